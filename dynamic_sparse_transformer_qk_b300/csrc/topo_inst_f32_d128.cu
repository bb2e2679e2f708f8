// Kernel instantiations for one (dtype, head dim) pair; compiled on its own
// so that the four pairs build in parallel.
#include "topo_launch.cuh"

namespace topo {
template struct Launcher<false, 128>;
}  // namespace topo
