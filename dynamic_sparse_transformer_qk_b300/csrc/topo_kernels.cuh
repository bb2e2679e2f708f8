// topo_kernels.cuh -- CUDA kernels for condensate-set ("topological")
// attention on sm_103a.
//
// Method: "The Condensate Theorem: Transformers are O(n), Not O(n^2)"
// explainer pages (gist.science, arXiv 2602.06317).  [fr S2]: per query the
// condensate set is the anchor 0, the W most recent positions and the top-k
// remaining positions by q . k.  [fr S3]: the softmax runs over that set only.
// [ko S3]: scores are recomputed every step, so every causal key is scored.
//
// Work decomposition (one CTA = one "split" of one column block):
//   column    one (query row, query head) pair.  The g = Hq/Hkv heads of a KV
//             group, and consecutive rows, share a KV head, so NC columns are
//             scored together against every K tile: one K read serves NC
//             queries (GQA sharing).
//   split     a contiguous key range of the column block.
//   producer  warp 4, lane 0: TMA loads of 64-key tiles (128-byte swizzle)
//             into a ring of `stages` shared-memory slots (mbarrier pipeline).
//   consumers warps 0..3: warp w scores tiles w, w+4, ...  Each lane scores 2
//             keys against NC columns with the float32 chain
//             acc = fma(q[c], k[c], acc), c = 0..d-1, the two keys sharing one
//             packed f32x2 FMA.
//   tail      the last CTA of a column block to finish (atomic counter; no CTA
//             ever waits on another) combines the splits' partial results.
#pragma once

#include <cuda_bf16.h>

#include "topo_device.cuh"

namespace topo {

// kSplitTail: the tensor-core select kernel only publishes its split lists;
// a dependent tail kernel merges them (one CTA per selection column).
// kEarlyBand: the tail kernel stages the window band before waiting for the
// select grid (measured to help when the select grid is one wave, and to cost
// ~25 us at B = 16 x 128K with seven waves).
enum : int { kDoIdx = 1, kDoPV = 2, kSaveThr = 4, kSplitTail = 8, kEarlyBand = 16 };

// Everything a kernel needs, passed by value.
struct Geom {
  int B, Hq, Hkv, g;
  long long n, nq, kv_stride;
  int W, topk;
  float scale;
  long long ncols;        // columns per (sequence, KV head) = nq * g
  long long ncb;          // column blocks per (sequence, KV head)
  long long L;            // keys per split (multiple of kTile)
  long long L2;           // keys per split of the units below hi_units (tensor-core select)
  long long hi_units;     // units that use L2 (one more split each); 0: none
  int nsplit_max;         // grid.x = ncb * nsplit_max
  int stages;             // ring depth
  int ncw;                // consumer warps that score tiles (1..kConsumerWarps, <= stages)
  int flags;
  const void* qp;
  const void* kp;
  const void* vp;
  float* out;
  int* idx;
  float* excl;
  int* status;
  int* counters;          // [unit]
  unsigned long long* lists;  // [unit][split][NC][KP]
  unsigned long long* thr;    // [unit][NC]
  float* partials;        // [unit][split][NC][...]
  // chunked-prefill tensor-core path (topo_prefill.cuh)
  unsigned* kmax;             // [B*Hkv] float bits of the largest |k_c| over keys 0..n-1
  float2* surv;               // [column][kPfLL] surviving candidates (tensor-core score, position bits)
  int* surv_cnt;              // [column] survivors, -1 when the buffer overflowed
  int* work;                  // work-queue counter of the scan kernel
  int* topsel;                // [row][k] selected positions ascending, -1 padded
  float* toplogit;            // [row][k] logits (scale * score) of topsel's positions
  long long nitems;           // scan work items (blocks of 128 columns)
  int items_per_head;         // blocks per (sequence, KV head)
  int thr_nc;                 // columns per unit of the excluded-mass pass
  // paged KV (tensor-core decode path): K and V are pools [blocks, Hkv,
  // block_size, d]; key j of sequence b lives in block
  // block_table[b * max_blocks + j / block_size].  Null table: contiguous.
  const int* block_table;
  const int* seq_lens;        // [B] causal length per sequence (clamped to nq..n), or null
  int max_blocks, block_size, num_blocks;
  int out_bf16;               // out holds bfloat16 values instead of float
};

constexpr int kStatusBadBlock = -7;  // TOPO_ERR_BAD_BLOCK: a block-table entry was out of range

// Row of key j of (sequence b, KV head h) in the K and V arrays: contiguous
// [B, Hkv, kv_stride] rows, or the paged pool's [blocks, Hkv, block_size]
// rows through the block table (an out-of-range entry is reported in the
// status word and read as block 0, so no access leaves the pool).
__device__ __forceinline__ long long kv_row(const Geom& G, int b, int h, long long j) {
  if (!G.block_table) return ((long long)b * G.Hkv + h) * G.kv_stride + j;
  int blk = G.block_table[(long long)b * G.max_blocks + j / G.block_size];
  if (blk < 0 || blk >= G.num_blocks) {
    if (G.status) atomicCAS(G.status, 0, kStatusBadBlock);
    blk = 0;
  }
  return ((long long)blk * G.Hkv + h) * G.block_size + j % G.block_size;
}

// Causal length of sequence b: the per-sequence length when given (clamped
// to nq..n, so that every query row has a position), else n.
__device__ __forceinline__ long long seq_len(const Geom& G, int b) {
  if (!G.seq_lens) return G.n;
  const long long s = G.seq_lens[b];
  return s < G.nq ? G.nq : (s > G.n ? G.n : s);
}

// Store output element i (float, or bf16 when G.out_bf16).
__device__ __forceinline__ void store_out(const Geom& G, long long i, float x) {
  if (G.out_bf16) reinterpret_cast<__nv_bfloat16*>(G.out)[i] = __float2bfloat16_rn(x);
  else G.out[i] = x;
}

struct ColInfo {
  long long pos;   // absolute position of the query row
  long long jhi;   // last candidate position (pos - W); < 1 means none
  long long row;   // flat row id over [B, Hq, nq]
  int active;
  int pad;
};

template <bool BF16, int D>
struct Shape {
  static constexpr int ES = BF16 ? 2 : 4;       // element bytes
  static constexpr int ROWB = D * ES;           // bytes per key row
  static constexpr int NCH = ROWB / 128;        // 128-byte column chunks per row
  static constexpr int EPC = 128 / ES;          // elements per column chunk
  static constexpr int EPV = 16 / ES;           // elements per 16-byte vector
  static constexpr int TILEB = kTile * ROWB;    // bytes of one K (or V) tile
  static constexpr int EPL = D / 32;            // output elements per lane
  static constexpr int BPL = ROWB / 32;         // row bytes per lane
  static_assert(ROWB % 128 == 0, "row must be a multiple of 128 bytes");
};

__host__ __device__ constexpr int cap_for(int KE) { return KE >= 2 ? 64 * KE : 128; }

// Shared-memory carve-up, identical on host and device.
struct Smem {
  int ring, bars, qd, buf, cols, misc, total;
  __host__ __device__ Smem(int stage_bytes, int stages, int D, int NC, int buf_bytes) {
    int o = 0;
    ring = o;  o += stages * stage_bytes;
    bars = o;  o += 2 * stages * 8;
    o = (o + 15) & ~15;
    qd = o;    o += D * NC * 8;
    buf = o;   o += (buf_bytes + 15) & ~15;
    cols = o;  o += NC * (int)sizeof(ColInfo);
    misc = o;  o += 64 + kConsumerWarps * 8 * 4;
    total = o + 1024;  // slack to align the base to 1024 bytes
  }
};

__device__ __forceinline__ uint8_t* aligned_smem_base() {
  extern __shared__ uint8_t dyn_smem[];
  const uint32_t a = smem_addr(dyn_smem);
  return dyn_smem + ((1024u - (a & 1023u)) & 1023u);
}

// Column table and the duplicated query vectors {q, q} of one column block.
template <bool BF16, int D, int NC>
__device__ void load_columns(const Geom& G, int b, int kvh, long long cb, ColInfo* cols,
                             float2* qd) {
  const long long nb = seq_len(G, b);
  const int tid = threadIdx.x;
  if (tid < NC) {
    const long long col = cb * NC + tid;
    ColInfo ci;
    ci.active = col < G.ncols;
    const long long r = ci.active ? col / G.g : 0;
    const int h = kvh * G.g + (ci.active ? (int)(col % G.g) : 0);
    ci.pos = nb - G.nq + r;
    ci.jhi = ci.active ? ci.pos - G.W : -1;
    ci.row = ((long long)b * G.Hq + h) * G.nq + r;
    ci.pad = 0;
    cols[tid] = ci;
  }
  __syncthreads();
  for (int i = tid; i < NC * D; i += blockDim.x) {
    const int hc = i / D, c = i % D;
    const float x = cols[hc].active ? load_elem<BF16>(G.qp, cols[hc].row * D + c) : 0.f;
    qd[c * NC + hc] = make_float2(x, x);
  }
}

// Score this lane's 2 keys (tile rows lane and lane+32) against NC columns
// with the float32 chain; .x is row lane, .y is row lane+32.
template <bool BF16, int D, int NC>
__device__ __forceinline__ void score_tile(const uint8_t* tile, const float2* qd, int lane,
                                           float2 (&acc)[NC]) {
  using S = Shape<BF16, D>;
#pragma unroll
  for (int h = 0; h < NC; ++h) acc[h] = make_float2(0.f, 0.f);
  const int sw = lane & 7;
  const uint8_t* row0 = tile + lane * 128;
  const uint8_t* row1 = tile + (lane + 32) * 128;
#pragma unroll
  for (int cc = 0; cc < S::NCH; ++cc) {
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16) {
      const int off = cc * (kTile * 128) + ((c16 ^ sw) << 4);
      const uint4 w0 = *reinterpret_cast<const uint4*>(row0 + off);
      const uint4 w1 = *reinterpret_cast<const uint4*>(row1 + off);
#pragma unroll
      for (int e = 0; e < S::EPV; ++e) {
        const float2 kv = make_float2(chunk_elem<BF16>(w0, e), chunk_elem<BF16>(w1, e));
        const int c = cc * S::EPC + c16 * S::EPV + e;
        if constexpr (NC == 1) {
          acc[0] = __ffma2_rn(qd[c], kv, acc[0]);
        } else {
          const float4* q4 = reinterpret_cast<const float4*>(qd + c * NC);
#pragma unroll
          for (int hp = 0; hp < NC / 2; ++hp) {
            const float4 qq = q4[hp];
            acc[2 * hp] = __ffma2_rn(make_float2(qq.x, qq.y), kv, acc[2 * hp]);
            acc[2 * hp + 1] = __ffma2_rn(make_float2(qq.z, qq.w), kv, acc[2 * hp + 1]);
          }
        }
      }
    }
  }
}

// The same float32 chain for one key row read from global memory.
template <bool BF16, int D, int NC>
__device__ __forceinline__ float score_row_global(const void* kbase, long long row,
                                                  const float2* qd, int hc) {
  using S = Shape<BF16, D>;
  const uint4* p =
      reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(kbase) + row * S::ROWB);
  uint4 w[S::ROWB / 16];  // every load of the row in flight at once
#pragma unroll
  for (int v = 0; v < S::ROWB / 16; ++v) w[v] = __ldg(p + v);
  float acc = 0.f;
#pragma unroll
  for (int v = 0; v < S::ROWB / 16; ++v) {
#pragma unroll
    for (int e = 0; e < S::EPV; ++e)
      acc = fmaf(qd[(v * S::EPV + e) * NC + hc].x, chunk_elem<BF16>(w[v], e), acc);
  }
  return acc;
}

// The same float32 chain with the query as plain floats in shared memory,
// read four at a time (one broadcast load per four products).
template <bool BF16, int D>
__device__ __forceinline__ float score_row_q4(const void* kbase, long long row, const float* q) {
  using S = Shape<BF16, D>;
  const uint4* p =
      reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(kbase) + row * S::ROWB);
  const float4* q4 = reinterpret_cast<const float4*>(q);
  float acc = 0.f;
#pragma unroll 4
  for (int v = 0; v < S::ROWB / 16; ++v) {
    const uint4 w = __ldg(p + v);
#pragma unroll
    for (int h = 0; h < S::EPV / 4; ++h) {
      const float4 qq = q4[v * (S::EPV / 4) + h];
      acc = fmaf(qq.x, chunk_elem<BF16>(w, 4 * h + 0), acc);
      acc = fmaf(qq.y, chunk_elem<BF16>(w, 4 * h + 1), acc);
      acc = fmaf(qq.z, chunk_elem<BF16>(w, 4 * h + 2), acc);
      acc = fmaf(qq.w, chunk_elem<BF16>(w, 4 * h + 3), acc);
    }
  }
  return acc;
}

// This lane's EPL consecutive elements (lane*EPL ...) of a row, widened.
template <bool BF16, int D>
__device__ __forceinline__ void lane_elems(const uint8_t* p, float (&v)[D / 32]) {
  using S = Shape<BF16, D>;
  if constexpr (S::BPL == 4) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    if constexpr (BF16) {
      v[0] = __uint_as_float(w << 16);
      v[1] = __uint_as_float(w & 0xffff0000u);
    } else {
      v[0] = __uint_as_float(w);
    }
  } else if constexpr (S::BPL == 8) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    if constexpr (BF16) {
      v[0] = __uint_as_float(w.x << 16);
      v[1] = __uint_as_float(w.x & 0xffff0000u);
      v[2] = __uint_as_float(w.y << 16);
      v[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
      v[0] = __uint_as_float(w.x);
      v[1] = __uint_as_float(w.y);
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    v[0] = __uint_as_float(w.x);
    v[1] = __uint_as_float(w.y);
    v[2] = __uint_as_float(w.z);
    v[3] = __uint_as_float(w.w);
  }
}

// Byte offset of this lane's slice of row r inside a swizzled tile of ROWS
// rows (each 128-byte column chunk of the rows stored contiguously).
template <bool BF16, int D, int ROWS = kTile>
__device__ __forceinline__ int tile_lane_offset(int r, int lane) {
  using S = Shape<BF16, D>;
  const int byte = lane * S::BPL;
  const int cc = byte >> 7, o = byte & 127;
  return cc * (ROWS * 128) + r * 128 + ((((o >> 4) ^ (r & 7))) << 4) + (o & 15);
}

// ------------------------------------------------------------ pipeline -----

// Producer (one thread): TMA loads of tiles [0, ntiles); each stage holds the
// K tile and, when map_v is given, the V tile behind it.  Returns the number
// of tiles issued.
template <bool BF16, int D>
__device__ int produce_tiles(const CUtensorMap* map_k, const CUtensorMap* map_v, long long row0,
                             int ntiles, int stages, uint8_t* ring, uint64_t* full,
                             uint64_t* empty, volatile int* abort_flag, int* status) {
  using S = Shape<BF16, D>;
  const int stage_bytes = map_v ? 2 * S::TILEB : S::TILEB;
  int t = 0;
  for (; t < ntiles; ++t) {
    if (*abort_flag) break;
    const int s = t % stages;
    const uint32_t round = (uint32_t)(t / stages);
    if (!mbar_wait(&empty[s], (round & 1u) ^ 1u)) {
      set_status(status, kStatusTimeout);
      *abort_flag = 1;
      break;
    }
    uint8_t* dst = ring + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
    const int y = (int)(row0 + (long long)t * kTile);
#pragma unroll
    for (int cc = 0; cc < S::NCH; ++cc)
      tma_load_2d(dst + cc * (kTile * 128), map_k, cc * S::EPC, y, &full[s]);
    if (map_v) {
#pragma unroll
      for (int cc = 0; cc < S::NCH; ++cc)
        tma_load_2d(dst + S::TILEB + cc * (kTile * 128), map_v, cc * S::EPC, y, &full[s]);
    }
  }
  return t;
}

// Producer clean-up: wait (bounded) until the last load issued into every
// stage has landed, so that no copy into shared memory outlives the CTA.
__device__ __forceinline__ void drain_tiles(int issued, int stages, uint64_t* full, int* status) {
  for (int s = 0; s < stages && s < issued; ++s) {
    const int last = s + stages * ((issued - 1 - s) / stages);
    if (!mbar_wait(&full[s], (uint32_t)(last / stages) & 1u)) set_status(status, kStatusTimeout);
  }
}

// Consumer loop of warp `warp` (< ncw <= stages): tiles warp, warp+ncw, ...;
// body(t, stage_ptr).  Tile t fills stage s = t % stages for the R-th time
// (R = t / stages).  A parity wait alone cannot tell fill R from fill R-2, and
// another warp may still hold fill R-1 of the stage, so the warp first waits
// until fill R-1 has been consumed (phase R-1 of empty[s]), then for fill R to
// land (phase R of full[s]).  The first wait is unambiguous because the
// producer issued tile t - stages (<= this warp's previous tile, as ncw <=
// stages) only after tile t - 2 stages had been consumed, and the second
// because tile t itself is not consumed yet.  Warps >= ncw take no tiles.
template <class Body>
__device__ __forceinline__ void consume_tiles(int warp, int ncw, int ntiles, int stages,
                                              int stage_bytes, uint8_t* ring, uint64_t* full,
                                              uint64_t* empty, volatile int* abort_flag,
                                              int* status, Body&& body) {
  const int lane = threadIdx.x & 31;
  if (warp >= ncw) return;
  for (int t = warp; t < ntiles; t += ncw) {
    const int s = t % stages;
    const uint32_t round = (uint32_t)(t / stages);
    const bool ok = __all_sync(kFull, (round == 0u || mbar_wait(&empty[s], (round - 1u) & 1u)) &&
                                          mbar_wait(&full[s], round & 1u));
    const int ab = __shfl_sync(kFull, *abort_flag, 0);
    if (!ok || ab) {
      if (!ok && lane == 0) {
        set_status(status, kStatusTimeout);
        *abort_flag = 1;
      }
      break;
    }
    body(t, ring + (size_t)s * stage_bytes);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// Pipeline set-up: barriers, misc flags.
__device__ __forceinline__ void init_pipeline(int stages, uint64_t* full, uint64_t* empty,
                                              volatile int* misc) {
  if (threadIdx.x == 0) {
    misc[0] = 0;  // abort
    misc[1] = 0;  // this CTA finishes its column block
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
}

// Announce completion of this split; true in the CTA that finished last.
__device__ __forceinline__ bool finish_split(int* counter, int nsplit, volatile int* misc) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(counter, 1);
    misc[1] = (prev == nsplit - 1);
  }
  __syncthreads();
  const bool last = misc[1] != 0;
  if (last) __threadfence();
  return last;
}

// ---------------------------------------------------- candidate buffers ----

// Sort the buffer, keep its k best at [0, k) and return the k-th best key,
// the new admission threshold (k >= 1).  The caller sets its count to k.
template <int EC, int KE>
__device__ __noinline__ uint64_t compact_buffer(uint64_t* buf, int cnt, int k, int lane) {
  __syncwarp();
  uint64_t x[EC];
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const int i = e * 32 + lane;
    x[e] = i < cnt ? buf[i] : 0ull;
  }
  warp_sort_desc<EC>(x, lane);
  __syncwarp();
#pragma unroll
  for (int e = 0; e < KE; ++e) buf[e * 32 + lane] = x[e];
  const uint64_t thr = warp_list_get<EC>(x, k - 1);
  __syncwarp();
  return thr;
}

// Offer one key per lane (0 = nothing) to a warp's candidate buffer.
template <int EC, int KE>
__device__ __forceinline__ void offer(uint64_t* buf, uint64_t& thr, int& cnt, uint64_t key, int k,
                                      int lane) {
  bool flag = key > thr;
  unsigned mask = __ballot_sync(kFull, flag);
  if (mask == 0u) return;
  if (cnt + __popc(mask) > 32 * EC) {
    thr = compact_buffer<EC, KE>(buf, cnt, k, lane);
    cnt = k;
    flag = key > thr;
    mask = __ballot_sync(kFull, flag);
    if (mask == 0u) return;
  }
  if (flag) buf[cnt + __popc(mask & ((1u << lane) - 1u))] = key;
  cnt += __popc(mask);
}

// ------------------------------------------------------ softmax over C_i ----

// One warp: out = sum_e w_e v_{j(e)} / sum_e w_e over entries e in [0, m) with
// positions j = entry(e) (negative: skip), w_e = exp(l_e - max l), l_e =
// scale * (float32 chain q . k_j); float32 online softmax in chunks of 256.
template <bool BF16, int D, class Entry, class Score, class RowOf>
__device__ void warp_softmax_pv_with(const Geom& G, RowOf&& row_of, Score&& score, long long m,
                                     Entry&& entry, float* wsm, int* jsm, long long out_off,
                                     int lane) {
  using S = Shape<BF16, D>;
  float mrun = -INFINITY, Z = 0.f;
  float acc[S::EPL];
#pragma unroll
  for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
  const uint8_t* vbase = reinterpret_cast<const uint8_t*>(G.vp);
  for (long long e0 = 0; e0 < m; e0 += 256) {
    const int cnt = (int)(m - e0 < 256 ? m - e0 : 256);
    float lmax = -INFINITY;
    for (int i = lane; i < cnt; i += 32) {
      const long long j = entry(e0 + i);
      float l = -INFINITY;
      if (j >= 0) {
        // start the V row on its way to L2 while the logit is computed
        const uint8_t* vrow = vbase + row_of(j) * S::ROWB;
#pragma unroll
        for (int o = 0; o < S::ROWB; o += 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(vrow + o));
        l = G.scale * score(row_of(j));
      }
      wsm[i] = l;
      jsm[i] = (int)j;
      lmax = fmaxf(lmax, l);
    }
    lmax = warp_max(lmax);
    const float mnew = fmaxf(mrun, lmax);
    __syncwarp();
    if (mnew == -INFINITY) continue;
    const float alpha = (mrun == -INFINITY) ? 0.f : expf(mrun - mnew);
    float zs = 0.f;
    for (int i = lane; i < cnt; i += 32) {
      const float l = wsm[i];
      const float w = (l == -INFINITY) ? 0.f : expf(l - mnew);
      wsm[i] = w;
      zs += w;
    }
    Z = Z * alpha + warp_sum(zs);
#pragma unroll
    for (int e = 0; e < S::EPL; ++e) acc[e] *= alpha;
    mrun = mnew;
    __syncwarp();
    // gather V in batches of 8 rows so that 8 loads are in flight per lane
    // (a skipped entry has weight 0 and reads row 0, which always exists)
    int i = 0;
    for (; i + 8 <= cnt; i += 8) {
      float v[8][S::EPL];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = jsm[i + u];
        lane_elems<BF16, D>(vbase + row_of(j >= 0 ? j : 0) * S::ROWB + lane * S::BPL, v[u]);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float w = wsm[i + u];
#pragma unroll
        for (int e = 0; e < S::EPL; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
      }
    }
    for (; i < cnt; ++i) {
      const int j = jsm[i];
      if (j < 0) continue;
      const float w = wsm[i];
      float v[S::EPL];
      lane_elems<BF16, D>(vbase + row_of(j) * S::ROWB + lane * S::BPL, v);
#pragma unroll
      for (int e = 0; e < S::EPL; ++e) acc[e] = fmaf(w, v[e], acc[e]);
    }
    __syncwarp();
  }
#pragma unroll
  for (int e = 0; e < S::EPL; ++e)
    store_out(G, out_off + lane * S::EPL + e, Z > 0.f ? acc[e] / Z : 0.f);
}

// The float32 chain for one key row held in shared memory (linear layout).
template <bool BF16, int D, int NC>
__device__ __forceinline__ float score_row_smem(const uint8_t* krow, const float2* qd, int hc) {
  using S = Shape<BF16, D>;
  const uint4* p = reinterpret_cast<const uint4*>(krow);
  float acc = 0.f;
#pragma unroll 4
  for (int v = 0; v < S::ROWB / 16; ++v) {
    const uint4 w = p[v];
#pragma unroll
    for (int e = 0; e < S::EPV; ++e)
      acc = fmaf(qd[(v * S::EPV + e) * NC + hc].x, chunk_elem<BF16>(w, e), acc);
  }
  return acc;
}

template <bool BF16, int D, int NC, class Entry>
__device__ __forceinline__ void warp_softmax_pv(const Geom& G, int b, int kvh, const float2* qd,
                                                int hc, long long m, Entry&& entry, float* wsm,
                                                int* jsm, long long out_off, int lane) {
  warp_softmax_pv_with<BF16, D>(
      G, [&](long long j) { return kv_row(G, b, kvh, j); },
      [&](long long row) { return score_row_global<BF16, D, NC>(G.kp, row, qd, hc); }, m, entry,
      wsm, jsm, out_off, lane);
}

// Tail of the select kernels, run by the CTA that finished a column block
// last, or by a CTA of the dependent tail kernel for the columns h0..h1-1
// (the others inactive): merge the splits' exact top-k lists, then per column
// write C_i, the k-th key (for the excluded-mass pass) and the softmax over
// C_i.  `run` holds NC * KP keys; `scratch` (1024-byte aligned, at least
// NC*KP*4 + NC*8 + 1024 + NW*2048 bytes and one split's lists) is free shared
// memory.
//
// Fast path, when everything fits in `scratch`: the rows every softmax needs
// (the band covering the block's windows and the anchor, then each column's
// top-k) are staged with bulk copies, the band ones first (part 1 issues only
// those, part 2 does the rest, part 0 both); the lists of all splits come in
// with one bulk copy, or, for a single selection column, every warp merges a
// strided subset of its lists from L2 and warp 0 the warps' results; logits
// are computed by all threads, then one thread per (column, output element)
// forms the weighted sum of V.  Otherwise the lists are read in chunks and one
// warp per column reads its rows from global memory.  All threads of the CTA
// call this; warps 0..NW-1 do the per-column work.
//
// GROUP: the lists are per selection column s (one per row of the block, for
// the g heads col = s*g .. s*g+g-1, see topo_select_tc_kernel); after the
// merge every column takes its row's list, one idx row per (KV head, row) is
// written, and the top-k rows are staged once per row.
template <bool BF16, int D, int NC, int KE, int NW, bool GROUP = false>
__device__ __noinline__ void select_tail(const Geom& G, long long unit, int nsplit, int b, int kvh,
                                         const ColInfo* cols, const float2* qd, uint64_t* run,
                                         uint8_t* scratch, int scratch_bytes, int h0 = 0,
                                         int h1 = NC, int part = 0) {
  using S = Shape<BF16, D>;
  constexpr int KP = 32 * KE;
  // a staged slot: the K row, then the V row, then 16 bytes of padding, so
  // that consecutive slots start four banks apart (threads scoring
  // consecutive entries read without bank conflicts)
  constexpr int SLOT = 2 * S::ROWB + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kk = G.topk;
  const long long cmax = 1 + (long long)G.W + kk;
  const int nsel = GROUP ? NC / G.g : NC;  // selection columns

  // fixed part of the scratch
  int* topj_all = reinterpret_cast<int*>(scratch);                       // [NC][KP]
  int* tcount = reinterpret_cast<int*>(scratch + NC * KP * 4);            // [NC]
  float* zsum = reinterpret_cast<float*>(scratch + NC * KP * 4 + NC * 4); // [NC]
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      scratch + ((NC * KP * 4 + NC * 8 + 15) & ~15));                     // lists, band, top-k
  const int v0 = (NC * KP * 4 + NC * 8 + 32 + 1023) & ~1023;
  // variable part: lists | logits | staged rows
  const int per_split = NC * KP;  // entries
  const long long list_bytes = (long long)nsplit * per_split * 8;
  const int off_lw = (int)((v0 + list_bytes + 1023) & ~1023LL);
  const long long mmax = cmax;  // entries per column at most
  const int off_stage = (int)((off_lw + NC * mmax * 4 + NC * 4 + 1023) & ~1023LL);

  long long plo = 0x7fffffffffffffffLL, phi = -1;
  for (int h = 0; h < NC; ++h)
    if (cols[h].active) {
      plo = cols[h].pos < plo ? cols[h].pos : plo;
      phi = cols[h].pos > phi ? cols[h].pos : phi;
    }
  const long long band_lo = plo - G.W + 1 > 0 ? plo - G.W + 1 : 0;
  const long long nb = phi - band_lo + 1;
  const long long anchor_slot = band_lo == 0 ? 0 : nb;
  const long long top0 = nb + 1;
  // top-k slots for columns h0..h1-1 (the columns that may be active)
  const long long nslots = top0 + (long long)(h1 - h0) * kk;
  const bool fast = (G.flags & kDoPV) && phi >= 0 &&
                    (long long)off_stage + nslots * SLOT + (long long)NC * mmax * 4 <=
                        scratch_bytes;
  uint8_t* stage = scratch + off_stage;
  float* lw = reinterpret_cast<float*>(scratch + off_lw);
  const uint8_t* kb = reinterpret_cast<const uint8_t*>(G.kp);
  const uint8_t* vb = reinterpret_cast<const uint8_t*>(G.vp);

  for (int i = tid; i < NC * KP; i += blockDim.x) run[i] = 0ull;
  // One selection column (the tail kernel's CTAs): every warp merges a
  // strided subset of the splits' lists of that column, read from L2, and
  // warp 0 merges the warps' results (NW partial lists in the list area).
  const bool one_sel = (GROUP ? h1 - h0 == G.g : h1 - h0 == 1) &&
                       (long long)nsplit * NC >= NW;
  // part 1 issues the band and anchor rows only (they do not depend on the
  // selection: the tail kernel starts them before waiting for the lists);
  // part 2 is the rest; part 0 both.
  if (fast && part != 2) {
    if (tid == 0) {
      for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
      mbar_arrive_expect_tx(&bars[1], (uint32_t)((nb + (band_lo == 0 ? 0 : 1)) * 2 * S::ROWB));
    for (long long sl = tid; sl < top0; sl += blockDim.x) {
      long long row = sl < nb ? band_lo + sl : (band_lo == 0 ? -1 : 0);
      if (row < 0) continue;
      uint8_t* dst = stage + (size_t)sl * SLOT;
      const long long gr = kv_row(G, b, kvh, row);
      bulk_copy_g2s(dst, kb + gr * S::ROWB, S::ROWB, &bars[1]);
      bulk_copy_g2s(dst + S::ROWB, vb + gr * S::ROWB, S::ROWB, &bars[1]);
    }
  }
  if (part == 1) return;
  if (fast) {
    // the split lists were written by other CTAs through the generic proxy
    asm volatile("fence.proxy.async;" ::: "memory");
    __syncthreads();
    if (tid == 0 && !one_sel) {
      mbar_arrive_expect_tx(&bars[0], (uint32_t)list_bytes);
      bulk_copy_g2s(scratch + v0, G.lists + (size_t)unit * G.nsplit_max * per_split,
                    (uint32_t)list_bytes, &bars[0]);
    }
    if (one_sel) {
      const int hs = GROUP ? h0 / G.g : h0;
      uint64_t a[KE];
#pragma unroll
      for (int e = 0; e < KE; ++e) a[e] = 0ull;
      for (int s2 = warp; s2 < nsplit; s2 += NW) {
        const unsigned long long* src =
            G.lists + ((size_t)unit * G.nsplit_max + s2) * per_split + (size_t)hs * KP;
        uint64_t bb[KE];
#pragma unroll
        for (int e = 0; e < KE; ++e) bb[e] = __ldcg(src + e * 32 + lane);
        warp_merge_desc<KE>(a, bb, lane);
      }
      uint64_t* part = reinterpret_cast<uint64_t*>(scratch + v0);  // [NW][KP]
#pragma unroll
      for (int e = 0; e < KE; ++e) part[warp * KP + e * 32 + lane] = a[e];
      __syncthreads();
      if (warp == 0) {
        for (int w = 1; w < NW; ++w) {
          uint64_t bb[KE];
#pragma unroll
          for (int e = 0; e < KE; ++e) bb[e] = part[w * KP + e * 32 + lane];
          warp_merge_desc<KE>(a, bb, lane);
        }
#pragma unroll
        for (int e = 0; e < KE; ++e) run[hs * KP + e * 32 + lane] = a[e];
      }
      __syncthreads();
    }
    if (!one_sel && !mbar_wait(&bars[0], 0) && tid == 0) set_status(G.status, kStatusTimeout);
    for (int h = warp; h < nsel && !one_sel; h += NW) {
      if (!cols[GROUP ? h * G.g : h].active) continue;
      const uint64_t* lb = reinterpret_cast<const uint64_t*>(scratch + v0);
      uint64_t a[KE];
#pragma unroll
      for (int e = 0; e < KE; ++e) a[e] = lb[h * KP + e * 32 + lane];
      for (int s = 1; s < nsplit; ++s) {
        uint64_t bb[KE];
#pragma unroll
        for (int e = 0; e < KE; ++e) bb[e] = lb[(size_t)s * per_split + h * KP + e * 32 + lane];
        warp_merge_desc<KE>(a, bb, lane);
      }
#pragma unroll
      for (int e = 0; e < KE; ++e) run[h * KP + e * 32 + lane] = a[e];
    }
    __syncthreads();
  } else {
    int chunk = (scratch_bytes - v0) / (per_split * 8);
    if (chunk < 1) chunk = 1;
    uint64_t* lbuf = reinterpret_cast<uint64_t*>(scratch + v0);
    __syncthreads();
    for (int s0 = 0; s0 < nsplit; s0 += chunk) {
      const int s1 = s0 + chunk < nsplit ? s0 + chunk : nsplit;
      const unsigned long long* src = G.lists + ((size_t)unit * G.nsplit_max + s0) * per_split;
      const int total = (s1 - s0) * per_split;
      for (int i = tid; i < total; i += blockDim.x) lbuf[i] = __ldcg(src + i);
      __syncthreads();
      for (int h = warp; h < nsel; h += NW) {
        if (!cols[GROUP ? h * G.g : h].active) continue;
        uint64_t a[KE];
#pragma unroll
        for (int e = 0; e < KE; ++e) a[e] = run[h * KP + e * 32 + lane];
        for (int s = 0; s < s1 - s0; ++s) {
          uint64_t bb[KE];
#pragma unroll
          for (int e = 0; e < KE; ++e) bb[e] = lbuf[(size_t)s * per_split + h * KP + e * 32 + lane];
          warp_merge_desc<KE>(a, bb, lane);
        }
#pragma unroll
        for (int e = 0; e < KE; ++e) run[h * KP + e * 32 + lane] = a[e];
      }
      __syncthreads();
    }
  }

  if constexpr (GROUP) {
    // every column takes its row's merged list (read all, then write)
    constexpr int PER = (NC * KP + 255) / 256;
    uint64_t tmp[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int i = tid + q * blockDim.x;
      tmp[q] = i < NC * KP ? run[((i / KP) / G.g) * KP + i % KP] : 0ull;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int i = tid + q * blockDim.x;
      if (i < NC * KP) run[i] = tmp[q];
    }
    __syncthreads();
  }

  // per column: the k-th key, the selected positions (ascending) and C_i
  for (int h = warp; h < NC; h += NW) {
    if (!cols[h].active) continue;
    uint64_t a[KE];
#pragma unroll
    for (int e = 0; e < KE; ++e) {
      const int i = e * 32 + lane;
      a[e] = i < kk ? run[h * KP + i] : 0ull;
    }
    int t = 0;
#pragma unroll
    for (int e = 0; e < KE; ++e) t += __popc(__ballot_sync(kFull, a[e] != 0ull));
    if (G.flags & kSaveThr) {
      const uint64_t kth = kk > 0 ? warp_list_get<KE>(a, kk - 1) : 0ull;
      if (lane == 0)
        G.thr[(size_t)unit * NC + h] = kk == 0 ? ~0ull : (t < kk ? 0ull : kth);
    }
    uint64_t y[KE];
#pragma unroll
    for (int e = 0; e < KE; ++e) y[e] = a[e] ? (~0ull - (uint64_t)key_pos(a[e])) : 0ull;
    warp_sort_desc<KE>(y, lane);
    int* topj = topj_all + h * KP;
#pragma unroll
    for (int e = 0; e < KE; ++e) topj[e * 32 + lane] = y[e] ? (int)(~0ull - y[e]) : -1;
    if (lane == 0) tcount[h] = t;
    __syncwarp();
    if ((G.flags & kDoIdx) && (!GROUP || h % G.g == 0)) {
      const long long p = cols[h].pos;
      const bool wide = p - G.W + 1 <= 0;  // the window reaches the anchor
      const long long mEnt = wide ? p + 1 : 1 + t + G.W;
      const long long wlo = p - G.W + 1;
      // one row per (sequence, KV head, row) in group mode
      const long long irow =
          GROUP ? ((long long)b * G.Hkv + kvh) * G.nq + (p - (seq_len(G, b) - G.nq)) : cols[h].row;
      int* dst = G.idx + irow * cmax;
      for (long long e = lane; e < cmax; e += 32) {
        long long v = -1;
        if (e < mEnt) v = wide ? e : (e == 0 ? 0 : (e <= t ? topj[e - 1] : wlo + (e - 1 - t)));
        dst[e] = (int)v;
      }
    }
  }
  if (!(G.flags & kDoPV)) return;
  __syncthreads();

  if (!fast) {
    // one warp per column, rows from global memory
    float* wsm_all = reinterpret_cast<float*>(scratch + v0);
    for (int h = warp; h < NC; h += NW) {
      if (!cols[h].active) continue;
      const int t = tcount[h];
      const int* topj = topj_all + h * KP;
      const long long p = cols[h].pos;
      const bool wide = p - G.W + 1 <= 0;
      const long long mEnt = wide ? p + 1 : 1 + t + G.W;
      const long long wlo = p - G.W + 1;
      float* wsm = wsm_all + warp * 512;
      int* jsm = reinterpret_cast<int*>(wsm + 256);
      auto entry = [&](long long e) -> long long {
        if (wide) return e;
        if (e == 0) return 0;
        if (e <= t) return topj[e - 1];
        return wlo + (e - 1 - t);
      };
      warp_softmax_pv<BF16, D, NC>(G, b, kvh, qd, h, mEnt, entry, wsm, jsm, cols[h].row * D,
                                   lane);
      __syncwarp();
    }
    return;
  }

  // the columns' top-k rows
  {
    long long tbytes = 0;
    for (int h = 0; h < NC; ++h)
      if (cols[h].active && (!GROUP || h % G.g == 0)) tbytes += (long long)tcount[h] * 2 * S::ROWB;
    if (tid == 0) mbar_arrive_expect_tx(&bars[2], (uint32_t)tbytes);
    for (long long sl = tid; sl < (long long)NC * kk; sl += blockDim.x) {
      const int h = (int)(sl / kk), i = (int)(sl % kk);
      if (!cols[h].active || i >= tcount[h] || (GROUP && h % G.g != 0)) continue;
      const long long row = topj_all[h * KP + i];
      uint8_t* dst = stage + (size_t)(top0 + (long long)(h - h0) * kk + i) * SLOT;
      const long long gr = kv_row(G, b, kvh, row);
      bulk_copy_g2s(dst, kb + gr * S::ROWB, S::ROWB, &bars[2]);
      bulk_copy_g2s(dst + S::ROWB, vb + gr * S::ROWB, S::ROWB, &bars[2]);
    }
    const bool ok = mbar_wait(&bars[1], 0) && mbar_wait(&bars[2], 0);
    if (!ok && tid == 0) set_status(G.status, kStatusTimeout);
    if (__syncthreads_or(!ok)) return;
  }

  // per-column constants, once: entries m, top-k count t, window start
  int* cm = reinterpret_cast<int*>(scratch + off_lw + NC * mmax * 4);   // [NC] entries
  int* slot_tab = reinterpret_cast<int*>(stage + nslots * SLOT);  // [NC][mmax]
  if (tid < NC) {
    const int h = tid;
    const long long p = cols[h].pos;
    cm[h] = !cols[h].active ? 0 : (int)(p - G.W + 1 <= 0 ? p + 1 : 1 + tcount[h] + G.W);
  }
  __syncthreads();
  const float scale = G.scale;
  const long long W = G.W;
  // logits of every (column, entry), all threads; the entry's staged slot is
  // kept for the weighted sum
  for (long long i = tid; i < (long long)NC * mmax; i += blockDim.x) {
    const int h = (int)(i / mmax);
    const int e = (int)(i % mmax);
    if (e >= cm[h]) continue;
    const long long p = cols[h].pos;
    const int t = tcount[h];
    long long sl;
    if (p - W + 1 <= 0) sl = e - band_lo;  // 0..p lies in the band, which starts at 0
    else if (e == 0) sl = anchor_slot;
    else if (e <= t) sl = top0 + (long long)((GROUP ? h - h % G.g : h) - h0) * kk + (e - 1);
    else sl = (p - W + 1) + (e - 1 - t) - band_lo;
    slot_tab[i] = (int)sl;
    lw[i] = scale * score_row_smem<BF16, D, NC>(stage + (size_t)sl * SLOT, qd, h);
  }
  __syncthreads();
  // per column: max, weights, normaliser
  for (int h = warp; h < NC; h += NW) {
    const int m = cm[h];
    if (m == 0) continue;
    float* l = lw + (size_t)h * mmax;
    float mx = -INFINITY;
    for (int e = lane; e < m; e += 32) mx = fmaxf(mx, l[e]);
    mx = warp_max(mx);
    float zs = 0.f;
    for (int e = lane; e < m; e += 32) {
      const float w = expf(l[e] - mx);
      l[e] = w;
      zs += w;
    }
    zs = warp_sum(zs);
    if (lane == 0) zsum[h] = zs;
  }
  __syncthreads();
  // out[h][c..c+1] = sum_e w_e v_e[c..c+1] / Z, one thread per (column, element pair)
  for (int i = tid; i < NC * (D / 2); i += blockDim.x) {
    const int h = i / (D / 2), c = 2 * (i % (D / 2));
    const int m = cm[h];
    if (m == 0) continue;
    const float* w = lw + (size_t)h * mmax;
    const int* st = slot_tab + (size_t)h * mmax;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
    for (int e = 0; e < m; ++e) {
      const uint8_t* vr = stage + (size_t)st[e] * SLOT + S::ROWB;
      float v0, v1;
      if constexpr (BF16) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(vr + c * 2);
        v0 = __uint_as_float(u << 16);
        v1 = __uint_as_float(u & 0xffff0000u);
      } else {
        const float2 f = *reinterpret_cast<const float2*>(vr + c * 4);
        v0 = f.x;
        v1 = f.y;
      }
      a0 = fmaf(w[e], v0, a0);
      a1 = fmaf(w[e], v1, a1);
    }
    const float z = zsum[h];
    const long long o = cols[h].row * D + c;
    store_out(G, o, z > 0.f ? a0 / z : 0.f);
    store_out(G, o + 1, z > 0.f ? a1 / z : 0.f);
  }
}

// ================================================== fused select kernel =====
//
// Scores the candidates 1..p-W of every column in this split, keeps each
// column's top-k, and in the last CTA of the column block: merges the
// splits' lists, writes C_i (idx), the k-th key (for the excluded-mass pass)
// and the softmax-over-C_i output.
template <bool BF16, int D, int NC, int KE>
__global__ void __launch_bounds__(kThreads, 1)
    topo_select_kernel(const __grid_constant__ CUtensorMap map_k, const Geom G) {
  using S = Shape<BF16, D>;
  constexpr int EC = cap_for(KE) / 32;
  constexpr int CAP = 32 * EC;
  constexpr int KP = 32 * KE;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const long long cb = blockIdx.x / G.nsplit_max;
  const int split = (int)(blockIdx.x % G.nsplit_max);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kk = G.topk;

  // candidate range of this column block: 1..jmax (the last column has the
  // largest position)
  const long long last_col = ((cb + 1) * NC < G.ncols ? (cb + 1) * NC : G.ncols) - 1;
  const long long pos_max = G.n - G.nq + last_col / G.g;
  const long long jmax = kk > 0 ? pos_max - G.W : 0;
  const long long ncand = jmax > 0 ? jmax : 0;
  const int nsplit = ncand > 0 ? (int)((ncand + G.L - 1) / G.L) : 1;
  if (split >= nsplit) return;
  const long long ks = 1 + (long long)split * G.L;
  const long long ke = (ks + G.L - 1 < jmax) ? ks + G.L - 1 : jmax;  // inclusive
  const int ntiles = ke >= ks ? (int)((ke - ks + kTile) / kTile) : 0;
  const long long unit = ((long long)b * G.Hkv + kvh) * G.ncb + cb;

  uint8_t* sm = aligned_smem_base();
  const Smem L(S::TILEB, G.stages, D, NC, kConsumerWarps * NC * CAP * 8);
  uint8_t* ring = sm + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + G.stages;
  float2* qd = reinterpret_cast<float2*>(sm + L.qd);
  uint64_t* wbuf = reinterpret_cast<uint64_t*>(sm + L.buf);
  ColInfo* cols = reinterpret_cast<ColInfo*>(sm + L.cols);
  volatile int* misc = reinterpret_cast<volatile int*>(sm + L.misc);

  init_pipeline(G.stages, full, empty, misc);
  load_columns<BF16, D, NC>(G, b, kvh, cb, cols, qd);
  __syncthreads();

  const long long row0 = ((long long)b * G.Hkv + kvh) * G.kv_stride + ks;
  int issued = 0;
  if (warp == kConsumerWarps) {
    if (lane == 0 && ntiles > 0) {
      prefetch_tmap(&map_k);
      issued = produce_tiles<BF16, D>(&map_k, nullptr, row0, ntiles, G.stages, ring, full, empty,
                                      misc, G.status);
      drain_tiles(issued, G.stages, full, G.status);
    }
  } else {
    uint64_t thr[NC];
    int cnt[NC];
#pragma unroll
    for (int h = 0; h < NC; ++h) {
      thr[h] = 0ull;
      cnt[h] = 0;
    }
    uint64_t* mybuf = wbuf + (size_t)warp * NC * CAP;
    long long jh[NC];
#pragma unroll
    for (int h = 0; h < NC; ++h) jh[h] = cols[h].jhi < ke ? cols[h].jhi : ke;
    consume_tiles(warp, G.ncw, ntiles, G.stages, S::TILEB, ring, full, empty, misc, G.status,
                  [&](int t, const uint8_t* tile) {
                    float2 acc[NC];
                    score_tile<BF16, D, NC>(tile, qd, lane, acc);
                    const long long jA = ks + (long long)t * kTile + lane, jB = jA + 32;
#pragma unroll
                    for (int h = 0; h < NC; ++h) {
                      const uint64_t kA = jA <= jh[h] ? rank_key(acc[h].x, (uint32_t)jA) : 0ull;
                      const uint64_t kB = jB <= jh[h] ? rank_key(acc[h].y, (uint32_t)jB) : 0ull;
                      offer<EC, KE>(mybuf + h * CAP, thr[h], cnt[h], kA, kk, lane);
                      offer<EC, KE>(mybuf + h * CAP, thr[h], cnt[h], kB, kk, lane);
                    }
                  });
    // final per-warp list: the k best, sorted, at [0, KP) of each buffer
    int* wcnt = reinterpret_cast<int*>(sm + L.misc) + 16 + warp * NC;
#pragma unroll
    for (int h = 0; h < NC; ++h)
      if (lane == 0) wcnt[h] = cnt[h];
    __syncwarp();
#pragma unroll 1
    for (int h = 0; h < NC; ++h) {
      __syncwarp();
      const int ch = wcnt[h];
      uint64_t x[EC];
#pragma unroll
      for (int e = 0; e < EC; ++e) {
        const int i = e * 32 + lane;
        x[e] = i < ch ? mybuf[h * CAP + i] : 0ull;
      }
      warp_sort_desc<EC>(x, lane);
      __syncwarp();
#pragma unroll
      for (int e = 0; e < KE; ++e) {
        const int i = e * 32 + lane;
        mybuf[h * CAP + i] = i < kk ? x[e] : 0ull;
      }
    }
  }
  __syncthreads();

  // merge the consumer warps' lists and publish this split's list
  for (int h = warp; h < NC; h += kWarps) {
    uint64_t a[KE];
#pragma unroll
    for (int e = 0; e < KE; ++e) a[e] = wbuf[h * CAP + e * 32 + lane];
    for (int w = 1; w < kConsumerWarps; ++w) {
      uint64_t bb[KE];
#pragma unroll
      for (int e = 0; e < KE; ++e) bb[e] = wbuf[((size_t)w * NC + h) * CAP + e * 32 + lane];
      warp_merge_desc<KE>(a, bb, lane);
    }
    unsigned long long* dst = G.lists + (((size_t)unit * G.nsplit_max + split) * NC + h) * KP;
#pragma unroll
    for (int e = 0; e < KE; ++e) dst[e * 32 + lane] = (e * 32 + lane < kk) ? a[e] : 0ull;
  }
  if (!finish_split(G.counters + unit, nsplit, misc)) return;

  // ---------------- tail: this CTA finished the column block last ----------
  select_tail<BF16, D, NC, KE, kWarps>(G, unit, nsplit, b, kvh, cols, qd, wbuf, ring,
                                       G.stages * S::TILEB);
}

// ================================================ excluded-mass pass ========
//
// Second sweep over keys 0..p: dense-softmax normaliser Z and the part Zx of
// it that falls outside C_i (membership: anchor, window, or key >= the k-th
// selected key saved by the select kernel).  excl = Zx / Z.
struct Online3 {
  float m, z, x;
};

__device__ __forceinline__ Online3 online3_merge(Online3 a, Online3 b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f, 0.f};
  const float fa = a.m == -INFINITY ? 0.f : expf(a.m - m);
  const float fb = b.m == -INFINITY ? 0.f : expf(b.m - m);
  return {m, a.z * fa + b.z * fb, a.x * fa + b.x * fb};
}

__device__ __forceinline__ void online3_add(Online3& s, float l, bool excluded) {
  if (l > s.m) {
    const float f = s.m == -INFINITY ? 0.f : expf(s.m - l);
    s.z = s.z * f + 1.f;
    s.x = s.x * f + (excluded ? 1.f : 0.f);
    s.m = l;
  } else {
    const float w = expf(l - s.m);
    s.z += w;
    if (excluded) s.x += w;
  }
}

template <bool BF16, int D, int NC>
__global__ void __launch_bounds__(kThreads, 1)
    topo_excl_kernel(const __grid_constant__ CUtensorMap map_k, const Geom G) {
  using S = Shape<BF16, D>;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const long long cb = blockIdx.x / G.nsplit_max;
  const int split = (int)(blockIdx.x % G.nsplit_max);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const long long last_col = ((cb + 1) * NC < G.ncols ? (cb + 1) * NC : G.ncols) - 1;
  const long long pos_max = G.n - G.nq + last_col / G.g;
  const long long nkeys = pos_max + 1;
  const int nsplit = (int)((nkeys + G.L - 1) / G.L);
  if (split >= nsplit) return;
  const long long ks = (long long)split * G.L;
  const long long ke = (ks + G.L - 1 < pos_max) ? ks + G.L - 1 : pos_max;
  const int ntiles = (int)((ke - ks + kTile) / kTile);
  const long long unit = ((long long)b * G.Hkv + kvh) * G.ncb + cb;

  uint8_t* sm = aligned_smem_base();
  const Smem L(S::TILEB, G.stages, D, NC, kWarps * NC * 16);
  uint8_t* ring = sm + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + G.stages;
  float2* qd = reinterpret_cast<float2*>(sm + L.qd);
  Online3* red = reinterpret_cast<Online3*>(sm + L.buf);  // [warp][NC]
  ColInfo* cols = reinterpret_cast<ColInfo*>(sm + L.cols);
  volatile int* misc = reinterpret_cast<volatile int*>(sm + L.misc);

  init_pipeline(G.stages, full, empty, misc);
  load_columns<BF16, D, NC>(G, b, kvh, cb, cols, qd);
  __syncthreads();

  const long long row0 = ((long long)b * G.Hkv + kvh) * G.kv_stride + ks;
  int issued = 0;
  Online3 st[NC];
#pragma unroll
  for (int h = 0; h < NC; ++h) st[h] = {-INFINITY, 0.f, 0.f};
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      prefetch_tmap(&map_k);
      issued = produce_tiles<BF16, D>(&map_k, nullptr, row0, ntiles, G.stages, ring, full, empty,
                                      misc, G.status);
      drain_tiles(issued, G.stages, full, G.status);
    }
  } else {
    uint64_t thr[NC];
    long long lim[NC], wlo[NC];
#pragma unroll
    for (int h = 0; h < NC; ++h) {
      thr[h] = G.thr[(size_t)unit * NC + h];
      const long long p = cols[h].active ? cols[h].pos : -1;
      lim[h] = p < ke ? p : ke;
      wlo[h] = p - G.W + 1;
    }
    consume_tiles(warp, G.ncw, ntiles, G.stages, S::TILEB, ring, full, empty, misc, G.status,
                  [&](int t, const uint8_t* tile) {
                    float2 acc[NC];
                    score_tile<BF16, D, NC>(tile, qd, lane, acc);
                    const long long jA = ks + (long long)t * kTile + lane, jB = jA + 32;
#pragma unroll
                    for (int h = 0; h < NC; ++h) {
                      if (jA <= lim[h]) {
                        const bool in = jA == 0 || jA >= wlo[h] ||
                                        rank_key(acc[h].x, (uint32_t)jA) >= thr[h];
                        online3_add(st[h], G.scale * acc[h].x, !in);
                      }
                      if (jB <= lim[h]) {
                        const bool in = jB >= wlo[h] || rank_key(acc[h].y, (uint32_t)jB) >= thr[h];
                        online3_add(st[h], G.scale * acc[h].y, !in);
                      }
                    }
                  });
  }
  // warp reduction, then across warps
#pragma unroll
  for (int h = 0; h < NC; ++h) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Online3 other;
      other.m = __shfl_xor_sync(kFull, st[h].m, o);
      other.z = __shfl_xor_sync(kFull, st[h].z, o);
      other.x = __shfl_xor_sync(kFull, st[h].x, o);
      st[h] = online3_merge(st[h], other);
    }
    if (lane == 0) red[warp * NC + h] = st[h];
  }
  __syncthreads();
  if (tid < NC) {
    Online3 a = red[tid];
    for (int w = 1; w < kWarps; ++w) a = online3_merge(a, red[w * NC + tid]);
    float* dst = G.partials + (((size_t)unit * G.nsplit_max + split) * NC + tid) * 4;
    dst[0] = a.m;
    dst[1] = a.z;
    dst[2] = a.x;
  }
  if (!finish_split(G.counters + unit, nsplit, misc)) return;
  if (tid < NC && cols[tid].active) {
    Online3 a = {-INFINITY, 0.f, 0.f};
    for (int s = 0; s < nsplit; ++s) {
      const float* src = G.partials + (((size_t)unit * G.nsplit_max + s) * NC + tid) * 4;
      a = online3_merge(a, Online3{__ldcg(src), __ldcg(src + 1), __ldcg(src + 2)});
    }
    G.excl[cols[tid].row] = a.z > 0.f ? a.x / a.z : 0.f;
  }
}

// ==================================================== dense attention =======
//
// Split-n flash-decode style dense causal attention over keys 0..p: each
// stage holds a K tile and the V tile behind it; per column an online
// softmax (m, l) and a float32 accumulator over d (lanes own d/32 outputs).
template <bool BF16, int D, int NC>
__global__ void __launch_bounds__(kThreads, 1)
    dense_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                 const Geom G) {
  using S = Shape<BF16, D>;
  constexpr int EPL = S::EPL;
  constexpr int PART = D + 2;  // m, l, acc[D]
  const int b = blockIdx.z, kvh = blockIdx.y;
  const long long cb = blockIdx.x / G.nsplit_max;
  const int split = (int)(blockIdx.x % G.nsplit_max);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const long long last_col = ((cb + 1) * NC < G.ncols ? (cb + 1) * NC : G.ncols) - 1;
  const long long pos_max = G.n - G.nq + last_col / G.g;
  const long long nkeys = pos_max + 1;
  const int nsplit = (int)((nkeys + G.L - 1) / G.L);
  if (split >= nsplit) return;
  const long long ks = (long long)split * G.L;
  const long long ke = (ks + G.L - 1 < pos_max) ? ks + G.L - 1 : pos_max;
  const int ntiles = (int)((ke - ks + kTile) / kTile);
  const long long unit = ((long long)b * G.Hkv + kvh) * G.ncb + cb;

  uint8_t* sm = aligned_smem_base();
  const Smem L(2 * S::TILEB, G.stages, D, NC, kConsumerWarps * kTile * NC * 4);
  uint8_t* ring = sm + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + G.stages;
  float2* qd = reinterpret_cast<float2*>(sm + L.qd);
  float* pbuf_all = reinterpret_cast<float*>(sm + L.buf);  // [warp][kTile][NC]
  ColInfo* cols = reinterpret_cast<ColInfo*>(sm + L.cols);
  volatile int* misc = reinterpret_cast<volatile int*>(sm + L.misc);

  init_pipeline(G.stages, full, empty, misc);
  load_columns<BF16, D, NC>(G, b, kvh, cb, cols, qd);
  __syncthreads();

  const long long row0 = ((long long)b * G.Hkv + kvh) * G.kv_stride + ks;
  int issued = 0;
  static_assert(EPL % 2 == 0, "element pairs per lane");
  // acc[h][i]: this lane's output elements 2i, 2i+1 of column h (paired FMAs)
  float m[NC], l[NC];
  float2 acc[NC][EPL / 2];
#pragma unroll
  for (int h = 0; h < NC; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
  }
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      prefetch_tmap(&map_k);
      prefetch_tmap(&map_v);
      issued = produce_tiles<BF16, D>(&map_k, &map_v, row0, ntiles, G.stages, ring, full, empty,
                                      misc, G.status);
      drain_tiles(issued, G.stages, full, G.status);
    }
  } else {
    float* pbuf = pbuf_all + warp * kTile * NC;
    long long lim[NC];
#pragma unroll
    for (int h = 0; h < NC; ++h) {
      const long long p = cols[h].active ? cols[h].pos : -1;
      lim[h] = p < ke ? p : ke;
    }
    consume_tiles(warp, G.ncw, ntiles, G.stages, 2 * S::TILEB, ring, full, empty, misc, G.status,
                  [&](int t, const uint8_t* stage) {
                    float2 sc[NC];
                    score_tile<BF16, D, NC>(stage, qd, lane, sc);
                    const long long t0 = ks + (long long)t * kTile;
                    const long long jA = t0 + lane, jB = jA + 32;
#pragma unroll
                    for (int h = 0; h < NC; ++h) {
                      const float lA = jA <= lim[h] ? G.scale * sc[h].x : -INFINITY;
                      const float lB = jB <= lim[h] ? G.scale * sc[h].y : -INFINITY;
                      const float mnew = fmaxf(m[h], warp_max(fmaxf(lA, lB)));
                      float pA = 0.f, pB = 0.f, alpha = 1.f;
                      if (mnew != -INFINITY) {
                        alpha = m[h] == -INFINITY ? 0.f : expf(m[h] - mnew);
                        pA = lA == -INFINITY ? 0.f : expf(lA - mnew);
                        pB = lB == -INFINITY ? 0.f : expf(lB - mnew);
                      }
                      l[h] = l[h] * alpha + warp_sum(pA + pB);
#pragma unroll
                      for (int e = 0; e < EPL / 2; ++e) {
                        acc[h][e].x *= alpha;
                        acc[h][e].y *= alpha;
                      }
                      m[h] = mnew;
                      pbuf[lane * NC + h] = pA;
                      pbuf[(lane + 32) * NC + h] = pB;
                    }
                    __syncwarp();
                    const int nrows = (int)(ke - t0 + 1 < kTile ? ke - t0 + 1 : kTile);
                    const uint8_t* vt = stage + S::TILEB;
#pragma unroll 2
                    for (int r = 0; r < nrows; ++r) {
                      float v[EPL];
                      lane_elems<BF16, D>(vt + tile_lane_offset<BF16, D>(r, lane), v);
                      float pr[NC];
                      if constexpr (NC % 4 == 0) {
#pragma unroll
                        for (int h = 0; h < NC; h += 4) {
                          const float4 p4 = *reinterpret_cast<const float4*>(pbuf + r * NC + h);
                          pr[h] = p4.x;
                          pr[h + 1] = p4.y;
                          pr[h + 2] = p4.z;
                          pr[h + 3] = p4.w;
                        }
                      } else {
#pragma unroll
                        for (int h = 0; h < NC; ++h) pr[h] = pbuf[r * NC + h];
                      }
#pragma unroll
                      for (int h = 0; h < NC; ++h)
#pragma unroll
                        for (int e = 0; e < EPL / 2; ++e)
                          acc[h][e] = __ffma2_rn(make_float2(pr[h], pr[h]),
                                                 make_float2(v[2 * e], v[2 * e + 1]), acc[h][e]);
                    }
                  });
  }
  __syncthreads();
  // combine the consumer warps in shared memory (ring is free), publish
  float* red = reinterpret_cast<float*>(ring);  // [warp][NC][PART]
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int h = 0; h < NC; ++h) {
      float* r = red + ((size_t)warp * NC + h) * PART;
      if (lane == 0) {
        r[0] = m[h];
        r[1] = l[h];
      }
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) {
        r[2 + lane * EPL + 2 * e] = acc[h][e].x;
        r[2 + lane * EPL + 2 * e + 1] = acc[h][e].y;
      }
    }
  }
  __syncthreads();
  for (int h = warp; h < NC; h += kWarps) {
    float mm = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w) mm = fmaxf(mm, red[((size_t)w * NC + h) * PART]);
    float ll = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    if (mm != -INFINITY) {
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* r = red + ((size_t)w * NC + h) * PART;
        const float f = r[0] == -INFINITY ? 0.f : expf(r[0] - mm);
        ll += r[1] * f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] += r[2 + lane * EPL + e] * f;
      }
    }
    float* dst = G.partials + (((size_t)unit * G.nsplit_max + split) * NC + h) * PART;
    if (lane == 0) {
      dst[0] = mm;
      dst[1] = ll;
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[2 + lane * EPL + e] = o[e];
  }
  if (!finish_split(G.counters + unit, nsplit, misc)) return;
  for (int h = warp; h < NC; h += kWarps) {
    if (!cols[h].active) continue;
    float mm = -INFINITY;
    for (int s = 0; s < nsplit; ++s)
      mm = fmaxf(mm, __ldcg(G.partials + (((size_t)unit * G.nsplit_max + s) * NC + h) * PART));
    float ll = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float* r = G.partials + (((size_t)unit * G.nsplit_max + s) * NC + h) * PART;
      const float rm = __ldcg(r);
      const float f = rm == -INFINITY ? 0.f : expf(rm - mm);
      ll += __ldcg(r + 1) * f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[e] += __ldcg(r + 2 + lane * EPL + e) * f;
    }
    float* outp = G.out + cols[h].row * D;
#pragma unroll
    for (int e = 0; e < EPL; ++e) outp[lane * EPL + e] = ll > 0.f ? o[e] / ll : 0.f;
  }
}

// ============================================ softmax over given sets =======
//
// One warp per query row: out = softmax over the listed positions.
template <bool BF16, int D>
__global__ void __launch_bounds__(128) sparse_pv_kernel(const Geom G) {
  __shared__ float2 qs[4][D];
  __shared__ float wsm[4][256];
  __shared__ int jsm[4][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + warp;
  const long long nrows = (long long)G.B * G.Hq * G.nq;
  if (row >= nrows) return;
  const long long r = row % G.nq;
  const int h = (int)((row / G.nq) % G.Hq);
  const int b = (int)(row / (G.nq * G.Hq));
  const int kvh = h / G.g;
  const long long p = G.n - G.nq + r;
  for (int c = lane; c < D; c += 32) {
    const float x = load_elem<BF16>(G.qp, row * D + c);
    qs[warp][c] = make_float2(x, x);
  }
  __syncwarp();
  const long long cmax = 1 + (long long)G.W + G.topk;
  const int* irow = G.idx + row * cmax;
  auto entry = [&](long long e) -> long long {
    const int j = irow[e];
    return (j >= 0 && j <= p) ? j : -1;
  };
  warp_softmax_pv<BF16, D, 1>(G, b, kvh, qs[warp], 0, cmax, entry, wsm[warp], jsm[warp],
                              row * D, lane);
}

// ================================================ condensate KV compaction ==
//
// out[row][e] = rows idx[row][e] of K and V of the row's KV head (zero rows
// for entries outside 0..n-1).  One warp per (row, entry group of 8): a lane
// moves 16 bytes of each row.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) compact_kv_kernel(const Geom G, void* k_out, void* v_out) {
  using S = Shape<BF16, D>;
  constexpr int VPR = S::ROWB / 16;  // 16-byte vectors per row
  const long long cmax = 1 + (long long)G.W + G.topk;
  const long long nrows = (long long)G.B * G.Hq * G.nq;
  const long long total = nrows * cmax * VPR;
  const uint4* kin = reinterpret_cast<const uint4*>(G.kp);
  const uint4* vin = reinterpret_cast<const uint4*>(G.vp);
  uint4* ko = reinterpret_cast<uint4*>(k_out);
  uint4* vo = reinterpret_cast<uint4*>(v_out);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long ent = i / VPR;  // (row, entry)
    const int vv = (int)(i % VPR);
    const long long row = ent / cmax;
    const int h = (int)((row / G.nq) % G.Hq);
    const int b = (int)(row / (G.nq * G.Hq));
    const int j = G.idx[ent];
    uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
    if (j >= 0 && j < G.n) {
      const long long src = (((long long)b * G.Hkv + h / G.g) * G.kv_stride + j) * VPR + vv;
      kx = __ldg(kin + src);
      vx = __ldg(vin + src);
    }
    ko[i] = kx;
    vo[i] = vx;
  }
}

}  // namespace topo
