// topo_api.cu -- the C ABI of libtopoattn.so (declared in include/topo_attn.h):
// argument checks, launch planning, workspace layout, TMA descriptors and
// kernel dispatch.  No allocation, no synchronisation (except the explicit
// status read-back).  Global state: lazily resolved driver entry points,
// per-kernel attribute set-up and a small mutex-guarded cache of launch plans
// (a plan depends only on the parameters and the device).  Each call clears
// the split counters it uses (one cudaMemsetAsync on the caller's stream), so
// a workspace may be shared by calls of any shapes, in stream order.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "topo_attn.h"
#include "topo_launch.cuh"

namespace {

using topo::Geom;
using topo::kTile;

constexpr long long kMaxRows = (1LL << 31) - 2 * kTile;  // TMA row coordinate is int32

struct Plan {
  bool bf16 = false;
  bool tc = false;  // tensor-core select kernel (bf16, <= 8 columns per KV head, 1 <= k <= 64)
  bool pf = false;  // tensor-core chunked-prefill path (bf16, > 8 columns per KV head, k <= 32)
  bool dtc = false;  // tensor-core dense kernel (bf16, <= 8 columns per KV head)
  int pf_stages = 0, pf_smem = 0, pf_items_per_head = 0, pf_grid = 0, pf_kmax_grid = 1;
  long long pf_nitems = 0;
  int D = 0, NC = 1, KE = 1, KP = 32;
  long long ncols = 0, ncb = 0, units = 0;
  // select (or dense) pass
  long long L = kTile, L2 = kTile, hi_units = 0;
  int nsplit = 1, stages = 2, ncw = 2, smem = 0;
  // excluded-mass pass
  long long Le = kTile;
  int nsplit_e = 1, stages_e = 2, ncw_e = 2, smem_e = 0;
  // its column blocks: the select pass's, except that 16 tensor-core columns
  // are two blocks of 8 (the saved k-th keys keep the layout unit * NC + h)
  int NCe = 1;
  long long ncbe = 1, units_e = 0;
  // workspace layout (bytes)
  size_t off_cnt = 0, off_cnt_e = 0, off_kmax = 0, off_work = 0, off_zero_end = 0;
  size_t off_lists = 0, off_thr = 0, off_part = 0, off_surv = 0, off_scnt = 0, off_topk = 0;
  size_t off_topl = 0;
  size_t total = 0;
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline int pow2_at_least(long long x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

int check_params(const topo_attn_params* p) {
  if (!p) return TOPO_ERR_INVALID_ARG;
  if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0) return TOPO_ERR_INVALID_ARG;
  if (p->B > 65535 || p->Hkv > 65535) return TOPO_ERR_INVALID_ARG;
  if (p->n < 1 || p->nq < 1 || p->nq > p->n || p->kv_stride < p->n) return TOPO_ERR_INVALID_ARG;
  if (p->n > (1LL << 31) - 1) return TOPO_ERR_INVALID_ARG;
  if (p->W < 1 || p->k < 0) return TOPO_ERR_INVALID_ARG;
  if (!isfinite(p->scale)) return TOPO_ERR_INVALID_ARG;
  if (p->dtype != TOPO_F32 && p->dtype != TOPO_BF16) return TOPO_ERR_UNSUPPORTED;
  if (p->d != 64 && p->d != 128) return TOPO_ERR_UNSUPPORTED;
  if (p->k > TOPO_KMAX) return TOPO_ERR_UNSUPPORTED;
  if ((long long)p->B * p->Hkv * p->kv_stride > kMaxRows) return TOPO_ERR_UNSUPPORTED;
  return TOPO_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

// Keys per split: enough CTAs to fill every SM, chosen so that the last wave
// is as full as possible (all splits of a pass take about the same time).
long long choose_split(long long units, long long nkeys, int slots, long long tile = kTile) {
  if (nkeys <= tile) return tile;
  const long long smax = nkeys / (4 * tile) > 1 ? nkeys / (4 * tile) : 1;
  double best = -1.0;
  long long best_s = 1;
  for (long long s = 1; s <= smax && s <= 4096; ++s) {
    const long long total = units * s;
    const long long waves = ceil_div(total, slots);
    const double eff = (double)total / (double)(waves * slots);
    if (eff > best + 1e-9) {
      best = eff;
      best_s = s;
    }
    if (total >= 8LL * slots) break;
  }
  return ceil_div(ceil_div(nkeys, best_s), tile) * tile;
}

// Keys per split for the tensor-core select kernel: minimises the estimated
// time waves x (keys per split + fixed), where `fixed` is the per-CTA cost
// (set-up, exact rescoring and publishing) expressed in keys streamed.
long long choose_split_tc(long long units, long long nkeys, int slots, long long fixed) {
  const long long tile = topo::kTcTile;
  if (nkeys <= tile) return tile;
  double best = 1e300;
  long long best_l = ceil_div(nkeys, tile) * tile;
  for (long long s = 1; s <= 4096 && (s - 1) * tile < nkeys; ++s) {
    const long long l = ceil_div(ceil_div(nkeys, s), tile) * tile;
    const long long nsp = ceil_div(nkeys, l);
    const long long waves = ceil_div(units * nsp, slots);
    const double cost = (double)waves * (double)(l + fixed);
    if (cost < best - 1e-9) {
      best = cost;
      best_l = l;
    }
  }
  return best_l;
}

int stages_for(int stage_bytes, int fixed_bytes, int min_ring) {
  int st = (topo::kMaxSmem - fixed_bytes) / stage_bytes;
  if (st > 16) st = 16;
  while (st > 2 && st * stage_bytes > topo::kMaxSmem - fixed_bytes) --st;
  if (st * stage_bytes < min_ring) st = (min_ring + stage_bytes - 1) / stage_bytes;
  return st;
}

// Ring depth and consumer-warp count of the CUDA-core kernels: the consumer
// count may not exceed the depth (see consume_tiles for why).
void ring_shape(int stage_bytes, int fixed_bytes, int min_ring, int* stages, int* ncw) {
  *stages = stages_for(stage_bytes, fixed_bytes, min_ring);
  *ncw = *stages < topo::kConsumerWarps ? *stages : topo::kConsumerWarps;
}

// Shared memory that select_tail's staged softmax needs for one selection
// column of gsz columns (its layout: top-k positions and counts, the split
// lists, logits, the band, anchor and top-k rows, the slot table).  One
// selection column is one query row, so the band is W rows.
int tail_scratch_bytes(const topo_attn_params* p, const Plan& P, int gsz) {
  const long long NC = P.NC, KP = P.KP, kk = p->k;
  const long long mmax = 1 + (long long)p->W + kk;
  const long long slot = 2LL * P.D * 2 + 16;
  const long long v0 = (NC * KP * 4 + NC * 8 + 32 + 1023) & ~1023LL;
  const long long lists = (long long)P.nsplit * NC * KP * 8;
  const long long off_lw = (v0 + lists + 1023) & ~1023LL;
  const long long off_stage = (off_lw + NC * mmax * 4 + NC * 4 + 1023) & ~1023LL;
  const long long nslots = (long long)p->W + 1 + gsz * kk;
  const long long need = off_stage + nslots * slot + NC * mmax * 4;
  return need > (1LL << 30) ? (1 << 30) : (int)need;
}

// Plan for the condensate-set passes (dense=false) or the dense pass.  A
// paged cache scans from key 0 (block-aligned tiles), one more key per
// split range.
int make_plan(const topo_attn_params* p, bool dense, Plan* P, bool paged = false) {
  int rc = check_params(p);
  if (rc != TOPO_OK) return rc;
  P->bf16 = p->dtype == TOPO_BF16;
  P->D = p->d;
  const int g = p->Hq / p->Hkv;
  P->ncols = p->nq * g;
  P->NC = pow2_at_least(P->ncols) < 8 ? pow2_at_least(P->ncols) : 8;
  P->ncb = ceil_div(P->ncols, P->NC);
  P->units = (long long)p->B * p->Hkv * P->ncb;
  P->KP = pow2_at_least(p->k > 32 ? p->k : 32);
  P->KE = P->KP / 32;
  const int es = P->bf16 ? 2 : 4;
  const int tileb = kTile * P->D * es;
  const int slots = sm_count();
  const long long pos_max = p->n - 1;
  P->tc = !dense && P->bf16 && p->k >= 1 &&
          ((p->k <= 32 && P->ncols <= 16) || (p->k <= 64 && P->ncols <= 4));
  P->pf = !dense && P->bf16 && !P->tc && p->k >= 1 && p->k <= 32 && P->ncols > 8;
  if (P->tc) {
    // tensor-core scorer: all columns of a KV head in one block
    P->NC = (int)pow2_at_least(P->ncols);
    P->ncb = 1;
    P->units = (long long)p->B * p->Hkv;
  }
  if (!dense) {
    long long ncand = p->k > 0 ? pos_max - p->W : 0;
    if (paged && ncand > 0) ncand += 1;
    P->L = P->tc ? choose_split_tc(P->units, ncand > 0 ? ncand : 0, slots, 1200)
                 : choose_split(P->units, ncand > 0 ? ncand : 0, slots);
    P->nsplit = ncand > 0 ? (int)ceil_div(ncand, P->L) : 1;
    const int cap = topo::cap_for(P->KE);
    const topo::Smem base(0, 0, P->D, P->NC, topo::kConsumerWarps * P->NC * cap * 8);
    const int tail = P->NC * P->KP * 8 > P->NC * P->KP * 4 + topo::kWarps * 2048
                         ? P->NC * P->KP * 8
                         : P->NC * P->KP * 4 + topo::kWarps * 2048;
    ring_shape(tileb + 16, base.total, tail > 32768 ? tail : 32768, &P->stages, &P->ncw);
    P->smem = topo::Smem(tileb, P->stages, P->D, P->NC, topo::kConsumerWarps * P->NC * cap * 8).total;
    if (P->tc && P->units * 2 <= slots && ncand > (long long)slots * topo::kTcTile) {
      // one wave: every unit gets slots/units splits, the first slots%units one more
      const long long s_lo = slots / P->units;
      P->hi_units = slots - s_lo * P->units;
      P->L = ceil_div(ceil_div(ncand, s_lo), topo::kTcTile) * topo::kTcTile;
      P->L2 = ceil_div(ceil_div(ncand, s_lo + 1), topo::kTcTile) * topo::kTcTile;
      P->nsplit = (int)ceil_div(ncand, P->hi_units > 0 ? P->L2 : P->L);
    }
    if (P->tc) {
      const int tct = topo::kTcTile * P->D * 2;
      const int fixed = topo::TcSmem(tct, 0, P->D, P->NC, P->KE).total;
      int st = (topo::kMaxSmem - fixed) / (tct + 24);
      if (st > 8) st = 8;
      if (st < 2) return TOPO_ERR_UNSUPPORTED;
      // after the scan the ring holds every column's concatenated survivors
      // (one area per column with at most four columns, else one per epilogue warp)
      const long long areas = P->NC < topo::kTcEpiWarps ? P->NC : topo::kTcEpiWarps;
      if ((long long)st * tct < areas * topo::kTcEpiWarps * topo::tc_cap(P->KE) * 8)
        return TOPO_ERR_UNSUPPORTED;
      P->stages = st;
      P->smem = topo::TcSmem(tct, st, P->D, P->NC, P->KE).total;
    }
    if (P->pf) {
      const int tile = topo::kPfKeys * P->D * 2;
      const int fixed = topo::PfSmem(P->D, 0).total;
      int st = (topo::kMaxSmem - fixed) / (tile + 16);
      if (st > 8) st = 8;
      if (st < 2) return TOPO_ERR_UNSUPPORTED;
      P->pf_stages = st;
      P->pf_smem = topo::PfSmem(P->D, st).total;
      P->pf_items_per_head = (int)ceil_div(P->ncols, topo::kPfCols);
      P->pf_nitems = (long long)p->B * p->Hkv * P->pf_items_per_head;
      P->pf_grid = (int)(P->pf_nitems < slots ? P->pf_nitems : slots);
      const long long nvec = p->n * (P->D / 8);
      long long kg = ceil_div(nvec, 1024);
      P->pf_kmax_grid = (int)(kg < 1 ? 1 : (kg > 64 ? 64 : kg));
      if (P->pf_smem > topo::kMaxSmem) return TOPO_ERR_UNSUPPORTED;
    }
    // excluded-mass pass: keys 0..p
    P->NCe = P->NC > 8 ? 8 : P->NC;
    P->ncbe = P->NC > 8 ? ceil_div(P->ncols, 8) : P->ncb;
    P->units_e = (long long)p->B * p->Hkv * P->ncbe;
    P->Le = choose_split(P->units_e, pos_max + 1, slots);
    P->nsplit_e = (int)ceil_div(pos_max + 1, P->Le);
    const topo::Smem base_e(0, 0, P->D, P->NCe, topo::kWarps * P->NCe * 16);
    ring_shape(tileb + 16, base_e.total, 32768, &P->stages_e, &P->ncw_e);
    P->smem_e = topo::Smem(tileb, P->stages_e, P->D, P->NCe, topo::kWarps * P->NCe * 16).total;
  } else if (P->bf16 && P->ncols <= 8) {
    // tensor-core dense kernel: all columns of a KV head in one block
    const int stageb = 2 * topo::kTcTile * P->D * 2;
    const int fixed = topo::DenseTcSmem(stageb, 0, P->D, P->NC).total;
    int st = (topo::kMaxSmem - fixed) / (stageb + 24);
    if (st > 8) st = 8;
    if (st < 2 || (long long)st * stageb < (long long)topo::kTcEpiWarps * P->NC * (P->D + 2) * 4)
      return TOPO_ERR_UNSUPPORTED;
    P->dtc = true;
    P->stages = st;
    P->smem = topo::DenseTcSmem(stageb, st, P->D, P->NC).total;
    P->L = choose_split(P->units, pos_max + 1, slots, topo::kTcTile);
    P->nsplit = (int)ceil_div(pos_max + 1, P->L);
  } else {
    const int pbuf = topo::kConsumerWarps * kTile * P->NC * 4;
    const topo::Smem base(0, 0, P->D, P->NC, pbuf);
    const int red = topo::kConsumerWarps * P->NC * (P->D + 2) * 4;
    ring_shape(2 * tileb + 16, base.total, red > 32768 ? red : 32768, &P->stages, &P->ncw);
    P->L = choose_split(P->units, pos_max + 1, slots);
    P->nsplit = (int)ceil_div(pos_max + 1, P->L);
    P->smem = topo::Smem(2 * tileb, P->stages, P->D, P->NC, pbuf).total;
  }
  if (P->smem > topo::kMaxSmem || P->smem_e > topo::kMaxSmem) return TOPO_ERR_UNSUPPORTED;
  if (P->ncb * P->nsplit > 0x7fffffffLL || P->ncbe * P->nsplit_e > 0x7fffffffLL)
    return TOPO_ERR_UNSUPPORTED;
  // workspace: status word, counters, then per-pass buffers
  size_t o = 256;
  P->off_cnt = o;
  o = align256(o + (size_t)P->units * 4);
  P->off_cnt_e = o;
  o = align256(o + (size_t)(P->units_e > P->units ? P->units_e : P->units) * 4);
  P->off_kmax = o;
  o = align256(o + (size_t)p->B * p->Hkv * 4);
  P->off_work = o;
  o = align256(o + 4);
  P->off_zero_end = o;  // everything before this is cleared on every call
  if (!dense) {
    P->off_lists = o;
    if (!P->pf) o = align256(o + (size_t)P->units * P->nsplit * P->NC * P->KP * 8);
    P->off_thr = o;
    o = align256(o + (size_t)P->units * P->NC * 8);
    P->off_part = o;
    o = align256(o + (size_t)P->units_e * P->nsplit_e * P->NCe * 16);
    if (P->pf) {
      const size_t ncolumns = (size_t)p->B * p->Hkv * P->ncols;
      P->off_surv = o;
      o = align256(o + ncolumns * topo::kPfLL * 8);
      P->off_scnt = o;
      o = align256(o + ncolumns * 4);
      P->off_topk = o;
      o = align256(o + ncolumns * p->k * 4);
      P->off_topl = o;
      o = align256(o + ncolumns * p->k * 4);
    }
  } else {
    P->off_part = o;
    o = align256(o + (size_t)P->units * P->nsplit * P->NC * (P->D + 2) * 4);
  }
  P->total = o;
  return TOPO_OK;
}

// make_plan, memoised: the last kPlanCache distinct (parameters, pass, device)
// triples (the split search costs tens of microseconds for long caches).
constexpr int kPlanCache = 32;
struct PlanEntry {
  topo_attn_params p;
  int dense, paged, dev, rc, valid;
  Plan plan;
};
std::mutex g_plan_mu;
PlanEntry g_plans[kPlanCache];
int g_plan_next = 0;

bool same_params(const topo_attn_params& a, const topo_attn_params& b) {
  return a.B == b.B && a.Hq == b.Hq && a.Hkv == b.Hkv && a.d == b.d && a.n == b.n &&
         a.nq == b.nq && a.kv_stride == b.kv_stride && a.W == b.W && a.k == b.k &&
         memcmp(&a.scale, &b.scale, sizeof a.scale) == 0 && a.dtype == b.dtype;
}

int make_plan_cached(const topo_attn_params* p, bool dense, Plan* P, bool paged = false) {
  if (!p) return TOPO_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (int i = 0; i < kPlanCache; ++i) {
      const PlanEntry& e = g_plans[i];
      if (e.valid && e.dense == (int)dense && e.paged == (int)paged && e.dev == dev &&
          same_params(e.p, *p)) {
        *P = e.plan;
        return e.rc;
      }
    }
  }
  const int rc = make_plan(p, dense, P, paged);
  std::lock_guard<std::mutex> lock(g_plan_mu);
  PlanEntry& e = g_plans[g_plan_next];
  g_plan_next = (g_plan_next + 1) % kPlanCache;
  e.p = *p;
  e.dense = (int)dense;
  e.paged = (int)paged;
  e.dev = dev;
  e.rc = rc;
  e.plan = *P;
  e.valid = 1;
  return rc;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 2-D map over the rows of k or v ([B*Hkv*kv_stride, d], or `nrows` rows of
// a paged pool); box = 128 bytes of one row x box_rows rows, 128-byte swizzle.
int make_map(CUtensorMap* map, const void* base, const topo_attn_params* p,
             int box_rows = kTile, long long nrows = 0) {
  auto fn = encode_fn();
  if (!fn) return TOPO_ERR_CUDA;
  const bool bf16 = p->dtype == TOPO_BF16;
  const int es = bf16 ? 2 : 4;
  const cuuint64_t rows = nrows > 0 ? (cuuint64_t)nrows : (cuuint64_t)p->B * p->Hkv * p->kv_stride;
  const cuuint64_t dims[2] = {(cuuint64_t)p->d, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)p->d * es};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TOPO_OK : TOPO_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

Geom base_geom(const topo_attn_params* p, const Plan& P) {
  Geom G;
  memset(&G, 0, sizeof G);
  G.B = p->B;
  G.Hq = p->Hq;
  G.Hkv = p->Hkv;
  G.g = p->Hq / p->Hkv;
  G.n = p->n;
  G.nq = p->nq;
  G.kv_stride = p->kv_stride;
  G.W = p->W;
  G.topk = p->k;
  G.scale = p->scale;
  G.ncols = P.ncols;
  G.ncb = P.ncb;
  return G;
}

// The parameters of one layer of a multi-layer step: the shared shapes of
// `p` with the layer's own window and top-k (a pillar layer ignores both).
topo_attn_params layer_params(const topo_attn_params* p, const topo_layer& l) {
  topo_attn_params q = *p;
  q.W = l.dense ? 1 : l.W;
  q.k = l.dense ? 0 : l.k_top;
  return q;
}

int to_status(cudaError_t e) {
  if (e == cudaSuccess) return TOPO_OK;
  return TOPO_ERR_CUDA;
}

template <class F>
int dispatch(bool bf16, int D, F&& f) {
  if (bf16) {
    if (D == 128) return to_status(f(topo::Launcher<true, 128>()));
    return to_status(f(topo::Launcher<true, 64>()));
  }
  if (D == 128) return to_status(f(topo::Launcher<false, 128>()));
  return to_status(f(topo::Launcher<false, 64>()));
}

// The select pass (and, with excl, the excluded-mass pass).  `group`: one
// condensate set per (sequence, KV head, row) shared by the KV head's query
// heads (tensor-core decode shapes only; no excluded mass).
int run_topo(const topo_attn_params* p, const void* q, const void* k, const void* v, float* out,
             int32_t* idx, float* excl, void* ws, size_t ws_bytes, cudaStream_t st,
             bool group = false, const topo_paged_kv* paged = nullptr) {
  const bool pool = paged && paged->block_table;
  Plan P;
  int rc = make_plan_cached(p, false, &P, pool);
  if (rc != TOPO_OK) return rc;
  if (group && (!P.tc || p->Hq / p->Hkv < 2 || excl)) return TOPO_ERR_UNSUPPORTED;
  if (paged && (!P.tc || excl)) return TOPO_ERR_UNSUPPORTED;
  if (!q || !k) return TOPO_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || (v && !aligned16(v))) return TOPO_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < P.total)
    return TOPO_ERR_WORKSPACE;
  const long long pool_rows =
      pool ? (long long)paged->num_blocks * p->Hkv * paged->block_size : 0;
  CUtensorMap mk;
  rc = make_map(&mk, k, p, kTile, pool_rows);
  if (rc != TOPO_OK) return rc;
  uint8_t* w = static_cast<uint8_t*>(ws);
  Geom G = base_geom(p, P);
  if (paged) {
    G.block_table = paged->block_table;
    G.seq_lens = paged->seq_lens;
    G.max_blocks = paged->max_blocks;
    G.block_size = paged->block_size;
    G.num_blocks = paged->num_blocks;
    G.out_bf16 = paged->out_bf16 ? 1 : 0;
  }
  G.qp = q;
  G.kp = k;
  G.vp = v;
  G.out = out;
  G.idx = idx;
  G.excl = excl;
  G.status = reinterpret_cast<int*>(w);
  G.counters = reinterpret_cast<int*>(w + P.off_cnt);
  G.lists = reinterpret_cast<unsigned long long*>(w + P.off_lists);
  G.thr = reinterpret_cast<unsigned long long*>(w + P.off_thr);
  G.partials = reinterpret_cast<float*>(w + P.off_part);
  G.L = P.L;
  G.L2 = P.L2;
  G.hi_units = P.hi_units;
  G.nsplit_max = P.nsplit;
  G.stages = P.stages;
  G.ncw = P.ncw;
  G.flags = (out ? topo::kDoPV : 0) | (idx ? topo::kDoIdx : 0) | (excl ? topo::kSaveThr : 0);
  // split counters, K scales and the work counter start at zero on every call
  rc = to_status(cudaMemsetAsync(w + P.off_cnt, 0, P.off_zero_end - P.off_cnt, st));
  if (rc != TOPO_OK) return rc;
  const dim3 grid((unsigned)(P.ncb * P.nsplit), (unsigned)p->Hkv, (unsigned)p->B);
  if (P.pf) {
    CUtensorMap mk128;
    rc = make_map(&mk128, k, p, topo::kPfKeys);
    if (rc != TOPO_OK) return rc;
    G.kmax = reinterpret_cast<unsigned*>(w + P.off_kmax);
    G.work = reinterpret_cast<int*>(w + P.off_work);
    G.surv = reinterpret_cast<float2*>(w + P.off_surv);
    G.surv_cnt = reinterpret_cast<int*>(w + P.off_scnt);
    G.topsel = reinterpret_cast<int*>(w + P.off_topk);
    G.toplogit = out ? reinterpret_cast<float*>(w + P.off_topl) : nullptr;  // softmax logits
    G.nitems = P.pf_nitems;
    G.items_per_head = P.pf_items_per_head;
    G.thr_nc = P.NC;
    G.stages = P.pf_stages;
    if (!excl) G.thr = nullptr;
    rc = dispatch(P.bf16, P.D, [&](auto L) {
      return L.prefill(mk128, G, P.pf_grid, P.pf_smem, P.pf_kmax_grid, out != nullptr, st);
    });
    G.stages = P.stages;
    G.thr = reinterpret_cast<unsigned long long*>(w + P.off_thr);
  } else if (P.tc) {
    CUtensorMap mk128;
    rc = make_map(&mk128, k, p, topo::kTcTile, pool_rows);
    if (rc != TOPO_OK) return rc;
    // the tail as a dependent kernel, one CTA per selection column, when its
    // staged softmax fits in one CTA's shared memory
    const int gsz = group ? p->Hq / p->Hkv : 1;
    const int tail_scratch = tail_scratch_bytes(p, P, gsz);
    const int tail_smem =
        topo::TailSmem(tail_scratch, P.D, P.NC, P.KP).total;
    const bool split_tail = tail_smem <= topo::kMaxSmem;
    if (split_tail) G.flags |= topo::kSplitTail;
    // one wave of select CTAs: the tail's band staging may overlap its end
    if (split_tail && (P.hi_units > 0 || P.units * P.nsplit <= sm_count()))
      G.flags |= topo::kEarlyBand;
    rc = dispatch(P.bf16, P.D, [&](auto L) {
      return L.select_tc(P.NC, P.KE, group, mk128, G, grid, P.smem, st);
    });
    if (rc == TOPO_OK && split_tail) {
      const dim3 tgrid((unsigned)(P.ncols / gsz), (unsigned)p->Hkv, (unsigned)p->B);
      rc = dispatch(P.bf16, P.D, [&](auto L) {
        return L.tail_tc(P.NC, P.KE, group, G, tgrid, tail_smem, tail_scratch, st);
      });
    }
  } else {
    rc = dispatch(P.bf16, P.D,
                  [&](auto L) { return L.select(P.NC, P.KE, mk, G, grid, P.smem, st); });
  }
  if (rc != TOPO_OK || !excl) return rc;
  Geom E = G;
  E.counters = reinterpret_cast<int*>(w + P.off_cnt_e);
  E.L = P.Le;
  E.nsplit_max = P.nsplit_e;
  E.stages = P.stages_e;
  E.ncw = P.ncw_e;
  E.ncb = P.ncbe;
  const dim3 grid_e((unsigned)(P.ncbe * P.nsplit_e), (unsigned)p->Hkv, (unsigned)p->B);
  return dispatch(P.bf16, P.D, [&](auto L) { return L.excl(P.NCe, mk, E, grid_e, P.smem_e, st); });
}

}  // namespace

extern "C" {

size_t topo_attn_workspace_size(const topo_attn_params* p) {
  Plan P;
  return make_plan_cached(p, false, &P) == TOPO_OK ? P.total : 0;
}

size_t dense_attn_workspace_size(const topo_attn_params* p) {
  Plan P;
  return make_plan_cached(p, true, &P) == TOPO_OK ? P.total : 0;
}

int topo_attn_workspace_init(void* ws, size_t bytes, topo_stream_t stream) {
  if (!ws) return TOPO_ERR_INVALID_ARG;
  return to_status(cudaMemsetAsync(ws, 0, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int topo_attn_forward(const topo_attn_params* p, const void* q, const void* k, const void* v,
                      float* out, int32_t* idx, float* excl, void* ws, size_t ws_bytes,
                      topo_stream_t stream) {
  if (!out || !v) return TOPO_ERR_INVALID_ARG;
  return run_topo(p, q, k, v, out, idx, excl, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t topo_attn_paged_workspace_size(const topo_attn_params* p, const topo_paged_kv* kv) {
  Plan P;
  return make_plan_cached(p, false, &P, kv && kv->block_table) == TOPO_OK ? P.total : 0;
}

int topo_attn_forward_paged(const topo_attn_params* p, const topo_paged_kv* kv, const void* q,
                            const void* k_pool, const void* v_pool, void* out, int32_t* idx,
                            void* ws, size_t ws_bytes, topo_stream_t stream) {
  if (!kv || !out || !v_pool) return TOPO_ERR_INVALID_ARG;
  const int rc = check_params(p);
  if (rc != TOPO_OK) return rc;
  if (kv->block_table) {
    if (kv->block_size < topo::kTcTile || kv->block_size % topo::kTcTile || kv->num_blocks < 1 ||
        kv->max_blocks < 1 || (long long)kv->max_blocks * kv->block_size < p->n)
      return TOPO_ERR_INVALID_ARG;
    if ((long long)kv->num_blocks * p->Hkv * kv->block_size > kMaxRows)
      return TOPO_ERR_UNSUPPORTED;
  }
  return run_topo(p, q, k_pool, v_pool, static_cast<float*>(out), idx, nullptr, ws, ws_bytes,
                  reinterpret_cast<cudaStream_t>(stream), false, kv);
}

int topo_attn_forward_grouped(const topo_attn_params* p, const void* q, const void* k,
                              const void* v, float* out, int32_t* idx, void* ws, size_t ws_bytes,
                              topo_stream_t stream) {
  if (!out || !v) return TOPO_ERR_INVALID_ARG;
  return run_topo(p, q, k, v, out, idx, nullptr, ws, ws_bytes,
                  reinterpret_cast<cudaStream_t>(stream), true);
}

int topo_attn_score_select(const topo_attn_params* p, const void* q, const void* k, int32_t* idx,
                           void* ws, size_t ws_bytes, topo_stream_t stream) {
  if (!idx) return TOPO_ERR_INVALID_ARG;
  return run_topo(p, q, k, nullptr, nullptr, idx, nullptr, ws, ws_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

int topo_attn_sparse_softmax_pv(const topo_attn_params* p, const void* q, const void* k,
                                const void* v, const int32_t* idx, float* out,
                                topo_stream_t stream) {
  const int rc = check_params(p);
  if (rc != TOPO_OK) return rc;
  if (!q || !k || !v || !idx || !out) return TOPO_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return TOPO_ERR_INVALID_ARG;
  Plan P;
  P.ncols = p->nq * (p->Hq / p->Hkv);
  P.ncb = 1;
  Geom G = base_geom(p, P);
  G.qp = q;
  G.kp = k;
  G.vp = v;
  G.out = out;
  G.idx = const_cast<int*>(idx);
  const long long nrows = (long long)p->B * p->Hq * p->nq;
  if ((nrows + 3) / 4 > 0x7fffffffLL) return TOPO_ERR_UNSUPPORTED;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return dispatch(p->dtype == TOPO_BF16, p->d, [&](auto L) { return L.pv(G, nrows, st); });
}

int topo_attn_compact_kv(const topo_attn_params* p, const void* k, const void* v,
                         const int32_t* idx, void* k_out, void* v_out, topo_stream_t stream) {
  const int rc = check_params(p);
  if (rc != TOPO_OK) return rc;
  if (!k || !v || !idx || !k_out || !v_out) return TOPO_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out))
    return TOPO_ERR_INVALID_ARG;
  Plan P;
  P.ncols = p->nq * (p->Hq / p->Hkv);
  P.ncb = 1;
  Geom G = base_geom(p, P);
  G.kp = k;
  G.vp = v;
  G.idx = const_cast<int32_t*>(idx);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return dispatch(p->dtype == TOPO_BF16, p->d,
                  [&](auto L) { return L.compact(G, k_out, v_out, st); });
}

int dense_attn_forward(const topo_attn_params* p, const void* q, const void* k, const void* v,
                       float* out, void* ws, size_t ws_bytes, topo_stream_t stream) {
  Plan P;
  int rc = make_plan_cached(p, true, &P);
  if (rc != TOPO_OK) return rc;
  if (!q || !k || !v || !out) return TOPO_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return TOPO_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < P.total)
    return TOPO_ERR_WORKSPACE;
  CUtensorMap mk, mv;
  const int box = P.dtc ? topo::kTcTile : kTile;
  rc = make_map(&mk, k, p, box);
  if (rc == TOPO_OK) rc = make_map(&mv, v, p, box);
  if (rc != TOPO_OK) return rc;
  uint8_t* w = static_cast<uint8_t*>(ws);
  Geom G = base_geom(p, P);
  G.qp = q;
  G.kp = k;
  G.vp = v;
  G.out = out;
  G.status = reinterpret_cast<int*>(w);
  G.counters = reinterpret_cast<int*>(w + P.off_cnt);
  G.partials = reinterpret_cast<float*>(w + P.off_part);
  G.L = P.L;
  G.nsplit_max = P.nsplit;
  G.stages = P.stages;
  G.ncw = P.ncw;
  const dim3 grid((unsigned)(P.ncb * P.nsplit), (unsigned)p->Hkv, (unsigned)p->B);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = to_status(cudaMemsetAsync(w + P.off_cnt, 0, P.off_part - P.off_cnt, st));
  if (rc != TOPO_OK) return rc;
  return dispatch(P.bf16, P.D, [&](auto L) {
    return P.dtc ? L.dense_tc(P.NC, mk, mv, G, grid, P.smem, st)
                 : L.dense(P.NC, mk, mv, G, grid, P.smem, st);
  });
}

int topo_attn_layer_schedule(int32_t L, int32_t pillar_every, const int32_t* windows,
                             int32_t n_windows, int32_t k, topo_layer* layers) {
  if (L < 1 || n_windows < 1 || !windows || !layers || k < 0 || k > TOPO_KMAX ||
      pillar_every < 0)
    return TOPO_ERR_INVALID_ARG;
  for (int i = 0; i < n_windows; ++i)
    if (windows[i] < 1) return TOPO_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l) {
    layers[l].dense = (pillar_every > 0 && l % pillar_every == 0) ? 1 : 0;
    layers[l].W = windows[(long long)l * n_windows / L];
    layers[l].k_top = k;
    layers[l].reserved = 0;
  }
  return TOPO_OK;
}

size_t topo_attn_layers_workspace_size(const topo_attn_params* p, const topo_layer* layers,
                                       int32_t L) {
  if (!p || !layers || L < 1) return 0;
  size_t need = 256;
  for (int l = 0; l < L; ++l) {
    const topo_attn_params lp = layer_params(p, layers[l]);
    Plan P;
    if (make_plan_cached(&lp, layers[l].dense != 0, &P) != TOPO_OK) return 0;
    need = P.total > need ? P.total : need;
  }
  return need;
}

int topo_attn_layers_forward(const topo_attn_params* p, const topo_layer* layers, int32_t L,
                             void* ws, size_t ws_bytes, topo_stream_t stream) {
  if (!p || !layers || L < 1) return TOPO_ERR_INVALID_ARG;
  // every layer is checked before the first one is enqueued
  for (int l = 0; l < L; ++l) {
    const topo_layer& ly = layers[l];
    const topo_attn_params lp = layer_params(p, ly);
    Plan P;
    const int rc = make_plan_cached(&lp, ly.dense != 0, &P);
    if (rc != TOPO_OK) return rc;
    if (ly.reserved != 0 || !ly.q || !ly.k || !ly.v || !ly.out) return TOPO_ERR_INVALID_ARG;
    if (!aligned16(ly.q) || !aligned16(ly.k) || !aligned16(ly.v)) return TOPO_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < P.total)
      return TOPO_ERR_WORKSPACE;
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  for (int l = 0; l < L; ++l) {
    const topo_layer& ly = layers[l];
    const topo_attn_params lp = layer_params(p, ly);
    const int rc = ly.dense ? dense_attn_forward(&lp, ly.q, ly.k, ly.v, ly.out, ws, ws_bytes,
                                                 stream)
                            : run_topo(&lp, ly.q, ly.k, ly.v, ly.out, nullptr, nullptr, ws,
                                       ws_bytes, st);
    if (rc != TOPO_OK) return rc;
  }
  return TOPO_OK;
}

const char* topo_attn_strerror(int status) {
  switch (status) {
    case TOPO_OK: return "ok";
    case TOPO_ERR_INVALID_ARG: return "invalid argument (shape, pointer or alignment)";
    case TOPO_ERR_UNSUPPORTED: return "unsupported configuration (d, k, dtype or size)";
    case TOPO_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case TOPO_ERR_CUDA: return "a CUDA call failed while enqueueing work";
    case TOPO_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case TOPO_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the no-allocation entry point's fixed buffer";
    case TOPO_ERR_BAD_BLOCK:
      return "a block-table entry was outside the pool (the block was read as block 0)";
    default: return "unknown status";
  }
}

int topo_attn_device_status(void* ws, int* status, topo_stream_t stream) {
  if (!ws || !status) return TOPO_ERR_INVALID_ARG;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaMemcpyAsync(&h, ws, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemsetAsync(ws, 0, sizeof h, st) != cudaSuccess)
    return TOPO_ERR_CUDA;
  *status = h;
  return TOPO_OK;
}

}  // extern "C"
