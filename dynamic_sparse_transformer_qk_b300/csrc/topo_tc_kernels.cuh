// topo_tc_kernels.cuh -- tensor-core (tcgen05) kernels for bf16 inputs with
// up to 16 query columns per KV head (decode): the condensate-set select
// kernel, its dependent tail kernel, and dense attention (pillar layers).
//
// Method ("The Condensate Theorem" explainer pages, technical summary
// sections 2-3): per query the condensate set is the anchor, the W most recent
// positions and the top-k remaining positions by q . k, re-identified at every
// step (every causal key is scored).  The selection must be the exact top-k
// under the float32 ranking score acc = fma(q[c], k[c], acc), c = 0..d-1.
//
// Scoring every key with that float32 chain costs d FMAs per (key, query
// head) on the CUDA cores.  Here the tensor cores score each 128-key tile
// against all query columns of the KV head in one MMA (bf16 products are
// exact, the accumulation is float32 but its rounding is not the chain's),
// and the exact chain is run only for the few keys that could still be in
// the top-k:
//
//   For a key j and query q, let s_j be the float32 chain and t_j the tensor
//   core result.  Both are within (gamma_d + beta_d) * sum_c |q_c k_jc| of the
//   exact dot product (gamma_d = d u / (1 - d u), u = 2^-24, for the chain; the
//   tensor cores' float32 accumulation is taken to be within beta_d = d 2^-21
//   relative to the same sum: the package's bound test, which runs this MMA on
//   random and cancellation-heavy rows, saw at most 14.2 * 2^-24 for d = 128,
//   some 70x below), so |t_j - s_j| <= delta_j <= F * ||q||_1 * max_c |k_jc|.
//   Each warp keeps an unordered candidate buffer.  If at least k buffered
//   keys have t >= T, their exact scores are >= T - delta*, delta* the
//   largest delta seen, so a key with t_j < T - 2 delta* (hence
//   s_j < T - delta*) is beaten by k keys and cannot be selected; T comes from
//   a search for (a lower bound of) the buffer's k-th best t.  Keys above that
//   cut are kept; at the end of the split the union of the warps' survivors is
//   cut again, the survivors (a few more than k) are rescored with the exact
//   chain and the exact top-k of the split is published, in the same format
//   the CUDA-core kernel uses.  If more near-ties than the buffers hold
//   survive (only with massively repeated scores), the split falls back to
//   scoring its keys with the exact chain on the CUDA cores.  The splits'
//   lists are merged, C_i written and the softmax taken by the dependent tail
//   kernel (one CTA per selection column), or by the last CTA of the unit.
//
// CTA layout: warp 0 lane 0 issues TMA loads of 128-key K tiles (two 128-byte
// column chunks, 128-byte swizzle) into a ring of stages; warp 1 owns the TMEM
// accumulators (16 columns per stage) and its lane 0 issues the MMAs
// (M = 128 keys, N = 16 padded query columns, K = d) and commits them to a
// per-stage barrier; warps 2..9 are the epilogue, two per TMEM lane quarter,
// taking alternate tiles: each thread owns one key of the tile, reads its
// column scores from TMEM and the key row's magnitude from shared memory, then
// the stage is released and the scores are offered to the warp's buffers.
#pragma once

#include <cuda_bf16.h>

#include "tc_device.cuh"
#include "topo_kernels.cuh"

namespace topo {

constexpr int kTcTile = 128;                  // keys per tile (MMA M)
constexpr int kTcN = 16;                      // MMA N: query columns, zero padded
constexpr int kTcEpiWarps = 8;                // epilogue warps
constexpr int kTcWarps = 2 + kTcEpiWarps;     // + TMA producer + MMA issuer
constexpr int kTcThreads = 32 * kTcWarps;
constexpr int kTcColsPerStage = kTcN;         // TMEM columns per stage

// candidate buffer entries per warp and column: room for the k-plus-near-ties
// survivors (2 * 32 * KE) plus one warp's worth of offers
__host__ __device__ constexpr int tc_cap(int KE) { return KE <= 1 ? 128 : 256; }

// F = 2 (gamma_d + beta_d), with gamma_d rounded up by 1 %; the factor 2 leaves
// room for the float32 rounding of ||q||_1 and of the threshold itself.
__host__ __device__ constexpr float tc_delta_factor(int D) {
  return 2.0f * ((float)D * 5.9604645e-8f * 1.01f + (float)D * 4.76837158e-7f);
}

// Shared-memory carve-up of the tensor-core select kernel (host and device).
struct TcSmem {
  int ring, qtile, bars, qd, buf, wmeta, cols, misc, total;
  __host__ __device__ TcSmem(int tile_bytes, int stages, int D, int NC, int KE) {
    int o = 0;
    ring = o;   o += stages * tile_bytes;          // multiple of 1024
    qtile = o;  o += kTcN * D * 2;                 // bf16 B operand (1024-aligned)
    bars = o;   o += 3 * stages * 8;               // full, empty, mma_done
    o = (o + 15) & ~15;
    qd = o;     o += D * NC * 8;                   // {q, q} float pairs, [c][col]
    buf = o;    o += kTcEpiWarps * NC * tc_cap(KE) * 8;
    wmeta = o;  o += kTcEpiWarps * NC * 16;        // per warp and column: TcMeta
    cols = o;   o += NC * (int)sizeof(ColInfo);
    misc = o;   o += 64;
    total = o + 1024;
  }
};

struct TcMeta {
  float delta;
  int overflow;
  int count;  // entries in the buffer at the end of the scan
  int pad;
};

// ------------------------------------------------ approximate-key buffer ----
//
// A warp's candidate buffer holds keys rank_key(t, j) (t: tensor-core score),
// in no particular order.

struct TcKept {
  int keep;
  float T;
};

// Rounds of the k-th-best search: each round counts the entries at or above
// three thresholds that split [lo, hi] into quarters (the three warp
// reductions are independent), so T ends within (max - min) / 4^rounds below
// the k-th best: a slightly lower cut, which only keeps a few more entries.
constexpr int kTcRounds = 5;

// Largest of lo and the quarter points tried, with at least k of the values
// at or above it; count(lo) >= k must hold, count(t) is warp-uniform.
template <typename F>
__device__ __forceinline__ float tc_search(float lo, float hi, int k, F count3) {
#pragma unroll 1
  for (int r = 0; r < kTcRounds && lo < hi; ++r) {
    const float q = 0.25f * (hi - lo);
    const float t1 = lo + q, t2 = lo + 2.f * q, t3 = lo + 3.f * q;
    int c1, c2, c3;
    count3(t1, t2, t3, c1, c2, c3);
    if (c3 >= k) lo = t3;
    else if (c2 >= k) { lo = t2; hi = t3; }
    else if (c1 >= k) { lo = t1; hi = t2; }
    else hi = t1;
  }
  return lo;
}

// Cut a warp's candidate buffer (cnt entries, any order) without sorting it:
// T is a lower bound of its k-th best tensor-core score (at least k entries
// score >= T), and the entries with t >= T - 2 delta move, in their order, to
// the front.  Fewer than k entries: unchanged, T = -inf.
template <int EC>
__device__ __noinline__ TcKept tc_cut(uint64_t* buf, int cnt, int k, float two_delta, int lane) {
  __syncwarp();
  if (k <= 0 || cnt < k) return TcKept{cnt, -INFINITY};
  uint64_t x[EC];
  float v[EC];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const int i = e * 32 + lane;
    x[e] = i < cnt ? buf[i] : 0ull;
    v[e] = i < cnt ? key_score(x[e]) : -INFINITY;
    mn = i < cnt ? fminf(mn, v[e]) : mn;
    mx = fmaxf(mx, v[e]);
  }
  mn = warp_min(mn);
  mx = warp_max(mx);
  const float T = tc_search(mn, mx, k, [&](float t1, float t2, float t3, int& c1, int& c2,
                                            int& c3) {
    int a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
    for (int e = 0; e < EC; ++e) {
      a1 += v[e] >= t1 ? 1 : 0;
      a2 += v[e] >= t2 ? 1 : 0;
      a3 += v[e] >= t3 ? 1 : 0;
    }
    c1 = __reduce_add_sync(kFull, a1);
    c2 = __reduce_add_sync(kFull, a2);
    c3 = __reduce_add_sync(kFull, a3);
  });
  const float cut = T - two_delta;
  __syncwarp();
  int keep = 0;
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const bool kp = v[e] >= cut;
    const unsigned m = __ballot_sync(kFull, kp);
    if (kp) buf[keep + __popc(m & ((1u << lane) - 1u))] = x[e];
    keep += __popc(m);
  }
  __syncwarp();
  return TcKept{keep, T};
}

template <bool BF16, int D>
__device__ __forceinline__ float row_magnitude(const uint8_t* tile, int r);

// Largest |k_c| of key row r of a bf16 tile (two 128-byte column chunks per
// row for d = 128, one for d = 64), read in swizzled order (conflict-free).
template <>
__device__ __forceinline__ float row_magnitude<true, 128>(const uint8_t* tile, int r) {
  __nv_bfloat162 m = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint4 w = *reinterpret_cast<const uint4*>(tile + cc * (kTcTile * 128) + r * 128 +
                                                      ((g ^ (r & 7)) << 4));
      m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.x)));
      m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.y)));
      m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.z)));
      m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.w)));
    }
  }
  return fmaxf(__low2float(m), __high2float(m));
}

template <>
__device__ __forceinline__ float row_magnitude<true, 64>(const uint8_t* tile, int r) {
  __nv_bfloat162 m = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint4 w = *reinterpret_cast<const uint4*>(tile + r * 128 + ((g ^ (r & 7)) << 4));
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.x)));
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.y)));
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.z)));
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.w)));
  }
  return fmaxf(__low2float(m), __high2float(m));
}

template <int NL>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[NL]);
template <>
__device__ __forceinline__ void tmem_ld_cols<4>(uint32_t taddr, float (&v)[4]) {
  tc::tmem_ld4(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, float (&v)[8]) {
  tc::tmem_ld8(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, float (&v)[16]) {
  tc::tmem_ld16(taddr, v);
}

// Split geometry of one (sequence, KV head, column block) unit of the
// tensor-core select kernel: splits cover keys kbase..jmax, from key 1 (the
// first candidate), or, for a paged cache, from key 0 so that every 128-key
// tile starts on a block boundary (key 0, the anchor, is then masked out of
// the candidates).  The tail kernel recomputes it to find the split lists.
struct TcSplits {
  long long jmax, kbase, unit, Lu;
  int nsplit;
};

__device__ __forceinline__ TcSplits tc_splits(const Geom& G, int b, int kvh, long long cb) {
  TcSplits r;
  const long long last_col = G.ncols - 1;  // the tensor-core kernel has one column block
  const long long pos_max = seq_len(G, b) - G.nq + last_col / G.g;
  r.jmax = G.topk > 0 ? pos_max - G.W : 0;
  r.kbase = G.block_table ? 0 : 1;
  const long long ncand = r.jmax > 0 ? r.jmax + 1 - r.kbase : 0;
  r.unit = ((long long)b * G.Hkv + kvh) * G.ncb + cb;
  r.Lu = r.unit < G.hi_units ? G.L2 : G.L;  // keys per split of this unit
  r.nsplit = ncand > 0 ? (int)((ncand + r.Lu - 1) / r.Lu) : 1;
  return r;
}

// ======================================== tensor-core select kernel ==========
//
// Grid and workspace as topo_select_kernel (grid.x = column block x split,
// grid.y = KV head, grid.z = sequence); a split is G.L keys (a multiple of
// 128).  bf16 only; k <= 32 * KE, KE <= 2; NC <= 16 columns per block (the
// MMA's N) with KE = 1, NC <= 4 with KE = 2.
//
// GROUP: group-shared selection (grouped-query attention).  The block's
// columns are (row, head) pairs, col = row * g + head; the g heads of a row
// share one condensate set, whose top-k ranks key j by the largest of the
// heads' float32 scores.  Selection runs on "selection columns" s = col / g
// (one per row): the epilogue offers max over the group's tensor-core scores
// (each within delta_h of its exact score, so the max is within max_h
// delta_h of the exact max), survivors are rescored as the max of the heads'
// exact chains, and the tail gives every head of the row the row's set.
template <int D, int NC, int KE, bool GROUP>
__global__ void __launch_bounds__(kTcThreads, 1)
    topo_select_tc_kernel(const __grid_constant__ CUtensorMap map_k, const Geom G) {
  using S = Shape<true, D>;
  constexpr int CAP = tc_cap(KE);
  constexpr int EC = CAP / 32;
  constexpr int KP = 32 * KE;
  constexpr int LE = 2 * KE;          // union list length / 32 (k plus near ties)
  constexpr int LL = 32 * LE;
  constexpr int TILEB = kTcTile * S::ROWB;
  constexpr int KSTEPS = D / 16;      // MMA K = 16 bf16 per instruction
  constexpr int NL = NC <= 4 ? 4 : (NC <= 8 ? 8 : 16);
  static_assert((KE == 1 ? NC <= kTcN : NC <= 4) && KE <= 2 && LL + 32 <= CAP &&
                    cap_for(KE) <= CAP,
                "tensor-core select shape");

  const int b = blockIdx.z, kvh = blockIdx.y;
  const long long cb = blockIdx.x / G.nsplit_max;
  const int split = (int)(blockIdx.x % G.nsplit_max);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kk = G.topk;

  // a dependent tail kernel may start its set-up now (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const TcSplits sp = tc_splits(G, b, kvh, cb);
  const long long jmax = sp.jmax, kbase = sp.kbase, unit = sp.unit, Lu = sp.Lu;
  const int nsplit = sp.nsplit;
  if (split >= nsplit) return;
  const long long ks = kbase + (long long)split * Lu;
  const long long ke = (ks + Lu - 1 < jmax) ? ks + Lu - 1 : jmax;  // inclusive
  const int ntiles = ke >= ks ? (int)((ke - ks + kTcTile) / kTcTile) : 0;
  const int stages = G.stages;

  uint8_t* sm = aligned_smem_base();
  const TcSmem L(TILEB, stages, D, NC, KE);
  uint8_t* ring = sm + L.ring;
  uint8_t* qtile = sm + L.qtile;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + stages;
  uint64_t* mdone = empty + stages;
  float2* qd = reinterpret_cast<float2*>(sm + L.qd);
  uint64_t* wbuf = reinterpret_cast<uint64_t*>(sm + L.buf);
  TcMeta* meta = reinterpret_cast<TcMeta*>(sm + L.wmeta);
  ColInfo* cols = reinterpret_cast<ColInfo*>(sm + L.cols);
  volatile int* misc = reinterpret_cast<volatile int*>(sm + L.misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L.misc + 32);

  if (tid == 0) {
    misc[0] = 0;  // abort
    misc[1] = 0;  // last CTA of the column block
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
      mbar_init(&mdone[s], 1);
    }
    fence_mbar_init();
  }
  load_columns<true, D, NC>(G, b, kvh, cb, cols, qd);
  __syncthreads();
  // B operand: query columns as bf16 rows (exact: the inputs are bf16), rows
  // NC..15 zero, K-major with the 128-byte swizzle
  for (int i = tid; i < kTcN * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    const float x = r < NC ? qd[c * NC + r].x : 0.f;
    *reinterpret_cast<__nv_bfloat16*>(qtile + tc::sw128_offset_bf16(r, c, kTcN)) =
        __float2bfloat16_rn(x);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const uint32_t tmem_cols = 32u < (uint32_t)(stages * kTcColsPerStage)
                                 ? (stages * kTcColsPerStage <= 64
                                        ? 64u
                                        : (stages * kTcColsPerStage <= 128 ? 128u : 256u))
                                 : 32u;
  if (warp == 1) {
    tc::tmem_alloc(tslot, tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;


  if (warp == 0) {
    // ---------------- TMA producer ------------------------------------------
    if (lane == 0 && ntiles > 0) {
      prefetch_tmap(&map_k);
      int t = 0;
      for (; t < ntiles; ++t) {
        if (misc[0]) break;
        const int s = t % stages;
        const uint32_t round = (uint32_t)(t / stages);
        if (!mbar_wait(&empty[s], (round & 1u) ^ 1u)) {
          set_status(G.status, kStatusTimeout);
          misc[0] = 1;
          break;
        }
        uint8_t* dst = ring + (size_t)s * TILEB;
        mbar_arrive_expect_tx(&full[s], (uint32_t)TILEB);
        const int y = (int)kv_row(G, b, kvh, ks + (long long)t * kTcTile);
#pragma unroll
        for (int cc = 0; cc < S::NCH; ++cc)
          tma_load_2d(dst + cc * (kTcTile * 128), &map_k, cc * S::EPC, y, &full[s]);
      }
      drain_tiles(t, stages, full, G.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer --------------------------------------------
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTcTile, kTcN);
      const uint32_t qaddr = smem_addr(qtile);
      int t = 0;
      for (; t < ntiles; ++t) {
        if (misc[0]) break;
        const int s = t % stages;
        const uint32_t round = (uint32_t)(t / stages);
        // the epilogue has released this stage's accumulator, and its tile landed
        if (!mbar_wait(&empty[s], (round & 1u) ^ 1u) || !mbar_wait(&full[s], round & 1u)) {
          set_status(G.status, kStatusTimeout);
          misc[0] = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t aaddr = smem_addr(ring + (size_t)s * TILEB);
#pragma unroll
        for (int ks16 = 0; ks16 < KSTEPS; ++ks16) {
          const uint32_t ao = aaddr + (ks16 >> 2) * (kTcTile * 128) + (ks16 & 3) * 32;
          const uint32_t bo = qaddr + (ks16 >> 2) * (kTcN * 128) + (ks16 & 3) * 32;
          tc::mma_bf16(tmem + (uint32_t)(s * kTcColsPerStage), tc::smem_desc_sw128(ao),
                       tc::smem_desc_sw128(bo), idesc, ks16 > 0);
        }
        tc::mma_commit(&mdone[s]);
      }
      // no MMA may still be running when the accumulators are freed
      if (t > 0) {
        const int tl = t - 1;
        if (!mbar_wait(&mdone[tl % stages], (uint32_t)(tl / stages) & 1u))
          set_status(G.status, kStatusTimeout);
      }
    }
  } else {
    // ---------------- epilogue ----------------------------------------------
    const int e = warp - 2;           // 0..7
    const int half = e >> 2;          // tiles t with t % 2 == half
    const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;  // this thread's key row in a tile
    uint64_t* mybuf = wbuf + (size_t)e * NC * CAP;
    float coef[NC], T[NC], thr[NC];
    int cnt[NC];
    bool ovf[NC];
    int jh[NC];  // last candidate position per column (< 2^31)
    const int gsz = GROUP ? G.g : 1;  // heads per selection column
#pragma unroll
    for (int h = 0; h < NC; ++h) {
      float a = 0.f;
      for (int c = lane; c < D; c += 32) a += fabsf(qd[c * NC + h].x);
      coef[h] = tc_delta_factor(D) * warp_sum(a) * 1.001f;
      T[h] = -INFINITY;
      thr[h] = -INFINITY;
      cnt[h] = 0;
      ovf[h] = false;
      jh[h] = cols[h].active ? (int)(cols[h].jhi < ke ? cols[h].jhi : ke) : 0;
    }
    if constexpr (GROUP) {
      // selection column s covers columns s*g .. s*g+g-1: the largest
      // coefficient of its heads bounds the error of the max
#pragma unroll
      for (int h = 0; h < NC; ++h) {
        if (h % gsz != 0) continue;
        float cm = coef[h];
#pragma unroll
        for (int i = 1; i < NC; ++i)
          if (i < gsz && h + i < NC) cm = fmaxf(cm, coef[h + i]);
        coef[h / gsz] = cm;
        jh[h / gsz] = jh[h];
      }
    }
    float kmag = 0.f;  // largest |k_c| seen by this warp
    for (int t = half; t < ntiles; t += 2) {
      const int s = t % stages;
      const uint32_t round = (uint32_t)(t / stages);
      const bool ok = __all_sync(kFull, mbar_wait(&mdone[s], round & 1u));
      if (!ok || misc[0]) {
        if (!ok && lane == 0) {
          set_status(G.status, kStatusTimeout);
          misc[0] = 1;
        }
        break;
      }
      tc::fence_after_sync();
      float sc[NL];
      tmem_ld_cols<NL>(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(s * kTcColsPerStage),
                       sc);
      tc::tmem_ld_wait();
      if constexpr (GROUP) {
        // selection column h: the largest score of its heads
#pragma unroll
        for (int h = 0; h < NC; ++h) {
          if (h * gsz >= NC) continue;
          float m = sc[h * gsz];
#pragma unroll
          for (int i = 1; i < NC; ++i)
            if (i < gsz && h * gsz + i < NC) m = fmaxf(m, sc[h * gsz + i]);
          sc[h] = m;
        }
      }
      const long long j = ks + (long long)t * kTcTile + r;
      const float mk = j <= ke ? row_magnitude<true, D>(ring + (size_t)s * TILEB, r) : 0.f;
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      const float wm = warp_max(mk);
      if (wm > kmag) {  // larger keys: widen the admission margin
        kmag = wm;
#pragma unroll
        for (int h = 0; h < NC; ++h)
          if (!ovf[h]) thr[h] = T[h] - 2.f * coef[h] * kmag;
      }
#pragma unroll
      for (int h = 0; h < NC; ++h) {
        if (GROUP && h * gsz >= NC) continue;
        const bool cand = j <= jh[h] && j >= 1;
        bool flag = cand && sc[h] >= thr[h];
        unsigned mask = __ballot_sync(kFull, flag);
        if (mask == 0u) continue;
        uint64_t* hb = mybuf + h * CAP;
        if (cnt[h] + __popc(mask) > CAP) {
          const TcKept kept = tc_cut<EC>(hb, cnt[h], kk, 2.f * coef[h] * kmag, lane);
          cnt[h] = kept.keep;
          T[h] = kept.T;
          thr[h] = T[h] - 2.f * coef[h] * kmag;
          if (cnt[h] + 32 > CAP) {  // the buffer is full of near ties
            ovf[h] = true;
            thr[h] = INFINITY;
          }
          flag = cand && sc[h] >= thr[h];
          mask = __ballot_sync(kFull, flag);
          if (mask == 0u) continue;
        }
        if (flag) hb[cnt[h] + __popc(mask & ((1u << lane) - 1u))] = rank_key(sc[h], (uint32_t)j);
        cnt[h] += __popc(mask);
      }
    }
    // the buffers go to the per-column stage as they are
#pragma unroll 1
    for (int h = 0; h < (GROUP ? NC / gsz : NC); ++h)
      if (lane == 0) {
        meta[e * NC + h].delta = coef[h] * kmag;
        meta[e * NC + h].overflow = ovf[h] ? 1 : 0;
        meta[e * NC + h].count = cnt[h];
      }
  }
  // every role is done with the ring and the accumulators
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols);
  }

  // ---------------- per column: exact top-k of this split ----------------
  const int nsel = GROUP ? NC / G.g : NC;
  // the exact score of a selection column: one head's chain, or the largest
  // of the group's heads' chains
  auto exact_score = [&](long long row, int h) -> float {
    if constexpr (GROUP) {
      float m = score_row_global<true, D, NC>(G.kp, row, qd, h * G.g);
      for (int i = 1; i < G.g; ++i)
        m = fmaxf(m, score_row_global<true, D, NC>(G.kp, row, qd, h * G.g + i));
      return m;
    } else {
      return score_row_global<true, D, NC>(G.kp, row, qd, h);
    }
  };
  // Per selection column: the warps' buffers concatenated in the (now idle)
  // ring, cut at T - 2 delta* (T a lower bound of the union's k-th best), the
  // survivors gathered at the front.  Returns the overflow flag (more near
  // ties than LL slots, or a warp's buffer overflowed).
  auto gather = [&](int h, uint64_t* cat, int& ns) -> int {
    float dmax = 0.f;
    int ov = 0, total = 0;
    for (int w = 0; w < kTcEpiWarps; ++w) {
      const TcMeta mt = meta[w * NC + h];
      dmax = fmaxf(dmax, mt.delta);
      ov |= mt.overflow;
      const uint64_t* src = wbuf + ((size_t)w * NC + h) * CAP;
      for (int i = lane; i < mt.count; i += 32) cat[total + i] = src[i];
      total += mt.count;
    }
    __syncwarp();
    // none are cut while the union holds fewer than k entries
    float cut = -INFINITY;
    if (kk > 0 && total >= kk) {
      float mn = INFINITY, mx = -INFINITY;
      for (int i = lane; i < total; i += 32) {
        const float t = key_score(cat[i]);
        mn = fminf(mn, t);
        mx = fmaxf(mx, t);
      }
      mn = warp_min(mn);
      mx = warp_max(mx);
      const float T = tc_search(mn, mx, kk, [&](float t1, float t2, float t3, int& c1, int& c2,
                                                 int& c3) {
        int a1 = 0, a2 = 0, a3 = 0;
#pragma unroll 4
        for (int i = lane; i < total; i += 32) {
          const float t = key_score(cat[i]);
          a1 += t >= t1 ? 1 : 0;
          a2 += t >= t2 ? 1 : 0;
          a3 += t >= t3 ? 1 : 0;
        }
        c1 = __reduce_add_sync(kFull, a1);
        c2 = __reduce_add_sync(kFull, a2);
        c3 = __reduce_add_sync(kFull, a3);
      });
      cut = T - 2.f * dmax;
    }
    // in place: a write never passes its read
    ns = 0;
    for (int i0 = 0; i0 < total && !ov; i0 += 32) {
      const uint64_t key = i0 + lane < total ? cat[i0 + lane] : 0ull;
      const bool kp = key != 0ull && key_score(key) >= cut;
      const unsigned m = __ballot_sync(kFull, kp);
      __syncwarp();
      if (kp) cat[ns + __popc(m & ((1u << lane) - 1u))] = key;
      ns += __popc(m);
      __syncwarp();
    }
    return (ov || ns > LL) ? 1 : 0;
  };
  // rescore gathered entry i (< ns) with the exact float32 chain
  auto rescore = [&](int h, const uint64_t* cat, int ns, int i) -> uint64_t {
    const uint64_t key = i < ns ? cat[i] : 0ull;
    if (key == 0ull) return 0ull;
    const uint32_t jj = key_pos(key);
    return rank_key(exact_score(kv_row(G, b, kvh, jj), h), jj);
  };
  // sort the rescored keys (or score the split on the CUDA cores after an
  // overflow) and publish the split's exact top-k of column h
  auto publish = [&](int h, uint64_t (&x)[LE], int ov) {
    uint64_t* scratch = wbuf + (size_t)h * CAP;  // the fallback's buffer
    if (!ov) {
      warp_sort_desc<LE>(x, lane);
    } else {
      // fallback: every key of the split through the exact chain (CUDA cores)
      constexpr int FEC = cap_for(KE) / 32;
      uint64_t fthr = 0ull;
      int fcnt = 0;
      const int hc = GROUP ? h * G.g : h;  // a column of the selection column
      const long long lim = cols[hc].active ? (cols[hc].jhi < ke ? cols[hc].jhi : ke) : 0;
      for (long long j0 = ks; j0 <= lim; j0 += 32) {
        const long long j = j0 + lane;
        const uint64_t key = (j <= lim && j >= 1)
                                 ? rank_key(exact_score(kv_row(G, b, kvh, j), h), (uint32_t)j)
                                 : 0ull;
        offer<FEC, KE>(scratch, fthr, fcnt, key, kk, lane);
      }
      __syncwarp();
      uint64_t y[FEC];
#pragma unroll
      for (int ee = 0; ee < FEC; ++ee) {
        const int i = ee * 32 + lane;
        y[ee] = i < fcnt ? scratch[i] : 0ull;
      }
      warp_sort_desc<FEC>(y, lane);
#pragma unroll
      for (int ee = 0; ee < LE; ++ee) x[ee] = ee < FEC ? y[ee] : 0ull;
    }
    unsigned long long* dst = G.lists + (((size_t)unit * G.nsplit_max + split) * NC + h) * KP;
#pragma unroll
    for (int ee = 0; ee < KE; ++ee) {
      const int i = ee * 32 + lane;
      const int hc = GROUP ? h * G.g : h;
      dst[i] = (i < kk && cols[hc].active) ? x[ee] : 0ull;
      // the V rows the final softmax may gather, on their way to L2
      if (i < kk && cols[hc].active && x[ee] != 0ull && G.vp)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(
            reinterpret_cast<const uint8_t*>(G.vp) + kv_row(G, b, kvh, key_pos(x[ee])) * S::ROWB));
    }
  };
  const int ew = warp - 2;  // epilogue warp, or < 0
  if (ew >= 0 && 2 * nsel <= kTcEpiWarps) {
    // two warps per column: the leader gathers, both rescore alternate
    // 32-entry blocks (into slots LL..2LL of the ring area), the leader sorts
    // and publishes; a named barrier per column pairs them
    constexpr int HALF = kTcEpiWarps / 2;
    const int h = ew % HALF, role = ew / HALF;
    if (h < nsel) {
      uint64_t* cat = reinterpret_cast<uint64_t*>(ring) + (size_t)h * kTcEpiWarps * CAP;
      if (role == 0) {
        int ns = 0;
        const int ov = gather(h, cat, ns);
        if (lane == 0) cat[2 * LL] = (uint64_t)(uint32_t)ns | ((uint64_t)ov << 32);
      }
      asm volatile("bar.sync %0, 64;" ::"r"(1 + h) : "memory");
      const uint64_t info = cat[2 * LL];
      const int ns = (int)(uint32_t)info, ov = (int)(info >> 32);
      if (!ov) {
#pragma unroll
        for (int ee = 0; ee < LE; ++ee)
          if ((ee & 1) == role) cat[LL + ee * 32 + lane] = rescore(h, cat, ns, ee * 32 + lane);
      }
      asm volatile("bar.sync %0, 64;" ::"r"(1 + h) : "memory");
      if (role == 0) {
        uint64_t x[LE];
#pragma unroll
        for (int ee = 0; ee < LE; ++ee) x[ee] = ov ? 0ull : cat[LL + ee * 32 + lane];
        publish(h, x, ov);
      }
    }
  } else {
    // one warp per column, each warp reusing its own area of the ring
    for (int h = ew; h >= 0 && h < nsel; h += kTcEpiWarps) {
      uint64_t* cat = reinterpret_cast<uint64_t*>(ring) + (size_t)ew * kTcEpiWarps * CAP;
      int ns = 0;
      const int ov = gather(h, cat, ns);
      uint64_t x[LE];
#pragma unroll
      for (int ee = 0; ee < LE; ++ee) x[ee] = ov ? 0ull : rescore(h, cat, ns, ee * 32 + lane);
      publish(h, x, ov);
    }
  }
  if (G.flags & kSplitTail) return;  // the tail kernel takes it from here
  if (!finish_split(G.counters + unit, nsplit, misc)) return;
  select_tail<true, D, NC, KE, kTcWarps, GROUP>(G, unit, nsplit, b, kvh, cols, qd, wbuf, ring,
                                                stages * TILEB);
}

// ============================================== tensor-core select: tail ====
//
// With kSplitTail the select kernel stops after publishing its split lists
// and this kernel, launched as its programmatic dependent, does the tail one
// selection column per CTA (grid.x: columns, or rows of group-shared sets):
// merge the splits' lists, write C_i, stage the set's K and V rows and take
// the softmax (select_tail restricted to the CTA's columns).  Its set-up
// overlaps the end of the scan; the lists are read only after the wait on
// the select grid, whose completion makes them visible.
struct TailSmem {
  int run, cols, qd, misc, total;
  __host__ __device__ TailSmem(int scratch_bytes, int D, int NC, int KP) {
    int o = (scratch_bytes + 1023) & ~1023;  // select_tail's scratch first
    run = o;   o += NC * KP * 8;
    cols = o;  o += NC * (int)sizeof(ColInfo);
    qd = o;    o += D * NC * 8;
    misc = o;  o += 64;
    total = o + 1024;
  }
};

// Two CTAs per SM (registers <= 102): batched decode runs hundreds of tails.
template <int D, int NC, int KE, bool GROUP>
__global__ void __launch_bounds__(kTcThreads, 2)
    topo_tail_tc_kernel(const Geom G, int scratch_bytes) {
  constexpr int KP = 32 * KE;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int gsz = GROUP ? G.g : 1;
  const int h0 = (int)blockIdx.x * gsz, h1 = h0 + gsz;
  uint8_t* sm = aligned_smem_base();
  const TailSmem L(scratch_bytes, D, NC, KP);
  uint64_t* run = reinterpret_cast<uint64_t*>(sm + L.run);
  ColInfo* cols = reinterpret_cast<ColInfo*>(sm + L.cols);
  float2* qd = reinterpret_cast<float2*>(sm + L.qd);
  load_columns<true, D, NC>(G, b, kvh, 0, cols, qd);
  __syncthreads();
  if (threadIdx.x < NC && ((int)threadIdx.x < h0 || (int)threadIdx.x >= h1))
    cols[threadIdx.x].active = 0;
  const TcSplits sp = tc_splits(G, b, kvh, 0);
  // the window band and anchor rows do not depend on the selection: with
  // kEarlyBand, start staging them before waiting
  const bool early = (G.flags & kEarlyBand) != 0;
  if (early)
    select_tail<true, D, NC, KE, kTcWarps, GROUP>(G, sp.unit, sp.nsplit, b, kvh, cols, qd, run,
                                                  sm, scratch_bytes, h0, h1, 1);
  // the select grid has completed and its lists are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  select_tail<true, D, NC, KE, kTcWarps, GROUP>(G, sp.unit, sp.nsplit, b, kvh, cols, qd, run, sm,
                                                scratch_bytes, h0, h1, early ? 2 : 0);
}

// ============================================ tensor-core dense attention ====
//
// Dense causal attention over keys 0..p (the pillar layers, and the
// reference the condensate set is compared with) for bf16 inputs with every
// query column of a KV head in one block.  Split-n as the CUDA-core dense
// kernel; per 128-key tile one MMA scores all columns into TMEM exactly as in
// the select kernel, and eight epilogue warps -- two per TMEM lane quarter,
// taking alternate tiles -- each keep an online softmax (m, l) per column
// over the keys they own and a float32 weighted sum of those keys' V rows,
// read from the same ring stage (K tile, then V tile).  The warps' states
// merge in shared memory, the splits' in the CTA that finishes last.
struct DenseTcSmem {
  int ring, qtile, bars, qd, pbuf, cols, misc, total;
  __host__ __device__ DenseTcSmem(int stage_bytes, int stages, int D, int NC) {
    int o = 0;
    ring = o;   o += stages * stage_bytes;      // K tile | V tile (multiples of 1024)
    qtile = o;  o += kTcN * D * 2;              // bf16 B operand (1024-aligned)
    bars = o;   o += 3 * stages * 8;            // full, empty, mma_done
    o = (o + 15) & ~15;
    qd = o;     o += D * NC * 8;
    pbuf = o;   o += kTcEpiWarps * 32 * NC * 4;  // per warp: weights of its 32 keys
    cols = o;   o += NC * (int)sizeof(ColInfo);
    misc = o;   o += 64;
    total = o + 1024;
  }
};

template <int D, int NC>
__global__ void __launch_bounds__(kTcThreads, 1)
    dense_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const Geom G) {
  using S = Shape<true, D>;
  constexpr int TILEB = kTcTile * S::ROWB;
  constexpr int STAGEB = 2 * TILEB;
  constexpr int KSTEPS = D / 16;
  constexpr int NL = NC <= 4 ? 4 : 8;
  constexpr int EPL = S::EPL;
  constexpr int PART = D + 2;  // m, l, acc[D]
  static_assert(NC <= 8 && EPL % 2 == 0, "dense tensor-core shape");

  const int b = blockIdx.z, kvh = blockIdx.y;
  const int split = (int)blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long pos_max = seq_len(G, b) - G.nq + (G.ncols - 1) / G.g;
  const long long nkeys = pos_max + 1;
  const int nsplit = (int)((nkeys + G.L - 1) / G.L);
  if (split >= nsplit) return;
  const long long ks = (long long)split * G.L;
  const long long ke = (ks + G.L - 1 < pos_max) ? ks + G.L - 1 : pos_max;
  const int ntiles = (int)((ke - ks + kTcTile) / kTcTile);
  const long long unit = (long long)b * G.Hkv + kvh;
  const int stages = G.stages;

  uint8_t* sm = aligned_smem_base();
  const DenseTcSmem L(STAGEB, stages, D, NC);
  uint8_t* ring = sm + L.ring;
  uint8_t* qtile = sm + L.qtile;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + stages;
  uint64_t* mdone = empty + stages;
  float2* qd = reinterpret_cast<float2*>(sm + L.qd);
  float* pbuf_all = reinterpret_cast<float*>(sm + L.pbuf);
  ColInfo* cols = reinterpret_cast<ColInfo*>(sm + L.cols);
  volatile int* misc = reinterpret_cast<volatile int*>(sm + L.misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L.misc + 32);

  if (tid == 0) {
    misc[0] = 0;  // abort
    misc[1] = 0;  // last CTA of the unit
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
      mbar_init(&mdone[s], 1);
    }
    fence_mbar_init();
  }
  load_columns<true, D, NC>(G, b, kvh, 0, cols, qd);
  __syncthreads();
  for (int i = tid; i < kTcN * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    const float x = r < NC ? qd[c * NC + r].x : 0.f;
    *reinterpret_cast<__nv_bfloat16*>(qtile + tc::sw128_offset_bf16(r, c, kTcN)) =
        __float2bfloat16_rn(x);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const uint32_t tmem_cols = stages * kTcColsPerStage <= 32
                                 ? 32u
                                 : (stages * kTcColsPerStage <= 64
                                        ? 64u
                                        : (stages * kTcColsPerStage <= 128 ? 128u : 256u));
  if (warp == 1) {
    tc::tmem_alloc(tslot, tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  float m[NC], l[NC];
  float2 acc[NC][EPL / 2];  // this lane's output elements 2i, 2i+1 (paired FMAs)
#pragma unroll
  for (int h = 0; h < NC; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
  }

  if (warp == 0) {
    // ---------------- TMA producer: K tile, then V tile, per stage ----------
    if (lane == 0 && ntiles > 0) {
      prefetch_tmap(&map_k);
      prefetch_tmap(&map_v);
      const long long row0 = ((long long)b * G.Hkv + kvh) * G.kv_stride + ks;
      int t = 0;
      for (; t < ntiles; ++t) {
        if (misc[0]) break;
        const int s = t % stages;
        const uint32_t round = (uint32_t)(t / stages);
        if (!mbar_wait(&empty[s], (round & 1u) ^ 1u)) {
          set_status(G.status, kStatusTimeout);
          misc[0] = 1;
          break;
        }
        uint8_t* dst = ring + (size_t)s * STAGEB;
        mbar_arrive_expect_tx(&full[s], (uint32_t)STAGEB);
        const int y = (int)(row0 + (long long)t * kTcTile);
#pragma unroll
        for (int cc = 0; cc < S::NCH; ++cc) {
          tma_load_2d(dst + cc * (kTcTile * 128), &map_k, cc * S::EPC, y, &full[s]);
          tma_load_2d(dst + TILEB + cc * (kTcTile * 128), &map_v, cc * S::EPC, y, &full[s]);
        }
      }
      drain_tiles(t, stages, full, G.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer --------------------------------------------
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTcTile, kTcN);
      const uint32_t qaddr = smem_addr(qtile);
      int t = 0;
      for (; t < ntiles; ++t) {
        if (misc[0]) break;
        const int s = t % stages;
        const uint32_t round = (uint32_t)(t / stages);
        if (!mbar_wait(&empty[s], (round & 1u) ^ 1u) || !mbar_wait(&full[s], round & 1u)) {
          set_status(G.status, kStatusTimeout);
          misc[0] = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t aaddr = smem_addr(ring + (size_t)s * STAGEB);
#pragma unroll
        for (int ks16 = 0; ks16 < KSTEPS; ++ks16) {
          const uint32_t ao = aaddr + (ks16 >> 2) * (kTcTile * 128) + (ks16 & 3) * 32;
          const uint32_t bo = qaddr + (ks16 >> 2) * (kTcN * 128) + (ks16 & 3) * 32;
          tc::mma_bf16(tmem + (uint32_t)(s * kTcColsPerStage), tc::smem_desc_sw128(ao),
                       tc::smem_desc_sw128(bo), idesc, ks16 > 0);
        }
        tc::mma_commit(&mdone[s]);
      }
      if (t > 0) {
        const int tl = t - 1;
        if (!mbar_wait(&mdone[tl % stages], (uint32_t)(tl / stages) & 1u))
          set_status(G.status, kStatusTimeout);
      }
    }
  } else {
    // ---------------- epilogue: online softmax and weighted sum -------------
    const int e = warp - 2;           // 0..7
    const int half = e >> 2;          // tiles t with t % 2 == half
    const int quarter = warp & 3;     // TMEM lanes (tile rows) 32*quarter .. +31
    float* pb = pbuf_all + e * 32 * NC;
    long long lim[NC];
#pragma unroll
    for (int h = 0; h < NC; ++h) {
      const long long p = cols[h].active ? cols[h].pos : -1;
      lim[h] = p < ke ? p : ke;
    }
    for (int t = half; t < ntiles; t += 2) {
      const int s = t % stages;
      const uint32_t round = (uint32_t)(t / stages);
      const bool ok = __all_sync(kFull, mbar_wait(&mdone[s], round & 1u));
      if (!ok || misc[0]) {
        if (!ok && lane == 0) {
          set_status(G.status, kStatusTimeout);
          misc[0] = 1;
        }
        break;
      }
      tc::fence_after_sync();
      float sc[NL];
      tmem_ld_cols<NL>(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(s * kTcColsPerStage),
                       sc);
      tc::tmem_ld_wait();
      const long long r0 = ks + (long long)t * kTcTile + quarter * 32;  // this warp's first key
      const long long j = r0 + lane;
#pragma unroll
      for (int h = 0; h < NC; ++h) {
        const float lg = j <= lim[h] ? G.scale * sc[h] : -INFINITY;
        const float mnew = fmaxf(m[h], warp_max(lg));
        float p = 0.f, alpha = 1.f;
        if (mnew != -INFINITY) {
          alpha = m[h] == -INFINITY ? 0.f : expf(m[h] - mnew);
          p = lg == -INFINITY ? 0.f : expf(lg - mnew);
        }
        l[h] = l[h] * alpha + warp_sum(p);
#pragma unroll
        for (int i = 0; i < EPL / 2; ++i) {
          acc[h][i].x *= alpha;
          acc[h][i].y *= alpha;
        }
        m[h] = mnew;
        pb[lane * NC + h] = p;
      }
      __syncwarp();
      // rows past the split's last key are skipped (their V may be anything)
      const int nrows = (int)(ke - r0 + 1 < 32 ? (ke - r0 + 1 > 0 ? ke - r0 + 1 : 0) : 32);
      const uint8_t* vt = ring + (size_t)s * STAGEB + TILEB;
#pragma unroll 2
      for (int rr = 0; rr < nrows; ++rr) {
        float v[EPL];
        lane_elems<true, D>(vt + tile_lane_offset<true, D, kTcTile>(quarter * 32 + rr, lane), v);
        float pr[NC];
        if constexpr (NC % 4 == 0) {
#pragma unroll
          for (int h = 0; h < NC; h += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(pb + rr * NC + h);
            pr[h] = p4.x;
            pr[h + 1] = p4.y;
            pr[h + 2] = p4.z;
            pr[h + 3] = p4.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < NC; ++h) pr[h] = pb[rr * NC + h];
        }
#pragma unroll
        for (int h = 0; h < NC; ++h)
#pragma unroll
          for (int i = 0; i < EPL / 2; ++i)
            acc[h][i] = __ffma2_rn(make_float2(pr[h], pr[h]), make_float2(v[2 * i], v[2 * i + 1]),
                                   acc[h][i]);
      }
      // this warp is done with the stage's accumulator and V rows
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
  // combine the epilogue warps in shared memory (the ring is free), publish
  float* red = reinterpret_cast<float*>(ring);  // [epilogue warp][NC][PART]
  if (warp >= 2) {
    const int e = warp - 2;
#pragma unroll
    for (int h = 0; h < NC; ++h) {
      float* r = red + ((size_t)e * NC + h) * PART;
      if (lane == 0) {
        r[0] = m[h];
        r[1] = l[h];
      }
#pragma unroll
      for (int i = 0; i < EPL / 2; ++i) {
        r[2 + lane * EPL + 2 * i] = acc[h][i].x;
        r[2 + lane * EPL + 2 * i + 1] = acc[h][i].y;
      }
    }
  }
  __syncthreads();
  for (int h = warp; h < NC; h += kTcWarps) {
    float mm = -INFINITY;
    for (int w = 0; w < kTcEpiWarps; ++w) mm = fmaxf(mm, red[((size_t)w * NC + h) * PART]);
    float ll = 0.f, o[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) o[i] = 0.f;
    if (mm != -INFINITY) {
      for (int w = 0; w < kTcEpiWarps; ++w) {
        const float* r = red + ((size_t)w * NC + h) * PART;
        const float f = r[0] == -INFINITY ? 0.f : expf(r[0] - mm);
        ll += r[1] * f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) o[i] += r[2 + lane * EPL + i] * f;
      }
    }
    float* dst = G.partials + (((size_t)unit * G.nsplit_max + split) * NC + h) * PART;
    if (lane == 0) {
      dst[0] = mm;
      dst[1] = ll;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) dst[2 + lane * EPL + i] = o[i];
  }
  if (!finish_split(G.counters + unit, nsplit, misc)) return;
  for (int h = warp; h < NC; h += kTcWarps) {
    if (!cols[h].active) continue;
    float mm = -INFINITY;
    for (int s2 = 0; s2 < nsplit; ++s2)
      mm = fmaxf(mm, __ldcg(G.partials + (((size_t)unit * G.nsplit_max + s2) * NC + h) * PART));
    float ll = 0.f, o[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) o[i] = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const float* r = G.partials + (((size_t)unit * G.nsplit_max + s2) * NC + h) * PART;
      const float rm = __ldcg(r);
      const float f = rm == -INFINITY ? 0.f : expf(rm - mm);
      ll += __ldcg(r + 1) * f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) o[i] += __ldcg(r + 2 + lane * EPL + i) * f;
    }
    const long long ob = cols[h].row * D + lane * EPL;
#pragma unroll
    for (int i = 0; i < EPL; ++i) store_out(G, ob + i, ll > 0.f ? o[i] / ll : 0.f);
  }
}

}  // namespace topo
