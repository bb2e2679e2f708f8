// topo_prefill.cuh -- chunked causal prefill of condensate-set attention on
// the tcgen05 tensor cores (bf16 inputs, many query rows per call).
//
// Method ("The Condensate Theorem" explainer pages, technical summary
// sections 2-3): every query row p selects the anchor 0, the window
// {p-W+1..p} and the top-k of the keys 1..p-W by q . k (re-identified for every
// query, so every causal pair is scored), then takes the softmax over that
// set.  In prefill the scoring of every causal (query, key) pair is a dense
// contraction: it runs on the tensor cores, and the exact float32 ranking
// score (acc = fma(q[c], k[c], acc), c = 0..d-1) is recomputed only for the
// few keys per query that can still be in its top-k.
//
// Kernels of one call (launched in this order by topo_api.cu):
//   prefill_kmax_kernel      largest |k_c| over the causal keys of each KV head
//                            (the scale of the tensor-core rounding bound);
//   prefill_scan_kernel      persistent; one work item = 128 query columns
//                            (query row x head pairs of one KV head) against
//                            all their candidate keys, 256 keys per tile, in
//                            two passes over the same tiles: M = 128 columns
//                            (A: queries, resident in shared memory), N = 256
//                            keys (B: K tile by TMA), the accumulator in TMEM
//                            (two buffers).  Each epilogue thread owns one
//                            column.  Pass 1 offers only the maxima of groups
//                            of keys (whole 128-key halves of a tile for long
//                            items, down to 8-key groups for short ones) to
//                            the column's candidate buffer; their k-th
//                            largest U bounds the column's k-th best
//                            tensor-core score from below (k distinct keys
//                            reach it), so U - 2 delta starts pass 2's cut
//                            (delta: the bound on |tensor core - exact chain|,
//                            see topo_tc_kernels.cuh).  Pass 2 appends every
//                            score above the cut and, when a buffer fills,
//                            compacts that column (its owner thread bisects
//                            over the buffered scores in registers), raising
//                            the cut.  Survivors,
//                            with their tensor-core scores, go to the
//                            workspace;
//   prefill_finalize_kernel  one warp per column: the exact top-k (ties to the
//                            lower position) from the survivors.  Survivors
//                            whose tensor-core score clears the boundary by
//                            2 delta are in without rescoring; the others are
//                            rescored with the exact chain.  Writes the sorted
//                            top-k, C_i (idx) and, when the excluded mass is
//                            requested, the exact k-th key.  A column whose
//                            near ties overflowed its buffer is rescanned
//                            exactly on CUDA cores;
//   prefill_pv_band_kernel   32 consecutive rows of one head share their
//                            window band, staged once in shared memory; per
//                            row the float32 softmax over C_i (band, anchor,
//                            and the top-k with the finalize kernel's exact
//                            logits) and the weighted sum of V;
//   prefill_pv_kernel        the same with one warp per row and rows read from
//                            global memory, when the band does not fit.
#pragma once

#include <cuda_bf16.h>

#include "topo_tc_kernels.cuh"

namespace topo {

constexpr int kPfCols = 128;   // query columns per work item (MMA M)
constexpr int kPfKeys = 256;   // keys per tile (MMA N)
constexpr int kPfSubKeys = 128;  // keys per epilogue step (one TMEM read of a column)
constexpr int kPfCap = 64;     // candidate slots per column
constexpr int kPfSub = 8;      // scores offered between room checks
constexpr int kPfLL = 64;      // survivors published per column
constexpr int kPfStride = kPfCols + 1;  // buffer row stride (entries)
constexpr int kPfEpiWarps = 4; // one per TMEM lane quarter
constexpr int kPfAcc = 2;      // TMEM accumulator buffers (kPfKeys columns each: all 512)
constexpr int kPfWarps = 2 + kPfEpiWarps;  // + TMA producer + MMA issuer
constexpr int kPfThreads = 32 * kPfWarps;

// Shared-memory carve-up of the scan kernel (host and device).
struct PfSmem {
  int ring, qtile, buf, bars, misc, total;
  __host__ __device__ PfSmem(int D, int stages) {
    const int tile = kPfKeys * D * 2;
    int o = 0;
    ring = o;   o += stages * tile;               // multiple of 1024
    qtile = o;  o += kPfCols * D * 2;             // A operand (1024-aligned)
    buf = o;    o += kPfCap * kPfStride * 8;      // (score, position) entries [slot][column]
    bars = o;   o += (2 * stages + 2 * kPfAcc) * 8;  // full, empty, acc_full[], acc_empty[]
    misc = o;   o += 64;
    total = o + 1024;
  }
};

// ------------------------------------------------------------- K scale ----

// kmax[b*Hkv + h] = max over keys 0..n-1 and c of |k_c| (float bits; the
// buffer starts at zero).  grid = (x blocks, B*Hkv), 256 threads.
template <int D>
__global__ void __launch_bounds__(256) prefill_kmax_kernel(const Geom G) {
  const int bh = blockIdx.y;
  const uint4* base = reinterpret_cast<const uint4*>(G.kp) + (long long)bh * G.kv_stride * (D / 8);
  const long long nvec = G.n * (D / 8);
  __nv_bfloat162 m = __floats2bfloat162_rn(0.f, 0.f);
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
       v += (long long)gridDim.x * blockDim.x) {
    const uint4 w = __ldg(base + v);
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.x)));
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.y)));
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.z)));
    m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w.w)));
  }
  float f = warp_max(fmaxf(__low2float(m), __high2float(m)));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = f;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) f = fmaxf(f, red[w]);
    atomicMax(G.kmax + bh, __float_as_uint(f));  // non-negative floats order as integers
  }
}

// ------------------------------------------------------------ scan ---------

// Candidate-buffer state of one column (held by the column's thread).
struct PfState {
  int cnt;    // candidates in the buffer
  float thr;  // scores must exceed this to enter
  int ovf;    // the buffer filled up with near ties
};

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float max8(const float* v) {
  return fmaxf(max3f(v[0], v[1], v[2]), max3f(v[3], v[4], max3f(v[5], v[6], v[7])));
}

// Compact the buffer of column c of this warp.  A bisection on warp-wide
// counts finds U with at least k buffered scores >= U (so U is at most the
// k-th best, within 1/1024 of the buffered range); entries with score >=
// U - 2 delta are kept (in any order) and lane c's count and cut are updated.
// While the column has fewer than k entries everything is kept.  `final`
// never flags overflow.  An entry is (score, position bits).
static __device__ __noinline__ PfState pf_compact(float2* be, int quarter, int lane, int kk,
                                                  int c, float two_delta, PfState st,
                                                  bool final) {
  constexpr int R = (kPfCap + 31) / 32;
  const int cc = quarter * 32 + c;
  const int cnt_c = __shfl_sync(kFull, st.cnt, c);
  const float td = __shfl_sync(kFull, two_delta, c);
  float2 e[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int slot = lane + 32 * r;
    e[r] = slot < cnt_c ? be[slot * kPfStride + cc] : make_float2(-INFINITY, 0.f);
  }
  float cut = -INFINITY;
  if (kk > 0 && cnt_c >= kk) {
    float hi = -INFINITY, lo = INFINITY;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      hi = fmaxf(hi, e[r].x);
      lo = fminf(lo, e[r].x == -INFINITY ? INFINITY : e[r].x);
    }
    hi = warp_max(hi);
    lo = -warp_max(-lo);  // at least k entries are >= lo
#pragma unroll 1
    for (int it = 0; it < 10; ++it) {
      const float mid = 0.5f * (lo + hi);
      int n = 0;
#pragma unroll
      for (int r = 0; r < R; ++r) n += __popc(__ballot_sync(kFull, e[r].x >= mid));
      if (n >= kk) lo = mid;
      else hi = mid;
    }
    cut = lo - td;
  }
  unsigned b[R];
  int keep = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    b[r] = __ballot_sync(kFull, e[r].x != -INFINITY && e[r].x >= cut);
    keep += __popc(b[r]);
  }
  __syncwarp();
  const unsigned below = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (b[r] & (1u << lane)) be[(base + __popc(b[r] & below)) * kPfStride + cc] = e[r];
    base += __popc(b[r]);
  }
  __syncwarp();
  if (lane == c) {
    st.cnt = keep;
    st.thr = fmaxf(st.thr, cut);
    if (!final && keep + kPfSub > kPfCap) {  // the buffer is full of near ties
      st.ovf = 1;
      st.thr = INFINITY;
    }
  }
  return st;
}

// Compact this thread's own column (every lane of the warp at once, no
// cross-lane work): the same bisection as pf_compact on per-lane counts,
// entries >= U - 2 delta kept in place, the cut never lowered.  Columns with
// fewer than max(k, at_least) entries, or already overflowed, are left as
// they are.  A column left with fewer than `room` free slots overflows; with
// `hold` its cut stays finite (appends stop), else the cut becomes +inf.
static __device__ __noinline__ PfState pf_compact_lane(float2* be, int cl, int kk, float two_delta,
                                                       PfState st, int at_least, int room,
                                                       bool hold) {
  const int n = st.cnt;
  if (st.ovf || kk <= 0 || n < kk || n < at_least) return st;
  // the column's scores in registers (absent slots -inf), then the bisection
  float v[kPfCap];
  float lo = INFINITY, hi = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPfCap; ++i) {
    v[i] = i < n ? be[i * kPfStride + cl].x : -INFINITY;
    lo = i < n ? fminf(lo, v[i]) : lo;
    hi = fmaxf(hi, v[i]);
  }
#pragma unroll 1
  for (int it = 0; it < 10; ++it) {
    const float mid = 0.5f * (lo + hi);
    int c = 0;
#pragma unroll
    for (int i = 0; i < kPfCap; ++i) c += v[i] >= mid ? 1 : 0;
    if (c >= kk) lo = mid;
    else hi = mid;
  }
  const float cut = lo - two_delta;
  int w = 0;
  for (int i = 0; i < n; ++i) {  // in place: the write slot never passes the read slot
    const float2 e = be[i * kPfStride + cl];
    be[w * kPfStride + cl] = e;
    w += e.x >= cut ? 1 : 0;
  }
  st.cnt = w;
  st.thr = fmaxf(st.thr, cut);
  if (w + room > kPfCap) {
    st.ovf = 1;
    if (!hold) st.thr = INFINITY;
  }
  return st;
}

// Offer 64 consecutive scores (positions jg..jg+63) of this thread's column,
// given the maxima m[0..7] of their eight 8-score groups: one warp reduction,
// and the append path only for the groups where some column has a
// candidate.  The append writes every score of the group to the next free
// slot and advances the count only past the ones above the cut (no branch,
// one 64-bit store per score); the room check keeps 8 slots free.
__device__ __forceinline__ void pf_offer64(const float (&sa)[32], const float (&sb)[32],
                                           const float* m, long long jg, float2* be,
                                           int quarter, int lane, int cl, int kk,
                                           float two_delta, PfState& st) {
  unsigned lm = 0u;
#pragma unroll
  for (int s = 0; s < 8; ++s) lm |= (m[s] > st.thr) ? (1u << s) : 0u;
  const unsigned wm = __reduce_or_sync(kFull, lm);
  if (wm == 0u) return;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    if (!(wm & (1u << s))) continue;
    unsigned full = __ballot_sync(kFull, !st.ovf && st.cnt + kPfSub > kPfCap);
    while (full) {
      const int c = __ffs(full) - 1;
      full &= full - 1;
      st = pf_compact(be, quarter, lane, kk, c, two_delta, st, false);
    }
    const float* v = s < 4 ? sa + 8 * s : sb + 8 * (s - 4);
    const int j0 = (int)(jg + 8 * s);
    // the group's candidates go to consecutive free slots: the eight compares
    // first, then each slot from a prefix count (independent stores)
    unsigned bits = 0u;
#pragma unroll
    for (int i = 0; i < kPfSub; ++i) bits |= (v[i] > st.thr) ? (1u << i) : 0u;
    if (st.ovf) bits = 0u;
    const int n = st.cnt;
#pragma unroll
    for (int i = 0; i < kPfSub; ++i) {
      if (bits & (1u << i))
        be[(n + __popc(bits & ((1u << i) - 1u))) * kPfStride + cl] =
            make_float2(v[i], __int_as_float(j0 + i));
    }
    const int nn = n + __popc(bits);
    st.cnt = nn;
  }
}

__device__ __forceinline__ float max64(const float (&a)[32], const float (&b)[32]) {
  float m[8];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    m[s] = max8(a + 8 * s);
    m[4 + s] = max8(b + 8 * s);
  }
  return max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_scan_kernel(const __grid_constant__ CUtensorMap map_k, const Geom G) {
  using S = Shape<true, D>;
  constexpr int TILEB = kPfKeys * S::ROWB;
  constexpr int KSTEPS = D / 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int stages = G.stages;
  const int kk = G.topk;

  uint8_t* sm = aligned_smem_base();
  const PfSmem L(D, stages);
  uint8_t* ring = sm + L.ring;
  uint8_t* qtile = sm + L.qtile;
  float2* be = reinterpret_cast<float2*>(sm + L.buf);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + stages;
  uint64_t* accf = empty + stages;
  uint64_t* acce = accf + kPfAcc;
  volatile int* misc = reinterpret_cast<volatile int*>(sm + L.misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L.misc + 32);

  if (tid == 0) {
    misc[0] = 0;  // abort
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kPfAcc; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], kPfEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tslot, kPfAcc * kPfKeys);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  long long seq = 0;     // tiles this CTA has run (phases of the ring and accumulator barriers)
  long long issued = 0;  // tiles the producer has issued (equals seq unless aborted)
  for (;;) {
    __syncthreads();
    if (tid == 0) misc[2] = atomicAdd(G.work, 1);
    __syncthreads();
    const long long item = misc[2];
    if (item >= G.nitems || misc[0]) break;
    // one KV head at a time (its K tiles stay in L2 for the CTAs that share
    // it), the longest blocks (latest rows) of each head first
    const int bh = (int)(item / G.items_per_head);
    const int blk = G.items_per_head - 1 - (int)(item % G.items_per_head);
    const int b = bh / G.Hkv, kvh = bh % G.Hkv;
    const long long c0 = (long long)blk * kPfCols;
    const long long cend = (c0 + kPfCols < G.ncols) ? c0 + kPfCols : G.ncols;
    const long long r_last = (cend - 1) / G.g;
    const long long jmax = G.n - G.nq + r_last - G.W;
    const int ntiles = jmax >= 1 ? (int)((jmax + kPfKeys - 1) / kPfKeys) : 0;
    const long long kvrow0 = ((long long)b * G.Hkv + kvh) * G.kv_stride;

    // queries of the block: bf16, K-major, 128-byte swizzle; missing columns zero
    for (int i = tid; i < kPfCols * (D / 8); i += blockDim.x) {
      const int r = i / (D / 8), v = i % (D / 8);
      const long long col = c0 + r;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (col < cend) {
        const long long rr = col / G.g;
        const int hh = (int)(col % G.g);
        const long long qrow = ((long long)b * G.Hq + (long long)kvh * G.g + hh) * G.nq + rr;
        w = __ldg(reinterpret_cast<const uint4*>(G.qp) + qrow * (D / 8) + v);
      }
      *reinterpret_cast<uint4*>(qtile + (v >> 3) * (kPfCols * 128) + r * 128 +
                                (((v & 7) ^ (r & 7)) << 4)) = w;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    if (warp == 0) {
      // ---------------- TMA producer ----------------------------------------
      if (lane == 0) {
        if (ntiles > 0) prefetch_tmap(&map_k);
        // ring slot and round of tile seq + t, advanced without a division per tile
        int s = (int)(seq % stages);
        uint32_t round = (uint32_t)(seq / stages);
        for (int t = 0; t < 2 * ntiles; ++t, s = (s + 1 == stages) ? 0 : s + 1,
                 round += (s == 0) ? 1u : 0u) {
          if (misc[0]) break;
          if (!mbar_wait(&empty[s], (round & 1u) ^ 1u)) {
            set_status(G.status, kStatusTimeout);
            misc[0] = 1;
            break;
          }
          uint8_t* dst = ring + (size_t)s * TILEB;
          mbar_arrive_expect_tx(&full[s], (uint32_t)TILEB);
          ++issued;
          const int tt = t < ntiles ? t : t - ntiles;  // both passes run the same tiles
          const int y = (int)(kvrow0 + 1 + (long long)tt * kPfKeys);
#pragma unroll
          for (int cc = 0; cc < S::NCH; ++cc)
            tma_load_2d(dst + cc * (kPfKeys * 128), &map_k, cc * S::EPC, y, &full[s]);
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer --------------------------------------------
      if (lane == 0) {
        constexpr uint32_t idesc = tc::idesc_bf16_f32(kPfCols, kPfKeys);
        // descriptors of the A operand and of ring slot 0; a 16-byte step of the
        // start address is +1 in the descriptor's low field (addresses < 256 KB)
        const uint64_t adesc = tc::smem_desc_sw128(smem_addr(qtile));
        const uint64_t bdesc0 = tc::smem_desc_sw128(smem_addr(ring));
        int s = (int)(seq % stages);
        uint32_t round = (uint32_t)(seq / stages);
        for (int t = 0; t < 2 * ntiles; ++t, s = (s + 1 == stages) ? 0 : s + 1,
                 round += (s == 0) ? 1u : 0u) {
          if (misc[0]) break;
          const long long gs = seq + t;
          const int ab = (int)(gs % kPfAcc);
          const uint32_t around = (uint32_t)(gs / kPfAcc);
          if (!mbar_wait(&acce[ab], (around & 1u) ^ 1u) || !mbar_wait(&full[s], round & 1u)) {
            set_status(G.status, kStatusTimeout);
            misc[0] = 1;
            break;
          }
          tc::fence_after_sync();
          const uint64_t bdesc = bdesc0 + (uint64_t)((s * TILEB) >> 4);
          const uint32_t dt = tmem + (uint32_t)(ab * kPfKeys);
#pragma unroll
          for (int ks16 = 0; ks16 < KSTEPS; ++ks16) {
            const uint32_t offa = ((ks16 >> 2) * (kPfCols * 128) + (ks16 & 3) * 32) >> 4;
            const uint32_t offb = ((ks16 >> 2) * (kPfKeys * 128) + (ks16 & 3) * 32) >> 4;
            tc::mma_bf16(dt, adesc + offa, bdesc + offb, idesc, ks16 > 0);
          }
          tc::mma_commit(&empty[s]);  // the K stage is free once these MMAs are done
          tc::mma_commit(&accf[ab]);
        }
      }
    } else {
      // ---------------- epilogue: one column per thread -----------------------
      const int quarter = warp & 3;
      const int cl = quarter * 32 + lane;
      const long long col = c0 + cl;
      const bool active = col < cend;
      const long long pos = G.n - G.nq + (active ? col / G.g : 0);
      const long long jhi = active ? pos - G.W : 0;
      float qn1 = 0.f;  // ||q||_1 of this column
#pragma unroll 4
      for (int v = 0; v < D / 8; ++v) {
        const uint4 w = *reinterpret_cast<const uint4*>(qtile + (v >> 3) * (kPfCols * 128) +
                                                        cl * 128 + (((v & 7) ^ (cl & 7)) << 4));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          qn1 += fabsf(__uint_as_float(u[q] << 16)) + fabsf(__uint_as_float(u[q] & 0xffff0000u));
      }
      const float kmx = __uint_as_float(G.kmax[bh]);
      const float two_delta = 2.f * tc_delta_factor(D) * qn1 * 1.001f * kmx;
      PfState st{0, -INFINITY, 0};
      // pass-1 values per 128 keys: enough group maxima (>= 4k) per column
      int vpt = 1;
      while (vpt < 16 && vpt * ntiles * (kPfKeys / kPfSubKeys) < 4 * kk) vpt <<= 1;
      const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
      for (int t = 0; t < 2 * ntiles; ++t) {
        const bool p1 = t < ntiles;
        if (t == ntiles) {
          // U from the pass-1 group maxima (k distinct keys reach it)
          st = pf_compact_lane(be, cl, kk, two_delta, st, 0, 0, true);
          st.cnt = 0;
          st.ovf = 0;
        }
        const long long gs = seq + t;
        const int ab = (int)(gs % kPfAcc);
        const uint32_t around = (uint32_t)(gs / kPfAcc);
        const bool ok = __all_sync(kFull, mbar_wait(&accf[ab], around & 1u));
        if (!ok || misc[0]) {
          if (!ok && lane == 0) {
            set_status(G.status, kStatusTimeout);
            misc[0] = 1;
          }
          break;
        }
        tc::fence_after_sync();
        const int tt = p1 ? t : t - ntiles;
#pragma unroll 1
        for (int sub = 0; sub < kPfKeys / kPfSubKeys; ++sub) {
          const long long js = 1 + (long long)tt * kPfKeys + sub * kPfSubKeys;
          // 128 scores of this column in registers; after the last read of the
          // tile the accumulator goes straight back to the MMA issuer
          float sa[32], sb[32], sc[32], sd[32];
          {
            const uint32_t ta = tq + (uint32_t)(ab * kPfKeys + sub * kPfSubKeys);
            tc::tmem_ld16(ta, *reinterpret_cast<float(*)[16]>(sa));
            tc::tmem_ld16(ta + 16, *reinterpret_cast<float(*)[16]>(sa + 16));
            tc::tmem_ld16(ta + 32, *reinterpret_cast<float(*)[16]>(sb));
            tc::tmem_ld16(ta + 48, *reinterpret_cast<float(*)[16]>(sb + 16));
            tc::tmem_ld16(ta + 64, *reinterpret_cast<float(*)[16]>(sc));
            tc::tmem_ld16(ta + 80, *reinterpret_cast<float(*)[16]>(sc + 16));
            tc::tmem_ld16(ta + 96, *reinterpret_cast<float(*)[16]>(sd));
            tc::tmem_ld16(ta + 112, *reinterpret_cast<float(*)[16]>(sd + 16));
            tc::tmem_ld_wait();
            if (sub == kPfKeys / kPfSubKeys - 1) {
              tc::fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acce[ab]);
            }
          }
          if (js + kPfSubKeys - 1 > jhi) {  // keys past the column's last candidate
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (js + i > jhi) sa[i] = -INFINITY;
              if (js + 32 + i > jhi) sb[i] = -INFINITY;
              if (js + 64 + i > jhi) sc[i] = -INFINITY;
              if (js + 96 + i > jhi) sd[i] = -INFINITY;
            }
          }
          // the maxima of the sixteen 8-score groups (independent)
          float m[16];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            m[g] = max8(sa + 8 * g);
            m[4 + g] = max8(sb + 8 * g);
            m[8 + g] = max8(sc + 8 * g);
            m[12 + g] = max8(sd + 8 * g);
          }
          if (p1) {
            // the maxima of 128 / vpt-key groups (distinct keys), offered to
            // the buffer; their kk-th largest bounds the column's kk-th best
            float gm[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) gm[i] = m[i];
#pragma unroll
            for (int l = 0; l < 4; ++l) {
              if ((16 >> l) > vpt) {
#pragma unroll
                for (int i = 0; i < (8 >> l); ++i) gm[i] = fmaxf(gm[2 * i], gm[2 * i + 1]);
              }
            }
            if (__any_sync(kFull, !st.ovf && st.cnt + vpt > kPfCap))
              st = pf_compact_lane(be, cl, kk, two_delta, st, 0, vpt, true);
            if (!st.ovf) {
              int n = st.cnt;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                if (i < vpt) {
                  be[n * kPfStride + cl] = make_float2(gm[i], __int_as_float((int)js));
                  n += gm[i] > st.thr ? 1 : 0;
                }
              }
              st.cnt = n;
            }
            continue;
          }
          // one vote: most steps hold no candidate for any column of the warp
          const float mt = fmaxf(max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]),
                                       max3f(m[6], m[7], m[8])),
                                 max3f(max3f(m[9], m[10], m[11]), max3f(m[12], m[13], m[14]),
                                       m[15]));
          if (__any_sync(kFull, mt > st.thr)) {
            pf_offer64(sa, sb, m, js, be, quarter, lane, cl, kk, two_delta, st);
            pf_offer64(sc, sd, m + 8, js + 64, be, quarter, lane, cl, kk, two_delta, st);
          }
        }
      }
      // survivors of each column (any order) to the workspace
      if (__any_sync(kFull, !st.ovf && st.cnt > kPfLL))
        st = pf_compact_lane(be, cl, kk, two_delta, st, kPfLL + 1, 0, false);
#pragma unroll 1
      for (int c = 0; c < 32; ++c) {
        const int cc = quarter * 32 + c;
        if (c0 + cc >= cend) break;
        const int cnt_c = __shfl_sync(kFull, st.cnt, c);
        const bool ov_c = __shfl_sync(kFull, st.ovf, c) != 0;
        const long long gcol = (long long)bh * G.ncols + c0 + cc;
        float2* dst = G.surv + gcol * kPfLL;
        const bool ovl = ov_c || cnt_c > kPfLL;  // more survivors than slots: exact rescan
#pragma unroll
        for (int r = 0; r < kPfLL / 32; ++r) {
          const int ee = lane + 32 * r;
          if (ee < cnt_c) dst[ee] = be[ee * kPfStride + cc];  // (tensor-core score, position)
        }
        if (lane == 0) G.surv_cnt[gcol] = ovl ? -1 : cnt_c;
      }
    }
    seq += 2 * ntiles;
  }

  // no copy into shared memory and no MMA may outlive the CTA: the producer
  // waits (bounded) for the last ring fills it issued
  if (warp == 0 && lane == 0) {
    for (long long gs = issued - 1; gs >= 0 && gs >= issued - stages; --gs) {
      if (!mbar_wait(&empty[gs % stages], (uint32_t)(gs / stages) & 1u))
        set_status(G.status, kStatusTimeout);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kPfAcc * kPfKeys);
  }
}

// ------------------------------------------------------------ finalize -----

// The float32 chain (acc = fma(q[c], k[c], acc), c = 0..D-1) of two bf16 key
// rows against one query held as floats in shared memory; every load of both
// rows is issued before the arithmetic, and the two chains are independent.
template <int D>
__device__ __forceinline__ void score_two_rows(const void* kbase, long long ra, long long rb,
                                               const float* q, float& sa, float& sb) {
  constexpr int NV = D / 8;  // 16-byte vectors per row
  const uint4* pa = reinterpret_cast<const uint4*>(kbase) + ra * NV;
  const uint4* pb = reinterpret_cast<const uint4*>(kbase) + rb * NV;
  uint4 wa[NV], wb[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    wa[v] = __ldg(pa + v);
    wb[v] = __ldg(pb + v);
  }
  const float4* q4 = reinterpret_cast<const float4*>(q);
  float a = 0.f, b = 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float4 qq = q4[v * 2 + h];
      a = fmaf(qq.x, chunk_elem<true>(wa[v], 4 * h + 0), a);
      b = fmaf(qq.x, chunk_elem<true>(wb[v], 4 * h + 0), b);
      a = fmaf(qq.y, chunk_elem<true>(wa[v], 4 * h + 1), a);
      b = fmaf(qq.y, chunk_elem<true>(wb[v], 4 * h + 1), b);
      a = fmaf(qq.z, chunk_elem<true>(wa[v], 4 * h + 2), a);
      b = fmaf(qq.z, chunk_elem<true>(wb[v], 4 * h + 2), b);
      a = fmaf(qq.w, chunk_elem<true>(wa[v], 4 * h + 3), a);
      b = fmaf(qq.w, chunk_elem<true>(wb[v], 4 * h + 3), b);
    }
  }
  sa = a;
  sb = b;
}

// One warp per column (= per output row): exact top-k from the survivors,
// then the sorted top-k positions, C_i and the k-th key.  4 warps per block.
// At least 12 CTAs per SM (<= 40 registers): each warp is a chain of dependent
// global loads, so occupancy hides the latency (44.65 -> 44.37 ms per 64K
// prefill at W = 64).
template <int D>
__global__ void __launch_bounds__(128, 12) prefill_finalize_kernel(const Geom G) {
  __shared__ __align__(16) float qs[4][D];
  __shared__ uint64_t scratch[4][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gcol = (long long)blockIdx.x * 4 + warp;
  const long long total = (long long)G.B * G.Hkv * G.ncols;
  if (gcol >= total) return;
  const int kk = G.topk;
  const long long bh = gcol / G.ncols, col = gcol % G.ncols;
  const int b = (int)(bh / G.Hkv), kvh = (int)(bh % G.Hkv);
  const long long rr = col / G.g;
  const int hh = (int)(col % G.g);
  const long long row = ((long long)b * G.Hq + (long long)kvh * G.g + hh) * G.nq + rr;
  const long long p = G.n - G.nq + rr;
  const long long jhi = p - G.W;
  const long long kvrow0 = ((long long)b * G.Hkv + kvh) * G.kv_stride;
  for (int c = lane; c < D; c += 32) qs[warp][c] = load_elem<true>(G.qp, row * D + c);
  __syncwarp();
  const int cnt = G.surv_cnt[gcol];
  uint64_t x0;
  if (cnt >= 0 && (cnt <= kk || G.thr)) {
    // every survivor is selected, or the exact k-th key is needed (for the
    // excluded mass): all survivors through the exact chain; a lane's two
    // rows are loaded up front and their chains interleaved (independent)
    uint64_t x[2];
    {
      const float2 e0 = lane < cnt ? G.surv[gcol * kPfLL + lane] : make_float2(0.f, 0.f);
      const float2 e1 = lane + 32 < cnt ? G.surv[gcol * kPfLL + lane + 32] : make_float2(0.f, 0.f);
      const uint32_t j0 = (uint32_t)__float_as_int(e0.y), j1 = (uint32_t)__float_as_int(e1.y);
      float s0, s1;
      score_two_rows<D>(G.kp, kvrow0 + j0, kvrow0 + j1, qs[warp], s0, s1);
      x[0] = lane < cnt ? rank_key(s0, j0) : 0ull;
      x[1] = lane + 32 < cnt ? rank_key(s1, j1) : 0ull;
    }
    warp_sort_desc<2>(x, lane);
    x0 = x[0];
  } else if (cnt >= 0) {
    // More survivors than k.  A bisection on the tensor-core scores t finds V
    // with fewer than k survivors at t >= V.  A survivor with t > V + 2 delta
    // is in the exact top-k without rescoring: any key that beats it exactly
    // has t > V (|t - exact| <= delta), every key with t > V is a survivor,
    // and fewer than k of them exist.  Only the other survivors (near the
    // boundary, typically a handful) are rescored with the exact chain, and
    // the best of them fill the remaining slots.
    const float2 e0 = lane < cnt ? G.surv[gcol * kPfLL + lane] : make_float2(-INFINITY, 0.f);
    const float2 e1 = lane + 32 < cnt ? G.surv[gcol * kPfLL + lane + 32]
                                      : make_float2(-INFINITY, 0.f);
    float lo = warp_max(-fminf(e0.x == -INFINITY ? INFINITY : e0.x,
                               e1.x == -INFINITY ? INFINITY : e1.x));
    lo = -lo;  // smallest t: kk <= cnt survivors are >= it
    float hi = warp_max(fmaxf(e0.x, e1.x));
    hi = hi + fabsf(hi) * 1e-6f + 1e-30f;  // no survivor is >= it
#pragma unroll 1
    for (int it = 0; it < 16; ++it) {
      const float mid = 0.5f * (lo + hi);
      const int c = __popc(__ballot_sync(kFull, e0.x >= mid)) +
                    __popc(__ballot_sync(kFull, e1.x >= mid));
      if (c >= kk) lo = mid;
      else hi = mid;
    }
    float qn1 = 0.f;
    for (int c = lane; c < D; c += 32) qn1 += fabsf(qs[warp][c]);  // the bf16 inputs, exactly
    qn1 = warp_sum(qn1);
    const float two_delta =
        2.f * tc_delta_factor(D) * qn1 * 1.01f * __uint_as_float(G.kmax[bh]);
    const float V = hi + two_delta;
    const bool c0 = e0.x > V, c1 = e1.x > V;                  // certain
    const bool u0 = lane < cnt && !c0, u1 = lane + 32 < cnt && !c1;  // to rescore
    const unsigned bc0 = __ballot_sync(kFull, c0), bc1 = __ballot_sync(kFull, c1);
    const unsigned bu0 = __ballot_sync(kFull, u0), bu1 = __ballot_sync(kFull, u1);
    const int m = __popc(bc0) + __popc(bc1);  // < kk
    const int u = __popc(bu0) + __popc(bu1);  // >= kk - m
    const unsigned below = (1u << lane) - 1u;
    uint64_t* sb = scratch[warp];
    if (c0) sb[__popc(bc0 & below)] = rank_key(e0.x, (uint32_t)__float_as_int(e0.y));
    if (c1) sb[__popc(bc0) + __popc(bc1 & below)] = rank_key(e1.x, (uint32_t)__float_as_int(e1.y));
    if (u0) sb[64 + __popc(bu0 & below)] = (uint64_t)(uint32_t)__float_as_int(e0.y);
    if (u1) sb[64 + __popc(bu0) + __popc(bu1 & below)] = (uint64_t)(uint32_t)__float_as_int(e1.y);
    __syncwarp();
    uint64_t x[2] = {0ull, 0ull};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = lane + 32 * r;
      if (i < u) {
        const uint32_t j = (uint32_t)sb[64 + i];
        x[r] = rank_key(score_row_q4<true, D>(G.kp, kvrow0 + j, qs[warp]), j);
      }
    }
    if (u > 32) {
      warp_sort_desc<2>(x, lane);
    } else {
      uint64_t y1[1] = {x[0]};
      warp_sort_desc<1>(y1, lane);
      x[0] = y1[0];
    }
    const uint64_t unc = __shfl_sync(kFull, x[0], (lane - m) & 31);
    uint64_t cer = lane < m ? sb[lane] : 0ull;
    if (lane < m && G.toplogit) {
      // a certain key's exact score (its logit in the softmax; the selection
      // did not need it)
      const uint32_t j = key_pos(sb[lane]);
      cer = rank_key(score_row_q4<true, D>(G.kp, kvrow0 + j, qs[warp]), j);
    }
    x0 = lane < m ? cer : unc;  // lanes < k: the selected set (not in exact order)
  } else {
    // the near ties overflowed: every candidate through the exact chain
    uint64_t fthr = 0ull;
    int fcnt = 0;
    uint64_t* sb = scratch[warp];
    for (long long j0 = 1; j0 <= jhi; j0 += 32) {
      const long long j = j0 + lane;
      const uint64_t key =
          j <= jhi ? rank_key(score_row_q4<true, D>(G.kp, kvrow0 + j, qs[warp]), (uint32_t)j)
                   : 0ull;
      offer<4, 1>(sb, fthr, fcnt, key, kk, lane);
    }
    __syncwarp();
    uint64_t y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = e * 32 + lane;
      y[e] = i < fcnt ? sb[i] : 0ull;
    }
    warp_sort_desc<4>(y, lane);
    x0 = y[0];
  }
  // x0 at lane i is the i-th best (k <= 32)
  const uint64_t mine = lane < kk ? x0 : 0ull;
  const int t = __popc(__ballot_sync(kFull, mine != 0ull));
  if (G.thr) {
    const uint64_t kth = __shfl_sync(kFull, x0, (kk > 0 ? kk - 1 : 0) & 31);
    if (lane == 0) {
      const long long cb = col / G.thr_nc;
      const int slot = (int)(col % G.thr_nc);
      const long long unit = bh * G.ncb + cb;
      G.thr[(size_t)unit * G.thr_nc + slot] = kk == 0 ? ~0ull : (t < kk ? 0ull : kth);
    }
  }
  // selected positions ascending, each with its exact score
  uint64_t y = mine ? (((uint64_t)(0xffffffffu - key_pos(mine)) << 32) |
                       __float_as_uint(key_score(mine)))
                    : 0ull;
  {
    uint64_t ya[1] = {y};
    warp_sort_desc<1>(ya, lane);
    y = ya[0];
  }
  const int tj = y ? (int)(0xffffffffu - (uint32_t)(y >> 32)) : -1;
  if (lane < kk) {
    G.topsel[row * kk + lane] = tj;
    if (G.toplogit) G.toplogit[row * kk + lane] = y ? G.scale * __uint_as_float((uint32_t)y) : 0.f;
  }
  if (G.idx) {
    const long long cmax = 1 + (long long)G.W + kk;
    const bool wide = p - G.W + 1 <= 0;
    const long long mEnt = wide ? p + 1 : 1 + t + G.W;
    const long long wlo = p - G.W + 1;
    int* dst = G.idx + row * cmax;
    for (long long e0 = 0; e0 < cmax; e0 += 32) {
      const long long e = e0 + lane;
      const int from_top = __shfl_sync(kFull, tj, (int)((e - 1) & 31));
      long long v = -1;
      if (e < mEnt) {
        if (wide) v = e;
        else if (e == 0) v = 0;
        else if (e <= t) v = from_top;
        else v = wlo + (e - 1 - t);
      }
      if (e < cmax) dst[e] = (int)v;
    }
  }
}

// ------------------------------------------------------------ softmax ------

// One warp per row: softmax over C_i = {0} U top-k U window and the weighted
// sum of V (4 rows per block).
template <int D>
__global__ void __launch_bounds__(128) prefill_pv_kernel(const Geom G) {
  __shared__ __align__(16) float qs[4][D];
  __shared__ float wsm[4][256];
  __shared__ int jsm[4][256];
  __shared__ int tsm[4][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + warp;
  const long long nrows = (long long)G.B * G.Hq * G.nq;
  if (row >= nrows) return;
  const int kk = G.topk;
  const long long r = row % G.nq;
  const int h = (int)((row / G.nq) % G.Hq);
  const int b = (int)(row / (G.nq * G.Hq));
  const int kvh = h / G.g;
  const long long p = G.n - G.nq + r;
  const long long kvrow0 = ((long long)b * G.Hkv + kvh) * G.kv_stride;
  for (int c = lane; c < D; c += 32) qs[warp][c] = load_elem<true>(G.qp, row * D + c);
  const int tj = lane < kk ? G.topsel[row * kk + lane] : -1;
  tsm[warp][lane] = tj;
  const int t = __popc(__ballot_sync(kFull, tj >= 0));
  __syncwarp();
  const bool wide = p - G.W + 1 <= 0;
  const long long mEnt = wide ? p + 1 : 1 + t + G.W;
  const long long wlo = p - G.W + 1;
  const int* top = tsm[warp];
  auto entry = [&](long long e) -> long long {
    if (wide) return e;
    if (e == 0) return 0;
    if (e <= t) return top[e - 1];
    return wlo + (e - 1 - t);
  };
  const float* qw = qs[warp];
  warp_softmax_pv_with<true, D>(
      G, [&](long long j) { return kvrow0 + j; },
      [&](long long kr) { return score_row_q4<true, D>(G.kp, kr, qw); }, mEnt, entry, wsm[warp],
      jsm[warp], row * D, lane);
}

// ------------------------------------------------------- banded softmax ----
//
// The softmax over C_i and the weighted sum of V for a block of kPbRows
// consecutive rows of every query head of one KV head.  Their windows all lie
// in the band [p0 - W + 1, p0 + kPbRows - 1] (p0: the block's first
// position), whose K and V rows are staged in shared memory once and shared
// by the block's g * kPbRows (row, head) pairs.  A warp takes four rows of one
// head at a time, so every staged row it reads serves four rows.  The anchor's
// rows are staged too.  The top-k entries' logits come from the finalize step
// (scale times the exact float32 score); only their V rows are gathered from
// global memory.  Logits of window keys are float32 dot products of the
// bf16 inputs; the softmax and the sums are float32.
constexpr int kPbRows = 32;   // rows per block (per query head)
constexpr int kPbWarps = 8;
constexpr int kPbUnit = 4;    // rows per warp step

// Shared-memory carve-up of the banded kernel (host and device).  Staged rows
// are padded by 16 bytes so that consecutive rows start four banks apart.
struct PbSmem {
  int kb, vb, k0, v0, q, lw, bars, total;
  __host__ __device__ PbSmem(int D, int W) {
    const int rowb = D * 2 + 16;
    const int nb = W + kPbRows - 1;
    const int wb = W + kPbUnit - 1;
    int o = 0;
    kb = o; o += nb * rowb;
    vb = o; o += nb * rowb;
    k0 = o; o += rowb;
    v0 = o; o += rowb;
    q = o;  o += kPbWarps * kPbUnit * D * 4;                 // float q rows per warp
    lw = o; o += kPbWarps * kPbUnit * ((wb + 3) & ~3) * 4;   // window logits / weights
    bars = o; o += 16;
    total = o + 16;
  }
};

template <int D>
__global__ void __launch_bounds__(kPbWarps * 32, 1) prefill_pv_band_kernel(const Geom G) {
  using S = Shape<true, D>;
  constexpr int ROWP = S::ROWB + 16;  // staged row pitch
  constexpr int EPL = D / 32;         // output elements per lane
  extern __shared__ __align__(16) uint8_t pb_raw[];
  uint8_t* sm = pb_raw + ((16u - (smem_addr(pb_raw) & 15u)) & 15u);
  const PbSmem L(D, G.W);
  uint8_t* kb = sm + L.kb;
  uint8_t* vb = sm + L.vb;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kk = G.topk;
  const int W = G.W;
  const int wb = W + kPbUnit - 1;
  const int wbp = (wb + 3) & ~3;
  float* qw = reinterpret_cast<float*>(sm + L.q) + warp * kPbUnit * D;
  float* lw = reinterpret_cast<float*>(sm + L.lw) + warp * kPbUnit * wbp;

  const int b = blockIdx.z, kvh = blockIdx.y;
  const long long r0 = (long long)blockIdx.x * kPbRows;  // first row of the block
  const long long rend = r0 + kPbRows < G.nq ? r0 + kPbRows : G.nq;
  const long long p0 = G.n - G.nq + r0;
  const long long band_lo = p0 - W + 1 > 0 ? p0 - W + 1 : 0;
  const long long band_hi = G.n - G.nq + rend - 1;
  const int nb = (int)(band_hi - band_lo + 1);
  const long long kvrow0 = ((long long)b * G.Hkv + kvh) * G.kv_stride;
  const uint8_t* kg = reinterpret_cast<const uint8_t*>(G.kp);
  const uint8_t* vg = reinterpret_cast<const uint8_t*>(G.vp);

  // stage the band and the anchor (bulk copies completing on one barrier)
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) mbar_arrive_expect_tx(bar, (uint32_t)((nb + 1) * 2 * S::ROWB));
  for (int i = tid; i <= nb; i += blockDim.x) {
    const long long row = i < nb ? band_lo + i : 0;
    uint8_t* dk = i < nb ? kb + (size_t)i * ROWP : sm + L.k0;
    uint8_t* dv = i < nb ? vb + (size_t)i * ROWP : sm + L.v0;
    bulk_copy_g2s(dk, kg + (kvrow0 + row) * S::ROWB, S::ROWB, bar);
    bulk_copy_g2s(dv, vg + (kvrow0 + row) * S::ROWB, S::ROWB, bar);
  }
  const bool staged = mbar_wait(bar, 0);
  if (!staged && tid == 0) set_status(G.status, kStatusTimeout);
  if (__syncthreads_or(!staged)) return;

  const int units = G.g * kPbRows / kPbUnit;
  for (int u = warp; u < units; u += kPbWarps) {
    const int hh = u / (kPbRows / kPbUnit);
    const long long ru = r0 + (long long)(u % (kPbRows / kPbUnit)) * kPbUnit;  // first row
    if (ru >= rend) continue;
    const int nr = (int)(rend - ru < kPbUnit ? rend - ru : kPbUnit);
    const int h = kvh * G.g + hh;
    const long long rowbase = ((long long)b * G.Hq + h) * G.nq;
    const long long pu = G.n - G.nq + ru;  // position of the unit's first row
    __syncwarp();
    for (int i = lane; i < kPbUnit * D; i += 32) {
      const int r = i / D, c = i % D;
      qw[i] = r < nr ? load_elem<true>(G.qp, (rowbase + ru + r) * D + c) : 0.f;
    }
    // top-k entries of the unit's rows (lane i: entry i of each row)
    int tp[kPbUnit];
    float tl[kPbUnit];
#pragma unroll
    for (int r = 0; r < kPbUnit; ++r) {
      tp[r] = -1;
      tl[r] = -INFINITY;
      if (r < nr && lane < kk) {
        const long long row = rowbase + ru + r;
        tp[r] = G.topsel[row * kk + lane];
        if (tp[r] >= 0) tl[r] = G.toplogit[row * kk + lane];
      }
    }
    __syncwarp();
    // window logits: the union of the rows' windows [jlo, pu + nr - 1]
    const long long jlo = pu - W + 1 > 0 ? pu - W + 1 : 0;
    const int nw = (int)(pu + nr - 1 - jlo + 1);
    float mx[kPbUnit];
#pragma unroll
    for (int r = 0; r < kPbUnit; ++r) mx[r] = -INFINITY;
    // two keys per lane at a time (e and e + 32), every query load serving
    // both; the dot products run as paired FMAs over (even, odd) elements
    // (softmax logits only: the selection is already made, so the two halves
    // may be added at the end)
    for (int e0 = 0; e0 < nw; e0 += 64) {
      const int ea = e0 + lane, eb = e0 + 32 + lane;
      const bool va = ea < nw, vbk = eb < nw;
      const uint4* kra = reinterpret_cast<const uint4*>(kb + (size_t)(jlo + (va ? ea : 0) - band_lo) * ROWP);
      const uint4* krb = reinterpret_cast<const uint4*>(kb + (size_t)(jlo + (vbk ? eb : 0) - band_lo) * ROWP);
      float2 a2[kPbUnit], b2[kPbUnit];
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r) {
        a2[r] = make_float2(0.f, 0.f);
        b2[r] = make_float2(0.f, 0.f);
      }
#pragma unroll 2
      for (int v = 0; v < S::ROWB / 16; ++v) {
        const uint4 wa4 = kra[v], wb4 = krb[v];
        const uint32_t ua[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
        const uint32_t ub[4] = {wb4.x, wb4.y, wb4.z, wb4.w};
        float2 xa[4], xb[4];  // elements (2i, 2i+1) of the two rows
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xa[i] = make_float2(__uint_as_float(ua[i] << 16), __uint_as_float(ua[i] & 0xffff0000u));
          xb[i] = make_float2(__uint_as_float(ub[i] << 16), __uint_as_float(ub[i] & 0xffff0000u));
        }
#pragma unroll
        for (int r = 0; r < kPbUnit; ++r) {
          const float4* q4 = reinterpret_cast<const float4*>(qw + r * D + v * 8);
          const float4 qa = q4[0], qb = q4[1];
          const float2 qp[4] = {make_float2(qa.x, qa.y), make_float2(qa.z, qa.w),
                                make_float2(qb.x, qb.y), make_float2(qb.z, qb.w)};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a2[r] = __ffma2_rn(qp[i], xa[i], a2[r]);
            b2[r] = __ffma2_rn(qp[i], xb[i], b2[r]);
          }
        }
      }
      float aa[kPbUnit], ab[kPbUnit];
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r) {
        aa[r] = a2[r].x + a2[r].y;
        ab[r] = b2[r].x + b2[r].y;
      }
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r) {
        const long long p = pu + r;
        const long long ja = jlo + ea, jb = jlo + eb;
        const bool ina = va && r < nr && ja <= p && ja >= p - W + 1;
        const bool inb = vbk && r < nr && jb <= p && jb >= p - W + 1;
        const float la = ina ? G.scale * aa[r] : -INFINITY;
        const float lb = inb ? G.scale * ab[r] : -INFINITY;
        if (va) lw[r * wbp + ea] = la;
        if (vbk) lw[r * wbp + eb] = lb;
        mx[r] = fmaxf(mx[r], fmaxf(la, lb));
      }
    }
    // anchor logit of rows whose window does not reach position 0
    float la[kPbUnit];
    {
      float pa[kPbUnit];
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r) pa[r] = 0.f;
      const uint32_t* k0w = reinterpret_cast<const uint32_t*>(sm + L.k0);
      for (int c2 = lane; c2 < D / 2; c2 += 32) {
        const uint32_t wv = k0w[c2];
        const float ka = __uint_as_float(wv << 16), kb2 = __uint_as_float(wv & 0xffff0000u);
#pragma unroll
        for (int r = 0; r < kPbUnit; ++r)
          pa[r] = fmaf(qw[r * D + 2 * c2 + 1], kb2, fmaf(qw[r * D + 2 * c2], ka, pa[r]));
      }
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r) {
        const float sa = warp_sum(pa[r]);
        const bool sep = r < nr && pu + r - W + 1 > 0;  // anchor outside the window
        la[r] = sep ? G.scale * sa : -INFINITY;
        mx[r] = fmaxf(fmaxf(mx[r], la[r]), tl[r]);
      }
    }
    float z[kPbUnit], tw[kPbUnit], wa[kPbUnit];
#pragma unroll
    for (int r = 0; r < kPbUnit; ++r) {
      mx[r] = warp_max(mx[r]);
      tw[r] = tl[r] == -INFINITY ? 0.f : expf(tl[r] - mx[r]);
      wa[r] = la[r] == -INFINITY ? 0.f : expf(la[r] - mx[r]);
      z[r] = tw[r] + (lane == 0 ? wa[r] : 0.f);
    }
    __syncwarp();
    for (int e = lane; e < nw; e += 32) {
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r) {
        const float l = lw[r * wbp + e];
        const float w = l == -INFINITY ? 0.f : expf(l - mx[r]);
        lw[r * wbp + e] = w;
        z[r] += w;
      }
    }
#pragma unroll
    for (int r = 0; r < kPbUnit; ++r) z[r] = warp_sum(z[r]);
    __syncwarp();
    // weighted sums: lane owns output elements lane*EPL ..
    float acc[kPbUnit][EPL];
    {
      float va[EPL];
      lane_elems<true, D>(sm + L.v0 + lane * S::BPL, va);
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r) {
        const float w0 = __shfl_sync(kFull, wa[r], 0);
#pragma unroll
        for (int x = 0; x < EPL; ++x) acc[r][x] = w0 * va[x];
      }
    }
    {
      static_assert(EPL % 2 == 0, "element pairs per lane");
      float2 acc2[kPbUnit][EPL / 2];
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r)
#pragma unroll
        for (int x = 0; x < EPL / 2; ++x) acc2[r][x] = make_float2(acc[r][2 * x], acc[r][2 * x + 1]);
#pragma unroll 2
      for (int e = 0; e < nw; ++e) {
        float vv[EPL];
        lane_elems<true, D>(vb + (size_t)(jlo + e - band_lo) * ROWP + lane * S::BPL, vv);
#pragma unroll
        for (int r = 0; r < kPbUnit; ++r) {
          const float w = lw[r * wbp + e];
#pragma unroll
          for (int x = 0; x < EPL / 2; ++x)
            acc2[r][x] = __ffma2_rn(make_float2(w, w), make_float2(vv[2 * x], vv[2 * x + 1]),
                                    acc2[r][x]);
        }
      }
#pragma unroll
      for (int r = 0; r < kPbUnit; ++r)
#pragma unroll
        for (int x = 0; x < EPL / 2; ++x) {
          acc[r][2 * x] = acc2[r][x].x;
          acc[r][2 * x + 1] = acc2[r][x].y;
        }
    }
#pragma unroll
    for (int r = 0; r < kPbUnit; ++r) {
      const int t = __popc(__ballot_sync(kFull, tp[r] >= 0));
      // the gathered V rows, eight loads in flight per lane
      int i = 0;
      for (; i + 8 <= t; i += 8) {
        float vv[8][EPL];
        float ww[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = __shfl_sync(kFull, tp[r], i + q);
          ww[q] = __shfl_sync(kFull, tw[r], i + q);
          lane_elems<true, D>(vg + (kvrow0 + j) * S::ROWB + lane * S::BPL, vv[q]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int x = 0; x < EPL; ++x) acc[r][x] = fmaf(ww[q], vv[q][x], acc[r][x]);
      }
      for (; i < t; ++i) {
        const int j = __shfl_sync(kFull, tp[r], i);
        const float w = __shfl_sync(kFull, tw[r], i);
        float vv[EPL];
        lane_elems<true, D>(vg + (kvrow0 + j) * S::ROWB + lane * S::BPL, vv);
#pragma unroll
        for (int x = 0; x < EPL; ++x) acc[r][x] = fmaf(w, vv[x], acc[r][x]);
      }
      if (r < nr) {
        float* o = G.out + (rowbase + ru + r) * D + lane * EPL;
#pragma unroll
        for (int x = 0; x < EPL; ++x) o[x] = z[r] > 0.f ? acc[r][x] / z[r] : 0.f;
      }
    }
  }
}

}  // namespace topo
