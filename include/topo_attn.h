/*
 * topo_attn.h -- C ABI of libtopoattn.so: condensate-set ("topological")
 * attention on one NVIDIA B300 (sm_103a).
 *
 * Method: "The Condensate Theorem: Transformers are O(n), Not O(n^2)"
 * (J. L. Ruiz Williams, arXiv 2602.06317), as restated by the gist.science
 * explainer pages; cited below as [fr S2] = French page, Resume Technique
 * section 2, [ko S3] = Korean page, technical summary section 3, and so on.
 *
 *   [fr S2] / [zh S3]  for each query position i the condensate set is
 *                      C_i = {anchor 0} U {the W most recent positions}
 *                            U {the k positions with the largest q_i . k_j}.
 *   [fr S3]            the softmax is taken over the indices in C_i only.
 *   [ko S3]            q . K^T scores are recomputed at every step to find C_i
 *                      (dynamic selection), so every causal key is scored.
 *   [fr S3] / [ko S2]  the weights left out are claimed to fall below the
 *                      float32 ULP; the optional `excl` output measures them.
 *   [zh S3]            "pillar" layers keep full attention: dense_attn_forward.
 *
 * Readings fixed by this library where the pages are silent:
 *   - query row r of a call sits at absolute position p = n - nq + r and sees
 *     keys 0..p (causal);
 *   - the window is {max(0, p-W+1) .. p} (it includes p);
 *   - top-k candidates are 1 .. p-W; with fewer than k candidates all are
 *     taken;
 *   - ranking uses the float32 score acc = +0; for c in 0..d-1:
 *     acc = fma(q[c], k[c], acc) (one rounding per step), ordered by (score
 *     descending, index ascending): equal scores go to the lower index;
 *   - query head h reads KV head h / (Hq / Hkv).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates nothing.  Its only global mutable state is a small
 *     mutex-guarded cache of launch plans (keyed by the parameters and the
 *     device) and topo_attn_forward_noalloc's fixed scratch array; it is
 *     thread-safe.  Work is enqueued on `stream` (a cudaStream_t, 0 = legacy
 *     default stream) and the call returns without synchronising.
 *   - Layouts are row-major with d fastest:
 *       q    [B, Hq,  nq,        d]  dtype
 *       k, v [B, Hkv, kv_stride, d]  dtype (rows n .. kv_stride-1 are never read)
 *       out  [B, Hq,  nq,        d]  float32
 *       idx  [B, Hq,  nq, 1+W+k]     int32, C_i ascending, padded with -1
 *       excl [B, Hq,  nq]            float32
 *     q, k, v must be 16-byte aligned.
 *   - Return value: TOPO_OK or a negative TOPO_ERR_* code.  Argument errors
 *     are detected on the host before anything is enqueued.  Faults of
 *     kernels already enqueued surface at the caller's next synchronisation,
 *     as usual in CUDA.  Inputs are assumed finite; NaN or Inf inputs give
 *     unspecified (but memory-safe) results.
 *   - Workspace: `ws` is a caller-owned device buffer of at least
 *     topo_attn_workspace_size() (resp. dense_attn_workspace_size()) bytes,
 *     256-byte aligned.  Each call clears the part it needs on `stream`
 *     (one small cudaMemsetAsync), so one workspace may serve calls of any
 *     shapes.  Its first 4 bytes are a sticky device status word (see
 *     topo_attn_device_status): zero them once when the buffer is created,
 *     for instance with topo_attn_workspace_init.  Calls sharing one
 *     workspace must be ordered on one stream.
 */
#ifndef TOPO_ATTN_H
#define TOPO_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */
typedef struct CUstream_st *topo_stream_t;

#define TOPO_KMAX 256 /* largest supported k */

enum {
  TOPO_OK = 0,
  TOPO_ERR_INVALID_ARG = -1,      /* bad shape, null required pointer, misaligned pointer */
  TOPO_ERR_UNSUPPORTED = -2,      /* d, k or dtype outside the supported set */
  TOPO_ERR_WORKSPACE = -3,        /* workspace missing, too small or misaligned */
  TOPO_ERR_CUDA = -4,             /* a CUDA runtime/driver call failed at enqueue time */
  TOPO_ERR_DEVICE_TIMEOUT = -5,   /* a bounded device-side wait gave up (see topo_attn_device_status) */
  TOPO_ERR_SCRATCH_LIMIT = -6,    /* topo_attn_forward_noalloc: the problem needs more scratch than
                                     TOPO_NOALLOC_SCRATCH_BYTES */
  TOPO_ERR_BAD_BLOCK = -7         /* device status only: a block-table entry of
                                     topo_attn_forward_paged was outside the pool */
};

typedef enum { TOPO_F32 = 0, TOPO_BF16 = 1 } topo_dtype;

typedef struct {
  int32_t B;          /* sequences, >= 1 */
  int32_t Hq;         /* query heads, >= 1, multiple of Hkv */
  int32_t Hkv;        /* key/value heads, >= 1 */
  int32_t d;          /* head dimension: 64 or 128 */
  int64_t n;          /* causal length: keys 0..n-1 are valid, >= 1 */
  int64_t nq;         /* query rows per (sequence, head), 1 <= nq <= n */
  int64_t kv_stride;  /* rows allocated per (sequence, KV head) in k and v, >= n */
  int32_t W;          /* window length, >= 1 */
  int32_t k;          /* top-k, 0 <= k <= TOPO_KMAX */
  float scale;        /* logit = scale * (q . k_j); finite */
  int32_t dtype;      /* topo_dtype of q, k, v */
} topo_attn_params;

/* Workspace bytes needed by topo_attn_forward / topo_attn_score_select for
 * these parameters; 0 if the parameters are invalid or unsupported. */
size_t topo_attn_workspace_size(const topo_attn_params *p);

/* Workspace bytes needed by dense_attn_forward; 0 if invalid. */
size_t dense_attn_workspace_size(const topo_attn_params *p);

/* Zero `bytes` of a new workspace on `stream` (cudaMemsetAsync), including
 * its status word. */
int topo_attn_workspace_init(void *ws, size_t bytes, topo_stream_t stream);

/*
 * Condensate-set attention [fr S2-S3]: per query row, score every causal key
 * in float32 (the ranking score above), select C_i, take the softmax over C_i
 * in float32 and write out = sum_j w_j v_j / sum_j w_j.
 *   out  : required.
 *   idx  : optional (NULL to skip): C_i per row.
 *   excl : optional (NULL to skip): the dense-softmax mass outside C_i,
 *          sum_{j <= p, j not in C_i} softmax_j(scale * q . k), computed by a
 *          second pass over K.
 */
int topo_attn_forward(const topo_attn_params *p, const void *q, const void *k, const void *v,
                      float *out, int32_t *idx, float *excl, void *ws, size_t ws_bytes,
                      topo_stream_t stream);

/*
 * Group-shared condensate-set attention for grouped-query attention models
 * (the method is validated on GQA architectures [fr S4]; the pages give no
 * rule for sharing, this is the reading this library takes): one condensate
 * set per (sequence, KV head, query row), shared by the Hq/Hkv query heads
 * that read that KV head.  Its top-k ranks key j by the largest of those
 * heads' float32 ranking scores (ties to the lower index); anchor and window
 * as for topo_attn_forward.  Each head then takes its own float32 softmax
 * over the shared set.  One selection per group instead of per head, and the
 * selected K/V rows are gathered once per group.
 *   out : required, [B, Hq, nq, d] float32.
 *   idx : optional, [B, Hkv, nq, 1+W+k] int32 (one row per group).
 * Workspace: topo_attn_workspace_size(p).  Supported: bf16, Hq/Hkv >= 2,
 * nq * Hq/Hkv <= 16 (<= 4 when k > 32), 1 <= k <= 64 (the tensor-core decode
 * shapes); otherwise TOPO_ERR_UNSUPPORTED.
 */
int topo_attn_forward_grouped(const topo_attn_params *p, const void *q, const void *k,
                              const void *v, float *out, int32_t *idx, void *ws,
                              size_t ws_bytes, topo_stream_t stream);

/*
 * Paged KV cache and output dtype (a serving-shaped boundary for the KV-cache
 * setting of the pages [zh S4]).
 *
 * With block_table != NULL, k_pool and v_pool are pools of fixed-size blocks,
 *     [num_blocks, Hkv, block_size, d]  (dtype of q),
 * and key j of sequence b lives in block block_table[b * max_blocks +
 * j / block_size] at offset j % block_size.  block_size must be a multiple of
 * 128 (so that every 128-key tile the scorer loads lies in one block) and
 * max_blocks * block_size >= n.  Entries outside 0..num_blocks-1 are read as
 * block 0 and reported through the device status word (TOPO_ERR_BAD_BLOCK);
 * no access leaves the pool.  With block_table == NULL, k_pool and v_pool are
 * the usual contiguous [B, Hkv, kv_stride, d] caches.
 * seq_lens (device, optional): the causal length of each sequence (the query
 * rows sit at positions seq_lens[b] - nq + r), clamped to nq..n; NULL: all n.
 * out_bf16 != 0: out is bfloat16 [B, Hq, nq, d] (round to nearest even),
 * else float32.
 */
typedef struct {
  const int32_t *block_table; /* [B, max_blocks] device, or NULL */
  const int32_t *seq_lens;    /* [B] device, or NULL */
  int32_t max_blocks;
  int32_t block_size;
  int32_t num_blocks;
  int32_t out_bf16;
} topo_paged_kv;

/* Workspace bytes for topo_attn_forward_paged; 0 if invalid or unsupported. */
size_t topo_attn_paged_workspace_size(const topo_attn_params *p, const topo_paged_kv *kv);

/*
 * Condensate-set attention (as topo_attn_forward, without the excluded mass)
 * over a paged or contiguous KV cache with per-sequence lengths and a float32
 * or bfloat16 output.  p->n is the largest sequence length (p->kv_stride is
 * read only for a contiguous cache).  Supported on the tensor-core decode
 * shapes: bf16, nq * Hq/Hkv <= 16 (<= 4 when k > 32), 1 <= k <= 64; otherwise
 * TOPO_ERR_UNSUPPORTED.  idx (optional) as for topo_attn_forward.
 */
int topo_attn_forward_paged(const topo_attn_params *p, const topo_paged_kv *kv, const void *q,
                            const void *k_pool, const void *v_pool, void *out, int32_t *idx,
                            void *ws, size_t ws_bytes, topo_stream_t stream);

/* The scoring and selection steps alone [fr S2, ko S3]: writes idx (required). */
int topo_attn_score_select(const topo_attn_params *p, const void *q, const void *k,
                           int32_t *idx, void *ws, size_t ws_bytes, topo_stream_t stream);

/*
 * The softmax-over-the-set step alone [fr S3]: given index rows idx
 * [B, Hq, nq, 1+W+k], writes out.  Entries that are negative or outside
 * 0..p of their row are ignored; every other entry takes part once per
 * occurrence.  A row with no usable entry gets out = 0.  Needs no workspace.
 */
int topo_attn_sparse_softmax_pv(const topo_attn_params *p, const void *q, const void *k,
                                const void *v, const int32_t *idx, float *out,
                                topo_stream_t stream);

/*
 * Condensate KV compaction [zh S4: storing only the condensate set's KV;
 * ko S4 (2): memory saving].  For each query row, gathers the K and V rows
 * its condensate set names into a compact cache:
 *   k_out, v_out [B, Hq, nq, 1+W+k, d]  (dtype of k / v)
 *   k_out[b,h,r,e] = k[b, h/(Hq/Hkv), idx[b,h,r,e]]  for idx >= 0, zero rows
 *   where idx is -1.
 * idx is [B, Hq, nq, 1+W+k] as written by topo_attn_forward /
 * topo_attn_score_select.  The compact cache is exact for these queries:
 * their outputs depend only on these rows, so the softmax over the compact
 * rows (topo_attn_sparse_softmax_pv with entries 0..|C|-1, n = 1+W+k)
 * reproduces them.  It cannot serve other queries: with dynamic top-k a new
 * query may select any earlier key, so the full cache stays the source of
 * truth.  Entries of idx outside 0..n-1 are treated as -1.  Needs no
 * workspace.
 */
int topo_attn_compact_kv(const topo_attn_params *p, const void *k, const void *v,
                         const int32_t *idx, void *k_out, void *v_out, topo_stream_t stream);

/* Dense causal attention over keys 0..p (the full-attention "pillar" layer,
 * [zh S3]); W and k are ignored. */
int dense_attn_forward(const topo_attn_params *p, const void *q, const void *k, const void *v,
                       float *out, void *ws, size_t ws_bytes, topo_stream_t stream);

/*
 * Multi-layer step with layer-adaptive sets and pillar layers [zh S3,
 * "implementation strategy": early layers use wider windows, later layers
 * leaner sets, and a few layers (e.g. L/16) keep full attention so that
 * global information still flows; ko S3, "layer-adaptive configuration"].
 *
 * One topo_layer per layer: that layer's own q, k, v and out (layouts and
 * alignment as for topo_attn_forward), its window W and top-k k, and whether
 * it is a pillar (dense != 0: dense_attn_forward, W and k ignored).
 */
typedef struct {
  const void *q;      /* [B, Hq, nq, d] */
  const void *k;      /* [B, Hkv, kv_stride, d] */
  const void *v;      /* [B, Hkv, kv_stride, d] */
  float *out;         /* [B, Hq, nq, d] float32 */
  int32_t W;          /* window of a sparse layer, >= 1 */
  int32_t k_top;      /* top-k of a sparse layer, 0 <= k_top <= TOPO_KMAX */
  int32_t dense;      /* nonzero: pillar layer (full causal attention) */
  int32_t reserved;   /* set to 0 */
} topo_layer;

/*
 * Fill the W, k_top and dense fields of layers[0..L) with the schedule this
 * library reads from the pages (they fix no numbers beyond "e.g. L/16"):
 *   - layer l is a pillar when pillar_every > 0 and l % pillar_every == 0
 *     (pillar_every = 16 gives L/16 pillars, the first at layer 0);
 *   - the sparse layers take their window from `windows` (n_windows values,
 *     widest first) by depth tier: layer l uses windows[l * n_windows / L];
 *   - every sparse layer uses top-k `k`.
 * Pointers in layers[] are left as they are.  Returns TOPO_ERR_INVALID_ARG for
 * L < 1, n_windows < 1, a window < 1, k outside 0..TOPO_KMAX or pillar_every < 0.
 */
int topo_attn_layer_schedule(int32_t L, int32_t pillar_every, const int32_t *windows,
                             int32_t n_windows, int32_t k, topo_layer *layers);

/* Workspace bytes for topo_attn_layers_forward: the largest need of any
 * layer (layers run one after another on the stream and share it); 0 if
 * any layer is invalid or unsupported. */
size_t topo_attn_layers_workspace_size(const topo_attn_params *p, const topo_layer *layers,
                                       int32_t L);

/*
 * Run L layers in order on `stream`: layer l computes condensate-set
 * attention (topo_attn_forward with its own W and k_top) or, for a pillar,
 * dense causal attention, on its own q, k, v into its own out.  `p` gives the
 * shapes every layer shares (B, Hq, Hkv, d, n, nq, kv_stride, scale, dtype);
 * its W and k are ignored.  Every layer is checked before anything is
 * enqueued, so an argument error enqueues no work.  The layers' inputs are
 * independent here: a model would compute layer l+1's q, k, v from layer l's
 * out between the layers, which is outside this library.
 */
int topo_attn_layers_forward(const topo_attn_params *p, const topo_layer *layers, int32_t L,
                             void *ws, size_t ws_bytes, topo_stream_t stream);

/*
 * topo_attn_forward without a caller-supplied workspace.  (The paper has no
 * counterpart; this is a deployment convenience of this library.)
 *
 * For callers that cannot allocate device memory: plugin hosts that hand an
 * operator only its input and output buffers, and latency-critical serving
 * loops where cudaMalloc is not allowed after start-up because it can
 * synchronise the device.  Same arguments, results and status codes as
 * topo_attn_forward, minus ws / ws_bytes; q, k, v, out (and idx, excl when
 * given) are still the caller's device buffers.
 *
 * Scratch: a fixed array of TOPO_NOALLOC_SCRATCH_BYTES (8 MiB) inside the
 * library's device image.  Every GPU on which the library is used holds it
 * until the process exits.  Problems whose topo_attn_workspace_size exceeds it
 * are rejected with TOPO_ERR_SCRATCH_LIMIT before anything is enqueued (the
 * decode shapes fit; long chunked-prefill calls need the regular entry point).
 * This call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress and caches it.  Make that
 * first call before any stream capture on that device.  The current device
 * must be the one that owns q, k, v and out.  The cached address belongs to
 * the device's primary context: after cudaDeviceReset (which destroys that
 * context) it is stale, so do not use this entry point again in that process.
 *
 * Sharing: every call, on every stream and host thread, uses the same array,
 * which keeps the previous call's contents; each call clears what must start
 * at zero on its own stream.  Calls whose GPU work overlaps (different streams
 * not ordered by events, or concurrent host threads) race on the array and
 * give undefined results: order them on one stream.  The array's device status
 * word cannot be read back through this entry point.
 */
#define TOPO_NOALLOC_SCRATCH_BYTES (8u << 20)
int topo_attn_forward_noalloc(const topo_attn_params *p, const void *q, const void *k,
                              const void *v, float *out, int32_t *idx, float *excl,
                              topo_stream_t stream);

/* Human-readable text of a status code (static storage). */
const char *topo_attn_strerror(int status);

/* Copy the workspace's device status word to *status (TOPO_OK or
 * TOPO_ERR_DEVICE_TIMEOUT) and clear it.  Synchronises `stream`. */
int topo_attn_device_status(void *ws, int *status, topo_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TOPO_ATTN_H */
