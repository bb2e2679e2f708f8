"""Condensate-set ("topological") attention on one B300: Python binding.

A thin ctypes layer over ``libtopoattn.so`` (C ABI in ``include/topo_attn.h``).
It only marshals arguments: shapes are read off torch tensors, outputs and
the workspace are allocated with torch on the tensors' device, and the current
torch stream is passed down.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback.  If the library
is missing, every call raises.

Method ("The Condensate Theorem: Transformers are O(n), Not O(n^2)",
gist.science explainers of arXiv 2602.06317, technical summary sections 2-3):
for query position p the condensate set is {0} + {max(0, p-W+1)..p} + the top-k
of the positions 1..p-W by q . k (float32 score, ties to the lower position);
the output is the softmax-weighted sum of V over that set.

Layouts: q [B, Hq, nq, d]; k, v [B, Hkv, kv_stride, d] (float32 or bfloat16,
contiguous, on CUDA); query row r sits at position n - nq + r.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = ["forward", "forward_grouped", "forward_noalloc", "score_select", "sparse_softmax_pv",
           "dense_forward", "compact_kv", "forward_paged",
           "layer_schedule", "layers_forward", "Workspace", "TopoError", "library_path",
           "load_library", "workspace_size", "dense_workspace_size", "device_status", "EXPORTS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libtopoattn.so")
_lock = threading.Lock()
_lib = None

# every entry point the header declares
EXPORTS = ("topo_attn_workspace_size", "dense_attn_workspace_size", "topo_attn_workspace_init",
           "topo_attn_forward", "topo_attn_score_select", "topo_attn_sparse_softmax_pv",
           "dense_attn_forward", "topo_attn_strerror", "topo_attn_device_status",
           "topo_attn_forward_noalloc", "topo_attn_layer_schedule",
           "topo_attn_layers_workspace_size", "topo_attn_layers_forward",
           "topo_attn_forward_grouped", "topo_attn_compact_kv", "topo_attn_paged_workspace_size",
           "topo_attn_forward_paged")

TOPO_OK = 0
TOPO_KMAX = 256


class TopoError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_strerror(status)} (status {status})")


class Params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n", ctypes.c_int64), ("nq", ctypes.c_int64),
                ("kv_stride", ctypes.c_int64), ("W", ctypes.c_int32), ("k", ctypes.c_int32),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


class PagedKV(ctypes.Structure):
    """topo_paged_kv (include/topo_attn.h)."""
    _fields_ = [("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("max_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("out_bf16", ctypes.c_int32)]


class TopoLayer(ctypes.Structure):
    """One layer of topo_attn_layers_forward (include/topo_attn.h)."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("W", ctypes.c_int32), ("k_top", ctypes.c_int32),
                ("dense", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def library_path() -> str:
    return _SO


def load_library():
    """Load libtopoattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_SO):
            raise RuntimeError(f"{_SO} is missing: build it with "
                               "`python -m dynamic_sparse_transformer_qk_b300.build`")
        lib = ctypes.CDLL(_SO)
        P = ctypes.POINTER(Params)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        sig = {
            "topo_attn_workspace_size": (sz, [P]),
            "dense_attn_workspace_size": (sz, [P]),
            "topo_attn_workspace_init": (i, [vp, sz, vp]),
            "topo_attn_forward": (i, [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "topo_attn_score_select": (i, [P, vp, vp, vp, vp, sz, vp]),
            "topo_attn_sparse_softmax_pv": (i, [P, vp, vp, vp, vp, vp, vp]),
            "dense_attn_forward": (i, [P, vp, vp, vp, vp, vp, sz, vp]),
            "topo_attn_strerror": (ctypes.c_char_p, [i]),
            "topo_attn_device_status": (i, [vp, ctypes.POINTER(ctypes.c_int), vp]),
            "topo_attn_forward_noalloc": (i, [P, vp, vp, vp, vp, vp, vp, vp]),
            "topo_attn_layer_schedule": (i, [ctypes.c_int32, ctypes.c_int32, vp, ctypes.c_int32,
                                             ctypes.c_int32, vp]),
            "topo_attn_layers_workspace_size": (sz, [P, vp, ctypes.c_int32]),
            "topo_attn_layers_forward": (i, [P, vp, ctypes.c_int32, vp, sz, vp]),
            "topo_attn_forward_grouped": (i, [P, vp, vp, vp, vp, vp, vp, sz, vp]),
            "topo_attn_compact_kv": (i, [P, vp, vp, vp, vp, vp, vp]),
            "topo_attn_paged_workspace_size": (sz, [P, vp]),
            "topo_attn_forward_paged": (i, [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _strerror(status: int) -> str:
    try:
        return load_library().topo_attn_strerror(status).decode()
    except Exception:  # library not loadable: still say something
        return "status"


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def make_params(q: torch.Tensor, k: torch.Tensor, *, W: int, topk: int, n: int | None = None,
                scale: float | None = None) -> Params:
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, Hq, nq, d] and k [B, Hkv, kv_stride, d]")
    B, Hq, nq, d = q.shape
    Bk, Hkv, stride, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} vs k {tuple(k.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Params(B, Hq, Hkv, d, stride if n is None else n, nq, stride, W, topk, scale,
                  _dtype_code(q))


def _check(*ts: torch.Tensor):
    dev = ts[0].device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for t in ts:
        if t.device != dev or not t.is_contiguous():
            raise ValueError("tensors must be contiguous and on one device")
        if t.dtype != ts[0].dtype:
            raise ValueError("q, k, v must share one dtype")


def _stream(stream, device=None) -> int:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


_ws_sizes: dict = {}


def _params_key(p: Params) -> tuple:
    return (p.B, p.Hq, p.Hkv, p.d, p.n, p.nq, p.kv_stride, p.W, p.k, p.scale, p.dtype)


def workspace_size(p: Params) -> int:
    key = _params_key(p)
    need = _ws_sizes.get(key)
    if need is None:
        need = _ws_sizes[key] = int(load_library().topo_attn_workspace_size(ctypes.byref(p)))
    return need


def dense_workspace_size(p: Params) -> int:
    return int(load_library().dense_attn_workspace_size(ctypes.byref(p)))


class Workspace:
    """A device buffer the library uses for scratch (split lists, counters).

    It starts zeroed (which clears the sticky status word); each call clears
    the counters it needs, so one Workspace can serve any number of
    stream-ordered calls of any shapes."""

    def __init__(self, device=None, nbytes: int = 0):
        self.device = torch.device(device or "cuda")
        self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes: int) -> "Workspace":
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


_default_ws: dict = {}


def _workspace(ws: Workspace | None, device, nbytes: int, stream) -> Workspace:
    if ws is None:
        key = (device, _stream(stream, device))
        ws = _default_ws.get(key)
        if ws is None:
            ws = _default_ws[key] = Workspace(device, nbytes)
    return ws.ensure(nbytes)


def _raise(rc: int, what: str):
    if rc != TOPO_OK:
        raise TopoError(rc, what)


def forward(q, k, v, *, W: int, topk: int, n: int | None = None, scale: float | None = None,
            want_idx: bool = False, want_excl: bool = False, out=None, idx=None, excl=None,
            workspace: Workspace | None = None, stream=None):
    """Condensate-set attention.  Returns (out, idx or None, excl or None)."""
    _check(q, k, v)
    lib = load_library()
    p = make_params(q, k, W=W, topk=topk, n=n, scale=scale)
    B, Hq, nq, d = q.shape
    if out is None:
        out = torch.empty((B, Hq, nq, d), dtype=torch.float32, device=q.device)
    if want_idx and idx is None:
        idx = torch.empty((B, Hq, nq, 1 + W + topk), dtype=torch.int32, device=q.device)
    if want_excl and excl is None:
        excl = torch.empty((B, Hq, nq), dtype=torch.float32, device=q.device)
    need = workspace_size(p)
    if need == 0:
        _raise(-1 if p.d in (64, 128) else -2, "topo_attn_workspace_size")
    ws = _workspace(workspace, q.device, need, stream)
    with torch.cuda.device(q.device):
        rc = lib.topo_attn_forward(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   out.data_ptr(), idx.data_ptr() if idx is not None else None,
                                   excl.data_ptr() if excl is not None else None, ws.ptr,
                                   ws.nbytes, _stream(stream, q.device))
    _raise(rc, "topo_attn_forward")
    return out, idx, excl


def forward_grouped(q, k, v, *, W: int, topk: int, n: int | None = None,
                    scale: float | None = None, want_idx: bool = False, out=None, idx=None,
                    workspace: Workspace | None = None, stream=None):
    """Group-shared condensate-set attention: one set per (sequence, KV head,
    row) shared by the KV head's query heads (top-k by the largest of their
    scores).  Returns (out [B, Hq, nq, d], idx [B, Hkv, nq, 1+W+k] or None)."""
    _check(q, k, v)
    lib = load_library()
    p = make_params(q, k, W=W, topk=topk, n=n, scale=scale)
    B, Hq, nq, d = q.shape
    if out is None:
        out = torch.empty((B, Hq, nq, d), dtype=torch.float32, device=q.device)
    if want_idx and idx is None:
        idx = torch.empty((B, k.shape[1], nq, 1 + W + topk), dtype=torch.int32, device=q.device)
    need = workspace_size(p)
    if need == 0:
        _raise(-1 if p.d in (64, 128) else -2, "topo_attn_workspace_size")
    ws = _workspace(workspace, q.device, need, stream)
    with torch.cuda.device(q.device):
        rc = lib.topo_attn_forward_grouped(ctypes.byref(p), q.data_ptr(), k.data_ptr(),
                                           v.data_ptr(), out.data_ptr(),
                                           idx.data_ptr() if idx is not None else None,
                                           ws.ptr, ws.nbytes, _stream(stream, q.device))
    _raise(rc, "topo_attn_forward_grouped")
    return out, idx


def score_select(q, k, *, W: int, topk: int, n: int | None = None, scale: float | None = None,
                 idx=None, workspace: Workspace | None = None, stream=None):
    """The condensate sets alone: int32 [B, Hq, nq, 1+W+k], ascending, -1 padded."""
    _check(q, k)
    lib = load_library()
    p = make_params(q, k, W=W, topk=topk, n=n, scale=scale)
    B, Hq, nq, _ = q.shape
    if idx is None:
        idx = torch.empty((B, Hq, nq, 1 + W + topk), dtype=torch.int32, device=q.device)
    need = workspace_size(p)
    if need == 0:
        _raise(-1 if p.d in (64, 128) else -2, "topo_attn_workspace_size")
    ws = _workspace(workspace, q.device, need, stream)
    with torch.cuda.device(q.device):
        rc = lib.topo_attn_score_select(ctypes.byref(p), q.data_ptr(), k.data_ptr(),
                                        idx.data_ptr(), ws.ptr, ws.nbytes,
                                        _stream(stream, q.device))
    _raise(rc, "topo_attn_score_select")
    return idx


def sparse_softmax_pv(q, k, v, idx, *, W: int, topk: int, n: int | None = None,
                      scale: float | None = None, out=None, stream=None):
    """Softmax over given index rows idx [B, Hq, nq, 1+W+k] and the weighted sum of V."""
    _check(q, k, v)
    lib = load_library()
    p = make_params(q, k, W=W, topk=topk, n=n, scale=scale)
    B, Hq, nq, d = q.shape
    if idx.dtype != torch.int32 or tuple(idx.shape) != (B, Hq, nq, 1 + W + topk) \
            or not idx.is_contiguous() or idx.device != q.device:
        raise ValueError("idx must be contiguous int32 [B, Hq, nq, 1+W+k] on q's device")
    if out is None:
        out = torch.empty((B, Hq, nq, d), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.topo_attn_sparse_softmax_pv(ctypes.byref(p), q.data_ptr(), k.data_ptr(),
                                             v.data_ptr(), idx.data_ptr(), out.data_ptr(),
                                             _stream(stream, q.device))
    _raise(rc, "topo_attn_sparse_softmax_pv")
    return out


def compact_kv(k, v, idx, *, Hq: int, n: int | None = None, k_out=None, v_out=None,
               stream=None):
    """topo_attn_compact_kv: the K and V rows each query row's condensate set
    names (idx [B, Hq, nq, 1+W+k]), gathered into [B, Hq, nq, 1+W+k, d]
    (zero rows for -1 entries).  W and k are read off idx: pass the same n."""
    _check(k, v)
    lib = load_library()
    B, Hkv, stride, d = k.shape
    if idx.dtype != torch.int32 or idx.dim() != 4 or idx.shape[0] != B or idx.shape[1] != Hq \
            or not idx.is_contiguous() or idx.device != k.device:
        raise ValueError("idx must be contiguous int32 [B, Hq, nq, 1+W+k] on k's device")
    nq, cmax = idx.shape[2], idx.shape[3]
    # only the row length 1 + W + k matters here
    p = Params(B, Hq, Hkv, d, stride if n is None else n, nq, stride, cmax - 1, 0, 1.0,
               _dtype_code(k))
    if k_out is None:
        k_out = torch.empty((B, Hq, nq, cmax, d), dtype=k.dtype, device=k.device)
    if v_out is None:
        v_out = torch.empty((B, Hq, nq, cmax, d), dtype=v.dtype, device=v.device)
    with torch.cuda.device(k.device):
        rc = lib.topo_attn_compact_kv(ctypes.byref(p), k.data_ptr(), v.data_ptr(),
                                      idx.data_ptr(), k_out.data_ptr(), v_out.data_ptr(),
                                      _stream(stream, k.device))
    _raise(rc, "topo_attn_compact_kv")
    return k_out, v_out


def forward_paged(q, k_pool, v_pool, *, W: int, topk: int, n: int, block_table=None,
                  seq_lens=None, block_size: int = 0, scale: float | None = None,
                  out_bf16: bool = False, want_idx: bool = False, out=None, idx=None,
                  workspace: Workspace | None = None, stream=None):
    """topo_attn_forward_paged: condensate-set attention over a paged KV cache
    (k_pool, v_pool [num_blocks, Hkv, block_size, d] with block_table
    [B, max_blocks] int32) or a contiguous one (block_table None), with
    optional per-sequence lengths seq_lens [B] int32 and a bf16 or float32
    output.  n: the largest sequence length.  Returns (out, idx or None)."""
    _check(q, k_pool, v_pool)
    lib = load_library()
    B, Hq, nq, d = q.shape
    Hkv = k_pool.shape[1]
    paged = block_table is not None
    kv = PagedKV(None, None, 0, 0, 0, int(out_bf16))
    if paged:
        if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
                or not block_table.is_contiguous() or block_table.device != q.device:
            raise ValueError("block_table must be contiguous int32 [B, max_blocks] on q's device")
        kv.block_table = block_table.data_ptr()
        kv.max_blocks = block_table.shape[1]
        kv.block_size = block_size or k_pool.shape[2]
        kv.num_blocks = k_pool.shape[0]
        stride = n
    else:
        stride = k_pool.shape[2]
    if seq_lens is not None:
        if seq_lens.dtype != torch.int32 or seq_lens.numel() != B or seq_lens.device != q.device:
            raise ValueError("seq_lens must be int32 [B] on q's device")
        kv.seq_lens = seq_lens.data_ptr()
    p = Params(B, Hq, Hkv, d, n, nq, stride, W, topk,
               scale if scale is not None else 1.0 / math.sqrt(d), _dtype_code(q))
    if out is None:
        out = torch.empty((B, Hq, nq, d), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                          device=q.device)
    if want_idx and idx is None:
        idx = torch.empty((B, Hq, nq, 1 + W + topk), dtype=torch.int32, device=q.device)
    need = int(lib.topo_attn_paged_workspace_size(ctypes.byref(p), ctypes.byref(kv)))
    if need == 0:
        _raise(-2, "topo_attn_paged_workspace_size")
    ws = _workspace(workspace, q.device, need, stream)
    with torch.cuda.device(q.device):
        rc = lib.topo_attn_forward_paged(ctypes.byref(p), ctypes.byref(kv), q.data_ptr(),
                                         k_pool.data_ptr(), v_pool.data_ptr(), out.data_ptr(),
                                         idx.data_ptr() if idx is not None else None, ws.ptr,
                                         ws.nbytes, _stream(stream, q.device))
    _raise(rc, "topo_attn_forward_paged")
    return out, idx


def dense_forward(q, k, v, *, n: int | None = None, scale: float | None = None, out=None,
                  workspace: Workspace | None = None, stream=None):
    """Dense causal attention over keys 0..p (the full-attention layer)."""
    _check(q, k, v)
    lib = load_library()
    p = make_params(q, k, W=1, topk=0, n=n, scale=scale)
    B, Hq, nq, d = q.shape
    if out is None:
        out = torch.empty((B, Hq, nq, d), dtype=torch.float32, device=q.device)
    need = dense_workspace_size(p)
    if need == 0:
        _raise(-1 if p.d in (64, 128) else -2, "dense_attn_workspace_size")
    ws = _workspace(workspace, q.device, need, stream)
    with torch.cuda.device(q.device):
        rc = lib.dense_attn_forward(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                    out.data_ptr(), ws.ptr, ws.nbytes, _stream(stream, q.device))
    _raise(rc, "dense_attn_forward")
    return out


def forward_noalloc(q, k, v, *, W: int, topk: int, n: int | None = None,
                    scale: float | None = None, out=None, idx=None, excl=None, stream=None):
    """topo_attn_forward_noalloc: like forward() but the library uses its own
    fixed device scratch array instead of a workspace.  out / idx / excl are
    allocated here only when not given; pass them to allocate nothing at all.
    Calls must not overlap on the GPU (they share the array)."""
    _check(q, k, v)
    lib = load_library()
    p = make_params(q, k, W=W, topk=topk, n=n, scale=scale)
    B, Hq, nq, d = q.shape
    if out is None:
        out = torch.empty((B, Hq, nq, d), dtype=torch.float32, device=q.device)
    # the library looks up its scratch array on the current device: make it q's
    with torch.cuda.device(q.device):
        rc = lib.topo_attn_forward_noalloc(ctypes.byref(p), q.data_ptr(), k.data_ptr(),
                                           v.data_ptr(), out.data_ptr(),
                                           idx.data_ptr() if idx is not None else None,
                                           excl.data_ptr() if excl is not None else None,
                                           _stream(stream, q.device))
    _raise(rc, "topo_attn_forward_noalloc")
    return out, idx, excl


def layer_schedule(L: int, *, pillar_every: int = 16, windows=(256, 128, 64),
                   topk: int = 32) -> list:
    """The per-layer settings topo_attn_layer_schedule assigns: a list of L
    dicts {"W", "topk", "dense"} (pillar layers every `pillar_every` layers
    from layer 0; sparse layers take `windows` by depth tier, widest first)."""
    lib = load_library()
    arr = (TopoLayer * L)() if L > 0 else None
    win = (ctypes.c_int32 * len(windows))(*windows)
    rc = lib.topo_attn_layer_schedule(L, pillar_every, ctypes.addressof(win), len(windows),
                                      topk, ctypes.addressof(arr) if arr is not None else None)
    _raise(rc, "topo_attn_layer_schedule")
    return [{"W": a.W, "topk": a.k_top, "dense": bool(a.dense)} for a in arr]


def layers_forward(qs, ks, vs, schedule, *, n: int | None = None, scale: float | None = None,
                   outs=None, workspace: Workspace | None = None, stream=None):
    """topo_attn_layers_forward: layer l attends with its own q, k, v and
    schedule[l] (a dict as from layer_schedule); returns the list of outputs."""
    L = len(schedule)
    if not (len(qs) == len(ks) == len(vs) == L) or L < 1:
        raise ValueError("one q, k, v and schedule entry per layer")
    for q, k, v in zip(qs, ks, vs):
        _check(q, k, v)
        if q.shape != qs[0].shape or k.shape != ks[0].shape or v.shape != ks[0].shape \
                or q.dtype != qs[0].dtype or q.device != qs[0].device:
            raise ValueError("every layer must have the same shapes, dtype and device")
    lib = load_library()
    q0 = qs[0]
    p = make_params(q0, ks[0], W=1, topk=0, n=n, scale=scale)
    B, Hq, nq, d = q0.shape
    if outs is None:
        outs = [torch.empty((B, Hq, nq, d), dtype=torch.float32, device=q0.device)
                for _ in range(L)]
    arr = (TopoLayer * L)()
    for a, q, k, v, o, sch in zip(arr, qs, ks, vs, outs, schedule):
        a.q, a.k, a.v, a.out = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
        a.W, a.k_top, a.dense, a.reserved = int(sch["W"]), int(sch["topk"]), int(sch["dense"]), 0
    need = int(lib.topo_attn_layers_workspace_size(ctypes.byref(p), ctypes.addressof(arr), L))
    if need == 0:
        _raise(-1 if p.d in (64, 128) else -2, "topo_attn_layers_workspace_size")
    ws = _workspace(workspace, q0.device, need, stream)
    with torch.cuda.device(q0.device):
        rc = lib.topo_attn_layers_forward(ctypes.byref(p), ctypes.addressof(arr), L, ws.ptr,
                                          ws.nbytes, _stream(stream, q0.device))
    _raise(rc, "topo_attn_layers_forward")
    return outs


def device_status(ws: Workspace, stream=None) -> int:
    """Read and clear the workspace's device status word (synchronises)."""
    st = ctypes.c_int(0)
    with torch.cuda.device(ws.device):
        rc = load_library().topo_attn_device_status(ws.ptr, ctypes.byref(st),
                                                    _stream(stream, ws.device))
    _raise(rc, "topo_attn_device_status")
    return st.value
