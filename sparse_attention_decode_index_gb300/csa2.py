"""Python binding of libcsa2.so (ctypes).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Functions take torch CUDA tensors (PyTorch supplies
device memory and streams) and mirror the C entry points of ``csa2.h``
without the ``csa2_`` prefix.  The library is loaded on first use and a
missing build raises immediately; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcsa2.so")

FULL, REINDEX, REUSE, SWA = 0, 1, 2, 3
BF16, F32 = 0, 1

OK = 0
STATUS = {0: "CSA2_OK", -1: "CSA2_ERR_INVALID_ARG", -2: "CSA2_ERR_UNSUPPORTED", -3: "CSA2_ERR_WORKSPACE",
          -4: "CSA2_ERR_CUDA", -5: "CSA2_ERR_DEVICE_CHECK", -6: "CSA2_ERR_TIMEOUT"}


class CSA2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_str(status)})")


class CShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_entries", ctypes.c_int32), ("idx_heads", ctypes.c_int32),
                ("idx_dim", ctypes.c_int32), ("block", ctypes.c_int32), ("pool_blocks", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("q_heads", ctypes.c_int32), ("k_dim", ctypes.c_int32),
                ("v_dim", ctypes.c_int32), ("swa", ctypes.c_int32), ("scale", ctypes.c_float),
                ("relu", ctypes.c_int32), ("dtype", ctypes.c_int32), ("tokens", ctypes.c_int32)]


class CLayer(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("hier", ctypes.c_int32), ("q", ctypes.c_void_p),
                ("q_idx", ctypes.c_void_p), ("w_idx", ctypes.c_void_p), ("k_swa", ctypes.c_void_p),
                ("v_swa", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("idx_out", ctypes.c_void_p)]


_lib = None
_VP, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_SIGS = {
    "csa2_workspace_bytes": (_SZ, [ctypes.POINTER(CShape)]),
    "csa2_workspace_init": (ctypes.c_int, [_VP, _SZ, _VP]),
    "csa2_block_keys": (ctypes.c_int, [ctypes.POINTER(CShape), _VP, _VP, _I32, _VP, _VP, _SZ, _VP]),
    "csa2_kv_append": (ctypes.c_int, [ctypes.POINTER(CShape), _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                      _I32, _VP, _SZ, _VP]),
    "csa2_swa_append": (ctypes.c_int, [ctypes.POINTER(CShape), ctypes.c_void_p, _I32, _VP, _VP, _VP, _SZ, _VP]),
    "csa2_index_blocks": (ctypes.c_int, [ctypes.POINTER(CShape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "csa2_index_tokens": (ctypes.c_int, [ctypes.POINTER(CShape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                         _VP, _SZ, _VP]),
    "csa2_index_topk": (ctypes.c_int, [ctypes.POINTER(CShape), _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP,
                                       _SZ, _VP]),
    "csa2_topk": (ctypes.c_int, [ctypes.POINTER(CShape), _VP, _I32, _VP, _VP, _I32, _VP, _VP, _VP, _SZ, _VP]),
    "csa2_sparse_attn": (ctypes.c_int, [ctypes.POINTER(CShape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                        _VP, _SZ, _VP]),
    "csa2_layer_group": (ctypes.c_int, [ctypes.POINTER(CShape), ctypes.POINTER(CLayer), _I32, _VP, _VP, _VP,
                                        _VP, _VP, _VP, _VP, _SZ, _VP]),
    "csa2_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "csa2_read_device_error": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(_I32)]),
    "csa2_fast_path": (ctypes.c_int, [ctypes.POINTER(CShape), ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "csa2_launch_count": (ctypes.c_ulonglong, []),
    "csa2_layer_group_static": (ctypes.c_int, [ctypes.POINTER(CShape), ctypes.POINTER(CLayer), _I32, _VP, _VP,
                                               _VP, _VP, _VP, _VP, _VP]),
    "csa2_read_static_device_error": (ctypes.c_int, [_VP, ctypes.POINTER(_I32)]),
    "csa2_shard_slice": (ctypes.c_int, [_VP, _I32, _I32, _I32, _I32, _I32, _VP, _I32, _VP, _VP, _SZ, _VP]),
    "csa2_shard_counts": (ctypes.c_int, [_VP, _I32, _I32, _I32, _I32, _VP, _VP]),
    "csa2_concat_parts": (ctypes.c_int, [_I32, _I32, _I32, _VP, _VP, _VP, _VP, _VP]),
    "csa2_merge_attn": (ctypes.c_int, [_I32, _I32, _I32, _VP, _VP, _VP, _VP, _VP]),
    "csa2_debug_wait_timeout": (ctypes.c_int, [ctypes.POINTER(CShape), _VP, _VP, _VP, _VP, _I32, _VP, ctypes.c_uint32,
                                               _VP, _SZ, _VP]),
}


def lib() -> ctypes.CDLL:
    """Load libcsa2.so (built in-tree); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -m sparse_attention_decode_index_gb300.build` "
                               "(or __graft_entry__.build()); the CSA2 path has no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols() -> Sequence[str]:
    return list(_SIGS)


def status_str(code: int) -> str:
    try:
        return lib().csa2_status_str(int(code)).decode()
    except RuntimeError:
        return STATUS.get(code, "unknown")


# ------------------------------------------------------------------ marshalling helpers

def c_shape(shape) -> CShape:
    """Build the C shape from any object with the csa2_shape fields (e.g. workloads.Shape)."""
    dt = getattr(shape, "dtype", "bf16")
    dt = {"bf16": BF16, "f32": F32}.get(dt, dt)
    return CShape(int(shape.batch), int(shape.n_entries), int(shape.idx_heads), int(shape.idx_dim),
                  int(shape.block), int(shape.pool_blocks), int(shape.topk), int(shape.q_heads),
                  int(shape.k_dim), int(shape.v_dim), int(shape.swa), float(getattr(shape, "scale", 0.0)),
                  int(getattr(shape, "relu", 1)), int(dt), int(getattr(shape, "tokens", 1)))


def elem_dtype(shape) -> torch.dtype:
    return torch.float32 if getattr(shape, "dtype", "bf16") in ("f32", F32) else torch.bfloat16


def _ptr(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None, name: str = "tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library takes device pointers)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ws(ws):
    """(pointer, bytes) of a workspace; None passes no workspace (NULL, 0)."""
    if ws is None:
        return None, 0
    return _ptr(ws, torch.uint8, "ws"), ws.numel()


def _check(status: int, what: str):
    if status != OK:
        raise CSA2Error(status, what)


# ------------------------------------------------------------------ entry points

def workspace_bytes(shape) -> int:
    s = c_shape(shape)
    n = lib().csa2_workspace_bytes(ctypes.byref(s))
    if n == 0:
        raise CSA2Error(-1, "csa2_workspace_bytes")
    return int(n)


def workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().csa2_workspace_init(_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)),
           "csa2_workspace_init")


def workspace(shape, device=None, stream=None) -> torch.Tensor:
    """Allocate (with torch) and initialise a workspace for ``shape``."""
    ws = torch.empty(workspace_bytes(shape), dtype=torch.uint8, device=device or "cuda")
    workspace_init(ws, stream)
    return ws


def block_keys(shape, k_idx, n_valid, kb, ws, round_to_int: bool = True, stream=None):
    """Block summary keys into kb.  ``ws`` may be None: device errors then go to the
    static scratch's error word (read_static_device_error)."""
    s = c_shape(shape)
    e = elem_dtype(shape)
    _check(lib().csa2_block_keys(ctypes.byref(s), _ptr(k_idx, e, "k_idx"), _ptr(n_valid, torch.int32, "n_valid"),
                                 int(bool(round_to_int)), _ptr(kb, e, "kb"), *_ws(ws), _stream(stream)),
           "csa2_block_keys")


def kv_append(shape, n_new, k_new, v_new, kidx_new, k_main, v_main, k_idx, kb, n_valid, ws,
              round_to_int: bool = True, stream=None):
    """Append n_new[b] compressed entries per query (rows of k_new / v_new / kidx_new, shaped
    [B, max_new, ...]) at n_valid[b]; recompute the touched block keys (kb may be None); grow n_valid."""
    s = c_shape(shape)
    e = elem_dtype(shape)
    max_new = int(k_new.shape[1]) if k_new is not None else 0
    _check(lib().csa2_kv_append(ctypes.byref(s), max_new, _ptr(n_new, torch.int32, "n_new"), _ptr(k_new, e, "k_new"),
                                _ptr(v_new, e, "v_new"), _ptr(kidx_new, e, "kidx_new"), _ptr(k_main, e, "k_main"),
                                _ptr(v_main, e, "v_main"), _ptr(k_idx, e, "k_idx"), _ptr(kb, e, "kb"),
                                _ptr(n_valid, torch.int32, "n_valid"), int(bool(round_to_int)), *_ws(ws),
                                _stream(stream)), "csa2_kv_append")


class CSwaSlot(ctypes.Structure):
    _fields_ = [("k_tok", ctypes.c_void_p), ("v_tok", ctypes.c_void_p), ("k_swa", ctypes.c_void_p),
                ("v_swa", ctypes.c_void_p)]


def swa_append(shape, slots, swa_head, n_swa, ws, stream=None):
    """Push one token per query into the SWA ring of every layer in ``slots`` (a list of
    (k_tok [B, dk], v_tok [B, dv], k_swa [B, W, dk], v_swa [B, W, dv])); the shared
    swa_head advances once and n_swa grows up to W."""
    s = c_shape(shape)
    e = elem_dtype(shape)
    arr = (CSwaSlot * len(slots))(*[CSwaSlot(_ptr(kt, e, "k_tok"), _ptr(vt, e, "v_tok"), _ptr(ks, e, "k_swa"),
                                             _ptr(vs, e, "v_swa")) for kt, vt, ks, vs in slots])
    _check(lib().csa2_swa_append(ctypes.byref(s), ctypes.cast(arr, ctypes.c_void_p), len(slots),
                                 _ptr(swa_head, torch.int32, "swa_head"), _ptr(n_swa, torch.int32, "n_swa"),
                                 *_ws(ws), _stream(stream)), "csa2_swa_append")


def index_blocks(shape, q_idx, w, kb, n_valid, pool_out, n_pool_out, ws, stream=None):
    s = c_shape(shape)
    e = elem_dtype(shape)
    _check(lib().csa2_index_blocks(ctypes.byref(s), _ptr(q_idx, e, "q_idx"), _ptr(w, torch.float32, "w"),
                                   _ptr(kb, e, "kb"), _ptr(n_valid, torch.int32, "n_valid"),
                                   _ptr(pool_out, torch.int32, "pool_out"),
                                   _ptr(n_pool_out, torch.int32, "n_pool_out"), _ptr(ws, torch.uint8, "ws"),
                                   ws.numel(), _stream(stream)), "csa2_index_blocks")


def index_tokens(shape, q_idx, w, k_idx, n_valid, scores_out, ws, pool=None, n_pool=None, cand_out=None,
                 n_cand_out=None, stream=None):
    s = c_shape(shape)
    e = elem_dtype(shape)
    _check(lib().csa2_index_tokens(ctypes.byref(s), _ptr(q_idx, e, "q_idx"), _ptr(w, torch.float32, "w"),
                                   _ptr(k_idx, e, "k_idx"), _ptr(n_valid, torch.int32, "n_valid"),
                                   _ptr(pool, torch.int32, "pool"), _ptr(n_pool, torch.int32, "n_pool"),
                                   _ptr(scores_out, torch.float32, "scores_out"),
                                   _ptr(cand_out, torch.int32, "cand_out"),
                                   _ptr(n_cand_out, torch.int32, "n_cand_out"), _ptr(ws, torch.uint8, "ws"),
                                   ws.numel(), _stream(stream)), "csa2_index_tokens")


def index_topk(shape, q_idx, w, k_idx, n_valid, k: int, idx_out, ws, pool=None, n_pool=None, n_out=None,
               stream=None):
    """Score the candidates (flat, or the pooled blocks' entries) and select the Top-k in one call."""
    s = c_shape(shape)
    e = elem_dtype(shape)
    _check(lib().csa2_index_topk(ctypes.byref(s), _ptr(q_idx, e, "q_idx"), _ptr(w, torch.float32, "w"),
                                 _ptr(k_idx, e, "k_idx"), _ptr(n_valid, torch.int32, "n_valid"),
                                 _ptr(pool, torch.int32, "pool"), _ptr(n_pool, torch.int32, "n_pool"), int(k),
                                 _ptr(idx_out, torch.int32, "idx_out"), _ptr(n_out, torch.int32, "n_out"),
                                 _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "csa2_index_topk")


def topk(shape, scores, k: int, idx_out, ws, cand=None, n_cand=None, score_out=None, stream=None):
    s = c_shape(shape)
    ld = scores.shape[-1]
    _check(lib().csa2_topk(ctypes.byref(s), _ptr(scores, torch.float32, "scores"), int(ld),
                           _ptr(cand, torch.int32, "cand"), _ptr(n_cand, torch.int32, "n_cand"), int(k),
                           _ptr(idx_out, torch.int32, "idx_out"), _ptr(score_out, torch.float32, "score_out"),
                           _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "csa2_topk")


def sparse_attn(shape, q, k_main, v_main, idx, k_swa, v_swa, n_swa, out, ws, lse=None, stream=None):
    s = c_shape(shape)
    e = elem_dtype(shape)
    _check(lib().csa2_sparse_attn(ctypes.byref(s), _ptr(q, e, "q"), _ptr(k_main, e, "k_main"),
                                  _ptr(v_main, e, "v_main"), _ptr(idx, torch.int32, "idx"),
                                  _ptr(k_swa, e, "k_swa"), _ptr(v_swa, e, "v_swa"),
                                  _ptr(n_swa, torch.int32, "n_swa"), _ptr(out, torch.float32, "out"),
                                  _ptr(lse, torch.float32, "lse"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                  _stream(stream)), "csa2_sparse_attn")


def _layer(L, e) -> CLayer:
    g = (lambda k: L.get(k)) if isinstance(L, dict) else (lambda k: getattr(L, k, None))
    return CLayer(int(g("mode")), int(g("hier") or 0), _ptr(g("q"), e, "q"), _ptr(g("q_idx"), e, "q_idx"),
                  _ptr(g("w_idx"), torch.float32, "w_idx"), _ptr(g("k_swa"), e, "k_swa"),
                  _ptr(g("v_swa"), e, "v_swa"), _ptr(g("out"), torch.float32, "out"),
                  _ptr(g("lse"), torch.float32, "lse"), _ptr(g("idx_out"), torch.int32, "idx_out"))


class LayerGroupCall:
    """A prepared csa2_layer_group call (marshalled once, launched many times)."""

    def __init__(self, shape, layers: Iterable, k_main, v_main, k_idx, kb, n_valid, n_swa, ws):
        e = elem_dtype(shape)
        self._keep = (layers, k_main, v_main, k_idx, kb, n_valid, n_swa, ws)
        self.shape = c_shape(shape)
        ls = [_layer(L, e) for L in layers]
        self.layers = (CLayer * len(ls))(*ls)
        self.n = len(ls)
        self.args = (_ptr(k_main, e, "k_main"), _ptr(v_main, e, "v_main"), _ptr(k_idx, e, "k_idx"),
                     _ptr(kb, e, "kb"), _ptr(n_valid, torch.int32, "n_valid"), _ptr(n_swa, torch.int32, "n_swa"),
                     _ptr(ws, torch.uint8, "ws"), ws.numel())

    def __call__(self, stream=None):
        _check(lib().csa2_layer_group(ctypes.byref(self.shape), self.layers, self.n, *self.args, _stream(stream)),
               "csa2_layer_group")


def layer_group(shape, layers, k_main, v_main, k_idx, kb, n_valid, n_swa, ws, stream=None):
    LayerGroupCall(shape, layers, k_main, v_main, k_idx, kb, n_valid, n_swa, ws)(stream)


def layer_group_static(shape, layers, k_main, v_main, k_idx, kb, n_valid, n_swa, stream=None):
    """csa2_layer_group on the library's own 32 MiB device scratch (no workspace argument).

    For callers that cannot allocate device memory (a plugin whose host
    framework owns all allocations, or a decode loop that must not call
    cudaMalloc).  Calls share the scratch, so calls that may overlap on the
    GPU must be serialised by the caller."""
    e = elem_dtype(shape)
    s = c_shape(shape)
    ls = [_layer(L, e) for L in layers]
    arr = (CLayer * len(ls))(*ls)
    _check(lib().csa2_layer_group_static(ctypes.byref(s), arr, len(ls), _ptr(k_main, e, "k_main"),
                                         _ptr(v_main, e, "v_main"), _ptr(k_idx, e, "k_idx"), _ptr(kb, e, "kb"),
                                         _ptr(n_valid, torch.int32, "n_valid"), _ptr(n_swa, torch.int32, "n_swa"),
                                         _stream(stream)), "csa2_layer_group_static")


def read_device_error(ws, stream=None):
    """Synchronise and read/clear the sticky device error word: (status, detail bits)."""
    d = _I32(0)
    st = lib().csa2_read_device_error(_ptr(ws, torch.uint8, "ws"), _stream(stream), ctypes.byref(d))
    return int(st), int(d.value)


def read_static_device_error(stream=None):
    """Synchronise and read/clear the error word of the library's static scratch on the
    current device (csa2_layer_group_static, and cache-maintenance calls made with
    ws=None): (status, detail bits)."""
    d = _I32(0)
    st = lib().csa2_read_static_device_error(_stream(stream), ctypes.byref(d))
    return int(st), int(d.value)


def shard_slice(ids, lo: int, hi: int, delta: int, out, ws, n_out=None, stream=None):
    """Keep each row's ids in [lo, hi), shifted by delta, compacted into out (-1 padded)."""
    _check(lib().csa2_shard_slice(_ptr(ids, torch.int32, "ids"), int(ids.shape[0]), int(ids.shape[1]), int(lo),
                                  int(hi), int(delta), _ptr(out, torch.int32, "out"), int(out.shape[1]),
                                  _ptr(n_out, torch.int32, "n_out"), *_ws(ws), _stream(stream)), "csa2_shard_slice")


def shard_counts(n_valid, e0: int, n_loc: int, out, div: int = 1, stream=None):
    """A rank's valid entries (div 1) or blocks (div = block): ceil(clamp(n_valid - e0, 0, n_loc) / div)."""
    _check(lib().csa2_shard_counts(_ptr(n_valid, torch.int32, "n_valid"), int(n_valid.shape[0]), int(e0), int(n_loc),
                                   int(div), _ptr(out, torch.int32, "out"), _stream(stream)), "csa2_shard_counts")


def concat_parts(ids, scores, ids_out, scores_out, stream=None):
    """[parts, batch, k] lists side by side into [batch, parts * k] rows (scores may be None)."""
    parts, batch, k = (int(x) for x in ids.shape)
    _check(lib().csa2_concat_parts(parts, batch, k, _ptr(ids, torch.int32, "ids"), _ptr(scores, torch.float32, "scores"),
                                   _ptr(ids_out, torch.int32, "ids_out"), _ptr(scores_out, torch.float32, "scores_out"),
                                   _stream(stream)), "csa2_concat_parts")


def merge_attn(out_parts, lse_parts, out, lse=None, stream=None):
    """Combine softmax partials [parts, ..., v_dim] / [parts, ...] in part order into out / lse."""
    parts = int(out_parts.shape[0])
    v_dim = int(out_parts.shape[-1])
    rows = int(lse_parts[0].numel())
    _check(lib().csa2_merge_attn(parts, rows, v_dim, _ptr(out_parts, torch.float32, "out_parts"),
                                 _ptr(lse_parts, torch.float32, "lse_parts"), _ptr(out, torch.float32, "out"),
                                 _ptr(lse, torch.float32, "lse"), _stream(stream)), "csa2_merge_attn")


def debug_wait_timeout(shape, q_idx, w, k_idx, n_valid, k: int, idx_out, wait_limit_ns: int, ws, stream=None):
    """Test hook of the bounded device waits (csa2_debug_wait_timeout): the fused flat selection
    with every CTA's first tile left uncopied and waits limited to ``wait_limit_ns``."""
    s = c_shape(shape)
    e = elem_dtype(shape)
    _check(lib().csa2_debug_wait_timeout(ctypes.byref(s), _ptr(q_idx, e, "q_idx"), _ptr(w, torch.float32, "w"),
                                         _ptr(k_idx, e, "k_idx"), _ptr(n_valid, torch.int32, "n_valid"), int(k),
                                         _ptr(idx_out, torch.int32, "idx_out"), int(wait_limit_ns),
                                         *_ws(ws), _stream(stream)), "csa2_debug_wait_timeout")


def launch_count() -> int:
    """Kernel launches enqueued by the library so far (captured graph launches count once)."""
    return int(lib().csa2_launch_count())


def fast_path(shape):
    s = c_shape(shape)
    a, b = _I32(0), _I32(0)
    lib().csa2_fast_path(ctypes.byref(s), ctypes.byref(a), ctypes.byref(b))
    return bool(a.value), bool(b.value)


# ------------------------------------------------------------------ workload upload

def to_device_tensor(arr, device="cuda") -> torch.Tensor:
    """numpy -> device tensor; uint16 arrays hold bf16 bit patterns."""
    import numpy as np
    a = np.ascontiguousarray(arr)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def upload(wl, device="cuda", with_outputs: bool = True):
    """Copy a workloads.Workload to the device and allocate outputs / workspace.

    Returns a dict with the group tensors, the per-layer dicts (accepted by
    ``layer_group``) and a workspace.  Block summary keys are left to
    ``block_keys`` (cache-side maintenance)."""
    sh = wl.shape
    d = dict(k_main=to_device_tensor(wl.k_main, device), v_main=to_device_tensor(wl.v_main, device),
             k_idx=to_device_tensor(wl.k_idx, device),
             n_valid=torch.from_numpy(wl.n_valid.astype("int32")).to(device),
             n_swa=torch.from_numpy(wl.n_swa.astype("int32")).to(device))
    nb = -(-sh.n_entries // sh.block)
    d["kb"] = torch.zeros((sh.batch, nb, sh.idx_dim), dtype=elem_dtype(sh), device=device)
    layers = []
    for L in wl.layers:
        y = dict(mode=L.mode, hier=L.hier, q=to_device_tensor(L.q, device), k_swa=to_device_tensor(L.k_swa, device),
                 v_swa=to_device_tensor(L.v_swa, device))
        if L.q_idx is not None:
            y["q_idx"] = to_device_tensor(L.q_idx, device)
            y["w_idx"] = to_device_tensor(L.w_idx, device)
        if with_outputs:
            y["out"] = torch.empty((sh.batch, sh.q_heads, sh.v_dim), dtype=torch.float32, device=device)
            y["lse"] = torch.empty((sh.batch, sh.q_heads), dtype=torch.float32, device=device)
            if L.mode in (FULL, REINDEX):
                y["idx_out"] = torch.empty((sh.batch, sh.topk), dtype=torch.int32, device=device)
        layers.append(y)
    d["layers"] = layers
    d["ws"] = workspace(sh, device)
    return d
