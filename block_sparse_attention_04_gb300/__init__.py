"""MiniMax Sparse Attention (MSA) forward on GB300: Python binding of libmsa.

Argument marshalling only.  Every step of the path runs in the CUDA kernels
of libmsa.so (include/msa.h); there is no fallback.  If the library is not
built, loading raises.  Tensors are torch CUDA tensors with 2-byte elements
(bf16, int16 or uint16 holding bf16 bit patterns) in the layouts msa.h
states; q_start and kv_len are host sequences of B ints.
"""
import ctypes
import math
import os

from . import _build

__all__ = ["MsaParams", "MsaError", "params", "load", "msa_workspace_bytes", "msa_index_topk",
           "msa_sparse_attn", "msa_forward", "msa_workspace_status", "msa_status_string",
           "msa_kernel_launch_count", "msa_index_topk_noalloc", "msa_debug_set_wait_polls",
           "msa_quality_workspace_bytes", "msa_selection_quality", "quality_workspace",
           "msa_cache_append", "msa_forward_paged", "msa_dense_workspace_bytes",
           "msa_dense_attn", "dense_workspace", "msa_index_kl_workspace_bytes", "msa_index_kl",
           "kl_workspace",
           "workspace", "BLOCK", "TOPK"]

BLOCK = 128
TOPK = 16
KERNELS = {"auto": 0, "streaming": 1, "tensorcore": 2}
EXPORTS = ("msa_workspace_bytes", "msa_index_topk", "msa_sparse_attn", "msa_forward",
           "msa_workspace_status", "msa_status_string", "msa_kernel_launch_count",
           "msa_index_topk_noalloc", "msa_debug_set_wait_polls", "msa_quality_workspace_bytes",
           "msa_selection_quality", "msa_cache_append", "msa_forward_paged",
           "msa_dense_workspace_bytes", "msa_dense_attn", "msa_index_kl_workspace_bytes",
           "msa_index_kl")


class MsaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (what, msa_status_string(status), status))


class MsaParams(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("G", ctypes.c_int), ("D", ctypes.c_int), ("Di", ctypes.c_int),
                ("block", ctypes.c_int), ("topk", ctypes.c_int), ("max_blocks", ctypes.c_int),
                ("scale", ctypes.c_float), ("kernels", ctypes.c_int)]


def params(B, T, H, G, D, Di, max_blocks, scale=None, kernels="auto"):
    return MsaParams(B, T, H, G, D, Di, BLOCK, TOPK, max_blocks,
                     1.0 / math.sqrt(D) if scale is None else scale,
                     KERNELS[kernels] if isinstance(kernels, str) else int(kernels))


_lib = None


def load(path=None):
    """Load libmsa.so (built in-tree by _build.build()); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIBMSA
    if not os.path.exists(path):
        raise RuntimeError("libmsa.so is not built (%s); run __graft_entry__.build()" % path)
    L = ctypes.CDLL(path)
    P, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    PP = ctypes.POINTER(MsaParams)
    L.msa_workspace_bytes.argtypes = [PP]
    L.msa_workspace_bytes.restype = sz
    L.msa_index_topk.argtypes = [PP, P, P, P, P, P, P, sz, P]
    L.msa_sparse_attn.argtypes = [PP, P, P, P, P, P, P, P, P, sz, P]
    L.msa_forward.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, sz, P]
    L.msa_workspace_status.argtypes = [P, P]
    L.msa_index_topk_noalloc.argtypes = [PP, P, P, P, P, P, P]
    L.msa_cache_append.argtypes = [PP, P, ci, P, P, P, P, P, P, P, P, sz, P]
    L.msa_index_kl_workspace_bytes.argtypes = [PP]
    L.msa_index_kl_workspace_bytes.restype = sz
    L.msa_index_kl.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, P, sz, P]
    L.msa_dense_workspace_bytes.argtypes = [PP]
    L.msa_dense_workspace_bytes.restype = sz
    L.msa_dense_attn.argtypes = [PP, P, P, P, P, P, P, P, sz, P]
    L.msa_forward_paged.argtypes = [PP, P, ci, P, P, P, P, P, P, P, P, P, P, sz, P]
    L.msa_quality_workspace_bytes.argtypes = [PP]
    L.msa_quality_workspace_bytes.restype = sz
    L.msa_selection_quality.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, sz, P]
    L.msa_debug_set_wait_polls.argtypes = [ctypes.c_uint32]
    L.msa_debug_set_wait_polls.restype = None
    L.msa_kernel_launch_count.argtypes = []
    L.msa_kernel_launch_count.restype = ctypes.c_uint64
    L.msa_status_string.argtypes = [ci]
    L.msa_status_string.restype = ctypes.c_char_p
    for f in ("msa_index_topk", "msa_sparse_attn", "msa_forward", "msa_workspace_status",
              "msa_index_topk_noalloc", "msa_selection_quality", "msa_cache_append",
              "msa_forward_paged", "msa_dense_attn", "msa_index_kl"):
        getattr(L, f).restype = ci
    if path == _build.LIBMSA:
        _lib = L
    return L


def msa_status_string(status):
    return load().msa_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def _host_i32(x, B):
    vals = [int(v) for v in (x if hasattr(x, "__len__") else [x] * B)]
    if len(vals) != B:
        raise ValueError("expected %d positions, got %d" % (B, len(vals)))
    return (ctypes.c_int32 * B)(*vals)


def msa_kernel_launch_count():
    return int(load().msa_kernel_launch_count())


def msa_debug_set_wait_polls(polls):
    """Test-only: cap the tensor-core kernels' pipeline waits at `polls` polls
    (0 restores the default wall-clock bound)."""
    load().msa_debug_set_wait_polls(int(polls))


def msa_workspace_bytes(p):
    return int(load().msa_workspace_bytes(ctypes.byref(p)))


def workspace(p, device="cuda"):
    """A device scratch buffer of msa_workspace_bytes(p) bytes."""
    import torch
    n = msa_workspace_bytes(p)
    if n == 0:
        raise MsaError(-2, "msa_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _call(rc, what):
    if rc != 0:
        raise MsaError(rc, what)


def msa_index_topk(p, q_idx, k_idx, q_start, kv_len, sel, ws, stream=None):
    _call(load().msa_index_topk(ctypes.byref(p), _ptr(q_idx), _ptr(k_idx),
                                _host_i32(q_start, p.B), _host_i32(kv_len, p.B), _ptr(sel),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
          "msa_index_topk")


def msa_index_topk_noalloc(p, q_idx, k_idx, q_start, kv_len, sel, stream=None):
    """msa_index_topk without a workspace: for callers that cannot allocate
    device memory (scratch lives in a static array inside the library)."""
    _call(load().msa_index_topk_noalloc(ctypes.byref(p), _ptr(q_idx), _ptr(k_idx),
                                        _host_i32(q_start, p.B), _host_i32(kv_len, p.B),
                                        _ptr(sel), _stream(stream)), "msa_index_topk_noalloc")


def msa_sparse_attn(p, q, k_cache, v_cache, sel, q_start, kv_len, out, ws, stream=None):
    _call(load().msa_sparse_attn(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(sel), _host_i32(q_start, p.B), _host_i32(kv_len, p.B),
                                 _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                 _stream(stream)), "msa_sparse_attn")


def msa_forward(p, q_idx, k_idx, q, k_cache, v_cache, q_start, kv_len, out, ws, sel_out=None,
                stream=None):
    _call(load().msa_forward(ctypes.byref(p), _ptr(q_idx), _ptr(k_idx), _ptr(q), _ptr(k_cache),
                             _ptr(v_cache), _host_i32(q_start, p.B), _host_i32(kv_len, p.B),
                             _ptr(sel_out), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "msa_forward")


def msa_index_kl_workspace_bytes(p):
    return int(load().msa_index_kl_workspace_bytes(ctypes.byref(p)))


def kl_workspace(p, device="cuda"):
    """A device scratch buffer of msa_index_kl_workspace_bytes(p) bytes."""
    import torch
    n = msa_index_kl_workspace_bytes(p)
    if n == 0:
        raise MsaError(-2, "msa_index_kl_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def msa_index_kl(p, q_idx, k_idx, q, k_cache, sel, q_start, kv_len, kl, dq_idx, dk_idx, ws,
                 stream=None):
    """KL(P||Q) of the index branch per (query, group), dQ_idx, and dK_idx
    accumulated into (see msa.h)."""
    _call(load().msa_index_kl(ctypes.byref(p), _ptr(q_idx), _ptr(k_idx), _ptr(q), _ptr(k_cache),
                              _ptr(sel), _host_i32(q_start, p.B), _host_i32(kv_len, p.B),
                              _ptr(kl), _ptr(dq_idx), _ptr(dk_idx), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "msa_index_kl")


def msa_dense_workspace_bytes(p):
    return int(load().msa_dense_workspace_bytes(ctypes.byref(p)))


def dense_workspace(p, device="cuda"):
    """A device scratch buffer of msa_dense_workspace_bytes(p) bytes."""
    import torch
    n = msa_dense_workspace_bytes(p)
    if n == 0:
        raise MsaError(-2, "msa_dense_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def msa_dense_attn(p, q, k_cache, v_cache, q_start, kv_len, out, ws, stream=None):
    """Dense causal GQA attention over every token <= t (see msa.h)."""
    _call(load().msa_dense_attn(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                _host_i32(q_start, p.B), _host_i32(kv_len, p.B), _ptr(out),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
          "msa_dense_attn")


def msa_quality_workspace_bytes(p):
    return int(load().msa_quality_workspace_bytes(ctypes.byref(p)))


def quality_workspace(p, device="cuda"):
    """A device scratch buffer of msa_quality_workspace_bytes(p) bytes."""
    import torch
    n = msa_quality_workspace_bytes(p)
    if n == 0:
        raise MsaError(-2, "msa_quality_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def msa_selection_quality(p, q, k_cache, sel, q_start, kv_len, coverage, best_coverage,
                          dense_sel, hits, ws, stream=None):
    """Attention-mass coverage of sel and of the ideal selection, the ideal
    selection itself and the recall hits (see msa.h)."""
    _call(load().msa_selection_quality(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(sel),
                                       _host_i32(q_start, p.B), _host_i32(kv_len, p.B),
                                       _ptr(coverage), _ptr(best_coverage), _ptr(dense_sel),
                                       _ptr(hits), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)), "msa_selection_quality")


def msa_cache_append(p, k_new, v_new, k_idx_new, q_start, k_cache, v_cache, k_idx_cache, ws,
                     block_table=None, num_pool_blocks=0, stream=None):
    """Write p.T new tokens per sequence at positions q_start[b] + i, through
    block_table when the caches are pools (see msa.h)."""
    _call(load().msa_cache_append(ctypes.byref(p), _ptr(block_table), int(num_pool_blocks),
                                  _ptr(k_new), _ptr(v_new), _ptr(k_idx_new),
                                  _host_i32(q_start, p.B), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(k_idx_cache), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "msa_cache_append")


def msa_forward_paged(p, block_table, num_pool_blocks, q_idx, k_idx_pool, q, k_pool, v_pool,
                      q_start, kv_len, out, ws, sel_out=None, stream=None):
    _call(load().msa_forward_paged(ctypes.byref(p), _ptr(block_table), int(num_pool_blocks),
                                   _ptr(q_idx), _ptr(k_idx_pool), _ptr(q), _ptr(k_pool),
                                   _ptr(v_pool), _host_i32(q_start, p.B), _host_i32(kv_len, p.B),
                                   _ptr(sel_out), _ptr(out), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
          "msa_forward_paged")


def msa_workspace_status(ws, stream=None):
    """Waits for the stream; raises MsaError if a kernel recorded an error in ws."""
    _call(load().msa_workspace_status(_ptr(ws), _stream(stream)), "kernel status")
