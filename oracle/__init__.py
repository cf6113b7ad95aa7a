"""MSA CPU oracle (ctypes binding) -- TEST INFRASTRUCTURE ONLY.

Loads the plain-C oracle in msa_ref.c (compiled by ``build()``) and exposes it
on numpy arrays of bf16 bit patterns (uint16).  Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package; the
product library never does.
"""
import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libmsa_ref.so")
_lib = None


def build(force=False):
    """Compile msa_ref.c into _lib/libmsa_ref.so (gcc, OpenMP, IEEE double)."""
    src = os.path.join(_HERE, "msa_ref.c")
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "msa_ref.h"))):
        return _LIB
    os.makedirs(_LIBDIR, exist_ok=True)
    tmp = _LIB + ".%d.tmp" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                           "-fno-fast-math", src, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


class Dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("G", ctypes.c_int), ("D", ctypes.c_int),
                ("Di", ctypes.c_int), ("block", ctypes.c_int), ("topk", ctypes.c_int),
                ("scale", ctypes.c_double)]


def dims(H, G, D, Di, block=128, topk=16, scale=None):
    return Dims(H, G, D, Di, block, topk, 1.0 / math.sqrt(D) if scale is None else scale)


def _bind(path):
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    ci = ctypes.c_int
    L.msa_ref_select.argtypes = [ctypes.POINTER(Dims), i64, P, P, P, P]
    L.msa_ref_attend.argtypes = [ctypes.POINTER(Dims), i64, P, P, P, P, P]
    L.msa_ref_dense.argtypes = [ctypes.POINTER(Dims), i64, P, P, P, P]
    L.msa_ref_quality.argtypes = [ctypes.POINTER(Dims), i64, P, P, P, P, P, P, P, P]
    L.msa_ref_index_kl.argtypes = [ctypes.POINTER(Dims), i64, P, P, P, P, P, P, P, P]
    L.msa_ref_index_kl_batch.argtypes = [ctypes.POINTER(Dims), ci, ci, ci, P, P, P, P, P, P, P,
                                         P, P, P, ci]
    L.msa_ref_index_topk.argtypes = [ctypes.POINTER(Dims), ci, ci, ci, P, P, P, P, P, ci]
    L.msa_ref_sparse_attn.argtypes = [ctypes.POINTER(Dims), ci, ci, ci, P, P, P, P, P, P,
                                      P, ci]
    L.msa_ref_dense_attn.argtypes = [ctypes.POINTER(Dims), ci, ci, ci, P, P, P, P, P, P, ci]
    for f in ("msa_ref_select", "msa_ref_attend", "msa_ref_dense", "msa_ref_quality",
              "msa_ref_index_kl", "msa_ref_index_kl_batch", "msa_ref_index_topk",
              "msa_ref_sparse_attn", "msa_ref_dense_attn"):
        getattr(L, f).restype = ctypes.c_int
    return L


_override = None


def lib():
    """The loaded oracle library (a test may swap in another build with use_library)."""
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


class use_library:
    """Context manager: route this module's functions to the oracle built at `path`."""

    def __init__(self, path):
        self.L = _bind(path)

    def __enter__(self):
        global _override
        _override = self.L
        return self

    def __exit__(self, *exc):
        global _override
        _override = None


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError("oracle %s rejected its arguments (rc=%d)" % (what, rc))


def nthreads_default():
    return os.cpu_count() or 1


def select(d, t, q_idx_t, k_idx_seq, want_pooled=False):
    """One query: q_idx_t [G][Di], k_idx_seq [>= t+1][Di] -> sel [G][topk]."""
    q_idx_t, k_idx_seq = _u16(q_idx_t), _u16(k_idx_seq)
    sel = np.empty((d.G, d.topk), np.int32)
    lb = t // d.block
    pooled = np.empty((d.G, max(lb, 1)), np.float64) if want_pooled else None
    _check(lib().msa_ref_select(ctypes.byref(d), t, _p(q_idx_t), _p(k_idx_seq), _p(sel),
                                _p(pooled) if want_pooled else None), "select")
    return (sel, pooled[:, :lb]) if want_pooled else sel


def attend(d, t, q_t, k_seq, v_seq, sel_t):
    """One query: q_t [H][D], k/v [nblocks][block][G][D], sel_t [G][topk] -> [H][D]."""
    q_t, k_seq, v_seq = _u16(q_t), _u16(k_seq), _u16(v_seq)
    sel_t = np.ascontiguousarray(sel_t, np.int32)
    out = np.empty((d.H, d.D), np.float64)
    _check(lib().msa_ref_attend(ctypes.byref(d), t, _p(q_t), _p(k_seq), _p(v_seq), _p(sel_t),
                                _p(out)), "attend")
    return out


def dense(d, t, q_t, k_seq, v_seq):
    q_t, k_seq, v_seq = _u16(q_t), _u16(k_seq), _u16(v_seq)
    out = np.empty((d.H, d.D), np.float64)
    _check(lib().msa_ref_dense(ctypes.byref(d), t, _p(q_t), _p(k_seq), _p(v_seq), _p(out)),
           "dense")
    return out


def quality(d, t, q_t, k_seq, sel_t, want_mass=False):
    """Selection quality of one query (see msa_ref.h): q_t [H][D], k_seq
    [nblocks][block][G][D], sel_t [G][topk] -> dict(coverage [H],
    best_coverage [H], dense_sel [G][topk], hits [G], mass [G][lb+1] if asked)."""
    q_t, k_seq = _u16(q_t), _u16(k_seq)
    sel_t = np.ascontiguousarray(sel_t, np.int32)
    cov = np.empty(d.H, np.float64)
    best = np.empty(d.H, np.float64)
    ds = np.empty((d.G, d.topk), np.int32)
    hits = np.empty(d.G, np.int32)
    mass = np.empty((d.G, t // d.block + 1), np.float64) if want_mass else None
    _check(lib().msa_ref_quality(ctypes.byref(d), t, _p(q_t), _p(k_seq), _p(sel_t), _p(cov),
                                 _p(best), _p(ds), _p(hits), _p(mass) if want_mass else None),
           "quality")
    r = dict(coverage=cov, best_coverage=best, dense_sel=ds, hits=hits)
    if want_mass:
        r["mass"] = mass
    return r


def index_kl(d, t, q_idx_t, k_idx_seq, q_t, k_seq, sel_t, dk_idx=None):
    """One query's KL(P||Q) per group and its gradient (see msa_ref.h):
    returns (kl [G], dq_idx [G][Di]); dk_idx [>= t+1][Di] float64 is
    accumulated into when given (by default a scratch array as long as
    k_idx_seq, so that a write past token t stays inside it)."""
    q_idx_t, k_idx_seq, q_t, k_seq = _u16(q_idx_t), _u16(k_idx_seq), _u16(q_t), _u16(k_seq)
    sel_t = np.ascontiguousarray(sel_t, np.int32)
    kl = np.empty(d.G, np.float64)
    dq = np.empty((d.G, d.Di), np.float64)
    if dk_idx is None:
        dk_idx = np.zeros((max(t + 1, k_idx_seq.shape[0]), d.Di), np.float64)
    assert dk_idx.dtype == np.float64 and dk_idx.flags.c_contiguous and dk_idx.shape[0] > t
    _check(lib().msa_ref_index_kl(ctypes.byref(d), t, _p(q_idx_t), _p(k_idx_seq), _p(q_t),
                                  _p(k_seq), _p(sel_t), _p(kl), _p(dq), _p(dk_idx)), "index_kl")
    return kl, dq


def index_kl_batch(d, q_idx, k_idx, q, k, sel, q_start, kv_len, max_blocks, nthreads=None):
    """kl [B][T][G], dq_idx [B][T][G][Di], dk_idx [B][max_blocks*block][Di]."""
    q_idx, k_idx, q, k = _u16(q_idx), _u16(k_idx), _u16(q), _u16(k)
    sel = np.ascontiguousarray(sel, np.int32)
    B, T = q.shape[0], q.shape[1]
    qs, kl_ = _pos(B, q_start, kv_len)
    kl = np.empty((B, T, d.G), np.float64)
    dq = np.empty((B, T, d.G, d.Di), np.float64)
    dk = np.zeros((B, max_blocks * d.block, d.Di), np.float64)
    _check(lib().msa_ref_index_kl_batch(ctypes.byref(d), B, T, max_blocks, _p(q_idx), _p(k_idx),
                                        _p(q), _p(k), _p(sel), _p(qs), _p(kl_), _p(kl), _p(dq),
                                        _p(dk), nthreads or nthreads_default()), "index_kl_batch")
    return kl, dq, dk


def _pos(B, q_start, kv_len):
    return (np.ascontiguousarray(np.broadcast_to(np.asarray(q_start, np.int32), (B,))),
            np.ascontiguousarray(np.broadcast_to(np.asarray(kv_len, np.int32), (B,))))


def index_topk(d, q_idx, k_idx, q_start, kv_len, max_blocks, nthreads=None):
    """q_idx [B][T][G][Di], k_idx [B][max_blocks*block][Di] -> sel [B][T][G][topk]."""
    q_idx, k_idx = _u16(q_idx), _u16(k_idx)
    B, T = q_idx.shape[0], q_idx.shape[1]
    qs, kl = _pos(B, q_start, kv_len)
    sel = np.empty((B, T, d.G, d.topk), np.int32)
    _check(lib().msa_ref_index_topk(ctypes.byref(d), B, T, max_blocks, _p(q_idx), _p(k_idx),
                                    _p(qs), _p(kl), _p(sel), nthreads or nthreads_default()),
           "index_topk")
    return sel


def sparse_attn(d, q, k, v, sel, q_start, kv_len, max_blocks, nthreads=None):
    q, k, v = _u16(q), _u16(k), _u16(v)
    sel = np.ascontiguousarray(sel, np.int32)
    B, T = q.shape[0], q.shape[1]
    qs, kl = _pos(B, q_start, kv_len)
    out = np.empty((B, T, d.H, d.D), np.float64)
    _check(lib().msa_ref_sparse_attn(ctypes.byref(d), B, T, max_blocks, _p(q), _p(k), _p(v),
                                     _p(sel), _p(qs), _p(kl), _p(out),
                                     nthreads or nthreads_default()), "sparse_attn")
    return out


def dense_attn(d, q, k, v, q_start, kv_len, max_blocks, nthreads=None):
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, T = q.shape[0], q.shape[1]
    qs, kl = _pos(B, q_start, kv_len)
    out = np.empty((B, T, d.H, d.D), np.float64)
    _check(lib().msa_ref_dense_attn(ctypes.byref(d), B, T, max_blocks, _p(q), _p(k), _p(v),
                                    _p(qs), _p(kl), _p(out), nthreads or nthreads_default()),
           "dense_attn")
    return out


def forward(d, q_idx, k_idx, q, k, v, q_start, kv_len, max_blocks, nthreads=None):
    sel = index_topk(d, q_idx, k_idx, q_start, kv_len, max_blocks, nthreads)
    return sel, sparse_attn(d, q, k, v, sel, q_start, kv_len, max_blocks, nthreads)
