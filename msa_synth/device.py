"""Device fill of the synthetic inputs (msa_synth/synth.cu), ctypes binding.

Same definition as the numpy generator in msa_synth/__init__.py; used to build
large inputs directly in device memory.  Tensors are torch CUDA tensors of a
2-byte dtype (bf16/int16/uint16) holding bf16 bit patterns.
"""
import ctypes
import os
import subprocess

from . import (TID_K, TID_KIDX, TID_Q, TID_QIDX, TID_V, BLOCK)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "_lib", "libmsa_synth.so")
_lib = None


def build(force=False):
    src = os.path.join(_HERE, "synth.cu")
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(src):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    nvcc = os.path.join(cuda, "bin", "nvcc")
    nvcc = nvcc if os.path.exists(nvcc) else "nvcc"
    tmp = LIB + ".%d.tmp" % os.getpid()
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
                           src, "-o", tmp, "-Xlinker", "-rpath=" + os.path.join(cuda, "lib64")])
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("msa_synth device library not built: run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        P, i64, u64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
        for f in ("msa_synth_normal", "msa_synth_grid"):
            getattr(L, f).argtypes = [P, i64, u64, ci, ci, i64, P]
            getattr(L, f).restype = ci
        L.msa_synth_needles.argtypes = [P, i64, ci, u64, ci, P]
        L.msa_synth_needles.restype = ci
        _lib = L
    return _lib


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _chk(rc):
    if rc != 0:
        raise RuntimeError("msa_synth fill failed: cudaError %d" % rc)


def fill(kind, t, seed, tid, b, idx0=0):
    """Fill the whole tensor t (one sequence's slice) with h(seed, tid, b, idx0 + k)."""
    assert t.is_cuda and t.element_size() == 2 and t.is_contiguous()
    f = lib().msa_synth_normal if kind == "normal" else lib().msa_synth_grid
    _chk(f(ctypes.c_void_p(t.data_ptr()), t.numel(), seed, tid, b, idx0, _stream()))


def plant_needles(kidx_seq, ctx_len, Di, seed, b):
    _chk(lib().msa_synth_needles(ctypes.c_void_p(kidx_seq.data_ptr()), ctx_len, Di, seed, b,
                                 _stream()))


def make_inputs(B, H, G, D, Di, max_blocks, ctx_len, seed, q_rows=None, with_qk=True, b0=0):
    """Device tensors (torch.int16 bit patterns) of a whole workload.

    ctx_len: the whole context of every sequence (needles are planted for it).
    q_rows:  (t0, t1) absolute query positions to generate for Q and Q_idx
             (default: the whole context).
    b0:      generator index of the first sequence (sequence b uses b0 + b).
    Returns dict(q_idx, k_idx, q, k, v); q/q_idx omitted when with_qk is False.
    """
    import torch
    t0, t1 = q_rows if q_rows is not None else (0, ctx_len)
    T = t1 - t0
    cap = max_blocks * BLOCK
    dev = torch.device("cuda")
    out = {}
    out["k_idx"] = torch.empty((B, cap, Di), dtype=torch.int16, device=dev)
    out["k"] = torch.empty((B, max_blocks, BLOCK, G, D), dtype=torch.int16, device=dev)
    out["v"] = torch.empty((B, max_blocks, BLOCK, G, D), dtype=torch.int16, device=dev)
    if with_qk:
        out["q_idx"] = torch.empty((B, T, G, Di), dtype=torch.int16, device=dev)
        out["q"] = torch.empty((B, T, H, D), dtype=torch.int16, device=dev)
    for b in range(B):
        gb = b0 + b
        fill("grid", out["k_idx"][b], seed, TID_KIDX, gb)
        plant_needles(out["k_idx"][b], ctx_len, Di, seed, gb)
        fill("normal", out["k"][b], seed, TID_K, gb)
        fill("normal", out["v"][b], seed, TID_V, gb)
        if with_qk:
            fill("grid", out["q_idx"][b], seed, TID_QIDX, gb, t0 * G * Di)
            fill("normal", out["q"][b], seed, TID_Q, gb, t0 * H * D)
    return out
