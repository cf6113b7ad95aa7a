"""C-ABI checks that need no GPU: the library loads, exports every function
include/msa.h declares, and rejects bad arguments on the host before any CUDA
call (a T == 0 call with valid arguments returns MSA_OK without touching CUDA).
"""
import ctypes
import os
import re

import pytest

import block_sparse_attention_04_gb300 as msa
from block_sparse_attention_04_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WORKSPACE = 0, -1, -2, -3


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return msa.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "msa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(msa_\w+)\s*\(", text, re.M)))


def exported(path):
    import subprocess
    out = subprocess.check_output(["nm", "-D", "--defined-only", path]).decode()
    return {l.split()[-1] for l in out.splitlines() if " T " in l}


def test_exports_every_header_function(lib):
    decl = header_functions()
    assert set(decl) >= {"msa_index_topk", "msa_sparse_attn", "msa_forward",
                         "msa_workspace_bytes", "msa_workspace_status", "msa_status_string"}
    syms = exported(_build.LIBMSA)
    missing = [f for f in decl if f not in syms]
    assert not missing, missing
    for f in decl:
        assert hasattr(lib, f)


def test_status_strings(lib):
    for code, text in [(0, "ok"), (-1, "invalid argument"), (-2, "unsupported shape"),
                       (-3, "workspace too small"), (-4, "CUDA error"),
                       (-5, "kernel wait timed out")]:
        assert msa.msa_status_string(code) == text
    assert msa.msa_status_string(7) == "unknown status"


def P(**kw):
    base = dict(B=1, T=0, H=48, G=8, D=128, Di=64, max_blocks=256)
    base.update(kw)
    return msa.params(**base)


def test_workspace_bytes(lib):
    assert msa.msa_workspace_bytes(P(T=128)) > 0
    assert msa.msa_workspace_bytes(P(T=4096)) >= msa.msa_workspace_bytes(P(T=128))
    assert msa.msa_workspace_bytes(P(H=47)) == 0        # H % G != 0
    assert msa.msa_workspace_bytes(P(D=96)) == 0
    assert lib.msa_workspace_bytes(None) == 0


class Buf:
    """A fake, 256-byte aligned address that is never dereferenced."""
    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def call_index(p, q_start=(0,), kv_len=None, q_idx=0x10000, k_idx=0x20000, sel=0x30000,
               ws=0x40000, ws_bytes=None):
    L = msa.load()
    B = p.B
    qs = (ctypes.c_int32 * B)(*(list(q_start) * B)[:B])
    kl = (ctypes.c_int32 * B)(*([p.T] * B if kv_len is None else list(kv_len) * B)[:B])
    nb = msa.msa_workspace_bytes(p) if ws_bytes is None else ws_bytes
    return L.msa_index_topk(ctypes.byref(p), q_idx, k_idx, qs, kl, sel, ws, nb, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(), OK),
    (dict(H=47), INVALID),
    (dict(B=0), INVALID),
    (dict(T=-1), INVALID),
    (dict(B=257), UNSUPPORTED),
    (dict(D=96), UNSUPPORTED),
    (dict(Di=48), UNSUPPORTED),
    (dict(G=16, H=32), UNSUPPORTED),
    (dict(max_blocks=40000), UNSUPPORTED),
])
def test_host_validation_of_params(lib, kw, expect):
    assert call_index(P(**kw)) == expect


def test_host_validation_of_block_and_topk(lib):
    p = P()
    p.block = 64
    assert call_index(p) == UNSUPPORTED
    p = P()
    p.topk = 8
    assert call_index(p) == UNSUPPORTED
    p = P()
    p.scale = float("nan")
    assert call_index(p) == INVALID
    p = P()
    p.kernels = 9
    assert call_index(p) == INVALID


def test_host_validation_of_positions_pointers_and_workspace(lib):
    p = P(T=0, max_blocks=4)
    assert call_index(p, q_start=(0,), kv_len=(4 * 128,)) == OK
    assert call_index(p, q_start=(-1,), kv_len=(10,)) == INVALID
    assert call_index(p, q_start=(0,), kv_len=(4 * 128 + 1,)) == INVALID     # beyond capacity
    p1 = P(T=5, max_blocks=4)
    assert call_index(p1, q_start=(10,), kv_len=(14,)) == INVALID            # q_start+T > kv_len
    assert call_index(p, q_idx=None) == INVALID
    assert call_index(p, sel=0x30004) == INVALID                             # misaligned
    assert call_index(p, ws=0x40010) == INVALID                              # ws not 256-aligned
    assert call_index(p, ws=None) == INVALID
    assert call_index(p1, q_start=(0,), kv_len=(5,),
                      ws_bytes=msa.msa_workspace_bytes(p1) - 1) == WORKSPACE
    L = msa.load()
    assert L.msa_index_topk(None, 1, 1, None, None, 1, 1, 1, None) == INVALID
    assert L.msa_workspace_status(None, None) == INVALID


def test_forward_and_attn_validate_pointers(lib):
    L = msa.load()
    p = P(T=0, max_blocks=4)
    qs = (ctypes.c_int32 * 1)(0)
    kl = (ctypes.c_int32 * 1)(0)
    n = msa.msa_workspace_bytes(p)
    a = 0x100000
    assert L.msa_forward(ctypes.byref(p), a, a, a, a, a, qs, kl, None, a, a, n, None) == OK
    assert L.msa_forward(ctypes.byref(p), a, a, a, a, None, qs, kl, None, a, a, n, None) == INVALID
    assert L.msa_forward(ctypes.byref(p), a, a, a, a, a, qs, kl, a + 4, a, a, n, None) == INVALID
    assert L.msa_sparse_attn(ctypes.byref(p), a, a, a, a, qs, kl, a, a, n, None) == OK
    assert L.msa_sparse_attn(ctypes.byref(p), a, a, a, None, qs, kl, a, a, n, None) == INVALID
    assert L.msa_sparse_attn(ctypes.byref(p), a, a, a, a, None, kl, a, a, n, None) == INVALID


def test_noalloc_rejects_calls_beyond_its_scratch(lib):
    # 256 sequences x 4M-token contexts need 256*128*8*15*8 bytes of candidate
    # lists, more than the static 16 MiB: rejected on the host, before any
    # CUDA call (the pointers are never dereferenced)
    p = msa.params(256, 1, 48, 8, 128, 64, 32768)
    qs = [32768 * 128 - 1] * 256
    kl = [32768 * 128] * 256
    with pytest.raises(msa.MsaError) as e:
        msa.msa_index_topk_noalloc(p, 0x10000, 0x20000, qs, kl, 0x30000, stream=0)
    assert e.value.status == WORKSPACE
    p = msa.params(300, 1, 48, 8, 128, 64, 4)                  # B beyond MSA_MAX_BATCH
    with pytest.raises(msa.MsaError) as e:
        msa.msa_index_topk_noalloc(p, 0x10000, 0x20000, [0] * 300, [1] * 300, 0x30000,
                                   stream=0)
    assert e.value.status == UNSUPPORTED


def test_large_single_prefill_call_is_accepted(lib):
    # T*G above 2^24 (query, group) rows in one call: more than 2^17 row
    # tiles of the tensor-core index scan.  The host accepts the shape and
    # sizes the workspace for every row (the parity of such a call is a GPU
    # test); the positions check still applies.
    T = (1 << 21) + 700
    nb = (T + 127) // 128
    p = msa.params(1, T, 8, 8, 64, 64, nb, kernels="tensorcore")
    n = msa.msa_workspace_bytes(p)
    cand = T * ((nb - 1 + 1023) // 1024) * 8 * 15 * 8     # per-split top-15 lists
    assert n >= cand + T * 8 * 16 * 4
    assert call_index(p, q_start=(0,), kv_len=(T,), ws_bytes=n - 1) == WORKSPACE
    assert call_index(p, q_start=(1,), kv_len=(T,), ws_bytes=n) == INVALID


def test_paged_entry_points_validate_on_the_host(lib):
    L = msa.load()
    p = P(T=0, max_blocks=4)
    qs = (ctypes.c_int32 * 1)(0)
    kl = (ctypes.c_int32 * 1)(0)
    n = msa.msa_workspace_bytes(p)
    a, bt = 0x100000, 0x200000
    fwd = L.msa_forward_paged
    assert fwd(ctypes.byref(p), bt, 10, a, a, a, a, a, qs, kl, None, a, a, n, None) == OK
    assert fwd(ctypes.byref(p), None, 10, a, a, a, a, a, qs, kl, None, a, a, n, None) == INVALID
    assert fwd(ctypes.byref(p), bt, 0, a, a, a, a, a, qs, kl, None, a, a, n, None) == INVALID
    assert fwd(ctypes.byref(p), bt + 2, 10, a, a, a, a, a, qs, kl, None, a, a, n, None) == INVALID
    assert fwd(ctypes.byref(p), bt, 1 << 24, a, a, a, a, a, qs, kl, None, a, a, n,
               None) == UNSUPPORTED
    assert fwd(ctypes.byref(p), bt, 10, a, None, a, a, a, qs, kl, None, a, a, n, None) == INVALID
    app = L.msa_cache_append
    p1 = P(T=3, max_blocks=4)
    ok_qs = (ctypes.c_int32 * 1)(4 * 128 - 3)
    bad_qs = (ctypes.c_int32 * 1)(4 * 128 - 2)                  # runs past the capacity
    z = P(T=0, max_blocks=4)
    assert app(ctypes.byref(z), None, 0, a, a, a, ok_qs, a, a, a, a, 256, None) == OK
    assert app(ctypes.byref(p1), None, 0, a, a, a, bad_qs, a, a, a, a, 256, None) == INVALID
    assert app(ctypes.byref(p1), bt, 0, a, a, a, ok_qs, a, a, a, a, 256, None) == INVALID
    assert app(ctypes.byref(p1), None, 0, a, a, a, ok_qs, a, a, a, a, 255, None) == WORKSPACE
    assert app(ctypes.byref(p1), None, 0, a, a + 8, a, ok_qs, a, a, a, a, 256, None) == INVALID
    assert app(ctypes.byref(p1), None, 0, a, a, a, None, a, a, a, a, 256, None) == INVALID


def test_dense_entry_point_validates_on_the_host(lib):
    L = msa.load()
    p = P(T=0, max_blocks=4)
    qs = (ctypes.c_int32 * 1)(0)
    kl = (ctypes.c_int32 * 1)(0)
    n = msa.msa_dense_workspace_bytes(p)
    assert n > 0 and msa.msa_dense_workspace_bytes(P(D=96)) == 0
    p1 = P(T=64, max_blocks=4)
    # tensor-core shapes keep everything on chip: the status word only;
    # streaming shapes add fp32 running accumulators
    assert msa.msa_dense_workspace_bytes(p1) == 256
    assert msa.msa_dense_workspace_bytes(P(T=64, max_blocks=4, kernels="streaming")) >= \
        64 * 48 * (128 + 2) * 4
    a = 0x100000
    f = L.msa_dense_attn
    assert f(ctypes.byref(p), a, a, a, qs, kl, a, a, n, None) == OK
    assert f(ctypes.byref(p), a, None, a, qs, kl, a, a, n, None) == INVALID
    assert f(ctypes.byref(p), a, a, a + 2, qs, kl, a, a, n, None) == INVALID
    assert f(ctypes.byref(p), a, a, a, qs, kl, a, a + 16, n, None) == INVALID
    qs1 = (ctypes.c_int32 * 1)(0)
    kl1 = (ctypes.c_int32 * 1)(64)
    n1 = msa.msa_dense_workspace_bytes(p1)
    assert f(ctypes.byref(p1), a, a, a, qs1, kl1, a, a, n1 - 1, None) == WORKSPACE


def test_workspace_sizes_above_two_gigabytes_come_back_whole(lib):
    # every *_workspace_bytes call returns size_t: a 64K dense call on the
    # streaming kernels needs about 2.5 GB, more than a 32-bit return could hold
    p = msa.params(1, 65536, 48, 8, 128, 64, 512, kernels="streaming")
    n = msa.msa_dense_workspace_bytes(p)
    assert n > (1 << 31)
    assert n >= 65536 * 48 * 128 * 4                   # the fp32 output accumulators alone
    for f in (msa.msa_workspace_bytes, msa.msa_quality_workspace_bytes,
              msa.msa_index_kl_workspace_bytes, msa.msa_dense_workspace_bytes):
        assert f(p) > 0
    big = msa.params(256, 1, 48, 8, 128, 64, 32768)    # 256 decode rows at 4M: quality scratch
    assert msa.msa_quality_workspace_bytes(big) > (1 << 31)
