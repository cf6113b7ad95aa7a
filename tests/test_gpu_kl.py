"""Parity of msa_index_kl (the index branch's KL(P||Q) loss and its gradient,
through the C ABI) with the oracle (msa_ref_index_kl, pinned by finite
differences and torch SDPA in tests/test_oracle_kl.py).

Index inputs lie on the 2^-3 grid, so the pooled scores and the maximising
token of every block (ties to the first token) are exact and identical on
both sides.  The rest is fp32 on the GPU: P carries the relative error of
fp32 attention statistics (about 1e-6), Q and the logarithms that of expf
and logf, so the loss and the gradients are compared within
|got - want| <= 1e-4 + 1e-4 |want|.
"""
import numpy as np
import pytest

from tests.helpers import Workload

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-4, 1e-4


@pytest.fixture(scope="module")
def msa():
    import torch
    assert torch.cuda.is_available()
    import block_sparse_attention_04_gb300 as m
    m.load()
    return m


def run_kl(msa, wl, sel):
    import torch
    dev = wl.device()
    p = wl.params(msa)
    ws = msa.kl_workspace(p)
    kl = torch.full((wl.B, wl.T, wl.G), float("nan"), dtype=torch.float32, device="cuda")
    dq = torch.full((wl.B, wl.T, wl.G, wl.Di), float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.zeros((wl.B, wl.max_blocks * 128, wl.Di), dtype=torch.float32, device="cuda")
    msa.msa_index_kl(p, dev["q_idx"], dev["k_idx"], dev["q"], dev["k"],
                     torch.from_numpy(np.ascontiguousarray(sel)).cuda(), wl.q_start, wl.kv_len,
                     kl, dq, dk, ws)
    torch.cuda.synchronize()
    return [x.cpu().numpy().astype(np.float64) for x in (kl, dq, dk)]


def check(ref, wl, sel, got):
    want = ref.index_kl_batch(wl.dims(ref), wl.q_idx, wl.k_idx, wl.q, wl.k, sel,
                              np.array(wl.q_start, np.int32), np.array(wl.kv_len, np.int32),
                              wl.max_blocks)
    for name, g, w in zip(("kl", "dq_idx", "dk_idx"), got, want):
        err = np.abs(g - w) - (ATOL + RTOL * np.abs(w))
        assert np.all(np.isfinite(g)) and err.max() <= 0, (name, np.abs(g - w).max())


def test_kl_prefill_m2_layout(msa, ref):
    wl = Workload(B=1, T=2500, H=48, G=8, D=128, Di=64, ctx=[2500], q_start=[0])
    sel, _ = wl.oracle(ref)
    check(ref, wl, sel, run_kl(msa, wl, sel))


def test_kl_full_128k_context(msa, ref):
    # 64 queries at the end of a 131072-token context (1024 blocks), the 128K
    # prefill's longest rows; the gradient dK_idx spans the whole context
    wl = Workload(B=1, T=64, H=48, G=8, D=128, Di=64, ctx=[131072], q_start=[131008])
    sel, _ = wl.oracle(ref)
    check(ref, wl, sel, run_kl(msa, wl, sel))


def test_kl_long_context_chunk_and_decode_batch(msa, ref):
    wl = Workload(B=1, T=200, H=12, G=4, D=128, Di=64, ctx=[9000], q_start=[8800])
    sel, _ = wl.oracle(ref)
    check(ref, wl, sel, run_kl(msa, wl, sel))
    ctx = [1, 130, 2049, 7000]
    wl = Workload(B=4, T=1, H=48, G=8, D=128, Di=64, ctx=ctx, q_start=[c - 1 for c in ctx])
    sel, _ = wl.oracle(ref)
    check(ref, wl, sel, run_kl(msa, wl, sel))


@pytest.mark.parametrize("H,G,D,Di", [(64, 4, 64, 32), (4, 1, 64, 32)])
def test_kl_head_layouts(msa, ref, H, G, D, Di):
    wl = Workload(B=1, T=300, H=H, G=G, D=D, Di=Di, ctx=[3300], q_start=[3000])
    sel, _ = wl.oracle(ref)
    check(ref, wl, sel, run_kl(msa, wl, sel))


def test_kl_caller_selection_with_duplicates_and_holes(msa, ref):
    wl = Workload(B=2, T=100, H=8, G=2, D=64, Di=64, ctx=[5000, 5000], q_start=[4900, 3000])
    rng = np.random.default_rng(9)
    sel = np.full((2, 100, 2, 16), -1, np.int32)
    for b in range(2):
        for i in range(100):
            lb = (wl.q_start[b] + i) // 128
            for g in range(2):
                ids = rng.integers(0, lb + 3, size=rng.integers(1, 17))
                sel[b, i, g, :len(ids)] = ids
    check(ref, wl, sel, run_kl(msa, wl, sel))
