"""Failure path of the tensor-core kernels: a pipeline wait that runs out.

Every wait between the warps of the tcgen05 index scan and of the KV-outer
attention is bounded.  A test-only poll cap (msa_debug_set_wait_polls) makes
those waits give up after one unsuccessful poll, so that a correct kernel on a
healthy GPU meets the expiry path: it must record MSA_ERR_TIMEOUT in the
workspace, drain the copies and MMAs it already issued, free its tensor memory
and exit, leaving the CUDA context usable.  The very next call on the same
workspace, with the cap removed, must then be bit-exact against the oracle.
No GPU fault or hang is involved: the waits that run out are on work that
would have completed a moment later.
"""
import numpy as np
import pytest

from tests.helpers import Workload, assert_close, assert_sel_equal, bf16_to_f64

pytestmark = pytest.mark.gpu

TIMEOUT = -5


@pytest.fixture(scope="module")
def msa():
    import torch
    assert torch.cuda.is_available()
    import block_sparse_attention_04_gb300 as m
    m.load()
    return m


def _status(msa, ws):
    try:
        msa.msa_workspace_status(ws)
        return 0
    except msa.MsaError as e:
        return e.status


# the tensor-core prefill kernels, and the streaming path's TMA-fed attention
# on a decode batch (its index scan has no pipeline waits)
CASES = {
    "tensorcore": dict(B=1, T=3000, H=48, G=8, D=128, Di=64, ctx=[6000], q_start=[3000]),
    "streaming": dict(B=6, T=1, H=48, G=8, D=128, Di=64, ctx=[9000, 4097, 128, 20000, 2500, 700],
                      q_start=[8999, 4096, 127, 19999, 2499, 699]),
}


@pytest.mark.parametrize("kernels", sorted(CASES))
def test_pipeline_wait_expiry_is_reported_then_next_call_is_exact(msa, ref, kernels):
    import torch
    wl = Workload(**CASES[kernels])
    want_sel, want_out = wl.oracle(ref)
    dev = wl.device()
    p = wl.params(msa, kernels)
    ws = msa.workspace(p)
    sel = torch.full((wl.B, wl.T, wl.G, 16), -7, dtype=torch.int32, device="cuda")
    out = torch.zeros((wl.B, wl.T, wl.H, wl.D), dtype=torch.int16, device="cuda")
    ref_sel = torch.from_numpy(want_sel).cuda()

    seen = {"index": [], "attn": []}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # larger than L2
    try:
        msa.msa_debug_set_wait_polls(1)
        for i in range(4):
            # every call starts with cold caches, so that its copies take long
            # enough for a one-poll wait to run out
            flush.fill_(i)
            msa.msa_index_topk(p, dev["q_idx"], dev["k_idx"], wl.q_start, wl.kv_len, sel, ws)
            seen["index"].append(_status(msa, ws))
            flush.fill_(i + 1)
            msa.msa_sparse_attn(p, dev["q"], dev["k"], dev["v"], ref_sel, wl.q_start, wl.kv_len,
                                out, ws)
            seen["attn"].append(_status(msa, ws))
    finally:
        msa.msa_debug_set_wait_polls(0)
    torch.cuda.synchronize()          # the context is still usable
    for k, v in seen.items():
        assert set(v) <= {0, TIMEOUT}, (k, v)
        if k == "attn" or kernels == "tensorcore":
            assert TIMEOUT in v, ("no wait ran out", k, v)

    # the next calls on the same workspace: the status word is reset and the
    # results are exact again
    sel.fill_(-7)
    out.fill_(0x7FC0)
    msa.msa_index_topk(p, dev["q_idx"], dev["k_idx"], wl.q_start, wl.kv_len, sel, ws)
    assert _status(msa, ws) == 0
    msa.msa_sparse_attn(p, dev["q"], dev["k"], dev["v"], sel, wl.q_start, wl.kv_len, out, ws)
    assert _status(msa, ws) == 0
    assert_sel_equal(sel.cpu().numpy(), want_sel)
    assert_close(bf16_to_f64(out.cpu().numpy()), want_out)


def test_dense_kernel_wait_expiry_is_reported_then_next_call_is_exact(msa, ref):
    # the query-outer dense kernel (msa_dense_attn on a prefill-sized call)
    import torch
    wl = Workload(B=1, T=1000, H=12, G=4, D=128, Di=64, ctx=[3000], q_start=[2000])
    want = ref.dense_attn(wl.dims(ref), wl.q, wl.k, wl.v, np.array(wl.q_start, np.int32),
                          np.array(wl.kv_len, np.int32), wl.max_blocks)
    dev = wl.device()
    p = wl.params(msa, "tensorcore")
    ws = msa.dense_workspace(p)
    out = torch.zeros((wl.B, wl.T, wl.H, wl.D), dtype=torch.int16, device="cuda")
    seen = []
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # larger than L2
    try:
        msa.msa_debug_set_wait_polls(1)
        for i in range(4):
            flush.fill_(i)
            msa.msa_dense_attn(p, dev["q"], dev["k"], dev["v"], wl.q_start, wl.kv_len, out, ws)
            seen.append(_status(msa, ws))
    finally:
        msa.msa_debug_set_wait_polls(0)
    torch.cuda.synchronize()
    assert set(seen) <= {0, TIMEOUT} and TIMEOUT in seen, seen
    out.fill_(0x7FC0)
    msa.msa_dense_attn(p, dev["q"], dev["k"], dev["v"], wl.q_start, wl.kv_len, out, ws)
    assert _status(msa, ws) == 0
    assert_close(bf16_to_f64(out.cpu().numpy()), want)
