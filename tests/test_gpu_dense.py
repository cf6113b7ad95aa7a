"""Parity of msa_dense_attn (dense causal GQA attention on the block-major
caches, through the C ABI) with the oracle's dense routine, which is pinned to
torch's scaled_dot_product_attention in float64 (tests/test_oracle.py).
Outputs within max-abs 2e-2 and mean-abs 2e-3, on both kernel families, for
contexts of one to several 16-block chunks.
"""
import numpy as np
import pytest

from tests.helpers import Workload, assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu

KERNELS = ["streaming", "tensorcore"]


@pytest.fixture(scope="module")
def msa():
    import torch
    assert torch.cuda.is_available()
    import block_sparse_attention_04_gb300 as m
    m.load()
    return m


def run_dense(msa, wl, kernels):
    import torch
    dev = wl.device()
    p = wl.params(msa, kernels)
    ws = msa.dense_workspace(p)
    out = torch.full((wl.B, wl.T, wl.H, wl.D), 0x7FC0, dtype=torch.int16, device="cuda")
    msa.msa_dense_attn(p, dev["q"], dev["k"], dev["v"], wl.q_start, wl.kv_len, out, ws)
    msa.msa_workspace_status(ws)
    torch.cuda.synchronize()
    return bf16_to_f64(out.cpu().numpy())


def oracle_dense(ref, wl):
    return ref.dense_attn(wl.dims(ref), wl.q, wl.k, wl.v, np.array(wl.q_start, np.int32),
                          np.array(wl.kv_len, np.int32), wl.max_blocks)


@pytest.mark.parametrize("kernels", KERNELS)
def test_dense_prefill_m2_layout_two_chunks(msa, ref, kernels):
    # 2500 tokens: 20 blocks, i.e. one full chunk of 16 and a ragged second one
    wl = Workload(B=1, T=2500, H=48, G=8, D=128, Di=64, ctx=[2500], q_start=[0])
    assert_close(run_dense(msa, wl, kernels), oracle_dense(ref, wl))


@pytest.mark.parametrize("kernels", KERNELS)
def test_dense_long_context_chunk(msa, ref, kernels):
    # 300 queries at the end of a 6000-token context: 47 blocks, 3 chunks
    wl = Workload(B=1, T=300, H=12, G=4, D=128, Di=64, ctx=[6000], q_start=[5700])
    assert_close(run_dense(msa, wl, kernels), oracle_dense(ref, wl))


@pytest.mark.parametrize("kernels", KERNELS)
def test_dense_decode_ragged_batch(msa, ref, kernels):
    ctx = [1, 127, 128, 2049, 5000, 9000]
    wl = Workload(B=len(ctx), T=1, H=48, G=8, D=128, Di=64, ctx=ctx,
                  q_start=[c - 1 for c in ctx], max_blocks=72)
    assert_close(run_dense(msa, wl, kernels), oracle_dense(ref, wl))


@pytest.mark.parametrize("H,G,D", [(64, 4, 64), (64, 4, 128), (4, 1, 64)])
def test_dense_head_layouts_on_tensor_cores(msa, ref, H, G, D):
    # M3's own layout (64 query / 4 KV heads) among them
    wl = Workload(B=1, T=600, H=H, G=G, D=D, Di=32, ctx=[2600], q_start=[2000])
    assert_close(run_dense(msa, wl, "tensorcore"), oracle_dense(ref, wl))


@pytest.mark.parametrize("kernels", KERNELS)
def test_dense_negative_scale_and_spread_scores(msa, ref, kernels):
    from tests.test_gpu_parity import spike_keys
    wl = Workload(B=2, T=400, H=12, G=4, D=128, Di=64, ctx=[2400, 3000], q_start=[2000, 2600],
                  scale=-0.0625)
    wl.k = spike_keys(wl.k)
    assert_close(run_dense(msa, wl, kernels), oracle_dense(ref, wl))


def test_dense_equals_sparse_below_sixteen_blocks(msa, ref):
    # with at most 16 causal blocks the MSA selection holds every block, so the
    # sparse forward pass and the dense one agree (both against the oracle)
    wl = Workload(B=1, T=2048, H=12, G=4, D=128, Di=64, ctx=[2048], q_start=[0])
    want = oracle_dense(ref, wl)
    from tests.helpers import run_forward
    _, sparse = run_forward(msa, wl, "tensorcore")
    assert_close(sparse, want)
    assert_close(run_dense(msa, wl, "tensorcore"), want)
