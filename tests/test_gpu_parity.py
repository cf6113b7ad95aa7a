"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Block selections must be bit-exact (index inputs lie on the 2^-3 grid, so
fp32 sums are exact in any order); outputs within max-abs 2e-2 and mean-abs
2e-3 of the oracle's double-precision result.
"""
import numpy as np
import pytest

import msa_synth as syn
from tests.helpers import Workload, assert_close, assert_sel_equal, run_forward, bf16_to_f64

pytestmark = pytest.mark.gpu

KERNELS = ["streaming", "tensorcore"]


@pytest.fixture(scope="module")
def msa():
    import torch
    assert torch.cuda.is_available()
    import block_sparse_attention_04_gb300 as m
    m.load()
    return m


def test_device_generator_equals_numpy_generator():
    import torch
    import msa_synth.device as sd
    B, H, G, D, Di, nb = 2, 6, 2, 64, 32, 5
    dev = sd.make_inputs(B, H, G, D, Di, nb, ctx_len=nb * 128, seed=77, q_rows=(100, 300))
    for b in range(B):
        assert np.array_equal(dev["k_idx"][b].cpu().numpy().view(np.uint16),
                              syn.kidx_seq(77, b, nb * 128, Di))
        assert np.array_equal(dev["k"][b].cpu().numpy().view(np.uint16),
                              syn.kv_cache(77, syn.TID_K, b, nb, G, D))
        assert np.array_equal(dev["v"][b].cpu().numpy().view(np.uint16),
                              syn.kv_cache(77, syn.TID_V, b, nb, G, D))
        assert np.array_equal(dev["q"][b].cpu().numpy().view(np.uint16),
                              syn.q_rows(77, b, 100, 300, H, D))
        assert np.array_equal(dev["q_idx"][b].cpu().numpy().view(np.uint16),
                              syn.qidx_rows(77, b, 100, 300, G, Di))


@pytest.mark.parametrize("kernels", KERNELS)
@pytest.mark.parametrize("split", [False, True])
def test_tiny_prefill_3072(msa, ref, kernels, split):
    # 24 blocks of 128, 1 group of 4 heads, D 64, Di 32, every row checked
    wl = Workload(B=1, T=3072, H=4, G=1, D=64, Di=32, ctx=[3072], q_start=[0])
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, kernels, split=split)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("kernels", KERNELS)
def test_prefill_m2_layout_ragged_tail(msa, ref, kernels):
    # 48 query / 8 KV heads, D 128, Di 64; T not a multiple of the block
    wl = Workload(B=1, T=2500, H=48, G=8, D=128, Di=64, ctx=[2500], q_start=[0])
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


def spike_keys(k, every=7, shift=5):
    """Every `every`-th token's K row (all groups) times 2^shift, on bf16 bits.

    k is [B][blocks][128][G][D]. Scaling by a power of two only moves the
    exponent field, so the spiked keys are exact bf16 values."""
    k = np.array(k, dtype=np.uint16)
    tok = np.arange(k.shape[1] * k.shape[2]).reshape(1, k.shape[1], k.shape[2], 1, 1)
    hit = (tok % every == 3) & ((k & 0x7F80) != 0)
    return np.where(hit, k + np.uint16(shift << 7), k).astype(np.uint16)


@pytest.mark.parametrize("kernels", KERNELS)
def test_spiked_keys_spread_the_scores(msa, ref, kernels):
    # keys 32x larger at every 7th token spread a block's scaled scores over
    # about a hundred powers of two: the softmax maximum is far from most
    # scores, most weights underflow, and each output follows few values
    wl = Workload(B=1, T=2500, H=48, G=8, D=128, Di=64, ctx=[2500], q_start=[0])
    wl.k = spike_keys(wl.k)
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("kernels", KERNELS)
@pytest.mark.parametrize("scale", [-0.0625, 0.25])
def test_caller_scale_of_either_sign(msa, ref, kernels, scale):
    # the softmax scale is the caller's: with a negative one the largest scaled
    # score comes from the smallest raw score
    wl = Workload(B=1, T=1500, H=12, G=4, D=128, Di=64, ctx=[700 + 1500], q_start=[700],
                  scale=scale)
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,G", [(4, 4), (8, 4), (12, 4), (20, 4), (48, 8), (28, 4), (32, 4),
                                 (40, 4), (48, 4), (64, 4), (16, 1)])
def test_head_layouts_on_tensor_cores(msa, ref, H, G, D):
    # heads per group 1..16: the KV-outer tiles hold whole groups of heads per
    # query, padded to 8 or 16 rows, and copy them as 8-row boxes
    wl = Workload(B=1, T=700, H=H, G=G, D=D, Di=64, ctx=[700 + 1300], q_start=[1300])
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, "tensorcore")
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("kernels", KERNELS)
def test_chunked_prefill_matches_whole(msa, ref, kernels):
    L = 2944
    whole = Workload(B=1, T=L, H=12, G=2, D=128, Di=64, ctx=[L], q_start=[0])
    want_sel, want_out = whole.oracle(ref)
    for c0, c1 in [(0, 1024), (1024, 2048), (2048, 2900), (2900, 2944)]:
        wl = Workload(B=1, T=c1 - c0, H=12, G=2, D=128, Di=64, ctx=[L], q_start=[c0],
                      max_blocks=whole.max_blocks)
        sel, out = run_forward(msa, wl, kernels)
        assert_sel_equal(sel[0], want_sel[0, c0:c1])
        assert_close(out[0], want_out[0, c0:c1])


def test_attention_in_slices_equals_one_call(msa):
    # msa_sparse_attn over a long prefill in consecutive calls of fewer queries
    # (aligned with the tensor-core path's 8192-query passes, or not) gives
    # the same bits as one call: every query-head row's scores, softmax and
    # partial outputs depend on its own row and selection only.  The bench's
    # end-to-end leg splits a single long prefill this way.
    import torch
    import msa_synth.device as sd
    L, H_, G_, D_, DI_ = 19968, 48, 8, 128, 64
    nb = L // 128
    dev = sd.make_inputs(1, H_, G_, D_, DI_, nb, L, syn.BASE_SEED + 11)
    p = msa.params(1, L, H_, G_, D_, DI_, nb)
    ws = msa.workspace(p)
    sel = torch.empty((1, L, G_, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((1, L, H_, D_), dtype=torch.int16, device="cuda")
    msa.msa_index_topk(p, dev["q_idx"], dev["k_idx"], [0], [L], sel, ws)
    msa.msa_sparse_attn(p, dev["q"], dev["k"], dev["v"], sel, [0], [L], out, ws)
    for step in (8192, 5000):
        got = torch.full_like(out, -1)
        for a in range(0, L, step):
            n = min(step, L - a)
            ps = msa.params(1, n, H_, G_, D_, DI_, nb)
            msa.msa_sparse_attn(ps, dev["q"][:, a:a + n], dev["k"], dev["v"], sel[:, a:a + n],
                                [a], [L], got[:, a:a + n], ws)
        torch.cuda.synchronize()
        assert torch.equal(got, out), step


@pytest.mark.parametrize("kernels", KERNELS)
def test_decode_batch_ragged_contexts(msa, ref, kernels):
    ctx = [1, 127, 128, 129, 2048, 2049, 5000, 9000]
    B = len(ctx)
    wl = Workload(B=B, T=1, H=48, G=8, D=128, Di=64, ctx=ctx, q_start=[c - 1 for c in ctx],
                  max_blocks=72)
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)
    for b, c in enumerate(ctx):   # invariants: min(16, lb+1) ids, local block in
        lb = (c - 1) // 128
        for g in range(8):
            ids = [x for x in sel[b, 0, g] if x >= 0]
            assert len(ids) == min(16, lb + 1) and lb in ids and ids == sorted(ids)


@pytest.mark.parametrize("kernels", KERNELS)
def test_unaligned_starts_in_several_sequences(msa, ref, kernels):
    # rows of one work item straddle query blocks and sequences start mid-block
    wl = Workload(B=3, T=700, H=12, G=4, D=64, Di=64, ctx=[700, 1033, 1700],
                  q_start=[0, 333, 1000])
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("kernels", KERNELS)
def test_long_context_chunk_spans_several_splits(msa, ref, kernels):
    # lb up to 312: the streaming scan splits the key range into 64-block
    # splits (the tensor-core scan's 1024-block splits are crossed at full
    # size, by the 1M chunked prefill of the full-size tests)
    L = 40000
    wl = Workload(B=1, T=1000, H=4, G=2, D=64, Di=64, ctx=[L], q_start=[L - 1000])
    want_sel, want_out = wl.oracle(ref)
    sel, out = run_forward(msa, wl, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("kernels", KERNELS)
def test_sparse_attn_with_caller_selection(msa, ref, kernels):
    import torch
    wl = Workload(B=2, T=300, H=8, G=2, D=64, Di=32, ctx=[4000, 4000], q_start=[3700, 3000],
                  max_blocks=32)
    rng = np.random.default_rng(1)
    sel = np.full((2, 300, 2, 16), -1, np.int32)
    for b in range(2):
        for i in range(300):
            lb = (wl.q_start[b] + i) // 128
            for g in range(2):
                n = rng.integers(1, 17)
                ids = rng.choice(lb + 1, size=min(n, lb + 1), replace=False)
                slots = rng.choice(16, size=len(ids), replace=False)
                sel[b, i, g, slots] = ids                  # unsorted, with -1 holes
    d = wl.dims(ref)
    want = ref.sparse_attn(d, wl.q, wl.k, wl.v, sel, np.array(wl.q_start, np.int32),
                           np.array(wl.kv_len, np.int32), wl.max_blocks)
    dev = wl.device()
    p = wl.params(msa, kernels)
    ws = msa.workspace(p)
    out = torch.full((2, 300, 8, 64), 0x7FC0, dtype=torch.int16, device="cuda")
    msa.msa_sparse_attn(p, dev["q"], dev["k"], dev["v"], torch.from_numpy(sel).cuda(),
                        wl.q_start, wl.kv_len, out, ws)
    msa.msa_workspace_status(ws)
    assert_close(bf16_to_f64(out.cpu().numpy()), want)


@pytest.mark.parametrize("kernels", KERNELS)
def test_out_of_range_selection_is_reported_not_read(msa, kernels):
    import torch
    wl = Workload(B=1, T=4, H=4, G=1, D=64, Di=32, ctx=[600], q_start=[500], max_blocks=5)
    dev = wl.device()
    p = wl.params(msa, kernels)
    ws = msa.workspace(p)
    sel = torch.full((1, 4, 1, 16), -1, dtype=torch.int32, device="cuda")
    sel[0, :, 0, 0] = 3
    sel[0, 0, 0, 1] = 4          # the block after query 500's local block 3
    out = torch.empty((1, 4, 4, 64), dtype=torch.int16, device="cuda")
    msa.msa_sparse_attn(p, dev["q"], dev["k"], dev["v"], sel, wl.q_start, wl.kv_len, out, ws)
    with pytest.raises(msa.MsaError) as e:
        msa.msa_workspace_status(ws)
    assert e.value.status == -1


def test_zero_length_call_is_a_noop(msa):
    import torch
    p = msa.params(2, 0, 4, 1, 64, 32, 4)
    ws = msa.workspace(p)
    z = torch.zeros(16, dtype=torch.int16, device="cuda")
    msa.msa_forward(p, z, z, z, z, z, [0, 5], [0, 5], z, ws)
    torch.cuda.synchronize()
