"""Parity of msa_selection_quality (through the C ABI) with the oracle.

The quality outputs are fp32 sums of softmax masses (bf16 inputs, fp32 scores
and exponentials), compared with the oracle's double-precision values within
QTOL.  Derivation: an fp32 score of a bf16 dot product over D <= 128 terms
carries a relative error near 2^-24 * sqrt(D) (about 1e-6 on scaled scores of
magnitude <= 10), the exponential turns it into a relative mass error of the
same size, and the hardware 2^x adds about 2^-22; a coverage sums at most 16
block masses of total <= 1, so its error stays near 1e-5.  QTOL = 1e-4 leaves
a factor of ten.

The ideal selection is decided by fp32 masses on the GPU and double ones in
the oracle, so near-ties may order differently: it is checked for validity
against the oracle's masses (local block in, right size, every chosen block
at least as heavy as every other candidate, within PTOL), and the hits are
checked against the GPU's own ideal set (and against the oracle's whenever
the two sets agree).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from tests.helpers import Workload

pytestmark = pytest.mark.gpu

QTOL = 1e-4
PTOL = 1e-6


@pytest.fixture(scope="module")
def msa():
    import torch
    assert torch.cuda.is_available()
    import block_sparse_attention_04_gb300 as m
    m.load()
    return m


def run_quality(msa, wl, sel):
    import torch
    dev = wl.device()
    p = wl.params(msa)
    ws = msa.quality_workspace(p)
    B, T, H, G = wl.B, wl.T, wl.H, wl.G
    cov = torch.full((B, T, H), float("nan"), dtype=torch.float32, device="cuda")
    best = torch.full((B, T, H), float("nan"), dtype=torch.float32, device="cuda")
    ds = torch.full((B, T, G, 16), -7, dtype=torch.int32, device="cuda")
    hits = torch.full((B, T, G), -7, dtype=torch.int32, device="cuda")
    msa.msa_selection_quality(p, dev["q"], dev["k"], torch.from_numpy(sel).cuda(), wl.q_start,
                              wl.kv_len, cov, best, ds, hits, ws)
    torch.cuda.synchronize()
    return (cov.cpu().numpy().astype(np.float64), best.cpu().numpy().astype(np.float64),
            ds.cpu().numpy(), hits.cpu().numpy())


def check_quality(ref, wl, sel, got):
    cov, best, ds, hits = got
    d = wl.dims(ref)
    rows = [(b, i) for b in range(wl.B) for i in range(wl.T)]

    def oracle_row(bi):
        b, i = bi
        return ref.quality(d, wl.q_start[b] + i, wl.q[b, i], wl.k[b], sel[b, i], want_mass=True)

    with ThreadPoolExecutor(os.cpu_count() or 4) as pool:
        want = dict(zip(rows, pool.map(oracle_row, rows)))
    for (b, i), r in want.items():
        t = wl.q_start[b] + i
        lb = t // 128
        nsel = min(16, lb + 1)
        assert np.max(np.abs(cov[b, i] - r["coverage"])) <= QTOL, (b, t)
        assert np.max(np.abs(best[b, i] - r["best_coverage"])) <= QTOL, (b, t)
        for g in range(wl.G):
            got_ids = [int(x) for x in ds[b, i, g] if x >= 0]
            assert list(ds[b, i, g, len(got_ids):]) == [-1] * (16 - len(got_ids))
            assert len(got_ids) == nsel and lb in got_ids and got_ids == sorted(set(got_ids))
            P = r["mass"][g]
            chosen = [x for x in got_ids if x != lb]
            others = [x for x in range(lb) if x not in set(chosen)]
            if chosen and others:
                assert min(P[chosen]) >= max(P[others]) - PTOL, (b, t, g)
            given = {int(x) for x in sel[b, i, g] if 0 <= x <= lb}
            assert hits[b, i, g] == len(given & set(got_ids)), (b, t, g)
            if set(got_ids) == {int(x) for x in r["dense_sel"][g] if x >= 0}:
                assert hits[b, i, g] == r["hits"][g]


def oracle_selection(ref, wl):
    sel, _ = wl.oracle(ref)
    return sel


def test_quality_m2_layout_prefill_rows(msa, ref):
    # 48/8 heads, D 128; 100 queries after 2300 tokens (two passes of rows;
    # local blocks 17-19, so 16 of up to 20 blocks are selected)
    wl = Workload(B=1, T=100, H=48, G=8, D=128, Di=64, ctx=[2400], q_start=[2300])
    sel = oracle_selection(ref, wl)
    check_quality(ref, wl, sel, run_quality(msa, wl, sel))


def test_quality_long_context(msa, ref):
    wl = Workload(B=1, T=12, H=48, G=8, D=128, Di=64, ctx=[40000], q_start=[40000 - 12])
    sel = oracle_selection(ref, wl)
    got = run_quality(msa, wl, sel)
    check_quality(ref, wl, sel, got)
    # most of a long context's mass lies outside any 16 blocks
    assert np.all(got[0] < 0.9) and np.all(got[1] >= 0)


def test_quality_full_128k_context(msa, ref):
    # the last 16 queries of a 131072-token context (1024 blocks, the 128K
    # prefill's longest rows): every block's mass over the whole context
    wl = Workload(B=1, T=16, H=48, G=8, D=128, Di=64, ctx=[131072], q_start=[131056])
    sel = oracle_selection(ref, wl)
    check_quality(ref, wl, sel, run_quality(msa, wl, sel))


def test_quality_decode_batch_ragged_contexts(msa, ref):
    ctx = [1, 127, 128, 129, 2048, 2049, 5000, 9000]
    wl = Workload(B=len(ctx), T=1, H=48, G=8, D=128, Di=64, ctx=ctx,
                  q_start=[c - 1 for c in ctx], max_blocks=72)
    sel = oracle_selection(ref, wl)
    cov, best, ds, hits = got = run_quality(msa, wl, sel)
    check_quality(ref, wl, sel, got)
    for b, c in enumerate(ctx):           # at most 16 blocks: everything recalled
        if (c - 1) // 128 < 16:
            assert np.all(np.abs(cov[b] - 1) < QTOL) and np.all(hits[b] == (c - 1) // 128 + 1)


@pytest.mark.parametrize("H,G,D", [(64, 4, 64), (4, 1, 64), (12, 4, 128)])
def test_quality_head_layouts(msa, ref, H, G, D):
    wl = Workload(B=1, T=40, H=H, G=G, D=D, Di=32, ctx=[4000], q_start=[3960])
    sel = oracle_selection(ref, wl)
    check_quality(ref, wl, sel, run_quality(msa, wl, sel))


def test_quality_negative_scale_and_caller_selection(msa, ref):
    # a caller selection with duplicates, holes and out-of-range ids (ignored)
    wl = Workload(B=2, T=30, H=12, G=4, D=128, Di=64, ctx=[5000, 5000], q_start=[4970, 3000],
                  scale=-0.0625)
    rng = np.random.default_rng(3)
    sel = np.full((2, 30, 4, 16), -1, np.int32)
    for b in range(2):
        for i in range(30):
            lb = (wl.q_start[b] + i) // 128
            for g in range(4):
                ids = rng.integers(0, lb + 3, size=rng.integers(1, 17))
                sel[b, i, g, :len(ids)] = ids
    check_quality(ref, wl, sel, run_quality(msa, wl, sel))
