"""Parity at the full workload sizes, in the launch configuration bench.py times.

The GPU side is bench.Job (device-generated inputs, the same chunked calls).
The CPU oracle checks sampled rows it can compute one by one; the numpy
generator rebuilds exactly the inputs the device fill made (pinned by
test_device_generator_equals_numpy_generator).  Selections are compared
bit-exactly, outputs within max-abs 2e-2 / mean-abs 2e-3.
"""
import numpy as np
import pytest

import msa_synth as syn
from tests.helpers import MAX_ABS, MEAN_ABS, bf16_to_f64, record_err

pytestmark = pytest.mark.gpu

H, G, D, DI, BLK = 48, 8, 128, 64, 128


def special_positions(L):
    return [t for t in (0, 1, 127, 128, 129, 2047, 2048, 2049, L - 129, L - 128, L - 1) if t < L]


def sample_positions(L, n, seed):
    rng = np.random.default_rng(seed)
    ts = set(special_positions(L)) | set(int(x) for x in rng.choice(L, size=n, replace=False))
    return sorted(ts)


def run_job(name):
    import torch
    import bench
    job = bench.Job(name, 0)
    job.step()
    job.msa.msa_workspace_status(job.ws)
    torch.cuda.synchronize()
    return job


def check_rows(ref, job, rows, kidx, attn_rows=None, kv=None):
    """rows: list of (b, t).  Compares sel for every row and out for attn_rows.
    Oracle calls run on a thread pool (the C oracle releases the GIL)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    d = ref.dims(H, G, D, DI)
    sel_gpu = job.sel.cpu().numpy()
    base = job.calls[0]["q_start"][0] if job.w["kind"] == "decode" else 0
    attn_rows = rows if attn_rows is None else attn_rows
    pool = ThreadPoolExecutor(os.cpu_count() or 4)

    def select(bt):
        b, t = bt
        qi = syn.qidx_rows(job.seed, b, t, t + 1, G, DI)[0]
        return ref.select(d, t, qi, kidx[b])

    want_sel = dict(zip(rows, pool.map(select, rows)))
    for b, t in rows:
        got = sel_gpu[b, t - base]
        assert np.array_equal(got, want_sel[(b, t)]), (b, t, got.tolist(),
                                                       want_sel[(b, t)].tolist())
    caches = {bt: kv(bt[0], want_sel[bt]) for bt in attn_rows}   # fills needed blocks

    def attend(bt):
        b, t = bt
        kc, vc = caches[bt]
        qt = syn.q_rows(job.seed, b, t, t + 1, H, D)[0]
        return ref.attend(d, t, qt, kc, vc, want_sel[bt])

    wants = list(pool.map(attend, attn_rows))
    pool.shutdown()
    err = np.concatenate([
        np.abs(bf16_to_f64(job.out[b, t - base].cpu().numpy()) - w).reshape(-1)
        for (b, t), w in zip(attn_rows, wants)])
    record_err(err)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
    return err.max(), err.mean()


def lazy_kv(seed, nb):
    """K/V caches holding only the blocks a selection needs (zeros elsewhere)."""
    cache = {}

    def get(b, sel):
        if b not in cache:
            cache[b] = (np.zeros((nb, BLK, G, D), np.uint16), np.zeros((nb, BLK, G, D), np.uint16),
                        set())
        kc, vc, have = cache[b]
        need = sorted({int(x) for x in sel.reshape(-1) if x >= 0} - have)
        if need:
            kc[need] = syn.kv_blocks(seed, syn.TID_K, b, need, G, D)
            vc[need] = syn.kv_blocks(seed, syn.TID_V, b, need, G, D)
            have.update(need)
        return kc, vc

    return get


def test_prefill_32k_all_selections(ref):
    job = run_job("prefill_32k")
    L = job.L
    kidx = {0: syn.kidx_seq(job.seed, 0, L, DI)}
    d = ref.dims(H, G, D, DI)
    q_idx = syn.qidx_rows(job.seed, 0, 0, L, G, DI)[None]
    want = ref.index_topk(d, q_idx, kidx[0][None], 0, L, L // BLK)
    assert np.array_equal(job.sel.cpu().numpy(), want)
    rows = [(0, t) for t in sample_positions(L, 4096, 1)]
    check_rows(ref, job, rows, kidx, kv=lazy_kv(job.seed, L // BLK))


def whole_query_blocks(L, n):
    """n query blocks (128 queries each) spread evenly over [0, L/128), first
    and last included."""
    nb = L // BLK
    return sorted({round(k * (nb - 1) / (n - 1)) for k in range(n)})


def test_prefill_128k_whole_query_blocks_and_sample(ref):
    # Selections: every row of 64 whole query blocks spread evenly over the
    # 131072 queries (8192 queries x 8 groups), plus the sampled rows below.
    # A whole query block is 8 row tiles of the tensor-core scan, so every one
    # of the 128 row positions of a tile (16 queries x 8 groups) is checked,
    # for local blocks from 0 to 1023 (odd and even candidate counts, i.e.
    # both halves of the last key-block pair), in tiles that the heaviest-
    # first item order hands to CTAs early and late.  Attention: >= 4096
    # sampled positions including the special ones.
    job = run_job("prefill_128k")
    L = job.L
    kidx = {0: syn.kidx_seq(job.seed, 0, L, DI)}
    d = ref.dims(H, G, D, DI)
    sel_gpu = job.sel.cpu().numpy()
    for qb in whole_query_blocks(L, 64):
        t0 = qb * BLK
        q_idx = syn.qidx_rows(job.seed, 0, t0, t0 + BLK, G, DI)[None]
        want = ref.index_topk(d, q_idx, kidx[0][None], t0, L, L // BLK)
        assert np.array_equal(sel_gpu[0, t0:t0 + BLK], want[0]), qb
    rows = [(0, t) for t in sample_positions(L, 4096, 2)]
    check_rows(ref, job, rows, kidx, kv=lazy_kv(job.seed, L // BLK))


def test_decode_256k_all_sequences(ref):
    job = run_job("decode_256k")
    L = job.L
    kidx = {b: syn.kidx_seq(job.seed, b, L, DI) for b in range(job.B)}
    rows = [(b, L - 1) for b in range(job.B)]
    check_rows(ref, job, rows, kidx, attn_rows=rows[:8], kv=lazy_kv(job.seed, L // BLK))


def test_dense_32k_sampled_rows(ref):
    # msa_dense_attn over the whole 32K causal context (the query-outer
    # tensor-core kernel), against the oracle's dense attention on >= 256 rows
    import os
    from concurrent.futures import ThreadPoolExecutor
    job = run_job("dense_32k")
    L, nb = job.L, job.L // BLK
    kc = syn.kv_cache(job.seed, syn.TID_K, 0, nb, G, D)
    vc = syn.kv_cache(job.seed, syn.TID_V, 0, nb, G, D)
    ts = sample_positions(L, 256, 20261207)
    d = ref.dims(H, G, D, DI)

    def dense(t):
        return ref.dense(d, t, syn.q_rows(job.seed, 0, t, t + 1, H, D)[0], kc, vc)

    with ThreadPoolExecutor(os.cpu_count() or 4) as pool:
        wants = list(pool.map(dense, ts))
    err = np.concatenate([np.abs(bf16_to_f64(job.out[0, t].cpu().numpy()) - w).reshape(-1)
                          for t, w in zip(ts, wants)])
    record_err(err)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


def test_prefill_1m_chunked_sampled(ref):
    job = run_job("prefill_1m")
    L = job.L
    kidx = {0: syn.kidx_seq(job.seed, 0, L, DI)}
    # >= 256 positions across all 128 chunks, plus chunk edges
    edges = [c * 8192 + o for c in (1, 64, 127) for o in (-1, 0, 1)]
    rows = [(0, t) for t in sorted(set(sample_positions(L, 256, 4)) | set(edges))]
    check_rows(ref, job, rows, kidx, kv=lazy_kv(job.seed, L // BLK))


def test_index_scan_row_tiles_beyond_2_17(ref):
    # One prefill call with T*G > 2^24 (query, group) rows: the tensor-core
    # scan's row tiles (128 rows each) then number more than 2^17.  Only the
    # index step runs (steps 1-3), so no Q/K/V of this length is made.  Rows
    # on both sides of tile 2^17 (query 2^21 at G = 8) are checked.
    import torch
    import block_sparse_attention_04_gb300 as msa
    import msa_synth.device as sd
    Gt, Dit = 8, 64
    T = (1 << 21) + 700
    nb = (T + BLK - 1) // BLK
    seed = syn.BASE_SEED + 11
    k_idx = torch.empty((1, nb * BLK, Dit), dtype=torch.int16, device="cuda")
    sd.fill("grid", k_idx[0], seed, syn.TID_KIDX, 0)
    sd.plant_needles(k_idx[0], T, Dit, seed, 0)
    q_idx = torch.empty((1, T, Gt, Dit), dtype=torch.int16, device="cuda")
    sd.fill("grid", q_idx[0], seed, syn.TID_QIDX, 0, 0)
    p = msa.params(1, T, Gt, Gt, 64, Dit, nb, kernels="tensorcore")
    ws = msa.workspace(p)
    sel = torch.full((1, T, Gt, 16), -7, dtype=torch.int32, device="cuda")
    msa.msa_index_topk(p, q_idx, k_idx, [0], [T], sel, ws)
    msa.msa_workspace_status(ws)
    torch.cuda.synchronize()
    del ws, q_idx, k_idx
    edge = 1 << 21          # first query of row tile 2^17
    rng = np.random.default_rng(5)
    ts = {edge - 17, edge - 16, edge - 1, edge, edge + 1, edge + 15, edge + 16, T - 1, T - 2,
          300000}
    ts |= {int(x) for x in rng.integers(edge, T, size=12)}
    ts = sorted(ts)
    got = sel[0, ts].cpu().numpy()
    del sel
    torch.cuda.empty_cache()
    assert np.all(got != -7), "rows left unwritten"
    kidx = syn.kidx_seq(seed, 0, T, Dit)
    d = ref.dims(Gt, Gt, 64, Dit)
    from concurrent.futures import ThreadPoolExecutor
    import os
    with ThreadPoolExecutor(os.cpu_count() or 4) as pool:
        want = list(pool.map(
            lambda t: ref.select(d, t, syn.qidx_rows(seed, 0, t, t + 1, Gt, Dit)[0], kidx), ts))
    for k, t in enumerate(ts):
        assert np.array_equal(got[k], want[k]), (t, got[k].tolist(), want[k].tolist())
