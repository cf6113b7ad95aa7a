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
from tests.helpers import MAX_ABS, MEAN_ABS, bf16_to_f64

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
    rows = [(0, t) for t in sample_positions(L, 1024, 1)]
    check_rows(ref, job, rows, kidx, kv=lazy_kv(job.seed, L // BLK))


def test_prefill_128k_sampled(ref):
    job = run_job("prefill_128k")
    L = job.L
    kidx = {0: syn.kidx_seq(job.seed, 0, L, DI)}
    rows = [(0, t) for t in sample_positions(L, 4096, 2)]
    check_rows(ref, job, rows, kidx, kv=lazy_kv(job.seed, L // BLK))


def test_decode_256k_all_sequences(ref):
    job = run_job("decode_256k")
    L = job.L
    kidx = {b: syn.kidx_seq(job.seed, b, L, DI) for b in range(job.B)}
    rows = [(b, L - 1) for b in range(job.B)]
    check_rows(ref, job, rows, kidx, attn_rows=rows[:8], kv=lazy_kv(job.seed, L // BLK))


def test_prefill_1m_chunked_sampled(ref):
    job = run_job("prefill_1m")
    L = job.L
    kidx = {0: syn.kidx_seq(job.seed, 0, L, DI)}
    # >= 256 positions across all 128 chunks, plus chunk edges
    edges = [c * 8192 + o for c in (1, 64, 127) for o in (-1, 0, 1)]
    rows = [(0, t) for t in sorted(set(sample_positions(L, 256, 4)) | set(edges))]
    check_rows(ref, job, rows, kidx, kv=lazy_kv(job.seed, L // BLK))
