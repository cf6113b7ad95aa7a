"""The algorithmic work that bench.py divides by, counted from the oracle.

bench.py reports roofline fractions from closed forms:
- attended tokens per query;
- index flops, from the candidate keys per query;
- decode bytes.
Here the same quantities are counted from the oracle's own selections and pooled scores on
seeded inputs, so a wrong closed form (an off-by-one in the local block, scoring the local block,
a missing group factor) fails.
"""
import os
import sys

import numpy as np

import msa_synth as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402  (numpy only at import time)

BLK = 128


def attended_by_selection(sel_t, t):
    """Tokens <= t inside the selected blocks of one (query, group)."""
    n = 0
    for b in sel_t:
        if b >= 0:
            n += min(BLK, t - BLK * int(b) + 1)
    return n


def test_attended_tokens_and_index_keys_match_the_oracle(ref):
    G, Di, L = 2, 32, 40 * BLK + 77
    d = ref.dims(4, G, 64, Di)
    k_idx = syn.kidx_seq(syn.BASE_SEED, 0, L, Di)
    ts = sorted({0, 1, 127, 128, 129, 255, 2047, 2048, 2049, 2175, 2176, 3000, L - 1}
                | set(range(1900, 2200, 37)))
    for t in ts:
        q_idx_t = syn.qidx_rows(syn.BASE_SEED, 0, t, t + 1, G, Di)[0]
        sel, pooled = ref.select(d, t, q_idx_t, k_idx[:t + 1], want_pooled=True)
        for g in range(G):
            assert attended_by_selection(sel[g], t) == int(bench.attended_tokens(t)), (t, g)
        # candidate keys per group: the whole blocks before the local one, which
        # the oracle pools; each costs 2 * Di flop per group
        assert pooled.shape == (G, t // BLK)
        assert bench.index_flops([t]) == 2.0 * bench.DI * bench.G * BLK * pooled.shape[1]


def test_attention_flops_count_every_head():
    t = np.array([0, 5, 2047, 2048, 100000])
    want = sum(4.0 * bench.D * bench.H * float(bench.attended_tokens(x)) for x in t)
    assert bench.attn_flops(t) == want
    # at most 16 blocks, the local one partial: 15 * 128 + (t mod 128) + 1
    assert int(bench.attended_tokens(100000)) == 15 * BLK + 100000 % BLK + 1
    assert int(bench.attended_tokens(2047)) == 2048


def test_decode_bytes_match_a_counted_gather(ref):
    # one decode query at the end of an L-token context: K_idx of every candidate
    # block, plus K and V of the selected tokens of every group
    G, D, Di, L = 2, 64, 32, 30 * BLK + 10
    d = ref.dims(4, G, D, Di)
    t = L - 1
    k_idx = syn.kidx_seq(syn.BASE_SEED, 0, L, Di)
    sel = ref.select(d, t, syn.qidx_rows(syn.BASE_SEED, 0, t, t + 1, G, Di)[0], k_idx)
    kidx_bytes = (t // BLK) * BLK * Di * 2
    kv_bytes = sum(attended_by_selection(sel[g], t) for g in range(G)) * D * 2 * 2
    # bench's closed form, evaluated for these dims
    saved = bench.G, bench.D, bench.DI
    try:
        bench.G, bench.D, bench.DI = G, D, Di
        got_kidx, got_rest = bench.decode_bytes(1, L)
    finally:
        bench.G, bench.D, bench.DI = saved
    small = bench.H * D * 2 * 2 + G * Di * 2 + G * 16 * 4
    assert got_kidx == kidx_bytes
    assert got_rest == kv_bytes + small


def test_recorded_traffic_is_null_once_the_kernel_sources_change(tmp_path, monkeypatch):
    # roofline.traffic comes from a recorded capture that carries a hash of
    # the kernel sources it was taken on; a capture of other sources is not
    # reported, and the recorded bytes scale with the units of the launch
    import json
    import bench
    f = tmp_path / "traffic.json"
    sha = bench.kernel_sources_sha("index_tc")
    f.write_text(json.dumps({"index_tc": {"sources_sha": sha, "dram_bytes": 1000.0,
                                          "units": 10.0}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("index_tc", 25.0) == 2500.0
    assert bench.recorded_traffic("index_stream", 25.0) is None
    f.write_text(json.dumps({"index_tc": {"sources_sha": "0" * 16, "dram_bytes": 1000.0,
                                          "units": 10.0}}))
    assert bench.recorded_traffic("index_tc", 25.0) is None
