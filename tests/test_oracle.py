"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own formulas: selections are
checked against brute-force subset enumeration and numpy pooling, attention
against torch's scaled_dot_product_attention (a library routine) in float64,
plus closed forms and invariants.  See oracle/msa_ref.c for the method steps
("MiniMax 模型迭代与竞品分析", section 2, inference steps 1-4 and the full
attention equation).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import msa_synth as syn


def bf(x):
    return syn.f32_to_bf16_bits(np.asarray(x, np.float32))


def f64(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def grid_bits(rng, shape, levels=8):
    return bf(rng.integers(-levels, levels + 1, size=shape).astype(np.float32) / 8.0)


def normal_bits(rng, shape):
    return bf(rng.standard_normal(shape).astype(np.float32))


def pooled_numpy(q_idx_t, k_idx, lb, block):
    """[G][lb] block maxima of token scores, by numpy matmul (exact on the grid)."""
    G = q_idx_t.shape[0]
    if lb == 0:
        return np.zeros((G, 0))
    s = f64(k_idx[: lb * block]) @ f64(q_idx_t).T          # [tok][G]
    return s.reshape(lb, block, G).max(axis=1).T


def beats(P, x, y):
    return P[x] > P[y] or (P[x] == P[y] and x < y)


def brute_force_selection(P, lb, topk):
    """The unique candidate subset that dominates its complement, plus lb."""
    k = min(topk - 1, lb)
    winners = []
    for S in itertools.combinations(range(lb), k):
        inside = set(S)
        if all(beats(P, x, y) for x in S for y in range(lb) if y not in inside):
            winners.append(S)
    assert len(winners) == 1, "the tie rule must make the selection unique"
    return sorted(set(winners[0]) | {lb})


def check_invariants(sel_g, t, block, topk):
    lb = t // block
    valid = [s for s in sel_g if s >= 0]
    assert len(valid) == min(topk, lb + 1)
    assert list(sel_g[len(valid):]) == [-1] * (topk - len(valid))
    assert valid == sorted(set(valid))
    assert lb in valid
    assert all(0 <= s <= lb for s in valid)


# ----------------------------------------------------------- generator pins --
def test_splitmix64_published_sequence():
    path = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed1234567.txt")
    want = [int(l) for l in open(path) if l.strip() and not l.startswith("#")]
    got = [syn.mix64_int(1234567 + 0x9E3779B97F4A7C15 * (i + 1)) for i in range(len(want))]
    assert got == want
    h = syn.hashes(0, 0, 0, np.arange(3))  # vectorised form equals the scalar form
    key = syn.stream_key(0, 0, 0)
    assert [int(x) for x in h] == [syn.mix64_int(key + 0x9E3779B97F4A7C15 * (i + 1))
                                   for i in range(3)]


def test_generator_distributions_and_chunk_consistency():
    x = syn.bf16_bits_to_f32(syn.normal_elems(7, syn.TID_Q, 0, np.arange(200000)))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01 and np.abs(x).max() <= 3.0
    g = syn.bf16_bits_to_f32(syn.grid_elems(7, syn.TID_QIDX, 0, np.arange(100000)))
    assert set(np.unique(g * 8).astype(int)) == set(range(-8, 9))
    # a chunk of rows equals the same rows of the whole tensor (absolute positions)
    whole = syn.q_rows(3, 1, 0, 40, 4, 8)
    assert np.array_equal(syn.q_rows(3, 1, 17, 40, 4, 8), whole[17:])
    k = syn.kidx_seq(3, 0, 1024, 16)
    toks, dims = syn.needles(3, 0, 1024, 16)
    assert len(toks) == (1024 // 128 - 1) * 4 * 8
    qb = np.repeat(np.arange(1, 8), 4 * 8)
    assert np.all(toks < qb * 128)
    assert np.all(syn.bf16_bits_to_f32(k[toks, dims]) == 4.0)


def test_golden_constants_match_header():
    path = os.path.join(os.path.dirname(__file__), "golden", "msa_constants.txt")
    c = dict(l.split() for l in open(path) if l.strip() and not l.startswith("#"))
    assert int(c["block_tokens"]) * int(c["topk_blocks"]) == int(c["max_attended_tokens"])
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "msa.h")).read()
    assert "#define MSA_BLOCK %s" % c["block_tokens"] in hdr
    assert "#define MSA_TOPK %s" % c["topk_blocks"] in hdr


# ------------------------------------------------------------ selection pins --
@pytest.mark.parametrize("block,topk,Di,levels", [(4, 4, 2, 1), (4, 5, 3, 2), (8, 6, 4, 8)])
def test_selection_equals_bruteforce_small_blocks(ref, block, topk, Di, levels):
    rng = np.random.default_rng(block * 100 + topk)
    G, T = 3, 18 * block
    d = ref.dims(H=G, G=G, D=8, Di=Di, block=block, topk=topk)
    q_idx = grid_bits(rng, (T, G, Di), levels)
    k_idx = grid_bits(rng, (T, Di), levels)
    ties = 0
    for t in range(T):
        sel, pooled = ref.select(d, t, q_idx[t], k_idx, want_pooled=True)
        lb = t // block
        P = pooled_numpy(q_idx[t], k_idx, lb, block)
        assert np.array_equal(pooled, P)
        for g in range(G):
            check_invariants(list(sel[g]), t, block, topk)
            want = brute_force_selection(P[g], lb, topk)
            assert [s for s in sel[g] if s >= 0] == want
            ties += len(P[g]) - len(set(P[g]))
    assert ties > 0, "the case must exercise the tie rule"


def test_selection_equals_bruteforce_block128(ref):
    rng = np.random.default_rng(11)
    G, Di, block, topk = 2, 4, 128, 16
    T = 21 * block                          # lb up to 20: C(20, 15) subsets
    d = ref.dims(H=2, G=G, D=8, Di=Di, block=block, topk=topk)
    q_idx = grid_bits(rng, (T, G, Di), 2)
    k_idx = grid_bits(rng, (T, Di), 2)
    for t in [0, 127, 128, 1919, 2047, 2048, 2049, 2175, 2431, 2559, 2687]:
        sel = ref.select(d, t, q_idx[t], k_idx)
        lb = t // block
        P = pooled_numpy(q_idx[t], k_idx, lb, block)
        for g in range(G):
            check_invariants(list(sel[g]), t, block, topk)
            assert [s for s in sel[g] if s >= 0] == brute_force_selection(P[g], lb, topk)


def test_selection_matches_lexsort_on_long_context(ref):
    rng = np.random.default_rng(5)
    G, Di, block, topk = 2, 8, 128, 16
    T = 300 * block
    d = ref.dims(H=2, G=G, D=8, Di=Di, block=block, topk=topk)
    q_idx = grid_bits(rng, (T, G, Di))
    k_idx = grid_bits(rng, (T, Di))
    for t in [38399, 20000, 5000, 2049]:
        sel = ref.select(d, t, q_idx[t], k_idx)
        lb = t // block
        P = pooled_numpy(q_idx[t], k_idx, lb, block)
        for g in range(G):
            order = np.lexsort((np.arange(lb), -P[g]))   # score desc, id asc
            want = sorted(set(order[: topk - 1].tolist()) | {lb})
            assert [s for s in sel[g] if s >= 0] == want


def test_needle_block_is_selected(ref):
    # max pooling: one strong token is enough to recall its block
    rng = np.random.default_rng(2)
    G, Di, block, topk = 1, 8, 128, 16
    T = 64 * block
    d = ref.dims(H=1, G=G, D=8, Di=Di, block=block, topk=topk)
    k_idx = grid_bits(rng, (T, Di), 1)
    q = bf(np.full((1, Di), 1.0, np.float32))
    t = T - 1
    for needle_blk in [0, 17, 40, 62]:
        k2 = k_idx.copy()
        k2[needle_blk * block + 77] = bf(np.full(Di, 4.0, np.float32))  # score 32 > any grid score 8
        sel = ref.select(d, t, q, k2)
        assert needle_blk in sel[0]


def test_selection_invariant_to_token_order_in_block_and_positive_scale(ref):
    rng = np.random.default_rng(3)
    G, Di, block, topk = 2, 8, 128, 16
    T = 40 * block
    d = ref.dims(H=2, G=G, D=8, Di=Di, block=block, topk=topk)
    q_idx = grid_bits(rng, (T, G, Di))
    k_idx = grid_bits(rng, (T, Di))
    t = T - 1
    base = ref.select(d, t, q_idx[t], k_idx)
    perm = k_idx.copy()
    for b in range(t // block):
        perm[b * block:(b + 1) * block] = k_idx[b * block + rng.permutation(block)]
    assert np.array_equal(ref.select(d, t, q_idx[t], perm), base)
    # ranking is exp-free: a positive scale (exact, x2) cannot change it
    q2 = bf(syn.bf16_bits_to_f32(q_idx[t]) * 2.0)
    assert np.array_equal(ref.select(d, t, q2, k_idx), base)


# ------------------------------------------------------------ attention pins --
def sdpa_f64(q, k, v, mask, scale):
    """torch SDPA in float64.  q [T][H][D]; k, v [S][G][D]; mask [H][T][S] bool."""
    H, G = q.shape[1], k.shape[1]
    qt = torch.from_numpy(f64(q)).permute(1, 0, 2)                      # [H][T][D]
    kt = torch.from_numpy(f64(k)).permute(1, 0, 2).repeat_interleave(H // G, 0)
    vt = torch.from_numpy(f64(v)).permute(1, 0, 2).repeat_interleave(H // G, 0)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask), scale=scale)
    return o.permute(1, 0, 2).numpy()


def test_short_context_equals_full_causal_attention(ref):
    # with at most topk causal blocks MSA keeps every block: full GQA attention
    rng = np.random.default_rng(4)
    H, G, D, Di, block, topk = 6, 2, 32, 8, 128, 16
    T = 2048
    d = ref.dims(H=H, G=G, D=D, Di=Di, block=block, topk=topk)
    nb = T // block
    q_idx, k_idx = grid_bits(rng, (1, T, G, Di)), grid_bits(rng, (1, T, Di))
    q = normal_bits(rng, (1, T, H, D))
    k = normal_bits(rng, (1, nb, block, G, D))
    v = normal_bits(rng, (1, nb, block, G, D))
    sel, out = ref.forward(d, q_idx, k_idx, q, k, v, 0, T, nb)
    assert np.array_equal(sel[0, -1], np.tile(np.arange(nb, dtype=np.int32), (G, 1)))
    causal = np.tril(np.ones((T, T), bool))[None].repeat(H, 0)
    want = sdpa_f64(q[0], k[0].reshape(T, G, D), v[0].reshape(T, G, D), causal, d.scale)
    assert np.max(np.abs(out[0] - want)) < 1e-12
    dense = ref.dense_attn(d, q, k, v, 0, T, nb)
    assert np.max(np.abs(dense[0] - want)) < 1e-12


def test_sparse_equals_masked_sdpa(ref):
    rng = np.random.default_rng(6)
    H, G, D, Di, block, topk = 6, 2, 16, 4, 8, 4
    T = 15 * block + 5
    nb = (T + block - 1) // block
    d = ref.dims(H=H, G=G, D=D, Di=Di, block=block, topk=topk)
    q_idx, k_idx = grid_bits(rng, (1, T, G, Di)), grid_bits(rng, (1, nb * block, Di))
    q = normal_bits(rng, (1, T, H, D))
    k = normal_bits(rng, (1, nb, block, G, D))
    v = normal_bits(rng, (1, nb, block, G, D))
    sel, out = ref.forward(d, q_idx, k_idx, q, k, v, 0, T, nb)
    S = nb * block
    mask = np.zeros((H, T, S), bool)
    hpg = H // G
    for t in range(T):
        for h in range(H):
            for s in sel[0, t, h // hpg]:
                if s >= 0:
                    lo = s * block
                    mask[h, t, lo:min(lo + block, t + 1)] = True
    want = sdpa_f64(q[0], k[0].reshape(S, G, D), v[0].reshape(S, G, D), mask, d.scale)
    assert np.max(np.abs(out[0] - want)) < 1e-12


def test_closed_forms(ref):
    rng = np.random.default_rng(8)
    H, G, D, Di = 4, 2, 16, 8
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    nb = 40
    q = normal_bits(rng, (H, D))
    k = normal_bits(rng, (nb, 128, G, D))
    v = np.empty((nb, 128, G, D), np.uint16)
    v[:, :, 0, :] = bf(np.float32(0.75))
    v[:, :, 1, :] = bf(np.float32(-2.5))
    t = nb * 128 - 3
    sel = ref.select(d, t, grid_bits(rng, (G, Di)), grid_bits(rng, (nb * 128, Di)))
    out = ref.attend(d, t, q, k, v, sel)
    # constant V: the output is that constant (up to double rounding of sum(w*c)/sum(w))
    assert np.allclose(out[:2], 0.75, rtol=1e-14, atol=0) and np.allclose(out[2:], -2.5, rtol=1e-14, atol=0)
    # t = 0: one causal token, the output is that token's V row
    v0 = normal_bits(rng, (nb, 128, G, D))
    sel0 = ref.select(d, 0, grid_bits(rng, (G, Di)), grid_bits(rng, (128, Di)))
    assert [list(s) for s in sel0] == [[0] + [-1] * 15] * G
    out0 = ref.attend(d, 0, q, k, v0, sel0)
    for h in range(H):
        assert np.array_equal(out0[h], f64(v0[0, 0, h // (H // G)]))


def test_chunked_equals_unchunked(ref):
    rng = np.random.default_rng(9)
    H, G, D, Di, block, topk = 4, 2, 16, 8, 16, 4
    T, nb = 256, 16
    d = ref.dims(H=H, G=G, D=D, Di=Di, block=block, topk=topk)
    q_idx, k_idx = grid_bits(rng, (1, T, G, Di)), grid_bits(rng, (1, T, Di))
    q = normal_bits(rng, (1, T, H, D))
    k = normal_bits(rng, (1, nb, block, G, D))
    v = normal_bits(rng, (1, nb, block, G, D))
    sel, out = ref.forward(d, q_idx, k_idx, q, k, v, 0, T, nb)
    for c0, c1 in [(0, 64), (64, 128), (128, 200), (200, 256)]:
        s2, o2 = ref.forward(d, q_idx[:, c0:c1], k_idx, q[:, c0:c1], k, v, c0, c1, nb)
        assert np.array_equal(s2, sel[:, c0:c1])
        assert np.array_equal(o2, out[:, c0:c1])


def test_batched_sequences_are_independent(ref):
    rng = np.random.default_rng(10)
    H, G, D, Di = 2, 1, 8, 4
    d = ref.dims(H=H, G=G, D=D, Di=Di, block=8, topk=3)
    B, T, nb = 3, 20, 6
    q_idx, k_idx = grid_bits(rng, (B, T, G, Di)), grid_bits(rng, (B, nb * 8, Di))
    q = normal_bits(rng, (B, T, H, D))
    k = normal_bits(rng, (B, nb, 8, G, D))
    v = normal_bits(rng, (B, nb, 8, G, D))
    qs = np.array([0, 10, 28], np.int32)
    kl = qs + T
    sel, out = ref.forward(d, q_idx, k_idx, q, k, v, qs, kl, nb)
    for b in range(B):
        s1, o1 = ref.forward(d, q_idx[b:b + 1], k_idx[b:b + 1], q[b:b + 1], k[b:b + 1],
                             v[b:b + 1], qs[b], kl[b], nb)
        assert np.array_equal(s1[0], sel[b]) and np.array_equal(o1[0], out[b])


def test_rejects_bad_arguments(ref):
    d = ref.dims(H=3, G=2, D=8, Di=4)          # H % G != 0
    with pytest.raises(ValueError):
        ref.select(d, 5, np.zeros((2, 4), np.uint16), np.zeros((8, 4), np.uint16))
    d = ref.dims(H=2, G=1, D=8, Di=4, block=8, topk=2)
    z = np.zeros((1, 4, 1, 4), np.uint16)
    with pytest.raises(ValueError):                       # q_start + T > kv_len
        ref.index_topk(d, z, np.zeros((1, 16, 4), np.uint16), 2, 5, 2)
    bad = np.array([[[5, -1]]], np.int32)                 # block after the local one
    with pytest.raises(ValueError):
        ref.attend(d, 3, np.zeros((2, 8), np.uint16), np.zeros((2, 8, 1, 8), np.uint16),
                   np.zeros((2, 8, 1, 8), np.uint16), bad[0])
