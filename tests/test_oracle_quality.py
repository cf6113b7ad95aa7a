"""Pins of the oracle's selection-quality function (msa_ref_quality).

The pages ask that MSA be judged by how much attention its selected blocks
recall ("MiniMax 模型迭代与竞品分析", section 2, the closing paragraph on the
indexer's recall risk).  These pins do not re-type the oracle's arithmetic:
block masses are checked against torch's scaled_dot_product_attention in
float64 with one-hot block indicators as values (the attention output onto an
indicator is exactly the mass of its tokens), the ideal selection against a
numpy lexsort of those masses, plus closed forms and invariants.
"""
import numpy as np
import torch

from tests.test_oracle import bf, normal_bits


def sdpa_block_mass(q_t, k_tok, t, block, G, scale):
    """A[h][b]: softmax mass of head h over block b's tokens <= t, by SDPA."""
    H, D = q_t.shape
    hpg = H // G
    n = t + 1
    nblk = t // block + 1
    qf = torch.from_numpy(syn_f64(q_t)).reshape(H, 1, D)                  # [H][1][D]
    kf = torch.from_numpy(syn_f64(k_tok[:n]))                              # [n][G][D]
    kf = kf[:, torch.arange(H) // hpg, :].permute(1, 0, 2)                 # [H][n][D]
    ind = torch.zeros(n, nblk, dtype=torch.float64)
    ind[torch.arange(n), torch.arange(n) // block] = 1.0
    v = ind.unsqueeze(0).expand(H, n, nblk)
    out = torch.nn.functional.scaled_dot_product_attention(qf, kf, v, scale=scale)
    return out[:, 0, :].numpy()                                            # [H][nblk]


def syn_f64(bits):
    import msa_synth as syn
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def ideal_selection(P, lb, topk):
    cand = np.arange(lb)
    order = np.lexsort((cand, -P[:lb]))                 # mass desc, id asc
    ids = sorted(set(cand[order[:min(topk, lb + 1) - 1]].tolist()) | {lb})
    return ids + [-1] * (topk - len(ids))


def test_quality_block_masses_and_ideal_selection_match_sdpa(ref):
    rng = np.random.default_rng(21)
    H, G, D, Di, block, topk = 6, 2, 16, 4, 8, 4
    hpg = H // G
    nb = 12
    d = ref.dims(H=H, G=G, D=D, Di=Di, block=block, topk=topk)
    k = normal_bits(rng, (nb, block, G, D))
    for t in (0, 5, 8, 31, 45, 90, nb * block - 1):
        q_t = normal_bits(rng, (H, D))
        lb = t // block
        # a selection with the local block, a duplicate and a -1 hole
        sel = np.full((G, topk), -1, np.int32)
        for g in range(G):
            ids = rng.choice(lb + 1, size=min(topk - 1, lb + 1), replace=False)
            sel[g, :len(ids)] = ids
            sel[g, -1] = ids[0]
        r = ref.quality(d, t, q_t, k, sel, want_mass=True)
        A = sdpa_block_mass(q_t, k.reshape(nb * block, G, D), t, block, G, d.scale)
        for g in range(G):
            P = A[g * hpg:(g + 1) * hpg].mean(axis=0)
            assert np.max(np.abs(r["mass"][g] - P)) < 1e-12
            want_ds = ideal_selection(P, lb, topk)
            assert r["dense_sel"][g].tolist() == want_ds
            given = {int(x) for x in sel[g] if 0 <= x <= lb}
            assert r["hits"][g] == len(given & {x for x in want_ds if x >= 0})
            for hh in range(hpg):
                h = g * hpg + hh
                assert abs(r["coverage"][h] - sum(A[h][b] for b in given)) < 1e-12
                assert abs(r["best_coverage"][h] -
                           sum(A[h][b] for b in want_ds if b >= 0)) < 1e-12


def test_quality_short_context_recalls_everything(ref):
    # with at most topk causal blocks every block is selected: coverage 1 and
    # recall 1 for any query
    rng = np.random.default_rng(22)
    H, G, D, Di = 4, 2, 32, 8
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    nb = 16
    k = normal_bits(rng, (nb, 128, G, D))
    k_idx = bf(rng.integers(-8, 9, size=(nb * 128, Di)).astype(np.float32) / 8)
    for t in (0, 127, 128, 1000, 2047):
        q_t = normal_bits(rng, (H, D))
        q_idx = bf(rng.integers(-8, 9, size=(G, Di)).astype(np.float32) / 8)
        sel = ref.select(d, t, q_idx, k_idx)
        r = ref.quality(d, t, q_t, k, sel)
        lb = t // 128
        assert np.all(np.abs(r["coverage"] - 1.0) < 1e-12)
        assert np.all(np.abs(r["best_coverage"] - 1.0) < 1e-12)
        assert np.all(r["hits"] == lb + 1)
        assert np.array_equal(r["dense_sel"], sel)


def test_quality_dominant_key_closed_form(ref):
    # one token whose scaled score (1/8 * 64 * 16 = 128) exceeds every other
    # by ~127: the rest of the mass is below e^-118, so its block is in the
    # ideal selection and coverage is 1 (to rounding) when the given
    # selection holds it, below 1e-40 when it does not
    rng = np.random.default_rng(23)
    H, G, D, Di = 2, 1, 64, 8
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    nb = 40
    t = nb * 128 - 1
    k = bf(rng.uniform(-0.2, 0.2, size=(nb, 128, G, D)).astype(np.float32))
    q_t = bf(np.ones((H, D), np.float32))
    star = 7 * 128 + 33
    k.reshape(nb * 128, G, D)[star] = bf(np.full((G, D), 16.0, np.float32))
    with_star = np.array([[3, 7, 20, 39] + [-1] * 12], np.int32)
    without = np.array([[3, 8, 20, 39] + [-1] * 12], np.int32)
    r1 = ref.quality(d, t, q_t, k, with_star)
    r0 = ref.quality(d, t, q_t, k, without)
    assert 7 in r1["dense_sel"][0] and 39 in r1["dense_sel"][0]
    assert np.all(r1["coverage"] > 1 - 1e-12) and np.all(r0["coverage"] < 1e-40)
    assert np.all(r1["best_coverage"] > 1 - 1e-12)
    for r, sel in ((r1, with_star), (r0, without)):
        ideal = {int(x) for x in r["dense_sel"][0] if x >= 0}
        assert r["hits"][0] == len(ideal & {int(x) for x in sel[0] if x >= 0})


def test_quality_ideal_selection_dominates_the_index_selection(ref):
    # the ideal selection maximises the group-averaged mass under the same
    # rule, so no index-branch selection (which holds the local block and at
    # most topk blocks) can recall more of it
    rng = np.random.default_rng(24)
    H, G, D, Di = 6, 2, 32, 16
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    nb = 30
    k = normal_bits(rng, (nb, 128, G, D))
    k_idx = bf(rng.integers(-8, 9, size=(nb * 128, Di)).astype(np.float32) / 8)
    hpg = H // G
    for t in (2048, 2500, 3000, nb * 128 - 1):
        q_t = normal_bits(rng, (H, D))
        q_idx = bf(rng.integers(-8, 9, size=(G, Di)).astype(np.float32) / 8)
        sel = ref.select(d, t, q_idx, k_idx)
        r = ref.quality(d, t, q_t, k, sel)
        lb = t // 128
        for g in range(G):
            ds = [x for x in r["dense_sel"][g] if x >= 0]
            assert len(ds) == 16 and lb in ds and ds == sorted(set(ds))
            assert 1 <= r["hits"][g] <= 16
            cov = r["coverage"][g * hpg:(g + 1) * hpg].mean()
            best = r["best_coverage"][g * hpg:(g + 1) * hpg].mean()
            assert best >= cov - 1e-12 and 0 < cov <= 1 + 1e-12
