"""Pins of the oracle's index-branch training signal (msa_ref_index_kl).

"MiniMax 模型迭代与竞品分析" section 2 states the loss: the main branch's
group-averaged block distribution P over the candidate blocks is the teacher
(no gradient), the indexer's distribution Q the student, D_KL(P || Q).  None
of these pins re-types the oracle: P is checked against torch's SDPA in
float64 with block indicators as values and a mask on the selected tokens, Q
against numpy pooling and numpy's softmax normalisation, the gradients against
central finite differences of the oracle's own loss, plus a closed form (a
single candidate) and the tie rule of the pooled maximum.
"""
import numpy as np
import torch

import msa_synth as syn
from tests.test_oracle import bf, normal_bits


def f64(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def setup(rng, H=6, G=2, D=32, Di=16, nb=24, idx_scale=0.25):
    q_idx = bf(rng.standard_normal((G, Di)).astype(np.float32) * idx_scale)
    k_idx = bf(rng.standard_normal((nb * 128, Di)).astype(np.float32))
    q = normal_bits(rng, (H, D))
    k = normal_bits(rng, (nb, 128, G, D))
    return q_idx, k_idx, q, k


def some_selection(rng, G, lb, n=16):
    sel = np.full((G, 16), -1, np.int32)
    for g in range(G):
        ids = rng.choice(lb, size=min(n - 1, lb), replace=False) if lb > 0 else []
        sel[g, :len(ids) + 1] = sorted(list(ids) + [lb])
    return sel


def test_single_candidate_gives_zero_loss_and_gradient(ref):
    rng = np.random.default_rng(31)
    d = ref.dims(H=6, G=2, D=32, Di=16)
    q_idx, k_idx, q, k = setup(rng)
    for t in (0, 60, 127):
        sel = np.full((2, 16), -1, np.int32)
        sel[:, 0] = 0
        dk = np.zeros((len(k_idx), 16))
        kl, dq = ref.index_kl(d, t, q_idx, k_idx, q, k, sel, dk)
        # P = Q = 1 up to the rounding of one softmax sum
        assert np.all(np.abs(kl) < 1e-13) and np.all(np.abs(dq) < 1e-13)
        assert np.all(np.abs(dk) < 1e-13)


def test_teacher_and_student_distributions(ref):
    # P from SDPA (block indicators as values, selected tokens <= t as mask),
    # Q from numpy pooling and normalisation: the oracle's loss must be the
    # pages' D_KL of these two independently computed distributions
    rng = np.random.default_rng(32)
    H, G, D, Di, nb = 6, 2, 32, 16, 24
    hpg = H // G
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    q_idx, k_idx, q, k = setup(rng, H, G, D, Di, nb)
    for t in (200, 1500, nb * 128 - 1):
        lb = t // 128
        sel = some_selection(rng, G, lb)
        kl, dq = ref.index_kl(d, t, q_idx, k_idx, q, k, sel)
        assert np.all(kl >= -1e-15)
        kt = torch.from_numpy(f64(k.reshape(nb * 128, G, D)[:t + 1]))
        for g in range(G):
            cand = [int(x) for x in sel[g] if x >= 0]
            mask = np.zeros(t + 1, bool)
            ind = np.zeros((t + 1, len(cand)))
            for j, c in enumerate(cand):
                mask[c * 128:min(c * 128 + 128, t + 1)] = True
                ind[c * 128:min(c * 128 + 128, t + 1), j] = 1.0
            qh = torch.from_numpy(f64(q[g * hpg:(g + 1) * hpg])).reshape(hpg, 1, D)
            kk = kt[:, g, :].unsqueeze(0).expand(hpg, t + 1, D)
            v = torch.from_numpy(ind).unsqueeze(0).expand(hpg, t + 1, len(cand))
            A = torch.nn.functional.scaled_dot_product_attention(
                qh, kk, v, attn_mask=torch.from_numpy(mask).reshape(1, 1, t + 1),
                scale=d.scale)[:, 0, :].numpy()
            P = A.mean(axis=0)
            s = f64(k_idx[:t + 1]) @ f64(q_idx[g])
            z = np.array([s[c * 128:min(c * 128 + 128, t + 1)].max() for c in cand])
            Q = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
            want = float(np.sum(P * np.log(P / Q)))
            assert abs(kl[g] - want) < 1e-12


def test_gradients_match_finite_differences_of_the_loss(ref):
    # perturb components that are exactly zero, so that +-2^-9 is exact in
    # bf16; the data are continuous, so the pooled maxima keep their tokens
    rng = np.random.default_rng(33)
    H, G, D, Di, nb = 6, 2, 32, 16, 24
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    q_idx, k_idx, q, k = setup(rng, H, G, D, Di, nb)
    t = nb * 128 - 40
    sel = some_selection(rng, G, t // 128)
    h = 2.0 ** -9
    for g, dim in [(0, 3), (1, 11), (0, 15)]:
        qz = q_idx.copy()
        qz[g, dim] = 0
        kl, dq = ref.index_kl(d, t, qz, k_idx, q, k, sel)
        qp, qm = qz.copy(), qz.copy()
        qp[g, dim] = bf([h])[0]
        qm[g, dim] = bf([-h])[0]
        fd = (ref.index_kl(d, t, qp, k_idx, q, k, sel)[0][g] -
              ref.index_kl(d, t, qm, k_idx, q, k, sel)[0][g]) / (2 * h)
        assert abs(fd - dq[g, dim]) < 1e-6 + 1e-3 * abs(dq[g, dim]), (g, dim, fd, dq[g, dim])
    # dk: perturb one component of a token that is some block's maximum; no
    # gradient reaches a token after t (the pooled scores are causal)
    dk = np.zeros((len(k_idx), Di))
    ref.index_kl(d, t, q_idx, k_idx, q, k, sel, dk)
    assert np.all(dk[t + 1:] == 0)
    tok = int(np.argmax(np.abs(dk).sum(axis=1)))
    for dim in (2, 9):
        kz = k_idx.copy()
        kz[tok, dim] = 0
        dk = np.zeros((len(k_idx), Di))
        ref.index_kl(d, t, q_idx, kz, q, k, sel, dk)
        kp, km = kz.copy(), kz.copy()
        kp[tok, dim] = bf([h])[0]
        km[tok, dim] = bf([-h])[0]
        fd = (ref.index_kl(d, t, q_idx, kp, q, k, sel)[0].sum() -
              ref.index_kl(d, t, q_idx, km, q, k, sel)[0].sum()) / (2 * h)
        assert abs(fd - dk[tok, dim]) < 1e-6 + 1e-3 * abs(dk[tok, dim]), (tok, dim, fd)


def test_tied_maximum_sends_the_gradient_to_the_first_token(ref):
    # two equal K_idx rows inside one candidate block: the pooled score is
    # attained at both, and the gradient goes to the lower token only
    rng = np.random.default_rng(34)
    H, G, D, Di, nb = 6, 1, 32, 16, 8
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    q_idx, k_idx, q, k = setup(rng, H, G, D, Di, nb)
    big = bf(np.full(Di, 2.0, np.float32) * np.sign(syn.bf16_bits_to_f32(q_idx[0])))
    k_idx[2 * 128 + 70] = big                      # equal rows: the block's maximum
    k_idx[2 * 128 + 9] = big
    t = nb * 128 - 1
    sel = np.array([[2, 5, 7] + [-1] * 13], np.int32)
    dk = np.zeros((len(k_idx), Di))
    ref.index_kl(d, t, q_idx, k_idx, q, k, sel, dk)
    assert np.any(dk[2 * 128 + 9] != 0) and np.all(dk[2 * 128 + 70] == 0)


def test_batch_equals_per_query(ref):
    rng = np.random.default_rng(35)
    H, G, D, Di, nb = 6, 2, 32, 16, 12
    d = ref.dims(H=H, G=G, D=D, Di=Di)
    T, q0 = 40, 1000
    q_idx = bf(rng.standard_normal((1, T, G, Di)).astype(np.float32) * 0.25)
    k_idx = bf(rng.standard_normal((1, nb * 128, Di)).astype(np.float32))
    q = normal_bits(rng, (1, T, H, D))
    k = normal_bits(rng, (1, nb, 128, G, D))
    sel = np.stack([some_selection(rng, G, (q0 + i) // 128) for i in range(T)])[None]
    kl, dq, dk = ref.index_kl_batch(d, q_idx, k_idx, q, k, sel, q0, q0 + T, nb)
    dk1 = np.zeros((nb * 128, Di))
    for i in range(T):
        kli, dqi = ref.index_kl(d, q0 + i, q_idx[0, i], k_idx[0], q[0, i], k[0], sel[0, i], dk1)
        assert np.array_equal(kli, kl[0, i]) and np.array_equal(dqi, dq[0, i])
    assert np.max(np.abs(dk1 - dk[0])) < 1e-12
