"""Paged caches ("前沿架构解码手记（三）" section 2.1, block-major KV served by a
paged engine): msa_cache_append and msa_forward_paged through the C ABI.

The writer moves bytes, so it is checked bit-exactly against a numpy scatter
of the same rows, with every other row of the pools unchanged.  The paged
forward pass is checked against the oracle run on the logical (gathered)
caches: block ids bit-exact, outputs within max-abs 2e-2 / mean-abs 2e-3,
for both kernel families.  Block-table entries outside the pool are reported
through the workspace status and never dereferenced.
"""
import numpy as np
import pytest

import msa_synth as syn
from tests.helpers import Workload, assert_close, assert_sel_equal, bf16_to_f64

pytestmark = pytest.mark.gpu

KERNELS = ["streaming", "tensorcore"]


@pytest.fixture(scope="module")
def msa():
    import torch
    assert torch.cuda.is_available()
    import block_sparse_attention_04_gb300 as m
    m.load()
    return m


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def make_pools(wl, extra, seed):
    """Pools holding the workload's caches in shuffled blocks (plus `extra`
    blocks of noise), and the block table that finds them."""
    rng = np.random.default_rng(seed)
    nb = wl.max_blocks
    npool = wl.B * nb + extra
    perm = rng.permutation(npool).astype(np.int32)
    table = perm[:wl.B * nb].reshape(wl.B, nb)
    G, D, Di = wl.G, wl.D, wl.Di
    kp = rng.integers(0, 1 << 16, size=(npool, 128, G, D), dtype=np.uint16)
    vp = rng.integers(0, 1 << 16, size=(npool, 128, G, D), dtype=np.uint16)
    kip = rng.integers(0, 1 << 16, size=(npool, 128, Di), dtype=np.uint16)
    for b in range(wl.B):
        kp[table[b]] = wl.k[b]
        vp[table[b]] = wl.v[b]
        kip[table[b]] = wl.k_idx[b].reshape(nb, 128, Di)
    # pool entries are bf16 bit patterns; keep the noise finite (no NaN/inf)
    for a in (kp, vp, kip):
        a &= np.uint16(0xBFFF)
    for b in range(wl.B):
        kp[table[b]] = wl.k[b]
        vp[table[b]] = wl.v[b]
        kip[table[b]] = wl.k_idx[b].reshape(nb, 128, Di)
    return table, kp, vp, kip


def run_paged(msa, wl, table, kp, vp, kip, kernels):
    import torch
    p = wl.params(msa, kernels)
    ws = msa.workspace(p)
    sel = torch.full((wl.B, wl.T, wl.G, 16), -7, dtype=torch.int32, device="cuda")
    out = torch.full((wl.B, wl.T, wl.H, wl.D), 0x7FC0, dtype=torch.int16, device="cuda")
    msa.msa_forward_paged(p, torch.from_numpy(table).cuda(), kp.shape[0], dev(wl.q_idx), dev(kip),
                          dev(wl.q), dev(kp), dev(vp), wl.q_start, wl.kv_len, out, ws,
                          sel_out=sel)
    msa.msa_workspace_status(ws)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), bf16_to_f64(out.cpu().numpy())


@pytest.mark.parametrize("kernels", KERNELS)
def test_paged_decode_ragged_contexts(msa, ref, kernels):
    ctx = [1, 127, 128, 129, 2048, 2049, 5000, 9000]
    wl = Workload(B=len(ctx), T=1, H=48, G=8, D=128, Di=64, ctx=ctx,
                  q_start=[c - 1 for c in ctx], max_blocks=72)
    want_sel, want_out = wl.oracle(ref)
    table, kp, vp, kip = make_pools(wl, extra=37, seed=1)
    sel, out = run_paged(msa, wl, table, kp, vp, kip, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("kernels", KERNELS)
def test_paged_prefill_chunk(msa, ref, kernels):
    # a chunk of 700 queries after 1300 tokens in two sequences whose blocks
    # are interleaved in one pool
    wl = Workload(B=2, T=700, H=12, G=4, D=128, Di=64, ctx=[2000, 2300], q_start=[1300, 1600])
    want_sel, want_out = wl.oracle(ref)
    table, kp, vp, kip = make_pools(wl, extra=5, seed=2)
    sel, out = run_paged(msa, wl, table, kp, vp, kip, kernels)
    assert_sel_equal(sel, want_sel)
    assert_close(out, want_out)


@pytest.mark.parametrize("paged", [False, True])
def test_cache_append_writes_exactly_the_new_rows(msa, paged):
    import torch
    rng = np.random.default_rng(3)
    B, T, H, G, D, Di, nb = 3, 5, 4, 2, 64, 32, 4
    q_start = [0, 125, 300]                 # the second crosses a block boundary
    p = msa.params(B, T, H, G, D, Di, nb)
    npool = B * nb + 3 if paged else B * nb
    table = rng.permutation(npool)[:B * nb].astype(np.int32).reshape(B, nb)
    if not paged:
        table = np.arange(B * nb, dtype=np.int32).reshape(B, nb)
    kp = rng.integers(0, 1 << 16, size=(npool, 128, G, D), dtype=np.uint16)
    vp = rng.integers(0, 1 << 16, size=(npool, 128, G, D), dtype=np.uint16)
    kip = rng.integers(0, 1 << 16, size=(npool, 128, Di), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, size=(B, T, G, D), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, size=(B, T, G, D), dtype=np.uint16)
    kin = rng.integers(0, 1 << 16, size=(B, T, Di), dtype=np.uint16)
    dk, dv, dki = dev(kp), dev(vp), dev(kip)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    msa.msa_cache_append(p, dev(kn), dev(vn), dev(kin), q_start, dk, dv, dki, ws,
                         block_table=torch.from_numpy(table).cuda() if paged else None,
                         num_pool_blocks=npool)
    msa.msa_workspace_status(ws)
    want_k, want_v, want_ki = kp.copy(), vp.copy(), kip.copy()
    for b in range(B):
        for i in range(T):
            t = q_start[b] + i
            blk, r = table[b, t // 128], t % 128
            want_k[blk, r], want_v[blk, r], want_ki[blk, r] = kn[b, i], vn[b, i], kin[b, i]
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), want_k)
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), want_v)
    assert np.array_equal(dki.cpu().numpy().view(np.uint16), want_ki)


@pytest.mark.parametrize("kernels", KERNELS)
def test_append_then_decode_through_the_table(msa, ref, kernels):
    # the serving step: the pools hold every sequence's context but its newest
    # token; the token is appended through the table, then decoded
    import torch
    ctx = [130, 2049, 6000, 9001]
    wl = Workload(B=len(ctx), T=1, H=48, G=8, D=128, Di=64, ctx=ctx,
                  q_start=[c - 1 for c in ctx], max_blocks=72)
    want_sel, want_out = wl.oracle(ref)
    table, kp, vp, kip = make_pools(wl, extra=11, seed=4)
    for b, c in enumerate(ctx):             # erase the newest rows
        blk, r = table[b, (c - 1) // 128], (c - 1) % 128
        kp[blk, r] = 0
        vp[blk, r] = 0
        kip[blk, r] = 0
    kn = np.stack([wl.k[b].reshape(-1, wl.G, wl.D)[c - 1] for b, c in enumerate(ctx)])[:, None]
    vn = np.stack([wl.v[b].reshape(-1, wl.G, wl.D)[c - 1] for b, c in enumerate(ctx)])[:, None]
    kin = np.stack([wl.k_idx[b][c - 1] for b, c in enumerate(ctx)])[:, None]
    p = wl.params(msa, kernels)
    ws = msa.workspace(p)
    tab = torch.from_numpy(table).cuda()
    dk, dv, dki = dev(kp), dev(vp), dev(kip)
    msa.msa_cache_append(p, dev(kn), dev(vn), dev(kin), wl.q_start, dk, dv, dki, ws,
                         block_table=tab, num_pool_blocks=kp.shape[0])
    msa.msa_workspace_status(ws)
    sel = torch.full((wl.B, 1, wl.G, 16), -7, dtype=torch.int32, device="cuda")
    out = torch.full((wl.B, 1, wl.H, wl.D), 0x7FC0, dtype=torch.int16, device="cuda")
    msa.msa_forward_paged(p, tab, kp.shape[0], dev(wl.q_idx), dki, dev(wl.q), dk, dv, wl.q_start,
                          wl.kv_len, out, ws, sel_out=sel)
    msa.msa_workspace_status(ws)
    assert_sel_equal(sel.cpu().numpy(), want_sel)
    assert_close(bf16_to_f64(out.cpu().numpy()), want_out)


@pytest.mark.parametrize("kernels", KERNELS)
def test_table_entry_outside_the_pool_is_reported_not_read(msa, kernels):
    import torch
    wl = Workload(B=2, T=1, H=8, G=2, D=64, Di=32, ctx=[900, 700], q_start=[899, 699],
                  max_blocks=8)
    table, kp, vp, kip = make_pools(wl, extra=0, seed=5)
    table = table.copy()
    table[0, 3] = kp.shape[0] + 1000        # a block every query of sequence 0 scans
    p = wl.params(msa, kernels)
    ws = msa.workspace(p)
    out = torch.empty((2, 1, 8, 64), dtype=torch.int16, device="cuda")
    msa.msa_forward_paged(p, torch.from_numpy(table).cuda(), kp.shape[0], dev(wl.q_idx), dev(kip),
                          dev(wl.q), dev(kp), dev(vp), wl.q_start, wl.kv_len, out, ws)
    with pytest.raises(msa.MsaError) as e:
        msa.msa_workspace_status(ws)
    assert e.value.status == -1
    # the writer: a new token whose block maps outside the pool is not written
    kn = np.ones((2, 1, 2, 64), np.uint16)
    kin = np.ones((2, 1, 32), np.uint16)
    dk = dev(kp)
    before = dk.cpu().numpy()
    msa.msa_cache_append(p, dev(kn), dev(kn), dev(kin), [3 * 128 + 5, 5], dk, dev(vp), dev(kip), ws,
                         block_table=torch.from_numpy(table).cuda(), num_pool_blocks=kp.shape[0])
    with pytest.raises(msa.MsaError) as e:
        msa.msa_workspace_status(ws)
    assert e.value.status == -1
    after = dk.cpu().numpy()
    changed = np.argwhere(np.any(before != after, axis=(2, 3)))
    assert [tuple(x) for x in changed] == [(table[1, 0], 5)]
