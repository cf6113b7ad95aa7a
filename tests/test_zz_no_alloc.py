"""msa_index_topk_noalloc: the index scan for callers that cannot allocate
device memory (for example a serving engine that gave all free GPU memory to
its KV-cache pool, or a plugin host that passes only input and output
buffers).  Its scratch is a static array inside the library.

Checked through the C ABI against msa_index_topk (which takes a caller
workspace): selections must be bit-identical, on two calls in a row with
different shapes, so that leftovers of the first call in the shared array
cannot go unnoticed.  Both calls are also checked against the CPU oracle
directly, so that a fault shared by the two entry points (they run the same
streaming kernels) cannot pass either.  This file sorts last so that a run stopping at the
first failure has already run every other test; it builds and loads what it
needs itself, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _selections(msa, wl, noalloc):
    import torch
    dev = wl.device()
    p = wl.params(msa, "streaming")
    sel = torch.full((wl.B, wl.T, wl.G, 16), -7, dtype=torch.int32, device="cuda")
    if noalloc:
        msa.msa_index_topk_noalloc(p, dev["q_idx"], dev["k_idx"], wl.q_start, wl.kv_len, sel)
    else:
        ws = msa.workspace(p)
        msa.msa_index_topk(p, dev["q_idx"], dev["k_idx"], wl.q_start, wl.kv_len, sel, ws)
    torch.cuda.synchronize()
    return sel.cpu().numpy()


def test_noalloc_index_matches_workspace_entry_point_twice():
    import torch
    assert torch.cuda.is_available()
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_04_gb300 as msa
    import oracle
    from tests.helpers import Workload

    # first call: a decode batch with long, ragged contexts (many splits)
    ctx = [300, 4096, 9000, 20000, 33000, 65536]
    first = Workload(B=len(ctx), T=1, H=48, G=8, D=128, Di=64, ctx=ctx,
                     q_start=[c - 1 for c in ctx], max_blocks=512)
    # second call: a different shape with fewer splits per row, so stale
    # candidate lists of the first call would be read if a split were missed
    second = Workload(B=1, T=700, H=4, G=1, D=64, Di=32, ctx=[2500], q_start=[1800],
                      max_blocks=20)
    for wl in (first, second):
        want = _selections(msa, wl, noalloc=False)
        got = _selections(msa, wl, noalloc=True)
        assert np.array_equal(got, want)
        d = wl.dims(oracle)
        ref = oracle.index_topk(d, wl.q_idx, wl.k_idx, np.array(wl.q_start, np.int32),
                                np.array(wl.kv_len, np.int32), wl.max_blocks)
        assert np.array_equal(got, ref)
