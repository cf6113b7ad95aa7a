"""msa_index_topk_noalloc: the index scan for callers that cannot allocate
device memory (for example a serving engine that gave all free GPU memory to
its KV-cache pool, or a plugin host that passes only input and output
buffers).  Its scratch is a static array inside the library.

Checked through the C ABI against msa_index_topk (which takes a caller
workspace): selections must be bit-identical, on two calls in a row with
different shapes, so that leftovers of the first call in the shared array
cannot go unnoticed.  This file sorts last so that a run stopping at the
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


def test_noalloc_rejects_calls_beyond_its_scratch():
    import ctypes
    import block_sparse_attention_04_gb300 as msa
    # 256 sequences x 4M-token context needs 256*128*8*15*8 bytes > 16 MiB
    p = msa.params(256, 1, 48, 8, 128, 64, 32768)
    qs = [32768 * 128 - 1] * 256
    kl = [32768 * 128] * 256
    with pytest.raises(msa.MsaError) as e:
        msa.msa_index_topk_noalloc(p, 0x10000, 0x20000, qs, kl, 0x30000)
    assert e.value.status == -3
