"""Shared helpers for the GPU parity tests: seeded workloads (msa_synth),
device copies, calls through the C ABI and comparison against the oracle."""
import numpy as np

import msa_synth as syn

MAX_ABS = 2e-2      # tolerance on outputs (bf16 in, fp32 accumulate, bf16 out)
MEAN_ABS = 2e-3

# (test id, max|err|, mean|err|, compared values) of every output comparison
# in this session; the terminal summary prints them (tests/conftest.py)
ERRSTATS = []
CURRENT_TEST = [""]


def record_err(err):
    ERRSTATS.append((CURRENT_TEST[0], float(err.max()), float(err.mean()), int(err.size)))


class Workload:
    """Host (numpy, bf16 bits) inputs of B sequences.

    ctx[b]: whole context length of sequence b (its needles and its kv_len);
    q_start[b], T: the call's queries are positions q_start[b] .. q_start[b]+T-1.
    """

    def __init__(self, B, T, H, G, D, Di, ctx, q_start, max_blocks=None, seed=syn.BASE_SEED,
                 scale=None):
        self.B, self.T, self.H, self.G, self.D, self.Di = B, T, H, G, D, Di
        self.scale = scale      # softmax scale; None is 1/sqrt(D)
        self.ctx = [int(c) for c in ctx]
        self.q_start = [int(s) for s in q_start]
        self.kv_len = [self.q_start[b] + T for b in range(B)]
        need = max((c + 127) // 128 for c in self.ctx)
        self.max_blocks = max_blocks or need
        self.seed = seed
        cap = self.max_blocks * 128
        self.k_idx = np.stack([syn.kidx_seq(seed, b, self.ctx[b], Di, cap) for b in range(B)])
        self.k = np.stack([syn.kv_cache(seed, syn.TID_K, b, self.max_blocks, G, D)
                           for b in range(B)])
        self.v = np.stack([syn.kv_cache(seed, syn.TID_V, b, self.max_blocks, G, D)
                           for b in range(B)])
        self.q_idx = np.stack([syn.qidx_rows(seed, b, self.q_start[b], self.q_start[b] + T, G, Di)
                               for b in range(B)])
        self.q = np.stack([syn.q_rows(seed, b, self.q_start[b], self.q_start[b] + T, H, D)
                           for b in range(B)])

    def dims(self, ref):
        return ref.dims(self.H, self.G, self.D, self.Di, scale=self.scale)

    def params(self, msa, kernels="auto"):
        return msa.params(self.B, self.T, self.H, self.G, self.D, self.Di, self.max_blocks,
                          scale=self.scale, kernels=kernels)

    def device(self):
        import torch

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()

        return {k: dev(getattr(self, k)) for k in ("q_idx", "k_idx", "q", "k", "v")}

    def oracle(self, ref, rows=None):
        """Oracle sel [B][T][G][16] and out [B][T][H][D] (all rows)."""
        d = self.dims(ref)
        return ref.forward(d, self.q_idx, self.k_idx, self.q, self.k, self.v,
                           np.array(self.q_start, np.int32), np.array(self.kv_len, np.int32),
                           self.max_blocks)


def run_forward(msa, wl, kernels="auto", dev=None, split=False):
    """CUDA path through the C ABI; returns (sel, out as float64)."""
    import torch
    dev = dev or wl.device()
    p = wl.params(msa, kernels)
    ws = msa.workspace(p)
    sel = torch.full((wl.B, wl.T, wl.G, 16), -7, dtype=torch.int32, device="cuda")
    out = torch.full((wl.B, wl.T, wl.H, wl.D), 0x7FC0, dtype=torch.int16, device="cuda")  # NaN
    if split:
        msa.msa_index_topk(p, dev["q_idx"], dev["k_idx"], wl.q_start, wl.kv_len, sel, ws)
        msa.msa_sparse_attn(p, dev["q"], dev["k"], dev["v"], sel, wl.q_start, wl.kv_len, out, ws)
    else:
        msa.msa_forward(p, dev["q_idx"], dev["k_idx"], dev["q"], dev["k"], dev["v"], wl.q_start,
                        wl.kv_len, out, ws, sel_out=sel)
    msa.msa_workspace_status(ws)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), bf16_to_f64(out.cpu().numpy())


def bf16_to_f64(a):
    return syn.bf16_bits_to_f32(np.asarray(a).view(np.uint16)).astype(np.float64)


def assert_close(got, want, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    assert np.all(np.isfinite(got)), "non-finite outputs (unwritten rows?)"
    err = np.abs(got - want)
    record_err(err)
    assert err.max() <= max_abs and err.mean() <= mean_abs, (
        "max|err| %.4g (tol %.1g), mean|err| %.4g (tol %.1g)" % (err.max(), max_abs, err.mean(),
                                                                 mean_abs))
    return err.max(), err.mean()


def assert_sel_equal(got, want):
    if not np.array_equal(got, want):
        bad = np.argwhere(np.any(got != want, axis=-1))
        i = tuple(bad[0])
        raise AssertionError("%d (b,t,g) selections differ; first at %s: got %s want %s" % (
            len(bad), i, got[i].tolist(), want[i].tolist()))
