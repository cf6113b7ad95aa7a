"""Seeded synthetic inputs for MiniMax Sparse Attention (MSA) workloads.

This module is the single definition of every input that both the CUDA path
and the CPU oracle see.  It holds none of the method's arithmetic: it only
turns (seed, tensor, sequence, element) into bf16 bit patterns.

Generator (counter-based, SplitMix64 of Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014):

    GAMMA    = 0x9E3779B97F4A7C15
    mix64(z) : z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
    key(seed, tid, b) = mix64(mix64(seed + GAMMA*(tid+1)) + GAMMA*(b+1))
    h(seed, tid, b, i) = mix64(key(seed, tid, b) + GAMMA*(i+1))      (mod 2^64)

Element index i inside sequence b (t and tok are ABSOLUTE positions, so a
chunk of a sequence is bit-identical to the same rows of the whole sequence):

    Q     [t][H][D]     i = (t*H + h)*D + d          tid 1   "normal"
    K     [tok][G][D]   i = (tok*G + g)*D + d        tid 2   "normal"
    V     [tok][G][D]   i = (tok*G + g)*D + d        tid 3   "normal"
    Q_idx [t][G][Di]    i = (t*G + g)*Di + d         tid 4   "grid"
    K_idx [tok][Di]     i = tok*Di + d               tid 5   "grid" + needles

The KV caches are block-major [block][128][G][D]; flattened, a block's
element (r, g, d) sits at token tok = block*128 + r, so the same formula holds.

    normal(h): u_k = (h >> 16k) & 0xFFFF (k = 0, 1, 2);
               x = (2*(u0+u1+u2) - 196605) * 2^-16      (Irwin-Hall of 3,
               mean 0, standard deviation 1.0000, |x| <= 3), rounded to bf16
               with round-to-nearest-even.  Integer arithmetic plus one exact
               scaling, so every machine gives the same bits.
    grid(h)  : x = ((h mod 17) - 8) / 8, a multiple of 2^-3 in [-1, 1], exact
               in bf16.

Needles in K_idx ("4 K_idx needle tokens per query range planted at +4.0"),
for a sequence whose whole context is L tokens (NB = ceil(L/128) blocks):
for every query block qb in [1, NB) and j in [0, 4), with n = 4*qb + j,

    tok   = h(seed, 6, b, n) mod (128*qb)              a token before block qb
    dim_m = h(seed, 7, b, 8*n + m) mod Di,  m in [0, 8)
    K_idx[tok][dim_m] = 4.0

Setting a value is idempotent, so overlapping needles commute.  Every index
score stays a multiple of 2^-6 below 2^7 in magnitude, which fp32 holds
exactly under any order of summation.

Default seeds: 20261202 + workload number.
"""

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
MASK64 = (1 << 64) - 1

TID_Q, TID_K, TID_V, TID_QIDX, TID_KIDX, TID_NEEDLE_TOK, TID_NEEDLE_DIM = 1, 2, 3, 4, 5, 6, 7
BLOCK = 128
NEEDLES_PER_QBLOCK = 4
NEEDLE_DIMS = 8
NEEDLE_VALUE = 4.0
BASE_SEED = 20261202


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2^64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tid: int, b: int) -> int:
    k = mix64_int(seed + 0x9E3779B97F4A7C15 * (tid + 1))
    return mix64_int(k + 0x9E3779B97F4A7C15 * (b + 1))


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def hashes(seed: int, tid: int, b: int, idx) -> np.ndarray:
    """h(seed, tid, b, i) for an array of element indices i (int64/uint64)."""
    key = np.uint64(stream_key(seed, tid, b))
    i = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + GAMMA * (i + np.uint64(1)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE float32 -> bf16 bit pattern, round to nearest even (no NaNs here)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_from_hash(h: np.ndarray) -> np.ndarray:
    m = np.uint64(0xFFFF)
    s = (h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m)
    x = (2 * s.astype(np.int64) - 196605).astype(np.float32) * np.float32(2.0 ** -16)
    return f32_to_bf16_bits(x)


def grid_from_hash(h: np.ndarray) -> np.ndarray:
    k = (h % np.uint64(17)).astype(np.int64) - 8
    return f32_to_bf16_bits(k.astype(np.float32) * np.float32(0.125))


def normal_elems(seed: int, tid: int, b: int, idx) -> np.ndarray:
    return normal_from_hash(hashes(seed, tid, b, idx))


def grid_elems(seed: int, tid: int, b: int, idx) -> np.ndarray:
    return grid_from_hash(hashes(seed, tid, b, idx))


# ---------------------------------------------------------------- tensors --
def q_rows(seed, b, t0, t1, H, D):
    """Q[b] rows t in [t0, t1) as bf16 bits, shape [t1-t0][H][D]."""
    n = (t1 - t0) * H * D
    idx = np.arange(n, dtype=np.uint64) + np.uint64(t0 * H * D)
    return normal_elems(seed, TID_Q, b, idx).reshape(t1 - t0, H, D)


def qidx_rows(seed, b, t0, t1, G, Di):
    n = (t1 - t0) * G * Di
    idx = np.arange(n, dtype=np.uint64) + np.uint64(t0 * G * Di)
    return grid_elems(seed, TID_QIDX, b, idx).reshape(t1 - t0, G, Di)


def kv_blocks(seed, tid, b, blocks, G, D):
    """K (tid 2) or V (tid 3) cache blocks of sequence b: [len(blocks)][128][G][D]."""
    blocks = np.asarray(blocks, dtype=np.int64).reshape(-1)
    per = BLOCK * G * D
    idx = (blocks[:, None].astype(np.uint64) * np.uint64(per)
           + np.arange(per, dtype=np.uint64)[None, :])
    return normal_elems(seed, tid, b, idx).reshape(len(blocks), BLOCK, G, D)


def needles(seed, b, L, Di):
    """Needle (token, dim) pairs of sequence b whose whole context is L tokens."""
    nb = (L + BLOCK - 1) // BLOCK
    if nb < 2:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    qb = np.repeat(np.arange(1, nb, dtype=np.uint64), NEEDLES_PER_QBLOCK)
    n = np.arange(NEEDLES_PER_QBLOCK, nb * NEEDLES_PER_QBLOCK, dtype=np.uint64)
    tok = hashes(seed, TID_NEEDLE_TOK, b, n) % (qb * np.uint64(BLOCK))
    m = (n[:, None] * np.uint64(NEEDLE_DIMS)
         + np.arange(NEEDLE_DIMS, dtype=np.uint64)[None, :])
    dim = hashes(seed, TID_NEEDLE_DIM, b, m) % np.uint64(Di)
    toks = np.repeat(tok.astype(np.int64), NEEDLE_DIMS)
    return toks, dim.reshape(-1).astype(np.int64)


def kidx_seq(seed, b, L, Di, ntok=None):
    """K_idx of sequence b, [ntok][Di] bf16 bits (ntok >= L; rows >= L are grid
    values without needles).  L is the sequence's whole context length."""
    ntok = L if ntok is None else ntok
    idx = np.arange(ntok * Di, dtype=np.uint64)
    k = grid_elems(seed, TID_KIDX, b, idx).reshape(ntok, Di)
    toks, dims = needles(seed, b, L, Di)
    if toks.size:
        k[toks, dims] = f32_to_bf16_bits(np.array([NEEDLE_VALUE], np.float32))[0]
    return k


def kv_cache(seed, tid, b, nblocks, G, D):
    return kv_blocks(seed, tid, b, np.arange(nblocks), G, D)
