"""Philox4x32-10 counter-based generator, written from its published definition.

TEST INFRASTRUCTURE: part of the CPU oracle. Only tests/, the smoke check and
the bench's CPU-baseline leg may import this module.

Definition followed: Salmon, Moraes, Dror & Shaw, "Parallel random numbers: as
easy as 1, 2, 3" (SC'11), section 3.2 (Philox): a 4x32 counter, a 2x32 key,
ten rounds; each round multiplies counter words 0 and 2 by the two Philox
multipliers, recombines the high/low halves with words 1 and 3 and the key,
and the key is bumped by the two Weyl constants between rounds.

The stream layout (which counter word carries what) is this project's reading
of the method's "counter RNG keyed by (seed, request, position)":
    key     = (seed & 0xffffffff, seed >> 32)
    counter = (c0, position & 0xffffffff, request, tag)
with c0 = vocab_id >> 2 for Gumbel draws (output word vocab_id & 3) and the
proposal index for residual draws.
"""
import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85

TAG_GUMBEL = 1
TAG_ACCEPT = 2
TAG_RESID = 3
TAG_BONUS = 4
TAG_MATCH = 5   # the target's own sample at each position (match verification)
TAG_HIST = 6    # synthetic history K/V of the history-KV control
TAG_TARGET = 7  # synthetic target tokens of the acceptance workloads
TAG_PICK = 8    # the draw inside the chosen vocabulary chunk (two-level sampling)
HIST_SEED = 0x4849535400000001   # fixed key of the synthetic history

_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10. Inputs broadcast; returns four uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK for c in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK
        p0 = m0 * c0          # 32x32 -> 64 bit products, exact in uint64
        p1 = m1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(np.asarray(c, dtype=np.uint32) for c in (c0, c1, c2, c3))


def seed_key(seed):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def uniform_open(x):
    """Map a 32-bit word to a uniform in the open interval (0, 1).

    Uses the top 23 bits: u = (floor(x / 2^9) + 1/2) / 2^23. Every value is
    exactly representable in float32 and float64, so both precisions agree.
    """
    x = np.asarray(x, dtype=np.uint64)
    return ((x >> np.uint64(9)).astype(np.float64) + 0.5) * (2.0 ** -23)


def draw(seed, c0, position, request, tag, word):
    """One uniform from word `word` of Philox(counter=(c0, pos, req, tag), key=seed)."""
    k0, k1 = seed_key(seed)
    out = philox4x32_10(c0, np.asarray(position, dtype=np.int64).astype(np.uint64) & _MASK,
                        request, tag, k0, k1)
    w = np.asarray(word)
    sel = np.choose(w, out) if w.ndim else out[int(w)]
    return uniform_open(sel)


def words(seed, c0, position, request, tag):
    """The four raw 32-bit words of Philox(counter=(c0, pos, req, tag), key=seed)."""
    k0, k1 = seed_key(seed)
    return philox4x32_10(c0, np.asarray(position, dtype=np.int64).astype(np.uint64) & _MASK,
                         request, tag, k0, k1)


def gumbel_row(seed, position, request, V):
    """Gumbel noise G_v = -log(-log u_v) for v = 0..V-1 of one draft slot."""
    v = np.arange(V, dtype=np.int64)
    k0, k1 = seed_key(seed)
    words = philox4x32_10(v >> 2, np.uint64(int(position) & 0xFFFFFFFF), request, TAG_GUMBEL, k0, k1)
    x = np.choose(v & 3, words)
    u = uniform_open(x)
    return -np.log(-np.log(u))
