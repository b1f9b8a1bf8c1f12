"""Temperature sampling for the oracle (test infrastructure only).

The pages name sampling and stopping only in passing (SGLang page,
Optimizations / Engineering Appendix: early-EOS divergence between attention
backends), with no parameters.  Reading taken: a frame's code k is drawn from
softmax(logits / T) by the Gumbel-max rule,

    code = argmax_i ( logits_i / T + G_i ),   G_i = -ln(-ln U_i),

with U_i from Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel random
numbers: as easy as 1, 2, 3", SC'11), key = (seed low 32 bits, seed high 32
bits) and counter = (i // 4, codebook k, position p of the slow step that
produced the frame, sequence id); word i % 4 of the output is used, mapped to
the odd multiples of 2^-24 in (0, 1).  T = 0 means greedy.

Top-p (nucleus) filtering, with no parameters on the pages either: with
scaled logits v = logits / T and p = softmax(v), sort v in descending order,
take the first k whose cumulative probability reaches top_p, and keep every
candidate whose v is at least the k-th largest value (ties at the cut are all
kept); the Gumbel-max draw is then taken over the kept candidates only.  An
equivalent statement, used as the check: candidate i is kept exactly when the
probability of the candidates strictly above it is below top_p.
"""

import numpy as np

TEST_ONLY = True

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds on arrays: ctr uint [..., 4], key uint [..., 2]."""
    c = np.asarray(ctr, dtype=np.uint64) & MASK
    k = np.asarray(key, dtype=np.uint64) & MASK
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0, k1 = k[..., 0], k[..., 1]
    for _ in range(10):
        p0 = np.uint64(M0) * c0
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + np.uint64(W0)) & np.uint64(MASK)
        k1 = (k1 + np.uint64(W1)) & np.uint64(MASK)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniforms(seed, seq, pos, codebook, n):
    """U_0 .. U_{n-1} in (0, 1) (float32, odd multiples of 2^-24)."""
    i = np.arange(n)
    blocks = np.arange((n + 3) // 4, dtype=np.uint64)
    ctr = np.stack([blocks, np.full_like(blocks, codebook), np.full_like(blocks, pos),
                    np.full_like(blocks, seq)], axis=-1)
    key = np.array([seed & MASK, (seed >> 32) & MASK], dtype=np.uint64)
    words = philox4x32_10(ctr, np.broadcast_to(key, ctr.shape[:-1] + (2,))).reshape(-1)[:n]
    odd = (words >> np.uint32(9)).astype(np.uint64) * np.uint64(2) + np.uint64(1)
    return (odd.astype(np.float64) * 2.0 ** -24).astype(np.float32)


def gumbel(seed, seq, pos, codebook, n):
    u = uniforms(seed, seq, pos, codebook, n)
    return -np.log(-np.log(u))


def nucleus(v, top_p):
    """Kept mask of top-p filtering over scaled logits v (probabilities in
    float64); top_p >= 1 keeps every candidate."""
    v = np.asarray(v, dtype=np.float64)
    if top_p >= 1.0:
        return np.ones(v.shape, bool)
    p = np.exp(v - v.max())
    p /= p.sum()
    order = np.argsort(-v, kind="stable")
    cum = np.cumsum(p[order])
    k = min(int(np.searchsorted(cum, top_p, side="left")), len(v) - 1)
    return v >= v[order[k]]


def pick(logits, temperature, top_p, seed, seq, pos, codebook):
    """Greedy for temperature 0 (lowest index on ties), else the Gumbel-max
    draw over the top-p nucleus of softmax(logits / T) (float32 scores)."""
    lg = np.asarray(logits, dtype=np.float32)
    if temperature <= 0:
        return int(np.argmax(lg))
    v = lg / np.float32(temperature)
    z = v + gumbel(seed, seq, pos, codebook, lg.shape[-1])
    z[~nucleus(v, top_p)] = -np.inf
    return int(np.argmax(z))


def sample(logits, temperature, seed, seq, pos, codebook):
    """Greedy for temperature 0, else the Gumbel-max draw (float32 decision)."""
    lg = np.asarray(logits, dtype=np.float32)
    if temperature <= 0:
        return int(np.argmax(lg))
    z = lg / np.float32(temperature) + gumbel(seed, seq, pos, codebook, lg.shape[-1])
    return int(np.argmax(z))
