"""A second, independent re-statement of the verify step in pure Python (tiny inputs only).

Used to cross-check the C++ oracle token for token on many random tiny cases. It is written
from the same definitions (speculative-decoding explainer, section "修正拒绝采样"; Philox4x32-10
from Salmon et al., SC'11) but shares no code with the oracle. fp32 operations are done with
numpy float32 scalars, one IEEE round-to-nearest operation each.
"""

import math

import numpy as np

MASK32 = 0xFFFFFFFF


def philox(c, k):
    c = list(c)
    k0, k1 = k
    for _ in range(10):
        p0 = 0xD2511F53 * c[0]
        p1 = 0xCD9E8D57 * c[2]
        c = [((p1 >> 32) ^ c[1] ^ k0) & MASK32, p1 & MASK32,
             ((p0 >> 32) ^ c[3] ^ k1) & MASK32, p0 & MASK32]
        k0 = (k0 + 0x9E3779B9) & MASK32
        k1 = (k1 + 0xBB67AE85) & MASK32
    return c


def key_of(seed):
    return (seed & MASK32, (seed >> 32) & MASK32)


def u_accept(seed, r, j):
    w = philox((0, j, r, 0), key_of(seed))[0]
    return (w >> 8) / float(1 << 24)


def e_race(seed, r, j, x):
    w = philox((x >> 2, j, r, 1), key_of(seed))[x & 3]
    return np.float32(-math.log((w + 0.5) / 4294967296.0))


def race(p, q, seed, r, j):
    best, best_x = np.float32(-1.0), 0
    for x in range(len(p)):
        d = np.float32(p[x]) - (np.float32(q[x]) if q is not None else np.float32(0.0))
        res = d if d > 0 else np.float32(0.0)
        key = np.float32(res / e_race(seed, r, j, x))
        if key > best:
            best, best_x = key, x
    return best_x if best > 0 else -1


def verify_one(p_rows, q_rows, drafts, greedy, seed, r):
    """p_rows [K+1, V], q_rows [K, V] float32; returns (a, out_tokens list)."""
    K = len(drafts)
    V = p_rows.shape[1]
    a = K
    for j in range(K):
        d = int(drafts[j])
        if d < 0 or d >= V:
            a = j
            break
        if greedy:
            ok = int(np.argmax(p_rows[j])) == d
        else:
            ok = u_accept(seed, r, j) * float(q_rows[j][d]) < float(p_rows[j][d])
        if not ok:
            a = j
            break
    if greedy:
        b = int(np.argmax(p_rows[a]))
    elif a < K:
        b = race(p_rows[a], q_rows[a], seed, r, a)
        if b < 0:
            b = race(p_rows[a], None, seed, r, a)
    else:
        b = race(p_rows[K], None, seed, r, K)
    if b < 0:
        b = 0
    toks = [int(drafts[t]) if t < a else (b if t == a else -1) for t in range(K + 1)]
    return a, toks
