"""Scalar, loop-by-loop restatement of BDLM attention for tiny inputs.

TEST INFRASTRUCTURE ONLY (see bdlm_oracle.py). It is written a second way, on
purpose: the visibility rule is stated per (query, key) pair from the roles
the paper gives (Block Parallelism abstract; rit.work CSBP post, first
section), and softmax is taken with math.exp over Python lists, so that the
vectorised oracle can be checked against it on sizes where loops finish.
"""
from __future__ import annotations

import math


def sees(i: int, j: int, n: int, block: int) -> bool:
    """Does query position i see key position j in one [clean | corrupted] sequence?"""
    q_is_clean, k_is_clean = i < n, j < n
    q_block = (i if q_is_clean else i - n) // block
    k_block = (j if k_is_clean else j - n) // block
    if q_is_clean:
        # autoregressive across clean blocks, all of its own block
        return k_is_clean and k_block <= q_block
    if k_is_clean:
        # the correct previous blocks only
        return k_block < q_block
    # its own noised block, bidirectionally
    return k_block == q_block


def forward(q, k, v, n, block, scale):
    """q [2n][H][d], k/v [2n][Hk][d] as nested lists or arrays; returns
    (o [2n][H][d], lse [H][2n]) as nested lists of floats."""
    T = 2 * n
    H, Hk, d = len(q[0]), len(k[0]), len(q[0][0])
    G = H // Hk
    o = [[[0.0] * d for _ in range(H)] for _ in range(T)]
    lse = [[-math.inf] * T for _ in range(H)]
    for h in range(H):
        g = h // G
        for i in range(T):
            logits = []
            for j in range(T):
                if sees(i, j, n, block):
                    dot = 0.0
                    for c in range(d):
                        dot += float(q[i][h][c]) * float(k[j][g][c])
                    logits.append((j, scale * dot))
            if not logits:
                continue
            top = max(x for _, x in logits)
            z = sum(math.exp(x - top) for _, x in logits)
            lse[h][i] = top + math.log(z)
            for j, x in logits:
                w = math.exp(x - top) / z
                for c in range(d):
                    o[i][h][c] += w * float(v[j][g][c])
    return o, lse
