"""Brute-force attention in high-precision decimal arithmetic.

Used only to pin the oracle on tiny inputs.  It takes a different route from
the oracle: Python's ``decimal`` module at 50 significant digits, no max
subtraction, every exponential computed directly, and its own gather of the
paged layout written with plain Python indexing.
"""
from __future__ import annotations

import decimal
from decimal import Decimal

import numpy as np

_CTX = decimal.Context(prec=50)


def attention_rows(q, K, V, scale):
    """softmax(scale * q.K_j) weighted sum of V_j, all in 50-digit decimal.

    q: sequence of D floats; K, V: sequences of ctx rows of D floats.
    Returns a list of D Python floats (rounded once at the end).
    """
    ctx = len(K)
    D = len(q)
    if ctx == 0:
        return [0.0] * D
    with decimal.localcontext(_CTX):
        sc = Decimal(float(scale))
        qd = [Decimal(float(x)) for x in q]
        weights = []
        for j in range(ctx):
            dot = sum((qd[d] * Decimal(float(K[j][d])) for d in range(D)), Decimal(0))
            weights.append((sc * dot).exp())
        total = sum(weights, Decimal(0))
        out = []
        for d in range(D):
            acc = sum((weights[j] * Decimal(float(V[j][d])) for j in range(ctx)), Decimal(0))
            out.append(float(acc / total))
    return out


def gather_logical(pool, block_tables, s, g, ctx, block_size):
    """Rows of kv head g for logical positions 0..ctx-1 of sequence s.

    pool: array-like [NB][Hkv][BS][D] of floats.
    """
    rows = []
    for pos in range(ctx):
        blk = int(block_tables[s][pos // block_size])
        rows.append([float(x) for x in pool[blk][g][pos % block_size]])
    return rows


def paged_decode(q, k_pool, v_pool, block_tables, context_lens, scale):
    """[S][H][D] float64 numpy array by brute force (tiny inputs only)."""
    q = np.asarray(q, dtype=np.float64)
    kp = np.asarray(k_pool, dtype=np.float64)
    vp = np.asarray(v_pool, dtype=np.float64)
    S, H, D = q.shape
    Hkv, BS = kp.shape[1], kp.shape[2]
    G = H // Hkv
    out = np.zeros((S, H, D))
    for s in range(S):
        ctx = int(context_lens[s])
        for h in range(H):
            g = h // G
            K = gather_logical(kp, block_tables, s, g, ctx, BS)
            V = gather_logical(vp, block_tables, s, g, ctx, BS)
            out[s, h] = attention_rows(q[s, h].tolist(), K, V, scale)
    return out
