"""Pure-Python brute-force twin of the oracle, for tiny inputs only.

TEST INFRASTRUCTURE (same import rule as ``oracle/attention.py``).

It takes a different road to the same definition so that the two pin each
other: explicit triple loops over Python floats, the softmax normalised
without subtracting the row maximum, and the backward written with the full
softmax Jacobian ``dP_ij/dS_ik = P_ij (delta_jk - P_ik)`` instead of the
``D_i = rowsum(P * dP)`` shortcut used by ``attn_bwd_unit``.
Definition: SDPA tutorial page, section "Overview" (scaled dot-product
attention), causal mask from its "Causal Self Attention" section, top-left
aligned.
"""
from __future__ import annotations

import math

__all__ = ["fwd_bruteforce", "bwd_bruteforce"]


def _visible(i: int, j: int, is_causal: bool, allowed=None) -> bool:
    """Key j is visible to query i: causal (top-left) and, when given, the
    explicit set ``allowed`` of (i, j) pairs (block-sparse attention)."""
    if allowed is not None and (i, j) not in allowed:
        return False
    return (not is_causal) or j <= i


def _probs(q, k, scale, is_causal, allowed=None, bias=None):
    lq, lk, d = len(q), len(k), len(q[0]) if q else 0
    p = [[0.0] * lk for _ in range(lq)]
    lse = [0.0] * lq
    for i in range(lq):
        w = [0.0] * lk
        z = 0.0
        for j in range(lk):
            if _visible(i, j, is_causal, allowed):
                dot = 0.0
                for c in range(d):
                    dot += q[i][c] * k[j][c]
                sc = scale * dot + (0.0 if bias is None else bias[i][j])
                w[j] = 0.0 if sc == -math.inf else math.exp(sc)
                z += w[j]
        if z == 0.0:
            # no visible key (possible only with `allowed`): the row's
            # probabilities are all zero and its log-sum-exp is -inf
            lse[i] = -math.inf
            continue
        for j in range(lk):
            p[i][j] = w[j] / z
        lse[i] = math.log(z)
    return p, lse


def fwd_bruteforce(q, k, v, scale, is_causal=False, allowed=None, bias=None, drop=None):
    """q: list[Lq][d], k: list[Lk][d], v: list[Lk][dv] -> (O list[Lq][dv], LSE list[Lq]).
    ``allowed``: optional set of visible (query, key) index pairs; ``bias``:
    optional list[Lq][Lk] added to every score (-inf excludes it)."""
    p, lse = _probs(q, k, scale, is_causal, allowed, bias)
    dv = len(v[0])
    z = (lambda i, j: 1.0) if drop is None else (lambda i, j: drop[i][j])
    o = [[sum(p[i][j] * z(i, j) * v[j][c] for j in range(len(k))) for c in range(dv)] for i in range(len(q))]
    return o, lse


def bwd_bruteforce(q, k, v, do, scale, is_causal=False, allowed=None, bias=None, drop=None):
    """Gradients of sum(dO * O) by the explicit softmax Jacobian; ``drop``: the
    dropout factors that multiply P in O."""
    lq, lk, d, dv_ = len(q), len(k), len(q[0]), len(v[0])
    p, _ = _probs(q, k, scale, is_causal, allowed, bias)
    z = (lambda i, j: 1.0) if drop is None else (lambda i, j: drop[i][j])
    # dL/dP_ij = z_ij * sum_c dO_ic V_jc
    gp = [[z(i, j) * sum(do[i][c] * v[j][c] for c in range(dv_)) for j in range(lk)] for i in range(lq)]
    # dL/dS_ik = sum_j gp_ij * P_ij * (delta_jk - P_ik)
    gs = [[0.0] * lk for _ in range(lq)]
    for i in range(lq):
        for kk in range(lk):
            acc = 0.0
            for j in range(lk):
                jac = p[i][j] * ((1.0 if j == kk else 0.0) - p[i][kk])
                acc += gp[i][j] * jac
            gs[i][kk] = acc
    dq = [[scale * sum(gs[i][j] * k[j][c] for j in range(lk)) for c in range(d)] for i in range(lq)]
    dk = [[scale * sum(gs[i][j] * q[i][c] for i in range(lq)) for c in range(d)] for j in range(lk)]
    dv = [[sum(p[i][j] * z(i, j) * do[i][c] for i in range(lq)) for c in range(dv_)] for j in range(lk)]
    return dq, dk, dv
