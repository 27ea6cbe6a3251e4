"""Pins for the fp64 oracle: checks against what the mathematics fixes.

None of these retypes the oracle's formula. They compare it with a
brute-force twin that takes another road (explicit loops, no max shift, full
softmax Jacobian), with central finite differences, with closed forms and
invariants of the definition (SDPA tutorial page, section "Overview";
causal: section "Causal Self Attention"; packed batches: section
"NestedTensor and Dense tensor support"), and with the library's own math
path. The last block plants mistakes in copies of the oracle and checks that
the pins catch each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import (attention_probs, attn_bwd_ref, attn_bwd_unit, attn_fwd_ref,
                    attn_fwd_rows, attn_fwd_unit, bwd_bruteforce, dropout_keep, dropout_threshold,
                    expand_block_mask, fwd_bruteforce, philox4x32_10)
from exact_attention_softmax_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(*shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("lq,lk,d,causal", [
    (1, 1, 1, False), (3, 3, 8, False), (3, 3, 8, True), (2, 4, 3, False),
    (4, 2, 3, True), (4, 4, 5, True), (3, 1, 2, True)])
def test_fwd_matches_bruteforce(lq, lk, d, causal):
    q, k, v = rnd(lq, d, seed=1), rnd(lk, d, seed=2), rnd(lk, d + 1, seed=3)
    scale = 0.7
    o, lse = attn_fwd_unit(q, k, v, scale, causal)
    ob, lseb = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(lseb), rtol=0, atol=1e-13)


@pytest.mark.parametrize("lq,lk,d,causal", [
    (3, 3, 8, False), (3, 3, 8, True), (2, 4, 3, False), (4, 3, 2, True), (1, 3, 2, False)])
def test_bwd_matches_bruteforce_jacobian(lq, lk, d, causal):
    q, k, v, do = rnd(lq, d, seed=4), rnd(lk, d, seed=5), rnd(lk, d, seed=6), rnd(lq, d, seed=7)
    scale = 1 / math.sqrt(d)
    got = attn_bwd_unit(q, k, v, do, scale, causal)
    ref = bwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), do.tolist(), scale, causal)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, np.array(r), rtol=0, atol=1e-13)


# ---------------------------------------------------------- finite differences

def _fd_check(bwd, causal, seed=0, h=1e-6):
    """Central differences of L = sum(dO * O) against the analytic gradients on
    the tiny workload's shape (B=2, H=1, L=3, d=8)."""
    shp = (2, 1, 3, 8)
    q, k, v, do = (rnd(*shp, seed=seed + i) for i in range(4))
    scale = 1 / math.sqrt(8)

    def loss(q_, k_, v_):
        o, _ = attn_fwd_ref(q_, k_, v_, scale, causal)
        return float(np.sum(do * o))

    grads = bwd(q, k, v, do, scale, causal)
    worst = 0.0
    for which, g in enumerate(grads):
        args = [q, k, v]
        num = np.zeros_like(args[which])
        it = np.nditer(args[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            num[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(num), 1e-30)
        worst = max(worst, err)
    return worst


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_finite_differences(causal):
    assert _fd_check(attn_bwd_ref, causal) <= 1e-7


# ---------------------------------------------------------- invariants / forms

def test_probability_rows_sum_to_one():
    for causal in (False, True):
        p, _ = attention_probs(rnd(7, 5, seed=1), rnd(9, 5, seed=2), 0.4, causal)
        np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-14)
        assert np.all(p >= 0)
        if causal:
            assert np.all(np.triu(p, 1) == 0)


def test_single_key_gives_its_value_and_lse():
    q, k, v = rnd(5, 4, seed=1), rnd(1, 4, seed=2), rnd(1, 4, seed=3)
    o, lse = attn_fwd_unit(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.repeat(v, 5, 0), atol=1e-15)
    np.testing.assert_allclose(lse, 0.3 * (q @ k[0]), atol=1e-14)


def test_constant_values_give_constant_output():
    v = np.tile(rnd(1, 6, seed=3), (8, 1))
    for causal in (False, True):
        o, _ = attn_fwd_unit(rnd(8, 6, seed=1), rnd(8, 6, seed=2), v, 1.1, causal)
        np.testing.assert_allclose(o, np.tile(v[:1], (8, 1)), atol=1e-14)


def test_causal_first_row_sees_only_first_key():
    q, k, v = rnd(6, 4, seed=1), rnd(6, 4, seed=2), rnd(6, 4, seed=3)
    o, lse = attn_fwd_unit(q, k, v, 0.5, True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    assert abs(lse[0] - 0.5 * q[0] @ k[0]) < 1e-14


def test_zero_scale_gives_mean_and_log_count():
    q, k, v = rnd(5, 3, seed=1), rnd(7, 3, seed=2), rnd(7, 3, seed=3)
    o, lse = attn_fwd_unit(q, k, v, 0.0, False)
    np.testing.assert_allclose(o, np.tile(v.mean(0), (5, 1)), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(7), atol=1e-14)
    o, lse = attn_fwd_unit(q, k, v, 0.0, True)
    for i in range(5):
        np.testing.assert_allclose(o[i], v[: i + 1].mean(0), atol=1e-14)
        assert abs(lse[i] - math.log(i + 1)) < 1e-14


def test_two_keys_closed_form():
    q, k, v = rnd(4, 3, seed=1), rnd(2, 3, seed=2), rnd(2, 5, seed=3)
    sc = 0.8
    o, lse = attn_fwd_unit(q, k, v, sc, False)
    s = sc * q @ k.T
    sig = 1 / (1 + np.exp(-(s[:, 0] - s[:, 1])))
    np.testing.assert_allclose(o, sig[:, None] * v[0] + (1 - sig)[:, None] * v[1], atol=1e-14)
    np.testing.assert_allclose(lse, np.logaddexp(s[:, 0], s[:, 1]), atol=1e-14)


def test_key_shift_invariance():
    q, k, v = rnd(6, 4, seed=1), rnd(6, 4, seed=2), rnd(6, 4, seed=3)
    u = rnd(4, seed=9)
    for causal in (False, True):
        o, lse = attn_fwd_unit(q, k, v, 0.6, causal)
        o2, lse2 = attn_fwd_unit(q, k + u, v, 0.6, causal)
        np.testing.assert_allclose(o2, o, atol=1e-13)
        np.testing.assert_allclose(lse2, lse + 0.6 * q @ u, atol=1e-13)


def test_key_value_permutation_invariance():
    q, k, v = rnd(5, 4, seed=1), rnd(9, 4, seed=2), rnd(9, 3, seed=3)
    perm = np.random.default_rng(0).permutation(9)
    o, lse = attn_fwd_unit(q, k, v, 0.5, False)
    o2, lse2 = attn_fwd_unit(q, k[perm], v[perm], 0.5, False)
    np.testing.assert_allclose(o2, o, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, atol=1e-14)


def test_packed_equals_dense_per_sequence():
    lens = [3, 1, 5, 0, 2]
    H, d = 2, 4
    x = wl.varlen_inputs(lens, H, d, "f32", "normal", seed=3)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens"].numpy()
    for causal in (False, True):
        o, lse = attn_fwd_ref(q, k, v, 0.5, causal, cu)
        dq, dk, dv = attn_bwd_ref(q, k, v, do, 0.5, causal, cu)
        assert lse.shape == (H, sum(lens))
        for s in range(len(lens)):
            a, b = cu[s], cu[s + 1]
            for h in range(H):
                od, ld = attn_fwd_unit(q[a:b, h], k[a:b, h], v[a:b, h], 0.5, causal)
                np.testing.assert_array_equal(o[a:b, h], od)
                np.testing.assert_array_equal(lse[h, a:b], ld)
                g = attn_bwd_unit(q[a:b, h], k[a:b, h], v[a:b, h], do[a:b, h], 0.5, causal)
                np.testing.assert_array_equal(dq[a:b, h], g[0])
                np.testing.assert_array_equal(dk[a:b, h], g[1])
                np.testing.assert_array_equal(dv[a:b, h], g[2])


def _cross_bruteforce(q, k, v, do, cq, ck, scale, causal):
    """Per-sequence brute force for a packed cross-attention batch, written
    with explicit row lists so that it shares no slicing with the oracle."""
    H = q.shape[1]
    o, lse = np.zeros(q.shape), np.zeros((H, q.shape[0]))
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for s in range(len(cq) - 1):
        qrows = list(range(cq[s], cq[s + 1]))
        krows = list(range(ck[s], ck[s + 1]))
        if not qrows:
            continue
        for h in range(H):
            qs = [q[r, h].tolist() for r in qrows]
            ks = [k[r, h].tolist() for r in krows]
            vs = [v[r, h].tolist() for r in krows]
            ds = [do[r, h].tolist() for r in qrows]
            ob, lb = fwd_bruteforce(qs, ks, vs, scale, causal)
            gq, gk, gv = bwd_bruteforce(qs, ks, vs, ds, scale, causal)
            for i, r in enumerate(qrows):
                o[r, h], lse[h, r], dq[r, h] = ob[i], lb[i], gq[i]
            for j, r in enumerate(krows):
                dk[r, h], dv[r, h] = gk[j], gv[j]
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
def test_packed_cross_matches_bruteforce(causal):
    # queries and keys of unequal lengths on their own token axes, including
    # a sequence with keys but no queries (its dK, dV must stay zero)
    lq, lk = [2, 0, 4, 1, 3], [3, 2, 2, 5, 3]
    x = wl.varlen_cross_inputs(lq, lk, 2, 3, "f32", "normal", seed=11)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    cq, ck = x["cu_seqlens_q"].numpy(), x["cu_seqlens_k"].numpy()
    o, lse = attn_fwd_ref(q, k, v, 0.6, causal, cq, ck)
    grads = attn_bwd_ref(q, k, v, do, 0.6, causal, cq, ck)
    ref = _cross_bruteforce(q, k, v, do, cq.tolist(), ck.tolist(), 0.6, causal)
    for got, want in zip((o, lse) + tuple(grads), ref):
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)
    assert np.all(grads[1][ck[1]:ck[2]] == 0) and np.all(grads[2][ck[1]:ck[2]] == 0)


def test_packed_cross_with_shared_offsets_is_self_attention():
    lens = [3, 1, 5, 0, 2]
    x = wl.varlen_inputs(lens, 2, 4, "f32", "normal", seed=3)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens"].numpy()
    for causal in (False, True):
        a = attn_fwd_ref(q, k, v, 0.5, causal, cu) + attn_bwd_ref(q, k, v, do, 0.5, causal, cu)
        b = attn_fwd_ref(q, k, v, 0.5, causal, cu, cu.copy()) + attn_bwd_ref(q, k, v, do, 0.5, causal, cu, cu.copy())
        for x1, x2 in zip(a, b):
            np.testing.assert_array_equal(x1, x2)


@pytest.mark.parametrize("causal", [False, True])
def test_blhd_batch_is_packed_with_uniform_offsets(causal):
    # a [B, L, H, d] batch read through uniform offsets s*L equals the dense
    # [B, H, L, d] definition (queries and keys of different lengths)
    B, Lq, Lk, H, d = 3, 4, 6, 2, 3
    q, k, v, do = rnd(B, Lq, H, d, seed=1), rnd(B, Lk, H, d, seed=2), rnd(B, Lk, H, d, seed=3), rnd(B, Lq, H, d, seed=4)
    cq, ck = np.arange(B + 1) * Lq, np.arange(B + 1) * Lk
    flat = lambda t: t.reshape(-1, H, d)
    o, lse = attn_fwd_ref(flat(q), flat(k), flat(v), 0.5, causal, cq, ck)
    dq, dk, dv = attn_bwd_ref(flat(q), flat(k), flat(v), flat(do), 0.5, causal, cq, ck)
    T = lambda t: t.transpose(0, 2, 1, 3)   # [B, L, H, d] -> [B, H, L, d]
    od, lsed = attn_fwd_ref(T(q), T(k), T(v), 0.5, causal)
    gd = attn_bwd_ref(T(q), T(k), T(v), T(do), 0.5, causal)
    np.testing.assert_allclose(o.reshape(B, Lq, H, d), T(od), atol=1e-14)
    np.testing.assert_allclose(lse.reshape(H, B, Lq).transpose(1, 0, 2), lsed, atol=1e-14)
    for g, r, L in zip((dq, dk, dv), gd, (Lq, Lk, Lk)):
        np.testing.assert_allclose(g.reshape(B, L, H, d), T(r), atol=1e-14)


# ------------------------------------------------------------- block-sparse

def _allowed_pairs(bm, lq, lk, block):
    """Visible (i, j) pairs of a block mask, enumerated with plain loops."""
    out = set()
    for i in range(lq):
        for j in range(lk):
            if bm[i // block][j // block]:
                out.add((i, j))
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_matches_bruteforce(causal):
    # tiles of 2 on a 7 x 9 score matrix (ragged last tiles); row block 1 keeps
    # nothing, so its rows must come out empty
    lq, lk, d, blk = 7, 9, 3, 2
    bm = np.array([[1, 0, 1, 0, 1], [0, 0, 0, 0, 0], [0, 1, 1, 0, 0], [1, 0, 0, 1, 1]])
    q, k, v, do = rnd(lq, d, seed=31), rnd(lk, d, seed=32), rnd(lk, d, seed=33), rnd(lq, d, seed=34)
    o, lse = attn_fwd_ref(q[None], k[None], v[None], 0.7, causal, block_mask=bm, block_size=blk)
    grads = attn_bwd_ref(q[None], k[None], v[None], do[None], 0.7, causal, block_mask=bm, block_size=blk)
    allowed = _allowed_pairs(bm, lq, lk, blk)
    ob, lb = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.7, causal, allowed)
    gb = bwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), do.tolist(), 0.7, causal, allowed)
    np.testing.assert_allclose(o[0], np.array(ob), rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(lse[0]), np.isinf(np.array(lb)))
    fin = np.isfinite(lse[0])
    np.testing.assert_allclose(lse[0][fin], np.array(lb)[fin], rtol=0, atol=1e-13)
    for g, r in zip(grads, gb):
        np.testing.assert_allclose(g[0], np.array(r), rtol=0, atol=1e-13)
    # rows 2 and 3 (row block 1) see nothing: O = 0, LSE = -inf, no gradient
    assert np.all(o[0][2:4] == 0) and np.all(np.isneginf(lse[0][2:4])) and np.all(grads[0][0][2:4] == 0)


def test_block_mask_of_ones_is_plain_attention():
    q, k, v, do = rnd(2, 3, 10, 4, seed=1), rnd(2, 3, 6, 4, seed=2), rnd(2, 3, 6, 4, seed=3), rnd(2, 3, 10, 4, seed=4)
    for causal in (False, True):
        a = attn_fwd_ref(q, k, v, 0.5, causal) + attn_bwd_ref(q, k, v, do, 0.5, causal)
        b = (attn_fwd_ref(q, k, v, 0.5, causal, block_mask=np.ones((4, 2)), block_size=3)
             + attn_bwd_ref(q, k, v, do, 0.5, causal, block_mask=np.ones((4, 2)), block_size=3))
        for x1, x2 in zip(a, b):
            np.testing.assert_array_equal(x1, x2)


def test_block_diagonal_mask_is_independent_blocks():
    # a block-diagonal mask splits the sequence into independent pieces: each
    # equals plain attention over its own slice
    n, blk, d = 3, 4, 5
    q, k, v, do = (rnd(1, 2, n * blk, d, seed=s) for s in (5, 6, 7, 8))
    o, lse = attn_fwd_ref(q, k, v, 0.4, False, block_mask=np.eye(n), block_size=blk)
    dq, dk, dv = attn_bwd_ref(q, k, v, do, 0.4, False, block_mask=np.eye(n), block_size=blk)
    for h in range(2):
        for b in range(n):
            sl = slice(b * blk, (b + 1) * blk)
            od, ld = attn_fwd_unit(q[0, h, sl], k[0, h, sl], v[0, h, sl], 0.4)
            gd = attn_bwd_unit(q[0, h, sl], k[0, h, sl], v[0, h, sl], do[0, h, sl], 0.4)
            np.testing.assert_allclose(o[0, h, sl], od, atol=1e-14)
            np.testing.assert_allclose(lse[0, h, sl], ld, atol=1e-14)
            for g, r in zip((dq, dk, dv), gd):
                np.testing.assert_allclose(g[0, h, sl], r, atol=1e-14)


def test_block_sparse_backward_finite_differences():
    lq, lk, d, blk = 5, 6, 3, 2
    bm = np.array([[1, 1, 0], [0, 1, 1], [1, 0, 1]])
    q, k, v, do = rnd(lq, d, seed=41), rnd(lk, d, seed=42), rnd(lk, d, seed=43), rnd(lq, d, seed=44)
    dq, dk, dv = attn_bwd_ref(q, k, v, do, 0.6, True, block_mask=bm, block_size=blk)

    def loss(qq, kk, vv):
        o, _ = attn_fwd_ref(qq, kk, vv, 0.6, True, block_mask=bm, block_size=blk)
        return float(np.sum(do * o))
    h = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(num - g)) <= 1e-7 * max(1.0, np.max(np.abs(g)))


def test_expand_block_mask_shapes():
    bm = np.array([[1, 0], [0, 1], [1, 1]])
    full = expand_block_mask(bm, 5, 3, 2)
    assert full.shape == (5, 3)
    assert full[0].tolist() == [True, True, False] and full[2].tolist() == [False, False, True]
    assert full[4].tolist() == [True, True, True]
    with pytest.raises(ValueError):
        expand_block_mask(bm, 7, 3, 2)


# ------------------------------------------------------------ additive mask

@pytest.mark.parametrize("causal", [False, True])
def test_additive_mask_matches_bruteforce(causal):
    lq, lk, d = 5, 7, 3
    q, k, v, do = rnd(lq, d, seed=61), rnd(lk, d, seed=62), rnd(lk, d, seed=63), rnd(lq, d, seed=64)
    m = rnd(lq, lk, seed=65)
    m[1, :] = -np.inf              # an empty row
    m[3, [0, 4]] = -np.inf         # scattered exclusions
    o, lse = attn_fwd_ref(q[None], k[None], v[None], 0.8, causal, attn_mask=m)
    grads = attn_bwd_ref(q[None], k[None], v[None], do[None], 0.8, causal, attn_mask=m)
    ob, lb = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.8, causal, bias=m.tolist())
    gb = bwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), do.tolist(), 0.8, causal, bias=m.tolist())
    np.testing.assert_allclose(o[0], np.array(ob), rtol=0, atol=1e-13)
    fin = np.isfinite(np.array(lb))
    np.testing.assert_array_equal(np.isneginf(lse[0]), ~fin)
    np.testing.assert_allclose(lse[0][fin], np.array(lb)[fin], rtol=0, atol=1e-13)
    for g, r in zip(grads, gb):
        np.testing.assert_allclose(g[0], np.array(r), rtol=0, atol=1e-13)
    assert np.all(o[0][1] == 0) and np.isneginf(lse[0][1])


def test_additive_mask_special_cases():
    q, k, v, do = rnd(2, 3, 6, 4, seed=71), rnd(2, 3, 6, 4, seed=72), rnd(2, 3, 6, 4, seed=73), rnd(2, 3, 6, 4, seed=74)
    plain = attn_fwd_ref(q, k, v, 0.5, False) + attn_bwd_ref(q, k, v, do, 0.5, False)
    # a zero mask changes nothing
    zero = attn_fwd_ref(q, k, v, 0.5, False, attn_mask=np.zeros((6, 6))) + attn_bwd_ref(
        q, k, v, do, 0.5, False, attn_mask=np.zeros((6, 6)))
    for a, b in zip(plain, zero):
        np.testing.assert_array_equal(a, b)
    # -inf above the diagonal is the causal mask
    tri = np.where(np.arange(6)[None, :] > np.arange(6)[:, None], -np.inf, 0.0)
    caus = attn_fwd_ref(q, k, v, 0.5, True) + attn_bwd_ref(q, k, v, do, 0.5, True)
    viam = attn_fwd_ref(q, k, v, 0.5, False, attn_mask=tri) + attn_bwd_ref(q, k, v, do, 0.5, False, attn_mask=tri)
    for a, b in zip(caus, viam):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    # a constant shifts LSE by that constant and leaves O and the gradients alone
    sh = attn_fwd_ref(q, k, v, 0.5, False, attn_mask=np.full((6, 6), 2.5)) + attn_bwd_ref(
        q, k, v, do, 0.5, False, attn_mask=np.full((6, 6), 2.5))
    np.testing.assert_allclose(sh[0], plain[0], atol=1e-13)
    np.testing.assert_allclose(sh[1], plain[1] + 2.5, atol=1e-13)
    for a, b in zip(plain[2:], sh[2:]):
        np.testing.assert_allclose(a, b, atol=1e-12)
    # -inf on the last keys (padding) is attention over the first keys only
    pad = np.zeros((6, 6))
    pad[:, 4:] = -np.inf
    o, lse = attn_fwd_ref(q, k, v, 0.5, False, attn_mask=pad)
    o2, lse2 = attn_fwd_ref(q, k[..., :4, :], v[..., :4, :], 0.5, False)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)


def test_additive_mask_broadcast_axes():
    """A mask shared across the batch ([H, Lq, Lk]) or across heads
    ([B, 1, Lq, Lk]) reaches unit (b, h) as its own slice: each unit of the
    batched result equals a single-unit call with that slice, so a mask
    aligned against the wrong axis fails."""
    B, H, lq, lk, d = 2, 3, 5, 6, 4
    q, k, v, do = rnd(B, H, lq, d, seed=81), rnd(B, H, lk, d, seed=82), rnd(B, H, lk, d, seed=83), rnd(B, H, lq, d, seed=84)
    per_head = rnd(H, lq, lk, seed=85)
    per_batch = rnd(B, 1, lq, lk, seed=86)
    for mask, pick in ((per_head, lambda b, h: per_head[h]), (per_batch, lambda b, h: per_batch[b, 0])):
        full = attn_fwd_ref(q, k, v, 0.7, False, attn_mask=mask) + attn_bwd_ref(q, k, v, do, 0.7, False, attn_mask=mask)
        for b in range(B):
            for h in range(H):
                one = (attn_fwd_ref(q[b, h][None], k[b, h][None], v[b, h][None], 0.7, False, attn_mask=pick(b, h))
                       + attn_bwd_ref(q[b, h][None], k[b, h][None], v[b, h][None], do[b, h][None], 0.7, False,
                                      attn_mask=pick(b, h)))
                for a, r in zip(full, one):
                    np.testing.assert_allclose(a[b, h], r[0], rtol=0, atol=1e-13)
    # and the two layouts differ, so the check above can tell them apart
    a = attn_fwd_ref(q, k, v, 0.7, False, attn_mask=per_head)[0]
    c = attn_fwd_ref(q, k, v, 0.7, False, attn_mask=per_batch)[0]
    assert np.max(np.abs(a - c)) > 1e-3


def test_additive_mask_backward_finite_differences():
    lq, lk, d = 4, 5, 3
    q, k, v, do = rnd(lq, d, seed=81), rnd(lk, d, seed=82), rnd(lk, d, seed=83), rnd(lq, d, seed=84)
    m = rnd(lq, lk, seed=85)
    dq, dk, dv = attn_bwd_ref(q, k, v, do, 0.6, False, attn_mask=m)

    def loss(qq, kk, vv):
        o, _ = attn_fwd_ref(qq, kk, vv, 0.6, False, attn_mask=m)
        return float(np.sum(do * o))
    h = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap, am = [q, k, v], [q, k, v]
            ap[which], am[which] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        assert np.max(np.abs(num - g)) <= 1e-7 * max(1.0, np.max(np.abs(g)))


# ------------------------------------------------------------------ dropout

def test_philox_known_answers():
    kat = json.load(open(os.path.join(HERE, "golden", "philox_kat.json")))
    for vec in kat["vectors"]:
        ctr = np.array([int(x, 16) for x in vec["counter"]], dtype=np.uint32)
        key = np.array([int(x, 16) for x in vec["key"]], dtype=np.uint32)
        out = philox4x32_10(ctr, key)
        assert [f"{int(w):08x}" for w in out] == vec["output"]


def _philox_scalar(ctr, key):
    """Philox4x32-10 for one counter, in plain Python integers: a second
    statement of the SC 2011 generator (ten rounds; each multiplies counter
    words 0 and 2 by 0xD2511F53 and 0xCD9E8D57, splits the 64-bit products
    into high and low words, and xors the high words with the other two
    counter words and the round key; the key advances by 0x9E3779B9 and
    0xBB67AE85 after every round but the last)."""
    x0, x1, x2, x3 = ctr
    k0, k1 = key
    for rnd_ in range(10):
        p0, p1 = 0xD2511F53 * x0, 0xCD9E8D57 * x2
        x0, x1, x2, x3 = ((p1 >> 32) ^ x1 ^ k0, p1 & 0xFFFFFFFF, (p0 >> 32) ^ x3 ^ k1, p0 & 0xFFFFFFFF)
        if rnd_ < 9:
            k0, k1 = (k0 + 0x9E3779B9) & 0xFFFFFFFF, (k1 + 0xBB67AE85) & 0xFFFFFFFF
    return x0, x1, x2, x3


def test_scalar_philox_known_answers():
    kat = json.load(open(os.path.join(HERE, "golden", "philox_kat.json")))
    for vec in kat["vectors"]:
        out = _philox_scalar([int(x, 16) for x in vec["counter"]], [int(x, 16) for x in vec["key"]])
        assert [f"{w:08x}" for w in out] == vec["output"]


def test_dropout_keep_bytes_from_published_vector():
    """Keep bits read by hand off Random123's first vector (counter 0, key 0):
    byte order within a word, the >= comparison and t = round(256 p)."""
    g = json.load(open(os.path.join(HERE, "golden", "dropout_keep_kat.json")))
    for case in g["cases"]:
        p = case["t"] / 256.0
        assert dropout_threshold(p) == case["t"]
        keep = dropout_keep(g["seed"], g["unit"], 1, 16, p)[0]
        assert keep.astype(int).tolist() == case["keep"], case["why"]


@pytest.mark.parametrize("seed", [0, 0x9E3779B97F4A7C15, (5 << 32) | 7])
def test_dropout_keep_one_counter_at_a_time(seed):
    """The vectorised keep mask against an explicit loop: for each score
    (i, j) of unit u, one Philox call at counter (j // 16, i, u, 0) with key
    (seed mod 2^32, seed div 2^32), then byte j mod 16 taken by shifting the
    word j mod 16 div 4 right by 8 (j mod 4) bits. Keys cross the 16- and
    32-key counter steps; rows and units differ so a swapped counter word or
    key word shows."""
    lq, lk, t = 5, 41, 77
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for u in (0, 3):
        got = dropout_keep(seed, u, lq, lk, t / 256.0)
        want = np.zeros((lq, lk), dtype=bool)
        for i in range(lq):
            for j in range(lk):
                words = _philox_scalar((j // 16, i, u, 0), key)
                byte = (words[(j % 16) // 4] >> (8 * (j % 4))) & 0xFF
                want[i, j] = byte >= t
        assert np.array_equal(got, want)
    # the unit and the row are different counter words
    assert not np.array_equal(dropout_keep(seed, 1, 2, 32, 0.5)[0], dropout_keep(seed, 0, 2, 32, 0.5)[1])


def test_dropout_keep_rate_and_independence():
    for p in (0.1, 0.5, 0.9):
        keep = dropout_keep(1234, 3, 256, 512, p)
        rate = 1.0 - dropout_threshold(p) / 256.0
        n = keep.size
        assert abs(keep.mean() - rate) < 6.0 * np.sqrt(rate * (1 - rate) / n)
    a = dropout_keep(7, 0, 64, 64, 0.5)
    b = dropout_keep(7, 1, 64, 64, 0.5)
    c = dropout_keep(8, 0, 64, 64, 0.5)
    assert (a != b).mean() > 0.3 and (a != c).mean() > 0.3
    assert np.array_equal(a, dropout_keep(7, 0, 64, 64, 0.5))     # deterministic
    assert dropout_keep(7, 0, 8, 8, 0.0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_matches_bruteforce(causal):
    lq, lk, d, p, seed = 6, 21, 3, 0.3, 99
    q, k, v, do = rnd(lq, d, seed=101), rnd(lk, d, seed=102), rnd(lk, d, seed=103), rnd(lq, d, seed=104)
    o, lse = attn_fwd_ref(q[None], k[None], v[None], 0.7, causal, dropout_p=p, dropout_seed=seed)
    grads = attn_bwd_ref(q[None], k[None], v[None], do[None], 0.7, causal, dropout_p=p, dropout_seed=seed)
    z = dropout_keep(seed, 0, lq, lk, p) * (256.0 / (256.0 - dropout_threshold(p)))
    ob, lb = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.7, causal, drop=z.tolist())
    gb = bwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), do.tolist(), 0.7, causal, drop=z.tolist())
    np.testing.assert_allclose(o[0], np.array(ob), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], np.array(lb), rtol=0, atol=1e-13)   # LSE ignores dropout
    for g, r in zip(grads, gb):
        np.testing.assert_allclose(g[0], np.array(r), rtol=0, atol=1e-13)
    plain = attn_fwd_ref(q[None], k[None], v[None], 0.7, causal)
    np.testing.assert_array_equal(plain[1], lse)
    zero = attn_fwd_ref(q[None], k[None], v[None], 0.7, causal, dropout_p=0.0, dropout_seed=seed)
    np.testing.assert_array_equal(plain[0], zero[0])


def test_dropout_backward_finite_differences():
    lq, lk, d = 4, 18, 3
    q, k, v, do = rnd(lq, d, seed=111), rnd(lk, d, seed=112), rnd(lk, d, seed=113), rnd(lq, d, seed=114)
    kw = dict(dropout_p=0.4, dropout_seed=5)
    dq, dk, dv = attn_bwd_ref(q, k, v, do, 0.6, False, **kw)

    def loss(qq, kk, vv):
        o, _ = attn_fwd_ref(qq, kk, vv, 0.6, False, **kw)
        return float(np.sum(do * o))
    h = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap, am = [q, k, v], [q, k, v]
            ap[which], am[which] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        assert np.max(np.abs(num - g)) <= 1e-7 * max(1.0, np.max(np.abs(g)))


def test_rows_helper_matches_full_unit():
    q, k, v = rnd(10, 4, seed=1), rnd(10, 4, seed=2), rnd(10, 4, seed=3)
    rows = np.array([0, 3, 9])
    for causal in (False, True):
        o, lse = attn_fwd_unit(q, k, v, 0.5, causal)
        o2, lse2 = attn_fwd_rows(q[rows], k, v, rows, 0.5, causal)
        np.testing.assert_allclose(o2, o[rows], atol=1e-14)
        np.testing.assert_allclose(lse2, lse[rows], atol=1e-14)


def test_backward_invariants():
    q, k, v, do = rnd(6, 4, seed=1), rnd(8, 4, seed=2), rnd(8, 4, seed=3), rnd(6, 4, seed=4)
    for causal in (False, True):
        dq, dk, dv = attn_bwd_unit(q, k, v, do, 0.5, causal)
        # softmax Jacobian rows sum to zero: the key gradients sum to zero
        np.testing.assert_allclose(dk.sum(0), 0, atol=1e-13)
        # P rows sum to one: value gradients sum to the summed output gradient
        np.testing.assert_allclose(dv.sum(0), do.sum(0), atol=1e-13)
        # a common shift of the keys leaves every gradient unchanged
        g2 = attn_bwd_unit(q, k + rnd(4, seed=5), v, do, 0.5, causal)
        for a, b in zip((dq, dk, dv), g2):
            np.testing.assert_allclose(b, a, atol=1e-12)
        # linear in dO
        g3 = attn_bwd_unit(q, k, v, -2.5 * do, 0.5, causal)
        for a, b in zip((dq, dk, dv), g3):
            np.testing.assert_allclose(b, -2.5 * a, atol=1e-12)


def test_empty_and_invalid_units():
    o, lse = attn_fwd_unit(np.zeros((0, 4)), rnd(3, 4), rnd(3, 4), 1.0)
    assert o.shape == (0, 4) and lse.shape == (0,)
    with pytest.raises(ValueError):
        attn_fwd_unit(rnd(2, 4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    with pytest.raises(ValueError):
        attn_fwd_ref(rnd(4, 1, 2), rnd(4, 1, 2), rnd(4, 1, 2), 1.0, cu_seqlens=[0, 3])


# ------------------------------------------------------ library cross-check

@pytest.mark.parametrize("lq,lk,causal", [(5, 5, False), (5, 5, True), (3, 7, True), (7, 3, True)])
def test_matches_library_math_path(lq, lk, causal):
    g = torch.Generator().manual_seed(0)
    q = torch.randn(2, 3, lq, 8, generator=g, dtype=torch.float64, requires_grad=True)
    k = torch.randn(2, 3, lk, 8, generator=g, dtype=torch.float64, requires_grad=True)
    v = torch.randn(2, 3, lk, 8, generator=g, dtype=torch.float64, requires_grad=True)
    do = torch.randn(2, 3, lq, 8, generator=g, dtype=torch.float64)
    o_t = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=0.35)
    o_t.backward(do)
    o, _ = attn_fwd_ref(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), 0.35, causal)
    np.testing.assert_allclose(o, o_t.detach().numpy(), atol=1e-12)
    dq, dk, dv = attn_bwd_ref(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(),
                              do.numpy(), 0.35, causal)
    np.testing.assert_allclose(dq, q.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, k.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, v.grad.numpy(), atol=1e-12)


# ------------------------------------------------------------ golden fixture

def test_golden_tiny_workload():
    """Stored oracle outputs for the tiny workload (written by
    tests/golden/make_golden.py, which calls only the oracle)."""
    with open(os.path.join(HERE, "golden", "tiny_f32.json")) as f:
        gold = json.load(f)
    x = wl.workload_inputs(wl.WORKLOADS["tiny_f32"], seed=gold["seed"])
    for n in ("q", "k", "v", "do"):
        np.testing.assert_array_equal(x[n].reshape(-1).numpy(), np.array(gold["inputs"][n], np.float32))
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    o, lse = attn_fwd_ref(q, k, v, gold["scale"], False)
    dq, dk, dv = attn_bwd_ref(q, k, v, do, gold["scale"], False)
    for name, val in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(val.reshape(-1), np.array(gold["outputs"][name]), rtol=0, atol=1e-14)


# ------------------------------------------------ planted mistakes get caught

def _bwd_mut(kind):
    def bwd(q, k, v, do, scale, causal):
        qu, ku, vu, du = (x.reshape((-1,) + x.shape[-2:]) for x in (q, k, v, do))
        outs = [np.empty_like(qu), np.empty_like(ku), np.empty_like(vu)]
        for u in range(qu.shape[0]):
            p, _ = attention_probs(qu[u], ku[u], scale, causal)
            dv = p.T @ du[u]
            dp = du[u] @ vu[u].T
            dsum = np.sum(p * dp, axis=1, keepdims=True)
            if kind == "D_sign":
                ds = p * (dp + dsum)
            elif kind == "D_axis":
                ds = p * (dp - np.sum(p * dp, axis=0, keepdims=True))
            else:
                ds = p * (dp - dsum)
            dq = scale * (ds @ ku[u])
            dk = scale * (ds.T @ qu[u])
            if kind == "no_scale":
                dq = ds @ ku[u]
            if kind == "dv_transpose":
                dv = p @ du[u]  # P used untransposed (square units only)
            outs[0][u], outs[1][u], outs[2][u] = dq, dk, dv
        return tuple(o.reshape(x.shape) for o, x in zip(outs, (q, k, v)))
    return bwd


@pytest.mark.parametrize("kind", ["D_sign", "D_axis", "no_scale", "dv_transpose"])
def test_finite_differences_catch_planted_backward_mistakes(kind):
    assert _fd_check(_bwd_mut(kind), causal=True) > 1e-3


def test_cross_bruteforce_catches_keys_read_at_query_offsets():
    # a packed cross-attention oracle that slices keys with the query offsets
    lq, lk = [2, 3], [4, 1]
    x = wl.varlen_cross_inputs(lq, lk, 1, 3, "f32", "normal", seed=5)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    cq, ck = x["cu_seqlens_q"].numpy().tolist(), x["cu_seqlens_k"].numpy().tolist()
    wrong = np.zeros(q.shape)
    for s in range(2):
        a, b = cq[s], cq[s + 1]
        wrong[a:b, 0], _ = attn_fwd_unit(q[a:b, 0], k[a:b, 0], v[a:b, 0], 0.5, False)
    ob = _cross_bruteforce(q, k, v, do, cq, ck, 0.5, False)[0]
    assert np.max(np.abs(wrong - ob)) > 1e-3


def test_bruteforce_catches_transposed_block_mask():
    # an oracle that applied the block mask transposed (key blocks as rows)
    lq = lk = 6
    bm = np.array([[1, 0, 0], [1, 1, 0], [0, 1, 1]])
    q, k, v = rnd(lq, 3, seed=51), rnd(lk, 3, seed=52), rnd(lk, 3, seed=53)
    wrong, _ = attn_fwd_ref(q[None], k[None], v[None], 0.5, False, block_mask=bm.T, block_size=2)
    ob, _ = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.5, False, _allowed_pairs(bm, lq, lk, 2))
    assert np.max(np.abs(wrong[0] - np.array(ob))) > 1e-3


def test_bruteforce_catches_mask_added_before_the_scale():
    # an oracle that scaled the mask along with Q K^T
    q, k, v = rnd(4, 3, seed=91), rnd(5, 3, seed=92), rnd(5, 3, seed=93)
    m = rnd(4, 5, seed=94)
    wrong, _ = attn_fwd_unit(q, k, v, 0.3, False, bias=m * 0.3)
    ob, _ = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.3, False, bias=m.tolist())
    assert np.max(np.abs(wrong - np.array(ob))) > 1e-3


def test_bruteforce_catches_dropout_in_the_normaliser():
    # an oracle that renormalised over the kept probabilities
    lq, lk = 4, 16
    q, k, v = rnd(lq, 3, seed=121), rnd(lk, 3, seed=122), rnd(lk, 3, seed=123)
    keep = dropout_keep(3, 0, lq, lk, 0.5)
    p, _ = attention_probs(q, k, 0.5)
    pk = p * keep
    wrong = (pk / pk.sum(1, keepdims=True)) @ v
    z = keep * (256.0 / (256.0 - dropout_threshold(0.5)))
    ob, _ = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.5, False, drop=z.tolist())
    assert np.max(np.abs(wrong - np.array(ob))) > 1e-3


def test_bruteforce_catches_planted_mask_mistake():
    q, k, v = rnd(4, 3, seed=1), rnd(4, 3, seed=2), rnd(4, 3, seed=3)
    s = 0.5 * q @ k.T
    s = np.where(np.arange(4)[None, :] >= np.arange(4)[:, None], -np.inf, s)  # j >= i: wrong
    s[0, 0] = 0.5 * q[0] @ k[0]
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ob, _ = fwd_bruteforce(q.tolist(), k.tolist(), v.tolist(), 0.5, True)
    assert np.max(np.abs(p @ v - np.array(ob))) > 1e-3


def _keep_variant(seed, unit, lq, lk, t, order="<u4", counter=lambda g, i, u: (g, i, u, 0), cmp=np.greater_equal):
    """A copy of the keep-mask construction with one planted change."""
    groups = -(-lk // 16)
    ctr = np.array([[counter(g, i, unit) for g in range(groups)] for i in range(lq)], dtype=np.uint32)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
    words = philox4x32_10(ctr, key).astype(np.uint32)
    by = words.astype(order).view(np.uint8).reshape(lq, groups * 16)[:, :lk]
    return cmp(by, t)


def test_dropout_pins_catch_planted_mistakes():
    g = json.load(open(os.path.join(HERE, "golden", "dropout_keep_kat.json")))
    # the unchanged copy passes both pins
    for case in g["cases"]:
        assert _keep_variant(0, 0, 1, 16, case["t"])[0].astype(int).tolist() == case["keep"]
    # big-endian bytes, and > instead of >=: the published-vector bytes catch them
    caught = [any(_keep_variant(0, 0, 1, 16, c["t"], **kw)[0].astype(int).tolist() != c["keep"] for c in g["cases"])
              for kw in (dict(order=">u4"), dict(cmp=np.greater))]
    assert all(caught)
    # row and unit swapped in the counter: the one-counter-at-a-time loop catches it
    seed = (5 << 32) | 7
    wrong = _keep_variant(seed, 3, 5, 41, 77, counter=lambda g_, i, u: (g_, u, i, 0))
    assert not np.array_equal(wrong, dropout_keep(seed, 3, 5, 41, 77 / 256.0))
