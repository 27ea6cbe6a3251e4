"""fp64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import or
run anything in ``oracle/``. The CUDA library never links it and the Python
binding never imports it; it shares no code, header, table or helper with the
GPU path.

What it computes is the plain definition, materialised, in float64:

* Forward -- the SDPA tutorial page ("(Beta) Implementing High-Performance
  Transformers with Scaled Dot Product Attention", section "Overview") defines
  the op as the scaled dot-product attention of "Attention Is All You Need":
  ``O = softmax(scale * Q K^T [+ causal mask]) V``; the same page, section
  "Causal Self Attention", passes ``is_causal`` to it.  The FlashAttention
  news article (QbitAI repost, section "FlashAttention") states that the tiled
  algorithm is *exact*, so the un-tiled definition is the oracle.
* The per-row log-sum-exp ``LSE_i = log sum_j exp(S_ij)`` (natural log) is
  what an IO-aware forward saves for the recomputing backward (same article,
  same section: attention is recomputed in the backward pass). The pages do
  not print it; this is the plainest reading of "recompute".
* Backward -- calculus on the definition (the pages only say the backward
  recomputes attention): with P the probabilities and dO the output gradient,
  ``dV = P^T dO``, ``dP = dO V^T``, ``D_i = sum_j P_ij dP_ij``,
  ``dS = P * (dP - D)``, ``dQ = scale dS K``, ``dK = scale dS^T Q``.

Readings taken where the pages are silent (each listed in the design notes):
causal masking is top-left aligned (key j is visible to query i iff j <= i);
``scale`` is always passed explicitly; LSE is natural-log, fp32 on the GPU,
shape ``[B, H, Lq]`` dense and ``[H, total]`` packed; a unit with Lq = 0
yields empty outputs; Lk = 0 with Lq > 0 is an error.

Block-sparse attention (the FlashAttention article's "block-sparse
FlashAttention", section "FlashAttention", which it only names): the
attention of the plain definition restricted to the (query block, key block)
tiles a 0/1 block mask keeps; every other score is excluded like a causally
masked one. Reading taken where the article is silent: a query row left with
no visible key gets O = 0 and LSE = -inf (and no gradient).

Additive mask (the SDPA tutorial's ``attn_mask`` argument, section "Causal
Self Attention", which passes ``None``): a float matrix M added to the scaled
scores, ``softmax(scale * Q K^T + M)``; -inf entries exclude a score, and a
row left with no finite score is empty as above.

Dropout (the tutorial's ``dropout_p`` argument of the same call): the
probabilities, not the normaliser, are dropped; O = (P * Z) V with Z = 0 for a
dropped score and 1/(1 - t/256) for a kept one, where t = round(256 p) is the
byte threshold of the keep test (so the realised drop rate is t/256, which
equals p when p is a multiple of 1/256), and LSE that of the full softmax.
The keep pattern comes from Philox4x32-10 (``oracle/philox.py``).

Layouts: dense tensors are ``[..., L, d]`` (any leading batch/head dims, the
tutorial's ``[B, H, L, d]`` and its ``[2, 3, 8]`` example both fit); packed
variable-length tensors (the tutorial's NestedTensor section) are
``[total, H, d]`` with ``cu_seqlens`` of length ``nseq + 1``; the same
offsets serve queries and keys (self-attention) unless ``cu_seqlens_k`` gives
the keys their own offsets on their own token axis (cross-attention: k/v
``[total_k, H, d]``; query i of a sequence sees that sequence's keys, causal
ones j <= i as in the dense case). A ``[B, L, H, d]`` batch is the packed
case with offsets ``s * L``.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "attention_probs",
    "attn_fwd_unit",
    "attn_bwd_unit",
    "attn_fwd_ref",
    "attn_bwd_ref",
    "attn_fwd_rows",
    "expand_block_mask",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _scores(q: np.ndarray, k: np.ndarray, scale: float, is_causal: bool, visible=None, bias=None) -> np.ndarray:
    """S = scale * Q K^T [+ bias] with masked entries set to -inf (SDPA tutorial,
    "Overview"; causal mask: "Causal Self Attention"; ``visible``: an extra
    [Lq, Lk] boolean mask, e.g. a block-sparse pattern; ``bias``: an additive
    [Lq, Lk] mask)."""
    s = float(scale) * (q @ k.T)
    if bias is not None:
        s = s + _f64(bias)
    if visible is not None:
        s = np.where(visible, s, -np.inf)
    if is_causal:
        lq, lk = s.shape
        i = np.arange(lq)[:, None]
        j = np.arange(lk)[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def attention_probs(q, k, scale: float, is_causal: bool = False, visible=None, bias=None):
    """P = softmax_j(S_ij) and LSE_i for one (batch, head) unit.

    ``q``: [Lq, d], ``k``: [Lk, d]. Returns ``(P [Lq, Lk], LSE [Lq])`` in float64.
    The row maximum is subtracted before exponentiating (a rounding measure
    only; softmax is shift invariant). ``visible`` ([Lq, Lk] bool, optional)
    excludes further scores; a row it leaves empty gets P = 0, LSE = -inf.
    """
    q, k = _f64(q), _f64(k)
    lq, lk = q.shape[0], k.shape[0]
    if lq == 0:
        return np.zeros((0, lk)), np.zeros((0,))
    if lk == 0:
        raise ValueError("softmax over an empty key set is undefined (Lk = 0 with Lq > 0)")
    s = _scores(q, k, scale, is_causal, visible, bias)
    m = np.max(s, axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m)
    z = np.sum(e, axis=1, keepdims=True)
    p = e / np.where(z > 0, z, 1.0)
    with np.errstate(divide="ignore"):
        lse = (m + np.log(z))[:, 0]
    lse[empty] = -np.inf
    return p, lse


def attn_fwd_unit(q, k, v, scale: float, is_causal: bool = False, visible=None, bias=None, drop=None):
    """O = P V and LSE for one unit. ``v``: [Lk, dv]. Returns (O [Lq, dv], LSE [Lq]).
    ``drop`` ([Lq, Lk], optional): dropout factors Z multiplying P in O only."""
    v = _f64(v)
    p, lse = attention_probs(q, k, scale, is_causal, visible, bias)
    if drop is not None:
        p = p * drop
    return p @ v, lse


def attn_bwd_unit(q, k, v, do, scale: float, is_causal: bool = False, visible=None, bias=None, drop=None):
    """Gradients of sum(dO * O) w.r.t. Q, K, V for one unit (chain rule through
    the softmax; the pages only say the backward recomputes attention)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    if q.shape[0] == 0:
        return np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    p, _ = attention_probs(q, k, scale, is_causal, visible, bias)
    z = np.ones_like(p) if drop is None else _f64(drop)
    dv = (p * z).T @ do
    dp = (do @ v.T) * z                      # gradient with respect to P
    dsum = np.sum(p * dp, axis=1, keepdims=True)
    ds = p * (dp - dsum)
    dq = float(scale) * (ds @ k)
    dk = float(scale) * (ds.T @ q)
    return dq, dk, dv


def _units_dense(x: np.ndarray) -> np.ndarray:
    return x.reshape((-1,) + x.shape[-2:])


def expand_block_mask(block_mask, lq: int, lk: int, block: int = 128) -> np.ndarray:
    """[..., ceil(Lq/block), ceil(Lk/block)] 0/1 block mask -> [..., Lq, Lk]
    booleans: score (i, j) is kept iff its tile (i // block, j // block) is."""
    bm = np.asarray(block_mask) != 0
    nq, nk = -(-lq // block), -(-lk // block)
    if bm.shape[-2:] != (nq, nk):
        raise ValueError(f"block mask must end in ({nq}, {nk}) for Lq={lq}, Lk={lk}, block={block}")
    rows = np.arange(lq) // block
    cols = np.arange(lk) // block
    return bm[..., rows, :][..., :, cols]


def _unit_masks(block_mask, lead, lq, lk, block):
    """Per-unit [Lq, Lk] masks for a dense batch with leading dims ``lead``."""
    if block_mask is None:
        return None
    full = expand_block_mask(block_mask, lq, lk, block)
    full = np.broadcast_to(full, tuple(lead) + (lq, lk))
    return full.reshape((-1, lq, lk))


def _check_cu(cu_seqlens, total: int) -> np.ndarray:
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] != total:
        raise ValueError("cu_seqlens must start at 0, be non-decreasing and end at the packed length")
    return cu


def _packed_spans(cu_seqlens, cu_seqlens_k, total_q: int, total_k: int):
    """Per sequence: (query rows a:b, key rows c:e)."""
    cq = _check_cu(cu_seqlens, total_q)
    ck = cq if cu_seqlens_k is None else _check_cu(cu_seqlens_k, total_k)
    if ck.size != cq.size:
        raise ValueError("cu_seqlens and cu_seqlens_k must describe the same number of sequences")
    return [(int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])) for s in range(cq.size - 1)]


def _unit_bias(attn_mask, lead, lq, lk):
    """Per-unit [Lq, Lk] additive masks for a dense batch with leading dims ``lead``."""
    if attn_mask is None:
        return None
    m = np.broadcast_to(_f64(attn_mask), tuple(lead) + (lq, lk))
    return m.reshape((-1, lq, lk))


def _unit_drops(dropout_p, seed, nunits, lq, lk):
    """Dropout factors Z per unit (None when p = 0)."""
    if not dropout_p:
        return None
    from .philox import dropout_keep, dropout_threshold
    t = dropout_threshold(dropout_p)
    kept = 256.0 / (256.0 - t)
    return [dropout_keep(seed, u, lq, lk, dropout_p) * kept for u in range(nunits)]


def attn_fwd_ref(q, k, v, scale: float, is_causal: bool = False, cu_seqlens=None, cu_seqlens_k=None,
                 block_mask=None, block_size: int = 128, attn_mask=None, dropout_p: float = 0.0, dropout_seed: int = 0):
    """Forward over a whole batch.

    Dense: ``q`` [..., Lq, d], ``k``/``v`` [..., Lk, d] -> ``O`` [..., Lq, d],
    ``LSE`` [..., Lq]. Packed (``cu_seqlens`` given): ``q``/``k``/``v``
    [total, H, d] -> ``O`` [total, H, d], ``LSE`` [H, total]; sequence s owns
    rows ``cu_seqlens[s] : cu_seqlens[s+1]`` of queries and keys (the
    tutorial's NestedTensor batches without padding). With ``cu_seqlens_k``
    the keys/values are [total_k, H, d] and sequence s owns key rows
    ``cu_seqlens_k[s] : cu_seqlens_k[s+1]``.
    Dense only: ``block_mask`` [..., ceil(Lq/block_size), ceil(Lk/block_size)]
    (broadcast over the leading dims) keeps or drops whole score tiles;
    ``attn_mask`` [..., Lq, Lk] (broadcast likewise) is added to the scores.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if cu_seqlens is None:
        lead = q.shape[:-2]
        qu, ku, vu = _units_dense(q), _units_dense(k), _units_dense(v)
        vis = _unit_masks(block_mask, lead, q.shape[-2], k.shape[-2], block_size)
        bias = _unit_bias(attn_mask, lead, q.shape[-2], k.shape[-2])
        drops = _unit_drops(dropout_p, dropout_seed, qu.shape[0], q.shape[-2], k.shape[-2])
        o = np.empty(qu.shape[:2] + (vu.shape[-1],))
        lse = np.empty(qu.shape[:2])
        for u in range(qu.shape[0]):
            o[u], lse[u] = attn_fwd_unit(qu[u], ku[u], vu[u], scale, is_causal, None if vis is None else vis[u],
                                         None if bias is None else bias[u], None if drops is None else drops[u])
        return o.reshape(lead + o.shape[1:]), lse.reshape(lead + lse.shape[1:])
    if block_mask is not None or attn_mask is not None or dropout_p:
        raise ValueError("block masks and additive masks apply to dense batches only")
    total, nh, _ = q.shape
    o = np.zeros((total, nh, v.shape[-1]))
    lse = np.zeros((nh, total))
    for a, b, c, e in _packed_spans(cu_seqlens, cu_seqlens_k, total, k.shape[0]):
        if b == a:
            continue
        for h in range(nh):
            o[a:b, h], lse[h, a:b] = attn_fwd_unit(q[a:b, h], k[c:e, h], v[c:e, h], scale, is_causal)
    return o, lse


def attn_bwd_ref(q, k, v, do, scale: float, is_causal: bool = False, cu_seqlens=None, cu_seqlens_k=None,
                 block_mask=None, block_size: int = 128, attn_mask=None, dropout_p: float = 0.0, dropout_seed: int = 0):
    """Backward over a whole batch; same layouts as :func:`attn_fwd_ref`.
    Returns ``(dQ, dK, dV)`` in float64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    if cu_seqlens is None:
        qu, ku, vu, du = (_units_dense(x) for x in (q, k, v, do))
        vis = _unit_masks(block_mask, q.shape[:-2], q.shape[-2], k.shape[-2], block_size)
        bias = _unit_bias(attn_mask, q.shape[:-2], q.shape[-2], k.shape[-2])
        drops = _unit_drops(dropout_p, dropout_seed, qu.shape[0], q.shape[-2], k.shape[-2])
        dq, dk, dv = np.empty_like(qu), np.empty_like(ku), np.empty_like(vu)
        for u in range(qu.shape[0]):
            dq[u], dk[u], dv[u] = attn_bwd_unit(qu[u], ku[u], vu[u], du[u], scale, is_causal,
                                                None if vis is None else vis[u], None if bias is None else bias[u],
                                                None if drops is None else drops[u])
        return dq.reshape(q.shape), dk.reshape(k.shape), dv.reshape(v.shape)
    if block_mask is not None or attn_mask is not None or dropout_p:
        raise ValueError("block masks and additive masks apply to dense batches only")
    total, nh, _ = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for a, b, c, e in _packed_spans(cu_seqlens, cu_seqlens_k, total, k.shape[0]):
        if b == a:
            continue
        for h in range(nh):
            dq[a:b, h], dk[c:e, h], dv[c:e, h] = attn_bwd_unit(
                q[a:b, h], k[c:e, h], v[c:e, h], do[a:b, h], scale, is_causal)
    return dq, dk, dv


def attn_fwd_rows(q_rows, k, v, row_index, scale: float, is_causal: bool = False):
    """Forward for selected query rows of one unit (for sampled checks at full size).

    ``q_rows`` [n, d] are the queries at absolute positions ``row_index`` [n]
    within a unit whose keys/values are ``k`` [Lk, d], ``v`` [Lk, dv]. Row i
    sees keys j <= row_index[i] when causal. Returns (O [n, dv], LSE [n]).
    """
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    rows = np.asarray(row_index, dtype=np.int64)
    s = float(scale) * (q_rows @ k.T)
    if is_causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > rows[:, None], -np.inf, s)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=1, keepdims=True)
    return (e / z) @ v, (m + np.log(z))[:, 0]
