"""Exact scaled dot-product attention for GB300 (sm_103a): a thin PyTorch
binding over the C ABI of ``libsdpa_gb300.so`` (``include/sdpa.h``).

The functions here only marshal arguments: they check shapes, allocate
outputs with PyTorch when the caller passes none, and hand raw device
pointers plus the current CUDA stream to the library, whose kernels do all of
the work. Nothing falls back to PyTorch or the CPU; a missing library raises.

Definition (SDPA tutorial page, section "Overview"):
``O = softmax(scale * Q K^T [+ causal mask]) V`` with the natural-log row
log-sum-exp ``LSE`` saved for the backward (FlashAttention news article,
section "FlashAttention": tiled, exact, recomputed in the backward).
"""
from __future__ import annotations

import ctypes
import math

from . import _abi
from ._abi import SdpaError  # noqa: F401

__all__ = ["sdpa_fwd", "sdpa_bwd", "sdpa_fwd_varlen", "sdpa_bwd_varlen", "sdpa_fwd_blocksparse",
           "sdpa_bwd_blocksparse", "sdpa_fwd_masked", "sdpa_bwd_masked", "sdpa_fwd_dropout",
           "sdpa_bwd_dropout", "sdpa_bwd_workspace_size",
           "sdpa_device_status", "sdpa_trace_events",
           "sdpa_debug_set", "sdpa_debug_build", "sdpa_last_error", "sdpa_version", "SdpaError"]


def _dtype_code(t):
    import torch
    codes = {torch.float32: _abi.SDPA_F32, torch.float16: _abi.SDPA_F16, torch.bfloat16: _abi.SDPA_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _vp(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _stream(dev, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    return ctypes.c_void_p(stream.cuda_stream)


def _geometry(q, k, cu_seqlens, max_seqlen):
    """(B, H, Lq, Lk, d, packed) in the C ABI's convention."""
    if cu_seqlens is not None:
        if q.dim() != 3:
            raise ValueError("packed q must be [total, H, d]")
        total, H, d = q.shape
        if max_seqlen is None:
            raise ValueError("packed batches need max_seqlen (an upper bound on every length)")
        return cu_seqlens.numel() - 1, H, total, int(max_seqlen), d, True
    if q.dim() == 3:  # [B, L, d]: one head
        return q.shape[0], 1, q.shape[1], k.shape[1], q.shape[2], False
    if q.dim() != 4:
        raise ValueError("dense q must be [B, H, L, d] (or [B, L, d])")
    B, H, Lq, d = q.shape
    return B, H, Lq, k.shape[2], d, False


def _check_tensors(ts, dev, dt, strided_ok=False):
    """Device, dtype and layout checks. With ``strided_ok`` (dense calls) a
    tensor may have any strides whose innermost one is 1; otherwise it must
    be contiguous."""
    if dev.type != "cuda":
        raise ValueError(f"q is on {dev}: the attention ops take CUDA tensors only (there is no CPU implementation)")
    for name, t in ts.items():
        if t is None:
            continue
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, expected {dev}")
        if t.dtype != dt:
            raise TypeError(f"{name} has dtype {t.dtype}, expected {dt}")
        if strided_ok and t.dim() >= 3 and t.stride(-1) == 1:
            continue
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous" + (" or have a unit innermost stride" if strided_ok else ""))


def _strides(ts):
    """ctypes array of the (batch, head, row) element strides of dense
    [B, H, L, d] (or one-head [B, L, d]) tensors, in the C ABI's order."""
    vals = []
    for t in ts:
        st = t.stride()
        vals += list(st[:3]) if t.dim() == 4 else [st[0], st[0], st[1]]
    return (ctypes.c_longlong * len(vals))(*vals)


def _is_strided(ts):
    return any(t is not None and not t.is_contiguous() for t in ts)


def sdpa_fwd(q, k, v, o=None, lse=None, *, scale=None, is_causal=False, cu_seqlens=None,
             max_seqlen=None, stream=None):
    """Forward pass. Returns ``(O, LSE)``.

    Dense: q [B,H,Lq,d] (or [B,Lq,d]), k/v [B,H,Lk,d]; LSE [B,H,Lq] fp32.
    Packed: q/k/v [total,H,d], ``cu_seqlens`` int32 [nseq+1] on the device,
    ``max_seqlen`` >= every length; LSE [H,total] fp32.
    ``scale`` defaults to 1/sqrt(d).
    """
    import torch
    lib = _abi.load()
    B, H, Lq, Lk, d, packed = _geometry(q, k, cu_seqlens, max_seqlen)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        shape = (H, Lq) if packed else tuple(q.shape[:-1])
        lse = torch.empty(shape, dtype=torch.float32, device=q.device)
    _check_tensors({"q": q, "k": k, "v": v, "o": o}, q.device, q.dtype, strided_ok=not packed)
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise TypeError("lse must be contiguous float32")
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or cu_seqlens.device != q.device):
        raise TypeError("cu_seqlens must be int32 on the device of q")
    if not packed and _is_strided((q, k, v, o)):
        # dense tensors at any strides (e.g. the [B, L, H, d] projections
        # viewed as [B, H, L, d]): no copy
        _abi.check(lib.sdpa_fwd_strided(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), B, H, Lq, Lk, d, float(scale),
                                        int(bool(is_causal)), _strides((q, k, v, o)), _dtype_code(q),
                                        _stream(q.device, stream)))
        return o, lse
    _abi.check(lib.sdpa_fwd(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), B, H, Lq, Lk, d, float(scale),
                            int(bool(is_causal)), _vp(cu_seqlens), _dtype_code(q), _stream(q.device, stream)))
    return o, lse


def sdpa_bwd_workspace_size(B, H, Lq, d, dtype_code):
    """Bytes of device scratch :func:`sdpa_bwd` needs (packed: B=1, Lq=total)."""
    return int(_abi.load().sdpa_bwd_workspace_size(B, H, Lq, d, dtype_code))


def sdpa_bwd(q, k, v, o, lse, dO, dq=None, dk=None, dv=None, *, scale=None, is_causal=False,
             cu_seqlens=None, max_seqlen=None, workspace=None, stream=None):
    """Backward pass. Returns ``(dQ, dK, dV)``; layouts as :func:`sdpa_fwd`.
    ``workspace`` (a uint8 CUDA tensor) is allocated here when not given."""
    import torch
    lib = _abi.load()
    B, H, Lq, Lk, d, packed = _geometry(q, k, cu_seqlens, max_seqlen)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors({"q": q, "k": k, "v": v, "o": o, "dO": dO, "dq": dq, "dk": dk, "dv": dv}, q.device, q.dtype,
                   strided_ok=not packed)
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise TypeError("lse must be contiguous float32")
    code = _dtype_code(q)
    need = lib.sdpa_bwd_workspace_size(1 if packed else B, H, Lq, d, code)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if not packed and _is_strided((q, k, v, o, dO, dq, dk, dv)):
        _abi.check(lib.sdpa_bwd_strided(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), _vp(dO), _vp(dq), _vp(dk),
                                        _vp(dv), B, H, Lq, Lk, d, float(scale), int(bool(is_causal)),
                                        _strides((q, k, v, o, dO, dq, dk, dv)), code, _vp(workspace),
                                        workspace.numel(), _stream(q.device, stream)))
        return dq, dk, dv
    _abi.check(lib.sdpa_bwd(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), _vp(dO), _vp(dq), _vp(dk), _vp(dv),
                            B, H, Lq, Lk, d, float(scale), int(bool(is_causal)), _vp(cu_seqlens), code,
                            _vp(workspace), workspace.numel(), _stream(q.device, stream)))
    return dq, dk, dv


def _varlen_geometry(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k):
    """(nseq, H, total_q, total_k, max_q, max_k, d) for the cross-attention calls."""
    import torch
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("varlen q and k must be [total, H, d]")
    if k.shape[1:] != q.shape[1:]:
        raise ValueError("q and k must agree in H and d")
    for name, cu in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if cu.dtype != torch.int32 or cu.device != q.device or cu.dim() != 1 or not cu.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int32 vector on the device of q")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold nseq + 1 offsets")
    total_q, H, d = q.shape
    return cu_seqlens_q.numel() - 1, H, total_q, k.shape[0], int(max_seqlen_q), int(max_seqlen_k), d


def sdpa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, o=None, lse=None, *,
                    scale=None, is_causal=False, stream=None):
    """Forward over packed sequences with separate query and key offsets.

    q/o [total_q,H,d], k/v [total_k,H,d]; sequence s owns query rows
    ``cu_seqlens_q[s]:cu_seqlens_q[s+1]`` and key rows
    ``cu_seqlens_k[s]:cu_seqlens_k[s+1]``; the max_seqlen bounds cover every
    length. Returns ``(O, LSE)`` with LSE [H,total_q] fp32. A [B,L,H,d] batch
    is the case of uniform offsets ``s*L``.
    """
    import torch
    lib = _abi.load()
    nseq, H, tq, tk, mq, mk, d = _varlen_geometry(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((H, tq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensors({"k": k, "v": v, "o": o}, q.device, q.dtype)
    if v.shape != k.shape or o.shape != q.shape:
        raise ValueError("v must match k and o must match q")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (H, tq):
        raise TypeError("lse must be contiguous float32 [H, total_q]")
    _abi.check(lib.sdpa_fwd_varlen(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), nseq, H, tq, tk, mq, mk, d,
                                   float(scale), int(bool(is_causal)), _vp(cu_seqlens_q), _vp(cu_seqlens_k),
                                   _dtype_code(q), _stream(q.device, stream)))
    return o, lse


def sdpa_bwd_varlen(q, k, v, o, lse, dO, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    dq=None, dk=None, dv=None, *, scale=None, is_causal=False, workspace=None, stream=None):
    """Backward of :func:`sdpa_fwd_varlen`. Returns ``(dQ, dK, dV)``."""
    import torch
    lib = _abi.load()
    nseq, H, tq, tk, mq, mk, d = _varlen_geometry(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors({"k": k, "v": v, "o": o, "dO": dO, "dq": dq, "dk": dk, "dv": dv}, q.device, q.dtype)
    if v.shape != k.shape or o.shape != q.shape or dO.shape != q.shape or dq.shape != q.shape \
            or dk.shape != k.shape or dv.shape != k.shape:
        raise ValueError("gradient and output shapes must match their inputs")
    code = _dtype_code(q)
    need = lib.sdpa_bwd_workspace_size(1, H, tq, d, code)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _abi.check(lib.sdpa_bwd_varlen(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), _vp(dO), _vp(dq), _vp(dk), _vp(dv),
                                   nseq, H, tq, tk, mq, mk, d, float(scale), int(bool(is_causal)),
                                   _vp(cu_seqlens_q), _vp(cu_seqlens_k), code, _vp(workspace), workspace.numel(),
                                   _stream(q.device, stream)))
    return dq, dk, dv


MASK_BLOCK = 128   # rows and keys per tile of a block-sparse mask


def _mask_args(block_mask, B, H, Lq, Lk, dev):
    """(pointer, stride_b, stride_h, stride_row) of a uint8 block mask of shape
    [nqb, nkb], [H, nqb, nkb] or [B, H, nqb, nkb] (size-1 or expanded dims broadcast)."""
    import torch
    nq, nk = -(-Lq // MASK_BLOCK), -(-Lk // MASK_BLOCK)
    if block_mask.dtype not in (torch.uint8, torch.bool) or block_mask.device != dev:
        raise TypeError("block_mask must be uint8 or bool on the device of q")
    m = block_mask
    while m.dim() < 4:
        m = m.unsqueeze(0)
    if m.dim() != 4 or tuple(m.shape[-2:]) != (nq, nk):
        raise ValueError(f"block_mask must end in ({nq}, {nk}) for Lq={Lq}, Lk={Lk}")
    if m.stride(-1) != 1:
        raise ValueError("block_mask rows must be contiguous")
    sb = 0 if m.shape[0] == 1 else m.stride(0)
    sh = 0 if m.shape[1] == 1 else m.stride(1)
    if m.shape[0] not in (1, B) or m.shape[1] not in (1, H):
        raise ValueError("block_mask batch / head dims must be 1 or match q")
    return ctypes.c_void_p(m.data_ptr()), sb, sh, m.stride(2)


def sdpa_fwd_blocksparse(q, k, v, block_mask, o=None, lse=None, *, scale=None, is_causal=False, stream=None):
    """Block-sparse forward: exact attention over the 128x128 score tiles
    ``block_mask`` keeps (uint8/bool, [..., ceil(Lq/128), ceil(Lk/128)]).
    Dense [B,H,L,d] layout. Rows with no visible key get O = 0, LSE = -inf."""
    import torch
    lib = _abi.load()
    if q.dim() != 4:
        raise ValueError("block-sparse q must be [B, H, L, d]")
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensors({"k": k, "v": v, "o": o}, q.device, q.dtype)
    mp, sb, sh, sq = _mask_args(block_mask, B, H, Lq, Lk, q.device)
    _abi.check(lib.sdpa_fwd_blocksparse(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), B, H, Lq, Lk, d, float(scale),
                                        int(bool(is_causal)), mp, sb, sh, sq, _dtype_code(q),
                                        _stream(q.device, stream)))
    return o, lse


def sdpa_bwd_blocksparse(q, k, v, o, lse, dO, block_mask, dq=None, dk=None, dv=None, *, scale=None,
                         is_causal=False, workspace=None, stream=None):
    """Backward of :func:`sdpa_fwd_blocksparse`. Returns ``(dQ, dK, dV)``."""
    import torch
    lib = _abi.load()
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors({"k": k, "v": v, "o": o, "dO": dO, "dq": dq, "dk": dk, "dv": dv}, q.device, q.dtype)
    code = _dtype_code(q)
    need = lib.sdpa_bwd_workspace_size(B, H, Lq, d, code)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    mp, sb, sh, sq = _mask_args(block_mask, B, H, Lq, Lk, q.device)
    _abi.check(lib.sdpa_bwd_blocksparse(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), _vp(dO), _vp(dq), _vp(dk), _vp(dv),
                                        B, H, Lq, Lk, d, float(scale), int(bool(is_causal)), mp, sb, sh, sq, code,
                                        _vp(workspace), workspace.numel(), _stream(q.device, stream)))
    return dq, dk, dv


def _attn_mask_args(attn_mask, q, Lq, Lk):
    """(pointer, stride_b, stride_h, stride_row) of an additive mask [..., Lq, Lk]
    in q's dtype, keys contiguous; size-1 or expanded leading dims broadcast."""
    m = attn_mask
    if m.dtype != q.dtype or m.device != q.device:
        raise TypeError("attn_mask must have the dtype and device of q")
    while m.dim() < 4:
        m = m.unsqueeze(0)
    if m.dim() != 4 or tuple(m.shape[-2:]) != (Lq, Lk) or m.stride(-1) != 1:
        raise ValueError(f"attn_mask must be [..., {Lq}, {Lk}] with contiguous keys")
    B, H = q.shape[0], q.shape[1]
    if m.shape[0] not in (1, B) or m.shape[1] not in (1, H):
        raise ValueError("attn_mask batch / head dims must be 1 or match q")
    sb = 0 if m.shape[0] == 1 else m.stride(0)
    sh = 0 if m.shape[1] == 1 else m.stride(1)
    return ctypes.c_void_p(m.data_ptr()), sb, sh, m.stride(2)


def sdpa_fwd_masked(q, k, v, attn_mask, o=None, lse=None, *, scale=None, is_causal=False, stream=None):
    """Forward with an additive mask: ``softmax(scale * Q K^T + attn_mask) V``
    (dense [B,H,L,d]; -inf entries exclude a score). For fp16/bf16 the mask's
    base must be 16-byte aligned and its strides multiples of 8 elements
    (pad the key axis to a multiple of 8; the padding is never read). Rows
    with no visible key get O = 0, LSE = -inf."""
    import torch
    lib = _abi.load()
    if q.dim() != 4:
        raise ValueError("masked q must be [B, H, L, d]")
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensors({"k": k, "v": v, "o": o}, q.device, q.dtype)
    mp, sb, sh, sq = _attn_mask_args(attn_mask, q, Lq, Lk)
    _abi.check(lib.sdpa_fwd_masked(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), B, H, Lq, Lk, d, float(scale),
                                   int(bool(is_causal)), mp, sb, sh, sq, _dtype_code(q), _stream(q.device, stream)))
    return o, lse


def sdpa_bwd_masked(q, k, v, o, lse, dO, attn_mask, dq=None, dk=None, dv=None, *, scale=None, is_causal=False,
                    workspace=None, stream=None):
    """Backward of :func:`sdpa_fwd_masked` (gradients for q, k, v)."""
    import torch
    lib = _abi.load()
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors({"k": k, "v": v, "o": o, "dO": dO, "dq": dq, "dk": dk, "dv": dv}, q.device, q.dtype)
    code = _dtype_code(q)
    need = lib.sdpa_bwd_workspace_size(B, H, Lq, d, code)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    mp, sb, sh, sq = _attn_mask_args(attn_mask, q, Lq, Lk)
    _abi.check(lib.sdpa_bwd_masked(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), _vp(dO), _vp(dq), _vp(dk), _vp(dv),
                                   B, H, Lq, Lk, d, float(scale), int(bool(is_causal)), mp, sb, sh, sq, code,
                                   _vp(workspace), workspace.numel(), _stream(q.device, stream)))
    return dq, dk, dv


def sdpa_fwd_dropout(q, k, v, dropout_p, seed, o=None, lse=None, *, scale=None, is_causal=False, stream=None):
    """Forward with dropout on the probabilities (dense [B,H,L,d]); the keep
    pattern is a pure function of ``seed`` (Philox4x32-10, see the C header).
    LSE is that of the full softmax."""
    import torch
    lib = _abi.load()
    if q.dim() != 4:
        raise ValueError("dropout q must be [B, H, L, d]")
    B, H, Lq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensors({"k": k, "v": v, "o": o}, q.device, q.dtype)
    _abi.check(lib.sdpa_fwd_dropout(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), B, H, Lq, k.shape[2], d, float(scale),
                                    int(bool(is_causal)), float(dropout_p), int(seed) & ((1 << 64) - 1),
                                    _dtype_code(q), _stream(q.device, stream)))
    return o, lse


def sdpa_bwd_dropout(q, k, v, o, lse, dO, dropout_p, seed, dq=None, dk=None, dv=None, *, scale=None,
                     is_causal=False, workspace=None, stream=None):
    """Backward of :func:`sdpa_fwd_dropout` (same ``dropout_p`` and ``seed``)."""
    import torch
    lib = _abi.load()
    B, H, Lq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors({"k": k, "v": v, "o": o, "dO": dO, "dq": dq, "dk": dk, "dv": dv}, q.device, q.dtype)
    code = _dtype_code(q)
    need = lib.sdpa_bwd_workspace_size(B, H, Lq, d, code)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _abi.check(lib.sdpa_bwd_dropout(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), _vp(dO), _vp(dq), _vp(dk), _vp(dv),
                                    B, H, Lq, k.shape[2], d, float(scale), int(bool(is_causal)), float(dropout_p),
                                    int(seed) & ((1 << 64) - 1), code, _vp(workspace), workspace.numel(),
                                    _stream(q.device, stream)))
    return dq, dk, dv


def sdpa_device_status(stream=None):
    """Synchronise and read/clear the device status word. Returns the raw bits;
    raises :class:`SdpaError` when a kernel reported a problem."""
    import torch
    lib = _abi.load()
    bits = ctypes.c_uint(0)
    s = ctypes.c_void_p(stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    _abi.check(lib.sdpa_device_status(s, ctypes.byref(bits)))
    return bits.value


def sdpa_trace_events(which, begin=None, end=None):
    """Kernel timing aid: later calls record ``begin`` and ``end``
    (``torch.cuda.Event(enable_timing=True)``) on their stream around their
    main attention kernel -- the forward's for ``which`` = 0 (or "fwd"), the
    backward's for 1 (or "bwd"); ``None`` for both removes them. Read the time
    with ``begin.elapsed_time(end)`` after synchronising."""
    import torch
    w = {"fwd": 0, "bwd": 1}.get(which, which)

    def handle(ev):
        if ev is None:
            return ctypes.c_void_p(0)
        if ev.cuda_event == 0:      # PyTorch creates the CUDA event on its first record
            ev.record(torch.cuda.current_stream())
        return ctypes.c_void_p(ev.cuda_event)
    _abi.check(_abi.load().sdpa_trace_events(int(w), handle(begin), handle(end)))


def sdpa_debug_set(flags: int) -> int:
    return int(_abi.load().sdpa_debug_set(int(flags)))


def sdpa_last_error() -> str:
    return _abi.load().sdpa_last_error().decode()


def sdpa_version() -> int:
    return int(_abi.load().sdpa_version())


def sdpa_debug_build() -> int:
    """1 if the loaded library is the debug build (device-side bounds checks)."""
    return int(_abi.load().sdpa_debug_build())
