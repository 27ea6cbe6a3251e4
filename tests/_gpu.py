"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
(via the ctypes binding) on seeded inputs and compare with the fp64 oracle."""
import numpy as np
import torch

import exact_attention_softmax_gb300 as ops
from oracle import attn_bwd_ref, attn_fwd_ref

# Tolerances against the fp64 oracle (forward max-abs per dtype; gradients by
# relative Frobenius error per tensor).
FWD_ATOL = {"f32": 1e-5, "f16": 4e-3, "bf16": 2e-2}
LSE_ATOL = {"f32": 1e-5, "f16": 1e-3, "bf16": 1e-3}
GRAD_RTOL = {"f32": 1e-5, "f16": 1e-2, "bf16": 1e-2}
SENTINEL = -12345.0
PAD = 256  # elements of canary on each side of every output


def cuda():
    return torch.device("cuda", 0)


def guarded_empty(shape, dtype, device):
    """An output tensor with canary padding before and after it."""
    n = int(np.prod(shape)) if len(shape) else 1
    buf = torch.full((n + 2 * PAD,), SENTINEL, dtype=dtype, device=device)
    return buf, buf[PAD:PAD + n].view(shape)


def check_guard(buf):
    head = buf[:PAD].float().cpu()
    tail = buf[-PAD:].float().cpu()
    s = torch.tensor(SENTINEL, dtype=buf.dtype).float()
    assert torch.all(head == s) and torch.all(tail == s), "store outside the output tensor"


def f64(t):
    return t.detach().double().cpu().numpy()


def rel_fro(a, b):
    """Relative Frobenius error. The denominator is floored at 1e-4 * sqrt(n): with
    a single visible key the softmax Jacobian vanishes and the exact dQ, dK are
    identically zero, so there the error is judged in absolute terms."""
    floor = 1e-4 * np.sqrt(max(b.size, 1))
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), floor))


def run_fwd(x, causal, scale, packed=False):
    """x: dict of CPU tensors from the workload generator. Returns (O, LSE) on CPU
    as float64 numpy, after checking canaries and the device status word."""
    dev = cuda()
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    ob, o = guarded_empty(tuple(q.shape), q.dtype, dev)
    lshape = (q.shape[1], q.shape[0]) if packed else tuple(q.shape[:-1])
    lb, lse = guarded_empty(lshape, torch.float32, dev)
    kw = {}
    if packed:
        kw = dict(cu_seqlens=x["cu_seqlens"].to(dev), max_seqlen=max(x["max_seqlen"], 1))
    ops.sdpa_fwd(q, k, v, o, lse, scale=scale, is_causal=causal, **kw)
    assert ops.sdpa_device_status() == 0
    check_guard(ob)
    check_guard(lb)
    return f64(o), f64(lse)


def run_fwd_bwd(x, causal, scale):
    dev = cuda()
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = ops.sdpa_fwd(q, k, v, scale=scale, is_causal=causal)
    gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
    dq, dk, dv = ops.sdpa_bwd(q, k, v, o, lse, do, gb[0][1], gb[1][1], gb[2][1], scale=scale, is_causal=causal)
    assert ops.sdpa_device_status() == 0
    for b, _ in gb:
        check_guard(b)
    return f64(o), f64(lse), f64(dq), f64(dk), f64(dv)


def run_fwd_bwd_packed(x, causal, scale):
    """Packed fwd + bwd through the C ABI; returns (O, LSE, dQ, dK, dV) as float64."""
    dev = cuda()
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = dict(cu_seqlens=x["cu_seqlens"].to(dev), max_seqlen=max(x["max_seqlen"], 1))
    o, lse = ops.sdpa_fwd(q, k, v, scale=scale, is_causal=causal, **kw)
    gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
    dq, dk, dv = ops.sdpa_bwd(q, k, v, o, lse, do, gb[0][1], gb[1][1], gb[2][1], scale=scale, is_causal=causal, **kw)
    assert ops.sdpa_device_status() == 0
    for b, _ in gb:
        check_guard(b)
    return f64(o), f64(lse), f64(dq), f64(dk), f64(dv)


def run_varlen_cross(x, causal, scale, bwd=True):
    """Cross-attention packed fwd (+ bwd) through sdpa_fwd_varlen / sdpa_bwd_varlen;
    returns (O, LSE[, dQ, dK, dV]) as float64 after the canary and status checks."""
    dev = cuda()
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    cq, ck = x["cu_seqlens_q"].to(dev), x["cu_seqlens_k"].to(dev)
    mq, mk = max(x["max_seqlen_q"], 1), max(x["max_seqlen_k"], 1)
    ob, o = guarded_empty(tuple(q.shape), q.dtype, dev)
    lb, lse = guarded_empty((q.shape[1], q.shape[0]), torch.float32, dev)
    ops.sdpa_fwd_varlen(q, k, v, cq, ck, mq, mk, o, lse, scale=scale, is_causal=causal)
    out = [o, lse]
    bufs = [ob, lb]
    if bwd:
        do = x["do"].to(dev)
        gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
        ops.sdpa_bwd_varlen(q, k, v, o, lse, do, cq, ck, mq, mk, gb[0][1], gb[1][1], gb[2][1],
                            scale=scale, is_causal=causal)
        out += [g for _, g in gb]
        bufs += [b for b, _ in gb]
    assert ops.sdpa_device_status() == 0
    for b in bufs:
        check_guard(b)
    return tuple(f64(t) for t in out)


def oracle_varlen_cross(x, causal, scale, bwd=True):
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    cq, ck = x["cu_seqlens_q"].numpy(), x["cu_seqlens_k"].numpy()
    out = attn_fwd_ref(q, k, v, scale, causal, cq, ck)
    if bwd:
        out = out + attn_bwd_ref(q, k, v, f64(x["do"]), scale, causal, cq, ck)
    return out


def oracle_bwd_packed(x, causal, scale):
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "do"))
    return attn_bwd_ref(q, k, v, do, scale, causal, x["cu_seqlens"].numpy())


def oracle_fwd(x, causal, scale, packed=False):
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    return attn_fwd_ref(q, k, v, scale, causal, x["cu_seqlens"].numpy() if packed else None)


def oracle_bwd(x, causal, scale):
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "do"))
    return attn_bwd_ref(q, k, v, do, scale, causal)


def assert_fwd_close(got, ref, dtype):
    o, lse = got
    ro, rlse = ref
    err_o = float(np.max(np.abs(o - ro))) if o.size else 0.0
    err_l = float(np.max(np.abs(lse - rlse))) if lse.size else 0.0
    assert err_o <= FWD_ATOL[dtype], f"O max-abs error {err_o:.3e} > {FWD_ATOL[dtype]}"
    assert err_l <= LSE_ATOL[dtype], f"LSE max-abs error {err_l:.3e} > {LSE_ATOL[dtype]}"
    return err_o, err_l


def assert_grads_close(got, ref, dtype):
    errs = []
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        e = rel_fro(g, r)
        errs.append(e)
        assert e <= GRAD_RTOL[dtype], f"{name} relative Frobenius error {e:.3e} > {GRAD_RTOL[dtype]}"
    return errs
