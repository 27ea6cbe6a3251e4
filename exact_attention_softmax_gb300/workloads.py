"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and packs them; it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can take
their inputs from it.

Recipe (shapes from the SDPA tutorial page "(Beta) Implementing
High-Performance Transformers with SDPA"):

* Inputs are drawn with ``torch.Generator('cpu').manual_seed(seed)`` in the
  order q, k, v, dO, in float32, then cast to the workload dtype; the same
  cast values feed the GPU and (upcast exactly) the oracle.
* ``"uniform"`` draws U[0, 1) like the tutorial's ``torch.rand`` batch
  (section "Explicit Dispatcher Control"); ``"normal"`` draws N(0, 1) like its
  ``torch.randn`` inputs (sections "Overview" example and "NestedTensor and
  Dense tensor support").
* Packed variable-length batches follow the tutorial's ``generate_rand_batch``
  recipe: with ``random.Random(seed)``, each length is
  ``int(max_len * (1 - gauss(pad, 0.01)))`` (truncated toward zero), then one
  randomly chosen entry is set to ``max_len``; lengths are clamped to
  ``[1, max_len]``.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field

import torch

_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """One attention problem: dense ``[B, H, L, d]`` or packed ``[total, H, d]``."""

    name: str
    dtype: str
    H: int
    d: int
    dist: str
    causal: bool
    bwd: bool
    B: int = 0
    Lq: int = 0
    Lk: int = 0
    nseq: int = 0
    max_len: int = 0
    pad: float = 0.0
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def varlen(self) -> bool:
        return self.nseq > 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]


# The five workloads the measurements are quoted on.
WORKLOADS = {
    "tiny_f32": Workload(
        name="tiny_f32", dtype="f32", B=2, H=1, Lq=3, Lk=3, d=8, dist="normal",
        causal=False, bwd=True,
        note="the tutorial's [2,3,8] example shape, no head dim (B=2, H=1)"),
    "dense_f16_d32": Workload(
        name="dense_f16_d32", dtype="f16", B=32, H=32, Lq=1024, Lk=1024, d=32,
        dist="uniform", causal=False, bwd=False,
        note="tutorial dispatcher benchmark batch, torch.rand"),
    "causal_f16_d64": Workload(
        name="causal_f16_d64", dtype="f16", B=32, H=8, Lq=1024, Lk=1024, d=64,
        dist="normal", causal=True, bwd=True,
        note="CausalSelfAttention shape: embed 512, 8 heads"),
    "varlen_f16_d64": Workload(
        name="varlen_f16_d64", dtype="f16", H=8, d=64, dist="normal",
        causal=False, bwd=False, nseq=32, max_len=512, pad=0.5,
        note="NestedTensor batch, 32 sequences up to 512 tokens, packed"),
    "long_causal_bf16_d128": Workload(
        name="long_causal_bf16_d128", dtype="bf16", B=2, H=16, Lq=16384, Lk=16384,
        d=128, dist="normal", causal=True, bwd=True,
        note="long-context causal forward+backward"),
}


def _draw(gen: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32)
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def varlen_lengths(nseq: int, max_len: int, pad: float, seed: int = 0) -> list:
    """Sequence lengths by the tutorial's random-batch recipe (see module doc)."""
    rng = random.Random(seed)
    lens = [int(max_len * (1 - rng.gauss(pad, 0.01))) for _ in range(nseq)]
    lens[rng.randint(0, nseq - 1)] = max_len
    return [min(max(n, 1), max_len) for n in lens]


def cu_seqlens_from(lengths) -> torch.Tensor:
    """Offsets [nseq + 1] (int32) of each sequence in the packed token axis."""
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def dense_inputs(B, H, Lq, Lk, d, dtype="f16", dist="normal", seed=0, with_do=True):
    """q [B,H,Lq,d], k/v [B,H,Lk,d], dO [B,H,Lq,d] on the CPU in ``dtype``."""
    g = torch.Generator("cpu").manual_seed(seed)
    td = _DTYPES[dtype]
    out = {
        "q": _draw(g, (B, H, Lq, d), dist).to(td),
        "k": _draw(g, (B, H, Lk, d), dist).to(td),
        "v": _draw(g, (B, H, Lk, d), dist).to(td),
    }
    if with_do:
        out["do"] = _draw(g, (B, H, Lq, d), dist if dist == "normal" else "normal").to(td)
    return out


def varlen_inputs(lengths, H, d, dtype="f16", dist="normal", seed=0, with_do=True):
    """Packed q/k/v/dO [total, H, d] plus ``cu_seqlens`` (int32) and ``max_seqlen``."""
    g = torch.Generator("cpu").manual_seed(seed)
    td = _DTYPES[dtype]
    total = int(sum(lengths))
    out = {
        "q": _draw(g, (total, H, d), dist).to(td),
        "k": _draw(g, (total, H, d), dist).to(td),
        "v": _draw(g, (total, H, d), dist).to(td),
        "cu_seqlens": cu_seqlens_from(lengths),
        "max_seqlen": int(max(lengths)) if lengths else 0,
        "lengths": list(int(n) for n in lengths),
    }
    if with_do:
        out["do"] = _draw(g, (total, H, d), "normal").to(td)
    return out


def varlen_cross_inputs(lengths_q, lengths_k, H, d, dtype="f16", dist="normal", seed=0, with_do=True):
    """Packed cross-attention inputs: q/dO [total_q, H, d], k/v [total_k, H, d]
    with their own offsets ``cu_seqlens_q`` / ``cu_seqlens_k`` (int32) and
    length bounds ``max_seqlen_q`` / ``max_seqlen_k``."""
    if len(lengths_q) != len(lengths_k):
        raise ValueError("one key length per query length")
    g = torch.Generator("cpu").manual_seed(seed)
    td = _DTYPES[dtype]
    tq, tk = int(sum(lengths_q)), int(sum(lengths_k))
    out = {
        "q": _draw(g, (tq, H, d), dist).to(td),
        "k": _draw(g, (tk, H, d), dist).to(td),
        "v": _draw(g, (tk, H, d), dist).to(td),
        "cu_seqlens_q": cu_seqlens_from(lengths_q),
        "cu_seqlens_k": cu_seqlens_from(lengths_k),
        "max_seqlen_q": int(max(lengths_q)) if lengths_q else 0,
        "max_seqlen_k": int(max(lengths_k)) if lengths_k else 0,
    }
    if with_do:
        out["do"] = _draw(g, (tq, H, d), "normal").to(td)
    return out


def block_mask(shape, density: float = 0.5, seed: int = 0, empty_rows=()) -> torch.Tensor:
    """Seeded 0/1 block mask (uint8) of ``shape`` [..., nqb, nkb] for block-sparse
    attention: each tile kept with probability ``density``; the query blocks
    listed in ``empty_rows`` keep nothing."""
    g = torch.Generator("cpu").manual_seed(seed)
    m = (torch.rand(shape, generator=g) < density).to(torch.uint8)
    for r in empty_rows:
        m[..., r, :] = 0
    return m


def attn_mask(shape, dtype="f16", seed: int = 0, neg_inf: float = 0.1, empty_rows=(), pad_to: int = 8):
    """Seeded additive mask [..., Lq, Lk]: N(0,1) entries, a fraction
    ``neg_inf`` of them -inf, the rows in ``empty_rows`` entirely -inf. Returned
    with the key axis padded to a multiple of ``pad_to`` ([..., Lq, Lk_padded];
    take ``[..., :Lk]`` after moving it to the device, so the row stride stays
    a multiple of 8 entries, as the fp16/bf16 kernels' TMA reads of the mask
    need)."""
    g = torch.Generator("cpu").manual_seed(seed)
    *lead, lq, lk = shape
    lkp = (lk + pad_to - 1) // pad_to * pad_to
    full = torch.randn(tuple(lead) + (lq, lkp), generator=g)
    drop = torch.rand(tuple(lead) + (lq, lkp), generator=g) < neg_inf
    full[drop] = float("-inf")
    for r in empty_rows:
        full[..., r, :] = float("-inf")
    return full.to(_DTYPES[dtype])


def workload_inputs(w: Workload, seed: int = 0, with_do=None):
    """Inputs of a named workload (dO drawn when the workload has a backward)."""
    if with_do is None:
        with_do = w.bwd
    if w.varlen:
        lens = varlen_lengths(w.nseq, w.max_len, w.pad, seed)
        return varlen_inputs(lens, w.H, w.d, w.dtype, w.dist, seed, with_do)
    return dense_inputs(w.B, w.H, w.Lq, w.Lk, w.d, w.dtype, w.dist, seed, with_do)


def fwd_flops(w: Workload, lengths=None) -> float:
    """Algorithmic forward FLOPs: 4*B*H*Lq*Lk*d, halved under causal masking;
    packed batches count 4*H*d*sum(l_i^2)."""
    if w.varlen:
        tot = sum(int(n) ** 2 for n in lengths)
        f = 4.0 * w.H * w.d * tot
    else:
        f = 4.0 * w.B * w.H * w.Lq * w.Lk * w.d
    return f / 2 if w.causal else f


def bwd_flops(w: Workload, lengths=None) -> float:
    """Algorithmic backward FLOPs: 2.5x the forward count."""
    return 2.5 * fwd_flops(w, lengths)
