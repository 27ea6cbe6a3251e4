"""Parity of block-sparse attention (sdpa_fwd_blocksparse / sdpa_bwd_blocksparse)
with the fp64 oracle through the C ABI. The FlashAttention news article
(QbitAI repost, section "FlashAttention") names block-sparse FlashAttention;
the masks here are seeded random 0/1 tile masks, with whole query blocks left
empty and ragged last tiles, over both dtypes and head dims, causal or not."""
import numpy as np
import pytest
import torch

import exact_attention_softmax_gb300 as ops
from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _nb(n):
    return -(-n // ops.MASK_BLOCK)


def _run(x, mask, causal, scale, bwd=True):
    from _gpu import check_guard, cuda, f64, guarded_empty
    dev = cuda()
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    m = mask.to(dev)
    ob, o = guarded_empty(tuple(q.shape), q.dtype, dev)
    lb, lse = guarded_empty(tuple(q.shape[:-1]), torch.float32, dev)
    ops.sdpa_fwd_blocksparse(q, k, v, m, o, lse, scale=scale, is_causal=causal)
    out, bufs = [o, lse], [ob, lb]
    if bwd:
        do = x["do"].to(dev)
        gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
        ops.sdpa_bwd_blocksparse(q, k, v, o, lse, do, m, gb[0][1], gb[1][1], gb[2][1], scale=scale, is_causal=causal)
        out += [g for _, g in gb]
        bufs += [b for b, _ in gb]
    assert ops.sdpa_device_status() == 0
    for b in bufs:
        check_guard(b)
    return tuple(f64(t) for t in out)


def _oracle(x, mask, causal, scale, bwd=True):
    from _gpu import f64
    from oracle import attn_bwd_ref, attn_fwd_ref
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    m = mask.numpy()
    out = attn_fwd_ref(q, k, v, scale, causal, block_mask=m)
    if bwd:
        out = out + attn_bwd_ref(q, k, v, f64(x["do"]), scale, causal, block_mask=m)
    return out


def _check_fwd(got, ref, dtype):
    from _gpu import assert_fwd_close
    o, lse = got
    ro, rlse = ref
    # rows without a visible key: exactly O = 0 and LSE = -inf on both sides
    empty = np.isneginf(rlse)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(o[empty] == 0)
    lse_f = np.where(empty, 0.0, lse)
    rlse_f = np.where(empty, 0.0, rlse)
    assert_fwd_close((o, lse_f), (ro, rlse_f), dtype)


SHAPES = [(1, 2, 300, 333), (2, 1, 256, 512), (1, 1, 640, 200)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_blocksparse_fwd_bwd(dtype, d, causal, shape):
    from _gpu import assert_grads_close
    B, H, Lq, Lk = shape
    x = wl.dense_inputs(B, H, Lq, Lk, d, dtype, "normal", seed=41)
    mask = wl.block_mask((B, H, _nb(Lq), _nb(Lk)), 0.5, seed=42, empty_rows=(1,))
    scale = d ** -0.5
    got = _run(x, mask, causal, scale)
    ref = _oracle(x, mask, causal, scale)
    _check_fwd(got[:2], ref[:2], dtype)
    assert_grads_close(got[2:], ref[2:], dtype)


@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_broadcast_mask_and_d32_forward(causal):
    B, H, Lq, Lk, d = 2, 3, 520, 300, 32
    x = wl.dense_inputs(B, H, Lq, Lk, d, "f16", "normal", seed=43, with_do=False)
    mask = wl.block_mask((_nb(Lq), _nb(Lk)), 0.6, seed=44, empty_rows=(2,))   # shared by every (b, h)
    got = _run(x, mask, causal, 0.2, bwd=False)
    _check_fwd(got, _oracle(x, mask, causal, 0.2, bwd=False), "f16")


@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_f32(causal):
    from _gpu import assert_grads_close
    B, H, Lq, Lk, d = 1, 2, 270, 140, 24
    x = wl.dense_inputs(B, H, Lq, Lk, d, "f32", "normal", seed=45)
    mask = wl.block_mask((H, _nb(Lq), _nb(Lk)), 0.5, seed=46, empty_rows=(0,))
    got = _run(x, mask, causal, 0.3)
    ref = _oracle(x, mask, causal, 0.3)
    _check_fwd(got[:2], ref[:2], "f32")
    assert_grads_close(got[2:], ref[2:], "f32")


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_many_items_per_cta(d, causal):
    """More work items than SMs, so each persistent CTA runs several items in
    a row while its tiles drop some of their pair's loaded blocks: the path
    that carries barrier phases and the deferred epilogue from one item into
    the next. Sampled (batch, head) units against the oracle."""
    B, H, L = 8, 24, 1024          # 192 units x 4 items of 256 rows: 768 items on at most 152 CTAs
    scale = d ** -0.5
    x = wl.dense_inputs(B, H, L, L, d, "f16", "normal", seed=48, with_do=False)
    mask = wl.block_mask((B, H, _nb(L), _nb(L)), 0.5, seed=49)
    got = _run(x, mask, causal, scale, bwd=False)
    for b, h in [(0, 0), (3, 7), (7, 23)]:
        sub = {n: x[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
        ref = _oracle(sub, mask[b:b + 1, h:h + 1], causal, scale, bwd=False)
        _check_fwd((got[0][b:b + 1, h:h + 1], got[1][b:b + 1, h:h + 1]), ref, "f16")


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_uneven_tiles(d, causal):
    """The two 128-row query tiles of each 256-row item keep very different
    numbers of key blocks: one keeps every block, the other one or two, and
    the roles swap from head to head. One tile then runs through many more
    K/V fills than a ring holds before the other finishes, and on into its
    next item, on many items per CTA. Sampled units against the oracle."""
    B, H, L = 1, 40, 4096
    nb = _nb(L)
    m = np.zeros((H, nb, nb), dtype=np.uint8)
    for h in range(H):
        for r in range(nb):
            if (r + h) % 2 == 0:
                m[h, r, :] = 1               # every key block
            else:
                m[h, r, 0] = 1               # the first block, and under causal masking
                m[h, r, r] = 1               # the diagonal one
    mask = torch.from_numpy(m)
    scale = d ** -0.5
    x = wl.dense_inputs(B, H, L, L, d, "bf16", "normal", seed=50, with_do=False)
    got = _run(x, mask, causal, scale, bwd=False)
    for h in (0, 1, 38, 39):
        sub = {n: x[n][:, h:h + 1] for n in ("q", "k", "v")}
        ref = _oracle(sub, mask[h:h + 1], causal, scale, bwd=False)
        _check_fwd((got[0][:, h:h + 1], got[1][:, h:h + 1]), ref, "bf16")


def test_all_ones_mask_matches_dense_call():
    """With every tile kept the block-sparse forward gives the dense call's
    results bit for bit (same blocks, same order)."""
    from _gpu import cuda
    dev = cuda()
    x = wl.dense_inputs(2, 2, 384, 384, 64, "f16", "normal", seed=47)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    ones = torch.ones((3, 3), dtype=torch.uint8, device=dev)
    for causal in (False, True):
        a = ops.sdpa_fwd(q, k, v, is_causal=causal)
        b = ops.sdpa_fwd_blocksparse(q, k, v, ones, is_causal=causal)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        ga = ops.sdpa_bwd(q, k, v, a[0], a[1], do, is_causal=causal)
        gb = ops.sdpa_bwd_blocksparse(q, k, v, b[0], b[1], do, ones, is_causal=causal)
        assert torch.equal(ga[1], gb[1]) and torch.equal(ga[2], gb[2])
        assert torch.allclose(ga[0].float(), gb[0].float(), atol=2e-3, rtol=0)
    assert ops.sdpa_device_status() == 0


def test_blocksparse_argument_errors():
    from _gpu import cuda
    dev = cuda()
    x = wl.dense_inputs(1, 1, 256, 256, 64, "f16", "normal", seed=48, with_do=False)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    with pytest.raises(ValueError):
        ops.sdpa_fwd_blocksparse(q, k, v, torch.ones((3, 2), dtype=torch.uint8, device=dev))
    lib = ops._abi.load()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    m = torch.ones((2, 2), dtype=torch.uint8, device=dev)
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 256, 256, 64, 0.125, 0]
    assert lib.sdpa_fwd_blocksparse(*args, None, 0, 0, 2, 1, None) == ops._abi.SDPA_ERR_ARG
    assert lib.sdpa_fwd_blocksparse(*args, m.data_ptr(), 0, 0, 1, 1, None) == ops._abi.SDPA_ERR_ARG
    assert lib.sdpa_fwd_blocksparse(*args, m.data_ptr(), -4, 0, 2, 1, None) == ops._abi.SDPA_ERR_ARG
