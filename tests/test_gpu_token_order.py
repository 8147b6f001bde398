"""Token order inside the call (the Hilbert order of image and video tokens without separate V
and output passes): bit for bit the same mask and output as permuting q, k and v, calling, and
permuting the output back, in every precision and through every call that takes a
sparge_params; against the oracle on the reordered workload; permutation entries out of range
reported without a stray access."""
import math

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import COS_MIN, MAXABS, cos_maxabs, dev_bf16, f64, host_f64

pytestmark = pytest.mark.gpu

SMALL = {
    "flux": dict(name="flux", Hq=4, Hkv=4),
    "cogvideox": dict(name="cogvideox", Hq=2, Hkv=2, grid=(5, 30, 45)),
}
BF16, Q8, FP8PV = fbs.SPARGE_PRECISION_BF16, fbs.SPARGE_PRECISION_Q8, fbs.SPARGE_PRECISION_Q8_FP8PV
BF16PV = fbs.SPARGE_PRECISION_BF16_FP8PV


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbs.lib()
    assert torch.cuda.is_available()
    yield
    torch.cuda.synchronize()
    assert fbs.device_status() == 0


def _make(key):
    spec = dict(SMALL[key])
    w = W.make_config(spec.pop("name"), **spec)
    perm = (fbs.hilbert_perm_2d(w.n_prefix, *w.grid) if len(w.grid) == 2
            else fbs.hilbert_perm_3d(w.n_prefix, *w.grid))
    return w, perm


def _empty_mask(w):
    return torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("key,prec", [("flux", BF16), ("flux", Q8), ("flux", FP8PV), ("flux", BF16PV),
                                      ("cogvideox", BF16)])
def test_token_order_equals_explicit_permutes(key, prec):
    """With contiguous inputs the bf16 Q.K^T paths read Q and K in place (pooling through the order,
    the attention's tiles by TMA gathers, Q rows into TMEM at d = 64): no ordered copies."""
    w, perm_np = _make(key)
    perm = torch.from_numpy(perm_np).cuda()
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    pq, pk, pv = (fbs.permute_tokens(t, perm) for t in (q, k, v))
    m1, m2 = _empty_mask(w), _empty_mask(w)
    po = fbs.sparge_attn_ex(pq, pk, pv, w.topk, w.causal, theta=w.theta, lam=-8.0, precision=prec, mask_out=m1)
    o1 = fbs.unpermute_tokens(po, perm)
    o2 = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, lam=-8.0, precision=prec, mask_out=m2,
                            token_order=perm)
    assert torch.equal(m1, m2)
    assert torch.equal(o1, o2)
    # the block-sparse call on a mask of the reordered sequence
    b1 = fbs.unpermute_tokens(fbs.block_sparse_attn_ex(pq, pk, pv, m1, w.causal, precision=prec), perm)
    b2 = fbs.block_sparse_attn_ex(q, k, v, m1, w.causal, precision=prec, token_order=perm)
    assert torch.equal(b1, b2)
    # stage 1 alone
    p2 = fbs.predict_mask_ex(q, k, w.topk, w.causal, theta=w.theta, token_order=perm)
    assert torch.equal(p2, m1)
    assert fbs.device_status() == fbs.SPARGE_OK


def test_token_order_matches_oracle():
    w, perm_np = _make("cogvideox")
    perm = torch.from_numpy(perm_np).cuda()
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    m = _empty_mask(w)
    out = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, mask_out=m, token_order=perm)
    gm = m.cpu().numpy()
    wp = W.Workload(**{**w.__dict__})
    wp.q, wp.k, wp.v = w.q[:, :, perm_np], w.k[:, :, perm_np], w.v[:, :, perm_np]
    pred = oracle.predict_mask(f64(wp.q), f64(wp.k), w.topk, w.theta, w.causal)
    dec = oracle.decisive_rows(pred, w.topk, w.theta, w.causal)
    assert dec.mean() > 0.2
    assert not ((gm != pred["mask"]).any(axis=-1) & dec).any()
    ref = oracle.unpermute_tokens(
        oracle.block_sparse_attn(f64(wp.q), f64(wp.k), f64(wp.v), gm, -math.inf, w.causal), perm_np)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


@pytest.mark.parametrize("key", ["flux", "cogvideox"])
def test_token_order_entries_out_of_range_are_reported(key):
    """Entries outside 0..N-1 are never used as addresses: the call finishes, the status word
    reports SPARGE_ERR_INVALID_ARG, output rows that no valid entry targets keep their old
    contents, and every written row is finite (the ordered copies and the gathers read zero rows
    there; at d = 64 Q is gathered, not copied).  Mask prediction alone (rows gathered by the
    pooling, no copies) reports the same."""
    w, perm_np = _make(key)
    bad = [0, 700, w.N - 1]
    perm_np = perm_np.copy()
    lost = perm_np[bad].copy()              # tokens no entry points at any more
    perm_np[bad[0]], perm_np[bad[1]], perm_np[bad[2]] = -3, w.N, 1 << 30
    perm = torch.from_numpy(perm_np).cuda()
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    out = torch.full_like(q, 5.0)
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_OK
    fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, out=out, token_order=perm)
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_ERR_INVALID_ARG
    assert fbs.device_status() == fbs.SPARGE_OK
    o = out.float().cpu().numpy()
    assert (o[:, :, lost] == 5.0).all()
    written = np.setdiff1d(np.arange(w.N), lost)
    assert np.isfinite(o[:, :, written]).all() and not (o[:, :, written] == 5.0).all()
    m = fbs.predict_mask_ex(q, k, w.topk, w.causal, theta=w.theta, token_order=perm)
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_ERR_INVALID_ARG
    assert m.shape == (w.B, w.Hq, w.nqb, w.nkb)


@pytest.mark.parametrize("key", ["flux", "cogvideox"])
def test_token_order_with_strided_rows_falls_back_to_copies(key):
    """Q and K views whose heads are not packed back to back (a slice of longer sequences) cannot be
    gathered through one row map: the call copies them in order instead, with the same result."""
    w, perm_np = _make(key)
    perm = torch.from_numpy(perm_np).cuda()
    pad = 256
    big = [torch.zeros((t.shape[0], t.shape[1], w.N + pad, w.d), dtype=torch.bfloat16, device="cuda")
           for t in (w.q, w.k)]
    big[0][:, :, :w.N] = dev_bf16(w.q)
    big[1][:, :, :w.N] = dev_bf16(w.k)
    q, k = big[0][:, :, :w.N], big[1][:, :, :w.N]
    v = dev_bf16(w.v)
    assert q.stride(1) != w.N * w.d
    m1, m2 = _empty_mask(w), _empty_mask(w)
    o1 = fbs.sparge_attn_ex(q.contiguous(), k.contiguous(), v, w.topk, w.causal, theta=w.theta, mask_out=m1,
                            token_order=perm)
    o2 = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, mask_out=m2, token_order=perm)
    assert torch.equal(m1, m2)
    assert torch.equal(o1, o2)
    assert fbs.device_status() == fbs.SPARGE_OK
