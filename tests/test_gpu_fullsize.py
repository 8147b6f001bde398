"""GPU parity at the full sizes of the named workloads, in the launch configuration the bench
times (one sparge_attn_ex call with the predicted mask, or the block-sparse call on the custom
workload's own mask).  The oracle is too slow for whole outputs at these sizes, so sampled query
blocks are checked one by one: the mask row against the oracle's single-row prediction
(bit-exact where the row is decisive), and the output rows of the block against the oracle's
single-block attention given the GPU's mask row.  Properties that hold at any size (no kept tile
above the causal diagonal, at least one kept block per row) are checked on the whole mask."""
import functools
import math

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import COS_MIN, MAXABS, cos_maxabs, dev_bf16, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbs.lib()
    assert torch.cuda.is_available()
    yield
    torch.cuda.synchronize()
    assert fbs.device_status() == 0


@functools.lru_cache(maxsize=2)
def _workload(name):
    return W.make_config(name)


def _samples(w, n):
    """n (b, h, i) query blocks spread over batches, heads and positions, the first and last
    blocks included."""
    rng = np.random.Generator(np.random.PCG64(7))
    out = [(0, 0, 0), (w.B - 1, w.Hq - 1, w.nqb - 1), (0, w.Hq // 2, w.nqb // 2)]
    while len(out) < n:
        out.append((int(rng.integers(w.B)), int(rng.integers(w.Hq)), int(rng.integers(w.nqb))))
    return out


def _block(x16, b, h, i):
    return f64(x16[b, h, i * 128:min(x16.shape[2], (i + 1) * 128)])


def _check_whole_mask(w, gm):
    valid = oracle.block_valid(w.nqb, w.nkb, w.causal)
    assert not gm[:, :, ~valid].any(), "kept tiles above the causal diagonal"
    assert (gm.sum(axis=-1) >= 1).all(), "a row keeps no block"


def _check_cut_properties(w, pr, row, where, eps=1e-3):
    """What any correct cut satisfies on a row whose cut rounding may move: the always-keep
    blocks are kept, the kept mass reaches topk (within eps), no kept top-k block is more than
    eps below the oracle's cut probability and no dropped block more than eps above it."""
    valid, p, sk = pr["valid"], pr["P"], pr["sK"]
    kept = row.astype(bool)
    assert not (kept & ~valid).any(), where
    if pr["sQ"] < w.theta - eps:
        assert kept[valid].all(), where
        return
    assert kept[valid & (sk < w.theta - eps)].all(), where
    assert p[kept].sum() >= min(1.0, w.topk) - eps, where
    if w.topk >= 1.0:
        return
    order = np.nonzero(valid)[0]
    order = order[np.lexsort((order, -p[order]))]
    c = np.cumsum(p[order])
    kstar = int(np.nonzero(c >= w.topk)[0][0]) + 1 if (c >= w.topk).any() else order.size
    p_cut = p[order[kstar - 1]]
    topk_part = kept & valid & ~(sk < w.theta + eps)  # blocks kept for their probability
    assert (p[topk_part] >= p_cut - eps).all(), where
    assert (p[valid & ~kept] <= p_cut + eps).all(), where


def _check_block(w, gm, got, b, h, i, lam, predicted, cos_min=COS_MIN, maxabs=MAXABS):
    kvh = h // (w.Hq // w.Hkv)
    kh, vh = f64(w.k[b, kvh]), f64(w.v[b, kvh])
    qi = _block(w.q, b, h, i)
    row = gm[b, h, i]
    decisive = False
    if predicted:
        pr = oracle.predict_mask_row(qi, kh, i, w.topk, w.theta, w.causal)
        decisive = oracle.row_decisive(pr["P"], pr["valid"], pr["sQ"], pr["sK"], w.topk, w.theta)
        if decisive:
            assert np.array_equal(row, pr["mask"]), (b, h, i)
        else:
            _check_cut_properties(w, pr, row, (b, h, i))
    valid = oracle.block_valid(w.nqb, w.nkb, w.causal)[i]
    kept = np.nonzero(row.astype(bool) & valid)[0]
    ref, _ = oracle.attn_qblock(qi, kh, vh, i, kept, lam, w.causal, oracle.default_scale(w.d))
    g = got[b, h, i * 128:i * 128 + qi.shape[0]].float().cpu().numpy().astype(np.float64)
    cos, err = cos_maxabs(g, ref)
    assert cos >= cos_min and err <= maxabs, ((b, h, i), cos, err)
    return decisive


@pytest.mark.parametrize("name,nsamp", [("llama128k", 12), ("llama32k", 12), ("flux", 8), ("cogvideox", 8),
                                         ("vit", 8)])
def test_full_size_predicted_mask_and_attention(name, nsamp):
    w = _workload(name)
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    perm = None
    if w.grid is not None:
        # image and video tokens in Hilbert order, as the workload prescribes: the permuted
        # tensors bit-exact, then the whole check on the permuted workload, then the inverse
        perm_np = (fbs.hilbert_perm_2d(w.n_prefix, *w.grid) if len(w.grid) == 2
                   else fbs.hilbert_perm_3d(w.n_prefix, *w.grid))
        perm = torch.from_numpy(perm_np).cuda()
        q, k, v = (fbs.permute_tokens(t, perm) for t in (q, k, v))
        wp = W.Workload(**{**w.__dict__})
        wp.q, wp.k, wp.v = w.q[:, :, perm_np], w.k[:, :, perm_np], w.v[:, :, perm_np]
        for dev_t, host_t in ((q, wp.q), (k, wp.k), (v, wp.v)):
            assert np.array_equal(dev_t.cpu().view(torch.int16).numpy().view(np.uint16), host_t)
        w = wp
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, lam=w.lam, mask_out=mask)
    if perm is not None:
        natural = fbs.unpermute_tokens(out, perm)
        assert torch.equal(fbs.permute_tokens(natural, perm), out)
    torch.cuda.synchronize()
    gm = mask.cpu().numpy()
    _check_whole_mask(w, gm)
    n_dec = sum(_check_block(w, gm, out, b, h, i, w.lam, predicted=True) for b, h, i in _samples(w, nsamp))
    # at least one sampled row compared bit for bit (rows of many nearly equal block
    # probabilities, as at 128K or in Hilbert order, are often not decisive)
    assert n_dec >= 1, n_dec


@pytest.mark.parametrize("prec,cos_min", [(fbs.SPARGE_PRECISION_BF16, COS_MIN), (fbs.SPARGE_PRECISION_Q8, 0.999),
                                          (fbs.SPARGE_PRECISION_Q8_FP8PV, 0.998)])
def test_full_size_custom_mask(prec, cos_min):
    """The custom-mask workload at full size (B 2, 16 heads, N 65536) through the block-sparse
    call on its own mask, in each precision; the 8-bit ones at their cosine bounds only."""
    w = _workload("custom")
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    out = fbs.block_sparse_attn_ex(q, k, v, torch.from_numpy(w.mask).cuda(), w.causal, lam=w.lam, precision=prec)
    torch.cuda.synchronize()
    maxabs = MAXABS if prec == fbs.SPARGE_PRECISION_BF16 else math.inf
    for b, h, i in _samples(w, 6):
        _check_block(w, w.mask, out, b, h, i, w.lam, predicted=False, cos_min=cos_min, maxabs=maxabs)
