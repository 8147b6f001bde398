"""Per-query-head parameters (the tuned mode of the SpargeAttn overview page, one topk, theta
and lambda per head): every head's mask and output follow the oracle run on that head alone with
its own parameters; per-head arrays equal to the scalars give the scalar call bit for bit; an
entry out of range is reported in the device status word and its head falls back to keeping
every valid block (topk, theta) or to the filter off (lambda)."""
import math

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import COS_MIN, MAXABS, cos_maxabs, dev_bf16, f64, host_f64

pytestmark = pytest.mark.gpu

TOPK = [0.3, 0.5, 0.8, 1.0]
THETA = [0.2, 0.5, 0.9, 0.5]
LAM = [-math.inf, -12.0, -8.0, -4.0]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbs.lib()
    assert torch.cuda.is_available()
    yield
    torch.cuda.synchronize()
    assert fbs.device_status() == 0


def _workload():
    # Llama-like causal GQA with a ragged tail: 4 query heads over 2 KV heads
    return W.make_config("llama32k", N=2048 + 130, Hq=4, Hkv=2)


def _arr(x):
    return torch.tensor(x, dtype=torch.float32, device="cuda")


def _head(w, x, h):
    return f64(x[:, h:h + 1])


def test_per_head_parameters_match_oracle():
    w = _workload()
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, 0.5, w.causal, theta=0.5, lam=-8.0, mask_out=mask,
                             topk_per_head=_arr(TOPK), theta_per_head=_arr(THETA), lambda_per_head=_arr(LAM))
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_OK
    gm, got = mask.cpu().numpy(), host_f64(out)
    G = w.Hq // w.Hkv
    n_dec = 0
    for h in range(w.Hq):
        qh, kh, vh = _head(w, w.q, h), _head(w, w.k, h // G), _head(w, w.v, h // G)
        pred = oracle.predict_mask(qh, kh, TOPK[h], THETA[h], w.causal)
        dec = oracle.decisive_rows(pred, TOPK[h], THETA[h], w.causal)[0, 0]
        n_dec += int(dec.sum())
        np.testing.assert_array_equal(gm[0, h][dec], pred["mask"][0, 0][dec], err_msg="head %d" % h)
        ref = oracle.block_sparse_attn(qh, kh, vh, gm[:, h:h + 1], LAM[h], w.causal)
        cos, err = cos_maxabs(got[:, h:h + 1], ref)
        assert cos >= COS_MIN and err <= MAXABS, (h, cos, err)
    assert n_dec >= w.nqb  # at least a head's worth of rows compared bit for bit
    # the heads' masks differ as their parameters do (sparser for smaller topk)
    kept = gm.reshape(w.Hq, -1).sum(axis=1)
    assert kept[0] < kept[1] < kept[3]


def test_per_head_arrays_equal_to_scalars_are_the_scalar_call():
    w = _workload()
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    m1, m2 = (torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda") for _ in range(2))
    o1 = fbs.sparge_attn_ex(q, k, v, 0.4, w.causal, theta=0.6, lam=-6.0, mask_out=m1)
    # different scalars, overridden for every head by the first call's values
    o2 = fbs.sparge_attn_ex(q, k, v, 0.9, w.causal, theta=0.1, lam=-1.0, mask_out=m2,
                            topk_per_head=_arr([0.4] * w.Hq), theta_per_head=_arr([0.6] * w.Hq),
                            lambda_per_head=_arr([-6.0] * w.Hq))
    assert torch.equal(m1, m2) and torch.equal(o1, o2)
    p1 = fbs.predict_mask(q, k, 0.4, 0.6, w.causal)
    p2 = fbs.predict_mask_ex(q, k, 0.7, w.causal, theta=0.3, topk_per_head=_arr([0.4] * w.Hq),
                             theta_per_head=_arr([0.6] * w.Hq))
    assert torch.equal(p1, m1) and torch.equal(p2, m1)
    b1 = fbs.block_sparse_attn_ex(q, k, v, m1, w.causal, lam=-6.0)
    b2 = fbs.block_sparse_attn_ex(q, k, v, m1, w.causal, lam=-2.0, lambda_per_head=_arr([-6.0] * w.Hq))
    assert torch.equal(b1, o1) and torch.equal(b2, o1)
    assert fbs.device_status() == fbs.SPARGE_OK


def test_per_head_entries_out_of_range_are_reported():
    w = _workload()
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    topk = [0.5, 0.0, 0.5, 0.5]          # head 1: topk outside (0, 1]
    theta = [0.5, 0.5, math.nan, 0.5]    # head 2: theta not finite
    lam = [-8.0, -8.0, -8.0, 1.0]        # head 3: lambda > 0
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_OK
    out = fbs.sparge_attn_ex(q, k, v, 0.5, w.causal, theta=0.5, lam=-8.0, mask_out=mask,
                             topk_per_head=_arr(topk), theta_per_head=_arr(theta), lambda_per_head=_arr(lam))
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_ERR_INVALID_ARG
    assert fbs.device_status() == fbs.SPARGE_OK   # reading clears the word
    gm, got = mask.cpu().numpy(), host_f64(out)
    valid = oracle.block_valid(w.nqb, w.nkb, w.causal)
    for h in (1, 2):                     # a bad topk or theta keeps every valid block of the head
        assert np.array_equal(gm[0, h].astype(bool), valid), h
    G = w.Hq // w.Hkv
    for h, lam_ref in ((0, -8.0), (3, -math.inf)):   # a bad lambda turns the filter off
        qh, kh, vh = _head(w, w.q, h), _head(w, w.k, h // G), _head(w, w.v, h // G)
        ref = oracle.block_sparse_attn(qh, kh, vh, gm[:, h:h + 1], lam_ref, w.causal)
        cos, err = cos_maxabs(got[:, h:h + 1], ref)
        assert cos >= COS_MIN and err <= MAXABS, (h, cos, err)
