"""Queries shorter than keys (a chunk of queries continuing a longer key sequence: prefill in
chunks, decoding), and without the causal mask queries longer than keys: masks bit-exact on
decisive rows and outputs within the bf16 bounds against the oracle run on the same shapes; the
last query sits on the last key."""
import math

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import COS_MIN, MAXABS, cos_maxabs, dev_bf16, f64, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbs.lib()
    assert torch.cuda.is_available()
    yield
    torch.cuda.synchronize()
    assert fbs.device_status() == 0


def _tensors(seed, Nq, Nk, Hq, Hkv, d):
    """Block-structured Q and K (per 64-token block a common direction plus noise) and i.i.d. V."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = W._block_mean_tokens(rng, 1, Hq, Nq, d)
    k = W._block_mean_tokens(rng, 1, Hkv, Nk, d)
    v = W.random_qkv(seed + 1, 1, Hkv, Hkv, Nk, d)[2]
    return q, k, v


@pytest.mark.parametrize("causal,Nq,Nk,d", [
    (True, 256 + 40, 4096 + 100, 128),   # a chunk of a long prefill, ragged tails on both sides
    (True, 1024, 4096, 64),
    (True, 7, 3000, 128),                 # a few decoding steps
    (True, 1, 513, 64),                   # one query
    (False, 640, 1920, 128),
    (False, 1000, 300, 64),               # without the causal mask queries may outnumber keys
])
def test_short_query_matches_oracle(causal, Nq, Nk, d):
    Hq, Hkv, topk, theta, lam = 4, 2, 0.5, 0.5, -8.0
    qu, ku, vu = _tensors(Nq + Nk, Nq, Nk, Hq, Hkv, d)
    q, k, v = dev_bf16(qu), dev_bf16(ku), dev_bf16(vu)
    nqb, nkb = -(-Nq // 128), -(-Nk // 64)
    mask = torch.empty((1, Hq, nqb, nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, topk, causal, theta=theta, lam=lam, mask_out=mask)
    assert out.shape == q.shape
    gm = mask.cpu().numpy()
    pred = oracle.predict_mask(f64(qu), f64(ku), topk, theta, causal)
    assert pred["mask"].shape == gm.shape
    valid = oracle.block_valid(nqb, nkb, causal, Nk - Nq)
    assert not gm[:, :, ~valid].any()
    assert (gm.sum(axis=-1) >= 1).all()
    dec = oracle.decisive_rows(pred, topk, theta, causal)
    assert not ((gm != pred["mask"]).any(axis=-1) & dec).any()
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), gm, lam, causal)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    # stage 1 alone and the block-sparse call on the same mask give the same results
    assert torch.equal(fbs.predict_mask(q, k, topk, theta, causal), mask)
    assert torch.equal(fbs.block_sparse_attn(q, k, v, mask, lam, causal), out)


def test_short_query_dense_is_tail_of_full_causal():
    """topk 1: the chunk's output is the last Nq rows of causal attention over a sequence that
    ends with the chunk (the GPU's full-length call as the second route)."""
    Nq, Nk, Hq, Hkv, d = 300, 2000, 2, 1, 128
    qu, ku, vu = _tensors(77, Nq, Nk, Hq, Hkv, d)
    prefix = W.random_qkv(78, 1, Hq, Hkv, Nk - Nq, d)[0]
    qf = np.concatenate([prefix, qu], axis=2)
    q, k, v, qfd = dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), dev_bf16(qf)
    short = fbs.sparge_attn_ex(q, k, v, 1.0, True, theta=0.5)
    full = fbs.sparge_attn_ex(qfd, k, v, 1.0, True, theta=0.5)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, True)
    cos, err = cos_maxabs(host_f64(short), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    cos, err = cos_maxabs(host_f64(short), host_f64(full)[:, :, Nk - Nq:])
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


@pytest.mark.parametrize("prec", [
    fbs.SPARGE_PRECISION_Q8,            # measured 0.99926
    pytest.param(fbs.SPARGE_PRECISION_Q8_FP8PV,
                 marks=pytest.mark.xfail(strict=True, reason="e4m3 scores, P and V: measured cosine 0.99861 < 0.999")),
    fbs.SPARGE_PRECISION_BF16_FP8PV,    # measured 0.99935
])
def test_short_query_8bit(prec):
    """A short causal query chunk (Nq < Nk, ragged tails) on every 8-bit precision, held to the
    8-bit bound (cosine >= 0.999 against the float64 oracle)."""
    Nq, Nk, Hq, Hkv, d = 384 + 5, 2048 + 33, 4, 2, 128
    qu, ku, vu = W.random_qkv(79, 1, Hq, Hkv, Nk, d)
    qu = qu[:, :, :Nq].copy()
    q, k, v = dev_bf16(qu), dev_bf16(ku), dev_bf16(vu)
    out = fbs.block_sparse_attn(q, k, v, None, -math.inf, True, precision=prec)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, True)
    cos, _ = cos_maxabs(host_f64(out), ref)
    print("short query 8-bit precision %d: cosine %.6f" % (prec, cos))
    assert cos >= 0.999, cos
