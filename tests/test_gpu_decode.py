"""Decoding tiles (few queries per head against many keys): the G Nq query rows of the heads that
share a KV head are packed into one 128-row tile, the key blocks are split over CTAs and the
chunks' partial rows combined.  The library takes this path by itself for bf16 calls with the
lambda filter off, no token order and G Nq <= 128 against at least 32 key blocks; these tests hold
it to the float64 oracle (given mask: masks that differ per head, heads with nothing kept,
causal alignment of the last query on the last key, ragged key tails, d = 64 and 128) and to the
regular kernel."""
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


def _qkv(seed, B, Hq, Hkv, Nq, Nk, d):
    qu, _, _ = W.random_qkv(seed, B, Hq, Hkv, Nq, d)
    _, ku, vu = W.random_qkv(seed + 1, B, Hq, Hkv, Nk, d)
    return qu, ku, vu


def _mask(seed, B, Hq, Nq, Nk, p):
    rng = np.random.Generator(np.random.PCG64(seed))
    nqb, nkb = -(-Nq // 128), -(-Nk // 64)
    m = (rng.random((B, Hq, nqb, nkb)) < p).astype(np.uint8)
    m[..., -1] = 1  # the last key block (holding the last keys the causal queries see)
    return m


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,p", [
    (1, 32, 8, 1, 4096 + 77, 128, True, 0.3),     # single-token decoding, GQA 4, ragged key tail
    (1, 8, 2, 4, 3000, 64, False, 0.5),           # a few queries, d = 64, non-causal
    (2, 16, 2, 16, 8192, 128, True, 0.2),         # G Nq = 128 rows, two batches
    (1, 4, 4, 1, 2048, 128, False, 1.0),          # no GQA, every block kept
    (1, 8, 1, 12, 5000, 64, True, 0.25),          # G = 8, d = 64, causal
])
def test_decode_matches_oracle(B, Hq, Hkv, Nq, Nk, d, causal, p):
    qu, ku, vu = _qkv(40, B, Hq, Hkv, Nq, Nk, d)
    m = _mask(41, B, Hq, Nq, Nk, p)
    if Hq > 1:
        m[0, 1] = 0                      # a head that keeps nothing: zero rows
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), torch.from_numpy(m).cuda(), -math.inf,
                                causal)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), m, -math.inf, causal)
    got = host_f64(out)
    cos, err = cos_maxabs(got, ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    if Hq > 1:
        assert (got[0, 1] == 0).all()


def test_decode_equals_regular_kernel_closely():
    """The split over key chunks against the regular kernel (taken when the lambda filter is on; a
    lambda of -1e30 never skips) on the same mask."""
    B, Hq, Hkv, Nq, Nk, d = 1, 16, 4, 2, 6000, 128
    qu, ku, vu = _qkv(42, B, Hq, Hkv, Nq, Nk, d)
    m = torch.from_numpy(_mask(43, B, Hq, Nq, Nk, 0.4)).cuda()
    q, k, v = dev_bf16(qu), dev_bf16(ku), dev_bf16(vu)
    a = fbs.block_sparse_attn(q, k, v, m, -math.inf, True)
    b = fbs.block_sparse_attn(q, k, v, m, -1e30, True)
    cos, err = cos_maxabs(host_f64(a), host_f64(b))
    assert cos >= 0.99999 and err <= 1e-2, (cos, err)


@pytest.mark.parametrize("N,d", [(4096 + 200, 128), (40000 + 37, 128), (40000 + 37, 64)])
def test_decode_through_sparge_attn_ex(N, d):
    """A decoding step with the predicted mask: one query token per head continuing a Llama-like
    sequence (8 query heads, 2 KV heads); at 40037 keys the pooled scores of the few query rows
    come in three slices of 256 key blocks with their own row maxima."""
    w = W.make_config("llama32k", N=N, Hq=8, Hkv=2, d=d)
    # the pooled scores of the single query block (a row kernel at this shape) against the oracle's
    qs, kd = dev_bf16(np.ascontiguousarray(w.q[:, :, -1:])), dev_bf16(w.k)
    ws = torch.zeros(fbs.workspace_bytes(fbs.SPARGE_OP_PREDICT_MASK, 1, 8, 2, N, d), dtype=torch.uint8, device="cuda")
    fbs.predict_mask(qs, kd, w.topk, w.theta, True, ws=ws)
    torch.cuda.synchronize()
    S = fbs.predict_ws_views(ws, 1, 8, 2, 1, d, Nk=N)[4].cpu().numpy().astype(np.float64)
    rmuQ, _ = oracle.pool_sim(f64(w.q[:, :, -1:]), 128)
    rmuK, _ = oracle.pool_sim(f64(w.k), 64)
    rS = oracle.pooled_scores(rmuQ, rmuK, True, oracle.default_scale(d), off=N - 1)
    valid = np.isfinite(rS)
    np.testing.assert_allclose(S[valid], rS[valid], rtol=1e-4, atol=2e-4)
    q = w.q[:, :, -1:]
    qd, k, v = dev_bf16(np.ascontiguousarray(q)), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((1, 8, 1, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(qd, k, v, w.topk, True, theta=w.theta, mask_out=mask)
    gm = mask.cpu().numpy()
    pred = oracle.predict_mask(f64(q), f64(w.k), w.topk, w.theta, True)
    dec = oracle.decisive_rows(pred, w.topk, w.theta, True)
    assert not ((gm != pred["mask"]).any(axis=-1) & dec).any()
    ref = oracle.block_sparse_attn(f64(q), f64(w.k), f64(w.v), gm, -math.inf, True)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


@pytest.mark.parametrize("causal", [True, False])
def test_decode_without_mask_is_dense(causal):
    """No mask: every key block is shared out over the CTAs (no listing pass), against dense
    attention from the oracle."""
    B, Hq, Hkv, Nq, Nk, d = 1, 8, 2, 3, 5000 + 11, 128
    qu, ku, vu = _qkv(44, B, Hq, Hkv, Nq, Nk, d)
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, causal)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, causal)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


def test_decode_bunched_mask_matches_oracle():
    """Kept blocks bunched into a few stretches of the key range (the shape of real decoding masks:
    the first blocks, a few recent stretches, the last block), so that equal key ranges would give
    some CTAs most of the work; each head keeps its own subset of the stretches."""
    B, Hq, Hkv, Nq, Nk, d = 1, 16, 4, 1, 40000, 128
    qu, ku, vu = _qkv(45, B, Hq, Hkv, Nq, Nk, d)
    nkb = -(-Nk // 64)
    rng = np.random.Generator(np.random.PCG64(46))
    m = np.zeros((B, Hq, 1, nkb), dtype=np.uint8)
    for h in range(Hq):
        m[0, h, 0, :4] = 1
        for s in rng.choice(np.arange(0, nkb - 40, 40), size=3, replace=False):
            m[0, h, 0, s:s + int(rng.integers(5, 40))] = 1
        m[0, h, 0, -1] = 1
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), torch.from_numpy(m).cuda(), -math.inf, True)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), m, -math.inf, True)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
