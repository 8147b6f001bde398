"""GPU checks of the 8-bit attention paths (d = 128).

The pages fix only that the path is 8-bit with outlier smoothing, so its output is held to a
tolerance against the float64 oracle of the unquantised method, given the same mask: cosine
>= 0.999 for every 8-bit precision.

Where a precision is known to fall short of that bound the case is marked xfail(strict=True),
so it fails if the precision ever passes it, and the measured cosine is in the reason:

- SPARGE_PRECISION_BF16_FP8PV (bf16 Q.K^T, e4m3 P.V) meets it everywhere (measured 0.99925 -
  0.99968 on i.i.d. and Llama-like data, 0.999995 on Flux-like data);
- SPARGE_PRECISION_Q8 (e4m3 Q.K^T, f16 P.V) meets it on i.i.d. and Flux-like data but not on the
  Llama-like data (0.9953): its rotary structure and 8x-norm sink keys give large, aligned scores,
  on which the 3-bit mantissa of e4m3 (a relative error up to 2^-4, where the pages' INT8 has
  an absolute error of max/254) moves peaked softmax rows;
- SPARGE_PRECISION_Q8_FP8PV (e4m3 for both) falls short on i.i.d. data too (0.9986 - 0.9989):
  three e4m3 roundings (scores, P, V), each of rms relative size about 2^-4 / sqrt(3) x 0.7,
  cost 1 - cos of about 1.2e-3.

The quantised copies the path leaves in its workspace are checked against their definitions
(per-block and per-channel scales, K mean, e4m3 round-to-nearest within half a code step)."""
import math

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import cos_maxabs, dev_bf16, f64, host_f64

pytestmark = pytest.mark.gpu

Q8, FP8PV, BF16PV = fbs.SPARGE_PRECISION_Q8, fbs.SPARGE_PRECISION_Q8_FP8PV, fbs.SPARGE_PRECISION_BF16_FP8PV
COS_MIN = 0.999
PRECS = [Q8, FP8PV, BF16PV]


def short(prec, measured):
    """A precision parameter marked as known to fall short of COS_MIN on the case (strict)."""
    return pytest.param(prec, marks=pytest.mark.xfail(strict=True, reason="measured cosine %s < 0.999" % measured))


# i.i.d. data: FP8PV short; Llama-like data: Q8 and FP8PV short
PRECS_IID = [Q8, short(FP8PV, "0.9986-0.9989"), BF16PV]
PRECS_STRUCT = [short(Q8, "0.9953"), short(FP8PV, "0.9950"), BF16PV]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbs.lib()
    assert torch.cuda.is_available()
    yield
    torch.cuda.synchronize()
    assert fbs.device_status() == 0


def _e4m3_half_step(y: np.ndarray) -> np.ndarray:
    """Half the spacing of e4m3 codes around |y| (3 mantissa bits; subnormal step 2^-9)."""
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 0.5 * np.exp2(e - 3)


def _decode(codes: torch.Tensor) -> np.ndarray:
    return codes.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


DENSE_CASES = [(N, Hq, Hkv, causal) for N, Hq, Hkv in [(128, 1, 1), (1000, 4, 1), (2100, 2, 2)] for causal in (False, True)]
# FP8PV reaches the bound on the single causal tile (0.99918), not on the other cases
DENSE_PARAMS = ([(Q8,) + c for c in DENSE_CASES] + [(BF16PV,) + c for c in DENSE_CASES] +
                [(FP8PV,) + c if c == (128, 1, 1, True) else
                 pytest.param(FP8PV, *c, marks=pytest.mark.xfail(strict=True, reason="measured cosine 0.9986-0.9989 < 0.999"))
                 for c in DENSE_CASES])


@pytest.mark.parametrize("prec,N,Hq,Hkv,causal", DENSE_PARAMS)
def test_q8_dense_attention(prec, N, Hq, Hkv, causal):
    qu, ku, vu = W.random_qkv(31, 1, Hq, Hkv, N, 128)
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, causal, precision=prec)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, causal)
    cos, _ = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN, cos


@pytest.mark.parametrize("prec", PRECS_IID)
def test_q8_offset_keys_and_large_values(prec):
    """K with a large common offset (the case the mean smoothing is for) and V of magnitude 30."""
    N, H = 1500, 2
    rng = np.random.Generator(np.random.PCG64(32))
    qu, ku, vu = W.random_qkv(33, 1, H, H, N, 128)
    k = f64(ku) + 4.0 * rng.standard_normal((1, H, 1, 128))
    v = 30.0 * f64(vu)
    ku2, vu2 = W.bf16_bits(k), W.bf16_bits(v)
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku2), dev_bf16(vu2), None, -math.inf, False, precision=prec)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku2), f64(vu2), None, -math.inf, False)
    cos, _ = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN, cos


@pytest.mark.parametrize("prec", PRECS_IID)
@pytest.mark.parametrize("lam", [-math.inf, -12.0, -8.0, -4.0])
def test_q8_custom_mask_lambda_sweep(prec, lam):
    """The custom-mask workload shrunk (B 2, 2 heads, ragged N): Bernoulli(0.25) tiles with the
    diagonal forced on, through the block-sparse call, over the lambda sweep."""
    w = W.make_config("custom", Hq=2, Hkv=2, N=3000)
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.from_numpy(w.mask).cuda()
    out = fbs.block_sparse_attn(q, k, v, mask, lam, w.causal, precision=prec)
    ref = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), w.mask, lam, w.causal)
    cos, _ = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN, cos
    bf = fbs.block_sparse_attn(q, k, v, mask, lam, w.causal)
    cos_bf, _ = cos_maxabs(host_f64(bf), ref)
    assert cos_bf >= cos - 1e-6  # the bf16 path is the more accurate one


@pytest.mark.parametrize("prec", PRECS_STRUCT)
def test_q8_empty_row_and_causal_llama(prec):
    w = W.make_config("llama32k", N=2048 + 77, Hq=4, Hkv=1)
    mask = W.random_mask(34, 1, 4, w.N, p=0.4, force_diag=True)
    mask[0, 1, 5] = 0
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    out = fbs.block_sparse_attn(q, k, v, torch.from_numpy(mask).cuda(), -math.inf, True, precision=prec)
    ref = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), mask, -math.inf, True)
    got = host_f64(out)
    assert (got[0, 1, 5 * 128:6 * 128] == 0).all()
    cos, _ = cos_maxabs(got, ref)
    assert cos >= COS_MIN, cos


@pytest.mark.parametrize("prec", PRECS_STRUCT)
def test_q8_end_to_end_predicted_mask(prec):
    w = W.make_config("llama32k", N=4096 + 200, Hq=8, Hkv=2)
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, lam=w.lam, precision=prec, mask_out=mask)
    ref = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), mask.cpu().numpy(), w.lam, w.causal)
    cos, _ = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN, cos


@pytest.mark.parametrize("prec", PRECS)
def test_q8_end_to_end_flux_like(prec):
    """Flux-like image data (smooth fields, text prefix) through the predicted mask: every 8-bit
    precision meets the bound."""
    w = W.make_config("flux", Hq=4, Hkv=4)
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, lam=w.lam, precision=prec, mask_out=mask)
    ref = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), mask.cpu().numpy(), w.lam, w.causal)
    cos, _ = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN, cos


def test_q8_quantised_copies():
    B, Hq, Hkv, N, d = 2, 4, 2, 1000, 128
    qu, ku, vu = W.random_qkv(35, B, Hq, Hkv, N, d)
    ws = torch.zeros(fbs.workspace_bytes(fbs.SPARGE_OP_BLOCK_SPARSE_ATTN_Q8, B, Hq, Hkv, N, d), dtype=torch.uint8,
                     device="cuda")
    fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, False, precision=FP8PV, ws=ws)
    torch.cuda.synchronize()
    wv = fbs.q8_ws_views(ws, B, Hq, Hkv, N, d)
    q, k, v = f64(qu), f64(ku), f64(vu)
    nqb, nkb = -(-N // 128), -(-N // 64)
    # K mean over the tokens of each (batch, KV head)
    kmean = k.mean(axis=2)
    np.testing.assert_allclose(wv["kmean"].cpu().numpy(), kmean, rtol=1e-5, atol=1e-6)
    # Q per 128-token block, K - mean per 64-token block: scale = max|x| / 448
    ks = k - wv["kmean"].cpu().numpy().astype(np.float64)[:, :, None, :]
    for x, blk, nb, codes, sc in ((q, 128, nqb, wv["q8"], wv["sq"]), (ks, 64, nkb, wv["k8"], wv["sk"])):
        pad = nb * blk - N
        xb = np.pad(x, ((0, 0), (0, 0), (0, pad), (0, 0))).reshape(x.shape[0], x.shape[1], nb, blk * d)
        smax = np.abs(xb).max(axis=3) / 448.0
        s_gpu = sc.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(s_gpu, smax, rtol=1e-5)
        y = x / np.repeat(s_gpu, blk, axis=2)[:, :, :N, None]
        dec = _decode(codes)
        assert np.all(np.abs(dec - y) <= _e4m3_half_step(y) * 1.001 + 1e-9)
    # V per channel, stored channel-major with the keys padded to a multiple of 64 (zeros)
    sv = wv["sv"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(sv, np.abs(v).max(axis=2) / 448.0, rtol=1e-6)
    v8 = wv["v8"]
    dec = _decode(v8[..., :N].contiguous()).transpose(0, 1, 3, 2)
    y = v / sv[:, :, None, :]
    assert np.all(np.abs(dec - y) <= _e4m3_half_step(y) * 1.001 + 1e-9)
    assert int(v8[..., N:].count_nonzero()) == 0
    # bf16 Q.K^T with e4m3 P.V quantises V the same way (and leaves Q and K alone)
    ws2 = torch.zeros_like(ws)
    fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, False, precision=BF16PV, ws=ws2)
    torch.cuda.synchronize()
    wv2 = fbs.q8_ws_views(ws2, B, Hq, Hkv, N, d)
    assert torch.equal(wv2["v8"], v8) and torch.equal(wv2["sv"], wv["sv"])
    assert int(wv2["q8"].count_nonzero()) == 0 and int(wv2["k8"].count_nonzero()) == 0


@pytest.mark.parametrize("prec", PRECS)
def test_q8_rejects_d64_and_reports(prec):
    qu, ku, vu = W.random_qkv(36, 1, 1, 1, 256, 64)
    with pytest.raises(fbs.SpargeError) as e:
        fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, False, precision=prec,
                              ws=torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.code == fbs.SPARGE_ERR_UNSUPPORTED
    assert fbs.workspace_bytes(fbs.SPARGE_OP_BLOCK_SPARSE_ATTN_Q8, 1, 1, 1, 256, 64) == 0
