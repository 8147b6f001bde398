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
from mask_checks import EPS_SIM, cut_violations, decisive, score_error_bound, slack

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


def _check_attention(w, gm, got, b, h, i, lam, kh, vh, cos_min=COS_MIN, maxabs=MAXABS):
    """The output rows of query block (b, h, i) against the oracle's single-block attention over
    the GPU's mask row."""
    qi = _block(w.q, b, h, i)
    valid = oracle.block_valid(w.nqb, w.nkb, w.causal)[i]
    kept = np.nonzero(gm[b, h, i].astype(bool) & valid)[0]
    ref, _ = oracle.attn_qblock(qi, kh, vh, i, kept, lam, w.causal, oracle.default_scale(w.d))
    g = got[b, h, i * 128:i * 128 + qi.shape[0]].float().cpu().numpy().astype(np.float64)
    cos, err = cos_maxabs(g, ref)
    assert cos >= cos_min and err <= maxabs, ((b, h, i), cos, err)


def _check_mask_rows(w, gm, ws, rows, kh, kvh_pool, b):
    """Mask rows (b, h, i) of one key/value head against the oracle's single-row prediction.

    The library's pooled scores, s_Q and s_K (read from its workspace) are first held to the
    bounds the slack is derived from (mask_checks).  Rows that no rounding within the slack can
    change are compared bit for bit; the others must satisfy what a correct cut satisfies
    (cut_violations).  Returns (rows decisive under the derived slack, rows decisive under the
    absolute 1e-3 margins)."""
    S_v, sQ_v, sK_v = ws
    scale = oracle.default_scale(w.d)
    n_rel = n_abs = 0
    for h, i in rows:
        pr = oracle.predict_mask_row(_block(w.q, b, h, i), kh, i, w.topk, w.theta, w.causal, k_pool=kvh_pool)
        valid = pr["valid"]
        E = score_error_bound(pr["muQ"], kvh_pool[0], pr["S"], valid, scale)
        s_gpu = S_v[(b, h, i)]
        err = np.abs(s_gpu[valid] - pr["S"][valid])
        assert (err <= E[valid]).all(), ("pooled scores outside their bound", (b, h, i), float((err - E[valid]).max()))
        assert abs(sQ_v[(b, h, i)] - pr["sQ"]) <= EPS_SIM, (b, h, i)
        assert np.abs(sK_v[b][valid] - pr["sK"][valid]).max(initial=0.0) <= EPS_SIM, (b, h, i)
        eps_rel, eps_mass = slack(E)
        row = gm[b, h, i]
        if decisive(pr, w.topk, w.theta, eps_rel, eps_mass):
            assert np.array_equal(row, pr["mask"]), ("decisive row differs", (b, h, i))
            n_rel += 1
        else:
            bad = cut_violations(pr, row, w.topk, w.theta, eps_rel, eps_mass)
            assert not bad, ((b, h, i), bad)
        n_abs += oracle.row_decisive(pr["P"], valid, pr["sQ"], pr["sK"], w.topk, w.theta)
    return n_rel, n_abs


# mask rows and attention blocks checked per workload, and the mask rows that must be compared
# bit for bit (decisive under the derived slack)
FULL_SIZE = {"llama128k": (320, 12, 100), "llama32k": (160, 12, 60), "flux": (96, 8, 20),
             "cogvideox": (96, 8, 20), "vit": (96, 8, 20)}


@pytest.mark.parametrize("name", list(FULL_SIZE))
def test_full_size_predicted_mask_and_attention(name):
    n_mask, n_attn, n_dec_min = FULL_SIZE[name]
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
    # the prediction alone, with its workspace kept for the pooled scores and similarities
    ws = torch.empty(fbs.workspace_bytes(fbs.SPARGE_OP_PREDICT_MASK, w.B, w.Hq, w.Hkv, w.N, w.d), dtype=torch.uint8,
                     device="cuda")
    mask2 = fbs.predict_mask(q, k, w.topk, w.theta, w.causal, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(mask, mask2)
    gm = mask.cpu().numpy()
    _check_whole_mask(w, gm)
    muQ, sQ, muK, sK, S = fbs.predict_ws_views(ws, w.B, w.Hq, w.Hkv, w.N, w.d)
    samples = _samples(w, n_mask)
    S_v = {s: S[s].double().cpu().numpy() for s in set(samples)}
    sQ_v = {s: float(sQ[s]) for s in set(samples)}
    sK_h = sK.double().cpu().numpy()
    G = w.Hq // w.Hkv
    n_rel = n_abs = 0
    attn_set = set(samples[:n_attn])
    for b in range(w.B):
        for kvh in range(w.Hkv):
            rows = [(h, i) for (bb, h, i) in samples if bb == b and h // G == kvh]
            if not rows:
                continue
            kh, vh = f64(w.k[b, kvh]), f64(w.v[b, kvh])
            kp = oracle.pool_key_head(kh)
            r, a = _check_mask_rows(w, gm, (S_v, sQ_v, {b: sK_h[b, kvh]}), rows, kh, kp, b)
            n_rel += r
            n_abs += a
            for h, i in rows:
                if (b, h, i) in attn_set:
                    _check_attention(w, gm, out, b, h, i, w.lam, kh, vh)
    print("%s: %d mask rows, %d bit-exact (derived slack), %d decisive at 1e-3" % (name, len(samples), n_rel, n_abs))
    assert n_rel >= n_dec_min, (n_rel, n_dec_min)


@pytest.mark.parametrize("prec,cos_min", [
    (fbs.SPARGE_PRECISION_BF16, COS_MIN), (fbs.SPARGE_PRECISION_Q8, 0.999), (fbs.SPARGE_PRECISION_BF16_FP8PV, 0.999),
    pytest.param(fbs.SPARGE_PRECISION_Q8_FP8PV, 0.999,
                 marks=pytest.mark.xfail(strict=True, reason="e4m3 scores, P and V: measured cosine 0.9986 < 0.999"))])
def test_full_size_custom_mask(prec, cos_min):
    """The custom-mask workload at full size (B 2, 16 heads, N 65536) through the block-sparse
    call on its own mask, in each precision; the 8-bit ones at the cosine bound only."""
    w = _workload("custom")
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    out = fbs.block_sparse_attn_ex(q, k, v, torch.from_numpy(w.mask).cuda(), w.causal, lam=w.lam, precision=prec)
    torch.cuda.synchronize()
    maxabs = MAXABS if prec == fbs.SPARGE_PRECISION_BF16 else math.inf
    for b, h, i in _samples(w, 6):
        _check_attention(w, w.mask, out, b, h, i, w.lam, f64(w.k[b, h]), f64(w.v[b, h]), cos_min=cos_min,
                         maxabs=maxabs)
