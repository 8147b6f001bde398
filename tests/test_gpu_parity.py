"""GPU parity: the CUDA path through the C ABI against the float64 oracle on the same seeded
inputs.  Masks bit-exact on decisive rows; bf16 outputs given the same mask at cosine >= 0.9999
and max-abs error <= 1e-2; pooled statistics at fp32 tolerance; permutations bit-exact."""
import math

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import COS_MIN, MAXABS, cos_maxabs, dev_bf16, f64, host_f64

pytestmark = pytest.mark.gpu

# small members of each workload family: several tiles and a ragged tail where the family has one
SMALL = {
    "tiny": dict(name="tiny"),
    "llama": dict(name="llama32k", N=4096 + 200, Hq=8, Hkv=2),
    "flux": dict(name="flux", Hq=4, Hkv=4),
    "cogvideox": dict(name="cogvideox", Hq=2, Hkv=2, grid=(5, 30, 45)),
    "vit": dict(name="vit", Hq=2, Hkv=2, grid=(32, 32)),
}


def make(key):
    spec = dict(SMALL[key])
    return W.make_config(spec.pop("name"), **spec)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbs.lib()
    assert torch.cuda.is_available()
    yield
    torch.cuda.synchronize()
    assert fbs.device_status() == 0


# ------------------------------------------------------------------------------------------------
# stage 1
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("key", list(SMALL))
def test_pool_sim_matches_oracle(key):
    w = make(key)
    q, k = dev_bf16(w.q), dev_bf16(w.k)
    ws = torch.zeros(fbs.workspace_bytes(fbs.SPARGE_OP_PREDICT_MASK, w.B, w.Hq, w.Hkv, w.N, w.d),
                     dtype=torch.uint8, device="cuda")
    fbs.predict_mask(q, k, w.topk, w.theta, w.causal, ws=ws)
    torch.cuda.synchronize()
    muQ, sQ, muK, sK, S = (t.cpu().numpy().astype(np.float64) for t in fbs.predict_ws_views(ws, w.B, w.Hq, w.Hkv, w.N, w.d))
    rmuQ, rsQ = oracle.pool_sim(f64(w.q), 128)
    rmuK, rsK = oracle.pool_sim(f64(w.k), 64)
    np.testing.assert_allclose(muQ, rmuQ, rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(muK, rmuK, rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(sQ, rsQ, rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(sK, rsK, rtol=1e-5, atol=2e-6)
    # pooled scores on the valid tiles: tensor-core product of bf16 hi/lo splits, ~1e-5 relative
    rS = oracle.pooled_scores(rmuQ, rmuK, w.causal, oracle.default_scale(w.d))
    valid = np.isfinite(rS)
    np.testing.assert_allclose(S[valid], rS[valid], rtol=1e-4, atol=2e-4)


def check_mask(w, gm, topk=None, theta=None):
    topk = w.topk if topk is None else topk
    theta = w.theta if theta is None else theta
    pred = oracle.predict_mask(f64(w.q), f64(w.k), topk, theta, w.causal)
    dec = oracle.decisive_rows(pred, topk, theta, w.causal)
    valid = oracle.block_valid(w.nqb, w.nkb, w.causal)
    assert not gm[:, :, ~valid].any(), "mask keeps tiles above the causal diagonal"
    assert (gm.sum(axis=-1) >= 1).all(), "a row keeps no block"
    assert dec.mean() > 0.2, "too few decisive rows to be a meaningful check"
    bad = np.nonzero((gm != pred["mask"]).any(axis=-1) & dec)
    assert bad[0].size == 0, "mask differs on decisive rows %s" % (list(zip(*bad))[:5],)
    return pred, dec


@pytest.mark.parametrize("key", list(SMALL))
def test_mask_matches_oracle_on_decisive_rows(key):
    w = make(key)
    gm = fbs.predict_mask(dev_bf16(w.q), dev_bf16(w.k), w.topk, w.theta, w.causal).cpu().numpy()
    check_mask(w, gm)


@pytest.mark.parametrize("causal", [False, True])
def test_mask_equal_scores_keep_lowest_indices(causal):
    """Every key block identical, so each row's pooled scores are all equal: the cut falls among
    ties, which the (probability desc, index asc) order resolves to the lowest indices.  300 key
    blocks make rows with up to 32, up to 256 and more than 256 tied candidates (the sort, the
    split-list and the whole-row tie paths)."""
    B, Hq, Hkv, N, d = 1, 2, 1, 300 * 64, 64
    qu, ku, _ = W.random_qkv(26, B, Hq, Hkv, N, d)
    ku = np.broadcast_to(ku[:, :, :1, :], ku.shape).copy()
    topk, theta = 0.331, 0.0      # 0.331 n is never an integer for n <= 300; theta 0 keeps nothing extra
    gm = fbs.predict_mask(dev_bf16(qu), dev_bf16(ku), topk, theta, causal).cpu().numpy()
    pred = oracle.predict_mask(f64(qu), f64(ku), topk, theta, causal)
    assert np.array_equal(gm, pred["mask"])
    nvalid = pred["mask"].shape[-1] if not causal else None
    if nvalid:
        assert (gm.sum(axis=-1) == math.ceil(topk * nvalid)).all()
        assert gm[..., :math.ceil(topk * nvalid)].all()


@pytest.mark.parametrize("key,topk", [("tiny", 0.3), ("llama", 0.5), ("flux", 0.25), ("cogvideox", 0.1)])
def test_count_mode_mask_matches_oracle(key, topk):
    """The count reading of topk (ceil(topk * n_valid) blocks per row): bit-exact on the rows whose
    probability gap at the cut and similarity margins exceed 1e-3."""
    w = make(key)
    q, k = dev_bf16(w.q), dev_bf16(w.k)
    gm = fbs.predict_mask_ex(q, k, topk, w.causal, theta=w.theta, topk_mode=fbs.SPARGE_TOPK_COUNT).cpu().numpy()
    pred = oracle.predict_mask(f64(w.q), f64(w.k), topk, w.theta, w.causal, mode="count")
    dec = oracle.decisive_rows(pred, topk, w.theta, w.causal, mode="count")
    assert dec.mean() > 0.2
    bad = np.nonzero((gm != pred["mask"]).any(axis=-1) & dec)
    assert bad[0].size == 0, "count-mode mask differs on decisive rows %s" % (list(zip(*bad))[:5],)
    # rows that no similarity rule touches keep exactly the count
    valid = oracle.block_valid(w.nqb, w.nkb, w.causal)
    G = w.Hq // w.Hkv
    for b, h, i in zip(*np.nonzero(dec)):
        if pred["sQ"][b, h, i] >= w.theta and (pred["sK"][b, h // G][valid[i]] >= w.theta).all():
            assert gm[b, h, i].sum() == oracle.count_target(topk, int(valid[i].sum()))


@pytest.mark.parametrize("causal", [False, True])
def test_count_mode_equal_scores_keep_lowest_indices(causal):
    """All pooled scores of a row equal: the count reading keeps the lowest indices, through the
    same tie paths as the cumulative reading (up to 300 tied candidates per row), and rows where
    exp underflows are not an issue because every e is 1."""
    B, Hq, Hkv, N, d = 1, 2, 1, 300 * 64, 64
    qu, ku, _ = W.random_qkv(26, B, Hq, Hkv, N, d)
    ku = np.broadcast_to(ku[:, :, :1, :], ku.shape).copy()
    topk, theta = 0.331, 0.0
    gm = fbs.predict_mask_ex(dev_bf16(qu), dev_bf16(ku), topk, causal, theta=theta,
                             topk_mode=fbs.SPARGE_TOPK_COUNT).cpu().numpy()
    pred = oracle.predict_mask(f64(qu), f64(ku), topk, theta, causal, mode="count")
    assert np.array_equal(gm, pred["mask"])


def test_count_mode_through_sparge_attn_ex():
    """sparge_attn_ex with the count reading: its mask is predict_mask_ex's, its output the
    oracle's attention on that mask."""
    w = make("llama")
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, 0.4, w.causal, theta=w.theta, mask_out=mask, topk_mode=fbs.SPARGE_TOPK_COUNT)
    m2 = fbs.predict_mask_ex(q, k, 0.4, w.causal, theta=w.theta, topk_mode=fbs.SPARGE_TOPK_COUNT)
    assert torch.equal(mask, m2)
    ref = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), mask.cpu().numpy(), -math.inf, w.causal)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


@pytest.mark.parametrize("key,topk,topp", [("tiny", 0.1, 0.3), ("tiny", 0.2, 0.5), ("llama", 0.15, 0.4),
                                           ("llama", 0.12, 0.45)])
def test_hybrid_mode_mask_matches_oracle(key, topk, topp):
    """The hybrid reading (blocks kept by the count reading with topk or by the cumulative reading
    with topp): bit-exact on the rows where both cuts are decisive, and on every row at least
    the blocks each reading keeps alone."""
    w = make(key)
    q, k = dev_bf16(w.q), dev_bf16(w.k)
    gm = fbs.predict_mask_ex(q, k, topk, w.causal, theta=w.theta, topk_mode=fbs.SPARGE_TOPK_HYBRID,
                             topp=topp).cpu().numpy()
    pred = oracle.predict_mask(f64(w.q), f64(w.k), topk, w.theta, w.causal, mode="hybrid", topp=topp)
    dec = oracle.decisive_rows(pred, topk, w.theta, w.causal, mode="hybrid", topp=topp)
    assert dec.mean() > 0.2
    bad = np.nonzero((gm != pred["mask"]).any(axis=-1) & dec)
    assert bad[0].size == 0, "hybrid mask differs on decisive rows %s" % (list(zip(*bad))[:5],)
    # the GPU's own count-mode and cumulative-mode masks are subsets of its hybrid mask, and
    # together they make it up
    gc = fbs.predict_mask_ex(q, k, topk, w.causal, theta=w.theta, topk_mode=fbs.SPARGE_TOPK_COUNT).cpu().numpy()
    gp = fbs.predict_mask_ex(q, k, topp, w.causal, theta=w.theta).cpu().numpy()
    assert np.array_equal(gm, gc | gp)
    # both readings decide some rows (the union is not just one of them)
    assert (gm != gc).any() and (gm != gp).any()


def test_hybrid_mode_through_sparge_attn_ex():
    """sparge_attn_ex with the hybrid reading: its mask is predict_mask_ex's, its output the
    oracle's attention on that mask."""
    w = make("llama")
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, 0.1, w.causal, theta=w.theta, mask_out=mask, topk_mode=fbs.SPARGE_TOPK_HYBRID,
                             topp=0.4)
    m2 = fbs.predict_mask_ex(q, k, 0.1, w.causal, theta=w.theta, topk_mode=fbs.SPARGE_TOPK_HYBRID, topp=0.4)
    assert torch.equal(mask, m2)
    ref = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), mask.cpu().numpy(), -math.inf, w.causal)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


@pytest.mark.parametrize("topk,theta", [(0.05, 0.5), (0.3, 0.3), (0.9, 0.0), (1.0, 0.5), (0.5, 2.0)])
def test_mask_topk_theta_sweep(topk, theta):
    w = make("llama")
    gm = fbs.predict_mask(dev_bf16(w.q), dev_bf16(w.k), topk, theta, w.causal).cpu().numpy()
    check_mask(w, gm, topk, theta)
    if topk >= 1.0 or theta > 1.0:
        assert (gm == oracle.block_valid(w.nqb, w.nkb, True)[None, None]).all()


# ------------------------------------------------------------------------------------------------
# stage 2
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,Hq,Hkv", [(128, 1, 1), (1000, 4, 1), (777, 2, 2)])
def test_dense_attention_all_ones(causal, d, N, Hq, Hkv):
    qu, ku, vu = W.random_qkv(21, 1, Hq, Hkv, N, d)
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, causal)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, causal)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_random_mask_attention(causal, d):
    N, Hq, Hkv = 1500, 4, 2
    qu, ku, vu = W.random_qkv(22, 2, Hq, Hkv, N, d)
    mask = W.random_mask(23, 2, Hq, N, p=0.3, force_diag=False)
    mask[0, 0, 3] = 0                               # an empty row: output 0
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), torch.from_numpy(mask).cuda(),
                                -math.inf, causal)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), mask, -math.inf, causal)
    got = host_f64(out)
    cos, err = cos_maxabs(got, ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    assert (got[0, 0, 3 * 128:4 * 128] == 0).all()


@pytest.mark.parametrize("lam", [-12.0, -8.0, -4.0])
def test_lambda_filter_matches_oracle(lam):
    w = make("llama")
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    stats = torch.zeros(4, dtype=torch.int64, device="cuda")
    out = fbs.block_sparse_attn(q, k, v, None, lam, True, stats=stats)
    ref, st = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), None, lam, True, return_stats=True)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    s = stats.cpu().numpy()
    assert s[0] == st["kept_tiles"]
    assert abs(int(s[2]) - st["skipped_group_tiles"]) <= max(2, st["skipped_group_tiles"] // 1000)
    assert abs(int(s[1]) - st["pv_tiles"]) <= max(2, st["pv_tiles"] // 1000)
    if lam >= -8.0:
        assert s[2] > 0


def test_strided_inputs():
    """Q/K/V as views into one packed (B, N, 3, H, d) buffer: head and token strides differ
    from the contiguous ones."""
    B, N, H, d = 1, 700, 2, 64
    qu, ku, vu = W.random_qkv(24, B, H, H, N, d)
    packed = torch.empty((B, N, 3, H, d), dtype=torch.bfloat16, device="cuda")
    for s, u in enumerate((qu, ku, vu)):
        packed[:, :, s] = dev_bf16(u).transpose(1, 2)
    q, k, v = (packed[:, :, s].transpose(1, 2) for s in range(3))
    assert q.stride(2) == 3 * H * d
    out_full = torch.zeros((B, H, N, 2 * d), dtype=torch.bfloat16, device="cuda")
    out = out_full[..., :d]
    fbs.block_sparse_attn(q, k, v, None, -math.inf, False, out=out)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, False)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    assert (out_full[..., d:] == 0).all()


# ------------------------------------------------------------------------------------------------
# the whole path
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("key", ["tiny", "llama"])
def test_sparge_attn_end_to_end(key):
    w = make(key)
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    lam = w.lam if key == "llama" else -math.inf
    out = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, lam=lam, mask_out=mask)
    gm = mask.cpu().numpy()
    check_mask(w, gm)
    ref = oracle.block_sparse_attn(f64(w.q), f64(w.k), f64(w.v), gm, lam, w.causal)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    # the plug-and-play call is the same computation with theta 0.5, lambda -inf
    out2 = fbs.sparge_attn(q, k, v, w.topk, w.causal)
    if w.theta == 0.5 and lam == -math.inf:
        assert torch.equal(out, out2)


@pytest.mark.parametrize("key", ["flux", "cogvideox", "vit"])
def test_hilbert_pipeline(key):
    w = make(key)
    perm_np = (fbs.hilbert_perm_2d(w.n_prefix, *w.grid) if len(w.grid) == 2
               else fbs.hilbert_perm_3d(w.n_prefix, *w.grid))
    perm = torch.from_numpy(perm_np).cuda()
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    pq, pk, pv = (fbs.permute_tokens(t, perm) for t in (q, k, v))
    for dev_t, host_t in ((pq, w.q), (pk, w.k), (pv, w.v)):
        assert np.array_equal(dev_t.cpu().view(torch.int16).numpy().view(np.uint16), host_t[:, :, perm_np])
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    po = fbs.sparge_attn_ex(pq, pk, pv, w.topk, w.causal, theta=w.theta, mask_out=mask)
    out = fbs.unpermute_tokens(po, perm)
    assert torch.equal(fbs.permute_tokens(out, perm), po)
    gm = mask.cpu().numpy()
    wp = W.Workload(**{**w.__dict__})
    wp.q, wp.k, wp.v = w.q[:, :, perm_np], w.k[:, :, perm_np], w.v[:, :, perm_np]
    check_mask(wp, gm)
    ref = oracle.unpermute_tokens(
        oracle.block_sparse_attn(f64(wp.q), f64(wp.k), f64(wp.v), gm, -math.inf, w.causal), perm_np)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


@pytest.mark.parametrize("d,N", [(64, 1000), (128, 777), (128, 4096 + 33)])
def test_permute_strided_ragged(d, N):
    """Gather and scatter bit-exact against numpy on strided views (token stride 2d, heads
    interleaved) with N not a multiple of the kernel's row chunk."""
    rng = np.random.Generator(np.random.PCG64(N + d))
    B, H = 2, 3
    perm_np = rng.permutation(N).astype(np.int32)
    perm = torch.from_numpy(perm_np).cuda()
    base = torch.randn((B, N, H, 2 * d), generator=torch.Generator().manual_seed(N), dtype=torch.float32)
    x = base.to(torch.bfloat16).cuda().permute(0, 2, 1, 3)[..., :d]     # (B, H, N, d), stride_n = 2 H d
    yb = torch.zeros((B, H, N, 2 * d), dtype=torch.bfloat16, device="cuda")
    y = yb[..., d:]                                                     # stride_n = 2 d, offset d
    fbs.permute_tokens(x, perm, out=y)
    xn = x.float().cpu().numpy()
    np.testing.assert_array_equal(y.float().cpu().numpy(), xn[:, :, perm_np])
    assert not yb[..., :d].any()                                        # nothing written outside y
    z = torch.empty_like(x)
    fbs.unpermute_tokens(y, perm, out=z)
    np.testing.assert_array_equal(z.float().cpu().numpy(), xn)
    assert fbs.device_status() == fbs.SPARGE_OK


def test_permute_skips_entries_out_of_range():
    """Entries outside 0..N-1 are never used as addresses: their rows are left as they were and
    the device status word reports SPARGE_ERR_INVALID_ARG once; the next valid call is clean."""
    N, d = 300, 64
    rng = np.random.Generator(np.random.PCG64(5))
    perm_np = rng.permutation(N).astype(np.int32)
    bad = [3, 150, 299]
    perm_np[bad[0]], perm_np[bad[1]], perm_np[bad[2]] = -1, N, 1 << 30
    perm = torch.from_numpy(perm_np).cuda()
    x = torch.randn((1, 2, N, d), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    sentinel = torch.full_like(x, 7.0)
    y = sentinel.clone()
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_OK
    fbs.permute_tokens(x, perm, out=y)
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_ERR_INVALID_ARG
    assert b"permutation entry" in fbs.lib().sparge_last_error()
    assert fbs.device_status() == fbs.SPARGE_OK                 # reading clears the word
    good = np.setdiff1d(np.arange(N), bad)
    xn, yn = x.float().cpu().numpy(), y.float().cpu().numpy()
    np.testing.assert_array_equal(yn[:, :, good], xn[:, :, perm_np[good]])
    assert (yn[:, :, bad] == 7.0).all()
    z = sentinel.clone()
    fbs.unpermute_tokens(x, perm, out=z)
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_ERR_INVALID_ARG
    zn = z.float().cpu().numpy()
    np.testing.assert_array_equal(zn[:, :, perm_np[good]], xn[:, :, good])
    untouched = np.setdiff1d(np.arange(N), perm_np[good])
    assert (zn[:, :, untouched] == 7.0).all()
    fbs.permute_tokens(x, torch.arange(N, dtype=torch.int32, device="cuda"), out=y)
    assert torch.equal(y, x) and fbs.device_status() == fbs.SPARGE_OK


def test_empty_and_degenerate_shapes():
    for N in (1, 63, 64, 65, 127, 129):
        qu, ku, vu = W.random_qkv(25, 1, 2, 1, N, 128)
        q, k, v = dev_bf16(qu), dev_bf16(ku), dev_bf16(vu)
        out = fbs.sparge_attn(q, k, v, 0.5, True)
        mask = fbs.predict_mask(q, k, 0.5, 0.5, True)
        ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), mask.cpu().numpy(), -math.inf, True)
        cos, err = cos_maxabs(host_f64(out), ref)
        assert cos >= COS_MIN and err <= MAXABS, (N, cos, err)
    z = torch.zeros((0, 2, 128, 64), dtype=torch.bfloat16, device="cuda")
    fbs.sparge_attn(z, z, z, 0.5, False)
    torch.cuda.synchronize()


def test_block_sparse_ex_matches_and_times():
    """The _ex call with scale 0 is the plain call (bit-identical); an explicit scale is the
    oracle's scale; its six events bracket the V copy and the attention kernel."""
    N, Hq, Hkv, d = 900, 2, 1, 128
    qu, ku, vu = W.random_qkv(27, 1, Hq, Hkv, N, d)
    q, k, v = dev_bf16(qu), dev_bf16(ku), dev_bf16(vu)
    base = fbs.block_sparse_attn(q, k, v, None, -math.inf, True)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    ex = fbs.block_sparse_attn_ex(q, k, v, None, True, events=evs)
    torch.cuda.synchronize()
    assert torch.equal(base, ex)
    assert evs[0].elapsed_time(evs[4]) >= 0 and evs[4].elapsed_time(evs[5]) > 0
    out = fbs.block_sparse_attn_ex(q, k, v, None, True, scale=0.05)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, True, scale=0.05)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)


def test_cuda_graph_capture_and_replay():
    """The whole path (prediction and attention, 5 launches) captured once in a CUDA graph and
    replayed on new inputs copied into the captured buffers matches eager calls bit for bit."""
    w = make("llama")
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(fbs.workspace_bytes(fbs.SPARGE_OP_ATTN, w.B, w.Hq, w.Hkv, w.N, w.d), dtype=torch.uint8,
                     device="cuda")
    call = lambda: fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, lam=w.lam, mask_out=mask, out=out,
                                      ws=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()                      # first call on this shape sets kernel attributes, outside capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    # replay on the first inputs, then on perturbed ones
    for scale in (1.0, 0.5):
        qs = (dev_bf16(w.q).float() * scale).to(torch.bfloat16)
        q.copy_(qs)
        g.replay()
        torch.cuda.synchronize()
        got_o, got_m = out.clone(), mask.clone()
        ref_o = fbs.sparge_attn_ex(qs, k, v, w.topk, w.causal, theta=w.theta, lam=w.lam,
                                   mask_out=(ref_m := torch.empty_like(mask)))
        torch.cuda.synchronize()
        assert torch.equal(got_m, ref_m)
        assert torch.equal(got_o, ref_o)
