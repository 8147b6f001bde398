"""Pins of the float64 oracle against things other than itself: closed forms, brute-force
enumeration, a library attention routine, invariants and an independent construction of
the Hilbert curve.  CPU only."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def f64(u16):
    return W.bf16_to_f64(u16)


def sdpa_f64(q, k, v, causal):
    """torch's scaled_dot_product_attention in float64 on the CPU (GQA by repeating K/V)."""
    G = q.shape[1] // k.shape[1]
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(np.repeat(k, G, axis=1))
    tv = torch.from_numpy(np.repeat(v, G, axis=1))
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal).numpy()


# ----------------------------------------------------------------------------------------------
# pooling and self-similarity
# ----------------------------------------------------------------------------------------------
def pairwise_cosine_mean(xb):
    """Definition: the mean over all ordered pairs (a, b), a == b included, of cos(x_a, x_b)."""
    n = xb.shape[0]
    tot = 0.0
    for a in range(n):
        for b in range(n):
            na, nb = np.linalg.norm(xb[a]), np.linalg.norm(xb[b])
            tot += 0.0 if na == 0 or nb == 0 else float(xb[a] @ xb[b]) / (na * nb)
    return tot / (n * n)


def test_pool_sim_matches_pairwise_definition():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((1, 2, 200, 16)) + rng.standard_normal((1, 2, 1, 16))
    x[0, 1, 130] = 0.0  # a zero-norm token inside the tail block
    mu, s = oracle.pool_sim(x, 128)
    assert mu.shape == (1, 2, 2, 16) and s.shape == (1, 2, 2)
    for h in range(2):
        for i, (a, b) in enumerate([(0, 128), (128, 200)]):
            np.testing.assert_allclose(mu[0, h, i], x[0, h, a:b].mean(axis=0), rtol=1e-12, atol=1e-12)
            assert s[0, h, i] == pytest.approx(pairwise_cosine_mean(x[0, h, a:b]), abs=1e-12)


def test_pool_sim_special_cases():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(32)
    same = np.tile(v * 3.0, (64, 1))[None, None]
    _, s = oracle.pool_sim(same * rng.uniform(0.5, 2.0, (1, 1, 64, 1)), 64)
    assert s[0, 0, 0] == pytest.approx(1.0, abs=1e-12)      # every token points the same way
    anti = np.concatenate([np.tile(v, (32, 1)), np.tile(-2.0 * v, (32, 1))])[None, None]
    _, s = oracle.pool_sim(anti, 64)
    assert s[0, 0, 0] == pytest.approx(0.0, abs=1e-12)      # antipodal halves cancel
    orth = np.eye(64)[None, None]
    _, s = oracle.pool_sim(orth, 64)
    assert s[0, 0, 0] == pytest.approx(1.0 / 64, abs=1e-12)  # orthogonal tokens: only the diagonal


# ----------------------------------------------------------------------------------------------
# attention against a library routine
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,Hq,Hkv,d", [(1024, 2, 2, 64), (333, 4, 1, 32), (260, 2, 2, 128)])
def test_topk_one_equals_dense(causal, N, Hq, Hkv, d):
    q, k, v = (f64(t) for t in W.random_qkv(3, 1, Hq, Hkv, N, d))
    ref = sdpa_f64(q, k, v, causal)
    out = oracle.sparge_attn(q, k, v, topk=1.0, causal=causal, theta=0.5, lam=-math.inf)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------------------------
# short queries (Nq < Nk): the last query sits on the last key
# ----------------------------------------------------------------------------------------------
def sdpa_f64_offset(q, k, v, causal):
    """float64 SDPA with an explicit boolean mask: query r sees key c when c <= (Nk - Nq) + r."""
    G = q.shape[1] // k.shape[1]
    Nq, Nk = q.shape[2], k.shape[2]
    tq, tk = torch.from_numpy(q), torch.from_numpy(np.repeat(k, G, axis=1))
    tv = torch.from_numpy(np.repeat(v, G, axis=1))
    m = None
    if causal:
        m = torch.from_numpy(np.arange(Nk)[None, :] <= (Nk - Nq) + np.arange(Nq)[:, None])
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m).numpy()


@pytest.mark.parametrize("Nq,Nk", [(128, 1024), (300, 700), (1, 513), (700, 700)])
def test_block_valid_with_offset_brute_force(Nq, Nk):
    nqb, nkb, off = -(-Nq // 128), -(-Nk // 64), Nk - Nq
    got = oracle.block_valid(nqb, nkb, True, off)
    for i in range(nqb):
        for j in range(nkb):
            rows = np.arange(128 * i, min(Nq, 128 * i + 128))
            cols = np.arange(64 * j, min(Nk, 64 * j + 64))
            vis = (cols[None, :] <= off + rows[:, None]).any()
            assert got[i, j] == vis, (i, j)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk,Hq,Hkv,d", [(256, 1024, 2, 1, 64), (130, 700, 2, 2, 32), (1, 300, 1, 1, 64)])
def test_short_query_dense_equals_sdpa(causal, Nq, Nk, Hq, Hkv, d):
    rng = np.random.Generator(np.random.PCG64(Nq + Nk))
    q = f64(W.bf16_bits(rng.standard_normal((1, Hq, Nq, d)).astype(np.float32)))
    _, k, v = (f64(t) for t in W.random_qkv(5, 1, Hq, Hkv, Nk, d))
    ref = sdpa_f64_offset(q, k, v, causal)
    out = oracle.sparge_attn(q, k, v, topk=1.0, causal=causal, theta=0.5, lam=-math.inf)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    if causal:   # and it is the tail of the full causal attention over a sequence ending in q
        qf = np.concatenate([f64(W.random_qkv(6, 1, Hq, Hkv, Nk - Nq, d)[0]), q], axis=2) if Nk > Nq else q
        full = oracle.block_sparse_attn(qf, k, v, None, -math.inf, True)
        np.testing.assert_allclose(out, full[:, :, Nk - Nq:], rtol=1e-10, atol=1e-12)


def test_short_query_mask_brute_force():
    rng = np.random.Generator(np.random.PCG64(11))
    Nq, Nk, d = 384, 1280, 32
    q = rng.standard_normal((1, 1, 1, d)) + 0.3 * rng.standard_normal((1, 1, Nq, d))
    k = rng.standard_normal((1, 1, 20, d)).repeat(64, axis=2) + 0.3 * rng.standard_normal((1, 1, Nk, d))
    for causal in (False, True):
        pred = oracle.predict_mask(q, k, topk=0.6, theta=0.0, causal=causal)
        valid = oracle.block_valid(3, 20, causal, Nk - Nq)
        for i in range(3):
            keep = brute_force_keep(pred["P"][0, 0, i], valid[i], 0.6)
            np.testing.assert_array_equal(pred["mask"][0, 0, i].astype(bool), keep)
            assert not pred["mask"][0, 0, i][~valid[i]].any()


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_equals_dense(causal):
    q, k, v = (f64(t) for t in W.random_qkv(4, 2, 4, 2, 700, 64))
    ref = sdpa_f64(q, k, v, causal)
    nqb, nkb = oracle.n_blocks(700, 128), oracle.n_blocks(700, 64)
    ones = np.ones((2, 4, nqb, nkb), np.uint8)
    np.testing.assert_allclose(oracle.block_sparse_attn(q, k, v, ones, -math.inf, causal), ref,
                               rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(oracle.block_sparse_attn(q, k, v, None, -math.inf, causal), ref,
                               rtol=1e-10, atol=1e-12)


def test_masked_attention_equals_library_with_token_mask():
    """Block-sparse attention = SDPA with the block mask expanded to a token mask."""
    N, d = 300, 32
    q, k, v = (f64(t) for t in W.random_qkv(5, 1, 2, 2, N, d))
    mask = W.random_mask(6, 1, 2, N, p=0.5)
    out = oracle.block_sparse_attn(q, k, v, mask, -math.inf, causal=True)
    tok = np.repeat(np.repeat(mask.astype(bool), 128, axis=2), 64, axis=3)[:, :, :N, :N]
    tok &= np.tril(np.ones((N, N), bool))[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(tok)).numpy()
    empty = ~tok.any(axis=-1)
    ref[empty] = 0.0  # a row with no visible kept key outputs 0 (the library gives NaN there)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------------------------
# mask against brute force
# ----------------------------------------------------------------------------------------------
def brute_force_keep(p, valid, topk):
    """Over all subsets of the valid blocks: the fewest blocks whose probabilities sum to at
    least topk; among those the largest sum; among those the lexicographically smallest list of
    indices."""
    vj = np.nonzero(valid)[0]
    n = vj.size
    subsets = np.array(list(itertools.product([0, 1], repeat=n)), dtype=bool)
    sums = subsets.astype(np.float64) @ p[vj]
    card = subsets.sum(axis=1)
    ok = sums >= topk
    if not ok.any():
        best = np.ones(n, bool)
    else:
        cmin = card[ok].min()
        cand = ok & (card == cmin)
        smax = sums[cand].max()
        cand &= sums == smax
        idx = sorted(tuple(vj[s]) for s in subsets[cand])
        best = np.isin(vj, idx[0])
    keep = np.zeros(p.size, bool)
    keep[vj[best]] = True
    return keep


@pytest.mark.parametrize("theta,min_cut_rows", [(0.5, 5), (0.3, 16)])
def test_mask_matches_brute_force_tiny(theta, min_cut_rows):
    w = W.make_config("tiny")
    w.theta = theta
    q, k = f64(w.q), f64(w.k)
    pred = oracle.predict_mask(q, k, w.topk, w.theta, w.causal)
    # independent route to the probabilities: block means, einsum, scipy softmax
    from scipy.special import softmax
    d = q.shape[-1]
    mq = q.reshape(1, 2, 8, 128, d).mean(axis=3)
    mk = k.reshape(1, 2, 16, 64, d).mean(axis=3)
    P = softmax(np.einsum("bhid,bhjd->bhij", mq, mk) / math.sqrt(d), axis=-1)
    sq = np.array([[[pairwise_cosine_mean(q[0, h, 128 * i:128 * i + 128]) for i in range(8)] for h in range(2)]])
    sk = np.array([[[pairwise_cosine_mean(k[0, h, 64 * j:64 * j + 64]) for j in range(16)] for h in range(2)]])
    valid = np.ones(16, bool)
    nonfull = 0
    for h in range(2):
        for i in range(8):
            keep = brute_force_keep(P[0, h, i], valid, w.topk)
            if sq[0, h, i] < w.theta:
                keep[:] = True
            keep |= sk[0, h] < w.theta
            nonfull += int(not keep.all())
            np.testing.assert_array_equal(pred["mask"][0, h, i].astype(bool), keep)
    assert nonfull >= min_cut_rows   # the workload really exercises the top-k cut


def test_mask_brute_force_causal_with_ties():
    """Causal validity and the index tie-break, on pooled keys with exact duplicates."""
    rng = np.random.default_rng(7)
    N, d = 640, 16
    q = rng.standard_normal((1, 1, N, d)) * 0.2 + rng.standard_normal((1, 1, 1, d))
    kb = rng.standard_normal((1, 1, 10, d))
    kb[0, 0, 5] = kb[0, 0, 2]           # key blocks with identical means and similarity
    kb[0, 0, 7] = kb[0, 0, 2]
    k = np.repeat(kb, 64, axis=2) + 0.0
    pred = oracle.predict_mask(q, k, topk=0.6, theta=0.0, causal=True)
    P = pred["P"]
    valid = oracle.block_valid(5, 10, True)
    for i in range(5):
        keep = brute_force_keep(P[0, 0, i], valid[i], 0.6)
        np.testing.assert_array_equal(pred["mask"][0, 0, i].astype(bool), keep)
        assert not pred["mask"][0, 0, i][~valid[i]].any()


# ----------------------------------------------------------------------------------------------
# the count reading of topk: keep ceil(topk * n_valid) blocks
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("topk,n,k", [(0.3, 10, 3), (0.5, 16, 8), (0.3, 16, 5), (0.25, 8, 2), (1e-9, 100, 1),
                                      (1.0, 7, 7), (0.999, 7, 7), (0.5, 7, 4), (0.1, 2048, 205)])
def test_count_target_values(topk, n, k):
    assert oracle.count_target(topk, n) == k


def brute_force_count_keep(p, valid, kc):
    """Over all subsets of kc valid blocks: the largest probability sum; among those the
    lexicographically smallest list of indices."""
    vj = np.nonzero(valid)[0]
    best, best_sum = None, -1.0
    for sub in itertools.combinations(range(vj.size), kc):
        ssum = float(p[vj[list(sub)]].sum())
        if ssum > best_sum:
            best, best_sum = sub, ssum
    keep = np.zeros(p.size, bool)
    keep[vj[list(best)]] = True
    return keep


def test_count_mode_matches_brute_force_tiny():
    w = W.make_config("tiny")
    q, k = f64(w.q), f64(w.k)
    topk = 0.3                                     # 5 of the 16 key blocks of every row
    pred = oracle.predict_mask(q, k, topk, 0.0, w.causal, mode="count")   # theta 0: no always-keep
    from scipy.special import softmax
    d = q.shape[-1]
    mq = q.reshape(1, 2, 8, 128, d).mean(axis=3)
    mk = k.reshape(1, 2, 16, 64, d).mean(axis=3)
    P = softmax(np.einsum("bhid,bhjd->bhij", mq, mk) / math.sqrt(d), axis=-1)
    valid = np.ones(16, bool)
    for h in range(2):
        for i in range(8):
            keep = brute_force_count_keep(P[0, h, i], valid, 5)
            np.testing.assert_array_equal(pred["mask"][0, h, i].astype(bool), keep)
    assert (pred["mask"].sum(axis=-1) == 5).all()


def brute_force_hybrid_keep(p, valid, kc, topp):
    """Over all subsets of the valid blocks with at least kc blocks and a probability sum of at
    least topp: the fewest blocks; among those the largest sum; among those the lexicographically
    smallest list of indices."""
    vj = np.nonzero(valid)[0]
    n = vj.size
    subsets = np.array(list(itertools.product([0, 1], repeat=n)), dtype=bool)
    sums = subsets.astype(np.float64) @ p[vj]
    card = subsets.sum(axis=1)
    ok = (sums >= topp) & (card >= kc)
    cmin = card[ok].min()
    cand = ok & (card == cmin)
    cand &= sums == sums[cand].max()
    idx = sorted(tuple(vj[s]) for s in subsets[cand])
    keep = np.zeros(p.size, bool)
    keep[np.array(idx[0], dtype=int)] = True
    return keep


@pytest.mark.parametrize("topk,topp", [(0.2, 0.5), (0.35, 0.7), (0.1, 0.3)])
def test_hybrid_mode_matches_brute_force_tiny(topk, topp):
    """The hybrid reading (count topk or cumulative topp) against subset enumeration of its
    defining property, on every row of the tiny workload; both the count side and the mass side
    decide some rows."""
    w = W.make_config("tiny")
    q, k = f64(w.q), f64(w.k)
    pred = oracle.predict_mask(q, k, topk, 0.0, w.causal, mode="hybrid", topp=topp)
    from scipy.special import softmax
    d = q.shape[-1]
    mq = q.reshape(1, 2, 8, 128, d).mean(axis=3)
    mk = k.reshape(1, 2, 16, 64, d).mean(axis=3)
    P = softmax(np.einsum("bhid,bhjd->bhij", mq, mk) / math.sqrt(d), axis=-1)
    valid = np.ones(16, bool)
    kc = oracle.count_target(topk, 16)
    sides = set()
    for h in range(2):
        for i in range(8):
            keep = brute_force_hybrid_keep(P[0, h, i], valid, kc, topp)
            np.testing.assert_array_equal(pred["mask"][0, h, i].astype(bool), keep)
            by_mass = brute_force_keep(P[0, h, i], valid, topp).sum()
            sides.add("count" if kc > by_mass else "mass" if by_mass > kc else "tie")
    assert {"count", "mass"} <= sides, sides


def test_count_mode_ties_keep_lowest_indices_and_is_monotone():
    p = np.full(12, 1.0 / 12)
    valid = np.ones(12, bool)
    keep = oracle.topk_select(p, valid, 0.25, mode="count")
    np.testing.assert_array_equal(np.nonzero(keep)[0], [0, 1, 2])
    w = W.make_config("tiny")
    q, k = f64(w.q), f64(w.k)
    prev = None
    for t in (0.05, 0.2, 0.5, 0.8, 1.0):
        m = oracle.predict_mask(q, k, t, 0.0, False, mode="count")["mask"]
        assert (m.sum(axis=-1) == oracle.count_target(t, 16)).all()
        if prev is not None:
            assert np.all(m >= prev)
        prev = m


def test_topk_one_keeps_all_valid_and_monotone():
    w = W.make_config("tiny")
    q, k = f64(w.q), f64(w.k)
    prev = None
    for t in (0.05, 0.2, 0.5, 0.8, 0.95, 1.0):
        m = oracle.predict_mask(q, k, t, 0.0, False)["mask"]
        if prev is not None:
            assert np.all(m >= prev)
        prev = m
    assert prev.all()
    assert oracle.predict_mask(q, k, 1e-9, 0.0, False)["mask"].sum(axis=-1).min() == 1


def test_mask_invariant_to_constant_shift_of_keys():
    """Adding one vector to every key adds a per-row constant to the pooled scores, which the
    softmax ignores (theta = 0 switches the similarity rule off, since s >= 0)."""
    w = W.make_config("tiny")
    q, k = f64(w.q), f64(w.k)
    c = np.random.default_rng(8).standard_normal(q.shape[-1])
    m0 = oracle.predict_mask(q, k, 0.5, 0.0, False)
    m1 = oracle.predict_mask(q, k + c, 0.5, 0.0, False)
    dec = oracle.decisive_rows(m0, 0.5, 0.0, False) & oracle.decisive_rows(m1, 0.5, 0.0, False)
    assert dec.sum() > 8
    np.testing.assert_array_equal(m0["mask"][dec], m1["mask"][dec])


@pytest.mark.parametrize("causal,lam", [(False, -math.inf), (True, -math.inf), (True, -8.0)])
def test_output_invariant_to_key_mean_smoothing(causal, lam):
    """Subtracting the token mean of K (per batch and key/value head) shifts every score of a row
    by the same q . mean, which the softmax and the lambda filter (differences of maxima) ignore:
    the attention output is unchanged in float64 (the smoothing the 8-bit path applies)."""
    qu, ku, vu = W.random_qkv(12, 1, 4, 2, 700, 32)
    q, k, v = f64(qu), f64(ku) + 3.0, f64(vu)
    mask = W.random_mask(13, 1, 4, 700, p=0.5)
    ks = k - k.mean(axis=2, keepdims=True)
    o0 = oracle.block_sparse_attn(q, k, v, mask, lam, causal)
    o1 = oracle.block_sparse_attn(q, ks, v, mask, lam, causal)
    np.testing.assert_allclose(o1, o0, rtol=1e-9, atol=1e-11)


def test_always_keep_rows_and_columns():
    rng = np.random.default_rng(9)
    N, d = 512, 32
    base = rng.standard_normal((1, 2, 1, d))
    q = np.repeat(base, N, axis=2) + 0.05 * rng.standard_normal((1, 2, N, d))
    k = np.repeat(rng.standard_normal((1, 1, 1, d)), N, axis=2) + 0.05 * rng.standard_normal((1, 1, N, d))
    q[0, 1, 128:256] = rng.standard_normal((128, d))   # head 1, query block 1 not self-similar
    k[0, 0, 192:256] = rng.standard_normal((64, d))    # key block 3 not self-similar
    pred = oracle.predict_mask(q, k, 0.01, 0.5, causal=True)
    m = pred["mask"]
    valid = oracle.block_valid(4, 8, True)
    assert pred["sQ"][0, 1, 1] < 0.5 and pred["sK"][0, 0, 3] < 0.5
    np.testing.assert_array_equal(m[0, 1, 1].astype(bool), valid[1])
    for h in range(2):                      # column 3 kept in every valid row of both heads
        np.testing.assert_array_equal(m[0, h, :, 3].astype(bool), valid[:, 3])
    assert m[0, 0, 0].sum() == 1             # a similar row keeps only its top block otherwise


# ----------------------------------------------------------------------------------------------
# the lambda filter
# ----------------------------------------------------------------------------------------------
def test_lambda_minus_inf_never_skips_visible_rows():
    q, k, v = (f64(t) for t in W.random_qkv(10, 1, 2, 2, 512, 64))
    _, st = oracle.block_sparse_attn(q, k, v, None, -math.inf, False, return_stats=True)
    assert st["skipped_group_tiles"] == 0
    assert st["pv_tiles"] == st["kept_tiles"] == 2 * 4 * 8


def test_lambda_skip_keeps_row_sum():
    """Hand case: tile 0 holds a key far above every key of tile 1, so with lambda = -4 every
    group skips tile 1; the output is tile 0's weighted values over the sum of both tiles."""
    d = 16
    rng = np.random.default_rng(11)
    q = np.zeros((1, 1, 128, d)); q[..., 0] = 1.0
    k = np.zeros((1, 1, 128, d)); v = rng.standard_normal((1, 1, 128, d))
    k[0, 0, 0, 0] = 40.0                  # score 40/4 = 10 in tile 0
    k[0, 0, 64:, 0] = rng.uniform(-4.0, 20.0, 64)   # tile 1 scores in [-1, 5], all < 10 - 4
    out, st = oracle.block_sparse_attn(q, k, v, None, -4.0, False, return_stats=True)
    assert st["skipped_group_tiles"] == 4 and st["pv_tiles"] == 1
    s = k[0, 0, :, 0] / 4.0
    p = np.exp(s - s.max())
    expect = (p[:64] @ v[0, 0, :64]) / p.sum()
    np.testing.assert_allclose(out[0, 0], np.tile(expect, (128, 1)), rtol=1e-12)
    ref = oracle.block_sparse_attn(q, k, v, None, -math.inf, False)
    np.testing.assert_allclose(ref[0, 0], np.tile((p @ v[0, 0]) / p.sum(), (128, 1)), rtol=1e-12)


@pytest.mark.parametrize("lam", [-12.0, -8.0, -4.0, -2.0])
def test_lambda_error_bound(lam):
    """Each skipped tile drops P.V terms with every P below e^lambda (relative to the running
    max), so |O_lambda - O| <= kept_tiles * 64 * e^lambda * max|v| per row."""
    w = W.make_config("llama32k", N=2048, Hq=4, Hkv=1)
    q, k, v = f64(w.q), f64(w.k), f64(w.v)
    ref = oracle.block_sparse_attn(q, k, v, None, -math.inf, True)
    out, st = oracle.block_sparse_attn(q, k, v, None, lam, True, return_stats=True)
    kept_per_row = np.minimum(2 * (np.arange(2048) // 128) + 2, 32)
    bound = kept_per_row[None, None, :, None] * 64 * math.exp(lam) * np.abs(v).max()
    assert np.all(np.abs(out - ref) <= bound)
    if lam >= -8.0:
        assert st["skipped_group_tiles"] > 0   # the sink makes later tiles trail


# ----------------------------------------------------------------------------------------------
# Hilbert ordering and the token permutation
# ----------------------------------------------------------------------------------------------
def lsystem_hilbert(order):
    """Turtle walk of the Lindenmayer system A -> +BF-AFA-FB+, B -> -AF+BFB+FA- (an independent
    construction of the Hilbert curve)."""
    s = "A"
    for _ in range(order):
        s = "".join({"A": "+BF-AFA-FB+", "B": "-AF+BFB+FA-"}.get(ch, ch) for ch in s)
    x = y = 0
    dx, dy = 1, 0
    pts = [(0, 0)]
    for ch in s:
        if ch == "F":
            x, y = x + dx, y + dy
            pts.append((x, y))
        elif ch == "+":
            dx, dy = -dy, dx
        elif ch == "-":
            dx, dy = dy, -dx
    return pts


@pytest.mark.parametrize("order", [1, 2, 3, 4])
def test_hilbert_2d_matches_lsystem_up_to_symmetry(order):
    n = 1 << order
    ours = sorted(((oracle.hilbert_index_2d(x, y, order), (x, y)) for x in range(n) for y in range(n)))
    ours = [p for _, p in ours]
    ls = lsystem_hilbert(order)
    mnx = min(p[0] for p in ls); mny = min(p[1] for p in ls)
    ls = [(p[0] - mnx, p[1] - mny) for p in ls]
    syms = [lambda x, y: (x, y), lambda x, y: (y, x), lambda x, y: (n - 1 - x, y), lambda x, y: (x, n - 1 - y),
            lambda x, y: (n - 1 - x, n - 1 - y), lambda x, y: (y, n - 1 - x), lambda x, y: (n - 1 - y, x),
            lambda x, y: (n - 1 - y, n - 1 - x)]
    assert any([f(*p) for p in ls] == ours for f in syms)
    assert ours[0] == (0, 0) and ours[-1] == (n - 1, 0)


@pytest.mark.parametrize("bits", [1, 2, 3])
def test_hilbert_3d_bijective_and_adjacent(bits):
    n = 1 << bits
    idx = {oracle.hilbert_index_3d((a, b, c), bits): (a, b, c) for a in range(n) for b in range(n) for c in range(n)}
    assert sorted(idx) == list(range(n ** 3))
    assert idx[0] == (0, 0, 0)
    for t in range(n ** 3 - 1):
        assert sum(abs(u - w) for u, w in zip(idx[t], idx[t + 1])) == 1


def test_hilbert_perms():
    p2 = oracle.hilbert_perm_2d(5, 8, 8)
    assert sorted(p2) == list(range(69)) and list(p2[:5]) == list(range(5))
    for t in range(5, 68):   # full power-of-two grid: consecutive tokens are 4-neighbours
        a, b = p2[t] - 5, p2[t + 1] - 5
        assert abs(a // 8 - b // 8) + abs(a % 8 - b % 8) == 1
    p3 = oracle.hilbert_perm_3d(3, 3, 5, 6)
    assert sorted(p3) == list(range(3 + 90)) and list(p3[:3]) == [0, 1, 2]
    pf = oracle.hilbert_perm_2d(512, 64, 64)
    assert sorted(pf) == list(range(4608))


def test_permutation_equivariance_of_dense_attention():
    q, k, v = (f64(t) for t in W.random_qkv(12, 1, 2, 2, 4 + 64, 32))
    perm = oracle.hilbert_perm_2d(4, 8, 8)
    ref = oracle.block_sparse_attn(q, k, v, None, -math.inf, False)
    pq, pk, pv = (oracle.permute_tokens(t, perm) for t in (q, k, v))
    out = oracle.unpermute_tokens(oracle.block_sparse_attn(pq, pk, pv, None, -math.inf, False), perm)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(oracle.unpermute_tokens(oracle.permute_tokens(q, perm), perm), q)


def test_decisive_rows_flag_near_ties():
    w = W.make_config("tiny")
    q, k = f64(w.q), f64(w.k)
    pred = oracle.predict_mask(q, k, 0.5, 0.3, False)
    dec = oracle.decisive_rows(pred, 0.5, 0.3, False)
    assert dec.mean() > 0.5
    # moving topk onto a row's exact cumulative sum makes that row non-decisive
    p = pred["P"][0, 0, 0]
    t = float(np.cumsum(np.sort(p)[::-1])[1])
    pred2 = oracle.predict_mask(q, k, t, 0.3, False)
    assert not oracle.decisive_rows(pred2, t, 0.3, False)[0, 0, 0]


# ----------------------------------------------------------------------------------------------
# single-row mask prediction (used on workloads too large to predict whole)
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["cdf", "count"])
@pytest.mark.parametrize("causal,Nq,Nk,Hq,Hkv,topk,theta", [
    (True, 1000, 1000, 4, 2, 0.5, 0.5),     # causal GQA, ragged tails of both block sizes
    (False, 700, 700, 2, 2, 0.3, 0.6),      # non-causal
    (True, 300, 1100, 4, 1, 0.6, 0.4),      # a short query chunk continuing a longer key sequence
    (False, 900, 513, 2, 1, 0.9, 0.5),      # more queries than keys, non-causal
])
def test_predict_mask_row_equals_predict_mask(mode, causal, Nq, Nk, Hq, Hkv, topk, theta):
    """predict_mask_row (one query block against one pooled key head) gives, on every row, the
    mask, probabilities, scores and similarities of the pinned whole-tensor predict_mask, with the
    key head pooled per call or once (k_pool)."""
    w = W.make_config("tiny", B=1, Hq=Hq, Hkv=Hkv, N=max(Nq, Nk), d=64)
    q = f64(w.q)[:, :, :Nq]
    k = f64(w.k)[:, :, :Nk]
    pred = oracle.predict_mask(q, k, topk, theta, causal, mode=mode)
    off = Nk - Nq
    G = Hq // Hkv
    for h in range(Hq):
        kp = oracle.pool_key_head(k[0, h // G])
        for i in range(pred["mask"].shape[2]):
            qb = q[0, h, i * 128:min(Nq, (i + 1) * 128)]
            for pool in (None, kp):
                r = oracle.predict_mask_row(qb, k[0, h // G], i, topk, theta, causal, mode=mode, off=off, k_pool=pool)
                assert np.array_equal(r["mask"], pred["mask"][0, h, i]), (h, i)
                np.testing.assert_allclose(r["P"], pred["P"][0, h, i], rtol=1e-12, atol=1e-15)
                np.testing.assert_array_equal(np.isneginf(r["S"]), np.isneginf(pred["S"][0, h, i]))
                fin = ~np.isneginf(r["S"])
                np.testing.assert_allclose(r["S"][fin], pred["S"][0, h, i][fin], rtol=1e-12, atol=1e-12)
                assert r["sQ"] == pytest.approx(pred["sQ"][0, h, i], abs=1e-14)
                np.testing.assert_allclose(r["sK"], pred["sK"][0, h // G], rtol=0, atol=1e-14)
                np.testing.assert_array_equal(r["valid"], oracle.block_valid(i + 1, r["valid"].size, causal, off)[i])


def test_cut_margins_agree_with_topk_select():
    """cut_margins places the cut where topk_select does, in both readings of topk."""
    rng = np.random.default_rng(5)
    for trial in range(200):
        n = int(rng.integers(1, 40))
        p = rng.dirichlet(np.full(n, 0.3))
        valid = rng.random(n) < 0.8
        valid[int(rng.integers(n))] = True
        p = np.where(valid, p, 0.0)
        p /= p.sum()
        topk = float(rng.uniform(0.05, 0.95))
        for mode in ("cdf", "count"):
            keep = oracle.topk_select(p, valid, topk, mode)
            m = oracle.cut_margins(p, valid, topk, mode)
            assert keep.sum() == m["kstar"]
            assert set(np.nonzero(keep)[0]) == set(m["order"][:m["kstar"]])
            assert m["p_cut"] == p[keep].min()
            assert m["c_at"] == pytest.approx(p[keep].sum(), abs=1e-12)
