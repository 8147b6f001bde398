"""Float64 CPU oracle of the SpargeAttn two-stage sparse attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module.  The CUDA library never calls it, and it shares
no code with the CUDA library.

Sources (page titles of the SpargeAttn material, cited by section):
  [abstract]  "SpargeAttention: Accurate and Training-free Sparse Attention Accelerating Any
              Model Inference" (paper abstract page) -- two-stage online filter: stage 1
              predicts the attention map so some matrix multiplications are skipped; stage 2
              is an online softmax-aware filter that skips further updates.
  [summary]   same title (paper summary page), method paragraph -- blocks with high internal
              similarity are compressed, non-similar blocks are always computed, the second
              filter works at GPU-warp level, Hilbert-curve reordering for visual tokens.
  [overview]  "SpargeAttn: accelerate LLM inference without training" -- plug-and-play API
              ``f(q, k, v, topk=0.5, is_causal=False)``, drop-in for scaled_dot_product_attention,
              per-head block mask of shape (B, H, ceil(N/128), ceil(N/64)), fixed 128x64 blocks,
              topk in (0, 1], lower is sparser.
  [readme-cn] "SpargeAttention" (Chinese README): custom block-sparse mask API; the mask is made
              of 0 and 1 with 1 meaning the block is kept; topk=0.5 keeps the top 50% of the
              attention weights.

Where the pages leave a step open, the reading taken is stated at the function that takes it.
Every function computes in float64 on inputs that are the bf16 values upcast exactly.

Parity status: pool_sim, pooled_scores, topk_select, predict_mask, block_sparse_attn,
sparge_attn, the Hilbert orderings and the token permutation are pinned by the tests
(closed forms, brute force, library routines, textbook curves).  The 8-bit path has no
oracle of its own rounding: it is checked only by tolerance against block_sparse_attn.
"""
from __future__ import annotations

import math
from typing import Dict, Tuple

import numpy as np

QBLK = 128       # query tokens per block  [overview: "128x64 block granularity"]
KBLK = 64        # key tokens per block
WARP_ROWS = 32   # rows whose P.V update is skipped together  [summary: "at the GPU warp level"]


def n_blocks(N: int, blk: int) -> int:
    return -(-N // blk)


def default_scale(d: int) -> float:
    """Softmax scale 1/sqrt(d): the SDPA default, implied by the drop-in-replacement claim
    [overview, "Using the plug-and-play API"].  Reading: the pooled scores use the same scale."""
    return 1.0 / math.sqrt(d)


# ---------------------------------------------------------------------------------------------
# Stage 1a: block mean pooling and intra-block self-similarity
# ---------------------------------------------------------------------------------------------
def pool_sim(x: np.ndarray, blk: int) -> Tuple[np.ndarray, np.ndarray]:
    """Mean of each block of ``blk`` tokens and its self-similarity.

    [summary, method paragraph] stage 1 compresses token blocks that show high internal
    similarity.  Reading of "internal similarity": the mean cosine similarity over all ordered
    pairs (a, b) of tokens in the block, the pairs a == b included.  That mean equals
    ||(1/n) sum_a x_a/||x_a|| ||^2, which is what is computed here; a token of zero norm
    contributes a zero unit vector.  A partial tail block uses its valid tokens only.

    x: (B, H, N, d) float64.  Returns mu (B, H, nb, d) and s (B, H, nb)."""
    B, H, N, d = x.shape
    nb = n_blocks(N, blk)
    mu = np.zeros((B, H, nb, d))
    s = np.zeros((B, H, nb))
    for i in range(nb):
        xb = x[:, :, i * blk:min(N, (i + 1) * blk), :]
        n = xb.shape[2]
        mu[:, :, i, :] = xb.sum(axis=2) / n
        nrm = np.sqrt((xb * xb).sum(axis=-1, keepdims=True))
        unit = np.divide(xb, nrm, out=np.zeros_like(xb), where=nrm > 0)
        h = unit.sum(axis=2) / n
        s[:, :, i] = (h * h).sum(axis=-1)
    return mu, s


# ---------------------------------------------------------------------------------------------
# Stage 1b: pooled score map, row softmax, cumulative top-k, always-keep
# ---------------------------------------------------------------------------------------------
def block_valid(nqb: int, nkb: int, causal: bool, off: int = 0) -> np.ndarray:
    """(nqb, nkb) bool: a 128x64 tile is valid unless causal attention hides all of it.
    Query row r sees key column c when c <= off + r, where off = Nk - Nq puts the last query on
    the last key (a short query block continues the key sequence; reading for Nq < Nk, the
    pages only treat Nq = Nk, off = 0).  Tile (i, j) holds some visible element iff
    64*j <= off + 128*i + 127."""
    i = np.arange(nqb)[:, None]
    j = np.arange(nkb)[None, :]
    if not causal:
        return np.ones((nqb, nkb), dtype=bool)
    return KBLK * j <= off + QBLK * i + (QBLK - 1)


def pooled_scores(muQ: np.ndarray, muK: np.ndarray, causal: bool, scale: float, off: int = 0) -> np.ndarray:
    """S_hat[b, h, i, j] = scale * muQ[b, h, i] . muK[b, h // G, j], -inf on invalid tiles.

    [abstract] stage 1 predicts the attention map from a compressed form of Q and K; the
    compressed tokens are the block means.  G = Hq / Hkv (reading: query heads share the pooled
    keys of their key/value head, as grouped-query attention shares K and V)."""
    B, Hq, nqb, d = muQ.shape
    Hkv, nkb = muK.shape[1], muK.shape[2]
    G = Hq // Hkv
    S = np.empty((B, Hq, nqb, nkb))
    for b in range(B):
        for h in range(Hq):
            S[b, h] = scale * (muQ[b, h] @ muK[b, h // G].T)
    S[:, :, ~block_valid(nqb, nkb, causal, off)] = -np.inf
    return S


def row_softmax(S: np.ndarray) -> np.ndarray:
    """Softmax over the last axis, -inf entries get probability 0."""
    m = S.max(axis=-1, keepdims=True)
    e = np.exp(S - m)
    return e / e.sum(axis=-1, keepdims=True)


def count_target(topk: float, n: int) -> int:
    """Blocks kept by the count reading of topk for a row of n valid blocks: ceil(topk * n),
    taken with topk as the float32 the library receives and a 1e-3 allowance below each integer
    (so 0.3 of 10 blocks is 3, not 4 through rounding), at least 1 and at most n."""
    t = float(np.float32(topk)) * n - 1e-3
    return int(min(n, max(1, math.ceil(t))))


def topk_select(p: np.ndarray, valid: np.ndarray, topk: float, mode: str = "cdf", topp: float = None) -> np.ndarray:
    """Keep set of one row of block probabilities.

    [overview, FAQ] topk lies in (0, 1]; lower means sparser.  [readme-cn, quick start]
    topk = 0.5 keeps the top 50% of the attention weights.  Reading ("cdf", the library's
    default): order the valid blocks by (probability descending, index ascending) and keep the
    shortest prefix whose cumulative probability reaches topk; topk >= 1 keeps every valid
    block; at least one block is kept.  The other reading of the knob ("count"): keep the first
    count_target(topk, n_valid) blocks of that order.

    "hybrid": [readme-cn, citation list] names a hybrid Top-k + Top-p mask (SpargeAttention2)
    without a rule.  Reading: a block is kept when the count reading with topk keeps it or the
    cumulative reading with topp keeps it (the union of a top-k set and a top-p set).

    p: (nkb,) probabilities, valid: (nkb,) bool with at least one True.  Returns bool (nkb,)."""
    if mode == "hybrid":
        return topk_select(p, valid, topk, "count") | topk_select(p, valid, topp, "cdf")
    keep = np.zeros(p.shape[0], dtype=bool)
    if topk >= 1.0:
        keep[valid] = True
        return keep
    vj = np.nonzero(valid)[0]
    order = vj[np.lexsort((vj, -p[vj]))]
    if mode == "count":
        keep[order[:count_target(topk, order.size)]] = True
        return keep
    assert mode == "cdf", mode
    c = np.cumsum(p[order])
    hit = np.nonzero(c >= topk)[0]
    kstar = (hit[0] + 1) if hit.size else order.size
    keep[order[:kstar]] = True
    return keep


def predict_mask(q: np.ndarray, k: np.ndarray, topk: float, theta: float, causal: bool,
                 scale: float = None, mode: str = "cdf", topp: float = None) -> Dict[str, np.ndarray]:
    """Stage 1 of SpargeAttn: the (B, Hq, ceil(N/128), ceil(N/64)) uint8 block mask.

    [overview, "Strengths"] mask shape and 128x64 granularity; [readme-cn, custom mask] 1 = keep.
    [summary, method paragraph] non-similar blocks are always computed.  Reading of that rule:
    after top-k, a query block i with s_Q < theta keeps every valid key block of its row, and a
    key block j with s_K < theta is kept in every valid row of every query head that shares its
    key/value head.  The softmax is taken over all valid blocks, similar or not.  Comparisons
    with theta are strict.

    q: (B, Hq, Nq, d), k: (B, Hkv, Nk, d) float64 (Nq <= Nk when causal; off = Nk - Nq as in
    block_valid).  mode: the reading of topk (topk_select; topp is the top-p mass of "hybrid")."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    off = k.shape[2] - N
    G = Hq // Hkv
    if scale is None:
        scale = default_scale(d)
    muQ, sQ = pool_sim(q, QBLK)
    muK, sK = pool_sim(k, KBLK)
    S = pooled_scores(muQ, muK, causal, scale, off)
    P = row_softmax(S)
    nqb, nkb = S.shape[2], S.shape[3]
    valid = block_valid(nqb, nkb, causal, off)
    mask = np.zeros((B, Hq, nqb, nkb), dtype=np.uint8)
    for b in range(B):
        for h in range(Hq):
            colkeep = sK[b, h // G] < theta
            for i in range(nqb):
                keep = topk_select(P[b, h, i], valid[i], topk, mode, topp)
                if sQ[b, h, i] < theta:
                    keep |= valid[i]
                keep |= colkeep & valid[i]
                mask[b, h, i] = keep
    return dict(mask=mask, muQ=muQ, sQ=sQ, muK=muK, sK=sK, S=S, P=P, off=off)


def row_decisive(p: np.ndarray, valid: np.ndarray, sq: float, sk: np.ndarray, topk: float, theta: float,
                 eps: float = 1e-3, mode: str = "cdf", topp: float = None) -> bool:
    """Whether no rounding within ``eps`` can change one mask row (the bit-exact comparison set).

    A row is decisive when its query similarity is farther than eps from theta and either it
    keeps every block because s_Q < theta, or (i) the cumulative sum at the cut and the one
    before it are farther than eps from topk, (ii) the probability gap at the cut exceeds eps,
    and (iii) every valid key block similarity is farther than eps from theta.  In the count
    reading only (ii) and (iii) apply (the number kept does not depend on rounding); in the
    hybrid reading both cuts (count with topk, cumulative with topp) must be decisive.
    p: row probabilities (nkb,), valid: bool (nkb,), sq: s_Q of the row, sk: s_K (nkb,)."""
    if abs(sq - theta) <= eps:
        return False
    if sq < theta:
        return True
    if not np.all(np.abs(sk[valid] - theta) > eps):
        return False
    if mode == "hybrid":
        return (row_decisive(p, valid, sq, sk, topk, theta, eps, "count") and
                row_decisive(p, valid, sq, sk, topp, theta, eps, "cdf"))
    if topk >= 1.0:
        return True
    m = cut_margins(p, valid, topk, mode)
    if mode == "count":
        return bool(m["kstar"] >= m["n"] or m["gap"] > eps)
    return bool(abs(m["c_at"] - topk) > eps and abs(topk - m["c_before"]) > eps and m["gap"] > eps)


def cut_margins(p: np.ndarray, valid: np.ndarray, topk: float, mode: str = "cdf") -> Dict[str, float]:
    """Where the top-k cut of one row falls and how far it is from moving (topk < 1).

    Returns the valid blocks in (probability desc, index asc) order ("order"), their count n,
    the number kept by the cut ("kstar", as topk_select), the probability of the last kept block
    ("p_cut") and of the first dropped one ("p_next", 0 if none), their difference ("gap"), and
    the cumulative probability through the cut ("c_at") and through the block before it
    ("c_before", 0 if none)."""
    vj = np.nonzero(valid)[0]
    order = vj[np.lexsort((vj, -p[vj]))]
    ps = p[order]
    c = np.cumsum(ps)
    if mode == "count":
        kstar = count_target(topk, order.size)
    else:
        assert mode == "cdf", mode
        hit = np.nonzero(c >= topk)[0]
        kstar = int(hit[0] + 1) if hit.size else order.size
    p_next = float(ps[kstar]) if kstar < ps.size else 0.0
    return dict(order=order, n=int(order.size), kstar=int(kstar), p_cut=float(ps[kstar - 1]), p_next=p_next,
                gap=float(ps[kstar - 1]) - p_next, c_at=float(c[kstar - 1]),
                c_before=float(c[kstar - 2]) if kstar >= 2 else 0.0)


def decisive_rows(pred: Dict[str, np.ndarray], topk: float, theta: float, causal: bool,
                  eps: float = 1e-3, mode: str = "cdf", topp: float = None) -> np.ndarray:
    """row_decisive for every row of a predict_mask result: bool (B, Hq, nqb)."""
    P, sQ, sK = pred["P"], pred["sQ"], pred["sK"]
    B, Hq, nqb, nkb = P.shape
    G = Hq // sK.shape[1]
    valid = block_valid(nqb, nkb, causal, pred.get("off", 0))
    out = np.zeros((B, Hq, nqb), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            for i in range(nqb):
                out[b, h, i] = row_decisive(P[b, h, i], valid[i], sQ[b, h, i], sK[b, h // G], topk, theta, eps,
                                            mode, topp)
    return out


def pool_key_head(k_head: np.ndarray):
    """Pooled means and similarities of every 64-key block of one key/value head, (nkb, d) and
    (nkb,): the key half of stage 1, computed once and shared by the rows of that head."""
    muk, sk = pool_sim(k_head[None, None], KBLK)
    return muk[0, 0], sk[0, 0]


def predict_mask_row(q_block: np.ndarray, k_head: np.ndarray, i: int, topk: float, theta: float,
                     causal: bool, scale: float = None, mode: str = "cdf", off: int = 0,
                     k_pool=None, topp: float = None) -> Dict[str, np.ndarray]:
    """predict_mask for a single query block: q_block (n_i, d) the tokens of query block i,
    k_head (N, d) every key of its key/value head.  Same steps as predict_mask, for checking
    rows of workloads too large to run whole.  k_pool, if given, is pool_key_head(k_head),
    so that many rows of one head pool its keys once.  Returns mask (nkb,) uint8, P (nkb,),
    S (nkb,) the scaled pooled scores (-inf on invalid blocks), muQ (d,) and sQ (float) of the
    query block, sK (nkb,), valid (nkb,) bool."""
    N, d = k_head.shape
    if scale is None:
        scale = default_scale(d)
    muq, sq = pool_sim(q_block[None, None], QBLK)
    muk, sk = pool_key_head(k_head) if k_pool is None else k_pool
    nkb = muk.shape[0]
    valid = block_valid(i + 1, nkb, causal, off)[i]
    s = scale * (muk @ muq[0, 0, 0])
    s[~valid] = -np.inf
    p = row_softmax(s)
    keep = topk_select(p, valid, topk, mode, topp)
    if sq[0, 0, 0] < theta:
        keep |= valid
    keep |= (sk < theta) & valid
    return dict(mask=keep.astype(np.uint8), P=p, S=s, muQ=muq[0, 0, 0], sQ=float(sq[0, 0, 0]), sK=sk, valid=valid)


# ---------------------------------------------------------------------------------------------
# Stage 2: block-sparse flash attention with the lambda warp filter
# ---------------------------------------------------------------------------------------------
def attn_qblock(Qi: np.ndarray, Kh: np.ndarray, Vh: np.ndarray, i: int, kept, lam: float, causal: bool,
                scale: float, group: int = WARP_ROWS, off: int = 0):
    """The rows of one query block: Qi (n_i, d), Kh/Vh (Nk, d) of its key/value head, kept the
    ascending key-block indices to visit (already restricted to valid tiles); causal rows see
    the columns c <= off + row (block_valid).  Returns the output rows (n_i, d) and (kept tiles,
    skipped group-tiles, tiles with a P.V update)."""
    N, d = Kh.shape
    r0 = i * QBLK
    nr = Qi.shape[0]
    grp = np.arange(nr) // group
    ngrp = grp[-1] + 1
    m = np.full(nr, -np.inf)
    l = np.zeros(nr)
    acc = np.zeros((nr, d))
    rows = np.arange(r0, r0 + nr)
    n_skip = n_pv = n_tiles = 0
    for j in kept:
        c0, c1 = j * KBLK, min(N, (j + 1) * KBLK)
        n_tiles += 1
        S = scale * (Qi @ Kh[c0:c1].T)
        if causal:
            S = np.where(np.arange(c0, c1)[None, :] > off + rows[:, None], -np.inf, S)
        m_loc = S.max(axis=1)
        m_new = np.maximum(m, m_loc)
        with np.errstate(invalid="ignore"):
            trailing = np.isneginf(m_loc) | np.isneginf(m_new) | ((m_loc - m_new) < lam)
        skip_g = np.array([trailing[grp == g].all() for g in range(ngrp)])
        n_skip += int(skip_g.sum())
        fin = ~np.isneginf(m_new)
        m_ref = np.where(fin, m_new, 0.0)
        alpha = np.where(fin, np.exp(m - m_ref), 1.0)
        Pm = np.where(fin[:, None], np.exp(S - m_ref[:, None]), 0.0)
        l = alpha * l + Pm.sum(axis=1)
        upd = Pm @ Vh[c0:c1]
        upd[skip_g[grp]] = 0.0
        if not skip_g.all():
            n_pv += 1
        acc = alpha[:, None] * acc + upd
        m = m_new
    out = np.divide(acc, l[:, None], out=np.zeros_like(acc), where=l[:, None] > 0)
    return out, (n_tiles, n_skip, n_pv)


def block_sparse_attn(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask, lam: float,
                      causal: bool, scale: float = None, group: int = WARP_ROWS,
                      return_stats: bool = False, qblocks=None):
    """Stage 2 of SpargeAttn, step by step as an online-softmax attention over kept tiles.

    [abstract] only the tiles the mask keeps are multiplied; the second-stage online
    softmax-aware filter skips further updates.  [summary] the filter acts at warp level.
    Reading of the filter: rows are grouped 32 at a time (one warp's rows); the key tiles of a
    query block are visited in ascending order; for tile j the group skips its P.V update when
    for every row r of the group m_local[r] - m_new[r] < lam (m_local the row max over tile j,
    m_new the running max after tile j; a row with m_local = -inf or m_new = -inf counts as
    trailing).  The running max and the row sum l are updated even for a skipped group; only
    P.V is left out.  lam = -inf disables the filter.  A row with no visible kept key outputs 0.

    mask: (B, Hq, nqb, nkb) uint8 or None (all ones).  Tiles above the causal diagonal are never
    visited.  ``qblocks`` optionally restricts the work to a list of (b, h, i) query blocks (the
    other rows of O stay 0).  q may be shorter than k and v (Nq <= Nk when causal, off = Nk - Nq
    as in block_valid).  Returns O (B, Hq, Nq, d) float64 (and statistics when asked)."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    off = k.shape[2] - N
    G = Hq // Hkv
    if scale is None:
        scale = default_scale(d)
    nqb, nkb = n_blocks(N, QBLK), n_blocks(k.shape[2], KBLK)
    valid = block_valid(nqb, nkb, causal, off)
    O = np.zeros((B, Hq, N, d))
    tot = np.zeros(3, dtype=np.int64)
    if qblocks is None:
        qblocks = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(nqb)]
    for b, h, i in qblocks:
        r0, r1 = i * QBLK, min(N, (i + 1) * QBLK)
        kept = np.ones(nkb, bool) if mask is None else (mask[b, h, i] != 0)
        js = np.nonzero(kept & valid[i])[0]
        O[b, h, r0:r1], st = attn_qblock(q[b, h, r0:r1], k[b, h // G], v[b, h // G], i, js, lam, causal,
                                         scale, group, off)
        tot += st
    if return_stats:
        return O, dict(kept_tiles=int(tot[0]), skipped_group_tiles=int(tot[1]), pv_tiles=int(tot[2]))
    return O


def sparge_attn(q, k, v, topk: float, causal: bool, theta: float = 0.5, lam: float = -math.inf,
                scale: float = None, return_all: bool = False):
    """The plug-and-play call [overview, "Using the plug-and-play API"]: stage 1 mask, then
    stage 2 attention.  Reading: theta defaults to 0.5 and lambda to -inf (no second filter),
    since the plug-and-play call takes neither."""
    pred = predict_mask(q, k, topk, theta, causal, scale)
    O = block_sparse_attn(q, k, v, pred["mask"], lam, causal, scale)
    if return_all:
        return O, pred
    return O


# ---------------------------------------------------------------------------------------------
# Hilbert-curve token order for image and video tokens  [summary, method paragraph]
# ---------------------------------------------------------------------------------------------
def hilbert_index_2d(x: int, y: int, order: int) -> int:
    """Position of cell (x, y) on the order-``order`` Hilbert curve over a 2^order square.

    The curve starts at (0, 0) and ends at (2^order - 1, 0).  Written from the recursive
    definition: the square splits into quadrants visited lower-left, upper-left, upper-right,
    lower-right; the lower-left copy is mirrored about the main diagonal and the lower-right
    copy about the anti-diagonal so that the pieces join end to end."""
    idx = 0
    for lev in range(order, 0, -1):
        h = 1 << (lev - 1)
        if x < h and y < h:
            qd, x, y = 0, y, x
        elif x < h:
            qd, x, y = 1, x, y - h
        elif y >= h:
            qd, x, y = 2, x - h, y - h
        else:
            qd, x, y = 3, h - 1 - y, h - 1 - (x - h)
        idx += qd * h * h
    return idx


def hilbert_index_3d(coords, bits: int) -> int:
    """Position of a point on the 3-D Hilbert curve of a 2^bits cube (J. Skilling, "Programming
    the Hilbert curve", AIP Conf. Proc. 707, 2004: transform the axes to the 'transposed' index,
    then read its bits most significant first, axis 0 first).  coords = (a0, a1, a2)."""
    X = [int(c) for c in coords]
    n = len(X)
    top = 1 << (bits - 1)
    qb = top
    while qb > 1:
        low = qb - 1
        for a in range(n):
            if X[a] & qb:
                X[0] ^= low
            else:
                t = (X[0] ^ X[a]) & low
                X[0] ^= t
                X[a] ^= t
        qb >>= 1
    for a in range(1, n):
        X[a] ^= X[a - 1]
    t = 0
    qb = top
    while qb > 1:
        if X[n - 1] & qb:
            t ^= qb - 1
        qb >>= 1
    for a in range(n):
        X[a] ^= t
    idx = 0
    for bit in range(bits - 1, -1, -1):
        for a in range(n):
            idx = (idx << 1) | ((X[a] >> bit) & 1)
    return idx


def _order_for(*extent) -> int:
    o = 0
    while (1 << o) < max(extent):
        o += 1
    return max(o, 1)


def hilbert_perm_2d(n_prefix: int, H: int, W: int) -> np.ndarray:
    """Gather permutation pi (int32, length n_prefix + H*W): new position t takes old token pi[t].
    Text tokens stay first and in order; image token (r, c), stored row-major after the prefix,
    is placed by its Hilbert index with x = c, y = r on the smallest 2^k square covering the grid
    (points outside the grid are skipped)."""
    k = _order_for(H, W)
    keys = np.array([hilbert_index_2d(c, r, k) for r in range(H) for c in range(W)], dtype=np.int64)
    order = np.argsort(keys, kind="stable")
    return np.concatenate([np.arange(n_prefix), n_prefix + order]).astype(np.int32)


def hilbert_perm_3d(n_prefix: int, T: int, H: int, W: int) -> np.ndarray:
    """As hilbert_perm_2d for a (T, H, W) video grid stored (t, r, c) row-major, ordered by the
    3-D Hilbert index of (t, r, c) on the smallest 2^k cube covering the grid."""
    k = _order_for(T, H, W)
    keys = np.array([hilbert_index_3d((t, r, c), k) for t in range(T) for r in range(H) for c in range(W)],
                    dtype=np.int64)
    order = np.argsort(keys, kind="stable")
    return np.concatenate([np.arange(n_prefix), n_prefix + order]).astype(np.int32)


def permute_tokens(x: np.ndarray, perm: np.ndarray) -> np.ndarray:
    """y[:, :, t] = x[:, :, perm[t]]."""
    return x[:, :, perm, :]


def unpermute_tokens(y: np.ndarray, perm: np.ndarray) -> np.ndarray:
    """Inverse of permute_tokens: x[:, :, perm[t]] = y[:, :, t]."""
    x = np.empty_like(y)
    x[:, :, perm, :] = y
    return x
