"""Seeded synthetic inputs shaped like the SpargeAttn workloads.

This module only draws random numbers and rounds them to bf16.  It holds none
of the method's arithmetic (no pooling, scoring, selection or attention) and it
imports neither the oracle nor the CUDA package, so both sides can take their
inputs from here.

Every generator uses ``numpy.random.Generator(PCG64(seed))``.  Draw order is
Q, K, V, then the custom mask; within a tensor the draws go batch-major, then
head, as written in each function.  ``N(m, s)`` means standard deviation ``s``.

The shapes stand in for the workloads the SpargeAttn pages evaluate on
(SpargeAttention paper summary: Llama 3.1 at 128K context, Flux image
generation, CogVideoX video generation).  None of those models or datasets is
used; only their attention shapes and a token structure with the same kind of
locality.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import numpy as np

QBLK = 128  # query rows per mask block (fixed 128x64 granularity of the mask API)
KBLK = 64   # key rows per mask block


# --------------------------------------------------------------------------
# bf16 helpers (storage format only)
# --------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Expand bf16 bit patterns (uint16) to float32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_to_f32(b).astype(np.float64)


# --------------------------------------------------------------------------
# configuration records
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    topk: float
    theta: float
    lam: float
    n_prefix: int = 0                      # text tokens that precede the image/video grid
    grid: Optional[Tuple[int, ...]] = None  # (H, W) image grid or (T, H, W) video grid
    q: Optional[np.ndarray] = None          # uint16 bf16 bits, (B, Hq, N, d)
    k: Optional[np.ndarray] = None          # (B, Hkv, N, d)
    v: Optional[np.ndarray] = None          # (B, Hkv, N, d)
    mask: Optional[np.ndarray] = None       # uint8 (B, Hq, ceil(N/128), ceil(N/64)) for the custom-mask workload

    @property
    def nqb(self) -> int:
        return -(-self.N // QBLK)

    @property
    def nkb(self) -> int:
        return -(-self.N // KBLK)

    def dense_flops(self) -> float:
        """Dense-equivalent attention work, 4*B*Hq*N^2*d (full square even when causal)."""
        return 4.0 * self.B * self.Hq * float(self.N) ** 2 * self.d


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


# --------------------------------------------------------------------------
# token structures
# --------------------------------------------------------------------------
def _block_mean_tokens(rng, B, H, N, d, blk=64, noise=0.3):
    """Per (head, 64-token block) a mean mu ~ N(0,1)^d, every token = mu + N(0, noise)."""
    nb = -(-N // blk)
    out = np.empty((B, H, N, d), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            mu = _normal(rng, (nb, d))
            x = np.repeat(mu, blk, axis=0)[:N] + _normal(rng, (N, d), noise)
            out[b, h] = bf16_bits(x)
    return out


def _periodic_gauss_tf(shape, sigmas):
    """Fourier transform of a unit-mass periodic Gaussian kernel on a grid (for FFT smoothing)."""
    tf = np.ones(shape, dtype=np.float64)
    for ax, (n, s) in enumerate(zip(shape, sigmas)):
        r = np.arange(n)
        r = np.minimum(r, n - r).astype(np.float64)       # wrap-around distance
        g = np.exp(-0.5 * (r / s) ** 2)
        g /= g.sum()
        gf = np.real(np.fft.fft(g))
        sh = [1] * len(shape)
        sh[ax] = n
        tf = tf * gf.reshape(sh)
    return tf


def _smooth_field_tokens(rng, B, H, d, n_prefix, grid, sigmas, noise=0.2):
    """Text prefix iid N(0,1), then a grid of tokens: per (head, dim) white noise smoothed by
    a periodic Gaussian (via FFT), renormalised to unit variance, plus N(0, noise).
    Grid tokens are laid out in row-major order of the grid."""
    ng = int(np.prod(grid))
    N = n_prefix + ng
    tf = _periodic_gauss_tf(grid, sigmas)
    axes = tuple(range(1, 1 + len(grid)))
    out = np.empty((B, H, N, d), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            pre = _normal(rng, (n_prefix, d))
            white = rng.standard_normal(size=(d,) + tuple(grid))
            f = np.real(np.fft.ifftn(np.fft.fftn(white, axes=axes) * tf[None], axes=axes))
            f /= f.reshape(d, -1).std(axis=1).reshape((d,) + (1,) * len(grid))
            tok = f.reshape(d, ng).T.astype(np.float32) + _normal(rng, (ng, d), noise)
            out[b, h] = bf16_bits(np.concatenate([pre, tok], axis=0))
    return out


ROTARY_BASE = 500000.0
ROTARY_AMPLITUDE = 2.0


def _rotary_tokens(rng, B, H, N, d, sink_tokens=0, sink_scale=8.0, amplitude=ROTARY_AMPLITUDE):
    """N(0,1) tokens plus slowly varying rotary-style components: for each dim pair (2p, 2p+1)
    whose period 2*pi/w_p is at least 128 tokens, w_p = 500000^(-2p/d), add
    amplitude*(cos(t w_p + phi), sin(t w_p + phi)) with a phase phi drawn per (head, pair).
    The first ``sink_tokens`` tokens are then scaled by ``sink_scale`` (an attention sink)."""
    p = np.arange(d // 2)
    omega = ROTARY_BASE ** (-2.0 * p / d)
    slow = np.nonzero(2.0 * np.pi / omega >= 128.0)[0]
    t = np.arange(N, dtype=np.float64)
    out = np.empty((B, H, N, d), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            x = _normal(rng, (N, d))
            phi = rng.uniform(0.0, 2.0 * np.pi, size=d // 2)
            ang = t[:, None] * omega[None, slow] + phi[None, slow]
            x[:, 2 * slow] += (amplitude * np.cos(ang)).astype(np.float32)
            x[:, 2 * slow + 1] += (amplitude * np.sin(ang)).astype(np.float32)
            if sink_tokens:
                x[:sink_tokens] *= np.float32(sink_scale)
            out[b, h] = bf16_bits(x)
    return out


def _iid_tokens(rng, B, H, N, d):
    out = np.empty((B, H, N, d), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            out[b, h] = bf16_bits(_normal(rng, (N, d)))
    return out


def _bernoulli_mask(rng, B, H, N, p=0.25):
    nqb, nkb = -(-N // QBLK), -(-N // KBLK)
    m = (rng.random(size=(B, H, nqb, nkb)) < p).astype(np.uint8)
    i = np.arange(nqb)
    for jj in (2 * i, 2 * i + 1):
        ok = jj < nkb
        m[:, :, i[ok], jj[ok]] = 1
    return m


# --------------------------------------------------------------------------
# named workloads
# --------------------------------------------------------------------------
CONFIG_NAMES = ("tiny", "flux", "cogvideox", "llama32k", "llama128k", "custom", "vit")

# one line per workload on how its tokens are drawn (for reports)
DATA_DESCRIPTIONS = {
    "tiny": "per-block mean N(0,1) plus N(0,0.3) token noise",
    "flux": "text prefix N(0,1) plus a 2-D Gaussian random field image grid with N(0,0.2) noise",
    "cogvideox": "text prefix N(0,1) plus a 3-D smooth Gaussian field video grid with N(0,0.2) noise",
    "llama32k": "Llama-like rotary structure with attention sink",
    "llama128k": "Llama-like rotary structure with attention sink",
    "custom": "i.i.d. N(0,1) Q/K/V with a Bernoulli(0.25) tile mask, diagonal tiles on",
    "vit": "a 64 x 64 patch grid, 2-D Gaussian random field (correlation length 4 patches) with N(0,0.2) noise",
}


def describe(name: str, **over) -> Workload:
    """Shape and settings of a named workload without drawing its tensors."""
    if name == "tiny":
        w = Workload(name, 1, 2, 2, 1024, 64, False, 0.5, 0.5, -math.inf)
    elif name == "flux":
        w = Workload(name, 1, 24, 24, 512 + 64 * 64, 128, False, 0.5, 0.5, -math.inf,
                     n_prefix=512, grid=(64, 64))
    elif name == "cogvideox":
        w = Workload(name, 1, 30, 30, 226 + 13 * 30 * 45, 64, False, 0.3, 0.5, -math.inf,
                     n_prefix=226, grid=(13, 30, 45))
    elif name == "llama32k":
        w = Workload(name, 1, 32, 8, 32768, 128, True, 0.5, 0.5, -8.0)
    elif name == "llama128k":
        w = Workload(name, 1, 32, 8, 131072, 128, True, 0.5, 0.5, -8.0)
    elif name == "custom":
        w = Workload(name, 2, 16, 16, 65536, 128, False, 1.0, 0.5, -math.inf)
    elif name == "vit":
        # ViT-like image encoder: small batch, non-causal, 64 x 64 patches, no text prefix
        w = Workload(name, 2, 12, 12, 64 * 64, 64, False, 0.5, 0.5, -math.inf, n_prefix=0, grid=(64, 64))
    else:
        raise KeyError(name)
    for key, val in over.items():
        setattr(w, key, val)
    if w.grid is not None:
        w.N = w.n_prefix + int(np.prod(w.grid))
    return w


def make_config(name: str, seed: int = 0, **over) -> Workload:
    """Draw the tensors of a named workload.

    ``over`` may shrink a workload for quick checks (``Hq``, ``Hkv``, ``N``, ``B``, ``grid``,
    ``n_prefix``) while keeping its token structure.  For the grid workloads N is recomputed
    from ``n_prefix`` and ``grid``."""
    w = describe(name, **over)
    rng = np.random.Generator(np.random.PCG64(seed))
    B, Hq, Hkv, N, d = w.B, w.Hq, w.Hkv, w.N, w.d
    if name == "tiny":
        w.q = _block_mean_tokens(rng, B, Hq, N, d)
        w.k = _block_mean_tokens(rng, B, Hkv, N, d)
        w.v = _block_mean_tokens(rng, B, Hkv, N, d)
    elif name == "flux":
        sig = (6.0, 6.0)
        w.q = _smooth_field_tokens(rng, B, Hq, d, w.n_prefix, w.grid, sig)
        w.k = _smooth_field_tokens(rng, B, Hkv, d, w.n_prefix, w.grid, sig)
        w.v = _smooth_field_tokens(rng, B, Hkv, d, w.n_prefix, w.grid, sig)
    elif name == "vit":
        sig = (4.0, 4.0)
        w.q = _smooth_field_tokens(rng, B, Hq, d, w.n_prefix, w.grid, sig)
        w.k = _smooth_field_tokens(rng, B, Hkv, d, w.n_prefix, w.grid, sig)
        w.v = _smooth_field_tokens(rng, B, Hkv, d, w.n_prefix, w.grid, sig)
    elif name == "cogvideox":
        sig = (3.0, 5.0, 5.0)
        w.q = _smooth_field_tokens(rng, B, Hq, d, w.n_prefix, w.grid, sig)
        w.k = _smooth_field_tokens(rng, B, Hkv, d, w.n_prefix, w.grid, sig)
        w.v = _smooth_field_tokens(rng, B, Hkv, d, w.n_prefix, w.grid, sig)
    elif name in ("llama32k", "llama128k"):
        w.q = _rotary_tokens(rng, B, Hq, N, d)
        w.k = _rotary_tokens(rng, B, Hkv, N, d, sink_tokens=4)
        w.v = _iid_tokens(rng, B, Hkv, N, d)
    elif name == "custom":
        w.q = _iid_tokens(rng, B, Hq, N, d)
        w.k = _iid_tokens(rng, B, Hkv, N, d)
        w.v = _iid_tokens(rng, B, Hkv, N, d)
        w.mask = _bernoulli_mask(rng, B, Hq, N)
    return w


def random_qkv(seed, B, Hq, Hkv, N, d, std=1.0):
    """Plain iid N(0, std) bf16 Q/K/V for edge-case tests."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = bf16_bits(_normal(rng, (B, Hq, N, d), std))
    k = bf16_bits(_normal(rng, (B, Hkv, N, d), std))
    v = bf16_bits(_normal(rng, (B, Hkv, N, d), std))
    return q, k, v


def climbing_qkv(seed, B, Hq, Hkv, N, d, step_log2=9.0, alpha=4.0):
    """Q/K whose scores climb from each 64-key block to the next (edge-case tests of the O rescale).

    Every query is alpha * u plus N(0, 0.1) noise and every key of key block b is beta_b * u plus
    N(0, 0.1) noise, for one random unit vector u per head, with beta_b chosen so that the score
    q.k / sqrt(d) grows by step_log2 (in log2 units) per key block; V is iid N(0, 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    u = _normal(rng, (B, Hkv, 1, d), 1.0)
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    G = Hq // Hkv
    uq = np.repeat(u, G, axis=1)
    dbeta = step_log2 * math.log(2.0) * math.sqrt(d) / alpha
    beta = (np.arange(N) // KBLK).astype(np.float32) * np.float32(dbeta)
    q = alpha * uq + _normal(rng, (B, Hq, N, d), 0.1)
    k = beta[None, None, :, None] * u + _normal(rng, (B, Hkv, N, d), 0.1)
    v = _normal(rng, (B, Hkv, N, d), 1.0)
    return bf16_bits(q), bf16_bits(k), bf16_bits(v)


def random_mask(seed, B, H, N, p=0.25, force_diag=True):
    """Bernoulli(p) tile mask, optionally with the diagonal tiles (2i, 2i+1) forced on."""
    rng = np.random.Generator(np.random.PCG64(seed))
    nqb, nkb = -(-N // QBLK), -(-N // KBLK)
    m = (rng.random(size=(B, H, nqb, nkb)) < p).astype(np.uint8)
    if force_diag:
        i = np.arange(nqb)
        for jj in (2 * i, 2 * i + 1):
            ok = jj < nkb
            m[:, :, i[ok], jj[ok]] = 1
    return m
