"""GB300 (sm_103a) SpargeAttn: two-stage sparse attention forward behind a C ABI.

Thin Python binding over ``libsparge.so`` (see include/sparge.h for the contract of every
call).  This module only marshals arguments: torch provides device memory and the current CUDA
stream, every step of the computation runs in the library's CUDA kernels.  There is no CPU
path: if the library is missing or no CUDA device is present the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsparge.so")

SPARGE_OK = 0
SPARGE_ERR_INVALID_ARG = -1
SPARGE_ERR_UNSUPPORTED = -2
SPARGE_ERR_WORKSPACE_TOO_SMALL = -3
SPARGE_ERR_CUDA = -4
SPARGE_ERR_DEVICE_TIMEOUT = -5
SPARGE_BF16 = 1
SPARGE_PRECISION_BF16 = 0
SPARGE_PRECISION_Q8 = 1
SPARGE_PRECISION_Q8_FP8PV = 2
SPARGE_PRECISION_BF16_FP8PV = 3
# precisions with an 8-bit product: d = 128 and the 8-bit workspace (SPARGE_OP_*_Q8)
PRECISIONS_8BIT = (SPARGE_PRECISION_Q8, SPARGE_PRECISION_Q8_FP8PV, SPARGE_PRECISION_BF16_FP8PV)
SPARGE_OP_PREDICT_MASK = 1
SPARGE_OP_BLOCK_SPARSE_ATTN = 2
SPARGE_OP_ATTN = 3
SPARGE_OP_BLOCK_SPARSE_ATTN_Q8 = 4
SPARGE_OP_ATTN_Q8 = 5
SPARGE_OP_TOKEN_ORDER = 0x100  # flag OR-ed into an op: room for token-ordered copies of Q and K
SPARGE_TOPK_CUMULATIVE = 0      # topk is a cumulative probability fraction (default)
SPARGE_TOPK_COUNT = 1           # topk is a fraction of the valid blocks to keep
SPARGE_TOPK_HYBRID = 2          # the count set of topk united with the cumulative set of topp
QBLK, KBLK = 128, 64


class SpargeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("sparge error %d: %s" % (code, msg))
        self.code = code


class sparge_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64), ("d", ctypes.c_int64),
                ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64), ("stride_n", ctypes.c_int64)]


class sparge_params(ctypes.Structure):
    _fields_ = [("theta", ctypes.c_float), ("lambda_", ctypes.c_float), ("scale", ctypes.c_float),
                ("precision", ctypes.c_int32), ("stats", ctypes.c_void_p), ("timing_events", ctypes.c_void_p),
                ("topk_per_head", ctypes.c_void_p), ("theta_per_head", ctypes.c_void_p),
                ("lambda_per_head", ctypes.c_void_p), ("token_order", ctypes.c_void_p), ("topk_mode", ctypes.c_int32),
                ("topp", ctypes.c_float)]


_lib = None

EXPORTS = {
    "sparge_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] + [ctypes.c_int64] * 5),
    "sparge_predict_mask": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_void_p]),
    "sparge_predict_mask_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_void_p]),
    "sparge_block_sparse_attn": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "sparge_block_sparse_attn_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_size_t, ctypes.c_void_p]),
    "sparge_attn": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_int,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "sparge_attn_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_size_t, ctypes.c_void_p]),
    "sparge_permute_tokens": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "sparge_unpermute_tokens": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "sparge_hilbert_perm_2d": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "sparge_hilbert_perm_3d": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "sparge_predict_mask_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_float,
                                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "sparge_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p]),
    "sparge_last_error": (ctypes.c_char_p, []),
    "sparge_get_device_status": (ctypes.c_int, [ctypes.c_void_p]),
}


def lib():
    """Load libsparge.so (built by ``free_block_sparse_gb300.build``); raise if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libsparge.so is not built (%s); run free_block_sparse_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc: int):
    if rc != SPARGE_OK:
        raise SpargeError(rc, lib().sparge_last_error().decode())


def _torch():
    import torch
    return torch


def _stream():
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _desc(t) -> sparge_tensor:
    torch = _torch()
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise TypeError("expected a CUDA tensor")
    if t.dtype != torch.bfloat16 or t.dim() != 4 or t.stride(-1) != 1:
        raise TypeError("expected a bf16 (B, H, N, d) tensor with contiguous last dim")
    B, H, N, d = t.shape
    sb, sh, sn, _ = t.stride()
    return sparge_tensor(t.data_ptr(), SPARGE_BF16, 0, B, H, N, d, sb, sh, sn)


def workspace_bytes(op: int, B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    return int(lib().sparge_workspace_bytes(op, B, Hq, Hkv, N, d))


def n_blocks(N: int):
    return -(-N // QBLK), -(-N // KBLK)


def _workspace(op, q, k, ws):
    torch = _torch()
    B, Hq, Nq, d = q.shape
    need = workspace_bytes(op, B, Hq, k.shape[1], max(Nq, k.shape[2]), d)   # N: an upper bound of both
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    return ws


def predict_mask(q, k, topk: float, theta: float = 0.5, causal: bool = False, ws=None, mask=None):
    """Stage 1: the (B, Hq, ceil(Nq/128), ceil(Nk/64)) uint8 block mask."""
    torch = _torch()
    B, Hq, Nq, d = q.shape
    nqb, nkb = -(-Nq // 128), -(-k.shape[2] // 64)
    if mask is None:
        mask = torch.empty((B, Hq, nqb, nkb), dtype=torch.uint8, device=q.device)
    ws = _workspace(SPARGE_OP_PREDICT_MASK, q, k, ws)
    dq, dk = _desc(q), _desc(k)
    _check(lib().sparge_predict_mask(ctypes.byref(dq), ctypes.byref(dk), float(topk), float(theta), int(causal),
                                     mask.data_ptr(), ws.data_ptr(), ws.numel(), _stream()))
    return mask


def predict_mask_ex(q, k, topk: float, causal: bool = False, theta: float = 0.5, scale: float = 0.0,
                    topk_per_head=None, theta_per_head=None, ws=None, mask=None, events=None, token_order=None,
                    topk_mode: int = SPARGE_TOPK_CUMULATIVE, topp: float = 1.0):
    """predict_mask with an explicit pooled-score scale, optional per-query-head topk and theta
    (float32 CUDA tensors of Hq entries), optional timing events ([0]-[3] are recorded), an
    optional token order (int32 CUDA tensor of N entries; the mask refers to the reordered
    sequence) and the reading of topk (topk_mode; topp is the top-p mass of the hybrid rule)."""
    torch = _torch()
    B, Hq, Nq, _ = q.shape
    if mask is None:
        mask = torch.empty((B, Hq, -(-Nq // 128), -(-k.shape[2] // 64)), dtype=torch.uint8, device=q.device)
    ws = _workspace(SPARGE_OP_PREDICT_MASK | (SPARGE_OP_TOKEN_ORDER if token_order is not None else 0), q, k, ws)
    p = _params(theta, -math.inf, scale, SPARGE_PRECISION_BF16, None, events, topk_per_head, theta_per_head,
                order=token_order, topk_mode=topk_mode, topp=topp)
    dq, dk = _desc(q), _desc(k)
    _check(lib().sparge_predict_mask_ex(ctypes.byref(dq), ctypes.byref(dk), float(topk), int(causal), ctypes.byref(p),
                                        mask.data_ptr(), ws.data_ptr(), ws.numel(), _stream()))
    return mask


def predict_ws_views(ws, B, Hq, Hkv, N, d, Nk=None):
    """Views of the stage-1 workspace after predict_mask: muQ (B,Hq,nqb,d), sQ (B,Hq,nqb),
    muK (B,Hkv,nkb,d), sK (B,Hkv,nkb) and the scaled pooled scores S (B,Hq,nqb,nkb), following
    the layout the library writes (regions 256-byte aligned; fp32 except the bf16 hi/lo copies of
    the means, which are skipped here).  N is the query length, Nk the key length (default N)."""
    torch = _torch()
    nqb = n_blocks(N)[0]
    nkb = n_blocks(N if Nk is None else Nk)[1]
    nkb_pad = -(-nkb // 4) * 4
    u8 = ws if ws.dtype == torch.uint8 else ws.view(torch.uint8)

    def take(off, nbytes):
        return u8[off:off + nbytes], off + ((nbytes + 255) // 256) * 256

    off = 0
    muQ, off = take(off, 4 * B * Hq * nqb * d)
    sQ, off = take(off, 4 * B * Hq * nqb)
    muK, off = take(off, 4 * B * Hkv * nkb * d)
    sK, off = take(off, 4 * B * Hkv * nkb_pad)
    _, off = take(off, 2 * B * Hq * nqb * d)
    _, off = take(off, 2 * B * Hq * nqb * d)
    _, off = take(off, 2 * B * Hkv * nkb * d)
    _, off = take(off, 2 * B * Hkv * nkb * d)
    S, off = take(off, 4 * B * Hq * nqb * nkb_pad)
    f = lambda t: t.view(torch.float32)
    return (f(muQ).view(B, Hq, nqb, d), f(sQ).view(B, Hq, nqb), f(muK).view(B, Hkv, nkb, d),
            f(sK).view(B, Hkv, nkb_pad)[..., :nkb], f(S).view(B, Hq, nqb, nkb_pad)[..., :nkb])


def q8_ws_views(ws, B, Hq, Hkv, N, d):
    """Views of the 8-bit attention workspace after block_sparse_attn with an 8-bit precision: q8
    (B,Hq,N,d) and k8 (B,Hkv,N,d) e4m3 codes (uint8), v8 (B,Hkv,d,npad) channel-major e4m3 codes
    (meaningful after SPARGE_PRECISION_Q8_FP8PV), sq (B,Hq,nqb), sk (B,Hkv,nkb), kmean (B,Hkv,d),
    sv (B,Hkv,d), following the layout the library writes (regions 256-byte aligned)."""
    torch = _torch()
    nqb, nkb = n_blocks(N)
    npad = -(-N // 64) * 64
    u8 = ws if ws.dtype == torch.uint8 else ws.view(torch.uint8)

    def take(off, nbytes):
        return u8[off:off + nbytes], off + ((nbytes + 255) // 256) * 256

    off = 0
    q8, off = take(off, B * Hq * N * d)
    k8, off = take(off, B * Hkv * N * d)
    v8, _ = take(off, B * Hkv * d * npad)
    _, off = take(off, max(B * Hkv * d * npad, 2 * B * Hkv * N * d))
    sq, off = take(off, 4 * B * Hq * nqb)
    sk, off = take(off, 4 * B * Hkv * nkb)
    km, off = take(off, 4 * B * Hkv * d)
    sv, off = take(off, 4 * B * Hkv * d)
    f = lambda t: t.view(torch.float32)
    return dict(q8=q8.view(B, Hq, N, d), k8=k8.view(B, Hkv, N, d), v8=v8.view(B, Hkv, d, npad),
                sq=f(sq).view(B, Hq, nqb), sk=f(sk).view(B, Hkv, nkb), kmean=f(km).view(B, Hkv, d),
                sv=f(sv).view(B, Hkv, d))


def block_sparse_attn(q, k, v, mask=None, lam: float = -math.inf, causal: bool = False, out=None, stats=None,
                      precision: int = SPARGE_PRECISION_BF16, ws=None):
    """Stage 2: attention over the kept 128x64 tiles with the lambda warp filter.
    precision SPARGE_PRECISION_Q8 (e4m3 Q.K^T, f16 P.V), SPARGE_PRECISION_Q8_FP8PV (both
    products e4m3) or SPARGE_PRECISION_BF16_FP8PV (bf16 Q.K^T, e4m3 P.V) runs an 8-bit path
    (d = 128); its workspace then holds the quantised copies and scales (see q8_ws_views)."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    op = SPARGE_OP_BLOCK_SPARSE_ATTN_Q8 if precision in PRECISIONS_8BIT \
        else SPARGE_OP_BLOCK_SPARSE_ATTN
    ws = _workspace(op, q, k, ws)
    dq, dk, dv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    mp = 0 if mask is None else mask.data_ptr()
    sp = 0 if stats is None else stats.data_ptr()
    _check(lib().sparge_block_sparse_attn(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), mp, float(lam),
                                          int(causal), int(precision), ctypes.byref(do), ws.data_ptr(), ws.numel(),
                                          sp, _stream()))
    return out


def sparge_attn(q, k, v, topk: float = 0.5, causal: bool = False, out=None, ws=None):
    """The plug-and-play call: predicted mask (theta 0.5) then block-sparse attention."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    ws = _workspace(SPARGE_OP_ATTN, q, k, ws)
    dq, dk, dv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    _check(lib().sparge_attn(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), float(topk), int(causal),
                             ctypes.byref(do), ws.data_ptr(), ws.numel(), _stream()))
    return out


def _head_array(x, name):
    """A per-head parameter array as a device pointer (0 for None); x is a float32 CUDA tensor."""
    if x is None:
        return 0
    torch = _torch()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32 and x.dim() == 1
            and x.is_contiguous()):
        raise TypeError("%s must be a contiguous float32 CUDA tensor of Hq entries" % name)
    return x.data_ptr()


def _order_ptr(order):
    """A token order as a device pointer (0 for None); order is an int32 CUDA tensor of N entries."""
    if order is None:
        return 0
    torch = _torch()
    if not (isinstance(order, torch.Tensor) and order.is_cuda and order.dtype == torch.int32 and order.dim() == 1
            and order.is_contiguous()):
        raise TypeError("token_order must be a contiguous int32 CUDA tensor of N entries")
    return order.data_ptr()


def _params(theta, lam, scale, precision, stats, events, topk_h=None, theta_h=None, lam_h=None, order=None,
            topk_mode=0, topp=1.0):
    """A sparge_params; `events` (6 torch.cuda.Event or None) are passed as cudaEvent_t handles.
    The handle array is kept on the returned struct so it outlives the call.  topk_h, theta_h and
    lam_h are optional per-query-head float32 CUDA tensors; order an optional int32 token order."""
    evp = None
    if events is not None:
        assert len(events) == 6
        for ev in events:
            if not ev.cuda_event:
                ev.record()   # torch creates the event on its first record
        evp = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
    p = sparge_params(float(theta), float(lam), float(scale), int(precision),
                      0 if stats is None else stats.data_ptr(),
                      ctypes.cast(evp, ctypes.c_void_p) if evp is not None else None,
                      _head_array(topk_h, "topk_per_head"), _head_array(theta_h, "theta_per_head"),
                      _head_array(lam_h, "lambda_per_head"), _order_ptr(order), int(topk_mode), float(topp))
    p._evp = evp
    p._arrays = (topk_h, theta_h, lam_h, order)
    return p


def block_sparse_attn_ex(q, k, v, mask=None, causal: bool = False, lam: float = -math.inf, scale: float = 0.0,
                         precision: int = SPARGE_PRECISION_BF16, stats=None, out=None, ws=None, events=None,
                         lambda_per_head=None, token_order=None):
    """block_sparse_attn with an explicit scale, optional timing events (6 torch.cuda.Event:
    [0] before the V copy or quantisation, [4] after it, [5] after the attention kernel) and an
    optional per-query-head lambda (float32 CUDA tensor of Hq entries) and an optional token order
    (int32 CUDA tensor of N entries; the mask then refers to the reordered sequence and the output
    comes back in the original order)."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    op = SPARGE_OP_BLOCK_SPARSE_ATTN_Q8 if precision in PRECISIONS_8BIT \
        else SPARGE_OP_BLOCK_SPARSE_ATTN
    ws = _workspace(op | (SPARGE_OP_TOKEN_ORDER if token_order is not None else 0), q, k, ws)
    p = _params(0.5, lam, scale, precision, stats, events, lam_h=lambda_per_head, order=token_order)
    dq, dk, dv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    mp = 0 if mask is None else mask.data_ptr()
    _check(lib().sparge_block_sparse_attn_ex(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), mp, int(causal),
                                             ctypes.byref(p), ctypes.byref(do), ws.data_ptr(), ws.numel(), _stream()))
    return out


def sparge_attn_ex(q, k, v, topk: float, causal: bool, theta: float = 0.5, lam: float = -math.inf,
                   scale: float = 0.0, precision: int = SPARGE_PRECISION_BF16, stats=None, mask_out=None,
                   out=None, ws=None, events=None, topk_per_head=None, theta_per_head=None, lambda_per_head=None,
                   token_order=None, topk_mode: int = SPARGE_TOPK_CUMULATIVE, topp: float = 1.0):
    """sparge_attn with explicit theta, lambda, scale, counters, an optional mask output,
    optional timing events (6 torch.cuda.Event, recorded around the five kernels), optional
    per-query-head topk, theta and lambda (float32 CUDA tensors of Hq entries) and an optional
    token order (int32 CUDA tensor of N entries: blocks and mask_out refer to the reordered
    sequence, the output comes back in the original order)."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    q8 = precision in PRECISIONS_8BIT
    ws = _workspace((SPARGE_OP_ATTN_Q8 if q8 else SPARGE_OP_ATTN) | (SPARGE_OP_TOKEN_ORDER if token_order is not None else 0),
                    q, k, ws)
    p = _params(theta, lam, scale, precision, stats, events, topk_per_head, theta_per_head, lambda_per_head,
                token_order, topk_mode, topp)
    dq, dk, dv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    mp = 0 if mask_out is None else mask_out.data_ptr()
    _check(lib().sparge_attn_ex(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), float(topk), int(causal),
                                ctypes.byref(p), ctypes.byref(do), mp, ws.data_ptr(), ws.numel(), _stream()))
    return out


def permute_tokens(x, perm, out=None):
    """y[:, :, t] = x[:, :, perm[t]] (perm: int32 CUDA tensor)."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(x)
    dx, dy = _desc(x), _desc(out)
    _check(lib().sparge_permute_tokens(ctypes.byref(dx), perm.data_ptr(), ctypes.byref(dy), _stream()))
    return out


def unpermute_tokens(x, perm, out=None):
    """y[:, :, perm[t]] = x[:, :, t]."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(x)
    dx, dy = _desc(x), _desc(out)
    _check(lib().sparge_unpermute_tokens(ctypes.byref(dx), perm.data_ptr(), ctypes.byref(dy), _stream()))
    return out


def hilbert_perm_2d(n_prefix: int, H: int, W: int) -> np.ndarray:
    out = np.empty(n_prefix + H * W, dtype=np.int32)
    _check(lib().sparge_hilbert_perm_2d(n_prefix, H, W, out.ctypes.data))
    return out


def hilbert_perm_3d(n_prefix: int, T: int, H: int, W: int) -> np.ndarray:
    out = np.empty(n_prefix + T * H * W, dtype=np.int32)
    _check(lib().sparge_hilbert_perm_3d(n_prefix, T, H, W, out.ctypes.data))
    return out


def selftest_bounded_wait(limit_ns: int = 50_000_000):
    """Enqueue the library's bounded-wait self test (a wait that is made to run out)."""
    _check(lib().sparge_selftest_bounded_wait(int(limit_ns), _stream()))


def device_status() -> int:
    """Reads and clears the library's device status word (0 = fine)."""
    return int(lib().sparge_get_device_status(_stream()))
