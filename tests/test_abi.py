"""The C-ABI library without a GPU: it loads, exports every call include/sparge.h declares,
and its host-only parts (workspace sizes, argument validation that fails before any CUDA call,
Hilbert permutation builders) behave as documented."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import free_block_sparse_gb300 as fbs
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fbs.LIB_PATH):
        from free_block_sparse_gb300 import build
        build.build()
    return fbs.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(sparge_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "sparge_attn" in names and "sparge_predict_mask" in names and "sparge_block_sparse_attn" in names
    for n in names:
        assert hasattr(lib, n), n
    assert names <= set(fbs.EXPORTS)


def test_struct_layouts_match_the_header(tmp_path):
    """The binding's ctypes structs have the sizes and field offsets the C compiler gives the
    header's structs."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"sparge.h\"\n"
        "int main(void) {\n"
        "  printf(\"%zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(sparge_params), offsetof(sparge_params, stats),\n"
        "         offsetof(sparge_params, timing_events), offsetof(sparge_params, topk_per_head),\n"
        "         offsetof(sparge_params, theta_per_head), offsetof(sparge_params, lambda_per_head),\n"
        "         offsetof(sparge_params, token_order), offsetof(sparge_params, topk_mode));\n"
        "  printf(\"%zu\\n\", offsetof(sparge_params, topp));\n"
        "  printf(\"%zu %zu %zu\\n\", sizeof(sparge_tensor), offsetof(sparge_tensor, B),\n"
        "         offsetof(sparge_tensor, stride_n));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P, T = fbs.sparge_params, fbs.sparge_tensor
    want = [ctypes.sizeof(P), P.stats.offset, P.timing_events.offset, P.topk_per_head.offset,
            P.theta_per_head.offset, P.lambda_per_head.offset, P.token_order.offset, P.topk_mode.offset,
            P.topp.offset, ctypes.sizeof(T), T.B.offset,
            T.stride_n.offset]
    assert got == want


@pytest.mark.parametrize("case", ["null_params", "bad_topk", "bad_theta", "neg_scale", "bad_mode", "bad_topp",
                                  "nan_topp"])
def test_predict_mask_ex_rejects_bad_parameters(lib, case):
    q = _t()
    p = fbs.sparge_params(0.5, -math.inf, 0.0, fbs.SPARGE_PRECISION_BF16, 0, None)
    topk = 0.5
    if case == "bad_mode":
        p.topk_mode = 7
    if case in ("bad_topp", "nan_topp"):
        p.topk_mode = fbs.SPARGE_TOPK_HYBRID
        p.topp = 0.0 if case == "bad_topp" else math.nan
    if case == "bad_topk":
        topk = 1.5
    elif case == "bad_theta":
        p.theta = math.nan
    elif case == "neg_scale":
        p.scale = -1.0
    pp = None if case == "null_params" else ctypes.byref(p)
    rc = lib.sparge_predict_mask_ex(ctypes.byref(q), ctypes.byref(q), topk, 0, pp, None, None, 0, None)
    assert rc == fbs.SPARGE_ERR_INVALID_ARG, lib.sparge_last_error()


def test_workspace_bytes(lib):
    B, Hq, Hkv, N, d = 1, 32, 8, 131072, 128
    nqb, nkb = 1024, 2048
    pred = fbs.workspace_bytes(fbs.SPARGE_OP_PREDICT_MASK, B, Hq, Hkv, N, d)
    assert pred >= 4 * (Hq * nqb * d + Hq * nqb + Hkv * d * nkb + Hkv * nkb)
    full = fbs.workspace_bytes(fbs.SPARGE_OP_ATTN, B, Hq, Hkv, N, d)
    attn = fbs.workspace_bytes(fbs.SPARGE_OP_BLOCK_SPARSE_ATTN, B, Hq, Hkv, N, d)
    assert attn >= 2 * B * Hkv * N * d
    assert full >= pred + Hq * nqb * nkb + attn
    assert fbs.workspace_bytes(fbs.SPARGE_OP_ATTN, B, Hq, Hkv, N, 96) == 0
    # 8-bit path: e4m3 copies of Q, K and V (V keys padded to 64) plus fp32 scales; d = 128 only
    q8 = fbs.workspace_bytes(fbs.SPARGE_OP_BLOCK_SPARSE_ATTN_Q8, B, Hq, Hkv, N, d)
    assert q8 >= B * (Hq + 2 * Hkv) * N * d + 4 * B * (Hq * nqb + Hkv * nkb + 2 * Hkv * d)
    assert fbs.workspace_bytes(fbs.SPARGE_OP_ATTN_Q8, B, Hq, Hkv, N, d) >= pred + Hq * nqb * nkb + q8
    assert fbs.workspace_bytes(fbs.SPARGE_OP_BLOCK_SPARSE_ATTN_Q8, B, Hq, Hkv, N, 64) == 0
    assert fbs.workspace_bytes(fbs.SPARGE_OP_ATTN_Q8, B, Hq, Hkv, N, 64) == 0
    # with a token order: the op's bytes plus bf16 copies of Q and K
    for op in (fbs.SPARGE_OP_PREDICT_MASK, fbs.SPARGE_OP_BLOCK_SPARSE_ATTN, fbs.SPARGE_OP_ATTN,
               fbs.SPARGE_OP_BLOCK_SPARSE_ATTN_Q8, fbs.SPARGE_OP_ATTN_Q8):
        base = fbs.workspace_bytes(op, B, Hq, Hkv, N, d)
        assert fbs.workspace_bytes(op | fbs.SPARGE_OP_TOKEN_ORDER, B, Hq, Hkv, N, d) == base + 2 * B * (Hq + Hkv) * N * d
    assert fbs.workspace_bytes(fbs.SPARGE_OP_ATTN_Q8 | fbs.SPARGE_OP_TOKEN_ORDER, B, Hq, Hkv, N, 64) == 0
    assert fbs.workspace_bytes(0x200 | fbs.SPARGE_OP_ATTN, B, Hq, Hkv, N, d) == 0


def _t(ptr=0x1000, B=1, H=2, N=256, d=64, dtype=fbs.SPARGE_BF16, sb=None, sh=None, sn=None):
    sn = d if sn is None else sn
    sh = N * sn if sh is None else sh
    sb = H * sh if sb is None else sb
    return fbs.sparge_tensor(ptr, dtype, 0, B, H, N, d, sb, sh, sn)


@pytest.mark.parametrize("case,code", [
    ("null_q", fbs.SPARGE_ERR_INVALID_ARG),
    ("bad_d", fbs.SPARGE_ERR_UNSUPPORTED),
    ("bad_dtype", fbs.SPARGE_ERR_UNSUPPORTED),
    ("gqa_ratio", fbs.SPARGE_ERR_UNSUPPORTED),
    ("topk_zero", fbs.SPARGE_ERR_INVALID_ARG),
    ("topk_nan", fbs.SPARGE_ERR_INVALID_ARG),
    ("topk_big", fbs.SPARGE_ERR_INVALID_ARG),
    ("theta_nan", fbs.SPARGE_ERR_INVALID_ARG),
    ("stride", fbs.SPARGE_ERR_INVALID_ARG),
    ("misaligned", fbs.SPARGE_ERR_INVALID_ARG),
    ("null_mask", fbs.SPARGE_ERR_INVALID_ARG),
    ("small_ws", fbs.SPARGE_ERR_WORKSPACE_TOO_SMALL),
    ("too_long", fbs.SPARGE_ERR_UNSUPPORTED),
])
def test_predict_mask_rejects_bad_arguments(lib, case, code):
    q, k = _t(), _t()
    topk, theta, mask, ws, wsb = 0.5, 0.5, 0x2000, 0x3000, 1 << 30
    if case == "null_q":
        rc = lib.sparge_predict_mask(None, ctypes.byref(k), topk, theta, 0, mask, ws, wsb, None)
        assert rc == code and b"NULL" in lib.sparge_last_error()
        return
    if case == "bad_d":
        q, k = _t(d=96), _t(d=96)
    elif case == "bad_dtype":
        q = _t(dtype=7)
    elif case == "gqa_ratio":
        q, k = _t(H=3), _t(H=2)
    elif case == "topk_zero":
        topk = 0.0
    elif case == "topk_nan":
        topk = math.nan
    elif case == "topk_big":
        topk = 1.5
    elif case == "theta_nan":
        theta = math.nan
    elif case == "stride":
        q = _t(sn=65)
    elif case == "misaligned":
        q = _t(ptr=0x1002)
    elif case == "null_mask":
        mask = None
    elif case == "small_ws":
        wsb = 16
    elif case == "too_long":
        q, k = _t(N=131073), _t(N=131073)
    rc = lib.sparge_predict_mask(ctypes.byref(q), ctypes.byref(k), topk, theta, 0, mask, ws, wsb, None)
    assert rc == code, lib.sparge_last_error()
    assert lib.sparge_last_error()


@pytest.mark.parametrize("lam", [0.5, math.nan])
def test_attention_rejects_bad_lambda(lib, lam):
    q = _t()
    rc = lib.sparge_block_sparse_attn(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), None, lam, 0, 0,
                                      ctypes.byref(q), None, 0, None, None)
    assert rc == fbs.SPARGE_ERR_INVALID_ARG


@pytest.mark.parametrize("case", ["null_params", "bad_lambda", "neg_scale", "inf_scale", "q8_d64"])
def test_block_sparse_ex_rejects_bad_parameters(lib, case):
    q = _t()
    p = fbs.sparge_params(0.5, -math.inf, 0.0, fbs.SPARGE_PRECISION_BF16, 0, None)
    code = fbs.SPARGE_ERR_INVALID_ARG
    if case == "bad_lambda":
        p.lambda_ = 1.0
    elif case == "neg_scale":
        p.scale = -1.0
    elif case == "inf_scale":
        p.scale = math.inf
    elif case == "q8_d64":
        p.precision = fbs.SPARGE_PRECISION_Q8
        code = fbs.SPARGE_ERR_UNSUPPORTED
    pp = None if case == "null_params" else ctypes.byref(p)
    rc = lib.sparge_block_sparse_attn_ex(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), None, 0, pp,
                                         ctypes.byref(q), None, 0, None)
    assert rc == code, lib.sparge_last_error()


def test_short_query_checks(lib):
    """Causal attention needs Nq <= Nk; a token order needs Nq = Nk (checked before any CUDA call)."""
    q, k = _t(N=512), _t(N=256)
    rc = lib.sparge_predict_mask(ctypes.byref(q), ctypes.byref(k), 0.5, 0.5, 1, ctypes.c_void_p(0x2000), None, 0, None)
    assert rc == fbs.SPARGE_ERR_INVALID_ARG and b"Nq <= Nk" in lib.sparge_last_error()
    p = fbs.sparge_params(0.5, -math.inf, 0.0, fbs.SPARGE_PRECISION_BF16, 0, None)
    p.token_order = 0x3000
    q2 = _t(N=128)
    rc = lib.sparge_attn_ex(ctypes.byref(q2), ctypes.byref(k), ctypes.byref(k), 0.5, 1, ctypes.byref(p),
                            ctypes.byref(q2), None, None, 0, None)
    assert rc == fbs.SPARGE_ERR_UNSUPPORTED and b"token order" in lib.sparge_last_error()


def test_attention_rejects_mismatched_output(lib):
    q, o = _t(), _t(H=4)
    rc = lib.sparge_block_sparse_attn(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), None, -math.inf, 0, 0,
                                      ctypes.byref(o), None, 0, None, None)
    assert rc == fbs.SPARGE_ERR_INVALID_ARG
    rc = lib.sparge_block_sparse_attn(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), None, -math.inf, 0,
                                      fbs.SPARGE_PRECISION_Q8, ctypes.byref(q), None, 0, None, None)
    assert rc == fbs.SPARGE_ERR_UNSUPPORTED


@pytest.mark.parametrize("n_prefix,H,W", [(0, 1, 1), (5, 8, 8), (512, 64, 64), (3, 7, 13), (0, 30, 45)])
def test_hilbert_2d_matches_oracle(lib, n_prefix, H, W):
    np.testing.assert_array_equal(fbs.hilbert_perm_2d(n_prefix, H, W), oracle.hilbert_perm_2d(n_prefix, H, W))


@pytest.mark.parametrize("n_prefix,T,H,W", [(0, 2, 2, 2), (3, 3, 5, 6), (0, 8, 8, 8), (226, 13, 30, 45)])
def test_hilbert_3d_matches_oracle(lib, n_prefix, T, H, W):
    np.testing.assert_array_equal(fbs.hilbert_perm_3d(n_prefix, T, H, W),
                                  oracle.hilbert_perm_3d(n_prefix, T, H, W))


def test_hilbert_rejects_bad_arguments(lib):
    assert lib.sparge_hilbert_perm_2d(0, 0, 4, None) == fbs.SPARGE_ERR_INVALID_ARG
    assert lib.sparge_hilbert_perm_3d(-1, 2, 2, 2, None) == fbs.SPARGE_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fbs.sparge_attn(x, x, x)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,precision", [
    (1, 32, 8, 1, 131072, 128, 1, fbs.SPARGE_PRECISION_BF16),       # a decoding step: row scores, lists
    (1, 32, 8, 131072, 131072, 128, 1, fbs.SPARGE_PRECISION_BF16),  # the 128K prefill
    (2, 16, 4, 16, 40000, 64, 1, fbs.SPARGE_PRECISION_BF16),
    (1, 76, 76, 16384, 16385, 64, 0, fbs.SPARGE_PRECISION_BF16),   # score splits on one side of a group
    (1, 76, 76, 16385, 16384, 64, 0, fbs.SPARGE_PRECISION_BF16),
    (3, 8, 2, 300, 20000, 128, 1, fbs.SPARGE_PRECISION_BF16_FP8PV),
    (1, 4, 1, 7000, 900, 128, 0, fbs.SPARGE_PRECISION_Q8),
    (8, 32, 8, 1, 32768, 128, 1, fbs.SPARGE_PRECISION_BF16),
])
def test_public_workspace_size_covers_every_shorter_query(lib, B, Hq, Hkv, Nq, Nk, d, causal, precision):
    """sparge_workspace_bytes for N = max(Nq, Nk) is enough for sparge_attn_ex on (Nq, Nk): the
    call passes its workspace check and stops at the next check (an unknown topk_mode), before
    anything is enqueued; 16 bytes fail the workspace check."""
    q8 = precision in fbs.PRECISIONS_8BIT
    op = fbs.SPARGE_OP_ATTN_Q8 if q8 else fbs.SPARGE_OP_ATTN
    wsb = fbs.workspace_bytes(op, B, Hq, Hkv, max(Nq, Nk), d)
    assert wsb > 0
    q, o = _t(B=B, H=Hq, N=Nq, d=d), _t(B=B, H=Hq, N=Nq, d=d)
    k = _t(B=B, H=Hkv, N=Nk, d=d)
    p = fbs.sparge_params(0.5, -math.inf, 0.0, precision, 0, None)
    p.topk_mode = 99
    for size, code in ((wsb, fbs.SPARGE_ERR_INVALID_ARG), (16, fbs.SPARGE_ERR_WORKSPACE_TOO_SMALL)):
        rc = lib.sparge_attn_ex(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), 0.5, causal, ctypes.byref(p),
                                ctypes.byref(o), None, 0x100000, size, None)
        err = lib.sparge_last_error()
        assert rc == code, (size, err)
        if code == fbs.SPARGE_ERR_INVALID_ARG:
            assert b"topk_mode" in err, err


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 32, 8, 1, 131072, 128, 1),     # decoding tiles: partial rows, lists and counts
    (2, 16, 2, 16, 8192, 128, 1),
    (1, 8, 1, 12, 5000, 64, 1),
    (1, 24, 24, 4608, 4608, 128, 0),
])
def test_public_workspace_size_covers_block_sparse_attention(lib, B, Hq, Hkv, Nq, Nk, d, causal):
    """The same for the block-sparse call alone (the decoding tiles' workspace included): with the
    public size the call passes its workspace-size check and stops at the workspace alignment
    check (a deliberately misaligned pointer), before anything is enqueued."""
    wsb = fbs.workspace_bytes(fbs.SPARGE_OP_BLOCK_SPARSE_ATTN, B, Hq, Hkv, max(Nq, Nk), d)
    q, o = _t(B=B, H=Hq, N=Nq, d=d), _t(B=B, H=Hq, N=Nq, d=d)
    k = _t(B=B, H=Hkv, N=Nk, d=d)
    p = fbs.sparge_params(0.5, -math.inf, 0.0, fbs.SPARGE_PRECISION_BF16, 0, None)
    for size, code, word in ((wsb, fbs.SPARGE_ERR_INVALID_ARG, b"aligned"), (16, fbs.SPARGE_ERR_WORKSPACE_TOO_SMALL, b"need")):
        rc = lib.sparge_block_sparse_attn_ex(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), 0x2000, causal,
                                             ctypes.byref(p), ctypes.byref(o), 0x100010, size, None)
        err = lib.sparge_last_error()
        assert rc == code and word in err, (size, err)
