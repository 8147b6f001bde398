"""The allocation-free mask prediction entry point.

sparge_predict_mask_noalloc exists for callers that may not call cudaMalloc (a plug-in whose
host application owns the device memory, a loop that cannot take the synchronisation an
allocation may cause).  It must give exactly the mask of sparge_predict_mask, call after call,
although its scratch array keeps whatever the previous call left in it.  This file is collected
last so that a run stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
import workloads as W
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


def _noalloc_mask(q, k, topk, theta, causal):
    B, Hq, N, d = q.shape
    nqb, nkb = fbs.n_blocks(N)
    mask = torch.full((B, Hq, nqb, nkb), 7, dtype=torch.uint8, device=q.device)
    dq, dk = fbs._desc(q), fbs._desc(k)
    rc = fbs.lib().sparge_predict_mask_noalloc(ctypes.byref(dq), ctypes.byref(dk), float(topk), float(theta),
                                               int(causal), mask.data_ptr(), fbs._stream())
    assert rc == fbs.SPARGE_OK, fbs.lib().sparge_last_error()
    return mask


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [W.make_config("llama32k", N=4096 + 200, Hq=8, Hkv=2), W.make_config("tiny")]
    for w in cases:   # two calls in a row, on different shapes: stale scratch must not matter
        q, k = dev_bf16(w.q), dev_bf16(w.k)
        got = _noalloc_mask(q, k, w.topk, w.theta, w.causal)
        ref = fbs.predict_mask(q, k, w.topk, w.theta, w.causal)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)   # integer output: bit-exact
        assert int(got.max()) <= 1
    again = _noalloc_mask(dev_bf16(cases[0].q), dev_bf16(cases[0].k), cases[0].topk, cases[0].theta, True)
    ref0 = fbs.predict_mask(dev_bf16(cases[0].q), dev_bf16(cases[0].k), cases[0].topk, cases[0].theta, True)
    assert torch.equal(again, ref0)
    assert fbs.device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    w = W.describe("llama128k")
    need = fbs.workspace_bytes(fbs.SPARGE_OP_PREDICT_MASK, w.B, w.Hq, w.Hkv, w.N, w.d)
    assert need > (8 << 20)
    q = torch.empty((w.B, w.Hq, w.N, w.d), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((w.B, w.Hkv, w.N, w.d), dtype=torch.bfloat16, device="cuda")
    mask = torch.zeros((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    dq, dk = fbs._desc(q), fbs._desc(k)
    rc = fbs.lib().sparge_predict_mask_noalloc(ctypes.byref(dq), ctypes.byref(dk), 0.5, 0.5, 1, mask.data_ptr(),
                                               fbs._stream())
    assert rc == fbs.SPARGE_ERR_UNSUPPORTED
    assert b"scratch" in fbs.lib().sparge_last_error()
    torch.cuda.synchronize()
    assert int(mask.max()) == 0   # nothing was enqueued
