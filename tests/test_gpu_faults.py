"""Failure detection on the GPU without a fault: a bounded device wait is made to run out (the
barrier it waits on never gets an arrival), the kernel returns, the host reads the timeout from
the library's status word, and the context keeps working."""
import math

import pytest
import torch

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import COS_MIN, MAXABS, cos_maxabs, dev_bf16, f64, host_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    fbs.lib()
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_OK
    fbs.selftest_bounded_wait(50_000_000)  # 50 ms
    torch.cuda.synchronize()
    assert fbs.device_status() == fbs.SPARGE_ERR_DEVICE_TIMEOUT
    assert b"timed out" in fbs.lib().sparge_last_error()
    assert fbs.device_status() == fbs.SPARGE_OK   # reading clears the word
    qu, ku, vu = W.random_qkv(31, 1, 2, 2, 300, 64)
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, False)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, False)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS
    assert fbs.device_status() == fbs.SPARGE_OK
