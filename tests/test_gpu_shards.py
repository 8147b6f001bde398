"""The (batch, key/value head) partition on the CUDA path: the library's calls on the views of
each unit give, bit for bit, the mask rows and output rows of one call on the whole tensors (what
each rank of a multi-GPU run computes is exactly its share of the single-GPU result)."""
import math

import numpy as np
import pytest
import torch

import free_block_sparse_gb300 as fbs
from free_block_sparse_gb300 import shards
import workloads as W
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 3])
def test_units_on_views_equal_the_whole_call(world):
    w = W.make_config("llama32k", B=2, Hq=8, Hkv=4, N=3000)
    q, k, v = dev_bf16(w.q), dev_bf16(w.k), dev_bf16(w.v)
    mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
    out = fbs.sparge_attn_ex(q, k, v, w.topk, w.causal, theta=w.theta, lam=w.lam, mask_out=mask)
    got_o = torch.zeros_like(out)
    got_m = torch.zeros_like(mask)
    for rank in range(world):
        for unit in shards.shard_units(w.B, w.Hkv, world, rank):
            b, hs, kvh = shards.unit_heads(unit, w.Hq, w.Hkv)
            m = torch.empty((1, hs.stop - hs.start, w.nqb, w.nkb), dtype=torch.uint8, device="cuda")
            o = fbs.sparge_attn_ex(q[b:b + 1, hs], k[b:b + 1, kvh:kvh + 1], v[b:b + 1, kvh:kvh + 1], w.topk, w.causal,
                                   theta=w.theta, lam=w.lam, mask_out=m)
            got_o[b:b + 1, hs] = o
            got_m[b:b + 1, hs] = m
    torch.cuda.synchronize()
    assert torch.equal(got_m, mask)
    assert torch.equal(got_o, out)
    assert fbs.device_status() == 0
