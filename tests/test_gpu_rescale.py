"""O rescaled on every tile: key scores climb by more than 8 (log2 units) from each 64-key block
to the next, so every new tile lifts the running maximum past the exponent reference and the
softmax warps rescale O in TMEM, waiting first for the P.V product of the previous tile while the
score products of later tiles are already in flight.  Dense (mask = None), ragged tail, GQA,
causal and not, both head sizes, against the float64 oracle."""
import math

import pytest

import free_block_sparse_gb300 as fbs
import oracle
import workloads as W
from gpu_util import COS_MIN, MAXABS, cos_maxabs, dev_bf16, f64, host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_on_every_tile(d, causal):
    qu, ku, vu = W.climbing_qkv(7, 1, 4, 2, 1280 - 17, d)
    out = fbs.block_sparse_attn(dev_bf16(qu), dev_bf16(ku), dev_bf16(vu), None, -math.inf, causal)
    ref = oracle.block_sparse_attn(f64(qu), f64(ku), f64(vu), None, -math.inf, causal)
    cos, err = cos_maxabs(host_f64(out), ref)
    assert cos >= COS_MIN and err <= MAXABS, (cos, err)
    assert fbs.device_status() == fbs.SPARGE_OK
