#!/usr/bin/env python3
"""Benchmark of the SpargeAttn hot path on one GB300: mask prediction (pooling + similarity,
pooled scores + softmax + cumulative top-k) followed by block-sparse attention with the lambda
filter, on the Llama-3.1-8B-like causal prefill at 128K tokens (B=1, 32 query heads, 8 KV heads,
d=128, topk 0.5, theta 0.5, lambda -8; synthetic bf16 inputs).

One step = one sparge_attn_ex call (five kernel launches: pooling, pooled-score GEMM, selection,
V to f16, attention) over inputs resident in HBM; CUDA events recorded by the library around each kernel
give the per-kernel times.
Prints one JSON line.  ``--impl reference`` times the float64 CPU oracle instead, on a bounded
sample of the same workload.  Under torchrun every rank runs its own full replica (weak scaling,
no collective on the data path); timings are reduced with a max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


# ------------------------------------------------------------------------------------------------
# CPU oracle sample (reference arm and cpu_baseline)
# ------------------------------------------------------------------------------------------------
def _oracle_sample_job(args):
    q_blocks, k_head, v_head, idx, N, d, topk, theta, lam, causal, mask_rows = args
    import oracle as O
    t0 = time.perf_counter()
    rows = 0
    for n, (qb, i) in enumerate(zip(q_blocks, idx)):
        if mask_rows is None:   # predicted mask row, then attention
            pr = O.predict_mask_row(qb, k_head, i, topk, theta, causal)
            kept = np.nonzero(pr["mask"])[0]
        else:                   # the workload's own mask row
            kept = np.nonzero(mask_rows[n])[0]
        O.attn_qblock(qb, k_head, v_head, i, kept, lam, causal, O.default_scale(d))
        rows += qb.shape[0]
    return time.perf_counter() - t0, rows


def oracle_sample(w, n_blocks_sample: int, workers: int):
    """Time the oracle on ``n_blocks_sample`` query blocks of head 0 spread over the sequence,
    in ``workers`` spawned processes (one BLAS thread each).  Each worker pools the whole key
    head itself (part of the timed work).  Returns (dense-equivalent TOPS, seconds, description)."""
    import multiprocessing as mp
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    N, d = w.N, w.d
    kh = W.bf16_to_f64(w.k[0, 0])
    vh = W.bf16_to_f64(w.v[0, 0])
    idx = np.linspace(0, w.nqb - 1, n_blocks_sample).round().astype(int)
    per = [idx[r::workers] for r in range(workers)]
    jobs = []
    for part in per:
        if len(part) == 0:
            continue
        qbs = [W.bf16_to_f64(w.q[0, 0, i * 128:min(N, i * 128 + 128)]) for i in part]
        mrows = None if w.mask is None else [w.mask[0, 0, i] for i in part]
        jobs.append((qbs, kh, vh, list(part), N, d, w.topk, w.theta, w.lam, w.causal, mrows))
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(len(jobs)) as pool:
        res = pool.map(_oracle_sample_job, jobs)
    wall = time.perf_counter() - t0
    rows = sum(r for _, r in res)
    tops = 4.0 * rows * N * d / wall / 1e12
    what = "mask row + attention each" if w.mask is None else "attention over the workload's mask row each"
    desc = ("%d query blocks (%d rows) of head 0 spread over the sequence, %s, "
            "%d processes x 1 BLAS thread, key/value head pooled per process" % (n_blocks_sample, rows, what, len(jobs)))
    return tops, wall, desc, len(jobs)


# ------------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        # the raw samples (nvidia-smi CSV); SPARGE_CLOCKS_CSV picks where they go
        self.path = os.environ.get("SPARGE_CLOCKS_CSV") or os.path.join(tempfile.gettempdir(), "sparge_clocks_bench.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# multi-rank bookkeeping (each rank runs its own replica; no collective on the data path)
# ------------------------------------------------------------------------------------------------
def max_over_ranks(seconds: float, dist=None, device=None) -> float:
    """The slowest rank's timed-region length (the job is done when every replica is done)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, dense_flops_per_step: float, steps: int, seconds: float) -> float:
    """Whole-job dense-equivalent TOPS: every rank processed `steps` full steps in `seconds`."""
    return world * dense_flops_per_step * steps / seconds / 1e12


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------
PRECISIONS = {  # name: (C enum, dtype label, Q.K^T peak ratio to bf16, P.V peak ratio to bf16)
    "bf16": (0, "bf16", 1.0, 1.0),
    "q8": (1, "e4m3 Q.K^T + f16 P.V", 2.0, 1.0),
    "fp8pv": (2, "e4m3", 2.0, 2.0),
    "bf16fp8pv": (3, "bf16 Q.K^T + e4m3 P.V", 1.0, 2.0),
}


def code_digest(paths) -> str:
    """sha256 (first 16 hex digits) of C++/CUDA sources with their comments and whitespace removed,
    so that a capture stays attached to the code it measured across edits of comments alone."""
    import re
    text = ""
    for p in paths:
        s = open(p).read()
        s = re.sub(r"/\*.*?\*/", " ", s, flags=re.S)
        s = re.sub(r"//[^\n]*", " ", s)
        text += " ".join(s.split()) + "\n"
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def profile_traffic(w, precision):
    """DRAM bytes of one full attention launch from the committed ncu capture of the same kernel
    (4 of the 32 query heads, scaled by 8), or None when the workload differs or the kernel source
    has changed since the capture."""
    if w.name != "llama128k" or precision != "bf16" or (w.Hq, w.Hkv) != (32, 8):
        return None
    sha = code_digest(os.path.join(ROOT, "free_block_sparse_gb300", "csrc", f) for f in ("bsattn.cu", "common.cuh"))
    path = os.path.join(ROOT, "profiles", "bsattn_llama128k_h4.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("code sha256 (bsattn.cu + common.cuh)") != sha:
        return None
    return int(fields["traffic per full launch (bytes)"])


def measure_permute(steps, warmup, dev, peaks):
    """The Hilbert token order of the video-like workload's shape (B 1, H 30, N 17776 = 226 text
    + 13 x 30 x 45 grid tokens, d 64): one step permutes q, k and v into curve order and
    unpermutes the output (four launches); eight 68 MB tensors, 546 MB in all, more than L2.
    Algorithmic bytes: each launch reads and writes every token row once (the 71 KB
    permutation is not counted)."""
    import torch
    import free_block_sparse_gb300 as fbs
    wd = W.describe("cogvideox")
    perm = torch.from_numpy(fbs.hilbert_perm_3d(wd.n_prefix, *wd.grid)).to(dev)
    g = torch.Generator(device=dev).manual_seed(11)
    xs = [torch.randn((wd.B, wd.Hq, wd.N, wd.d), generator=g, device=dev).to(torch.bfloat16) for _ in range(4)]
    ys = [torch.empty_like(x) for x in xs]

    def step():
        for i in range(3):
            fbs.permute_tokens(xs[i], perm, out=ys[i])
        fbs.unpermute_tokens(xs[3], perm, out=ys[3])

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    assert fbs.device_status() == 0
    t = e0.elapsed_time(e1) / 1e3 / steps
    nbytes = 4 * 2 * xs[0].numel() * 2
    gbs = nbytes / t / 1e9
    return {"workload": "cogvideox-like shape, q/k/v into Hilbert order + output back (B1 H30 N17776 d64)",
            "launches_per_step": 4, "ms": round(t * 1e3, 4), "bytes_per_step": nbytes, "gbs": round(gbs, 1),
            "pct_hbm": round(100 * gbs / float(peaks["hbm_gbs"]), 2)}


def measure_decode(q, k, w, steps, warmup, dev, peaks, v):
    """One decoding step of a causal workload: the last query token of every head against all the
    keys (mask prediction of that token, then the decoding tiles that pack the G query rows of a
    KV head into one tile and split the keys over CTAs), on the bench's own device tensors.  The
    lambda filter is off (the split over key chunks needs it off).  A decoding loop replays its
    step as a CUDA graph, so the step, the prediction alone and the attention alone are each timed
    as graph replays (device time without the host's launch work); `eager_ms` is the same step
    called directly.  Algorithmic bytes of the attention: a K and a V tile per key block that any
    head of a KV head keeps (counted by the kernel), the token's Q and O rows and the mask."""
    import torch
    import free_block_sparse_gb300 as fbs
    B, Hq, _, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    nkb = -(-Nk // 64)
    qd = q[:, :, -1:]
    mask = torch.empty((B, Hq, 1, nkb), dtype=torch.uint8, device=dev)
    ws = torch.empty(fbs.workspace_bytes(fbs.SPARGE_OP_ATTN, B, Hq, Hkv, Nk, d), dtype=torch.uint8, device=dev)
    o = torch.empty((B, Hq, 1, d), dtype=torch.bfloat16, device=dev)
    stats = torch.zeros(4, dtype=torch.int64, device=dev)
    s = torch.cuda.Stream(device=dev)

    def step(counters=None):
        fbs.sparge_attn_ex(qd, k, v, w.topk, True, theta=w.theta, lam=-math.inf, mask_out=mask, out=o, ws=ws,
                           stats=counters)

    def predict():
        fbs.predict_mask(qd, k, w.topk, w.theta, True, ws=ws, mask=mask)

    def attend():
        fbs.block_sparse_attn(qd, k, v, mask, -math.inf, True, out=o, ws=ws)

    def per_replay(fn):
        """Device time of one call of fn, replayed from a CUDA graph (median of `steps` replays)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        for _ in range(max(warmup, 3)):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for e0, e1 in evs:
            e0.record(s)
            g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3

    with torch.cuda.stream(s):
        step(counters=stats)
        torch.cuda.synchronize()
        tiles = int(stats[0].item())
        ref = o.clone()
        for _ in range(max(warmup, 3)):
            step()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for e0, e1 in evs:
            e0.record(s)
            step()
            e1.record(s)
        torch.cuda.synchronize()
        t_eager = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3
        t_step = per_replay(step)
        t_pred = per_replay(predict)
        t_attn = per_replay(attend)
    torch.cuda.synchronize()
    assert torch.equal(o, ref)
    assert fbs.device_status() == 0
    nbytes = tiles * 64 * d * 2 * 2 + 2 * 2 * B * Hq * d + mask.numel()
    gbs = nbytes / t_attn / 1e9
    return {"workload": "%s decoding step: the last query token of each of the %d heads against the %d keys, "
                        "predicted mask, lambda off; device times of CUDA-graph replays" % (w.name, Hq, Nk),
            "ms": round(t_step * 1e3, 4), "eager_ms": round(t_eager * 1e3, 4), "mask_pred_ms": round(t_pred * 1e3, 4),
            "attn_ms": round(t_attn * 1e3, 4), "kv_tiles": tiles, "attn_bytes": nbytes, "attn_gbs": round(gbs, 1),
            "attn_pct_hbm": round(100 * gbs / float(peaks["hbm_gbs"]), 2),
            "tokens_per_s": round(B / t_step, 1)}


def run_ours(args, rank, world, local_rank):
    import torch
    import free_block_sparse_gb300 as fbs

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    peaks = load_peaks()
    w = make_workload(args)
    dev = torch.device("cuda", local_rank)

    def to_dev(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = to_dev(w.q), to_dev(w.k), to_dev(w.v)
    o = torch.empty_like(q)
    prec, dtype_label, r_s, r_pv = PRECISIONS[args.precision]
    given_mask = w.mask is not None   # the custom-mask workload: the block-sparse call on its own mask
    lam = w.lam if args.lam is None else args.lam
    if given_mask:
        mask = torch.from_numpy(w.mask).to(dev)
        op = fbs.SPARGE_OP_BLOCK_SPARSE_ATTN if prec == 0 else fbs.SPARGE_OP_BLOCK_SPARSE_ATTN_Q8
    else:
        mask = torch.empty((w.B, w.Hq, w.nqb, w.nkb), dtype=torch.uint8, device=dev)
        op = fbs.SPARGE_OP_ATTN if prec == 0 else fbs.SPARGE_OP_ATTN_Q8
    ws = torch.empty(fbs.workspace_bytes(op, w.B, w.Hq, w.Hkv, w.N, w.d), dtype=torch.uint8, device=dev)
    stats = torch.zeros(4, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()
    # image / video workloads run in Hilbert token order, inside the call (sparge_params.token_order):
    # the call copies Q and K in that order, gathers V while converting it and writes each output
    # row back to its original position
    perm = None
    if w.grid is not None:
        perm_np = (fbs.hilbert_perm_2d(w.n_prefix, *w.grid) if len(w.grid) == 2
                   else fbs.hilbert_perm_3d(w.n_prefix, *w.grid))
        perm = torch.from_numpy(perm_np).to(dev)
        ws = torch.empty(fbs.workspace_bytes(op | fbs.SPARGE_OP_TOKEN_ORDER, w.B, w.Hq, w.Hkv, w.N, w.d),
                         dtype=torch.uint8, device=dev)

    def call(qq, kk, vv, events=None, counters=None, oo=None, outer=None):
        """One step through the public call; `outer` (2 events) brackets the whole call."""
        oo = o if oo is None else oo
        if outer is not None:
            outer[0].record(stream)
        if given_mask:
            fbs.block_sparse_attn_ex(qq, kk, vv, mask, w.causal, lam=lam, out=oo, ws=ws, precision=prec,
                                     stats=counters, events=events, token_order=perm)
        else:
            fbs.sparge_attn_ex(qq, kk, vv, w.topk, w.causal, theta=w.theta, lam=lam, mask_out=mask, out=oo, ws=ws,
                               precision=prec, events=events, stats=counters, token_order=perm)
        if outer is not None:
            outer[1].record(stream)

    # one run with counters for the executed-work figures (same inputs -> same mask every step)
    call(q, k, v, counters=stats)
    torch.cuda.synchronize()
    kept, pv, skipped, valid = (int(x) for x in stats.cpu().tolist())
    assert fbs.device_status() == 0

    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    # inputs smaller than twice L2 (129 MB): flush L2 between steps and sum the steps' own spans
    in_bytes = w.q.nbytes + w.k.nbytes + w.v.nbytes
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < 2 * 129e6 else None

    def step(events=None):
        call(q, k, v, events=None if events is None else events[:6], outer=None if events is None else events[6:])

    for evs in ev_sets:   # create every event once (torch creates events on first record)
        for ev in evs:
            ev.record(stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.5)
    for s in range(args.steps):
        if flush is not None:
            flush.zero_()    # evict the previous step's data from L2 (outside the step's own span)
        step(ev_sets[s])
    torch.cuda.synchronize()
    clk = clocks.stop()
    # per step: [0] before pooling, [1] after pooling, [2] after the score GEMM, [3] after selection,
    # [4] after the V copy (8-bit: quantisation), [5] after attention.  With the workload's own
    # mask there is no prediction: [0] and [4] bracket the V copy or quantisation.
    t_pool = [e[0].elapsed_time(e[1]) / 1e3 for e in ev_sets]
    t_gemm = [e[1].elapsed_time(e[2]) / 1e3 for e in ev_sets]
    t_sel = [e[2].elapsed_time(e[3]) / 1e3 for e in ev_sets]
    t_conv = [e[0 if given_mask else 3].elapsed_time(e[4]) / 1e3 for e in ev_sets]
    t_attn = [e[4].elapsed_time(e[5]) / 1e3 for e in ev_sets]
    t_pred = [0.0 if given_mask else a + b + c for a, b, c in zip(t_pool, t_gemm, t_sel)]
    # [6] before the call and [7] after it: with a token order, [6]-[0] holds the ordered copies of Q and K
    t_perm = [e[6].elapsed_time(e[0]) / 1e3 + e[5].elapsed_time(e[7]) / 1e3 for e in ev_sets] if perm is not None else None
    first, last = 6, 7
    if flush is None:
        total = ev_sets[0][first].elapsed_time(ev_sets[-1][last]) / 1e3
    else:
        total = sum(e[first].elapsed_time(e[last]) for e in ev_sets) / 1e3
    total = max_over_ranks(total, dist, dev)
    assert fbs.device_status() == 0

    # end to end through the public call: every step copies its inputs in from pinned host memory
    # and its output back.  Two device buffer sets and two copy streams pipeline the steps: the
    # inputs of step s + 1 go in and the output of step s - 1 comes back while step s computes.
    hq = q.cpu().pin_memory()
    hk = k.cpu().pin_memory()
    hv = v.cpu().pin_memory()
    ho = [torch.empty_like(hq).pin_memory() for _ in range(2)]
    dqkv = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]
    dout = [torch.empty_like(o) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]      # inputs of a set copied in
    in_free = [ev(), ev()]       # the compute that read a set's inputs has finished
    out_ready = [ev(), ev()]     # a set's output written
    out_free = [ev(), ev()]      # a set's output copied back
    for e in in_free + out_free:
        e.record(stream)

    def e2e_step(i):
        b = i % 2
        dq, dk, dv = dqkv[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[b])
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])
        call(dq, dk, dv, oo=dout[b])
        in_free[b].record(stream)
        out_ready[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            ho[b].copy_(dout[b], non_blocking=True)
            out_free[b].record(s_out)

    # as many steps as the device-timed region: the first copy in and the last copy back are the
    # pipeline's fill and drain, inside the timed region and spread over the steps
    e2e_steps = max(4, args.steps)
    e2e_step(0)
    e2e_step(1)
    torch.cuda.synchronize()
    e2e_clocks = ClockSampler(local_rank)   # the clocks of this region too (copies and compute together)
    e2e_clocks.start()
    time.sleep(0.5)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(s_in)              # before the first copy in
    s_in.wait_event(a0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    a1.record(stream)            # after the last copy back
    torch.cuda.synchronize()
    e2e_clk = e2e_clocks.stop()
    e2e_t = a0.elapsed_time(a1) / 1e3 / e2e_steps
    for b in range(2):
        assert torch.equal(ho[b], o.cpu())

    dense = w.dense_flops()
    ms_step = total / args.steps * 1e3
    value = job_value(world, dense, args.steps, total)
    avg = lambda xs: sum(xs) / len(xs)
    t_attn_avg, t_pred_avg = avg(t_attn), avg(t_pred)
    tile_flops = 2.0 * 128 * 64 * w.d
    executed = (kept + pv) * tile_flops
    attn_tflops = executed / t_attn_avg / 1e12
    # The attention kernel runs for milliseconds inside a short timed region.  When its SM clock
    # held the maximum (median of the samples taken during the timed steps), the burst bf16 figure
    # (cuBLAS timed alone, at full clock) is its peak; otherwise the sustained one (cuBLAS in a
    # seconds-long loop under the power cap).  Both fractions are reported.
    burst, sustained = float(peaks["bf16_tflops"]), float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    at_max = (clk.get("sm_mhz") is not None and clk.get("sm_max_mhz") and
              clk["sm_mhz"] >= 0.97 * float(clk["sm_max_mhz"]))
    peak_bf16 = burst if at_max else sustained

    def mix_peak(p_bf16):
        # the peak of the executed mix: Q.K^T work at r_s x and P.V work at r_pv x the bf16 rate
        # (e4m3 = 2 x bf16, the nominal dense ratio 4.5 / 2.25 PFLOP/s)
        return executed / (kept * tile_flops / (r_s * p_bf16) + pv * tile_flops / (r_pv * p_bf16)) if kept else p_bf16

    peak_tc = mix_peak(peak_bf16)
    pred_bytes = (w.q.nbytes + w.k.nbytes + mask.numel())
    pred_gbs = pred_bytes / t_pred_avg / 1e9 if t_pred_avg > 0 else 0.0
    hbm = float(peaks["hbm_gbs"])
    tag = "of measured" if peaks.get("source") == "measured" else "of fallback"

    kernels_ms = ({"attn_prep": round(avg(t_conv) * 1e3, 4), "bsattn": round(t_attn_avg * 1e3, 4)} if given_mask else
                  {"pool_sim": round(avg(t_pool) * 1e3, 4), "score_gemm": round(avg(t_gemm) * 1e3, 4),
                   "score_select": round(avg(t_sel) * 1e3, 4),
                   "attn_prep": round(avg(t_conv) * 1e3, 4), "bsattn": round(t_attn_avg * 1e3, 4)})
    # under a token order the mask prediction's pooling writes the ordered copies of Q and K that the
    # attention reads (no copy launch); a call on a given mask copies them in separate launches (K,
    # and Q where TMA or the 8-bit quantiser reads it)
    order_copies = 0 if (perm is None or not given_mask) else (2 if (w.d != 64 or args.precision != "bf16") else 1)
    if t_perm is not None:
        # the time between the call's outer events and its first / after its last kernel: ordered
        # copies when the call makes them, otherwise only the gaps of the launches
        kernels_ms["token_order_outside_kernels"] = round(avg(t_perm) * 1e3, 4)

    line = {
        "metric": "dense-equiv attention TOPS and % tensor peak at 128K causal; mask-pred GB/s",
        "value": round(value, 2),
        "unit": "dense-equiv TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_label,
        "data": "synthetic (seeded, bf16; %s)" % W.DATA_DESCRIPTIONS[w.name],
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                   "causal": w.causal, "topk": w.topk, "theta": w.theta, "lambda": lam,
                   "mask": "the workload's Bernoulli(0.25) tile mask" if given_mask else "predicted",
                   "l2": ("inputs larger than L2 (Q+K+V %.2f GB), no flush" % (in_bytes / 1e9) if flush is None else
                          "Q+K+V %.3f GB: L2 flushed (256 MB write) before every step, steps timed apart" % (in_bytes / 1e9)),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "kernels_ms": kernels_ms,
        "attn": {"ms": round(t_attn_avg * 1e3, 4), "dense_equiv_tops": round(dense / t_attn_avg / 1e12, 2),
                 "executed_tflops": round(attn_tflops, 2), "pct_tensor_peak": round(100 * attn_tflops / peak_tc, 2),
                 "kept_tiles": kept, "valid_tiles": valid, "sparsity": round(1 - kept / max(valid, 1), 4),
                 "pv_tiles": pv, "lambda_skipped_warp_tiles": skipped,
                 "lambda_skip_fraction": round(skipped / max(4 * kept, 1), 4)},
        "mask_pred": None if given_mask else {"ms": round(t_pred_avg * 1e3, 4), "gbs": round(pred_gbs, 1),
                                              "pct_hbm": round(100 * pred_gbs / hbm, 2), "bytes": pred_bytes},
        "roofline": {"bound": "tensor", "kernel": KERNEL_NAMES[(args.precision, w.d)], "achieved": round(attn_tflops, 2),
                     "peak": round(peak_tc, 1), "unit": "TFLOP/s", "frac": round(attn_tflops / peak_tc, 4),
                     "peak_source": (("bf16_tflops (burst; SM clock at max during the timed steps) " if at_max else
                                      "bf16_tflops_sustained (SM clock below max during the timed steps) ") + tag +
                                     ("" if args.precision == "bf16" else
                                      ", e4m3 products at 2x (nominal 4.5 / 2.25 PFLOP/s), weighted by the executed mix")),
                     "frac_of_sustained": round(attn_tflops / mix_peak(sustained), 4),
                     "traffic": profile_traffic(w, args.precision)},
        "e2e": {"value": round(world * dense / e2e_t / 1e12, 2), "unit": "dense-equiv TOPS",
                "h2d_bytes_per_step": int(w.q.nbytes + w.k.nbytes + w.v.nbytes),
                "d2h_bytes_per_step": int(o.numel() * 2), "clocks": e2e_clk},
        "gpu_launches": (LAUNCHES_PER_STEP[(args.precision, given_mask)] + order_copies) * args.steps,
        "clocks": clk,
    }
    line["permute"] = measure_permute(max(args.steps, 10), args.warmup, dev, peaks)
    if w.causal and w.mask is None and w.N // 64 >= 32:
        line["decode"] = measure_decode(q, k, w, max(args.steps, 10), args.warmup, dev, peaks, v)
    if rank == 0 and not args.no_cpu_baseline:
        tops, wall, desc, ncores = oracle_sample(w, args.cpu_blocks, min(args.cpu_workers, os.cpu_count() or 1))
        line["cpu_baseline"] = {"value": round(tops, 6), "unit": "dense-equiv TOPS", "cores": ncores,
                                "kind": "oracle", "sample": desc, "seconds": round(wall, 2)}
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


KERNEL_NAMES = {("bf16", 128): "bsattn_kernel<128,3,2,0,0>", ("bf16", 64): "bsattn_kernel<64,4,3,0,0>",
                ("q8", 128): "bsattn_kernel<128,4,2,1,0>", ("fp8pv", 128): "bsattn_kernel<128,4,3,1,1>",
                ("bf16fp8pv", 128): "bsattn_kernel<128,3,3,0,1>"}
# kernels per step: prediction (pool_sim, score_gemm, score_select) unless the mask is given, then
# the V copy (bf16) or the quantisation (K/V partial sums, their reduction, Q, K, and the V copy or
# the V quantisation; bf16 Q.K^T with e4m3 P.V: the V maxima, the V scales and the V quantisation),
# then the attention kernel
LAUNCHES_PER_STEP = {("bf16", False): 5, ("bf16", True): 2, ("q8", False): 9, ("q8", True): 6,
                     ("fp8pv", False): 9, ("fp8pv", True): 6, ("bf16fp8pv", False): 7, ("bf16fp8pv", True): 4}


def make_workload(args):
    over = {}
    if args.heads:
        hq, hkv = (int(x) for x in args.heads.split(","))
        over.update(Hq=hq, Hkv=hkv)
    if getattr(args, "topk", None) is not None:
        over["topk"] = args.topk
    return W.make_config(args.config, **over)


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = make_workload(args)
    for _ in range(args.warmup):
        oracle_sample(w, 2, 1)
    vals, walls = [], []
    desc, cores = "", 1
    for _ in range(args.steps):
        tops, wall, desc, cores = oracle_sample(w, args.cpu_blocks, min(args.cpu_workers, os.cpu_count() or 1))
        vals.append(tops)
        walls.append(wall)
    value = statistics.median(vals)
    line = {
        "impl": "reference",
        "metric": "dense-equiv attention TOPS and % tensor peak at 128K causal; mask-pred GB/s",
        "value": round(value, 6), "unit": "dense-equiv TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.median(walls), 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d, "causal": w.causal,
                   "topk": w.topk, "theta": w.theta, "lambda": w.lam},
        "cpu_baseline": {"value": round(value, 6), "unit": "dense-equiv TOPS", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "dense-equiv TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama128k", choices=list(W.CONFIG_NAMES))
    ap.add_argument("--cpu-blocks", type=int, default=384)
    ap.add_argument("--cpu-workers", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--precision", default="bf16", choices=list(PRECISIONS),
                    help="bf16, q8 (e4m3 Q.K^T, f16 P.V), fp8pv (both products e4m3) or bf16fp8pv (bf16 Q.K^T, "
                         "e4m3 P.V); 8-bit needs d = 128")
    ap.add_argument("--lam", type=float, default=None, help="lambda override (default: the workload's)")
    ap.add_argument("--topk", type=float, default=None,
                    help="topk override (default: the workload's), e.g. a denser mask than the synthetic data gives")
    ap.add_argument("--heads", default=None,
                    help="Hq,Hkv override (smaller cases of a workload for profiling; not a bench line)")
    ap.add_argument("--permute-only", action="store_true",
                    help="time only the Hilbert permute step (for profiling; not a bench line)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.permute_only:
        import torch
        torch.cuda.set_device(local_rank)
        print(json.dumps({"permute": measure_permute(max(args.steps, 10), args.warmup,
                                                     torch.device("cuda", local_rank), load_peaks())}))
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
