// Stage 1a: block mean pooling and intra-block self-similarity (SpargeAttention summary page,
// method paragraph: token blocks with high internal similarity are compressed).
//
// For each 128-token query block and 64-token key block this kernel produces the fp32 mean of
// the valid tokens and s = ||(1/n) sum_a x_a / ||x_a|| ||^2, the mean cosine similarity over
// all ordered token pairs of the block (pairs a == b included).  A zero token contributes a
// zero unit vector.  Memory-bound: one pass over Q and K with 16-byte streaming loads, fp32
// accumulation, warp-shuffle reductions; every load of a CTA is issued before any arithmetic.
#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

struct PoolArgs {
  const __nv_bfloat16 *q, *k;
  int64_t q_sb, q_sh, q_sn, k_sb, k_sh, k_sn;
  int B, Hq, Hkv, N, nqb, nkb;
  int64_t nq_total;  // B * Hq * nqb
  PredictWs ws;
};

template <int D>
__global__ void __launch_bounds__(256) pool_sim_kernel(PoolArgs a) {
  constexpr int LPT = D / 8;        // lanes per token, 8 bf16 (16 bytes) per lane
  constexpr int TPW = 32 / LPT;     // tokens per warp per step
  constexpr int TPS = 8 * TPW;      // tokens per CTA step
  constexpr int MAXSTEPS = QBLK / TPS;

  __shared__ float red[8][2][D];
  __shared__ float red_s[D / 32];

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPT, part = lane % LPT;

  int64_t bid = blockIdx.x;
  const bool isQ = bid < a.nq_total;
  const __nv_bfloat16 *base;
  int blk, tok0, b, h, blkidx;
  if (isQ) {
    blkidx = static_cast<int>(bid % a.nqb);
    int64_t bh = bid / a.nqb;
    h = static_cast<int>(bh % a.Hq);
    b = static_cast<int>(bh / a.Hq);
    base = a.q + b * a.q_sb + h * a.q_sh;
    blk = QBLK;
    tok0 = blkidx * QBLK;
  } else {
    bid -= a.nq_total;
    blkidx = static_cast<int>(bid % a.nkb);
    int64_t bh = bid / a.nkb;
    h = static_cast<int>(bh % a.Hkv);
    b = static_cast<int>(bh / a.Hkv);
    base = a.k + b * a.k_sb + h * a.k_sh;
    blk = KBLK;
    tok0 = blkidx * KBLK;
  }
  const int64_t sn = isQ ? a.q_sn : a.k_sn;
  const int n = min(blk, a.N - tok0);
  const int steps = blk / TPS;

  uint4 v[MAXSTEPS];
#pragma unroll
  for (int s = 0; s < MAXSTEPS; ++s) {
    const int t = s * TPS + w * TPW + sub;
    v[s] = make_uint4(0, 0, 0, 0);
    if (s < steps && t < n) v[s] = ld_stream_v4(base + (tok0 + t) * sn + part * 8);
  }

  float sx[8], sh[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) sx[c] = sh[c] = 0.f;

#pragma unroll
  for (int s = 0; s < MAXSTEPS; ++s) {
    if (s < steps) {
      const uint32_t wd[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
      float x[8];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        x[2 * c] = bf16lo(wd[c]);
        x[2 * c + 1] = bf16hi(wd[c]);
      }
      float n2 = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) n2 = fmaf(x[c], x[c], n2);
#pragma unroll
      for (int off = LPT / 2; off > 0; off >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, off);
      const float inv = n2 > 0.f ? rsqrtf(n2) : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        sx[c] += x[c];
        sh[c] = fmaf(x[c], inv, sh[c]);
      }
    }
  }
  // sum over the token slots of the warp: lanes with the same `part`
#pragma unroll
  for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      sx[c] += __shfl_xor_sync(0xffffffffu, sx[c], off);
      sh[c] += __shfl_xor_sync(0xffffffffu, sh[c], off);
    }
  }
  if (sub == 0) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      red[w][0][part * 8 + c] = sx[c];
      red[w][1][part * 8 + c] = sh[c];
    }
  }
  __syncthreads();
  const int t = threadIdx.x;
  float hsq = 0.f;
  const float invn = 1.f / static_cast<float>(n);
  if (t < D) {
    float mx = 0.f, hx = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {
      mx += red[ww][0][t];
      hx += red[ww][1][t];
    }
    mx *= invn;
    hx *= invn;
    hsq = hx * hx;
    if (isQ)
      a.ws.muQ[((static_cast<int64_t>(b) * a.Hq + h) * a.nqb + blkidx) * D + t] = mx;
    else
      a.ws.muKt[((static_cast<int64_t>(b) * a.Hkv + h) * D + t) * a.ws.nkb_pad + blkidx] = mx;
  }
  if (t < D) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) hsq += __shfl_xor_sync(0xffffffffu, hsq, off);
    if (lane == 0) red_s[w] = hsq;
  }
  __syncthreads();
  if (t == 0) {
    float s = 0.f;
#pragma unroll
    for (int ww = 0; ww < D / 32; ++ww) s += red_s[ww];
    if (isQ)
      a.ws.sQ[(static_cast<int64_t>(b) * a.Hq + h) * a.nqb + blkidx] = s;
    else
      a.ws.sK[(static_cast<int64_t>(b) * a.Hkv + h) * a.ws.nkb_pad + blkidx] = s;
  }
}

}  // namespace

cudaError_t launch_pool_sim(const View &q, const View &k, const PredictWs &ws, cudaStream_t st) {
  PoolArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(q.data);
  a.k = static_cast<const __nv_bfloat16 *>(k.data);
  a.q_sb = q.sb; a.q_sh = q.sh; a.q_sn = q.sn;
  a.k_sb = k.sb; a.k_sh = k.sh; a.k_sn = k.sn;
  a.B = static_cast<int>(q.B); a.Hq = static_cast<int>(q.H); a.Hkv = static_cast<int>(k.H);
  a.N = static_cast<int>(q.N);
  a.nqb = (a.N + QBLK - 1) / QBLK;
  a.nkb = (a.N + KBLK - 1) / KBLK;
  a.nq_total = static_cast<int64_t>(a.B) * a.Hq * a.nqb;
  a.ws = ws;
  const int64_t grid = a.nq_total + static_cast<int64_t>(a.B) * a.Hkv * a.nkb;
  if (grid == 0) return cudaSuccess;
  if (q.d == 128)
    pool_sim_kernel<128><<<static_cast<unsigned>(grid), 256, 0, st>>>(a);
  else
    pool_sim_kernel<64><<<static_cast<unsigned>(grid), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sparge
