// Stage 1a: block mean pooling and intra-block self-similarity (SpargeAttention summary page,
// method paragraph: token blocks with high internal similarity are compressed).
//
// For each 128-token query block and 64-token key block this kernel produces the fp32 mean of
// the valid tokens and s = ||(1/n) sum_a x_a / ||x_a|| ||^2, the mean cosine similarity over
// all ordered token pairs of the block (pairs a == b included).  A zero token contributes a
// zero unit vector.  Memory-bound: one pass over Q and K with 16-byte streaming loads, fp32
// accumulation (packed pair arithmetic), warp-shuffle reductions.
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

struct BlockRef {
  const __nv_bfloat16 *base;  // first token row of the block
  int64_t sn;                  // token stride (elements)
  int n;                       // valid tokens
  int steps;                   // CTA load steps covering the block
  float *mu;                   // where the mean goes (d contiguous floats)
  uint16_t *hi, *lo;           // where its bf16 hi/lo split goes
  float *s;                    // where the similarity goes
};

template <int TPS>
__device__ __forceinline__ BlockRef block_ref(const PoolArgs &a, int64_t bid, int D) {
  BlockRef r;
  if (bid < a.nq_total) {
    const int i = static_cast<int>(bid % a.nqb);
    const int64_t bh = bid / a.nqb;
    const int h = static_cast<int>(bh % a.Hq), b = static_cast<int>(bh / a.Hq);
    r.base = a.q + b * a.q_sb + h * a.q_sh + static_cast<int64_t>(i) * QBLK * a.q_sn;
    r.sn = a.q_sn;
    r.n = min(QBLK, a.N - i * QBLK);
    r.steps = QBLK / TPS;
    const int64_t row = (static_cast<int64_t>(b) * a.Hq + h) * a.nqb + i;
    r.mu = a.ws.muQ + row * D;
    r.hi = a.ws.qhi + row * D;
    r.lo = a.ws.qlo + row * D;
    r.s = a.ws.sQ + row;
  } else {
    bid -= a.nq_total;
    const int j = static_cast<int>(bid % a.nkb);
    const int64_t bh = bid / a.nkb;
    const int h = static_cast<int>(bh % a.Hkv), b = static_cast<int>(bh / a.Hkv);
    r.base = a.k + b * a.k_sb + h * a.k_sh + static_cast<int64_t>(j) * KBLK * a.k_sn;
    r.sn = a.k_sn;
    r.n = min(KBLK, a.N - j * KBLK);
    r.steps = KBLK / TPS;
    const int64_t row = (static_cast<int64_t>(b) * a.Hkv + h) * a.nkb + j;
    r.mu = a.ws.muK + row * D;
    r.hi = a.ws.khi + row * D;
    r.lo = a.ws.klo + row * D;
    r.s = a.ws.sK + (static_cast<int64_t>(b) * a.Hkv + h) * a.ws.nkb_pad + j;
  }
  return r;
}

// Persistent CTAs walk the blocks (all query blocks, then all key blocks) with a stride of the
// grid size.  Each thread keeps the 16-byte vectors of the next block in flight (registers)
// while it reduces the current one, so the loads of a CTA overlap its arithmetic.
template <int D>
__global__ void __launch_bounds__(256, (D == 128 ? 2 : 3)) pool_sim_kernel(PoolArgs a) {
  constexpr int LPT = D / 8;        // lanes per token, 8 bf16 (16 bytes) per lane
  constexpr int TPW = 32 / LPT;     // tokens per warp per step
  constexpr int TPS = 8 * TPW;      // tokens per CTA step
  constexpr int MAXSTEPS = QBLK / TPS;

  __shared__ float red[2][8][2][D];  // double-buffered per-warp partial sums (x and unit x)
  __shared__ float red_s[2][8];      // per-warp partial sums of squares of the mean unit vector

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPT, part = lane % LPT;
  const int64_t total = a.nq_total + static_cast<int64_t>(a.B) * a.Hkv * a.nkb;

  auto load = [&](const BlockRef &r, uint4 (&v)[MAXSTEPS]) {
#pragma unroll
    for (int st = 0; st < MAXSTEPS; ++st) {
      const int t = st * TPS + w * TPW + sub;
      v[st] = make_uint4(0, 0, 0, 0);
      if (st < r.steps && t < r.n) v[st] = ld_stream_v4(r.base + t * r.sn + part * 8);
    }
  };

  int64_t bid = blockIdx.x;
  if (bid >= total) return;
  BlockRef cur = block_ref<TPS>(a, bid, D);
  uint4 vc[MAXSTEPS], vn[MAXSTEPS];
  load(cur, vc);
  float *prev_s = nullptr;
  int it = 0;
  for (; bid < total; ++it) {
    const int64_t nbid = bid + gridDim.x;
    BlockRef nxt = cur;
    if (nbid < total) {
      nxt = block_ref<TPS>(a, nbid, D);
      load(nxt, vn);
    }
    float2 sx2[4], sh2[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) sx2[c] = sh2[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int st = 0; st < MAXSTEPS; ++st) {
      if (st < cur.steps) {
        const uint32_t wd[4] = {vc[st].x, vc[st].y, vc[st].z, vc[st].w};
        float2 x2[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) x2[c] = make_float2(bf16lo(wd[c]), bf16hi(wd[c]));
        float2 n2 = fmul2(x2[0], x2[0]);
#pragma unroll
        for (int c = 1; c < 4; ++c) n2 = ffma2(x2[c], x2[c], n2);
        float nn = n2.x + n2.y;
#pragma unroll
        for (int off = LPT / 2; off > 0; off >>= 1) nn += __shfl_xor_sync(0xffffffffu, nn, off);
        const float inv = nn > 0.f ? rsqrtf(nn) : 0.f;
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          sx2[c] = fadd2(sx2[c], x2[c]);
          sh2[c] = ffma2(x2[c], inv2, sh2[c]);
        }
      }
    }
    // sum over the token slots of the warp: lanes with the same `part`
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        sx2[c].x += __shfl_xor_sync(0xffffffffu, sx2[c].x, off);
        sx2[c].y += __shfl_xor_sync(0xffffffffu, sx2[c].y, off);
        sh2[c].x += __shfl_xor_sync(0xffffffffu, sh2[c].x, off);
        sh2[c].y += __shfl_xor_sync(0xffffffffu, sh2[c].y, off);
      }
    }
    float(*rb)[2][D] = red[it & 1];
    if (sub == 0) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        rb[w][0][part * 8 + 2 * c] = sx2[c].x;
        rb[w][0][part * 8 + 2 * c + 1] = sx2[c].y;
        rb[w][1][part * 8 + 2 * c] = sh2[c].x;
        rb[w][1][part * 8 + 2 * c + 1] = sh2[c].y;
      }
    }
    __syncthreads();
    // the similarity of the previous block: its eight per-warp partial sums of squares
    if (threadIdx.x == 0 && prev_s) {
      float sprev = 0.f;
#pragma unroll
      for (int ww = 0; ww < 8; ++ww) sprev += red_s[(it - 1) & 1][ww];
      *prev_s = sprev;
    }
    // every warp finishes D/8 dimensions of this block (the partial sums alternate between two
    // buffers, so the next barrier orders their reuse)
    {
      constexpr int DPW = D / 8;
      const float invn = 1.f / static_cast<float>(cur.n);
      float hsq = 0.f;
      if (lane < DPW) {
        const int dim = w * DPW + lane;
        float mx = 0.f, hx = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) {
          mx += rb[ww][0][dim];
          hx += rb[ww][1][dim];
        }
        hx *= invn;
        hsq = hx * hx;
        const float mean = mx * invn;
        cur.mu[dim] = mean;
        const __nv_bfloat16 hb = __float2bfloat16_rn(mean);
        cur.hi[dim] = __bfloat16_as_ushort(hb);
        cur.lo[dim] = __bfloat16_as_ushort(__float2bfloat16_rn(mean - __bfloat162float(hb)));
      }
#pragma unroll
      for (int off = DPW / 2; off > 0; off >>= 1) hsq += __shfl_xor_sync(0xffffffffu, hsq, off);
      if (lane == 0) red_s[it & 1][w] = hsq;
    }
    prev_s = cur.s;
    cur = nxt;
#pragma unroll
    for (int st = 0; st < MAXSTEPS; ++st) vc[st] = vn[st];
    bid = nbid;
  }
  __syncthreads();
  if (threadIdx.x == 0 && prev_s) {
    float sprev = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) sprev += red_s[(it - 1) & 1][ww];
    *prev_s = sprev;
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
  const int64_t total = a.nq_total + static_cast<int64_t>(a.B) * a.Hkv * a.nkb;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * (q.d == 128 ? 2 : 3);  // resident CTAs
  const unsigned grid = static_cast<unsigned>(total < cap ? total : cap);
  if (q.d == 128)
    pool_sim_kernel<128><<<grid, 256, 0, st>>>(a);
  else
    pool_sim_kernel<64><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sparge
