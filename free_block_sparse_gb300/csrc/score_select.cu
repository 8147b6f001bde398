// Stage 1b: pooled score map, row softmax, cumulative top-k and always-keep rule, written as
// the uint8 block mask (SpargeAttention abstract: the attention map is predicted from a
// compressed Q/K so that matrix multiplications of dropped tiles are skipped; summary page:
// non-similar blocks are always computed; overview page "Strengths": mask of shape
// (B, H, ceil(N/128), ceil(N/64)); Chinese README quick start: topk = 0.5 keeps the top 50%
// of the attention weights).
//
// One CTA takes 16 query blocks of one head.  Phase 1 computes their pooled scores against
// every valid key block with an fp32 register-tiled product (4 rows x 4 key blocks per thread,
// key means staged through shared memory 32 dims at a time) into a shared-memory score tile.
// Phase 2 gives each warp one row at a time with the row's values in registers (lane l holds
// key blocks l, l+32, ...): max, exponentials, their sum Z, then a bisection over the bit
// pattern of the threshold value v* (the largest value whose mass at or above it still
// reaches topk * Z), ties at v* kept in ascending index order, and the mask row written.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

constexpr int ROWS = 16;      // query blocks per CTA
constexpr int JCHUNK = 256;   // key blocks per product chunk
constexpr int KSLAB = 32;     // dims per staged slab
constexpr int KPITCH = JCHUNK + 4;

struct ScoreArgs {
  PredictWs ws;
  uint8_t *mask;
  int B, Hq, Hkv, G, N, nqb, nkb, causal, ngroups;
  float topk, theta, scale;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

template <int D, int VPL>
__global__ void __launch_bounds__(256, 1) score_select_kernel(ScoreArgs a) {
  constexpr int SP = 32 * VPL;  // score row pitch (>= nkb)
  extern __shared__ __align__(16) float smem[];
  float *S = smem;                       // [ROWS][SP]
  float *qT = S + ROWS * SP;             // [D][ROWS]
  float *kT = qT + D * ROWS;             // [KSLAB][KPITCH]

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // heavy (late, causal) row groups first
  const int gidx = a.ngroups - 1 - static_cast<int>(blockIdx.x % a.ngroups);
  const int bh = static_cast<int>(blockIdx.x / a.ngroups);
  const int h = bh % a.Hq, b = bh / a.Hq;
  const int kvh = h / a.G;
  const int i0 = gidx * ROWS;
  const int ilast = min(i0 + ROWS - 1, a.nqb - 1);
  const int ncols = a.causal ? min(a.nkb, 2 * ilast + 2) : a.nkb;

  const float *muQ = a.ws.muQ + ((static_cast<int64_t>(b) * a.Hq + h) * a.nqb) * D;
  const float *muKt = a.ws.muKt + (static_cast<int64_t>(b) * a.Hkv + kvh) * D * a.ws.nkb_pad;

  for (int e = tid; e < ROWS * D; e += 256) {
    const int r = e / D, kk = e % D;
    qT[kk * ROWS + r] = (i0 + r < a.nqb) ? muQ[static_cast<int64_t>(i0 + r) * D + kk] : 0.f;
  }

  const int ty = tid / 64, tx = tid % 64;  // rows 4ty..4ty+3, key blocks 4tx..4tx+3 of the chunk
  for (int jc = 0; jc < ncols; jc += JCHUNK) {
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    for (int ks = 0; ks < D; ks += KSLAB) {
      __syncthreads();
#pragma unroll
      for (int rep = 0; rep < (KSLAB * JCHUNK / 4) / 256; ++rep) {
        const int e = tid + rep * 256;
        const int kk = e / (JCHUNK / 4), jj = (e % (JCHUNK / 4)) * 4;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (jc + jj < a.ws.nkb_pad)
          val = *reinterpret_cast<const float4 *>(muKt + static_cast<int64_t>(ks + kk) * a.ws.nkb_pad + jc + jj);
        *reinterpret_cast<float4 *>(kT + kk * KPITCH + jj) = val;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < KSLAB; ++kk) {
        const float4 qa = *reinterpret_cast<const float4 *>(qT + (ks + kk) * ROWS + 4 * ty);
        const float4 kb = *reinterpret_cast<const float4 *>(kT + kk * KPITCH + 4 * tx);
        const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
        const float kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(qv[r], kv[c], acc[r][c]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float4 o = make_float4(acc[r][0] * a.scale, acc[r][1] * a.scale, acc[r][2] * a.scale, acc[r][3] * a.scale);
      *reinterpret_cast<float4 *>(S + (4 * ty + r) * SP + jc + 4 * tx) = o;
    }
  }
  __syncthreads();

  // ---------------- phase 2: per-row softmax, top-k threshold and mask write ----------------
  const float *sKrow = a.ws.sK + (static_cast<int64_t>(b) * a.Hkv + kvh) * a.ws.nkb_pad;
  for (int r = w; r < ROWS; r += 8) {
    const int i = i0 + r;
    if (i >= a.nqb) break;
    const int nvalid = a.causal ? min(a.nkb, 2 * i + 2) : a.nkb;
    float e[VPL];
    float m = -FLT_MAX;
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      const int j = lane + 32 * c;
      e[c] = (j < nvalid) ? S[r * SP + j] : -FLT_MAX;
      m = fmaxf(m, e[c]);
    }
    m = warp_max(m);
    float zl = 0.f;
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      const int j = lane + 32 * c;
      e[c] = (j < nvalid) ? expf(e[c] - m) : 0.f;
      zl += e[c];
    }
    const float Z = warp_sum(zl);
    const bool keep_all = a.topk >= 1.f || a.ws.sQ[(static_cast<int64_t>(b) * a.Hq + h) * a.nqb + i] < a.theta;
    float vstar = 0.f;
    uint64_t tiekeep = 0;
    if (!keep_all) {
      const float target = a.topk * Z;
      // invariant: mass(e >= float(lo)) >= target > mass(e >= float(hi))
      uint32_t lo = 0u, hi = 0x3F800001u;
      while (hi - lo > 1u) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        const float tv = __uint_as_float(mid);
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < VPL; ++c) part += (e[c] >= tv) ? e[c] : 0.f;
        if (warp_sum(part) >= target)
          lo = mid;
        else
          hi = mid;
      }
      vstar = __uint_as_float(lo);
      float above = 0.f;
#pragma unroll
      for (int c = 0; c < VPL; ++c) above += (e[c] > vstar) ? e[c] : 0.f;
      float cum = warp_sum(above);
      // elements equal to v*: keep them in ascending key-block order until the mass reaches target
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        uint32_t bal = __ballot_sync(0xffffffffu, e[c] == vstar && (lane + 32 * c) < nvalid);
        while (bal != 0u && cum < target) {
          const int l = __ffs(bal) - 1;
          if (lane == l) tiekeep |= (1ull << c);
          cum += vstar;
          bal &= bal - 1u;
        }
      }
    }
    uint8_t *mrow = a.mask + ((static_cast<int64_t>(b) * a.Hq + h) * a.nqb + i) * a.nkb;
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      const int j = lane + 32 * c;
      if (j < a.nkb) {
        bool keep = false;
        if (j < nvalid)
          keep = keep_all || e[c] > vstar || ((tiekeep >> c) & 1ull) || sKrow[j] < a.theta;
        mrow[j] = keep ? 1 : 0;
      }
    }
  }
}

template <int D, int VPL>
cudaError_t launch_t(const ScoreArgs &a, cudaStream_t st) {
  const size_t smem = sizeof(float) * (static_cast<size_t>(ROWS) * 32 * VPL + D * ROWS + KSLAB * KPITCH);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(score_select_kernel<D, VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t grid = static_cast<int64_t>(a.B) * a.Hq * a.ngroups;
  score_select_kernel<D, VPL><<<static_cast<unsigned>(grid), 256, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const ScoreArgs &a, cudaStream_t st) {
  if (a.nkb <= 256) return launch_t<D, 8>(a, st);
  if (a.nkb <= 512) return launch_t<D, 16>(a, st);
  if (a.nkb <= 1024) return launch_t<D, 32>(a, st);
  return launch_t<D, 64>(a, st);
}

}  // namespace

cudaError_t launch_score_select(const PredictWs &ws, int B, int Hq, int Hkv, int N, int d, float topk,
                                float theta, int causal, float scale, uint8_t *mask, cudaStream_t st) {
  ScoreArgs a;
  a.ws = ws;
  a.mask = mask;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.N = N;
  a.nqb = (N + QBLK - 1) / QBLK;
  a.nkb = (N + KBLK - 1) / KBLK;
  a.causal = causal;
  a.ngroups = (a.nqb + ROWS - 1) / ROWS;
  a.topk = topk; a.theta = theta; a.scale = scale;
  if (static_cast<int64_t>(B) * Hq * a.ngroups == 0) return cudaSuccess;
  return d == 128 ? launch_d<128>(a, st) : launch_d<64>(a, st);
}

}  // namespace sparge
