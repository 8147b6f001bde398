// Stage 1b, part 2: row softmax of the pooled scores, cumulative top-k and the always-keep rule,
// written as the uint8 block mask (SpargeAttention summary page: non-similar blocks are always
// computed; overview page "Strengths": mask of shape (B, H, ceil(N/128), ceil(N/64)); Chinese
// README quick start: topk = 0.5 keeps the top 50% of the attention weights).
//
// One warp per mask row, the row's valid scores in registers (lane l holds key blocks l, l+32,
// ...).  With e_j = exp(s_j - max) and Z = sum e_j, the kept set is every e_j > v* plus, among
// the e_j equal to v*, the lowest indices until the kept mass reaches topk * Z; v* is the largest
// value whose mass at or above it reaches topk * Z.  The search is two-level: a 32-bin histogram
// of the mass over the bit pattern of e (bins ordered by value, per-lane private columns in
// shared memory, no shared counters) finds the bin holding v*; then a bisection over that bin's
// bit patterns runs on the few elements inside it, compacted to a short list.  Elements more
// than log2(n / (1 - topk)) + 0.1 below the maximum (in log2 units) can never reach v* (the
// elements from v* down carry more than (1 - topk) Z, so v* >= (1 - topk) Z / n >= (1 - topk) / n),
// so they stay out of the histogram.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

constexpr int WARPS = 8;
constexpr int NBIN = 32;

struct SelArgs {
  const float *S;
  const float *sQ, *sK;
  uint8_t *mask;
  int64_t nkb_pad, rows;
  int Hq, Hkv, G, nqb, nkb, causal;
  float topk, theta;
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
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <int VPL>
__global__ void __launch_bounds__(WARPS * 32) score_select_kernel(SelArgs a) {
  __shared__ float hist[WARPS][NBIN * 32];  // per warp: [bin][lane]; reused for the candidate list
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *H = hist[w];
  const int64_t row = static_cast<int64_t>(blockIdx.x) * WARPS + w;
  if (row >= a.rows) return;
  const int i = static_cast<int>(row % a.nqb);
  const int64_t bh = row / a.nqb;
  const int h = static_cast<int>(bh % a.Hq), b = static_cast<int>(bh / a.Hq);
  const int kvh = h / a.G;
  const int nvalid = a.causal ? min(a.nkb, 2 * i + 2) : a.nkb;
  const float *srow = a.S + row * a.nkb_pad;
  const float *sKrow = a.sK + (static_cast<int64_t>(b) * a.Hkv + kvh) * a.nkb_pad;
  constexpr float LOG2E = 1.4426950408889634f;

  float e[VPL];
  float m = -FLT_MAX;
#pragma unroll
  for (int c = 0; c < VPL; ++c) {
    const int j = lane + 32 * c;
    e[c] = (j < nvalid) ? srow[j] : -FLT_MAX;
    m = fmaxf(m, e[c]);
  }
  m = warp_max(m);
  float zl = 0.f;
#pragma unroll
  for (int c = 0; c < VPL; ++c) {
    const int j = lane + 32 * c;
    e[c] = (j < nvalid) ? exp2f((e[c] - m) * LOG2E) : 0.f;
    zl += e[c];
  }
  const float Z = warp_sum(zl);
  const bool keep_all = a.topk >= 1.f || a.sQ[row] < a.theta;
  float vstar = 0.f;
  uint64_t tiekeep = 0;
  bool sorted = false;          // threshold found by sorting the crossing bin:
  float et = 0.f;               //   keep e > et, or e == et with index <= jt
  int jt = -1;
  if (!keep_all) {
    const float target = a.topk * Z;
    // Level 0: bins of width 2^sh bit patterns (2^(sh-23) log2 units) below 1.0f, wide enough that
    // 32 of them reach the bound past which no element can be v*.  Each further level splits the
    // crossing bin of the previous one into 32 sub-bins.  All levels use one formula:
    // bin = (hi - 1 - bits(e)) >> shift for e in [lo, hi).
    const float r2 = log2f(static_cast<float>(nvalid) / (1.f - a.topk)) + 0.1f;
    int shift = 16;
    while (static_cast<float>(NBIN) * exp2f(static_cast<float>(shift - 23)) < r2) ++shift;
    uint32_t lo = 1u, hi = 0x3F800001u;  // bit patterns: mass(e >= lo) >= target > mass(e >= hi)
    float above = 0.f;                   // mass of the elements >= hi
    int nc = 0x7fffffff;                 // elements in [lo, hi)
    for (int level = 0; level < 3 && nc > 32 && shift >= 0; ++level) {
#pragma unroll
      for (int k = 0; k < NBIN; ++k) H[k * 32 + lane] = 0.f;
      __syncwarp();
      const uint32_t top = hi - 1u;
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        const uint32_t u = __float_as_uint(e[c]);
        const uint32_t bin = (top - u) >> shift;
        if (e[c] > 0.f && u >= lo && u < hi && bin < NBIN) H[bin * 32 + lane] += e[c];  // lane-private column
      }
      __syncwarp();
      float mass = 0.f;  // lane = bin
#pragma unroll
      for (int k = 0; k < 32; ++k) mass += H[lane * 32 + ((k + lane) & 31)];
      float cum = mass;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, cum, off);
        if (lane >= off) cum += o;
      }
      const uint32_t hit = __ballot_sync(0xffffffffu, above + cum >= target);
      if (!hit) break;  // rounding left the crossing outside the bins: resolve [lo, hi) below
      const int bstar = __ffs(hit) - 1;
      const uint32_t nhi = top + 1u - (static_cast<uint32_t>(bstar) << shift);
      const uint32_t width = 1u << shift;
      const uint32_t nlo = (nhi > lo + width) ? nhi - width : lo;
      above += __shfl_sync(0xffffffffu, cum - mass, bstar);
      hi = nhi;
      lo = nlo;
      int cnt = 0;
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        const uint32_t u = __float_as_uint(e[c]);
        cnt += (e[c] > 0.f && u >= lo && u < hi) ? 1 : 0;
      }
      nc = warp_sum_i(cnt);
      shift -= 5;
      __syncwarp();
    }
    if (nc <= 32) {
      // one candidate per lane: sort by (e desc, index asc), then the first prefix reaching target
      int cnt = 0;
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        const uint32_t u = __float_as_uint(e[c]);
        cnt += (e[c] > 0.f && u >= lo && u < hi) ? 1 : 0;
      }
      int off = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, off, o);
        if (lane >= o) off += v;
      }
      off -= cnt;
      __syncwarp();
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        const uint32_t u = __float_as_uint(e[c]);
        if (e[c] > 0.f && u >= lo && u < hi) {
          H[off] = e[c];
          H[32 + off] = __int_as_float(lane + 32 * c);
          ++off;
        }
      }
      __syncwarp();
      float ce = lane < nc ? H[lane] : -1.f;
      int cj = lane < nc ? __float_as_int(H[32 + lane]) : 0x7fffffff;
#pragma unroll
      for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
          const float oe = __shfl_xor_sync(0xffffffffu, ce, jj);
          const int oj = __shfl_xor_sync(0xffffffffu, cj, jj);
          const bool mine_first = ce > oe || (ce == oe && cj < oj);
          const bool take_first = ((lane & jj) == 0) == ((lane & kk) == 0);
          if (mine_first != take_first) {
            ce = oe;
            cj = oj;
          }
        }
      }
      float ps = ce > 0.f ? ce : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, ps, o);
        if (lane >= o) ps += v;
      }
      const uint32_t reach = __ballot_sync(0xffffffffu, lane < nc && above + ps >= target);
      if (reach) {
        const int kstar = __ffs(reach) - 1;
        et = __shfl_sync(0xffffffffu, ce, kstar);
        jt = __shfl_sync(0xffffffffu, cj, kstar);
        sorted = true;
      }
    }
    if (!sorted) {
      // bisection over every element in [lo, hi) (rare: many equal-looking values or rounding)
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
    }
  }
  if (!keep_all && !sorted) {
    const float target = a.topk * Z;
    // elements equal to v*: keep them in ascending key-block order until the mass reaches target
    int nties = 0;
    float abovev = 0.f;
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      abovev += (e[c] > vstar) ? e[c] : 0.f;
      nties += (e[c] == vstar && (lane + 32 * c) < nvalid) ? 1 : 0;
    }
    nties = warp_sum_i(nties);
    if (nties == 1) {
#pragma unroll
      for (int c = 0; c < VPL; ++c)
        if (e[c] == vstar && (lane + 32 * c) < nvalid) tiekeep |= (1ull << c);
    } else if (nties > 1) {
      float cumv = warp_sum(abovev);
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        uint32_t bal = __ballot_sync(0xffffffffu, e[c] == vstar && (lane + 32 * c) < nvalid);
        while (bal != 0u && cumv < target) {
          const int l = __ffs(bal) - 1;
          if (lane == l) tiekeep |= (1ull << c);
          cumv += vstar;
          bal &= bal - 1u;
        }
      }
    }
  }
  uint8_t *mrow = a.mask + row * a.nkb;
#pragma unroll
  for (int c = 0; c < VPL; ++c) {
    const int j = lane + 32 * c;
    if (j < a.nkb) {
      bool keep = false;
      if (j < nvalid) {
        const bool topk_keep = sorted ? (e[c] > et || (e[c] == et && j <= jt))
                                      : (e[c] > vstar || ((tiekeep >> c) & 1ull));
        keep = keep_all || topk_keep || sKrow[j] < a.theta;
      }
      mrow[j] = keep ? 1 : 0;
    }
  }
}

template <int VPL>
cudaError_t launch_t(const SelArgs &a, cudaStream_t st) {
  const int64_t grid = (a.rows + WARPS - 1) / WARPS;
  score_select_kernel<VPL><<<static_cast<unsigned>(grid), WARPS * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_select(const PredictWs &ws, int B, int Hq, int Hkv, int N, int d, float topk,
                                float theta, int causal, uint8_t *mask, cudaStream_t st) {
  (void)d;
  SelArgs a;
  a.S = ws.S;
  a.sQ = ws.sQ;
  a.sK = ws.sK;
  a.mask = mask;
  a.nkb_pad = ws.nkb_pad;
  a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv;
  a.nqb = (N + QBLK - 1) / QBLK;
  a.nkb = (N + KBLK - 1) / KBLK;
  a.causal = causal;
  a.rows = static_cast<int64_t>(B) * Hq * a.nqb;
  a.topk = topk;
  a.theta = theta;
  if (a.rows == 0) return cudaSuccess;
  if (a.nkb <= 256) return launch_t<8>(a, st);
  if (a.nkb <= 512) return launch_t<16>(a, st);
  if (a.nkb <= 1024) return launch_t<32>(a, st);
  return launch_t<64>(a, st);
}

}  // namespace sparge
