// Stage 1b, part 2: row softmax of the pooled scores, cumulative top-k and the always-keep rule,
// written as the uint8 block mask (SpargeAttention summary page: non-similar blocks are always
// computed; overview page "Strengths": mask of shape (B, H, ceil(N/128), ceil(N/64)); Chinese
// README quick start: topk = 0.5 keeps the top 50% of the attention weights).
//
// One warp per mask row, the row's valid scores in registers (lane l holds key blocks l, l+32,
// ...; the register count per lane is chosen per row from its number of valid blocks).  With
// e_j = exp(s_j - max) and Z = sum e_j, the kept set is the shortest prefix, in (e desc, index
// asc) order, whose mass reaches topk * Z.  The cut is found without sorting the row: a 32-bin
// histogram of the mass over the bit pattern of e (bins ordered by value, per-lane private
// columns in shared memory, no shared counters) finds the bin holding the cut; that bin is split
// again into 32 sub-bins (after the few elements inside it have been compacted into a short
// list) until at most 32 remain, which one warp-wide bitonic sort orders exactly.  Elements more
// than log2(n / (1 - topk)) + 0.1 below the maximum (in log2 units) never reach the cut (the
// elements from the cut down carry more than (1 - topk) Z, so the cut value is at least
// (1 - topk) Z / n >= (1 - topk) / n), so they stay out of the histogram.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

constexpr int WARPS = 8;
constexpr int NBIN = 32;
constexpr int CMAX = 256;  // crossing-bin elements compacted into the short list (8 per lane)

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
__device__ __forceinline__ bool in_range(float x, uint32_t lo, uint32_t hi) {
  const uint32_t u = __float_as_uint(x);
  return x > 0.f && u >= lo && u < hi;
}

// The search state: bit patterns [lo, hi) hold the cut (mass(e >= lo) >= target > mass(e >= hi)),
// `above` is the mass of the elements >= hi, `nc` the number of elements in [lo, hi).
struct Cut {
  uint32_t lo, hi;
  float above;
  int nc, shift;
};

// One histogram level over the elements of x inside [lo, hi): 32 bins of 2^shift patterns from
// hi - 1 down; narrows the state to the bin where the cumulative mass first reaches target.
// Returns false (state unchanged) if rounding left no bin reaching it.
template <int V>
__device__ __forceinline__ bool hist_level(const float (&x)[V], float *H, int lane, float target, Cut &st) {
#pragma unroll
  for (int k = 0; k < NBIN; ++k) H[k * 32 + lane] = 0.f;
  __syncwarp();
  const uint32_t top = st.hi - 1u;
#pragma unroll
  for (int c = 0; c < V; ++c) {
    const uint32_t bin = (top - __float_as_uint(x[c])) >> st.shift;
    if (in_range(x[c], st.lo, st.hi) && bin < NBIN) H[bin * 32 + lane] += x[c];  // lane-private column
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
  const uint32_t hit = __ballot_sync(0xffffffffu, st.above + cum >= target);
  __syncwarp();
  if (!hit) return false;
  const int bstar = __ffs(hit) - 1;
  const uint32_t nhi = st.hi - (static_cast<uint32_t>(bstar) << st.shift);
  const uint32_t width = 1u << st.shift;
  st.lo = (nhi > st.lo + width) ? nhi - width : st.lo;
  st.hi = nhi;
  st.above += __shfl_sync(0xffffffffu, cum - mass, bstar);
  int cnt = 0;
#pragma unroll
  for (int c = 0; c < V; ++c) cnt += in_range(x[c], st.lo, st.hi) ? 1 : 0;
  st.nc = warp_sum_i(cnt);
  st.shift -= 5;
  return true;
}

// Exclusive prefix over lanes of per-lane counts.
__device__ __forceinline__ int lane_offset(int cnt, int lane) {
  int off = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, off, o);
    if (lane >= o) off += v;
  }
  return off - cnt;
}

template <int V>
__device__ __forceinline__ void select_row(const SelArgs &a, float *H, int lane, int64_t row, int nvalid,
                                           const float *srow, const float *sKrow) {
  constexpr float LOG2E = 1.4426950408889634f;
  float e[V];
  float m = -FLT_MAX;
#pragma unroll
  for (int c = 0; c < V; ++c) {
    const int j = lane + 32 * c;
    e[c] = (j < nvalid) ? srow[j] : -FLT_MAX;
    m = fmaxf(m, e[c]);
  }
  m = warp_max(m);
  float zl = 0.f;
#pragma unroll
  for (int c = 0; c < V; ++c) {
    const int j = lane + 32 * c;
    e[c] = (j < nvalid) ? exp2f((e[c] - m) * LOG2E) : 0.f;
    zl += e[c];
  }
  const float Z = warp_sum(zl);
  const bool keep_all = a.topk >= 1.f || a.sQ[row] < a.theta;
  bool sorted = false;  // cut found by the sort: keep e > et, or e == et with index <= jt
  float et = 0.f, vstar = 0.f;
  int jt = -1;
  uint64_t tiekeep = 0;
  if (!keep_all) {
    const float target = a.topk * Z;
    const float r2 = log2f(static_cast<float>(nvalid) / (1.f - a.topk)) + 0.1f;
    Cut st;
    st.lo = 1u;
    st.hi = 0x3F800001u;
    st.above = 0.f;
    st.nc = 0x7fffffff;
    st.shift = 16;
    while (static_cast<float>(NBIN) * exp2f(static_cast<float>(st.shift - 23)) < r2) ++st.shift;
    bool ok = hist_level(e, H, lane, target, st);
    // the short list: crossing-bin elements with their key-block indices
    float ce[CMAX / 32];
    int cj[CMAX / 32];
    bool compact = false;
    if (ok && st.nc > 32 && st.nc <= CMAX) {
      int cnt = 0;
#pragma unroll
      for (int c = 0; c < V; ++c) cnt += in_range(e[c], st.lo, st.hi) ? 1 : 0;
      int off = lane_offset(cnt, lane);
#pragma unroll
      for (int c = 0; c < V; ++c)
        if (in_range(e[c], st.lo, st.hi)) {
          H[off] = e[c];
          H[CMAX + off] = __int_as_float(lane + 32 * c);
          ++off;
        }
      __syncwarp();
#pragma unroll
      for (int k = 0; k < CMAX / 32; ++k) {
        const int idx = lane + 32 * k;
        ce[k] = idx < st.nc ? H[idx] : 0.f;
        cj[k] = idx < st.nc ? __float_as_int(H[CMAX + idx]) : 0x7fffffff;
      }
      __syncwarp();
      compact = true;
      for (int lev = 0; lev < 3 && ok && st.nc > 32 && st.shift >= 0; ++lev) ok = hist_level(ce, H, lane, target, st);
    } else {
      for (int lev = 0; lev < 2 && ok && st.nc > 32 && st.shift >= 0; ++lev) ok = hist_level(e, H, lane, target, st);
    }
    if (ok && st.nc <= 32) {
      // one candidate per lane, sorted by (e desc, index asc); the first prefix reaching target
      float x = -1.f;
      int xj = 0x7fffffff;
      int cnt = 0;
      if (compact) {
#pragma unroll
        for (int k = 0; k < CMAX / 32; ++k) cnt += in_range(ce[k], st.lo, st.hi) ? 1 : 0;
      } else {
#pragma unroll
        for (int c = 0; c < V; ++c) cnt += in_range(e[c], st.lo, st.hi) ? 1 : 0;
      }
      int off = lane_offset(cnt, lane);
      if (compact) {
#pragma unroll
        for (int k = 0; k < CMAX / 32; ++k)
          if (in_range(ce[k], st.lo, st.hi)) {
            H[off] = ce[k];
            H[32 + off] = __int_as_float(cj[k]);
            ++off;
          }
      } else {
#pragma unroll
        for (int c = 0; c < V; ++c)
          if (in_range(e[c], st.lo, st.hi)) {
            H[off] = e[c];
            H[32 + off] = __int_as_float(lane + 32 * c);
            ++off;
          }
      }
      __syncwarp();
      if (lane < st.nc) {
        x = H[lane];
        xj = __float_as_int(H[32 + lane]);
      }
      __syncwarp();
#pragma unroll
      for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
          const float oe = __shfl_xor_sync(0xffffffffu, x, jj);
          const int oj = __shfl_xor_sync(0xffffffffu, xj, jj);
          const bool mine_first = x > oe || (x == oe && xj < oj);
          const bool take_first = ((lane & jj) == 0) == ((lane & kk) == 0);
          if (mine_first != take_first) {
            x = oe;
            xj = oj;
          }
        }
      }
      float ps = x > 0.f ? x : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, ps, o);
        if (lane >= o) ps += v;
      }
      const uint32_t reach = __ballot_sync(0xffffffffu, lane < st.nc && st.above + ps >= target);
      if (reach) {
        const int kstar = __ffs(reach) - 1;
        et = __shfl_sync(0xffffffffu, x, kstar);
        jt = __shfl_sync(0xffffffffu, xj, kstar);
        sorted = true;
      }
    }
    if (!sorted) {
      // bisection over every element in [lo, hi) (rare: many equal values, or rounding)
      uint32_t lo = ok ? st.lo : 1u, hi = ok ? st.hi : 0x3F800001u;
      while (hi - lo > 1u) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        const float tv = __uint_as_float(mid);
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < V; ++c) part += (e[c] >= tv) ? e[c] : 0.f;
        if (warp_sum(part) >= target)
          lo = mid;
        else
          hi = mid;
      }
      vstar = __uint_as_float(lo);
      // elements equal to v*: keep them in ascending key-block order until the mass reaches target
      float abovev = 0.f;
      int nties = 0;
#pragma unroll
      for (int c = 0; c < V; ++c) {
        abovev += (e[c] > vstar) ? e[c] : 0.f;
        nties += (e[c] == vstar && (lane + 32 * c) < nvalid) ? 1 : 0;
      }
      nties = warp_sum_i(nties);
      float cumv = warp_sum(abovev);
      if (nties > 0) {
#pragma unroll
        for (int c = 0; c < V; ++c) {
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
  }
  uint8_t *mrow = a.mask + row * a.nkb;
#pragma unroll
  for (int c = 0; c < V; ++c) {
    const int j = lane + 32 * c;
    if (j < nvalid) {
      const bool topk_keep =
          sorted ? (e[c] > et || (e[c] == et && j <= jt)) : (e[c] > vstar || ((tiekeep >> c) & 1ull));
      mrow[j] = (keep_all || topk_keep || sKrow[j] < a.theta) ? 1 : 0;
    }
  }
  for (int j = nvalid + lane; j < a.nkb; j += 32) mrow[j] = 0;  // causally hidden blocks
}

template <int VMAX>
__global__ void __launch_bounds__(WARPS * 32) score_select_kernel(SelArgs a) {
  __shared__ float hist[WARPS][NBIN * 32];  // per warp: [bin][lane]; reused for the short lists
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * WARPS + w;
  if (row >= a.rows) return;
  const int i = static_cast<int>(row % a.nqb);
  const int64_t bh = row / a.nqb;
  const int h = static_cast<int>(bh % a.Hq), b = static_cast<int>(bh / a.Hq);
  const int kvh = h / a.G;
  const int nvalid = a.causal ? min(a.nkb, 2 * i + 2) : a.nkb;
  const float *srow = a.S + row * a.nkb_pad;
  const float *sKrow = a.sK + (static_cast<int64_t>(b) * a.Hkv + kvh) * a.nkb_pad;
  // the fewest registers per lane that cover this row's valid blocks
  if (VMAX == 8 || nvalid <= 256) {
    select_row<8>(a, hist[w], lane, row, nvalid, srow, sKrow);
  } else if (VMAX == 16 || nvalid <= 512) {
    select_row<(VMAX >= 16 ? 16 : 8)>(a, hist[w], lane, row, nvalid, srow, sKrow);
  } else if (VMAX == 32 || nvalid <= 1024) {
    select_row<(VMAX >= 32 ? 32 : 8)>(a, hist[w], lane, row, nvalid, srow, sKrow);
  } else {
    select_row<VMAX>(a, hist[w], lane, row, nvalid, srow, sKrow);
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
