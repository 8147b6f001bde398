// Stage 1b, part 2: row softmax of the pooled scores, cumulative top-k and the always-keep rule,
// written as the uint8 block mask (SpargeAttention summary page: non-similar blocks are always
// computed; overview page "Strengths": mask of shape (B, H, ceil(N/128), ceil(N/64)); Chinese
// README quick start: topk = 0.5 keeps the top 50% of the attention weights).
//
// One warp per mask row.  Lane l handles the key blocks 128 t + 4 l .. 128 t + 4 l + 3 of each
// 128-block stretch t, so every global access is 16 bytes per lane and the mask goes out as
// 32-bit words.  The row maximum comes from the score kernel; every pass re-reads the row (from
// L2 after the first) and recomputes e_j = exp(s_j - max) with the same expression, so no row
// buffer limits how many warps an SM holds.  The first pass sums Z and builds a 32-bin
// histogram of the mass over the bit pattern of e (bins ordered by value, lane-private columns in
// shared memory, no shared counters).  With the kept set defined as the shortest prefix, in (e desc, index asc)
// order, whose mass reaches topk * Z, the bin where the cumulative mass first reaches the target
// holds the cut.  Its elements are compacted into a short list (ballot offsets); further 32-bin
// levels split the list until at most 32 remain, which one warp-wide bitonic sort orders
// exactly.  Elements more than log2(n / (1 - topk)) + 0.1 below the maximum (in log2 units) never
// reach the cut (the elements from the cut down carry more than (1 - topk) Z, so the cut value is
// at least (1 - topk) Z / n >= (1 - topk) / n), so they stay out of the histogram.  A bisection
// over the whole row, with an index-ordered tie rule, covers the rare rows the levels cannot
// split (many equal values, or rounding).  The last pass writes the mask: kept by the cut, or the
// whole row when s_Q < theta, or the column when s_K < theta; causally hidden blocks are 0.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

constexpr int WARPS = 8;
constexpr int NBIN = 32;
constexpr int CMAX = 256;  // crossing-bin elements compacted into the short list (8 per lane)

struct SelArgs {
  const float *S, *Smax;  // Smax: smax_splits slices of `rows` row maxima
  int smax_splits;
  int64_t smax_stride;
  const float *sQ, *sK;
  uint8_t *mask;
  int64_t nkb_pad, rows;
  int Hq, Hkv, G, nqb, nkb, causal, off;  // off = Nk - Nq (causal alignment)
  float topk, theta;
  const float *topk_h, *theta_h;  // per query head, or nullptr
  int *status;
  int count_mode;  // 0: keep the shortest prefix reaching topk of the mass; 1: keep ceil(topk * n) blocks
  int or_into;     // OR the row into the mask already written (the second half of the hybrid rule)
};

constexpr float LOG2E = 1.4426950408889634f;

// e of the key blocks j0 .. j0 + 3 of a row (`none` past the valid blocks: 0 for the mass
// reading, -1 for the count reading, where an e of 0 is still a block to count); every pass uses
// this one expression, so the values agree bit for bit between passes.  s - max is exact zero
// for the maximum, and the hardware exponential is clamped at 1, so e <= 1 always.
// The loads and the exponentials are split (load_s, to_e) so that the row passes can load the
// next 4 blocks while they work on these; load_e is the two together.
__device__ __forceinline__ float4 load_s(const float *srow, int j0, int nvalid) {
  return j0 < nvalid ? __ldg(reinterpret_cast<const float4 *>(srow + j0)) : make_float4(0.f, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ float4 to_e(const float4 v, int j0, int nvalid, float negm, float none) {
  float4 e = make_float4(none, none, none, none);
  if (j0 < nvalid) {
    const float2 l2 = make_float2(LOG2E, LOG2E), nm = make_float2(negm, negm);
    const float2 a = fmul2(fadd2(make_float2(v.x, v.y), nm), l2);
    const float2 b = fmul2(fadd2(make_float2(v.z, v.w), nm), l2);
    e.x = fminf(fast_exp2(a.x), 1.f);
    e.y = j0 + 1 < nvalid ? fminf(fast_exp2(a.y), 1.f) : none;
    e.z = j0 + 2 < nvalid ? fminf(fast_exp2(b.x), 1.f) : none;
    e.w = j0 + 3 < nvalid ? fminf(fast_exp2(b.y), 1.f) : none;
  }
  return e;
}
// to_e for a stretch that lies wholly inside the valid blocks (a warp-uniform case: no per-block
// range checks; the same expression, so the same values)
__device__ __forceinline__ float4 to_e_full(const float4 v, float negm) {
  const float2 l2 = make_float2(LOG2E, LOG2E), nm = make_float2(negm, negm);
  const float2 a = fmul2(fadd2(make_float2(v.x, v.y), nm), l2);
  const float2 b = fmul2(fadd2(make_float2(v.z, v.w), nm), l2);
  return make_float4(fminf(fast_exp2(a.x), 1.f), fminf(fast_exp2(a.y), 1.f), fminf(fast_exp2(b.x), 1.f),
                     fminf(fast_exp2(b.y), 1.f));
}
__device__ __forceinline__ float4 load_e(const float *srow, int j0, int nvalid, float negm, float none = 0.f) {
  float4 e = make_float4(none, none, none, none);
  if (j0 < nvalid) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(srow + j0));
    const float2 l2 = make_float2(LOG2E, LOG2E), nm = make_float2(negm, negm);
    const float2 a = fmul2(fadd2(make_float2(v.x, v.y), nm), l2);
    const float2 b = fmul2(fadd2(make_float2(v.z, v.w), nm), l2);
    e.x = fminf(fast_exp2(a.x), 1.f);
    e.y = j0 + 1 < nvalid ? fminf(fast_exp2(a.y), 1.f) : none;
    e.z = j0 + 2 < nvalid ? fminf(fast_exp2(b.x), 1.f) : none;
    e.w = j0 + 3 < nvalid ? fminf(fast_exp2(b.y), 1.f) : none;
  }
  return e;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
// x has a bit pattern in [lo, hi) (patterns of e >= 0 are ordered like the values; -1, the
// count reading's mark for an invalid block, has the sign bit and is never inside)
__device__ __forceinline__ bool in_range(float x, uint32_t lo, uint32_t hi) {
  return __float_as_uint(x) - lo < hi - lo;
}
__device__ __forceinline__ float comp(const float4 &v, int u) {
  return u == 0 ? v.x : (u == 1 ? v.y : (u == 2 ? v.z : v.w));
}

// The search state: bit patterns [lo, hi) hold the cut (mass(e >= lo) >= target > mass(e >= hi)),
// `above` is the mass of the elements >= hi, `nc` the number of elements in [lo, hi).
struct Cut {
  uint32_t lo, hi;
  float above;
  int nc, shift;
};

__device__ __forceinline__ void hist_zero(float *H, int lane) {
#pragma unroll
  for (int k = 0; k < NBIN; ++k) H[k * 32 + lane] = 0.f;
  __syncwarp();
}
// 32 bins of 2^shift patterns from hi - 1 down, lane-private column; each element adds its mass
// e (mass reading) or 1 (count reading, cnt).  With d = hi - 1 - bits, x is in [lo, hi) and in
// one of the 32 bins exactly when d < lim = min(hi - lo, 32 << shift).
__device__ __forceinline__ uint32_t hist_lim(const Cut &st) {
  const uint32_t w = st.hi - st.lo, b = static_cast<uint32_t>(NBIN) << st.shift;
  return w < b ? w : b;
}
__device__ __forceinline__ void hist_add(float *H, int lane, float x, const Cut &st, uint32_t lim, bool cnt) {
  const uint32_t d = st.hi - 1u - __float_as_uint(x);
  if (d < lim) H[(d >> st.shift) * 32 + lane] += cnt ? 1.f : x;
}
__device__ __forceinline__ void hist_add4(float *H, int lane, const float4 &v, const Cut &st, uint32_t lim,
                                          bool cnt) {
  hist_add(H, lane, v.x, st, lim, cnt);
  hist_add(H, lane, v.y, st, lim, cnt);
  hist_add(H, lane, v.z, st, lim, cnt);
  hist_add(H, lane, v.w, st, lim, cnt);
}
// Narrows the state to the bin where the cumulative mass first reaches target (st.nc is left for
// the caller to recount).  Returns false (state unchanged) if rounding left no bin reaching it.
__device__ __forceinline__ bool hist_pick(float *H, int lane, float target, Cut &st) {
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
  st.shift -= 5;
  return true;
}

// Appends the elements of e (4 per lane, key blocks j0 .. j0 + 3) inside [lo, hi) to the short
// list Lv/Lj at slots n, n + 1, ... (any order; slots >= CMAX are dropped); returns the new count.
__device__ __forceinline__ int list_append(const float4 &e, int j0, const Cut &st, float *Lv, int *Lj, int n,
                                           int lane) {
  bool f[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) f[u] = in_range(comp(e, u), st.lo, st.hi);
  if (!__any_sync(0xffffffffu, f[0] || f[1] || f[2] || f[3])) return n;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint32_t bb = __ballot_sync(0xffffffffu, f[u]);
    const int slot = n + __popc(bb & lt);
    if (f[u] && slot < CMAX) {
      Lv[slot] = comp(e, u);
      Lj[slot] = j0 + u;
    }
    n += __popc(bb);
  }
  return n;
}

__global__ void __launch_bounds__(WARPS * 32, 4) score_select_kernel(SelArgs a) {
  __shared__ float sel_smem[WARPS][NBIN * 32 + 2 * CMAX];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 32-bit row arithmetic (the host keeps rows below 2^31): the divisions below are per row
  const uint32_t row = blockIdx.x * WARPS + w;
  if (row >= static_cast<uint32_t>(a.rows)) return;
  float *H = sel_smem[w];                        // histogram [bin][lane]
  float *Lv = H + NBIN * 32;                     // short list: values
  int *Lj = reinterpret_cast<int *>(Lv + CMAX);  // and key-block indices

  const uint32_t bh = row / static_cast<uint32_t>(a.nqb);
  const int i = static_cast<int>(row - bh * static_cast<uint32_t>(a.nqb));
  const uint32_t b = bh / static_cast<uint32_t>(a.Hq);
  const int h = static_cast<int>(bh - b * static_cast<uint32_t>(a.Hq));
  const int kvh = h / a.G;
  const int nvalid = a.causal ? min(a.nkb, causal_key_blocks(i, a.off)) : a.nkb;
  const int nit = (nvalid + 127) >> 7;
  const float *srow = a.S + static_cast<int64_t>(row) * a.nkb_pad;
  const float *sKrow = a.sK + (static_cast<int64_t>(b) * a.Hkv + kvh) * a.nkb_pad;
  float smax = a.Smax[row];
  for (int z = 1; z < a.smax_splits; ++z) smax = fmaxf(smax, a.Smax[z * a.smax_stride + row]);
  const float negm = -smax;
  // this head's parameters; an entry out of range keeps every valid block of the head
  float topk = a.topk, theta = a.theta;
  bool bad = false;
  if (a.topk_h) {
    const float t = a.topk_h[h];
    if (t > 0.f && t <= 1.f) topk = t; else { topk = 1.f; bad = true; }
  }
  if (a.theta_h) {
    const float th = a.theta_h[h];
    if (isfinite(th)) theta = th; else { theta = INFINITY; bad = true; }
  }
  if (bad && lane == 0) record_status(a.status, -1 /* SPARGE_ERR_INVALID_ARG */);

  // The count reading keeps kc = ceil(topk * nvalid) blocks (a 1e-3 allowance below each integer
  // keeps fp32 rounding of the product from adding a block), at least one: the cut is taken on
  // block counts instead of mass, over every e in [0, 1] (an e that underflows to 0 still counts).
  const bool cnt = a.count_mode != 0;
  const float none = cnt ? -1.f : 0.f;
  int kc = 0;
  if (cnt) kc = min(nvalid, max(1, static_cast<int>(ceilf(topk * static_cast<float>(nvalid) - 1e-3f))));
  const bool keep_all = topk >= 1.f || a.sQ[row] < theta || (cnt && kc >= nvalid);
  Cut st;
  st.lo = cnt ? 0u : 1u;
  st.hi = 0x3F800001u;  // e <= 1: the maximum gives exactly 1
  st.above = 0.f;
  st.nc = 0x7fffffff;
  st.shift = 16;
  if (!keep_all) {
    if (cnt) {
      st.shift = 25;  // 32 bins of 2^25 patterns cover [0, 1]
    } else {
      const float r2 = log2f(static_cast<float>(nvalid) / (1.f - topk)) + 0.1f;
      while (static_cast<float>(NBIN) * exp2f(static_cast<float>(st.shift - 23)) < r2) ++st.shift;
    }
    hist_zero(H, lane);
  }
  // the mask row: 4 key blocks per lane, 32-bit stores when the rows are 4-byte aligned
  uint8_t *mrow = a.mask + static_cast<int64_t>(row) * a.nkb;
  const bool words = (a.nkb & 3) == 0 && (reinterpret_cast<uintptr_t>(a.mask) & 3u) == 0;
  auto put_word = [&](int j0, uint32_t word) {
    if (j0 >= a.nkb) return;
    if (words) {
      uint32_t *dst = reinterpret_cast<uint32_t *>(mrow + j0);
      *dst = a.or_into ? (*dst | word) : word;
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (j0 + u < a.nkb) {
          const uint8_t bt = static_cast<uint8_t>(word >> (8 * u));
          mrow[j0 + u] = a.or_into ? static_cast<uint8_t>(mrow[j0 + u] | bt) : bt;
        }
    }
  };
  // first pass (rows not kept whole): Z (mass reading) and the first histogram level
  float2 z2 = make_float2(0.f, 0.f);
  if (!keep_all) {
    const uint32_t lim1 = hist_lim(st);
    float4 sn = load_s(srow, 4 * lane, nvalid);  // one stretch of 128 blocks loaded ahead
    for (int t = 0; t < nit; ++t) {
      const int j0 = 128 * t + 4 * lane;
      const float4 sv = sn;
      if (t + 1 < nit) sn = load_s(srow, j0 + 128, nvalid);
      const bool full = 128 * t + 128 <= nvalid;  // the whole stretch is valid (warp-uniform)
      const float4 v = full ? to_e_full(sv, negm) : to_e(sv, j0, nvalid, negm, none);
      if (!cnt) z2 = fadd2(z2, fadd2(make_float2(v.x, v.y), make_float2(v.z, v.w)));
      hist_add4(H, lane, v, st, lim1, cnt);
    }
  }
  const float Z = warp_sum(z2.x + z2.y);

  // the cut: keep e > et, or e == et with index <= jt
  float et = 2.f;
  int jt = -1;
  bool mask_done = false;  // the row was written by the last compaction pass and patched
  if (!keep_all) {
    const float target = cnt ? static_cast<float>(kc) : topk * Z;
    bool ok = hist_pick(H, lane, target, st);
    bool listed = false;
    // compact the crossing bin; while it does not fit the short list, split it over the row.
    // Each compaction pass also writes the mask row as far as the range decides it: blocks above
    // [lo, hi) are kept, blocks below it dropped, blocks inside it kept only by the s_K rule
    // until the cut among them is known (patched below).
    while (ok) {
      int n = 0;
      // the scores and the key blocks' similarities, both loaded one stretch ahead (s_K has
      // nkb_pad >= j0 + 4 entries per row)
      float4 sn = load_s(srow, 4 * lane, nvalid);
      float4 kn = load_s(sKrow, 4 * lane, nvalid);
      for (int t = 0; t < nit; ++t) {
        const int j0 = 128 * t + 4 * lane;
        const float4 sv = sn, sk = kn;
        if (t + 1 < nit) {
          sn = load_s(srow, j0 + 128, nvalid);
          kn = load_s(sKrow, j0 + 128, nvalid);
        }
        const bool full = 128 * t + 128 <= nvalid;  // the whole stretch is valid (warp-uniform)
        const float4 v = full ? to_e_full(sv, negm) : to_e(sv, j0, nvalid, negm, none);
        n = list_append(v, j0, st, Lv, Lj, n, lane);
        uint32_t word = 0u;
        if (full) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const bool keep = __float_as_uint(comp(v, u)) >= st.hi || comp(sk, u) < theta;
            word |= (keep ? 1u : 0u) << (8 * u);
          }
        } else if (j0 < nvalid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const bool keep = j0 + u < nvalid && (__float_as_uint(comp(v, u)) >= st.hi || comp(sk, u) < theta);
            word |= (keep ? 1u : 0u) << (8 * u);
          }
        }
        put_word(j0, word);
      }
      st.nc = n;
      if (n <= CMAX) {
        listed = true;
        break;
      }
      if (st.shift < 0) break;
      hist_zero(H, lane);
      const uint32_t lim = hist_lim(st);
      for (int t = 0; t < nit; ++t)
        hist_add4(H, lane, load_e(srow, 128 * t + 4 * lane, nvalid, negm, none), st, lim, cnt);
      ok = hist_pick(H, lane, target, st);
    }
    bool sorted = false;
    if (listed) {
      __syncwarp();
      float ce[CMAX / 32];
      int cj[CMAX / 32];
#pragma unroll
      for (int k = 0; k < CMAX / 32; ++k) {
        const int idx = lane + 32 * k;
        ce[k] = idx < st.nc ? Lv[idx] : none;
        cj[k] = idx < st.nc ? Lj[idx] : 0x7fffffff;
      }
      __syncwarp();
      // split the list in registers until at most 32 candidates remain
      while (ok && st.nc > 32 && st.shift >= 0) {
        hist_zero(H, lane);
        const uint32_t lim = hist_lim(st);
#pragma unroll
        for (int k = 0; k < CMAX / 32; ++k) hist_add(H, lane, ce[k], st, lim, cnt);
        ok = hist_pick(H, lane, target, st);
        if (ok) {
          int cnt = 0;
#pragma unroll
          for (int k = 0; k < CMAX / 32; ++k) cnt += in_range(ce[k], st.lo, st.hi) ? 1 : 0;
          st.nc = warp_sum_i(cnt);
        }
      }
      if (ok && st.nc <= 32) {
        // one candidate per lane, sorted by (e desc, index asc); the first prefix reaching target
        int n = 0;
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int k = 0; k < CMAX / 32; ++k) {
          const bool f = in_range(ce[k], st.lo, st.hi);
          const uint32_t bb = __ballot_sync(0xffffffffu, f);
          if (f) {
            Lv[n + __popc(bb & lt)] = ce[k];
            Lj[n + __popc(bb & lt)] = cj[k];
          }
          n += __popc(bb);
        }
        __syncwarp();
        float x = -1.f;
        int xj = 0x7fffffff;
        if (lane < st.nc) {
          x = Lv[lane];
          xj = Lj[lane];
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
        float ps = cnt ? (lane < st.nc ? 1.f : 0.f) : (x > 0.f ? x : 0.f);
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
          // the listed blocks the cut keeps (the compaction pass left them to the s_K rule)
          __syncwarp();
#pragma unroll
          for (int k = 0; k < CMAX / 32; ++k)
            if (cj[k] != 0x7fffffff && (ce[k] > et || (ce[k] == et && cj[k] <= jt))) mrow[cj[k]] = 1;
          mask_done = true;
        }
      }
    }
    if (!sorted) {
      // bisection over the whole row for v* = the largest value with mass(e >= v*) >= target
      // each element weighs its mass, or 1 in the count reading (tv >= 0 leaves out the -1 marks)
      auto wt = [&](float x, bool in) { return in ? (cnt ? 1.f : x) : 0.f; };
      uint32_t lo = cnt ? 0u : 1u, hi = 0x3F800001u;
      while (hi - lo > 1u) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        const float tv = __uint_as_float(mid);
        float part = 0.f;
        for (int t = 0; t < nit; ++t) {
          const float4 v = load_e(srow, 128 * t + 4 * lane, nvalid, negm, none);
          part += wt(v.x, v.x >= tv) + wt(v.y, v.y >= tv) + wt(v.z, v.z >= tv) + wt(v.w, v.w >= tv);
        }
        if (warp_sum(part) >= target)
          lo = mid;
        else
          hi = mid;
      }
      et = __uint_as_float(lo);
      // elements equal to v* are kept in ascending key-block order until the mass reaches target
      float above = 0.f;
      for (int t = 0; t < nit; ++t) {
        const float4 v = load_e(srow, 128 * t + 4 * lane, nvalid, negm, none);
        above += wt(v.x, v.x > et) + wt(v.y, v.y > et) + wt(v.z, v.z > et) + wt(v.w, v.w > et);
      }
      float cum = warp_sum(above);
      jt = -1;
      for (int t = 0; t < nit && cum < target; ++t) {
        const int j0 = 128 * t + 4 * lane;
        const float4 v = load_e(srow, j0, nvalid, negm, none);
        int mine = 0;  // ties held by this lane
#pragma unroll
        for (int u = 0; u < 4; ++u) mine += (comp(v, u) == et && j0 + u < nvalid) ? 1 : 0;
        int upto = mine;  // ties of this stretch up to and including this lane (index order)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, upto, o);
          if (lane >= o) upto += x;
        }
        const int total = __shfl_sync(0xffffffffu, upto, 31);
        // ties still needed to bring the mass to target
        const int take = cnt ? static_cast<int>(target - cum) : max(1, static_cast<int>(ceilf((target - cum) / et)));
        if (take <= total) {
          const int first = upto - mine;  // ties before this lane
          int jsel = -1;
          if (take > first && take <= upto) {
            int c = first;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (comp(v, u) == et && j0 + u < nvalid && ++c == take) jsel = j0 + u;
          }
          jt = __reduce_max_sync(0xffffffffu, jsel);
          cum = target;
        } else {
          cum += (cnt ? 1.f : et) * static_cast<float>(total);
          jt = 128 * t + 127;  // every tie of this stretch is kept
        }
      }
    }
  }

  // the mask row where no compaction pass wrote it (rows kept whole, the bisection path); the
  // causally hidden part of the row is zero-filled
  for (int t = 0; t < nit && !mask_done; ++t) {
    const int j0 = 128 * t + 4 * lane;
    uint32_t word = 0u;
    if (j0 < nvalid) {
      const float4 v = keep_all ? make_float4(0.f, 0.f, 0.f, 0.f) : load_e(srow, j0, nvalid, negm, none);
      const float4 sk = keep_all ? v : __ldg(reinterpret_cast<const float4 *>(sKrow + j0));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        const float e = comp(v, u);
        const bool keep = j < nvalid && (keep_all || e > et || (e == et && j <= jt) || comp(sk, u) < theta);
        word |= (keep ? 1u : 0u) << (8 * u);
      }
    }
    put_word(j0, word);
  }
  const int nall = a.or_into ? 0 : (a.nkb + 127) >> 7;  // OR-ed rows: that part is zero already
  for (int t = nit; t < nall; ++t) {
    const int j0 = 128 * t + 4 * lane;
    if (j0 >= a.nkb) continue;
    if (words) {
      *reinterpret_cast<uint32_t *>(mrow + j0) = 0u;
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (j0 + u < a.nkb) mrow[j0 + u] = 0;
    }
  }
}

}  // namespace

cudaError_t launch_score_select(const PredictWs &ws, int B, int Hq, int Hkv, int Nq, int Nk, int d, float topk,
                                float theta, int causal, uint8_t *mask, const float *topk_h, const float *theta_h,
                                int *status, int count_mode, bool or_into, cudaStream_t st) {
  (void)d;
  SelArgs a;
  a.S = ws.S;
  a.Smax = ws.Smax;
  a.smax_splits = ws.smax_splits;
  a.smax_stride = ws.smax_stride;
  a.sQ = ws.sQ;
  a.sK = ws.sK;
  a.mask = mask;
  a.nkb_pad = ws.nkb_pad;
  a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv;
  a.nqb = (Nq + QBLK - 1) / QBLK;
  a.nkb = (Nk + KBLK - 1) / KBLK;
  a.causal = causal;
  a.off = Nk - Nq;
  a.rows = static_cast<int64_t>(B) * Hq * a.nqb;
  a.topk = topk;
  a.theta = theta;
  a.topk_h = topk_h;
  a.theta_h = theta_h;
  a.status = status;
  a.count_mode = count_mode;
  a.or_into = or_into ? 1 : 0;
  if (a.rows == 0) return cudaSuccess;
  if (a.rows > 0x7fffffffLL) return cudaErrorInvalidValue;  // the kernel indexes rows in 32 bits
  const int64_t grid = (a.rows + WARPS - 1) / WARPS;
  score_select_kernel<<<static_cast<unsigned>(grid), WARPS * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sparge
