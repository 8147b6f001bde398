// Stage 1b, part 1: the pooled score map S = scale * muQ . muK^T (SpargeAttention abstract: the
// attention map is predicted from a compressed Q and K).  A batched GEMM per head on tcgen05:
// M = 128 query blocks, N = 128 key blocks per chunk, K = d.  The fp32 means are carried as bf16
// hi/lo pairs and multiplied as hi.hi + hi.lo + lo.hi with fp32 accumulation, which keeps about
// 16 significant bits (relative error ~1e-5, far inside the 1e-3 decision margins of the mask).
// Only chunks holding valid (causal) key blocks are computed.  One CTA per (128 query blocks,
// head); warp 4 loads operands by TMA (Q once, K chunks into a 2-stage ring), warp 5 issues the
// MMAs into two TMEM accumulators, warps 0-3 move each finished accumulator to S: each thread
// owns one row, scales it, keeps the maximum over the row's valid key blocks, and writes it in
// 32-column quarters into the K stage the chunk's MMAs have just finished with (128-byte
// swizzle), from where one thread stores the quarters to S by TMA (whole 128-byte lines instead
// of one 16-byte piece per row per instruction).  The stage goes back to the producer once the
// stores have read it.  The row maxima go to Smax for the selection.
#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

constexpr int GROWS = 128;  // query blocks per CTA (MMA M)
constexpr int GCOLS = 128;  // key blocks per chunk (MMA N)

struct GemmArgs {
  float *Smax;
  int64_t nkb_pad, smax_stride;
  int B, Hq, Hkv, G, nqb, nkb, causal, off, ngroups;  // off = Nk - Nq (causal alignment)
  int per_split;  // key chunks per split (blockIdx.z): split z takes chunks [z per_split, ...)
  float scale;
  int *status;
};

template <int D>
struct GL {
  static constexpr int KCH = D / 64;                     // 64-wide k chunks (128-byte rows)
  static constexpr uint32_t OP_BYTES = KCH * 128 * 128;  // one 128-row bf16 operand
  static constexpr uint32_t OFF_QHI = 0;
  static constexpr uint32_t OFF_QLO = OP_BYTES;
  static constexpr uint32_t OFF_K = 2 * OP_BYTES;        // stage s: hi at OFF_K + 2 s OP_BYTES, lo after it
  static constexpr int KST = 2;
  static constexpr uint32_t STAGE_BYTES = 2 * OP_BYTES;  // K hi + lo; reused to stage S quarters
  static constexpr int QPR = STAGE_BYTES / 16384 < 4 ? STAGE_BYTES / 16384 : 4;  // 16 KB quarters per round
  static constexpr int ROUNDS = 4 / QPR;
  static constexpr uint32_t OFF_CTRL = OFF_K + KST * STAGE_BYTES;
  static constexpr uint32_t TOTAL = OFF_CTRL + 256;
};

struct GCtrl {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    score_gemm_kernel(const __grid_constant__ CUtensorMap tqh, const __grid_constant__ CUtensorMap tql,
                      const __grid_constant__ CUtensorMap tkh, const __grid_constant__ CUtensorMap tkl,
                      const __grid_constant__ CUtensorMap ts, const GemmArgs a) {
  using L = GL<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_status(a.status, -4 /* SPARGE_ERR_CUDA */);
    return;
  }
  GCtrl &cs = *reinterpret_cast<GCtrl *>(smem + L::OFF_CTRL);
  volatile int *abort = &cs.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int group = a.ngroups - 1 - static_cast<int>(blockIdx.y);  // longest causal rows first
  const int bh = blockIdx.x, b = bh / a.Hq, h = bh % a.Hq, kvh = h / a.G;
  const int i0 = group * GROWS;
  const int ilast = min(i0 + GROWS - 1, a.nqb - 1);
  const int ncols = a.causal ? min(a.nkb, causal_key_blocks(ilast, a.off)) : a.nkb;
  // this CTA's key chunks [ch0, ch0 + nch) of the group's (ncols + 127) / 128
  const int ch0 = static_cast<int>(blockIdx.z) * a.per_split;
  const int nch = max(0, min((ncols + GCOLS - 1) / GCOLS - ch0, a.per_split));
  constexpr uint32_t IDESC = idesc_f32acc(128, GCOLS, FMT_BF16, false);

  if (threadIdx.x == 0) {
    mbar_init(&cs.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&cs.k_full[s], 1);
      mbar_init(&cs.k_empty[s], 2);  // the chunk's MMAs, and the S stores out of the stage
      mbar_init(&cs.acc_full[s], 1);
      mbar_init(&cs.acc_empty[s], 128);
    }
    mbar_init(&cs.final_bar, 1);
    cs.abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&cs.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cs.tmem_base;

  if (warp == 4) {
    if (lane == 0 && nch > 0) {
      mbar_arrive_expect_tx(&cs.q_full, 2 * L::OP_BYTES);
      for (int c = 0; c < L::KCH; ++c) {
        tma_load_3d(smem + L::OFF_QHI + c * 16384, &tqh, &cs.q_full, 64 * c, i0, bh);
        tma_load_3d(smem + L::OFF_QLO + c * 16384, &tql, &cs.q_full, 64 * c, i0, bh);
      }
      for (int ch = 0; ch < nch; ++ch) {
        const int st = ch % L::KST;
        if (!mbar_wait(&cs.k_empty[st], ((ch / L::KST) & 1) ^ 1, abort, a.status)) break;
        uint8_t *kh = smem + L::OFF_K + st * 2 * L::OP_BYTES;
        uint8_t *kl = kh + L::OP_BYTES;
        mbar_arrive_expect_tx(&cs.k_full[st], 2 * L::OP_BYTES);
        for (int c = 0; c < L::KCH; ++c) {
          tma_load_3d(kh + c * 16384, &tkh, &cs.k_full[st], 64 * c, GCOLS * (ch0 + ch), b * a.Hkv + kvh);
          tma_load_3d(kl + c * 16384, &tkl, &cs.k_full[st], 64 * c, GCOLS * (ch0 + ch), b * a.Hkv + kvh);
        }
      }
      if (*abort) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0 && nch > 0 && mbar_wait(&cs.q_full, 0, abort, a.status)) {
      tc_fence_after();
      const uint32_t qh = smem_u32(smem + L::OFF_QHI), ql = smem_u32(smem + L::OFF_QLO);
      for (int ch = 0; ch < nch; ++ch) {
        const int st = ch % L::KST, ab = ch & 1;
        if (!mbar_wait(&cs.k_full[st], (ch / L::KST) & 1, abort, a.status)) break;
        if (!mbar_wait(&cs.acc_empty[ab], ((ch >> 1) & 1) ^ 1, abort, a.status)) break;
        tc_fence_after();
        const uint32_t kh = smem_u32(smem + L::OFF_K + st * 2 * L::OP_BYTES), kl = kh + L::OP_BYTES;
        const uint32_t acc = tmem + ab * GCOLS;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
          const uint64_t dqh = smem_desc_sw128(qh + off, 16, 1024), dql = smem_desc_sw128(ql + off, 16, 1024);
          const uint64_t dkh = smem_desc_sw128(kh + off, 16, 1024), dkl = smem_desc_sw128(kl + off, 16, 1024);
          mma_bf16_ss(acc, dqh, dkh, IDESC, s > 0 ? 1u : 0u);
          mma_bf16_ss(acc, dqh, dkl, IDESC, 1u);
          mma_bf16_ss(acc, dql, dkh, IDESC, 1u);
        }
        mma_commit(&cs.k_empty[st]);
        mma_commit(&cs.acc_full[ab]);
      }
      mma_commit(&cs.final_bar);
      mbar_wait(&cs.final_bar, 0, abort, a.status);
    }
    __syncwarp();
  } else {
    const int r = warp * 32 + lane;
    const int i = i0 + r;
    const int nv = (i < a.nqb) ? (a.causal ? min(a.nkb, causal_key_blocks(i, a.off)) : a.nkb) : 0;  // valid key blocks
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float rmax = -3.402823466e38f;
    for (int ch = 0; ch < nch; ++ch) {
      const int ab = ch & 1, st = ch % L::KST;
      // all 128 epilogue threads leave together if any wait gave up (they meet at named barriers)
      const bool ok = mbar_wait(&cs.acc_full[ab], (ch >> 1) & 1, abort, a.status);
      if (bar_red_or(1, 128, !ok)) break;
      tc_fence_after();
      uint8_t *stage = smem + L::OFF_K + st * L::STAGE_BYTES;  // free: the chunk's MMAs are done
      for (int rd = 0; rd < L::ROUNDS; ++rd) {
        if (rd > 0) {  // the previous round's stores must have read the stage
          if (threadIdx.x == 0) bulk_wait_read_all();
          bar_sync(1, 128);
        }
#pragma unroll 1
        for (int qq = 0; qq < L::QPR; ++qq) {
          const int q = rd * L::QPR + qq;
          uint32_t v[32];
          tmem_ld32(tl + ab * GCOLS + 32 * q, v);
          tmem_ld_wait();
          const int j0 = GCOLS * (ch0 + ch) + 32 * q;
          uint8_t *row = stage + qq * 16384 + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float4 o;
            o.x = __uint_as_float(v[4 * c]) * a.scale;
            o.y = __uint_as_float(v[4 * c + 1]) * a.scale;
            o.z = __uint_as_float(v[4 * c + 2]) * a.scale;
            o.w = __uint_as_float(v[4 * c + 3]) * a.scale;
            const int j = j0 + 4 * c;
            if (j < nv) rmax = fmaxf(rmax, o.x);
            if (j + 1 < nv) rmax = fmaxf(rmax, o.y);
            if (j + 2 < nv) rmax = fmaxf(rmax, o.z);
            if (j + 3 < nv) rmax = fmaxf(rmax, o.w);
            *reinterpret_cast<float4 *>(row + ((c ^ (r & 7)) << 4)) = o;
          }
        }
        if (rd == L::ROUNDS - 1) {  // this thread's TMEM reads of the accumulator are done
          tc_fence_before();
          mbar_arrive(&cs.acc_empty[ab]);
        }
        fence_proxy_async_smem();
        bar_sync(1, 128);
        if (threadIdx.x == 0) {
          for (int qq = 0; qq < L::QPR; ++qq)
            tma_store_3d(&ts, stage + qq * 16384, GCOLS * (ch0 + ch) + 32 * (rd * L::QPR + qq), i0, bh);
          bulk_commit();
        }
      }
      if (threadIdx.x == 0) {  // the stage returns to the producer once the stores have read it
        bulk_wait_read_all();
        mbar_arrive(&cs.k_empty[st]);
      }
    }
    if (threadIdx.x == 0) bulk_wait_all();
    if (i < a.nqb) a.Smax[blockIdx.z * a.smax_stride + static_cast<int64_t>(bh) * a.nqb + i] = rmax;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 256);
}

// The few-row path: S[row][j] = scale * muQ[row] . muK[j] in fp32 for the valid key blocks of
// each row, one CTA per (row, 256 key blocks) and one key block per thread: the row's mean is
// staged in shared memory (read as a broadcast), each thread streams its block's mean as D / 4
// independent 16-byte loads into four FMA chains, and the threads' scores go out as one
// coalesced row; the CTA's maximum over its valid blocks goes to its own Smax slice.
template <int D>
__global__ void __launch_bounds__(256) score_rows_kernel(const float *__restrict__ muQ, const float *__restrict__ muK,
                                                         float *S, float *Smax, int64_t smax_stride, int64_t nkb_pad,
                                                         int Hq, int Hkv, int nqb, int nkb, int causal, int off,
                                                         float scale) {
  __shared__ float4 qs[D / 4];
  __shared__ float wmax[8];
  const int row = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = row / nqb, i = row - bh * nqb, b = bh / Hq, h = bh - b * Hq, kvh = h / (Hq / Hkv);
  const int nvalid = causal ? min(nkb, causal_key_blocks(i, off)) : nkb;
  if (threadIdx.x < D / 4) qs[threadIdx.x] = __ldg(reinterpret_cast<const float4 *>(muQ + static_cast<int64_t>(row) * D) + threadIdx.x);
  __syncthreads();
  const int j = static_cast<int>(blockIdx.y) * 256 + static_cast<int>(threadIdx.x);
  float m = -3.402823466e38f;
  if (j < nvalid) {
    const float4 *kr = reinterpret_cast<const float4 *>(muK + ((static_cast<int64_t>(b) * Hkv + kvh) * nkb + j) * D);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < D / 4; ++u) {
      const float4 kv = __ldg(kr + u), qv = qs[u];
      float a = acc[u & 3];
      a = fmaf(qv.x, kv.x, a);
      a = fmaf(qv.y, kv.y, a);
      a = fmaf(qv.z, kv.z, a);
      a = fmaf(qv.w, kv.w, a);
      acc[u & 3] = a;
    }
    const float sc = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * scale;
    S[static_cast<int64_t>(row) * nkb_pad + j] = sc;
    m = sc;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wmax[w] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = wmax[0];
    for (int u = 1; u < 8; ++u) mm = fmaxf(mm, wmax[u]);
    Smax[blockIdx.y * smax_stride + row] = mm;
  }
}

template <int D>
cudaError_t launch_d(const ScoreGemmLaunch &l, const GemmArgs &a, cudaStream_t st) {
  const uint32_t smem = GL<D>::TOTAL;
  static std::atomic<unsigned long long> smem_set{0};
  if (cudaError_t e = set_smem_limit_once(score_gemm_kernel<D>, static_cast<int>(smem), smem_set); e != cudaSuccess) return e;
  const int nch_all = (a.nkb + GCOLS - 1) / GCOLS;
  dim3 grid(static_cast<unsigned>(a.B * a.Hq), static_cast<unsigned>(a.ngroups),
            static_cast<unsigned>((nch_all + a.per_split - 1) / a.per_split));
  score_gemm_kernel<D><<<grid, 192, smem, st>>>(l.qhi, l.qlo, l.khi, l.klo, l.ts, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_gemm(const ScoreGemmLaunch &l, cudaStream_t st) {
  GemmArgs a;
  a.Smax = l.Smax;
  a.nkb_pad = l.nkb_pad;
  a.smax_stride = l.smax_stride;
  a.B = l.B; a.Hq = l.Hq; a.Hkv = l.Hkv; a.G = l.Hq / l.Hkv;
  a.nqb = (l.Nq + QBLK - 1) / QBLK;
  a.nkb = (l.Nk + KBLK - 1) / KBLK;
  a.causal = l.causal;
  a.off = l.Nk - l.Nq;
  a.ngroups = (a.nqb + GROWS - 1) / GROWS;
  a.scale = l.scale;
  a.status = l.status;
  {
    const int nch_all = (a.nkb + GCOLS - 1) / GCOLS, sp = l.splits > 0 ? l.splits : 1;
    a.per_split = (nch_all + sp - 1) / sp;
    if (a.per_split < 1) a.per_split = 1;
    if ((nch_all + a.per_split - 1) / a.per_split > sp) return cudaErrorInvalidValue;  // more slices than Smax has
  }
  if (static_cast<int64_t>(a.B) * a.Hq * a.ngroups == 0) return cudaSuccess;
  if (score_use_rows(l.B, l.Hq, l.Nq)) {
    const int64_t rows = static_cast<int64_t>(a.B) * a.Hq * a.nqb;
    const unsigned zs = static_cast<unsigned>((a.nkb + 255) / 256);
    if (static_cast<int>(zs) != l.splits || !l.muQ || !l.muK || !l.S) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(rows), zs);
    if (l.d == 128)
      score_rows_kernel<128><<<grid, 256, 0, st>>>(l.muQ, l.muK, l.S, a.Smax, a.smax_stride, a.nkb_pad, a.Hq, a.Hkv,
                                                   a.nqb, a.nkb, a.causal, a.off, a.scale);
    else
      score_rows_kernel<64><<<grid, 256, 0, st>>>(l.muQ, l.muK, l.S, a.Smax, a.smax_stride, a.nkb_pad, a.Hq, a.Hkv,
                                                  a.nqb, a.nkb, a.causal, a.off, a.scale);
    return cudaGetLastError();
  }
  return l.d == 128 ? launch_d<128>(l, a, st) : launch_d<64>(l, a, st);
}

}  // namespace sparge
