// Stage 1a: block mean pooling and intra-block self-similarity (SpargeAttention summary page,
// method paragraph: token blocks with high internal similarity are compressed).
//
// For each 128-token query block and 64-token key block this kernel produces the fp32 mean of
// the valid tokens and s = ||(1/n) sum_a x_a / ||x_a|| ||^2, the mean cosine similarity over
// all ordered token pairs of the block (pairs a == b included).  A zero token contributes a
// zero unit vector.  Memory-bound: one pass over Q and K.  One persistent CTA per SM: a producer
// warp streams blocks by TMA into a deep shared-memory ring (so enough bytes are in flight to keep
// HBM busy), eight consumer warps reduce each block from shared memory with fp32 (packed pair)
// arithmetic and warp shuffles, then split the finishing work of the block among themselves.
#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

struct PoolArgs {
  int B, Hq, Hkv, N, nqb, nkb;
  int64_t nq_total, total;
  PredictWs ws;
  int *status;
};

template <int D>
struct PL {
  static constexpr int NST = D == 128 ? 6 : 10;         // ring stages
  static constexpr uint32_t STAGE = QBLK * D * 2;        // room for one query block
  static constexpr uint32_t OFF_RED = NST * STAGE;       // [8 warps][2][D] partial sums
  static constexpr uint32_t OFF_REDS = OFF_RED + 8 * 2 * D * 4;
  static constexpr uint32_t OFF_CTRL = OFF_REDS + 64;
  static constexpr uint32_t TOTAL = OFF_CTRL + 256;
};

struct PCtrl {
  uint64_t full[10], empty[10];
  int abort;
};

struct BlockRef {
  bool isQ;
  int b, h, idx;  // batch, head, block index within the head
  int n;          // valid tokens
};

__device__ __forceinline__ BlockRef block_ref(const PoolArgs &a, int64_t bid) {
  BlockRef r;
  r.isQ = bid < a.nq_total;
  if (r.isQ) {
    r.idx = static_cast<int>(bid % a.nqb);
    const int64_t bh = bid / a.nqb;
    r.h = static_cast<int>(bh % a.Hq);
    r.b = static_cast<int>(bh / a.Hq);
    r.n = min(QBLK, a.N - r.idx * QBLK);
  } else {
    bid -= a.nq_total;
    r.idx = static_cast<int>(bid % a.nkb);
    const int64_t bh = bid / a.nkb;
    r.h = static_cast<int>(bh % a.Hkv);
    r.b = static_cast<int>(bh / a.Hkv);
    r.n = min(KBLK, a.N - r.idx * KBLK);
  }
  return r;
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(288, 1)
    pool_sim_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const PoolArgs a) {
  using L = PL<D>;
  constexpr int LPT = D / 8;     // lanes per token, 8 bf16 (16 bytes) per lane
  constexpr int TPW = 32 / LPT;  // tokens per warp per step
  constexpr int TPS = 8 * TPW;   // tokens per step of the 8 consumer warps
  constexpr int NBOX = D / 64;   // 64-column boxes per token row
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_status(a.status, -4 /* SPARGE_ERR_CUDA */);
    return;
  }
  PCtrl &cs = *reinterpret_cast<PCtrl *>(smem + L::OFF_CTRL);
  float(*red)[2][D] = reinterpret_cast<float(*)[2][D]>(smem + L::OFF_RED);
  float *red_s = reinterpret_cast<float *>(smem + L::OFF_REDS);
  volatile int *abort = &cs.abort;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < L::NST; ++st) {
      mbar_init(&cs.full[st], 1);
      mbar_init(&cs.empty[st], 1);
    }
    cs.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (w == 8) {
    // ------------------------------- producer: TMA into the ring -------------------------------
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      int k = 0;
      for (int64_t bid = blockIdx.x; bid < a.total; bid += gridDim.x, ++k) {
        const int st = k % L::NST;
        if (!mbar_wait(&cs.empty[st], ((k / L::NST) & 1) ^ 1, abort, a.status)) break;
        const BlockRef r = block_ref(a, bid);
        const int rows = r.isQ ? QBLK : KBLK;
        uint8_t *dst = smem + st * L::STAGE;
        mbar_arrive_expect_tx(&cs.full[st], static_cast<uint32_t>(rows * D * 2));
        for (int bx = 0; bx < NBOX; ++bx)
          tma_load_4d(dst + bx * rows * 128, r.isQ ? &tq : &tk, &cs.full[st], 64 * bx, rows * r.idx, r.h, r.b);
      }
      if (*abort) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
    return;
  }

  // ------------------------------- consumers: 8 warps -------------------------------
  const int sub = lane / LPT, part = lane % LPT;
  const int bx = part >> 3, chunk = part & 7;
  int k = 0;
  for (int64_t bid = blockIdx.x; bid < a.total; bid += gridDim.x, ++k) {
    const int st = k % L::NST;
    // after a timeout the wait returns at once and the data is stale, but every consumer warp
    // still takes part in the barriers below, so none of them can hang
    mbar_wait(&cs.full[st], (k / L::NST) & 1, abort, a.status);
    const BlockRef r = block_ref(a, bid);
    const int rows = r.isQ ? QBLK : KBLK;
    const uint8_t *src = smem + st * L::STAGE + bx * rows * 128;
    float2 sx2[4], sh2[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) sx2[c] = sh2[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int step = 0; step < QBLK / TPS; ++step) {
      const int t = step * TPS + w * TPW + sub;
      if (t < rows) {  // rows past the valid tokens were zero-filled by TMA and add nothing
        const uint4 v = *reinterpret_cast<const uint4 *>(src + t * 128 + ((chunk ^ (t & 7)) << 4));
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
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
    if (sub == 0) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        red[w][0][part * 8 + 2 * c] = sx2[c].x;
        red[w][0][part * 8 + 2 * c + 1] = sx2[c].y;
        red[w][1][part * 8 + 2 * c] = sh2[c].x;
        red[w][1][part * 8 + 2 * c + 1] = sh2[c].y;
      }
    }
    consumer_sync();
    if (threadIdx.x == 0) mbar_arrive(&cs.empty[st]);  // every consumer is done with this stage
    {
      constexpr int DPW = D / 8;
      const float invn = 1.f / static_cast<float>(r.n);
      float hsq = 0.f;
      if (lane < DPW) {
        const int dim = w * DPW + lane;
        float mx = 0.f, hx = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) {
          mx += red[ww][0][dim];
          hx += red[ww][1][dim];
        }
        hx *= invn;
        hsq = hx * hx;
        const float mean = mx * invn;
        const int64_t row = r.isQ ? (static_cast<int64_t>(r.b) * a.Hq + r.h) * a.nqb + r.idx
                                  : (static_cast<int64_t>(r.b) * a.Hkv + r.h) * a.nkb + r.idx;
        float *mu = (r.isQ ? a.ws.muQ : a.ws.muK) + row * D;
        uint16_t *hi = (r.isQ ? a.ws.qhi : a.ws.khi) + row * D;
        uint16_t *lo = (r.isQ ? a.ws.qlo : a.ws.klo) + row * D;
        mu[dim] = mean;
        const __nv_bfloat16 hb = __float2bfloat16_rn(mean);
        hi[dim] = __bfloat16_as_ushort(hb);
        lo[dim] = __bfloat16_as_ushort(__float2bfloat16_rn(mean - __bfloat162float(hb)));
      }
#pragma unroll
      for (int off = DPW / 2; off > 0; off >>= 1) hsq += __shfl_xor_sync(0xffffffffu, hsq, off);
      if (lane == 0) red_s[w] = hsq;
    }
    consumer_sync();
    if (threadIdx.x == 0) {
      float sv = 0.f;
#pragma unroll
      for (int ww = 0; ww < 8; ++ww) sv += red_s[ww];
      if (r.isQ)
        a.ws.sQ[(static_cast<int64_t>(r.b) * a.Hq + r.h) * a.nqb + r.idx] = sv;
      else
        a.ws.sK[(static_cast<int64_t>(r.b) * a.Hkv + r.h) * a.ws.nkb_pad + r.idx] = sv;
    }
  }
}

template <int D>
cudaError_t launch_d(const CUtensorMap &tq, const CUtensorMap &tk, const PoolArgs &a, cudaStream_t st) {
  const uint32_t smem = PL<D>::TOTAL;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(pool_sim_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = sms > 0 ? sms : 152;  // one persistent CTA per SM
  const unsigned grid = static_cast<unsigned>(a.total < cap ? a.total : cap);
  pool_sim_kernel<D><<<grid, 288, smem, st>>>(tq, tk, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pool_sim(const View &q, const View &k, const CUtensorMap &tq, const CUtensorMap &tk,
                            const PredictWs &ws, int *status, cudaStream_t st) {
  PoolArgs a;
  a.B = static_cast<int>(q.B); a.Hq = static_cast<int>(q.H); a.Hkv = static_cast<int>(k.H);
  a.N = static_cast<int>(q.N);
  a.nqb = (a.N + QBLK - 1) / QBLK;
  a.nkb = (a.N + KBLK - 1) / KBLK;
  a.nq_total = static_cast<int64_t>(a.B) * a.Hq * a.nqb;
  a.total = a.nq_total + static_cast<int64_t>(a.B) * a.Hkv * a.nkb;
  a.ws = ws;
  a.status = status;
  if (a.total == 0) return cudaSuccess;
  return q.d == 128 ? launch_d<128>(tq, tk, a, st) : launch_d<64>(tq, tk, a, st);
}

}  // namespace sparge
