// Stage 1a: block mean pooling and intra-block self-similarity (SpargeAttention summary page,
// method paragraph: token blocks with high internal similarity are compressed).
//
// For each 128-token query block and 64-token key block this kernel produces the fp32 mean of
// the valid tokens and s = ||(1/n) sum_a x_a / ||x_a|| ||^2, the mean cosine similarity over
// all ordered token pairs of the block (pairs a == b included).  A zero token contributes a
// zero unit vector.  Memory-bound: one pass over Q and K.  One warp per block, no block-level
// barriers, fp32 (packed pair) arithmetic, warp-shuffle reductions, vector stores of the results.
// A block's rows stream through a per-lane ring of shared-memory slots filled by cp.async well
// ahead of the arithmetic, so the bytes in flight cost no registers.  Under a token order (Hilbert
// order of image or video tokens) the rows are gathered whole through the order (the block's
// indices read once into shared memory), so the pooling needs no ordered copy of Q or K; it writes
// the ordered copies the later kernels read as it goes (the rows pass through its registers).
#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

struct PoolArgs {
  const __nv_bfloat16 *q, *k;
  int64_t q_sb, q_sh, q_sn, k_sb, k_sh, k_sn;
  int B, Hq, Hkv, Nq, Nk, nqb, nkb;  // query and key lengths may differ
  int64_t nq_total, total;
  PredictWs ws;
  const int32_t *qperm, *kperm;  // token orders (or nullptr): block row t is token perm[t]
  int *status;
  __nv_bfloat16 *qcopy, *kcopy;  // with a token order: contiguous (B, H, N, d) copies in that order
                                 // that the pooling writes as it reads the rows (or nullptr)
};

// One block's place in the inputs and outputs: block ub of the Q blocks then the K blocks
// (32-bit arithmetic: the host keeps the block count below 2^31).
struct BlockRef {
  const __nv_bfloat16 *base;  // the block's first row
  int64_t sn, row;            // row stride; the block's index in the pooled outputs
  int b, h, idx, n, rows, ntok;
  bool isQ;
};
__device__ __forceinline__ BlockRef block_ref(const PoolArgs &a, uint32_t ub) {
  BlockRef r;
  const uint32_t nqt = static_cast<uint32_t>(a.nq_total);
  r.isQ = ub < nqt;
  if (r.isQ) {
    const uint32_t bh = ub / static_cast<uint32_t>(a.nqb);
    r.idx = static_cast<int>(ub - bh * static_cast<uint32_t>(a.nqb));
    r.h = static_cast<int>(bh % static_cast<uint32_t>(a.Hq));
    r.b = static_cast<int>(bh / static_cast<uint32_t>(a.Hq));
    r.rows = QBLK;
    r.sn = a.q_sn;
    r.base = a.q + r.b * a.q_sb + r.h * a.q_sh + static_cast<int64_t>(r.idx) * QBLK * r.sn;
    r.row = (static_cast<int64_t>(r.b) * a.Hq + r.h) * a.nqb + r.idx;
    r.ntok = a.Nq;
  } else {
    const uint32_t kb = ub - nqt;
    const uint32_t bh = kb / static_cast<uint32_t>(a.nkb);
    r.idx = static_cast<int>(kb - bh * static_cast<uint32_t>(a.nkb));
    r.h = static_cast<int>(bh % static_cast<uint32_t>(a.Hkv));
    r.b = static_cast<int>(bh / static_cast<uint32_t>(a.Hkv));
    r.rows = KBLK;
    r.sn = a.k_sn;
    r.base = a.k + r.b * a.k_sb + r.h * a.k_sh + static_cast<int64_t>(r.idx) * KBLK * r.sn;
    r.row = (static_cast<int64_t>(r.b) * a.Hkv + r.h) * a.nkb + r.idx;
    r.ntok = a.Nk;
  }
  r.n = min(r.rows, r.ntok - r.idx * r.rows);
  return r;
}

// One token's 8 coordinates held by this lane (LPT lanes per token): adds them to the running
// sum and their share of the unit vector x / ||x|| (the norm from a shuffle over the LPT lanes).
template <int LPT>
__device__ __forceinline__ void pool_accumulate(const uint4 v, float2 (&sx2)[4], float2 (&sh2)[4]) {
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

// The block's results from the lanes' sums: the mean, its bf16 hi/lo split and s.
template <int D>
__device__ __forceinline__ void pool_finish(const PoolArgs &a, const BlockRef &r, int lane, float2 (&sx2)[4],
                                            float2 (&sh2)[4]) {
  constexpr int LPT = D / 8;
  const int sub = lane / LPT, part = lane % LPT;
  // sum over the token slots of the warp (lanes with the same part)
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
  const float invn = 1.f / static_cast<float>(r.n);
  float hsq = 0.f;
  if (sub == 0) {  // lanes 0..LPT-1 own dims 8 part .. 8 part + 7
    float mean[8];
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      mean[2 * c] = sx2[c].x * invn;
      mean[2 * c + 1] = sx2[c].y * invn;
      const float h0 = sh2[c].x * invn, h1 = sh2[c].y * invn;
      hsq = fmaf(h0, h0, fmaf(h1, h1, hsq));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __nv_bfloat16 a0 = __float2bfloat16_rn(mean[2 * c]), a1 = __float2bfloat16_rn(mean[2 * c + 1]);
      const __nv_bfloat16 b0 = __float2bfloat16_rn(mean[2 * c] - __bfloat162float(a0));
      const __nv_bfloat16 b1 = __float2bfloat16_rn(mean[2 * c + 1] - __bfloat162float(a1));
      hi[c] = static_cast<uint32_t>(__bfloat16_as_ushort(a0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(a1)) << 16);
      lo[c] = static_cast<uint32_t>(__bfloat16_as_ushort(b0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b1)) << 16);
    }
    float *mu = (r.isQ ? a.ws.muQ : a.ws.muK) + r.row * D + part * 8;
    *reinterpret_cast<float4 *>(mu) = make_float4(mean[0], mean[1], mean[2], mean[3]);
    *reinterpret_cast<float4 *>(mu + 4) = make_float4(mean[4], mean[5], mean[6], mean[7]);
    *reinterpret_cast<uint4 *>((r.isQ ? a.ws.qhi : a.ws.khi) + r.row * D + part * 8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4 *>((r.isQ ? a.ws.qlo : a.ws.klo) + r.row * D + part * 8) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) hsq += __shfl_xor_sync(0xffffffffu, hsq, off);
  if (lane == 0) {
    if (r.isQ)
      a.ws.sQ[r.row] = hsq;
    else
      a.ws.sK[(static_cast<int64_t>(r.b) * a.Hkv + r.h) * a.ws.nkb_pad + r.idx] = hsq;
  }
}

// The plain (unordered) pooling: each warp takes its blocks one after another and streams a
// block's rows through a ring of RING 16-byte slots per lane in shared memory, filled by cp.async
// RING warp-wide steps ahead of the arithmetic (rows past the block's valid tokens zero-filled),
// so the bytes in flight cost no registers; each lane reads back only the slots it filled.
// (Letting the ring run on into the warp's next block, with no drain at block ends, measured
// slower: 0.28 against 0.235 ms at 128K.)
constexpr int RING = 16;
template <int D>
__global__ void __launch_bounds__(128, 5) pool_stream_kernel(PoolArgs a) {
  __shared__ __align__(16) uint8_t ring_smem[4][RING * 512];
  constexpr int LPT = D / 8;     // lanes per token, 8 bf16 (16 bytes) per lane
  constexpr int TPW = 32 / LPT;  // tokens per warp-wide step
  const int lane = threadIdx.x & 31, sub = lane / LPT, part = lane % LPT;
  const uint32_t ring = smem_u32(ring_smem[threadIdx.x >> 5]) + lane * 16;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t bid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; bid < a.total;
       bid += nwarps) {
    const BlockRef r = block_ref(a, static_cast<uint32_t>(bid));
    const int steps = r.rows / TPW;
    const __nv_bfloat16 *p = r.base + sub * r.sn + part * 8;
    auto issue = [&](int s) {
      const int t = s * TPW + sub;
      const bool in = t < r.n;
      const __nv_bfloat16 *src = in ? p + static_cast<int64_t>(s) * TPW * r.sn : p;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ring + (s % RING) * 512), "l"(src),
                   "r"(in ? 16u : 0u)
                   : "memory");
    };
    // steps go in pairs (a block has an even number of steps): one group per pair
#pragma unroll
    for (int s = 0; s < RING; s += 2) {
      if (s < steps) {
        issue(s);
        issue(s + 1);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");  // one group per pair, empty or not
    }
    float2 sx2[4], sh2[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) sx2[c] = sh2[c] = make_float2(0.f, 0.f);
    for (int s = 0; s < steps; s += 2) {
      asm volatile("cp.async.wait_group %0;" ::"n"(RING / 2 - 1) : "memory");  // pair s has landed
      uint4 v0, v1;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v0.x), "=r"(v0.y), "=r"(v0.z), "=r"(v0.w)
                   : "r"(ring + (s % RING) * 512)
                   : "memory");
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v1.x), "=r"(v1.y), "=r"(v1.z), "=r"(v1.w)
                   : "r"(ring + ((s + 1) % RING) * 512)
                   : "memory");
      pool_accumulate<LPT>(v0, sx2, sh2);
      pool_accumulate<LPT>(v1, sx2, sh2);
      if (s + RING < steps) {  // into the slots just read (v0, v1 are used above)
        issue(s + RING);
        issue(s + RING + 1);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    pool_finish<D>(a, r, lane, sx2, sh2);
  }
}

// Under a token order: a block's token indices are read once into shared memory and its rows
// gathered through them into the warp's cp.async ring; the rows also go out, from registers, to
// the ordered copies the later kernels read.
template <int D>
__global__ void __launch_bounds__(128, 5) pool_gather_kernel(PoolArgs a) {
  __shared__ __align__(16) uint8_t ring_smem[4][RING * 512];
  __shared__ int sperm[4][QBLK];  // the block's token indices, per warp
  constexpr int LPT = D / 8;     // lanes per token, 8 bf16 (16 bytes) per lane
  constexpr int TPW = 32 / LPT;  // tokens per warp-wide load
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPT, part = lane % LPT;
  const uint32_t ring = smem_u32(ring_smem[threadIdx.x >> 5]) + lane * 16;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t bid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; bid < a.total;
       bid += nwarps) {
    const BlockRef r = block_ref(a, static_cast<uint32_t>(bid));
    const int n = r.n, steps = r.rows / TPW;  // warp-wide steps covering the block
    const __nv_bfloat16 *p = r.base + sub * r.sn + part * 8;
    // the block's row t is token perm[t] of the head (gathered whole rows)
    const int32_t *perm = r.isQ ? a.qperm : a.kperm;
    const __nv_bfloat16 *hbase = r.base - static_cast<int64_t>(r.idx) * r.rows * r.sn + part * 8;
    int *wperm = sperm[(threadIdx.x >> 5) & 3];
    // the block's rows of the ordered copy (this lane's 16 bytes of row 0), when one is wanted
    __nv_bfloat16 *cpy = nullptr;
    __nv_bfloat16 *cbase = r.isQ ? a.qcopy : a.kcopy;
    if (cbase != nullptr)
      cpy = cbase + ((static_cast<int64_t>(r.b) * (r.isQ ? a.Hq : a.Hkv) + r.h) * r.ntok +
                     static_cast<int64_t>(r.idx) * r.rows) * D + part * 8;
    if (perm != nullptr) {  // one coalesced read of the block's indices; bad ones become -1
      __syncwarp();  // every lane is done with the previous block's indices
      for (int u = lane; u < n; u += 32) {
        const int src = __ldg(perm + r.idx * r.rows + u);
        const bool good = static_cast<unsigned>(src) < static_cast<unsigned>(r.ntok);
        if (!good) record_status(a.status, -1 /* SPARGE_ERR_INVALID_ARG */);
        wperm[u] = good ? src : -1;
      }
      __syncwarp();
    }
    // the rows (gathered through the order, or in place) through the warp's cp.async ring, as in
    // pool_stream_kernel; entries outside the order's range read as zero rows
    auto issue = [&](int s) {
      const int t = s * TPW + sub;
      const __nv_bfloat16 *src = p;
      bool in = t < n;
      if (in) {
        if (perm == nullptr) {
          src = p + static_cast<int64_t>(s) * TPW * r.sn;
        } else {
          const int g = wperm[t];
          in = g >= 0;
          src = in ? hbase + static_cast<int64_t>(g) * r.sn : p;
        }
      }
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ring + (s % RING) * 512), "l"(src),
                   "r"(in ? 16u : 0u)
                   : "memory");
    };
#pragma unroll
    for (int s = 0; s < RING; ++s) {
      if (s < steps) issue(s);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    float2 sx2[4], sh2[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) sx2[c] = sh2[c] = make_float2(0.f, 0.f);
    for (int s = 0; s < steps; ++s) {
      asm volatile("cp.async.wait_group %0;" ::"n"(RING - 1) : "memory");
      uint4 v;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(ring + (s % RING) * 512)
                   : "memory");
      const int t = s * TPW + sub;
      if (cpy != nullptr && t < n) *reinterpret_cast<uint4 *>(cpy + static_cast<int64_t>(t) * D) = v;
      pool_accumulate<LPT>(v, sx2, sh2);
      if (s + RING < steps) issue(s + RING);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    pool_finish<D>(a, r, lane, sx2, sh2);
  }
}

}  // namespace

cudaError_t launch_pool_sim(const View &q, const View &k, const PredictWs &ws, cudaStream_t st, const int32_t *qperm,
                            const int32_t *kperm, int *status, void *qcopy, void *kcopy) {
  PoolArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(q.data);
  a.k = static_cast<const __nv_bfloat16 *>(k.data);
  a.q_sb = q.sb; a.q_sh = q.sh; a.q_sn = q.sn;
  a.k_sb = k.sb; a.k_sh = k.sh; a.k_sn = k.sn;
  a.B = static_cast<int>(q.B); a.Hq = static_cast<int>(q.H); a.Hkv = static_cast<int>(k.H);
  a.Nq = static_cast<int>(q.N);
  a.Nk = static_cast<int>(k.N);
  a.nqb = (a.Nq + QBLK - 1) / QBLK;
  a.nkb = (a.Nk + KBLK - 1) / KBLK;
  a.nq_total = static_cast<int64_t>(a.B) * a.Hq * a.nqb;
  a.total = a.nq_total + static_cast<int64_t>(a.B) * a.Hkv * a.nkb;
  a.ws = ws;
  a.qperm = qperm;
  a.kperm = kperm;
  a.status = status;
  a.qcopy = qperm ? static_cast<__nv_bfloat16 *>(qcopy) : nullptr;
  a.kcopy = kperm ? static_cast<__nv_bfloat16 *>(kcopy) : nullptr;
  if (a.total == 0) return cudaSuccess;
  if (a.total > 0x7fffffffLL) return cudaErrorInvalidValue;  // the kernel's block arithmetic is 32-bit
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (a.total + 3) / 4;
  const bool gather = qperm != nullptr || kperm != nullptr;
  // 5 resident CTAs of 4 warps per SM (33-35 KB of ring and indices each)
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 5;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (q.d == 128) {
    if (gather)
      pool_gather_kernel<128><<<grid, 128, 0, st>>>(a);
    else
      pool_stream_kernel<128><<<grid, 128, 0, st>>>(a);
  } else {
    if (gather)
      pool_gather_kernel<64><<<grid, 128, 0, st>>>(a);
    else
      pool_stream_kernel<64><<<grid, 128, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace sparge
