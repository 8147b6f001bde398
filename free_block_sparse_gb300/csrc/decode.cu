// Decoding tiles, the kernels around the attention kernel: the list of key blocks that the
// attention CTAs share out, and the combination of their partial rows (SpargeAttention overview
// page, "Strengths": the sparse kernel stands in for attention in any model, decoding included).
#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

// The key blocks that any of the G heads of a (batch, KV head) keeps, in ascending order, for the
// decoding tiles to share out evenly (one CTA of 1024 threads per (batch, KV head), a flag per
// thread, the heads' flags read four at a time; query block 0 of each head's mask, the only one a
// decoding call has).
constexpr int UNION_THREADS = 1024;
__global__ void __launch_bounds__(UNION_THREADS) decode_union_kernel(const uint8_t *mask, int Hq, int Hkv, int nqb,
                                                                     int nkb, int32_t *list, int *count) {
  __shared__ int wcount[UNION_THREADS / 32];
  const int bk = blockIdx.x, b = bk / Hkv, kvh = bk % Hkv, G = Hq / Hkv;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint8_t *m0 = mask + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(kvh) * G) * nqb * nkb;
  const int64_t gstride = static_cast<int64_t>(nqb) * nkb;
  int32_t *out = list + static_cast<int64_t>(bk) * nkb;
  int base = 0;
  for (int j0 = 0; j0 < nkb; j0 += UNION_THREADS) {
    const int j = j0 + static_cast<int>(threadIdx.x);
    uint32_t f = 0u;
    for (int g0 = 0; g0 < G; g0 += 4) {
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = (j < nkb && g0 + u < G) ? __ldg(m0 + (g0 + u) * gstride + j) : 0u;
      f |= v[0] | v[1] | v[2] | v[3];
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, f != 0u);
    if (lane == 0) wcount[w] = __popc(bal);
    __syncthreads();
    int off = base, tot = 0;
    for (int u = 0; u < UNION_THREADS / 32; ++u) {
      off += u < w ? wcount[u] : 0;
      tot += wcount[u];
    }
    if (f != 0u) out[off + __popc(bal & ((1u << lane) - 1u))] = j;
    base += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) count[bk] = base;
}

// The partial rows of a decoding call's chunks combined into the output: one CTA of D threads per
// output row (b, h, qi).  The chunks' exponent references and row sums are staged in shared
// memory, the largest reference M and the weights 2^(m_c - M) found by the first warp, then
// thread t sums channel t over the chunks (coalesced rows of the partial outputs, the first 64
// chunks' values loaded into registers before the weights are known):
// O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c (0 where no chunk saw a visible key).
constexpr int MAX_DECODE_CHUNKS = 1024;
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float *part_o, const float *part_ml, int nchunk,
                                                           int Hq, int Hkv, int Nq, __nv_bfloat16 *o, int64_t o_sb,
                                                           int64_t o_sh, int64_t o_sn) {
  constexpr int PREG = 64;  // chunks whose partial outputs a thread holds in registers
  __shared__ float wgt[MAX_DECODE_CHUNKS];
  __shared__ float lsum[MAX_DECODE_CHUNKS];
  __shared__ float inv_sum;
  const int row = blockIdx.x, t = threadIdx.x;
  const int qi = row % Nq, bh = row / Nq, h = bh % Hq, b = bh / Hq;
  const int G = Hq / Hkv, kvh = h / G, r = (h % G) * Nq + qi;
  const int64_t base = (static_cast<int64_t>(b) * Hkv + kvh) * nchunk;
  // this thread's channel of every chunk's partial output, loaded first: none of these loads
  // waits for the weights
  float po[PREG];
#pragma unroll
  for (int c = 0; c < PREG; ++c) po[c] = c < nchunk ? part_o[((base + c) * 128 + r) * D + t] : 0.f;
  for (int c = t; c < nchunk; c += D) {  // m_c where the chunk saw a visible key, else -inf; l_c
    const int64_t pr = (base + c) * 128 + r;
    const float l = part_ml[2 * pr + 1];
    wgt[c] = l > 0.f ? part_ml[2 * pr] : -INFINITY;
    lsum[c] = l;
  }
  __syncthreads();
  if (t < 32) {
    float M = -INFINITY;
    for (int c = t; c < nchunk; c += 32) M = fmaxf(M, wgt[c]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int c = t; c < nchunk; c += 32) {
      const float w = (M == -INFINITY || wgt[c] == -INFINITY) ? 0.f : exp2f(wgt[c] - M);
      wgt[c] = w;
      L = fmaf(w, lsum[c], L);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (t == 0) inv_sum = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < PREG; ++c) acc = fmaf(wgt[c < nchunk ? c : 0], po[c], acc);  // po is 0 past nchunk
#pragma unroll 4
  for (int c = PREG; c < nchunk; ++c) acc = fmaf(wgt[c], part_o[((base + c) * 128 + r) * D + t], acc);
  o[b * o_sb + h * o_sh + static_cast<int64_t>(qi) * o_sn + t] = __float2bfloat16_rn(acc * inv_sum);
}

}  // namespace

cudaError_t launch_decode_union(const uint8_t *mask, int B, int Hq, int Hkv, int nqb, int nkb, int32_t *list, int *count,
                                cudaStream_t st) {
  if (static_cast<int64_t>(B) * Hkv == 0) return cudaSuccess;
  decode_union_kernel<<<static_cast<unsigned>(static_cast<int64_t>(B) * Hkv), UNION_THREADS, 0, st>>>(mask, Hq, Hkv, nqb,
                                                                                                    nkb, list, count);
  return cudaGetLastError();
}

cudaError_t launch_decode_combine(const float *part_o, const float *part_ml, int nchunk, int B, int Hq, int Hkv, int Nq,
                                  int d, void *o, int64_t o_sb, int64_t o_sh, int64_t o_sn, cudaStream_t st) {
  if (nchunk <= 0 || nchunk > MAX_DECODE_CHUNKS || (d != 64 && d != 128)) return cudaErrorInvalidValue;
  const unsigned rows = static_cast<unsigned>(static_cast<int64_t>(B) * Hq * Nq);
  if (rows == 0) return cudaSuccess;
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(o);
  if (d == 128)
    decode_combine_kernel<128><<<rows, 128, 0, st>>>(part_o, part_ml, nchunk, Hq, Hkv, Nq, out, o_sb, o_sh, o_sn);
  else
    decode_combine_kernel<64><<<rows, 64, 0, st>>>(part_o, part_ml, nchunk, Hq, Hkv, Nq, out, o_sb, o_sh, o_sn);
  return cudaGetLastError();
}

}  // namespace sparge
