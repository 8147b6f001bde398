// Layout kernels: token permutation along the Hilbert curve, and the f16 copy of V.
//
// Token permutation along the Hilbert curve and its inverse (SpargeAttention summary page: a
// space-filling Hilbert-curve reordering improves token locality and sparsity for visual
// tasks).  y[:, :, t] = x[:, :, perm[t]] (gather) or y[:, :, perm[t]] = x[:, :, t] (scatter).
// A pure row copy: each group of d/8 lanes moves one token row with 16-byte loads and stores;
// a grid-stride loop over all (b, h, t) rows.
#include "common.cuh"
#include "kernels.h"

#include <cuda_fp16.h>

namespace sparge {
namespace {

struct PermArgs {
  const __nv_bfloat16 *x;
  __nv_bfloat16 *y;
  const int32_t *perm;
  int64_t xsb, xsh, xsn, ysb, ysh, ysn;
  int B, H, N;
  int inverse;
};

template <int D>
__global__ void __launch_bounds__(256) permute_kernel(PermArgs a) {
  constexpr int LPT = D / 8;
  constexpr int RPW = 32 / LPT;  // rows per warp per step
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPT, part = lane % LPT;
  const int64_t rows = static_cast<int64_t>(a.B) * a.H * a.N;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = warp0 * RPW + sub; r < rows; r += nwarps * RPW) {
    const int t = static_cast<int>(r % a.N);
    const int64_t bh = r / a.N;
    const int h = static_cast<int>(bh % a.H), b = static_cast<int>(bh / a.H);
    const int p = __ldg(a.perm + t);
    const int src = a.inverse ? t : p;
    const int dst = a.inverse ? p : t;
    const uint4 v = ld_stream_v4(a.x + b * a.xsb + h * a.xsh + static_cast<int64_t>(src) * a.xsn + part * 8);
    *reinterpret_cast<uint4 *>(a.y + b * a.ysb + h * a.ysh + static_cast<int64_t>(dst) * a.ysn + part * 8) = v;
  }
}

// V (bf16, any legal strides) -> contiguous f16 copy for the P.V product of the attention kernel.
// cvt.rn.satfinite: exact for |v| <= 65504 (every bf16 value in f16 range keeps its 8 significant
// bits), larger magnitudes saturate.  Grid (token chunks, H, B); each thread moves 16 bytes per
// step with streaming loads, two independent vectors in flight.
template <int D>
__global__ void __launch_bounds__(256) convert_v_f16_kernel(const __nv_bfloat16 *x, int64_t sb, int64_t sh,
                                                             int64_t sn, __half *y, int N) {
  constexpr int VPR = D / 8;                 // 16-byte vectors per token row
  constexpr int ROWS = 2 * 256 / VPR;        // token rows per CTA
  const int h = blockIdx.y, b = blockIdx.z, H = gridDim.y;
  const __nv_bfloat16 *xb = x + b * sb + h * sh;
  __half *yb = y + (static_cast<int64_t>(b) * H + h) * N * D;
  const int t0 = blockIdx.x * ROWS;
  uint4 v[2];
  int t[2], part[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int e = threadIdx.x + u * 256;
    t[u] = t0 + e / VPR;
    part[u] = e % VPR;
    if (t[u] < N) v[u] = ld_stream_v4(xb + static_cast<int64_t>(t[u]) * sn + part[u] * 8);
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (t[u] < N) {
      uint4 o;
      o.x = pack_f16x2(bf16lo(v[u].x), bf16hi(v[u].x));
      o.y = pack_f16x2(bf16lo(v[u].y), bf16hi(v[u].y));
      o.z = pack_f16x2(bf16lo(v[u].z), bf16hi(v[u].z));
      o.w = pack_f16x2(bf16lo(v[u].w), bf16hi(v[u].w));
      *reinterpret_cast<uint4 *>(yb + static_cast<int64_t>(t[u]) * D + part[u] * 8) = o;
    }
  }
}

}  // namespace

cudaError_t launch_convert_v_f16(const View &v, void *v16, cudaStream_t st) {
  if (v.B * v.H * v.N == 0) return cudaSuccess;
  const int rows = 2 * 256 / static_cast<int>(v.d / 8);
  dim3 grid(static_cast<unsigned>((v.N + rows - 1) / rows), static_cast<unsigned>(v.H), static_cast<unsigned>(v.B));
  const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(v.data);
  if (v.d == 128)
    convert_v_f16_kernel<128><<<grid, 256, 0, st>>>(x, v.sb, v.sh, v.sn, static_cast<__half *>(v16), (int)v.N);
  else
    convert_v_f16_kernel<64><<<grid, 256, 0, st>>>(x, v.sb, v.sh, v.sn, static_cast<__half *>(v16), (int)v.N);
  return cudaGetLastError();
}

cudaError_t launch_permute(const View &x, const int32_t *perm, void *y, int64_t ysb, int64_t ysh, int64_t ysn,
                           bool inverse, cudaStream_t st) {
  PermArgs a;
  a.x = static_cast<const __nv_bfloat16 *>(x.data);
  a.y = static_cast<__nv_bfloat16 *>(y);
  a.perm = perm;
  a.xsb = x.sb; a.xsh = x.sh; a.xsn = x.sn;
  a.ysb = ysb; a.ysh = ysh; a.ysn = ysn;
  a.B = static_cast<int>(x.B); a.H = static_cast<int>(x.H); a.N = static_cast<int>(x.N);
  a.inverse = inverse ? 1 : 0;
  const int64_t rows = x.B * x.H * x.N;
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int rpb = 8 * (32 / (static_cast<int>(x.d) / 8));  // rows per CTA per step
  int64_t want = (rows + rpb - 1) / rpb;
  int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 8;  // 8 resident CTAs of 256 threads per SM
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (x.d == 128)
    permute_kernel<128><<<grid, 256, 0, st>>>(a);
  else
    permute_kernel<64><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sparge
