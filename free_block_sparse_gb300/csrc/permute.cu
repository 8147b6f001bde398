// Token permutation along the Hilbert curve and its inverse (SpargeAttention summary page: a
// space-filling Hilbert-curve reordering improves token locality and sparsity for visual
// tasks).  y[:, :, t] = x[:, :, perm[t]] (gather) or y[:, :, perm[t]] = x[:, :, t] (scatter).
// A pure row copy: each group of d/8 lanes moves one token row with 16-byte loads and stores;
// a grid-stride loop over all (b, h, t) rows.
#include "common.cuh"
#include "kernels.h"

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

}  // namespace

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
