// Layout kernels: token permutation along the Hilbert curve, and the f16 copy of V.
//
// Token permutation along the Hilbert curve and its inverse (SpargeAttention summary page: a
// space-filling Hilbert-curve reordering improves token locality and sparsity for visual
// tasks).  y[:, :, t] = x[:, :, perm[t]] (gather) or y[:, :, perm[t]] = x[:, :, t] (scatter).
// A pure row copy: each group of d/8 lanes moves one token row with 16-byte loads and stores.
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
  int zero_bad;  // gather: a bad entry writes a zero row instead of leaving the row alone
  int *status;
};

// Grid (token chunks, H, B), 256 threads; each thread moves U 16-byte pieces of token rows, all
// U loads issued before the first store, so each SM keeps many bytes in flight; 32-bit index
// arithmetic within a head.  A perm entry outside 0..N-1 is never used as an address: its row is
// skipped (or, for the library's own ordered copies, written as zeros) and the device status word
// records SPARGE_ERR_INVALID_ARG.
constexpr int PERM_U = 4;

template <int D>
__global__ void __launch_bounds__(256) permute_kernel(PermArgs a) {
  constexpr int VPR = D / 8;                 // 16-byte pieces per token row
  constexpr int ROWS = PERM_U * 256 / VPR;   // token rows per CTA
  const int h = blockIdx.y, b = blockIdx.z;
  const __nv_bfloat16 *xb = a.x + b * a.xsb + h * a.xsh;
  __nv_bfloat16 *yb = a.y + b * a.ysb + h * a.ysh;
  const int t0 = blockIdx.x * ROWS;
  uint4 v[PERM_U];
  int dst[PERM_U], part[PERM_U];
#pragma unroll
  for (int u = 0; u < PERM_U; ++u) {
    const int e = threadIdx.x + u * 256;
    const int t = t0 + e / VPR;
    part[u] = e % VPR;
    dst[u] = -1;
    if (t < a.N) {
      const int p = __ldg(a.perm + t);
      if (static_cast<unsigned>(p) >= static_cast<unsigned>(a.N)) {  // not a token index: skip the row
        if (part[u] == 0) record_status(a.status, -1 /* SPARGE_ERR_INVALID_ARG */);
        if (a.zero_bad && !a.inverse) {
          dst[u] = t;
          v[u] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int src = a.inverse ? t : p;
      dst[u] = a.inverse ? p : t;
      v[u] = ld_stream_v4(xb + static_cast<int64_t>(src) * a.xsn + part[u] * 8);
    }
  }
#pragma unroll
  for (int u = 0; u < PERM_U; ++u)
    if (dst[u] >= 0) *reinterpret_cast<uint4 *>(yb + static_cast<int64_t>(dst[u]) * a.ysn + part[u] * 8) = v[u];
}

// V (bf16, any legal strides) -> contiguous f16 copy for the P.V product of the attention kernel.
// cvt.rn.satfinite: exact for |v| <= 65504 (every bf16 value in f16 range keeps its 8 significant
// bits), larger magnitudes saturate.  Grid (token chunks, H, B); each thread moves 16 bytes per
// step with streaming loads, two independent vectors in flight.  With a token order, row t of
// the copy is token perm[t] of V (an entry outside 0..N-1 gives a zero row and is reported).
template <int D>
__global__ void __launch_bounds__(256) convert_v_f16_kernel(const __nv_bfloat16 *x, int64_t sb, int64_t sh,
                                                             int64_t sn, __half *y, int N, const int32_t *perm,
                                                             int *status) {
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
    if (t[u] < N) {
      int src = t[u];
      if (perm) {
        src = __ldg(perm + t[u]);
        if (static_cast<unsigned>(src) >= static_cast<unsigned>(N)) {
          if (part[u] == 0) record_status(status, -1 /* SPARGE_ERR_INVALID_ARG */);
          v[u] = make_uint4(0, 0, 0, 0);
          continue;
        }
      }
      v[u] = ld_stream_v4(xb + static_cast<int64_t>(src) * sn + part[u] * 8);
    }
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

cudaError_t launch_convert_v_f16(const View &v, void *v16, const int32_t *perm, int *status, cudaStream_t st) {
  if (v.B * v.H * v.N == 0) return cudaSuccess;
  const int rows = 2 * 256 / static_cast<int>(v.d / 8);
  dim3 grid(static_cast<unsigned>((v.N + rows - 1) / rows), static_cast<unsigned>(v.H), static_cast<unsigned>(v.B));
  const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(v.data);
  if (v.d == 128)
    convert_v_f16_kernel<128><<<grid, 256, 0, st>>>(x, v.sb, v.sh, v.sn, static_cast<__half *>(v16), (int)v.N, perm,
                                                    status);
  else
    convert_v_f16_kernel<64><<<grid, 256, 0, st>>>(x, v.sb, v.sh, v.sn, static_cast<__half *>(v16), (int)v.N, perm,
                                                   status);
  return cudaGetLastError();
}

cudaError_t launch_permute(const View &x, const int32_t *perm, void *y, int64_t ysb, int64_t ysh, int64_t ysn,
                           bool inverse, int *status, cudaStream_t st, bool zero_bad) {
  PermArgs a;
  a.x = static_cast<const __nv_bfloat16 *>(x.data);
  a.y = static_cast<__nv_bfloat16 *>(y);
  a.perm = perm;
  a.xsb = x.sb; a.xsh = x.sh; a.xsn = x.sn;
  a.ysb = ysb; a.ysh = ysh; a.ysn = ysn;
  a.B = static_cast<int>(x.B); a.H = static_cast<int>(x.H); a.N = static_cast<int>(x.N);
  a.inverse = inverse ? 1 : 0;
  a.zero_bad = zero_bad ? 1 : 0;
  a.status = status;
  if (x.B * x.H * x.N == 0) return cudaSuccess;
  const int rows = PERM_U * 256 / static_cast<int>(x.d / 8);
  dim3 grid(static_cast<unsigned>((x.N + rows - 1) / rows), static_cast<unsigned>(x.H), static_cast<unsigned>(x.B));
  if (x.d == 128)
    permute_kernel<128><<<grid, 256, 0, st>>>(a);
  else
    permute_kernel<64><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sparge
