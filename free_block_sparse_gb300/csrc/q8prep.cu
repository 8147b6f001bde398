// Quantisation for the 8-bit attention path (SpargeAttention overview page: SpargeAttn builds on
// SageAttention's 8-bit quantisation and outlier smoothing; abstract: "sparse and quantized
// attention").
//
//   K is smoothed by its per-(batch, KV head) token mean, K~ = K - mean_t K (a per-row constant
//   shift of the scores, which the row softmax ignores), then Q and K~ are quantised to FP8 e4m3
//   with one scale per 128-token query block and per 64-token key block (scale = max|x| / 448,
//   round to nearest even, saturating); V is quantised to e4m3 with one scale per channel
//   (max over the head's tokens), stored channel-major.  INT8 tensor-core products (tcgen05 kind::i8) are not available
//   on sm_103a, so Q.K^T also runs in e4m3 (kind::f8f6f4).
//
// Kernels: per-chunk partial sums of K (and maxima of |V| when V is quantised) per (batch, KV
// head, channel); their reduction into the K mean and the V scales; one CTA per query / key block
// for Q and K~ (block maximum, then quantise, the block held in registers); a tiled transpose for V.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

constexpr int CHUNK = 2048;    // tokens per partial of the K mean / V maximum
constexpr float E4M3_MAX = 448.f;

// grid (B*Hkv, chunks); 256 threads: 16 lanes per token (d = 128) or 8 (d = 64), 8 dims per lane;
// each lane loads U tokens (of K, and of V when its scales are wanted) before it accumulates.
constexpr int U = 4;

template <int D, bool WITH_K, bool WITH_V>
__global__ void __launch_bounds__(256) kv_partials_kernel(const __nv_bfloat16 *k, int64_t ksb, int64_t ksh,
                                                          int64_t ksn, const __nv_bfloat16 *v, int64_t vsb,
                                                          int64_t vsh, int64_t vsn, int Hkv, int N,
                                                          float *part) {
  constexpr int LPT = D / 8, TPW = 32 / LPT, TPS = 8 * TPW;
  __shared__ float red[8][2][D];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane / LPT, p = lane % LPT;
  const int bh = blockIdx.x, b = bh / Hkv, h = bh % Hkv;
  const int t0 = blockIdx.y * CHUNK, t1 = min(N, t0 + CHUNK);
  const __nv_bfloat16 *kb = k + b * ksb + h * ksh + p * 8, *vb = v + b * vsb + h * vsh + p * 8;
  float s[8], mx[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) s[c] = mx[c] = 0.f;
  for (int t = t0 + w * TPW + sub; t < t1; t += U * TPS) {
    uint4 kx[U], vx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tt = t + u * TPS;
      kx[u] = vx[u] = make_uint4(0, 0, 0, 0);  // zeros add nothing to the sum or the maximum
      if (tt < t1) {
        if (WITH_K) kx[u] = ld_stream_v4(kb + static_cast<int64_t>(tt) * ksn);
        if (WITH_V) vx[u] = ld_stream_v4(vb + static_cast<int64_t>(tt) * vsn);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t kw[4] = {kx[u].x, kx[u].y, kx[u].z, kx[u].w}, vw[4] = {vx[u].x, vx[u].y, vx[u].z, vx[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        s[2 * c] += bf16lo(kw[c]);
        s[2 * c + 1] += bf16hi(kw[c]);
        if (WITH_V) {
          mx[2 * c] = fmaxf(mx[2 * c], fabsf(bf16lo(vw[c])));
          mx[2 * c + 1] = fmaxf(mx[2 * c + 1], fabsf(bf16hi(vw[c])));
        }
      }
    }
  }
#pragma unroll
  for (int off = LPT; off < 32; off <<= 1)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      s[c] += __shfl_xor_sync(0xffffffffu, s[c], off);
      mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
    }
  if (sub == 0)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      red[w][0][p * 8 + c] = s[c];
      red[w][1][p * 8 + c] = mx[c];
    }
  __syncthreads();
  if (threadIdx.x < D) {
    float ss = 0.f, mm = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {
      ss += red[ww][0][threadIdx.x];
      mm = fmaxf(mm, red[ww][1][threadIdx.x]);
    }
    float *dst = part + (static_cast<int64_t>(bh) * gridDim.y + blockIdx.y) * 2 * D;
    dst[threadIdx.x] = ss;
    dst[D + threadIdx.x] = mm;
  }
}

// grid B*Hkv, D threads: K mean and (with_v) V scale per channel
template <int D>
__global__ void kv_finish_kernel(const float *part, int nchunks, int N, int with_v, float *kmean, float *sv) {
  const int bh = blockIdx.x, c = threadIdx.x;
  float ss = 0.f, mm = 0.f;
  for (int k = 0; k < nchunks; ++k) {
    const float *src = part + (static_cast<int64_t>(bh) * nchunks + k) * 2 * D;
    ss += src[c];
    mm = fmaxf(mm, src[D + c]);
  }
  kmean[static_cast<int64_t>(bh) * D + c] = ss / static_cast<float>(N);
  if (with_v) sv[static_cast<int64_t>(bh) * D + c] = mm > 0.f ? mm / E4M3_MAX : 1.f;
}

// One CTA of 256 threads per block of ROWS tokens, held in registers between the two steps (one
// read of the block): the block maximum of |x - mean| (mean per channel when given, else 0), the
// scale max / 448, then the e4m3 codes.  Grid: one CTA per (b h, block), x = bh * nblk + block.
// out is contiguous [B][H][N][D] bytes; scale[bh * nblk + block].
template <int D, int ROWS>
__global__ void __launch_bounds__(256) quant_block_kernel(const __nv_bfloat16 *x, int64_t sb, int64_t sh,
                                                          int64_t sn, int H, int N, int nblk,
                                                          const float *mean, uint8_t *out, float *scale) {
  constexpr int LPT = D / 8, TPC = 256 / LPT;  // tokens per CTA-wide load
  constexpr int STEPS = ROWS / TPC;
  __shared__ float red[8];
  const int bi = static_cast<int>(blockIdx.x % static_cast<unsigned>(nblk));
  const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(nblk));
  const int h = bh % H, b = bh / H;
  const int tok = threadIdx.x / LPT, p = threadIdx.x % LPT;
  const int t0 = bi * ROWS;
  float mu[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) mu[c] = mean ? mean[static_cast<int64_t>(bh) * D + p * 8 + c] : 0.f;
  const __nv_bfloat16 *base = x + b * sb + h * sh + p * 8;
  uint4 xv[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int t = t0 + s * TPC + tok;
    xv[s] = t < N ? ld_stream_v4(base + static_cast<int64_t>(t) * sn) : make_uint4(0, 0, 0, 0);
  }
  float m = 0.f;
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (t0 + s * TPC + tok >= N) continue;  // rows past N do not count (0 - mean would)
    const uint32_t wd[4] = {xv[s].x, xv[s].y, xv[s].z, xv[s].w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      m = fmaxf(m, fmaxf(fabsf(bf16lo(wd[c]) - mu[2 * c]), fabsf(bf16hi(wd[c]) - mu[2 * c + 1])));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) m = fmaxf(m, red[w]);
  const float sc = m > 0.f ? m / E4M3_MAX : 1.f;
  const float inv = 1.f / sc;
  if (threadIdx.x == 0) scale[blockIdx.x] = sc;
  uint8_t *obase = out + static_cast<int64_t>(bh) * N * D + p * 8;
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int t = t0 + s * TPC + tok;
    if (t >= N) continue;
    const uint32_t wd[4] = {xv[s].x, xv[s].y, xv[s].z, xv[s].w};
    float f[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      f[2 * c] = (bf16lo(wd[c]) - mu[2 * c]) * inv;
      f[2 * c + 1] = (bf16hi(wd[c]) - mu[2 * c + 1]) * inv;
    }
    uint2 o;
    o.x = pack_e4m3x4(f[0], f[1], f[2], f[3]);
    o.y = pack_e4m3x4(f[4], f[5], f[6], f[7]);
    *reinterpret_cast<uint2 *>(obase + static_cast<int64_t>(t) * D) = o;
  }
}

// V -> e4m3 with a scale per (batch, KV head, channel), written channel-major: out is
// [B][Hkv][D][npad] bytes (npad = N rounded up to 64, the tail zero), so that a 64-key tile is a
// K-major operand of P.V; with a token order, key t of the copy is token perm[t] of V (an entry
// outside 0..N-1 gives zero codes and is reported).  grid (B*Hkv, npad / 64), 256 threads.  Each CTA quantises one tile of
// 64 keys into shared memory token-major (coalesced 16-byte loads, all issued first; 8-byte
// stores), then each of D * 2 threads gathers 32 keys of one channel and writes them as two
// 16-byte pieces (one whole 32-byte sector).
template <int D>
__global__ void __launch_bounds__(256) quant_vt_kernel(const __nv_bfloat16 *v, int64_t sb, int64_t sh, int64_t sn,
                                                       int H, int N, int npad, const float *sv, uint8_t *out,
                                                       const int32_t *perm, int *status) {
  constexpr int VPR = D / 8;           // 16-byte input pieces per token
  constexpr int TPC = 256 / VPR;       // tokens per CTA-wide load
  constexpr int STEPS = 64 / TPC;
  __shared__ __align__(16) uint8_t tile[64][D];  // token-major codes
  const int bh = blockIdx.x, b = bh / H, h = bh % H;
  const int t0 = blockIdx.y * 64;
  const int tok = threadIdx.x / VPR, p = threadIdx.x % VPR;
  const __nv_bfloat16 *base = v + b * sb + h * sh + p * 8;
  float inv[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) inv[c] = 1.f / sv[static_cast<int64_t>(bh) * D + p * 8 + c];
  uint4 xv[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int t = t0 + s * TPC + tok;
    int src = t;
    if (perm && t < N) {
      src = __ldg(perm + t);
      if (static_cast<unsigned>(src) >= static_cast<unsigned>(N)) {
        if (p == 0) record_status(status, -1 /* SPARGE_ERR_INVALID_ARG */);
        src = N;  // read nothing: zero codes
      }
    }
    xv[s] = (t < N && src < N) ? ld_stream_v4(base + static_cast<int64_t>(src) * sn) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const uint32_t wd[4] = {xv[s].x, xv[s].y, xv[s].z, xv[s].w};
    uint2 o;
    o.x = pack_e4m3x4(bf16lo(wd[0]) * inv[0], bf16hi(wd[0]) * inv[1], bf16lo(wd[1]) * inv[2], bf16hi(wd[1]) * inv[3]);
    o.y = pack_e4m3x4(bf16lo(wd[2]) * inv[4], bf16hi(wd[2]) * inv[5], bf16lo(wd[3]) * inv[6], bf16hi(wd[3]) * inv[7]);
    *reinterpret_cast<uint2 *>(&tile[s * TPC + tok][p * 8]) = o;  // zero codes past N
  }
  __syncthreads();
  uint8_t *obase = out + static_cast<int64_t>(bh) * D * npad + t0;
  for (int e = threadIdx.x; e < D * 2; e += 256) {
    const int ch = e % D, half = e / D;  // keys 32 half .. 32 half + 31 of channel ch
    uint32_t wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = 32 * half + 4 * j;
      wv[j] = static_cast<uint32_t>(tile[r][ch]) | (static_cast<uint32_t>(tile[r + 1][ch]) << 8) |
              (static_cast<uint32_t>(tile[r + 2][ch]) << 16) | (static_cast<uint32_t>(tile[r + 3][ch]) << 24);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(obase + static_cast<int64_t>(ch) * npad + 32 * half);
    dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
  }
}

template <int D>
cudaError_t run(const View &q, const View &k, const View &v, const Q8Ws &w, bool quant_qk, bool quant_v,
                const int32_t *perm, int *status, cudaStream_t st) {
  const int B = static_cast<int>(q.B), Hq = static_cast<int>(q.H), Hkv = static_cast<int>(k.H);
  const int Nq = static_cast<int>(q.N), N = static_cast<int>(k.N);  // N: keys and values
  const int nchunks = (N + CHUNK - 1) / CHUNK;
  const dim3 pgrid(B * Hkv, nchunks);
  const __nv_bfloat16 *kp = static_cast<const __nv_bfloat16 *>(k.data), *vp = static_cast<const __nv_bfloat16 *>(v.data);
  if (quant_qk && quant_v)
    kv_partials_kernel<D, true, true><<<pgrid, 256, 0, st>>>(kp, k.sb, k.sh, k.sn, vp, v.sb, v.sh, v.sn, Hkv, N, w.partial);
  else if (quant_qk)
    kv_partials_kernel<D, true, false><<<pgrid, 256, 0, st>>>(kp, k.sb, k.sh, k.sn, vp, v.sb, v.sh, v.sn, Hkv, N, w.partial);
  else if (quant_v)  // V scales only (bf16 Q.K^T): K is not read, its mean comes out 0 and is unused
    kv_partials_kernel<D, false, true><<<pgrid, 256, 0, st>>>(kp, k.sb, k.sh, k.sn, vp, v.sb, v.sh, v.sn, Hkv, N, w.partial);
  else
    return cudaSuccess;
  kv_finish_kernel<D><<<B * Hkv, D, 0, st>>>(w.partial, nchunks, N, quant_v ? 1 : 0, w.kmean, w.sv);
  const int nqb = (Nq + QBLK - 1) / QBLK, nkb = (N + KBLK - 1) / KBLK;
  const int64_t nq = static_cast<int64_t>(B) * Hq * nqb, nk = static_cast<int64_t>(B) * Hkv * nkb;
  if (quant_qk) {
    quant_block_kernel<D, QBLK><<<static_cast<unsigned>(nq), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(q.data), q.sb, q.sh, q.sn, Hq, Nq, nqb, nullptr, w.q8, w.sq);
    quant_block_kernel<D, KBLK><<<static_cast<unsigned>(nk), 256, 0, st>>>(kp, k.sb, k.sh, k.sn, Hkv, N, nkb, w.kmean,
                                                                            w.k8, w.sk);
  }
  const int npad = (N + 63) / 64 * 64;
  if (quant_v)
    quant_vt_kernel<D><<<dim3(B * Hkv, npad / 64), 256, 0, st>>>(vp, v.sb, v.sh, v.sn, Hkv, N, npad, w.sv, w.v8, perm,
                                                              status);
  return cudaGetLastError();
}

}  // namespace

size_t q8_ws_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t N, int64_t d) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int64_t nqb = (Nq + QBLK - 1) / QBLK, nkb = (N + KBLK - 1) / KBLK, nch = (N + CHUNK - 1) / CHUNK;
  const int64_t npad = (N + 63) / 64 * 64;
  const int64_t vbytes = std::max(B * Hkv * d * npad, 2 * B * Hkv * N * d);  // e4m3 V^T or the f16 copy
  return al(B * Hq * Nq * d) + al(B * Hkv * N * d) + al(vbytes) + al(4 * B * Hq * nqb) + al(4 * B * Hkv * nkb) +
         2 * al(4 * B * Hkv * d) + al(4 * B * Hkv * nch * 2 * d);
}

Q8Ws q8_ws_carve(void *ws, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t N, int64_t d) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int64_t nqb = (Nq + QBLK - 1) / QBLK, nkb = (N + KBLK - 1) / KBLK;
  const int64_t npad = (N + 63) / 64 * 64;
  char *p = static_cast<char *>(ws);
  Q8Ws w;
  w.q8 = reinterpret_cast<uint8_t *>(p); p += al(B * Hq * Nq * d);
  w.k8 = reinterpret_cast<uint8_t *>(p); p += al(B * Hkv * N * d);
  w.v8 = reinterpret_cast<uint8_t *>(p); p += al(std::max(B * Hkv * d * npad, 2 * B * Hkv * N * d));
  w.sq = reinterpret_cast<float *>(p); p += al(4 * B * Hq * nqb);
  w.sk = reinterpret_cast<float *>(p); p += al(4 * B * Hkv * nkb);
  w.kmean = reinterpret_cast<float *>(p); p += al(4 * B * Hkv * d);
  w.sv = reinterpret_cast<float *>(p); p += al(4 * B * Hkv * d);
  w.partial = reinterpret_cast<float *>(p);
  return w;
}

cudaError_t launch_q8_prep(const View &q, const View &k, const View &v, const Q8Ws &w, bool quant_qk, bool quant_v,
                           const int32_t *perm, int *status, cudaStream_t st) {
  if (q.B * q.N == 0) return cudaSuccess;
  return q.d == 128 ? run<128>(q, k, v, w, quant_qk, quant_v, perm, status, st)
                    : run<64>(q, k, v, w, quant_qk, quant_v, perm, status, st);
}

}  // namespace sparge
