// C-ABI layer of libsparge: argument validation, workspace layout, TMA descriptor creation,
// the device status word and kernel launches.  Every entry point is declared (and its
// arguments documented) in include/sparge.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/sparge.h"
#include "common.cuh"
#include "kernels.h"

using namespace sparge;

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char *where) {
  return fail(SPARGE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// One status word per process in device memory (a __device__ variable, not an allocation);
// kernels record a timed-out bounded wait there.
__device__ int g_status_word = 0;

// One thread waits on an mbarrier that nothing arrives on, through the same bounded wait the
// attention and score kernels use; the wait runs out after limit_ns and records a timeout.
__global__ void bounded_wait_probe_kernel(int *status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
}

int *status_ptr() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int *>(p);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int check_tensor(const sparge_tensor *t, const char *name, View *v) {
  if (!t) return fail(SPARGE_ERR_INVALID_ARG, "%s is NULL", name);
  if (!t->data && t->B * t->H * t->N != 0) return fail(SPARGE_ERR_INVALID_ARG, "%s->data is NULL", name);
  if (t->dtype != SPARGE_BF16) return fail(SPARGE_ERR_UNSUPPORTED, "%s: only bf16 is supported", name);
  if (t->d != 64 && t->d != 128) return fail(SPARGE_ERR_UNSUPPORTED, "%s: head dim %lld not in {64,128}", name, (long long)t->d);
  if (t->B < 0 || t->H <= 0 || t->N < 0)
    return fail(SPARGE_ERR_INVALID_ARG, "%s: bad shape B=%lld H=%lld N=%lld", name, (long long)t->B,
                (long long)t->H, (long long)t->N);
  if (t->N > (int64_t(1) << 30) || t->B * t->H > (int64_t(1) << 24) || t->B > 65535 || t->H > 65535)
    return fail(SPARGE_ERR_UNSUPPORTED, "%s: shape too large", name);
  if ((reinterpret_cast<uintptr_t>(t->data) & 15u) != 0)
    return fail(SPARGE_ERR_INVALID_ARG, "%s: data not 16-byte aligned", name);
  int64_t sb = t->stride_b, sh = t->stride_h, sn = t->stride_n;
  // strides of unit dimensions do not matter; give them a harmless legal value
  if (t->N == 1) sn = t->d;
  if (t->H == 1) sh = sn * (t->N > 0 ? t->N : 1);
  if (t->B == 1) sb = sh * t->H;
  if (sn < t->d || sh <= 0 || sb <= 0 || sn % 8 || sh % 8 || sb % 8)
    return fail(SPARGE_ERR_INVALID_ARG, "%s: strides (%lld,%lld,%lld) must be positive multiples of 8 with stride_n >= d",
                name, (long long)t->stride_b, (long long)t->stride_h, (long long)t->stride_n);
  *v = View{t->data, t->B, t->H, t->N, t->d, sb, sh, sn};
  return SPARGE_OK;
}

// q may be shorter (or, without the causal mask, longer) than k; the causal case is checked where
// the mask kind is known (check_lengths).
int check_qk(const View &q, const View &k) {
  if (k.B != q.B || k.d != q.d)
    return fail(SPARGE_ERR_INVALID_ARG, "q and k disagree in B or d");
  if (q.H % k.H != 0) return fail(SPARGE_ERR_UNSUPPORTED, "Hq=%lld not a multiple of Hkv=%lld", (long long)q.H, (long long)k.H);
  return SPARGE_OK;
}

// Causal attention with Nq != Nk puts the last query on the last key, so it needs Nq <= Nk; a
// call with queries needs keys.
int check_lengths(const View &q, const View &k, int causal) {
  if (causal && q.N > k.N)
    return fail(SPARGE_ERR_INVALID_ARG, "causal attention needs Nq <= Nk (got %lld > %lld)", (long long)q.N,
                (long long)k.N);
  if (q.N > 0 && k.N == 0) return fail(SPARGE_ERR_INVALID_ARG, "k and v have no tokens");
  return SPARGE_OK;
}

typedef CUresult (*encode_fn_t)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

encode_fn_t get_encode() {
  static encode_fn_t fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<encode_fn_t>(p);
  });
  return fn;
}

int make_map(CUtensorMap *m, const View &v, int box_rows, const char *name,
             CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  encode_fn_t enc = get_encode();
  if (!enc) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[4] = {(cuuint64_t)v.d, (cuuint64_t)v.N, (cuuint64_t)v.H, (cuuint64_t)v.B};
  cuuint64_t strides[3] = {(cuuint64_t)v.sn * 2, (cuuint64_t)v.sh * 2, (cuuint64_t)v.sb * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, dt, 4, const_cast<void *>(v.data), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return SPARGE_OK;
}

// 3-D map over a contiguous bf16 array [planes][rows][d], box 64 columns x 128 rows, 128-byte swizzle.
int make_map3(CUtensorMap *m, void *base, int64_t d, int64_t rows, int64_t planes, const char *name) {
  encode_fn_t enc = get_encode();
  if (!enc) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)(rows * d * 2)};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return SPARGE_OK;
}

// 4-D map over a byte array (e4m3 codes): dims and byte strides innermost first, box
// box0 x box1, the given swizzle.
int make_map_u8(CUtensorMap *m, void *base, const int64_t dims_[4], const int64_t strides_[3], int box0, int box1,
                CUtensorMapSwizzle swz, const char *name) {
  encode_fn_t enc = get_encode();
  if (!enc) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[4], strides[3];
  for (int i = 0; i < 4; ++i) dims[i] = (cuuint64_t)dims_[i];
  for (int i = 0; i < 3; ++i) strides[i] = (cuuint64_t)strides_[i];
  cuuint32_t box[4] = {(cuuint32_t)box0, (cuuint32_t)box1, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return SPARGE_OK;
}

// 3-D map over the fp32 pooled scores [planes][rows][nkb_pad] for TMA stores: box 32 columns
// (128 bytes) x 128 rows, 128-byte swizzle.
int make_map_s(CUtensorMap *m, float *base, int64_t nkb_pad, int64_t rows, int64_t planes) {
  encode_fn_t enc = get_encode();
  if (!enc) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[3] = {(cuuint64_t)nkb_pad, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)nkb_pad * 4, (cuuint64_t)(rows * nkb_pad * 4)};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPARGE_ERR_CUDA, "cuTensorMapEncodeTiled(S) failed with %d", (int)r);
  return SPARGE_OK;
}

int check_topk_theta(float topk, float theta) {
  if (!(topk > 0.f && topk <= 1.f)) return fail(SPARGE_ERR_INVALID_ARG, "topk=%g not in (0, 1]", (double)topk);
  if (!std::isfinite(theta)) return fail(SPARGE_ERR_INVALID_ARG, "theta must be finite");
  return SPARGE_OK;
}

int check_lambda(float lambda) {
  if (std::isnan(lambda) || lambda > 0.f) return fail(SPARGE_ERR_INVALID_ARG, "lambda=%g must be <= 0 or -inf", (double)lambda);
  return SPARGE_OK;
}

// Records timing event `idx` of `ev` (an array of 6 cudaEvent_t, or nullptr) on stream s.
int record_event(void *const *ev, int idx, cudaStream_t s) {
  if (!ev || !ev[idx]) return SPARGE_OK;
  cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(ev[idx]), s);
  return e == cudaSuccess ? SPARGE_OK : cuda_fail(e, "timing event record");
}

size_t order_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d) {
  return align256((size_t)2 * B * Hq * N * d) + align256((size_t)2 * B * Hkv * N * d);
}

// Calls with a token order: places copies of q and/or k in that order at the front of the
// workspace (contiguous (B, H, N, d) bf16), replaces them by the copies and moves ws past the space
// of both (the space is reserved whether or not a copy is made).  With launch the copies are made
// here by permute kernels; without it the caller has them written by another kernel (the pooling
// of mask prediction, which reads every row through the order anyway).  A tensor that is not
// copied is read through the permutation by the kernels instead (pooling, and the d = 64
// attention's Q rows).
int order_qk(View &q, View &k, const int32_t *perm, void *&ws, size_t &ws_bytes, cudaStream_t s, bool copy_q = true,
             bool copy_k = true, bool launch = true) {
  const size_t need = order_bytes(q.B, q.H, k.H, q.N, q.d);
  if (!ws || ws_bytes < need)
    return fail(SPARGE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu for the token-ordered copies", ws_bytes,
                need);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(SPARGE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  uint8_t *base = static_cast<uint8_t *>(ws);
  void *qc = base, *kc = base + align256((size_t)2 * q.B * q.H * q.N * q.d);
  cudaError_t e = cudaSuccess;
  if (launch && copy_q) e = launch_permute(q, perm, qc, q.H * q.N * q.d, q.N * q.d, q.d, false, status_ptr(), s, true);
  if (launch && e == cudaSuccess && copy_k)
    e = launch_permute(k, perm, kc, k.H * k.N * k.d, k.N * k.d, k.d, false, status_ptr(), s, true);
  if (e != cudaSuccess) return cuda_fail(e, "token-order copy launch");
  if (copy_q) q = View{qc, q.B, q.H, q.N, q.d, q.H * q.N * q.d, q.N * q.d, q.d};
  if (copy_k) k = View{kc, k.B, k.H, k.N, k.d, k.H * k.N * k.d, k.N * k.d, k.d};
  ws = base + need;
  ws_bytes -= need;
  return SPARGE_OK;
}

bool is_q8(int precision);
// Under a token order Q gets an ordered copy only where TMA (d = 128) or the 8-bit quantiser reads
// it; at d = 64 the attention loads Q rows itself and gathers them through the permutation (the
// 8-bit precisions need d = 128).
bool order_copies_q(int64_t d, int precision) { return d != 64 || is_q8(precision); }

// Per-query-head parameter arrays of a sparge_params (device pointers, each may be null).
struct HeadParams {
  const float *topk = nullptr, *theta = nullptr, *lambda = nullptr;
  int topk_mode = SPARGE_TOPK_CUMULATIVE;  // how topk selects blocks (enum sparge_topk_mode)
  float topp = 1.f;                        // the top-p mass of SPARGE_TOPK_HYBRID
};

// topk_mode and, for the hybrid rule, topp
int check_topk_mode(const sparge_params *p) {
  if (p->topk_mode != SPARGE_TOPK_CUMULATIVE && p->topk_mode != SPARGE_TOPK_COUNT && p->topk_mode != SPARGE_TOPK_HYBRID)
    return fail(SPARGE_ERR_INVALID_ARG, "topk_mode %d unknown", p->topk_mode);
  if (p->topk_mode == SPARGE_TOPK_HYBRID && !(p->topp > 0.f && p->topp <= 1.f))
    return fail(SPARGE_ERR_INVALID_ARG, "topp=%g not in (0, 1]", (double)p->topp);
  return SPARGE_OK;
}

int predict_impl(const View &q, const View &k, float topk, float theta, int causal, float scale, uint8_t *mask,
                 void *ws, size_t ws_bytes, cudaStream_t s, void *const *ev = nullptr, const HeadParams &hp = {},
                 const int32_t *qperm = nullptr, const int32_t *kperm = nullptr, void *qcopy = nullptr,
                 void *kcopy = nullptr) {
  if (!mask) return fail(SPARGE_ERR_INVALID_ARG, "mask is NULL");
  int rc;
  if ((rc = check_lengths(q, k, causal))) return rc;
  if (k.N > 131072) return fail(SPARGE_ERR_UNSUPPORTED, "mask prediction supports Nk <= 131072 (got %lld)", (long long)k.N);
  if (q.B * q.H * cdiv(q.N, QBLK) > 0x7fffffffLL)
    return fail(SPARGE_ERR_UNSUPPORTED, "mask prediction supports at most 2^31 - 1 mask rows");
  const size_t need = predict_ws_bytes(q.B, q.H, k.H, q.N, k.N, q.d);
  if (need && (!ws || ws_bytes < need))
    return fail(SPARGE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, need);
  if (q.B == 0 || q.N == 0) return SPARGE_OK;
  PredictWs pw = predict_ws_carve(ws, q.B, q.H, k.H, q.N, k.N, q.d);
  if ((rc = record_event(ev, 0, s))) return rc;
  cudaError_t e = launch_pool_sim(q, k, pw, s, qperm, kperm, status_ptr(), qcopy, kcopy);
  if (e != cudaSuccess) return cuda_fail(e, "pool_sim launch");
  if ((rc = record_event(ev, 1, s))) return rc;
  {
    ScoreGemmLaunch g;
    memset(&g, 0, sizeof(g));
    const int64_t nqb = cdiv(q.N, QBLK), nkb = cdiv(k.N, KBLK);
    if ((rc = make_map3(&g.qhi, pw.qhi, q.d, nqb, q.B * q.H, "qhi")) || (rc = make_map3(&g.qlo, pw.qlo, q.d, nqb, q.B * q.H, "qlo")) ||
        (rc = make_map3(&g.khi, pw.khi, q.d, nkb, q.B * k.H, "khi")) || (rc = make_map3(&g.klo, pw.klo, q.d, nkb, q.B * k.H, "klo")) ||
        (rc = make_map_s(&g.ts, pw.S, pw.nkb_pad, nqb, q.B * q.H)))
      return rc;
    g.Smax = pw.Smax;
    g.muQ = pw.muQ;
    g.muK = pw.muK;
    g.S = pw.S;
    g.splits = pw.smax_splits;
    g.smax_stride = pw.smax_stride;
    g.nkb_pad = pw.nkb_pad;
    g.B = (int)q.B; g.Hq = (int)q.H; g.Hkv = (int)k.H; g.Nq = (int)q.N; g.Nk = (int)k.N; g.d = (int)q.d;
    g.causal = causal;
    g.scale = scale;
    g.status = status_ptr();
    e = launch_score_gemm(g, s);
    if (e != cudaSuccess) return cuda_fail(e, "score_gemm launch");
    if ((rc = record_event(ev, 2, s))) return rc;
  }
  // the hybrid rule: the count reading with topk, then the cumulative reading with topp OR-ed into
  // the same mask rows (the union of the two sets)
  const bool hybrid = hp.topk_mode == SPARGE_TOPK_HYBRID;
  e = launch_score_select(pw, (int)q.B, (int)q.H, (int)k.H, (int)q.N, (int)k.N, (int)q.d, topk, theta, causal, mask, hp.topk,
                          hp.theta, status_ptr(), hp.topk_mode != SPARGE_TOPK_CUMULATIVE ? 1 : 0, false, s);
  if (e == cudaSuccess && hybrid)
    e = launch_score_select(pw, (int)q.B, (int)q.H, (int)k.H, (int)q.N, (int)k.N, (int)q.d, hp.topp, theta, causal, mask,
                            nullptr, hp.theta, status_ptr(), 0, true, s);
  if (e != cudaSuccess) return cuda_fail(e, "score_select launch");
  return record_event(ev, 3, s);
}

size_t v16_bytes(int64_t B, int64_t Hkv, int64_t N, int64_t d) { return align256((size_t)B * Hkv * N * d * 2); }

// Attention workspace for a precision: the f16 copy of V, or the 8-bit copies and scales (every
// precision with an 8-bit product uses the 8-bit layout).
bool is_q8(int precision) {
  return precision == SPARGE_PRECISION_Q8 || precision == SPARGE_PRECISION_Q8_FP8PV ||
         precision == SPARGE_PRECISION_BF16_FP8PV;
}

// bf16: the f16 copy of V, or (decoding calls) the chunks' partial rows, whichever is larger
size_t attn_ws_bytes(int precision, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d) {
  if (is_q8(precision)) return d == 128 ? q8_ws_bytes(B, Hq, Hkv, Nq, Nk, d) : 0;
  const size_t v16 = v16_bytes(B, Hkv, Nk, d), part = decode_part_bytes(B, Hkv, Nk, d);
  return v16 > part ? v16 : part;
}

// Few queries per head against many keys (decoding, short chunks): the G Nq rows of a KV head's
// heads share one tile and the key blocks are split over CTAs (bf16, lambda off, no token order;
// the split needs the order of visiting tiles not to matter, which holds without the filter).
bool use_decode(const View &q, const View &k, int precision, float lambda, const HeadParams &hp, const int32_t *perm) {
  const int64_t G = q.H / k.H;
  return precision == SPARGE_PRECISION_BF16 && lambda == -INFINITY && hp.lambda == nullptr && perm == nullptr &&
         G * q.N <= 128 && cdiv(k.N, KBLK) >= 32;
}

int attn_impl(const View &q, const View &k, const View &v, const uint8_t *mask, float lambda, int causal, float scale,
              int precision, sparge_tensor *o, unsigned long long *stats, void *ws, size_t ws_bytes,
              cudaStream_t s, void *const *ev = nullptr, const HeadParams &hp = {}, const int32_t *perm = nullptr,
              const int32_t *qperm = nullptr) {
  if (precision != SPARGE_PRECISION_BF16 && !is_q8(precision))
    return fail(SPARGE_ERR_UNSUPPORTED, "precision %d not supported", precision);
  const bool q8 = is_q8(precision);  // an 8-bit product: d = 128, the 8-bit workspace
  const bool qk8 = precision == SPARGE_PRECISION_Q8 || precision == SPARGE_PRECISION_Q8_FP8PV;
  const bool pv8 = precision == SPARGE_PRECISION_Q8_FP8PV || precision == SPARGE_PRECISION_BF16_FP8PV;
  if (q8 && q.d != 128) return fail(SPARGE_ERR_UNSUPPORTED, "the 8-bit path needs d = 128 (got %lld)", (long long)q.d);
  if (q8 && k.N > 65535LL * 64) return fail(SPARGE_ERR_UNSUPPORTED, "the 8-bit path supports Nk <= %lld", 65535LL * 64);
  View ov{};
  int rc = check_tensor(o, "o", &ov);
  if (rc) return rc;
  if ((rc = check_lengths(q, k, causal))) return rc;
  if (v.B != q.B || v.N != k.N || v.d != q.d || v.H != k.H) return fail(SPARGE_ERR_INVALID_ARG, "v disagrees with q/k");
  if (ov.B != q.B || ov.N != q.N || ov.d != q.d || ov.H != q.H) return fail(SPARGE_ERR_INVALID_ARG, "o disagrees with q");
  const size_t need = attn_ws_bytes(precision, q.B, q.H, k.H, q.N, k.N, q.d);
  if (ws_bytes < need || (need && !ws))
    return fail(SPARGE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, need);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(SPARGE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (q.B == 0 || q.N == 0) return SPARGE_OK;
  AttnLaunch l;
  memset(&l, 0, sizeof(l));
  if (q8) {
    const Q8Ws w = q8_ws_carve(ws, q.B, q.H, k.H, q.N, k.N, q.d);
    cudaError_t e = launch_q8_prep(q, k, v, w, qk8, pv8, perm, status_ptr(), s);
    if (e != cudaSuccess) return cuda_fail(e, "8-bit quantisation launch");
    if (!pv8 && (e = launch_convert_v_f16(v, w.v8, perm, status_ptr(), s)) != cudaSuccess)
      return cuda_fail(e, "convert_v launch");
    if ((rc = record_event(ev, 4, s))) return rc;
    const int64_t d = q.d, Nq = q.N, N = k.N, npad = cdiv(N, 64) * 64;
    const int64_t qd[4] = {d, Nq, q.H, q.B}, qs[3] = {d, Nq * d, q.H * Nq * d};
    const int64_t kd[4] = {d, N, k.H, k.B}, ks[3] = {d, N * d, k.H * N * d};
    const int64_t vd[4] = {npad, d, k.H, k.B}, vs[3] = {npad, d * npad, k.H * d * npad};
    if (qk8) {
      if ((rc = make_map_u8(&l.tq, w.q8, qd, qs, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B, "q8")) ||
          (rc = make_map_u8(&l.tk, w.k8, kd, ks, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B, "k8")))
        return rc;
    } else if ((rc = make_map(&l.tq, q, 128, "q")) || (rc = make_map(&l.tk, k, 64, "k"))) {
      return rc;  // bf16 Q.K^T reads the (ordered) bf16 inputs as the bf16 path does
    }
    if (pv8) {
      if ((rc = make_map_u8(&l.tv, w.v8, vd, vs, 64, (int)d, CU_TENSOR_MAP_SWIZZLE_64B, "v8"))) return rc;
    } else {
      View v16{w.v8, v.B, v.H, v.N, v.d, v.H * v.N * v.d, v.N * v.d, v.d};
      if ((rc = make_map(&l.tv, v16, 64, "v", CU_TENSOR_MAP_DATA_TYPE_FLOAT16))) return rc;
    }
    l.q8 = qk8 ? (pv8 ? 2 : 1) : 3;
    l.sq = w.sq;
    l.sk = w.sk;
    l.sv = w.sv;
  } else if (use_decode(q, k, precision, lambda, hp, perm)) {
    // decoding tiles read Q rows, K and V (bf16) in place; the workspace holds the partial rows
    if ((rc = record_event(ev, 4, s))) return rc;
    const DecodeSplit sp = decode_split(k.B, k.H, k.N);
    const size_t rows = static_cast<size_t>(k.B * k.H) * sp.nchunk * 128;
    l.decode = 1;
    l.nchunk = sp.nchunk;
    l.chunk_blocks = sp.chunk_blocks;
    l.part_o = static_cast<float *>(ws);
    l.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + align256(rows * q.d * 4));
    const size_t lists_off = align256(rows * q.d * 4) + align256(rows * 2 * 4);
    l.dlist = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + lists_off);
    l.dcount = reinterpret_cast<int *>(static_cast<uint8_t *>(ws) + lists_off +
                                       align256(static_cast<size_t>(k.B * k.H) * cdiv(k.N, KBLK) * 4));
    if ((rc = make_map(&l.tq, q, 128, "q"))) return rc;  // checks the alignment the row reads rely on
    l.q = q.data;
    l.q_sb = q.sb; l.q_sh = q.sh; l.q_sn = q.sn;
    if ((rc = make_map(&l.tk, k, 64, "k")) || (rc = make_map(&l.tv, v, 64, "v"))) return rc;
  } else {
    cudaError_t e = launch_convert_v_f16(v, ws, perm, status_ptr(), s);
    if (e != cudaSuccess) return cuda_fail(e, "convert_v launch");
    if ((rc = record_event(ev, 4, s))) return rc;
    View v16{ws, v.B, v.H, v.N, v.d, v.H * v.N * v.d, v.N * v.d, v.d};
    if ((rc = make_map(&l.tq, q, 128, "q"))) return rc;  // checks the alignment the row reads rely on
    l.q = q.data;
    l.qperm = qperm;  // d = 64 under a token order: q is the caller's tensor, gathered by row
    l.q_sb = q.sb; l.q_sh = q.sh; l.q_sn = q.sn;
    if ((rc = make_map(&l.tk, k, 64, "k"))) return rc;
    if ((rc = make_map(&l.tv, v16, 64, "v", CU_TENSOR_MAP_DATA_TYPE_FLOAT16))) return rc;
  }
  l.mask = mask;
  l.o = o->data;
  l.o_sb = ov.sb; l.o_sh = ov.sh; l.o_sn = ov.sn;
  l.B = (int)q.B; l.Hq = (int)q.H; l.Hkv = (int)k.H; l.Nq = (int)q.N; l.Nk = (int)k.N; l.d = (int)q.d;
  l.causal = causal ? 1 : 0;
  l.scale = scale;
  l.lambda = lambda;
  l.lambda_h = hp.lambda;
  l.perm = perm;
  l.stats = stats;
  l.status = status_ptr();
  cudaError_t e = launch_bsattn(l, s);
  if (e != cudaSuccess) return cuda_fail(e, "bsattn launch");
  return record_event(ev, 5, s);
}

}  // namespace

namespace sparge {

int validate_predict_args(const sparge_tensor *q, const sparge_tensor *k, float topk, float theta, View *qv,
                          View *kv) {
  g_last_error[0] = 0;
  int rc;
  if ((rc = check_tensor(q, "q", qv)) || (rc = check_tensor(k, "k", kv)) || (rc = check_qk(*qv, *kv))) return rc;
  return check_topk_theta(topk, theta);
}

int run_predict(const View &q, const View &k, float topk, float theta, int causal, uint8_t *mask, void *ws,
                size_t ws_bytes, cudaStream_t s) {
  return predict_impl(q, k, topk, theta, causal, 1.f / sqrtf((float)q.d), mask, ws, ws_bytes, s);
}

int report_error(int code, const char *msg) { return fail(code, "%s", msg); }

size_t predict_ws_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d) {
  const int64_t nqb = cdiv(Nq, QBLK), nkb = cdiv(Nk, KBLK), nkb_pad = cdiv(nkb, 4) * 4;
  size_t s = 0;
  s += align256(sizeof(float) * B * Hq * nqb * d);      // muQ
  s += align256(sizeof(float) * B * Hq * nqb);          // sQ
  s += align256(sizeof(float) * B * Hkv * nkb * d);     // muK
  s += align256(sizeof(float) * B * Hkv * nkb_pad);     // sK
  s += 2 * align256(2 * B * Hq * nqb * d);              // qhi, qlo
  s += 2 * align256(2 * B * Hkv * nkb * d);             // khi, klo
  s += align256(sizeof(float) * B * Hq * nqb * nkb_pad);  // S
  s += align256(sizeof(float) * score_gemm_slices(Nk) * B * Hq * nqb);  // Smax slices
  return s;
}

PredictWs predict_ws_carve(void *ws, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d) {
  const int64_t nqb = cdiv(Nq, QBLK), nkb = cdiv(Nk, KBLK), nkb_pad = cdiv(nkb, 4) * 4;
  char *p = static_cast<char *>(ws);
  PredictWs w;
  auto take = [&](size_t bytes) {
    char *r = p;
    p += align256(bytes);
    return r;
  };
  w.muQ = reinterpret_cast<float *>(take(sizeof(float) * B * Hq * nqb * d));
  w.sQ = reinterpret_cast<float *>(take(sizeof(float) * B * Hq * nqb));
  w.muK = reinterpret_cast<float *>(take(sizeof(float) * B * Hkv * nkb * d));
  w.sK = reinterpret_cast<float *>(take(sizeof(float) * B * Hkv * nkb_pad));
  w.qhi = reinterpret_cast<uint16_t *>(take(2 * B * Hq * nqb * d));
  w.qlo = reinterpret_cast<uint16_t *>(take(2 * B * Hq * nqb * d));
  w.khi = reinterpret_cast<uint16_t *>(take(2 * B * Hkv * nkb * d));
  w.klo = reinterpret_cast<uint16_t *>(take(2 * B * Hkv * nkb * d));
  w.S = reinterpret_cast<float *>(take(sizeof(float) * B * Hq * nqb * nkb_pad));
  w.smax_splits = score_gemm_splits(B, Hq, Nq, Nk);
  w.smax_stride = B * Hq * nqb;
  w.Smax = reinterpret_cast<float *>(take(sizeof(float) * score_gemm_slices(Nk) * B * Hq * nqb));
  w.nkb_pad = nkb_pad;
  return w;
}

}  // namespace sparge

extern "C" {

size_t sparge_workspace_bytes(int op, int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || (d != 64 && d != 128)) return 0;
  if (op & SPARGE_OP_TOKEN_ORDER) {
    const size_t base = sparge_workspace_bytes(op & ~SPARGE_OP_TOKEN_ORDER, B, Hq, Hkv, N, d);
    return base ? base + order_bytes(B, Hq, Hkv, N, d) : 0;
  }
  switch (op) {
    case SPARGE_OP_PREDICT_MASK:
      return predict_ws_bytes(B, Hq, Hkv, N, N, d);
    case SPARGE_OP_BLOCK_SPARSE_ATTN:
      return attn_ws_bytes(SPARGE_PRECISION_BF16, B, Hq, Hkv, N, N, d);
    case SPARGE_OP_ATTN:
      return predict_ws_bytes(B, Hq, Hkv, N, N, d) + align256((size_t)B * Hq * cdiv(N, QBLK) * cdiv(N, KBLK)) +
             attn_ws_bytes(SPARGE_PRECISION_BF16, B, Hq, Hkv, N, N, d);
    case SPARGE_OP_BLOCK_SPARSE_ATTN_Q8:
      return attn_ws_bytes(SPARGE_PRECISION_Q8, B, Hq, Hkv, N, N, d);
    case SPARGE_OP_ATTN_Q8:
      if (d != 128) return 0;
      return predict_ws_bytes(B, Hq, Hkv, N, N, d) + align256((size_t)B * Hq * cdiv(N, QBLK) * cdiv(N, KBLK)) +
             attn_ws_bytes(SPARGE_PRECISION_Q8, B, Hq, Hkv, N, N, d);
    default:
      return 0;
  }
}

const char *sparge_last_error(void) { return g_last_error; }

int sparge_predict_mask(const sparge_tensor *q, const sparge_tensor *k, float topk, float theta, int is_causal,
                        uint8_t *mask, void *ws, size_t ws_bytes, sparge_stream_t stream) {
  g_last_error[0] = 0;
  View qv, kv;
  int rc;
  if ((rc = check_tensor(q, "q", &qv)) || (rc = check_tensor(k, "k", &kv)) || (rc = check_qk(qv, kv))) return rc;
  if ((rc = check_topk_theta(topk, theta))) return rc;
  return predict_impl(qv, kv, topk, theta, is_causal, 1.f / sqrtf((float)qv.d), mask, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream));
}

int sparge_predict_mask_ex(const sparge_tensor *q, const sparge_tensor *k, float topk, int is_causal,
                           const sparge_params *p, uint8_t *mask, void *ws, size_t ws_bytes, sparge_stream_t stream) {
  g_last_error[0] = 0;
  if (!p) return fail(SPARGE_ERR_INVALID_ARG, "params is NULL");
  View qv, kv;
  int rc;
  if ((rc = check_tensor(q, "q", &qv)) || (rc = check_tensor(k, "k", &kv)) || (rc = check_qk(qv, kv))) return rc;
  if ((rc = check_topk_theta(topk, p->theta))) return rc;
  if (std::isnan(p->scale) || p->scale < 0.f || std::isinf(p->scale))
    return fail(SPARGE_ERR_INVALID_ARG, "scale must be finite and >= 0");
  const float scale = p->scale > 0.f ? p->scale : 1.f / sqrtf((float)qv.d);
  if ((rc = check_topk_mode(p))) return rc;
  HeadParams hp;
  hp.topk = p->topk_per_head;
  hp.theta = p->theta_per_head;
  hp.topk_mode = p->topk_mode;
  hp.topp = p->topp;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->token_order) {
    if (qv.N != kv.N) return fail(SPARGE_ERR_UNSUPPORTED, "a token order needs Nq = Nk");
    const size_t need = order_bytes(qv.B, qv.H, kv.H, qv.N, qv.d) + predict_ws_bytes(qv.B, qv.H, kv.H, qv.N, kv.N, qv.d);
    if (!mask) return fail(SPARGE_ERR_INVALID_ARG, "mask is NULL");
    if (!ws || ws_bytes < need) return fail(SPARGE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, need);
    // pooling reads q and k through the permutation: no ordered copies (the space stays reserved)
    if (qv.B * qv.N > 0 && (rc = order_qk(qv, kv, p->token_order, ws, ws_bytes, s, false, false))) return rc;
  }
  return predict_impl(qv, kv, topk, p->theta, is_causal, scale, mask, ws, ws_bytes, s, p->timing_events, hp,
                      p->token_order, p->token_order);
}

int sparge_block_sparse_attn(const sparge_tensor *q, const sparge_tensor *k, const sparge_tensor *v,
                             const uint8_t *mask, float lambda, int is_causal, int precision, sparge_tensor *o,
                             void *ws, size_t ws_bytes, unsigned long long *stats, sparge_stream_t stream) {
  g_last_error[0] = 0;
  View qv, kv, vv;
  int rc;
  if ((rc = check_tensor(q, "q", &qv)) || (rc = check_tensor(k, "k", &kv)) || (rc = check_tensor(v, "v", &vv)) ||
      (rc = check_qk(qv, kv)))
    return rc;
  if ((rc = check_lambda(lambda))) return rc;
  return attn_impl(qv, kv, vv, mask, lambda, is_causal, 1.f / sqrtf((float)qv.d), precision, o, stats, ws,
                   ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int sparge_block_sparse_attn_ex(const sparge_tensor *q, const sparge_tensor *k, const sparge_tensor *v,
                                const uint8_t *mask, int is_causal, const sparge_params *p, sparge_tensor *o, void *ws,
                                size_t ws_bytes, sparge_stream_t stream) {
  g_last_error[0] = 0;
  if (!p) return fail(SPARGE_ERR_INVALID_ARG, "params is NULL");
  View qv, kv, vv;
  int rc;
  if ((rc = check_tensor(q, "q", &qv)) || (rc = check_tensor(k, "k", &kv)) || (rc = check_tensor(v, "v", &vv)) ||
      (rc = check_qk(qv, kv)))
    return rc;
  if ((rc = check_lambda(p->lambda))) return rc;
  if (std::isnan(p->scale) || p->scale < 0.f || std::isinf(p->scale))
    return fail(SPARGE_ERR_INVALID_ARG, "scale must be finite and >= 0");
  const float scale = p->scale > 0.f ? p->scale : 1.f / sqrtf((float)qv.d);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->token_order) {
    if (qv.N != kv.N) return fail(SPARGE_ERR_UNSUPPORTED, "a token order needs Nq = Nk");
    const size_t need =
        order_bytes(qv.B, qv.H, kv.H, qv.N, qv.d) + attn_ws_bytes(p->precision, qv.B, qv.H, kv.H, qv.N, kv.N, qv.d);
    if (!ws || ws_bytes < need) return fail(SPARGE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, need);
  }
  if ((rc = record_event(p->timing_events, 0, s))) return rc;
  const bool copy_q = order_copies_q(qv.d, p->precision);
  if (p->token_order && qv.B * qv.N > 0 &&
      (rc = order_qk(qv, kv, p->token_order, ws, ws_bytes, s, copy_q, true)))
    return rc;
  HeadParams hp;
  hp.lambda = p->lambda_per_head;
  return attn_impl(qv, kv, vv, mask, p->lambda, is_causal, scale, p->precision, o, p->stats, ws, ws_bytes, s,
                   p->timing_events, hp, p->token_order, (p->token_order && !copy_q) ? p->token_order : nullptr);
}

int sparge_attn_ex(const sparge_tensor *q, const sparge_tensor *k, const sparge_tensor *v, float topk, int is_causal,
                   const sparge_params *p, sparge_tensor *o, uint8_t *mask_out, void *ws, size_t ws_bytes,
                   sparge_stream_t stream) {
  g_last_error[0] = 0;
  if (!p) return fail(SPARGE_ERR_INVALID_ARG, "params is NULL");
  View qv, kv, vv;
  int rc;
  if ((rc = check_tensor(q, "q", &qv)) || (rc = check_tensor(k, "k", &kv)) || (rc = check_tensor(v, "v", &vv)) ||
      (rc = check_qk(qv, kv)))
    return rc;
  if ((rc = check_topk_theta(topk, p->theta)) || (rc = check_lambda(p->lambda))) return rc;
  if (std::isnan(p->scale) || p->scale < 0.f || std::isinf(p->scale))
    return fail(SPARGE_ERR_INVALID_ARG, "scale must be finite and >= 0");
  const float scale = p->scale > 0.f ? p->scale : 1.f / sqrtf((float)qv.d);
  if (p->token_order && qv.N != kv.N) return fail(SPARGE_ERR_UNSUPPORTED, "a token order needs Nq = Nk");
  const size_t need_pred = predict_ws_bytes(qv.B, qv.H, kv.H, qv.N, kv.N, qv.d);
  const size_t mask_bytes = mask_out ? 0 : align256((size_t)qv.B * qv.H * cdiv(qv.N, QBLK) * cdiv(kv.N, KBLK));
  if (is_q8(p->precision) && qv.d != 128)
    return fail(SPARGE_ERR_UNSUPPORTED, "the 8-bit path needs d = 128 (got %lld)", (long long)qv.d);
  const size_t need_v = attn_ws_bytes(p->precision, qv.B, qv.H, kv.H, qv.N, kv.N, qv.d);
  const size_t need_order = p->token_order ? order_bytes(qv.B, qv.H, kv.H, qv.N, qv.d) : 0;
  const size_t need = need_order + need_pred + mask_bytes + need_v;
  if (!ws || ws_bytes < need) return fail(SPARGE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool copy_q = order_copies_q(qv.d, p->precision);
  // Under a token order the pooling reads Q and K through it and writes the ordered copies the
  // attention (or the 8-bit quantiser) reads, so no separate copy pass runs.
  const View q_in = qv, k_in = kv;
  if (p->token_order && qv.B * qv.N > 0 &&
      (rc = order_qk(qv, kv, p->token_order, ws, ws_bytes, s, copy_q, true, false)))
    return rc;
  const int32_t *ord = p->token_order;
  const int32_t *qperm = (ord && !copy_q) ? ord : nullptr;  // q not copied: the attention gathers its rows
  uint8_t *mask = mask_out ? mask_out : static_cast<uint8_t *>(ws) + need_pred;
  void *ws_v = static_cast<uint8_t *>(ws) + need_pred + mask_bytes;
  if ((rc = check_topk_mode(p))) return rc;
  HeadParams hp;
  hp.topk = p->topk_per_head;
  hp.theta = p->theta_per_head;
  hp.lambda = p->lambda_per_head;
  hp.topk_mode = p->topk_mode;
  hp.topp = p->topp;
  if (ord) {
    if ((rc = predict_impl(q_in, k_in, topk, p->theta, is_causal, scale, mask, ws, need_pred, s, p->timing_events, hp,
                           ord, ord, copy_q ? const_cast<void *>(qv.data) : nullptr, const_cast<void *>(kv.data))))
      return rc;
  } else if ((rc = predict_impl(qv, kv, topk, p->theta, is_causal, scale, mask, ws, need_pred, s, p->timing_events,
                                hp))) {
    return rc;
  }
  return attn_impl(qv, kv, vv, mask, p->lambda, is_causal, scale, p->precision, o, p->stats, ws_v, need_v, s,
                   p->timing_events, hp, p->token_order, qperm);
}

int sparge_attn(const sparge_tensor *q, const sparge_tensor *k, const sparge_tensor *v, float topk, int is_causal,
                sparge_tensor *o, void *ws, size_t ws_bytes, sparge_stream_t stream) {
  sparge_params p;
  memset(&p, 0, sizeof(p));  // every optional pointer null
  p.theta = 0.5f;
  p.lambda = -INFINITY;
  p.scale = 0.f;
  p.precision = SPARGE_PRECISION_BF16;
  p.stats = nullptr;
  p.timing_events = nullptr;
  return sparge_attn_ex(q, k, v, topk, is_causal, &p, o, nullptr, ws, ws_bytes, stream);
}

static int permute_common(const sparge_tensor *x, const int32_t *perm, sparge_tensor *y, bool inverse,
                          sparge_stream_t stream) {
  g_last_error[0] = 0;
  View xv, yv;
  int rc;
  if ((rc = check_tensor(x, "x", &xv)) || (rc = check_tensor(y, "y", &yv))) return rc;
  if (!perm) return fail(SPARGE_ERR_INVALID_ARG, "perm is NULL");
  if (xv.B != yv.B || xv.H != yv.H || xv.N != yv.N || xv.d != yv.d) return fail(SPARGE_ERR_INVALID_ARG, "x and y shapes differ");
  if (x->data == y->data) return fail(SPARGE_ERR_INVALID_ARG, "x and y must not overlap");
  cudaError_t e = launch_permute(xv, perm, y->data, yv.sb, yv.sh, yv.sn, inverse, status_ptr(),
                                 reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "permute launch");
  return SPARGE_OK;
}

int sparge_permute_tokens(const sparge_tensor *x, const int32_t *perm, sparge_tensor *y, sparge_stream_t stream) {
  return permute_common(x, perm, y, false, stream);
}

int sparge_unpermute_tokens(const sparge_tensor *x, const int32_t *perm, sparge_tensor *y, sparge_stream_t stream) {
  return permute_common(x, perm, y, true, stream);
}

int sparge_selftest_bounded_wait(int64_t limit_ns, sparge_stream_t stream) {
  g_last_error[0] = 0;
  if (limit_ns < 1000000) limit_ns = 1000000;
  if (limit_ns > 1000000000) limit_ns = 1000000000;
  int *st = status_ptr();
  if (!st) return fail(SPARGE_ERR_CUDA, "device status word unavailable");
  bounded_wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(st, (uint64_t)limit_ns);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SPARGE_OK : cuda_fail(e, "bounded wait probe launch");
}

int sparge_get_device_status(sparge_stream_t stream) {
  g_last_error[0] = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_status_word, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (host != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return fail(host, host == SPARGE_ERR_DEVICE_TIMEOUT ? "a device-side wait timed out"
                                                        : "a kernel skipped a permutation entry outside 0..N-1");
  }
  return SPARGE_OK;
}

}  // extern "C"
