// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sparge {

struct View {  // a validated bf16 (B, H, N, d) tensor, strides in elements
  const void *data;
  int64_t B, H, N, d;
  int64_t sb, sh, sn;
};

// Stage-1 workspace.  fp32 block means and similarities, the means again as bf16 hi/lo pairs
// (mu ~= hi + lo, about 16 significant bits) for the tensor-core score product, and the scaled
// pooled scores S, one fp32 row of nkb_pad entries per query block.
struct PredictWs {
  float *muQ;       // [B][Hq][nqb][d]
  float *sQ;        // [B][Hq][nqb]
  float *muK;       // [B][Hkv][nkb][d]
  float *sK;        // [B][Hkv][nkb_pad]
  uint16_t *qhi, *qlo;  // bf16 [B][Hq][nqb][d]
  uint16_t *khi, *klo;  // bf16 [B][Hkv][nkb][d]
  float *S;         // [B][Hq][nqb][nkb_pad]
  float *Smax;      // [smax_splits][B][Hq][nqb] maximum of each S row over its valid key blocks, one
                    // slice per key-chunk split of the score product (the row maximum is theirs)
  int64_t nkb_pad;
  int smax_splits;
  int64_t smax_stride;  // B Hq nqb: floats between two slices
};

// Key-chunk splits of the pooled-score product.  One CTA per (head, group of 128 query blocks)
// leaves most of a 152-SM part idle when there are few such tiles (decoding, short queries): the
// key chunks of 128 blocks are then divided among up to about two CTAs per SM (at most 8 splits),
// each writing the maxima of its chunks to its own Smax slice.  The workspace holds
// score_gemm_slices(Nk) slices, a bound that grows with Nk alone, so a workspace sized for the
// longer of the two lengths covers every shorter query.
constexpr int SCORE_GEMM_MAX_SPLITS = 8;
inline int score_gemm_slices(int64_t Nk) {
  const int64_t nch = ((Nk + 63) / 64 + 127) / 128;
  return static_cast<int>(nch < 1 ? 1 : (nch < SCORE_GEMM_MAX_SPLITS ? nch : SCORE_GEMM_MAX_SPLITS));
}
// With at most SCORE_ROW_KERNEL_ROWS query-block rows in all (decoding steps, short chunks) the
// pooled scores come from a row kernel instead of the tensor-core product (a 128-row MMA tile
// would be almost empty): one CTA per (row, 256 key blocks), fp32 dot products of the fp32 means,
// each CTA's row maximum in its own Smax slice (at most 8, as 2048 key blocks is the longest row).
constexpr int64_t SCORE_ROW_KERNEL_ROWS = 256;
inline bool score_use_rows(int64_t B, int64_t Hq, int64_t Nq) {
  return B * Hq * ((Nq + 127) / 128) <= SCORE_ROW_KERNEL_ROWS;
}
inline int score_gemm_splits(int64_t B, int64_t Hq, int64_t Nq, int64_t Nk) {
  const int64_t nqb = (Nq + 127) / 128, nkb = (Nk + 63) / 64;
  if (score_use_rows(B, Hq, Nq)) {
    const int64_t s = (nkb + 255) / 256;
    return static_cast<int>(s < 1 ? 1 : s);
  }
  const int64_t tiles = B * Hq * ((nqb + 127) / 128), nch = (nkb + 127) / 128;
  if (tiles <= 0 || nch <= 1 || tiles >= 152) return 1;
  int64_t s = (2 * 152 + tiles - 1) / tiles;
  if (s > score_gemm_slices(Nk)) s = score_gemm_slices(Nk);
  const int64_t per = (nch + s - 1) / s;  // chunks per split
  return static_cast<int>((nch + per - 1) / per);
}

// Nq: query length, Nk: key length
size_t predict_ws_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d);
PredictWs predict_ws_carve(void *ws, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d);

}  // namespace sparge
struct sparge_tensor;
namespace sparge {
// Host-side pieces of the C-ABI layer (api.cu) that other entry points reuse.
int validate_predict_args(const ::sparge_tensor *q, const ::sparge_tensor *k, float topk, float theta, View *qv,
                          View *kv);
int run_predict(const View &q, const View &k, float topk, float theta, int causal, uint8_t *mask, void *ws,
                size_t ws_bytes, cudaStream_t s);
int report_error(int code, const char *msg);

// qperm / kperm (or nullptr): token order of q / k; block row t of the pooling is token perm[t] (an
// entry outside 0..N-1 is reported in *status and read as a zero token).  qcopy / kcopy (or
// nullptr; used only with the order): contiguous (B, H, N, d) bf16 buffers that receive the rows
// in that order as they are read (zero rows for bad entries).
cudaError_t launch_pool_sim(const View &q, const View &k, const PredictWs &ws, cudaStream_t st,
                            const int32_t *qperm = nullptr, const int32_t *kperm = nullptr, int *status = nullptr,
                            void *qcopy = nullptr, void *kcopy = nullptr);

// Pooled scores S = scale * muQ . muK^T on tcgen05 (bf16 hi/lo split, three products), for the
// valid (causal) key blocks of every query block.  The four maps cover qhi, qlo (3-D: d, nqb,
// B*Hq; box 64 x 128) and khi, klo (d, nkb, B*Hkv; box 64 x 128).
struct ScoreGemmLaunch {
  CUtensorMap qhi, qlo, khi, klo;
  CUtensorMap ts;  // 3-D map over S (nkb_pad, nqb, B*Hq) fp32, box 32 x 128, 128-byte swizzle
  float *Smax;     // [splits][B][Hq][nqb] row maxima over the valid key blocks of each split's chunks
  int64_t nkb_pad;
  int splits;      // score_gemm_splits of the shape
  int64_t smax_stride;
  const float *muQ, *muK;  // the fp32 means and S itself, for the row kernel of few-row shapes
  float *S;
  int B, Hq, Hkv, Nq, Nk, d, causal;  // query and key lengths (causal: Nq <= Nk, the last query on the last key)
  float scale;
  int *status;
};
cudaError_t launch_score_gemm(const ScoreGemmLaunch &l, cudaStream_t st);

// Row softmax, cumulative top-k and the always-keep rule on S: writes the uint8 mask.  topk_h and
// theta_h (device, Hq floats, or nullptr) override topk and theta per query head; a bad entry is
// recorded in *status and its head keeps every valid block.  count_mode: topk is a fraction of the
// valid blocks instead of the mass; or_into: the kept blocks are OR-ed into the mask rows already
// there instead of replacing them.
cudaError_t launch_score_select(const PredictWs &ws, int B, int Hq, int Hkv, int Nq, int Nk, int d, float topk,
                                float theta, int causal, uint8_t *mask, const float *topk_h, const float *theta_h,
                                int *status, int count_mode, bool or_into, cudaStream_t st);

struct AttnLaunch {
  CUtensorMap tq, tk, tv;  // 4-D maps (d, N, H, B), 128-byte swizzle, boxes 64 x 128 (Q) / 64 x 64 (K, V);
                           // Q, K bf16, V the f16 copy
  const uint8_t *mask;     // (B, Hq, nqb, nkb) or nullptr
  void *o;
  int64_t o_sb, o_sh, o_sn;
  int B, Hq, Hkv, Nq, Nk, d;  // query and key lengths (causal: Nq <= Nk, the last query on the last key)
  int causal;
  float scale;
  float lambda;
  const float *lambda_h;   // per query head (device, Hq floats) or nullptr; a bad entry turns the filter off
  unsigned long long *stats;
  int *status;
  int q8;                  // 0: bf16 Q.K^T, f16 P.V; 1: e4m3 Q.K^T (maps over the e4m3 copies, scales sq, sk),
                           // f16 P.V; 2: as 1 with e4m3 P.V (channel-major e4m3 V, scales sv); 3: bf16
                           // Q.K^T (maps over the bf16 inputs) with e4m3 P.V as in 2
  const float *sq, *sk, *sv;
  const int32_t *perm;     // token order or nullptr: output row t goes to token perm[t] of o
  const void *q;           // bf16 Q, read row by row into TMEM at d = 64 (the ordered copy under a token order
                           // at d = 128, where the rows come by TMA)
  const int32_t *qperm;    // d = 64 under a token order: Q row t of the block is token qperm[t] of q
  int64_t q_sb, q_sh, q_sn;
  // decoding tiles (decode != 0, bf16): the G Nq <= 128 query rows of a KV head's heads in one
  // tile; the key blocks that any of the G heads keeps are listed in ascending order (dlist,
  // [B Hkv][nkb], with their count in dcount) and split into nchunk equal shares, one per CTA
  // (decode_split); the shares' partial rows go to part_o / part_ml, then are combined; V is read in
  // place as bf16
  int decode, nchunk, chunk_blocks;
  float *part_o, *part_ml;
  int32_t *dlist;
  int *dcount;
};

// How a decoding call splits the key blocks of each (batch, KV head): about two CTAs per SM of a
// 152-SM part, at least 16 key blocks per chunk.  Sizes both the workspace and the launch.
struct DecodeSplit {
  int nchunk, chunk_blocks;
};
inline DecodeSplit decode_split(int64_t B, int64_t Hkv, int64_t Nk) {
  const int64_t nkb = (Nk + 63) / 64, units = B * Hkv > 0 ? B * Hkv : 1;
  int64_t nchunk = (304 + units - 1) / units;
  const int64_t most = nkb >= 16 ? nkb / 16 : 1;
  if (nchunk > most) nchunk = most;
  if (nchunk < 1) nchunk = 1;
  const int64_t cb = (nkb + nchunk - 1) / nchunk;
  DecodeSplit s;
  s.chunk_blocks = static_cast<int>(cb > 0 ? cb : 1);
  s.nchunk = static_cast<int>((nkb + s.chunk_blocks - 1) / s.chunk_blocks);
  return s;
}
// Workspace of a decoding call: the partial rows [B Hkv][nchunk][128][d] fp32, then (m, l) per
// row, then the kept-block lists [B Hkv][nkb] int32 and their counts [B Hkv].
inline size_t decode_part_bytes(int64_t B, int64_t Hkv, int64_t Nk, int64_t d) {
  const DecodeSplit s = decode_split(B, Hkv, Nk);
  const size_t rows = static_cast<size_t>(B * Hkv) * s.nchunk * 128;
  const size_t units = static_cast<size_t>(B * Hkv), nkb = static_cast<size_t>((Nk + 63) / 64);
  return ((rows * d * 4 + 255) & ~size_t(255)) + ((rows * 2 * 4 + 255) & ~size_t(255)) +
         ((units * nkb * 4 + 255) & ~size_t(255)) + ((units * 4 + 255) & ~size_t(255));
}

cudaError_t launch_bsattn(const AttnLaunch &a, cudaStream_t st);

// Decoding tiles (decode.cu): before the attention, the ascending list of key blocks that any of
// the G heads of each (batch, KV head) keeps in query block 0 (list [B Hkv][nkb], count [B Hkv]);
// after it, the shares' partial rows combined into o (bf16, strides in elements).
cudaError_t launch_decode_union(const uint8_t *mask, int B, int Hq, int Hkv, int nqb, int nkb, int32_t *list, int *count,
                                cudaStream_t st);
cudaError_t launch_decode_combine(const float *part_o, const float *part_ml, int nchunk, int B, int Hq, int Hkv, int Nq,
                                  int d, void *o, int64_t o_sb, int64_t o_sh, int64_t o_sn, cudaStream_t st);

// perm (or nullptr): row t of the copy is token perm[t] of v; bad entries are reported in *status.
cudaError_t launch_convert_v_f16(const View &v, void *v16, const int32_t *perm, int *status, cudaStream_t st);

// 8-bit path: e4m3 copies of Q, K - mean(K) and V with their scales (all contiguous).
struct Q8Ws {
  uint8_t *q8;      // [B][Hq][N][d]
  uint8_t *k8;      // [B][Hkv][N][d]
  uint8_t *v8;      // e4m3 P.V: [B][Hkv][d][npad] channel-major, npad = N rounded up to 64 (tail zero);
                    // f16 P.V: the f16 copy of V, [B][Hkv][N][d]
  float *sq;        // [B][Hq][nqb]   per 128-token query block
  float *sk;        // [B][Hkv][nkb]  per 64-token key block
  float *kmean;     // [B][Hkv][d]
  float *sv;        // [B][Hkv][d]    per channel
  float *partial;   // [B*Hkv][chunks][2][d]
};
// Nq: query length, N: key / value length
size_t q8_ws_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t N, int64_t d);
Q8Ws q8_ws_carve(void *ws, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t N, int64_t d);
// With quant_qk: the K mean and e4m3 Q and K - mean with their block scales.  With quant_v: the V
// channel scales and the channel-major e4m3 V (otherwise v8 is left to the caller), whose key t is
// token perm[t] of v when perm is given (Q and K are used in the order they come in).
cudaError_t launch_q8_prep(const View &q, const View &k, const View &v, const Q8Ws &w, bool quant_qk, bool quant_v,
                           const int32_t *perm, int *status, cudaStream_t st);

cudaError_t launch_permute(const View &x, const int32_t *perm, void *y, int64_t ysb, int64_t ysh, int64_t ysn,
                           bool inverse, int *status, cudaStream_t st, bool zero_bad = false);

}  // namespace sparge
