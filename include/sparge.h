/*
 * sparge.h -- C ABI of the GB300 (sm_103a) SpargeAttn sparse-attention forward.
 *
 * The method (SpargeAttention: Accurate and Training-free Sparse Attention Accelerating Any
 * Model Inference, abstract and summary pages) is a two-stage online filter:
 *   stage 1 predicts a 128x64 block mask from mean-pooled Q/K blocks (sparge_predict_mask);
 *   stage 2 runs flash attention over the kept tiles only, and inside its online softmax
 *   skips a warp's P.V update when its row maxima trail the running maxima by more than
 *   lambda (sparge_block_sparse_attn).
 * sparge_attn chains the two, as the plug-and-play call of the SpargeAttn overview page
 * ("Using the plug-and-play API": attn(q, k, v, topk=0.5, is_causal=False)).
 *
 * Conventions shared by every call
 *   - Tensors are bf16 in (B, H, N, d) order ("HND"), described by sparge_tensor.  The d axis
 *     must be contiguous; stride_n, stride_h and stride_b are in elements and must be
 *     multiples of 8 (16 bytes); data must be 16-byte aligned.  d is 64 or 128.
 *   - K and V may have fewer heads than Q (grouped-query attention): Hq % Hkv == 0 and query
 *     head h reads key/value head h / (Hq / Hkv).
 *   - Q may have a different length Nq from K and V (Nk): a chunk of queries continuing a longer
 *     key sequence (prefill in chunks, decoding).  With the causal mask Nq <= Nk and the last
 *     query sits on the last key: query row r sees key c when c <= (Nk - Nq) + r (Nq = Nk is
 *     the usual square case).  Without it any Nq and Nk > 0.  Blocks and masks then have
 *     ceil(Nq/128) query rows and ceil(Nk/64) key columns, and sparge_workspace_bytes is
 *     called with N = max(Nq, Nk).  A token order (sparge_params.token_order) needs Nq = Nk.
 *   - The block mask is uint8, contiguous, shape (B, Hq, ceil(Nq/128), ceil(Nk/64)); 1 keeps
 *     the 128x64 tile, 0 drops it (SpargeAttention Chinese README, custom block-sparse mask).
 *   - Every pointer except the *_host ones is a device pointer.  The caller owns every buffer
 *     (inputs, outputs, mask, workspace); the library allocates no device memory.  All work
 *     is enqueued asynchronously on the caller's stream; no call synchronises except
 *     sparge_get_device_status.
 *   - Every call returns SPARGE_OK (0) or a negative status; sparge_last_error() then gives a
 *     message (thread-local).  Arguments are validated on the host before anything is
 *     enqueued, so a failed validation leaves the outputs untouched.
 *   - Device-side waits are bounded; a wait that runs out records SPARGE_ERR_DEVICE_TIMEOUT in
 *     a device status word that sparge_get_device_status reads.
 */
#ifndef SPARGE_H
#define SPARGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *sparge_stream_t; /* the same handle type as cudaStream_t */

enum sparge_status {
  SPARGE_OK = 0,
  SPARGE_ERR_INVALID_ARG = -1,        /* null pointer, bad shape/stride, topk/theta/lambda out of range */
  SPARGE_ERR_UNSUPPORTED = -2,        /* d not in {64,128}, dtype not bf16, Hq % Hkv != 0, N too large */
  SPARGE_ERR_WORKSPACE_TOO_SMALL = -3,
  SPARGE_ERR_CUDA = -4,               /* a CUDA runtime/driver call or a launch failed */
  SPARGE_ERR_DEVICE_TIMEOUT = -5      /* a bounded device-side wait ran out */
};

enum sparge_dtype { SPARGE_BF16 = 1 };

enum sparge_precision {
  SPARGE_PRECISION_BF16 = 0,          /* bf16 tensor-core products, fp32 accumulation */
  SPARGE_PRECISION_Q8 = 1,            /* 8-bit Q.K^T (e4m3, K smoothed), f16 P.V; d = 128 */
  SPARGE_PRECISION_Q8_FP8PV = 2,      /* 8-bit Q.K^T and P.V (both e4m3); d = 128 */
  SPARGE_PRECISION_BF16_FP8PV = 3     /* bf16 Q.K^T, 8-bit P.V (e4m3); d = 128 */
};

/* How topk picks a mask row's blocks (sparge_params.topk_mode). */
enum sparge_topk_mode {
  SPARGE_TOPK_CUMULATIVE = 0,  /* the shortest prefix, in (probability desc, index asc) order, whose
                                  cumulative probability reaches topk (the pages' "top 50% of the
                                  attention weights"; the default) */
  SPARGE_TOPK_COUNT = 1,       /* the first ceil(topk * n_valid) blocks of that order (at least one;
                                  the product is taken in fp32 with topk as given, less 1e-3, so
                                  that rounding never adds a block) */
  SPARGE_TOPK_HYBRID = 2       /* a block is kept when SPARGE_TOPK_COUNT with topk keeps it or
                                  SPARGE_TOPK_CUMULATIVE with sparge_params.topp keeps it (the
                                  union of a top-k and a top-p set: the longer of the two prefixes;
                                  reading of the hybrid Top-k + Top-p mask that the Chinese README's
                                  citation list names for SpargeAttention2 without a rule) */
};

enum sparge_op {
  SPARGE_OP_PREDICT_MASK = 1,
  SPARGE_OP_BLOCK_SPARSE_ATTN = 2,
  SPARGE_OP_ATTN = 3,
  SPARGE_OP_BLOCK_SPARSE_ATTN_Q8 = 4, /* sparge_block_sparse_attn with an 8-bit precision */
  SPARGE_OP_ATTN_Q8 = 5,              /* sparge_attn_ex with an 8-bit precision */
  SPARGE_OP_TOKEN_ORDER = 0x100       /* flag OR-ed into an op: room for the token-ordered copies of
                                         Q and K that a call with sparge_params.token_order makes */
};

/* A strided bf16 tensor of logical shape (B, H, N, d); data is a device pointer. */
typedef struct sparge_tensor {
  void *data;
  int32_t dtype; /* SPARGE_BF16 */
  int32_t pad_;
  int64_t B, H, N, d;
  int64_t stride_b, stride_h, stride_n; /* in elements */
} sparge_tensor;

/* Zero-initialise a sparge_params before setting its fields (sparge_params p = {0};): every
 * optional pointer must be NULL unless it is meant to be used.
 * Counters the attention kernel can add to (device memory, 4 x uint64, caller-zeroed):
 *   [0] kept tiles visited, [1] tiles whose P.V product was issued,
 *   [2] (32-row group, tile) pairs whose P.V update the lambda filter skipped,
 *   [3] valid tiles (tiles not wholly above the causal diagonal). */
typedef struct sparge_params {
  float theta;   /* similarity threshold; blocks with self-similarity < theta are always kept */
  float lambda;  /* <= 0 or -INFINITY (filter off) */
  float scale;   /* softmax scale; 0 means 1/sqrt(d) */
  int32_t precision;            /* enum sparge_precision */
  unsigned long long *stats;    /* optional device pointer to 4 counters, or NULL */
  void *const *timing_events;   /* optional: 6 cudaEvent_t handles recorded on the stream before the
                                   pooling kernel and after the pooling, pooled-score, selection,
                                   V-copy (8-bit path: quantisation) and attention kernels (for per-kernel timing), or NULL */
  /* Optional per-query-head parameters (the tuned mode of the SpargeAttn overview page, where
   * every head of every layer has its own thresholds): device arrays of Hq floats, or NULL.
   * When given, entry h replaces the scalar for query head h: topk_per_head in the mask rows of
   * head h (the topk argument otherwise), theta_per_head in its always-keep rules (both the
   * row rule on s_Q and the column rule on s_K), lambda_per_head in its attention rows.  The
   * entries are read on the device; an entry out of range (topk outside (0, 1], a theta that is
   * not finite, a lambda that is NaN or > 0) records SPARGE_ERR_INVALID_ARG in the device status
   * word and that head runs with every valid block kept (bad topk or theta) or with the filter
   * off (bad lambda). */
  const float *topk_per_head;
  const float *theta_per_head;
  const float *lambda_per_head;
  /* Optional token order (device, N int32, or NULL), e.g. the Hilbert order of image or video
   * tokens (SpargeAttention summary page: reordering by a space-filling curve raises the
   * similarity inside blocks).  The call then works on the sequence whose token t is token
   * token_order[t] of q, k and v: blocks, mask (and mask_out) refer to that sequence, and o is
   * written back in the original order (o token token_order[t] receives row t).  The result is
   * that of sparge_permute_tokens on q, k and v, the call, and sparge_unpermute_tokens on the
   * output, without the separate V and output passes: the attention reads K, and Q where d = 128
   * or an 8-bit precision needs it, from copies in the new order in the workspace (the space is
   * sparge_workspace_bytes(op | SPARGE_OP_TOKEN_ORDER, ...) either way).  In sparge_attn_ex the
   * mask prediction's pooling, which reads every row through the order, writes those copies as
   * it goes (no separate copy pass); sparge_block_sparse_attn_ex, which has no pooling, copies
   * them in a pass of its own.  The d = 64 attention reads Q rows through the order itself,
   * mask prediction alone copies nothing, V is gathered while it is converted or quantised, and
   * the attention kernel writes each output row straight to its original position.
   * token_order should be a permutation of 0..N-1; an entry outside that range is never used as
   * an address (its row is skipped or zero) and records SPARGE_ERR_INVALID_ARG in the device
   * status word. */
  const int32_t *token_order;
  /* How topk (and topk_per_head) picks blocks: enum sparge_topk_mode (0, the cumulative reading,
   * when the struct is zeroed).  Used by sparge_predict_mask_ex and sparge_attn_ex. */
  int32_t topk_mode;
  /* SPARGE_TOPK_HYBRID only: the cumulative probability of the top-p set, in (0, 1] (else
   * SPARGE_ERR_INVALID_ARG); topk (or topk_per_head) is then the count fraction of the top-k set.
   * Unused by the other modes. */
  float topp;
} sparge_params;

/*
 * Workspace bytes needed by an op for the given shape (0 if the op needs none).
 * SPARGE_OP_PREDICT_MASK: pooled means and similarities (fp32).
 * SPARGE_OP_BLOCK_SPARSE_ATTN: an f16 copy of V.
 * SPARGE_OP_ATTN: all of the above plus the uint8 mask.
 * SPARGE_OP_BLOCK_SPARSE_ATTN_Q8: e4m3 copies of Q and K - mean(K), room for either V copy (f16,
 *   or e4m3 channel-major with the keys padded to a multiple of 64) and the fp32 scales;
 *   SPARGE_OP_ATTN_Q8: that plus the mask-prediction workspace and the mask.  Both return 0
 *   unless d = 128.
 * op | SPARGE_OP_TOKEN_ORDER: the op's bytes plus room for bf16 copies of Q and K in a given
 *   token order (at the front of the workspace), for calls whose sparge_params.token_order is set
 *   (a call uses only the copies it needs; the room is reserved in full).
 * Returns 0 for an unknown op or an unsupported shape.
 */
size_t sparge_workspace_bytes(int op, int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d);

/*
 * Stage 1, mask prediction (SpargeAttention summary page, method paragraph: blocks with high
 * internal similarity are compressed, non-similar blocks always computed; abstract: the
 * attention map is predicted so that some matrix multiplications are skipped).
 *   For each 128-token query block and 64-token key block: the mean over its valid tokens and
 *   its self-similarity s = mean pairwise cosine = ||mean of unit tokens||^2.  Then per query
 *   head and query block i: pooled scores scale * muQ_i . muK_j over the valid key blocks
 *   (causal: 64 j <= 128 i + 127), a row softmax, and the shortest prefix of blocks in
 *   (probability desc, index asc) order whose cumulative probability reaches topk (all valid
 *   blocks when topk >= 1).  The row is then OR-ed with every valid block if s_Q(i) < theta,
 *   and with block j if s_K(j) < theta (per key/value head).
 * q: (B,Hq,N,d), k: (B,Hkv,N,d).  topk in (0,1]; theta finite.  mask: device, (B,Hq,nqb,nkb).
 * ws/ws_bytes: device workspace of at least sparge_workspace_bytes(SPARGE_OP_PREDICT_MASK,...).
 * Supports N <= 131072 (nkb <= 2048).
 */
int sparge_predict_mask(const sparge_tensor *q, const sparge_tensor *k, float topk, float theta,
                        int is_causal, uint8_t *mask, void *ws, size_t ws_bytes,
                        sparge_stream_t stream);

/*
 * sparge_predict_mask with its parameters in a sparge_params: theta, scale (0 means 1/sqrt(d);
 * the pooled scores are scale * muQ . muK), topk_per_head and theta_per_head, token_order, and
 * timing events [0]-[3] (before pooling, after pooling, after the pooled scores, after the
 * selection).  lambda, precision, stats and lambda_per_head are unused.  Same workspace and
 * errors as sparge_predict_mask (with SPARGE_OP_TOKEN_ORDER when token_order is set).
 */
int sparge_predict_mask_ex(const sparge_tensor *q, const sparge_tensor *k, float topk, int is_causal,
                           const sparge_params *params, uint8_t *mask, void *ws, size_t ws_bytes,
                           sparge_stream_t stream);

/*
 * Stage 2, block-sparse attention (SpargeAttention abstract: the second-stage online
 * softmax-aware filter; summary: it works at GPU-warp level; Chinese README: custom mask API).
 *   O = softmax(scale * Q K^T) V restricted to the kept tiles, visited in ascending key-block
 *   order with an online softmax.  Rows are grouped 32 per warp; for each kept tile a group
 *   leaves out its P.V update when every row's tile maximum trails its running maximum by more
 *   than |lambda| (the running maximum and the row sum are still updated).  Rows with no
 *   visible kept key output 0.  mask may be NULL (every tile kept).  Tiles wholly above the
 *   causal diagonal are never visited, whatever the mask says.
 * lambda <= 0 or -INFINITY.  o: (B,Hq,N,d) bf16 output.
 * precision SPARGE_PRECISION_BF16: Q.K^T runs on bf16 operands; P.V runs on f16 operands (P in
 * [0, 256], V copied to f16 into the workspace first: exact for |v| <= 65504, larger magnitudes
 * saturate), both with fp32 accumulation.  ws: 256-byte aligned device workspace of at least
 * sparge_workspace_bytes(SPARGE_OP_BLOCK_SPARSE_ATTN, ...) bytes (the f16 copy of V).
 * precision SPARGE_PRECISION_Q8 and SPARGE_PRECISION_Q8_FP8PV (d = 128 only, else
 * SPARGE_ERR_UNSUPPORTED; SpargeAttention overview page: built on SageAttention's 8-bit
 * quantisation with outlier smoothing): K is smoothed by its per-(batch, KV head) token mean (a
 * per-row shift of the scores that the softmax ignores); Q and K - mean are quantised to FP8
 * e4m3 with one scale per 128-token query block and per 64-token key block (scale = max|x| /
 * 448, round to nearest even) and Q.K^T runs as e4m3 x e4m3 with fp32 accumulation.  INT8
 * Q.K^T (tcgen05 kind::i8) is not available on sm_103a, hence e4m3, whose 3-bit mantissa
 * leaves a larger score error than INT8 would.  SPARGE_PRECISION_Q8 keeps P.V on f16 operands
 * as above; SPARGE_PRECISION_Q8_FP8PV also quantises V to e4m3 with one scale per channel and
 * P to e4m3 (P <= 256) and runs P.V as e4m3 x e4m3 (faster tensor work, about twice the output
 * error).  SPARGE_PRECISION_BF16_FP8PV (d = 128 only) keeps Q.K^T on the bf16 inputs and runs
 * P.V in e4m3 as SPARGE_PRECISION_Q8_FP8PV does: e4m3 Q.K^T moves peaked softmax rows (large,
 * aligned scores) much more than INT8 would, while e4m3 P.V alone stays within cosine 0.999 of
 * the exact output on every workload measured.  ws: 256-byte aligned, at least
 * sparge_workspace_bytes(SPARGE_OP_BLOCK_SPARSE_ATTN_Q8, ...) bytes (every precision with an
 * 8-bit product); it holds the quantised copies after the call.
 * Few queries against many keys (decoding, short chunks): with precision SPARGE_PRECISION_BF16,
 * lambda = -INFINITY (and no per-head lambda), no token order, G Nq <= 128 (G = Hq / Hkv) and at
 * least 32 key blocks, the call packs the Nq query rows of the G heads of each KV head into one
 * tile, lists the key blocks any of the G heads keeps and splits that list into equal shares over
 * CTAs (each row masking the blocks its own head does not keep), and combines the shares' partial
 * rows in a last kernel; P.V then runs on bf16 P and V read in place (no f16 copy of
 * V; the workspace holds the partial rows and the block lists instead).  The result is the same computation within
 * the bf16 tolerances; the lambda filter needs the tiles visited in order, so calls with it keep
 * one tile per query block and head.  Counters then count a tile once per (batch, KV head).
 * stats: optional counters (see sparge_params), may be NULL.
 */
int sparge_block_sparse_attn(const sparge_tensor *q, const sparge_tensor *k,
                             const sparge_tensor *v, const uint8_t *mask, float lambda,
                             int is_causal, int precision, sparge_tensor *o, void *ws,
                             size_t ws_bytes, unsigned long long *stats, sparge_stream_t stream);

/*
 * sparge_block_sparse_attn with its parameters in a sparge_params (theta, topk_per_head and
 * theta_per_head are unused): lambda or lambda_per_head, scale (0 means 1/sqrt(d)), precision,
 * counters, and timing events; of the six events, [0] is recorded before the V copy or
 * quantisation, [4] after it and [5] after the attention kernel ([1]-[3] are left alone).  Same
 * workspace and errors as sparge_block_sparse_attn.
 */
int sparge_block_sparse_attn_ex(const sparge_tensor *q, const sparge_tensor *k, const sparge_tensor *v,
                                const uint8_t *mask, int is_causal, const sparge_params *params,
                                sparge_tensor *o, void *ws, size_t ws_bytes, sparge_stream_t stream);

/*
 * The plug-and-play call: sparge_predict_mask with theta = 0.5, then sparge_block_sparse_attn
 * with lambda = -INFINITY, scale 1/sqrt(d).  ws: sparge_workspace_bytes(SPARGE_OP_ATTN, ...).
 */
int sparge_attn(const sparge_tensor *q, const sparge_tensor *k, const sparge_tensor *v,
                float topk, int is_causal, sparge_tensor *o, void *ws, size_t ws_bytes,
                sparge_stream_t stream);

/*
 * sparge_attn with every parameter explicit (theta, lambda, scale, precision, counters, and the
 * optional per-head topk, theta and lambda arrays).
 * ws: sparge_workspace_bytes(SPARGE_OP_ATTN, ...) bytes, or SPARGE_OP_ATTN_Q8 for the 8-bit path.
 * mask_out: optional device buffer (B,Hq,nqb,nkb) that receives the predicted mask; when
 * NULL the mask lives in the workspace.
 */
int sparge_attn_ex(const sparge_tensor *q, const sparge_tensor *k, const sparge_tensor *v,
                   float topk, int is_causal, const sparge_params *params, sparge_tensor *o,
                   uint8_t *mask_out, void *ws, size_t ws_bytes, sparge_stream_t stream);

/*
 * Hilbert-curve token order (SpargeAttention summary page: a space-filling Hilbert-curve
 * reordering improves token locality and sparsity for visual tasks).
 * perm (device, int32, length N): y[:, :, t, :] = x[:, :, perm[t], :] (permute) and
 * y[:, :, perm[t], :] = x[:, :, t, :] (unpermute).  x and y have the same shape; they must
 * not overlap.  perm should be a permutation of 0..N-1.  An entry outside 0..N-1 is never used
 * as an address: its token row is skipped (left unwritten in y) and the kernel records
 * SPARGE_ERR_INVALID_ARG in the device status word (read by sparge_get_device_status).  Entries
 * in range that repeat leave some rows of y unwritten (permute) or written more than once
 * (unpermute, last writer unspecified).
 */
int sparge_permute_tokens(const sparge_tensor *x, const int32_t *perm, sparge_tensor *y,
                          sparge_stream_t stream);
int sparge_unpermute_tokens(const sparge_tensor *x, const int32_t *perm, sparge_tensor *y,
                            sparge_stream_t stream);

/*
 * Host-side builders of the gather permutation (integer only, host memory, length
 * n_prefix + H*W or n_prefix + T*H*W).  Text tokens 0..n_prefix-1 stay in place; grid tokens
 * (stored row-major after the prefix) are ordered by their index on the Hilbert curve of the
 * smallest power-of-two square (2-D, x = column, y = row, curve from (0,0) to (2^k-1,0)) or
 * cube (3-D, Skilling's transpose construction on (t, row, column)) covering the grid.
 */
int sparge_hilbert_perm_2d(int n_prefix, int H, int W, int32_t *perm_host);
int sparge_hilbert_perm_3d(int n_prefix, int T, int H, int W, int32_t *perm_host);

/*
 * Mask prediction without any device allocation, for callers that cannot call cudaMalloc (a
 * plug-in inside a host application whose allocator already holds the device memory it hands
 * out; a latency-critical loop that cannot afford the device synchronisation cudaMalloc and
 * cudaFree may cause).  The paper has no counterpart: this is a packaging variant of
 * sparge_predict_mask, with the same arguments minus the workspace and the same result.
 * The scratch (pooled means and similarities) is a fixed 8 MiB array in device memory that every
 * GPU loading the library holds until the process exits; a shape whose scratch
 * (sparge_workspace_bytes(SPARGE_OP_PREDICT_MASK, ...)) exceeds 8 MiB is rejected with
 * SPARGE_ERR_UNSUPPORTED before anything is enqueued.  The first call on a device looks up the
 * array's device address with that device current (and so does the first call in a new context of
 * the device, e.g. after cudaDeviceReset, which gives the array a new home); make that first call
 * before any stream capture.  All calls on a device share the array and it keeps the last call's contents (no
 * part of it needs to start at zero): calls that can overlap on the GPU (different streams, no
 * ordering between them) race on it and must be serialised by the caller.
 */
int sparge_predict_mask_noalloc(const sparge_tensor *q, const sparge_tensor *k, float topk, float theta,
                                int is_causal, uint8_t *mask, sparge_stream_t stream);

/*
 * Failure-detection test support.  Enqueues a one-thread kernel whose mbarrier wait gets no
 * arrival: the wait gives up after limit_ns (clamped to [1 ms, 1 s]) exactly like the bounded
 * waits of the library's kernels and records SPARGE_ERR_DEVICE_TIMEOUT in the device status word,
 * which sparge_get_device_status then reports (and clears).  Nothing faults or hangs; the context
 * stays usable.  No passage of the method corresponds to it.
 */
int sparge_selftest_bounded_wait(int64_t limit_ns, sparge_stream_t stream);

/* Message of the last failed call on this thread ("" if none). */
const char *sparge_last_error(void);

/* Reads and clears the device status word after synchronising the stream: SPARGE_OK,
 * SPARGE_ERR_DEVICE_TIMEOUT (a bounded wait ran out), SPARGE_ERR_INVALID_ARG (a permutation entry
 * outside 0..N-1 was skipped), or SPARGE_ERR_CUDA if the read itself failed.  The first code
 * recorded since the last read is kept. */
int sparge_get_device_status(sparge_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARGE_H */
