// Stage 2: block-sparse flash attention with the lambda warp filter, on tcgen05 tensor cores.
//
// SpargeAttention abstract: only the kept tiles of the predicted map are multiplied, and an
// online softmax-aware filter skips further updates; summary page: that filter works at GPU
// warp level; Chinese README: arbitrary per-head block masks of 128x64 tiles.
//
// One CTA computes one 128-row query block of one head.  Warp roles (224 threads):
//   warps 0-3  softmax + epilogue; warp w owns TMEM lanes 32w..32w+31, i.e. rows 32w.. of the
//              block, one row per thread (the 32-row group of the lambda filter).
//   warp 4     producer: TMA loads of the Q block once, then of only the kept tiles: K into a
//              KST-deep ring that is freed as soon as Q.K^T of a tile completes (so K runs well
//              ahead), V into a VST-deep ring freed when P.V completes; the key-block index of
//              each tile goes to the softmax warps through a small ring of its own.
//   warp 5     score issuer: S_t = Q K_t^T (bf16) into one of two TMEM score buffers, as soon as
//              K_t has landed and P.V of tile t - 2 (the buffer's last P) has completed.
//   warp 6     P.V issuer: O += P_t V_t (f16) with P_t read back from TMEM (written over S_t) and
//              V_t from shared memory.  A tcgen05.mma issue returns only once the tensor unit
//              has taken the product, about 150 cycles per product here, so one thread issuing
//              both kinds serialised them; two issuers overlap them.
// P and V enter the second product as f16 (V converted once from bf16 by convert_v_f16 before
// the kernel): P lies in [0, 256] and f16 keeps 3 more mantissa bits than bf16, so the P.V
// rounding error is 8x smaller at the same tensor-core rate.
// TMEM columns: O at [0, D), score buffers at [128, 192) and [192, 256) (D = 128) or [64, 128)
// and [128, 192) (D = 64, where Q also moves into TMEM at [192, 224) as the A operand of Q.K^T);
// 256 columns are allocated, so two CTAs share an SM.  The tensor core reads the shared-memory
// operands of one 128 x 64 x 16 product at about 128 bytes per clock, so with Q in shared memory
// the score product takes 48 cycles instead of 32 and the operand reads bound the kernel.
//
// Online softmax per row in the log2 domain.  The exponent reference m_ref is moved only when
// the running maximum exceeds it by more than 8 (P <= 2^8 before the move), so O is rescaled
// in TMEM only then; O and l share the reference so O / l is exact.  The lambda filter compares
// each row's tile maximum with its true running maximum; a warp whose 32 rows all trail writes
// P = 0 (its row sums still include the tile) and the P.V product is not issued when all four
// warps trail.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace sparge {
namespace {

constexpr int NTHREADS = 224;
constexpr int RESCALE_LOG2 = 8;   // bf16 path: O is rescaled when the running max passes m_ref + 8
constexpr int RESCALE_LOG2_P8 = 4;  // e4m3 P: P = 2^(x - m_ref + 4) <= 256 < 448 (e4m3 maximum)

struct AttnArgs {
  const uint8_t *mask;
  __nv_bfloat16 *o;
  int64_t o_sb, o_sh, o_sn;
  int B, Hq, Hkv, G, Nq, Nk, nqb, nkb, causal, off;  // query and key lengths; off = Nk - Nq
  float scale_log2, lam_log2;
  const float *lam_h;  // lambda per query head (natural-log units), or nullptr
  const int32_t *perm; // token order or nullptr: output row t is token perm[t] of o
  unsigned long long *stats;
  int *status;
  const float *sq, *sk, *sv;  // 8-bit path: scales of the Q blocks, K blocks and V channels
  const __nv_bfloat16 *q;     // bf16 path: Q rows, copied into TMEM by the softmax warps
  const int32_t *qperm;       // token order of those rows (or nullptr)
  int64_t q_sb, q_sh, q_sn;
  // decoding tiles: the key blocks that any head of a (batch, KV head) keeps, listed in dlist
  // ([B Hkv][nkb], count in dcount; without a mask every block), are split into nchunk equal
  // shares; partial results go to part_o [B Hkv][nchunk][128][D] and part_ml (m, l) per row
  int nchunk, chunk_blocks;
  float *part_o, *part_ml;
  const int32_t *dlist;
  const int *dcount;
};

// Warp-collective walk over the kept, valid key blocks of one mask row in ascending order, run
// by the producer warp only: windows of 512 candidates, 16 per lane loaded as independent bytes,
// then lowest lane / lowest bit first.  Returns -1 after the last kept block.
// A decoding tile walks the union of the mask rows of its G heads (gstride bytes apart) from block
// lo on.
struct KeptScan {
  const uint8_t *row;
  int n, base, t, G;
  int64_t gstride;
  uint32_t bits;  // this lane's 16 flags of the current window
  __device__ void init(const uint8_t *r, int n_valid, int lo = 0, int g = 1, int64_t gs = 0) {
    row = r;
    n = n_valid;
    base = lo - 512;
    t = lo;
    G = g;
    gstride = gs;
    bits = 0u;
  }
  __device__ int next(int lane) {
    if (row == nullptr) return t < n ? t++ : -1;
    for (;;) {
      const uint32_t any = __ballot_sync(0xffffffffu, bits != 0u);
      if (any) {
        const int l = __ffs(any) - 1;
        const uint32_t lb = __shfl_sync(0xffffffffu, bits, l);
        if (lane == l) bits &= bits - 1u;
        return base + 16 * l + (__ffs(lb) - 1);
      }
      base += 512;
      if (base >= n) return -1;
      // per row of the group: the lane's 16 flags are all loaded before any is used, so the loads
      // of a window are in flight together (one memory latency per row, not one per flag)
      uint32_t f = 0u;
      for (int g = 0; g < G; ++g) {
        const uint8_t *rg = row + g * gstride;
        uint32_t m[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int j = base + 16 * lane + c;
          m[c] = j < n ? __ldg(rg + j) : 0u;
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) f |= (m[c] != 0u ? 1u : 0u) << c;
      }
      bits = f;
    }
  }
};

// Operand precisions: Q.K^T on bf16 or e4m3 (QK8) operands, P.V on f16 or e4m3 (PV8) operands.
// Shared memory of one CTA.  Q and K tiles are rows of D elements in 128-byte chunks (bf16: D / 64
// chunks; e4m3: one chunk for D = 128).  A V tile is 64 keys x D channels, either key-major f16
// (MN-major operand, 128-byte chunks of 64 channels) or channel-major e4m3 with 64-byte rows
// (K-major operand, 64-byte swizzle).
template <int D, int KST, int VST, bool QK8, bool PV8>
struct Smem {
  static constexpr int EB = QK8 ? 1 : 2;                 // bytes per element of Q and K
  static constexpr int QCH = D * EB / 128;               // 128-byte chunks of a Q or K row
  static constexpr int VCH = D * (PV8 ? 1 : 2) / 128;    // 128 bytes of V row data per chunk
  // TMEM score buffers.  At d = 64 a third buffer fits if Q leaves TMEM (O 64 + 3 x 64 columns);
  // measured no faster than two buffers with Q in TMEM (video-like 0.516 vs 0.506 ms).
  static constexpr int NSB = 2;
  static constexpr bool QTM = !QK8 && D == 64;  // Q in TMEM where two score buffers still fit
  static constexpr uint32_t Q_BYTES = QTM ? 0u : QCH * 128 * 128;  // 128 rows x 128 B per chunk
  static constexpr uint32_t KV_CHUNK = 64 * 128;         // 64 rows x 128 B
  static constexpr uint32_t K_BYTES = QCH * KV_CHUNK;    // one K tile
  static constexpr uint32_t V_BYTES = VCH * KV_CHUNK;    // one V tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KST * K_BYTES;
  static constexpr uint32_t OFF_CTRL = OFF_V + VST * V_BYTES;
  static constexpr uint32_t CTRL_BYTES = 512;
  static constexpr uint32_t TOTAL = OFF_CTRL + CTRL_BYTES;
};

constexpr int JRING = 8;  // key-block indices handed from the producer to the softmax warps

struct Ctrl {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4];    // K ring: filled by TMA, freed when Q.K^T of the tile completes
  uint64_t v_full[4], v_empty[4];    // V ring: filled by TMA, freed when P.V of the tile completes
  uint64_t j_full[JRING], j_empty[JRING];
  uint64_t s_full[4];
  uint64_t p_full[4];
  uint64_t mma_done;
  uint64_t final_bar, final_bar2;  // completions of each issuer's products
  uint64_t pv_done[4];             // P.V of the score buffer's last tile completed (buffer free)
  uint32_t tmem_base;
  int jring[JRING];  // key block of tile t at t % JRING; -1 marks the end of the row
  int jk[4];         // key block of the tile in each K stage (-1: end of the row)
  int abort;
  int pv_any;
  int row_end;  // the row's tile count T, set by the softmax warps with their p_full arrival of phase T
  uint8_t skip[4][4];
};
static_assert(sizeof(Ctrl) <= 512, "control block");

template <int D, int KST, int VST, bool QK8, bool PV8, bool DEC>
__global__ void __launch_bounds__(NTHREADS, 2)
    bsattn_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const AttnArgs a) {
  using L = Smem<D, KST, VST, QK8, PV8>;
  static_assert((!QK8 && !PV8) || D == 128, "the 8-bit operands cover d = 128");
  extern __shared__ __align__(1024) uint8_t smem[];
  // the 128-byte swizzle of TMA and of the MMA descriptors assumes 1024-byte aligned tiles
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_status(a.status, -4 /* SPARGE_ERR_CUDA */);
    return;
  }
  Ctrl &cs = *reinterpret_cast<Ctrl *>(smem + L::OFF_CTRL);
  volatile int *abort = &cs.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work item: (b, kvh) outermost so concurrently resident CTAs share K/V in L2; within it the
  // query blocks go from last to first (most causal work first), heads of a group adjacent.
  // A decoding tile (DEC) holds the Nq query rows of all G heads of one KV head (row g Nq + qi is
  // query qi of head kvh G + g) against one share of the key blocks those heads keep (lo and
  // n_valid only count the chunk's key range for the counters).
  int b, kvh, i, h, lo = 0, n_valid;
  if constexpr (DEC) {
    const int chunk = blockIdx.x % a.nchunk, bk = blockIdx.x / a.nchunk;
    b = bk / a.Hkv;
    kvh = bk % a.Hkv;
    i = 0;
    h = kvh * a.G;  // the group's first head
    lo = chunk * a.chunk_blocks;
    n_valid = min(a.nkb, lo + a.chunk_blocks);  // causal visibility is row by row in the softmax
  } else {
    const int per_bk = a.nqb * a.G;
    const int bk = blockIdx.x / per_bk, rem = blockIdx.x % per_bk;
    b = bk / a.Hkv;
    kvh = bk % a.Hkv;
    i = a.nqb - 1 - rem / a.G;
    h = kvh * a.G + rem % a.G;
    n_valid = a.causal ? min(a.nkb, causal_key_blocks(i, a.off)) : a.nkb;
  }
  const uint8_t *mrow = a.mask ? a.mask + ((static_cast<int64_t>(b) * a.Hq + h) * a.nqb + i) * a.nkb : nullptr;

  // TMEM columns: d = 128: O [0, 128), score buffers [128, 192) and [192, 256), Q in shared memory;
  // d = 64 (bf16): O [0, 64), score buffers [64, 128) and [128, 192), and Q [192, 224) as the TMEM
  // A operand of Q.K^T, so the tensor core reads only K from shared memory.  (Q in TMEM at d = 128
  // leaves room for one score buffer only; measured slower, as Q.K^T of the next tile can then not
  // run during the softmax of this one.)
  constexpr bool QTM = L::QTM;
  constexpr int NSB = L::NSB;  // score buffers
  static_assert(!QTM || D == 64, "Q in TMEM at d = 64 only");
  constexpr int SCOL0 = (D == 128) ? 128 : 64;
  constexpr int QCOL = (D == 128) ? 128 : 192;
  constexpr uint32_t TMEM_COLS = 256;
  constexpr uint32_t IDESC_S = QK8 ? idesc_f32acc(128, 64, FMT_E4M3, false) : idesc_f32acc(128, 64, FMT_BF16, false);
  // P.V: e4m3, f16 (V copied to f16), or bf16 for decoding tiles, which read V in place
  constexpr uint32_t IDESC_PV = PV8 ? idesc_f32acc(128, D, FMT_E4M3, false)
                                    : idesc_f32acc(128, D, DEC ? FMT_BF16 : FMT_F16, true);
  constexpr int KSTEPS = D * L::EB / 32;  // 32 bytes of the contraction per MMA: K = 16 (bf16) or 32 (e4m3)

  if (threadIdx.x == 0) {
    // the 128 softmax threads after their Q rows are in TMEM (d = 64 bf16) or in shared memory
    // (decoding tiles); else the producer's TMA load
    mbar_init(&cs.q_full, (QTM || DEC) ? 128 : 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&cs.k_full[s], 1);
      mbar_init(&cs.k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&cs.v_full[s], 1);
      mbar_init(&cs.v_empty[s], 1);
    }
    for (int s = 0; s < JRING; ++s) {
      mbar_init(&cs.j_full[s], 1);
      mbar_init(&cs.j_empty[s], 4);
    }
    for (int s = 0; s < L::NSB; ++s) {
      mbar_init(&cs.s_full[s], 1);
      mbar_init(&cs.p_full[s], 128);
      mbar_init(&cs.pv_done[s], 1);
    }
    mbar_init(&cs.mma_done, 1);
    mbar_init(&cs.final_bar, 1);
    mbar_init(&cs.final_bar2, 1);
    cs.row_end = -1;
    cs.abort = 0;
    cs.pv_any = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&cs.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cs.tmem_base;

  const uint32_t sQ = smem_u32(smem + L::OFF_Q);
  const uint32_t sK = smem_u32(smem + L::OFF_K);
  const uint32_t sV = smem_u32(smem + L::OFF_V);

  if (warp == 4) {
    // ------------------------------------ producer ------------------------------------
    // For tile t: the key block index into the j ring, K_t into the K ring (Q with the first
    // tile), then V_{t-1} into the V ring, so K runs up to KST tiles ahead of Q.K^T while V
    // follows P.V.  After the last tile the next K stage and j slot get the end mark (-1, a plain
    // arrive without data).
    KeptScan ks;
    ks.init(mrow, n_valid);
    // decoding tile: share `chunk` of the (batch, KV head)'s kept-block list, [d_lo, d_hi)
    int d_lo = 0, d_hi = 0;
    const int32_t *dl = nullptr;
    if constexpr (DEC) {
      const int chunk = blockIdx.x % a.nchunk, bk = blockIdx.x / a.nchunk;
      const int cnt = a.mask ? __ldg(a.dcount + bk) : a.nkb;
      d_lo = static_cast<int>(static_cast<int64_t>(chunk) * cnt / a.nchunk);
      d_hi = static_cast<int>(static_cast<int64_t>(chunk + 1) * cnt / a.nchunk);
      if (a.mask) dl = a.dlist + static_cast<int64_t>(bk) * a.nkb;
    }
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    int jprev = -1;
    for (int t = 0;; ++t) {
      int j;
      if constexpr (DEC)
        j = d_lo + t < d_hi ? (dl ? __ldg(dl + d_lo + t) : d_lo + t) : -1;
      else
        j = ks.next(lane);
      const int kst = t % KST, js = t % JRING;
      if (!mbar_wait(&cs.k_empty[kst], ((t / KST) & 1) ^ 1, abort, a.status)) break;
      if (!mbar_wait(&cs.j_empty[js], ((t / JRING) & 1) ^ 1, abort, a.status)) break;
      if (lane == 0) {
        cs.jring[js] = j;
        mbar_arrive(&cs.j_full[js]);
        cs.jk[kst] = j;
        if (j >= 0) {
          if (!QTM && !DEC && t == 0) {
            mbar_arrive_expect_tx(&cs.q_full, L::Q_BYTES);
            for (int c = 0; c < L::QCH; ++c)
              tma_load_4d(smem + L::OFF_Q + c * 16384, &tq, &cs.q_full, (128 / L::EB) * c, QBLK * i, h, b);
          }
          uint8_t *kdst = smem + L::OFF_K + kst * L::K_BYTES;
          mbar_arrive_expect_tx(&cs.k_full[kst], L::K_BYTES);
          for (int c = 0; c < L::QCH; ++c)
            tma_load_4d(kdst + c * L::KV_CHUNK, &tk, &cs.k_full[kst], (128 / L::EB) * c, KBLK * j, kvh, b);
        } else {
          mbar_arrive(&cs.k_full[kst]);
        }
      }
      __syncwarp();
      if (jprev >= 0) {
        const int u = t - 1, vst = u % VST;
        if (!mbar_wait(&cs.v_empty[vst], ((u / VST) & 1) ^ 1, abort, a.status)) break;
        if (lane == 0) {
          uint8_t *vdst = smem + L::OFF_V + vst * L::V_BYTES;
          mbar_arrive_expect_tx(&cs.v_full[vst], L::V_BYTES);
          if constexpr (PV8) {
            tma_load_4d(vdst, &tv, &cs.v_full[vst], KBLK * jprev, 0, kvh, b);  // [D channels][64 keys]
          } else {
            for (int c = 0; c < L::VCH; ++c)
              tma_load_4d(vdst + c * L::KV_CHUNK, &tv, &cs.v_full[vst], 64 * c, KBLK * jprev, kvh, b);
          }
        }
        __syncwarp();
      }
      jprev = j;
      if (j < 0) break;
    }
    if (*abort) {  // let copies already in flight land before the CTA exits
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 1000000ull) {
      }
    }
  } else if (warp == 5) {
    // ------------------------------ score-product issuer ------------------------------
    // Q.K^T of tile u as soon as K_u has landed and the score buffer is free: it last held P of
    // tile u - 2, so that P.V must have completed.  A second warp issues the P.V products, so
    // neither kind of product waits behind the other's issue.
    // next_tile(u): waits for K stage u % KST and returns its key block (-1 = end of row)
    auto next_tile = [&](int u) -> int {
      const int st = u % KST;
      if (!mbar_wait(&cs.k_full[st], (u / KST) & 1, abort, a.status)) return -2;
      tc_fence_after();
      return cs.jk[st];
    };
    // Descriptors: the start address is the low field (address / 16), so a tile's descriptor for an
    // operand offset is the base descriptor plus offset / 16; only these adds remain per MMA.
    const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
    auto issue_s = [&](int u) {
      if (lane == 0) {
        const uint64_t dk = dk0 + static_cast<uint64_t>(((u % KST) * L::K_BYTES) >> 4);
        const uint32_t dS = tmem + SCOL0 + (u % NSB) * 64;
#pragma unroll
        for (int s = 0; s < KSTEPS; ++s) {
          const uint64_t db = dk + static_cast<uint64_t>(((s >> 2) * L::KV_CHUNK + (s & 3) * 32) >> 4);
          if constexpr (QTM) {
            mma_bf16_ts(dS, tmem + QCOL + s * 8, db, IDESC_S, s > 0 ? 1u : 0u);  // 16 bf16 of Q = 8 columns
          } else {
            const uint64_t da = dq0 + static_cast<uint64_t>(((s >> 2) * 16384 + (s & 3) * 32) >> 4);
            if constexpr (QK8)
              mma_f8_ss(dS, da, db, IDESC_S, s > 0 ? 1u : 0u);
            else
              mma_bf16_ss(dS, da, db, IDESC_S, s > 0 ? 1u : 0u);
          }
        }
        mma_commit(&cs.s_full[u % NSB]);
        mma_commit(&cs.k_empty[u % KST]);  // the K stage is free once this product completes
      }
      __syncwarp();
    };
    int u = 0;
    for (;; ++u) {
      const int jn = next_tile(u);
      if (jn < 0) break;  // -1: end of the row, -2: timeout
      if (u == 0) {
        if (!mbar_wait(&cs.q_full, 0, abort, a.status)) break;
        tc_fence_after();
      } else if (u >= NSB) {
        if (!mbar_wait(&cs.pv_done[u % NSB], ((u - NSB) / NSB) & 1, abort, a.status)) break;
        tc_fence_after();
      }
      issue_s(u);
    }
    if (lane == 0) {
      if (u > 0) {
        mma_commit(&cs.final_bar);  // completes once every product this thread issued has finished
        mbar_wait(&cs.final_bar, 0, abort, a.status);
      }
      if (a.stats) {
        atomicAdd(a.stats + 0, static_cast<unsigned long long>(u));
        atomicAdd(a.stats + 3, static_cast<unsigned long long>(n_valid - lo));
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------ P.V issuer ------------------------------
    // O += P_t V_t once the softmax has written P_t and V_t has landed; the softmax warps mark the
    // end of the row with one more p_full arrival, phase T, after storing T in row_end (the flag may
    // already hold T while earlier phases are still being consumed, hence the comparison with t).
    int pv_count = 0, t = 0;
    uint32_t pv_issued = 0;
    for (;; ++t) {
      if (!mbar_wait(&cs.p_full[t % NSB], (t / NSB) & 1, abort, a.status)) break;
      if (*reinterpret_cast<volatile int *>(&cs.row_end) == t) break;  // set before phase t's arrival
      const int vst = t % VST;
      if (!mbar_wait(&cs.v_full[vst], (t / VST) & 1, abort, a.status)) break;
      tc_fence_after();
      const int sb = t % NSB;
      const bool all_skip = cs.skip[sb][0] && cs.skip[sb][1] && cs.skip[sb][2] && cs.skip[sb][3];
      if (lane == 0) {
        if (!all_skip) {
          const uint32_t vaddr = sV + vst * L::V_BYTES;
          const uint32_t aP = tmem + SCOL0 + sb * 64;
          if constexpr (PV8) {
            // P: 4 e4m3 per TMEM column, 8 columns per 32 keys; V tile rows of 64 keys
            const uint64_t dv = smem_desc_sw64(vaddr, 512);
#pragma unroll
            for (int s = 0; s < 2; ++s)
              mma_f8_ts(tmem, aP + s * 8, dv + static_cast<uint64_t>((s * 32) >> 4), IDESC_PV, (pv_issued | (s > 0 ? 1u : 0u)));
          } else {
            const uint64_t dv = smem_desc_sw128(vaddr, L::KV_CHUNK, 1024);
#pragma unroll
            for (int s = 0; s < 4; ++s)
              mma_bf16_ts(tmem, aP + s * 8, dv + static_cast<uint64_t>((s * 2048) >> 4), IDESC_PV, (pv_issued | (s > 0 ? 1u : 0u)));
          }
          pv_issued = 1;
          ++pv_count;
        }
        mma_commit(&cs.v_empty[vst]);
        mma_commit(&cs.pv_done[sb]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      if (t > 0) {
        mma_commit(&cs.final_bar2);  // completes once every P.V product has finished
        mbar_wait(&cs.final_bar2, 0, abort, a.status);
      }
      cs.pv_any = static_cast<int>(pv_issued);
      mbar_arrive(&cs.mma_done);  // the epilogue may read O
      if (a.stats) atomicAdd(a.stats + 1, static_cast<unsigned long long>(pv_count));
    }
    __syncwarp();
  } else {
    // ------------------------------------ softmax warps ------------------------------------
    const int r = warp * 32 + lane;
    // the row's query index and head: row r of query block i of head h, or (decoding tile) query
    // r % Nq of head h + r / Nq, rows past G Nq empty
    int row_g = QBLK * i + r, hrow = h;
    bool row_ok = row_g < a.Nq;
    const uint8_t *hmask = nullptr;  // decoding tile: this row's head's mask row
    if constexpr (DEC) {
      row_ok = r < a.G * a.Nq;
      row_g = row_ok ? r % a.Nq : 0;
      hrow = h + (row_ok ? r / a.Nq : 0);
      if (a.mask) hmask = a.mask + (static_cast<int64_t>(b) * a.Hq + hrow) * a.nqb * a.nkb;
    }
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m_run = -INFINITY, m_ref = -INFINITY, l = 0.f;
    int nskip = 0, T = 0;
    bool ok = true;
    constexpr float RESC = static_cast<float>(PV8 ? RESCALE_LOG2_P8 : RESCALE_LOG2);
    constexpr float POFF = PV8 ? static_cast<float>(8 - RESCALE_LOG2_P8) : 0.f;  // exponent offset of P
    // this head's filter threshold in log2 units; a bad per-head entry turns the filter off
    float lam_log2 = a.lam_log2;
    if (a.lam_h) {
      const float lh = a.lam_h[h];
      const bool good = lh <= 0.f;  // false for NaN and for lambda > 0
      lam_log2 = (!good || lh == -INFINITY) ? -INFINITY : lh * 1.4426950408889634f;
      if (!good && r == 0) record_status(a.status, -1 /* SPARGE_ERR_INVALID_ARG */);
    }
    if constexpr (QTM) {
      // this thread's Q row (zeros past the query length) into TMEM columns QCOL.., two bf16 per column
      // under a token order the row is token qperm[row] of q (an entry outside 0..Nq-1 is
      // reported and read as a zero row)
      int qrow = row_ok ? row_g : 0;
      bool qok = row_ok;
      if (a.qperm != nullptr && row_ok) {
        qrow = __ldg(a.qperm + row_g);
        if (static_cast<unsigned>(qrow) >= static_cast<unsigned>(a.Nq)) {
          record_status(a.status, -1 /* SPARGE_ERR_INVALID_ARG */);
          qrow = 0;
          qok = false;
        }
      }
      const uint4 *qsrc = reinterpret_cast<const uint4 *>(a.q + b * a.q_sb + hrow * a.q_sh + static_cast<int64_t>(qrow) * a.q_sn);
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = qok ? __ldg(qsrc + 8 * half + c) : make_uint4(0u, 0u, 0u, 0u);
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        tmem_st32(tl + QCOL + 32 * half, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&cs.q_full);
    } else if constexpr (DEC) {
      // this thread's Q row (zeros for the empty rows) into the shared-memory Q tile, 16-byte pieces
      // in the 128-byte swizzle the score product's descriptor expects
      const uint4 *qsrc = reinterpret_cast<const uint4 *>(a.q + b * a.q_sb + hrow * a.q_sh + static_cast<int64_t>(row_g) * a.q_sn);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const uint4 v = row_ok ? __ldg(qsrc + 8 * c + p) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4 *>(smem + L::OFF_Q + c * 16384 + r * 128 + ((p ^ (r & 7)) << 4)) = v;
        }
      fence_proxy_async_smem();  // generic writes read by the tensor core
      mbar_arrive(&cs.q_full);
    }
    float sq_blk = 1.f;
    const float *skrow = nullptr;
    if constexpr (QK8) {
      sq_blk = a.sq[(static_cast<int64_t>(b) * a.Hq + h) * a.nqb + i];
      skrow = a.sk + (static_cast<int64_t>(b) * a.Hkv + kvh) * a.nkb;
    }
    for (int t = 0;; ++t) {
      const int js = t % JRING;
      if (!mbar_wait(&cs.j_full[js], (t / JRING) & 1, abort, a.status)) {
        ok = false;
        break;
      }
      const int j = cs.jring[js];
      __syncwarp();
      if (lane == 0) mbar_arrive(&cs.j_empty[js]);
      if (j < 0) {  // tell the P.V issuer: phase t of p_full carries no tile (t = T, the tile count)
        // That is one more phase of p_full[t % NSB], with no score product before it: its previous
        // phase (tile t - NSB) must have been taken by the P.V issuer first, or both complete
        // before the issuer's parity wait for the earlier one, which then never passes.
        if (t >= NSB && !mbar_wait(&cs.pv_done[t % NSB], ((t - NSB) / NSB) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        if (r == 0) cs.row_end = t;
        mbar_arrive(&cs.p_full[t % NSB]);
        break;
      }
      T = t + 1;
      const int buf = t % NSB;
      if (!mbar_wait(&cs.s_full[buf], (t / NSB) & 1, abort, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sc = tl + SCOL0 + buf * 64;
      float x[64];  // raw scores Q.K^T of this row; hidden columns become -inf
      float mhw;    // their maximum, from the loads' max reduction
      {
        uint32_t r0[32], r1[32];
        float m0, m1;
        tmem_ld32_max(sc, r0, m0);
        tmem_ld32_max(sc + 32, r1, m1);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0[c]);
          x[32 + c] = __uint_as_float(r1[c]);
        }
        mhw = fmaxf(m0, m1);
      }
      // a tile with hidden columns (causal diagonal, ragged key tail) or rows past the query length;
      // the vote makes the branch warp-uniform, so interior tiles skip the masking code entirely
      // (decoding tiles always take it: their rows have their own heads' masks)
      const bool edge = DEC || (a.causal && KBLK * j + KBLK - 1 > a.off + QBLK * i) || (KBLK * j + KBLK > a.Nk) ||
                        (QBLK * i + QBLK > a.Nq);
      float mraw = mhw;
      if (__any_sync(0xffffffffu, edge)) {
        int lim = a.causal ? a.off + row_g - KBLK * j : 1 << 30;  // cols c > lim are hidden
        lim = min(lim, a.Nk - 1 - KBLK * j);
        if (!row_ok) lim = -1;
        if constexpr (DEC) {
          if (hmask != nullptr && __ldg(hmask + j) == 0) lim = -1;  // not kept by this row's head
        }
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = (c > lim) ? -INFINITY : x[c];
        // the maximum of what stays visible
        mraw = fmax3(x[0], x[1], x[2]);
#pragma unroll
        for (int c = 3; c < 63; c += 2) mraw = fmax3(mraw, x[c], x[c + 1]);
        mraw = fmaxf(mraw, x[63]);
      }
      // score multiplier of this tile (8-bit path: times the Q block and K block scales)
      const float tsc = QK8 ? a.scale_log2 * sq_blk * __ldg(skrow + j) : a.scale_log2;
      const float mloc = mraw * tsc;  // the multiplier is positive: max commutes with it
      const float m_new = fmaxf(m_run, mloc);
      const bool trailing = !row_ok || mloc == -INFINITY || m_new == -INFINITY || (mloc - m_new < lam_log2);
      const bool wskip = __all_sync(0xffffffffu, trailing);
      const bool resc = m_new > m_ref + RESC;
      const float alpha = resc ? fast_exp2(m_ref - m_new) : 1.f;
      if (__any_sync(0xffffffffu, resc) && t > 0) {
        // O must hold P_{t-1} V_{t-1} before it is rescaled
        // P.V of tile t - 1 completed: phase (t - 1) / NSB of its buffer's barrier (that barrier's
        // phases are NSB tiles apart, so a pending P.V of tile t - 2 cannot alias the wait)
        if (!mbar_wait(&cs.pv_done[(t - 1) % NSB], ((t - 1) / NSB) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float2 al2 = make_float2(alpha, alpha);
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t rr[32];
          tmem_ld32(tl + 32 * q, rr);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 o2 = fmul2(make_float2(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1])), al2);
            rr[2 * c] = __float_as_uint(o2.x);
            rr[2 * c + 1] = __float_as_uint(o2.y);
          }
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            lo[c] = rr[c];
            hi[c] = rr[16 + c];
          }
          tmem_st16(tl + 32 * q, lo);
          tmem_st16(tl + 32 * q + 16, hi);
        }
      }
      if (resc) m_ref = m_new;
      m_run = m_new;
      l *= alpha;
      // P = 2^(x * scale_log2 - m_ref); a row whose reference is still -inf has only hidden columns
      const float nref = (m_ref == -INFINITY) ? 0.f : POFF - m_ref;
      const float2 sc2 = make_float2(tsc, tsc), nr2 = make_float2(nref, nref);
      float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[32];  // P of columns 2c, 2c + 1 (two f16, or two e4m3 in the low half)
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float2 e2 = ffma2(make_float2(x[2 * c], x[2 * c + 1]), sc2, nr2);
        const float2 p2 = make_float2(fast_exp2(e2.x), fast_exp2(e2.y));
        rs2[c & 3] = fadd2(rs2[c & 3], p2);  // four independent chains
        pk[c] = PV8 ? pack_e4m3x2(p2.x, p2.y) : (DEC ? pack_bf16x2(p2.x, p2.y) : pack_f16x2(p2.x, p2.y));
      }
      {
        const float2 rs = fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3]));
        l += rs.x + rs.y;
      }
      if constexpr (PV8) {
        uint32_t w[16];  // 4 e4m3 per column, keys in order
#pragma unroll
        for (int c = 0; c < 16; ++c) w[c] = wskip ? 0u : (pk[2 * c] | (pk[2 * c + 1] << 16));
        tmem_st16(sc, w);
      } else if (wskip) {
        uint32_t z[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) z[c] = 0u;
        tmem_st32(sc, z);
      } else {
        tmem_st32(sc, pk);
      }
      tmem_st_wait();
      if (lane == 0) cs.skip[buf][warp] = wskip ? 1 : 0;
      nskip += (wskip && (DEC ? warp * 32 < a.G * a.Nq : QBLK * i + warp * 32 < a.Nq)) ? 1 : 0;
      tc_fence_before();
      mbar_arrive(&cs.p_full[buf]);
    }
    // ------------------------------------ epilogue ------------------------------------
    bool have_o = false;
    if (T > 0 && ok) {
      ok = mbar_wait(&cs.mma_done, 0, abort, a.status);  // every P.V product has completed
      tc_fence_after();
      have_o = ok && cs.pv_any != 0;
    }
    if constexpr (DEC) {
      // decoding tile: this row's partial result over the chunk, relative to 2^m_ref (O and l share
      // the exponent reference), for the combining kernel; rows that saw no visible key give l = 0
      const int chunk = blockIdx.x % a.nchunk, bk = blockIdx.x / a.nchunk;
      const int64_t prow = (static_cast<int64_t>(bk) * a.nchunk + chunk) * 128 + r;
      float4 *po = reinterpret_cast<float4 *>(a.part_o + prow * D);
      // only the G Nq rows the combining kernel reads (a warp of empty rows skips it all)
      const bool warp_rows = __any_sync(0xffffffffu, row_ok);
#pragma unroll 1
      for (int q = 0; q < (warp_rows ? D / 16 : 0); ++q) {
        uint32_t rr[16];
        if (have_o) {
          tmem_ld16(tl + 16 * q, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) rr[c] = 0u;
        }
        if (row_ok)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            po[4 * q + c] = make_float4(__uint_as_float(rr[4 * c]), __uint_as_float(rr[4 * c + 1]),
                                        __uint_as_float(rr[4 * c + 2]), __uint_as_float(rr[4 * c + 3]));
      }
      if (row_ok) {
        const bool any = have_o && l > 0.f;
        a.part_ml[2 * prow] = any ? m_ref : -INFINITY;
        a.part_ml[2 * prow + 1] = any ? l : 0.f;
      }
    } else {
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const float *svrow = PV8 ? a.sv + (static_cast<int64_t>(b) * a.Hkv + kvh) * D : nullptr;
      // the output row: token row_g, or token perm[row_g] of o under a token order (an entry outside
      // 0..N-1 is reported and its row left unwritten)
      int orow_t = row_g;
      bool write_row = row_ok;
      if (a.perm && row_ok) {
        orow_t = __ldg(a.perm + row_g);
        if (static_cast<unsigned>(orow_t) >= static_cast<unsigned>(a.Nq)) {
          record_status(a.status, -1 /* SPARGE_ERR_INVALID_ARG */);
          write_row = false;
          orow_t = 0;
        }
      }
      __nv_bfloat16 *orow = a.o + b * a.o_sb + h * a.o_sh + static_cast<int64_t>(orow_t) * a.o_sn;
  #pragma unroll 1
      for (int q = 0; q < D / 16; ++q) {
        uint32_t rr[16];
        if (have_o) {
          tmem_ld16(tl + 16 * q, rr);
          tmem_ld_wait();
        } else {
  #pragma unroll
          for (int c = 0; c < 16; ++c) rr[c] = 0u;
        }
        if constexpr (PV8) {  // undo the per-channel V scale
  #pragma unroll
          for (int c = 0; c < 16; c += 4) {
            const float4 s4 = __ldg(reinterpret_cast<const float4 *>(svrow + 16 * q + c));
            rr[c] = __float_as_uint(__uint_as_float(rr[c]) * s4.x);
            rr[c + 1] = __float_as_uint(__uint_as_float(rr[c + 1]) * s4.y);
            rr[c + 2] = __float_as_uint(__uint_as_float(rr[c + 2]) * s4.z);
            rr[c + 3] = __float_as_uint(__uint_as_float(rr[c + 3]) * s4.w);
          }
        }
        uint4 o0, o1;
        o0.x = pack_bf16x2(__uint_as_float(rr[0]) * inv_l, __uint_as_float(rr[1]) * inv_l);
        o0.y = pack_bf16x2(__uint_as_float(rr[2]) * inv_l, __uint_as_float(rr[3]) * inv_l);
        o0.z = pack_bf16x2(__uint_as_float(rr[4]) * inv_l, __uint_as_float(rr[5]) * inv_l);
        o0.w = pack_bf16x2(__uint_as_float(rr[6]) * inv_l, __uint_as_float(rr[7]) * inv_l);
        o1.x = pack_bf16x2(__uint_as_float(rr[8]) * inv_l, __uint_as_float(rr[9]) * inv_l);
        o1.y = pack_bf16x2(__uint_as_float(rr[10]) * inv_l, __uint_as_float(rr[11]) * inv_l);
        o1.z = pack_bf16x2(__uint_as_float(rr[12]) * inv_l, __uint_as_float(rr[13]) * inv_l);
        o1.w = pack_bf16x2(__uint_as_float(rr[14]) * inv_l, __uint_as_float(rr[15]) * inv_l);
        if (write_row) {
          *reinterpret_cast<uint4 *>(orow + 16 * q) = o0;
          *reinterpret_cast<uint4 *>(orow + 16 * q + 8) = o1;
        }
      }
    }
    if (a.stats && lane == 0 && nskip) atomicAdd(a.stats + 2, static_cast<unsigned long long>(nskip));
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

template <int D, int KST, int VST, bool QK8, bool PV8, bool DEC = false>
cudaError_t launch_t(const AttnLaunch &l, const AttnArgs &a, cudaStream_t st) {
  // each CTA allocates 256 TMEM columns, half of the SM's: at least 77 KB of shared memory keeps a
  // third CTA off the SM (it would only wait in tcgen05.alloc)
  constexpr uint32_t MIN_SMEM = 77u * 1024u;
  const uint32_t smem = Smem<D, KST, VST, QK8, PV8>::TOTAL > MIN_SMEM ? Smem<D, KST, VST, QK8, PV8>::TOTAL : MIN_SMEM;
  static std::atomic<unsigned long long> smem_set{0};
  if (cudaError_t e = set_smem_limit_once(bsattn_kernel<D, KST, VST, QK8, PV8, DEC>, static_cast<int>(smem), smem_set);
      e != cudaSuccess)
    return e;
  const int64_t grid = DEC ? static_cast<int64_t>(a.B) * a.Hkv * a.nchunk : static_cast<int64_t>(a.B) * a.Hq * a.nqb;
  bsattn_kernel<D, KST, VST, QK8, PV8, DEC><<<static_cast<unsigned>(grid), NTHREADS, smem, st>>>(l.tq, l.tk, l.tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bsattn(const AttnLaunch &l, cudaStream_t st) {
  AttnArgs a;
  a.mask = l.mask;
  a.o = static_cast<__nv_bfloat16 *>(l.o);
  a.o_sb = l.o_sb; a.o_sh = l.o_sh; a.o_sn = l.o_sn;
  a.B = l.B; a.Hq = l.Hq; a.Hkv = l.Hkv; a.G = l.Hq / l.Hkv;
  a.Nq = l.Nq;
  a.Nk = l.Nk;
  a.off = l.Nk - l.Nq;
  a.nqb = (l.Nq + QBLK - 1) / QBLK;
  a.nkb = (l.Nk + KBLK - 1) / KBLK;
  a.causal = l.causal;
  const float LOG2E = 1.4426950408889634f;
  a.scale_log2 = l.scale * LOG2E;
  a.lam_log2 = (l.lambda == -INFINITY) ? -INFINITY : l.lambda * LOG2E;
  a.lam_h = l.lambda_h;
  a.perm = l.perm;
  a.stats = l.stats;
  a.status = l.status;
  a.sq = l.sq;
  a.sk = l.sk;
  a.sv = l.sv;
  a.q = static_cast<const __nv_bfloat16 *>(l.q);
  a.q_sb = l.q_sb; a.q_sh = l.q_sh; a.q_sn = l.q_sn;
  a.qperm = l.qperm;
  if (static_cast<int64_t>(a.B) * a.Hq * a.nqb == 0) return cudaSuccess;
  if (l.q8 != 0 && l.d != 128) return cudaErrorInvalidValue;
  if (l.decode) {  // bf16 only: the host picks this path for few queries per head, lambda off
    if (l.q8 != 0 || a.G * a.Nq > 128 || l.nchunk <= 0) return cudaErrorInvalidValue;
    a.nchunk = l.nchunk;
    a.chunk_blocks = l.chunk_blocks;
    a.part_o = l.part_o;
    a.part_ml = l.part_ml;
    a.dlist = l.dlist;
    a.dcount = l.dcount;
    if (a.mask) {
      if (!l.dlist || !l.dcount) return cudaErrorInvalidValue;
      if (cudaError_t e = launch_decode_union(a.mask, a.B, a.Hq, a.Hkv, a.nqb, a.nkb, l.dlist, l.dcount, st);
          e != cudaSuccess)
        return e;
    }
    cudaError_t e = l.d == 128 ? launch_t<128, 3, 2, false, false, true>(l, a, st)
                               : launch_t<64, 4, 3, false, false, true>(l, a, st);
    if (e != cudaSuccess) return e;
    return launch_decode_combine(l.part_o, l.part_ml, l.nchunk, a.B, a.Hq, a.Hkv, a.Nq, l.d, a.o, a.o_sb, a.o_sh, a.o_sn,
                                 st);
  }
  if (l.q8 == 3) return launch_t<128, 3, 3, false, true>(l, a, st);  // bf16 Q.K^T, e4m3 P.V
  if (l.q8 == 2) return launch_t<128, 4, 3, true, true>(l, a, st);
  if (l.q8 == 1) return launch_t<128, 4, 2, true, false>(l, a, st);
  return l.d == 128 ? launch_t<128, 3, 2, false, false>(l, a, st) : launch_t<64, 4, 3, false, false>(l, a, st);
}

}  // namespace sparge
