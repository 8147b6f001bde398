// Host-side builders of the Hilbert-curve token order (SpargeAttention summary page: a
// space-filling Hilbert-curve reordering improves token locality for visual tasks).
// Integer only; the result is a gather permutation in host memory.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#include "../../include/sparge.h"

namespace {

int order_for(int64_t extent) {
  int o = 1;
  while ((int64_t(1) << o) < extent) ++o;
  return o;
}

// 2-D: walk the levels from the coarsest; at each level the quadrant number is (3 rx) xor ry
// (lower-left 0, upper-left 1, upper-right 2, lower-right 3), and the local frame is turned so
// that the sub-curve again runs from its own (0,0) to (h-1,0): the lower-left quadrant is
// mirrored about the diagonal, the lower-right one about the anti-diagonal.
uint64_t hilbert2(uint32_t x, uint32_t y, int order) {
  uint64_t d = 0;
  for (uint32_t h = 1u << (order - 1); h; h >>= 1) {
    const uint32_t rx = (x & h) ? 1u : 0u, ry = (y & h) ? 1u : 0u;
    d += static_cast<uint64_t>(h) * h * ((3u * rx) ^ ry);
    x &= h - 1;
    y &= h - 1;
    if (!ry) {
      if (rx) {
        x = h - 1 - x;
        y = h - 1 - y;
      }
      std::swap(x, y);
    }
  }
  return d;
}

// 3-D: J. Skilling, "Programming the Hilbert curve" (AIP Conf. Proc. 707, 2004).  The axes are
// turned into the "transposed" Hilbert index in place, whose bits, read most significant
// first and axis 0 first, form the index.
uint64_t hilbert3(uint32_t a0, uint32_t a1, uint32_t a2, int bits) {
  uint32_t X[3] = {a0, a1, a2};
  const uint32_t top = 1u << (bits - 1);
  for (uint32_t q = top; q > 1; q >>= 1) {
    const uint32_t low = q - 1;
    for (int i = 0; i < 3; ++i) {
      if (X[i] & q) {
        X[0] ^= low;
      } else {
        const uint32_t t = (X[0] ^ X[i]) & low;
        X[0] ^= t;
        X[i] ^= t;
      }
    }
  }
  X[1] ^= X[0];
  X[2] ^= X[1];
  uint32_t t = 0;
  for (uint32_t q = top; q > 1; q >>= 1)
    if (X[2] & q) t ^= q - 1;
  for (int i = 0; i < 3; ++i) X[i] ^= t;
  uint64_t idx = 0;
  for (int bit = bits - 1; bit >= 0; --bit)
    for (int i = 0; i < 3; ++i) idx = (idx << 1) | ((X[i] >> bit) & 1u);
  return idx;
}

void order_by_keys(const std::vector<uint64_t> &keys, int n_prefix, int32_t *perm) {
  std::vector<int32_t> idx(keys.size());
  std::iota(idx.begin(), idx.end(), 0);
  std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return keys[a] < keys[b]; });
  for (int t = 0; t < n_prefix; ++t) perm[t] = t;
  for (size_t t = 0; t < idx.size(); ++t) perm[n_prefix + t] = n_prefix + idx[t];
}

}  // namespace

extern "C" {

int sparge_hilbert_perm_2d(int n_prefix, int H, int W, int32_t *perm_host) {
  if (!perm_host || n_prefix < 0 || H <= 0 || W <= 0 || int64_t(H) * W > (int64_t(1) << 30))
    return SPARGE_ERR_INVALID_ARG;
  const int k = order_for(std::max(H, W));
  std::vector<uint64_t> keys(static_cast<size_t>(H) * W);
  for (int r = 0; r < H; ++r)
    for (int c = 0; c < W; ++c) keys[static_cast<size_t>(r) * W + c] = hilbert2(c, r, k);
  order_by_keys(keys, n_prefix, perm_host);
  return SPARGE_OK;
}

int sparge_hilbert_perm_3d(int n_prefix, int T, int H, int W, int32_t *perm_host) {
  if (!perm_host || n_prefix < 0 || T <= 0 || H <= 0 || W <= 0 || int64_t(T) * H * W > (int64_t(1) << 30))
    return SPARGE_ERR_INVALID_ARG;
  const int k = order_for(std::max(T, std::max(H, W)));
  if (3 * k > 63) return SPARGE_ERR_UNSUPPORTED;
  std::vector<uint64_t> keys(static_cast<size_t>(T) * H * W);
  size_t n = 0;
  for (int t = 0; t < T; ++t)
    for (int r = 0; r < H; ++r)
      for (int c = 0; c < W; ++c) keys[n++] = hilbert3(t, r, c, k);
  order_by_keys(keys, n_prefix, perm_host);
  return SPARGE_OK;
}

}  // extern "C"
