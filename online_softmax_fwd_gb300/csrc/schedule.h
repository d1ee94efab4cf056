// Static work lists for the persistent attention kernels.
//
// A work item is one pair of 128-row Q tiles of one (batch, head). Items are
// numbered in bands of `band` heads (heads whose K and V fit in L2 together);
// inside a band the pairs come last-first, i.e. heaviest first under the
// causal mask, head index fastest. The host assigns the items to CTAs by list
// scheduling -- in that order, each item goes to the CTA that a cost model
// says becomes free first -- so CTAs finish together even though causal items
// differ in cost, while the CTAs busy at any moment still work on one band.
// The list travels to the kernel as a launch parameter; no device memory is
// involved.
#pragma once

#include <cstdint>

namespace attn {

constexpr int kListMaxCtas = 256;
constexpr int kListMaxItems = 8192;

// CTA c runs items item[first[c]], ..., item[first[c + 1] - 1] in that order.
struct WorkList {
  uint16_t first[kListMaxCtas + 1];
  uint16_t item[kListMaxItems];
};

// (head, pair) of item `it` in the banded order above.
__host__ __device__ inline void item_coords(int it, int bh, int n_pairs, int band, int& head, int& pair) {
  const int per_band = band * n_pairs;
  const int band_id = it / per_band;
  const int r = it - band_id * per_band;
  const int heads = (bh - band_id * band) < band ? (bh - band_id * band) : band;
  pair = n_pairs - 1 - r / heads;
  head = band_id * band + r % heads;
}

// Builds the list for `ctas` CTAs (cached per shape). Returns false, leaving
// `out` untouched, when the items or CTAs exceed the list's capacity.
bool work_list_for(int bh, int n_pairs, int n_kv_blocks, int band, bool causal, int ctas, WorkList* out);

}  // namespace attn
