// Host side of the static work lists: list scheduling with a cost model, and a
// small cache so a shape is scheduled once.
#include "schedule.h"

#include <cstring>
#include <deque>
#include <functional>
#include <memory>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

namespace attn {
namespace {

struct Key {
  int bh, n_pairs, n_kv_blocks, band, causal, ctas;
  bool operator==(const Key& o) const {
    return bh == o.bh && n_pairs == o.n_pairs && n_kv_blocks == o.n_kv_blocks && band == o.band &&
           causal == o.causal && ctas == o.ctas;
  }
};

constexpr size_t kCacheEntries = 32;

// Cost of a pair in units of one 128 x 128 block of one Q tile (its S and
// P V products and its softmax): tile 0 sees 2p + 1 key blocks under the
// causal mask, tile 1 2p + 2, both all of them otherwise; the epilogue and the
// hand-over between items cost about three more units.
long long pair_cost(int pair, int n_kv_blocks, bool causal) {
  auto cap = [&](long long n) { return n < n_kv_blocks ? n : n_kv_blocks; };
  const long long n0 = causal ? cap(2LL * pair + 1) : n_kv_blocks;
  const long long n1 = causal ? cap(2LL * pair + 2) : n_kv_blocks;
  return n0 + n1 + 3;
}

void build(const Key& k, WorkList* wl) {
  const int total = k.bh * k.n_pairs;
  std::vector<std::vector<uint16_t>> lists(k.ctas);
  // (time the CTA becomes free, CTA); ties go to the lower CTA index
  using Slot = std::pair<long long, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < k.ctas; ++c) free_at.push({0, c});
  for (int it = 0; it < total; ++it) {
    int head, pair;
    item_coords(it, k.bh, k.n_pairs, k.band, head, pair);
    Slot s = free_at.top();
    free_at.pop();
    lists[s.second].push_back(static_cast<uint16_t>(it));
    s.first += pair_cost(pair, k.n_kv_blocks, k.causal != 0);
    free_at.push(s);
  }
  std::memset(wl, 0, sizeof(*wl));
  int pos = 0;
  for (int c = 0; c < k.ctas; ++c) {
    wl->first[c] = static_cast<uint16_t>(pos);
    for (uint16_t it : lists[c]) wl->item[pos++] = it;
  }
  for (int c = k.ctas; c <= kListMaxCtas; ++c) wl->first[c] = static_cast<uint16_t>(pos);
}

}  // namespace

bool work_list_for(int bh, int n_pairs, int n_kv_blocks, int band, bool causal, int ctas, WorkList* out) {
  if (bh <= 0 || n_pairs <= 0 || band <= 0 || ctas <= 0 || ctas > kListMaxCtas) return false;
  if (static_cast<long long>(bh) * n_pairs > kListMaxItems) return false;
  static std::mutex mu;
  static std::deque<std::pair<Key, std::unique_ptr<WorkList>>> cache;
  const Key key{bh, n_pairs, n_kv_blocks, band, causal ? 1 : 0, ctas};
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& e : cache)
    if (e.first == key) {
      std::memcpy(out, e.second.get(), sizeof(WorkList));
      return true;
    }
  auto wl = std::make_unique<WorkList>();
  build(key, wl.get());
  std::memcpy(out, wl.get(), sizeof(WorkList));
  if (cache.size() == kCacheEntries) cache.pop_front();
  cache.emplace_back(key, std::move(wl));
  return true;
}

}  // namespace attn
