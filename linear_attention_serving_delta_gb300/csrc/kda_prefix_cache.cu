// kda_prefix_cache.cu -- the snapshot retention policy of a serving host:
// which states of earlier prompts to keep in a fixed pool of device rows,
// and which one a new prompt can resume from.  Host code only; contract in
// include/kda.h.
//
// The recurrent state is overwritten as a prompt advances, so reusing the
// work of an earlier prompt needs a saved copy of the state at a shared
// prefix ("Kimi K3: The Manos, The Mythos, The Legendos", Context: the
// engine keeps selected checkpoints, prompt boundaries among them; more
// checkpoints cost memory and save recomputation, so the retention policy
// matters).  The policy here:
//   * an entry is the state after the first p tokens of some prompt, keyed
//     by p and two independent 64-bit polynomial hashes of those p token ids;
//   * a lookup returns the longest cached prefix of the new prompt;
//   * when the pool is full, an interval checkpoint (one taken every few
//     chunks) is evicted before a prompt-boundary checkpoint, least recently
//     used first within each class: a boundary state is where a later turn of
//     the same conversation resumes, so it is worth more;
//   * a reservation places prompt-boundary checkpoints first, then interval
//     checkpoints from the latest position back (a later checkpoint saves
//     more recomputation), and never evicts a row it placed itself or the
//     row the prefill resumes from.
#include <cstdint>
#include <list>
#include <map>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/kda.h"

namespace {

constexpr uint64_t kMul1 = 0x9E3779B97F4A7C15ull;  // odd multipliers of the two hashes
constexpr uint64_t kMul2 = 0xC2B2AE3D27D4EB4Full;

struct Key {
  uint64_t h1, h2;
  int64_t len;
  bool operator==(const Key& o) const { return h1 == o.h1 && h2 == o.h2 && len == o.len; }
};
struct KeyHash {
  size_t operator()(const Key& k) const { return (size_t)(k.h1 ^ (k.h2 * 31) ^ (uint64_t)k.len); }
};

// Hash state after consuming tokens one by one (token id + 1, so that id 0 counts).
struct Rolling {
  uint64_t h1 = 0, h2 = 0;
  void push(int32_t t) {
    const uint64_t x = (uint64_t)(uint32_t)t + 1;
    h1 = h1 * kMul1 + x;
    h2 = (h2 ^ x) * kMul2;
  }
};

struct Row {
  bool live = false;
  bool boundary = false;
  Key key{};
  std::list<int32_t>::iterator lru;  // position in its class's recency list
};

}  // namespace

struct kda_prefix_cache {
  std::mutex mu;
  std::vector<Row> rows;
  std::vector<int32_t> free_rows;
  std::unordered_map<Key, int32_t, KeyHash> index;
  std::map<int64_t, int64_t> lengths;        // cached prefix length -> entries
  std::list<int32_t> lru[2];                 // [interval, boundary]: front = least recent

  void touch(int32_t r) {
    Row& x = rows[r];
    std::list<int32_t>& l = lru[x.boundary ? 1 : 0];
    l.splice(l.end(), l, x.lru);
  }
  void drop(int32_t r) {
    Row& x = rows[r];
    index.erase(x.key);
    auto it = lengths.find(x.key.len);
    if (it != lengths.end() && --it->second == 0) lengths.erase(it);
    lru[x.boundary ? 1 : 0].erase(x.lru);
    x.live = false;
  }
  void put(int32_t r, const Key& k, bool boundary) {
    Row& x = rows[r];
    x.live = true;
    x.boundary = boundary;
    x.key = k;
    index[k] = r;
    ++lengths[k.len];
    std::list<int32_t>& l = lru[boundary ? 1 : 0];
    x.lru = l.insert(l.end(), r);
  }
  // a row to reuse: a free one, else the least recently used interval entry,
  // else the least recently used boundary entry; rows in `held` are skipped
  int32_t victim(const std::vector<char>& held) {
    for (size_t i = free_rows.size(); i-- > 0;) {
      const int32_t r = free_rows[i];
      if (held[r]) continue;
      free_rows[i] = free_rows.back();
      free_rows.pop_back();
      return r;
    }
    for (int cls = 0; cls < 2; ++cls)
      for (int32_t r : lru[cls])
        if (!held[r]) {
          drop(r);
          return r;
        }
    return -1;
  }
};

extern "C" {

kda_prefix_cache* kda_prefix_cache_create(int64_t num_rows) {
  if (num_rows < 1 || num_rows > INT32_MAX) return nullptr;
  kda_prefix_cache* c = new (std::nothrow) kda_prefix_cache();
  if (!c) return nullptr;
  try {
    c->rows.resize((size_t)num_rows);
    c->free_rows.reserve((size_t)num_rows);
    for (int64_t r = num_rows - 1; r >= 0; --r) c->free_rows.push_back((int32_t)r);
  } catch (...) {
    delete c;
    return nullptr;
  }
  return c;
}

void kda_prefix_cache_destroy(kda_prefix_cache* c) { delete c; }

int64_t kda_prefix_cache_entries(kda_prefix_cache* c) {
  if (!c) return -1;
  std::lock_guard<std::mutex> lock(c->mu);
  return (int64_t)c->index.size();
}

int64_t kda_prefix_cache_lookup(kda_prefix_cache* c, const int32_t* tokens, int64_t n, int32_t* row) {
  if (!c || n < 0 || (n > 0 && !tokens) || !row) return -1;
  std::lock_guard<std::mutex> lock(c->mu);
  *row = -1;
  int64_t best = 0;
  Rolling h;
  int64_t done = 0;
  // probe only the lengths some entry has, in increasing order
  for (auto it = c->lengths.begin(); it != c->lengths.end() && it->first <= n; ++it) {
    const int64_t len = it->first;
    for (; done < len; ++done) h.push(tokens[done]);
    auto f = c->index.find(Key{h.h1, h.h2, len});
    if (f != c->index.end()) {
      best = len;
      *row = f->second;
    }
  }
  if (*row >= 0) c->touch(*row);
  return best;
}

int64_t kda_prefix_cache_reserve(kda_prefix_cache* c, const int32_t* tokens, int64_t n,
                                 const int64_t* pos, const uint8_t* is_boundary, int64_t m,
                                 int32_t keep_row, int32_t* rows_out) {
  if (!c || n < 0 || m < 0 || (n > 0 && !tokens) || (m > 0 && (!pos || !rows_out))) return -1;
  if (keep_row < -1 || keep_row >= (int64_t)c->rows.size()) return -1;
  for (int64_t i = 0; i < m; ++i)
    if (pos[i] < 1 || pos[i] > n || (i > 0 && pos[i] <= pos[i - 1])) return -1;
  std::lock_guard<std::mutex> lock(c->mu);
  // keys of every position, in one pass over the tokens
  std::vector<Key> keys((size_t)m);
  {
    Rolling h;
    int64_t done = 0;
    for (int64_t i = 0; i < m; ++i) {
      for (; done < pos[i]; ++done) h.push(tokens[done]);
      keys[(size_t)i] = Key{h.h1, h.h2, pos[i]};
    }
  }
  // placement order: boundaries first, then the rest from the latest back
  std::vector<int64_t> order;
  order.reserve((size_t)m);
  for (int64_t i = m - 1; i >= 0; --i)
    if (is_boundary && is_boundary[i]) order.push_back(i);
  for (int64_t i = m - 1; i >= 0; --i)
    if (!(is_boundary && is_boundary[i])) order.push_back(i);
  std::vector<char> held(c->rows.size(), 0);
  if (keep_row >= 0) held[keep_row] = 1;  // the row the prefill resumes from
  int64_t placed = 0;
  for (int64_t i : order) {
    rows_out[i] = -1;
    const bool bnd = is_boundary && is_boundary[i];
    auto f = c->index.find(keys[(size_t)i]);
    if (f != c->index.end()) {  // already kept: no need to write it again
      const int32_t r = f->second;
      held[r] = 1;
      if (bnd && !c->rows[r].boundary) {  // promote to the boundary class
        c->drop(r);
        c->put(r, keys[(size_t)i], true);
      } else {
        c->touch(r);
      }
      continue;
    }
    const int32_t r = c->victim(held);
    if (r < 0) continue;  // every row is held by this reservation
    c->put(r, keys[(size_t)i], bnd);
    held[r] = 1;
    rows_out[i] = r;
    ++placed;
  }
  return placed;
}

int64_t kda_prefix_cache_forget(kda_prefix_cache* c, const int32_t* rows, int64_t m) {
  if (!c || m < 0 || (m > 0 && !rows)) return -1;
  for (int64_t i = 0; i < m; ++i)
    if (rows[i] < -1 || rows[i] >= (int64_t)c->rows.size()) return -1;
  std::lock_guard<std::mutex> lock(c->mu);
  int64_t freed = 0;
  for (int64_t i = 0; i < m; ++i) {
    const int32_t r = rows[i];
    if (r < 0 || !c->rows[r].live) continue;  // -1 entries of a reservation, or already free
    c->drop(r);
    c->free_rows.push_back(r);
    ++freed;
  }
  return freed;
}

}  // extern "C"
