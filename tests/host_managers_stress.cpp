// Stress driver for the library's host-side managers (pkv_bm_* and pkv_pc_*),
// built with AddressSanitizer and UndefinedBehaviorSanitizer by
// tests/test_host_sanitizers.py.  Long seeded random streams of the calls a
// serving loop makes (add, fork, append, free; prefix hits, evictions,
// refused appends), with the managers' invariants checked through the public
// API after every call:
//   * every block is either free or referenced: num_free + #(refcount > 0)
//     equals the pool size;
//   * a block's count equals the number of live tables holding it;
//   * a table holds ceil(tokens / block_size) blocks;
//   * (prefix cache) a cached block's key equals the chained key of the
//     tokens the sequence put there.
// Exit status 0 when every check holds; the sanitizers abort on any memory or
// undefined-behaviour error.
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <random>
#include <vector>

#include "../include/paged_kv.h"

namespace {

int g_failures = 0;
#define CHECK(cond)                                                      \
  do {                                                                   \
    if (!(cond)) {                                                       \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      if (++g_failures > 20) return false;                               \
    }                                                                    \
  } while (0)

template <typename Table, typename Count, typename Free>
bool pool_invariants(int N, int B, const std::vector<int64_t> &live, Table table, Count count,
                     Free num_free) {
  std::vector<int> held(N, 0);
  for (int64_t s : live) {
    std::vector<int32_t> t(4096);
    int nb = 0;
    int64_t tokens = 0;
    CHECK(table(s, t.data(), (int)t.size(), &nb, &tokens) == PKV_OK);
    CHECK(nb == (int)((tokens + B - 1) / B));
    for (int i = 0; i < nb; ++i) {
      CHECK(t[i] >= 0 && t[i] < N);
      if (t[i] >= 0 && t[i] < N) ++held[t[i]];
    }
  }
  int used = 0;
  for (int b = 0; b < N; ++b) {
    CHECK(count(b) == held[b]);
    used += count(b) > 0;
  }
  CHECK(num_free() + used == N);
  return true;
}

bool stress_block_manager(uint32_t seed, int N, int B) {
  std::mt19937 rng(seed);
  std::vector<int32_t> order(N);
  for (int i = 0; i < N; ++i) order[i] = i;
  std::shuffle(order.begin(), order.end(), rng);
  pkv_block_manager *bm = pkv_bm_create(N, B, order.data());
  CHECK(bm != nullptr);
  std::vector<int64_t> live;
  int64_t next = 0;
  auto table = [&](int64_t s, int32_t *o, int cap, int *nb, int64_t *nt) {
    return pkv_bm_table(bm, s, o, cap, nb, nt);
  };
  auto count = [&](int b) { return pkv_bm_refcount(bm, b); };
  auto nfree = [&]() { return pkv_bm_num_free(bm); };
  for (int step = 0; step < 3000; ++step) {
    const int op = (int)(rng() % 100);
    if (op < 20 || live.empty()) {
      CHECK(pkv_bm_add_sequence(bm, next) == PKV_OK);
      live.push_back(next++);
    } else if (op < 35) {
      const int64_t parent = live[rng() % live.size()];
      CHECK(pkv_bm_fork(bm, parent, next) == PKV_OK);
      live.push_back(next++);
    } else if (op < 85) {
      // a batch of appends, some sequences more than once
      const int n = 1 + (int)(rng() % 24);
      std::vector<int64_t> seqs(n), slots(n), pairs(2 * n);
      for (int i = 0; i < n; ++i) seqs[i] = live[rng() % live.size()];
      int np = -1;
      const pkv_status st = pkv_bm_append(bm, seqs.data(), n, slots.data(), pairs.data(), &np);
      CHECK(st == PKV_OK || st == PKV_ERR_NO_BLOCKS);
      if (st == PKV_OK) {
        CHECK(np >= 0 && np <= n);
        for (int i = 0; i < n; ++i) CHECK(slots[i] >= 0 && slots[i] < (int64_t)N * B);
        for (int i = 0; i < np; ++i)
          CHECK(pairs[2 * i] >= 0 && pairs[2 * i] < N && pairs[2 * i + 1] >= 0 &&
                pairs[2 * i + 1] < N && pairs[2 * i] != pairs[2 * i + 1]);
      }
    } else {
      const size_t i = rng() % live.size();
      CHECK(pkv_bm_free_sequence(bm, live[i]) == PKV_OK);
      live.erase(live.begin() + (long)i);
    }
    // errors leave the manager unchanged
    if (step % 97 == 0) {
      if (!live.empty()) CHECK(pkv_bm_add_sequence(bm, live[0]) != PKV_OK);
      CHECK(pkv_bm_free_sequence(bm, next + 1000) != PKV_OK);
      CHECK(pkv_bm_fork(bm, next + 1000, next + 1001) != PKV_OK);
    }
    if (step % 10 == 0 && !pool_invariants(N, B, live, table, count, nfree)) return false;
  }
  for (int64_t s : live) CHECK(pkv_bm_free_sequence(bm, s) == PKV_OK);
  CHECK(pkv_bm_num_free(bm) == N);
  pkv_bm_destroy(bm);
  return g_failures == 0;
}

bool stress_prefix_cache(uint32_t seed, int N, int B) {
  std::mt19937 rng(seed);
  std::vector<int32_t> order(N);
  for (int i = 0; i < N; ++i) order[i] = i;
  std::shuffle(order.begin(), order.end(), rng);
  pkv_prefix_cache *pc = pkv_pc_create(N, B, order.data());
  CHECK(pc != nullptr);
  std::vector<std::vector<int32_t>> systems(4);
  for (auto &sp : systems) {
    sp.resize(B + rng() % (5 * B));
    for (auto &t : sp) t = (int32_t)(rng() % 100);
  }
  std::map<int64_t, std::vector<int32_t>> tokens;   // every token of each live sequence
  std::map<int64_t, uint64_t> extra;
  std::vector<int64_t> live;
  int64_t next = 0;
  auto table = [&](int64_t s, int32_t *o, int cap, int *nb, int64_t *nt) {
    return pkv_pc_table(pc, s, o, cap, nb, nt);
  };
  auto count = [&](int b) { return pkv_pc_refcount(pc, b); };
  auto nfree = [&]() { return pkv_pc_num_free(pc); };
  for (int step = 0; step < 3000; ++step) {
    const int op = (int)(rng() % 100);
    if (op < 40 || live.empty()) {
      std::vector<int32_t> prompt;
      if (rng() % 5) prompt = systems[rng() % systems.size()];
      const int own = 1 + (int)(rng() % (3 * B));
      for (int i = 0; i < own; ++i) prompt.push_back((int32_t)(rng() % 100));
      const uint64_t ex = rng() % 2;
      int cached = -1;
      CHECK(pkv_pc_add_sequence(pc, next, prompt.data(), (int)prompt.size(), ex, &cached) ==
            PKV_OK);
      CHECK(cached >= 0 && cached % B == 0 && cached < (int)prompt.size());
      std::vector<int64_t> slots(prompt.size());
      const int rest = (int)prompt.size() - cached;
      const pkv_status st = pkv_pc_append(pc, next, prompt.data() + cached, rest, slots.data());
      CHECK(st == PKV_OK || st == PKV_ERR_NO_BLOCKS);
      if (st == PKV_OK) {
        tokens[next] = prompt;
        extra[next] = ex;
        live.push_back(next);
      } else {
        CHECK(pkv_pc_free_sequence(pc, next) == PKV_OK);
      }
      ++next;
    } else if (op < 75) {
      const int64_t s = live[rng() % live.size()];
      const int n = 1 + (int)(rng() % (2 * B));
      std::vector<int32_t> more(n);
      for (auto &t : more) t = (int32_t)(rng() % 100);
      std::vector<int64_t> slots(n);
      const pkv_status st = pkv_pc_append(pc, s, more.data(), n, slots.data());
      CHECK(st == PKV_OK || st == PKV_ERR_NO_BLOCKS);
      if (st == PKV_OK) tokens[s].insert(tokens[s].end(), more.begin(), more.end());
    } else {
      const size_t i = rng() % live.size();
      CHECK(pkv_pc_free_sequence(pc, live[i]) == PKV_OK);
      tokens.erase(live[i]);
      live.erase(live.begin() + (long)i);
    }
    if (step % 10 == 0) {
      if (!pool_invariants(N, B, live, table, count, nfree)) return false;
      // the free queue lists each free block once
      std::vector<int32_t> q(N);
      int nq = -1;
      CHECK(pkv_pc_free_queue(pc, q.data(), N, &nq) == PKV_OK);
      CHECK(nq == pkv_pc_num_free(pc));
      std::vector<int> seen(N, 0);
      for (int i = 0; i < nq; ++i) {
        CHECK(q[i] >= 0 && q[i] < N);
        if (q[i] >= 0 && q[i] < N) CHECK(++seen[q[i]] == 1);
      }
      // a live sequence's full blocks that are cached carry its chained keys
      for (int64_t s : live) {
        const auto &tk = tokens[s];
        const int full = (int)tk.size() / B;
        std::vector<uint8_t> keys(32 * (size_t)(full + 1));
        CHECK(pkv_pc_chain_keys(tk.data(), (int)tk.size(), B, extra[s], keys.data()) == PKV_OK);
        std::vector<int32_t> t(4096);
        int nb = 0;
        int64_t nt = 0;
        CHECK(pkv_pc_table(pc, s, t.data(), (int)t.size(), &nb, &nt) == PKV_OK);
        CHECK(nt == (int64_t)tk.size());
        for (int i = 0; i < full && i < nb; ++i) {
          uint8_t key[32];
          int cached = 0;
          CHECK(pkv_pc_block_key(pc, t[i], key, &cached) == PKV_OK);
          if (cached) CHECK(memcmp(key, keys.data() + 32 * (size_t)i, 32) == 0);
        }
      }
    }
  }
  for (int64_t s : live) CHECK(pkv_pc_free_sequence(pc, s) == PKV_OK);
  CHECK(pkv_pc_num_free(pc) == N);
  pkv_pc_destroy(pc);
  // digests of every padding length
  std::vector<uint8_t> msg(600);
  for (auto &c : msg) c = (uint8_t)rng();
  uint8_t d[32];
  for (size_t n = 0; n <= msg.size(); ++n) CHECK(pkv_sha256(msg.data(), n, d) == PKV_OK);
  return g_failures == 0;
}

}  // namespace

int main() {
  bool ok = true;
  ok &= stress_block_manager(1, 64, 4);
  ok &= stress_block_manager(2, 200, 16);
  ok &= stress_block_manager(3, 40, 1);
  ok &= stress_prefix_cache(4, 64, 4);
  ok &= stress_prefix_cache(5, 200, 16);
  ok &= stress_prefix_cache(6, 48, 8);
  printf(ok ? "host managers: all checks passed\n" : "host managers: FAILED\n");
  return ok ? 0 : 1;
}
