// Host-side block manager with a prefix cache: full blocks are keyed by a
// chained SHA-256 and kept in a key -> block map after their request
// finishes, so that a later request with the same prefix takes them over
// instead of recomputing them.  No device code.
//
// The rules are the pages' ("PagedAttention and vLLM: Paging the KV Cache
// Like an OS" ..., section 2.4, "V1's block pool and hash chain", and summary
// point 5):
//  * one free queue ordered by recency of release: released blocks go to the
//    back, allocation takes the front, and a block taken from the front that
//    still holds cached content leaves the map first -- the queue order is the
//    eviction order;
//  * a block's key is SHA-256(previous block's key, its tokens, an extra key);
//    only full blocks are keyed and cached;
//  * a new request walks its prompt's chain block by block, each hit raising
//    the block's count (taking it out of the free queue if it was there), and
//    stops at the first miss; the last prompt token is always recomputed, so
//    hits only cover blocks inside the first prompt_len - 1 tokens;
//  * cached blocks are full and never written again, so no copy-on-write.
// Readings where the pages are silent: the hashed message is the parent's 32
// bytes, each token as 4 little-endian bytes, then the extra key as 8
// little-endian bytes; the first block's parent is 32 zero bytes; a finished
// request's blocks enter the free queue last block first; a block that fills
// with content already cached stays uncached.
#include <stdint.h>
#include <string.h>

#include <array>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/paged_kv.h"

namespace {

// ---- SHA-256 (FIPS 180-4) ---------------------------------------------------------
// Round constants: the first 32 bits of the fractional parts of the cube roots
// of the first 64 primes; initial value: the same of the square roots of the
// first 8 primes.
const uint32_t K256[64] = {
    0x428a2f98u, 0x71374491u, 0xb5c0fbcfu, 0xe9b5dba5u, 0x3956c25bu, 0x59f111f1u, 0x923f82a4u,
    0xab1c5ed5u, 0xd807aa98u, 0x12835b01u, 0x243185beu, 0x550c7dc3u, 0x72be5d74u, 0x80deb1feu,
    0x9bdc06a7u, 0xc19bf174u, 0xe49b69c1u, 0xefbe4786u, 0x0fc19dc6u, 0x240ca1ccu, 0x2de92c6fu,
    0x4a7484aau, 0x5cb0a9dcu, 0x76f988dau, 0x983e5152u, 0xa831c66du, 0xb00327c8u, 0xbf597fc7u,
    0xc6e00bf3u, 0xd5a79147u, 0x06ca6351u, 0x14292967u, 0x27b70a85u, 0x2e1b2138u, 0x4d2c6dfcu,
    0x53380d13u, 0x650a7354u, 0x766a0abbu, 0x81c2c92eu, 0x92722c85u, 0xa2bfe8a1u, 0xa81a664bu,
    0xc24b8b70u, 0xc76c51a3u, 0xd192e819u, 0xd6990624u, 0xf40e3585u, 0x106aa070u, 0x19a4c116u,
    0x1e376c08u, 0x2748774cu, 0x34b0bcb5u, 0x391c0cb3u, 0x4ed8aa4au, 0x5b9cca4fu, 0x682e6ff3u,
    0x748f82eeu, 0x78a5636fu, 0x84c87814u, 0x8cc70208u, 0x90befffau, 0xa4506cebu, 0xbef9a3f7u,
    0xc67178f2u};
const uint32_t H256[8] = {0x6a09e667u, 0xbb67ae85u, 0x3c6ef372u, 0xa54ff53au,
                          0x510e527fu, 0x9b05688cu, 0x1f83d9abu, 0x5be0cd19u};

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void sha256_block(uint32_t h[8], const uint8_t *p) {
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = (uint32_t)p[4 * t] << 24 | (uint32_t)p[4 * t + 1] << 16 | (uint32_t)p[4 * t + 2] << 8 |
           (uint32_t)p[4 * t + 3];
  for (int t = 16; t < 64; ++t) {
    const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
    const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
    w[t] = w[t - 16] + s0 + w[t - 7] + s1;
  }
  uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], k = h[7];
  for (int t = 0; t < 64; ++t) {
    const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t t1 = k + S1 + ch + K256[t] + w[t];
    const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    const uint32_t mj = (a & b) ^ (a & c) ^ (b & c);
    const uint32_t t2 = S0 + mj;
    k = g;
    g = f;
    f = e;
    e = d + t1;
    d = c;
    c = b;
    b = a;
    a = t1 + t2;
  }
  h[0] += a;
  h[1] += b;
  h[2] += c;
  h[3] += d;
  h[4] += e;
  h[5] += f;
  h[6] += g;
  h[7] += k;
}

// Digest of msg[0..n) into out[32].
void sha256(const uint8_t *msg, size_t n, uint8_t out[32]) {
  uint32_t h[8];
  memcpy(h, H256, sizeof(h));
  size_t i = 0;
  for (; i + 64 <= n; i += 64) sha256_block(h, msg + i);
  uint8_t last[128] = {0};
  const size_t rem = n - i;
  memcpy(last, msg + i, rem);
  last[rem] = 0x80;
  const size_t tot = rem + 9 <= 64 ? 64 : 128;
  const uint64_t bits = (uint64_t)n * 8u;
  for (int j = 0; j < 8; ++j) last[tot - 1 - j] = (uint8_t)(bits >> (8 * j));
  sha256_block(h, last);
  if (tot == 128) sha256_block(h, last + 64);
  for (int j = 0; j < 8; ++j) {
    out[4 * j] = (uint8_t)(h[j] >> 24);
    out[4 * j + 1] = (uint8_t)(h[j] >> 16);
    out[4 * j + 2] = (uint8_t)(h[j] >> 8);
    out[4 * j + 3] = (uint8_t)h[j];
  }
}

using Key = std::array<uint8_t, 32>;

struct KeyHash {
  size_t operator()(const Key &k) const {
    size_t v;
    memcpy(&v, k.data(), sizeof(v));
    return v;
  }
};

// Chained key of one full block (message layout: see the file comment).
Key block_key(const Key &parent, const int32_t *tokens, int n, uint64_t extra) {
  std::vector<uint8_t> msg(32 + 4 * (size_t)n + 8);
  memcpy(msg.data(), parent.data(), 32);
  for (int i = 0; i < n; ++i) {
    const uint32_t t = (uint32_t)tokens[i];
    for (int j = 0; j < 4; ++j) msg[32 + 4 * (size_t)i + j] = (uint8_t)(t >> (8 * j));
  }
  for (int j = 0; j < 8; ++j) msg[32 + 4 * (size_t)n + j] = (uint8_t)(extra >> (8 * j));
  Key k;
  sha256(msg.data(), msg.size(), k.data());
  return k;
}

const Key ROOT_KEY = {};

}  // namespace

struct pkv_prefix_cache {
  struct Seq {
    uint64_t extra = 0;
    std::vector<int32_t> table;
    std::vector<Key> keys;          // keys of the full blocks, in order
    std::vector<int32_t> tail;      // tokens of the partly filled last block
    int64_t len = 0;
  };
  int num_blocks = 0;
  int block_size = 0;
  // free queue: a doubly linked list through prev/next, front = head
  std::vector<int32_t> prev, next;
  std::vector<char> in_free;
  int32_t head = -1, tail = -1;
  int num_free = 0;
  std::vector<int32_t> refs;
  std::vector<char> keyed;          // block holds a cached key
  std::vector<Key> key;
  std::unordered_map<Key, int32_t, KeyHash> cache;
  std::unordered_map<int64_t, Seq> seqs;

  void push_back(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b;
    else head = b;
    tail = b;
    in_free[b] = 1;
    ++num_free;
  }
  void unlink(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b];
    else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b];
    else tail = prev[b];
    prev[b] = next[b] = -1;
    in_free[b] = 0;
    --num_free;
  }
  // Front of the queue, its cached content evicted first.
  int32_t allocate() {
    const int32_t b = head;
    unlink(b);
    if (keyed[b]) {
      auto it = cache.find(key[b]);
      if (it != cache.end() && it->second == b) cache.erase(it);
      keyed[b] = 0;
    }
    refs[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--refs[b] == 0) push_back(b);
  }
};

extern "C" {

pkv_prefix_cache *pkv_pc_create(int num_blocks, int block_size, const int32_t *free_order) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pkv_prefix_cache *pc = new (std::nothrow) pkv_prefix_cache;
  if (!pc) return nullptr;
  pc->num_blocks = num_blocks;
  pc->block_size = block_size;
  pc->prev.assign((size_t)num_blocks, -1);
  pc->next.assign((size_t)num_blocks, -1);
  pc->in_free.assign((size_t)num_blocks, 0);
  pc->refs.assign((size_t)num_blocks, 0);
  pc->keyed.assign((size_t)num_blocks, 0);
  pc->key.resize((size_t)num_blocks);
  for (int i = 0; i < num_blocks; ++i) {
    const int32_t b = free_order ? free_order[i] : i;
    if (b < 0 || b >= num_blocks || pc->in_free[(size_t)b]) {   // not a permutation
      delete pc;
      return nullptr;
    }
    pc->push_back(b);
  }
  return pc;
}

void pkv_pc_destroy(pkv_prefix_cache *pc) { delete pc; }

pkv_status pkv_pc_add_sequence(pkv_prefix_cache *pc, int64_t seq, const int32_t *prompt,
                               int prompt_len, uint64_t extra_key, int *num_cached_tokens) {
  if (!pc || !num_cached_tokens) return PKV_ERR_NULL;
  if (prompt_len < 0 || pc->seqs.count(seq)) return PKV_ERR_RANGE;
  if (prompt_len > 0 && !prompt) return PKV_ERR_NULL;
  pkv_prefix_cache::Seq s;
  s.extra = extra_key;
  const int B = pc->block_size;
  const int usable = prompt_len > 0 ? (prompt_len - 1) / B : 0;   // last token recomputed
  Key parent = ROOT_KEY;
  for (int i = 0; i < usable; ++i) {
    const Key k = block_key(parent, prompt + (size_t)i * B, B, extra_key);
    auto it = pc->cache.find(k);
    if (it == pc->cache.end()) break;
    const int32_t b = it->second;
    if (pc->refs[b] == 0) pc->unlink(b);
    ++pc->refs[b];
    s.table.push_back(b);
    s.keys.push_back(k);
    parent = k;
  }
  s.len = (int64_t)s.table.size() * B;
  *num_cached_tokens = (int)s.len;
  pc->seqs.emplace(seq, std::move(s));
  return PKV_OK;
}

pkv_status pkv_pc_append(pkv_prefix_cache *pc, int64_t seq, const int32_t *tokens, int n,
                         int64_t *slots) {
  if (!pc) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_RANGE;
  auto it = pc->seqs.find(seq);
  if (it == pc->seqs.end()) return PKV_ERR_RANGE;
  if (n == 0) return PKV_OK;
  if (!tokens || !slots) return PKV_ERR_NULL;
  pkv_prefix_cache::Seq &s = it->second;
  const int B = pc->block_size;
  long long need = 0;   // blocks this call takes: refused up front if they are not free
  for (int i = 0; i < n; ++i)
    if ((s.len + i) % B == 0) ++need;
  if (need > pc->num_free) return PKV_ERR_NO_BLOCKS;
  for (int i = 0; i < n; ++i) {
    const int off = (int)(s.len % B);
    if (off == 0) s.table.push_back(pc->allocate());
    const int32_t blk = s.table.back();
    slots[i] = (int64_t)blk * B + off;
    s.tail.push_back(tokens[i]);
    ++s.len;
    if ((int)s.tail.size() == B) {
      const Key k = block_key(s.keys.empty() ? ROOT_KEY : s.keys.back(), s.tail.data(), B, s.extra);
      s.keys.push_back(k);
      s.tail.clear();
      if (!pc->cache.count(k)) {
        pc->cache.emplace(k, blk);
        pc->key[(size_t)blk] = k;
        pc->keyed[(size_t)blk] = 1;
      }
    }
  }
  return PKV_OK;
}

pkv_status pkv_pc_free_sequence(pkv_prefix_cache *pc, int64_t seq) {
  if (!pc) return PKV_ERR_NULL;
  auto it = pc->seqs.find(seq);
  if (it == pc->seqs.end()) return PKV_ERR_RANGE;
  const std::vector<int32_t> &t = it->second.table;
  for (size_t i = t.size(); i-- > 0;) pc->release(t[i]);   // last block first
  pc->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_pc_table(const pkv_prefix_cache *pc, int64_t seq, int32_t *out, int capacity,
                        int *num_blocks, int64_t *num_tokens) {
  if (!pc || !num_blocks || !num_tokens) return PKV_ERR_NULL;
  auto it = pc->seqs.find(seq);
  if (it == pc->seqs.end()) return PKV_ERR_RANGE;
  const std::vector<int32_t> &t = it->second.table;
  *num_blocks = (int)t.size();
  *num_tokens = it->second.len;
  if (capacity > 0 && !out) return PKV_ERR_NULL;
  for (int i = 0; i < capacity && i < (int)t.size(); ++i) out[i] = t[(size_t)i];
  return PKV_OK;
}

int pkv_pc_num_free(const pkv_prefix_cache *pc) { return pc ? pc->num_free : -1; }

int pkv_pc_num_cached(const pkv_prefix_cache *pc) { return pc ? (int)pc->cache.size() : -1; }

int pkv_pc_refcount(const pkv_prefix_cache *pc, int block) {
  if (!pc || block < 0 || block >= pc->num_blocks) return -1;
  return pc->refs[(size_t)block];
}

pkv_status pkv_pc_block_key(const pkv_prefix_cache *pc, int block, uint8_t *key32, int *cached) {
  if (!pc || !key32 || !cached) return PKV_ERR_NULL;
  if (block < 0 || block >= pc->num_blocks) return PKV_ERR_RANGE;
  *cached = pc->keyed[(size_t)block] ? 1 : 0;
  if (*cached) memcpy(key32, pc->key[(size_t)block].data(), 32);
  return PKV_OK;
}

pkv_status pkv_pc_free_queue(const pkv_prefix_cache *pc, int32_t *out, int capacity, int *count) {
  if (!pc || !count) return PKV_ERR_NULL;
  *count = pc->num_free;
  if (capacity > 0 && !out) return PKV_ERR_NULL;
  int i = 0;
  for (int32_t b = pc->head; b >= 0 && i < capacity; b = pc->next[(size_t)b]) out[i++] = b;
  return PKV_OK;
}

pkv_status pkv_pc_chain_keys(const int32_t *tokens, int num_tokens, int block_size,
                             uint64_t extra_key, uint8_t *keys_out) {
  if (num_tokens < 0 || block_size <= 0) return PKV_ERR_RANGE;
  const int nb = num_tokens / block_size;
  if (nb == 0) return PKV_OK;
  if (!tokens || !keys_out) return PKV_ERR_NULL;
  Key parent = ROOT_KEY;
  for (int i = 0; i < nb; ++i) {
    parent = block_key(parent, tokens + (size_t)i * block_size, block_size, extra_key);
    memcpy(keys_out + 32 * (size_t)i, parent.data(), 32);
  }
  return PKV_OK;
}

pkv_status pkv_sha256(const void *msg, size_t len, uint8_t *digest32) {
  if (!digest32 || (len > 0 && !msg)) return PKV_ERR_NULL;
  sha256(static_cast<const uint8_t *>(msg), len, digest32);
  return PKV_OK;
}

}  // extern "C"
