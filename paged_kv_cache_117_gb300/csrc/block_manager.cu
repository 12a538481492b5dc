// Host-side block manager: on-demand block allocation, reference counts and
// copy-on-write, producing the block tables, slot mapping and copy pairs that
// the GPU calls consume.  No device code.
//
// The rules are the pages':
//  * a sequence takes a new block only when its last block is full
//    ("PagedAttention" (tensortonic), section 3; "PagedAttention and vLLM:
//    Paging the KV Cache Like an OS", Step 3);
//  * free blocks are handed out first in, first out, and a sequence's blocks
//    return to the back of the queue when their count reaches zero
//    ("vLLM's PagedAttention ...", sections 2.4 and 7);
//  * forking copies the block table and raises each block's count (Step 4,
//    beam search);
//  * a writer whose last block has a count above one first copies it to a
//    fresh block and repoints its table; a writer that finds the count at one
//    writes in place (Step 4, parallel sampling).
#include <stdint.h>

#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/paged_kv.h"

struct pkv_block_manager {
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
  };
  int num_blocks = 0;
  int block_size = 0;
  std::deque<int32_t> free_q;
  std::vector<int32_t> refs;
  std::unordered_map<int64_t, Seq> seqs;
};

namespace {

int32_t take_free(pkv_block_manager *bm) {
  const int32_t b = bm->free_q.front();
  bm->free_q.pop_front();
  bm->refs[b] = 1;
  return b;
}

void drop_ref(pkv_block_manager *bm, int32_t b) {
  if (--bm->refs[b] == 0) bm->free_q.push_back(b);
}

}  // namespace

extern "C" {

pkv_block_manager *pkv_bm_create(int num_blocks, int block_size, const int32_t *free_order) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pkv_block_manager *bm = new (std::nothrow) pkv_block_manager;
  if (!bm) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refs.assign((size_t)num_blocks, 0);
  if (free_order) {
    std::vector<char> seen((size_t)num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
      const int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[(size_t)b]) {   // not a permutation
        delete bm;
        return nullptr;
      }
      seen[(size_t)b] = 1;
      bm->free_q.push_back(b);
    }
  } else {
    for (int32_t b = 0; b < num_blocks; ++b) bm->free_q.push_back(b);
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq) {
  if (!bm) return PKV_ERR_NULL;
  if (bm->seqs.count(seq)) return PKV_ERR_RANGE;
  bm->seqs.emplace(seq, pkv_block_manager::Seq{});
  return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child) {
  if (!bm) return PKV_ERR_NULL;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end() || bm->seqs.count(child)) return PKV_ERR_RANGE;
  pkv_block_manager::Seq copy = it->second;
  for (int32_t b : copy.table) ++bm->refs[b];
  bm->seqs.emplace(child, std::move(copy));
  return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq) {
  if (!bm) return PKV_ERR_NULL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ERR_RANGE;
  for (int32_t b : it->second.table) drop_ref(bm, b);
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager *bm, const int64_t *seqs, int n, int64_t *slots,
                         int64_t *pairs, int *num_pairs) {
  if (!bm || !num_pairs) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_RANGE;
  *num_pairs = 0;
  if (n == 0) return PKV_OK;
  if (!seqs || !slots || !pairs) return PKV_ERR_NULL;
  for (int i = 0; i < n; ++i)
    if (!bm->seqs.count(seqs[i])) return PKV_ERR_RANGE;
  const int B = bm->block_size;
  // Dry run: count the blocks this batch takes, so that a batch that does not
  // fit is refused before anything changes.
  {
    struct Tmp {
      int64_t len;
      bool own_last;   // last block taken in this batch (count 1)
    };
    std::unordered_map<int64_t, Tmp> tmp;
    std::unordered_map<int32_t, int32_t> dref;
    long long need = 0;
    for (int i = 0; i < n; ++i) {
      const pkv_block_manager::Seq &s = bm->seqs[seqs[i]];
      auto it = tmp.find(seqs[i]);
      if (it == tmp.end()) it = tmp.emplace(seqs[i], Tmp{s.len, false}).first;
      Tmp &t = it->second;
      if (t.len % B == 0) {
        ++need;
        t.own_last = true;
      } else if (!t.own_last) {
        const int32_t last = s.table.back();
        if (bm->refs[last] + dref[last] > 1) {
          ++need;
          --dref[last];
          t.own_last = true;
        }
      }
      ++t.len;
    }
    if ((long long)bm->free_q.size() < need) return PKV_ERR_NO_BLOCKS;
  }
  for (int i = 0; i < n; ++i) {
    pkv_block_manager::Seq &s = bm->seqs[seqs[i]];
    const int off = (int)(s.len % B);
    if (off == 0) {
      s.table.push_back(take_free(bm));
    } else {
      const int32_t last = s.table.back();
      if (bm->refs[last] > 1) {   // shared partial block: copy before writing
        const int32_t fresh = take_free(bm);
        --bm->refs[last];
        s.table.back() = fresh;
        pairs[2 * *num_pairs + 0] = last;
        pairs[2 * *num_pairs + 1] = fresh;
        ++*num_pairs;
      }
    }
    slots[i] = (int64_t)s.table[(size_t)(s.len / B)] * B + off;
    ++s.len;
  }
  return PKV_OK;
}

pkv_status pkv_bm_table(const pkv_block_manager *bm, int64_t seq, int32_t *out, int capacity,
                        int *num_blocks, int64_t *num_tokens) {
  if (!bm || !num_blocks || !num_tokens) return PKV_ERR_NULL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ERR_RANGE;
  const std::vector<int32_t> &t = it->second.table;
  *num_blocks = (int)t.size();
  *num_tokens = it->second.len;
  if (capacity > 0 && !out) return PKV_ERR_NULL;
  for (int i = 0; i < capacity && i < (int)t.size(); ++i) out[i] = t[(size_t)i];
  return PKV_OK;
}

int pkv_bm_num_free(const pkv_block_manager *bm) { return bm ? (int)bm->free_q.size() : -1; }

int pkv_bm_refcount(const pkv_block_manager *bm, int block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refs[(size_t)block];
}

}  // extern "C"
