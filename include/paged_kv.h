/*
 * paged_kv.h -- C ABI of the GB300 (sm_103a) paged KV cache decode library.
 *
 * The library implements the data-parallel hot path of PagedAttention: the
 * KV cache lives in one pool of fixed-size blocks, and every sequence reaches
 * its tokens through its own block table.  Three operations keep that pool
 * live and read it:
 *
 *   paged_kv_write          store this step's new keys/values into the slots
 *                           the block manager assigned ("reshape and cache")
 *   paged_block_copy        the batched copy-on-write block copy
 *   paged_attention_decode  single-query attention over the paged context
 *   paged_attention_decode_append
 *                           the step's KV write and decode attention in one
 *                           call
 *   paged_attention_chunked multi-query attention over the paged context:
 *                           chunked prefill and decode in one batch
 *
 * Sources for what each call computes: "PagedAttention and vLLM: Paging the
 * KV Cache Like an OS" (vidyal.ai), Step 5, the three kernels (write, read and
 * attend, copy) and Step 4 (reference counts and copy-on-write);
 * "PagedAttention" (tensortonic.com), section 5 (write before attending,
 * softmax over all valid positions, the table [3, 0, 6]);
 * "PagedAttention: Virtual Memory for the KV Cache" (alexdo.xyz), the
 * block-wise attention equation.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers, owned by the caller, dense
 *    (row-major, no padding) and 16-byte aligned.  The library allocates no
 *    memory: scratch for the attention pass is passed in (see
 *    paged_attention_workspace_bytes).
 *  - Pool layout: k_cache and v_cache are [num_blocks, block_size,
 *    num_kv_heads, head_dim] of the cache dtype.  Slot s of the pool is
 *    (block s / block_size, offset s % block_size).
 *  - Supported shapes: head_dim in {64, 128}; block_size in {4, 8, 16, 32};
 *    cache dtype PKV_F16 or PKV_BF16; num_q_heads a multiple of num_kv_heads.
 *  - Query head hq reads KV head hq / (num_q_heads / num_kv_heads).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are found on the host before anything
 *    is launched and returned as a status; nothing is launched then.  A
 *    launch failure returns PKV_ERR_CUDA.  Calls never abort the process.
 *  - Device-side values (block ids, slots, lengths, copy pairs) are checked
 *    inside the kernels: an out-of-range value is never dereferenced; the
 *    access is skipped (or the length clamped), and a bit is set in the
 *    library's device flag word, read back with pkv_read_device_flags.
 *  - Results of calls that overlap in time on the same buffers are undefined;
 *    order them on one stream: block copy, then write, then attend.
 */
#ifndef PAGED_KV_H
#define PAGED_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pkv_stream_t; /* same type as cudaStream_t */

typedef enum {
  PKV_OK = 0,
  PKV_ERR_NULL = 1,      /* a required pointer is NULL */
  PKV_ERR_SHAPE = 2,     /* unsupported or inconsistent sizes */
  PKV_ERR_DTYPE = 3,     /* unsupported dtype */
  PKV_ERR_RANGE = 4,     /* a size is negative or too large */
  PKV_ERR_ALIAS = 5,     /* buffers that must be distinct overlap */
  PKV_ERR_CUDA = 6,      /* a CUDA runtime / driver call failed */
  PKV_ERR_WORKSPACE = 7, /* workspace missing or too small */
  PKV_ERR_ALIGN = 8,     /* a pointer is not aligned as required */
  PKV_ERR_NO_BLOCKS = 9  /* the block manager has too few free blocks */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 } pkv_dtype;

/* Bits of the device flag word. */
#define PKV_FLAG_BLOCK_RANGE 0x1u /* a block table entry was outside [0, num_blocks) */
#define PKV_FLAG_SLOT_RANGE 0x2u  /* a slot was >= num_blocks * block_size */
#define PKV_FLAG_PAIR_RANGE 0x4u  /* a copy pair named a block outside the pool */
#define PKV_FLAG_LEN_RANGE 0x8u   /* a context length was < 0 or > max_blocks * block_size */
#define PKV_FLAG_TIMEOUT 0x10u    /* a kernel gave up waiting on its own tile loads */
#define PKV_FLAG_V_RANGE 0x20u    /* PKV_P_F16 met a bf16 V value beyond the f16 range (clamped) */
#define PKV_FLAG_PAIR_CONFLICT 0x40u /* a copy pair's dst was another pair's dst or src (skipped) */

/*
 * paged_kv_write -- store new keys/values into their slots.
 *
 * Each new token's key and value rows are stored at the block and offset
 * that its slot names ("PagedAttention", section 5); one launch writes the
 * rows of every token of the step ("PagedAttention and vLLM ...", Step 5,
 * "Write").
 *
 *   key, value    [num_tokens, num_kv_heads, head_dim], cache dtype
 *   k_cache,
 *   v_cache       [num_blocks, block_size, num_kv_heads, head_dim]
 *   slot_mapping  int64 [num_tokens]; token t goes to slot slot_mapping[t]
 *                 (= block * block_size + offset).  A negative slot skips the
 *                 token.  A slot >= num_blocks * block_size is skipped and
 *                 flagged (PKV_FLAG_SLOT_RANGE).
 *
 * The copy is bit-exact.  Two tokens naming one slot race (one of them wins).
 * num_tokens == 0 is a no-op that launches nothing.
 */
pkv_status paged_kv_write(const void *key, const void *value, void *k_cache,
                          void *v_cache, const int64_t *slot_mapping,
                          int num_tokens, int num_blocks, int block_size,
                          int num_kv_heads, int head_dim, pkv_dtype dtype,
                          pkv_stream_t stream);

/*
 * paged_block_copy -- batched copy-on-write block copy.
 *
 * A step's copy-on-write may ask for many small block copies; they all run in
 * a single launch ("PagedAttention and vLLM ...", Step 5, "Copy").  For
 * every pair, all block_size slots of block src are copied to block dst, in
 * k_cache and in v_cache, bit-exactly, in one launch.
 *
 *   block_pairs  int64 [num_pairs][2] = (src, dst), DEVICE memory.
 *
 * Preconditions (the block manager's invariants): every dst appears once and
 * no dst is also a src in the same call.  The pairs live on the device, so
 * the kernel checks them: a pair naming a block outside [0, num_blocks) is
 * skipped and flagged (PKV_FLAG_PAIR_RANGE) and copies nothing; a pair whose
 * dst is another in-pool pair's dst or src is skipped and flagged
 * (PKV_FLAG_PAIR_CONFLICT) -- the copies of one call run in no particular
 * order.  A pair that copies a block onto itself conflicts only through other
 * pairs.  num_pairs == 0 is a no-op.
 *
 * Cost of the check: each CTA compares its pair with every other pair
 * (O(num_pairs) reads per CTA, from L2), which is nothing for the few copies
 * of a decode step.  For long pair lists (beam search forking many beams,
 * a scheduler moving many requests at once) use paged_block_copy_ws, whose
 * check costs O(1) per CTA.
 */
pkv_status paged_block_copy(void *k_cache, void *v_cache,
                            const int64_t *block_pairs, int num_pairs,
                            int num_blocks, int block_size, int num_kv_heads,
                            int head_dim, pkv_dtype dtype, pkv_stream_t stream);

/*
 * paged_block_copy_ws -- paged_block_copy with the pair check done through a
 * caller-owned counter workspace, so that its cost does not grow with the
 * number of pairs.  Same copies, same skips and flags, same results.
 *
 *   workspace        DEVICE memory of at least
 *                    paged_block_copy_workspace_bytes(num_blocks) bytes
 *                    (two uint32 counters per pool block), 256-byte aligned.
 *                    It must be all zero before the first call; every call
 *                    leaves it all zero again when its work on the stream is
 *                    done, so allocate it zeroed once and reuse it.  Calls
 *                    that share one workspace must not overlap in time
 *                    (issue them on one stream).
 *
 * Three kernels run in stream order: a counting pass (per pair, one atomic
 * increment of cnt_dst[dst] and of cnt_src[src]), the copy (a pair is
 * skipped and flagged when cnt_dst[dst] > 1, or when cnt_src[dst] counts a
 * src other than the pair's own), and a reset pass that zeroes the counters
 * the counting pass raised.  A null workspace returns PKV_ERR_WORKSPACE;
 * other errors as paged_block_copy.
 */
size_t paged_block_copy_workspace_bytes(int num_blocks);
pkv_status paged_block_copy_ws(void *k_cache, void *v_cache,
                               const int64_t *block_pairs, int num_pairs,
                               int num_blocks, int block_size, int num_kv_heads,
                               int head_dim, pkv_dtype dtype, void *workspace,
                               size_t workspace_bytes, pkv_stream_t stream);

/*
 * paged_attention_decode -- single-query attention over the paged context.
 *
 * For sequence s and query head hq (KV head h = hq / G):
 *   out[s, hq, :] = sum_t softmax_t(scale * q[s, hq, :] . K_t) V_t
 * over the L_s = context_lens[s] tokens of the sequence, token t read from
 * physical block block_tables[s, t / block_size], offset t % block_size
 * ("PagedAttention and vLLM ...", Step 5; "PagedAttention", sections 4-5).
 * The softmax is over all L_s positions at once; slots of the last block at
 * or past L_s are never read.  L_s counts this step's token, which must
 * already be written (paged_kv_write earlier on the same stream).  L_s == 0
 * gives zeros.
 *
 *   out            [num_seqs, num_q_heads, head_dim] of out_dtype (F32, F16
 *                  or BF16; arithmetic is fp32 regardless)
 *   q              [num_seqs, num_q_heads, head_dim], cache dtype
 *   block_tables   int32 [num_seqs, max_blocks]; entries past a sequence's
 *                  last block are ignored
 *   context_lens   int32 [num_seqs]; a length outside [0, max_blocks *
 *                  block_size] is clamped and flagged (PKV_FLAG_LEN_RANGE)
 *   scale          softmax scale, normally 1/sqrt(head_dim)
 *   partition_tokens
 *                  0: one partition per sequence.  Otherwise a multiple of
 *                  block_size: each sequence's context is cut into partitions
 *                  of this many tokens, processed in parallel; the CTA that
 *                  finishes a sequence's last partition merges the partition
 *                  results, rescaling each by its running max (log-sum-exp
 *                  merge, unnormalised records).
 *   workspace      device scratch, 256-byte aligned, of at least
 *                  paged_attention_workspace_bytes(num_seqs, num_q_heads,
 *                  head_dim, max_blocks * block_size, partition_tokens)
 *                  bytes.  Contents on entry do not matter; the call leaves
 *                  its work list and partition records there.  Two calls
 *                  that share a workspace must not overlap in time.
 *
 * Two launches: a one-CTA pass that lists the (sequence, partition) work
 * items in the workspace, then the persistent attention pass.
 */
pkv_status paged_attention_decode(
    void *out, pkv_dtype out_dtype, const void *q, const void *k_cache,
    const void *v_cache, pkv_dtype dtype, const int32_t *block_tables,
    int max_blocks, const int32_t *context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, float scale, int partition_tokens, void *workspace,
    size_t workspace_bytes, pkv_stream_t stream);

/*
 * paged_attention_decode_append -- the decode step's KV write and decode
 * attention in one call.
 *
 * Computes what paged_kv_write followed by paged_attention_decode computes
 * when this step's token of sequence s (L_s = context_lens[s] >= 1 counting
 * it) goes to position L_s - 1, i.e. to slot block_tables[s, (L_s - 1) /
 * block_size] * block_size + (L_s - 1) % block_size ("PagedAttention",
 * section 5: the new key and value are written first, then the query attends
 * over every valid position including its own).  key and value hold the
 * step's rows, [num_seqs, num_kv_heads, head_dim] of the cache dtype,
 * 16-byte aligned, overlapping neither pool, out nor the workspace.  The
 * attention takes position L_s - 1 from these rows directly and the call
 * stores them into both pools, so the pools afterwards hold exactly what
 * paged_kv_write would have left.  Sequences with L_s == 0 append nothing
 * (zeros out); a length past the table is clamped and flagged
 * (PKV_FLAG_LEN_RANGE) and appends nothing; a bad block id for the slot is
 * flagged (PKV_FLAG_BLOCK_RANGE) and nothing is stored.  The slot's block
 * must belong to sequence s alone during the call (copy-on-write done
 * before, as the block manager guarantees): another sequence reading it in
 * the same call would see either the old or the new row.  Every other
 * argument, the workspace and the launches are those of
 * paged_attention_decode.
 */
pkv_status paged_attention_decode_append(
    void *out, pkv_dtype out_dtype, const void *q, const void *key,
    const void *value, void *k_cache, void *v_cache, pkv_dtype dtype,
    const int32_t *block_tables, int max_blocks, const int32_t *context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, int partition_tokens,
    void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* How P (the softmax weights) enters the P.V product of
 * paged_attention_chunked; scores, the softmax and accumulation are fp32
 * either way. */
typedef enum {
  PKV_P_HILO = 0, /* P = hi + lo, two 16-bit MMA operands of the cache dtype:
                     about 16 significant bits (errors ~1e-5) */
  PKV_P_F16 = 1   /* P as one f16 operand (11 significant bits) and V as f16
                     (a bf16 V tile is converted in shared memory; values
                     beyond +-65504 are clamped and flagged
                     PKV_FLAG_V_RANGE); half the P.V tensor work; each
                     output row is an exact convex combination of the f16
                     values with the rounded weights, error per element below
                     2^-11 * max|V - out| */
} pkv_p_format;

/*
 * paged_attention_chunked -- multi-query attention over the paged context:
 * chunks of prompts (chunked prefill) and decode tokens in one batch.
 *
 * "Paging the KV Cache Like an OS" (continuous batching; chunked prefill): a
 * prompt is prefilled a piece at a time over several steps, each piece
 * filling blocks taken on demand, alongside other sequences' decode tokens.  Sequence s contributes the n_s = query_start[s+1]
 * - query_start[s] query rows q[query_start[s] .. query_start[s+1]-1], its
 * LAST n_s positions: with L_s = context_lens[s] (which counts them), row i
 * sits at position p = L_s - n_s + i and attends to positions 0..p of its own
 * sequence (causal attention; a decode token is the case n_s = 1):
 *   out[row, hq, :] = sum_{t <= p} softmax_t(scale * q[row, hq, :] . K_t) V_t
 * The chunk's keys and values must already be in the pool (paged_kv_write of
 * its n_s tokens earlier on the same stream).
 *
 *   out            [num_tokens, num_q_heads, head_dim] of out_dtype (F32, F16
 *                  or BF16), 16-byte aligned
 *   q              [num_tokens, num_q_heads, head_dim], cache dtype
 *   block_tables   int32 [num_seqs, max_blocks]
 *   context_lens   int32 [num_seqs]; L_s >= n_s
 *   query_start    int32 [num_seqs + 1], non-decreasing, query_start[0] = 0,
 *                  query_start[num_seqs] = num_tokens
 *   max_query_len  an upper bound of every n_s (sizes the launch)
 *   p_format       PKV_P_HILO or PKV_P_F16 (see pkv_p_format)
 *
 * Extra shape limits: num_q_heads / num_kv_heads <= 128; block_size 8, 16 or
 * 32 (the tiles are staged in 128-byte-swizzled shared memory whose 1 KiB
 * atoms a 4-token block cannot fill).  Accuracy: scores
 * and the online softmax in fp32; P enters P.V as a 16-bit hi + lo pair.
 * Device-side checks: a sequence whose query_start entries are out of order
 * or past num_tokens, whose n_s exceeds max_query_len, or whose L_s < n_s is
 * skipped (its rows are left untouched) and flagged PKV_FLAG_LEN_RANGE; L_s
 * past the table is clamped and flagged; bad block ids are read as zeros and
 * flagged PKV_FLAG_BLOCK_RANGE.  No workspace: one launch, one CTA per
 * (two query tiles of 128 / G tokens each, sequence, KV head); with up to
 * 2,048 sequences of which some have fewer query tiles than the longest, the
 * grid holds only the units that exist, which query ranges that overlap
 * (against the non-decreasing rule above) can exceed: then some units are not
 * run and PKV_FLAG_LEN_RANGE is set.  Up to 64 sequences launch longest
 * context first (the order changes no result).
 */
pkv_status paged_attention_chunked(
    void *out, pkv_dtype out_dtype, const void *q, const void *k_cache,
    const void *v_cache, pkv_dtype dtype, const int32_t *block_tables,
    int max_blocks, const int32_t *context_lens, const int32_t *query_start,
    int num_seqs, int num_tokens, int max_query_len, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int num_blocks,
    float scale, pkv_p_format p_format, pkv_stream_t stream);

/*
 * paged_attention_mixed -- paged_attention_chunked for a batch that mixes
 * decode tokens with prompt chunks, as continuous batching builds one step
 * ("Paging the KV Cache Like an OS", continuous batching: a step takes all
 * sequences that are decoding first and spends what is left of its token
 * budget on pieces of prompts).
 *
 * Same arguments, layouts and result as paged_attention_chunked, plus the
 * decode attention's partition size and workspace.  A sequence with exactly
 * one query row (n_s = 1: a decode token) goes to the decode kernel (the one
 * paged_attention_decode runs: the block table walked in partitions, each
 * K/V block read once for the whole query group, CUDA cores and warp-level
 * MMAs), its query and output rows found through query_start; the sequences
 * with more rows go to the tensor-core kernel of paged_attention_chunked,
 * which skips the single-row ones.  In one chunked launch a decode row fills
 * 1 of the 128 rows of its MMA tile; here it costs what a decode step costs.
 *
 *   partition_tokens  as paged_attention_decode (multiple of block_size;
 *                     0 = one partition per sequence)
 *   workspace         DEVICE memory of at least
 *                     paged_attention_workspace_bytes(num_seqs, num_q_heads,
 *                     head_dim, max_blocks * block_size, partition_tokens)
 *                     bytes, 256-byte aligned, no initial contents needed;
 *                     calls that share one must not overlap in time.
 *
 * Two or three kernels (the decode work list, the decode pass, then the
 * chunked pass when max_query_len > 1); they write disjoint rows of out.
 * With max_query_len > 1 and at most 8 query heads per KV head the two
 * passes run at the same time on disjoint SMs: the work list gives the
 * decode pass the share of the SMs that a model of the two passes (its K/V
 * bytes against the chunks' query-key pairs) says balances them, and the
 * chunked pass starts on the rest at once.  The call still behaves as stream
 * ordered: the chunked grid ends only after the decode grid, so work queued
 * behind the call on `stream` sees out complete.  (The workspace's first
 * bytes carry the split and a finished-CTA count for this.)  Every argument
 * is checked before the first launch; errors as paged_attention_chunked and
 * paged_attention_decode.  A single-row sequence
 * whose row lies outside [0, num_tokens) or whose context length is below 1
 * is skipped and flagged (PKV_FLAG_LEN_RANGE).
 */
pkv_status paged_attention_mixed(
    void *out, pkv_dtype out_dtype, const void *q, const void *k_cache,
    const void *v_cache, pkv_dtype dtype, const int32_t *block_tables,
    int max_blocks, const int32_t *context_lens, const int32_t *query_start,
    int num_seqs, int num_tokens, int max_query_len, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int num_blocks,
    float scale, pkv_p_format p_format, int partition_tokens, void *workspace,
    size_t workspace_bytes, pkv_stream_t stream);

/*
 * Scratch bytes paged_attention_decode needs, with
 * P = ceil(max_context / partition_tokens) (P = 1 when partition_tokens is 0)
 * and max_context the capacity of one block-table row (max_blocks *
 * block_size), each part rounded up to 256 bytes:
 *   256 (control words) + 4 * num_seqs * num_q_heads (completion counters)
 *   + 8 * num_seqs * P (work list)
 *   + when P > 1: 4 * num_seqs * num_q_heads * P * (head_dim + 2)
 *     (one fp32 (max, sum, unnormalised output) record per sequence, query
 *     head and partition).
 * Returns (size_t)-1 on invalid arguments.
 */
size_t paged_attention_workspace_bytes(int num_seqs, int num_q_heads,
                                       int head_dim, int max_context,
                                       int partition_tokens);

/*
 * paged_attention_decode_noalloc -- paged_attention_decode without a
 * caller-provided workspace.  (The pages describe no such call: it exists for
 * callers of this library that cannot allocate device memory.)
 *
 * Some callers cannot hand the library a scratch buffer: a host program
 * whose device memory belongs to another memory manager that gives out no
 * extra buffers, a plugin inside a host process with a fixed memory budget
 * reserved up front, or a latency-critical loop that must not call cudaMalloc
 * (it can synchronise the device).  This entry point computes exactly what
 * paged_attention_decode computes, with the same arguments minus `workspace`
 * and `workspace_bytes`; its scratch is a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES that is part of the library's device image, held
 * on every GPU that loads the library until the process exits.  Nothing is
 * allocated by the call.
 *
 *  - Limit: a request whose paged_attention_workspace_bytes(num_seqs,
 *    num_q_heads, head_dim, max_blocks * block_size, partition_tokens)
 *    exceeds PKV_NOALLOC_SCRATCH_BYTES returns PKV_ERR_WORKSPACE before any
 *    CUDA call.
 *  - Set-up: the first call on a device (with that device current) looks up
 *    the array's device address once and keeps it for the life of the
 *    process; make that first call before any stream capture.  The kept
 *    address is not refreshed: after cudaDeviceReset on a device this entry
 *    point must not be called on that device again in the same process (the
 *    module may be reloaded elsewhere and the kept address would be stale).
 *  - Sharing: every call on a device uses the same array, which keeps the
 *    last call's contents (the call resets what must start at zero).  Calls
 *    that overlap in time on one device race; order them on one stream.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (64u << 20)
pkv_status paged_attention_decode_noalloc(
    void *out, pkv_dtype out_dtype, const void *q, const void *k_cache,
    const void *v_cache, pkv_dtype dtype, const int32_t *block_tables,
    int max_blocks, const int32_t *context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, float scale, int partition_tokens, pkv_stream_t stream);

/*
 * Host-side block manager (no device memory involved): on-demand block
 * allocation, reference counts and copy-on-write, producing the block tables,
 * slot mapping and copy pairs that the calls above consume.
 *
 * The rules follow the pages: a sequence takes a new block only when its last
 * one is full ("PagedAttention" (tensortonic), section 3; "PagedAttention and
 * vLLM ...", Step 3); free blocks are handed out first in, first out and come
 * back when their count reaches zero ("vLLM's PagedAttention ...", sections
 * 2.4 and 7); forking copies the block table and raises the counts; a writer
 * whose last block is shared (count > 1) copies it to a fresh block first,
 * while a writer that finds the count at one writes in place ("PagedAttention
 * and vLLM ...", Step 4).  Not thread-safe: one manager, one thread at a time.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager of num_blocks blocks of block_size tokens.  free_order (may be
 * NULL = ascending) is the order in which free blocks are first handed out; it
 * must be a permutation of 0..num_blocks-1.  Returns NULL on invalid
 * arguments or allocation failure.  Release with pkv_bm_destroy. */
pkv_block_manager *pkv_bm_create(int num_blocks, int block_size,
                                 const int32_t *free_order);
void pkv_bm_destroy(pkv_block_manager *bm);

/* New empty sequence (PKV_ERR_RANGE if the id exists). */
pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq);
/* child shares every block of parent (PKV_ERR_RANGE: unknown parent or
 * existing child). */
pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child);
/* Drops the sequence; blocks whose count reaches zero return to the free
 * queue. */
pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq);

/*
 * Reserves the next token slot of each of seqs[0..n-1], in that order (a
 * sequence may appear more than once).  slots[i] = block * block_size +
 * offset.  Every copy-on-write appends one (src, dst) pair to pairs (room for
 * n pairs) and *num_pairs receives their count; the copies must run
 * (paged_block_copy) before the writes.  Refuses with PKV_ERR_NO_BLOCKS,
 * changing nothing, when the batch needs more blocks than are free.
 */
pkv_status pkv_bm_append(pkv_block_manager *bm, const int64_t *seqs, int n,
                         int64_t *slots, int64_t *pairs, int *num_pairs);

/* Copies up to `capacity` entries of the sequence's block table to out;
 * *num_blocks receives the table length and *num_tokens its token count. */
pkv_status pkv_bm_table(const pkv_block_manager *bm, int64_t seq, int32_t *out,
                        int capacity, int *num_blocks, int64_t *num_tokens);

/* Free blocks, and a block's reference count (-1 on invalid arguments). */
int pkv_bm_num_free(const pkv_block_manager *bm);
int pkv_bm_refcount(const pkv_block_manager *bm, int block);

/* Human-readable name of a status code (static storage, never NULL). */
const char *pkv_status_string(pkv_status status);

/*
 * Read (and with clear != 0, reset) the library's device flag word for the
 * current device.  Synchronises `stream` first so every earlier call on it
 * has finished.  *flags_out receives an OR of PKV_FLAG_* bits.
 */
pkv_status pkv_read_device_flags(uint32_t *flags_out, int clear,
                                 pkv_stream_t stream);

/*
 * Text of the CUDA error behind the last PKV_ERR_CUDA returned on the calling
 * thread (error name, message and the step that failed); "no error" before
 * any.  Static per-thread storage, valid until the next failing call.
 */
const char *pkv_last_error_string(void);

/*
 * Host-side block manager with a prefix cache (no device memory involved).
 *
 * "PagedAttention and vLLM: Paging the KV Cache Like an OS" ..., section 2.4
 * (V1's block pool and hash chain) and summary point 5: full blocks are keyed
 * by a chained hash and stay in a key -> block map after their request
 * finishes, so that a later request whose prompt starts the same way takes
 * them over and skips their prefill.
 *  - Key of a full block: SHA-256 of the message (parent key: 32 bytes; each
 *    of the block's block_size token ids: 4 bytes little-endian; extra key:
 *    8 bytes little-endian).  The first block's parent key is 32 zero bytes.
 *    The extra key separates caches that must not mix (e.g. adapters).
 *  - Free blocks wait in one queue ordered by recency of release: a finished
 *    request's blocks go to the back (its last block first), allocation takes
 *    the front, and a block taken from the front leaves the map if it was
 *    cached.  The queue order is the eviction order.
 *  - Cached blocks are full and never written again: each request fills its
 *    own last block, so nothing is ever copied on write.
 * Not thread-safe: one manager, one thread at a time.
 */
typedef struct pkv_prefix_cache pkv_prefix_cache;

/* A manager of num_blocks blocks of block_size tokens; free_order (NULL =
 * ascending) is the initial queue, a permutation of 0..num_blocks-1.  Returns
 * NULL on invalid arguments.  Release with pkv_pc_destroy. */
pkv_prefix_cache *pkv_pc_create(int num_blocks, int block_size,
                                const int32_t *free_order);
void pkv_pc_destroy(pkv_prefix_cache *pc);

/* New request `seq` with prompt[0..prompt_len): walks the prompt's key chain
 * over the full blocks inside its first prompt_len - 1 tokens (the last
 * token is always recomputed) and takes over every block up to the first
 * miss.  *num_cached_tokens = the prompt tokens already in the cache (a
 * multiple of block_size); the caller appends the rest with pkv_pc_append.
 * PKV_ERR_RANGE if seq exists or prompt_len < 0. */
pkv_status pkv_pc_add_sequence(pkv_prefix_cache *pc, int64_t seq,
                               const int32_t *prompt, int prompt_len,
                               uint64_t extra_key, int *num_cached_tokens);

/* Reserves slots for the sequence's next n tokens (their ids in tokens[]):
 * slots[i] = block * block_size + offset.  A block that becomes full is keyed
 * and entered in the map unless its key is cached already.  Refuses with
 * PKV_ERR_NO_BLOCKS, changing nothing, when the call needs more blocks than
 * the free queue holds. */
pkv_status pkv_pc_append(pkv_prefix_cache *pc, int64_t seq,
                         const int32_t *tokens, int n, int64_t *slots);

/* Finishes the request: every block's count drops; blocks reaching zero go
 * to the back of the free queue, keeping their cached keys. */
pkv_status pkv_pc_free_sequence(pkv_prefix_cache *pc, int64_t seq);

/* The sequence's block table (up to capacity entries), its block and token
 * counts. */
pkv_status pkv_pc_table(const pkv_prefix_cache *pc, int64_t seq, int32_t *out,
                        int capacity, int *num_blocks, int64_t *num_tokens);

/* Blocks in the free queue (cached ones included); entries in the map. */
int pkv_pc_num_free(const pkv_prefix_cache *pc);
int pkv_pc_num_cached(const pkv_prefix_cache *pc);
/* Reference count of a block (-1 if out of range). */
int pkv_pc_refcount(const pkv_prefix_cache *pc, int block);
/* *cached = 1 and key32[0..32) = the block's key when the block is cached. */
pkv_status pkv_pc_block_key(const pkv_prefix_cache *pc, int block,
                            uint8_t *key32, int *cached);
/* The free queue from front to back (up to capacity entries); *count = its
 * length. */
pkv_status pkv_pc_free_queue(const pkv_prefix_cache *pc, int32_t *out,
                             int capacity, int *count);
/* Keys of the num_tokens / block_size full blocks of a token stream (32
 * bytes each, in order) -- the chain a request would look up. */
pkv_status pkv_pc_chain_keys(const int32_t *tokens, int num_tokens,
                             int block_size, uint64_t extra_key,
                             uint8_t *keys_out);
/* SHA-256 (FIPS 180-4) of msg[0..len) into digest32[0..32). */
pkv_status pkv_sha256(const void *msg, size_t len, uint8_t *digest32);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H */
