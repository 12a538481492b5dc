// Multi-query paged attention on the fifth-generation tensor cores: chunked
// prefill (a piece of a long prompt processed in one pass, its queries
// attending causally to the sequence's earlier tokens and to each other) and
// decode tokens in the same batch ("Paging the KV Cache Like an OS",
// continuous batching and chunked prefill).
//
// One CTA = one work unit: a sequence s, a KV head h and two query tiles A
// and B of that sequence.  A query tile is 128 rows: TQ = 128 / G consecutive
// query tokens times the G query heads that share KV head h (row r = token
// r / G, head r % G); tile B holds the TQ tokens before tile A's.  The CTA
// walks the sequence's block table in KV tiles of 128 tokens, each K and V
// tile loaded once and used by both query tiles:
//
//   S_x = Q_x K^T    tcgen05.mma (A and B from shared memory), M = 128 rows,
//                    N = 128 keys, K = head_dim, into TMEM
//   P_x = exp2(S_x * scale * log2 e - m)   per row, causal mask on diagonal
//                    tiles, written over S_x in TMEM as 16-bit hi and lo
//                    parts (P = hi + lo to about 2^-16 relative)
//   O_x += P_x V     tcgen05.mma with A (P hi, then P lo) from TMEM and V from
//                    shared memory, M = 128, N = head_dim, K = 128 keys
//
// with an online softmax whose running maximum is only raised when a score
// exceeds it by more than 2^8 (O_x in TMEM is then rescaled), and the
// normalisation by the running sum in the epilogue.  The tensor core
// alternates between the tiles (S_A, S_B, P_A V, S_A next, P_B V, S_B next,
// ...), so that it works on one tile while the softmax warps work on the
// other.  An MMA issued after another by the same thread runs after it, so
// S_x of the next KV tile may overwrite P_x once P_x V has been issued; and a
// commit tracks every earlier MMA of its thread, so when S_x is seen
// complete, the previous P_x V (and so O_x) is complete too.
//
// Warp roles (384 threads; 448 when V is converted): warps 0-7 are two
// softmax warpgroups; warpgroup x owns query tile x, thread t of it query row
// t % 128 (TMEM lane) with all 128 key columns, so the two tiles' softmax run
// side by side.  (When V is converted, the four extra warps leave fewer
// registers: there thread t of warpgroup wg owns key columns wg*64 ..
// wg*64+63 of row t % 128 of both tiles, and the two threads of a row agree
// on its maximum through shared memory.)  Warp 8 issues the TMA loads of the
// two Q tiles (once) and of the K tiles, warp 10 those of the V tiles (warp
// 8 both when warp 10 converts V), through rings, one box per block (all its
// tokens) and 64 dims, the block-table entries fetched a group of 32 ahead.
// Warp 9 allocates TMEM and issues the MMAs (one lane).  Warps 10-13 convert
// V tiles to f16 when P goes in as f16 and the cache is bf16; otherwise warp
// 10 loads V and warp 11 idles.  All hand-offs are mbarriers; every wait is
// bounded and a timeout sets PKV_FLAG_TIMEOUT, after which each role stops
// issuing and drains what it has in flight before the CTA frees its TMEM and
// exits.
//
// Shared memory (head_dim 128): Q_A and Q_B 32 KiB each, five K/V stages of
// 32 KiB (3 K + 2 V; 2 K + 3 V when V is converted, which then also waits
// for its conversion), in the 128-byte swizzled layout (rows of 64
// elements); one CTA per SM.  TMEM columns: tile
// x at 256 x: S_x / P_x (P hi 0..63, P lo 64..127), O_x at 128.
#pragma once

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_launch.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int CK_ROWS = 128;     // query rows per tile (MMA M)
constexpr int CK_BN = 128;       // keys per KV tile
constexpr int CK_PRODUCER = 8;   // warp ids
constexpr int CK_MMA = 9;
constexpr int CK_CONV = 10;      // first V-converting warp (f16 P from a bf16 cache)
// Threads: 8 softmax warps, the TMA warp, the MMA warp and the converting
// warps -- four (one per SM sub-partition) when a bf16 V tile is converted to
// f16, two otherwise (then idle).
__host__ __device__ constexpr int ck_threads(bool convert) { return convert ? 448 : 384; }
// K and V rings share five tile stages: 3 K + 2 V, or 2 K + 3 V when V is
// converted to f16 (a V stage then also waits for its conversion)
constexpr int CK_STAGES = 5;
constexpr int CK_ST_MAX = 3;     // barrier slots per ring
__host__ __device__ constexpr int ck_kst(bool convert) { return convert ? 2 : 3; }
__host__ __device__ constexpr int ck_vst(bool convert) { return CK_STAGES - ck_kst(convert); }
constexpr float CK_SLACK = 8.0f; // lazy rescale threshold (log2 domain)
constexpr int CK_ORDER_MAX = 64; // sequences ranked by length at launch (at most)
constexpr int CK_SCAN_MAX = 2048;   // up to this many sequences the grid holds only real units

template <int D>
struct ChunkCfg {
  static constexpr int NH = D / 64;            // 64-element column halves
  static constexpr int HALF = CK_ROWS * 128;   // one half-tile: 128 rows x 128 bytes
  static constexpr int Q_BYTES = NH * HALF;
  static constexpr int KV_BYTES = NH * HALF;
  static constexpr int OFF_Q = 0;              // Q_A, then Q_B
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_BAR = OFF_K + CK_STAGES * KV_BYTES;   // K stages, then V stages
  static constexpr int NBAR = 26;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  // (V converted) row-maximum exchange of the two softmax warpgroups:
  // [2 rounds][2][128]
  static constexpr int OFF_RED = OFF_TMEM + 16;
  static constexpr int SMEM = OFF_RED + 2 * 2 * CK_ROWS * 4;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TILE_COLS = 256;   // TMEM columns per query tile
  static constexpr uint32_t COL_O = 128;       // within a tile
  static constexpr uint32_t COL_PL = 64;       // P lo within a tile (P hi at 0)
};

// mbarrier slots
enum : int {
  CB_Q = 0,                  // both Q tiles landed (tx)
  CB_KF = 1,                 // K stage full [K stages] (tx)
  CB_KE = CB_KF + CK_ST_MAX, // K stage free [K stages] (MMA commit)
  CB_VF = CB_KE + CK_ST_MAX, // V stage full [V stages] (tx)
  CB_VE = CB_VF + CK_ST_MAX, // V stage free [V stages] (MMA commit)
  CB_SF = CB_VE + CK_ST_MAX, // S_x computed [2: tiles A, B] (MMA commit)
  CB_PF = CB_SF + 2,         // P_x written [2] (one arrival per softmax warp writing P_x)
  CB_OF = CB_PF + 2,         // O_x final [2] (MMA commit)
  CB_PAIR = CB_OF + 2,       // (V converted) row-maximum exchange of warps w, w + 4 [4] (64 arrivals)
  CB_VC = CB_PAIR + 4,       // V stage converted to f16 [V stages] (one arrival per converting thread)
  CB_COUNT = CB_VC + CK_ST_MAX,
};

// max(a, b, c) in one instruction (sm_100 and later); like fmaxf, a NaN
// operand is ignored
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// In-place exclusive prefix sum of v[0..n) in shared memory by the whole
// CTA of NT threads; returns the total.  red[0..NT/32) is scratch.  Every
// thread must call it.
template <int NT>
__device__ __forceinline__ int cta_exclusive_scan(int *v, int n, int *red) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int NWARP = NT / 32;
  const int per = (n + NT - 1) / NT;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int sum = 0;
  for (int i = b0; i < b1; ++i) sum += v[i];
  int x = sum;   // inclusive within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(FULL_MASK, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) red[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = lane < NWARP ? red[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, t, off);
      if (lane >= off) t += y;
    }
    if (lane < NWARP) red[lane] = t;   // inclusive over warps
  }
  __syncthreads();
  int run = x - sum + (wid ? red[wid - 1] : 0);
  for (int i = b0; i < b1; ++i) {
    const int c = v[i];
    v[i] = run;
    run += c;
  }
  const int total = red[NWARP - 1];
  __syncthreads();
  return total;
}

// Every lane of the warp waits; the result is the same on all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait_bounded(bar, parity);
  return __all_sync(FULL_MASK, ok);
}

__device__ __forceinline__ void store_row32(void *out, size_t base, int out_dtype,
                                            const float *v) {
  if (out_dtype == PKV_F32) {
    float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
#pragma unroll
    for (int e = 0; e < 8; ++e) d[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
  } else {
    uint32_t w[16];
    if (out_dtype == PKV_BF16) {
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = Mma<__nv_bfloat16>::pack(v[2 * e], v[2 * e + 1]);
      uint4 *d = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + base);
#pragma unroll
      for (int e = 0; e < 4; ++e) d[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = Mma<__half>::pack(v[2 * e], v[2 * e + 1]);
      uint4 *d = reinterpret_cast<uint4 *>(static_cast<__half *>(out) + base);
#pragma unroll
      for (int e = 0; e < 4; ++e) d[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    }
  }
}

// OVL: the chunked pass of a mixed batch whose decode pass (the kernel
// before this one, launched first) still runs on other SMs.  The decode
// grid lets this one start as soon as it holds its SMs, and everything this
// kernel reads was complete before the decode grid started, so it does not
// wait for its predecessor at the start; instead the last of its CTAs to
// leave waits for the decode grid, so that this grid ends after it and the
// stream's next work sees both passes done.
template <typename T, int D, int B, bool P16, bool OVL>
__global__ void __launch_bounds__(ck_threads(P16 && std::is_same<T, __nv_bfloat16>::value), 1)
    chunked_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const ChunkedParams p) {
  using C = ChunkCfg<D>;
  static_assert(CB_COUNT <= C::NBAR, "mbarrier slots");
  constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
  // P16: P enters P.V as one f16 MMA operand (instead of hi + lo halves of the
  // cache dtype); a bf16 V tile is then converted to f16 in shared memory.
  constexpr bool CONVERT = P16 && BF16;
  constexpr int NT = ck_threads(CONVERT);
  constexpr int NCONV = NT - CK_CONV * 32;       // converting threads
  constexpr int CK_KST = ck_kst(CONVERT), CK_VST = ck_vst(CONVERT);
  constexpr int OFF_V = C::OFF_K + CK_KST * C::KV_BYTES;
  static_assert(B * 128 % 1024 == 0, "boxes land on 1 KiB boundaries (128-byte swizzle atoms)");
  constexpr int BLOCKS_PER_TILE = CK_BN / B;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sm = smem_raw;
  const uint32_t sb = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * (uint32_t)i; };

  // ---- the unit: the query-tile pairs of one (sequence, KV head) are
  // adjacent in the grid, heaviest (last) pair first, so that they run at
  // the same time and read each K/V tile from L2 rather than from HBM.
  int s, kvh, pr_rev;
  // (OVL) every way out of the kernel passes here once per CTA
  auto ovl_leave = [&]() {
    if constexpr (OVL) {
      if (tid == 0 && atomicAdd(p.ovl_done, 1u) == gridDim.x - 1) pdl_wait_predecessors();
    }
  };
  if constexpr (!OVL) pdl_wait_predecessors();
  // Up to CK_ORDER_MAX sequences launch longest context first (ties by
  // index; more keep index order): the CTAs of the longest contexts start in
  // the first waves and the last wave holds short ones, so the SMs run out of
  // work at nearly the same time.  Every CTA ranks the lengths the same way.
  const int S = p.num_seqs;
  const bool ranked = S > 1 && S <= CK_ORDER_MAX;
  int *qs_s = reinterpret_cast<int *>(sm + C::OFF_K);   // scratch: the K ring is still empty
  int *cnt_s = qs_s + CK_SCAN_MAX + 1;   // lengths, then units per launch slot, then offsets
  int *ord_s = cnt_s + CK_SCAN_MAX;      // launch slot -> sequence
  int *red = ord_s + CK_SCAN_MAX;        // [32] scan partials, [32] the slot found
  auto rank_sequences = [&]() {
    for (int i = tid; i < S; i += NT) {
      int r = i;
      if (ranked) {
        const int li = cnt_s[i];
        r = 0;
        for (int j = 0; j < S; ++j) {
          const int lj = cnt_s[j];
          r += (lj > li) || (lj == li && j < i);
        }
      }
      ord_s[r] = i;
    }
  };
  if (p.compact) {
    // The grid holds only units that exist (many sequences have fewer query
    // tiles than the longest): every CTA lists the sequences' unit counts
    // (query-tile pairs x KV heads; a sequence whose query range is invalid
    // keeps one unit, which flags it) in launch order, takes the exclusive
    // sum and finds its own unit.
    const int TQ = p.tile_tokens;
    for (int i = tid; i <= S; i += NT) qs_s[i] = p.query_start[i];
    for (int i = tid; i < S; i += NT) cnt_s[i] = p.context_lens[i];
    __syncthreads();
    rank_sequences();
    __syncthreads();
    for (int r = tid; r < S; r += NT) {
      const int q = ord_s[r];
      const int a = qs_s[q], b = qs_s[q + 1], n = b - a;
      const bool valid = a >= 0 && n >= 0 && b <= p.num_tokens && n <= p.max_query_len;
      const int pairs = !valid ? 1 : (p.skip_single && n == 1 ? 0 : ((n + TQ - 1) / TQ + 1) / 2);
      cnt_s[r] = pairs * p.num_kv_heads;
    }
    if (tid == 0) red[32] = -1;
    __syncthreads();
    const int total = cta_exclusive_scan<NT>(cnt_s, S, red);
    const int b = (int)blockIdx.x;
    for (int r = tid; r < S; r += NT)
      if (cnt_s[r] <= b && b < (r + 1 < S ? cnt_s[r + 1] : total)) red[32] = r;
    __syncthreads();
    const int r = red[32];
    // (the grid is an upper bound; it falls short only when query ranges
    // overlap, which no valid batch has)
    if (b == 0 && tid == 0 && total > (int)gridDim.x) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    if (b >= total || r < 0) {
      ovl_leave();
      return;
    }
    s = ord_s[r];
    const int units = (r + 1 < S ? cnt_s[r + 1] : total) - cnt_s[r];
    const int npairs = units / p.num_kv_heads;
    kvh = (b - cnt_s[r]) / npairs;
    pr_rev = (b - cnt_s[r]) % npairs;
  } else {
    // every (sequence, KV head, pair) slot of the longest query range
    int id = blockIdx.x;
    pr_rev = id % p.num_qpairs;
    id /= p.num_qpairs;
    kvh = id % p.num_kv_heads;
    s = id / p.num_kv_heads;               // rank of the sequence in launch order
    if (ranked) {
      for (int i = tid; i < S; i += NT) cnt_s[i] = p.context_lens[i];
      __syncthreads();
      rank_sequences();
      __syncthreads();
      s = ord_s[s];
    }
  }
  fence_proxy_async_smem();   // the scratch is a TMA destination later
  const int q0 = p.query_start[s], q1 = p.query_start[s + 1];
  const int n = q1 - q0;
  if (p.skip_single && n == 1) {   // a decode row: the decode kernel's
    ovl_leave();
    return;
  }
  int L = p.context_lens[s];
  if (q0 < 0 || n < 0 || q1 > p.num_tokens || n > p.max_query_len || L < n) {
    if (tid == 0 && pr_rev == 0 && kvh == 0) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    ovl_leave();
    return;
  }
  if (L > p.max_blocks * B) {
    if (tid == 0 && pr_rev == 0 && kvh == 0) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    L = p.max_blocks * B;
    if (L < n) {
      ovl_leave();
      return;
    }
  }
  const int TQ = p.tile_tokens;
  const int G = p.group;
  const int nq = (n + TQ - 1) / TQ;
  if (2 * pr_rev >= nq) {
    ovl_leave();
    return;
  }
  int tb[2], te[2], pm[2], nk[2];              // per query tile: tokens [tb, te), last
  tb[0] = (nq - 1 - 2 * pr_rev) * TQ;          // position, KV tiles it needs
  tb[1] = tb[0] - TQ;                          // tile B: the TQ tokens before A's
  for (int x = 0; x < 2; ++x) {
    te[x] = min(n, tb[x] + TQ);
    pm[x] = L - n + te[x] - 1;
    nk[x] = tb[x] >= 0 ? pm[x] / CK_BN + 1 : 0;
  }
  const int ntile = 1 + (nk[1] > 0);           // query tiles in this unit
  const int nkv = nk[0];                       // KV tiles streamed (tile A needs most)
  const int nb_valid = (L + B - 1) / B;

  if (sb & 1023u) {   // the swizzled tiles need a 1 KiB-aligned base
    if (tid == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
    ovl_leave();
    return;
  }
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C::OFF_TMEM);
  if (tid == 0) {
    mbar_init(bar(CB_Q), 1);
    for (int i = 0; i < CK_KST; ++i) {
      mbar_init(bar(CB_KF + i), 1);
      mbar_init(bar(CB_KE + i), 1);
    }
    for (int i = 0; i < CK_VST; ++i) {
      mbar_init(bar(CB_VF + i), 1);
      mbar_init(bar(CB_VE + i), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(CB_SF + x), 1);
      mbar_init(bar(CB_PF + x), CONVERT ? 8 : 4);   // softmax warps writing P_x
      mbar_init(bar(CB_OF + x), 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(bar(CB_PAIR + i), 64);
    for (int i = 0; i < CK_VST; ++i) mbar_init(bar(CB_VC + i), NCONV);
    fence_barrier_init();
  }
  // rows of the Q tiles that no token fills (G not dividing 128) are zero
  const int q_rows = TQ * G;
  if (q_rows < CK_ROWS) {
    const int per = (CK_ROWS - q_rows) * 8;    // 16-byte chunks per half-tile
    for (int x = tid; x < 2 * C::NH * per; x += NT) {
      const int h = x / per, rem = x % per;    // h: (tile, column half)
      *reinterpret_cast<uint4 *>(sm + C::OFF_Q + h * C::HALF + (q_rows + rem / 8) * 128 +
                                 (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == CK_MMA) {
    tc::tmem_alloc(smem_addr(tslot), C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  bool ok = true;

  if (warp == CK_PRODUCER || (!CONVERT && warp == CK_CONV)) {
    // ------------------------------------------------------------ producers
    // Warp 8 loads the Q tiles and the K tiles, warp 10 the V tiles (when it
    // does not convert V; then warp 8 loads both), so that K runs ahead of V
    // as far as its ring allows.  A producer warp runs the loop as a whole:
    // lane i holds block-table entry i of the current group of 32 (TPG
    // tiles), the next group's entries are already in flight, and the lanes
    // issue the TMA loads.
    const bool do_k = warp == CK_PRODUCER;
    const bool do_v = warp == CK_CONV || CONVERT;
    constexpr int TPG = 32 / BLOCKS_PER_TILE;    // tiles per group of 32 entries
    const int32_t *tbl = p.block_tables + (size_t)s * p.max_blocks;
    const int nb_used = min(nb_valid, nkv * BLOCKS_PER_TILE);
    auto fetch = [&](int grp) -> int {
      const int lb = grp * 32 + lane;
      int blk = p.num_blocks;                    // past the pool: TMA fills zeros
      if (lb < nb_used) {
        const int x = __ldg(tbl + lb);
        if (x < 0 || x >= p.num_blocks) atomicOr(p.flags, PKV_FLAG_BLOCK_RANGE);
        else blk = x;
      }
      return blk;
    };
    if (do_k && lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      mbar_arrive_expect_tx(bar(CB_Q), (uint32_t)(ntile * C::NH * 128 * q_rows));
      for (int x = 0; x < ntile; ++x)
        for (int h = 0; h < C::NH; ++h)
          tma_load_3d(sb + C::OFF_Q + x * C::Q_BYTES + h * C::HALF, &qmap, h * 64, kvh * G,
                      q0 + tb[x], bar(CB_Q));
    }
    // one TMA box per (block, 64-dim half) of the tile, lane i issuing box i
    // (issuing them from one lane in turn is a little slower)
    static_assert(BLOCKS_PER_TILE * C::NH <= 32, "one box per lane");
    auto load_tile = [&](const CUtensorMap *map, uint32_t dst, const int (&blk)[BLOCKS_PER_TILE],
                         uint32_t full) {
      if (lane < BLOCKS_PER_TILE * C::NH) {
        const int b = lane / C::NH, h = lane % C::NH;
        int bb = blk[0];
#pragma unroll
        for (int i = 1; i < BLOCKS_PER_TILE; ++i)
          if (b == i) bb = blk[i];
        tma_load_4d_keep(dst + h * C::HALF + b * B * 128, map, h * 64, kvh, 0, bb, full);
      }
    };
    int cur = fetch(0), nxt = fetch(1);
    int nk_issued = 0, nv_issued = 0;
    for (int j = 0; j < nkv; ++j) {
      if (j > 0 && j % TPG == 0) {
        cur = nxt;
        nxt = fetch(j / TPG + 1);
      }
      int blk[BLOCKS_PER_TILE];
#pragma unroll
      for (int b = 0; b < BLOCKS_PER_TILE; ++b)
        blk[b] = __shfl_sync(FULL_MASK, cur, (j % TPG) * BLOCKS_PER_TILE + b);
      const int ks = j % CK_KST, vs = j % CK_VST;
      if (do_k) {
        if (j >= CK_KST && !warp_wait(bar(CB_KE + ks), ((uint32_t)(j / CK_KST) & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(CB_KF + ks), (uint32_t)C::KV_BYTES);
        __syncwarp();
        load_tile(&kmap, sb + C::OFF_K + ks * C::KV_BYTES, blk, bar(CB_KF + ks));
        nk_issued = j + 1;
      }
      if (do_v) {
        if (j >= CK_VST && !warp_wait(bar(CB_VE + vs), ((uint32_t)(j / CK_VST) & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(CB_VF + vs), (uint32_t)C::KV_BYTES);
        __syncwarp();
        load_tile(&vmap, sb + OFF_V + vs * C::KV_BYTES, blk, bar(CB_VF + vs));
        nv_issued = j + 1;
      }
    }
    // drain: every load issued has landed before the CTA may exit (loads
    // older than a ring's worth were consumed, so they have landed)
    if (lane == 0) {
      if (do_k) mbar_wait_bounded(bar(CB_Q), 0);
      for (int j = max(0, nk_issued - CK_KST); j < nk_issued; ++j)
        mbar_wait_bounded(bar(CB_KF + j % CK_KST), (uint32_t)(j / CK_KST) & 1u);
      for (int j = max(0, nv_issued - CK_VST); j < nv_issued; ++j)
        mbar_wait_bounded(bar(CB_VF + j % CK_VST), (uint32_t)(j / CK_VST) & 1u);
      if (!ok) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
    }
  } else if (warp == CK_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // Order: S_A(0), S_B(0); then per KV tile j: P_A(j) V(j), S_A(j+1),
    // P_B(j) V(j), S_B(j+1).
    constexpr uint32_t ID_S = tc::idesc_f16(BF16, CK_ROWS, CK_BN, false);
    constexpr uint32_t ID_PV = tc::idesc_f16(BF16 && !P16, CK_ROWS, D, true);
    // The MMA issue rate is set by this one thread, and an MMA whose
    // descriptors are rebuilt from addresses just before it issues well below
    // the pipe's rate (measured on this GPU: ~100 cycles apart instead of 66
    // for a 128 x 128 x 16 MMA).  So the descriptors' high words (stride,
    // version, swizzle: the same for every tile) and the Q tiles' low words
    // are built once, a K or V stage's low word before the barrier waits that
    // precede its MMAs, and each K step adds its offset in 16-byte units to
    // the low word's start-address field (no carry: shared-memory addresses
    // stay below 2^18).
    const uint32_t hqk = (uint32_t)(tc::sdesc_sw128(sb, 16, 1024) >> 32);
    const uint32_t hv = (uint32_t)(tc::sdesc_sw128(sb, C::HALF, 1024) >> 32);
    const uint32_t lq[2] = {(uint32_t)tc::sdesc_sw128(sb + C::OFF_Q, 16, 1024),
                            (uint32_t)tc::sdesc_sw128(sb + C::OFF_Q + C::Q_BYTES, 16, 1024)};
    auto k_lo = [&](int j) {                     // low word of K(j)'s stage
      return (uint32_t)tc::sdesc_sw128(sb + C::OFF_K + (j % CK_KST) * C::KV_BYTES, 16, 1024);
    };
    auto v_lo = [&](int j) {
      return (uint32_t)tc::sdesc_sw128(sb + OFF_V + (j % CK_VST) * C::KV_BYTES, C::HALF, 1024);
    };
    auto issue_s = [&](int x, uint32_t lk) {     // S_x = Q_x K^T, K's stage low word lk
      if (lane == 0) {
        const uint32_t d = tmem + (uint32_t)x * C::TILE_COLS;
        const uint32_t lqx = x ? lq[1] : lq[0];
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)(((k >> 2) * C::HALF + (k & 3) * 32) >> 4);
          tc::mma_f16_ss(d, tc::desc_pack(lqx + off, hqk), tc::desc_pack(lk + off, hqk), ID_S,
                         k > 0 ? 1u : 0u);
        }
        tc::commit(bar(CB_SF + x));
      }
    };
    auto issue_pv = [&](int x, int j, uint32_t lv) {   // O_x += P_x(j) V(j), V's low word lv
      if (lane == 0) {
        const uint32_t t0 = tmem + (uint32_t)x * C::TILE_COLS;
        const uint32_t first = j > 0 ? 1u : 0u;
#pragma unroll
        for (int k = 0; k < CK_BN / 16; ++k) {
          const uint64_t bv = tc::desc_pack(lv + (uint32_t)(k * (2048 >> 4)), hv);   // 16 V rows a step
          tc::mma_f16_ts(t0 + C::COL_O, t0 + 8u * k, bv, ID_PV, k > 0 ? 1u : first);
          if (!P16) tc::mma_f16_ts(t0 + C::COL_O, t0 + C::COL_PL + 8u * k, bv, ID_PV, 1u);
        }
        if (j == nk[x] - 1) tc::commit(bar(CB_OF + x));
      }
    };
    auto wait_k = [&](int j) {
      return warp_wait(bar(CB_KF + j % CK_KST), (uint32_t)(j / CK_KST) & 1u);
    };
    // Up to three barriers polled together with one vote at the end: in this
    // warp, which shares its issue slots with two softmax warps, even a
    // satisfied wait-and-vote costs ~150-230 cycles (measured).
    auto wait3 = [&](uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1, bool use2, uint32_t b2,
                     uint32_t p2) {
      bool d0 = false, d1 = false, d2 = !use2;
      for (uint32_t it = 0; it < WAIT_LIMIT && !(d0 && d1 && d2); ++it) {
        if (!d0) d0 = mbar_try_wait(b0, p0);
        if (!d1) d1 = mbar_try_wait(b1, p1);
        if (!d2) d2 = mbar_try_wait(b2, p2);
      }
      return __all_sync(FULL_MASK, d0 && d1 && d2);
    };
    const int tail_tile = (L % CK_BN) ? (L - 1) / CK_BN : -1;
    ok = wait3(bar(CB_Q), 0, bar(CB_KF + 0), 0, false, 0, 0);
    if (ok) {
      tc::fence_after_sync();
      issue_s(0, k_lo(0));
      if (nk[1] > 0) issue_s(1, k_lo(0));
      if (lane == 0) tc::commit(bar(CB_KE + 0));
      __syncwarp();
    }
    for (int j = 0; j < nkv && ok; ++j) {
      const uint32_t lv = v_lo(j), lk1 = k_lo(j + 1);   // before the waits
      // V(j), P_A(j) and K(j + 1) (usually long landed) are all waited for
      // first, so that P_A(j) V(j) and S_A(j + 1) issue back to back
      const bool next_a = j + 1 < nk[0];
      if (!wait3(bar((CONVERT ? CB_VC : CB_VF) + j % CK_VST), (uint32_t)(j / CK_VST) & 1u,
                 bar(CB_PF + 0), (uint32_t)j & 1u, next_a, bar(CB_KF + (j + 1) % CK_KST),
                 (uint32_t)((j + 1) / CK_KST) & 1u)) {
        ok = false;
        break;
      }
      if (!CONVERT && j == tail_tile) {
        // V rows past the sequence hold whatever the pool holds there; their
        // probabilities are exactly zero, but 0 * NaN is not, so zero them
        const int z0 = L - j * CK_BN;
        unsigned char *vsm = sm + OFF_V + (j % CK_VST) * C::KV_BYTES;
        for (int x = lane; x < (CK_BN - z0) * 8 * C::NH; x += 32) {
          const int h = x / ((CK_BN - z0) * 8), rem = x % ((CK_BN - z0) * 8);
          *reinterpret_cast<uint4 *>(vsm + h * C::HALF + (z0 + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc::fence_after_sync();
      issue_pv(0, j, lv);
      if (next_a) {
        issue_s(0, lk1);
        if (j + 1 >= nk[1] && lane == 0) tc::commit(bar(CB_KE + (j + 1) % CK_KST));
      }
      if (j < nk[1]) {
        if (!warp_wait(bar(CB_PF + 1), (uint32_t)j & 1u)) { ok = false; break; }
        tc::fence_after_sync();
        issue_pv(1, j, lv);
      }
      if (lane == 0) tc::commit(bar(CB_VE + j % CK_VST));
      if (j + 1 < nk[1]) {
        issue_s(1, lk1);
        if (lane == 0) tc::commit(bar(CB_KE + (j + 1) % CK_KST));
      }
      __syncwarp();
    }
    // drain: the MMAs issued have completed before TMEM is freed (the O
    // commits come after every MMA of a complete run; after a timeout these
    // waits give up in their turn)
    for (int x = 0; x < ntile; ++x) warp_wait(bar(CB_OF + x), 0);
    if (!ok && lane == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
  } else if (warp >= CK_CONV) {
    // ------------------------------------------------------------ V to f16
    // (P16 with a bf16 cache only.)  Each V tile is converted in place, 16
    // bytes at a time (the swizzle only moves whole 16-byte chunks, so a chunk
    // converts where it lies); rows past the sequence become zeros.  f16 holds
    // every bf16 value of magnitude 2^-14 .. 65504 exactly; smaller ones lose
    // at most 2^-25 absolutely; larger ones saturate to +-65504 and are flagged
    // (NaN stays NaN).
    if constexpr (CONVERT) {
      const int ct = tid - CK_CONV * 32;           // 0..NCONV-1
      uint32_t vmax = 0;                           // largest |V| met, as bf16 bits
      for (int j = 0; j < nkv && ok; ++j) {
        const int vs = j % CK_VST;
        if (!warp_wait(bar(CB_VF + vs), (uint32_t)(j / CK_VST) & 1u)) { ok = false; break; }
        unsigned char *vsm = sm + OFF_V + vs * C::KV_BYTES;
        const int live = min(CK_BN, L - j * CK_BN);  // rows holding tokens of the sequence
#pragma unroll 4
        for (int c = ct; c < CK_BN * 8 * C::NH; c += NCONV) {
          const int h = c / (CK_BN * 8), rem = c % (CK_BN * 8), r = rem / 8;
          uint4 *ptr = reinterpret_cast<uint4 *>(vsm + h * C::HALF + r * 128 + (rem % 8) * 16);
          uint4 w = make_uint4(0, 0, 0, 0);
          if (r < live) {
            w = *ptr;
            uint32_t *ww = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              // largest magnitude seen (bf16 bits without the sign, both halves)
              vmax = max(vmax, max(ww[e] & 0x7fffu, (ww[e] >> 16) & 0x7fffu));
              const float2 f = Widen<__nv_bfloat16>::pair(ww[e]);
              asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(ww[e]) : "f"(f.y), "f"(f.x));
            }
          }
          *ptr = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(CB_VC + vs));
      }
      // bf16 magnitudes above 65504 (0x477f) became +-65504
      if (vmax > 0x477fu) atomicOr(p.flags, PKV_FLAG_V_RANGE);
      if (!ok && lane == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax
    if constexpr (!CONVERT) {
      // Warpgroup x owns query tile x: thread t holds row t (TMEM lane t) of it,
      // all CK_BN key columns, so a row's maximum and sum need no exchange and
      // the two tiles' softmax run side by side.
      const int x = warp >> 2;                  // query tile of this warpgroup
      const int r = tid & (CK_ROWS - 1);        // query row = TMEM lane
      const int tl = r / G, g = r % G;
      const uint32_t tt = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)x * C::TILE_COLS;
      const float sl2 = p.scale_log2;
      const int tok = tb[x] + tl;
      const bool valid = x < ntile && tl < TQ && tok < te[x];
      const int p_row = valid ? (L - n + tok) : pm[x];
      float m = -INFINITY, l = 0.f;
      uint32_t sr[CK_BN];
      const int njx = x < ntile ? nk[x] : 0;
      for (int j = 0; j < njx && ok; ++j) {
        if (!warp_wait(bar(CB_SF + x), (uint32_t)j & 1u)) { ok = false; break; }
        tc::fence_after_sync();
        const int lim = p_row - j * CK_BN;      // columns 0..lim are visible
        float alpha = 1.f;
        bool resc = false;
        const float2 sl2x2 = make_float2(sl2, sl2);
        float2 lsum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        {
          // S all in registers, so P may overwrite its columns as it goes
#pragma unroll
          for (int c = 0; c < CK_BN / 32; ++c) tc::ld_32x32b_x32(tt + (uint32_t)(c * 32), sr + 32 * c);
          tc::wait_ld();
          if (lim < CK_BN - 1) {
#pragma unroll
            for (int c = 0; c < CK_BN; ++c)
              if (c > lim) sr[c] = __float_as_uint(-INFINITY);
          }
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < CK_BN; c += 2)
            m4[(c >> 1) & 3] = fmax3(m4[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          // running maximum in the exp2 domain, raised lazily
          const float mnew = fmaxf(m, mx * sl2);
          resc = mnew > m + CK_SLACK;
          if (resc) {
            alpha = fast_exp2(m - mnew);
            m = mnew;
          }
          // P = exp2(s * scale * log2 e - m), 32 keys at a time: hi + lo pairs
          // of the cache dtype, or (P16) f16 pairs with the row sum taken over
          // the rounded values (each output row is then an exact convex
          // combination)
          const float2 negm = make_float2(-m, -m);
#pragma unroll
          for (int c = 0; c < CK_BN / 32; ++c) {
            uint32_t hiw[16], low[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int k0 = 32 * c + 2 * e;
              const float2 v = fma2(make_float2(__uint_as_float(sr[k0]), __uint_as_float(sr[k0 + 1])),
                                    sl2x2, negm);
              const float2 pe = make_float2(fast_exp2(v.x), fast_exp2(v.y));
              if constexpr (P16) {
                hiw[e] = Mma<__half>::pack(pe.x, pe.y);
                const float2 hf = Widen<__half>::pair(hiw[e]);
                lsum[e & 1] = make_float2(lsum[e & 1].x + hf.x, lsum[e & 1].y + hf.y);
              } else {
                lsum[e & 1] = make_float2(lsum[e & 1].x + pe.x, lsum[e & 1].y + pe.y);
                hiw[e] = Mma<T>::pack(pe.x, pe.y);
                const float2 hf = Widen<T>::pair(hiw[e]);
                low[e] = Mma<T>::pack(pe.x - hf.x, pe.y - hf.y);
              }
            }
            tc::st_32x32b_x16(tt + (uint32_t)(16 * c), hiw);
            if (!P16) tc::st_32x32b_x16(tt + C::COL_PL + (uint32_t)(16 * c), low);
          }
        }
        l = l * alpha + ((lsum[0].x + lsum[0].y) + (lsum[1].x + lsum[1].y));
        // O_x is quiet: the P_x V before this S_x has completed
        if (j > 0 && __any_sync(FULL_MASK, resc)) {
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            const uint32_t ta = tt + C::COL_O + (uint32_t)(c * 32);
            tc::ld_32x32b_x32(ta, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st_32x32b_x32(ta, o);
          }
        }
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(CB_PF + x));
      }
      // ---- epilogue: O_x / l_x
      if (x < ntile && ok) {
        if (!warp_wait(bar(CB_OF + x), 0)) {
          ok = false;
        } else {
          tc::fence_after_sync();
          const float inv = l > 0.f ? 1.f / l : 0.f;
          const size_t row = ((size_t)(q0 + (valid ? tok : 0)) * p.num_q_heads +
                              (size_t)kvh * G + g) * (size_t)D;
          uint32_t o[32];
          float v[32];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            tc::ld_32x32b_x32(tt + C::COL_O + (uint32_t)(c * 32), o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
            if (valid) store_row32(p.out, row + (size_t)c * 32, p.out_dtype, v);
          }
        }
      }
    } else {
      // (f16 P with a converted bf16 V: the converting warps leave fewer
      // registers, so the two warpgroups split each tile's key columns and
      // take tile A, then tile B, agreeing on a row's maximum through shared
      // memory.)
      constexpr int HC = CK_BN / 2;             // key columns per thread
      constexpr int HD = D / 2;                 // output columns per thread
      const int wg = warp >> 2;
      const int r = tid & (CK_ROWS - 1);        // query row = TMEM lane
      const int tl = r / G, g = r % G;
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t pair = bar(CB_PAIR + (warp & 3));
      float *red = reinterpret_cast<float *>(sm + C::OFF_RED);   // [2][2][128]
      const float sl2 = p.scale_log2;
      bool valid[2];
      int tok[2], p_row[2];
      float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
      for (int x = 0; x < 2; ++x) {
        tok[x] = tb[x] + tl;
        valid[x] = x < ntile && tl < TQ && tok[x] < te[x];
        p_row[x] = valid[x] ? (L - n + tok[x]) : pm[x];
      }
      int round = 0;                            // row-statistics exchanges so far
      // the two threads of a row combine v (max or sum) through shared memory
      auto exchange = [&](float v, bool is_max) -> float {
        float *rb = red + (round & 1) * 2 * CK_ROWS;
        rb[wg * CK_ROWS + r] = v;
        mbar_arrive(pair);
        if (!warp_wait(pair, (uint32_t)round & 1u)) ok = false;
        ++round;
        const float o = rb[(wg ^ 1) * CK_ROWS + r];
        return is_max ? fmaxf(v, o) : v + o;
      };
      uint32_t sr[HC];
      for (int j = 0; j < nkv && ok; ++j) {
        for (int x = 0; x < ntile && ok; ++x) {
          if (j >= nk[x]) continue;
          const uint32_t tt = tmem + lane_base + (uint32_t)x * C::TILE_COLS;
          if (!warp_wait(bar(CB_SF + x), (uint32_t)j & 1u)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < HC / 32; ++c) tc::ld_32x32b_x32(tt + (uint32_t)(wg * HC + c * 32), sr + 32 * c);
          tc::wait_ld();
          const int lim = p_row[x] - j * CK_BN - wg * HC;   // own columns 0..lim are visible
          if (lim < HC - 1) {
#pragma unroll
            for (int c = 0; c < HC; ++c)
              if (c > lim) sr[c] = __float_as_uint(-INFINITY);
          }
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < HC; c += 2)
            m4[(c >> 1) & 3] = fmax3(m4[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          // both threads have read their S columns once they meet, so P may
          // then overwrite any of the row's S columns
          const float mx = exchange(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])), true);
          if (!ok) break;
          // running maximum in the exp2 domain, raised lazily
          const float mnew = fmaxf(m[x], mx * sl2);
          const bool resc = mnew > m[x] + CK_SLACK;
          float alpha = 1.f;
          if (resc) {
            alpha = fast_exp2(m[x] - mnew);
            m[x] = mnew;
          }
          // P = exp2(s * scale * log2 e - m): as hi + lo pairs of the cache
          // dtype, or (P16) as f16 pairs with the row sum taken over the
          // rounded values (each output row is then an exact convex combination)
          const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m[x], -m[x]);
          float2 lsum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          uint32_t hiw[HC / 2], low[HC / 2];
#pragma unroll
          for (int e = 0; e < HC / 2; ++e) {
            const float2 v = fma2(make_float2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                                  sl2x2, negm);
            const float2 pe = make_float2(fast_exp2(v.x), fast_exp2(v.y));
            if constexpr (P16) {
              hiw[e] = Mma<__half>::pack(pe.x, pe.y);
              const float2 hf = Widen<__half>::pair(hiw[e]);
              lsum[e & 1] = make_float2(lsum[e & 1].x + hf.x, lsum[e & 1].y + hf.y);
            } else {
              lsum[e & 1] = make_float2(lsum[e & 1].x + pe.x, lsum[e & 1].y + pe.y);
              hiw[e] = Mma<T>::pack(pe.x, pe.y);
              const float2 hf = Widen<T>::pair(hiw[e]);
              low[e] = Mma<T>::pack(pe.x - hf.x, pe.y - hf.y);
            }
          }
          l[x] = l[x] * alpha + ((lsum[0].x + lsum[0].y) + (lsum[1].x + lsum[1].y));
          // O_x is quiet: the P_x V before this S_x has completed
          if (j > 0 && __any_sync(FULL_MASK, resc)) {
            uint32_t o[32];
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              const uint32_t ta = tt + C::COL_O + (uint32_t)(wg * HD + c * 32);
              tc::ld_32x32b_x32(ta, o);
              tc::wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tc::st_32x32b_x32(ta, o);
            }
          }
          tc::st_32x32b_x32(tt + (uint32_t)(wg * (HC / 2)), hiw);
          if (!P16) tc::st_32x32b_x32(tt + C::COL_PL + (uint32_t)(wg * (HC / 2)), low);
          tc::wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(CB_PF + x));
        }
      }
      // ---- epilogue: O_x / l_x, a row's sum being its two threads' partial sums
      for (int x = 0; x < ntile && ok; ++x) {
        l[x] = exchange(l[x], false);
        if (!ok || !warp_wait(bar(CB_OF + x), 0)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t tt = tmem + lane_base + (uint32_t)x * C::TILE_COLS;
        const float inv = l[x] > 0.f ? 1.f / l[x] : 0.f;
        const size_t row = ((size_t)(q0 + (valid[x] ? tok[x] : 0)) * p.num_q_heads +
                            (size_t)kvh * G + g) * (size_t)D + (size_t)(wg * HD);
        uint32_t o[32];
        float v[32];
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          tc::ld_32x32b_x32(tt + C::COL_O + (uint32_t)(wg * HD + c * 32), o);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
          if (valid[x]) store_row32(p.out, row + (size_t)c * 32, p.out_dtype, v);
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == CK_MMA) tc::tmem_dealloc(tmem, C::TMEM_COLS);
  ovl_leave();
  pdl_launch_dependents();
}

// ---- host side ---------------------------------------------------------------

template <typename T, int D, int B, bool P16, bool OVL>
cudaError_t launch_chunked_p(const CUtensorMap &qmap, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, const ChunkedParams &p,
                             cudaStream_t stream) {
  using C = ChunkCfg<D>;
  auto kern = chunked_kernel<T, D, B, P16, OVL>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // every (sequence, KV head, pair of query tiles) of the longest query
  // range; or, when that is smaller and there are at most CK_SCAN_MAX
  // sequences, only the units that exist (compact), bounded by
  // S + ceil(tokens / 2 tiles) pairs per KV head (a sequence of n > 0 queries
  // has ceil(ceil(n / TQ) / 2) <= n / (2 TQ) + 1 pairs; an invalid one keeps one)
  ChunkedParams pc = p;
  long long units = (long long)p.num_qpairs * p.num_seqs * p.num_kv_heads;
  const long long bound =
      ((long long)p.num_seqs + (p.num_tokens + 2LL * p.tile_tokens - 1) / (2LL * p.tile_tokens)) *
      p.num_kv_heads;
  pc.compact = p.num_seqs <= CK_SCAN_MAX && bound < units ? 1 : 0;
  if (pc.compact) units = bound;
  if (units <= 0) return cudaSuccess;
  constexpr int NT = ck_threads(P16 && std::is_same<T, __nv_bfloat16>::value);
  return launch_pdl(kern, dim3((unsigned)units), dim3(NT), (size_t)C::SMEM, stream, qmap,
                    kmap, vmap, pc);
}

template <typename T, int D, int B>
cudaError_t launch_chunked_cfg(const CUtensorMap &qmap, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, const ChunkedParams &p,
                               cudaStream_t stream) {
  if (p.ovl_done)   // beside a running decode pass (mixed batch)
    return p.p_format == PKV_P_F16
               ? launch_chunked_p<T, D, B, true, true>(qmap, kmap, vmap, p, stream)
               : launch_chunked_p<T, D, B, false, true>(qmap, kmap, vmap, p, stream);
  return p.p_format == PKV_P_F16
             ? launch_chunked_p<T, D, B, true, false>(qmap, kmap, vmap, p, stream)
             : launch_chunked_p<T, D, B, false, false>(qmap, kmap, vmap, p, stream);
}

template <typename T, int D>
cudaError_t launch_chunked_d(const CUtensorMap &qmap, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, const ChunkedParams &p, int block_size,
                             cudaStream_t stream) {
  switch (block_size) {
    case 8: return launch_chunked_cfg<T, D, 8>(qmap, kmap, vmap, p, stream);
    case 16: return launch_chunked_cfg<T, D, 16>(qmap, kmap, vmap, p, stream);
    case 32: return launch_chunked_cfg<T, D, 32>(qmap, kmap, vmap, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_chunked_t(const CUtensorMap &qmap, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, const ChunkedParams &p, int head_dim,
                             int block_size, cudaStream_t stream) {
  if (head_dim == 64) return launch_chunked_d<T, 64>(qmap, kmap, vmap, p, block_size, stream);
  if (head_dim == 128) return launch_chunked_d<T, 128>(qmap, kmap, vmap, p, block_size, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
