// Multi-query paged attention on the fifth-generation tensor cores: chunked
// prefill (a piece of a long prompt processed in one pass, its queries
// attending causally to the sequence's earlier tokens and to each other) and
// decode tokens in the same batch ("Paging the KV Cache Like an OS",
// continuous batching and chunked prefill).
//
// One CTA = one work unit (sequence s, KV head h, query tile i).  A query tile
// is 128 rows: TQ = 128 / G consecutive query tokens of the sequence times the
// G query heads that share KV head h (row r = token r / G, head r % G).  The
// CTA walks the sequence's block table in KV tiles of 128 tokens:
//
//   S   = Q K^T      tcgen05.mma (A and B from shared memory), M = 128 rows,
//                    N = 128 keys, K = head_dim, into TMEM; two S buffers, so
//                    the tensor core computes the next S while the current
//                    one is softmaxed
//   P   = exp2(S * scale * log2 e - m)   per row, causal mask on diagonal tiles,
//                    written back to TMEM as 16-bit hi and lo parts (P = hi +
//                    lo to about 2^-16 relative)
//   O  += P V        tcgen05.mma with A (P hi, then P lo) from TMEM and V from
//                    shared memory, M = 128, N = head_dim, K = 128 keys
//
// with an online softmax whose running maximum is only raised when a score
// exceeds it by more than 2^8 (the accumulator in TMEM is then rescaled), and
// the normalisation by the running sum in the epilogue.
//
// Warp roles (320 threads): warps 0-7 are two softmax warpgroups; thread t of
// warpgroup wg owns query row t % 128 (TMEM lane) and key columns wg*64 ..
// wg*64+63 of every tile, the two threads of a row agreeing on its maximum
// through shared memory once per tile.  Warp 8 issues the TMA loads (Q once;
// K and V tiles through three-stage rings, one box per 16 tokens of a block
// and 64 dims, the block-table entries fetched a group of 32 ahead).  Warp 9
// allocates TMEM and issues the MMAs (one lane).  All hand-offs are
// mbarriers; every wait is bounded and a timeout sets PKV_FLAG_TIMEOUT, after
// which each role stops issuing and drains what it has in flight before the
// CTA frees its TMEM and exits.
//
// Shared memory (head_dim 128): Q 32 KiB, K and V 3 x 32 KiB each, in the
// 128-byte swizzled layout (rows of 64 elements); one CTA per SM.  TMEM
// columns: S buffers 0 and 128, O 256, P hi 384, P lo 448.
#pragma once

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_launch.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int CK_ROWS = 128;     // query rows per tile (MMA M)
constexpr int CK_BN = 128;       // keys per KV tile
constexpr int CK_THREADS = 320;
constexpr int CK_PRODUCER = 8;   // warp ids
constexpr int CK_MMA = 9;
constexpr int CK_NST = 3;        // K / V ring stages
constexpr float CK_SLACK = 8.0f; // lazy rescale threshold (log2 domain)

template <int D>
struct ChunkCfg {
  static constexpr int NH = D / 64;            // 64-element column halves
  static constexpr int HALF = CK_ROWS * 128;   // one half-tile: 128 rows x 128 bytes
  static constexpr int Q_BYTES = NH * HALF;
  static constexpr int KV_BYTES = NH * HALF;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + CK_NST * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + CK_NST * KV_BYTES;
  static constexpr int NBAR = 24;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  // row-max exchange between the two softmax warpgroups: [2 tiles][2][128]
  static constexpr int OFF_RED = OFF_TMEM + 16;
  static constexpr int SMEM = OFF_RED + 2 * 2 * CK_ROWS * 4;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 256;
  static constexpr uint32_t COL_PH = 384;
  static constexpr uint32_t COL_PL = 448;
};

// mbarrier slots
enum : int {
  CB_Q = 0,                  // Q tile landed (tx)
  CB_KF = 1,                 // K stage full [CK_NST] (tx)
  CB_KE = CB_KF + CK_NST,    // K stage free [CK_NST] (MMA commit)
  CB_VF = CB_KE + CK_NST,    // V stage full [CK_NST] (tx)
  CB_VE = CB_VF + CK_NST,    // V stage free [CK_NST] (MMA commit)
  CB_SF = CB_VE + CK_NST,    // S buffer computed [2] (MMA commit)
  CB_SE = CB_SF + 2,         // S buffer read by the softmax warps [2] (8 arrivals)
  CB_PF = CB_SE + 2,         // P written (8 arrivals)
  CB_PV = CB_PF + 1,         // P V of a tile done (MMA commit)
  CB_PAIR = CB_PV + 1,       // row-statistics exchange of warps w and w + 4 [4] (64 arrivals)
  CB_COUNT = CB_PAIR + 4,
};

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

template <typename T, int D, int B>
__global__ void __launch_bounds__(CK_THREADS, 1)
    chunked_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const ChunkedParams p) {
  using C = ChunkCfg<D>;
  static_assert(CB_COUNT <= C::NBAR, "mbarrier slots");
  constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int BT = B < 16 ? B : 16;          // tokens per TMA box
  static_assert(BT * 128 % 1024 == 0, "boxes land on 1 KiB boundaries (128-byte swizzle atoms)");
  constexpr int BLOCKS_PER_TILE = CK_BN / B;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sm = smem_raw;
  const uint32_t sb = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * (uint32_t)i; };

  // ---- the unit: the query tiles of one (sequence, KV head) are adjacent in
  // the grid, heaviest (last) tile first, so that they run at the same time
  // and read each K/V tile from L2 rather than from HBM
  int id = blockIdx.x;
  const int qt_rev = id % p.num_qtiles;
  id /= p.num_qtiles;
  const int kvh = id % p.num_kv_heads;
  const int s = id / p.num_kv_heads;

  pdl_wait_predecessors();
  const int q0 = p.query_start[s], q1 = p.query_start[s + 1];
  const int n = q1 - q0;
  int L = p.context_lens[s];
  if (q0 < 0 || n < 0 || q1 > p.num_tokens || n > p.max_query_len || L < n) {
    if (tid == 0 && qt_rev == 0 && kvh == 0) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    return;
  }
  if (L > p.max_blocks * B) {
    if (tid == 0 && qt_rev == 0 && kvh == 0) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    L = p.max_blocks * B;
    if (L < n) return;
  }
  const int TQ = p.tile_tokens;
  const int G = p.group;
  const int nq = (n + TQ - 1) / TQ;
  if (qt_rev >= nq) return;
  const int qt = nq - 1 - qt_rev;
  const int t_begin = qt * TQ;
  const int t_end = min(n, t_begin + TQ);
  const int p_max = L - n + t_end - 1;           // last query position of the tile
  const int nkv = p_max / CK_BN + 1;             // KV tiles the tile needs
  const int nb_valid = (L + B - 1) / B;

  if (sb & 1023u) {   // the swizzled tiles need a 1 KiB-aligned base
    if (tid == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
    return;
  }
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C::OFF_TMEM);
  if (tid == 0) {
    mbar_init(bar(CB_Q), 1);
    for (int i = 0; i < CK_NST; ++i) {
      mbar_init(bar(CB_KF + i), 1);
      mbar_init(bar(CB_KE + i), 1);
      mbar_init(bar(CB_VF + i), 1);
      mbar_init(bar(CB_VE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(CB_SF + i), 1);
      mbar_init(bar(CB_SE + i), 8);
    }
    mbar_init(bar(CB_PF), 8);
    mbar_init(bar(CB_PV), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(CB_PAIR + i), 64);
    fence_barrier_init();
  }
  // rows of the Q tile that no token fills (G not dividing 128) are zero
  const int q_rows = TQ * G;
  if (q_rows < CK_ROWS) {
    for (int x = tid; x < (CK_ROWS - q_rows) * 8 * C::NH; x += CK_THREADS) {
      const int h = x / ((CK_ROWS - q_rows) * 8), rem = x % ((CK_ROWS - q_rows) * 8);
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

  if (warp == CK_PRODUCER) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop: lane i holds block-table entry i of the
    // current group of 32 (TPG tiles), the next group's entries are already
    // in flight, and lane 0 issues the TMA loads.
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
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      mbar_arrive_expect_tx(bar(CB_Q), (uint32_t)(C::NH * 128 * q_rows));
      for (int h = 0; h < C::NH; ++h)
        tma_load_3d(sb + C::OFF_Q + h * C::HALF, &qmap, h * 64, kvh * G, q0 + t_begin, bar(CB_Q));
    }
    auto load_tile = [&](const CUtensorMap *map, uint32_t dst, const int (&blk)[BLOCKS_PER_TILE],
                         uint32_t full) {
#pragma unroll
      for (int b = 0; b < BLOCKS_PER_TILE; ++b)
#pragma unroll
        for (int sub = 0; sub < B / BT; ++sub)
#pragma unroll
          for (int h = 0; h < C::NH; ++h)
            tma_load_4d_keep(dst + h * C::HALF + (b * B + sub * BT) * 128, map, h * 64, kvh,
                             sub * BT, blk[b], full);
    };
    int cur = fetch(0), nxt = fetch(1);
    int issued = 0;
    for (int j = 0; j < nkv; ++j) {
      if (j > 0 && j % TPG == 0) {
        cur = nxt;
        nxt = fetch(j / TPG + 1);
      }
      int blk[BLOCKS_PER_TILE];
#pragma unroll
      for (int b = 0; b < BLOCKS_PER_TILE; ++b)
        blk[b] = __shfl_sync(FULL_MASK, cur, (j % TPG) * BLOCKS_PER_TILE + b);
      const int st = j % CK_NST;
      const uint32_t ph = (uint32_t)(j / CK_NST) & 1u;
      if (j >= CK_NST && !warp_wait(bar(CB_KE + st), ph ^ 1u)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(CB_KF + st), (uint32_t)C::KV_BYTES);
        load_tile(&kmap, sb + C::OFF_K + st * C::KV_BYTES, blk, bar(CB_KF + st));
      }
      if (j >= CK_NST && !warp_wait(bar(CB_VE + st), ph ^ 1u)) { ok = false; issued = 2 * j + 1; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(CB_VF + st), (uint32_t)C::KV_BYTES);
        load_tile(&vmap, sb + C::OFF_V + st * C::KV_BYTES, blk, bar(CB_VF + st));
      }
      issued = 2 * j + 2;
    }
    // drain: every load issued has landed before the CTA may exit (loads
    // older than the last ring's worth were consumed, so they have landed)
    if (lane == 0) {
      mbar_wait_bounded(bar(CB_Q), 0);
      for (int x = issued - 1; x >= 0 && x >= issued - 2 * CK_NST; --x) {
        const int j = x >> 1, st = j % CK_NST;
        mbar_wait_bounded(bar(((x & 1) ? CB_VF : CB_KF) + st), (uint32_t)(j / CK_NST) & 1u);
      }
      if (!ok) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
    }
  } else if (warp == CK_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // Per tile j: S(j+1) = Q K(j+1)^T first (the tensor core computes it while
    // the softmax warps work on S(j)), then O += P(j) V(j).
    constexpr uint32_t ID_S = tc::idesc_f16(BF16, CK_ROWS, CK_BN, false);
    constexpr uint32_t ID_PV = tc::idesc_f16(BF16, CK_ROWS, D, true);
    const uint32_t tO = tmem + C::COL_O;
    int pv_issued = 0, s_issued = 0;
    auto issue_s = [&](int j) -> bool {
      const int st = j % CK_NST, b = j & 1;
      if (!warp_wait(bar(CB_KF + st), (uint32_t)(j / CK_NST) & 1u)) return false;
      if (j >= 2 && !warp_wait(bar(CB_SE + b), (uint32_t)((j >> 1) - 1) & 1u)) return false;
      tc::fence_after_sync();
      if (lane == 0) {
        const uint32_t qa = sb + C::OFF_Q, ka = sb + C::OFF_K + st * C::KV_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)(k >> 2) * C::HALF + (uint32_t)(k & 3) * 32u;
          tc::mma_f16_ss(tmem + (uint32_t)b * 128u, tc::sdesc_sw128(qa + off, 16, 1024),
                         tc::sdesc_sw128(ka + off, 16, 1024), ID_S, k > 0 ? 1u : 0u);
        }
        tc::commit(bar(CB_SF + b));
        tc::commit(bar(CB_KE + st));
      }
      __syncwarp();
      s_issued = j + 1;
      return true;
    };
    ok = warp_wait(bar(CB_Q), 0) && issue_s(0);
    const int tail_tile = (L % CK_BN) ? (L - 1) / CK_BN : -1;
    for (int j = 0; j < nkv && ok; ++j) {
      if (j + 1 < nkv && !issue_s(j + 1)) { ok = false; break; }
      const int st = j % CK_NST;
      if (!warp_wait(bar(CB_PF), (uint32_t)j & 1u) ||
          !warp_wait(bar(CB_VF + st), (uint32_t)(j / CK_NST) & 1u)) {
        ok = false;
        break;
      }
      if (j == tail_tile) {
        // V rows past the sequence hold whatever the pool holds there; their
        // probabilities are exactly zero, but 0 * NaN is not, so zero them
        const int z0 = L - j * CK_BN;
        unsigned char *vs = sm + C::OFF_V + st * C::KV_BYTES;
        for (int x = lane; x < (CK_BN - z0) * 8 * C::NH; x += 32) {
          const int h = x / ((CK_BN - z0) * 8), rem = x % ((CK_BN - z0) * 8);
          *reinterpret_cast<uint4 *>(vs + h * C::HALF + (z0 + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc::fence_after_sync();
      if (lane == 0) {
        const uint32_t va = sb + C::OFF_V + st * C::KV_BYTES;
#pragma unroll
        for (int k = 0; k < CK_BN / 16; ++k) {
          const uint64_t bv = tc::sdesc_sw128(va + (uint32_t)k * 2048u, C::HALF, 1024);
          tc::mma_f16_ts(tO, tmem + C::COL_PH + 8u * k, bv, ID_PV, (j > 0 || k > 0) ? 1u : 0u);
          tc::mma_f16_ts(tO, tmem + C::COL_PL + 8u * k, bv, ID_PV, 1u);
        }
        tc::commit(bar(CB_PV));
        tc::commit(bar(CB_VE + st));
      }
      __syncwarp();
      pv_issued = j + 1;
    }
    // drain: the MMAs issued have completed before TMEM is freed
    if (pv_issued > 0) warp_wait(bar(CB_PV), (uint32_t)(pv_issued - 1) & 1u);
    if (s_issued > 0)
      warp_wait(bar(CB_SF + ((s_issued - 1) & 1)), (uint32_t)((s_issued - 1) >> 1) & 1u);
    if (!ok && lane == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
  } else {
    // ------------------------------------------------------------ softmax
    constexpr int HC = CK_BN / 2;             // key columns per thread
    constexpr int HD = D / 2;                 // output columns per thread
    const int wg = warp >> 2;
    const int r = tid & (CK_ROWS - 1);        // query row = TMEM lane
    const int tl = r / G, g = r % G;
    const int tok = t_begin + tl;
    const bool valid = tl < TQ && tok < t_end;
    const int p_row = valid ? (L - n + tok) : p_max;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t pair = bar(CB_PAIR + (warp & 3));
    float *red = reinterpret_cast<float *>(sm + C::OFF_RED);   // [2][2][128]
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    uint32_t sr[HC];
    int j = 0;
    for (; j < nkv; ++j) {
      const int b = j & 1;
      if (!warp_wait(bar(CB_SF + b), (uint32_t)(j >> 1) & 1u)) { ok = false; break; }
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < HC / 32; ++c)
        tc::ld_32x32b_x32(tmem + lane_base + (uint32_t)(b * 128 + wg * HC + c * 32), sr + 32 * c);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(CB_SE + b));

      const int lim = p_row - j * CK_BN - wg * HC;   // own columns 0..lim are visible
      if (lim < HC - 1) {
#pragma unroll
        for (int c = 0; c < HC; ++c)
          if (c > lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < HC; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sr[c]));
      float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      float *rb = red + (j & 1) * 2 * CK_ROWS;
      rb[wg * CK_ROWS + r] = mx;
      mbar_arrive(pair);
      if (!warp_wait(pair, (uint32_t)j & 1u)) { ok = false; break; }
      mx = fmaxf(mx, rb[(wg ^ 1) * CK_ROWS + r]);
      // running maximum in the exp2 domain, raised lazily
      const float mnew = fmaxf(m, mx * sl2);
      const bool resc = mnew > m + CK_SLACK;
      float alpha = 1.f;
      if (resc) {
        alpha = fast_exp2(m - mnew);
        m = mnew;
      }
      // P = exp2(s * scale * log2 e - m) as hi + lo 16-bit pairs
      const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m, -m);
      float2 lsum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t hiw[HC / 2], low[HC / 2];
#pragma unroll
      for (int e = 0; e < HC / 2; ++e) {
        const float2 x = fma2(make_float2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                              sl2x2, negm);
        const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        lsum[e & 1] = make_float2(lsum[e & 1].x + pe.x, lsum[e & 1].y + pe.y);
        hiw[e] = Mma<T>::pack(pe.x, pe.y);
        const float2 hf = Widen<T>::pair(hiw[e]);
        low[e] = Mma<T>::pack(pe.x - hf.x, pe.y - hf.y);
      }
      l = l * alpha + ((lsum[0].x + lsum[0].y) + (lsum[1].x + lsum[1].y));
      // P in TMEM and O are free once the previous tile's P V is done
      if (j > 0 && !warp_wait(bar(CB_PV), (uint32_t)(j - 1) & 1u)) { ok = false; break; }
      tc::fence_after_sync();
      if (j > 0 && __any_sync(FULL_MASK, resc)) {
        uint32_t o[32];
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          const uint32_t ta = tmem + lane_base + C::COL_O + (uint32_t)(wg * HD + c * 32);
          tc::ld_32x32b_x32(ta, o);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::st_32x32b_x32(ta, o);
        }
      }
      tc::st_32x32b_x32(tmem + lane_base + C::COL_PH + (uint32_t)(wg * (HC / 2)), hiw);
      tc::st_32x32b_x32(tmem + lane_base + C::COL_PL + (uint32_t)(wg * (HC / 2)), low);
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(CB_PF));
    }
    // ---- epilogue: O / l, the row's sum being the two threads' partial sums
    if (ok) {
      float *rb = red + (j & 1) * 2 * CK_ROWS;
      rb[wg * CK_ROWS + r] = l;
      mbar_arrive(pair);
      ok = warp_wait(pair, (uint32_t)j & 1u);
      if (ok) l += rb[(wg ^ 1) * CK_ROWS + r];
    }
    if (ok && warp_wait(bar(CB_PV), (uint32_t)(nkv - 1) & 1u)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t row = ((size_t)(q0 + (valid ? tok : 0)) * p.num_q_heads + (size_t)kvh * G + g) *
                             (size_t)D + (size_t)(wg * HD);
      uint32_t o[32];
      float v[32];
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        tc::ld_32x32b_x32(tmem + lane_base + C::COL_O + (uint32_t)(wg * HD + c * 32), o);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
        if (valid) store_row32(p.out, row + (size_t)c * 32, p.out_dtype, v);
      }
    } else {
      ok = false;
    }
    if (!ok && lane == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == CK_MMA) tc::tmem_dealloc(tmem, C::TMEM_COLS);
  pdl_launch_dependents();
}

// ---- host side ---------------------------------------------------------------

template <typename T, int D, int B>
cudaError_t launch_chunked_cfg(const CUtensorMap &qmap, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, const ChunkedParams &p,
                               cudaStream_t stream) {
  using C = ChunkCfg<D>;
  auto kern = chunked_kernel<T, D, B>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const long long units = (long long)p.num_qtiles * p.num_seqs * p.num_kv_heads;
  if (units <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3((unsigned)units), dim3(CK_THREADS), (size_t)C::SMEM, stream, qmap,
                    kmap, vmap, p);
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
