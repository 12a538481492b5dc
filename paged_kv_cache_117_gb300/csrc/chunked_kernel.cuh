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
//   S   = Q K^T      tcgen05.mma, M = 128 rows, N = 128 keys, K = head_dim,
//                    accumulated in TMEM (two S buffers, so the tensor core
//                    computes the next S while the current one is softmaxed)
//   P   = exp2(S * scale * log2 e - m)   per row, causal mask on diagonal tiles
//   O  += P V        tcgen05.mma, M = 128, N = head_dim, K = 128 keys; P is
//                    split into bf16/f16 hi and lo parts (P = hi + lo to about
//                    2^-16 relative) so the product keeps fp32-like accuracy
//
// with an online softmax whose running maximum is only raised when a score
// exceeds it by more than 2^8 (the accumulator in TMEM is then rescaled), and
// the normalisation by the running sum in the epilogue.
//
// Warp roles (192 threads): warps 0-3 own TMEM lanes 0-127, one query row per
// thread (softmax, rescale, epilogue); warp 4 issues the TMA loads (Q once;
// K and V tiles through two-stage rings, one box per 16 tokens of a block
// and 64 dims); warp 5 allocates TMEM and issues the MMAs (one lane).  All
// hand-offs are mbarriers; every wait is bounded and a timeout sets
// PKV_FLAG_TIMEOUT, after which each role stops issuing and drains what it
// has in flight before the CTA frees its TMEM and exits.
//
// Shared memory (head_dim 128): Q 32 KiB, K 2 x 32 KiB, V 2 x 32 KiB, P hi
// and lo 32 KiB each, all in the 128-byte swizzled layout (rows of 64
// elements); one CTA per SM.  TMEM: S buffers at columns 0 and 128, O at 256.
#pragma once

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_launch.h"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int CK_ROWS = 128;     // query rows per tile (MMA M)
constexpr int CK_BN = 128;       // keys per KV tile
constexpr int CK_THREADS = 192;
constexpr float CK_SLACK = 8.0f; // lazy rescale threshold (log2 domain)

template <int D>
struct ChunkCfg {
  static constexpr int NH = D / 64;            // 64-element column halves
  static constexpr int HALF = CK_ROWS * 128;   // one half-tile: 128 rows x 128 bytes
  static constexpr int Q_BYTES = NH * HALF;
  static constexpr int KV_BYTES = NH * HALF;
  static constexpr int P_BYTES = 2 * HALF;     // 128 keys
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr int OFF_PH = OFF_V + 2 * KV_BYTES;
  static constexpr int OFF_PL = OFF_PH + P_BYTES;
  static constexpr int OFF_BAR = OFF_PL + P_BYTES;
  static constexpr int NBAR = 16;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEM + 16 + 1024;   // + room to align the base to 1 KiB
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 256;
};

// mbarrier slots
enum : int {
  CB_Q = 0,        // Q tile landed (tx)
  CB_KF = 1,       // K stage full [2] (tx)
  CB_KE = 3,       // K stage free [2] (MMA commit)
  CB_VF = 5,       // V stage full [2] (tx)
  CB_VE = 7,       // V stage free [2] (MMA commit)
  CB_SF = 9,       // S buffer computed [2] (MMA commit)
  CB_SE = 11,      // S buffer read by the softmax warps [2] (4 arrivals)
  CB_PF = 13,      // P written (4 arrivals)
  CB_PV = 14,      // P V of a tile done (MMA commit)
};

// Every lane of the warp waits; the result is the same on all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait_bounded(bar, parity);
  return __all_sync(FULL_MASK, ok);
}

template <typename T>
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
  constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int BT = B < 16 ? B : 16;          // tokens per TMA box
  static_assert(BT * 128 % 1024 == 0, "boxes land on 1 KiB boundaries (128-byte swizzle atoms)");
  constexpr int BLOCKS_PER_TILE = CK_BN / B;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * (uint32_t)i; };

  // ---- the unit: heaviest query tiles first (the last tile of a sequence
  // sees the most keys), then sequence, then KV head
  int id = blockIdx.x;
  const int kvh = id % p.num_kv_heads;
  id /= p.num_kv_heads;
  const int s = id % p.num_seqs;
  const int qt_rev = id / p.num_seqs;

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

  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C::OFF_TMEM);
  if (tid == 0) {
    mbar_init(bar(CB_Q), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(CB_KF + i), 1);
      mbar_init(bar(CB_KE + i), 1);
      mbar_init(bar(CB_VF + i), 1);
      mbar_init(bar(CB_VE + i), 1);
      mbar_init(bar(CB_SF + i), 1);
      mbar_init(bar(CB_SE + i), 4);
    }
    mbar_init(bar(CB_PF), 4);
    mbar_init(bar(CB_PV), 1);
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
  if (warp == 5) {
    tc::tmem_alloc(smem_addr(tslot), C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  bool ok = true;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      mbar_arrive_expect_tx(bar(CB_Q), (uint32_t)(C::NH * 128 * q_rows));
      for (int h = 0; h < C::NH; ++h)
        tma_load_3d(sb + C::OFF_Q + h * C::HALF, &qmap, h * 64, kvh * G, q0 + t_begin, bar(CB_Q));
      const int32_t *tbl = p.block_tables + (size_t)s * p.max_blocks;
      auto load_tile = [&](const CUtensorMap *map, uint32_t dst, int j, uint32_t full) {
        for (int b = 0; b < BLOCKS_PER_TILE; ++b) {
          const int lb = j * BLOCKS_PER_TILE + b;
          int blk = p.num_blocks;                  // past the pool: TMA fills zeros
          if (lb < nb_valid) {
            const int x = tbl[lb];
            if (x < 0 || x >= p.num_blocks) atomicOr(p.flags, PKV_FLAG_BLOCK_RANGE);
            else blk = x;
          }
#pragma unroll
          for (int sub = 0; sub < B / BT; ++sub)
#pragma unroll
            for (int h = 0; h < C::NH; ++h)
              tma_load_4d_keep(dst + h * C::HALF + (b * B + sub * BT) * 128, map, h * 64, kvh,
                               sub * BT, blk, full);
        }
      };
      int issued = 0;
      for (int j = 0; j < nkv && ok; ++j) {
        const int st = j & 1;
        const uint32_t ph = (uint32_t)(j >> 1) & 1u;
        if (j >= 2 && !mbar_wait_bounded(bar(CB_KE + st), ph ^ 1u)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(CB_KF + st), (uint32_t)C::KV_BYTES);
        load_tile(&kmap, sb + C::OFF_K + st * C::KV_BYTES, j, bar(CB_KF + st));
        if (j >= 2 && !mbar_wait_bounded(bar(CB_VE + st), ph ^ 1u)) { ok = false; issued = 2 * j + 1; break; }
        mbar_arrive_expect_tx(bar(CB_VF + st), (uint32_t)C::KV_BYTES);
        load_tile(&vmap, sb + C::OFF_V + st * C::KV_BYTES, j, bar(CB_VF + st));
        issued = 2 * j + 2;
      }
      // drain: every load issued has landed before the CTA may exit
      mbar_wait_bounded(bar(CB_Q), 0);
      for (int x = issued - 1; x >= 0 && x >= issued - 4; --x) {
        const int j = x >> 1, st = j & 1;
        mbar_wait_bounded(bar(((x & 1) ? CB_VF : CB_KF) + st), (uint32_t)(j >> 1) & 1u);
      }
      if (!ok) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t ID_S = tc::idesc_f16(BF16, CK_ROWS, CK_BN, false);
    constexpr uint32_t ID_PV = tc::idesc_f16(BF16, CK_ROWS, D, true);
    const uint32_t tO = tmem + C::COL_O;
    int pv_issued = 0, s_issued = 0;
    auto issue_s = [&](int j) -> bool {
      const int st = j & 1;
      if (!warp_wait(bar(CB_KF + st), (uint32_t)(j >> 1) & 1u)) return false;
      if (j >= 2 && !warp_wait(bar(CB_SE + st), (uint32_t)((j >> 1) - 1) & 1u)) return false;
      tc::fence_after_sync();
      if (lane == 0) {
        const uint32_t qa = sb + C::OFF_Q, ka = sb + C::OFF_K + st * C::KV_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)(k >> 2) * C::HALF + (uint32_t)(k & 3) * 32u;
          tc::mma_f16_ss(tmem + (uint32_t)st * 128u, tc::sdesc_sw128(qa + off, 16, 1024),
                         tc::sdesc_sw128(ka + off, 16, 1024), ID_S, k > 0 ? 1u : 0u);
        }
        tc::commit(bar(CB_SF + st));
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
      const int st = j & 1;
      if (!warp_wait(bar(CB_PF), (uint32_t)j & 1u) ||
          !warp_wait(bar(CB_VF + st), (uint32_t)(j >> 1) & 1u)) { ok = false; break; }
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
          const uint32_t poff = (uint32_t)(k >> 2) * C::HALF + (uint32_t)(k & 3) * 32u;
          const uint64_t bv = tc::sdesc_sw128(va + (uint32_t)k * 2048u, C::HALF, 1024);
          tc::mma_f16_ss(tO, tc::sdesc_sw128(sb + C::OFF_PH + poff, 16, 1024), bv, ID_PV,
                         (j > 0 || k > 0) ? 1u : 0u);
          tc::mma_f16_ss(tO, tc::sdesc_sw128(sb + C::OFF_PL + poff, 16, 1024), bv, ID_PV, 1u);
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
    const int r = tid;                        // query row = TMEM lane
    const int tl = r / G, g = r % G;
    const int tok = t_begin + tl;
    const bool valid = tl < TQ && tok < t_end;
    const int p_row = valid ? (L - n + tok) : p_max;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    uint32_t sr[CK_BN];
    for (int j = 0; j < nkv; ++j) {
      const int b = j & 1;
      if (!warp_wait(bar(CB_SF + b), (uint32_t)(j >> 1) & 1u)) { ok = false; break; }
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < CK_BN / 32; ++c)
        tc::ld_32x32b_x32(tmem + lane_base + (uint32_t)b * 128u + (uint32_t)c * 32u, sr + 32 * c);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(CB_SE + b));

      const int lim = p_row - j * CK_BN;      // columns 0..lim are visible
      float mx = -INFINITY;
      if (lim >= CK_BN - 1) {
#pragma unroll
        for (int c = 0; c < CK_BN; ++c) {
          const float v = __uint_as_float(sr[c]) * sl2;
          sr[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      } else {
#pragma unroll
        for (int c = 0; c < CK_BN; ++c) {
          const float v = c <= lim ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
          sr[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      }
      const float mnew = fmaxf(m, mx);
      const bool resc = mnew > m + CK_SLACK;
      // the P buffers and O are free once the previous tile's P V is done
      if (j > 0 && !warp_wait(bar(CB_PV), (uint32_t)(j - 1) & 1u)) { ok = false; break; }
      tc::fence_after_sync();
      float alpha = 1.f;
      if (resc) {
        alpha = fast_exp2(m - mnew);
        m = mnew;
      }
      if (j > 0 && __any_sync(FULL_MASK, resc)) {
        uint32_t o[32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint32_t ta = tmem + lane_base + C::COL_O + (uint32_t)c * 32u;
          tc::ld_32x32b_x32(ta, o);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::st_32x32b_x32(ta, o);
        }
        tc::wait_st();
      }
      l *= alpha;
#pragma unroll
      for (int c8 = 0; c8 < CK_BN / 8; ++c8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = fast_exp2(__uint_as_float(sr[8 * c8 + 2 * e]) - m);
          const float bb = fast_exp2(__uint_as_float(sr[8 * c8 + 2 * e + 1]) - m);
          l += a + bb;
          hi[e] = Mma<T>::pack(a, bb);
          const float2 hf = Widen<T>::pair(hi[e]);
          lo[e] = Mma<T>::pack(a - hf.x, bb - hf.y);
        }
        const uint32_t off = (uint32_t)(c8 >> 3) * C::HALF + tc::sw128_offset(r, c8 & 7);
        *reinterpret_cast<uint4 *>(sm + C::OFF_PH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(sm + C::OFF_PL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(CB_PF));
    }
    // ---- epilogue: O / l
    if (ok && warp_wait(bar(CB_PV), (uint32_t)(nkv - 1) & 1u)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t row = ((size_t)(q0 + (valid ? tok : 0)) * p.num_q_heads + (size_t)kvh * G + g) *
                         (size_t)D;
      uint32_t o[32];
      float v[32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        tc::ld_32x32b_x32(tmem + lane_base + C::COL_O + (uint32_t)c * 32u, o);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
        if (valid) store_row32<T>(p.out, row + (size_t)c * 32, p.out_dtype, v);
      }
    } else {
      ok = false;
    }
    if (!ok && lane == 0) atomicOr(p.flags, PKV_FLAG_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) tc::tmem_dealloc(tmem, C::TMEM_COLS);
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
