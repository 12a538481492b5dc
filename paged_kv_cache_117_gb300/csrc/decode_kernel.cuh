// Paged decode attention for sm_103a: one CTA per (sequence, KV head, query
// head chunk, context partition).
//
// What is computed (PagedAttention, "PagedAttention and vLLM: Paging the KV
// Cache Like an OS", Step 5; "PagedAttention: Virtual Memory for the KV
// Cache", block-wise attention equation): for each query head of the GQA
// group, walk the sequence's block table, score the query against every valid
// key of every block, run one softmax over all valid positions, and weight the
// values.  Each gathered K/V block is read once from HBM for the whole query
// group.
//
// How, on GB300:
//  * Each warp streams its own share of the partition's blocks (block
//    jb + w, jb + w + NW, ...) through a private ring of STAGES shared-memory
//    stages.  One lane issues two 4-D TMA tile loads per block (K and V tile
//    [block_size, head_dim] of one KV head; the pool is [N, B, Hkv, D], so
//    the tile is block_size rows of head_dim*2 bytes at a stride of
//    Hkv*head_dim*2 bytes) completing on the stage's mbarrier.  No cross-warp
//    synchronisation is needed inside the loop.
//  * A block is processed in chunks of up to 16 tokens.  Half-warp h takes
//    tokens h*CH/2 .. of the chunk; lane li of the half owns head_dim/16
//    consecutive dims.  Q.K partial dot products use the packed fp32x2 FMA;
//    the (token, head) partials are summed across the 16 lanes by a
//    reduce-scatter butterfly (about one shuffle per partial instead of four).
//  * Online softmax in fp32 in the exp2 domain (q is pre-scaled by
//    scale*log2 e).  Running (max, sum) per head, output accumulators per
//    (head, owned dims); slots at or past the context length are masked
//    before the max and skipped in P.V, so whatever bytes they hold never
//    reach the result.
//  * At the end the warps' states are merged in shared memory (log-sum-exp
//    rescale).  With one partition the CTA writes out = O / L; otherwise it
//    writes the partition's (M, L, O) record and decode_merge_kernel combines
//    the records of a sequence: o = sum_p e^(M_p - M) O_p / sum_p e^(M_p - M) L_p.
//    Normalising each partition and adding the results would be wrong
//    ("PagedAttention" (tensortonic), section 5), so records stay
//    unnormalised.
#pragma once

#include <math.h>

#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

constexpr int ilog2_c(int v) { return v <= 1 ? 0 : 1 + ilog2_c(v >> 1); }
constexpr int max_c(int a, int b) { return a > b ? a : b; }
constexpr int min_c(int a, int b) { return a < b ? a : b; }
constexpr int round_up_c(int v, int a) { return (v + a - 1) / a * a; }

template <typename T, int D, int B, int GT, int NW, int STAGES>
struct DecodeCfg {
  static constexpr int CH = min_c(B, 16);        // tokens per compute chunk
  static constexpr int NCH = B / CH;             // chunks per block
  static constexpr int HT = CH / 2;              // tokens per half-warp per chunk
  static constexpr int DPL = D / 16;             // dims owned by a lane
  static constexpr int WPL = DPL / 2;            // 32-bit words per lane row slice
  static constexpr int TILE_ELEMS = B * D;
  static constexpr int TILE_BYTES = TILE_ELEMS * (int)sizeof(T);
  static constexpr int V = HT * GT;              // partial scores per lane per chunk
  static constexpr int LPG = 16 / GT;            // lanes per head within a half-warp
  static constexpr int SCAT = V >= 16 ? 4 : ilog2_c(V);
  static constexpr int DUP_BITS = 4 - SCAT;      // lanes holding copies of one sum
  static constexpr int R = V >= 16 ? V / 16 : 1; // sums owned per lane
  // shared memory (bytes)
  static constexpr int STAGES_BYTES = NW * STAGES * 2 * TILE_BYTES;
  static constexpr int MERGE_BYTES = NW * GT * (D + 2) * 4;
  static constexpr int BIG_BYTES = round_up_c(max_c(STAGES_BYTES, MERGE_BYTES), 128);
  static constexpr int P_FLOATS = NW * 2 * HT * GT;
  static constexpr int A_FLOATS = NW * GT;
  static constexpr int SMALL_BYTES = round_up_c((P_FLOATS + A_FLOATS) * 4, 16);
  static constexpr int BAR_BYTES = NW * STAGES * 8;
  static constexpr int SMEM_BYTES = 1024 + BIG_BYTES + SMALL_BYTES + BAR_BYTES + 16;

  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(B == 4 || B == 8 || B == 16 || B == 32, "block_size");
  static_assert(GT == 1 || GT == 2 || GT == 4 || GT == 8, "query head chunk");
  static_assert(R <= HT, "a lane's sums belong to one head");
};

// Sum v[] over the 16 lanes of each half-warp.  Afterwards lane li holds, in
// v[0 .. R-1], the full sums of the original entries
// [(li >> DUP_BITS) * R, ... + R).  Each exchange step sends half of the live
// entries to the partner lane and keeps the other half.
template <int V>
__device__ __forceinline__ void half_reduce_scatter(float (&v)[V], int li) {
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int off = 8 >> step;
    const int n = (V >> step) > 1 ? (V >> step) : 1;
    if (n > 1) {
      const int h = n >> 1;
      const bool upper = (li & off) != 0;
#pragma unroll
      for (int k = 0; k < h; ++k) {
        const float send = upper ? v[k] : v[k + h];
        const float keep = upper ? v[k + h] : v[k];
        v[k] = keep + __shfl_xor_sync(FULL_MASK, send, off);
      }
    } else {
      v[0] += __shfl_xor_sync(FULL_MASK, v[0], off);
    }
  }
}

template <int W>
__device__ __forceinline__ void load_words(const void *p, uint32_t (&w)[W]);
template <>
__device__ __forceinline__ void load_words<4>(const void *p, uint32_t (&w)[4]) {
  const uint4 x = *reinterpret_cast<const uint4 *>(p);
  w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
}
template <>
__device__ __forceinline__ void load_words<2>(const void *p, uint32_t (&w)[2]) {
  const uint2 x = *reinterpret_cast<const uint2 *>(p);
  w[0] = x.x; w[1] = x.y;
}

template <int W>
__device__ __forceinline__ void ldg_words(const void *p, uint32_t (&w)[W]);
template <>
__device__ __forceinline__ void ldg_words<4>(const void *p, uint32_t (&w)[4]) {
  const uint4 x = __ldg(reinterpret_cast<const uint4 *>(p));
  w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
}
template <>
__device__ __forceinline__ void ldg_words<2>(const void *p, uint32_t (&w)[2]) {
  const uint2 x = __ldg(reinterpret_cast<const uint2 *>(p));
  w[0] = x.x; w[1] = x.y;
}

template <typename T, int D, int B, int GT, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using C = DecodeCfg<T, D, B, GT, NW, STAGES>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  T *stages = reinterpret_cast<T *>(smem);
  float *p_s = reinterpret_cast<float *>(smem + C::BIG_BYTES);
  float *a_s = p_s + C::P_FLOATS;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BIG_BYTES + C::SMALL_BYTES);
  volatile int *s_abort = reinterpret_cast<volatile int *>(bars + NW * STAGES);

  const int part = blockIdx.x;
  const int kvh = blockIdx.y / p.num_gchunks;
  const int gc = blockIdx.y - kvh * p.num_gchunks;
  const int s = blockIdx.z;
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5, half = lane >> 4, li = lane & 15;

  int L = __ldg(p.context_lens + s);
  const int cap = p.max_blocks * B;
  if (L < 0 || L > cap) {
    if (tid == 0 && part == 0 && blockIdx.y == 0) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    L = L < 0 ? 0 : cap;
  }
  const int nb = (L + B - 1) / B;
  const int g0 = gc * GT;
  const int gcount = min(GT, p.group - g0);
  const int hq0 = kvh * p.group + g0;
  const size_t out_base = ((size_t)s * p.num_q_heads + hq0) * D;
  if (nb == 0) {  // nothing to attend to: zeros
    if (part == 0)
      for (int idx = tid; idx < gcount * D; idx += NW * 32)
        store_out(p.out, out_base + idx, p.out_dtype, 0.f);
    return;
  }
  const int jb = part * p.part_blocks;
  if (jb >= nb) return;
  const int je = min(nb, jb + p.part_blocks);
  const int nparts = (nb + p.part_blocks - 1) / p.part_blocks;

  if (tid == 0) {
#pragma unroll 1
    for (int i = 0; i < NW * STAGES; ++i) mbar_init(smem_addr(bars + i), 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (tid == 32 || (NW == 1 && tid == 0)) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncthreads();

  // ---- this warp's blocks and its slice of the block table ----------------
  const int j0 = jb + w;
  const int n_w = j0 < je ? (je - j0 + NW - 1) / NW : 0;
  const int32_t *trow = p.block_tables + (size_t)s * p.max_blocks;
  int kbase = 0;
  int tbl = lane < n_w ? __ldg(trow + j0 + lane * NW) : 0;
  T *wst = stages + (size_t)w * STAGES * 2 * C::TILE_ELEMS;
  const uint32_t bar0 = smem_addr(bars + w * STAGES);
  const uint64_t pol = l2_policy_evict_first();

  auto issue = [&](int i_load, int stage) {
    if (i_load - kbase >= 32) {
      kbase += 32;
      tbl = kbase + lane < n_w ? __ldg(trow + j0 + (kbase + lane) * NW) : 0;
    }
    const int pb = __shfl_sync(FULL_MASK, tbl, i_load - kbase);
    if (lane == 0) {
      if ((unsigned)pb >= (unsigned)p.num_blocks) atomicOr(p.flags, PKV_FLAG_BLOCK_RANGE);
      const uint32_t bar = bar0 + stage * 8;
      T *kdst = wst + stage * 2 * C::TILE_ELEMS;
      mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
      // out-of-range block ids read as zeros (TMA bounds), never fault
      tma_load_4d(smem_addr(kdst), &kmap, 0, kvh, 0, pb, bar, pol);
      tma_load_4d(smem_addr(kdst + C::TILE_ELEMS), &vmap, 0, kvh, 0, pb, bar, pol);
    }
  };

  int issued = 0;
  for (; issued < n_w && issued < STAGES; ++issued) issue(issued, issued);

  // ---- query slice in registers, pre-scaled into the exp2 domain ----------
  float2 q2[GT][C::WPL];
  {
    const T *qb = static_cast<const T *>(p.q) + out_base + li * C::DPL;
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      uint32_t wv[C::WPL];
      if (g < gcount) {
        ldg_words<C::WPL>(qb + g * D, wv);
      } else {
#pragma unroll
        for (int k = 0; k < C::WPL; ++k) wv[k] = 0u;
      }
#pragma unroll
      for (int k = 0; k < C::WPL; ++k) {
        const float2 f = Widen<T>::pair(wv[k]);
        q2[g][k] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
      }
    }
  }

  const int g_own = li / C::LPG;
  const int base_idx = (li >> C::DUP_BITS) * C::R;
  const int tt0 = base_idx - g_own * C::HT;
  const bool primary = (li & ((1 << C::DUP_BITS) - 1)) == 0;
  float m_run = -INFINITY, l_run = 0.f;
  float2 o2[GT][C::WPL];
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int k = 0; k < C::WPL; ++k) o2[g][k] = make_float2(0.f, 0.f);

  float *pw = p_s + w * (2 * C::HT * GT);
  float *aw = a_s + w * GT;

  bool ok = true;
  int i = 0;
#pragma unroll 1
  for (; i < n_w; ++i) {
    const int stage = i % STAGES;
    const bool got = mbar_wait_bounded(bar0 + stage * 8, (uint32_t)((i / STAGES) & 1));
    if (!__all_sync(FULL_MASK, got)) {
      ok = false;
      break;
    }
    const int j = j0 + i * NW;
    const int valid_blk = min(B, L - j * B);
    const T *kt = wst + stage * 2 * C::TILE_ELEMS;
    const T *vt = kt + C::TILE_ELEMS;

#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      const int valid = valid_blk - c * C::CH;   // may be <= 0 for a tail chunk
      if (valid <= 0) break;                     // warp-uniform
      const T *kc = kt + c * C::CH * D;
      const T *vc = vt + c * C::CH * D;

      // scores of this half's tokens against every head of the chunk
      float sc[C::V];
#pragma unroll
      for (int tt = 0; tt < C::HT; ++tt) {
        const int t = half * C::HT + tt;
        uint32_t kw[C::WPL];
        load_words<C::WPL>(kc + t * D + li * C::DPL, kw);
        float2 kf[C::WPL];
#pragma unroll
        for (int k = 0; k < C::WPL; ++k) kf[k] = Widen<T>::pair(kw[k]);
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < C::WPL; ++k) acc = fma2(q2[g][k], kf[k], acc);
          sc[g * C::HT + tt] = acc.x + acc.y;
        }
      }
      half_reduce_scatter<C::V>(sc, li);

      // online softmax for head g_own (identical in all lanes of the group
      // and in both halves)
      float own[C::R];
      float bmax = -INFINITY;
#pragma unroll
      for (int r = 0; r < C::R; ++r) {
        const int t = half * C::HT + tt0 + r;
        own[r] = t < valid ? sc[r] : -INFINITY;
        bmax = fmaxf(bmax, own[r]);
      }
#pragma unroll
      for (int off = 1; off < C::LPG; off <<= 1)
        bmax = fmaxf(bmax, __shfl_xor_sync(FULL_MASK, bmax, off));
      bmax = fmaxf(bmax, __shfl_xor_sync(FULL_MASK, bmax, 16));
      const float m_new = fmaxf(m_run, bmax);
      const float alpha = fast_exp2(m_run - m_new);
      float lsum = 0.f;
#pragma unroll
      for (int r = 0; r < C::R; ++r) {
        own[r] = fast_exp2(own[r] - m_new);
        lsum += own[r];
      }
      if (!primary) lsum = 0.f;
#pragma unroll
      for (int off = 1; off < C::LPG; off <<= 1)
        lsum += __shfl_xor_sync(FULL_MASK, lsum, off);
      lsum += __shfl_xor_sync(FULL_MASK, lsum, 16);
      l_run = l_run * alpha + lsum;
      m_run = m_new;

      // publish P[half][tt][g] and alpha[g] to the warp
      if (primary) {
#pragma unroll
        for (int r = 0; r < C::R; ++r) pw[(half * C::HT + tt0 + r) * GT + g_own] = own[r];
      }
      if (half == 0 && (li % C::LPG) == 0) aw[g_own] = alpha;
      __syncwarp();

#pragma unroll
      for (int g = 0; g < GT; ++g) {
        const float a = aw[g];
#pragma unroll
        for (int k = 0; k < C::WPL; ++k) {
          o2[g][k].x *= a;
          o2[g][k].y *= a;
        }
      }
#pragma unroll
      for (int tt = 0; tt < C::HT; ++tt) {
        const int t = half * C::HT + tt;
        uint32_t vw[C::WPL];
        load_words<C::WPL>(vc + t * D + li * C::DPL, vw);
        float pg[GT];
#pragma unroll
        for (int g = 0; g < GT; ++g) pg[g] = pw[(half * C::HT + tt) * GT + g];
        if (t < valid) {
#pragma unroll
          for (int k = 0; k < C::WPL; ++k) {
            const float2 vf = Widen<T>::pair(vw[k]);
#pragma unroll
            for (int g = 0; g < GT; ++g)
              o2[g][k] = fma2(make_float2(pg[g], pg[g]), vf, o2[g][k]);
          }
        }
      }
      __syncwarp();  // P / alpha and this chunk's K, V reads are done
    }

    if (i + STAGES < n_w) {
      fence_proxy_async_smem();
      issue(i + STAGES, stage);
      ++issued;
    }
  }

  if (!ok) {
    if (lane == 0) {
      atomicOr(p.flags, PKV_FLAG_TIMEOUT);
      *s_abort = 1;
    }
    for (int k = i; k < issued; ++k)   // let this warp's copies land first
      (void)mbar_wait_bounded(bar0 + (k % STAGES) * 8, (uint32_t)((k / STAGES) & 1));
  }

  // both halves accumulated different tokens of the same heads and dims
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int k = 0; k < C::WPL; ++k) {
      o2[g][k].x += __shfl_xor_sync(FULL_MASK, o2[g][k].x, 16);
      o2[g][k].y += __shfl_xor_sync(FULL_MASK, o2[g][k].y, 16);
    }

  __syncthreads();  // every stage consumed: the stage area becomes merge space
  float *mg_o = reinterpret_cast<float *>(smem);    // [NW][GT][D]
  float *mg_ml = mg_o + NW * GT * D;                 // [NW][GT][2]
  if (half == 0) {
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int k = 0; k < C::WPL; ++k)
        *reinterpret_cast<float2 *>(mg_o + (w * GT + g) * D + li * C::DPL + 2 * k) = o2[g][k];
    if (li % C::LPG == 0) {
      mg_ml[(w * GT + g_own) * 2 + 0] = m_run;
      mg_ml[(w * GT + g_own) * 2 + 1] = l_run;
    }
  }
  __syncthreads();
  if (*s_abort) return;

  for (int idx = tid; idx < gcount * D; idx += NW * 32) {
    const int g = idx / D;
    const int d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int u = 0; u < NW; ++u) M = fmaxf(M, mg_ml[(u * GT + g) * 2]);
    float Lt = 0.f, O = 0.f;
#pragma unroll
    for (int u = 0; u < NW; ++u) {
      const float f = fast_exp2(mg_ml[(u * GT + g) * 2] - M);
      Lt += f * mg_ml[(u * GT + g) * 2 + 1];
      O += f * mg_o[(u * GT + g) * D + d];
    }
    if (nparts == 1) {
      store_out(p.out, out_base + idx, p.out_dtype, O / Lt);
    } else {
      const size_t rec = ((size_t)s * p.num_q_heads + hq0 + g) * p.max_parts + part;
      p.part_o[rec * D + d] = O;
      if (d == 0) {
        p.part_ml[rec * 2 + 0] = M;
        p.part_ml[rec * 2 + 1] = Lt;
      }
    }
  }
}

// Combines the partition records of every (sequence, query head) with more
// than one partition.  One warp per (sequence, query head).
template <int D, int B>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
  constexpr int DL = D / 32;
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.num_seqs * p.num_q_heads) return;
  const int s = gw / p.num_q_heads;
  const int hq = gw - s * p.num_q_heads;
  int L = __ldg(p.context_lens + s);
  const int cap = p.max_blocks * B;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int nb = (L + B - 1) / B;
  const int nparts = (nb + p.part_blocks - 1) / p.part_blocks;
  if (nparts <= 1) return;
  const size_t rec0 = ((size_t)s * p.num_q_heads + hq) * p.max_parts;
  float M = -INFINITY;
  for (int k = lane; k < nparts; k += 32) M = fmaxf(M, p.part_ml[(rec0 + k) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, off));
  float acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] = 0.f;
  float Lt = 0.f;
#pragma unroll 1
  for (int k = 0; k < nparts; ++k) {
    const float2 ml = *reinterpret_cast<const float2 *>(p.part_ml + (rec0 + k) * 2);
    const float f = fast_exp2(ml.x - M);
    Lt += f * ml.y;
    const float *o = p.part_o + (rec0 + k) * D + lane * DL;
    if constexpr (DL == 4) {
      const float4 x = *reinterpret_cast<const float4 *>(o);
      acc[0] += f * x.x; acc[1] += f * x.y; acc[2] += f * x.z; acc[3] += f * x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2 *>(o);
      acc[0] += f * x.x; acc[1] += f * x.y;
    }
  }
  const float inv = 1.f / Lt;
  const size_t ob = ((size_t)s * p.num_q_heads + hq) * D + lane * DL;
#pragma unroll
  for (int e = 0; e < DL; ++e) store_out(p.out, ob + e, p.out_dtype, acc[e] * inv);
}

// ---- host-side launch -------------------------------------------------------

template <int B, int D>
constexpr int stages_for(int tile_bytes_kv) {
  // about 24 KiB of K+V in flight per warp, 2..4 stages
  return max_c(2, min_c(4, (24 * 1024) / tile_bytes_kv));
}

template <typename T, int D, int B, int GT>
cudaError_t launch_decode_cfg(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeParams &p, cudaStream_t stream, int *launches) {
  constexpr int NW = 4;
  constexpr int STAGES = stages_for<B, D>(2 * B * D * (int)sizeof(T));
  using C = DecodeCfg<T, D, B, GT, NW, STAGES>;
  auto kern = decode_kernel<T, D, B, GT, NW, STAGES>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_done[64] = {false};
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  dim3 grid(p.max_parts, p.num_kv_heads * p.num_gchunks, p.num_seqs);
  kern<<<grid, NW * 32, C::SMEM_BYTES, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  if (p.max_parts > 1) {
    const int warps = p.num_seqs * p.num_q_heads;
    decode_merge_kernel<D, B><<<(warps + 3) / 4, 128, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  return cudaSuccess;
}

template <typename T, int D, int B>
cudaError_t launch_decode_gt(const CUtensorMap &kmap, const CUtensorMap &vmap,
                             const DecodeParams &p, cudaStream_t stream, int *launches) {
  const int g = p.group >= 8 ? 8 : p.group;
  if (g <= 1) return launch_decode_cfg<T, D, B, 1>(kmap, vmap, p, stream, launches);
  if (g <= 2) return launch_decode_cfg<T, D, B, 2>(kmap, vmap, p, stream, launches);
  if (g <= 4) return launch_decode_cfg<T, D, B, 4>(kmap, vmap, p, stream, launches);
  return launch_decode_cfg<T, D, B, 8>(kmap, vmap, p, stream, launches);
}

template <typename T, int D>
cudaError_t launch_decode_b(const CUtensorMap &kmap, const CUtensorMap &vmap,
                            const DecodeParams &p, int block_size, cudaStream_t stream,
                            int *launches) {
  switch (block_size) {
    case 4: return launch_decode_gt<T, D, 4>(kmap, vmap, p, stream, launches);
    case 8: return launch_decode_gt<T, D, 8>(kmap, vmap, p, stream, launches);
    case 16: return launch_decode_gt<T, D, 16>(kmap, vmap, p, stream, launches);
    case 32: return launch_decode_gt<T, D, 32>(kmap, vmap, p, stream, launches);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_decode_typed(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeParams &p, int head_dim, int block_size,
                                cudaStream_t stream, int *launches) {
  switch (head_dim) {
    case 64: return launch_decode_b<T, 64>(kmap, vmap, p, block_size, stream, launches);
    case 128: return launch_decode_b<T, 128>(kmap, vmap, p, block_size, stream, launches);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
