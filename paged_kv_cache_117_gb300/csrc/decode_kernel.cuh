// Paged decode attention for sm_103a.
//
// What is computed (PagedAttention, "PagedAttention and vLLM: Paging the KV
// Cache Like an OS", Step 5; "PagedAttention: Virtual Memory for the KV
// Cache", block-wise attention equation): for each query head of a GQA group,
// walk the sequence's block table, score the query against every valid key of
// every block, run one softmax over all valid positions, and weight the
// values.  Each gathered K/V block is read once from HBM for the whole query
// group of its KV head.
//
// Work decomposition.  A sequence's context is cut into partitions of
// part_blocks blocks.  A work unit is (sequence, partition, KV head, query
// head chunk of <= 8).  decode_plan_kernel (one CTA) lists the (sequence,
// partition) items in the workspace -- all full partitions first, then the
// shorter last partitions -- and resets the work counter and the per-sequence
// completion counters.  decode_kernel runs as a persistent grid sized to fill
// the SMs; each CTA takes the next unit with one atomicAdd (fetched while the
// current unit is processed), so no CTA slot is spent on empty work and the
// short units land at the end.
//
// Inside a CTA (4 warps), warp w streams blocks jb + w, jb + w + 4, ... of the
// partition through a private ring of STAGES shared-memory stages.  One lane
// issues two 4-D TMA tile loads per chunk of <= 16 tokens (K and V tile
// [chunk, head_dim] of one KV head; pool layout [N, B, Hkv, D], so a tile is
// `chunk` rows of head_dim*2 bytes at a stride of Hkv*head_dim*2 bytes),
// completing on the stage's mbarrier; the stage/phase counters run on across
// units, so barriers are initialised once per CTA.
//
// Per chunk: half-warp h takes half of the chunk's tokens; lane li owns
// head_dim/16 consecutive dims.  Q.K partial dot products use the packed fp32x2
// FMA; the (token, head) partials are summed across the 16 lanes by a
// reduce-scatter butterfly (about one shuffle per partial instead of four).
// Online softmax in fp32 in the exp2 domain (q pre-scaled by scale*log2 e);
// slots at or past the context length are masked before the max and skipped
// in P.V, so whatever bytes they hold never reach the result.  P goes to the
// warp through shared memory as (p, p) pairs that feed the packed FMA as is.
//
// End of a unit: the warps' (max, sum, output) states merge in shared memory.
// A one-partition sequence writes out = O / L.  Otherwise the unit writes its
// unnormalised (M, L, O) record, bumps the sequence's completion counter, and
// the CTA that completes the last partition merges all records:
// o = sum_p e^(M_p - M) O_p / sum_p e^(M_p - M) L_p.  Normalising each
// partition and adding the results would be wrong ("PagedAttention"
// (tensortonic), section 5).  No CTA ever waits on another.
#pragma once

#include <math.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

constexpr int ilog2_c(int v) { return v <= 1 ? 0 : 1 + ilog2_c(v >> 1); }
constexpr int max_c(int a, int b) { return a > b ? a : b; }
constexpr int min_c(int a, int b) { return a < b ? a : b; }
constexpr int round_up_c(int v, int a) { return (v + a - 1) / a * a; }

constexpr int DECODE_WARPS = 4;

// CTAs per SM the kernel is shaped for: 3 when the register budget allows
// (up to 4 query heads per CTA), otherwise 2.
constexpr int occupancy_for(int GT) { return GT >= 8 ? 2 : 3; }

// Stages per warp: fill about 220 KiB of shared memory across the CTAs of an
// SM, 2..4 stages.
constexpr int stages_for(int stage_bytes, int occ) {
  return max_c(2, min_c(4, (220 * 1024 / occ - 4096) / (DECODE_WARPS * stage_bytes)));
}

template <typename T, int D, int B, int GT>
struct DecodeCfg {
  static constexpr int NW = DECODE_WARPS;
  static constexpr int OCC = occupancy_for(GT);
  static constexpr int CH = min_c(B, 16);        // tokens per chunk (one TMA box)
  static constexpr int NCH = B / CH;             // chunks per block
  static constexpr int HT = CH / 2;              // tokens per half-warp per chunk
  static constexpr int DPL = D / 16;             // dims owned by a lane
  static constexpr int WPL = DPL / 2;            // 32-bit words per lane row slice
  static constexpr int CHUNK_ELEMS = CH * D;
  static constexpr int CHUNK_BYTES = CHUNK_ELEMS * (int)sizeof(T);
  static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;   // K + V
  static constexpr int STAGES = stages_for(STAGE_BYTES, OCC);
  static constexpr int GP = min_c(GT, 4);        // heads per score pass
  static constexpr int NPASS = GT / GP;
  static constexpr int V = HT * GP;              // partial scores per lane per pass
  static constexpr int LPG = 16 / GP;            // lanes per head within a half-warp
  static constexpr int SCAT = V >= 16 ? 4 : ilog2_c(V);
  static constexpr int DUP_BITS = 4 - SCAT;      // lanes holding copies of one sum
  static constexpr int R = V >= 16 ? V / 16 : 1; // sums owned per lane
  // shared memory (bytes)
  static constexpr int STAGES_BYTES = NW * STAGES * STAGE_BYTES;
  static constexpr int MERGE_BYTES = NW * GT * (D + 2) * 4;
  static constexpr int BIG_BYTES = round_up_c(max_c(STAGES_BYTES, MERGE_BYTES), 128);
  static constexpr int P_FLOATS = NW * 2 * HT * GT * 2;   // (p, p) pairs
  static constexpr int A_FLOATS = NW * GT;
  static constexpr int SMALL_BYTES = round_up_c((P_FLOATS + A_FLOATS) * 4, 16);
  static constexpr int BAR_BYTES = NW * STAGES * 8;
  static constexpr int SMEM_BYTES = 1024 + BIG_BYTES + SMALL_BYTES + BAR_BYTES + 16;

  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(B == 4 || B == 8 || B == 16 || B == 32, "block_size");
  static_assert(GT == 1 || GT == 2 || GT == 4 || GT == 8, "query head chunk");
  static_assert(R <= HT, "a lane's sums belong to one head");
  static_assert(SMEM_BYTES * OCC <= 227 * 1024, "shared memory budget");
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

__device__ __forceinline__ int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

// ---------------------------------------------------------------------------
// Work list: one CTA of 1024 threads.
static __global__ void __launch_bounds__(1024) decode_plan_kernel(const DecodeParams p) {
  __shared__ int wsum_f[32], wsum_p[32];
  const int S = p.num_seqs, PB = p.part_blocks, Bs = p.block_size;
  const int cap = p.max_blocks * Bs;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (S + 1023) / 1024;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  int nf = 0, np = 0;
  for (int s = s0; s < s1; ++s) {
    const int L0 = __ldg(p.context_lens + s);
    if (L0 < 0 || L0 > cap) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    const int nb = (clamp_len(L0, cap) + Bs - 1) / Bs;
    nf += nb / PB;
    np += (nb % PB) != 0;
  }
  // block-wide exclusive scans of nf and np
  int xf = nf, xp = np;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int yf = __shfl_up_sync(FULL_MASK, xf, off);
    const int yp = __shfl_up_sync(FULL_MASK, xp, off);
    if (lane >= off) { xf += yf; xp += yp; }
  }
  if (lane == 31) { wsum_f[wid] = xf; wsum_p[wid] = xp; }
  __syncthreads();
  if (wid == 0) {
    int tf = wsum_f[lane], tp = wsum_p[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int yf = __shfl_up_sync(FULL_MASK, tf, off);
      const int yp = __shfl_up_sync(FULL_MASK, tp, off);
      if (lane >= off) { tf += yf; tp += yp; }
    }
    wsum_f[lane] = tf;   // inclusive over warps
    wsum_p[lane] = tp;
  }
  __syncthreads();
  const int total_f = wsum_f[31], total_p = wsum_p[31];
  int fo = xf - nf + (wid ? wsum_f[wid - 1] : 0);
  int po = total_f + xp - np + (wid ? wsum_p[wid - 1] : 0);
  for (int s = s0; s < s1; ++s) {
    const int L = clamp_len(__ldg(p.context_lens + s), cap);
    const int nb = (L + Bs - 1) / Bs;
    const int F = nb / PB;
    for (int q = 0; q < F; ++q) p.items[fo++] = make_int2(s, q);
    if (nb % PB) p.items[po++] = make_int2(s, F);
    if (L == 0) {   // nothing to attend to: zeros
      const size_t base = (size_t)s * p.num_q_heads * p.head_dim;
      for (int e = 0; e < p.num_q_heads * p.head_dim; ++e) store_out(p.out, base + e, p.out_dtype, 0.f);
    }
  }
  for (int i = tid; i < S * p.num_hc; i += 1024) p.seq_done[i] = 0u;
  if (tid == 0) {
    p.ctrl[0] = 0u;
    p.ctrl[1] = (unsigned)(total_f + total_p) * (unsigned)p.num_hc;
  }
}

// ---------------------------------------------------------------------------
template <typename T, int D, int B, int GT>
__global__ void __launch_bounds__(DECODE_WARPS * 32, occupancy_for(GT))
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using C = DecodeCfg<T, D, B, GT>;
  constexpr int NW = C::NW;
  constexpr int STAGES = C::STAGES;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  T *stages = reinterpret_cast<T *>(smem);
  float *p_s = reinterpret_cast<float *>(smem + C::BIG_BYTES);
  float *a_s = p_s + C::P_FLOATS;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BIG_BYTES + C::SMALL_BYTES);
  volatile int *s_int = reinterpret_cast<volatile int *>(bars + NW * STAGES);  // next, abort, last

  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5, half = lane >> 4, li = lane & 15;
  const int HC = p.num_hc;
  const int cap = p.max_blocks * B;

  if (tid == 0) {
#pragma unroll 1
    for (int i = 0; i < NW * STAGES; ++i) mbar_init(smem_addr(bars + i), 1);
    s_int[1] = 0;
    s_int[0] = (int)atomicAdd(p.ctrl, 1u);
    fence_barrier_init();
  }
  if (tid == 32 || (NW == 1 && tid == 0)) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  const unsigned total = __ldcg(p.ctrl + 1);
  __syncthreads();

  T *wst = stages + (size_t)w * STAGES * 2 * C::CHUNK_ELEMS;
  const uint32_t bar0 = smem_addr(bars + w * STAGES);
  const uint64_t pol = l2_policy_evict_first();
  float2 *pw = reinterpret_cast<float2 *>(p_s) + w * (2 * C::HT * GT);
  float *aw = a_s + w * GT;
  uint32_t ld_cnt = 0, use_cnt = 0;   // this warp's loads issued / consumed, all units

  const int g_loc = li / C::LPG;                      // head within a score pass
  const int base_idx = (li >> C::DUP_BITS) * C::R;
  const int tt0 = base_idx - g_loc * C::HT;
  const bool primary = (li & ((1 << C::DUP_BITS) - 1)) == 0;

  unsigned unit = (unsigned)s_int[0];
#pragma unroll 1
  while (unit < total) {
    __syncthreads();   // every thread has read s_int[0]
    if (tid == 0) s_int[0] = (int)atomicAdd(p.ctrl, 1u);

    const int2 item = __ldcg(p.items + unit / HC);
    const int hc = (int)(unit % HC);
    const int s = item.x, part = item.y;
    const int kvh = hc / p.num_gchunks;
    const int gc = hc - kvh * p.num_gchunks;
    const int L = clamp_len(__ldg(p.context_lens + s), cap);
    const int nb = (L + B - 1) / B;
    const int jb = part * p.part_blocks;
    const int je = min(nb, jb + p.part_blocks);
    const int nparts = (nb + p.part_blocks - 1) / p.part_blocks;
    const int g0 = gc * GT;
    const int gcount = min(GT, p.group - g0);
    const int hq0 = kvh * p.group + g0;
    const size_t out_base = ((size_t)s * p.num_q_heads + hq0) * D;

    // ---- this warp's blocks, chunks and slice of the block table ----------
    const int j0 = jb + w;
    const int n_w = j0 < je ? (je - j0 + NW - 1) / NW : 0;
    int n_units = n_w * C::NCH;
    if (C::NCH > 1 && n_w > 0 && j0 + (n_w - 1) * NW == nb - 1) {
      const int tail = L - (nb - 1) * B;                 // tokens in the last block
      n_units -= C::NCH - (tail + C::CH - 1) / C::CH;
    }
    const int32_t *trow = p.block_tables + (size_t)s * p.max_blocks;
    int kbase = 0;
    int tbl = lane < n_w ? __ldg(trow + j0 + lane * NW) : 0;

    auto issue = [&](int u) {
      const int i = u / C::NCH;
      const int c = u - i * C::NCH;
      if (i - kbase >= 32) {
        kbase += 32;
        tbl = kbase + lane < n_w ? __ldg(trow + j0 + (kbase + lane) * NW) : 0;
      }
      const int pb = __shfl_sync(FULL_MASK, tbl, i - kbase);
      if (lane == 0) {
        if ((unsigned)pb >= (unsigned)p.num_blocks) atomicOr(p.flags, PKV_FLAG_BLOCK_RANGE);
        const int stage = (int)(ld_cnt % STAGES);
        const uint32_t bar = bar0 + stage * 8;
        T *kdst = wst + stage * 2 * C::CHUNK_ELEMS;
        mbar_arrive_expect_tx(bar, 2 * C::CHUNK_BYTES);
        // out-of-range block ids read as zeros (TMA bounds), never fault
        tma_load_4d(smem_addr(kdst), &kmap, 0, kvh, c * C::CH, pb, bar, pol);
        tma_load_4d(smem_addr(kdst + C::CHUNK_ELEMS), &vmap, 0, kvh, c * C::CH, pb, bar, pol);
      }
      ++ld_cnt;
    };

    // The stage area held the previous unit's merge data (generic-proxy
    // writes); order those before this unit's TMA writes.  Within a unit a
    // stage is refilled only after every lane's reads of it have returned.
    if (lane == 0) fence_proxy_async_smem();
    int issued = 0;
    for (; issued < n_units && issued < STAGES; ++issued) issue(issued);

    // ---- query slice in registers, pre-scaled into the exp2 domain --------
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

    float m_run[C::NPASS], l_run[C::NPASS];
#pragma unroll
    for (int ps = 0; ps < C::NPASS; ++ps) { m_run[ps] = -INFINITY; l_run[ps] = 0.f; }
    float2 o2[GT][C::WPL];
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int k = 0; k < C::WPL; ++k) o2[g][k] = make_float2(0.f, 0.f);

    bool ok = true;
    int u = 0;
#pragma unroll 1
    for (; u < n_units; ++u) {
      const uint32_t stage = use_cnt % STAGES;
      const bool got = mbar_wait_bounded(bar0 + stage * 8, (use_cnt / STAGES) & 1u);
      if (!__all_sync(FULL_MASK, got)) {
        ok = false;
        break;
      }
      const int i = u / C::NCH;
      const int c = u - i * C::NCH;
      const int j = j0 + i * NW;
      const int valid = min(C::CH, L - j * B - c * C::CH);   // >= 1
      const T *kt = wst + stage * 2 * C::CHUNK_ELEMS;
      const T *vt = kt + C::CHUNK_ELEMS;

      float alpha_own[C::NPASS];
#pragma unroll
      for (int ps = 0; ps < C::NPASS; ++ps) {
        // scores of this half's tokens against heads ps*GP .. ps*GP+GP-1
        float sc[C::V];
#pragma unroll
        for (int tt = 0; tt < C::HT; ++tt) {
          const int t = half * C::HT + tt;
          uint32_t kw[C::WPL];
          load_words<C::WPL>(kt + t * D + li * C::DPL, kw);
          float2 kf[C::WPL];
#pragma unroll
          for (int k = 0; k < C::WPL; ++k) kf[k] = Widen<T>::pair(kw[k]);
#pragma unroll
          for (int gl = 0; gl < C::GP; ++gl) {
            const int g = ps * C::GP + gl;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < C::WPL; ++k) acc = fma2(q2[g][k], kf[k], acc);
            sc[gl * C::HT + tt] = acc.x + acc.y;
          }
        }
        half_reduce_scatter<C::V>(sc, li);

        // online softmax of head ps*GP + g_loc (identical in all lanes of the
        // group and in both halves)
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
        const float m_new = fmaxf(m_run[ps], bmax);
        const float alpha = fast_exp2(m_run[ps] - m_new);
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
        l_run[ps] = l_run[ps] * alpha + lsum;
        m_run[ps] = m_new;
        alpha_own[ps] = alpha;
        if (primary) {
#pragma unroll
          for (int r = 0; r < C::R; ++r)
            pw[(half * C::HT + tt0 + r) * GT + ps * C::GP + g_loc] = make_float2(own[r], own[r]);
        }
      }
      if (half == 0 && (li % C::LPG) == 0) {
#pragma unroll
        for (int ps = 0; ps < C::NPASS; ++ps) aw[ps * C::GP + g_loc] = alpha_own[ps];
      }
      __syncwarp();

#pragma unroll
      for (int g = 0; g < GT; ++g) {
        const float a = aw[g];
        const float2 aa = make_float2(a, a);
#pragma unroll
        for (int k = 0; k < C::WPL; ++k) o2[g][k] = __fmul2_rn(o2[g][k], aa);
      }
#pragma unroll
      for (int tt = 0; tt < C::HT; ++tt) {
        const int t = half * C::HT + tt;
        uint32_t vw[C::WPL];
        load_words<C::WPL>(vt + t * D + li * C::DPL, vw);
        float2 pp[GT];
#pragma unroll
        for (int g = 0; g < GT; ++g) pp[g] = pw[(half * C::HT + tt) * GT + g];
        if (t < valid) {
#pragma unroll
          for (int k = 0; k < C::WPL; ++k) {
            const float2 vf = Widen<T>::pair(vw[k]);
#pragma unroll
            for (int g = 0; g < GT; ++g) o2[g][k] = fma2(pp[g], vf, o2[g][k]);
          }
        }
      }
      __syncwarp();   // P / alpha and this stage's K, V reads are done
      ++use_cnt;
      if (issued < n_units) {
        issue(issued);
        ++issued;
      }
    }

    if (!ok) {
      if (lane == 0) {
        atomicOr(p.flags, PKV_FLAG_TIMEOUT);
        s_int[1] = 1;
      }
      // let this warp's copies land before the stages are reused or released
      for (; use_cnt < ld_cnt; ++use_cnt)
        (void)mbar_wait_bounded(bar0 + (use_cnt % STAGES) * 8, (use_cnt / STAGES) & 1u);
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
#pragma unroll
        for (int ps = 0; ps < C::NPASS; ++ps) {
          mg_ml[(w * GT + ps * C::GP + g_loc) * 2 + 0] = m_run[ps];
          mg_ml[(w * GT + ps * C::GP + g_loc) * 2 + 1] = l_run[ps];
        }
      }
    }
    __syncthreads();
    const bool abort = s_int[1] != 0;
    if (!abort) {
      for (int idx = tid; idx < gcount * D; idx += NW * 32) {
        const int g = idx / D;
        const int d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int x = 0; x < NW; ++x) M = fmaxf(M, mg_ml[(x * GT + g) * 2]);
        float Lt = 0.f, O = 0.f;
#pragma unroll
        for (int x = 0; x < NW; ++x) {
          const float f = fast_exp2(mg_ml[(x * GT + g) * 2] - M);
          Lt += f * mg_ml[(x * GT + g) * 2 + 1];
          O += f * mg_o[(x * GT + g) * D + d];
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
      if (nparts > 1) {
        // Release this CTA's records (ordered before thread 0 by the barrier)
        // with one gpu-scope fence before the counter update; the CTA that
        // sees the final count fences again before reading the others'.
        __syncthreads();
        if (tid == 0) {
          __threadfence();
          const unsigned prev = atomicAdd(p.seq_done + (size_t)s * HC + hc, 1u);
          const bool last = prev == (unsigned)(nparts - 1);
          if (last) __threadfence();
          s_int[2] = last;
        }
        __syncthreads();
        if (s_int[2]) {   // this CTA completed the sequence's last partition
          for (int idx = tid; idx < gcount * D; idx += NW * 32) {
            const int g = idx / D;
            const int d = idx - g * D;
            const size_t rec0 = ((size_t)s * p.num_q_heads + hq0 + g) * p.max_parts;
            float M = -INFINITY;
            for (int q = 0; q < nparts; ++q) M = fmaxf(M, __ldcg(p.part_ml + (rec0 + q) * 2));
            float Lt = 0.f, O = 0.f;
            for (int q = 0; q < nparts; ++q) {
              const float f = fast_exp2(__ldcg(p.part_ml + (rec0 + q) * 2) - M);
              Lt += f * __ldcg(p.part_ml + (rec0 + q) * 2 + 1);
              O += f * __ldcg(p.part_o + (rec0 + q) * D + d);
            }
            store_out(p.out, out_base + idx, p.out_dtype, O / Lt);
          }
        }
      }
    }
    __syncthreads();  // merge space is free again; s_int[0] holds the next unit
    if (abort) break;
    unit = (unsigned)s_int[0];
  }
}

// ---- host-side launch -------------------------------------------------------

// Per (kernel, device) launch facts: the dynamic shared memory attribute is
// set once and the resident CTAs per SM and the SM count are cached.  The
// table has internal linkage, so two copies of this library loaded in one
// process never share it.
namespace {
struct LaunchInfo {
  const void *fn;
  int dev;
  int ctas_per_sm;
  int sms;
};
LaunchInfo g_launch_info[256];
int g_launch_info_n = 0;
std::mutex g_launch_mu;

cudaError_t launch_info(const void *fn, int threads, int smem, int dev, LaunchInfo *out) {
  std::lock_guard<std::mutex> lock(g_launch_mu);
  for (int i = 0; i < g_launch_info_n; ++i)
    if (g_launch_info[i].fn == fn && g_launch_info[i].dev == dev) {
      *out = g_launch_info[i];
      return cudaSuccess;
    }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int n = 0, m = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const LaunchInfo li{fn, dev, n > 0 ? n : 1, m};
  if (g_launch_info_n < 256) g_launch_info[g_launch_info_n++] = li;
  *out = li;
  return cudaSuccess;
}
}  // namespace

template <typename T, int D, int B, int GT>
cudaError_t launch_decode_cfg(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeParams &p, cudaStream_t stream, int *launches) {
  using C = DecodeCfg<T, D, B, GT>;
  auto kern = decode_kernel<T, D, B, GT>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  LaunchInfo li;
  e = launch_info(reinterpret_cast<const void *>(kern), C::NW * 32, C::SMEM_BYTES, dev, &li);
  if (e != cudaSuccess) return e;
  decode_plan_kernel<<<1, 1024, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  const long long units_max =
      (long long)p.num_seqs * p.max_parts * p.num_hc;   // upper bound on work units
  long long grid = (long long)li.sms * li.ctas_per_sm;
  if (grid > units_max) grid = units_max;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, C::NW * 32, C::SMEM_BYTES, stream>>>(kmap, vmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
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
