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

// CTAs per SM the kernel is shaped for: 3 up to 8 query heads per CTA,
// 2 for 16 (larger merge area).
constexpr int occupancy_for(int GT) { return GT >= 16 ? 2 : 3; }

// Stages per warp: fill the shared memory of an SM across its CTAs, 2..4.
constexpr int stages_for(int stage_bytes, int occ) {
  return max_c(2, min_c(4, (227 * 1024 / occ - 3 * 1024) / (DECODE_WARPS * stage_bytes)));
}

// Softmax reference-max slack (log2 domain): the running maximum used for
// the exponentials is raised only when a score exceeds it by more than this,
// so P stays <= 2^8 and the rescale of O is rare.  Exact: O and L always use
// the same reference.
constexpr float RESCALE_SLACK = 8.0f;

template <typename T, int D, int B, int GT>
struct DecodeCfg {
  static constexpr int NW = DECODE_WARPS;
  static constexpr int OCC = occupancy_for(GT);
  static constexpr int CH = min_c(B, 16);        // tokens per chunk (one TMA box high)
  static constexpr int NCH = B / CH;             // chunks per block
  static constexpr int NT = (CH + 7) / 8;        // 8-token MMA n-tiles in Q.K^T
  static constexpr int NSUB = D / 64;            // 128-byte column slabs of a row
  static constexpr int KS = D / 16;              // k-steps of Q.K^T
  static constexpr int NTD = D / 8;              // 8-dim MMA n-tiles of P.V
  static constexpr int SUB_BYTES = 16 * 128;     // one slab: 16 rows x 128 B, 128B-swizzled
  static constexpr int CHUNK_BYTES = NSUB * SUB_BYTES;   // K (or V) of one chunk
  static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;    // K + V
  static constexpr int TX_BYTES = 2 * NSUB * CH * 128;   // bytes the TMA loads deliver
  static constexpr int STAGES = stages_for(STAGE_BYTES, OCC);
  // shared memory (bytes)
  static constexpr int STAGES_BYTES = NW * STAGES * STAGE_BYTES;
  static constexpr int MERGE_BYTES = NW * GT * (D + 2) * 4;
  static constexpr int BIG_BYTES = round_up_c(max_c(STAGES_BYTES, MERGE_BYTES), 1024);
  static constexpr int BAR_BYTES = NW * STAGES * 8;
  static constexpr int SMEM_BYTES = 1024 + BIG_BYTES + BAR_BYTES + 16;

  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(B == 4 || B == 8 || B == 16 || B == 32, "block_size");
  static_assert(GT == 1 || GT == 4 || GT == 8 || GT == 16, "query head rows");
  static_assert(SMEM_BYTES * OCC <= 227 * 1024, "shared memory budget");
};

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
  const uint32_t stage_smem = smem_addr(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BIG_BYTES);
  volatile int *s_int = reinterpret_cast<volatile int *>(bars + NW * STAGES);  // next, abort, last

  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  const int HC = p.num_hc;
  const int cap = p.max_blocks * B;

  // Rows a chunk never loads (block_size < 16) must read as zeros in P.V.
  if (C::CH < 16) {
    for (int i = tid; i < C::STAGES_BYTES / 16; i += NW * 32)
      *reinterpret_cast<uint4 *>(smem + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
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

  const uint32_t wst = stage_smem + w * STAGES * C::STAGE_BYTES;
  const uint32_t bar0 = smem_addr(bars + w * STAGES);
  const uint64_t pol = l2_policy_evict_first();
  uint32_t ld_cnt = 0, use_cnt = 0;   // this warp's loads issued / consumed, all units

  // fragment coordinates of this lane
  const int r0 = lane >> 2;                         // C rows r0 and r0 + 8 (query heads)
  const int cq = 2 * (lane & 3);                    // C columns cq, cq + 1
  const int k_tok = ((lane >> 4) & 1) * 8 + (lane & 7);   // ldmatrix row for K (B operand)
  const int k_chb = (lane >> 3) & 1;
  const int v_tok = ((lane >> 3) & 1) * 8 + (lane & 7);   // ldmatrix row for V (trans)
  const int v_chb = (lane >> 4) & 1;

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
        const uint32_t dst = wst + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(bar, C::TX_BYTES);
        // out-of-range block ids read as zeros (TMA bounds), never fault
#pragma unroll
        for (int sb = 0; sb < C::NSUB; ++sb) {
          tma_load_4d(dst + sb * C::SUB_BYTES, &kmap, sb * 64, kvh, c * C::CH, pb, bar, pol);
          tma_load_4d(dst + C::CHUNK_BYTES + sb * C::SUB_BYTES, &vmap, sb * 64, kvh,
                      c * C::CH, pb, bar, pol);
        }
      }
      ++ld_cnt;
    };

    // The stage area held the previous unit's merge data: every thread
    // fenced its generic writes before the unit barrier; order them ahead of
    // this unit's TMA writes.  Within a unit a stage is refilled only after
    // every lane's reads of it have returned.
    if (lane == 0) fence_proxy_async_smem();
    int issued = 0;
    for (; issued < n_units && issued < STAGES; ++issued) issue(issued);

    // ---- query rows as MMA A fragments (rows >= gcount are zero) ----------
    uint32_t qa[C::KS][4];
    {
      const T *qb = static_cast<const T *>(p.q) + out_base;
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = r0 + ((e & 1) ? 8 : 0);
          const int kk = ks * 16 + cq + ((e & 2) ? 8 : 0);
          qa[ks][e] = row < gcount
                          ? __ldg(reinterpret_cast<const unsigned int *>(qb + row * D + kk))
                          : 0u;
        }
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[C::NTD][4];
#pragma unroll
    for (int nt = 0; nt < C::NTD; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;

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
      const uint32_t kb = wst + stage * C::STAGE_BYTES;
      const uint32_t vb = kb + C::CHUNK_BYTES;

      if (valid < C::CH) {
        // rows at or past the context length hold stale pool bytes: zero the
        // V rows so that 0 * V stays 0 in P.V (K rows are masked below)
        unsigned char *vrow = smem + (vb - stage_smem);
        for (int x = lane; x < (C::CH - valid) * C::NSUB * 8; x += 32) {
          const int piece = x & 7;
          const int rr = x >> 3;
          const int sb = rr % C::NSUB;
          const int row = valid + rr / C::NSUB;
          *reinterpret_cast<uint4 *>(vrow + sb * C::SUB_BYTES + row * 128 + piece * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // S = Q K^T (rows: query heads, columns: the chunk's tokens)
      float sa[C::NT][4];
#pragma unroll
      for (int jn = 0; jn < C::NT; ++jn)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[jn][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        const int sb = ks >> 2;
        const int ch = (ks & 3) * 2 + k_chb;
        const uint32_t addr = kb + sb * C::SUB_BYTES + k_tok * 128 + ((ch ^ (k_tok & 7)) << 4);
        if (C::NT == 2) {
          uint32_t r[4];
          ldsm_x4(r, addr);
          Mma<T>::run(sa[0], qa[ks], r[0], r[1]);
          Mma<T>::run(sa[C::NT - 1], qa[ks], r[2], r[3]);
        } else {
          uint32_t r[2];
          ldsm_x2(r, addr);
          Mma<T>::run(sa[0], qa[ks], r[0], r[1]);
        }
      }

      // online softmax (exp2 domain) with a lazily raised reference max
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int jn = 0; jn < C::NT; ++jn)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = 8 * jn + cq + (e & 1);
          const float x = tok < valid ? sa[jn][e] * p.scale_log2 : -INFINITY;
          sa[jn][e] = x;
          if (e < 2) mx0 = fmaxf(mx0, x); else mx1 = fmaxf(mx1, x);
        }
      mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 2));
      const bool up0 = mx0 > m0 + RESCALE_SLACK, up1 = mx1 > m1 + RESCALE_SLACK;
      if (__any_sync(FULL_MASK, up0 || up1)) {
        const float n0 = up0 ? mx0 : m0, n1 = up1 ? mx1 : m1;
        const float a0 = fast_exp2(m0 - n0), a1 = fast_exp2(m1 - n1);
        m0 = n0;
        m1 = n1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int nt = 0; nt < C::NTD; ++nt) {
          o[nt][0] *= a0; o[nt][1] *= a0;
          o[nt][2] *= a1; o[nt][3] *= a1;
        }
      }
      uint32_t ah[4], al[4];
#pragma unroll
      for (int jn = 0; jn < 2; ++jn) {
        if (jn < C::NT) {
          const float p00 = fast_exp2(sa[jn][0] - m0), p01 = fast_exp2(sa[jn][1] - m0);
          const float p10 = fast_exp2(sa[jn][2] - m1), p11 = fast_exp2(sa[jn][3] - m1);
          l0 += p00 + p01;
          l1 += p10 + p11;
          // P in two 16-bit pieces (hi + lo) keeps about 16 mantissa bits
          const uint32_t h0 = Mma<T>::pack(p00, p01), h1 = Mma<T>::pack(p10, p11);
          const float2 b0 = Widen<T>::pair(h0), b1 = Widen<T>::pair(h1);
          ah[2 * jn + 0] = h0;
          ah[2 * jn + 1] = h1;
          al[2 * jn + 0] = Mma<T>::pack(p00 - b0.x, p01 - b0.y);
          al[2 * jn + 1] = Mma<T>::pack(p10 - b1.x, p11 - b1.y);
        } else {
          ah[2 * jn] = ah[2 * jn + 1] = al[2 * jn] = al[2 * jn + 1] = 0u;
        }
      }

      // O += P V
#pragma unroll
      for (int nt = 0; nt < C::NTD; nt += 2) {
        const int sb = nt >> 3;
        const int ch = (nt & 7) + v_chb;
        uint32_t r[4];
        ldsm_x4_trans(r, vb + sb * C::SUB_BYTES + v_tok * 128 + ((ch ^ (v_tok & 7)) << 4));
        Mma<T>::run(o[nt], ah, r[0], r[1]);
        Mma<T>::run(o[nt], al, r[0], r[1]);
        Mma<T>::run(o[nt + 1], ah, r[2], r[3]);
        Mma<T>::run(o[nt + 1], al, r[2], r[3]);
      }
      __syncwarp();   // every lane's reads of this stage have returned
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

    // row sums: the 4 lanes of a row hold different columns
    l0 += __shfl_xor_sync(FULL_MASK, l0, 1);
    l0 += __shfl_xor_sync(FULL_MASK, l0, 2);
    l1 += __shfl_xor_sync(FULL_MASK, l1, 1);
    l1 += __shfl_xor_sync(FULL_MASK, l1, 2);

    __syncthreads();  // every stage consumed: the stage area becomes merge space
    float *mg_o = reinterpret_cast<float *>(smem);    // [NW][GT][D]
    float *mg_ml = mg_o + NW * GT * D;                 // [NW][GT][2]
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int row = r0 + 8 * hr;
      if (row < gcount) {
#pragma unroll
        for (int nt = 0; nt < C::NTD; ++nt)
          *reinterpret_cast<float2 *>(mg_o + (w * GT + row) * D + 8 * nt + cq) =
              make_float2(o[nt][2 * hr], o[nt][2 * hr + 1]);
        if ((lane & 3) == 0) {
          mg_ml[(w * GT + row) * 2 + 0] = hr ? m1 : m0;
          mg_ml[(w * GT + row) * 2 + 1] = hr ? l1 : l0;
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
    __syncthreads();  // merge reads done
    if (C::CH < 16) {   // the merge overwrote rows that must stay zero
      for (int i2 = tid; i2 < C::MERGE_BYTES / 16; i2 += NW * 32)
        *reinterpret_cast<uint4 *>(smem + i2 * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncthreads();  // stage area free again; s_int[0] holds the next unit
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
  const int g = p.group >= 16 ? 16 : p.group;
  if (g <= 1) return launch_decode_cfg<T, D, B, 1>(kmap, vmap, p, stream, launches);
  if (g <= 4) return launch_decode_cfg<T, D, B, 4>(kmap, vmap, p, stream, launches);
  if (g <= 8) return launch_decode_cfg<T, D, B, 8>(kmap, vmap, p, stream, launches);
  return launch_decode_cfg<T, D, B, 16>(kmap, vmap, p, stream, launches);
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
