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
// part_blocks blocks.  A work unit is (sequence, partition, KV head, chunk of
// up to 16 query heads).  decode_plan_kernel (one CTA) lists the (sequence,
// partition) items in the workspace -- the full partitions of the sequences
// that span several, then their shorter last partitions, then the
// one-partition sequences, the last two groups longest first -- and resets
// the work counter and the per-sequence completion counters.  decode_kernel runs as a persistent
// grid sized to fill the SMs; CTA c starts with units c and c + grid, then
// takes units with atomicAdd, two ahead of the one it is processing, so that
// every warp knows its next unit while it works on the current one.
//
// Streaming.  Warp w of the CTA takes blocks jb + w, jb + w + 4, ... of the
// unit's partition, in chunks of up to 16 tokens, through a private ring of
// STAGES shared-memory stages.  One lane issues the TMA tile loads of a chunk
// (K and V, one 128-byte-wide, 128B-swizzled slab of 64 dims per load; pool
// layout [N, B, Hkv, D]) completing on the stage's mbarrier.  When the current
// unit has no chunk left to load, the warp keeps loading its chunks of the
// next unit, so the ring stays full across unit boundaries and merges.
//
// Arithmetic per chunk, on the tensor cores (warp-level m16n8k16, fp32
// accumulate), with the chunk's tokens as rows:
//   S^T = K Q^T    A = K tile (ldmatrix), B = Q^T fragments kept in registers
//   online softmax per query head (column), exp2 domain, fp32
//   O^T += V^T P^T A = V tile (ldmatrix.trans), B = P^T from the S^T
//                  fragments by an in-register 8x8 transpose (movmatrix)
// P is fed as two 16-bit pieces (hi + lo) so that P.V keeps about 16 mantissa
// bits; Q.K products of 16-bit inputs are exact in fp32.  The running maximum
// used for the exponentials is raised only when a score exceeds it by more
// than RESCALE_SLACK (exact: O and L always share the reference).  Slots at
// or past the context length are masked before the max, and their V rows are
// zeroed in shared memory, so whatever bytes they hold never reach the result.
//
// End of a unit: the four warps' (max, sum, O) states merge in shared memory,
// four heads per round.  A one-partition sequence writes out = O / L.
// Otherwise the unit writes its unnormalised (M, L, O) record and bumps the
// sequence's completion counter; the CTA that completes the last partition
// merges all records: o = sum_p e^(M_p - M) O_p / sum_p e^(M_p - M) L_p.
// Normalising each partition and adding the results would be wrong
// ("PagedAttention" (tensortonic), section 5).  No CTA ever waits on another.
#pragma once

#include <math.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

constexpr int max_c(int a, int b) { return a > b ? a : b; }
constexpr int min_c(int a, int b) { return a < b ? a : b; }
constexpr int round_up_c(int v, int a) { return (v + a - 1) / a * a; }

constexpr int DECODE_WARPS = 4;
constexpr int SMEM_PER_SM = 228 * 1024;   // shared memory of one SM
constexpr int SMEM_RESERVED = 1024;       // reserved by the system per CTA
constexpr int MERGE_HEADS = 4;            // query heads merged per round
constexpr int MERGE_BATCH = 16;           // partition records fetched together by a final merge

// Softmax reference-max slack (log2 domain): P stays <= 2^8 and the rescale
// of O is rare.
constexpr float RESCALE_SLACK = 8.0f;

template <int D>
constexpr int stage_bytes_c() { return 2 * (D / 64) * 2048; }
template <int D>
constexpr int merge_bytes_c() { return DECODE_WARPS * MERGE_HEADS * (D + 2) * 4; }
template <int D>
constexpr int smem_bytes_c(int stages) {
  return 1024 + round_up_c(DECODE_WARPS * stages * stage_bytes_c<D>(), 1024) +
         merge_bytes_c<D>() + DECODE_WARPS * stages * 8 + 64;
}
template <int D>
constexpr bool fits_c(int stages, int occ) {
  return (smem_bytes_c<D>(stages) + SMEM_RESERVED) * occ <= SMEM_PER_SM;
}
// CTAs per SM: 3 when two stages per warp fit and the registers allow it
// (one 8-head tile), else 2.
template <int D, int NH>
constexpr int occupancy_c() { return (NH == 1 && fits_c<D>(2, 3)) ? 3 : 2; }
// Stages per warp: as many as fit (2..4).
template <int D, int NH>
constexpr int stages_c() {
  return fits_c<D>(4, occupancy_c<D, NH>()) ? 4 : (fits_c<D>(3, occupancy_c<D, NH>()) ? 3 : 2);
}

template <typename T, int D, int B, int NH>
struct DecodeCfg {
  static constexpr int NW = DECODE_WARPS;
  static constexpr int HEADS = 8 * NH;           // query heads per CTA (MMA N)
  static constexpr int OCC = occupancy_c<D, NH>();
  static constexpr int STAGES = stages_c<D, NH>();
  static constexpr int CH = min_c(B, 16);        // tokens per chunk (one TMA box high)
  static constexpr int NCH = B / CH;             // chunks per block
  static constexpr int NSUB = D / 64;            // 128-byte column slabs of a row
  static constexpr int KS = D / 16;              // k-steps of K Q^T
  static constexpr int MT = D / 16;              // m-tiles (16 dims) of V^T P^T
  static constexpr int SUB_BYTES = 16 * 128;     // one slab: 16 rows x 128 B, 128B-swizzled
  static constexpr int CHUNK_BYTES = NSUB * SUB_BYTES;   // K (or V) of one chunk
  static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;    // K + V
  static constexpr int TX_BYTES = 2 * NSUB * CH * 128;   // bytes the TMA loads deliver
  static constexpr int STAGES_BYTES = round_up_c(NW * STAGES * STAGE_BYTES, 1024);
  static constexpr int MERGE_FLOATS = NW * MERGE_HEADS * (D + 2);
  static constexpr int SMEM_BYTES = smem_bytes_c<D>(STAGES);
  // Grouped form (WG groups of NW warps in one CTA, each an independent
  // decoder with its own shared memory): the groups' regions, 1 KiB apart.
  static constexpr int GROUP_STRIDE = round_up_c(SMEM_BYTES - 1024, 1024);
  static constexpr int smem_for(int wg) { return wg == 1 ? SMEM_BYTES : 1024 + wg * GROUP_STRIDE; }

  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(B == 4 || B == 8 || B == 16 || B == 32, "block_size");
  static_assert(NH == 1 || NH == 2, "query head tiles");
  static_assert(STAGE_BYTES == stage_bytes_c<D>(), "stage size");
  static_assert(fits_c<D>(STAGES, OCC), "shared memory budget");
};

__device__ __forceinline__ int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

// ---------------------------------------------------------------------------
// Work list: one CTA of 1024 threads.  First the full partitions of the
// sequences that span several partitions (in sequence order), then their
// shorter last partitions, then the sequences that fit in one partition; the
// last two groups longest first (a counting sort over PLAN_BUCKETS / 2
// length classes each).  So the units handed out last are the shortest, and
// they merge no partitions (a one-partition sequence writes its output
// directly): the CTAs run out of work at nearly the same time.  The order
// changes no result: every unit is computed the same way wherever it runs,
// and a sequence's records are merged in partition order.
constexpr int PLAN_BUCKETS = 1024;

// Length class of r blocks (0 < r < pb) among nbk <= pb classes: the longer,
// the lower.
__device__ __forceinline__ int plan_bucket(int r, int pb, int nbk) {
  return (int)((long long)(pb - r) * nbk / pb);
}

static __global__ void __launch_bounds__(1024, 1) decode_plan_kernel(const DecodeParams p) {
  __shared__ int wsum[32];
  __shared__ int slot[PLAN_BUCKETS];   // last partitions per length class, then the next free slot
  pdl_launch_dependents();   // the attention grid may start its prologue
  pdl_wait_predecessors();   // context_lens / out may come from earlier kernels
  const int S = p.num_seqs, PB = p.part_blocks, Bs = p.block_size;
  const int cap = p.max_blocks * Bs;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (S + 1023) / 1024;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  const int nbk = min(PB, PLAN_BUCKETS / 2);
  // the class of a sequence's item that does not come first: the last
  // partition (r blocks) of a longer sequence, or the whole of a sequence of
  // at most PB blocks
  auto cls = [=](int nb) {
    return nb > PB ? plan_bucket(nb % PB, PB, nbk) : nbk + plan_bucket(nb, PB + 1, nbk);
  };
  // a mixed batch: only the sequences with exactly one query row are this
  // kernel's; one whose row lies outside q, or whose context cannot hold it,
  // is flagged and skipped
  auto mine = [&](int s, bool flag) -> bool {
    if (!p.query_start) return true;
    const int a = __ldg(p.query_start + s), b = __ldg(p.query_start + s + 1);
    if (b - a != 1) return false;
    if (a < 0 || b > p.num_tokens || __ldg(p.context_lens + s) < 1) {
      if (flag) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
      return false;
    }
    return true;
  };
  slot[tid] = 0;
  __syncthreads();
  int nf = 0;
  // (overlap) decode tokens and visible (query, key) pairs of the chunks, exact
  long long dec_tok = 0, ch_pairs = 0;
  for (int s = s0; s < s1; ++s) {
    if (p.overlap) {
      const int a = __ldg(p.query_start + s), n = __ldg(p.query_start + s + 1) - a;
      const int Lc = clamp_len(__ldg(p.context_lens + s), cap);
      if (n == 1) dec_tok += Lc;
      else if (n >= 2 && Lc >= n)
        ch_pairs += (long long)n * (Lc - n + 1) + (long long)n * (n - 1) / 2;
    }
    if (!mine(s, true)) continue;
    const int L0 = __ldg(p.context_lens + s);
    if (L0 < 0 || L0 > cap) atomicOr(p.flags, PKV_FLAG_LEN_RANGE);
    const int nb = (clamp_len(L0, cap) + Bs - 1) / Bs;
    if (nb > PB) nf += nb / PB;
    if (nb > 0 && (nb <= PB || nb % PB)) atomicAdd(&slot[cls(nb)], 1);
  }
  __syncthreads();
  // block-wide exclusive scans: first-group partitions per thread, the other
  // items per class (thread t holds class t)
  const int np = slot[tid];
  int xf = nf, xp = np;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int yf = __shfl_up_sync(FULL_MASK, xf, off);
    const int yp = __shfl_up_sync(FULL_MASK, xp, off);
    if (lane >= off) { xf += yf; xp += yp; }
  }
  __shared__ int wsum_p[32];
  if (lane == 31) { wsum[wid] = xf; wsum_p[wid] = xp; }
  __syncthreads();
  if (wid == 0) {
    int tf = wsum[lane], tp = wsum_p[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int yf = __shfl_up_sync(FULL_MASK, tf, off);
      const int yp = __shfl_up_sync(FULL_MASK, tp, off);
      if (lane >= off) { tf += yf; tp += yp; }
    }
    wsum[lane] = tf;   // inclusive over warps
    wsum_p[lane] = tp;
  }
  __syncthreads();
  const int total_f = wsum[31], total_p = wsum_p[31];
  int fo = xf - nf + (wid ? wsum[wid - 1] : 0);
  slot[tid] = total_f + xp - np + (wid ? wsum_p[wid - 1] : 0);
  __syncthreads();
  for (int s = s0; s < s1; ++s) {
    if (!mine(s, false)) continue;
    const int L = clamp_len(__ldg(p.context_lens + s), cap);
    const int nb = (L + Bs - 1) / Bs;
    const int F = nb > PB ? nb / PB : 0;
    for (int q = 0; q < F; ++q) p.items[fo++] = make_int2(s, q);
    if (nb > 0 && (nb <= PB || nb % PB)) p.items[atomicAdd(&slot[cls(nb)], 1)] = make_int2(s, F);
    if (L == 0) {   // nothing to attend to: zeros
      const size_t base = (size_t)s * p.num_q_heads * p.head_dim;
      for (int e = 0; e < p.num_q_heads * p.head_dim; ++e)
        store_out(p.out, base + e, p.out_dtype, 0.f);
    }
  }
  for (int i = tid; i < S * p.num_hc; i += 1024) p.seq_done[i] = 0u;
  unsigned active = (unsigned)p.grid;
  if (p.overlap) {
    // The decode pass's share of the SMs when the chunked pass runs beside
    // it.  With x SMs the decode rows' K/V stream at
    //   bw(x) = min(per_sm * x, peak * x / (x + half))
    // (linear while each SM's own rate binds, then saturating), and the
    // chunks' query-key pairs run at a fixed tensor rate on the other M - x.
    // Every x in [1, M) is tried (one thread each) for the smallest
    // max(decode time, chunked time); unless that beats running the passes
    // in turn by ovl_margin, the decode pass takes every SM (and the chunked
    // CTAs follow as its CTAs leave).
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      dec_tok += __shfl_xor_sync(FULL_MASK, dec_tok, off);
      ch_pairs += __shfl_xor_sync(FULL_MASK, ch_pairs, off);
    }
    __shared__ long long red[2][32];
    __shared__ unsigned long long best[32];
    if (lane == 0) { red[0][wid] = dec_tok; red[1][wid] = ch_pairs; }
    __syncthreads();
    long long dt = 0, cp = 0;
    for (int i = 0; i < 32; ++i) { dt += red[0][i]; cp += red[1][i]; }   // every thread
    const float bytes = (float)dt * (float)(p.num_kv_heads * p.head_dim * 4);   // K + V, 2 B
    const float flops = (float)cp * (float)(p.num_q_heads * p.head_dim * 4);
    const int M = p.ovl_sms;
    auto bw = [&](float x) { return fminf(p.ovl_sm_bps * x, p.ovl_peak_bps * x / (x + p.ovl_half_sms)); };
    // key: the time's bits (non-negative floats order as unsigned) above x
    unsigned long long key = ~0ull;
    for (int x = tid + 1; x < M; x += 1024) {
      const float t = fmaxf(bytes / bw((float)x), flops / ((float)(M - x) * p.ovl_flops_sm));
      const unsigned long long k = ((unsigned long long)__float_as_uint(t) << 32) | (unsigned)x;
      key = k < key ? k : key;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(FULL_MASK, key, off);
      key = o < key ? o : key;
    }
    if (lane == 0) best[wid] = key;
    __syncthreads();
    if (tid == 0) {
      for (int i = 1; i < 32; ++i) key = best[i] < key ? best[i] : key;
      const int gcta = p.grid / p.ovl_wg;   // decode CTAs launched
      int xi = gcta;                        // the passes in turn
      if (bytes <= 0.f) xi = 0;             // no decode rows: every SM to the chunks
      else if (flops > 0.f && key != ~0ull) {
        const float t_best = __uint_as_float((unsigned)(key >> 32));
        const float t_turn = bytes / bw((float)M) + flops / ((float)M * p.ovl_flops_sm);
        if (t_best < (1.f - p.ovl_margin) * t_turn) xi = (int)(key & 0xffffffffu);
      }
      xi = xi > gcta ? gcta : xi;
      active = (unsigned)(xi * p.ovl_wg);
    }
  }
  if (tid == 0) {
    // CTA c of the attention grid starts with units c and c + (CTAs running)
    // without asking; the counter hands out the rest
    p.ctrl[0] = 2u * active;
    p.ctrl[1] = (unsigned)(total_f + total_p) * (unsigned)p.num_hc;
    p.ctrl[2] = active;   // decoders that run (all, unless a chunked pass runs beside)
    p.ctrl[WS_CTRL_CHUNKED_DONE] = 0u;   // chunked CTAs finished (when it does)
  }
}

// ---------------------------------------------------------------------------
// A warp's view of one work unit for loading: which blocks (and chunks) it
// streams and its slice of the block table.
struct WarpLoads {
  int s;            // sequence
  int row;          // its row of q and out
  int part;         // partition
  int hc;           // KV head x query-head chunk index
  int L;            // context length (clamped)
  bool append;      // position L - 1 comes from the step's new K/V rows
  int kvh;          // KV head
  int j0;           // first block of this warp
  int n_w;          // blocks of this warp
  int n_units;      // chunks of this warp
  int issued;       // chunks already issued
  int kbase;        // first warp-block index held in `tbl`
  int tbl;          // lane i: physical block of warp-block kbase + i
  const int32_t *trow;
};

// `item` = the work list's entry unit / num_hc.
template <int B, int NCH, int CH, int NW>
__device__ __forceinline__ void decode_unit_loads(WarpLoads &wl, const DecodeParams &p,
                                                  unsigned unit, int2 item, int w, int lane) {
  const int HC = p.num_hc;
  const int hc = (int)(unit % HC);
  const int s = item.x, part = item.y;
  const int L0 = __ldg(p.context_lens + s);
  const int L = clamp_len(L0, p.max_blocks * B);
  const int nb = (L + B - 1) / B;
  const int jb = part * p.part_blocks;
  const int je = min(nb, jb + p.part_blocks);
  wl.s = s;
  wl.row = p.query_start ? __ldg(p.query_start + s) : s;
  wl.part = part;
  wl.hc = hc;
  wl.L = L;
  wl.append = p.key_new != nullptr && L0 >= 1 && L0 == L;
  wl.kvh = hc / p.num_gchunks;
  wl.j0 = jb + w;
  wl.n_w = wl.j0 < je ? (je - wl.j0 + NW - 1) / NW : 0;
  wl.n_units = wl.n_w * NCH;
  if (NCH > 1 && wl.n_w > 0 && wl.j0 + (wl.n_w - 1) * NW == nb - 1) {
    const int tail = L - (nb - 1) * B;   // tokens in the last block
    wl.n_units -= NCH - (tail + CH - 1) / CH;
  }
  wl.issued = 0;
  wl.kbase = 0;
  wl.trow = p.block_tables + (size_t)s * p.max_blocks;
  wl.tbl = lane < wl.n_w ? __ldg(wl.trow + wl.j0 + lane * NW) : 0;
}

// Q^T of one unit as MMA B fragments (k: dims, n: heads); heads past the
// group are zero.
template <typename T, int D, int NH, int HEADS>
__device__ __forceinline__ void load_q_frags(uint32_t (&qb)[D / 16][NH][2], const DecodeParams &p,
                                             const WarpLoads &wl, int cr, int cq) {
  const int gc = wl.hc - wl.kvh * p.num_gchunks;
  const int g0 = gc * HEADS;
  const int gcount = min(HEADS, p.group - g0);
  const T *qp = static_cast<const T *>(p.q) +
                ((size_t)wl.row * p.num_q_heads + wl.kvh * p.group + g0) * D;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int head = 8 * nh + cr;
        const int kk = ks * 16 + cq + 8 * e;
        qb[ks][nh][e] =
            head < gcount ? __ldg(reinterpret_cast<const unsigned int *>(qp + head * D + kk)) : 0u;
      }
}

// ---------------------------------------------------------------------------
// WG = 1: one decoder per CTA (several CTAs per SM).  WG = 3: three
// decoders of NW warps each in one CTA that takes a whole SM -- the form a
// mixed batch uses, so that the decode pass holds whole SMs and the chunked
// pass can run on the others at the same time.  Each group works exactly as
// a CTA of the WG = 1 form (own shared memory, own barrier, own units); only
// the group-wide barrier and the virtual CTA index differ.
template <typename T, int D, int B, int NH, int WG>
__global__ void __launch_bounds__(DECODE_WARPS * 32 * WG, WG == 1 ? occupancy_c<D, NH>() : 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using C = DecodeCfg<T, D, B, NH>;
  constexpr int NW = C::NW;
  constexpr int STAGES = C::STAGES;
  static_assert(WG == 1 || (NH == 1 && C::OCC == 3), "grouped form: one 8-head tile, 3 per SM");
  extern __shared__ unsigned char smem_raw[];
  const int wg = WG == 1 ? 0 : (int)(threadIdx.x / (NW * 32));
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023)) + wg * C::GROUP_STRIDE;
  // the group's barrier: the whole CTA in the WG = 1 form, else named
  // barrier 1 + wg over the group's NW warps
  auto group_sync = [&]() {
    if (WG == 1) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"r"(1 + wg), "r"(NW * 32) : "memory");
  };
  const uint32_t stage_smem = smem_addr(smem);
  float *mg_o = reinterpret_cast<float *>(smem + C::STAGES_BYTES);      // [NW][4][D]
  float *mg_ml = mg_o + NW * MERGE_HEADS * D;                          // [NW][4][2]
  uint64_t *bars = reinterpret_cast<uint64_t *>(mg_o + C::MERGE_FLOATS);
  // s_int[0..2]: ring of upcoming unit ids, s_int[3]: abort, s_int[4]: last
  volatile int *s_int = reinterpret_cast<volatile int *>(bars + NW * STAGES);

  const int tid = (int)threadIdx.x - wg * NW * 32;   // thread within the group
  const int lane = tid & 31, w = tid >> 5;
  const int HC = p.num_hc;

  // Rows a chunk never loads (block_size < 16) must read as zeros in P.V.
  if (C::CH < 16) {
    for (int i = tid; i < C::STAGES_BYTES / 16; i += NW * 32)
      *reinterpret_cast<uint4 *>(smem + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  if (tid == 0) {
#pragma unroll 1
    for (int i = 0; i < NW * STAGES; ++i) mbar_init(smem_addr(bars + i), 1);
    s_int[3] = 0;
    fence_barrier_init();
  }
  if (tid == 32 || (NW == 1 && tid == 0)) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  // everything above is local; the work list, the pool and q come from the
  // kernels before this one
  pdl_wait_predecessors();
  // Decoders (groups) of the grid: vb is this one's index.  The grouped form
  // runs only the first ctrl[2] of them (the work list's share of the SMs):
  // it lets the next kernel on the stream start now, and a CTA with no
  // running group leaves at once so that its SM goes to that kernel.
  const unsigned vb = blockIdx.x * WG + wg;
  unsigned vgrid = gridDim.x * WG;
  if (WG > 1) {
    vgrid = __ldcg(p.ctrl + 2);
    pdl_launch_dependents();
    if (blockIdx.x * WG >= vgrid) return;
  }
  // The first two units need no atomic (the counter starts past them), and
  // their work-list entries are fetched together with the unit count (an
  // entry past the list is read, from inside the array, but never used).
  unsigned cur_unit = vb < vgrid ? vb : 0xFFFFFFFFu;
  unsigned nxt_unit = vb < vgrid ? vb + vgrid : 0xFFFFFFFFu;
  const size_t last_item = (size_t)p.num_seqs * p.max_parts - 1;
  const int2 item0 = __ldcg(p.items + min((size_t)(cur_unit / HC), last_item));
  const int2 item1 = __ldcg(p.items + min((size_t)(nxt_unit / HC), last_item));
  const unsigned total = __ldcg(p.ctrl + 1);
  group_sync();

  const uint32_t wst = stage_smem + w * STAGES * C::STAGE_BYTES;
  const uint32_t bar0 = smem_addr(bars + w * STAGES);
  const uint64_t pol = l2_policy_evict_first();
  uint32_t ld_cnt = 0, use_cnt = 0;   // this warp's loads issued / consumed, all units

  // fragment coordinates of this lane
  const int cr = lane >> 2;              // C row (token, or dim within an m-tile)
  const int cq = 2 * (lane & 3);         // C columns (query heads) cq, cq + 1
  const int a_tok = ((lane >> 3) & 1) * 8 + (lane & 7);   // ldmatrix row for K (A operand)
  const int a_chb = (lane >> 4) & 1;
  const int v_tok = ((lane >> 4) & 1) * 8 + (lane & 7);   // ldmatrix row for V (A, trans)
  const int v_chb = (lane >> 3) & 1;

  WarpLoads cur, nxt;
  if (cur_unit < total) decode_unit_loads<B, C::NCH, C::CH, NW>(cur, p, cur_unit, item0, w, lane);
  if (nxt_unit < total) decode_unit_loads<B, C::NCH, C::CH, NW>(nxt, p, nxt_unit, item1, w, lane);

  auto issue_chunk = [&](WarpLoads &wl) {
    const int u = wl.issued++;
    const int i = u / C::NCH;
    const int c = u - i * C::NCH;
    if (i - wl.kbase >= 32) {
      wl.kbase += 32;
      wl.tbl = wl.kbase + lane < wl.n_w ? __ldg(wl.trow + wl.j0 + (wl.kbase + lane) * NW) : 0;
    }
    const int pb = __shfl_sync(FULL_MASK, wl.tbl, i - wl.kbase);
    if (lane == 0) {
      if ((unsigned)pb >= (unsigned)p.num_blocks) atomicOr(p.flags, PKV_FLAG_BLOCK_RANGE);
      const int stage = (int)(ld_cnt % STAGES);
      const uint32_t bar = bar0 + stage * 8;
      const uint32_t dst = wst + stage * C::STAGE_BYTES;
      mbar_arrive_expect_tx(bar, C::TX_BYTES);
      // out-of-range block ids read as zeros (TMA bounds), never fault
#pragma unroll
      for (int sb = 0; sb < C::NSUB; ++sb) {
        tma_load_4d(dst + sb * C::SUB_BYTES, &kmap, sb * 64, wl.kvh, c * C::CH, pb, bar, pol);
        tma_load_4d(dst + C::CHUNK_BYTES + sb * C::SUB_BYTES, &vmap, sb * 64, wl.kvh,
                    c * C::CH, pb, bar, pol);
      }
    }
    ++ld_cnt;
  };
  // Keep STAGES chunks in flight: the current unit's first, then the next's.
  auto top_up = [&](bool have_cur, bool have_nxt) {
    while (ld_cnt - use_cnt < (uint32_t)STAGES) {
      if (have_cur && cur.issued < cur.n_units) issue_chunk(cur);
      else if (have_nxt && nxt.issued < nxt.n_units) issue_chunk(nxt);
      else break;
    }
  };
  top_up(cur_unit < total, nxt_unit < total);

  // query fragments of the current unit; the next unit's are loaded one unit
  // ahead so that a unit starts without waiting for them
  uint32_t qb[C::KS][NH][2], qb_next[C::KS][NH][2];
  if (cur_unit < total) load_q_frags<T, D, NH, C::HEADS>(qb, p, cur, cr, cq);

  int qn = 2;   // ring slot the next atomicAdd result goes to
  bool ok = true;
#pragma unroll 1
  while (cur_unit < total) {
    // the unit after `nxt_unit`; visible to all after this unit's merge barriers
    if (tid == 0) s_int[qn] = (int)atomicAdd(p.ctrl, 1u);

    if (nxt_unit < total) load_q_frags<T, D, NH, C::HEADS>(qb_next, p, nxt, cr, cq);
    const int s = cur.s, part = cur.part, hc = cur.hc, L = cur.L;
    const int kvh = cur.kvh;
    const int gc = hc - kvh * p.num_gchunks;
    const int nb = (L + B - 1) / B;
    const int nparts = (nb + p.part_blocks - 1) / p.part_blocks;
    const int g0 = gc * C::HEADS;
    const int gcount = min(C::HEADS, p.group - g0);
    const int hq0 = kvh * p.group + g0;
    const size_t out_base = ((size_t)cur.row * p.num_q_heads + hq0) * D;

    // Appending: the warp whose blocks include position L - 1 fetches this
    // step's K (lanes 0..D/8-1) or V (the next D/8 lanes) row piece now, so
    // the load is long done when that chunk comes up.
    constexpr int PIECES = D / 8;              // 16-byte pieces of one row
    const bool app_warp = cur.append && cur.n_w > 0 && cur.j0 + (cur.n_w - 1) * NW == nb - 1;
    uint4 app_val = make_uint4(0u, 0u, 0u, 0u);
    if (app_warp && lane < 2 * PIECES) {
      const bool isv = lane >= PIECES;
      const T *src = static_cast<const T *>(isv ? p.value_new : p.key_new) +
                     ((size_t)s * p.num_kv_heads + kvh) * D;
      app_val = __ldg(reinterpret_cast<const uint4 *>(src) + (isv ? lane - PIECES : lane));
    }

    // softmax state of heads 8nh + cq + {0, 1}
    float mr[NH][2], lr[NH][2];
    float o[NH][C::MT][4];
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
      mr[nh][0] = mr[nh][1] = -INFINITY;
      lr[nh][0] = lr[nh][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nh][mt][e] = 0.f;
    }

#pragma unroll 1
    for (int u = 0; u < cur.n_units; ++u) {
      const uint32_t stage = use_cnt % STAGES;
      const bool got = mbar_wait_bounded(bar0 + stage * 8, (use_cnt / STAGES) & 1u);
      if (!__all_sync(FULL_MASK, got)) {
        ok = false;
        break;
      }
      const int i = u / C::NCH;
      const int c = u - i * C::NCH;
      const int j = cur.j0 + i * NW;
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
      if (app_warp && j * B + c * C::CH + valid == L) {
        // this step's token (position L - 1, row valid - 1 of the chunk): its
        // K and V rows come from the step's inputs, whatever the slot holds,
        // and the unit of query-head chunk 0 stores them in the pool.  No
        // unit of this call takes that slot's bytes from the pool.
        const int row = valid - 1;
        if (lane < 2 * PIECES) {
          const bool isv = lane >= PIECES;
          const int pc = isv ? lane - PIECES : lane;
          const int sb = pc >> 3, ch = pc & 7;
          const uint4 val = app_val;
          unsigned char *base = smem + ((isv ? vb : kb) - stage_smem);
          *reinterpret_cast<uint4 *>(base + sb * C::SUB_BYTES + row * 128 + ((ch ^ (row & 7)) << 4)) =
              val;
          if (gc == 0) {
            const int pb = __ldg(cur.trow + j);
            if ((unsigned)pb < (unsigned)p.num_blocks) {   // a bad id was flagged at load
              const size_t dst = (((size_t)pb * B + (L - 1) % B) * p.num_kv_heads + kvh) * D;
              reinterpret_cast<uint4 *>(static_cast<T *>(isv ? p.v_pool : p.k_pool) + dst)[pc] =
                  val;
            }
          }
        }
        fence_proxy_async_smem();   // before a later TMA load refills this stage
        __syncwarp();
      }

      // S^T = K Q^T: rows = the chunk's tokens, columns = query heads
      float sa[NH][4];
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[nh][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        const int sb = ks >> 2;
        const int ch = (ks & 3) * 2 + a_chb;
        uint32_t a[4];
        ldsm_x4(a, kb + sb * C::SUB_BYTES + a_tok * 128 + ((ch ^ (a_tok & 7)) << 4));
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) Mma<T>::run(sa[nh], a, qb[ks][nh][0], qb[ks][nh][1]);
      }

      // online softmax per head (column), exp2 domain, lazily raised reference
      const bool v0 = cr < valid, v1 = cr + 8 < valid;
      bool up_any = false;
      float mx[NH][2];
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {
        sa[nh][0] = v0 ? sa[nh][0] * p.scale_log2 : -INFINITY;
        sa[nh][1] = v0 ? sa[nh][1] * p.scale_log2 : -INFINITY;
        sa[nh][2] = v1 ? sa[nh][2] * p.scale_log2 : -INFINITY;
        sa[nh][3] = v1 ? sa[nh][3] * p.scale_log2 : -INFINITY;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float x = fmaxf(sa[nh][hh], sa[nh][hh + 2]);
          x = fmaxf(x, __shfl_xor_sync(FULL_MASK, x, 4));
          x = fmaxf(x, __shfl_xor_sync(FULL_MASK, x, 8));
          x = fmaxf(x, __shfl_xor_sync(FULL_MASK, x, 16));
          mx[nh][hh] = x;
          up_any |= x > mr[nh][hh] + RESCALE_SLACK;
        }
      }
      if (__any_sync(FULL_MASK, up_any)) {
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
          float a2[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float nm = mx[nh][hh] > mr[nh][hh] + RESCALE_SLACK ? mx[nh][hh] : mr[nh][hh];
            a2[hh] = fast_exp2(mr[nh][hh] - nm);
            mr[nh][hh] = nm;
            lr[nh][hh] *= a2[hh];
          }
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            o[nh][mt][0] *= a2[0];
            o[nh][mt][1] *= a2[1];
            o[nh][mt][2] *= a2[0];
            o[nh][mt][3] *= a2[1];
          }
        }
      }
      uint32_t bh[NH][2], bl[NH][2];
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {
        const float p0 = fast_exp2(sa[nh][0] - mr[nh][0]), p1 = fast_exp2(sa[nh][1] - mr[nh][1]);
        const float p2 = fast_exp2(sa[nh][2] - mr[nh][0]), p3 = fast_exp2(sa[nh][3] - mr[nh][1]);
        lr[nh][0] += p0 + p2;
        lr[nh][1] += p1 + p3;
        // P^T rows (tokens) as 16-bit pairs, hi and lo pieces, transposed into
        // B fragments (k: tokens, n: heads)
        const uint32_t ht = Mma<T>::pack(p0, p1), hb = Mma<T>::pack(p2, p3);
        const float2 ft = Widen<T>::pair(ht), fb = Widen<T>::pair(hb);
        const uint32_t lt = Mma<T>::pack(p0 - ft.x, p1 - ft.y);
        const uint32_t lb = Mma<T>::pack(p2 - fb.x, p3 - fb.y);
        bh[nh][0] = movmatrix_trans(ht);
        bh[nh][1] = movmatrix_trans(hb);
        bl[nh][0] = movmatrix_trans(lt);
        bl[nh][1] = movmatrix_trans(lb);
      }

      // O^T += V^T P^T: rows = dims (m-tiles of 16), columns = query heads
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) {
        const int sb = mt >> 2;
        const int ch = (mt & 3) * 2 + v_chb;
        uint32_t a[4];
        ldsm_x4_trans(a, vb + sb * C::SUB_BYTES + v_tok * 128 + ((ch ^ (v_tok & 7)) << 4));
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
          Mma<T>::run(o[nh][mt], a, bh[nh][0], bh[nh][1]);
          Mma<T>::run(o[nh][mt], a, bl[nh][0], bl[nh][1]);
        }
      }
      __syncwarp();   // every lane's reads of this stage have returned
      ++use_cnt;
      top_up(true, nxt_unit < total);
    }

    if (!ok && lane == 0) {
      atomicOr(p.flags, PKV_FLAG_TIMEOUT);
      s_int[3] = 1;
    }

    // ---- merge the four warps' states, MERGE_HEADS heads per round --------
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float x = lr[nh][hh];
        x += __shfl_xor_sync(FULL_MASK, x, 4);
        x += __shfl_xor_sync(FULL_MASK, x, 8);
        x += __shfl_xor_sync(FULL_MASK, x, 16);
        lr[nh][hh] = x;
      }
    for (int h0 = 0; h0 < gcount; h0 += MERGE_HEADS) {
      const int hn = min(MERGE_HEADS, gcount - h0);
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int head = 8 * nh + cq + hh;
          if (head >= h0 && head < h0 + hn) {
            const int slot = w * MERGE_HEADS + (head - h0);
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
              mg_o[slot * D + 16 * mt + cr] = o[nh][mt][hh];
              mg_o[slot * D + 16 * mt + cr + 8] = o[nh][mt][hh + 2];
            }
            if (cr == 0) {
              mg_ml[slot * 2 + 0] = mr[nh][hh];
              mg_ml[slot * 2 + 1] = lr[nh][hh];
            }
          }
        }
      group_sync();
      if (s_int[3] == 0) {
        for (int idx = tid; idx < hn * D; idx += NW * 32) {
          const int g = idx / D;
          const int d = idx - g * D;
          float M = -INFINITY;
#pragma unroll
          for (int x = 0; x < NW; ++x) M = fmaxf(M, mg_ml[(x * MERGE_HEADS + g) * 2]);
          float Lt = 0.f, O = 0.f;
#pragma unroll
          for (int x = 0; x < NW; ++x) {
            const float f = fast_exp2(mg_ml[(x * MERGE_HEADS + g) * 2] - M);
            Lt += f * mg_ml[(x * MERGE_HEADS + g) * 2 + 1];
            O += f * mg_o[(x * MERGE_HEADS + g) * D + d];
          }
          const int head = h0 + g;
          if (nparts == 1) {
            store_out(p.out, out_base + (size_t)head * D + d, p.out_dtype, O / Lt);
          } else {
            const size_t rec = ((size_t)s * p.num_q_heads + hq0 + head) * p.max_parts + part;
            p.part_o[rec * D + d] = O;
            if (d == 0) {
              p.part_ml[rec * 2 + 0] = M;
              p.part_ml[rec * 2 + 1] = Lt;
            }
          }
        }
      }
      group_sync();   // merge slots free again; this round's records written
    }
    const bool abort = s_int[3] != 0;

    // ---- split-context completion: the CTA that wrote a sequence's last
    // partition record merges all of them ------------------------------------
    if (!abort && nparts > 1) {
      if (tid == 0) {
        // release: the records (ordered before this by the barrier) are
        // visible to whoever sees the count; acquire: the last one sees all
        unsigned prev;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(p.seq_done + (size_t)s * HC + hc)
                     : "memory");
        s_int[4] = prev == (unsigned)(nparts - 1);
      }
      group_sync();
      if (s_int[4]) {
        // Each thread takes 4 dims (a float4) of one head and combines that
        // slice of all nparts records, MERGE_BATCH records at a time with
        // every load of a batch in flight: the running sum is rescaled to
        // each batch's maximum, so a merge costs ceil(nparts / MERGE_BATCH)
        // round trips to L2 per slice.
        constexpr int Q4 = D / 4;
        for (int idx = tid; idx < gcount * Q4; idx += NW * 32) {
          const int g = idx / Q4;
          const int d4 = idx - g * Q4;
          const size_t rec0 = ((size_t)s * p.num_q_heads + hq0 + g) * p.max_parts;
          const float2 *mlp = reinterpret_cast<const float2 *>(p.part_ml) + rec0;
          const float4 *op = reinterpret_cast<const float4 *>(p.part_o + rec0 * D) + d4;
          float M = -INFINITY, Lt = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int q0 = 0; q0 < nparts; q0 += MERGE_BATCH) {
            float2 ml[MERGE_BATCH];
            float4 ov[MERGE_BATCH];
#pragma unroll
            for (int i = 0; i < MERGE_BATCH; ++i) {
              if (q0 + i < nparts) {
                ml[i] = __ldcg(mlp + q0 + i);
                ov[i] = __ldcg(op + (size_t)(q0 + i) * Q4);
              } else {
                ml[i] = make_float2(-INFINITY, 0.f);
                ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
            float Mb = M;
#pragma unroll
            for (int i = 0; i < MERGE_BATCH; ++i) Mb = fmaxf(Mb, ml[i].x);
            // exp2(-inf) = 0: the first batch, and padding entries, weigh nothing
            const float a = fast_exp2(M - Mb);
            acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
            Lt *= a;
#pragma unroll
            for (int i = 0; i < MERGE_BATCH; ++i) {
              const float f = fast_exp2(ml[i].x - Mb);
              acc.x += f * ov[i].x;
              acc.y += f * ov[i].y;
              acc.z += f * ov[i].z;
              acc.w += f * ov[i].w;
              Lt += f * ml[i].y;
            }
            M = Mb;
          }
          const float inv = 1.f / Lt;
          const size_t ob = out_base + (size_t)g * D + 4 * d4;
          store_out(p.out, ob + 0, p.out_dtype, acc.x * inv);
          store_out(p.out, ob + 1, p.out_dtype, acc.y * inv);
          store_out(p.out, ob + 2, p.out_dtype, acc.z * inv);
          store_out(p.out, ob + 3, p.out_dtype, acc.w * inv);
        }
      }
    }
    if (abort) break;

    // ---- advance: the next unit becomes current (its first chunks may be
    // in flight already); learn the one after it from the ring -------------
    cur_unit = nxt_unit;
    cur = nxt;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks)
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {
        qb[ks][nh][0] = qb_next[ks][nh][0];
        qb[ks][nh][1] = qb_next[ks][nh][1];
      }
    nxt_unit = (unsigned)s_int[qn];
    qn = qn == 2 ? 0 : qn + 1;
    if (nxt_unit < total)
      decode_unit_loads<B, C::NCH, C::CH, NW>(nxt, p, nxt_unit, __ldcg(p.items + nxt_unit / HC), w,
                                              lane);
    top_up(cur_unit < total, nxt_unit < total);
  }

  // never leave with copies in flight into this CTA's shared memory
  for (; use_cnt < ld_cnt; ++use_cnt)
    (void)mbar_wait_bounded(bar0 + (use_cnt % STAGES) * 8, (use_cnt / STAGES) & 1u);
  if (WG == 1) pdl_launch_dependents();
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

template <typename T, int D, int B, int NH, int WG>
cudaError_t launch_decode_cfg(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeParams &p, cudaStream_t stream, int *launches) {
  using C = DecodeCfg<T, D, B, NH>;
  auto kern = decode_kernel<T, D, B, NH, WG>;
  constexpr int smem = C::smem_for(WG);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  LaunchInfo li;
  e = launch_info(reinterpret_cast<const void *>(kern), C::NW * 32 * WG, smem, dev, &li);
  if (e != cudaSuccess) return e;
  const long long units_max =
      (long long)p.num_seqs * p.max_parts * p.num_hc;   // upper bound on work units
  long long grid = (long long)li.sms * li.ctas_per_sm;   // CTAs
  if (grid * WG > units_max) grid = (units_max + WG - 1) / WG;
  if (grid < 1) grid = 1;
  DecodeParams pg = p;
  pg.grid = (int)grid * WG;   // decoders
  pg.ovl_wg = WG;
  pg.ovl_sms = li.sms;
  e = launch_pdl(decode_plan_kernel, dim3(1), dim3(1024), 0, stream, pg);
  if (e != cudaSuccess) return e;
  ++*launches;
  e = launch_pdl(kern, dim3((unsigned)grid), dim3(C::NW * 32 * WG), smem, stream, kmap, vmap, pg);
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaSuccess;
}

template <typename T, int D, int B>
cudaError_t launch_decode_nh(const CUtensorMap &kmap, const CUtensorMap &vmap,
                             const DecodeParams &p, cudaStream_t stream, int *launches) {
  if (p.group <= 8) {
    // a mixed batch whose chunked pass runs beside: the grouped form
    if (p.overlap) return launch_decode_cfg<T, D, B, 1, 3>(kmap, vmap, p, stream, launches);
    return launch_decode_cfg<T, D, B, 1, 1>(kmap, vmap, p, stream, launches);
  }
  return launch_decode_cfg<T, D, B, 2, 1>(kmap, vmap, p, stream, launches);
}

template <typename T, int D>
cudaError_t launch_decode_b(const CUtensorMap &kmap, const CUtensorMap &vmap,
                            const DecodeParams &p, int block_size, cudaStream_t stream,
                            int *launches) {
  switch (block_size) {
    case 4: return launch_decode_nh<T, D, 4>(kmap, vmap, p, stream, launches);
    case 8: return launch_decode_nh<T, D, 8>(kmap, vmap, p, stream, launches);
    case 16: return launch_decode_nh<T, D, 16>(kmap, vmap, p, stream, launches);
    case 32: return launch_decode_nh<T, D, 32>(kmap, vmap, p, stream, launches);
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
