// Packed / chunked causal prefill attention for sm_103a.
//
// Operation (see include/unip.h): token t of segment s, local index i, attends
// to the segment's P_s cached prefix keys (paged) and to its own tokens
// 0..i.  Sources: "Chunked Prefill" glossary page, section "Como funciona o
// pre-preenchimento segmentado" (chunk = cached K/V of earlier chunks + own
// tokens under a causal mask over absolute positions, SDPA softmax) and
// section "Tecnicas de servico relacionadas" (fixed-size KV pages); the
// Prepacking summary, sections "技术框架"/"关键设计" (block-diagonal mask,
// per-prompt positions).
//
// Design
//   * A device planner (one CTA) validates cu_seqlens / positions, cuts every
//     segment into 128-token items and orders them longest-first by their
//     number of 128-key KV tiles, with light items (prefix-streaming tiles of
//     fewer than 128 valid rows) spread evenly among the heavy ones.
//   * Persistent grid, one CTA per SM: the TMA warp claims work items in that
//     order from a global counter and publishes them to the other roles; the
//     K/V ring, the Q buffers and every barrier run on across items.
//   * One work item = two 128-row query tiles that share every K/V tile.  With an
//     even GQA group G dividing 128, a tile's rows are (token, head) pairs of
//     the G query heads of one kv head (128 / G tokens per tile, so a decode
//     token fills G rows); otherwise 128 tokens of query heads h0 and h0 + 1.
//     A KV tile is either 128 prefix keys (read page by page through the
//     block table) or 128 of the segment's own keys; masks only where a tile
//     crosses the prefix end or a row's own token.
//   * Warp roles: 8 softmax warps per query tile, each owning 16 TMEM lanes
//     (16 query rows, all 128 columns) read with the 16x256b shape, so that
//     4 threads share a row and its maximum and sum need only quad shuffles.
//     Warp 16 is the TMA producer, warp 17 the tcgen05 issuer, warps 18-19
//     share the page copies of prefix tiles with warp 16 (TMA copies issue
//     one after another within a warp).
//   * K and V tiles stream through a 5-slot ring of 128-byte-swizzled TMA
//     tiles; a slot is released by a tcgen05.commit after its last MMA.
//   * TMEM (512 columns): S of each query tile (128 fp32 columns) and O of
//     each query tile (D columns).  P is written back as bf16 pairs over the
//     first 64 columns of its S region and read by the PV MMA from TMEM; V is
//     the MN-major B operand straight from its TMA tile.  Two tiles: the MMA
//     order PV0(j), QK0(j+1), PV1(j), QK1(j+1) lets one tile's softmax run
//     while the other tile's MMAs execute.  One tile: S is double-buffered
//     over both S regions and QK(j+2) runs during the softmax of j.
//   * Online softmax in base 2 with a lazy rescale: the running maximum is
//     only moved (and O rescaled in TMEM) when a row's maximum grows by more
//     than 8 (log2 units), which bounds P by 2^8; the final O / l is exact.
//     The epilogue reads O in the same 16x256b layout, so each thread holds
//     its rows' statistics and no shared-memory exchange is needed.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <queue>
#include <vector>

#include "unip_attention_common.cuh"
#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kHistBins = 4096;
constexpr int kPlanThreads = 1024;
constexpr int kWsHeaderBytes = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;  // first TMEM column of the O accumulator
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct AttnArgs {
  CUtensorMap tm_q, tm_qp, tm_k, tm_v, tm_kc, tm_vc;
  const int32_t *cu;
  const int32_t *pos;
  const int32_t *prefix_lens;  // compacted stream: cached prefix length per segment (else the first position)
  const int32_t *block_table;
  const int2 *pairs;
  const int32_t *num_pairs;
  int32_t *work_counter;  // next unclaimed work item (set to 0 by the planner)
  __nv_bfloat16 *out;
  float *lse;
  uint32_t *status;
  int32_t S, N, Hq, group, heads_per_pair, num_pages, page_size, max_pages;
  int32_t lg;  // 0: a tile's rows are 128 tokens of one head; log2(group): rows are (token, head of the group)
  int32_t single;  // 1: every work item is one query tile (calls with too few items to fill the GPU)
  float scale_log2;
};

// ---------------------------------------------------------------------------
// Planner
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads) attn_plan_kernel(const int32_t *__restrict__ cu,
                                                                 const int32_t *__restrict__ pos,
                                                                 const int32_t *__restrict__ prefix_lens, int32_t S,
                                                                 int32_t N, int32_t has_cache, int32_t page_size,
                                                                 int32_t max_pages, int32_t lg,
                                                                 int32_t *__restrict__ header,
                                                                 int2 *__restrict__ pairs, int32_t max_pairs,
                                                                 uint32_t *__restrict__ status) {
  // [0]: heavy pairs (every tile row valid, or no cached prefix), [1]: light ones
  __shared__ int32_t s_hist[2][kHistBins];
  __shared__ int32_t s_scan[32];
  __shared__ int32_t s_base[kPlanThreads + 1];
  __shared__ uint32_t s_err;
  const int tid = threadIdx.x;
  // the attention grid may be scheduled now: it sets itself up, then waits for this plan
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int b = tid; b < 2 * kHistBins; b += kPlanThreads) (&s_hist[0][0])[b] = 0;
  if (tid == 0) s_err = (cu[0] != 0 || cu[S] != N) ? UNIP_DEV_BAD_SEQLENS : 0u;
  __syncthreads();

  // Each thread owns a contiguous range of segments.
  const int per = (S + kPlanThreads - 1) / kPlanThreads;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  // Phase A: cu_seqlens must be non-decreasing (with cu[0] = 0, cu[S] = N every entry is then in range).
  bool mono = true;
  for (int s = s0; s < s1; ++s) mono &= cu[s + 1] >= cu[s];
  if (!mono) atomicOr(&s_err, UNIP_DEV_BAD_SEQLENS);
  __syncthreads();
  if (s_err != 0) {
    if (tid == 0) {
      header[0] = 0;
      header[1] = 0;
      atomicOr(status, s_err);
    }
    return;
  }
  // Phase B: prefixes, pages and positions; count query tiles.
  int32_t my_pairs = 0;
  uint32_t err = 0;
  for (int s = s0; s < s1; ++s) {
    const int32_t n = cu[s + 1] - cu[s];
    if (n == 0) continue;
    const int32_t P = prefix_lens ? prefix_lens[s] : pos[cu[s]];
    if (P < 0 || pos[cu[s]] < 0) err |= UNIP_DEV_BAD_POSITIONS;
    if (P > 0 && (!has_cache || (P + page_size - 1) / page_size > max_pages)) err |= UNIP_DEV_BAD_PAGES;
    my_pairs += (n + kBlockM - 1) / kBlockM;
  }
  // Positions contiguous inside each segment: pos[t] - pos[t-1] == 1 unless t starts a segment.
  // Each thread issues the loads of kPosBatch tokens before it compares any: after an L2 flush the
  // positions come from HBM, and four tokens in flight left a 32k-token call with ~16 dependent
  // rounds of HBM latency in its planner.
  {
    constexpr int kPosBatch = 16;
    for (int t0 = tid; t0 < N; t0 += kPlanThreads * kPosBatch) {
      int32_t prv[kPosBatch], cur[kPosBatch];
#pragma unroll
      for (int u = 0; u < kPosBatch; ++u) {
        const int t = t0 + u * kPlanThreads;
        const bool in = t > 0 && t < N;
        cur[u] = in ? pos[t] : 0;
        prv[u] = in ? pos[t - 1] : 0;
      }
#pragma unroll
      for (int u = 0; u < kPosBatch; ++u) {
        const int t = t0 + u * kPlanThreads;
        // contiguous positions, or (compacted stream) increasing ones
        if (t > 0 && t < N && (prefix_lens ? cur[u] <= prv[u] : cur[u] != prv[u] + 1)) {
          // allowed only at a segment start (some s with cu[s] == t)
          const int32_t s_cur = find_segment(cu, S, t);
          if (cu[s_cur] != t) err |= UNIP_DEV_BAD_POSITIONS;
        }
      }
    }
  }
  if (err) atomicOr(&s_err, err);
  int32_t total_pairs;
  const int32_t my_base = block_excl_scan<int32_t>(my_pairs, s_scan, &total_pairs);
  if (s_err != 0 || total_pairs > max_pairs) {
    if (tid == 0) {
      header[0] = 0;
      header[1] = 0;
      atomicOr(status, s_err ? s_err : UNIP_DEV_BAD_SEQLENS);
    }
    return;
  }
  // Pairs are spread over all threads (one long segment would otherwise sit on one thread):
  // pair p belongs to the thread j with s_base[j] <= p < s_base[j+1], and to one of j's segments.
  s_base[tid] = my_base;
  if (tid == 0) s_base[kPlanThreads] = total_pairs;
  __syncthreads();
  // A pair is light when the first query tile of its CTAs has fewer than 128 valid rows and its
  // keys include a cached prefix (a decode token, a short chunk): such CTAs stream the prefix at
  // HBM speed with an idle tensor pipe.
  auto locate = [&](int32_t p, int32_t &seg, int32_t &m, int32_t &cost, int32_t &light) {
    int32_t lo = 0, hi = kPlanThreads - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (s_base[mid] <= p) lo = mid; else hi = mid - 1;
    }
    int32_t rem = p - s_base[lo];
    for (int32_t sg = min(S, lo * per);; ++sg) {
      const int32_t len = cu[sg + 1] - cu[sg];
      const int32_t nt = (len + kBlockM - 1) / kBlockM;
      if (rem < nt) {
        seg = sg;
        m = rem;
        const int32_t P = prefix_lens ? prefix_lens[sg] : pos[cu[sg]];
        cost = (P + kBlockN - 1) / kBlockN + rem + 1;
        const int32_t tok = len - rem * kBlockM;
        light = (P > 0 && tok < (kBlockM >> lg)) ? 1 : 0;
        return;
      }
      rem -= nt;
    }
  };
  // Histograms of pair costs (number of KV tiles), per class.
  for (int32_t p = tid; p < total_pairs; p += kPlanThreads) {
    int32_t sg, m, cost, light;
    locate(p, sg, m, cost, light);
    atomicAdd(&s_hist[light][min(cost, kHistBins - 1)], 1);
  }
  __syncthreads();
  // Bin start offsets in decreasing cost order: ranks inside each class.
  constexpr int kPer = kHistBins / kPlanThreads;
  int32_t class_total[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    int32_t cnt[kPer];
    int32_t local = 0;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      cnt[r] = s_hist[c][kHistBins - 1 - (tid * kPer + r)];
      local += cnt[r];
    }
    int32_t run = block_excl_scan<int32_t>(local, s_scan, &class_total[c]);
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      s_hist[c][kHistBins - 1 - (tid * kPer + r)] = run;
      run += cnt[r];
    }
  }
  __syncthreads();
  // Merge the two longest-first lists so that both advance at the same rate: heavy rank i sits
  // at fraction i / H of the order and light rank k at k / L (heavy first on ties), so the
  // prefix streaming of light pairs overlaps the tensor work of heavy ones.
  const int64_t H = class_total[0], Lc = class_total[1];
  for (int32_t p = tid; p < total_pairs; p += kPlanThreads) {
    int32_t sg, m, cost, light;
    locate(p, sg, m, cost, light);
    const int64_t r = atomicAdd(&s_hist[light][min(cost, kHistBins - 1)], 1);
    int64_t at = r;
    if (H > 0 && Lc > 0) at = light ? r + (r * H) / Lc + 1 : r + (r * Lc + H - 1) / H;
    pairs[at] = make_int2(sg, m);
  }
  if (tid == 0) {
    header[0] = total_pairs;
    header[1] = 0;  // work counter of the attention grid
  }
}

// ---------------------------------------------------------------------------
// Attention kernel
// ---------------------------------------------------------------------------
constexpr int kStages = 5;        // K/V ring slots (each holds one K or one V tile)
// 4 softmax warpgroups (8 warps per query tile, 16 rows each) + one control
// warpgroup (TMA warp, MMA warp, 2 idle warps); 96 registers per thread.
constexpr int kThreads = 640;
constexpr int kWarpTma = 16;
constexpr int kWarpMma = 17;
constexpr int kWarpAux0 = 18;     // warps 18, 19: extra issuers of paged K/V copies
constexpr int kPageIssuers = 3;   // TMA copies issue one at a time per warp: pages go to 3 warps
constexpr int kUnitSlots = 4;     // published work items in flight (a power of two)
constexpr int kUnitReaders = 19;  // warps that read a published work item: 16 softmax, MMA, 2 helpers

template <int D>
struct SmemLayout {
  static constexpr uint32_t kHalfBytes = kBlockM * 128;    // 128 rows x 128 B (64 bf16)
  static constexpr uint32_t kTileBytes = kBlockM * D * 2;  // one Q / K / V tile
  static constexpr uint32_t kQ0 = 0;
  static constexpr uint32_t kQ1 = kTileBytes;
  static constexpr uint32_t kRing = 2 * kTileBytes;
  static constexpr uint32_t kBytes = kRing + kStages * kTileBytes;
  static constexpr uint32_t kDynamic = kBytes + 1024;      // slack for 1024-byte alignment
};

enum BarId {
  kBarQFull = 0,
  kBarSlotFull0 = 1,                      // + slot
  kBarSlotEmpty0 = 1 + kStages,        // + slot
  kBarSFull0 = 1 + 2 * kStages,        // + tile: S in TMEM
  kBarPFull0 = 3 + 2 * kStages,        // + tile: P in TMEM and O rescaled (both column halves)
  kBarODone0 = 5 + 2 * kStages,        // + tile: last PV done
  kBarFinal = 7 + 2 * kStages,
  kBarPVDone = 8 + 2 * kStages,        // one query tile: each PV done (O may be rescaled)
  kBarQEmpty = 9 + 2 * kStages,        // last QK of a work item done: Q buffers may be reloaded
  kBarOFree0 = 10 + 2 * kStages,       // + tile: epilogue read O (count 256)
  kBarSlotGo0 = 12 + 2 * kStages,      // + slot: a prefix fill of the slot may be issued (helpers)
  kBarUnitFull0 = 12 + 3 * kStages,    // + k: work item i (k = i % kUnitSlots) published in s_unit[k]
  kBarUnitEmpty0 = 16 + 3 * kStages,   // + k: every consumer warp has read s_unit[k]
  kBarSplitStored0 = 20 + 3 * kStages,  // + tile: split epilogue, every thread stored its partial (count 256)
  kBarSplitDecided0 = 22 + 3 * kStages, // + tile: split epilogue, the ticket was taken (count 1)
  kBarTile1Start = 24 + 3 * kStages,    // every warp of tile 1 has started work item i (count 8)
  kNumBars = 25 + 3 * kStages
};

__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}


__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Softmax, P write-back, O rescale and epilogue of one query tile, run by the
// tile's 8 warps.  Warp (q, g) with q = warp % 4 and g = (warp / 4) % 2 owns the
// 16 TMEM lanes 32q + 16g .. 32q + 16g + 15 (16 query rows, all 128 columns)
// and reads them with the 16x256b shape: each thread holds two rows (r, r + 8)
// and two adjacent columns of every 8-column chunk, so a row's maximum and sum
// are completed with two shuffles inside a 4-thread quad.  P goes back into
// the first 64 columns of the tile's S region with the 16x128b shape, in the
// packed layout the PV MMA reads as its A operand.  The epilogue reads O in
// the same layout, so each thread already holds its rows' maximum and sum.

// sb0 / sb1, pvb and ob: completions of S-full 0 / 1, PV-done and this tile's O-done before this
// work item (the barriers run on across the items of a persistent CTA).  Returns false on a timeout.
// Split of a host-planned item whose unit's key range is divided over several items.
struct SplitCtx {
  float *partial;
  unsigned long long *tickets;
  int32_t *last;  // shared memory, one flag per tile
  uint32_t gen;
  int32_t split, nsplit, g0;
};

// Counts this split into the ticket of its (unit, tile); true for the split that completes the
// count.  The ticket carries the launch generation in its upper half, so a count left by an
// earlier launch (or an aborted one) reads as zero.
__device__ __forceinline__ bool split_ticket(unsigned long long *tk, uint32_t gen, int32_t nsplit, uint32_t *status) {
  const unsigned long long tag = static_cast<unsigned long long>(gen) << 32;
  unsigned long long cur = atomicAdd(tk, 0ull);
  for (int it = 0; it < (1 << 20); ++it) {
    const unsigned long long want = ((cur >> 32) == gen) ? cur + 1 : (tag | 1ull);
    const unsigned long long prev = atomicCAS(tk, cur, want);
    if (prev == cur) return static_cast<uint32_t>(want) == static_cast<uint32_t>(nsplit);
    cur = prev;
  }
  atomicOr(status, UNIP_DEV_TIMEOUT);
  return false;
}

// Epilogue of a split item.  Every thread of the tile stores the accumulator values it holds and its
// rows' (m, l) into the split's partial slot; the split that finishes a (unit, tile) last merges the
// slots of all splits in split order (so the result does not depend on which split finished last):
//   M = max_k m_k,  w_k = 2^(m_k - M),  out = sum_k w_k O_k / sum_k w_k l_k,  lse = ln 2 (M + log2 sum_k w_k l_k).
// Warps past the tile's valid rows keep only the barrier protocol.  sep: split epilogues this tile
// ran before (phase of its two split barriers).  Returns false when a bounded wait gave up.
template <int D>
__device__ __noinline__ bool split_epilogue(const AttnArgs &a, const SplitCtx &sp, int tile, const TileRows tr,
                                            bool active, uint32_t tw, uint32_t o_col, uint32_t bar_free,
                                            float m0, float l0, float m1, float l1, int32_t c0, uint64_t *bars,
                                            volatile int *abort_flag, uint32_t sep) {
  using SL = SplitLayout<D>;
  constexpr int kC = SL::kChunks;
  const int lane = threadIdx.x & 31;
  const int t = threadIdx.x & 255;  // thread of the tile's 256 softmax threads
  const int wt = (threadIdx.x >> 5) & 7;
  const int R0 = 32 * (wt & 3) + 16 * (wt >> 2) + (lane >> 2), R1 = R0 + 8;
  const int cq = 2 * (lane & 3);
  auto slot_chunk = [&](int32_t k, int c) {
    const size_t slot = (size_t)(sp.g0 + k) * 2 + tile;
    return reinterpret_cast<float4 *>(sp.partial) + (slot * kC + c) * 256 + t;
  };
  if (active) {
    float o[D / 2];
#pragma unroll
    for (int part = 0; part < D / 32; ++part) tmem_ld_16x256b_x4(tw + o_col + part * 32, o + 16 * part);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(bar_free);  // O is in registers: the next item's first PV may overwrite it
#pragma unroll
    for (int c = 0; c < D / 8; ++c) __stcg(slot_chunk(sp.split, c), make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]));
    __stcg(slot_chunk(sp.split, D / 8), make_float4(m0, l0, m1, l1));
  } else {
    mbar_arrive(bar_free);
  }
  // Every thread's partial is stored before thread 0 counts the split in: the mbarrier orders the
  // tile's stores before thread 0's fence, which makes them visible to the whole GPU before its
  // ticket update (the pattern of a grid-wide barrier).
  const uint32_t bar_stored = smem_u32(&bars[kBarSplitStored0 + tile]);
  const uint32_t bar_decided = smem_u32(&bars[kBarSplitDecided0 + tile]);
  mbar_arrive(bar_stored);
  if (t == 0) {
    const bool ok = mbar_wait(bar_stored, sep & 1, abort_flag, a.status);
    __threadfence();
    sp.last[tile] =
        ok && split_ticket(sp.tickets + (size_t)sp.g0 * 2 + tile, sp.gen, sp.nsplit, a.status) ? 1 : 0;
    __threadfence();
    mbar_arrive(bar_decided);  // also after a timeout, so that no thread of the tile waits for it
  }
  if (!mbar_wait(bar_decided, sep & 1, abort_flag, a.status)) return false;
  if (!sp.last[tile] || !active) return true;
  // Merge.  Loads are batched across splits (independent loads in flight) so that the merge costs a
  // few L2 round trips rather than one per split.
  const int32_t n = sp.nsplit;
  float M0 = -INFINITY, M1 = -INFINITY;
  for (int32_t k0 = 0; k0 < n; k0 += 8) {
    float4 st[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) st[u] = k0 + u < n ? __ldcg(slot_chunk(k0 + u, D / 8)) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      M0 = fmaxf(M0, st[u].x);
      M1 = fmaxf(M1, st[u].z);
    }
  }
  const int32_t tok_r0 = tr.tok0 + (R0 >> tr.lg), tok_r1 = tr.tok0 + (R1 >> tr.lg);
  const int32_t t0 = c0 + tok_r0, t1 = c0 + tok_r1;
  const int32_t hm = (1 << tr.lg) - 1;
  const int32_t h0 = tr.head0 + (R0 & hm), h1 = tr.head0 + (R1 & hm);
  const bool st0 = R0 < tr.rows_valid, st1 = R1 < tr.rows_valid;
  __nv_bfloat16 *o0 = a.out + ((int64_t)t0 * a.Hq + h0) * D + cq;
  __nv_bfloat16 *o1 = a.out + ((int64_t)t1 * a.Hq + h1) * D + cq;
  // chunk c holds columns 8c + cq + {0, 1} of rows R0 (x, y) and R1 (z, w); four chunks at a time,
  // three splits per batch of loads
  constexpr int kG = 4, kB = 3;
  float L0 = 0.f, L1 = 0.f;
#pragma unroll 1
  for (int grp = 0; grp < D / 8 / kG; ++grp) {
    float4 acc[kG];
#pragma unroll
    for (int c = 0; c < kG; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int32_t k0 = 0; k0 < n; k0 += kB) {
      float4 st[kB], v[kB][kG];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const bool in = k0 + u < n;
        st[u] = in ? __ldcg(slot_chunk(k0 + u, D / 8)) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
#pragma unroll
        for (int c = 0; c < kG; ++c)
          v[u][c] = in ? __ldcg(slot_chunk(k0 + u, grp * kG + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const float w0 = ex2_approx(st[u].x - M0), w1 = ex2_approx(st[u].z - M1);
        if (grp == 0) {
          L0 += w0 * st[u].y;
          L1 += w1 * st[u].w;
        }
#pragma unroll
        for (int c = 0; c < kG; ++c) {
          acc[c].x += w0 * v[u][c].x;
          acc[c].y += w0 * v[u][c].y;
          acc[c].z += w1 * v[u][c].z;
          acc[c].w += w1 * v[u][c].w;
        }
      }
    }
    const float inv0 = 1.f / L0, inv1 = 1.f / L1;
#pragma unroll
    for (int c = 0; c < kG; ++c) {
      const int col = 8 * (grp * kG + c);
      if (st0) *reinterpret_cast<uint32_t *>(o0 + col) = pack_bf16x2(acc[c].x * inv0, acc[c].y * inv0);
      if (st1) *reinterpret_cast<uint32_t *>(o1 + col) = pack_bf16x2(acc[c].z * inv1, acc[c].w * inv1);
    }
  }
  if ((lane & 3) == 0 && a.lse) {
    if (st0) a.lse[(int64_t)h0 * a.N + t0] = (M0 + log2f(L0)) * kLn2;
    if (st1) a.lse[(int64_t)h1 * a.N + t1] = (M1 + log2f(L1)) * kLn2;
  }
  return true;
}

// j0: first key tile of this item within its unit's key range (0 unless the range is split).
template <int D, bool db, bool kHost>
__device__ __forceinline__ bool softmax_tile_role(const AttnArgs &a, int tile, const TileRows tr, int32_t j0,
                                                  int32_t T, int32_t Tp, int32_t P, int32_t c0, uint32_t tmem,
                                                  uint64_t *bars, volatile int *abort_flag, uint32_t sb0,
                                                  uint32_t sb1, uint32_t pvb, uint32_t ob, const SplitCtx &sp,
                                                  uint32_t &sep) {
  const int wt = (threadIdx.x >> 5) & 7;
  const int lane = threadIdx.x & 31;
  const int q = wt & 3, g = wt >> 2;
  const uint32_t lane_base = 32 * q + 16 * g;
  const int R0 = lane_base + (lane >> 2), R1 = R0 + 8;  // tile rows held by this thread
  const int cq = 2 * (lane & 3);                         // first column of this thread in a chunk
  const uint32_t tw = tmem + (lane_base << 16);
  // db (one query tile): S and P of KV tile j alternate between the two S regions and their barriers.
  const uint32_t o_col = kTmemO + tile * 128;
  const uint32_t bar_o = smem_u32(&bars[kBarODone0 + tile]);
  const float c = a.scale_log2;
  const int32_t tok_r0 = tr.tok0 + (R0 >> tr.lg), tok_r1 = tr.tok0 + (R1 >> tr.lg);
  // A warp whose 16 rows are all past the tile's valid rows only keeps the barrier protocol.
  const bool active = static_cast<int32_t>(lane_base) < tr.rows_valid;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  for (int32_t j = 0; j < T; ++j) {
    const int buf = db ? (j & 1) : tile;
    const uint32_t par = ((buf ? sb1 : sb0) + static_cast<uint32_t>(db ? (j >> 1) : j)) & 1u;
    const uint32_t s_col = buf * kBlockN;
    const uint32_t bar_p = smem_u32(&bars[kBarPFull0 + buf]);
    if (!mbar_wait(smem_u32(&bars[kBarSFull0 + buf]), par, abort_flag, a.status)) return false;
    if (!active) {
      mbar_arrive(bar_p);
      continue;
    }
    tc_fence_after();
    float sv[64];  // sv[4k + {0,1}]: row R0, columns 8k + cq + {0,1}; sv[4k + {2,3}]: row R1
    tmem_ld_16x256b_x8(tw + s_col, sv);
    tmem_ld_16x256b_x8(tw + s_col + 64, sv + 32);
    tmem_wait_ld();
    const int32_t jg = j0 + j;  // key tile within the unit's range
    if (jg < Tp) {
      if (jg == Tp - 1) {
        const int lim = P - jg * kBlockN;  // keys at or past the prefix end are not cached tokens
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int col = 8 * k + cq;
          if (col >= lim) { sv[4 * k] = -INFINITY; sv[4 * k + 2] = -INFINITY; }
          if (col + 1 >= lim) { sv[4 * k + 1] = -INFINITY; sv[4 * k + 3] = -INFINITY; }
        }
      }
    } else {
      // own keys: key (jg - Tp) * 128 + col is visible to a row whose token index is at least that
      const int32_t lim0 = tok_r0 - (jg - Tp) * kBlockN, lim1 = tok_r1 - (jg - Tp) * kBlockN;
      if (min(lim0, lim1) < kBlockN - 1) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int col = 8 * k + cq;
          if (col > lim0) sv[4 * k] = -INFINITY;
          if (col + 1 > lim0) sv[4 * k + 1] = -INFINITY;
          if (col > lim1) sv[4 * k + 2] = -INFINITY;
          if (col + 1 > lim1) sv[4 * k + 3] = -INFINITY;
        }
      }
    }
    float a0 = fmaxf(sv[0], sv[1]), a1 = fmaxf(sv[4], sv[5]);
    float b0 = fmaxf(sv[2], sv[3]), b1 = fmaxf(sv[6], sv[7]);
#pragma unroll
    for (int k = 2; k < 16; k += 2) {
      a0 = fmax3(a0, sv[4 * k], sv[4 * k + 1]);
      a1 = fmax3(a1, sv[4 * k + 4], sv[4 * k + 5]);
      b0 = fmax3(b0, sv[4 * k + 2], sv[4 * k + 3]);
      b1 = fmax3(b1, sv[4 * k + 6], sv[4 * k + 7]);
    }
    float mx0 = fmaxf(a0, a1), mx1 = fmaxf(b0, b1);
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0 * c), n1 = fmaxf(m1, mx1 * c);
    const bool need0 = n0 > m0 + kRescaleThreshold, need1 = n1 > m1 + kRescaleThreshold;
    float al0 = 1.f, al1 = 1.f;
    if (need0) { al0 = ex2_approx(m0 - n0); m0 = n0; }
    if (need1) { al1 = ex2_approx(m1 - n1); m1 = n1; }
    const float mb0 = (m0 == -INFINITY) ? 0.f : m0, mb1 = (m1 == -INFINITY) ? 0.f : m1;
    float r00 = 0.f, r01 = 0.f, r10 = 0.f, r11 = 0.f;
    // O is rescaled before the PV of this tile accumulates into it.  With two query tiles the PV of
    // the previous KV tile is complete here because S of this one was committed after it; with
    // one (db) S runs ahead, so that PV is waited for.
    if (j >= 1 && __any_sync(0xffffffffu, need0 || need1)) {
      if (db && !mbar_wait(smem_u32(&bars[kBarPVDone]), (pvb + j - 1) & 1, abort_flag, a.status)) return false;
      tc_fence_after();
#pragma unroll 1
      for (int part = 0; part < D / 32; ++part) {
        float o[16];
        tmem_ld_16x256b_x4(tw + o_col + part * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          o[4 * k] *= al0; o[4 * k + 1] *= al0; o[4 * k + 2] *= al1; o[4 * k + 3] *= al1;
        }
        tmem_st_16x256b_x4(tw + o_col + part * 32, o);
      }
    }
    // P in two halves of 64 keys; all of S is already in registers, so P may overwrite it.
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t pk[16];  // pk[2k]: row R0, P column 4(8hf+k) + lane%4; pk[2k+1]: row R1
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int e = 4 * (8 * hf + k);
        float x0, x1, y0, y1;
        ffma2(x0, x1, sv[e], sv[e + 1], c, c, -mb0, -mb0);
        ffma2(y0, y1, sv[e + 2], sv[e + 3], c, c, -mb1, -mb1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(y0), p3 = ex2_approx(y1);
        fadd2_acc(r00, r01, p0, p1);
        fadd2_acc(r10, r11, p2, p3);
        pk[2 * k] = pack_bf16x2(p0, p1);
        pk[2 * k + 1] = pack_bf16x2(p2, p3);
      }
      tmem_st_16x128b_x8(tw + s_col + 32 * hf, pk);
    }
    l0 = l0 * al0 + (r00 + r01);
    l1 = l1 * al1 + (r10 + r11);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar_p);
  }
  // Row sums over the quad: all four threads of a quad then hold their two rows' m and l.
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  // Every warp waits for this item's last PV before it arrives on O-free, also one with no valid
  // row: an arrival before that could land in the previous item's O-free phase and release O while
  // that item's epilogue still reads it.
  const uint32_t bar_free = smem_u32(&bars[kBarOFree0 + tile]);
  if (!mbar_wait(bar_o, ob & 1, abort_flag, a.status)) return false;
  if constexpr (kHost) {
    if (sp.nsplit > 1) {
      tc_fence_after();
      return split_epilogue<D>(a, sp, tile, tr, active, tw, o_col, bar_free, m0, l0, m1, l1, c0, bars, abort_flag,
                               sep++);
    }
  }
  if (!active) {  // warp-uniform: no row of this warp is stored, O is not read
    mbar_arrive(bar_free);
    return true;
  }
  tc_fence_after();
  // Epilogue in the softmax layout: O of rows R0, R1 in 32-column parts (16x256b), each thread
  // writing two adjacent bf16 per 8-column chunk; a quad covers 16 contiguous bytes of a row.
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int32_t t0 = c0 + tok_r0, t1 = c0 + tok_r1;
  const int32_t hm = (1 << tr.lg) - 1;
  const int32_t h0 = tr.head0 + (R0 & hm), h1 = tr.head0 + (R1 & hm);
  const bool st0 = R0 < tr.rows_valid, st1 = R1 < tr.rows_valid;
  __nv_bfloat16 *o0 = a.out + ((int64_t)t0 * a.Hq + h0) * D + cq;
  __nv_bfloat16 *o1 = a.out + ((int64_t)t1 * a.Hq + h1) * D + cq;
  // all of O (D / 32 parts of 16 values) in flight before one wait, then the stores
  float o[D / 2];  // o[16 part + 4k + {0,1}]: row R0, columns 32 part + 8k + cq + {0,1}; + {2,3}: row R1
#pragma unroll
  for (int part = 0; part < D / 32; ++part) tmem_ld_16x256b_x4(tw + o_col + part * 32, o + 16 * part);
  tmem_wait_ld();
#pragma unroll
  for (int part = 0; part < D / 32; ++part) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int col = part * 32 + 8 * k;
      const float *v = o + 16 * part + 4 * k;
      if (st0) *reinterpret_cast<uint32_t *>(o0 + col) = pack_bf16x2(v[0] * inv0, v[1] * inv0);
      if (st1) *reinterpret_cast<uint32_t *>(o1 + col) = pack_bf16x2(v[2] * inv1, v[3] * inv1);
    }
  }
  if ((lane & 3) == 0 && a.lse) {
    if (st0) a.lse[(int64_t)h0 * a.N + t0] = (m0 + log2f(l0)) * kLn2;
    if (st1) a.lse[(int64_t)h1 * a.N + t1] = (m1 + log2f(l1)) * kLn2;
  }
  // this warp's TMEM loads of O are complete: the next work item's first PV may overwrite it
  tc_fence_before();
  mbar_arrive(bar_free);
  return true;
}

// One work item = two 128-row query tiles of one segment that share every K/V
// tile (one tile when the second would hold no valid row); see unit_geometry.
// When a call holds too few items to give every SM one (a short chunk),
// `single` makes every item one tile, twice as many items at the same total
// work.  A host-planned call may also split a unit's key range over several
// items (WorkItem::j0, T, split, nsplit), merged by the last one to finish.
// What unit_geometry needs of a device-planned unit: three dependent reads of global memory
// (the planner's pair, the segment's bounds, its cached prefix), done once by the warp that claims
// the unit and published with it in shared memory.
struct ItemInputs {
  int32_t s, m, hsel, c0, n, P;
};
__device__ __forceinline__ ItemInputs item_inputs(const AttnArgs &a, int32_t unit) {
  const int32_t pair_idx = unit / a.heads_per_pair, hsel = unit % a.heads_per_pair;
  const int2 pr = a.pairs[pair_idx];
  const int32_t c0 = a.cu[pr.x];
  const int32_t n = a.cu[pr.x + 1] - c0;
  const int32_t P = a.prefix_lens ? a.prefix_lens[pr.x] : a.pos[c0];
  return ItemInputs{pr.x, pr.y, hsel, c0, n, P};
}
__device__ __forceinline__ WorkItem item_geometry(const AttnArgs &a, const ItemInputs &in) {
  return unit_geometry(in.s, in.m, in.hsel, in.c0, in.n, in.P, a.lg, a.group, a.single);
}

// Item u of a host-built plan.
__device__ __forceinline__ WorkItem decode_plan_item(const AttnArgs &a, const HostPlanArgs &hp, int32_t u) {
  const PlanItem it = hp.items[u];
  const int32_t s = it.w0 & 0xFFFF, hsel = (int32_t)((uint32_t)it.w0 >> 16);
  const int32_t m = it.w1 & 0xFFFFFF, nsplit = (int32_t)((uint32_t)it.w1 >> 24);
  WorkItem w = unit_geometry(s, m, hsel, hp.seg[s][0], hp.seg[s][1], hp.seg[s][2], a.lg, a.group, a.single);
  w.j0 = it.w2 & 0xFFFF;
  w.T = (int32_t)((uint32_t)it.w2 >> 16);
  w.nsplit = nsplit;
  w.g0 = it.w3 & 0xFFFFFF;
  w.split = (int32_t)((uint32_t)it.w3 >> 24);
  return w;
}

// Kernel parameter of the host-planned variant; the device-planned one gets a placeholder.
template <bool kHost>
struct PlanParam {
  int32_t unused;
};
template <>
struct PlanParam<true> : HostPlanArgs {};

// Persistent: the TMA warp claims the next non-empty work item of the
// planner's longest-first list from a global counter (dynamic longest-first
// scheduling over the SMs) and publishes it to the other roles through a
// two-entry queue in shared memory; every role walks the same sequence.  The K/V
// ring and all barriers run on across items, so the producer streams the next
// item's Q and K/V while the current one finishes, and the next item's first
// QK overlaps the current epilogue (its first PV waits until O has been read).
// kHost: the work items come from a plan built on the host (kernel parameter hp): CTA b runs items
// hp.cta_first[b] .. hp.cta_first[b + 1] - 1 in order, and an item may cover part of its unit's key
// range (split items, merged in the epilogue).  Otherwise a device planner wrote the item list and
// the CTAs claim items dynamically.
template <int D, bool kHost>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnArgs a,
                                                               const __grid_constant__ PlanParam<kHost> hp) {
  using L = SmemLayout<D>;
  constexpr int kHalves = D / 64;
  constexpr int ns = kStages;  // ring slots, after both Q buffers
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tmem_busy;  // 1: tensor-core work could not be confirmed finished, TMEM is kept
  __shared__ int32_t s_unit[kUnitSlots][8];  // published items: id, then its ItemInputs (device planner)
  __shared__ int32_t s_last[2];  // split epilogue: this CTA's split finished its (unit, tile) last

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto slot_addr = [&](int slot) { return sbase + L::kRing + slot * L::kTileBytes; };
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarSlotFull0 + i), 1);
      mbar_init(bar(kBarSlotEmpty0 + i), 1);
      mbar_init(bar(kBarSlotGo0 + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull0 + i), 1);
      mbar_init(bar(kBarPFull0 + i), 2 * kBlockM);
      mbar_init(bar(kBarODone0 + i), 1);
      mbar_init(bar(kBarOFree0 + i), 2 * kBlockM);
    }
    mbar_init(bar(kBarFinal), 1);
    mbar_init(bar(kBarPVDone), 1);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(bar(kBarUnitFull0 + i), 1);
      mbar_init(bar(kBarUnitEmpty0 + i), kUnitReaders);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSplitStored0 + i), 2 * kBlockM);
      mbar_init(bar(kBarSplitDecided0 + i), 1);
    }
    mbar_init(bar(kBarTile1Start), 8);
    s_abort = 0;
    s_tmem_busy = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int *abort_flag = &s_abort;
  // This grid runs as a programmatic dependent of its planner: the set-up above overlaps the plan,
  // which is read only past here.  A CTA that finds no work left claims nothing and tears down.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int32_t n_units = 0, first_item = 0;
  if constexpr (kHost) {
    first_item = hp.cta_first[blockIdx.x];
    n_units = hp.cta_first[blockIdx.x + 1] - first_item;
  } else {
    n_units = *a.num_pairs * a.heads_per_pair;
  }
  auto decode = [&](int32_t u, const ItemInputs &in) -> WorkItem {
    if constexpr (kHost) return decode_plan_item(a, hp, u);
    else return item_geometry(a, in);
  };
  SplitCtx sp;
  if constexpr (kHost) {
    sp.partial = hp.partial;
    sp.tickets = hp.tickets;
    sp.gen = hp.gen;
  } else {
    sp.partial = nullptr;
    sp.tickets = nullptr;
    sp.gen = 0;
  }
  sp.last = s_last;

  // Barrier completions before the current item, replayed identically by every role:
  // S-full / P-full per buffer, PV-done, O-done and O-free uses per tile, items done.
  uint32_t cs0 = 0, cs1 = 0, cpv = 0, co0 = 0, co1 = 0, items = 0;
  auto advance = [&](const WorkItem &w) {
    if (w.two) {
      cs0 += w.T;
      cs1 += w.T;
      ++co0;
      ++co1;
    } else {
      cs0 += (w.T + 1) >> 1;
      cs1 += w.T >> 1;
      cpv += w.T;
      ++co0;
    }
    ++items;
  };
  // Work item i of this CTA as published by the TMA warp (-1: none left).  Every lane of a reading
  // warp waits and reads; lane 0 then frees the entry for item i + kUnitSlots.
  auto next_unit = [&](uint32_t i, int32_t &u, ItemInputs &in) -> bool {
    const int k = i & (kUnitSlots - 1);
    if (!mbar_wait(bar(kBarUnitFull0 + k), (i / kUnitSlots) & 1, abort_flag, a.status)) return false;
    const volatile int32_t *e = s_unit[k];
    u = e[0];
    in = ItemInputs{e[1], e[2], e[3], e[4], e[5], e[6]};
    __syncwarp(__activemask());  // the MMA warp reads with lane 0 alone
    if (lane == 0) mbar_arrive(bar(kBarUnitEmpty0 + k));
    return true;
  };

  if (warp < 16) {
    // ------------------------------------------------------------ softmax + epilogue
    const int tile = warp >> 3;
    uint32_t sep = 0;  // split epilogues of this warp's tile so far
    for (uint32_t i = 0;; ++i) {
      int32_t u;
      ItemInputs in;
      if (!next_unit(i, u, in) || u < 0) break;
      // Tile 1 idles through one-tile items on tile 0's O-done barrier, so it must never fall two of
      // that barrier's phases behind (a warp of tile 1 may be late, merging the partials of a split
      // item): the MMA warp completes an item's O-done only after all of tile 1 has started the item.
      if (tile == 1 && lane == 0) mbar_arrive(smem_u32(&bars[kBarTile1Start]));
      const WorkItem w = decode(u, in);
      sp.split = w.split;
      sp.nsplit = w.nsplit;
      sp.g0 = w.g0;
      bool ok = true;
      if (w.two)
        ok = softmax_tile_role<D, false, kHost>(a, tile, tile ? w.tr1 : w.tr0, w.j0, w.T, w.Tp, w.P, w.c0, tmem,
                                                bars, abort_flag, cs0, cs1, cpv, tile ? co1 : co0, sp, sep);
      else if (tile == 0)
        ok = softmax_tile_role<D, true, kHost>(a, 0, w.tr0, w.j0, w.T, w.Tp, w.P, w.c0, tmem, bars, abort_flag,
                                               cs0, cs1, cpv, co0, sp, sep);
      else  // tile 1 idles through a one-tile item but may not run ahead of its S-full completions
        ok = mbar_wait(smem_u32(&bars[kBarODone0 + 0]), co0 & 1, abort_flag, a.status);
      if (!ok) break;
      advance(w);
    }
  } else if (warp == kWarpTma || warp >= kWarpAux0) {
    // ------------------------------------------------------------ TMA producers
    // Warp 16 loads Q and the segment's own K/V tiles and arms every slot; the page copies of a
    // prefix tile are split over warps 16, 18 and 19 (page pi by warp pi mod 3), since one warp
    // issues its TMA copies one after another.  All three follow the same load sequence.
    const int pw = warp == kWarpTma ? 0 : warp - kWarpAux0 + 1;
    if (pw == 0 && lane == 0) {
      tma_prefetch_desc(a.lg > 0 ? &a.tm_qp : &a.tm_q);
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
      if (a.num_pages > 0) {
        tma_prefetch_desc(&a.tm_kc);
        tma_prefetch_desc(&a.tm_vc);
      }
    }
    const int32_t ppt = kBlockN / a.page_size;  // 1, 2, 4 or 8
    const int32_t tpb = 32 / ppt;               // tiles per block-table batch (a power of two)
    const uint32_t page_bytes = a.page_size * 128u;
    // Helpers do not wait on slot-empty (they skip the fills they take no part in, so they could drift
    // two phases from it): warp 16 arrives on the slot's go barrier for every prefix fill after its
    // own slot-empty wait, and the helpers wait on those in order, one go per prefix fill of a slot.
    uint32_t go[kStages] = {0, 0, 0, 0, 0};
    const bool helpers = ppt > 1;
    int64_t lbase = 0;  // ring loads issued before the current item (all producer warps count them)
    int64_t issued = 0;
    uint32_t q_issued = 0;  // Q loads issued (warp 16)
    bool ok = true;
    // Work items are claimed and published ahead: when item i starts, items i + 1 and i + 2 are
    // already out, so the claim (an atomic on the work counter and three dependent reads of the
    // item's metadata) is off the path from one item's last PV to the next item's first QK even when
    // items are short.  Publishing item j waits only for every reader to have taken item
    // j - kUnitSlots, at most item i - 2.
    static_assert(kUnitSlots >= 4, "items i .. i + 2 published while readers may still hold item i - 1");
    // lane 0 of warp 16: item i of this CTA (-1 for none) and, device-planned, its inputs
    auto claim = [&](uint32_t i, ItemInputs &in) -> int32_t {
      in = ItemInputs{0, 0, 0, 0, 0, 0};
      if constexpr (kHost) {
        return static_cast<int32_t>(i) < n_units ? first_item + static_cast<int32_t>(i) : -1;
      } else {
        for (;;) {
          const int32_t c = atomicAdd(a.work_counter, 1);
          if (c >= n_units) return -1;
          in = item_inputs(a, c);
          if (item_geometry(a, in).valid) return c;
        }
      }
    };
    uint32_t n_published = 0;  // lane 0 of warp 16: items published so far
    bool end_published = false;  // lane 0 of warp 16: the -1 that ends the list is out
    auto publish_to = [&](uint32_t upto) -> int {  // lane 0 of warp 16; 0 when a wait gave up
      for (; !end_published && n_published < upto; ++n_published) {
        const uint32_t i = n_published;
        const int k = i & (kUnitSlots - 1);
        if (i >= kUnitSlots &&
            !mbar_wait(bar(kBarUnitEmpty0 + k), (i / kUnitSlots - 1) & 1, abort_flag, a.status))
          return 0;
        ItemInputs in;
        const int32_t u = claim(i, in);
        s_unit[k][0] = u;
        s_unit[k][1] = in.s;
        s_unit[k][2] = in.m;
        s_unit[k][3] = in.hsel;
        s_unit[k][4] = in.c0;
        s_unit[k][5] = in.n;
        s_unit[k][6] = in.P;
        mbar_arrive(bar(kBarUnitFull0 + k));
        if (u < 0) end_published = true;
      }
      return 1;
    };
    for (uint32_t i = 0; ok; ++i) {
      int32_t u = -1;
      ItemInputs in{0, 0, 0, 0, 0, 0};
      if (pw == 0) {
        int okq = 1;
        if (lane == 0) {
          okq = publish_to(i + 3);
          // item i as this lane published it (its own earlier shared-memory stores)
          const int k = i & (kUnitSlots - 1);
          u = s_unit[k][0];
          in = ItemInputs{s_unit[k][1], s_unit[k][2], s_unit[k][3], s_unit[k][4], s_unit[k][5], s_unit[k][6]};
        }
        if (!__shfl_sync(0xffffffffu, okq, 0)) break;
        u = __shfl_sync(0xffffffffu, u, 0);
        in.s = __shfl_sync(0xffffffffu, in.s, 0);
        in.m = __shfl_sync(0xffffffffu, in.m, 0);
        in.hsel = __shfl_sync(0xffffffffu, in.hsel, 0);
        in.c0 = __shfl_sync(0xffffffffu, in.c0, 0);
        in.n = __shfl_sync(0xffffffffu, in.n, 0);
        in.P = __shfl_sync(0xffffffffu, in.P, 0);
      } else if (!next_unit(i, u, in)) {
        break;
      }
      if (u < 0) break;
      const WorkItem w = decode(u, in);
      const int32_t T = w.T, Tp = w.Tp, P = w.P, c0 = w.c0, g = w.g, j0 = w.j0;
      const int32_t Tpl = max(0, min(T, Tp - j0));  // prefix tiles among this item's key tiles
      const bool two = w.two;
      if (pw == 0 && lane == 0) {
        // Q of this item once the previous item's last QK has read the buffers
        if (items > 0) ok = mbar_wait(bar(kBarQEmpty), (items - 1) & 1, abort_flag, a.status);
        if (ok) {
          mbar_arrive_expect_tx(bar(kBarQFull), (two ? 2 : 1) * L::kTileBytes);
          // box {64, 1, 128} of tm_q, or {64, G, 128 / G} of tm_qp: 128 rows of 128 bytes either way
          const void *qmap = a.lg > 0 ? static_cast<const void *>(&a.tm_qp) : static_cast<const void *>(&a.tm_q);
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf) {
            tma_load_3d(sbase + L::kQ0 + hf * L::kHalfBytes, qmap, bar(kBarQFull), hf * 64, w.tr0.head0,
                        c0 + w.tr0.tok0);
            if (two)
              tma_load_3d(sbase + L::kQ1 + hf * L::kHalfBytes, qmap, bar(kBarQFull), hf * 64, w.tr1.head0,
                          c0 + w.tr1.tok0);
          }
          q_issued = items + 1;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      // Page ids in warp-wide batches of 32 entries, fetched two batches ahead, validated at use.
      const int64_t bt_row = (int64_t)w.s * a.max_pages;
      auto fetch = [&](int32_t jb) -> int32_t {  // raw entry of logical page jb * ppt + lane, or -1
        const int32_t lp = jb * ppt + lane;
        return (jb < Tp && lp * a.page_size < P) ? __ldg(&a.block_table[bt_row + lp]) : -1;
      };
      const int32_t jb0 = j0 & ~(tpb - 1);  // block-table batch holding the item's first key tile
      int32_t bt_cur = fetch(jb0), bt_nxt = fetch(jb0 + tpb), bt_nx2 = fetch(jb0 + 2 * tpb);
      int32_t ph0 = a.num_pages, ph1 = a.num_pages;  // this lane's page of the last two K tiles
      int32_t last_k = -1;
      // Helper warps stop after the item's last prefix copy: V_(Tp-1), load 2Tp - 1 with two query
      // tiles, else 2Tp while K runs ahead (Tp - 1 < T - 2) and Tp - 1 + T after.
      // A helper that owns no page of a tile (page size 64 or 128) waits for nothing at all.
      const int32_t n_loads =
          pw == 0 ? 2 * T
                  : (Tpl == 0 || ppt <= pw ? 0 : (two ? 2 * Tpl : (Tpl - 1 < T - 2 ? 2 * Tpl + 1 : Tpl + T)));
      for (int32_t ld = 0; ld < n_loads; ++ld) {
        const int64_t gl = lbase + ld;
        const int slot = (int)(gl % ns);
        const int64_t round = gl / ns;
        // Loads follow the order the MMAs consume them: K_j, V_j alternating with two query tiles;
        // with one, K runs two tiles ahead of V: K0, K1, V0, K2, V1, ..., K(T-1), V(T-2), V(T-1).
        int32_t j;
        bool is_v;
        if (two) {
          j = ld >> 1;
          is_v = ld & 1;
        } else if (ld < 2) {
          is_v = ld == 1 && T == 1;
          j = is_v ? 0 : ld;
        } else {
          const int32_t t = ld - 2;
          if (t < 2 * (T - 2)) {
            is_v = (t & 1) == 0;
            j = is_v ? (t >> 1) : (t >> 1) + 2;
          } else {
            is_v = true;
            j = t - T + 2;
          }
        }
        const int32_t jg = j0 + j;  // key tile within the unit's range
        const uint32_t dst = slot_addr(slot);
        const uint32_t fb = bar(kBarSlotFull0 + slot);
        int okw = 1;
        if (pw == 0) {
          if (lane == 0) {
            if (round > 0)
              okw = mbar_wait(bar(kBarSlotEmpty0 + slot), (uint32_t)(round - 1) & 1, abort_flag, a.status);
            if (okw) {
              mbar_arrive_expect_tx(fb, L::kTileBytes);
              if (helpers && jg < Tp) mbar_arrive(bar(kBarSlotGo0 + slot));
            }
          }
        } else if (jg < Tp) {
          uint32_t k = 0;
#pragma unroll
          for (int sl = 0; sl < kStages; ++sl)
            if (sl == slot) k = go[sl]++;
          if (lane == 0) okw = mbar_wait(bar(kBarSlotGo0 + slot), k & 1, abort_flag, a.status);
        }
        if (!__shfl_sync(0xffffffffu, okw, 0)) {
          ok = false;
          break;
        }
        int32_t phys = a.num_pages;  // past the prefix end, or a bad entry: zero fill
        if (!is_v) {
          if (jg < Tp) {
            if (jg > j0 && (jg & (tpb - 1)) == 0) {
              bt_cur = bt_nxt;
              bt_nxt = bt_nx2;
              bt_nx2 = fetch(jg + 2 * tpb);
            }
            const int32_t e = __shfl_sync(0xffffffffu, bt_cur, (jg & (tpb - 1)) * ppt + (lane & (ppt - 1)));
            if (lane < ppt && (jg * ppt + lane) * a.page_size < P) {
              if (e >= 0 && e < a.num_pages) phys = e;
              else if (lane % kPageIssuers == pw) atomicOr(a.status, UNIP_DEV_BAD_PAGES);
            }
          }
          ph1 = ph0;
          ph0 = phys;
          last_k = j;
        } else {
          phys = last_k == j ? ph0 : ph1;  // V_j follows K_j or K_(j+1)
        }
        if (jg < Tp) {
          const void *map = is_v ? static_cast<const void *>(&a.tm_vc) : static_cast<const void *>(&a.tm_kc);
          if (lane < ppt && lane % kPageIssuers == pw) {
#pragma unroll
            for (int hf = 0; hf < kHalves; ++hf)
              tma_load_4d(dst + hf * L::kHalfBytes + lane * page_bytes, map, fb, hf * 64, g, 0, phys);
          }
        } else if (pw == 0 && lane == 0) {
          const void *map = is_v ? static_cast<const void *>(&a.tm_v) : static_cast<const void *>(&a.tm_k);
          const int32_t krow = c0 + (jg - Tp) * kBlockN;
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf) tma_load_3d(dst + hf * L::kHalfBytes, map, fb, hf * 64, g, krow);
        }
        issued = gl + 1;
      }
      lbase += 2 * T;
      advance(w);
    }
    if (lane == 0 && *abort_flag) {
      // Let copies already in flight land before the CTA's shared memory is released.
      for (int64_t gl = max((int64_t)0, issued - ns); gl < issued; ++gl) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar(kBarSlotFull0 + (int)(gl % ns)), (uint32_t)(gl / ns) & 1) &&
               globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      if (pw == 0 && q_issued > 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar(kBarQFull), (q_issued - 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, D, false, true);
      // Shared-memory descriptors are built once; a K step or another slot only adds an offset
      // (in 16-byte units) to the start-address field.
      const uint64_t dq0 = sdesc_sw128(sbase + L::kQ0, 16, 1024);
      const uint64_t dq1 = sdesc_sw128(sbase + L::kQ1, 16, 1024);
      const uint64_t dk = sdesc_sw128(sbase + L::kRing, 16, 1024);
      const uint64_t dv = sdesc_sw128(sbase + L::kRing, L::kHalfBytes, 1024);
      const uint32_t d_s0 = tmem, d_s1 = tmem + kBlockN;
      const uint32_t d_o0 = tmem + kTmemO, d_o1 = tmem + kTmemO + 128;
      auto slot_desc = [&](uint64_t d, int slot) { return d + ((uint64_t)(slot * L::kTileBytes) >> 4); };
      auto qk = [&](uint32_t d_s, uint64_t dq, uint64_t dkb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4);
          umma_bf16_ss(d_s, dq + off, dkb + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto pv = [&](uint32_t d_o, uint32_t p_tmem, uint64_t dvb, uint32_t acc_first) {
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          umma_bf16_ts(d_o, p_tmem + kk * 8, dvb + (uint64_t)((kk * 2048) >> 4), idesc_pv, kk > 0 ? 1u : acc_first);
      };
      // ring load gl sits in slot gl % ns and completes phase (gl / ns) & 1
      auto full = [&](int64_t gl) {
        return mbar_wait(bar(kBarSlotFull0 + (int)(gl % ns)), (uint32_t)(gl / ns) & 1, abort_flag, a.status);
      };
      auto release = [&](int64_t gl) { umma_commit(bar(kBarSlotEmpty0 + (int)(gl % ns))); };
      // O of tile t may be overwritten once the previous item's epilogue has read it
      auto o_free = [&](int t, uint32_t uses) {
        return uses == 0 || mbar_wait(bar(kBarOFree0 + t), (uses - 1) & 1, abort_flag, a.status);
      };
      // before the PV that completes this item's O-done of tile 0: every warp of tile 1 started the item
      auto tile1_started = [&]() { return mbar_wait(bar(kBarTile1Start), items & 1, abort_flag, a.status); };
      int64_t lbase = 0;
      bool ok = true;
      for (uint32_t i = 0; ok; ++i) {
        int32_t u;
        ItemInputs in;
        if (!next_unit(i, u, in) || u < 0) break;
        const WorkItem w = decode(u, in);
        const int32_t T = w.T;
        ok = mbar_wait(bar(kBarQFull), items & 1, abort_flag, a.status) && full(lbase);
        if (!ok) break;
        tc_fence_after();
        if (!w.two) {
          // One query tile: S is double-buffered over both S regions, so QK(j+2) runs while the
          // softmax of KV tile j does.  Order: QK(0), QK(1), then PV(j), QK(j+2) for each j.
          // Load index of K_0, K_1: 0, 1; of K_m (m >= 2): 2m - 1; of V_j: 2j + 2 while K still runs
          // ahead (j < T - 2), then j + T.
          qk(d_s0, dq0, slot_desc(dk, (int)(lbase % ns)));
          umma_commit(bar(kBarSFull0 + 0));
          release(lbase);
          if (T > 1) {
            if (!(ok = full(lbase + 1))) break;
            qk(d_s1, dq0, slot_desc(dk, (int)((lbase + 1) % ns)));
            umma_commit(bar(kBarSFull0 + 1));
            release(lbase + 1);
          }
          if (T <= 2) umma_commit(bar(kBarQEmpty));
          for (int32_t j = 0; ok && j < T; ++j) {
            const int buf = j & 1;
            const uint32_t d_s = tmem + buf * kBlockN;
            const int64_t iv = lbase + (j < T - 2 ? 2 * j + 2 : j + T), ik = lbase + 2 * j + 3;
            ok = mbar_wait(bar(kBarPFull0 + buf), ((buf ? cs1 : cs0) + (j >> 1)) & 1, abort_flag, a.status) &&
                 full(iv) && (j > 0 || o_free(0, co0)) && (j + 1 < T || tile1_started());
            if (!ok) break;
            tc_fence_after();
            pv(d_o0, d_s, slot_desc(dv, (int)(iv % ns)), j > 0 ? 1u : 0u);
            umma_commit(bar(kBarPVDone));
            release(iv);
            if (j + 1 == T) umma_commit(bar(kBarODone0 + 0));
            if (j + 2 < T) {
              if (!(ok = full(ik))) break;
              qk(d_s, dq0, slot_desc(dk, (int)(ik % ns)));
              umma_commit(bar(kBarSFull0 + buf));
              release(ik);
              if (j + 3 == T) umma_commit(bar(kBarQEmpty));  // QK(T-1): the last read of Q
            }
          }
        } else {
          // Two query tiles: K_j is load 2j, V_j load 2j + 1.
          const uint64_t dk0 = slot_desc(dk, (int)(lbase % ns));
          qk(d_s0, dq0, dk0);
          umma_commit(bar(kBarSFull0 + 0));
          qk(d_s1, dq1, dk0);
          umma_commit(bar(kBarSFull0 + 1));
          release(lbase);
          if (T == 1) umma_commit(bar(kBarQEmpty));
          for (int32_t j = 0; ok && j < T; ++j) {
            const bool more = j + 1 < T;
            const int64_t iv = lbase + 2 * j + 1, ik = lbase + 2 * j + 2;
            const uint64_t dvj = slot_desc(dv, (int)(iv % ns)), dkn = slot_desc(dk, (int)(ik % ns));
            const uint32_t acc = j > 0 ? 1u : 0u;
            // tile 0: PV(j), then QK(j+1); K_(j+1) is waited for first so that both go out back to back
            ok = full(iv) && (!more || full(ik)) &&
                 mbar_wait(bar(kBarPFull0 + 0), (cs0 + j) & 1, abort_flag, a.status) && (j > 0 || o_free(0, co0)) &&
                 (more || tile1_started());
            if (!ok) break;
            tc_fence_after();
            pv(d_o0, d_s0, dvj, acc);
            if (!more) umma_commit(bar(kBarODone0 + 0));
            if (more) {
              qk(d_s0, dq0, dkn);
              umma_commit(bar(kBarSFull0 + 0));
            }
            // tile 1: PV(j), then QK(j+1)
            if (!(ok = mbar_wait(bar(kBarPFull0 + 1), (cs1 + j) & 1, abort_flag, a.status) &&
                       (j > 0 || o_free(1, co1))))
              break;
            tc_fence_after();
            pv(d_o1, d_s1, dvj, acc);
            if (!more) umma_commit(bar(kBarODone0 + 1));
            if (more) {
              qk(d_s1, dq1, dkn);
              umma_commit(bar(kBarSFull0 + 1));  // first: the softmax of tile 1 waits on it
              release(ik);
              if (j + 2 == T) umma_commit(bar(kBarQEmpty));  // QK(T-1): the last read of Q
            }
            release(iv);
          }
        }
        lbase += 2 * T;
        advance(w);
      }
      // Every tcgen05 op of this CTA has landed before TMEM is released.  If that cannot be confirmed
      // within two wait limits, the columns are not freed under running MMAs: the CTA leaves them
      // allocated and raises the timeout bit (the context should then be torn down by its owner).
      umma_commit(bar(kBarFinal));
      bool drained = false;
      for (int round = 0; round < 2 && !drained; ++round) {
        const uint64_t t0 = globaltimer_ns();
        while (!(drained = mbar_try_wait(bar(kBarFinal), 0)) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      if (!drained) {
        s_tmem_busy = 1;
        atomicOr(a.status, UNIP_DEV_TIMEOUT);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma && !s_tmem_busy) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kHost>
cudaError_t launch_attention(const AttnArgs &args, const PlanParam<kHost> &plan, int grid, cudaStream_t stream) {
  using L = SmemLayout<D>;
  const cudaError_t e = ensure_dynamic_smem((const void *)attn_fwd_kernel<D, kHost>, (int)L::kDynamic);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kDynamic;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the planner runs
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // A host-planned call has no planner: its set-up overlaps the tail of whatever ran before it on the
  // stream (the kernel reads nothing before griddepcontrol.wait).
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D, kHost>, args, plan);
}

// Work-item shape of every attention call of the process (unip_set_attention_schedule).
std::atomic<int> g_attention_schedule{UNIP_ATTN_SCHEDULE_AUTO};

int32_t max_pairs_for(int32_t total_tokens, int32_t num_segs) {
  return (total_tokens + kBlockM - 1) / kBlockM + num_segs;
}

}  // namespace
}  // namespace unip

using namespace unip;

extern "C" {

UNIP_API int32_t unip_set_attention_schedule(int32_t mode) {
  if (mode != UNIP_ATTN_SCHEDULE_AUTO && mode != UNIP_ATTN_SCHEDULE_PAIRED && mode != UNIP_ATTN_SCHEDULE_SINGLE)
    return UNIP_ERR_INVALID_ARGUMENT;
  g_attention_schedule.store(mode, std::memory_order_relaxed);
  return UNIP_OK;
}

UNIP_API size_t unip_attention_workspace_size(int32_t total_tokens, int32_t num_segs, const unip_attn_params *prm) {
  (void)prm;
  if (total_tokens < 0 || num_segs < 0) return 0;
  return kWsHeaderBytes + align_up(sizeof(int2) * (size_t)max_pairs_for(total_tokens, num_segs), 256);
}

// Tensor maps and shape fields shared by every attention launch (q, k, v token-major; the cache,
// when given, [page][slot][H_kv][D]).  Returns UNIP_OK or UNIP_ERR_CUDA.
static int32_t prepare_args(AttnArgs &args, const void *q, const void *k, const void *v, int32_t total_tokens,
                            const unip_paged_kv *cache, const unip_attn_params *prm, void *out, float *lse) {
  const int32_t Hq = prm->num_heads_q, Hkv = prm->num_heads_kv, D = prm->head_dim;
  memset(&args, 0, sizeof(args));
  const cuuint32_t box3[3] = {64, 1, kBlockM};
  // Even groups that divide 128 put (token, head) pairs on a tile's rows.
  const int32_t G = Hq / Hkv;
  int32_t lg = 0;
  if (G % 2 == 0 && kBlockM % G == 0)
    while ((1 << lg) < G) ++lg;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)total_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
    if (encode_tiled(&args.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box3,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return UNIP_ERR_CUDA;
    const cuuint32_t boxp[3] = {64, (cuuint32_t)G, (cuuint32_t)(kBlockM / G)};
    if (lg > 0 && encode_tiled(&args.tm_qp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims,
                               strides, boxp, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return UNIP_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)total_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
    if (encode_tiled(&args.tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(k), dims, strides, box3,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tiled(&args.tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(v), dims, strides, box3,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return UNIP_ERR_CUDA;
  }
  if (cache) {
    const int32_t ps = cache->page_size;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)ps, (cuuint64_t)cache->num_pages};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2, (cuuint64_t)ps * Hkv * D * 2};
    const cuuint32_t box4[4] = {64, 1, (cuuint32_t)ps, 1};
    if (encode_tiled(&args.tm_kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache->k_cache), dims,
                     strides, box4, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tiled(&args.tm_vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache->v_cache), dims,
                     strides, box4, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return UNIP_ERR_CUDA;
    args.block_table = cache->block_table;
    args.num_pages = cache->num_pages;
    args.page_size = cache->page_size;
    args.max_pages = cache->max_pages_per_seq;
  } else {
    args.page_size = 16;
  }
  args.out = static_cast<__nv_bfloat16 *>(out);
  args.lse = lse;
  args.N = total_tokens;
  args.Hq = Hq;
  args.group = G;
  args.lg = lg;
  const float scale = prm->scale > 0.f ? prm->scale : 1.0f / sqrtf((float)D);
  args.scale_log2 = scale * kLog2e;
  return UNIP_OK;
}

// Both entry points: prefix_lens == NULL takes each segment's prefix length from its first position
// (contiguous positions); otherwise the stream is compacted (increasing positions, explicit prefixes).
static int32_t attention_entry(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                               int32_t num_segs, const int32_t *positions, const int32_t *prefix_lens,
                               int32_t total_tokens, const unip_paged_kv *paged, const unip_attn_params *prm,
                               void *out, float *lse, void *workspace, size_t workspace_bytes, void *stream) {
  if (!prm || !cu_seqlens || num_segs < 0 || total_tokens < 0) return UNIP_ERR_INVALID_ARGUMENT;
  const int32_t Hq = prm->num_heads_q, Hkv = prm->num_heads_kv, D = prm->head_dim;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return UNIP_ERR_INVALID_ARGUMENT;
  if (D != 64 && D != 128) return UNIP_ERR_UNSUPPORTED;
  if (total_tokens == 0) return UNIP_OK;
  if (num_segs == 0 || !q || !k || !v || !positions || !out) return UNIP_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return UNIP_ERR_ALIGNMENT;
  const size_t need_ws = unip_attention_workspace_size(total_tokens, num_segs, prm);
  if (!workspace || workspace_bytes < need_ws || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return UNIP_ERR_WORKSPACE;
  const bool has_cache = paged && paged->k_cache && paged->v_cache && paged->block_table && paged->num_pages > 0;
  if (has_cache) {
    const int32_t ps = paged->page_size;
    if (ps != 16 && ps != 32 && ps != 64 && ps != 128) return UNIP_ERR_UNSUPPORTED;
    if (paged->max_pages_per_seq <= 0) return UNIP_ERR_INVALID_ARGUMENT;
    if (!aligned16(paged->k_cache) || !aligned16(paged->v_cache)) return UNIP_ERR_ALIGNMENT;
  }
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;

  AttnArgs args;
  const int32_t prc = prepare_args(args, q, k, v, total_tokens, has_cache ? paged : nullptr, prm, out, lse);
  if (prc != UNIP_OK) return prc;
  const int32_t G = args.group, lg = args.lg;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t *header = static_cast<int32_t *>(workspace);
  int2 *pairs = reinterpret_cast<int2 *>(static_cast<uint8_t *>(workspace) + kWsHeaderBytes);
  const int32_t max_pairs = max_pairs_for(total_tokens, num_segs);
  attn_plan_kernel<<<1, kPlanThreads, 0, st>>>(cu_seqlens, positions, prefix_lens, num_segs, total_tokens,
                                               has_cache ? 1 : 0,
                                               has_cache ? paged->page_size : 16,
                                               has_cache ? paged->max_pages_per_seq : 0, lg, header, pairs,
                                               max_pairs, status);
  if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;

  args.cu = cu_seqlens;
  args.pos = positions;
  args.prefix_lens = prefix_lens;
  args.pairs = pairs;
  args.num_pairs = header;
  args.work_counter = header + 1;
  args.status = status;
  args.S = num_segs;
  // Two query tiles per work item when the group is even, unless even twice the
  // most items the call can hold leave SMs idle: then one tile per item.
  // Query tiles: sum over segments of ceil(n_s / 128) <= ceil(N / 128) + S - 1.
  const int sms = device_sm_count();
  const bool even = G % 2 == 0;
  const int64_t tiles_hi = (int64_t)(total_tokens + kBlockM - 1) / kBlockM + (num_segs > 0 ? num_segs - 1 : 0);
  const int mode = g_attention_schedule.load(std::memory_order_relaxed);
  args.single = !even ? 0
                : mode == UNIP_ATTN_SCHEDULE_SINGLE ? 1
                : mode == UNIP_ATTN_SCHEDULE_PAIRED ? 0
                : (2 * tiles_hi * (Hq / 2) <= (int64_t)(sms > 0 ? sms : 1) ? 1 : 0);
  args.heads_per_pair = (even && !args.single) ? Hq / 2 : Hq;
  // persistent grid: one CTA per SM (fewer when the plan cannot hold that many work items)
  const int64_t units_bound = (int64_t)max_pairs * args.heads_per_pair;
  if (units_bound > 0x7FFFFFFF) return UNIP_ERR_UNSUPPORTED;
  const int64_t grid = std::min<int64_t>(units_bound, sms > 0 ? sms : 1);
  const PlanParam<false> none{0};
  const cudaError_t e = D == 128 ? launch_attention<128, false>(args, none, (int)grid, st)
                                 : launch_attention<64, false>(args, none, (int)grid, st);
  return e == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
}

UNIP_API int32_t unip_prefill_attention(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                                        int32_t num_segs, const int32_t *positions, int32_t total_tokens,
                                        const unip_paged_kv *paged, const unip_attn_params *prm, void *out,
                                        float *lse, void *workspace, size_t workspace_bytes, void *stream) {
  return attention_entry(q, k, v, cu_seqlens, num_segs, positions, nullptr, total_tokens, paged, prm, out, lse,
                         workspace, workspace_bytes, stream);
}

UNIP_API int32_t unip_compacted_attention(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                                          int32_t num_segs, const int32_t *positions, const int32_t *prefix_lens,
                                          int32_t total_tokens, const unip_paged_kv *paged,
                                          const unip_attn_params *prm, void *out, float *lse, void *workspace,
                                          size_t workspace_bytes, void *stream) {
  if (num_segs > 0 && !prefix_lens) return UNIP_ERR_INVALID_ARGUMENT;
  return attention_entry(q, k, v, cu_seqlens, num_segs, positions, prefix_lens, total_tokens, paged, prm, out,
                         lse, workspace, workspace_bytes, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Host-built plans
// ---------------------------------------------------------------------------
struct unip_attn_plan {
  int32_t N = 0, S = 0, Hq = 0, Hkv = 0, D = 0, page_size = 16, max_pages = 0;
  float scale = 0.f;
  bool any_prefix = false;
  bool device = false;  // run the device planner instead
  int32_t single = 0, n_items = 0, n_ctas = 0, n_split_units = 0, n_splits = 0;
  size_t ticket_bytes = 0, partial_bytes = 0, ws_bytes = 0;
  unip::HostPlanArgs args;  // seg, cta_first, items (pointers and generation are set per run)
  std::atomic<void *> ready_ws{nullptr};  // workspace whose ticket area this plan has cleared
};

namespace unip {
namespace {

// Cost model of the host planner, in SM cycles (measured periods of the kernel on GB300): a key tile
// of a two-tile item costs ~3.4k cycles (32 MMAs, one tile's softmax overlapping the other's MMAs);
// of a one-tile item ~1.6k, ~2.9k when it streams cached pages (its K and V tiles serve one query
// tile, so page copies bound it); every item adds its Q load, pipeline fill and epilogue.  A split
// item also stores its fp32 partial (~70 KB per full tile) and takes a ticket, and the split that
// merges reads every split's partial back through L2: a few round trips of ~3k cycles when many
// tiles merge at once.  Both scale with the tile's valid rows (warps past them store nothing), so
// splitting pays for decode-like tiles far more readily than for full prefill tiles.
constexpr double kCostTile2 = 3400.0, kCostTile2Prefix = 3900.0, kCostTile1 = 1600.0, kCostTile1Prefix = 2900.0;
constexpr double kCostItem = 3000.0, kCostSplitFixed = 2000.0, kCostSplitStore = 3000.0;
constexpr double kCostMergeRound = 5000.0;  // a round of the merge's loads reads partials another SM wrote
constexpr int32_t kMinSplitTiles = 2;
constexpr int32_t kMaxSplits = 8;        // the merge reads every split: more would lengthen the tail
constexpr int32_t kMaxSplitsFull = 2;    // tiles whose rows are mostly valid

double merge_rounds(int32_t n) { return 1.0 + 4.0 * ((n + 2) / 3); }

struct PlanUnit {
  int32_t s, m, hsel, T, Tp;
  bool two;
  double active;  // fraction of the item's softmax warps that hold valid rows (partial-store volume)
};

double range_cost(const PlanUnit &u, int32_t j0, int32_t T) {
  const int32_t pre = std::max(0, std::min(T, u.Tp - j0));  // key tiles read through the block table
  if (u.two) return kCostTile2Prefix * pre + kCostTile2 * (T - pre);
  return kCostTile1Prefix * pre + kCostTile1 * (T - pre);
}

struct Candidate {
  int32_t single = 0;
  int32_t L = 0;  // largest key range of one item (INT32_MAX: no split)
  double makespan = 0.0;
  int32_t n_items = 0;
  std::vector<PlanItem> items;       // in CTA order
  std::vector<uint16_t> cta_first;
  int32_t n_ctas = 0, n_split_units = 0, n_splits = 0;
};

// Items of one shape and split length, balanced over `sms` CTAs longest-processing-time first.
// forced > 0: every unit is split into min(forced, T) ranges instead (L unused).
bool build_candidate(const std::vector<PlanUnit> &units, int32_t single, int32_t L, int sms, Candidate &c,
                     int32_t forced = 0) {
  struct It {
    PlanItem pi;
    double cost;
  };
  std::vector<It> its;
  int32_t g = 0, nsu = 0;
  for (const PlanUnit &u : units) {
    int32_t n = (u.T > L) ? (u.T + L - 1) / L : 1;
    n = std::min(n, std::min(u.T, u.active > 0.5 ? kMaxSplitsFull : kMaxSplits));
    if (forced > 0) n = std::min(forced, u.T);
    const int32_t base = u.T / n, rem = u.T % n;
    int32_t j0 = 0;
    for (int32_t k = 0; k < n; ++k) {
      const int32_t T = base + (k < rem ? 1 : 0);
      It it;
      it.pi.w0 = (int32_t)((uint32_t)u.s | ((uint32_t)u.hsel << 16));
      it.pi.w1 = (int32_t)((uint32_t)u.m | ((uint32_t)n << 24));
      it.pi.w2 = (int32_t)((uint32_t)j0 | ((uint32_t)T << 16));
      it.pi.w3 = (int32_t)((uint32_t)(n > 1 ? g : 0) | ((uint32_t)k << 24));
      // the last split holds the unit's own (diagonal) tiles and is charged the merge
      const double vol = 0.25 + 0.75 * u.active;
      it.cost = kCostItem + range_cost(u, j0, T);
      if (n > 1) it.cost += kCostSplitFixed + kCostSplitStore * vol;
      if (n > 1 && k == n - 1) it.cost += kCostMergeRound * merge_rounds(n) * vol;
      its.push_back(it);
      j0 += T;
    }
    if (n > 1) {
      g += n;
      ++nsu;
    }
    if ((int64_t)its.size() > kPlanMaxItems || g >= (1 << 24)) return false;
  }
  const int32_t n_items = (int32_t)its.size();
  const int ctas = std::max(1, std::min(sms, n_items));
  if (ctas > kPlanMaxCtas) return false;
  std::vector<int32_t> order(n_items);
  for (int32_t i = 0; i < n_items; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return its[x].cost > its[y].cost; });
  // least-loaded CTA first (ties: lower index)
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int b = 0; b < ctas; ++b) heap.push({0.0, b});
  std::vector<std::vector<int32_t>> per(ctas);
  double mk = 0.0;
  for (int32_t i : order) {
    Slot sl = heap.top();
    heap.pop();
    per[sl.second].push_back(i);
    sl.first += its[i].cost;
    mk = std::max(mk, sl.first);
    heap.push(sl);
  }
  c.single = single;
  c.L = L;
  c.makespan = mk;
  c.n_items = n_items;
  c.n_ctas = ctas;
  c.n_split_units = nsu;
  c.n_splits = g;
  c.items.clear();
  c.cta_first.assign(ctas + 1, 0);
  for (int b = 0; b < ctas; ++b) {
    c.cta_first[b] = (uint16_t)c.items.size();
    for (int32_t i : per[b]) c.items.push_back(its[i].pi);
  }
  c.cta_first[ctas] = (uint16_t)c.items.size();
  return true;
}

void plan_units(const unip_attn_plan &p, const std::vector<int32_t> &cu, const std::vector<int32_t> &pre,
                int32_t lg, int32_t single, std::vector<PlanUnit> &units) {
  const int32_t G = p.Hq / p.Hkv;
  const bool even = G % 2 == 0;
  const int32_t hpp = (even && !single) ? p.Hq / 2 : p.Hq;
  units.clear();
  for (int32_t s = 0; s < p.S; ++s) {
    const int32_t n = cu[s + 1] - cu[s];
    for (int32_t m = 0; m * kBlockM < n; ++m)
      for (int32_t h = 0; h < hpp; ++h) {
        const WorkItem w = unit_geometry(s, m, h, cu[s], n, pre[s], lg, G, single);
        if (!w.valid) continue;
        const int32_t rows = w.tr0.rows_valid + (w.two ? w.tr1.rows_valid : 0);
        const double active = (double)((rows + 15) / 16) / (w.two ? 16.0 : 8.0);
        units.push_back({s, m, h, w.T, w.Tp, w.two, active});
      }
  }
}

}  // namespace
}  // namespace unip

extern "C" {

UNIP_API int32_t unip_attention_plan_create(const int32_t *cu_seqlens, int32_t num_segs, const int32_t *prefix_lens,
                                            int32_t total_tokens, const unip_attn_params *prm, int32_t page_size,
                                            int32_t max_pages_per_seq, int32_t flags, int32_t num_sms,
                                            unip_attn_plan **plan) {
  if (!plan) return UNIP_ERR_INVALID_ARGUMENT;
  *plan = nullptr;
  if (!prm || !cu_seqlens || num_segs < 0 || total_tokens < 0 || (flags & ~0xFF03) || num_sms < 0)
    return UNIP_ERR_INVALID_ARGUMENT;
  const int32_t forced = (flags >> 8) & 0xFF;  // UNIP_PLAN_SPLITS(n)
  if (forced && (flags & UNIP_PLAN_NO_SPLIT)) return UNIP_ERR_INVALID_ARGUMENT;
  const int32_t Hq = prm->num_heads_q, Hkv = prm->num_heads_kv, D = prm->head_dim;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return UNIP_ERR_INVALID_ARGUMENT;
  if (D != 64 && D != 128) return UNIP_ERR_UNSUPPORTED;
  std::vector<int32_t> cu(cu_seqlens, cu_seqlens + num_segs + 1);
  std::vector<int32_t> pre(num_segs, 0);
  if (cu[0] != 0 || cu[num_segs] != total_tokens) return UNIP_ERR_INVALID_ARGUMENT;
  bool any_prefix = false;
  for (int32_t s = 0; s < num_segs; ++s) {
    if (cu[s + 1] < cu[s]) return UNIP_ERR_INVALID_ARGUMENT;
    pre[s] = prefix_lens ? prefix_lens[s] : 0;
    if (pre[s] < 0) return UNIP_ERR_INVALID_ARGUMENT;
    if (pre[s] > 0 && cu[s + 1] > cu[s]) any_prefix = true;
  }
  if (any_prefix) {
    if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return UNIP_ERR_UNSUPPORTED;
    if (max_pages_per_seq <= 0) return UNIP_ERR_INVALID_ARGUMENT;
    for (int32_t s = 0; s < num_segs; ++s)
      if (cu[s + 1] > cu[s] && ((int64_t)pre[s] + page_size - 1) / page_size > max_pages_per_seq)
        return UNIP_ERR_INVALID_ARGUMENT;
  }
  unip_attn_plan *p = new (std::nothrow) unip_attn_plan();
  if (!p) return UNIP_ERR_TOO_LARGE;
  p->N = total_tokens;
  p->S = num_segs;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->D = D;
  p->scale = prm->scale;
  p->page_size = any_prefix ? page_size : 16;
  p->max_pages = any_prefix ? max_pages_per_seq : 0;
  p->any_prefix = any_prefix;
  const int32_t G = Hq / Hkv;
  int32_t lg = 0;
  if (G % 2 == 0 && kBlockM % G == 0)
    while ((1 << lg) < G) ++lg;
  bool host = !(flags & UNIP_PLAN_DEVICE) && num_segs <= kPlanMaxSegs && total_tokens > 0 &&
              Hq < (1 << 16) && (int64_t)total_tokens / kBlockM < (1 << 24);
  if (host) {
    // the key range of a unit must fit the item's 16-bit fields
    for (int32_t s = 0; s < num_segs && host; ++s)
      if ((int64_t)(pre[s] + kBlockN - 1) / kBlockN + (int64_t)(cu[s + 1] - cu[s] + kBlockN - 1) / kBlockN >= 65535)
        host = false;
  }
  int sms = num_sms > 0 ? num_sms : device_sm_count();
  if (sms <= 0) sms = 1;
  sms = std::min(sms, kPlanMaxCtas);
  Candidate best;
  bool found = false;
  if (host) {
    const int mode = g_attention_schedule.load(std::memory_order_relaxed);
    std::vector<int32_t> shapes;
    if (G % 2 != 0) shapes = {0};
    else if (mode == UNIP_ATTN_SCHEDULE_PAIRED) shapes = {0};
    else if (mode == UNIP_ATTN_SCHEDULE_SINGLE) shapes = {1};
    else shapes = {0, 1};
    std::vector<PlanUnit> units;
    Candidate c;
    for (int32_t single : shapes) {
      plan_units(*p, cu, pre, lg, single, units);
      if (units.empty()) continue;
      int64_t wt = 0;
      for (const PlanUnit &u : units) wt += u.T;
      std::vector<int32_t> Ls = {INT32_MAX};
      if (!(flags & UNIP_PLAN_NO_SPLIT))
        for (double f : {1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 8.0}) {
          const int64_t L = std::max<int64_t>(kMinSplitTiles, (int64_t)std::ceil((double)wt / (f * sms)));
          if (std::find(Ls.begin(), Ls.end(), (int32_t)L) == Ls.end()) Ls.push_back((int32_t)L);
        }
      if (forced) Ls = {INT32_MAX};
      for (int32_t L : Ls) {
        if (!build_candidate(units, single, L, sms, c, forced)) continue;
        // a clearly shorter makespan wins; within 2 %, fewer items (less fixed and split overhead)
        if (!found || c.makespan < best.makespan * 0.98 ||
            (c.makespan <= best.makespan * 1.02 && c.n_items < best.n_items)) {
          best = c;
          found = true;
        }
      }
    }
  }
  if (!found) {
    p->device = true;
    p->ws_bytes = unip_attention_workspace_size(total_tokens, num_segs, prm);
    *plan = p;
    return UNIP_OK;
  }
  p->single = best.single;
  p->n_items = best.n_items;
  p->n_ctas = best.n_ctas;
  p->n_split_units = best.n_split_units;
  p->n_splits = best.n_splits;
  memset(&p->args, 0, sizeof(p->args));
  for (int32_t s = 0; s < num_segs; ++s) {
    p->args.seg[s][0] = cu[s];
    p->args.seg[s][1] = cu[s + 1] - cu[s];
    p->args.seg[s][2] = pre[s];
  }
  std::copy(best.cta_first.begin(), best.cta_first.end(), p->args.cta_first);
  std::copy(best.items.begin(), best.items.end(), p->args.items);
  p->ticket_bytes = align_up(sizeof(unsigned long long) * 2 * (size_t)best.n_splits, 256);
  p->partial_bytes = split_slot_bytes(D) * 2 * (size_t)best.n_splits;
  p->ws_bytes = std::max<size_t>(256, p->ticket_bytes + p->partial_bytes);
  *plan = p;
  return UNIP_OK;
}

UNIP_API size_t unip_attention_plan_workspace_size(const unip_attn_plan *plan) { return plan ? plan->ws_bytes : 0; }

UNIP_API int32_t unip_attention_plan_info(const unip_attn_plan *plan, int32_t *info) {
  if (!plan || !info) return UNIP_ERR_INVALID_ARGUMENT;
  info[0] = plan->device ? 0 : 1;
  info[1] = plan->n_items;
  info[2] = plan->n_ctas;
  info[3] = plan->n_split_units;
  info[4] = plan->n_splits;
  info[5] = plan->single;
  return UNIP_OK;
}

UNIP_API void unip_attention_plan_destroy(unip_attn_plan *plan) { delete plan; }

UNIP_API int32_t unip_prefill_attention_planned(const unip_attn_plan *plan, const void *q, const void *k,
                                                const void *v, const int32_t *cu_seqlens, const int32_t *positions,
                                                const int32_t *prefix_lens, const unip_paged_kv *paged, void *out,
                                                float *lse, void *workspace, size_t workspace_bytes, void *stream) {
  if (!plan) return UNIP_ERR_INVALID_ARGUMENT;
  unip_attn_params prm;
  prm.num_heads_q = plan->Hq;
  prm.num_heads_kv = plan->Hkv;
  prm.head_dim = plan->D;
  prm.scale = plan->scale;
  if (plan->device)
    return attention_entry(q, k, v, cu_seqlens, plan->S, positions, prefix_lens, plan->N, paged, &prm, out, lse,
                           workspace, workspace_bytes, stream);
  if (!q || !k || !v || !out) return UNIP_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return UNIP_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < plan->ws_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return UNIP_ERR_WORKSPACE;
  const bool has_cache = paged && paged->k_cache && paged->v_cache && paged->block_table && paged->num_pages > 0;
  if (plan->any_prefix) {
    if (!has_cache) return UNIP_ERR_INVALID_ARGUMENT;
    if (paged->page_size != plan->page_size || paged->max_pages_per_seq != plan->max_pages)
      return UNIP_ERR_INVALID_ARGUMENT;
    if (!aligned16(paged->k_cache) || !aligned16(paged->v_cache)) return UNIP_ERR_ALIGNMENT;
  }
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  AttnArgs args;
  const int32_t prc = prepare_args(args, q, k, v, plan->N, plan->any_prefix ? paged : nullptr, &prm, out, lse);
  if (prc != UNIP_OK) return prc;
  args.status = status;
  args.S = plan->S;
  args.single = plan->single;
  args.heads_per_pair = 0;  // unused: items name their head selection
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PlanParam<true> hp;
  static_cast<HostPlanArgs &>(hp) = plan->args;
  hp.tickets = reinterpret_cast<unsigned long long *>(workspace);
  hp.partial = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + plan->ticket_bytes);
  static std::atomic<uint32_t> g_gen{0};
  hp.gen = g_gen.fetch_add(1, std::memory_order_relaxed) % 0xFFFFFFFEu + 1u;  // never 0 (cleared tickets)
  if (plan->n_splits > 0 && plan->ready_ws.load(std::memory_order_relaxed) != workspace) {
    if (cudaMemsetAsync(workspace, 0, plan->ticket_bytes, st) != cudaSuccess) return UNIP_ERR_CUDA;
    const_cast<unip_attn_plan *>(plan)->ready_ws.store(workspace, std::memory_order_relaxed);
  }
  const cudaError_t e = plan->D == 128 ? launch_attention<128, true>(args, hp, plan->n_ctas, st)
                                       : launch_attention<64, true>(args, hp, plan->n_ctas, st);
  return e == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation variant: the tile plan lives in a fixed device array.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxDevices = 64;

// Scratch of unip_prefill_attention_noalloc (planner header + tile pairs).
static __device__ __align__(256) uint8_t g_noalloc_scratch[UNIP_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoAllocMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device with that device current (host code cannot use the symbol itself).
void *noalloc_scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_noalloc_addr[dev] = ptr;
  }
  return g_noalloc_addr[dev];
}

}  // namespace

extern "C" {

UNIP_API int32_t unip_prefill_attention_noalloc(const void *q, const void *k, const void *v,
                                                const int32_t *cu_seqlens, int32_t num_segs,
                                                const int32_t *positions, int32_t total_tokens,
                                                const unip_paged_kv *paged, const unip_attn_params *prm,
                                                void *out, float *lse, void *stream) {
  if (!prm || num_segs < 0 || total_tokens < 0) return UNIP_ERR_INVALID_ARGUMENT;
  const int64_t tiles = ((int64_t)total_tokens + kBlockM - 1) / kBlockM + num_segs;
  if (tiles > UNIP_NOALLOC_MAX_TILES) return UNIP_ERR_TOO_LARGE;
  const size_t need = unip_attention_workspace_size(total_tokens, num_segs, prm);
  if (need > (size_t)UNIP_NOALLOC_SCRATCH_BYTES) return UNIP_ERR_TOO_LARGE;
  void *scratch = noalloc_scratch_address();
  if (!scratch) return UNIP_ERR_CUDA;
  return unip_prefill_attention(q, k, v, cu_seqlens, num_segs, positions, total_tokens, paged, prm, out, lse,
                                scratch, (size_t)UNIP_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
