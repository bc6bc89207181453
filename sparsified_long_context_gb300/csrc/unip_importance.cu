// Block importance from the last query rows of each segment.
//
// Source: "[논문리뷰] UniPrefill ..." review, section 3 -- the sequence is cut
// into blocks whose importance is estimated at a full-attention layer.  The
// scoring rule (last min(B, n) query rows, attention probability mass per
// own-key block, summed over query heads, normalised per segment) is the
// reading this library fixes; it reuses the row log-sum-exp that the
// attention kernel stores, so no second softmax pass is needed.
//
// Kernels
//   imp_plan_kernel   one CTA: block offsets blk_cu, list of (segment, 128-key
//                     chunk) work items of the scored segments.
//   imp_score_tc_kernel  one CTA per (work item, kv head): TMA loads the
//                     128-key tile and the window rows of the kv head's query
//                     heads; one tcgen05 MMA chain computes S^T = K Q_w^T into
//                     TMEM (keys on lanes, window rows x heads on columns);
//                     128 threads, one key each, sum exp(s - lse) over their
//                     visible columns; per-block partial masses are reduced
//                     with shuffles and written without atomics (deterministic).
//   imp_norm_kernel   one CTA per segment: sums the kv-head partials in a
//                     fixed order and divides by the segment total.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kChunk = 128;        // keys per score CTA
constexpr int kPlanThreads = 1024;
constexpr int kNormThreads = kImpNormThreads;
constexpr int kWsHeaderBytes = 256;
constexpr float kLog2e = 1.44269504088896340736f;

__global__ void __launch_bounds__(kPlanThreads) imp_plan_kernel(const int32_t *__restrict__ cu, int32_t S,
                                                                int32_t N, const uint8_t *__restrict__ seg_mask,
                                                                int32_t B, int32_t *__restrict__ blk_cu,
                                                                int32_t imp_capacity, int32_t *__restrict__ header,
                                                                int2 *__restrict__ items, int32_t max_items,
                                                                uint32_t *__restrict__ status) {
  __shared__ int32_t s_scan[32];
  __shared__ uint32_t s_err;
  const int tid = threadIdx.x;
  // the score grid may be scheduled now; it waits for this plan before reading it
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int per = (S + kPlanThreads - 1) / kPlanThreads;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  if (tid == 0) s_err = (cu[0] != 0 || cu[S] != N) ? UNIP_DEV_BAD_SEQLENS : 0u;
  __syncthreads();
  int32_t my_blocks = 0, my_items = 0;
  bool bad = false;
  for (int s = s0; s < s1; ++s) {
    const int32_t n = cu[s + 1] - cu[s];
    if (n < 0) { bad = true; continue; }
    if (n > 0 && (!seg_mask || seg_mask[s])) {
      my_blocks += (n + B - 1) / B;
      my_items += (n + kChunk - 1) / kChunk;
    }
  }
  if (bad) atomicOr(&s_err, UNIP_DEV_BAD_SEQLENS);
  int32_t tot_blocks, tot_items;
  int32_t blk_base = block_excl_scan<int32_t>(my_blocks, s_scan, &tot_blocks);
  int32_t item_base = block_excl_scan<int32_t>(my_items, s_scan, &tot_items);
  if (s_err != 0 || tot_blocks > imp_capacity || tot_items > max_items) {
    for (int s = tid; s <= S; s += kPlanThreads) blk_cu[s] = 0;
    if (tid == 0) {
      header[0] = 0;
      atomicOr(status, s_err ? s_err : UNIP_DEV_BAD_SEQLENS);
    }
    return;
  }
  if (tid == 0) blk_cu[0] = 0;
  for (int s = s0; s < s1; ++s) {
    const int32_t n = cu[s + 1] - cu[s];
    if (n > 0 && (!seg_mask || seg_mask[s])) {
      blk_base += (n + B - 1) / B;
      const int32_t nc = (n + kChunk - 1) / kChunk;
      for (int c = 0; c < nc; ++c) items[item_base + c] = make_int2(s, c);
      item_base += nc;
    }
    blk_cu[s + 1] = blk_base;
  }
  if (tid == 0) header[0] = tot_items;
}

struct ScoreArgs {
  CUtensorMap tm_k;   // k  [N][H_kv][D], box 64 x 1 x 128
  CUtensorMap tm_q;   // q  [N][H_q][D],  box 64 x 1 x B
  const float *lse;   // [H_q][N]
  const int32_t *cu;
  const int32_t *blk_cu;
  const int2 *items;
  const int32_t *num_items;
  float *partial;     // [blocks][H_kv]
  uint32_t *status;
  int32_t N, Hq, Hkv, B, heads_per_group;
  float scale_log2;
};

// 16 score warps (four per TMEM lane quarter, each summing 64 of a unit's columns), TMA warp, MMA
// warp.  The score warps are latency-bound (TMEM loads, exp chains, per-unit barriers), so four per
// scheduler hide more of it than two did.
constexpr int kScoreWarps = 16;
constexpr int kScoreWarpTma = kScoreWarps;
constexpr int kScoreWarpMma = kScoreWarps + 1;
constexpr int kScoreThreadsTc = 32 * (kScoreWarps + 2);
constexpr int kScoreCompute = 32 * kScoreWarps;
constexpr int kScoreCols = kScoreWarps / 4 > 0 ? 256 / (kScoreWarps / 4) : 256;  // columns per score warp
constexpr int kMaxCols = 256;  // columns of S^T per MMA group (window rows x heads)

template <int D>
struct ScoreSmem {
  static constexpr uint32_t kHalf = 128 * 128;            // 128 rows x 128 B
  static constexpr uint32_t kKTile = (D / 64) * kHalf;     // one K tile: D/64 halves of 128 rows
  static constexpr uint32_t kQ = 2 * kKTile;               // after two K slots: Q window, D/64 halves of 256 rows
  static constexpr uint32_t kQHalf = kMaxCols * 128;
  static constexpr uint32_t kBytes = kQ + (D / 64) * kQHalf;
  static constexpr uint32_t kDynamic = kBytes + 1024;
};

enum ScoreBar {
  kSbQFull = 0,
  kSbQEmpty = 1,
  kSbKFull0 = 2,   // + slot
  kSbKEmpty0 = 4,  // + slot
  kSbSFull0 = 6,   // + TMEM buffer
  kSbSEmpty0 = 8,  // + TMEM buffer
  kSbFinal = 10,
  kSbNum = 11
};

// Persistent: CTA b walks a contiguous range of units (kv head g, 128-key
// chunk c of segment s), ordered head-major so that consecutive units mostly
// share a segment's window.  Per unit and query-head group: S^T = K Q_w^T on
// the tensor cores (M = 128 keys on TMEM lanes, N = window rows x heads on
// columns, K = D).  The window Q is loaded once per (segment, g, group); K
// tiles and S buffers are double-buffered so the next MMA runs while the
// score warps sum exp(s - lse) of the current one (warp w: lane quarter w % 4,
// column group w / 4 of kScoreCols columns).
template <int D>
__global__ void __launch_bounds__(kScoreThreadsTc, 1) imp_score_tc_kernel(const __grid_constant__ ScoreArgs a) {
  using L = ScoreSmem<D>;
  constexpr int kHalves = D / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kSbNum];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tmem_busy;  // 1: tensor-core work could not be confirmed finished, TMEM is kept
  __shared__ __align__(16) float s_lse[kMaxCols];
  __shared__ float s_key[kScoreWarps / 4 - 1][128];
  __shared__ float s_red[4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  // launched as a programmatic dependent of the planner: its work list is complete after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t n_items = *a.num_items;
  const int64_t U = (int64_t)n_items * a.Hkv;
  const int64_t u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  if (u0 >= u1) {  // uniform over the CTA
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }
  const int32_t B = a.B;
  const int32_t group = a.Hq / a.Hkv;
  const int32_t hpg = a.heads_per_group;     // heads per MMA group
  const int32_t ngroups = (group + hpg - 1) / hpg;
  const int64_t n_iter = (u1 - u0) * ngroups;  // iteration i: unit u0 + i / ngroups, group i % ngroups
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto bar = [&](int k) { return smem_u32(&bars[k]); };
  if (tid == 0) {
    for (int k = 0; k < kSbNum; ++k) mbar_init(bar(k), (k == kSbSEmpty0 || k == kSbSEmpty0 + 1) ? kScoreCompute : 1);
    s_abort = 0;
    s_tmem_busy = 0;
    fence_mbar_init();
  }
  if (warp == kScoreWarpMma) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int *abort_flag = &s_abort;
  struct It {
    int32_t g, s, c, gi, c0, n, bk0, nbs;  // bk0, nbs: the segment's first block and block count
  };
  // Each role decodes iteration i + 1 while it works on i: the work-list and cu_seqlens reads are a
  // chain of dependent global loads that would otherwise sit in front of every unit.
  auto decode = [&](int64_t i) {
    It r;
    if (i >= n_iter) {
      r.g = r.s = r.c = r.gi = -1;
      r.c0 = r.n = r.bk0 = r.nbs = 0;
      return r;
    }
    const int64_t u = u0 + i / ngroups;
    r.gi = (int32_t)(i % ngroups);
    r.g = (int32_t)(u / n_items);
    const int2 item = a.items[u % n_items];
    r.s = item.x;
    r.c = item.y;
    r.c0 = a.cu[r.s];
    r.n = a.cu[r.s + 1] - r.c0;
    r.bk0 = a.blk_cu[r.s];
    r.nbs = a.blk_cu[r.s + 1] - r.bk0;
    return r;
  };
  auto same_q = [](const It &x, const It &y) { return x.s == y.s && x.g == y.g && x.gi == y.gi; };

  if (warp == kScoreWarpTma) {
    if (lane == 0) {
      It prev = {-1, -1, -1, -1, 0, 0, 0, 0};
      uint32_t qn = 0;
      int64_t issued = 0;
      It nxt = decode(0);
      for (int64_t i = 0; i < n_iter; ++i) {
        const It it = nxt;
        nxt = decode(i + 1);
        const int32_t c0 = it.c0, n = it.n;
        if (!same_q(it, prev)) {
          if (qn > 0 && !mbar_wait(bar(kSbQEmpty), (qn - 1) & 1, abort_flag, a.status)) break;
          const int32_t W = min(B, n), hn = min(hpg, group - it.gi * hpg);
          mbar_arrive_expect_tx(bar(kSbQFull), kHalves * hn * B * 128);
          for (int32_t hh = 0; hh < hn; ++hh) {
            const int32_t h = it.g * group + it.gi * hpg + hh;
#pragma unroll
            for (int hf = 0; hf < kHalves; ++hf)
              tma_load_3d(sbase + L::kQ + hf * L::kQHalf + hh * B * 128, &a.tm_q, bar(kSbQFull), hf * 64, h,
                          c0 + n - W);
          }
          ++qn;
          prev = it;
        }
        const int slot = (int)(i & 1);
        if (i >= 2 && !mbar_wait(bar(kSbKEmpty0 + slot), ((i >> 1) - 1) & 1, abort_flag, a.status)) break;
        mbar_arrive_expect_tx(bar(kSbKFull0 + slot), L::kKTile);
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf)
          tma_load_3d(sbase + slot * L::kKTile + hf * L::kHalf, &a.tm_k, bar(kSbKFull0 + slot), hf * 64, it.g,
                      c0 + it.c * 128);
        issued = i + 1;
      }
      if (*abort_flag) {  // copies in flight land before the CTA's shared memory is released
        for (int64_t i = max((int64_t)0, issued - 2); i < issued; ++i) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar(kSbKFull0 + (int)(i & 1)), (i >> 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
        if (qn > 0) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar(kSbQFull), (qn - 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == kScoreWarpMma) {
    if (lane == 0) {
      It prev = {-1, -1, -1, -1, 0, 0, 0, 0};
      uint32_t qn = 0;
      bool ok = true;
      It nxt = decode(0);
      for (int64_t i = 0; ok && i < n_iter; ++i) {
        const It it = nxt;
        nxt = decode(i + 1);
        if (!same_q(it, prev)) {
          ok = mbar_wait(bar(kSbQFull), qn & 1, abort_flag, a.status);
          ++qn;
          prev = it;
        }
        const int slot = (int)(i & 1);
        ok = ok && mbar_wait(bar(kSbKFull0 + slot), (i >> 1) & 1, abort_flag, a.status) &&
             (i < 2 || mbar_wait(bar(kSbSEmpty0 + slot), ((i >> 1) - 1) & 1, abort_flag, a.status));
        if (!ok) break;
        tc_fence_after();
        const int32_t hn = min(hpg, group - it.gi * hpg);
        const uint32_t idesc = idesc_bf16_f32(128, hn * B, false, false);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = slot * L::kKTile + (kk >> 2) * L::kHalf + (kk & 3) * 32;
          const uint32_t qoff = L::kQ + (kk >> 2) * L::kQHalf + (kk & 3) * 32;
          umma_bf16_ss(tmem + slot * kMaxCols, sdesc_sw128(sbase + koff, 16, 1024), sdesc_sw128(sbase + qoff, 16, 1024),
                       idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(kSbSFull0 + slot));
        umma_commit(bar(kSbKEmpty0 + slot));
        if (i + 1 == n_iter || !same_q(nxt, it)) umma_commit(bar(kSbQEmpty));  // last MMA on this Q
      }
      // Every tcgen05 op of this CTA has landed before TMEM is released; if that cannot be confirmed
      // within two wait limits the columns are kept (not freed under running MMAs) and the timeout
      // bit is raised.
      umma_commit(bar(kSbFinal));
      bool drained = false;
      for (int round = 0; round < 2 && !drained; ++round) {
        const uint64_t t0 = globaltimer_ns();
        while (!(drained = mbar_try_wait(bar(kSbFinal), 0)) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      if (!drained) {
        s_tmem_busy = 1;
        atomicOr(a.status, UNIP_DEV_TIMEOUT);
      }
    }
  } else {
    // Score warps.  Every one of them runs all n_iter iterations and every named barrier, also
    // after a timed-out wait (live = false then skips the work), so none is left at a barrier.
    const int qd = warp & 3, ch = warp >> 2;
    const int key = 32 * qd + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    const int32_t bpc = 128 / B;
    bool live = true;
    It prev = {-1, -1, -1, -1, 0, 0, 0, 0};
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    It nxt = decode(0);
    for (int64_t i = 0; i < n_iter; ++i) {
      const It it = nxt;
      nxt = decode(i + 1);
      const int32_t c0 = it.c0, n = it.n;
      const int32_t W = min(B, n), wrow0 = n - W;
      const int32_t hn = min(hpg, group - it.gi * hpg), ncols = hn * B;
      if (!same_q(it, prev)) {
        // row normalisers of this window (log2 domain); window slots past the segment are masked
        asm volatile("bar.sync 1, %0;" ::"n"(kScoreCompute) : "memory");
        if (tid < ncols) {
          const int32_t hh = tid / B, t = tid & (B - 1);
          const int32_t h = it.g * group + it.gi * hpg + hh;
          s_lse[tid] = t < W ? a.lse[(int64_t)h * a.N + c0 + wrow0 + t] * kLog2e : INFINITY;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kScoreCompute) : "memory");
        prev = it;
      }
      const int slot = (int)(i & 1);
      live = live && mbar_wait(bar(kSbSFull0 + slot), (i >> 1) & 1, abort_flag, a.status);
      const int32_t j = it.c * 128 + key;
      const bool kvalid = j < n;
      // Every key of the chunk lies in the segment and before the window's first row: all columns
      // are visible (window slots past the segment carry an infinite normaliser and give 0).
      const bool open_chunk = it.c * 128 + 127 < n && it.c * 128 + 127 <= wrow0;
      if (live) {
        tc_fence_after();
        // this warp's columns: [kScoreCols ch, kScoreCols (ch + 1)) of the group's hn * B (a multiple of 16)
        // (32 columns per TMEM load keeps the score warps within 96 registers)
        for (int32_t col0 = kScoreCols * ch; col0 < min(kScoreCols * (ch + 1), ncols); col0 += 32) {
          float sv[32];
          tmem_ld32(tl + slot * kMaxCols + col0, sv);
          tmem_wait_ld();
          if (open_chunk && col0 + 32 <= ncols) {
            // no masks: packed (s * c - lse) pairs, four normalisers per shared-memory load
#pragma unroll
            for (int x = 0; x < 32; x += 4) {
              const float4 l4 = *reinterpret_cast<const float4 *>(&s_lse[col0 + x]);
              float y0, y1, y2, y3;
              ffma2(y0, y1, sv[x], sv[x + 1], a.scale_log2, a.scale_log2, -l4.x, -l4.y);
              ffma2(y2, y3, sv[x + 2], sv[x + 3], a.scale_log2, a.scale_log2, -l4.z, -l4.w);
              fadd2_acc(acc0, acc1, ex2_approx(y0), ex2_approx(y1));
              fadd2_acc(acc2, acc3, ex2_approx(y2), ex2_approx(y3));
            }
            continue;
          }
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            float e[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int32_t col = col0 + x + u;
              // visible: window slot inside the segment and key j at or before row wrow0 + slot
              const bool vis = kvalid && col < ncols && j <= wrow0 + (col & (B - 1));
              e[u] = vis ? ex2_approx(fmaf(sv[x + u], a.scale_log2, -s_lse[col])) : 0.f;
            }
            acc0 += e[0];
            acc1 += e[1];
            acc2 += e[2];
            acc3 += e[3];
          }
        }
        tc_fence_before();
      }
      mbar_arrive(bar(kSbSEmpty0 + slot));
      if (it.gi != ngroups - 1) continue;  // the unit's mass sums over all head groups
      // unit done: key masses of the column groups (summed in group order), then per-block sums over
      // the chunk's keys
      float v = (acc0 + acc1) + (acc2 + acc3);
      acc0 = acc1 = acc2 = acc3 = 0.f;
      asm volatile("bar.sync 1, %0;" ::"n"(kScoreCompute) : "memory");
      if (ch > 0) s_key[ch - 1][key] = v;
      asm volatile("bar.sync 1, %0;" ::"n"(kScoreCompute) : "memory");
      if (ch == 0) {
#pragma unroll
        for (int g2 = 0; g2 < kScoreWarps / 4 - 1; ++g2) v += s_key[g2][key];
        const int32_t nb_seg = it.nbs;
        const int64_t pbase = (int64_t)it.bk0 + it.c * bpc;
        if (B <= 32) {
          for (int off = B / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if ((key & (B - 1)) == 0) {
            const int32_t b = key / B;
            if (it.c * bpc + b < nb_seg && live) a.partial[(pbase + b) * a.Hkv + it.g] = v;
          }
        } else {
          for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == 0) s_red[qd] = v;
          asm volatile("bar.sync 2, 128;" ::: "memory");
          const int wpb = B / 32;
          if (key < bpc) {
            float t = 0.f;
            for (int w = 0; w < wpb; ++w) t += s_red[key * wpb + w];
            if (it.c * bpc + key < nb_seg && live) a.partial[(pbase + key) * a.Hkv + it.g] = t;
          }
          asm volatile("bar.sync 2, 128;" ::: "memory");
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // the normaliser may be scheduled now; it waits for every score CTA before reading the masses
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kScoreWarpMma && !s_tmem_busy) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void __launch_bounds__(kNormThreads) imp_norm_kernel(const int32_t *__restrict__ blk_cu,
                                                                 const float *__restrict__ partial, int32_t Hkv,
                                                                 float *__restrict__ imp) {
  __shared__ float sred[kImpNormThreads];
  // a Top-p grid launched as a programmatic dependent may be scheduled now; it waits for this one
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // launched as a programmatic dependent of the score grid: its masses are complete after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t s = blockIdx.x;
  const int32_t b0 = blk_cu[s], nb = blk_cu[s + 1] - b0;
  if (nb <= 0) return;
  normalise_segment(partial, b0, nb, Hkv, imp, sred);
}

template <int D>
cudaError_t launch_score(const ScoreArgs &args, int grid, cudaStream_t stream) {
  using L = ScoreSmem<D>;
  const cudaError_t e = ensure_dynamic_smem((const void *)imp_score_tc_kernel<D>, (int)L::kDynamic);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kScoreThreadsTc);
  cfg.dynamicSmemBytes = L::kDynamic;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the planner runs
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, imp_score_tc_kernel<D>, args);
}

cudaError_t launch_norm(const int32_t *blk_cu, const float *partial, int32_t Hkv, float *imp, int32_t num_segs,
                        cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_segs);
  cfg.blockDim = dim3(kNormThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the score grid drains
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, imp_norm_kernel, blk_cu, partial, Hkv, imp);
}

int32_t max_items_for(int32_t total_tokens, int32_t num_segs) {
  return (total_tokens + kChunk - 1) / kChunk + num_segs;
}

}  // namespace
}  // namespace unip

using namespace unip;

extern "C" {

UNIP_API int32_t unip_importance_capacity(int32_t total_tokens, int32_t num_segs, int32_t block_size) {
  if (total_tokens < 0 || num_segs < 0 || block_size <= 0) return 0;
  return total_tokens / block_size + num_segs + 1;
}

UNIP_API size_t unip_importance_workspace_size(int32_t total_tokens, int32_t num_segs, int32_t block_size,
                                               const unip_attn_params *prm) {
  if (!prm || total_tokens < 0 || num_segs < 0 || block_size <= 0) return 0;
  const size_t items = align_up(sizeof(int2) * (size_t)max_items_for(total_tokens, num_segs), 256);
  const size_t part = align_up(sizeof(float) * (size_t)unip_importance_capacity(total_tokens, num_segs, block_size) *
                                   (size_t)(prm->num_heads_kv > 0 ? prm->num_heads_kv : 1),
                               256);
  return kWsHeaderBytes + items + part;
}

}  // extern "C"

int32_t unip::importance_scores(const void *q, const void *k, const float *lse, const int32_t *cu_seqlens,
                                int32_t num_segs, int32_t total_tokens, const uint8_t *seg_mask, int32_t block_size,
                                const unip_attn_params *prm, float *imp, int32_t imp_capacity, int32_t *blk_cu,
                                void *workspace, size_t workspace_bytes, cudaStream_t st, float **partial_out) {
  *partial_out = nullptr;
  if (!prm || !cu_seqlens || !blk_cu || num_segs < 0 || total_tokens < 0) return UNIP_ERR_INVALID_ARGUMENT;
  const int32_t Hq = prm->num_heads_q, Hkv = prm->num_heads_kv, D = prm->head_dim;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return UNIP_ERR_INVALID_ARGUMENT;
  if (D != 64 && D != 128) return UNIP_ERR_UNSUPPORTED;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128) return UNIP_ERR_UNSUPPORTED;
  if (num_segs == 0) return UNIP_OK;
  if (total_tokens > 0 && (!q || !k || !lse || !imp)) return UNIP_ERR_INVALID_ARGUMENT;
  if ((q && !aligned16(q)) || (k && !aligned16(k))) return UNIP_ERR_ALIGNMENT;
  if (imp_capacity < unip_importance_capacity(total_tokens, num_segs, block_size)) return UNIP_ERR_INVALID_ARGUMENT;
  const size_t need = unip_importance_workspace_size(total_tokens, num_segs, block_size, prm);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return UNIP_ERR_WORKSPACE;
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *header = reinterpret_cast<int32_t *>(ws);
  const int32_t max_items = max_items_for(total_tokens, num_segs);
  int2 *items = reinterpret_cast<int2 *>(ws + kWsHeaderBytes);
  float *partial = reinterpret_cast<float *>(ws + kWsHeaderBytes + align_up(sizeof(int2) * (size_t)max_items, 256));
  imp_plan_kernel<<<1, kPlanThreads, 0, st>>>(cu_seqlens, num_segs, total_tokens, seg_mask, block_size, blk_cu,
                                              imp_capacity, header, items, max_items, status);
  if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;
  if (total_tokens == 0) return UNIP_OK;
  const float scale = prm->scale > 0.f ? prm->scale : 1.0f / sqrtf((float)D);
  // persistent score grid: one CTA per SM (each takes a contiguous range of (kv head, chunk) units)
  const int64_t units_bound = (int64_t)max_items * Hkv;
  const int sms = device_sm_count();
  const int64_t grid = std::min<int64_t>(units_bound, sms > 0 ? sms : 1);
  ScoreArgs args;
  memset(&args, 0, sizeof(args));
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)total_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
    const cuuint32_t box[3] = {64, 1, 128};
    if (encode_tiled(&args.tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(k), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return UNIP_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)total_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)block_size};
    if (encode_tiled(&args.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return UNIP_ERR_CUDA;
  }
  args.lse = lse;
  args.cu = cu_seqlens;
  args.blk_cu = blk_cu;
  args.items = items;
  args.num_items = header;
  args.partial = partial;
  args.status = status;
  args.N = total_tokens;
  args.Hq = Hq;
  args.Hkv = Hkv;
  args.B = block_size;
  args.heads_per_group = std::min(Hq / Hkv, kMaxCols / block_size);
  args.scale_log2 = scale * kLog2e;
  cudaError_t e = D == 128 ? launch_score<128>(args, (int)grid, st) : launch_score<64>(args, (int)grid, st);
  if (e != cudaSuccess) return UNIP_ERR_CUDA;
  *partial_out = partial;
  return UNIP_OK;
}

extern "C" {

UNIP_API int32_t unip_block_importance(const void *q, const void *k, const float *lse, const int32_t *cu_seqlens,
                                       int32_t num_segs, int32_t total_tokens, const uint8_t *seg_mask,
                                       int32_t block_size, const unip_attn_params *prm, float *imp,
                                       int32_t imp_capacity, int32_t *blk_cu, void *workspace,
                                       size_t workspace_bytes, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float *partial = nullptr;
  const int32_t rc = importance_scores(q, k, lse, cu_seqlens, num_segs, total_tokens, seg_mask, block_size, prm, imp,
                                       imp_capacity, blk_cu, workspace, workspace_bytes, st, &partial);
  if (rc != UNIP_OK || !partial) return rc;
  if (launch_norm(blk_cu, partial, prm->num_heads_kv, imp, num_segs, st) != cudaSuccess) return UNIP_ERR_CUDA;
  return UNIP_OK;
}

}  // extern "C"
