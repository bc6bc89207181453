// Top-p block selection and compaction indices.
//
// Source: "[논문리뷰] UniPrefill ..." review, section 1 ("Top-p Token
// Selection": the fewest blocks whose cumulative importance reaches p) and
// section 3 (dropped tokens are excluded from every later sub-layer).
//
// Bit-exact, summation-order-free selection: scores become 32.32 fixed-point
// integers, the total and all running sums are exact uint64, the threshold is
// one IEEE double multiply, and the ranking is a total order (score bits
// descending, block index ascending).  Greedy-by-rank gives the fewest blocks
// because, for any count, the largest reachable mass is the sum of the
// top-ranked blocks.
//
// Kernels
//   topp_kernel   one CTA per segment: bitonic sort of 64-bit rank keys
//                 (each key also carries its block's score, so the ranked
//                 masses need no second read), exclusive scan of the ranked
//                 integer masses, keep decision per block, exclusive scan of
//                 kept lengths; writes the segment's count.  Segments of at
//                 most 32 blocks are selected by one warp.
//   norm_select_kernel  the same per segment after importance's normaliser,
//                 in the CTA that normalised the scores.
//   select_gather_kernel  the row copy after either of them (a programmatic
//                 dependent): kept offsets staged in shared memory, one warp
//                 per kept row.
//   select_gather_onepass_kernel, norm_select_gather_onepass_kernel  one
//                 segment in the call: every CTA (one per SM) selects the
//                 segment's blocks itself (the second also normalises the
//                 masses first), stages the kept offsets and copies its share
//                 of the kept rows (one launch, no grid waits for another).
//   index_kernel  one thread per source token: every CTA scans the
//                 per-segment counts into shared memory (CTA 0 also writes
//                 cu_seqlens_kept and n_kept), then writes gather_idx and
//                 positions_kept at the token's compacted slot.  With very
//                 many segments a one-CTA scan kernel writes the offsets to
//                 global memory first.
#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kToppThreads = 512;
static_assert(kToppThreads <= 512, "block_sum2 holds one slot per warp for at most 16 warps");
constexpr int kIndexThreads = 256;
constexpr int kMaxBlocks = UNIP_TOPP_MAX_BLOCKS;
constexpr int kRankCountMax = 1024;  // segments up to this many blocks rank by counting instead of sorting
constexpr int kWsHeaderBytes = 256;
constexpr int kIndexSmemSegs = 12000;  // segments whose offsets the index kernel keeps in shared memory
constexpr int kGatherCtasPerSm = 2;    // fused gather grid: 16 warps per SM, each with 4 KB of loads in flight
constexpr int kGatherStageBytes = 48 * 1024;  // shared memory of the fused gather (no opt-in needed)

// floor(f * 2^32) for 0 <= f <= 1, exactly and without FP64 arithmetic (a slow pipe on this
// part): f = m * 2^(e - 150) with the 24-bit significand m and biased exponent e, so
// f * 2^32 = m * 2^(e - 118).  Zero and subnormal scores are below 2^-126 and give 0.
__device__ __forceinline__ unsigned long long fixed_mass(float f) {
  const uint32_t u = __float_as_uint(f);
  const int e = static_cast<int>(u >> 23);  // f >= 0 with the sign bit clear (-0 is read as +0)
  if (e == 0) return 0ull;
  const unsigned long long m = (u & 0x7FFFFFu) | 0x800000u;
  const int sh = e - 118;
  return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}

// Keep test in integers: for an integer mass x below 2^53 (exact in fp64), x < thr holds exactly
// when x < ceil(thr), with thr = p * T the one IEEE multiply of the selection rule.
__device__ __forceinline__ unsigned long long mass_threshold(double p, unsigned long long T) {
  return static_cast<unsigned long long>(ceil(__dmul_rn(p, static_cast<double>(T))));
}

// Rank key of a non-forced block: score descending (bits of a non-negative
// float order like the float), then block index ascending.
__device__ __forceinline__ unsigned long long rank_key(float f, int b) {
  return (static_cast<unsigned long long>(~__float_as_uint(f)) << 32) | static_cast<uint32_t>(b);
}
__device__ __forceinline__ float key_score(unsigned long long key) {
  return __uint_as_float(~static_cast<uint32_t>(key >> 32));
}

// Bitonic sort of npow keys (a power of two, at most the CTA's threads), one per thread (threads
// past npow hold padding): strides below 32 exchange through warp shuffles, larger ones through
// shared memory.  The loop over sizes is not unrolled: a selection runs once per call, usually
// after other work has pushed its code out of L2, and a fully unrolled 45-stage network for 512 keys
// spent longer fetching its instructions than executing them.
__device__ __forceinline__ void bitonic_sort_regs(unsigned long long &key, unsigned long long *skeys, int tid,
                                                  int npow) {
#pragma unroll 1
  for (int size = 2; size <= npow; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride >= 32; stride >>= 1) {
      __syncthreads();
      if (tid < npow) skeys[tid] = key;
      __syncthreads();
      const unsigned long long other = tid < npow ? skeys[tid ^ stride] : key;
      const bool take_min = ((tid & stride) == 0) == ((tid & size) == 0);
      key = take_min ? (other < key ? other : key) : (other > key ? other : key);
    }
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
      if (stride < size) {  // uniform over the CTA
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, stride);
        const bool take_min = ((tid & stride) == 0) == ((tid & size) == 0);
        key = take_min ? (other < key ? other : key) : (other > key ? other : key);
      }
    }
  }
}

// Sums of a and b over the CTA (at most 16 warps), returned to every thread.  Integer sums are exact,
// so their order does not matter.  sh: 32 elements of shared memory, free again on return.
__device__ __forceinline__ void block_sum2(unsigned long long &a, unsigned long long &b, unsigned long long *sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
  if (lane == 0) {
    sh[wid] = a;
    sh[16 + wid] = b;
  }
  __syncthreads();
  a = 0;
  b = 0;
  for (int w = 0; w < nw; ++w) {
    a += sh[w];
    b += sh[16 + w];
  }
  __syncthreads();
}

// Keep flags of one scored segment (nb blocks from imp[b0]) into skeep[0, nb), run by all
// kToppThreads threads of the CTA: fixed-point masses, exact totals, rank keys sorted (register
// bitonic up to 512 blocks, rank counting up to 1024, shared-memory bitonic beyond; skeys holds
// the padded sort), ranked exclusive scan, keep while below the integer threshold.  Returns false
// (status raised) when a score is not in [0, 1].
__device__ bool select_segment_blocks(const float *__restrict__ imp, int32_t b0, int32_t nb, double p,
                                      uint32_t flags, unsigned long long *skeys, uint8_t *skeep,
                                      unsigned long long *sh64, uint32_t *s_bad, uint32_t *status) {
  const int tid = threadIdx.x;
  if (tid == 0) *s_bad = 0;
  int npow = 1;
  while (npow < nb) npow <<= 1;
  const bool f_first = (flags & UNIP_KEEP_FIRST) != 0;
  const bool f_last = (flags & UNIP_KEEP_LAST) != 0;
  __syncthreads();

  // 1. scores -> rank keys (forced blocks and padding sort last), exact totals
  unsigned long long tsum = 0, fsum = 0;
  uint32_t bad = 0;
  for (int b = tid; b < npow; b += kToppThreads) {
    unsigned long long key = ~0ull;
    uint8_t kf = 0;
    if (b < nb) {
      float f = imp[b0 + b];
      // a zero score is +0 whatever its sign bit: no mass, and ranked as zero
      if (__float_as_uint(f) == 0x80000000u) f = __uint_as_float(0u);
      if (!(f >= 0.f) || f > 1.f) {
        bad = 1;
      } else {
        const unsigned long long qb = fixed_mass(f);
        tsum += qb;
        if ((f_first && b == 0) || (f_last && b == nb - 1)) {
          fsum += qb;
          kf = 1;
        } else {
          key = rank_key(f, b);
        }
      }
      skeep[b] = kf;
    }
    skeys[b] = key;
  }
  if (bad) atomicOr(s_bad, 1u);
  unsigned long long T = tsum, CF = fsum;
  block_sum2(T, CF, sh64);  // its barrier also publishes s_bad
  if (*s_bad) {
    if (tid == 0) atomicOr(status, UNIP_DEV_BAD_SCORES);
    return false;
  }
  if (T == 0) {
    for (int b = tid; b < nb; b += kToppThreads) skeep[b] = 1;
  } else if (npow <= kToppThreads) {
    // Up to 512 blocks: bitonic sort with one key per thread, in registers.
    const unsigned long long kthr = mass_threshold(p, T);
    unsigned long long key = tid < npow ? skeys[tid] : ~0ull;
    bitonic_sort_regs(key, skeys, tid, npow);
    // thread tid now holds the key of rank tid; forced blocks and padding sort last
    const unsigned long long m = key != ~0ull ? fixed_mass(key_score(key)) : 0ull;
    unsigned long long tot;
    const unsigned long long ex = block_excl_scan<unsigned long long>(m, sh64, &tot);
    if (key != ~0ull) skeep[key & 0xFFFFFFFFull] = CF + ex < kthr ? 1 : 0;
  } else if (nb <= kRankCountMax) {
    // Small segment: the rank of a block is the number of smaller keys (keys are unique), so
    // no sort is needed.  Forced blocks and padding hold the largest key and are never counted.
    const unsigned long long kthr = mass_threshold(p, T);
    constexpr int kPer = kRankCountMax / kToppThreads;
    const int npad = (nb + 15) & ~15;  // keys past npow are padded with the largest key up to npad
    for (int b = npow + tid; b < npad; b += kToppThreads) skeys[b] = ~0ull;
    __syncthreads();
    int rank[kPer];
    unsigned long long mine[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int b = tid + e * kToppThreads;
      rank[e] = -1;
      mine[e] = b < nb ? skeys[b] : ~0ull;
      if (mine[e] != ~0ull) {
        const ulonglong2 *k2 = reinterpret_cast<const ulonglong2 *>(skeys);  // two keys per load
        int r = 0;
        for (int o = 0; o < npad / 2; o += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const ulonglong2 kk = k2[o + u];
            r += (kk.x < mine[e] ? 1 : 0) + (kk.y < mine[e] ? 1 : 0);
          }
        }
        rank[e] = r;
      }
    }
    __syncthreads();  // every key has been read; the key array now holds masses in rank order
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (rank[e] >= 0) skeys[rank[e]] = fixed_mass(key_score(mine[e]));
    __syncthreads();
    const int R = nb - (f_first ? 1 : 0) - ((f_last && !(f_first && nb == 1)) ? 1 : 0);
    const int ipt = (R + kToppThreads - 1) / kToppThreads;
    const int r0 = tid * ipt;
    unsigned long long local = 0;
    for (int e = 0; e < ipt; ++e)
      if (r0 + e < R) local += skeys[r0 + e];
    unsigned long long tot;
    unsigned long long run = block_excl_scan<unsigned long long>(local, sh64, &tot);
    for (int e = 0; e < ipt; ++e) {
      if (r0 + e < R) {
        const unsigned long long m = skeys[r0 + e];
        skeys[r0 + e] = run;  // exclusive prefix of ranked masses, in place
        run += m;
      }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (rank[e] >= 0) skeep[tid + e * kToppThreads] = CF + skeys[rank[e]] < kthr ? 1 : 0;
  } else {
    const unsigned long long kthr = mass_threshold(p, T);
    // 2. bitonic sort, ascending key = score descending, index ascending
    for (int size = 2; size <= npow; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < npow / 2; i += kToppThreads) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool asc = (lo & size) == 0;
          const unsigned long long x = skeys[lo], y = skeys[hi];
          if ((x > y) == asc) {
            skeys[lo] = y;
            skeys[hi] = x;
          }
        }
        __syncthreads();
      }
    }
    // 3. ranked masses (recovered from the keys), exclusive scan, keep while below the threshold
    const int R = nb - (f_first ? 1 : 0) - ((f_last && !(f_first && nb == 1)) ? 1 : 0);
    const int ipt = (R + kToppThreads - 1) / kToppThreads;  // contiguous ranks per thread
    const int r0 = tid * ipt;
    unsigned long long local = 0;
    for (int e = 0; e < ipt; ++e) {
      const int r = r0 + e;
      if (r < R) local += fixed_mass(key_score(skeys[r]));
    }
    unsigned long long tot;
    unsigned long long run = block_excl_scan<unsigned long long>(local, sh64, &tot);
    for (int e = 0; e < ipt; ++e) {
      const int r = r0 + e;
      if (r < R) {
        const unsigned long long key = skeys[r];
        skeep[key & 0xFFFFFFFFull] = CF + run < kthr ? 1 : 0;
        run += fixed_mass(key_score(key));
      }
    }
  }
  __syncthreads();
  return true;
}

// Keep flags of a selected segment out to global memory, with the kept-token offset of every block
// (exclusive, in block order) and the segment's kept-token count.
__device__ __forceinline__ void write_segment_selection(int32_t s, int32_t b0, int32_t nb, int32_t n, int32_t B,
                                                        const uint8_t *skeep, uint8_t *__restrict__ keep,
                                                        int32_t *__restrict__ kept_off,
                                                        int32_t *__restrict__ seg_kept, int32_t *sh32) {
  const int tid = threadIdx.x;
  const int ipb = (nb + kToppThreads - 1) / kToppThreads;
  const int bb0 = tid * ipb;
  int32_t lsum = 0;
  for (int e = 0; e < ipb; ++e) {
    const int b = bb0 + e;
    if (b < nb && skeep[b]) lsum += min(B, n - b * B);
  }
  int32_t tot;
  int32_t run = block_excl_scan<int32_t>(lsum, sh32, &tot);
  for (int e = 0; e < ipb; ++e) {
    const int b = bb0 + e;
    if (b < nb) {
      keep[b0 + b] = skeep[b];
      kept_off[b0 + b] = run;
      if (skeep[b]) run += min(B, n - b * B);
    }
  }
  if (tid == 0) seg_kept[s] = tot;
}

// Selection of a segment of at most 32 blocks by one warp, block b on lane b (f: its score, read by
// lanes below nb), in registers: the same fixed-point masses, exact totals and integer threshold as
// select_segment_blocks, with the exclusive mass of the blocks ranked before a block summed over
// the lanes holding a smaller key (keys are unique, so that set is exactly the blocks ranked
// before it).  Writes keep, the kept-token offsets and the segment's count, or only a zero count
// (status raised) when a score is not in [0, 1].
__device__ void select_small_segment(float f, int32_t s, int32_t b0, int32_t nb, int32_t n, int32_t B, double p,
                                     uint32_t flags, uint8_t *__restrict__ keep, int32_t *__restrict__ kept_off,
                                     int32_t *__restrict__ seg_kept, uint32_t *__restrict__ status) {
  const int lane = threadIdx.x & 31;
  const bool live = lane < nb;
  if (__float_as_uint(f) == 0x80000000u) f = __uint_as_float(0u);  // a zero score is +0
  const bool bad = live && (!(f >= 0.f) || f > 1.f);
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) {
      atomicOr(status, UNIP_DEV_BAD_SCORES);
      seg_kept[s] = 0;
    }
    return;
  }
  const bool forced = live && (((flags & UNIP_KEEP_FIRST) && lane == 0) || ((flags & UNIP_KEEP_LAST) && lane == nb - 1));
  const unsigned long long qb = live ? fixed_mass(f) : 0ull;
  unsigned long long T = qb, CF = forced ? qb : 0ull;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    T += __shfl_xor_sync(0xffffffffu, T, off);
    CF += __shfl_xor_sync(0xffffffffu, CF, off);
  }
  bool kf = live;  // a zero total keeps every block
  if (T != 0) {
    const unsigned long long kthr = mass_threshold(p, T);
    const unsigned long long key = live && !forced ? rank_key(f, lane) : ~0ull;
    unsigned long long pre = 0;
    for (int j = 0; j < nb; ++j) {
      const unsigned long long kj = __shfl_sync(0xffffffffu, key, j);
      const unsigned long long qj = __shfl_sync(0xffffffffu, qb, j);
      if (kj < key) pre += qj;
    }
    kf = forced || (live && CF + pre < kthr);
  }
  // kept-token offsets in block order (exclusive) and the segment's count
  const int32_t len = kf ? min(B, n - lane * B) : 0;
  const int32_t incl = warp_incl_scan(len);
  const int32_t tot = __shfl_sync(0xffffffffu, incl, 31);
  if (live) {
    keep[b0 + lane] = kf ? 1 : 0;
    kept_off[b0 + lane] = incl - len;
  }
  if (lane == 0) seg_kept[s] = tot;
}

__global__ void __launch_bounds__(kToppThreads) topp_kernel(
    const float *__restrict__ imp, const int32_t *__restrict__ blk_cu, const int32_t *__restrict__ cu, int32_t B,
    double p, uint32_t flags, uint8_t *__restrict__ keep, int32_t *__restrict__ kept_off,
    int32_t *__restrict__ seg_kept, int32_t cap, uint32_t *__restrict__ status) {
  extern __shared__ unsigned long long skeys[];  // cap rank keys, then cap keep flags
  uint8_t *skeep = reinterpret_cast<uint8_t *>(skeys + cap);
  __shared__ unsigned long long sh64[32];
  __shared__ int32_t sh32[32];
  __shared__ uint32_t s_bad;
  const int tid = threadIdx.x;
  // A gather launched as a programmatic dependent may start now; it waits for this grid's results.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // This grid may itself run as a programmatic dependent of the importance kernels: no memory is
  // touched before their results are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t s = blockIdx.x;
  const int32_t n = cu[s + 1] - cu[s];
  const int32_t b0 = blk_cu[s], nb = blk_cu[s + 1] - blk_cu[s];

  if (nb == 0) {  // not scored: every token is kept
    if (tid == 0) seg_kept[s] = n > 0 ? n : 0;
    return;
  }
  // cap (a power of two) bounds the padded sort of every segment that fits the call's token count
  if (nb > kMaxBlocks || nb > cap || n <= 0 || nb != (n + B - 1) / B) {
    if (tid == 0) {
      atomicOr(status, nb > kMaxBlocks ? UNIP_DEV_TOO_MANY_BLOCKS : UNIP_DEV_BAD_BLOCKS);
      seg_kept[s] = 0;
    }
    return;
  }
  if (nb <= 32) {  // one warp, no barriers
    if (tid < 32)
      select_small_segment(tid < nb ? imp[b0 + tid] : 0.f, s, b0, nb, n, B, p, flags, keep, kept_off, seg_kept,
                           status);
    return;
  }
  if (!select_segment_blocks(imp, b0, nb, p, flags, skeys, skeep, sh64, &s_bad, status)) {
    if (tid == 0) seg_kept[s] = 0;
    return;
  }
  write_segment_selection(s, b0, nb, n, B, skeep, keep, kept_off, seg_kept, sh32);
}

// Normalisation and Top-p of one segment per CTA: the normaliser of unip_block_importance (the same
// fp32 arithmetic, so imp has the same bits) followed, in the same CTA, by the selection of
// topp_kernel on the scores it just wrote; launched as a programmatic dependent of the score grid.
__global__ void __launch_bounds__(kToppThreads) norm_select_kernel(
    const int32_t *__restrict__ blk_cu, const int32_t *__restrict__ cu, const float *__restrict__ partial,
    int32_t Hkv, int32_t B, double p, uint32_t flags, int32_t cap, float *__restrict__ imp,
    uint8_t *__restrict__ keep, int32_t *__restrict__ kept_off, int32_t *__restrict__ seg_kept,
    uint32_t *__restrict__ status) {
  extern __shared__ unsigned long long skeys[];  // cap rank keys, then cap keep flags
  uint8_t *skeep = reinterpret_cast<uint8_t *>(skeys + cap);
  __shared__ unsigned long long sh64[32];
  __shared__ int32_t sh32[32];
  __shared__ uint32_t s_bad;
  __shared__ float sred[kImpNormThreads];
  const int tid = threadIdx.x;
  // the row-copy grid may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the score grid's masses are complete past here
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t s = blockIdx.x;
  const int32_t n = cu[s + 1] - cu[s];
  const int32_t b0 = blk_cu[s], nb = blk_cu[s + 1] - blk_cu[s];
  if (nb == 0) {  // not scored: every token is kept
    if (tid == 0) seg_kept[s] = n > 0 ? n : 0;
    return;
  }
  if (nb > kMaxBlocks || nb > cap || n <= 0 || nb != (n + B - 1) / B) {
    if (tid == 0) {
      atomicOr(status, nb > kMaxBlocks ? UNIP_DEV_TOO_MANY_BLOCKS : UNIP_DEV_BAD_BLOCKS);
      seg_kept[s] = 0;
    }
    return;
  }
  if (nb <= 32) {
    // One warp, block b on lane b.  The normaliser's tree over at most 32 nonzero masses (the
    // other slots add exact zeros) pairs the same partial sums as the lanes' xor butterfly, so the
    // scores have the bits normalise_segment gives them.
    if (tid < 32) {
      float m = 0.f;
      if (tid < nb)
        for (int32_t g = 0; g < Hkv; ++g) m += partial[(int64_t)(b0 + tid) * Hkv + g];
      float t = m;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
      const float f = m * (1.f / t);
      if (tid < nb) imp[b0 + tid] = f;
      select_small_segment(f, s, b0, nb, n, B, p, flags, keep, kept_off, seg_kept, status);
    }
    return;
  }
  normalise_segment(partial, b0, nb, Hkv, imp, sred);
  __syncthreads();  // this CTA's scores are written before it reads them back
  if (!select_segment_blocks(imp, b0, nb, p, flags, skeys, skeep, sh64, &s_bad, status)) {
    if (tid == 0) seg_kept[s] = 0;
    return;
  }
  write_segment_selection(s, b0, nb, n, B, skeep, keep, kept_off, seg_kept, sh32);
}

// Copies n0 ints of src0 to dst0 and n1 ints of src1 to dst1 (shared memory), each thread issuing
// all of its loads of a round before any store, so the copy costs about one memory round trip.
__device__ __forceinline__ void stage_two(int32_t *__restrict__ dst0, const int32_t *__restrict__ src0, int32_t n0,
                                          int32_t *__restrict__ dst1, const int32_t *__restrict__ src1, int32_t n1) {
  constexpr int kPer = 8;
  const int32_t n = n0 + n1;
  for (int32_t base = 0; base < n; base += kIndexThreads * kPer) {
    int32_t v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int32_t i = base + u * kIndexThreads + threadIdx.x;
      v[u] = i < n0 ? src0[i] : (i < n ? src1[i - n0] : 0);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int32_t i = base + u * kIndexThreads + threadIdx.x;
      if (i < n0) dst0[i] = v[u];
      else if (i < n) dst1[i - n0] = v[u];
    }
  }
}

// Kept-token offsets of every segment, exclusive, in place: soff[0, S) holds the per-segment kept
// counts on entry (written by this CTA's threads), the offsets on exit, and soff[S] the total.
// Every CTA of a gather grid recomputes them: S is small next to N, and this saves a launch and
// any cross-CTA handshake.
__device__ void segment_offsets_inplace(int32_t S, int32_t *__restrict__ soff, int32_t *sh32) {
  __syncthreads();
  const int32_t per = (S + kIndexThreads - 1) / kIndexThreads;
  const int32_t i0 = threadIdx.x * per;
  int32_t run = 0;
  for (int32_t e = 0; e < per && i0 + e < S; ++e) run += soff[i0 + e];
  int32_t tot;
  run = block_excl_scan<int32_t>(run, sh32, &tot);  // every count has been read past its barriers
  for (int32_t e = 0; e < per && i0 + e < S; ++e) {
    const int32_t c = soff[i0 + e];
    soff[i0 + e] = run;
    run += c;
  }
  if (threadIdx.x == 0) soff[S] = tot;
  __syncthreads();
}

// The same from the counts in global memory.
__device__ void segment_offsets(const int32_t *__restrict__ seg_kept, int32_t S, int32_t *__restrict__ soff,
                                int32_t *sh32) {
  stage_two(soff, seg_kept, S, nullptr, nullptr, 0);
  segment_offsets_inplace(S, soff, sh32);
}

__global__ void __launch_bounds__(kIndexThreads) index_kernel(
    const int32_t *__restrict__ cu, const int32_t *__restrict__ pos, const int32_t *__restrict__ blk_cu,
    const uint8_t *__restrict__ keep, const int32_t *__restrict__ kept_off, const int32_t *__restrict__ seg_kept,
    int32_t S, int32_t N, int32_t B, int32_t *__restrict__ cu_kept, int32_t *__restrict__ n_kept,
    int32_t *__restrict__ gather_idx, int32_t *__restrict__ pos_kept) {
  extern __shared__ int32_t soff[];  // S + 1 kept-token offsets
  __shared__ int32_t sh32[32];
  segment_offsets(seg_kept, S, soff, sh32);
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= S; i += kIndexThreads) cu_kept[i] = soff[i];
    if (threadIdx.x == 0) *n_kept = soff[S];
  }
  const int32_t t = blockIdx.x * kIndexThreads + threadIdx.x;
  if (t >= N) return;
  const int32_t s = find_segment(cu, S, t);
  const int32_t c0 = cu[s], n = cu[s + 1] - c0, i = t - c0;
  const int32_t nb = blk_cu[s + 1] - blk_cu[s];
  int32_t dest;
  if (nb == 0) {
    dest = soff[s] + i;
  } else {
    if (nb > kMaxBlocks || nb != (n + B - 1) / B) return;
    const int32_t b = i / B;
    if (!keep[blk_cu[s] + b]) return;
    dest = soff[s] + kept_off[blk_cu[s] + b] + (i - b * B);
  }
  if (dest < soff[s] || dest >= soff[s + 1]) return;  // a rejected segment keeps nothing
  gather_idx[dest] = t;
  pos_kept[dest] = pos[t];
}

// Same offsets for very many segments: one CTA writes them to global memory first.
__global__ void __launch_bounds__(kIndexThreads) kept_offsets_kernel(const int32_t *__restrict__ seg_kept,
                                                                     int32_t S, int32_t *__restrict__ cu_kept,
                                                                     int32_t *__restrict__ n_kept) {
  __shared__ int32_t sh32[32];
  int32_t carry = 0;
  for (int base = 0; base < S; base += kIndexThreads) {
    const int sidx = base + threadIdx.x;
    const int32_t v = sidx < S ? seg_kept[sidx] : 0;
    int32_t tot;
    const int32_t ex = block_excl_scan<int32_t>(v, sh32, &tot);
    if (sidx < S) cu_kept[sidx] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    cu_kept[S] = carry;
    *n_kept = carry;
  }
}

__global__ void __launch_bounds__(kIndexThreads) index_global_kernel(
    const int32_t *__restrict__ cu, const int32_t *__restrict__ pos, const int32_t *__restrict__ blk_cu,
    const uint8_t *__restrict__ keep, const int32_t *__restrict__ kept_off, const int32_t *__restrict__ cu_kept,
    int32_t S, int32_t N, int32_t B, int32_t *__restrict__ gather_idx, int32_t *__restrict__ pos_kept) {
  const int32_t t = blockIdx.x * kIndexThreads + threadIdx.x;
  if (t >= N) return;
  const int32_t s = find_segment(cu, S, t);
  const int32_t c0 = cu[s], n = cu[s + 1] - c0, i = t - c0;
  const int32_t nb = blk_cu[s + 1] - blk_cu[s];
  int32_t dest;
  if (nb == 0) {
    dest = cu_kept[s] + i;
  } else {
    if (nb > kMaxBlocks || nb != (n + B - 1) / B) return;
    const int32_t b = i / B;
    if (!keep[blk_cu[s] + b]) return;
    dest = cu_kept[s] + kept_off[blk_cu[s] + b] + (i - b * B);
  }
  if (dest < cu_kept[s] || dest >= cu_kept[s + 1]) return;
  gather_idx[dest] = t;
  pos_kept[dest] = pos[t];
}

// Fused index build + row gather: kept row r is found from the per-segment
// counts (shared-memory scan) and the per-block kept offsets (binary search,
// staged in shared memory when they fit); one warp writes gather_idx /
// positions_kept and copies the hidden row.
__global__ void __launch_bounds__(kIndexThreads) select_gather_kernel(
    const uint4 *__restrict__ hidden, int32_t num_rows, int64_t stride16, int32_t vec_per_row,
    const int32_t *__restrict__ cu, const int32_t *__restrict__ pos, const int32_t *__restrict__ blk_cu,
    const uint8_t *__restrict__ keep, const int32_t *__restrict__ kept_off, const int32_t *__restrict__ seg_kept,
    int32_t S, int32_t B, int32_t capacity, uint4 *__restrict__ out, int64_t out_stride16,
    int32_t *__restrict__ cu_kept, int32_t *__restrict__ n_kept, int32_t *__restrict__ gather_idx,
    int32_t *__restrict__ pos_kept, int32_t stage_blocks, uint32_t *__restrict__ status) {
  extern __shared__ int32_t soff[];  // S + 1 kept-token offsets, then (optionally) per-block kept offsets
  __shared__ int32_t sh32[32];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the Top-p grid's results are visible past here
  // The block count, the staged block offsets and the segment counts are loaded in one round trip:
  // stage_blocks bounds the call's blocks and the workspace holds that many offsets, so the entries
  // past the real count are read (never used) instead of waiting for the count first.
  const int32_t nblk = blk_cu[S];
  int32_t *skoff = soff + S + 1;
  stage_two(soff, seg_kept, S, skoff, kept_off, stage_blocks);
  const bool staged = nblk <= stage_blocks;
  segment_offsets_inplace(S, soff, sh32);  // its barriers publish skoff
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= S; i += kIndexThreads) cu_kept[i] = soff[i];
    if (threadIdx.x == 0) *n_kept = soff[S];
  }
  int32_t total = soff[S];
  if (total > capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, UNIP_DEV_BAD_INDEX);
    total = capacity;
  }
  const int lane = threadIdx.x & 31;
  const int warps_per_block = kIndexThreads / 32;
  const int32_t nwarps = gridDim.x * warps_per_block;
  for (int32_t r = blockIdx.x * warps_per_block + (threadIdx.x >> 5); r < total; r += nwarps) {
    int32_t lo = 0, hi = S - 1;  // segment: last s with soff[s] <= r
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (soff[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int32_t sg = lo, local = r - soff[sg], c0 = cu[sg];
    const int32_t b0 = blk_cu[sg], nb = blk_cu[sg + 1] - b0;
    int32_t src;
    if (nb == 0) {
      src = c0 + local;
    } else {
      // block: last b with kept_off[b] <= local.  kept_off is non-decreasing and a dropped block
      // shares its offset with the next kept one, so the answer is always a kept block.
      const int32_t *ko = staged ? skoff + b0 : kept_off + b0;
      int32_t blo = 0, bhi = nb - 1;
      while (blo < bhi) {
        const int32_t mid = (blo + bhi + 1) >> 1;
        if (ko[mid] <= local) blo = mid; else bhi = mid - 1;
      }
      if (!keep[b0 + blo]) continue;
      src = c0 + blo * B + (local - ko[blo]);
    }
    if (src < 0 || src >= num_rows) {
      if (lane == 0) atomicOr(status, UNIP_DEV_BAD_INDEX);
      continue;
    }
    if (lane == 0) {
      gather_idx[r] = src;
      pos_kept[r] = pos[src];
    }
    warp_copy_row(hidden + (int64_t)src * stride16, out + (int64_t)r * out_stride16, vec_per_row, lane);
  }
}

// Kept-token offsets of a one-segment call's blocks (exclusive, in block order) into skoff from the
// keep flags the CTA selected itself; CTA 0 also writes the keep mask.  Returns the kept-token count.
__device__ __forceinline__ int32_t onepass_offsets(int32_t n, int32_t b0, int32_t nb, int32_t B, const uint8_t *skeep,
                                                   int32_t *skoff, uint8_t *__restrict__ keep, int32_t *sh32) {
  const int tid = threadIdx.x;
  const int ipb = (nb + kToppThreads - 1) / kToppThreads;
  const int bb0 = tid * ipb;
  int32_t lsum = 0;
  for (int e = 0; e < ipb; ++e) {
    const int b = bb0 + e;
    if (b < nb && skeep[b]) lsum += min(B, n - b * B);
  }
  int32_t total;
  int32_t run = block_excl_scan<int32_t>(lsum, sh32, &total);
  for (int e = 0; e < ipb; ++e) {
    const int b = bb0 + e;
    if (b < nb) {
      skoff[b] = run;
      if (blockIdx.x == 0) keep[b0 + b] = skeep[b];
      if (skeep[b]) run += min(B, n - b * B);
    }
  }
  return total;
}

// The rest of a one-segment call once every CTA knows the kept blocks (skeep, skoff) and their token
// count: CTA 0 writes cu_seqlens_kept and n_kept, and each warp of the grid takes kept rows r in turn,
// writing gather_idx / positions_kept and copying the hidden row.  Consecutive rows go to consecutive
// CTAs, so a short list of rows still spreads over every SM.  nb == 0: every token is kept.
__device__ __forceinline__ void onepass_copy(int32_t total, int32_t c0, int32_t nb, int32_t B, const uint8_t *skeep,
                                             const int32_t *skoff, const int32_t *__restrict__ pos,
                                             const uint4 *__restrict__ hidden, int32_t num_rows, int64_t stride16,
                                             int32_t vec_per_row, uint4 *__restrict__ out, int64_t out_stride16,
                                             int32_t *__restrict__ cu_kept, int32_t *__restrict__ n_kept,
                                             int32_t *__restrict__ gather_idx, int32_t *__restrict__ pos_kept,
                                             uint32_t *__restrict__ status) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (blockIdx.x == 0 && tid == 0) {
    cu_kept[0] = 0;
    cu_kept[1] = total;
    *n_kept = total;
  }
  __syncthreads();
  const int warps_per_block = kToppThreads / 32;
  for (int32_t r = (tid >> 5) * gridDim.x + blockIdx.x; r < total; r += gridDim.x * warps_per_block) {
    int32_t src;
    if (nb == 0) {
      src = c0 + r;
    } else {
      // block: last b with skoff[b] <= r (a dropped block shares its offset with the next kept one)
      int32_t lo = 0, hi = nb - 1;
      while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (skoff[mid] <= r) lo = mid; else hi = mid - 1;
      }
      if (!skeep[lo]) continue;
      src = c0 + lo * B + (r - skoff[lo]);
    }
    if (src < 0 || src >= num_rows) {
      if (lane == 0) atomicOr(status, UNIP_DEV_BAD_INDEX);
      continue;
    }
    if (lane == 0) {
      gather_idx[r] = src;
      pos_kept[r] = pos[src];
    }
    warp_copy_row(hidden + (int64_t)src * stride16, out + (int64_t)r * out_stride16, vec_per_row, lane);
  }
}

// One segment in the call (a single long prompt): every CTA selects the segment's blocks itself
// (a few microseconds of shared-memory work on at most UNIP_TOPP_MAX_BLOCKS scores), stages the
// kept offsets and copies its share of the kept rows, so no grid waits for another; CTA 0 writes
// the keep mask, cu_seqlens_kept and n_kept.  Same results as topp_kernel + select_gather_kernel.
__global__ void __launch_bounds__(kToppThreads) select_gather_onepass_kernel(
    const float *__restrict__ imp, const int32_t *__restrict__ blk_cu, const int32_t *__restrict__ cu,
    const int32_t *__restrict__ pos, int32_t B, double p, uint32_t flags, int32_t cap, uint8_t *__restrict__ keep,
    const uint4 *__restrict__ hidden, int32_t num_rows, int64_t stride16, int32_t vec_per_row,
    uint4 *__restrict__ out, int64_t out_stride16, int32_t *__restrict__ cu_kept, int32_t *__restrict__ n_kept,
    int32_t *__restrict__ gather_idx, int32_t *__restrict__ pos_kept, uint32_t *__restrict__ status) {
  extern __shared__ unsigned long long skeys[];  // cap rank keys, cap kept offsets (int32), cap flags
  int32_t *skoff = reinterpret_cast<int32_t *>(skeys + cap);
  uint8_t *skeep = reinterpret_cast<uint8_t *>(skoff + cap);
  __shared__ unsigned long long sh64[32];
  __shared__ int32_t sh32[32];
  __shared__ uint32_t s_bad;
  // the importance results are visible past here (this grid is a programmatic dependent of them)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t c0 = cu[0], n = cu[1] - cu[0];
  const int32_t b0 = blk_cu[0], nb = blk_cu[1] - blk_cu[0];
  int32_t total = 0;
  if (nb == 0) {  // not scored: every token is kept
    total = n > 0 ? n : 0;
  } else if (nb > kMaxBlocks || nb > cap || n <= 0 || nb != (n + B - 1) / B) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      atomicOr(status, nb > kMaxBlocks ? UNIP_DEV_TOO_MANY_BLOCKS : UNIP_DEV_BAD_BLOCKS);
  } else if (select_segment_blocks(imp, b0, nb, p, flags, skeys, skeep, sh64, &s_bad, status)) {
    total = onepass_offsets(n, b0, nb, B, skeep, skoff, keep, sh32);
  }
  onepass_copy(total, c0, nb, B, skeep, skoff, pos, hidden, num_rows, stride16, vec_per_row, out, out_stride16,
               cu_kept, n_kept, gather_idx, pos_kept, status);
}

// The fused importance call with one segment: every CTA normalises the segment's block masses itself
// (the normaliser of unip_block_importance, so the scores have the same bits; CTA 0 writes them out),
// selects from its own copy of the scores in shared memory and copies its share of the kept rows, as
// select_gather_onepass_kernel does.  One grid after the score grid, none waiting for another.
__global__ void __launch_bounds__(kToppThreads) norm_select_gather_onepass_kernel(
    const int32_t *__restrict__ blk_cu, const int32_t *__restrict__ cu, const float *__restrict__ partial,
    int32_t Hkv, const int32_t *__restrict__ pos, int32_t B, double p, uint32_t flags, int32_t cap,
    float *__restrict__ imp, uint8_t *__restrict__ keep, const uint4 *__restrict__ hidden, int32_t num_rows,
    int64_t stride16, int32_t vec_per_row, uint4 *__restrict__ out, int64_t out_stride16,
    int32_t *__restrict__ cu_kept, int32_t *__restrict__ n_kept, int32_t *__restrict__ gather_idx,
    int32_t *__restrict__ pos_kept, uint32_t *__restrict__ status) {
  // cap rank keys, cap int32 that hold the scores during the selection and the kept offsets after
  // it (the selection reads each score once, before it writes anything else), cap flags
  extern __shared__ unsigned long long skeys[];
  int32_t *skoff = reinterpret_cast<int32_t *>(skeys + cap);
  float *sscore = reinterpret_cast<float *>(skoff);
  uint8_t *skeep = reinterpret_cast<uint8_t *>(skoff + cap);
  __shared__ unsigned long long sh64[32];
  __shared__ int32_t sh32[32];
  __shared__ uint32_t s_bad;
  __shared__ float sred[kImpNormThreads];
  // the score grid's masses are complete past here
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t c0 = cu[0], n = cu[1] - cu[0];
  const int32_t b0 = blk_cu[0], nb = blk_cu[1] - blk_cu[0];
  int32_t total = 0;
  if (nb == 0) {  // not scored: every token is kept
    total = n > 0 ? n : 0;
  } else if (nb > kMaxBlocks || nb > cap || n <= 0 || nb != (n + B - 1) / B) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      atomicOr(status, nb > kMaxBlocks ? UNIP_DEV_TOO_MANY_BLOCKS : UNIP_DEV_BAD_BLOCKS);
  } else {
    normalise_segment(partial, b0, nb, Hkv, blockIdx.x == 0 ? imp : nullptr, sred, sscore);
    __syncthreads();  // the scores in shared memory are complete
    if (select_segment_blocks(sscore, 0, nb, p, flags, skeys, skeep, sh64, &s_bad, status))
      total = onepass_offsets(n, b0, nb, B, skeep, skoff, keep, sh32);
  }
  onepass_copy(total, c0, nb, B, skeep, skoff, pos, hidden, num_rows, stride16, vec_per_row, out, out_stride16,
               cu_kept, n_kept, gather_idx, pos_kept, status);
}

// Top-p launch: shared memory for the padded sort of the largest segment the call can hold
// (a power of two of at least total_tokens / B + 2 blocks, at most UNIP_TOPP_MAX_BLOCKS).
cudaError_t launch_topp(const float *imp, const int32_t *blk_cu, const int32_t *cu_seqlens, int32_t num_segs,
                        int32_t total_tokens, int32_t block_size, double p, uint32_t flags, uint8_t *keep,
                        int32_t *kept_off, int32_t *seg_kept, uint32_t *status, cudaStream_t st) {
  {
    const cudaError_t e =
        ensure_dynamic_smem((const void *)topp_kernel, kMaxBlocks * ((int)sizeof(unsigned long long) + 1));
    if (e != cudaSuccess) return e;
  }
  int32_t cap = 16;
  const int64_t need = (int64_t)total_tokens / block_size + 2;
  while (cap < need && cap < kMaxBlocks) cap <<= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_segs);
  cfg.blockDim = dim3(kToppThreads);
  cfg.dynamicSmemBytes = (size_t)cap * (sizeof(unsigned long long) + 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topp_kernel, imp, blk_cu, cu_seqlens, block_size, p, flags, keep, kept_off,
                            seg_kept, cap, status);
}

// Row copy after a selection grid (programmatic dependent of it): kept-token offsets per segment,
// then one warp per kept row writes gather_idx / positions_kept and copies the hidden row.
cudaError_t launch_gather_rows(const void *hidden, int64_t row_stride, int32_t d_model, bool rows,
                               const int32_t *cu_seqlens, const int32_t *positions, const int32_t *blk_cu,
                               const uint8_t *keep, const int32_t *kept_off, const int32_t *seg_kept,
                               int32_t num_segs, int32_t total_tokens, int32_t block_size, void *hidden_out,
                               int64_t out_row_stride, int32_t *cu_seqlens_kept, int32_t *n_kept,
                               int32_t *gather_idx, int32_t *positions_kept, uint32_t *status, cudaStream_t st) {
  const int sms = device_sm_count();
  const int warps_per_block = kIndexThreads / 32;
  int64_t blocks = ((int64_t)(total_tokens > 0 ? total_tokens : 1) + warps_per_block - 1) / warps_per_block;
  const int64_t max_blocks = (int64_t)(sms > 0 ? sms : 1) * kGatherCtasPerSm;
  if (blocks > max_blocks) blocks = max_blocks;
  // per-block kept offsets are staged in shared memory when the upper bound on blocks fits
  const int32_t blk_bound = unip_importance_capacity(total_tokens, num_segs, block_size);
  const int32_t stage_blocks =
      (int64_t)(num_segs + 1 + blk_bound) * 4 <= kGatherStageBytes ? blk_bound : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kIndexThreads);
  cfg.dynamicSmemBytes = (size_t)(num_segs + 1 + stage_blocks) * sizeof(int32_t);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(
      &cfg, select_gather_kernel, static_cast<const uint4 *>(hidden), total_tokens,
      rows ? (int64_t)(row_stride / 8) : 0, (int32_t)(d_model / 8), cu_seqlens, positions, blk_cu, keep, kept_off,
      seg_kept, num_segs, block_size, total_tokens, static_cast<uint4 *>(hidden_out),
      rows ? (int64_t)(out_row_stride / 8) : 0, cu_seqlens_kept, n_kept, gather_idx, positions_kept, stage_blocks,
      status);
}

}  // namespace
}  // namespace unip

using namespace unip;

extern "C" {

UNIP_API size_t unip_topp_workspace_size(int32_t total_tokens, int32_t num_segs, int32_t block_size) {
  if (total_tokens < 0 || num_segs < 0 || block_size <= 0) return 0;
  const size_t cap = (size_t)total_tokens / block_size + num_segs + 1;
  return kWsHeaderBytes + align_up(sizeof(int32_t) * (size_t)num_segs, 256) + align_up(sizeof(int32_t) * cap, 256);
}

UNIP_API int32_t unip_topp_select(const float *imp, const int32_t *blk_cu, const int32_t *cu_seqlens,
                                  const int32_t *positions, int32_t num_segs, int32_t total_tokens,
                                  int32_t block_size, double p, uint32_t flags, uint8_t *keep,
                                  int32_t keep_capacity, int32_t *gather_idx, int32_t *cu_seqlens_kept,
                                  int32_t *positions_kept, int32_t *n_kept, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  if (!blk_cu || !cu_seqlens || !cu_seqlens_kept || !n_kept || num_segs < 0 || total_tokens < 0)
    return UNIP_ERR_INVALID_ARGUMENT;
  if (block_size <= 0 || !(p >= 0.0 && p <= 1.0) || (flags & ~(UNIP_KEEP_FIRST | UNIP_KEEP_LAST)))
    return UNIP_ERR_INVALID_ARGUMENT;
  if (total_tokens > 0 && (!positions || !gather_idx || !positions_kept)) return UNIP_ERR_INVALID_ARGUMENT;
  if (keep_capacity < unip_importance_capacity(total_tokens, num_segs, block_size)) return UNIP_ERR_INVALID_ARGUMENT;
  if (!keep || !imp) return UNIP_ERR_INVALID_ARGUMENT;
  const size_t need = unip_topp_workspace_size(total_tokens, num_segs, block_size);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return UNIP_ERR_WORKSPACE;
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (num_segs == 0) {
    if (cudaMemsetAsync(cu_seqlens_kept, 0, sizeof(int32_t), st) != cudaSuccess ||
        cudaMemsetAsync(n_kept, 0, sizeof(int32_t), st) != cudaSuccess)
      return UNIP_ERR_CUDA;
    return UNIP_OK;
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *seg_kept = reinterpret_cast<int32_t *>(ws + kWsHeaderBytes);
  int32_t *kept_off = reinterpret_cast<int32_t *>(ws + kWsHeaderBytes + align_up(sizeof(int32_t) * num_segs, 256));
  if (launch_topp(imp, blk_cu, cu_seqlens, num_segs, total_tokens, block_size, p, flags, keep, kept_off, seg_kept,
                  status, st) != cudaSuccess)
    return UNIP_ERR_CUDA;
  const int grid = total_tokens > 0 ? (total_tokens + kIndexThreads - 1) / kIndexThreads : 1;
  if (num_segs < kIndexSmemSegs) {
    index_kernel<<<grid, kIndexThreads, (num_segs + 1) * sizeof(int32_t), st>>>(
        cu_seqlens, positions, blk_cu, keep, kept_off, seg_kept, num_segs, total_tokens, block_size,
        cu_seqlens_kept, n_kept, gather_idx, positions_kept);
  } else {
    kept_offsets_kernel<<<1, kIndexThreads, 0, st>>>(seg_kept, num_segs, cu_seqlens_kept, n_kept);
    if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;
    if (total_tokens > 0)
      index_global_kernel<<<grid, kIndexThreads, 0, st>>>(cu_seqlens, positions, blk_cu, keep, kept_off,
                                                          cu_seqlens_kept, num_segs, total_tokens, block_size,
                                                          gather_idx, positions_kept);
  }
  if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;
  return UNIP_OK;
}

UNIP_API int32_t unip_select_gather(const float *imp, const int32_t *blk_cu, const int32_t *cu_seqlens,
                                    const int32_t *positions, int32_t num_segs, int32_t total_tokens,
                                    int32_t block_size, double p, uint32_t flags, uint8_t *keep,
                                    int32_t keep_capacity, int32_t *gather_idx, int32_t *cu_seqlens_kept,
                                    int32_t *positions_kept, int32_t *n_kept, const void *hidden,
                                    int64_t row_stride, int32_t d_model, void *hidden_out, int64_t out_row_stride,
                                    void *workspace, size_t workspace_bytes, void *stream) {
  // d_model == 0 with both row pointers NULL: selection and indices only, no rows copied.
  const bool rows = d_model != 0 || hidden || hidden_out;
  if (rows) {
    if (!hidden || !hidden_out || d_model <= 0 || row_stride < d_model || out_row_stride < d_model)
      return UNIP_ERR_INVALID_ARGUMENT;
    if (!aligned16(hidden) || !aligned16(hidden_out) || (d_model % 8) || (row_stride % 8) || (out_row_stride % 8))
      return UNIP_ERR_ALIGNMENT;
  }
  if (num_segs >= kIndexSmemSegs) {  // very many segments: the two-call path
    const int32_t rc = unip_topp_select(imp, blk_cu, cu_seqlens, positions, num_segs, total_tokens, block_size, p,
                                        flags, keep, keep_capacity, gather_idx, cu_seqlens_kept, positions_kept,
                                        n_kept, workspace, workspace_bytes, stream);
    if (rc != UNIP_OK || !rows) return rc;
    return unip_gather_tokens(hidden, total_tokens, row_stride, d_model, gather_idx, n_kept, total_tokens,
                              hidden_out, out_row_stride, stream);
  }
  if (!blk_cu || !cu_seqlens || !cu_seqlens_kept || !n_kept || num_segs < 0 || total_tokens < 0)
    return UNIP_ERR_INVALID_ARGUMENT;
  if (block_size <= 0 || !(p >= 0.0 && p <= 1.0) || (flags & ~(UNIP_KEEP_FIRST | UNIP_KEEP_LAST)))
    return UNIP_ERR_INVALID_ARGUMENT;
  if (total_tokens > 0 && (!positions || !gather_idx || !positions_kept)) return UNIP_ERR_INVALID_ARGUMENT;
  if (keep_capacity < unip_importance_capacity(total_tokens, num_segs, block_size)) return UNIP_ERR_INVALID_ARGUMENT;
  if (!keep || !imp) return UNIP_ERR_INVALID_ARGUMENT;
  const size_t need = unip_topp_workspace_size(total_tokens, num_segs, block_size);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return UNIP_ERR_WORKSPACE;
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (num_segs == 0) {
    if (cudaMemsetAsync(cu_seqlens_kept, 0, sizeof(int32_t), st) != cudaSuccess ||
        cudaMemsetAsync(n_kept, 0, sizeof(int32_t), st) != cudaSuccess)
      return UNIP_ERR_CUDA;
    return UNIP_OK;
  }
  // One segment: selection and gather in one grid.  One CTA per SM, since every CTA runs the same
  // selection and two CTAs on an SM would share its issue slots.
  if (num_segs == 1) {
    if (ensure_dynamic_smem((const void *)select_gather_onepass_kernel,
                            kMaxBlocks * ((int)sizeof(unsigned long long) + 5)) != cudaSuccess)
      return UNIP_ERR_CUDA;
    int32_t cap = 16;
    const int64_t need = (int64_t)total_tokens / block_size + 2;
    while (cap < need && cap < kMaxBlocks) cap <<= 1;
    const int sms1 = device_sm_count();
    const int warps = kToppThreads / 32;
    int64_t blocks1 = ((int64_t)(total_tokens > 0 ? total_tokens : 1) + warps - 1) / warps;
    const int64_t max_blocks1 = sms1 > 0 ? sms1 : 1;
    if (blocks1 > max_blocks1) blocks1 = max_blocks1;
    cudaLaunchConfig_t cfg1 = {};
    cfg1.gridDim = dim3((unsigned)blocks1);
    cfg1.blockDim = dim3(kToppThreads);
    cfg1.dynamicSmemBytes = (size_t)cap * (sizeof(unsigned long long) + 5);
    cfg1.stream = st;
    cudaLaunchAttribute attr1[1];
    attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr1[0].val.programmaticStreamSerializationAllowed = 1;
    cfg1.attrs = attr1;
    cfg1.numAttrs = 1;
    const cudaError_t e1 = cudaLaunchKernelEx(
        &cfg1, select_gather_onepass_kernel, imp, blk_cu, cu_seqlens, positions, block_size, p, flags, cap, keep,
        static_cast<const uint4 *>(hidden), total_tokens, rows ? (int64_t)(row_stride / 8) : 0,
        (int32_t)(d_model / 8), static_cast<uint4 *>(hidden_out), rows ? (int64_t)(out_row_stride / 8) : 0,
        cu_seqlens_kept, n_kept, gather_idx, positions_kept, status);
    return e1 == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *seg_kept = reinterpret_cast<int32_t *>(ws + kWsHeaderBytes);
  int32_t *kept_off = reinterpret_cast<int32_t *>(ws + kWsHeaderBytes + align_up(sizeof(int32_t) * num_segs, 256));
  if (launch_topp(imp, blk_cu, cu_seqlens, num_segs, total_tokens, block_size, p, flags, keep, kept_off, seg_kept,
                  status, st) != cudaSuccess)
    return UNIP_ERR_CUDA;
  const cudaError_t e = launch_gather_rows(hidden, row_stride, d_model, rows, cu_seqlens, positions, blk_cu, keep,
                                           kept_off, seg_kept, num_segs, total_tokens, block_size, hidden_out,
                                           out_row_stride, cu_seqlens_kept, n_kept, gather_idx, positions_kept,
                                           status, st);
  return e == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
}

UNIP_API size_t unip_importance_select_gather_workspace_size(int32_t total_tokens, int32_t num_segs,
                                                             int32_t block_size, const unip_attn_params *prm) {
  const size_t a = unip_importance_workspace_size(total_tokens, num_segs, block_size, prm);
  const size_t b = unip_topp_workspace_size(total_tokens, num_segs, block_size);
  if (!a || !b) return 0;
  return align_up(a, 256) + b;
}

UNIP_API int32_t unip_importance_select_gather(
    const void *q, const void *k, const float *lse, const int32_t *cu_seqlens, const int32_t *positions,
    int32_t num_segs, int32_t total_tokens, const uint8_t *seg_mask, int32_t block_size,
    const unip_attn_params *prm, double p, uint32_t flags, float *imp, int32_t imp_capacity, int32_t *blk_cu,
    uint8_t *keep, int32_t *gather_idx, int32_t *cu_seqlens_kept, int32_t *positions_kept, int32_t *n_kept,
    const void *hidden, int64_t row_stride, int32_t d_model, void *hidden_out, int64_t out_row_stride,
    void *workspace, size_t workspace_bytes, void *stream) {
  const bool rows = d_model != 0 || hidden || hidden_out;
  if (rows) {
    if (!hidden || !hidden_out || d_model <= 0 || row_stride < d_model || out_row_stride < d_model)
      return UNIP_ERR_INVALID_ARGUMENT;
    if (!aligned16(hidden) || !aligned16(hidden_out) || (d_model % 8) || (row_stride % 8) || (out_row_stride % 8))
      return UNIP_ERR_ALIGNMENT;
  }
  if (!prm || !cu_seqlens || !blk_cu || !cu_seqlens_kept || !n_kept || num_segs < 0 || total_tokens < 0)
    return UNIP_ERR_INVALID_ARGUMENT;
  if (!(p >= 0.0 && p <= 1.0) || (flags & ~(UNIP_KEEP_FIRST | UNIP_KEEP_LAST))) return UNIP_ERR_INVALID_ARGUMENT;
  if (total_tokens > 0 && (!positions || !gather_idx || !positions_kept)) return UNIP_ERR_INVALID_ARGUMENT;
  if (!keep || !imp || imp_capacity < unip_importance_capacity(total_tokens, num_segs, block_size))
    return UNIP_ERR_INVALID_ARGUMENT;
  const size_t need = unip_importance_select_gather_workspace_size(total_tokens, num_segs, block_size, prm);
  if (!need || !workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return UNIP_ERR_WORKSPACE;
  const size_t ws_imp = align_up(unip_importance_workspace_size(total_tokens, num_segs, block_size, prm), 256);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  void *ws_sel = ws + ws_imp;
  const size_t ws_sel_bytes = workspace_bytes - ws_imp;
  if (num_segs >= kIndexSmemSegs) {  // very many segments: the separate calls
    const int32_t rc = unip_block_importance(q, k, lse, cu_seqlens, num_segs, total_tokens, seg_mask, block_size, prm,
                                             imp, imp_capacity, blk_cu, workspace, ws_imp, stream);
    if (rc != UNIP_OK) return rc;
    return unip_select_gather(imp, blk_cu, cu_seqlens, positions, num_segs, total_tokens, block_size, p, flags, keep,
                              imp_capacity, gather_idx, cu_seqlens_kept, positions_kept, n_kept, hidden, row_stride,
                              d_model, hidden_out, out_row_stride, ws_sel, ws_sel_bytes, stream);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float *partial = nullptr;
  int32_t rc = importance_scores(q, k, lse, cu_seqlens, num_segs, total_tokens, seg_mask, block_size, prm, imp,
                                 imp_capacity, blk_cu, workspace, ws_imp, st, &partial);
  if (rc != UNIP_OK) return rc;
  if (!partial)  // nothing was scored (no segment, or no token): every segment keeps all its tokens
    return unip_select_gather(imp, blk_cu, cu_seqlens, positions, num_segs, total_tokens, block_size, p, flags, keep,
                              imp_capacity, gather_idx, cu_seqlens_kept, positions_kept, n_kept, hidden, row_stride,
                              d_model, hidden_out, out_row_stride, ws_sel, ws_sel_bytes, stream);
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  int32_t cap = 16;
  const int64_t cap_need = (int64_t)total_tokens / block_size + 2;
  while (cap < cap_need && cap < kMaxBlocks) cap <<= 1;
  if (num_segs == 1) {  // one segment: normalisation, selection and row copy in one grid
    if (ensure_dynamic_smem((const void *)norm_select_gather_onepass_kernel,
                            kMaxBlocks * ((int)sizeof(unsigned long long) + 5)) != cudaSuccess)
      return UNIP_ERR_CUDA;
    // One CTA per SM: every CTA runs the same selection, and two on an SM share its issue slots
    // (the 45-stage network of 512 blocks took ~6 us instead of ~4.3 us); 16 copying warps per SM
    // still keep 128 KB of row loads in flight there.
    const int sms1 = device_sm_count();
    const int warps = kToppThreads / 32;
    int64_t blocks1 = ((int64_t)(total_tokens > 0 ? total_tokens : 1) + warps - 1) / warps;
    const int64_t max_blocks1 = sms1 > 0 ? sms1 : 1;
    if (blocks1 > max_blocks1) blocks1 = max_blocks1;
    cudaLaunchConfig_t cfg1 = {};
    cfg1.gridDim = dim3((unsigned)blocks1);
    cfg1.blockDim = dim3(kToppThreads);
    cfg1.dynamicSmemBytes = (size_t)cap * (sizeof(unsigned long long) + 5);
    cfg1.stream = st;
    cudaLaunchAttribute attr1[1];
    attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the score grid drains
    attr1[0].val.programmaticStreamSerializationAllowed = 1;
    cfg1.attrs = attr1;
    cfg1.numAttrs = 1;
    const cudaError_t e1 = cudaLaunchKernelEx(
        &cfg1, norm_select_gather_onepass_kernel, (const int32_t *)blk_cu, cu_seqlens, (const float *)partial,
        prm->num_heads_kv, positions, block_size, p, flags, cap, imp, keep, static_cast<const uint4 *>(hidden),
        total_tokens, rows ? (int64_t)(row_stride / 8) : 0, (int32_t)(d_model / 8),
        static_cast<uint4 *>(hidden_out), rows ? (int64_t)(out_row_stride / 8) : 0, cu_seqlens_kept, n_kept,
        gather_idx, positions_kept, status);
    return e1 == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
  }
  if (ensure_dynamic_smem((const void *)norm_select_kernel, kMaxBlocks * ((int)sizeof(unsigned long long) + 1)) !=
      cudaSuccess)
    return UNIP_ERR_CUDA;
  int32_t *seg_kept = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws_sel) + kWsHeaderBytes);
  int32_t *kept_off = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws_sel) + kWsHeaderBytes +
                                                  align_up(sizeof(int32_t) * num_segs, 256));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_segs);
  cfg.blockDim = dim3(kToppThreads);
  cfg.dynamicSmemBytes = (size_t)cap * (sizeof(unsigned long long) + 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the score grid drains
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, norm_select_kernel, (const int32_t *)blk_cu, cu_seqlens, (const float *)partial,
                         prm->num_heads_kv, block_size, p, flags, cap, imp, keep, kept_off, seg_kept,
                         status) != cudaSuccess)
    return UNIP_ERR_CUDA;
  const cudaError_t e = launch_gather_rows(hidden, row_stride, d_model, rows, cu_seqlens, positions, blk_cu, keep,
                                           kept_off, seg_kept, num_segs, total_tokens, block_size, hidden_out,
                                           out_row_stride, cu_seqlens_kept, n_kept, gather_idx, positions_kept,
                                           status, st);
  return e == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
}

}  // extern "C"
