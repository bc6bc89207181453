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
//   topp_kernel   one CTA per segment: bitonic sort of 64-bit rank keys in
//                 shared memory, exclusive scan of the ranked integer masses,
//                 keep decision per block, exclusive scan of kept lengths.
//                 The last CTA to finish (threadfence + ticket) scans the
//                 per-segment kept counts into cu_seqlens_kept and n_kept.
//   index_kernel  one thread per source token: writes gather_idx and
//                 positions_kept at the token's compacted slot.
#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kToppThreads = 512;
constexpr int kIndexThreads = 256;
constexpr int kMaxBlocks = UNIP_TOPP_MAX_BLOCKS;
constexpr int kWsHeaderBytes = 256;

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Exclusive scan of one value per thread over the CTA; *total gets the sum.
template <typename T>
__device__ T block_excl_scan(T v, T *sh_warp, T *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const T incl = warp_incl_scan(v);
  if (lane == 31) sh_warp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    T w = lane < nw ? sh_warp[lane] : T(0);
    w = warp_incl_scan(w);
    if (lane < nw) sh_warp[lane] = w;
  }
  __syncthreads();
  const T before = wid > 0 ? sh_warp[wid - 1] : T(0);
  *total = sh_warp[nw - 1];
  __syncthreads();
  return before + incl - v;
}

__global__ void __launch_bounds__(kToppThreads) topp_kernel(
    const float *__restrict__ imp, const int32_t *__restrict__ blk_cu, const int32_t *__restrict__ cu, int32_t S,
    int32_t B, double p, uint32_t flags, uint8_t *__restrict__ keep, int32_t *__restrict__ kept_off,
    int32_t *__restrict__ seg_kept, int32_t *__restrict__ ticket, int32_t *__restrict__ cu_kept,
    int32_t *__restrict__ n_kept, uint32_t *__restrict__ status) {
  extern __shared__ unsigned long long skeys[];  // kMaxBlocks rank keys
  __shared__ unsigned long long sh64[32];
  __shared__ int32_t sh32[32];
  __shared__ int s_last;
  __shared__ uint32_t s_bad;
  const int tid = threadIdx.x;
  const int32_t s = blockIdx.x;
  const int32_t n = cu[s + 1] - cu[s];
  const int32_t b0 = blk_cu[s], nb = blk_cu[s + 1] - blk_cu[s];
  constexpr int kItems = kMaxBlocks / kToppThreads;  // blocks per thread in the scans

  if (tid == 0) s_bad = 0;
  __syncthreads();
  int32_t kept_tokens = 0;
  if (nb == 0) {
    kept_tokens = n > 0 ? n : 0;
  } else if (nb > kMaxBlocks || n <= 0 || nb != (n + B - 1) / B) {
    if (tid == 0) atomicOr(status, nb > kMaxBlocks ? UNIP_DEV_TOO_MANY_BLOCKS : UNIP_DEV_BAD_BLOCKS);
    kept_tokens = 0;
  } else {
    // 1. fixed-point masses and their exact total
    unsigned long long tsum = 0;
    uint32_t bad = 0;
    for (int b = tid; b < nb; b += kToppThreads) {
      const float f = imp[b0 + b];
      if (!(f >= 0.f) || f > 1.f) bad = 1;
      else tsum += static_cast<unsigned long long>(floor(static_cast<double>(f) * 4294967296.0));
    }
    if (bad) atomicOr(&s_bad, 1u);
    unsigned long long T;
    block_excl_scan<unsigned long long>(tsum, sh64, &T);
    if (s_bad) {
      if (tid == 0) atomicOr(status, UNIP_DEV_BAD_SCORES);
      // leave kept_tokens = 0 for a segment with invalid scores
    } else if (T == 0) {
      for (int b = tid; b < nb; b += kToppThreads) keep[b0 + b] = 1;
    } else {
      const double thr = __dmul_rn(p, static_cast<double>(T));
      const bool f_first = (flags & UNIP_KEEP_FIRST) != 0;
      const bool f_last = (flags & UNIP_KEEP_LAST) != 0;
      auto forced = [&](int b) { return (f_first && b == 0) || (f_last && b == nb - 1); };
      // 2. rank keys: forced blocks (and padding) sort last
      int npow = 1;
      while (npow < nb) npow <<= 1;
      unsigned long long cum_f = 0;
      for (int b = tid; b < npow; b += kToppThreads) {
        unsigned long long key = ~0ull;
        if (b < nb) {
          const float f = imp[b0 + b];
          if (forced(b)) cum_f += static_cast<unsigned long long>(floor(static_cast<double>(f) * 4294967296.0));
          else key = (static_cast<unsigned long long>(~__float_as_uint(f)) << 32) | static_cast<uint32_t>(b);
        }
        skeys[b] = key;
      }
      unsigned long long CF;
      block_excl_scan<unsigned long long>(cum_f, sh64, &CF);
      // 3. bitonic sort, ascending key = score descending, index ascending
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
      // 4. ranked masses, exclusive scan, keep while the running mass is below thr
      const int R = nb - (f_first ? 1 : 0) - ((f_last && !(f_first && nb == 1)) ? 1 : 0);
      unsigned long long qv[kItems];
      unsigned long long local = 0;
#pragma unroll
      for (int e = 0; e < kItems; ++e) {
        const int r = tid * kItems + e;
        qv[e] = 0;
        if (r < R) {
          const uint32_t bi = static_cast<uint32_t>(skeys[r] & 0xFFFFFFFFull);
          qv[e] = static_cast<unsigned long long>(floor(static_cast<double>(imp[b0 + bi]) * 4294967296.0));
        }
        local += qv[e];
      }
      unsigned long long tot;
      unsigned long long run = block_excl_scan<unsigned long long>(local, sh64, &tot);
#pragma unroll
      for (int e = 0; e < kItems; ++e) {
        const int r = tid * kItems + e;
        if (r < R) {
          const uint32_t bi = static_cast<uint32_t>(skeys[r] & 0xFFFFFFFFull);
          keep[b0 + bi] = static_cast<double>(CF + run) < thr ? 1 : 0;
        }
        run += qv[e];
      }
      if (tid == 0) {
        if (f_first) keep[b0] = 1;
        if (f_last) keep[b0 + nb - 1] = 1;
      }
    }
    __syncthreads();
    // 5. kept token offsets in block order
    if (!s_bad) {
      int32_t lens[kItems];
      int32_t lsum = 0;
#pragma unroll
      for (int e = 0; e < kItems; ++e) {
        const int b = tid * kItems + e;
        lens[e] = 0;
        if (b < nb && keep[b0 + b]) lens[e] = min(B, n - b * B);
        lsum += lens[e];
      }
      int32_t tot;
      int32_t run = block_excl_scan<int32_t>(lsum, sh32, &tot);
#pragma unroll
      for (int e = 0; e < kItems; ++e) {
        const int b = tid * kItems + e;
        if (b < nb) kept_off[b0 + b] = run;
        run += lens[e];
      }
      kept_tokens = tot;
    }
  }
  if (tid == 0) seg_kept[s] = kept_tokens;
  // Last CTA: per-segment kept counts -> cu_seqlens_kept, n_kept.
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(ticket, 1) == static_cast<int32_t>(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int32_t carry = 0;
  for (int base = 0; base < S; base += kToppThreads) {
    const int sidx = base + tid;
    const int32_t v = sidx < S ? __ldcg(seg_kept + sidx) : 0;
    int32_t tot;
    const int32_t ex = block_excl_scan<int32_t>(v, sh32, &tot);
    if (sidx < S) cu_kept[sidx] = carry + ex;
    carry += tot;
  }
  if (tid == 0) {
    cu_kept[S] = carry;
    *n_kept = carry;
    *ticket = 0;
  }
}

__global__ void __launch_bounds__(kIndexThreads) index_kernel(
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
  if (dest < cu_kept[s] || dest >= cu_kept[s + 1]) return;  // a rejected segment keeps nothing
  gather_idx[dest] = t;
  pos_kept[dest] = pos[t];
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
  int32_t *ticket = reinterpret_cast<int32_t *>(ws);
  int32_t *seg_kept = reinterpret_cast<int32_t *>(ws + kWsHeaderBytes);
  int32_t *kept_off = reinterpret_cast<int32_t *>(ws + kWsHeaderBytes + align_up(sizeof(int32_t) * num_segs, 256));
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = kMaxBlocks * (int)sizeof(unsigned long long);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    if (cudaFuncSetAttribute(topp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return UNIP_ERR_CUDA;
    configured[dev] = true;
  }
  if (cudaMemsetAsync(ticket, 0, sizeof(int32_t), st) != cudaSuccess) return UNIP_ERR_CUDA;
  topp_kernel<<<num_segs, kToppThreads, smem, st>>>(imp, blk_cu, cu_seqlens, num_segs, block_size, p, flags, keep,
                                                    kept_off, seg_kept, ticket, cu_seqlens_kept, n_kept, status);
  if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;
  if (total_tokens > 0) {
    const int grid = (total_tokens + kIndexThreads - 1) / kIndexThreads;
    index_kernel<<<grid, kIndexThreads, 0, st>>>(cu_seqlens, positions, blk_cu, keep, kept_off, cu_seqlens_kept,
                                                 num_segs, total_tokens, block_size, gather_idx, positions_kept);
    if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;
  }
  return UNIP_OK;
}

}  // extern "C"
