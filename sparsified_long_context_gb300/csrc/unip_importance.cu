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
//   imp_score_kernel  one CTA per (work item, kv head): 128 threads, one key
//                     each; the window rows of the kv head's query-head group
//                     are staged in shared memory; per-block partial masses
//                     are reduced in registers/shuffles and written without
//                     atomics (deterministic).
//   imp_norm_kernel   one CTA per segment: sums the kv-head partials in a
//                     fixed order and divides by the segment total.
#include <cuda_bf16.h>

#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kChunk = 128;        // keys per score CTA
constexpr int kScoreThreads = 128;
constexpr int kRowsPerPass = 16;   // window rows staged per pass
constexpr int kPlanThreads = 1024;
constexpr int kNormThreads = 256;
constexpr int kWsHeaderBytes = 256;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ int32_t scan1024(int32_t v, int32_t *sh, int32_t *total) {
  const int tid = threadIdx.x;
  sh[tid] = v;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    const int32_t add = tid >= off ? sh[tid - off] : 0;
    __syncthreads();
    sh[tid] += add;
    __syncthreads();
  }
  const int32_t incl = sh[tid];
  *total = sh[kPlanThreads - 1];
  __syncthreads();
  return incl - v;
}

__global__ void __launch_bounds__(kPlanThreads) imp_plan_kernel(const int32_t *__restrict__ cu, int32_t S,
                                                                int32_t N, const uint8_t *__restrict__ seg_mask,
                                                                int32_t B, int32_t *__restrict__ blk_cu,
                                                                int32_t imp_capacity, int32_t *__restrict__ header,
                                                                int2 *__restrict__ items, int32_t max_items,
                                                                uint32_t *__restrict__ status) {
  __shared__ int32_t s_scan[kPlanThreads];
  __shared__ uint32_t s_err;
  const int tid = threadIdx.x;
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
  int32_t blk_base = scan1024(my_blocks, s_scan, &tot_blocks);
  int32_t item_base = scan1024(my_items, s_scan, &tot_items);
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

template <int D>
__global__ void __launch_bounds__(kScoreThreads) imp_score_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k, const float *__restrict__ lse,
    const int32_t *__restrict__ cu, const int32_t *__restrict__ blk_cu, const int2 *__restrict__ items,
    const int32_t *__restrict__ num_items, int32_t N, int32_t Hq, int32_t Hkv, int32_t B, float scale_log2,
    float *__restrict__ partial) {
  __shared__ float sq[kRowsPerPass][D];
  __shared__ float sl[kRowsPerPass];
  __shared__ float sred[kScoreThreads / 32];
  const int32_t item = blockIdx.x / Hkv;
  if (item >= *num_items) return;
  const int32_t g = blockIdx.x % Hkv;
  const int2 it = items[item];
  const int32_t s = it.x, c = it.y;
  const int32_t c0 = cu[s], n = cu[s + 1] - c0;
  const int32_t W = min(B, n);
  const int32_t group = Hq / Hkv;
  const int tid = threadIdx.x;
  const int32_t j = c * kChunk + tid;  // segment-local key index
  const bool valid = j < n;

  float kf[D];
  if (valid) {
    const uint4 *src = reinterpret_cast<const uint4 *>(k + ((int64_t)(c0 + j) * Hkv + g) * D);
#pragma unroll
    for (int v = 0; v < D / 8; ++v) {
      const uint4 w = src[v];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kf[v * 8 + 2 * e] = __uint_as_float(ws[e] << 16);
        kf[v * 8 + 2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) kf[d] = 0.f;
  }

  float acc = 0.f;
  for (int32_t hh = 0; hh < group; ++hh) {
    const int32_t h = g * group + hh;
    for (int32_t r0 = n - W; r0 < n; r0 += kRowsPerPass) {
      const int32_t nr = min(kRowsPerPass, n - r0);
      __syncthreads();
      for (int e = tid; e < kRowsPerPass * D; e += kScoreThreads) {
        const int r = e / D, d = e % D;
        sq[r][d] = r < nr ? __bfloat162float(q[((int64_t)(c0 + r0 + r) * Hq + h) * D + d]) : 0.f;
      }
      if (tid < kRowsPerPass) sl[tid] = tid < nr ? lse[(int64_t)h * N + c0 + r0 + tid] * kLog2e : 0.f;
      __syncthreads();
      for (int r = 0; r < nr; ++r) {
        float dot = 0.f;
#pragma unroll
        for (int d = 0; d < D; d += 4) {
          const float4 qv = *reinterpret_cast<const float4 *>(&sq[r][d]);
          dot = fmaf(qv.x, kf[d], dot);
          dot = fmaf(qv.y, kf[d + 1], dot);
          dot = fmaf(qv.z, kf[d + 2], dot);
          dot = fmaf(qv.w, kf[d + 3], dot);
        }
        if (valid && j <= r0 + r) acc += ex2_approx(fmaf(dot, scale_log2, -sl[r]));
      }
    }
  }
  // Per-block sums over the chunk's keys (block size divides the chunk).
  const int32_t nb_seg = blk_cu[s + 1] - blk_cu[s];
  const int32_t blocks_per_chunk = kChunk / B;
  if (B <= 32) {
    float v = acc;
    for (int off = B / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((tid % B) == 0) {
      const int32_t b = c * blocks_per_chunk + tid / B;
      if (b < nb_seg) partial[(int64_t)(blk_cu[s] + b) * Hkv + g] = v;
    }
  } else {
    float v = acc;
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((tid & 31) == 0) sred[tid >> 5] = v;
    __syncthreads();
    const int wpb = B / 32;
    if (tid < blocks_per_chunk) {
      float t = 0.f;
      for (int w = 0; w < wpb; ++w) t += sred[tid * wpb + w];
      const int32_t b = c * blocks_per_chunk + tid;
      if (b < nb_seg) partial[(int64_t)(blk_cu[s] + b) * Hkv + g] = t;
    }
  }
}

__global__ void __launch_bounds__(kNormThreads) imp_norm_kernel(const int32_t *__restrict__ blk_cu,
                                                                 const float *__restrict__ partial, int32_t Hkv,
                                                                 float *__restrict__ imp) {
  __shared__ float sred[kNormThreads];
  const int32_t s = blockIdx.x;
  const int32_t b0 = blk_cu[s], nb = blk_cu[s + 1] - b0;
  if (nb <= 0) return;
  const int tid = threadIdx.x;
  float t = 0.f;
  for (int32_t b = tid; b < nb; b += kNormThreads) {
    float m = 0.f;
    for (int32_t g = 0; g < Hkv; ++g) m += partial[(int64_t)(b0 + b) * Hkv + g];
    t += m;
  }
  sred[tid] = t;
  __syncthreads();
  for (int off = kNormThreads / 2; off >= 1; off >>= 1) {
    if (tid < off) sred[tid] += sred[tid + off];
    __syncthreads();
  }
  const float inv = 1.f / sred[0];
  for (int32_t b = tid; b < nb; b += kNormThreads) {
    float m = 0.f;
    for (int32_t g = 0; g < Hkv; ++g) m += partial[(int64_t)(b0 + b) * Hkv + g];
    imp[b0 + b] = m * inv;
  }
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

UNIP_API int32_t unip_block_importance(const void *q, const void *k, const float *lse, const int32_t *cu_seqlens,
                                       int32_t num_segs, int32_t total_tokens, const uint8_t *seg_mask,
                                       int32_t block_size, const unip_attn_params *prm, float *imp,
                                       int32_t imp_capacity, int32_t *blk_cu, void *workspace,
                                       size_t workspace_bytes, void *stream) {
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
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
  const int64_t grid = (int64_t)max_items * Hkv;
  if (grid > 0x7FFFFFFF) return UNIP_ERR_UNSUPPORTED;
  const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(q);
  const __nv_bfloat16 *kb = static_cast<const __nv_bfloat16 *>(k);
  if (D == 128)
    imp_score_kernel<128><<<(int)grid, kScoreThreads, 0, st>>>(qb, kb, lse, cu_seqlens, blk_cu, items, header,
                                                               total_tokens, Hq, Hkv, block_size, scale * kLog2e,
                                                               partial);
  else
    imp_score_kernel<64><<<(int)grid, kScoreThreads, 0, st>>>(qb, kb, lse, cu_seqlens, blk_cu, items, header,
                                                              total_tokens, Hq, Hkv, block_size, scale * kLog2e,
                                                              partial);
  if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;
  imp_norm_kernel<<<num_segs, kNormThreads, 0, st>>>(blk_cu, partial, Hkv, imp);
  if (cudaGetLastError() != cudaSuccess) return UNIP_ERR_CUDA;
  return UNIP_OK;
}

}  // extern "C"
