// Compaction of the kept tokens' hidden-state rows.
//
// Source: "[논문리뷰] UniPrefill ..." review, section 3 -- tokens dropped by the
// selection are excluded from every later sub-layer, so the later layers run
// on the compacted stream out[i] = hidden[gather_idx[i]].
//
// HBM-bound row copy: one warp per row, 16-byte vector loads with a
// streaming (no L1 allocation) hint, 8 independent loads in flight per lane
// before the stores, and a grid sized to a multiple of the SM count that
// strides over the rows.  The number of rows is read on the device, so the
// call never waits for the selection's result on the host.
#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const uint4 *__restrict__ hidden,
                                                                     int32_t num_rows, int64_t stride16,
                                                                     int32_t vec_per_row,
                                                                     const int32_t *__restrict__ gather_idx,
                                                                     const int32_t *__restrict__ n_kept_ptr,
                                                                     int32_t capacity, uint4 *__restrict__ out,
                                                                     int64_t out_stride16, uint32_t *status) {
  int32_t n = *n_kept_ptr;
  if (n > capacity || n < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, UNIP_DEV_BAD_INDEX);
    n = n < 0 ? 0 : capacity;
  }
  const int lane = threadIdx.x & 31;
  const int warps_per_block = kGatherThreads / 32;
  const int64_t nwarps = (int64_t)gridDim.x * warps_per_block;
  for (int64_t row = (int64_t)blockIdx.x * warps_per_block + (threadIdx.x >> 5); row < n; row += nwarps) {
    const int32_t src = gather_idx[row];
    if (src < 0 || src >= num_rows) {
      if (lane == 0) atomicOr(status, UNIP_DEV_BAD_INDEX);
      continue;
    }
    warp_copy_row(hidden + (int64_t)src * stride16, out + row * out_stride16, vec_per_row, lane);
  }
}

}  // namespace
}  // namespace unip

using namespace unip;

extern "C" {

UNIP_API int32_t unip_gather_tokens(const void *hidden, int32_t num_rows, int64_t row_stride, int32_t d_model,
                                    const int32_t *gather_idx, const int32_t *n_kept, int32_t capacity, void *out,
                                    int64_t out_row_stride, void *stream) {
  if (num_rows < 0 || d_model < 0 || capacity < 0 || !n_kept) return UNIP_ERR_INVALID_ARGUMENT;
  if (capacity == 0 || d_model == 0) return UNIP_OK;
  if (!hidden || !gather_idx || !out) return UNIP_ERR_INVALID_ARGUMENT;
  if (row_stride < d_model || out_row_stride < d_model) return UNIP_ERR_INVALID_ARGUMENT;
  if (!aligned16(hidden) || !aligned16(out) || (d_model % 8) || (row_stride % 8) || (out_row_stride % 8))
    return UNIP_ERR_ALIGNMENT;
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  const int sms = device_sm_count();
  const int warps_per_block = kGatherThreads / 32;
  int64_t blocks = ((int64_t)capacity + warps_per_block - 1) / warps_per_block;
  const int64_t max_blocks = (int64_t)(sms > 0 ? sms : 1) * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  gather_rows_kernel<<<(int)blocks, kGatherThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(hidden), num_rows, row_stride / 8, d_model / 8, gather_idx, n_kept, capacity,
      static_cast<uint4 *>(out), out_row_stride / 8, status);
  return cudaGetLastError() == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
}

}  // extern "C"
