// Host plumbing shared by every entry point: per-device status word,
// SM count, driver entry point for tensor maps, version and error strings.
#include <map>
#include <mutex>
#include <utility>

#include "unip_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

// One status word per device; kernels OR error bits into it.
__device__ uint32_t g_status_word;

std::mutex g_mu;
uint32_t *g_status_ptr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

}  // namespace

namespace unip {

uint32_t *device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<uint32_t *>(p);
  }
  return g_status_ptr[dev];
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

cudaError_t ensure_dynamic_smem(const void *fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // The attribute is one value per kernel and device: it is only ever raised, so that a launch that
  // needs less shared memory never lowers the limit a larger launch relies on.
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, int> limit;
  const auto key = std::make_pair(fn, dev);
  std::lock_guard<std::mutex> lk(mu);
  const auto it = limit.find(key);
  if (it != limit.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) limit[key] = bytes;
  return e;
}

CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank, void *gaddr,
                      const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                      CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return CUDA_ERROR_NOT_FOUND;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return g_encode(map, dtype, rank, gaddr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace unip

extern "C" {

UNIP_API const char *unip_version(void) { return "unip 0.1.0 (sm_103a)"; }

UNIP_API const char *unip_status_string(int32_t code) {
  switch (code) {
    case UNIP_OK: return "ok";
    case UNIP_ERR_INVALID_ARGUMENT: return "invalid argument";
    case UNIP_ERR_UNSUPPORTED: return "unsupported shape";
    case UNIP_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case UNIP_ERR_CUDA: return "CUDA runtime or launch failure";
    case UNIP_ERR_ALIGNMENT: return "pointer or row stride not 16-byte aligned";
    case UNIP_ERR_TOO_LARGE: return "problem too large (no-allocation scratch, page budget, int32 sizes or host memory)";
    default: return "unknown status";
  }
}

UNIP_API const char *unip_last_cuda_error(void) { return cudaGetErrorString(cudaGetLastError()); }

UNIP_API int32_t unip_get_device_status(uint32_t *bits, int32_t clear) {
  if (!bits) return UNIP_ERR_INVALID_ARGUMENT;
  uint32_t *p = unip::device_status_ptr();
  if (!p) return UNIP_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return UNIP_ERR_CUDA;
  if (cudaMemcpy(bits, p, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return UNIP_ERR_CUDA;
  if (clear && cudaMemset(p, 0, sizeof(uint32_t)) != cudaSuccess) return UNIP_ERR_CUDA;
  if (clear && cudaDeviceSynchronize() != cudaSuccess) return UNIP_ERR_CUDA;
  return UNIP_OK;
}

}  // extern "C"
