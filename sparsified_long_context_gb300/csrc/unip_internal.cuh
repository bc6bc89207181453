// Internal helpers of libunip: status word access, tensor-map creation and
// the inline-PTX wrappers (mbarrier, TMA, tcgen05) the sm_103a kernels use.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "unip.h"

namespace unip {

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Device address of the current device's status word (set up once per device).
uint32_t *device_status_ptr();
// Streaming-multiprocessor count of the current device.
int device_sm_count();
// Raises the dynamic shared-memory limit of kernel `fn` on the current device to at least `bytes`
// (never lowers it); safe to call from several host threads.
cudaError_t ensure_dynamic_smem(const void *fn, int bytes);
// Importance without its normalisation (plan + persistent score grid of unip_block_importance, same
// checks and return codes): block masses per kv head land in the workspace; *partial receives their
// address.  The normalisation follows as a programmatic dependent of the score grid.
int32_t importance_scores(const void *q, const void *k, const float *lse, const int32_t *cu_seqlens,
                          int32_t num_segs, int32_t total_tokens, const uint8_t *seg_mask, int32_t block_size,
                          const unip_attn_params *prm, float *imp, int32_t imp_capacity, int32_t *blk_cu,
                          void *workspace, size_t workspace_bytes, cudaStream_t st, float **partial);
// cuTensorMapEncodeTiled, fetched from the driver at first use.
CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank, void *gaddr,
                      const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                      CUtensorMapSwizzle swizzle);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Limit of every bounded device-side wait (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// mbarrier -------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of an mbarrier.  Returns false (and raises
// *abort and the status bit) when the limit runs out, or false at once when
// another role of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t *status, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, UNIP_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// TMA --------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// Generic-proxy shared-memory writes become visible to the async proxy (tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// tcgen05 -------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem], bf16 x bf16 -> f32, one CTA.
__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t *r = reinterpret_cast<uint32_t *>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  const uint32_t *r = reinterpret_cast<const uint32_t *>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 lanes x 8N columns (16x256b shape): thread t holds, per 8-column chunk k,
// columns 8k + 2(t%4) + {0,1} of lanes t/4 and t/4 + 8, as registers
// 4k + {0,1} (lane t/4) and 4k + {2,3} (lane t/4 + 8).  8 chunks per call.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, float *v) {
  uint32_t *r = reinterpret_cast<uint32_t *>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_16x256b_x8(uint32_t taddr, const float *v) {
  const uint32_t *r = reinterpret_cast<const uint32_t *>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, float *v) {
  uint32_t *r = reinterpret_cast<uint32_t *>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const float *v) {
  const uint32_t *r = reinterpret_cast<const uint32_t *>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 16 lanes x 4N columns (16x128b shape): thread t holds column 4k + t%4 of lanes
// t/4 (register 2k) and t/4 + 8 (register 2k + 1).  16 chunks per call.
__device__ __forceinline__ void tmem_st_16x128b_x16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//   K-major operand: rows of 128 B (64 bf16 along K), 8-row groups 1024 B
//     apart (SBO); a K step of 16 elements advances the start by 32 B.
//   MN-major operand: 128 B along MN per K row, 8 K rows per 1024 B group
//     (SBO = step between K groups), LBO = step between 64-element MN groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1) in one packed instruction.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
// (d0, d1) += (a0, a1) in one packed instruction.
__device__ __forceinline__ void fadd2_acc(float &d0, float &d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rd, {%0, %1};\n\t"
      "add.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

// Two floats -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

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

// Exclusive scan of one value per thread over the CTA (blockDim a multiple of 32, at most 1024);
// *total gets the sum.  sh_warp: 32 elements of shared memory.
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

// 16-byte global load that does not allocate in L1 / streaming store (row copies).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// One warp copies one row of vec_per_row 16-byte vectors, 16 loads in flight per lane.
__device__ __forceinline__ void warp_copy_row(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                              int32_t vec_per_row, int lane) {
  constexpr int kUnroll = 16;  // 16 x 16 B per lane: an 8 KB row in one round trip
  int v = lane;
  for (; v + 32 * (kUnroll - 1) < vec_per_row; v += 32 * kUnroll) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = ld_stream(src + v + 32 * u);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) st_stream(dst + v + 32 * u, r[u]);
  }
  for (; v < vec_per_row; v += 32) st_stream(dst + v, ld_stream(src + v));
}

// M_b = sum over kv heads g = 0, 1, ... of row[g], in that order, with the loads of a group of heads
// issued before its adds (one memory round trip per 8 heads instead of one per head).
__device__ __forceinline__ float block_mass(const float *__restrict__ row, int32_t Hkv) {
  constexpr int kG = 8;
  float m = 0.f;
  for (int32_t g0 = 0; g0 < Hkv; g0 += kG) {
    float v[kG];
#pragma unroll
    for (int u = 0; u < kG; ++u) v[u] = g0 + u < Hkv ? row[g0 + u] : 0.f;
#pragma unroll
    for (int u = 0; u < kG; ++u)
      if (g0 + u < Hkv) m += v[u];
  }
  return m;
}

// Block masses of one scored segment normalised to importance: imp[b] = M_b / sum_b' M_b', with
// M_b = sum over kv heads g of partial[b][g].  Run by the first kImpNormThreads threads of a CTA in a
// fixed order (strided per-thread sums, then a pairwise tree: element i takes element i + off for
// off = 128, 64, ..., 1), so every caller produces the same fp32 bits.  The tree's levels from 128
// down to 32 are summed by warp 0 from registers and the last five by an xor butterfly: both pair
// exactly the elements the in-place tree pairs.  sred: kImpNormThreads floats of shared memory.
// The scores go to imp[b0 + b] and, when sdst is given, also to sdst[b] (shared memory); imp may be
// null.  Threads past kImpNormThreads take no part but must reach the same __syncthreads.
constexpr int kImpNormThreads = 256;
__device__ __forceinline__ void normalise_segment(const float *__restrict__ partial, int32_t b0, int32_t nb,
                                                  int32_t Hkv, float *__restrict__ imp, float *sred,
                                                  float *sdst = nullptr) {
  static_assert(kImpNormThreads == 256, "the register tree below covers 8 warps");
  constexpr int kHeld = 4;  // masses of a thread's first kHeld blocks stay in registers
  const int tid = threadIdx.x;
  const bool part = tid < kImpNormThreads;
  float held[kHeld];
  float t = 0.f;
  if (part) {
#pragma unroll
    for (int k = 0; k < kHeld; ++k) {
      const int32_t b = tid + k * kImpNormThreads;
      held[k] = b < nb ? block_mass(partial + (int64_t)(b0 + b) * Hkv, Hkv) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kHeld; ++k)
      if (tid + k * kImpNormThreads < nb) t += held[k];
    for (int32_t b = tid + kHeld * kImpNormThreads; b < nb; b += kImpNormThreads)
      t += block_mass(partial + (int64_t)(b0 + b) * Hkv, Hkv);
    sred[tid] = t;
  }
  __syncthreads();
  if (tid < 32) {
    float e[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) e[k] = sred[tid + 32 * k];
#pragma unroll
    for (int k = 0; k < 4; ++k) e[k] += e[k + 4];  // off = 128
#pragma unroll
    for (int k = 0; k < 2; ++k) e[k] += e[k + 2];  // off = 64
    float v = e[0] + e[1];                          // off = 32
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncwarp();
    if (tid == 0) sred[0] = v;
  }
  __syncthreads();
  const float inv = 1.f / sred[0];
  if (part) {
#pragma unroll
    for (int k = 0; k < kHeld; ++k) {
      const int32_t b = tid + k * kImpNormThreads;
      if (b < nb) {
        const float f = held[k] * inv;
        if (imp) imp[b0 + b] = f;
        if (sdst) sdst[b] = f;
      }
    }
    for (int32_t b = tid + kHeld * kImpNormThreads; b < nb; b += kImpNormThreads) {
      const float f = block_mass(partial + (int64_t)(b0 + b) * Hkv, Hkv) * inv;
      if (imp) imp[b0 + b] = f;
      if (sdst) sdst[b] = f;
    }
  }
}

// Segment holding token t: largest s with cu[s] <= t (cu non-decreasing, t < cu[S]).
__device__ __forceinline__ int32_t find_segment(const int32_t *cu, int32_t S, int32_t t) {
  int32_t lo = 0, hi = S - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace unip
