// Rotary position embedding of q and k by each token's own position, fused
// with the append of the rotated k and of v into the paged KV cache.
//
// Sources:
//   "Prepacking: A Simple Method for Fast Prefilling and Increased Throughput
//   in Large Language Models" summary, sections "技术框架" and "关键设计": a
//   packed sequence changes its positional encoding so that every prompt
//   restarts at position 0.  The encoding is taken to be the rotary embedding
//   (RoFormer): channel pair i of a head of width D turns by the angle
//   position * theta^(-2i/D); pairs are channels (i, i + D/2) in the "half"
//   layout and (2i, 2i + 1) in the interleaved one.
//   "Chunked Prefill" (Ultralytics glossary), section "Como funciona o
//   pre-preenchimento segmentado": a chunk's K/V join the cache that later
//   chunks attend to; section "Tecnicas de servico relacionadas": the cache is
//   paged.  Token i's rows go to cache slot slot_mapping[i] = page * page_size
//   + offset.
//
// HBM-bound, one pass: every q and k element is read once and written once in
// place, and the rotated k and the v rows are written once more into the
// cache.  A CTA takes 16 tokens at a time: first the (cos, sin) table of those
// tokens goes to shared memory, shared by all heads; then one flat loop runs
// over the 16-byte units of the q rows, the k rows and the v rows of the 16
// tokens (each a contiguous range of memory), four units per thread in
// flight, so the three streams overlap.
//
// Angle: each frequency theta^(-2i/D) is turned, once per CTA, into the turns
// it makes per position, a fraction F_i of a full turn held as a 64-bit
// fixed-point number.  A token's angle is then position * F_i modulo one
// turn, which 64-bit integer multiplication gives exactly (the wrap-around is
// the modulo), so the range reduction costs no floating point; the top 32
// bits become a single-precision argument of sincospif.  The only errors are
// F_i's double-precision rounding (below 3e-16 relative, ~6e-7 rad at
// position 2^31, ~1e-9 rad at 2^22) and the 24-bit argument (2e-7 rad).
#include <cmath>

#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kRopeTok = 16;      // tokens per CTA iteration
constexpr int kRopeBatch = 4;     // units per thread in flight
constexpr int kRopeMaxHalf = 128; // D <= 256

// 2*pi rounded to double.
constexpr double kTwoPi = 6.283185307179586;

struct RopeArgs {
  uint4 *q;                 // [N][Hq][D] bf16, rotated in place (may be null)
  uint4 *k;                 // [N][Hkv][D] bf16, rotated in place
  const uint4 *v;           // [N][Hkv][D] bf16 (read only when appending)
  const int32_t *pos;       // [N]
  const int32_t *slots;     // [N] or null (no append)
  uint4 *kc;                // [num_slots][Hkv][D]
  uint4 *vc;
  int64_t num_slots;
  int32_t N, Hq, Hkv, D;
  double log2_theta;
  int rotate;
  uint32_t *status;
};

// Plain 16-byte global accesses; the load does not allocate in L1 (every
// element is touched once).
__device__ __forceinline__ uint4 ld_v4(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_v4(uint4 *p, const uint4 &v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One word of a and one of b (two pairs each) turned by (c, s) of two frequencies.
__device__ __forceinline__ void turn2(uint32_t &wa, uint32_t &wb, float2 cs0, float2 cs1) {
  const float a0 = bf_lo(wa), a1 = bf_hi(wa), b0 = bf_lo(wb), b1 = bf_hi(wb);
  wa = pack_bf16x2(a0 * cs0.x - b0 * cs0.y, a1 * cs1.x - b1 * cs1.y);
  wb = pack_bf16x2(b0 * cs0.x + a0 * cs0.y, b1 * cs1.x + a1 * cs1.y);
}
// Half layout: va holds channels i..i+7 of the first half, vb the matching
// channels of the second half; cs points at frequency i.
__device__ __forceinline__ void turn_half(uint4 &va, uint4 &vb, const float2 *cs) {
  turn2(va.x, vb.x, cs[0], cs[1]);
  turn2(va.y, vb.y, cs[2], cs[3]);
  turn2(va.z, vb.z, cs[4], cs[5]);
  turn2(va.w, vb.w, cs[6], cs[7]);
}
// Interleaved layout: v holds pairs (2i, 2i+1) .. (2i+6, 2i+7); cs points at frequency i.
__device__ __forceinline__ uint32_t turn_pair(uint32_t w, float2 cs) {
  const float a = bf_lo(w), b = bf_hi(w);
  return pack_bf16x2(a * cs.x - b * cs.y, b * cs.x + a * cs.y);
}
__device__ __forceinline__ void turn_inter(uint4 &v, const float2 *cs) {
  v.x = turn_pair(v.x, cs[0]);
  v.y = turn_pair(v.y, cs[1]);
  v.z = turn_pair(v.z, cs[2]);
  v.w = turn_pair(v.w, cs[3]);
}

template <bool kInter>
__global__ void __launch_bounds__(kRopeThreads, 3) rope_append_kernel(RopeArgs a) {
  __shared__ uint64_t s_turn[kRopeMaxHalf];          // F_i: turns per position, 64-bit fraction
  __shared__ float2 s_cs[kRopeTok * kRopeMaxHalf];   // (cos, sin) per token and frequency
  const int half = a.D >> 1;
  const int vr = a.D >> 3;                 // 16-byte vectors per head row
  const int ur = kInter ? vr : vr >> 1;    // rotation units per head row
  if (a.rotate)
    for (int i = threadIdx.x; i < half; i += kRopeThreads) {
      double turns = exp2(-(2.0 * i / a.D) * a.log2_theta) / kTwoPi;   // < 1/(2 pi) when theta >= 1
      turns = fmod(turns, 1.0);                                         // whole turns do not matter
      s_turn[i] = (uint64_t)(turns * 18446744073709551616.0);          // * 2^64
    }
  const int per_q = a.Hq * ur, per_k = a.Hkv * ur, per_v = a.Hkv * vr;
  const int64_t groups = ((int64_t)a.N + kRopeTok - 1) / kRopeTok;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t t0 = g * kRopeTok;
    const int nt = (a.N - t0) < kRopeTok ? (int)(a.N - t0) : kRopeTok;
    __syncthreads();  // s_turn written; the previous group's table no longer read
    if (a.rotate) {
      for (int e = threadIdx.x; e < nt * half; e += kRopeThreads) {
        const int tl = e / half, i = e - tl * half;
        const uint64_t frac = (uint64_t)(int64_t)a.pos[t0 + tl] * s_turn[i];  // mod 2^64 = mod one turn
        float sn, cs;
        sincospif((float)(int32_t)(frac >> 32) * 0x1p-31f, &sn, &cs);         // half-turns in [-1, 1)
        s_cs[tl * half + i] = make_float2(cs, sn);
      }
    }
    __syncthreads();
    const int n_q = (a.q && a.rotate) ? nt * per_q : 0;
    const int n_qk = n_q + nt * per_k;
    const int total = n_qk + (a.slots ? nt * per_v : 0);
    uint4 *qg = a.q ? a.q + t0 * a.Hq * vr : nullptr;
    uint4 *kg = a.k + t0 * a.Hkv * vr;
    const uint4 *vg = a.slots ? a.v + t0 * per_v : nullptr;
    const int32_t *slots = a.slots ? a.slots + t0 : nullptr;
    for (int u0 = threadIdx.x; u0 < total; u0 += kRopeThreads * kRopeBatch) {
      uint4 va[kRopeBatch], vb[kRopeBatch];
#pragma unroll
      for (int b = 0; b < kRopeBatch; ++b) {
        const int u = u0 + b * kRopeThreads;
        if (u < n_qk) {
          const bool is_q = u < n_q;
          const int w = is_q ? u : u - n_q;
          const int row = w / ur, c = w - row * ur;
          const uint4 *p = (is_q ? qg : kg) + row * vr + c;
          va[b] = ld_v4(p);
          if (!kInter) vb[b] = ld_v4(p + (vr >> 1));
        } else if (u < total) {
          va[b] = ld_v4(vg + (u - n_qk));
        }
      }
#pragma unroll
      for (int b = 0; b < kRopeBatch; ++b) {
        const int u = u0 + b * kRopeThreads;
        if (u >= total) break;
        if (u < n_qk) {
          const bool is_q = u < n_q;
          const int w = is_q ? u : u - n_q;
          const int H = is_q ? a.Hq : a.Hkv;
          const int row = w / ur, c = w - row * ur;
          const int tl = row / H, h = row - tl * H;
          uint4 *p = (is_q ? qg : kg) + row * vr + c;
          if (a.rotate) {
            if (kInter) {
              turn_inter(va[b], s_cs + tl * half + 4 * c);
            } else {
              turn_half(va[b], vb[b], s_cs + tl * half + 8 * c);
            }
            st_v4(p, va[b]);
            if (!kInter) st_v4(p + (vr >> 1), vb[b]);
          }
          if (!is_q && slots) {
            const int32_t slot = slots[tl];
            if (slot >= 0 && slot < a.num_slots) {
              uint4 *dst = a.kc + ((int64_t)slot * a.Hkv + h) * vr + c;
              st_v4(dst, va[b]);
              if (!kInter) st_v4(dst + (vr >> 1), vb[b]);
            } else if (slot >= a.num_slots && h == 0 && c == 0) {
              atomicOr(a.status, UNIP_DEV_BAD_INDEX);
            }
          }
        } else {
          const int w = u - n_qk;
          const int tl = w / per_v;
          const int32_t slot = slots[tl];
          if (slot >= 0 && slot < a.num_slots) st_v4(a.vc + (int64_t)slot * per_v + (w - tl * per_v), va[b]);
        }
      }
    }
  }
}

}  // namespace
}  // namespace unip

using namespace unip;

extern "C" {

UNIP_API int32_t unip_rope_append_kv(void *q, void *k, const void *v, const int32_t *positions, int32_t num_tokens,
                                     const unip_attn_params *prm, double rope_theta, int32_t interleaved,
                                     const int32_t *slot_mapping, void *k_cache, void *v_cache, int32_t num_pages,
                                     int32_t page_size, void *stream) {
  if (!prm || num_tokens < 0 || (interleaved != 0 && interleaved != 1)) return UNIP_ERR_INVALID_ARGUMENT;
  const int32_t hq = prm->num_heads_q, hkv = prm->num_heads_kv, d = prm->head_dim;
  if (hq < 1 || hkv < 1) return UNIP_ERR_INVALID_ARGUMENT;
  if (d < 16 || d > 2 * kRopeMaxHalf || d % 16) return UNIP_ERR_UNSUPPORTED;
  const bool rotate = rope_theta > 0.0;
  const bool append = slot_mapping != nullptr;
  if (!std::isfinite(rope_theta)) return UNIP_ERR_INVALID_ARGUMENT;  // NaN or infinite base
  if (num_tokens == 0 || (!rotate && !append)) return UNIP_OK;
  if (!k || (rotate && !positions)) return UNIP_ERR_INVALID_ARGUMENT;
  if (append && (!v || !k_cache || !v_cache || num_pages < 0 || page_size <= 0)) return UNIP_ERR_INVALID_ARGUMENT;
  if ((q && !aligned16(q)) || !aligned16(k) || (append && (!aligned16(v) || !aligned16(k_cache) ||
                                                          !aligned16(v_cache))))
    return UNIP_ERR_ALIGNMENT;
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  RopeArgs a;
  a.q = static_cast<uint4 *>(q);
  a.k = static_cast<uint4 *>(k);
  a.v = static_cast<const uint4 *>(v);
  a.pos = positions;
  a.slots = slot_mapping;
  a.kc = static_cast<uint4 *>(k_cache);
  a.vc = static_cast<uint4 *>(v_cache);
  a.num_slots = append ? (int64_t)num_pages * page_size : 0;
  a.N = num_tokens;
  a.Hq = hq;
  a.Hkv = hkv;
  a.D = d;
  a.log2_theta = rotate ? log2(rope_theta) : 0.0;
  a.rotate = rotate ? 1 : 0;
  a.status = status;
  const int sms = device_sm_count();
  const int64_t groups = ((int64_t)num_tokens + kRopeTok - 1) / kRopeTok;
  const int64_t max_blocks = (int64_t)(sms > 0 ? sms : 1) * 8;
  const int blocks = (int)(groups < max_blocks ? groups : max_blocks);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (interleaved)
    rope_append_kernel<true><<<blocks, kRopeThreads, 0, st>>>(a);
  else
    rope_append_kernel<false><<<blocks, kRopeThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
}

}  // extern "C"
