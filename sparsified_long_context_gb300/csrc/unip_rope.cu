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
// cache.  A CTA takes 8 tokens at a time: first the (cos, sin) table of those
// tokens goes to shared memory, shared by all heads; then the q rows, the k
// rows and the v rows of the 8 tokens, each a contiguous range of memory, are
// streamed with 16-byte accesses, four units per thread in flight.
//
// Angle accuracy: the frequencies theta^(-2i/D) and the product with the
// position are formed in double precision and reduced to [-pi, pi] with a
// two-part 2*pi (Cody-Waite reduction), after which sincosf of the reduced
// single-precision angle is within ~1e-7 rad of the exact rotation even for
// positions in the millions (frequencies in single precision would be off by
// up to ~1e-2 rad at position 65536).
#include "unip_internal.cuh"

namespace unip {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kRopeTok = 8;       // tokens per CTA iteration
constexpr int kRopeBatch = 4;     // units per thread in flight
constexpr int kRopeMaxHalf = 128; // D <= 256

// 2*pi as a double plus the double nearest to its remainder, and 1/(2*pi).
constexpr double kTwoPiHi = 6.283185307179586;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189535;

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

// Rotates (and/or appends) the rows of H heads of nt tokens starting at
// `rows`; a unit is one 16-byte vector (interleaved) or a pair of vectors
// half a row apart (half layout).  slots is offset to the first token.
template <bool kInter>
__device__ __forceinline__ void rotate_rows(uint4 *rows, int nt, int H, int vr, int half, const float2 *cs,
                                            bool rotate, const int32_t *slots, uint4 *cache, int64_t num_slots,
                                            uint32_t *status) {
  const int ur = kInter ? vr : vr / 2;  // units per head row
  const int n_units = nt * H * ur;
  for (int u0 = threadIdx.x; u0 < n_units; u0 += kRopeThreads * kRopeBatch) {
    uint4 va[kRopeBatch], vb[kRopeBatch];
#pragma unroll
    for (int b = 0; b < kRopeBatch; ++b) {
      const int u = u0 + b * kRopeThreads;
      if (u < n_units) {
        const int row = u / ur, c = u - row * ur;
        const int off = row * vr + c;
        va[b] = ld_v4(rows + off);
        if (!kInter) vb[b] = ld_v4(rows + off + vr / 2);
      }
    }
#pragma unroll
    for (int b = 0; b < kRopeBatch; ++b) {
      const int u = u0 + b * kRopeThreads;
      if (u >= n_units) break;
      const int row = u / ur, c = u - row * ur;
      const int tl = row / H, h = row - tl * H;
      const int off = row * vr + c;
      if (rotate) {
        if (kInter) {
          turn_inter(va[b], cs + tl * half + 4 * c);
        } else {
          turn_half(va[b], vb[b], cs + tl * half + 8 * c);
        }
        st_v4(rows + off, va[b]);
        if (!kInter) st_v4(rows + off + vr / 2, vb[b]);
      }
      if (slots) {
        const int32_t slot = slots[tl];
        if (slot >= 0 && slot < num_slots) {
          uint4 *dst = cache + ((int64_t)slot * H + h) * vr + c;
          st_v4(dst, va[b]);
          if (!kInter) st_v4(dst + vr / 2, vb[b]);
        } else if (slot >= num_slots && h == 0 && c == 0) {
          atomicOr(status, UNIP_DEV_BAD_INDEX);
        }
      }
    }
  }
}

template <bool kInter>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(RopeArgs a) {
  __shared__ double s_inv[kRopeMaxHalf];
  __shared__ float2 s_cs[kRopeTok * kRopeMaxHalf];
  const int half = a.D >> 1;
  const int vr = a.D >> 3;  // 16-byte vectors per head row
  if (a.rotate)
    for (int i = threadIdx.x; i < half; i += kRopeThreads) s_inv[i] = exp2(-(2.0 * i / a.D) * a.log2_theta);
  const int64_t groups = ((int64_t)a.N + kRopeTok - 1) / kRopeTok;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t t0 = g * kRopeTok;
    const int nt = (a.N - t0) < kRopeTok ? (int)(a.N - t0) : kRopeTok;
    __syncthreads();  // s_inv written; the previous group's table no longer read
    if (a.rotate) {
      for (int e = threadIdx.x; e < nt * half; e += kRopeThreads) {
        const int tl = e / half, i = e - tl * half;
        const double ang = (double)a.pos[t0 + tl] * s_inv[i];
        const double turns = rint(ang * kInvTwoPi);
        double r = fma(-turns, kTwoPiHi, ang);
        r = fma(-turns, kTwoPiLo, r);
        float s, c;
        sincosf((float)r, &s, &c);
        s_cs[tl * half + i] = make_float2(c, s);
      }
    }
    __syncthreads();
    const int32_t *slots = a.slots ? a.slots + t0 : nullptr;
    if (a.q && a.rotate)
      rotate_rows<kInter>(a.q + t0 * a.Hq * vr, nt, a.Hq, vr, half, s_cs, true, nullptr, nullptr, 0, a.status);
    rotate_rows<kInter>(a.k + t0 * a.Hkv * vr, nt, a.Hkv, vr, half, s_cs, a.rotate != 0, slots, a.kc,
                        a.num_slots, a.status);
    if (slots) {
      // v rows of the group are contiguous; copy them to their slots.
      const int per_tok = a.Hkv * vr;
      const int n_units = nt * per_tok;
      const uint4 *src = a.v + t0 * per_tok;
      for (int u0 = threadIdx.x; u0 < n_units; u0 += kRopeThreads * kRopeBatch) {
        uint4 r[kRopeBatch];
#pragma unroll
        for (int b = 0; b < kRopeBatch; ++b) {
          const int u = u0 + b * kRopeThreads;
          if (u < n_units) r[b] = ld_v4(src + u);
        }
#pragma unroll
        for (int b = 0; b < kRopeBatch; ++b) {
          const int u = u0 + b * kRopeThreads;
          if (u >= n_units) break;
          const int tl = u / per_tok;
          const int32_t slot = slots[tl];
          if (slot >= 0 && slot < a.num_slots) st_v4(a.vc + (int64_t)slot * per_tok + (u - tl * per_tok), r[b]);
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
  if (!(rope_theta == rope_theta)) return UNIP_ERR_INVALID_ARGUMENT;  // NaN
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
