// Work-unit geometry of the attention kernel, shared by the device code and
// the host planner (both must cut a call into the same units), and the layout
// of a host-built plan passed to the kernel as a parameter.
//
// A unit is (segment s, 128-token pair index m, head selection hsel): one or
// two 128-row query tiles that share every K/V tile of the unit's key range.
// With an even GQA group G dividing 128 (lg = log2 G) a tile's rows are
// (token, head) pairs of the G query heads of one kv head (128 / G tokens);
// otherwise 128 tokens of one query head.  A unit's key range is its P_s
// prefix keys (ceil(P_s / 128) tiles, read through the block table) followed
// by its segment's own keys up to the tile holding its last token.
#pragma once

#include <stdint.h>

namespace unip {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per KV tile

// Rows of one query tile: row R is token tok0 + (R >> lg) (segment-local) and
// query head head0 + (R & (2^lg - 1)); rows at or past rows_valid are not stored.
struct TileRows {
  int32_t tok0, head0, lg, rows_valid;
};

// One work item: a unit, or one KV range of a unit split across items.
struct WorkItem {
  TileRows tr0, tr1;
  int32_t s, c0, P, g;
  int32_t Tp;      // prefix KV tiles of the unit (its key tiles 0 .. Tp - 1 are cached keys)
  int32_t j0, T;   // this item's key tiles: j0 .. j0 + T - 1 of the unit's range
  int32_t split, nsplit, g0;  // KV split `split` of `nsplit` (1: the whole range); g0: first split id
  bool two, valid;
};

__host__ __device__ inline int32_t imin32(int32_t a, int32_t b) { return a < b ? a : b; }
__host__ __device__ inline int32_t imax32(int32_t a, int32_t b) { return a > b ? a : b; }

// Geometry of unit (s, m, hsel) of a segment starting at token c0 with n tokens and a P-token
// cached prefix.  single: one query tile per unit (else two when the group allows).  The item
// covers the unit's whole key range.
__host__ __device__ inline WorkItem unit_geometry(int32_t s, int32_t m, int32_t hsel, int32_t c0, int32_t n,
                                                  int32_t P, int32_t lg, int32_t group, int32_t single) {
  WorkItem w;
  w.s = s;
  w.c0 = c0;
  w.P = P;
  if (lg > 0) {
    const int32_t subs = single ? group : (group >> 1);  // units per kv head for one 128-token pair
    w.g = hsel / subs;
    const int32_t tpt = kBlockM >> lg;
    w.tr0.tok0 = m * kBlockM + (hsel - w.g * subs) * (single ? 1 : 2) * tpt;
    w.tr1.tok0 = w.tr0.tok0 + tpt;
    w.tr0.head0 = w.tr1.head0 = w.g * group;
    w.tr0.lg = w.tr1.lg = lg;
    w.tr0.rows_valid = imin32(kBlockM, imax32(0, n - w.tr0.tok0) << lg);
    w.tr1.rows_valid = imin32(kBlockM, imax32(0, n - w.tr1.tok0) << lg);
    w.two = !single && w.tr1.rows_valid > 0;
  } else {
    w.two = !single && (group & 1) == 0;
    const int32_t h0 = w.two ? 2 * hsel : hsel;
    w.g = h0 / group;
    w.tr0.tok0 = w.tr1.tok0 = m * kBlockM;
    w.tr0.head0 = h0;
    w.tr1.head0 = h0 + 1;
    w.tr0.lg = w.tr1.lg = 0;
    w.tr0.rows_valid = w.tr1.rows_valid = imin32(kBlockM, n - m * kBlockM);
  }
  w.valid = w.tr0.rows_valid > 0;  // else every token of the unit lies past the segment
  const TileRows &trl = w.two ? w.tr1 : w.tr0;  // the tile holding the unit's last token
  const int32_t end_tok = trl.tok0 + (trl.rows_valid >> trl.lg);
  w.Tp = (P + kBlockN - 1) / kBlockN;                       // prefix KV tiles
  w.T = w.valid ? w.Tp + (end_tok - 1) / kBlockN + 1 : 0;    // + own tiles up to the last token's
  w.j0 = 0;
  w.split = 0;
  w.nsplit = 1;
  w.g0 = 0;
  return w;
}

// ---------------------------------------------------------------------------
// Host-built plan (kernel parameter)
// ---------------------------------------------------------------------------
constexpr int kPlanMaxItems = 1024;
constexpr int kPlanMaxSegs = 128;
constexpr int kPlanMaxCtas = 256;

// Item words: w0 = s | hsel << 16; w1 = m | nsplit << 24; w2 = j0 | T << 16; w3 = g0 | split << 24.
struct PlanItem {
  int32_t w0, w1, w2, w3;
};

struct HostPlanArgs {
  int32_t seg[kPlanMaxSegs][3];            // c0, n, P of every segment
  uint16_t cta_first[kPlanMaxCtas + 1];    // CTA b runs items cta_first[b] .. cta_first[b + 1] - 1, in order
  PlanItem items[kPlanMaxItems];
  float *partial;                          // fp32 partial results of split items
  unsigned long long *tickets;             // one per (split unit, tile): generation << 32 | finished splits
  uint32_t gen;                            // this launch's generation (tags the tickets)
};

// Split partials: per (split, tile) slot, per thread of the tile's 256 softmax threads, the D / 2
// accumulator values it holds plus (m0, l0, m1, l1) of its two rows, stored as float4 chunks
// chunk-major (each store of a warp covers 512 contiguous bytes).
template <int D>
struct SplitLayout {
  static constexpr int kChunks = D / 8 + 1;
  static constexpr size_t kSlotBytes = (size_t)kChunks * 256 * 16;
};
inline size_t split_slot_bytes(int32_t D) { return (size_t)(D / 8 + 1) * 256 * 16; }

}  // namespace unip
