"""fp64 oracle of the rotary position embedding and the paged-cache append --
TEST INFRASTRUCTURE (only the test suite may import it).

The Prepacking summary ("Prepacking: A Simple Method for Fast Prefilling and
Increased Throughput in Large Language Models", sections "技术框架" and
"关键设计") changes the positional encoding of a packed sequence so that every
prompt is encoded as if alone: positions restart at 0 per prompt.  The pages
do not spell out the encoding itself; the reading taken is the rotary
embedding as published with RoFormer: channel pair i of a head of width D is
turned by the angle  position * theta^(-2i/D),

    (a, b)  ->  (a cos w - b sin w,  b cos w + a sin w).

Which channels form pair i is a layout choice of the model:
  * "half" layout: channels i and i + D/2;
  * "interleaved" layout: channels 2i and 2i + 1.

Everything here is double precision on the bf16 input values; the result is
returned unrounded.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def inv_frequencies(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2i/D) for i = 0 .. D/2-1."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope(x: np.ndarray, positions: np.ndarray, theta: float, interleaved: bool = False) -> np.ndarray:
    """Rotate x [N, H, D] (float64 values) by each token's position; returns float64."""
    x = np.asarray(x, np.float64)
    n, h, d = x.shape
    ang = np.asarray(positions, np.float64)[:, None] * inv_frequencies(d, theta)[None, :]   # [N, D/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if interleaved:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        a, b = x[..., : d // 2], x[..., d // 2:]
    ra = a * c - b * s
    rb = b * c + a * s
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : d // 2], out[..., d // 2:] = ra, rb
    return out


def append_to_cache(k_cache: np.ndarray, v_cache: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray,
                    slot_mapping: np.ndarray) -> None:
    """Write token i's rows at cache slot slot_mapping[i] (page * page_size + offset)
    of caches shaped [num_pages, page_size, H_kv, D]; negative slots are skipped."""
    num_pages, page_size = k_cache.shape[:2]
    for i, s in enumerate(np.asarray(slot_mapping)):
        if s < 0:
            continue
        k_cache[s // page_size, s % page_size] = k_rows[i]
        v_cache[s // page_size, s % page_size] = v_rows[i]
