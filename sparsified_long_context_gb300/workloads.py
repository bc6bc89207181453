"""Seeded synthetic inputs for packed / chunked prefill with block selection.

This module only draws numbers and lays them out; it holds none of the
method's arithmetic (no attention, no scoring, no selection).  Both the CUDA
path (tests, bench) and the CPU oracle's tests take their inputs from here.

Every floating-point input is drawn as float32 and rounded to bfloat16 (round
to nearest, ties to even); arrays hold the bfloat16 bit patterns as uint16.

Workloads (one builder per shape):

* ``tiny_packed``    4 prompts (37, 100, 64, 255) packed into 456 tokens,
  H_q=4, H_kv=2, D=64, 5% heavy keys, block 16, p=0.9, hidden d=256.
* ``chunked``        one 4096-token prompt prefilled in 8 chunks of 512 that
  read earlier chunks through a 16-token paged cache, H_q=32, H_kv=8, D=128.
* ``prepacked``      64 lognormal prompts (median 512, sigma 1, clipped to
  32..8192) packed into 16384-token bins by a packer the caller passes in
  (the library's first-fit-decreasing packer, or the oracle's).
* ``long_single``    one 32768-token prompt, heavy keys in 10 spans, block 64,
  p=0.95, hidden d=4096.
* ``mixed_step``     an 8192-token continuous-batching step: 256 decode tokens
  over paged contexts of 1k..32k plus four 1984-token prefill chunks of
  65536-token prompts; selection applies to the prefill chunks only.

The pages behind these shapes: the "Chunked Prefill" glossary page (token
budget, chunks attending to cached K/V plus themselves, KV pages of fixed
size), the Prepacking summary (prompts of varying length packed with a
bin-packing algorithm, per-prompt mask and restarted positions) and the
UniPrefill review (block-wise importance, Top-p block selection).

Draw order inside one workload: lengths or offsets, heavy-key mask, q, k, v,
cache contents, physical page permutation, hidden states.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

M32 = 0xFFFFFFFF


# ---------------------------------------------------------------------------
# bfloat16 bit helpers (input encoding only)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    # work in slabs to bound temporaries on large arrays
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for a in range(0, flat_u.size, step):
        s = flat_u[a:a + step]
        flat_o[a:a + step] = ((s + np.uint32(0x7FFF) + ((s >> np.uint32(16)) & np.uint32(1)))
                              >> np.uint32(16)).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bits -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, scale_rows: Optional[np.ndarray] = None) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if scale_rows is not None:
        x[scale_rows] *= np.float32(4.0)
    return f32_to_bf16_bits(x)


# ---------------------------------------------------------------------------
# Counter-based generator for very large paged caches.
#
# A paged context of tens of GB is too large to draw on the host, so its
# contents are a pure function of (seed, stream, flat element index), written
# out twice: with numpy on the host and with torch integer ops on a device.
# Both use only exact integer steps plus one correctly rounded float32
# multiply, so they agree bit for bit.  Hash: Wellons' "lowbias32" mixer
# (hash-prospector).  Values: Irwin-Hall sum of eight 16-bit uniforms,
# centred and scaled to unit variance.
# ---------------------------------------------------------------------------
_IH_KAPPA = np.float32(1.0 / (131072.0 * math.sqrt(8.0 / 12.0)))


def _mul32(x, c: int):
    """(x * c) mod 2^32 for x < 2^32 held in a 64-bit integer array, without overflow."""
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & M32


def _mix32(x):
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _hash_normal_f32_bits_numpy(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    idx = idx.astype(np.uint64)
    lo = idx & np.uint64(M32)
    hi = idx >> np.uint64(32)
    key = _mix32(np.uint64((seed * 2 + stream) & M32))
    base = _mix32(lo ^ _mix32(hi ^ key))
    acc = np.zeros(idx.shape, dtype=np.uint64)
    for j in range(1, 5):
        h = _mix32((base + np.uint64((j * 0x9E3779B9) & M32)) & np.uint64(M32))
        acc += (h & np.uint64(0xFFFF)) + (h >> np.uint64(16))
    c = (acc.astype(np.int64) * 2 - 8 * 65535).astype(np.float32)
    return (c * _IH_KAPPA).astype(np.float32)


def hash_normal_bf16_numpy(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    return f32_to_bf16_bits(_hash_normal_f32_bits_numpy(seed, stream, idx))


def hash_normal_bf16_torch(seed: int, stream: int, idx):
    """Same values as :func:`hash_normal_bf16_numpy`, as a torch.bfloat16 tensor on idx's device."""
    import torch
    idx = idx.to(torch.int64)
    lo = idx & M32
    hi = idx >> 32
    key = int(_mix32(np.uint64((seed * 2 + stream) & M32)))
    base = _mix32(lo ^ _mix32(hi ^ key))
    acc = torch.zeros_like(idx)
    for j in range(1, 5):
        h = _mix32((base + ((j * 0x9E3779B9) & M32)) & M32)
        acc += (h & 0xFFFF) + (h >> 16)
    c = (acc * 2 - 8 * 65535).to(torch.float32)
    x = c * torch.tensor(float(_IH_KAPPA), dtype=torch.float32, device=idx.device)
    u = x.view(torch.int32).to(torch.int64) & M32
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF
    r = torch.where(r >= 0x8000, r - 0x10000, r)
    return r.to(torch.int16).view(torch.bfloat16)


# ---------------------------------------------------------------------------
# Paged KV cache description
# ---------------------------------------------------------------------------
@dataclass
class PagedCache:
    """K/V pages laid out [num_pages][page_size][H_kv][D] (bf16 bits).

    ``kind == "array"``: contents held in ``k_pages`` / ``v_pages``.
    ``kind == "hash"``: contents are the counter-based values for ``seed``
    (stream 0 = K, stream 1 = V) at each flat element index.
    """
    num_pages: int
    page_size: int
    num_heads_kv: int
    head_dim: int
    kind: str = "array"
    k_pages: Optional[np.ndarray] = None
    v_pages: Optional[np.ndarray] = None
    seed: int = 0

    @property
    def page_elems(self) -> int:
        return self.page_size * self.num_heads_kv * self.head_dim

    def pages_numpy(self, page_ids: np.ndarray):
        """Return (k, v) uint16 arrays [len(page_ids), page, H_kv, D] for these physical pages."""
        page_ids = np.asarray(page_ids, dtype=np.int64)
        shp = (len(page_ids), self.page_size, self.num_heads_kv, self.head_dim)
        if self.kind == "array":
            return self.k_pages[page_ids], self.v_pages[page_ids]
        e = self.page_elems
        idx = (page_ids[:, None] * e + np.arange(e, dtype=np.int64)[None, :]).reshape(-1)
        k = hash_normal_bf16_numpy(self.seed, 0, idx).reshape(shp)
        v = hash_normal_bf16_numpy(self.seed, 1, idx).reshape(shp)
        return k, v

    def to_torch(self, device, pages_per_slab: int = 2048):
        """Materialise the cache as two torch.bfloat16 tensors on ``device``."""
        import torch
        shp = (self.num_pages, self.page_size, self.num_heads_kv, self.head_dim)
        if self.kind == "array":
            k = torch.from_numpy(self.k_pages).view(torch.bfloat16).to(device)
            v = torch.from_numpy(self.v_pages).view(torch.bfloat16).to(device)
            return k.reshape(shp), v.reshape(shp)
        k = torch.empty(shp, dtype=torch.bfloat16, device=device)
        v = torch.empty(shp, dtype=torch.bfloat16, device=device)
        e = self.page_elems
        for p0 in range(0, self.num_pages, pages_per_slab):
            p1 = min(self.num_pages, p0 + pages_per_slab)
            idx = torch.arange(p0 * e, p1 * e, dtype=torch.int64, device=device)
            k[p0:p1] = hash_normal_bf16_torch(self.seed, 0, idx).reshape(p1 - p0, *shp[1:])
            v[p0:p1] = hash_normal_bf16_torch(self.seed, 1, idx).reshape(p1 - p0, *shp[1:])
        return k, v


# ---------------------------------------------------------------------------
# Workload container
# ---------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    cu_seqlens: np.ndarray            # int32 [S+1]
    positions: np.ndarray             # int32 [N]
    q: np.ndarray                     # uint16 [N, H_q, D]
    k: np.ndarray                     # uint16 [N, H_kv, D]
    v: np.ndarray                     # uint16 [N, H_kv, D]
    cache: Optional[PagedCache] = None
    block_table: Optional[np.ndarray] = None   # int32 [S, max_pages]
    block_size: Optional[int] = None
    top_p: Optional[float] = None
    seg_mask: Optional[np.ndarray] = None      # uint8 [S], 1 = score and select this segment
    hidden: Optional[np.ndarray] = None        # uint16 [N, d_model]
    meta: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_segs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def seq_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens).astype(np.int64)

    @property
    def prefix_lens(self) -> np.ndarray:
        """Cached-prefix length of each segment: the position of its first token."""
        cu = self.cu_seqlens
        out = np.zeros(self.num_segs, dtype=np.int64)
        for s in range(self.num_segs):
            if cu[s + 1] > cu[s]:
                out[s] = self.positions[cu[s]]
        return out


def _positions_for(lengths, prefixes) -> np.ndarray:
    parts = [np.arange(p, p + n, dtype=np.int32) for n, p in zip(lengths, prefixes)]
    return np.concatenate(parts) if parts else np.zeros(0, np.int32)


def _cu(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def _heavy_rows(rng, n_tokens: int, frac: float = 0.05) -> np.ndarray:
    n_heavy = int(round(frac * n_tokens))
    return np.sort(rng.choice(n_tokens, n_heavy, replace=False))


# ---------------------------------------------------------------------------
# Builders
# ---------------------------------------------------------------------------
def packed(lengths, num_heads_q: int, num_heads_kv: int, head_dim: int, seed: int,
           heavy_frac: float = 0.05, block_size: Optional[int] = None, top_p: Optional[float] = None,
           d_model: Optional[int] = None, name: str = "packed") -> Workload:
    """Prompts packed back to back with restarted positions and no cached prefix."""
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in lengths]
    n = sum(lengths)
    heavy = _heavy_rows(rng, n, heavy_frac) if heavy_frac > 0 else None
    q = _normal_bf16(rng, (n, num_heads_q, head_dim))
    k = _normal_bf16(rng, (n, num_heads_kv, head_dim), heavy)
    v = _normal_bf16(rng, (n, num_heads_kv, head_dim))
    hidden = _normal_bf16(rng, (n, d_model)) if d_model else None
    return Workload(name, num_heads_q, num_heads_kv, head_dim, _cu(lengths),
                    _positions_for(lengths, [0] * len(lengths)), q, k, v,
                    block_size=block_size, top_p=top_p,
                    seg_mask=np.ones(len(lengths), np.uint8), hidden=hidden,
                    meta={"lengths": lengths, "heavy_rows": heavy})


def tiny_packed(seed: int = 1) -> Workload:
    return packed([37, 100, 64, 255], 4, 2, 64, seed, 0.05, block_size=16, top_p=0.9,
                  d_model=256, name="tiny_packed")


def prepacked(pack, seed: int = 3, num_prompts: int = 64, bin_tokens: int = 16384,
              num_heads_q: int = 32, num_heads_kv: int = 8, head_dim: int = 128) -> Workload:
    """64 lognormal prompts packed into ``bin_tokens``-token bins.

    The packing itself is method arithmetic, so it is not done here: ``pack``
    is the packer under use, called as ``pack(lengths, bin_tokens)`` and
    returning ``(order, bin_cu)`` (the prompts in packed order and the bin
    boundaries in that order), e.g. the library's ``unip_ffd_pack`` or an
    adapter over the oracle's.  Prompt contents are drawn per prompt, in
    prompt order, and then laid out in the packed order, so every packer that
    returns the same order yields the same stream.
    """
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(num_prompts)
    lengths = np.clip(np.round(np.exp(math.log(512.0) + 1.0 * z)), 32, 8192).astype(np.int64)
    n = int(lengths.sum())
    heavy = _heavy_rows(rng, n, 0.05)   # rows of the prompt-order concatenation
    q = _normal_bf16(rng, (n, num_heads_q, head_dim))
    k = _normal_bf16(rng, (n, num_heads_kv, head_dim), heavy)
    v = _normal_bf16(rng, (n, num_heads_kv, head_dim))
    order, bin_cu = pack([int(x) for x in lengths], bin_tokens)
    order = [int(i) for i in order]
    bin_cu = [int(x) for x in bin_cu]
    if sorted(order) != list(range(num_prompts)):
        raise ValueError("the packer must place every prompt exactly once")
    starts = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    rows = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in order])
    packed_lengths = [int(lengths[i]) for i in order]
    bins = [order[bin_cu[b]:bin_cu[b + 1]] for b in range(len(bin_cu) - 1)]
    inv = np.empty(n, np.int64)
    inv[rows] = np.arange(n)
    return Workload("prepacked", num_heads_q, num_heads_kv, head_dim, _cu(packed_lengths),
                    _positions_for(packed_lengths, [0] * num_prompts), q[rows], k[rows], v[rows],
                    block_size=64, top_p=0.95,  # selection settings of the long-context layer
                    seg_mask=np.ones(num_prompts, np.uint8),
                    meta={"lengths": packed_lengths, "prompt_order": order, "bins": bins,
                          "bin_tokens": bin_tokens, "heavy_rows": np.sort(inv[heavy])})


def long_single(seed: int = 4, n: int = 32768, num_heads_q: int = 32, num_heads_kv: int = 8,
                head_dim: int = 128, num_spans: int = 10, heavy_frac: float = 0.05,
                block_size: int = 64, top_p: float = 0.95, d_model: int = 4096) -> Workload:
    rng = np.random.default_rng(seed)
    n_heavy = int(round(heavy_frac * n))
    span_len = [n_heavy // num_spans + (1 if i < n_heavy % num_spans else 0) for i in range(num_spans)]
    gaps = np.sort(rng.choice(n - n_heavy + 1, num_spans, replace=False))
    starts = [int(gaps[i]) + sum(span_len[:i]) for i in range(num_spans)]
    heavy = np.concatenate([np.arange(s, s + l) for s, l in zip(starts, span_len)])
    q = _normal_bf16(rng, (n, num_heads_q, head_dim))
    k = _normal_bf16(rng, (n, num_heads_kv, head_dim), heavy)
    v = _normal_bf16(rng, (n, num_heads_kv, head_dim))
    hidden = _normal_bf16(rng, (n, d_model)) if d_model else None
    return Workload("long_single", num_heads_q, num_heads_kv, head_dim, _cu([n]),
                    np.arange(n, dtype=np.int32), q, k, v, block_size=block_size, top_p=top_p,
                    seg_mask=np.ones(1, np.uint8), hidden=hidden,
                    meta={"heavy_rows": heavy, "span_starts": starts, "span_lens": span_len})


def _paged_from_tokens(k: np.ndarray, v: np.ndarray, page_size: int, perm: np.ndarray):
    """Scatter one prompt's K/V into pages; logical page p lives in physical page perm[p]."""
    n, hkv, d = k.shape
    n_pages = len(perm)
    kp = np.zeros((n_pages, page_size, hkv, d), np.uint16)
    vp = np.zeros((n_pages, page_size, hkv, d), np.uint16)
    for p in range(n_pages):
        a, b = p * page_size, min(n, (p + 1) * page_size)
        kp[perm[p], : b - a] = k[a:b]
        vp[perm[p], : b - a] = v[a:b]
    return kp, vp


def chunked(seed: int = 2, prompt_len: int = 4096, chunk: int = 512, page_size: int = 16,
            num_heads_q: int = 32, num_heads_kv: int = 8, head_dim: int = 128):
    """One prompt, its one-shot workload and its chunk-by-chunk workloads.

    Returns (one_shot, chunks): chunk c holds tokens [c*chunk, (c+1)*chunk), positions
    starting at c*chunk, and reads tokens before it from a shared paged cache whose
    physical pages are a random permutation of the logical ones.
    """
    rng = np.random.default_rng(seed)
    q = _normal_bf16(rng, (prompt_len, num_heads_q, head_dim))
    k = _normal_bf16(rng, (prompt_len, num_heads_kv, head_dim))
    v = _normal_bf16(rng, (prompt_len, num_heads_kv, head_dim))
    n_pages = -(-prompt_len // page_size)
    perm = rng.permutation(n_pages).astype(np.int32)
    kp, vp = _paged_from_tokens(k, v, page_size, perm)
    cache = PagedCache(n_pages, page_size, num_heads_kv, head_dim, "array", kp, vp)
    one = Workload("chunked_one_shot", num_heads_q, num_heads_kv, head_dim, _cu([prompt_len]),
                   np.arange(prompt_len, dtype=np.int32), q, k, v, meta={"perm": perm})
    chunks = []
    for start in range(0, prompt_len, chunk):
        end = min(start + chunk, prompt_len)
        bt = perm[None, :].copy()
        chunks.append(Workload(f"chunk_{start}", num_heads_q, num_heads_kv, head_dim, _cu([end - start]),
                               np.arange(start, end, dtype=np.int32), q[start:end], k[start:end],
                               v[start:end], cache=cache, block_table=bt,
                               meta={"start": start, "end": end}))
    return one, chunks


def mixed_step(seed: int = 5, budget: int = 8192, num_decode: int = 256, num_prefill: int = 4,
               prompt_len: int = 65536, ctx_lo: int = 1024, ctx_hi: int = 32768, page_size: int = 16,
               num_heads_q: int = 32, num_heads_kv: int = 8, head_dim: int = 128,
               block_size: int = 64, top_p: float = 0.95, d_model: int = 4096,
               offset_align: int = 64) -> Workload:
    """A continuous-batching step: decode tokens first, then prefill chunks fill the budget."""
    rng = np.random.default_rng(seed)
    chunk = (budget - num_decode) // num_prefill
    ctx = rng.integers(ctx_lo, ctx_hi + 1, num_decode).astype(np.int64)
    max_off = (prompt_len - chunk) // offset_align * offset_align
    offs = (rng.integers(0, max_off // offset_align + 1, num_prefill) * offset_align).astype(np.int64)
    lengths = [1] * num_decode + [chunk] * num_prefill
    prefixes = [int(c) for c in ctx] + [int(o) for o in offs]
    n = sum(lengths)
    q = _normal_bf16(rng, (n, num_heads_q, head_dim))
    k = _normal_bf16(rng, (n, num_heads_kv, head_dim))
    v = _normal_bf16(rng, (n, num_heads_kv, head_dim))
    cache_seed = int(rng.integers(0, 2**31 - 1))
    pages_per_seg = [-(-p // page_size) for p in prefixes]
    total_pages = int(sum(pages_per_seg))
    perm = rng.permutation(total_pages).astype(np.int32)
    max_pages = max(max(pages_per_seg), 1)
    bt = np.full((len(lengths), max_pages), -1, np.int32)
    off = 0
    for s, np_s in enumerate(pages_per_seg):
        bt[s, :np_s] = perm[off:off + np_s]
        off += np_s
    hidden = _normal_bf16(rng, (n, d_model)) if d_model else None
    cache = PagedCache(total_pages, page_size, num_heads_kv, head_dim, "hash", seed=cache_seed)
    seg_mask = np.array([0] * num_decode + [1] * num_prefill, np.uint8)
    return Workload("mixed_step", num_heads_q, num_heads_kv, head_dim, _cu(lengths),
                    _positions_for(lengths, prefixes), q, k, v, cache=cache, block_table=bt,
                    block_size=block_size, top_p=top_p, seg_mask=seg_mask, hidden=hidden,
                    meta={"decode_ctx": ctx, "chunk_offsets": offs, "chunk": chunk})


def workload_by_name(name: str, **kw):
    table = {"tiny_packed": tiny_packed, "prepacked": prepacked, "long_single": long_single,
             "mixed_step": mixed_step, "chunked": chunked}
    return table[name](**kw)
