"""fp64 CPU oracle for the packed / chunked prefill path -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never calls it and shares no code with it.

The numerics live in ``unip_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use (or via :func:`build`) and marshals
numpy arrays through ctypes.

Pins: every function here is checked by the ``-m "not gpu"`` tests against
values fixed by the pages or by mathematics (library SDPA in fp64, closed
forms, brute force, the chunked-prefill demo printed on the "Chunked Prefill"
page).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "unip_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()

KEEP_FIRST = 1
KEEP_LAST = 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64, u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_uint32
            lib.oracle_attention.argtypes = [P, P, P, P, i32, P, i32, P, P, i32, i32, P, i32,
                                             i32, i32, i32, f64, P, i32, P, P, i32]
            lib.oracle_block_importance.argtypes = [P, P, P, P, i32, i32, P, i32, i32, i32, i32, f64,
                                                    P, i64, P, i32]
            lib.oracle_topp_select.argtypes = [P, P, i32, f64, u32, P]
            lib.oracle_index_build.argtypes = [P, P, P, P, i32, i32, P, P, P, P]
            lib.oracle_gather.argtypes = [P, i64, i32, P, i32, i32, P]
            lib.oracle_attention_compacted.argtypes = [P, P, P, P, i32, P, P, i32, P, P, i32, i32, P, i32,
                                                       i32, i32, i32, f64, P, i32, P, P, i32]
            for f in (lib.oracle_attention, lib.oracle_block_importance, lib.oracle_topp_select,
                      lib.oracle_index_build, lib.oracle_gather, lib.oracle_attention_compacted):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: oracle rejected its inputs (code {rc})")


def attention(q, k, v, cu_seqlens, positions, num_heads_q, num_heads_kv, head_dim,
              k_cache=None, v_cache=None, block_table=None, page_size=16, scale=None,
              rows=None, nthreads=None, prefix_lens=None):
    """Causal packed / chunked attention in fp64.

    q [N,Hq,D], k/v [N,Hkv,D] (uint16 bf16 bits); k_cache/v_cache
    [num_pages,page,Hkv,D]; block_table [S,max_pages].  Returns (out, lse):
    out float64 [R,Hq,D], lse float64 [R,Hq] with R = len(rows) or N.

    prefix_lens (int32 [S]): a compacted stream (kept tokens after selection):
    positions only increase inside a segment, a token sees its segment's tokens
    at or before its position, and segment s's cached prefix holds prefix_lens[s]
    tokens.  Without it positions are contiguous and the prefix is the first one.
    """
    lib = _load()
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    cu, pos = _c(cu_seqlens, np.int32), _c(positions, np.int32)
    n = int(cu[-1])
    kc, vc = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    bt = _c(block_table, np.int32)
    num_pages = 0 if kc is None else kc.shape[0]
    max_pages = 0 if bt is None else (bt.shape[1] if bt.ndim == 2 else bt.shape[0])
    rows_a = _c(rows, np.int32)
    r = n if rows_a is None else len(rows_a)
    out = np.zeros((r, num_heads_q, head_dim), np.float64)
    lse = np.zeros((r, num_heads_q), np.float64)
    if prefix_lens is None:
        rc = lib.oracle_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, _ptr(pos), n,
                                  _ptr(kc), _ptr(vc), num_pages, page_size, _ptr(bt), max_pages,
                                  num_heads_q, num_heads_kv, head_dim, float(scale or 0.0),
                                  _ptr(rows_a), r, _ptr(out), _ptr(lse),
                                  int(nthreads or default_threads()))
    else:
        pl = _c(prefix_lens, np.int32)
        rc = lib.oracle_attention_compacted(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, _ptr(pos),
                                            _ptr(pl), n, _ptr(kc), _ptr(vc), num_pages, page_size, _ptr(bt),
                                            max_pages, num_heads_q, num_heads_kv, head_dim, float(scale or 0.0),
                                            _ptr(rows_a), r, _ptr(out), _ptr(lse),
                                            int(nthreads or default_threads()))
    _check(rc, "attention")
    return out, lse


def block_importance(q, k, lse_full, cu_seqlens, num_heads_q, num_heads_kv, head_dim, block_size,
                     seg_mask=None, scale=None, nthreads=None):
    """Per-block importance (float64) and block offsets blk_cu (int32 [S+1]).

    lse_full: float64 [N,Hq] (only the scoring-window rows are read).
    """
    lib = _load()
    q, k = _c(q, np.uint16), _c(k, np.uint16)
    cu = _c(cu_seqlens, np.int32)
    n, S = int(cu[-1]), len(cu) - 1
    lse_a = _c(lse_full, np.float64)
    sm = _c(seg_mask, np.uint8)
    cap = n // block_size + S + 1
    imp = np.zeros(cap, np.float64)
    blk_cu = np.zeros(S + 1, np.int32)
    rc = lib.oracle_block_importance(_ptr(q), _ptr(k), _ptr(lse_a), _ptr(cu), S, n, _ptr(sm),
                                     block_size, num_heads_q, num_heads_kv, head_dim,
                                     float(scale or 0.0), _ptr(imp), cap, _ptr(blk_cu),
                                     int(nthreads or default_threads()))
    _check(rc, "block_importance")
    return imp[: blk_cu[-1]].copy(), blk_cu


def topp_select(imp_f32, blk_cu, p, flags=KEEP_FIRST | KEEP_LAST):
    """Top-p keep mask (uint8 per block) from float32 block scores."""
    lib = _load()
    imp_a = _c(imp_f32, np.float32)
    bc = _c(blk_cu, np.int32)
    keep = np.zeros(max(int(bc[-1]), 1), np.uint8)
    rc = lib.oracle_topp_select(_ptr(imp_a), _ptr(bc), len(bc) - 1, float(p), int(flags), _ptr(keep))
    _check(rc, "topp_select")
    return keep[: int(bc[-1])].copy()


def index_build(keep, blk_cu, cu_seqlens, positions, block_size):
    """(gather_idx, cu_seqlens_kept, positions_kept, n_kept) for a keep mask."""
    lib = _load()
    kp = _c(keep, np.uint8)
    if kp.size == 0:
        kp = np.zeros(1, np.uint8)
    bc, cu, pos = _c(blk_cu, np.int32), _c(cu_seqlens, np.int32), _c(positions, np.int32)
    n = int(cu[-1])
    gi = np.zeros(max(n, 1), np.int32)
    pk = np.zeros(max(n, 1), np.int32)
    ck = np.zeros(len(cu), np.int32)
    nk = np.zeros(1, np.int32)
    rc = lib.oracle_index_build(_ptr(kp), _ptr(bc), _ptr(cu), _ptr(pos), len(cu) - 1, block_size,
                                _ptr(gi), _ptr(ck), _ptr(pk), _ptr(nk))
    _check(rc, "index_build")
    m = int(nk[0])
    return gi[:m].copy(), ck, pk[:m].copy(), m


def gather(hidden, gather_idx):
    """Bit-exact row gather of uint16 (bf16 bits) hidden states."""
    lib = _load()
    h = _c(hidden, np.uint16)
    gi = _c(gather_idx, np.int32)
    out = np.zeros((len(gi), h.shape[1]), np.uint16)
    rc = lib.oracle_gather(_ptr(h), h.shape[1], h.shape[1], _ptr(gi), len(gi), h.shape[0], _ptr(out))
    _check(rc, "gather")
    return out
