"""Thin ctypes binding of libunip (argument marshalling only).

Each function carries the name of the C entry point it calls and forwards
device pointers taken from torch tensors; every step of the path runs in the
library's CUDA kernels.  There is no CPU fallback: when libunip.so cannot be
loaded, or a tensor is not on a CUDA device, the call raises.

torch serves only as the owner of device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import native_build

_lib = None
_lock = threading.Lock()

UNIP_OK = 0
UNIP_KEEP_FIRST = 0x1
UNIP_KEEP_LAST = 0x2
UNIP_TOPP_MAX_BLOCKS = 8192
UNIP_ATTN_SCHEDULE_AUTO, UNIP_ATTN_SCHEDULE_PAIRED, UNIP_ATTN_SCHEDULE_SINGLE = 0, 1, 2

# device status bits (include/unip.h)
UNIP_DEV_BAD_SEQLENS, UNIP_DEV_BAD_POSITIONS, UNIP_DEV_BAD_PAGES, UNIP_DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8
UNIP_DEV_BAD_SCORES, UNIP_DEV_TOO_MANY_BLOCKS, UNIP_DEV_BAD_INDEX, UNIP_DEV_BAD_BLOCKS = 0x10, 0x20, 0x40, 0x80

DEV_STATUS_BITS = {
    0x1: "bad cu_seqlens", 0x2: "bad positions", 0x4: "bad pages", 0x8: "device wait timeout",
    0x10: "bad importance scores", 0x20: "too many blocks in a segment", 0x40: "bad gather index",
    0x80: "blk_cu does not match cu_seqlens",
}


class UnipError(RuntimeError):
    pass


class _AttnParams(ctypes.Structure):
    _fields_ = [("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("scale", ctypes.c_float)]


class _PagedKV(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("block_table", ctypes.c_void_p),
                ("max_pages_per_seq", ctypes.c_int32)]


class _StepBuffers(ctypes.Structure):
    _fields_ = [("cu_seqlens", ctypes.c_void_p), ("positions", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("request_ids", ctypes.c_void_p), ("seg_mask", ctypes.c_void_p),
                ("finished_ids", ctypes.c_void_p)]


class _StepCounts(ctypes.Structure):
    _fields_ = [("num_segs", ctypes.c_int32), ("num_tokens", ctypes.c_int32), ("num_decode", ctypes.c_int32),
                ("num_finished", ctypes.c_int32)]


def library_path() -> str:
    return native_build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load libunip.so (building it in-tree first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = native_build.LIB_PATH
        if build_if_missing and not native_build.up_to_date():
            native_build.build()
        if not os.path.exists(path):
            raise UnipError(f"libunip.so not found at {path}; run native_build.build()")
        lib = ctypes.CDLL(path)
        P, i32, i64, u32, f64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                     ctypes.c_double, ctypes.c_size_t)
        pp = ctypes.POINTER(_AttnParams)
        lib.unip_version.restype = ctypes.c_char_p
        lib.unip_status_string.restype = ctypes.c_char_p
        lib.unip_status_string.argtypes = [i32]
        lib.unip_last_cuda_error.restype = ctypes.c_char_p
        lib.unip_last_cuda_error.argtypes = []
        lib.unip_get_device_status.restype = i32
        lib.unip_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        lib.unip_attention_workspace_size.restype = sz
        lib.unip_attention_workspace_size.argtypes = [i32, i32, pp]
        lib.unip_prefill_attention.restype = i32
        lib.unip_prefill_attention.argtypes = [P, P, P, P, i32, P, i32, ctypes.POINTER(_PagedKV), pp, P, P, P, sz, P]
        lib.unip_compacted_attention.restype = i32
        lib.unip_compacted_attention.argtypes = [P, P, P, P, i32, P, P, i32, ctypes.POINTER(_PagedKV), pp, P, P, P,
                                                 sz, P]
        lib.unip_prefill_attention_noalloc.restype = i32
        lib.unip_prefill_attention_noalloc.argtypes = [P, P, P, P, i32, P, i32, ctypes.POINTER(_PagedKV), pp, P, P,
                                                       P]
        lib.unip_attention_plan_create.restype = i32
        lib.unip_attention_plan_create.argtypes = [P, i32, P, i32, pp, i32, i32, i32, i32, ctypes.POINTER(P)]
        lib.unip_attention_plan_workspace_size.restype = sz
        lib.unip_attention_plan_workspace_size.argtypes = [P]
        lib.unip_attention_plan_info.restype = i32
        lib.unip_attention_plan_info.argtypes = [P, P]
        lib.unip_attention_plan_destroy.restype = None
        lib.unip_attention_plan_destroy.argtypes = [P]
        lib.unip_prefill_attention_planned.restype = i32
        lib.unip_prefill_attention_planned.argtypes = [P, P, P, P, P, P, P, ctypes.POINTER(_PagedKV), P, P, P, sz,
                                                       P]
        lib.unip_importance_capacity.restype = i32
        lib.unip_importance_capacity.argtypes = [i32, i32, i32]
        lib.unip_importance_workspace_size.restype = sz
        lib.unip_importance_workspace_size.argtypes = [i32, i32, i32, pp]
        lib.unip_block_importance.restype = i32
        lib.unip_block_importance.argtypes = [P, P, P, P, i32, i32, P, i32, pp, P, i32, P, P, sz, P]
        lib.unip_topp_workspace_size.restype = sz
        lib.unip_topp_workspace_size.argtypes = [i32, i32, i32]
        lib.unip_topp_select.restype = i32
        lib.unip_topp_select.argtypes = [P, P, P, P, i32, i32, i32, f64, u32, P, i32, P, P, P, P, P, sz, P]
        lib.unip_select_gather.restype = i32
        lib.unip_select_gather.argtypes = [P, P, P, P, i32, i32, i32, f64, u32, P, i32, P, P, P, P, P, i64, i32, P, i64,
                                           P, sz, P]
        lib.unip_importance_select_gather_workspace_size.restype = sz
        lib.unip_importance_select_gather_workspace_size.argtypes = [i32, i32, i32, pp]
        lib.unip_importance_select_gather.restype = i32
        lib.unip_importance_select_gather.argtypes = [P, P, P, P, P, i32, i32, P, i32, pp, f64, u32, P, i32, P, P,
                                                      P, P, P, P, P, i64, i32, P, i64, P, sz, P]
        lib.unip_gather_tokens.restype = i32
        lib.unip_gather_tokens.argtypes = [P, i32, i64, i32, P, P, i32, P, i64, P]
        lib.unip_selftest_bounded_wait.restype = i32
        lib.unip_selftest_bounded_wait.argtypes = [u32, P, P]
        lib.unip_set_attention_schedule.restype = i32
        lib.unip_set_attention_schedule.argtypes = [i32]
        lib.unip_rope_append_kv.restype = i32
        lib.unip_rope_append_kv.argtypes = [P, P, P, P, i32, pp, f64, i32, P, P, P, i32, i32, P]
        lib.unip_ffd_pack.restype = i32
        lib.unip_ffd_pack.argtypes = [P, i32, i32, P, P, P]
        lib.unip_pack_metadata.restype = i32
        lib.unip_pack_metadata.argtypes = [P, i32, P, P, P, P]
        lib.unip_step_builder_create.restype = i32
        lib.unip_step_builder_create.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(P)]
        lib.unip_step_builder_destroy.restype = None
        lib.unip_step_builder_destroy.argtypes = [P]
        lib.unip_step_builder_add.restype = i32
        lib.unip_step_builder_add.argtypes = [P, i32, i32, ctypes.POINTER(ctypes.c_int32)]
        lib.unip_step_builder_next.restype = i32
        lib.unip_step_builder_next.argtypes = [P, ctypes.POINTER(_StepBuffers), ctypes.POINTER(_StepCounts)]
        lib.unip_step_builder_state.restype = i32
        lib.unip_step_builder_state.argtypes = [P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                                ctypes.POINTER(ctypes.c_int32)]
        _lib = lib
        return lib


UNIP_ERR_CUDA = -4


def _check(rc: int, what: str):
    if rc != UNIP_OK:
        lib = load()
        msg = lib.unip_status_string(rc).decode()
        if rc == UNIP_ERR_CUDA:
            msg += f": {lib.unip_last_cuda_error().decode()}"
        raise UnipError(f"{what} failed: {msg} (code {rc})")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise UnipError("libunip takes CUDA tensors only (no CPU fallback)")
    if not t.is_contiguous():
        raise UnipError("libunip takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _params(hq, hkv, d, scale):
    return _AttnParams(int(hq), int(hkv), int(d), float(scale or 0.0))


def _workspace(nbytes: int, device):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def unip_version() -> str:
    return load().unip_version().decode()


def unip_get_device_status(clear: bool = True) -> int:
    """Device status bits (synchronises the current device)."""
    bits = ctypes.c_uint32(0)
    _check(load().unip_get_device_status(ctypes.byref(bits), 1 if clear else 0), "unip_get_device_status")
    return int(bits.value)


def describe_status(bits: int) -> str:
    return ", ".join(v for k, v in DEV_STATUS_BITS.items() if bits & k) or "ok"


def unip_selftest_bounded_wait(limit_us: int, gave_up, stream=None):
    """Runs the bounded-wait self-test (gave_up: int32 CUDA tensor of 3 elements)."""
    _check(load().unip_selftest_bounded_wait(int(limit_us), _ptr(gave_up), _stream(stream)),
           "unip_selftest_bounded_wait")


def unip_set_attention_schedule(mode: int):
    """Work-item shape of later attention calls: AUTO, PAIRED (two query tiles) or SINGLE (one)."""
    _check(load().unip_set_attention_schedule(int(mode)), "unip_set_attention_schedule")


def unip_attention_workspace_size(total_tokens, num_segs, hq, hkv, d) -> int:
    p = _params(hq, hkv, d, 0.0)
    return int(load().unip_attention_workspace_size(int(total_tokens), int(num_segs), ctypes.byref(p)))


def unip_prefill_attention(q, k, v, cu_seqlens, positions, out, lse=None, *, num_heads_q, num_heads_kv,
                           head_dim, k_cache=None, v_cache=None, block_table=None, page_size=16,
                           scale=None, workspace=None, stream=None):
    """Packed / chunked causal attention: writes out [N,Hq,D] bf16 and lse [Hq,N] fp32."""
    lib = load()
    n = int(q.shape[0])
    S = int(cu_seqlens.shape[0]) - 1
    prm = _params(num_heads_q, num_heads_kv, head_dim, scale)
    need = lib.unip_attention_workspace_size(n, S, ctypes.byref(prm))
    if workspace is None:
        workspace = _workspace(need, q.device)
    paged_p = None
    if k_cache is not None:
        paged = _PagedKV(_ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]), int(page_size), _ptr(block_table),
                         int(block_table.shape[1]))
        paged_p = ctypes.byref(paged)
    rc = lib.unip_prefill_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), S, _ptr(positions), n, paged_p,
                                    ctypes.byref(prm), _ptr(out), _ptr(lse), _ptr(workspace),
                                    workspace.numel(), _stream(stream))
    _check(rc, "unip_prefill_attention")
    return out, lse


def unip_compacted_attention(q, k, v, cu_seqlens, positions, prefix_lens, out, lse=None, *, num_heads_q,
                             num_heads_kv, head_dim, k_cache=None, v_cache=None, block_table=None, page_size=16,
                             scale=None, workspace=None, stream=None):
    """Attention over a compacted stream: kept tokens with their (increasing) original positions and an
    explicit cached-prefix length per segment (prefix_lens, int32 [S] on the device)."""
    lib = load()
    n = int(q.shape[0])
    S = int(cu_seqlens.shape[0]) - 1
    prm = _params(num_heads_q, num_heads_kv, head_dim, scale)
    need = lib.unip_attention_workspace_size(n, S, ctypes.byref(prm))
    if workspace is None:
        workspace = _workspace(need, q.device)
    paged_p = None
    if k_cache is not None:
        paged = _PagedKV(_ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]), int(page_size), _ptr(block_table),
                         int(block_table.shape[1]))
        paged_p = ctypes.byref(paged)
    rc = lib.unip_compacted_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), S, _ptr(positions),
                                      _ptr(prefix_lens), n, paged_p, ctypes.byref(prm), _ptr(out), _ptr(lse),
                                      _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "unip_compacted_attention")
    return out, lse


UNIP_PLAN_NO_SPLIT = 0x1
UNIP_PLAN_DEVICE = 0x2


def UNIP_PLAN_SPLITS(n: int) -> int:
    return (int(n) & 0xFF) << 8


class AttentionPlan:
    """Host-built work plan of attention calls over one batch layout (unip_attention_plan_*).

    cu_seqlens and prefix_lens are host arrays (numpy or lists); the plan is reused by every call
    with that layout.  ``workspace_bytes`` is the device workspace a run needs; ``info`` reports
    whether the plan is host-built, its items, CTAs, split units, key splits and tile shape."""

    def __init__(self, cu_seqlens, prefix_lens, *, num_heads_q, num_heads_kv, head_dim, page_size=16,
                 max_pages_per_seq=0, scale=None, flags=0, num_sms=0):
        import numpy as np
        lib = load()
        self._lib = lib
        self._h = None
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        S = int(cu.shape[0]) - 1
        pre = None if prefix_lens is None else np.ascontiguousarray(prefix_lens, dtype=np.int32)
        if pre is not None and pre.shape[0] != S:
            raise UnipError("prefix_lens must have one entry per segment")
        self.num_tokens = int(cu[-1])
        self.num_segs = S
        self.head_dim = int(head_dim)
        self.num_heads_q = int(num_heads_q)
        prm = _params(num_heads_q, num_heads_kv, head_dim, scale)
        h = ctypes.c_void_p()
        _check(lib.unip_attention_plan_create(cu.ctypes.data, S, None if pre is None else pre.ctypes.data,
                                              self.num_tokens, ctypes.byref(prm), int(page_size),
                                              int(max_pages_per_seq), int(flags), int(num_sms), ctypes.byref(h)),
               "unip_attention_plan_create")
        self._h = h
        self.workspace_bytes = int(lib.unip_attention_plan_workspace_size(h))
        info = (ctypes.c_int32 * 6)()
        _check(lib.unip_attention_plan_info(h, info), "unip_attention_plan_info")
        self.info = {"host": bool(info[0]), "items": info[1], "ctas": info[2], "split_units": info[3],
                     "splits": info[4], "single": bool(info[5])}

    def close(self):
        if self._h is not None:
            self._lib.unip_attention_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def run(self, q, k, v, out, lse=None, *, cu_seqlens=None, positions=None, prefix_lens=None, k_cache=None,
            v_cache=None, block_table=None, page_size=16, workspace=None, stream=None):
        """unip_prefill_attention_planned: out [N,Hq,D] bf16 and lse [Hq,N] fp32 (device tensors).
        cu_seqlens / positions / prefix_lens: the device copies of the layout (read only when the plan
        fell back to the device planner)."""
        if workspace is None:
            workspace = _workspace(self.workspace_bytes, q.device)
        paged_p = None
        if k_cache is not None:
            paged = _PagedKV(_ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]), int(page_size), _ptr(block_table),
                             int(block_table.shape[1]))
            paged_p = ctypes.byref(paged)
        rc = self._lib.unip_prefill_attention_planned(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens),
                                                      _ptr(positions), _ptr(prefix_lens), paged_p, _ptr(out),
                                                      _ptr(lse), _ptr(workspace), workspace.numel(),
                                                      _stream(stream))
        _check(rc, "unip_prefill_attention_planned")
        return out, lse


def unip_prefill_attention_noalloc(q, k, v, cu_seqlens, positions, out, lse=None, *, num_heads_q, num_heads_kv,
                                   head_dim, k_cache=None, v_cache=None, block_table=None, page_size=16,
                                   scale=None, stream=None):
    """Same result as unip_prefill_attention, with the library's built-in scratch.

    For callers that cannot allocate device memory: nothing is allocated here
    either (no workspace tensor).  The library's one scratch array per device
    is shared by every call, so calls that may overlap on the GPU must be
    serialised by the caller; the first call on a device should come before
    any stream capture.
    """
    lib = load()
    n = int(q.shape[0])
    S = int(cu_seqlens.shape[0]) - 1
    prm = _params(num_heads_q, num_heads_kv, head_dim, scale)
    paged_p = None
    if k_cache is not None:
        paged = _PagedKV(_ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]), int(page_size), _ptr(block_table),
                         int(block_table.shape[1]))
        paged_p = ctypes.byref(paged)
    rc = lib.unip_prefill_attention_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), S, _ptr(positions), n,
                                            paged_p, ctypes.byref(prm), _ptr(out), _ptr(lse), _stream(stream))
    _check(rc, "unip_prefill_attention_noalloc")
    return out, lse


def unip_importance_capacity(total_tokens, num_segs, block_size) -> int:
    return int(load().unip_importance_capacity(int(total_tokens), int(num_segs), int(block_size)))


def unip_block_importance(q, k, lse, cu_seqlens, imp, blk_cu, *, block_size, num_heads_q, num_heads_kv,
                          head_dim, seg_mask=None, scale=None, workspace=None, stream=None):
    """Per-block importance imp (fp32) and block offsets blk_cu (int32 [S+1])."""
    lib = load()
    n = int(q.shape[0])
    S = int(cu_seqlens.shape[0]) - 1
    prm = _params(num_heads_q, num_heads_kv, head_dim, scale)
    need = lib.unip_importance_workspace_size(n, S, int(block_size), ctypes.byref(prm))
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.unip_block_importance(_ptr(q), _ptr(k), _ptr(lse), _ptr(cu_seqlens), S, n, _ptr(seg_mask),
                                   int(block_size), ctypes.byref(prm), _ptr(imp), int(imp.numel()), _ptr(blk_cu),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "unip_block_importance")
    return imp, blk_cu


def unip_topp_workspace_size(total_tokens, num_segs, block_size) -> int:
    return int(load().unip_topp_workspace_size(int(total_tokens), int(num_segs), int(block_size)))


def unip_topp_select(imp, blk_cu, cu_seqlens, positions, keep, gather_idx, cu_seqlens_kept, positions_kept,
                     n_kept, *, block_size, p, flags=UNIP_KEEP_FIRST | UNIP_KEEP_LAST, workspace=None,
                     stream=None):
    """Top-p keep mask and compaction indices; n_kept stays on the device."""
    lib = load()
    n = int(positions.shape[0])
    S = int(cu_seqlens.shape[0]) - 1
    need = lib.unip_topp_workspace_size(n, S, int(block_size))
    if workspace is None:
        workspace = _workspace(need, imp.device)
    rc = lib.unip_topp_select(_ptr(imp), _ptr(blk_cu), _ptr(cu_seqlens), _ptr(positions), S, n, int(block_size),
                              float(p), int(flags), _ptr(keep), int(keep.numel()), _ptr(gather_idx),
                              _ptr(cu_seqlens_kept), _ptr(positions_kept), _ptr(n_kept), _ptr(workspace),
                              workspace.numel(), _stream(stream))
    _check(rc, "unip_topp_select")


def unip_select_gather(imp, blk_cu, cu_seqlens, positions, keep, gather_idx, cu_seqlens_kept, positions_kept,
                       n_kept, hidden, hidden_out, *, block_size, p, flags=UNIP_KEEP_FIRST | UNIP_KEEP_LAST,
                       workspace=None, stream=None):
    """Top-p selection, compaction indices and the hidden-state gather in two kernel launches."""
    lib = load()
    n = int(positions.shape[0])
    S = int(cu_seqlens.shape[0]) - 1
    need = lib.unip_topp_workspace_size(n, S, int(block_size))
    if workspace is None:
        workspace = _workspace(need, imp.device)
    if (hidden is None) != (hidden_out is None):
        raise UnipError("hidden and hidden_out are given together or not at all")
    if hidden is None:  # selection and indices only
        h_ptr = o_ptr = None
        h_stride = o_stride = d_model = 0
    else:
        for t in (hidden, hidden_out):
            if not t.is_cuda:
                raise UnipError("libunip takes CUDA tensors only (no CPU fallback)")
        h_ptr, o_ptr = hidden.data_ptr(), hidden_out.data_ptr()
        h_stride, o_stride, d_model = int(hidden.stride(0)), int(hidden_out.stride(0)), int(hidden.shape[1])
    rc = lib.unip_select_gather(_ptr(imp), _ptr(blk_cu), _ptr(cu_seqlens), _ptr(positions), S, n, int(block_size),
                                float(p), int(flags), _ptr(keep), int(keep.numel()), _ptr(gather_idx),
                                _ptr(cu_seqlens_kept), _ptr(positions_kept), _ptr(n_kept), h_ptr, h_stride,
                                d_model, o_ptr, o_stride, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "unip_select_gather")


def unip_importance_select_gather_workspace_size(total_tokens, num_segs, block_size, hq, hkv, d) -> int:
    p = _params(hq, hkv, d, 0.0)
    return int(load().unip_importance_select_gather_workspace_size(int(total_tokens), int(num_segs), int(block_size),
                                                                   ctypes.byref(p)))


def unip_importance_select_gather(q, k, lse, cu_seqlens, positions, imp, blk_cu, keep, gather_idx, cu_seqlens_kept,
                                  positions_kept, n_kept, hidden, hidden_out, *, block_size, p, num_heads_q,
                                  num_heads_kv, head_dim, seg_mask=None, scale=None,
                                  flags=UNIP_KEEP_FIRST | UNIP_KEEP_LAST, workspace=None, stream=None):
    """Block importance, Top-p selection and compaction in one call (the outputs of
    unip_block_importance and unip_select_gather)."""
    lib = load()
    n = int(positions.shape[0])
    S = int(cu_seqlens.shape[0]) - 1
    prm = _params(num_heads_q, num_heads_kv, head_dim, scale)
    need = lib.unip_importance_select_gather_workspace_size(n, S, int(block_size), ctypes.byref(prm))
    if workspace is None:
        workspace = _workspace(need, q.device)
    if (hidden is None) != (hidden_out is None):
        raise UnipError("hidden and hidden_out are given together or not at all")
    if hidden is None:
        h_ptr = o_ptr = None
        h_stride = o_stride = d_model = 0
    else:
        for t in (hidden, hidden_out):
            if not t.is_cuda:
                raise UnipError("libunip takes CUDA tensors only (no CPU fallback)")
        h_ptr, o_ptr = hidden.data_ptr(), hidden_out.data_ptr()
        h_stride, o_stride, d_model = int(hidden.stride(0)), int(hidden_out.stride(0)), int(hidden.shape[1])
    rc = lib.unip_importance_select_gather(_ptr(q), _ptr(k), _ptr(lse), _ptr(cu_seqlens), _ptr(positions), S, n,
                                           _ptr(seg_mask), int(block_size), ctypes.byref(prm), float(p), int(flags),
                                           _ptr(imp), int(imp.numel()), _ptr(blk_cu), _ptr(keep), _ptr(gather_idx),
                                           _ptr(cu_seqlens_kept), _ptr(positions_kept), _ptr(n_kept), h_ptr, h_stride,
                                           d_model, o_ptr, o_stride, _ptr(workspace), workspace.numel(),
                                           _stream(stream))
    _check(rc, "unip_importance_select_gather")


def unip_gather_tokens(hidden, gather_idx, n_kept, out, *, stream=None):
    """out[i] = hidden[gather_idx[i]] for i < n_kept (device scalar)."""
    lib = load()
    rows, d = int(hidden.shape[0]), int(hidden.shape[1])
    rc = lib.unip_gather_tokens(_ptr(hidden), rows, int(hidden.stride(0)), d, _ptr(gather_idx), _ptr(n_kept),
                                int(out.shape[0]), _ptr(out), int(out.stride(0)), _stream(stream))
    _check(rc, "unip_gather_tokens")
    return out


def unip_rope_append_kv(q, k, v=None, positions=None, *, num_heads_q, num_heads_kv, head_dim,
                        rope_theta=10000.0, interleaved=False, slot_mapping=None, k_cache=None, v_cache=None,
                        page_size=16, stream=None):
    """Rotary embedding of q and k in place by `positions`; with `slot_mapping`,
    also writes the rotated k and v rows into the paged caches."""
    lib = load()
    n = int(k.shape[0])
    prm = _params(num_heads_q, num_heads_kv, head_dim, 0.0)
    num_pages = int(k_cache.shape[0]) if k_cache is not None else 0
    rc = lib.unip_rope_append_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), n, ctypes.byref(prm),
                                 float(rope_theta), 1 if interleaved else 0, _ptr(slot_mapping), _ptr(k_cache),
                                 _ptr(v_cache), num_pages, int(page_size), _stream(stream))
    _check(rc, "unip_rope_append_kv")
    return q, k

# ---------------------------------------------------------------------------
# Host-side batch builders (include/unip_sched.h).  These take and return
# numpy arrays in host memory; the library does the packing and scheduling.

def _host_i32(a):
    import numpy as np
    return np.ascontiguousarray(a, dtype=np.int32)


def unip_ffd_pack(lengths, capacity: int):
    """First-fit-decreasing packing -> (order int32[n], bin_cu int32[num_bins + 1])."""
    import numpy as np
    lengths = _host_i32(lengths)
    n = int(lengths.size)
    order = np.empty(n, np.int32)
    bin_cu = np.zeros(n + 1, np.int32)
    nb = ctypes.c_int32(0)
    _check(load().unip_ffd_pack(lengths.ctypes.data if n else None, n, int(capacity),
                                order.ctypes.data if n else None, bin_cu.ctypes.data, ctypes.byref(nb)),
           "unip_ffd_pack")
    return order, bin_cu[: nb.value + 1].copy()


def unip_pack_metadata(lengths, order):
    """Packed-stream metadata -> (cu_seqlens, positions, src_index), int32 host arrays."""
    import numpy as np
    lengths = _host_i32(lengths)
    order = _host_i32(order)
    n = int(lengths.size)
    if order.size != n:
        raise UnipError("order must have one entry per prompt")
    total = int(lengths.astype(np.int64).sum())
    cu = np.zeros(n + 1, np.int32)
    pos = np.empty(total, np.int32)
    src = np.empty(total, np.int32)
    _check(load().unip_pack_metadata(lengths.ctypes.data if n else None, n, order.ctypes.data if n else None,
                                     cu.ctypes.data, pos.ctypes.data if total else None,
                                     src.ctypes.data if total else None), "unip_pack_metadata")
    return cu, pos, src


class StepBuilder:
    """Token-budget step builder with a paged KV cache (unip_step_builder_*).

    ``next()`` returns a dict of host int32/uint8 arrays trimmed to the step:
    cu_seqlens, positions, slot_mapping, block_table [S, max_pages_per_seq],
    request_ids, seg_mask, finished_ids, num_decode.
    """

    def __init__(self, token_budget: int, page_size: int, num_pages: int, max_pages_per_seq: int,
                 max_seqs: int, chunk_multiple: int = 1):
        import numpy as np
        self._lib = load()
        h = ctypes.c_void_p(None)
        _check(self._lib.unip_step_builder_create(int(token_budget), int(page_size), int(num_pages),
                                                  int(max_pages_per_seq), int(max_seqs), int(chunk_multiple),
                                                  ctypes.byref(h)), "unip_step_builder_create")
        self._h = h
        self.token_budget, self.page_size, self.num_pages = int(token_budget), int(page_size), int(num_pages)
        self.max_pages_per_seq, self.max_seqs = int(max_pages_per_seq), int(max_seqs)
        self._cu = np.zeros(self.max_seqs + 1, np.int32)
        self._pos = np.zeros(self.token_budget, np.int32)
        self._slot = np.zeros(self.token_budget, np.int32)
        self._bt = np.zeros((self.max_seqs, self.max_pages_per_seq), np.int32)
        self._rid = np.zeros(self.max_seqs, np.int32)
        self._mask = np.zeros(self.max_seqs, np.uint8)
        self._fin = np.zeros(self.max_seqs, np.int32)
        self._bufs = _StepBuffers(*(a.ctypes.data for a in (self._cu, self._pos, self._slot, self._bt, self._rid,
                                                              self._mask, self._fin)))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value is not None:
            self._lib.unip_step_builder_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, prompt_len: int, max_new_tokens: int) -> int:
        rid = ctypes.c_int32(-1)
        _check(self._lib.unip_step_builder_add(self._h, int(prompt_len), int(max_new_tokens), ctypes.byref(rid)),
               "unip_step_builder_add")
        return rid.value

    def state(self):
        """(requests with prompt tokens left, requests decoding, free pages)."""
        a, b, c = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        _check(self._lib.unip_step_builder_state(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "unip_step_builder_state")
        return a.value, b.value, c.value

    def next(self) -> dict:
        cnt = _StepCounts()
        _check(self._lib.unip_step_builder_next(self._h, ctypes.byref(self._bufs), ctypes.byref(cnt)),
               "unip_step_builder_next")
        s, n = cnt.num_segs, cnt.num_tokens
        return {"cu_seqlens": self._cu[: s + 1].copy(), "positions": self._pos[:n].copy(),
                "slot_mapping": self._slot[:n].copy(), "block_table": self._bt[:s].copy(),
                "request_ids": self._rid[:s].copy(), "seg_mask": self._mask[:s].copy(),
                "finished_ids": self._fin[: cnt.num_finished].copy(), "num_decode": cnt.num_decode}
