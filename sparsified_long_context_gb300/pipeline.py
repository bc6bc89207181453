"""Device buffers and the four-call step of the path (marshalling only).

A step is: prefill attention -> block importance -> Top-p selection ->
gather of the kept tokens' hidden states.  Every call goes through the C ABI;
this module only owns the torch tensors (device memory) and the workspaces.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import binding as B
from .workloads import Workload


def _to_dev(a: Optional[np.ndarray], device, bf16: bool = False):
    import torch
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if bf16:
        t = t.view(torch.bfloat16)
    return t.to(device)


@dataclass
class DeviceInputs:
    """A workload's inputs resident in device memory."""
    wl: Workload
    q: object
    k: object
    v: object
    cu_seqlens: object
    positions: object
    k_cache: object = None
    v_cache: object = None
    block_table: object = None
    seg_mask: object = None
    hidden: object = None

    @classmethod
    def from_workload(cls, wl: Workload, device="cuda", with_hidden: bool = True):
        kc = vc = bt = None
        if wl.cache is not None:
            kc, vc = wl.cache.to_torch(device)
            bt = _to_dev(wl.block_table, device)
        return cls(wl, _to_dev(wl.q, device, True), _to_dev(wl.k, device, True), _to_dev(wl.v, device, True),
                   _to_dev(wl.cu_seqlens, device), _to_dev(wl.positions, device), kc, vc, bt,
                   _to_dev(wl.seg_mask, device),
                   _to_dev(wl.hidden, device, True) if (with_hidden and wl.hidden is not None) else None)


class StepBuffers:
    """Outputs and workspaces of one step, allocated once (torch owns the memory)."""

    def __init__(self, di: DeviceInputs, block_size: Optional[int] = None):
        import torch
        wl = di.wl
        dev = di.q.device
        n, S = wl.num_tokens, wl.num_segs
        hq, hkv, d = wl.num_heads_q, wl.num_heads_kv, wl.head_dim
        self.block_size = block_size or wl.block_size or 64
        bs = self.block_size
        self.out = torch.empty((n, hq, d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((hq, n), dtype=torch.float32, device=dev)
        cap = B.unip_importance_capacity(n, S, bs)
        self.imp = torch.empty(cap, dtype=torch.float32, device=dev)
        self.blk_cu = torch.empty(S + 1, dtype=torch.int32, device=dev)
        self.keep = torch.empty(cap, dtype=torch.uint8, device=dev)
        self.gather_idx = torch.empty(max(n, 1), dtype=torch.int32, device=dev)
        self.positions_kept = torch.empty(max(n, 1), dtype=torch.int32, device=dev)
        self.cu_seqlens_kept = torch.empty(S + 1, dtype=torch.int32, device=dev)
        self.n_kept = torch.empty(1, dtype=torch.int32, device=dev)
        self.hidden_out = None
        if di.hidden is not None:
            self.hidden_out = torch.empty_like(di.hidden)
        self.ws_attn = torch.empty(max(B.unip_attention_workspace_size(n, S, hq, hkv, d), 256), dtype=torch.uint8,
                                   device=dev)
        lib = B.load()
        prm = B._params(hq, hkv, d, 0.0)
        import ctypes
        self.ws_imp = torch.empty(max(int(lib.unip_importance_workspace_size(n, S, bs, ctypes.byref(prm))), 256),
                                  dtype=torch.uint8, device=dev)
        self.ws_topp = torch.empty(max(B.unip_topp_workspace_size(n, S, bs), 256), dtype=torch.uint8, device=dev)
        self.ws_fused = torch.empty(max(B.unip_importance_select_gather_workspace_size(n, S, bs, hq, hkv, d), 256),
                                    dtype=torch.uint8, device=dev)


def run_attention(di: DeviceInputs, bufs: StepBuffers, stream=None):
    wl = di.wl
    B.unip_prefill_attention(di.q, di.k, di.v, di.cu_seqlens, di.positions, bufs.out, bufs.lse,
                             num_heads_q=wl.num_heads_q, num_heads_kv=wl.num_heads_kv, head_dim=wl.head_dim,
                             k_cache=di.k_cache, v_cache=di.v_cache, block_table=di.block_table,
                             page_size=wl.cache.page_size if wl.cache is not None else 16,
                             workspace=bufs.ws_attn, stream=stream)


def attention_plan(wl: Workload, flags: int = 0) -> "B.AttentionPlan":
    """Host-built plan of the workload's attention calls, from its host-side layout."""
    return B.AttentionPlan(wl.cu_seqlens, wl.prefix_lens, num_heads_q=wl.num_heads_q,
                           num_heads_kv=wl.num_heads_kv, head_dim=wl.head_dim,
                           page_size=wl.cache.page_size if wl.cache is not None else 16,
                           max_pages_per_seq=wl.block_table.shape[1] if wl.block_table is not None else 0,
                           flags=flags)


def plan_workspace(plan, device):
    import torch
    return torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)


def run_attention_planned(di: DeviceInputs, bufs: StepBuffers, plan, workspace, stream=None):
    """unip_prefill_attention_planned with a plan from attention_plan() and its workspace."""
    wl = di.wl
    plan.run(di.q, di.k, di.v, bufs.out, bufs.lse, cu_seqlens=di.cu_seqlens, positions=di.positions,
             k_cache=di.k_cache, v_cache=di.v_cache, block_table=di.block_table,
             page_size=wl.cache.page_size if wl.cache is not None else 16, workspace=workspace, stream=stream)


def run_importance(di: DeviceInputs, bufs: StepBuffers, stream=None):
    wl = di.wl
    B.unip_block_importance(di.q, di.k, bufs.lse, di.cu_seqlens, bufs.imp, bufs.blk_cu,
                            block_size=bufs.block_size, num_heads_q=wl.num_heads_q,
                            num_heads_kv=wl.num_heads_kv, head_dim=wl.head_dim, seg_mask=di.seg_mask,
                            workspace=bufs.ws_imp, stream=stream)


def run_topp_gather(di: DeviceInputs, bufs: StepBuffers, p: Optional[float] = None, stream=None,
                    flags: int = B.UNIP_KEEP_FIRST | B.UNIP_KEEP_LAST):
    wl = di.wl
    B.unip_topp_select(bufs.imp, bufs.blk_cu, di.cu_seqlens, di.positions, bufs.keep, bufs.gather_idx,
                       bufs.cu_seqlens_kept, bufs.positions_kept, bufs.n_kept, block_size=bufs.block_size,
                       p=wl.top_p if p is None else p, flags=flags, workspace=bufs.ws_topp, stream=stream)
    if di.hidden is not None:
        B.unip_gather_tokens(di.hidden, bufs.gather_idx, bufs.n_kept, bufs.hidden_out, stream=stream)


def run_select_gather(di: DeviceInputs, bufs: StepBuffers, p: Optional[float] = None, stream=None,
                      flags: int = B.UNIP_KEEP_FIRST | B.UNIP_KEEP_LAST):
    """Top-p + index build + gather through the fused entry point (two kernel launches)."""
    wl = di.wl
    B.unip_select_gather(bufs.imp, bufs.blk_cu, di.cu_seqlens, di.positions, bufs.keep, bufs.gather_idx,
                         bufs.cu_seqlens_kept, bufs.positions_kept, bufs.n_kept, di.hidden, bufs.hidden_out,
                         block_size=bufs.block_size, p=wl.top_p if p is None else p, flags=flags,
                         workspace=bufs.ws_topp, stream=stream)


def run_importance_select_gather(di: DeviceInputs, bufs: StepBuffers, p: Optional[float] = None, stream=None,
                                 flags: int = B.UNIP_KEEP_FIRST | B.UNIP_KEEP_LAST, rows: bool = True):
    """Importance, Top-p and compaction through the fused entry point (importance's normaliser and the
    selection share one grid; the row copy follows as a programmatic dependent).  rows=False: the
    selection and the compaction indices only, no hidden row copied."""
    wl = di.wl
    hidden, hidden_out = (di.hidden, bufs.hidden_out) if rows else (None, None)
    B.unip_importance_select_gather(di.q, di.k, bufs.lse, di.cu_seqlens, di.positions, bufs.imp, bufs.blk_cu,
                                    bufs.keep, bufs.gather_idx, bufs.cu_seqlens_kept, bufs.positions_kept,
                                    bufs.n_kept, hidden, hidden_out, block_size=bufs.block_size,
                                    p=wl.top_p if p is None else p, num_heads_q=wl.num_heads_q,
                                    num_heads_kv=wl.num_heads_kv, head_dim=wl.head_dim, seg_mask=di.seg_mask,
                                    flags=flags, workspace=bufs.ws_fused, stream=stream)


def run_select(di: DeviceInputs, bufs: StepBuffers, p: Optional[float] = None, stream=None,
               flags: int = B.UNIP_KEEP_FIRST | B.UNIP_KEEP_LAST):
    run_importance(di, bufs, stream)
    run_topp_gather(di, bufs, p, stream, flags)


def run_step(di: DeviceInputs, bufs: StepBuffers, stream=None):
    """One pass of the whole path over one batch."""
    run_attention(di, bufs, stream)
    run_select(di, bufs, stream=stream)


def kernels_per_step(has_hidden: bool = True, fused_select: bool = False, num_segs: int = 2,
                     fused_importance: bool = False) -> int:
    """libunip kernels one step launches (device-planned attention, up to 12000 segments)."""
    # attention: plan + attention; importance: plan + score + norm;
    # Top-p: select + index, gather: 1  -- or the fused select + gather: 2,
    # one launch when the stream holds a single segment -- or importance, selection and
    # compaction in one call: plan + score + normalise-and-select + row copy, the last two one
    # grid when the stream holds a single segment
    if fused_importance:
        return 2 + (3 if num_segs == 1 else 4)
    if fused_select:
        return 2 + 3 + (1 if num_segs == 1 else 2)
    return 2 + 3 + 2 + (1 if has_hidden else 0)


class StreamedSteps:
    """The step over batches that live in pinned host memory, with the copies
    overlapped with the kernels.

    Two device sets (inputs + step buffers) alternate.  While batch i's kernels
    run on the compute stream, batch i+1's inputs are uploaded on an upload
    stream and batch i-1's results (attention output, n_kept and the n_kept
    compacted hidden rows) are downloaded on a download stream into pinned host
    buffers.  Events order the three streams; the host waits only for a batch's
    n_kept (to size its hidden-row copy) after the next batch is already queued,
    and for a set's last download before uploading into it again.
    """

    FIELDS = ("q", "k", "v", "hidden", "cu_seqlens", "positions", "seg_mask")

    def __init__(self, sets, compute_stream=None):
        import torch
        if len(sets) != 2:
            raise ValueError("StreamedSteps alternates between two device sets")
        self.sets = sets
        dev = sets[0][0].q.device
        self.cs = compute_stream or torch.cuda.current_stream(dev)
        self.up = torch.cuda.Stream(device=dev)
        self.down = torch.cuda.Stream(device=dev)
        self.out_host = [torch.empty(b.out.shape, dtype=b.out.dtype).pin_memory() for _, b in sets]
        self.hid_host = [None if b.hidden_out is None else
                         torch.empty(b.hidden_out.shape, dtype=b.hidden_out.dtype).pin_memory() for _, b in sets]
        self.nk_host = torch.zeros(2, dtype=torch.int32).pin_memory()
        self.fields = [f for f in self.FIELDS if getattr(sets[0][0], f) is not None]

    def host_batch(self, di: DeviceInputs):
        """Pinned host copies of a device set's input fields (a batch to stream)."""
        return {f: getattr(di, f).cpu().pin_memory() for f in self.fields}

    def bytes_up(self, batch) -> int:
        return sum(t.numel() * t.element_size() for t in batch.values())

    def run(self, batches, steps: int, on_result=None):
        """Runs `steps` steps, step i on batches[i % len(batches)].  Returns the
        n_kept of every step; on_result(i, out_host, hidden_rows_host, n_kept) is
        called once step i's downloads have landed (before its buffers are reused)."""
        import torch
        if steps < 0 or (steps > 0 and not batches):
            raise ValueError("StreamedSteps.run needs at least one batch and steps >= 0")
        ev = [[torch.cuda.Event() for _ in range(4)] for _ in range(2)]  # uploaded, computed, nk, downloaded
        n_kept = [0] * steps
        used = [None, None]   # step whose results a set holds

        def finish_download(i, s):
            _, bufs = self.sets[s]
            ev[s][2].synchronize()
            m = int(self.nk_host[s])
            n_kept[i] = m
            with torch.cuda.stream(self.down):
                if self.hid_host[s] is not None and m > 0:
                    self.hid_host[s][:m].copy_(bufs.hidden_out[:m], non_blocking=True)
                self.down.record_event(ev[s][3])

        def release(s):
            i = used[s]
            if i is None:
                return
            ev[s][3].synchronize()
            if on_result is not None:
                hid = None if self.hid_host[s] is None else self.hid_host[s][:n_kept[i]]
                on_result(i, self.out_host[s], hid, n_kept[i])
            used[s] = None

        pending = None
        for i in range(steps):
            s = i % 2
            di, bufs = self.sets[s]
            batch = batches[i % len(batches)]
            if used[s] is not None:
                release(s)
            with torch.cuda.stream(self.up):
                for f, t in batch.items():
                    getattr(di, f).copy_(t, non_blocking=True)
                self.up.record_event(ev[s][0])
            self.cs.wait_event(ev[s][0])
            run_attention(di, bufs, self.cs)
            run_importance_select_gather(di, bufs, stream=self.cs)
            self.cs.record_event(ev[s][1])
            # The previous step's hidden rows go on the download stream before this
            # step's downloads, which wait for this step's kernels.
            if pending is not None:
                finish_download(*pending)
            with torch.cuda.stream(self.down):
                self.down.wait_event(ev[s][1])
                self.out_host[s].copy_(bufs.out, non_blocking=True)
                self.nk_host[s:s + 1].copy_(bufs.n_kept, non_blocking=True)
                self.down.record_event(ev[s][2])
            used[s] = i
            pending = (i, s)
        if pending is not None:
            finish_download(*pending)
        for s in sorted((s for s in (0, 1) if used[s] is not None), key=lambda s: used[s]):
            release(s)
        torch.cuda.synchronize()
        return n_kept
