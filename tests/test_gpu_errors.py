"""Metadata errors that only the device can see (the error model of include/unip.h): each kernel's own
check turns the bad input into a status bit before any access that would use it, the call writes
nothing it should not, and the next call on the same context is clean and correct.

Every case here is one of the checks the kernels carry: cu_seqlens and positions are validated by the
attention planner before it publishes any work item, a page id outside the cache becomes an
out-of-range TMA page coordinate (which reads zeros), Top-p rejects a segment whose block count does
not match its length before reading its scores, and the row copy tests every source index and the
kept count against the buffers before it copies."""
import numpy as np
import pytest

from sparsified_long_context_gb300 import workloads as W

from gpu_harness import assert_close, bf16_tensor_to_f64, oracle_attention_rows, LSE_ABS
from test_gpu_attention import _chunk_with_prefix

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

_POISON = 0x5A5A


def _attention_after(wl, edit):
    """Runs attention on the workload's device inputs after edit(di); returns (status bits, buffers)."""
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import DeviceInputs, StepBuffers, run_attention
    B.unip_get_device_status(clear=True)
    di = DeviceInputs.from_workload(wl, "cuda", with_hidden=False)
    bufs = StepBuffers(di, block_size=64)
    edit(di)
    bufs.out.view(torch.int16).fill_(_POISON)
    run_attention(di, bufs)
    torch.cuda.synchronize()
    return B.unip_get_device_status(clear=True), bufs


def _clean_call_still_correct():
    """A valid call right after the failed one: no status bit, and the oracle's result."""
    wl = W.tiny_packed()
    st, bufs = _attention_after(wl, lambda di: None)
    assert st == 0
    ref_o, ref_l = oracle_attention_rows(wl, None)
    assert_close(bf16_tensor_to_f64(bufs.out), ref_o, what="attention after the error")
    assert_close(bufs.lse.cpu().numpy().astype(np.float64).T, ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS,
                 what="lse after the error")


def test_non_monotone_cu_seqlens_raise_and_write_nothing():
    from sparsified_long_context_gb300 import binding as B
    wl = W.packed([100, 156], 4, 2, 64, seed=81)

    def edit(di):
        di.cu_seqlens[1] = 300  # after cu[2] = 256: the second segment would have -44 tokens

    st, bufs = _attention_after(wl, edit)
    assert st & B.UNIP_DEV_BAD_SEQLENS, B.describe_status(st)
    assert not st & B.UNIP_DEV_TIMEOUT
    assert bool((bufs.out.view(torch.int16) == _POISON).all())
    _clean_call_still_correct()


def test_positions_with_a_gap_inside_a_segment_raise_and_write_nothing():
    from sparsified_long_context_gb300 import binding as B
    wl = W.packed([100, 156], 4, 2, 64, seed=82)

    def edit(di):
        di.positions[150:] += 3  # segment 1 (tokens 100..255) jumps from position 49 to 53

    st, bufs = _attention_after(wl, edit)
    assert st & B.UNIP_DEV_BAD_POSITIONS, B.describe_status(st)
    assert not st & B.UNIP_DEV_TIMEOUT
    assert bool((bufs.out.view(torch.int16) == _POISON).all())
    _clean_call_still_correct()


def test_page_id_outside_the_cache_raises_and_reads_zeros():
    """Page 1 of the prefix names a page past the cache: the call raises UNIP_DEV_BAD_PAGES, still
    finishes, and reads that page as zeros, which is the oracle's result with the block table pointing
    at one of the cache's unused (all-zero) pages instead."""
    from sparsified_long_context_gb300 import binding as B
    wl = _chunk_with_prefix(64, 40, 4, 2, 64, 16, seed=83)
    num_pages = wl.cache.num_pages
    unused = sorted(set(range(num_pages)) - set(int(x) for x in wl.block_table[0]))
    assert unused

    def edit(di):
        di.block_table[0, 1] = num_pages

    st, bufs = _attention_after(wl, edit)
    assert st & B.UNIP_DEV_BAD_PAGES, B.describe_status(st)
    assert not st & B.UNIP_DEV_TIMEOUT
    zeroed = W.Workload(wl.name + "_zero_page", wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.cu_seqlens,
                        wl.positions, wl.q, wl.k, wl.v, cache=wl.cache, block_table=wl.block_table.copy())
    zeroed.block_table[0, 1] = unused[0]
    ref_o, ref_l = oracle_attention_rows(zeroed, None)
    assert_close(bf16_tensor_to_f64(bufs.out), ref_o, what="out with a zero page")
    assert_close(bufs.lse.cpu().numpy().astype(np.float64).T, ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS,
                 what="lse with a zero page")
    _clean_call_still_correct()


def test_block_counts_that_do_not_match_the_lengths_keep_nothing():
    from sparsified_long_context_gb300 import binding as B
    dev = "cuda"
    B.unip_get_device_status(clear=True)
    cu = np.array([0, 100, 300], np.int32)          # 7 and 13 blocks of 16
    blk_cu = np.array([0, 8, 20], np.int32)         # claims 8 and 12
    n, S, B_ = 300, 2, 16
    pos = np.concatenate([np.arange(100), np.arange(200)]).astype(np.int32)
    cap = B.unip_importance_capacity(n, S, B_)
    imp = torch.full((cap,), 0.05, dtype=torch.float32, device=dev)
    keep = torch.full((cap,), 7, dtype=torch.uint8, device=dev)
    gi = torch.full((n,), -1, dtype=torch.int32, device=dev)
    pk = torch.full((n,), -1, dtype=torch.int32, device=dev)
    ck = torch.full((S + 1,), -1, dtype=torch.int32, device=dev)
    nk = torch.full((1,), -1, dtype=torch.int32, device=dev)
    B.unip_topp_select(imp, torch.from_numpy(blk_cu).to(dev), torch.from_numpy(cu).to(dev),
                       torch.from_numpy(pos).to(dev), keep, gi, ck, pk, nk, block_size=B_, p=0.9)
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st & B.UNIP_DEV_BAD_BLOCKS, B.describe_status(st)
    assert int(nk.item()) == 0
    assert ck.cpu().numpy().tolist() == [0, 0, 0]
    assert bool((gi == -1).all()) and bool((pk == -1).all())


def test_gather_indices_out_of_range_are_skipped():
    """Rows whose source index is outside the hidden matrix are not copied (their output rows keep
    their old bytes), the others are, and a kept count above the output's rows is cut to them."""
    from sparsified_long_context_gb300 import binding as B
    dev = "cuda"
    rng = np.random.default_rng(84)
    rows, d = 50, 64
    hid = torch.from_numpy(W.f32_to_bf16_bits(rng.standard_normal((rows, d), dtype=np.float32))).view(
        torch.bfloat16).to(dev)
    idx = np.array([3, 49, 50, -1, 7, 1 << 30, 0], np.int32)
    out = torch.zeros((len(idx), d), dtype=torch.bfloat16, device=dev)
    out.view(torch.int16).fill_(_POISON)
    B.unip_get_device_status(clear=True)
    B.unip_gather_tokens(hid, torch.from_numpy(idx).to(dev), torch.tensor([len(idx)], dtype=torch.int32,
                                                                           device=dev), out)
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st & B.UNIP_DEV_BAD_INDEX, B.describe_status(st)
    got = out.view(torch.int16).cpu().numpy()
    src = hid.view(torch.int16).cpu().numpy()
    for r, s in enumerate(idx):
        if 0 <= s < rows:
            assert np.array_equal(got[r], src[s]), r
        else:
            assert (got[r] == _POISON).all(), r
    # a kept count above the output's rows: the first len(idx) rows are copied, nothing past them
    big = torch.zeros((len(idx) + 8, d), dtype=torch.bfloat16, device=dev)
    idx2 = torch.from_numpy(np.arange(len(idx) + 8, dtype=np.int32) % rows).to(dev)
    B.unip_gather_tokens(hid, idx2, torch.tensor([len(idx) + 100], dtype=torch.int32, device=dev),
                         big[: len(idx)])
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st & B.UNIP_DEV_BAD_INDEX, B.describe_status(st)
    assert np.array_equal(big[: len(idx)].view(torch.int16).cpu().numpy(), src[np.arange(len(idx)) % rows])
    assert bool((big[len(idx):] == 0).all())
