"""GPU parity of block importance, Top-p selection, index build and gather.

Importance is compared with the oracle within the attention tolerance;
selection, indices and gathered rows are compared bit for bit with the oracle
fed the GPU's own fp32 scores.
"""
import numpy as np
import pytest

import oracle
from sparsified_long_context_gb300 import workloads as W

from gpu_harness import LSE_ABS, assert_close, library_ffd, oracle_attention_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _step(wl):
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import DeviceInputs, StepBuffers, run_step
    B.unip_get_device_status(clear=True)
    di = DeviceInputs.from_workload(wl, "cuda")
    bufs = StepBuffers(di)
    run_step(di, bufs)
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st == 0, B.describe_status(st)
    return di, bufs


def _check_selection(wl, bufs, flags=oracle.KEEP_FIRST | oracle.KEEP_LAST):
    blk_cu = bufs.blk_cu.cpu().numpy()
    nblk = int(blk_cu[-1])
    imp = bufs.imp[:nblk].cpu().numpy()
    keep = bufs.keep[:nblk].cpu().numpy()
    ref_keep = oracle.topp_select(imp, blk_cu, wl.top_p, flags)
    assert np.array_equal(keep, ref_keep)
    gi, ck, pk, m = oracle.index_build(ref_keep, blk_cu, wl.cu_seqlens, wl.positions, wl.block_size)
    n_kept = int(bufs.n_kept.cpu().item())
    assert n_kept == m
    assert np.array_equal(bufs.cu_seqlens_kept.cpu().numpy(), ck)
    assert np.array_equal(bufs.gather_idx[:m].cpu().numpy(), gi)
    assert np.array_equal(bufs.positions_kept[:m].cpu().numpy(), pk)
    if wl.hidden is not None:
        ref_h = oracle.gather(wl.hidden, gi)
        got = bufs.hidden_out[:m].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, ref_h)
    return imp, blk_cu, m


def test_tiny_full_chain():
    wl = W.tiny_packed()
    di, bufs = _step(wl)
    _, lse = oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, 4, 2, 64)
    ref_imp, ref_bc = oracle.block_importance(wl.q, wl.k, lse, wl.cu_seqlens, 4, 2, 64, wl.block_size,
                                              seg_mask=wl.seg_mask)
    imp, blk_cu, m = _check_selection(wl, bufs)
    assert np.array_equal(blk_cu, ref_bc)
    assert_close(imp.astype(np.float64), ref_imp, what="importance")
    assert 0 < m <= wl.num_tokens


def _window_rows(wl):
    """Token rows of every scored segment's scoring window: its last min(B, n) rows."""
    cu, B_ = wl.cu_seqlens, wl.block_size
    rows = []
    for s in range(wl.num_segs):
        a, b = int(cu[s]), int(cu[s + 1])
        if b > a and (wl.seg_mask is None or wl.seg_mask[s]):
            rows.extend(range(b - min(B_, b - a), b))
    return np.array(rows, np.int32)


def _importance_vs_oracle(wl, bufs):
    """Importance against the oracle computed from the oracle's own inputs only: the window rows'
    LSE comes from the oracle's attention over those rows (prefix pages included), never from the
    GPU.  The GPU's LSE of the same rows is checked against it on the way."""
    rows = _window_rows(wl)
    _, lse_rows = oracle_attention_rows(wl, rows)           # [R, H_q]
    lse_gpu = bufs.lse.cpu().numpy().astype(np.float64).T    # [N, H_q]
    assert_close(lse_gpu[rows], lse_rows, max_abs=LSE_ABS, mean_abs=LSE_ABS, what="window-row lse")
    lse_full = np.zeros((wl.num_tokens, wl.num_heads_q), np.float64)   # only window rows are read
    lse_full[rows] = lse_rows
    ref_imp, ref_bc = oracle.block_importance(wl.q, wl.k, lse_full, wl.cu_seqlens, wl.num_heads_q,
                                              wl.num_heads_kv, wl.head_dim, wl.block_size, seg_mask=wl.seg_mask)
    blk_cu = bufs.blk_cu.cpu().numpy()
    assert np.array_equal(blk_cu, ref_bc)
    imp = bufs.imp[: int(blk_cu[-1])].cpu().numpy().astype(np.float64)
    assert_close(imp, ref_imp, what="importance")
    for s in range(wl.num_segs):
        a, b = blk_cu[s], blk_cu[s + 1]
        if b > a:
            assert abs(imp[a:b].sum() - 1.0) < 1e-4


def test_long_single_chain():
    wl = W.long_single()
    di, bufs = _step(wl)
    _importance_vs_oracle(wl, bufs)
    _, _, m = _check_selection(wl, bufs)
    assert 0 < m < wl.num_tokens


def test_mixed_step_chain():
    wl = W.mixed_step()
    di, bufs = _step(wl)
    _importance_vs_oracle(wl, bufs)
    _, _, m = _check_selection(wl, bufs)
    assert m >= 256  # decode tokens are never dropped


def test_prepacked_chain():
    """The prepacked batch (64 prompts, every one scored): importance of all 64 segments against the
    oracle, then selection and indices bit-exact."""
    wl = W.prepacked(library_ffd)
    di, bufs = _step(wl)
    _importance_vs_oracle(wl, bufs)
    _, _, m = _check_selection(wl, bufs)
    assert 0 < m < wl.num_tokens


def _topp_direct(imp_np, blk_cu_np, cu_np, B_, p, flags):
    from sparsified_long_context_gb300 import binding as Bd
    dev = "cuda"
    n = int(cu_np[-1])
    S = len(cu_np) - 1
    pos = np.concatenate([np.arange(cu_np[s + 1] - cu_np[s]) for s in range(S)]).astype(np.int32)
    cap = Bd.unip_importance_capacity(n, S, B_)
    imp_t = torch.zeros(cap, dtype=torch.float32, device=dev)
    imp_t[: len(imp_np)] = torch.from_numpy(imp_np)
    keep = torch.full((cap,), 7, dtype=torch.uint8, device=dev)
    gi = torch.full((n,), -1, dtype=torch.int32, device=dev)
    pk = torch.full((n,), -1, dtype=torch.int32, device=dev)
    ck = torch.empty(S + 1, dtype=torch.int32, device=dev)
    nk = torch.empty(1, dtype=torch.int32, device=dev)
    Bd.unip_topp_select(imp_t, torch.from_numpy(blk_cu_np).to(dev), torch.from_numpy(cu_np).to(dev),
                        torch.from_numpy(pos).to(dev), keep, gi, ck, pk, nk, block_size=B_, p=p, flags=flags)
    torch.cuda.synchronize()
    m = int(nk.item())
    return keep[: len(imp_np)].cpu().numpy(), gi[:m].cpu().numpy(), ck.cpu().numpy(), pk[:m].cpu().numpy(), pos


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_topp_edge_cases_bit_exact(flags):
    rng = np.random.default_rng(50 + flags)
    B_ = 16
    lengths = [1, 16, 17, 300, 0, 5000, 64, 33, 20000]   # 20000 tokens = 1250 blocks: the sorting path
    scored = [1, 1, 1, 1, 1, 1, 0, 1, 1]
    nbs = [(-(-L // B_) if (sc and L > 0) else 0) for L, sc in zip(lengths, scored)]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    bc = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    parts = []
    for s, nb in enumerate(nbs):
        if nb == 0:
            continue
        kind = s % 3
        if kind == 0:
            x = rng.random(nb) ** 4
        elif kind == 1:
            x = np.round(rng.random(nb) * 3) + 1.0    # many exact ties
        else:
            x = np.zeros(nb)
            x[rng.integers(0, nb)] = 1.0
        x = (x / x.sum()).astype(np.float32)
        parts.append(x)
    imp = np.concatenate(parts).astype(np.float32)
    for p in (0.0, 0.5, 0.9, 0.95, 1.0):
        keep, gi, ck, pk, pos = _topp_direct(imp, bc, cu, B_, p, flags)
        ref = oracle.topp_select(imp, bc, p, flags)
        assert np.array_equal(keep, ref), (p, flags)
        rgi, rck, rpk, rm = oracle.index_build(ref, bc, cu, pos, B_)
        assert np.array_equal(gi, rgi) and np.array_equal(ck, rck) and np.array_equal(pk, rpk)


@pytest.mark.parametrize("nb", [13, 32, 40])   # one-warp path (up to 32 blocks) and the CTA path
def test_topp_negative_zero_scores(nb):
    """-0 scores through the public Top-p call: read as zero (mass and rank), like the oracle."""
    rng = np.random.default_rng(77 + nb)
    x = rng.random(nb).astype(np.float32)
    x[::5] = 0.0
    x = (x / x.sum()).astype(np.float32)
    x[::5] = np.float32(-0.0)
    bc = np.array([0, nb], np.int32)
    cu = np.array([0, nb * 16], np.int32)
    for p, flags in [(0.5, 0), (0.9, 3), (1.0, 0), (1.0, 3)]:
        keep, gi, ck, pk, pos = _topp_direct(x, bc, cu, 16, p, flags)
        assert np.array_equal(keep, oracle.topp_select(x, bc, p, flags)), (p, flags)


@pytest.mark.parametrize("bad", [np.nan, -0.25, 1.5])
def test_topp_invalid_scores_raise_status(bad):
    """A score outside [0, 1] (or NaN) in a segment of either selection path raises the bad-scores bit
    and that segment keeps nothing; a valid segment in the same call is still selected exactly."""
    rng = np.random.default_rng(11)
    B_ = 16
    nbs = [5, 40, 8]                       # one-warp path, CTA path, one-warp path
    parts = []
    for nb in nbs:
        x = rng.random(nb)
        parts.append((x / x.sum()).astype(np.float32))
    from sparsified_long_context_gb300 import binding as B
    parts[0][2] = bad
    parts[1][7] = bad
    imp = np.concatenate(parts).astype(np.float32)
    bc = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    cu = (bc * B_).astype(np.int32)
    B.unip_get_device_status(clear=True)
    keep, gi, ck, pk, pos = _topp_direct(imp, bc, cu, B_, 0.9, 0)
    st = B.unip_get_device_status(clear=True)
    assert st & 0x10, B.describe_status(st)                  # UNIP_DEV_BAD_SCORES
    assert ck[1] - ck[0] == 0 and ck[2] - ck[1] == 0         # the two invalid segments keep nothing
    good = parts[2]
    ref = oracle.topp_select(good, np.array([0, len(good)], np.int32), 0.9, 0)
    assert np.array_equal(keep[bc[2]:bc[3]], ref)
    assert ck[3] - ck[2] == int(ref.sum()) * B_


def test_topp_zero_mass_keeps_all():
    imp = np.zeros(4, np.float32)
    keep, gi, ck, pk, pos = _topp_direct(imp, np.array([0, 4], np.int32), np.array([0, 50], np.int32), 16, 0.5, 3)
    assert keep.tolist() == [1, 1, 1, 1] and len(gi) == 50


@pytest.mark.parametrize("n_rows,d,extra", [(37, 8, 0), (1000, 256, 0), (3000, 4096, 0), (64, 512, 64)])
def test_gather_bit_exact_and_strides(n_rows, d, extra):
    from sparsified_long_context_gb300 import binding as Bd
    rng = np.random.default_rng(n_rows + d)
    hid = W.f32_to_bf16_bits(rng.standard_normal((n_rows, d + extra), dtype=np.float32))
    idx = np.sort(rng.choice(n_rows, n_rows // 2 + 1, replace=False)).astype(np.int32)
    h_t = torch.from_numpy(hid).view(torch.bfloat16).cuda()[:, :d]
    cap = n_rows
    out = torch.zeros((cap, d + extra), dtype=torch.bfloat16, device="cuda")[:, :d]
    gi = torch.zeros(cap, dtype=torch.int32, device="cuda")
    gi[: len(idx)] = torch.from_numpy(idx).cuda()
    nk = torch.tensor([len(idx)], dtype=torch.int32, device="cuda")
    lib = Bd.load()
    rc = lib.unip_gather_tokens(h_t.data_ptr(), n_rows, h_t.stride(0), d, gi.data_ptr(), nk.data_ptr(), cap,
                                out.data_ptr(), out.stride(0), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    got = out[: len(idx)].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.gather(np.ascontiguousarray(hid[:, :d]), idx))
    assert Bd.unip_get_device_status() == 0


@pytest.mark.parametrize("lengths,hq,hkv,d,B", [
    ([37, 100, 64, 255], 4, 2, 64, 16), ([5, 130, 300], 8, 2, 128, 32), ([1000, 64], 4, 1, 64, 128),
    ([7, 260], 8, 8, 128, 64), ([513], 16, 2, 128, 64), ([129, 1, 0, 40], 2, 1, 128, 16)])
def test_importance_shapes_vs_oracle(lengths, hq, hkv, d, B):
    from sparsified_long_context_gb300 import binding as Bd
    from sparsified_long_context_gb300.pipeline import DeviceInputs, StepBuffers, run_attention, run_importance
    wl = W.packed(lengths, hq, hkv, d, seed=sum(lengths) + B, block_size=B, top_p=0.9)
    Bd.unip_get_device_status(clear=True)
    di = DeviceInputs.from_workload(wl, "cuda", with_hidden=False)
    bufs = StepBuffers(di, block_size=B)
    run_attention(di, bufs)
    run_importance(di, bufs)
    torch.cuda.synchronize()
    assert Bd.unip_get_device_status() == 0
    _, lse = oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, hq, hkv, d)
    ref_imp, ref_bc = oracle.block_importance(wl.q, wl.k, lse, wl.cu_seqlens, hq, hkv, d, B, seg_mask=wl.seg_mask)
    blk_cu = bufs.blk_cu.cpu().numpy()
    assert np.array_equal(blk_cu, ref_bc)
    imp = bufs.imp[: blk_cu[-1]].cpu().numpy().astype(np.float64)
    assert_close(imp, ref_imp, what="importance")


@pytest.mark.parametrize("name", ["tiny_packed", "long_single", "mixed_step", "prepacked"])
def test_fused_select_gather_matches_oracle(name):
    """unip_select_gather against the oracle fed the same scores (and so against the two-call path)."""
    from sparsified_long_context_gb300 import binding as Bd
    from sparsified_long_context_gb300.pipeline import (DeviceInputs, StepBuffers, run_attention, run_importance,
                                                        run_select_gather)
    wl = W.prepacked(library_ffd) if name == "prepacked" else W.workload_by_name(name)
    Bd.unip_get_device_status(clear=True)
    di = DeviceInputs.from_workload(wl, "cuda")
    bufs = StepBuffers(di)
    run_attention(di, bufs)
    run_importance(di, bufs)
    if bufs.hidden_out is not None:
        bufs.hidden_out.zero_()
    run_select_gather(di, bufs)
    torch.cuda.synchronize()
    assert Bd.unip_get_device_status(clear=True) == 0
    _check_selection(wl, bufs)


@pytest.mark.parametrize("L,B_,with_hidden", [(1, 16, True), (300 * 16 - 5, 16, True), (1000 * 16, 16, False),
                                              (1250 * 16 - 3, 16, True), (777, 64, False)])
def test_single_segment_one_launch_path(L, B_, with_hidden):
    """unip_select_gather with one segment (the one-launch path): every sort regime of the selection,
    with and without hidden rows, bit-exact against the oracle fed the same scores."""
    from sparsified_long_context_gb300 import binding as Bd
    rng = np.random.default_rng(L + B_)
    nb = -(-L // B_)
    x = rng.random(nb) ** 6
    x[rng.integers(0, nb, max(1, nb // 10))] = 0.0          # zero-mass blocks
    x[: nb // 3] = np.round(x[: nb // 3] * 8) / 8 + 1e-3     # many exact ties
    if x.sum() == 0:
        x[0] = 1.0
    imp = (x / x.sum()).astype(np.float32)
    cu = np.array([0, L], np.int32)
    bc = np.array([0, nb], np.int32)
    pos = np.arange(7, 7 + L, dtype=np.int32)                # positions past a 7-token prefix
    d = 64
    hid = W.f32_to_bf16_bits(rng.standard_normal((L, d), dtype=np.float32))
    dev = "cuda"
    cap = Bd.unip_importance_capacity(L, 1, B_)
    imp_t = torch.zeros(cap, dtype=torch.float32, device=dev)
    imp_t[:nb] = torch.from_numpy(imp)
    for p, flags in [(0.0, 3), (0.5, 1), (0.95, 3), (1.0, 0), (0.9, 2)]:
        keep = torch.full((cap,), 9, dtype=torch.uint8, device=dev)
        gi = torch.full((L,), -1, dtype=torch.int32, device=dev)
        pk = torch.full((L,), -1, dtype=torch.int32, device=dev)
        ck = torch.empty(2, dtype=torch.int32, device=dev)
        nk = torch.empty(1, dtype=torch.int32, device=dev)
        h_t = torch.from_numpy(hid).view(torch.bfloat16).to(dev) if with_hidden else None
        out = torch.zeros((L, d), dtype=torch.bfloat16, device=dev) if with_hidden else None
        Bd.unip_get_device_status(clear=True)
        Bd.unip_select_gather(imp_t, torch.from_numpy(bc).to(dev), torch.from_numpy(cu).to(dev),
                              torch.from_numpy(pos).to(dev), keep, gi, ck, pk, nk, h_t, out, block_size=B_, p=p,
                              flags=flags)
        torch.cuda.synchronize()
        assert Bd.unip_get_device_status(clear=True) == 0
        ref = oracle.topp_select(imp, bc, p, flags)
        assert np.array_equal(keep[:nb].cpu().numpy(), ref), (L, p, flags)
        rgi, rck, rpk, rm = oracle.index_build(ref, bc, cu, pos, B_)
        m = int(nk.item())
        assert m == rm and np.array_equal(ck.cpu().numpy(), rck)
        assert np.array_equal(gi[:m].cpu().numpy(), rgi) and np.array_equal(pk[:m].cpu().numpy(), rpk)
        if with_hidden:
            got = out[:m].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, oracle.gather(hid, rgi))


def test_single_unscored_segment_keeps_everything():
    from sparsified_long_context_gb300 import binding as Bd
    L, B_ = 333, 64
    dev = "cuda"
    cap = Bd.unip_importance_capacity(L, 1, B_)
    imp_t = torch.zeros(cap, dtype=torch.float32, device=dev)
    keep = torch.zeros(cap, dtype=torch.uint8, device=dev)
    gi = torch.full((L,), -1, dtype=torch.int32, device=dev)
    pk = torch.full((L,), -1, dtype=torch.int32, device=dev)
    ck = torch.empty(2, dtype=torch.int32, device=dev)
    nk = torch.empty(1, dtype=torch.int32, device=dev)
    pos = torch.arange(L, dtype=torch.int32, device=dev)
    Bd.unip_select_gather(imp_t, torch.tensor([0, 0], dtype=torch.int32, device=dev),
                          torch.tensor([0, L], dtype=torch.int32, device=dev), pos, keep, gi, ck, pk, nk, None, None,
                          block_size=B_, p=0.5)
    torch.cuda.synchronize()
    assert Bd.unip_get_device_status(clear=True) == 0
    assert int(nk.item()) == L and ck.cpu().tolist() == [0, L]
    assert np.array_equal(gi.cpu().numpy(), np.arange(L)) and np.array_equal(pk.cpu().numpy(), np.arange(L))


@pytest.mark.parametrize("S", [11999, 12500])
def test_select_gather_many_segments(S):
    """unip_select_gather on either side of the segment count where the kept-token offsets stop fitting
    in shared memory (12000: the call switches to Top-p + index + gather as separate grids): masks,
    indices, kept offsets, kept positions and gathered rows bit-exact against the oracle."""
    from sparsified_long_context_gb300 import binding as Bd
    rng = np.random.default_rng(S)
    B_, d = 16, 64
    lengths = rng.integers(0, 120, S)
    lengths[rng.random(S) < 0.05] = 1
    scored = rng.random(S) > 0.1                       # some segments are not scored (decode-like)
    nbs = np.where(scored & (lengths > 0), -(-lengths // B_), 0)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    bc = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    parts = []
    for nb in nbs:
        if nb:
            x = rng.random(nb) ** 3
            parts.append((x / x.sum()).astype(np.float32))
    imp = np.concatenate(parts).astype(np.float32)
    n = int(cu[-1])
    pos = np.concatenate([np.arange(L) + (7 if s % 3 == 0 else 0) for s, L in enumerate(lengths)]).astype(np.int32)
    hid = W.f32_to_bf16_bits(rng.standard_normal((n, d), dtype=np.float32))
    dev = "cuda"
    cap = Bd.unip_importance_capacity(n, S, B_)
    imp_t = torch.zeros(cap, dtype=torch.float32, device=dev)
    imp_t[: len(imp)] = torch.from_numpy(imp)
    keep = torch.full((cap,), 7, dtype=torch.uint8, device=dev)
    gi = torch.full((n,), -1, dtype=torch.int32, device=dev)
    pk = torch.full((n,), -1, dtype=torch.int32, device=dev)
    ck = torch.empty(S + 1, dtype=torch.int32, device=dev)
    nk = torch.empty(1, dtype=torch.int32, device=dev)
    h_t = torch.from_numpy(hid).view(torch.bfloat16).to(dev)
    out = torch.zeros_like(h_t)
    Bd.unip_get_device_status(clear=True)
    Bd.unip_select_gather(imp_t, torch.from_numpy(bc).to(dev), torch.from_numpy(cu).to(dev),
                          torch.from_numpy(pos).to(dev), keep, gi, ck, pk, nk, h_t, out, block_size=B_, p=0.9)
    torch.cuda.synchronize()
    st = Bd.unip_get_device_status(clear=True)
    assert st == 0, Bd.describe_status(st)
    ref = oracle.topp_select(imp, bc, 0.9)
    assert np.array_equal(keep[: len(imp)].cpu().numpy(), ref)
    rgi, rck, rpk, rm = oracle.index_build(ref, bc, cu, pos, B_)
    m = int(nk.item())
    assert m == rm
    assert np.array_equal(gi[:m].cpu().numpy(), rgi) and np.array_equal(ck.cpu().numpy(), rck)
    assert np.array_equal(pk[:m].cpu().numpy(), rpk)
    got = out[:m].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.gather(hid, rgi))


def _fused_vs_separate(wl, flags=oracle.KEEP_FIRST | oracle.KEEP_LAST):
    from sparsified_long_context_gb300 import binding as Bd
    from sparsified_long_context_gb300.pipeline import (DeviceInputs, StepBuffers, run_attention, run_importance,
                                                        run_importance_select_gather, run_select_gather)
    Bd.unip_get_device_status(clear=True)
    di = DeviceInputs.from_workload(wl, "cuda")
    bufs = StepBuffers(di)
    run_attention(di, bufs)
    run_importance(di, bufs)
    run_select_gather(di, bufs, flags=flags)
    torch.cuda.synchronize()
    assert Bd.unip_get_device_status(clear=True) == 0
    names = ["imp", "blk_cu", "keep", "gather_idx", "cu_seqlens_kept", "positions_kept", "n_kept"]
    if bufs.hidden_out is not None:
        names.append("hidden_out")
    ref = {n: getattr(bufs, n).clone() for n in names}
    for n in names:   # poison every output, so the fused call must write each one
        t = getattr(bufs, n)
        t.view(torch.uint8).fill_(0xA5)
    run_importance_select_gather(di, bufs, flags=flags)
    torch.cuda.synchronize()
    st = Bd.unip_get_device_status(clear=True)
    assert st == 0, Bd.describe_status(st)
    n_blk = int(ref["blk_cu"][-1].item())
    m = int(ref["n_kept"].item())
    lim = {"imp": n_blk, "keep": n_blk, "gather_idx": m, "positions_kept": m, "hidden_out": m}
    for n in names:
        a, b = getattr(bufs, n), ref[n]
        if n in lim:
            a, b = a[: lim[n]], b[: lim[n]]
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), n
    return bufs


@pytest.mark.parametrize("name", ["tiny_packed", "long_single", "mixed_step", "prepacked"])
def test_fused_importance_select_gather_matches_the_separate_calls(name):
    """unip_importance_select_gather: the bits of unip_block_importance + unip_select_gather (scores, keep
    mask, indices, kept offsets and positions, compacted rows), and bit-exact against the oracle fed its
    scores."""
    wl = W.prepacked(library_ffd) if name == "prepacked" else W.workload_by_name(name)
    bufs = _fused_vs_separate(wl)
    _check_selection(wl, bufs)


@pytest.mark.parametrize("L,B_,p,d_model,flags", [
    (1, 16, 0.9, 64, 3),         # one token, one block
    (63, 64, 0.5, 64, 0),        # one partial block, no forced blocks
    (65, 64, 0.99, 64, 1),       # a full block and a one-token block
    (1500, 64, 0.9, 256, 3),     # 24 blocks
    (5000, 16, 0.8, 0, 0),       # 313 blocks, register network; selection and indices only
    (8192 - 37, 16, 0.95, 128, 1),  # 510 blocks
    (12000, 16, 0.95, 128, 2),   # 750 blocks: ranks by counting
    (40000 + 5, 16, 0.9, 64, 3),  # 2501 blocks: shared-memory network, ragged last block
])
def test_fused_single_segment_matches_the_separate_calls(L, B_, p, d_model, flags):
    """One segment in the fused call: every CTA of one grid normalises the block masses, selects and
    copies its share of the rows.  Scores, keep mask, indices and rows must have the bits of the separate
    calls and match the oracle's selection on those scores, for every flag combination."""
    wl = W.packed([L], 4, 2, 64, seed=90 + L % 97, block_size=B_, top_p=p, d_model=d_model)
    bufs = _fused_vs_separate(wl, flags)
    _check_selection(wl, bufs, flags)


def test_fused_single_unscored_segment_keeps_everything():
    """One segment that is not scored: the fused call scores nothing and keeps every token and row."""
    wl = W.packed([333], 4, 2, 64, seed=91, block_size=64, top_p=0.5, d_model=64)
    wl.seg_mask = np.array([0], np.uint8)
    bufs = _fused_vs_separate(wl)
    _check_selection(wl, bufs)
    assert int(bufs.n_kept.item()) == 333


def test_fused_path_with_unscored_and_empty_segments():
    wl = W.packed([0, 300, 1, 0, 700, 64, 17], 8, 2, 128, seed=61, block_size=32, top_p=0.8, d_model=512)
    wl.seg_mask = np.array([1, 1, 0, 1, 0, 1, 1], np.uint8)
    bufs = _fused_vs_separate(wl)
    _check_selection(wl, bufs)


def test_launches_with_growing_and_shrinking_shared_memory():
    """The compaction's shared memory grows with the number of segments and blocks: a large call after a
    smaller one must still launch (a kernel's shared-memory limit is only ever raised)."""
    from sparsified_long_context_gb300.pipeline import (DeviceInputs, StepBuffers, run_attention, run_importance,
                                                        run_select_gather)
    big = W.packed([20] * 300, 4, 2, 64, seed=71, block_size=16, top_p=0.9, d_model=256)
    small = W.packed([500, 300], 4, 2, 64, seed=72, block_size=16, top_p=0.9, d_model=256)
    for wl in (big, small, big):
        di = DeviceInputs.from_workload(wl, "cuda")
        bufs = StepBuffers(di)
        run_attention(di, bufs)
        run_importance(di, bufs)
        run_select_gather(di, bufs)
        torch.cuda.synchronize()
        _check_selection(wl, bufs)
