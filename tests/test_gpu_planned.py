"""GPU parity of host-planned attention (unip_prefill_attention_planned) through the C ABI.

The plan is built on the host from the batch layout; calls with few work items also split the
key range of their query tiles over several items and merge the fp32 partials in key order.
Split and unsplit items are held against the fp64 oracle; an unsplit plan must give exactly
the bits of the device-planned entry point (the same items, each row's keys in the same order).
"""
import numpy as np
import pytest

import oracle
from sparsified_long_context_gb300 import workloads as W

from gpu_harness import LSE_ABS, assert_close, bf16_tensor_to_f64, oracle_attention_rows, sample_rows
from test_gpu_attention import _batch_with_prefixes, _chunk_with_prefix, _run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run_planned(wl, flags=0, reps=1):
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import (DeviceInputs, StepBuffers, attention_plan, plan_workspace,
                                                        run_attention_planned)
    B.unip_get_device_status(clear=True)
    di = DeviceInputs.from_workload(wl, "cuda", with_hidden=False)
    bufs = StepBuffers(di, block_size=wl.block_size or 64)
    plan = attention_plan(wl, flags)
    ws = plan_workspace(plan, "cuda")
    outs = []
    for _ in range(reps):
        bufs.out.fill_(float("nan"))
        bufs.lse.fill_(float("nan"))
        run_attention_planned(di, bufs, plan, ws)
        torch.cuda.synchronize()
        st = B.unip_get_device_status(clear=True)
        assert st == 0, B.describe_status(st)
        outs.append((bf16_tensor_to_f64(bufs.out), bufs.lse.cpu().numpy().astype(np.float64)))
    info = plan.info
    plan.close()
    return outs, info


def _check_oracle(wl, out, lse, rows=None):
    ref_o, ref_l = oracle_attention_rows(wl, rows)
    sel = slice(None) if rows is None else rows
    assert_close(out[sel], ref_o, what=f"{wl.name} out (planned)")
    assert_close(lse.T[sel], ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS, what=f"{wl.name} lse (planned)")


def _few_long_decodes(ctx, hq=32, hkv=8, d=128, page=16, seed=9):
    return _batch_with_prefixes(ctx, [1] * len(ctx), hq, hkv, d, page, seed)


_PLANNED_CASES = [
    lambda: _chunk_with_prefix(3584, 512, 32, 8, 128, 16, seed=41),   # the last chunk of 4096/512
    lambda: _chunk_with_prefix(1000, 257, 4, 2, 64, 64, seed=42),
    lambda: _chunk_with_prefix(4096, 130, 8, 1, 128, 128, seed=43),   # G 8
    lambda: _chunk_with_prefix(700, 300, 12, 2, 128, 32, seed=44),    # even G 6 (tokens of one head)
    lambda: _chunk_with_prefix(900, 77, 6, 2, 64, 16, seed=45),       # odd G 3
    lambda: _few_long_decodes([32768, 30000, 17, 32001]),            # four decodes, long contexts
    lambda: W.packed([37, 100, 64, 255], 4, 2, 64, seed=1),           # no prefix
    lambda: _batch_with_prefixes([1000, 17, 300, 2048, 5, 64, 129, 0], [1, 1, 2, 5, 33, 65, 1, 3],
                                 32, 8, 128, 16, seed=3328),
]
_PLANNED_IDS = ["chunk7_of_4096", "prefix1000_g2", "prefix4096_g8", "g6", "g3", "four_decodes", "tiny_packed",
                "decode_batch"]


@pytest.mark.parametrize("make", _PLANNED_CASES, ids=_PLANNED_IDS)
@pytest.mark.parametrize("splits", [0, 2, 5])
def test_planned_against_oracle(make, splits):
    """The plan's own choice (0), and every unit's key range forced into 2 or 5 items."""
    from sparsified_long_context_gb300 import binding as B
    wl = make()
    (res,), info = _run_planned(wl, flags=B.UNIP_PLAN_SPLITS(splits) if splits else 0)
    assert info["host"]
    if splits:
        assert info["split_units"] > 0, info
    rows = None if wl.num_tokens <= 600 else sample_rows(wl, 200)
    _check_oracle(wl, res[0], res[1], rows)


def test_few_long_decodes_are_split_by_the_cost_model():
    (res,), info = _run_planned(_few_long_decodes([20000, 9000, 31000]))
    assert info["split_units"] > 0


@pytest.mark.parametrize("make", [
    lambda: _chunk_with_prefix(3584, 512, 32, 8, 128, 16, seed=41),
    lambda: _few_long_decodes([20000, 9000, 31000]),
    lambda: _batch_with_prefixes([1000, 17, 300, 2048, 5, 64, 129, 0], [1, 1, 2, 5, 33, 65, 1, 3],
                                 32, 8, 128, 16, seed=3328),
], ids=["chunk", "decodes", "decode_batch"])
def test_split_merge_is_deterministic_and_close_to_unsplit(make):
    """Two runs of a split plan give identical bits (the merge order is fixed, whichever split finishes
    last); the split result stays within the tolerance of the unsplit one."""
    from sparsified_long_context_gb300 import binding as B
    wl = make()
    (r1, r2), info = _run_planned(wl, flags=B.UNIP_PLAN_SPLITS(3), reps=2)
    assert info["split_units"] > 0
    assert np.array_equal(r1[0], r2[0]) and np.array_equal(r1[1], r2[1])
    (u,), info_u = _run_planned(wl, flags=B.UNIP_PLAN_NO_SPLIT)
    assert info_u["split_units"] == 0
    assert_close(r1[0], u[0], what="split vs unsplit out")
    assert_close(r1[1], u[1], max_abs=LSE_ABS, mean_abs=LSE_ABS, what="split vs unsplit lse")


@pytest.mark.parametrize("make", [
    lambda: W.packed([0, 300, 0, 5], 8, 2, 128, seed=313),
    lambda: W.packed([1000], 8, 1, 64, seed=1073),
    lambda: W.packed([5, 70, 131], 12, 2, 64, seed=282),
    lambda: W.packed([9, 130], 6, 2, 128, seed=139),
    lambda: _chunk_with_prefix(513, 512, 4, 2, 128, 16, seed=1025),
    lambda: _batch_with_prefixes([1000, 17, 300, 2048, 5, 64, 129, 0], [1, 1, 2, 5, 33, 65, 1, 3],
                                 32, 8, 128, 16, seed=3328),
], ids=["g4", "g8", "g6", "g3", "chunk", "decode_batch"])
def test_unsplit_plan_is_bit_identical_to_device_planner(make):
    """A host plan without splits and the device planner make the same units (each row's keys in the same
    order), so the outputs agree bit for bit; the device fallback of a plan too."""
    from sparsified_long_context_gb300 import binding as B
    wl = make()
    ref_o, ref_l = _run(wl)
    (u,), info = _run_planned(wl, flags=B.UNIP_PLAN_NO_SPLIT)
    assert info["host"] and info["split_units"] == 0
    assert np.array_equal(u[0], ref_o) and np.array_equal(u[1], ref_l)
    (d,), info_d = _run_planned(wl, flags=B.UNIP_PLAN_DEVICE)
    assert not info_d["host"]
    assert np.array_equal(d[0], ref_o) and np.array_equal(d[1], ref_l)


def test_planned_chunked_equals_one_shot():
    """The 4096-token prompt in eight planned 512-token calls behind its paged prefix ([CP]: chunked
    prefill reproduces one-pass prefill), against the one-shot call and the oracle."""
    one, chunks = W.chunked()
    outs, infos = [], []
    for wl in chunks:
        (r,), info = _run_planned(wl)
        outs.append(r[0])
        infos.append(info)
    chunked = np.concatenate(outs, 0)
    full, _ = _run(one)
    assert_close(chunked, full, what="planned chunks vs one-shot")
    rows = sample_rows(one, 160)
    ref, _ = oracle.attention(one.q, one.k, one.v, one.cu_seqlens, one.positions, 32, 8, 128, rows=rows)
    assert_close(chunked[rows], ref, what="planned chunks vs oracle")


def test_planned_compacted_stream():
    """A compacted stream (kept tokens with gaps, explicit prefix lengths) through a host plan."""
    from sparsified_long_context_gb300 import binding as B
    from test_gpu_attention import _compact
    wl = _batch_with_prefixes([3000, 17, 300, 2048, 0, 64], [900, 1, 130, 65, 300, 3], 32, 8, 128, 16, seed=77)
    rng = np.random.default_rng(5)
    q, k, v, cu_k, pos_k, plen = _compact(wl, 16, rng, 0.5)
    n = int(cu_k[-1])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kct, vct = wl.cache.to_torch("cuda")
    plan = B.AttentionPlan(cu_k, plen, num_heads_q=32, num_heads_kv=8, head_dim=128, page_size=16,
                           max_pages_per_seq=wl.block_table.shape[1], flags=B.UNIP_PLAN_SPLITS(3))
    assert plan.info["host"] and plan.info["split_units"] > 0
    out = torch.empty((n, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((32, n), dtype=torch.float32, device="cuda")
    B.unip_get_device_status(clear=True)
    plan.run(dev(q).view(torch.bfloat16), dev(k).view(torch.bfloat16), dev(v).view(torch.bfloat16), out, lse,
             k_cache=kct, v_cache=vct, block_table=dev(wl.block_table), page_size=16)
    torch.cuda.synchronize()
    assert B.unip_get_device_status(clear=True) == 0
    kc, vc = wl.cache.pages_numpy(np.arange(wl.cache.num_pages))
    ref_o, ref_l = oracle.attention(q, k, v, cu_k, pos_k, 32, 8, 128, prefix_lens=plen, k_cache=kc, v_cache=vc,
                                    block_table=wl.block_table, page_size=16)
    assert_close(bf16_tensor_to_f64(out), ref_o, what="planned compacted out")
    assert_close(lse.cpu().numpy().astype(np.float64).T, ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS,
                 what="planned compacted lse")
    plan.close()


def test_plan_reused_across_workspaces_and_calls():
    """One plan run on two workspaces alternately (each cleared at its first use) and repeatedly: every
    run gives the same bits."""
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import (DeviceInputs, StepBuffers, attention_plan, plan_workspace,
                                                        run_attention_planned)
    wl = _chunk_with_prefix(2048, 384, 32, 8, 128, 16, seed=88)
    di = DeviceInputs.from_workload(wl, "cuda", with_hidden=False)
    bufs = StepBuffers(di)
    plan = attention_plan(wl, B.UNIP_PLAN_SPLITS(4))
    assert plan.info["split_units"] > 0
    ws = [plan_workspace(plan, "cuda"), plan_workspace(plan, "cuda")]
    ws[1].fill_(0xAB)   # stale bytes in the ticket area must not matter
    res = []
    for i in range(5):
        run_attention_planned(di, bufs, plan, ws[i % 2])
        torch.cuda.synchronize()
        res.append(bufs.out.clone())
    assert B.unip_get_device_status(clear=True) == 0
    for r in res[1:]:
        assert torch.equal(r.view(torch.int16), res[0].view(torch.int16))
    plan.close()


def test_split_items_repeated_without_timeouts():
    """Split items whose merge keeps some warps of a tile busy while one-tile items follow: 200 runs of a
    compacted stream with forced splits (2 to 5) must never trip a bounded device wait, and every run
    gives the bits of the first run with the same split count."""
    from sparsified_long_context_gb300 import binding as B
    from test_gpu_attention import _compact
    wl = _batch_with_prefixes([3000, 17, 300, 2048, 0, 64], [900, 1, 130, 65, 300, 3], 32, 8, 128, 16, seed=77)
    q, k, v, cu_k, pos_k, plen = _compact(wl, 16, np.random.default_rng(5), 0.5)
    n = int(cu_k[-1])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    qd, kd, vd = dev(q).view(torch.bfloat16), dev(k).view(torch.bfloat16), dev(v).view(torch.bfloat16)
    kct, vct = wl.cache.to_torch("cuda")
    bt = dev(wl.block_table)
    plans = {s: B.AttentionPlan(cu_k, plen, num_heads_q=32, num_heads_kv=8, head_dim=128, page_size=16,
                                max_pages_per_seq=wl.block_table.shape[1], flags=B.UNIP_PLAN_SPLITS(s))
             for s in (2, 3, 4, 5)}
    ws = {s: torch.empty(max(p.workspace_bytes, 256), dtype=torch.uint8, device="cuda") for s, p in plans.items()}
    out = torch.empty((n, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((32, n), dtype=torch.float32, device="cuda")
    first = {}
    B.unip_get_device_status(clear=True)
    for it in range(200):
        s = 2 + it % 4
        plans[s].run(qd, kd, vd, out, lse, k_cache=kct, v_cache=vct, block_table=bt, page_size=16,
                     workspace=ws[s])
        if it % 20 == 19 or it < 4:
            torch.cuda.synchronize()
            st = B.unip_get_device_status(clear=True)
            assert st == 0, (it, B.describe_status(st))
            if s not in first:
                first[s] = out.clone()
            else:
                assert torch.equal(out.view(torch.int16), first[s].view(torch.int16)), it
    for p in plans.values():
        p.close()
