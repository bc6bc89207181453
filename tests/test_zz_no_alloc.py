"""The no-allocation attention entry point against the workspace entry point.

unip_prefill_attention_noalloc serves callers that cannot allocate device
memory (an operator interface that hands out only its tensors, a path that
must not risk the device synchronisation an allocation can cause).  It runs
the same planner and kernel as unip_prefill_attention, only with the plan in
the library's own scratch array, so its outputs must be bit for bit those of
unip_prefill_attention; one case is also held against the fp64 oracle.  This
file runs last so that a failure here never hides another test.  Each call
below goes through the C ABI.
"""
import ctypes

import numpy as np
import pytest

from sparsified_long_context_gb300 import workloads as W

from gpu_harness import LSE_ABS, assert_close, bf16_tensor_to_f64, oracle_attention_rows

torch = pytest.importorskip("torch")


def _device_inputs(wl):
    from sparsified_long_context_gb300.pipeline import DeviceInputs
    return DeviceInputs.from_workload(wl, "cuda", with_hidden=False)


def _outputs(wl):
    n = wl.num_tokens
    out = torch.full((n, wl.num_heads_q, wl.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((wl.num_heads_q, n), float("nan"), dtype=torch.float32, device="cuda")
    return out, lse


def _kw(wl, di):
    return dict(num_heads_q=wl.num_heads_q, num_heads_kv=wl.num_heads_kv, head_dim=wl.head_dim,
                k_cache=di.k_cache, v_cache=di.v_cache, block_table=di.block_table,
                page_size=wl.cache.page_size if wl.cache is not None else 16)


def _prefix_workload(seed):
    rng = np.random.default_rng(seed)
    P, n, hq, hkv, d, page = 700, 300, 8, 2, 128, 16
    k_all = W.f32_to_bf16_bits(rng.standard_normal((P + n, hkv, d), dtype=np.float32))
    v_all = W.f32_to_bf16_bits(rng.standard_normal((P + n, hkv, d), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((n, hq, d), dtype=np.float32))
    n_pages = -(-P // page)
    perm = rng.permutation(n_pages).astype(np.int32)
    kp = np.zeros((n_pages, page, hkv, d), np.uint16)
    vp = np.zeros_like(kp)
    for p in range(n_pages):
        a, b = p * page, min(P, (p + 1) * page)
        kp[perm[p], : b - a], vp[perm[p], : b - a] = k_all[a:b], v_all[a:b]
    return W.Workload("prefix", hq, hkv, d, np.array([0, n], np.int32), np.arange(P, P + n, dtype=np.int32), q,
                      k_all[P:], v_all[P:], cache=W.PagedCache(n_pages, page, hkv, d, "array", kp, vp),
                      block_table=perm[None, :])


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    from sparsified_long_context_gb300 import binding as B
    B.unip_get_device_status(clear=True)
    # two calls in a row on different problems: the shared scratch keeps the first call's plan
    for wl in (W.packed([37, 300, 1, 129], 8, 2, 128, seed=11), _prefix_workload(12)):
        di = _device_inputs(wl)
        ref_out, ref_lse = _outputs(wl)
        B.unip_prefill_attention(di.q, di.k, di.v, di.cu_seqlens, di.positions, ref_out, ref_lse, **_kw(wl, di))
        out, lse = _outputs(wl)
        B.unip_prefill_attention_noalloc(di.q, di.k, di.v, di.cu_seqlens, di.positions, out, lse, **_kw(wl, di))
        torch.cuda.synchronize()
        assert B.unip_get_device_status(clear=True) == 0
        assert torch.isfinite(out.float()).all()
        # the same plan and kernel: identical bits
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        if wl.cache is not None:   # the paged-prefix case, also against the oracle
            ref_o, ref_l = oracle_attention_rows(wl, None)
            assert_close(bf16_tensor_to_f64(out), ref_o, what="no-allocation out vs oracle")
            assert_close(lse.cpu().numpy().astype(np.float64).T, ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS,
                         what="no-allocation lse vs oracle")


def test_noalloc_rejects_problems_beyond_its_scratch():
    from sparsified_long_context_gb300 import binding as B
    lib = B.load()
    prm = B._params(32, 8, 128, 0.0)
    too_many_tokens = 128 * 32768
    rc = lib.unip_prefill_attention_noalloc(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                            ctypes.c_void_p(16), 1, ctypes.c_void_p(16), too_many_tokens, None,
                                            ctypes.byref(prm), ctypes.c_void_p(16), None, None)
    assert rc == -6
    assert "no-allocation" in lib.unip_status_string(rc).decode()
