"""Guard bands around every output of the path: each output buffer sits
between two bands filled with a bit pattern, and after the calls the bands
must be untouched (a stand-in for a memory checker: an out-of-range write by a
kernel shows up here), while the outputs still match the oracle."""
import numpy as np
import pytest

import oracle
from sparsified_long_context_gb300 import workloads as W

from gpu_harness import assert_close, bf16_tensor_to_f64, oracle_attention_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 8192  # elements before and after each output
_INT = {torch.bfloat16: torch.int16, torch.float32: torch.int32, torch.int32: torch.int32, torch.uint8: torch.uint8}
_FILL = {torch.int16: 0x5A5A, torch.int32: 0x5A5A5A5A, torch.uint8: 0xA5}


class Banded:
    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.n, self.dtype = n, dtype
        self.full = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        it = _INT[dtype]
        self.full.view(it).fill_(_FILL[it])
        self.t = self.full[GUARD:GUARD + n].view(*shape)

    def intact(self):
        raw = self.full.view(_INT[self.dtype])
        fill = _FILL[_INT[self.dtype]]
        return bool(torch.all(raw[:GUARD] == fill)) and bool(torch.all(raw[GUARD + self.n:] == fill))


def _decode_batch():
    from test_gpu_attention import _batch_with_prefixes
    wl = _batch_with_prefixes([1000, 17, 300, 2048, 5, 64, 129, 0], [1, 1, 2, 5, 33, 65, 1, 3], 32, 8, 128, 16, 77)
    rng = np.random.default_rng(78)
    wl.hidden = W.f32_to_bf16_bits(rng.standard_normal((wl.num_tokens, 512), dtype=np.float32))
    wl.block_size, wl.top_p, wl.seg_mask = 16, 0.9, np.ones(wl.num_segs, np.uint8)
    return wl


@pytest.mark.parametrize("make", [W.tiny_packed, _decode_batch], ids=["tiny_packed", "paged_decode_batch"])
def test_outputs_stay_inside_their_buffers(make):
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import DeviceInputs
    wl = make()
    di = DeviceInputs.from_workload(wl, "cuda")
    n, S, hq, hkv, d = wl.num_tokens, wl.num_segs, wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    bs = wl.block_size
    cap = B.unip_importance_capacity(n, S, bs)
    dm = di.hidden.shape[1]
    bufs = {"out": Banded((n, hq, d), torch.bfloat16), "lse": Banded((hq, n), torch.float32),
            "imp": Banded((cap,), torch.float32), "blk_cu": Banded((S + 1,), torch.int32),
            "keep": Banded((cap,), torch.uint8), "gather_idx": Banded((n,), torch.int32),
            "positions_kept": Banded((n,), torch.int32), "cu_kept": Banded((S + 1,), torch.int32),
            "n_kept": Banded((1,), torch.int32), "hidden_out": Banded((n, dm), torch.bfloat16)}
    B.unip_get_device_status(clear=True)
    page = wl.cache.page_size if wl.cache is not None else 16
    B.unip_prefill_attention(di.q, di.k, di.v, di.cu_seqlens, di.positions, bufs["out"].t, bufs["lse"].t,
                             num_heads_q=hq, num_heads_kv=hkv, head_dim=d, k_cache=di.k_cache, v_cache=di.v_cache,
                             block_table=di.block_table, page_size=page)
    B.unip_block_importance(di.q, di.k, bufs["lse"].t, di.cu_seqlens, bufs["imp"].t, bufs["blk_cu"].t,
                            block_size=bs, num_heads_q=hq, num_heads_kv=hkv, head_dim=d, seg_mask=di.seg_mask)
    B.unip_select_gather(bufs["imp"].t, bufs["blk_cu"].t, di.cu_seqlens, di.positions, bufs["keep"].t,
                         bufs["gather_idx"].t, bufs["cu_kept"].t, bufs["positions_kept"].t, bufs["n_kept"].t,
                         di.hidden, bufs["hidden_out"].t, block_size=bs, p=wl.top_p)
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st == 0, B.describe_status(st)
    bad = [k for k, b in bufs.items() if not b.intact()]
    assert not bad, f"writes outside the output buffers: {bad}"
    # and the outputs inside the bands are right
    ref_o, _ = oracle_attention_rows(wl, None)
    assert_close(bf16_tensor_to_f64(bufs["out"].t), ref_o, what="attention")
    nb = int(bufs["blk_cu"].t[-1].item())
    imp = bufs["imp"].t[:nb].cpu().numpy()
    bc = bufs["blk_cu"].t.cpu().numpy()
    ref_keep = oracle.topp_select(imp, bc, wl.top_p)
    assert np.array_equal(bufs["keep"].t[:nb].cpu().numpy(), ref_keep)
    gi, ck, pk, m = oracle.index_build(ref_keep, bc, wl.cu_seqlens, wl.positions, bs)
    assert int(bufs["n_kept"].t.item()) == m
    assert np.array_equal(bufs["gather_idx"].t[:m].cpu().numpy(), gi)
    got = bufs["hidden_out"].t[:m].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.gather(wl.hidden, gi))
