"""StreamedSteps (uploads and downloads overlapped with the kernels of the
neighbouring steps) gives, step for step, the same results as one plain step
on the same batch: attention output, n_kept and compacted hidden rows, bit for
bit.  Two different batches alternate, so results from the wrong set, or
copies racing the kernels, show up as mismatches."""
import dataclasses

import numpy as np
import pytest

from sparsified_long_context_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _plain(wl):
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import (DeviceInputs, StepBuffers, run_attention, run_importance,
                                                        run_select_gather)
    di = DeviceInputs.from_workload(wl, "cuda")
    bufs = StepBuffers(di)
    run_attention(di, bufs)
    run_importance(di, bufs)
    run_select_gather(di, bufs)
    torch.cuda.synchronize()
    m = int(bufs.n_kept.item())
    st = B.unip_get_device_status(clear=True)
    assert st == 0, B.describe_status(st)
    hid = None if bufs.hidden_out is None else bufs.hidden_out[:m].cpu().clone()
    return bufs.out.cpu().clone(), m, hid


@pytest.mark.parametrize("steps", [1, 2, 7])
def test_streamed_steps_match_plain_steps(steps):
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import DeviceInputs, StepBuffers, StreamedSteps
    wl_a = W.tiny_packed(seed=1)
    wl_b = W.packed([37, 100, 64, 255], 4, 2, 64, 9, 0.05, block_size=16, top_p=0.9, d_model=256, name="tiny_b")
    ref = [_plain(wl_a), _plain(wl_b)]
    assert ref[0][1] != ref[1][1] or not torch.equal(ref[0][0], ref[1][0])   # the batches differ
    di = DeviceInputs.from_workload(wl_a, "cuda")
    di2 = dataclasses.replace(di, **{f: getattr(di, f).clone() for f in StreamedSteps.FIELDS
                                     if getattr(di, f) is not None})
    streamer = StreamedSteps([(di, StepBuffers(di)), (di2, StepBuffers(di2))])
    di_b = DeviceInputs.from_workload(wl_b, "cuda")
    batches = [streamer.host_batch(di), streamer.host_batch(di_b)]
    seen = {}

    def on_result(i, out_host, hid_host, m):
        seen[i] = (out_host.clone(), m, hid_host.clone())

    kept = streamer.run(batches, steps, on_result)
    st = B.unip_get_device_status(clear=True)
    assert st == 0, B.describe_status(st)
    assert sorted(seen) == list(range(steps))
    for i in range(steps):
        out, m, hid = seen[i]
        r_out, r_m, r_hid = ref[i % 2]
        assert m == r_m == kept[i], (i, m, r_m, kept[i])
        assert torch.equal(out.view(torch.int16), r_out.view(torch.int16)), f"step {i}: attention output differs"
        assert torch.equal(hid.view(torch.int16), r_hid.view(torch.int16)), f"step {i}: hidden rows differ"


def test_streamed_chunks_behind_a_paged_prefix():
    """Chunked-prefill batches (512 tokens behind 1536 and 2560 cached tokens of one paged cache, which
    both device sets share and which is not re-uploaded) alternate through StreamedSteps; every step's
    attention output and compaction equal a plain step on the same chunk."""
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import DeviceInputs, StepBuffers, StreamedSteps
    _, chunks = W.chunked()
    wls = [dataclasses.replace(chunks[c], block_size=64, top_p=0.9, seg_mask=np.ones(1, np.uint8))
           for c in (3, 5)]
    ref = [_plain(w) for w in wls]
    di = DeviceInputs.from_workload(wls[0], "cuda")
    di2 = dataclasses.replace(di, **{f: getattr(di, f).clone() for f in StreamedSteps.FIELDS
                                     if getattr(di, f) is not None})
    streamer = StreamedSteps([(di, StepBuffers(di)), (di2, StepBuffers(di2))])
    di_b = DeviceInputs.from_workload(wls[1], "cuda")
    batches = [streamer.host_batch(di), streamer.host_batch(di_b)]
    seen = {}
    kept = streamer.run(batches, 5, lambda i, o, h, m: seen.__setitem__(i, (o.clone(), m)))
    st = B.unip_get_device_status(clear=True)
    assert st == 0, B.describe_status(st)
    for i in range(5):
        out, m = seen[i]
        r_out, r_m, _ = ref[i % 2]
        assert m == r_m == kept[i]
        assert torch.equal(out.view(torch.int16), r_out.view(torch.int16)), f"step {i}"
