"""Host-side helpers of bench.py: useful-FLOP counts against independently
computed pair counts, the per-workload bounds, the recorded-traffic lookup and
the per-step launch count (no GPU)."""
import hashlib
import json
import os

import numpy as np

import bench
from oracle.scheduling import ffd_order
from sparsified_long_context_gb300 import workloads as W
from sparsified_long_context_gb300.pipeline import kernels_per_step


def _pairs(wl):
    return bench.useful_attention_flops(wl) / (4.0 * wl.head_dim * wl.num_heads_q)


def test_useful_pairs_by_brute_force_on_the_tiny_batch():
    wl = W.tiny_packed()
    visible = 0
    for s in range(wl.num_segs):
        n = int(wl.cu_seqlens[s + 1] - wl.cu_seqlens[s])
        visible += sum(1 for i in range(n) for j in range(n) if j <= i)
    assert _pairs(wl) == visible == 40473


def test_useful_pairs_of_the_chunked_and_long_prompts():
    one, chunks = W.chunked()
    assert _pairs(one) == 4096 * 4097 // 2 == 8390656
    assert sum(_pairs(c) for c in chunks) == 8390656          # chunking does not change the useful work
    n = 32768
    assert n * (n + 1) // 2 == 536887296                       # the long prompt's pairs (closed form)


def test_rows_flops_matches_the_whole_count():
    wl = W.tiny_packed()
    assert bench.rows_flops(wl, range(wl.num_tokens)) == bench.useful_attention_flops(wl)


def test_mixed_step_bound_is_prefill_flops_plus_decode_bytes():
    wl = W.mixed_step(d_model=0)
    ctx = bench.workload_context(wl, attn_ms=10.0, bf16_peak=1000.0, hbm_peak=5000.0)
    pre = wl.seg_mask.astype(bool)
    n, P = wl.seq_lens.astype(np.float64), wl.prefix_lens.astype(np.float64)
    f_pre = float(np.sum(4.0 * 128 * 32 * (n * P + n * (n + 1) / 2)[pre]))
    kv = float(np.sum((P + n)[~pre])) * 8 * 128 * 2 * 2
    assert ctx["prefill_flops"] == f_pre and ctx["decode_kv_bytes"] == kv
    assert abs(ctx["roofline_ms"] - (f_pre / 1e15 + kv / 5e12) * 1e3) < 1e-9
    assert abs(ctx["attention_frac_of_roofline"] - ctx["roofline_ms"] / 10.0) < 1e-12


def test_prepacked_padding_context():
    wl = W.prepacked(ffd_order)
    ctx = bench.workload_context(wl, 1.0, 1000.0, 5000.0)
    lmax = int(wl.seq_lens.max())
    c = 4.0 * 128 * 32
    assert ctx["padded_to_max_flops"] == c * 64 * lmax * (lmax + 1) / 2
    assert ctx["padded_to_bin_flops"] == c * len(wl.meta["bins"]) * 16384 * 16385 / 2
    assert ctx["useful_flops"] <= ctx["padded_to_bin_flops"] <= ctx["padded_to_max_flops"]
    assert bench.workload_context(W.tiny_packed(), 1.0, 1000.0, 5000.0) is None


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha1(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(
        {"k": {"kernel_source": "kernel.cu", "kernel_source_sha1": sha, "dram_bytes_per_launch": 12345}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k") == 12345.0
    src.write_text("// kernel v2\n")                           # changed since the capture: no traffic
    assert bench.recorded_traffic("k") is None
    assert bench.recorded_traffic("missing") is None


def test_launches_per_step():
    assert kernels_per_step(True, fused_select=True, num_segs=1) == 6
    assert kernels_per_step(True, fused_select=True, num_segs=260) == 7
    assert kernels_per_step(True, fused_select=False) == 8
    assert kernels_per_step(False, fused_select=False) == 7
    assert kernels_per_step(fused_importance=True) == 6
    assert kernels_per_step(fused_importance=True, num_segs=1) == 5


def test_committed_traffic_records_follow_their_sources():
    """bench.py attaches a recorded DRAM figure only while the kernel source still hashes as at capture."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    table = json.load(open(os.path.join(root, "profiles", "dram_traffic.json")))
    for name, rec in table.items():
        if name.startswith("_"):
            continue
        src = os.path.join(root, rec["kernel_source"])
        sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
        assert (bench.recorded_traffic(name) is not None) == (sha == rec["kernel_source_sha1"])


def test_select_copy_split_reports_the_copy_rate_of_the_kept_rows():
    # 2176 kept rows of 4096 bf16: 17.8 MB read and as much written
    sp = bench.select_copy_split(0.012, (0.006, 0.0055), 2176, 4096, 6744.6)
    assert sp["row_copy_bytes"] == 2 * 2 * 4096 * 2176
    assert abs(sp["row_copy_gbs"] - sp["row_copy_bytes"] / 0.0055e-3 / 1e9) < 1e-6
    assert abs(sp["row_copy_frac_hbm"] - sp["row_copy_gbs"] / 6744.6) < 1e-12
    assert abs(sp["overlap_ms"] - (0.006 + 0.0055 - 0.012)) < 1e-12
    # no hidden rows in the workload: nothing to split
    assert bench.select_copy_split(0.03, None, 100, 0, 6744.6) is None
    assert bench.select_copy_split(0.03, (0.01, 0.01), 100, 0, 6744.6) is None
