"""Checks of the seeded input generators (shapes and structure of each workload)."""
import numpy as np
import torch

from oracle.scheduling import ffd_order
from sparsified_long_context_gb300 import workloads as W


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-7 + 2**-9, -2.5, 3.0e-3], np.float32)
    bits = W.f32_to_bf16_bits(vals)
    back = W.bf16_bits_to_f32(bits)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 is a tie -> even (1+2^-6); 1+2^-7+2^-9 rounds down
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0 + 2**-6)
    assert back[3] == np.float32(1.0 + 2**-7) and back[4] == -2.5
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)


def test_tiny_packed_shape():
    wl = W.tiny_packed()
    assert wl.num_tokens == 456 and wl.num_segs == 4
    assert list(wl.seq_lens) == [37, 100, 64, 255]
    assert list(-(-wl.seq_lens // 16)) == [3, 7, 4, 16]
    assert len(wl.meta["heavy_rows"]) == 23
    assert wl.q.shape == (456, 4, 64) and wl.k.shape == (456, 2, 64) and wl.hidden.shape == (456, 256)
    assert list(wl.prefix_lens) == [0, 0, 0, 0]


def test_prepacked_ffd_structure():
    wl = W.prepacked(ffd_order)
    L = wl.meta["lengths"]
    assert len(L) == 64 and min(L) >= 32 and max(L) <= 8192
    for b in wl.meta["bins"]:
        assert sum(wl.meta["lengths"][wl.meta["prompt_order"].index(i)] for i in b) <= 16384
    assert 30000 < wl.num_tokens < 80000
    assert np.all(wl.positions[wl.cu_seqlens[:-1]] == 0)


def test_long_single_spans():
    wl = W.long_single(d_model=0)
    h = wl.meta["heavy_rows"]
    assert len(h) == 1638 and len(np.unique(h)) == 1638
    starts, lens = wl.meta["span_starts"], wl.meta["span_lens"]
    for i in range(9):
        assert starts[i] + lens[i] < starts[i + 1]
    assert wl.num_tokens == 32768


def test_mixed_step_budget_and_pages():
    wl = W.mixed_step(d_model=0)
    assert wl.num_tokens == 8192 and wl.num_segs == 260
    L = wl.seq_lens
    assert np.all(L[:256] == 1) and np.all(L[256:] == 1984)
    P = wl.prefix_lens
    assert np.all((P[:256] >= 1024) & (P[:256] <= 32768))
    assert np.all(P[256:] % 64 == 0) and np.all(P[256:] <= 65536 - 1984)
    assert list(-(-L[256:] // 64)) == [31] * 4
    bt = wl.block_table
    used = np.concatenate([bt[s, : -(-int(P[s]) // 16)] for s in range(260)])
    assert len(np.unique(used)) == len(used) == wl.cache.num_pages


def test_chunked_layout():
    one, chunks = W.chunked()
    assert len(chunks) == 8 and one.num_tokens == 4096
    for c, wl in enumerate(chunks):
        assert wl.prefix_lens[0] == 512 * c
        k_pages, _ = wl.cache.pages_numpy(wl.block_table[0, :4])
        assert np.array_equal(k_pages.reshape(64, 8, 128), one.k[:64])


def test_hash_generator_numpy_matches_torch():
    idx = np.concatenate([np.arange(5000), np.array([2**32 - 1, 2**32, 2**33 + 12345, 7 * 2**32 + 99])])
    a = W.hash_normal_bf16_numpy(1234, 1, idx)
    b = W.hash_normal_bf16_torch(1234, 1, torch.from_numpy(idx)).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(a, b)
    x = W.bf16_bits_to_f32(a[:5000]).astype(np.float64)
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1.0) < 0.05


def test_prepacked_stream_is_the_same_under_the_library_and_oracle_packers():
    """The bench packs the prepacked batch with the library's packer, the reference arm and the CPU tests
    with the oracle's; both must yield the same stream."""
    from sparsified_long_context_gb300 import binding as B
    a, b = W.prepacked(B.unip_ffd_pack), W.prepacked(ffd_order)
    assert a.meta["prompt_order"] == b.meta["prompt_order"] and a.meta["bins"] == b.meta["bins"]
    for f in ("cu_seqlens", "positions", "q", "k", "v"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    # rows are laid out prompt by prompt in the packed order: heavy keys follow their rows
    assert np.array_equal(a.meta["heavy_rows"], b.meta["heavy_rows"])
