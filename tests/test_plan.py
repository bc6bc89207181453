"""Host-side checks of the attention planner (unip_attention_plan_create): argument validation, the
choice between a host plan and the device planner, and the split decision.  No GPU is used: the
SM count is passed explicitly."""
import ctypes

import numpy as np
import pytest

from sparsified_long_context_gb300 import binding as B


def _plan(cu, pre, **kw):
    args = dict(num_heads_q=32, num_heads_kv=8, head_dim=128, page_size=16, max_pages_per_seq=4096, num_sms=152)
    args.update(kw)
    return B.AttentionPlan(np.array(cu), None if pre is None else np.array(pre), **args)


@pytest.mark.parametrize("cu,pre,kw", [
    ([1, 512], [0], {}),                       # cu[0] != 0
    ([0, 300, 200], [0, 0], {}),               # not monotone
    ([0, 512], [-1], {}),                      # negative prefix
    ([0, 512], [16 * 4096 + 1], {}),           # prefix beyond the block-table row
    ([0, 512], [100], {"page_size": 24}),      # unsupported page size
    ([0, 512], [100], {"max_pages_per_seq": 0}),
    ([0, 512], [0], {"head_dim": 96}),
    ([0, 512], [0], {"num_heads_q": 30}),      # 30 % 8 != 0
    ([0, 512], [0], {"num_sms": -1}),
    ([0, 512], [0], {"flags": 4}),
])
def test_invalid_layouts_are_rejected(cu, pre, kw):
    with pytest.raises(B.UnipError):
        _plan(cu, pre, **kw)


def test_null_plan_pointer_and_info():
    lib = B.load()
    prm = B._params(32, 8, 128, 0.0)
    cu = np.array([0, 10], np.int32)
    assert lib.unip_attention_plan_create(cu.ctypes.data, 1, None, 10, ctypes.byref(prm), 16, 0, 0, 152,
                                          None) == -1
    assert lib.unip_attention_plan_info(None, None) == -1
    assert lib.unip_attention_plan_workspace_size(None) == 0
    lib.unip_attention_plan_destroy(None)   # a no-op


def test_short_chunk_behind_long_prefix_is_split():
    """A 512-token chunk behind 8192 cached tokens has 64-128 query units for 152 SMs: the plan splits
    their key ranges (two-tile units, two splits each); without splitting nothing is split.  Behind
    3584 cached tokens (the last chunk of a 4096-token prompt) the merge costs more than it saves
    (measured: 53.9 us split against 46.8 us unsplit one-tile items), so that chunk is not split."""
    p = _plan([0, 512], [8192])
    assert p.info["host"] and p.info["split_units"] > 0 and p.info["items"] <= 1024
    assert p.workspace_bytes >= p.info["splits"] * 2 * (128 // 8 + 1) * 256 * 16
    q = _plan([0, 512], [8192], flags=B.UNIP_PLAN_NO_SPLIT)
    assert q.info["host"] and q.info["split_units"] == 0 and q.workspace_bytes == 256
    r = _plan([0, 512], [3584])
    assert r.info["host"] and r.info["split_units"] == 0 and r.info["single"]


def test_few_decodes_with_long_contexts_are_split():
    p = _plan([0, 1, 2, 3, 4], [32768, 30000, 17, 32001], max_pages_per_seq=2048)
    assert p.info["host"] and p.info["split_units"] == 24   # the 17-token context has one key tile


def test_large_calls_fall_back_to_the_device_planner():
    assert not _plan([0, 32768], None).info["host"]                       # 4096 units > 1024 items
    cu = np.arange(0, 130 * 8 + 1, 8)                                     # 130 segments > 128
    assert not _plan(cu, None).info["host"]
    p = _plan([0, 512], [3584], flags=B.UNIP_PLAN_DEVICE)
    assert not p.info["host"]
    assert p.workspace_bytes == B.unip_attention_workspace_size(512, 1, 32, 8, 128)


def test_no_prefix_needs_no_cache_arguments():
    p = _plan([0, 37, 137, 201, 456], None, num_heads_q=4, num_heads_kv=2, head_dim=64, page_size=0,
              max_pages_per_seq=0)
    assert p.info["host"] and p.info["split_units"] == 0


def test_every_unit_appears_once_per_key_range():
    """Item count = units when nothing is split; with splits, more items than units."""
    p = _plan([0, 256, 300], [1024, 0], flags=B.UNIP_PLAN_NO_SPLIT, num_sms=8)
    # G = 4 (token, head) rows: 128-token pairs x 32 heads / 2 per two-tile unit, or x 32 one-tile units
    n_pairs = 2 + 1
    assert p.info["items"] in (n_pairs * 16, n_pairs * 32) or p.info["items"] < n_pairs * 32
    assert p.info["ctas"] <= 8
