"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
entry point declared in include/*.h (no compute calls here)."""
import ctypes
import os
import re

from sparsified_long_context_gb300 import binding, native_build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_symbols():
    names = []
    for f in sorted(os.listdir(INCLUDE)):
        if f.endswith(".h"):
            text = open(os.path.join(INCLUDE, f)).read()
            names += re.findall(r"UNIP_API\s+[\w\s\*]+?\b(unip_\w+)\s*\(", text)
    return names


def test_header_declares_the_four_calls():
    names = set(declared_symbols())
    for n in ("unip_prefill_attention", "unip_block_importance", "unip_topp_select", "unip_gather_tokens",
              "unip_ffd_pack", "unip_step_builder_next"):
        assert n in names


def test_library_exports_every_declared_symbol():
    path = native_build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_helpers_without_gpu():
    lib = binding.load()
    assert binding.unip_version().startswith("unip")
    assert lib.unip_status_string(-2).decode() == "unsupported shape"
    assert binding.unip_importance_capacity(32768, 1, 64) >= 512
    assert binding.unip_attention_workspace_size(32768, 1, 32, 8, 128) >= 256 + 8 * 257
    assert binding.unip_topp_workspace_size(8192, 260, 64) > 0


def test_host_rejects_bad_arguments_before_launch():
    lib = binding.load()
    prm = binding._params(32, 8, 96, 0.0)   # head_dim 96 is not covered
    rc = lib.unip_prefill_attention(None, None, None, ctypes.c_void_p(16), 1, None, 10, None, ctypes.byref(prm),
                                    None, None, None, 0, None)
    assert rc == -2
    prm = binding._params(32, 7, 128, 0.0)  # H_q not a multiple of H_kv
    rc = lib.unip_prefill_attention(None, None, None, ctypes.c_void_p(16), 1, None, 10, None, ctypes.byref(prm),
                                    None, None, None, 0, None)
    assert rc == -1
    rc = lib.unip_topp_select(None, None, None, None, 1, 10, 16, 1.5, 3, None, 0, None, None, None, None, None, 0,
                              None)
    assert rc == -1


def test_rope_host_checks_before_launch():
    lib = binding.load()
    prm = binding._params(8, 2, 72, 0.0)    # D not a multiple of 16
    assert lib.unip_rope_append_kv(None, ctypes.c_void_p(16), None, ctypes.c_void_p(16), 10, ctypes.byref(prm),
                                   10000.0, 0, None, None, None, 0, 16, None) == -2
    prm = binding._params(8, 2, 128, 0.0)
    assert lib.unip_rope_append_kv(None, ctypes.c_void_p(16), None, ctypes.c_void_p(16), 10, ctypes.byref(prm),
                                   10000.0, 2, None, None, None, 0, 16, None) == -1     # layout flag
    assert lib.unip_rope_append_kv(None, None, None, None, 10, ctypes.byref(prm),
                                   10000.0, 0, None, None, None, 0, 16, None) == -1     # k missing
    assert lib.unip_rope_append_kv(None, ctypes.c_void_p(16), None, ctypes.c_void_p(16), 10, ctypes.byref(prm),
                                   10000.0, 0, ctypes.c_void_p(16), None, None, 4, 16, None) == -1  # caches missing
    assert lib.unip_rope_append_kv(None, ctypes.c_void_p(24), None, ctypes.c_void_p(16), 10, ctypes.byref(prm),
                                   10000.0, 0, None, None, None, 0, 16, None) == -5     # misaligned k
    assert lib.unip_rope_append_kv(None, None, None, None, 0, ctypes.byref(prm),
                                   10000.0, 0, None, None, None, 0, 16, None) == 0      # nothing to do
    for bad in (float("inf"), float("nan")):
        assert lib.unip_rope_append_kv(None, ctypes.c_void_p(16), None, ctypes.c_void_p(16), 10, ctypes.byref(prm),
                                       bad, 0, None, None, None, 0, 16, None) == -1


def test_attention_schedule_modes():
    lib = binding.load()
    assert lib.unip_set_attention_schedule(7) == -1
    for m in (1, 2, 0):
        assert lib.unip_set_attention_schedule(m) == 0


def test_bounded_wait_selftest_checks_its_arguments():
    lib = binding.load()
    assert lib.unip_selftest_bounded_wait(0, ctypes.c_void_p(16), None) == -1         # limit 0
    assert lib.unip_selftest_bounded_wait(2000000, ctypes.c_void_p(16), None) == -1   # above one second
    assert lib.unip_selftest_bounded_wait(1000, None, None) == -1                      # no result buffer


def test_binding_status_bits_match_the_header():
    text = open(os.path.join(INCLUDE, "unip.h")).read()
    bits = {name: int(val, 16) for name, val in re.findall(r"#define (UNIP_DEV_\w+) (0x[0-9a-fA-F]+)u", text)}
    assert len(bits) == 8
    for name, val in bits.items():
        assert getattr(binding, name) == val, name
        assert val in binding.DEV_STATUS_BITS, name
