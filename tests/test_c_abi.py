"""The C ABI from plain C: the headers compile as strict C11 and a C program
linked against libunip.so packs prompts and builds chunked-prefill steps that
match the oracle (host calls only, no GPU)."""
import os
import shutil
import subprocess

import pytest

from oracle import scheduling as osch
from sparsified_long_context_gb300 import native_build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")


def test_headers_compile_as_c11():
    for h in ("unip.h", "unip_sched.h"):
        r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                            "-I", INCLUDE, "-x", "c", os.path.join(INCLUDE, h)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_c_program_matches_the_oracle(tmp_path):
    lib = native_build.build()
    exe = tmp_path / "host_builders"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", INCLUDE, os.path.join(HERE, "c", "host_builders.c"),
                        "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lengths = [5, 7, 5, 2, 4, 2, 5, 1, 6]
    out = subprocess.run([str(exe), "10"] + [str(x) for x in lengths], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.strip().splitlines()
    assert lines[0] == "pack 0 ok"
    bins = [[int(x) for x in ln.split()[1:]] for ln in lines if ln.startswith("bin")]
    assert bins == osch.ffd_pack(lengths, 10)
    sched = osch.ChunkedScheduler(8, 4, 256, 8, 1)
    for L in lengths:
        sched.add(L, 2)
    expect = []
    while True:
        segs, _ = sched.step()
        if not segs:
            break
        expect.append("step" + "".join(f" [{i} {a} {n} {int(p)}]" for (i, a, n, p) in segs))
    assert [ln for ln in lines if ln.startswith("step")] == expect
    assert lines[-1] == "bad invalid argument"
