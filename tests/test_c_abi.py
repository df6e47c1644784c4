"""The C ABI used from plain C (CPU).

`include/pa.h` must compile as strict C99 and `libpa.so` must link and run from a C
program with no C++ or Python in between.  tests/c/bm_worked_trace.c drives the
block manager through the worked allocation trace of "PagedAttention, simply
explained" (100 frames of 10 slots, prompts A:8 B:5 C:12 D:9, three decode steps);
its output is compared with the trace's printed tables and free list
(tests/golden/worked_allocation_trace.json) and with the slots the translation
frame * B + offset gives for them.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "paged_kv_cache_126_gb300")


@pytest.fixture(scope="module")
def trace_output(pa, tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("cabi") / "bm_worked_trace")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "bm_worked_trace.c"), "-o", exe, "-L", LIBDIR, "-lpa",
           f"-Wl,-rpath,{LIBDIR}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, res.stdout + res.stderr
    return [line.split() for line in res.stdout.splitlines()]


def test_worked_trace_from_c(trace_output, golden):
    g = golden("worked_allocation_trace.json")
    lines = {(t[0], t[1]) if t[0] in ("step", "seq") else (t[0],): t for t in trace_output}
    # decode steps: every token's slot is frame * 10 + offset of the printed final tables
    final = g["steps"][-1]["tables"]
    names = g["order"]
    lens0 = [g["prefill"][n] for n in names]
    for k in range(3):
        t = lines[("step", str(k + 1))]
        got = [int(x) for x in t[3:7]]
        want = [final[n][(lens0[i] + k) // 10] * 10 + (lens0[i] + k) % 10 for i, n in enumerate(names)]
        assert got == want
        assert t[7:] == ["copies", "0"]
    for i, n in enumerate(names):
        t = lines[("seq", str(i))]
        assert int(t[3]) == lens0[i] + 3
        assert [int(x) for x in t[5:]] == final[n]
    st = g["steps"][-1]
    f = lines[("free",)]
    assert int(f[1]) == st["free_len"]
    assert [int(x) for x in f[3:6]] == st["free_head"] and int(f[7]) == st["free_last"]
    u = [int(x) for x in lines[("usage",)][1:]]
    fill = st["fill"]
    assert u == [sum(len(v) for v in fill.values()), sum(n for v in fill.values() for _, n in v),
                 sum(lens0) + 12, sum(len(v) for v in fill.values()),
                 max(10 * len(v) - sum(n for _, n in v) for v in fill.values())]


@pytest.mark.gpu
def test_device_path_from_c(pa, tmp_path):
    # pa_cache_append + pa_decode from a C program (CUDA runtime only, descriptors filled by
    # hand): a one-token context returns its value row, equal keys return the mean of the
    # value rows, bit for bit in fp16 (tests/c/decode_from_c.c).
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "decode_from_c")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "decode_from_c.c"), "-o", exe,
           "-L", LIBDIR, "-lpa", "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{LIBDIR}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "mismatches 0 status 0" in res.stdout
