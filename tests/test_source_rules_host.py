"""Static rules over the committed sources (CPU): device code never traps,
every mbarrier wait goes through a bounded wait, nothing uses multi-GPU
multicast, every ncu command in the profile summaries leaves the clocks
alone, nothing changes a GPU's settings, and code and comments stand on their
own (no build notes or machine paths)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_mla_decode_token_gb300", "csrc")
SKIP_DIRS = {".git", "_work", "gpurun_out", "_build", "__pycache__", "baseline", ".pytest_cache"}
CODE_EXT = (".py", ".cu", ".cuh", ".h", ".c", ".sh")


def files(exts, top=ROOT):
    for d, dirs, names in os.walk(top):
        dirs[:] = [x for x in dirs if x not in SKIP_DIRS]
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def strip_comments(text):
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return re.sub(r"//[^\n]*", " ", text)


DEVICE_SOURCES = sorted(files((".cu", ".cuh"), CSRC))


def test_device_sources_exist():
    names = {os.path.basename(f) for f in DEVICE_SOURCES}
    assert {"decode_tcgen05.cu", "decode_cuda_core.cu", "combine.cu", "tc_ptx.cuh"} <= names


@pytest.mark.parametrize("path", DEVICE_SOURCES, ids=os.path.basename)
def test_device_code_never_traps(path):
    code = strip_comments(open(path).read())
    assert "__trap" not in code
    assert not re.search(r"\btrap\s*;", code)
    assert "brkpt" not in code
    assert not re.search(r"(?<!static_)\bassert\s*\(", code)       # device asserts trap


@pytest.mark.parametrize("path", DEVICE_SOURCES, ids=os.path.basename)
def test_no_multi_gpu_multicast(path):
    """One GPU only: no NVLink multicast objects or multimem accesses (TMA
    multicast within a cluster reads this GPU's own memory and stays allowed)."""
    code = strip_comments(open(path).read())
    assert "multimem" not in code
    assert "cuMulticast" not in code


def function_body(code, name):
    m = re.search(r"\b" + name + r"\s*\([^)]*\)\s*\{", code)
    assert m, name
    depth, i = 1, m.end()
    while depth:
        depth += {"{": 1, "}": -1}.get(code[i], 0)
        i += 1
    return code[m.end():i]


def test_every_mbarrier_wait_is_bounded():
    """Raw try-waits are defined in tc_ptx.cuh and called only from the two
    bounded waits the tcgen05 kernels share (tc_common.cuh): wait_bar
    (timeout -> abort flag and error word) and drain_wait (timeout, not cut
    short by the abort flag)."""
    ptx = strip_comments(open(os.path.join(CSRC, "tc_ptx.cuh")).read())
    assert ptx.count("mbarrier.try_wait") == 2 and "mbarrier.test_wait" not in ptx
    for path in DEVICE_SOURCES:
        code = strip_comments(open(path).read())
        if os.path.basename(path) == "tc_ptx.cuh":
            continue
        assert "mbarrier.try_wait" not in code and "mbarrier.test_wait" not in code, path
        calls = len(re.findall(r"\bmbar_try_wait(_cluster)?\s*\(", code))
        if os.path.basename(path) != "tc_common.cuh":
            assert calls == 0, path
            continue
        wait_bar, drain = function_body(code, "wait_bar"), function_body(code, "drain_wait")
        inside = sum(len(re.findall(r"\bmbar_try_wait(_cluster)?\s*\(", b)) for b in (wait_bar, drain))
        assert calls == inside == 3
        assert "kTimeoutNs" in wait_bar and "kTimeoutNs" in drain
        assert "SMLA_DEVERR_TIMEOUT" in wait_bar and "abort_flag" in wait_bar


def test_ncu_commands_leave_the_clocks_alone():
    found = 0
    for path in files((".md", ".txt"), os.path.join(ROOT, "profiles")):
        for line in open(path):
            if re.match(r"^\s*ncu\s+--", line):
                found += 1
                assert "--clock-control none" in line, (path, line)
    assert found >= 5


def test_nothing_changes_gpu_settings():
    smi = "nvidia" + "-smi"
    bad = re.compile(smi + r"[^\n]*\s(-lgc|-rgc|-ac|-rac|-pl|-pm|-mig|-e|-r|--lock|--reset)\b")
    for path in files(CODE_EXT):
        text = open(path, errors="ignore").read()
        assert not bad.search(text), path


def test_code_and_comments_stand_on_their_own():
    """No file of code names the build's notes, the machine's paths or the
    tooling around the build (pieces joined here so this file names none)."""
    needles = ["BASELINE" + ".json", "BASELINE" + ".md", "north" + "_star", "PAPER" + ".md", "SURVEY" + ".md",
               "DESIGN" + ".md", "VERDICT" + ".md", "ADVICE" + ".md", "/root" + "/", "gpu" + "run", "configs" + "["]
    me = os.path.abspath(__file__)
    for path in files(CODE_EXT):
        if os.path.abspath(path) == me:
            continue
        text = open(path, errors="ignore").read()
        for n in needles:
            assert n not in text, (os.path.relpath(path, ROOT), n)


def test_the_product_never_imports_the_oracle():
    """The library package and build() leave the oracle unimported (only the
    tests, smoke() and the benchmark's CPU-baseline leg may run it)."""
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "sparse_mla_decode_token_gb300")
    for path in files((".py",), pkg):
        text = open(path).read()
        assert not re.search(r"^\s*(import oracle|from oracle)", text, flags=re.M), path
    code = ("import sys; import __graft_entry__ as g; g.build(); "
            "import sparse_mla_decode_token_gb300.binding, sparse_mla_decode_token_gb300.workloads; "
            "assert 'oracle' not in sys.modules and 'oracle.oracle' not in sys.modules, sorted(sys.modules)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
