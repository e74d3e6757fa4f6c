"""Host-only checks of the C ABI: the library builds, loads, exports every
declared symbol, its struct layout matches the header, and host-detectable
argument errors return their own status codes (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import build as smla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smla.h")


@pytest.fixture(scope="module")
def lib():
    smla_build.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(smla_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"smla_decode", "smla_plan_decode", "smla_workspace_size", "smla_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(B.EXPORTS)
    assert B.smla_abi_version() == 9


def test_struct_layout_matches_header(tmp_path):
    fields = {"smla_args": [f for f, _ in B.SmlaArgs._fields_],
              "smla_plan": [f for f, _ in B.SmlaPlan._fields_]}
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'  printf("{st} %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'  printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", str(src), "-o", str(exe)], check=True)
    out = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                   check=True).stdout.splitlines())
    for st, cls in (("smla_args", B.SmlaArgs), ("smla_plan", B.SmlaPlan)):
        assert int(out[st]) == ctypes.sizeof(cls), st
        for f in fields[st]:
            assert int(out[f"{st}.{f}"]) == getattr(cls, f).offset, f"{st}.{f}"


def test_header_constants_match_pages():
    import json
    c = json.load(open(os.path.join(ROOT, "tests", "golden", "page_constants.json")))
    text = open(HEADER).read()
    assert re.search(r"#define SMLA_HEAD_DIM (\d+)", text).group(1) == str(c["head_dim"]["value"])
    assert re.search(r"#define SMLA_SWA_COLS (\d+)", text).group(1) == str(c["swa_columns"]["value"])


def good_args():
    a = B.SmlaArgs()
    a.sum_q, a.batch, a.num_heads, a.width, a.dtype = 4, 2, 128, 640, B.SMLA_BF16
    a.swa_rows, a.comp_rows = 256, 1024
    return a


def status(lib, a):
    return lib.smla_decode(ctypes.byref(a) if a is not None else None, None)


@pytest.mark.parametrize("mutate,code,needle", [
    (lambda a: setattr(a, "num_heads", 96), B.SMLA_ERR_UNSUPPORTED, "num_heads"),
    (lambda a: setattr(a, "num_heads", 16), B.SMLA_ERR_UNSUPPORTED, "num_heads"),
    (lambda a: setattr(a, "dtype", 7), B.SMLA_ERR_INVALID_ARG, "dtype"),
    (lambda a: setattr(a, "width", 127), B.SMLA_ERR_INVALID_ARG, "width"),
    (lambda a: setattr(a, "sum_q", 5), B.SMLA_ERR_INVALID_ARG, "multiple of batch"),
    (lambda a: setattr(a, "sum_q", -1), B.SMLA_ERR_INVALID_ARG, "sum_q"),
    (lambda a: setattr(a, "batch", 0), B.SMLA_ERR_INVALID_ARG, "batch"),
    (lambda a: setattr(a, "num_splits", 65), B.SMLA_ERR_INVALID_ARG, "num_splits"),
    (lambda a: setattr(a, "max_splits", -2), B.SMLA_ERR_INVALID_ARG, "max_splits"),
    (lambda a: setattr(a, "kernel", 9), B.SMLA_ERR_INVALID_ARG, "kernel"),
    (lambda a: setattr(a, "swa_row_stride", 500), B.SMLA_ERR_INVALID_ARG, "stride"),
    (lambda a: setattr(a, "comp_row_stride", 516), B.SMLA_ERR_INVALID_ARG, "stride"),
    (lambda a: setattr(a, "q_stride_token", 128 * 512 + 4), B.SMLA_ERR_INVALID_ARG, "q_stride_token"),
    (lambda a: setattr(a, "indices_row_stride", 600), B.SMLA_ERR_INVALID_ARG, "indices_row_stride"),
    (lambda a: setattr(a, "comp_rows", -1), B.SMLA_ERR_INVALID_ARG, "row count"),
])
def test_host_argument_errors(lib, mutate, code, needle):
    a = good_args()
    mutate(a)
    assert status(lib, a) == code
    assert needle in B.smla_last_error()


def pointer_args():
    """Every pointer a 256-byte-aligned marker (host checks never dereference)."""
    a = good_args()
    for i, f in enumerate(("q", "swa_kv", "compressed_kv", "sparse_indices", "seq_lens", "out")):
        setattr(a, f, 0x10000 * (i + 1))
    return a


WORD_ARRAYS = ("sparse_indices", "sparse_topk_lens", "seq_lens", "cum_seq_lens_q", "sinks",
               "bmm1_scale_dev", "bmm2_scale_dev", "out_lse", "error_word", "comp_block_tables",
               "hca_seq_lens", "swa_topk_lens")


@pytest.mark.parametrize("field", WORD_ARRAYS)
def test_misaligned_word_arrays_are_rejected_on_the_host(lib, field):
    """int32 / float32 arrays must be 4-byte aligned; the check runs before
    any CUDA call, so it answers here without a GPU."""
    a = pointer_args()
    if field in ("comp_block_tables", "hca_seq_lens"):
        a.comp_block_tables, a.comp_max_pages, a.comp_page_size, a.hca_seq_lens = 0x90000, 4, 128, 0xa0000
    setattr(a, field, 0x80002)
    assert status(lib, a) == B.SMLA_ERR_INVALID_ARG
    assert f"{field} must be 4-byte aligned" in B.smla_last_error()


@pytest.mark.parametrize("field", ["q", "swa_kv", "compressed_kv", "out"])
def test_misaligned_rows_are_rejected_on_the_host(lib, field):
    a = pointer_args()
    setattr(a, field, 0x80008)
    assert status(lib, a) == B.SMLA_ERR_INVALID_ARG
    assert "16-byte aligned" in B.smla_last_error()


@pytest.mark.parametrize("field", ["q", "swa_kv", "compressed_kv", "sparse_indices", "seq_lens", "out"])
def test_missing_required_pointer_is_rejected_on_the_host(lib, field):
    a = pointer_args()
    setattr(a, field, None)
    assert status(lib, a) == B.SMLA_ERR_INVALID_ARG
    assert "required" in B.smla_last_error()


def test_page_table_without_hca_seq_lens_is_rejected_on_the_host(lib):
    a = pointer_args()
    a.comp_block_tables, a.comp_max_pages, a.comp_page_size = 0x90000, 4, 128
    assert status(lib, a) == B.SMLA_ERR_INVALID_ARG
    assert "hca_seq_lens is required" in B.smla_last_error()


def paged_args():
    """Page-table form: 4 pages of 128 rows cover the 512 compressed columns of
    width 640; the pointers are markers only (host checks never read them)."""
    a = good_args()
    a.comp_block_tables, a.comp_max_pages, a.comp_page_size = 64, 4, 128
    a.hca_seq_lens = 64
    return a


@pytest.mark.parametrize("mutate,code,needle", [
    (lambda a: setattr(a, "comp_page_size", 0), B.SMLA_ERR_INVALID_ARG, "comp_page_size"),
    (lambda a: setattr(a, "comp_max_pages", 3), B.SMLA_ERR_INVALID_ARG, "exceed"),
    (lambda a: setattr(a, "block_table_stride", 2), B.SMLA_ERR_INVALID_ARG, "block_table_stride"),
    (lambda a: setattr(a, "indices_row_stride", 100), B.SMLA_ERR_INVALID_ARG, "indices_row_stride"),
    (lambda a: setattr(a, "comp_rows", 1 << 31), B.SMLA_ERR_UNSUPPORTED, "int32"),
])
def test_page_table_argument_errors(lib, mutate, code, needle):
    a = paged_args()
    mutate(a)
    assert status(lib, a) == code
    assert needle in B.smla_last_error()


def test_page_table_index_table_holds_swa_columns_only(lib):
    a = paged_args()
    a.sum_q = 0
    a.indices_row_stride = 128                     # the index form would need >= width (640)
    assert status(lib, a) == B.SMLA_OK
    b = good_args()
    b.sum_q = 0
    b.indices_row_stride = 128
    assert status(lib, b) == B.SMLA_ERR_INVALID_ARG


def test_null_args_and_empty_batch(lib):
    assert status(lib, None) == B.SMLA_ERR_INVALID_ARG
    a = good_args()
    a.sum_q = 0
    assert status(lib, a) == B.SMLA_OK            # nothing to launch, no device needed
    a.dtype = B.SMLA_E4M3
    a.swa_row_stride = 528                        # 528 B: multiple of 16 for FP8 rows
    assert status(lib, a) == B.SMLA_OK


def test_varlen_needs_no_divisibility(lib):
    a = good_args()
    a.sum_q = 0
    a.cum_seq_lens_q = 16                          # any non-NULL value marks varlen; not read on host
    assert status(lib, a) == B.SMLA_OK


def test_status_strings(lib):
    for code, name in ((0, "SMLA_OK"), (1, "SMLA_ERR_INVALID_ARG"), (2, "SMLA_ERR_UNSUPPORTED"),
                       (3, "SMLA_ERR_WORKSPACE_TOO_SMALL"), (4, "SMLA_ERR_CUDA")):
        assert B.smla_status_string(code) == name


def test_binding_raises_on_missing_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        B.lib()


def test_binding_rejects_host_tensors():
    """Host tensors never reach the library (a host pointer read by a kernel
    would fault the GPU): make_args raises before any CUDA call."""
    import torch
    from sparse_mla_decode_token_gb300 import binding as B
    q = torch.zeros(2, 64, 512, dtype=torch.bfloat16)
    kv = torch.zeros(256, 512, dtype=torch.bfloat16)
    idx = torch.zeros(2, 256, dtype=torch.int32)
    seq = torch.full((2,), 300, dtype=torch.int32)
    out = torch.empty(2, 64, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA device"):
        B.make_args(q=q, swa_kv=kv, compressed_kv=kv, sparse_indices=idx, seq_lens=seq, out=out)


def _host_call(**over):
    """A well-formed call's tensors, on the host (layout checks precede the
    device check, so every layout error below answers without a GPU)."""
    import torch
    T, H, B = 4, 64, 2
    kw = dict(q=torch.zeros(T, H, 512, dtype=torch.bfloat16),
              swa_kv=torch.zeros(256, 512, dtype=torch.bfloat16),
              compressed_kv=torch.zeros(256, 512, dtype=torch.bfloat16),
              sparse_indices=torch.zeros(T, 256, dtype=torch.int32),
              seq_lens=torch.full((B,), 300, dtype=torch.int32),
              out=torch.empty(T, H, 512, dtype=torch.bfloat16),
              sparse_topk_lens=torch.full((T,), 200, dtype=torch.int32),
              cum_seq_lens_q=torch.tensor([0, 1, 4], dtype=torch.int32),
              sinks=torch.zeros(H, dtype=torch.float32),
              error_word=torch.zeros(1, dtype=torch.int32))
    kw.update(over)
    return kw


def _bad_layouts():
    import torch
    i32 = torch.int32
    return [
        ("short_topk_lens", dict(sparse_topk_lens=torch.zeros(3, dtype=i32)), ValueError, "sparse_topk_lens has 3"),
        ("short_cum", dict(cum_seq_lens_q=torch.tensor([0, 4], dtype=i32)), ValueError, "cum_seq_lens_q has 2"),
        ("short_sinks", dict(sinks=torch.zeros(63)), ValueError, "sinks has 63"),
        ("strided_sinks", dict(sinks=torch.zeros(128)[::2]), ValueError, "sinks must be contiguous"),
        ("f64_sinks", dict(sinks=torch.zeros(64, dtype=torch.float64)), ValueError, "float32"),
        ("strided_seq_lens", dict(seq_lens=torch.zeros(4, dtype=i32)[::2]), ValueError, "seq_lens must be contiguous"),
        ("short_swa_topk_lens", dict(swa_topk_lens=torch.zeros(2, dtype=i32)), ValueError, "swa_topk_lens has 2"),
        ("i64_error_word", dict(error_word=torch.zeros(1, dtype=torch.int64)), TypeError, "error_word must be int32"),
        ("empty_error_word", dict(error_word=torch.zeros(0, dtype=i32)), ValueError, "error_word has 0"),
        ("i64_seq_lens", dict(seq_lens=torch.zeros(2, dtype=torch.int64)), TypeError, "seq_lens must be int32"),
        ("f16_scale", dict(bmm1_scale=torch.ones(1, dtype=torch.float16)), TypeError, "bmm1_scale"),
        ("empty_scale", dict(bmm2_scale=torch.ones(0)), ValueError, "bmm2_scale tensor is empty"),
        ("few_index_rows", dict(sparse_indices=torch.zeros(3, 256, dtype=i32)), ValueError, "3 rows for 4"),
        ("index_dim1_not_1", dict(sparse_indices=torch.zeros(4, 2, 256, dtype=i32)), ValueError, "1 in dim 1"),
        ("strided_index_cols", dict(sparse_indices=torch.zeros(4, 512, dtype=i32)[:, ::2]), ValueError, "contiguous last dim"),
        ("dense_query_needs_copy", dict(q=torch.zeros(2, 64, 2, 512, dtype=torch.bfloat16).transpose(1, 2)),
         ValueError, "without a copy"),
    ]


@pytest.mark.parametrize("case", _bad_layouts(), ids=lambda c: c[0])
def test_binding_rejects_bad_layouts_before_the_device_check(case):
    _, over, exc, match = case
    with pytest.raises(exc, match=match):
        B.make_args(**_host_call(**over))


def test_binding_well_formed_host_call_fails_only_on_placement():
    with pytest.raises(ValueError, match="CUDA device"):
        B.make_args(**_host_call())
    import torch
    # a dense [B, q_len, H, 512] query that flattens without a copy passes layout
    with pytest.raises(ValueError, match="CUDA device"):
        B.make_args(**_host_call(q=torch.zeros(2, 2, 64, 512, dtype=torch.bfloat16)))


@pytest.mark.parametrize("compiler", [["gcc", "-std=c99"], ["g++", "-std=c++17", "-x", "c++"]],
                         ids=["c99", "c++17"])
def test_plain_c_caller_links_and_runs(lib, tmp_path, compiler):
    """A C program (no Python, no CUDA headers), built as C99 and as C++,
    links libsmla.so and gets plans and host-side statuses from it without a
    GPU."""
    src = os.path.join(ROOT, "tests", "c", "abi_from_c.c")
    exe = tmp_path / "abi_from_c"
    libdir = os.path.dirname(B.LIB_PATH)
    subprocess.run(compiler + ["-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                               src, "-x", "none", "-o", str(exe), "-L", libdir, "-lsmla", f"-Wl,-rpath,{libdir}"],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and r.stdout.count("ok ") == 11
