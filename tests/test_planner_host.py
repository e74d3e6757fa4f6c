"""The planner, called through the C ABI as a pure function of shapes and the
SM count (no GPU): its documented rules, and the plans the committed
measurements were taken with.

Rules (tcgen05 kernel, 2-CTA clusters, 152 SMs = 76 pairs on GB300):

* balanced mode when the schedule is BALANCED, num_splits and max_splits
  are 0, the kernel is TCGEN05, W <= 2304 and T <= 14 x pairs: P = min(pairs, T W / 64)
  clusters (at least 1) take equal shares of the T x W columns; grid = 2 P,
  num_splits = 1; with P > 1 the workspace holds 2 P x H BF16 pieces of
  512, their fp32 LSEs (one copy per CTA of a pair) and 2 P counters (each
  part 256-byte aligned);
* otherwise (and under the default schedule) grid mode, one cluster per
  (token, split): S = floor(pairs / T)
  so that every cluster runs in one wave, at least 1, capped by max_splits
  (default 32) and by ceil(W / 64) (at least 64 columns per split), then
  raised to ceil(W / 2304) (the columns one CTA stages).  A forced num_splits
  below that minimum is an error.

The CUDA-core kernel targets 2 resident CTAs per SM with at least 256 columns
per split.
"""
import json
import math
import os

import numpy as np
import pytest

from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import build as smla_build
from sparse_mla_decode_token_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GB300_SMS = 152


@pytest.fixture(scope="module", autouse=True)
def lib():
    smla_build.build()
    return B.lib()


def args(T, W_, *, H=128, dtype=B.SMLA_E4M3, batch=None, varlen=False, num_splits=0, max_splits=0,
         kernel=B.KERNEL_AUTO, schedule=B.SCHEDULE_AUTO):
    a = B.SmlaArgs()
    a.sum_q, a.batch, a.num_heads, a.width, a.dtype = T, batch or max(T, 1), H, W_, dtype
    if varlen:
        a.cum_seq_lens_q = 16                 # marks varlen; never read by the planner
    a.num_splits, a.max_splits, a.kernel, a.schedule = num_splits, max_splits, kernel, schedule
    return a


def plan(a, sms=GB300_SMS):
    return B.smla_plan_decode_for_sm_count(a, sms).as_dict()


def expected_clusters(T, W_, num_splits=0, max_splits=0, sms=GB300_SMS, schedule=B.SCHEDULE_BALANCED):
    """Balanced-mode cluster count, 0 where grid mode applies."""
    pairs = sms // 2
    if schedule != B.SCHEDULE_BALANCED or num_splits or max_splits or W_ > 2304 or T > 14 * pairs:
        return 0
    return max(1, min(pairs, T * W_ // 64))


def expected_tc_splits(T, W_, max_splits=0, sms=GB300_SMS):
    pairs = sms // 2
    want = pairs // T if T > 0 else 1
    want = min(want, math.ceil(W_ / 64), max_splits or 32)
    want = max(want, math.ceil(W_ / 2304))
    return max(want, 1)


def workload_args(n):
    w = W.config_workload(n)
    dt = {"bf16": B.SMLA_BF16, "e4m3": B.SMLA_E4M3, "packed_fp8": B.SMLA_PACKED_FP8,
          "nvfp4": B.SMLA_NVFP4}[w.dtype]
    return args(w.sum_q, w.width, H=w.num_heads, dtype=dt, batch=w.batch,
                varlen=w.cum_seq_lens_q is not None)


def test_plans_of_the_committed_traffic_records():
    """traffic.json stores the launch plan and device-code hash of each ncu
    capture.  A record of the current device code must match the planner's
    plan for its workload on a GB300; a record of older device code is one
    that bench.py reports as stale (traffic null), never as a measurement of
    this code."""
    import bench
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    by_name = {name: n for n, name in W.CONFIG_NAMES.items()}
    sha = bench.kernel_sources_sha()
    for name, ent in rec.items():
        if name.startswith("_"):
            continue
        got = plan(workload_args(by_name[name]))
        traffic, note = bench.traffic_record(name, got)
        if ent.get("kernel_sources_sha") == sha:
            for k, v in ent["plan"].items():
                assert got[k] == v, (name, k, got[k], v)
            assert traffic == ent["dram_bytes_per_launch"]
        else:
            assert traffic is None and sha in note


@pytest.mark.parametrize("n,splits,grid", [(1, 4, 16), (2, 2, 128), (3, 1, 256), (4, 1, 324),
                                           (5, 19, 152), (6, 1, 256)])
def test_named_workload_plans(n, splits, grid):
    """E4M3 workloads (3, 5, 6) take the slot-split kernel, BF16 ones the
    dims-split kernel; both by the grid-mode rule."""
    p = plan(workload_args(n))
    kernel = B.KERNEL_TCGEN05_SLOT_SPLIT if workload_args(n).dtype == B.SMLA_E4M3 else B.KERNEL_TCGEN05
    assert (p["kernel"], p["num_splits"], p["grid"], p["ctas_per_split"], p["clusters"]) == \
        (kernel, splits, grid, 2, 0)


@pytest.mark.parametrize("n,grid,clusters", [(1, 16, 8), (2, 152, 76), (3, 152, 76), (4, 152, 76),
                                             (5, 152, 0), (6, 152, 76)])
def test_named_workload_balanced_plans(n, grid, clusters):
    a = workload_args(n)
    a.schedule = B.SCHEDULE_BALANCED
    p = plan(a)
    assert (p["kernel"], p["grid"], p["clusters"]) == (B.KERNEL_TCGEN05, grid, clusters)


def test_head_owned_form_is_opt_in_and_e4m3_only():
    """The head-owned softmax form runs only when asked for and only on E4M3
    rows; BF16 rows asking for it get the default tensor-core kernel.  It has
    no balanced mode: one cluster per (token, split), by the grid-mode rule."""
    ref = plan(args(128, 2176, schedule=B.SCHEDULE_BALANCED))
    ho = plan(args(128, 2176, kernel=B.KERNEL_TCGEN05_HEAD_OWNED, schedule=B.SCHEDULE_BALANCED))
    assert ref["kernel"] == B.KERNEL_TCGEN05 and ho["kernel"] == B.KERNEL_TCGEN05_HEAD_OWNED
    assert ref["clusters"] == 76 and ho["clusters"] == 0
    assert (ho["num_splits"], ho["grid"], ho["ctas_per_split"]) == (expected_tc_splits(128, 2176), 256, 2)
    bf = plan(args(32, 640, dtype=B.SMLA_BF16, kernel=B.KERNEL_TCGEN05_HEAD_OWNED, schedule=B.SCHEDULE_BALANCED))
    assert bf["kernel"] == B.KERNEL_TCGEN05 and bf["clusters"] == 76


def test_slot_split_form_is_the_e4m3_default():
    """The slot-split form runs on E4M3 rows only (BF16 rows asking for it get
    the dims-split kernel); it is what AUTO picks for E4M3 rows, except under
    the balanced schedule, which only the dims-split kernel runs.  Like the
    head-owned form it has no balanced mode and takes the grid-mode rule."""
    auto = plan(args(128, 2176))
    assert auto["kernel"] == B.KERNEL_TCGEN05_SLOT_SPLIT and auto["clusters"] == 0
    bal = plan(args(128, 2176, schedule=B.SCHEDULE_BALANCED))
    assert bal["kernel"] == B.KERNEL_TCGEN05 and bal["clusters"] == 76
    assert plan(args(32, 640, dtype=B.SMLA_BF16))["kernel"] == B.KERNEL_TCGEN05
    ss = plan(args(128, 2176, kernel=B.KERNEL_TCGEN05_SLOT_SPLIT, schedule=B.SCHEDULE_BALANCED))
    assert ss["kernel"] == B.KERNEL_TCGEN05_SLOT_SPLIT and ss["clusters"] == 0
    assert (ss["num_splits"], ss["grid"], ss["ctas_per_split"]) == (expected_tc_splits(128, 2176), 256, 2)
    assert ss["threads"] == 512 and ss["smem_bytes"] <= 232448
    for T, W_ in [(4, 16512), (32, 640), (1, 65536)]:
        p = plan(args(T, W_, kernel=B.KERNEL_TCGEN05_SLOT_SPLIT))
        assert p["kernel"] == B.KERNEL_TCGEN05_SLOT_SPLIT and p["num_splits"] == expected_tc_splits(T, W_)
    bf = plan(args(32, 640, dtype=B.SMLA_BF16, kernel=B.KERNEL_TCGEN05_SLOT_SPLIT))
    assert bf["kernel"] == B.KERNEL_TCGEN05


@pytest.mark.parametrize("T", [1, 2, 3, 75, 151, 152, 153, 301, 1000])
@pytest.mark.parametrize("W_", [128, 640, 2304, 2305, 16512])
@pytest.mark.parametrize("dtype", [B.SMLA_BF16, B.SMLA_E4M3])
def test_token_pair_plan_rule(T, W_, dtype):
    """The token-pair form: ceil(T / 2) units of two tokens, split by the
    grid-mode rule over units; the split partials stay per token."""
    for schedule in (B.SCHEDULE_AUTO, B.SCHEDULE_BALANCED):
        p = plan(args(T, W_, H=64, dtype=dtype, kernel=B.KERNEL_TCGEN05_TOKEN_PAIRS, schedule=schedule))
        U = (T + 1) // 2
        assert p["kernel"] == B.KERNEL_TCGEN05_TOKEN_PAIRS and p["clusters"] == 0
        S = p["num_splits"]
        # as many splits as keep one wave of units, at least 64 union columns
        # (up to 2W) per split, and at most 2304 columns of each token (1152
        # for E4M3, whose pairs run the slot-split kernel's pair form)
        cap = 1152 if dtype == B.SMLA_E4M3 else 2304
        want = min(GB300_SMS // 2 // U, math.ceil(2 * W_ / 64), 32)
        assert S == max(want, math.ceil(W_ / cap), 1)
        slot = plan(args(T, W_, dtype=B.SMLA_E4M3, kernel=B.KERNEL_TCGEN05_SLOT_SPLIT))
        if dtype == B.SMLA_E4M3:
            assert p["smem_bytes"] == slot["smem_bytes"]
        assert p["grid"] == 2 * U * S and p["ctas_per_split"] == 2
        assert p["workspace_bytes"] == (0 if S == 1 else workspace(T * 64 * S))
        assert p["threads"] == 512 and p["smem_bytes"] <= 232448


def test_auto_takes_token_pairs_for_e4m3_64_heads_past_a_wave():
    """AUTO: E4M3 rows with 64 heads, at most 1152 columns and more tokens
    than SM pairs run the slot-split kernel's token-pair form; otherwise the
    slot-split kernel (and BF16 rows the dims-split kernel)."""
    pairs = GB300_SMS // 2
    for T, W_, want in [(pairs + 1, 640, B.KERNEL_TCGEN05_TOKEN_PAIRS), (300, 1152, B.KERNEL_TCGEN05_TOKEN_PAIRS),
                        (pairs, 640, B.KERNEL_TCGEN05_SLOT_SPLIT), (300, 1153, B.KERNEL_TCGEN05_SLOT_SPLIT),
                        (300, 2176, B.KERNEL_TCGEN05_SLOT_SPLIT)]:
        p = plan(args(T, W_, H=64))
        assert p["kernel"] == want, (T, W_, p)
        if want == B.KERNEL_TCGEN05_TOKEN_PAIRS:
            assert p["grid"] == 2 * ((T + 1) // 2) * p["num_splits"]
    assert plan(args(300, 640, H=128))["kernel"] == B.KERNEL_TCGEN05_SLOT_SPLIT
    assert plan(args(300, 640, H=64, dtype=B.SMLA_BF16))["kernel"] == B.KERNEL_TCGEN05
    assert plan(args(300, 640, H=64, schedule=B.SCHEDULE_BALANCED))["kernel"] == B.KERNEL_TCGEN05


def test_token_pair_form_needs_64_heads():
    """H = 128 fills the MMA rows alone: a token-pair request runs the
    dims-split kernel."""
    for dtype in (B.SMLA_BF16, B.SMLA_E4M3):
        p = plan(args(77, 640, H=128, dtype=dtype, kernel=B.KERNEL_TCGEN05_TOKEN_PAIRS))
        assert p["kernel"] == B.KERNEL_TCGEN05 and p["grid"] == 2 * 77 * p["num_splits"]


def workspace(rows):
    return -(-rows * 512 * 2 // 256) * 256 + -(-rows * 4 // 256) * 256


@pytest.mark.parametrize("T", [1, 2, 3, 4, 7, 19, 38, 75, 76, 77, 128, 1000, 1064, 1065])
@pytest.mark.parametrize("W_", [128, 129, 256, 640, 2176, 2304, 2305, 4608, 16512, 65536])
@pytest.mark.parametrize("max_splits", [0, 1, 8])
@pytest.mark.parametrize("schedule", [B.SCHEDULE_AUTO, B.SCHEDULE_GRID, B.SCHEDULE_BALANCED])
def test_tc_plan_rule(T, W_, max_splits, schedule):
    p = plan(args(T, W_, max_splits=max_splits, schedule=schedule))
    P = expected_clusters(T, W_, max_splits=max_splits, schedule=schedule)
    assert p["clusters"] == P
    if P:
        # balanced mode: equal shares, pieces of cut tokens in the workspace
        assert p["num_splits"] == 1 and p["grid"] == 2 * P
        assert P <= GB300_SMS // 2 and (P == GB300_SMS // 2 or P == max(1, T * W_ // 64))
        rows = 2 * P * 128
        want = -(-rows * 1024 // 256) * 256 + -(-2 * rows * 4 // 256) * 256 + -(-2 * P * 4 // 256) * 256
        assert p["workspace_bytes"] == (want if P > 1 else 0)
        return
    S = p["num_splits"]
    assert S == expected_tc_splits(T, W_, max_splits)
    assert p["grid"] == T * S * 2
    assert S >= math.ceil(W_ / 2304)                       # no split stages more than 2304 columns
    if S > math.ceil(W_ / 2304):
        assert T * S <= GB300_SMS // 2                      # extra splits only while one wave holds
    # workspace: BF16 partials + fp32 LSEs, each 256-byte aligned; none for S = 1
    assert p["workspace_bytes"] == (0 if S == 1 else workspace(T * 128 * S))


def test_balanced_shares_are_whole_waves_of_one_cluster_per_pair():
    """Balanced mode uses every SM pair once the columns allow 64 per share,
    and never more clusters than pairs."""
    for sms in (16, 132, 148, 152):
        pairs = sms // 2
        bal = B.SCHEDULE_BALANCED
        assert plan(args(min(128, 14 * pairs), 2176, schedule=bal), sms)["clusters"] == pairs
        assert plan(args(1, 256, schedule=bal), sms)["clusters"] == min(pairs, 4)
        assert plan(args(14 * pairs + 1, 128, schedule=bal), sms)["clusters"] == 0   # beyond 14 tokens per pair
        assert plan(args(128, 2176), sms)["clusters"] == 0                           # the default schedule: grid


def test_sm_count_scales_the_split():
    a = args(4, 16512)
    assert plan(a, 152)["num_splits"] == 19
    assert plan(a, 304)["num_splits"] == 32                  # capped by the default max_splits
    assert plan(a, 16)["num_splits"] == 8                    # ceil(16512 / 2304) = 8 is the floor


def test_forced_splits():
    assert plan(args(3, 2176, num_splits=5))["num_splits"] == 5
    with pytest.raises(B.SmlaError) as e:
        plan(args(3, 4608 + 1, num_splits=2))                 # needs >= 3 splits of <= 2304 columns
    assert e.value.status == B.SMLA_ERR_INVALID_ARG and "num_splits 2 < 3" in str(e.value)


def test_cuda_core_rule():
    for T, W_, H in ((1, 2176, 128), (32, 640, 128), (128, 2176, 64), (4, 16512, 128)):
        p = plan(args(T, W_, H=H, kernel=B.KERNEL_CUDA_CORE))
        units = T * p["ctas_per_split"]
        want = min(math.ceil(GB300_SMS * 2 / units), math.ceil(W_ / 256), 32)
        assert p["kernel"] == B.KERNEL_CUDA_CORE and p["num_splits"] == max(want, 1)
        assert p["grid"] == T * p["num_splits"] * p["ctas_per_split"]


def test_bad_sm_count_and_null_plan():
    with pytest.raises(B.SmlaError) as e:
        plan(args(1, 256), sms=0)
    assert e.value.status == B.SMLA_ERR_INVALID_ARG and "sm_count" in str(e.value)
    assert B.lib().smla_plan_decode_for_sm_count(None, 152, None) == B.SMLA_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value", [("kernel", 6), ("kernel", -1), ("schedule", 3), ("schedule", -1)])
def test_unknown_kernel_or_schedule_is_an_error(field, value):
    a = args(8, 640)
    setattr(a, field, value)
    with pytest.raises(B.SmlaError) as e:
        plan(a)
    assert e.value.status == B.SMLA_ERR_INVALID_ARG and field in str(e.value)


def test_shape_errors_match_the_decode_call():
    a = args(1, 100)                                         # width < 128 SWA columns
    with pytest.raises(B.SmlaError) as e:
        plan(a)
    assert e.value.status == B.SMLA_ERR_INVALID_ARG and "width" in str(e.value)


@pytest.mark.gpu
def test_device_plan_equals_the_sm_count_plan():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for n in (1, 2, 3, 5):
        a = workload_args(n)
        assert B.smla_plan_decode(a, 0).as_dict() == B.smla_plan_decode_for_sm_count(a, sms).as_dict()


@pytest.mark.parametrize("dtype", [B.SMLA_PACKED_FP8, B.SMLA_NVFP4])
def test_packed_rows_plan(dtype):
    """Packed KV rows run the dims-split tensor-core kernel (the BF16 plan:
    grid schedule, its split rule, smem and workspace), whatever tensor-core
    form or schedule was asked for, and the CUDA-core kernel when that is
    asked for."""
    for T, W_ in [(128, 2176), (4, 16512), (2, 256)]:
        for kernel in (B.KERNEL_AUTO, B.KERNEL_TCGEN05, B.KERNEL_TCGEN05_HEAD_OWNED,
                       B.KERNEL_TCGEN05_SLOT_SPLIT, B.KERNEL_TCGEN05_TOKEN_PAIRS):
            for schedule in (B.SCHEDULE_AUTO, B.SCHEDULE_BALANCED):
                for H in (64, 128):
                    p = plan(args(T, W_, H=H, dtype=dtype, kernel=kernel, schedule=schedule))
                    ref = plan(args(T, W_, H=H, dtype=B.SMLA_BF16, kernel=B.KERNEL_TCGEN05,
                                    schedule=B.SCHEDULE_GRID))
                    assert p["kernel"] == B.KERNEL_TCGEN05 and p["clusters"] == 0
                    assert p == ref
        p = plan(args(T, W_, dtype=dtype, kernel=B.KERNEL_CUDA_CORE))
        assert p == plan(args(T, W_, dtype=B.SMLA_BF16, kernel=B.KERNEL_CUDA_CORE))


@pytest.mark.parametrize("dtype,row,align", [(B.SMLA_PACKED_FP8, 584, 8), (B.SMLA_NVFP4, 384, 16)])
def test_packed_row_strides(dtype, row, align):
    """Packed pools count their row strides in bytes: at least the row size
    and a multiple of 8 (packed FP8) or 16 (NVFP4) bytes."""
    for stride, ok in ((0, True), (row, True), (row + align, True), (row - align, False),
                       (row + align // 2, False), (512, row <= 512)):
        a = args(4, 256, dtype=dtype)
        a.swa_row_stride = a.comp_row_stride = stride
        if ok:
            plan(a)
        else:
            with pytest.raises(B.SmlaError) as e:
                plan(a)
            assert e.value.status == B.SMLA_ERR_INVALID_ARG and "strides" in str(e.value)


def test_unknown_dtype_is_an_error():
    a = args(4, 256)
    a.dtype = 4
    with pytest.raises(B.SmlaError) as e:
        plan(a)
    assert e.value.status == B.SMLA_ERR_INVALID_ARG and "dtype" in str(e.value)
