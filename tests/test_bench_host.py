"""Host checks of the benchmark's accounting: the slots it counts per token
(the basis of the algorithmic bytes and FLOPs behind every roofline number)
equal the oracle's slot lists, in the index and the page-table forms."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from oracle import oracle as orc  # noqa: E402
from sparse_mla_decode_token_gb300 import workloads as W  # noqa: E402


def oracle_counts(w, tokens):
    return np.array([len(orc.valid_slots(
        t, indices=w.indices, topk_lens=w.topk_lens, seq_lens=w.seq_lens,
        cum_seq_lens_q=w.cum_seq_lens_q, batch=w.batch, swa_rows=w.swa_kv.shape[0],
        comp_rows=w.comp_kv.shape[0], width=w.width, swa_topk_lens=w.swa_topk_lens,
        comp_block_tables=w.comp_block_tables, comp_page_size=w.comp_page_size,
        hca_seq_lens=w.hca_seq_lens, invalid_index="mask")) for t in tokens])


@pytest.mark.parametrize("n", [1, 2, 4, 6])
def test_slot_accounting_matches_oracle(n):
    w = W.config_workload(n)
    got = bench.valid_slots_per_token(w)
    tokens = range(w.sum_q) if w.sum_q <= 200 else range(0, w.sum_q, 7)
    np.testing.assert_array_equal(got[list(tokens)], oracle_counts(w, tokens))


def test_slot_accounting_page_table_edge_cases():
    """Footprints below 128, top-k cuts inside a page, windows 0 and past 128."""
    w = W.make_paged_workload(seed=3, dtype="bf16", batch=3, q_lens=[1, 2, 1], num_heads=64,
                              swa_rows=3 * 130 + 10, comp_pages=32, page_size=16, max_pages=20,
                              hca_seq_lens=[128 + 300, 100, 128 + 17], seq_lens=[5000, 90, 3000],
                              ring_len=130, topk_lens=[200, 140, 450, 129], swa_topk_lens=[0, 300, 64, 128],
                              varlen=True)
    np.testing.assert_array_equal(bench.valid_slots_per_token(w), oracle_counts(w, range(w.sum_q)))


def test_workload_config_names_the_page_table_form():
    cfg = bench.workload_config(W.config_workload(6), 6)
    assert cfg["workload"] == "paged_fp8_b128_h128"
    assert cfg["page_size"] == 128 and cfg["pages_per_token"] == 16 and cfg["index_width"] == 2176
    assert "page_size" not in bench.workload_config(W.config_workload(1), 1)


def test_recorded_traffic_needs_the_same_device_code_and_plan(monkeypatch):
    """A stored ncu traffic figure is reported only for the device code and
    launch plan it was captured on."""
    import json
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    name = "fp8_decode_b128_h128"
    plan = dict(rec[name]["plan"], workspace_bytes=0)
    want = rec[name]["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: rec[name]["kernel_sources_sha"])
    assert bench.recorded_traffic(name, plan) == want
    assert bench.recorded_traffic(name, dict(plan, num_splits=2)) is None
    assert bench.recorded_traffic(name, dict(plan, grid=plan["grid"] + 2)) is None
    assert bench.recorded_traffic("no_such_workload", plan) is None
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "0" * 16)
    assert bench.recorded_traffic(name, plan) is None
    value, note = bench.traffic_record(name, plan)
    assert value is None and rec[name]["kernel_sources_sha"] in note and "0" * 16 in note


def test_host_only_sources_hold_no_device_code():
    """Files left out of the device-code hash must not define device code."""
    csrc = os.path.join(ROOT, "sparse_mla_decode_token_gb300", "csrc")
    for f in bench.HOST_ONLY_SOURCES:
        code = bench.code_only(open(os.path.join(csrc, f)).read())
        for word in ("__global__", "__device__", "__constant__", "__shared__", "asm(", "asm volatile"):
            assert word not in code, (f, word)


def test_cpu_baseline_cycles_the_workload_until_its_budget():
    w = W.config_workload(1)                                  # 2 tokens: a fraction of a second
    done, seconds = bench.time_oracle(w, 0.3)
    assert done > w.sum_q and seconds >= 0.3
    done, _ = bench.time_oracle(w, 1e9, max_tokens=3)
    assert done == 3


def test_clock_summary_reports_median_max_and_throttle_reasons(tmp_path):
    """The clocks entry of the JSON line from nvidia-smi's CSV samples
    (noheader, nounits): the median SM clock under load, the maximum, and
    every throttle reason seen Active (a run with a slowdown is rejected)."""
    csv = tmp_path / "clocks.csv"
    na = "Not Active"
    csv.write_text("\n".join([
        f"0, 2070, 2070, 610.5, 0x0000000000000000, {na}, {na}, {na}, {na}",
        f"0, 1900, 2070, 1395.0, 0x0000000000000004, {na}, {na}, {na}, Active",
        f"0, 2000, 2070, 700.0, 0x0000000000000008, Active, {na}, {na}, {na}",
        f"0, 1980, 2070, [N/A], 0x0000000000000000, {na}, {na}, {na}, {na}",   # unparsable: skipped
        "garbage line",
    ]) + "\n")
    s = bench.ClockSampler(0)
    s.proc, s.path = object(), str(csv)
    out = s.summary()
    assert out["sm_mhz"] == 2000 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["power_w_max"] == 1395.0
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    s2 = bench.ClockSampler(0)
    assert s2.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_roofline_peaks_come_from_the_measured_file_else_the_fallback(monkeypatch, tmp_path):
    import json
    rec = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    assert bench.peaks() == (rec["hbm_gbs"], rec["bf16_tflops"], "measured")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))                  # no measured file there
    assert bench.peaks() == (6800.0, 1900.0, "fallback")              # the recipe's fallback figures


def test_fp8_tensor_peak_comes_from_the_measured_record(monkeypatch, tmp_path):
    """The FP8 tensor peak is the E4M3 tcgen05 burst rate recorded in
    profiles/mma_peak.json; without that record it falls back to twice the
    BF16 peak."""
    import json
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "mma_peak.json")))
    tf, src = bench.fp8_tensor_peak(1000.0)
    assert tf == rec["e4m3_tflops"] and "measured" in src
    assert rec["e4m3_tflops"] > rec["bf16_tflops"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    tf, src = bench.fp8_tensor_peak(1000.0)
    assert tf == 2000.0 and "nominal" in src


def oracle_union_rows(w, S):
    """Brute force from the oracle's slot lists: per (token pair, split) the
    distinct (pool, row) pairs, or every slot when a token reads a row twice."""
    per = -(-w.width // S)
    if w.paged:
        per = -(-per // 64) * 64
    slots = [orc.valid_slots(
        t, indices=w.indices, topk_lens=w.topk_lens, seq_lens=w.seq_lens,
        cum_seq_lens_q=w.cum_seq_lens_q, batch=w.batch, swa_rows=w.swa_kv.shape[0],
        comp_rows=w.comp_kv.shape[0], width=w.width, swa_topk_lens=w.swa_topk_lens,
        comp_block_tables=w.comp_block_tables, comp_page_size=w.comp_page_size,
        hca_seq_lens=w.hca_seq_lens, invalid_index="mask") for t in range(w.sum_q)]
    total = 0
    for u in range(0, w.sum_q, 2):
        for s in range(S):
            lists = [[(p, r) for (j, p, r) in slots[t] if s * per <= j < s * per + per]
                     for t in range(u, min(u + 2, w.sum_q))]
            if any(len(set(x)) < len(x) for x in lists):
                total += sum(len(x) for x in lists)
            else:
                total += len(set(lists[0]) | (set(lists[1]) if len(lists) > 1 else set()))
    return total


@pytest.mark.parametrize("S", [1, 2, 3])
def test_token_pair_rows_match_the_oracle_slot_lists(S):
    """Rows the token-pair kernel gathers (bench accounting) = brute-force
    unions of the oracle's slot lists: shared SWA windows of a request's
    consecutive tokens, copied and shuffled compressed rows, a row read twice,
    equal row numbers in the two pools, an odd token count."""
    rng = np.random.default_rng(5)
    w = W.make_workload(seed=5, dtype="bf16", batch=4, q_lens=[2, 3, 1, 3], num_heads=64,
                        swa_rows=4 * 128 + 64, comp_rows=1024, width=128 + 200,
                        seq_lens=[3000, 60, 4000, 5000], ring_len=128,
                        topk_lens=rng.integers(100, 329, size=9), varlen=True)
    w.indices[1, 128:] = w.indices[0, 128:]
    w.indices[3, 128:] = rng.permutation(w.indices[2, 128:])
    w.indices[5, 128:228] = w.indices[4, :100]            # SWA row numbers in compressed columns
    w.indices[6, 130] = w.indices[6, 131]                 # a row read twice
    got = bench.token_pair_rows(w, S)
    assert got == oracle_union_rows(w, S)
    assert got < bench.valid_slots_per_token(w).sum()


def test_token_pair_rows_page_table_form():
    w = W.make_paged_workload(seed=3, dtype="bf16", batch=3, q_lens=[2, 3, 2], num_heads=64,
                              swa_rows=3 * 130 + 10, comp_pages=32, page_size=16, max_pages=20,
                              hca_seq_lens=[128 + 300, 100, 128 + 17], seq_lens=[5000, 90, 3000],
                              ring_len=130, topk_lens=[200, 140, 450, 129, 300, 300, 180],
                              swa_topk_lens=[0, 128, 64, 128, 100, 128, 128], varlen=True)
    for S in (1, 2):
        assert bench.token_pair_rows(w, S) == oracle_union_rows(w, S)


def test_workload_4_token_pairs_gather_fewer_rows():
    """The varlen workload (64 requests of 1-4 tokens, H = 64): pairs of a
    request's consecutive tokens share their SWA window."""
    w = W.config_workload(4)
    assert bench.token_pair_rows(w, 1) < bench.valid_slots_per_token(w).sum()
