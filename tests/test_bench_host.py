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
