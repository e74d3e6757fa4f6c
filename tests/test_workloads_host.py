"""The six named synthetic workloads have the shapes, value distributions and
index structure their recipe states (CPU only).

The recipe: N(0, 1) query and pools, FP8 with per-tensor scales amax / 448
and bmm1 = softmax_scale * q_scale * kv_scale, bmm2 = kv_scale (vLLM
DeepseekV4FlashInferMLAAttention, FP8 scale folding); 128 SWA columns holding
the request's ring rows in position order, then unique random compressed rows
(or -1 padding); lengths and sinks per workload.  Values are decoded here with
torch's own BF16 / E4M3 types, independently of the oracle and the CUDA path.
"""
import math

import numpy as np
import pytest
import torch

from sparse_mla_decode_token_gb300 import workloads as W

SWA = 128

# n: (name, dtype, batch, heads, width, swa_rows, comp_rows, seq_lens range, sinks)
RECIPE = {
    1: ("tiny_bf16_h64", "bf16", 2, 64, 256, 256, 512, (4096, 4096), False),
    2: ("bf16_decode_b32_h128", "bf16", 32, 128, 640, 32 * 128, 65536, (4096, 32768), True),
    3: ("fp8_decode_b128_h128", "e4m3", 128, 128, 2176, 128 * 128, 262144, (8192, 65536), False),
    4: ("varlen_spec_bf16_h64", "bf16", 64, 64, 1152, 64 * 256, 65536, (4096, 32768), True),
    5: ("long_splitk_fp8_b4_h128", "e4m3", 4, 128, 128 + 16384, 4 * 128, 1 << 20, (1 << 20, 1 << 20), True),
    6: ("paged_fp8_b128_h128", "e4m3", 128, 128, 2176, 128 * 128, 262144, (8192, 65536), False),
}


def decoded(bits: np.ndarray, dtype: str, scale: float) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits))
    if dtype == "bf16":
        return t.view(torch.int16).view(torch.bfloat16).to(torch.float64)
    return t.view(torch.float8_e4m3fn).to(torch.float64) * scale


def check_standard_normal(x: torch.Tensor, tol_std: float):
    x = x.flatten()[: 1 << 22]
    assert abs(float(x.mean())) < 0.01
    assert abs(float(x.std()) - 1.0) < tol_std


@pytest.mark.parametrize("n", sorted(RECIPE))
def test_named_workload_matches_its_recipe(n):
    name, dtype, batch, H, width, swa_rows, comp_rows, (lo, hi), sinks = RECIPE[n]
    w = W.config_workload(n)
    paged = w.comp_block_tables is not None
    assert (w.name, w.dtype, w.batch, w.num_heads) == (name, dtype, batch, H)
    assert w.width == width
    assert w.swa_kv.shape == (swa_rows, 512) and w.comp_kv.shape == (comp_rows, 512)
    assert (w.sinks is not None) == sinks and (not sinks or w.sinks.shape == (H,))
    assert int(w.seq_lens.min()) >= lo and int(w.seq_lens.max()) <= hi

    # query lengths: one token per request except the varlen workload (1..4)
    if n == 4:
        q_lens = np.diff(w.cum_seq_lens_q)
        assert q_lens.min() >= 1 and q_lens.max() <= 4 and len(q_lens) == batch
        assert len(set(q_lens.tolist())) > 1
    else:
        assert w.cum_seq_lens_q is None
        q_lens = np.ones(batch, np.int64)
    T = int(q_lens.sum())
    assert w.q.shape == (T, H, 512) and w.sum_q == T

    # values: N(0, 1); FP8 per-tensor scales amax / 448, folded into bmm1 / bmm2
    tol = 0.01 if dtype == "bf16" else 0.03
    check_standard_normal(decoded(w.q, dtype, w.q_scale), tol)
    check_standard_normal(decoded(w.comp_kv[: 1 << 13], dtype, w.kv_scale), tol)
    check_standard_normal(decoded(w.swa_kv[: 1 << 13], dtype, w.kv_scale), tol)
    if dtype == "e4m3":
        assert float(decoded(w.q, dtype, 1.0).abs().max()) == 448.0
        kv_amax = max(float(decoded(w.swa_kv, dtype, 1.0).abs().max()),
                      float(decoded(w.comp_kv, dtype, 1.0).abs().max()))
        assert kv_amax == 448.0
    else:
        assert w.q_scale == w.kv_scale == 1.0
    assert w.bmm1_scale == float(np.float32(w.q_scale * w.kv_scale / math.sqrt(512)))
    assert w.bmm2_scale == float(np.float32(w.kv_scale))

    # SWA columns: the request's ring rows in position order (every token here
    # is at position >= 127, so all 128 columns are filled)
    ring = swa_rows // batch
    req = np.repeat(np.arange(batch), q_lens)
    pos = np.repeat(w.seq_lens.astype(np.int64), q_lens) - np.repeat(q_lens, q_lens) + \
        np.concatenate([np.arange(q) for q in q_lens])
    assert pos.min() >= SWA - 1
    want_swa = req[:, None] * ring + (pos[:, None] - (SWA - 1) + np.arange(SWA)[None, :]) % ring
    np.testing.assert_array_equal(w.indices[:, :SWA], want_swa)

    if paged:
        # 16 distinct random pages of 128 rows per request, 2048 slots each
        assert w.indices.shape == (T, SWA)
        assert w.comp_page_size == 128 and w.comp_block_tables.shape == (T, 16)
        assert np.all(w.hca_seq_lens == SWA + 2048)
        for t in range(T):
            pages = w.comp_block_tables[t]
            assert len(set(pages.tolist())) == 16 and pages.min() >= 0 and pages.max() < comp_rows // 128
        assert np.all(w.topk_lens == 2176) and w.swa_topk_lens is None
        return

    comp = w.indices[:, SWA:]
    assert comp.shape == (T, width - SWA)
    valid = comp != -1
    n_valid = valid.sum(axis=1)
    for t in range(T):
        k = int(n_valid[t])
        assert valid[t, :k].all() and not valid[t, k:].any()          # valid rows, then -1
        rows = comp[t, :k]
        assert rows.min() >= 0 and rows.max() < comp_rows and len(np.unique(rows)) == k
    if n == 2:
        assert n_valid.min() >= 256 and n_valid.max() <= 512
        even = np.arange(T) % 2 == 0
        assert np.all(w.topk_lens[even] == 640)
        np.testing.assert_array_equal(w.topk_lens[~even], SWA + n_valid[~even])
    else:
        assert np.all(n_valid == width - SWA)
    if n in (1, 4):
        assert w.topk_lens.min() >= SWA + 1 and w.topk_lens.max() <= width
        assert len(np.unique(w.topk_lens)) > 1
    if n in (3, 5):
        assert np.all(w.topk_lens == width)


def test_named_workloads_are_deterministic():
    a, b = W.config_workload(1), W.config_workload(1)
    for f in ("q", "swa_kv", "comp_kv", "indices", "topk_lens", "seq_lens"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
