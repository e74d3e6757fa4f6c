"""Pins for the CPU oracle: closed forms, library special cases and invariants.

Each test ties the oracle to something other than itself -- a value fixed by
the mathematics, a library routine on a case that reduces to it, or an
invariant stated by the documentation pages -- so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import oracle as orc

HERE = os.path.dirname(os.path.abspath(__file__))
LOG2E = 1.0 / math.log(2.0)


# ---------------------------------------------------------------- helpers

def bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_round(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def e4m3_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).clamp(-448, 448)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def case(*, H=4, q=None, swa=None, comp=None, indices, topk_lens=None, seq_lens=(100000,),
         cum=None, sinks=None, bmm1=0.125, bmm2=1.0, dtype="bf16", batch=None, **kw):
    enc = bf16_bits if dtype == "bf16" else e4m3_bits
    indices = np.asarray(indices, dtype=np.int32)
    if indices.ndim == 1:
        indices = indices[None, :]
    T = indices.shape[0]
    q = np.zeros((T, H, 512), np.float32) if q is None else np.asarray(q, np.float32)
    swa = np.zeros((4, 512), np.float32) if swa is None else np.asarray(swa, np.float32)
    comp = np.zeros((4, 512), np.float32) if comp is None else np.asarray(comp, np.float32)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    batch = len(seq_lens) if batch is None else batch
    return orc.sparse_mla_decode(
        dtype=dtype, batch=batch, q=enc(q), swa_kv=enc(swa), comp_kv=enc(comp),
        indices=indices, topk_lens=None if topk_lens is None else np.asarray(topk_lens, np.int32),
        seq_lens=seq_lens, cum_seq_lens_q=None if cum is None else np.asarray(cum, np.int32),
        sinks=None if sinks is None else np.asarray(sinks, np.float32),
        bmm1_scale=bmm1, bmm2_scale=bmm2, **kw)


def table(swa_cols, comp_cols, width=None):
    """Index row: SWA columns padded with -1 to 128, then compressed columns."""
    row = list(swa_cols) + [-1] * (128 - len(swa_cols)) + list(comp_cols)
    if width is not None:
        row += [-1] * (width - len(row))
    return row


def rand_rows(rng, n, scale=1.0):
    return bf16_round(rng.standard_normal((n, 512)) * scale)


# ------------------------------------------------------- element formats

def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_bf16_decode_matches_torch_for_every_code():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = orc.bf16_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_page_constants():
    c = json.load(open(os.path.join(HERE, "golden", "page_constants.json")))
    assert orc.HEAD_DIM == c["head_dim"]["value"] == c["nope_dim"]["value"] + c["rope_dim"]["value"]
    assert orc.SWA_COLS == c["swa_columns"]["value"]
    assert c["lse_base"]["value"] == 2 and c["masked_index"]["value"] == -1


# ------------------------------------------- whole formula vs a library

@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_dense_case_equals_torch_sdpa(dtype):
    """All slots selected, identity indices: plain dense attention (library routine)."""
    rng = np.random.default_rng(1)
    H, n_swa, n_comp = 8, 128, 37
    qf = rng.standard_normal((1, H, 512)) * (1.0 if dtype == "bf16" else 20.0)
    swa = rng.standard_normal((n_swa, 512)) * (1.0 if dtype == "bf16" else 20.0)
    comp = rng.standard_normal((n_comp, 512)) * (1.0 if dtype == "bf16" else 20.0)
    bmm1, bmm2 = 0.0441941738, 0.75
    idx = table(range(n_swa), range(n_comp))
    o, lse = case(H=H, q=qf, swa=swa, comp=comp, indices=idx, bmm1=bmm1, bmm2=bmm2, dtype=dtype)
    # decode the same bits with torch itself, then run torch's SDPA in float64
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float8_e4m3fn
    def dec(x):
        t = torch.as_tensor(np.asarray(x, np.float32))
        if dtype == "e4m3":
            t = t.clamp(-448, 448)
        return t.to(tdt).to(torch.float64)
    Q = dec(qf)[0][None]                                  # [1, H, 512]
    K = torch.cat([dec(swa), dec(comp)])[None, None]      # [1, 1, n, 512]
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q[:, :, None, :], K.expand(1, H, -1, -1),
        K.expand(1, H, -1, -1), scale=bmm1)[0, :, 0, :] * bmm2
    np.testing.assert_allclose(o[0], ref.numpy(), rtol=1e-11, atol=1e-12)
    logits = (Q[0] @ K[0, 0].T * bmm1).numpy()
    from scipy.special import logsumexp
    np.testing.assert_allclose(lse[0], logsumexp(logits, axis=1) / math.log(2), rtol=0, atol=1e-11)


# ---------------------------------------------------------- closed forms

def test_two_slot_worked_example():
    """q = 2 e0, rows e0 and e1, bmm1 = 1/2: logits 1 and 0.

    softmax weights e/(1+e) and 1/(1+e); O = those weights on dims 0 and 1;
    LSE2 = log2(1 + e).
    """
    q = np.zeros((1, 1, 512)); q[0, 0, 0] = 2.0
    swa = np.zeros((16, 512)); swa[5, 0] = 1.0; swa[9, 1] = 1.0
    o, lse = case(H=1, q=q, swa=swa, indices=table([5, 9], []), bmm1=0.5, bmm2=1.0)
    e = math.e
    assert o[0, 0, 0] == pytest.approx(e / (1 + e), abs=1e-15)
    assert o[0, 0, 1] == pytest.approx(1 / (1 + e), abs=1e-15)
    assert np.count_nonzero(o[0, 0, 2:]) == 0
    assert lse[0, 0] == pytest.approx(math.log2(1 + e), abs=1e-15)


def test_single_valid_slot_returns_row_times_bmm2():
    rng = np.random.default_rng(2)
    H = 6
    qf = rng.standard_normal((1, H, 512))
    comp = rand_rows(rng, 8)
    sinks = rng.standard_normal(H).astype(np.float32)
    idx = table([], [-1, 3, -1], width=140)
    bmm1, bmm2 = 0.03, 1.7
    o, lse = case(H=H, q=qf, comp=comp, indices=idx, bmm1=bmm1, bmm2=bmm2)
    qd = bf16_round(qf)[0]
    l = bmm1 * qd @ comp[3]                                   # [H]
    np.testing.assert_allclose(o[0], bmm2 * np.tile(comp[3], (H, 1)), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse[0], l * LOG2E, rtol=1e-13, atol=1e-13)
    o_s, lse_s = case(H=H, q=qf, comp=comp, indices=idx, bmm1=bmm1, bmm2=bmm2, sinks=sinks)
    w = np.exp(l) / (np.exp(l) + np.exp(sinks.astype(np.float64)))
    np.testing.assert_allclose(o_s[0], bmm2 * w[:, None] * comp[3][None], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse_s[0], lse[0], rtol=0, atol=0)


def test_zero_query_gives_mean_and_log2_n():
    rng = np.random.default_rng(3)
    H, n_swa, n_comp = 3, 5, 9
    swa, comp = rand_rows(rng, 10), rand_rows(rng, 20)
    sw, cp = [1, 7, 2, 0, 9], [4, 19, 3, 11, 12, 5, 6, 0, 8]
    o, lse = case(H=H, swa=swa, comp=comp, indices=table(sw, cp), bmm2=2.5)
    mean = (swa[sw].sum(0) + comp[cp].sum(0)) / (n_swa + n_comp)
    np.testing.assert_allclose(o[0], 2.5 * np.tile(mean, (H, 1)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log2(n_swa + n_comp), rtol=0, atol=1e-14)
    sinks = np.array([0.0, 1.5, -2.0], np.float32)
    o2, lse2 = case(H=H, swa=swa, comp=comp, indices=table(sw, cp), bmm2=2.5, sinks=sinks)
    n = n_swa + n_comp
    f = n / (n + np.exp(sinks.astype(np.float64)))
    np.testing.assert_allclose(o2[0], 2.5 * f[:, None] * mean[None], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse2[0], lse[0], atol=0)


def test_equal_logit_sink_closed_form():
    """Every selected row identical => equal logits l; O = row*bmm2*n/(n + e^{sink - l})."""
    rng = np.random.default_rng(4)
    H = 5
    row = rand_rows(rng, 1)[0]
    comp = np.tile(row, (12, 1))
    qf = rng.standard_normal((1, H, 512))
    sinks = rng.standard_normal(H).astype(np.float32)
    bmm1, bmm2, n = 0.05, 0.5, 12
    o, lse = case(H=H, q=qf, comp=comp, indices=table([], range(12)), sinks=sinks, bmm1=bmm1, bmm2=bmm2)
    l = bmm1 * bf16_round(qf)[0] @ row
    f = n / (n + np.exp(sinks.astype(np.float64) - l))
    np.testing.assert_allclose(o[0], bmm2 * f[:, None] * row[None], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[0], math.log2(n) + l * LOG2E, rtol=1e-13, atol=1e-13)


def test_combine_of_two_partials_closed_form():
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal((1, 512)), rng.standard_normal((1, 512))
    L1, L2 = 3.25, 1.5
    o, lse = orc.combine_partials(np.stack([a, b]), np.array([[L1], [L2]]), 1.0, None)
    w1, w2 = 2.0 ** L1, 2.0 ** L2
    np.testing.assert_allclose(o, (w1 * a + w2 * b) / (w1 + w2), rtol=1e-13, atol=1e-15)
    assert lse[0] == pytest.approx(math.log2(w1 + w2), abs=1e-14)
    o, lse = orc.combine_partials(np.stack([a, b]), np.array([[-np.inf], [L2]]), 2.0, None)
    np.testing.assert_allclose(o, 2.0 * b, rtol=1e-15)
    assert lse[0] == L2


def test_fully_masked_token_is_zero_with_minus_inf_lse():
    o, lse = case(H=2, indices=table([-1, -1], [-1]), sinks=[0.5, -0.5])
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    o, lse = case(H=2, indices=table([1], [2]), topk_lens=[0])
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_duplicate_index_counts_twice():
    q = np.zeros((1, 1, 512)); q[0, 0, 0] = 1.0
    comp = np.zeros((4, 512)); comp[1, 0] = 1.0; comp[2, 1] = 1.0
    o, lse = case(H=1, q=q, comp=comp, indices=table([], [1, 1, 2]), bmm1=1.0)
    e = math.e
    assert o[0, 0, 0] == pytest.approx(2 * e / (2 * e + 1), abs=1e-15)
    assert o[0, 0, 1] == pytest.approx(1 / (2 * e + 1), abs=1e-15)
    assert lse[0, 0] == pytest.approx(math.log2(2 * e + 1), abs=1e-15)


def test_dominant_logit_selects_its_row_without_overflow():
    """Logits near 1e3 (e^1000 overflows float64): the largest logit's row
    takes all the weight; O = that row * bmm2, LSE2 = its logit in base 2."""
    q = np.zeros((1, 1, 512)); q[0, 0, 0] = 64.0
    comp = np.zeros((8, 512))
    comp[2, 0], comp[5, 0], comp[6, 0] = 16.0, 15.0, 14.0          # logits 1024, 960, 896 (bmm1 = 1)
    comp[2, 1], comp[5, 2] = 3.0, 5.0
    o, lse = case(H=1, q=q, comp=comp, indices=table([], [5, 2, 6]), bmm1=1.0, bmm2=0.5)
    assert np.all(np.isfinite(o)) and np.isfinite(lse[0, 0])
    np.testing.assert_allclose(o[0, 0], 0.5 * comp[2], rtol=0, atol=1e-25)
    assert lse[0, 0] == pytest.approx(1024.0 * LOG2E, rel=1e-15)


def test_sink_limits():
    """A very negative sink is no sink; a very large one sends O to 0 while
    the LSE (sink excluded) stays.  Sinks of +-600 keep e^{sink - max logit}
    inside float64's range, so no step relies on overflow."""
    rng = np.random.default_rng(12)
    q, swa, comp, idx = _random_case(rng, T=1)
    kw = dict(H=4, q=q, swa=swa, comp=comp, indices=idx)
    o0, l0 = case(**kw)
    o1, l1 = case(sinks=np.full(4, -600.0, np.float32), **kw)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
    o2, l2 = case(sinks=np.full(4, 600.0, np.float32), **kw)
    assert 0 < np.abs(o2).max() < 1e-240
    np.testing.assert_array_equal(l0, l2)


def test_output_is_linear_in_bmm2_and_lse_ignores_it():
    rng = np.random.default_rng(13)
    q, swa, comp, idx = _random_case(rng, T=2)
    kw = dict(H=4, q=q, swa=swa, comp=comp, indices=idx, seq_lens=[10 ** 6] * 2,
              sinks=np.array([0.3, -1.0, 2.0, 0.0], np.float32))
    o1, l1 = case(bmm2=1.0, **kw)
    o3, l3 = case(bmm2=3.0, **kw)
    np.testing.assert_allclose(o3, 3.0 * o1, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(l1, l3)


def test_power_of_two_query_scale_trades_with_bmm1():
    """BF16 q * 2 is exact, so (2q, bmm1 / 2) gives bit-identical logits."""
    rng = np.random.default_rng(14)
    q, swa, comp, idx = _random_case(rng, T=1)
    kw = dict(H=4, swa=swa, comp=comp, indices=idx, sinks=np.array([0.5, 0.0, -0.5, 1.0], np.float32))
    qb = bf16_round(q)
    o1, l1 = case(q=qb, bmm1=0.125, **kw)
    o2, l2 = case(q=2.0 * qb, bmm1=0.0625, **kw)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    o3, _ = case(q=qb, bmm1=0.0625, **kw)                 # and bmm1 does matter
    assert np.abs(o3 - o1).max() > 1e-6


# ------------------------------------------------------------ invariants

def _random_case(rng, T=3, H=4, n_comp=40, width=128 + 64, comp_rows=100):
    q = rng.standard_normal((T, H, 512))
    swa = rand_rows(rng, 128 * T)
    comp = rand_rows(rng, comp_rows)
    idx = np.full((T, width), -1, np.int32)
    for t in range(T):
        idx[t, :128] = 128 * t + rng.permutation(128)
        idx[t, 128:128 + n_comp] = rng.choice(comp_rows, n_comp, replace=False)
    return q, swa, comp, idx


def test_minus_one_equals_dropping_the_column():
    rng = np.random.default_rng(6)
    q, swa, comp, idx = _random_case(rng)
    sinks = rng.standard_normal(4).astype(np.float32)
    T = idx.shape[0]
    kw = dict(H=4, q=q, swa=swa, comp=comp, seq_lens=[10 ** 6] * T, sinks=sinks)
    holed = idx.copy()
    holed[:, [3, 77, 130, 141, 150]] = -1
    o1, l1 = case(indices=holed, **kw)
    # drop the compressed holes by shifting left; SWA holes stay -1 in place
    dropped = np.full_like(idx, -1)
    for t in range(T):
        dropped[t, :128] = holed[t, :128]
        keep = [c for c in holed[t, 128:] if c != -1]
        dropped[t, 128:128 + len(keep)] = keep
    o2, l2 = case(indices=dropped, **kw)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-13)
    # and a hole changes the result relative to no hole
    o3, _ = case(indices=idx, **kw)
    assert np.abs(o3 - o1).max() > 1e-6


def test_topk_lens_mask_equals_minus_one_mask():
    rng = np.random.default_rng(7)
    q, swa, comp, idx = _random_case(rng)
    T = idx.shape[0]
    lens = np.array([150, 128, 170])
    kw = dict(H=4, q=q, swa=swa, comp=comp, seq_lens=[10 ** 6] * T)
    o1, l1 = case(indices=idx, topk_lens=lens, **kw)
    cut = idx.copy()
    for t in range(T):
        cut[t, lens[t]:] = -1
    o2, l2 = case(indices=cut, **kw)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # out-of-range lens clamp to [0, W]
    o3, _ = case(indices=idx, topk_lens=[10 ** 6, -5, 10 ** 6], **kw)
    o4, _ = case(indices=idx, **kw)
    np.testing.assert_array_equal(o3[[0, 2]], o4[[0, 2]])
    assert np.all(o3[1] == 0)


def test_permutation_invariance():
    rng = np.random.default_rng(8)
    q, swa, comp, idx = _random_case(rng)
    T = idx.shape[0]
    sinks = rng.standard_normal(4).astype(np.float32)
    kw = dict(H=4, q=q, swa=swa, comp=comp, seq_lens=[10 ** 6] * T, sinks=sinks)
    o1, l1 = case(indices=idx, **kw)
    perm = idx.copy()
    for t in range(T):
        perm[t, :128] = rng.permutation(perm[t, :128])
        perm[t, 128:168] = rng.permutation(perm[t, 128:168])
    o2, l2 = case(indices=perm, **kw)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_split_combine_matches_unsplit(splits):
    rng = np.random.default_rng(9)
    q, swa, comp, idx = _random_case(rng)
    T = idx.shape[0]
    sinks = rng.standard_normal(4).astype(np.float32)
    kw = dict(H=4, q=q, swa=swa, comp=comp, seq_lens=[10 ** 6] * T, sinks=sinks,
              topk_lens=[192, 140, 128], bmm2=1.3)
    o1, l1 = case(indices=idx, **kw)
    o2, l2 = case(indices=idx, splits=splits, **kw)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-12)


def test_swa_window_reading():
    """Reading of the SWA window: only the first min(128, pos + 1) SWA columns count."""
    rng = np.random.default_rng(10)
    q, swa, comp, idx = _random_case(rng, T=1)
    # pos = seq_len - q_len + i = 40 - 1 + 0 = 39 -> 40 SWA columns
    o1, l1 = case(H=4, q=q, swa=swa, comp=comp, indices=idx, seq_lens=[40])
    cut = idx.copy()
    cut[0, 40:128] = -1
    o2, l2 = case(H=4, q=q, swa=swa, comp=comp, indices=cut, seq_lens=[10 ** 6])
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_varlen_right_aligned_positions():
    cum = np.array([0, 2, 3, 7], np.int32)
    got = [orc.token_request(t, 7, 3, cum) for t in range(7)]
    assert got == [(0, 0, 2), (0, 1, 2), (1, 0, 1), (2, 0, 4), (2, 1, 4), (2, 2, 4), (2, 3, 4)]
    seq = np.array([10, 5, 100], np.int32)
    assert [orc.token_position(t, 7, 3, cum, seq) for t in range(7)] == [8, 9, 4, 96, 97, 98, 99]
    # dense query: q_len = sum_q / batch
    assert [orc.token_request(t, 6, 2, None) for t in range(6)] == [
        (0, 0, 3), (0, 1, 3), (0, 2, 3), (1, 0, 3), (1, 1, 3), (1, 2, 3)]


def test_invalid_index_raises_or_masks():
    with pytest.raises(IndexError):
        case(H=1, indices=table([1], [99]))
    o1, l1 = case(H=1, indices=table([1], [99, 2]), invalid_index="mask")
    o2, l2 = case(H=1, indices=table([1], [-1, 2]))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_lse_with_sink_reading_differs_only_in_lse():
    rng = np.random.default_rng(11)
    q, swa, comp, idx = _random_case(rng, T=1)
    sinks = np.array([1.0, 2.0, -1.0, 0.0], np.float32)
    kw = dict(H=4, q=q, swa=swa, comp=comp, indices=idx, sinks=sinks)
    o1, l1 = case(**kw)
    o2, l2 = case(lse_with_sink=True, **kw)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_allclose(l2, np.logaddexp2(l1, sinks * LOG2E), rtol=1e-11)


# ---------------------------------------------------------------- page-table form

def _golden_page_table():
    with open(os.path.join(HERE, "golden", "page_table_expansion.json")) as f:
        return json.load(f)


def test_page_table_slots_golden():
    """Hand-worked slot lists of the page-table form (fixture cites its rules)."""
    g = _golden_page_table()
    T = len(g["block_tables"])
    indices = np.array([[200 + 128 * t + j for j in range(128)] for t in range(T)], dtype=np.int32)
    for e in g["expected"]:
        t = e["token"]
        got = orc.valid_slots(t, indices=indices, topk_lens=np.asarray(g["sparse_topk_lens"]),
                              seq_lens=np.full(g["batch"], 100000), cum_seq_lens_q=None,
                              batch=g["batch"], swa_rows=g["swa_rows"], comp_rows=g["comp_rows"],
                              width=g["width"], swa_topk_lens=np.asarray(g["swa_topk_lens"]),
                              comp_block_tables=np.asarray(g["block_tables"], dtype=np.int32),
                              comp_page_size=g["page_size"], hca_seq_lens=np.asarray(g["hca_seq_lens"]))
        if e.get("swa_all"):
            want = [(j, "swa", 200 + 128 * t + j) for j in range(128)]
        else:
            want = [tuple(x) for x in e["slots"]]
        assert got == want, (t, got, want)


def test_page_table_is_indexed_by_token():
    """Hand-worked: the table has one row per token, so two tokens of one
    request may list different pages and each reads its own.

    Varlen query cum = [0, 2, 3]: tokens 0 and 1 belong to request 0 (3
    compressed slots: hca_seq_lens 131 - 128), token 2 to request 1 (2 slots).
    Page size 2, tables t0 [4, 1], t1 [0, 6], t2 [3, 5]; slot c is row
    table[c // 2] * 2 + c % 2:
      t0: rows 8, 9 (page 4), 2 (page 1)
      t1: rows 0, 1 (page 0), 12 (page 6)
      t2: rows 6, 7 (page 3); its second page lies past the footprint.
    """
    tables = np.array([[4, 1], [0, 6], [3, 5]], np.int32)
    want = {0: [8, 9, 2], 1: [0, 1, 12], 2: [6, 7]}
    for t, rows in want.items():
        got = orc.valid_slots(t, indices=np.zeros((3, 128), np.int32), topk_lens=None,
                              seq_lens=np.array([9000, 9000]), cum_seq_lens_q=np.array([0, 2, 3]),
                              batch=2, swa_rows=8, comp_rows=14, width=131,
                              swa_topk_lens=np.zeros(3, np.int32), comp_block_tables=tables,
                              comp_page_size=2, hca_seq_lens=np.array([131, 130]))
        assert got == [(128 + c, "comp", r) for c, r in enumerate(rows)], (t, got)


def test_page_table_single_slot_closed_form():
    """One page-table slot: O = row * bmm2 and LSE2 = l * log2 e."""
    rng = np.random.default_rng(5)
    comp = rng.standard_normal((8, 512)).astype(np.float32)
    q = rng.standard_normal((1, 4, 512)).astype(np.float32)
    indices = np.zeros((1, 128), np.int32)
    o, lse = case(H=4, q=q, comp=comp, indices=indices, bmm1=0.03, bmm2=0.5, width=130,
                  swa_topk_lens=np.array([0], np.int32), comp_block_tables=np.array([[3]], np.int32),
                  comp_page_size=2, hca_seq_lens=np.array([129], np.int32))
    row = bf16_round(comp[6])                     # page 3, offset 0 -> row 3 * 2 + 0
    qd = bf16_round(q[0])
    np.testing.assert_allclose(o[0], np.broadcast_to(0.5 * row, (4, 512)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], 0.03 * (qd @ row) * LOG2E, rtol=1e-12, atol=1e-12)


def _paged_small(fill_unused=-1, seed=11, per_token_pages=False):
    from sparse_mla_decode_token_gb300 import workloads as W
    return W.make_paged_workload(seed=seed, dtype="bf16", batch=3, q_lens=[1, 2, 1], num_heads=4,
                                 swa_rows=3 * 130, comp_pages=16, page_size=8, max_pages=5,
                                 hca_seq_lens=[128 + 37, 128 + 8, 100], seq_lens=[5000, 60, 3000],
                                 topk_lens=[160, 170, 140, 200], swa_topk_lens=[128, 17, 0, 64],
                                 fill_unused=fill_unused, varlen=True, sinks=True,
                                 per_token_pages=per_token_pages)


@pytest.mark.parametrize("per_token_pages", [False, True])
def test_page_table_equals_expanded_index_table(per_token_pages):
    """The page-table form equals the index form with the rows written out."""
    w = _paged_small(seed=12 if per_token_pages else 11, per_token_pages=per_token_pages)
    if per_token_pages:
        assert not np.array_equal(w.comp_block_tables[1], w.comp_block_tables[2])   # one request
    o, lse = orc.run_workload(w)
    T, W = w.sum_q, w.width
    ind = np.full((T, W), -1, np.int32)
    ind[:, :128] = w.indices
    cum = w.cum_seq_lens_q
    for t in range(T):
        b = int(np.searchsorted(cum, t, side="right") - 1)
        n_c = max(0, int(w.hca_seq_lens[b]) - 128)
        c = np.arange(n_c)
        ind[t, 128:128 + n_c] = w.comp_block_tables[t, c // w.comp_page_size] * w.comp_page_size + c % w.comp_page_size
        ind[t, :128][np.arange(128) >= min(max(int(w.swa_topk_lens[t]), 0), 128)] = -1
    o2, lse2 = orc.sparse_mla_decode(dtype=w.dtype, batch=w.batch, q=w.q, swa_kv=w.swa_kv, comp_kv=w.comp_kv,
                                     indices=ind, topk_lens=w.topk_lens, seq_lens=np.full(w.batch, 100000),
                                     cum_seq_lens_q=cum, sinks=w.sinks, bmm1_scale=w.bmm1_scale,
                                     bmm2_scale=w.bmm2_scale)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_page_table_entries_past_the_footprint_are_never_read():
    o1, l1 = orc.run_workload(_paged_small(fill_unused=-1))
    o2, l2 = orc.run_workload(_paged_small(fill_unused=7))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_swa_topk_lens_equals_minus_one_mask():
    """A visible window of k columns is the same as -1 in SWA columns >= k."""
    rng = np.random.default_rng(3)
    swa = rng.standard_normal((200, 512)).astype(np.float32)
    q = rng.standard_normal((2, 4, 512)).astype(np.float32)
    ind = np.stack([rng.choice(200, size=128, replace=False) for _ in range(2)]).astype(np.int32)
    k = [37, 128]
    o1, l1 = case(H=4, q=q, swa=swa, indices=ind, seq_lens=(100000, 100000),
                  swa_topk_lens=np.asarray(k, np.int32))
    masked = ind.copy()
    masked[0, 37:] = -1
    o2, l2 = case(H=4, q=q, swa=swa, indices=masked, seq_lens=(100000, 100000))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # the window overrides the seq_lens rule (position 9 would allow 10 columns)
    o3, _ = case(H=4, q=q, swa=swa, indices=ind, seq_lens=(10, 100000), swa_topk_lens=np.asarray(k, np.int32))
    np.testing.assert_array_equal(o1, o3)
