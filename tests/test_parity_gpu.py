"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances: max |dO| <= 2e-2 (BF16 inputs) or 4e-2 (FP8 E4M3 inputs),
|dLSE| <= 1e-3, and the set of attended slots exact (masking probes)."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import workloads as W

from gpu_helpers import compare, device_inputs, run_gpu

pytestmark = pytest.mark.gpu

KERNELS = [B.KERNEL_CUDA_CORE, B.KERNEL_TCGEN05, B.KERNEL_TCGEN05_HEAD_OWNED, B.KERNEL_TCGEN05_SLOT_SPLIT,
           B.KERNEL_TCGEN05_TOKEN_PAIRS]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_decode_token_gb300 import build
    build.build()
    B.lib()


# ------------------------------------------------------- the five workloads

# tokens checked per workload: every token (the oracle takes about a second
# for the 128 tokens of the FP8 workload)
SAMPLE = {1: None, 2: None, 3: None, 4: None, 5: None}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_config_parity(n, kernel):
    w = W.config_workload(n)
    out, lse, plan = run_gpu(w, kernel=kernel)
    tokens = SAMPLE[n]
    if tokens is not None:
        tokens = [t for t in tokens if t < w.sum_q]
    compare(w, out, lse, tokens=tokens)


# ------------------------------------------- small cases: tiles + ragged tails

def small_case(seed, *, dtype="bf16", H=128, width=128 + 300, batch=3, q_lens=1,
               sinks=True, holes=True, topk="random", comp_rows=2048, seq_len=100000):
    rng = np.random.default_rng(seed)
    q_lens_arr = np.broadcast_to(np.asarray(q_lens), (batch,))
    T = int(q_lens_arr.sum())
    n_comp = width - 128
    comp_valid = rng.integers(n_comp // 2, n_comp + 1, size=T) if holes else None
    if isinstance(topk, str) and topk == "random":
        topk_lens = rng.integers(129, width + 1, size=T)
    elif isinstance(topk, str) and topk == "none":
        topk_lens = None
    else:
        topk_lens = topk
    return W.make_workload(name=f"small{seed}", seed=seed, dtype=dtype, batch=batch, q_lens=q_lens,
                           num_heads=H, swa_rows=128 * batch + 64, comp_rows=comp_rows,
                           width=width, seq_lens=seq_len, ring_len=128, comp_valid=comp_valid,
                           topk_lens=topk_lens, sinks=sinks)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("splits", [1, 2, 3, 0])
def test_small_parity(kernel, dtype, H, splits):
    w = small_case(100 + H + splits, dtype=dtype, H=H)
    out, lse, plan = run_gpu(w, kernel=kernel, num_splits=splits)
    if splits:
        assert plan["num_splits"] == splits
    compare(w, out, lse)


# ------------------------------------- balanced mode: shares of the columns

def expected_clusters(T, width, sms):
    """The planner's cluster count under the balanced schedule (see the
    header's smla_schedule)."""
    pairs = max(sms // 2, 1)
    if width > 2304 or T > 14 * pairs:
        return 0
    return max(1, min(pairs, T * width // 64))


@pytest.mark.parametrize("dtype,H,batch,q_lens,width,topk", [
    ("e4m3", 128, 1, 1, 128 + 2048, "none"),     # one token in 34 pieces
    ("bf16", 64, 3, 1, 128 + 512, "random"),     # three tokens in 10 pieces each
    ("e4m3", 128, 7, 11, 128 + 512, "random"),   # 77 tokens: most shares cut two tokens
    ("bf16", 128, 8, 25, 256, "random"),         # 200 tokens: 3 to 4 units per share
    ("e4m3", 64, 8, 133, 128, "none"),           # 1064 tokens: 14 whole tokens per share
    ("e4m3", 128, 5, 20, 128 + 128, "zeros"),    # every third token has no active column
])
def test_balanced_mode_parity(dtype, H, batch, q_lens, width, topk):
    """The balanced schedule: each CTA pair takes an equal share of the T x W
    columns, whole tokens plus pieces of tokens cut at the share boundaries,
    merged by the piece combine."""
    T = batch * q_lens
    if isinstance(topk, str) and topk == "zeros":
        rng = np.random.default_rng(5)
        topk = rng.integers(129, width + 1, size=T)
        topk[::3] = 0
    w = small_case(300 + T, dtype=dtype, H=H, width=width, batch=batch, q_lens=q_lens, topk=topk,
                   seq_len=4000)
    out, lse, plan = run_gpu(w, kernel=B.KERNEL_TCGEN05, schedule=B.SCHEDULE_BALANCED)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan["clusters"] == expected_clusters(T, width, sms)
    assert plan["grid"] == 2 * plan["clusters"] and plan["num_splits"] == 1
    compare(w, out, lse)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_balanced_and_grid_modes_agree(dtype):
    """The same workload in balanced mode (which cuts some tokens into
    pieces) and in grid mode (one pair per token): both match the oracle."""
    w = small_case(41, dtype=dtype, H=128, width=128 + 640, batch=4, q_lens=40, seq_len=4000)
    out_b, lse_b, plan_b = run_gpu(w, kernel=B.KERNEL_TCGEN05, schedule=B.SCHEDULE_BALANCED)
    out_g, lse_g, plan_g = run_gpu(w, kernel=B.KERNEL_TCGEN05)
    assert plan_b["clusters"] > 1 and plan_g["clusters"] == 0
    compare(w, out_b, lse_b)
    compare(w, out_g, lse_g)
    P, Wd = plan_b["clusters"], w.width
    cut = {(w.sum_q * Wd * c // P) // Wd for c in range(1, P) if (w.sum_q * Wd * c // P) % Wd}
    assert cut and len(cut) < w.sum_q


@pytest.mark.parametrize("kernel", KERNELS)
def test_varlen_parity(kernel):
    w = small_case(7, dtype="bf16", H=64, batch=6, q_lens=[1, 4, 2, 3, 1, 4], seq_len=5000)
    assert w.cum_seq_lens_q is not None
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype,H,q_lens,width", [("bf16", 64, [1, 150, 40], 128 + 128),
                                                   ("e4m3", 128, [2, 64, 1], 128 + 448),
                                                   ("e4m3", 128, [3, 40, 1], 128 + 16)])
def test_mixed_prefill_and_decode_batch(kernel, dtype, H, q_lens, width):
    """Requests with q_len from 1 to 150 in one call (a mixed prefill/decode
    batch, flattened tokens on the grid, per-token windows shifted by i).
    The second E4M3 case has at most 144 slots per token, where the E4M3
    rounding of P weighs most (short chains follow the exact running maximum)."""
    w = small_case(21 + H, dtype=dtype, H=H, width=width, batch=len(q_lens), q_lens=q_lens, seq_len=4000)
    assert w.cum_seq_lens_q is not None and w.sum_q == sum(q_lens)
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", [B.KERNEL_TCGEN05, B.KERNEL_TCGEN05_SLOT_SPLIT])
def test_e4m3_exact_maximum_boundary(kernel):
    """E4M3 P: a split of at most 512 valid slots follows the exact running
    maximum, a longer one the lazy reference (threshold 2^8).  Tokens of 511,
    512 and 513 valid slots in one unsplit call, on both tensor-core kernels."""
    w = small_case(31, dtype="e4m3", H=128, width=128 + 400, batch=3, holes=False,
                   topk=np.array([511, 512, 513]))
    counts = [len(oracle.valid_slots(t, indices=w.indices, topk_lens=w.topk_lens, seq_lens=w.seq_lens,
                                     cum_seq_lens_q=None, batch=w.batch, swa_rows=w.swa_kv.shape[0],
                                     comp_rows=w.comp_kv.shape[0])) for t in range(w.sum_q)]
    assert counts == [511, 512, 513]
    out, lse, plan = run_gpu(w, kernel=kernel, num_splits=1)
    assert plan["num_splits"] == 1
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
def test_swa_only_width_128(kernel):
    w = small_case(8, dtype="e4m3", H=128, width=128, holes=False, topk="none")
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
def test_forced_max_splits(kernel):
    w = small_case(9, dtype="bf16", H=64, width=128 + 900, batch=2)
    out, lse, plan = run_gpu(w, kernel=kernel, num_splits=B.MAX_SPLITS)
    assert plan["num_splits"] == B.MAX_SPLITS
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
def test_short_sequences_trim_swa_window(kernel):
    # seq_len < 128: only the first pos + 1 SWA columns are in the window
    w = small_case(10, dtype="bf16", H=64, batch=4, q_lens=2, seq_len=[3, 60, 127, 128], topk="none")
    # put real rows into every SWA column so that the window, not -1, does the masking
    rng = np.random.default_rng(10)
    for t in range(w.sum_q):
        w.indices[t, :128] = rng.choice(w.swa_kv.shape[0], 128, replace=False)
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse)


# ------------------------------------------------------------ masking probes

def probe_case(indices, *, seq_lens, topk_lens=None, H=64, dtype="bf16", sinks=None, bmm2=1.0):
    """q = 0 and basis-vector rows: row r of the pools has a single 1 at dim r % 512
    (SWA rows at dims 0..255, compressed rows at 256..511), so every output dim
    shows whether its slot contributed, and LSE2 = log2(number of slots)."""
    indices = np.asarray(indices, np.int32)
    T = indices.shape[0]
    one = 0x3F80 if dtype == "bf16" else 0x38
    nptype = np.uint16 if dtype == "bf16" else np.uint8
    swa = np.zeros((256, 512), nptype)
    comp = np.zeros((256, 512), nptype)
    for r in range(256):
        swa[r, r] = one
        comp[r, 256 + r] = one
    seq_lens = np.asarray(seq_lens, np.int32)
    return W.Workload(name="probe", dtype=dtype, batch=len(seq_lens), num_heads=H,
                      q=np.zeros((T, H, 512), nptype), swa_kv=swa, comp_kv=comp, indices=indices,
                      topk_lens=None if topk_lens is None else np.asarray(topk_lens, np.int32),
                      seq_lens=seq_lens, cum_seq_lens_q=None,
                      sinks=None if sinks is None else np.asarray(sinks, np.float32),
                      bmm1_scale=1.0, bmm2_scale=bmm2)


def check_probe(w, out, lse):
    """Exact attended-slot set per token, checked against the oracle's slot list."""
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for t in range(w.sum_q):
        slots = oracle.valid_slots(t, indices=w.indices, topk_lens=w.topk_lens, seq_lens=w.seq_lens,
                                   cum_seq_lens_q=None, batch=w.batch, swa_rows=256, comp_rows=256)
        counts = np.zeros(512)
        for (_, pool, row) in slots:
            counts[row if pool == "swa" else 256 + row] += 1
        n = len(slots)
        nz_gpu = o[t] != 0
        assert np.array_equal(nz_gpu, np.broadcast_to(counts > 0, nz_gpu.shape)), f"token {t}: slot set differs"
        if n:
            np.testing.assert_allclose(o[t], np.broadcast_to(counts / n * w.bmm2_scale, o[t].shape),
                                       atol=TOL_PROBE)
            np.testing.assert_allclose(l[t], math.log2(n), atol=1e-5)
        else:
            assert np.all(np.isneginf(l[t]))


TOL_PROBE = 4e-3


def probe_row(swa, comp, width):
    row = np.full(width, -1, np.int32)
    row[:len(swa)] = swa
    row[128:128 + len(comp)] = comp
    return row


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("H", [64, 128])
def test_masking_probes(kernel, dtype, H):
    W_ = 128 + 200
    rng = np.random.default_rng(11)
    rows = []
    # 0: -1 holes in both segments
    r = probe_row(rng.permutation(256)[:128], rng.permutation(256)[:200], W_)
    r[[0, 5, 127, 128, 200, 327]] = -1
    rows.append(r)
    # 1: topk_lens = 128 (SWA only)
    rows.append(probe_row(rng.permutation(256)[:128], rng.permutation(256)[:200], W_))
    # 2: topk_lens = W
    rows.append(probe_row(rng.permutation(256)[:128], rng.permutation(256)[:200], W_))
    # 3: random topk_lens with -1 tail
    rows.append(probe_row(rng.permutation(256)[:100], rng.permutation(256)[:150], W_))
    # 4: fully masked token
    rows.append(np.full(W_, -1, np.int32))
    # 5: everything beyond topk_lens = 0
    rows.append(probe_row(rng.permutation(256)[:128], rng.permutation(256)[:200], W_))
    # 6: duplicate rows count twice
    rows.append(probe_row([3, 3, 3, 9], [7, 7, 8], W_))
    # 7: short sequence (pos = 4): only 5 SWA columns in the window
    rows.append(probe_row(rng.permutation(256)[:128], [1, 2], W_))
    idx = np.stack(rows)
    topk = np.array([W_, 128, W_, 200, W_, 0, W_, W_])
    seq = [10 ** 6] * 7 + [5]
    w = probe_case(idx, seq_lens=seq, topk_lens=topk, H=H, dtype=dtype, bmm2=0.5)
    out, lse, _ = run_gpu(w, kernel=kernel)
    check_probe(w, out, lse)
    for splits in (2, 5):
        out, lse, _ = run_gpu(w, kernel=kernel, num_splits=splits)
        check_probe(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
def test_out_of_range_index_is_masked_and_flagged(kernel):
    W_ = 128 + 8
    idx = np.stack([probe_row([0, 1, 2], [4, 300, 5], W_), probe_row([0, -7], [4], W_),
                    probe_row([0], [1], W_)])
    w = probe_case(idx, seq_lens=[10 ** 6] * 3)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = run_gpu(w, kernel=kernel, error_word=err)
    assert int(err.item()) & B.DEVERR_INDEX_OUT_OF_RANGE
    masked = w.indices.copy()
    masked[0, 129] = -1
    masked[1, 1] = -1
    w2 = probe_case(masked, seq_lens=[10 ** 6] * 3)
    check_probe(w2, out, lse)
    err.zero_()
    run_gpu(w2, kernel=kernel, error_word=err)
    assert int(err.item()) == 0


# ------------------------------------------------------------ edge cases

def test_empty_batch_is_a_noop():
    w = small_case(12, H=64)
    d = device_inputs(w)
    out = torch.empty((0, 64, 512), dtype=torch.bfloat16, device="cuda")
    args = B.make_args(q=d["q"][:0], swa_kv=d["swa"], compressed_kv=d["comp"],
                       sparse_indices=d["indices"][:0], seq_lens=d["seq_lens"], out=out)
    B.smla_decode(args)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kernel", KERNELS)
def test_scales_as_device_tensors(kernel):
    w = small_case(13, dtype="e4m3", H=128)
    o1, l1, _ = run_gpu(w, kernel=kernel)
    o2, l2, _ = run_gpu(w, kernel=kernel, bmm_as_tensor=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("kernel", KERNELS)
def test_deterministic(kernel):
    w = small_case(14, dtype="bf16", H=128)
    d = device_inputs(w)
    o1, l1, _ = run_gpu(w, d, kernel=kernel, num_splits=3)
    o2, l2, _ = run_gpu(w, d, kernel=kernel, num_splits=3)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_and_strided_layouts(kernel):
    """Pools as paged HND views [pages, 1, page_size, 512] and a padded row stride;
    the query as a slice of a wider buffer (token stride > H * 512)."""
    w = small_case(15, dtype="bf16", H=64, comp_rows=64 * 32)
    d = device_inputs(w)
    ref_o, ref_l, _ = run_gpu(w, d, kernel=kernel)
    comp_paged = d["comp"].view(64, 1, 32, 512)
    swa_pad = torch.zeros((d["swa"].shape[0], 520), dtype=d["swa"].dtype, device="cuda")
    swa_pad[:, :512] = d["swa"]
    q_wide = torch.zeros((w.sum_q, 64 * 512 + 64), dtype=d["q"].dtype, device="cuda")
    q_wide[:, :64 * 512] = d["q"].reshape(w.sum_q, -1)
    q_view = torch.as_strided(q_wide, (w.sum_q, 64, 512), (64 * 512 + 64, 512, 1))
    out = torch.empty_like(ref_o)
    lse = torch.empty_like(ref_l)
    args = B.make_args(q=q_view, swa_kv=swa_pad[:, :512], compressed_kv=comp_paged,
                       sparse_indices=d["indices"], seq_lens=d["seq_lens"], out=out,
                       sparse_topk_lens=d["topk_lens"], sinks=d["sinks"],
                       bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale, out_lse=lse, kernel=kernel)
    assert args.swa_row_stride == 520 and args.q_stride_token == 64 * 512 + 64
    ws = torch.empty(max(B.smla_plan_decode(args).workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    B.smla_decode(args)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_workspace_too_small_is_rejected():
    w = small_case(16, H=64)
    d = device_inputs(w)
    out = torch.empty((w.sum_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    args = B.make_args(q=d["q"], swa_kv=d["swa"], compressed_kv=d["comp"], sparse_indices=d["indices"],
                       seq_lens=d["seq_lens"], out=out, num_splits=4)
    need = B.smla_plan_decode(args).workspace_bytes
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), need - 256
    with pytest.raises(B.SmlaError) as e:
        B.smla_decode(args)
    assert e.value.status == B.SMLA_ERR_WORKSPACE_TOO_SMALL
    args.out = out.data_ptr() + 2                  # misaligned output
    args.workspace_bytes = need
    with pytest.raises(B.SmlaError) as e:
        B.smla_decode(args)
    assert e.value.status == B.SMLA_ERR_INVALID_ARG


@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("splits", [1, 2])
def test_slot_split_many_units(H, splits):
    """More (token, split) units than SM pairs (several waves of the
    slot-split kernel): tokens of one to four 128-slot tiles, every fourth
    token fully masked (no slot at all), and split partials."""
    w = small_case(500 + H + splits, dtype="e4m3", H=H, batch=200, width=128 + 400)
    w.indices[::4, :] = -1
    out, lse, plan = run_gpu(w, kernel=B.KERNEL_TCGEN05_SLOT_SPLIT, num_splits=splits)
    assert plan["kernel"] == B.KERNEL_TCGEN05_SLOT_SPLIT and plan["num_splits"] == splits
    assert plan["grid"] == 2 * 200 * splits
    compare(w, out, lse)


def packed_kernel(dtype, asked):
    """Kernel a packed form plans to: the dims-split kernel unless the
    CUDA-core kernel is asked for."""
    return B.KERNEL_CUDA_CORE if asked == B.KERNEL_CUDA_CORE else B.KERNEL_TCGEN05


@pytest.mark.parametrize("dtype", ["packed_fp8", "nvfp4"])
@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("kernel", [B.KERNEL_AUTO, B.KERNEL_CUDA_CORE, B.KERNEL_TCGEN05_SLOT_SPLIT,
                                    B.KERNEL_TCGEN05_TOKEN_PAIRS])
def test_packed_rows_parity(dtype, H, splits, kernel):
    """Packed KV rows (584-byte packed FP8, 384-byte NVFP4; BF16 query): the
    dims-split tensor-core kernel's producers dequantise each row into exact
    BF16 tiles (AUTO, and the E4M3-only and token-pair requests; NVFP4's row
    scale applied to the logits and P in fp32), the CUDA-core kernel into fp32
    shared memory; ragged tiles, masked slots, sinks and split partials."""
    w = small_case(600 + H + splits, dtype=dtype, H=H)
    out, lse, plan = run_gpu(w, kernel=kernel, num_splits=splits)
    assert plan["kernel"] == packed_kernel(dtype, kernel)
    if splits:
        assert plan["num_splits"] == splits
    compare(w, out, lse)


@pytest.mark.parametrize("n", [7, 8])
@pytest.mark.parametrize("kernel", [B.KERNEL_AUTO, B.KERNEL_CUDA_CORE])
def test_packed_rows_workload_sampled(n, kernel):
    """Workload 3's shape with NVFP4 / packed FP8 rows (the bench workloads 7
    and 8): every 4th token of the tensor-core path, every 8th of the
    CUDA-core path, against the oracle."""
    w = W.config_workload(n)
    out, lse, plan = run_gpu(w, kernel=kernel)
    assert plan["kernel"] == packed_kernel(w.dtype, kernel)
    compare(w, out, lse, tokens=list(range(0, w.sum_q, 8 if plan["kernel"] == B.KERNEL_CUDA_CORE else 4)))


def test_many_tokens_grid():
    """More than 65535 tokens: tokens live on grid.x, so no launch limit is hit.

    q = 0 keeps the inputs small: every output is the mean of the token's rows."""
    T, H = 70000, 64
    rng = np.random.default_rng(17)
    gen = torch.Generator().manual_seed(17)
    swa_bits = W._to_bf16_bits(torch.randn(256, 512, generator=gen))
    comp_bits = W._to_bf16_bits(torch.randn(512, 512, generator=gen))
    idx = np.full((T, 136), -1, np.int32)
    idx[:, :8] = rng.integers(0, 256, size=(T, 8))
    idx[:, 128:136] = rng.integers(0, 512, size=(T, 8))
    zero_q = np.broadcast_to(np.zeros((1, H, 512), np.uint16), (T, H, 512))   # a view, no memory
    w = W.Workload(name="many", dtype="bf16", batch=T, num_heads=H, q=zero_q, swa_kv=swa_bits,
                   comp_kv=comp_bits, indices=idx, topk_lens=None,
                   seq_lens=np.full(T, 10 ** 6, np.int32), cum_seq_lens_q=None, sinks=None,
                   bmm1_scale=1.0, bmm2_scale=1.0)
    bf = lambda a: torch.from_numpy(a).view(torch.int16).view(torch.bfloat16).cuda()
    d = dict(q=torch.zeros((T, H, 512), dtype=torch.bfloat16, device="cuda"), swa=bf(swa_bits),
             comp=bf(comp_bits), indices=torch.from_numpy(idx).cuda(), topk_lens=None,
             seq_lens=torch.from_numpy(w.seq_lens).cuda(), cum=None, sinks=None)
    out, lse, plan = run_gpu(w, d)
    assert plan["grid"] >= T
    compare(w, out, lse, tokens=[0, 1, 65535, 65536, T - 1])
