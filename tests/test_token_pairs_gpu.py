"""GPU parity of the token-pair kernel (SMLA_KERNEL_TCGEN05_TOKEN_PAIRS: two
tokens of 64 heads per CTA pair over the union of their selected rows) in the
cases that decide what the union holds: rows both tokens select (the shared
SWA window of a request's consecutive tokens; compressed rows copied from the
previous token, in the same or a shuffled column order), a row one token
selects twice (the unit then shares nothing), equal row numbers in different
pools (never shared), an odd token count (the last unit holds one token),
empty tokens, split partials, page tables and CUDA-graph replays.  Same
tolerances as the other parity tests."""
import numpy as np
import pytest
import torch

from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import workloads as W

from gpu_helpers import compare, device_inputs, run_gpu

pytestmark = pytest.mark.gpu

PAIRS = B.KERNEL_TCGEN05_TOKEN_PAIRS


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_decode_token_gb300 import build
    build.build()
    B.lib()


def pair_case(seed, *, dtype="bf16", q_lens=(2, 3, 1, 2), width=128 + 300, overlap="copy", topk="random",
              comp_rows=4096):
    """H = 64 workload whose odd-numbered tokens take (part of) the previous
    token's compressed rows: overlap = "none" (independent draws), "copy"
    (same rows, same columns), "shuffle" (same rows, permuted columns),
    "half" (the first half of the compressed columns copied)."""
    rng = np.random.default_rng(seed)
    q_lens = list(q_lens)
    batch, T = len(q_lens), int(sum(q_lens))
    n_comp = width - 128
    topk_lens = rng.integers(129, width + 1, size=T) if topk == "random" else topk
    w = W.make_workload(name=f"pairs{seed}", seed=seed, dtype=dtype, batch=batch, q_lens=q_lens,
                        num_heads=64, swa_rows=128 * batch + 64, comp_rows=comp_rows, width=width,
                        seq_lens=rng.integers(3000, 9000, size=batch), ring_len=128,
                        comp_valid=rng.integers(n_comp // 2, n_comp + 1, size=T), topk_lens=topk_lens,
                        sinks=True, varlen=True)
    for t in range(1, T, 2):
        prev = w.indices[t - 1, 128:]
        if overlap == "copy":
            w.indices[t, 128:] = prev
        elif overlap == "shuffle":
            w.indices[t, 128:] = rng.permutation(prev)
        elif overlap == "half":
            w.indices[t, 128:128 + n_comp // 2] = prev[:n_comp // 2]
    return w


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("overlap", ["none", "shuffle"])
def test_wide_tables(dtype, overlap):
    """128 + 2048 columns: the E4M3 pair form takes at most 1152 columns of
    each token per split (two splits at least), the BF16 one up to 2304."""
    w = pair_case(780, dtype=dtype, q_lens=(2, 2, 1), width=128 + 2048, overlap=overlap, comp_rows=65536)
    out, lse, plan = run_gpu(w, kernel=PAIRS)
    check_plan(plan, w.sum_q)
    assert plan["num_splits"] >= (2 if dtype == "e4m3" else 1)
    compare(w, out, lse)


def test_auto_takes_pairs_past_a_wave():
    """AUTO runs the slot-split kernel's token-pair form for E4M3 rows with
    64 heads, at most 1152 columns and more tokens than SM pairs (here 160
    tokens of 128 + 512 columns, requests of two tokens): every token against
    the oracle."""
    w = pair_case(790, dtype="e4m3", q_lens=[2] * 80, width=128 + 512, overlap="half")
    out, lse, plan = run_gpu(w)
    check_plan(plan, w.sum_q)
    compare(w, out, lse)


def check_plan(plan, T, splits=None):
    assert plan["kernel"] == PAIRS
    S = plan["num_splits"]
    if splits:
        assert S == splits
    assert plan["grid"] == 2 * ((T + 1) // 2) * S


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("overlap", ["none", "copy", "shuffle", "half"])
@pytest.mark.parametrize("splits", [1, 2, 3, 0])
def test_pairs_parity(dtype, overlap, splits):
    w = pair_case(700 + splits, dtype=dtype, overlap=overlap)
    out, lse, plan = run_gpu(w, kernel=PAIRS, num_splits=splits)
    check_plan(plan, w.sum_q, splits)
    compare(w, out, lse)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("where", ["a", "b", "both"])
def test_row_selected_twice_shares_nothing(dtype, where):
    """A token that selects a row in two slots counts it twice; its unit falls
    back to the concatenation of the two lists (the other units still share)."""
    w = pair_case(720, dtype=dtype, overlap="copy", topk=None)
    if where in ("a", "both"):
        w.indices[0, 131] = w.indices[0, 130] = 7         # token 0 (A of unit 0): row 7 twice
        w.indices[1, 140] = 7                             # and token 1 selects it once
    if where in ("b", "both"):
        w.indices[3, 5] = w.indices[3, 6]                 # token 3 (B of unit 1): a SWA row twice
    out, lse, plan = run_gpu(w, kernel=PAIRS)
    check_plan(plan, w.sum_q)
    compare(w, out, lse)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_same_row_number_in_other_pool_is_not_shared(dtype):
    """Token B's compressed columns hold token A's SWA row numbers: the same
    integers in another pool, so different rows."""
    w = pair_case(730, dtype=dtype, overlap="none", topk=None)
    for t in range(1, w.sum_q, 2):
        w.indices[t, 128:256] = w.indices[t - 1, :128]
    out, lse, plan = run_gpu(w, kernel=PAIRS)
    check_plan(plan, w.sum_q)
    compare(w, out, lse)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("splits", [1, 2])
def test_odd_tokens_empty_tokens_and_many_units(dtype, splits):
    """301 tokens (151 units: more than the SM pairs, and a last unit of one
    token), every fifth token with no active slot, every seventh with only
    SWA slots."""
    T = 301
    w = pair_case(740 + splits, dtype=dtype, q_lens=[2] * 150 + [1], width=128 + 200, overlap="shuffle")
    w.indices[::5, :] = -1
    w.topk_lens = np.asarray(w.topk_lens).copy()
    w.topk_lens[::7] = 128
    out, lse, plan = run_gpu(w, kernel=PAIRS, num_splits=splits)
    check_plan(plan, T, splits)
    compare(w, out, lse)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_pairs_page_table_form(dtype):
    """Compressed segment from per-token page tables (consecutive tokens of a
    request share their request's pages), per-row window lengths."""
    w = W.make_paged_workload(seed=750, dtype=dtype, batch=3, q_lens=[2, 3, 2], num_heads=64,
                              swa_rows=3 * 130 + 10, comp_pages=64, page_size=64, max_pages=5,
                              hca_seq_lens=[128 + 300, 128 + 64, 200], seq_lens=[5000, 900, 3000],
                              ring_len=130, topk_lens=np.full(7, 128 + 320), swa_topk_lens=[128, 17, 0, 64, 128, 90, 128],
                              sinks=True, varlen=True)
    out, lse, plan = run_gpu(w, kernel=PAIRS)
    check_plan(plan, w.sum_q)
    compare(w, out, lse)


@pytest.mark.parametrize("splits", [1, 3])
def test_pairs_replay_from_a_cuda_graph(splits):
    w = pair_case(770, dtype="bf16", overlap="half")
    d = device_inputs(w)
    out = torch.empty((w.sum_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.sum_q, 64), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = B.make_args(q=d["q"], swa_kv=d["swa"], compressed_kv=d["comp"], sparse_indices=d["indices"],
                       seq_lens=d["seq_lens"], out=out, sparse_topk_lens=d["topk_lens"], cum_seq_lens_q=d["cum"],
                       sinks=d["sinks"], bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale, out_lse=lse,
                       num_splits=splits, kernel=PAIRS, error_word=err)
    plan = B.smla_plan_decode(args, torch.cuda.current_device())
    check_plan(plan.as_dict(), w.sum_q, splits)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    cap = torch.cuda.Stream()
    B.smla_decode(args, cap.cuda_stream)          # first launch outside the graph (kernel attributes set)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        B.smla_decode(args, cap.cuda_stream)
    w2 = pair_case(771, dtype="bf16", overlap="half")
    w.q = w2.q
    d["q"].copy_(device_inputs(w)["q"])
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    compare(w, out, lse)
