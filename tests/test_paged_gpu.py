"""GPU parity of the page-table form of the compressed segment, per-row SWA
window lengths, and whole-tile copies of consecutive rows, against the fp64
CPU oracle (same tolerances as the other parity tests)."""
import numpy as np
import pytest
import torch

from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import workloads as W

from gpu_helpers import compare, run_gpu

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


def paged_case(seed, *, dtype="bf16", H=128, page_size=64, hca=(128 + 300, 128 + 64, 100),
               q_lens=(1, 2, 1), topk="random", swa_topk=(128, 17, 0, 64), sinks=True,
               fill_unused=-1, comp_pages=64, per_token_pages=False):
    rng = np.random.default_rng(seed)
    batch = len(hca)
    max_pages = -(-max(h - 128 for h in hca) // page_size)
    T = int(sum(q_lens))
    width = 128 + max_pages * page_size
    topk_lens = rng.integers(129, width + 1, size=T) if topk == "random" else topk
    return W.make_paged_workload(seed=seed, dtype=dtype, batch=batch, q_lens=list(q_lens), num_heads=H,
                                 swa_rows=batch * 130 + 10, comp_pages=comp_pages, page_size=page_size,
                                 max_pages=max_pages, hca_seq_lens=list(hca),
                                 seq_lens=[5000, 90, 3000, 7000][:batch], ring_len=130,
                                 topk_lens=topk_lens, swa_topk_lens=swa_topk, sinks=sinks,
                                 varlen=True, fill_unused=fill_unused, per_token_pages=per_token_pages)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("page_size", [64, 128])
def test_paged_parity(kernel, dtype, H, splits, page_size):
    w = paged_case(300 + H + splits + page_size, dtype=dtype, H=H, page_size=page_size)
    out, lse, plan = run_gpu(w, kernel=kernel, num_splits=splits)
    if splits:
        assert plan["num_splits"] == splits
    compare(w, out, lse)


@pytest.mark.parametrize("dtype", ["packed_fp8", "nvfp4"])
@pytest.mark.parametrize("page_size", [16, 128])
@pytest.mark.parametrize("splits", [1, 2])
def test_paged_packed_rows(dtype, page_size, splits):
    """The page-table form with packed KV rows, on the dims-split tensor-core
    kernel (AUTO) and the CUDA-core kernel."""
    w = paged_case(700 + page_size + splits, dtype=dtype, H=128, page_size=page_size)
    for kernel in (B.KERNEL_AUTO, B.KERNEL_CUDA_CORE):
        out, lse, plan = run_gpu(w, num_splits=splits, kernel=kernel)
        want = B.KERNEL_CUDA_CORE if kernel == B.KERNEL_CUDA_CORE else B.KERNEL_TCGEN05
        assert plan["kernel"] == want and plan["num_splits"] == splits
        compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("page_size", [1, 16, 24, 256])
def test_paged_page_sizes_off_the_tile_grid(kernel, dtype, page_size):
    """Pages smaller than a tile or not a multiple of it: tiles span pages
    (row gathers), except where consecutive page IDs happen to form a run."""
    w = paged_case(500 + page_size, dtype=dtype, page_size=page_size, hca=(128 + 300, 128 + 200, 128 + 1),
                   topk=None, swa_topk=None, comp_pages=max(64, 3 * 300 // page_size + 8))
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("splits", [1, 0])
def test_paged_per_token_tables(kernel, dtype, splits):
    """Tokens of one request list different pages: each reads its own table row."""
    w = paged_case(700 + splits, dtype=dtype, q_lens=(3, 2, 1), hca=(128 + 300, 128 + 64, 128 + 9),
                   swa_topk=None, per_token_pages=True)
    bt = w.comp_block_tables
    assert not np.array_equal(bt[0], bt[1]) and not np.array_equal(bt[3], bt[4])
    out, lse, _ = run_gpu(w, kernel=kernel, num_splits=splits)
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_consecutive_pages_form_long_runs(kernel):
    """Page tables that list consecutive pages: whole compressed segments are
    runs of consecutive rows (whole-tile copies across page boundaries)."""
    w = paged_case(611, dtype="e4m3", page_size=64, topk=None, swa_topk=None)
    w.comp_block_tables[:] = np.where(w.comp_block_tables >= 0,
                                      10 + np.arange(w.comp_block_tables.shape[1])[None, :], -1)
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits", [1, 2])
def test_paged_empty_and_window_only_tokens(kernel, splits):
    """hca_seq_lens below 128 backs no compressed slot; window 0 then leaves
    the token empty (O = 0, LSE = -inf)."""
    w = paged_case(71, dtype="bf16", hca=(100, 128, 128 + 64), q_lens=(1, 1, 1), topk=None,
                   swa_topk=(0, 5, 0))
    out, lse, _ = run_gpu(w, kernel=kernel, num_splits=splits)
    compare(w, out, lse)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_out_of_range_page_is_masked_and_flagged(kernel):
    w = paged_case(81, dtype="e4m3", page_size=64, topk=None, swa_topk=None, comp_pages=64)
    w.comp_block_tables[0, 1] = 64          # one page past the pool: rows 4096..4159
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = run_gpu(w, kernel=kernel, error_word=err)
    assert int(err.item()) & B.DEVERR_INDEX_OUT_OF_RANGE
    compare(w, out, lse, invalid_index="mask")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_index_form_runs_of_consecutive_rows(kernel, dtype):
    """Index-form compressed columns that hold runs of consecutive rows, some
    aligned to tiles, some not, one ending on the pool's last row, one broken
    in the middle of a tile: runs take whole-tile copies, the rest gathers."""
    comp_rows = 2048
    w = W.make_workload(name="runs", seed=91, dtype=dtype, batch=4, q_lens=1, num_heads=128,
                        swa_rows=4 * 128 + 64, comp_rows=comp_rows, width=128 + 320, seq_lens=100000,
                        ring_len=128, topk_lens=None, sinks=True)
    cols = 320
    w.indices[0, 128:] = 100 + np.arange(cols)                        # one run, start not tile-aligned
    w.indices[1, 128:] = comp_rows - cols + np.arange(cols)           # ends on the last row
    w.indices[2, 128:] = 64 + np.arange(cols)
    w.indices[2, 128 + 90] = 7                                        # broken inside the second tile
    w.indices[3, 128:128 + 64] = 500 + np.arange(64)                  # one run, then -1 holes
    w.indices[3, 128 + 64:] = np.where(np.arange(cols - 64) % 3 == 0, -1, 900 + np.arange(cols - 64))
    for splits in (1, 2):
        out, lse, _ = run_gpu(w, kernel=kernel, num_splits=splits)
        compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_index_form_per_row_window_lengths(kernel, dtype):
    """swa_topk_lens in the index form, including 0, 128 and values past 128
    (clamped), overriding the seq_lens rule."""
    w = W.make_workload(name="win", seed=93, dtype=dtype, batch=5, q_lens=1, num_heads=64,
                        swa_rows=5 * 128 + 64, comp_rows=2048, width=128 + 200, seq_lens=[100000, 40, 100000, 3, 100000],
                        ring_len=128, topk_lens=None, sinks=False)
    w.indices[:, :128] = np.arange(128)[None, :] + 128 * np.arange(5)[:, None]   # every SWA column a legal row
    w.swa_topk_lens = np.array([0, 128, 300, 77, 1], dtype=np.int32)
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_full_size_sampled(kernel):
    """The paged FP8 workload (128 tokens, H=128, 128 SWA + 2048 compressed
    slots on 16 pages of 128 rows) in the launch configuration the benchmark
    times, checked on sampled tokens."""
    w = W.config_workload(6)
    out, lse, _ = run_gpu(w, kernel=kernel)
    compare(w, out, lse, tokens=[0, 1, 63, 64, 127])
