"""The allocation-free entry point, smla_decode_static_workspace.

It is for callers that cannot allocate device memory where they run the
decode (an inference runtime's plugin enqueue callback that must not allocate,
a process whose device memory another allocator has fully reserved, a plain C
caller with no device allocator).  Its split-K scratch is a library-owned
static device array, so the test checks, through the C ABI, that two calls in
a row give bit for bit the output of smla_decode with a caller workspace (the
same plan runs the same deterministic kernels, so any difference would be a
misplaced scratch region), and that an over-size call is refused with a clear
error.

The file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import workloads as W

from gpu_helpers import device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_decode_token_gb300 import build
    build.build()
    B.lib()


def _args(w, d, out, lse, splits, kernel=B.KERNEL_AUTO):
    return B.make_args(q=d["q"], swa_kv=d["swa"], compressed_kv=d["comp"], sparse_indices=d["indices"],
                       seq_lens=d["seq_lens"], out=out, sparse_topk_lens=d["topk_lens"],
                       cum_seq_lens_q=d["cum"], sinks=d["sinks"], bmm1_scale=w.bmm1_scale,
                       bmm2_scale=w.bmm2_scale, out_lse=lse, num_splits=splits, kernel=kernel)


@pytest.mark.parametrize("dtype,H,splits", [("bf16", 128, 4), ("e4m3", 64, 7)])
def test_static_workspace_matches_caller_workspace(dtype, H, splits):
    w = W.make_workload(name="noalloc", seed=4242 + H, dtype=dtype, batch=3, q_lens=1, num_heads=H,
                        swa_rows=3 * 128, comp_rows=4096, width=128 + 900, seq_lens=100000,
                        ring_len=128, topk_lens=np.array([1028, 700, 300]), sinks=True)
    d = device_inputs(w)
    T = w.sum_q
    # reference: the existing entry point with a caller-owned workspace
    ref_o = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    ref_l = torch.empty((T, H), dtype=torch.float32, device="cuda")
    a = _args(w, d, ref_o, ref_l, splits)
    need = B.smla_plan_decode(a).workspace_bytes
    assert 0 < need <= B.STATIC_WORKSPACE_BYTES        # the call really uses split-K scratch
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), need
    B.smla_decode(a)
    torch.cuda.synchronize()
    for _ in range(2):                                 # two calls in a row share the static array
        out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        b = _args(w, d, out, lse, splits)
        B.smla_decode_static_workspace(b)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref_o)
        assert not torch.isnan(lse).any()
        assert torch.equal(lse, ref_l)                 # -inf == -inf for empty heads


def test_static_workspace_rejects_oversize_calls():
    w = W.make_workload(name="noalloc_big", seed=77, dtype="bf16", batch=64, q_lens=1, num_heads=128,
                        swa_rows=64 * 128, comp_rows=4096, width=128 + 64 * 40, seq_lens=100000,
                        ring_len=128, topk_lens=None, sinks=False)
    d = device_inputs(w)
    out = torch.empty((w.sum_q, 128, 512), dtype=torch.bfloat16, device="cuda")
    b = _args(w, d, out, None, 64)        # 64 tokens x 128 heads x 64 splits x 2 KB > 64 MiB
    assert B.smla_plan_decode(b).workspace_bytes > B.STATIC_WORKSPACE_BYTES
    with pytest.raises(B.SmlaError) as e:
        B.smla_decode_static_workspace(b)
    assert e.value.status == B.SMLA_ERR_WORKSPACE_TOO_SMALL
    assert "static workspace" in str(e.value)
