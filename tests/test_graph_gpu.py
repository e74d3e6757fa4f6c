"""The public call inside a CUDA graph: smla_decode is captured (single-split,
and split kernel + combine as a programmatic dependent launch), the graph is
replayed after new query values are written into the captured input buffer,
and every replay matches the fp64 oracle for the inputs it saw."""
import numpy as np
import pytest
import torch

from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import workloads as W

from gpu_helpers import compare, device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_decode_token_gb300 import build
    build.build()
    B.lib()


@pytest.mark.parametrize("kernel", [B.KERNEL_TCGEN05, B.KERNEL_TCGEN05_HEAD_OWNED, B.KERNEL_TCGEN05_SLOT_SPLIT, B.KERNEL_CUDA_CORE])
@pytest.mark.parametrize("dtype,splits", [("bf16", 1), ("e4m3", 1), ("bf16", 3), ("e4m3", 2)])
def test_decode_replays_from_a_cuda_graph(kernel, dtype, splits):
    w = W.make_workload(name="graph", seed=41, dtype=dtype, batch=3, q_lens=[1, 2, 1], num_heads=128,
                        swa_rows=3 * 128 + 64, comp_rows=2048, width=128 + 300, seq_lens=100000,
                        ring_len=128, topk_lens=[300, 428, 200, 350], sinks=True)
    d = device_inputs(w)
    out = torch.empty((w.sum_q, w.num_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.sum_q, w.num_heads), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = B.make_args(q=d["q"], swa_kv=d["swa"], compressed_kv=d["comp"], sparse_indices=d["indices"],
                       seq_lens=d["seq_lens"], out=out, sparse_topk_lens=d["topk_lens"], cum_seq_lens_q=d["cum"],
                       sinks=d["sinks"], bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale, out_lse=lse,
                       num_splits=splits, kernel=kernel, error_word=err)
    plan = B.smla_plan_decode(args, torch.cuda.current_device())
    assert plan.num_splits == splits
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    cap = torch.cuda.Stream()
    B.smla_decode(args, cap.cuda_stream)          # first launch outside the graph (kernel attributes set)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        B.smla_decode(args, cap.cuda_stream)
    for seed in (1, 2):
        # new query values in the captured buffer, then replay
        w2 = W.make_workload(name="graph", seed=41 + 100 * seed, dtype=dtype, batch=3, q_lens=[1, 2, 1],
                             num_heads=128, swa_rows=3 * 128 + 64, comp_rows=2048, width=128 + 300,
                             seq_lens=100000, ring_len=128, topk_lens=[300, 428, 200, 350], sinks=True)
        w.q = w2.q
        d["q"].copy_(device_inputs(w)["q"])
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        compare(w, out, lse)
