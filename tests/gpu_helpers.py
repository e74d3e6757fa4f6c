"""Shared helpers of the GPU tests: move a Workload to the device, run the
CUDA path through the C ABI binding, and compare it with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_mla_decode_token_gb300 import binding as B

# max |dO| allowed vs the fp64 oracle (packed rows: exact dequantisation in
# fp32 on the CUDA cores, so the BF16 bound applies)
TOL_O = {"bf16": 2e-2, "e4m3": 4e-2, "packed_fp8": 2e-2, "nvfp4": 2e-2}
TOL_LSE = 1e-3                          # max |dLSE| (base 2)


def device_inputs(w, device="cuda"):
    def kv(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:                       # BF16 bits (query, or BF16 rows)
            return t.view(torch.int16).view(torch.bfloat16).to(device)
        if getattr(w, "packed", False):                # packed KV rows: uint8
            return t.to(device)
        return t.view(torch.float8_e4m3fn).to(device)

    def i32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    return dict(
        q=kv(w.q), swa=kv(w.swa_kv), comp=kv(w.comp_kv), indices=i32(w.indices),
        topk_lens=i32(w.topk_lens), seq_lens=i32(w.seq_lens), cum=i32(w.cum_seq_lens_q),
        sinks=None if w.sinks is None else torch.from_numpy(w.sinks).to(device),
        swa_topk_lens=i32(getattr(w, "swa_topk_lens", None)),
        block_tables=i32(getattr(w, "comp_block_tables", None)),
        hca_seq_lens=i32(getattr(w, "hca_seq_lens", None)),
    )


DEVERR_FATAL = 0x2 | 0x4      # a bounded on-device wait expired / an internal limit was hit


def run_gpu(w, d=None, *, num_splits=0, max_splits=0, kernel=B.KERNEL_AUTO, bmm_as_tensor=False,
            error_word=None, sync=True, schedule=B.SCHEDULE_AUTO):
    """Run the decode on the GPU; returns (out bf16 tensor, lse tensor, plan dict).

    Every run carries a device error word; a timeout or internal-limit bit fails
    the call (index range errors are left to the caller to inspect)."""
    own_err = error_word is None
    if own_err:
        error_word = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = device_inputs(w) if d is None else d
    T, H = w.sum_q, w.num_heads
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    bmm1, bmm2 = w.bmm1_scale, w.bmm2_scale
    if bmm_as_tensor:
        bmm1 = torch.tensor([bmm1], dtype=torch.float32, device="cuda")
        bmm2 = torch.tensor([bmm2], dtype=torch.float32, device="cuda")
    args = B.make_args(q=d["q"], swa_kv=d["swa"], compressed_kv=d["comp"],
                       sparse_indices=d["indices"], seq_lens=d["seq_lens"], out=out,
                       sparse_topk_lens=d["topk_lens"], cum_seq_lens_q=d["cum"], sinks=d["sinks"],
                       bmm1_scale=bmm1, bmm2_scale=bmm2, out_lse=lse, num_splits=num_splits,
                       max_splits=max_splits, kernel=kernel, error_word=error_word, schedule=schedule,
                       swa_topk_lens=d.get("swa_topk_lens"), comp_block_tables=d.get("block_tables"),
                       comp_page_size=getattr(w, "comp_page_size", 0), hca_seq_lens=d.get("hca_seq_lens"),
                       width=w.width if getattr(w, "comp_block_tables", None) is not None else None)
    plan = B.smla_plan_decode(args, torch.cuda.current_device()) if T > 0 else None
    ws = None
    if plan is not None and plan.workspace_bytes:
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        args.workspace, args.workspace_bytes = ws.data_ptr(), plan.workspace_bytes
    B.smla_decode(args)
    if sync:
        torch.cuda.synchronize()
        assert int(error_word.item()) & DEVERR_FATAL == 0, f"device error word {int(error_word.item()):#x}"
    return out, lse, (plan.as_dict() if plan is not None else None)


def compare(w, out, lse, tokens=None, tol_o=None, tol_lse=TOL_LSE, **oracle_kw):
    """Assert the GPU result matches the oracle on ``tokens`` (default: all)."""
    tokens = list(range(w.sum_q)) if tokens is None else list(tokens)
    o_ref, l_ref = oracle.run_workload(w, tokens=tokens, **oracle_kw)
    o_gpu = out.float().cpu().numpy()[tokens].astype(np.float64)
    l_gpu = lse.cpu().numpy()[tokens].astype(np.float64)
    tol_o = TOL_O[w.dtype] if tol_o is None else tol_o
    assert np.all(np.isfinite(o_gpu)), "non-finite output"
    err_o = np.abs(o_gpu - o_ref).max() if o_gpu.size else 0.0
    assert err_o <= tol_o, f"max |dO| = {err_o:.3e} > {tol_o}"
    ninf_ref, ninf_gpu = np.isneginf(l_ref), np.isneginf(l_gpu)
    assert np.array_equal(ninf_ref, ninf_gpu), "empty-token (-inf LSE) pattern differs"
    fin = ~ninf_ref
    err_l = np.abs(l_gpu[fin] - l_ref[fin]).max() if fin.any() else 0.0
    assert err_l <= tol_lse, f"max |dLSE| = {err_l:.3e} > {tol_lse}"
    return err_o, err_l
