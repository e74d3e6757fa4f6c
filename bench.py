"""Benchmark of the sparse MLA decode hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

One step = one whole decode (the decode kernel, plus the combine kernel when
the plan has one) over one batch of the synthetic workload.  Default workload:
FP8 E4M3, 128 tokens, H=128, 128 SWA + 2048 compressed slots per token over a
256k-row compressed pool.  L2 is flushed (a write of twice the L2 size)
between timed steps, outside the timed events.  Prints one JSON line.
"""
from __future__ import annotations

import os

_NCPU = os.cpu_count() or 1
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_NCPU))   # the CPU oracle's BLAS threads
os.environ.setdefault("OMP_NUM_THREADS", str(_NCPU))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import re  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mla_decode_token_gb300 import workloads as W  # noqa: E402

METRIC = "sparse-MLA decode query-tokens/s; gathered-KV GB/s and % of roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
HEAD_DIM, SWA_COLS = 512, 128
# fp32 FMA peak of the CUDA cores (the CUDA-core kernel's bound, which the
# packed KV forms run on): 152 SMs x 128 FP32 lanes x 2 flops x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


# ------------------------------------------------------------------ accounting

def active_slots(w) -> np.ndarray:
    """[T, W] mask of the slots each token reads: columns below
    clamp(topk_lens, 0, W) that are not -1 and, for SWA columns, inside the
    window min(128, pos + 1) (or the per-row window lengths); in the
    page-table form the compressed columns below the request's backed count
    hca_seq_lens[b]."""
    T, width = w.sum_q, w.width
    n_lim = np.full(T, width) if w.topk_lens is None else np.clip(w.topk_lens, 0, width)
    q_lens = (np.full(w.batch, T // w.batch) if w.cum_seq_lens_q is None
              else np.diff(w.cum_seq_lens_q))
    pos = np.concatenate([np.arange(ql) + sl - ql for sl, ql in zip(w.seq_lens, q_lens)])
    w_swa = np.clip(pos + 1 if w.swa_topk_lens is None else w.swa_topk_lens, 0, SWA_COLS)
    j = np.arange(width)[None, :]
    if w.paged:
        req = np.repeat(np.arange(w.batch), q_lens)
        n_lim = np.minimum(n_lim, np.maximum(SWA_COLS, w.hca_seq_lens[req]))
        swa_ok = np.zeros((T, width), dtype=bool)
        swa_ok[:, :SWA_COLS] = (w.indices[:, :SWA_COLS] != -1) & (j[:, :SWA_COLS] < w_swa[:, None])
        return (j < n_lim[:, None]) & (swa_ok | (j >= SWA_COLS))
    return (j < n_lim[:, None]) & (w.indices != -1) & ((j >= SWA_COLS) | (j < w_swa[:, None]))


def valid_slots_per_token(w) -> np.ndarray:
    """Slots each token reads (see active_slots)."""
    return active_slots(w).sum(axis=1)


def slot_rows(w) -> np.ndarray:
    """[T, W] row read by each column (int64): SWA rows as given, compressed
    rows + 2^32 (their own pool); in the page-table form the compressed rows
    come from the page tables."""
    T, width = w.sum_q, w.width
    rows = np.empty((T, width), dtype=np.int64)
    rows[:, :SWA_COLS] = w.indices[:, :SWA_COLS]
    if w.paged:
        c = np.arange(width - SWA_COLS)
        pages = w.comp_block_tables[:, c // w.comp_page_size].astype(np.int64)
        rows[:, SWA_COLS:] = pages * w.comp_page_size + c % w.comp_page_size
    else:
        rows[:, SWA_COLS:] = w.indices[:, SWA_COLS:]
    rows[:, SWA_COLS:] += 1 << 32
    return rows


def token_pair_rows(w, num_splits: int) -> int:
    """Rows the token-pair kernel gathers per launch.  A unit is (tokens 2u
    and 2u + 1, split s) over the split's columns [s P, s P + P), P =
    ceil(W / S) (in the page-table form rounded up to a multiple of 64); it
    reads the union of the two tokens' rows there, or both lists whole when
    either token reads some row twice."""
    act, rows = active_slots(w), slot_rows(w)
    T, width, S = w.sum_q, w.width, num_splits
    per = -(-width // S)
    if w.paged:
        per = -(-per // 64) * 64
    total = 0
    for u in range(0, T, 2):
        for s in range(S):
            c0, c1 = min(width, s * per), min(width, s * per + per)
            lists = [rows[t, c0:c1][act[t, c0:c1]] for t in range(u, min(u + 2, T))]
            if any(len(np.unique(x)) < len(x) for x in lists):
                total += sum(len(x) for x in lists)
            else:
                total += len(np.unique(np.concatenate(lists)))
    return total


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def fp8_tensor_peak(bf16_tf: float):
    """FP8 dense tensor peak: the E4M3 tcgen05.mma burst rate measured on a
    GB300 (profiles/mma_peak.json, written by mma_peak.cu), else twice the
    BF16 figure (the nominal ratio)."""
    try:
        with open(os.path.join(ROOT, "profiles", "mma_peak.json")) as f:
            return float(json.load(f)["e4m3_tflops"]), "measured (profiles/mma_peak.json)"
    except (OSError, KeyError, ValueError):
        return 2.0 * bf16_tf, "2x the BF16 peak (nominal ratio)"


def code_only(text: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace collapsed (a
    comment edit leaves the compiled kernel, and so its counters, unchanged)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


# Sources with no device code: argument checks, the planner and parameter
# packing.  What they decide about a launch (kernel, splits, grid, block, shared
# memory) is matched through the plan stored with each traffic record instead.
HOST_ONLY_SOURCES = ("smla_api.cu",)
PLAN_KEYS = ("kernel", "num_splits", "ctas_per_split", "grid", "threads", "smem_bytes", "clusters")


def kernel_sources_sha() -> str:
    """Hash of the device-code sources (comments and whitespace ignored)."""
    csrc = os.path.join(ROOT, "sparse_mla_decode_token_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")) and f not in HOST_ONLY_SOURCES:
            h.update(f.encode())
            h.update(code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, plan: dict):
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    if it was taken on the current device code with this run's launch plan;
    else None."""
    return traffic_record(workload, plan)[0]


def traffic_record(workload: str, plan: dict):
    """(DRAM bytes per launch or None, a note saying where it came from or why
    there is none)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, "no profiles/traffic.json"
    ent = rec.get(workload)
    if not ent:
        return None, f"no ncu capture of workload {workload}"
    sha = kernel_sources_sha()
    if ent.get("kernel_sources_sha") != sha:
        return None, (f"the capture was taken on device code {ent.get('kernel_sources_sha')}; "
                      f"the current device code is {sha}")
    want = ent.get("plan")
    if not want or any(want.get(k) != plan.get(k) for k in PLAN_KEYS):
        return None, f"the capture's launch plan {want} differs from this run's"
    return ent.get("dram_bytes_per_launch"), f"profiles/traffic.json, device code {sha}, same launch plan"


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3][1:5]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "power_w_max": max(r[2] for r in rows), "reasons": reasons}


# -------------------------------------------------------------- oracle timing

def time_oracle(w, budget_s: float, max_tokens: int | None = None):
    """Run the CPU oracle token by token, cycling over the workload's tokens,
    until ``budget_s`` is spent or ``max_tokens`` are done; returns (tokens
    done, seconds)."""
    import oracle
    t0 = time.perf_counter()
    done = 0
    while max_tokens is None or done < max_tokens:
        oracle.run_workload(w, tokens=[done % w.sum_q])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return done, time.perf_counter() - t0


def blas_threads() -> int:
    try:
        return int(os.environ.get("OPENBLAS_NUM_THREADS", _NCPU))
    except ValueError:
        return _NCPU


# ----------------------------------------------------------------- the bench

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device="cpu") -> float:
    """The largest x over the replicas (the job's time is that of its slowest
    replica).  Needs an initialised process group when ws > 1."""
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank: int, seconds: float, ws: int, device="cpu") -> float:
    """Whole-job tokens/s of ws independent replicas: all tokens over the
    slowest replica's time."""
    return tokens_per_rank * ws / max_over_ranks(seconds, ws, device)


def workload_config(w, n: int) -> dict:
    extra = {"page_size": w.comp_page_size, "pages_per_token": int(w.comp_block_tables.shape[1])} if w.paged else {}
    return {"workload": W.CONFIG_NAMES[n], **extra, "dtype": w.dtype, "batch": w.batch, "sum_q": w.sum_q,
            "num_heads": w.num_heads, "head_dim": HEAD_DIM, "index_width": w.width,
            "swa_rows": int(w.swa_kv.shape[0]), "compressed_rows": int(w.comp_kv.shape[0]),
            "sinks": w.sinks is not None, "varlen": w.cum_seq_lens_q is not None,
            "l2": "flushed between timed steps (write of 2x L2 size, outside the timed events)",
            "parallelism": "replicas"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = W.config_workload(args.config)
    per_step = max(1, min(w.sum_q, args.ref_tokens))
    for _ in range(args.warmup):
        time_oracle(w, 1e9, max_tokens=1)
    t_total = 0.0
    tokens = 0
    for _ in range(args.steps):
        n, dt = time_oracle(w, 1e9, max_tokens=per_step)
        tokens += n
        t_total += dt
    value = tokens / t_total
    cores = blas_threads()
    sample = f"first {per_step} tokens of the workload per step, {args.steps} steps"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, args.config),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_gpu(args):
    from sparse_mla_decode_token_gb300 import binding as B
    from sparse_mla_decode_token_gb300 import build as smla_build

    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    smla_build.build()
    B.lib()
    dev = torch.device("cuda", local)
    w = W.config_workload(args.config)
    n_valid = valid_slots_per_token(w)
    gathered_bytes = int(n_valid.sum()) * w.row_bytes             # per step (the packed rows' own size)
    flops = int(n_valid.sum()) * 2 * 2 * HEAD_DIM * w.num_heads   # QK + PV, 2 flops per MAC

    def kv(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:                                # BF16 bits (query, or BF16 rows)
            return t.view(torch.int16).view(torch.bfloat16)
        return t if w.packed else t.view(torch.float8_e4m3fn)   # packed rows stay uint8

    def i32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))

    # host (pinned) per-step inputs and outputs for the end-to-end leg
    h_q = kv(w.q).pin_memory()
    h_idx = i32(w.indices).pin_memory()
    h_lens = i32(w.topk_lens).pin_memory() if w.topk_lens is not None else None
    h_seq = i32(w.seq_lens).pin_memory()
    h_cum = i32(w.cum_seq_lens_q).pin_memory() if w.cum_seq_lens_q is not None else None
    h_bt = i32(w.comp_block_tables).pin_memory() if w.paged else None
    h_hca = i32(w.hca_seq_lens).pin_memory() if w.paged else None
    h_win = i32(w.swa_topk_lens).pin_memory() if w.swa_topk_lens is not None else None
    # device-resident state: KV pools, sinks
    d_swa = kv(w.swa_kv).to(dev)
    d_comp = kv(w.comp_kv).to(dev)
    d_sinks = torch.from_numpy(w.sinks).to(dev) if w.sinks is not None else None
    d_q, d_idx, d_seq = h_q.to(dev), h_idx.to(dev), h_seq.to(dev)
    d_lens = h_lens.to(dev) if h_lens is not None else None
    d_cum = h_cum.to(dev) if h_cum is not None else None
    d_bt = h_bt.to(dev) if h_bt is not None else None
    d_hca = h_hca.to(dev) if h_hca is not None else None
    d_win = h_win.to(dev) if h_win is not None else None
    out = torch.empty((w.sum_q, w.num_heads, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.sum_q, w.num_heads), dtype=torch.float32, device=dev)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    err_word = torch.zeros(1, dtype=torch.int32, device=dev)
    args_c = B.make_args(q=d_q, swa_kv=d_swa, compressed_kv=d_comp, sparse_indices=d_idx,
                         seq_lens=d_seq, out=out, sparse_topk_lens=d_lens, cum_seq_lens_q=d_cum,
                         sinks=d_sinks, bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale,
                         out_lse=lse, kernel=args.kernel, num_splits=args.num_splits, error_word=err_word,
                         schedule=args.schedule,
                         swa_topk_lens=d_win, comp_block_tables=d_bt, comp_page_size=w.comp_page_size,
                         hca_seq_lens=d_hca, width=w.width if w.paged else None)
    plan = B.smla_plan_decode(args_c, local)
    if plan.kernel == B.KERNEL_TCGEN05_TOKEN_PAIRS:
        # rows that both tokens of a unit select are gathered once
        gathered_bytes = token_pair_rows(w, plan.num_splits) * w.row_bytes
    workspace = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    args_c.workspace, args_c.workspace_bytes = workspace.data_ptr(), workspace.numel()
    has_combine = plan.num_splits > 1
    launches_per_step = 1 + (1 if has_combine else 0)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    def new_event():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)          # materialise the CUDA event handle
        return e

    def step():
        B.smla_decode(args_c, sptr)

    # two buffer sets of the per-step tensors for the end-to-end leg; each set
    # keeps all of a step's inputs in one allocation and its outputs in another
    # (one copy in and one copy out per step: the host issues few calls)
    per_step = [(k_, h_) for k_, h_ in (("q", h_q), ("idx", h_idx), ("seq", h_seq), ("lens", h_lens),
                                        ("cum", h_cum), ("bt", h_bt), ("hca", h_hca), ("win", h_win))
                if h_ is not None]

    def packed(parts, device):
        """One uint8 buffer holding `parts` (name, like-tensor) at 256-byte
        aligned offsets, and typed views of it."""
        offs, n = {}, 0
        for k_, t_ in parts:
            offs[k_] = n
            n += (t_.numel() * t_.element_size() + 255) // 256 * 256
        buf = torch.empty(n, dtype=torch.uint8, device=device)
        if device == "cpu":
            buf = buf.pin_memory()
        views = {k_: buf[offs[k_]:offs[k_] + t_.numel() * t_.element_size()].view(t_.dtype).view(t_.shape)
                 for k_, t_ in parts}
        return buf, views

    h_in, h_in_views = packed(per_step, "cpu")
    for k_, h_ in per_step:
        h_in_views[k_].copy_(h_)
    e2e_sets = []
    for _b in range(2):
        d_in, dd = packed(per_step, dev)
        d_res, res = packed([("out", out), ("lse", lse)], dev)
        h_res, _ = packed([("out", out), ("lse", lse)], "cpu")
        a_b = B.make_args(q=dd["q"], swa_kv=d_swa, compressed_kv=d_comp, sparse_indices=dd["idx"],
                          seq_lens=dd["seq"], out=res["out"], sparse_topk_lens=dd.get("lens"),
                          cum_seq_lens_q=dd.get("cum"), sinks=d_sinks, bmm1_scale=w.bmm1_scale,
                          bmm2_scale=w.bmm2_scale, out_lse=res["lse"], kernel=args.kernel,
                          num_splits=args.num_splits, error_word=err_word, swa_topk_lens=dd.get("win"),
                          schedule=args.schedule,
                          comp_block_tables=dd.get("bt"), comp_page_size=w.comp_page_size,
                          hca_seq_lens=dd.get("hca"), width=w.width if w.paged else None)
        a_b.workspace, a_b.workspace_bytes = workspace.data_ptr(), workspace.numel()   # decodes are serial
        e2e_sets.append(dict(d_in=d_in, d_res=d_res, h_res=h_res, res=res, args=a_b,
                             ev_in=torch.cuda.Event(), ev_done=torch.cuda.Event(), ev_out=torch.cuda.Event()))
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def e2e_enqueue(steps, comp):
        """Enqueue `steps` pipelined end-to-end steps; decodes on stream `comp`."""
        for k_ in range(steps):
            st_ = e2e_sets[k_ & 1]
            if k_ >= 2:
                s_in.wait_event(st_["ev_done"])           # step k - 2 has read this set's inputs
            with torch.cuda.stream(s_in):
                st_["d_in"].copy_(h_in, non_blocking=True)
                st_["ev_in"].record(s_in)
            comp.wait_event(st_["ev_in"])
            if k_ >= 2:
                comp.wait_event(st_["ev_out"])            # step k - 2's outputs are copied out
            B.smla_decode(st_["args"], comp.cuda_stream)
            st_["ev_done"].record(comp)
            s_out.wait_event(st_["ev_done"])
            with torch.cuda.stream(s_out):
                st_["h_res"].copy_(st_["d_res"], non_blocking=True)
                st_["ev_out"].record(s_out)

    def e2e_check(steps):
        last = e2e_sets[(steps - 1) & 1]
        n_out = out.numel() * out.element_size()
        return bool(torch.equal(last["h_res"][:n_out], last["d_res"][:n_out].cpu())) and \
            bool(torch.equal(last["res"]["out"].cpu(), out.cpu())) and bool(torch.equal(last["res"]["lse"].cpu(), lse.cpu()))

    def e2e_pipelined(steps):
        """Host-loop form: seconds for `steps` pipelined end-to-end steps, and
        whether the last step's copied-back output equals the device-resident leg's."""
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ev0.record(s_in)
        e2e_enqueue(steps, stream)
        ev1.record(s_out)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / 1e3, e2e_check(steps)

    def e2e_graphed(steps):
        """The same `steps` captured once in a CUDA graph (the public call
        captured with its copies), then one replay timed: no host time inside."""
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            s_in.wait_stream(cap)
            s_out.wait_stream(cap)
            e2e_enqueue(steps, cap)
            cap.wait_stream(s_in)
            cap.wait_stream(s_out)
        g.replay()                                        # warm
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / 1e3, e2e_check(steps)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    e2e_pipelined(max(2, args.warmup))                 # warm the end-to-end path (streams, pinned copies)

    K = args.steps
    ev_step = [(new_event(), new_event()) for _ in range(K)]
    ev_main = [(new_event(), new_event()) for _ in range(K)]
    torch.cuda.synchronize()

    def barrier():
        if ws_ > 1:
            import torch.distributed as dist
            dist.barrier()

    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        for k in range(K):
            flush.zero_()
            args_c.profile_event_begin = ev_main[k][0].cuda_event
            args_c.profile_event_end = ev_main[k][1].cuda_event
            ev_step[k][0].record(stream)
            step()
            ev_step[k][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        args_c.profile_event_begin = args_c.profile_event_end = None
        # end-to-end leg through the public call: every step copies its inputs
        # from pinned host memory, decodes and copies out and LSE back to pinned
        # host memory.  Copies in, decodes and copies out run on three streams
        # with two buffer sets, so step k's copies overlap the decodes of steps
        # k - 1 and k + 1 (a serving loop's pipeline); the timed region spans
        # all K steps, every copy included.
        try:
            e2e_s, e2e_ok = e2e_graphed(K)
            e2e_how = "one CUDA graph of the K steps (captured once, replayed once)"
        except RuntimeError as exc:                      # capture refused: time the host loop instead
            print(f"e2e graph capture failed ({exc}); timing the host loop", file=sys.stderr)
            torch.cuda.synchronize()
            e2e_s, e2e_ok = e2e_pipelined(K)
            e2e_how = "host loop"
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    main_ms = [a.elapsed_time(b) for a, b in ev_main]
    total_s = max_over_ranks(sum(step_ms) / 1e3, ws_, dev)
    value = w.sum_q * K * ws_ / total_s                 # all replicas' tokens over the slowest replica's time
    e2e_value = replica_throughput(w.sum_q * K, e2e_s, ws_, dev)
    pool_mb = (d_swa.numel() * d_swa.element_size() + d_comp.numel() * d_comp.element_size()) // 2**20
    h2d = h_in.numel()                                  # bytes of the one packed copy in per step
    d2h = e2e_sets[0]["h_res"].numel()                  # bytes of the one packed copy out per step

    hbm_gbs, bf16_tf, peak_src = peaks()
    cuda_core = plan.kernel == B.KERNEL_CUDA_CORE
    if cuda_core:
        # fp32 FMA on the CUDA cores: 152 SMs x 128 lanes x 2 flops x 2.07 GHz
        dtype_tf, tensor_src = FP32_ALU_TFLOPS, "fp32 FMA lanes x clock (152 SMs x 128 x 2 x 2.07 GHz)"
    elif w.dtype == "e4m3":
        dtype_tf, tensor_src = fp8_tensor_peak(bf16_tf)
    else:
        dtype_tf, tensor_src = bf16_tf, peak_src
    main_s = statistics.mean(main_ms) / 1e3
    t_hbm = gathered_bytes / (hbm_gbs * 1e9)
    t_tc = flops / (dtype_tf * 1e12)
    if cuda_core and t_tc > t_hbm:
        roof = {"bound": "alu", "achieved": flops / main_s / 1e12, "peak": dtype_tf, "unit": "TFLOP/s"}
    elif t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": gathered_bytes / main_s / 1e9, "peak": hbm_gbs,
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / main_s / 1e12, "peak": dtype_tf,
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "alu":                          # no measured ALU peak: unit counts x clock
        roof["peak_source"] = "derived: " + tensor_src
    else:
        roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
    roof["tensor_peak_tflops"], roof["tensor_peak_source"] = dtype_tf, tensor_src
    roof["tensor_time_us"] = 1e6 * t_tc
    roof["traffic"], roof["traffic_source"] = traffic_record(W.CONFIG_NAMES[args.config], plan.as_dict())
    roof["algorithmic_bytes_per_launch"] = gathered_bytes
    roof["roofline_time_us"] = 1e6 * max(t_hbm, t_tc)
    roof["main_kernel_us"] = 1e6 * main_s
    roof["kernels_timed"] = ("decode kernel + combine (programmatic dependent launch)" if has_combine
                             else "counter memset + decode kernel" if plan.clusters > 1 else "decode kernel")
    roof["roofline_frac_whole_step"] = max(t_hbm, t_tc) / (total_s / (K * 1.0)) if ws_ == 1 else None

    if rank != 0:
        return
    cpu = None
    if ws_ == 1 and not args.no_cpu_baseline:
        n_done, dt = time_oracle(w, args.cpu_budget)
        cpu = {"value": n_done / dt, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": (f"{n_done} tokens of the same workload (its {w.sum_q} tokens in order, cycled), "
                          f"fp64 numpy, {dt:.1f} s")}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_, "steps": K, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("f32" if plan.kernel == B.KERNEL_CUDA_CORE else
                                       "e4m3" if w.dtype == "e4m3" else "bf16"), "data": "synthetic",
        "config": workload_config(w, args.config),
        "gathered_kv_gbs": gathered_bytes * K * ws_ / total_s / 1e9,
        "roofline": roof,
        "plan": plan.as_dict(),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "copy in, decode and copy out on three streams, two buffer sets; " + e2e_how,
                "l2": ("not flushed: the KV pools (%d MB) are larger than L2 (%d MB)" if pool_mb > l2 // 2**20
                       else "warm: the KV pools (%d MB) fit in L2 (%d MB)") % (pool_mb, l2 // 2**20),
                "output_matches_device_leg": e2e_ok},
        "gpu_launches": K * launches_per_step,
        "device_error_word": int(err_word.item()),
        "clocks": clocks.summary(),
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5, 6, 7, 8],
                    help="workload (3 = FP8 decode, 128 tokens, H=128; 6 = the same with page-table "
                         "compressed segments)")
    ap.add_argument("--kernel", type=int, default=0, help="smla_kernel: 0 auto, 1 CUDA-core, 2 tcgen05, 3 tcgen05 head-owned, 4 tcgen05 slot-split")
    ap.add_argument("--num-splits", type=int, default=0, help="0 = the planner's choice")
    ap.add_argument("--schedule", type=int, default=0, help="0 = auto, 1 = grid, 2 = balanced (smla_schedule)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of CPU oracle timing")
    ap.add_argument("--ref-tokens", type=int, default=4, help="oracle tokens per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
