"""CPU oracle for DeepSeek-V4 sparse MLA decode attention (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this file; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` do.
It shares no code with the CUDA path.

What it computes is the plain definition of the operation, written out in
float64 with no blocking, fusion or reordering:

for every flattened query token t and head h, over the set V_t of slots the
token's index row selects,

    l_j   = bmm1_scale * <q[t, h, :], kv_j>                      (natural-log units)
    O[d]  = bmm2_scale * sum_j e^{l_j} kv_j[d] / (sum_j e^{l_j} + e^{sink_h})
    LSE2  = log2 sum_j e^{l_j}                                   (sink excluded)

Sources (FlashInfer and vLLM documentation pages):

* trtllm_batch_decode_sparse_mla_dsv4, description (SM100/SM103 paragraph):
  head dim 512; BF16 or per-tensor FP8 E4M3 query and KV; BF16 output; the
  first 128 index columns address the SWA pool, the rest the compressed pool;
  ``sparse_topk_lens`` counts active columns including the 128 SWA ones;
  ``seq_lens`` bounds the SWA validity window.
* same page, Parameters: ``bmm1_scale`` (QK and softmax scale), ``bmm2_scale``
  (VO scale), ``sinks`` (per-head sink logits), ``cum_seq_lens_q`` (varlen
  query, top-k lengths in flattened token order).
* cake_sparse_mla_sm120_dsv4_nvfp4_decode, Parameters: -1 masks a slot;
  ``out_lse`` is the base-2 log-sum-exp; ``attn_sink`` joins the softmax
  normalisation; ``mid_out`` / ``mid_lse`` are split partials.
* msa_sparse_decode_attention, description: decode tokens are right-aligned,
  token i of a request sits at position seq_len - q_len + i.
* vLLM DeepseekV4FlashInferMLAAttention: FP8 scale folding
  ``bmm1 = scale * q_scale * kv_scale``, ``bmm2 = kv_scale``.

Readings where the pages are silent (each is listed in the design notes):

* SWA window: SWA column j is valid iff j < min(128, pos + 1), pos being the
  right-aligned token position.  PARITY UNPINNED by the pages (our reading).
* A fully masked token yields O = 0 and LSE = -inf.
* The sink is a natural-log logit, not multiplied by bmm1_scale.
* LSE2 excludes the sink.  PARITY UNPINNED by the pages (our reading);
  ``lse_with_sink=True`` gives the other reading.
* ``sparse_topk_lens`` outside [0, W] is clamped to that range.
* V = K = the whole 512-wide row.
* Duplicate indices each count as their own slot.
* An index < -1 or >= the pool's row count is a caller error: raised by
  default, or treated as masked with ``invalid_index="mask"``.

Packed KV rows (§8(f) f2; trtllm_batch_decode_sparse_mla_dsv4, description,
SM120/SM121 paragraph: "packed uint8 ... 584 bytes per token", BF16 query;
cake_sparse_mla_sm120_dsv4_nvfp4_decode, Parameters: kv_cache "NVFP4 ...
384 bytes per token", q "448 NoPE dims, then 64 RoPE dims").  The pages give
only the sizes; the byte layouts are our reading (PARITY UNPINNED by the
pages for the layout; pinned here against the bit-format definitions):

* ``packed_fp8`` (584 B): bytes [0, 448) the 448 NoPE values in E4M3; bytes
  [448, 455) seven UE8M0 block exponents e_b, NoPE dim d scaled by
  2^(e_{d // 64} - 127); byte 455 unused; bytes [456, 584) the 64 RoPE values
  in BF16 (little-endian).
* ``nvfp4`` (384 B): bytes [0, 224) the 448 NoPE values in E2M1, dim 2i in
  the low nibble and dim 2i + 1 in the high nibble of byte i; bytes
  [224, 252) 28 E4M3 block scales, NoPE dim d scaled by scale_{d // 16};
  bytes [252, 380) the 64 RoPE values in BF16; bytes [380, 384) an fp32 row
  scale applied to every NoPE value.
* With either, the query is BF16; K = V = the decoded 512-wide row.

Page-table form of the compressed segment (trtllm_batch_decode_sparse_mla_dsv4,
Parameters: hca_swa_indices, hca_compressed_block_tables, hca_seq_lens,
swa_topk_lens, hca_sparse_indices_format):

* the index table then holds only the 128 SWA columns; compressed slot c of
  token t (logical column 128 + c) is row
  ``block_tables[t, c // page_size] * page_size + c % page_size`` of the
  compressed pool (the canonical page_id * page_size + page_offset expansion);
* request b backs ``hca_seq_lens[b] - 128`` compressed slots (the count
  includes the 128 window slots); slots past it are not read, and
  ``sparse_topk_lens`` (logical columns) may cut further;
* ``swa_topk_lens[t]`` (optional, in either form), clamped to [0, 128], is the
  token's visible window and replaces the seq_lens rule.  Reading: the window
  is a leading prefix of the SWA columns, as for the seq_lens rule.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

HEAD_DIM = 512
SWA_COLS = 128
LN2 = math.log(2.0)
LOG2E = 1.0 / LN2


# --------------------------------------------------------------------------
# element decoding, from the bit-format definitions
# --------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 is the upper 16 bits of an IEEE-754 binary32."""
    wide = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return wide.view(np.float32).astype(np.float64)


def _e4m3_value(code: int) -> float:
    """OCP 8-bit floating point E4M3 ("fn" variant).

    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field 0
    encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity,
    so the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(bits, dtype=np.uint8)]


def _e2m1_value(code: int) -> float:
    """OCP 4-bit floating point E2M1: 1 sign bit, 2 exponent bits (bias 1),
    1 mantissa bit; exponent field 0 encodes the subnormal m/2."""
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * m * 0.5
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)

PACKED_ROW_BYTES = {"packed_fp8": 584, "nvfp4": 384}
NOPE_DIMS = 448


def ue8m0_to_f64(bits: np.ndarray) -> np.ndarray:
    """UE8M0 (unsigned exponent-only scale): 2^(e - 127)."""
    return np.exp2(np.asarray(bits, dtype=np.float64) - 127.0)


def _bf16_pairs(raw: np.ndarray) -> np.ndarray:
    """[..., 2n] bytes (little-endian) -> [..., n] BF16 values."""
    u16 = raw[..., 0::2].astype(np.uint16) | (raw[..., 1::2].astype(np.uint16) << np.uint16(8))
    return bf16_to_f64(u16)


def decode_packed_fp8_rows(rows: np.ndarray) -> np.ndarray:
    """[n, 584] uint8 -> [n, 512] float64 (layout in the module docstring)."""
    rows = np.asarray(rows, dtype=np.uint8)
    nope = e4m3_to_f64(rows[:, :NOPE_DIMS])
    scale = ue8m0_to_f64(rows[:, NOPE_DIMS:NOPE_DIMS + 7])            # [n, 7]
    nope = nope * np.repeat(scale, 64, axis=1)
    rope = _bf16_pairs(rows[:, 456:584])
    return np.concatenate([nope, rope], axis=1)


def decode_nvfp4_rows(rows: np.ndarray) -> np.ndarray:
    """[n, 384] uint8 -> [n, 512] float64 (layout in the module docstring)."""
    rows = np.asarray(rows, dtype=np.uint8)
    packed = rows[:, :224]
    codes = np.empty((rows.shape[0], NOPE_DIMS), dtype=np.uint8)
    codes[:, 0::2] = packed & 0x0F
    codes[:, 1::2] = packed >> 4
    block = e4m3_to_f64(rows[:, 224:252])                              # [n, 28]
    row_scale = rows[:, 380:384].copy().view(np.float32).astype(np.float64)   # [n, 1]
    nope = E2M1_TABLE[codes] * np.repeat(block, 16, axis=1) * row_scale
    rope = _bf16_pairs(rows[:, 252:380])
    return np.concatenate([nope, rope], axis=1)


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Query elements (bf16 / e4m3 bits; BF16 for the packed KV forms)."""
    if dtype in ("bf16", "packed_fp8", "nvfp4"):
        return bf16_to_f64(bits)
    if dtype == "e4m3":
        return e4m3_to_f64(bits)
    raise ValueError(dtype)


def decode_rows(rows: np.ndarray, dtype: str) -> np.ndarray:
    """KV rows of one pool -> [n, 512] float64."""
    if dtype == "packed_fp8":
        return decode_packed_fp8_rows(rows)
    if dtype == "nvfp4":
        return decode_nvfp4_rows(rows)
    return decode(rows, dtype)


# --------------------------------------------------------------------------
# step a1: token metadata
# --------------------------------------------------------------------------

def token_request(t: int, sum_q: int, batch: int,
                  cum_seq_lens_q: Optional[np.ndarray]) -> tuple[int, int, int]:
    """(request b, index i inside the request, q_len of the request).

    Without ``cum_seq_lens_q`` the query is dense ``[batch, q_len, ...]`` with
    q_len = sum_q / batch.
    """
    if cum_seq_lens_q is None:
        q_len = sum_q // batch
        return t // q_len, t % q_len, q_len
    cum = [int(c) for c in cum_seq_lens_q]
    for b in range(batch):
        if cum[b] <= t < cum[b + 1]:
            return b, t - cum[b], cum[b + 1] - cum[b]
    raise ValueError(f"token {t} is outside cum_seq_lens_q")


def token_position(t, sum_q, batch, cum_seq_lens_q, seq_lens) -> int:
    """Right-aligned absolute position seq_len - q_len + i."""
    b, i, q_len = token_request(t, sum_q, batch, cum_seq_lens_q)
    return int(seq_lens[b]) - q_len + i


# --------------------------------------------------------------------------
# step a2: which slots a token reads
# --------------------------------------------------------------------------

def valid_slots(t: int, *, indices, topk_lens, seq_lens, cum_seq_lens_q,
                batch: int, swa_rows: int, comp_rows: int,
                invalid_index: str = "raise", width: Optional[int] = None,
                swa_topk_lens=None, comp_block_tables=None,
                comp_page_size: int = 0, hca_seq_lens=None) -> list[tuple[int, str, int]]:
    """List of (column j, pool name, row) that token t attends to, in column order.

    ``width`` is the logical column count W (default: the index table's
    width); with ``comp_block_tables`` the compressed columns come from the
    page table (see the module docstring) and ``indices`` needs only the 128
    SWA columns.
    """
    sum_q = indices.shape[0]
    width = indices.shape[1] if width is None else int(width)
    n_lim = width if topk_lens is None else min(max(int(topk_lens[t]), 0), width)
    b, i, q_len = token_request(t, sum_q, batch, cum_seq_lens_q)
    if swa_topk_lens is None:
        w_swa = min(SWA_COLS, max(0, int(seq_lens[b]) - q_len + i + 1))
    else:
        w_swa = min(max(int(swa_topk_lens[t]), 0), SWA_COLS)
    paged = comp_block_tables is not None
    if paged:
        n_comp = max(0, int(hca_seq_lens[b]) - SWA_COLS)
    out = []
    for j in range(n_lim):
        if j < SWA_COLS:
            idx = int(indices[t, j])
            if idx == -1 or j >= w_swa:
                continue
            pool, rows = "swa", swa_rows
        elif paged:
            c = j - SWA_COLS
            if c >= n_comp:
                continue
            idx = int(comp_block_tables[t, c // comp_page_size]) * comp_page_size + c % comp_page_size
            pool, rows = "comp", comp_rows
        else:
            idx = int(indices[t, j])
            if idx == -1:
                continue
            pool, rows = "comp", comp_rows
        if not 0 <= idx < rows:
            if invalid_index == "raise":
                raise IndexError(f"token {t} column {j}: index {idx} outside {pool} pool of {rows} rows")
            continue
        out.append((j, pool, idx))
    return out


# --------------------------------------------------------------------------
# steps a4-a6 and a9 for one token: masked softmax attention over the slots
# --------------------------------------------------------------------------

def attend(q_t: np.ndarray, kv: np.ndarray, bmm1: float, bmm2: float,
           sinks: Optional[np.ndarray], lse_with_sink: bool = False):
    """q_t [H, 512], kv [n, 512] (both float64) -> (O [H, 512], LSE2 [H])."""
    H = q_t.shape[0]
    if kv.shape[0] == 0:
        return np.zeros((H, HEAD_DIM)), np.full(H, -np.inf)
    logits = bmm1 * (q_t @ kv.T)                        # [H, n]
    m = logits.max(axis=1)                               # [H]
    e = np.exp(logits - m[:, None])                      # [H, n]
    z = e.sum(axis=1)                                    # [H]
    denom = z.copy()
    if sinks is not None:
        denom = denom + np.exp(np.asarray(sinks, dtype=np.float64) - m)
    o = bmm2 * (e @ kv) / denom[:, None]
    lse2 = (m + np.log(denom if lse_with_sink else z)) * LOG2E
    return o, lse2


# --------------------------------------------------------------------------
# steps a7-a9: split partials and their log-sum-exp combine
# --------------------------------------------------------------------------

def partial(q_t: np.ndarray, kv: np.ndarray, bmm1: float):
    """Unsunk, unscaled normalised partial (O_s, LSE2_s) over one slot subset."""
    return attend(q_t, kv, bmm1, 1.0, None)


def combine_partials(o_s: np.ndarray, lse_s: np.ndarray, bmm2: float,
                     sinks: Optional[np.ndarray], lse_with_sink: bool = False):
    """o_s [S, H, 512], lse_s [S, H] -> (O [H, 512], LSE2 [H]).

    LSE2 = log2 sum_s 2^{LSE2_s};  O = sum_s 2^{LSE2_s - LSE2} O_s; then the
    sink joins the normaliser: O *= 1 / (1 + 2^{sink * log2 e - LSE2}); then
    O *= bmm2.
    """
    H = o_s.shape[1]
    mx = lse_s.max(axis=0)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    w = np.where(np.isfinite(lse_s), np.exp2(lse_s - mx_safe[None, :]), 0.0)  # [S, H]
    wsum = w.sum(axis=0)
    out = np.zeros((H, HEAD_DIM))
    lse = np.full(H, -np.inf)
    ok = ~empty
    out[ok] = (w[:, ok, None] * o_s[:, ok, :]).sum(axis=0) / wsum[ok, None]
    lse[ok] = mx_safe[ok] + np.log2(wsum[ok])
    if sinks is not None:
        sink2 = np.asarray(sinks, dtype=np.float64) * LOG2E
        factor = np.where(ok, 1.0 / (1.0 + np.exp2(sink2 - np.where(ok, lse, 0.0))), 0.0)
        out = out * factor[:, None]
        if lse_with_sink:
            lse = np.where(ok, np.logaddexp2(lse, sink2), lse)
    return bmm2 * out, lse


# --------------------------------------------------------------------------
# the whole operation
# --------------------------------------------------------------------------

def _gather(pool_bits: dict, slots, dtype: str) -> np.ndarray:
    if not slots:
        return np.zeros((0, HEAD_DIM))
    rows = [pool_bits[p][r] for (_, p, r) in slots]
    return decode_rows(np.stack(rows), dtype)


def sparse_mla_decode(*, dtype: str, batch: int, q, swa_kv, comp_kv, indices,
                      topk_lens=None, seq_lens, cum_seq_lens_q=None, sinks=None,
                      bmm1_scale: float, bmm2_scale: float,
                      tokens: Optional[Sequence[int]] = None,
                      splits: Optional[int] = None, lse_with_sink: bool = False,
                      invalid_index: str = "raise", width: Optional[int] = None,
                      swa_topk_lens=None, comp_block_tables=None,
                      comp_page_size: int = 0, hca_seq_lens=None):
    """Return (O [T, H, 512] float64, LSE2 [T, H] float64) for ``tokens``.

    Arguments are raw element bits as the operation takes them (see the module
    docstring).  ``splits`` (optional) evaluates every token as that many
    contiguous column ranges of its active columns and merges them with
    ``combine_partials``; it must agree with the unsplit result.
    """
    sum_q = q.shape[0]
    tokens = range(sum_q) if tokens is None else list(tokens)
    pools = {"swa": swa_kv, "comp": comp_kv}
    bmm1 = float(bmm1_scale)
    bmm2 = float(bmm2_scale)
    O, L = [], []
    for t in tokens:
        slots = valid_slots(t, indices=indices, topk_lens=topk_lens, seq_lens=seq_lens,
                            cum_seq_lens_q=cum_seq_lens_q, batch=batch,
                            swa_rows=swa_kv.shape[0], comp_rows=comp_kv.shape[0],
                            invalid_index=invalid_index, width=width,
                            swa_topk_lens=swa_topk_lens, comp_block_tables=comp_block_tables,
                            comp_page_size=comp_page_size, hca_seq_lens=hca_seq_lens)
        q_t = decode(q[t], dtype)                         # [H, 512]
        if splits is None:
            o, lse = attend(q_t, _gather(pools, slots, dtype), bmm1, bmm2, sinks, lse_with_sink)
        else:
            w_all = indices.shape[1] if width is None else int(width)
            n_lim = w_all if topk_lens is None else min(max(int(topk_lens[t]), 0), w_all)
            per = -(-n_lim // splits) if n_lim > 0 else 0
            o_s, lse_s = [], []
            for s in range(splits):
                lo, hi = s * per, min(n_lim, (s + 1) * per)
                part = [sl for sl in slots if lo <= sl[0] < hi]
                o_p, l_p = partial(q_t, _gather(pools, part, dtype), bmm1)
                o_s.append(o_p)
                lse_s.append(l_p)
            o, lse = combine_partials(np.stack(o_s), np.stack(lse_s), bmm2, sinks, lse_with_sink)
        O.append(o)
        L.append(lse)
    H = q.shape[1]
    if not O:
        return np.zeros((0, H, HEAD_DIM)), np.zeros((0, H))
    return np.stack(O), np.stack(L)


def run_workload(w, **kw):
    """Convenience: evaluate a ``Workload`` (duck-typed) with the oracle."""
    return sparse_mla_decode(dtype=w.dtype, batch=w.batch, q=w.q, swa_kv=w.swa_kv,
                             comp_kv=w.comp_kv, indices=w.indices, topk_lens=w.topk_lens,
                             seq_lens=w.seq_lens, cum_seq_lens_q=w.cum_seq_lens_q,
                             sinks=w.sinks, bmm1_scale=w.bmm1_scale,
                             bmm2_scale=w.bmm2_scale, width=w.width,
                             swa_topk_lens=getattr(w, "swa_topk_lens", None),
                             comp_block_tables=getattr(w, "comp_block_tables", None),
                             comp_page_size=getattr(w, "comp_page_size", 0),
                             hca_seq_lens=getattr(w, "hca_seq_lens", None), **kw)
