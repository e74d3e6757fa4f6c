"""Seeded synthetic inputs for DeepSeek-V4 sparse MLA decode.

This module only draws inputs.  It holds none of the attention arithmetic, so
the CPU oracle (``oracle/``) and the CUDA path can both consume the very same
bytes without sharing any code of the method.

A ``Workload`` carries raw host buffers exactly as the operation takes them:

* ``q``        -- ``[sum_q, H, 512]`` BF16 bits (``uint16``) or FP8 E4M3 bits (``uint8``)
* ``swa_kv``   -- ``[swa_rows, 512]``  same element type as ``q``
* ``comp_kv``  -- ``[comp_rows, 512]`` same element type as ``q``
* ``indices``  -- ``[sum_q, W]`` int32; columns 0..127 index ``swa_kv``, the
  rest index ``comp_kv``; -1 masks a slot
* ``topk_lens``-- ``[sum_q]`` int32 or ``None`` (every column active)
* ``seq_lens`` -- ``[batch]`` int32, original KV length per request
* ``cum_seq_lens_q`` -- ``[batch + 1]`` int32 or ``None`` (uniform q_len)
* ``sinks``    -- ``[H]`` float32 or ``None``
* ``bmm1_scale``, ``bmm2_scale`` -- float32-representable Python floats

A page-table workload (``make_paged_workload``) instead holds only the 128 SWA
columns in ``indices`` and gives the compressed segment as per-token rows of
page IDs ``comp_block_tables`` with ``comp_page_size`` rows per page and
per-request slot counts ``hca_seq_lens`` (FlashInfer
``trtllm_batch_decode_sparse_mla_dsv4`` page, Parameters:
hca_compressed_block_tables, hca_seq_lens, swa_topk_lens).

The five named workloads follow the shapes of the FlashInfer
``trtllm_batch_decode_sparse_mla_dsv4`` page (head dim 512, 128 SWA columns,
H in {64, 128}, BF16 or per-tensor FP8 E4M3) and the vLLM DeepSeek-V4 caller's
scale folding (``bmm1 = softmax_scale * q_scale * kv_scale``, ``bmm2 = kv_scale``).
Values are N(0, 1); FP8 tensors are quantised with a per-tensor scale
``amax / 448`` by round-to-nearest-even after clamping to the E4M3 range.

Packed KV rows (``dtype`` ``"packed_fp8"``: 584 bytes, ``"nvfp4"``: 384
bytes per row; the byte layouts are the oracle's reading of the FlashInfer
pages, which give only the sizes) hold the same N(0, 1) values: the 448 NoPE
dims quantised per block (packed_fp8: a power-of-two UE8M0 exponent per 64
dims so that the block fits E4M3; nvfp4: an fp32 row scale amax / (6 * 448)
and an E4M3 scale per 16 dims so that the block fits E2M1), the 64 RoPE dims
in BF16.  The query is BF16 with these rows.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

HEAD_DIM = 512
SWA_COLS = 128
E4M3_MAX = 448.0
NOPE_DIMS = 448
PACKED_ROW_BYTES = {"packed_fp8": 584, "nvfp4": 384}
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                      # "bf16", "e4m3", "packed_fp8" or "nvfp4"
    batch: int
    num_heads: int
    q: np.ndarray
    swa_kv: np.ndarray
    comp_kv: np.ndarray
    indices: np.ndarray
    topk_lens: Optional[np.ndarray]
    seq_lens: np.ndarray
    cum_seq_lens_q: Optional[np.ndarray]
    sinks: Optional[np.ndarray]
    bmm1_scale: float
    bmm2_scale: float
    q_scale: float = 1.0
    kv_scale: float = 1.0
    # page-table form of the compressed segment (None: index form)
    comp_block_tables: Optional[np.ndarray] = None   # [sum_q, max_pages] int32 page IDs
    comp_page_size: int = 0
    hca_seq_lens: Optional[np.ndarray] = None        # [batch] int32: 128 window + compressed slots
    swa_topk_lens: Optional[np.ndarray] = None       # [sum_q] int32 visible window, or None
    logical_width: Optional[int] = None              # W when the index table holds SWA columns only

    @property
    def sum_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def width(self) -> int:
        return int(self.logical_width if self.logical_width is not None else self.indices.shape[1])

    @property
    def paged(self) -> bool:
        return self.comp_block_tables is not None

    @property
    def elem_bytes(self) -> int:
        """Bytes per KV element (packed rows: per byte of the row)."""
        return 2 if self.dtype == "bf16" else 1

    @property
    def packed(self) -> bool:
        return self.dtype in PACKED_ROW_BYTES

    @property
    def row_bytes(self) -> int:
        """Bytes of one KV row (512 elements, or the packed row size)."""
        return PACKED_ROW_BYTES[self.dtype] if self.packed else HEAD_DIM * self.elem_bytes


# --------------------------------------------------------------------------
# element encodings (input synthesis only)
# --------------------------------------------------------------------------

def _to_bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _to_e4m3_bits(x: torch.Tensor, scale: float) -> np.ndarray:
    y = (x / scale).clamp_(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _normal(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def _encode(x: torch.Tensor, dtype: str, scale: float) -> np.ndarray:
    return _to_bf16_bits(x) if dtype == "bf16" else _to_e4m3_bits(x, scale)


def _bf16_bytes(x: torch.Tensor) -> np.ndarray:
    """[n, k] values -> [n, 2k] bytes of their BF16 bits, little-endian."""
    return np.ascontiguousarray(_to_bf16_bits(x)).view(np.uint8)


def _to_packed_fp8_rows(x: torch.Tensor) -> np.ndarray:
    """[n, 512] values -> [n, 584] packed rows (448 E4M3 NoPE scaled by a
    UE8M0 exponent per 64 dims, 8 bytes of exponents, 64 BF16 RoPE)."""
    n = x.shape[0]
    nope = x[:, :NOPE_DIMS].reshape(n, 7, 64)
    amax = nope.abs().amax(dim=2).clamp_min(1e-30)
    e = torch.ceil(torch.log2(amax / E4M3_MAX)).clamp(-127, 127)        # block / 2^e fits E4M3
    codes = _to_e4m3_bits((nope / torch.exp2(e)[:, :, None]).reshape(n, NOPE_DIMS), 1.0)
    rows = np.zeros((n, 584), dtype=np.uint8)
    rows[:, :NOPE_DIMS] = codes
    rows[:, NOPE_DIMS:NOPE_DIMS + 7] = (e + 127).to(torch.int64).numpy().astype(np.uint8)
    rows[:, 456:584] = _bf16_bytes(x[:, NOPE_DIMS:])
    return rows


def _to_e2m1_codes(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code of each value (|v| <= 6 expected)."""
    mid = (E2M1_MAGNITUDES[1:] + E2M1_MAGNITUDES[:-1]) / 2.0
    mag = np.searchsorted(mid, np.abs(v)).astype(np.uint8)              # 0..7
    return mag | np.where(v < 0, 8, 0).astype(np.uint8)


def _to_nvfp4_rows(x: torch.Tensor) -> np.ndarray:
    """[n, 512] values -> [n, 384] rows (448 E2M1 NoPE, 28 E4M3 block scales
    per 16 dims, 64 BF16 RoPE, an fp32 row scale)."""
    n = x.shape[0]
    nope = x[:, :NOPE_DIMS].double()
    g = (nope.abs().amax(dim=1) / (6.0 * E4M3_MAX)).clamp_min(1e-30).float()           # fp32 row scale
    blocks = nope.reshape(n, 28, 16)
    bscale = (blocks.abs().amax(dim=2) / 6.0 / g.double()[:, None]).float()
    bcodes = _to_e4m3_bits(bscale, 1.0)                                                  # [n, 28]
    bval = torch.from_numpy(bcodes.copy()).view(torch.float8_e4m3fn).double()
    denom = (bval * g.double()[:, None]).clamp_min(1e-300)
    v = (blocks / denom[:, :, None]).reshape(n, NOPE_DIMS).numpy()
    codes = _to_e2m1_codes(v)
    rows = np.zeros((n, 384), dtype=np.uint8)
    rows[:, :224] = codes[:, 0::2] | (codes[:, 1::2] << 4)
    rows[:, 224:252] = bcodes
    rows[:, 252:380] = _bf16_bytes(x[:, NOPE_DIMS:])
    rows[:, 380:384] = np.ascontiguousarray(g.numpy().astype(np.float32)).view(np.uint8).reshape(n, 4)
    return rows


def _encode_rows(x: torch.Tensor, dtype: str, scale: float) -> np.ndarray:
    """KV pool values -> the pool's stored form."""
    if dtype == "packed_fp8":
        return _to_packed_fp8_rows(x)
    if dtype == "nvfp4":
        return _to_nvfp4_rows(x)
    return _encode(x, dtype, scale)


def _pertensor_scale(*xs: torch.Tensor) -> float:
    amax = max(float(x.abs().max()) for x in xs)
    return float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0


def f32(x: float) -> float:
    """Round a Python float to the nearest float32 (scales travel as fp32)."""
    return float(np.float32(x))


# --------------------------------------------------------------------------
# index-table construction
# --------------------------------------------------------------------------

def token_positions(seq_lens: np.ndarray, q_lens: np.ndarray) -> np.ndarray:
    """Absolute position of every flattened query token.

    Decode tokens are right-aligned: token i of a request of q_len tokens
    sits at position seq_len - q_len + i (FlashInfer msa_sparse_decode_attention
    page, description).  Used here only to lay out the SWA ring columns.
    """
    out = []
    for sl, ql in zip(seq_lens.tolist(), q_lens.tolist()):
        out.extend(sl - ql + i for i in range(ql))
    return np.asarray(out, dtype=np.int64)


def swa_ring_columns(pos: int, ring_base: int, ring_len: int) -> np.ndarray:
    """128 SWA columns for a token at ``pos`` whose request owns a ring of rows.

    Column c < w holds the row of position ``pos - (w - 1) + c`` with
    ``w = min(128, pos + 1)``; columns past ``w`` are -1.
    """
    w = min(SWA_COLS, max(0, pos + 1))
    cols = np.full(SWA_COLS, -1, dtype=np.int32)
    p = pos - (w - 1) + np.arange(w)
    cols[:w] = ring_base + (p % ring_len)
    return cols


def _unique_rows(rng: np.random.Generator, n_rows: int, k: int) -> np.ndarray:
    return rng.choice(n_rows, size=k, replace=False).astype(np.int32)


def _draw_values(gen: torch.Generator, dtype: str, sum_q: int, num_heads: int,
                 swa_rows: int, comp_rows: int):
    """N(0, 1) query and pools, encoded; FP8 takes per-tensor scales amax / 448;
    packed rows carry their own scales and go with a BF16 query."""
    qf = _normal(gen, (sum_q, num_heads, HEAD_DIM))
    swaf = _normal(gen, (swa_rows, HEAD_DIM))
    compf = _normal(gen, (comp_rows, HEAD_DIM))
    if dtype == "e4m3":
        q_scale = _pertensor_scale(qf)
        kv_scale = _pertensor_scale(swaf, compf)
    else:
        q_scale = kv_scale = 1.0
    q_dtype = "e4m3" if dtype == "e4m3" else "bf16"
    return (_encode(qf, q_dtype, q_scale), _encode_rows(swaf, dtype, kv_scale),
            _encode_rows(compf, dtype, kv_scale), q_scale, kv_scale)


def _lengths(q_lens, seq_lens, batch: int):
    q_lens = np.broadcast_to(np.asarray(q_lens, dtype=np.int64), (batch,)).copy()
    seq_lens = np.broadcast_to(np.asarray(seq_lens, dtype=np.int64), (batch,)).astype(np.int32)
    cum = np.zeros(batch + 1, dtype=np.int32)
    cum[1:] = np.cumsum(q_lens)
    return q_lens, seq_lens, cum


# --------------------------------------------------------------------------
# generic generator
# --------------------------------------------------------------------------

def make_workload(*, name: str = "custom", seed: int, dtype: str, batch: int,
                  q_lens, num_heads: int, swa_rows: int, comp_rows: int,
                  width: int, seq_lens, ring_len: Optional[int] = None,
                  comp_valid=None, topk_lens=None, sinks: bool = False,
                  varlen: Optional[bool] = None,
                  softmax_scale: float = 1.0 / math.sqrt(HEAD_DIM)) -> Workload:
    """Draw one workload.

    ``q_lens`` and ``seq_lens`` are per-request sequences (or scalars).
    ``comp_valid[t]`` (default: every compressed column) is the number of
    leading compressed columns of token t that hold a real row; the rest are
    -1.  ``topk_lens`` is ``None`` (every column active), a scalar, or a
    per-token sequence.  SWA columns come from a per-request ring of
    ``ring_len`` rows (default ``swa_rows // batch``).
    """
    assert dtype in ("bf16", "e4m3", "packed_fp8", "nvfp4")
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    q_lens, seq_lens, cum = _lengths(q_lens, seq_lens, batch)
    sum_q = int(q_lens.sum())
    if varlen is None:
        varlen = bool((q_lens != q_lens[0]).any())
    ring_len = ring_len if ring_len is not None else swa_rows // batch
    n_comp_cols = width - SWA_COLS
    assert n_comp_cols >= 0

    q, swa_kv, comp_kv, q_scale, kv_scale = _draw_values(gen, dtype, sum_q, num_heads, swa_rows, comp_rows)

    # index table
    pos = token_positions(seq_lens, q_lens)
    req_of_token = np.repeat(np.arange(batch), q_lens)
    indices = np.full((sum_q, width), -1, dtype=np.int32)
    if comp_valid is None:
        comp_valid = np.full(sum_q, n_comp_cols, dtype=np.int64)
    comp_valid = np.broadcast_to(np.asarray(comp_valid, dtype=np.int64), (sum_q,))
    for t in range(sum_q):
        b = int(req_of_token[t])
        indices[t, :SWA_COLS] = swa_ring_columns(int(pos[t]), b * ring_len, ring_len)
        k = int(comp_valid[t])
        if k > 0:
            indices[t, SWA_COLS:SWA_COLS + k] = _unique_rows(rng, comp_rows, k)
    if topk_lens is not None:
        topk_lens = np.broadcast_to(np.asarray(topk_lens, dtype=np.int64), (sum_q,)).astype(np.int32)

    sink_vals = _normal(gen, (num_heads,)).numpy().astype(np.float32) if sinks else None
    bmm1 = f32(softmax_scale * q_scale * kv_scale)
    bmm2 = f32(kv_scale)
    return Workload(name=name, dtype=dtype, batch=batch, num_heads=num_heads,
                    q=q, swa_kv=swa_kv, comp_kv=comp_kv, indices=indices,
                    topk_lens=topk_lens, seq_lens=seq_lens,
                    cum_seq_lens_q=cum if varlen else None, sinks=sink_vals,
                    bmm1_scale=bmm1, bmm2_scale=bmm2, q_scale=q_scale,
                    kv_scale=kv_scale)


def make_paged_workload(*, name: str = "paged", seed: int, dtype: str, batch: int,
                        q_lens, num_heads: int, swa_rows: int, comp_pages: int,
                        page_size: int, max_pages: int, hca_seq_lens, seq_lens,
                        ring_len: Optional[int] = None, topk_lens=None,
                        swa_topk_lens=None, sinks: bool = False,
                        varlen: Optional[bool] = None, fill_unused: int = -1,
                        width: Optional[int] = None, per_token_pages: bool = False,
                        softmax_scale: float = 1.0 / math.sqrt(HEAD_DIM)) -> Workload:
    """Draw a workload whose compressed segment is a page table.

    Every request owns ``max_pages`` distinct random pages of the compressed
    pool (``comp_pages * page_size`` rows); its tokens share that page list,
    unless ``per_token_pages``, where every token draws a list of its own (the
    table has one row per token, so a token must read its own row, not its
    request's).
    Table entries past the request's footprint ``ceil((hca_seq_lens[b] - 128)
    / page_size)`` hold ``fill_unused`` (never read as rows).  All 128 SWA
    columns hold legal ring rows; the visible window is ``swa_topk_lens`` when
    given, else the seq_lens rule.  ``width`` (logical columns) defaults to
    ``128 + max_pages * page_size``.
    """
    assert dtype in ("bf16", "e4m3", "packed_fp8", "nvfp4")
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    q_lens, seq_lens, cum = _lengths(q_lens, seq_lens, batch)
    sum_q = int(q_lens.sum())
    if varlen is None:
        varlen = bool((q_lens != q_lens[0]).any())
    ring_len = ring_len if ring_len is not None else swa_rows // batch
    assert ring_len >= SWA_COLS and batch * ring_len <= swa_rows
    comp_rows = comp_pages * page_size
    assert max_pages <= comp_pages
    hca = np.broadcast_to(np.asarray(hca_seq_lens, dtype=np.int64), (batch,)).astype(np.int32)
    assert int(hca.max()) - SWA_COLS <= max_pages * page_size
    width = SWA_COLS + max_pages * page_size if width is None else int(width)

    q, swa_kv, comp_kv, q_scale, kv_scale = _draw_values(gen, dtype, sum_q, num_heads, swa_rows, comp_rows)

    pos = token_positions(seq_lens, q_lens)
    req_of_token = np.repeat(np.arange(batch), q_lens)
    indices = np.empty((sum_q, SWA_COLS), dtype=np.int32)
    tables = np.full((sum_q, max_pages), fill_unused, dtype=np.int32)
    pages_of = [rng.choice(comp_pages, size=max_pages, replace=False).astype(np.int32) for _ in range(batch)]
    if per_token_pages:            # drawn after the shared lists: the default stream is unchanged
        token_pages = [rng.choice(comp_pages, size=max_pages, replace=False).astype(np.int32)
                       for _ in range(sum_q)]
    for t in range(sum_q):
        b = int(req_of_token[t])
        p = int(pos[t]) - (SWA_COLS - 1) + np.arange(SWA_COLS)       # every column a legal ring row
        indices[t] = b * ring_len + (p % ring_len)
        used = -(-max(0, int(hca[b]) - SWA_COLS) // page_size)
        tables[t, :used] = (token_pages[t] if per_token_pages else pages_of[b])[:used]
    if topk_lens is not None:
        topk_lens = np.broadcast_to(np.asarray(topk_lens, dtype=np.int64), (sum_q,)).astype(np.int32)
    if swa_topk_lens is not None:
        swa_topk_lens = np.broadcast_to(np.asarray(swa_topk_lens, dtype=np.int64), (sum_q,)).astype(np.int32)
    sink_vals = _normal(gen, (num_heads,)).numpy().astype(np.float32) if sinks else None
    return Workload(name=name, dtype=dtype, batch=batch, num_heads=num_heads,
                    q=q, swa_kv=swa_kv, comp_kv=comp_kv, indices=indices,
                    topk_lens=topk_lens, seq_lens=seq_lens,
                    cum_seq_lens_q=cum if varlen else None, sinks=sink_vals,
                    bmm1_scale=f32(softmax_scale * q_scale * kv_scale), bmm2_scale=f32(kv_scale),
                    q_scale=q_scale, kv_scale=kv_scale, comp_block_tables=tables,
                    comp_page_size=page_size, hca_seq_lens=hca, swa_topk_lens=swa_topk_lens,
                    logical_width=width)


# --------------------------------------------------------------------------
# the named workloads
# --------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny_bf16_h64",
    2: "bf16_decode_b32_h128",
    3: "fp8_decode_b128_h128",
    4: "varlen_spec_bf16_h64",
    5: "long_splitk_fp8_b4_h128",
    6: "paged_fp8_b128_h128",
    7: "nvfp4_decode_b128_h128",
    8: "packed_fp8_decode_b128_h128",
}


def config_workload(n: int) -> Workload:
    """Workload ``n`` (1..8); seed 1000 + n.  Workload 6 is workload 3's shape
    with the compressed segment given as page tables; workloads 7 and 8 are
    workload 3's shape with 384-byte NVFP4 and 584-byte packed FP8 KV rows
    (BF16 query)."""
    seed = 1000 + n
    rng = np.random.default_rng(seed + 7919)
    if n == 1:
        # 2 tokens, H=64, BF16; 128 SWA + 128 compressed unique rows; lens U[129, 256].
        return make_workload(name=CONFIG_NAMES[1], seed=seed, dtype="bf16", batch=2,
                             q_lens=1, num_heads=64, swa_rows=256, comp_rows=512,
                             width=256, seq_lens=4096, ring_len=128,
                             topk_lens=rng.integers(129, 257, size=2), sinks=False)
    if n == 2:
        # 32 tokens, H=128, BF16; 128 SWA + c_t ~ U[256, 512] compressed then -1.
        c = rng.integers(256, 513, size=32)
        lens = np.where(np.arange(32) % 2 == 0, 640, 128 + c)
        return make_workload(name=CONFIG_NAMES[2], seed=seed, dtype="bf16", batch=32,
                             q_lens=1, num_heads=128, swa_rows=32 * 128,
                             comp_rows=65536, width=640,
                             seq_lens=rng.integers(4096, 32769, size=32),
                             ring_len=128, comp_valid=c, topk_lens=lens, sinks=True)
    if n == 3:
        # 128 tokens, H=128, FP8 E4M3; 128 SWA + 2048 compressed, all valid.
        return make_workload(name=CONFIG_NAMES[3], seed=seed, dtype="e4m3", batch=128,
                             q_lens=1, num_heads=128, swa_rows=128 * 128,
                             comp_rows=262144, width=2176,
                             seq_lens=rng.integers(8192, 65537, size=128),
                             ring_len=128, topk_lens=2176, sinks=False)
    if n == 4:
        # 64 requests, q_len U{1..4} (varlen), H=64, BF16; 128 SWA + 1024 compressed.
        q_lens = rng.integers(1, 5, size=64)
        sum_q = int(q_lens.sum())
        return make_workload(name=CONFIG_NAMES[4], seed=seed, dtype="bf16", batch=64,
                             q_lens=q_lens, num_heads=64, swa_rows=64 * 256,
                             comp_rows=65536, width=1152,
                             seq_lens=rng.integers(4096, 32769, size=64),
                             ring_len=256, topk_lens=rng.integers(129, 1153, size=sum_q),
                             sinks=True, varlen=True)
    if n == 5:
        # 4 tokens, H=128, FP8; 128 SWA + 16384 compressed over a 1M-row pool.
        return make_workload(name=CONFIG_NAMES[5], seed=seed, dtype="e4m3", batch=4,
                             q_lens=1, num_heads=128, swa_rows=4 * 128,
                             comp_rows=1 << 20, width=128 + 16384,
                             seq_lens=1 << 20, ring_len=128, topk_lens=128 + 16384,
                             sinks=True)
    if n == 6:
        # 128 tokens, H=128, FP8 E4M3; 128 SWA + 2048 compressed slots per token on
        # 16 pages of 128 rows (each request its own random pages of a 262,144-row pool).
        return make_paged_workload(name=CONFIG_NAMES[6], seed=seed, dtype="e4m3", batch=128,
                                   q_lens=1, num_heads=128, swa_rows=128 * 128, comp_pages=2048,
                                   page_size=128, max_pages=16, hca_seq_lens=128 + 2048,
                                   seq_lens=rng.integers(8192, 65537, size=128), ring_len=128,
                                   topk_lens=2176)
    if n in (7, 8):
        # workload 3's shape (128 tokens, H=128, 128 SWA + 2048 compressed,
        # all valid) with packed KV rows and a BF16 query
        return make_workload(name=CONFIG_NAMES[n], seed=seed, dtype="nvfp4" if n == 7 else "packed_fp8",
                             batch=128, q_lens=1, num_heads=128, swa_rows=128 * 128,
                             comp_rows=262144, width=2176,
                             seq_lens=rng.integers(8192, 65537, size=128),
                             ring_len=128, topk_lens=2176, sinks=False)
    raise ValueError(f"no workload {n}")

