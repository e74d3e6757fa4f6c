"""Python binding of the C ABI in ``include/smla.h`` (argument marshalling only).

Every step of the decode runs in the CUDA kernels of ``libsmla.so``; this
module only fills the ``smla_args`` struct from torch tensors and forwards the
call.  There is no fallback: if the library is missing, the first call raises.

Names follow the C ABI: ``smla_decode``, ``smla_plan_decode``,
``smla_workspace_size``, ``smla_status_string``, ``smla_last_error``; plus
``sparse_mla_decode(...)``, the tensor-level call whose argument list follows
the FlashInfer ``trtllm_batch_decode_sparse_mla_dsv4`` signature.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsmla.so")

HEAD_DIM = 512
SWA_COLS = 128
MAX_SPLITS = 64

SMLA_OK, SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED, SMLA_ERR_WORKSPACE_TOO_SMALL, SMLA_ERR_CUDA = range(5)
SMLA_BF16, SMLA_E4M3, SMLA_PACKED_FP8, SMLA_NVFP4 = 0, 1, 2, 3
# bytes of one KV row of the packed forms (BF16 query; layouts in include/smla.h)
PACKED_ROW_BYTES = {SMLA_PACKED_FP8: 584, SMLA_NVFP4: 384}
(KERNEL_AUTO, KERNEL_CUDA_CORE, KERNEL_TCGEN05, KERNEL_TCGEN05_HEAD_OWNED, KERNEL_TCGEN05_SLOT_SPLIT,
 KERNEL_TCGEN05_TOKEN_PAIRS) = 0, 1, 2, 3, 4, 5
SCHEDULE_AUTO, SCHEDULE_GRID, SCHEDULE_BALANCED = 0, 1, 2
DEVERR_INDEX_OUT_OF_RANGE = 0x1

_c_void_p = ctypes.c_void_p


class SmlaArgs(ctypes.Structure):
    _fields_ = [
        ("sum_q", ctypes.c_int32), ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
        ("width", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("q", _c_void_p), ("q_stride_token", ctypes.c_int64),
        ("swa_kv", _c_void_p), ("swa_rows", ctypes.c_int64), ("swa_row_stride", ctypes.c_int64),
        ("compressed_kv", _c_void_p), ("comp_rows", ctypes.c_int64), ("comp_row_stride", ctypes.c_int64),
        ("sparse_indices", _c_void_p), ("indices_row_stride", ctypes.c_int64),
        ("sparse_topk_lens", _c_void_p), ("seq_lens", _c_void_p),
        ("cum_seq_lens_q", _c_void_p), ("sinks", _c_void_p),
        ("bmm1_scale", ctypes.c_float), ("bmm2_scale", ctypes.c_float),
        ("bmm1_scale_dev", _c_void_p), ("bmm2_scale_dev", _c_void_p),
        ("out", _c_void_p), ("out_lse", _c_void_p),
        ("workspace", _c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("num_splits", ctypes.c_int32), ("max_splits", ctypes.c_int32), ("kernel", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("error_word", _c_void_p),
        ("profile_event_begin", _c_void_p), ("profile_event_end", _c_void_p),
        ("comp_block_tables", _c_void_p), ("block_table_stride", ctypes.c_int64),
        ("comp_max_pages", ctypes.c_int32), ("comp_page_size", ctypes.c_int32),
        ("hca_seq_lens", _c_void_p), ("swa_topk_lens", _c_void_p),
    ]


class SmlaPlan(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int32), ("num_splits", ctypes.c_int32),
        ("ctas_per_split", ctypes.c_int32), ("grid", ctypes.c_int32),
        ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
        ("clusters", ctypes.c_int32), ("workspace_bytes", ctypes.c_size_t),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class SmlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{smla_status_string(status)}: {message}")
        self.status = status


_lib = None

# (symbol, restype, argtypes) of every entry point the header declares
EXPORTS = {
    "smla_plan_decode": (ctypes.c_int, [ctypes.POINTER(SmlaArgs), ctypes.c_int, ctypes.POINTER(SmlaPlan)]),
    "smla_plan_decode_for_sm_count": (ctypes.c_int, [ctypes.POINTER(SmlaArgs), ctypes.c_int,
                                                     ctypes.POINTER(SmlaPlan)]),
    "smla_validate_host": (ctypes.c_int, [ctypes.POINTER(SmlaArgs)]),
    "smla_workspace_size": (ctypes.c_int, [ctypes.POINTER(SmlaArgs), ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "smla_decode": (ctypes.c_int, [ctypes.POINTER(SmlaArgs), _c_void_p]),
    "smla_decode_static_workspace": (ctypes.c_int, [ctypes.POINTER(SmlaArgs), _c_void_p]),
    "smla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "smla_last_error": (ctypes.c_char_p, []),
    "smla_abi_version": (ctypes.c_int, []),
}


def lib():
    """Load ``libsmla.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libsmla.so is not built ({LIB_PATH}); run "
                              "sparse_mla_decode_token_gb300.build.build() first")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, argt) in EXPORTS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = argt
        _lib = handle
    return _lib


# ------------------------------------------------------------- raw ABI calls

def smla_status_string(status: int) -> str:
    return lib().smla_status_string(status).decode()


def smla_last_error() -> str:
    return lib().smla_last_error().decode()


def smla_abi_version() -> int:
    return lib().smla_abi_version()


def _check(status: int) -> None:
    if status != SMLA_OK:
        raise SmlaError(status, smla_last_error())


def smla_plan_decode(args: SmlaArgs, device: int = 0) -> SmlaPlan:
    plan = SmlaPlan()
    _check(lib().smla_plan_decode(ctypes.byref(args), device, ctypes.byref(plan)))
    return plan


def smla_plan_decode_for_sm_count(args: SmlaArgs, sm_count: int) -> SmlaPlan:
    """The plan for a device with ``sm_count`` SMs; queries no device."""
    plan = SmlaPlan()
    _check(lib().smla_plan_decode_for_sm_count(ctypes.byref(args), sm_count, ctypes.byref(plan)))
    return plan


def smla_validate_host(args: SmlaArgs) -> None:
    """Check a call's index data; its index-data pointers must be HOST memory
    (raises ``SmlaError`` naming the first bad entry)."""
    _check(lib().smla_validate_host(ctypes.byref(args)))


def _validate_on_host(a: SmlaArgs, **tensors) -> None:
    """``smla_validate_host`` on host copies of the call's index data (one
    device-to-host copy each: a debugging aid, enabled by SMLA_VALIDATE=1)."""
    h = SmlaArgs.from_buffer_copy(a)
    keep = []

    def host(t):
        c = t.detach().to("cpu").contiguous()
        keep.append(c)
        return c

    si = host(tensors["sparse_indices"])
    h.sparse_indices, h.indices_row_stride = si.data_ptr(), si.stride(0)
    h.seq_lens = host(tensors["seq_lens"]).data_ptr()
    for name in ("sparse_topk_lens", "cum_seq_lens_q", "hca_seq_lens", "swa_topk_lens"):
        t = tensors.get(name)
        setattr(h, name, None if t is None else host(t).data_ptr())
    bt = tensors.get("comp_block_tables")
    if bt is not None:
        bt = host(bt)
        h.comp_block_tables, h.block_table_stride = bt.data_ptr(), bt.stride(0)
    smla_validate_host(h)


def smla_workspace_size(args: SmlaArgs, device: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().smla_workspace_size(ctypes.byref(args), device, ctypes.byref(n)))
    return int(n.value)


def smla_decode(args: SmlaArgs, stream: Optional[int] = None) -> None:
    """Launch on ``stream`` (a raw cudaStream_t value; default: torch's current stream)."""
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check(lib().smla_decode(ctypes.byref(args), _c_void_p(stream)))


STATIC_WORKSPACE_BYTES = 64 << 20


def smla_decode_static_workspace(args: SmlaArgs, stream: Optional[int] = None) -> None:
    """Like ``smla_decode`` but with the library's own static split-K scratch
    (``args.workspace`` is ignored; nothing is allocated).  For callers that
    cannot allocate device memory; calls that overlap on the GPU race."""
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check(lib().smla_decode_static_workspace(ctypes.byref(args), _c_void_p(stream)))


# ---------------------------------------------------------- tensor marshalling

def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SMLA_BF16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return SMLA_E4M3
    raise TypeError(f"q/KV dtype {t.dtype} is not bfloat16 or float8_e4m3fn")


def _kv_dtype_code(q: torch.Tensor, kv: torch.Tensor) -> int:
    """KV element type: the query's, or a packed row form (uint8 rows of 584 or
    384 bytes with a BF16 query)."""
    if q.dtype == torch.bfloat16 and kv.dtype == torch.uint8:
        for code, nbytes in PACKED_ROW_BYTES.items():
            if kv.shape[-1] == nbytes:
                return code
    return _dtype_code(kv)


def _rows_and_stride(kv: torch.Tensor, row: int = HEAD_DIM) -> tuple[int, int]:
    """Flatten a KV pool view ([..., row], any page layout) to (rows, row stride)."""
    if kv.shape[-1] != row or kv.stride(-1) != 1:
        raise ValueError(f"KV pool must end in a contiguous dim of {row}; got {tuple(kv.shape)}")
    flat = kv.reshape(-1, row) if kv.dim() != 2 else kv
    if flat.data_ptr() != kv.data_ptr():
        raise ValueError("KV pool view cannot be flattened to rows without a copy")
    return flat.shape[0], flat.stride(0)


def make_args(*, q: torch.Tensor, swa_kv: torch.Tensor, compressed_kv: torch.Tensor,
              sparse_indices: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
              sparse_topk_lens: Optional[torch.Tensor] = None,
              cum_seq_lens_q: Optional[torch.Tensor] = None,
              sinks: Optional[torch.Tensor] = None,
              bmm1_scale=1.0, bmm2_scale=1.0,
              out_lse: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None,
              num_splits: int = 0, max_splits: int = 0, kernel: int = KERNEL_AUTO,
              error_word: Optional[torch.Tensor] = None,
              swa_topk_lens: Optional[torch.Tensor] = None,
              schedule: int = 0,
              comp_block_tables: Optional[torch.Tensor] = None,
              comp_page_size: int = 0, hca_seq_lens: Optional[torch.Tensor] = None,
              width: Optional[int] = None) -> SmlaArgs:
    """Fill ``smla_args`` from tensors (no copies; wrong layouts raise).  Every
    tensor must live on the CUDA device of ``q`` (the library reads raw device
    pointers; a host pointer would fault the GPU), and the call must then be
    made with that device current (``sparse_mla_decode`` does both).

    Page-table form: ``comp_block_tables`` ``[T, max_pages]`` int32 page IDs,
    ``comp_page_size`` rows per page and ``hca_seq_lens`` ``[B]``; the index
    table then holds the 128 SWA columns and ``width`` (logical columns)
    defaults to ``128 + max_pages * comp_page_size``."""
    # layout first (tensor metadata only), so that a wrong shape, dtype or
    # length answers the same on any device; placement after
    if q.dim() == 4:                       # dense [B, q_len, H, 512]
        try:
            q = q.view(-1, q.shape[2], q.shape[3])     # a copy would leave the library a dangling pointer
        except RuntimeError as exc:
            raise ValueError(f"dense query [B, q_len, H, {HEAD_DIM}] must flatten to [T, H, {HEAD_DIM}] "
                             f"without a copy: {exc}") from None
    if q.dim() != 3 or q.shape[-1] != HEAD_DIM or q.stride(-1) != 1 or q.stride(1) != HEAD_DIM:
        raise ValueError(f"query must be [T, H, {HEAD_DIM}] with contiguous heads; got {tuple(q.shape)}")
    T, H = q.shape[0], q.shape[1]
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.numel() != T * H * HEAD_DIM:
        raise ValueError("out must be a contiguous bfloat16 tensor of T*H*512 elements")
    if out_lse is not None and (out_lse.dtype != torch.float32 or not out_lse.is_contiguous()
                                or out_lse.numel() != T * H):
        raise ValueError("out_lse must be a contiguous float32 tensor of T*H elements")
    for name, t in (("sparse_indices", sparse_indices), ("seq_lens", seq_lens),
                    ("sparse_topk_lens", sparse_topk_lens), ("cum_seq_lens_q", cum_seq_lens_q),
                    ("swa_topk_lens", swa_topk_lens), ("comp_block_tables", comp_block_tables),
                    ("hca_seq_lens", hca_seq_lens), ("error_word", error_word)):
        if t is not None and t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    B = seq_lens.numel()
    # arrays the kernels index by token, request or head: contiguous and long
    # enough (a short one would be read past its end on the device)
    for name, t, need in (("seq_lens", seq_lens, B), ("sparse_topk_lens", sparse_topk_lens, T),
                          ("cum_seq_lens_q", cum_seq_lens_q, B + 1), ("swa_topk_lens", swa_topk_lens, T),
                          ("hca_seq_lens", hca_seq_lens, B), ("sinks", sinks, H),
                          ("error_word", error_word, 1)):
        if t is None:
            continue
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.numel() < need:
            raise ValueError(f"{name} has {t.numel()} entries; the call reads {need}")
    if sinks is not None and sinks.dtype != torch.float32:
        raise ValueError("sinks must be float32 with at least H entries")
    for name, val in (("bmm1", bmm1_scale), ("bmm2", bmm2_scale)):
        if isinstance(val, torch.Tensor):
            if val.dtype != torch.float32:
                raise TypeError(f"{name}_scale tensor must be float32")
            if val.numel() < 1:
                raise ValueError(f"{name}_scale tensor is empty")
    if sparse_indices.dim() == 3:          # [T, 1, W]
        if sparse_indices.shape[1] != 1:
            raise ValueError(f"sparse_indices [T, 1, W] must have 1 in dim 1; got {tuple(sparse_indices.shape)}")
        sparse_indices = sparse_indices[:, 0, :]
    if sparse_indices.dim() != 2 or sparse_indices.stride(-1) != 1:
        raise ValueError("sparse_indices must be [T, W] with a contiguous last dim")
    if sparse_indices.shape[0] < T:
        raise ValueError(f"sparse_indices has {sparse_indices.shape[0]} rows for {T} query tokens")

    kv_code = _kv_dtype_code(q, swa_kv)
    if _kv_dtype_code(q, compressed_kv) != kv_code:
        raise TypeError("swa_kv and compressed_kv must share one element type")
    row = PACKED_ROW_BYTES.get(kv_code, HEAD_DIM)
    swa_rows, swa_stride = _rows_and_stride(swa_kv, row)
    comp_rows, comp_stride = _rows_and_stride(compressed_kv, row)
    a = SmlaArgs()
    a.sum_q, a.num_heads, a.width = T, H, sparse_indices.shape[-1]
    if comp_block_tables is not None:
        if comp_block_tables.dim() != 2 or comp_block_tables.stride(-1) != 1 or comp_block_tables.shape[0] != T:
            raise ValueError("comp_block_tables must be [T, max_pages] with a contiguous last dim")
        if hca_seq_lens is None or comp_page_size < 1:
            raise ValueError("the page-table form needs hca_seq_lens and comp_page_size >= 1")
        a.comp_block_tables, a.block_table_stride = comp_block_tables.data_ptr(), comp_block_tables.stride(0)
        a.comp_max_pages, a.comp_page_size = comp_block_tables.shape[1], int(comp_page_size)
        a.hca_seq_lens = hca_seq_lens.data_ptr()
        a.width = SWA_COLS + a.comp_max_pages * a.comp_page_size if width is None else int(width)
    elif width is not None and width != a.width:
        raise ValueError("width is the index table's width in the index form")
    a.swa_topk_lens = _ptr(swa_topk_lens)
    a.batch = B
    a.dtype = kv_code
    if kv_code not in PACKED_ROW_BYTES and _dtype_code(q) != kv_code:
        raise TypeError("query, swa_kv and compressed_kv must share one dtype")
    a.q, a.q_stride_token = q.data_ptr(), q.stride(0)
    a.swa_kv, a.swa_rows, a.swa_row_stride = swa_kv.data_ptr(), swa_rows, swa_stride
    a.compressed_kv, a.comp_rows, a.comp_row_stride = compressed_kv.data_ptr(), comp_rows, comp_stride
    a.sparse_indices, a.indices_row_stride = sparse_indices.data_ptr(), sparse_indices.stride(0)
    a.sparse_topk_lens = _ptr(sparse_topk_lens)
    a.seq_lens = seq_lens.data_ptr()
    a.cum_seq_lens_q = _ptr(cum_seq_lens_q)
    a.sinks = _ptr(sinks)
    for name, val in (("bmm1", bmm1_scale), ("bmm2", bmm2_scale)):
        if isinstance(val, torch.Tensor):
            setattr(a, f"{name}_scale_dev", val.data_ptr())
            setattr(a, f"{name}_scale", 1.0)
        else:
            setattr(a, f"{name}_scale", float(val))
    a.out, a.out_lse = out.data_ptr(), _ptr(out_lse)
    if workspace is not None:
        a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    a.num_splits, a.max_splits, a.kernel, a.schedule = num_splits, max_splits, kernel, schedule
    a.error_word = _ptr(error_word)
    if os.environ.get("SMLA_VALIDATE") == "1":
        _validate_on_host(a, sparse_indices=sparse_indices, seq_lens=seq_lens, sparse_topk_lens=sparse_topk_lens,
                          cum_seq_lens_q=cum_seq_lens_q, hca_seq_lens=hca_seq_lens, swa_topk_lens=swa_topk_lens,
                          comp_block_tables=comp_block_tables)

    dev = q.device
    for name, t in (("q", q), ("swa_kv", swa_kv), ("compressed_kv", compressed_kv),
                    ("sparse_indices", sparse_indices), ("seq_lens", seq_lens), ("out", out),
                    ("sparse_topk_lens", sparse_topk_lens), ("cum_seq_lens_q", cum_seq_lens_q),
                    ("sinks", sinks), ("out_lse", out_lse), ("workspace", workspace),
                    ("error_word", error_word), ("bmm1_scale", bmm1_scale), ("bmm2_scale", bmm2_scale),
                    ("swa_topk_lens", swa_topk_lens), ("comp_block_tables", comp_block_tables),
                    ("hca_seq_lens", hca_seq_lens)):
        if isinstance(t, torch.Tensor) and (t.device.type != "cuda" or t.device != dev):
            raise ValueError(f"{name} is on {t.device}; every tensor must be on the CUDA device of q ({dev})")
    if dev.type != "cuda":
        raise ValueError(f"q is on {dev}; the decode runs on a CUDA device")
    return a


def sparse_mla_decode(query: torch.Tensor, swa_kv_cache: torch.Tensor, workspace_buffer: Optional[torch.Tensor],
                      sparse_indices: torch.Tensor, compressed_kv_cache: torch.Tensor,
                      sparse_topk_lens: Optional[torch.Tensor], seq_lens: torch.Tensor,
                      out: Optional[torch.Tensor] = None, bmm1_scale=1.0, bmm2_scale=1.0,
                      sinks: Optional[torch.Tensor] = None,
                      cum_seq_lens_q: Optional[torch.Tensor] = None,
                      out_lse: Optional[torch.Tensor] = None,
                      num_splits: int = 0, max_splits: int = 0, kernel: int = KERNEL_AUTO,
                      error_word: Optional[torch.Tensor] = None,
                      stream: Optional[int] = None,
                      schedule: int = 0,
                      swa_topk_lens: Optional[torch.Tensor] = None,
                      hca_compressed_block_tables: Optional[torch.Tensor] = None,
                      hca_seq_lens: Optional[torch.Tensor] = None,
                      comp_page_size: Optional[int] = None,
                      width: Optional[int] = None):
    """Decode; returns ``(out, out_lse)``.  ``out`` / ``out_lse`` are allocated when not given.

    With ``hca_compressed_block_tables`` the compressed segment is given as
    page tables; ``comp_page_size`` defaults to the compressed cache view's
    rows per page (``[num_pages, page_size, 512]``)."""
    if hca_compressed_block_tables is not None and comp_page_size is None:
        if compressed_kv_cache.dim() < 3:
            raise ValueError("pass comp_page_size, or a compressed cache view [num_pages, page_size, 512]")
        comp_page_size = compressed_kv_cache.shape[-2]
    T = query.shape[0] if query.dim() == 3 else query.shape[0] * query.shape[1]
    H = query.shape[-2]
    if out is None:
        out = torch.empty((T, H, HEAD_DIM), dtype=torch.bfloat16, device=query.device)
    if out_lse is None:
        out_lse = torch.empty((T, H), dtype=torch.float32, device=query.device)
    args = make_args(q=query, swa_kv=swa_kv_cache, compressed_kv=compressed_kv_cache,
                     sparse_indices=sparse_indices, seq_lens=seq_lens, out=out,
                     sparse_topk_lens=sparse_topk_lens, cum_seq_lens_q=cum_seq_lens_q,
                     sinks=sinks, bmm1_scale=bmm1_scale, bmm2_scale=bmm2_scale,
                     out_lse=out_lse, workspace=workspace_buffer, num_splits=num_splits,
                     max_splits=max_splits, kernel=kernel, error_word=error_word, schedule=schedule,
                     swa_topk_lens=swa_topk_lens, comp_block_tables=hca_compressed_block_tables,
                     comp_page_size=comp_page_size or 0, hca_seq_lens=hca_seq_lens, width=width)
    with torch.cuda.device(query.device):   # the library plans and launches on the current device
        smla_decode(args, stream)
    return out, out_lse


def workspace_size(query, sparse_indices, seq_lens, *, num_splits=0, max_splits=0,
                   kernel=KERNEL_AUTO, cum_seq_lens_q=None, device: int = 0,
                   width: Optional[int] = None, schedule: int = 0, kv_cache=None) -> int:
    """Workspace bytes for a call with these shapes (no device memory is read);
    ``width`` = logical columns in the page-table form; ``kv_cache`` (a pool
    view, metadata only) gives the KV element type when it differs from the
    query's (packed rows)."""
    a = SmlaArgs()
    q3 = query if query.dim() == 3 else query.view(-1, query.shape[2], query.shape[3])
    a.sum_q, a.num_heads = q3.shape[0], q3.shape[1]
    a.width = sparse_indices.shape[-1] if width is None else int(width)
    a.batch = seq_lens.numel()
    a.dtype = _dtype_code(q3) if kv_cache is None else _kv_dtype_code(q3, kv_cache)
    a.cum_seq_lens_q = _ptr(cum_seq_lens_q)
    a.num_splits, a.max_splits, a.kernel, a.schedule = num_splits, max_splits, kernel, schedule
    return smla_workspace_size(a, device)
