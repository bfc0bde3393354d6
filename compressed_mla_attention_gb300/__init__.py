"""Python binding of libqsfm, the quantized shared-KV sparse MLA attention
forward for sm_103a (QuantSparseFlashMla / KvQuantSparseAttnSharedKv, and the
bf16-KV SparseCompressedFlashAttention).

This module only marshals arguments: it fills the C ``qsfm_params`` struct
from torch tensors (device pointers, shapes) and calls the C ABI declared in
``include/qsfm.h`` through ctypes. Every step of the computation runs in the
library's CUDA kernels. There is no CPU or PyTorch fallback: if the library
is missing, importing the op functions raises.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libqsfm.so")

NUM_HEADS = 64
HEAD_DIM = 512
BLOCK_SIZE = 128
METADATA_INTS = 1024
MAX_CTAS = 256
LAYOUT_BSND = 0
LAYOUT_TND = 1
KV_FP8_FP32_SCALES = 0
KV_PACKED640 = 1
KV_BF16 = 2
PACKED_ROW_BYTES = 640

STATUS = {
    0: "QSFM_OK",
    1: "QSFM_ERR_INVALID_ARG",
    2: "QSFM_ERR_UNSUPPORTED",
    3: "QSFM_ERR_CUDA",
    4: "QSFM_ERR_WORKSPACE",
    5: "QSFM_ERR_DEVICE_FAULT",
    6: "QSFM_ERR_TIMEOUT",
}
FAULT_ORI_BLOCK_ID = 0x1
FAULT_CMP_BLOCK_ID = 0x2
FAULT_ORI_TABLE_COL = 0x4
FAULT_CMP_TABLE_COL = 0x8
FAULT_METADATA = 0x10
FAULT_TIMEOUT = 0x20
FAULT_RANGE = 0x40
FAULT_KV_ROW = 0x80
LAYOUT_KV = {"PA_BBND": 0, "BSND": 1, "TND": 2}

_i32 = ctypes.c_int32
_ptr = ctypes.c_void_p


class QsfmParams(ctypes.Structure):
    """Mirror of ``qsfm_params`` (include/qsfm.h); field order must match."""

    _fields_ = [
        ("batch", _i32), ("max_s1", _i32), ("total_t", _i32), ("n1", _i32), ("d", _i32),
        ("k2", _i32), ("ori_block_size", _i32), ("cmp_block_size", _i32),
        ("ori_max_blocks", _i32), ("cmp_max_blocks", _i32), ("ori_num_blocks", _i32),
        ("cmp_num_blocks", _i32), ("num_ctas", _i32),
        ("q", _ptr), ("ori_kv", _ptr), ("ori_scale", _ptr), ("cmp_kv", _ptr), ("cmp_scale", _ptr),
        ("cmp_sparse_indices", _ptr), ("ori_block_table", _ptr), ("cmp_block_table", _ptr),
        ("cu_seqlens_q", _ptr), ("seqused_q", _ptr), ("seqused_ori_kv", _ptr),
        ("seqused_cmp_kv", _ptr), ("cmp_residual_kv", _ptr), ("cmp_topk_length", _ptr),
        ("sinks", _ptr), ("metadata", _ptr),
        ("softmax_scale", ctypes.c_float), ("cmp_ratio", _i32), ("ori_mask_mode", _i32),
        ("cmp_mask_mode", _i32), ("ori_win_left", _i32), ("ori_win_right", _i32),
        ("layout_q", _i32), ("return_lse", _i32),
        ("attn_out", _ptr), ("softmax_lse", _ptr),
        ("kv_layout", _i32),
        ("layout_kv", _i32), ("ori_kv_len", _i32), ("cmp_kv_len", _i32), ("k1", _i32),
        ("cu_seqlens_ori_kv", _ptr), ("cu_seqlens_cmp_kv", _ptr), ("ori_sparse_indices", _ptr),
        ("ori_topk_length", _ptr),
    ]


class IndexerParams(ctypes.Structure):
    """Mirror of ``qsfm_indexer_params`` (include/qsfm.h); field order must match."""

    _fields_ = [
        ("batch", _i32), ("max_s1", _i32), ("total_t", _i32), ("heads", _i32), ("dim", _i32), ("topk", _i32),
        ("block_size", _i32), ("max_blocks", _i32), ("num_blocks", _i32), ("layout_q", _i32),
        ("mask_mode", _i32), ("cmp_ratio", _i32), ("return_value", _i32),
        ("query", _ptr), ("query_scale", _ptr), ("weights", _ptr), ("key", _ptr), ("key_scale", _ptr),
        ("block_table", _ptr), ("seqused_k", _ptr), ("cmp_residual_k", _ptr), ("cu_seqlens_q", _ptr),
        ("seqused_q", _ptr), ("sparse_indices", _ptr), ("sparse_values", _ptr),
        ("layout_k", _i32), ("max_sk", _i32), ("total_k", _i32), ("cu_seqlens_k", _ptr),
        ("output_idx_offset", _ptr),
    ]


class QsfmError(RuntimeError):
    def __init__(self, fn: str, code: int, cuda_error: str = ""):
        detail = f" ({cuda_error})" if cuda_error else ""
        super().__init__(f"{fn} returned {STATUS.get(code, code)}{detail}")
        self.code = code
        self.cuda_error = cuda_error


_LIB: Optional[ctypes.CDLL] = None

EXPORTS = {
    "qsfm_params_init": (None, [ctypes.POINTER(QsfmParams)]),
    "qsfm_metadata": (_i32, [ctypes.POINTER(QsfmParams), _ptr, _ptr]),
    "qsfm_forward_workspace_size": (_i32, [ctypes.POINTER(QsfmParams), ctypes.POINTER(ctypes.c_size_t)]),
    "qsfm_forward": (_i32, [ctypes.POINTER(QsfmParams), _ptr, ctypes.c_size_t, _ptr]),
    "qsfm_attention": (_i32, [ctypes.POINTER(QsfmParams), _ptr, ctypes.c_size_t, _ptr]),
    "qsfm_combine": (_i32, [ctypes.POINTER(QsfmParams), _ptr, ctypes.c_size_t, _ptr]),
    "qsfm_forward_noalloc": (_i32, [ctypes.POINTER(QsfmParams), _ptr]),
    "qsfm_debug_gather": (_i32, [ctypes.POINTER(QsfmParams), _ptr, _i32, _i32, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "qsfm_debug_bounded_wait": (_i32, [ctypes.c_uint64, _ptr, _ptr]),
    "qsfm_get_device_status": (_i32, [ctypes.POINTER(_i32)]),
    "qsfm_status_string": (ctypes.c_char_p, [_i32]),
    "qsfm_abi_version": (_i32, []),
    "qsfm_last_cuda_error": (_i32, [ctypes.POINTER(ctypes.c_char_p)]),
    "qsfm_indexer_params_init": (None, [ctypes.POINTER(IndexerParams)]),
    "qsfm_lightning_indexer_workspace_size": (_i32, [ctypes.POINTER(IndexerParams),
                                                     ctypes.POINTER(ctypes.c_size_t)]),
    "qsfm_lightning_indexer": (_i32, [ctypes.POINTER(IndexerParams), _ptr, ctypes.c_size_t, _ptr]),
}


def lib() -> ctypes.CDLL:
    """The loaded C library. Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m compressed_mla_attention_gb300.build` (no fallback exists)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(fn: str, code: int):
    if code != 0:
        name = ""
        if code == 3:  # QSFM_ERR_CUDA: name the runtime error behind it
            s = ctypes.c_char_p()
            lib().qsfm_last_cuda_error(ctypes.byref(s))
            name = (s.value or b"").decode()
        raise QsfmError(fn, code, name)


def _dptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to qsfm must be contiguous")
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_params(
    *,
    q,
    attn_out,
    ori_kv,
    ori_scale,
    ori_block_table,
    seqused_ori_kv,
    layout: str = "BSND",
    batch: Optional[int] = None,
    cmp_kv=None,
    cmp_scale=None,
    cmp_block_table=None,
    cmp_sparse_indices=None,
    cu_seqlens_q=None,
    seqused_q=None,
    seqused_cmp_kv=None,
    cmp_residual_kv=None,
    cmp_topk_length=None,
    sinks=None,
    metadata=None,
    softmax_lse=None,
    softmax_scale: float = HEAD_DIM ** -0.5,
    cmp_ratio: int = 1,
    ori_mask_mode: int = 4,
    cmp_mask_mode: int = 3,
    ori_win_left: int = 127,
    ori_win_right: int = 0,
    return_lse: bool = False,
    num_ctas: int = 0,
    layout_kv: str = "PA_BBND",
    cu_seqlens_ori_kv=None,
    cu_seqlens_cmp_kv=None,
    ori_sparse_indices=None,
    ori_topk_length=None,
) -> QsfmParams:
    """Fill a QsfmParams from device tensors (shapes as in include/qsfm.h).

    q / attn_out: BSND [B, S1, N1, 512] or TND [T1, N1, 512] bf16, N1 = 64 or 128.
    Paged KV (layout_kv "PA_BBND"): [blocks, 128, 1, 512] uint8 (fp8 e4m3fn
    bytes) with fp32 scales [blocks, 128, 1, 8], or packed [blocks, 128, 1,
    640] uint8 rows (bf16 rope, e4m3fn nope, e8m0 scales; scales None), or
    bf16 rows [blocks, 128, 1, 512] (scales None); block tables int32 [B,
    width]. Non-paged KV: layout_kv "BSND" ([B, S, 1, row], q BSND) or "TND"
    ([T, 1, row], q TND, cu_seqlens_ori_kv / cu_seqlens_cmp_kv int32 [B+1]),
    no block tables. ori_sparse_indices int32 [T, 1, K1] (or BSND
    [B, S1, 1, K1]) with optional ori_topk_length int32 [T].
    """
    p = QsfmParams()
    lib().qsfm_params_init(ctypes.byref(p))
    if layout == "BSND":
        p.layout_q = LAYOUT_BSND
        if q.dim() == 4:
            p.batch, p.max_s1 = int(q.shape[0]), int(q.shape[1])
        else:  # flat [B * S1, 64, 512]
            if batch is None:
                raise ValueError("flat BSND q needs batch=")
            p.batch = int(batch)
            p.max_s1 = int(q.shape[0]) // max(1, p.batch)
        p.total_t = p.batch * p.max_s1
    elif layout == "TND":
        p.layout_q = LAYOUT_TND
        p.total_t = int(q.shape[0])
        p.batch = int(cu_seqlens_q.shape[0]) - 1 if cu_seqlens_q is not None else int(batch or 0)
        p.max_s1 = 0
    else:
        raise ValueError(layout)
    p.n1, p.d = int(q.shape[-2]), int(q.shape[-1])
    p.k2 = int(cmp_sparse_indices.shape[-1]) if cmp_sparse_indices is not None else 0
    # bf16 rows, packed 640-byte rows (bf16 rope, e4m3 nope, e8m0 scales) or fp8 rows + fp32 scales
    if cmp_kv is not None and (cmp_kv.dtype != ori_kv.dtype or cmp_kv.shape[-1] != ori_kv.shape[-1]):
        raise ValueError("ori_kv and cmp_kv must have the same row format")
    if str(ori_kv.dtype) == "torch.bfloat16":
        p.kv_layout = KV_BF16
    elif int(ori_kv.shape[-1]) == PACKED_ROW_BYTES:
        p.kv_layout = KV_PACKED640
    else:
        p.kv_layout = KV_FP8_FP32_SCALES
    if layout_kv not in LAYOUT_KV:
        raise ValueError(layout_kv)
    p.layout_kv = LAYOUT_KV[layout_kv]
    if layout_kv == "PA_BBND":
        p.ori_block_size = int(ori_kv.shape[1])
        p.ori_max_blocks = int(ori_block_table.shape[-1])
        p.ori_num_blocks = int(ori_kv.shape[0])
        if cmp_kv is not None:
            p.cmp_block_size = int(cmp_kv.shape[1])
            p.cmp_max_blocks = int(cmp_block_table.shape[-1])
            p.cmp_num_blocks = int(cmp_kv.shape[0])
    else:  # the length of the sequence axis: S of [B, S, 1, row], T of [T, 1, row]
        axis = 1 if layout_kv == "BSND" else 0
        p.ori_kv_len = int(ori_kv.shape[axis])
        if cmp_kv is not None:
            p.cmp_kv_len = int(cmp_kv.shape[axis])
    p.k1 = int(ori_sparse_indices.shape[-1]) if ori_sparse_indices is not None else 0
    p.cu_seqlens_ori_kv, p.cu_seqlens_cmp_kv = _dptr(cu_seqlens_ori_kv), _dptr(cu_seqlens_cmp_kv)
    p.ori_sparse_indices, p.ori_topk_length = _dptr(ori_sparse_indices), _dptr(ori_topk_length)
    p.num_ctas = int(num_ctas)
    p.q, p.attn_out = _dptr(q), _dptr(attn_out)
    p.ori_kv, p.ori_scale = _dptr(ori_kv), _dptr(ori_scale)
    p.cmp_kv, p.cmp_scale = _dptr(cmp_kv), _dptr(cmp_scale)
    p.cmp_sparse_indices = _dptr(cmp_sparse_indices)
    p.ori_block_table, p.cmp_block_table = _dptr(ori_block_table), _dptr(cmp_block_table)
    p.cu_seqlens_q, p.seqused_q = _dptr(cu_seqlens_q), _dptr(seqused_q)
    p.seqused_ori_kv, p.seqused_cmp_kv = _dptr(seqused_ori_kv), _dptr(seqused_cmp_kv)
    p.cmp_residual_kv, p.cmp_topk_length = _dptr(cmp_residual_kv), _dptr(cmp_topk_length)
    p.sinks, p.metadata, p.softmax_lse = _dptr(sinks), _dptr(metadata), _dptr(softmax_lse)
    p.softmax_scale = float(softmax_scale)
    p.cmp_ratio = int(cmp_ratio)
    p.ori_mask_mode, p.cmp_mask_mode = int(ori_mask_mode), int(cmp_mask_mode)
    p.ori_win_left, p.ori_win_right = int(ori_win_left), int(ori_win_right)
    p.return_lse = int(bool(return_lse))
    return p


def metadata(params: QsfmParams, metadata_out, stream=None) -> None:
    """qsfm_metadata(): plan the split over CTAs into metadata_out (int32[1024])."""
    _check("qsfm_metadata", lib().qsfm_metadata(ctypes.byref(params), _dptr(metadata_out),
                                                _stream_ptr(stream)))


def workspace_size(params: QsfmParams) -> int:
    n = ctypes.c_size_t(0)
    _check("qsfm_forward_workspace_size",
           lib().qsfm_forward_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return int(n.value)


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _dptr(workspace), workspace.numel() * workspace.element_size()


def forward(params: QsfmParams, workspace=None, stream=None) -> None:
    """qsfm_forward(): attention + combine into params' output pointers."""
    w, n = _ws(workspace)
    _check("qsfm_forward", lib().qsfm_forward(ctypes.byref(params), w, n, _stream_ptr(stream)))


def attention(params: QsfmParams, workspace=None, stream=None) -> None:
    w, n = _ws(workspace)
    _check("qsfm_attention", lib().qsfm_attention(ctypes.byref(params), w, n, _stream_ptr(stream)))


def combine(params: QsfmParams, workspace=None, stream=None) -> None:
    w, n = _ws(workspace)
    _check("qsfm_combine", lib().qsfm_combine(ctypes.byref(params), w, n, _stream_ptr(stream)))


def _header_scratch_bytes() -> int:
    """QSFM_NOALLOC_SCRATCH_BYTES as the C header defines it."""
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qsfm.h")
    m = re.search(r"#define QSFM_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", open(path).read())
    if m is None:
        raise RuntimeError("QSFM_NOALLOC_SCRATCH_BYTES not found in qsfm.h")
    return int(m.group(1)) << int(m.group(2))


NOALLOC_SCRATCH_BYTES = _header_scratch_bytes()


def forward_noalloc(params: QsfmParams, stream=None) -> None:
    """qsfm_forward_noalloc(): the forward pass using the library's fixed
    device scratch array instead of a caller workspace (allocates nothing)."""
    _check("qsfm_forward_noalloc", lib().qsfm_forward_noalloc(ctypes.byref(params), _stream_ptr(stream)))


def debug_gather(params: QsfmParams, tokens, max_rows: int, rows_out, scales_out, row_ids_out,
                 counts_out, stream=None) -> None:
    """qsfm_debug_gather(): the rows the attention kernel resolves per token
    (rows_out = scales_out = None: row ids and counts only, any row format)."""
    _check("qsfm_debug_gather", lib().qsfm_debug_gather(
        ctypes.byref(params), _dptr(tokens), int(tokens.numel()), int(max_rows), _dptr(rows_out),
        _dptr(scales_out), _dptr(row_ids_out), _dptr(counts_out), _stream_ptr(stream)))


def debug_bounded_wait(timeout_ns: int, elapsed_out, stream=None) -> None:
    """qsfm_debug_bounded_wait(): runs out a bounded wait on purpose (sets
    the timeout bit of the fault word; the device stays usable)."""
    _check("qsfm_debug_bounded_wait", lib().qsfm_debug_bounded_wait(
        int(timeout_ns), _dptr(elapsed_out), _stream_ptr(stream)))


def device_status() -> int:
    """Read and clear the device fault word (synchronous)."""
    v = _i32(0)
    code = lib().qsfm_get_device_status(ctypes.byref(v))
    if code not in (0, 5):
        raise QsfmError("qsfm_get_device_status", code)
    return int(v.value)


def status_string(code: int) -> str:
    return lib().qsfm_status_string(int(code)).decode()


def quant_sparse_flash_mla(
    q,
    ori_kv,
    ori_scale,
    ori_block_table,
    seqused_ori_kv,
    *,
    layout: str = "BSND",
    batch: Optional[int] = None,
    cmp_kv=None,
    cmp_scale=None,
    cmp_block_table=None,
    cmp_sparse_indices=None,
    cu_seqlens_q=None,
    seqused_q=None,
    seqused_cmp_kv=None,
    cmp_residual_kv=None,
    cmp_topk_length=None,
    sinks=None,
    softmax_scale: float = HEAD_DIM ** -0.5,
    cmp_ratio: int = 1,
    ori_mask_mode: int = 4,
    cmp_mask_mode: int = 3,
    ori_win_left: int = 127,
    ori_win_right: int = 0,
    return_softmax_lse: bool = False,
    metadata=None,
    workspace=None,
    num_ctas: int = 0,
    out=None,
    stream=None,
    layout_kv: str = "PA_BBND",
    cu_seqlens_ori_kv=None,
    cu_seqlens_cmp_kv=None,
    ori_sparse_indices=None,
    ori_topk_length=None,
):
    """One forward call: plan (unless metadata is given), attention, combine.

    Allocates the outputs (and the plan / workspace when not given) with
    torch on q's device and returns (attn_out, softmax_lse or None). The
    argument names are those of QuantSparseFlashMla's parameter table.
    """
    import torch

    dev = q.device
    attn_out = torch.empty_like(q) if out is None else out
    lse = None
    if return_softmax_lse:
        T = int(q.shape[0] * q.shape[1]) if (layout == "BSND" and q.dim() == 4) else int(q.shape[0])
        lse = torch.empty(T, int(q.shape[-2]), dtype=torch.float32, device=dev)
    plan = metadata if metadata is not None else torch.empty(METADATA_INTS, dtype=torch.int32, device=dev)
    p = make_params(
        q=q, attn_out=attn_out, ori_kv=ori_kv, ori_scale=ori_scale, ori_block_table=ori_block_table,
        seqused_ori_kv=seqused_ori_kv, layout=layout, batch=batch, cmp_kv=cmp_kv,
        cmp_scale=cmp_scale, cmp_block_table=cmp_block_table,
        cmp_sparse_indices=cmp_sparse_indices, cu_seqlens_q=cu_seqlens_q, seqused_q=seqused_q,
        seqused_cmp_kv=seqused_cmp_kv, cmp_residual_kv=cmp_residual_kv,
        cmp_topk_length=cmp_topk_length, sinks=sinks, metadata=plan, softmax_lse=lse,
        softmax_scale=softmax_scale, cmp_ratio=cmp_ratio, ori_mask_mode=ori_mask_mode,
        cmp_mask_mode=cmp_mask_mode, ori_win_left=ori_win_left, ori_win_right=ori_win_right,
        return_lse=return_softmax_lse, num_ctas=num_ctas, layout_kv=layout_kv,
        cu_seqlens_ori_kv=cu_seqlens_ori_kv, cu_seqlens_cmp_kv=cu_seqlens_cmp_kv,
        ori_sparse_indices=ori_sparse_indices, ori_topk_length=ori_topk_length)
    if metadata is None:
        globals()["metadata"](p, plan, stream)
    if workspace is None:
        nbytes = workspace_size(p)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev) if nbytes else None
    forward(p, workspace, stream)
    return attn_out, lse


def sparse_compressed_flash_attention(
    query,
    q_act_seqs,
    ori_kv,
    cmp_kv,
    ori_block_table,
    cmp_block_table,
    atten_sink,
    seqused_kv,
    cmp_sparse_indices,
    softmax_scale: float,
    win_size: int = 128,
    cmp_ratio: int = 4,
    stream=None,
):
    """The bf16-KV entry point with SparseCompressedFlashAttention's argument
    names and shapes (its parameter table; TND only), on the same kernels.

    query [T1 * N1, 512] bf16 (N1 = 64); q_act_seqs int32 [B], the running
    token totals per batch (no leading zero); ori_kv / cmp_kv bf16
    [block_num * 128, 512]; block tables int32 [B, width]; atten_sink fp32
    [N1]; seqused_kv int32 [B]; cmp_sparse_indices int32 [T1, K2].
    The window of win_size tokens ending at the query is band mode 4 with
    ori_win_left = win_size - 1 and ori_win_right = 0; the compressed part
    takes the causal mode 3. Returns attention_out [T1 * N1, 512] bf16.
    Argument marshalling only: views of the given tensors, and cu_seqlens_q
    = [0, q_act_seqs...] (one small device concatenation).
    """
    import torch

    n1 = int(atten_sink.shape[0])
    if query.dim() != 2 or int(query.shape[0]) % n1:
        raise ValueError("query must be [T1 * N1, D] with N1 = atten_sink.shape[0]")
    if win_size < 1:
        raise ValueError("win_size must be >= 1")
    t1 = int(query.shape[0]) // n1
    d = int(query.shape[1])

    def paged(kv):  # [block_num * 128, D] -> [block_num, 128, 1, D] (a view)
        if kv.dim() != 2 or int(kv.shape[0]) % BLOCK_SIZE:
            raise ValueError("ori_kv / cmp_kv must be [block_num * 128, D]")
        return kv.view(int(kv.shape[0]) // BLOCK_SIZE, BLOCK_SIZE, 1, int(kv.shape[1]))

    cu = torch.cat([torch.zeros(1, dtype=q_act_seqs.dtype, device=q_act_seqs.device), q_act_seqs])
    out, _ = quant_sparse_flash_mla(
        query.view(t1, n1, d), paged(ori_kv), None, ori_block_table, seqused_kv,
        layout="TND", cmp_kv=paged(cmp_kv), cmp_block_table=cmp_block_table,
        cmp_sparse_indices=cmp_sparse_indices.view(t1, 1, int(cmp_sparse_indices.shape[-1])),
        cu_seqlens_q=cu, sinks=atten_sink, softmax_scale=float(softmax_scale), cmp_ratio=int(cmp_ratio),
        ori_mask_mode=4, cmp_mask_mode=3, ori_win_left=int(win_size) - 1, ori_win_right=0,
        stream=stream)
    return out.view(t1 * n1, d)


def lightning_indexer(
    query,
    query_scale,
    weights,
    key,
    key_scale,
    block_table,
    seqused_k,
    *,
    layout: str = "BSND",
    batch: Optional[int] = None,
    cu_seqlens_q=None,
    seqused_q=None,
    cmp_residual_k=None,
    topk: int = 2048,
    mask_mode: int = 0,
    cmp_ratio: int = 1,
    return_value: bool = False,
    layout_k: str = "PA_BBND",
    cu_seqlens_k=None,
    output_idx_offset=None,
    out=None,
    values=None,
    workspace=None,
    stream=None,
):
    """QuantLightningIndexerV2's top-k (quant mode 1) through qsfm_lightning_indexer.

    query uint8 e4m3fn bytes BSND [B, S1, g, 128] or TND [T, g, 128];
    query_scale, weights fp32 [T, g]. key uint8 e4m3fn bytes by layout_k:
    "PA_BBND" [blocks, 128, 1, 128] with block_table int32 [B, width] and
    seqused_k int32 [B]; "BSND" [B, Sk, 1, 128] with seqused_k or None;
    "TND" [Tk, 1, 128] with cu_seqlens_k int32 [B + 1] (block_table and
    seqused_k None). key_scale fp32, key's shape without the last axis.
    output_idx_offset int32 [B] or None. Returns (sparse_indices int32 [T, 1, topk],
    sparse_values bf16 [T, 1, topk] or None). workspace: a device uint8
    tensor of at least indexer_workspace_size() bytes, allocated when None.
    Argument marshalling only.
    """
    import torch

    p = IndexerParams()
    lib().qsfm_indexer_params_init(ctypes.byref(p))
    if layout == "BSND":
        p.layout_q = LAYOUT_BSND
        if query.dim() == 4:
            p.batch, p.max_s1 = int(query.shape[0]), int(query.shape[1])
        else:
            if batch is None:
                raise ValueError("flat BSND query needs batch=")
            p.batch = int(batch)
            p.max_s1 = int(query.shape[0]) // max(1, p.batch)
        T = p.batch * p.max_s1
    elif layout == "TND":
        p.layout_q = LAYOUT_TND
        p.total_t = T = int(query.shape[0])
        p.batch = int(cu_seqlens_q.shape[0]) - 1 if cu_seqlens_q is not None else int(batch or 0)
    else:
        raise ValueError(layout)
    p.heads, p.dim = int(query.shape[-2]), int(query.shape[-1])
    p.topk, p.mask_mode, p.cmp_ratio, p.return_value = int(topk), int(mask_mode), int(cmp_ratio), int(bool(return_value))
    p.layout_k = LAYOUT_KV[layout_k]
    if layout_k == "PA_BBND":
        p.block_size, p.num_blocks = int(key.shape[1]), int(key.shape[0])
        p.max_blocks = int(block_table.shape[-1])
    elif layout_k == "BSND":
        p.max_sk = int(key.shape[1])
    else:
        p.total_k = int(key.shape[0])
    dev = query.device
    if out is None:
        out = torch.empty(T, 1, int(topk), dtype=torch.int32, device=dev)
    if return_value and values is None:
        values = torch.empty(T, 1, int(topk), dtype=torch.bfloat16, device=dev)
    p.query, p.query_scale, p.weights = _dptr(query), _dptr(query_scale), _dptr(weights)
    p.key, p.key_scale, p.block_table = _dptr(key), _dptr(key_scale), _dptr(block_table)
    p.seqused_k, p.cmp_residual_k = _dptr(seqused_k), _dptr(cmp_residual_k)
    p.cu_seqlens_q, p.seqused_q = _dptr(cu_seqlens_q), _dptr(seqused_q)
    p.cu_seqlens_k, p.output_idx_offset = _dptr(cu_seqlens_k), _dptr(output_idx_offset)
    p.sparse_indices = _dptr(out)
    p.sparse_values = _dptr(values) if return_value else None
    need = ctypes.c_size_t(0)
    _check("qsfm_lightning_indexer_workspace_size",
           lib().qsfm_lightning_indexer_workspace_size(ctypes.byref(p), ctypes.byref(need)))
    if workspace is None:
        workspace = torch.empty(max(16, need.value), dtype=torch.uint8, device=dev)
    _check("qsfm_lightning_indexer", lib().qsfm_lightning_indexer(
        ctypes.byref(p), _dptr(workspace), workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, (values if return_value else None)
