"""Seeded synthetic inputs for the quantized shared-KV sparse MLA attention.

This module builds inputs only. It holds none of the attention arithmetic:
no masking, no dequantisation, no softmax. The oracle and the CUDA path both
take what it returns. Everything is drawn on the CPU from one
``torch.Generator`` seeded per workload.

Value distributions follow the five workloads of the spec description
(tiny CSA decode, SWA prefill, CSA decode batch, HCA long decode, CSA chunked
prefill):

* q ~ N(0, 1) in bf16.
* KV rows ~ N(0, 1), quantised per 64-element tile to fp8 e4m3fn with
  scale = amax / 448 (KvQuantSparseAttnSharedKv, parameter table rows
  kv_quant_mode / tile_size: per-tile quantisation, tile 64). The fp32 scales
  are stored beside the KV in a [blocks, 128, 1, 8] tensor paged like it.
* sinks ~ N(0, 1) fp32 [64].
* KV lives in 128-token blocks. Each batch takes its blocks from a randomly
  permuted physical pool sized to the exact total, so block tables are
  shuffled.
* KV storage is paged (PA_BBND, the default: 128-token blocks through block
  tables) or, for the non-paged layouts of QuantSparseFlashMla's layout_kv,
  BSND ([B, S2max, 1, row] with each batch's rows from row 0 of its slab)
  or TND ([T2, 1, row] with the batches' rows back to back, located by
  cu_seqlens_ori_kv / cu_seqlens_cmp_kv).
* ori_sparse_indices (when asked for) are drawn distinct and uniform from
  the ori rows inside the token's mask range, valid entries first, -1 after.
* CSA indices are drawn distinct and uniform from the compressed rows a token
  can see. The bound used for drawing is computed here from the
  bottom-right-aligned position; the oracle and the kernel each apply their
  own visibility rule, so a wrong bound here would show up as a mismatch or
  as masked entries, never be hidden.

Large pools (more than ``BANK_ROWS`` rows) are filled from a bank of
``BANK_ROWS`` distinct random rows through a seeded random map. Each row is
still a quantised N(0, 1) row; rows repeat across the pool. The attention
output depends only on the rows a token attends to, so this changes neither
the results' distribution nor the memory traffic of the kernel.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

NUM_HEADS = 64
HEAD_DIM = 512
BLOCK = 128
TILE = 64
SCALES_PER_ROW = HEAD_DIM // TILE
FP8_MAX = 448.0
BANK_ROWS = 1 << 18


@dataclasses.dataclass
class Workload:
    """All inputs of one forward call, as CPU tensors (numpy-convertible)."""

    name: str
    layout: str  # "BSND" or "TND"
    batch: int
    max_s1: int  # BSND: S1; TND: max chunk length
    q_lens: np.ndarray  # int64 [B]: query tokens per batch
    cu_seqlens_q: Optional[torch.Tensor]  # int32 [B+1] (TND)
    q: torch.Tensor  # bf16 [T, N1, 512], N1 = 64 or 128 (BSND memory is identical)
    ori_kv: torch.Tensor  # paged pool [nb, 128, 1, row] (uint8 512 fp8 / 640 packed, or bf16 512); see layout_kv
    ori_scale: Optional[torch.Tensor]  # fp32 [nb, 128, 1, 8]; None for packed and bf16 rows
    ori_block_table: Optional[torch.Tensor]  # int32 [B, wo]; None for non-paged KV
    seqused_ori_kv: Optional[torch.Tensor]  # int32 [B]; None for TND KV (and optionally BSND KV)
    cmp_kv: Optional[torch.Tensor]
    cmp_scale: Optional[torch.Tensor]
    cmp_block_table: Optional[torch.Tensor]
    cmp_sparse_indices: Optional[torch.Tensor]  # int32 [T, 1, K2]
    seqused_cmp_kv: Optional[torch.Tensor]
    cmp_residual_kv: Optional[torch.Tensor]
    cmp_topk_length: Optional[torch.Tensor]
    seqused_q: Optional[torch.Tensor]
    sinks: Optional[torch.Tensor]  # fp32 [64]
    softmax_scale: float
    cmp_ratio: int
    ori_mask_mode: int
    cmp_mask_mode: int
    ori_win_left: int
    ori_win_right: int
    return_lse: bool
    seed: int
    # KV storage: "PA_BBND" (paged, the tensors above are pools and the
    # tables map blocks), "BSND" (ori_kv [B, S2max, 1, row], cmp_kv
    # [B, S3max, 1, row], no tables) or "TND" (ori_kv [T2, 1, row], cmp_kv
    # [T3, 1, row], rows of batch b from cu_seqlens_*_kv[b])
    layout_kv: str = "PA_BBND"
    cu_seqlens_ori_kv: Optional[torch.Tensor] = None  # int32 [B+1] (TND KV)
    cu_seqlens_cmp_kv: Optional[torch.Tensor] = None  # int32 [B+1] (TND KV with cmp_kv)
    ori_sparse_indices: Optional[torch.Tensor] = None  # int32 [T, 1, K1]
    ori_topk_length: Optional[torch.Tensor] = None  # int32 [T]

    @property
    def total_t(self) -> int:
        return int(self.q.shape[0])

    @property
    def n1(self) -> int:
        return int(self.q.shape[1])

    @property
    def k2(self) -> int:
        return 0 if self.cmp_sparse_indices is None else int(self.cmp_sparse_indices.shape[-1])

    @property
    def k1(self) -> int:
        return 0 if self.ori_sparse_indices is None else int(self.ori_sparse_indices.shape[-1])

    @property
    def mode(self) -> str:
        if self.cmp_kv is None:
            return "SWA"
        return "CSA" if self.cmp_sparse_indices is not None else "HCA"

    def token_batch(self) -> np.ndarray:
        """Batch index of every query token (int64 [T])."""
        return np.repeat(np.arange(self.batch), self.q_lens)

    def token_pos(self) -> np.ndarray:
        """Position s of every query token inside its batch's chunk."""
        return np.concatenate([np.arange(n) for n in self.q_lens]) if self.total_t else np.zeros(0, np.int64)


def _quantize_rows(x: torch.Tensor):
    """Quantise fp32 rows [n, 512] per 64-tile to e4m3fn bytes + fp32 scales."""
    n = x.shape[0]
    t = x.view(n, SCALES_PER_ROW, TILE)
    amax = t.abs().amax(dim=-1)
    scale = torch.clamp(amax, min=1e-12) / FP8_MAX
    q8 = (t / scale.unsqueeze(-1)).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8).view(n, HEAD_DIM), scale.to(torch.float32)


PACKED_ROW = 640     # bf16 rope 64 (128 B) + e4m3fn nope 448 + e8m0 scales 7 + pad
ROPE_DIM = 64
NOPE_DIM = HEAD_DIM - ROPE_DIM


def _quantize_packed_rows(x: torch.Tensor):
    """fp32 rows [n, 512] as packed 640-byte rows: the first 64 elements in
    bf16, the other 448 per 64-tile as e4m3fn with a power-of-two scale
    (e8m0: 2^(e - 127)), the smallest that keeps the tile within the e4m3fn
    range."""
    n = x.shape[0]
    rope = x[:, :ROPE_DIM].to(torch.bfloat16)
    t = x[:, ROPE_DIM:].reshape(n, NOPE_DIM // TILE, TILE)
    amax = torch.clamp(t.abs().amax(dim=-1), min=1e-30)
    e = torch.ceil(torch.log2(amax / FP8_MAX)).clamp(-127, 127)
    scale = torch.pow(2.0, e)
    q8 = (t / scale.unsqueeze(-1)).to(torch.float8_e4m3fn)
    out = torch.zeros(n, PACKED_ROW, dtype=torch.uint8)
    out[:, :2 * ROPE_DIM] = rope.view(torch.uint8).view(n, 2 * ROPE_DIM)
    out[:, 2 * ROPE_DIM:2 * ROPE_DIM + NOPE_DIM] = q8.view(torch.uint8).reshape(n, NOPE_DIM)
    out[:, 2 * ROPE_DIM + NOPE_DIM:2 * ROPE_DIM + NOPE_DIM + NOPE_DIM // TILE] = (e + 127).to(torch.uint8)
    return out


def _random_packed_rows(n: int, gen: torch.Generator, chunk: int = 1 << 16):
    rows = torch.empty(n, PACKED_ROW, dtype=torch.uint8)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        rows[lo:hi] = _quantize_packed_rows(torch.randn(hi - lo, HEAD_DIM, generator=gen, dtype=torch.float32))
    return rows


def _random_bf16_rows(n: int, gen: torch.Generator, chunk: int = 1 << 16):
    """Unquantised rows: N(0, 1) draws rounded to bf16."""
    rows = torch.empty(n, HEAD_DIM, dtype=torch.bfloat16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        rows[lo:hi] = torch.randn(hi - lo, HEAD_DIM, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return rows


def _random_rows(n: int, gen: torch.Generator, chunk: int = 1 << 16):
    rows = torch.empty(n, HEAD_DIM, dtype=torch.uint8)
    scales = torch.empty(n, SCALES_PER_ROW, dtype=torch.float32)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        x = torch.randn(hi - lo, HEAD_DIM, generator=gen, dtype=torch.float32)
        r, s = _quantize_rows(x)
        rows[lo:hi] = r
        scales[lo:hi] = s
    return rows, scales


def _paged_pool(lengths: np.ndarray, gen: torch.Generator, min_width: int = 0,
                block: int = BLOCK, fmt: str = "fp8_fp32_scales"):
    """Pool + shuffled block table holding lengths[b] rows for each batch
    (fmt packed640: 640-byte rows, bf16: bf16 rows; neither has a scale
    tensor)."""
    nblk = [(int(l) + block - 1) // block for l in lengths]
    total = sum(nblk)
    width = max([min_width] + nblk + [1])
    perm = torch.randperm(max(total, 1), generator=gen)[:total].to(torch.int32)
    table = torch.full((len(lengths), width), -1, dtype=torch.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[off:off + k]
        off += k
    nrows = max(total, 1) * block
    if fmt in ("packed640", "bf16"):
        make, width_b = (_random_packed_rows, PACKED_ROW) if fmt == "packed640" else (_random_bf16_rows, HEAD_DIM)
        if nrows <= BANK_ROWS:
            rows = make(nrows, gen)
        else:
            bank = make(BANK_ROWS, gen)
            rows = bank[torch.randint(0, BANK_ROWS, (nrows,), generator=gen)]
        return rows.view(max(total, 1), block, 1, width_b), None, table
    if nrows <= BANK_ROWS:
        rows, scales = _random_rows(nrows, gen)
    else:
        bank_r, bank_s = _random_rows(BANK_ROWS, gen)
        pick = torch.randint(0, BANK_ROWS, (nrows,), generator=gen)
        rows, scales = bank_r[pick], bank_s[pick]
    kv = rows.view(max(total, 1), block, 1, HEAD_DIM)
    sc = scales.view(max(total, 1), block, 1, SCALES_PER_ROW)
    return kv, sc, table


def _dense_rows(n: int, gen: torch.Generator, fmt: str):
    """n random rows of a row format: (rows, scales or None); rows are uint8
    [n, 512] (fp8), uint8 [n, 640] (packed) or bf16 [n, 512]."""
    if fmt == "packed640":
        return _random_packed_rows(n, gen), None
    if fmt == "bf16":
        return _random_bf16_rows(n, gen), None
    return _random_rows(n, gen)


def _dense_kv(lengths: np.ndarray, gen: torch.Generator, layout_kv: str, fmt: str, pad: int = 0):
    """Non-paged KV of the given per-batch lengths: BSND [B, max + pad, 1, row]
    (rows past a batch's length are random filler) or TND [sum + pad, 1, row]
    with the prefix sums of the lengths. Returns (kv, scales, cu or None)."""
    B = len(lengths)
    if layout_kv == "BSND":
        s = max([int(l) for l in lengths] + [0]) + pad
        rows, sc = _dense_rows(max(B * s, 1), gen, fmt)
        rows = rows[:B * s].reshape(B, s, 1, rows.shape[-1])
        sc = None if sc is None else sc[:B * s].reshape(B, s, 1, SCALES_PER_ROW)
        return rows, sc, None
    assert layout_kv == "TND"
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.from_numpy(np.cumsum(np.asarray(lengths, dtype=np.int64))).to(torch.int32)
    n = int(cu[-1]) + pad
    rows, sc = _dense_rows(max(n, 1), gen, fmt)
    rows = rows[:max(n, 1)].reshape(max(n, 1), 1, rows.shape[-1])
    sc = None if sc is None else sc[:max(n, 1)].reshape(max(n, 1), 1, SCALES_PER_ROW)
    return rows, sc, cu


def _ori_draw_range(s2: int, s1: int, s: int, mode: int, wl: int, wr: int):
    """Inclusive [lo, hi] of ori rows token s may draw ori indices from (the
    bottom-right-aligned mask range; empty when hi < lo)."""
    p = s2 - s1 + s
    if mode == 0:
        return 0, s2 - 1
    if mode == 3:
        return 0, min(s2 - 1, p)
    lo = 0 if wl == -1 else max(0, p - wl)
    hi = s2 - 1 if wr == -1 else min(s2 - 1, p + wr)
    return lo, hi


def _index_draw_bound(s2: int, s1: int, s: int, cmp_len: int, res: int, r: int) -> int:
    """Number of compressed rows token s may draw indices from (see module doc)."""
    p_c = cmp_len * r + res - s1 + s
    return max(0, min(cmp_len, (p_c + 1) // r))


def build(
    name: str,
    *,
    layout: str,
    q_lens,
    s2,
    cmp_ratio: int = 1,
    mode: str = "SWA",
    k2: int = 512,
    n_valid: Optional[int] = None,
    seed: int = 0,
    ori_mask_mode: int = 4,
    cmp_mask_mode: int = 3,
    ori_win_left: int = 127,
    ori_win_right: int = 0,
    return_lse: bool = False,
    sinks: bool = True,
    with_residual: bool = True,
    softmax_scale: Optional[float] = None,
    cmp_topk_length: Optional[list] = None,
    seqused_q: Optional[list] = None,
    q_scale: float = 1.0,
    block_size: int = BLOCK,
    n1: int = NUM_HEADS,
    kv_format: str = "fp8_fp32_scales",
    layout_kv: str = "PA_BBND",
    kv_pad: int = 0,
    bsnd_seqused: bool = True,
    ori_k1: Optional[int] = None,
    ori_n_valid: Optional[int] = None,
    ori_topk_length: Optional[list] = None,
) -> Workload:
    """Build one workload. q_lens / s2 are per-batch query and ori lengths.

    layout_kv: "PA_BBND" (paged), "BSND" or "TND" (non-paged); kv_pad adds
    filler rows past the last batch's rows (BSND: to every batch's slab);
    bsnd_seqused False leaves seqused_ori_kv / seqused_cmp_kv out for BSND KV
    (the lengths are then the tensors' S dimensions: every batch must fill
    its slab). ori_k1 > 0 adds ori_sparse_indices [T, 1, K1] with up to
    ori_n_valid (default K1) distinct rows of the token's ori mask range,
    -1 after; ori_topk_length [T] optionally cuts each row.
    """
    gen = torch.Generator().manual_seed(seed)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    s2 = np.asarray(s2, dtype=np.int64)
    B = len(q_lens)
    assert len(s2) == B
    T = int(q_lens.sum())
    q = (torch.randn(T, n1, HEAD_DIM, generator=gen) * q_scale).to(torch.bfloat16)
    assert kv_format in ("fp8_fp32_scales", "packed640", "bf16")
    assert layout_kv in ("PA_BBND", "BSND", "TND")
    paged = layout_kv == "PA_BBND"
    cu_ori = cu_cmp = None
    if paged:
        ori_kv, ori_scale, ori_table = _paged_pool(s2, gen, block=block_size, fmt=kv_format)
    else:
        assert layout_kv == layout, "non-paged KV needs layout_kv == layout_q"
        ori_kv, ori_scale, cu_ori = _dense_kv(s2, gen, layout_kv, kv_format, pad=kv_pad)
        ori_table = None
    sink = torch.randn(n1, generator=gen, dtype=torch.float32) if sinks else None
    cu = None
    if layout == "TND":
        cu = torch.zeros(B + 1, dtype=torch.int32)
        cu[1:] = torch.from_numpy(np.cumsum(q_lens)).to(torch.int32)
    else:
        assert len(set(q_lens.tolist())) <= 1, "BSND needs equal S1"
    cmp_kv = cmp_scale = cmp_table = idx = used_cmp = resid = topk = None
    if mode in ("CSA", "HCA"):
        cmp_len = s2 // cmp_ratio
        res = (s2 % cmp_ratio) if with_residual else np.zeros_like(s2)
        cmp_w = (int(s2.max()) // cmp_ratio + block_size - 1) // block_size if B else 1
        if paged:
            cmp_kv, cmp_scale, cmp_table = _paged_pool(cmp_len, gen, min_width=cmp_w,
                                                       block=block_size, fmt=kv_format)
        else:
            cmp_kv, cmp_scale, cu_cmp = _dense_kv(cmp_len, gen, layout_kv, kv_format, pad=kv_pad)
            if layout_kv == "BSND" and bsnd_seqused:
                used_cmp = torch.from_numpy(cmp_len.astype(np.int32))
        resid = torch.from_numpy(res.astype(np.int32))
        if mode == "CSA":
            idx = torch.full((T, 1, k2), -1, dtype=torch.int32)
            t = 0
            for b in range(B):
                for s in range(int(q_lens[b])):
                    v = _index_draw_bound(int(s2[b]), int(q_lens[b]), s, int(cmp_len[b]), int(res[b]), cmp_ratio)
                    n = min(k2 if n_valid is None else n_valid, v)
                    if n > 0:
                        idx[t, 0, :n] = torch.randperm(v, generator=gen)[:n].to(torch.int32)
                    t += 1
        if cmp_topk_length is not None:
            topk = torch.tensor(cmp_topk_length, dtype=torch.int32)
    used_q = torch.tensor(seqused_q, dtype=torch.int32) if seqused_q is not None else None
    ori_idx = ori_topk = None
    if ori_k1:
        ori_idx = torch.full((T, 1, ori_k1), -1, dtype=torch.int32)
        t = 0
        for b in range(B):
            for s in range(int(q_lens[b])):
                lo, hi = _ori_draw_range(int(s2[b]), int(q_lens[b]), s, ori_mask_mode, ori_win_left, ori_win_right)
                v = max(0, hi - lo + 1)
                n = min(ori_k1 if ori_n_valid is None else ori_n_valid, v)
                if n > 0:
                    ori_idx[t, 0, :n] = (torch.randperm(v, generator=gen)[:n] + lo).to(torch.int32)
                t += 1
        if ori_topk_length is not None:
            ori_topk = torch.tensor(ori_topk_length, dtype=torch.int32)
    if layout_kv == "TND":
        used_ori = None  # the lengths come from cu_seqlens_ori_kv
    elif layout_kv == "BSND" and not bsnd_seqused:
        assert len(set(s2.tolist())) <= 1 and kv_pad == 0, "without seqused every batch fills its slab"
        used_ori = None
    else:
        used_ori = torch.from_numpy(s2.astype(np.int32))
    return Workload(
        name=name, layout=layout, batch=B, max_s1=int(q_lens.max()) if B else 0,
        q_lens=q_lens, cu_seqlens_q=cu, q=q,
        ori_kv=ori_kv, ori_scale=ori_scale, ori_block_table=ori_table,
        seqused_ori_kv=used_ori,
        cmp_kv=cmp_kv, cmp_scale=cmp_scale, cmp_block_table=cmp_table,
        cmp_sparse_indices=idx, seqused_cmp_kv=used_cmp, cmp_residual_kv=resid,
        cmp_topk_length=topk, seqused_q=used_q, sinks=sink,
        softmax_scale=(1.0 / math.sqrt(HEAD_DIM)) if softmax_scale is None else softmax_scale,
        cmp_ratio=cmp_ratio if mode != "SWA" else 1,
        ori_mask_mode=ori_mask_mode, cmp_mask_mode=cmp_mask_mode,
        ori_win_left=ori_win_left, ori_win_right=ori_win_right,
        return_lse=return_lse, seed=seed,
        layout_kv=layout_kv, cu_seqlens_ori_kv=cu_ori, cu_seqlens_cmp_kv=cu_cmp,
        ori_sparse_indices=ori_idx, ori_topk_length=ori_topk,
    )


_build = build


def _uniform_int(gen: torch.Generator, lo: int, hi: int, n: int) -> np.ndarray:
    """n integers uniform on the inclusive range [lo, hi]."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).numpy().astype(np.int64)


def config(index: int, seed: Optional[int] = None, kv_format: str = "fp8_fp32_scales",
           n1: int = NUM_HEADS) -> Workload:
    """The five spec workloads; seed defaults to the workload index.

    kv_format / n1 give the same workload with another KV row format or head
    count (the indices, lengths and block tables are drawn the same way; the
    name says what changed)."""
    seed = index if seed is None else seed
    gen = torch.Generator().manual_seed(10_000 + seed)
    extra = dict(kv_format=kv_format, n1=n1)
    tag = ("" if kv_format == "fp8_fp32_scales" else f" kv={kv_format}") + ("" if n1 == NUM_HEADS else f" N1={n1}")

    def build(name, **kw):  # the module-level build with the format / head count applied
        return _build(name + tag, **kw, **extra)

    if index == 0:  # tiny CSA decode
        return build("tiny CSA decode B=2 S1=1 S2=4096 r=4 K2=512 (384 valid)",
                     layout="BSND", q_lens=[1, 1], s2=[4096, 4096], cmp_ratio=4,
                     mode="CSA", k2=512, n_valid=384, seed=seed)
    if index == 1:  # SWA-only prefill
        return build("SWA prefill TND B=4 S1=S2=2048",
                     layout="TND", q_lens=[2048] * 4, s2=[2048] * 4, mode="SWA", seed=seed)
    if index == 2:  # CSA decode batch
        s2 = _uniform_int(gen, 4096, 65536, 128)
        return build("CSA decode batch B=128 S1=2 S2~U[4K,64K] r=4 K2=512",
                     layout="BSND", q_lens=[2] * 128, s2=s2, cmp_ratio=4, mode="CSA",
                     k2=512, seed=seed)
    if index == 3:  # HCA long-context decode
        s2 = _uniform_int(gen, 32768, 131072, 64)
        return build("HCA long decode B=64 S1=1 S2~U[32K,128K] r=128",
                     layout="BSND", q_lens=[1] * 64, s2=s2, cmp_ratio=128, mode="HCA", seed=seed)
    if index == 4:  # CSA chunked prefill
        q_lens = _uniform_int(gen, 512, 4096, 8)
        s2 = _uniform_int(gen, 8192, 32768, 8)
        s2 = np.maximum(s2, q_lens)
        return build("CSA chunked prefill TND B=8 S1~U[512,4096] S2~U[8K,32K] r=4 K2=512 lse",
                     layout="TND", q_lens=q_lens, s2=s2, cmp_ratio=4, mode="CSA",
                     k2=512, seed=seed, return_lse=True)
    raise ValueError(index)


def profile_case(seed: int = 2) -> Workload:
    """The CSA decode batch at profiling size: same B = 128, S1 = 2, K2 = 512
    and per-token work (640 rows) as workload 2, with S2 ~ U[4K, 8K] so the
    KV pools stay under 1 GB on the device."""
    gen = torch.Generator().manual_seed(30_000 + seed)
    s2 = _uniform_int(gen, 4096, 8192, 128)
    return build("CSA decode batch (profiling size) B=128 S1=2 S2~U[4K,8K] r=4 K2=512",
                 layout="BSND", q_lens=[2] * 128, s2=s2, cmp_ratio=4, mode="CSA", k2=512, seed=seed)


def subset_tokens(w: Workload, n: int, seed: int = 0) -> np.ndarray:
    """A seeded sample of n query-token indices of w (sorted)."""
    gen = torch.Generator().manual_seed(20_000 + seed)
    n = min(n, w.total_t)
    return np.sort(torch.randperm(w.total_t, generator=gen)[:n].numpy())


def device_inputs(w: Workload, device) -> dict:
    """The workload's tensors on `device`, keyed by the op's argument names.

    Pure data movement (no arithmetic): uint8 fp8 bytes, bf16 rows, fp32 scales, int32
    tables / lengths / indices and the bf16 query are copied as they are.
    """
    def mv(t):
        return None if t is None else t.contiguous().to(device)

    return dict(
        q=mv(w.q), ori_kv=mv(w.ori_kv), ori_scale=mv(w.ori_scale),
        ori_block_table=mv(w.ori_block_table), seqused_ori_kv=mv(w.seqused_ori_kv),
        layout=w.layout, batch=w.batch, cmp_kv=mv(w.cmp_kv), cmp_scale=mv(w.cmp_scale),
        cmp_block_table=mv(w.cmp_block_table), cmp_sparse_indices=mv(w.cmp_sparse_indices),
        cu_seqlens_q=mv(w.cu_seqlens_q), seqused_q=mv(w.seqused_q),
        seqused_cmp_kv=mv(w.seqused_cmp_kv), cmp_residual_kv=mv(w.cmp_residual_kv),
        cmp_topk_length=mv(w.cmp_topk_length), sinks=mv(w.sinks),
        softmax_scale=w.softmax_scale, cmp_ratio=w.cmp_ratio, ori_mask_mode=w.ori_mask_mode,
        cmp_mask_mode=w.cmp_mask_mode, ori_win_left=w.ori_win_left,
        ori_win_right=w.ori_win_right, return_softmax_lse=w.return_lse,
        layout_kv=w.layout_kv, cu_seqlens_ori_kv=mv(w.cu_seqlens_ori_kv),
        cu_seqlens_cmp_kv=mv(w.cu_seqlens_cmp_kv), ori_sparse_indices=mv(w.ori_sparse_indices),
        ori_topk_length=mv(w.ori_topk_length),
    )


# --------------------------------------------------------------------------
# Inputs of the lightning-indexer top-k (QuantLightningIndexerV2, quant
# mode 1): e4m3fn index queries and keys with fp32 dequant scales, fp32
# head weights. Rows ~ N(0, 1) quantised with scale = amax / 448 (one scale
# per query head of a token, one per key row); weights ~ N(0, 1). Keys are
# paged in 128-row blocks through a shuffled block table.
# --------------------------------------------------------------------------
@dataclasses.dataclass
class IndexerWorkload:
    name: str
    layout: str  # "BSND" or "TND"
    batch: int
    q_lens: np.ndarray  # int64 [B]
    cu_seqlens_q: Optional[torch.Tensor]  # int32 [B+1] (TND)
    query: torch.Tensor  # uint8 e4m3fn bytes [T, g, d]
    query_scale: torch.Tensor  # fp32 [T, g]
    weights: torch.Tensor  # fp32 [T, g]
    key: torch.Tensor  # uint8 e4m3fn bytes: PA_BBND [blocks, 128, 1, d], BSND [B, Sk, 1, d], TND [Tk, 1, d]
    key_scale: torch.Tensor  # fp32, the key's shape without d
    block_table: Optional[torch.Tensor]  # int32 [B, width] (PA_BBND)
    seqused_k: Optional[torch.Tensor]  # int32 [B] (PA_BBND; BSND, default Sk; None for TND)
    cmp_residual_k: Optional[torch.Tensor]  # int32 [B]
    seqused_q: Optional[torch.Tensor]  # int32 [B]
    topk: int
    mask_mode: int
    cmp_ratio: int
    seed: int
    layout_k: str = "PA_BBND"  # "PA_BBND", "BSND" or "TND"
    cu_seqlens_k: Optional[torch.Tensor] = None  # int32 [B+1] (TND keys)
    output_idx_offset: Optional[torch.Tensor] = None  # int32 [B]

    @property
    def total_t(self) -> int:
        return int(self.query.shape[0])

    @property
    def heads(self) -> int:
        return int(self.query.shape[1])

    def key_len(self, b: int) -> int:
        """Keys of batch b (a length, not a rule of the method)."""
        if self.layout_k == "TND":
            return int(self.cu_seqlens_k[b + 1] - self.cu_seqlens_k[b])
        if self.seqused_k is None:
            return int(self.key.shape[1])
        return int(self.seqused_k[b])

    def token_batch(self) -> np.ndarray:
        return np.repeat(np.arange(self.batch), self.q_lens)

    def token_pos(self) -> np.ndarray:
        return np.concatenate([np.arange(n) for n in self.q_lens]) if self.total_t else np.zeros(0, np.int64)


def _quantize_rows_e4m3(x: torch.Tensor):
    """Rows of x as e4m3fn bytes with one fp32 scale per row (amax / 448)."""
    amax = x.abs().amax(dim=-1, keepdim=True).clamp(min=1e-12)
    scale = amax / FP8_MAX
    q = (x / scale).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale.squeeze(-1).to(torch.float32)


def build_indexer(name: str, *, layout: str, q_lens, sk, heads: int = 64, dim: int = 128, topk: int = 512,
                  mask_mode: int = 3, cmp_ratio: int = 4, with_residual: bool = True,
                  seqused_q: Optional[list] = None, residual=None, layout_k: str = "PA_BBND",
                  bsnd_seqused: bool = True, output_idx_offset=None, seed: int = 0) -> IndexerWorkload:
    """One indexer call: q_lens query tokens and sk keys per batch. The
    logical keys of a batch are drawn the same way for every layout_k and
    then stored paged (random block permutation), as BSND slabs [B, max sk]
    (with seqused_k, or without when bsnd_seqused is False and every batch
    fills its slab) or as TND rows with cu_seqlens_k."""
    gen = torch.Generator().manual_seed(seed)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    sk = np.asarray(sk, dtype=np.int64)
    B, T = len(q_lens), int(q_lens.sum())
    qx = torch.randn(T, heads, dim, generator=gen)
    query, qscale = _quantize_rows_e4m3(qx)
    weights = torch.randn(T, heads, generator=gen, dtype=torch.float32)
    nblk = [(int(l) + BLOCK - 1) // BLOCK for l in sk]
    total = max(sum(nblk), 1)
    perm = torch.randperm(total, generator=gen)[:sum(nblk)].to(torch.int32)
    width = max(nblk + [1])
    table = torch.full((B, width), -1, dtype=torch.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[off:off + k]
        off += k
    kx = torch.randn(total * BLOCK, dim, generator=gen)
    key, kscale = _quantize_rows_e4m3(kx)
    cu = None
    if layout == "TND":
        cu = torch.zeros(B + 1, dtype=torch.int32)
        cu[1:] = torch.from_numpy(np.cumsum(q_lens)).to(torch.int32)
    else:
        assert len(set(q_lens.tolist())) <= 1, "BSND needs equal S1"
    res = None
    if residual is not None:
        res = torch.as_tensor(np.asarray(residual), dtype=torch.int32).clone()
    elif with_residual and mask_mode == 3:
        res = torch.from_numpy((torch.randint(0, cmp_ratio, (B,), generator=gen)).numpy().astype(np.int32))
    key = key.view(total, BLOCK, 1, dim)
    kscale = kscale.view(total, BLOCK, 1)
    used_k = torch.from_numpy(sk.astype(np.int32))
    cu_k = None
    if layout_k != "PA_BBND":
        # batch b's logical key j is the paged pool's row table[b, j // 128], j % 128
        rows = [[(int(table[b, j // BLOCK]), j % BLOCK) for j in range(int(sk[b]))] for b in range(B)]
        if layout_k == "BSND":
            width = int(sk.max()) if B else 0
            k2 = torch.zeros(B, width, 1, dim, dtype=torch.uint8)
            s2 = torch.zeros(B, width, 1, dtype=torch.float32)
            for b in range(B):
                for j, (blk, off) in enumerate(rows[b]):
                    k2[b, j] = key[blk, off]
                    s2[b, j] = kscale[blk, off]
            if not bsnd_seqused:
                assert len(set(sk.tolist())) <= 1, "without seqused_k every batch fills its slab"
                used_k = None
        else:
            flat = [r for rb in rows for r in rb]
            k2 = torch.zeros(len(flat), 1, dim, dtype=torch.uint8)
            s2 = torch.zeros(len(flat), 1, dtype=torch.float32)
            for i, (blk, off) in enumerate(flat):
                k2[i] = key[blk, off]
                s2[i] = kscale[blk, off]
            cu_k = torch.zeros(B + 1, dtype=torch.int32)
            cu_k[1:] = torch.from_numpy(np.cumsum(sk)).to(torch.int32)
            used_k = None
        key, kscale, table = k2, s2, None
    offs = None if output_idx_offset is None else torch.as_tensor(np.asarray(output_idx_offset), dtype=torch.int32)
    return IndexerWorkload(
        name=name, layout=layout, batch=B, q_lens=q_lens, cu_seqlens_q=cu, query=query, query_scale=qscale,
        weights=weights, key=key, key_scale=kscale, layout_k=layout_k, cu_seqlens_k=cu_k, output_idx_offset=offs,
        block_table=table, seqused_k=used_k, cmp_residual_k=res,
        seqused_q=torch.tensor(seqused_q, dtype=torch.int32) if seqused_q is not None else None,
        topk=topk, mask_mode=mask_mode, cmp_ratio=cmp_ratio, seed=seed)


def indexer_for(w: "Workload", seed: int = 0, heads: int = 64) -> IndexerWorkload:
    """The indexer call that produces a CSA workload's index rows: the same
    batches, query chunks, layout and padded query rows; one index key per
    compressed row of the workload (seqused_k = its compressed length, the
    generator's own s2 // cmp_ratio when the workload leaves it implicit),
    paged in a pool of its own; the same residual, ratio and causal mask 3;
    topk = the index row width K2. Its rows can be passed as the workload's
    cmp_sparse_indices."""
    if w.seqused_cmp_kv is not None:
        sk = np.asarray(w.seqused_cmp_kv, dtype=np.int64)
    else:
        sk = np.asarray(w.seqused_ori_kv, dtype=np.int64) // w.cmp_ratio
    res = (np.asarray(w.cmp_residual_kv, dtype=np.int64) if w.cmp_residual_kv is not None
           else np.zeros(w.batch, dtype=np.int64))
    used_q = None if w.seqused_q is None else np.asarray(w.seqused_q).tolist()
    return build_indexer(f"indexer for {w.name}", layout=w.layout, q_lens=w.q_lens, sk=sk, heads=heads,
                         topk=w.k2, mask_mode=3, cmp_ratio=w.cmp_ratio, seqused_q=used_q, residual=res,
                         seed=seed)


def indexer_decode_batch(seed: int = 2) -> IndexerWorkload:
    """The indexer call that feeds the CSA decode batch: B = 128, S1 = 2,
    64 index heads of 128, compressed keys S2 / 4 with S2 ~ U[4K, 64K],
    top-512 under the causal mask."""
    gen = torch.Generator().manual_seed(10_000 + seed)
    s2 = _uniform_int(gen, 4096, 65536, 128)
    return build_indexer("indexer for the CSA decode batch B=128 S1=2 Sk=S2/4 g=64 d=128 top-512",
                         layout="BSND", q_lens=[2] * 128, sk=s2 // 4, topk=512, mask_mode=3,
                         cmp_ratio=4, seed=seed)


def indexer_device_inputs(w: IndexerWorkload, device) -> dict:
    """The indexer workload's tensors on `device` (data movement only)."""
    def mv(t):
        return None if t is None else t.contiguous().to(device)

    return dict(query=mv(w.query), query_scale=mv(w.query_scale), weights=mv(w.weights), key=mv(w.key),
                key_scale=mv(w.key_scale), block_table=mv(w.block_table), seqused_k=mv(w.seqused_k),
                cmp_residual_k=mv(w.cmp_residual_k), seqused_q=mv(w.seqused_q), cu_seqlens_q=mv(w.cu_seqlens_q),
                cu_seqlens_k=mv(w.cu_seqlens_k), output_idx_offset=mv(w.output_idx_offset), layout_k=w.layout_k,
                layout=w.layout, batch=w.batch, topk=w.topk, mask_mode=w.mask_mode, cmp_ratio=w.cmp_ratio)
