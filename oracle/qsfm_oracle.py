"""fp64 CPU oracle of the quantized shared-KV sparse MLA attention forward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module. The product path (the CUDA library and its Python binding)
never calls it, and it shares no code with that path.

It evaluates, token by token and straight from the definitions,

    O = softmax([Q K~^T * softmax_scale, sink]) V~,   K~ = V~

over the rows each query token attends to. Every step is written in float64
with numpy; the one library primitive is a matrix product.

Sources (page title, section):
  * QuantSparseFlashMla, "功能说明" (function description): the three modes
    SWA / CSA / HCA and the formula O = softmax(Q K~^T softmax_scale) V~ with
    K~ = V~ made of the ori window part and the cmp part.
  * QuantSparseFlashMla, "参数说明" (parameter table): cmp_sparse_indices
    (-1 = invalid), seqused_*, cmp_residual_kv, cmp_topk_length, sinks,
    cmp_ratio, ori/cmp_mask_mode (0 none, 3 RightDownCausal, 4 band),
    ori_win_left/right (-1 = unbounded).
  * QuantSparseFlashMla, "约束说明" (constraints): PageAttention layout, the
    cmp length default and cmp_len * cmp_ratio + residual.
  * SparseCompressedFlashAttention, parameter table: the same attention over
    unquantised bf16 KV rows.
  * KvQuantSparseAttnSharedKv, parameter table: fp8 e4m3fn KV with per-tile
    quantisation (tile 64), softmax_lse definition; its constraints: indices
    valid-first, -1 after.
  * torch_npu.npu_fused_infer_attention_score, "参数说明" (sparse_mode 3 and
    4), "输出说明" (softmaxLse), "约束说明" (an empty KV gives a zero output).

Readings where the pages are silent or ambiguous (each is also listed in the
design notes of the repository):
  R1 query positions are aligned bottom-right: p = S2 - S1_b + s (ori) and
     p_c = cmp_len * cmp_ratio + residual - S1_b + s (cmp);
  R2 band bounds are inclusive: rows max(0, p - wl) .. min(S2 - 1, p + wr);
  R3 compressed row c covers original tokens c*r .. c*r + r - 1 and is
     visible under mask mode 3 when that whole range is <= p_c, i.e.
     c < floor((p_c + 1) / r), clipped to [0, cmp_len];
  R4 an index names a logical compressed row of the token's own batch,
     resolved through cmp_block_table; entries that are -1 or outside the
     visible range are dropped; duplicates count once per occurrence;
  R5 the sink is a logit of its own in the softmax denominator, not scaled
     by softmax_scale and with no value vector;
  R6 lse = log sum_j exp(x_j) over attended rows, the sink excluded;
  R7 a token with no attended row (or a padded query row) gets O = 0 and
     lse = -inf, even when a sink is given;
  R16 ori_sparse_indices (QuantSparseFlashMla parameter table: discrete
     picks from ori_kv, -1 = invalid; ori_topk_length: how many entries
     take part) replace the contiguous ori range: the token's ori rows are
     the entries of its index row (the first ori_topk_length of them when
     given) that are not -1 and lie inside its ori mask range (R1, R2),
     each occurrence counted, in index order;
  R17 non-paged KV (QuantSparseFlashMla constraints on layout_kv): BSND
     ori_kv [B, S2, 1, D] holds batch b's row j at [b, j]; TND ori_kv
     [T2, 1, D] holds it at cu_seqlens_ori_kv[b] + j (cmp_kv alike with
     cu_seqlens_cmp_kv). The ori length S2_b is seqused_ori_kv[b] (BSND;
     the tensor's S dimension when absent) or cu[b + 1] - cu[b] (TND); the
     cmp length is seqused_cmp_kv[b] when given, else the tensor's S
     dimension (BSND) or the cu_seqlens_cmp_kv difference (TND), and
     floor(S2 / cmp_ratio) for paged KV as before.
"""

from __future__ import annotations

import math

import numpy as np

NUM_HEADS = 64
HEAD_DIM = 512
TILE = 64


# --------------------------------------------------------------------------
# fp8 e4m3fn decoding (KvQuantSparseAttnSharedKv, parameter table rows
# ori_kv / cmp_kv: FLOAT8_E4M3FN). Format: 1 sign bit, 4 exponent bits with
# bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); the only
# non-finite codes are S.1111.111 (NaN); there is no infinity.
# --------------------------------------------------------------------------
def decode_e4m3fn_code(code: int) -> float:
    """Value of one e4m3fn byte, from the bit fields."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3FN_TABLE = np.array([decode_e4m3fn_code(c) for c in range(256)], dtype=np.float64)


def decode_e8m0_code(code: int) -> float:
    """Value of one e8m0 (float8_e8m0fnu) byte: 2^(code - 127); 0xFF is NaN."""
    return math.nan if code == 0xFF else 2.0 ** (code - 127)


E8M0_TABLE = np.array([decode_e8m0_code(c) for c in range(256)], dtype=np.float64)
ROPE_DIM = 64
PACKED_ROW = 640


def dequant_packed_rows(rows: np.ndarray) -> np.ndarray:
    """K~ of packed 640-byte rows [n, 640] -> fp64 [n, 512], exactly.

    KvQuantSparseAttnSharedKv constraints: a row is kv_rope (64 bf16,
    bytes 0..127), kv_nope (448 e4m3fn, bytes 128..575) and the nope scales
    (7 e8m0, bytes 576..582, one per 64 nope elements), padded to 640 bytes.
    The 512 elements are rope then nope (R12).
    """
    rows = np.ascontiguousarray(rows)
    n = rows.shape[0]
    bits = rows[:, :2 * ROPE_DIM].copy().view("<u2").astype(np.uint32) << 16
    rope = bits.view(np.float32).astype(np.float64)
    nope_end = 2 * ROPE_DIM + (HEAD_DIM - ROPE_DIM)
    nope = E4M3FN_TABLE[rows[:, 2 * ROPE_DIM:nope_end].astype(np.int64)]
    scales = E8M0_TABLE[rows[:, nope_end:nope_end + (HEAD_DIM - ROPE_DIM) // TILE].astype(np.int64)]
    return np.concatenate([rope, nope * np.repeat(scales, TILE, axis=1)], axis=1).reshape(n, HEAD_DIM)


BF16_ROW = 2 * HEAD_DIM


def decode_bf16_rows(rows: np.ndarray) -> np.ndarray:
    """K~ of unquantised bf16 rows given as little-endian bytes [n, 1024] ->
    fp64 [n, 512], exactly.

    SparseCompressedFlashAttention, parameter table rows ori_kv / cmp_kv:
    bf16 [block_num, block_size, 1, 512]. A bf16 value is the top half of
    the fp32 with the same sign, exponent and leading mantissa bits, so its
    16 bits shifted up by 16 are that fp32 exactly.
    """
    rows = np.ascontiguousarray(rows)
    bits = rows.view("<u2").astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64).reshape(rows.shape[0], HEAD_DIM)


def dequant_rows(kv_bytes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """K~[j, d] = e4m3fn(kv[j, d]) * scale[j, d // 64], exactly, in fp64.

    kv_bytes uint8 [n, 512], scales fp32 [n, 8] -> fp64 [n, 512].
    """
    vals = E4M3FN_TABLE[kv_bytes.astype(np.int64)]
    per_col = np.repeat(scales.astype(np.float64), TILE, axis=1)
    return vals * per_col


# --------------------------------------------------------------------------
# Row sets (QuantSparseFlashMla parameter table rows ori_mask_mode,
# cmp_mask_mode, ori_win_left/right, cmp_residual_kv; its constraints on
# seqused_cmp_kv and cmp_len * cmp_ratio + residual).
# --------------------------------------------------------------------------
def ori_row_range(p: int, s2: int, mode: int, wl: int, wr: int):
    """Inclusive [lo, hi] of ori rows a query at position p attends (R1, R2).

    Returns (0, -1) for an empty set.
    """
    if mode == 0:
        lo, hi = 0, s2 - 1
    elif mode == 3:
        lo, hi = 0, min(s2 - 1, p)
    elif mode == 4:
        lo = 0 if wl == -1 else max(0, p - wl)
        hi = s2 - 1 if wr == -1 else min(s2 - 1, p + wr)
    else:
        raise ValueError(f"ori_mask_mode {mode}")
    if hi < lo:
        return 0, -1
    return lo, hi


def cmp_visible_count(p_c: int, cmp_len: int, ratio: int, mode: int) -> int:
    """Number V of leading compressed rows visible at cmp position p_c (R3)."""
    if mode == 0:
        return cmp_len
    if mode == 3:
        return max(0, min(cmp_len, (p_c + 1) // ratio))
    raise ValueError(f"cmp_mask_mode {mode}")


def kv_layout_of(w) -> str:
    return getattr(w, "layout_kv", "PA_BBND")


def ori_length(w, b: int) -> int:
    """S2 of batch b (R17)."""
    lay = kv_layout_of(w)
    if lay == "TND":
        cu = w.cu_seqlens_ori_kv
        return int(cu[b + 1]) - int(cu[b])
    if w.seqused_ori_kv is not None:
        return int(w.seqused_ori_kv[b])
    if lay == "BSND":
        return int(w.ori_kv.shape[1])
    raise ValueError("paged KV needs seqused_ori_kv")


def cmp_length(w, b: int, s2: int) -> int:
    """Compressed length of batch b (QuantSparseFlashMla constraints on
    seqused_cmp_kv; R17)."""
    if w.seqused_cmp_kv is not None:
        return int(w.seqused_cmp_kv[b])
    lay = kv_layout_of(w)
    if lay == "BSND":
        return int(w.cmp_kv.shape[1])
    if lay == "TND":
        cu = w.cu_seqlens_cmp_kv
        return int(cu[b + 1]) - int(cu[b])
    return s2 // int(w.cmp_ratio)


def ori_picks(w, t: int, lo: int, hi: int) -> list:
    """ori rows of token t picked by ori_sparse_indices (R16): the entries
    of its index row (the first ori_topk_length[t] when given) that are not
    -1 and lie in the mask range [lo, hi], in index order, repeats kept."""
    idx = w.ori_sparse_indices
    n = int(idx.shape[-1])
    if w.ori_topk_length is not None:
        n = min(n, int(w.ori_topk_length[t]))
    return [int(e) for e in np.asarray(idx[t, 0, :max(n, 0)]).tolist() if e != -1 and lo <= e <= hi]


def token_rows(w, t: int, b: int, s: int):
    """Attended rows of query token t (batch b, position s in the chunk).

    Returns (ori_rows, cmp_rows) as lists of logical row indices; either may
    be empty. For a padded query row both are None.
    """
    s1_b = int(w.q_lens[b])
    if w.seqused_q is not None and s >= int(w.seqused_q[b]):
        return None, None
    s2 = ori_length(w, b)
    p = s2 - s1_b + s
    lo, hi = ori_row_range(p, s2, w.ori_mask_mode, w.ori_win_left, w.ori_win_right)
    if getattr(w, "ori_sparse_indices", None) is None:
        ori = list(range(lo, hi + 1))
    else:
        ori = ori_picks(w, t, lo, hi)
    cmp_rows: list = []
    if w.cmp_kv is not None:
        r = int(w.cmp_ratio)
        cmp_len = cmp_length(w, b, s2)
        res = int(w.cmp_residual_kv[b]) if w.cmp_residual_kv is not None else 0
        p_c = cmp_len * r + res - s1_b + s
        v = cmp_visible_count(p_c, cmp_len, r, w.cmp_mask_mode)
        if w.cmp_sparse_indices is None:  # HCA: a contiguous segment
            cmp_rows = list(range(v))
        else:  # CSA: valid top-k entries (R4)
            n = int(w.cmp_sparse_indices.shape[-1])
            if w.cmp_topk_length is not None:
                n = min(n, int(w.cmp_topk_length[t]))
            for e in np.asarray(w.cmp_sparse_indices[t, 0, :n]).tolist():
                if e != -1 and 0 <= e < v:
                    cmp_rows.append(int(e))
    return ori, cmp_rows


def gather_paged(kv_pool, scale_pool, table_row, rows):
    """Bytes and scales of logical rows through one batch's block table.

    (QuantSparseFlashMla constraints, PageAttention: kv is
    [block_num, block_size, KV_N, D] and the table maps a batch's logical
    block to a physical block.)
    """
    bs = kv_pool.shape[1]
    n = len(rows)
    out_b = np.zeros((n, kv_pool.shape[-1]), dtype=np.uint8)
    out_s = None if scale_pool is None else np.zeros((n, HEAD_DIM // TILE), dtype=np.float32)
    for i, j in enumerate(rows):
        blk = int(table_row[j // bs])
        out_b[i] = kv_pool[blk, j % bs, 0]
        if out_s is not None:
            out_s[i] = scale_pool[blk, j % bs, 0]
    return out_b, out_s


def decode_rows(kv_bytes: np.ndarray, scales) -> np.ndarray:
    """K~ of gathered rows: packed 640-byte rows carry their scales, bf16
    rows (1024 bytes) need none; 512-byte fp8 rows come with a separate fp32
    scale row."""
    if kv_bytes.shape[-1] == PACKED_ROW:
        return dequant_packed_rows(kv_bytes)
    if kv_bytes.shape[-1] == BF16_ROW:
        return decode_bf16_rows(kv_bytes)
    return dequant_rows(kv_bytes, scales)


# --------------------------------------------------------------------------
# Attention of one token (QuantSparseFlashMla function description formula;
# sink per its parameter table row "sinks"; lse per
# KvQuantSparseAttnSharedKv parameter table row softmax_lse).
# --------------------------------------------------------------------------
def attend(q: np.ndarray, k: np.ndarray, softmax_scale: float, sinks):
    """O[N1, 512] and lse[N1] of one token over its rows k [n, 512] (fp64).

    x = softmax_scale * q k^T; m = max(max_j x_j, sink_h);
    O = sum_j e^{x_j - m} k_j / (sum_j e^{x_j - m} + e^{sink_h - m});
    lse = log sum_j e^{x_j} (sink excluded).  (R5, R6, R7)
    """
    nh = q.shape[0]
    if k.shape[0] == 0:
        return np.zeros((nh, HEAD_DIM)), np.full(nh, -np.inf)
    x = softmax_scale * (q @ k.T)  # [64, n]
    sink = np.full(nh, -np.inf) if sinks is None else np.asarray(sinks, dtype=np.float64)
    xmax = x.max(axis=1)
    m = np.maximum(xmax, sink)
    e = np.exp(x - m[:, None])
    den = e.sum(axis=1) + np.exp(sink - m)
    o = (e @ k) / den[:, None]
    lse = xmax + np.log(np.exp(x - xmax[:, None]).sum(axis=1))
    return o, lse


def pool_bytes(pool) -> np.ndarray:
    """A KV pool as a byte array [blocks, block_size, 1, row bytes] (bf16
    rows are taken as their 1024 little-endian bytes)."""
    if str(getattr(pool, "dtype", "")) == "torch.bfloat16":
        import torch  # the workload's tensors are torch tensors; numpy has no bf16

        pool = pool.contiguous().view(torch.uint8)  # last dim 512 -> 1024 bytes
    return np.asarray(pool)


def gather_dense(kv, scales, w, b: int, rows, cu):
    """Bytes and scales of logical rows of batch b in non-paged KV (R17):
    BSND kv [B, S, 1, row] at [b, j]; TND kv [T, 1, row] at cu[b] + j."""
    kv = pool_bytes(kv)
    sc = None if scales is None else np.asarray(scales)
    idx = np.asarray(rows, dtype=np.int64)
    if kv_layout_of(w) == "BSND":
        out_b = kv[b, idx, 0]
        out_s = None if sc is None else sc[b, idx, 0]
    else:
        flat = int(cu[b]) + idx
        out_b = kv[flat, 0]
        out_s = None if sc is None else sc[flat, 0]
    out_b = np.asarray(out_b).reshape(len(idx), kv.shape[-1])
    return out_b, None if out_s is None else np.asarray(out_s).reshape(len(idx), sc.shape[-1])


def token_kv(w, t: int, b: int, s: int):
    """Dequantised K~ = V~ rows [n, 512] of token t: ori rows, then cmp rows."""
    ori, cmp_rows = token_rows(w, t, b, s)
    if ori is None:
        return None
    parts = []
    paged = kv_layout_of(w) == "PA_BBND"
    if paged:
        ob, os_ = gather_paged(pool_bytes(w.ori_kv), None if w.ori_scale is None else np.asarray(w.ori_scale),
                               np.asarray(w.ori_block_table[b]), ori)
    else:
        ob, os_ = gather_dense(w.ori_kv, w.ori_scale, w, b, ori, w.cu_seqlens_ori_kv)
    parts.append(decode_rows(ob, os_))
    if cmp_rows:
        if paged:
            cb, cs = gather_paged(pool_bytes(w.cmp_kv), None if w.cmp_scale is None else np.asarray(w.cmp_scale),
                                  np.asarray(w.cmp_block_table[b]), cmp_rows)
        else:
            cb, cs = gather_dense(w.cmp_kv, w.cmp_scale, w, b, cmp_rows, w.cu_seqlens_cmp_kv)
        parts.append(decode_rows(cb, cs))
    return np.concatenate(parts, axis=0)


def q_fp64(w, t: int) -> np.ndarray:
    """Query of token t as fp64 [N1, 512] (bf16 -> fp32 -> fp64 is exact)."""
    return w.q[t].float().numpy().astype(np.float64)


def reference(w, tokens=None):
    """O (fp64 [n, N1, 512]) and lse (fp64 [n, N1]) for the given tokens.

    tokens: iterable of query-token indices; default all tokens.
    """
    tokens = range(w.total_t) if tokens is None else tokens
    tokens = list(tokens)
    tb, tp = w.token_batch(), w.token_pos()
    nh = int(w.q.shape[1])  # N1: 64 or 128
    out = np.zeros((len(tokens), nh, HEAD_DIM))
    lse = np.full((len(tokens), nh), -np.inf)
    sinks = None if w.sinks is None else np.asarray(w.sinks, dtype=np.float64)
    for i, t in enumerate(tokens):
        k = token_kv(w, t, int(tb[t]), int(tp[t]))
        if k is None:  # padded query row (R7)
            continue
        out[i], lse[i] = attend(q_fp64(w, t), k, float(w.softmax_scale), sinks)
    return out, lse


def logits(w, t: int) -> np.ndarray:
    """softmax_scale * Q K~^T of token t, fp64 [64, n] (for the lse pin)."""
    k = token_kv(w, t, int(w.token_batch()[t]), int(w.token_pos()[t]))
    return float(w.softmax_scale) * (q_fp64(w, t) @ k.T)


_FORK_WORKLOAD = None


def _worker_init():
    # a forked worker must not enter the parent's OpenMP pool
    import sys

    if "torch" in sys.modules:
        sys.modules["torch"].set_num_threads(1)


def _reference_chunk(tokens):
    return reference(_FORK_WORKLOAD, tokens)


def reference_parallel(w, tokens, processes: int):
    """reference() split over a pool of `processes` forked workers.

    The workers inherit w through fork (no copy of the KV pools). A process
    forked after CUDA is initialised can hang, so once the calling process
    has initialised CUDA this runs serially instead.
    """
    import multiprocessing as mp
    import sys

    global _FORK_WORKLOAD
    tokens = list(tokens)
    torch_mod = sys.modules.get("torch")
    cuda_up = torch_mod is not None and torch_mod.cuda.is_initialized()
    if processes <= 1 or len(tokens) < 2 or cuda_up:
        return reference(w, tokens)
    chunks = [tokens[i::processes] for i in range(processes)]
    _FORK_WORKLOAD = w
    try:
        with mp.get_context("fork").Pool(processes, initializer=_worker_init) as pool:
            res = pool.map(_reference_chunk, chunks)
    finally:
        _FORK_WORKLOAD = None
    nh = int(w.q.shape[1])
    out = np.zeros((len(tokens), nh, HEAD_DIM))
    lse = np.zeros((len(tokens), nh))
    for i, (o, l) in enumerate(res):
        out[i::processes] = o
        lse[i::processes] = l
    return out, lse
