"""fp64 CPU oracle of the lightning-indexer top-k (QuantLightningIndexerV2).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` may import or run this module. The product path
never calls it and shares no code with it.

It evaluates, query token by query token and straight from the formula of
QuantLightningIndexerV2 ("功能说明", 计算公式 and the three steps under it),

    score_j = sum_h W[h] * ReLU( Sq[h] * Sk[j] * (Q[h, :] . K[j, :]) )
    out     = the top-k keys j by score

with Q = the token's index query (g heads x d, FLOAT8_e4m3fn, decoded
exactly), K = the batch's compressed index keys (S_k x d, FLOAT8_e4m3fn),
Sq = query_dequant_scale (one fp32 per head of the token, the shape of
weights), Sk = key_dequant_scale (one fp32 per key row), W = weights (fp32
per head). Every step is written in float64 with numpy; the one library
primitive is a matrix product.

Readings where the page is silent (each is also listed in the design
notes of the repository):
  I1 quant_mode 1 only: query and key e4m3fn, both scales and the weights
     fp32 (the constraints section pairs FLOAT8_e4m3fn with fp32 scales
     and fp32 weights in quant_mode 1);
  I2 keys are paged like the attention's compressed KV: key
     [blocks, 128, 1, d] and key_dequant_scale [blocks, 128, 1] through
     block_table, seqused_k[b] keys in batch b;
  I3 mask_mode 0 attends every key j < seqused_k[b]; mask_mode 3 only the
     causally visible ones, j < floor((p_c + 1) / cmp_ratio) with
     p_c = S_k * cmp_ratio + cmp_residual_k[b] - S1_b + s (the same
     bottom-right alignment and visibility as the attention's compressed
     rows);
  I4 the top-k takes the k visible keys of largest score, a smaller key
     index first among equal scores; sparse_indices lists them in
     ascending key order (the attention treats its index row as a set)
     and fills the rest of the row with -1 (valid first, -1 after, as
     KvQuantSparseAttnSharedKv's constraints require of its indices);
     sparse_values holds their scores (bf16), -inf where the index is -1;
  I5 a padded query row (seqused_q) gets an all -1 row (BSND and TND);
     the other rows keep their positions (p_c takes the chunk length S1_b);
  I6 output_idx_offset, when given, is int32 [B]: every valid index of a
     batch-b row is reported plus output_idx_offset[b]; -1 stays -1;
  I7 layout_k: PA_BBND keys are paged through block_table (I2); BSND keys
     [B, S_k, 1, d] hold batch b's key j at [b, j], with seqused_k[b] keys
     (S_k when seqused_k is absent); TND keys [T_k, 1, d] hold it at
     cu_seqlens_k[b] + j, with cu_seqlens_k[b + 1] - cu_seqlens_k[b] keys.
     The scales follow the keys' layout without the d axis.
"""

from __future__ import annotations

import numpy as np

from oracle.qsfm_oracle import E4M3FN_TABLE, cmp_visible_count


def key_count(w, b: int) -> int:
    """Keys of batch b (I2, I7)."""
    layout = getattr(w, "layout_k", "PA_BBND")
    if layout == "TND":
        return int(w.cu_seqlens_k[b + 1]) - int(w.cu_seqlens_k[b])
    if layout == "BSND" and w.seqused_k is None:
        return int(w.key.shape[1])
    return int(w.seqused_k[b])


def key_rows(w, b: int, v: int):
    """Batch b's keys 0 .. v - 1: e4m3 bytes [v, d] and fp32 scales [v] (I2, I7)."""
    layout = getattr(w, "layout_k", "PA_BBND")
    if layout == "PA_BBND":
        bs = int(w.key.shape[1])
        rows = [(int(w.block_table[b, j // bs]), j % bs) for j in range(v)]
        k = np.stack([np.asarray(w.key[blk, off, 0]) for blk, off in rows])
        sk = np.array([float(w.key_scale[blk, off, 0]) for blk, off in rows], dtype=np.float64)
    elif layout == "BSND":
        k = np.asarray(w.key[b, :v, 0])
        sk = np.asarray(w.key_scale[b, :v, 0], dtype=np.float64)
    else:
        base = int(w.cu_seqlens_k[b])
        k = np.asarray(w.key[base:base + v, 0])
        sk = np.asarray(w.key_scale[base:base + v, 0], dtype=np.float64)
    return k, sk


def token_scores(w, t: int) -> np.ndarray:
    """fp64 scores of every visible key of query token t (length V)."""
    b, s = int(w.token_batch()[t]), int(w.token_pos()[t])
    v = visible_keys(w, b, s)
    if v == 0:
        return np.zeros(0)
    kb, sk = key_rows(w, b, v)
    k = E4M3FN_TABLE[np.asarray(kb).astype(np.int64)]
    q = E4M3FN_TABLE[np.asarray(w.query[t]).astype(np.int64)]           # [g, d]
    sq = np.asarray(w.query_scale[t], dtype=np.float64)                 # [g]
    wt = np.asarray(w.weights[t], dtype=np.float64)                     # [g]
    dots = q @ k.T                                                      # [g, V]
    relu = np.maximum(0.0, (sq[:, None] * sk[None, :]) * dots)
    return wt @ relu                                                    # [V]


def visible_keys(w, b: int, s: int) -> int:
    """Keys query token s of batch b may select (I3, I5)."""
    if w.seqused_q is not None and s >= int(w.seqused_q[b]):
        return 0
    sk_len = key_count(w, b)
    if w.mask_mode == 0:
        return sk_len
    s1 = int(w.q_lens[b])
    res = int(w.cmp_residual_k[b]) if w.cmp_residual_k is not None else 0
    p_c = sk_len * int(w.cmp_ratio) + res - s1 + s
    return cmp_visible_count(p_c, sk_len, int(w.cmp_ratio), 3)


def select(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the top-k scores (I4): largest first, the smaller index
    among equals; returned in ascending index order."""
    order = np.lexsort((np.arange(scores.size), -scores))  # by -score, then index
    return np.sort(order[:k])


def reference(w, tokens=None):
    """sparse_indices int32 [n, topk] and scores fp64 [n, topk] (NaN-free;
    -inf where the index is -1) for the given tokens (default all)."""
    tokens = range(w.total_t) if tokens is None else list(tokens)
    tokens = list(tokens)
    k = int(w.topk)
    idx = np.full((len(tokens), k), -1, dtype=np.int32)
    val = np.full((len(tokens), k), -np.inf)
    offs = getattr(w, "output_idx_offset", None)
    tb = w.token_batch()
    for i, t in enumerate(tokens):
        sc = token_scores(w, t)
        sel = select(sc, k)
        off = 0 if offs is None else int(offs[int(tb[t])])
        idx[i, :sel.size] = sel + off
        val[i, :sel.size] = sc[sel]
    return idx, val


def boundary_gap(w, t: int) -> float:
    """Score gap at token t's top-k boundary: the k-th largest visible score
    minus the (k+1)-th (inf when every visible key is selected). A GPU
    computing the scores within half this gap selects the same set."""
    sc = np.sort(token_scores(w, t))[::-1]
    k = int(w.topk)
    if sc.size <= k:
        return np.inf
    return float(sc[k - 1] - sc[k])
