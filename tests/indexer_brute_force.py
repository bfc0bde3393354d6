"""Dense brute force of the lightning-indexer top-k, independent of the
oracle (used only to pin it on small inputs).

A different route to the same definition (QuantLightningIndexerV2,
"功能说明" formula): each batch's whole key cache is materialised by
indexing the paged key tensor with the block table (or slicing the BSND
slab / TND rows) and decoded with
torch's own float8_e4m3fn type; the scores of all keys come from one
einsum per batch, in the order the formula writes them
([1]_{1 x g} @ [(W @ [1]_{1 x S_k}) * ReLU((Sq @ Sk^T) * (Q @ K^T))]);
visibility is a per-key predicate (a compressed key covers original tokens
c r .. c r + r - 1 and is visible once its last token is <= p_c); the
top-k is a Python sort by (-score, key index).
"""

from __future__ import annotations

import torch


def _cache(w, b):
    """Batch b's whole key cache, decoded: paged keys by indexing the pool
    with the block table, BSND keys by slicing the batch's slab to seqused_k
    (all of it when absent), TND keys by slicing rows cu_seqlens_k[b] ..
    cu_seqlens_k[b + 1]."""
    layout = getattr(w, "layout_k", "PA_BBND")
    if layout == "PA_BBND":
        n = int(w.seqused_k[b])
        bs = w.key.shape[1]
        blocks = w.block_table[b, :(n + bs - 1) // bs].long()
        raw = w.key[blocks].reshape(-1, w.key.shape[-1])[:n]
        sk = w.key_scale[blocks].reshape(-1)[:n]
    elif layout == "BSND":
        n = int(w.key.shape[1]) if w.seqused_k is None else int(w.seqused_k[b])
        raw = w.key[b, :n, 0]
        sk = w.key_scale[b, :n, 0]
    else:
        lo, hi = int(w.cu_seqlens_k[b]), int(w.cu_seqlens_k[b + 1])
        raw = w.key[lo:hi, 0]
        sk = w.key_scale[lo:hi, 0]
    return raw.contiguous().view(torch.float8_e4m3fn).to(torch.float64), sk.to(torch.float64)


def _visible(c, p_c, r):
    return c * r + r - 1 <= p_c


def brute_force(w):
    """(indices int32 [T, topk], values fp64 [T, topk]) for every query token."""
    T, k = w.total_t, int(w.topk)
    idx = torch.full((T, k), -1, dtype=torch.int32)
    val = torch.full((T, k), float("-inf"), dtype=torch.float64)
    t = 0
    for b in range(w.batch):
        keys, sk = _cache(w, b)
        n = keys.shape[0]
        s1 = int(w.q_lens[b])
        for s in range(s1):
            if w.seqused_q is not None and s >= int(w.seqused_q[b]):
                t += 1
                continue
            q = w.query[t].contiguous().view(torch.float8_e4m3fn).to(torch.float64)  # [g, d]
            sq = w.query_scale[t].to(torch.float64)
            wt = w.weights[t].to(torch.float64)
            ones_g = torch.ones(1, q.shape[0], dtype=torch.float64)
            ones_s = torch.ones(1, n, dtype=torch.float64)
            inner = torch.relu((sq[:, None] @ sk[None, :]) * torch.einsum("hd,jd->hj", q, keys))
            scores = (ones_g @ ((wt[:, None] @ ones_s) * inner)).reshape(-1)  # [n]
            if w.mask_mode == 3:
                res = int(w.cmp_residual_k[b]) if w.cmp_residual_k is not None else 0
                p_c = n * w.cmp_ratio + res - s1 + s
                cand = [j for j in range(n) if _visible(j, p_c, w.cmp_ratio)]
            else:
                cand = list(range(n))
            ranked = sorted(cand, key=lambda j: (-float(scores[j]), j))[:k]
            ranked.sort()
            offs = getattr(w, "output_idx_offset", None)
            shift = 0 if offs is None else int(offs[b])
            for i, j in enumerate(ranked):
                idx[t, i] = j + shift
                val[t, i] = scores[j]
            t += 1
    return idx, val
