"""Dense brute-force evaluation of the attention, independent of the oracle.

Used only to pin the oracle on tiny inputs. It shares no code with
``oracle/`` and takes a different route to the same definition:

* the whole logical KV cache of a batch is materialised by indexing the pool
  with the block table (paged KV) or by slicing the batch's rows out of a
  BSND / TND tensor (non-paged KV), and decoded with torch's own
  float8_e4m3fn, float8_e8m0fnu and bfloat16 types;
* every query token is scored against *every* key of both caches, and a
  per-key weight (0 = masked, k = the key occurs k times among the CSA or
  ori sparse indices) is built from predicates written per key;
* the softmax with a sink is evaluated densely in float64.

Definitions followed: QuantSparseFlashMla, function description (formula,
modes), parameter table (masks, windows, sinks, residual); the readings are
the same ones the oracle documents (bottom-right alignment, inclusive band,
compressed row c covers tokens c*r .. c*r + r - 1).
"""

from __future__ import annotations

import torch


def _batch_rows(w, pool, scale_pool, table_row, cu, b, length):
    """Raw rows 0..length-1 of batch b (and their scale rows) in storage order."""
    layout_kv = getattr(w, "layout_kv", "PA_BBND")
    if layout_kv == "BSND":
        raw = pool[b, :length, 0]
        return raw, None if scale_pool is None else scale_pool[b, :length, 0]
    if layout_kv == "TND":
        start = int(cu[b])
        raw = pool[start:start + length, 0]
        return raw, None if scale_pool is None else scale_pool[start:start + length, 0]
    bs = pool.shape[1]
    nblk = (length + bs - 1) // bs
    blocks = table_row[:nblk].long()
    raw = pool[blocks].reshape(-1, pool.shape[-1])[:length]
    sc = None if scale_pool is None else scale_pool[blocks].reshape(-1, scale_pool.shape[-1])[:length]
    return raw, sc


def _logical_cache(w, pool, scale_pool, table_row, cu, b, length):
    """Decoded logical rows 0..length-1 of one batch, fp64 [length, 512]."""
    if length == 0:
        return torch.zeros(0, 512, dtype=torch.float64)
    raw, sc = _batch_rows(w, pool, scale_pool, table_row, cu, b, length)
    if raw.dtype == torch.bfloat16:  # unquantised bf16 rows
        return raw.to(torch.float64)
    if scale_pool is None:  # packed 640-byte rows: bf16 rope | e4m3fn nope | e8m0 scales | pad
        rope = raw[:, :128].contiguous().view(torch.bfloat16).to(torch.float64)
        nope = raw[:, 128:576].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
        sc = raw[:, 576:583].contiguous().view(torch.float8_e8m0fnu).to(torch.float64)
        return torch.cat([rope, nope * sc.repeat_interleave(64, dim=1)], dim=1)
    vals = raw.contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    tile = raw.shape[-1] // sc.shape[-1]
    return vals * sc.to(torch.float64).repeat_interleave(tile, dim=1)


def _ori_visible(j: int, p: int, s2: int, mode: int, wl: int, wr: int) -> bool:
    if j >= s2:
        return False
    if mode == 0:
        return True
    if mode == 3:
        return j <= p
    left_ok = wl == -1 or j >= p - wl
    right_ok = wr == -1 or j <= p + wr
    return left_ok and right_ok


def _cmp_visible(c: int, p_c: int, cmp_len: int, r: int, mode: int) -> bool:
    if c >= cmp_len or c < 0:
        return False
    if mode == 0:
        return True
    last_token = c * r + r - 1  # last original token the row summarises
    return last_token <= p_c


def brute_force(w):
    """O fp64 [T, 64, 512] and lse fp64 [T, 64] for every query token of w."""
    T = w.total_t
    nh, d = w.q.shape[1], w.q.shape[2]
    out = torch.zeros(T, nh, d, dtype=torch.float64)
    lse = torch.full((T, nh), float("-inf"), dtype=torch.float64)
    sink = (torch.full((nh,), float("-inf"), dtype=torch.float64) if w.sinks is None
            else w.sinks.to(torch.float64))
    layout_kv = getattr(w, "layout_kv", "PA_BBND")
    ori_idx = getattr(w, "ori_sparse_indices", None)
    t = 0
    for b in range(w.batch):
        s1 = int(w.q_lens[b])
        if layout_kv == "TND":
            s2 = int(w.cu_seqlens_ori_kv[b + 1] - w.cu_seqlens_ori_kv[b])
        elif w.seqused_ori_kv is not None:
            s2 = int(w.seqused_ori_kv[b])
        else:  # BSND without seqused: the tensor's S dimension
            s2 = int(w.ori_kv.shape[1])
        table = None if w.ori_block_table is None else w.ori_block_table[b]
        k_ori = _logical_cache(w, w.ori_kv, w.ori_scale, table, w.cu_seqlens_ori_kv, b, s2)
        k_cmp = torch.zeros(0, d, dtype=torch.float64)
        cmp_len, r, res = 0, 1, 0
        if w.cmp_kv is not None:
            r = int(w.cmp_ratio)
            if w.seqused_cmp_kv is not None:
                cmp_len = int(w.seqused_cmp_kv[b])
            elif layout_kv == "BSND":
                cmp_len = int(w.cmp_kv.shape[1])
            elif layout_kv == "TND":
                cmp_len = int(w.cu_seqlens_cmp_kv[b + 1] - w.cu_seqlens_cmp_kv[b])
            else:
                cmp_len = s2 // r
            res = int(w.cmp_residual_kv[b]) if w.cmp_residual_kv is not None else 0
            ctable = None if w.cmp_block_table is None else w.cmp_block_table[b]
            k_cmp = _logical_cache(w, w.cmp_kv, w.cmp_scale, ctable, w.cu_seqlens_cmp_kv, b, cmp_len)
        keys = torch.cat([k_ori, k_cmp], dim=0)
        for s in range(s1):
            if w.seqused_q is not None and s >= int(w.seqused_q[b]):
                t += 1
                continue
            p = s2 - s1 + s
            p_c = cmp_len * r + res - s1 + s
            weight = torch.zeros(keys.shape[0], dtype=torch.float64)
            if ori_idx is None:
                for j in range(s2):
                    if _ori_visible(j, p, s2, w.ori_mask_mode, w.ori_win_left, w.ori_win_right):
                        weight[j] = 1.0
            else:  # one weight per occurrence of a visible ori index
                n = ori_idx.shape[-1]
                if w.ori_topk_length is not None:
                    n = min(n, int(w.ori_topk_length[t]))
                for e in ori_idx[t, 0, :max(n, 0)].tolist():
                    if e >= 0 and _ori_visible(e, p, s2, w.ori_mask_mode, w.ori_win_left, w.ori_win_right):
                        weight[e] += 1.0
            if w.cmp_kv is not None:
                if w.cmp_sparse_indices is None:
                    for c in range(cmp_len):
                        if _cmp_visible(c, p_c, cmp_len, r, w.cmp_mask_mode):
                            weight[s2 + c] += 1.0
                else:
                    n = w.cmp_sparse_indices.shape[-1]
                    if w.cmp_topk_length is not None:
                        n = min(n, int(w.cmp_topk_length[t]))
                    for e in w.cmp_sparse_indices[t, 0, :n].tolist():
                        if _cmp_visible(e, p_c, cmp_len, r, w.cmp_mask_mode):
                            weight[s2 + e] += 1.0
            if weight.sum() == 0:
                t += 1
                continue
            q = w.q[t].to(torch.float64)
            x = w.softmax_scale * (q @ keys.T)  # [64, n_keys]
            live = weight > 0
            xl = x[:, live]
            wl_ = weight[live]
            m = torch.maximum(xl.max(dim=1).values, sink)
            e = torch.exp(xl - m[:, None]) * wl_[None, :]
            den = e.sum(dim=1) + torch.exp(sink - m)
            out[t] = (e @ keys[live]) / den[:, None]
            xm = xl.max(dim=1).values
            lse[t] = xm + torch.log((torch.exp(xl - xm[:, None]) * wl_[None, :]).sum(dim=1))
            t += 1
    return out, lse
