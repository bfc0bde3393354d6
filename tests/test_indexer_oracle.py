"""Pins for the fp64 oracle of the lightning-indexer top-k (CPU only).

QuantLightningIndexerV2, "功能说明" (formula and its three steps), "参数说明"
(query / key / weights / dequant scales, seqused, cmp_residual_k, topk,
mask_mode, cmp_ratio, sparse_indices, sparse_values). Each test checks the
oracle against something other than itself: the dense brute force built a
different way, closed forms, invariances of the formula, and planted
mistakes.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import indexer_oracle as I
from tests.indexer_brute_force import brute_force

CASES = [
    dict(layout="BSND", q_lens=[2, 2], sk=[300, 900], topk=64, mask_mode=3, cmp_ratio=4),
    dict(layout="TND", q_lens=[3, 1, 5], sk=[40, 700, 129], topk=50, mask_mode=3, cmp_ratio=3, heads=8),
    dict(layout="BSND", q_lens=[1, 1, 1], sk=[10, 0, 130], topk=32, mask_mode=0, heads=16, dim=64),
    dict(layout="TND", q_lens=[4, 2], sk=[256, 77], topk=300, mask_mode=3, cmp_ratio=128, heads=4),
    dict(layout="BSND", q_lens=[3, 3], sk=[200, 500], topk=20, mask_mode=3, cmp_ratio=4, seqused_q=[1, 3]),
    dict(layout="TND", q_lens=[4, 2, 5], sk=[150, 90, 400], topk=24, mask_mode=3, cmp_ratio=4, seqused_q=[2, 2, 0],
         heads=8),
    dict(layout="BSND", q_lens=[2, 2], sk=[300, 900], topk=40, mask_mode=3, cmp_ratio=4, layout_k="BSND",
         output_idx_offset=[1000, 5]),
    dict(layout="TND", q_lens=[3, 1, 5], sk=[40, 700, 129], topk=50, mask_mode=3, cmp_ratio=3, heads=8,
         layout_k="TND", output_idx_offset=[0, 40, 740]),
    dict(layout="BSND", q_lens=[1, 1], sk=[260, 260], topk=30, mask_mode=0, layout_k="BSND", bsnd_seqused=False),
]


def _check(w):
    idx, val = I.reference(w)
    bi, bv = brute_force(w)
    assert np.array_equal(idx, bi.numpy())
    fin = np.isfinite(val)
    assert np.array_equal(fin, np.isfinite(bv.numpy()))
    assert np.allclose(val[fin], bv.numpy()[fin], rtol=1e-12, atol=1e-12)
    return idx, val


@pytest.mark.parametrize("i", range(len(CASES)))
def test_oracle_matches_brute_force(i):
    _check(W.build_indexer(f"ix{i}", seed=70 + i, **CASES[i]))


def test_rows_are_valid_first_and_padded():
    w = W.build_indexer("pad", layout="TND", q_lens=[2, 2], sk=[30, 600], topk=100, mask_mode=3, seed=3)
    idx, val = I.reference(w)
    for t in range(w.total_t):
        row = idx[t]
        v = row[row >= 0]
        assert np.all(row[v.size:] == -1) and np.all(np.diff(v) > 0)  # ascending, then -1
        assert np.all(np.isinf(val[t, v.size:]))
    assert (idx[0] >= 0).sum() < 100  # 30 keys / r = 4: fewer visible than topk


def test_one_head_one_hot_query_closed_form():
    """One head, weight 1, query e_0 (e4m3 byte 0x38 = 1.0): the score of key
    j is max(0, Sq * Sk_j * K[j, 0]), computed here from the bytes."""
    w = W.build_indexer("onehot", layout="BSND", q_lens=[1], sk=[200], topk=10, mask_mode=0, heads=1, dim=64,
                        seed=4)
    w.query.zero_()
    w.query[0, 0, 0] = 0x38
    w.weights.fill_(1.0)
    idx, val = I.reference(w)
    k0 = w.key[w.block_table[0, :2].long()].reshape(-1, 64)[:200, 0]
    ks = w.key_scale[w.block_table[0, :2].long()].reshape(-1)[:200].double()
    x = k0.view(torch.float8_e4m3fn).double() * ks * float(w.query_scale[0, 0])
    expect = np.maximum(0.0, x.numpy())
    order = sorted(range(200), key=lambda j: (-expect[j], j))[:10]
    assert idx[0].tolist() == sorted(order)
    assert np.allclose(val[0], expect[sorted(order)], rtol=1e-15)


def test_ties_take_the_smaller_index():
    """Zero weights make every score 0: the top-k is the k smallest visible
    key indices, as the brute force's (-score, index) sort gives."""
    w = W.build_indexer("ties", layout="BSND", q_lens=[2], sk=[100], topk=5, mask_mode=3, seed=8)
    w.weights.zero_()
    idx, _ = _check(w)
    assert idx[0].tolist() == list(range(5))


def test_permuting_heads_leaves_scores_unchanged():
    w = W.build_indexer("perm", layout="BSND", q_lens=[2], sk=[500], topk=40, mask_mode=3, seed=5)
    ref = I.reference(w)
    p = torch.randperm(w.heads, generator=torch.Generator().manual_seed(1))
    w.query, w.query_scale, w.weights = w.query[:, p], w.query_scale[:, p], w.weights[:, p]
    idx, val = I.reference(w)
    assert np.array_equal(idx, ref[0]) and np.allclose(val, ref[1], rtol=1e-12)


def test_positive_weight_scaling_scales_scores_exactly():
    w = W.build_indexer("scale", layout="BSND", q_lens=[2], sk=[500], topk=40, mask_mode=3, seed=6)
    ref = I.reference(w)
    w.weights *= 4.0
    idx, val = I.reference(w)
    assert np.array_equal(idx, ref[0]) and np.array_equal(val, 4.0 * ref[1])


def test_relu_drops_negative_correlations():
    """With the query negated, a head's contribution is ReLU of the negated
    product: the two scores add up to sum_h W |Sq Sk q.k|."""
    w = W.build_indexer("neg", layout="BSND", q_lens=[1], sk=[128], topk=128, mask_mode=0, heads=8, seed=7)
    s_pos = I.token_scores(w, 0)
    w.query ^= 0x80  # the e4m3 sign bit
    s_neg = I.token_scores(w, 0)
    w.query ^= 0x80
    from oracle.qsfm_oracle import E4M3FN_TABLE
    q = E4M3FN_TABLE[w.query[0].numpy().astype(np.int64)]
    k = E4M3FN_TABLE[w.key[w.block_table[0, 0].long(), :, 0].numpy().astype(np.int64)]
    sk = w.key_scale[w.block_table[0, 0].long(), :, 0].double().numpy()
    absval = np.abs(w.query_scale[0].double().numpy()[:, None] * sk[None, :] * (q @ k.T))
    assert np.allclose(s_pos + s_neg, w.weights[0].double().numpy() @ absval, rtol=1e-12)


# ------------------------------------------------ planted mistakes (oracle)
def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def _brute_pins():
    return [lambda i=i: test_oracle_matches_brute_force(i) for i in range(len(CASES))]


def _scores_variant(w, t, relu_after_weight=False, drop_key_scale=False):
    """The oracle's score with one planted mistake (written out here)."""
    from oracle.qsfm_oracle import E4M3FN_TABLE
    b, s = int(w.token_batch()[t]), int(w.token_pos()[t])
    v = I.visible_keys(w, b, s)
    if v == 0:
        return np.zeros(0)
    bs = int(w.key.shape[1])
    blk = [int(w.block_table[b, j // bs]) for j in range(v)]
    k = E4M3FN_TABLE[np.stack([w.key[blk[j], j % bs, 0].numpy() for j in range(v)]).astype(np.int64)]
    sk = np.array([float(w.key_scale[blk[j], j % bs, 0]) for j in range(v)])
    if drop_key_scale:
        sk = np.ones_like(sk)
    q = E4M3FN_TABLE[w.query[t].numpy().astype(np.int64)]
    x = (w.query_scale[t].double().numpy()[:, None] * sk[None, :]) * (q @ k.T)
    wt = w.weights[t].double().numpy()
    if relu_after_weight:
        return np.maximum(0.0, wt[:, None] * x).sum(axis=0)
    return wt @ np.maximum(0.0, x)


@pytest.mark.parametrize("mistake", ["relu_after_weight", "drop_key_scale"])
def test_score_mistakes_are_caught(monkeypatch, mistake):
    monkeypatch.setattr(I, "token_scores", lambda w, t: _scores_variant(w, t, **{mistake: True}))
    assert any(_fails(p) for p in _brute_pins())


def test_largest_index_first_on_ties_is_caught(monkeypatch):
    monkeypatch.setattr(I, "select", lambda sc, k: np.sort(np.lexsort((-np.arange(sc.size), -sc))[:k]))
    assert _fails(test_ties_take_the_smaller_index)


def test_visibility_off_by_one_is_caught(monkeypatch):
    real = I.visible_keys
    monkeypatch.setattr(I, "visible_keys", lambda w, b, s: real(w, b, s) + (1 if w.mask_mode == 3 else 0))
    assert any(_fails(p) for p in _brute_pins())


def test_key_layouts_give_the_same_rows():
    """The same logical keys stored paged, as BSND slabs and as TND rows
    (the generator stores one draw three ways) give identical rows and
    scores; an offset shifts every valid index of its batch and no -1."""
    base = dict(layout="TND", q_lens=[3, 2], sk=[500, 140], topk=200, mask_mode=3, cmp_ratio=4, seed=40)
    ref = I.reference(W.build_indexer("pa", **base))
    for lk in ("BSND", "TND"):
        got = I.reference(W.build_indexer(lk, layout_k=lk, **base))
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    idx, _ = I.reference(W.build_indexer("off", layout_k="TND", output_idx_offset=[7, 500], **base))
    tb = np.repeat([0, 1], [3, 2])
    shift = np.where(ref[0] >= 0, np.array([7, 500])[tb][:, None], 0)
    assert np.array_equal(idx, ref[0] + shift)


def test_tnd_key_base_off_by_one_is_caught(monkeypatch):
    real = I.key_rows

    def shifted(w, b, v):
        if getattr(w, "layout_k", "PA_BBND") == "TND" and b > 0:
            base = int(w.cu_seqlens_k[b]) + 1
            return np.asarray(w.key[base:base + v, 0]), np.asarray(w.key_scale[base:base + v, 0], dtype=np.float64)
        return real(w, b, v)

    monkeypatch.setattr(I, "key_rows", shifted)
    assert any(_fails(p) for p in _brute_pins())


def test_missing_offset_is_caught(monkeypatch):
    real = I.reference

    def no_offset(w, tokens=None):
        saved = w.output_idx_offset
        w.output_idx_offset = None
        try:
            return real(w, tokens)
        finally:
            w.output_idx_offset = saved

    monkeypatch.setattr(I, "reference", no_offset)
    assert any(_fails(p) for p in _brute_pins())
