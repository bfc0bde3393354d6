"""Pins for the oracle's ori_sparse_indices / ori_topk_length and its
non-paged BSND / TND KV layouts (CPU only).

QuantSparseFlashMla, parameter table rows ori_sparse_indices (discrete
picks from ori_kv, -1 = invalid), ori_topk_length (how many entries take
part), cu_seqlens_ori_kv / cu_seqlens_cmp_kv (TND prefix sums), layout_kv;
its constraints on the BSND / TND KV layouts and on seqused_cmp_kv.

Each test checks the oracle against something other than itself: the dense
brute force (which slices each batch's rows out of the BSND / TND tensors
and weights every key by per-key predicates), the same logical rows stored
in a paged pool by this file's own scatter, closed forms (no attended row
gives O = 0 and lse = -inf), and invariances of the definition.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import qsfm_oracle as O
from tests.brute_force import brute_force


def _close(a, b):
    o1, l1 = a
    o2, l2 = b
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-13)
    f1, f2 = np.isfinite(l1), np.isfinite(l2)
    assert np.array_equal(f1, f2)
    assert np.allclose(l1[f1], l2[f2], rtol=1e-12, atol=1e-12)


def _bf(w):
    o, l = brute_force(w)
    return o.numpy(), l.numpy()


CASES = [
    # non-paged BSND KV, window picks (20 of up to 24 slots valid)
    dict(layout="BSND", q_lens=[2, 2], s2=[50, 90], cmp_ratio=4, mode="CSA", k2=16, block_size=16,
         layout_kv="BSND", ori_k1=24, ori_n_valid=20),
    # TND KV with filler rows past the last batch, HCA, window 20
    dict(layout="TND", q_lens=[3, 1, 4], s2=[50, 9, 130], cmp_ratio=4, mode="HCA", block_size=16,
         layout_kv="TND", kv_pad=7, ori_win_left=20),
    # paged KV with causal ori picks cut by ori_topk_length (one row cut to 0)
    dict(layout="BSND", q_lens=[2, 2], s2=[64, 90], cmp_ratio=4, mode="CSA", k2=8, block_size=16,
         ori_k1=12, ori_topk_length=[3, 12, 0, 7], ori_mask_mode=3, ori_win_left=-1, ori_win_right=-1),
    # TND KV, SWA with ori picks over the whole sequence (mask mode 0)
    dict(layout="TND", q_lens=[5, 2], s2=[40, 70], mode="SWA", block_size=16, layout_kv="TND",
         ori_k1=16, ori_mask_mode=0, ori_win_left=-1, ori_win_right=-1),
    # BSND KV without seqused (every batch fills its slab), band 10 / 2
    dict(layout="BSND", q_lens=[3, 3], s2=[60, 60], cmp_ratio=3, mode="HCA", block_size=16,
         layout_kv="BSND", bsnd_seqused=False, ori_win_left=10, ori_win_right=2),
    # packed rows and bf16 rows in the non-paged layouts
    dict(layout="BSND", q_lens=[1, 1], s2=[80, 33], cmp_ratio=4, mode="CSA", k2=8, block_size=16,
         layout_kv="BSND", kv_format="packed640", ori_k1=10),
    dict(layout="TND", q_lens=[2, 3], s2=[45, 77], cmp_ratio=4, mode="CSA", k2=8, block_size=16,
         layout_kv="TND", kv_format="bf16", ori_k1=6, ori_win_left=30),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_oracle_matches_brute_force(i):
    w = W.build(f"oriL{i}", seed=400 + i, **CASES[i])
    _close(O.reference(w), _bf(w))


def test_brute_force_counts_duplicate_and_drops_masked_ori_picks():
    w = W.build("dup", layout="BSND", q_lens=[1], s2=[64], mode="SWA", block_size=16, ori_k1=8,
                ori_win_left=10, seed=41)
    # p = 63, band 53..63: 60 twice, 53 and 63 at the edges, 52 and 64 outside
    w.ori_sparse_indices[0, 0] = torch.tensor([60, 60, 53, -1, 63, 52, 64, -7], dtype=torch.int32)
    ori, _ = O.token_rows(w, 0, 0, 0)
    assert ori == [60, 60, 53, 63]
    _close(O.reference(w), _bf(w))


def test_window_listed_as_picks_equals_the_window():
    """Picks that list the window rows in order give the window's rows in
    the same order, so the oracle's result is bit-identical."""
    kw = dict(layout="BSND", q_lens=[2, 2], s2=[100, 300], cmp_ratio=4, mode="CSA", k2=16,
              block_size=16, ori_win_left=30, seed=42)
    w = W.build("win", **kw)
    o1, l1 = O.reference(w)
    w.ori_sparse_indices = torch.full((w.total_t, 1, 40), -1, dtype=torch.int32)
    w.ori_topk_length = None
    for t, (b, s) in enumerate(zip(w.token_batch(), w.token_pos())):
        s2, s1 = int(w.seqused_ori_kv[b]), int(w.q_lens[b])
        p = s2 - s1 + int(s)
        rows = list(range(max(0, p - 30), p + 1))
        w.ori_sparse_indices[t, 0, :len(rows)] = torch.tensor(rows, dtype=torch.int32)
    o2, l2 = O.reference(w)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_permuting_ori_picks_leaves_output_unchanged():
    w = W.build("perm", layout="TND", q_lens=[3, 2], s2=[200, 333], cmp_ratio=4, mode="CSA", k2=16,
                block_size=16, layout_kv="TND", ori_k1=48, ori_n_valid=40, ori_win_left=100, seed=43)
    ref = O.reference(w)
    g = torch.Generator().manual_seed(9)
    for t in range(w.total_t):
        w.ori_sparse_indices[t, 0] = w.ori_sparse_indices[t, 0, torch.randperm(w.k1, generator=g)]
    _close(O.reference(w), ref)


def test_topk_length_equals_cutting_the_row():
    w = W.build("cut", layout="BSND", q_lens=[2, 2], s2=[90, 120], mode="SWA", block_size=16,
                ori_k1=16, ori_topk_length=[5, 16, 0, 9], ori_win_left=60, seed=44)
    ref = O.reference(w)
    for t, n in enumerate([5, 16, 0, 9]):
        w.ori_sparse_indices[t, 0, n:] = -1
    w.ori_topk_length = None
    o, l = O.reference(w)
    assert np.array_equal(o, ref[0]) and np.array_equal(l, ref[1])


def test_no_valid_pick_without_cmp_gives_zero_and_minus_inf():
    """SWA with every ori pick -1: no attended row (O = 0, lse = -inf, even
    with a sink)."""
    w = W.build("none", layout="TND", q_lens=[2, 3], s2=[40, 50], mode="SWA", block_size=16,
                layout_kv="TND", ori_k1=8, seed=45)
    w.ori_sparse_indices.fill_(-1)
    o, l = O.reference(w)
    assert np.all(o == 0) and np.all(l == -np.inf)


def _paged_copy(w, block=16, seed=0):
    """The same logical rows in a paged pool: this test's own scatter of
    each batch's rows into shuffled blocks of `block` rows."""
    g = torch.Generator().manual_seed(seed)

    def scatter(kv, sc, cu, lengths):
        nblk = [(n + block - 1) // block for n in lengths]
        perm = torch.randperm(sum(nblk), generator=g)
        width = max(nblk)
        row = kv.shape[-1]
        pool = torch.zeros((sum(nblk), block, 1, row), dtype=kv.dtype)
        spool = None if sc is None else torch.zeros((sum(nblk), block, 1, sc.shape[-1]), dtype=sc.dtype)
        table = torch.full((len(lengths), width), -1, dtype=torch.int32)
        k = 0
        for b, n in enumerate(lengths):
            src = kv[b, :n, 0] if cu is None else kv[int(cu[b]):int(cu[b]) + n, 0]
            ssrc = None if sc is None else (sc[b, :n, 0] if cu is None else sc[int(cu[b]):int(cu[b]) + n, 0])
            for i in range(nblk[b]):
                blk = int(perm[k])
                k += 1
                table[b, i] = blk
                lo, hi = i * block, min(n, (i + 1) * block)
                pool[blk, :hi - lo, 0] = src[lo:hi]
                if spool is not None:
                    spool[blk, :hi - lo, 0] = ssrc[lo:hi]
        return pool, spool, table

    cu_o = w.cu_seqlens_ori_kv
    s2 = [int(cu_o[b + 1] - cu_o[b]) for b in range(w.batch)] if cu_o is not None else \
        [int(x) for x in (w.seqused_ori_kv if w.seqused_ori_kv is not None else [w.ori_kv.shape[1]] * w.batch)]
    pa = W.Workload(**{f: getattr(w, f) for f in w.__dataclass_fields__})
    pa.layout_kv = "PA_BBND"
    pa.cu_seqlens_ori_kv = pa.cu_seqlens_cmp_kv = None
    pa.ori_kv, pa.ori_scale, pa.ori_block_table = scatter(w.ori_kv, w.ori_scale, cu_o, s2)
    pa.seqused_ori_kv = torch.tensor(s2, dtype=torch.int32)
    if w.cmp_kv is not None:
        cu_c = w.cu_seqlens_cmp_kv
        if w.seqused_cmp_kv is not None:
            s3 = [int(x) for x in w.seqused_cmp_kv]
        elif cu_c is not None:
            s3 = [int(cu_c[b + 1] - cu_c[b]) for b in range(w.batch)]
        else:
            s3 = [int(w.cmp_kv.shape[1])] * w.batch
        pa.cmp_kv, pa.cmp_scale, pa.cmp_block_table = scatter(w.cmp_kv, w.cmp_scale, cu_c, s3)
        pa.seqused_cmp_kv = torch.tensor(s3, dtype=torch.int32)
    return pa


@pytest.mark.parametrize("i", [0, 1, 4, 5, 6])
def test_non_paged_layouts_equal_the_same_rows_paged(i):
    w = W.build(f"dense{i}", seed=500 + i, **CASES[i])
    assert w.layout_kv in ("BSND", "TND")
    o1, l1 = O.reference(w)
    o2, l2 = O.reference(_paged_copy(w, seed=i))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_bsnd_cmp_length_is_the_tensor_s_dimension():
    """BSND KV without seqused_cmp_kv: the cmp length is cmp_kv's S
    dimension, here 3 rows more than floor(S2 / cmp_ratio) (HCA, no cmp
    mask, so every row of the slab is attended)."""
    w = W.build("s3", layout="BSND", q_lens=[2, 2], s2=[60, 60], cmp_ratio=3, mode="HCA", block_size=16,
                layout_kv="BSND", bsnd_seqused=False, cmp_mask_mode=0, seed=48)
    g = torch.Generator().manual_seed(3)
    extra = torch.randint(0, 120, (2, 3, 1, 512), generator=g, dtype=torch.uint8)
    w.cmp_kv = torch.cat([w.cmp_kv, extra], dim=1)
    w.cmp_scale = torch.cat([w.cmp_scale, torch.rand(2, 3, 1, 8, generator=g)], dim=1)
    _, cmp_rows = O.token_rows(w, 0, 0, 0)
    assert cmp_rows == list(range(23))
    _close(O.reference(w), _bf(w))


def test_generator_layouts_and_shapes():
    w = W.build("shape", layout="TND", q_lens=[3, 2], s2=[50, 70], cmp_ratio=4, mode="CSA", k2=8,
                block_size=16, layout_kv="TND", kv_pad=5, ori_k1=12, seed=46)
    assert w.ori_block_table is None and w.seqused_ori_kv is None
    assert tuple(w.ori_kv.shape) == (125, 1, 512) and tuple(w.ori_scale.shape) == (125, 1, 8)
    assert w.cu_seqlens_ori_kv.tolist() == [0, 50, 120]
    assert w.cu_seqlens_cmp_kv.tolist() == [0, 12, 29]
    assert tuple(w.ori_sparse_indices.shape) == (5, 1, 12) and w.k1 == 12
    w = W.build("shape2", layout="BSND", q_lens=[2, 2], s2=[50, 70], cmp_ratio=4, mode="HCA",
                block_size=16, layout_kv="BSND", seed=47)
    assert tuple(w.ori_kv.shape) == (2, 70, 1, 512) and tuple(w.cmp_kv.shape) == (2, 17, 1, 512)
    assert w.seqused_cmp_kv.tolist() == [12, 17]


# ------------------------------------------------ planted mistakes (oracle)
def _fails(pins):
    """The pins that fail under the planted mistake (a wrong value or a
    crash on an out-of-range row both count)."""
    failed = []
    for pin in pins:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failed.append(pin)
    return failed


BRUTE = [lambda i=i: test_oracle_matches_brute_force(i) for i in range(len(CASES))]


def test_unmasked_ori_picks_are_caught(monkeypatch):
    def picks(w, t, lo, hi):
        idx = w.ori_sparse_indices
        n = int(idx.shape[-1]) if w.ori_topk_length is None else min(int(idx.shape[-1]), int(w.ori_topk_length[t]))
        return [int(e) for e in idx[t, 0, :max(n, 0)].tolist() if e != -1]  # mask range not applied
    monkeypatch.setattr(O, "ori_picks", picks)
    with pytest.raises(Exception):
        test_brute_force_counts_duplicate_and_drops_masked_ori_picks()


def test_ignored_topk_length_is_caught(monkeypatch):
    def picks(w, t, lo, hi):
        return [int(e) for e in w.ori_sparse_indices[t, 0].tolist() if e != -1 and lo <= e <= hi]
    monkeypatch.setattr(O, "ori_picks", picks)
    assert _fails([test_topk_length_equals_cutting_the_row] + BRUTE)


def test_wrong_tnd_row_base_is_caught(monkeypatch):
    real = O.gather_dense

    def gather(kv, scales, w, b, rows, cu):
        if O.kv_layout_of(w) == "TND":
            cu = [int(x) for x in cu[1:]] + [0]  # batch b read from batch b + 1's start
        return real(kv, scales, w, b, rows, cu)
    monkeypatch.setattr(O, "gather_dense", gather)
    assert _fails(BRUTE)


def test_paged_cmp_length_rule_on_bsnd_kv_is_caught(monkeypatch):
    def cmp_len(w, b, s2):
        if w.seqused_cmp_kv is not None:
            return int(w.seqused_cmp_kv[b])
        return s2 // int(w.cmp_ratio)  # the paged default applied to every layout
    monkeypatch.setattr(O, "cmp_length", cmp_len)
    assert _fails([test_bsnd_cmp_length_is_the_tensor_s_dimension])
