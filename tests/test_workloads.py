"""The seeded synthetic inputs follow their stated recipe (CPU only).

Checks the generators in ``workloads/`` against the input recipe: distinct,
visible, valid-first CSA indices; block tables that are a permutation of
the pool; per-64-tile e4m3fn quantisation with scale = amax / 448; packed
and bf16 rows; lengths inside their stated ranges; determinism per seed.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W


def _visible(w, t):
    """Visible compressed rows V of token t (floor((p_c + 1) / r), clipped)."""
    b, s = int(w.token_batch()[t]), int(w.token_pos()[t])
    s2, s1 = int(w.seqused_ori_kv[b]), int(w.q_lens[b])
    cmp_len = s2 // w.cmp_ratio
    res = int(w.cmp_residual_kv[b]) if w.cmp_residual_kv is not None else 0
    p_c = cmp_len * w.cmp_ratio + res - s1 + s
    return max(0, min(cmp_len, (p_c + 1) // w.cmp_ratio))


def _check_indices(w, tokens, n_valid=None):
    idx = w.cmp_sparse_indices.numpy()
    for t in tokens:
        row = idx[t, 0]
        valid = row[row >= 0]
        n = len(valid)
        assert np.all(row[:n] >= 0) and np.all(row[n:] == -1), "valid entries first, then -1"
        assert len(np.unique(valid)) == n, "indices are distinct"
        v = _visible(w, t)
        assert np.all(valid < v), "indices name visible compressed rows only"
        want = min(w.k2 if n_valid is None else n_valid, v)
        assert n == want


@pytest.mark.parametrize("i", [0, 2])
def test_csa_indices_are_distinct_visible_and_valid_first(i):
    w = W.config(i)
    _check_indices(w, range(w.total_t), n_valid=384 if i == 0 else None)


def test_chunked_prefill_indices_on_a_sample():
    w = W.config(4)
    _check_indices(w, W.subset_tokens(w, 200, seed=3))


@pytest.mark.parametrize("i", [0, 2, 3])
def test_block_tables_are_a_permutation_of_the_pool(i):
    w = W.config(i)
    for pool, table, lengths in [(w.ori_kv, w.ori_block_table, w.seqused_ori_kv.numpy()),
                                 (w.cmp_kv, w.cmp_block_table,
                                  None if w.cmp_kv is None else w.seqused_ori_kv.numpy() // w.cmp_ratio)]:
        if pool is None:
            continue
        tab = table.numpy()
        used = []
        for b, n in enumerate(lengths):
            k = (int(n) + 127) // 128
            assert np.all(tab[b, :k] >= 0) and np.all(tab[b, k:] == -1)
            used.append(tab[b, :k])
        used = np.concatenate(used)
        assert np.array_equal(np.sort(used), np.arange(pool.shape[0])), "each physical block used once"


def test_lengths_are_inside_the_stated_ranges():
    w2, w3, w4 = W.config(2), W.config(3), W.config(4)
    assert w2.batch == 128 and np.all(w2.q_lens == 2)
    s2 = w2.seqused_ori_kv.numpy()
    assert s2.min() >= 4096 and s2.max() <= 65536
    s3 = w3.seqused_ori_kv.numpy()
    assert w3.batch == 64 and s3.min() >= 32768 and s3.max() <= 131072
    assert w4.batch == 8 and w4.q_lens.min() >= 512 and w4.q_lens.max() <= 4096
    s4 = w4.seqused_ori_kv.numpy()
    assert s4.min() >= 8192 and s4.max() <= 32768 and np.all(s4 >= w4.q_lens)
    assert w4.return_lse


def test_fp8_rows_are_tile_quantised_with_amax_over_448():
    w = W.config(0)
    kv = w.ori_kv.reshape(-1, 512)
    sc = w.ori_scale.reshape(-1, 8)
    codes = kv.numpy()
    assert not np.any((codes & 0x7F) == 0x7F), "no NaN codes"
    vals = kv.view(torch.float8_e4m3fn).to(torch.float64).reshape(-1, 8, 64)
    amax_q = vals.abs().amax(dim=-1)  # largest code magnitude per tile
    # scale = amax / 448 puts each tile's largest element at the top code
    assert torch.all(amax_q == 448.0)
    assert torch.all(sc > 0)


def test_packed_rows_follow_the_row_layout():
    w = W.config(0, kv_format="packed640")
    rows = w.ori_kv.reshape(-1, 640).numpy()
    assert np.all(rows[:, 583:] == 0), "zero padding after the seven scale bytes"
    nope = torch.from_numpy(rows[:, 128:576].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    tiles = nope.reshape(-1, 7, 64).abs().amax(dim=-1)
    # power-of-two scales, the smallest that keep a tile within e4m3fn's range:
    # amax / scale lies in (224, 448], and its e4m3fn code in [224, 448]
    assert torch.all(tiles <= 448.0) and torch.all(tiles >= 224.0)
    assert not np.any((rows[:, 128:576] & 0x7F) == 0x7F)


def test_bf16_rows_are_finite_normal_draws():
    w = W.config(0, kv_format="bf16")
    kv = w.ori_kv.reshape(-1, 512).float()
    assert torch.isfinite(kv).all()
    assert abs(kv.mean().item()) < 0.02 and abs(kv.std().item() - 1.0) < 0.02


def test_common_recipe_values():
    w = W.config(2)
    assert w.q.dtype == torch.bfloat16 and tuple(w.q.shape) == (256, 64, 512)
    assert w.sinks.dtype == torch.float32 and tuple(w.sinks.shape) == (64,)
    assert w.softmax_scale == pytest.approx(1 / math.sqrt(512))
    assert (w.ori_mask_mode, w.ori_win_left, w.ori_win_right, w.cmp_mask_mode) == (4, 127, 0, 3)
    assert w.cmp_ratio == 4 and w.k2 == 512


def test_same_seed_same_inputs():
    a, b = W.config(0), W.config(0)
    for name in ("q", "ori_kv", "ori_scale", "ori_block_table", "cmp_sparse_indices", "sinks"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    c = W.config(0, seed=1)
    assert not torch.equal(a.q, c.q)
