"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: the fp8
format definition, hand-derived mask fixtures, a dense brute force built a
different way, torch's SDPA, torch.logsumexp, closed forms of the sink
softmax, and invariances of the definition.
"""

import json
import math
import os
import types

import numpy as np
import pytest
import torch

import workloads as W
from oracle import qsfm_oracle as O
from tests.brute_force import brute_force

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp8 decode
def test_e4m3fn_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.E4M3FN_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    # signed zeros too
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_e4m3fn_golden_codes():
    n = 0
    for line in open(os.path.join(GOLDEN, "e4m3fn_codes.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()
        v = O.decode_e4m3fn_code(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))
        n += 1
    assert n >= 15


def test_dequant_uses_tile_of_column():
    b = np.full((1, 512), 0x38, dtype=np.uint8)  # 1.0 everywhere
    s = np.arange(1, 9, dtype=np.float32)[None, :]
    k = O.dequant_rows(b, s)
    for d in (0, 63, 64, 127, 448, 511):
        assert k[0, d] == float(d // 64 + 1)


def test_e8m0_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = O.E8M0_TABLE
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_packed_row_by_hand():
    """A 640-byte row built by hand: rope bf16 bit patterns, nope e4m3fn
    codes and e8m0 scales written from the format definitions."""
    row = np.zeros((1, 640), dtype=np.uint8)
    # rope element 0 = 1.5 (bf16 0x3FC0), element 63 = -2.0 (0xC000), little-endian
    row[0, 0:2] = [0xC0, 0x3F]
    row[0, 126:128] = [0x00, 0xC0]
    # nope element 0 (output 64) = 0x38 = 1.0, scale byte 126 = 2^-1 -> 0.5
    row[0, 128] = 0x38
    # nope element 447 (output 511) = 0xC4 (sign 1, exponent 1000b -> 2^1,
    # mantissa 100b -> 1.5) = -3.0, scale byte 6 = 130 = 2^3 -> -24
    row[0, 128 + 447] = 0xC4
    row[0, 576 + 0] = 126
    row[0, 576 + 6] = 130
    k = O.dequant_packed_rows(row)
    assert k.shape == (1, 512)
    assert k[0, 0] == 1.5 and k[0, 63] == -2.0
    assert k[0, 64] == 0.5 and k[0, 511] == -24.0
    assert np.count_nonzero(k) == 4


PACKED_CASES = [
    dict(layout="BSND", q_lens=[2, 2], s2=[100, 300], cmp_ratio=4, mode="CSA", k2=16, block_size=16,
         ori_win_left=40),
    dict(layout="TND", q_lens=[3, 4], s2=[60, 200], cmp_ratio=3, mode="HCA", block_size=16),
]


@pytest.mark.parametrize("i", range(len(PACKED_CASES)))
def test_oracle_matches_brute_force_packed_rows(i):
    w = W.build(f"packed{i}", seed=200 + i, kv_format="packed640", **PACKED_CASES[i])
    assert w.ori_kv.shape[-1] == 640 and w.ori_scale is None
    o_ref, l_ref = O.reference(w)
    o_bf, l_bf = brute_force(w)
    assert np.allclose(o_ref, o_bf.numpy(), rtol=1e-12, atol=1e-13)
    fin = np.isfinite(l_ref)
    assert np.allclose(l_ref[fin], l_bf.numpy()[fin], rtol=1e-12)


def test_bf16_all_bit_patterns_match_torch():
    """Every one of the 65,536 bf16 bit patterns, decoded by the oracle, equals
    torch's own bfloat16 -> float64 conversion (NaNs compared as NaNs)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype("<u2")
    rows = bits.view(np.uint8).reshape(-1, 1024)  # 64 rows of 512 elements
    with np.errstate(invalid="ignore"):  # the signalling-NaN patterns
        got = O.decode_bf16_rows(rows).reshape(-1)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))  # -0.0 kept


def test_bf16_row_by_hand():
    """A bf16 row (1024 little-endian bytes) built from the bf16 format
    definition: 1 sign bit, 8 exponent bits with bias 127, 7 mantissa bits."""
    row = np.zeros((1, 1024), dtype=np.uint8)
    row[0, 0:2] = [0xC0, 0x3F]      # element 0: 0x3FC0 = +2^0 * 1.5
    row[0, 2:4] = [0x80, 0xC0]      # element 1: 0xC080 = -2^(129-127) * 1.0
    row[0, 1022:1024] = [0x01, 0x00]  # element 511: 0x0001, the smallest subnormal 2^-133
    row[0, 600:602] = [0x49, 0x42]  # element 300: 0x4249 = 2^5 * (1 + 73/128) = 50.25
    k = O.decode_bf16_rows(row)
    assert k.shape == (1, 512)
    assert k[0, 0] == 1.5 and k[0, 1] == -4.0 and k[0, 300] == 50.25
    assert k[0, 511] == 2.0 ** -133
    assert np.count_nonzero(k) == 4


BF16_CASES = [
    dict(layout="TND", q_lens=[3, 2], s2=[90, 260], cmp_ratio=4, mode="CSA", k2=16, block_size=16,
         ori_win_left=31),
    dict(layout="TND", q_lens=[2, 3], s2=[70, 150], cmp_ratio=4, mode="HCA", block_size=16),
]


@pytest.mark.parametrize("i", range(len(BF16_CASES)))
def test_oracle_matches_brute_force_bf16_rows(i):
    w = W.build(f"bf16_{i}", seed=300 + i, kv_format="bf16", **BF16_CASES[i])
    assert str(w.ori_kv.dtype) == "torch.bfloat16" and w.ori_scale is None
    o_ref, l_ref = O.reference(w)
    o_bf, l_bf = brute_force(w)
    assert np.allclose(o_ref, o_bf.numpy(), rtol=1e-12, atol=1e-13)
    fin = np.isfinite(l_ref)
    assert np.allclose(l_ref[fin], l_bf.numpy()[fin], rtol=1e-12)


# -------------------------------------------------------------- mask fixtures
def _fake(S2, S1, mode=4, wl=127, wr=0, r=1, cmp_len=None, res=None, cmp_mode=3, cmp=False):
    return types.SimpleNamespace(
        q_lens=np.array([S1]), seqused_q=None, seqused_ori_kv=np.array([S2]),
        ori_mask_mode=mode, ori_win_left=wl, ori_win_right=wr,
        cmp_kv=object() if cmp else None, cmp_ratio=r,
        seqused_cmp_kv=None if cmp_len is None else np.array([cmp_len]),
        cmp_residual_kv=None if res is None else np.array([res]),
        cmp_mask_mode=cmp_mode, cmp_sparse_indices=None, cmp_topk_length=None)


def test_golden_ori_row_sets():
    cases = json.load(open(os.path.join(GOLDEN, "mask_cases.json")))["ori"]
    for c in cases:
        w = _fake(c["S2"], c["S1"], c["mode"], c["wl"], c["wr"])
        for s, exp in enumerate(c["ori"]):
            ori, _ = O.token_rows(w, s, 0, s)
            if exp is None:
                assert ori == [], (c["why"], s, ori)
            else:
                assert ori == list(range(exp[0], exp[1] + 1)), (c["why"], s)


def test_golden_cmp_visibility():
    cases = json.load(open(os.path.join(GOLDEN, "mask_cases.json")))["cmp"]
    for c in cases:
        # cmp_len passed explicitly only where it differs from floor(S2 / r)
        explicit = None if c["cmp_len"] == c["S2"] // c["r"] else c["cmp_len"]
        w = _fake(c["S2"], c["S1"], mode=0, r=c["r"], cmp_len=explicit, res=c["res"],
                  cmp_mode=c["mode"], cmp=True)
        for s, exp in enumerate(c["cmp_visible"]):
            _, cmp_rows = O.token_rows(w, s, 0, s)
            assert cmp_rows == list(range(exp)), (c["why"], s, len(cmp_rows), exp)


# ------------------------------------------------------------- brute force
SMALL_CASES = [
    dict(layout="BSND", q_lens=[1, 1], s2=[100, 300], cmp_ratio=4, mode="CSA", k2=16, n_valid=12,
         block_size=16, ori_win_left=40),
    dict(layout="BSND", q_lens=[3, 3], s2=[37, 130], cmp_ratio=4, mode="CSA", k2=24,
         block_size=16, ori_win_left=20, ori_win_right=1),
    dict(layout="TND", q_lens=[5, 2, 7], s2=[60, 9, 200], cmp_ratio=3, mode="HCA",
         block_size=16, ori_win_left=10, ori_win_right=0),
    dict(layout="TND", q_lens=[6, 4], s2=[6, 70], mode="SWA", block_size=16,
         ori_mask_mode=3, ori_win_left=-1, ori_win_right=-1),
    dict(layout="BSND", q_lens=[4, 4], s2=[3, 50], cmp_ratio=2, mode="HCA", block_size=8,
         ori_mask_mode=0, ori_win_left=-1, ori_win_right=-1, cmp_mask_mode=0),
    dict(layout="BSND", q_lens=[2, 2], s2=[64, 90], cmp_ratio=4, mode="CSA", k2=8,
         block_size=16, sinks=False, cmp_topk_length=[3, 8, 0, 5]),
    dict(layout="BSND", q_lens=[3, 3], s2=[64, 90], cmp_ratio=4, mode="CSA", k2=8,
         block_size=16, seqused_q=[2, 3], ori_win_left=5),
    dict(layout="TND", q_lens=[4], s2=[21], cmp_ratio=4, mode="HCA", block_size=4,
         with_residual=True, ori_win_left=3, ori_win_right=2),
]


@pytest.mark.parametrize("i", range(len(SMALL_CASES)))
def test_oracle_matches_brute_force(i):
    w = W.build(f"small{i}", seed=100 + i, **SMALL_CASES[i])
    o_ref, l_ref = O.reference(w)
    o_bf, l_bf = brute_force(w)
    o_bf, l_bf = o_bf.numpy(), l_bf.numpy()
    assert np.allclose(o_ref, o_bf, rtol=1e-12, atol=1e-13)
    fin = np.isfinite(l_bf)
    assert np.array_equal(fin, np.isfinite(l_ref))
    assert np.allclose(l_ref[fin], l_bf[fin], rtol=1e-12, atol=1e-12)
    assert np.all(l_ref[~fin] == -np.inf)


def test_oracle_matches_brute_force_128_heads():
    """N1 = 128 (the pages allow 64 and 128): same definition per head."""
    w = W.build("h128", layout="BSND", q_lens=[2, 2], s2=[80, 150], cmp_ratio=4, mode="CSA", k2=16,
                block_size=16, ori_win_left=20, n1=128, seed=31)
    assert tuple(w.q.shape[1:]) == (128, 512) and tuple(w.sinks.shape) == (128,)
    o_ref, l_ref = O.reference(w)
    o_bf, l_bf = brute_force(w)
    assert o_ref.shape == (4, 128, 512)
    assert np.allclose(o_ref, o_bf.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(l_ref, l_bf.numpy(), rtol=1e-12)


def test_brute_force_sees_duplicate_indices_as_multiset():
    w = W.build("dup", layout="BSND", q_lens=[1], s2=[64], cmp_ratio=4, mode="CSA", k2=8,
                block_size=16, seed=7)
    w.cmp_sparse_indices[0, 0, :] = torch.tensor([3, 3, 5, -1, 7, 3, -1, 2], dtype=torch.int32)
    o_ref, l_ref = O.reference(w)
    o_bf, l_bf = brute_force(w)
    assert np.allclose(o_ref, o_bf.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(l_ref, l_bf.numpy(), rtol=1e-12)


# --------------------------------------------------- library / closed forms
def test_causal_no_cmp_no_sink_equals_sdpa():
    """Mode 3 (or band with wl = -1, wr = 0), no cmp, no sink == causal SDPA."""
    for mode, wl, wr in ((3, -1, -1), (4, -1, 0)):
        w = W.build("causal", layout="TND", q_lens=[7, 5], s2=[40, 5], mode="SWA",
                    block_size=16, sinks=False, ori_mask_mode=mode, ori_win_left=wl,
                    ori_win_right=wr, seed=3)
        o_ref, _ = O.reference(w)
        t = 0
        for b in range(w.batch):
            s1, s2 = int(w.q_lens[b]), int(w.seqused_ori_kv[b])
            rows = list(range(s2))
            kb, ks = O.gather_paged(w.ori_kv.numpy(), w.ori_scale.numpy(),
                                    w.ori_block_table[b].numpy(), rows)
            k = torch.from_numpy(O.dequant_rows(kb, ks))
            q = w.q[t:t + s1].to(torch.float64).permute(1, 0, 2)  # [64, s1, 512]
            mask = torch.ones(s1, s2, dtype=torch.bool).tril(diagonal=s2 - s1)
            ref = torch.nn.functional.scaled_dot_product_attention(
                q, k[None].expand(64, -1, -1), k[None].expand(64, -1, -1),
                attn_mask=mask, scale=w.softmax_scale)
            assert np.allclose(o_ref[t:t + s1], ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-13)
            t += s1


def test_sink_minus_inf_is_plain_softmax():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((64, 512))
    k = rng.standard_normal((9, 512))
    o, lse = O.attend(q, k, 0.05, np.full(64, -np.inf))
    x = 0.05 * q @ k.T
    p = torch.softmax(torch.from_numpy(x), dim=1).numpy()
    assert np.allclose(o, p @ k, rtol=1e-13, atol=1e-14)
    o2, _ = O.attend(q, k, 0.05, None)
    assert np.array_equal(o, o2)


def test_single_key_sink_closed_form():
    """One key: O = sigmoid(x - sink) * v, with x = scale * q.k (sink unscaled)."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal((64, 512))
    k = rng.standard_normal((1, 512))
    sink = rng.standard_normal(64)
    o, lse = O.attend(q, k, 0.07, sink)
    x = 0.07 * (q @ k[0])
    sig = 1.0 / (1.0 + np.exp(-(x - sink)))
    assert np.allclose(o, sig[:, None] * k[0][None, :], rtol=1e-13, atol=1e-15)
    assert np.allclose(lse, x, rtol=1e-14)


def test_zero_query_gives_sink_damped_mean():
    """q = 0: every logit is 0, O = n / (n + e^sink) * mean_j v_j."""
    rng = np.random.default_rng(2)
    k = rng.standard_normal((13, 512))
    sink = rng.standard_normal(64)
    o, lse = O.attend(np.zeros((64, 512)), k, 0.1, sink)
    n = k.shape[0]
    exp = (n / (n + np.exp(sink)))[:, None] * k.mean(axis=0)[None, :]
    assert np.allclose(o, exp, rtol=1e-13, atol=1e-15)
    assert np.allclose(lse, np.log(n), rtol=1e-14)


def test_identical_rows_give_row_times_mass():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(512)
    k = np.repeat(v[None], 5, axis=0)
    q = rng.standard_normal((64, 512))
    sink = rng.standard_normal(64)
    o, _ = O.attend(q, k, 0.04, sink)
    x = 0.04 * q @ v
    mass = 5 * np.exp(x) / (5 * np.exp(x) + np.exp(sink))
    assert np.allclose(o, mass[:, None] * v[None, :], rtol=1e-13, atol=1e-15)


def test_empty_rows_give_zero_and_minus_inf():
    o, lse = O.attend(np.ones((64, 512)), np.zeros((0, 512)), 0.1, np.zeros(64))
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_lse_equals_torch_logsumexp_of_logits():
    w = W.build("lse", layout="BSND", q_lens=[2, 2], s2=[150, 260], cmp_ratio=4, mode="CSA",
                k2=32, block_size=16, ori_win_left=30, seed=11)
    _, lse = O.reference(w)
    for t in range(w.total_t):
        x = torch.from_numpy(O.logits(w, t))
        assert np.allclose(lse[t], torch.logsumexp(x, dim=1).numpy(), rtol=1e-13)


# ----------------------------------------------------------- invariances
def test_permuting_index_rows_leaves_output_unchanged():
    w = W.build("perm", layout="BSND", q_lens=[2, 2], s2=[200, 333], cmp_ratio=4, mode="CSA",
                k2=40, n_valid=30, block_size=16, seed=5)
    o1, l1 = O.reference(w)
    g = torch.Generator().manual_seed(9)
    for t in range(w.total_t):
        perm = torch.randperm(w.k2, generator=g)
        w.cmp_sparse_indices[t, 0] = w.cmp_sparse_indices[t, 0, perm]
    o2, l2 = O.reference(w)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14)
    assert np.allclose(l1, l2, rtol=1e-13)


def test_all_invalid_indices_equal_swa_only():
    w = W.build("neg", layout="BSND", q_lens=[2], s2=[300], cmp_ratio=4, mode="CSA", k2=16,
                block_size=16, seed=6)
    w.cmp_sparse_indices.fill_(-1)
    o_csa, l_csa = O.reference(w)
    w.cmp_kv = w.cmp_scale = w.cmp_block_table = w.cmp_sparse_indices = None
    w.cmp_ratio = 1
    o_swa, l_swa = O.reference(w)
    assert np.array_equal(o_csa, o_swa) and np.array_equal(l_csa, l_swa)


def test_invisible_indices_are_dropped():
    w = W.build("vis", layout="BSND", q_lens=[1], s2=[64], cmp_ratio=4, mode="CSA", k2=4,
                block_size=16, seed=8)
    # cmp_len = 16, p_c = 63 -> V = 16: entries 16, 99 and -5 must be ignored
    w.cmp_sparse_indices[0, 0] = torch.tensor([2, 16, 99, -5], dtype=torch.int32)
    _, rows = O.token_rows(w, 0, 0, 0)
    assert rows == [2]


def test_padded_query_rows_are_zero():
    w = W.build("pad", layout="BSND", q_lens=[3, 3], s2=[40, 40], mode="SWA", block_size=16,
                seqused_q=[1, 3], seed=12)
    o, lse = O.reference(w)
    assert np.all(o[1:3] == 0) and np.all(lse[1:3] == -np.inf)
    assert np.all(np.isfinite(lse[0])) and np.all(np.isfinite(lse[3:]))


def test_config_workloads_shapes():
    w = W.config(0)
    assert w.total_t == 2 and w.k2 == 512 and w.mode == "CSA"
    assert int((w.cmp_sparse_indices >= 0).sum()) == 2 * 384
    o, lse = O.reference(w)
    assert o.shape == (2, 64, 512) and np.all(np.isfinite(lse))


def test_reference_parallel_matches_serial():
    w = W.build("par", layout="BSND", q_lens=[2, 2], s2=[300, 500], cmp_ratio=4, mode="CSA", k2=32,
                block_size=16, seed=13)
    o1, l1 = O.reference(w)
    o2, l2 = O.reference_parallel(w, range(w.total_t), 2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
