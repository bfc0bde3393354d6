"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each test swaps one step of ``oracle/qsfm_oracle.py`` for a plausible wrong
version (a dropped term, a wrong sign or bound, a transposed index, a
misread formula) and checks that at least one pin of ``tests/test_oracle.py``
fails under it. The mistakes are planted in the oracle module only, for the
duration of one test; the product path is not involved.
"""

import math

import numpy as np
import pytest

from oracle import qsfm_oracle as O
from tests import test_oracle as P

# pins that evaluate the oracle end to end on several inputs
BRUTE = [lambda i=i: P.test_oracle_matches_brute_force(i) for i in range(len(P.SMALL_CASES))]


def _fails(pins):
    """Names of the pins that fail (raise AssertionError) under the mutant."""
    failed = []
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed.append(getattr(pin, "__name__", "brute force"))
    return failed


def _attend_variant(sink_scaled=False, lse_with_sink=False, drop_sink_den=False, max_without_sink=False):
    def attend(q, k, softmax_scale, sinks):
        nh = q.shape[0]
        if k.shape[0] == 0:
            return np.zeros((nh, O.HEAD_DIM)), np.full(nh, -np.inf)
        x = softmax_scale * (q @ k.T)
        sink = np.full(nh, -np.inf) if sinks is None else np.asarray(sinks, dtype=np.float64)
        if sink_scaled:
            sink = sink * softmax_scale
        xmax = x.max(axis=1)
        m = xmax if max_without_sink else np.maximum(xmax, sink)
        e = np.exp(x - m[:, None])
        den = e.sum(axis=1) + (0.0 if drop_sink_den else np.exp(sink - m))
        o = (e @ k) / den[:, None]
        lse = xmax + np.log(np.exp(x - xmax[:, None]).sum(axis=1))
        if lse_with_sink:
            lse = np.logaddexp(lse, sink)
        return o, lse
    return attend


SINK_PINS = [P.test_sink_minus_inf_is_plain_softmax, P.test_single_key_sink_closed_form,
             P.test_zero_query_gives_sink_damped_mean, P.test_identical_rows_give_row_times_mass,
             P.test_lse_equals_torch_logsumexp_of_logits]


@pytest.mark.parametrize("mistake", ["sink_scaled", "lse_with_sink", "drop_sink_den"])
def test_sink_mistakes_are_caught(monkeypatch, mistake):
    monkeypatch.setattr(O, "attend", _attend_variant(**{mistake: True}))
    assert _fails(SINK_PINS + BRUTE)


def test_max_without_sink_is_harmless():
    """Leaving the sink out of the running max is not a mistake: it only
    shifts the exponents, so the result is the same (a reading check)."""
    rng = np.random.default_rng(4)
    q, k, sink = rng.standard_normal((64, 512)), rng.standard_normal((7, 512)), rng.standard_normal(64)
    a = O.attend(q, k, 0.05, sink)
    b = _attend_variant(max_without_sink=True)(q, k, 0.05, sink)
    assert np.allclose(a[0], b[0], rtol=1e-12) and np.allclose(a[1], b[1], rtol=1e-14)


def test_exclusive_band_bound_is_caught(monkeypatch):
    """Band rows p - wl + 1 .. p (an exclusive left bound)."""
    orig = O.ori_row_range

    def ori_row_range(p, s2, mode, wl, wr):
        lo, hi = orig(p, s2, mode, wl, wr)
        if mode == 4 and wl != -1 and hi >= lo:
            lo = max(lo, p - wl + 1)
        return (lo, hi) if hi >= lo else (0, -1)

    monkeypatch.setattr(O, "ori_row_range", ori_row_range)
    assert _fails([P.test_golden_ori_row_sets] + BRUTE)


def test_top_left_alignment_is_caught(monkeypatch):
    """Ori positions aligned top-left (p = s) instead of bottom-right."""
    orig = O.token_rows

    def token_rows(w, t, b, s):
        ori, cmp_rows = orig(w, t, b, s)
        if ori is None:
            return ori, cmp_rows
        lo, hi = O.ori_row_range(s, int(w.seqused_ori_kv[b]), w.ori_mask_mode, w.ori_win_left,
                                 w.ori_win_right)
        return list(range(lo, hi + 1)), cmp_rows

    monkeypatch.setattr(O, "token_rows", token_rows)
    assert _fails([P.test_golden_ori_row_sets] + BRUTE)


def test_cmp_visibility_off_by_one_is_caught(monkeypatch):
    """V = floor(p_c / r) instead of floor((p_c + 1) / r)."""
    def cmp_visible_count(p_c, cmp_len, ratio, mode):
        if mode == 0:
            return cmp_len
        return max(0, min(cmp_len, p_c // ratio))

    monkeypatch.setattr(O, "cmp_visible_count", cmp_visible_count)
    assert _fails([P.test_golden_cmp_visibility] + BRUTE)


def test_transposed_scale_index_is_caught(monkeypatch):
    """scale[j, d % 8] (tiled) instead of scale[j, d // 64] (repeated)."""
    def dequant_rows(kv_bytes, scales):
        vals = O.E4M3FN_TABLE[kv_bytes.astype(np.int64)]
        per_col = np.tile(scales.astype(np.float64), (1, O.TILE))
        return vals * per_col

    monkeypatch.setattr(O, "dequant_rows", dequant_rows)
    assert _fails([P.test_dequant_uses_tile_of_column] + BRUTE)


def test_subnormal_exponent_mistake_is_caught(monkeypatch):
    """e4m3fn subnormals as m/8 * 2^-7 instead of 2^-6."""
    table = O.E4M3FN_TABLE.copy()
    for c in range(256):
        if (c >> 3) & 0xF == 0:
            table[c] = table[c] / 2.0
    monkeypatch.setattr(O, "E4M3FN_TABLE", table)
    assert _fails([P.test_e4m3fn_all_codes_match_torch])


def test_swapped_sign_bit_is_caught(monkeypatch):
    """Sign taken from bit 6 instead of bit 7."""
    def decode(code):
        sign = -1.0 if (code >> 6) & 1 else 1.0
        exp, man = (code >> 3) & 0xF, code & 0x7
        if exp == 0xF and man == 0x7:
            return math.nan
        if exp == 0:
            return sign * (man / 8.0) * 2.0 ** -6
        return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)

    monkeypatch.setattr(O, "decode_e4m3fn_code", decode)
    monkeypatch.setattr(O, "E4M3FN_TABLE", np.array([decode(c) for c in range(256)]))
    assert _fails([P.test_e4m3fn_all_codes_match_torch, P.test_e4m3fn_golden_codes])


def test_dropped_invalid_index_filter_is_caught(monkeypatch):
    """Index entries beyond the visible range kept instead of dropped (CSA
    pins only: an unbounded visible count would make HCA rows endless)."""
    monkeypatch.setattr(O, "cmp_visible_count", lambda p_c, cmp_len, ratio, mode: 10 ** 9)
    assert _fails([P.test_invisible_indices_are_dropped])


def test_e8m0_bias_mistake_is_caught(monkeypatch):
    """e8m0 as 2^(e - 126) instead of 2^(e - 127)."""
    monkeypatch.setattr(O, "E8M0_TABLE", O.E8M0_TABLE * 2.0)
    assert _fails([P.test_e8m0_all_codes_match_torch, P.test_packed_row_by_hand])


def test_nope_before_rope_is_caught(monkeypatch):
    """The 512 elements of a packed row taken as nope then rope."""
    orig = O.dequant_packed_rows

    def dequant_packed_rows(rows):
        k = orig(rows)
        return np.concatenate([k[:, 64:], k[:, :64]], axis=1)

    monkeypatch.setattr(O, "dequant_packed_rows", dequant_packed_rows)
    assert _fails([P.test_packed_row_by_hand] + [lambda i=i: P.test_oracle_matches_brute_force_packed_rows(i)
                                                 for i in range(len(P.PACKED_CASES))])


def test_big_endian_bf16_is_caught(monkeypatch):
    """bf16 rows read with the two bytes of an element swapped."""
    def decode_bf16_rows(rows):
        rows = np.ascontiguousarray(rows)
        bits = rows.view(">u2").astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64).reshape(rows.shape[0], O.HEAD_DIM)

    monkeypatch.setattr(O, "decode_bf16_rows", decode_bf16_rows)
    assert _fails([P.test_bf16_row_by_hand] + [lambda i=i: P.test_oracle_matches_brute_force_bf16_rows(i)
                                               for i in range(len(P.BF16_CASES))])


def test_bf16_subnormal_flush_is_caught(monkeypatch):
    """bf16 subnormals (and -0.0) flushed to +0.0."""
    orig = O.decode_bf16_rows

    def decode_bf16_rows(rows):
        k = orig(rows)
        k[np.abs(k) < 2.0 ** -126] = 0.0
        return k

    monkeypatch.setattr(O, "decode_bf16_rows", decode_bf16_rows)
    assert _fails([P.test_bf16_all_bit_patterns_match_torch, P.test_bf16_row_by_hand])
