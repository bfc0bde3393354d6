"""Helpers for the GPU parity tests: run the CUDA path, compare with the oracle.

Tolerances stated for the path: each bf16 output element within
1e-2 + 2e-2 * |ref| of the fp64 oracle, lse within 1e-3 absolute.
"""

from __future__ import annotations

import numpy as np
import torch

import compressed_mla_attention_gb300 as Q
import workloads as W
from oracle import qsfm_oracle as O

O_ATOL = 1e-2
O_RTOL = 2e-2
LSE_ATOL = 1e-3


def run_gpu(w, device, num_ctas: int = 0, lse: bool | None = None):
    """Forward on the GPU through the public API; returns CPU fp32 out / lse."""
    args = W.device_inputs(w, device)
    if lse is not None:
        args["return_softmax_lse"] = lse
    out, l = Q.quant_sparse_flash_mla(num_ctas=num_ctas, **args)
    torch.cuda.synchronize()
    assert Q.device_status() == 0
    out = out.float().cpu().reshape(w.total_t, int(w.q.shape[1]), 512).numpy()
    return out, (None if l is None else l.cpu().numpy())


def rounding_bounds(w, tokens, sigmas: float = 6.0):
    """Error bounds that follow from the kernel's bf16 operands.

    K~ = e4m3 * scale is rounded once to bf16 before the tensor-core
    products (relative error uniform in +-2^-9, independent per element), so
    a logit x_j = scale * q . k_j moves by a zero-mean error of standard
    deviation s_j = scale * 2^-9 / sqrt(3) * sqrt(sum_d q_d^2 k_jd^2).
    With dx = `sigmas` * max_j s_j:
      |d lse| <= dx,
      |d O_hd| <= 2 dx sum_j w_j |v_jd| + 2^-8 sum_j w_j |v_jd| + 2^-9 |O_hd|
    (softmax weight shift, bf16 V~ and P, bf16 output). Returns per-token
    arrays (lse_extra [n, N1], o_extra [n, N1, 512]) to add to the stated
    tolerances.
    """
    tb, tp = w.token_batch(), w.token_pos()
    sink = None if w.sinks is None else np.asarray(w.sinks, dtype=np.float64)
    nh = int(w.q.shape[1])
    lse_extra = np.zeros((len(tokens), nh))
    o_extra = np.zeros((len(tokens), nh, 512))
    for i, t in enumerate(tokens):
        k = O.token_kv(w, t, int(tb[t]), int(tp[t]))
        if k is None or k.shape[0] == 0:
            continue
        q = O.q_fp64(w, t)
        s = w.softmax_scale * 2.0 ** -9 / np.sqrt(3.0) * np.sqrt((q * q) @ (k * k).T)  # [N1, n]
        dx = sigmas * s.max(axis=1)
        x = w.softmax_scale * (q @ k.T)
        m = x.max(axis=1) if sink is None else np.maximum(x.max(axis=1), sink)
        e = np.exp(x - m[:, None])
        den = e.sum(axis=1) + (0.0 if sink is None else np.exp(sink - m))
        wv = (e / den[:, None]) @ np.abs(k)  # sum_j w_j |v_jd|
        o = (e / den[:, None]) @ k
        lse_extra[i] = dx
        o_extra[i] = (2 * dx[:, None] + 2.0 ** -8) * wv + 2.0 ** -9 * np.abs(o)
    return lse_extra, o_extra


def assert_parity(out, lse, w, tokens, o_ref=None, l_ref=None, lse_atol=LSE_ATOL, derived=False):
    """Element-wise check of sampled tokens against the oracle.

    derived=True adds the bf16-rounding bounds of rounding_bounds() to the
    stated tolerances (used for inputs outside the five workloads, e.g.
    tokens with a handful of rows or very peaked softmax).
    """
    tokens = list(tokens)
    if o_ref is None:
        o_ref, l_ref = O.reference(w, tokens)
    got = out[tokens]
    err = np.abs(got - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    lse_tol = np.full((len(tokens), o_ref.shape[1]), lse_atol)
    if derived:
        l_extra, o_extra = rounding_bounds(w, tokens)
        bound = bound + o_extra
        lse_tol = lse_tol + l_extra
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} outputs out of tolerance; first at token "
            f"{tokens[i[0]]} head {i[1]} d {i[2]}: got {got[tuple(i)]} ref {o_ref[tuple(i)]}; "
            f"max err {err.max():.3g}")
    if lse is not None:
        lg = lse[tokens]
        fin = np.isfinite(l_ref)
        assert np.array_equal(fin, np.isfinite(lg)), "lse finiteness differs"
        assert np.all(lg[~fin] == -np.inf)
        if fin.any():
            e = np.abs(lg[fin] - l_ref[fin])
            over = e > lse_tol[fin]
            assert not over.any(), f"lse: {int(over.sum())} over tolerance, max err {e.max():.3g}"
    return float(err.max())
