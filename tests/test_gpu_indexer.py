"""GPU parity of the lightning-indexer top-k (qsfm_lightning_indexer) with the
fp64 oracle (QuantLightningIndexerV2, formula and parameter table; quant
mode 1).

The kernel computes each score in fp32 (e4m3 products exact, fp32 sums on
the tensor cores and in the epilogue); the oracle in fp64. Where the scores
of the k-th and (k+1)-th key differ by more than twice the fp32 error bound
the selection is unique and the index row must match the oracle's bit for
bit; otherwise (a near tie at the boundary) the row must be a valid top-k
within that bound. sparse_values are checked against the oracle's scores
at bf16 rounding.
"""

import numpy as np
import pytest
import torch

import compressed_mla_attention_gb300 as Q
import workloads as W
from oracle import indexer_oracle as I
from oracle.qsfm_oracle import E4M3FN_TABLE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from compressed_mla_attention_gb300 import build

    build.build()
    Q.lib()


def run(w, device, return_value=True):
    a = W.indexer_device_inputs(w, device)
    idx, val = Q.lightning_indexer(a["query"], a["query_scale"], a["weights"], a["key"], a["key_scale"],
                                   a["block_table"], a["seqused_k"], layout=w.layout, batch=w.batch,
                                   cu_seqlens_q=a["cu_seqlens_q"], seqused_q=a["seqused_q"],
                                   cmp_residual_k=a["cmp_residual_k"], topk=w.topk, mask_mode=w.mask_mode,
                                   cmp_ratio=w.cmp_ratio, return_value=return_value, layout_k=w.layout_k,
                                   cu_seqlens_k=a["cu_seqlens_k"], output_idx_offset=a["output_idx_offset"])
    torch.cuda.synchronize()
    idx = idx.reshape(w.total_t, w.topk).cpu().numpy()
    val = None if val is None else val.reshape(w.total_t, w.topk).float().cpu().numpy()
    return idx, val


def fp32_bound(w, t):
    """An upper bound of the fp32 error of any score of token t: 2^-24 times
    (d + heads + 4) times the largest sum of absolute terms."""
    b, s = int(w.token_batch()[t]), int(w.token_pos()[t])
    v = I.visible_keys(w, b, s)
    if v == 0:
        return 0.0
    kb, sk = I.key_rows(w, b, v)
    k = E4M3FN_TABLE[np.asarray(kb).astype(np.int64)]
    q = E4M3FN_TABLE[w.query[t].numpy().astype(np.int64)]
    absum = (np.abs(w.weights[t].double().numpy()) * np.abs(w.query_scale[t].double().numpy())) @ (np.abs(q) @ np.abs(k).T)
    return float((absum * np.abs(sk)).max()) * 2.0 ** -24 * (q.shape[1] + q.shape[0] + 4)


def check(w, idx, val, tokens=None):
    tokens = range(w.total_t) if tokens is None else tokens
    ref_i, ref_v = I.reference(w, tokens)
    exact = same = 0
    for n, t in enumerate(tokens):
        got, want = idx[t], ref_i[n]
        same += int(np.array_equal(got, want))
        nv = int((want >= 0).sum())
        assert int((got >= 0).sum()) == nv, t
        assert np.all(got[nv:] == -1) and np.all(np.diff(got[:nv]) > 0), t  # ascending, then -1
        offs = getattr(w, "output_idx_offset", None)
        if offs is not None:  # compare key indices from here on
            shift = int(offs[int(w.token_batch()[t])])
            got = np.where(got >= 0, got - shift, got)
            want = np.where(want >= 0, want - shift, want)
        eps = fp32_bound(w, t)
        if I.boundary_gap(w, t) > 2 * eps:
            assert np.array_equal(got, want), t  # a unique selection: bit for bit
            exact += 1
        else:  # a near tie: every pick scores at least the k-th largest minus the bound
            sc = I.token_scores(w, t)
            kth = np.sort(sc)[::-1][nv - 1] if nv else 0.0
            assert np.all(got[:nv] < sc.size) and np.all(sc[got[:nv]] >= kth - 2 * eps), t
        if val is not None and nv:
            sc = I.token_scores(w, t)
            r = sc[got[:nv]]
            assert np.all(np.abs(val[t, :nv] - r) <= 2.0 ** -8 * np.abs(r) + 2 * eps + 1e-30), t
            assert np.all(np.isneginf(val[t, nv:])), t
    return exact, same


CASES = {
    "bsnd_causal": dict(layout="BSND", q_lens=[2, 2, 2], sk=[300, 900, 5000], topk=64, mask_mode=3, cmp_ratio=4),
    "tnd_mixed_heads8": dict(layout="TND", q_lens=[3, 1, 5], sk=[40, 700, 129], topk=50, mask_mode=3, cmp_ratio=3,
                             heads=8),
    "no_mask_fewer_keys_than_topk": dict(layout="BSND", q_lens=[1, 1, 1], sk=[10, 0, 130], topk=512, mask_mode=0,
                                         heads=16),
    "heads48_r128": dict(layout="TND", q_lens=[4, 2], sk=[256, 1077], topk=300, mask_mode=3, cmp_ratio=128,
                         heads=48),
    "padded_queries": dict(layout="BSND", q_lens=[3, 3], sk=[200, 500], topk=20, mask_mode=3, cmp_ratio=4,
                           seqused_q=[1, 3]),
    "tnd_padding": dict(layout="TND", q_lens=[4, 2, 5], sk=[1500, 90, 4000], topk=40, mask_mode=3, cmp_ratio=4,
                        seqused_q=[2, 2, 0], heads=32),
    "bsnd_keys_offsets": dict(layout="BSND", q_lens=[2, 2, 2], sk=[300, 2900, 5000], topk=64, mask_mode=3,
                              cmp_ratio=4, layout_k="BSND", output_idx_offset=[0, 300, 3200]),
    "tnd_keys": dict(layout="TND", q_lens=[3, 1, 5], sk=[1040, 700, 129], topk=50, mask_mode=3, cmp_ratio=3,
                     heads=8, layout_k="TND", output_idx_offset=[0, 1040, 1740]),
    "bsnd_keys_full_slabs": dict(layout="BSND", q_lens=[1, 1], sk=[700, 700], topk=100, mask_mode=0,
                                 layout_k="BSND", bsnd_seqused=False),
    "topk_8192_long": dict(layout="BSND", q_lens=[1, 1], sk=[30000, 9000], topk=8192, mask_mode=0, heads=64),
    # more query rows than the score kernel has threads (its start-up scan
    # then takes two tokens per thread), rows of four 64-head tokens (N = 256)
    "tnd_prefill_650": dict(layout="TND", q_lens=[250, 400], sk=[500, 1200], topk=48, mask_mode=3, cmp_ratio=4,
                            heads=64),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_indexer_parity(cuda_device, name):
    w = W.build_indexer(name, seed=len(name), **CASES[name])
    idx, val = run(w, cuda_device)
    assert Q.device_status() == 0
    check(w, idx, val)


def test_indexer_decode_batch_full_size(cuda_device):
    """The indexer call feeding the CSA decode batch (B = 128, S1 = 2, 64
    heads, up to 16K keys, top-512): 48 sampled tokens checked. The error
    bound is a worst case (every rounding in one direction), so few tokens
    qualify for the bit-for-bit comparison by it; the rows must still equal
    the oracle's on nearly all tokens (a difference is a swap of near-equal
    scores at the boundary, which the validity check covers)."""
    w = W.indexer_decode_batch()
    idx, _ = run(w, cuda_device, return_value=False)
    assert Q.device_status() == 0
    toks = W.subset_tokens(w, 48, seed=5).tolist() if hasattr(W, "subset_tokens") else list(range(48))
    exact, same = check(w, idx, None, toks)
    assert same >= 0.9 * len(toks)


def test_indexer_ties_take_the_smaller_key(cuda_device):
    """Zero weights: every score is 0, so the top-k is the k smallest
    visible keys."""
    w = W.build_indexer("ties", layout="BSND", q_lens=[2], sk=[1000], topk=100, mask_mode=3, seed=9)
    w.weights.zero_()
    idx, val = run(w, cuda_device)
    assert np.array_equal(idx, I.reference(w)[0])
    assert np.all(val[:, :100] == 0)


def test_indexer_bad_block_is_reported_not_read(cuda_device):
    w = W.build_indexer("bad", layout="BSND", q_lens=[1], sk=[400], topk=16, mask_mode=0, seed=10)
    w.block_table[0, 1] = int(w.key.shape[0]) + 7
    idx, _ = run(w, cuda_device, return_value=False)
    assert Q.device_status() & Q.FAULT_CMP_BLOCK_ID
    row = idx[0]
    assert np.all((row < 128) | (row >= 256))  # the bad block's keys are never picked


@pytest.mark.parametrize("sk,topk", [([6000, 2000], 300), ([700, 90], 64)])
def test_indexer_groups_of_equal_scores(cuda_device, sk, topk):
    """Every key is one of 16 distinct rows (same bytes, same scale), so each
    token's scores take at most 16 values and the k-th largest falls inside a
    group of equal scores: the smaller key indices of that group are taken.
    Large groups go through the full-depth radix and the tie bitmap, small
    ones through the ranked boundary list."""
    w = W.build_indexer("dups", layout="BSND", q_lens=[2, 2], sk=sk, topk=topk, mask_mode=3, cmp_ratio=4, seed=12)
    flat = w.key.reshape(-1, w.key.shape[-1])
    fs = w.key_scale.reshape(-1)
    src = torch.arange(flat.shape[0]) % 16
    flat.copy_(flat[src].clone())
    fs.copy_(fs[src].clone())
    idx, val = run(w, cuda_device)
    assert Q.device_status() == 0
    ref_i, _ = I.reference(w)
    assert np.array_equal(idx, ref_i)
    check(w, idx, val)


def test_indexer_keys_past_the_table_are_cut_and_flagged(cuda_device):
    """seqused_k larger than the block table holds: the row is cut to the
    table's keys (max_blocks * 128) and QSFM_FAULT_CMP_TABLE_COL is raised."""
    w = W.build_indexer("cut", layout="BSND", q_lens=[1], sk=[500], topk=16, mask_mode=0, seed=13)
    w.seqused_k[0] = 900  # the table holds 4 blocks = 512 keys
    idx, _ = run(w, cuda_device, return_value=False)
    assert Q.device_status() & Q.FAULT_CMP_TABLE_COL
    row = idx[0]
    assert np.all((row >= 0) & (row < 512))


@pytest.mark.parametrize("layout_k", ["BSND", "TND"])
def test_non_paged_keys_equal_paged_bitwise(cuda_device, layout_k):
    """The same logical keys as BSND slabs or TND rows give the paged
    layout's rows and values bit for bit (the scores of a key do not depend
    on where its row is stored)."""
    base = dict(layout="BSND", q_lens=[2, 2], sk=[1800, 4300], topk=256, mask_mode=3, cmp_ratio=4, seed=41)
    ref = run(W.build_indexer("paged", **base), cuda_device)
    got = run(W.build_indexer(layout_k, layout_k=layout_k, **base), cuda_device)
    assert Q.device_status() == 0
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
