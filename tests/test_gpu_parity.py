"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

The five spec workloads run at full size in the launch configuration
the bench uses; sampled tokens are compared element by element with the
oracle. Small edge cases are compared on every token. Row resolution is
checked bit-exactly through the exported debug gather.
"""

import zlib

import numpy as np
import pytest
import torch

import compressed_mla_attention_gb300 as Q
import workloads as W
from oracle import qsfm_oracle as O
from tests.harness import assert_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from compressed_mla_attention_gb300 import build

    build.build()
    Q.lib()


# ------------------------------------------------------- the five workloads
def _plan_starts(w, device, num_ctas=0):
    """First unit of every planned CTA (the plan the bench's launch uses)."""
    a = {k: v for k, v in W.device_inputs(w, device).items() if k != "return_softmax_lse"}
    plan = torch.empty(1024, dtype=torch.int32, device=device)
    p = Q.make_params(attn_out=torch.empty_like(a["q"]), metadata=plan, num_ctas=num_ctas, **a)
    Q.metadata(p, plan)
    m = plan.cpu().numpy()
    g = int(m[1])
    return [int(m[8 + 2 * c]) for c in range(g)]


def _config_tokens(i, w, device):
    """Tokens compared element by element with the oracle: every token of the
    decode workloads; for the prefill workloads, every batch's first and last
    token, every planned CTA's first and last token, and a seeded sample."""
    if i in (0, 2, 3):
        return list(range(w.total_t))
    ends = np.cumsum(w.q_lens)
    edges = [int(x) - 1 for x in ends] + [int(x) for x in ends[:-1]] + [0]
    starts = _plan_starts(w, device)
    cta_edges = starts + [s - 1 for s in starts if s > 0]
    if i == 1:  # early positions (short windows), a random sample, batch and CTA ends
        early = list(range(0, 160))
        return sorted(set(early + edges + cta_edges + W.subset_tokens(w, 96, seed=1).tolist()))
    # chunked prefill: 128 random tokens of each batch (1024 in all), plus the edges
    tb = w.token_batch()
    g = torch.Generator().manual_seed(4)
    strat = []
    for b in range(w.batch):
        idx = np.flatnonzero(tb == b)
        pick = torch.randperm(idx.size, generator=g)[:128].numpy()
        strat += idx[pick].tolist()
    return sorted(set(strat + edges + cta_edges))


@pytest.mark.parametrize("i", range(5))
def test_config_parity(cuda_device, i):
    w = W.config(i)
    out, lse = run_gpu(w, cuda_device, lse=True)
    toks = _config_tokens(i, w, cuda_device)
    assert np.isfinite(out).all()
    # Workload 1 returns no lse; its first tokens attend 1..127 rows, where the
    # lse carries the bf16 rounding of single logits, so its lse is held to
    # the derived bound. Every output element is held to the stated bound.
    if i == 1:
        assert_parity(out, lse, w, toks, derived=True)
        lse = None
    err = assert_parity(out, lse, w, toks)
    print(f"config {i}: {len(toks)} tokens checked, max |err| {err:.3g}")


@pytest.mark.parametrize("kv_format,n1", [("packed640", 64), ("bf16", 64), ("fp8_fp32_scales", 128)])
def test_config2_other_formats_full_size(cuda_device, kv_format, n1):
    """The CSA decode batch at full size with the other row formats and head
    count, in the launch configuration the bench times (default CTA count),
    on sampled tokens (every output element of each)."""
    w = W.config(2, kv_format=kv_format, n1=n1)
    out, lse = run_gpu(w, cuda_device, lse=True)
    assert np.isfinite(out).all()
    toks = W.subset_tokens(w, 24, seed=6).tolist()
    assert_parity(out, lse, w, toks)


def test_config2_all_ctas_variants(cuda_device):
    """The decode batch planned over fewer CTAs than SMs gives the same result."""
    w = W.config(2)
    toks = W.subset_tokens(w, 16, seed=5).tolist()
    o_ref, l_ref = O.reference(w, toks)
    for ctas in (1, 37, 152):
        out, lse = run_gpu(w, cuda_device, num_ctas=ctas, lse=True)
        assert_parity(out, lse, w, toks, o_ref, l_ref)


def test_plan_uses_fewest_ctas_with_same_tokens_per_cta(cuda_device):
    """256 equal-cost tokens on at most n CTAs: the plan keeps ceil(256 / n)
    tokens per CTA on the fewest CTAs that need (152 -> 128 CTAs of 2)."""
    w = W.build("equal tokens", layout="BSND", q_lens=[2] * 128, s2=[300] * 128, mode="SWA", seed=3)
    a = {k: v for k, v in W.device_inputs(w, cuda_device).items() if k != "return_softmax_lse"}
    plan = torch.empty(1024, dtype=torch.int32, device=cuda_device)
    for n, g in ((152, 128), (100, 86), (37, 37)):
        p = Q.make_params(attn_out=torch.empty_like(a["q"]), metadata=plan, num_ctas=n, **a)
        Q.metadata(p, plan)
        m = plan.cpu().numpy()
        assert m[1] == g
        starts = [int(m[8 + 2 * c]) for c in range(g + 1)]
        per = -(-256 // n)
        assert max(b - a_ for a_, b in zip(starts, starts[1:])) == per
        out, _ = run_gpu(w, cuda_device, num_ctas=n)
        assert_parity(out, None, w, range(0, w.total_t, 17))


# ----------------------------------------------------------- edge cases
EDGE = {
    "short_seq_decode": dict(layout="BSND", q_lens=[1, 1, 1], s2=[1, 50, 127], cmp_ratio=4, mode="CSA",
                             k2=64),
    "empty_kv_batch": dict(layout="BSND", q_lens=[2, 2], s2=[0, 300], cmp_ratio=4, mode="HCA"),
    "ragged_tnd_swa": dict(layout="TND", q_lens=[1, 129, 300, 7], s2=[1, 200, 300, 1000], mode="SWA"),
    "unbounded_causal_long": dict(layout="TND", q_lens=[5, 3], s2=[700, 260], mode="SWA",
                                  ori_mask_mode=3, ori_win_left=-1, ori_win_right=-1),
    "band_future_tokens": dict(layout="TND", q_lens=[40], s2=[300], mode="SWA", ori_win_left=20,
                               ori_win_right=9),
    "no_mask_hca": dict(layout="BSND", q_lens=[3, 3], s2=[400, 90], cmp_ratio=2, mode="HCA",
                        ori_mask_mode=0, ori_win_left=-1, ori_win_right=-1, cmp_mask_mode=0),
    "no_sinks_csa": dict(layout="BSND", q_lens=[2, 2], s2=[2000, 5000], cmp_ratio=4, mode="CSA",
                         k2=512, sinks=False),
    "topk_length": dict(layout="BSND", q_lens=[2, 2], s2=[900, 3000], cmp_ratio=4, mode="CSA", k2=256,
                        cmp_topk_length=[0, 1, 200, 256]),
    "padded_queries": dict(layout="BSND", q_lens=[4, 4], s2=[600, 700], cmp_ratio=4, mode="CSA", k2=128,
                           seqused_q=[1, 4]),
    "hca_r128_many_tiles": dict(layout="BSND", q_lens=[1, 1], s2=[131072, 40000], cmp_ratio=128,
                                mode="HCA"),
    "hca_r3_residual": dict(layout="TND", q_lens=[6, 9], s2=[500, 1001], cmp_ratio=3, mode="HCA"),
    "k2_1024": dict(layout="BSND", q_lens=[1], s2=[20000], cmp_ratio=4, mode="CSA", k2=1024),
    "large_logits": dict(layout="BSND", q_lens=[2], s2=[3000], cmp_ratio=4, mode="CSA", k2=512,
                         q_scale=12.0),
    # one token of 64 tiles: with the default CTA count it is split into more
    # than 32 parts, which the combine merges in groups of 32
    "one_token_many_parts": dict(layout="BSND", q_lens=[1], s2=[250000], cmp_ratio=64, mode="HCA"),
}


# the pages' other shapes: N1 = 128 heads (two 64-head units per token) and
# K2 = 1024 index entries
WIDE = {
    "n1_128_csa_decode": dict(layout="BSND", q_lens=[2] * 6, s2=[5000, 9000, 700, 20000, 4096, 3000],
                              cmp_ratio=4, mode="CSA", k2=512, n1=128),
    "n1_128_split": dict(layout="BSND", q_lens=[1], s2=[9000], cmp_ratio=4, mode="CSA", k2=512, n1=128),
    "n1_128_hca_tnd": dict(layout="TND", q_lens=[3, 5], s2=[3000, 40000], cmp_ratio=128, mode="HCA", n1=128),
    "k2_1024": dict(layout="BSND", q_lens=[2] * 4, s2=[8000, 30000, 5000, 12000], cmp_ratio=4, mode="CSA",
                    k2=1024),
    "n1_128_k2_1024": dict(layout="BSND", q_lens=[2, 2], s2=[20000, 9000], cmp_ratio=4, mode="CSA", k2=1024,
                           n1=128),
    # packed 640-byte KV rows (bf16 rope | e4m3fn nope | e8m0 scales)
    "packed_csa_decode": dict(layout="BSND", q_lens=[2] * 6, s2=[5000, 9000, 700, 20000, 4096, 3000],
                              cmp_ratio=4, mode="CSA", k2=512, kv_format="packed640"),
    "packed_hca_tnd": dict(layout="TND", q_lens=[3, 5], s2=[3000, 40000], cmp_ratio=128, mode="HCA",
                           kv_format="packed640"),
    "packed_split": dict(layout="BSND", q_lens=[1], s2=[9000], cmp_ratio=4, mode="CSA", k2=512,
                         kv_format="packed640"),
    "packed_n1_128_swa": dict(layout="TND", q_lens=[40, 9], s2=[300, 9], mode="SWA", n1=128,
                              kv_format="packed640"),
    # unquantised bf16 KV rows (SparseCompressedFlashAttention: TND, K2 = 512,
    # window 128, cmp_ratio 4)
    "bf16_csa_tnd": dict(layout="TND", q_lens=[3, 1, 4, 2], s2=[5000, 700, 20000, 130], cmp_ratio=4,
                         mode="CSA", k2=512, kv_format="bf16"),
    "bf16_split": dict(layout="TND", q_lens=[1], s2=[9000], cmp_ratio=4, mode="CSA", k2=512,
                       kv_format="bf16"),
    "bf16_n1_128_hca": dict(layout="TND", q_lens=[3, 5], s2=[3000, 40000], cmp_ratio=128, mode="HCA",
                            n1=128, kv_format="bf16"),
}


@pytest.mark.parametrize("name", sorted(WIDE))
@pytest.mark.parametrize("ctas", [0, 5])
def test_wide_shape_parity(cuda_device, name, ctas):
    w = W.build(name, seed=zlib.crc32(name.encode()) % 1000, return_lse=True, **WIDE[name])
    out, lse = run_gpu(w, cuda_device, num_ctas=ctas)
    assert out.shape[1] == w.q.shape[1]
    assert_parity(out, lse, w, range(w.total_t))


# KV storage layouts and ori picks (QuantSparseFlashMla parameter table rows
# layout_kv, cu_seqlens_ori_kv / cu_seqlens_cmp_kv, ori_sparse_indices,
# ori_topk_length; its constraints on the BSND / TND KV layouts)
LAYOUTS = {
    "bsnd_kv_csa_decode_picks": dict(layout="BSND", q_lens=[2] * 8,
                                     s2=[5000, 9000, 700, 20000, 4096, 3000, 130, 12000], cmp_ratio=4,
                                     mode="CSA", k2=512, layout_kv="BSND", ori_k1=128),
    "tnd_kv_csa_prefill_picks_topk": dict(layout="TND", q_lens=[40, 7, 100], s2=[3000, 900, 8000], cmp_ratio=4,
                                          mode="CSA", k2=512, layout_kv="TND", kv_pad=33, ori_k1=256,
                                          ori_mask_mode=3, ori_win_left=-1, ori_win_right=-1,
                                          ori_topk_length=[(37 * i) % 300 for i in range(147)]),
    "tnd_kv_hca_packed": dict(layout="TND", q_lens=[3, 5], s2=[3000, 40000], cmp_ratio=64, mode="HCA",
                              layout_kv="TND", kv_format="packed640"),
    "bsnd_kv_swa_no_seqused": dict(layout="BSND", q_lens=[3, 3], s2=[500, 500], mode="SWA", layout_kv="BSND",
                                   bsnd_seqused=False, ori_win_left=200, ori_win_right=3),
    "paged_picks_no_mask": dict(layout="BSND", q_lens=[2, 2, 2], s2=[9000, 300, 20000], cmp_ratio=4, mode="CSA",
                                k2=512, ori_k1=512, ori_n_valid=480, ori_mask_mode=0, ori_win_left=-1,
                                ori_win_right=-1),
    "bsnd_kv_bf16_picks_n1_128": dict(layout="BSND", q_lens=[2, 2], s2=[6000, 2500], cmp_ratio=4, mode="CSA",
                                      k2=512, layout_kv="BSND", kv_format="bf16", ori_k1=64, n1=128),
    "tnd_kv_swa_picks_none_valid": dict(layout="TND", q_lens=[5, 9], s2=[64, 900], mode="SWA",
                                        layout_kv="TND", ori_k1=32, ori_n_valid=0),
}


@pytest.mark.parametrize("name", sorted(LAYOUTS))
@pytest.mark.parametrize("ctas", [0, 5])
def test_kv_layout_and_ori_picks_parity(cuda_device, name, ctas):
    w = W.build(name, seed=zlib.crc32(name.encode()) % 1000, return_lse=True, **LAYOUTS[name])
    out, lse = run_gpu(w, cuda_device, num_ctas=ctas)
    assert_parity(out, lse, w, range(w.total_t), derived=True)


def test_non_paged_kv_equals_paged_bitwise(cuda_device):
    """The same logical rows stored BSND and paged give the same bits: the
    storage only changes where a row is read from."""
    from tests.test_oracle_ori_sparse_layouts import _paged_copy

    w = W.build("same rows", layout="BSND", q_lens=[2] * 4, s2=[5000, 900, 12000, 3000], cmp_ratio=4,
                mode="CSA", k2=512, layout_kv="BSND", ori_k1=100, seed=51, return_lse=True)
    pa = _paged_copy(w, block=128, seed=2)
    out1, lse1 = run_gpu(w, cuda_device)
    out2, lse2 = run_gpu(pa, cuda_device)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_sparse_compressed_flash_attention_entry(cuda_device):
    """The bf16-KV entry point with SparseCompressedFlashAttention's argument
    layout (flat query and KV, q_act_seqs without the leading zero, win_size)
    matches the oracle and gives the same bits as the general entry point."""
    w = W.build("scfa", layout="TND", q_lens=[3, 1, 4], s2=[5000, 700, 20000], cmp_ratio=4, mode="CSA",
                k2=512, kv_format="bf16", with_residual=False, seed=41)
    a = W.device_inputs(w, cuda_device)
    T = w.total_t
    out = Q.sparse_compressed_flash_attention(
        a["q"].reshape(T * 64, 512), a["cu_seqlens_q"][1:].contiguous(), a["ori_kv"].reshape(-1, 512),
        a["cmp_kv"].reshape(-1, 512), a["ori_block_table"], a["cmp_block_table"], a["sinks"],
        a["seqused_ori_kv"], a["cmp_sparse_indices"].reshape(T, 512), w.softmax_scale,
        win_size=128, cmp_ratio=4)
    torch.cuda.synchronize()
    assert Q.device_status() == 0
    assert out.shape == (T * 64, 512)
    got = out.float().cpu().reshape(T, 64, 512).numpy()
    general, _ = run_gpu(w, cuda_device)
    assert np.array_equal(got, general)
    assert_parity(got, None, w, range(T))


@pytest.mark.parametrize("name", sorted(EDGE))
@pytest.mark.parametrize("ctas", [0, 3])
def test_edge_case_parity(cuda_device, name, ctas):
    w = W.build(name, seed=zlib.crc32(name.encode()) % 1000, return_lse=True, **EDGE[name])
    out, lse = run_gpu(w, cuda_device, num_ctas=ctas)
    assert_parity(out, lse, w, range(w.total_t), derived=True)


def test_duplicate_and_invalid_indices(cuda_device):
    w = W.build("dup", layout="BSND", q_lens=[2], s2=[4096], cmp_ratio=4, mode="CSA", k2=512, seed=3,
                return_lse=True)
    idx = w.cmp_sparse_indices
    idx[0, 0, 100:200] = idx[0, 0, 0:100]            # duplicates count twice
    idx[0, 0, 200:260] = -1                          # -1 in the middle
    idx[1, 0, 0:10] = torch.tensor([-7, 1024, 5000, 2**30, -2**31, 3, 3, 3, 1023, 0],
                                   dtype=torch.int32)  # out of range entries are ignored
    out, lse = run_gpu(w, cuda_device)
    assert_parity(out, lse, w, range(2))


def test_all_invalid_equals_swa_bitwise(cuda_device):
    w = W.build("neg", layout="BSND", q_lens=[2, 2], s2=[3000, 700], cmp_ratio=4, mode="CSA", k2=512,
                seed=9, return_lse=True)
    w.cmp_sparse_indices.fill_(-1)
    # 2 CTAs for 4 tokens: tokens are never split, so both runs take the same path
    out_csa, lse_csa = run_gpu(w, cuda_device, num_ctas=2)
    w.cmp_kv = w.cmp_scale = w.cmp_block_table = w.cmp_sparse_indices = None
    w.cmp_ratio, w.cmp_residual_kv = 1, None
    out_swa, lse_swa = run_gpu(w, cuda_device, num_ctas=2)
    assert np.array_equal(out_csa, out_swa) and np.array_equal(lse_csa, lse_swa)


def test_index_permutation_invariance(cuda_device):
    w = W.build("perm", layout="BSND", q_lens=[2, 2], s2=[5000, 9000], cmp_ratio=4, mode="CSA",
                k2=512, n_valid=400, seed=4, return_lse=True)
    out1, lse1 = run_gpu(w, cuda_device)
    g = torch.Generator().manual_seed(1)
    for t in range(w.total_t):
        w.cmp_sparse_indices[t, 0] = w.cmp_sparse_indices[t, 0, torch.randperm(512, generator=g)]
    out2, lse2 = run_gpu(w, cuda_device)
    assert np.abs(out1 - out2).max() <= 2e-3
    assert np.abs(lse1 - lse2).max() <= 1e-4
    assert_parity(out2, lse2, w, range(w.total_t))


# ------------------------------------------------------ row resolution
def _storage_row(w, kv, b, e, table, cu):
    """Row e of batch b in a KV tensor of any storage layout, found here from
    the layout's definition: paged [blocks, 128, ...] through the block
    table, BSND [B, S, 1, ...] at [b, e], TND [T, 1, ...] at cu[b] + e."""
    lay = getattr(w, "layout_kv", "PA_BBND")
    if lay == "BSND":
        return kv[b, e].reshape(-1)
    if lay == "TND":
        return kv[int(cu[b]) + e].reshape(-1)
    return kv[table[e // 128], e % 128].reshape(-1)


def _raw(kv):
    """KV tensor as raw row bytes keeping its leading axes (bf16 -> 2 bytes per element)."""
    if kv.dtype == torch.bfloat16:
        kv = kv.contiguous().view(torch.uint8)
    return kv.numpy()


def _expected_slots(w, t, with_bytes=True):
    """(row ids, row bytes, scales) of token t's slots in the kernel's order
    (ori slots, then cmp slots), resolved in Python from the token's mask
    ranges, its index rows and the KV storage (with_bytes=False: ids only).
    A slot that attends nothing has id -1 and zero bytes. Scales are
    separate only for fp8 rows (else None)."""
    b, s = int(w.token_batch()[t]), int(w.token_pos()[t])
    fp8 = w.ori_scale is not None
    ids, rows_b, rows_s = [], [], []
    if w.seqused_q is not None and s >= int(w.seqused_q[b]):
        return ids, rows_b, (rows_s if fp8 else None)
    s1, s2 = int(w.q_lens[b]), O.ori_length(w, b)
    lo, hi = O.ori_row_range(s2 - s1 + s, s2, w.ori_mask_mode, w.ori_win_left, w.ori_win_right)
    if w.ori_sparse_indices is None:
        ori_ids = list(range(lo, hi + 1))
    else:
        n = w.k1 if w.ori_topk_length is None else max(0, min(w.k1, int(w.ori_topk_length[t])))
        ori_ids = [e if (e != -1 and lo <= e <= hi) else -1 for e in w.ori_sparse_indices[t, 0, :n].tolist()]
    slots = [(0, e) for e in ori_ids]
    if w.cmp_kv is not None:
        cmp_len = O.cmp_length(w, b, s2)
        res = int(w.cmp_residual_kv[b]) if w.cmp_residual_kv is not None else 0
        v = O.cmp_visible_count(cmp_len * w.cmp_ratio + res - s1 + s, cmp_len, w.cmp_ratio,
                                w.cmp_mask_mode)
        entries = (w.cmp_sparse_indices[t, 0].tolist() if w.cmp_sparse_indices is not None
                   else list(range(v)))
        if w.cmp_topk_length is not None:
            entries = entries[:int(w.cmp_topk_length[t])]
        slots += [(1, e if 0 <= e < v else -1) for e in entries]
    if with_bytes:
        kvs = {0: _raw(w.ori_kv), 1: None if w.cmp_kv is None else _raw(w.cmp_kv)}
        scs = {0: w.ori_scale.numpy() if fp8 else None, 1: w.cmp_scale.numpy() if fp8 and w.cmp_kv is not None else None}
        tabs = {0: None if w.ori_block_table is None else w.ori_block_table[b].numpy(),
                1: None if w.cmp_block_table is None else w.cmp_block_table[b].numpy()}
        cus = {0: w.cu_seqlens_ori_kv, 1: w.cu_seqlens_cmp_kv}
    for src, e in slots:
        ids.append(-1 if e < 0 else (src << 30) | e)
        if with_bytes:
            width = kvs[src].shape[-1]
            rows_b.append(np.zeros(width, np.uint8) if e < 0 else
                          _storage_row(w, kvs[src], b, e, tabs[src], cus[src]))
            if fp8:
                rows_s.append(np.zeros(8, np.float32) if e < 0 else
                              _storage_row(w, scs[src], b, e, tabs[src], cus[src]))
    return ids, rows_b, (rows_s if fp8 else None)


GATHER_CASES = {
    "tiny_csa_decode": lambda: W.config(0),
    "csa_decode_batch": lambda: W.config(2),
    "csa_decode_batch_n1_128": lambda: W.config(2, n1=128),
    "hca_long_decode": lambda: W.config(3),
    "csa_chunked_prefill": lambda: W.config(4),
    "k2_1024": lambda: W.build("k2 1024", layout="BSND", q_lens=[2] * 4, s2=[8000, 30000, 5000, 12000],
                               cmp_ratio=4, mode="CSA", k2=1024, seed=7),
    "tiny_csa_decode_packed": lambda: W.config(0, kv_format="packed640"),
    "csa_decode_batch_packed": lambda: W.config(2, kv_format="packed640"),
    "hca_long_decode_bf16": lambda: W.config(3, kv_format="bf16"),
    "csa_chunked_prefill_bf16": lambda: W.config(4, kv_format="bf16"),
    "hca_tnd_packed": lambda: W.build("hca tnd", layout="TND", q_lens=[3, 5], s2=[3000, 40000], cmp_ratio=128,
                                      mode="HCA", kv_format="packed640", seed=5),
    "k2_1024_bf16": lambda: W.build("k2 1024 bf16", layout="BSND", q_lens=[2] * 2, s2=[30000, 9000],
                                    cmp_ratio=4, mode="CSA", k2=1024, kv_format="bf16", seed=8),
    # non-paged KV and ori picks
    "bsnd_kv_csa_ori_picks": lambda: W.build("bsnd kv picks", **LAYOUTS["bsnd_kv_csa_decode_picks"], seed=9),
    "tnd_kv_prefill_picks_topk": lambda: W.build("tnd kv picks", **LAYOUTS["tnd_kv_csa_prefill_picks_topk"],
                                                 seed=10),
    "tnd_kv_hca_packed": lambda: W.build("tnd kv hca packed", **LAYOUTS["tnd_kv_hca_packed"], seed=11),
    "paged_picks_mode0": lambda: W.build("paged picks", **LAYOUTS["paged_picks_no_mask"], seed=12),
}


@pytest.mark.parametrize("case", sorted(GATHER_CASES))
def test_debug_gather_bit_exact(cuda_device, case):
    """The row resolution of the attention kernel (the same device function
    its resolver warp runs, with the same lane mapping) exported for sampled
    tokens: logical row ids, the bytes of each resolved row in the pool's own
    format and, for fp8 rows, the scale row, all bit for bit against a Python
    gather through the block tables."""
    w = GATHER_CASES[case]()
    toks = W.subset_tokens(w, 12, seed=len(case)).tolist()
    args = W.device_inputs(w, cuda_device)
    out = torch.empty_like(args["q"])
    p = Q.make_params(attn_out=out, **{k: v for k, v in args.items() if k != "return_softmax_lse"})
    fp8 = w.ori_scale is not None
    row_bytes = _raw(w.ori_kv).shape[-1]
    max_rows = 1280
    n = len(toks)
    tok = torch.tensor(toks, dtype=torch.int32, device=cuda_device)
    rows = torch.empty(n, max_rows, row_bytes, dtype=torch.uint8, device=cuda_device)
    scales = torch.empty(n, max_rows, 8, dtype=torch.float32, device=cuda_device) if fp8 else None
    ids = torch.empty(n, max_rows, dtype=torch.int32, device=cuda_device)
    counts = torch.empty(n, dtype=torch.int32, device=cuda_device)
    Q.debug_gather(p, tok, max_rows, rows, scales, ids, counts)
    torch.cuda.synchronize()
    assert Q.device_status() == 0
    rows, ids, counts = rows.cpu().numpy(), ids.cpu().numpy(), counts.cpu().numpy()
    if fp8:
        scales = scales.cpu().numpy()
    for j, t in enumerate(toks):
        e_ids, e_b, e_s = _expected_slots(w, t)
        assert counts[j] == len(e_ids)
        m = min(len(e_ids), max_rows)
        assert np.array_equal(ids[j, :m], np.array(e_ids[:m], dtype=np.int32))
        assert np.array_equal(rows[j, :m], np.stack(e_b[:m]))
        if fp8:
            assert np.array_equal(scales[j, :m].view(np.uint32), np.stack(e_s[:m]).view(np.uint32))


def test_debug_gather_row_ids_only(cuda_device):
    """Row ids and counts alone (no row bytes), as the bench counts rows."""
    w = W.config(4, kv_format="packed640")
    toks = W.subset_tokens(w, 12, seed=3).tolist()
    args = W.device_inputs(w, cuda_device)
    out = torch.empty_like(args["q"])
    p = Q.make_params(attn_out=out, **{k: v for k, v in args.items() if k != "return_softmax_lse"})
    max_rows = 1280
    n = len(toks)
    tok = torch.tensor(toks, dtype=torch.int32, device=cuda_device)
    ids = torch.empty(n, max_rows, dtype=torch.int32, device=cuda_device)
    counts = torch.empty(n, dtype=torch.int32, device=cuda_device)
    Q.debug_gather(p, tok, max_rows, None, None, ids, counts)
    torch.cuda.synchronize()
    assert Q.device_status() == 0
    ids, counts = ids.cpu().numpy(), counts.cpu().numpy()
    for j, t in enumerate(toks):
        e_ids, _, _ = _expected_slots(w, t, with_bytes=False)
        assert counts[j] == len(e_ids)
        m = min(len(e_ids), max_rows)
        assert np.array_equal(ids[j, :m], np.array(e_ids[:m], dtype=np.int32))


# --------------------------------------------------------- fault reporting
def test_bad_block_id_is_reported_not_read(cuda_device):
    w = W.build("bad", layout="BSND", q_lens=[1, 1], s2=[500, 500], mode="SWA", seed=2)
    b0_last = (500 - 1) // 128
    w.ori_block_table[1, b0_last] = 10 ** 6  # outside the pool
    args = W.device_inputs(w, cuda_device)
    out, _ = Q.quant_sparse_flash_mla(num_ctas=4, **args)
    torch.cuda.synchronize()
    fault = Q.device_status()
    assert fault & Q.FAULT_ORI_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    assert Q.device_status() == 0  # reading clears the word


def test_bounded_wait_runs_out_without_faulting(cuda_device):
    """A wait on a barrier nothing arrives on ends at its limit with the
    timeout bit set, a second wait ends on the abort flag, and the device
    keeps working."""
    Q.device_status()  # clear
    elapsed = torch.zeros(2, dtype=torch.int64, device=cuda_device)
    Q.debug_bounded_wait(2_000_000, elapsed)  # 2 ms
    torch.cuda.synchronize()
    assert Q.device_status() & Q.FAULT_TIMEOUT
    first, second = elapsed.cpu().tolist()
    assert 2_000_000 <= first < 200_000_000
    assert first <= second < first + 1_000_000  # well before its own 2 s limit
    w = W.build("after timeout", layout="BSND", q_lens=[1] * 3, s2=[300, 700, 1200], cmp_ratio=4,
                mode="CSA", k2=64, seed=11)
    out, lse = run_gpu(w, cuda_device)
    assert_parity(out, lse, w, range(w.total_t), derived=True)
    assert Q.device_status() == 0


def test_stale_metadata_is_rejected(cuda_device):
    """A plan made for other lengths is detected; nothing is written."""
    w1 = W.build("m1", layout="BSND", q_lens=[1] * 4, s2=[300] * 4, mode="SWA", seed=1)
    w2 = W.build("m2", layout="BSND", q_lens=[1] * 6, s2=[300] * 6, mode="SWA", seed=1)
    a1, a2 = W.device_inputs(w1, cuda_device), W.device_inputs(w2, cuda_device)
    plan = torch.empty(1024, dtype=torch.int32, device=cuda_device)
    p1 = Q.make_params(attn_out=torch.empty_like(a1["q"]), metadata=plan, num_ctas=8,
                       **{k: v for k, v in a1.items() if k != "return_softmax_lse"})
    Q.metadata(p1, plan)
    out = torch.zeros_like(a2["q"])
    p2 = Q.make_params(attn_out=out, metadata=plan, num_ctas=8,
                       **{k: v for k, v in a2.items() if k != "return_softmax_lse"})
    ws = torch.empty(max(Q.workspace_size(p2), 1), dtype=torch.uint8, device=cuda_device)
    Q.forward(p2, ws)
    torch.cuda.synchronize()
    assert Q.device_status() & Q.FAULT_METADATA
    assert (out.float() == 0).all()


def test_plan_for_more_ctas_than_the_call_is_refused(cuda_device):
    """A split plan made for 24 CTAs, reused by a forward call planned over 8
    (whose workspace holds 8 CTAs' partial results): both kernels see the
    mismatch, set the metadata fault bit and write nothing."""
    w = W.config(0)
    a = {k: v for k, v in W.device_inputs(w, cuda_device).items() if k != "return_softmax_lse"}
    plan = torch.empty(1024, dtype=torch.int32, device=cuda_device)
    big = Q.make_params(attn_out=torch.empty_like(a["q"]), metadata=plan, num_ctas=24, **a)
    Q.metadata(big, plan)
    assert int(plan[1].item()) > 8  # split over more CTAs than the call below plans
    out = torch.zeros_like(a["q"])
    small = Q.make_params(attn_out=out, metadata=plan, num_ctas=8, **a)
    ws = torch.empty(Q.workspace_size(small), dtype=torch.uint8, device=cuda_device)
    assert 0 < ws.numel() < Q.workspace_size(big)
    Q.forward(small, ws)
    torch.cuda.synchronize()
    assert Q.device_status() & Q.FAULT_METADATA
    assert (out.float() == 0).all()
