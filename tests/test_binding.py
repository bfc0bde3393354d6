"""Argument marshalling of the Python entry points (CPU only, no kernel runs).

The page-named wrappers must hand the C-ABI path exactly the tensors and
attribute values their parameter tables define. The compute call is
replaced by a recorder, so nothing here touches a GPU.
"""

import pytest
import torch

import compressed_mla_attention_gb300 as Q


def _record(monkeypatch):
    seen = {}

    def fake(q, ori_kv, ori_scale, ori_block_table, seqused_ori_kv, **kw):
        seen.update(q=q, ori_kv=ori_kv, ori_scale=ori_scale, ori_block_table=ori_block_table,
                    seqused_ori_kv=seqused_ori_kv, **kw)
        return torch.zeros_like(q), None

    monkeypatch.setattr(Q, "quant_sparse_flash_mla", fake)
    return seen


def test_sparse_compressed_flash_attention_marshalling(monkeypatch):
    """SparseCompressedFlashAttention parameter table: query [T1 * N1, D],
    q_act_seqs = running token totals, PA_ND KV [block_num * 128, D],
    cmp_sparse_indices [T1, K2], win_size and cmp_ratio."""
    seen = _record(monkeypatch)
    t1, n1, k2 = 7, 64, 512
    query = torch.randn(t1 * n1, 512).to(torch.bfloat16)
    q_act = torch.tensor([3, 7], dtype=torch.int32)
    ori = torch.zeros(3 * 128, 512, dtype=torch.bfloat16)
    cmp_ = torch.zeros(2 * 128, 512, dtype=torch.bfloat16)
    ot, ct = torch.zeros(2, 2, dtype=torch.int32), torch.zeros(2, 1, dtype=torch.int32)
    sink = torch.randn(n1)
    used = torch.tensor([200, 50], dtype=torch.int32)
    idx = torch.randint(-1, 40, (t1, k2), dtype=torch.int32)
    out = Q.sparse_compressed_flash_attention(query, q_act, ori, cmp_, ot, ct, sink, used, idx,
                                              softmax_scale=0.04, win_size=128, cmp_ratio=4)
    assert out.shape == (t1 * n1, 512)
    assert seen["layout"] == "TND"
    assert seen["q"].shape == (t1, n1, 512) and seen["q"].data_ptr() == query.data_ptr()
    assert torch.equal(seen["cu_seqlens_q"], torch.tensor([0, 3, 7], dtype=torch.int32))
    assert seen["ori_kv"].shape == (3, 128, 1, 512) and seen["ori_kv"].data_ptr() == ori.data_ptr()
    assert seen["cmp_kv"].shape == (2, 128, 1, 512) and seen["cmp_kv"].data_ptr() == cmp_.data_ptr()
    assert seen["ori_scale"] is None and seen.get("cmp_scale") is None
    assert seen["cmp_sparse_indices"].shape == (t1, 1, k2)
    assert torch.equal(seen["cmp_sparse_indices"].reshape(t1, k2), idx)
    assert seen["sinks"] is sink and seen["seqused_ori_kv"] is used
    assert seen["ori_block_table"] is ot and seen["cmp_block_table"] is ct
    # a window of 128 tokens ending at the query: 127 before it, none after
    assert (seen["ori_mask_mode"], seen["ori_win_left"], seen["ori_win_right"]) == (4, 127, 0)
    assert seen["cmp_mask_mode"] == 3 and seen["cmp_ratio"] == 4 and seen["softmax_scale"] == 0.04
    assert seen.get("cmp_residual_kv") is None and seen.get("seqused_cmp_kv") is None


def test_sparse_compressed_flash_attention_rejects_bad_shapes(monkeypatch):
    _record(monkeypatch)
    sink = torch.zeros(64)
    kv = torch.zeros(128, 512, dtype=torch.bfloat16)
    tab = torch.zeros(1, 1, dtype=torch.int32)
    q_act = torch.tensor([1], dtype=torch.int32)
    used = torch.tensor([5], dtype=torch.int32)
    idx = torch.zeros(1, 512, dtype=torch.int32)
    with pytest.raises(ValueError):  # T1 * N1 rows needed
        Q.sparse_compressed_flash_attention(torch.zeros(65, 512, dtype=torch.bfloat16), q_act, kv, kv,
                                            tab, tab, sink, used, idx, 0.04)
    with pytest.raises(ValueError):  # whole 128-row blocks needed
        Q.sparse_compressed_flash_attention(torch.zeros(64, 512, dtype=torch.bfloat16), q_act,
                                            torch.zeros(100, 512, dtype=torch.bfloat16), kv, tab, tab,
                                            sink, used, idx, 0.04)
    with pytest.raises(ValueError):
        Q.sparse_compressed_flash_attention(torch.zeros(64, 512, dtype=torch.bfloat16), q_act, kv, kv,
                                            tab, tab, sink, used, idx, 0.04, win_size=0)
