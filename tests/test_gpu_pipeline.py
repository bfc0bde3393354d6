"""The CSA decode step with its index rows made on the device: the lightning
indexer's output (QuantLightningIndexerV2's sparse_indices) is passed as the
attention's cmp_sparse_indices (QuantSparseFlashMla / KvQuantSparseAttnSharedKv
parameter tables) without a trip through the host, and each stage is
checked against its own oracle: the index rows against the indexer oracle,
the attention output against the attention oracle fed the same rows.
"""

import dataclasses

import numpy as np
import pytest
import torch

import compressed_mla_attention_gb300 as Q
import workloads as W
from tests.harness import assert_parity
from tests.test_gpu_indexer import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from compressed_mla_attention_gb300 import build

    build.build()
    Q.lib()


def indexer_rows(wi, dev):
    a = W.indexer_device_inputs(wi, dev)
    idx, _ = Q.lightning_indexer(a["query"], a["query_scale"], a["weights"], a["key"], a["key_scale"],
                                 a["block_table"], a["seqused_k"], layout=wi.layout, batch=wi.batch,
                                 cu_seqlens_q=a["cu_seqlens_q"], seqused_q=a["seqused_q"],
                                 cmp_residual_k=a["cmp_residual_k"], topk=wi.topk, mask_mode=wi.mask_mode,
                                 cmp_ratio=wi.cmp_ratio)
    return idx


CASES = {
    "bsnd decode": dict(layout="BSND", q_lens=[2, 2, 2], s2=[5000, 9000, 4100]),
    "tnd chunks": dict(layout="TND", q_lens=[3, 1, 4], s2=[6000, 2500, 12000]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_indexer_rows_drive_the_attention(cuda_device, name):
    wa = W.build(f"pipeline {name}", cmp_ratio=4, mode="CSA", k2=512, seed=31, **CASES[name])
    wi = W.indexer_for(wa, seed=32)
    idx = indexer_rows(wi, cuda_device)  # [T, 1, 512] int32, on the device
    args = W.device_inputs(wa, cuda_device)
    args["cmp_sparse_indices"] = idx
    out, lse = Q.quant_sparse_flash_mla(**dict(args, return_softmax_lse=True))
    torch.cuda.synchronize()
    assert Q.device_status() == 0
    rows = idx.reshape(wi.total_t, wi.topk).cpu().numpy()
    check(wi, rows, None)  # stage 1: the indexer against its oracle
    w2 = dataclasses.replace(wa, cmp_sparse_indices=torch.from_numpy(rows.copy()).reshape(wa.total_t, 1, wi.topk))
    got = out.float().cpu().reshape(wa.total_t, 64, 512).numpy()
    assert_parity(got, lse.cpu().numpy(), w2, range(wa.total_t))  # stage 2: the attention on those rows
