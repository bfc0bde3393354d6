"""qsfm_forward_noalloc(): the forward pass for callers that cannot allocate.

Some callers cannot call cudaMalloc (a framework that owns the device memory
pool, a plugin host, a serving loop that forbids allocation). The entry
point takes its split-KV scratch from a fixed array the library reserves on
the device. These tests call it through the C ABI, twice in a row on
different inputs, with a plan that splits tokens over CTAs (so the scratch is
really used), and compare each result with qsfm_forward() run with a
torch-allocated workspace, within the tolerances of the other GPU tests.
This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import compressed_mla_attention_gb300 as Q
import workloads as W

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 1e-2, 2e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from compressed_mla_attention_gb300 import build

    build.build()
    Q.lib()


def _params(w, dev, num_ctas):
    a = W.device_inputs(w, dev)
    a.pop("return_softmax_lse")
    out = torch.full_like(a["q"], float("nan"))
    lse = torch.full((w.total_t, w.n1), float("nan"), dtype=torch.float32, device=dev)
    plan = torch.empty(1024, dtype=torch.int32, device=dev)
    p = Q.make_params(attn_out=out, softmax_lse=lse, metadata=plan, return_lse=True,
                      num_ctas=num_ctas, **a)
    Q.metadata(p, plan)
    # p holds raw device pointers: keep every tensor it points to alive
    return p, out, lse, (a, plan)


def _existing(p, out, lse):
    """Result of the existing entry point, qsfm_forward(), with a workspace."""
    ws = torch.empty(max(Q.workspace_size(p), 1), dtype=torch.uint8, device=out.device)
    Q.forward(p, ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().copy(), lse.cpu().numpy().copy()


def _same_bits(o, l, o_ref, l_ref):
    """Both entry points run the same kernels on the same plan, so the
    results must agree bit for bit (a scratch-offset mistake that moves a
    few partial results would show here even inside the float tolerance)."""
    assert np.array_equal(o.view(np.uint32), o_ref.view(np.uint32))
    assert np.array_equal(l.view(np.uint32), l_ref.view(np.uint32))


CASES = {
    # 2 tokens of 5 tiles over 24 CTAs: every token split into many parts
    "tiny CSA decode": lambda: W.config(0),
    "HCA decode": lambda: W.build("noalloc HCA", layout="BSND", q_lens=[1, 1, 1], s2=[9000, 40000, 130000],
                                  cmp_ratio=128, mode="HCA", seed=21),
    # two 64-head units per token
    "N1 = 128 decode": lambda: W.build("noalloc N1=128", layout="BSND", q_lens=[2, 2], s2=[5000, 20000],
                                       cmp_ratio=4, mode="CSA", k2=512, n1=128, seed=22),
    # a short TND chunk with fewer tokens than CTAs
    "TND chunk": lambda: W.build("noalloc TND", layout="TND", q_lens=[5, 3, 9], s2=[700, 3000, 9000],
                                 cmp_ratio=4, mode="CSA", k2=512, seed=23),
}


def test_noalloc_matches_forward_on_two_calls(cuda_device):
    """Two calls in a row on different inputs (the scratch keeps the first
    call's contents when the second starts)."""
    num_ctas = 24  # more CTAs than query tokens: tokens are split, scratch is used
    for name, make in CASES.items():
        w = make()
        p, out, lse, keep = _params(w, cuda_device, num_ctas)
        need = Q.workspace_size(p)
        assert 0 < need <= Q.NOALLOC_SCRATCH_BYTES, name
        o_ref, l_ref = _existing(p, out, lse)
        st = Q.device_status()
        assert st == 0, (name, "qsfm_forward", st)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        Q.forward_noalloc(p)
        torch.cuda.synchronize()
        st = Q.device_status()
        assert st == 0, (name, "qsfm_forward_noalloc", st)
        _same_bits(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref)


def test_noalloc_against_the_oracle(cuda_device):
    """One case compared with the fp64 oracle directly, at the tolerances of
    the other GPU tests."""
    from oracle import qsfm_oracle as O

    w = W.config(0)
    p, out, lse, keep = _params(w, cuda_device, 24)
    Q.forward_noalloc(p)
    torch.cuda.synchronize()
    assert Q.device_status() == 0
    o = out.float().cpu().numpy().reshape(w.total_t, 64, 512)
    l = lse.cpu().numpy()
    o_ref, l_ref = O.reference(w)
    assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
    assert np.all(np.abs(l - l_ref) <= LSE_ATOL)


def test_noalloc_rejects_plans_beyond_the_scratch(cuda_device):
    w = W.config(0)
    p, out, lse, keep = _params(w, cuda_device, 64)  # 2 tokens over 64 CTAs: ~16.8 MB of partials
    assert Q.workspace_size(p) > Q.NOALLOC_SCRATCH_BYTES
    with pytest.raises(Q.QsfmError) as e:
        Q.forward_noalloc(p)
    assert e.value.code == 4  # QSFM_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()  # nothing was launched
