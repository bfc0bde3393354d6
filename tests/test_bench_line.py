"""The JSON line bench.py prints, assembled on CPU from a faked GPU result.

The GPU arm is replaced by a function returning fixed timings and work
counts, and the library build by a no-op, so these tests check only the
host-side assembly: the keys of the contract, the algorithmic bytes and
FLOPs for each KV row format and head count, the recorded traffic (only
for the default format), and --quick lines without e2e.
"""

import json
import sys

import pytest

import bench
import compressed_mla_attention_gb300.build as B


def _line(monkeypatch, capsys, argv, work=(1000, 2000), with_e2e=False):
    res = dict(ms=0.05, ms_attn=0.04, ms_plan=0.01, ms_comb=None, launches=6, split=False,
               clocks=None, ctas=2, work=work)
    if with_e2e:
        res["e2e"] = dict(ms=0.2, h2d=100, d2h=50, n=3, sets=3)
    monkeypatch.setattr(B, "build", lambda *a, **k: None)
    monkeypatch.setattr(bench, "run_gpu_arm", lambda args, w, rank, world, local: dict(res))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "3", "--warmup", "3", *argv])
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main()
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    return json.loads(out[0])


@pytest.mark.parametrize("fmt,row_bytes", [("fp8_fp32_scales", 544), ("packed640", 640), ("bf16", 1024)])
@pytest.mark.parametrize("n1", [64, 128])
def test_quick_line_counts_bytes_and_flops_per_format(monkeypatch, capsys, fmt, row_bytes, n1):
    line = _line(monkeypatch, capsys, ["--quick", "--workload", "0", "--kv-format", fmt, "--n1", str(n1)])
    assert "e2e" not in line and "cpu_baseline" not in line
    T, k2 = 2, 512  # tiny CSA decode: 2 tokens, 512 indices each
    r = line["roofline"]
    alg = 1000 * row_bytes + 2 * T * n1 * 512 * 2 + T * k2 * 4
    flops = 2000 * 4 * 512 * n1
    assert r["hbm"]["algorithmic_bytes"] == alg
    assert r["hbm"]["achieved"] == pytest.approx(alg / 0.04e-3 / 1e9)
    assert r["tensor"]["algorithmic_flops"] == flops
    assert r["tensor"]["achieved"] == pytest.approx(flops / 0.04e-3 / 1e12)
    # by hand: the roofline time is the slower floor; frac = that / measured
    hbm, tf, _ = bench.measured_peaks()
    t_roof = max(alg / (hbm * 1e9), flops / (tf * 1e12))
    assert r["roofline_ms"] == pytest.approx(t_roof * 1e3)
    assert r["frac"] == pytest.approx(t_roof / 0.04e-3)
    assert r["frac"] == pytest.approx(max(r["hbm"]["frac"], r["tensor"]["frac"]))
    assert r["bound"] == ("tensor" if flops / (tf * 1e12) > alg / (hbm * 1e9) else "hbm")
    assert r["achieved"] / r["peak"] == pytest.approx(r["frac"])
    assert line["dtype"] == ("f16" if fmt == "fp8_fp32_scales" else "bf16")
    assert r["traffic"] is None  # recorded for the bench workload only
    assert line["value"] == pytest.approx(T / 0.05e-3)
    assert ("kv=" in line["config"]["workload"]) == (fmt != "fp8_fp32_scales")
    assert ("N1=128" in line["config"]["workload"]) == (n1 == 128)


def test_default_line_has_the_contract_keys(monkeypatch, capsys):
    monkeypatch.setattr(bench, "oracle_throughput", lambda w, toks, cores, secs: (1234.0, 3, 12.0))
    line = _line(monkeypatch, capsys, [], with_e2e=True)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "gpu_launches", "roofline", "e2e",
                "cpu_baseline"):
        assert key in line, key
    assert line["config"]["workload"].startswith("CSA decode batch B=128")
    assert line["e2e"]["h2d_bytes_per_step"] == 100 and line["e2e"]["d2h_bytes_per_step"] == 50
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == 1234.0
    # the traffic figure is reported only while the kernel source hash matches the record
    assert line["roofline"]["traffic"] == bench.recorded_traffic(2)


def test_e2e_input_sets_and_packing():
    """The e2e pipeline's host inputs: rotating sets keep every block-table
    entry inside its pool (a permutation of the pool's blocks, -1 kept), and
    the packed pinned buffer views give back each tensor bit for bit."""
    import torch

    import workloads as W

    w = W.build("e2e sets", layout="BSND", q_lens=[2, 2], s2=[300, 700], cmp_ratio=4, mode="CSA", k2=16,
                block_size=128, seed=3)
    a = W.device_inputs(w, "cpu")
    sets = bench._step_input_sets(a, 3, seed=1)
    assert len(sets) == 3 and sets[0]["q"] is not sets[1]["q"]
    for s in sets[1:]:
        for tk, pool in (("ori_block_table", "ori_kv"), ("cmp_block_table", "cmp_kv")):
            t0, t1 = sets[0][tk], s[tk]
            assert torch.equal(t0 < 0, t1 < 0)
            assert int(t1.max()) < a[pool].shape[0]
            assert sorted(t1[t1 >= 0].tolist()) != t1[t1 >= 0].tolist() or not torch.equal(t0, t1)
    buf, layout = bench._pack(sets[1], pin=False)  # pinning needs a GPU driver
    views = bench._views(buf, layout)
    for k, t in sets[1].items():
        assert layout[k][0] % 256 == 0
        assert torch.equal(views[k], t)
