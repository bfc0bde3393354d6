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
        res["e2e"] = dict(ms=0.2, eager_ms=0.25, graph=True, h2d=100, d2h=50)
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
    assert r["algorithmic_bytes"] == 1000 * row_bytes + 2 * T * n1 * 512 * 2 + T * k2 * 4
    assert r["achieved"] == pytest.approx(r["algorithmic_bytes"] / 0.04e-3 / 1e9)
    assert r["tensor_tflops"] == pytest.approx(2000 * 4 * 512 * n1 / 0.04e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
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
