"""bench.py's host logic on CPU: the reference arm's JSON line (it times the oracle and
needs no GPU), the algorithmic-work and roofline arithmetic against hand-worked values,
and the rule that a recorded DRAM traffic figure is used only for the sources and the
workload it was captured on."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from padding_free_variable_gb300 import synthetic  # noqa: E402

PEAKS = {"hbm_gbs": 6764.0, "bf16_tflops_sustained": 1719.1, "sm_max_mhz": 2070.0, "source": "test"}


def test_reference_arm_prints_one_contract_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    d = json.loads(lines[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "frames/s"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["config"]["workload"] == "uni-1x32-d16-b8" and d["config"]["frames_per_step"] == 204
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # frames/s and ms/step describe the same run
    assert d["value"] == pytest.approx(204 / (d["ms_per_step"] / 1e3), rel=1e-3)


def test_recurrent_smem_bytes_and_peak_by_hand():
    spec = synthetic.WORKLOADS[2]                       # bi, 1 layer, H = 256, fp32
    rows, T, ctas = 9564, 720, 8
    # per direction: T steps x |R| (4H x H fp32) + ctas x rows x H x 4 bytes of staged h
    per_dir = T * 4 * 256 * 256 * 4 + ctas * rows * 256 * 4
    assert bench.rec_smem_bytes("rec_fwd", spec, rows, T, ctas) == 2 * per_dir == 1666646016
    cfg = {"kernel": "cluster", "ctas_per_direction": ctas}
    r = bench.roofline_of("rec_fwd", 2.0, 1, spec, rows, T, 40, PEAKS, cfg)
    assert r["bound"] == "smem" and r["unit"] == "GB/s"
    assert r["peak"] == pytest.approx(16 * 128 * 2070e6 / 1e9, abs=0.1)          # 16 SMs x 128 B/clk
    assert r["achieved"] == pytest.approx(1666646016 / 2e-3 / 1e9, abs=0.1)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], abs=1e-4)


def test_gemm_work_and_bound_by_hand():
    spec = synthetic.WORKLOADS[3]                       # bi, 5 layers, D = 40 then 1024, H = 512, bf16
    rows = 40555
    fl, by = bench.kind_work("input_gemm", spec, rows, 40)
    G4 = 2 * 4 * 512
    assert fl == pytest.approx(2.0 * rows * G4 * (40 + 4 * 1024))
    # X (bf16) + W (bf16) read, fp32 pre-activations written, every layer
    exp_by = sum(rows * D * 2 + G4 * D * 2 + rows * G4 * 4 for D in [40] + [1024] * 4)
    assert by == pytest.approx(exp_by)
    r = bench.roofline_of("input_gemm", 1.0, 5, spec, rows, 1569, 40, PEAKS, None)
    assert r["bound"] == "tensor" and r["peak"] == pytest.approx(1719.1)
    assert r["achieved"] == pytest.approx(fl / 1e-3 / 1e12, rel=1e-3)
    # a K = 16 fp32 product is bound by its bytes, not its flops
    r1 = bench.roofline_of("input_gemm", 0.01, 1, synthetic.WORKLOADS[1], 204, 37, 16, PEAKS, None)
    assert r1["bound"] == "hbm" and r1["unit"] == "GB/s"


def test_recorded_traffic_is_keyed_to_sources_and_workload(tmp_path, monkeypatch):
    rec = {"rec_fwd@w": {"workload": "w", "dram_bytes_per_launch": 123, "source_digest": bench.source_digest("rec_fwd")}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda kind="": rec["rec_fwd@w"]["source_digest"])
    assert bench.recorded_traffic("rec_fwd", "w") == 123
    assert bench.recorded_traffic("rec_fwd", "other") is None          # another workload
    assert bench.recorded_traffic("rec_bwd", "w") is None              # nothing recorded
    monkeypatch.setattr(bench, "source_digest", lambda kind="": "changed")
    assert bench.recorded_traffic("rec_fwd", "w") is None              # the kernels changed since


def test_source_digest_sees_code_not_comments():
    """The digest that keys a traffic record follows what the compiler sees: a comment or a
    whitespace change keeps it, a changed token (also inside a string literal) moves it."""
    base = 'int f(int a) { return a + 1; }  // adds one\nconst char* s = "x // y";\n'
    same = '/* header */\nint f(int a)\n{\n    return a + 1;   // one more\n}\nconst char* s = "x // y";\n'
    assert bench.code_only(base) == bench.code_only(same)
    assert bench.code_only(base) != bench.code_only(base.replace("a + 1", "a + 2"))
    assert bench.code_only(base) != bench.code_only(base.replace('"x // y"', '"x // z"'))
    assert "adds" not in bench.code_only(base) and "x // y" in bench.code_only(base)


def test_md_work_counts():
    """The 2-D phases' algorithmic flops: per cell 20 H^2 + 25 H forward (two recurrent products
    and the cell), 20 H^2 + 40 H backward; the input projection 10 D H per pixel and direction."""
    N, nd, D, H = 1000, 4, 16, 32
    assert bench.md_kind_work("md_fwd", N, nd, D, H) == N * nd * (20 * H * H + 25 * H)
    assert bench.md_kind_work("md_bwd", N, nd, D, H) == N * nd * (20 * H * H + 40 * H)
    assert bench.md_kind_work("md_input", N, nd, D, H) == 2 * N * D * nd * 5 * H
    assert bench.md_kind_work("nothing", N, nd, D, H) == 0.0
