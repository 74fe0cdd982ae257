"""Host-side logic of bench.py (no GPU): the algorithmic byte counts the
GB/s figures divide by, workload lookup, the staleness rule for committed
DRAM-traffic records, and the reference arm's JSON line (the float64
oracle on the host cores)."""
import io
import json
import os
import shutil
import contextlib

import pytest

import bench
import workloads as W


# Bytes per call printed in the scope table for the RMSNorm configurations
# (fwd = 2RNs + 4R + Ns, bwd = 3RNs + 4R + Ns + 4N), checked against the
# workloads' own counts.
SCOPE_TABLE = {
    "fp32_256x1024": (2_102_272, 3_154_944),
    "llama_bf16_4096x4096": (67_133_440, 100_704_256),
    "gemma_bf16_8192x3072": (100_702_208, 151_046_144),
    "large_bf16_16384x8192_once": (536_952_832, 805_421_056),
    "large_bf16_16384x8192_twice": (536_952_832, 805_421_056),
}

# fwd+bwd bytes of the fp16 sweep at 4096 rows, N = 1024 ... 32768.
FP16_SWEEP_STEP = [41_984_000, 83_935_232, 167_837_696, 335_642_624, 671_252_480,
                   1_342_472_192]


@pytest.mark.parametrize("name", sorted(SCOPE_TABLE))
def test_algorithmic_bytes_match_the_scope_table(name):
    w = bench.workload_by_name(name)
    assert (w.fwd_bytes(), w.bwd_bytes()) == SCOPE_TABLE[name]


def test_fp16_sweep_step_bytes():
    got = [bench.workload_by_name(f"fp16_4096x{n}").step_bytes()
           for n in (1024, 2048, 4096, 8192, 16384, 32768)]
    assert got == FP16_SWEEP_STEP


def test_every_workload_resolves_with_its_metric():
    names = (list(W.all_workloads()) + list(W.layer_norm_workloads()) +
             list(W.fp8_workloads()) + list(W.softmax_workloads()) +
             list(W.group_norm_workloads()))
    assert len(names) == len(set(names))
    for name in names:
        w = bench.workload_by_name(name)
        assert w.name == name
        metric = bench.metric_for(w)
        assert metric.endswith("GB/s and % of GB300 peak; µs per call")
        assert w.step_bytes() > 0
    with pytest.raises((KeyError, SystemExit, ValueError)):
        bench.workload_by_name("no_such_workload")


def test_traffic_records_go_stale_with_their_sources(tmp_path, monkeypatch):
    """A committed DRAM-traffic record is used only while the code of the
    CUDA sources it lists (comments and whitespace aside) hashes to the
    recorded value."""
    csrc = tmp_path / "bwd_rms_norm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_text("__global__ void k() {}\n")
    (csrc / "b.cuh").write_text("// helpers\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    srcs = ["a.cu", "b.cuh"]
    rec = {"w": {"fwd": 10, "bwd": 20, "sources": srcs,
                 "sources_sha256_16": bench.sources_hash(srcs)}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("w")["bwd"] == 20
    assert bench.load_traffic("other") == {}
    # comments and layout do not change the kernels: the record stands
    (csrc / "a.cu").write_text("/* the kernel */\n__global__  void k()\n{}  // empty\n")
    assert bench.load_traffic("w")["bwd"] == 20
    # code does: the record is dropped
    (csrc / "b.cuh").write_text("#define HELPER 1\n")
    assert bench.load_traffic("w") == {}


def test_committed_traffic_records_name_existing_sources():
    path = os.path.join(bench.ROOT, "profiles", "traffic.json")
    with open(path) as f:
        recs = json.load(f)
    for name, rec in recs.items():
        bench.workload_by_name(name)
        for src in rec["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, "bwd_rms_norm_gb300", "csrc", src))
        assert rec["fwd"] > 0 and rec["bwd"] > 0


def test_reference_arm_prints_one_contract_line():
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main(["--impl", "reference", "--workload", "fp32_256x1024", "--steps", "1",
                    "--warmup", "3"])
    lines = [l for l in out.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "fp32_256x1024"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_fewer_than_three_warmup_steps_are_refused():
    with pytest.raises(SystemExit):
        with contextlib.redirect_stderr(io.StringIO()):
            bench.main(["--warmup", "2"])


def test_default_workload_is_the_largest_single_gpu_config():
    """The headline line runs 16384 x 8192 bf16 (round once), the largest
    configuration, and times the round-twice store in the same run."""
    assert bench.DEFAULT_WORKLOAD == "large_bf16_16384x8192_once"
    sizes = {n: w.step_bytes() for n, w in W.all_workloads().items()}
    assert sizes[bench.DEFAULT_WORKLOAD] >= max(sizes.values()) - 200_000
    assert bench.paired_variant(bench.DEFAULT_WORKLOAD) == "large_bf16_16384x8192_twice"
    assert bench.paired_variant("large_bf16_16384x8192_twice") == "large_bf16_16384x8192_once"
    assert bench.paired_variant("llama_bf16_4096x4096") is None


def test_threaded_oracle_matches_one_thread():
    """The all-core oracle baseline runs the unchanged oracle on contiguous
    row ranges: y and dx are those of one pass over all rows, and the weight
    gradient is the per-range sums added in range order."""
    import numpy as np
    from oracle import rms_norm as orm
    from oracle import threads as OT
    w = W.LLAMA_BF16_4096x4096.with_(rows=37, hidden=256)
    inp = W.make_inputs(w)
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    y1, r1 = orm.forward(xd, gd, w.eps, 0, "bf16")
    dx1, dw1 = orm.backward_exact(dyd, xd, gd, r1, 0)

    def run(sl):
        y, r = orm.forward(xd[sl], gd, w.eps, 0, "bf16")
        dx, dw = orm.backward_exact(dyd[sl], xd[sl], gd, r, 0)
        return y, dx, dw

    parts = OT.map_rows(run, w.rows, 4)
    assert [len(r) for r in OT.row_ranges(37, 4)] == [9, 9, 9, 10]
    assert np.array_equal(np.concatenate([p[0] for p in parts]), y1)
    assert np.array_equal(np.concatenate([p[1] for p in parts]), dx1)
    dw = OT.sum_in_order([p[2] for p in parts])
    np.testing.assert_allclose(dw, dw1, rtol=1e-12, atol=1e-12)
    assert np.array_equal(dw, ((parts[0][2] + parts[1][2]) + parts[2][2]) + parts[3][2])


def test_oracle_baseline_reports_both_core_counts(monkeypatch):
    monkeypatch.setattr(bench, "host_threads", lambda: 3)
    w = W.FP32_256x1024.with_(rows=64, hidden=128)
    cpu = bench.oracle_baseline(w, "tiny", budget_s=0.05)
    assert cpu["kind"] == "oracle" and cpu["cores"] == 3
    assert cpu["single_thread"]["cores"] == 1 and cpu["single_thread"]["value"] > 0
    assert cpu["value"] > 0 and "3 threads" in cpu["sample"]
