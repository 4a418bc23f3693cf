"""bench.py's JSON line, assembled on the CPU from made-up op times for every
path, so that a formatting error cannot first show up on the GPU."""
import argparse
import json

import pytest

import bench
from dequant_kvc8_store_gb300 import workloads as W

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "ops",
        "roofline", "gpu_launches", "clocks", "e2e"}


def test_default_workload_is_the_decode_batch():
    ap_default = bench.DEFAULT_WORKLOAD
    assert ap_default == "decode"
    w = W.decode()
    # the largest batch that runs both ops: a store and a gather of > 1 M positions
    assert w.has_store and w.num_tokens == 256 and w.total_context > 1_000_000


@pytest.mark.parametrize("path", ["c8", "bf16", "fused", "attention"])
@pytest.mark.parametrize("gather_only", [False, True])
def test_result_line_for_every_path(path, gather_only):
    w = W.tiny() if not gather_only else W.make_workload(
        "g", q_lens=[0, 0], ctx_before=[3, 17], kv_heads=2, head_dim=64, block_size=16,
        num_blocks=8, quant_mode=0, seed=1, gather_only=True)
    args = argparse.Namespace(path=path, workload="tiny", steps=7, warmup=3)
    one_op = path in ("fused", "attention")
    t = {"step_ms": 0.05, "store_ms": 0.0 if one_op else 0.02, "gather_ms": 0.03, "wall_s": 1.0}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}
    e2e = {"value": 1.0, "unit": "GB/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 1}
    line = bench.result_line(args, 1, w, bench.path_bytes(w, path), t, clocks, e2e,
                             w.has_store and w.num_tokens > 0 and path != "attention")
    assert KEYS <= set(line)
    json.dumps(line)
    assert line["value"] > 0 and line["roofline"]["achieved"] > 0
    if path == "attention":
        assert line["gpu_launches"] == 7 * 3 and "decode_attention" in line["ops"]
    else:
        assert line["gpu_launches"] == 7 * (2 if one_op or gather_only else 3)
    if path == "fused":
        assert line["ops"]["store"]["ms"] == 0.0
    assert line["config"] == bench.config_of(args)


def test_result_line_carries_the_workload_sweep():
    w = W.tiny()
    args = argparse.Namespace(path="c8", workload="tiny", steps=7, warmup=3)
    t = {"step_ms": 0.05, "store_ms": 0.02, "gather_ms": 0.03, "wall_s": 1.0}
    peak, _ = bench.measured_peak()
    sweep = {"steps": 7, "warmup": 3, "clocks": {"sm_mhz": 2070.0}}
    for name in bench.SWEEP_WORKLOADS:
        sweep[name] = bench.op_figures(w, bench.path_bytes(w, "c8"), t, peak)
    line = bench.result_line(args, 1, w, bench.path_bytes(w, "c8"), t, {}, None, True, sweep)
    json.dumps(line)
    by = line["ops"]["by_workload"]
    for name in bench.SWEEP_WORKLOADS:
        for op in ("store", "dequant_gather"):
            e = by[name][op]
            assert e["ms"] > 0 and e["GB_s"] > 0 and 0 < e["frac"] and e["tokens_per_s"] > 0


def test_reference_arm_prints_the_same_config(capsys):
    args = argparse.Namespace(path="c8", workload="tiny", steps=3, warmup=3)
    bench.run_reference(args, 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.config_of(args)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["value"] == line["value"]
    assert "nproc" in line["cpu_baseline"]["host"]


def test_traffic_entries_follow_their_kernel_sources(tmp_path, monkeypatch):
    """A committed traffic figure is used only while its own kernel's sources
    hash as they did at capture; editing one kernel leaves the others valid."""
    root = tmp_path
    csrc = root / "dequant_kvc8_store_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("kvc8_store.cu", "kvc8_gather.cu", "kvc8_internal.cuh"):
        (csrc / f).write_text(f"// {f}\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    (root / "profiles").mkdir()
    entries = {"store_kernel": {"bytes": 11, "source_hash": bench.kernel_hash("store_kernel")},
               "gather_kernel": {"bytes": 22, "source_hash": bench.kernel_hash("gather_kernel")}}
    (root / "profiles" / "ncu_traffic.json").write_text(
        json.dumps({"workloads": {"prefill": entries}}))
    assert bench.ncu_traffic("prefill", "store_kernel") == 11
    assert bench.ncu_traffic("prefill", "gather_kernel") == 22
    assert bench.ncu_traffic("decode", "gather_kernel") is None
    (csrc / "kvc8_store.cu").write_text("// changed\n")
    assert bench.ncu_traffic("prefill", "store_kernel") is None
    assert bench.ncu_traffic("prefill", "gather_kernel") == 22
    (csrc / "kvc8_internal.cuh").write_text("// shared header changed\n")
    assert bench.ncu_traffic("prefill", "gather_kernel") is None


def test_dram_fraction_from_the_captured_launch(tmp_path, monkeypatch):
    root = tmp_path
    csrc = root / "dequant_kvc8_store_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("kvc8_gather.cu", "kvc8_internal.cuh"):
        (csrc / f).write_text(f"// {f}\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    (root / "profiles").mkdir()
    e = {"bytes": 4000, "captured_on": "decode_small", "captured_bytes": 1000,
         "captured_ns": 1000.0, "source_hash": bench.kernel_hash("gather_kernel")}
    (root / "profiles" / "ncu_traffic.json").write_text(
        json.dumps({"workloads": {"decode": {"gather_kernel": e}}}))
    # 1000 bytes in 1 us = 1 GB/s
    assert bench.ncu_dram_frac("decode", "gather_kernel", 2.0) == 0.5
    assert bench.ncu_traffic("decode", "gather_kernel") == 4000
    assert bench.ncu_dram_frac("decode", "store_kernel", 2.0) is None


def test_committed_traffic_file_is_well_formed():
    with open(bench.os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    for wl, ks in d["workloads"].items():
        assert wl in W.NAMED
        for k, e in ks.items():
            assert k in bench.KERNEL_FILES
            assert int(e["bytes"]) > 0 and len(e["source_hash"]) == 16
            if "captured_ns" in e:
                assert int(e["captured_bytes"]) > 0 and float(e["captured_ns"]) > 0
                assert e["captured_on"] in W.NAMED
