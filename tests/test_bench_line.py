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


def test_committed_traffic_file_is_well_formed():
    with open(bench.os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    for wl, ks in d["workloads"].items():
        assert wl in W.NAMED
        for k, e in ks.items():
            assert k in bench.KERNEL_FILES
            assert int(e["bytes"]) > 0 and len(e["source_hash"]) == 16
