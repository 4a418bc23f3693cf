"""Readers for the hand-worked golden files under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _strip(line):
    return line.split("#", 1)[0].strip()


def quantize_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "quantize_rows.txt")) as f:
        for raw in f:
            line = _strip(raw)
            if not line:
                continue
            if line.startswith("[case"):
                cur = {"name": line[len("[case"):-1].strip()}
                cases.append(cur)
                continue
            key, val = (t.strip() for t in line.split("=", 1))
            cur[key] = val.split()
    out = []
    for c in cases:
        H, D = int(c["heads"][0]), int(c["head_dim"][0])
        d = {"name": c["name"], "mode": int(c["mode"][0]), "heads": H, "head_dim": D,
             "x": [v for v in c["x"]],
             "codes": np.array([int(v) for v in c["expect_codes"]], np.int64).reshape(H, D)}
        if "expect_scale_bits" in c:
            d["scale_bits"] = [int(v, 16) for v in c["expect_scale_bits"]]
        if "static_scale_bits" in c:
            d["static_bits"] = np.array([int(v, 16) for v in c["static_scale_bits"]],
                                        np.uint32).reshape(H, D)
        assert len(d["x"]) == H * D and d["codes"].size == H * D
        out.append(d)
    return out


def dequant_values():
    rows = []
    with open(os.path.join(GOLDEN, "dequant_values.txt")) as f:
        for raw in f:
            line = _strip(raw)
            if not line:
                continue
            q, s, e = line.split()
            rows.append((int(q), int(s, 16), int(e, 16)))
    return rows


def placement():
    kv = {}
    with open(os.path.join(GOLDEN, "placement_tiny.txt")) as f:
        for raw in f:
            line = _strip(raw)
            if not line:
                continue
            key, val = (t.strip() for t in line.split("=", 1))
            kv[key] = val
    g = {
        "block_size": int(kv["block_size"]),
        "num_blocks": int(kv["num_blocks"]),
        "block_table": np.array([[int(v) for v in row.split()] for row in kv["block_table"].split("|")],
                                np.int32),
        "cu_q_lens": np.array(kv["cu_q_lens"].split(), np.int32),
        "context_kv_lens": np.array(kv["context_kv_lens"].split(), np.int32),
        "expect_slot": {},
        "gathers": [],
    }
    for item in kv["expect_slot"].split():
        t, bs = item.split(":")
        blk, slot = bs.split(",")
        g["expect_slot"][int(t)] = (int(blk), int(slot))
    for i in (1, 2, 3):
        pre = f"gather{i}_"
        gg = {"context_lengths": np.array(kv[pre + "context_lengths"].split(), np.int32),
              "rows": kv[pre + "rows"].split()}
        if pre + "offsets" in kv:
            gg["offsets"] = np.array(kv[pre + "offsets"].split(), np.int64)
            gg["out_rows"] = int(kv[pre + "out_rows"])
        g["gathers"].append(gg)
    return g
