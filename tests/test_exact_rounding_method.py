"""The dynamic-scale store decides flagged (near-tie) values without a
division: code = n or n + 1 from the sign of the exact remainder
|x| - (n + 1/2) s, or the even one of them when fl(|x|/s) is exactly n + 1/2.
This checks that rule on the host against one IEEE division per value, for
every bf16 value under scales amax/127 from every bf16 amax mantissa and for
random fp32 scales (the GPU parity tests check the kernel itself)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_remainder_rule_matches_division(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "exact_rounding_check"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe),
                    os.path.join(HERE, "exact_rounding_check.c"), "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    checked, bad = map(int, out.stdout.split()[-2:])
    assert checked > 10_000_000
    assert out.returncode == 0 and bad == 0, out.stdout
