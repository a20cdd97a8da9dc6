"""The separately built library with the plane kernels' per-phase clocks
(`python bench.py --phase-clocks`): run in a subprocess (a process loads one library), on a
small workload, it must count every plane of every call and attribute cycles to phases."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_phase_clocks_count_every_plane():
    steps = 2
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--phase-clocks",
                          "--workload", "c2_fp32_train", "--steps", str(steps), "--warmup", "1"],
                         capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    out = json.loads(res.stdout.strip().splitlines()[-1])
    planes = 8 * 64 * steps  # c2: N = 8, C = 64, one plane-kernel call a step each
    for name in ("wt_fwd_plane_kernel", "wt_dw_plane_kernel"):
        k = out["kernels"][name]
        assert k["planes"] == planes, (name, k["planes"])
        assert k["cycles_per_plane"] > 0
        shares = [r["share"] for r in k["phases"].values()]
        assert abs(sum(shares) - 1.0) < 1e-6
        assert len(shares) >= 6, k["phases"].keys()
