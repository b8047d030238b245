"""bench.py's contract on the CPU: the reference arm's JSON line (the oracle
timed on the host cores, run here on the tiny workload) and the count of
library launches it reports for a slot-path step."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402
from offloaded_expert_slot_gb300.configs import C1, C2, C5, scaled  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "c1_tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "c1_tiny" and d["data"] == "synthetic"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    # cores is numpy's BLAS pool, which bench.py sizes before numpy loads
    assert "numpy's BLAS with %d threads" % d["cpu_baseline"]["cores"] in d["cpu_baseline"]["sample"]
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("cfg,want", [
    # restore, topk, distinct, 3 ensures, 6 copies (queries of 128, 128 and
    # 64 ids: two parts each), flags, one-CTA align, hits GEMM1/2, 6 part
    # GEMM1/2 pairs, combine
    (C2, 1 + 1 + 1 + 3 + 6 + 1 + 1 + 2 + 12 + 1),
    # restore, gate logits, topk, distinct, 1 ensure, 1 copy (8 ids: one
    # part), flags, one-CTA align, hits pair, one part pair, combine
    (C1, 1 + 1 + 1 + 1 + 1 + 1 + 1 + 1 + 2 + 2 + 1),
    # restore, topk, distinct, 4 ensures, 8 copies, flags, count/scan/scatter
    # align, hits pair, 8 part pairs, combine, x -> f16 (NVFP4)
    (C5, 1 + 1 + 1 + 4 + 8 + 1 + 3 + 2 + 16 + 1 + 1),
    # one-token decode: 10 ids, one query in one part
    (scaled(C2, T=1), 1 + 1 + 1 + 1 + 1 + 1 + 1 + 2 + 2 + 1),
], ids=["decode_width", "tiny", "long_prefill", "one_token"])
def test_gpu_launch_count_follows_the_slot_path(cfg, want):
    assert bench.gpu_launches(cfg) == want


def test_blas_pool_is_sized_before_numpy_loads():
    """A caller's OPENBLAS_NUM_THREADS stands; otherwise bench.py sets it to
    the cores the process may run on, and the baselines report that."""
    code = ("import os, bench; print(os.environ['OPENBLAS_NUM_THREADS'], bench.blas_threads(), "
            "len(os.sched_getaffinity(0)))")
    env = {k: v for k, v in os.environ.items() if k != "OPENBLAS_NUM_THREADS"}
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT,
                         env=env, timeout=300, check=True).stdout.split()
    assert out[0] == out[1] == out[2]
    env["OPENBLAS_NUM_THREADS"] = "3"
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT,
                         env=env, timeout=300, check=True).stdout.split()
    assert out[0] == out[1] == "3"
