"""Host-side pieces of bench.py (no GPU): the oracle cast sweep's threaded slabs
give the single calls' bytes, and the sweep prints one JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
import oracle
from scaled_quantize_gemm_amax_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.mark.parametrize("kind", [oracle.KIND_TENSOR, oracle.KIND_1x128, oracle.KIND_128x128, oracle.KIND_MX])
@pytest.mark.parametrize("threads", [1, 2, 3])
def test_threaded_slabs_equal_the_single_calls(kind, threads):
    xh = bench._bits(wl.normal_bf16((384, 640), 91, 1.0, "cpu"))
    xh[5, 7] = 0x4700          # 32768: a block whose scale differs from its neighbours
    scale = oracle.tensor_scale(oracle.amax(xh), oracle.E4M3)[0] if kind == oracle.KIND_TENSOR else None
    row_parts, col_parts = bench._oracle_cast_both(oracle, xh, kind, threads, scale)
    for parts, ref in ((row_parts, oracle.quantize_rowwise(xh, kind, oracle.E4M3, scale)),
                       (col_parts, oracle.quantize_colwise(xh, kind, oracle.E4M3, scale))):
        q = np.concatenate([p[0] for p in parts])
        assert np.array_equal(q, ref[0])
        if kind == oracle.KIND_TENSOR:
            assert all(np.array_equal(p[1], ref[1]) for p in parts)
        else:
            s = np.concatenate([p[1] for p in parts])
            assert np.array_equal(s.view(np.uint8), ref[1].view(np.uint8))


def test_cpu_baseline_sweep_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-baseline-sweep", "256"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["kind"] == "oracle" and d["cores"] >= 1
    got = {(r["recipe"], r["threads"]) for r in d["runs"]}
    assert got == {(name, t) for name in ("TENSOR", "BLOCK_1x128", "BLOCK_128x128", "MX_1x32")
                   for t in {1, d["cores"]}}
    assert all(r["size"] == 256 and r["s"] > 0 and r["GB/s"] > 0 for r in d["runs"])
