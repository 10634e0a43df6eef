"""bench.py's reference arm on the CPU: the oracle timed on the host cores.

The arm needs no GPU: it draws the workload's inputs and times the oracle on
a bounded sample.  One process prints one JSON line with the contract's keys;
under a two-rank launcher (gloo) rank 0 alone runs and prints, and both ranks
exit 0.
"""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORKLOAD = "all_gather_v_bf16_w5"   # the V workloads run in full and are small


def _lines(out):
    return [json.loads(x) for x in out.splitlines() if x.startswith("{")]


def _check_line(d, n_gpus):
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == n_gpus and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["name"] == WORKLOAD
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["host_cores"] == os.cpu_count() and d["cpu_baseline"]["cpu_model"]
    # the workload only: the own arm prints the same object (see below)
    assert set(d["config"]) == {"workload", "name", "world", "algorithmic_bytes_per_step", "l2"}
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_one_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                        "--workload", WORKLOAD], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def test_reference_arm_two_ranks_prints_once():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--gpus", "2", "--workload", WORKLOAD],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)


def test_both_arms_describe_the_workload_alike():
    """The own arm and the reference arm build `config` with one function from
    the workload alone, so the two lines of a workload carry equal objects."""
    sys.path.insert(0, ROOT)
    import bench
    import workload_inputs as inputs
    from collective_datapath_reduce_gb300 import purlin as P
    wl = bench.workloads(P, inputs)[WORKLOAD]
    x = wl.make_inputs()
    import numpy as np
    a, b = bench.config_of(wl, x), bench.config_of(wl, [np.copy(v) for v in x])
    assert a == b and a["name"] == WORKLOAD and "MiB" in a["l2"]
