"""The N>1 path of bench.py on CPU (gloo, world size 2).  Every CP rank is
emulated on one GPU, so N GPUs run N independent replicas: the step time is
the slowest replica's (a MAX over the process group) and the job's value adds
up the replicas' work; the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _torchrun(args, timeout):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    env = dict(os.environ, OMP_NUM_THREADS="2")
    return subprocess.run(cmd, capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=env)


def _json_lines(text):
    return [json.loads(line) for line in text.splitlines() if line.startswith("{")]


def test_max_over_ranks_and_whole_job_value_world2(tmp_path):
    out = _torchrun([os.path.join(ROOT, "tests", "replica_reduce_worker.py"), str(tmp_path)], 300)
    assert out.returncode == 0, out.stderr[-3000:]
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [d["rank"] for d in res] == [0, 1]
    for d in res:
        assert d["ws"] == 2
        assert d["max"] == [2.0, 10.0, 3.5]          # element-wise max over both ranks
        # two replicas of 2 TFLOP per step in the slower one's 2 ms
        assert d["value"] == pytest.approx(2 * 2e12 / 2e-3 / 1e12)


def test_reference_arm_under_torchrun_prints_once():
    out = _torchrun([os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                     "--steps", "1", "--warmup", "3"], 900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = _json_lines(out.stdout)
    assert len(lines) == 1                           # rank 0 alone runs and prints
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_roofline_peak_choice():
    """The burst BF16 peak is the denominator while the median SM clock stays
    within 10% of its maximum (a barely binding power cap included); the
    sustained one once the clock is pulled well below it; without clock
    samples the region's length decides."""
    sys.path.insert(0, ROOT)
    import bench
    at_max = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    capped = {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    slow = {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    none = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    assert bench._pick_peak(0.5, at_max, 1943.5, 1725.2) == (1943.5, "burst")
    assert bench._pick_peak(2.0, at_max, 1943.5, 1725.2) == (1943.5, "burst")
    assert bench._pick_peak(1.0, capped, 1943.5, 1725.2) == (1943.5, "burst")
    assert bench._pick_peak(1.0, slow, 1943.5, 1725.2) == (1725.2, "sustained")
    assert bench._pick_peak(0.5, none, 1943.5, 1725.2) == (1943.5, "burst")
    assert bench._pick_peak(2.0, none, 1943.5, 1725.2) == (1725.2, "sustained")
