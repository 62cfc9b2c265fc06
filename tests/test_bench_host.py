"""Host-side logic of bench.py, on the CPU: the multi-rank aggregation (two
gloo ranks), the algorithmic byte count, and the reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402

_RANK_SCRIPT = r"""
import json, os, sys, torch
sys.path.insert(0, sys.argv[1])
import bench
world, rank, local = bench.dist_env()
bench.init_dist(world, "gloo")
bench.barrier()
mx = bench.reduce_max(1.5 + rank, torch.device("cpu"))
sm = bench.reduce_sum(10.0 * (rank + 1), torch.device("cpu"))
bench.barrier()
print(json.dumps({"rank": rank, "world": world, "max": mx, "sum": sm}))
torch.distributed.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_max_time_and_total_units():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2
        assert o["max"] == 2.5          # max over ranks of 1.5 + rank
        assert o["sum"] == 30.0         # 10 + 20


def test_single_process_reductions_are_identity():
    assert bench.reduce_max(3.25, torch.device("cpu")) == 3.25
    assert bench.reduce_sum(7.0, torch.device("cpu")) == 7.0


def test_algorithmic_bytes_by_hand():
    specs = [workloads.TableSpec(100, 16, "f32", ("fixed", 2), ("uniform",)),
             workloads.TableSpec(50, 32, "bf16", ("fixed", 1), ("uniform",))]
    B, T = 3, 2
    lengths = torch.tensor([2, 2, 2, 1, 1, 1])
    N, U, passes = 9, 5, 1
    b = bench.algorithmic_bytes(specs, lengths, N, B, T, 8, True, "adagrad", U, passes)
    gathered = 6 * 16 * 4 + 3 * 32 * 2
    out = B * 48 * 4
    fwd = gathered + N * 8 + (T * B + 1) * 8 + N * 4 + out
    assert b["forward"] == fwd
    prep = N * 8 + (T * B + 1) * 8 + N * 12 + passes * N * 16 - N * 4 + N * 4 + U * 8
    assert b["prepare"] == prep
    grad_rows = 6 * 16 * 4 + 3 * 32 * 4
    avg_row = (16 * 4 + 32 * 2) / 2
    apply = grad_rows + N * 12 + U * 8 + 2 * U * avg_row + 2 * U * 4
    assert b["apply"] == apply
    assert b["step"] == fwd + prep + apply


def test_reference_arm_prints_contract_line(capsys):
    pytest.importorskip("numpy")
    bench.main(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_length_order_rule_follows_the_length_law():
    """The bench turns the length-keyed order on only for lengths drawn
    uniformly over a wide range (workload 5), and --length-order on|off
    overrides it."""
    for cid, want in [(1, False), (2, False), (3, False), (4, False), (5, True)]:
        specs = workloads.realize_tables(workloads.get_config(cid))
        assert bench.wants_length_order(specs, "auto") is want, cid
        assert bench.wants_length_order(specs, "on") is True
        assert bench.wants_length_order(specs, "off") is False


def test_histogram_forward_only_where_a_workload_prescribes_it():
    assert [workloads.get_config(c).histogram_forward for c in (1, 2, 3, 4, 5)] == [False] * 4 + [True]
    # shrunk parity variants keep the prescription
    assert workloads.get_config(5).scaled(B=160, rows_div=1000, rows_min=512).histogram_forward
