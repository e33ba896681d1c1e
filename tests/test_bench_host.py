"""CPU tests of bench.py's host logic: the work model and the multi-rank
plumbing (barrier and max over ranks) with two gloo ranks."""
import os
import socket
import subprocess
import sys
import textwrap

import bench
from linear_attention_recurrence_gated_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_work_model_matches_hand_count():
    w = W.WORKLOADS["hymo_bf16"]
    # per head-token: C(6dk+4dv) + 6 dk dv + C^2/3 with C=64, dk=dv=64
    assert bench.flops_per_head_token(64, 64) == 64 * (6 * 64 + 4 * 64) + 6 * 64 * 64 + 64 * 64 / 3
    assert bench.bytes_per_head_token(64, 64, 2) == 518
    tokens = 8 * 4096
    b = bench.algorithmic_bytes(w, tokens, 8, with_init=False)
    assert abs(b - (tokens * 16 * 518 + 8 * 16 * 64 * 64 * 4)) < 1
    assert 273e6 < b < 275e6
    assert abs(bench.algorithmic_flops(w, tokens) / 1e9 - 35.07) < 0.05


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_gloo_ranks_max_over_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import os, sys
        sys.path.insert(0, {ROOT!r})
        import bench, torch
        rank, world, local = bench.dist_setup()
        assert world == 2 and torch.distributed.get_backend() == "gloo"
        bench.barrier(world)
        m = bench.max_over_ranks(1.5 + rank, world)
        assert m == 2.5, m
        print("rank", rank, "ok", flush=True)
        torch.distributed.destroy_process_group()
    """))
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()),
               WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    procs = []
    for r in range(2):
        e = dict(env, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=e,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=120)[0] for p in procs]
    assert all(p.returncode == 0 for p in procs), outs
    assert all("ok" in o for o in outs)


def test_reference_arm_only_rank0_prints(tmp_path):
    """Non-zero ranks of the reference arm exit without work."""
    import argparse
    args = argparse.Namespace(steps=1, warmup=3)
    assert bench.bench_reference(args, W.WORKLOADS["tiny_fp32"], rank=1, world=2) == 0


def test_reference_arm_line(capsys):
    import argparse, json
    args = argparse.Namespace(steps=2, warmup=3)
    bench.bench_reference(args, W.WORKLOADS["tiny_fp32"], rank=0, world=1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
