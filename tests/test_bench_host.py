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


def test_source_hash_ignores_comments_only():
    """The profile hash covers code, not comments: editing a comment keeps a
    profile's counters valid, editing code does not."""
    src = 'int f(int x) {  // doubles\n  /* twice\n */ return 2 * x;  \n}\nconst char *s = "a // b";\n'
    assert bench.code_only(src) == 'int f(int x) {\n   return 2 * x;\n}\nconst char *s = "a // b";'
    assert bench.code_only(src.replace("doubles", "twice x")) == bench.code_only(src)
    assert bench.code_only(src.replace("2 * x", "3 * x")) != bench.code_only(src)
    assert bench.code_only("char c = '\\'';  // q\n") == "char c = '\\'';"


def test_committed_profiles_name_their_sources():
    """Every ncu summary that carries counters names a kernel bench.py knows
    and the hash of the code it was taken on (bench.py reports the counters
    only while that hash matches the sources)."""
    import glob
    import re
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path).read()
        if "dram_bytes_per_launch" not in text:
            continue
        name = os.path.basename(path)[:-3]
        assert any(name.startswith(k + "_") for k in bench.KERNEL_SOURCES), path
        assert re.search(r"source_sha:\s*[0-9a-f]{16}\b", text), path
