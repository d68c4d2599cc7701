"""The bench's multi-rank path on CPU: two ranks over gloo, launched the way
a multi-GPU run is (torch.distributed.run, one process per rank, rendezvous
on 127.0.0.1).

Each rank runs an independent replica, so the only exchanges are the
barrier around the timed region and the max over ranks of its duration;
the value is the units of all ranks over that max, and rank 0 alone prints
the JSON line.  The GPU arm reaches the same `Ranks` object over nccl.
"""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(nproc, argv, cwd, timeout=240):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={nproc}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}"] + argv
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    env.pop("LOCAL_RANK", None)
    env["OMP_NUM_THREADS"] = "1"
    return subprocess.run(cmd, cwd=cwd, env=env, capture_output=True, text=True, timeout=timeout)


def _json_lines(text):
    out = []
    for ln in text.splitlines():
        ln = ln.strip()
        if ln.startswith("{"):
            out.append(json.loads(ln))
    return out


WORKER = textwrap.dedent("""
    import json, os, sys
    sys.path.insert(0, {root!r})
    import bench

    r = bench.Ranks("gloo")
    assert r.world == 2 and r.rank in (0, 1), (r.world, r.rank)
    # a rank-dependent "timed region": rank 1 is the slow one
    mine_ms = 10.0 + 5.0 * r.rank
    r.barrier()
    mx = r.max(mine_ms)
    units = 4.0e9                      # units one rank processed
    value = r.aggregate(units, mx * 1e-3)
    with open(os.path.join({tmp!r}, "rank%d.json" % r.rank), "w") as f:
        json.dump({{"rank": r.rank, "max_ms": mx, "value": value}}, f)
    r.emit({{"rank": r.rank, "world": r.world, "max_ms": mx, "value": value}})
    r.close()
""")


def test_ranks_max_and_rank0_line_over_gloo(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT, tmp=str(tmp_path)))
    p = _torchrun(2, [str(script)], cwd=str(tmp_path))
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    # every rank got the slowest rank's time and the same whole-job value
    per_rank = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(2)]
    expect_value = 2 * 4.0e9 / 15.0e-3
    for d in per_rank:
        assert d["max_ms"] == 15.0
        assert abs(d["value"] - expect_value) <= 1e-9 * expect_value
    # one line, from rank 0
    lines = _json_lines(p.stdout)
    assert len(lines) == 1, p.stdout
    assert lines[0]["rank"] == 0 and lines[0]["world"] == 2


def test_reference_arm_two_ranks_one_line():
    """`bench.py --impl reference` under torchrun: rank 0 times the oracle and
    prints the line; rank 1 exits 0 without work."""
    p = _torchrun(2, ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"], cwd=ROOT)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    lines = _json_lines(p.stdout)
    assert len(lines) == 1, p.stdout
    d = lines[0]
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_ranks_single_process_needs_no_group(monkeypatch, capsys):
    """N = 1 (no torchrun environment): no process group, the max is the
    rank's own value, and the line is printed."""
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks("gloo")
    assert (r.world, r.rank, r.dist) == (1, 0, None)
    assert r.max(3.5) == 3.5
    assert r.aggregate(10.0, 2.0) == 5.0
    r.emit({"x": 1})
    r.close()
    assert _json_lines(capsys.readouterr().out) == [{"x": 1}]
