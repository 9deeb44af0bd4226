"""bench.py with more than one rank, on the CPU (gloo, world size 2).

With N > 1 the benchmark runs one process per GPU with independent replicas
of the workload (no data-path collective): the only collectives are the
barriers around the timed region and the max over ranks of the timed
milliseconds.  These tests run that code under torch.distributed.run with
two CPU ranks: the max-over-ranks reduction and barriers of bench.DistCtx,
and the reference arm, where rank 0 alone times the oracle and prints the
one JSON line while the other rank exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}"] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def _json_lines(text):
    return [json.loads(l) for l in text.splitlines() if l.startswith("{")]


def test_max_over_ranks_and_barriers_with_two_gloo_ranks(tmp_path):
    r = _torchrun([os.path.join(ROOT, "tests", "dist_rank_probe.py"), str(tmp_path)], timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / f"rank{k}.json").read_text()) for k in range(2)]
    assert [d["rank"] for d in lines] == [0, 1]
    for d in lines:
        assert d["world"] == 2 and d["backend"] == "gloo"
        assert d["max"] == 17.5  # the slower rank's time, seen by both ranks


def test_reference_arm_prints_one_line_from_rank_zero():
    r = _torchrun([os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                   "--steps", "3", "--warmup", "3"], timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "layer-steps/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
