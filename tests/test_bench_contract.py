"""The benchmark's output contract, on the arm that needs no GPU (CPU only).

`bench.py --impl reference` times the oracle on host cores and prints one JSON
line with the same metric, unit and config as the GPU arm, plus the oracle's
own cpu_baseline and an e2e object with no host-device traffic.  Under a
multi-process launch only rank 0 prints; the other ranks exit 0 without work.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*argv, env_extra=None, timeout=240):
    env = {**os.environ, **(env_extra or {})}
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], capture_output=True, text=True,
                          timeout=timeout, env=env, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    proc = _bench("--impl", "reference", "--workload", "ragged", "--steps", "2", "--warmup", "1",
                  "--cpu-threads", "2", "--ref-step-seconds", "0.3")
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, proc.stdout
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"].startswith("SGEMM TFLOPS") and line["unit"] == "TFLOP/s"
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 3  # warm-up raised to the three-step minimum
    assert line["n_gpus"] == 1 and line["vs_baseline"] is None
    cfg = line["config"]
    assert (cfg["m"], cfg["n"], cfg["k"]) == (3000, 1500, 777) and "3000x1500x777" in cfg["workload"]
    # the GPU arm builds its config with the same function and arguments: same keys, same values
    sys.path.insert(0, ROOT)
    import bench
    ours = bench.make_config("ragged", bench.WORKLOADS["ragged"][1], ["ffma", "tf32", "3xtf32"], 1)
    assert cfg == ours
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == line["value"] and cb["sample"]
    assert cb["unit"] == line["unit"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    proc = _bench("--impl", "reference", "--workload", "ragged", "--steps", "1", "--warmup", "3",
                  "--ref-step-seconds", "0.3", env_extra={"RANK": "1", "WORLD_SIZE": "2"}, timeout=120)
    assert proc.returncode == 0, proc.stderr[-2000:]
    assert proc.stdout.strip() == ""


@pytest.mark.parametrize("flag", ["--help"])
def test_cli_lists_the_contract_flags(flag):
    proc = _bench(flag, timeout=120)
    assert proc.returncode == 0
    for opt in ("--gpus", "--steps", "--warmup", "--impl"):
        assert opt in proc.stdout


def test_reference_arm_under_torchrun_prints_once():
    """The launch the scaling run uses (torchrun, two ranks on this host): rank 0
    alone prints the line, every rank exits 0."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    proc = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                           "--gpus", "2", "--impl", "reference", "--workload", "ragged", "--steps", "1",
                           "--warmup", "3", "--cpu-threads", "2", "--ref-step-seconds", "0.3"],
                          capture_output=True, text=True, timeout=300, cwd=ROOT,
                          env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, proc.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def _profile_commands(text):
    """Logical command lines (backslash continuations joined) of a profile summary."""
    out, cur = [], ""
    for raw in text.splitlines():
        line = raw.strip()
        if not cur and not (line.startswith("ncu ") or line.startswith("python ") or line.startswith("SNIP=")):
            continue
        cur += " " + line.rstrip("\\").strip()
        if not line.endswith("\\"):
            out.append(cur.strip())
            cur = ""
    return out


def test_profile_summaries_give_runnable_commands():
    """Each ncu summary under profiles/ names the command that made it; the
    command runs committed files only, with bench.py flags and workloads that
    exist, and every ncu invocation leaves the clocks alone."""
    import re
    sys.path.insert(0, ROOT)
    import bench
    help_text = _bench("--help", timeout=120).stdout
    pdir = os.path.join(ROOT, "profiles")
    names = sorted(f for f in os.listdir(pdir) if f.endswith(".md"))
    assert names
    for name in names:
        cmds = _profile_commands(open(os.path.join(pdir, name)).read())
        assert any(c.startswith("ncu ") for c in cmds), name
        for c in cmds:
            if c.startswith("ncu "):
                assert "--clock-control none" in c, (name, c)
            if "bench.py" in c:
                tail = c.split("bench.py", 1)[1].split()
                for tok in tail:
                    if tok.startswith("--"):
                        assert tok in help_text, (name, tok)
                m = re.search(r"--workload (\S+)", c)
                if m:
                    assert m.group(1) in bench.WORKLOADS, (name, m.group(1))


def test_bench_figures_and_config_helpers():
    """The arithmetic behind the GPU arm's JSON line, without a GPU: per-mode
    TFLOP/s, the roofline min(compute, AI x HBM) and its bound, the tensor-pipe
    fraction (3xTF32 counts its three products), and one config for both arms."""
    sys.path.insert(0, ROOT)
    import bench
    from precision_gemm_gb300 import synth
    pk = {"fp32": 80.0, "tf32": 900.0, "hbm": 6800.0, "pipe": 1289.0}
    big = synth.Problem(8192, 8192, 8192, beta=1.0)
    f = bench.mode_figures("ffma", big, 17.2, pk)
    assert abs(f["tflops"] - 2 * 8192 ** 3 / 17.2e-3 / 1e12) < 1e-9
    assert f["bound"] == "compute" and f["roofline_tflops"] == 80.0 and "frac_of_tensor_pipe" not in f
    t = bench.mode_figures("3xtf32", big, 3.0, pk)
    assert t["compute_peak_tflops"] == 300.0 and abs(t["frac_of_tensor_pipe"] - 3 * t["tflops"] / 1289.0) < 1e-12
    skinny = synth.Problem(16384, 16384, 64, beta=0.0)
    s = bench.mode_figures("tf32", skinny, 0.2, pk)
    ai = 2 * 16384 * 16384 * 64 / bench.alg_bytes(skinny)
    assert s["bound"] == "hbm" and abs(s["roofline_tflops"] - ai * 6800.0 / 1e3) < 1e-9
    assert bench.alg_bytes(skinny) == 4 * (16384 * 64 * 2 + 16384 * 16384)
    cfg = bench.make_config("square8192", bench.WORKLOADS["square8192"][1], ["ffma"], 1)
    assert cfg["l2"].startswith("inputs larger than L2") and cfg["parallelism"] == "single GPU"
    assert bench.make_config("square8192", bench.WORKLOADS["square8192"][1], ["ffma"], 4)["parallelism"] == "replicas"
    assert set(bench.SWEEP) <= set(synth.config_problems())


def test_roofline_traffic_comes_only_from_a_matching_profile():
    """roofline.traffic is read from the committed summary of the dominant kernel
    only while the kernel source hash and the tile shape the planner picks both
    match the ones the capture was taken on; otherwise it is null."""
    sys.path.insert(0, ROOT)
    import bench
    import hashlib
    text = open(os.path.join(ROOT, "profiles", "ffma_square8192.md")).read()
    fields = dict(line.split(":", 1) for line in text.splitlines() if ":" in line and not line.startswith("#"))
    tile = fields["tile"].strip()
    want = int(fields["traffic_bytes_per_launch"].strip())
    src = os.path.join(ROOT, "precision_gemm_gb300", "csrc", "ffma_kernel.cu")
    current = hashlib.sha256(open(src, "rb").read()).hexdigest() == fields["source_sha256"].strip()
    got = bench.read_traffic("ffma", "ffma", tile, "square8192")
    assert got == (want if current else None)
    other = "128x128" if tile != "128x128" else "128x64"
    assert bench.read_traffic("ffma", "ffma", other, "square8192") is None
    assert bench.read_traffic("ffma", "ffma", tile, "no_such_workload") is None
