"""The benchmark's reference arm runs on the host alone: one JSON line with
the metric, the oracle's CPU baseline and the end-to-end block the contract
asks for (no GPU needed)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e",
                "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "varlen64k"
    assert d["gpu_launches"] == 0


def test_algorithmic_bytes_of_the_measured_workload():
    """The roofline numerator, counted by hand for the packed 64K workload
    (65536 tokens x 32 heads, dk = dv = 128, 8 documents with h0):
    forward q, k, v, o bf16 (2 B each) + a fp32 per (token, head), plus h0 in
    and hT out per (document, head); backward q, k, v, dO bf16 and a in, dq,
    dk, dv, da fp32 out, plus h0 per (document, head)."""
    sys.path.insert(0, ROOT)
    import bench
    from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS
    w = WORKLOADS["varlen64k"]
    th, units, state = 65536 * 32, 8 * 32, 128 * 128 * 4
    per_fwd = 2 * 128 * 4 + 4               # q, k, v, o at 2 B + a
    per_bwd = 2 * 128 * 4 + 4 + 4 * 128 * 3 + 4   # q, k, v, dO in + a; dq, dk, dv, da out
    assert (per_fwd, per_bwd) == (1028, 2568)
    got = bench.algorithmic_bytes(w, 8)
    assert got["fwd"] == th * per_fwd + 2 * units * state
    assert got["bwd"] == th * per_bwd + units * state
    assert got["bwd"] == 5402263552


def test_algorithmic_bytes_with_fp32_checkpoints():
    """The 256K stage as its config asks (fp32 state every 16 tokens): the
    forward also writes the 128-token block starts, the expansion kernel the
    7 inner states of every block (reading k, v and the tile cumsums once),
    and the backward reads one checkpoint per block."""
    sys.path.insert(0, ROOT)
    import bench
    from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS
    w = WORKLOADS["c256k"]
    th = 262144 * 16
    blocks = 262144 // 128 * 16
    state = 128 * 256 * 4
    got = bench.algorithmic_bytes(w, 1)
    assert got["states"] == th * (2 * 128 + 2 * 256 + 4) + blocks * 7 * state
    assert got["states"] == 33302773760
    plain = bench.algorithmic_bytes(WORKLOADS["c8k"], 4)
    assert "states" not in plain
    assert got["fwd"] - blocks * state == th * (2 * 128 * 2 + 2 * 256 + 4 + 2 * 256) + 16 * state
