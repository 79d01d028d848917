"""The benchmark's reference arm (the oracle timed on the host cores) keeps
the JSON-line contract, and under a multi-rank launch only rank 0 prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       cwd=ROOT, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_reference_arm_json_line():
    # the 131,072-node workload keeps the graph generation on the CPU short
    out = _run(["--impl", "reference", "--workload", "gcn3-rmat17-131k", "--steps", "1",
                "--warmup", "0"]).strip().splitlines()
    line = json.loads(out[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["unit"] == "edges/s" and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["config"]["workload"] == "gcn3-rmat17-131k"
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert "scaled linearly" in line["cpu_baseline"]["sample"] and line["scaled_step_s"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    out = _run(["--impl", "reference", "--workload", "gcn3-rmat17-131k", "--steps", "1", "--warmup", "0"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.strip() == ""


def test_single_gpu_workloads_other_ranks_are_silent():
    for wl in ("gat-rmat20-1m", "aggregate-rmat24-16.8m"):
        out = _run(["--workload", wl, "--steps", "1", "--warmup", "0"], {"RANK": "1", "WORLD_SIZE": "2",
                                                                         "LOCAL_RANK": "1"})
        assert out.strip() == ""


def test_aggregation_bytes_by_hand():
    """The roofline numerator: compulsory bytes of one aggregation, worked by
    hand for a small case (n = 10 rows, 30 edges, d = 64, b = 2, 4 marginal
    rows): row pointers, column ids, the two degree norms, the mask, each
    packed row once, each fp32 row once, the output; a gated launch adds the
    gate bits (ceil(64 / 32) words per row)."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    import quantized_gnn_message_gb300 as q
    from quantized_gnn_message_gb300 import build
    build.build()  # the host-side pitch query of libgq (no GPU needed)
    pitch = q.packed_pitch(64, 2)
    assert pitch == 32  # 8-byte header after 16 payload bytes, padded to 16
    meta = 11 * 4 + 30 * 4 + 2 * 10 * 4 + 10
    comp, stream = bench.spmm_bytes(10, 30, 64, 2, 4, 12, 2, q)
    assert comp == meta + 4 * pitch + 6 * 64 * 4 + 10 * 64 * 2
    # streaming: metadata read per edge (column id and coefficient), the mask
    # byte per edge, every gathered row
    assert stream == 11 * 4 + 30 * 8 + 30 + 10 * 4 + 10 * 64 * 2 + 12 * pitch + 18 * 64 * 4
    comp_g, _ = bench.spmm_bytes(10, 30, 64, 2, 4, 12, 2, q, gated=True)
    assert comp_g - comp == 10 * 2 * 4
