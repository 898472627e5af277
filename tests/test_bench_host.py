"""Host-side pieces of bench.py: the FLOP convention and the reference arm."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def read_golden(name):
    vals = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    return vals


def test_flop_convention_reproduces_the_pages_131_tflop():
    g = read_golden("flop_convention.txt")
    n = int(g["tokens"])
    per_layer = bench.prefill_flops(n, n, 0, int(g["n_q_heads"]))
    total = per_layer * int(g["layers"])
    assert round(total / 1e12) == int(g["tflop"])


def test_visible_pairs_closed_forms():
    # causal square: n (n + 1) / 2
    assert bench.visible_pairs(100, 100, 0) == 100 * 101 // 2
    # bottom-right chunk: rows see q_offset + i + 1 keys
    assert bench.visible_pairs(8192, 16384, 8192) == sum(8192 + i + 1 for i in range(8192))
    # window W: every row past W-1 sees exactly W keys
    assert bench.visible_pairs(10, 10, 0, window=3) == 1 + 2 + 3 * 8
    assert bench.visible_pairs(5, 7, 0, causal=False) == 35


def test_decode_bytes_counts_live_kv():
    b, n = 64, 28672
    assert bench.decode_bytes(b, n, 8, 4) >= b * n * 4 * 512 * 2 * 2


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--ref-rows", "2"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
