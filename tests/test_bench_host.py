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


def test_decode_bytes_fp8_cache_is_half_the_kv_bytes():
    b, n, hq, hk = 64, 28672, 8, 4
    kv16 = b * n * hk * 512 * 2 * 2
    kv8 = b * n * hk * 512 * 1 * 2
    other = bench.decode_bytes(b, n, hq, hk) - kv16
    assert bench.decode_bytes(b, n, hq, hk, kv_elem_bytes=1) == kv8 + other
    # several tokens add their q / out / lse rows, not K/V bytes
    assert (bench.decode_bytes(b, n, hq, hk, q_len=4) - bench.decode_bytes(b, n, hq, hk)
            == 3 * (b * hq * 512 * 2 * 2 + b * hq * 4))


def test_recorded_traffic_needs_the_current_source_digest():
    dec = bench.source_digest(["decode_sm103.cu", "fa512_device.cuh", "fa512_internal.h"])
    pf = bench.source_digest(["prefill_so_sm103.cu", "fa512_pair.cuh", "fa512_device.cuh",
                              "fa512_internal.h"])
    # a stale digest finds nothing; an unknown kernel finds nothing
    assert bench.recorded_traffic("decode_bf16_mma_kernel", "0" * 16) is None
    assert bench.recorded_traffic("no_such_kernel", dec) is None
    # a record taken on the current source holds at least the algorithmic
    # bytes of the shape it names (a source edited since has no record: None)
    pf_bytes = bench.recorded_traffic("prefill_kernel", pf)
    d_bytes = bench.recorded_traffic("decode_bf16_mma_kernel", dec)
    f_bytes = bench.recorded_traffic("decode_fp8_mma_kernel", dec)
    if pf_bytes is not None:
        assert pf_bytes >= 0.9 * 8192 * 32 * 512 * 2 * 2    # Q and O of the chunked config
    if d_bytes is not None:
        assert d_bytes >= 64 * 28672 * 4 * 512 * 2 * 2
    if f_bytes is not None:
        assert f_bytes >= 64 * 28672 * 4 * 512 * 2
