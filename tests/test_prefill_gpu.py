"""Parity of fa512_prefill (CUDA, through the C ABI) with the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flashattention_gb300 import workloads
from parity import compare_lse, compare_o

pytestmark = pytest.mark.gpu
D = 512


@pytest.fixture(scope="module")
def fa(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    import head_dim_flashattention_gb300 as fa
    fa.load_library()
    return fa


def run(fa, q, k, v, q_offset=0, causal=True, window=0, scale=None, dev="cuda"):
    out, lse = fa.fa512_prefill(q.to(dev), k.to(dev), v.to(dev), q_offset=q_offset, scale=scale,
                                causal=causal, window=window)
    torch.cuda.synchronize()
    assert fa.fa512_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(fa, q, k, v, rows=None, stress=False, **kw):
    o, l = run(fa, q, k, v, **kw)
    ro, rl = oracle.prefill(q, k, v, rows=rows, **kw)
    if rows is not None:
        o, l = o[rows], l[:, rows]
    st = compare_o(o, ro, stress=stress)
    compare_lse(l, rl)
    return st


def rand(shape, seed):
    return workloads.randn_bf16(shape, seed)


def test_tiny_config(fa):
    cfg = workloads.PREFILL_CONFIGS["tiny"]
    q, k, v = workloads.prefill_inputs(cfg)
    check(fa, q, k, v, q_offset=cfg.q_offset, scale=cfg.scale, causal=cfg.causal)


@pytest.mark.parametrize("sq,sk,hq,hk,off", [
    (256, 256, 8, 1, 0),       # G = 8: 16 tokens per tile
    (100, 100, 8, 2, 0),       # ragged last q tile, keys not a multiple of 64
    (33, 97, 4, 4, 64),        # G = 1, chunk at an offset
    (70, 70, 16, 1, 0),        # MQA-style G = 16: 8 tokens per tile
    (50, 130, 6, 2, 80),       # G = 3: 42 tokens (126 rows) per tile
    (9, 200, 32, 1, 191),      # G = 32: 4 tokens per tile
    (1, 1, 2, 2, 0),
])
def test_shapes_causal(fa, sq, sk, hq, hk, off):
    q, k, v = rand((sq, hq, D), 1), rand((sk, hk, D), 2), rand((sk, hk, D), 3)
    check(fa, q, k, v, q_offset=off, causal=True)


@pytest.mark.parametrize("window", [1, 17, 64, 100])
def test_sliding_window(fa, window):
    q, k, v = rand((150, 8, D), 4), rand((150, 2, D), 5), rand((150, 2, D), 6)
    check(fa, q, k, v, causal=True, window=window)


def test_non_causal(fa):
    q, k, v = rand((77, 8, D), 7), rand((190, 4, D), 8), rand((190, 4, D), 9)
    check(fa, q, k, v, causal=False)


def test_empty_rows_and_empty_keys(fa):
    # window and offset leave no key for any row: O = 0, LSE = -inf
    q, k, v = rand((5, 4, D), 10), rand((4, 1, D), 11), rand((4, 1, D), 12)
    o, l = run(fa, q, k, v, q_offset=10, causal=True, window=2)
    assert np.all(o == 0) and np.all(np.isneginf(l))
    o, l = run(fa, q, k[:0], v[:0], q_offset=0)
    assert np.all(o == 0) and np.all(np.isneginf(l))
    # some rows empty, some not: keys exist only below position 20
    q, k, v = rand((40, 8, D), 13), rand((20, 2, D), 14), rand((20, 2, D), 15)
    check(fa, q, k, v, q_offset=10, causal=True, window=12)


def test_causal_row0_is_v0(fa):
    q, k, v = rand((64, 8, D), 16), rand((64, 1, D), 17), rand((64, 1, D), 18)
    o, l = run(fa, q, k, v)
    for h in range(8):
        np.testing.assert_array_equal(o[0, h], v[0, 0].float().numpy())


def test_q0_v1_long_is_exactly_one(fa):
    """PR #199 review: q = 0, V = 1 must give 1.000 at every length."""
    n = 32768
    q = torch.zeros((256, 8, D), dtype=torch.bfloat16)
    k = rand((n, 1, D), 19)
    v = torch.ones((n, 1, D), dtype=torch.bfloat16)
    o, l = run(fa, q, k, v, q_offset=n - 256)
    assert np.all(o == 1.0)
    np.testing.assert_allclose(l[:, -1], math.log(n), atol=1e-3)


def test_softmax_tail_late_key(fa):
    """PR #199 review item F1 at 32K keys: one late key ahead by 12."""
    n = 32768
    q = torch.zeros((1, 1, D), dtype=torch.bfloat16)
    q[0, 0, 0] = 3.0
    k = torch.zeros((n, 1, D), dtype=torch.bfloat16)
    k[n - 1, 0, 0] = 4.0
    v = torch.zeros((n, 1, D), dtype=torch.bfloat16)
    v[n - 1, 0, 0] = 1.0
    v[:, 0, 1] = 1.0
    o, l = run(fa, q, k, v, q_offset=n - 1, scale=1.0)
    w = math.exp(12) / (math.exp(12) + n - 1)
    assert abs(o[0, 0, 0] - w) <= 1e-2
    assert abs(o[0, 0, 1] - 1.0) <= 1e-2
    assert abs(l[0, 0] - math.log(math.exp(12) + n - 1)) <= 1e-3


def test_large_logits_stress_rows(fa):
    """Every 64th K row x8 forces large max rescales (the stress variant)."""
    cfg = workloads.PrefillConfig("s", 512, 512, 0, 8, 2, stress=True, seed=77)
    q, k, v = workloads.prefill_inputs(cfg)
    check(fa, q, k, v, causal=True, stress=True)


@pytest.mark.parametrize("name", ["chunked", "full_stress"])
def test_full_size_configs_sampled_rows(fa, name):
    cfg = workloads.PREFILL_CONFIGS[name]
    q, k, v = workloads.prefill_inputs(cfg)
    rows = workloads.sample_rows(cfg, tokens_per_tile=128 // (cfg.n_q_heads // cfg.n_kv_heads),
                                 every=997)
    check(fa, q, k, v, rows=rows, q_offset=cfg.q_offset, scale=cfg.scale, causal=cfg.causal,
          stress=cfg.stress)


def test_mqa_long_context_sampled_rows(fa):
    cfg = workloads.PREFILL_CONFIGS["mqa"]
    q, k, v = workloads.prefill_inputs(cfg)
    rows = [0, 1, 7, 8, 4095, 4096, 24575, 49144, 49151]
    check(fa, q, k, v, rows=rows, q_offset=cfg.q_offset, scale=cfg.scale, causal=cfg.causal)


def test_repeat_calls_are_bitwise_identical(fa):
    q, k, v = rand((300, 8, D), 20), rand((300, 1, D), 21), rand((300, 1, D), 22)
    o1, l1 = run(fa, q, k, v)
    o2, l2 = run(fa, q, k, v)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
