"""Parity of fa512_prefill_d256 (heads of 256 dimensions, the sliding-window
local layers; CUDA through the C ABI) with the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flashattention_gb300 import workloads
from parity import compare_lse, compare_o

pytestmark = pytest.mark.gpu
D = 256


@pytest.fixture(scope="module")
def fa(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    import head_dim_flashattention_gb300 as fa
    fa.load_library()
    return fa


def rand(shape, seed):
    return workloads.randn_bf16(shape, seed)


def run(fa, q, k, v, **kw):
    out, lse = fa.fa512_prefill_d256(q.cuda(), k.cuda(), v.cuda(), **kw)
    torch.cuda.synchronize()
    assert fa.fa512_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(fa, q, k, v, rows=None, **kw):
    o, l = run(fa, q, k, v, **kw)
    ro, rl = oracle.prefill(q, k, v, rows=rows, **kw)
    if rows is not None:
        o, l = o[rows], l[:, rows]
    compare_o(o, ro)
    compare_lse(l, rl)
    return o, l


@pytest.mark.parametrize("sq,sk,hq,hk,off,window", [
    (300, 300, 8, 1, 0, 1024),      # every row inside the window
    (1500, 1500, 8, 2, 0, 1024),    # window edges cross 128-key tiles
    (700, 2100, 32, 4, 1400, 1024), # a chunk at an offset
    (333, 333, 4, 4, 0, 100),       # G = 1, short window
    (260, 900, 6, 2, 640, 17),      # G = 3 (126-row tiles), window inside one tile
    (129, 129, 16, 1, 0, 1),        # a window of one key: O = V of the row's own position
    (400, 400, 32, 1, 0, 0),        # G = 32, full causal
    (1, 1, 2, 2, 0, 1024),
])
def test_shapes_and_windows(fa, sq, sk, hq, hk, off, window):
    q, k, v = rand((sq, hq, D), 1), rand((sk, hk, D), 2), rand((sk, hk, D), 3)
    check(fa, q, k, v, q_offset=off, window=window)


def test_non_causal(fa):
    q, k, v = rand((77, 8, D), 4), rand((390, 4, D), 5), rand((390, 4, D), 6)
    check(fa, q, k, v, causal=False)
    check(fa, q, k, v, causal=False, window=64, q_offset=200)


def test_items_without_keys_between_items_with_keys(fa):
    """Rows past the end of the keys by more than the window see nothing
    (O = 0, LSE = -inf) while earlier rows of the same range see keys."""
    q, k, v = rand((600, 8, D), 7), rand((1500, 2, D), 8), rand((1500, 2, D), 9)
    o, l = check(fa, q, k, v, q_offset=2000, window=700)
    assert np.all(o[300:] == 0) and np.all(np.isneginf(l[:, 300:]))
    o, l = run(fa, q, k[:0], v[:0], q_offset=0, window=1024)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_window_one_returns_own_value(fa):
    q, k, v = rand((64, 8, D), 10), rand((64, 1, D), 11), rand((64, 1, D), 12)
    o, _ = run(fa, q, k, v, window=1)
    for i in (0, 13, 63):
        for h in range(8):
            np.testing.assert_array_equal(o[i, h], v[i, 0].float().numpy())


def test_q0_v1_is_exactly_one(fa):
    n = 8192
    q = torch.zeros((n, 8, D), dtype=torch.bfloat16)
    k = rand((n, 1, D), 13)
    v = torch.ones((n, 1, D), dtype=torch.bfloat16)
    o, l = run(fa, q, k, v, window=1024)
    assert np.all(o == 1.0)
    np.testing.assert_allclose(l[:, -1], math.log(1024), atol=1e-3)


def test_local_layer_workload_sampled_rows(fa):
    """The 20k-token local-layer config (window 1024, 32 over 4 heads): every
    cluster walks many items; sampled rows against the oracle."""
    cfg = workloads.PREFILL_CONFIGS["local256"]
    q, k, v = workloads.prefill_inputs(cfg)
    rows = workloads.sample_rows(cfg, tokens_per_tile=16, every=331)
    check(fa, q, k, v, rows=rows, q_offset=cfg.q_offset, window=cfg.window, scale=cfg.scale)


def test_repeat_calls_are_bitwise_identical(fa):
    q, k, v = rand((3000, 8, D), 14), rand((3000, 2, D), 15), rand((3000, 2, D), 16)
    o1, l1 = run(fa, q, k, v, window=1024)
    o2, l2 = run(fa, q, k, v, window=1024)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
