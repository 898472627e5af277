"""Parity of fa512_decode_paged_fp8 -- decode over a paged KV cache stored in
FP8 E4M3 with per-tensor K and V scales (vllm-project/flash-attention PR
#199, "Summary") -- (CUDA, through the C ABI) with the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from head_dim_flashattention_gb300 import workloads
from parity import compare_lse, compare_o

pytestmark = pytest.mark.gpu
D = 512
# scales that are not powers of two, so every dequantised value is rounded
# differently from the bf16 grid
K_SCALE, V_SCALE = 0.0371, 0.0517


@pytest.fixture(scope="module")
def fa(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    import head_dim_flashattention_gb300 as fa
    fa.load_library()
    return fa


def run(fa, pc, q=None, k_pages=None, v_pages=None, k_scale=K_SCALE, v_scale=V_SCALE,
        num_splits=0, window=0, scale=None, max_kv_len=None):
    q = pc.q if q is None else q
    kp = pc.k_pages if k_pages is None else k_pages
    vp = pc.v_pages if v_pages is None else v_pages
    out, lse = fa.fa512_decode_paged_fp8(
        q.cuda(), kp.cuda(), vp.cuda(), pc.page_table.cuda(), pc.kv_lens.cuda(),
        k_scale=k_scale, v_scale=v_scale, scale=scale, window=window, num_splits=num_splits,
        max_kv_len=pc.max_kv_len if max_kv_len is None else max_kv_len)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(fa, pc, q=None, k_scale=K_SCALE, v_scale=V_SCALE, num_splits=0, window=0, scale=None):
    """GPU vs oracle.  A one-key window (window 1) makes every output a single
    dequantised value that bf16 cannot hold: that case is compared with the
    mean of the error beyond the bf16 rounding floor (tests/parity.py)."""
    q = pc.q if q is None else q
    o, l = run(fa, pc, q=q, k_scale=k_scale, v_scale=v_scale, num_splits=num_splits,
               window=window, scale=scale)
    assert fa.fa512_device_status() == 0
    ro, rl = oracle.decode_paged_fp8(q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                     k_scale=k_scale, v_scale=v_scale, window=window,
                                     scale=scale)
    compare_o(o, ro, one_key_fp8=(window == 1))
    compare_lse(l, rl)
    return o, l


def fp8_cache(batch, lens, hq=8, hk=4, page=64, seed=70, **kw):
    pc, _, _ = workloads.paged_fp8_inputs(batch, lens, hq, hk, page, seed=seed,
                                          k_scale=K_SCALE, v_scale=V_SCALE, **kw)
    return pc


@pytest.mark.parametrize("batch,kv_len", [(1, 4096), (1, 16384), (1, 28672), (16, 4096),
                                          (16, 16384), (16, 28672), (64, 4096)])
def test_decode_shapes(fa, batch, kv_len):
    """The decode table's shapes (8 q heads over 4 KV heads, page 64, q_len 1)
    with an FP8 cache, NaN codes in every slot outside a live band."""
    check(fa, fp8_cache(batch, [kv_len] * batch, seed=70 + batch))


@pytest.mark.parametrize("hq,hk,q_len", [(4, 4, 1), (8, 4, 1), (8, 4, 3), (16, 2, 2),
                                         (16, 1, 1), (12, 4, 5)])
def test_groupings_and_tokens(fa, hq, hk, q_len):
    """Up to 8 (token, head) rows take the streaming tensor-core kernel
    (f16 products of the exactly widened bytes); more rows take the split
    kernel that converts each FP8 tile into a bf16 tile."""
    pc = fp8_cache(3, [513, 100, 1], hq, hk, seed=71)
    q = workloads.draft_queries(3, q_len, hq, seed=71) if q_len > 1 else pc.q
    check(fa, pc, q=q)


@pytest.mark.parametrize("splits", [1, 3, 64, 1024])
def test_split_invariance(fa, splits):
    pc = fp8_cache(3, [1000, 64, 4097], seed=72)
    check(fa, pc, num_splits=splits)
    q = workloads.draft_queries(3, 4, 8, seed=72)
    check(fa, pc, q=q, num_splits=splits)


@pytest.mark.parametrize("window", [1, 3, 50, 1000])
def test_window_band(fa, window):
    pc = fp8_cache(3, [40, 129, 3000], seed=73)
    check(fa, pc, window=window)
    check(fa, pc, window=window, num_splits=5)
    check(fa, pc, q=workloads.draft_queries(3, 4, 8, seed=73), window=window)


@pytest.mark.parametrize("page_size", [16, 32, 128, 256])
def test_page_sizes(fa, page_size):
    pc = fp8_cache(4, [1, 31, 33, 700], page=page_size, seed=74)
    check(fa, pc)
    check(fa, pc, q=workloads.draft_queries(4, 2, 8, seed=74))


def test_empty_and_short_sequences(fa):
    pc = fp8_cache(3, [0, 2, 5], seed=75)
    o, l = check(fa, pc, num_splits=4)
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    q = workloads.draft_queries(3, 4, 8, seed=75)
    o, l = check(fa, pc, q=q)
    assert np.all(o[1, :2] == 0) and np.all(np.isneginf(l[1, :2]))


def _dequant_bf16(pages_u8, scale):
    # exact when scale is a power of two
    return (pages_u8.view(torch.float8_e4m3fn).float() * scale).to(torch.bfloat16)


@pytest.mark.parametrize("hq,hk,q_len", [(16, 2, 2), (16, 1, 1), (12, 4, 3)])
def test_split_path_equals_bf16_decode_bitwise(fa, hq, hk, q_len):
    """More than 8 rows: with power-of-two scales the dequantised cache is a
    bf16 cache, and the split kernel converts each FP8 tile exactly into the
    bf16 tile the bf16 split kernel reads, so the two calls agree bit for bit."""
    s = 1.0 / 32
    pc = fp8_cache(3, [3000, 129, 64], hq, hk, seed=76)
    q = workloads.draft_queries(3, q_len, hq, seed=76)
    o8, l8 = fa.fa512_decode_paged_fp8(q.cuda(), pc.k_pages.cuda(), pc.v_pages.cuda(),
                                       pc.page_table.cuda(), pc.kv_lens.cuda(), k_scale=s,
                                       v_scale=s, max_kv_len=pc.max_kv_len)
    o16, l16 = fa.fa512_decode_paged_q(q.cuda(), _dequant_bf16(pc.k_pages, s).cuda(),
                                       _dequant_bf16(pc.v_pages, s).cuda(), pc.page_table.cuda(),
                                       pc.kv_lens.cuda(), max_kv_len=pc.max_kv_len)
    torch.cuda.synchronize()
    assert torch.equal(o8, o16) and torch.equal(l8, l16)


@pytest.mark.parametrize("hq,hk,q_len", [(8, 4, 1), (4, 4, 1), (8, 4, 4), (16, 4, 2), (8, 1, 1)])
def test_streaming_path_agrees_with_bf16_decode(fa, hq, hk, q_len):
    """Up to 8 rows: the FP8 kernel's f16 tensor-core products of the exactly
    widened cache against the bf16 decode of the same values (power-of-two
    scales): the scores are the same exact products summed in another order,
    P is rounded to f16 instead of kept in fp32 or rounded to bf16, so the two
    agree within the rounding of the output."""
    s = 1.0 / 16
    pc = fp8_cache(4, [4096, 777, 64, 1], hq, hk, seed=77)
    q = workloads.draft_queries(4, q_len, hq, seed=77)
    o8, l8 = run(fa, pc, q=q, k_scale=s, v_scale=s)
    o16, l16 = fa.fa512_decode_paged_q(q.cuda(), _dequant_bf16(pc.k_pages, s).cuda(),
                                       _dequant_bf16(pc.v_pages, s).cuda(), pc.page_table.cuda(),
                                       pc.kv_lens.cuda(), max_kv_len=pc.max_kv_len)
    torch.cuda.synchronize()
    # two bf16 spacings relative, plus the fp32 rounding of small values
    np.testing.assert_allclose(o8, o16.float().cpu().numpy(), atol=2e-3, rtol=8e-3)
    fin = np.isfinite(l8)
    assert np.array_equal(fin, np.isfinite(l16.cpu().numpy()))
    np.testing.assert_allclose(l8[fin], l16.cpu().numpy()[fin], atol=1e-5, rtol=0)


def test_large_and_small_query_rows(fa):
    """The tensor-core kernel scales each query row by a power of two before
    the f16 products, so rows far outside the f16 range keep their scores:
    one head's query times 2^20 (elements up to ~2^22, beyond f16's 65504)
    with the softmax scale times 2^-20, and one head's query times 2^-50
    (below f16's subnormals; its attention is uniform)."""
    pc = fp8_cache(2, [300, 4097], 8, 4, seed=83)
    q = pc.q.clone()
    q[:, 0] *= 2.0 ** 20
    q[1, 5] *= 2.0 ** -50
    check(fa, pc, q=q, scale=D ** -0.5 * 2.0 ** -20)


@pytest.mark.parametrize("q_len", [1, 4])
def test_q0_v1_long_split_is_exact(fa, q_len):
    """PR #199 review: with q = 0 and V = 1 the output must be 1 (here
    v_scale) at every length; the FP8 WGMMA kernel returned 0.5 at 32K keys
    and 0.125 at 128K with one split.  Here: 131072 keys, one split."""
    n = 131072
    pc = fp8_cache(1, [n], 8, 4, seed=78, spare_pages=1)
    q = torch.zeros((1, q_len, 8, D), dtype=torch.bfloat16)
    ones = torch.full_like(pc.v_pages, 0x38)      # e4m3 1.0
    for splits in (1, 7):
        o, l = run(fa, pc, q=q, v_pages=ones, k_scale=0.25, v_scale=0.5, num_splits=splits)
        assert np.all(o == 0.5)
        ref = [math.log(n - q_len + 1 + t) for t in range(q_len)]
        np.testing.assert_allclose(l[0], np.array(ref)[:, None].repeat(8, 1), atol=1e-3)


def test_late_key_softmax_tail(fa):
    """PR #199 review F1: one key ahead by 12 logits among n = 131072 keys
    carries the weight e^12 / (e^12 + n - 1); the value channels give that
    weight and 1 exactly (closed form), and the GPU matches the oracle."""
    n = 131072
    pc = fp8_cache(1, [n], 2, 1, seed=79, spare_pages=1)
    k = torch.zeros_like(pc.k_pages)
    v = torch.zeros_like(pc.v_pages)
    last = int(pc.page_table[0, (n - 1) // 64])
    k[last, (n - 1) % 64, 0, 0] = 0x48             # 4.0
    v[:, :, 0, 1] = 0x38                           # 1.0 in channel 1 everywhere
    v[last, (n - 1) % 64, 0, 0] = 0x38             # 1.0 in channel 0 for the late key
    q = torch.zeros_like(pc.q)
    q[0, :, 0] = 3.0
    o, l = run(fa, pc, q=q, k_pages=k, v_pages=v, k_scale=1.0, v_scale=1.0, scale=1.0,
               num_splits=1)
    w = math.exp(12) / (math.exp(12) + n - 1)
    np.testing.assert_allclose(o[0, :, 0], w, atol=3e-3)   # bf16 half spacing at 0.55: 2e-3
    assert np.all(o[0, :, 1] == 1.0)
    np.testing.assert_allclose(l[0], math.log(math.exp(12) + n - 1), atol=1e-3)
    ro, rl = oracle.decode_paged_fp8(q, k, v, pc.page_table, pc.kv_lens, scale=1.0)
    compare_o(o, ro)
    compare_lse(l, rl)


def test_float8_dtype_is_accepted(fa):
    pc = fp8_cache(2, [300, 64], seed=80)
    o1, l1 = run(fa, pc)
    o2, l2 = run(fa, pc, k_pages=pc.k_pages.view(torch.float8_e4m3fn),
                 v_pages=pc.v_pages.view(torch.float8_e4m3fn))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_bad_page_index_is_reported_not_read(fa):
    pc = fp8_cache(2, [200, 100], seed=81)
    pc.page_table[1, 0] = 10 ** 6
    run(fa, pc)
    assert fa.fa512_device_status() == 6
    assert fa.fa512_device_status() == 0


def test_rejected_arguments(fa):
    pc = fp8_cache(1, [100], seed=82)
    with pytest.raises(fa.Fa512Error):
        run(fa, pc, k_scale=float("inf"))
    with pytest.raises(fa.Fa512Error):
        run(fa, pc, v_scale=float("nan"))
    with pytest.raises(fa.Fa512Error):
        run(fa, pc, q=workloads.draft_queries(1, 9, 8, seed=82))
    with pytest.raises(fa.Fa512Error):
        # a bf16 cache is not an FP8 cache
        fa.fa512_decode_paged_fp8(pc.q.cuda(), pc.k_pages.cuda().to(torch.bfloat16),
                                  pc.v_pages.cuda().to(torch.bfloat16), pc.page_table.cuda(),
                                  pc.kv_lens.cuda())
