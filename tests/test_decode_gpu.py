"""Parity of fa512_decode_paged (CUDA, through the C ABI) with the fp64 oracle."""
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


def run(fa, pc, num_splits=0, window=0, max_kv_len=None, dev="cuda", q=None, v_pages=None):
    q = pc.q if q is None else q
    vp = pc.v_pages if v_pages is None else v_pages
    out, lse = fa.fa512_decode_paged(q.to(dev), pc.k_pages.to(dev), vp.to(dev),
                                     pc.page_table.to(dev), pc.kv_lens.to(dev),
                                     max_kv_len=pc.max_kv_len if max_kv_len is None else max_kv_len,
                                     num_splits=num_splits, window=window)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(fa, pc, num_splits=0, window=0):
    o, l = run(fa, pc, num_splits=num_splits, window=window)
    assert fa.fa512_device_status() == 0
    ro, rl = oracle.decode_paged(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                 window=window)
    compare_o(o, ro)
    compare_lse(l, rl)
    return o, l


@pytest.mark.parametrize("name", sorted(workloads.DECODE_CONFIGS))
def test_decode_configs(fa, name):
    """Batch {1,16,64} x KV {4K,16K,28K}, 8 q heads over 4 KV heads, page 64,
    NaN-poisoned outside every live band, num_splits auto."""
    cfg = workloads.DECODE_CONFIGS[name]
    check(fa, workloads.decode_inputs(cfg))


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 1024])
def test_split_invariance(fa, splits):
    # 3 sequences x 8 heads = 24 rows: the merge takes each row in four
    # column slices (128 splits loaded up front, the rest in its loop)
    pc = workloads.paged_decode_inputs(3, [1000, 64, 4097], 8, 4, 64, seed=31)
    check(fa, pc, num_splits=splits)


@pytest.mark.parametrize("splits", [33, 100, 1024])
def test_split_invariance_whole_rows(fa, splits):
    # 6 sequences x 8 heads = 48 rows: the merge takes whole rows (32 splits
    # loaded up front, the rest in its unrolled loop, with a remainder)
    pc = workloads.paged_decode_inputs(6, [1000, 64, 4097, 0, 2500, 3333], 8, 4, 64, seed=41)
    check(fa, pc, num_splits=splits)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
def test_page_sizes(fa, page_size):
    pc = workloads.paged_decode_inputs(4, [1, 31, 33, 700], 8, 4, page_size, seed=32)
    check(fa, pc)


@pytest.mark.parametrize("hq,hk", [(16, 1), (4, 4), (8, 1), (12, 4)])
def test_head_groupings(fa, hq, hk):
    pc = workloads.paged_decode_inputs(2, [513, 100], hq, hk, 64, seed=33)
    check(fa, pc)


@pytest.mark.parametrize("window", [1, 50, 64, 1000])
def test_window_band(fa, window):
    pc = workloads.paged_decode_inputs(3, [40, 129, 3000], 8, 4, 64, seed=34)
    check(fa, pc, window=window, num_splits=0)
    check(fa, pc, window=window, num_splits=5)


def test_empty_sequences(fa):
    pc = workloads.paged_decode_inputs(3, [0, 5, 0], 8, 4, 64, seed=35)
    o, l = check(fa, pc, num_splits=4)
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))


def test_q0_v1_long_is_exactly_one(fa):
    pc = workloads.paged_decode_inputs(2, [28672, 28672], 8, 4, 64, seed=36, spare_pages=2)
    q = torch.zeros_like(pc.q)
    v = torch.ones_like(pc.v_pages)
    for splits in (1, 9):
        o, l = run(fa, pc, num_splits=splits, q=q, v_pages=v)
        assert np.all(o == 1.0)
        np.testing.assert_allclose(l, math.log(28672), atol=1e-3)


def test_agrees_with_prefill_last_row(fa):
    """A decode step equals the last row of a prefill over the same keys."""
    n, hq, hk = 777, 8, 4
    pc = workloads.paged_decode_inputs(1, [n], hq, hk, 64, seed=37)
    npg = (n + 63) // 64
    idx = pc.page_table[0, :npg].long()
    k_lin = pc.k_pages[idx].reshape(npg * 64, hk, D)[:n].contiguous()
    v_lin = pc.v_pages[idx].reshape(npg * 64, hk, D)[:n].contiguous()
    od, ld = run(fa, pc)
    op, lp = fa.fa512_prefill(pc.q[0][None].cuda(), k_lin.cuda(), v_lin.cuda(), q_offset=n - 1)
    torch.cuda.synchronize()
    np.testing.assert_allclose(od[0], op[0].float().cpu().numpy(), atol=1e-2)
    np.testing.assert_allclose(ld[0], lp[:, 0].cpu().numpy(), atol=1e-3)


def test_bad_page_index_is_reported_not_read(fa):
    pc = workloads.paged_decode_inputs(2, [200, 100], 8, 4, 64, seed=38)
    pc.page_table[1, 0] = 10 ** 6
    run(fa, pc)
    assert fa.fa512_device_status() == 6   # FA512_ERR_DEVICE_INDEX
    assert fa.fa512_device_status() == 0   # cleared


def test_kv_len_beyond_bound_is_reported(fa):
    pc = workloads.paged_decode_inputs(1, [300], 8, 4, 64, seed=39)
    run(fa, pc, max_kv_len=200)
    assert fa.fa512_device_status() == 6
