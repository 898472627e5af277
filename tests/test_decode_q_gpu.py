"""Parity of fa512_decode_paged_q -- several query tokens per sequence, the
last q_len positions of a paged cache -- (CUDA, through the C ABI) with the
fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from head_dim_flashattention_gb300 import workloads
from parity import compare_lse, compare_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    import head_dim_flashattention_gb300 as fa
    fa.load_library()
    return fa


def run(fa, pc, q, num_splits=0, window=0, dev="cuda"):
    out, lse = fa.fa512_decode_paged_q(q.to(dev), pc.k_pages.to(dev), pc.v_pages.to(dev),
                                       pc.page_table.to(dev), pc.kv_lens.to(dev),
                                       max_kv_len=pc.max_kv_len, num_splits=num_splits,
                                       window=window)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(fa, pc, q, num_splits=0, window=0):
    o, l = run(fa, pc, q, num_splits=num_splits, window=window)
    assert fa.fa512_device_status() == 0
    ro, rl = oracle.decode_paged_q(q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                   window=window)
    compare_o(o, ro)
    compare_lse(l, rl)
    return o, l


@pytest.mark.parametrize("q_len", [2, 4, 8])
def test_draft_tokens_8_over_4_heads(fa, q_len):
    """The decode config's heads (8 over 4, page 64) with q_len tokens per
    sequence, NaN-poisoned outside every live band."""
    pc = workloads.paged_decode_inputs(4, [4096, 777, 64, 3001], 8, 4, 64, seed=41)
    q = workloads.draft_queries(4, q_len, 8, seed=41 + q_len)
    check(fa, pc, q)


@pytest.mark.parametrize("hq,hk,q_len", [(16, 16, 16), (8, 1, 2), (12, 4, 5), (4, 4, 3)])
def test_groupings_up_to_16_rows(fa, hq, hk, q_len):
    pc = workloads.paged_decode_inputs(2, [513, 100], hq, hk, 64, seed=42)
    q = workloads.draft_queries(2, q_len, hq, seed=42)
    check(fa, pc, q)


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_split_invariance(fa, splits):
    pc = workloads.paged_decode_inputs(3, [1000, 64, 4097], 8, 4, 64, seed=43)
    q = workloads.draft_queries(3, 4, 8, seed=43)
    check(fa, pc, q, num_splits=splits)


@pytest.mark.parametrize("window", [1, 3, 50, 1000])
def test_windows_give_each_token_its_own_band(fa, window):
    pc = workloads.paged_decode_inputs(3, [40, 129, 3000], 8, 4, 64, seed=44)
    q = workloads.draft_queries(3, 4, 8, seed=44)
    check(fa, pc, q, window=window)
    check(fa, pc, q, window=window, num_splits=5)


@pytest.mark.parametrize("page_size", [16, 32, 128])
def test_page_sizes(fa, page_size):
    pc = workloads.paged_decode_inputs(3, [1, 33, 700], 8, 4, page_size, seed=45)
    q = workloads.draft_queries(3, 4, 8, seed=45)
    check(fa, pc, q)


def test_caches_shorter_than_the_draft(fa):
    """A query whose position would be negative (kv_len < q_len) sees nothing:
    O = 0, LSE = -inf; the others see the keys up to their own position."""
    pc = workloads.paged_decode_inputs(3, [0, 2, 5], 8, 4, 64, seed=46)
    q = workloads.draft_queries(3, 4, 8, seed=46)
    o, l = check(fa, pc, q)
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    assert np.all(o[1, :2] == 0) and np.all(np.isneginf(l[1, :2]))
    assert np.all(np.isfinite(l[1, 2:])) and np.all(np.isfinite(l[2]))


def test_q_len_one_matches_single_token_decode_bitwise(fa):
    pc = workloads.paged_decode_inputs(2, [3000, 129], 8, 4, 64, seed=47)
    o1, l1 = fa.fa512_decode_paged(pc.q.cuda(), pc.k_pages.cuda(), pc.v_pages.cuda(),
                                   pc.page_table.cuda(), pc.kv_lens.cuda(), max_kv_len=pc.max_kv_len)
    o2, l2 = fa.fa512_decode_paged_q(pc.q[:, None].cuda(), pc.k_pages.cuda(), pc.v_pages.cuda(),
                                     pc.page_table.cuda(), pc.kv_lens.cuda(),
                                     max_kv_len=pc.max_kv_len)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:, 0]) and torch.equal(l1, l2[:, 0])


def test_rows_past_sixteen_are_rejected(fa):
    pc = workloads.paged_decode_inputs(1, [100], 8, 4, 64, seed=48)
    q = workloads.draft_queries(1, 9, 8, seed=48)
    with pytest.raises(fa.Fa512Error):
        run(fa, pc, q)
