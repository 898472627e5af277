"""Parity of fa512_prefill_paged (CUDA, through the C ABI) with the fp64 oracle:
a batch of prefill chunks of different lengths over a paged KV cache."""
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


def make(lens_k, lens_q, hq, hk, page, seed, poison=True):
    """Paged cache (NaN in every slot no sequence uses, out-of-range entries in
    unused table slots) and packed chunk rows."""
    pc = workloads.paged_decode_inputs(len(lens_k), lens_k, hq, hk, page, seed=seed,
                                       poison=poison)
    q, cu = workloads.varlen_queries(lens_q, hq, seed=seed)
    return pc, q, cu, torch.tensor(lens_k, dtype=torch.int32)


def run(fa, pc, q, cu, used, max_seqlen_q=None, expect_status=0, **kw):
    dev = "cuda"
    if max_seqlen_q is None:
        max_seqlen_q = int((cu[1:] - cu[:-1]).max()) if cu.numel() > 1 else 0
    out, lse = fa.fa512_prefill_paged(q.to(dev), pc.k_pages.to(dev), pc.v_pages.to(dev),
                                      pc.page_table.to(dev), cu.to(dev), used.to(dev),
                                      max_seqlen_q=max_seqlen_q, **kw)
    torch.cuda.synchronize()
    assert fa.fa512_device_status() == expect_status
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(fa, pc, q, cu, used, **kw):
    o, l = run(fa, pc, q, cu, used, **kw)
    ro, rl = oracle.prefill_paged(q, pc.k_pages, pc.v_pages, pc.page_table, cu, used, **kw)
    st = compare_o(o, ro)
    compare_lse(l, rl)
    return o, l, st


def test_varlen_batch_over_poisoned_pages(fa):
    """Whole prompts, chunks at an offset, page-aligned and ragged lengths."""
    lens_k = [300, 129, 64, 1000, 7, 200]
    lens_q = [300, 50, 64, 129, 7, 1]
    pc, q, cu, used = make(lens_k, lens_q, 8, 2, 64, seed=51)
    check(fa, pc, q, cu, used)


@pytest.mark.parametrize("page", [64, 128, 256])
@pytest.mark.parametrize("tail", [0, 1, 63, 65, 127])
def test_page_sizes_and_cache_tails(fa, page, tail):
    """Cache lengths ending anywhere in a 128-key tile: the rows past the end
    of the last page hold NaN and must not reach O."""
    n = 256 + tail
    pc, q, cu, used = make([n, n + 64], [n, 100], 8, 4, page, seed=52 + tail)
    check(fa, pc, q, cu, used)


@pytest.mark.parametrize("hq,hk", [(32, 4), (16, 1), (6, 2), (4, 4), (12, 4)])
def test_groupings(fa, hq, hk):
    pc, q, cu, used = make([333, 90], [200, 90], hq, hk, 64, seed=53)
    check(fa, pc, q, cu, used)


@pytest.mark.parametrize("window", [1, 17, 100, 1000])
def test_sliding_windows(fa, window):
    pc, q, cu, used = make([400, 150, 70], [300, 150, 5], 8, 2, 64, seed=54)
    check(fa, pc, q, cu, used, window=window)


def test_non_causal(fa):
    pc, q, cu, used = make([190, 77], [77, 30], 8, 4, 64, seed=55)
    check(fa, pc, q, cu, used, causal=False)


def test_empty_caches_empty_chunks_and_short_caches(fa):
    """A cache shorter than its chunk leaves the first rows with negative
    positions (O = 0, LSE = -inf); an empty cache empties every row; an empty
    chunk writes nothing."""
    lens_k = [0, 10, 100, 50]
    lens_q = [5, 40, 0, 50]
    pc, q, cu, used = make(lens_k, lens_q, 8, 2, 64, seed=56)
    o, l, _ = check(fa, pc, q, cu, used)
    assert np.all(o[:5] == 0) and np.all(np.isneginf(l[:, :5]))
    assert np.all(o[5:35] == 0) and np.all(np.isneginf(l[:, 5:35]))


def test_bitwise_equal_to_contiguous_prefill(fa):
    """One sequence through a shuffled page table gives the contiguous
    kernel's bits: same tiles, same arithmetic, only the addresses differ."""
    n, s, hq, hk = 1000, 700, 32, 4
    pc, q, cu, used = make([n], [s], hq, hk, 64, seed=57)
    o_p, l_p = run(fa, pc, q, cu, used)
    npg = (n + 63) // 64
    idx = pc.page_table[0, :npg].long()
    k_lin = pc.k_pages[idx].reshape(npg * 64, hk, D)[:n].contiguous()
    v_lin = pc.v_pages[idx].reshape(npg * 64, hk, D)[:n].contiguous()
    o_c, l_c = fa.fa512_prefill(q.cuda(), k_lin.cuda(), v_lin.cuda(), q_offset=n - s)
    torch.cuda.synchronize()
    assert np.array_equal(o_p, o_c.float().cpu().numpy())
    assert np.array_equal(l_p, l_c.cpu().numpy())


def test_chunked_config_through_a_page_table_sampled_rows(fa):
    """The chunked workload (8192 rows after 8192 cached, 32 over 4 heads)
    with its keys in shuffled 64-key pages: sampled rows against the oracle,
    every row bit-equal to the contiguous kernel."""
    cfg = workloads.PREFILL_CONFIGS["chunked"]
    n, s = cfg.seqlen_k, cfg.seqlen_q
    pc, q, cu, used = make([n], [s], cfg.n_q_heads, cfg.n_kv_heads, 64, seed=58)
    o, l = run(fa, pc, q, cu, used)
    npg = n // 64
    idx = pc.page_table[0, :npg].long()
    k_lin = pc.k_pages[idx].reshape(n, cfg.n_kv_heads, D)
    v_lin = pc.v_pages[idx].reshape(n, cfg.n_kv_heads, D)
    rows = workloads.sample_rows(cfg, tokens_per_tile=16, every=997)
    ro, rl = oracle.prefill(q, k_lin, v_lin, rows=rows, q_offset=n - s)
    compare_o(o[rows], ro)
    compare_lse(l[:, rows], rl)
    o_c, l_c = fa.fa512_prefill(q.cuda(), k_lin.cuda(), v_lin.cuda(), q_offset=n - s)
    torch.cuda.synchronize()
    assert np.array_equal(o, o_c.float().cpu().numpy())


def test_out_of_range_pages_and_lengths_are_recorded_not_read(fa):
    """Bad device-side metadata sets the device error word
    (FA512_ERR_DEVICE_INDEX) and is read as zeros or clipped, never out of
    bounds; the library stays usable."""
    pc, q, cu, used = make([200, 100], [100, 100], 8, 2, 64, seed=59)
    bad = pc.page_table.clone()
    bad[0, 1] = 10_000
    run(fa, workloads.PagedCache(pc.q, pc.k_pages, pc.v_pages, bad, pc.kv_lens, pc.max_kv_len),
        q, cu, used, expect_status=6)
    assert fa.fa512_device_status() == 0
    # a cache length beyond the page table's capacity
    run(fa, pc, q, cu, torch.tensor([200, 10_000], dtype=torch.int32), expect_status=6)
    # a chunk longer than the host-side bound
    run(fa, pc, q, cu, used, max_seqlen_q=50, expect_status=6)
    # and a clean call afterwards
    check(fa, pc, q, cu, used)


def test_repeat_calls_are_bitwise_identical(fa):
    pc, q, cu, used = make([500, 260], [300, 260], 16, 2, 128, seed=60)
    o1, l1 = run(fa, pc, q, cu, used)
    o2, l2 = run(fa, pc, q, cu, used)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
