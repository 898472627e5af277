"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

None of these re-types the oracle's formula: each case is built so that the
answer follows from a closed form, an invariance or a special case, and so
that a plausible slip in the oracle (a dropped max shift, a wrong head or
key index, a transposed operand, a misplaced scale, an off-by-one mask)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from head_dim_flashattention_gb300 import workloads

D = 512
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    """Round to bf16 (nearest even).  Cases that need exact values build them
    from small integers and dyadic fractions, or round first and reuse the
    rounded values on both sides."""
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split("=", 1)
            vals[key.strip()] = val.strip()
    return vals


# ----------------------------------------------------------------- prefill

def test_single_visible_key_returns_its_value():
    """Causal row 0 (q_offset 0) sees only key 0: O = V[0], LSE = s_00."""
    rng = np.random.default_rng(1)
    sq, hq = 4, 2
    q = np.zeros((sq, hq, D), np.float32)
    q[:, :, 3] = 2.0
    k = rng.integers(-4, 5, size=(sq, 1, D)).astype(np.float32)
    k[0, 0, 3] = 3.0
    v = rng.integers(-8, 9, size=(sq, 1, D)).astype(np.float32) / 4
    q[0, :, 100] = 0.0
    out, lse = oracle.prefill(bf16(q), bf16(k), bf16(v), scale=0.125, causal=True)
    np.testing.assert_array_equal(out[0, 0], v[0, 0])
    np.testing.assert_array_equal(out[0, 1], v[0, 0])
    assert lse[0, 0] == pytest.approx(2.0 * 3.0 * 0.125, abs=1e-15)


def test_uniform_logits_give_mean_and_log_count():
    """q = 0: every visible key has logit 0, so O is the mean of the visible V
    rows and LSE = ln(#visible)."""
    rng = np.random.default_rng(2)
    sq, sk, off = 5, 12, 7
    q = np.zeros((sq, 2, D), np.float32)
    k = rng.standard_normal((sk, 1, D)).astype(np.float32)
    v = bf16(rng.standard_normal((sk, 1, D))).float().numpy()
    out, lse = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=off, causal=True)
    for i in range(sq):
        n = off + i + 1
        np.testing.assert_allclose(out[i, 0], v[:n, 0].astype(np.float64).mean(0), atol=1e-14)
        assert lse[1, i] == pytest.approx(math.log(n), abs=1e-14)


def test_causal_positions_and_window_bands():
    """V[j] = j with q = 0: row i (position p = q_offset + i) averages the
    visible positions, p/2 causally and p - (W-1)/2 inside a window of W keys."""
    sk, off, sq = 200, 40, 160
    q = np.zeros((sq, 1, D), np.float32)
    k = np.ones((sk, 1, D), np.float32)
    v = np.repeat(np.arange(sk, dtype=np.float32)[:, None, None], D, axis=2)
    out, _ = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=off, causal=True)
    for i in (0, 1, 17, 159):
        p = off + i
        assert out[i, 0, 0] == pytest.approx(p / 2, abs=1e-12)
    W = 9
    out, lse = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=off, causal=True, window=W)
    for i in (0, 5, 159):
        p = off + i
        assert out[i, 0, 7] == pytest.approx(p - (W - 1) / 2, abs=1e-12)
        assert lse[0, i] == pytest.approx(math.log(W), abs=1e-13)
    # window reaching before key 0 keeps only [0, p]
    out, _ = oracle.prefill(bf16(q[:1]), bf16(k), bf16(v), q_offset=3, causal=True, window=W)
    assert out[0, 0, 0] == pytest.approx(1.5, abs=1e-13)


def test_q_offset_is_bottom_right_for_chunks():
    """A chunk at q_offset = seqlen_k - seqlen_q: its last row sees every key."""
    sk, sq = 64, 16
    q = np.zeros((sq, 1, D), np.float32)
    k = np.zeros((sk, 1, D), np.float32)
    v = np.repeat(np.arange(sk, dtype=np.float32)[:, None, None], D, axis=2)
    out, lse = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=sk - sq)
    assert out[-1, 0, 0] == pytest.approx((sk - 1) / 2, abs=1e-12)
    assert lse[0, -1] == pytest.approx(math.log(sk), abs=1e-13)
    assert lse[0, 0] == pytest.approx(math.log(sk - sq + 1), abs=1e-13)


def test_head_mapping_is_consecutive_groups():
    """Query head h reads KV head h // G: V of KV head c is the constant c+1."""
    hq, hk, sk = 12, 3, 9
    G = hq // hk
    q = np.zeros((2, hq, D), np.float32)
    k = np.zeros((sk, hk, D), np.float32)
    v = np.zeros((sk, hk, D), np.float32)
    for c in range(hk):
        v[:, c, :] = c + 1
    out, _ = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=sk - 2)
    for h in range(hq):
        np.testing.assert_allclose(out[:, h, :], h // G + 1, atol=1e-14)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(3)
    sq, sk, hq, hk = 6, 11, 8, 2
    q = bf16(rng.standard_normal((sq, hq, D)))
    k = bf16(rng.standard_normal((sk, hk, D)))
    v = bf16(rng.standard_normal((sk, hk, D)))
    G = hq // hk
    kr = k.repeat_interleave(G, dim=1)
    vr = v.repeat_interleave(G, dim=1)
    o1, l1 = oracle.prefill(q, k, v, q_offset=5)
    o2, l2 = oracle.prefill(q, kr, vr, q_offset=5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("a,b", [(2.0, 3.0), (-1.5, 4.0), (32.0, 25.0)])
def test_two_keys_closed_form(a, b):
    """Two keys with logits s0 = scale*a*b and s1 = 0 give weights
    sigmoid(s0) and 1 - sigmoid(s0); LSE = ln(1 + e^s0).  The (32, 25) case
    puts the logit at 800, beyond exp's range, so a missing max shift fails."""
    rng = np.random.default_rng(4)
    scale = 1.0 if a * b > 100 else 0.25
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = a
    k = np.zeros((2, 1, D), np.float32)
    k[0, 0, 0] = b
    k[1, 0, 1] = 7.0          # orthogonal to q: logit 0
    v = bf16(rng.standard_normal((2, 1, D))).float().numpy().astype(np.float64)
    out, lse = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=1, scale=scale)
    s0 = scale * a * b
    w0 = 1.0 / (1.0 + math.exp(-s0)) if s0 > -700 else 0.0
    np.testing.assert_allclose(out[0, 0], w0 * v[0, 0] + (1 - w0) * v[1, 0], rtol=1e-13,
                               atol=1e-14)
    want = s0 + math.log1p(math.exp(-s0)) if s0 > 0 else math.log1p(math.exp(s0))
    assert lse[0, 0] == pytest.approx(want, rel=1e-14)


def test_dominant_key_returns_its_row_not_column():
    """One key 60 logits above the rest: O equals that key's V row to ~e^-60.
    V rows and columns differ everywhere, so a transposed V fails."""
    rng = np.random.default_rng(5)
    sk = 24
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 5] = 6.0
    k = np.zeros((sk, 1, D), np.float32)
    k[13, 0, 5] = 10.0
    v = bf16(rng.standard_normal((sk, 1, D))).float().numpy().astype(np.float64)
    out, lse = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=sk - 1, scale=1.0)
    np.testing.assert_allclose(out[0, 0], v[13, 0], atol=1e-20 * sk + 1e-24, rtol=1e-15)
    assert lse[0, 0] == pytest.approx(60.0 + math.log1p((sk - 1) * math.exp(-60)), abs=1e-14)


def test_common_logit_shift_moves_lse_only():
    """Adding c to every logit (through a spare dimension) leaves O unchanged
    and adds c to LSE."""
    rng = np.random.default_rng(6)
    sq, sk = 3, 10
    q = rng.standard_normal((sq, 1, D)).astype(np.float32)
    k = rng.standard_normal((sk, 1, D)).astype(np.float32)
    q[:, :, D - 1] = 0.0
    k[:, :, D - 1] = 0.0
    v = rng.standard_normal((sk, 1, D)).astype(np.float32)
    q2, k2 = q.copy(), k.copy()
    q2[:, :, D - 1] = 4.0
    k2[:, :, D - 1] = 8.0
    scale = 0.0625
    o1, l1 = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=sk - sq, scale=scale)
    o2, l2 = oracle.prefill(bf16(q2), bf16(k2), bf16(v), q_offset=sk - sq, scale=scale)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, scale * 32.0, atol=1e-12)


def test_key_order_is_irrelevant_without_mask():
    rng = np.random.default_rng(7)
    sq, sk = 4, 30
    q = bf16(rng.standard_normal((sq, 2, D)))
    k = bf16(rng.standard_normal((sk, 1, D)))
    v = bf16(rng.standard_normal((sk, 1, D)))
    perm = torch.as_tensor(rng.permutation(sk))
    o1, l1 = oracle.prefill(q, k, v, causal=False)
    o2, l2 = oracle.prefill(q, k[perm], v[perm], causal=False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_empty_rows_are_zero_with_minus_inf_lse():
    """No visible key: O = 0, LSE = -inf (PR #199, review item F4)."""
    q = bf16(np.ones((2, 2, D)))
    k = bf16(np.ones((4, 1, D)))
    out, lse = oracle.prefill(q, k, k, q_offset=10, causal=True, window=2)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    out, lse = oracle.prefill(q, k[:0], k[:0], q_offset=0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_sampled_rows_match_full_run():
    """Asking for a subset of rows returns exactly those rows."""
    cfg = workloads.PrefillConfig("t", 40, 40, 0, 4, 2, seed=11)
    q, k, v = workloads.prefill_inputs(cfg)
    o_all, l_all = oracle.prefill(q, k, v)
    rows = [0, 7, 39]
    o_s, l_s = oracle.prefill(q, k, v, rows=rows)
    np.testing.assert_array_equal(o_s, o_all[rows])
    np.testing.assert_array_equal(l_s, l_all[:, rows])


def test_thread_count_does_not_change_bits():
    cfg = workloads.PrefillConfig("t", 33, 33, 0, 4, 1, seed=12)
    q, k, v = workloads.prefill_inputs(cfg)
    o1, l1 = oracle.prefill(q, k, v, threads=1)
    o2, l2 = oracle.prefill(q, k, v, threads=5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ------------------------------------------------------- pages' worked cases

def test_q_zero_v_one_is_one_at_every_length():
    """PR #199 review: with q = 0 and V = 1 the exact output is 1.000 at any
    key count (the page saw 0.500 at 32K and 0.125 at 128K from a
    low-precision accumulator)."""
    g = read_golden("q0_v1_long_split.txt")
    for n in [int(x) for x in g["key_counts"].split(",")]:
        q = torch.zeros((1, 1, D), dtype=torch.bfloat16)
        k = workloads.randn_bf16((n, 1, D), 99)
        v = torch.ones((n, 1, D), dtype=torch.bfloat16)
        out, lse = oracle.prefill(q, k, v, q_offset=n - 1)
        assert np.max(np.abs(out - float(g["expected_output"]))) < 1e-9
        assert lse[0, 0] == pytest.approx(math.log(n), abs=1e-10)


def test_softmax_tail_one_late_key_ahead():
    """PR #199 review item F1: n keys, every logit 0 except one late key
    ahead by delta.  Its weight is e^delta / (e^delta + n - 1) exactly."""
    g = read_golden("late_key_tail.txt")
    n = int(g["keys"])
    for delta_s in g["deltas"].split(","):
        delta = int(delta_s)
        a, b = {12: (3.0, 4.0), 13: (1.0, 13.0)}[delta]
        q = np.zeros((1, 1, D), np.float32)
        q[0, 0, 0] = a
        k = torch.zeros((n, 1, D), dtype=torch.bfloat16)
        k[n - 1, 0, 0] = b
        v = torch.zeros((n, 1, D), dtype=torch.bfloat16)
        v[n - 1, 0, 0] = 1.0
        v[:, 0, 1] = 1.0
        out, lse = oracle.prefill(bf16(q), k, v, q_offset=n - 1, scale=1.0)
        w = math.exp(delta) / (math.exp(delta) + n - 1)
        assert out[0, 0, 0] == pytest.approx(w, rel=1e-12)
        assert out[0, 0, 1] == pytest.approx(1.0, abs=1e-12)
        assert lse[0, 0] == pytest.approx(math.log(math.exp(delta) + n - 1), abs=1e-12)


# ------------------------------------------------------------------ decode

def test_decode_band_and_positions():
    """V at logical position j is the constant j / 8 and q = 0: the output is
    the mean of the live band, (len - 1) / 2 / 8, or the window mean."""
    page = 16
    lens = [1, 15, 16, 17, 100]
    pc = workloads.paged_decode_inputs(len(lens), lens, 4, 2, page, seed=21)
    q = torch.zeros_like(pc.q)
    for b, n in enumerate(lens):
        for j in range(n):
            pg = int(pc.page_table[b, j // page])
            pc.v_pages[pg, j % page] = j / 8
    out, lse = oracle.decode_paged(q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens)
    for b, n in enumerate(lens):
        np.testing.assert_allclose(out[b], (n - 1) / 2 / 8, atol=1e-12)
        np.testing.assert_allclose(lse[b], math.log(n), atol=1e-13)
    W = 5
    out, lse = oracle.decode_paged(q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                   window=W)
    for b, n in enumerate(lens):
        lo = max(0, n - W)
        np.testing.assert_allclose(out[b], (lo + n - 1) / 2 / 8, atol=1e-12)
        np.testing.assert_allclose(lse[b], math.log(n - lo), atol=1e-13)


def test_decode_ignores_poisoned_slots_and_empty_sequences():
    pc = workloads.paged_decode_inputs(3, [0, 70, 64], 8, 4, 64, seed=22)
    out, lse = oracle.decode_paged(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens)
    assert np.all(np.isfinite(out))
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1:]))


def test_decode_page_permutation_invariance_and_prefill_agreement():
    """The same logical cache laid out through two different page tables
    gives the same result, equal to the last row of a contiguous prefill."""
    page, n, hq, hk = 32, 150, 8, 4
    pc = workloads.paged_decode_inputs(1, [n], hq, hk, page, seed=23)
    o1, l1 = oracle.decode_paged(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens)
    npg = (n + page - 1) // page
    # gather the logical K/V contiguously, then re-page in reversed order
    idx = pc.page_table[0, :npg].long()
    k_lin = pc.k_pages[idx].reshape(npg * page, hk, D)[:n]
    v_lin = pc.v_pages[idx].reshape(npg * page, hk, D)[:n]
    o_pre, l_pre = oracle.prefill(pc.q[0][None], k_lin, v_lin, q_offset=n - 1)
    np.testing.assert_array_equal(o1[0], o_pre[0])
    np.testing.assert_array_equal(l1[0], l_pre[:, 0])
    rev = torch.arange(npg - 1, -1, -1)
    k2 = pc.k_pages[idx][rev]
    v2 = pc.v_pages[idx][rev]
    pt2 = (npg - 1 - torch.arange(npg, dtype=torch.int32))[None]
    o2, l2 = oracle.decode_paged(pc.q, k2, v2, pt2, pc.kv_lens)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_decode_q0_v1_long():
    n = 28672
    pc = workloads.paged_decode_inputs(1, [n], 8, 4, 64, seed=24, spare_pages=1)
    q = torch.zeros_like(pc.q)
    v = torch.ones_like(pc.v_pages)
    out, _ = oracle.decode_paged(q, pc.k_pages, v, pc.page_table, pc.kv_lens)
    assert np.max(np.abs(out - 1.0)) < 1e-9


def test_decode_rejects_out_of_range_tables():
    pc = workloads.paged_decode_inputs(1, [10], 2, 1, 16, seed=25)
    bad = pc.page_table.clone()
    bad[0, 0] = 10_000
    with pytest.raises(ValueError):
        oracle.decode_paged(pc.q, pc.k_pages, pc.v_pages, bad, pc.kv_lens)


# ----------------------------------------------- decode with several query tokens

def test_decode_q_positions_and_window_closed_form():
    """q = 0, V at logical position j is the constant j / 8: query t of a
    q_len-token decode sits at p = len - q_len + t and averages the positions
    [lo, p] it sees (lo = 0, or p - W + 1 under a window W); a query whose
    position is negative (len < q_len) sees nothing."""
    page, q_len = 16, 4
    lens = [1, 3, 4, 15, 17, 100]
    pc = workloads.paged_decode_inputs(len(lens), lens, 4, 2, page, seed=31)
    q = torch.zeros((len(lens), q_len, 4, D), dtype=torch.bfloat16)
    for b, n in enumerate(lens):
        for j in range(n):
            pg = int(pc.page_table[b, j // page])
            pc.v_pages[pg, j % page] = j / 8
    for W in (0, 3):
        out, lse = oracle.decode_paged_q(q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                         window=W)
        for b, n in enumerate(lens):
            for t in range(q_len):
                p = n - q_len + t
                if p < 0:
                    assert np.all(out[b, t] == 0) and np.all(np.isneginf(lse[b, t]))
                    continue
                lo = max(0, p - W + 1) if W > 0 else 0
                np.testing.assert_allclose(out[b, t], (lo + p) / 2 / 8, atol=1e-12)
                np.testing.assert_allclose(lse[b, t], math.log(p - lo + 1), atol=1e-13)


def test_decode_q_rows_are_the_last_prefill_rows():
    """A q_len-token decode over a paged cache equals the last q_len rows of a
    causal prefill over the same keys laid out contiguously (q_offset = len - q_len)."""
    page, n, hq, hk, q_len = 32, 150, 8, 4, 5
    pc = workloads.paged_decode_inputs(1, [n], hq, hk, page, seed=32)
    q = workloads.draft_queries(1, q_len, hq, seed=32)
    out, lse = oracle.decode_paged_q(q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens)
    npg = (n + page - 1) // page
    idx = pc.page_table[0, :npg].long()
    k_lin = pc.k_pages[idx].reshape(npg * page, hk, D)[:n]
    v_lin = pc.v_pages[idx].reshape(npg * page, hk, D)[:n]
    o_pre, l_pre = oracle.prefill(q[0], k_lin, v_lin, q_offset=n - q_len)
    np.testing.assert_array_equal(out[0], o_pre)
    np.testing.assert_array_equal(lse[0], l_pre.T)
    # the same with a window: row t keeps its own band
    out_w, lse_w = oracle.decode_paged_q(q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                         window=40)
    o_prw, l_prw = oracle.prefill(q[0], k_lin, v_lin, q_offset=n - q_len, window=40)
    np.testing.assert_array_equal(out_w[0], o_prw)
    np.testing.assert_array_equal(lse_w[0], l_prw.T)


def test_decode_q_len_one_is_single_token_decode():
    pc = workloads.paged_decode_inputs(3, [5, 64, 90], 8, 4, 32, seed=33)
    o1, l1 = oracle.decode_paged(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens)
    o2, l2 = oracle.decode_paged_q(pc.q[:, None], pc.k_pages, pc.v_pages, pc.page_table,
                                   pc.kv_lens)
    np.testing.assert_array_equal(o1, o2[:, 0])
    np.testing.assert_array_equal(l1, l2[:, 0])


# ------------------------------------------------ varlen prefill over a paged cache

def _paged_v_positions(pc, lens, page):
    """V channel 0 at logical position j of sequence b is j / 8, channel 1 is b
    (both exact in bf16); the other channels keep their random values."""
    for b, n in enumerate(lens):
        for j in range(n):
            pg = int(pc.page_table[b, j // page])
            pc.v_pages[pg, j % page, :, 0] = j / 8
            pc.v_pages[pg, j % page, :, 1] = b


def test_prefill_paged_positions_closed_form():
    """q = 0: every visible key has logit 0, so channel 0 of O is the mean of
    the visible positions / 8 and channel 1 names the sequence.  Row i of a
    chunk of S rows over a cache of n positions sits at p = n - S + i (the
    chunk is the tail of its sequence) and sees [lo, p]; a negative p sees
    nothing.  Slots outside the live positions are NaN, so a read past a
    sequence's length or through an unused table entry shows up."""
    page = 16
    lens_k = [37, 5, 64, 0, 20]
    lens_q = [6, 9, 1, 3, 0]
    pc = workloads.paged_decode_inputs(len(lens_k), lens_k, 4, 2, page, seed=41)
    _paged_v_positions(pc, lens_k, page)
    _, cu = workloads.varlen_queries(lens_q, 4, seed=41)
    q = torch.zeros((int(cu[-1]), 4, D), dtype=torch.bfloat16)
    used = torch.tensor(lens_k, dtype=torch.int32)
    for W in (0, 3):
        out, lse = oracle.prefill_paged(q, pc.k_pages, pc.v_pages, pc.page_table, cu, used,
                                        window=W)
        assert np.all(np.isfinite(out))
        for b, (n, s) in enumerate(zip(lens_k, lens_q)):
            for i in range(s):
                r, p = int(cu[b]) + i, n - s + i
                if p < 0:
                    assert np.all(out[r] == 0) and np.all(np.isneginf(lse[:, r]))
                    continue
                lo = max(0, p - W + 1) if W > 0 else 0
                np.testing.assert_allclose(out[r, :, 0], (lo + p) / 2 / 8, atol=1e-12)
                np.testing.assert_allclose(out[r, :, 1], b, atol=1e-12)
                np.testing.assert_allclose(lse[:, r], math.log(p - lo + 1), atol=1e-13)
    # without the causal mask every row sees the whole cache of its sequence
    out, lse = oracle.prefill_paged(q, pc.k_pages, pc.v_pages, pc.page_table, cu, used,
                                    causal=False)
    for b, (n, s) in enumerate(zip(lens_k, lens_q)):
        for i in range(s):
            r = int(cu[b]) + i
            if n == 0:
                assert np.all(out[r] == 0) and np.all(np.isneginf(lse[:, r]))
                continue
            np.testing.assert_allclose(out[r, :, 0], (n - 1) / 2 / 8, atol=1e-12)
            np.testing.assert_allclose(lse[:, r], math.log(n), atol=1e-13)


def test_prefill_paged_equals_multi_token_decode():
    """Chunks of S rows each equal an S-token decode over the same cache (a
    separate code path that walks the page table itself), bit for bit."""
    page, s, hq, hk = 32, 4, 8, 4
    lens_k = [40, 100, 7]
    pc = workloads.paged_decode_inputs(len(lens_k), lens_k, hq, hk, page, seed=42)
    q, cu = workloads.varlen_queries([s] * len(lens_k), hq, seed=42)
    used = torch.tensor(lens_k, dtype=torch.int32)
    for W in (0, 20):
        o_p, l_p = oracle.prefill_paged(q, pc.k_pages, pc.v_pages, pc.page_table, cu, used,
                                        window=W)
        o_d, l_d = oracle.decode_paged_q(q.reshape(len(lens_k), s, hq, D), pc.k_pages,
                                         pc.v_pages, pc.page_table, used, window=W)
        np.testing.assert_array_equal(o_p, o_d.reshape(-1, hq, D))
        np.testing.assert_array_equal(l_p, l_d.reshape(-1, hq).T)


def test_prefill_paged_page_permutation_invariance():
    """Moving every physical page elsewhere in the pool and rewriting the
    table to match leaves the result unchanged, bit for bit."""
    page, hq, hk = 16, 4, 1
    lens_k, lens_q = [50, 33], [20, 33]
    pc = workloads.paged_decode_inputs(2, lens_k, hq, hk, page, seed=43)
    q, cu = workloads.varlen_queries(lens_q, hq, seed=43)
    used = torch.tensor(lens_k, dtype=torch.int32)
    o1, l1 = oracle.prefill_paged(q, pc.k_pages, pc.v_pages, pc.page_table, cu, used)
    npg = pc.k_pages.shape[0]
    perm = torch.randperm(npg, generator=torch.Generator().manual_seed(43))
    k2 = torch.empty_like(pc.k_pages)
    v2 = torch.empty_like(pc.v_pages)
    k2[perm] = pc.k_pages
    v2[perm] = pc.v_pages
    pt2 = pc.page_table.clone()
    live = pt2 < npg
    pt2[live] = perm[pt2[live].long()].to(torch.int32)
    o2, l2 = oracle.prefill_paged(q, k2, v2, pt2, cu, used)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # and a contiguous prefill over the gathered keys agrees for a full-length chunk
    idx = pc.page_table[1, :3].long()
    k_lin = pc.k_pages[idx].reshape(3 * page, hk, D)[:33]
    v_lin = pc.v_pages[idx].reshape(3 * page, hk, D)[:33]
    o3, l3 = oracle.prefill(q[20:53], k_lin, v_lin, q_offset=0)
    np.testing.assert_array_equal(o1[20:53], o3)
    np.testing.assert_array_equal(l1[:, 20:53], l3)


def test_prefill_paged_rejects_bad_tables_and_offsets():
    pc = workloads.paged_decode_inputs(2, [10, 30], 2, 1, 16, seed=44)
    q, cu = workloads.varlen_queries([4, 5], 2, seed=44)
    used = torch.tensor([10, 30], dtype=torch.int32)
    bad = pc.page_table.clone()
    bad[1, 1] = 10_000
    with pytest.raises(ValueError):
        oracle.prefill_paged(q, pc.k_pages, pc.v_pages, bad, cu, used)
    with pytest.raises(ValueError):
        oracle.prefill_paged(q, pc.k_pages, pc.v_pages, pc.page_table,
                             torch.tensor([0, 5, 4], dtype=torch.int32), used)
    with pytest.raises(ValueError):
        oracle.prefill_paged(q, pc.k_pages, pc.v_pages, pc.page_table, cu,
                             torch.tensor([10, 33], dtype=torch.int32))


# --------------------------------------- head dim 256 (the sliding-window local layers)

D256 = 256


def test_d256_window_band_closed_form():
    """Head dim 256, window 1024 ("A custom attention kernel for Gemma 4 on the
    RTX PRO 6000", "The deployment": the local layers attend to the last 1,024
    tokens with heads of 256 dimensions).  q = 0 and V channel c at position j
    equal to j / 64 (exact in bf16 for j < 2048): row i at p = q_offset + i
    averages the (bf16-rounded) values of [max(0, p - W + 1), p] and
    LSE = ln(count)."""
    sk, off, sq, W = 1500, 300, 1200, 1024
    q = np.zeros((sq, 2, D256), np.float32)
    k = np.ones((sk, 1, D256), np.float32)
    vb = bf16(np.repeat((np.arange(sk, dtype=np.float32) / 64)[:, None, None], D256, axis=2))
    vr = vb.float().numpy().astype(np.float64)[:, 0, D256 - 1]
    rows = [0, 1, 700, 723, 724, 725, 1199]
    out, lse = oracle.prefill(bf16(q), bf16(k), vb, q_offset=off, window=W, rows=rows)
    for r, i in enumerate(rows):
        p = off + i
        lo = max(0, p - W + 1)
        np.testing.assert_allclose(out[r, :, D256 - 1], vr[lo:p + 1].mean(), atol=1e-12)
        np.testing.assert_allclose(lse[:, r], math.log(p - lo + 1), atol=1e-12)


def test_d256_two_keys_and_scale():
    """Two visible keys with q.k0 = a * b over one channel and q.k1 = 0: the
    weights are sigmoid(+-s), s = a * b / 16, the default scale 1/sqrt(256)."""
    a, b = 3.0, 5.0
    q = np.zeros((1, 1, D256), np.float32)
    q[0, 0, 255] = a
    k = np.zeros((2, 1, D256), np.float32)
    k[0, 0, 255] = b
    v = np.zeros((2, 1, D256), np.float32)
    v[0, 0, 0] = 1.0
    v[1, 0, 1] = 1.0
    out, lse = oracle.prefill(bf16(q), bf16(k), bf16(v), q_offset=1)
    s = a * b / 16
    w0 = 1 / (1 + math.exp(-s))
    assert out[0, 0, 0] == pytest.approx(w0, rel=1e-13)
    assert out[0, 0, 1] == pytest.approx(1 - w0, rel=1e-12)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(s) + 1), rel=1e-13)


def test_d256_head_mapping_and_last_channel():
    """Query head h reads KV head h // G and every one of the 256 channels:
    V of KV head c is c + 1 + channel / 256, rounded to bf16 once and used
    rounded on both sides."""
    hq, hk, sk = 8, 2, 5
    q = np.zeros((3, hq, D256), np.float32)
    k = np.zeros((sk, hk, D256), np.float32)
    ch = np.arange(D256, dtype=np.float32) / 256
    v = np.zeros((sk, hk, D256), np.float32)
    for c in range(hk):
        v[:, c, :] = c + 1 + ch
    vb = bf16(v)
    vr = vb.float().numpy().astype(np.float64)
    out, _ = oracle.prefill(bf16(q), bf16(k), vb, q_offset=sk - 3)
    for h in range(hq):
        np.testing.assert_allclose(out[:, h, :], np.broadcast_to(vr[0, h // (hq // hk)], (3, D256)),
                                   atol=1e-14)


# ------------------------------------------------------------- FP8 E4M3 cache

def test_e4m3_decoding_fixed_points_and_torch_agreement():
    """The oracle's E4M3 decoding against the format's fixed points (the
    largest finite value is 448: vllm-project/flash-attention PR #199, review
    F1, "256 < 448") and against torch's float8_e4m3fn for all 256 codes."""
    t = oracle.e4m3_table()
    fixed = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0x08: 2.0 ** -6,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0xFE: -448.0, 0xB8: -1.0}
    for code, val in fixed.items():
        assert t[code] == val, hex(code)
    assert np.signbit(t[0x80]) and t[0x80] == 0.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.all(np.diff(t[:0x7F]) > 0)                        # monotone over the positive codes
    np.testing.assert_array_equal(t[0x80:0xFF], -t[0x00:0x7F])   # sign bit
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(t), np.isnan(ref))
    np.testing.assert_array_equal(t[~np.isnan(t)], ref[~np.isnan(ref)])


def _fp8_to_bf16_cache(pages_u8, scale):
    """The dequantised cache in bf16: scale * e4m3 is exact in bf16 when the
    scale is a power of two."""
    return (pages_u8.view(torch.float8_e4m3fn).float() * scale).to(torch.bfloat16)


@pytest.mark.parametrize("scale_pow2", [1.0, 1 / 32])
def test_fp8_decode_equals_bf16_decode_on_the_same_values(scale_pow2):
    """With power-of-two scales every dequantised element is a bf16 value, so
    the FP8 decode must equal the (pinned) bf16 decode bit for bit, including
    the poisoned slots it must not read."""
    lens = [1, 63, 64, 130, 300]
    pc, _, _ = workloads.paged_fp8_inputs(len(lens), lens, 8, 4, 64, seed=61)
    kb = _fp8_to_bf16_cache(pc.k_pages, scale_pow2)
    vb = _fp8_to_bf16_cache(pc.v_pages, scale_pow2)
    o8, l8 = oracle.decode_paged_fp8(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                     k_scale=scale_pow2, v_scale=scale_pow2)
    o16, l16 = oracle.decode_paged(pc.q, kb, vb, pc.page_table, pc.kv_lens)
    np.testing.assert_array_equal(o8, o16)
    np.testing.assert_array_equal(l8, l16)
    # several query tokens and a window take the same path
    q4 = workloads.draft_queries(len(lens), 3, 8, seed=61)
    o8, l8 = oracle.decode_paged_fp8(q4, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                     k_scale=scale_pow2, v_scale=scale_pow2, window=50)
    o16, l16 = oracle.decode_paged_q(q4, kb, vb, pc.page_table, pc.kv_lens, window=50)
    np.testing.assert_array_equal(o8, o16)
    np.testing.assert_array_equal(l8, l16)


def test_fp8_scale_laws():
    """k_scale multiplies every logit (the same as scaling the softmax scale);
    v_scale multiplies O and leaves LSE alone."""
    pc, _, _ = workloads.paged_fp8_inputs(2, [100, 37], 4, 2, 64, seed=62)
    base_o, base_l = oracle.decode_paged_fp8(pc.q, pc.k_pages, pc.v_pages, pc.page_table,
                                             pc.kv_lens, k_scale=0.03, v_scale=0.05)
    o, l = oracle.decode_paged_fp8(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                   k_scale=1.0, v_scale=0.05, scale=D ** -0.5 * 0.03)
    np.testing.assert_allclose(o, base_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, base_l, rtol=1e-12, atol=1e-12)
    o, l = oracle.decode_paged_fp8(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                                   k_scale=0.03, v_scale=0.15)
    np.testing.assert_allclose(o, 3 * base_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(l, base_l)


def test_fp8_q0_v1_and_softmax_tail_closed_forms():
    """PR #199 review: q = 0 and V = 1 give exactly 1 (here v_scale) at every
    length; review F1: one late key ahead by 12 among n keys carries the
    weight e^12 / (e^12 + n - 1)."""
    n = 32768
    pc, _, _ = workloads.paged_fp8_inputs(1, [n], 2, 1, 64, seed=63, spare_pages=1)
    q = torch.zeros_like(pc.q)
    ones = torch.full_like(pc.v_pages, 0x38)        # e4m3 1.0
    o, _ = oracle.decode_paged_fp8(q, pc.k_pages, ones, pc.page_table, pc.kv_lens, v_scale=0.5)
    np.testing.assert_allclose(o, 0.5, rtol=1e-12)
    # the tail case: K = 0 except k[n-1][0] = 4 (code 0x48), q[0] = 3, scale 1
    k = torch.zeros_like(pc.k_pages)
    v = torch.zeros_like(pc.v_pages)
    last = int(pc.page_table[0, (n - 1) // 64])
    k[last, (n - 1) % 64, 0, 0] = 0x48
    v[:, :, 0, 1] = 0x38
    v[last, (n - 1) % 64, 0, 0] = 0x38
    q = torch.zeros_like(pc.q)
    q[0, :, 0] = 3.0
    o, l = oracle.decode_paged_fp8(q, k, v, pc.page_table, pc.kv_lens, scale=1.0)
    w = math.exp(12) / (math.exp(12) + n - 1)
    np.testing.assert_allclose(o[0, :, 0], w, rtol=1e-12)
    np.testing.assert_allclose(o[0, :, 1], 1.0, rtol=1e-12)
    np.testing.assert_allclose(l[0], math.log(math.exp(12) + n - 1), rtol=1e-13)
