"""Seeded synthetic inputs for hd512 prefill and paged decode.

This module holds shapes and random draws only -- none of the attention
arithmetic -- so that the CUDA path and the fp64 oracle can be fed the very
same tensors.  Everything is drawn on the CPU with a seeded torch generator in
fp32 and rounded to bf16 (round-to-nearest-even), Q, K and V independently.

Shapes follow the workloads the pages measure:
  * pegainfer issue #1051, "Description": one 8192-row chunk against all the
    context before it, 32 query heads over 4 KV heads, bf16, causal;
  * "A custom attention kernel for Gemma 4 on the RTX PRO 6000": 20k-token
    prefill of the head-dim-512 global layers, 8 query heads per KV head;
  * "Flash-Decoding for MQA in CUDA": long-context MQA (one KV head);
  * vllm-project/flash-attention PR #199, "Performance": decode with q_len 1,
    8 query heads over 4 KV heads, head dim 512, page size 64, batch
    {1, 16, 64} at KV length {4K, 16K, 28K}.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

HEAD_DIM = 512
SEED_BASE = 0x5EED


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    seqlen_q: int
    seqlen_k: int
    q_offset: int
    n_q_heads: int
    n_kv_heads: int
    causal: bool = True
    window: int = 0
    stress: bool = False          # every 64th K row multiplied by 8
    seed: int = SEED_BASE
    head_dim: int = HEAD_DIM

    @property
    def scale(self) -> float:
        return self.head_dim ** -0.5


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    kv_len: int
    n_q_heads: int = 8
    n_kv_heads: int = 4
    page_size: int = 64
    window: int = 0
    spare_pages: int = 8          # poisoned pages no sequence points at
    seed: int = SEED_BASE + 5

    @property
    def scale(self) -> float:
        return HEAD_DIM ** -0.5


PREFILL_CONFIGS = {
    "tiny": PrefillConfig("tiny", 256, 256, 0, 8, 1, seed=SEED_BASE + 1),
    "chunked": PrefillConfig("chunked", 8192, 16384, 8192, 32, 4, seed=SEED_BASE + 2),
    "full": PrefillConfig("full", 20480, 20480, 0, 32, 4, seed=SEED_BASE + 3),
    "full_stress": PrefillConfig("full_stress", 20480, 20480, 0, 32, 4, stress=True,
                                 seed=SEED_BASE + 3),
    "mqa": PrefillConfig("mqa", 49152, 49152, 0, 16, 1, seed=SEED_BASE + 4),
    # the sliding-window local layers: heads of 256 dimensions over the last
    # 1,024 tokens, a 20k-token prompt (RTX PRO 6000 page, "The deployment");
    # the head counts are the global layers' (the pages give none for these)
    "local256": PrefillConfig("local256", 20480, 20480, 0, 32, 4, window=1024,
                              seed=SEED_BASE + 8, head_dim=256),
}

DECODE_CONFIGS = {
    "b%d_kv%d" % (b, n): DecodeConfig("b%d_kv%d" % (b, n), b, n)
    for b in (1, 16, 64) for n in (4096, 16384, 28672)
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, seed: int) -> torch.Tensor:
    """N(0,1) draws in fp32 from a seeded CPU generator, rounded to bf16."""
    return torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(cfg: PrefillConfig):
    """(q, k, v) on the CPU: q [sq, Hq, D], k/v [sk, Hkv, D], bf16 (D = cfg.head_dim)."""
    q = randn_bf16((cfg.seqlen_q, cfg.n_q_heads, cfg.head_dim), cfg.seed * 3 + 0)
    k = randn_bf16((cfg.seqlen_k, cfg.n_kv_heads, cfg.head_dim), cfg.seed * 3 + 1)
    v = randn_bf16((cfg.seqlen_k, cfg.n_kv_heads, cfg.head_dim), cfg.seed * 3 + 2)
    if cfg.stress:
        # x8 is exact in bf16 (an exponent change), so the stressed rows stay
        # exact copies of 8 * (the unstressed bf16 value).
        k[::64] *= 8
    return q, k, v


@dataclass
class PagedCache:
    q: torch.Tensor            # [batch, Hq, 512] bf16
    k_pages: torch.Tensor      # [num_pages, page_size, Hkv, 512] bf16
    v_pages: torch.Tensor
    page_table: torch.Tensor   # [batch, max_pages_per_seq] int32
    kv_lens: torch.Tensor      # [batch] int32
    max_kv_len: int
    extra: dict = field(default_factory=dict)


def paged_decode_inputs(batch: int, kv_lens, n_q_heads: int = 8, n_kv_heads: int = 4,
                        page_size: int = 64, seed: int = SEED_BASE + 5, spare_pages: int = 8,
                        poison: bool = True, max_pages_per_seq: int | None = None) -> PagedCache:
    """A paged KV cache with a seeded random page permutation.

    Each sequence b gets ceil(kv_lens[b] / page_size) pages, drawn from a
    seeded random permutation of a pool that also holds ``spare_pages``
    pages nobody points at.  With ``poison`` set, every slot outside a live
    band (spare pages, the tail of each last page) is NaN, so any read
    outside the band shows up in the output.  Unused page-table entries hold
    an out-of-range page index.
    """
    kv_lens = [int(x) for x in (kv_lens if hasattr(kv_lens, "__len__") else [kv_lens] * batch)]
    assert len(kv_lens) == batch
    pages_per_seq = [(n + page_size - 1) // page_size for n in kv_lens]
    mpps = max(1, max(pages_per_seq) if pages_per_seq else 1)
    if max_pages_per_seq is not None:
        assert max_pages_per_seq >= mpps
        mpps = max_pages_per_seq
    num_pages = sum(pages_per_seq) + spare_pages
    g = _gen(seed * 7 + 1)
    perm = torch.randperm(num_pages, generator=g)
    q = randn_bf16((batch, n_q_heads, HEAD_DIM), seed * 7 + 2)
    k_pages = randn_bf16((num_pages, page_size, n_kv_heads, HEAD_DIM), seed * 7 + 3)
    v_pages = randn_bf16((num_pages, page_size, n_kv_heads, HEAD_DIM), seed * 7 + 4)
    page_table = torch.full((batch, mpps), num_pages + 12345, dtype=torch.int32)
    live = torch.zeros((num_pages, page_size), dtype=torch.bool)
    cursor = 0
    for b in range(batch):
        for p in range(pages_per_seq[b]):
            pg = int(perm[cursor])
            cursor += 1
            page_table[b, p] = pg
            n_in_page = min(page_size, kv_lens[b] - p * page_size)
            live[pg, :n_in_page] = True
    if poison:
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
        k_pages[~live] = nan
        v_pages[~live] = nan
    return PagedCache(q, k_pages, v_pages, page_table,
                      torch.tensor(kv_lens, dtype=torch.int32), max(kv_lens) if kv_lens else 0,
                      extra={"num_pages": num_pages, "page_size": page_size,
                             "n_q_heads": n_q_heads, "n_kv_heads": n_kv_heads})


E4M3_NAN = 0x7F


def to_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """x / scale rounded to the nearest FP8 E4M3 value (torch's float8_e4m3fn
    cast), returned as the uint8 codes; |x / scale| must stay below 448."""
    return (x.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8)


def paged_fp8_inputs(batch: int, kv_lens, n_q_heads: int = 8, n_kv_heads: int = 4,
                     page_size: int = 64, seed: int = SEED_BASE + 9, spare_pages: int = 8,
                     poison: bool = True, k_scale: float = 1 / 32, v_scale: float = 1 / 32):
    """The paged layout of paged_decode_inputs with an FP8 E4M3 cache: K and V
    are N(0,1) draws stored as e4m3(x / scale) with per-tensor scales (the
    dequantised element is scale * e4m3).  With ``poison`` every slot outside
    a live band holds the E4M3 NaN code.  Returns (PagedCache with uint8
    k_pages / v_pages, k_scale, v_scale)."""
    pc = paged_decode_inputs(batch, kv_lens, n_q_heads, n_kv_heads, page_size, seed,
                             spare_pages, poison=False)
    g = _gen(seed * 7 + 8)
    shape = tuple(pc.k_pages.shape)
    k8 = to_e4m3(torch.randn(shape, generator=g, dtype=torch.float32), k_scale)
    v8 = to_e4m3(torch.randn(shape, generator=g, dtype=torch.float32), v_scale)
    if poison:
        live = torch.zeros(shape[:2], dtype=torch.bool)
        for b in range(batch):
            n = int(pc.kv_lens[b])
            for lp in range((n + page_size - 1) // page_size):
                live[int(pc.page_table[b, lp]), :min(page_size, n - lp * page_size)] = True
        k8[~live] = E4M3_NAN
        v8[~live] = E4M3_NAN
    pc.k_pages, pc.v_pages = k8, v8
    return pc, k_scale, v_scale


def draft_queries(batch: int, q_len: int, n_q_heads: int, seed: int) -> torch.Tensor:
    """q_len query tokens per sequence (the last q_len positions of each
    cache, e.g. draft tokens being verified): [batch, q_len, n_q_heads, D] bf16."""
    return randn_bf16((batch, q_len, n_q_heads, HEAD_DIM), seed * 7 + 5)


def varlen_queries(seqlens_q, n_q_heads: int, seed: int):
    """Packed query rows of a batch of prefill chunks: (q [total_q, n_q_heads,
    D] bf16, cu_seqlens_q [batch + 1] int32), chunk b at rows
    cu_seqlens_q[b] .. cu_seqlens_q[b + 1] - 1."""
    lens = [int(x) for x in seqlens_q]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    q = randn_bf16((cu[-1], n_q_heads, HEAD_DIM), seed * 7 + 6)
    return q, torch.tensor(cu, dtype=torch.int32)


def decode_inputs(cfg: DecodeConfig, poison: bool = True) -> PagedCache:
    return paged_decode_inputs(cfg.batch, [cfg.kv_len] * cfg.batch, cfg.n_q_heads,
                               cfg.n_kv_heads, cfg.page_size, cfg.seed, cfg.spare_pages, poison)


def sample_rows(cfg: PrefillConfig, tokens_per_tile: int = 16, every: int = 97) -> list[int]:
    """Stratified query-row sample for configs too large to check in full:
    the first and last 64 rows, rows at q-tile boundaries near both ends, the
    rows just after stressed keys (stress variant), and every 97th row."""
    n = cfg.seqlen_q
    rows = set(range(min(64, n))) | set(range(max(0, n - 64), n))
    for t in range(0, n, tokens_per_tile * 64):
        rows.update(x for x in (t - 1, t, t + tokens_per_tile - 1, t + tokens_per_tile)
                    if 0 <= x < n)
    if cfg.stress:
        for j in range(0, cfg.seqlen_k, 64 * 41):
            i = j - cfg.q_offset
            rows.update(x for x in (i, i + 1) if 0 <= x < n)
    rows.update(range(0, n, every))
    return sorted(rows)
