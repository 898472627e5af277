"""Parity at the benchmark's own sizes and launch configuration: the decode
legs bench.py times (batch 64, 8 query over 4 KV heads, page 64, shuffled
pages, num_splits auto), drawn on the device as the bench draws them, with
sampled sequences checked against the fp64 oracle (the oracle reads only the
pages those sequences own)."""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_lse, compare_o

pytestmark = pytest.mark.gpu
D, PAGE, HQ, HK = 512, 64, 8, 4
SAMPLE = [0, 21, 42, 63]


@pytest.fixture(scope="module")
def fa(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    import head_dim_flashattention_gb300 as fa
    fa.load_library()
    return fa


def device_cache(batch, kv_len, seed, fp8_scale=None):
    """Pools of batch * ceil(kv_len / 64) pages, N(0,1) (bf16, or e4m3 of
    N(0,1) / scale), a seeded permutation as page table: on the device."""
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    npg = (kv_len + PAGE - 1) // PAGE
    shape = (batch * npg, PAGE, HK, D)
    if fp8_scale is None:
        kp = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
        vp = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    else:
        kp = (torch.randn(shape, generator=g, device=dev) / fp8_scale).to(torch.float8_e4m3fn)
        vp = (torch.randn(shape, generator=g, device=dev) / fp8_scale).to(torch.float8_e4m3fn)
    gc = torch.Generator()
    gc.manual_seed(seed + 1)
    pt = torch.randperm(batch * npg, generator=gc).to(torch.int32).view(batch, npg)
    kl = torch.full((batch,), kv_len, dtype=torch.int32)
    return kp, vp, pt, kl


def sub_cache(kp, vp, pt, kl, rows):
    """The pages of the sampled sequences, renumbered 0.., on the host."""
    sel = pt[rows]
    idx = sel.reshape(-1).to(torch.int64)
    kp_s = kp.index_select(0, idx.cuda()).cpu()
    vp_s = vp.index_select(0, idx.cuda()).cpu()
    pt_s = torch.arange(idx.numel(), dtype=torch.int32).view(sel.shape)
    return kp_s, vp_s, pt_s, kl[rows]


def test_fp8_decode_at_bench_size(fa):
    """b64 x kv28672 over an FP8 cache (scales 1/32), the largest shape of
    the bench's FP8 leg."""
    s = 1.0 / 32
    kp, vp, pt, kl = device_cache(64, 28672, seed=101, fp8_scale=s)
    g = torch.Generator(device="cuda")
    g.manual_seed(102)
    q = torch.randn((64, HQ, D), generator=g, device="cuda").to(torch.bfloat16)
    out, lse = fa.fa512_decode_paged_fp8(q, kp, vp, pt.cuda(), kl.cuda(), k_scale=s, v_scale=s,
                                         max_kv_len=28672)
    torch.cuda.synchronize()
    assert fa.fa512_device_status() == 0
    kp_s, vp_s, pt_s, kl_s = sub_cache(kp.view(torch.uint8), vp.view(torch.uint8), pt, kl, SAMPLE)
    ro, rl = oracle.decode_paged_fp8(q[SAMPLE].cpu(), kp_s, vp_s, pt_s, kl_s, k_scale=s, v_scale=s)
    compare_o(out[SAMPLE].float().cpu().numpy(), ro)
    compare_lse(lse[SAMPLE].cpu().numpy(), rl)


def test_multi_token_decode_at_bench_size(fa):
    """b64 x kv16384 x 4 tokens (bf16), the bench's several-token leg."""
    kp, vp, pt, kl = device_cache(64, 16384, seed=103)
    g = torch.Generator(device="cuda")
    g.manual_seed(104)
    q = torch.randn((64, 4, HQ, D), generator=g, device="cuda").to(torch.bfloat16)
    out, lse = fa.fa512_decode_paged_q(q, kp, vp, pt.cuda(), kl.cuda(), max_kv_len=16384)
    torch.cuda.synchronize()
    assert fa.fa512_device_status() == 0
    kp_s, vp_s, pt_s, kl_s = sub_cache(kp, vp, pt, kl, SAMPLE)
    ro, rl = oracle.decode_paged_q(q[SAMPLE].cpu(), kp_s, vp_s, pt_s, kl_s)
    compare_o(out[SAMPLE].float().cpu().numpy(), ro)
    compare_lse(lse[SAMPLE].cpu().numpy(), rl)


def test_fp8_several_tokens_at_bench_size(fa):
    """The FP8 cache with 4 tokens per sequence (8 rows: the tensor-core
    streaming kernel at its largest row count), b64 x kv16384."""
    s = 1.0 / 32
    kp, vp, pt, kl = device_cache(64, 16384, seed=105, fp8_scale=s)
    g = torch.Generator(device="cuda")
    g.manual_seed(106)
    q = torch.randn((64, 4, HQ, D), generator=g, device="cuda").to(torch.bfloat16)
    out, lse = fa.fa512_decode_paged_fp8(q, kp, vp, pt.cuda(), kl.cuda(), k_scale=s, v_scale=s,
                                         max_kv_len=16384)
    torch.cuda.synchronize()
    assert fa.fa512_device_status() == 0
    kp_s, vp_s, pt_s, kl_s = sub_cache(kp.view(torch.uint8), vp.view(torch.uint8), pt, kl, SAMPLE)
    ro, rl = oracle.decode_paged_fp8(q[SAMPLE].cpu(), kp_s, vp_s, pt_s, kl_s, k_scale=s, v_scale=s)
    compare_o(out[SAMPLE].float().cpu().numpy(), ro)
    compare_lse(lse[SAMPLE].cpu().numpy(), rl)
