"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/fa512.h declares; host-side validation answers without touching
a device."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import head_dim_flashattention_gb300 as fa
from head_dim_flashattention_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa512.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa512_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_two_hot_path_calls():
    names = declared_functions()
    assert "fa512_prefill" in names and "fa512_decode_paged" in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in _binding._STATUS.items():
        assert fa.fa512_status_string(code) == name


def _prefill(lib, **kw):
    args = dict(q=16, k=16, v=16, out=16, lse=None, sq=4, sk=4, off=0, hq=8, hk=2,
                scale=0.05, causal=1, window=0)
    args.update(kw)
    return lib.fa512_prefill(args["q"], args["k"], args["v"], args["out"], args["lse"],
                             args["sq"], args["sk"], args["off"], args["hq"], args["hk"],
                             args["scale"], args["causal"], args["window"], None)


def test_prefill_rejects_bad_arguments_before_any_launch(lib):
    assert _prefill(lib, hq=6, hk=4) == 1            # heads not a multiple
    assert _prefill(lib, hk=0) == 1
    assert _prefill(lib, sq=-1) == 1
    assert _prefill(lib, off=-3) == 1
    assert _prefill(lib, q=None) == 1
    assert _prefill(lib, q=24) == 1                  # misaligned
    assert _prefill(lib, scale=float("nan")) == 1
    assert _prefill(lib, hq=256, hk=1) == 2          # G > 128
    assert _prefill(lib, off=2**31 - 2, sq=4) == 1   # positions overflow
    assert _prefill(lib, sq=0, q=None) == 0          # empty chunk: no-op
    assert "multiple" in lib.fa512_last_error_message().decode() or True


def _decode(lib, **kw):
    a = dict(q=16, kp=16, vp=16, pt=16, kl=16, out=16, lse=None, b=2, hq=8, hk=4, ps=64,
             npages=10, mpps=4, maxlen=200, scale=0.05, window=0, splits=0, ws=256,
             wsb=1 << 30)
    a.update(kw)
    return lib.fa512_decode_paged(a["q"], a["kp"], a["vp"], a["pt"], a["kl"], a["out"], a["lse"],
                                  a["b"], a["hq"], a["hk"], a["ps"], a["npages"], a["mpps"],
                                  a["maxlen"], a["scale"], a["window"], a["splits"], a["ws"],
                                  a["wsb"], None)


def test_decode_rejects_bad_arguments_before_any_launch(lib):
    assert _decode(lib, ps=48) == 2
    assert _decode(lib, hq=68, hk=2) == 2            # G > 16
    assert _decode(lib, hq=6, hk=4) == 1
    assert _decode(lib, maxlen=300) == 1             # beyond the page table
    assert _decode(lib, splits=2000) == 1
    assert _decode(lib, npages=0) == 1
    assert _decode(lib, ws=None) == 5
    assert _decode(lib, wsb=16) == 5
    assert _decode(lib, ws=272) == 5                 # not 256-byte aligned
    assert _decode(lib, b=0, q=None) == 0            # empty batch: no-op


def test_workspace_size_and_auto_splits(lib):
    n = fa.fa512_decode_workspace_bytes(4, 8, 4, 64, 4096, 3)
    assert n == 4 * 8 * 3 * 512 * 4 + ((4 * 8 * 3 * 2 * 4 + 255) // 256) * 256
    assert fa.fa512_decode_auto_splits(1, 4, 64, 0) == 1
    s = fa.fa512_decode_auto_splits(1, 4, 64, 4096)
    assert 1 <= s <= 4096 // 32
    # more work per sequence never asks for fewer splits of a single sequence
    assert fa.fa512_decode_auto_splits(1, 4, 64, 28672) >= s
    assert fa.fa512_decode_workspace_bytes(-1, 8, 4, 64, 10, 0) == 0


def test_fp8_workspace_and_auto_splits(lib):
    # an explicit split count: the partial layout of the bf16 calls
    assert (fa.fa512_decode_workspace_bytes_fp8(4, 1, 8, 4, 64, 4096, 3)
            == fa.fa512_decode_workspace_bytes(4, 8, 4, 64, 4096, 3))
    assert (fa.fa512_decode_workspace_bytes_fp8(4, 2, 8, 4, 64, 4096, 3)
            == lib.fa512_decode_workspace_bytes_q(4, 2, 8, 4, 64, 4096, 3))
    # the automatic choice of the one-split-per-CTA kernel: at most 128
    # splits, at most one per tile, and the workspace query sizes for it
    for b, n in ((1, 4096), (16, 16384), (64, 28672)):
        s = fa.fa512_decode_auto_splits_fp8(b, 1, 8, 4, 64, n)
        assert 1 <= s <= min(128, n // 32)
        assert (fa.fa512_decode_workspace_bytes_fp8(b, 1, 8, 4, 64, n, 0)
                == fa.fa512_decode_workspace_bytes_fp8(b, 1, 8, 4, 64, n, s))
    # more rows than that kernel takes (q_len x G > 8): the bf16 choice
    assert (fa.fa512_decode_auto_splits_fp8(16, 8, 8, 4, 64, 16384)
            == fa.fa512_decode_auto_splits(16, 4, 64, 16384))
    assert fa.fa512_decode_auto_splits_fp8(1, 1, 8, 4, 64, 0) == 1
    assert fa.fa512_decode_workspace_bytes_fp8(-1, 1, 8, 4, 64, 10, 0) == 0
    assert fa.fa512_decode_workspace_bytes_fp8(4, 0, 8, 4, 64, 10, 0) == 0


def test_fp8_auto_splits_on_152_sms(lib):
    # with no GPU the library plans for 152 SMs: the counts the fitted time
    # models give on the nine decode shapes (8/4 heads, page 64)
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the counts are for 152 SMs")
    want = {(1, 4096): 64, (1, 16384): 74, (1, 28672): 75,
            (16, 4096): 16, (16, 16384): 32, (16, 28672): 39,
            (64, 4096): 8, (64, 16384): 19, (64, 28672): 28}
    got = {(b, n): fa.fa512_decode_auto_splits_fp8(b, 1, 8, 4, 64, n) for b, n in want}
    assert got == want


def _decode_q(lib, **kw):
    a = dict(q=16, kp=16, vp=16, pt=16, kl=16, out=16, lse=None, b=2, ql=4, hq=8, hk=4, ps=64,
             npages=10, mpps=4, maxlen=200, scale=0.05, window=0, splits=0, ws=256,
             wsb=1 << 30)
    a.update(kw)
    return lib.fa512_decode_paged_q(a["q"], a["kp"], a["vp"], a["pt"], a["kl"], a["out"],
                                    a["lse"], a["b"], a["ql"], a["hq"], a["hk"], a["ps"],
                                    a["npages"], a["mpps"], a["maxlen"], a["scale"], a["window"],
                                    a["splits"], a["ws"], a["wsb"], None)


def test_multi_token_decode_validation_and_workspace(lib):
    assert _decode_q(lib, ql=0) == 1                 # q_len >= 1
    assert _decode_q(lib, ql=9, hq=8, hk=4) == 2     # 9 tokens x G 2 > 16 rows
    assert _decode_q(lib, ql=3, hq=48, hk=8) == 2    # 3 x G 6 = 18 > 16
    assert _decode_q(lib, wsb=16) == 5
    assert _decode_q(lib, b=0, q=None) == 0
    # the workspace covers batch x q_len query rows; q_len 1 is the single-token size
    n4 = lib.fa512_decode_workspace_bytes_q(4, 4, 8, 4, 64, 4096, 3)
    assert n4 == 16 * 8 * 3 * 512 * 4 + ((16 * 8 * 3 * 2 * 4 + 255) // 256) * 256
    assert (lib.fa512_decode_workspace_bytes_q(4, 1, 8, 4, 64, 4096, 3)
            == fa.fa512_decode_workspace_bytes(4, 8, 4, 64, 4096, 3))
    assert lib.fa512_decode_workspace_bytes_q(4, 0, 8, 4, 64, 4096, 3) == 0


def _prefill_paged(lib, **kw):
    args = dict(q=16, k=16, v=16, pt=16, cu=16, used=16, out=16, lse=None, batch=2, total_q=8,
                max_q=4, hq=8, hk=2, page=64, npages=4, mpps=2, scale=0.05, causal=1, window=0)
    args.update(kw)
    a = args
    return lib.fa512_prefill_paged(a["q"], a["k"], a["v"], a["pt"], a["cu"], a["used"], a["out"],
                                   a["lse"], a["batch"], a["total_q"], a["max_q"], a["hq"],
                                   a["hk"], a["page"], a["npages"], a["mpps"], a["scale"],
                                   a["causal"], a["window"], None)


def test_prefill_paged_rejects_bad_arguments_before_any_launch(lib):
    assert _prefill_paged(lib, batch=-1) == 1
    assert _prefill_paged(lib, total_q=-1) == 1
    assert _prefill_paged(lib, hq=6, hk=4) == 1
    assert _prefill_paged(lib, page=32) == 2          # a page must hold whole 64-key half tiles
    assert _prefill_paged(lib, page=100) == 2
    assert _prefill_paged(lib, npages=0) == 1
    assert _prefill_paged(lib, mpps=0) == 1
    assert _prefill_paged(lib, npages=1 << 24, page=256) == 2   # pool rows past int32
    assert _prefill_paged(lib, scale=float("inf")) == 1
    assert _prefill_paged(lib, q=None) == 1
    assert _prefill_paged(lib, cu=None) == 1
    assert _prefill_paged(lib, out=24) == 1           # misaligned
    assert _prefill_paged(lib, used=18) == 1          # int32 array misaligned
    assert _prefill_paged(lib, hq=256, hk=1) == 2
    # empty batches are no-ops that touch nothing
    assert _prefill_paged(lib, batch=0, q=None) == 0
    assert _prefill_paged(lib, total_q=0, q=None) == 0
    assert _prefill_paged(lib, max_q=0, q=None) == 0


def test_prefill_d256_rejects_bad_arguments_before_any_launch(lib):
    def call(**kw):
        a = dict(q=16, k=16, v=16, out=16, lse=None, sq=4, sk=4, off=0, hq=8, hk=2,
                 scale=0.05, causal=1, window=1024)
        a.update(kw)
        return lib.fa512_prefill_d256(a["q"], a["k"], a["v"], a["out"], a["lse"], a["sq"],
                                      a["sk"], a["off"], a["hq"], a["hk"], a["scale"],
                                      a["causal"], a["window"], None)
    assert call(hq=6, hk=4) == 1
    assert call(sq=-1) == 1
    assert call(off=-1) == 1
    assert call(q=None) == 1
    assert call(out=8) == 1
    assert call(scale=float("nan")) == 1
    assert call(hq=256, hk=1) == 2
    assert call(sq=0, q=None) == 0


def _decode_fp8(lib, **kw):
    a = dict(q=16, kp=16, vp=16, pt=16, kl=16, out=16, lse=None, b=2, ql=1, hq=8, hk=4, ps=64,
             npages=10, mpps=4, maxlen=200, scale=0.05, ks=0.03, vs=0.04, window=0, splits=0,
             ws=256, wsb=1 << 30)
    a.update(kw)
    return lib.fa512_decode_paged_fp8(a["q"], a["kp"], a["vp"], a["pt"], a["kl"], a["out"],
                                      a["lse"], a["b"], a["ql"], a["hq"], a["hk"], a["ps"],
                                      a["npages"], a["mpps"], a["maxlen"], a["scale"], a["ks"],
                                      a["vs"], a["window"], a["splits"], a["ws"], a["wsb"], None)


def test_fp8_decode_rejects_bad_arguments_before_any_launch(lib):
    inf, nan = float("inf"), float("nan")
    assert _decode_fp8(lib, ks=inf) == 1             # scales must be finite
    assert _decode_fp8(lib, vs=nan) == 1
    assert _decode_fp8(lib, scale=nan) == 1
    assert _decode_fp8(lib, ql=0) == 1
    assert _decode_fp8(lib, ql=9, hq=8, hk=4) == 2   # 18 rows > 16
    assert _decode_fp8(lib, ps=48) == 2
    assert _decode_fp8(lib, maxlen=300) == 1         # beyond the page table
    assert _decode_fp8(lib, ws=None) == 5
    assert _decode_fp8(lib, wsb=16) == 5
    assert _decode_fp8(lib, kp=8) == 1               # pages not 16-byte aligned
    assert _decode_fp8(lib, b=0, q=None) == 0        # empty batch: no-op
    assert _decode_fp8(lib, ks=inf) == 1 and b"finite" in lib.fa512_last_error_message()


def test_fp8_binding_rejects_a_bf16_cache_before_the_library():
    torch = pytest.importorskip("torch")
    q = torch.zeros((1, 8, 512), dtype=torch.bfloat16)
    pages = torch.zeros((1, 64, 4, 512), dtype=torch.bfloat16)
    with pytest.raises(fa.Fa512Error):
        fa.fa512_decode_paged_fp8(q, pages, pages, torch.zeros((1, 1), dtype=torch.int32),
                                  torch.ones(1, dtype=torch.int32))


def test_timeout_hook_rejects_bad_bounds_before_any_launch(lib):
    """The test hook that exhausts a prefill wait refuses bounds outside
    [1 ms, 2 s] and an empty key sequence on the host."""
    f = lib.fa512_test_prefill_missing_load
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int,
                                                                ctypes.c_int, ctypes.c_uint64,
                                                                ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(16, 16, 16, 16, None, 4, 4, 0, 8, 2, 0.05, 1, 0, 10, None) == 1
    assert f(16, 16, 16, 16, None, 4, 4, 0, 8, 2, 0.05, 1, 0, 3_000_000_000, None) == 1
    assert f(16, 16, 16, 16, None, 4, 0, 0, 8, 2, 0.05, 1, 0, 5_000_000, None) == 1
