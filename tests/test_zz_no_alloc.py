"""fa512_decode_paged_noalloc: the decode entry point for callers that cannot
call cudaMalloc (they get device pointers for inputs and outputs from another
framework and have no allocator of their own).  It keeps the split partials
in the library's fixed static device array instead of a caller workspace.

Called through the C ABI with ctypes and compared with fa512_decode_paged on
the same inputs, on two calls in a row (the second with a different shape,
so stale contents of the shared array from the first call would show).  Both
entry points run the same kernels with the same split count, so O and LSE
must agree bit for bit.  A third test checks that a call allocates nothing:
neither torch's allocator nor the device's free memory moves.  The file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from head_dim_flashattention_gb300 import workloads

pytestmark = pytest.mark.gpu
STATIC_SCRATCH_BYTES = 32 * 1024 * 1024


@pytest.fixture(scope="module")
def lib(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    import head_dim_flashattention_gb300 as fa
    lib = fa.load_library()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa512_decode_paged_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P]
    lib.fa512_decode_paged_noalloc.restype = I
    return lib


def _dev(pc):
    return {k: getattr(pc, k).cuda() for k in ("q", "k_pages", "v_pages", "page_table", "kv_lens")}


def _outputs(pc):
    bsz, hq, _ = pc.q.shape
    return (torch.full((bsz, hq, 512), float("nan"), dtype=torch.bfloat16, device="cuda"),
            torch.full((bsz, hq), float("nan"), dtype=torch.float32, device="cuda"))


def _noalloc(lib, pc, d, num_splits, window=0, outputs=None):
    bsz, hq, _ = pc.q.shape
    npages, psz, hk, _ = pc.k_pages.shape
    out, lse = outputs if outputs is not None else _outputs(pc)
    st = lib.fa512_decode_paged_noalloc(
        d["q"].data_ptr(), d["k_pages"].data_ptr(), d["v_pages"].data_ptr(),
        d["page_table"].data_ptr(), d["kv_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
        bsz, hq, hk, psz, npages, pc.page_table.shape[1], pc.max_kv_len, 512 ** -0.5, window,
        num_splits, torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.fa512_last_error_message()
    return out, lse


def _with_workspace(pc, d, num_splits, window=0):
    import head_dim_flashattention_gb300 as fa
    return fa.fa512_decode_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"],
                                 d["kv_lens"], max_kv_len=pc.max_kv_len, num_splits=num_splits,
                                 window=window)


def _same(a, b):
    (oa, la), (ob, lb) = a, b
    assert torch.isfinite(oa.float()).all()
    assert torch.equal(oa, ob), "O differs from the workspace entry point"
    assert np.array_equal(la.cpu().numpy(), lb.cpu().numpy()), "LSE differs"


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    first = workloads.paged_decode_inputs(16, [4096] * 16, 8, 4, 64, seed=51)
    second = workloads.paged_decode_inputs(3, [1000, 64, 0], 8, 4, 64, seed=52)
    d1, d2 = _dev(first), _dev(second)
    a1 = _noalloc(lib, first, d1, 0)
    a2 = _noalloc(lib, second, d2, 5, window=300)
    torch.cuda.synchronize()
    b1 = _with_workspace(first, d1, 0)
    b2 = _with_workspace(second, d2, 5, window=300)
    torch.cuda.synchronize()
    _same(a1, b1)
    _same(a2, b2)


def test_noalloc_rejects_shapes_beyond_the_static_array(lib):
    # 64 sequences x 8 heads x 1024 splits of 2 KiB partials > 32 MiB
    st = lib.fa512_decode_paged_noalloc(16, 16, 16, 16, 16, 16, None, 64, 8, 4, 64, 10, 448,
                                        28672, 0.04, 0, 1024, None)
    assert st == 5
    assert b"static array" in lib.fa512_last_error_message()


def test_noalloc_call_allocates_nothing(lib):
    """After a first call (which looks up the static array), further calls on
    other shapes leave torch's allocator and the device's free memory as
    they were."""
    first = workloads.paged_decode_inputs(4, [2048, 700, 64, 1], 8, 4, 64, seed=53)
    second = workloads.paged_decode_inputs(2, [5000, 300], 8, 4, 64, seed=54)
    d1, d2 = _dev(first), _dev(second)
    # every kernel these shapes use has run once (loading device code can take memory)
    _with_workspace(first, d1, 0)
    _with_workspace(second, d2, 3)
    out1 = _noalloc(lib, first, d1, 0)
    outs2, outs3 = _outputs(second), _outputs(first)
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    _noalloc(lib, second, d2, 3, outputs=outs2)
    _noalloc(lib, first, d1, 0, outputs=outs3)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    assert after[0] == before[0], ("torch allocator moved", before, after)
    assert after[1] == before[1], ("device free memory moved", before, after)
    _same(out1, outs3)
    _same(outs2, _with_workspace(second, d2, 3))
