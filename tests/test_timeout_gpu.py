"""The bounded pipeline waits of the prefill kernel, driven to their bound.

Every mbarrier wait in the kernels is bounded by %globaltimer; a wait that
runs out records FA512_ERR_TIMEOUT in the device error word, the CTA pair
drains the MMAs it issued, frees its tensor memory and returns, so the
context stays usable.  Ordinary inputs never exhaust a wait, so this test
uses the library's test hook fa512_test_prefill_missing_load: the first CTA
pair's even CTA leaves out its first K load (a barrier nothing completes)
and every wait is bounded by 5 ms instead of 2 s.  Nothing faults, traps or
hangs: the waits end by their bound.

Checked: the call itself returns FA512_OK, fa512_device_status reports
FA512_ERR_TIMEOUT within a fraction of a second, and the next ordinary call
in the same process matches the fp64 oracle with a clean status.
"""
import ctypes
import time

import pytest
import torch

import oracle
from head_dim_flashattention_gb300 import workloads
from parity import compare_lse, compare_o

pytestmark = pytest.mark.gpu
D = 512
FA512_ERR_TIMEOUT = 4
WAIT_LIMIT_NS = 5_000_000


@pytest.fixture(scope="module")
def fa(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    import head_dim_flashattention_gb300 as fa
    lib = fa.load_library()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa512_test_prefill_missing_load.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I,
                                                    ctypes.c_uint64, P]
    lib.fa512_test_prefill_missing_load.restype = I
    return fa


def test_prefill_wait_bound_reports_timeout_and_next_call_is_correct(fa):
    lib = fa.load_library()
    assert fa.fa512_device_status(clear=True) == 0
    sq, hq, hk = 512, 8, 1
    q = workloads.randn_bf16((sq, hq, D), 91)
    k = workloads.randn_bf16((sq, hk, D), 92)
    v = workloads.randn_bf16((sq, hk, D), 93)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.zeros((sq, hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((hq, sq), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    t0 = time.perf_counter()
    st = lib.fa512_test_prefill_missing_load(
        qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), lse.data_ptr(), sq, sq, 0,
        hq, hk, D ** -0.5, 1, 0, WAIT_LIMIT_NS, stream.cuda_stream)
    assert st == 0, lib.fa512_last_error_message()
    status = fa.fa512_device_status(stream, clear=True)      # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == FA512_ERR_TIMEOUT
    assert elapsed < 1.0, elapsed                            # a few 5 ms bounds, not 2 s ones
    assert fa.fa512_device_status(stream, clear=True) == 0   # cleared

    # the same process, the same device: an ordinary call is correct
    o, l = fa.fa512_prefill(qd, kd, vd, q_offset=0, causal=True)
    assert fa.fa512_device_status(stream, clear=False) == 0
    ro, rl = oracle.prefill(q, k, v, q_offset=0, causal=True)
    compare_o(o.float().cpu().numpy(), ro)
    compare_lse(l.cpu().numpy(), rl)
