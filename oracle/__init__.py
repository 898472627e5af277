"""fp64 CPU oracle for head-dim-512 attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does: it shares no
code, header, table or helper with the CUDA path.

The arithmetic lives in ``fa512_oracle.c`` (plain fp64 loops, one
(row, head) pair at a time, the score vector materialised).  This module only
compiles it with gcc, marshals arrays through ctypes and returns numpy fp64
results.  Every input arrives as bf16 bit patterns and is widened exactly.

Sources: "Writing a FlashAttention Prefill Kernel for Gemma 4" (the score
matrix a classical attention materialises defines the result); "Flash-Decoding
for MQA in CUDA", section "The test that catches what parity misses" (an FP64
host reference over the same bf16-rounded inputs) and section "One KV head
breaks the textbook" (the live band of a decode query); vllm-project/
flash-attention PR #199, review item F4 (an empty row has LSE = -inf);
pegainfer issue #1051, "Proposed Plan" (a varlen prefill over the paged pool);
vllm-project/flash-attention PR #199, "Summary" (an FP8 paged KV cache).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa512_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfa512_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (idempotent)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_prefill.argtypes = [P, P, P, P, P, i, i, i, i, i, i,
                                           ctypes.c_double, i, i, P, i, i]
            lib.oracle_prefill.restype = i
            lib.oracle_decode_paged.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, i,
                                                ctypes.c_double, i, i]
            lib.oracle_decode_paged.restype = i
            lib.oracle_decode_paged_q.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, i, i,
                                                  ctypes.c_double, i, i]
            lib.oracle_decode_paged_q.restype = i
            lib.oracle_decode_paged_fp8.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, i, i,
                                                    ctypes.c_double, ctypes.c_double,
                                                    ctypes.c_double, i, i]
            lib.oracle_decode_paged_fp8.restype = i
            lib.oracle_e4m3_table.argtypes = [P]
            lib.oracle_e4m3_table.restype = None
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _bits(x) -> np.ndarray:
    """bf16 tensor/array -> contiguous uint16 numpy array of its bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype != torch.bfloat16:
                raise TypeError("oracle inputs must be bf16, got %s" % x.dtype)
            return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                        .view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype != np.uint16:
        raise TypeError("expected bf16 bit patterns as uint16, got %s" % a.dtype)
    return np.ascontiguousarray(a)


def _i32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def prefill(q, k, v, *, q_offset: int = 0, scale: float | None = None, causal: bool = True,
            window: int = 0, rows=None, threads: int | None = None):
    """Reference attention for a prefill chunk.

    q [seqlen_q, n_q_heads, D], k/v [seqlen_k, n_kv_heads, D] (bf16).
    Query row i sits at absolute position q_offset + i.  ``rows`` selects a
    subset of query rows (default: all).  Returns ``(out, lse)``:
    out [n_rows, n_q_heads, D] fp64 and lse [n_q_heads, n_rows] fp64.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if qb.ndim != 3 or kb.ndim != 3 or vb.shape != kb.shape:
        raise ValueError("bad shapes")
    sq, hq, d = qb.shape
    sk, hk, d2 = kb.shape
    if d2 != d:
        raise ValueError("head_dim mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows_arr = None if rows is None else _i32(rows)
    n_rows = sq if rows_arr is None else int(rows_arr.shape[0])
    out = np.zeros((n_rows, hq, d), dtype=np.float64)
    lse = np.zeros((hq, n_rows), dtype=np.float64)
    rc = _load().oracle_prefill(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(out), _ptr(lse),
                                sq, sk, int(q_offset), hq, hk, d, float(scale),
                                1 if causal else 0, int(window),
                                None if rows_arr is None else _ptr(rows_arr), n_rows,
                                threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_prefill rejected its arguments")
    return out, lse


def decode_paged(q, k_pages, v_pages, page_table, kv_lens, *, scale: float | None = None,
                 window: int = 0, threads: int | None = None):
    """Reference attention of one query token per sequence over a paged cache.

    q [batch, n_q_heads, D]; k_pages/v_pages [num_pages, page_size, n_kv_heads, D];
    page_table [batch, max_pages_per_seq] int; kv_lens [batch] int.
    Returns ``(out, lse)``: out [batch, n_q_heads, D] fp64, lse [batch, n_q_heads].
    """
    qb, kb, vb = _bits(q), _bits(k_pages), _bits(v_pages)
    pt, kl = _i32(page_table), _i32(kv_lens)
    bsz, hq, d = qb.shape
    npages, psz, hk, d2 = kb.shape
    if d2 != d or vb.shape != kb.shape or pt.ndim != 2 or pt.shape[0] != bsz:
        raise ValueError("bad shapes")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    lse = np.zeros((bsz, hq), dtype=np.float64)
    rc = _load().oracle_decode_paged(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pt), _ptr(kl),
                                     _ptr(out), _ptr(lse), bsz, hq, hk, d, psz, pt.shape[1],
                                     npages, float(scale), int(window),
                                     threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_decode_paged rejected its arguments")
    return out, lse


def decode_paged_q(q, k_pages, v_pages, page_table, kv_lens, *, scale: float | None = None,
                   window: int = 0, threads: int | None = None):
    """Reference attention of the last q_len tokens of each sequence over a paged cache.

    q [batch, q_len, n_q_heads, D]: query t of sequence b sits at position
    kv_lens[b] - q_len + t and sees the cache causally (and through the window).
    k_pages/v_pages [num_pages, page_size, n_kv_heads, D]; page_table
    [batch, max_pages_per_seq] int; kv_lens [batch] int.
    Returns ``(out, lse)``: out [batch, q_len, n_q_heads, D] fp64, lse [batch, q_len, n_q_heads].
    """
    qb, kb, vb = _bits(q), _bits(k_pages), _bits(v_pages)
    pt, kl = _i32(page_table), _i32(kv_lens)
    bsz, qlen, hq, d = qb.shape
    npages, psz, hk, d2 = kb.shape
    if d2 != d or vb.shape != kb.shape or pt.ndim != 2 or pt.shape[0] != bsz:
        raise ValueError("bad shapes")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((bsz, qlen, hq, d), dtype=np.float64)
    lse = np.zeros((bsz, qlen, hq), dtype=np.float64)
    rc = _load().oracle_decode_paged_q(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pt), _ptr(kl),
                                       _ptr(out), _ptr(lse), bsz, qlen, hq, hk, d, psz,
                                       pt.shape[1], npages, float(scale), int(window),
                                       threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_decode_paged_q rejected its arguments")
    return out, lse


def prefill_paged(q, k_pages, v_pages, page_table, cu_seqlens_q, seqused_k, *,
                  scale: float | None = None, causal: bool = True, window: int = 0,
                  threads: int | None = None):
    """Reference attention of a batch of prefill chunks over a paged KV cache.

    q [total_q, n_q_heads, D]: the chunk of sequence b is
    q[cu_seqlens_q[b]:cu_seqlens_q[b + 1]].  k_pages/v_pages [num_pages,
    page_size, n_kv_heads, D]; page_table [batch, max_pages_per_seq] int;
    seqused_k [batch] int.  The cache of sequence b holds positions
    0 .. seqused_k[b] - 1, position j in slot j % page_size of physical page
    page_table[b, j // page_size] (pegainfer issue #1051, "Proposed Plan": a
    varlen prefill reading the paged pool).  A chunk is the tail of its
    sequence, as in the chunked prefill of the same issue's "Description"
    (one chunk against everything before it): its row i sits at position
    seqused_k[b] - seqlen_q_b + i; a negative position sees no key under the
    causal mask.

    Steps: gather the used positions of each sequence in order through its
    page table (numpy indexing), then the contiguous prefill reference.
    Returns ``(out, lse)``: out [total_q, n_q_heads, D] fp64,
    lse [n_q_heads, total_q] fp64.
    """
    qb, kb, vb = _bits(q), _bits(k_pages), _bits(v_pages)
    pt, cu, used = _i32(page_table), _i32(cu_seqlens_q), _i32(seqused_k)
    total_q, hq, d = qb.shape
    npages, psz, hk, d2 = kb.shape
    batch = int(used.shape[0])
    if (d2 != d or vb.shape != kb.shape or pt.ndim != 2 or pt.shape[0] != batch
            or cu.shape != (batch + 1,)):
        raise ValueError("bad shapes")
    if cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] > total_q:
        raise ValueError("cu_seqlens_q must rise from 0 to at most total_q")
    if np.any(used < 0) or np.any(used > pt.shape[1] * psz):
        raise ValueError("seqused_k outside [0, max_pages_per_seq * page_size]")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((total_q, hq, d), dtype=np.float64)
    lse = np.zeros((hq, total_q), dtype=np.float64)
    for b in range(batch):
        r0, r1 = int(cu[b]), int(cu[b + 1])
        if r1 == r0:
            continue
        n = int(used[b])
        pos = np.arange(n)
        phys = pt[b, pos // psz]
        if np.any(phys < 0) or np.any(phys >= npages):
            raise ValueError("page table of sequence %d points outside the pool" % b)
        k_lin = np.ascontiguousarray(kb[phys, pos % psz])
        v_lin = np.ascontiguousarray(vb[phys, pos % psz])
        o_b, l_b = prefill(qb[r0:r1], k_lin, v_lin, q_offset=n - (r1 - r0), scale=scale,
                           causal=causal, window=window, threads=threads)
        out[r0:r1] = o_b
        lse[:, r0:r1] = l_b
    return out, lse


def _u8(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous().view(torch.uint8).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype != np.uint8:
        raise TypeError("expected e4m3 bytes as uint8, got %s" % a.dtype)
    return np.ascontiguousarray(a)


def e4m3_table() -> np.ndarray:
    """The 256 E4M3 codes decoded by the oracle (fp64; code 0x7F and 0xFF are NaN)."""
    out = np.zeros(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def decode_paged_fp8(q, k_pages, v_pages, page_table, kv_lens, *, k_scale: float = 1.0,
                     v_scale: float = 1.0, scale: float | None = None, window: int = 0,
                     threads: int | None = None):
    """Reference decode over an FP8 E4M3 paged cache.

    q [batch, n_q_heads, D] (one token) or [batch, q_len, n_q_heads, D] bf16;
    k_pages/v_pages [num_pages, page_size, n_kv_heads, D] e4m3 bytes (uint8 or
    torch.float8_e4m3fn); a key element is k_scale * e4m3(byte), a value
    element v_scale * e4m3(byte).  Returns ``(out, lse)`` shaped like q
    (lse without the head-dim axis), fp64.
    """
    qb, kb, vb = _bits(q), _u8(k_pages), _u8(v_pages)
    pt, kl = _i32(page_table), _i32(kv_lens)
    single = qb.ndim == 3
    if single:
        qb = qb[:, None]
    bsz, qlen, hq, d = qb.shape
    npages, psz, hk, d2 = kb.shape
    if d2 != d or vb.shape != kb.shape or pt.ndim != 2 or pt.shape[0] != bsz:
        raise ValueError("bad shapes")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    qb = np.ascontiguousarray(qb)
    out = np.zeros((bsz, qlen, hq, d), dtype=np.float64)
    lse = np.zeros((bsz, qlen, hq), dtype=np.float64)
    rc = _load().oracle_decode_paged_fp8(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pt), _ptr(kl),
                                         _ptr(out), _ptr(lse), bsz, qlen, hq, hk, d, psz,
                                         pt.shape[1], npages, float(scale), float(k_scale),
                                         float(v_scale), int(window),
                                         threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_decode_paged_fp8 rejected its arguments")
    if single:
        return out[:, 0], lse[:, 0]
    return out, lse
