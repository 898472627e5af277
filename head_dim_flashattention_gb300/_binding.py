"""ctypes binding of the fa512 C ABI (``include/fa512.h``).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the ``stream`` argument, and a non-zero status becomes a
:class:`Fa512Error`.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback of any kind.  torch supplies device memory
(outputs and the decode workspace when the caller passes none) and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HEAD_DIM = 512
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libfa512.so"
_lock = threading.Lock()
_lib = None

_STATUS = {
    0: "FA512_OK",
    1: "FA512_ERR_INVALID_ARG",
    2: "FA512_ERR_UNSUPPORTED",
    3: "FA512_ERR_CUDA",
    4: "FA512_ERR_TIMEOUT",
    5: "FA512_ERR_WORKSPACE",
    6: "FA512_ERR_DEVICE_INDEX",
}


class Fa512Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s (%d): %s" % (_STATUS.get(status, "?"), status, message))
        self.status = status


def library_path() -> str:
    return os.environ.get("FA512_LIBRARY", os.path.join(_HERE, _LIB_NAME))


def load_library():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise Fa512Error(3, "CUDA library %s is missing; build it with "
                                "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa512_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P]
        lib.fa512_prefill.restype = I
        lib.fa512_prefill_d256.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P]
        lib.fa512_prefill_d256.restype = I
        lib.fa512_prefill_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F,
                                            I, I, P]
        lib.fa512_prefill_paged.restype = I
        lib.fa512_decode_paged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I,
                                           P, Z, P]
        lib.fa512_decode_paged.restype = I
        lib.fa512_decode_paged_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I,
                                                   I, P]
        lib.fa512_decode_paged_noalloc.restype = I
        lib.fa512_decode_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.fa512_decode_workspace_bytes.restype = Z
        lib.fa512_decode_paged_q.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I,
                                             P, Z, P]
        lib.fa512_decode_paged_q.restype = I
        lib.fa512_decode_paged_fp8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, F,
                                               F, I, I, P, Z, P]
        lib.fa512_decode_paged_fp8.restype = I
        lib.fa512_decode_workspace_bytes_q.argtypes = [I, I, I, I, I, I, I]
        lib.fa512_decode_workspace_bytes_q.restype = Z
        lib.fa512_decode_auto_splits.argtypes = [I, I, I, I]
        lib.fa512_decode_auto_splits.restype = I
        lib.fa512_decode_auto_splits_fp8.argtypes = [I, I, I, I, I, I]
        lib.fa512_decode_auto_splits_fp8.restype = I
        lib.fa512_decode_workspace_bytes_fp8.argtypes = [I, I, I, I, I, I, I]
        lib.fa512_decode_workspace_bytes_fp8.restype = Z
        lib.fa512_device_status.argtypes = [P, I]
        lib.fa512_device_status.restype = I
        lib.fa512_status_string.argtypes = [I]
        lib.fa512_status_string.restype = ctypes.c_char_p
        lib.fa512_last_error_message.argtypes = []
        lib.fa512_last_error_message.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != 0:
        lib = load_library()
        msg = lib.fa512_last_error_message()
        raise Fa512Error(status, msg.decode() if msg else "")


def _dptr(t: torch.Tensor | None, name: str, dtype=None) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise Fa512Error(1, "%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise Fa512Error(1, "%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise Fa512Error(1, "%s must be contiguous" % name)
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def fa512_status_string(status: int) -> str:
    return load_library().fa512_status_string(int(status)).decode()


def fa512_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  out: torch.Tensor | None = None, lse: torch.Tensor | None = None, *,
                  q_offset: int = 0, scale: float | None = None, causal: bool = True,
                  window: int = 0, return_lse: bool = True, stream=None):
    """Attention forward of one prefill chunk; returns ``(out, lse)``.

    q [seqlen_q, n_q_heads, 512], k/v [seqlen_k, n_kv_heads, 512], bf16 CUDA.
    out is allocated when not given; lse [n_q_heads, seqlen_q] fp32 likewise
    (``return_lse=False`` passes NULL).
    """
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape != v.shape:
        raise Fa512Error(1, "q, k, v must be [seq, heads, 512] with k.shape == v.shape")
    sq, hq, d = q.shape
    sk, hk, _ = k.shape
    if out is None:
        out = torch.empty((sq, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((hq, sq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    _check(lib.fa512_prefill(_dptr(q, "q", torch.bfloat16), _dptr(k, "k", torch.bfloat16),
                             _dptr(v, "v", torch.bfloat16), _dptr(out, "out", torch.bfloat16),
                             _dptr(lse, "lse", torch.float32), sq, sk, int(q_offset), hq, hk,
                             float(scale), 1 if causal else 0, int(window), _stream(stream)))
    return out, lse


def fa512_prefill_d256(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       out: torch.Tensor | None = None, lse: torch.Tensor | None = None, *,
                       q_offset: int = 0, scale: float | None = None, causal: bool = True,
                       window: int = 0, return_lse: bool = True, stream=None):
    """Attention forward of one prefill chunk with heads of 256 dimensions
    (the sliding-window local layers); returns ``(out, lse)``.

    q [seqlen_q, n_q_heads, 256], k/v [seqlen_k, n_kv_heads, 256], bf16 CUDA.
    """
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape != v.shape:
        raise Fa512Error(1, "q, k, v must be [seq, heads, 256] with k.shape == v.shape")
    sq, hq, d = q.shape
    sk, hk, dk = k.shape
    if d != 256 or dk != 256:
        raise Fa512Error(1, "fa512_prefill_d256 takes heads of 256 dimensions")
    if out is None:
        out = torch.empty((sq, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((hq, sq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    _check(lib.fa512_prefill_d256(_dptr(q, "q", torch.bfloat16), _dptr(k, "k", torch.bfloat16),
                                  _dptr(v, "v", torch.bfloat16), _dptr(out, "out", torch.bfloat16),
                                  _dptr(lse, "lse", torch.float32), sq, sk, int(q_offset), hq, hk,
                                  float(scale), 1 if causal else 0, int(window), _stream(stream)))
    return out, lse


def fa512_prefill_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                        page_table: torch.Tensor, cu_seqlens_q: torch.Tensor,
                        seqused_k: torch.Tensor, out: torch.Tensor | None = None,
                        lse: torch.Tensor | None = None, *, max_seqlen_q: int,
                        scale: float | None = None, causal: bool = True, window: int = 0,
                        return_lse: bool = True, stream=None):
    """Attention forward of a batch of prefill chunks (varlen rows) over a
    paged KV cache; returns ``(out, lse)``.

    q [total_q, n_q_heads, 512] bf16; k_pages/v_pages [num_pages, page_size,
    n_kv_heads, 512] bf16; page_table [batch, max_pages_per_seq] int32;
    cu_seqlens_q [batch + 1] int32; seqused_k [batch] int32 (all CUDA).
    ``max_seqlen_q`` bounds the chunk lengths on the host.  out is allocated
    when not given; lse [n_q_heads, total_q] fp32 likewise.
    """
    if q.dim() != 3 or k_pages.dim() != 4 or k_pages.shape != v_pages.shape:
        raise Fa512Error(1, "q must be [total_q, heads, 512], pages [n, page, heads, 512]")
    if page_table.dim() != 2 or cu_seqlens_q.dim() != 1 or seqused_k.dim() != 1:
        raise Fa512Error(1, "page_table [batch, pages], cu_seqlens_q [batch + 1], seqused_k [batch]")
    total_q, hq, d = q.shape
    npages, psz, hk, _ = k_pages.shape
    bsz, mpps = page_table.shape
    if cu_seqlens_q.shape[0] != bsz + 1 or seqused_k.shape[0] != bsz:
        raise Fa512Error(1, "cu_seqlens_q must have batch + 1 entries and seqused_k batch")
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((hq, total_q), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    _check(lib.fa512_prefill_paged(
        _dptr(q, "q", torch.bfloat16), _dptr(k_pages, "k_pages", torch.bfloat16),
        _dptr(v_pages, "v_pages", torch.bfloat16), _dptr(page_table, "page_table", torch.int32),
        _dptr(cu_seqlens_q, "cu_seqlens_q", torch.int32),
        _dptr(seqused_k, "seqused_k", torch.int32), _dptr(out, "out", torch.bfloat16),
        _dptr(lse, "lse", torch.float32), bsz, total_q, int(max_seqlen_q), hq, hk, psz, npages,
        mpps, float(scale), 1 if causal else 0, int(window), _stream(stream)))
    return out, lse


def fa512_decode_workspace_bytes(batch: int, n_q_heads: int, n_kv_heads: int, page_size: int,
                                 max_kv_len: int, num_splits: int = 0) -> int:
    return int(load_library().fa512_decode_workspace_bytes(batch, n_q_heads, n_kv_heads,
                                                           page_size, max_kv_len, num_splits))


def fa512_decode_auto_splits(batch: int, n_kv_heads: int, page_size: int, max_kv_len: int) -> int:
    return int(load_library().fa512_decode_auto_splits(batch, n_kv_heads, page_size, max_kv_len))


def fa512_decode_auto_splits_fp8(batch: int, q_len: int, n_q_heads: int, n_kv_heads: int,
                                 page_size: int, max_kv_len: int) -> int:
    return int(load_library().fa512_decode_auto_splits_fp8(batch, q_len, n_q_heads, n_kv_heads,
                                                           page_size, max_kv_len))


def fa512_decode_workspace_bytes_fp8(batch: int, q_len: int, n_q_heads: int, n_kv_heads: int,
                                     page_size: int, max_kv_len: int, num_splits: int = 0) -> int:
    return int(load_library().fa512_decode_workspace_bytes_fp8(batch, q_len, n_q_heads, n_kv_heads,
                                                               page_size, max_kv_len, num_splits))


def fa512_decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                       page_table: torch.Tensor, kv_lens: torch.Tensor,
                       out: torch.Tensor | None = None, lse: torch.Tensor | None = None, *,
                       max_kv_len: int | None = None, scale: float | None = None,
                       window: int = 0, num_splits: int = 0,
                       workspace: torch.Tensor | None = None, return_lse: bool = True,
                       stream=None):
    """One query token per sequence over a paged KV cache; returns ``(out, lse)``.

    q [batch, n_q_heads, 512]; k_pages/v_pages [num_pages, page_size,
    n_kv_heads, 512] bf16; page_table [batch, max_pages_per_seq] int32;
    kv_lens [batch] int32 (all CUDA).  ``max_kv_len`` bounds kv_lens on the
    host (default: the page table's capacity).
    """
    if q.dim() != 3 or k_pages.dim() != 4 or k_pages.shape != v_pages.shape:
        raise Fa512Error(1, "q must be [batch, heads, 512], pages [n, page, heads, 512]")
    bsz, hq, d = q.shape
    npages, psz, hk, _ = k_pages.shape
    if page_table.dim() != 2:
        raise Fa512Error(1, "page_table must be [batch, max_pages_per_seq]")
    mpps = page_table.shape[1]
    if max_kv_len is None:
        max_kv_len = mpps * psz
    if out is None:
        out = torch.empty((bsz, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((bsz, hq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    need = int(lib.fa512_decode_workspace_bytes(bsz, hq, hk, psz, int(max_kv_len),
                                                int(num_splits)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.fa512_decode_paged(
        _dptr(q, "q", torch.bfloat16), _dptr(k_pages, "k_pages", torch.bfloat16),
        _dptr(v_pages, "v_pages", torch.bfloat16), _dptr(page_table, "page_table", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), _dptr(out, "out", torch.bfloat16),
        _dptr(lse, "lse", torch.float32), bsz, hq, hk, psz, npages, mpps, int(max_kv_len),
        float(scale), int(window), int(num_splits), _dptr(workspace, "workspace"), ws_bytes,
        _stream(stream)))
    return out, lse


def fa512_decode_paged_noalloc(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                               page_table: torch.Tensor, kv_lens: torch.Tensor,
                               out: torch.Tensor, lse: torch.Tensor | None = None, *,
                               max_kv_len: int | None = None, scale: float | None = None,
                               window: int = 0, num_splits: int = 0, stream=None):
    """fa512_decode_paged without a workspace: the split partials go to the
    library's static device array (for callers that cannot allocate).  The
    caller passes ``out`` (and ``lse``, or None); nothing is allocated here
    either.  Arguments as for :func:`fa512_decode_paged`."""
    if q.dim() != 3 or k_pages.dim() != 4 or k_pages.shape != v_pages.shape:
        raise Fa512Error(1, "q must be [batch, heads, 512], pages [n, page, heads, 512]")
    bsz, hq, d = q.shape
    npages, psz, hk, _ = k_pages.shape
    if page_table.dim() != 2:
        raise Fa512Error(1, "page_table must be [batch, max_pages_per_seq]")
    mpps = page_table.shape[1]
    if max_kv_len is None:
        max_kv_len = mpps * psz
    if scale is None:
        scale = d ** -0.5
    _check(load_library().fa512_decode_paged_noalloc(
        _dptr(q, "q", torch.bfloat16), _dptr(k_pages, "k_pages", torch.bfloat16),
        _dptr(v_pages, "v_pages", torch.bfloat16), _dptr(page_table, "page_table", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), _dptr(out, "out", torch.bfloat16),
        _dptr(lse, "lse", torch.float32), bsz, hq, hk, psz, npages, mpps, int(max_kv_len),
        float(scale), int(window), int(num_splits), _stream(stream)))
    return out, lse


def fa512_decode_paged_q(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                         page_table: torch.Tensor, kv_lens: torch.Tensor,
                         out: torch.Tensor | None = None, lse: torch.Tensor | None = None, *,
                         max_kv_len: int | None = None, scale: float | None = None,
                         window: int = 0, num_splits: int = 0,
                         workspace: torch.Tensor | None = None, return_lse: bool = True,
                         stream=None):
    """q_len query tokens per sequence (its last q_len positions) over a paged
    KV cache; returns ``(out, lse)``.

    q [batch, q_len, n_q_heads, 512]; out like q; lse [batch, q_len, n_q_heads].
    Other arguments as :func:`fa512_decode_paged`.
    """
    if q.dim() != 4 or k_pages.dim() != 4 or k_pages.shape != v_pages.shape:
        raise Fa512Error(1, "q must be [batch, q_len, heads, 512], pages [n, page, heads, 512]")
    bsz, qlen, hq, d = q.shape
    npages, psz, hk, _ = k_pages.shape
    if page_table.dim() != 2:
        raise Fa512Error(1, "page_table must be [batch, max_pages_per_seq]")
    mpps = page_table.shape[1]
    if max_kv_len is None:
        max_kv_len = mpps * psz
    if out is None:
        out = torch.empty((bsz, qlen, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((bsz, qlen, hq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    need = int(lib.fa512_decode_workspace_bytes_q(bsz, qlen, hq, hk, psz, int(max_kv_len),
                                                  int(num_splits)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.fa512_decode_paged_q(
        _dptr(q, "q", torch.bfloat16), _dptr(k_pages, "k_pages", torch.bfloat16),
        _dptr(v_pages, "v_pages", torch.bfloat16), _dptr(page_table, "page_table", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), _dptr(out, "out", torch.bfloat16),
        _dptr(lse, "lse", torch.float32), bsz, qlen, hq, hk, psz, npages, mpps, int(max_kv_len),
        float(scale), int(window), int(num_splits), _dptr(workspace, "workspace"), ws_bytes,
        _stream(stream)))
    return out, lse


def _e4m3_bytes(t: torch.Tensor, name: str) -> int | None:
    """Device pointer of an E4M3 cache given as uint8 codes or torch.float8_e4m3fn."""
    if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn:
        return _dptr(t, name)
    return _dptr(t, name, torch.uint8)


def fa512_decode_paged_fp8(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                           page_table: torch.Tensor, kv_lens: torch.Tensor,
                           out: torch.Tensor | None = None, lse: torch.Tensor | None = None, *,
                           k_scale: float = 1.0, v_scale: float = 1.0,
                           max_kv_len: int | None = None, scale: float | None = None,
                           window: int = 0, num_splits: int = 0,
                           workspace: torch.Tensor | None = None, return_lse: bool = True,
                           stream=None):
    """Decode over a paged KV cache stored in FP8 E4M3; returns ``(out, lse)``.

    q [batch, n_q_heads, 512] (one token) or [batch, q_len, n_q_heads, 512] bf16;
    k_pages / v_pages [num_pages, page_size, n_kv_heads, 512] as uint8 codes or
    torch.float8_e4m3fn; a key element is k_scale * e4m3, a value element
    v_scale * e4m3.  out / lse are shaped like q (lse without the head dim).
    Other arguments as :func:`fa512_decode_paged_q`.
    """
    single = q.dim() == 3
    q4 = q.unsqueeze(1) if single else q
    if q4.dim() != 4 or k_pages.dim() != 4 or k_pages.shape != v_pages.shape:
        raise Fa512Error(1, "q must be [batch, (q_len,) heads, 512], pages [n, page, heads, 512]")
    bsz, qlen, hq, d = q4.shape
    npages, psz, hk, _ = k_pages.shape
    if page_table.dim() != 2:
        raise Fa512Error(1, "page_table must be [batch, max_pages_per_seq]")
    mpps = page_table.shape[1]
    if max_kv_len is None:
        max_kv_len = mpps * psz
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    need = int(lib.fa512_decode_workspace_bytes_fp8(bsz, qlen, hq, hk, psz, int(max_kv_len),
                                                    int(num_splits)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.fa512_decode_paged_fp8(
        _dptr(q, "q", torch.bfloat16), _e4m3_bytes(k_pages, "k_pages"),
        _e4m3_bytes(v_pages, "v_pages"), _dptr(page_table, "page_table", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), _dptr(out, "out", torch.bfloat16),
        _dptr(lse, "lse", torch.float32), bsz, qlen, hq, hk, psz, npages, mpps, int(max_kv_len),
        float(scale), float(k_scale), float(v_scale), int(window), int(num_splits),
        _dptr(workspace, "workspace"), ws_bytes, _stream(stream)))
    return out, lse


def fa512_device_status(stream=None, clear: bool = True) -> int:
    """Synchronise ``stream`` and return (optionally clearing) the device error word."""
    return int(load_library().fa512_device_status(_stream(stream), 1 if clear else 0))
