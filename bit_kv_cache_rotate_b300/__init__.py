"""bit_kv_cache_rotate_b300 -- 4-bit rotated KV-cache decode attention on B300.

Thin Python binding over the C ABI of ``libkv4.so`` (declared in
``include/kv4.h``).  Every function here only marshals torch tensors into
pointers and sizes and calls the entry point of the same name; all the work
runs in the library's CUDA kernels on the current torch stream.  There is no
CPU fallback: the first call raises ImportError if the library has not been
built (``python -m bit_kv_cache_rotate_b300.build``).  The library is loaded
on first use so that the workload generator in this package can be imported
on machines without the build.

Method: "UltraQuant on AMD Instinct" (section "What is UltraQuant"): each key
and value head vector is Walsh-Hadamard rotated and stored as FP4 E2M1 codes
with one power-of-two UE8M0 scale per 32 channels (17 bytes per 32 values);
decode attention reads the codes directly.  An FP8 E4M3 cache with per-head
scales is provided as the comparison path (section "UltraQuant vs 8-bit KV").
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkv4.so")

KV4_OK, KV4_ERR_INVALID_ARG, KV4_ERR_UNSUPPORTED, KV4_ERR_CUDA, KV4_ERR_DEVICE_BOUNDS = range(5)
KV4_DEVERR_PAGE, KV4_DEVERR_CONTEXT, KV4_DEVERR_SLOT, KV4_DEVERR_TIMEOUT = 1, 2, 4, 8
# kernel choices and test controls of kv4_decode_attention_select (include/kv4.h)
(KV4_KERNEL_AUTO, KV4_KERNEL_WARP_MMA, KV4_KERNEL_EXTEND, KV4_KERNEL_LATENT, KV4_KERNEL_GENERAL,
 KV4_KERNEL_TCGEN05, KV4_KERNEL_LATENT_TC, KV4_KERNEL_BALANCED) = range(8)
KV4_DIAG_EXPIRE_FIRST_WAIT = 1
KV4_MAX_Q_PER_SEQ = 4096  # include/kv4.h
PAGE_SIZE = 16

EXPORTS = ("kv4_status_string", "kv4_cache_bytes", "kv4_append_quantize", "kv4_decode_auto_splits",
           "kv4_decode_workspace_bytes", "kv4_decode_attention", "kv4_decode_partials", "kv4_split_combine",
           "fp8_cache_bytes", "fp8_append_quantize", "fp8_decode_attention",
           "kv4_decode_attention_noalloc", "kv4_decode_attention_select", "kv4_decode_partials_prefix",
           "kv4_decode_kernel_choice")


class Kv4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {lib().kv4_status_string(status).decode()} (status {status})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing; build it with `python -m bit_kv_cache_rotate_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    L.kv4_status_string.argtypes = [i32]
    L.kv4_status_string.restype = ctypes.c_char_p
    L.kv4_cache_bytes.argtypes = [i32, i32, i32, i32]
    L.kv4_cache_bytes.restype = sz
    L.fp8_cache_bytes.argtypes = [i32, i32, i32, i32]
    L.fp8_cache_bytes.restype = sz
    L.kv4_append_quantize.argtypes = [P, P, i32, i32, i32, P, P, P, i32, i32, P, P]
    L.kv4_append_quantize.restype = i32
    L.fp8_append_quantize.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, i32, i32, P, P]
    L.fp8_append_quantize.restype = i32
    L.kv4_decode_auto_splits.argtypes = [i32] * 7
    L.kv4_decode_auto_splits.restype = i32
    L.kv4_decode_kernel_choice.argtypes = [i32] * 7
    L.kv4_decode_kernel_choice.restype = i32
    L.kv4_decode_workspace_bytes.argtypes = [i32] * 5
    L.kv4_decode_workspace_bytes.restype = sz
    L.kv4_decode_attention.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                       P, sz, P, P, P]
    L.kv4_decode_attention.restype = i32
    L.kv4_decode_partials.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                      P, sz, P, P]
    L.kv4_decode_partials.restype = i32
    L.kv4_decode_partials_prefix.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                             P, sz, P, P]
    L.kv4_decode_partials_prefix.restype = i32
    L.fp8_decode_attention.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                       i32, P, sz, P, P, P]
    L.fp8_decode_attention.restype = i32
    L.kv4_split_combine.argtypes = [P, P, i32, i32, i32, i32, i32, P, P]
    L.kv4_split_combine.restype = i32
    L.kv4_decode_attention_noalloc.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                               i32, P, P, P]
    L.kv4_decode_attention_noalloc.restype = i32
    L.kv4_decode_attention_select.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                              P, sz, P, P, i32, i32, P]
    L.kv4_decode_attention_select.restype = i32
    return L


_lib_handle: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    """The loaded libkv4.so (loaded on first use; ImportError if it was never built)."""
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _load()
    return _lib_handle


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != KV4_OK:
        raise Kv4Error(fn, status)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ---------------------------------------------------------------- sizes
def kv4_cache_bytes(num_pages: int, num_kv_heads: int, page_size: int, head_dim: int) -> int:
    return int(lib().kv4_cache_bytes(num_pages, num_kv_heads, page_size, head_dim))


def fp8_cache_bytes(num_pages: int, num_kv_heads: int, page_size: int, head_dim: int) -> int:
    return int(lib().fp8_cache_bytes(num_pages, num_kv_heads, page_size, head_dim))


def kv4_decode_kernel_choice(batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, num_splits, latent=False) -> int:
    """The KV4_KERNEL_* id kv4_decode_attention runs for this shape (-1: invalid shape)."""
    return int(lib().kv4_decode_kernel_choice(batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, num_splits,
                                              1 if latent else 0))


def kv4_decode_auto_splits(batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, page_size,
                           max_pages_per_seq) -> int:
    return int(lib().kv4_decode_auto_splits(batch, q_per_seq, num_q_heads, num_kv_heads, head_dim,
                                           page_size, max_pages_per_seq))


def kv4_decode_workspace_bytes(batch, q_per_seq, num_q_heads, head_dim, num_splits) -> int:
    return int(lib().kv4_decode_workspace_bytes(batch, q_per_seq, num_q_heads, head_dim, num_splits))


def empty_cache(num_pages: int, num_kv_heads: int, head_dim: int, fp8: bool = False,
                device="cuda") -> torch.Tensor:
    n = (fp8_cache_bytes if fp8 else kv4_cache_bytes)(num_pages, num_kv_heads, PAGE_SIZE, head_dim)
    return torch.empty(n, dtype=torch.uint8, device=device)


def workspace(batch, q_per_seq, num_q_heads, head_dim, num_splits, device="cuda") -> torch.Tensor:
    n = kv4_decode_workspace_bytes(batch, q_per_seq, num_q_heads, head_dim, num_splits)
    return torch.empty(n, dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- 4-bit path
def kv4_append_quantize(k: torch.Tensor, v: torch.Tensor | None, slot_mapping: torch.Tensor,
                        k_cache: torch.Tensor, v_cache: torch.Tensor | None, num_pages: int,
                        page_size: int = PAGE_SIZE, dev_error: torch.Tensor | None = None,
                        stream=None) -> None:
    """k, v: bf16 [num_tokens, num_kv_heads, head_dim] (v None: latent cache)."""
    _dev(k, "k", torch.bfloat16)
    if v is not None:
        _dev(v, "v", torch.bfloat16)
    _dev(slot_mapping, "slot_mapping", torch.int32)
    n, hkv, d = k.shape
    st = lib().kv4_append_quantize(_ptr(k), _ptr(v), n, hkv, d, _ptr(slot_mapping), _ptr(k_cache),
                                  _ptr(v_cache), num_pages, page_size, _ptr(dev_error), _stream(stream))
    _check("kv4_append_quantize", st)


def kv4_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor | None,
                         block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int,
                         num_pages: int, softmax_scale: float, num_splits: int = 0,
                         workspace_buf: torch.Tensor | None = None, out: torch.Tensor | None = None,
                         dev_error: torch.Tensor | None = None, page_size: int = PAGE_SIZE,
                         stream=None) -> torch.Tensor:
    """q: bf16 [B, T, Hq, D] -> fp32 [B, T, Hq, D].  v_cache None: latent cache."""
    _dev(q, "q", torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    B, T, Hq, D = q.shape
    max_pages = block_tables.shape[1]
    S = num_splits or kv4_decode_auto_splits(B, T, Hq, num_kv_heads, D, page_size, max_pages)
    if workspace_buf is None:
        workspace_buf = workspace(B, T, Hq, D, S, device=q.device)
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.float32, device=q.device)
    st = lib().kv4_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), B, T, Hq, num_kv_heads, D, page_size, max_pages,
                                   num_pages, float(softmax_scale), S, _ptr(workspace_buf),
                                   workspace_buf.numel(), _ptr(out), _ptr(dev_error), _stream(stream))
    _check("kv4_decode_attention", st)
    return out


def kv4_decode_attention_select(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor | None,
                                block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int,
                                num_pages: int, softmax_scale: float, kernel: int, diag_flags: int = 0,
                                num_splits: int = 0, workspace_buf: torch.Tensor | None = None,
                                out: torch.Tensor | None = None, dev_error: torch.Tensor | None = None,
                                page_size: int = PAGE_SIZE, stream=None) -> torch.Tensor:
    """kv4_decode_attention with an explicit split kernel (KV4_KERNEL_*) and
    test controls (KV4_DIAG_*), for tests and measurements."""
    _dev(q, "q", torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    B, T, Hq, D = q.shape
    max_pages = block_tables.shape[1]
    S = num_splits or kv4_decode_auto_splits(B, T, Hq, num_kv_heads, D, page_size, max_pages)
    if workspace_buf is None:
        workspace_buf = workspace(B, T, Hq, D, S, device=q.device)
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.float32, device=q.device)
    st = lib().kv4_decode_attention_select(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                          _ptr(context_lens), B, T, Hq, num_kv_heads, D, page_size, max_pages,
                                          num_pages, float(softmax_scale), S, _ptr(workspace_buf),
                                          workspace_buf.numel(), _ptr(out), _ptr(dev_error), int(kernel),
                                          int(diag_flags), _stream(stream))
    _check("kv4_decode_attention_select", st)
    return out


def kv4_decode_partials(q, k_cache, v_cache, block_tables, context_lens, num_kv_heads: int,
                        num_pages: int, softmax_scale: float, num_splits: int, workspace_buf,
                        dev_error=None, page_size: int = PAGE_SIZE, stream=None) -> None:
    """Split stage only: partial outputs and log-sum-exps into workspace_buf."""
    B, T, Hq, D = q.shape
    st = lib().kv4_decode_partials(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), B, T, Hq, num_kv_heads, D, page_size,
                                   block_tables.shape[1], num_pages, float(softmax_scale), num_splits,
                                   _ptr(workspace_buf), workspace_buf.numel(), _ptr(dev_error),
                                   _stream(stream))
    _check("kv4_decode_partials", st)


def kv4_decode_partials_prefix(q, k_cache, v_cache, block_tables, context_lens, num_kv_heads: int,
                               num_pages: int, softmax_scale: float, num_splits: int, workspace_buf,
                               dev_error=None, page_size: int = PAGE_SIZE, stream=None) -> None:
    """Split stage over a leading share of each sequence (every cached token
    precedes the queries and is visible to all of them): the non-final shares
    of a sequence split across devices (see seqsplit)."""
    B, T, Hq, D = q.shape
    st = lib().kv4_decode_partials_prefix(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                          _ptr(context_lens), B, T, Hq, num_kv_heads, D, page_size,
                                          block_tables.shape[1], num_pages, float(softmax_scale), num_splits,
                                          _ptr(workspace_buf), workspace_buf.numel(), _ptr(dev_error),
                                          _stream(stream))
    _check("kv4_decode_partials_prefix", st)


def split_views(workspace_buf, B, T, Hq, D, S):
    """(partial_o [B,T,Hq,S,D], partial_lse [B,T,Hq,S]) fp32 views of a decode workspace."""
    n_o = B * T * Hq * S * D
    off = ((n_o * 4 + 255) // 256) * 256
    po = workspace_buf[:n_o * 4].view(torch.float32).view(B, T, Hq, S, D)
    pl = workspace_buf[off:off + B * T * Hq * S * 4].view(torch.float32).view(B, T, Hq, S)
    return po, pl


def kv4_split_combine(partial_o: torch.Tensor, partial_lse: torch.Tensor,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """partial_o: fp32 [B, T, Hq, S, D], partial_lse: fp32 [B, T, Hq, S] -> fp32 [B, T, Hq, D]."""
    _dev(partial_o, "partial_o", torch.float32)
    _dev(partial_lse, "partial_lse", torch.float32)
    B, T, Hq, S, D = partial_o.shape
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.float32, device=partial_o.device)
    st = lib().kv4_split_combine(_ptr(partial_o), _ptr(partial_lse), B, T, Hq, D, S, _ptr(out),
                                _stream(stream))
    _check("kv4_split_combine", st)
    return out


def kv4_decode_attention_noalloc(q, k_cache, v_cache, block_tables, context_lens, num_kv_heads: int,
                                 num_pages: int, softmax_scale: float, num_splits: int = 0,
                                 out: torch.Tensor | None = None, dev_error=None,
                                 page_size: int = PAGE_SIZE, stream=None) -> torch.Tensor:
    """kv4_decode_attention without a workspace: for callers that cannot allocate
    device memory.  The split partials go to a fixed array inside libkv4 shared
    by all calls, so calls whose GPU work overlaps must be ordered."""
    _dev(q, "q", torch.bfloat16)
    B, T, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.float32, device=q.device)
    st = lib().kv4_decode_attention_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                            _ptr(context_lens), B, T, Hq, num_kv_heads, D, page_size,
                                            block_tables.shape[1], num_pages, float(softmax_scale), num_splits,
                                            _ptr(out), _ptr(dev_error), _stream(stream))
    _check("kv4_decode_attention_noalloc", st)
    return out


# ---------------------------------------------------------------- FP8 comparator
def fp8_append_quantize(k, v, slot_mapping, k_inv_scale, v_inv_scale, k_cache, v_cache, num_pages,
                        page_size: int = PAGE_SIZE, dev_error=None, stream=None) -> None:
    _dev(k, "k", torch.bfloat16)
    _dev(v, "v", torch.bfloat16)
    _dev(slot_mapping, "slot_mapping", torch.int32)
    _dev(k_inv_scale, "k_inv_scale", torch.float32)
    _dev(v_inv_scale, "v_inv_scale", torch.float32)
    n, hkv, d = k.shape
    st = lib().fp8_append_quantize(_ptr(k), _ptr(v), n, hkv, d, _ptr(slot_mapping), _ptr(k_inv_scale),
                                  _ptr(v_inv_scale), _ptr(k_cache), _ptr(v_cache), num_pages, page_size,
                                  _ptr(dev_error), _stream(stream))
    _check("fp8_append_quantize", st)


def fp8_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                         num_kv_heads, num_pages, softmax_scale, num_splits=0, workspace_buf=None,
                         out=None, dev_error=None, page_size: int = PAGE_SIZE, stream=None):
    _dev(q, "q", torch.bfloat16)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    B, T, Hq, D = q.shape
    max_pages = block_tables.shape[1]
    S = num_splits or kv4_decode_auto_splits(B, T, Hq, num_kv_heads, D, page_size, max_pages)
    if workspace_buf is None:
        workspace_buf = workspace(B, T, Hq, D, S, device=q.device)
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.float32, device=q.device)
    st = lib().fp8_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(block_tables), _ptr(context_lens), B, T, Hq, num_kv_heads, D,
                                   page_size, max_pages, num_pages, float(softmax_scale), S,
                                   _ptr(workspace_buf), workspace_buf.numel(), _ptr(out), _ptr(dev_error),
                                   _stream(stream))
    _check("fp8_decode_attention", st)
    return out
