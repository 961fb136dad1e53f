"""CPU oracle for 4-bit rotated KV-cache decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library in ``bit_kv_cache_rotate_b300``; it is compiled
from ``kv4_oracle.c`` with the host C compiler.

What it computes follows the "UltraQuant on AMD Instinct" blog page:
  * section "What is UltraQuant": Walsh-Hadamard rotation, FP4 (E2M1) codes
    with one power-of-two scale per 32 channels, 17 bytes per 32 values;
  * section "Why UltraQuant beats 8-bit KV": UE8M0 scales; decoding re-reads
    the whole cache every token;
  * section "Throughput-latency trade-off": 3-position MTP verify rows share
    one paged cache (causal among the new positions).
The readings taken where the page is silent (rotation arithmetic, scale
rule, rounding, block layout, FP8 comparator) are listed at the top of the C
source and in the design notes.  Every function is pinned by ``tests/``
against facts the page and the mathematics fix.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

OK, BAD_ARG, INEXACT = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.orc_hadamard_pm1.argtypes = [i32, P]
        L.orc_rotate_bf16.argtypes = [P, i32, P]
        L.orc_rotate_f64.argtypes = [P, i32, P]
        L.orc_group_exponent.argtypes = [P, i32]
        L.orc_e2m1_encode.argtypes = [f64]
        L.orc_e2m1_decode.argtypes = [i32]
        L.orc_e2m1_decode.restype = f64
        L.orc_quantize_vector.argtypes = [P, i32, P, P]
        L.orc_quantize_rotated.argtypes = [P, i32, P, P]
        L.orc_quantize_vectors.argtypes = [P, i64, i32, P, P]
        L.orc_quantize_vectors.restype = i64
        L.orc_block_bytes.argtypes = [i32, i32]
        L.orc_block_bytes.restype = ctypes.c_size_t
        L.orc_pack_k_token.argtypes = [P, i32, i32, i32, P, P]
        L.orc_pack_v_token.argtypes = [P, i32, i32, i32, P, P]
        L.orc_unpack_k_token.argtypes = [P, i32, i32, i32, P]
        L.orc_unpack_v_token.argtypes = [P, i32, i32, i32, P]
        L.orc_append_quantize.argtypes = [P, P, i32, i32, i32, P, P, P, i32, i32]
        L.orc_attend_row.argtypes = [P, P, P, i32, i32, f64, P]
        L.orc_attend_row.restype = f64
        L.orc_decode_attention.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                           f64, i32, P, i32, P]
        L.orc_e4m3_decode.argtypes = [i32]
        L.orc_e4m3_decode.restype = f64
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode_array.argtypes = [P, i64, P]
        L.orc_e4m3_encode_array.argtypes = [P, i64, P]
        L.orc_e4m3_decode_array.argtypes = [P, i64, P]
        L.orc_fp8_append.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, i32, i32]
        L.orc_set_threads.argtypes = [i32]
        L.orc_max_threads.restype = i32
        L.orc_fp8_decode_attention.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                               i32, i32, f64, P, i32, P]
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ---------------------------------------------------------------- rotation
def hadamard_pm1(D: int) -> np.ndarray:
    H = np.zeros((D, D), dtype=np.int8)
    assert lib().orc_hadamard_pm1(D, _p(H)) == OK
    return H


def rotate_bf16(x) -> tuple[np.ndarray, int]:
    x = _u16(x)
    D = x.shape[-1]
    y = np.zeros(D, dtype=np.float32)
    st = lib().orc_rotate_bf16(_p(x), D, _p(y))
    return y, st


def rotate_f64(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    lib().orc_rotate_f64(_p(v), v.shape[-1], _p(out))
    return out


# ---------------------------------------------------------------- FP4 codes
def group_exponent(y: np.ndarray) -> int:
    y = np.ascontiguousarray(y, dtype=np.float32)
    return lib().orc_group_exponent(_p(y), y.size)


def e2m1_encode(z) -> np.ndarray:
    z = np.ascontiguousarray(np.atleast_1d(np.asarray(z, dtype=np.float64)))
    out = np.zeros(z.shape, dtype=np.uint8)
    lib().orc_e2m1_encode_array(_p(z), z.size, _p(out))
    return out


def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def quantize_rotated(y: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """y: fp32 [D] already rotated -> (codes [D] uint8, exponents [D/32] int32)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    D = y.shape[-1]
    codes = np.zeros(D, dtype=np.uint8)
    expo = np.zeros(D // 32, dtype=np.int32)
    lib().orc_quantize_rotated(_p(y), D, _p(codes), _p(expo))
    return codes, expo


def quantize_vectors(x) -> tuple[np.ndarray, np.ndarray, int]:
    """x: [..., D] bf16 -> (codes [..., D] uint8, exponents [..., D/32] int32, n_inexact)."""
    x = _u16(x)
    D = x.shape[-1]
    n = x.size // D
    codes = np.zeros(x.shape, dtype=np.uint8)
    expo = np.zeros(x.shape[:-1] + (D // 32,), dtype=np.int32)
    bad = lib().orc_quantize_vectors(_p(x), n, D, _p(codes), _p(expo))
    return codes, expo, int(bad)


def block_bytes(page_size: int, D: int) -> int:
    return int(lib().orc_block_bytes(page_size, D))


def unpack_k_token(block: np.ndarray, page_size: int, D: int, off: int) -> np.ndarray:
    out = np.zeros(D, dtype=np.float64)
    lib().orc_unpack_k_token(_p(np.ascontiguousarray(block)), page_size, D, off, _p(out))
    return out


def unpack_v_token(block: np.ndarray, page_size: int, D: int, off: int) -> np.ndarray:
    out = np.zeros(D, dtype=np.float64)
    lib().orc_unpack_v_token(_p(np.ascontiguousarray(block)), page_size, D, off, _p(out))
    return out


# ---------------------------------------------------------------- append + attention
def append_quantize(k, v, slot_mapping: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray | None,
                    num_pages: int, page_size: int) -> int:
    """k, v: bf16 [n, Hkv, D] (v None for the latent cache); caches: uint8, modified in place."""
    k = _u16(k)
    v = None if v is None else _u16(v)
    n, Hkv, D = k.shape
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    return lib().orc_append_quantize(_p(k), _p(v), n, Hkv, D, _p(slot_mapping), _p(k_cache),
                                     _p(v_cache), num_pages, page_size)


def attend_row(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> tuple[np.ndarray, float]:
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    out = np.zeros(q.shape[-1], dtype=np.float64)
    lse = lib().orc_attend_row(_p(q), _p(K), _p(V), K.shape[0], q.shape[-1], scale, _p(out))
    return out, lse


def decode_attention(q, k_cache: np.ndarray, v_cache: np.ndarray | None, block_tables: np.ndarray,
                     context_lens: np.ndarray, num_kv_heads: int, page_size: int, num_pages: int,
                     scale: float, latent: bool = False, seqs=None) -> np.ndarray:
    """q: bf16 [B, T, Hq, D] -> fp64 [B, T, Hq, D] (rows of unselected sequences stay 0)."""
    q = _u16(q)
    B, T, Hq, D = q.shape
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    sel = None if seqs is None else np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    st = lib().orc_decode_attention(_p(q), _p(k_cache), _p(k_cache if latent else v_cache),
                                    _p(block_tables), _p(context_lens), B, T, Hq, num_kv_heads, D,
                                    page_size, block_tables.shape[1], num_pages, scale, int(latent),
                                    _p(sel), 0 if sel is None else sel.size, _p(out))
    assert st == OK, f"oracle decode_attention failed ({st})"
    return out


# ---------------------------------------------------------------- FP8 comparator
def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(np.atleast_1d(np.asarray(x, dtype=np.float32)))
    out = np.zeros(x.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_decode(b) -> np.ndarray:
    b = np.ascontiguousarray(np.atleast_1d(np.asarray(b, dtype=np.uint8)))
    out = np.zeros(b.shape, dtype=np.float64)
    lib().orc_e4m3_decode_array(_p(b), b.size, _p(out))
    return out


def fp8_append(k, v, slot_mapping, k_inv_scale, v_inv_scale, k_cache, v_cache, num_pages, page_size) -> int:
    k = _u16(k)
    v = _u16(v)
    n, Hkv, D = k.shape
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    kis = np.ascontiguousarray(k_inv_scale, dtype=np.float32)
    vis = np.ascontiguousarray(v_inv_scale, dtype=np.float32)
    return lib().orc_fp8_append(_p(k), _p(v), n, Hkv, D, _p(slot_mapping), _p(kis), _p(vis),
                                _p(k_cache), _p(v_cache), num_pages, page_size)


def fp8_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                         num_kv_heads, page_size, num_pages, scale, seqs=None) -> np.ndarray:
    q = _u16(q)
    B, T, Hq, D = q.shape
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    sel = None if seqs is None else np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    st = lib().orc_fp8_decode_attention(_p(q), _p(k_cache), _p(v_cache), _p(ks), _p(vs),
                                        _p(block_tables), _p(context_lens), B, T, Hq, num_kv_heads,
                                        D, page_size, block_tables.shape[1], num_pages, scale,
                                        _p(sel), 0 if sel is None else sel.size, _p(out))
    assert st == OK, f"oracle fp8_decode_attention failed ({st})"
    return out


# ---------------------------------------------------------------- threads (timing only)
def set_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP loops; no result depends on it."""
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())
