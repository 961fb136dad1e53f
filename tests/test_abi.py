"""The C-ABI library loads on a machine without a GPU, exports every entry
point that include/kv4.h declares, and validates arguments on the host
before launching anything (these calls return before touching the device)."""
import ctypes
import os
import re

import pytest

import bit_kv_cache_rotate_b300 as kv4
from bit_kv_cache_rotate_b300 import build as kbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kv4.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M))
                  - {"if", "extern"})


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kv4.lib()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("kv4_append_quantize", "kv4_decode_attention", "kv4_split_combine",
              "fp8_append_quantize", "fp8_decode_attention"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(kv4.EXPORTS) <= set(_declared())


def test_sizes(lib):
    assert kv4.kv4_cache_bytes(16384, 8, 16, 128) == 16384 * 8 * 1088
    assert kv4.kv4_cache_bytes(1, 1, 16, 512) == 16 * 256 + 16 * 16
    assert kv4.fp8_cache_bytes(10, 8, 16, 128) == 10 * 8 * 2048
    assert kv4.kv4_cache_bytes(-1, 1, 16, 128) == 0
    ws = kv4.kv4_decode_workspace_bytes(32, 1, 64, 128, 4)
    assert ws >= 32 * 64 * 4 * (128 + 1) * 4
    assert 1 <= kv4.kv4_decode_auto_splits(32, 1, 64, 8, 128, 16, 2048) <= 2048


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    # null pointers
    assert lib.kv4_append_quantize(None, None, 4, 8, 128, None, None, None, 10, 16, None, None) == \
        kv4.KV4_ERR_INVALID_ARG
    # unsupported head dim / page size
    assert lib.kv4_append_quantize(fake, fake, 4, 8, 96, fake, fake, fake, 10, 16, None, None) == \
        kv4.KV4_ERR_UNSUPPORTED
    assert lib.kv4_append_quantize(fake, fake, 4, 8, 128, fake, fake, fake, 10, 32, None, None) == \
        kv4.KV4_ERR_UNSUPPORTED
    # v without v_cache
    assert lib.kv4_append_quantize(fake, fake, 4, 8, 128, fake, fake, None, 10, 16, None, None) == \
        kv4.KV4_ERR_INVALID_ARG
    # misaligned cache pointer
    assert lib.kv4_append_quantize(fake, fake, 4, 8, 128, fake, P(4097), fake, 10, 16, None, None) == \
        kv4.KV4_ERR_INVALID_ARG
    # zero tokens is a no-op
    assert lib.kv4_append_quantize(None, None, 0, 8, 128, None, None, None, 10, 16, None, None) == kv4.KV4_OK
    # decode: Hq not a multiple of Hkv, T too large, workspace too small
    dec = lib.kv4_decode_attention
    args = lambda **kw: [kw.get("q", fake), fake, fake, fake, fake, kw.get("B", 2), kw.get("T", 1),
                         kw.get("Hq", 8), kw.get("Hkv", 2), kw.get("D", 128), 16, 4, 8, 0.1,
                         kw.get("S", 1), P(4096 * 256), kw.get("ws", 1 << 20), fake, None, None]
    assert dec(*args(Hq=7)) == kv4.KV4_ERR_INVALID_ARG
    assert dec(*args(T=kv4.KV4_MAX_Q_PER_SEQ + 1)) == kv4.KV4_ERR_UNSUPPORTED
    assert dec(*args(D=80)) == kv4.KV4_ERR_UNSUPPORTED
    assert dec(*args(ws=16)) == kv4.KV4_ERR_INVALID_ARG
    assert dec(*args(q=None)) == kv4.KV4_ERR_INVALID_ARG
    assert dec(*args(B=0)) == kv4.KV4_OK
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        a_bad = args()
        a_bad[13] = bad
        assert dec(*a_bad) == kv4.KV4_ERR_INVALID_ARG, bad
    assert lib.kv4_split_combine(None, None, 1, 1, 8, 128, 2, None, None) == kv4.KV4_ERR_INVALID_ARG
    assert lib.kv4_split_combine(fake, fake, 1, 1, 8, 100, 2, fake, None) == kv4.KV4_ERR_UNSUPPORTED


def test_status_strings(lib):
    for s in range(5):
        assert lib.kv4_status_string(s)


def test_more_host_validation(lib):
    """Each of these returns before any launch or CUDA call."""
    P = ctypes.c_void_p
    fake = P(4096)
    ws = P(4096 * 256)
    dec = lib.kv4_decode_attention

    def args(q=fake, B=2, T=1, Hq=8, Hkv=2, D=128, S=1, ws_ptr=ws, ws_bytes=1 << 24, out=fake):
        return [q, fake, fake, fake, fake, B, T, Hq, Hkv, D, 16, 4, 8, 0.1, S, ws_ptr, ws_bytes, out, None, None]

    assert dec(*args(S=-1)) == kv4.KV4_ERR_INVALID_ARG
    assert dec(*args(S=4097)) == kv4.KV4_ERR_INVALID_ARG
    assert dec(*args(q=P(4098))) == kv4.KV4_ERR_INVALID_ARG          # q not 16-byte aligned
    assert dec(*args(ws_ptr=P(4096 * 256 + 128))) == kv4.KV4_ERR_INVALID_ARG  # workspace not 256-byte aligned
    assert dec(*args(out=P(4100))) == kv4.KV4_ERR_INVALID_ARG        # out not 16-byte aligned
    assert dec(*args(out=None)) == kv4.KV4_ERR_INVALID_ARG
    assert dec(*args(Hkv=0)) == kv4.KV4_ERR_INVALID_ARG
    # the general kernel's row limits: 64 rows at head_dim 64, 16 for the 512-wide latent cache
    assert dec(*args(D=64, T=9, Hq=16, Hkv=2)) == kv4.KV4_ERR_UNSUPPORTED
    lat = args(D=512, T=2, Hq=16, Hkv=1)
    lat[2] = None  # latent cache: no separate V
    assert dec(*lat) == kv4.KV4_ERR_UNSUPPORTED
    # the split stage alone needs an explicit split count
    part = args()
    del part[17]  # kv4_decode_partials has no output argument
    part[14] = 0
    assert lib.kv4_decode_partials(*part) == kv4.KV4_ERR_INVALID_ARG
    # FP8 decode needs both per-head scales
    f8 = lib.fp8_decode_attention
    f8_args = lambda ks, vs: [fake, fake, fake, ks, vs, fake, fake, 2, 1, 8, 2, 128, 16, 4, 8, 0.1, 1, ws, 1 << 24,
                              fake, None, None]
    assert f8(*f8_args(None, fake)) == kv4.KV4_ERR_INVALID_ARG
    assert f8(*f8_args(fake, None)) == kv4.KV4_ERR_INVALID_ARG
    # FP8 append: misaligned bf16 input
    assert lib.fp8_append_quantize(P(4100), fake, 4, 8, 128, fake, fake, fake, fake, fake, 10, 16, None, None) == \
        kv4.KV4_ERR_INVALID_ARG


def test_noalloc_rejects_before_touching_the_device(lib):
    """An explicit split count whose partials exceed the fixed scratch, or a
    negative one, is refused before the scratch address is looked up."""
    P = ctypes.c_void_p
    fake = P(4096)
    na = lib.kv4_decode_attention_noalloc
    B, T, Hq, Hkv, D = 64, 1, 64, 8, 128
    need = kv4.kv4_decode_workspace_bytes(B, T, Hq, D, 64)
    assert need > (16 << 20)
    assert na(fake, fake, fake, fake, fake, B, T, Hq, Hkv, D, 16, 4, 8, 0.1, 64, fake, None, None) == \
        kv4.KV4_ERR_INVALID_ARG
    assert na(fake, fake, fake, fake, fake, B, T, Hq, Hkv, D, 16, 4, 8, 0.1, -1, fake, None, None) == \
        kv4.KV4_ERR_INVALID_ARG
    assert na(fake, fake, fake, fake, fake, 0, T, Hq, Hkv, D, 16, 4, 8, 0.1, 0, fake, None, None) == kv4.KV4_OK
    # batch 0 is validated like kv4_decode_attention: a bad shape is still refused
    assert na(fake, fake, fake, fake, fake, 0, T, Hq, Hkv, 96, 16, 4, 8, 0.1, 0, fake, None, None) == \
        kv4.KV4_ERR_UNSUPPORTED
    assert na(fake, fake, fake, fake, fake, 0, T, 63, Hkv, D, 16, 4, 8, 0.1, 0, fake, None, None) == \
        kv4.KV4_ERR_INVALID_ARG


def test_kernel_choice_is_validated_before_launch(lib):
    """kv4_decode_attention_select: an unknown kernel id is an invalid argument,
    a kernel that does not serve the shape is unsupported; both return before
    any launch."""
    P = ctypes.c_void_p
    fake = P(4096)
    ws = P(4096 * 256)
    sel = lib.kv4_decode_attention_select

    def args(kernel, T=1, Hq=8, Hkv=2, D=128, v=fake, diag=0):
        return [fake, fake, v, fake, fake, 2, T, Hq, Hkv, D, 16, 4, 8, 0.1, 1, ws, 1 << 24, fake, None,
                kernel, diag, None]

    assert sel(*args(99)) == kv4.KV4_ERR_INVALID_ARG
    assert sel(*args(-1)) == kv4.KV4_ERR_INVALID_ARG
    assert sel(*args(kv4.KV4_KERNEL_LATENT)) == kv4.KV4_ERR_UNSUPPORTED        # not a latent cache
    assert sel(*args(kv4.KV4_KERNEL_LATENT_TC)) == kv4.KV4_ERR_UNSUPPORTED     # not a latent cache
    assert sel(*args(8)) == kv4.KV4_ERR_INVALID_ARG
    assert sel(*args(kv4.KV4_KERNEL_EXTEND)) == kv4.KV4_ERR_UNSUPPORTED        # 4 rows: not an extend tile
    assert sel(*args(kv4.KV4_KERNEL_WARP_MMA, D=64)) == kv4.KV4_ERR_UNSUPPORTED  # head_dim 64
    assert sel(*args(kv4.KV4_KERNEL_GENERAL, T=40, Hq=16)) == kv4.KV4_ERR_UNSUPPORTED  # 320 rows
    # the env switches of earlier versions are gone: nothing in the library reads the environment
    import subprocess
    out = subprocess.run(["nm", "-D", "--undefined-only", kv4.LIB_PATH], capture_output=True, text=True).stdout
    assert "getenv" not in out


def test_kernel_choice_query(lib):
    assert kv4.kv4_decode_kernel_choice(0, 1, 64, 8, 128, 4) == -1          # no sequences
    assert kv4.kv4_decode_kernel_choice(4, 1, 60, 8, 128, 4) == -1          # heads not a multiple
    assert kv4.kv4_decode_kernel_choice(4, 1, 64, 8, 96, 4) == -1           # unsupported head_dim
    assert kv4.kv4_decode_kernel_choice(8, 1, 16, 1, 512, 18, latent=True) == kv4.KV4_KERNEL_LATENT_TC
    assert kv4.kv4_decode_kernel_choice(4, 512, 64, 8, 128, 1) == kv4.KV4_KERNEL_EXTEND
    assert kv4.kv4_decode_kernel_choice(32, 3, 64, 8, 128, 4) == kv4.KV4_KERNEL_WARP_MMA   # 24 rows
    assert kv4.kv4_decode_kernel_choice(4, 1, 80, 8, 128, 4) == kv4.KV4_KERNEL_GENERAL     # G = 10
    # up to 8 rows: the flat mode where the slots fill a wave on this device, else the split form
    assert kv4.kv4_decode_kernel_choice(32, 1, 64, 8, 128, 4) in (kv4.KV4_KERNEL_BALANCED, kv4.KV4_KERNEL_WARP_MMA)
    assert kv4.kv4_decode_kernel_choice(32, 1, 64, 8, 128, 1) == kv4.KV4_KERNEL_WARP_MMA
