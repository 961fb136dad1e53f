"""Attention ignores cache slots that no token has written.

A serving engine hands the library cache memory it never cleared, and the
last page of a sequence is usually only partly filled, so the slots past a
sequence's context hold whatever bytes were there before.  Every decode
kernel must give the oracle's result (computed over zero-initialised
caches, reading only tokens below the context length) when those slots
hold hostile bytes: 0xFF is a UE8M0 scale of 2^128 and an E2M1 code of -6
in the 4-bit cache, and a NaN in the E4M3 cache.  Each case has ragged
contexts so that partial pages, partial chunks and splits ending mid-page
all occur, and routes through one kernel: the warp-MMA decode (T = 1) and
verify (T = 3) kernels, the opt-in tcgen05 decode kernel, the latent (MLA)
kernel, both extend kernels, the general CUDA-core kernel (G = 10, and
head_dim 64), and the FP8 comparator's kernels."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL, all_tokens, gpu_caches, gpu_tables, oracle_caches

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

_B32 = W.CONFIGS["b32_ctx8k"]
_EXT = W.CONFIGS["extend_b4_ctx32k_t512"]

# name -> (config, kernel choice)
CASES = {
    "decode": (W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)), 0),
    "decode_general": (W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)), 4),
    "decode_tcgen05": (W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)), 5),
    "decode_balanced": (W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)), 7),
    "verify": (W.scaled(W.CONFIGS["verify_agentic"], batch=4, ctx=("uniform", 300, 1500)), 0),
    "mla": (W.scaled(W.CONFIGS["mla_b8_ctx96k"], batch=3, ctx=("uniform", 17, 900)), 0),
    "mla_warp": (W.scaled(W.CONFIGS["mla_b8_ctx96k"], batch=3, ctx=("uniform", 17, 900)), 3),
    "extend_tcgen05": (dataclasses.replace(W.scaled(_EXT, batch=2, ctx=("uniform", 100, 700)), q_per_seq=40), 0),
    "extend_warp": (dataclasses.replace(W.scaled(_EXT, batch=2, ctx=("uniform", 100, 700)), q_per_seq=40), 1),
    "general_g10": (dataclasses.replace(W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)), num_q_heads=80), 0),
    "general_d64": (dataclasses.replace(W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)), head_dim=64), 0),
}


@pytest.mark.parametrize("fill", [0xFF, 0xC3])
@pytest.mark.parametrize("name", list(CASES))
def test_4bit_attention_ignores_unwritten_slots(name, fill):
    cfg, kernel = CASES[name]
    lay = W.make_layout(cfg)
    assert (lay.context_lens % cfg.page_size != 0).any(), "the case needs partly filled pages"
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots, fill=fill)
    q = W.queries(cfg)
    tab, lens = gpu_tables(lay)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for S in ((2, 3) if kernel == kv4.KV4_KERNEL_BALANCED else (1, 3)):
        out = kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                              cfg.softmax_scale, kernel, num_splits=S, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), (S, "non-finite output")
        ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                      lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                      cfg.softmax_scale, latent=cfg.latent)
        e = np.abs(got - ref).max()
        assert e <= TOL, (S, f"max abs error {e:.3e}")


FP8_CASES = {
    "decode": W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)),
    "verify": W.scaled(W.CONFIGS["verify_agentic"], batch=3, ctx=("uniform", 300, 900)),
    "general_g10": dataclasses.replace(W.scaled(_B32, batch=3, ctx=("uniform", 17, 700)), num_q_heads=80),
}


@pytest.mark.parametrize("fill", [0xFF, 0x7E])
@pytest.mark.parametrize("name", list(FP8_CASES))
def test_fp8_attention_ignores_unwritten_slots(name, fill):
    """0xFF is an E4M3 NaN, 0x7E the largest finite value (448)."""
    cfg = FP8_CASES[name]
    lay = W.make_layout(cfg)
    assert (lay.context_lens % cfg.page_size != 0).any()
    k, v, slots = all_tokens(cfg, lay)
    ks, vs, kinv, vinv = W.fp8_head_scales(k, v)
    bb = cfg.page_size * cfg.head_dim
    okc = np.zeros(lay.num_pages * cfg.num_kv_heads * bb, np.uint8)
    ovc = np.zeros_like(okc)
    assert oracle.fp8_append(k, v, slots, kinv, vinv, okc, ovc, lay.num_pages, cfg.page_size) == 0
    n = kv4.fp8_cache_bytes(lay.num_pages, cfg.num_kv_heads, cfg.page_size, cfg.head_dim)
    gkc = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
    gvc = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
    t = lambda a: torch.from_numpy(a).cuda()
    kv4.fp8_append_quantize(k.cuda(), v.cuda(), t(slots), t(kinv), t(vinv), gkc, gvc, lay.num_pages)
    q = W.queries(cfg)
    tab, lens = gpu_tables(lay)
    ref = oracle.fp8_decode_attention(q, okc, ovc, ks, vs, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                      lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                      cfg.softmax_scale)
    for S in (1, 3):
        out = kv4.fp8_decode_attention(q.cuda(), gkc, gvc, t(ks), t(vs), tab, lens, cfg.num_kv_heads,
                                       lay.num_pages, cfg.softmax_scale, num_splits=S)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), (S, "non-finite output")
        e = np.abs(got - ref).max()
        assert e <= TOL, (S, f"max abs error {e:.3e}")
