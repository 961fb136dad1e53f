"""GPU parity of extend steps: many new query positions per sequence (a chunk
of prompt tokens) over the cached prefix, causal among themselves, through
the same C ABI call as decode.  The 4-bit kernel tiles the positions over
CTAs; each CTA is checked through the whole output against the oracle's fp64
attention (max abs error 2e-3), across tile boundaries, ragged contexts,
split counts, GQA groups and the pure-prefill case (context == chunk)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL, all_tokens, gpu_caches, gpu_tables, oracle_caches

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

BASE = W.CONFIGS["extend_b4_ctx32k_t512"]


def _cfg(T, ctx, batch=2, Hq=64, Hkv=8, seed=None):
    c = W.scaled(BASE, batch=batch, ctx=ctx)
    return dataclasses.replace(c, q_per_seq=T, num_q_heads=Hq, num_kv_heads=Hkv,
                               seed=c.seed if seed is None else seed)


def _run(cfg, num_splits=0, fp8=False, kernel=0):
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    q = W.queries(cfg)
    tab, lens = gpu_tables(lay)
    otab = np.where(lay.block_tables < 0, 0, lay.block_tables)
    if not fp8:
        okc, ovc = oracle_caches(cfg, lay, k, v, slots)
        gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
        out = kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                              cfg.softmax_scale, kernel, num_splits=num_splits)
        torch.cuda.synchronize()
        ref = oracle.decode_attention(q, okc, ovc, otab, lay.context_lens, cfg.num_kv_heads, cfg.page_size,
                                      lay.num_pages, cfg.softmax_scale)
    else:
        ks, vs, kinv, vinv = W.fp8_head_scales(k, v)
        bb = cfg.page_size * cfg.head_dim
        okc = np.zeros(lay.num_pages * cfg.num_kv_heads * bb, np.uint8)
        ovc = np.zeros_like(okc)
        assert oracle.fp8_append(k, v, slots, kinv, vinv, okc, ovc, lay.num_pages, cfg.page_size) == 0
        n = kv4.fp8_cache_bytes(lay.num_pages, cfg.num_kv_heads, cfg.page_size, cfg.head_dim)
        gkc = torch.zeros(n, dtype=torch.uint8, device="cuda")
        gvc = torch.zeros(n, dtype=torch.uint8, device="cuda")
        t = lambda a: torch.from_numpy(a).cuda()
        kv4.fp8_append_quantize(k.cuda(), v.cuda(), t(slots), t(kinv), t(vinv), gkc, gvc, lay.num_pages)
        out = kv4.fp8_decode_attention(q.cuda(), gkc, gvc, t(ks), t(vs), tab, lens, cfg.num_kv_heads,
                                       lay.num_pages, cfg.softmax_scale, num_splits=num_splits)
        torch.cuda.synchronize()
        assert np.array_equal(gkc.cpu().numpy(), okc) and np.array_equal(gvc.cpu().numpy(), ovc)
        ref = oracle.fp8_decode_attention(q, okc, ovc, ks, vs, otab, lay.context_lens, cfg.num_kv_heads,
                                          cfg.page_size, lay.num_pages, cfg.softmax_scale)
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    return np.abs(got - ref).max()


@pytest.mark.parametrize("T,ctx", [(9, ("uniform", 200, 700)), (25, ("uniform", 300, 900)),
                                   (64, ("fixed", 1021)), (200, ("uniform", 400, 1200))])
def test_extend_parity(T, ctx):
    err = _run(_cfg(T, ctx))
    assert err <= TOL, f"max abs error {err:.3e}"


@pytest.mark.parametrize("T", [16, 100])
def test_prefill_chunk_is_whole_context(T):
    """No cached prefix: the chunk is the whole context (causal self-attention)."""
    err = _run(_cfg(T, ("fixed", T), batch=3))
    assert err <= TOL, f"max abs error {err:.3e}"


@pytest.mark.parametrize("Hq,Hkv,T", [(8, 2, 50), (8, 8, 70), (12, 4, 33), (40, 8, 11)])
def test_extend_other_groups(Hq, Hkv, T):
    """G = 4, 1, 3, 5: tiles of 6, 24, 8 and 4 positions (ragged last tiles)."""
    err = _run(_cfg(T, ("uniform", 100, 600), Hq=Hq, Hkv=Hkv))
    assert err <= TOL, f"max abs error {err:.3e}"


@pytest.mark.parametrize("S", [1, 2, 7])
def test_extend_split_counts(S):
    err = _run(_cfg(40, ("uniform", 500, 1500)), num_splits=S)
    assert err <= TOL, (S, err)


def test_extend_fp8_comparator():
    err = _run(_cfg(30, ("uniform", 300, 800)), fp8=True)
    assert err <= TOL, f"max abs error {err:.3e}"


@pytest.mark.parametrize("warp", [False, True])
def test_extend_both_kernels(warp):
    """G = 8 and 4 on the tcgen05 extend kernel (default) and on the warp-MMA
    kernel's position tiles (KV4_KERNEL_WARP_MMA)."""
    kernel = kv4.KV4_KERNEL_WARP_MMA if warp else kv4.KV4_KERNEL_AUTO
    for Hq, Hkv, T, ctx in [(64, 8, 48, ("uniform", 300, 1100)), (16, 4, 130, ("uniform", 200, 700))]:
        err = _run(_cfg(T, ctx, Hq=Hq, Hkv=Hkv), kernel=kernel)
        assert err <= TOL, (warp, Hq, Hkv, T, err)
