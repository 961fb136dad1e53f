"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Packed codes and scales must match bit-exactly; attention outputs must be
within max abs error 2e-3 of the oracle's fp64 attention over the same
dequantised cache.  Sizes are small enough for the oracle yet span several
pages, several splits and a ragged last page.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL, all_tokens, gpu_caches, gpu_tables, oracle_caches

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")


SMALL = {
    "tiny": W.CONFIGS["tiny"],
    "b32_small": W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("fixed", 1000)),
    "mla_small": W.scaled(W.CONFIGS["mla_b8_ctx96k"], batch=2, ctx=("fixed", 777)),
    "verify_small": W.scaled(W.CONFIGS["verify_agentic"], batch=4, ctx=("uniform", 300, 1500)),
    "verify6_small": W.scaled(W.CONFIGS["verify6_agentic"], batch=4, ctx=("uniform", 300, 1500)),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_append_codes_bit_exact(name):
    cfg = SMALL[name]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    g = gkc.cpu().numpy()
    diff = np.flatnonzero(g != okc)
    assert diff.size == 0, f"K cache differs at {diff[:10]} ({diff.size} bytes)"
    if ovc is not None:
        g = gvc.cpu().numpy()
        diff = np.flatnonzero(g != ovc)
        assert diff.size == 0, f"V cache differs at {diff[:10]} ({diff.size} bytes)"


def test_append_over_garbage_and_concurrent_neighbours():
    """Cache memory starts as garbage (0xFF); tokens sharing V bytes are
    appended in one launch; every written page must equal the oracle's."""
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=2, ctx=("fixed", 64))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots, fill=0xFF)
    assert np.array_equal(gkc.cpu().numpy(), okc)
    assert np.array_equal(gvc.cpu().numpy(), ovc)


def _decode_pair(cfg, lay, okc, ovc, gkc, gvc, q, num_splits=0):
    tab, lens = gpu_tables(lay)
    out = kv4.kv4_decode_attention(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                   cfg.softmax_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale, latent=cfg.latent)
    return out.cpu().numpy().astype(np.float64), ref


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_attention_parity(name):
    cfg = SMALL[name]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    got, ref = _decode_pair(cfg, lay, okc, ovc, gkc, gvc, q)
    err = np.abs(got - ref).max()
    assert np.isfinite(got).all()
    assert err <= TOL, f"max abs error {err:.3e}"


def test_decode_split_count_invariance():
    cfg = SMALL["b32_small"]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    outs = []
    for S in (1, 2, 5, 63):
        got, ref = _decode_pair(cfg, lay, okc, ovc, gkc, gvc, q, num_splits=S)
        assert np.abs(got - ref).max() <= TOL, S
        outs.append(got)
    # Split counts change which tokens share a warp's running row sum, and so
    # which tokens keep the lo part of P (a token above a share of that sum);
    # the others' f16 rounding of p (2^-11 relative) differs between counts.
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-3


@pytest.mark.parametrize("ctx", [1, 3, 15, 16, 17, 33])
def test_decode_short_and_ragged_contexts(ctx):
    T = 3 if ctx >= 3 else 1
    cfg = W.scaled(W.CONFIGS["verify_agentic"] if T == 3 else W.CONFIGS["b32_ctx8k"], batch=2,
                   ctx=("fixed", ctx))
    cfg = W.dataclasses.replace(cfg, shared_prefix=0.0)
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    got, ref = _decode_pair(cfg, lay, okc, ovc, gkc, gvc, q, num_splits=4)
    assert np.abs(got - ref).max() <= TOL


def test_empty_batch_is_a_no_op():
    q = torch.empty((0, 1, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1088 * 2, dtype=torch.uint8, device="cuda")
    tab = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    lens = torch.zeros((0,), dtype=torch.int32, device="cuda")
    out = kv4.kv4_decode_attention(q, kc, kc.clone(), tab, lens, 1, 1, 0.1, num_splits=1)
    assert out.shape == (0, 1, 8, 128)


def test_device_bounds_errors_are_flagged_not_fatal():
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=2, ctx=("fixed", 40))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    tab, lens = gpu_tables(lay)
    q = W.queries(cfg).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_tab = tab.clone()
    bad_tab[1, 1] = lay.num_pages + 5
    out = kv4.kv4_decode_attention(q, gkc, gvc, bad_tab, lens, cfg.num_kv_heads, lay.num_pages,
                                   cfg.softmax_scale, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kv4.KV4_DEVERR_PAGE
    assert torch.isfinite(out).all()
    err.zero_()
    bad_lens = lens.clone()
    bad_lens[0] = lay.max_pages * cfg.page_size + 1
    kv4.kv4_decode_attention(q, gkc, gvc, tab, bad_lens, cfg.num_kv_heads, lay.num_pages,
                             cfg.softmax_scale, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kv4.KV4_DEVERR_CONTEXT
    err.zero_()
    bad_slots = torch.tensor([lay.num_pages * cfg.page_size + 3], dtype=torch.int32, device="cuda")
    kv4.kv4_append_quantize(k[:1].cuda(), v[:1].cuda(), bad_slots, gkc, gvc, lay.num_pages, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kv4.KV4_DEVERR_SLOT


def test_split_combine_matches_direct_merge():
    torch.manual_seed(0)
    B, T, Hq, S, D = 2, 3, 4, 5, 128
    po = torch.randn(B, T, Hq, S, D, device="cuda")
    pl = torch.randn(B, T, Hq, S, device="cuda") * 3
    pl[0, 0, 0, 2] = float("-inf")
    out = kv4.kv4_split_combine(po, pl)
    w = torch.softmax(pl.double(), dim=-1)
    merged = (w.unsqueeze(-1) * po.double()).sum(-2).cpu().numpy()
    want = oracle.rotate_f64(merged.reshape(-1, D)[0])  # spot-check one row's rotation path
    got = out.double().cpu().numpy()
    H = np.stack([oracle.rotate_f64(np.eye(D)[i]) for i in range(D)])  # H (symmetric)
    full = merged @ H
    assert np.abs(got - full).max() < 1e-5
    assert np.abs(got.reshape(-1, D)[0] - want).max() < 1e-5


# ---------------------------------------------------------------- FP8 comparator
def _fp8_setup(cfg):
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
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
    torch.cuda.synchronize()
    return lay, okc, ovc, gkc, gvc, ks, vs


@pytest.mark.parametrize("name", ["b32_small", "verify_small"])
def test_fp8_append_and_decode_parity(name):
    cfg = SMALL[name]
    lay, okc, ovc, gkc, gvc, ks, vs = _fp8_setup(cfg)
    assert np.array_equal(gkc.cpu().numpy(), okc)
    assert np.array_equal(gvc.cpu().numpy(), ovc)
    q = W.queries(cfg)
    tab, lens = gpu_tables(lay)
    out = kv4.fp8_decode_attention(q.cuda(), gkc, gvc, torch.from_numpy(ks).cuda(),
                                   torch.from_numpy(vs).cuda(), tab, lens, cfg.num_kv_heads,
                                   lay.num_pages, cfg.softmax_scale)
    torch.cuda.synchronize()
    ref = oracle.fp8_decode_attention(q, okc, ovc, ks, vs, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                      lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                      cfg.softmax_scale)
    assert np.abs(out.cpu().numpy() - ref).max() <= TOL


@pytest.mark.parametrize("ctx", [1, 2, 15, 16, 17, 63, 64, 65, 127, 255, 257, 1021])
def test_decode_single_query_ragged_contexts(ctx):
    # T = 1, G = 8: the tensor-core kernel, with partial pages, partial chunks
    # and splits that end mid-chunk
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("fixed", ctx))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    for S in (1, 3):
        got, ref = _decode_pair(cfg, lay, okc, ovc, gkc, gvc, q, num_splits=S)
        assert np.abs(got - ref).max() <= TOL, S


def _fp8_pair(cfg, num_splits=0):
    lay, okc, ovc, gkc, gvc, ks, vs = _fp8_setup(cfg)
    q = W.queries(cfg)
    tab, lens = gpu_tables(lay)
    out = kv4.fp8_decode_attention(q.cuda(), gkc, gvc, torch.from_numpy(ks).cuda(),
                                   torch.from_numpy(vs).cuda(), tab, lens, cfg.num_kv_heads,
                                   lay.num_pages, cfg.softmax_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    ref = oracle.fp8_decode_attention(q, okc, ovc, ks, vs, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                      lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                      cfg.softmax_scale)
    return out.cpu().numpy().astype(np.float64), ref


def test_fp8_split_count_invariance_and_tiny():
    outs = []
    for S in (1, 2, 5, 63):
        got, ref = _fp8_pair(SMALL["b32_small"], num_splits=S)
        assert np.abs(got - ref).max() <= TOL, S
        outs.append(got)
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-4
    got, ref = _fp8_pair(SMALL["tiny"])  # G = 4, outlier channels x20
    assert np.abs(got - ref).max() <= TOL


@pytest.mark.parametrize("ctx", [1, 15, 17, 64, 65, 257])
def test_fp8_single_query_ragged_contexts(ctx):
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=2, ctx=("fixed", ctx))
    got, ref = _fp8_pair(cfg, num_splits=2)
    assert np.abs(got - ref).max() <= TOL


@pytest.mark.parametrize("ctx", [("fixed", 1), ("fixed", 33), ("uniform", 17, 900), ("fixed", 2049)])
def test_mla_latent_decode_ragged_and_split_invariant(ctx):
    # D = 512 latent cache (K = V), 16 query rows per latent head: the latent kernel
    cfg = W.scaled(W.CONFIGS["mla_b8_ctx96k"], batch=3, ctx=ctx)
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    outs = []
    for S in (1, 3, 7):
        got, ref = _decode_pair(cfg, lay, okc, ovc, gkc, gvc, q, num_splits=S)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= TOL, (S, np.abs(got - ref).max())
        outs.append(got)
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-4


def test_decode_with_moderately_dominant_tokens():
    """Rows whose weight sits on a few hundred tokens of a few tenths of a
    percent to a percent each (keys pushed along the query), with values four
    times the workload's: the warp-MMA kernel keeps the lo part of P only for
    tokens above a share of a row's running sum (smaller for larger V), and
    the rest (f16 rounding of p) must still stay within the parity
    tolerance."""
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=2, ctx=("fixed", 3000))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    q = W.queries(cfg)
    G, L = cfg.group, 3000
    gen = torch.Generator().manual_seed(7)
    k = k.float()
    for b in range(cfg.batch):
        base = b * L  # no shared prefix: sequence b's tokens are rows b*L .. b*L + L - 1, in order
        for h in range(cfg.num_kv_heads):
            qh = q[b, 0, h * G].float()
            qhat = qh / qh.norm()
            idx = torch.randperm(L, generator=gen)[:248]
            k[base + idx[:48], h] += 5.0 * qhat      # about 1 % of the row each
            k[base + idx[48:], h] += 3.5 * qhat      # just under 2^-8 of the row each
    k = k.to(torch.bfloat16)
    v = (v.float() * 4.0).to(torch.bfloat16)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    tab, lens = gpu_tables(lay)
    ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale)
    for kernel, S in ((kv4.KV4_KERNEL_AUTO, 0), (kv4.KV4_KERNEL_WARP_MMA, 1), (kv4.KV4_KERNEL_WARP_MMA, 3),
                      (kv4.KV4_KERNEL_BALANCED, 4)):
        out = kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                              cfg.softmax_scale, kernel, num_splits=S)
        torch.cuda.synchronize()
        e = np.abs(out.cpu().numpy().astype(np.float64) - ref).max()
        assert e <= TOL, (kernel, S, e)
