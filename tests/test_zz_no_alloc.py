"""The no-allocation decode entry point (kv4_decode_attention_noalloc) is for
callers that cannot allocate device memory, e.g. an operator plugin that only
receives its input and output buffers.  It keeps the split partials in a
fixed array inside libkv4.  These tests call it through the C ABI and check
it against kv4_decode_attention with a caller-allocated workspace, on two
calls in a row with different queries, so a second call cannot lean on what
the first left in the shared array.  The file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from bit_kv_cache_rotate_b300 import workloads as W

pytestmark = pytest.mark.gpu
kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

TOL = 2e-3  # the max abs error the parity tests allow


def _cache(cfg):
    lay = W.make_layout(cfg)
    ks, vs, ss = [], [], []
    for b in range(cfg.batch):
        k, v = W.sequence_tokens(cfg, lay, b)
        ks.append(k)
        vs.append(v)
        ss.append(W.slots_for(lay, b, 0, int(lay.context_lens[b]), cfg.page_size))
    k, v = torch.cat(ks).cuda(), torch.cat(vs).cuda()
    slots = torch.from_numpy(np.concatenate(ss).astype(np.int32)).cuda()
    kc = kv4.empty_cache(lay.num_pages, cfg.num_kv_heads, cfg.head_dim)
    vc = kv4.empty_cache(lay.num_pages, cfg.num_kv_heads, cfg.head_dim)
    kv4.kv4_append_quantize(k, v, slots, kc, vc, lay.num_pages)
    tab = torch.from_numpy(lay.block_tables.clip(min=0)).cuda()
    lens = torch.from_numpy(lay.context_lens).cuda()
    return lay, kc, vc, tab, lens


def _noalloc_c(q, kc, vc, tab, lens, cfg, lay, num_splits, out):
    fn = kv4.lib().kv4_decode_attention_noalloc
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, P, P, P]
    fn.restype = i32
    B, T, Hq, D = q.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return fn(p(q), p(kc), p(vc), p(tab), p(lens), B, T, Hq, cfg.num_kv_heads, D, cfg.page_size,
              tab.shape[1], lay.num_pages, cfg.softmax_scale, num_splits, p(out), None,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("fixed", 1000))
    lay, kc, vc, tab, lens = _cache(cfg)
    for call in range(2):
        q = (W.queries(cfg).float() * (1.0 + 0.5 * call)).to(torch.bfloat16).cuda()
        want = kv4.kv4_decode_attention(q, kc, vc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                        cfg.softmax_scale)
        got = torch.full_like(want, float("nan"))
        st = _noalloc_c(q, kc, vc, tab, lens, cfg, lay, 0, got)
        torch.cuda.synchronize()
        assert st == kv4.KV4_OK
        assert torch.isfinite(got).all()
        assert (got - want).abs().max().item() <= TOL, f"call {call}"


def test_noalloc_rejects_partials_beyond_its_scratch():
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=2, ctx=("fixed", 64))
    lay, kc, vc, tab, lens = _cache(cfg)
    q = W.queries(cfg).cuda()
    out = torch.full((cfg.batch, 1, cfg.num_q_heads, cfg.head_dim), 7.0, device="cuda")
    limit = 16 << 20
    per_split = cfg.batch * cfg.num_q_heads * cfg.head_dim * 4
    too_many = limit // per_split + 1
    st = _noalloc_c(q, kc, vc, tab, lens, cfg, lay, too_many, out)
    torch.cuda.synchronize()
    assert st == kv4.KV4_ERR_INVALID_ARG
    assert (out == 7.0).all()  # nothing was launched


def test_noalloc_lowers_an_automatic_split_count_that_does_not_fit():
    """head_dim 256, 24 query rows per kv head, 8 sequences: the automatic split
    count (130) needs about 24 MiB of partials, more than the fixed array holds.
    With num_splits = 0 the entry point lowers the count until they fit and
    must still match the workspace entry point (which keeps the 130 splits)."""
    import dataclasses
    cfg = dataclasses.replace(W.CONFIGS["b32_ctx8k"], name="d256_g24", batch=8, ctx=("fixed", 8320),
                              num_q_heads=24, num_kv_heads=1, head_dim=256)
    lay, kc, vc, tab, lens = _cache(cfg)
    S = kv4.kv4_decode_auto_splits(cfg.batch, 1, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim,
                                   cfg.page_size, tab.shape[1])
    assert kv4.kv4_decode_workspace_bytes(cfg.batch, 1, cfg.num_q_heads, cfg.head_dim, S) > 16 << 20
    q = W.queries(cfg).cuda()
    want = kv4.kv4_decode_attention(q, kc, vc, tab, lens, cfg.num_kv_heads, lay.num_pages, cfg.softmax_scale)
    got = torch.full_like(want, float("nan"))
    st = _noalloc_c(q, kc, vc, tab, lens, cfg, lay, 0, got)
    torch.cuda.synchronize()
    assert st == kv4.KV4_OK
    assert torch.isfinite(got).all()
    assert (got - want).abs().max().item() <= TOL


def test_noalloc_reserves_no_memory_after_its_first_call():
    """The fixed array is reserved when the library's module holding it loads on
    the device (at the first call, under CUDA's lazy module loading); from then
    on calls leave the device's free memory unchanged."""
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("fixed", 1000))
    lay, kc, vc, tab, lens = _cache(cfg)
    q = W.queries(cfg).cuda()
    out = torch.empty((cfg.batch, 1, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    assert _noalloc_c(q, kc, vc, tab, lens, cfg, lay, 0, out) == kv4.KV4_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc_c(q, kc, vc, tab, lens, cfg, lay, 0, out) == kv4.KV4_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
