"""Parity at the benchmarks' full size (batch 32, 32K context, 8 kv heads, 64
query heads, head_dim 128) in the launch configuration bench.py times: the
whole cache is built and one bench step (append of the new tokens + decode
with the automatic split count) runs on the GPU; sampled (sequence, kv head)
pairs are recomputed one by one by the oracle -- every cached K/V block of the
sample bit-exact, its attention rows within 2e-3.  The extend workload (batch 4,
a 512-token chunk over a 32K context) is checked the same way on both extend
kernels, at sampled chunk positions."""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

SAMPLES = [(0, 3), (17, 6), (31, 0)]  # (sequence, kv head)


@pytest.fixture(scope="module")
def fullsize():
    import bench
    cfg = W.CONFIGS["b32_ctx32k"]
    wl = bench.Workload(cfg, kv4, with_fp8=False)
    kv4.kv4_append_quantize(wl.new_k, wl.new_v, wl.new_slots, wl.kc, wl.vc, wl.lay.num_pages)
    out = kv4.kv4_decode_attention(wl.q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, wl.lay.num_pages,
                                   cfg.softmax_scale, num_splits=wl.S, workspace_buf=wl.ws)
    torch.cuda.synchronize()
    return cfg, wl, out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("b,h", SAMPLES)
def test_fullsize_sampled_parity(fullsize, b, h):
    cfg, wl, out = fullsize
    lay, P, D, G = wl.lay, cfg.page_size, cfg.head_dim, cfg.group
    L = int(lay.context_lens[b])
    n_pages = (L + P - 1) // P
    k, v = W.sequence_tokens(cfg, lay, b)
    k = k[:, h:h + 1].contiguous()
    v = v[:, h:h + 1].contiguous()
    bb = oracle.block_bytes(P, D)
    okc = np.zeros(n_pages * bb, np.uint8)
    ovc = np.zeros_like(okc)
    assert oracle.append_quantize(k, v, np.arange(L, dtype=np.int32), okc, ovc, n_pages, P) == oracle.OK
    # the sequence's blocks in the GPU cache, page by page
    phys = lay.block_tables[b, :n_pages].astype(np.int64)
    idx = ((phys * cfg.num_kv_heads + h) * bb)[:, None] + np.arange(bb)[None, :]
    gkc = wl.kc[torch.from_numpy(idx.reshape(-1)).cuda()].cpu().numpy()
    gvc = wl.vc[torch.from_numpy(idx.reshape(-1)).cuda()].cpu().numpy()
    assert np.array_equal(gkc, okc), "K blocks differ from the oracle"
    assert np.array_equal(gvc, ovc), "V blocks differ from the oracle"
    q = W.queries(cfg)[b:b + 1, :, h * G:(h + 1) * G].contiguous()
    ref = oracle.decode_attention(q, okc, ovc, np.arange(n_pages, dtype=np.int32)[None, :],
                                  np.array([L], dtype=np.int32), 1, P, n_pages, cfg.softmax_scale)
    got = out[b:b + 1, :, h * G:(h + 1) * G]
    err = np.abs(got - ref).max()
    assert err <= TOL, f"max abs error {err:.3e}"


# ---- extend step at full size: batch 4, a 512-token chunk over a 32K context
EXT_SAMPLES = [(0, 5, (0, 300, 511)), (3, 2, (17, 511))]  # (sequence, kv head, positions)


@pytest.fixture(scope="module", params=["tcgen05", "warp"])
def fullsize_extend(request):
    import os
    import bench
    if request.param == "warp":
        os.environ["KV4_EXTEND_WARPMMA"] = "1"
    try:
        cfg = W.CONFIGS["extend_b4_ctx32k_t512"]
        wl = bench.Workload(cfg, kv4, with_fp8=False)
        kv4.kv4_append_quantize(wl.new_k, wl.new_v, wl.new_slots, wl.kc, wl.vc, wl.lay.num_pages)
        out = kv4.kv4_decode_attention(wl.q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, wl.lay.num_pages,
                                       cfg.softmax_scale, num_splits=wl.S, workspace_buf=wl.ws)
        torch.cuda.synchronize()
    finally:
        os.environ.pop("KV4_EXTEND_WARPMMA", None)
    return cfg, wl, out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("b,h,positions", EXT_SAMPLES)
def test_fullsize_extend_sampled_parity(fullsize_extend, b, h, positions):
    """Position j of the chunk equals a single-query decode over the first
    L - T + 1 + j tokens, computed by the oracle from its own cache."""
    cfg, wl, out = fullsize_extend
    lay, P, D, G, T = wl.lay, cfg.page_size, cfg.head_dim, cfg.group, cfg.q_per_seq
    L = int(lay.context_lens[b])
    n_pages = (L + P - 1) // P
    k, v = W.sequence_tokens(cfg, lay, b)
    k = k[:, h:h + 1].contiguous()
    v = v[:, h:h + 1].contiguous()
    bb = oracle.block_bytes(P, D)
    okc = np.zeros(n_pages * bb, np.uint8)
    ovc = np.zeros_like(okc)
    assert oracle.append_quantize(k, v, np.arange(L, dtype=np.int32), okc, ovc, n_pages, P) == oracle.OK
    q_all = W.queries(cfg)
    for j in positions:
        q = q_all[b:b + 1, j:j + 1, h * G:(h + 1) * G].contiguous()
        ref = oracle.decode_attention(q, okc, ovc, np.arange(n_pages, dtype=np.int32)[None, :],
                                      np.array([L - T + 1 + j], dtype=np.int32), 1, P, n_pages, cfg.softmax_scale)
        got = out[b:b + 1, j:j + 1, h * G:(h + 1) * G]
        err = np.abs(got - ref).max()
        assert err <= TOL, f"position {j}: max abs error {err:.3e}"
