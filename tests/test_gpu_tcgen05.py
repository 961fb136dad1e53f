"""GPU parity of the warp-specialised tcgen05 decode kernel
(KV4_KERNEL_TCGEN05: Q.K^T as block-scaled mxf4 MMAs straight from the
cache's codes and scale bytes, "UltraQuant on AMD Instinct", section "What is
UltraQuant") against the CPU oracle, and agreement with the warp-MMA kernel on
the same cache: several chunks of 128 tokens per split, ragged contexts and
last pages, GQA groups of 4 and 8, two positions of 4 query heads, split
counts 1 to 3."""
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
CASES = {
    "tiny": W.CONFIGS["tiny"],                                     # G = 4, outliers x20
    "b32_small": W.scaled(_B32, batch=3, ctx=("fixed", 1000)),
    "ragged": W.scaled(_B32, batch=5, ctx=("uniform", 1, 900)),
    "long": W.scaled(_B32, batch=2, ctx=("fixed", 4099)),
    "t2_g4": dataclasses.replace(W.scaled(_B32, batch=3, ctx=("uniform", 50, 1300)), q_per_seq=2, num_q_heads=32),
}


def _run(cfg, lay, gkc, gvc, q, S, kernel):
    tab, lens = gpu_tables(lay)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                          cfg.softmax_scale, kernel, num_splits=S, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", list(CASES))
def test_tcgen05_decode_parity(name):
    cfg = CASES[name]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale)
    warp = _run(cfg, lay, gkc, gvc, q, 2, kv4.KV4_KERNEL_WARP_MMA)
    for S in (1, 2, 3):
        got = _run(cfg, lay, gkc, gvc, q, S, kv4.KV4_KERNEL_TCGEN05)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= TOL, (S, np.abs(got - ref).max())
        # the kernels keep the lo part of P for different tokens (f16 rounding of
        # the rest, 2^-11 relative)
        assert np.abs(got - warp).max() <= 1e-3, (S, np.abs(got - warp).max())


def test_tcgen05_decode_refuses_more_than_eight_rows():
    cfg = W.scaled(W.CONFIGS["verify_agentic"], batch=1, ctx=("fixed", 100))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    tab, lens = gpu_tables(lay)
    with pytest.raises(kv4.Kv4Error) as e:
        kv4.kv4_decode_attention_select(W.queries(cfg).cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads,
                                        lay.num_pages, cfg.softmax_scale, kv4.KV4_KERNEL_TCGEN05)
    assert e.value.status == kv4.KV4_ERR_UNSUPPORTED
