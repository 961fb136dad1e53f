"""GPU parity of the warp-specialised tcgen05 latent (MLA) kernel
(KV4_KERNEL_LATENT_TC: Q.K^T as block-scaled mxf4 MMAs straight from the
cached latent codes and scale bytes, P.V as f16 MMAs on V widened once per
chunk; "UltraQuant on AMD Instinct", section "What is UltraQuant", and the
512-value latent row of "GLM-5.3-Flash on MI300X") against the CPU oracle, and
agreement with the warp-MMA latent kernel on the same cache: several chunks of
128 tokens per split, ragged contexts and last pages, 16 query heads (and 8),
two positions of 8 heads, split counts 1 to 3, and pages shared by sequences."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL, all_tokens, gpu_caches, gpu_tables, oracle_caches

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

_MLA = W.CONFIGS["mla_b8_ctx96k"]
CASES = {
    "small": W.scaled(_MLA, batch=2, ctx=("fixed", 1000)),
    "ragged": W.scaled(_MLA, batch=5, ctx=("uniform", 1, 900)),
    "long": W.scaled(_MLA, batch=2, ctx=("fixed", 4099)),
    "g8": dataclasses.replace(W.scaled(_MLA, batch=3, ctx=("uniform", 100, 1500)), num_q_heads=8),
    "t2_g8": dataclasses.replace(W.scaled(_MLA, batch=3, ctx=("uniform", 50, 1300)), q_per_seq=2, num_q_heads=8),
    "shared": dataclasses.replace(W.scaled(_MLA, batch=3, ctx=("uniform", 600, 2000)), shared_prefix=0.9),
}


def _run(cfg, lay, gkc, q, S, kernel):
    tab, lens = gpu_tables(lay)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv4.kv4_decode_attention_select(q.cuda(), gkc, None, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                          cfg.softmax_scale, kernel, num_splits=S, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", list(CASES))
def test_latent_tc_parity(name):
    cfg = CASES[name]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, _ = oracle_caches(cfg, lay, k, v, slots)
    gkc, _ = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    ref = oracle.decode_attention(q, okc, None, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale, latent=True)
    warp = _run(cfg, lay, gkc, q, 2, kv4.KV4_KERNEL_LATENT)
    for S in (1, 2, 3):
        got = _run(cfg, lay, gkc, q, S, kv4.KV4_KERNEL_LATENT_TC)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= TOL, (S, np.abs(got - ref).max())
        assert np.abs(got - warp).max() <= 5e-4, (S, np.abs(got - warp).max())


def test_latent_tc_refuses_other_caches():
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=1, ctx=("fixed", 100))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    tab, lens = gpu_tables(lay)
    with pytest.raises(kv4.Kv4Error) as e:
        kv4.kv4_decode_attention_select(W.queries(cfg).cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads,
                                        lay.num_pages, cfg.softmax_scale, kv4.KV4_KERNEL_LATENT_TC)
    assert e.value.status == kv4.KV4_ERR_UNSUPPORTED
