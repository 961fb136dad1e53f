"""GPU parity of the tcgen05 block-scaled decode kernel (selected by
KV4_DECODE_TCGEN05=1) against the CPU oracle, and agreement with the default
warp-MMA kernel on the same cache."""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL, all_tokens, gpu_caches, oracle_caches

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

CASES = {
    "tiny": W.CONFIGS["tiny"],                                                       # G = 4, outliers x20
    "b32_small": W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("fixed", 1000)),
    "ragged": W.scaled(W.CONFIGS["b32_ctx8k"], batch=4, ctx=("uniform", 1, 700)),
    "long": W.scaled(W.CONFIGS["b32_ctx8k"], batch=2, ctx=("fixed", 4099)),
}


def _run(cfg, lay, gkc, gvc, q, S):
    tab = torch.from_numpy(np.where(lay.block_tables < 0, 0, lay.block_tables).astype(np.int32)).cuda()
    lens = torch.from_numpy(lay.context_lens.astype(np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv4.kv4_decode_attention(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                   cfg.softmax_scale, num_splits=S, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", list(CASES))
def test_tcgen05_decode_parity(name, monkeypatch):
    cfg = CASES[name]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale)
    default = _run(cfg, lay, gkc, gvc, q, 2)
    monkeypatch.setenv("KV4_DECODE_TCGEN05", "1")
    for S in (1, 2, 3):
        got = _run(cfg, lay, gkc, gvc, q, S)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= TOL, (S, np.abs(got - ref).max())
        assert np.abs(got - default).max() <= 2e-4, S
