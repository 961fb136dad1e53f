"""GPU side of one long context split across devices, emulated on one GPU.

Each sequence is cut into consecutive page-aligned shares (seqsplit.share_ranges).
The share with the newest tokens runs kv4_decode_partials, every other share
kv4_decode_partials_prefix, each on its own page table; the partials are
concatenated along the split axis as the gather would deliver them and merged
by kv4_split_combine.  The result must match the oracle's attention over the
whole sequence within 2e-3, for decode, verify, latent and extend shapes.
No collective runs here: the exchange itself is covered by the gloo test.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import seqsplit
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL, all_tokens, gpu_caches, oracle_caches

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

CASES = {
    "decode": W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("uniform", 40, 2000)),
    "verify": W.scaled(W.CONFIGS["verify_agentic"], batch=3, ctx=("uniform", 300, 2000)),
    "latent": W.scaled(W.CONFIGS["mla_b8_ctx96k"], batch=2, ctx=("uniform", 300, 1500)),
    "extend": dataclasses.replace(W.scaled(W.CONFIGS["extend_b4_ctx32k_t512"], batch=2,
                                           ctx=("uniform", 400, 1500)), q_per_seq=40),
}


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("name", list(CASES))
def test_shares_merge_to_whole_sequence_attention(name, world):
    cfg = CASES[name]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    B, T, Hq, D = q.shape
    tables = np.where(lay.block_tables < 0, 0, lay.block_tables).astype(np.int32)
    ranges = seqsplit.share_ranges(lay.context_lens, T, world, cfg.page_size)
    S = 2
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos, pls = [], []
    for r in range(world):
        tab, lens = seqsplit.local_tables(tables, ranges[r], cfg.page_size)
        ws = kv4.workspace(B, T, Hq, D, S)
        fn = kv4.kv4_decode_partials if r == world - 1 else kv4.kv4_decode_partials_prefix
        fn(q.cuda(), gkc, gvc, torch.from_numpy(tab).cuda(), torch.from_numpy(lens).cuda(), cfg.num_kv_heads,
           lay.num_pages, cfg.softmax_scale, S, ws, dev_error=err)
        po, pl = kv4.split_views(ws, B, T, Hq, D, S)
        pos.append(po.clone())
        pls.append(pl.clone())
    out = kv4.kv4_split_combine(torch.cat(pos, dim=3).contiguous(), torch.cat(pls, dim=3).contiguous())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.decode_attention(q, okc, ovc, tables, lay.context_lens, cfg.num_kv_heads, cfg.page_size,
                                  lay.num_pages, cfg.softmax_scale, latent=cfg.latent)
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    e = np.abs(got - ref).max()
    assert e <= TOL, f"max abs error {e:.3e}"
