"""GPU parity when V scales span a wide range inside one sequence.

The cache keeps one power-of-two scale per token and 32 channels ("UltraQuant
on AMD Instinct", section "What is UltraQuant"), so one token's values may lie
many binades above the others'.  Here every sequence holds one such token:
its V (or, for the latent cache, its whole row) is the ordinary draw times
2^16 or 2^40, and its K is the least-norm vector that gives every query row
of its group the same very negative logit, so its softmax weight is
negligible and the output is made by the ordinary tokens.  A kernel whose V
reference follows that token and flushes values far below it would lose the
ordinary tokens' contributions; the oracle computes the exact attention over
the dequantised cache.  Every 4-bit decode kernel must agree within 2e-3.
"""
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
_VER = dataclasses.replace(W.CONFIGS["verify_agentic"], shared_prefix=0.0)
_MLA = W.CONFIGS["mla_b8_ctx96k"]
_EXT = W.CONFIGS["extend_b4_ctx32k_t512"]

# name -> (config, kernel choice)
CASES = {
    "warp_t1": (W.scaled(_B32, batch=3, ctx=("uniform", 200, 1500)), 0),
    "warp_t2": (dataclasses.replace(W.scaled(_B32, batch=3, ctx=("uniform", 200, 1200)), q_per_seq=2), 0),
    "warp_t3": (W.scaled(_VER, batch=3, ctx=("uniform", 300, 1500)), 0),
    "general": (W.scaled(_B32, batch=2, ctx=("uniform", 200, 900)), 4),
    "tcgen05": (W.scaled(_B32, batch=3, ctx=("uniform", 200, 1500)), 5),
    "balanced": (W.scaled(_B32, batch=3, ctx=("uniform", 200, 1500)), 7),
    "latent": (W.scaled(_MLA, batch=2, ctx=("uniform", 300, 1200)), 3),
    "latent_tc": (W.scaled(_MLA, batch=2, ctx=("uniform", 300, 1200)), 6),
    "extend_tc": (dataclasses.replace(W.scaled(_EXT, batch=2, ctx=("uniform", 300, 1100)), q_per_seq=6), 2),
    "extend_warp": (dataclasses.replace(W.scaled(_EXT, batch=2, ctx=("uniform", 300, 1100)), q_per_seq=6), 1),
}


def _plant(cfg, lay, k, v, q, log2_scale, seed):
    """One token per sequence, at a seeded position before the new tokens:
    V (latent row) times 2^log2_scale, K chosen so that q . k = -c for every
    query row of its kv head (least-norm solution, fp64, rounded to bf16)."""
    rng = np.random.default_rng(seed)
    G, T, D = cfg.group, cfg.q_per_seq, cfg.head_dim
    offsets = np.concatenate([[0], np.cumsum(lay.context_lens)[:-1]])
    k = k.clone()
    v = None if v is None else v.clone()
    qf = q.float().numpy().astype(np.float64)
    planted = []
    for b in range(cfg.batch):
        L = int(lay.context_lens[b])
        pos = int(rng.integers(0, L - T))
        row = int(offsets[b]) + pos
        planted.append(pos)
        for h in range(cfg.num_kv_heads):
            Q = qf[b, :, h * G:(h + 1) * G].reshape(T * G, D)
            # logit = softmax_scale * q . k = -48 for every row (before quantisation)
            c = 48.0 / cfg.softmax_scale
            kk = -c * np.linalg.pinv(Q) @ np.ones(T * G)
            kk_t = torch.from_numpy(kk.astype(np.float32)).to(torch.bfloat16)
            if cfg.latent:
                k[row, h] = (kk_t.float() * 2.0 ** log2_scale).to(torch.bfloat16)
            else:
                k[row, h] = kk_t
                v[row, h] = (v[row, h].float() * 2.0 ** log2_scale).to(torch.bfloat16)
    return k, v, planted


@pytest.mark.parametrize("log2_scale", [16, 40])
@pytest.mark.parametrize("name", list(CASES))
def test_wide_v_scale_range(name, log2_scale):
    cfg, kernel = CASES[name]
    assert cfg.shared_prefix == 0.0  # sequences are laid out back to back by all_tokens
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    q = W.queries(cfg)
    k, v, _ = _plant(cfg, lay, k, v, q, log2_scale, seed=cfg.seed + log2_scale)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    assert np.array_equal(gkc.cpu().numpy(), okc), "K (latent) cache differs from the oracle"
    if ovc is not None:
        assert np.array_equal(gvc.cpu().numpy(), ovc), "V cache differs from the oracle"
    ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale, latent=cfg.latent)
    # the planted tokens carry no weight: the exact output is of ordinary size
    assert np.abs(ref).max() < 100.0
    tab, lens = gpu_tables(lay)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for S in ((2, 3) if kernel == kv4.KV4_KERNEL_BALANCED else (1, 3)):
        out = kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                              cfg.softmax_scale, kernel, num_splits=S, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), (S, "non-finite output")
        e = np.abs(got - ref).max()
        assert e <= TOL, (S, f"max abs error {e:.3e}")
