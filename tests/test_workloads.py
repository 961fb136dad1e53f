"""Host-side checks of the seeded workload generator (no GPU)."""
import numpy as np
import pytest

import oracle
from bit_kv_cache_rotate_b300 import workloads as W


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_layout_invariants(name):
    cfg = W.CONFIGS[name]
    if cfg.batch * (cfg.ctx[-1] // cfg.page_size) > 3_000_000:
        pytest.skip("layout too large for a unit test")
    lay = W.make_layout(cfg)
    P = cfg.page_size
    used = []
    for b in range(cfg.batch):
        L = int(lay.context_lens[b])
        n = (L + P - 1) // P
        row = lay.block_tables[b, :n]
        assert (row >= 0).all() and (row < lay.num_pages).all()
        assert (lay.block_tables[b, n:] == -1).all()
        k = int(lay.prefix_pages[b])
        assert np.array_equal(row[:k], lay.chain[:k])
        used.append(row[k:])
        # the step's new tokens never land on a shared page
        assert (L - cfg.q_per_seq) // P >= k
    priv = np.concatenate(used)
    assert len(np.unique(priv)) == priv.size                # private pages are private
    assert not set(priv.tolist()) & set(lay.chain.tolist())
    if cfg.shared_prefix:
        shared = lay.prefix_pages.sum() / ((lay.context_lens + P - 1) // P).sum()
        assert 0.90 < shared < 0.94


def test_sequences_regenerate_identically():
    cfg = W.scaled(W.CONFIGS["verify_agentic"], batch=3, ctx=("uniform", 100, 300))
    lay = W.make_layout(cfg)
    a = W.sequence_tokens(cfg, lay, 1)
    b = W.sequence_tokens(cfg, lay, 1)
    assert a[0].equal(b[0]) and a[1].equal(b[1])
    # the shared prefix content is the same across sequences
    k0, _ = W.sequence_tokens(cfg, lay, 0)
    k2, _ = W.sequence_tokens(cfg, lay, 2)
    n = min(lay.prefix_pages[0], lay.prefix_pages[2]) * cfg.page_size
    assert n > 0 and k0[:n].equal(k2[:n])


@pytest.mark.parametrize("name", ["tiny", "b32_ctx8k", "mla_b8_ctx96k"])
def test_generated_vectors_lie_in_the_exact_rotation_domain(name):
    cfg = W.scaled(W.CONFIGS[name], batch=2, ctx=("fixed", 2048))
    lay = W.make_layout(cfg)
    for b in range(cfg.batch):
        k, v = W.sequence_tokens(cfg, lay, b)
        for x in (k, v):
            if x is None:
                continue
            _, _, bad = oracle.quantize_vectors(x)
            assert bad == 0


def test_outlier_structure():
    cfg = W.scaled(W.CONFIGS["b32_ctx8k"], batch=1, ctx=("fixed", 4096))
    lay = W.make_layout(cfg)
    k, _ = W.sequence_tokens(cfg, lay, 0)
    std = k.float().std(dim=0)                     # [Hkv, D]
    big = (std > 8).sum(dim=1)
    assert (big == round(0.02 * cfg.head_dim)).all()
