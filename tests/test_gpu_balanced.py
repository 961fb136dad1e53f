"""GPU parity of the warp-MMA kernel's flat mode (KV4_KERNEL_BALANCED: one wave
of CTAs, each an equal part of the flat (sequence, kv head, 4-page chunk)
range, run as one unit per (sequence, kv head) it meets; "UltraQuant on AMD
Instinct", section "Why UltraQuant beats 8-bit KV": a decode step is one
stream over the whole cache) against the CPU oracle, and agreement with the
split form on the same cache: short and ragged contexts (a CTA's part then
crosses many (sequence, kv head) boundaries), many short sequences (parts of
one or two chunks), long ones, GQA groups of 4 and 8, two positions of 4 query
heads, split slot counts 2 to 4, and pages shared by sequences."""
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
    "many_short": W.scaled(_B32, batch=48, ctx=("uniform", 1, 200)),
    "long": W.scaled(_B32, batch=2, ctx=("fixed", 4099)),
    "t2_g4": dataclasses.replace(W.scaled(_B32, batch=3, ctx=("uniform", 50, 1300)), q_per_seq=2, num_q_heads=32),
    "verify_t3": W.scaled(W.CONFIGS["verify_agentic"], batch=4, ctx=("uniform", 300, 1500)),   # 24 rows
    "t2_g8": dataclasses.replace(W.scaled(_B32, batch=3, ctx=("uniform", 50, 1300)), q_per_seq=2),  # 16 rows
    "shared": dataclasses.replace(W.scaled(_B32, batch=4, ctx=("uniform", 600, 3000)), shared_prefix=0.9),
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
def test_balanced_decode_parity(name):
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
    for S in (2, 3, 4):
        got = _run(cfg, lay, gkc, gvc, q, S, kv4.KV4_KERNEL_BALANCED)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= TOL, (S, np.abs(got - ref).max())
        # the two forms give different tokens to a warp's running row sum, so
        # different tokens keep the lo part of P (f16 rounding, 2^-11 relative)
        assert np.abs(got - warp).max() <= 1e-3, (S, np.abs(got - warp).max())


def test_balanced_decode_refuses_other_shapes():
    cfg = W.scaled(W.CONFIGS["verify6_agentic"], batch=1, ctx=("fixed", 100))   # 48 rows
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    tab, lens = gpu_tables(lay)
    with pytest.raises(kv4.Kv4Error) as e:
        kv4.kv4_decode_attention_select(W.queries(cfg).cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads,
                                        lay.num_pages, cfg.softmax_scale, kv4.KV4_KERNEL_BALANCED, num_splits=2)
    assert e.value.status == kv4.KV4_ERR_UNSUPPORTED


def test_balanced_decode_flags_bad_inputs_and_keeps_the_rest():
    """A page id out of range is flagged and read as page 0; a sequence whose
    context length is out of range is flagged, takes no part of the flat range
    and comes out as zeros, and the other sequences keep their result."""
    cfg = W.scaled(_B32, batch=3, ctx=("fixed", 700))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    tab, lens = gpu_tables(lay)
    q = W.queries(cfg).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sel = lambda t_, l_: kv4.kv4_decode_attention_select(q, gkc, gvc, t_, l_, cfg.num_kv_heads, lay.num_pages,
                                                          cfg.softmax_scale, kv4.KV4_KERNEL_BALANCED,
                                                          num_splits=3, dev_error=err)
    good = sel(tab, lens)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bad_tab = tab.clone()
    bad_tab[1, 2] = lay.num_pages + 5
    out = sel(bad_tab, lens)
    torch.cuda.synchronize()
    assert int(err.item()) & kv4.KV4_DEVERR_PAGE
    assert torch.isfinite(out).all()
    err.zero_()
    bad_lens = lens.clone()
    bad_lens[0] = lay.max_pages * cfg.page_size + 1
    out = sel(tab, bad_lens)
    torch.cuda.synchronize()
    assert int(err.item()) & kv4.KV4_DEVERR_CONTEXT
    assert (out[0] == 0).all()
    # the other sequences' chunks are parted differently, so only the rounding differs
    assert (out[1:] - good[1:]).abs().max().item() <= 1e-3


def test_automatic_choice_takes_the_flat_mode_where_it_fills_a_wave():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # four resident CTAs per SM: batch 32 x 8 kv heads with 4 slots fills a wave
    assert kv4.kv4_decode_kernel_choice(32, 1, 64, 8, 128, 4) == (kv4.KV4_KERNEL_BALANCED if 3 * 256 >= 4 * sms
                                                                  else kv4.KV4_KERNEL_WARP_MMA)
    # 2 slots for 64 sequences: a part per sequence is too few for the wave
    assert kv4.kv4_decode_kernel_choice(64, 1, 64, 8, 128, 2) == (kv4.KV4_KERNEL_BALANCED if 512 >= 4 * sms
                                                                  else kv4.KV4_KERNEL_WARP_MMA)


@pytest.mark.parametrize("seed", range(6))
def test_balanced_decode_random_shapes_write_every_slot(seed):
    """Seeded random batches (sizes, context mixes, GQA groups, positions and
    slot counts): the flat mode's parts, units and empty slots must cover
    every partial the combine reads -- the workspace starts as NaN, so a
    partial left unwritten would reach the output -- and agree with the oracle
    and the split form."""
    rng = np.random.default_rng(1000 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    T = int(rng.choice([t for t in (1, 2, 3) if t * G <= 24]))
    Hkv = int(rng.choice([1, 2, 3, 8]))
    batch = int(rng.integers(1, 40))
    hi = int(rng.choice([40, 300, 2000]))
    cfg = dataclasses.replace(W.scaled(_B32, batch=batch, ctx=("uniform", T, max(T + 1, hi)),
                                       name=f"rand{seed}"),
                              num_kv_heads=Hkv, num_q_heads=Hkv * G, q_per_seq=T)
    S = int(rng.integers(2, 9))
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    tab, lens = gpu_tables(lay)
    ws = kv4.workspace(cfg.batch, T, cfg.num_q_heads, cfg.head_dim, S)
    ws.view(torch.float32).fill_(float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                          cfg.softmax_scale, kv4.KV4_KERNEL_BALANCED, num_splits=S,
                                          workspace_buf=ws, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), (G, T, Hkv, batch, hi, S)
    ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale)
    assert np.abs(got - ref).max() <= TOL, (G, T, Hkv, batch, hi, S, np.abs(got - ref).max())
    split = _run(cfg, lay, gkc, gvc, q, S, kv4.KV4_KERNEL_WARP_MMA)
    assert np.abs(got - split).max() <= 1e-3
