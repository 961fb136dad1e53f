"""The bounded-wait timeout path of the streaming kernels, run without a fault
or a hang.

Every wait of a kernel for streamed cache data is bounded; when one runs out
the kernel sets KV4_DEVERR_TIMEOUT, waits (bounded) for the copies and MMAs it
issued, releases its tensor memory and returns.  The test control
KV4_DIAG_EXPIRE_FIRST_WAIT makes each streaming warp's first wait give up
without trying, which takes exactly that path.  The call must return, flag
the timeout, and leave the context usable: the next normal call on the same
cache must match the oracle.
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

_EXT = W.CONFIGS["extend_b4_ctx32k_t512"]

CASES = {
    "warp_t1": (W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("uniform", 100, 900)), 1),
    "warp_t3": (W.scaled(W.CONFIGS["verify_agentic"], batch=3, ctx=("uniform", 300, 900)), 1),
    "tcgen05": (W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("uniform", 100, 900)), 5),
    "balanced": (W.scaled(W.CONFIGS["b32_ctx8k"], batch=3, ctx=("uniform", 100, 900)), 7),
    "latent": (W.scaled(W.CONFIGS["mla_b8_ctx96k"], batch=2, ctx=("uniform", 200, 700)), 3),
    "latent_tc": (W.scaled(W.CONFIGS["mla_b8_ctx96k"], batch=2, ctx=("uniform", 200, 700)), 6),
    "extend_tc": (dataclasses.replace(W.scaled(_EXT, batch=2, ctx=("uniform", 200, 700)), q_per_seq=40), 2),
    "extend_warp": (dataclasses.replace(W.scaled(_EXT, batch=2, ctx=("uniform", 200, 700)), q_per_seq=40), 1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_expired_wait_flags_timeout_and_the_next_call_is_correct(name):
    cfg, kernel = CASES[name]
    lay = W.make_layout(cfg)
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    gkc, gvc = gpu_caches(kv4, cfg, lay, k, v, slots)
    q = W.queries(cfg)
    tab, lens = gpu_tables(lay)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for S in ((2, 3) if kernel == kv4.KV4_KERNEL_BALANCED else (1, 2)):
        err.zero_()
        kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                        cfg.softmax_scale, kernel, diag_flags=kv4.KV4_DIAG_EXPIRE_FIRST_WAIT,
                                        num_splits=S, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) & kv4.KV4_DEVERR_TIMEOUT, "the expired wait was not flagged"
    err.zero_()
    out = kv4.kv4_decode_attention_select(q.cuda(), gkc, gvc, tab, lens, cfg.num_kv_heads, lay.num_pages,
                                          cfg.softmax_scale, kernel, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.decode_attention(q, okc, ovc, np.where(lay.block_tables < 0, 0, lay.block_tables),
                                  lay.context_lens, cfg.num_kv_heads, cfg.page_size, lay.num_pages,
                                  cfg.softmax_scale, latent=cfg.latent)
    e = np.abs(out.cpu().numpy().astype(np.float64) - ref).max()
    assert e <= TOL, f"max abs error {e:.3e}"
