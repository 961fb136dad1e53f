"""Shared test harness: builds the same cache on the GPU (through the C ABI)
and on the CPU (through the oracle) from one seeded workload."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W

TOL = 2e-3  # max abs error of attention outputs vs the fp64 oracle


def all_tokens(cfg, lay):
    """Every cached token once: (k, v, slots) with shared-prefix tokens appended once."""
    ks, vs, ss = [], [], []
    n_chain = int(lay.prefix_pages.max()) * cfg.page_size if cfg.batch else 0
    chain = None
    if n_chain:
        chain = W.chain_tokens(cfg, lay, 0, int(lay.chain.size) * cfg.page_size)
        ks.append(chain[0][:n_chain])
        vs.append(None if chain[1] is None else chain[1][:n_chain])
        ss.append(W.chain_slots(cfg, lay, 0, n_chain))
    for b in range(cfg.batch):
        start = int(lay.prefix_pages[b]) * cfg.page_size
        kp, vp = W.private_tokens(cfg, lay, b)
        ks.append(kp)
        vs.append(vp)
        ss.append(W.slots_for(lay, b, start, int(lay.context_lens[b]), cfg.page_size))
    k = torch.cat(ks, 0)
    v = None if cfg.latent else torch.cat(vs, 0)
    return k, v, np.concatenate(ss).astype(np.int32)


def oracle_caches(cfg, lay, k, v, slots):
    bb = oracle.block_bytes(cfg.page_size, cfg.head_dim)
    kc = np.zeros(lay.num_pages * cfg.num_kv_heads * bb, np.uint8)
    vc = None if cfg.latent else np.zeros_like(kc)
    st = oracle.append_quantize(k, v, slots, kc, vc, lay.num_pages, cfg.page_size)
    assert st == oracle.OK, st
    return kc, vc


def gpu_caches(kv4, cfg, lay, k, v, slots, fill=0):
    n = kv4.kv4_cache_bytes(lay.num_pages, cfg.num_kv_heads, cfg.page_size, cfg.head_dim)
    kc = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
    vc = None if cfg.latent else torch.full((n,), fill, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv4.kv4_append_quantize(k.cuda(), None if v is None else v.cuda(),
                            torch.from_numpy(slots).cuda(), kc, vc, lay.num_pages, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return kc, vc


def gpu_tables(lay):
    tab = torch.from_numpy(np.where(lay.block_tables < 0, 0, lay.block_tables).astype(np.int32)).cuda()
    return tab, torch.from_numpy(lay.context_lens.astype(np.int32)).cuda()
