"""Seeded synthetic workloads for 4-bit KV-cache decode attention.

This module only draws inputs (bf16 tensors, page tables, context lengths,
slot mappings).  It holds none of the method's arithmetic, so the CUDA path
and the CPU oracle can both be fed from it.

The shapes follow the long-context agentic serving described on the
"UltraQuant on AMD Instinct" page (section "Agentic serving / workload and
setup": long shared prefixes, prefix caching hit rate 91-95 %, 262K context;
section "Throughput-latency trade-off": 3-position MTP verify, with fused
multi-token decode as future work; the 6-token EAGLE verify of the OneNexus
"GLM-5.3-Flash MXFP4" page) and the MLA
latent row of the GLM serving note (512 values per token, no RoPE half).
The page replays an InferenceX agentic trace that is not available here;
these seeded generators stand in for it.

Every sequence's tokens are drawn from their own CPU generator seeded by
(config seed, sequence), so any single sequence can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    batch: int
    q_per_seq: int          # T: query positions per sequence (3 = MTP verify block)
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    ctx: tuple              # ("fixed", L) or ("uniform", lo, hi)
    latent: bool = False    # one cache holds K and V (MLA latent row)
    outliers: str = "none"  # "fixed4x20" | "pct2x16" | "studentt5pct"
    shared_prefix: float = 0.0
    seed: int = 1234

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


CONFIGS = {
    # 1 sequence, GQA 4, context 1024; 4 fixed outlier channels x20 in Q, K, V.
    "tiny": Config("tiny", 1, 1, 4, 1, 128, 16, ("fixed", 1024), outliers="fixed4x20", seed=1235),
    # batch 32, context 8K, GQA 8, 2 % outlier channels x16 in K and V.
    "b32_ctx8k": Config("b32_ctx8k", 32, 1, 64, 8, 128, 16, ("fixed", 8192), outliers="pct2x16", seed=1236),
    "b32_ctx16k": Config("b32_ctx16k", 32, 1, 64, 8, 128, 16, ("fixed", 16384), outliers="pct2x16", seed=1237),
    "b32_ctx32k": Config("b32_ctx32k", 32, 1, 64, 8, 128, 16, ("fixed", 32768), outliers="pct2x16", seed=1237),
    # MLA-style latent cache: one 512-wide latent row per token, 16 query heads.
    "mla_b8_ctx96k": Config("mla_b8_ctx96k", 8, 1, 16, 1, 512, 16, ("fixed", 98304), latent=True,
                            outliers="studentt5pct", seed=1238),
    # MTP verify + agentic traffic: ragged 16K..128K contexts, 93 % shared prefix pages, T = 3.
    "verify_agentic": Config("verify_agentic", 32, 3, 64, 8, 128, 16, ("uniform", 16384, 131072),
                             outliers="pct2x16", shared_prefix=0.93, seed=1239),
    # Longer verify block (EAGLE-style 6-token speculation): the same traffic, T = 6.
    "verify6_agentic": Config("verify6_agentic", 32, 6, 64, 8, 128, 16, ("uniform", 16384, 131072),
                              outliers="pct2x16", shared_prefix=0.93, seed=1241),
    # Extend step: a 512-token chunk of new prompt per sequence over a 32K cached
    # context (the chunk included), causal among the new tokens.
    "extend_b4_ctx32k_t512": Config("extend_b4_ctx32k_t512", 4, 512, 64, 8, 128, 16, ("fixed", 32768),
                                    outliers="pct2x16", seed=1240),
}


def scaled(cfg: Config, batch: int | None = None, ctx=None, name: str | None = None) -> Config:
    """A smaller copy of a config (same distributions) for oracle-sized tests."""
    return dataclasses.replace(cfg, batch=cfg.batch if batch is None else batch,
                               ctx=cfg.ctx if ctx is None else ctx,
                               name=name or (cfg.name + "_small"))


@dataclasses.dataclass
class Layout:
    context_lens: np.ndarray      # int32 [B], includes the T tokens of the step
    block_tables: np.ndarray      # int32 [B, max_pages], -1 past the sequence's pages
    num_pages: int
    prefix_pages: np.ndarray      # int32 [B]: leading table entries that point into the shared chain
    chain: np.ndarray             # int32 [n_chain]: physical pages of the shared prefix chain

    @property
    def max_pages(self) -> int:
        return int(self.block_tables.shape[1])


def _gen(cfg: Config, *key: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    s = cfg.seed
    for k in key:
        s = (s * 1000003 + int(k) + 17) % (2 ** 62)
    g.manual_seed(s)
    return g


def make_layout(cfg: Config) -> Layout:
    """Context lengths and a page table over one shared physical page pool."""
    B, P = cfg.batch, cfg.page_size
    rng = np.random.default_rng(cfg.seed)
    if cfg.ctx[0] == "fixed":
        lens = np.full(B, cfg.ctx[1], dtype=np.int64)
    else:
        lens = rng.integers(cfg.ctx[1], cfg.ctx[2] + 1, size=B)
    pages_needed = (lens + P - 1) // P
    # Shared prefix: sequence b's first floor(f * L_b / P) table entries point at
    # one common physical chain; the T new tokens always land on private pages.
    prefix = np.floor(cfg.shared_prefix * lens / P).astype(np.int64)
    prefix = np.minimum(prefix, (lens - cfg.q_per_seq) // P)
    n_chain = int(prefix.max()) if B else 0
    n_private = int((pages_needed - prefix).sum())
    num_pages = n_chain + n_private
    perm = rng.permutation(num_pages).astype(np.int32)
    chain = perm[:n_chain]
    private = perm[n_chain:]
    max_pages = int(pages_needed.max())
    tables = np.full((B, max_pages), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        k = int(prefix[b])
        tables[b, :k] = chain[:k]
        m = int(pages_needed[b] - k)
        tables[b, k:k + m] = private[pos:pos + m]
        pos += m
    return Layout(lens.astype(np.int32), tables, num_pages, prefix.astype(np.int32), chain)


def _outlier_channels(cfg: Config) -> list:
    """Per KV head, the channels that carry outliers (fixed by the config seed)."""
    rng = np.random.default_rng(cfg.seed + 99)
    D = cfg.head_dim
    if cfg.outliers == "fixed4x20":
        return [np.array([7, 31, 64, 100]) for _ in range(cfg.num_kv_heads)]
    if cfg.outliers == "pct2x16":
        n = int(round(0.02 * D))
        return [np.sort(rng.choice(D, n, replace=False)) for _ in range(cfg.num_kv_heads)]
    if cfg.outliers == "studentt5pct":
        n = int(round(0.05 * D))
        return [np.sort(rng.choice(D, n, replace=False)) for _ in range(cfg.num_kv_heads)]
    return [np.array([], dtype=np.int64) for _ in range(cfg.num_kv_heads)]


def _draw(cfg: Config, g: torch.Generator, n: int) -> torch.Tensor:
    """n tokens x Hkv heads x D channels, fp32, with the config's outlier structure."""
    Hkv, D = cfg.num_kv_heads, cfg.head_dim
    x = torch.randn((n, Hkv, D), generator=g, dtype=torch.float32)
    chans = _outlier_channels(cfg)
    for h in range(Hkv):
        c = torch.as_tensor(chans[h], dtype=torch.long)
        if c.numel() == 0:
            continue
        if cfg.outliers == "fixed4x20":
            x[:, h, c] *= 20.0
        elif cfg.outliers == "pct2x16":
            x[:, h, c] *= 16.0
        elif cfg.outliers == "studentt5pct":
            # Student-t with 3 degrees of freedom: Z / sqrt(chi2_3 / 3).
            z = torch.randn((n, c.numel()), generator=g, dtype=torch.float32)
            chi2 = (torch.randn((n, c.numel(), 3), generator=g, dtype=torch.float32) ** 2).sum(-1)
            x[:, h, c] = z / torch.sqrt(chi2 / 3.0)
    return x


def _draw_kv(cfg: Config, key: tuple, n: int):
    g = _gen(cfg, *key)
    k = _draw(cfg, g, n).to(torch.bfloat16)
    v = None if cfg.latent else _draw(cfg, g, n).to(torch.bfloat16)
    return k, v


def chain_tokens(cfg: Config, layout: Layout, lo: int, hi: int):
    """Tokens [lo, hi) of the shared prefix chain (K, V bf16 [n, Hkv, D])."""
    n_total = int(layout.chain.size) * cfg.page_size
    assert 0 <= lo <= hi <= n_total
    k, v = _draw_kv(cfg, (1, 0), n_total) if n_total else (None, None)
    if n_total == 0:
        return k, v
    return k[lo:hi], (None if v is None else v[lo:hi])


def private_tokens(cfg: Config, layout: Layout, b: int):
    """Sequence b's private tokens: positions [prefix_b * P, L_b)."""
    L = int(layout.context_lens[b])
    start = int(layout.prefix_pages[b]) * cfg.page_size
    return _draw_kv(cfg, (2, b), L - start)


def sequence_tokens(cfg: Config, layout: Layout, b: int, chain_cache=None):
    """All L_b tokens of sequence b in position order (K, V bf16 [L_b, Hkv, D])."""
    start = int(layout.prefix_pages[b]) * cfg.page_size
    kp, vp = private_tokens(cfg, layout, b)
    if start == 0:
        return kp, vp
    if chain_cache is None:
        chain_cache = chain_tokens(cfg, layout, 0, int(layout.chain.size) * cfg.page_size)
    kc, vc = chain_cache
    k = torch.cat([kc[:start], kp], 0)
    v = None if vp is None else torch.cat([vc[:start], vp], 0)
    return k, v


def slots_for(layout: Layout, b: int, lo: int, hi: int, page_size: int) -> np.ndarray:
    """Physical cache slots of sequence b's positions [lo, hi)."""
    pos = np.arange(lo, hi, dtype=np.int64)
    pages = layout.block_tables[b, pos // page_size].astype(np.int64)
    return (pages * page_size + pos % page_size).astype(np.int32)


def chain_slots(cfg: Config, layout: Layout, lo: int, hi: int) -> np.ndarray:
    pos = np.arange(lo, hi, dtype=np.int64)
    return (layout.chain[pos // cfg.page_size].astype(np.int64) * cfg.page_size
            + pos % cfg.page_size).astype(np.int32)


def queries(cfg: Config) -> torch.Tensor:
    """bf16 [B, T, Hq, D]; config 'tiny' carries the same x20 outlier channels in Q."""
    g = _gen(cfg, 3)
    q = torch.randn((cfg.batch, cfg.q_per_seq, cfg.num_q_heads, cfg.head_dim), generator=g,
                    dtype=torch.float32)
    if cfg.outliers == "fixed4x20":
        q[..., [7, 31, 64, 100]] *= 20.0
    return q.to(torch.bfloat16)


def fp8_head_scales(k: torch.Tensor, v: torch.Tensor):
    """Per-KV-head calibration for the FP8 comparator: scale_h = amax_h / 448.

    k, v: bf16 [n, Hkv, D] covering every token the cache will hold.
    Returns (k_scale, v_scale, k_inv_scale, v_inv_scale) as float32 numpy arrays,
    with inv_scale = fp32(1 / scale) computed here on the host.
    """
    def one(x):
        amax = x.float().abs().amax(dim=(0, 2)).numpy().astype(np.float64)
        s = (np.maximum(amax, 1e-30) / 448.0).astype(np.float32)
        inv = (1.0 / s.astype(np.float64)).astype(np.float32)
        return s, inv
    ks, kinv = one(k)
    vs, vinv = one(v)
    return ks, vs, kinv, vinv
