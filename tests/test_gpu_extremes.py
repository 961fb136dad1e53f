"""Quantise-on-append at the edges of the number range, bit-exact against the
oracle: all-zero vectors (scale byte 0, every code +0), one-hot vectors (the
rotation spreads them evenly), vectors scaled by 2^100 and 2^-120 (exponents
near both ends of the UE8M0 range), vectors of bf16 subnormals (a subnormal
group maximum clamps the exponent to -127) and negative zeros.  Every vector
stays inside the rotation's exact domain (its dynamic range is that of a
normal sample), so the oracle reports no inexact sum."""
import numpy as np
import pytest
import torch

import oracle
from _harness import gpu_caches

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

D, HKV, P = 128, 2, 16


def _vectors(seed):
    g = torch.Generator().manual_seed(seed)
    base = lambda n: torch.randn((n, HKV, D), generator=g, dtype=torch.float32)
    parts = [
        torch.zeros((8, HKV, D)),                                    # all zero
        -torch.zeros((4, HKV, D)),                                   # negative zeros
        torch.eye(D)[torch.randint(0, D, (8,), generator=g)].unsqueeze(1).repeat(1, HKV, 1),  # one-hot
        base(8) * 2.0 ** 100,                                        # large
        base(8) * 2.0 ** -120,                                       # small, still normal
        base(8) * 2.0 ** -130,                                       # bf16 subnormals
        base(5),                                                     # ordinary, ragged last page
    ]
    return torch.cat(parts).to(torch.bfloat16).contiguous()


class _Lay:
    def __init__(self, n_tokens):
        self.num_pages = (n_tokens + P - 1) // P


class _Cfg:
    num_kv_heads, head_dim, page_size, latent = HKV, D, P, False


def test_append_extremes_bit_exact():
    k, v = _vectors(1), _vectors(2)
    n = k.shape[0]
    lay = _Lay(n)
    perm = np.random.default_rng(3).permutation(lay.num_pages)
    slots = (perm[np.arange(n) // P] * P + np.arange(n) % P).astype(np.int32)
    bb = oracle.block_bytes(P, D)
    okc = np.zeros(lay.num_pages * HKV * bb, np.uint8)
    ovc = np.zeros_like(okc)
    assert oracle.append_quantize(k, v, slots, okc, ovc, lay.num_pages, P) == oracle.OK
    gkc, gvc = gpu_caches(kv4, _Cfg, lay, k, v, slots)
    for name, g, o in (("K", gkc, okc), ("V", gvc, ovc)):
        diff = np.flatnonzero(g.cpu().numpy() != o)
        assert diff.size == 0, f"{name} cache differs at bytes {diff[:10]} ({diff.size} bytes)"
