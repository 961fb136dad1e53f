"""Rotation accuracy study on synthetic data (run: python tests/rotation_accuracy.py).

"UltraQuant on AMD Instinct", section "What is UltraQuant": a Walsh-Hadamard
rotation before the 4-bit quantisation spreads outlier channels over the whole
head vector, so one power-of-two scale per 32 values fits every group.  The
pages defer the accuracy analysis to the paper and give no numbers; this study
measures it on synthetic vectors with the oracle's own quantiser (E2M1 codes,
one UE8M0 scale per 32 channels), rotated and unrotated:

  * K reconstruction error  ||k - k_hat||^2 / ||k||^2 (mean over tokens);
  * attention error         ||o - o_hat|| / ||o|| against exact fp64 attention,
    averaged over `n_q` queries attending to the whole context, and the
    largest |o - o_hat| over them.

Inputs: N(0, 1) head vectors (bf16-representable) with `n_out` seeded outlier
channels per vector scaled by `factor` in K and V (the decode workloads use
3 channels x 16 at head_dim 128), and N(0, 1) queries.  With large factors the
outlier channels dominate the logits and the softmax approaches one-hot, so
the attention error then measures whether the same few tokens win.  This file is test
infrastructure: it reads the oracle, nothing in the product calls it.
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def _bf16(a: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000  # round to nearest even
    return u.view(np.float32).astype(np.float64)


def _dequant(codes: np.ndarray, expo: np.ndarray, table: np.ndarray) -> np.ndarray:
    return table[codes] * np.repeat(np.ldexp(1.0, expo), 32)


def _quantize(x: np.ndarray, rotate: bool, table: np.ndarray) -> np.ndarray:
    """One head vector through the 4-bit format and back (fp64)."""
    y = oracle.rotate_f64(x) if rotate else x
    codes, expo = oracle.quantize_rotated(y.astype(np.float32))
    y_hat = _dequant(codes, expo, table)
    return oracle.rotate_f64(y_hat) if rotate else y_hat  # H is symmetric and orthonormal


def _attend(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    s = K @ q / np.sqrt(q.size)
    p = np.exp(s - s.max())
    return (p[:, None] * V).sum(0) / p.sum()


def study(n_tokens: int = 1024, D: int = 128, factors=(1, 4, 16, 64), n_out: int = 3, n_q: int = 16,
          seed: int = 0):
    table = np.array([oracle.e2m1_decode(c) for c in range(16)], dtype=np.float64)
    rows = []
    for f in factors:
        rng = np.random.default_rng(seed)
        K = rng.standard_normal((n_tokens, D))
        V = rng.standard_normal((n_tokens, D))
        ch = rng.choice(D, size=n_out, replace=False)
        K[:, ch] *= f
        V[:, ch] *= f
        K, V = _bf16(K), _bf16(V)
        Q = _bf16(rng.standard_normal((n_q, D)))
        O = np.stack([_attend(q, K, V) for q in Q])
        row = {"factor": f}
        for name, rot in (("rotated", True), ("plain", False)):
            Kh = np.stack([_quantize(k, rot, table) for k in K])
            Vh = np.stack([_quantize(v, rot, table) for v in V])
            mse = float(np.mean(np.sum((K - Kh) ** 2, 1) / np.sum(K ** 2, 1)))
            Oh = np.stack([_attend(q, Kh, Vh) for q in Q])
            rel = np.linalg.norm(O - Oh, axis=1) / np.linalg.norm(O, axis=1)
            row[name] = {"k_rel_mse": mse, "attn_max_abs": float(np.abs(O - Oh).max()),
                         "attn_rel_l2": float(rel.mean())}
        rows.append(row)
    return rows


def main():
    rows = study(factors=(1, 2, 4, 8, 16, 32, 64))
    print("| outlier factor | K rel. MSE rotated | K rel. MSE plain | attn max abs rotated | attn max abs plain "
          "| attn rel. L2 rotated (mean) | attn rel. L2 plain (mean) |")
    print("|---|---|---|---|---|---|---|")
    for r in rows:
        a, b = r["rotated"], r["plain"]
        print(f"| {r['factor']} | {a['k_rel_mse']:.2e} | {b['k_rel_mse']:.2e} | {a['attn_max_abs']:.2e} | "
              f"{b['attn_max_abs']:.2e} | {a['attn_rel_l2']:.2e} | {b['attn_rel_l2']:.2e} |")


if __name__ == "__main__":
    main()
