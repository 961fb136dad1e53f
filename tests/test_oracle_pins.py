"""Pins of the CPU oracle against facts fixed by the page and by mathematics.

None of these checks re-runs the oracle's own formula: each compares it with
an independent characterisation (closed forms, exact rational arithmetic, a
library routine, brute-force search, invariants), chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one.
"""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rn_inv_sqrt(D):
    getcontext().prec = 60
    return float(Decimal(1) / Decimal(D).sqrt())


# ------------------------------------------------------------------ Hadamard
@pytest.mark.parametrize("D", [2, 8, 64, 128, 512])
def test_hadamard_matches_scipy_and_closed_form(D):
    H = oracle.hadamard_pm1(D).astype(np.int64)
    assert np.array_equal(H, scipy.linalg.hadamard(D))
    i, j = np.meshgrid(np.arange(D), np.arange(D), indexing="ij")
    pop = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    assert np.array_equal(H, np.where(pop % 2 == 0, 1, -1))
    assert np.array_equal(H @ H.T, D * np.eye(D, dtype=np.int64))
    assert np.array_equal(H, H.T)


@pytest.mark.parametrize("D", [64, 128, 512])
def test_rotation_exact_against_rationals(D):
    rng = np.random.default_rng(D)
    H = scipy.linalg.hadamard(D)
    c = _rn_inv_sqrt(D)
    for trial in range(6):
        x = rng.standard_normal(D) * (20.0 if trial % 2 else 1.0)
        xb = _bf16(x)
        xs = xb.float().numpy().astype(np.float64)
        y, st = oracle.rotate_bf16(_bf16_bits(xb))
        assert st == oracle.OK
        for i in range(D):
            S = sum(Fraction(float(xs[j])) * int(H[i, j]) for j in range(D))
            Sf = float(S)
            assert Fraction(Sf) == S  # exact in binary64 for these inputs
            expect = np.float32(Sf * c)
            assert y[i].view(np.uint32) == expect.view(np.uint32), (trial, i)


@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_rotation_closed_forms(D):
    c = _rn_inv_sqrt(D)
    e0 = np.zeros(D, dtype=np.float32)
    e0[0] = 1.0
    y, st = oracle.rotate_bf16(_bf16_bits(_bf16(e0)))
    assert st == oracle.OK
    assert np.all(y == np.float32(c))                 # H e0 = (1/sqrt D) * ones
    y, st = oracle.rotate_bf16(_bf16_bits(_bf16(np.ones(D))))
    assert y[0] == np.float32(D * c)                   # H ones = sqrt(D) e0
    assert np.all(y[1:] == 0.0)
    # a single -1 at index k: row i gets -(-1)^popcount(i&k) / sqrt(D)
    k = 5
    x = np.zeros(D, dtype=np.float32)
    x[k] = -1.0
    y, _ = oracle.rotate_bf16(_bf16_bits(_bf16(x)))
    sign = np.array([(-1) ** bin(i & k).count("1") for i in range(D)])
    assert np.array_equal(y, (-sign * c).astype(np.float32))


@pytest.mark.parametrize("D", [128, 512])
def test_rotation_f64_is_orthonormal_involution(D):
    rng = np.random.default_rng(7)
    v = rng.standard_normal(D)
    hv = oracle.rotate_f64(v)
    assert abs(np.linalg.norm(hv) - np.linalg.norm(v)) < 1e-12 * np.linalg.norm(v)
    assert np.allclose(oracle.rotate_f64(hv), v, atol=1e-13, rtol=0)
    w = rng.standard_normal(D)
    assert abs(hv @ oracle.rotate_f64(w) - v @ w) < 1e-11  # inner products preserved


def test_rotation_flags_inputs_outside_exact_domain():
    x = np.zeros(128, dtype=np.float32)
    x[0], x[1] = 1e30, 1e-30
    _, st = oracle.rotate_bf16(_bf16_bits(_bf16(x)))
    assert st == oracle.INEXACT


# ------------------------------------------------------------------ E2M1 codes
def test_e2m1_decode_table_golden():
    for code, val in _read_golden("e2m1_grid.txt"):
        v = oracle.e2m1_decode(int(code))
        assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))


def test_e2m1_ties_and_saturation_golden():
    for z, code in _read_golden("e2m1_ties.txt"):
        assert int(oracle.e2m1_encode(float(z))[0]) == int(code), z


def _nearest_even_grid(z):
    """Independent brute-force: nearest magnitude on the grid, ties to the
    even code, saturating, sign kept."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    a = min(abs(z), 6.0)
    d = np.abs(grid - a)
    best = np.flatnonzero(d == d.min())
    idx = int(best[0]) if best.size == 1 else int(best[best % 2 == 0][0])
    return (8 if math.copysign(1, z) < 0 else 0) | idx


def test_e2m1_encode_brute_force_sweep():
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (grid[1:] + grid[:-1]) / 2
    pts = [np.linspace(-8, 8, 4097)]
    for m in mids:
        for s in (1, -1):
            pts.append(s * np.array([m, np.nextafter(m, 0), np.nextafter(m, 10)]))
    z = np.concatenate(pts)
    got = oracle.e2m1_encode(z)
    want = np.array([_nearest_even_grid(float(v)) for v in z])
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ scale rule
def test_group_exponent_puts_amax_in_top_binade():
    rng = np.random.default_rng(3)
    for _ in range(2000):
        y = (rng.standard_normal(32) * 2.0 ** rng.integers(-40, 40)).astype(np.float32)
        e = oracle.group_exponent(y)
        amax = float(np.abs(y).max())
        assert 4.0 <= amax / 2.0 ** e < 8.0  # OCP MX: largest element maps into [4, 8)
    assert oracle.group_exponent(np.zeros(32, np.float32)) == -127
    assert oracle.group_exponent(np.full(32, 6.0, np.float32)) == 0
    assert oracle.group_exponent(np.full(32, 8.0, np.float32)) == 1
    assert oracle.group_exponent(np.full(32, np.nextafter(np.float32(8), np.float32(0)))) == 0
    assert oracle.group_exponent(np.full(32, 2.0 ** -130, np.float32)) == -127  # clamped
    assert oracle.group_exponent(np.full(32, 2.0 ** 126, np.float32)) == 124


def test_zero_vectors_quantise_to_plus_zero_codes():
    """An all-zero vector, of either sign, rotates to an exact zero: every group
    gets exponent -127 (scale byte 0) and every code is +0, since the exact
    matrix product of zeros has no sign (the sign bit is kept only for nonzero
    values that round to zero)."""
    for z in (0.0, -0.0):
        x = torch.full((1, 1, 128), z, dtype=torch.bfloat16)
        codes, expo, bad = oracle.quantize_vectors(x)
        assert bad == 0
        assert np.all(codes == 0) and np.all(expo == -127)
    # a nonzero negative value far below the group's scale rounds to -0 (code 0b1000)
    y = np.zeros(32, np.float32)
    y[0], y[1] = 4.0, -2.0 ** -10
    codes, expo = oracle.quantize_rotated(y)
    assert expo[0] == 0 and codes[0] == 0b0110 and codes[1] == 0b1000 and np.all(codes[2:] == 0)


def test_on_grid_groups_round_trip_exactly():
    rng = np.random.default_rng(11)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    for _ in range(200):
        k = int(rng.integers(-60, 60))
        mags = grid[rng.integers(0, 8, 32)]
        mags[rng.integers(0, 32)] = rng.choice([4.0, 6.0])  # max in the top binade
        vals = mags * rng.choice([-1.0, 1.0], 32)
        y = (vals * 2.0 ** k).astype(np.float32)
        codes, expo = oracle.quantize_rotated(y)
        assert expo[0] == k
        back = np.array([oracle.e2m1_decode(int(c)) for c in codes]) * 2.0 ** k
        assert np.array_equal(back, y.astype(np.float64))


def test_scaling_a_group_by_power_of_two_moves_only_the_exponent():
    rng = np.random.default_rng(5)
    y = rng.standard_normal(128).astype(np.float32)
    c0, e0 = oracle.quantize_rotated(y)
    for k in (-20, -3, 1, 7, 40):
        c1, e1 = oracle.quantize_rotated((y * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(c0, c1)
        assert np.array_equal(e1, e0 + k)


# ------------------------------------------------------------------ layout
def test_format_bytes_golden():
    g = {k: float(v) for k, v in _read_golden("format_bytes.txt")}
    for D in (64, 128, 256, 512):
        for P in (16, 32):
            bb = oracle.block_bytes(P, D)
            assert bb * g["group_values"] == g["bytes_per_group_4bit"] * P * D
    assert round(100 * (1 - g["bytes_per_group_4bit"] / g["bytes_per_group_8bit"])) == g["capacity_saving_pct"]
    assert round(g["bytes_per_group_8bit"] / g["bytes_per_group_4bit"], 2) == g["values_per_byte_ratio"]


def test_block_layout_positions():
    """Codes/scales land where the layout says: K in 8-token x 32-channel tiles
    of 128 bytes (16 bytes per token, low nibble = even channel), V
    channel-major low-nibble-even token, scales after the codes."""
    P, D, Hkv = 16, 128, 2
    bb = oracle.block_bytes(P, D)
    rng = np.random.default_rng(2)
    k = _bf16(rng.standard_normal((3, Hkv, D)))
    v = _bf16(rng.standard_normal((3, Hkv, D)))
    slots = np.array([5 * P + 6, 2 * P + 7, 2 * P + 0], dtype=np.int32)
    kc = np.zeros(8 * Hkv * bb, np.uint8)
    vc = np.zeros(8 * Hkv * bb, np.uint8)
    assert oracle.append_quantize(k, v, slots, kc, vc, 8, P) == oracle.OK
    kcodes, kexp, _ = oracle.quantize_vectors(k)
    vcodes, vexp, _ = oracle.quantize_vectors(v)
    for i, s in enumerate(slots):
        page, off = divmod(int(s), P)
        for h in range(Hkv):
            base = (page * Hkv + h) * bb
            for d in range(D):
                kb = kc[base + ((off // 8) * (D // 32) + d // 32) * 128 + (off % 8) * 16 + (d % 32) // 2]
                assert ((kb >> 4) if d & 1 else (kb & 15)) == kcodes[i, h, d]
                vb = vc[base + d * (P // 2) + off // 2]
                assert ((vb >> 4) if off & 1 else (vb & 15)) == vcodes[i, h, d]
            for g in range(D // 32):
                assert kc[base + P * D // 2 + off * (D // 32) + g] == kexp[i, h, g] + 127
                assert vc[base + P * D // 2 + off * (D // 32) + g] == vexp[i, h, g] + 127
    # untouched slots stay zero
    used = {(int(s) // P, int(s) % P) for s in slots}
    page, off = 1, 3
    assert (page, off) not in used
    assert not kc[(page * Hkv) * bb:(page * Hkv + 1) * bb].any()


def test_unpack_is_code_times_power_of_two():
    P, D = 16, 128
    rng = np.random.default_rng(9)
    k = _bf16(rng.standard_normal((1, 1, D)) * 3)
    kc = np.zeros(oracle.block_bytes(P, D), np.uint8)
    vc = np.zeros_like(kc)
    oracle.append_quantize(k, k, np.array([9], np.int32), kc, vc, 1, P)
    codes, expo, _ = oracle.quantize_vectors(k)
    want = np.array([oracle.e2m1_decode(int(c)) for c in codes[0, 0]]) * np.repeat(2.0 ** expo[0, 0], 32)
    assert np.array_equal(oracle.unpack_k_token(kc, P, D, 9), want)
    assert np.array_equal(oracle.unpack_v_token(vc, P, D, 9), want)


# ------------------------------------------------------------------ attention
def _np_attend(q, K, V, scale):
    s = scale * (K @ q)
    w = np.exp(s - s.max())
    w /= w.sum()
    return w @ V


def test_attend_row_brute_force_tiny():
    rng = np.random.default_rng(1)
    for n in (1, 2, 3, 4):
        for D in (4, 8):
            q, K, V = rng.standard_normal(D), rng.standard_normal((n, D)), rng.standard_normal((n, D))
            out, lse = oracle.attend_row(q, K, V, 0.7)
            assert np.allclose(out, _np_attend(q, K, V, 0.7), atol=1e-14)
            assert abs(lse - np.log(np.exp(0.7 * (K @ q)).sum())) < 1e-12


def test_attend_row_special_cases():
    rng = np.random.default_rng(4)
    D = 8
    q = rng.standard_normal(D)
    V = rng.standard_normal((5, D))
    out, _ = oracle.attend_row(q, V[:1] * 0 + rng.standard_normal(D), V[:1], 1.0)
    assert np.array_equal(out, V[0])                                  # one key: o = v
    K = np.tile(rng.standard_normal(D), (5, 1))
    out, _ = oracle.attend_row(q, K, V, 1.0)
    assert np.allclose(out, V.mean(0), atol=1e-14)                    # equal keys: mean
    K = rng.standard_normal((5, D))
    K[2] = 60 * q / np.linalg.norm(q)
    out, _ = oracle.attend_row(q, K, V, 1.0)
    assert np.allclose(out, V[2], atol=1e-12)                         # dominant logit


def _dense_from_cache(kc, vc, tables, lens, b, h, Hkv, P, D, latent):
    bb = oracle.block_bytes(P, D)
    L = int(lens[b])
    K = np.zeros((L, D))
    V = np.zeros((L, D))
    for t in range(L):
        page = int(tables[b, t // P])
        blk = kc[(page * Hkv + h) * bb:(page * Hkv + h + 1) * bb]
        K[t] = oracle.unpack_k_token(blk, P, D, t % P)
        if latent:
            V[t] = K[t]
        else:
            V[t] = oracle.unpack_v_token(vc[(page * Hkv + h) * bb:(page * Hkv + h + 1) * bb], P, D, t % P)
    return K, V


def _small_cache(rng, B, Hkv, D, P, lens, perm=True, extra_pages=3):
    pages_per = [(L + P - 1) // P for L in lens]
    num_pages = sum(pages_per) + extra_pages
    ids = rng.permutation(num_pages) if perm else np.arange(num_pages)
    tables = np.full((B, max(pages_per)), -1, np.int32)
    pos = 0
    for b in range(B):
        tables[b, :pages_per[b]] = ids[pos:pos + pages_per[b]]
        pos += pages_per[b]
    bb = oracle.block_bytes(P, D)
    kc = np.zeros(num_pages * Hkv * bb, np.uint8)
    vc = np.zeros_like(kc)
    kv = []
    for b in range(B):
        k = _bf16(rng.standard_normal((lens[b], Hkv, D)))
        v = _bf16(rng.standard_normal((lens[b], Hkv, D)))
        slots = np.array([tables[b, t // P] * P + t % P for t in range(lens[b])], np.int32)
        assert oracle.append_quantize(k, v, slots, kc, vc, num_pages, P) == oracle.OK
        kv.append((k, v))
    return tables, num_pages, kc, vc, kv


@pytest.mark.parametrize("T", [1, 3])
def test_decode_attention_equals_unrotated_attention_over_dequantised_cache(T):
    """Reading R2: scores in the rotated space equal scores in the original
    space; the output is rotated back.  Checked with scipy's Hadamard and
    plain numpy on the dequantised cache (rotated back into the input space)."""
    rng = np.random.default_rng(20 + T)
    B, Hkv, G, D, P = 2, 2, 3, 64, 16
    lens = [37, 50]
    tables, num_pages, kc, vc, _ = _small_cache(rng, B, Hkv, D, P, lens)
    q = _bf16(rng.standard_normal((B, T, Hkv * G, D)))
    scale = 0.125
    out = oracle.decode_attention(q, kc, vc, tables, np.array(lens, np.int32), Hkv, P, num_pages, scale)
    Hn = scipy.linalg.hadamard(D) / math.sqrt(D)
    for b in range(B):
        for h in range(Hkv):
            Kr, Vr = _dense_from_cache(kc, vc, tables, np.array(lens), b, h, Hkv, P, D, False)
            K0, V0 = Kr @ Hn, Vr @ Hn  # back to the input space (H symmetric)
            for j in range(T):
                n = lens[b] - T + 1 + j
                for g in range(G):
                    qv = q[b, j, h * G + g].float().numpy().astype(np.float64)
                    want = _np_attend(qv, K0[:n], V0[:n], scale)
                    assert np.allclose(out[b, j, h * G + g], want, atol=1e-10)


def test_decode_invariances_page_permutation_shared_prefix_and_verify():
    rng = np.random.default_rng(33)
    Hkv, G, D, P = 1, 4, 128, 16
    L = 70
    k = _bf16(rng.standard_normal((L, Hkv, D)))
    v = _bf16(rng.standard_normal((L, Hkv, D)))
    q = _bf16(rng.standard_normal((1, 3, G, D)))
    bb = oracle.block_bytes(P, D)
    npages = (L + P - 1) // P

    def run(page_ids, total_pages, qq, ctx, T):
        kc = np.zeros(total_pages * bb, np.uint8)
        vc = np.zeros_like(kc)
        slots = np.array([page_ids[t // P] * P + t % P for t in range(ctx)], np.int32)
        oracle.append_quantize(k[:ctx], v[:ctx], slots, kc, vc, total_pages, P)
        tab = np.array([page_ids], np.int32)
        return oracle.decode_attention(qq, kc, vc, tab, np.array([ctx], np.int32), Hkv, P, total_pages, 0.088)

    base = run(list(range(npages)), npages, q, L, 3)
    perm = run([7, 2, 9, 0, 4], 10, q, L, 3)
    assert np.array_equal(base, perm)  # physical placement is irrelevant
    # verify position j equals a single-query decode at context L - 3 + 1 + j
    for j in range(3):
        single = run(list(range(npages)), npages, q[:, j:j + 1], L - 2 + j, 1)
        assert np.array_equal(base[:, j], single[:, 0])
    # two sequences sharing their first 3 physical pages == each with its own copy
    kc = np.zeros(12 * bb, np.uint8)
    vc = np.zeros_like(kc)
    shared = [0, 1, 2]
    tabs = np.array([shared + [3, 4], shared + [5, 6]], np.int32)
    for b in range(2):
        lo = 0 if b == 0 else 3 * P
        slots = np.array([tabs[b, t // P] * P + t % P for t in range(lo, L)], np.int32)
        oracle.append_quantize(k[lo:L], v[lo:L], slots, kc, vc, 12, P)
    qq = torch.cat([q, q], 0)
    both = oracle.decode_attention(qq, kc, vc, tabs, np.array([L, L], np.int32), Hkv, P, 12, 0.088)
    assert np.array_equal(both[0], base[0]) and np.array_equal(both[1], base[0])


def test_latent_mode_uses_one_cache_for_k_and_v():
    rng = np.random.default_rng(8)
    Hkv, G, D, P, L = 1, 2, 512, 16, 40
    k = _bf16(rng.standard_normal((L, Hkv, D)))
    bb = oracle.block_bytes(P, D)
    kc = np.zeros(3 * bb, np.uint8)
    oracle.append_quantize(k, None, np.arange(L, dtype=np.int32), kc, None, 3, P)
    q = _bf16(rng.standard_normal((1, 1, G, D)))
    tab = np.array([[0, 1, 2]], np.int32)
    out = oracle.decode_attention(q, kc, None, tab, np.array([L], np.int32), Hkv, P, 3, 1 / math.sqrt(D),
                                  latent=True)
    Hn = scipy.linalg.hadamard(D) / math.sqrt(D)
    K = np.stack([oracle.unpack_k_token(kc[(t // P) * bb:(t // P + 1) * bb], P, D, t % P) for t in range(L)]) @ Hn
    for g in range(G):
        qv = q[0, 0, g].float().numpy().astype(np.float64)
        assert np.allclose(out[0, 0, g], _np_attend(qv, K, K, 1 / math.sqrt(D)), atol=1e-10)


# ------------------------------------------------------------------ FP8 comparator
def test_e4m3_decode_matches_torch_and_closed_forms():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[finite], ref[finite])
    assert ours[0x7E] == 448 and ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-4, 2.5, 20000),
                        oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)),
                        (oracle.e4m3_decode(np.arange(0x7E, dtype=np.uint8))
                         + oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))) / 2]).astype(np.float32)
    x = np.concatenate([x, -x])
    x = x[np.abs(x) <= 448]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    big = np.array([448.5, 463.9, 464.0, 1e6, -1e6], np.float32)
    assert list(oracle.e4m3_encode(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(finite).astype(np.float32)), finite)


def test_fp8_attention_brute_force():
    rng = np.random.default_rng(12)
    Hkv, G, D, P, L = 2, 2, 64, 16, 45
    k = _bf16(rng.standard_normal((L, Hkv, D)) * 3)
    v = _bf16(rng.standard_normal((L, Hkv, D)))
    kamax = k.float().abs().amax(dim=(0, 2)).numpy()
    vamax = v.float().abs().amax(dim=(0, 2)).numpy()
    ks, vs = (kamax / 448).astype(np.float32), (vamax / 448).astype(np.float32)
    kinv, vinv = (1 / ks.astype(np.float64)).astype(np.float32), (1 / vs.astype(np.float64)).astype(np.float32)
    num_pages = 4
    kc = np.zeros(num_pages * Hkv * P * D, np.uint8)
    vc = np.zeros_like(kc)
    page_ids = [3, 0, 2]
    slots = np.array([page_ids[t // P] * P + t % P for t in range(L)], np.int32)
    oracle.fp8_append(k, v, slots, kinv, vinv, kc, vc, num_pages, P)
    q = _bf16(rng.standard_normal((1, 1, Hkv * G, D)))
    out = oracle.fp8_decode_attention(q, kc, vc, ks, vs, np.array([page_ids], np.int32),
                                      np.array([L], np.int32), Hkv, P, num_pages, 0.125)
    for h in range(Hkv):
        kf = k[:, h].float().numpy() * kinv[h]
        vf = v[:, h].float().numpy() * vinv[h]
        kq = torch.from_numpy(kf).to(torch.float8_e4m3fn).double().numpy() * ks[h]
        vq = torch.from_numpy(vf).to(torch.float8_e4m3fn).double().numpy() * vs[h]
        for g in range(G):
            qv = q[0, 0, h * G + g].float().numpy().astype(np.float64)
            assert np.allclose(out[0, 0, h * G + g], _np_attend(qv, kq, vq, 0.125), atol=1e-12)
