"""Parity at the benchmarks' full size in the launch configuration bench.py
times: the whole cache is built and one bench step (append of the new tokens +
decode with the automatic split count) runs on the GPU; sampled (sequence, kv
head) pairs are recomputed one by one by the oracle -- every cached K/V block
of the sample bit-exact, its attention rows within 2e-3.  Workloads covered:
batch 32 at a 32K context (4-bit path and the FP8 comparator on the same
inputs), at 16K, and at 8K (there every K and V vector of the cache is
checked, not a sample), the 512-wide MLA latent cache at batch 8 and a 96K context, the
3-position verify step over ragged 16K-128K contexts with a 93 % shared prefix
(every token the step appends checked bit-exact),
and the extend step (batch 4, a 512-token chunk over a 32K context) on both
extend kernels at sampled chunk positions."""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_rotate_b300 import workloads as W
from _harness import TOL

pytestmark = pytest.mark.gpu

kv4 = pytest.importorskip("bit_kv_cache_rotate_b300")

SAMPLES = [(0, 3), (17, 6), (31, 0)]  # (sequence, kv head)


@pytest.fixture(scope="module")
def fullsize():
    import bench
    cfg = W.CONFIGS["b32_ctx32k"]
    wl = bench.Workload(cfg, kv4, with_fp8=True)
    kv4.kv4_append_quantize(wl.new_k, wl.new_v, wl.new_slots, wl.kc, wl.vc, wl.lay.num_pages)
    out = kv4.kv4_decode_attention(wl.q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, wl.lay.num_pages,
                                   cfg.softmax_scale, num_splits=wl.S, workspace_buf=wl.ws)
    f = wl.fp8
    kv4.fp8_append_quantize(wl.new_k, wl.new_v, wl.new_slots, f["k_inv"], f["v_inv"], f["kc"], f["vc"],
                            wl.lay.num_pages)
    out8 = kv4.fp8_decode_attention(wl.q, f["kc"], f["vc"], f["k_scale"], f["v_scale"], wl.tab, wl.lens,
                                    cfg.num_kv_heads, wl.lay.num_pages, cfg.softmax_scale, num_splits=wl.S,
                                    workspace_buf=f["ws"])
    torch.cuda.synchronize()
    return cfg, wl, out.cpu().numpy().astype(np.float64), out8.cpu().numpy().astype(np.float64)


def _gpu_blocks(cache, lay, b, h, n_pages, num_kv_heads, bb):
    """Sequence b's cache blocks of kv head h, page by page, as the GPU wrote them."""
    phys = lay.block_tables[b, :n_pages].astype(np.int64)
    idx = ((phys * num_kv_heads + h) * bb)[:, None] + np.arange(bb)[None, :]
    return cache[torch.from_numpy(idx.reshape(-1)).cuda()].cpu().numpy()


def _written_bits(k, v, L, P, bb):
    """Bit mask of the bytes a sequence's tokens write into its blocks.  The
    cache memory is not initialised, so in a partly filled last page the
    slots past the context hold whatever was there.  Appending the last
    page's tokens into two oracle blocks that start as all-zero and all-one
    bits leaves exactly the unwritten bits different; the result is None
    when every page is full."""
    n_full, n_last = divmod(L, P)
    if n_last == 0:
        return None
    lo = n_full * P
    kl = k[lo:L].contiguous()
    vl = None if v is None else v[lo:L].contiguous()
    blocks = []
    for fill in (0x00, 0xFF):
        kb = np.full(bb, fill, np.uint8)
        vb = None if v is None else np.full(bb, fill, np.uint8)
        assert oracle.append_quantize(kl, vl, np.arange(n_last, dtype=np.int32), kb, vb, 1, P) == oracle.OK
        blocks.append((kb, vb))
    (k0, v0), (k1, v1) = blocks
    return n_full * bb, ~(k0 ^ k1), None if v is None else ~(v0 ^ v1)


def _same_written(gpu, ref, written, part):
    """Blocks equal on every written bit: all bits of the full pages, the
    masked bits of the last one (part 1 = K or latent, 2 = V)."""
    if written is None:
        return np.array_equal(gpu, ref)
    start, mask = written[0], written[part]
    return (np.array_equal(gpu[:start], ref[:start])
            and not np.any((gpu[start:] ^ ref[start:]) & mask))


def _check_sample(cfg, wl, out, b, h, chain=None):
    """Oracle cache and attention for one (sequence, kv head), built from the
    sequence's own tokens at logical slots 0..L-1, against the GPU's blocks
    (found through the page table) and output rows."""
    lay, P, D, G = wl.lay, cfg.page_size, cfg.head_dim, cfg.group
    L = int(lay.context_lens[b])
    n_pages = (L + P - 1) // P
    k, v = W.sequence_tokens(cfg, lay, b, chain_cache=chain)
    k = k[:, h:h + 1].contiguous()
    v = None if v is None else v[:, h:h + 1].contiguous()
    bb = oracle.block_bytes(P, D)
    okc = np.zeros(n_pages * bb, np.uint8)
    ovc = None if cfg.latent else np.zeros_like(okc)
    assert oracle.append_quantize(k, v, np.arange(L, dtype=np.int32), okc, ovc, n_pages, P) == oracle.OK
    written = _written_bits(k, v, L, P, bb)
    assert _same_written(_gpu_blocks(wl.kc, lay, b, h, n_pages, cfg.num_kv_heads, bb), okc, written, 1), \
        "K blocks differ from the oracle"
    if not cfg.latent:
        assert _same_written(_gpu_blocks(wl.vc, lay, b, h, n_pages, cfg.num_kv_heads, bb), ovc, written, 2), \
            "V blocks differ from the oracle"
    q = W.queries(cfg)[b:b + 1, :, h * G:(h + 1) * G].contiguous()
    ref = oracle.decode_attention(q, okc, ovc, np.arange(n_pages, dtype=np.int32)[None, :],
                                  np.array([L], dtype=np.int32), 1, P, n_pages, cfg.softmax_scale,
                                  latent=cfg.latent)
    got = out[b:b + 1, :, h * G:(h + 1) * G]
    err = np.abs(got - ref).max()
    assert err <= TOL, f"sequence {b}, kv head {h}: max abs error {err:.3e}"


@pytest.mark.parametrize("b,h", SAMPLES)
def test_fullsize_sampled_parity(fullsize, b, h):
    cfg, wl, out, _ = fullsize
    _check_sample(cfg, wl, out, b, h)


@pytest.mark.parametrize("b,h", SAMPLES[:2])
def test_fullsize_fp8_comparator_sampled_parity(fullsize, b, h):
    """The FP8 comparator on the same inputs: its E4M3 blocks bit-exact against
    the oracle's encoder under the same per-head scales, attention within 2e-3."""
    cfg, wl, _, out8 = fullsize
    lay, P, D, G, f = wl.lay, cfg.page_size, cfg.head_dim, cfg.group, wl.fp8
    L = int(lay.context_lens[b])
    n_pages = (L + P - 1) // P
    k, v = W.sequence_tokens(cfg, lay, b)
    k = k[:, h:h + 1].contiguous()
    v = v[:, h:h + 1].contiguous()
    fbb = P * D
    okc = np.zeros(n_pages * fbb, np.uint8)
    ovc = np.zeros_like(okc)
    k_inv, v_inv = f["k_inv"].cpu().numpy()[h:h + 1], f["v_inv"].cpu().numpy()[h:h + 1]
    k_sc, v_sc = f["k_scale"].cpu().numpy()[h:h + 1], f["v_scale"].cpu().numpy()[h:h + 1]
    assert oracle.fp8_append(k, v, np.arange(L, dtype=np.int32), k_inv, v_inv, okc, ovc, n_pages, P) == oracle.OK
    assert np.array_equal(_gpu_blocks(f["kc"], lay, b, h, n_pages, cfg.num_kv_heads, fbb), okc), \
        "FP8 K blocks differ from the oracle"
    assert np.array_equal(_gpu_blocks(f["vc"], lay, b, h, n_pages, cfg.num_kv_heads, fbb), ovc), \
        "FP8 V blocks differ from the oracle"
    q = W.queries(cfg)[b:b + 1, :, h * G:(h + 1) * G].contiguous()
    ref = oracle.fp8_decode_attention(q, okc, ovc, k_sc, v_sc, np.arange(n_pages, dtype=np.int32)[None, :],
                                      np.array([L], dtype=np.int32), 1, P, n_pages, cfg.softmax_scale)
    err = np.abs(out8[b:b + 1, :, h * G:(h + 1) * G] - ref).max()
    assert err <= TOL, f"max abs error {err:.3e}"


def _bench_step(name):
    import bench
    cfg = W.CONFIGS[name]
    wl = bench.Workload(cfg, kv4, with_fp8=False)
    kv4.kv4_append_quantize(wl.new_k, wl.new_v, wl.new_slots, wl.kc, wl.vc, wl.lay.num_pages)
    out = kv4.kv4_decode_attention(wl.q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, wl.lay.num_pages,
                                   cfg.softmax_scale, num_splits=wl.S, workspace_buf=wl.ws)
    torch.cuda.synchronize()
    return cfg, wl, out.cpu().numpy().astype(np.float64)


# ---- batch 32 at an 8K context (the same kernel, a quarter of the tokens per split)
@pytest.fixture(scope="module")
def fullsize_8k():
    return _bench_step("b32_ctx8k")


@pytest.mark.parametrize("b,h", [(5, 1), (30, 7)])
def test_fullsize_8k_sampled_parity(fullsize_8k, b, h):
    cfg, wl, out = fullsize_8k
    _check_sample(cfg, wl, out, b, h)


def test_fullsize_8k_every_vector_bit_exact(fullsize_8k):
    """Every K and V vector of the 8K step (32 sequences x 8192 tokens x 8 kv
    heads, the step's appended tokens included): the whole GPU cache equal to
    the oracle's, byte for byte.  Every page of this workload is full, so
    every byte of both caches is written."""
    from _harness import all_tokens, oracle_caches
    cfg, wl, _ = fullsize_8k
    lay = wl.lay
    assert (lay.context_lens % cfg.page_size == 0).all()
    k, v, slots = all_tokens(cfg, lay)
    okc, ovc = oracle_caches(cfg, lay, k, v, slots)
    for name, g, o in (("K", wl.kc, okc), ("V", wl.vc, ovc)):
        diff = np.flatnonzero(g.cpu().numpy() != o)
        assert diff.size == 0, f"{name} cache differs at {diff[:8]} ({diff.size} bytes)"


# ---- batch 32 at a 16K context: the middle of the context sweep
@pytest.fixture(scope="module")
def fullsize_16k():
    return _bench_step("b32_ctx16k")


@pytest.mark.parametrize("b,h", [(2, 4), (19, 0), (31, 7)])
def test_fullsize_16k_sampled_parity(fullsize_16k, b, h):
    cfg, wl, out = fullsize_16k
    _check_sample(cfg, wl, out, b, h)


# ---- MLA latent cache at full size: batch 8, a 98304-token context, one 512-wide latent head
@pytest.fixture(scope="module")
def fullsize_mla():
    return _bench_step("mla_b8_ctx96k")


@pytest.mark.parametrize("b", [0, 5])
def test_fullsize_mla_sampled_parity(fullsize_mla, b):
    cfg, wl, out = fullsize_mla
    _check_sample(cfg, wl, out, b, 0)


# ---- verify step at full size: batch 32, ragged 16K-128K contexts, 93 % shared prefix, T = 3
@pytest.fixture(scope="module")
def fullsize_verify():
    cfg, wl, out = _bench_step("verify_agentic")
    chain = W.chain_tokens(cfg, wl.lay, 0, int(wl.lay.chain.size) * cfg.page_size)
    return cfg, wl, out, chain


def _verify_samples():
    lay = W.make_layout(W.CONFIGS["verify_agentic"])
    lens = lay.context_lens
    return [(int(np.argmax(lens)), 7), (int(np.argmin(lens)), 2), (13, 4)]


def test_fullsize_verify_every_new_token_bit_exact(fullsize_verify):
    """Every token the verify step appends (3 per sequence, 32 sequences, 8 kv
    heads, K and V): the bits each one writes into its page equal the oracle's.
    The written bits are found by appending the page's new tokens into two
    oracle blocks that start all-zero and all-one."""
    cfg, wl, _, _ = fullsize_verify
    lay, P, D, T, Hkv = wl.lay, cfg.page_size, cfg.head_dim, cfg.q_per_seq, cfg.num_kv_heads
    bb = oracle.block_bytes(P, D)
    gk, gv = wl.kc.cpu().numpy(), wl.vc.cpu().numpy()
    checked = 0
    for b in range(cfg.batch):
        L = int(lay.context_lens[b])
        k, v = W.private_tokens(cfg, lay, b)
        k, v = k[-T:], v[-T:]
        pos = np.arange(L - T, L)
        for page_idx in np.unique(pos // P):
            sel = np.flatnonzero(pos // P == page_idx)
            phys = int(lay.block_tables[b, page_idx])
            for h in range(Hkv):
                kh = k[sel, h:h + 1].contiguous()
                vh = v[sel, h:h + 1].contiguous()
                offs = (pos[sel] % P).astype(np.int32)
                blk = []
                for fill in (0x00, 0xFF):
                    kb = np.full(bb, fill, np.uint8)
                    vb = np.full(bb, fill, np.uint8)
                    assert oracle.append_quantize(kh, vh, offs, kb, vb, 1, P) == oracle.OK
                    blk.append((kb, vb))
                (k0, v0), (k1, v1) = blk
                base = (phys * Hkv + h) * bb
                for g, o0, o1, part in ((gk, k0, k1, "K"), (gv, v0, v1, "V")):
                    mask = ~(o0 ^ o1)  # the bits the new tokens write
                    assert not np.any((g[base:base + bb] ^ o0) & mask), \
                        f"sequence {b}, kv head {h}, page {page_idx}: {part} bits of the new tokens differ"
                checked += len(sel)
    assert checked == cfg.batch * T * Hkv


@pytest.mark.parametrize("b,h", _verify_samples())
def test_fullsize_verify_sampled_parity(fullsize_verify, b, h):
    """The shortest and the longest sequence plus one more: their shared-prefix
    pages (written once, reached through several page tables) and private pages
    bit-exact, the three causal verify rows of each query head within 2e-3."""
    cfg, wl, out, chain = fullsize_verify
    _check_sample(cfg, wl, out, b, h, chain=chain)


# ---- 6-position verify at full size: the same traffic with T = 6 (48 rows per kv head)
@pytest.fixture(scope="module")
def fullsize_verify6():
    cfg, wl, out = _bench_step("verify6_agentic")
    chain = W.chain_tokens(cfg, wl.lay, 0, int(wl.lay.chain.size) * cfg.page_size)
    return cfg, wl, out, chain


def _verify6_samples():
    lens = W.make_layout(W.CONFIGS["verify6_agentic"]).context_lens
    return [(int(np.argmax(lens)), 3), (int(np.argmin(lens)), 6)]


@pytest.mark.parametrize("b,h", _verify6_samples())
def test_fullsize_verify6_sampled_parity(fullsize_verify6, b, h):
    cfg, wl, out, chain = fullsize_verify6
    _check_sample(cfg, wl, out, b, h, chain=chain)


# ---- extend step at full size: batch 4, a 512-token chunk over a 32K context
EXT_SAMPLES = [(0, 5, (0, 300, 511)), (3, 2, (17, 511))]  # (sequence, kv head, positions)


@pytest.fixture(scope="module", params=["tcgen05", "warp"])
def fullsize_extend(request):
    import bench
    kernel = kv4.KV4_KERNEL_WARP_MMA if request.param == "warp" else kv4.KV4_KERNEL_AUTO
    cfg = W.CONFIGS["extend_b4_ctx32k_t512"]
    wl = bench.Workload(cfg, kv4, with_fp8=False)
    kv4.kv4_append_quantize(wl.new_k, wl.new_v, wl.new_slots, wl.kc, wl.vc, wl.lay.num_pages)
    out = kv4.kv4_decode_attention_select(wl.q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, wl.lay.num_pages,
                                          cfg.softmax_scale, kernel, num_splits=wl.S, workspace_buf=wl.ws)
    torch.cuda.synchronize()
    return cfg, wl, out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("b,h,positions", EXT_SAMPLES)
def test_fullsize_extend_sampled_parity(fullsize_extend, b, h, positions):
    """Position j of the chunk equals a single-query decode over the first
    L - T + 1 + j tokens, computed by the oracle from its own cache."""
    cfg, wl, out = fullsize_extend
    lay, P, D, G, T = wl.lay, cfg.page_size, cfg.head_dim, cfg.group, cfg.q_per_seq
    L = int(lay.context_lens[b])
    n_pages = (L + P - 1) // P
    k, v = W.sequence_tokens(cfg, lay, b)
    k = k[:, h:h + 1].contiguous()
    v = v[:, h:h + 1].contiguous()
    bb = oracle.block_bytes(P, D)
    okc = np.zeros(n_pages * bb, np.uint8)
    ovc = np.zeros_like(okc)
    assert oracle.append_quantize(k, v, np.arange(L, dtype=np.int32), okc, ovc, n_pages, P) == oracle.OK
    q_all = W.queries(cfg)
    for j in positions:
        q = q_all[b:b + 1, j:j + 1, h * G:(h + 1) * G].contiguous()
        ref = oracle.decode_attention(q, okc, ovc, np.arange(n_pages, dtype=np.int32)[None, :],
                                      np.array([L - T + 1 + j], dtype=np.int32), 1, P, n_pages, cfg.softmax_scale)
        got = out[b:b + 1, j:j + 1, h * G:(h + 1) * G]
        err = np.abs(got - ref).max()
        assert err <= TOL, f"position {j}: max abs error {err:.3e}"
