"""Host logic of one long context split across devices ("GLM-5.3-Flash on
MI300X": a sharded, not replicated, KV cache), on CPU.

share_ranges cuts each sequence into consecutive page-aligned shares with the
newest tokens in the last one; two gloo ranks each compute their share's
partial attention (the oracle's fp64 attention over the share's tokens, with
the visibility rule of kv4_decode_partials on the newest share and of
kv4_decode_partials_prefix on the others), gather_partials brings them to rank
0, and the log-sum-exp merge of the gathered partials must equal the oracle's
attention over the whole sequence.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_kv_cache_rotate_b300 import seqsplit

P = 16


def test_shares_cover_each_sequence_in_order():
    lens = np.array([3, 16, 17, 100, 1000, 4099], dtype=np.int64)
    for T in (1, 3, 6):
        for W in (1, 2, 3, 5):
            r = seqsplit.share_ranges(np.maximum(lens, T), T, W, P)
            L = np.maximum(lens, T)
            assert r.shape == (W, lens.size, 2)
            assert (r[0, :, 0] == 0).all() and (r[W - 1, :, 1] == L).all()
            assert (r[1:, :, 0] == r[:-1, :, 1]).all()                # consecutive
            assert (r[:, :, 1] >= r[:, :, 0]).all()                    # possibly empty
            assert (r[:-1, :, :] % P == 0).all() and (r[W - 1, :, 0] % P == 0).all()  # page-aligned cuts
            assert (r[W - 1, :, 1] - r[W - 1, :, 0] >= T).all()        # the newest tokens in the last share
    # long sequences are divided about evenly by pages
    r = seqsplit.share_ranges(np.array([32768]), 1, 4, P)
    sizes = r[:, 0, 1] - r[:, 0, 0]
    assert sizes.max() - sizes.min() <= P
    with pytest.raises(ValueError):
        seqsplit.share_ranges(np.array([2]), 3, 2, P)


def test_local_tables_hold_the_share_pages():
    tables = np.arange(4 * 10, dtype=np.int32).reshape(4, 10) * 7
    lens = np.array([160, 33, 1, 100])
    r = seqsplit.share_ranges(lens, 1, 2, P)
    for w in range(2):
        tab, ll = seqsplit.local_tables(tables, r[w], P)
        for b in range(4):
            p0 = r[w, b, 0] // P
            n = (ll[b] + P - 1) // P
            assert (tab[b, :n] == tables[b, p0:p0 + n]).all()
            assert ll[b] == r[w, b, 1] - r[w, b, 0]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(seed=7, B=3, T=3, Hq=4, D=16):
    rng = np.random.default_rng(seed)
    lens = np.array([T + 5, 200, 611])[:B]
    K = [rng.standard_normal((L, D)) for L in lens]
    V = [rng.standard_normal((L, D)) for L in lens]
    q = rng.standard_normal((B, T, Hq, D))
    return lens, K, V, q


def _share_partials(rank, world, lens, K, V, q, scale):
    """This rank's partial (O, lse) per (b, j, hq): fp64 attention over its share."""
    import oracle
    B, T, Hq, D = q.shape
    r = seqsplit.share_ranges(lens, T, world, P)[rank]
    newest = rank == world - 1
    po = np.zeros((B, T, Hq, 1, D))
    pl = np.full((B, T, Hq, 1), -np.inf)
    for b in range(B):
        t0, t1 = int(r[b, 0]), int(r[b, 1])
        for j in range(T):
            # kv4_decode_partials on the newest share: causal among the T new tokens;
            # kv4_decode_partials_prefix elsewhere: every token of the share visible
            hi = (t1 - T + 1 + j) if newest else t1
            n = max(0, hi - t0)
            for h in range(Hq):
                if n == 0:
                    continue
                o, lse = oracle.attend_row(q[b, j, h], np.ascontiguousarray(K[b][t0:t0 + n]),
                                           np.ascontiguousarray(V[b][t0:t0 + n]), scale)
                po[b, j, h, 0] = o
                pl[b, j, h, 0] = lse
    return po, pl


def _worker(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lens, K, V, q = _problem()
        po, pl = _share_partials(rank, world, lens, K, V, q, 0.25)
        go, gl = seqsplit.gather_partials(torch.from_numpy(po), torch.from_numpy(pl))
        if rank == 0:
            np.savez(out_path, po=go.numpy(), pl=gl.numpy())
        else:
            assert go is None and gl is None
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gathered_shares_merge_to_the_whole_attention(world, tmp_path):
    import oracle
    out_path = str(tmp_path / "gathered.npz")
    mp.spawn(_worker, args=(world, _free_port(), out_path), nprocs=world, join=True)
    got = np.load(out_path)
    po, pl = got["po"], got["pl"]
    lens, K, V, q = _problem()
    B, T, Hq, D = q.shape
    assert po.shape == (B, T, Hq, world, D) and pl.shape == (B, T, Hq, world)
    # the log-sum-exp merge that kv4_split_combine performs, in fp64
    m = pl.max(axis=3, keepdims=True)
    w = np.where(np.isfinite(pl), np.exp(pl - m), 0.0)
    merged = (w[..., None] * po).sum(axis=3) / w.sum(axis=3)[..., None]
    for b in range(B):
        for j in range(T):
            n = int(lens[b]) - T + 1 + j
            for h in range(Hq):
                ref, _ = oracle.attend_row(q[b, j, h], np.ascontiguousarray(K[b][:n]),
                                           np.ascontiguousarray(V[b][:n]), 0.25)
                assert np.abs(merged[b, j, h] - ref).max() < 1e-12
