"""Host logic of the bench's multi-rank (replica) mode, on CPU with gloo.

Each rank simulates its own sequences with the bench's Trajectory, using the
trajectory's own expected outcome in place of the device's (the device path is
covered by the GPU parity tests).  Checked here: the ranks' pages and start
ids are disjoint, the committed-token count follows the page cap, and the
whole-job reduction takes the slowest rank's times and every rank's tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from moe_speculative_decoding_router_gb300 import synth as S

V, B, K, PAGE, STEPS = 512, 8, 3, 20, 30


def _table():
    return S.uniform_ids(V, 99, 7, V).astype(np.int64)


def _simulate(rank):
    g = _table()
    tr = bench.Trajectory(g, rank, B=B, K=K, p=0.75, page_tokens=PAGE)
    pages, verify, counted = set(tr.page_id.tolist()), [], 0
    for _ in range(STEPS):
        ctx_ids, drafts = tr.drafts()
        verify.append(np.concatenate([ctx_ids[:, None], drafts], axis=1))
        com, alen = tr.expected(ctx_ids, drafts)
        counted += tr.advance(com, alen)
        pages.update(tr.page_id.tolist())
    return pages, np.stack(verify), counted


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    pages, verify, counted = _simulate(rank)
    ms, e_s = 10.0 + rank, 20.0 - rank
    red = bench.whole_job(ms, e_s, float(counted), float(counted + rank), "cpu")
    dist.barrier()
    dist.destroy_process_group()
    np.savez(os.path.join(out_dir, f"r{rank}.npz"), pages=np.array(sorted(pages)),
             verify=verify, counted=counted, red=np.array(red))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_trajectory_counts_and_pages():
    g = _table()
    tr = bench.Trajectory(g, 0, B=B, K=K, p=1.0, page_tokens=PAGE)
    total = 0
    for step in range(12):
        ctx_ids, drafts = tr.drafts()
        # p = 1: every draft is the greedy chain of the last committed token
        x = ctx_ids.astype(np.int64)
        for j in range(K):
            x = g[x]
            assert np.array_equal(drafts[:, j], x)
        com, alen = tr.expected(ctx_ids, drafts)
        assert np.all(alen == K)
        total += tr.advance(com, alen)
    # pages of 20 tokens at 4 per step: 5 steps fill a page exactly
    assert total == 12 * B * (K + 1)
    assert tr.next_page == B + 2 * B


def test_draft_batch_equals_per_sequence():
    """The batched draft draws are the per-sequence draws (same counters)."""
    src = S.DraftSource(0.6, V, K)
    rng = np.random.default_rng(5)
    seqs = rng.integers(0, 3_000_000, 50)
    steps = rng.integers(0, 500, 50)
    truth = rng.integers(0, V, (50, K))
    a = src.drafts_batch(seqs, steps, truth)
    b = np.stack([src.drafts(int(seqs[i]), int(steps[i]), truth[i]) for i in range(50)])
    assert np.array_equal(a, b)
    assert 0 < np.mean(a == truth) < 1


def test_expected_commits_follow_the_prefix_rule():
    g = _table()
    tr = bench.Trajectory(g, 0, B=B, K=K, p=0.5, page_tokens=PAGE)
    for _ in range(6):
        ctx_ids, drafts = tr.drafts()
        com, n = tr.expected(ctx_ids, drafts)
        y = g[np.concatenate([ctx_ids[:, None], drafts], axis=1)]
        for b in range(B):
            m = 0
            while m < K and drafts[b, m] == y[b, m]:
                m += 1
            assert n[b] == m
            assert list(com[b, : m + 1]) == list(y[b, : m + 1])
            assert all(com[b, m + 1:] == -1)
        tr.advance(com, n)


def test_two_rank_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r = [np.load(tmp_path / f"r{i}.npz") for i in range(world)]
    # disjoint pages and different sequences on the two ranks
    assert not set(r[0]["pages"].tolist()) & set(r[1]["pages"].tolist())
    assert not np.array_equal(r[0]["verify"][0], r[1]["verify"][0])
    # each rank's own simulation is what a single process gets
    for i in range(world):
        pages, verify, counted = _simulate(i)
        assert np.array_equal(verify, r[i]["verify"])
        assert counted == int(r[i]["counted"])
    # whole job: max of the times, sum of the tokens, same on every rank
    c0, c1 = int(r[0]["counted"]), int(r[1]["counted"])
    want = np.array([11.0, 20.0, c0 + c1, c0 + c1 + 1])
    for i in range(world):
        assert np.array_equal(r[i]["red"], want)


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
