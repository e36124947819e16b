"""Multi-rank paths on CPU (gloo, world_size 2), with the CPU oracle standing in for each rank's GPU.

1. Request sharding (the N-GPU configuration of the decode step): each rank computes its own
   requests; the gathered result equals the single-process result on the whole batch, and the
   timing reduction takes the slowest rank.
2. The one-exchange variant for a single very long request (keys sharded by token range): each rank
   scores its key range and keeps a local top-k of (value, index) pairs; one all-gather of the
   candidates and a merge give the global top-k; each rank attends over the selected keys it owns
   and one more all-gather plus a log-sum-exp merge gives the attention output.  Both equal the
   unsharded computation.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)


def _oracle_chain(wl, pool, rows):
    import oracle
    lg = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q, rows,
                               wl.max_seq_len)
    idx = oracle.topk(lg, wl.seq_lens, wl.cu_q, rows, wl.topk)
    full = np.full((wl.T, wl.topk), -1, np.int32)
    full[rows] = idx
    out, lse = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, full, wl.scale,
                                 rows)
    return idx, out, lse


def _small_workload():
    from deepseek_sparse_attention_paged_gb300 import workloads
    return workloads.make_custom("shard", 77, [300, 520, 129, 1000, 64], 1, topk=128, heads=16)


def _build_pool(wl):
    import oracle
    pool = np.zeros((wl.num_pages, oracle.PAGE_BYTES), np.uint8)
    oracle.store_index_k(wl.index_keys(), wl.token_slots(), pool)
    return pool


def _worker_request_sharding(rank, port, result):
    _init(rank, port)
    try:
        from deepseek_sparse_attention_paged_gb300 import distributed as D
        wl = _small_workload()
        pool = _build_pool(wl)
        mine = D.shard_requests(wl.B, rank, WORLD)
        rows = np.concatenate([np.arange(wl.cu_q[b], wl.cu_q[b + 1]) for b in mine]).astype(np.int64)
        idx, out, lse = _oracle_chain(wl, pool, rows)
        payload = [None] * WORLD
        dist.all_gather_object(payload, (rows, idx, out, lse))
        slowest = D.max_over_ranks(float(rank + 1))
        if rank == 0:
            result["gathered"] = payload
            result["slowest"] = slowest
    finally:
        dist.destroy_process_group()


def test_request_sharding_matches_whole_batch():
    from deepseek_sparse_attention_paged_gb300 import distributed as D
    assert D.shard_requests(5, 0, 2) == [0, 1, 2] and D.shard_requests(5, 1, 2) == [3, 4]
    assert sorted(sum((D.shard_requests(7, r, 3) for r in range(3)), [])) == list(range(7))
    port = _free_port()
    mgr = mp.Manager()
    result = mgr.dict()
    mp.spawn(_worker_request_sharding, args=(port, result), nprocs=WORLD, join=True)
    wl = _small_workload()
    pool = _build_pool(wl)
    all_rows = np.arange(wl.T)
    idx, out, lse = _oracle_chain(wl, pool, all_rows)
    got_idx = np.zeros_like(idx)
    got_out = np.zeros_like(out)
    got_lse = np.zeros_like(lse)
    for rows, i, o, l in result["gathered"]:
        got_idx[rows] = i
        got_out[rows] = o
        got_lse[rows] = l
    assert np.array_equal(got_idx, idx)
    assert np.array_equal(got_out, out) and np.array_equal(got_lse, lse)
    assert result["slowest"] == float(WORLD)
    assert D.aggregate_rate(64, 2, 1.0) == 128000.0


# ------------------------------------------------------------------ one-exchange variant

def _long_request():
    from deepseek_sparse_attention_paged_gb300 import workloads
    return workloads.make_custom("long", 78, [3000], 1, topk=256, heads=16)


def _worker_exchange(rank, port, result):
    _init(rank, port)
    try:
        import oracle
        wl = _long_request()
        pool = _build_pool(wl)
        v = int(wl.visible_lens()[0])
        lg = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                                   np.array([0]), wl.max_seq_len)[0, :v]
        lo, hi = rank * v // WORLD, (rank + 1) * v // WORLD          # this rank's token range
        # local top-k over the owned range (values and global indices)
        order = np.argsort(-lg[lo:hi], kind="stable")[:wl.topk] + lo
        cand = (lg[order].astype(np.float32), order.astype(np.int64))
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, cand)
        vals = np.concatenate([g[0] for g in gathered])
        inds = np.concatenate([g[1] for g in gathered])
        # merge: larger value first, lower index on ties (the stable order of the whole row)
        merged = np.lexsort((inds, -vals.astype(np.float64)))[:wl.topk]
        sel = np.sort(inds[merged])
        # attention over the selected keys this rank owns, then an exchange of (o, lse)
        mine = sel[(sel >= lo) & (sel < hi)]
        idx = np.full((1, wl.topk), -1, np.int32)
        idx[0, :mine.size] = mine
        o, l = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, idx, wl.scale,
                                 np.array([0]))
        parts = [None] * WORLD
        dist.all_gather_object(parts, (o, l))
        om, lm = parts[0]
        for o2, l2 in parts[1:]:
            om, lm = oracle.lse_merge(om, lm, o2, l2)
        if rank == 0:
            result["sel"] = sel
            result["out"] = om
            result["lse"] = lm
    finally:
        dist.destroy_process_group()


def test_token_range_exchange_matches_unsharded():
    import oracle
    port = _free_port()
    mgr = mp.Manager()
    result = mgr.dict()
    mp.spawn(_worker_exchange, args=(port, result), nprocs=WORLD, join=True)
    wl = _long_request()
    pool = _build_pool(wl)
    idx, out, lse = _oracle_chain(wl, pool, np.array([0]))
    assert np.array_equal(result["sel"], idx[0][idx[0] >= 0])
    assert np.allclose(result["out"], out, rtol=1e-12, atol=1e-14)
    assert np.allclose(result["lse"], lse, rtol=1e-12)
