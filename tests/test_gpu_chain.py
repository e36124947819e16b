"""End-to-end GPU parity of one decode step (store -> logits -> top-k -> sparse MLA) against the
CPU oracle, in the launch configuration the benchmark times (the same DeviceBatch.step() calls,
row-tiled logits included): the whole tiny workload; every row of the 32 x 8K, 64-request 64K and
MTP 128K decode batches; every 64th row (and the last) of the 4096-row prefill chunk; and the whole
index-K cache of every workload byte for byte."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

from helpers import (bf16_to_np_f64, check_attention, check_logits, check_topk_valid, kth_gap_ok,
                     oracle_pool, record)

pytestmark = pytest.mark.gpu


def run_step_capturing_logits(db, rows):
    """One step; the logits of `rows` are copied out of each logits tile right after its indexer
    call (the tile buffer is reused by the next tile).  Returns them as a host array [n, ld]."""
    rows = np.asarray(rows, np.int64)
    got = torch.empty((len(rows), db.ld), dtype=torch.float32, device=db.device)
    pos = {int(r): i for i, r in enumerate(rows)}

    def hook(rb, re, lg):
        sel = [r for r in range(rb, re) if r in pos]
        if sel:
            dst = torch.tensor([pos[r] for r in sel], device=db.device)
            src = torch.tensor([r - rb for r in sel], device=db.device)
            got[dst] = lg[src]

    db.step(logits_hook=hook)
    torch.cuda.synchronize()
    return got.cpu().numpy()


def check_rows(wl, db, rows, pool, got_lg, key):
    rows = np.asarray(rows, np.int64)
    vis = wl.visible_lens()[rows]
    ld = db.ld
    ref_lg, mag, bad = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens,
                                             wl.cu_q, rows, ld, want_mag=True)
    assert bad == 0
    check_logits(got_lg, ref_lg, mag, vis, key=key)
    # top-k: GPU indices from GPU logits vs oracle indices from oracle logits
    ref_idx = oracle.topk(ref_lg, wl.seq_lens, wl.cu_q, rows, wl.topk)
    got_idx = db.idx[torch.from_numpy(rows).cuda()].cpu().numpy()
    exact_rows, gap_rows = [], 0
    for i, r in enumerate(rows):
        v = int(vis[i])
        if kth_gap_ok(ref_lg[i, :v], wl.topk):
            gap_rows += 1
            assert np.array_equal(got_idx[i], ref_idx[i]), f"row {r}: top-k set differs outside the tie band"
        check_topk_valid(got_idx[i], ref_lg[i, :v].astype(np.float64), wl.topk, mag[i, :v])
        if np.array_equal(got_idx[i], ref_idx[i]):
            exact_rows.append(i)
    record(key, topk_rows=len(rows), topk_rows_outside_tie_band=gap_rows, topk_rows_equal_to_oracle=len(exact_rows))
    # the GPU top-k kernel on the oracle's logits must match the oracle's top-k bit for bit
    lg_t = torch.from_numpy(np.ascontiguousarray(ref_lg)).cuda()
    if np.array_equal(rows, np.arange(rows[0], rows[0] + len(rows))):
        got = torch.empty((len(rows), wl.topk), dtype=torch.int32, device="cuda")
        db.topk(logits=lg_t, idx=got, row_begin=int(rows[0]), row_end=int(rows[0]) + len(rows))
        assert np.array_equal(got.cpu().numpy(), ref_idx)
    else:
        for i, r in enumerate(rows):
            one = torch.empty((1, wl.topk), dtype=torch.int32, device="cuda")
            db.topk(logits=lg_t[i:i + 1], idx=one, row_begin=int(r), row_end=int(r) + 1)
            assert np.array_equal(one.cpu().numpy()[0], ref_idx[i]), f"row {r}"
    record(key, topk_on_oracle_logits_rows=len(rows))
    # attention: rows whose GPU selection equals the oracle's compare the step's own output
    if db.kv_pool is not None:
        ref_o, ref_l = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                         _full_idx(wl, rows, ref_idx), wl.scale, rows)
        out = bf16_to_np_f64(db.out[torch.from_numpy(rows).cuda()])
        lse = db.lse[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
        ex = np.asarray(exact_rows, np.int64)
        if ex.size:
            check_attention(out[ex], lse[ex], ref_o[ex], ref_l[ex], key=key + "/attention_of_step")
        # and the GPU attention fed the oracle's selection for every checked row
        idx_all = db.idx.clone()
        idx_all[torch.from_numpy(rows).cuda()] = torch.from_numpy(ref_idx).cuda()
        db.sparse_mla(idx=idx_all)
        out2 = bf16_to_np_f64(db.out[torch.from_numpy(rows).cuda()])
        lse2 = db.lse[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
        check_attention(out2, lse2, ref_o, ref_l, key=key + "/attention_of_oracle_selection")
    return len(exact_rows)


def _full_idx(wl, rows, ref_idx):
    idx = np.full((wl.T, wl.topk), -1, np.int32)
    idx[rows] = ref_idx
    return idx


def test_chain_tiny_all_rows():
    wl = workloads.make("tiny")
    db = DeviceBatch(wl)
    got_lg = run_step_capturing_logits(db, np.arange(wl.T))
    assert db.device_error() == (0, 0)
    pool = oracle_pool(wl)
    assert np.array_equal(db.index_pool.cpu().numpy(), pool)
    n_exact = check_rows(wl, db, np.arange(wl.T), pool, got_lg, "chain/tiny")
    assert n_exact == wl.T


ROWS = {
    "decode_b32_8k": lambda wl: np.arange(wl.T),
    "decode_b64_logu64k": lambda wl: np.arange(wl.T),
    "mtp_b8_128k": lambda wl: np.arange(wl.T),
    "prefill_32k_4k": lambda wl: np.unique(np.concatenate([np.arange(0, wl.T, 64), [wl.T - 1]])),
}


@pytest.mark.parametrize("name", list(ROWS))
def test_chain_full_size(name):
    wl = workloads.make(name)
    db = DeviceBatch(wl)
    rows = ROWS[name](wl)
    got_lg = run_step_capturing_logits(db, rows)
    assert db.device_error() == (0, 0)
    if name == "prefill_32k_4k":
        assert len(db.tiles()) > 1          # the 4096 x 36864 logits are produced in row tiles
    # the whole index-K cache (every request's pages, this step's keys included) is bit-exact
    pool = oracle_pool(wl)
    assert np.array_equal(db.index_pool.cpu().numpy(), pool)
    record(f"chain/{name}", index_pages=wl.num_pages)
    check_rows(wl, db, rows, pool, got_lg, f"chain/{name}")


def test_step_io_graph_matches_eager_step():
    """DeviceBatch.step_io (copies + four calls as one CUDA graph) gives the eager step's outputs,
    and replays move fresh host data every time."""
    wl = workloads.make("tiny")
    db = DeviceBatch(wl)
    db.step()
    ref_out = db.out.cpu().clone()
    ref_lse = db.lse.cpu().clone()
    host_in = [t.cpu().pin_memory() for t in db.io_inputs()]
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in db.io_outputs()]
    for _ in range(2):   # capture, then replay
        for h in host_out:
            h.zero_()
        db.step_io(host_in, host_out)
        torch.cuda.synchronize()
        assert torch.equal(host_out[0], ref_out) and torch.equal(host_out[1], ref_lse)
    # a changed query on the host reaches the device on replay
    host_in[2].copy_(-host_in[2])
    db.step_io(host_in, host_out)
    torch.cuda.synchronize()
    assert not torch.equal(host_out[0], ref_out)
    assert db.device_error() == (0, 0)


def test_step_io_packed_buffers_match_eager_step():
    """The packed form of step_io (one pinned block in, one out) gives the eager step's outputs
    and moves fresh host data on every replay."""
    wl = workloads.make("tiny")
    db = DeviceBatch(wl)
    db.step()
    ref_out = db.out.clone()
    dev_in, dev_out = db.io_buffers()
    host_in = [dev_in.cpu().pin_memory()]
    host_out = [torch.empty_like(dev_out, device="cpu").pin_memory()]
    for _ in range(2):   # capture, then replay
        host_out[0].zero_()
        db.step_io(host_in, host_out)
        torch.cuda.synchronize()
        assert torch.equal(db.out, ref_out)
        assert torch.equal(host_out[0], dev_out.cpu())
    # a changed query on the host reaches the device on replay
    q_off = db.mla_q.data_ptr() - dev_in.data_ptr()
    mod = dev_in.clone()
    mod[q_off:q_off + db.mla_q.numel() * 2].view(torch.bfloat16).neg_()
    host_in[0].copy_(mod.cpu())
    db.step_io(host_in, host_out)
    torch.cuda.synchronize()
    assert not torch.equal(db.out, ref_out)
    assert torch.equal(host_out[0], dev_out.cpu())
    assert db.device_error() == (0, 0)


def test_run_io_pipelined_steps_match_eager_steps():
    """run_io over several steps with different host inputs: every step's outputs equal the eager
    step's outputs for that step's inputs (the two device I/O sets and the overlapped copies keep
    each step's data apart)."""
    wl = workloads.make("tiny")
    db = DeviceBatch(wl)
    dev_in, dev_out = db.io_buffers()
    q_off = db.mla_q.data_ptr() - dev_in.data_ptr()
    nq = db.mla_q.numel() * 2
    base = dev_in.clone()
    host_ins, refs = [], []
    for i in range(5):                       # step i: the query scaled by (1 + i / 4)
        mod = base.clone()
        mod[q_off:q_off + nq].view(torch.bfloat16).mul_(1.0 + i / 4.0)
        dev_in.copy_(mod)
        db.step()
        torch.cuda.synchronize()
        refs.append(dev_out.cpu().clone())
        host_ins.append(mod.cpu().pin_memory())
    host_outs = [torch.zeros_like(refs[0]).pin_memory() for _ in range(5)]
    db.run_io(host_ins, host_outs)
    torch.cuda.synchronize()
    for i in range(5):
        assert torch.equal(host_outs[i], refs[i]), f"step {i}"
    assert not torch.equal(refs[0], refs[1])
    assert db.device_error() == (0, 0)


def test_back_to_back_calls_keep_stream_order():
    """The logits, top-k and attention kernels overlap their successors' launch; a call that
    overwrites a buffer the previous call still reads must still see stream order.  Here a second
    top-k (on different logits, into the same idx) is enqueued right after the attention call that
    reads idx, and a second indexer call right after the top-k that reads the logits."""
    wl = workloads.make("tiny")
    db = DeviceBatch(wl)
    db.step()
    torch.cuda.synchronize()
    ref_out = db.out.clone()
    ref_idx = db.idx.clone()
    flipped = -db.logits   # made before the sequence, so that attention and top-k are adjacent launches
    # attention reads idx, then top-k rewrites idx from reversed logits, in one stream, no sync
    db.logits.zero_()
    db.indexer_logits()
    db.topk()
    db.sparse_mla()
    db.topk(logits=flipped)
    torch.cuda.synchronize()
    assert torch.equal(db.out, ref_out)            # attention used the first idx
    assert not torch.equal(db.idx, ref_idx)        # the second top-k did run afterwards
    # top-k reads the logits, then the indexer rewrites them with a rotated query, no sync
    db.indexer_logits()
    db.topk()
    idx_first = db.idx.clone()
    db.indexer_logits(flags=capi.DSA_Q_ROTATE)
    torch.cuda.synchronize()
    assert torch.equal(idx_first, ref_idx)
    assert db.device_error() == (0, 0)


def test_indexer_right_after_a_long_store_sees_the_stored_keys():
    """The one-call indexer enqueued right after a store of every key of its rows (no sync): the
    query prologue is a programmatic dependent of the store and the logits kernel streams key
    pages before its own wait, so the prologue lets it start only after its wait on the store.
    The store writes 240 K keys into a zeroed pool; the one-call indexer's logits are compared
    with the oracle's.  (An end-to-end check of the order: a premature start would show only where
    it overlapped the last pages written, which this timing does not force.)"""
    from helpers import check_logits, oracle_pool
    from deepseek_sparse_attention_paged_gb300.pipeline import lightning_logits_offset
    wl = workloads.make_custom("store_then_index", 261, [60000, 59000, 61000, 58000], 1, topk=2048, heads=16)
    db = DeviceBatch(wl, with_latent=False, build_index_cache=False)
    keys = torch.from_numpy(np.ascontiguousarray(wl.index_keys()).view(np.int16)).cuda().view(torch.bfloat16)
    slots = torch.from_numpy(wl.token_slots()).cuda()
    ws = torch.empty(capi.dsa_lightning_indexer_workspace_size(wl.T, wl.max_seq_len), dtype=torch.uint8,
                     device="cuda")
    idx = torch.empty((wl.T, wl.topk), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    capi.dsa_store_index_k(keys, slots, db.index_pool, db.dev_err)
    capi.dsa_lightning_indexer(db.index_q, db.weights, db.index_pool, db.block_table, db.seq_lens, db.cu_q,
                               wl.max_seq_len, wl.max_q_len, wl.topk, idx, ws, dev_err=db.dev_err)
    torch.cuda.synchronize()
    pool = oracle_pool(wl)
    assert np.array_equal(db.index_pool.cpu().numpy(), pool)
    rows = np.arange(wl.T)
    ref, mag, bad = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                                          rows, db.ld, want_mag=True)
    assert bad == 0
    off = lightning_logits_offset(wl.T)
    lg = ws[off:off + wl.T * db.ld * 4].view(torch.float32).view(wl.T, db.ld).cpu().numpy()
    check_logits(lg, ref, mag, wl.visible_lens(), key="chain/store_then_index")
    assert db.device_error() == (0, 0)
