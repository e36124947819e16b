"""GPU parity of the compressed-KV (DSV4, compress ratio 4) decode path against the oracle: the
indexer over compressed keys (DSA_KEYS_CMP4) element by element, its top-k through the one-call
indexer, and the window + compressed + sink attention fed the oracle's selection -- on ragged
next_n batches and on every row of the 64-request 64K batch."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import logits_ld

from helpers import bf16_to_np_f64, check_attention, check_logits, check_topk_valid, kth_gap_ok, record

pytestmark = pytest.mark.gpu


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _run_case(wl, c, key, rows=None, sinks=None):
    T = wl.T
    rows = np.arange(T) if rows is None else np.asarray(rows)
    # compressed index keys: FP8 cache written by the store call, bit-exact with the oracle's
    keys, slots = c.index_keys(), c.slots()
    ref_pool = np.zeros((c.num_pages, oracle.PAGE_BYTES), np.uint8)
    assert oracle.store_index_k(keys, slots, ref_pool) == 0
    pool = torch.zeros((c.num_pages, oracle.PAGE_BYTES), dtype=torch.uint8, device="cuda")
    capi.dsa_store_index_k(_dev_bf16(keys), torch.from_numpy(slots).cuda(), pool)
    assert np.array_equal(pool.cpu().numpy(), ref_pool)
    q, w = _dev_bf16(wl.index_q()), torch.from_numpy(wl.weights()).cuda()
    cbt, sl, cq = _i32(c.block_table), _i32(wl.seq_lens), _i32(wl.cu_q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ld = logits_ld(c.max_cmp_len)
    # logits over the compressed entries
    lg = torch.full((T, ld), float("nan"), dtype=torch.float32, device="cuda")
    capi.dsa_indexer_logits(q, w, pool, cbt, sl, cq, c.max_cmp_len, wl.max_q_len, lg, flags=capi.DSA_KEYS_CMP4,
                            dev_err=err)
    ref, mag, bad = oracle.indexer_logits(wl.index_q(), wl.weights(), ref_pool, c.block_table, wl.seq_lens, wl.cu_q,
                                          np.arange(T), ld, want_mag=True, cmp_ratio=c.ratio)
    assert bad == 0
    got = lg.cpu().numpy()
    vis = c.visible_cmp_lens()
    check_logits(got[rows], ref[rows], mag[rows], vis[rows], key=key + "/logits")
    for r in rows:
        assert np.all(np.isnan(got[r, vis[r]:]))
    # the one-call indexer: top-k of the compressed entries
    idx = torch.empty((T, c.topk), dtype=torch.int32, device="cuda")
    ws = torch.empty(capi.dsa_lightning_indexer_workspace_size(T, c.max_cmp_len), dtype=torch.uint8, device="cuda")
    capi.dsa_lightning_indexer(q, w, pool, cbt, sl, cq, c.max_cmp_len, wl.max_q_len, c.topk, idx, ws,
                               flags=capi.DSA_KEYS_CMP4, dev_err=err)
    got_idx = idx.cpu().numpy()
    ref_idx = oracle.topk(ref, wl.seq_lens, wl.cu_q, np.arange(T), c.topk, cmp_ratio=c.ratio)
    gap = 0
    for r in rows:
        v = int(vis[r])
        check_topk_valid(got_idx[r], ref[r, :v].astype(np.float64), c.topk, mag[r, :v])
        if kth_gap_ok(ref[r, :v], c.topk):
            gap += 1
            assert np.array_equal(got_idx[r], ref_idx[r])
    record(key + "/topk", rows=len(rows), rows_outside_tie_band=gap)
    # attention: window of the original cache + the oracle's selection of compressed entries + sinks
    sinks = c.sinks() if sinks is None else np.asarray(sinks, np.float32)
    H = wl.heads
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    capi.dsa_sparse_attn_swa_cmp(_dev_bf16(wl.mla_q()), _dev_bf16(wl.latent_pool()), _i32(wl.block_table),
                                 _dev_bf16(c.latent_pool()), cbt, sl, cq, _i32(ref_idx), c.window, c.ratio,
                                 torch.from_numpy(sinks).cuda(), wl.scale, out, lse=lse, dev_err=err)
    torch.cuda.synchronize()
    ref_o, ref_l, skipped = oracle.dsv4_attention(wl.mla_q(), wl.latent_pool(), wl.block_table, c.latent_pool(),
                                                  c.block_table, wl.seq_lens, wl.cu_q, ref_idx, c.window, sinks,
                                                  wl.scale, rows, ratio=c.ratio)
    assert skipped == 0
    check_attention(bf16_to_np_f64(out[torch.from_numpy(rows).cuda()]),
                    lse[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64), ref_o, ref_l,
                    key=key + "/attention")
    assert tuple(capi.dsa_read_device_error(err)) == (0, 0)


def test_dsv4_ragged_next_n_short_and_window_longer_than_context():
    wl = workloads.make_custom("dsv4_ragged", 301, [300, 1000, 7, 70, 2049], [1, 2, 1, 3, 1], topk=64, heads=16)
    c = workloads.make_compressed(wl, ratio=4, window=96, topk=64)
    _run_case(wl, c, "dsv4/ragged")


def test_dsv4_without_sinks_and_128_heads():
    wl = workloads.make_custom("dsv4_nosink", 302, [5000, 640, 129], 1, topk=128, heads=128)
    c = workloads.make_compressed(wl, ratio=4, window=128, topk=128)
    _run_case(wl, c, "dsv4/no_sink", sinks=np.full(128, -np.inf, np.float32))


def test_dsv4_full_size_every_row():
    wl = workloads.make("decode_b64_logu64k")
    c = workloads.make_compressed(wl)          # ratio 4, window 128, top-512 of the compressed entries
    _run_case(wl, c, "dsv4/decode_b64_logu64k")


def test_dsv4_attention_rejects_bad_ratio_and_short_workspace():
    wl = workloads.make_custom("dsv4_args", 303, [300], 1, topk=64, heads=16)
    c = workloads.make_compressed(wl, ratio=4, window=64, topk=64)
    T, H, k = wl.T, wl.heads, 2048                  # one row over 2112 entries: split, so scratch is needed
    args = (_dev_bf16(wl.mla_q()), _dev_bf16(wl.latent_pool()), _i32(wl.block_table), _dev_bf16(c.latent_pool()),
            _i32(c.block_table), _i32(wl.seq_lens), _i32(wl.cu_q), _i32(np.zeros((T, k), np.int32)))
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    sinks = torch.zeros(H, dtype=torch.float32, device="cuda")
    with pytest.raises(capi.DSAError) as e:
        capi.dsa_sparse_attn_swa_cmp(*args, 64, 3, sinks, wl.scale, out)
    assert e.value.status == capi.DSA_ERR_UNSUPPORTED
    need = capi.dsa_sparse_attn_swa_cmp_workspace_size(T, H, 64, k)
    assert need > 0
    with pytest.raises(capi.DSAError) as e:
        short = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
        capi.dsa_sparse_attn_swa_cmp(*args, 64, 4, sinks, wl.scale, out, workspace=short)
    assert e.value.status == capi.DSA_ERR_INVALID_ARG


def test_dsv4_split_rows_add_the_sink_in_the_combine():
    """Few rows and many entries: each row is split over several clusters and the sink enters in
    the split-K combine instead of the kernel's epilogue."""
    wl = workloads.make_custom("dsv4_split", 304, [20000, 9000], 1, topk=64, heads=32)
    c = workloads.make_compressed(wl, ratio=4, window=256, topk=2048)
    assert capi.dsa_sparse_attn_swa_cmp_workspace_size(wl.T, wl.heads, c.window, c.topk) > 0
    _run_case(wl, c, "dsv4/split")
