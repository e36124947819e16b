"""GPU parity of the int8 ("c8") index cache: dsa_store_index_k_c8 bit-exact against the oracle,
dsa_indexer_logits_c8 against the oracle's logits (the integer dot products are exact on both
sides; only the fp32 head sum differs), and the top-k over them, from tiny ragged cases to every row
and every index page of the 64-request 64K decode batch."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

from helpers import check_logits, check_topk_valid, kth_gap_ok, record

pytestmark = pytest.mark.gpu


def _bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def oracle_pool_c8(wl):
    pool = np.zeros((wl.num_pages, oracle.C8_PAGE_BYTES), np.uint8)
    assert oracle.store_index_k_c8(wl.index_keys(), wl.token_slots(), pool) == 0
    return pool


def test_store_c8_bit_exact_tiny():
    wl = workloads.make("tiny")
    db = DeviceBatch(wl, with_latent=False, c8=True)
    assert np.array_equal(db.index_pool_c8.cpu().numpy(), oracle_pool_c8(wl))
    assert db.device_error() == (0, 0)


def test_store_c8_scaled_zero_spike_padding_and_range():
    rng = np.random.default_rng(201)
    n = 777
    x = rng.standard_normal((n, 128)).astype(np.float32)
    x[:100] *= 1e-3
    x[100:200] *= 40.0
    x[200] = 0.0                              # zero key: scale 0, codes 0
    x[201, :] = 0.0
    x[201, 5] = 3.0                           # single spike: every rotated entry +-3c
    x[202] = 1e-30                            # subnormal-range fp16 scale
    x[203, :] = rng.standard_normal(128) * 1e-6
    x[203, 7] = 3000.0                        # exponent spread beyond fp32's 24 bits: the fp64 fallback
    x[204, ::2] = 1.0 + 2.0 ** -7             # products on bf16 midpoints
    keys = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pages = 20
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    slots[300] = -1                           # padding token
    slots[301] = pages * 64 + 3               # past the pool
    ref = np.full((pages, oracle.C8_PAGE_BYTES), 0x5A, np.uint8)
    assert oracle.store_index_k_c8(keys, slots, ref) == 1
    pool = torch.full((pages, oracle.C8_PAGE_BYTES), 0x5A, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_store_index_k_c8(_bf16_dev(keys), torch.from_numpy(slots).cuda(), pool, err)
    assert np.array_equal(pool.cpu().numpy(), ref)
    st, word = capi.dsa_read_device_error(err)
    assert st == capi.DSA_ERR_DEVICE_BOUNDS and word == capi.DSA_DEVERR_SLOT_RANGE


def _logits_c8_case(wl, key, row_begin=0, row_end=None, pool=None, db=None):
    db = db or DeviceBatch(wl, with_latent=False, c8=True)
    row_end = wl.T if row_end is None else row_end
    lg = torch.full((row_end - row_begin, db.ld), float("nan"), dtype=torch.float32, device="cuda")
    db.indexer_logits_c8(row_begin=row_begin, row_end=row_end, logits=lg)
    torch.cuda.synchronize()
    got = lg.cpu().numpy()
    pool = oracle_pool_c8(wl) if pool is None else pool
    rows = np.arange(row_begin, row_end)
    ref, mag, bad = oracle.indexer_logits_c8(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                                             rows, db.ld, want_mag=True)
    assert bad == 0
    vis = wl.visible_lens()[row_begin:row_end]
    check_logits(got, ref, mag, vis, key=key)
    for i, v in enumerate(vis):           # nothing past the visible length is written
        assert np.all(np.isnan(got[i, v:]))
    assert db.device_error() == (0, 0)
    return db, got, ref, mag


def test_logits_c8_tiny():
    _logits_c8_case(workloads.make("tiny"), "c8_logits/tiny")


def test_logits_c8_ragged_lengths_and_tails():
    lens = [1, 63, 64, 65, 127, 128, 129, 1000, 4097, 300]
    _logits_c8_case(workloads.make_custom("ragged", 202, lens, 1, topk=64, heads=16), "c8_logits/ragged")


def test_logits_c8_next_n_causal():
    _logits_c8_case(workloads.make_custom("mtp", 203, [200, 129, 2], 2, topk=64, heads=16), "c8_logits/next_n")


def test_logits_c8_mixed_query_counts_and_row_tiles():
    # q_len 5 -> groups of 2 rows with a 1-row tail; a request without query rows
    wl = workloads.make_custom("mixed", 204, [500, 64, 900, 130, 7, 260], [3, 0, 5, 1, 2, 4], topk=64, heads=16)
    db, full, _, _ = _logits_c8_case(wl, "c8_logits/mixed")
    _, part, _, _ = _logits_c8_case(wl, "c8_logits/mixed_tile", row_begin=3, row_end=11, db=db)
    assert np.array_equal(part, full[3:11], equal_nan=True)


def test_logits_c8_many_requests_shares_split_inside_requests():
    lens = np.random.default_rng(205).integers(1, 6000, size=120).tolist()
    _logits_c8_case(workloads.make_custom("many", 205, lens, 1, topk=64, heads=16), "c8_logits/many")


def test_logits_c8_bad_page_sets_error_word_and_does_not_fault():
    wl = workloads.make_custom("badpage", 206, [300, 200], 1, topk=64, heads=16)
    db = DeviceBatch(wl, with_latent=False, c8=True)
    bt = db.block_table.clone()
    bt[0, 2] = wl.num_pages + 5
    db.block_table = bt
    db.logits.fill_(float("nan"))
    db.indexer_logits_c8()
    st, word = db.device_error()
    assert st == capi.DSA_ERR_DEVICE_BOUNDS and word & capi.DSA_DEVERR_PAGE_RANGE
    got = db.logits.cpu().numpy()
    assert np.all(np.isfinite(got[1, :200]))
    assert np.all(np.isfinite(got[0, :128]))


def test_logits_c8_invalid_args():
    wl = workloads.make("tiny")
    db = DeviceBatch(wl, with_latent=False, c8=True)
    with pytest.raises(capi.DSAError) as e:   # workspace one byte short
        short = torch.empty(capi.dsa_indexer_logits_c8_workspace_size(wl.T) - 1, dtype=torch.uint8, device="cuda")
        capi.dsa_indexer_logits_c8(db.index_q, db.weights, db.index_pool_c8, db.block_table, db.seq_lens, db.cu_q,
                                   wl.max_seq_len, 1, db.logits, workspace=short)
    assert e.value.status == capi.DSA_ERR_INVALID_ARG


def test_c8_full_size_every_row_and_page():
    """The 64-request 64K decode batch: the whole int8 cache byte for byte, every row's logits, and
    the top-k over them (GPU indices from GPU logits vs the oracle's from its own logits, and the
    GPU top-k kernel on the oracle's logits bit for bit)."""
    wl = workloads.make("decode_b64_logu64k")
    db = DeviceBatch(wl, with_latent=False, c8=True)
    pool = oracle_pool_c8(wl)
    assert np.array_equal(db.index_pool_c8.cpu().numpy(), pool)
    record("c8/decode_b64_logu64k", index_pages=wl.num_pages)
    lg = torch.full((wl.T, db.ld), float("nan"), dtype=torch.float32, device="cuda")
    _, got, ref, mag = _logits_c8_case(wl, "c8/decode_b64_logu64k", pool=pool, db=db)
    rows = np.arange(wl.T)
    vis = wl.visible_lens()
    lg.copy_(torch.from_numpy(got))
    idx = torch.empty((wl.T, wl.topk), dtype=torch.int32, device="cuda")
    db.topk(logits=lg, idx=idx)
    got_idx = idx.cpu().numpy()
    ref_idx = oracle.topk(ref, wl.seq_lens, wl.cu_q, rows, wl.topk)
    gap = 0
    for r in rows:
        v = int(vis[r])
        check_topk_valid(got_idx[r], ref[r, :v].astype(np.float64), wl.topk, mag[r, :v])
        if kth_gap_ok(ref[r, :v], wl.topk):
            gap += 1
            assert np.array_equal(got_idx[r], ref_idx[r])
    lg_ref = torch.from_numpy(np.ascontiguousarray(ref)).cuda()
    db.topk(logits=lg_ref, idx=idx)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    record("c8/decode_b64_logu64k", topk_rows=wl.T, topk_rows_outside_tie_band=gap, topk_on_oracle_logits_rows=wl.T)
