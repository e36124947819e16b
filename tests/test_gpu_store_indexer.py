"""GPU parity of dsa_store_index_k (bit-exact) and dsa_indexer_logits (tolerance) against the
CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

from helpers import check_logits, oracle_pool

pytestmark = pytest.mark.gpu


def _bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def test_store_bit_exact_tiny():
    wl = workloads.make("tiny")
    db = DeviceBatch(wl, with_latent=False)
    got = db.index_pool.cpu().numpy()
    assert np.array_equal(got, oracle_pool(wl))
    assert db.device_error() == (0, 0)


def test_store_bit_exact_scaled_keys_padding_and_range():
    rng = np.random.default_rng(101)
    n = 777
    x = rng.standard_normal((n, 128)).astype(np.float32)
    x[:100] *= 1e-3
    x[100:200] *= 40.0
    x[200] = 0.0                              # zero key: scale 1e-4 / 448
    x[201, :] = 0.0
    x[201, 5] = 3.0                           # single spike
    keys = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pages = 20
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    slots[300] = -1                           # padding token
    slots[301] = pages * 64 + 3               # past the pool
    ref = np.full((pages, oracle.PAGE_BYTES), 0x5A, np.uint8)
    assert oracle.store_index_k(keys, slots, ref) == 1
    pool = torch.full((pages, oracle.PAGE_BYTES), 0x5A, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_store_index_k(_bf16_dev(keys), torch.from_numpy(slots).cuda(), pool, err)
    assert np.array_equal(pool.cpu().numpy(), ref)
    st, word = capi.dsa_read_device_error(err)
    assert st == capi.DSA_ERR_DEVICE_BOUNDS and word == capi.DSA_DEVERR_SLOT_RANGE


def test_store_empty_is_noop():
    pool = torch.zeros((1, oracle.PAGE_BYTES), dtype=torch.uint8, device="cuda")
    capi.dsa_store_index_k(torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda"),
                           torch.zeros(0, dtype=torch.int64, device="cuda"), pool)
    torch.cuda.synchronize()
    assert int(pool.sum()) == 0


def _logits_case(wl, flags=0, row_begin=0, row_end=None):
    db = DeviceBatch(wl, with_latent=False)
    T = wl.T
    row_end = T if row_end is None else row_end
    lg = torch.full((row_end - row_begin, db.ld), float("nan"), dtype=torch.float32, device="cuda")
    db.indexer_logits(row_begin=row_begin, row_end=row_end, logits=lg, flags=flags)
    got = lg.cpu().numpy()
    pool = oracle_pool(wl)
    rows = np.arange(row_begin, row_end)
    ref, mag, bad = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                                          rows, db.ld, rotate_q=bool(flags & capi.DSA_Q_ROTATE), want_mag=True,
                                          ue8m0_q=bool(flags & capi.DSA_SCALE_UE8M0))
    assert bad == 0
    vis = wl.visible_lens()[row_begin:row_end]
    check_logits(got, ref, mag, vis)
    for i, v in enumerate(vis):          # nothing past the visible length is written
        assert np.all(np.isnan(got[i, v:]))
    assert db.device_error() == (0, 0)
    return got


def test_logits_tiny():
    _logits_case(workloads.make("tiny"))


def test_logits_ragged_lengths_and_tails():
    lens = [1, 63, 64, 65, 127, 128, 129, 1000, 4097, 300]
    _logits_case(workloads.make_custom("ragged", 102, lens, 1, topk=64, heads=16))


def test_logits_next_n_causal():
    _logits_case(workloads.make_custom("mtp", 103, [200, 129, 2], 2, topk=64, heads=16))


def test_logits_prefill_chunk_causal_and_row_tiles():
    wl = workloads.make_custom("prefill", 104, [700], 150, topk=256, heads=16)
    full = _logits_case(wl)
    part = _logits_case(wl, row_begin=37, row_end=101)
    assert np.array_equal(part, full[37:101], equal_nan=True)


def test_logits_mixed_query_counts_and_empty_requests():
    # q_len 5 -> groups of 4 rows with a 1-row tail; a request without query rows; short contexts
    wl = workloads.make_custom("mixed", 106, [500, 64, 900, 130, 7, 260], [3, 0, 5, 1, 2, 4], topk=64, heads=16)
    _logits_case(wl)


def test_logits_fewer_tiles_than_sms():
    _logits_case(workloads.make_custom("few", 107, [5, 17, 3], 1, topk=64, heads=16))


def test_logits_many_requests_shares_split_inside_requests():
    # ~2900 key tiles over one CTA per SM: most CTAs start and end inside a request
    lens = np.random.default_rng(108).integers(1, 6000, size=120).tolist()
    _logits_case(workloads.make_custom("many", 108, lens, 1, topk=64, heads=16))


def test_logits_shares_spanning_many_short_segments():
    # 200 one-tile requests, then 56 long ones (256 segments): the CTAs holding the short requests
    # each span ~18 segments, more than the first ones they keep in shared memory
    rng = np.random.default_rng(109)
    lens = rng.integers(1, 129, size=200).tolist() + rng.integers(5000, 6001, size=56).tolist()
    _logits_case(workloads.make_custom("segments", 109, lens, 1, topk=64, heads=16))


def test_logits_rotate_q_flag():
    _logits_case(workloads.make("tiny"), flags=capi.DSA_Q_ROTATE)


def test_logits_ue8m0_query_scales():
    _logits_case(workloads.make_custom("ue8m0", 108, [300, 1000, 70], 2, topk=64, heads=16),
                 flags=capi.DSA_SCALE_UE8M0 | capi.DSA_Q_ROTATE)


def test_logits_bad_page_sets_error_word_and_does_not_fault():
    wl = workloads.make_custom("badpage", 105, [300, 200], 1, topk=64, heads=16)
    db = DeviceBatch(wl, with_latent=False)
    bt = db.block_table.clone()
    bt[0, 2] = wl.num_pages + 5
    db.block_table = bt
    db.logits.fill_(float("nan"))
    db.indexer_logits()
    st, word = db.device_error()
    assert st == capi.DSA_ERR_DEVICE_BOUNDS and word & capi.DSA_DEVERR_PAGE_RANGE
    got = db.logits.cpu().numpy()
    assert np.all(np.isfinite(got[1, :200]))        # the other request is fully scored
    assert np.all(np.isfinite(got[0, :128]))


def test_logits_invalid_args():
    wl = workloads.make("tiny")
    db = DeviceBatch(wl, with_latent=False)
    with pytest.raises(capi.DSAError) as e:
        narrow = torch.empty((wl.T, 10), dtype=torch.float32, device="cuda")   # ld = 10 < max_seq_len
        capi.dsa_indexer_logits(db.index_q, db.weights, db.index_pool, db.block_table, db.seq_lens, db.cu_q,
                                wl.max_seq_len, 1, narrow)
    assert e.value.status == capi.DSA_ERR_INVALID_ARG
    with pytest.raises(capi.DSAError) as e:   # workspace one byte short
        short = torch.empty(capi.dsa_indexer_logits_workspace_size(wl.T) - 1, dtype=torch.uint8, device="cuda")
        capi.dsa_indexer_logits(db.index_q, db.weights, db.index_pool, db.block_table, db.seq_lens, db.cu_q,
                                wl.max_seq_len, 1, db.logits, workspace=short)
    assert e.value.status == capi.DSA_ERR_INVALID_ARG
