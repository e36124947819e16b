"""GPU parity of dsa_topk (bit-exact) and dsa_sparse_mla_decode (tolerance) against the CPU oracle,
each fed the same oracle-side inputs, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

from helpers import bf16_to_np_f64, check_attention, check_topk_valid, kth_gap_ok, oracle_pool

pytestmark = pytest.mark.gpu


def _gpu_topk(logits_np, seq_lens, q_lens, k, max_seq_len=None):
    seq_lens = np.asarray(seq_lens, np.int32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(cu[-1])
    ld = logits_np.shape[1]
    lg = torch.from_numpy(np.ascontiguousarray(logits_np, np.float32)).cuda()
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    msl = int(seq_lens.max()) if max_seq_len is None else max_seq_len
    ws_n = capi.dsa_topk_workspace_size(T, k, msl)
    ws = torch.empty(max(1, ws_n), dtype=torch.uint8, device="cuda")
    capi.dsa_topk(lg, torch.from_numpy(seq_lens).cuda(), torch.from_numpy(cu).cuda(), msl, k, idx, workspace=ws)
    ref = oracle.topk(logits_np, seq_lens, cu, np.arange(T), k)
    return idx.cpu().numpy(), ref


def test_topk_on_oracle_logits_tiny():
    wl = workloads.make("tiny")
    pool = oracle_pool(wl)
    lg = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                               np.arange(wl.T), wl.max_seq_len)
    got, ref = _gpu_topk(lg, wl.seq_lens, wl.q_lens, wl.topk)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("v,k", [(0, 16), (1, 16), (15, 16), (16, 16), (17, 16), (2048, 2048), (2049, 2048),
                                 (5000, 2048), (70000, 2048), (131072, 2048), (3000, 1), (3000, 1999),
                                 (40, 3), (100, 7), (131071, 2048), (140000, 2048), (140000, 100),
                                 (20000, 2048), (20001, 2048), (33000, 100), (65536, 2048), (65792, 2048)])
def test_topk_lengths_and_ties(v, k):
    rng = np.random.default_rng(200 + v + k)
    width = max(v, 4)
    lg = np.full((3, width + 4), np.nan, np.float32)
    lg[0, :v] = rng.standard_normal(v).astype(np.float32)
    lg[1, :v] = rng.integers(-8, 8, v).astype(np.float32)            # heavy ties
    lg[2, :v] = np.where(rng.random(v) < 0.5, -0.0, 0.0)              # all zeros of both signs
    if v > 10:
        lg[2, 3] = np.nan
        lg[2, 7] = -np.inf
        lg[0, 5] = np.inf
    got, ref = _gpu_topk(lg, [v, v, v], [1, 1, 1], k, max_seq_len=max(v, 1))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("v,k", [(70000, 2048), (70000, 1500), (9000, 2048), (131072, 100), (40000, 2048)])
def test_topk_rows_that_mislead_the_sample(v, k):
    """Rows whose evenly spaced sample misjudges the cut: the largest values sit on sampled
    positions only (fewer than k keys reach the cut), everywhere but the sampled positions (far
    more keys than fit pass it), or the row is one value with sparse outliers."""
    S = 2048
    sampled = (np.arange(S, dtype=np.int64) * v) // S
    lg = np.zeros((4, v + 4), np.float32)
    lg[0, :v] = np.random.default_rng(220).standard_normal(v).astype(np.float32) - 10.0
    lg[0, sampled[::2]] = 50.0 + np.arange(S // 2, dtype=np.float32) * 1e-3   # large values only where sampled
    lg[1, :v] = 100.0
    lg[1, sampled] = -5.0                                                  # the sample sees only small values
    lg[2, :v] = 1.0
    lg[2, np.arange(0, v, 997)] = 2.0                                      # one value plus sparse outliers
    lg[3, :v] = np.random.default_rng(221).standard_normal(v).astype(np.float32)
    lg[3, sampled[::2]] = 7.0                                              # ties at the top on half the sample
    got, ref = _gpu_topk(lg, [v] * 4, [1] * 4, k, max_seq_len=v)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("v,k,n_init,n_local", [(100, 16, 2, 3), (5000, 2048, 4, 64), (20000, 2048, 1, 1),
                                                 (70000, 2048, 16, 512), (70000, 100, 0, 300), (140000, 2048, 4, 64),
                                                 (3000, 64, 3000, 0)])
def test_topk_forced_init_and_local_tokens(v, k, n_init, n_local):
    rng = np.random.default_rng(230 + v + n_local)
    lg = np.full((3, v + 4), np.nan, np.float32)
    lg[0, :v] = rng.standard_normal(v).astype(np.float32)
    lg[1, :v] = rng.integers(-8, 8, v).astype(np.float32)      # heavy ties
    lg[2, :v] = rng.standard_normal(v).astype(np.float32)
    lg[2, v // 3] = np.inf                                      # ties with the forced positions by index
    seq_lens = np.array([v, v, v], np.int32)
    cu = np.array([0, 1, 2, 3], np.int32)
    dev = torch.from_numpy(lg).cuda()
    idx = torch.empty((3, k), dtype=torch.int32, device="cuda")
    capi.dsa_topk(dev, torch.from_numpy(seq_lens).cuda(), torch.from_numpy(cu).cuda(), v, k, idx,
                  n_init=n_init, n_local=n_local)
    ref = oracle.topk_forced(lg, seq_lens, cu, np.arange(3), k, n_init, n_local)
    assert np.array_equal(idx.cpu().numpy(), ref)


def test_topk_next_n_rows_use_their_own_length():
    rng = np.random.default_rng(210)
    L = 3000
    lg = rng.standard_normal((2, L)).astype(np.float32)
    lg[:, L - 1] = 100.0      # only row 1 can see the last key
    got, ref = _gpu_topk(lg, [L], [2], 256)
    assert np.array_equal(got, ref)
    assert L - 1 not in got[0] and L - 1 in got[1]


def _mla_case(wl, idx, expect_bad=0):
    db = DeviceBatch(wl, with_latent=True, build_index_cache=False)
    db.sparse_mla(idx=torch.from_numpy(idx).cuda())
    out = bf16_to_np_f64(db.out)
    lse = db.lse.cpu().numpy().astype(np.float64)
    ref_o, ref_l, _, bad = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                             idx, wl.scale, np.arange(wl.T), want_psum=True)
    assert bad == expect_bad
    err = check_attention(out, lse, ref_o, ref_l)
    return db, err


def _random_idx(wl, k, fill, rng):
    idx = np.full((wl.T, k), -1, np.int32)
    vis = wl.visible_lens()
    for r in range(wl.T):
        n = min(int(fill * k), int(vis[r]))
        idx[r, :n] = np.sort(rng.choice(int(vis[r]), n, replace=False))
    return idx


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_mla_random_selection(H):
    rng = np.random.default_rng(300 + H)
    wl = workloads.make_custom("mla", 300 + H, [3000, 700, 129], 1, topk=512, heads=H)
    _mla_case(wl, _random_idx(wl, 512, 0.9, rng))


def test_mla_tiny_full_k_several_splits():
    rng = np.random.default_rng(311)
    wl = workloads.make_custom("mla2k", 311, [5000, 2048, 2100], 1, topk=2048, heads=128)
    idx = _random_idx(wl, 2048, 1.0, rng)
    _mla_case(wl, idx)


def test_mla_empty_rows_and_unsorted_entries():
    rng = np.random.default_rng(312)
    wl = workloads.make_custom("mla_e", 312, [400, 400], 1, topk=256, heads=16)
    idx = _random_idx(wl, 256, 0.5, rng)
    idx[1] = -1                                  # no valid entry: out = 0, lse = -inf
    idx[0, :128] = rng.permutation(idx[0, :128])  # order inside the list does not matter
    db, _ = _mla_case(wl, idx)
    assert float(db.out[1].abs().max()) == 0.0
    assert bool(torch.isneginf(db.lse[1]).all())


def test_mla_out_of_range_entries_are_skipped_and_reported():
    rng = np.random.default_rng(313)
    wl = workloads.make_custom("mla_bad", 313, [500, 300], 1, topk=128, heads=32)
    idx = _random_idx(wl, 128, 0.5, rng)
    idx[0, 100] = 500          # == v: future position
    idx[1, 120] = 10 ** 6
    db, _ = _mla_case(wl, idx, expect_bad=2)
    st, word = db.device_error()
    assert st == capi.DSA_ERR_DEVICE_BOUNDS and word & capi.DSA_DEVERR_INDEX_RANGE


def test_mla_workspace_too_small_is_rejected():
    wl = workloads.make_custom("mla_ws", 314, [3000], 1, topk=2048, heads=16)   # one row: split over k
    db = DeviceBatch(wl, with_latent=True, build_index_cache=False)
    assert capi.dsa_sparse_mla_workspace_size(wl.T, wl.heads, wl.topk) > 16
    idx = torch.full((1, 2048), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.DSAError) as e:
        capi.dsa_sparse_mla_decode(db.mla_q, db.kv_pool, db.block_table, db.seq_lens, db.cu_q, idx, wl.scale,
                                   db.out, db.mla_ws[:16])
    assert e.value.status == capi.DSA_ERR_INVALID_ARG


def test_lightning_indexer_equals_logits_then_topk():
    """The one-call indexer returns exactly the indices of the logits call followed by the top-k
    call (the same kernels), with and without forced tokens."""
    wl = workloads.make_custom("li", 240, [500, 64, 3000, 17000, 40000], [1, 2, 3, 1, 1], topk=256, heads=16)
    db = DeviceBatch(wl, with_latent=False)
    db.indexer_logits()
    ws = torch.empty(capi.dsa_lightning_indexer_workspace_size(wl.T, wl.max_seq_len), dtype=torch.uint8,
                     device="cuda")
    for n_init, n_local in ((0, 0), (2, 8)):
        ref = torch.empty((wl.T, wl.topk), dtype=torch.int32, device="cuda")
        capi.dsa_topk(db.logits, db.seq_lens, db.cu_q, wl.max_seq_len, wl.topk, ref, n_init=n_init, n_local=n_local)
        got = torch.full((wl.T, wl.topk), -7, dtype=torch.int32, device="cuda")
        capi.dsa_lightning_indexer(db.index_q, db.weights, db.index_pool, db.block_table, db.seq_lens, db.cu_q,
                                   wl.max_seq_len, wl.max_q_len, wl.topk, got, ws, n_init=n_init, n_local=n_local)
        assert torch.equal(got, ref)
    with pytest.raises(capi.DSAError):     # short workspace
        capi.dsa_lightning_indexer(db.index_q, db.weights, db.index_pool, db.block_table, db.seq_lens, db.cu_q,
                                   wl.max_seq_len, wl.max_q_len, wl.topk, got, ws[:1024])


def _li_case(name):
    if name == "cluster":   # long rows, few of them: the 2-CTA cluster top-k; row groups of 2
        return workloads.make_custom("li_oracle", 241, [500, 64, 3000, 17000, 40000, 70000], [1, 2, 3, 1, 1, 2],
                                     topk=256, heads=16)
    if name == "segments":   # 200 one-tile requests then 56 long ones: shares spanning many segments
        rng = np.random.default_rng(243)
        lens = rng.integers(1, 129, size=200).tolist() + rng.integers(5000, 6001, size=56).tolist()
        return workloads.make_custom("li_oracle_s", 243, lens, 1, topk=512, heads=16)
    rng = np.random.default_rng(242)   # many short rows: the one-CTA bitmap top-k
    lens = rng.integers(100, 12000, 90).tolist()
    return workloads.make_custom("li_oracle_b", 242, lens, rng.integers(1, 3, 90).tolist(), topk=512, heads=16)


@pytest.mark.parametrize("case", ["cluster", "bitmap", "segments"])
def test_lightning_indexer_matches_oracle(case):
    """The one-call indexer (histogram-fused: both cases have row groups of at most 2 rows) against
    the oracle: oracle.topk_forced on the oracle's logits, exactly wherever the k-th / (k+1)-th gap
    (with the forced positions at +inf) is outside the tie band, and a valid selection everywhere
    (forced positions kept, every other kept logit >= every dropped one up to the logit
    tolerance), with and without forced initial / local tokens; its logits stay in the workspace
    and match the oracle's."""
    from helpers import check_logits, oracle_pool, record
    from deepseek_sparse_attention_paged_gb300.pipeline import lightning_logits_offset
    wl = _li_case(case)
    assert wl.max_q_len < 4
    db = DeviceBatch(wl, with_latent=False)
    pool = oracle_pool(wl)
    rows = np.arange(wl.T)
    ref_lg, mag, bad = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                                             rows, db.ld, want_mag=True)
    assert bad == 0
    vis = wl.visible_lens()
    ws = torch.empty(capi.dsa_lightning_indexer_workspace_size(wl.T, wl.max_seq_len), dtype=torch.uint8,
                     device="cuda")
    off = lightning_logits_offset(wl.T)
    for n_init, n_local in ((0, 0), (2, 8)):
        got = torch.full((wl.T, wl.topk), -7, dtype=torch.int32, device="cuda")
        ws.fill_(0xAB)   # stale histograms / logits from elsewhere must not matter
        capi.dsa_lightning_indexer(db.index_q, db.weights, db.index_pool, db.block_table, db.seq_lens, db.cu_q,
                                   wl.max_seq_len, wl.max_q_len, wl.topk, got, ws, n_init=n_init, n_local=n_local)
        lg = ws[off:off + wl.T * db.ld * 4].view(torch.float32).view(wl.T, db.ld).cpu().numpy()
        check_logits(lg, ref_lg, mag, vis, key=f"lightning_indexer_vs_oracle/{case}")
        got = got.cpu().numpy()
        ref = oracle.topk_forced(ref_lg, wl.seq_lens, wl.cu_q, rows, wl.topk, n_init, n_local)
        exact = 0
        for r in rows:
            v = int(vis[r])
            row = ref_lg[r, :v].astype(np.float64).copy()
            forced = np.zeros(v, bool)
            forced[:min(n_init, v)] = True
            if n_local:
                forced[max(0, v - n_local):] = True
            row[forced] = np.inf
            assert np.all(np.isin(np.flatnonzero(forced), got[r])), f"row {r}: a forced position is missing"
            finite = row[np.isfinite(row)]
            if forced.sum() >= wl.topk or v <= wl.topk or kth_gap_ok(np.concatenate([row[forced], finite]), wl.topk):
                assert np.array_equal(got[r], ref[r]), f"row {r}: differs from the oracle outside the tie band"
                exact += 1
            check_topk_valid(got[r], row, wl.topk, mag[r, :v])
        record(f"lightning_indexer_vs_oracle/{case}", rows=len(rows), rows_exact=exact)
