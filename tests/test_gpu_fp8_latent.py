"""GPU parity of the FP8 latent-cache variant against the oracle, through the C ABI:
dsa_store_latent_fp8 (per-tensor E4M3 codes of the latent rows, by slot) bit for bit, and
dsa_sparse_mla_decode_fp8 (query quantised with q_scale, scores on E4M3 codes, values widened to
bf16) within the attention bar (2e-2 max-abs on the output, 1e-3 on lse)."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

from helpers import bf16_to_np_f64, check_attention, record

pytestmark = pytest.mark.gpu

K_SCALE = 0.0125   # ~ max |N(0,1)| / 448 over the synthetic caches: a few values saturate
Q_SCALE = 0.0125


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def test_store_latent_fp8_bit_exact():
    rng = np.random.default_rng(500)
    n, pages = 3000, 60
    lat = torch.randn(n, 576, generator=torch.Generator().manual_seed(500)).mul(2.0).to(torch.bfloat16)
    lat_bits = lat.view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    slots[3] = -1
    slots[9] = pages * 64 + 1
    ref = np.full((pages, 64, 576), 0x11, np.uint8)
    assert oracle.store_latent_fp8(lat_bits, slots, K_SCALE, ref) == 1
    pool = torch.full((pages, 64, 576), 0x11, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_store_latent_fp8(lat.cuda(), torch.from_numpy(slots).cuda(), K_SCALE, pool, dev_err=err)
    assert np.array_equal(pool.cpu().numpy(), ref)
    assert capi.dsa_read_device_error(err) == (capi.DSA_ERR_DEVICE_BOUNDS, capi.DSA_DEVERR_SLOT_RANGE)


def _fp8_cache(wl):
    """The workload's latent cache quantised by the GPU store (bit-exact with the oracle's store)."""
    lat = wl.latent_pool().reshape(-1, 576)
    pool = torch.empty((wl.num_pages, 64, 576), dtype=torch.uint8, device="cuda")
    slots = torch.arange(lat.shape[0], dtype=torch.int64, device="cuda")
    capi.dsa_store_latent_fp8(_dev_bf16(lat), slots, K_SCALE, pool)
    return pool


def _fp8_case(wl, idx, key, expect_bad=0):
    db = DeviceBatch(wl, with_latent=True, build_index_cache=False)
    pool = _fp8_cache(wl)
    kv8 = pool.cpu().numpy()
    ref_pool = oracle.quant_fp8_tensor(wl.latent_pool(), K_SCALE)
    assert np.array_equal(kv8, ref_pool.reshape(kv8.shape))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_sparse_mla_decode_fp8(db.mla_q, Q_SCALE, pool, K_SCALE, db.block_table, db.seq_lens, db.cu_q,
                                   torch.from_numpy(idx).cuda(), wl.scale, db.out, db.mla_ws, lse=db.lse, dev_err=err)
    out = bf16_to_np_f64(db.out)
    lse = db.lse.cpu().numpy().astype(np.float64)
    ref_o, ref_l = oracle.sparse_mla_fp8(wl.mla_q(), Q_SCALE, kv8, K_SCALE, wl.block_table, wl.seq_lens, wl.cu_q, idx,
                                         wl.scale, np.arange(wl.T))
    check_attention(out, lse, ref_o, ref_l, key=key)
    st, word = capi.dsa_read_device_error(err)
    assert (word != 0) == (expect_bad > 0)
    return db, out


def _random_idx(wl, k, fill, rng):
    idx = np.full((wl.T, k), -1, np.int32)
    vis = wl.visible_lens()
    for r in range(wl.T):
        n = min(int(fill * k), int(vis[r]))
        idx[r, :n] = np.sort(rng.choice(int(vis[r]), n, replace=False))
    return idx


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_fp8_mla_random_selection(H):
    rng = np.random.default_rng(510 + H)
    wl = workloads.make_custom("mla8", 510 + H, [3000, 700, 129], 1, topk=512, heads=H)
    _fp8_case(wl, _random_idx(wl, 512, 0.9, rng), "fp8_mla/random")


def test_fp8_mla_several_splits_empty_row_and_bad_entries():
    rng = np.random.default_rng(520)
    wl = workloads.make_custom("mla8s", 520, [5000, 2048, 2100, 300], 1, topk=2048, heads=128)
    idx = _random_idx(wl, 2048, 1.0, rng)
    idx[1] = -1                       # no valid entry: out = 0, lse = -inf
    idx[2, 7] = 2100                  # == v: not visible (skipped, reported)
    _, out = _fp8_case(wl, idx, "fp8_mla/splits", expect_bad=1)
    assert np.all(out[1] == 0.0)


def test_fp8_mla_full_size_every_row():
    """Every row of the 64-request 64K decode batch, selections from the step's own top-k."""
    wl = workloads.make("decode_b64_logu64k")
    db = DeviceBatch(wl)
    db.step()
    torch.cuda.synchronize()
    idx = db.idx.cpu().numpy()
    pool = _fp8_cache(wl)
    kv8 = pool.cpu().numpy()
    capi.dsa_sparse_mla_decode_fp8(db.mla_q, Q_SCALE, pool, K_SCALE, db.block_table, db.seq_lens, db.cu_q, db.idx,
                                   wl.scale, db.out, db.mla_ws, lse=db.lse)
    out = bf16_to_np_f64(db.out)
    lse = db.lse.cpu().numpy().astype(np.float64)
    ref_o, ref_l = oracle.sparse_mla_fp8(wl.mla_q(), Q_SCALE, kv8, K_SCALE, wl.block_table, wl.seq_lens, wl.cu_q, idx,
                                         wl.scale, np.arange(wl.T))
    check_attention(out, lse, ref_o, ref_l, key="fp8_mla/decode_b64_logu64k")
    record("fp8_mla/decode_b64_logu64k", full_rows=wl.T)
