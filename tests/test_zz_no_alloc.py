"""dsa_sparse_mla_decode_noalloc: the sparse-MLA entry point for callers that may not allocate device
memory (it takes no workspace and uses the library's fixed 16 MiB scratch instead).

Checked through the C ABI against the oracle and against the workspace-taking dsa_sparse_mla_decode
on the same inputs,
on two calls in a row with different inputs (the scratch is shared between calls and keeps the
previous call's contents), for device memory left unchanged by a call after the first, and for the
size limit.  This file is collected last so that a run that
stops at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

from helpers import bf16_to_np_f64, check_attention

pytestmark = pytest.mark.gpu

ATTN_ABS = 2e-2   # the attention tolerance of the parity tests


def _inputs(seed, lens, heads, k):
    wl = workloads.make_custom("noalloc", seed, lens, 1, topk=k, heads=heads)
    db = DeviceBatch(wl, with_latent=True, build_index_cache=False)
    rng = np.random.default_rng(seed)
    idx = np.full((wl.T, k), -1, np.int32)
    for r, v in enumerate(wl.visible_lens()):
        n = min(k, int(v))
        idx[r, :n] = np.sort(rng.choice(int(v), n, replace=False))
    return wl, db, torch.from_numpy(idx).cuda()


def _with_workspace(wl, db, idx):
    out = torch.empty_like(db.out)
    lse = torch.empty_like(db.lse)
    capi.dsa_sparse_mla_decode(db.mla_q, db.kv_pool, db.block_table, db.seq_lens, db.cu_q, idx, wl.scale, out,
                               db.mla_ws, lse=lse)
    return out, lse


def _no_alloc(wl, db, idx):
    out = torch.full_like(db.out, float("nan"))
    lse = torch.full_like(db.lse, float("nan"))
    capi.dsa_sparse_mla_decode_noalloc(db.mla_q, db.kv_pool, db.block_table, db.seq_lens, db.cu_q, idx, wl.scale,
                                       out, lse=lse)
    return out, lse


def _compare(a, b):
    oa, la = a
    ob, lb = b
    torch.cuda.synchronize()
    assert float((oa.float() - ob.float()).abs().max()) <= ATTN_ABS
    fin = torch.isfinite(la)
    assert torch.equal(fin, torch.isfinite(lb))
    assert float((la[fin] - lb[fin]).abs().max()) <= 1e-3 if bool(fin.any()) else True


def _against_oracle(wl, idx, got, key):
    torch.cuda.synchronize()
    rows = np.arange(wl.T)
    ref_o, ref_l = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                     idx.cpu().numpy(), wl.scale, rows)
    check_attention(bf16_to_np_f64(got[0]), got[1].cpu().numpy().astype(np.float64), ref_o, ref_l, key=key)


def test_no_alloc_matches_workspace_entry_point_twice_in_a_row():
    # first call: 3 rows, 128 heads, k = 2048 (8 splits: 6.3 MB of the 16 MiB scratch)
    wl1, db1, idx1 = _inputs(901, [4000, 2500, 9000], 128, 2048)
    got1 = _no_alloc(wl1, db1, idx1)
    _compare(got1, _with_workspace(wl1, db1, idx1))
    _against_oracle(wl1, idx1, got1, "no_alloc/first_call")
    # second call, different shapes and values: nothing left over from the first call may leak in
    wl2, db2, idx2 = _inputs(902, [700, 3000, 150, 2048, 64], 64, 512)
    idx2[2] = -1                                      # an empty row: out = 0, lse = -inf
    got = _no_alloc(wl2, db2, idx2)
    _compare(got, _with_workspace(wl2, db2, idx2))
    _against_oracle(wl2, idx2, got, "no_alloc/second_call")
    assert float(got[0][2].abs().max()) == 0.0 and bool(torch.isneginf(got[1][2]).all())


def test_no_alloc_call_after_the_first_leaves_device_memory_unchanged():
    """After one call on the device (which may load the library's device code and with it the
    fixed scratch), further calls take no device memory: the driver's free-memory count is the
    same before and after a call that uses the scratch (8 splits of 3 rows)."""
    wl, db, idx = _inputs(904, [4000, 2500, 9000], 128, 2048)
    assert capi.dsa_sparse_mla_workspace_size(wl.T, wl.heads, wl.topk) > 0
    out = torch.empty_like(db.out)
    lse = torch.empty_like(db.lse)

    def call():
        capi.dsa_sparse_mla_decode_noalloc(db.mla_q, db.kv_pool, db.block_table, db.seq_lens, db.cu_q, idx,
                                           wl.scale, out, lse=lse)

    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    _compare((out, lse), _with_workspace(wl, db, idx))


def test_no_alloc_rejects_problems_larger_than_its_scratch():
    wl, db, idx = _inputs(903, [2048] * 16, 128, 2048)   # 16 rows x 128 heads x 4 splits > 16 MiB
    assert capi.dsa_sparse_mla_workspace_size(wl.T, wl.heads, wl.topk) > (16 << 20)
    with pytest.raises(capi.DSAError) as e:
        _no_alloc(wl, db, idx)
    assert e.value.status == capi.DSA_ERR_UNSUPPORTED
