"""GPU parity of the projections around the absorbed attention (dsa_mla_absorb_q, dsa_mla_v_up)
against the CPU oracle, through the C ABI.

Tolerance: the oracle rounds the exact sum once to bf16; the kernel accumulates in fp32 on the
tensor cores and rounds once.  When the two sums fall on either side of a rounding boundary they
land on neighbouring bf16 values, one unit in the last place apart (up to 2^-7 relative: bf16
keeps 8 significant bits); the fp32 accumulation error is bounded by K * 2^-24 times the
magnitude sum |x| |w| (K <= 512 terms): |gpu - ref| <= 2^-7 |ref| + 2^-14 * mag."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _val(bits) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits)


def _check(got_bits, ref_bits, mag):
    got, ref = _val(got_bits), _val(ref_bits)
    bound = 2.0 ** -7 * np.abs(ref) + 2.0 ** -14 * mag
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max err {err.max()} (worst ratio {np.max(err / np.maximum(bound, 1e-30))})"


@pytest.mark.parametrize("T,H", [(64, 128), (1, 8), (100, 16), (300, 4), (1100, 8), (4096, 8)])
def test_absorb_matches_oracle_into_strided_query(T, H):
    g = torch.Generator().manual_seed(700 + T + H)
    q = torch.randn(T, H, 192, generator=g).to(torch.bfloat16).cuda()             # [q_nope 128 | q_pe 64]
    w = (torch.randn(H, 128, 512, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
    mla_q = torch.full((T, H, 576), 7.0, dtype=torch.bfloat16, device="cuda")       # sentinel
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_mla_absorb_q(q[..., :128], w, mla_q[..., :512], dev_err=err)
    ref, mag = oracle.mla_absorb_q(_bits(q[..., :128]), _bits(w), want_mag=True)
    _check(_bits(mla_q[..., :512]), ref, mag)
    assert bool((mla_q[..., 512:] == 7.0).all())                                   # rope columns untouched
    assert capi.dsa_read_device_error(err) == (0, 0)


@pytest.mark.parametrize("T,H", [(64, 128), (257, 4), (3, 2)])
def test_v_up_matches_oracle(T, H):
    g = torch.Generator().manual_seed(710 + T + H)
    o = torch.randn(T, H, 512, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(H, 512, 128, generator=g) / math.sqrt(512)).to(torch.bfloat16).cuda()
    out = torch.full((T, H * 128), 3.0, dtype=torch.bfloat16, device="cuda")
    capi.dsa_mla_v_up(o, w, out.view(T, H, 128))
    ref, mag = oracle.mla_v_up(_bits(o), _bits(w), want_mag=True)
    _check(_bits(out.view(T, H, 128)), ref, mag)


def test_absorb_attention_v_up_chain():
    """q_nope -> absorbed query (kernel) -> sparse MLA (kernel) -> v_up (kernel) against the same
    chain in the oracle, on the tiny workload's latent cache and a full selection."""
    wl = workloads.make_custom("chain", 720, [300, 1000], 1, topk=256, heads=16)
    db = DeviceBatch(wl, with_latent=True, build_index_cache=False)
    H, T = wl.heads, wl.T
    g = torch.Generator().manual_seed(721)
    q = torch.randn(T, H, 192, generator=g).to(torch.bfloat16).cuda()
    w_uk_t = (torch.randn(H, 128, 512, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
    w_uv = (torch.randn(H, 512, 128, generator=g) / math.sqrt(512)).to(torch.bfloat16).cuda()
    db.mla_q[..., 512:] = q[..., 128:]
    capi.dsa_mla_absorb_q(q[..., :128], w_uk_t, db.mla_q[..., :512])
    rng = np.random.default_rng(722)
    idx = np.full((T, 256), -1, np.int32)
    for r, v in enumerate(wl.visible_lens()):
        idx[r, :min(256, v)] = np.sort(rng.choice(v, min(256, v), replace=False))
    db.sparse_mla(idx=torch.from_numpy(idx).cuda())
    out = torch.empty(T, H * 128, dtype=torch.bfloat16, device="cuda")
    capi.dsa_mla_v_up(db.out, w_uv, out.view(T, H, 128))
    # oracle chain: its own absorbed query (bf16), its attention (float64, rounded to bf16), its v_up
    ql = oracle.mla_absorb_q(_bits(q[..., :128]), _bits(w_uk_t))
    q_abs = np.concatenate([ql, _bits(q[..., 128:])], axis=-1)
    o_ref, _ = oracle.sparse_mla(q_abs, wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, idx, wl.scale,
                                 np.arange(T))
    o_bits = oracle.f64_to_bf16_array(o_ref)
    ref, mag = oracle.mla_v_up(o_bits, _bits(w_uv), want_mag=True)
    got = _val(_bits(out.view(T, H, 128)))
    # attention output within the attention bar (2e-2 on unit data) propagates through W_UV:
    # |delta out| <= 2e-2 * sum_l |W_UV[l, v]| + the projection's own bound
    w_abs = np.abs(_val(_bits(w_uv))).sum(axis=1)                                   # [H, 128]
    bound = 2e-2 * w_abs[None] + 2.0 ** -7 * np.abs(_val(ref)) + 2.0 ** -14 * mag
    assert np.all(np.abs(got - _val(ref)) <= bound)


@pytest.mark.parametrize("T", [64, 5])
def test_v_up_into_output_rows_without_16_byte_strides(T):
    # head stride 130 elements: the 16-byte row stores do not apply, each value is stored alone
    H = 8
    g = torch.Generator().manual_seed(720 + T)
    o = torch.randn(T, H, 512, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(H, 512, 128, generator=g) / math.sqrt(512)).to(torch.bfloat16).cuda()
    out = torch.full((T, H, 130), 3.0, dtype=torch.bfloat16, device="cuda")
    capi.dsa_mla_v_up(o, w, out[..., :128])
    ref, mag = oracle.mla_v_up(_bits(o), _bits(w), want_mag=True)
    _check(_bits(out[..., :128]), ref, mag)
    assert bool((out[..., 128:] == 3.0).all())


def test_bad_strides_are_rejected():
    q = torch.zeros(4, 2, 132, dtype=torch.bfloat16, device="cuda")               # head stride 132: not 16-byte
    w = torch.zeros(2, 128, 512, dtype=torch.bfloat16, device="cuda")
    ql = torch.zeros(4, 2, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(capi.DSAError):
        capi.dsa_mla_absorb_q(q[..., :128], w, ql)
