"""CPU checks of the C-ABI library: it builds, loads without a GPU, and exports every function
that include/dsa.h declares.  No compute call is made here."""
import ctypes
import os

import pytest

from deepseek_sparse_attention_paged_gb300 import build, capi


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(capi.LIB_PATH)


def test_header_declares_the_four_path_calls():
    names = capi.header_functions()
    for n in ("dsa_store_index_k", "dsa_indexer_logits", "dsa_topk", "dsa_sparse_mla_decode"):
        assert n in names


def test_library_exports_every_header_symbol(lib):
    for name in capi.header_functions():
        assert hasattr(lib, name), f"{name} declared in include/dsa.h but not exported"


def test_status_strings_and_host_side_validation(lib):
    capi.load()
    assert capi._lib.dsa_status_str(0) == b"ok"
    assert capi._lib.dsa_status_str(2).startswith(b"unsupported")
    # argument checks return before touching the GPU
    L = capi._lib
    assert L.dsa_store_index_k(None, None, 0, None, 0, 64, None, None) == 0          # n = 0: nothing to do
    assert L.dsa_store_index_k(None, None, 4, None, 1, 32, None, None) == 2          # page size 32
    assert L.dsa_store_index_k(None, None, 4, None, 1, 64, None, None) == 1          # null pointers
    assert L.dsa_topk(None, 0, None, None, 1, 0, 0, 1, 0, None, None, 0, None) == 2  # k = 0
    assert L.dsa_topk(None, 0, None, None, 1, 0, 0, 1, 4096, None, None, 0, None) == 2
    assert L.dsa_sparse_mla_decode(None, None, 0, None, 0, None, None, 1, None, 64, 1, 24, 0.1, None, None,
                                   None, 0, None, None) == 2                          # H = 24
    assert L.dsa_indexer_logits(None, None, None, 0, None, 0, None, None, 1, 10, 1, 0, 1, None, 10, 0x40,
                                None, 0, None, None) == 1                             # unknown flag
    assert L.dsa_indexer_logits(None, None, None, 0, None, 0, None, None, 1, 10, 1, 0, 1, None, 10, 0,
                                None, 0, None, None) == 1                             # null pointers
    assert L.dsa_indexer_logits_workspace_size(3) == 3 * (64 * 128 + 64 * 4)          # codes + gates per row
    assert L.dsa_indexer_logits_workspace_size(0) == 0
    assert L.dsa_sparse_mla_workspace_size(64, 128, 2048) == 0     # one split per row: no scratch
    assert L.dsa_sparse_mla_workspace_size(16, 128, 2048) > 0      # few rows: split over k


def test_host_side_validation_of_the_next_row_calls(lib):
    """Argument checks of the prologue, projection, forced top-k and one-call indexer entry points
    (all return before any CUDA call)."""
    capi.load()
    L = capi._lib
    f = ctypes.c_float
    # key prologue: page size, unknown flag, nothing to do, null pointers
    assert L.dsa_store_index_k_prologue(None, None, None, f(1e-6), None, 8, None, None, 4, None, 1, 32, 0,
                                        None, None) == 2
    assert L.dsa_store_index_k_prologue(None, None, None, f(1e-6), None, 8, None, None, 4, None, 1, 64, 0x40,
                                        None, None) == 1
    assert L.dsa_store_index_k_prologue(None, None, None, f(1e-6), None, 8, None, None, 0, None, 1, 64, 0,
                                        None, None) == 0
    assert L.dsa_store_index_k_prologue(None, None, None, f(1e-6), None, 8, None, None, 4, None, 1, 64,
                                        capi.DSA_NORM_RMS | capi.DSA_SCALE_UE8M0, None, None) == 1
    # query rope
    assert L.dsa_indexer_rope_q(None, None, 8, None, 2, 0x1, None, None, None) == 1   # flag of another call
    assert L.dsa_indexer_rope_q(None, None, 8, None, 0, 0, None, None, None) == 0
    assert L.dsa_indexer_rope_q(None, None, 8, None, -1, 0, None, None, None) == 1
    # projections: empty, null, misaligned base, stride not a multiple of 8 elements, overlapping outputs
    assert L.dsa_mla_absorb_q(None, 0, 0, None, 0, 128, None, 0, 0, None, None) == 0
    assert L.dsa_mla_absorb_q(None, 24576, 192, None, 4, 128, None, 73728, 576, None, None) == 1
    assert L.dsa_mla_absorb_q(ctypes.c_void_p(0x1008), 24576, 192, ctypes.c_void_p(0x2000), 4, 128,
                              ctypes.c_void_p(0x3000), 73728, 576, None, None) == 1
    assert L.dsa_mla_absorb_q(ctypes.c_void_p(0x1000), 24576, 196, ctypes.c_void_p(0x2000), 4, 128,
                              ctypes.c_void_p(0x3000), 73728, 576, None, None) == 1
    assert L.dsa_mla_v_up(ctypes.c_void_p(0x1000), 65536, 512, ctypes.c_void_p(0x2000), 4, 128,
                          ctypes.c_void_p(0x3000), 16384, 64, None, None) == 1            # head stride < 128
    # forced top-k
    assert L.dsa_topk_forced(None, 0, None, None, 1, 0, 0, 1, 16, -1, 0, None, None, 0, None) == 1
    assert L.dsa_topk_forced(None, 0, None, None, 1, 0, 0, 1, 0, 0, 0, None, None, 0, None) == 2
    # one-call indexer: k, empty batch, missing or short workspace
    assert L.dsa_lightning_indexer(None, None, None, 0, None, 0, None, None, 1, 100, 1, 2, 0, 0, 0, 0, None,
                                   None, 0, None, None) == 1
    assert L.dsa_lightning_indexer(None, None, None, 0, None, 0, None, None, 1, 100, 1, 0, 16, 0, 0, 0, None,
                                   None, 0, None, None) == 0
    need = L.dsa_lightning_indexer_workspace_size(2, 100)
    # the per-row histograms, the logits call's scratch, the logits (each part 256-byte aligned)
    assert need == 2 * 4096 * 4 + (2 * (64 * 128 + 64 * 4) + 255) // 256 * 256 + 2 * 100 * 4
    assert L.dsa_lightning_indexer(None, None, None, 0, None, 0, None, None, 1, 100, 1, 2, 16, 0, 0, 0,
                                   ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), need - 16, None, None) == 1


def test_host_side_validation_of_the_c8_calls(lib):
    """The int8 ("c8") cache's store and logits calls check their arguments before any CUDA call."""
    capi.load()
    L = capi._lib
    assert L.dsa_store_index_k_c8(None, None, 0, None, 0, 64, None, None) == 0      # n = 0
    assert L.dsa_store_index_k_c8(None, None, 4, None, 1, 32, None, None) == 2      # page size 32
    assert L.dsa_store_index_k_c8(None, None, 4, None, 1, 64, None, None) == 1      # null pointers
    assert L.dsa_store_index_k_c8(ctypes.c_void_p(0x1008), ctypes.c_void_p(0x2000), 4, ctypes.c_void_p(0x3000), 1,
                                  64, None, None) == 1                              # misaligned keys
    # f16 query codes (64 heads x 128 dims x 2 B) + fp32 gates per row
    assert L.dsa_indexer_logits_c8_workspace_size(3) == 3 * (64 * 128 * 2 + 64 * 4)
    assert L.dsa_indexer_logits_c8_workspace_size(0) == 0
    assert L.dsa_indexer_logits_c8(None, None, None, 0, None, 0, None, None, 1, 10, 1, 0, 1, None, 10, None, 0,
                                   None, None) == 1                                 # null pointers
    assert L.dsa_indexer_logits_c8(None, None, None, 0, None, 0, None, None, 0, 10, 1, 0, 1, None, 10, None, 0,
                                   None, None) == 0                                 # empty batch


def test_host_side_validation_of_the_compressed_kv_calls(lib):
    """The compressed-KV attention and the DSA_KEYS_CMP4 flag are checked before any CUDA call."""
    capi.load()
    L = capi._lib
    f = ctypes.c_float
    # T = 0: nothing to do; ratio 3 and window 0 unsupported; null pointers rejected
    assert L.dsa_sparse_attn_swa_cmp(None, None, 0, None, 0, None, 0, None, 0, None, None, 1, None, 64, 128, 4, None,
                                     0, 128, f(0.1), None, None, None, 0, None, None) == 0
    assert L.dsa_sparse_attn_swa_cmp(None, None, 0, None, 0, None, 0, None, 0, None, None, 1, None, 64, 128, 3, None,
                                     1, 128, f(0.1), None, None, None, 0, None, None) == 2
    assert L.dsa_sparse_attn_swa_cmp(None, None, 0, None, 0, None, 0, None, 0, None, None, 1, None, 64, 0, 4, None,
                                     1, 128, f(0.1), None, None, None, 0, None, None) == 2
    assert L.dsa_sparse_attn_swa_cmp(None, None, 1, None, 1, None, 1, None, 1, None, None, 1, None, 64, 128, 4, None,
                                     1, 128, f(0.1), None, None, None, 0, None, None) == 1
    # split-K partials only when the rows are split (as dsa_sparse_mla_workspace_size for window + k entries)
    assert L.dsa_sparse_attn_swa_cmp_workspace_size(64, 128, 128, 512) == L.dsa_sparse_mla_workspace_size(64, 128, 640)
    assert L.dsa_sparse_attn_swa_cmp_workspace_size(2, 16, 128, 2048) == L.dsa_sparse_mla_workspace_size(2, 16, 2176)
    assert L.dsa_sparse_attn_swa_cmp_workspace_size(0, 16, 128, 64) == 0
    # the compressed-keys flag is a known flag of the logits call (null pointers are what is rejected)
    assert L.dsa_indexer_logits(None, None, None, 0, None, 0, None, None, 1, 10, 1, 0, 1, None, 10,
                                capi.DSA_KEYS_CMP4, None, 0, None, None) == 1


def test_host_side_validation_of_the_fp8_latent_calls(lib):
    """The FP8 latent store and attention check their arguments before any CUDA call."""
    capi.load()
    L = capi._lib
    f = ctypes.c_float
    assert L.dsa_store_latent_fp8(None, None, 0, f(0.5), None, 1, None, None) == 0          # n = 0
    assert L.dsa_store_latent_fp8(None, None, 4, f(0.0), None, 1, None, None) == 1          # k_scale <= 0
    assert L.dsa_store_latent_fp8(None, None, 4, f(float("inf")), None, 1, None, None) == 1  # k_scale not finite
    assert L.dsa_store_latent_fp8(None, None, 4, f(0.5), None, 1, None, None) == 1          # null pointers
    args = [None, f(0.5), None, f(0.5), 1, None, 1, None, None, 1, None, 64, 1, 128, f(0.1), None, None, None, 0,
            None, None]
    a = list(args); a[11] = 0
    assert L.dsa_sparse_mla_decode_fp8(*a) == 2                                              # k = 0
    a = list(args); a[13] = 24
    assert L.dsa_sparse_mla_decode_fp8(*a) == 2                                              # H = 24
    a = list(args); a[12] = 0
    assert L.dsa_sparse_mla_decode_fp8(*a) == 0                                              # T = 0
    assert L.dsa_sparse_mla_decode_fp8(*args) == 1                                           # null pointers

