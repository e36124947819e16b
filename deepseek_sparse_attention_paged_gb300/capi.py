"""Thin Python binding of the C ABI in ``include/dsa.h`` (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch CUDA tensors, checks
their dtype/shape/contiguity, passes raw device pointers and the caller's current CUDA stream,
and raises :class:`DSAError` on a non-OK status.  All computation happens in the CUDA library;
if the library is missing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa_gb300.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "dsa.h")

DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CUDA = 3
DSA_ERR_DEVICE_BOUNDS = 4
DSA_ERR_TIMEOUT = 5
DSA_DEVERR_SLOT_RANGE = 0x1
DSA_DEVERR_PAGE_RANGE = 0x2
DSA_DEVERR_INDEX_RANGE = 0x4
DSA_DEVERR_TIMEOUT = 0x8
DSA_DEVERR_POSITION = 0x10
DSA_Q_ROTATE = 0x1
DSA_NORM_RMS = 0x2
DSA_ROPE_INTERLEAVED = 0x4
DSA_K_NO_ROTATE = 0x8
DSA_SCALE_UE8M0 = 0x10
DSA_KEYS_CMP4 = 0x20          # the index cache holds compressed keys, one per 4 tokens
PAGE_SIZE = 64
INDEX_PAGE_BYTES = 64 * 132
C8_PAGE_BYTES = 64 * 130      # int8 index cache page: 64 x 128 codes + 64 fp16 scales
LATENT_DIM = 576
VALUE_DIM = 512
MAX_TOPK = 2048

_lib = None
_launches = 0   # kernels this process enqueued through the binding (graph captures included)


def launch_count() -> int:
    """Number of CUDA kernels enqueued through this binding so far (a captured launch counts once,
    at capture)."""
    return _launches


def _count(n: int) -> None:
    global _launches
    _launches += n


class DSAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _lib.dsa_status_str(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    sigs = {
        "dsa_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "dsa_store_index_k": (ctypes.c_int, [P, P, i64, P, i64, i32, P, P]),
        "dsa_store_index_k_prologue": (ctypes.c_int, [P, P, P, ctypes.c_float, P, i64, P, P, i64, P, i64, i32, u32,
                                                      P, P]),
        "dsa_indexer_rope_q": (ctypes.c_int, [P, P, i64, P, i64, u32, P, P, P]),
        "dsa_mla_absorb_q": (ctypes.c_int, [P, i64, i64, P, i32, i32, P, i64, i64, P, P]),
        "dsa_mla_v_up": (ctypes.c_int, [P, i64, i64, P, i32, i32, P, i64, i64, P, P]),
        "dsa_indexer_logits_workspace_size": (sz, [i32]),
        "dsa_indexer_logits": (ctypes.c_int, [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, P, i64, u32,
                                              P, sz, P, P]),
        "dsa_topk_workspace_size": (sz, [i32, i32, i32]),
        "dsa_topk": (ctypes.c_int, [P, i64, P, P, i32, i32, i32, i32, i32, P, P, sz, P]),
        "dsa_topk_forced": (ctypes.c_int, [P, i64, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, sz, P]),
        "dsa_lightning_indexer_workspace_size": (sz, [i32, i32]),
        "dsa_lightning_indexer": (ctypes.c_int, [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, u32,
                                                 P, P, sz, P, P]),
        "dsa_sparse_mla_workspace_size": (sz, [i32, i32, i32]),
        "dsa_sparse_mla_decode": (ctypes.c_int, [P, P, i64, P, i32, P, P, i32, P, i32, i32, i32, ctypes.c_float,
                                                 P, P, P, sz, P, P]),
        "dsa_read_device_error": (ctypes.c_int, [P, P, P]),
        "dsa_selftest_wait_timeout": (ctypes.c_int, [P, ctypes.c_uint64, P]),
        "dsa_sparse_mla_decode_noalloc": (ctypes.c_int, [P, P, i64, P, i32, P, P, i32, P, i32, i32, i32,
                                                         ctypes.c_float, P, P, P, P]),
        "dsa_store_latent_fp8": (ctypes.c_int, [P, P, i64, ctypes.c_float, P, i64, P, P]),
        "dsa_store_index_k_c8": (ctypes.c_int, [P, P, i64, P, i64, i32, P, P]),
        "dsa_sparse_attn_swa_cmp_workspace_size": (sz, [i32, i32, i32, i32]),
        "dsa_sparse_attn_swa_cmp": (ctypes.c_int, [P, P, i64, P, i32, P, i64, P, i32, P, P, i32, P, i32, i32, i32, P,
                                                   i32, i32, ctypes.c_float, P, P, P, sz, P, P]),
        "dsa_indexer_logits_c8_workspace_size": (sz, [i32]),
        "dsa_indexer_logits_c8": (ctypes.c_int, [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, P, i64, P, sz,
                                                 P, P]),
        "dsa_sparse_mla_decode_fp8": (ctypes.c_int, [P, ctypes.c_float, P, ctypes.c_float, i64, P, i32, P, P, i32, P,
                                                     i32, i32, i32, ctypes.c_float, P, P, P, sz, P, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(path: str = HEADER):
    """Names of the functions declared in ``include/dsa.h``."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(cond: bool, what: str):
    if not cond:
        raise ValueError(what)


def _cuda(t: torch.Tensor, dtype, name: str):
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")
    _need(t.is_contiguous(), f"{name} must be contiguous")


def _rows(t: torch.Tensor, dtype, name: str):
    """2-D tensor whose rows may be strided (the row stride is passed as ld) but are dense."""
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")
    _need(t.dim() == 2 and (t.stride(1) == 1 or t.shape[1] <= 1), f"{name} rows must be dense")


def _check(fn: str, status: int):
    if status != DSA_OK:
        raise DSAError(fn, status)


def dsa_store_index_k(k_bf16: torch.Tensor, slot_mapping: torch.Tensor, index_k_pool: torch.Tensor,
                      dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    lib = load()
    _cuda(k_bf16, torch.bfloat16, "k_bf16")
    _cuda(slot_mapping, torch.int64, "slot_mapping")
    _cuda(index_k_pool, torch.uint8, "index_k_pool")
    _need(k_bf16.dim() == 2 and k_bf16.shape[1] == 128, "k_bf16 must be [n, 128]")
    _need(slot_mapping.numel() == k_bf16.shape[0], "slot_mapping must have n entries")
    _need(index_k_pool.dim() == 2 and index_k_pool.shape[1] == INDEX_PAGE_BYTES, "pool must be [pages, 8448]")
    _check("dsa_store_index_k", lib.dsa_store_index_k(
        _ptr(k_bf16), _ptr(slot_mapping), k_bf16.shape[0], _ptr(index_k_pool), index_k_pool.shape[0], PAGE_SIZE,
        _ptr(dev_err), _stream(stream)))
    _count(1 if k_bf16.shape[0] > 0 else 0)


def dsa_store_index_k_prologue(k_raw_bf16: torch.Tensor, norm_weight: torch.Tensor,
                               norm_bias: Optional[torch.Tensor], eps: float, cos_sin_cache: torch.Tensor,
                               positions: torch.Tensor, slot_mapping: torch.Tensor, index_k_pool: torch.Tensor,
                               flags: int = 0, dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Key norm (LayerNorm, or RMSNorm with DSA_NORM_RMS), rotary embedding at `positions`, then
    the rotate / quantise / paged store of dsa_store_index_k (no rotation with DSA_K_NO_ROTATE)."""
    lib = load()
    _cuda(k_raw_bf16, torch.bfloat16, "k_raw_bf16")
    _cuda(norm_weight, torch.float32, "norm_weight")
    if not flags & DSA_NORM_RMS:
        _need(norm_bias is not None, "LayerNorm needs norm_bias")
    if norm_bias is not None:
        _cuda(norm_bias, torch.float32, "norm_bias")
        _need(norm_bias.numel() == 128, "norm_bias must have 128 entries")
    _cuda(cos_sin_cache, torch.float32, "cos_sin_cache")
    _cuda(positions, torch.int64, "positions")
    _cuda(slot_mapping, torch.int64, "slot_mapping")
    _cuda(index_k_pool, torch.uint8, "index_k_pool")
    _need(k_raw_bf16.dim() == 2 and k_raw_bf16.shape[1] == 128, "k_raw_bf16 must be [n, 128]")
    _need(norm_weight.numel() == 128, "norm_weight must have 128 entries")
    _need(cos_sin_cache.dim() == 2 and cos_sin_cache.shape[1] == 64, "cos_sin_cache must be [max_position, 64]")
    n = k_raw_bf16.shape[0]
    _need(positions.numel() == n and slot_mapping.numel() == n, "positions / slot_mapping must have n entries")
    _need(index_k_pool.dim() == 2 and index_k_pool.shape[1] == INDEX_PAGE_BYTES, "pool must be [pages, 8448]")
    _check("dsa_store_index_k_prologue", lib.dsa_store_index_k_prologue(
        _ptr(k_raw_bf16), _ptr(norm_weight), _ptr(norm_bias), float(eps), _ptr(cos_sin_cache),
        cos_sin_cache.shape[0], _ptr(positions), _ptr(slot_mapping), n, _ptr(index_k_pool), index_k_pool.shape[0],
        PAGE_SIZE, flags, _ptr(dev_err), _stream(stream)))
    _count(1 if n > 0 else 0)


def dsa_indexer_rope_q(q_raw_bf16: torch.Tensor, cos_sin_cache: torch.Tensor, positions: torch.Tensor,
                       q_out_bf16: torch.Tensor, flags: int = 0, dev_err: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """Rotary embedding of the first 64 dims of every head of the indexer query [T, 64, 128]
    (q_out_bf16 may be q_raw_bf16)."""
    lib = load()
    _cuda(q_raw_bf16, torch.bfloat16, "q_raw_bf16")
    _cuda(q_out_bf16, torch.bfloat16, "q_out_bf16")
    _cuda(cos_sin_cache, torch.float32, "cos_sin_cache")
    _cuda(positions, torch.int64, "positions")
    _need(q_raw_bf16.dim() == 3 and tuple(q_raw_bf16.shape[1:]) == (64, 128), "q_raw_bf16 must be [T, 64, 128]")
    _need(q_out_bf16.shape == q_raw_bf16.shape, "q_out_bf16 must match q_raw_bf16")
    _need(cos_sin_cache.dim() == 2 and cos_sin_cache.shape[1] == 64, "cos_sin_cache must be [max_position, 64]")
    T = q_raw_bf16.shape[0]
    _need(positions.numel() == T, "positions must have T entries")
    _check("dsa_indexer_rope_q", lib.dsa_indexer_rope_q(
        _ptr(q_raw_bf16), _ptr(cos_sin_cache), cos_sin_cache.shape[0], _ptr(positions), T, flags,
        _ptr(q_out_bf16), _ptr(dev_err), _stream(stream)))
    _count(1 if T > 0 else 0)


def _strided3(t: torch.Tensor, inner: int, name: str):
    """(row stride, head stride) of a [T, H, inner] bf16 CUDA view whose last dim is dense."""
    _need(t.is_cuda and t.dtype == torch.bfloat16, f"{name} must be a bf16 CUDA tensor")
    _need(t.dim() == 3 and t.shape[2] == inner and (t.stride(2) == 1), f"{name} must be [T, H, {inner}], last dim dense")
    return t.stride(0), t.stride(1)


def dsa_mla_absorb_q(q_nope: torch.Tensor, w_uk_t: torch.Tensor, ql: torch.Tensor,
                     dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """ql[t, n, :512] = q_nope[t, n, :128] @ w_uk_t[n] (q_nope / ql may be strided views, e.g.
    q[..., :128] of a [T, H, 192] projection and out[..., :512] of the [T, H, 576] MLA query)."""
    lib = load()
    qs_t, qs_n = _strided3(q_nope, 128, "q_nope")
    os_t, os_n = _strided3(ql, 512, "ql")
    _cuda(w_uk_t, torch.bfloat16, "w_uk_t")
    T, H = q_nope.shape[0], q_nope.shape[1]
    _need(tuple(w_uk_t.shape) == (H, 128, 512), "w_uk_t must be [H, 128, 512]")
    _need(tuple(ql.shape[:2]) == (T, H), "ql must be [T, H, 512]")
    _check("dsa_mla_absorb_q", lib.dsa_mla_absorb_q(_ptr(q_nope), qs_t, qs_n, _ptr(w_uk_t), T, H, _ptr(ql), os_t, os_n,
                                                    _ptr(dev_err), _stream(stream)))
    _count(1 if T > 0 and H > 0 else 0)


def dsa_mla_v_up(o_lat: torch.Tensor, w_uv: torch.Tensor, out: torch.Tensor,
                 dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """out[t, n, :128] = o_lat[t, n, :512] @ w_uv[n] (out may be a [T, H, 128] view of [T, H * 128])."""
    lib = load()
    is_t, is_n = _strided3(o_lat, 512, "o_lat")
    os_t, os_n = _strided3(out, 128, "out")
    _cuda(w_uv, torch.bfloat16, "w_uv")
    T, H = o_lat.shape[0], o_lat.shape[1]
    _need(tuple(w_uv.shape) == (H, 512, 128), "w_uv must be [H, 512, 128]")
    _need(tuple(out.shape[:2]) == (T, H), "out must be [T, H, 128]")
    _check("dsa_mla_v_up", lib.dsa_mla_v_up(_ptr(o_lat), is_t, is_n, _ptr(w_uv), T, H, _ptr(out), os_t, os_n,
                                            _ptr(dev_err), _stream(stream)))
    _count(1 if T > 0 and H > 0 else 0)


def dsa_indexer_logits(q_bf16: torch.Tensor, weights: torch.Tensor, index_k_pool: torch.Tensor,
                       block_table: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor,
                       max_seq_len: int, max_q_len: int, logits: torch.Tensor, row_begin: int = 0,
                       row_end: Optional[int] = None, flags: int = 0, dev_err: Optional[torch.Tensor] = None,
                       stream=None, workspace: Optional[torch.Tensor] = None) -> None:
    """Logits of rows [row_begin, row_end).  `workspace` is device scratch of at least
    dsa_indexer_logits_workspace_size(row_end - row_begin) bytes; when it is None a buffer of that
    size is taken from torch's allocator for this call."""
    lib = load()
    _cuda(q_bf16, torch.bfloat16, "q_bf16")
    _cuda(weights, torch.float32, "weights")
    _cuda(index_k_pool, torch.uint8, "index_k_pool")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(cu_q, torch.int32, "cu_q")
    _rows(logits, torch.float32, "logits")
    _need(q_bf16.dim() == 3 and tuple(q_bf16.shape[1:]) == (64, 128), "q_bf16 must be [T, 64, 128]")
    T = q_bf16.shape[0]
    _need(tuple(weights.shape) == (T, 64), "weights must be [T, 64]")
    B = seq_lens.numel()
    _need(cu_q.numel() == B + 1 and block_table.dim() == 2 and block_table.shape[0] == B, "metadata shapes")
    row_end = T if row_end is None else row_end
    _need(0 <= row_begin <= row_end <= T, "row range")
    _need(logits.dim() == 2 and logits.shape[0] >= row_end - row_begin, "logits rows")
    if workspace is None:
        workspace = torch.empty(max(16, dsa_indexer_logits_workspace_size(row_end - row_begin)), dtype=torch.uint8,
                                device=q_bf16.device)
    _need(workspace.is_cuda and workspace.is_contiguous(), "workspace must be a contiguous CUDA tensor")
    _check("dsa_indexer_logits", lib.dsa_indexer_logits(
        _ptr(q_bf16), _ptr(weights), _ptr(index_k_pool), index_k_pool.shape[0], _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), B, int(max_seq_len), int(max_q_len), int(row_begin),
        int(row_end), _ptr(logits), logits.stride(0), int(flags), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(stream)))
    _count(2 if row_end > row_begin else 0)


def dsa_indexer_logits_workspace_size(rows: int) -> int:
    return int(load().dsa_indexer_logits_workspace_size(int(rows)))


def dsa_store_index_k_c8(k_bf16: torch.Tensor, slot_mapping: torch.Tensor, index_k_pool_c8: torch.Tensor,
                         dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    lib = load()
    _cuda(k_bf16, torch.bfloat16, "k_bf16")
    _cuda(slot_mapping, torch.int64, "slot_mapping")
    _cuda(index_k_pool_c8, torch.uint8, "index_k_pool_c8")
    _need(k_bf16.dim() == 2 and k_bf16.shape[1] == 128, "k_bf16 must be [n, 128]")
    _need(slot_mapping.numel() == k_bf16.shape[0], "slot_mapping must have n entries")
    _need(index_k_pool_c8.dim() == 2 and index_k_pool_c8.shape[1] == C8_PAGE_BYTES, "pool must be [pages, 8320]")
    _check("dsa_store_index_k_c8", lib.dsa_store_index_k_c8(
        _ptr(k_bf16), _ptr(slot_mapping), k_bf16.shape[0], _ptr(index_k_pool_c8), index_k_pool_c8.shape[0],
        PAGE_SIZE, _ptr(dev_err), _stream(stream)))
    _count(1 if k_bf16.shape[0] > 0 else 0)


def dsa_indexer_logits_c8_workspace_size(rows: int) -> int:
    return int(load().dsa_indexer_logits_c8_workspace_size(int(rows)))


def dsa_indexer_logits_c8(q_bf16: torch.Tensor, weights: torch.Tensor, index_k_pool_c8: torch.Tensor,
                          block_table: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor,
                          max_seq_len: int, max_q_len: int, logits: torch.Tensor, row_begin: int = 0,
                          row_end: Optional[int] = None, dev_err: Optional[torch.Tensor] = None,
                          stream=None, workspace: Optional[torch.Tensor] = None) -> None:
    """Logits of rows [row_begin, row_end) over the int8 cache (dsa_store_index_k_c8)."""
    lib = load()
    _cuda(q_bf16, torch.bfloat16, "q_bf16")
    _cuda(weights, torch.float32, "weights")
    _cuda(index_k_pool_c8, torch.uint8, "index_k_pool_c8")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(cu_q, torch.int32, "cu_q")
    _rows(logits, torch.float32, "logits")
    _need(q_bf16.dim() == 3 and tuple(q_bf16.shape[1:]) == (64, 128), "q_bf16 must be [T, 64, 128]")
    _need(index_k_pool_c8.dim() == 2 and index_k_pool_c8.shape[1] == C8_PAGE_BYTES, "pool must be [pages, 8320]")
    T = q_bf16.shape[0]
    _need(tuple(weights.shape) == (T, 64), "weights must be [T, 64]")
    B = seq_lens.numel()
    _need(cu_q.numel() == B + 1 and block_table.dim() == 2 and block_table.shape[0] == B, "metadata shapes")
    row_end = T if row_end is None else row_end
    _need(0 <= row_begin <= row_end <= T, "row range")
    _need(logits.dim() == 2 and logits.shape[0] >= row_end - row_begin, "logits rows")
    if workspace is None:
        workspace = torch.empty(max(16, dsa_indexer_logits_c8_workspace_size(row_end - row_begin)),
                                dtype=torch.uint8, device=q_bf16.device)
    _need(workspace.is_cuda and workspace.is_contiguous(), "workspace must be a contiguous CUDA tensor")
    _check("dsa_indexer_logits_c8", lib.dsa_indexer_logits_c8(
        _ptr(q_bf16), _ptr(weights), _ptr(index_k_pool_c8), index_k_pool_c8.shape[0], _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), B, int(max_seq_len), int(max_q_len), int(row_begin),
        int(row_end), _ptr(logits), logits.stride(0), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_err), _stream(stream)))
    _count(2 if row_end > row_begin else 0)


def dsa_topk_workspace_size(rows: int, k: int, max_seq_len: int) -> int:
    return int(load().dsa_topk_workspace_size(int(rows), int(k), int(max_seq_len)))


def dsa_topk(logits: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor, max_seq_len: int, k: int,
             idx: torch.Tensor, row_begin: int = 0, row_end: Optional[int] = None,
             workspace: Optional[torch.Tensor] = None, stream=None, n_init: int = 0, n_local: int = 0) -> None:
    """Per-row top-k; with n_init / n_local > 0 (dsa_topk_forced) the first n_init and the last
    n_local visible positions of every row count as +inf."""
    lib = load()
    _rows(logits, torch.float32, "logits")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(cu_q, torch.int32, "cu_q")
    _cuda(idx, torch.int32, "idx")
    B = seq_lens.numel()
    row_end = (row_begin + logits.shape[0]) if row_end is None else row_end
    rows = row_end - row_begin
    _need(idx.dim() == 2 and idx.shape[0] >= rows and idx.shape[1] == k, "idx must be [rows, k]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if n_init or n_local:
        _check("dsa_topk_forced", lib.dsa_topk_forced(
            _ptr(logits), logits.stride(0), _ptr(seq_lens), _ptr(cu_q), B, int(max_seq_len), int(row_begin),
            int(row_end), int(k), int(n_init), int(n_local), _ptr(idx), _ptr(workspace), ws_bytes, _stream(stream)))
    else:
        _check("dsa_topk", lib.dsa_topk(
            _ptr(logits), logits.stride(0), _ptr(seq_lens), _ptr(cu_q), B, int(max_seq_len), int(row_begin),
            int(row_end), int(k), _ptr(idx), _ptr(workspace), ws_bytes, _stream(stream)))
    _count(1 if rows > 0 else 0)


def dsa_lightning_indexer_workspace_size(T: int, max_seq_len: int) -> int:
    return int(load().dsa_lightning_indexer_workspace_size(int(T), int(max_seq_len)))


def dsa_lightning_indexer(q_bf16: torch.Tensor, weights: torch.Tensor, index_k_pool: torch.Tensor,
                          block_table: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor, max_seq_len: int,
                          max_q_len: int, k: int, idx: torch.Tensor, workspace: torch.Tensor, n_init: int = 0,
                          n_local: int = 0, flags: int = 0, dev_err: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """Top-k indices of the indexer logits of every row in one call (the logits stay in
    `workspace`, dsa_lightning_indexer_workspace_size(T, max_seq_len) bytes)."""
    lib = load()
    _cuda(q_bf16, torch.bfloat16, "q_bf16")
    _cuda(weights, torch.float32, "weights")
    _cuda(index_k_pool, torch.uint8, "index_k_pool")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(cu_q, torch.int32, "cu_q")
    _cuda(idx, torch.int32, "idx")
    _cuda(workspace, torch.uint8, "workspace")
    T = q_bf16.shape[0]
    B = seq_lens.numel()
    _need(q_bf16.dim() == 3 and tuple(q_bf16.shape[1:]) == (64, 128), "q_bf16 must be [T, 64, 128]")
    _need(tuple(idx.shape) == (T, k), "idx must be [T, k]")
    _check("dsa_lightning_indexer", lib.dsa_lightning_indexer(
        _ptr(q_bf16), _ptr(weights), _ptr(index_k_pool), index_k_pool.shape[0], _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), B, int(max_seq_len), int(max_q_len), T, int(k),
        int(n_init), int(n_local), int(flags), _ptr(idx), _ptr(workspace), workspace.numel(), _ptr(dev_err),
        _stream(stream)))
    _count(3 if T > 0 else 0)


def dsa_sparse_mla_workspace_size(T: int, H: int, k: int) -> int:
    return int(load().dsa_sparse_mla_workspace_size(int(T), int(H), int(k)))


def dsa_sparse_mla_decode(q_bf16: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                          seq_lens: torch.Tensor, cu_q: torch.Tensor, idx: torch.Tensor, scale: float,
                          out: torch.Tensor, workspace: torch.Tensor, lse: Optional[torch.Tensor] = None,
                          dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    lib = load()
    _cuda(q_bf16, torch.bfloat16, "q_bf16")
    _cuda(kv_pool, torch.bfloat16, "kv_pool")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(cu_q, torch.int32, "cu_q")
    _cuda(idx, torch.int32, "idx")
    _cuda(out, torch.bfloat16, "out")
    _need(workspace.is_cuda and workspace.is_contiguous(), "workspace must be a contiguous CUDA tensor")
    if lse is not None:
        _cuda(lse, torch.float32, "lse")
    _need(q_bf16.dim() == 3 and q_bf16.shape[2] == LATENT_DIM, "q_bf16 must be [T, H, 576]")
    T, H, _ = q_bf16.shape
    _need(kv_pool.dim() == 3 and tuple(kv_pool.shape[1:]) == (64, LATENT_DIM), "kv_pool must be [pages, 64, 576]")
    _need(idx.dim() == 2 and idx.shape[0] == T, "idx must be [T, k]")
    _need(tuple(out.shape) == (T, H, VALUE_DIM), "out must be [T, H, 512]")
    B = seq_lens.numel()
    _check("dsa_sparse_mla_decode", lib.dsa_sparse_mla_decode(
        _ptr(q_bf16), _ptr(kv_pool), kv_pool.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        _ptr(cu_q), B, _ptr(idx), idx.shape[1], T, H, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(stream)))
    # the attention kernel, and the split-K combine when the rows are split (scratch needed)
    _count((1 + (1 if dsa_sparse_mla_workspace_size(T, H, idx.shape[1]) > 0 else 0)) if T > 0 else 0)


def dsa_sparse_attn_swa_cmp_workspace_size(T: int, H: int, window: int, k: int) -> int:
    return int(load().dsa_sparse_attn_swa_cmp_workspace_size(int(T), int(H), int(window), int(k)))


def dsa_sparse_attn_swa_cmp(q_bf16: torch.Tensor, swa_kv: torch.Tensor, swa_block_table: torch.Tensor,
                            cmp_kv: torch.Tensor, cmp_block_table: torch.Tensor, seq_lens: torch.Tensor,
                            cu_q: torch.Tensor, cmp_idx: torch.Tensor, window: int, cmp_ratio: int,
                            sinks: torch.Tensor, scale: float, out: torch.Tensor,
                            workspace: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Sliding window of the original cache + selected compressed entries + per-head sinks."""
    lib = load()
    _cuda(q_bf16, torch.bfloat16, "q_bf16")
    _cuda(swa_kv, torch.bfloat16, "swa_kv")
    _cuda(cmp_kv, torch.bfloat16, "cmp_kv")
    for t, n in ((swa_block_table, "swa_block_table"), (cmp_block_table, "cmp_block_table"), (seq_lens, "seq_lens"),
                 (cu_q, "cu_q"), (cmp_idx, "cmp_idx")):
        _cuda(t, torch.int32, n)
    _cuda(sinks, torch.float32, "sinks")
    _cuda(out, torch.bfloat16, "out")
    if lse is not None:
        _cuda(lse, torch.float32, "lse")
    _need(q_bf16.dim() == 3 and q_bf16.shape[2] == LATENT_DIM, "q_bf16 must be [T, H, 576]")
    T, H, _ = q_bf16.shape
    for kv, n in ((swa_kv, "swa_kv"), (cmp_kv, "cmp_kv")):
        _need(kv.dim() == 3 and tuple(kv.shape[1:]) == (64, LATENT_DIM), f"{n} must be [pages, 64, 576]")
    _need(cmp_idx.dim() == 2 and cmp_idx.shape[0] == T, "cmp_idx must be [T, k]")
    _need(sinks.numel() == H, "sinks must be [H]")
    _need(tuple(out.shape) == (T, H, VALUE_DIM), "out must be [T, H, 512]")
    if workspace is None:
        workspace = torch.empty(max(16, dsa_sparse_attn_swa_cmp_workspace_size(T, H, window, cmp_idx.shape[1])),
                                dtype=torch.uint8, device=q_bf16.device)
    _need(workspace.is_cuda and workspace.is_contiguous(), "workspace must be a contiguous CUDA tensor")
    B = seq_lens.numel()
    _check("dsa_sparse_attn_swa_cmp", lib.dsa_sparse_attn_swa_cmp(
        _ptr(q_bf16), _ptr(swa_kv), swa_kv.shape[0], _ptr(swa_block_table), swa_block_table.shape[1], _ptr(cmp_kv),
        cmp_kv.shape[0], _ptr(cmp_block_table), cmp_block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), B,
        _ptr(cmp_idx), cmp_idx.shape[1], int(window), int(cmp_ratio), _ptr(sinks), T, H, float(scale), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(stream)))
    split = dsa_sparse_attn_swa_cmp_workspace_size(T, H, window, cmp_idx.shape[1]) > 0
    _count((1 + (1 if split else 0)) if T > 0 else 0)   # the kernel (+ the combine when the rows are split)


def dsa_store_latent_fp8(latent_bf16: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                         kv_pool_fp8: torch.Tensor, dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Latent rows [n, 576] (bf16) into the FP8 latent cache (uint8 [pages, 64, 576]) by slot."""
    lib = load()
    _cuda(latent_bf16, torch.bfloat16, "latent_bf16")
    _cuda(slot_mapping, torch.int64, "slot_mapping")
    _cuda(kv_pool_fp8, torch.uint8, "kv_pool_fp8")
    _need(latent_bf16.dim() == 2 and latent_bf16.shape[1] == LATENT_DIM, "latent_bf16 must be [n, 576]")
    _need(slot_mapping.numel() == latent_bf16.shape[0], "one slot per row")
    _need(kv_pool_fp8.dim() == 3 and tuple(kv_pool_fp8.shape[1:]) == (64, LATENT_DIM),
          "kv_pool_fp8 must be [pages, 64, 576]")
    n = latent_bf16.shape[0]
    _check("dsa_store_latent_fp8", lib.dsa_store_latent_fp8(_ptr(latent_bf16), _ptr(slot_mapping), n, float(k_scale),
                                                            _ptr(kv_pool_fp8), kv_pool_fp8.shape[0], _ptr(dev_err),
                                                            _stream(stream)))
    _count(1 if n > 0 else 0)


def dsa_sparse_mla_decode_fp8(q_bf16: torch.Tensor, q_scale: float, kv_pool_fp8: torch.Tensor, k_scale: float,
                              block_table: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor, idx: torch.Tensor,
                              scale: float, out: torch.Tensor, workspace: torch.Tensor,
                              lse: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                              stream=None) -> None:
    """Sparse MLA over the FP8 latent cache; the query is quantised with q_scale inside the call."""
    lib = load()
    _cuda(q_bf16, torch.bfloat16, "q_bf16")
    _cuda(kv_pool_fp8, torch.uint8, "kv_pool_fp8")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(cu_q, torch.int32, "cu_q")
    _cuda(idx, torch.int32, "idx")
    _cuda(out, torch.bfloat16, "out")
    _need(workspace.is_cuda and workspace.is_contiguous(), "workspace must be a contiguous CUDA tensor")
    if lse is not None:
        _cuda(lse, torch.float32, "lse")
    _need(q_bf16.dim() == 3 and q_bf16.shape[2] == LATENT_DIM, "q_bf16 must be [T, H, 576]")
    T, H, _ = q_bf16.shape
    _need(kv_pool_fp8.dim() == 3 and tuple(kv_pool_fp8.shape[1:]) == (64, LATENT_DIM),
          "kv_pool_fp8 must be [pages, 64, 576]")
    _need(idx.dim() == 2 and idx.shape[0] == T, "idx must be [T, k]")
    _need(tuple(out.shape) == (T, H, VALUE_DIM), "out must be [T, H, 512]")
    B = seq_lens.numel()
    _check("dsa_sparse_mla_decode_fp8", lib.dsa_sparse_mla_decode_fp8(
        _ptr(q_bf16), float(q_scale), _ptr(kv_pool_fp8), float(k_scale), kv_pool_fp8.shape[0], _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), _ptr(cu_q), B, _ptr(idx), idx.shape[1], T, H, float(scale), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(stream)))
    _count((1 + (1 if dsa_sparse_mla_workspace_size(T, H, idx.shape[1]) > 0 else 0)) if T > 0 else 0)


def dsa_sparse_mla_decode_noalloc(q_bf16: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                                  seq_lens: torch.Tensor, cu_q: torch.Tensor, idx: torch.Tensor, scale: float,
                                  out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                                  dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """dsa_sparse_mla_decode without a workspace argument: the library's fixed 16 MiB scratch is
    used, for callers that may not allocate device memory.  Larger problems raise DSAError
    (DSA_ERR_UNSUPPORTED)."""
    lib = load()
    _cuda(q_bf16, torch.bfloat16, "q_bf16")
    _cuda(kv_pool, torch.bfloat16, "kv_pool")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(cu_q, torch.int32, "cu_q")
    _cuda(idx, torch.int32, "idx")
    _cuda(out, torch.bfloat16, "out")
    if lse is not None:
        _cuda(lse, torch.float32, "lse")
    _need(q_bf16.dim() == 3 and q_bf16.shape[2] == LATENT_DIM, "q_bf16 must be [T, H, 576]")
    T, H, _ = q_bf16.shape
    _need(kv_pool.dim() == 3 and tuple(kv_pool.shape[1:]) == (64, LATENT_DIM), "kv_pool must be [pages, 64, 576]")
    _need(idx.dim() == 2 and idx.shape[0] == T, "idx must be [T, k]")
    _need(tuple(out.shape) == (T, H, VALUE_DIM), "out must be [T, H, 512]")
    B = seq_lens.numel()
    _check("dsa_sparse_mla_decode_noalloc", lib.dsa_sparse_mla_decode_noalloc(
        _ptr(q_bf16), _ptr(kv_pool), kv_pool.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        _ptr(cu_q), B, _ptr(idx), idx.shape[1], T, H, float(scale), _ptr(out), _ptr(lse), _ptr(dev_err),
        _stream(stream)))
    _count(2 if T > 0 else 0)


def dsa_selftest_wait_timeout(dev_err: torch.Tensor, cycles: int, stream=None) -> None:
    """Runs a bounded wait that can never complete; it must give up and set DSA_DEVERR_TIMEOUT."""
    lib = load()
    _cuda(dev_err, torch.int32, "dev_err")
    _check("dsa_selftest_wait_timeout", lib.dsa_selftest_wait_timeout(_ptr(dev_err), int(cycles), _stream(stream)))
    _count(1)


def dsa_read_device_error(dev_err: torch.Tensor, stream=None):
    """Returns (status, raw word)."""
    lib = load()
    word = ctypes.c_int32(0)
    st = lib.dsa_read_device_error(_ptr(dev_err), ctypes.byref(word), _stream(stream))
    return int(st), int(word.value)
