"""CPU oracle for the DSA decode path -- TEST INFRASTRUCTURE ONLY.

This package wraps ``dsa_oracle.c``: a plain, slow, double-precision C implementation of what the
DSA decode path computes (Hadamard rotation, FP8-E4M3 quantisation, paged index-K store,
lightning-indexer logits, per-row top-k, absorbed sparse MLA, log-sum-exp merge, the indexer
prologues, and the per-head projections around the absorbed attention).  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may
import it.  The product library (``deepseek_sparse_attention_paged_gb300``) never imports, links or
runs anything here, and the two share no code.

Every function is pinned by ``-m "not gpu"`` tests against closed forms, library routines, brute
force and invariants (see ``tests/test_oracle_*.py``).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdsa_oracle.so")
_lib = None

PAGE = 64
DI = 128
HI = 64
ROW_BYTES = 132
PAGE_BYTES = PAGE * ROW_BYTES
C8_PAGE_BYTES = PAGE * DI + PAGE * 2      # int8 cache page: 64 x 128 codes + 64 fp16 scales
DQK = 576
DV = 512


_CMD = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared"]


def _digest() -> str:
    """Hash of the source, the compiler command and the machine type: the library is rebuilt
    whenever it differs from the one stored beside the last build."""
    import hashlib
    import platform
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(_CMD).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libdsa_oracle.so`` (host C, gcc, OpenMP)."""
    digest = _digest()
    stamp = _LIB_PATH + ".hash"
    if not force and os.path.exists(_LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(_CMD + [_SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    with open(stamp + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(stamp + f".tmp{os.getpid()}", stamp)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i64, i32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
    sig = {
        "dsa_oracle_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
        "dsa_oracle_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "dsa_oracle_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
        "dsa_oracle_f64_to_bf16_array": (None, [P, i64, P]),
        "dsa_oracle_e4m3_decode": (f64, [ctypes.c_uint8]),
        "dsa_oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "dsa_oracle_fwht128": (None, [P]),
        "dsa_oracle_rotate128": (None, [P, P]),
        "dsa_oracle_quant128": (None, [P, P, P]),
        "dsa_oracle_quant128_fmt": (None, [P, P, P, ctypes.c_int]),
        "dsa_oracle_store_index_k": (i64, [P, P, i64, P, i64]),
        "dsa_oracle_k_norm128": (None, [P, P, P, ctypes.c_float, ctypes.c_int, P]),
        "dsa_oracle_rope64": (None, [P, P, ctypes.c_int, P]),
        "dsa_oracle_store_index_k_prologue": (i64, [P, P, P, ctypes.c_float, ctypes.c_int, P, i64, P, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, P, i64, P, i64]),
        "dsa_oracle_rope_q": (i64, [P, P, i64, P, ctypes.c_int, i64, P]),
        "dsa_oracle_visible_len": (i32, [P, P, i32, i64]),
        "dsa_oracle_indexer_logits": (i64, [P, P, P, i64, P, i32, P, P, i32, i32, P, i64, P, i64, P]),
        "dsa_oracle_topk": (None, [P, i64, P, P, i32, P, i64, i32, P]),
        "dsa_oracle_sparse_mla": (i64, [P, P, i64, P, i32, P, P, i32, P, i32, i32, f64, P, i64, P, P, P]),
        "dsa_oracle_dense_mla": (None, [P, P, i64, P, i32, P, P, i32, i32, f64, P, i64, P, P]),
        "dsa_oracle_quant_fp8_tensor": (None, [P, i64, ctypes.c_float, P]),
        "dsa_oracle_store_latent_fp8": (i64, [P, P, i64, ctypes.c_float, P, i64]),
        "dsa_oracle_sparse_mla_fp8": (i64, [P, ctypes.c_float, P, ctypes.c_float, i64, P, i32, P, P, i32, P, i32, i32,
                                            f64, P, i64, P, P]),
        "dsa_oracle_lse_merge": (None, [P, P, P, P, i64, i32, P, P]),
        "dsa_oracle_f16_decode": (f64, [ctypes.c_uint16]),
        "dsa_oracle_visible_len_cmp": (i32, [P, P, i32, i64, i32]),
        "dsa_oracle_indexer_logits_cmp": (i64, [P, P, P, i64, P, i32, P, P, i32, i32, i32, P, i64, P, i64, P]),
        "dsa_oracle_topk_cmp": (None, [P, i64, P, P, i32, P, i64, i32, i32, P]),
        "dsa_oracle_dsv4_attention": (i64, [P, P, i64, P, i32, P, i64, P, i32, P, P, i32, P, i32, i32, i32, P, i32,
                                            f64, P, i64, P, P]),
        "dsa_oracle_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
        "dsa_oracle_c8_rotate128": (None, [P, P]),
        "dsa_oracle_quant_int8": (None, [P, ctypes.c_int, P, P]),
        "dsa_oracle_store_index_k_c8": (i64, [P, P, i64, P, i64]),
        "dsa_oracle_indexer_logits_c8": (i64, [P, P, P, i64, P, i32, P, P, i32, P, i64, P, i64, P]),
        "dsa_oracle_num_threads": (ctypes.c_int, []),
        "dsa_oracle_set_num_threads": (None, [ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ scalar helpers

def f32_to_bf16(x: float) -> int:
    return int(_load().dsa_oracle_f32_to_bf16(float(x)))


def bf16_to_f32(h: int) -> float:
    return float(_load().dsa_oracle_bf16_to_f32(int(h)))


def e4m3_decode(c: int) -> float:
    return float(_load().dsa_oracle_e4m3_decode(int(c)))


def e4m3_encode(x: float) -> int:
    return int(_load().dsa_oracle_e4m3_encode(float(x)))


def f32_to_bf16_array(x: np.ndarray) -> np.ndarray:
    fn = _load().dsa_oracle_f32_to_bf16
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.array([fn(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(x))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    fn = _load().dsa_oracle_e4m3_encode
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.array([fn(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


# ------------------------------------------------------------------ vector steps

def fwht128(x: np.ndarray) -> np.ndarray:
    """Unnormalised fp32 Walsh-Hadamard butterflies of one 128-vector (Sylvester order)."""
    v = _c(x, np.float32).copy()
    assert v.shape == (DI,)
    _load().dsa_oracle_fwht128(_p(v))
    return v


def rotate128(x_bf16: np.ndarray) -> np.ndarray:
    """Hadamard rotation of one bf16 128-vector (bits in, bits out)."""
    src = _c(x_bf16, np.uint16)
    assert src.shape == (DI,)
    out = np.empty(DI, np.uint16)
    _load().dsa_oracle_rotate128(_p(src), _p(out))
    return out


def quant128(y: np.ndarray, ue8m0: bool = False):
    """Per-128 FP8 quantisation: returns (codes uint8[128], scale float32); ``ue8m0`` rounds the
    scale up to a power of two."""
    v = _c(y, np.float32)
    assert v.shape == (DI,)
    codes = np.empty(DI, np.uint8)
    s = np.empty(1, np.float32)
    if ue8m0:
        _load().dsa_oracle_quant128_fmt(_p(v), _p(codes), _p(s), 1)
    else:
        _load().dsa_oracle_quant128(_p(v), _p(codes), _p(s))
    return codes, s[0]


# ------------------------------------------------------------------ path stages

def store_index_k(k_bf16: np.ndarray, slot_mapping: np.ndarray, pool: np.ndarray) -> int:
    """Rotate, quantise and scatter keys into ``pool`` (uint8 [num_pages, 64*132]) in place."""
    k = _c(k_bf16, np.uint16).reshape(-1, DI)
    slots = _c(slot_mapping, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"] and pool.shape[1] == PAGE_BYTES
    return int(_load().dsa_oracle_store_index_k(_p(k), _p(slots), k.shape[0], _p(pool), pool.shape[0]))


def k_norm128(x_bf16: np.ndarray, w: np.ndarray, b, eps: float, rms: bool = False) -> np.ndarray:
    """LayerNorm (or RMSNorm) of one bf16 128-vector, bf16 bits out."""
    src = _c(x_bf16, np.uint16)
    assert src.shape == (DI,)
    wv = _c(w, np.float32)
    bv = _c(np.zeros(DI) if b is None else b, np.float32)
    out = np.empty(DI, np.uint16)
    _load().dsa_oracle_k_norm128(_p(src), _p(wv), _p(bv), float(eps), int(bool(rms)), _p(out))
    return out


def rope64(x_bf16: np.ndarray, cos_sin_row: np.ndarray, neox: bool = True) -> np.ndarray:
    """Rotary embedding of dims 0..63 of one bf16 128-vector with one cos/sin cache row."""
    src = _c(x_bf16, np.uint16)
    cs = _c(cos_sin_row, np.float32)
    assert src.shape == (DI,) and cs.shape == (64,)
    out = np.empty(DI, np.uint16)
    _load().dsa_oracle_rope64(_p(src), _p(cs), int(bool(neox)), _p(out))
    return out


def store_index_k_prologue(k_raw: np.ndarray, w: np.ndarray, b, eps: float, cos_sin: np.ndarray,
                           positions: np.ndarray, slot_mapping: np.ndarray, pool: np.ndarray, rms: bool = False,
                           neox: bool = True, rotate: bool = True, ue8m0: bool = False) -> int:
    """Norm, rotary embedding, rotate (unless ``rotate`` is False), quantise (power-of-two scales
    with ``ue8m0``) and scatter raw keys into ``pool`` in place."""
    k = _c(k_raw, np.uint16).reshape(-1, DI)
    wv = _c(w, np.float32)
    bv = _c(np.zeros(DI) if b is None else b, np.float32)
    cs = _c(cos_sin, np.float32).reshape(-1, 64)
    pos = _c(positions, np.int64)
    slots = _c(slot_mapping, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"] and pool.shape[1] == PAGE_BYTES
    return int(_load().dsa_oracle_store_index_k_prologue(_p(k), _p(wv), _p(bv), float(eps), int(bool(rms)), _p(cs),
                                                         cs.shape[0], _p(pos), int(bool(neox)), int(bool(rotate)),
                                                         int(bool(ue8m0)), _p(slots),
                                                         k.shape[0], _p(pool), pool.shape[0]))


def rope_q(q_raw: np.ndarray, cos_sin: np.ndarray, positions: np.ndarray, neox: bool = True):
    """Rotary embedding of every head of every query row: returns (bf16 bits [T, 64, 128], bad rows)."""
    q = _c(q_raw, np.uint16).reshape(-1, HI, DI)
    cs = _c(cos_sin, np.float32).reshape(-1, 64)
    pos = _c(positions, np.int64)
    out = np.empty_like(q)
    bad = _load().dsa_oracle_rope_q(_p(q), _p(cs), cs.shape[0], _p(pos), int(bool(neox)), q.shape[0], _p(out))
    return out, int(bad)


def visible_len(seq_lens, cu_q, r: int) -> int:
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    return int(_load().dsa_oracle_visible_len(_p(sl), _p(cq), sl.shape[0], int(r)))


def indexer_logits(q_bf16, w, pool, block_table, seq_lens, cu_q, rows, ld, rotate_q=False,
                   want_mag=False, fill=np.nan, ue8m0_q=False, cmp_ratio=1):
    """Indexer logits for the global rows ``rows``; returns float32 [len(rows), ld] (and the
    float64 magnitude array when ``want_mag``).  Entries past each row's visible length (of
    compressed entries when ``cmp_ratio`` > 1) keep ``fill``."""
    q = _c(q_bf16, np.uint16)
    wv = _c(w, np.float32)
    pool = _c(pool, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    rr = _c(rows, np.int64)
    out = np.full((rr.shape[0], ld), fill, np.float32)
    mag = np.zeros((rr.shape[0], ld), np.float64) if want_mag else None
    bad = _load().dsa_oracle_indexer_logits_cmp(
        _p(q), _p(wv), _p(pool), pool.shape[0], _p(bt), bt.shape[1], _p(sl), _p(cq), sl.shape[0],
        int(bool(rotate_q)) | (int(bool(ue8m0_q)) << 1), int(cmp_ratio), _p(rr), rr.shape[0], _p(out), ld,
        _p(mag) if mag is not None else None)
    if want_mag:
        return out, mag, int(bad)
    return out


def topk(logits, seq_lens, cu_q, rows, k, cmp_ratio=1):
    """Per-row top-k indices (ascending index order, -1 padded) for logits rows of ``rows``."""
    lg = _c(logits, np.float32)
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    rr = _c(rows, np.int64)
    idx = np.empty((rr.shape[0], k), np.int32)
    _load().dsa_oracle_topk_cmp(_p(lg), lg.shape[1], _p(sl), _p(cq), sl.shape[0], _p(rr), rr.shape[0],
                                int(k), int(cmp_ratio), _p(idx))
    return idx


def visible_len_cmp(seq_lens, cu_q, r: int, ratio: int) -> int:
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    return int(_load().dsa_oracle_visible_len_cmp(_p(sl), _p(cq), sl.size, int(r), int(ratio)))


def dsv4_attention(q_bf16, swa_kv_bf16, swa_block_table, cmp_kv_bf16, cmp_block_table, seq_lens, cu_q, cmp_idx,
                   window, sinks, scale, rows, ratio=4):
    """Window + selected compressed entries + per-head sinks: (out [n, H, 512] f64, lse [n, H] f64, skipped)."""
    q = _c(q_bf16, np.uint16)
    T, H = q.shape[0], q.shape[1]
    sw = _c(swa_kv_bf16, np.uint16).reshape(-1, PAGE, DQK)
    ck = _c(cmp_kv_bf16, np.uint16).reshape(-1, PAGE, DQK)
    sbt = _c(swa_block_table, np.int32)
    cbt = _c(cmp_block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    ix = _c(cmp_idx, np.int32)
    sk = _c(sinks, np.float32)
    rw = _c(rows, np.int64)
    out = np.empty((rw.size, H, DV), np.float64)
    lse = np.empty((rw.size, H), np.float64)
    bad = _load().dsa_oracle_dsv4_attention(_p(q), _p(sw), sw.shape[0], _p(sbt), sbt.shape[1], _p(ck), ck.shape[0],
                                            _p(cbt), cbt.shape[1], _p(sl), _p(cq), sl.size, _p(ix), ix.shape[1],
                                            int(window), int(ratio), _p(sk), H, float(scale), _p(rw), rw.size,
                                            _p(out), _p(lse))
    return out, lse, int(bad)


def topk_forced(logits, seq_lens, cu_q, rows, k, n_init, n_local):
    """Top-k with forced initial and local tokens ([idx] Indexer._mask_init_and_local_tokens: the
    logits at the row's first n_init and last n_local positions are set to +inf before the top-k).
    Reading: the positions are taken inside the row's visible range [0, v_r); then ``topk``."""
    lg = np.array(logits, dtype=np.float32, copy=True)
    rr = np.asarray(rows, np.int64)
    for i, r in enumerate(rr):
        v = visible_len(seq_lens, cu_q, int(r))
        v = min(v, lg.shape[1])
        lg[i, :min(n_init, v)] = np.inf
        lg[i, max(0, v - n_local):v] = np.inf
    return topk(lg, seq_lens, cu_q, rows, k)


def sparse_mla(q_bf16, kv_bf16, block_table, seq_lens, cu_q, idx, scale, rows, want_psum=False):
    """Absorbed sparse MLA for the global rows ``rows``; returns (out float64 [n,H,512],
    lse float64 [n,H]) and, when ``want_psum``, the softmax-weight sums and the skipped count."""
    q = _c(q_bf16, np.uint16)
    T, H, D = q.shape
    assert D == DQK
    kv = _c(kv_bf16, np.uint16)
    num_pages = kv.shape[0]
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    ix = _c(idx, np.int32)
    rr = _c(rows, np.int64)
    n = rr.shape[0]
    out = np.zeros((n, H, DV), np.float64)
    lse = np.zeros((n, H), np.float64)
    psum = np.zeros((n, H), np.float64)
    bad = _load().dsa_oracle_sparse_mla(_p(q), _p(kv), num_pages, _p(bt), bt.shape[1], _p(sl), _p(cq),
                                        sl.shape[0], _p(ix), ix.shape[1], H, float(scale), _p(rr), n,
                                        _p(out), _p(lse), _p(psum))
    if want_psum:
        return out, lse, psum, int(bad)
    return out, lse


def f16_decode(h: int) -> float:
    return _load().dsa_oracle_f16_decode(int(h))


def f32_to_f16(x: float) -> int:
    return int(_load().dsa_oracle_f32_to_f16(float(x)))


def c8_rotate128(x_bf16: np.ndarray) -> np.ndarray:
    """The c8 rotation of one bf16 128-vector (bits): bf16(x @ (bf16 Hadamard / sqrt(128)))."""
    x = _c(x_bf16, np.uint16)
    assert x.size == DI
    out = np.empty(DI, np.uint16)
    _load().dsa_oracle_c8_rotate128(_p(x), _p(out))
    return out


def quant_int8(y: np.ndarray):
    """Dynamic int8 quantisation of one fp32 vector: (codes int8, fp32 scale)."""
    yy = _c(y, np.float32)
    codes = np.empty(yy.size, np.int8)
    sc = np.empty(1, np.float32)
    _load().dsa_oracle_quant_int8(_p(yy), yy.size, _p(codes), _p(sc))
    return codes, float(sc[0])


def store_index_k_c8(k_bf16: np.ndarray, slot_mapping: np.ndarray, pool: np.ndarray) -> int:
    """Keys [n, 128] (bf16 bits) into the int8 cache ``pool`` (uint8 [num_pages, C8_PAGE_BYTES]) by slot."""
    k = _c(k_bf16, np.uint16).reshape(-1, DI)
    slots = _c(slot_mapping, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"] and pool.shape[1] == C8_PAGE_BYTES
    return int(_load().dsa_oracle_store_index_k_c8(_p(k), _p(slots), k.shape[0], _p(pool), pool.shape[0]))


def indexer_logits_c8(q_bf16, w, pool, block_table, seq_lens, cu_q, rows, ld, want_mag=False):
    """Logits over the int8 cache for the listed rows: fp32 [n, ld] (NaN where not written)."""
    q = _c(q_bf16, np.uint16)
    ww = _c(w, np.float32)
    pl = _c(pool, np.uint8)
    assert pl.shape[1] == C8_PAGE_BYTES
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    rw = _c(rows, np.int64)
    out = np.full((rw.size, ld), np.nan, np.float32)
    mag = np.full((rw.size, ld), np.nan, np.float64) if want_mag else None
    bad = _load().dsa_oracle_indexer_logits_c8(_p(q), _p(ww), _p(pl), pl.shape[0], _p(bt), bt.shape[1], _p(sl),
                                              _p(cq), sl.size, _p(rw), rw.size, _p(out), ld,
                                              _p(mag) if want_mag else None)
    if want_mag:
        return out, mag, int(bad)
    return out, int(bad)


def quant_fp8_tensor(x_bf16: np.ndarray, scale: float) -> np.ndarray:
    """Per-tensor FP8 codes of bf16 values: E4M3FN(x / scale) (fp32 division, RNE, saturating)."""
    x = _c(x_bf16, np.uint16)
    out = np.empty(x.shape, np.uint8)
    _load().dsa_oracle_quant_fp8_tensor(_p(x), x.size, float(scale), _p(out))
    return out


def store_latent_fp8(latent_bf16: np.ndarray, slot_mapping: np.ndarray, k_scale: float, pool: np.ndarray) -> int:
    """Latent rows [n, 576] (bf16 bits) into the FP8 cache ``pool`` (uint8 [num_pages, 64, 576]) by slot."""
    x = _c(latent_bf16, np.uint16).reshape(-1, DQK)
    slots = _c(slot_mapping, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"] and pool.shape[-1] == DQK
    return int(_load().dsa_oracle_store_latent_fp8(_p(x), _p(slots), x.shape[0], float(k_scale), _p(pool),
                                                     pool.shape[0]))


def sparse_mla_fp8(q_bf16, q_scale, kv_fp8, k_scale, block_table, seq_lens, cu_q, idx, scale, rows):
    """Sparse MLA over the FP8 latent cache (query quantised with q_scale): (out [n, H, 512], lse [n, H])."""
    q = _c(q_bf16, np.uint16)
    T, H = q.shape[0], q.shape[1]
    kv = _c(kv_fp8, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    ix = _c(idx, np.int32)
    rw = _c(rows, np.int64)
    out = np.empty((rw.size, H, DV), np.float64)
    lse = np.empty((rw.size, H), np.float64)
    _load().dsa_oracle_sparse_mla_fp8(_p(q), float(q_scale), _p(kv), float(k_scale), kv.shape[0], _p(bt), bt.shape[1],
                                      _p(sl), _p(cq), sl.size, _p(ix), ix.shape[1], H, float(scale), _p(rw), rw.size,
                                      _p(out), _p(lse))
    return out, lse


def dense_mla(q_bf16, kv_bf16, block_table, seq_lens, cu_q, scale, rows):
    q = _c(q_bf16, np.uint16)
    T, H, D = q.shape
    kv = _c(kv_bf16, np.uint16)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    cq = _c(cu_q, np.int32)
    rr = _c(rows, np.int64)
    n = rr.shape[0]
    out = np.zeros((n, H, DV), np.float64)
    lse = np.zeros((n, H), np.float64)
    _load().dsa_oracle_dense_mla(_p(q), _p(kv), kv.shape[0], _p(bt), bt.shape[1], _p(sl), _p(cq),
                                 sl.shape[0], H, float(scale), _p(rr), n, _p(out), _p(lse))
    return out, lse


# ------------------------------------------------------------------ projections around the attention

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact float64 values of bf16 bit patterns."""
    b = np.ascontiguousarray(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_array(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 (ties to even) of each double, one rounding."""
    v = _c(x, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().dsa_oracle_f64_to_bf16_array(_p(v), v.size, _p(out))
    return out


def mla_absorb_q(q_nope_bf16, w_uk_t_bf16, want_mag=False):
    """Absorbed latent query ([mla] MLACommonImpl.forward decode branch and
    _q_proj_and_k_up_proj: ql_nope = bmm(q_nope as (N, B, P), W_UK_T (N, P, L)) with
    W_UK_T = W_UK.permute(1, 2, 0), W_UK the qk_nope part of kv_b_proj viewed (L, N, P)):
        ql[t, n, l] = sum_p q_nope[t, n, p] * W_UK_T[n, p, l].
    q_nope: bf16 bits [T, N, P]; W_UK_T: bf16 bits [N, P, L].  The products of bf16 values are
    exact in float64 and so are their sums for data of ordinary range; the result is rounded once
    to bf16 (the output dtype of the pages' bmm).  Returns bf16 bits [T, N, L] (and the float64
    magnitude sum_p |q| |W| when ``want_mag``)."""
    q = bf16_bits_to_f64(q_nope_bf16)
    w = bf16_bits_to_f64(w_uk_t_bf16)
    T, N, P = q.shape
    assert w.shape[0] == N and w.shape[1] == P
    acc = np.matmul(q.transpose(1, 0, 2), w).transpose(1, 0, 2)          # [T, N, L]
    out = f64_to_bf16_array(acc)
    if want_mag:
        return out, np.matmul(np.abs(q).transpose(1, 0, 2), np.abs(w)).transpose(1, 0, 2)
    return out


def mla_v_up(o_lat_bf16, w_uv_bf16, want_mag=False):
    """Value up-projection of the latent attention output ([mla] MLACommonImpl._v_up_proj:
    bmm(x as (N, B, L), W_UV (N, L, V)) with W_UV = the v part of kv_b_proj viewed (L, N, V),
    transposed to (N, L, V)):  out[t, n, v] = sum_l o_lat[t, n, l] * W_UV[n, l, v].
    o_lat: bf16 bits [T, N, L]; W_UV: bf16 bits [N, L, V]; float64 sums rounded once to bf16.
    Returns bf16 bits [T, N, V] (and the magnitude sum_l |o| |W| when ``want_mag``)."""
    o = bf16_bits_to_f64(o_lat_bf16)
    w = bf16_bits_to_f64(w_uv_bf16)
    T, N, L = o.shape
    assert w.shape[0] == N and w.shape[1] == L
    acc = np.matmul(o.transpose(1, 0, 2), w).transpose(1, 0, 2)          # [T, N, V]
    out = f64_to_bf16_array(acc)
    if want_mag:
        return out, np.matmul(np.abs(o).transpose(1, 0, 2), np.abs(w)).transpose(1, 0, 2)
    return out


def lse_merge(o1, lse1, o2, lse2):
    o1 = _c(o1, np.float64)
    o2 = _c(o2, np.float64)
    l1 = _c(lse1, np.float64)
    l2 = _c(lse2, np.float64)
    dv = o1.shape[-1]
    n = l1.size
    o = np.zeros_like(o1)
    lse = np.zeros_like(l1)
    _load().dsa_oracle_lse_merge(_p(o1), _p(l1), _p(o2), _p(l2), n, dv, _p(o), _p(lse))
    return o, lse


def num_threads() -> int:
    return int(_load().dsa_oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().dsa_oracle_set_num_threads(int(n))
