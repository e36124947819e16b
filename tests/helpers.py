"""Shared helpers of the GPU parity tests: oracle-side references and the tolerance rules.

Tolerances:
  * FP8 codes, scales and top-k indices: bit-exact.
  * logits: |I_gpu - I_ref| <= 1e-3 * |I_ref| + 1e-5 * M_ref, where M_ref = sum_h |w'| ReLU(...)
    is the magnitude of the summed terms (the sum cancels, so its rounding error scales with M, not
    with |I|: the fp32 accumulation of 128 exact FP8 products and the 64-term head sum each stay
    below ~2^-20 M, well inside 1e-5 M; 1e-3 |I| is the stated relative bar).
  * attention output: max |o_gpu - o_ref| <= 2e-2 on unit-variance data; lse within 1e-3.
"""
import numpy as np
import torch

import oracle

LOGIT_REL = 1e-3
LOGIT_MAG = 1e-5
ATTN_ABS = 2e-2
LSE_ABS = 1e-3
TOPK_GAP_REL = 1e-4


def bf16_to_np_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def oracle_pool(wl) -> np.ndarray:
    pool = np.zeros((wl.num_pages, oracle.PAGE_BYTES), np.uint8)
    bad = oracle.store_index_k(wl.index_keys(), wl.token_slots(), pool)
    assert bad == 0
    return pool


def check_logits(got_rows: np.ndarray, ref_rows: np.ndarray, mag_rows: np.ndarray, vis: np.ndarray, key=None):
    """got/ref/mag: [n, >= max vis]; only s < vis[i] is compared.  Records, under `key`, how many
    logits were compared and how many pass only through the 1e-5 M term (their error exceeds
    1e-3 |I_ref|)."""
    worst = 0.0
    n_el = n_mag = 0
    for i, v in enumerate(vis):
        g = got_rows[i, :v].astype(np.float64)
        r = ref_rows[i, :v].astype(np.float64)
        m = mag_rows[i, :v]
        assert np.all(np.isfinite(g)), f"row {i}: non-finite logits"
        err = np.abs(g - r)
        bound = LOGIT_REL * np.abs(r) + LOGIT_MAG * m
        bad = err > bound
        assert not bad.any(), (f"row {i}: {bad.sum()} logits out of tolerance; worst at s={int(np.argmax(err - bound))} "
                               f"got {g[np.argmax(err - bound)]} ref {r[np.argmax(err - bound)]}")
        n_el += int(v)
        n_mag += int(np.count_nonzero(err > LOGIT_REL * np.abs(r)))
        if v:
            worst = max(worst, float(np.max(err / np.maximum(bound, 1e-30))))
    if key is not None:
        record(key, logits=n_el, logits_only_by_mag_term=n_mag)
    return worst


def kth_gap_ok(ref_row: np.ndarray, k: int) -> bool:
    """True when the k-th and (k+1)-th largest reference logits are separated by more than the
    near-tie band, so the top-k set is unique under any admissible rounding."""
    if ref_row.shape[0] <= k:
        return True
    s = np.sort(ref_row.astype(np.float64))[::-1]
    a, b = s[k - 1], s[k]
    return (a - b) > TOPK_GAP_REL * max(abs(a), abs(b), 1e-30)


def check_topk_valid(idx_row: np.ndarray, ref_row: np.ndarray, k: int, mag_row=None):
    """A top-k row is valid when it has min(k, v) distinct in-range ascending indices, -1 after,
    and every kept logit is >= every dropped one up to the two logits' own tolerances
    (1e-3 |I| + 1e-5 M of each, M per element)."""
    v = ref_row.shape[0]
    n = min(k, v)
    kept = idx_row[:n]
    assert np.all(idx_row[n:] == -1)
    assert np.all(kept >= 0) and np.all(kept < v)
    assert np.all(np.diff(kept) > 0)
    if n < v:
        mask = np.ones(v, bool)
        mask[kept] = False
        tol = LOGIT_REL * np.abs(ref_row)
        if mag_row is not None:
            tol = tol + LOGIT_MAG * np.asarray(mag_row, np.float64)
        assert (ref_row[kept] + tol[kept]).min() >= (ref_row[mask] - tol[mask]).max()


def check_attention(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray, lse_ref: np.ndarray, key=None):
    err = np.abs(out_gpu - out_ref)
    assert err.max() <= ATTN_ABS, f"attention max abs err {err.max()}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse_gpu))
    if fin.any():
        assert np.abs(lse_gpu[fin] - lse_ref[fin]).max() <= LSE_ABS
    if key is not None:
        record(key, outputs=err.size, rows=err.shape[0])
        d = PARITY_COUNTS[key]
        d["max_abs_err_x1e6"] = max(d.get("max_abs_err_x1e6", 0), int(round(float(err.max()) * 1e6)))
    return float(err.max())


# ---------------------------------------------------------------- counters shown at the end of a run

PARITY_COUNTS: dict = {}


def record(key: str, **counts):
    """Adds `counts` to the named entry of the run summary (printed by conftest at the end)."""
    d = PARITY_COUNTS.setdefault(key, {})
    for k, v in counts.items():
        d[k] = d.get(k, 0) + int(v)


# ---------------------------------------------------------------- key prologue bar

_E4M3_VALUES = None


def _e4m3_values():
    global _E4M3_VALUES
    if _E4M3_VALUES is None:
        _E4M3_VALUES = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    return _E4M3_VALUES


def _pow2_at_least(s: float) -> float:
    m, e = np.frexp(np.float64(s))
    return float(np.ldexp(1.0, int(e) - 1)) if m == 0.5 else float(np.ldexp(1.0, int(e)))


def _bf16_ulp(v):
    """Unit in the last place of bf16 at magnitude |v| (8 significant bits); 2^-133 at 0."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, (np.floor(np.log2(a)) - 7).astype(np.int64))


def prologue_token_admissible(codes_gpu, scale_gpu, y_oracle, norm_oracle, rotate=True, ue8m0=False):
    """Bar of the fused key prologue for one token whose stored codes / scale differ from the
    oracle's.  The oracle normalises exactly (float64, one rounding to bf16); the kernel normalises
    in fp32, so one or two of its bf16 norm outputs may sit one bf16 unit u away from the oracle's
    (where the exact value is that close to a rounding boundary), u = the bf16 unit of the largest
    norm output.  Each moved norm output moves the two rotary outputs of its pair by at most u plus
    their own re-rounding (2 u): at most 6 u in L1 size per moved output, 12 u for two.  Without the
    Hadamard rotation that is the perturbation of the pre-quantisation values y directly (at most
    3 u on one value); the rotation's entries all have magnitude 1/sqrt(128), so with it every y_j
    moves by at most 12 u / sqrt(128).  Plus one bf16 unit of y_j for its own rounding:
    delta_j = (12 u / sqrt(128) or 3 u) + ulp(y_j).  Admissible: the scale the quantisation rule
    gives for a block maximum within delta of the oracle's, and every code one that E4M3 rounding
    gives for some value within delta_j / scale of the oracle's y_j / scale."""
    y = np.asarray(y_oracle, np.float64)
    u = float(_bf16_ulp(np.abs(np.asarray(norm_oracle, np.float64)).max()))
    delta = (12.0 * u / np.sqrt(128.0) if rotate else 3.0 * u) + _bf16_ulp(y)
    amax = float(np.abs(y).max())
    dmax = float(delta[int(np.argmax(np.abs(y)))])
    s_lo = float(np.float32(max(amax - dmax, 1e-4) / 448.0))
    s_hi = float(np.float32(max(amax + dmax, 1e-4) / 448.0))
    sg = float(scale_gpu)
    if ue8m0:
        if sg not in (_pow2_at_least(s_lo), _pow2_at_least(s_hi)):
            return False
    elif not (s_lo * (1 - 2.0 ** -22) <= sg <= s_hi * (1 + 2.0 ** -22)):
        return False
    lo = ((y - delta) / sg).astype(np.float32)
    hi = ((y + delta) / sg).astype(np.float32)
    vals = _e4m3_values()
    v_lo = vals[oracle.e4m3_encode_array(lo)]
    v_hi = vals[oracle.e4m3_encode_array(hi)]
    got = vals[np.asarray(codes_gpu, np.uint8)]
    return bool(np.all((got >= v_lo) & (got <= v_hi)))


def compare_prologue_pools(got_pool, ref_pool, keys, w, b, eps, cs, pos, slots, rms, neox, rotate, ue8m0,
                           max_boundary_frac=0.01, key="key_prologue"):
    """Token by token: stored codes and scale equal to the oracle's, or (for at most
    `max_boundary_frac` of the tokens) admissible by prologue_token_admissible().  Bytes of the pool
    that no valid token writes must be equal too.  Records the counts."""
    pages = ref_pool.shape[0]
    written = np.zeros(ref_pool.shape, bool)
    n_tok = n_exact = n_boundary = n_codes = 0
    for t in range(len(slots)):
        sl = int(slots[t])
        if sl < 0 or sl >= pages * 64 or pos[t] < 0 or pos[t] >= cs.shape[0]:
            continue
        pg, row = sl >> 6, sl & 63
        cpos = slice(row * 128, row * 128 + 128)
        spos = slice(64 * 128 + row * 4, 64 * 128 + row * 4 + 4)
        written[pg, cpos] = True
        written[pg, spos] = True
        n_tok += 1
        cg, co = got_pool[pg, cpos], ref_pool[pg, cpos]
        sgb, sob = got_pool[pg, spos], ref_pool[pg, spos]
        if np.array_equal(cg, co) and np.array_equal(sgb, sob):
            n_exact += 1
            continue
        nrm = oracle.k_norm128(keys[t], w, b, eps, rms=rms)
        rop = oracle.rope64(nrm, cs[pos[t]], neox=neox)
        y = oracle.rotate128(rop) if rotate else rop
        yv = oracle.bf16_bits_to_f64(y)
        sg = np.frombuffer(sgb.tobytes(), np.float32)[0]
        assert prologue_token_admissible(cg, sg, yv, oracle.bf16_bits_to_f64(nrm), rotate=rotate, ue8m0=ue8m0), \
            f"token {t}: codes/scale not admissible"
        n_boundary += 1
        n_codes += int((cg != co).sum())
    assert np.array_equal(got_pool[~written], ref_pool[~written]), "bytes outside the stored tokens differ"
    assert n_boundary <= max_boundary_frac * max(1, n_tok), f"{n_boundary} of {n_tok} tokens off the oracle"
    record(key, tokens=n_tok, exact=n_exact, boundary_tokens=n_boundary, boundary_codes=n_codes)
    return n_exact, n_boundary
