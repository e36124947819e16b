"""Seeded synthetic workloads for the DSA decode path.

This module only draws inputs: context lengths, page assignments, bf16 keys and queries, head
gates and the latent cache.  It holds none of the method's arithmetic (no rotation, no
quantisation, no scoring, no attention), so both the CUDA path and the CPU oracle may consume
what it produces.

Streams: ``numpy.random.SeedSequence(seed).spawn(7)`` gives one independent stream per input, in
this order: context lengths, page assignment, index keys, indexer queries, head gates, latent
cache, MLA queries.  The two large streams (index keys, latent cache) are further split into
fixed-size chunks, each with its own child seed, so that they can be drawn by several threads and
still give the same values on any machine.  Values are N(0, 1) drawn in float32 and rounded to
bf16 (round-to-nearest-even, by torch's conversion) -- bf16 tensors are carried as uint16 bits.

Named workloads (sizes from the decode scenarios the path is measured on):

====================  ========================================================================
``tiny``              2 requests, contexts 300 and 1000, 1 query token each; 21 pages in a
                      random permutation; top-k 256; 16 MLA heads; seed 0
``decode_b32_8k``     32 requests x 8192 tokens, 1 query token each; 4096 shuffled pages;
                      top-k 2048; 128 MLA heads; seed 1
``decode_b64_logu64k``  64 requests, contexts log-uniform in [4096, 65536], 1 query token each;
                      pages scattered over a 2M-token (32768-page) pool; top-k 2048; 128 heads;
                      seed 2
``mtp_b8_128k``       8 requests x 131072 tokens, 2 query tokens each (next_n = 2); 16384
                      shuffled pages; top-k 2048; 128 heads; seed 3
``prefill_32k_4k``    1 request: 32768 cached prefix tokens plus a 4096-token new chunk
                      (4096 query rows, causal); 576 shuffled pages; top-k 2048; 128 heads; seed 4
====================  ========================================================================
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

PAGE = 64            # page size of both caches (one shared block table)
INDEX_HEADS = 64     # lightning-indexer heads
INDEX_DIM = 128      # lightning-indexer head dim
INDEX_ROW_BYTES = 132
INDEX_PAGE_BYTES = PAGE * INDEX_ROW_BYTES
LATENT_DIM = 576     # 512 latent + 64 rope
VALUE_DIM = 512
MLA_SCALE = 1.0 / math.sqrt(192.0)   # softmax scale 1/sqrt(qk_nope 128 + qk_rope 64)

_STREAMS = ("lengths", "pages", "index_keys", "index_q", "weights", "latent", "mla_q")
_KEY_CHUNK = 1 << 14          # tokens per child stream of the index-key draw
_LATENT_CHUNK_PAGES = 256     # pages per child stream of the latent-cache draw


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits (uint16), round-to-nearest-even via torch's conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _normal_bf16_chunked(seq: np.random.SeedSequence, n_chunks: int, chunk_elems: int,
                         total_elems: int) -> np.ndarray:
    """N(0,1) bf16 bits, chunk i drawn from child i of ``seq`` (thread-count independent)."""
    kids = seq.spawn(n_chunks)
    out = np.empty(total_elems, np.uint16)

    def fill(i: int) -> None:
        lo = i * chunk_elems
        hi = min(total_elems, lo + chunk_elems)
        g = np.random.Generator(np.random.PCG64(kids[i]))
        out[lo:hi] = _to_bf16_bits(g.standard_normal(hi - lo, dtype=np.float32))

    if n_chunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


@dataclass
class Workload:
    """One synthetic batch: metadata up front, large tensors drawn on first use."""

    name: str
    seed: int
    seq_lens: np.ndarray          # int32 [B]   cached tokens per request, this step's included
    q_lens: np.ndarray            # int32 [B]   query tokens per request
    block_table: np.ndarray       # int32 [B, max_pages], unused tail entries = -1
    num_pages: int                # pages in each pool
    topk: int
    heads: int                    # MLA heads
    scale: float = MLA_SCALE
    _streams: dict = field(default_factory=dict, repr=False)
    _cache: dict = field(default_factory=dict, repr=False)

    # ---- metadata
    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def T(self) -> int:
        return int(self.q_lens.sum())

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max())

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max())

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def visible_lens(self) -> np.ndarray:
        """Keys each query row may see (row j of request b sits at position L_b - q_len_b + j)."""
        out = np.empty(self.T, np.int64)
        r = 0
        for L, ql in zip(self.seq_lens.tolist(), self.q_lens.tolist()):
            for j in range(ql):
                out[r] = max(0, L - ql + j + 1)
                r += 1
        return out

    def token_slots(self) -> np.ndarray:
        """Slot (page * 64 + offset) of every cached token, requests in order (int64)."""
        if "slots" not in self._cache:
            parts = []
            for b, L in enumerate(self.seq_lens.tolist()):
                pos = np.arange(L, dtype=np.int64)
                parts.append(self.block_table[b, pos // PAGE].astype(np.int64) * PAGE + pos % PAGE)
            self._cache["slots"] = np.concatenate(parts) if parts else np.zeros(0, np.int64)
        return self._cache["slots"]

    def new_token_ids(self) -> np.ndarray:
        """Indices (into the token order of ``token_slots``) of this step's query tokens."""
        starts = np.concatenate([[0], np.cumsum(self.seq_lens.astype(np.int64))[:-1]])
        ids = [starts[b] + self.seq_lens[b] - self.q_lens[b] + np.arange(self.q_lens[b])
               for b in range(self.B)]
        return np.concatenate(ids).astype(np.int64)

    # ---- large inputs
    def index_keys(self) -> np.ndarray:
        """bf16 bits [total_tokens, 128]: the indexer key of every cached token, before rotation."""
        if "keys" not in self._cache:
            n = self.total_tokens
            chunks = max(1, -(-n // _KEY_CHUNK))
            flat = _normal_bf16_chunked(self._streams["index_keys"], chunks, _KEY_CHUNK * INDEX_DIM,
                                        n * INDEX_DIM)
            self._cache["keys"] = flat.reshape(n, INDEX_DIM)
        return self._cache["keys"]

    def index_q(self) -> np.ndarray:
        """bf16 bits [T, 64, 128]: indexer queries."""
        if "iq" not in self._cache:
            g = np.random.Generator(np.random.PCG64(self._streams["index_q"]))
            x = g.standard_normal((self.T, INDEX_HEADS, INDEX_DIM), dtype=np.float32)
            self._cache["iq"] = _to_bf16_bits(x)
        return self._cache["iq"]

    def weights(self) -> np.ndarray:
        """float32 [T, 64]: head gates N(0,1) * 64^-0.5 * 128^-0.5."""
        if "w" not in self._cache:
            g = np.random.Generator(np.random.PCG64(self._streams["weights"]))
            x = g.standard_normal((self.T, INDEX_HEADS), dtype=np.float32)
            self._cache["w"] = (x * np.float32(INDEX_HEADS ** -0.5 * INDEX_DIM ** -0.5)).astype(np.float32)
        return self._cache["w"]

    def latent_pool(self) -> np.ndarray:
        """bf16 bits [num_pages, 64, 576]: the latent (MLA) cache, every page N(0,1)."""
        if "kv" not in self._cache:
            chunks = max(1, -(-self.num_pages // _LATENT_CHUNK_PAGES))
            per = _LATENT_CHUNK_PAGES * PAGE * LATENT_DIM
            flat = _normal_bf16_chunked(self._streams["latent"], chunks, per,
                                        self.num_pages * PAGE * LATENT_DIM)
            self._cache["kv"] = flat.reshape(self.num_pages, PAGE, LATENT_DIM)
        return self._cache["kv"]

    def mla_q(self) -> np.ndarray:
        """bf16 bits [T, H, 576]: absorbed MLA queries (512 latent + 64 rope)."""
        if "mq" not in self._cache:
            g = np.random.Generator(np.random.PCG64(self._streams["mla_q"]))
            x = g.standard_normal((self.T, self.heads, LATENT_DIM), dtype=np.float32)
            self._cache["mq"] = _to_bf16_bits(x)
        return self._cache["mq"]

    def drop(self, *names: str) -> None:
        for n in names:
            self._cache.pop(n, None)


def _block_table(seq_lens: Sequence[int], page_ids: np.ndarray) -> np.ndarray:
    need = [-(-int(L) // PAGE) for L in seq_lens]
    width = max(1, max(need) if need else 1)
    bt = np.full((len(seq_lens), width), -1, np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = page_ids[off:off + n]
        off += n
    return bt


def make_custom(name: str, seed: int, seq_lens: Sequence[int], q_lens: Sequence[int] | int,
                topk: int, heads: int, pool_pages: Optional[int] = None) -> Workload:
    """A workload with given context lengths.  Pages are drawn without replacement from a pool of
    ``pool_pages`` (default: exactly the pages needed, in a random permutation)."""
    ss = np.random.SeedSequence(seed)
    streams = dict(zip(_STREAMS, ss.spawn(len(_STREAMS))))
    seq_lens = np.asarray(seq_lens, np.int32)
    if np.isscalar(q_lens):
        q_lens = np.full(seq_lens.shape, int(q_lens), np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    need = int(sum(-(-int(L) // PAGE) for L in seq_lens))
    pool = need if pool_pages is None else int(pool_pages)
    assert pool >= need, "page pool smaller than the pages the contexts need"
    gp = np.random.Generator(np.random.PCG64(streams["pages"]))
    page_ids = gp.permutation(pool)[:need].astype(np.int32)
    return Workload(name=name, seed=seed, seq_lens=seq_lens, q_lens=q_lens,
                    block_table=_block_table(seq_lens, page_ids), num_pages=pool, topk=topk,
                    heads=heads, _streams=streams)


def make(name: str) -> Workload:
    """The named workloads listed in the module docstring."""
    if name == "tiny":
        return make_custom(name, 0, [300, 1000], 1, topk=256, heads=16)
    if name == "decode_b32_8k":
        return make_custom(name, 1, [8192] * 32, 1, topk=2048, heads=128)
    if name == "decode_b64_logu64k":
        ss = np.random.SeedSequence(2)
        streams = dict(zip(_STREAMS, ss.spawn(len(_STREAMS))))
        gl = np.random.Generator(np.random.PCG64(streams["lengths"]))
        u = gl.uniform(math.log(4096.0), math.log(65536.0), size=64)
        seq_lens = np.floor(np.exp(u)).astype(np.int32)
        w = make_custom(name, 2, seq_lens, 1, topk=2048, heads=128, pool_pages=(2 << 20) // PAGE)
        return w
    if name == "mtp_b8_128k":
        return make_custom(name, 3, [131072] * 8, 2, topk=2048, heads=128)
    if name == "prefill_32k_4k":
        return make_custom(name, 4, [32768 + 4096], 4096, topk=2048, heads=128)
    raise KeyError(f"unknown workload {name!r}")


NAMES = ("tiny", "decode_b32_8k", "decode_b64_logu64k", "mtp_b8_128k", "prefill_32k_4k")


@dataclass
class CompressedKV:
    """The compressed-KV companion of a workload (the DSV4 layers with compress ratio 4): request b
    holds floor(L_b / ratio) compressed entries, each with an indexer key and a 576-wide latent row
    drawn N(0, 1) as if written by the model's compressor (a trained module, not drawn here), on
    pages of its own; per-head sink logits N(0, 1); the sliding window and the top-k width over the
    compressed entries.  Streams: SeedSequence(seed + 1000).spawn(4) = pages, index keys, latent
    rows, sinks."""

    base: Workload
    ratio: int
    window: int
    topk: int
    cmp_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray       # int32 [B, max_cmp_pages], unused tail entries = -1
    num_pages: int
    _streams: dict = field(default_factory=dict, repr=False)
    _cache: dict = field(default_factory=dict, repr=False)

    @property
    def max_cmp_len(self) -> int:
        return max(1, int(self.cmp_lens.max()))

    def visible_cmp_lens(self) -> np.ndarray:
        """Compressed entries each query row may see: its visible tokens // ratio."""
        return self.base.visible_lens() // self.ratio

    def slots(self) -> np.ndarray:
        """Slot (page * 64 + offset) of every compressed entry, requests in order (int64)."""
        parts = []
        for b, n in enumerate(self.cmp_lens.tolist()):
            e = np.arange(n, dtype=np.int64)
            parts.append(self.block_table[b, e // PAGE].astype(np.int64) * PAGE + e % PAGE)
        return np.concatenate(parts) if parts else np.zeros(0, np.int64)

    def index_keys(self) -> np.ndarray:
        """bf16 bits [sum cmp_lens, 128]: the indexer key of every compressed entry."""
        if "ik" not in self._cache:
            n = int(self.cmp_lens.astype(np.int64).sum())
            chunks = max(1, -(-n // _KEY_CHUNK))
            self._cache["ik"] = _normal_bf16_chunked(self._streams["keys"], chunks, _KEY_CHUNK * INDEX_DIM,
                                                     n * INDEX_DIM).reshape(n, INDEX_DIM)
        return self._cache["ik"]

    def latent_pool(self) -> np.ndarray:
        """bf16 bits [num_pages, 64, 576]: the compressed latent rows."""
        if "kv" not in self._cache:
            chunks = max(1, -(-self.num_pages // _LATENT_CHUNK_PAGES))
            per = _LATENT_CHUNK_PAGES * PAGE * LATENT_DIM
            flat = _normal_bf16_chunked(self._streams["latent"], chunks, per, self.num_pages * PAGE * LATENT_DIM)
            self._cache["kv"] = flat.reshape(self.num_pages, PAGE, LATENT_DIM)
        return self._cache["kv"]

    def sinks(self) -> np.ndarray:
        """fp32 [heads]: per-head sink logits."""
        g = np.random.Generator(np.random.PCG64(self._streams["sinks"]))
        return g.standard_normal(self.base.heads, dtype=np.float32)


def make_compressed(wl: Workload, ratio: int = 4, window: int = 128, topk: int = 512) -> CompressedKV:
    """The compressed-KV companion of ``wl`` (see CompressedKV)."""
    ss = np.random.SeedSequence(wl.seed + 1000)
    streams = dict(zip(("pages", "keys", "latent", "sinks"), ss.spawn(4)))
    cmp_lens = (wl.seq_lens // ratio).astype(np.int32)
    need = [-(-int(n) // PAGE) for n in cmp_lens]
    pool = max(1, sum(need))
    gp = np.random.Generator(np.random.PCG64(streams["pages"]))
    page_ids = gp.permutation(pool).astype(np.int32)
    width = max(1, max(need))
    bt = np.full((wl.B, width), -1, np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = page_ids[off:off + n]
        off += n
    return CompressedKV(base=wl, ratio=ratio, window=window, topk=topk, cmp_lens=cmp_lens, block_table=bt,
                        num_pages=pool, _streams=streams)
