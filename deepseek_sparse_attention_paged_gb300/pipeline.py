"""Device-side buffers and the four-call DSA decode step, on top of the C-ABI binding.

``DeviceBatch`` uploads one :class:`~deepseek_sparse_attention_paged_gb300.workloads.Workload` to
the GPU (block table, lengths, queries, head gates, latent cache), builds the FP8 index-K cache
with ``dsa_store_index_k`` and owns the outputs (logits, top-k indices, attention output, lse) and
the scratch space.  ``step()`` runs one decode step of the hot path:

    dsa_store_index_k    this step's new keys -> paged FP8 index-K cache
    dsa_indexer_logits   lightning-indexer logits of every query row
    dsa_topk             per-row top-k indices
    dsa_sparse_mla_decode  absorbed sparse MLA over the selected latent rows

Nothing here computes: every step is a call into the CUDA library.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import capi
from .workloads import INDEX_DIM, INDEX_HEADS, INDEX_PAGE_BYTES, LATENT_DIM, VALUE_DIM, Workload


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def logits_ld(max_seq_len: int) -> int:
    """Row stride of the logits buffer: max_seq_len rounded up to 16 bytes."""
    return max(4, (max_seq_len + 3) // 4 * 4)


class DeviceBatch:
    def __init__(self, wl: Workload, device: str = "cuda", with_latent: bool = True,
                 build_index_cache: bool = True, key_chunk: int = 1 << 20):
        self.wl = wl
        self.device = torch.device(device)
        dev = self.device
        self.block_table = torch.from_numpy(wl.block_table).to(dev)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
        self.cu_q = torch.from_numpy(wl.cu_q).to(dev)
        self.index_q = _bf16(wl.index_q(), dev)
        self.weights = torch.from_numpy(wl.weights()).to(dev)
        self.index_pool = torch.zeros((wl.num_pages, INDEX_PAGE_BYTES), dtype=torch.uint8, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        new_ids = wl.new_token_ids()
        self.new_keys = _bf16(wl.index_keys()[new_ids], dev)
        self.new_slots = torch.from_numpy(wl.token_slots()[new_ids]).to(dev)
        if build_index_cache:
            keys = wl.index_keys()
            slots = wl.token_slots()
            for lo in range(0, keys.shape[0], key_chunk):
                k = _bf16(keys[lo:lo + key_chunk], dev)
                s = torch.from_numpy(slots[lo:lo + key_chunk]).to(dev)
                capi.dsa_store_index_k(k, s, self.index_pool, self.dev_err)
            torch.cuda.synchronize(dev)
        self.ld = logits_ld(wl.max_seq_len)
        self.logits = torch.empty((wl.T, self.ld), dtype=torch.float32, device=dev)
        self.idx = torch.empty((wl.T, wl.topk), dtype=torch.int32, device=dev)
        self.idx_ws = torch.empty(max(16, capi.dsa_indexer_logits_workspace_size(wl.T)), dtype=torch.uint8,
                                  device=dev)
        self.topk_ws = torch.empty(max(1, capi.dsa_topk_workspace_size(wl.T, wl.topk, wl.max_seq_len)),
                                   dtype=torch.uint8, device=dev)
        self.kv_pool = None
        self.mla_q = None
        if with_latent:
            self.kv_pool = _bf16(wl.latent_pool(), dev)
            self.mla_q = _bf16(wl.mla_q(), dev)
            self.out = torch.empty((wl.T, wl.heads, VALUE_DIM), dtype=torch.bfloat16, device=dev)
            self.lse = torch.empty((wl.T, wl.heads), dtype=torch.float32, device=dev)
            self.mla_ws = torch.empty(max(16, capi.dsa_sparse_mla_workspace_size(wl.T, wl.heads, wl.topk)),
                                      dtype=torch.uint8, device=dev)

    # ---- the four stages
    def store_new_keys(self, stream=None):
        capi.dsa_store_index_k(self.new_keys, self.new_slots, self.index_pool, self.dev_err, stream=stream)

    def indexer_logits(self, row_begin: int = 0, row_end: Optional[int] = None, logits=None, flags: int = 0,
                       q=None, stream=None):
        capi.dsa_indexer_logits(self.index_q if q is None else q, self.weights, self.index_pool,
                                self.block_table, self.seq_lens, self.cu_q, self.wl.max_seq_len,
                                self.wl.max_q_len, self.logits if logits is None else logits,
                                row_begin=row_begin, row_end=row_end, flags=flags, dev_err=self.dev_err,
                                stream=stream, workspace=self.idx_ws)

    def topk(self, logits=None, idx=None, row_begin: int = 0, row_end: Optional[int] = None, stream=None):
        lg = self.logits if logits is None else logits
        capi.dsa_topk(lg, self.seq_lens, self.cu_q, self.wl.max_seq_len, self.wl.topk,
                      self.idx if idx is None else idx, row_begin=row_begin,
                      row_end=row_end if row_end is not None else row_begin + lg.shape[0],
                      workspace=self.topk_ws, stream=stream)

    def sparse_mla(self, idx=None, stream=None):
        capi.dsa_sparse_mla_decode(self.mla_q, self.kv_pool, self.block_table, self.seq_lens, self.cu_q,
                                   self.idx if idx is None else idx, self.wl.scale, self.out, self.mla_ws,
                                   lse=self.lse, dev_err=self.dev_err, stream=stream)

    def step(self, stream=None):
        """One decode step: store the new keys, score, select, attend."""
        self.store_new_keys(stream)
        self.indexer_logits(stream=stream)
        self.topk(stream=stream)
        self.sparse_mla(stream=stream)

    # ---- end to end: host inputs -> step -> host outputs
    def io_inputs(self):
        """Device tensors a serving loop refills from the host before every step (queries, head
        gates, this step's new keys and slots, lengths, block table), in a fixed order."""
        return [self.index_q, self.weights, self.mla_q, self.new_keys, self.new_slots, self.seq_lens, self.cu_q,
                self.block_table]

    def io_outputs(self):
        """Device tensors a serving loop reads back after every step (attention output, lse)."""
        return [self.out, self.lse]

    def step_io(self, host_in, host_out, stream=None, graph: bool = True):
        """One decode step end to end: copy `host_in` (pinned host tensors shaped like
        io_inputs()) to the device, run step(), copy io_outputs() into `host_out` (pinned host
        tensors).  With graph=True the copies and the four library calls are captured once per
        (host_in, host_out) set as one CUDA graph and replayed on later calls; every replay moves
        the data again.  Returns when the work is enqueued on `stream`."""
        stream = torch.cuda.current_stream(self.device) if stream is None else stream
        ins, outs = self.io_inputs(), self.io_outputs()
        if len(host_in) != len(ins) or len(host_out) != len(outs):
            raise ValueError("host_in / host_out must match io_inputs() / io_outputs()")

        def enqueue():
            for d, h in zip(ins, host_in):
                d.copy_(h, non_blocking=True)
            self.step(stream=torch.cuda.current_stream(self.device))
            for h, d in zip(host_out, outs):
                h.copy_(d, non_blocking=True)

        if not graph:
            with torch.cuda.stream(stream):
                enqueue()
            return
        key = tuple(t.data_ptr() for t in host_in) + tuple(t.data_ptr() for t in host_out)
        g = getattr(self, "_io_graphs", {}).get(key)
        if g is None:
            side = torch.cuda.Stream(self.device)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                enqueue()   # one eager run first (library and allocator warm)
            stream.wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                enqueue()
            stream.wait_stream(side)
            if not hasattr(self, "_io_graphs"):
                self._io_graphs = {}
            self._io_graphs[key] = g
        with torch.cuda.stream(stream):
            g.replay()

    def device_error(self):
        return capi.dsa_read_device_error(self.dev_err)
