"""Writes tests/golden/tiny_oracle.json: regression values of the CPU oracle on the tiny workload
(2 requests, contexts 300 and 1000, seed 0).  Calls only the oracle and the input generator."""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from deepseek_sparse_attention_paged_gb300 import workloads  # noqa: E402


def compute():
    wl = workloads.make("tiny")
    pool = np.zeros((wl.num_pages, oracle.PAGE_BYTES), np.uint8)
    oracle.store_index_k(wl.index_keys(), wl.token_slots(), pool)
    rows = np.arange(wl.T)
    lg = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                               rows, wl.max_seq_len)
    idx = oracle.topk(lg, wl.seq_lens, wl.cu_q, rows, wl.topk)
    out, lse = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, idx,
                                 wl.scale, rows)
    return {
        "workload": "tiny",
        "index_pool_sha256": hashlib.sha256(pool.tobytes()).hexdigest(),
        "logits_row0_first8": [float(x) for x in lg[0, :8]],
        "logits_row1_last8": [float(x) for x in lg[1, 992:1000]],
        "topk_row0_first16": idx[0, :16].tolist(),
        "topk_row1_first16": idx[1, :16].tolist(),
        "topk_sha256": hashlib.sha256(idx.tobytes()).hexdigest(),
        "mla_out_r0h0_first8": [float(x) for x in out[0, 0, :8]],
        "mla_lse_row1": [float(x) for x in lse[1]],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
