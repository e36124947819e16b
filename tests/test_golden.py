"""Golden fixtures: the constants the pages print, and the oracle's regression values on the tiny
workload (written by tests/golden/make_golden.py, which calls only the oracle)."""
import json
import os

import pytest

import oracle
from deepseek_sparse_attention_paged_gb300 import workloads

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_page_constants_used_by_oracle_and_generator():
    c = json.load(open(os.path.join(HERE, "page_constants.json")))
    assert oracle.PAGE == c["page_size"]["value"] == workloads.PAGE
    assert oracle.ROW_BYTES == c["index_row_bytes"]["value"] == workloads.INDEX_ROW_BYTES
    assert oracle.HI == c["index_heads"]["value"] == workloads.INDEX_HEADS
    assert oracle.DI == c["index_head_dim"]["value"] == c["quant_block"]["value"]
    assert oracle.DQK == c["mla_head_size"]["value"] == workloads.LATENT_DIM
    assert oracle.DV == c["mla_latent_dim"]["value"]
    assert oracle.DQK - oracle.DV == c["mla_rope_dim"]["value"]
    assert workloads.make("decode_b32_8k").topk == c["topk"]["value"]


def test_tiny_oracle_regression():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    want = json.load(open(os.path.join(HERE, "tiny_oracle.json")))
    got = mod.compute()
    assert got == want
