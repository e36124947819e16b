"""Failure detection without a GPU fault: the kernels' bounded waits give up and report through the
device error word (a wait on a barrier that nothing ever arrives on), and data-dependent faults are
turned into error bits (covered in the parity tests); afterwards the CUDA context keeps working."""
import numpy as np
import pytest
import torch

from deepseek_sparse_attention_paged_gb300 import capi, workloads
from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_selftest_wait_timeout(err, 2_000_000)   # ~1 ms of SM cycles
    st, word = capi.dsa_read_device_error(err)
    assert st == capi.DSA_ERR_TIMEOUT and word == capi.DSA_DEVERR_TIMEOUT
    # the context is still usable: a normal call succeeds and reports no error
    wl = workloads.make("tiny")
    db = DeviceBatch(wl, with_latent=False)
    db.indexer_logits()
    torch.cuda.synchronize()
    assert db.device_error() == (0, 0)


def test_selftest_rejects_bad_arguments():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.DSAError) as e:
        capi.dsa_selftest_wait_timeout(err, 0)
    assert e.value.status == capi.DSA_ERR_INVALID_ARG
