"""Failure detection without a GPU fault: a CTA of the first pass never
fills its first shared-memory stage (host-side hook), its warps' bounded
waits on the stage run out after about a second, the CTA raises the device
flag and stops; the host reads DRS_ERR_DEVICE_TIMEOUT and the context keeps
working."""
import time

import numpy as np
import pytest
import torch

import workloads
from gpu_util import drs, gpu_row_stats, oracle_rows
from parity import check_row_stats

pytestmark = pytest.mark.gpu


def test_withheld_record_times_out_and_is_reported():
    lib = drs()
    w = workloads.make("tiny")
    x, t = w["logits"].cuda(), w["temps"].cuda()
    lib.drs_test_inject_fault(1)
    t0 = time.time()
    lib.row_stats(x, t, 16, 0, torch.bfloat16)
    status = lib.drs_get_device_error()
    elapsed = time.time() - t0
    assert status == lib.DRS_ERR_DEVICE_TIMEOUT
    assert 0.5 < elapsed < 30.0
    # the flag was cleared by reading it, and the next call is correct
    assert lib.drs_get_device_error() == lib.DRS_OK
    g = gpu_row_stats(x, t, 16, 0, 1)
    r = oracle_rows(x, w["temps"].numpy(), 16, 0, 1, np.arange(64))
    check_row_stats(g, r, 1, "after timeout")
