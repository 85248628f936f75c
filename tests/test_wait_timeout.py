"""Failure detection without a GPU fault: the metadata staging of the
gather and the load waits on an mbarrier for its TMA bulk copies with a
wall-time limit.  A test-only build of the library expects 16 bytes more
than the copies deliver, so the wait runs out (after 20 ms): the kernel
must report KVQ_DEVERR_TIMEOUT, write none of its rows, return normally,
and leave the context usable (the regular library works right after)."""
import ctypes
import os

import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import build as kbuild
from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import gpu_gather, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def timeout_lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("kvq_timeout") / "libkvq_timeout.so")
    kbuild.build(defines={"KVQ_TEST_EXTRA_TX": 16,
                          "KVQ_WAIT_LIMIT_NS": 20000000}, out=out)
    return out


def test_gather_wait_times_out_and_reports(timeout_lib, monkeypatch):
    wl = W.gather_workload(0)
    saved_path, saved_lib = kvq.LIB_PATH, kvq._lib
    monkeypatch.setattr(kvq, "LIB_PATH", timeout_lib)
    monkeypatch.setattr(kvq, "_lib", None)
    k, s, err = gpu_gather(wl)
    assert err & kvq.KVQ_DEVERR_TIMEOUT
    assert (k == 0xCD).all() and (s == 0xCD).all()  # nothing written
    # the context is still usable: the regular library runs normally
    monkeypatch.setattr(kvq, "LIB_PATH", saved_path)
    monkeypatch.setattr(kvq, "_lib", saved_lib)
    k2, s2, err2 = gpu_gather(wl)
    assert err2 == 0 and not (k2 == 0xCD).all()
    torch.cuda.synchronize()
