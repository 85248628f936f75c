"""Host-side logic of bench.py that needs no GPU: the all-cores CPU
baseline splits the oracle's calls over threads, which must write exactly
the bytes of the single-threaded step."""
import numpy as np
import pytest

import bench
import oracle
from paged_quantized_kv_gb300 import workloads as W


@pytest.mark.parametrize("threads", [1, 3, 7])
def test_threaded_oracle_step_matches_single_thread(threads):
    o = oracle.get()
    # interleaved K/V rows (row stride 2*H*D, nonzero value offset), skipped
    # slots, runs of blocks; sequences of uneven length including empty ones
    st = W.make_store("split_store", 11, 700, 2, 64, 16, 128, slots="runs",
                      request_len=100, row_mult=2, skip=9)
    ga = W.make_gather("split_gather", 12, [5, 0, 130, 64, 1, 0, 77], 64, 128,
                       64, scales="uniform")
    outs = []
    for split in (False, True):
        cache = np.full(st.cache_bytes, 0xAA, dtype=np.uint8)
        k = np.full(ga.total_tokens * ga.head_dim, 0xCD, dtype=np.uint8)
        s = np.full(ga.total_tokens * 4, 0xCD, dtype=np.uint8)
        if split:
            bench.oracle_step_threaded(o, st, ga, cache, k, s, threads)
        else:
            bench.oracle_step(o, st, ga, cache, k, s)
        outs.append((cache, k, s))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    # both steps wrote something (gathered e4m3 bytes may equal the 0xCD fill)
    assert (outs[0][0] != 0xAA).any() and (outs[0][1] != 0xCD).any()
