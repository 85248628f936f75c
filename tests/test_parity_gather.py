"""GPU parity of kvq_gather_indexer_k against the CPU oracle: both outputs
(K rows and scale bytes) identical, rows past the end untouched.

Covers the named workloads' gather parts at full size, sequences of 0, 1,
63, 64, 65 and 8192 tokens (the first published gather dropped the tail of
long sequences), head_dim other than 128 (the generic copy path), a block
table with a row stride wider than its used part, a total larger than
cu_seq_lens[-1] (flagged, extra rows untouched), and an out-of-range block
id (flagged, row untouched).  Each case also runs with
KVQ_F_PDL_EARLY_READ (cache reads issued before the wait on the
predecessor, every write after it), which must give the same bytes and
flags.
"""
import numpy as np
import pytest

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import assert_bytes_equal, gpu_gather
from tests.test_oracle_gather import run_gather

pytestmark = pytest.mark.gpu
FLAGS = [0, kvq.KVQ_F_PDL_EARLY_READ]
FLAG_IDS = ["plain", "early_read"]


def _compare(orc, wl, total=None, bt_cols=None, flags=0):
    k, s, err = gpu_gather(wl, total=total, bt_cols=bt_cols, flags=flags)
    wk, ws = run_gather(orc, wl, total=total)
    n = wl.total_tokens if total is None else total
    assert_bytes_equal(k, wk[: n * wl.head_dim], wl.name + " k_fp8")
    assert_bytes_equal(s, ws[: n * 4], wl.name + " k_scale")
    return err


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("index", [0, 3, 4])
def test_named_workload(orc, index, flags):
    assert _compare(orc, W.gather_workload(index), flags=flags) == 0


CASES = [
    ("boundaries_d32", [0, 1, 63, 64, 65, 0, 130], 16, 32, 64, 0),
    ("boundaries_d128", [0, 1, 63, 64, 65, 0, 130], 64, 128, 32, 0),
    ("long_8192", [8192, 1, 64, 3], 64, 128, 600, 0),
    ("d64_b32", [77, 5, 300], 32, 64, 40, 0),
    ("d256_wide_table", [90, 17], 16, 256, 30, 12),  # kernel sees 6 cols
    ("single_token", [1], 64, 128, 2, 0),
    ("many_short", [3] * 200, 4, 16, 400, 0),
    # more sequences than fit in the kernel's shared-memory copy of
    # cu_seq_lens: the search reads global memory instead
    ("many_seqs_global_cu", [1, 2, 0, 3] * 3300, 16, 16, 13300, 0),
    # a block table too large to stage: only cu_seq_lens goes to shared
    # memory and block ids are read from global memory
    ("big_table_global_bt", [11000] + [7] * 19, 16, 16, 14000, 700),
]


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("name,lens,B,D,nb,mb", CASES,
                         ids=[c[0] for c in CASES])
def test_case(orc, name, lens, B, D, nb, mb, flags):
    wl = W.make_gather(name, 30, lens, B, D, nb, max_blocks=mb)
    cols = None
    if mb and name == "d256_wide_table":
        cols = int(((np.asarray(lens) + B - 1) // B).max())
    assert _compare(orc, wl, bt_cols=cols, flags=flags) == 0


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_total_beyond_cu_is_flagged(orc, flags):
    wl = W.make_gather("beyond", 31, [20, 45], 16, 128, 8)
    err = _compare(orc, wl, total=wl.total_tokens + 5, flags=flags)
    assert err == kvq.KVQ_DEVERR_SEQ


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_bad_block_id_is_flagged(orc, flags):
    wl = W.make_gather("badblk", 32, [20, 45], 16, 128, 8)
    bt = wl.block_table.copy()
    bt[1, 1] = 10_000
    k, s, err = gpu_gather(wl, block_table=bt, flags=flags)
    assert err == kvq.KVQ_DEVERR_BLOCK
    # rows of the bad block stay untouched; the rest match the oracle
    wk, ws = run_gather(orc, wl)
    rows = np.arange(wl.total_tokens)
    bad = (rows >= 20 + 16) & (rows < 20 + 32)
    kr, wkr = k.reshape(-1, 128), wk.reshape(-1, 128)
    assert (kr[bad] == 0xCD).all()
    assert_bytes_equal(kr[~bad].reshape(-1), wkr[~bad].reshape(-1), "badblk")
    sr, wsr = s.reshape(-1, 4), ws.reshape(-1, 4)
    assert (sr[bad] == 0xCD).all()
    assert_bytes_equal(sr[~bad].reshape(-1), wsr[~bad].reshape(-1), "badblk")


def test_scale_view_float32():
    wl = W.gather_workload(4)
    k, s, err = gpu_gather(wl)
    v = s.view(np.float32)
    assert err == 0 and (v >= 1e-4 * 0.999).all() and (v <= 1.0).all()
