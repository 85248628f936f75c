"""GPU parity of kvq_store_nvfp4 against the CPU oracle: every byte of the
cache (written pages and untouched sentinel bytes) must be identical.

Covers the five named workloads' store parts at their full sizes (in the
launch configuration the benchmark uses), small ragged and degenerate
cases (one token, odd head counts, more than 256 chunks per token, a
non-power-of-two block size, NHD, swizzled K scales, strided rows, all
tokens skipped, zero tokens), an out-of-range slot, and crafted groups that
put the hardware conversions on every e2m1 and e4m3 rounding boundary.
"""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import assert_bytes_equal, gpu_store
from tests.test_oracle_store import SMALL_CASES, run_store

pytestmark = pytest.mark.gpu


def _compare(orc, wl):
    got, err = gpu_store(wl)
    want = run_store(orc, wl)
    assert err == 0
    assert_bytes_equal(got, want, wl.name)


@pytest.mark.parametrize("index", [0, 1, 2, 4])
def test_named_workload(orc, index):
    _compare(orc, W.store_workload(index))


FP16_CASES = [
    dict(name="fp16_decode_shape", seed=50, num_tokens=256, num_heads=8,
         head_size=128, block_size=16, num_blocks=4096),
    dict(name="fp16_prefill_shape", seed=51, num_tokens=4096, num_heads=8,
         head_size=128, block_size=16, num_blocks=1024, slots="runs",
         request_len=1024, row_mult=2, outlier_p=1e-3, outlier_mult=50.0),
    dict(name="fp16_long_shape_nhd", seed=52, num_tokens=8192, num_heads=4,
         head_size=256, block_size=32, num_blocks=512, slots="runs",
         request_len=512, layout=W.LAYOUT_NHD),
    dict(name="fp16_ragged_odd_heads", seed=53, num_tokens=37, num_heads=3,
         head_size=64, block_size=16, num_blocks=9, skip=5, flags=1),
    dict(name="fp16_tiny_scale", seed=54, num_tokens=16, num_heads=2,
         head_size=64, block_size=8, num_blocks=4, scales=(1e-4, 3e-5)),
]


@pytest.mark.parametrize("case", FP16_CASES, ids=lambda c: c["name"])
def test_fp16_input(orc, case):
    c = dict(case)
    _compare(orc, W.make_store(c.pop("name"), c.pop("seed"),
                               dtype=W.DTYPE_F16, **c))


EDGE_CASES = SMALL_CASES + [
    dict(name="one_token", seed=10, num_tokens=1, num_heads=1, head_size=64,
         block_size=4, num_blocks=3),
    dict(name="odd_heads_ragged", seed=11, num_tokens=37, num_heads=3,
         head_size=64, block_size=16, num_blocks=9, skip=5),
    dict(name="wide_token_slices", seed=12, num_tokens=23, num_heads=16,
         head_size=256, block_size=8, num_blocks=5, skip=2),
    dict(name="head_size_512", seed=13, num_tokens=11, num_heads=2,
         head_size=512, block_size=4, num_blocks=4),
    dict(name="head_size_192", seed=14, num_tokens=29, num_heads=5,
         head_size=192, block_size=8, num_blocks=6, layout=W.LAYOUT_NHD),
    dict(name="block_size_12", seed=15, num_tokens=40, num_heads=2,
         head_size=128, block_size=12, num_blocks=5),
    dict(name="runs_strided", seed=16, num_tokens=96, num_heads=4,
         head_size=128, block_size=16, num_blocks=12, slots="runs",
         request_len=32, row_mult=2, flags=1),
    dict(name="outliers", seed=17, num_tokens=64, num_heads=8,
         head_size=128, block_size=16, num_blocks=8, outlier_p=0.01,
         outlier_mult=300.0),
    dict(name="tiny_scale_saturates", seed=18, num_tokens=16, num_heads=2,
         head_size=64, block_size=8, num_blocks=4, scales=(1e-4, 3e-5)),
    dict(name="huge_scale_underflows", seed=19, num_tokens=16, num_heads=2,
         head_size=64, block_size=8, num_blocks=4, scales=(500.0, 90.0)),
]


@pytest.mark.parametrize("case", EDGE_CASES, ids=lambda c: c["name"])
def test_edge_case(orc, case):
    c = dict(case)
    _compare(orc, W.make_store(c.pop("name"), c.pop("seed"), **c))


def test_all_tokens_skipped(orc):
    wl = W.make_store("skip_all", 20, 9, 2, 64, 8, 4)
    wl.slot_mapping[:] = -1
    got, err = gpu_store(wl)
    assert err == 0 and (got == 0xAA).all()


def test_zero_tokens():
    wl = W.make_store("empty", 21, 0, 2, 64, 8, 4, slots="dense")
    got, err = gpu_store(wl)
    assert err == 0 and (got == 0xAA).all()


def test_out_of_range_slot_is_flagged_and_skipped(orc):
    wl = W.make_store("oob", 22, 12, 2, 64, 8, 4)
    bad = wl.slot_mapping.copy()
    bad[5] = wl.num_blocks * wl.block_size + 3
    got, err = gpu_store(wl, slot_mapping=bad)
    assert err == kvq.KVQ_DEVERR_SLOT
    wl.slot_mapping = bad.copy()
    wl.slot_mapping[5] = -1
    assert_bytes_equal(got, run_store(orc, wl), "oob")


# --- hardware conversions on every rounding boundary ---------------------------

def _e2m1_probe_values():
    """bf16 values in [-6, 6] on and around every e2m1 boundary."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)
    mids = (grid[:-1] + grid[1:]) / 2
    vals = [grid, mids]
    for m in mids:                      # one bf16 ulp either side
        b = np.float32(m).view(np.uint32) >> 16
        vals.append(((np.array([b - 1, b + 1], np.uint32)) << 16)
                    .view(np.float32))
    vals.append(np.float32([0.0, 1e-30, 2.0 ** -130, 5.99, 0.01]))
    v = np.concatenate(vals)
    v = np.concatenate([v, -v])
    return v[np.abs(v) <= 6]


def test_e2m1_boundaries(orc):
    """Groups [6, v1..v15] with g = 1 have sf = 1.0 and r = 1, so every
    v_i goes straight through the e2m1 conversion."""
    vals = _e2m1_probe_values()
    n_groups = -(-vals.size // 15)
    pad = np.zeros(n_groups * 15, np.float32)
    pad[: vals.size] = vals
    groups = np.concatenate([np.full((n_groups, 1), 6.0, np.float32),
                             pad.reshape(n_groups, 15)], axis=1)
    _probe_store(orc, groups, 1.0)


def _e4m3_probe_amax():
    """amax values whose amax/6 is every e4m3 value and midpoint (all exact
    in bf16), plus one bf16 ulp either side."""
    v = np.array([orc_val for orc_val in _e4m3_table()], np.float64)
    mids = (v[:-1] + v[1:]) / 2
    a = np.concatenate([v, mids]) * 6
    a = a[(a > 0) & (a < 3.3e38)].astype(np.float32)
    bits = a.view(np.uint32) >> 16
    assert ((a.view(np.uint32) & 0xFFFF) == 0).all()
    near = np.concatenate([bits - 1, bits + 1]).astype(np.uint32) << 16
    return np.concatenate([a, near.view(np.float32)])


def _e4m3_table():
    codes = torch.arange(127, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().tolist()


def test_e4m3_boundaries(orc):
    """Groups whose amax puts (amax/6)*g on every e4m3 value, midpoint and
    saturation boundary (g = 1)."""
    amax = _e4m3_probe_amax()
    amax = np.concatenate([amax, np.float32([448 * 6, 464 * 6, 500 * 6])])
    rng = np.random.default_rng(5)
    groups = rng.uniform(-1, 1, (amax.size, 16)).astype(np.float32)
    groups *= amax[:, None]
    groups[:, 3] = amax
    groups[:, 9] = -amax * np.float32(0.5)
    _probe_store(orc, groups, 1.0)


@pytest.mark.parametrize("scale", [1.0, 0.37, 2.0 ** -20])
def test_every_bf16_amax(orc, scale):
    """One group per finite non-negative bf16 amax (32640 groups): covers the
    kernel's division-free amax / 6 on every value it can see, and with
    k_scale = 2^-20 the overflow of (amax/6)*g to +inf (saturates to 448)."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    a = (bits << 16).view(np.float32)
    groups = np.zeros((a.size, 16), np.float32)
    groups[:, 0] = a
    groups[:, 5] = -a * np.float32(0.375)
    groups[:, 11] = a * np.float32(0.5)
    groups[:, 14] = -a
    _probe_store(orc, groups, scale)


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -20])
def test_every_fp16_amax(orc, scale):
    """One group per finite non-negative fp16 amax (31744 groups), fp16
    inputs (subnormals included)."""
    bits = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    a = bits.view(np.float16).astype(np.float32)
    groups = np.zeros((a.size, 16), np.float32)
    groups[:, 0] = a
    groups[:, 5] = -a * np.float32(0.375)
    groups[:, 11] = a * np.float32(0.5)
    groups[:, 14] = -a
    _probe_store(orc, groups, scale, dtype=W.DTYPE_F16)


def _probe_store(orc, groups, scale, dtype=W.DTYPE_BF16):
    """Store each 16-value group as one head of one token (H=1, D=16*...)."""
    n = groups.shape[0]
    per_tok = 4                          # head_size 64 = 4 groups
    T = -(-n // per_tok)
    x = np.zeros((T * per_tok, 16), np.float32)
    x[:n] = groups
    bits = W.element_bits(x.reshape(-1), dtype)
    src = np.concatenate([bits, bits[::-1].copy()])
    wl = W.StoreWorkload(
        name="probe", num_tokens=T, num_heads=1, head_size=64, block_size=4,
        num_blocks=-(-T // 4), src=src, key_offset=0, key_stride0=64,
        value_offset=T * 64, value_stride0=64,
        slot_mapping=np.arange(T, dtype=np.int64),
        k_scale=np.float32(scale), v_scale=np.float32(scale), dtype=dtype)
    _compare(orc, wl)
