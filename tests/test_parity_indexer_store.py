"""GPU parity of kvq_store_indexer_k (the write side of the indexer cache)
against the CPU oracle: every byte of the cache identical (rows, scales,
untouched sentinel bytes), at the long-context size and on small cases
(head_dim 16..256, fp16, all-zero rows, skipped and out-of-range slots,
extreme magnitudes), plus a PDL chain in which the early-metadata gather
reads back the rows the store just wrote."""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import assert_bytes_equal, to_dev

pytestmark = pytest.mark.gpu


def _oracle(orc, wl, slots=None):
    cache = np.full(wl.num_blocks * wl.block_stride, 0xAA, dtype=np.uint8)
    slots = wl.slot_mapping if slots is None else slots
    orc.store_indexer_k(np.ascontiguousarray(wl.k).reshape(-1), wl.head_dim,
                        wl.num_tokens, wl.head_dim, cache, wl.block_stride,
                        wl.block_size, wl.num_blocks, slots, wl.dtype)
    return cache


def _gpu(wl, slots=None, flags=0):
    tdt = torch.float16 if wl.dtype == W.DTYPE_F16 else torch.bfloat16
    k = torch.from_numpy(np.ascontiguousarray(wl.k).view(np.int16)).cuda(
    ).view(tdt)
    cache = torch.full((wl.num_blocks, wl.block_size, wl.head_dim + 4), 0xAA,
                       dtype=torch.uint8, device="cuda")
    sm = to_dev(wl.slot_mapping if slots is None else slots)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_store_indexer_k(k, cache, sm, flags=flags, dev_error=err)
    torch.cuda.synchronize()
    return cache, int(err.item())


def _compare(orc, wl):
    cache, err = _gpu(wl)
    assert err == 0
    assert_bytes_equal(cache.cpu().numpy().reshape(-1), _oracle(orc, wl),
                       wl.name)


def test_long_context(orc):
    _compare(orc, W.make_indexer_store("long", 80, [512] * 256, 64, 128,
                                       8192))


CASES = [
    ("d16", [5, 40], 16, 16, 8, W.DTYPE_BF16),
    ("d32_fp16", [33, 1, 0, 64], 8, 32, 32, W.DTYPE_F16),
    ("d64", [100], 16, 64, 10, W.DTYPE_BF16),
    ("d256", [7, 300], 32, 256, 24, W.DTYPE_BF16),
    ("d128_fp16", [257, 3], 64, 128, 10, W.DTYPE_F16),
    ("block_size_12", [30, 11], 12, 128, 8, W.DTYPE_BF16),
]


@pytest.mark.parametrize("name,lens,B,D,nb,dtype", CASES,
                         ids=[c[0] for c in CASES])
def test_case(orc, name, lens, B, D, nb, dtype):
    _compare(orc, W.make_indexer_store(name, 81, lens, B, D, nb, dtype))


def test_zero_rows_extremes_skips_and_flags(orc):
    wl = W.make_indexer_store("edge", 82, [40, 24], 16, 128, 8, spread=30)
    k = wl.k.copy()
    k[3] = 0                      # an all-zero row
    k[5, :7] = 0x8000             # negative zeros
    wl.k = k
    slots = wl.slot_mapping.copy()
    slots[10] = -1                # skipped
    slots[11] = 8 * 16 + 5        # beyond the cache: flagged, skipped
    cache, err = _gpu(wl, slots=slots)
    assert err == kvq.KVQ_DEVERR_SLOT
    slots_o = slots.copy()
    slots_o[11] = -1
    assert_bytes_equal(cache.cpu().numpy().reshape(-1),
                       _oracle(orc, wl, slots_o), "edge")


def test_pdl_gather_reads_rows_just_stored(orc):
    wl = W.make_indexer_store("chain", 83, [512] * 64, 64, 128, 1024)
    tdt = torch.bfloat16
    k = torch.from_numpy(wl.k.view(np.int16)).cuda().view(tdt)
    cache = torch.full((wl.num_blocks, wl.block_size, wl.head_dim + 4), 0xAA,
                       dtype=torch.uint8, device="cuda")
    n = wl.num_tokens
    out_k = torch.empty((n, 128), dtype=torch.uint8, device="cuda")
    out_s = torch.empty((n, 4), dtype=torch.uint8, device="cuda")
    kvq.kvq_store_indexer_k(k, cache, to_dev(wl.slot_mapping),
                            flags=kvq.KVQ_F_PDL)
    kvq.kvq_gather_indexer_k(cache, out_k, out_s, to_dev(wl.block_table),
                             to_dev(wl.cu_seq_lens),
                             flags=kvq.KVQ_F_PDL_EARLY_META)
    torch.cuda.synchronize()
    ref = _oracle(orc, wl).reshape(wl.num_blocks, -1)
    rows = np.empty((n, 128), np.uint8)
    scs = np.empty((n, 4), np.uint8)
    for i, slot in enumerate(wl.slot_mapping):
        blk, off = divmod(int(slot), 64)
        rows[i] = ref[blk, off * 128:(off + 1) * 128]
        scs[i] = ref[blk, 64 * 128 + 4 * off: 64 * 128 + 4 * off + 4]
    assert_bytes_equal(out_k.cpu().numpy().reshape(-1), rows.reshape(-1),
                       "rows")
    assert_bytes_equal(out_s.cpu().numpy().reshape(-1), scs.reshape(-1),
                       "scales")


@pytest.mark.parametrize("amax_mult", [1.0, 1.1, 0.73])
def test_quotients_on_e4m3_midpoints(orc, amax_mult):
    """Rows whose quotients k / scale fall exactly on e4m3 rounding
    midpoints (ties, where the kernel's division fast path must hand over to
    the IEEE division) and one bf16 step either side of them."""
    e4 = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mids = (e4[8:-1] + e4[9:]) / 2          # normal-range midpoints
    rng = np.random.default_rng(84)
    T, D = 64, 128
    x = np.zeros((T, D), np.float64)
    for t in range(T):
        e = 2.0 ** rng.integers(-8, 8)
        row = rng.choice(mids, D) * np.where(rng.random(D) < .5, -1, 1) * e
        row[0] = 448.0 * e * amax_mult
        x[t] = row
    bits = W.bf16_bits(x.astype(np.float32).reshape(-1)).reshape(T, D)
    near = bits.astype(np.int32) + rng.integers(-1, 2, size=bits.shape)
    near[:, 0] = bits[:, 0]
    bits[T // 2:] = near[T // 2:].astype(np.uint16)
    slots = np.arange(T, dtype=np.int64)
    wl = W.IndexerStoreWorkload(
        name="midpoints", k=bits, num_tokens=T, head_dim=D, block_size=16,
        num_blocks=T // 16, slot_mapping=slots,
        block_table=np.arange(T // 16, dtype=np.int32)[None, :],
        cu_seq_lens=np.array([0, T], np.int32))
    _compare(orc, wl)


@pytest.mark.parametrize("f16", [False, True], ids=["bf16", "fp16"])
@pytest.mark.parametrize("mult", [3.0, 5.0, 0.75, 1.25])
def test_midpoints_with_exact_non_power_of_two_scale(orc, mult, f16):
    """Rows whose amax is 448 * mult * 2^e, so that scale = amax / 448 is
    exact but not a power of two, and whose other elements are e4m3
    midpoints times mult * 2^e (exact in bf16): every quotient is exactly a
    rounding midpoint (ties to even), the case in which the kernel's
    division-free products cannot decide and the IEEE quotient must."""
    e4 = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mids = (e4[8:-1] + e4[9:]) / 2
    rng = np.random.default_rng(85)
    T, D = 64, 128
    x = np.zeros((T, D), np.float64)
    for t in range(T):
        e = 2.0 ** (rng.integers(-6, 4) if f16 else rng.integers(-8, 8))
        row = rng.choice(mids, D) * np.where(rng.random(D) < .5, -1, 1)
        row = row * mult * e
        row[0] = 448.0 * mult * e
        x[t] = row
    xf = x.astype(np.float32)
    if f16:
        bits = xf.astype(np.float16).view(np.uint16)
        back = bits.view(np.float16).astype(np.float32)
    else:
        bits = W.bf16_bits(xf.reshape(-1)).reshape(T, D)
        back = (bits.astype(np.uint32) << 16).view(np.float32)
    # every value above is exact in the input type (<= 8 significant bits)
    assert np.array_equal(back, xf)
    slots = np.arange(T, dtype=np.int64)
    wl = W.IndexerStoreWorkload(
        name="exact_mid", k=bits, num_tokens=T, head_dim=D, block_size=16,
        num_blocks=T // 16, slot_mapping=slots,
        block_table=np.arange(T // 16, dtype=np.int32)[None, :],
        cu_seq_lens=np.array([0, T], np.int32),
        dtype=W.DTYPE_F16 if f16 else W.DTYPE_BF16)
    _compare(orc, wl)


def test_tiny_scales_take_the_exact_path(orc):
    """Rows whose amax is so small that scale = amax / 448 is below 2^-125
    (1 / scale may overflow), mixed with ordinary rows, and rows of bf16
    subnormals beside large values."""
    rng = np.random.default_rng(86)
    T, D = 48, 128
    x = rng.standard_normal((T, D)).astype(np.float32)
    x[0:8] *= np.float32(2.0 ** -118)
    x[8:16] *= np.float32(2.0 ** -126)
    x[16:24, :5] = np.float32(2.0 ** -130)
    x[16:24, 5] = np.float32(3.0e4)
    bits = W.bf16_bits(x.reshape(-1)).reshape(T, D)
    slots = np.arange(T, dtype=np.int64)
    wl = W.IndexerStoreWorkload(
        name="tiny_scale", k=bits, num_tokens=T, head_dim=D, block_size=16,
        num_blocks=T // 16, slot_mapping=slots,
        block_table=np.arange(T // 16, dtype=np.int32)[None, :],
        cu_seq_lens=np.array([0, T], np.int32))
    _compare(orc, wl)


def test_quotients_within_an_ulp_of_a_midpoint(orc):
    """Rows where 448 * k == m * amax exactly for the e4m3 midpoint
    m = 1.3125 * 2^j while amax / 448 is inexact (amax has no factor 7):
    k / scale then lies within one fp32 ulp of m without equalling it, so
    the fp32 quotient lands on m (an e4m3 tie) for some elements and next
    to it for others -- the double-rounding case the kernel's products must
    settle exactly."""
    rng = np.random.default_rng(87)
    T, D = 256, 128
    x = np.zeros((T, D), np.float64)
    for t in range(T):
        a_int = int(rng.integers(32, 64))
        while a_int % 7 == 0:
            a_int = int(rng.integers(32, 64))
        a = a_int * 2.0 ** int(rng.integers(-20, 10))
        x[t, 0] = a
        j = rng.integers(-6, 9, size=D - 1)
        x[t, 1:] = (3 * a / 1024 * 2.0 ** j
                    * np.where(rng.random(D - 1) < .5, -1, 1))
    xf = x.astype(np.float32)
    assert np.array_equal(xf.astype(np.float64), x)
    bits = W.bf16_bits(xf.reshape(-1)).reshape(T, D)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32),
                          xf)
    slots = np.arange(T, dtype=np.int64)
    wl = W.IndexerStoreWorkload(
        name="near_mid", k=bits, num_tokens=T, head_dim=D, block_size=16,
        num_blocks=T // 16, slot_mapping=slots,
        block_table=np.arange(T // 16, dtype=np.int32)[None, :],
        cu_seq_lens=np.array([0, T], np.int32))
    _compare(orc, wl)


def test_long_context_early_read(orc):
    """KVQ_F_PDL_EARLY_READ: the first rows are loaded before the wait on
    the predecessor, every write after it -- same bytes as the oracle."""
    wl = W.make_indexer_store("long_er", 88, [512] * 256, 64, 128, 8192)
    cache, err = _gpu(wl, flags=kvq.KVQ_F_PDL_EARLY_READ)
    assert err == 0
    assert_bytes_equal(cache.cpu().numpy().reshape(-1), _oracle(orc, wl),
                       wl.name)


def test_early_read_chain_of_stores(orc):
    """Early-read stores back to back into the same slots, alternating two
    inputs (the kernel before each writes the cache, none of its inputs):
    the cache holds exactly the last store's bytes."""
    a = W.make_indexer_store("a", 89, [512] * 64, 64, 128, 1024)
    b = W.make_indexer_store("b", 90, [512] * 64, 64, 128, 1024)
    b.slot_mapping = a.slot_mapping.copy()
    ks = [torch.from_numpy(w.k.view(np.int16)).cuda().view(torch.bfloat16)
          for w in (a, b)]
    cache = torch.full((a.num_blocks, a.block_size, a.head_dim + 4), 0xAA,
                       dtype=torch.uint8, device="cuda")
    sm = to_dev(a.slot_mapping)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(7):
        kvq.kvq_store_indexer_k(ks[i % 2], cache, sm,
                                flags=kvq.KVQ_F_PDL_EARLY_READ, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bytes_equal(cache.cpu().numpy().reshape(-1), _oracle(orc, a), "a")
