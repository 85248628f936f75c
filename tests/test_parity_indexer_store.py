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
