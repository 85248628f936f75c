"""Pins for the oracle's indexer-K store (CPU only).

The pages give no rule for writing the indexer cache; the reading taken is
per-token absmax scaling, scale = amax / 448, q = e4m3(k / scale).  Pinned by
* exact cases: rows of e4m3 values times 2^e with amax 448 * 2^e store those
  codes (checked against torch's float8_e4m3fn cast) and scale 2^e;
* the e4m3 rounding bound |k - e4m3(q) * scale| <= half an e4m3 step of
  k / scale, times scale; the amax element always stores +-448;
* the scale bytes are the fp32 value amax / 448;
* structure: only the slots' rows and scale entries change, slot -1 writes
  nothing;
* a round trip through the gather oracle returns the stored rows.
"""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import workloads as W
from tests.test_oracle_gather import run_gather


def _cache(nb, B, D, sentinel=0xAA):
    return np.full(nb * B * (D + 4), sentinel, dtype=np.uint8)


def _store(o, bits, T, D, cache, B, nb, slots, dtype=W.DTYPE_BF16):
    o.store_indexer_k(bits, D, T, D, cache, B * (D + 4), B, nb, slots, dtype)


def check_exact_rows(o):
    rng = np.random.default_rng(70)
    T, D, B = 12, 128, 4
    e4m3 = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).float().numpy()
    codes = rng.integers(0, 127, size=(T, D))
    vals = e4m3[codes] * np.where(rng.random((T, D)) < 0.5, -1, 1)
    vals[:, 7] = 448.0
    e = rng.integers(-10, 10, size=(T, 1)).astype(np.float64)
    x = (vals * 2.0 ** e).astype(np.float32)
    bits = W.bf16_bits(x.reshape(-1))
    assert (W.bf16_values(bits) == x.reshape(-1)).all()
    cache = _cache(3, B, D)
    _store(o, bits, T, D, cache, B, 3, np.arange(T))
    blocks = cache.reshape(3, -1)
    for t in range(T):
        blk, off = divmod(t, B)
        row = blocks[blk, off * D:(off + 1) * D]
        want = torch.from_numpy(vals[t].astype(np.float32)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(row, want), t
        sc = blocks[blk, B * D + 4 * off: B * D + 4 * off + 4].view(
            np.float32)[0]
        assert sc == np.float32(2.0 ** e[t, 0])


def check_bound_and_scale(o):
    rng = np.random.default_rng(71)
    e4m3 = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).float().numpy().astype(np.float64)
    for dtype, T, D in ((W.DTYPE_BF16, 40, 128), (W.DTYPE_F16, 20, 64)):
        x = (rng.standard_normal((T, D)) *
             np.where(rng.random((T, D)) < 0.05, 30, 1) *
             10.0 ** rng.uniform(-3, 3, (T, 1))).astype(np.float32)
        x[3] = 0.0  # an all-zero row
        bits = W.element_bits(x.reshape(-1), dtype)
        xv = W.element_values(bits, dtype).reshape(T, D).astype(np.float64)
        B = 8
        nb = (T + B - 1) // B
        cache = _cache(nb, B, D)
        _store(o, bits, T, D, cache, B, nb, np.arange(T), dtype)
        blocks = cache.reshape(nb, -1)
        for t in range(T):
            blk, off = divmod(t, B)
            q = blocks[blk, off * D:(off + 1) * D]
            sc = float(blocks[blk, B * D + 4 * off: B * D + 4 * off + 4]
                       .view(np.float32)[0])
            amax = np.abs(xv[t]).max()
            assert sc == float(np.float32(amax) / np.float32(448.0))
            if amax == 0:
                assert (q == 0).all()
                continue
            mag = e4m3[q & 0x7F]
            dq = np.where(q & 0x80, -mag, mag)
            y = np.abs(xv[t]) / sc
            step = np.where(y >= 2.0 ** -6,
                            2.0 ** (np.floor(np.log2(np.maximum(y, 1e-300)))
                                    - 3), 2.0 ** -9)
            err = np.abs(xv[t] / sc - dq)
            assert (err <= 0.5 * step * (1 + 1e-6) + 1e-7 * y).all(), t
            big = np.argmax(np.abs(xv[t]))
            assert (q[big] & 0x7F) == 0x7E


def check_structure_and_round_trip(o):
    rng = np.random.default_rng(72)
    T, D, B, nb = 30, 128, 16, 6
    x = rng.standard_normal((T, D)).astype(np.float32)
    bits = W.bf16_bits(x.reshape(-1))
    lens = [13, 0, 17]
    perm = rng.permutation(nb)[:6].reshape(3, 2).astype(np.int32)
    slots = np.concatenate([perm[b, np.arange(n) // B] * B + np.arange(n) % B
                            for b, n in enumerate(lens) if n]).astype(np.int64)
    slots = np.concatenate([slots, [-1]])       # one skipped token
    T = slots.size
    a, b = _cache(nb, B, D, 0xAA), _cache(nb, B, D, 0x55)
    _store(o, bits, T, D, a, B, nb, slots)
    _store(o, bits, T, D, b, B, nb, slots)
    changed = (a != 0xAA) | (b != 0x55)
    assert changed.sum() == 30 * (D + 4)
    wl = W.GatherWorkload(name="rt", block_size=B, head_dim=D, num_blocks=nb,
                          cache=a, block_table=perm,
                          cu_seq_lens=np.array([0, 13, 13, 30], np.int32))
    k, s = run_gather(o, wl)
    blocks = a.reshape(nb, -1)
    for i, slot in enumerate(slots[:30]):
        blk, off = divmod(int(slot), B)
        assert np.array_equal(k.reshape(-1, D)[i],
                              blocks[blk, off * D:(off + 1) * D])
        assert np.array_equal(s.reshape(-1, 4)[i],
                              blocks[blk, B * D + 4 * off: B * D + 4 * off + 4])


CHECKS = [check_exact_rows, check_bound_and_scale,
          check_structure_and_round_trip]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_indexer_store_pins(orc, check):
    check(orc)
