"""Pins for the oracle's NVFP4 paged load (CPU only).

The pages state no dequantisation rule; the load takes the plain inverse of
the store's: x' = bf16_rn(e2m1(q) * (float(sf) * k_scale)).  Pinned by
* the fp32 -> bf16 rounding against torch's own cast (independent library)
  on every kind of boundary value;
* exact round trips: groups whose values are e2m1 codes times a power of
  two come back bit-for-bit after store -> load;
* the dequantisation error bound after store -> load on random sequences
  (HND, NHD, swizzled K, fp16 inputs): |x - x'| <= half an e2m1 step *
  float(sf) * k_scale plus the bf16 rounding of x' -- which also pins the
  page addressing and the unswizzle, because the store's layout is pinned
  independently;
* rows of sequences come out in cu_seq_lens order through the block table
  (sequences of 0, 1, B-1, B, B+1 tokens).
"""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import workloads as W
from tests.test_oracle_store import run_store

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def check_bf16_rounding(o):
    rng = np.random.default_rng(31)
    base = rng.standard_normal(3000).astype(np.float32) * 10
    bits = base.view(np.uint32) & 0xFFFF0000
    mids = (bits | 0x8000).view(np.float32)           # exact ties
    near = np.concatenate([(bits | 0x7FFF), (bits | 0x8001)]).view(
        np.float32)
    special = np.float32([0.0, -0.0, 1e-40, -1e-42, 3.4e38, -3.4e38,
                          np.inf, -np.inf, 1.00390625, 1.01171875])
    pts = np.concatenate([base, mids, near, special])
    ref = torch.from_numpy(pts).to(torch.bfloat16).view(torch.int16).numpy()
    ref = ref.view(np.uint16)
    got = np.array([o.float_to_bf16(v) for v in pts], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(pts[i]), hex(got[i]), hex(ref[i]))
                           for i in bad[:6]]


def _seq_store(o, wl, lens, B, rng):
    """Place sequences of the given lengths on random distinct blocks of
    the workload's cache and return (block_table, cu, slot_mapping)."""
    lens = np.asarray(lens, dtype=np.int64)
    need = (lens + B - 1) // B
    mb = max(int(need.max()) if lens.size else 1, 1)
    perm = rng.permutation(wl.num_blocks)[: lens.size * mb]
    bt = perm.reshape(lens.size, mb).astype(np.int32)
    cu = np.zeros(lens.size + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    slots = np.concatenate([bt[b, np.arange(n) // B] * B + np.arange(n) % B
                            for b, n in enumerate(lens)] or
                           [np.zeros(0, np.int64)]).astype(np.int64)
    return bt, cu, slots


def _load(o, wl, cache, bt, cu):
    return o.load_nvfp4(cache, 0, wl.value_side_offset, wl.page_stride,
                        wl.block_size, wl.num_blocks, wl.layout,
                        wl.num_heads, wl.head_size, bt, cu, int(cu[-1]),
                        wl.k_scale, wl.v_scale, wl.flags)


def check_exact_round_trip(o):
    rng = np.random.default_rng(32)
    T, H, D, B = 24, 2, 64, 8
    for scale in (1.0, 0.25, 8.0):
        codes = rng.integers(0, 16, size=(T, 2, H, D // 16, 16))
        vals = E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0)
        vals[..., 0] = 6.0                          # amax 6 * 2^e per group
        e = rng.integers(-6, 6, size=(T, 2, H, D // 16, 1))
        x = (vals * 2.0 ** e * scale).astype(np.float32)
        src = W.bf16_bits(x.reshape(-1))
        assert (W.bf16_values(src) == x.reshape(-1)).all()
        wl = W.StoreWorkload(
            name="exact", num_tokens=T, num_heads=H, head_size=D,
            block_size=B, num_blocks=4, src=src, key_offset=0,
            key_stride0=2 * H * D, value_offset=H * D,
            value_stride0=2 * H * D,
            slot_mapping=np.arange(T, dtype=np.int64),
            k_scale=np.float32(scale), v_scale=np.float32(scale))
        cache = run_store(o, wl)
        bt = np.arange(3, dtype=np.int32)[None, :]
        cu = np.array([0, T], dtype=np.int32)
        k, v = _load(o, wl, cache, bt, cu)
        assert np.array_equal(k, wl.key_array())
        assert np.array_equal(v, wl.value_array())


CASES = [
    dict(name="hnd", seed=33, num_heads=2, head_size=64, block_size=8,
         num_blocks=24, lens=[0, 1, 7, 8, 9, 30]),
    dict(name="nhd", seed=34, num_heads=3, head_size=128, block_size=4,
         num_blocks=40, lens=[5, 11, 3], layout=W.LAYOUT_NHD,
         scales=(0.02, 0.7)),
    dict(name="swzk_fp16", seed=35, num_heads=1, head_size=256,
         block_size=16, num_blocks=8, lens=[40, 17], flags=1,
         dtype=W.DTYPE_F16, scales=(0.1, 0.05)),
]


def check_round_trip_bound(o):
    for case in CASES:
        c = dict(case)
        rng = np.random.default_rng(c["seed"])
        lens = c.pop("lens")
        T = int(sum(lens))
        wl = W.make_store(c.pop("name"), c.pop("seed"), T, slots="dense",
                          **c)
        bt, cu, slots = _seq_store(o, wl, lens, wl.block_size, rng)
        wl.slot_mapping = slots
        cache = run_store(o, wl)
        k, v = _load(o, wl, cache, bt, cu)
        for src, out, sc in ((wl.key_array(), k, wl.k_scale),
                             (wl.value_array(), v, wl.v_scale)):
            g = float(np.float32(1.0) / np.float32(sc))
            bits = np.asarray(src)
            xd_all = W.bf16_values(out).astype(np.float64)
            for t in range(T):
                for h in range(wl.num_heads):
                    for j in range(wl.head_size // 16):
                        gb = bits[t, h, 16 * j:16 * j + 16]
                        x = W.element_values(gb, wl.dtype).astype(np.float64)
                        xd = xd_all[t, h, 16 * j:16 * j + 16]
                        _, sf = o.quantize_group(gb, g, wl.dtype)
                        s_ = o.e4m3_decode(sf)
                        if sf == 0:
                            assert (xd == 0).all()
                            continue
                        if np.abs(x).max() * g / 6.0 > 448.0:
                            continue  # saturated scale: no half-step bound
                        y = np.abs(x) * g / s_
                        step = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
                        bound = (0.5 * step * s_ / g * (1 + 1e-5)
                                 + np.abs(xd) * 2.0 ** -8 + 1e-30)
                        assert (np.abs(x - xd) <= bound).all(), (
                            case["name"], t, h, j)


def check_rows_in_sequence_order(o):
    """The load of sequence b, position p equals the load of a one-token
    sequence made of that token alone (block table row of one block)."""
    rng = np.random.default_rng(36)
    wl = W.make_store("order", 36, 20, 2, 64, 4, 16, slots="dense")
    lens = [3, 0, 9, 8]
    bt, cu, slots = _seq_store(o, wl, lens, 4, rng)
    wl.slot_mapping = slots
    cache = run_store(o, wl)
    k, v = _load(o, wl, cache, bt, cu)
    for b, n in enumerate(lens):
        for p in range(n):
            blk = int(bt[b, p // 4])
            one_bt = np.array([[blk]], dtype=np.int32)
            # a 1-token "sequence" starting at offset p % 4 of that block:
            # load the block's first p%4+1 tokens and take the last row
            k1, v1 = _load(o, wl, cache, one_bt,
                           np.array([0, p % 4 + 1], dtype=np.int32))
            row = cu[b] + p
            assert np.array_equal(k[row], k1[-1])
            assert np.array_equal(v[row], v1[-1])


CHECKS = [check_bf16_rounding, check_exact_round_trip,
          check_round_trip_bound, check_rows_in_sequence_order]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_load_pins(orc, check):
    check(orc)
