"""Pins for the oracle's NVFP4 group quantiser and paged store (CPU only).

* hand-worked groups (tests/golden/nvfp4_groups.txt);
* the dequantisation error bound: with s = float(sf), y = x*g/s in exact
  arithmetic, |y - e2m1(q)| <= half the e2m1 step at y (0.5 below 2, 1 below
  4, 2 above) -- i.e. |x - e2m1(q)*s/g| <= half a step * s/g -- whenever sf
  is a normal e4m3 value and (amax/6)*g does not saturate;
* the scale is the e4m3 value nearest to amax*g/6 (up to fp32 slack);
* the page layout: an independent numpy re-assembly of the cache from the
  per-group results, through reshaped views of the page (the dispatch's
  [H, B, D/2] / [B, H, D/2] data and [H, B, S] / [B, H, S] scale regions)
  and the page's reshape/permute statement of the scale swizzle;
* structure: exactly the stored tokens' bytes change, nothing else.
"""
import numpy as np
import pytest

from paged_quantized_kv_gb300 import workloads as W
from tests.golden_io import as_bits, nvfp4_groups

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_value(nib):
    v = E2M1[nib & 7]
    return -v if nib & 8 else v


def unpack(data8):
    q = []
    for b in data8:
        q.append(int(b) & 0xF)
        q.append(int(b) >> 4)
    return q


def check_golden_groups(o):
    for name, g, xs, sf, data, dtype in nvfp4_groups():
        got_data, got_sf = o.quantize_group(as_bits(xs, dtype), g, dtype)
        assert got_sf == sf, (name, hex(got_sf), hex(sf))
        assert bytes(got_data) == data, (name, bytes(got_data).hex(),
                                         data.hex())


def _groups(rng, n, dtype=W.DTYPE_BF16):
    """Random bf16 (or fp16) groups from several value distributions."""
    kinds = [
        lambda: rng.standard_normal(16),
        lambda: rng.standard_normal(16) * np.where(rng.random(16) < .1, 50, 1),
        lambda: rng.uniform(-1e-3, 1e-3, 16),
        lambda: rng.standard_normal(16) * 1e3,
        lambda: np.round(rng.uniform(-12, 12, 16) * 4) / 4,
    ]
    for i in range(n):
        x = kinds[i % len(kinds)]().astype(np.float32)
        if dtype == W.DTYPE_F16:
            x = np.clip(x, -60000, 60000)
        yield W.element_bits(x, dtype)


def check_error_bound(o):
    rng = np.random.default_rng(21)
    e4m3_min_normal = 2.0 ** -6
    checked = 0
    vals = np.array([o.e4m3_decode(c) for c in range(127)])
    cases = [(g, W.DTYPE_BF16) for g in (1.0, 0.37, 13.0, 580.0, 2.0 ** -5)]
    cases += [(g, W.DTYPE_F16) for g in (1.0, 41.0)]
    for g, dtype in cases:
        g32 = float(np.float32(g))
        for bits in _groups(rng, 300, dtype):
            x = W.element_values(bits, dtype).astype(np.float64)
            data, sf = o.quantize_group(bits, g32, dtype)
            s = o.e4m3_decode(sf)
            amax = np.abs(x).max()
            target = amax * g32 / 6.0  # exact-arithmetic scale
            # sf is the e4m3 value nearest the target (or 448 above it)
            if target >= 448.0:
                assert sf == 0x7E
            else:
                best = np.abs(vals - target).min()
                assert abs(s - target) <= best + 1e-6 * target + 1e-30
            if sf == 0:
                assert bytes(data) == bytes(8)
                continue
            if not (s >= e4m3_min_normal and target <= 448.0):
                continue
            q = unpack(data)
            for xi, qi in zip(x, q):
                y = xi * g32 / s
                ay = abs(y)
                step = 0.5 if ay < 2 else (1.0 if ay < 4 else 2.0)
                err = abs(y - e2m1_value(qi))
                assert err <= 0.5 * step + 1e-5 * max(ay, 1.0), (
                    xi, g32, s, qi, y)
                if xi != 0 and e2m1_value(qi) != 0:
                    assert np.sign(e2m1_value(qi)) == np.sign(xi)
                checked += 1
    assert checked > 10000


# --- page layout ----------------------------------------------------------------

def _side_views(cache, wl, side):
    H, B, D = wl.num_heads, wl.block_size, wl.head_size
    S = D // 16
    pages = cache.reshape(wl.num_blocks, wl.page_stride)
    base = 0 if side == 0 else wl.value_side_offset
    side_bytes = pages[:, base: base + wl.side_bytes]
    nd = H * B * D // 2
    if wl.layout == W.LAYOUT_HND:
        data = side_bytes[:, :nd].reshape(wl.num_blocks, H, B, D // 2)
        scale = side_bytes[:, nd:].reshape(wl.num_blocks, H, B, S)
        return (lambda blk, h, off: data[blk, h, off],
                lambda blk, h: scale[blk, h])
    data = side_bytes[:, :nd].reshape(wl.num_blocks, B, H, D // 2)
    scale = side_bytes[:, nd:].reshape(wl.num_blocks, B, H, S)
    return (lambda blk, h, off: data[blk, off, h],
            lambda blk, h: scale[blk, :, h])


def _swizzled_set(tile, t, s, value):
    """Write logical (t, s) of a physically swizzled [B, S] tile, using the
    page's statement: physical = logical viewed [B/4, 4, 4, S/4],
    permuted (0, 2, 3, 1), read back as [B, S]."""
    B, S = tile.shape
    logical = (tile.copy().reshape(B // 4, 4, S // 4, 4)
               .transpose(0, 3, 1, 2).reshape(B, S))
    logical[t, s] = value
    tile[...] = (logical.reshape(B // 4, 4, 4, S // 4)
                 .transpose(0, 2, 3, 1).reshape(B, S))


def expected_cache(o, wl, sentinel=0xAA):
    """Independent re-assembly of the store's output from per-group
    results."""
    cache = np.full(wl.cache_bytes, sentinel, dtype=np.uint8)
    keys, vals = wl.key_array(), wl.value_array()
    g = (1.0 / np.float32(wl.k_scale), 1.0 / np.float32(wl.v_scale))
    g = tuple(float(np.float32(v)) for v in g)
    for t in range(wl.num_tokens):
        slot = int(wl.slot_mapping[t])
        if slot < 0:
            continue
        blk, off = divmod(slot, wl.block_size)
        for side, src in ((0, keys), (1, vals)):
            data_row, scale_tile = _side_views(cache, wl, side)
            swz = side == 1 or (wl.flags & 1)
            for h in range(wl.num_heads):
                for j in range(wl.head_size // 16):
                    d8, sf = o.quantize_group(src[t, h, 16 * j:16 * j + 16],
                                              g[side], wl.dtype)
                    data_row(blk, h, off)[8 * j: 8 * j + 8] = d8
                    tile = scale_tile(blk, h)
                    if swz:
                        _swizzled_set(tile, off, j, sf)
                    else:
                        tile[off, j] = sf
    return cache


def run_store(o, wl, sentinel=0xAA):
    cache = np.full(wl.cache_bytes, sentinel, dtype=np.uint8)
    o.store_nvfp4(wl.src, wl.key_stride0, wl.src, wl.value_stride0,
                  wl.num_tokens, wl.num_heads, wl.head_size, cache, 0,
                  wl.value_side_offset, wl.page_stride, wl.block_size,
                  wl.num_blocks, wl.layout, wl.slot_mapping, wl.k_scale,
                  wl.v_scale, wl.flags, key_base=wl.key_offset,
                  value_base=wl.value_offset, dtype=wl.dtype)
    return cache


SMALL_CASES = [
    dict(name="hnd", seed=1, num_tokens=19, num_heads=2, head_size=64,
         block_size=8, num_blocks=6, skip=4, scales=(0.7, 0.05)),
    dict(name="nhd", seed=2, num_tokens=13, num_heads=3, head_size=128,
         block_size=4, num_blocks=5, skip=2, layout=W.LAYOUT_NHD,
         scales=(0.01, 1.5)),
    dict(name="swzk", seed=3, num_tokens=16, num_heads=1, head_size=64,
         block_size=16, num_blocks=2, slots="dense", flags=1),
    dict(name="nhd_swzk_stride", seed=4, num_tokens=9, num_heads=2,
         head_size=64, block_size=8, num_blocks=3, row_mult=2,
         layout=W.LAYOUT_NHD, flags=1),
    dict(name="fp16_hnd", seed=5, num_tokens=11, num_heads=2, head_size=128,
         block_size=8, num_blocks=4, skip=1, dtype=W.DTYPE_F16,
         scales=(0.02, 3.0)),
]


def _small(case):
    c = dict(case)
    return W.make_store(c.pop("name"), c.pop("seed"), **c)


def check_store_layout(o):
    for case in SMALL_CASES + [None]:
        wl = W.store_workload(0) if case is None else _small(case)
        got = run_store(o, wl)
        want = expected_cache(o, wl)
        assert np.array_equal(got, want), case


def check_store_structure(o):
    wl = W.store_workload(0)
    a = run_store(o, wl, 0xAA)
    b = run_store(o, wl, 0x55)
    changed = (a != 0xAA) | (b != 0x55)
    H, D = wl.num_heads, wl.head_size
    assert changed.sum() == wl.stored_tokens * 2 * H * (D // 2 + D // 16)
    assert wl.stored_tokens == 21
    assert np.array_equal(a[changed], b[changed])
    # a skipped token writes nothing: drop every slot and nothing changes
    wl.slot_mapping = np.full_like(wl.slot_mapping, -1)
    assert (run_store(o, wl, 0xAA) == 0xAA).all()


CHECKS = [check_golden_groups, check_error_bound, check_store_layout,
          check_store_structure]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_store_pins(orc, check):
    check(orc)
