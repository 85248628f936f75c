"""Pins for the oracle's paged decode attention over the NVFP4 cache (CPU).

vLLM PR #12348 "[ROCm] Faster Custom Paged Attention kernels" shows the
paged_attention op's signature only; the computation taken is plain softmax
attention of one query token per sequence over its cached context, on the
exactly dequantised cache (K^ = e2m1 * sf * k_scale), query head h reading
KV head h / (Hq / Hkv).  Pinned, independently of the oracle's own loops, by
* torch's scaled_dot_product_attention in float64 (an independent library
  routine) on the K/V rows the load oracle dequantises -- exact in bf16
  when k_scale and v_scale are powers of two -- with the KV heads repeated
  per query group (HND, NHD, swizzled K scales, fp16 queries, negative
  and zero softmax scales);
* closed forms: a zero query, or a zero softmax scale, averages the value
  rows; a one-token context returns that token's value row; an empty
  context returns zeros;
* invariances: k_scale * c with scale / c (c a power of two) changes
  nothing, v_scale * 2 doubles the output, moving pages to other blocks
  changes nothing;
* the one-hot limit: logits thousands apart return the value row of the
  largest logit (and overflow exp() if the max is not subtracted);
* the error-scale output: mag >= |out|, and mag == out for non-negative
  values.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_quantized_kv_gb300 import workloads as W

LAYOUTS = (W.LAYOUT_HND, W.LAYOUT_NHD)


def _wl(seed, lens, Hq=8, Hkv=2, D=64, B=16, **kw):
    kw.setdefault("k_scale", 0.25)
    kw.setdefault("v_scale", 0.5)
    return W.make_attention(f"pin{seed}", seed, lens, num_q_heads=Hq,
                            num_kv_heads=Hkv, head_size=D, block_size=B,
                            extra_blocks=3, **kw)


def _nhd(wl):
    """The same tokens re-laid out NHD: rebuild each page's bytes from the
    HND ones by the layout's definition (data [H][B][D/2] -> [B][H][D/2],
    scales likewise)."""
    H, B, D = wl.num_kv_heads, wl.block_size, wl.head_size
    data, S = D // 2, D // 16
    pages = wl.cache.reshape(wl.num_blocks, wl.page_stride).copy()
    out = np.zeros_like(pages)
    for s in range(2):
        base = s * wl.side_bytes
        d = pages[:, base:base + H * B * data].reshape(-1, H, B, data)
        out[:, base:base + H * B * data] = d.transpose(0, 2, 1, 3).reshape(
            wl.num_blocks, -1)
        sb = base + H * B * data
        sc = pages[:, sb:sb + H * B * S].reshape(-1, H, B, S)
        out[:, sb:sb + H * B * S] = sc.transpose(0, 2, 1, 3).reshape(
            wl.num_blocks, -1)
    wl.cache = out.reshape(-1)
    wl.layout = W.LAYOUT_NHD
    return wl


def _attend(o, wl):
    return o.paged_attention_nvfp4(
        wl.query, wl.cache, 0, wl.side_bytes, wl.page_stride, wl.block_size,
        wl.num_blocks, wl.layout, wl.num_kv_heads, wl.block_table,
        wl.context_lens, wl.k_scale, wl.v_scale, wl.scale, wl.flags,
        wl.dtype)


def _dequant(o, wl):
    """K^ and V^ per sequence (float64 [L, Hkv, D]) from the load oracle."""
    lens = wl.context_lens.astype(np.int64)
    cu = np.zeros(lens.size + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    k, v = o.load_nvfp4(wl.cache, 0, wl.side_bytes, wl.page_stride,
                        wl.block_size, wl.num_blocks, wl.layout,
                        wl.num_kv_heads, wl.head_size, wl.block_table, cu,
                        int(cu[-1]), wl.k_scale, wl.v_scale, wl.flags)
    k = W.bf16_values(k).astype(np.float64)
    v = W.bf16_values(v).astype(np.float64)
    return [(k[cu[b]:cu[b + 1]], v[cu[b]:cu[b + 1]])
            for b in range(lens.size)]


def _query(wl):
    return W.element_values(wl.query, wl.dtype).astype(np.float64)


def check_sdpa_agreement(o):
    cases = [
        dict(seed=1, lens=[1, 17, 40, 16]),
        dict(seed=2, lens=[33, 5], Hq=4, Hkv=4, D=128, B=8),
        dict(seed=3, lens=[50, 64], Hq=16, Hkv=2, D=64, B=32,
             flags=oracle.F_SWIZZLE_K_SCALE),
        dict(seed=4, lens=[21, 9], dtype=W.DTYPE_F16),
        dict(seed=5, lens=[30, 12], scale=-0.2),    # negative softmax scale
        dict(seed=6, lens=[25, 3], scale=0.0),      # zero: uniform weights
    ]
    for case in cases:
        for layout in LAYOUTS:
            wl = _wl(**case)
            if layout == W.LAYOUT_NHD:
                wl = _nhd(wl)
            out, _ = _attend(o, wl)
            rows = _dequant(o, wl)
            q = _query(wl)
            G = wl.num_q_heads // wl.num_kv_heads
            for b, (k, v) in enumerate(rows):
                kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(
                    G, dim=0)[None]
                vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(
                    G, dim=0)[None]
                qt = torch.from_numpy(q[b])[None, :, None, :]
                ref = torch.nn.functional.scaled_dot_product_attention(
                    qt, kt, vt, scale=float(wl.scale))[0, :, 0, :].numpy()
                err = np.abs(out[b] - ref).max()
                assert err <= 1e-12 * (1 + np.abs(ref).max()), (case, b, err)


def check_zero_query_is_mean(o):
    wl = _wl(11, [7, 30, 3])
    wl.query[:] = 0
    out, _ = _attend(o, wl)
    G = wl.num_q_heads // wl.num_kv_heads
    for b, (k, v) in enumerate(_dequant(o, wl)):
        mean = v.mean(axis=0)                       # [Hkv, D]
        assert np.allclose(out[b], np.repeat(mean, G, axis=0), rtol=0,
                           atol=1e-13 * (1 + np.abs(mean).max()))


def check_zero_scale_is_mean(o):
    wl = _wl(17, [9, 40, 2], scale=0.0)
    out, _ = _attend(o, wl)
    G = wl.num_q_heads // wl.num_kv_heads
    for b, (k, v) in enumerate(_dequant(o, wl)):
        mean = v.mean(axis=0)                       # [Hkv, D]
        assert np.allclose(out[b], np.repeat(mean, G, axis=0), rtol=0,
                           atol=1e-13 * (1 + np.abs(mean).max()))


def check_single_token_and_empty(o):
    wl = _wl(12, [1, 0, 1])
    out, mag = _attend(o, wl)
    G = wl.num_q_heads // wl.num_kv_heads
    rows = _dequant(o, wl)
    for b in (0, 2):
        v = rows[b][1][0]                           # [Hkv, D]
        assert np.array_equal(out[b], np.repeat(v, G, axis=0))
        assert np.array_equal(mag[b], np.abs(np.repeat(v, G, axis=0)))
    assert not out[1].any() and not mag[1].any()


def check_scale_invariances(o):
    lens = [25, 12]
    base, _ = _attend(o, _wl(13, lens, k_scale=0.25, scale=0.125))
    traded, _ = _attend(o, _wl(13, lens, k_scale=1.0, scale=0.125 / 4))
    assert np.array_equal(base, traded)
    doubled, _ = _attend(o, _wl(13, lens, v_scale=1.0, scale=0.125))
    assert np.array_equal(doubled, 2 * base)


def check_page_relocation(o):
    wl = _wl(14, [40, 19, 33])
    out, _ = _attend(o, wl)
    rng = np.random.default_rng(5)
    perm = rng.permutation(wl.num_blocks)          # block i moves to perm[i]
    pages = wl.cache.reshape(wl.num_blocks, wl.page_stride)
    moved = np.zeros_like(pages)
    moved[perm] = pages
    wl.cache = moved.reshape(-1)
    wl.block_table = perm[wl.block_table].astype(np.int32)
    out2, _ = _attend(o, wl)
    assert np.array_equal(out, out2)


def check_one_hot_limit(o):
    wl = _wl(15, [37, 64], query_mult=1.0, scale=5000.0)
    out, _ = _attend(o, wl)
    assert np.isfinite(out).all()
    q = _query(wl)
    G = wl.num_q_heads // wl.num_kv_heads
    checked = 0
    for b, (k, v) in enumerate(_dequant(o, wl)):
        for h in range(wl.num_q_heads):
            logits = k[:, h // G, :] @ q[b, h]
            order = np.sort(logits)
            if order.size > 1 and (order[-1] - order[-2]) * 5000.0 < 50:
                continue                            # not one-hot: skip head
            t = int(np.argmax(logits))
            assert np.allclose(out[b, h], v[t, h // G], rtol=1e-15,
                               atol=1e-15), (b, h)
            checked += 1
    assert checked >= wl.num_q_heads


def check_mag(o):
    wl = _wl(16, [45, 8])
    out, mag = _attend(o, wl)
    assert (mag >= np.abs(out) - 1e-15).all()
    assert (mag > np.abs(out) + 1e-9).any()         # signed values cancel
    # non-negative values: clear every sign bit of the V data
    H, B, D = wl.num_kv_heads, wl.block_size, wl.head_size
    pages = wl.cache.reshape(wl.num_blocks, wl.page_stride)
    vdata = slice(wl.side_bytes, wl.side_bytes + H * B * D // 2)
    pages[:, vdata] &= 0x77
    out, mag = _attend(o, wl)
    assert np.allclose(mag, out, rtol=1e-15, atol=0)


CHECKS = [check_sdpa_agreement, check_zero_query_is_mean,
          check_zero_scale_is_mean,
          check_single_token_and_empty, check_scale_invariances,
          check_page_relocation, check_one_hot_limit, check_mag]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_attention_pins(orc, check):
    check(orc)
