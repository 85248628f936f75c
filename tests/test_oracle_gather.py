"""Pins for the oracle's indexer-K gather (CPU only).

* brute-force index tracing: every cache row carries a tag naming its
  (block, offset); each output row must carry the tag of
  (block_table[b, p // B], p % B) for the (b, p) found by a linear scan of
  cu_seq_lens, and rows past the end stay untouched;
* the identity special case: one sequence over an identity block table
  yields the concatenated K regions;
* regression lengths around a block boundary and a sequence spanning 128
  blocks (the first published version of the gather dropped the tail of
  long sequences: vLLM PR #25931 review comment on its launch grid);
* the scale bytes, viewed as float32 as the consumer does (vLLM PR #26456),
  are exactly the cache's scale values.
"""
import numpy as np
import pytest

from paged_quantized_kv_gb300 import workloads as W


def run_gather(o, wl, total=None, sentinel=0xCD):
    total = wl.total_tokens if total is None else total
    k = np.full(max(total, 1) * wl.head_dim, sentinel, dtype=np.uint8)
    s = np.full(max(total, 1) * 4, sentinel, dtype=np.uint8)
    o.gather_indexer_k(wl.cache, wl.block_stride, wl.num_blocks,
                       wl.block_size, wl.head_dim, wl.block_table,
                       wl.cu_seq_lens, total, k, s)
    return k, s


def tagged(wl):
    """Overwrite the first 4 bytes of every K row with int32 tag
    blk*B + off and every scale with float32(tag)."""
    B, D = wl.block_size, wl.head_dim
    c = wl.cache.reshape(wl.num_blocks, wl.block_stride)
    tags = np.arange(wl.num_blocks * B, dtype=np.int32).reshape(-1, B)
    k = c[:, : B * D].reshape(wl.num_blocks, B, D)
    k[:, :, :4] = tags[..., None].view(np.uint8).reshape(wl.num_blocks, B, 4)
    c[:, B * D: B * D + 4 * B] = tags.astype(np.float32).view(
        np.uint8).reshape(wl.num_blocks, 4 * B)
    return wl


def check_trace(o):
    cases = [
        W.make_gather("t0", 5, [5, 37], 64, 128, 4, max_blocks=2),
        W.make_gather("t1", 6, [0, 1, 63, 64, 65, 0, 130], 16, 32, 64),
        W.make_gather("t2", 7, [3, 9, 4], 4, 16, 24, max_blocks=5),
    ]
    for wl in cases:
        tagged(wl)
        B, D = wl.block_size, wl.head_dim
        k, s = run_gather(o, wl, total=wl.total_tokens + 3)
        cu = wl.cu_seq_lens
        kr = k.reshape(-1, D)
        sc = s.view(np.float32)
        for i in range(wl.total_tokens):
            b = 0
            while not (cu[b] <= i < cu[b + 1]):  # linear scan
                b += 1
            p = i - cu[b]
            want = int(wl.block_table[b, p // B]) * B + p % B
            assert kr[i, :4].view(np.int32)[0] == want, (wl.name, i)
            blk, off = divmod(want, B)
            row = wl.cache.reshape(wl.num_blocks, -1)[blk,
                                                      off * D:(off + 1) * D]
            assert np.array_equal(kr[i], row)
            assert sc[i] == np.float32(want)
        tail = wl.total_tokens
        assert (kr[tail:] == 0xCD).all() and (s[4 * tail:] == 0xCD).all()


def check_identity(o):
    wl = W.make_gather("ident", 8, [200], 16, 64, 13)
    wl.block_table = np.arange(13, dtype=np.int32)[None, :]
    k, s = run_gather(o, wl)
    c = wl.cache.reshape(13, wl.block_stride)
    K = c[:, : 16 * 64].reshape(-1)[: 200 * 64]
    S = c[:, 16 * 64:].reshape(-1)[: 200 * 4]
    assert np.array_equal(k, K) and np.array_equal(s, S)


def check_long_sequence(o):
    wl = W.make_gather("long", 9, [8192, 1, 64], 64, 128, 400)
    tagged(wl)
    k, s = run_gather(o, wl)
    kr = k.reshape(-1, 128)[:, :4].copy().view(np.int32)[:, 0]
    p = np.arange(8192)
    want = wl.block_table[0, p // 64].astype(np.int64) * 64 + p % 64
    assert np.array_equal(kr[:8192], want)
    assert np.array_equal(s.view(np.float32)[:8192], want.astype(np.float32))


def check_scale_view(o):
    wl = W.gather_workload(0)
    k, s = run_gather(o, wl)
    v = s.view(np.float32)
    assert v.size == 42 and (v >= 1e-3).all() and (v <= 1.0).all()
    # every gathered scale is one of the cache's scale values of that block
    c = wl.cache.reshape(wl.num_blocks, wl.block_stride)
    allsc = c[:, 64 * 128:].copy().view(np.float32)
    assert np.isin(v, allsc).all()


CHECKS = [check_trace, check_identity, check_long_sequence, check_scale_view]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_gather_pins(orc, check):
    check(orc)
