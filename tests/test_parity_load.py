"""GPU parity of kvq_load_nvfp4 (the read side of the NVFP4 store) against
the CPU oracle: pages written by the GPU store (themselves checked against
the oracle's) are read back through a block table, and every output bf16
bit pattern must equal the oracle's load of the same pages.

Covers the long-context workload read back in full, HND / NHD, swizzled K
scales, fp16-stored pages, ragged sequences (0, 1, B-1, B, B+1 tokens),
pages never written (sentinel bytes), out-of-range flags, and PDL chains in
which the load reads pages the immediately preceding store wrote."""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import assert_bytes_equal, store_inputs, to_dev
from tests.test_oracle_load import _seq_store
from tests.test_oracle_store import run_store

pytestmark = pytest.mark.gpu
SENTINEL = 0x7FC1  # a NaN bit pattern no load writes


def _oracle_load(orc, wl, cache, bt, cu, total=None):
    total = int(cu[-1]) if total is None else total
    return orc.load_nvfp4(cache, 0, wl.value_side_offset, wl.page_stride,
                          wl.block_size, wl.num_blocks, wl.layout,
                          wl.num_heads, wl.head_size, bt, cu, total,
                          wl.k_scale, wl.v_scale, wl.flags & 1)


def _gpu_store_load(wl, bt, cu, total=None, store_flags=0, load_flags=0):
    key, value, slots, ks, vs = store_inputs(wl)
    kv, kc, vc = kvq.alloc_nvfp4_cache(wl.num_blocks, wl.block_size,
                                       wl.num_heads, wl.head_size,
                                       wl.layout, fill=0xAA)
    total = int(cu[-1]) if total is None else total
    shape = (max(total, 1), wl.num_heads, wl.head_size)
    ko = torch.full(shape, SENTINEL, dtype=torch.int16,
                    device="cuda").view(torch.bfloat16)[:total]
    vo = torch.full(shape, SENTINEL, dtype=torch.int16,
                    device="cuda").view(torch.bfloat16)[:total]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs,
                        flags=wl.flags | store_flags)
    kvq.kvq_load_nvfp4(kc, vc, to_dev(bt), to_dev(cu), ks, vs, ko, vo,
                       flags=(wl.flags & 1) | load_flags, dev_error=err)
    torch.cuda.synchronize()
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    return kv.cpu().numpy().reshape(-1), bits(ko), bits(vo), int(err.item())


def _compare(orc, wl, bt, cu, **kw):
    cache_g, kg, vg, err = _gpu_store_load(wl, bt, cu, **kw)
    cache_o = run_store(orc, wl)
    assert_bytes_equal(cache_g, cache_o, wl.name + " pages")
    ko, vo = _oracle_load(orc, wl, cache_o, bt, cu)
    assert_bytes_equal(kg.reshape(-1).view(np.uint8),
                       ko.reshape(-1).view(np.uint8), wl.name + " key")
    assert_bytes_equal(vg.reshape(-1).view(np.uint8),
                       vo.reshape(-1).view(np.uint8), wl.name + " value")
    return err


def test_long_context_read_back(orc):
    st = W.store_workload(4)
    bt, cu = W.sequences_of_store(st, 512)
    assert _compare(orc, st, bt, cu) == 0


def test_tiny_whole_cache_including_unwritten_pages(orc):
    st = W.store_workload(0)  # 24 random slots of 128, 3 skipped
    bt = np.arange(8, dtype=np.int32).reshape(2, 4)
    cu = np.array([0, 64, 128], dtype=np.int32)
    assert _compare(orc, st, bt, cu) == 0


CASES = [
    dict(name="hnd_ragged", seed=60, num_heads=2, head_size=64,
         block_size=8, num_blocks=24, lens=[0, 1, 7, 8, 9, 30]),
    dict(name="nhd", seed=61, num_heads=3, head_size=128, block_size=4,
         num_blocks=40, lens=[5, 11, 3], layout=W.LAYOUT_NHD,
         scales=(0.02, 0.7)),
    dict(name="swzk_fp16", seed=62, num_heads=1, head_size=256,
         block_size=16, num_blocks=8, lens=[40, 17], flags=1,
         dtype=W.DTYPE_F16, scales=(0.1, 0.05)),
    dict(name="wide_heads", seed=63, num_heads=16, head_size=256,
         block_size=32, num_blocks=12, lens=[100, 64, 1]),
    dict(name="block_size_12", seed=64, num_heads=2, head_size=128,
         block_size=12, num_blocks=20, lens=[25, 12, 13, 0, 11]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_case(orc, case):
    c = dict(case)
    rng = np.random.default_rng(c["seed"])
    lens = c.pop("lens")
    wl = W.make_store(c.pop("name"), c.pop("seed"), int(sum(lens)),
                      slots="dense", **c)
    bt, cu, slots = _seq_store(orc, wl, lens, wl.block_size, rng)
    wl.slot_mapping = slots
    assert _compare(orc, wl, bt, cu) == 0


def test_flags_for_bad_block_and_short_cu(orc):
    wl = W.make_store("flags", 65, 40, 2, 64, 8, 10, slots="dense")
    bt = np.arange(10, dtype=np.int32).reshape(2, 5)
    cu = np.array([0, 20, 40], dtype=np.int32)
    bad = bt.copy()
    bad[1, 2] = 99                      # rows 20 + 16 .. 20 + 23
    cache_g, kg, vg, err = _gpu_store_load(wl, bad, cu, total=44)
    assert err == kvq.KVQ_DEVERR_BLOCK | kvq.KVQ_DEVERR_SEQ
    cache_o = run_store(orc, wl)
    ko, vo = _oracle_load(orc, wl, cache_o, bt, cu)
    rows = np.arange(44)
    bad_rows = (rows >= 36) & (rows < 40) | (rows >= 40)
    assert (kg[bad_rows] == SENTINEL).all() and (vg[bad_rows] == SENTINEL).all()
    good = ~bad_rows
    assert np.array_equal(kg[good], ko[good[:40]])
    assert np.array_equal(vg[good], vo[good[:40]])


@pytest.mark.parametrize("load_flags", [kvq.KVQ_F_PDL,
                                        kvq.KVQ_F_PDL_EARLY_META])
def test_pdl_load_reads_pages_just_stored(orc, load_flags):
    st = W.make_store("pdl", 66, 8192, 4, 256, 32, 256, slots="runs",
                      request_len=512)
    bt, cu = W.sequences_of_store(st, 512)
    for _ in range(2):
        assert _compare(orc, st, bt, cu, store_flags=kvq.KVQ_F_PDL,
                        load_flags=load_flags) == 0
