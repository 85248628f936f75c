"""Calls launched with KVQ_F_PDL (programmatic dependent launch) give the
same bytes as the oracle, including when they run back to back with the
other call and with themselves on one stream: each kernel waits for the
previous kernel's completion before it touches memory, so a chain of
stores into the same pages ends with the last store's bytes."""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import assert_bytes_equal, store_inputs, to_dev
from tests.test_oracle_gather import run_gather
from tests.test_oracle_store import run_store

pytestmark = pytest.mark.gpu
PDL = kvq.KVQ_F_PDL


def _gather_args(g):
    cache = to_dev(g.cache).view(g.num_blocks, g.block_stride)
    n = g.total_tokens
    k = torch.full((n, g.head_dim), 0xCD, dtype=torch.uint8, device="cuda")
    s = torch.full((n, 4), 0xCD, dtype=torch.uint8, device="cuda")
    return cache, k, s, to_dev(g.block_table), to_dev(g.cu_seq_lens)


@pytest.mark.parametrize("index", [0, 4])
def test_store_then_gather_pdl(orc, index):
    st = W.store_workload(index)
    ga = W.gather_workload(index)
    key, value, slots, ks, vs = store_inputs(st)
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size,
                                       st.num_heads, st.head_size, fill=0xAA)
    cache, k, s, bt, cu = _gather_args(ga)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):  # back to back, each depending on nothing but order
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs, flags=PDL,
                            dev_error=err)
        kvq.kvq_gather_indexer_k(cache, k, s, bt, cu,
                                 block_size=ga.block_size, flags=PDL,
                                 dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bytes_equal(kv.cpu().numpy().reshape(-1), run_store(orc, st),
                       st.name)
    wk, ws = run_gather(orc, ga)
    assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, ga.name + " k")
    assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, ga.name + " s")


def test_chain_of_dependent_stores(orc):
    """Alternate two inputs into the same slots 9 times with PDL; the pages
    must hold exactly the last store's result."""
    a = W.make_store("a", 40, 4096, 4, 256, 32, 128, slots="runs",
                     request_len=512)
    b = W.make_store("b", 41, 4096, 4, 256, 32, 128, slots="runs",
                     request_len=512)
    b.slot_mapping = a.slot_mapping.copy()
    ins = [store_inputs(a), store_inputs(b)]
    kv, kc, vc = kvq.alloc_nvfp4_cache(a.num_blocks, a.block_size,
                                       a.num_heads, a.head_size, fill=0xAA)
    for i in range(9):
        key, value, slots, ks, vs = ins[i % 2]
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs, flags=PDL)
    torch.cuda.synchronize()
    assert_bytes_equal(kv.cpu().numpy().reshape(-1), run_store(orc, a), "a")


def test_pdl_after_foreign_kernel(orc):
    """A PDL launch right after an ordinary torch kernel that writes the
    store's input sees the finished input."""
    st = W.store_workload(0)
    key, value, slots, ks, vs = store_inputs(st)
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size,
                                       st.num_heads, st.head_size, fill=0xAA)
    k2 = torch.zeros_like(key)
    k2.copy_(key)  # torch kernel writing the input just before the launch
    kvq.kvq_store_nvfp4(k2, value, kc, vc, slots, ks, vs, flags=PDL)
    torch.cuda.synchronize()
    assert_bytes_equal(kv.cpu().numpy().reshape(-1), run_store(orc, st),
                       st.name)


EARLY = kvq.KVQ_F_PDL_EARLY_META


@pytest.mark.parametrize("index", [0, 3, 4])
def test_gather_early_meta(orc, index):
    ga = W.gather_workload(index)
    cache, k, s, bt, cu = _gather_args(ga)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        kvq.kvq_gather_indexer_k(cache, k, s, bt, cu,
                                 block_size=ga.block_size, flags=EARLY,
                                 dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, ws = run_gather(orc, ga)
    assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, ga.name + " k")
    assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, ga.name + " s")


def test_early_meta_gather_reads_bytes_the_store_just_wrote(orc):
    """The gather's cache is the very buffer the preceding PDL store
    writes: the early-metadata gather may start while the store runs, but
    must read the cache only after the store has finished."""
    st = W.make_store("src", 42, 4096, 4, 256, 32, 128, slots="runs",
                      request_len=512)
    key, value, slots, ks, vs = store_inputs(st)
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size,
                                       st.num_heads, st.head_size, fill=0xAA)
    B, D = 64, 128
    stride = B * (D + 4)
    nb = st.cache_bytes // stride
    g = W.make_gather("over_store", 43, [500, 700, 300, 1], B, D, nb)
    g_cache = kv.view(-1)[: nb * stride].view(nb, stride)
    n = g.total_tokens
    k = torch.full((n, D), 0xCD, dtype=torch.uint8, device="cuda")
    s = torch.full((n, 4), 0xCD, dtype=torch.uint8, device="cuda")
    bt, cu = to_dev(g.block_table), to_dev(g.cu_seq_lens)
    kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs, flags=PDL)
    kvq.kvq_gather_indexer_k(g_cache, k, s, bt, cu, block_size=B,
                             flags=EARLY)
    torch.cuda.synchronize()
    stored = run_store(orc, st)
    g.cache = stored[: nb * stride].copy()
    wk, ws = run_gather(orc, g)
    assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, "k over store")
    assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, "s over store")


EARLY_READ = kvq.KVQ_F_PDL_EARLY_READ


@pytest.mark.parametrize("index", [0, 4])
def test_store_then_early_read_gather(orc, index):
    """The step's order: a PDL store into the NVFP4 pages, then an
    early-read gather from the (separate) indexer cache, three times back
    to back; the gather's cache reads may overlap the store, its writes
    may not."""
    st = W.store_workload(index)
    ga = W.gather_workload(index)
    key, value, slots, ks, vs = store_inputs(st)
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size,
                                       st.num_heads, st.head_size, fill=0xAA)
    cache, k, s, bt, cu = _gather_args(ga)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs, flags=PDL,
                            dev_error=err)
        kvq.kvq_gather_indexer_k(cache, k, s, bt, cu,
                                 block_size=ga.block_size, flags=EARLY_READ,
                                 dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bytes_equal(kv.cpu().numpy().reshape(-1), run_store(orc, st),
                       st.name)
    wk, ws = run_gather(orc, ga)
    assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, ga.name + " k")
    assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, ga.name + " s")


def test_early_read_gathers_back_to_back(orc):
    """Early-read gathers in a row (twice over four buffer sets), each
    from its own cache copy into its own outputs: every output matches the
    oracle."""
    ga = W.gather_workload(4)
    sets = [_gather_args(ga) for _ in range(4)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        for cache, k, s, bt, cu in sets:
            kvq.kvq_gather_indexer_k(cache, k, s, bt, cu,
                                     block_size=ga.block_size,
                                     flags=EARLY_READ, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, ws = run_gather(orc, ga)
    for _, k, s, _, _ in sets:
        assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, "k")
        assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, "s")


def test_early_read_gather_after_torch_write(orc):
    """An early-read gather right after an ordinary torch kernel that
    writes a buffer the gather does not read (its contract) gives the
    oracle's bytes, and the torch kernel's result is intact."""
    ga = W.gather_workload(3)
    cache, k, s, bt, cu = _gather_args(ga)
    other = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    other.fill_(7)
    kvq.kvq_gather_indexer_k(cache, k, s, bt, cu, block_size=ga.block_size,
                             flags=EARLY_READ, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int((other != 7).sum().item()) == 0
    wk, ws = run_gather(orc, ga)
    assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, "k")
    assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, "s")


@pytest.mark.parametrize("index", [0, 4])
def test_early_read_step(orc, index):
    """The bench's step with both calls in early-read mode, three times back
    to back: each store's inputs are not written by the gather before it,
    and each gather's inputs are not written by the store before it."""
    st = W.store_workload(index)
    ga = W.gather_workload(index)
    key, value, slots, ks, vs = store_inputs(st)
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size,
                                       st.num_heads, st.head_size, fill=0xAA)
    cache, k, s, bt, cu = _gather_args(ga)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs,
                            flags=EARLY_READ, dev_error=err)
        kvq.kvq_gather_indexer_k(cache, k, s, bt, cu,
                                 block_size=ga.block_size, flags=EARLY_READ,
                                 dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bytes_equal(kv.cpu().numpy().reshape(-1), run_store(orc, st),
                       st.name)
    wk, ws = run_gather(orc, ga)
    assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, ga.name + " k")
    assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, ga.name + " s")


def test_early_read_chain_of_stores(orc):
    """Early-read stores alternating two inputs into the same slots 9
    times: each store's writes still follow its predecessor's, so the pages
    hold exactly the last store's result."""
    a = W.make_store("a", 44, 4096, 4, 256, 32, 128, slots="runs",
                     request_len=512)
    b = W.make_store("b", 45, 4096, 4, 256, 32, 128, slots="runs",
                     request_len=512)
    b.slot_mapping = a.slot_mapping.copy()
    ins = [store_inputs(a), store_inputs(b)]
    kv, kc, vc = kvq.alloc_nvfp4_cache(a.num_blocks, a.block_size,
                                       a.num_heads, a.head_size, fill=0xAA)
    for i in range(9):
        key, value, slots, ks, vs = ins[i % 2]
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs,
                            flags=EARLY_READ)
    torch.cuda.synchronize()
    assert_bytes_equal(kv.cpu().numpy().reshape(-1), run_store(orc, a), "a")
