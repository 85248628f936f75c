"""The sharded path on one GPU: the store split by request and the gather
split by sequence (the units the replicas of a multi-GPU run take, with no
exchange step), each shard run through the CUDA kernels in sequence.  The
union of the shards' writes must equal, byte for byte, both the unsharded
GPU call and the oracle -- cache pages (sentinels included) for the store,
k_fp8 / k_scale rows for the gather."""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import assert_bytes_equal, store_inputs, to_dev
from tests.test_oracle_gather import run_gather
from tests.test_oracle_store import run_store

pytestmark = pytest.mark.gpu


def _store_into(wl, kc, vc, err):
    key, value, slots, ks, vs = store_inputs(wl)
    kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs, flags=wl.flags,
                        dev_error=err)


@pytest.mark.parametrize("index,unit", [(2, 1024), (0, 1)],
                         ids=["prefill_store", "tiny_store"])
@pytest.mark.parametrize("world", [2, 3, 4])
def test_store_shards_union(orc, index, unit, world):
    full = W.store_workload(index)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches = []
    for sharded in (False, True):
        kv, kc, vc = kvq.alloc_nvfp4_cache(full.num_blocks, full.block_size,
                                           full.num_heads, full.head_size,
                                           full.layout, fill=0xAA)
        if sharded:
            for r in range(world):
                _store_into(W.shard_store(full, r, world, unit_tokens=unit),
                            kc, vc, err)
        else:
            _store_into(full, kc, vc, err)
        torch.cuda.synchronize()
        caches.append(kv.cpu().numpy().reshape(-1))
        del kv, kc, vc
    assert int(err.item()) == 0
    assert_bytes_equal(caches[1], caches[0], "shards vs one call")
    assert_bytes_equal(caches[1], run_store(orc, full), "shards vs oracle")


@pytest.mark.parametrize("index", [3, 4, 0],
                         ids=["prefill_gather", "long_gather", "tiny_gather"])
@pytest.mark.parametrize("world", [2, 3, 4])
def test_gather_shards_union(orc, index, world):
    full = W.gather_workload(index)
    n, D = full.total_tokens, full.head_dim
    cache = to_dev(full.cache).view(full.num_blocks, full.block_stride)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for sharded in (False, True):
        k = torch.full((n, D), 0xCD, dtype=torch.uint8, device="cuda")
        s = torch.full((n, 4), 0xCD, dtype=torch.uint8, device="cuda")
        parts = [W.shard_gather(full, r, world) for r in range(world)] \
            if sharded else [(full, 0)]
        for sub, first in parts:
            m = sub.total_tokens
            if m == 0 and sub.num_seqs == 0:
                continue
            kvq.kvq_gather_indexer_k(
                cache, k[first:first + m], s[first:first + m],
                to_dev(sub.block_table), to_dev(sub.cu_seq_lens),
                block_size=sub.block_size, dev_error=err)
        torch.cuda.synchronize()
        outs.append((k.cpu().numpy().reshape(-1), s.cpu().numpy().reshape(-1)))
    assert int(err.item()) == 0
    (k_one, s_one), (k_sh, s_sh) = outs
    wk, ws = run_gather(orc, full)
    assert_bytes_equal(k_sh, k_one, "k_fp8 shards vs one call")
    assert_bytes_equal(s_sh, s_one, "k_scale shards vs one call")
    assert_bytes_equal(k_sh, wk, "k_fp8 shards vs oracle")
    assert_bytes_equal(s_sh, ws, "k_scale shards vs oracle")
