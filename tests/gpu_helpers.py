"""Run the CUDA path (through the C-ABI binding) on workload inputs and
bring the results back as numpy byte arrays laid out like the oracle's."""
import numpy as np
import torch

from paged_quantized_kv_gb300 import kvq


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def store_inputs(wl, device="cuda"):
    tdt = torch.float16 if wl.dtype == 1 else torch.bfloat16
    src = torch.from_numpy(wl.src.view(np.int16)).to(device).view(tdt)
    T, H, D = wl.num_tokens, wl.num_heads, wl.head_size
    key = src.as_strided((T, H, D), (wl.key_stride0, D, 1), wl.key_offset)
    value = src.as_strided((T, H, D), (wl.value_stride0, D, 1),
                           wl.value_offset)
    slots = torch.from_numpy(wl.slot_mapping).to(device)
    ks = torch.tensor([float(wl.k_scale)], dtype=torch.float32,
                      device=device)
    vs = torch.tensor([float(wl.v_scale)], dtype=torch.float32,
                      device=device)
    return key, value, slots, ks, vs


def gpu_store(wl, sentinel=0xAA, slot_mapping=None):
    """Returns (cache bytes as the oracle lays them out, dev_error)."""
    key, value, slots, ks, vs = store_inputs(wl)
    if slot_mapping is not None:
        slots = torch.from_numpy(np.asarray(slot_mapping,
                                            dtype=np.int64)).cuda()
    kv, kc, vc = kvq.alloc_nvfp4_cache(wl.num_blocks, wl.block_size,
                                       wl.num_heads, wl.head_size,
                                       wl.layout, fill=sentinel)
    assert kc.stride(0) == wl.page_stride
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs, flags=wl.flags,
                        dev_error=err)
    torch.cuda.synchronize()
    return kv.cpu().numpy().reshape(-1), int(err.item())


def gpu_gather(wl, total=None, sentinel=0xCD, block_table=None,
               bt_cols=None, flags=0):
    """bt_cols: hand the kernel only the first bt_cols columns of the block
    table (a view whose row stride is wider than its used part)."""
    total = wl.total_tokens if total is None else total
    cache = to_dev(wl.cache).view(wl.num_blocks, wl.block_stride)
    bt = to_dev(wl.block_table if block_table is None else block_table)
    if bt_cols is not None:
        bt = bt[:, :bt_cols]
    cu = to_dev(wl.cu_seq_lens)
    k = torch.full((max(total, 1), wl.head_dim), sentinel, dtype=torch.uint8,
                   device="cuda")[:total]
    s = torch.full((max(total, 1), 4), sentinel, dtype=torch.uint8,
                   device="cuda")[:total]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_gather_indexer_k(cache, k, s, bt, cu, block_size=wl.block_size,
                             flags=flags, dev_error=err)
    torch.cuda.synchronize()
    return (k.cpu().numpy().reshape(-1), s.cpu().numpy().reshape(-1),
            int(err.item()))


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what=""):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (
        f"{what}: {bad.size} bytes differ; first at "
        + ", ".join(f"{i}: gpu {got[i]:#04x} oracle {want[i]:#04x}"
                    for i in bad[:6]))
