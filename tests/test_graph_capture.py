"""The hot-path calls allocate nothing, synchronise nothing and take their
stream from the caller, so a sequence of them can be captured once in a
CUDA graph and replayed with no per-call host work.  Captures the store ->
gather step (plain and PDL launches) and a decode attention call, replays
them, and checks the results against the oracle."""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import assert_bytes_equal, store_inputs, to_dev
from tests.test_oracle_gather import run_gather
from tests.test_oracle_store import run_store

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pdl", [False, True], ids=["plain", "pdl"])
def test_store_gather_step_in_a_graph(orc, pdl):
    st = W.store_workload(4)
    ga = W.gather_workload(4)
    key, value, slots, ks, vs = store_inputs(st)
    kv, kc, vc = kvq.alloc_nvfp4_cache(st.num_blocks, st.block_size,
                                       st.num_heads, st.head_size, fill=0xAA)
    cache = to_dev(ga.cache).view(ga.num_blocks, ga.block_stride)
    n = ga.total_tokens
    k = torch.full((n, ga.head_dim), 0xCD, dtype=torch.uint8, device="cuda")
    s = torch.full((n, 4), 0xCD, dtype=torch.uint8, device="cuda")
    bt, cu = to_dev(ga.block_table), to_dev(ga.cu_seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    f_store = kvq.KVQ_F_PDL if pdl else 0
    f_gather = kvq.KVQ_F_PDL_EARLY_READ if pdl else 0
    def step():
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs,
                            flags=f_store, dev_error=err)
        kvq.kvq_gather_indexer_k(cache, k, s, bt, cu,
                                 block_size=ga.block_size, flags=f_gather,
                                 dev_error=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture (one-time set-up calls)
    torch.cuda.synchronize()
    kv.fill_(0xAA)
    k.fill_(0xCD)
    s.fill_(0xCD)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(2):
                step()
    torch.cuda.synchronize()
    # capture ran nothing: the buffers still hold their fill
    assert int((kv != 0xAA).sum().item()) == 0
    assert int((k != 0xCD).sum().item()) == 0
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bytes_equal(kv.cpu().numpy().reshape(-1), run_store(orc, st),
                       st.name)
    wk, ws = run_gather(orc, ga)
    assert_bytes_equal(k.cpu().numpy().reshape(-1), wk, "k")
    assert_bytes_equal(s.cpu().numpy().reshape(-1), ws, "s")


def test_attention_in_a_graph(orc):
    from tests.test_parity_attention import (_upload, _vmax, assert_close,
                                             oracle_attention)
    wl = W.make_attention("graph", 96, [1, 700, 2049, 0, 513],
                          num_q_heads=16, num_kv_heads=2, head_size=128,
                          block_size=16)
    kv, kc, vc = _upload(wl)
    q = torch.from_numpy(wl.query.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    bt, lens = to_dev(wl.block_table), to_dev(wl.context_lens)
    ks = torch.tensor([float(wl.k_scale)], device="cuda")
    vs = torch.tensor([float(wl.v_scale)], device="cuda")
    mcl = int(wl.context_lens.max())
    scratch = kvq.attention_scratch(wl.num_seqs, wl.num_q_heads, mcl, 512,
                                    wl.head_size, torch.device("cuda"))
    es, ml, tmp = scratch
    def call():
        kvq.kvq_paged_attention_nvfp4(
            q, kc, vc, bt, lens, ks, vs, float(wl.scale), out, mcl, 512,
            es, ml, tmp, flags=kvq.KVQ_F_PDL)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # warm-up outside the capture (one-time set-up calls)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call()
    graph.replay()
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref, mag = oracle_attention(orc, wl)
    assert_close(got, ref, mag, _vmax(wl, wl.context_lens), "graph")
