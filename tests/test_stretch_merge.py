"""GPU tests of contexts split over several stretches and merged.

On contiguous pages the attention kernel splits a context of more than one
stretch (1792 tokens) into CTAs in the proportions 4 : ... : 4 : 1, each
writing its partial result to the caller's scratch, and the partition-merge
kernel combines them.  These tests run that path against the oracle over
contexts of two to ten stretches, with scratch full of random bits, twice in
a row on the same scratch, in a CUDA graph replayed with a new query each
time, and with partition sizes 512, 384 and 128 (which set the scratch rows
per head but not the stretches: the outputs are bitwise equal)."""
import dataclasses

import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import to_dev
from tests.test_oracle_attention import _nhd
from tests.test_parity_attention import (_upload, _vmax, assert_close,
                                         oracle_attention)

pytestmark = pytest.mark.gpu

LONG = [1281, 2560, 2561, 3841, 6400, 12800, 700, 1]


class Call:
    """One attention call's device buffers, the scratch filled with random
    bits."""

    def __init__(self, wl, partition_size=512, seed=0):
        self.wl, self.part = wl, partition_size
        self.caches = _upload(wl)
        self.q = torch.from_numpy(wl.query.view(np.int16)).cuda().view(
            torch.bfloat16)
        self.out = torch.full(self.q.shape, float("nan"),
                              dtype=torch.bfloat16, device="cuda")
        self.bt, self.lens = to_dev(wl.block_table), to_dev(wl.context_lens)
        self.ks = torch.tensor([float(wl.k_scale)], device="cuda")
        self.vs = torch.tensor([float(wl.v_scale)], device="cuda")
        self.mcl = int(wl.context_lens.max())
        self.scratch = kvq.attention_scratch(
            wl.num_seqs, wl.num_q_heads, self.mcl, partition_size,
            wl.head_size, torch.device("cuda"))
        g = torch.Generator(device="cuda").manual_seed(seed)
        for t in self.scratch:
            if t is None:  # every context within one partition: no scratch
                continue
            t.view(torch.int32).copy_(torch.randint(
                -2 ** 31, 2 ** 31 - 1, t.shape, dtype=torch.int32,
                device="cuda", generator=g))

    def __call__(self, flags=kvq.KVQ_F_PDL):
        _, kc, vc = self.caches
        es, ml, tmp = self.scratch
        kvq.kvq_paged_attention_nvfp4(
            self.q, kc, vc, self.bt, self.lens, self.ks, self.vs,
            float(self.wl.scale), self.out, self.mcl, self.part, es, ml, tmp,
            flags=flags | self.wl.flags)

    def result(self):
        torch.cuda.synchronize()
        return self.out.float().cpu().numpy().astype(np.float64)

    def check(self, orc, wl=None, what=""):
        wl = self.wl if wl is None else wl
        ref, mag = oracle_attention(orc, wl)
        return assert_close(self.result(), ref, mag,
                            _vmax(wl, wl.context_lens), what)


@pytest.mark.parametrize("part", [512, 128])
def test_many_stretches_random_scratch(orc, part):
    wl = W.make_attention(f"long{part}", 110, LONG, num_q_heads=16,
                          num_kv_heads=2, head_size=128, block_size=16)
    c = Call(wl, part, seed=part)
    c()
    c.check(orc, what="first call")
    first = c.result()
    c.out.fill_(float("nan"))
    c()
    c.check(orc, what="second call")
    assert np.array_equal(first, c.result())


def test_graph_replays_with_new_queries(orc):
    wl = W.make_attention("greplay", 112, [3000, 1281, 77, 2600, 5200],
                          num_q_heads=16, num_kv_heads=2, head_size=128,
                          block_size=16)
    c = Call(wl, 512, seed=7)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        c()  # the first call configures the kernel (outside the capture)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            c()
    rng = np.random.default_rng(113)
    for rep in range(3):
        qf = rng.standard_normal(wl.query.shape).astype(np.float32)
        bits = W.bf16_bits(qf.reshape(-1)).reshape(qf.shape)
        c.q.copy_(torch.from_numpy(bits.view(np.int16)).cuda().view(
            torch.bfloat16))
        c.out.fill_(float("nan"))
        graph.replay()
        c.check(orc, dataclasses.replace(wl, query=bits), f"replay {rep}")


def test_merge_matches_across_partition_sizes(orc):
    """The stretches do not depend on the caller's partition size; only the
    scratch row stride does, so the outputs are bitwise equal."""
    wl = W.make_attention("pstride", 114, [4000, 1500, 2561], num_q_heads=8,
                          num_kv_heads=1, head_size=128, block_size=16)
    outs = []
    for part in (512, 384, 128):
        c = Call(wl, part, seed=part + 1)
        c()
        outs.append(c.result())
    c.check(orc, what="partition strides")
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("swz", [0, 1])
@pytest.mark.parametrize("layout", [W.LAYOUT_HND, W.LAYOUT_NHD])
@pytest.mark.parametrize("B", [16, 32, 48, 8])
def test_stretch_boundaries(orc, B, layout, swz):
    """Contexts at the stretch length (1792) and at twice it, one token
    either side: the first of two stretches then holds up to 2848 tokens,
    a warp range up to 46 blocks of 16 (the block ids of its second 32
    blocks come from each lane's second entry); HND pages and NHD ones
    (with 2 KV heads, so that a head's token rows are 2 rows apart), K
    scales linear and swizzled; block size 8 (linear K scales) splits at
    1280 tokens, and 48 (and 8 with swizzled K scales) takes the
    per-fragment path with the caller's partitions."""
    wl = W.make_attention(f"edge{B}_{layout}_{swz}", 115,
                          [1792, 1793, 3584, 3585, 2000], num_q_heads=16,
                          num_kv_heads=2, head_size=128, block_size=B,
                          flags=swz)
    if layout == W.LAYOUT_NHD:
        wl = _nhd(wl)
    c = Call(wl, 512, seed=B)
    c()
    c.check(orc, what=f"stretch edges B={B} layout={layout} swz={swz}")


@pytest.mark.parametrize("B", [16, 8])
@pytest.mark.parametrize("layout", [W.LAYOUT_HND, W.LAYOUT_NHD])
def test_bad_blocks_in_long_ranges(orc, layout, B):
    """Out-of-range block ids among the second 32 blocks of a warp's range
    (block_size 16, contexts of 3584 and 3000 tokens: warp ranges of 736
    and 608 tokens, 46 and 38 blocks; block_size 8, 3584 and 3000 tokens:
    52 and 44 blocks) and among the first 32: flagged, and their tokens
    left out, as the oracle gives with those blocks removed from the
    table."""
    wl = W.make_attention(f"longbad{B}", 116, [3584, 3000, 2100],
                          num_q_heads=8, num_kv_heads=1, head_size=128,
                          block_size=B)
    if layout == W.LAYOUT_NHD:
        wl = _nhd(wl)
    # sequence -> block made bad (block_size 8: warp ranges of 52, 44 and
    # 52 blocks in the first stretches)
    drop = {0: 40, 1: 73, 2: 33} if B == 16 else {0: 40, 1: 33, 2: 5}
    wl.block_table[0, drop[0]] = -3
    wl.block_table[1, drop[1]] = wl.num_blocks
    wl.block_table[2, drop[2]] = wl.num_blocks + 100
    c = Call(wl, 512, seed=9)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, kc, vc = c.caches
    es, ml, tmp = c.scratch
    kvq.kvq_paged_attention_nvfp4(
        c.q, kc, vc, c.bt, c.lens, c.ks, c.vs, float(wl.scale), c.out,
        c.mcl, 512, es, ml, tmp, flags=kvq.KVQ_F_PDL, dev_error=err)
    got = c.result()
    assert int(err.item()) & kvq.KVQ_DEVERR_BLOCK
    bt = np.zeros_like(wl.block_table)
    lens = wl.context_lens.copy()
    for b in range(wl.num_seqs):
        row = list(wl.block_table[b])
        del row[drop[b]]
        row.append(0)
        lens[b] -= B
        bt[b] = row
    ref_wl = dataclasses.replace(wl, block_table=bt, context_lens=lens)
    ref, mag = oracle_attention(orc, ref_wl)
    assert_close(got, ref, mag, _vmax(ref_wl, lens), "bad blocks, long")


def test_early_metadata_back_to_back(orc):
    """Calls with KVQ_F_PDL_EARLY_META back to back on one stream (each
    after the previous call's merge kernel, which writes only the output):
    the lengths, block ids and query are read before the wait, the pages
    and every write after it; both results equal the plain call's and the
    oracle's."""
    wl = W.make_attention("early", 117, [3000, 77, 1800, 2600, 0, 1],
                          num_q_heads=16, num_kv_heads=2, head_size=128,
                          block_size=16)
    c = Call(wl, 512, seed=11)
    c(flags=0)
    plain = c.result()
    outs = []
    for _ in range(3):
        c.out.fill_(float("nan"))
        torch.cuda.synchronize()
        c(flags=kvq.KVQ_F_PDL_EARLY_META)
        c(flags=kvq.KVQ_F_PDL_EARLY_META)
        outs.append(c.result())
    c.check(orc, what="early metadata")
    for o in outs:
        assert np.array_equal(o, plain)


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F16])
@pytest.mark.parametrize("G", [8, 16, 3])
@pytest.mark.parametrize("layout", [W.LAYOUT_HND, W.LAYOUT_NHD])
def test_block_size_8_forms(orc, layout, G, dtype):
    """Block size 8 on HND and NHD pages with 3, 8 and 16 query heads per
    KV head and both query types, contexts from one token to several
    1280-token stretches, at the stretch length and twice it (ragged last
    steps and pieces)."""
    wl = W.make_attention(f"b8_{layout}_{G}_{dtype}", 118,
                          [1, 7, 8, 9, 33, 300, 1280, 1281, 2560, 2561,
                           4001],
                          num_q_heads=2 * G, num_kv_heads=2, head_size=128,
                          block_size=8, dtype=dtype)
    if layout == W.LAYOUT_NHD:
        wl = _nhd(wl)
    tdt = torch.float16 if dtype == W.DTYPE_F16 else torch.bfloat16
    c = Call(wl, 512, seed=G)
    c.q = torch.from_numpy(wl.query.view(np.int16)).cuda().view(tdt)
    c.out = torch.full(c.q.shape, float("nan"), dtype=tdt, device="cuda")
    c()
    c.check(orc, what=f"block_size 8 layout={layout} G={G} dtype={dtype}")


def _form_cases(n=20, seed=4049):
    """Seeded mixes aimed at the contiguous-page forms: block sizes 8 and
    powers of two from 16 to 128, HND and NHD pages, linear and swizzled K
    scales, 1 to 16 query heads per KV head, both query types, partition
    sizes 128 to 512, and contexts drawn around the block size, the step,
    the stretch lengths (1280 for block size 8, 1792 otherwise) and twice
    them."""
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(n):
        B = int(rng.choice([8, 16, 32, 64, 128]))
        S = 1280 if B == 8 else 1792
        G = int(rng.choice([1, 2, 4, 6, 8, 12, 16]))
        anchors = [B, 32, S, 2 * S, 3 * S]
        lens = [max(0, int(rng.choice(anchors)) + int(rng.integers(-3, 4)))
                for _ in range(int(rng.integers(2, 5)))]
        lens.append(int(rng.integers(0, 40)))
        cases.append(dict(name=f"form{k}", B=B, G=G, lens=lens,
                          layout=int(rng.integers(0, 2)),
                          swz=int(rng.integers(0, 2)),
                          dtype=int(rng.integers(0, 2)),
                          part=int(rng.choice([128, 256, 384, 512]))))
    return cases


@pytest.mark.parametrize("c", _form_cases(), ids=lambda c: c["name"])
def test_random_form_sweep(orc, c):
    wl = W.make_attention(c["name"], 500 + int(c["name"][4:]), c["lens"],
                          num_q_heads=c["G"] * 2, num_kv_heads=2,
                          head_size=128, block_size=c["B"],
                          flags=c["swz"], dtype=c["dtype"])
    if c["layout"] == W.LAYOUT_NHD:
        wl = _nhd(wl)
    tdt = torch.float16 if c["dtype"] == W.DTYPE_F16 else torch.bfloat16
    call = Call(wl, c["part"], seed=7 + int(c["name"][4:]))
    call.q = torch.from_numpy(wl.query.view(np.int16)).cuda().view(tdt)
    call.out = torch.full(call.q.shape, float("nan"), dtype=tdt,
                          device="cuda")
    call()
    call.check(orc, what=str(c))
