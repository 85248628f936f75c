"""GPU parity of kvq_paged_attention_nvfp4 against the CPU oracle.

The oracle computes the attention exactly (double, exact dequantisation);
the kernel rounds the query to fp16, accumulates q . (e2m1 * sf) and P . V'
in fp32 on the tensor cores, rounds P to fp16 and the output to bf16 / fp16.
Every output element must satisfy

    |out - ref| <= 2^-8 |ref| + 2^-9 mag + 2^-24 vmax

with ref and mag = sum_t p_t |V^[t, d]| from the oracle and vmax the
largest |V^| of the sequence: 2^-8 |ref| covers the final rounding to bf16
(half an ulp) and the fp32 accumulation error of out itself; 2^-9 mag covers
the fp16 rounding of each weight (2^-11 relative, once in the numerator and
once through the denominator) and the fp32 logit error; 2^-24 vmax covers
weights below the fp16 normal range (absolute error 2^-25 each).

Covers contexts of 0, 1, B-1, B, B+1, 127, 128, 129 .. 2049 tokens (partial
tiles, one to five partitions, the partition merge), partition sizes 128 to
512, GQA group sizes 1 to 16, bf16 and fp16 queries, HND and NHD pages,
swizzled K scales, block sizes 4 to 384 (12 and 384 not powers of two),
large logits (one-hot weights), pages written by the GPU store, a PDL chain
store -> attention, the Llama-3.1-70B-shaped decode batch (sampled rows),
clamped contexts and invalid block ids (flags), and bitwise determinism.
The ranges of the kernel's warps (a quarter of a stretch of up to 2048
tokens each, walked in steps of 32) end inside a step, at a step boundary
and one token past it across these lengths, so both the unmasked steps and
the masked last step run, and a bad block id makes a whole range masked."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.gpu_helpers import store_inputs, to_dev
from tests.test_oracle_attention import _nhd

pytestmark = pytest.mark.gpu


def _upload(wl):
    H, B, D = wl.num_kv_heads, wl.block_size, wl.head_size
    kv, kc, vc = kvq.alloc_nvfp4_cache(wl.num_blocks, B, H, D, wl.layout)
    assert kc.stride(0) == wl.page_stride
    kv.view(-1).copy_(torch.from_numpy(wl.cache))
    return kv, kc, vc


def gpu_attention(wl, partition_size=512, max_context_len=None, flags=None,
                  dev_error=None, caches=None):
    kv, kc, vc = _upload(wl) if caches is None else caches
    tdt = torch.float16 if wl.dtype == W.DTYPE_F16 else torch.bfloat16
    q = torch.from_numpy(wl.query.view(np.int16)).cuda().view(tdt)
    out = torch.full(q.shape, float("nan"), dtype=tdt, device="cuda")
    bt = to_dev(wl.block_table)
    lens = to_dev(wl.context_lens)
    ks = torch.tensor([float(wl.k_scale)], device="cuda")
    vs = torch.tensor([float(wl.v_scale)], device="cuda")
    mcl = (int(wl.context_lens.max()) if wl.context_lens.size else 0) \
        if max_context_len is None else max_context_len
    kvq.kvq_paged_attention_nvfp4(
        q, kc, vc, bt, lens, ks, vs, float(wl.scale), out, mcl,
        partition_size=partition_size,
        flags=wl.flags if flags is None else flags,
        dev_error=dev_error)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def oracle_attention(orc, wl, context_lens=None):
    lens = wl.context_lens if context_lens is None else context_lens
    out, mag = orc.paged_attention_nvfp4(
        wl.query, wl.cache, 0, wl.side_bytes, wl.page_stride, wl.block_size,
        wl.num_blocks, wl.layout, wl.num_kv_heads, wl.block_table, lens,
        wl.k_scale, wl.v_scale, wl.scale, wl.flags & 1, wl.dtype)
    return out, mag


def _vmax(wl, lens):
    """Largest possible |V^| of each sequence: 6 * largest V scale byte
    value of its pages * v_scale (a bound, from the page bytes)."""
    H, B, D = wl.num_kv_heads, wl.block_size, wl.head_size
    pages = wl.cache.reshape(wl.num_blocks, wl.page_stride)
    sc0 = wl.side_bytes + H * B * D // 2
    vs = pages[:, sc0:sc0 + H * B * D // 16].astype(np.int64)
    e4 = np.array([oracle.get().e4m3_decode(c) for c in range(127)])
    peak = e4[np.clip(vs, 0, 126)].max(axis=1)       # per block
    out = np.zeros(len(lens))
    for b, L in enumerate(lens):
        n = (int(L) + B - 1) // B
        if n:
            out[b] = 6.0 * peak[wl.block_table[b, :n]].max() * float(
                wl.v_scale)
    return out


def assert_close(got, ref, mag, vmax, what=""):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), what
    tol = (2.0 ** -8 * np.abs(ref) + 2.0 ** -9 * mag
           + 2.0 ** -24 * vmax[:, None, None])
    err = np.abs(got - ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (what, [(tuple(i), got[tuple(i)], ref[tuple(i)],
                                   tol[tuple(i)]) for i in bad[:5]])
    return float((err / np.maximum(tol, 1e-300)).max())


def _check(orc, wl, **kw):
    got = gpu_attention(wl, **kw)
    ref, mag = oracle_attention(orc, wl)
    return assert_close(got, ref, mag, _vmax(wl, wl.context_lens), wl.name)


LENS = [1, 15, 16, 17, 127, 128, 129, 255, 300, 511, 512, 513, 700, 1025,
        2049, 0]


@pytest.mark.parametrize("part", [512, 256, 128, 384])
def test_contexts_and_partitions(orc, part):
    wl = W.make_attention("ctx", 21, LENS, num_q_heads=16, num_kv_heads=2,
                          head_size=128, block_size=16)
    _check(orc, wl, partition_size=part)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_group_sizes(orc, G):
    Hkv = 2
    wl = W.make_attention(f"g{G}", 30 + G, [3, 200, 640, 129],
                          num_q_heads=G * Hkv, num_kv_heads=Hkv,
                          head_size=128, block_size=16)
    _check(orc, wl)


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F16])
@pytest.mark.parametrize("layout", [W.LAYOUT_HND, W.LAYOUT_NHD])
@pytest.mark.parametrize("swz", [0, oracle.F_SWIZZLE_K_SCALE])
def test_layouts_dtypes_swizzle(orc, dtype, layout, swz):
    wl = W.make_attention("lay", 40, [77, 600, 5, 1000], num_q_heads=8,
                          num_kv_heads=4, head_size=128, block_size=16,
                          dtype=dtype, flags=swz)
    if layout == W.LAYOUT_NHD:
        wl = _nhd(wl)
    _check(orc, wl)


@pytest.mark.parametrize("B", [4, 8, 12, 32, 64, 128, 256, 384])
def test_block_sizes(orc, B):
    lens = [B - 1, B, B + 1, 4 * B + 3, 900]
    wl = W.make_attention(f"B{B}", 50 + B, [n for n in lens if n <= 2100],
                          num_q_heads=8, num_kv_heads=1, head_size=128,
                          block_size=B)
    _check(orc, wl)


def test_one_hot_logits(orc):
    wl = W.make_attention("hot", 60, [300, 1200, 40], num_q_heads=8,
                          num_kv_heads=2, head_size=128, block_size=16,
                          scale=50.0)
    _check(orc, wl)


@pytest.mark.parametrize("scale", [-0.088, 0.0, -50.0])
@pytest.mark.parametrize("Hq", [16, 32])
def test_negative_and_zero_scale(orc, Hq, scale):
    """A negative softmax scale (the largest weights go to the smallest dot
    products; -50 makes them one-hot) and a zero one (every logit 0: each
    output is the mean of its context's values), over contexts of several
    stretches and partitions, with 8 and 16 query heads per KV head."""
    wl = W.make_attention(f"scale{scale}_{Hq}", 61, [300, 1500, 40, 2600],
                          num_q_heads=Hq, num_kv_heads=2, head_size=128,
                          block_size=16, scale=scale)
    _check(orc, wl)


def test_store_then_attention(orc):
    """Pages written by the GPU store from bf16 K/V (scales as a checkpoint
    would give), read by the attention, against the oracle on the same
    bytes; also as a PDL chain in which the attention reads what the store
    just wrote, with and without early metadata reads."""
    swl = W.make_store("sa", 70, num_tokens=3 * 512, num_heads=2,
                       head_size=128, block_size=16, num_blocks=200,
                       slots="runs", request_len=512)
    bt, _ = W.sequences_of_store(swl, 512)
    lens = np.array([512, 300, 77], dtype=np.int32)
    key, value, slots, ks, vs = store_inputs(swl)
    kv, kc, vc = kvq.alloc_nvfp4_cache(swl.num_blocks, 16, 2, 128)
    kv.zero_()
    rng = np.random.default_rng(71)
    qf = rng.standard_normal((3, 8, 128)).astype(np.float32)
    q_bits = W.bf16_bits(qf.reshape(-1)).reshape(qf.shape)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    outs = []
    bt_d, lens_d = to_dev(bt), to_dev(lens)
    for flags in (0, kvq.KVQ_F_PDL, kvq.KVQ_F_PDL_EARLY_META):
        out = torch.empty_like(q)
        kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs,
                            flags=flags & kvq.KVQ_F_PDL)
        # the store writes only the pages: the attention may read its
        # lengths, block ids and query before it finishes
        kvq.kvq_paged_attention_nvfp4(
            q, kc, vc, bt_d, lens_d, ks, vs, 0.088, out, 512, flags=flags)
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy().astype(np.float64))
        kv.zero_()
    kvq.kvq_store_nvfp4(key, value, kc, vc, slots, ks, vs)
    torch.cuda.synchronize()
    wl = W.AttentionWorkload(
        name="store_then_attention", query=q_bits, num_kv_heads=2,
        block_size=16, num_blocks=swl.num_blocks,
        cache=kv.cpu().numpy().reshape(-1), block_table=bt,
        context_lens=lens, k_scale=swl.k_scale, v_scale=swl.v_scale,
        scale=np.float32(0.088))
    ref, mag = oracle_attention(orc, wl)
    vmax = _vmax(wl, lens)
    for got in outs:
        assert_close(got, ref, mag, vmax, "store->attention")
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(outs[0], outs[2])


def test_llama70b_decode_batch_sampled(orc):
    """The benchmark's decode step (200 sequences, 64 query / 8 KV heads),
    run in full on the GPU; eight sequences checked against the oracle."""
    wl = W.attention_workload()
    got = gpu_attention(wl)
    rng = np.random.default_rng(72)
    pick = np.sort(rng.choice(wl.num_seqs, size=8, replace=False))
    pick[0] = int(np.argmax(wl.context_lens))       # the longest context
    sub = W.AttentionWorkload(
        name="sampled", query=wl.query[pick], num_kv_heads=8, block_size=16,
        num_blocks=wl.num_blocks, cache=wl.cache,
        block_table=wl.block_table[pick], context_lens=wl.context_lens[pick],
        k_scale=wl.k_scale, v_scale=wl.v_scale, scale=wl.scale)
    ref, mag = oracle_attention(orc, sub)
    assert_close(got[pick], ref, mag, _vmax(sub, sub.context_lens),
                 "llama70b_decode")


def test_deterministic(orc):
    wl = W.make_attention("det", 80, [900, 33, 1500], num_q_heads=16,
                          num_kv_heads=2, head_size=128, block_size=16)
    a = gpu_attention(wl)
    b = gpu_attention(wl)
    assert np.array_equal(a, b)


def test_clamped_context_and_flags(orc):
    wl = W.make_attention("clamp", 90, [700, 100], num_q_heads=8,
                          num_kv_heads=1, head_size=128, block_size=16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_attention(wl, max_context_len=600, dev_error=err)
    assert int(err.item()) & kvq.KVQ_DEVERR_SEQ
    ref, mag = oracle_attention(orc, wl, np.array([600, 100], np.int32))
    assert_close(got, ref, mag, _vmax(wl, [600, 100]), "clamped")

    # an out-of-range block id on the last page of sequence 0: flagged, its
    # tokens (48..63) left out -- the same result as a 48-token context
    bad = W.make_attention("badblk", 91, [64, 40], num_q_heads=8,
                           num_kv_heads=1, head_size=128, block_size=16)
    bad.block_table[0, 3] = bad.num_blocks + 5
    err.zero_()
    got = gpu_attention(bad, dev_error=err)
    assert int(err.item()) & kvq.KVQ_DEVERR_BLOCK
    lens = np.array([48, 40], np.int32)
    ref, mag = oracle_attention(orc, bad, lens)
    assert_close(got, ref, mag, _vmax(bad, lens), "bad block")


def test_bad_blocks_inside_contexts(orc):
    """Out-of-range block ids (negative and past the cache) in the middle of
    contexts: flagged, and their B tokens left out.  The attention of one
    query token does not depend on the order of the context's tokens, so
    the reference is the oracle over the block table with those entries
    removed and each context shortened by one block (a partial last block
    stays last)."""
    B = 16
    wl = W.make_attention("midbad", 96, [64, 40, 100, 1300], num_q_heads=8,
                          num_kv_heads=2, head_size=128, block_size=B)
    drop = {0: 1, 2: 2, 3: 40}           # sequence -> block index made bad
    wl.block_table[0, 1] = -1
    wl.block_table[2, 2] = wl.num_blocks + 7
    wl.block_table[3, 40] = wl.num_blocks
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_attention(wl, dev_error=err)
    assert int(err.item()) & kvq.KVQ_DEVERR_BLOCK
    bt = np.zeros_like(wl.block_table)
    lens = wl.context_lens.copy()
    for b in range(wl.num_seqs):
        row = list(wl.block_table[b])
        if b in drop:
            del row[drop[b]]
            row.append(0)
            lens[b] -= B
        bt[b] = row
    ref_wl = dataclasses.replace(wl, block_table=bt, context_lens=lens)
    ref, mag = oracle_attention(orc, ref_wl)
    assert_close(got, ref, mag, _vmax(ref_wl, lens), "bad blocks inside")


def test_long_contexts_many_partitions(orc):
    """Contexts of several thousand tokens (up to 17 partitions of 512; on
    these pages the kernel's CTAs cover stretches of up to 2048 tokens, the
    last of a context a quarter of the others) with a
    max_context_len above the longest context, so the scratch has more rows
    than used."""
    wl = W.make_attention("long", 95, [4097, 8191, 3000, 1, 1024, 2048],
                          num_q_heads=16, num_kv_heads=2, head_size=128,
                          block_size=16)
    _check(orc, wl, partition_size=512, max_context_len=9000)


def _sweep_cases(n=14, seed=2027):
    """Seeded random mixes of the attention's shape parameters: query heads
    per KV head, block size (powers of two and other multiples of 4, so
    both page paths run), layout, swizzled K scales, query type, partition
    size, and contexts drawn around the block size, the 32-token step, the
    partition size and the 1280-token stretch (split 4 : ... : 4 : 1 when a
    context needs several)."""
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(n):
        G = int(rng.choice([1, 2, 4, 8, 16]))
        Hkv = int(rng.choice([1, 2])) if G < 16 else 1
        B = int(rng.choice([16, 32, 48, 64, 12, 20]))
        part = int(rng.choice([128, 256, 384, 512]))
        anchors = [B, 32, part, 1280, 2560, 3840]
        lens = []
        for _ in range(int(rng.integers(2, 6))):
            a = int(rng.choice(anchors)) * int(rng.integers(1, 3))
            lens.append(max(0, a + int(rng.integers(-3, 4))))
        lens.append(int(rng.integers(0, 40)))
        cases.append(dict(name=f"sweep{k}", G=G, Hkv=Hkv, B=B, part=part,
                          lens=[min(x, 6000) for x in lens],
                          layout=int(rng.integers(0, 2)),
                          swz=int(rng.integers(0, 2)) if k % 3 == 0 else 0,
                          dtype=int(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("c", _sweep_cases(), ids=lambda c: c["name"])
def test_random_shape_sweep(orc, c):
    wl = W.make_attention(c["name"], 300 + int(c["name"][5:]), c["lens"],
                          num_q_heads=c["G"] * c["Hkv"],
                          num_kv_heads=c["Hkv"], head_size=128,
                          block_size=c["B"], layout=c["layout"],
                          flags=c["swz"], dtype=c["dtype"])
    _check(orc, wl, partition_size=c["part"])
