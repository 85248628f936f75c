"""GPU test of kvq_paged_attention_nvfp4_noalloc, the attention entry point
for callers that cannot allocate device memory (an engine that has reserved
all of it, a runtime that forbids allocation while serving).  It takes no
scratch from the caller and uses the library's built-in array instead.

Checked through the C ABI, on two calls in a row with different shapes (the
second finds the first one's leftovers in the shared array), against the
plain entry point given its own scratch, within the attention tests'
tolerance; and a call that needs more than the built-in array is refused
with KVQ_ERR_SCRATCH before anything is launched.  This file is collected
last so that a run stopping at its first failure has run everything else."""
import numpy as np
import pytest
import torch

from paged_quantized_kv_gb300 import kvq
from paged_quantized_kv_gb300 import workloads as W
from tests.test_parity_attention import (_upload, _vmax, oracle_attention,
                                         to_dev)

pytestmark = pytest.mark.gpu


def _inputs(wl):
    kv, kc, vc = _upload(wl)
    q = torch.from_numpy(wl.query.view(np.int16)).cuda().view(torch.bfloat16)
    return dict(kv=kv, kc=kc, vc=vc, q=q, bt=to_dev(wl.block_table),
                lens=to_dev(wl.context_lens),
                ks=torch.tensor([float(wl.k_scale)], device="cuda"),
                vs=torch.tensor([float(wl.v_scale)], device="cuda"),
                mcl=int(wl.context_lens.max()))


def _plain(wl, a, part):
    out = torch.full_like(a["q"], float("nan"))
    kvq.kvq_paged_attention_nvfp4(a["q"], a["kc"], a["vc"], a["bt"],
                                  a["lens"], a["ks"], a["vs"],
                                  float(wl.scale), out, a["mcl"],
                                  partition_size=part)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def _noalloc(wl, a, part):
    out = torch.full_like(a["q"], float("nan"))
    kvq.kvq_paged_attention_nvfp4_noalloc(a["q"], a["kc"], a["vc"], a["bt"],
                                          a["lens"], a["ks"], a["vs"],
                                          float(wl.scale), out, a["mcl"],
                                          partition_size=part)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def test_noalloc_matches_plain_entry_point(orc):
    cases = [
        (W.make_attention("noalloc_a", 101, [1500, 7, 900, 2049, 513, 0],
                          num_q_heads=16, num_kv_heads=2, head_size=128,
                          block_size=16), 256),
        (W.make_attention("noalloc_b", 102, [3000, 640, 128], num_q_heads=8,
                          num_kv_heads=8, head_size=128, block_size=32), 512),
    ]
    for wl, part in cases:  # two calls in a row, different shapes
        a = _inputs(wl)
        want = _plain(wl, a, part)
        got = _noalloc(wl, a, part)
        ref, mag = oracle_attention(orc, wl)
        tol = (2.0 ** -8 * np.abs(want) + 2.0 ** -9 * mag
               + 2.0 ** -24 * _vmax(wl, wl.context_lens)[:, None, None])
        assert np.isfinite(got).all(), wl.name
        bad = np.argwhere(np.abs(got - want) > tol)
        assert bad.size == 0, (wl.name, bad[:5])


def test_noalloc_refuses_requests_beyond_its_array():
    wl = W.make_attention("noalloc_big", 103, [16], num_q_heads=8,
                          num_kv_heads=1, head_size=128, block_size=16)
    a = _inputs(wl)
    # 8 heads x 1 sequence x P partitions x (128 + 2) floats > 32 MiB
    parts = kvq.KVQ_NOALLOC_SCRATCH_BYTES // (8 * 130 * 4) + 1
    out = torch.zeros_like(a["q"])
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_paged_attention_nvfp4_noalloc(
            a["q"], a["kc"], a["vc"], a["bt"], a["lens"], a["ks"], a["vs"],
            float(wl.scale), out, parts * 128, partition_size=128)
    assert e.value.status == kvq.KVQ_ERR_SCRATCH
    torch.cuda.synchronize()
    assert not out.any()  # nothing was launched


def test_noalloc_single_partition_uses_no_scratch(orc):
    """Every context within one partition: no scratch is needed, the array
    is not used, and the result equals the plain entry point's."""
    wl = W.make_attention("noalloc_one", 104, [512, 1, 300, 0, 129],
                          num_q_heads=8, num_kv_heads=1, head_size=128,
                          block_size=16)
    a = _inputs(wl)
    want = _plain(wl, a, 512)
    got = _noalloc(wl, a, 512)
    ref, mag = oracle_attention(orc, wl)
    tol = (2.0 ** -8 * np.abs(want) + 2.0 ** -9 * mag
           + 2.0 ** -24 * _vmax(wl, wl.context_lens)[:, None, None])
    assert np.isfinite(got).all()
    assert (np.abs(got - want) <= tol).all()


def test_noalloc_at_the_limit_and_one_partition_past_it(orc):
    """A call whose scratch is exactly the most rows the array holds is
    accepted (and matches the plain entry point); one more partition is
    refused.  rows = num_seqs * num_q_heads * partitions of the declared
    max_context_len, which may be far above the actual contexts."""
    cap = kvq.KVQ_NOALLOC_SCRATCH_BYTES // ((128 + 2) * 4)
    nseq, hq, parts = 137, 3, 157  # 137 * 3 * 157 == cap
    assert nseq * hq * parts == cap
    rng = np.random.default_rng(105)
    lens = rng.integers(1, 3001, size=nseq)
    lens[:3] = [3000, 1281, 2560]  # several stretches per context
    wl = W.make_attention("noalloc_cap", 105, lens, num_q_heads=hq,
                          num_kv_heads=1, head_size=128, block_size=16)
    a = _inputs(wl)
    a["mcl"] = parts * 512  # declared maximum: 157 partitions of 512
    want = _plain(wl, a, 512)
    got = _noalloc(wl, a, 512)
    ref, mag = oracle_attention(orc, wl)
    tol = (2.0 ** -8 * np.abs(want) + 2.0 ** -9 * mag
           + 2.0 ** -24 * _vmax(wl, wl.context_lens)[:, None, None])
    assert np.isfinite(got).all()
    assert (np.abs(got - want) <= tol).all()
    out = torch.zeros_like(a["q"])
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_paged_attention_nvfp4_noalloc(
            a["q"], a["kc"], a["vc"], a["bt"], a["lens"], a["ks"], a["vs"],
            float(wl.scale), out, (parts + 1) * 512, partition_size=512)
    assert e.value.status == kvq.KVQ_ERR_SCRATCH
    torch.cuda.synchronize()
    assert not out.any()


def test_noalloc_back_to_back_pdl_calls_share_the_array(orc):
    """Two calls with KVQ_F_PDL on one stream, different shapes, no
    synchronisation between them: the second call's kernels wait for the
    first call's merge before they touch the shared array, so both results
    match the plain entry point's."""
    wl1 = W.make_attention("noalloc_p1", 106, [2600, 900, 1700, 5],
                           num_q_heads=16, num_kv_heads=2, head_size=128,
                           block_size=16)
    wl2 = W.make_attention("noalloc_p2", 107, [4000, 2561, 130],
                           num_q_heads=8, num_kv_heads=1, head_size=128,
                           block_size=16)
    a1, a2 = _inputs(wl1), _inputs(wl2)
    want1 = _plain(wl1, a1, 256)
    want2 = _plain(wl2, a2, 512)
    out1 = torch.full_like(a1["q"], float("nan"))
    out2 = torch.full_like(a2["q"], float("nan"))
    for wl, a, out, part in ((wl1, a1, out1, 256), (wl2, a2, out2, 512)):
        kvq.kvq_paged_attention_nvfp4_noalloc(
            a["q"], a["kc"], a["vc"], a["bt"], a["lens"], a["ks"], a["vs"],
            float(wl.scale), out, a["mcl"], partition_size=part,
            flags=kvq.KVQ_F_PDL)
    torch.cuda.synchronize()
    for wl, out, want in ((wl1, out1, want1), (wl2, out2, want2)):
        got = out.float().cpu().numpy().astype(np.float64)
        ref, mag = oracle_attention(orc, wl)
        tol = (2.0 ** -8 * np.abs(want) + 2.0 ** -9 * mag
               + 2.0 ** -24 * _vmax(wl, wl.context_lens)[:, None, None])
        assert np.isfinite(got).all(), wl.name
        assert (np.abs(got - want) <= tol).all(), wl.name


def test_noalloc_rejects_bad_arguments_with_the_plain_codes():
    """Arguments the plain entry point rejects get its codes, even when the
    declared context would also need more scratch than the array holds."""
    wl = W.make_attention("noalloc_args", 108, [16], num_q_heads=8,
                          num_kv_heads=1, head_size=128, block_size=16)
    a = _inputs(wl)
    out = torch.zeros_like(a["q"])
    huge = 1 << 22  # partitions far past the array
    for part, flags, code in ((100, 0, kvq.KVQ_ERR_SHAPE),
                              (1024, 0, kvq.KVQ_ERR_SHAPE),
                              (512, 1 << 3, kvq.KVQ_ERR_ARG)):
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_paged_attention_nvfp4_noalloc(
                a["q"], a["kc"], a["vc"], a["bt"], a["lens"], a["ks"],
                a["vs"], float(wl.scale), out, huge, partition_size=part,
                flags=flags)
        assert e.value.status == code, (part, flags)
    torch.cuda.synchronize()
    assert not out.any()
