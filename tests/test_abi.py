"""Host-only checks of the C-ABI library (no GPU needed, nothing launched).

* libkvq.so builds for sm_103a, loads, and exports exactly the functions
  include/kvq.h declares;
* every validation rule returns its status code before any device memory is
  touched or any kernel launched (each call below breaks exactly one rule,
  so none of them reaches a launch);
* the binding fails loudly when the library is missing;
* no product source imports or links the oracle.
"""
import ctypes
import os
import re
import subprocess

import pytest

from paged_quantized_kv_gb300 import build as kbuild
from paged_quantized_kv_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvq.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(kvq_\w+)\s*\(", text))


def test_exports_match_header(lib):
    declared = header_functions()
    assert {"kvq_store_nvfp4", "kvq_gather_indexer_k", "kvq_load_nvfp4",
            "kvq_store_indexer_k", "kvq_paged_attention_nvfp4",
            "kvq_status_string", "kvq_version"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(kvq_\w+)$", out, flags=re.M))
    assert exported == declared
    for name in declared:
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert kvq.kvq_version() == 100
    for code in range(0, -8, -1):
        assert kvq.kvq_status_string(code) != "unknown status"
    assert kvq.kvq_status_string(-99) == "unknown status"


# fake, 16-byte aligned addresses: never dereferenced because every call
# below fails validation first
A = 0x10000


def store(lib, **kw):
    args = dict(key=A, key_stride0=128, value=A, value_stride0=128,
                dtype=0, num_tokens=4, num_heads=1, head_size=128,
                key_cache=A, value_cache=A, page_stride=2 * 1 * 16 * 72,
                block_size=16, num_blocks=8, layout=0, slot_mapping=A,
                k_scale=A, v_scale=A, flags=0, dev_error=None, stream=None)
    args.update(kw)
    return lib.kvq_store_nvfp4(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), kvq.KVQ_ERR_DTYPE),
    (dict(layout=2), kvq.KVQ_ERR_LAYOUT),
    (dict(flags=4), kvq.KVQ_ERR_ARG),
    (dict(head_size=96), kvq.KVQ_ERR_SHAPE),
    (dict(head_size=0), kvq.KVQ_ERR_SHAPE),
    (dict(block_size=6), kvq.KVQ_ERR_SHAPE),
    (dict(num_heads=0), kvq.KVQ_ERR_SHAPE),
    (dict(num_tokens=-1), kvq.KVQ_ERR_SHAPE),
    (dict(num_blocks=-1), kvq.KVQ_ERR_SHAPE),
    (dict(page_stride=100), kvq.KVQ_ERR_SHAPE),
    (dict(key_stride0=-8), kvq.KVQ_ERR_SHAPE),
    (dict(key=None), kvq.KVQ_ERR_NULL),
    (dict(slot_mapping=None), kvq.KVQ_ERR_NULL),
    (dict(v_scale=None), kvq.KVQ_ERR_NULL),
    (dict(key=A + 8), kvq.KVQ_ERR_ALIGN),
    (dict(value_cache=A + 4), kvq.KVQ_ERR_ALIGN),
    (dict(value_stride0=132), kvq.KVQ_ERR_ALIGN),
    (dict(page_stride=2 * 16 * 72 + 8), kvq.KVQ_ERR_ALIGN),
    (dict(slot_mapping=A + 4), kvq.KVQ_ERR_ALIGN),
    (dict(num_tokens=0, key=None, value=None, slot_mapping=None),
     kvq.KVQ_OK),
])
def test_store_validation(lib, kw, code):
    assert store(lib, **kw) == code


def gather(lib, **kw):
    args = dict(kv_cache=A, block_stride=64 * 132, num_blocks=8,
                block_size=64, head_dim=128, block_table=A,
                block_table_stride=4, max_blocks_per_seq=4, cu_seq_lens=A,
                num_seqs=2, total_tokens=100, k_fp8=A, k_scale=A, flags=0,
                dev_error=None, stream=None)
    args.update(kw)
    return lib.kvq_gather_indexer_k(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=20), kvq.KVQ_ERR_SHAPE),
    (dict(block_size=0), kvq.KVQ_ERR_SHAPE),
    (dict(block_stride=64 * 131), kvq.KVQ_ERR_SHAPE),
    (dict(block_table_stride=3), kvq.KVQ_ERR_SHAPE),
    (dict(num_seqs=-1), kvq.KVQ_ERR_SHAPE),
    (dict(total_tokens=-5), kvq.KVQ_ERR_SHAPE),
    (dict(total_tokens=1 << 31), kvq.KVQ_ERR_SHAPE),
    (dict(num_seqs=0), kvq.KVQ_ERR_ARG),
    (dict(flags=1), kvq.KVQ_ERR_ARG),
    (dict(flags=8), kvq.KVQ_ERR_ARG),
    (dict(k_fp8=None), kvq.KVQ_ERR_NULL),
    (dict(cu_seq_lens=None), kvq.KVQ_ERR_NULL),
    (dict(k_fp8=A + 4), kvq.KVQ_ERR_ALIGN),
    (dict(k_scale=A + 2), kvq.KVQ_ERR_ALIGN),
    (dict(kv_cache=A + 8), kvq.KVQ_ERR_ALIGN),
    (dict(block_stride=64 * 132 + 4), kvq.KVQ_ERR_ALIGN),
    (dict(total_tokens=0, k_fp8=None, kv_cache=None), kvq.KVQ_OK),
])
def test_gather_validation(lib, kw, code):
    assert gather(lib, **kw) == code


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(kvq, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(kvq, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        kvq.lib()


def test_product_never_touches_oracle():
    pkg = os.path.join(ROOT, "paged_quantized_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(
                    r"^\s*(import|from)\s+oracle\b|kvq_oracle|kvqo_", text,
                    flags=re.M), f


def load(lib, **kw):
    args = dict(key_cache=A, value_cache=A, page_stride=2 * 16 * 72,
                block_size=16, num_blocks=8, layout=0, num_heads=1,
                head_size=128, block_table=A, block_table_stride=4,
                max_blocks_per_seq=4, cu_seq_lens=A, num_seqs=2,
                total_tokens=100, k_scale=A, v_scale=A, out_dtype=0,
                key_out=A, value_out=A, out_stride0=128, flags=0,
                dev_error=None, stream=None)
    args.update(kw)
    return lib.kvq_load_nvfp4(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(out_dtype=1), kvq.KVQ_ERR_DTYPE),
    (dict(layout=3), kvq.KVQ_ERR_LAYOUT),
    (dict(flags=8), kvq.KVQ_ERR_ARG),
    (dict(head_size=96), kvq.KVQ_ERR_SHAPE),
    (dict(block_size=6), kvq.KVQ_ERR_SHAPE),
    (dict(page_stride=64), kvq.KVQ_ERR_SHAPE),
    (dict(out_stride0=64), kvq.KVQ_ERR_SHAPE),
    (dict(block_table_stride=2), kvq.KVQ_ERR_SHAPE),
    (dict(total_tokens=-1), kvq.KVQ_ERR_SHAPE),
    (dict(num_seqs=0), kvq.KVQ_ERR_ARG),
    (dict(key_out=None), kvq.KVQ_ERR_NULL),
    (dict(v_scale=None), kvq.KVQ_ERR_NULL),
    (dict(value_out=A + 8), kvq.KVQ_ERR_ALIGN),
    (dict(out_stride0=132), kvq.KVQ_ERR_ALIGN),
    (dict(key_cache=A + 4), kvq.KVQ_ERR_ALIGN),
    (dict(total_tokens=0, key_out=None, key_cache=None), kvq.KVQ_OK),
])
def test_load_validation(lib, kw, code):
    assert load(lib, **kw) == code


def istore(lib, **kw):
    args = dict(k=A, k_stride0=128, dtype=0, num_tokens=10, head_dim=128,
                kv_cache=A, block_stride=64 * 132, block_size=64,
                num_blocks=4, slot_mapping=A, flags=0, dev_error=None,
                stream=None)
    args.update(kw)
    return lib.kvq_store_indexer_k(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), kvq.KVQ_ERR_DTYPE),
    (dict(flags=1), kvq.KVQ_ERR_ARG),
    (dict(head_dim=96), kvq.KVQ_ERR_SHAPE),
    (dict(head_dim=512), kvq.KVQ_ERR_SHAPE),
    (dict(block_stride=64 * 131), kvq.KVQ_ERR_SHAPE),
    (dict(num_tokens=-2), kvq.KVQ_ERR_SHAPE),
    (dict(block_size=0), kvq.KVQ_ERR_SHAPE),
    (dict(k=None), kvq.KVQ_ERR_NULL),
    (dict(slot_mapping=None), kvq.KVQ_ERR_NULL),
    (dict(k=A + 8), kvq.KVQ_ERR_ALIGN),
    (dict(k_stride0=132), kvq.KVQ_ERR_ALIGN),
    (dict(block_stride=64 * 132 + 8), kvq.KVQ_ERR_ALIGN),
    (dict(slot_mapping=A + 4), kvq.KVQ_ERR_ALIGN),
    (dict(num_tokens=0, k=None), kvq.KVQ_OK),
])
def test_indexer_store_validation(lib, kw, code):
    assert istore(lib, **kw) == code


def attn(lib, **kw):
    args = dict(query=A, query_stride0=8 * 128, dtype=0, num_seqs=2,
                num_q_heads=8, num_kv_heads=1, head_size=128, key_cache=A,
                value_cache=A, page_stride=2 * 16 * 72, block_size=16,
                num_blocks=8, layout=0, block_table=A, block_table_stride=4,
                max_blocks_per_seq=4, context_lens=A, max_context_len=600,
                k_scale=A, v_scale=A, scale=0.088, partition_size=512,
                exp_sums=A, max_logits=A, tmp_out=A, out=A,
                out_stride0=8 * 128, flags=0, dev_error=None, stream=None)
    args.update(kw)
    return lib.kvq_paged_attention_nvfp4(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), kvq.KVQ_ERR_DTYPE),
    (dict(layout=2), kvq.KVQ_ERR_LAYOUT),
    (dict(flags=8), kvq.KVQ_ERR_ARG),
    (dict(flags=16), kvq.KVQ_ERR_ARG),
    (dict(scale=float("nan")), kvq.KVQ_ERR_ARG),
    (dict(scale=float("inf")), kvq.KVQ_ERR_ARG),
    (dict(head_size=64), kvq.KVQ_ERR_SHAPE),
    (dict(num_q_heads=6, num_kv_heads=4), kvq.KVQ_ERR_SHAPE),
    (dict(num_q_heads=17 * 2, num_kv_heads=2, query_stride0=34 * 128,
          out_stride0=34 * 128), kvq.KVQ_ERR_SHAPE),
    (dict(block_size=6), kvq.KVQ_ERR_SHAPE),
    (dict(partition_size=192), kvq.KVQ_ERR_SHAPE),
    (dict(partition_size=640), kvq.KVQ_ERR_SHAPE),
    (dict(page_stride=64), kvq.KVQ_ERR_SHAPE),
    (dict(query_stride0=4 * 128), kvq.KVQ_ERR_SHAPE),
    (dict(block_table_stride=2), kvq.KVQ_ERR_SHAPE),
    (dict(max_context_len=-1), kvq.KVQ_ERR_SHAPE),
    (dict(num_seqs=70000), kvq.KVQ_ERR_SHAPE),
    (dict(query=None), kvq.KVQ_ERR_NULL),
    (dict(tmp_out=None), kvq.KVQ_ERR_NULL),
    (dict(out=A + 8), kvq.KVQ_ERR_ALIGN),
    (dict(out_stride0=8 * 128 + 4), kvq.KVQ_ERR_ALIGN),
    (dict(key_cache=A + 4), kvq.KVQ_ERR_ALIGN),
    (dict(tmp_out=A + 4), kvq.KVQ_ERR_ALIGN),
    (dict(num_seqs=0, query=None, out=None), kvq.KVQ_OK),
])
def test_attention_validation(lib, kw, code):
    assert attn(lib, **kw) == code
