"""The bulk-copy form of the indexer-K gather, a build option of the
library (KVQ_GATHER_BULK=1: one warp per (sequence, block of its table),
whose rows move cache -> shared memory -> k_fp8 by TMA bulk copies, the
scale bytes by one bulk load and 4-byte stores).  The default build keeps
the per-row 16-byte copy, which is faster back to back with early-read
PDL; this form is 3-8 % faster as a cold single launch.  Both must give the same bytes: the
gather parity cases (named workloads, sequence-length boundaries, wide
tables, flagged rows, early-read PDL) and the sharded-gather cases run here
again against a library built with the option."""
import pytest

from paged_quantized_kv_gb300 import build as kbuild
from paged_quantized_kv_gb300 import kvq
from tests import test_parity_gather as G
from tests import test_parity_shards as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bulk_lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("kvq_bulk") / "libkvq_gather_bulk.so")
    return kbuild.build(defines={"KVQ_GATHER_BULK": 1}, out=out)


@pytest.fixture(autouse=True)
def _use_bulk_library(bulk_lib, monkeypatch):
    monkeypatch.setattr(kvq, "LIB_PATH", bulk_lib)
    monkeypatch.setattr(kvq, "_lib", None)
    yield
    assert kvq.LIB_PATH == bulk_lib


test_named_workload = G.test_named_workload
test_case = G.test_case
test_total_beyond_cu_is_flagged = G.test_total_beyond_cu_is_flagged
test_bad_block_id_is_flagged = G.test_bad_block_id_is_flagged
test_gather_shards_union = S.test_gather_shards_union
