"""The no-allocation selection entry point against the workspace one.

Some callers cannot allocate device memory while they run (a server that has
given all free memory to its KV pool up front, a step that cannot take
cudaMalloc's implicit synchronisation, a C caller without a workspace), so
kvs_select_critical_noalloc keeps its scratch in a fixed device array inside
the library.  This file is collected last so that a run stopping at the first
failure has already run every other test; it passes alone and after them."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
import harness as H


def run_both(seed, rows, row_elems, ratio):
    kc, kn, off = W.selection_inputs(seed, len(rows), rows, row_elems)
    n, max_rows = len(rows), max(max(rows), 1)
    kc_d, kn_d, off_d = H.bits_to_dev(kc), H.bits_to_dev(kn), H.i64(off)
    total = int(off[-1]) + 1
    idx_a = torch.full((total,), -7, dtype=torch.int32, device=H.DEV)
    off_a = torch.zeros(n + 1, dtype=torch.int64, device=H.DEV)
    idx_b = torch.full((total,), -9, dtype=torch.int32, device=H.DEV)
    off_b = torch.zeros(n + 1, dtype=torch.int64, device=H.DEV)
    ws = H.workspace(4 * n * max_rows)
    K.kvs_select_critical(kc_d, kn_d, off_d, n, max_rows, row_elems, ratio, idx_a, off_a, ws)
    K.kvs_select_critical_noalloc(kc_d, kn_d, off_d, n, max_rows, row_elems, ratio, idx_b, off_b)
    torch.cuda.synchronize()
    oa, ob = off_a.cpu().numpy(), off_b.cpu().numpy()
    np.testing.assert_array_equal(oa, ob)
    m = int(oa[-1])
    np.testing.assert_array_equal(idx_a.cpu().numpy()[:m], idx_b.cpu().numpy()[:m])
    return m


def test_noalloc_matches_workspace_entry_on_two_calls():
    # two calls in a row with different shapes: the second must not see the
    # first call's leftovers in the shared scratch
    m1 = run_both(21, [700, 3, 0, 2048, 129], 1024, 0.15)
    m2 = run_both(22, [64, 1500, 9], 256, 0.3)
    assert m1 > 0 and m2 > 0


def test_noalloc_rejects_oversize():
    z = torch.zeros(16, dtype=torch.int16, device=H.DEV)
    off = torch.zeros(3, dtype=torch.int64, device=H.DEV)
    idx = torch.zeros(4, dtype=torch.int32, device=H.DEV)
    with pytest.raises(K.KvsError) as e:
        K.kvs_select_critical_noalloc(z, z, off, 2, 65536 // 2 * 2 * 8, 8, 0.1, idx, off)
    assert e.value.status in (K.KVS_ERR_CAPACITY, K.KVS_ERR_INVALID_ARG)
    with pytest.raises(K.KvsError) as e:
        K.kvs_select_critical_noalloc(z, z, off, 17, 65536, 8, 0.1, idx, off)
    assert e.value.status == K.KVS_ERR_CAPACITY
