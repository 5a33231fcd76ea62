"""The no-allocation selection entry point against the workspace one and the
oracle.

Some callers cannot allocate device memory while they run: a server that has
given all free memory to its KV pool and caching allocator up front (another
cudaMalloc would fail or fragment it), a step that cannot take cudaMalloc's
implicit synchronisation, or a C caller that does not want to own a
workspace.  kvs_select_critical_noalloc serves them from a fixed device array
inside the library.  This file is collected last so that a run stopping at the
first failure has already run every other test; it passes alone and after
them."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
import harness as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
    gb = idx_b.cpu().numpy()
    np.testing.assert_array_equal(idx_a.cpu().numpy()[:m], gb[:m])
    H.check_selection(kc, kn, off, ratio, gb[:m], ob)
    return m


def test_noalloc_matches_workspace_entry_on_two_calls():
    # two calls in a row with different shapes: the second must not see the
    # first call's leftovers in the shared scratch
    m1 = run_both(21, [700, 3, 0, 2048, 129], 1024, 0.15)
    m2 = run_both(22, [64, 1500, 9], 256, 0.3)
    assert m1 > 0 and m2 > 0


def test_noalloc_rejects_oversize():
    z = torch.zeros(16, dtype=torch.int16, device=H.DEV)
    off = torch.zeros(40, dtype=torch.int64, device=H.DEV)
    idx = torch.zeros(4, dtype=torch.int32, device=H.DEV)
    # within 65536 rows per agent, but 33 x 32768 rows exceed the 2^20 scratch
    with pytest.raises(K.KvsError) as e:
        K.kvs_select_critical_noalloc(z, z, off, 33, 32768, 8, 0.1, idx, off)
    assert e.value.status == K.KVS_ERR_CAPACITY
    with pytest.raises(K.KvsError) as e:
        K.kvs_select_critical_noalloc(z, z, off, 17, 65536, 8, 0.1, idx, off)
    assert e.value.status == K.KVS_ERR_CAPACITY
    # more than 65536 rows per agent is a bad size, whatever the total
    with pytest.raises(K.KvsError) as e:
        K.kvs_select_critical_noalloc(z, z, off, 1, 65537, 8, 0.1, idx, off)
    assert e.value.status == K.KVS_ERR_INVALID_ARG
    # exactly the scratch size is accepted (every agent empty: nothing read)
    ooff = torch.full((17,), -1, dtype=torch.int64, device=H.DEV)
    K.kvs_select_critical_noalloc(z, z, off, 16, 65536, 8, 0.1, idx, ooff)
    torch.cuda.synchronize()
    assert ooff.cpu().numpy().tolist() == [0] * 17


# Run in a fresh interpreter: the device is reset between two calls, which
# invalidates every allocation of the process, so the child uses plain cudart
# through ctypes (no torch allocations) and compares each call with the
# workspace entry point.
_RESET_CHILD = r"""
import ctypes, json, sys
import numpy as np
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
lib = K.load()
cudart = None
with open("/proc/self/maps") as f:
    for line in f:
        if "libcudart.so" in line:
            cudart = ctypes.CDLL(line.split()[-1])
            break
assert cudart is not None, "libcudart not mapped"
P = ctypes.c_void_p

def ck(e, what):
    assert e == 0, f"{what}: cuda error {e}"

def dev_copy(a):
    a = np.ascontiguousarray(a)
    p = P()
    ck(cudart.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(max(a.nbytes, 16))), "cudaMalloc")
    ck(cudart.cudaMemcpy(p, a.ctypes.data_as(P), ctypes.c_size_t(a.nbytes), 1), "H2D")
    return p

def host_copy(p, n, dt):
    a = np.zeros(n, dt)
    ck(cudart.cudaMemcpy(a.ctypes.data_as(P), p, ctypes.c_size_t(a.nbytes), 2), "D2H")
    return a

def one_round(seed):
    rows = [300, 5, 1024, 77]
    kc, kn, off = W.selection_inputs(seed, len(rows), rows, 512)
    n, mr = len(rows), max(rows)
    bufs = [dev_copy(kc), dev_copy(kn), dev_copy(off)]
    total = int(off[-1])
    res = []
    for noalloc in (False, True):
        idx = dev_copy(np.full(total, -3, np.int32))
        ioff = dev_copy(np.zeros(n + 1, np.int64))
        if noalloc:
            st = lib.kvs_select_critical_noalloc(bufs[0], bufs[1], bufs[2], n, mr, 512, ctypes.c_float(0.2), idx, ioff, None)
        else:
            ws = dev_copy(np.zeros(n * mr, np.float32))
            st = lib.kvs_select_critical(bufs[0], bufs[1], bufs[2], n, mr, 512, ctypes.c_float(0.2), idx, ioff, ws,
                                         ctypes.c_size_t(4 * n * mr), None)
        assert st == 0, lib.kvs_last_error_string()
        ck(cudart.cudaDeviceSynchronize(), "sync")
        o = host_copy(ioff, n + 1, np.int64)
        res.append((o.tolist(), host_copy(idx, total, np.int32)[: int(o[-1])].tolist()))
    assert res[0] == res[1], "noalloc differs from the workspace entry point"
    return res[1]

first = one_round(31)
ck(cudart.cudaDeviceSynchronize(), "sync")
ck(cudart.cudaDeviceReset(), "cudaDeviceReset")
second = one_round(32)
print(json.dumps({"ok": True, "first": first[0], "second": second[0], "second_idx": second[1]}))
"""


def test_noalloc_after_device_reset():
    code = "ROOT = %r\n" % ROOT + _RESET_CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["ok"]
    # the call after the reset is also right against the oracle
    rows = [300, 5, 1024, 77]
    kc, kn, off = W.selection_inputs(32, len(rows), rows, 512)
    H.check_selection(kc, kn, off, 0.2, np.array(res["second_idx"], np.int32), np.array(res["second"], np.int64))
