"""Failure detection on the GPU without a fault: a ring stage that is never
armed makes a bounded mbarrier wait run out; the kernel records
KVS_DEVERR_WAIT_TIMEOUT, lets its other copies land and stops, and the
context stays usable for the next call."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from shared_paged_kv_gb300 import kvs as K
from shared_paged_kv_gb300 import workloads as W
from oracle import attention as OA, fingerprint as OF
import harness as H

f32 = W.bf16_bits_to_f32


def test_wait_timeout_is_reported_and_the_context_survives():
    w = W.make_tiny()
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    pool = H.bf16_pool(w)
    q_bits = w.q_layer(0)
    K.kvs_pool_set_test_flags(pool, K.KVS_TEST_STALL_ONE_STAGE | K.KVS_TEST_TOKEN_MAJOR)
    t0 = time.time()
    H.attn(pool, 0, q_bits, w, ref["block_table"])
    dt = time.time() - t0
    flags = K.kvs_pool_check(pool)
    assert flags & K.KVS_DEVERR_WAIT_TIMEOUT
    assert dt < 30, "the bounded wait must end by itself"
    # the flag was consumed and the context still computes correctly
    got = H.attn(pool, 0, q_bits, w, ref["block_table"])
    hst = pool.host[0]
    exp = OA.decode_attention(f32(q_bits), f32(hst["k"]), f32(hst["v"]), ref["block_table"], w.seq_len,
                              w.block_tokens, w.scale, diff_table=w.diff_table, dk_pool=f32(hst["dk"]),
                              dv_pool=f32(hst["dv"]))
    H.assert_close_attn(got, exp)
    assert K.kvs_pool_check(pool) == 0
