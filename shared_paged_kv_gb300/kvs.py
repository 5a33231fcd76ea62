"""Thin ctypes binding of libkvs (the C ABI in include/kvs.h).

Argument marshalling only: torch tensors become raw device pointers, the
current torch CUDA stream becomes the cudaStream_t, and a non-OK status raises
KvsError with the library's error string.  Every step of the hot path runs in
the library's CUDA kernels; there is no fallback when the library is missing —
loading fails loudly.
"""
from __future__ import annotations

import ctypes

import numpy as np
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvs.so")

KVS_OK = 0
KVS_ERR_INVALID_ARG = 1
KVS_ERR_CAPACITY = 2
KVS_ERR_CUDA = 3
KVS_ERR_DEVICE_BOUNDS = 4
KVS_ERR_UNSUPPORTED = 5

KVS_DEVERR_BLOCK_ID = 0x1
KVS_DEVERR_SEQ_LEN = 0x2
KVS_DEVERR_CAPACITY = 0x4
KVS_DEVERR_DIFF_ID = 0x8
KVS_DEVERR_WAIT_TIMEOUT = 0x10
KVS_DEVERR_ROPE_RANGE = 0x20
KVS_DEVERR_JOB = 0x40
KVS_DEVERR_PLAN = 0x80
KVS_DEVERR_REFCOUNT = 0x100
KVS_TEST_STALL_ONE_STAGE = 0x1
KVS_TEST_TOKEN_MAJOR = 0x2

KVS_DTYPE_BF16 = 0
KVS_DTYPE_Q4G64 = 1
KVS_DEDUP_TEST_WEAK_KEYS = 0x1
KVS_OP_DEDUP, KVS_OP_DECODE_ATTN, KVS_OP_DECODE_ATTN_Q4, KVS_OP_SELECT, KVS_OP_MIRROR, KVS_OP_BLOCKS = 0, 1, 2, 3, 4, 5

EXPORTED = [
    "kvs_pool_create", "kvs_pool_destroy", "kvs_fingerprint_dedup", "kvs_rope_rerotate",
    "kvs_select_critical", "kvs_select_critical_noalloc", "kvs_decode_plan", "kvs_decode_attn_planned",
    "kvs_decode_attn", "kvs_decode_attn_q4", "kvs_quantize_q4", "kvs_mirror_build",
    "kvs_blocks_init_free", "kvs_block_write", "kvs_seq_release", "kvs_evict_score",
    "kvs_pool_block_bytes", "kvs_pool_export", "kvs_pool_import", "kvs_pool_set_test_flags",
    "kvs_workspace_size", "kvs_pool_check", "kvs_pool_stats", "kvs_last_error_string",
    "kvs_launch_count",
]


class KvsError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kvs status {status}: {msg}")
        self.status = status


class PoolDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "num_kv_heads", "head_dim", "block_tokens", "dtype",
        "capacity_blocks", "diff_capacity_blocks", "max_seqs")]


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "unique_blocks", "shared_blocks", "total_refs", "pool_bytes", "dense_bytes")]


_lib = None


def load(path: str = LIB_PATH):
    """Load libkvs.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkvs.so not found at {path}; run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P, I32, I64, U32, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t)
    sigs = {
        "kvs_pool_create": [ctypes.POINTER(PoolDesc), P, P, P, P, P, P, ctypes.POINTER(P)],
        "kvs_pool_destroy": [P],
        "kvs_fingerprint_dedup": [P, P, P, I32, P, P, P, P, P, I32, P, P, P, P, P, U32, P, SZ, P],
        "kvs_rope_rerotate": [P, I32, P, I32, I32, F32, P, P, I32, P],
        "kvs_select_critical": [P, P, P, I32, I32, I32, F32, P, P, P, SZ, P],
        "kvs_select_critical_noalloc": [P, P, P, I32, I32, I32, F32, P, P, P],
        "kvs_mirror_build": [P, I32, P, I32, P, I32, P, P, P, P, P, P, F32, P, P, P, SZ, P],
        "kvs_blocks_init_free": [P, P, P, P, P, SZ, P],
        "kvs_block_write": [P, P, I32, I32, P, P, I32, P, P, P, P, SZ, P],
        "kvs_seq_release": [P, P, I32, P, I32, P, I32, P, P, P, P, SZ, P],
        "kvs_evict_score": [P, P, P, P, P, I32, I32, P, P, I32, I64, P, P, P, P, P],
        "kvs_pool_block_bytes": [P, ctypes.POINTER(SZ)],
        "kvs_pool_set_test_flags": [P, U32],
        "kvs_pool_export": [P, P, I32, P, SZ, P],
        "kvs_pool_import": [P, P, I32, P, SZ, P],
        "kvs_decode_attn": [P, I32, P, I32, P, I32, P, I32, P, P, P, F32, F32, P, P, SZ, P],
        "kvs_decode_attn_planned": [P, I32, P, I32, P, I32, P, I32, P, P, P, F32, F32, P, P, SZ, P],
        "kvs_decode_plan": [P, I32, P, I32, P, I32, P, P, P, P, SZ, P],
        "kvs_decode_attn_q4": [P, I32, P, I32, P, I32, P, I32, P, F32, P, P, SZ, P],
        "kvs_quantize_q4": [P, I32, P, P, P, I32, P],
        "kvs_workspace_size": [P, I32, I32, I32, I32, ctypes.POINTER(SZ)],
        "kvs_pool_check": [P, P, ctypes.POINTER(U32)],
        "kvs_pool_stats": [P, P, P, P, ctypes.POINTER(Stats)],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.kvs_last_error_string.argtypes = []
    lib.kvs_last_error_string.restype = ctypes.c_char_p
    lib.kvs_launch_count.argtypes = []
    lib.kvs_launch_count.restype = ctypes.c_uint64
    _lib = lib
    return lib


def _check(st: int):
    if st != KVS_OK:
        raise KvsError(st, load().kvs_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    # a plain int: ctypes passes it as the void* argument without a wrapper
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libkvs must be contiguous")
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_dev = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream=None):
    """The cudaStream_t of `stream`, or of torch's current stream on the
    current device (read without building a Stream object)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and _cur_dev is not None:
        return _raw_stream(_cur_dev())
    return torch.cuda.current_stream().cuda_stream


def _ptr_array(ts: Optional[Sequence[torch.Tensor]]):
    if ts is None:
        return None
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return arr


class Pool:
    """Owns a kvs_pool handle and keeps the slab tensors alive."""

    def __init__(self, handle, desc: PoolDesc, keep):
        self.handle = handle
        self.desc = desc
        self._keep = keep

    def __del__(self):
        try:
            if self.handle:
                kvs_pool_destroy(self)
        except Exception:
            pass


def kvs_pool_create(num_layers, num_kv_heads, head_dim, block_tokens, dtype, capacity_blocks,
                    max_seqs, k_layers, v_layers, k_sb_layers=None, v_sb_layers=None,
                    dk_layers=None, dv_layers=None, diff_capacity_blocks=0) -> Pool:
    lib = load()
    d = PoolDesc(num_layers, num_kv_heads, head_dim, block_tokens, dtype, capacity_blocks,
                 diff_capacity_blocks, max_seqs)
    arrs = [_ptr_array(x) for x in (k_layers, v_layers, k_sb_layers, v_sb_layers, dk_layers, dv_layers)]
    h = ctypes.c_void_p()
    _check(lib.kvs_pool_create(ctypes.byref(d), *arrs, ctypes.byref(h)))
    keep = [k_layers, v_layers, k_sb_layers, v_sb_layers, dk_layers, dv_layers]
    return Pool(h, d, keep)


def kvs_pool_destroy(pool: Pool):
    if pool.handle:
        _check(load().kvs_pool_destroy(pool.handle))
        pool.handle = None


def kvs_workspace_size(pool: Pool, op: int, n_seq: int, max_blocks: int, n_q_heads: int = 0) -> int:
    out = ctypes.c_size_t()
    _check(load().kvs_workspace_size(pool.handle, op, n_seq, max_blocks, n_q_heads, ctypes.byref(out)))
    return out.value


def kvs_fingerprint_dedup(pool: Pool, tokens, seq_off, n_seq, tier, seg_off, seg_blocks, fp_out,
                          block_table, max_blocks, refcount, n_phys, ws, flags=0, stream=None,
                          owner_seq=None, ref_off=None, ref_seq=None):
    """Fingerprints, block table, refcounts and n_phys; optionally the owner
    sequence of every physical block and the CSR of its references."""
    _check(load().kvs_fingerprint_dedup(
        pool.handle, _ptr(tokens), _ptr(seq_off), n_seq, _ptr(tier), _ptr(seg_off), _ptr(seg_blocks),
        _ptr(fp_out), _ptr(block_table), max_blocks, _ptr(refcount), _ptr(n_phys), _ptr(owner_seq),
        _ptr(ref_off), _ptr(ref_seq), flags, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def kvs_rope_rerotate(pool: Pool, layer, jobs, n_jobs, max_job_tokens, theta, src_table, dst_table,
                      max_blocks, stream=None):
    _check(load().kvs_rope_rerotate(pool.handle, layer, _ptr(jobs), n_jobs, max_job_tokens, theta,
                                    _ptr(src_table), _ptr(dst_table), max_blocks, _stream(stream)))


def kvs_select_critical(k_cached, k_new, row_off, n_agents, max_rows_per_agent, row_elems, ratio,
                        idx_out, idx_off, ws, stream=None):
    _check(load().kvs_select_critical(_ptr(k_cached), _ptr(k_new), _ptr(row_off), n_agents,
                                      max_rows_per_agent, row_elems, ratio, _ptr(idx_out), _ptr(idx_off),
                                      _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def kvs_mirror_build(pool: Pool, layer, block_table, max_blocks, seq_len, n_seq, idx, idx_off, k_new, v_new,
                     rope_off, rope_segs, theta, diff_table, n_diff, ws, stream=None):
    """Diff table and block-sparse diff tiles (written into the pool's diff
    slabs of `layer`) of every agent's refreshed positions against its master
    blocks; n_diff (device int32 [1]) receives the number of diff blocks."""
    _check(load().kvs_mirror_build(pool.handle, layer, _ptr(block_table), max_blocks, _ptr(seq_len), n_seq, _ptr(idx),
                                   _ptr(idx_off), _ptr(k_new), _ptr(v_new), _ptr(rope_off), _ptr(rope_segs), theta,
                                   _ptr(diff_table), _ptr(n_diff), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)))


def kvs_blocks_init_free(pool: Pool, refcount, free_ids, n_free, ws, stream=None):
    """Free stack = every block whose reference count is 0 (smallest id on top)."""
    _check(load().kvs_blocks_init_free(pool.handle, _ptr(refcount), _ptr(free_ids), _ptr(n_free), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)))


def kvs_block_write(pool: Pool, block_table, max_blocks, n_seq, write_seq, write_block, n_writes, refcount,
                    free_ids, n_free, ws, stream=None):
    """Copy-on-write for a batch of block writes, applied in list order."""
    _check(load().kvs_block_write(pool.handle, _ptr(block_table), max_blocks, n_seq, _ptr(write_seq),
                                  _ptr(write_block), n_writes, _ptr(refcount), _ptr(free_ids), _ptr(n_free), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)))


def kvs_seq_release(pool: Pool, block_table, max_blocks, seq_len, n_seq, release_seq, n_release, refcount,
                    free_ids, n_free, ws, stream=None):
    """Destroy sequences: decrement their blocks' counts, reclaim the zeros."""
    _check(load().kvs_seq_release(pool.handle, _ptr(block_table), max_blocks, _ptr(seq_len), n_seq,
                                  _ptr(release_seq), n_release, _ptr(refcount), _ptr(free_ids), _ptr(n_free),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def kvs_evict_score(pool: Pool, region, created, access, seq_len, n_seq, max_blocks, init, decay, step, k, scores,
                    victims, victims_off, stream=None):
    """Block scores and per-sequence lowest-scored victim blocks.  init and
    decay are host sequences of floats (one per region)."""
    init_a = np.ascontiguousarray(init, dtype=np.float32)
    decay_a = np.ascontiguousarray(decay, dtype=np.float32)
    _check(load().kvs_evict_score(pool.handle, _ptr(region), _ptr(created), _ptr(access), _ptr(seq_len), n_seq,
                                  max_blocks, init_a.ctypes.data, decay_a.ctypes.data, len(init_a), int(step), _ptr(k),
                                  _ptr(scores), _ptr(victims), _ptr(victims_off), _stream(stream)))


def kvs_pool_block_bytes(pool: Pool) -> int:
    """Bytes of one packed block record (every layer's slabs)."""
    b = ctypes.c_size_t(0)
    _check(load().kvs_pool_block_bytes(pool.handle, ctypes.byref(b)))
    return b.value


def kvs_pool_export(pool: Pool, blocks, n_blocks, dst, stream=None):
    """Pack the listed physical blocks (all layers) into dst, in list order."""
    _check(load().kvs_pool_export(pool.handle, _ptr(blocks), n_blocks, _ptr(dst), dst.numel() * dst.element_size(),
                                  _stream(stream)))


def kvs_pool_import(pool: Pool, blocks, n_blocks, src, stream=None):
    """Unpack records from src into the listed physical blocks."""
    _check(load().kvs_pool_import(pool.handle, _ptr(blocks), n_blocks, _ptr(src), src.numel() * src.element_size(),
                                  _stream(stream)))


def kvs_pool_set_test_flags(pool: Pool, flags: int):
    """Test-only switches (KVS_TEST_*); see include/kvs.h."""
    _check(load().kvs_pool_set_test_flags(pool.handle, flags))


def kvs_select_critical_noalloc(k_cached, k_new, row_off, n_agents, max_rows_per_agent, row_elems, ratio,
                                idx_out, idx_off, stream=None):
    """kvs_select_critical without a workspace argument: the library's fixed
    device scratch (2^20 rows) is used instead; nothing is allocated."""
    _check(load().kvs_select_critical_noalloc(_ptr(k_cached), _ptr(k_new), _ptr(row_off), n_agents,
                                              max_rows_per_agent, row_elems, ratio, _ptr(idx_out), _ptr(idx_off),
                                              _stream(stream)))


def kvs_decode_attn(pool: Pool, layer, q, n_q_heads, block_table, max_blocks, seq_len, n_seq,
                    diff_table, rope_off, rope_segs, theta, scale, out, ws, stream=None):
    _check(load().kvs_decode_attn(pool.handle, layer, _ptr(q), n_q_heads, _ptr(block_table), max_blocks,
                                  _ptr(seq_len), n_seq, _ptr(diff_table), _ptr(rope_off), _ptr(rope_segs),
                                  theta, scale, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)))


def kvs_decode_plan(pool: Pool, n_q_heads, block_table, max_blocks, seq_len, n_seq, diff_table, rope_off,
                    rope_segs, ws, stream=None):
    _check(load().kvs_decode_plan(pool.handle, n_q_heads, _ptr(block_table), max_blocks, _ptr(seq_len), n_seq,
                                  _ptr(diff_table), _ptr(rope_off), _ptr(rope_segs), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)))


def kvs_decode_attn_planned(pool: Pool, layer, q, n_q_heads, block_table, max_blocks, seq_len, n_seq,
                            diff_table, rope_off, rope_segs, theta, scale, out, ws, stream=None):
    _check(load().kvs_decode_attn_planned(pool.handle, layer, _ptr(q), n_q_heads, _ptr(block_table), max_blocks,
                                          _ptr(seq_len), n_seq, _ptr(diff_table), _ptr(rope_off), _ptr(rope_segs),
                                          theta, scale, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(stream)))


def kvs_decode_attn_q4(pool: Pool, layer, q, n_q_heads, block_table, max_blocks, seq_len, n_seq,
                       scale, out, ws, stream=None, diff_table=None):
    """Q4 decode attention; diff_table (int32 [n_seq][max_blocks * 16]) adds
    the pool's per-16-token mirror diffs."""
    _check(load().kvs_decode_attn_q4(pool.handle, layer, _ptr(q), n_q_heads, _ptr(block_table), max_blocks,
                                     _ptr(seq_len), n_seq, _ptr(diff_table), scale, _ptr(out), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)))


def kvs_quantize_q4(pool: Pool, layer, k_src, v_src, dst_blocks, n_blocks, stream=None):
    _check(load().kvs_quantize_q4(pool.handle, layer, _ptr(k_src), _ptr(v_src), _ptr(dst_blocks),
                                  n_blocks, _stream(stream)))


def kvs_pool_check(pool: Pool, stream=None) -> int:
    """Returns the device error bits (0 = clean); synchronises the stream."""
    flags = ctypes.c_uint32()
    st = load().kvs_pool_check(pool.handle, _stream(stream), ctypes.byref(flags))
    if st not in (KVS_OK, KVS_ERR_DEVICE_BOUNDS):
        _check(st)
    return flags.value


def kvs_pool_stats(pool: Pool, refcount, n_phys, stream=None) -> dict:
    s = Stats()
    _check(load().kvs_pool_stats(pool.handle, _ptr(refcount), _ptr(n_phys), _stream(stream), ctypes.byref(s)))
    return {n: getattr(s, n) for n, _ in Stats._fields_}


def kvs_last_error_string() -> str:
    return load().kvs_last_error_string().decode()


def kvs_launch_count() -> int:
    return int(load().kvs_launch_count())
