"""CPU oracle for the shared paged KV hot path — TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 restatements of what the method computes, written from the
five source pages:

* INMS walkthrough — "大模型多Agent系统显存优化：KV Cache共享机制解析"
  (memory tiers, block fingerprint + refcount, prefix sharing, RoPE offset
  compensation; §1.2 accounting; §2.2, §3.2, §5.1),
* TokenDance news summary — "TokenDance: Scaling Multi-Agent LLM Serving via
  Collective KV Cache Sharing" (collective reuse, master/mirror diffs, fused
  restore; sections 1-3, Fig. 6-8),
* shared-memory KV pool post — "共享内存KV Cache池" (per-token KV formula
  §1.1, CalcHash §3.2, longest-prefix match §3.3),
* Q4 edge paper summary — "Agent Memory Below the Prompt: Persistent Q4 KV
  Cache for Multi-Agent LLM Inference on Edge Devices" (§2.1 block pool, Q4
  ratio; §2.2 attention directly on Q4),
* MemDecay post — "MemDecay: Region-Aware KV Cache Eviction" (§4.2 scaled
  dot-product with 1/sqrt(head_dim)).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA library and never imports it.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (page-printed worked values, closed forms,
invariants, brute force on tiny inputs).  Parity unpinned: none of the
functions; the only unpinned matter is the pairing convention of RoPE
(rotate-half), which the pages do not state at all — see the readings list in
the design notes.
"""
