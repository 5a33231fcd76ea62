"""Benchmark of the shared paged KV decode step on GB300.

Headline workload (the configuration the metric is quoted on): 8 agents x
16384-token contexts, 32 query heads = 32 KV heads, head_dim 128, 16-token
blocks, 60 % common prefix stored once (614 shared + 8 x 410 private blocks
per layer), 32 layers, bf16 values ~N(0,1), one decode query per agent.

One step = the whole hot path on that batch: GPU block fingerprints + dedup
of the 8 token sequences (block tables, refcounts), one work plan, then
decode attention on all 32 layers through the deduplicated pool.  value =
decode tokens/s = agents / step time, timed with two CUDA events around the
K steps (no events inside them).  KV of one step is 32.7 GB, far above L2, so
no flush is needed between steps.  The per-layer attention time of the
roofline comes from a separate breakdown pass of the same steps with events
around every layer.

Also reported on the same line: KV GB/s, the attention kernel's roofline
(algorithmic bytes per launch / average launch time vs the measured HBM
peak), the end-to-end rate through the public API with pinned host buffers,
the CPU oracle on every host core over a bounded sample of the workload, and
one key per other synthetic workload (tiny, tiny x 4096, GQA fan-out,
all-gather round, Q4, selection, mirror build, RoPE re-rotation), each with
eager and CUDA-graph-replayed times, algorithmic bytes per launch and the
fraction of the measured HBM peak.

Multi-GPU: the path partitions by agent with no exchange, so N ranks each run
the full workload on their own agents (weak scaling, no collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode-attn tokens/s & KV GB/s vs GB300 HBM roofline; RoPE-reuse tokens/s"
UNIT = "tokens/s"
WORKLOAD = ("mha7b: 8 agents x 16384-token context, 60% shared prefix (614 shared + 8x410 private "
            "16-token blocks), 32 q heads = 32 kv heads, head_dim 128, bf16, 32 layers, 1 decode token per agent")
EXTRA_CONFIGS = ["tiny", "gqa_fanout", "allgather", "q4", "q4_mirror", "select", "mirror"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rope", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--extra-steps", type=int, default=10, help="timed steps of each extra workload")
    ap.add_argument("--layers", type=int, default=None, help="layers (default: the workload's own)")
    ap.add_argument("--workload", default="mha7b",
                    choices=["mha7b"] + EXTRA_CONFIGS + ["cow", "evict", "io"],
                    help="mha7b is the headline workload; the others print one record")
    ap.add_argument("--trace", action="store_true",
                    help="with --workload: add the kernels' start/end times of one CUDA-graph replay "
                         "(torch.profiler CUDA activity trace) to the record")
    ap.add_argument("--cpu-oracle", nargs=3, type=int, metavar=("LAYERS", "REPS", "PAIRS"),
                    help=argparse.SUPPRESS)
    return ap.parse_args()


# ----------------------------------------------------------- multi-rank ----
def rank_agents(n_per_rank: int, world: int, rank: int):
    """Global agent ids of this rank's replica: ranks hold disjoint,
    contiguous blocks of n_per_rank agents (weak scaling, no collective on
    the data path)."""
    if not 0 <= rank < world:
        raise ValueError("rank outside the world")
    return range(rank * n_per_rank, (rank + 1) * n_per_rank)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The job's time is the slowest rank's: an all-reduce MAX when world > 1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(n_per_rank: int, world: int, ms_step_max: float) -> float:
    """Whole-job decode tokens/s: every rank's agents over the slowest rank's step."""
    return world * n_per_rank / (ms_step_max * 1e-3)


# --------------------------------------------------------------- helpers ----
def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


ATTN_SOURCES = ["shared_paged_kv_gb300/csrc/attn_tm.cu", "shared_paged_kv_gb300/csrc/common.cuh"]
ATTN_KERNEL = "attn_tm_kernel<128,false,false>"


def profiled_traffic(kernel_src_hash):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "attn_bf16_mha7b.md")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_src_hash:
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(", ") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------- CPU oracle -----
# The oracle as it stands, on the host cores: the dedup of all 8 sequences
# (a sequential scan, one core) plus (agent, head) attention pairs of one
# layer (dense materialisation + fp64 attention) spread over a spawn pool of
# every usable core, then scaled to a full step of 8 agents x 32 heads x the
# step's layers.  The same sample serves the cpu_baseline key and the
# reference arm.
_ORACLE = {}


def _oracle_init(seed):
    """Worker start: the dedup result and one set of K/V values of one head
    (the oracle's cost does not depend on the values)."""
    from shared_paged_kv_gb300 import workloads as W
    from oracle import fingerprint as OF
    w = W.make_mha7b(n_layers=1)
    ref = OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
    rng = np.random.default_rng(seed)
    cap = ref["n_phys"]
    _ORACLE.update(w=w, table=ref["block_table"],
                   k=rng.standard_normal((cap, 1, 16, 128)).astype(np.float32),
                   v=rng.standard_normal((cap, 1, 16, 128)).astype(np.float32),
                   q=rng.standard_normal((1, 1, 128)).astype(np.float32))


def _oracle_warm(_):
    time.sleep(0.05)
    return len(_ORACLE)


def _oracle_pair(a):
    from oracle import attention as OA
    o = _ORACLE
    w = o["w"]
    OA.decode_attention(o["q"], o["k"], o["v"], o["table"][a:a + 1], w.seq_len[a:a + 1], 16, w.scale)
    return a


def host_cores() -> int:
    if hasattr(os, "sched_getaffinity"):
        return len(os.sched_getaffinity(0))
    return os.cpu_count() or 1


def cpu_oracle_run(layers: int, reps: int, n_pairs: int) -> dict:
    """Runs in its own interpreter (bench.py --cpu-oracle): returns the cores
    used and, per rep, the extrapolated seconds of one full step."""
    import multiprocessing as mp
    from shared_paged_kv_gb300 import workloads as W
    from oracle import fingerprint as OF
    cores = host_cores()
    w = W.make_mha7b(n_layers=1)
    agents = [p % 8 for p in range(n_pairs)]
    total_pairs = 8 * 32 * layers
    steps, dedup_s, pairs_s = [], [], []
    with mp.get_context("spawn").Pool(cores, initializer=_oracle_init, initargs=(0,)) as pool:
        pool.map(_oracle_warm, range(4 * cores), chunksize=1)
        for _ in range(reps):
            t0 = time.perf_counter()
            OF.dedup(w.tokens, w.seq_off, w.tier, w.block_tokens, w.max_blocks)
            t1 = time.perf_counter()
            pool.map(_oracle_pair, agents, chunksize=1)
            t2 = time.perf_counter()
            dedup_s.append(t1 - t0)
            pairs_s.append(t2 - t1)
            steps.append((t1 - t0) + (t2 - t1) * total_pairs / n_pairs)
    return {"cores": cores, "steps": steps, "dedup_s": dedup_s, "pairs_wall_s": pairs_s, "n_pairs": n_pairs,
            "scale": total_pairs / n_pairs}


def cpu_oracle(layers: int, reps: int) -> dict:
    """The oracle timing in a fresh interpreter (BLAS pinned to one thread per
    worker process); 4 pairs per core per rep."""
    n_pairs = 4 * host_cores()
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-oracle", str(layers), str(reps),
                        str(n_pairs)], capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_sample_text(res: dict, layers: int) -> str:
    return (f"per step: oracle dedup of all 8 sequences (one core, {statistics.median(res['dedup_s']):.3f} s) + "
            f"{res['n_pairs']} (agent, head) pairs of one mha7b layer through the fp64 oracle (dense materialise "
            f"+ attention) on a spawn pool of {res['cores']} processes "
            f"({statistics.median(res['pairs_wall_s']):.3f} s wall), the pairs' time scaled by "
            f"{res['scale']:.0f} to a full step of 8 agents x 32 heads x {layers} layers")


# ------------------------------------------------------------------ main ----
def main():
    args = parse()
    if args.cpu_oracle:
        layers, reps, n_pairs = args.cpu_oracle
        print(json.dumps(cpu_oracle_run(layers, reps, n_pairs)))
        return 0
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the CPU oracle as it stands, on the host cores; rank 0 only
        if rank != 0:
            return 0
        L = args.layers or 32
        res = cpu_oracle(L, args.warmup + args.steps)
        timed = res["steps"][args.warmup:]
        step_s = sum(timed) / len(timed)
        val = 8.0 / step_s
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": WORKLOAD, "agents": 8, "context": 16384, "layers": L},
                "cpu_baseline": {"kind": "oracle", "value": val, "unit": UNIT, "cores": res["cores"],
                                 "sample": cpu_sample_text(res, L)},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "ms_per_step_from": "extrapolated: the measured sample of each step (sample_ms_per_step) with its "
                                    "attention pairs scaled by sample_scale to a full step",
                "sample_ms_per_step": 1e3 * (sum(res["dedup_s"][args.warmup:]) +
                                             sum(res["pairs_wall_s"][args.warmup:])) / args.steps,
                "sample_scale": res["scale"]}
        print(json.dumps(line))
        return 0

    import torch
    import torch.distributed as dist
    import __graft_entry__ as G
    G.build()
    from shared_paged_kv_gb300 import kvs as K
    from shared_paged_kv_gb300 import workloads as W

    if args.workload != "mha7b" or args.trace:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        rec = run_extra(args.workload, torch, K, W, dev, args.steps, args.warmup, args.layers, trace=args.trace)
        print(json.dumps(rec))
        return 0

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    # ---- workload, resident in HBM
    L = args.layers or 32
    w = W.make_mha7b(n_layers=L)
    B, D, H, N = w.block_tokens, w.head_dim, w.n_kv_heads, w.n_seq
    cap = 614 + N * 410                       # physical blocks the dedup produces
    gen = torch.Generator(device=dev).manual_seed(1000 + rank)
    k_slabs = [torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16) for _ in range(L)]
    v_slabs = [torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16) for _ in range(L)]
    pool = K.kvs_pool_create(L, H, D, B, K.KVS_DTYPE_BF16, cap, N, [t.view(torch.int16) for t in k_slabs],
                             [t.view(torch.int16) for t in v_slabs])
    q = torch.randn((L, N, w.n_q_heads, D), generator=gen, device=dev, dtype=torch.bfloat16)
    tokens = torch.from_numpy(w.tokens.view(np.int32)).to(dev)
    seq_off = torch.from_numpy(w.seq_off).to(dev)
    seq_len = torch.from_numpy(w.seq_len).to(dev)
    fp = torch.zeros((N, w.max_blocks), dtype=torch.int64, device=dev)
    table = torch.zeros((N, w.max_blocks), dtype=torch.int32, device=dev)
    refc = torch.zeros(cap, dtype=torch.int32, device=dev)
    nphys = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_d = torch.zeros(K.kvs_workspace_size(pool, K.KVS_OP_DEDUP, N, w.max_blocks), dtype=torch.uint8, device=dev)
    ws_a = torch.zeros(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN, N, w.max_blocks, w.n_q_heads),
                       dtype=torch.uint8, device=dev)
    out = torch.zeros((L, N, w.n_q_heads, D), dtype=torch.float32, device=dev)

    def step(ev=None):
        # block tables change per step: fingerprint + dedup, then one work
        # plan for all layers, then attention on every layer
        K.kvs_fingerprint_dedup(pool, tokens, seq_off, N, None, None, None, fp, table, w.max_blocks, refc,
                                nphys, ws_d)
        K.kvs_decode_plan(pool, w.n_q_heads, table, w.max_blocks, seq_len, N, None, None, None, ws_a)
        for l in range(L):
            if ev is not None:
                ev[l][0].record(stream)
            K.kvs_decode_attn_planned(pool, l, q[l], w.n_q_heads, table, w.max_blocks, seq_len, N, None, None,
                                      None, w.theta, w.scale, out[l], ws_a)
            if ev is not None:
                ev[l][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags = K.kvs_pool_check(pool)
    if flags:
        raise RuntimeError(f"device status flags {flags:#x}")
    assert int(nphys.item()) == cap, (int(nphys.item()), cap)

    # ---- timed region: K steps between two events, nothing else recorded
    launches0 = K.kvs_launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = K.kvs_launch_count() - launches0
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_step = ms / args.steps
    value = job_tokens_per_s(N, world, ms_step)

    # ---- breakdown pass (outside the timed region): the same steps with an
    # event pair around every layer's attention call
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
          for _ in range(args.steps)]
    for i in range(args.steps):
        step([e for e in ev[i]])
    torch.cuda.synchronize()
    attn_ms = [a.elapsed_time(b) for row in ev for a, b in row]
    attn_avg_ms = sum(attn_ms) / len(attn_ms)

    # ---- algorithmic bytes of one attention launch (unique bytes leaving HBM)
    kv_bytes = cap * H * B * D * 2 * 2
    attn_bytes = kv_bytes + N * w.n_q_heads * D * 2 + N * w.max_blocks * 4 + N * 4 + N * w.n_q_heads * D * 4
    peak, peak_kind = read_peaks()
    achieved = attn_bytes / (attn_avg_ms * 1e-3) / 1e9
    step_bytes = L * attn_bytes + w.tokens.nbytes + N * w.max_blocks * (8 + 4)

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        h_tok = torch.from_numpy(w.tokens.view(np.int32)).pin_memory()
        h_off = torch.from_numpy(w.seq_off).pin_memory()
        h_q = q.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        d_tok, d_off, d_q = torch.empty_like(tokens), torch.empty_like(seq_off), torch.empty_like(q)

        def e2e_step():
            d_tok.copy_(h_tok, non_blocking=True)
            d_off.copy_(h_off, non_blocking=True)
            d_q.copy_(h_q, non_blocking=True)
            K.kvs_fingerprint_dedup(pool, d_tok, d_off, N, None, None, None, fp, table, w.max_blocks, refc,
                                    nphys, ws_d)
            K.kvs_decode_plan(pool, w.n_q_heads, table, w.max_blocks, seq_len, N, None, None, None, ws_a)
            for l in range(L):
                K.kvs_decode_attn_planned(pool, l, d_q[l], w.n_q_heads, table, w.max_blocks, seq_len, N, None,
                                          None, None, w.theta, w.scale, out[l], ws_a)
            h_out.copy_(out, non_blocking=True)
            torch.cuda.synchronize()

        for _ in range(2):
            e2e_step()
        if world > 1:
            dist.barrier()
        t_a = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        e2e_s = max_over_ranks((time.perf_counter() - t_a) / args.steps, world, dev)
        e2e = {"value": job_tokens_per_s(N, world, e2e_s * 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h_tok.numel() * 4 + h_off.numel() * 8 + h_q.numel() * 2),
               "d2h_bytes_per_step": int(h_out.numel() * 4)}
        del h_tok, h_off, h_q, h_out, d_tok, d_off, d_q
    flags |= K.kvs_pool_check(pool)
    del k_slabs, v_slabs, pool, q, out, ws_a, ws_d
    torch.cuda.empty_cache()

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "agents": N, "context": 16384, "layers": L,
                       "l2": "inputs larger than L2 (32.7 GB of unique KV per step), no flush",
                       "parallelism": f"replicas x{world} (agents partitioned, no collective)"},
            "kv_gbs": world * step_bytes / (ms_step * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(source_hash(ATTN_SOURCES)),
                         "kernel": ATTN_KERNEL, "peak_kind": peak_kind,
                         "bytes_per_launch": attn_bytes, "avg_launch_ms": attn_avg_ms,
                         "avg_launch_from": "breakdown pass after the timed region: the same steps with events "
                                            "around every layer's attention call"},
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "status_flags": flags,
        }

    # ---- RoPE re-rotation on one layer of the all-gather round
    if not args.no_rope and line is not None:
        line["rope_reuse"] = bench_rope(torch, K, W, dev, stream, args, peak)

    # ---- every other workload, one key each (one GPU only)
    if not args.no_extra and world == 1:
        for name in EXTRA_CONFIGS:
            try:
                line[name] = run_extra(name, torch, K, W, dev, args.extra_steps, min(args.warmup, 3), None)
            except Exception as ex:  # keep the headline line; record what failed
                line[name] = {"error": f"{type(ex).__name__}: {ex}"[:500]}
            torch.cuda.empty_cache()

    # ---- CPU oracle (rank 0, after all GPU work)
    if not args.no_cpu_baseline and rank == 0:
        res = cpu_oracle(L, 3)
        step_s = statistics.median(res["steps"])
        line["cpu_baseline"] = {"value": N / step_s, "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                                "sample": cpu_sample_text(res, L)}

    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------- other workloads --
# name -> (dominant kernels, committed ncu summary, workload description)
CONFIG_INFO = {
    "mha7b": ("attn_tm_kernel<128,0,0>, then tm_merge_kernel<128>", "profiles/attn_bf16_mha7b.md", WORKLOAD),
    "tiny": ("attn_bf16_kernel<64,1,0,8> (small-call path: one launch of 8-warp CTAs, latency-bound)",
             "profiles/attn_bf16_tiny.md",
             "tiny: 4 agents, 1 layer, 8 q / 2 kv heads, d 64, 256-token shared prefix + 64-128 private, "
             "2 mirror-diff blocks per agent"),
    "gqa_fanout": ("attn_wide_kernel<1,0> beside attn_tm_kernel<128,0,0>, then tm_merge_kernel<128>",
                   "profiles/launches_gqa_step.md",
                   "gqa_fanout: 32 sequences, 4096-token shared system prefix + 512-2048 private, 16 q / 2 kv heads, "
                   "d 128, 28 layers"),
    "allgather": ("attn_tm_kernel<128,1,1> beside attn_wide_kernel<2,1>, then tm_merge_kernel<128>",
                  "profiles/launches_allgather_step.md",
                  "allgather: 64 agents, private 1k-6k + 64 shared 128-token segments per agent with RoPE shifts "
                  "(theta 1e6), 31 mirror-diff blocks per agent, 40 q / 8 kv heads, d 128, 48 layers"),
    "q4": ("q4_attn_kernel<0>", "profiles/q4_attn_q4.md",
           "q4: 12 agents x 8192 tokens, 32 q / 8 kv heads, d 128, Q4G64 codes with fp16 scale+bias, "
           "256-token blocks, 32 layers"),
    "q4_mirror": ("q4_attn_kernel<1>", "profiles/q4_attn_q4_mirror.md",
                  "q4_mirror: the q4 workload with bf16 mirror diffs ~N(0,0.1) on 31 of each agent's 512 "
                  "16-token sub-blocks (6 %), restored inside the Q4 read"),
}


def graph_replay_ms(torch, fn, reps, flush):
    """Device time of one replay of fn captured in a CUDA graph (host launch
    cost removed).  The L2 is flushed (a buffer larger than L2 is written)
    before every replay, outside the timed events."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        flush.add_(1)
        a.record(st)
        g.replay()
        b.record(st)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / reps


def graph_timeline(torch, fn, tag):
    """Kernel start/end times (microseconds from the first kernel) of one
    replay of fn captured in a CUDA graph, from torch.profiler's CUDA
    activity trace: the real overlap of the kernels, which a serialising
    profiler does not show."""
    import tempfile
    from torch.profiler import ProfilerActivity, profile
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    # the first profiling session of a process records no kernel activity
    # here: run one to set the tracer up, then the one that is kept
    for _ in range(2):
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            g.replay()
            torch.cuda.synchronize()
    path = os.path.join(tempfile.gettempdir(), f"kvs_trace_{tag}_{os.getpid()}.json")
    prof.export_chrome_trace(path)
    with open(path) as f:
        ev = json.load(f)["traceEvents"]
    os.remove(path)
    ks = sorted((e for e in ev if e.get("cat") == "kernel" and "dur" in e), key=lambda e: e["ts"])
    if not ks:
        return []
    t0 = ks[0]["ts"]
    return [[e["name"].split("(")[0].replace("void ", "").replace("kvs::", ""), round(e["ts"] - t0, 2),
             round(e["ts"] + e["dur"] - t0, 2)] for e in ks]


def run_extra(name, torch, K, W, dev, steps, warmup, layers, trace=False):
    stream = torch.cuda.current_stream()
    if name == "select":
        return bench_select(torch, K, dev, stream, steps, warmup)
    if name == "mirror":
        return bench_mirror(torch, K, W, dev, steps)
    if name == "cow":
        return bench_cow(torch, K, W, dev, stream, steps, warmup)
    if name == "evict":
        return bench_evict(torch, K, dev, steps)
    if name == "io":
        return bench_io(torch, K, W, dev, steps)
    return workload_record(name, torch, K, W, dev, stream, steps, warmup, layers, trace)


def bench_select(torch, K, dev, stream, steps, warmup):
    """Critical-position selection of the all-gather round at one check layer:
    64 agents x 8192 shared positions x 8 KV heads x 128 dims, top 15 %."""
    n, rows, E = 64, 8192, 1024
    gen = torch.Generator(device=dev).manual_seed(11)
    kc = torch.randn((n * rows, E), generator=gen, device=dev)
    sig = 0.05 + 0.45 * torch.rand((n * rows, 1), generator=gen, device=dev)
    kn = (kc + torch.randn((n * rows, E), generator=gen, device=dev) * sig).to(torch.bfloat16).view(torch.int16)
    kc = kc.to(torch.bfloat16).view(torch.int16)
    off = torch.arange(n + 1, dtype=torch.int64, device=dev) * rows
    ws = torch.zeros(4 * n * rows, dtype=torch.uint8, device=dev)
    idx = torch.zeros(n * rows, dtype=torch.int32, device=dev)
    idx_off = torch.zeros(n + 1, dtype=torch.int64, device=dev)

    def run():
        K.kvs_select_critical(kc, kn, off, n, rows, E, 0.15, idx, idx_off, ws)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    byts = 2 * n * rows * E * 2
    peak, kind = read_peaks()
    return {"workload": "select: 64 agents x 8192 positions x (8 kv heads x 128), top 15 % by ||K_cached - K_new||",
            "kernel": "sel_scores + sel_topk", "profile": "profiles/sel_scores_select.md",
            "ms_per_call": ms, "rows_per_s": n * rows / (ms * 1e-3), "bytes_per_call": byts,
            "gbs": byts / (ms * 1e-3) / 1e9, "frac": byts / (ms * 1e-3) / 1e9 / peak, "peak": peak,
            "peak_kind": kind, "l2": "inputs (2.1 GB) larger than L2", "timing": "eager, back to back"}


def bench_tiny_replicated(torch, K, W, dev, reps, flush, n_inst=4096):
    """The tiny workload replicated: n_inst independent copies (own physical
    blocks, own mirror diffs) decoded by one plan + one attention launch."""
    w = W.make_tiny()
    N, H, D, B = w.n_seq, w.n_kv_heads, w.head_dim, w.block_tokens
    tokens = torch.from_numpy(w.tokens.view(np.int32)).to(dev)
    seq_off = torch.from_numpy(w.seq_off).to(dev)
    probe_k = torch.zeros(16, dtype=torch.int16, device=dev)
    probe = K.kvs_pool_create(1, H, D, B, K.KVS_DTYPE_BF16, w.capacity_blocks, N, [probe_k], [probe_k])
    fp = torch.zeros((N, w.max_blocks), dtype=torch.int64, device=dev)
    table = torch.zeros((N, w.max_blocks), dtype=torch.int32, device=dev)
    refc = torch.zeros(w.capacity_blocks, dtype=torch.int32, device=dev)
    nphys = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_d = torch.zeros(K.kvs_workspace_size(probe, K.KVS_OP_DEDUP, N, w.max_blocks), dtype=torch.uint8, device=dev)
    K.kvs_fingerprint_dedup(probe, tokens, seq_off, N, None, None, None, fp, table, w.max_blocks, refc, nphys, ws_d)
    n_phys = int(nphys.item())
    nd = w.diff_capacity_blocks
    rep = torch.arange(n_inst, device=dev, dtype=torch.int32).view(n_inst, 1, 1)
    t1 = table.view(1, N, w.max_blocks)
    table_r = torch.where(t1 >= 0, t1 + rep * n_phys, t1).reshape(n_inst * N, w.max_blocks).contiguous()
    d1 = torch.from_numpy(w.diff_table).to(dev).view(1, N, w.max_blocks)
    diff_r = torch.where(d1 >= 0, d1 + rep * nd, d1).reshape(n_inst * N, w.max_blocks).contiguous()
    seq_len = torch.from_numpy(w.seq_len).to(dev).repeat(n_inst)
    NS, cap, ndr = n_inst * N, n_inst * n_phys, n_inst * nd
    gen = torch.Generator(device=dev).manual_seed(17)
    k = torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
    v = torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
    dk = (0.1 * torch.randn((ndr, H, B, D), generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
    dv = (0.1 * torch.randn((ndr, H, B, D), generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
    pool = K.kvs_pool_create(1, H, D, B, K.KVS_DTYPE_BF16, cap, NS, [k], [v], dk_layers=[dk], dv_layers=[dv],
                             diff_capacity_blocks=ndr)
    q = torch.randn((NS, w.n_q_heads, D), generator=gen, device=dev, dtype=torch.bfloat16)
    out = torch.zeros((NS, w.n_q_heads, D), dtype=torch.float32, device=dev)
    ws = torch.zeros(K.kvs_workspace_size(pool, K.KVS_OP_DECODE_ATTN, NS, w.max_blocks, w.n_q_heads),
                     dtype=torch.uint8, device=dev)

    def run():
        K.kvs_decode_plan(pool, w.n_q_heads, table_r, w.max_blocks, seq_len, NS, diff_r, None, None, ws)
        K.kvs_decode_attn_planned(pool, 0, q, w.n_q_heads, table_r, w.max_blocks, seq_len, NS, diff_r, None,
                                  None, w.theta, w.scale, out, ws)

    ms = graph_replay_ms(torch, run, reps, flush)
    flags = K.kvs_pool_check(pool)
    byts = (cap + ndr) * H * B * D * 2 * 2 + NS * w.n_q_heads * D * (2 + 4) + NS * w.max_blocks * 4 * 2
    peak, _ = read_peaks()
    return {"instances": n_inst, "sequences": NS, "ms_plan_plus_attn": ms, "tokens_per_s": NS / (ms * 1e-3),
            "bytes": byts, "gbs": byts / (ms * 1e-3) / 1e9, "frac": byts / (ms * 1e-3) / 1e9 / peak,
            "timing": "CUDA graph of plan + attention, L2 flushed before every replay", "status_flags": flags}


def workload_record(name, torch, K, W, dev, stream, steps, warmup, layers, trace=False):
    """GPU dedup + plan + decode attention on every layer (Q4: attention only),
    eager through the public API and replayed from CUDA graphs."""
    mk = {"tiny": W.make_tiny, "gqa_fanout": W.make_gqa_fanout, "allgather": W.make_allgather, "q4": W.make_q4,
          "q4_mirror": W.make_q4_mirror, "mha7b": W.make_mha7b}
    w = mk[name]()
    L = layers or w.n_layers
    N, H, D, B = w.n_seq, w.n_kv_heads, w.head_dim, w.block_tokens
    q4 = name in ("q4", "q4_mirror")
    tokens = torch.from_numpy(w.tokens.view(np.int32)).to(dev)
    seq_off = torch.from_numpy(w.seq_off).to(dev)
    seq_len = torch.from_numpy(w.seq_len).to(dev)
    tier = torch.from_numpy(w.tier.view(np.int32)).to(dev) if (w.tier != 0).any() else None
    so = sb = None
    if w.seg_start_off is not None:
        so = torch.from_numpy(w.seg_start_off).to(dev)
        sb = torch.from_numpy(w.seg_start_blocks).to(dev)
    fp = torch.zeros((N, w.max_blocks), dtype=torch.int64, device=dev)
    table = torch.zeros((N, w.max_blocks), dtype=torch.int32, device=dev)
    # dedup once on a pool whose capacity is the upper bound, to size the slabs
    dummy = torch.zeros(16, dtype=torch.int16, device=dev)
    if q4:
        d8 = torch.zeros(16, dtype=torch.uint8, device=dev)
        dh = torch.zeros(16, dtype=torch.float16, device=dev)
        probe = K.kvs_pool_create(1, H, D, B, K.KVS_DTYPE_Q4G64, w.capacity_blocks, N, [d8], [d8], [dh], [dh])
    else:
        probe = K.kvs_pool_create(1, H, D, B, K.KVS_DTYPE_BF16, w.capacity_blocks, N, [dummy], [dummy])
    refc = torch.zeros(w.capacity_blocks, dtype=torch.int32, device=dev)
    nphys = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_d = torch.zeros(K.kvs_workspace_size(probe, K.KVS_OP_DEDUP, N, w.max_blocks), dtype=torch.uint8, device=dev)
    K.kvs_fingerprint_dedup(probe, tokens, seq_off, N, tier, so, sb, fp, table, w.max_blocks, refc, nphys, ws_d)
    cap = int(nphys.item())
    gen = torch.Generator(device=dev).manual_seed(7)
    nd = 0
    if q4:
        ks = [torch.empty(cap * H * B * D // 2, dtype=torch.uint8, device=dev) for _ in range(L)]
        vs = [torch.empty_like(ks[0]) for _ in range(L)]
        ksb = [torch.empty(cap * H * B * 4, dtype=torch.float16, device=dev) for _ in range(L)]
        vsb = [torch.empty_like(ksb[0]) for _ in range(L)]
        nd = w.diff_capacity_blocks
        dks = [(0.1 * torch.randn((nd, H, 16, D), generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
               for _ in range(L)] if nd else None
        dvs = [(0.1 * torch.randn((nd, H, 16, D), generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
               for _ in range(L)] if nd else None
        pool = K.kvs_pool_create(L, H, D, B, K.KVS_DTYPE_Q4G64, cap, N, ks, vs, ksb, vsb, dk_layers=dks,
                                 dv_layers=dvs, diff_capacity_blocks=nd)
        ids = torch.arange(cap, dtype=torch.int32, device=dev)
        for l in range(L):
            src_k = torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16)
            src_v = torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16)
            K.kvs_quantize_q4(pool, l, src_k.view(torch.int16), src_v.view(torch.int16), ids, cap)
            del src_k, src_v
        per_launch = cap * H * B * 144 + nd * H * 16 * D * 2 * 2
    else:
        ks = [torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
              for _ in range(L)]
        vs = [torch.randn((cap, H, B, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
              for _ in range(L)]
        nd = w.diff_capacity_blocks
        dks = [(0.1 * torch.randn((nd, H, B, D), generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
               for _ in range(L)] if nd else None
        dvs = [(0.1 * torch.randn((nd, H, B, D), generator=gen, device=dev)).to(torch.bfloat16).view(torch.int16)
               for _ in range(L)] if nd else None
        pool = K.kvs_pool_create(L, H, D, B, K.KVS_DTYPE_BF16, cap, N, ks, vs, dk_layers=dks, dv_layers=dvs,
                                 diff_capacity_blocks=nd)
        per_launch = (cap + nd) * H * B * D * 2 * 2
    per_launch += N * w.n_q_heads * D * (2 + 4) + N * w.max_blocks * 4
    if w.diff_table is not None:
        per_launch += w.diff_table.nbytes
    refc = torch.zeros(cap, dtype=torch.int32, device=dev)
    q = torch.randn((L, N, w.n_q_heads, D), generator=gen, device=dev, dtype=torch.bfloat16)
    out = torch.zeros((L, N, w.n_q_heads, D), dtype=torch.float32, device=dev)
    dt = torch.from_numpy(w.diff_table).to(dev) if w.diff_table is not None else None
    ro = torch.from_numpy(w.rope_off).to(dev) if w.rope_off is not None else None
    rs = torch.from_numpy(w.rope_segs).to(dev) if w.rope_segs is not None else None
    op = K.KVS_OP_DECODE_ATTN_Q4 if q4 else K.KVS_OP_DECODE_ATTN
    ws_a = torch.zeros(K.kvs_workspace_size(pool, op, N, w.max_blocks, w.n_q_heads), dtype=torch.uint8, device=dev)

    def attn(l):
        if q4:
            K.kvs_decode_attn_q4(pool, l, q[l], w.n_q_heads, table, w.max_blocks, seq_len, N, w.scale, out[l], ws_a,
                                 diff_table=dt)
        else:
            K.kvs_decode_attn_planned(pool, l, q[l], w.n_q_heads, table, w.max_blocks, seq_len, N, dt, ro, rs,
                                      w.theta, w.scale, out[l], ws_a)

    def step(ev=None):
        if not q4:
            K.kvs_fingerprint_dedup(pool, tokens, seq_off, N, tier, so, sb, fp, table, w.max_blocks, refc, nphys, ws_d)
            K.kvs_decode_plan(pool, w.n_q_heads, table, w.max_blocks, seq_len, N, dt, ro, rs, ws_a)
        for l in range(L):
            if ev is not None:
                ev[l][0].record(stream)
            attn(l)
            if ev is not None:
                ev[l][1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    flags = K.kvs_pool_check(pool)
    # eager, whole steps between two events
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms_step = t0.elapsed_time(t1) / steps
    # eager breakdown: events around every layer's attention call
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
          for _ in range(steps)]
    for i in range(steps):
        step(ev[i])
    torch.cuda.synchronize()
    attn_ms = sum(a.elapsed_time(b) for row in ev for a, b in row) / (steps * L)
    peak, kind = read_peaks()
    # the same work replayed from CUDA graphs (host launch cost removed): the
    # whole step, and the attention launches alone
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    g_step = graph_replay_ms(torch, step, steps, flush)
    g_attn = graph_replay_ms(torch, lambda: [attn(l) for l in range(L)], steps, flush) / L
    kern, prof, desc = CONFIG_INFO[name]

    def gbs(ms):
        return per_launch / (ms * 1e-3) / 1e9

    rec = {"workload": desc, "kernel": kern, "profile": prof, "layers": L, "n_phys": cap, "diff_blocks": nd,
           "attn_bytes_per_launch": per_launch, "peak": peak, "peak_kind": kind,
           "eager": {"tokens_per_s": N / (ms_step * 1e-3), "ms_per_step": ms_step, "attn_ms_per_layer": attn_ms,
                     "attn_gbs": gbs(attn_ms), "frac": gbs(attn_ms) / peak,
                     "timing": "public API calls from Python; step = dedup + plan + every layer" +
                               (" (Q4: attention only)" if q4 else "") +
                               "; per-layer time from a second pass with events around each call"},
           "graph": {"tokens_per_s": N / (g_step * 1e-3), "ms_per_step": g_step, "attn_ms_per_layer": g_attn,
                     "attn_gbs": gbs(g_attn), "frac": gbs(g_attn) / peak,
                     "timing": "CUDA graph replays, L2 flushed before every replay"},
           "status_flags": flags | K.kvs_pool_check(pool)}
    if trace:
        rec["timeline"] = {"what": "kernel [name, start_us, end_us] of one CUDA-graph replay of every layer's "
                                   "attention call (torch.profiler CUDA activity trace)",
                           "kernels": graph_timeline(torch, lambda: [attn(l) for l in range(L)], name)}
    if name == "tiny":
        rec["eager"]["l2"] = "the 0.43 MB working set stays in L2 between eager steps"
        rec["tiny_x4096"] = bench_tiny_replicated(torch, K, W, dev, steps, flush)
    return rec


def bench_mirror(torch, K, W, dev, steps):
    """Mirror construction of the all-gather round at one layer: 64 agents,
    each refreshing every row of 31 blocks among its 512 shared-segment
    blocks (the round's mirror structure), K rotated back by the segment
    shift."""
    w = W.make_allgather(n_layers=1)
    rng = np.random.default_rng(5)
    tokens = torch.from_numpy(w.tokens.view(np.int32)).to(dev)
    seq_off = torch.from_numpy(w.seq_off).to(dev)
    so = torch.from_numpy(w.seg_start_off).to(dev)
    sb = torch.from_numpy(w.seg_start_blocks).to(dev)
    N, H, D = w.n_seq, w.n_kv_heads, w.head_dim
    d16 = torch.zeros(16, dtype=torch.int16, device=dev)
    probe = K.kvs_pool_create(1, H, D, 16, K.KVS_DTYPE_BF16, w.capacity_blocks, N, [d16], [d16])
    fp = torch.zeros((N, w.max_blocks), dtype=torch.int64, device=dev)
    table = torch.zeros((N, w.max_blocks), dtype=torch.int32, device=dev)
    refc = torch.zeros(w.capacity_blocks, dtype=torch.int32, device=dev)
    nphys = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_d = torch.zeros(K.kvs_workspace_size(probe, K.KVS_OP_DEDUP, N, w.max_blocks), dtype=torch.uint8, device=dev)
    K.kvs_fingerprint_dedup(probe, tokens, seq_off, N, None, so, sb, fp, table, w.max_blocks, refc, nphys, ws_d)
    cap = int(nphys.item())
    idx, off = [], [0]
    for a in range(N):
        fb = int(w.rope_segs[w.rope_off[a]][0])
        for b in np.sort(rng.choice(512, size=31, replace=False)) + fb:
            idx.extend(range(int(b) * 16, int(b) * 16 + 16))
        off.append(len(idx))
    n_rows = len(idx)
    gen = torch.Generator(device=dev).manual_seed(9)
    k = torch.randn((cap, H, 16, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
    v = torch.randn((cap, H, 16, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
    kn = torch.randn((n_rows, H, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
    vn = torch.randn((n_rows, H, D), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
    cap_d = N * 31
    dk = torch.zeros((cap_d, H, 16, D), dtype=torch.int16, device=dev)
    dv = torch.zeros_like(dk)
    pool = K.kvs_pool_create(1, H, D, 16, K.KVS_DTYPE_BF16, cap, N, [k], [v], dk_layers=[dk], dv_layers=[dv],
                             diff_capacity_blocks=cap_d)
    idx_t = torch.tensor(idx, dtype=torch.int32, device=dev)
    off_t = torch.tensor(off, dtype=torch.int64, device=dev)
    ro = torch.from_numpy(w.rope_off).to(dev)
    rs = torch.from_numpy(w.rope_segs).to(dev)
    sl = torch.from_numpy(w.seq_len).to(dev)
    diff_table = torch.zeros((N, w.max_blocks), dtype=torch.int32, device=dev)
    n_diff = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(K.kvs_workspace_size(pool, K.KVS_OP_MIRROR, N, w.max_blocks), dtype=torch.uint8, device=dev)

    def run():
        K.kvs_mirror_build(pool, 0, table, w.max_blocks, sl, N, idx_t, off_t, kn, vn, ro, rs, w.theta,
                           diff_table, n_diff, ws)

    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    ms = graph_replay_ms(torch, run, steps, flush)
    flags = K.kvs_pool_check(pool)
    tile = 16 * D * 2
    byts = (cap_d * H * tile * 2) * 3 + n_rows * 4 + N * w.max_blocks * 4 * 2
    peak, _ = read_peaks()
    return {"workload": "mirror: all-gather round, 64 agents x 31 refreshed blocks among 512 shared-segment blocks, "
                        "8 kv heads x 128, K rotated back by the segment shift",
            "kernel": "mir_write + 2 index kernels (mir_agent, mir_apply)", "ms_per_call": ms, "dirty_blocks": cap_d, "rows": n_rows,
            "bytes": byts, "gbs": byts / (ms * 1e-3) / 1e9, "frac": byts / (ms * 1e-3) / 1e9 / peak,
            "timing": "CUDA graph replays, L2 flushed before every replay", "status_flags": flags}


def bench_cow(torch, K, W, dev, stream, steps, warmup):
    """Copy-on-write burst on the 7B multi-head tables (32 layers x 32 KV
    heads): agent 0 writes into all 614 shared blocks, so each is copied (K
    and V of every layer, 8 MiB per block); then all 8 sequences are
    released.  Tables, counts and the free stack are restored before every
    timed call, outside the timed region."""
    w = W.make_mha7b(n_layers=1)
    N, L, H, D = w.n_seq, 32, 32, 128
    tokens = torch.from_numpy(w.tokens.view(np.int32)).to(dev)
    seq_off = torch.from_numpy(w.seq_off).to(dev)
    cap = 614 + N * 410 + 614
    ks = [torch.zeros((cap, H, 16, D), dtype=torch.int16, device=dev) for _ in range(L)]
    vs = [torch.zeros_like(ks[0]) for _ in range(L)]
    pool = K.kvs_pool_create(L, H, D, 16, K.KVS_DTYPE_BF16, cap, N, ks, vs)
    fp = torch.zeros((N, w.max_blocks), dtype=torch.int64, device=dev)
    table0 = torch.zeros((N, w.max_blocks), dtype=torch.int32, device=dev)
    ref0 = torch.zeros(cap, dtype=torch.int32, device=dev)
    nphys = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_d = torch.zeros(K.kvs_workspace_size(pool, K.KVS_OP_DEDUP, N, w.max_blocks), dtype=torch.uint8, device=dev)
    K.kvs_fingerprint_dedup(pool, tokens, seq_off, N, None, None, None, fp, table0, w.max_blocks, ref0, nphys, ws_d)
    ws = torch.zeros(K.kvs_workspace_size(pool, K.KVS_OP_BLOCKS, 1024, 0), dtype=torch.uint8, device=dev)
    free0 = torch.zeros(cap, dtype=torch.int32, device=dev)
    nfree0 = torch.zeros(1, dtype=torch.int32, device=dev)
    K.kvs_blocks_init_free(pool, ref0, free0, nfree0, ws)
    table, ref, free, nfree = table0.clone(), ref0.clone(), free0.clone(), nfree0.clone()
    sl0 = torch.from_numpy(w.seq_len).to(dev)
    sl = sl0.clone()
    wseq = torch.zeros(614, dtype=torch.int32, device=dev)
    wblk = torch.arange(614, dtype=torch.int32, device=dev)
    rel = torch.arange(N, dtype=torch.int32, device=dev)

    def restore():
        table.copy_(table0); ref.copy_(ref0); free.copy_(free0); nfree.copy_(nfree0); sl.copy_(sl0)

    times_w, times_r = [], []
    for it in range(warmup + steps):
        restore()
        torch.cuda.synchronize()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        K.kvs_block_write(pool, table, w.max_blocks, N, wseq, wblk, 614, ref, free, nfree, ws)
        e1.record(stream)
        K.kvs_seq_release(pool, table, w.max_blocks, sl, N, rel, N, ref, free, nfree, ws)
        e2.record(stream)
        torch.cuda.synchronize()
        if it >= warmup:
            times_w.append(e0.elapsed_time(e1))
            times_r.append(e1.elapsed_time(e2))
    flags = K.kvs_pool_check(pool)
    ok = int(nfree.item()) == cap and int(ref.abs().sum().item()) == 0
    ms_w = sum(times_w) / len(times_w)
    ms_r = sum(times_r) / len(times_r)
    byts = 614 * L * 2 * (H * 16 * D * 2) * 2   # every copied byte read once and written once
    peak, _ = read_peaks()
    return ({"workload": "cow", "copies": 614, "bytes_per_copy": L * 2 * H * 16 * D * 2,
                      "write_batch_ms": ms_w, "gbs": byts / (ms_w * 1e-3) / 1e9,
                      "frac_of_measured_peak": byts / (ms_w * 1e-3) / 1e9 / peak,
                      "release_ms": ms_r, "released_blocks": cap - 614, "all_blocks_free_after": ok,
                      "status_flags": flags})


def bench_evict(torch, K, dev, steps):
    """Block-granular eviction scoring: 64 agents x 16,384 tokens (1,024
    blocks each), five regions with the MemDecay post's suggested initial
    scores, each agent evicting a quarter of its blocks."""
    n, mb, B = 64, 1024, 16
    T = mb * B
    rng = np.random.default_rng(3)
    region = np.full((n, T), 4, np.uint8)
    region[:, :64] = 0
    region[rng.random((n, T)) < 0.03] = 1
    region[rng.random((n, T)) < 0.05] = 2
    region[:, T - 256:] = 3
    created = np.tile(np.arange(T, dtype=np.int32), (n, 1))
    access = rng.poisson(1.5, size=(n, T)).astype(np.int32)
    d16 = torch.zeros(16, dtype=torch.int16, device=dev)
    pool = K.kvs_pool_create(1, 1, 64, B, K.KVS_DTYPE_BF16, 1, 1, [d16], [d16])
    reg_t = torch.from_numpy(region).to(dev)
    cr_t = torch.from_numpy(created).to(dev)
    ac_t = torch.from_numpy(access).to(dev)
    sl = torch.full((n,), T, dtype=torch.int32, device=dev)
    k = torch.full((n,), mb // 4, dtype=torch.int32, device=dev)
    scores = torch.zeros((n, mb), dtype=torch.float32, device=dev)
    victims = torch.zeros(n * mb // 4, dtype=torch.int32, device=dev)
    voff = torch.zeros(n + 1, dtype=torch.int64, device=dev)
    init, decay = [100.0, 10.0, 5.0, 2.0, 1.0], [0.0, 0.0092, 0.02, 0.05, 0.1]

    def run():
        K.kvs_evict_score(pool, reg_t, cr_t, ac_t, sl, n, mb, init, decay, T + 10, k, scores, victims, voff)

    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    ms = graph_replay_ms(torch, run, steps, flush)
    byts = n * T * 9 + n * mb * 4 + n * mb // 4 * 4
    return ({"workload": "evict", "ms_per_call": ms, "blocks_scored": n * mb, "victims": n * mb // 4,
                      "blocks_per_s": n * mb / (ms * 1e-3), "bytes": byts, "gbs": byts / (ms * 1e-3) / 1e9,
                      "note": "9.4 MB per call: latency-bound", "l2": "flushed before every replay",
                      "status_flags": K.kvs_pool_check(pool)})


def bench_io(torch, K, W, dev, steps):
    """Export and import of the Q4 configuration's whole pool: 12 agents x 32
    blocks of 256 tokens, 32 layers x 8 KV heads (codes and scale/bias), the
    device side of saving and reloading a persistent Q4 cache."""
    w = W.make_q4(n_layers=1)
    L, H, cap = 32, w.n_kv_heads, w.capacity_blocks
    g = torch.Generator(device=dev).manual_seed(4)
    codes = [torch.randint(0, 256, (cap, H, 256, 64), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
             for _ in range(2 * L)]
    sbs = [torch.randn((cap, H, 256, 4), generator=g, device=dev).to(torch.float16) for _ in range(2 * L)]
    pool = K.kvs_pool_create(L, H, 128, 256, K.KVS_DTYPE_Q4G64, 2 * cap, w.n_seq,
                             [torch.cat([c, torch.zeros_like(c)]) for c in codes[0::2]],
                             [torch.cat([c, torch.zeros_like(c)]) for c in codes[1::2]],
                             [torch.cat([s_, torch.zeros_like(s_)]) for s_ in sbs[0::2]],
                             [torch.cat([s_, torch.zeros_like(s_)]) for s_ in sbs[1::2]])
    del codes, sbs
    rec = K.kvs_pool_block_bytes(pool)
    packed = torch.zeros(cap * rec, dtype=torch.uint8, device=dev)
    src = torch.arange(cap, dtype=torch.int32, device=dev)
    dst = src + cap
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    ms_e = graph_replay_ms(torch, lambda: K.kvs_pool_export(pool, src, cap, packed), steps, flush)
    ms_i = graph_replay_ms(torch, lambda: K.kvs_pool_import(pool, dst, cap, packed), steps, flush)
    byts = 2 * cap * rec
    peak, _ = read_peaks()
    return ({"workload": "io", "blocks": cap, "record_bytes": rec, "export_ms": ms_e, "import_ms": ms_i,
                      "export_gbs": byts / (ms_e * 1e-3) / 1e9, "import_gbs": byts / (ms_i * 1e-3) / 1e9,
                      "frac_of_measured_peak": [byts / (ms_e * 1e-3) / 1e9 / peak, byts / (ms_i * 1e-3) / 1e9 / peak],
                      "status_flags": K.kvs_pool_check(pool)})


def bench_rope(torch, K, W, dev, stream, args, peak):
    """All-gather round, one layer: 64 agents x 64 shared 128-token segments
    re-rotated from the master copy into private blocks (524,288 rows)."""
    w = W.make_allgather(n_layers=1)
    # physical layout: masters = first occurrences; destinations after them
    n_master = 64 * 8
    rows = []
    B = w.block_tokens
    src_row = 0
    r_off = w.rope_off
    src_segs = w.rope_segs[r_off[0]:r_off[1]]
    # source table: row 0 maps its segment blocks to master blocks 0..511
    src_table = np.full((1, w.max_blocks), -1, np.int32)
    by_src = {}
    for j, (fb, nb, delta, _) in enumerate(src_segs):
        src_table[0, fb:fb + nb] = np.arange(j * nb, (j + 1) * nb)
        by_src[fb * B - delta] = fb * B
    jobs = []
    dst_table = np.full((w.n_seq, w.max_blocks), -1, np.int32)
    nxt = n_master
    for a in range(w.n_seq):
        for (fb, nb, delta, _) in w.rope_segs[r_off[a]:r_off[a + 1]]:
            dst_table[a, fb:fb + nb] = np.arange(nxt, nxt + nb)
            nxt += nb
            jobs.append((src_row, by_src[fb * B - delta], a, fb * B, nb * B, fb * B - delta, fb * B, 0))
    jobs = np.array(jobs, np.int32)
    cap = nxt
    k = torch.randn((cap, w.n_kv_heads, B, w.head_dim), device=dev, dtype=torch.bfloat16)
    v = torch.zeros(16, dtype=torch.int16, device=dev)
    pool = K.kvs_pool_create(1, w.n_kv_heads, w.head_dim, B, K.KVS_DTYPE_BF16, cap, w.n_seq, [k.view(torch.int16)], [v])
    jd = torch.from_numpy(jobs).to(dev)
    st = torch.from_numpy(src_table).to(dev)
    dt = torch.from_numpy(dst_table).to(dev)
    n_rows = int(jobs[:, 4].sum())

    def run():
        K.kvs_rope_rerotate(pool, 0, jd, len(jobs), 128, w.theta, st, dt, w.max_blocks)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(min(args.steps, 20)):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    flags = K.kvs_pool_check(pool)
    t = e0.elapsed_time(e1) / min(args.steps, 20) * 1e-3
    row_bytes = w.n_kv_heads * w.head_dim * 2
    algo = n_master * w.n_kv_heads * B * w.head_dim * 2 + n_rows * row_bytes + jobs.nbytes
    del k, pool
    return {"rows_per_s": n_rows / t, "unit": "rows/s (one row = one token's K over all KV heads)",
            "rows": n_rows, "ms": t * 1e3, "achieved_gbs": algo / t / 1e9, "frac": algo / t / 1e9 / peak,
            "status_flags": flags}


if __name__ == "__main__":
    sys.exit(main())
