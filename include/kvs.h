/*
 * kvs.h — C ABI of libkvs: decode-step attention over a pool of fixed-size KV
 * blocks shared by many agents, for NVIDIA GB300 (sm_103a).
 *
 * The operations follow these pages:
 *   [INMS]   "大模型多Agent系统显存优化：KV Cache共享机制解析" — a walkthrough of
 *            "INMS: Memory Sharing for LLM based Agents": fixed-size blocks,
 *            content fingerprints, refcounts, prefix sharing (§2.2, §3.2),
 *            RoPE offset compensation (§3.2), tier folded into the
 *            fingerprint (§5.1).
 *   [TD]     "TokenDance: Scaling Multi-Agent LLM Serving via Collective KV
 *            Cache Sharing" (news summary): segment hashing (section 1),
 *            batched RoPE and critical-position selection (section 2, Fig. 6),
 *            master/mirror block-sparse diffs with fused restore (section 3,
 *            Fig. 7, Fig. 8).
 *   [POOL]   "共享内存KV Cache池" — host shared-memory KV pool post: per-token KV
 *            formula (§1.1), CalcHash (§3.2), longest-prefix match (§3.3).
 *   [Q4]     "Agent Memory Below the Prompt: Persistent Q4 KV Cache for
 *            Multi-Agent LLM Inference on Edge Devices" (summary): 256-token
 *            4-bit blocks (§2.1), attention directly on Q4 (§2.2).
 *   [MD]     "MemDecay: Region-Aware KV Cache Eviction" (§4.2: scores are
 *            q.k / sqrt(head_dim)).
 *
 * Conventions for every call:
 *   - Pointers named *_dev or documented "device" are device pointers in the
 *     current CUDA device's memory; everything else is host memory.
 *   - Every device buffer is owned by the caller.  The library allocates
 *     device memory only in kvs_pool_create (a status word and the split-K
 *     arrival counters, freed by kvs_pool_destroy).
 *   - Calls that take a cudaStream_t only enqueue work on it and return
 *     without synchronising, except kvs_pool_check and kvs_pool_stats.
 *   - Calls on one pool must be ordered on one stream (the arrival counters
 *     and the status word are per pool).
 *   - Host-detectable argument errors return a status before anything is
 *     enqueued.  Errors the device detects (a block id outside the pool, a
 *     sequence longer than its block-table row, a capacity overflow, a
 *     bounded wait that ran out) set bits in the pool's status word, skip the
 *     offending access and never trap; read them with kvs_pool_check.
 *   - kvs_last_error_string() describes the last failure on this host thread.
 */
#ifndef KVS_H
#define KVS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVS_OK = 0,
  KVS_ERR_INVALID_ARG = 1,    /* a null/misaligned pointer or an out-of-range size */
  KVS_ERR_CAPACITY = 2,       /* a pool, table or workspace is too small */
  KVS_ERR_CUDA = 3,           /* a CUDA runtime call failed */
  KVS_ERR_DEVICE_BOUNDS = 4,  /* the device saw an out-of-range index (kvs_pool_check) */
  KVS_ERR_UNSUPPORTED = 5     /* a shape this build has no kernel for */
} kvs_status;

/* Device status-word bits reported by kvs_pool_check. */
#define KVS_DEVERR_BLOCK_ID     0x1u  /* block id < 0 or >= capacity in a table */
#define KVS_DEVERR_SEQ_LEN      0x2u  /* seq_len beyond max_blocks * block_tokens, or < 0 */
#define KVS_DEVERR_CAPACITY     0x4u  /* dedup produced more physical blocks than capacity */
#define KVS_DEVERR_DIFF_ID      0x8u  /* diff block id >= diff capacity */
#define KVS_DEVERR_WAIT_TIMEOUT 0x10u /* a bounded wait on a TMA copy ran out */
#define KVS_DEVERR_ROPE_RANGE   0x20u /* |position shift| >= 2^18 */
#define KVS_DEVERR_JOB          0x40u /* a RoPE job addresses tokens outside its table row */
#define KVS_DEVERR_PLAN         0x80u /* kvs_decode_attn_planned saw no matching plan in ws */
#define KVS_DEVERR_REFCOUNT     0x100u /* a release took a reference count below zero */

typedef enum { KVS_DTYPE_BF16 = 0, KVS_DTYPE_Q4G64 = 1 } kvs_dtype;

/* Pool geometry.  One K slab and one V slab per layer.
 *   BF16:   slab[capacity_blocks][num_kv_heads][block_tokens][head_dim] bf16.
 *   Q4G64:  codes[capacity_blocks][num_kv_heads][block_tokens][head_dim/2]
 *           uint8 (element 2i in the low nibble of byte i) plus scale/bias
 *           [capacity_blocks][num_kv_heads][block_tokens][head_dim/64][2] fp16
 *           (index 0 = scale, 1 = bias; value = scale * code + bias) — [Q4]
 *           §2.1 (ratio 0.281 fixes group 64 with fp16 scale and bias).
 *   Mirror diffs: dk/dv slabs [diff_capacity_blocks][num_kv_heads]
 *           [diff_tokens][head_dim] bf16 holding K and V differences added to
 *           a master block — [TD] section 3; diff_tokens = block_tokens for
 *           BF16 pools and 16 (one sub-block of a 256-token block) for Q4G64
 *           pools.
 * Supported by this build: head_dim 64 or 128; BF16 block_tokens 16;
 * Q4G64 block_tokens 256 with head_dim 128. */
typedef struct {
  int32_t num_layers;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_tokens;
  int32_t dtype;                 /* kvs_dtype */
  int32_t capacity_blocks;       /* physical blocks per layer slab */
  int32_t diff_capacity_blocks;  /* 0 = no mirror diffs */
  int32_t max_seqs;              /* largest n_seq any call will pass */
} kvs_pool_desc;

typedef struct kvs_pool kvs_pool;

/* Create a pool over caller-owned per-layer slabs.  The pointer arrays are
 * host arrays of num_layers device pointers (16-byte aligned); k_sb/v_sb are
 * required for Q4G64 and must be NULL for BF16; dk/dv are required when
 * diff_capacity_blocks > 0.  Builds one TMA tensor map per slab.  The pool
 * never frees the slabs.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
kvs_status kvs_pool_create(const kvs_pool_desc* desc,
                           void* const* k_layers, void* const* v_layers,
                           void* const* k_sb_layers, void* const* v_sb_layers,
                           void* const* dk_layers, void* const* dv_layers,
                           kvs_pool** out);
kvs_status kvs_pool_destroy(kvs_pool* pool);

/* ---------------------------------------------------------------------------
 * Block fingerprints + deduplication ([POOL] §3.2 CalcHash, §3.3; [INMS]
 * §2.2, §3.2, §5.1; [TD] section 1 segment hashing).
 *
 * tokens_dev    uint32 token ids of all sequences, concatenated.
 * seq_off_dev   int64 [n_seq+1] CSR offsets into tokens.
 * tier_dev      uint32 [n_seq] memory tier per sequence, or NULL (= tier 0).
 *               Tier 0xFFFFFFFF is PRIVATE: its blocks are never shared.
 * seg_off_dev / seg_blocks_dev   optional CSR (int64 [n_seq+1] / int32) of
 *               block indices where a hashed segment starts (block 0 always
 *               does); NULL for plain prefix hashing.  Ascending per sequence.
 * fp_out_dev    uint64 [n_seq][max_blocks]: CalcHash(block tokens, tier) of
 *               every full block, 0 elsewhere.
 * block_table_dev int32 [n_seq][max_blocks]: physical block id, -1 unused.
 * refcount_dev  int32 [pool capacity]: references per physical block
 *               (entries >= n_phys are zeroed).
 * n_phys_dev    int32 [1]: physical blocks used.
 * owner_seq_dev int32 [pool capacity] or NULL: the sequence of each physical
 *               block's first occurrence (the sequence that owns it, [INMS]
 *               §2.2); -1 for ids >= n_phys.
 * ref_off_dev / ref_seq_dev   int64 [capacity + 1] / int32 [n_seq *
 *               max_blocks], both NULL or both set: the references of every
 *               physical block as a CSR (the shared-reference lists that
 *               [INMS] §3.3 hooks walk and that the shared attention tiles
 *               group by): ref_off is the exclusive prefix sum of refcount
 *               (ref_off[capacity] = total references) and ref_seq[ref_off[id]
 *               .. ref_off[id + 1]) lists the sequence of every slot mapped to
 *               id, in ascending (sequence, block) order; a block is shared
 *               when it has more than one entry.  Costs one extra single-CTA
 *               kernel.
 * Rule: full blocks of equal tier (not PRIVATE), at the same index inside
 * their segment, with identical token runs from the segment start through the
 * block, share one physical block; tail and PRIVATE blocks get fresh ones; ids
 * follow first occurrence scanning sequence-major.  The result is exact: a
 * 64-bit hash collision is caught by a token compare and resolved.
 * ws/ws_bytes   device scratch of kvs_workspace_size(KVS_OP_DEDUP) bytes.
 * flags         0, or KVS_DEDUP_TEST_WEAK_KEYS (truncates the internal table
 *               keys to 6 bits so that the collision path runs; results are
 *               unchanged, only slower).
 * Device errors: SEQ_LEN (a sequence needs more than max_blocks blocks),
 * CAPACITY (more physical blocks than the pool holds). */
#define KVS_DEDUP_TEST_WEAK_KEYS 0x1u
kvs_status kvs_fingerprint_dedup(kvs_pool* pool,
                                 const uint32_t* tokens_dev, const int64_t* seq_off_dev,
                                 int32_t n_seq, const uint32_t* tier_dev,
                                 const int64_t* seg_off_dev, const int32_t* seg_blocks_dev,
                                 uint64_t* fp_out_dev, int32_t* block_table_dev,
                                 int32_t max_blocks, int32_t* refcount_dev, int32_t* n_phys_dev,
                                 int32_t* owner_seq_dev, int64_t* ref_off_dev, int32_t* ref_seq_dev,
                                 uint32_t flags, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Batched RoPE re-rotation of reused K ([INMS] §3.2; [TD] section 2, one
 * batched RoPE call per layer).  Each job moves n_tok tokens of K:
 *   K[dst] = R(dst_pos - src_pos) * K[src]
 * with rotate-half pairing (i, i + d/2) and frequency theta^(-2i/d); V is not
 * touched.  Source token t is token src_tok0+t of row src_row of
 * src_table_dev; the destination is token dst_tok0+t of row dst_row of
 * dst_table_dev; both tables are int32 [rows][max_blocks] into this layer's K
 * slab, all KV heads.  Destinations must not overlap sources.
 * jobs_dev      kvs_rope_job [n_jobs] (device).
 * max_job_tokens  an upper bound of n_tok over the jobs (sizes the grid).
 * |dst_pos - src_pos| must be < 2^18.  BF16 pools only. */
typedef struct {
  int32_t src_row, src_tok0, dst_row, dst_tok0, n_tok, src_pos, dst_pos, reserved;
} kvs_rope_job;
kvs_status kvs_rope_rerotate(kvs_pool* pool, int32_t layer, const kvs_rope_job* jobs_dev,
                             int32_t n_jobs, int32_t max_job_tokens, float theta,
                             const int32_t* src_table_dev, const int32_t* dst_table_dev,
                             int32_t max_blocks, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Critical-position selection ([TD] section 2: one batched difference
 * computation finds each request's positions whose cached and new K differ
 * most).  For agent a with rows [row_off[a], row_off[a+1]) of k_cached and
 * k_new (bf16 [rows][row_elems]):
 *   score_t = || k_cached[t] - k_new[t] ||_2   (fp32 accumulation)
 *   k_a = ceil(ratio * n_a)  (ratio as float32, product in fp64)
 * keeps the k_a largest scores (ties toward the lower position) and writes
 * their positions, relative to the agent's first row, ascending, to
 * idx_out_dev[idx_off[a] ...]; idx_off_dev (int64 [n_agents+1]) is the
 * exclusive prefix sum of k_a.  row_elems must be a multiple of 8.
 * max_rows_per_agent bounds n_a (<= 65536).  ws: kvs_workspace_size(SELECT).
 * row_off must be non-decreasing with every value in [0, n_agents *
 * max_rows_per_agent]; k_cached/k_new hold rows [row_off[0],
 * row_off[n_agents]).  Because row_off is device memory this is not checked
 * before launch: an agent whose range ends before it starts, or leaves
 * [max(row_off[0], 0), min(row_off[n_agents], n_agents * max_rows_per_agent)),
 * is treated as empty (k_a = 0, nothing written for it), and rows past
 * n_agents * max_rows_per_agent are ignored. */
kvs_status kvs_select_critical(const void* k_cached_dev, const void* k_new_dev,
                               const int64_t* row_off_dev, int32_t n_agents,
                               int32_t max_rows_per_agent, int32_t row_elems, float ratio,
                               int32_t* idx_out_dev, int64_t* idx_off_dev,
                               void* ws, size_t ws_bytes, cudaStream_t stream);

/* Same selection as kvs_select_critical, for callers that cannot allocate
 * device memory on the call path — for example a serving process that has
 * handed all free device memory to its KV pool and caching allocator up front
 * (a further cudaMalloc would fail or fragment it), a latency-critical step
 * that cannot afford cudaMalloc/cudaFree's implicit device synchronisation,
 * or a plain C caller that does not want to size and own a workspace.  The
 * pages have no counterpart to this entry point.
 * Scratch: a fixed device array of 2^20 fp32 scores inside the library,
 * reserved on every GPU that loads the library and held until the process
 * exits.  n_agents * max_rows_per_agent must not exceed 2^20, otherwise
 * KVS_ERR_CAPACITY is returned before anything is enqueued.  The caller still
 * passes all inputs and outputs (same meaning as kvs_select_critical).
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress: no allocation, and correct after a device reset).
 * The first call made with a given device current can load the library's
 * device code as part of that lookup; make that first call before any stream
 * capture.
 * All calls on a device share the one array and it keeps the previous call's
 * contents; every value a call reads is written earlier in the same call
 * (row_off rules as for kvs_select_critical).
 * Calls whose work can overlap on the GPU (different streams, or threads
 * without ordering) race on the array and give undefined results. */
kvs_status kvs_select_critical_noalloc(const void* k_cached_dev, const void* k_new_dev,
                                       const int64_t* row_off_dev, int32_t n_agents,
                                       int32_t max_rows_per_agent, int32_t row_elems, float ratio,
                                       int32_t* idx_out_dev, int64_t* idx_off_dev, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Paged decode attention with the mirror-diff overlay and segment RoPE
 * restore fused into the read ([TD] section 3, Fig. 8: blocks with a diff
 * are corrected on chip before attention, nothing dense is materialised;
 * [INMS] §3.2 rotation; [MD] §4.2 scaled dot product).  For every sequence a
 * and query head h (kv head = h / (n_q_heads / num_kv_heads)):
 *   out[a][h] = sum_t softmax_t(scale * <q[a][h], K~_a[t]>) V~_a[t]
 *   K~ = R(delta_seg) (K_blk + DK_blk),  V~ = V_blk + DV_blk
 * over t < seq_len[a]; DK/DV are the agent's diff block for that logical block
 * (diff_table >= 0) and delta_seg the shift of the RoPE segment covering it.
 * q_dev         bf16 [n_seq][n_q_heads][head_dim] (already position-encoded).
 * block_table_dev int32 [n_seq][max_blocks]; seq_len_dev int32 [n_seq].
 * diff_table_dev  int32 [n_seq][max_blocks] diff block id or -1; or NULL.
 * rope_off_dev / rope_segs_dev  optional CSR: int32 [n_seq+1] offsets into
 *               kvs_seg_rope entries {first_block, n_blocks, delta}; blocks
 *               outside every entry are not rotated; where entries overlap,
 *               the last one covering a block applies; |delta| < 2^18.
 * out_dev       float32 [n_seq][n_q_heads][head_dim]; an empty context
 *               (seq_len 0) yields zeros.
 * ws            kvs_workspace_size(KVS_OP_DECODE_ATTN) bytes of device memory.
 * Requires n_q_heads % num_kv_heads == 0 and a group of at most 16 query
 * heads per KV head; BF16 pools.
 * Two implementations, chosen from the call's shape on the host: groups of
 * 9-16 heads, and small calls (n_seq * num_kv_heads * max_blocks <= 2048)
 * with groups <= 8, run one kernel per layer with no plan; larger calls with
 * groups <= 8 run the planned token-major path (blocks that a group of
 * sequences shares are computed once for the group).  The results agree to
 * rounding. */
typedef struct { int32_t first_block, n_blocks, delta, reserved; } kvs_seg_rope;
kvs_status kvs_decode_attn(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                           const int32_t* block_table_dev, int32_t max_blocks,
                           const int32_t* seq_len_dev, int32_t n_seq,
                           const int32_t* diff_table_dev,
                           const int32_t* rope_off_dev, const kvs_seg_rope* rope_segs_dev,
                           float theta, float scale, float* out_dev,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* The same attention split in two steps so that the per-step work plan is
 * built once and reused by every layer (block tables change per decode step,
 * not per layer).  kvs_decode_plan writes the plan into ws (sized by
 * kvs_workspace_size(KVS_OP_DECODE_ATTN)): for query groups G <= 8 it records,
 * for groups of R = 8/G sequences (R = 1 when rope_off is given), which
 * logical blocks every member that reaches them holds in the same physical
 * block, the RoPE shift of every logical block (when rope_off is given: the
 * last rope_segs entry covering the block; |delta| >= 2^18 sets
 * KVS_DEVERR_ROPE_RANGE and that block is not rotated), and lists the work
 * items.  kvs_decode_attn_planned then runs one layer with arguments that
 * must match the plan's call (same tables, seq_len, n_seq, max_blocks,
 * n_q_heads, diff table and RoPE segments); a mismatch in shapes is detected
 * on the device (KVS_DEVERR_PLAN, no output written), a change of table or
 * segment contents without a new plan is not.
 * kvs_decode_attn is kvs_decode_plan followed by kvs_decode_attn_planned.
 * Groups of more than 8 query heads, and small calls, need no plan (the calls
 * accept them and kvs_decode_plan writes nothing). */
kvs_status kvs_decode_plan(kvs_pool* pool, int32_t n_q_heads, const int32_t* block_table_dev,
                           int32_t max_blocks, const int32_t* seq_len_dev, int32_t n_seq,
                           const int32_t* diff_table_dev, const int32_t* rope_off_dev,
                           const kvs_seg_rope* rope_segs_dev, void* ws, size_t ws_bytes,
                           cudaStream_t stream);
kvs_status kvs_decode_attn_planned(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                                   const int32_t* block_table_dev, int32_t max_blocks,
                                   const int32_t* seq_len_dev, int32_t n_seq,
                                   const int32_t* diff_table_dev,
                                   const int32_t* rope_off_dev, const kvs_seg_rope* rope_segs_dev,
                                   float theta, float scale, float* out_dev,
                                   void* ws, size_t ws_bytes, cudaStream_t stream);

/* Decode attention reading a Q4G64 pool directly, dequantising in registers
 * ([Q4] §2.2), with optional mirror diffs over the Q4 master ([TD] section 3,
 * Fig. 8: a mirror is the master plus block-sparse K/V differences, restored
 * inside the read):
 *   out[a][h] = sum_t softmax_t(scale * <q[a][h], K^_a[t] + DK>) (V^_a[t] + DV)
 * with K^, V^ the dequantised codes (scale * code + bias) and DK, DV the
 * agent's diff rows for token t (zero where it has none).  Q4 pools keep
 * their diffs per 16-token sub-block of a 256-token block (the bf16 pool's
 * block size, so a refreshed position dirties 16 rows, not 256):
 * diff_table_dev  int32 [n_seq][max_blocks * 16] (16-byte aligned): entry
 *               [a][t / 16] is the diff sub-block holding token t's K and V
 *               differences at row t % 16 of the pool's dk / dv slabs
 *               (bf16 [diff_capacity_blocks][num_kv_heads][16][head_dim]), or
 *               -1; NULL for no diffs.  Ids >= diff_capacity_blocks set
 *               KVS_DEVERR_DIFF_ID and are ignored.
 * Every finite bf16 query is accepted (each query row is scaled by a power of
 * two before the fp16 tensor-core products and the factor is folded back
 * into its scores).  Other arguments as kvs_decode_attn; no rotation. */
kvs_status kvs_decode_attn_q4(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                              const int32_t* block_table_dev, int32_t max_blocks,
                              const int32_t* seq_len_dev, int32_t n_seq,
                              const int32_t* diff_table_dev, float scale, float* out_dev,
                              void* ws, size_t ws_bytes, cudaStream_t stream);

/* Quantise bf16 K/V blocks into a Q4G64 pool ([Q4] §2.1).  k_src/v_src are
 * bf16 [n_blocks][num_kv_heads][block_tokens][head_dim]; block i is written to
 * physical block dst_blocks_dev[i] of `layer`.  Per 64-element group:
 * scale = fp16((max-min)/15), bias = fp16(min) (float32 arithmetic),
 * code = clamp(rint((x - bias)/scale), 0, 15), scale 0 -> code 0. */
kvs_status kvs_quantize_q4(kvs_pool* pool, int32_t layer, const void* k_src_dev,
                           const void* v_src_dev, const int32_t* dst_blocks_dev,
                           int32_t n_blocks, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Mirror construction from refreshed critical positions ([TD] section 2: at
 * the check layers only each request's critical positions of its cached K/V
 * are refreshed; section 3, Fig. 7: one master cache, every other cache kept
 * as block-sparse K/V differences from it; Fig. 8: a diff is applied before
 * the RoPE positions are restored, so it lives in the master's frame).
 * For agent a, idx_dev[idx_off_dev[a] .. idx_off_dev[a+1]) are logical token
 * positions of its sequence, strictly ascending and < seq_len[a]; row r of
 * k_new_dev / v_new_dev (bf16 [rows][num_kv_heads][head_dim]) holds the
 * refreshed values of position idx_dev[r], K in the agent's frame.  The master
 * value of position t is row t % block_tokens of physical block
 * block_table[a][t / block_tokens] of `layer`.
 * Writes diff_table_dev (int32 [n_seq][max_blocks]): -1 for a block with no
 * refreshed position, else its diff block id; ids are consecutive from 0 in
 * agent order, then logical-block order, and *n_diff_dev (device int32)
 * receives their number.  Each dirty block's tiles in the pool's diff slabs of
 * `layer` get, on a refreshed row, bf16(R(-delta) k_new - K_master) and
 * bf16(v_new - V_master) (delta: the RoPE shift of the block's segment as in
 * kvs_decode_attn, 0 without rope_off_dev), and zero on every other row.
 * Those diff slabs then serve kvs_decode_attn as the agent's mirror diffs.
 * Device-detected errors: a position out of order or out of range
 * (KVS_DEVERR_JOB, the row is ignored), a block id out of range
 * (KVS_DEVERR_BLOCK_ID, the block's tiles are zeroed), more dirty blocks than
 * diff_capacity_blocks (KVS_DEVERR_DIFF_ID, the excess is not written).
 * ws: kvs_workspace_size(KVS_OP_MIRROR) bytes.  BF16 pools with diff slabs. */
kvs_status kvs_mirror_build(kvs_pool* pool, int32_t layer, const int32_t* block_table_dev, int32_t max_blocks,
                            const int32_t* seq_len_dev, int32_t n_seq, const int32_t* idx_dev,
                            const int64_t* idx_off_dev, const void* k_new_dev, const void* v_new_dev,
                            const int32_t* rope_off_dev, const kvs_seg_rope* rope_segs_dev, float theta,
                            int32_t* diff_table_dev, int32_t* n_diff_dev, void* ws, size_t ws_bytes,
                            cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Block lifetime: copy-on-write and sequence release ([INMS] §2.2: shared
 * blocks are read-only; a sequence about to write into a block that others
 * also reference gets a private copy, the old block's reference count drops,
 * otherwise it writes in place; §3.3: destroying a sequence decrements the
 * counts of its blocks and reclaims what becomes unused; §5.3: a missed
 * release leaks).  State, all caller-owned device memory: refcount_dev int32
 * [capacity] (as kvs_fingerprint_dedup writes it), a free stack free_ids_dev
 * int32 [capacity] with n_free_dev int32 [1] (entries [0, n_free), the top at
 * n_free - 1).  Blocks are pushed in descending id order, so the smallest id
 * is on top and taken first.  A block of sequence a is referenced at logical
 * block b < ceil(seq_len[a] / block_tokens).  ws: kvs_workspace_size(
 * KVS_OP_BLOCKS, n_items = max(n_writes, n_seq)) bytes.
 *
 * kvs_blocks_init_free: the stack = every block whose count is 0.
 *
 * kvs_block_write: applies the writes w = 0 .. n_writes-1 in list order, each
 * to logical block write_block[w] of sequence write_seq[w], with the pages'
 * write_to_block rule: when the block's count is above 1 the sequence takes
 * the block on top of the stack, every layer's K and V (Q4: codes and
 * scale/bias) of the old block are copied into it, its count becomes 1, the
 * old one's drops by 1 and the table entry is redirected; otherwise nothing
 * changes (the caller writes in place).  A write whose (sequence, block)
 * appeared earlier in the batch targets the private copy made then.  An empty
 * stack leaves the write on the shared block (KVS_DEVERR_CAPACITY); a bad
 * sequence/block index (KVS_DEVERR_JOB) or table entry (KVS_DEVERR_BLOCK_ID)
 * skips the write.
 *
 * kvs_seq_release: for every sequence listed (duplicates count once),
 * decrements the counts of its referenced blocks, sets its table row to -1
 * and seq_len to 0; the blocks that reached 0 are pushed.  A count going
 * below zero sets KVS_DEVERR_REFCOUNT. */
kvs_status kvs_blocks_init_free(kvs_pool* pool, const int32_t* refcount_dev, int32_t* free_ids_dev,
                                int32_t* n_free_dev, void* ws, size_t ws_bytes, cudaStream_t stream);
kvs_status kvs_block_write(kvs_pool* pool, int32_t* block_table_dev, int32_t max_blocks, int32_t n_seq,
                           const int32_t* write_seq_dev, const int32_t* write_block_dev, int32_t n_writes,
                           int32_t* refcount_dev, int32_t* free_ids_dev, int32_t* n_free_dev, void* ws,
                           size_t ws_bytes, cudaStream_t stream);
kvs_status kvs_seq_release(kvs_pool* pool, int32_t* block_table_dev, int32_t max_blocks, int32_t* seq_len_dev,
                           int32_t n_seq, const int32_t* release_seq_dev, int32_t n_release,
                           int32_t* refcount_dev, int32_t* free_ids_dev, int32_t* n_free_dev, void* ws,
                           size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Block-granular eviction scoring ([MD] §3.2: a token's current score is its
 * region's initial score times exp(-decay * (step - created)); §4.1 scoring
 * code: times (1 + 0.1 ln(1 + access)) when access > 0; §5.3: whole blocks
 * are evicted, judged by the mean score of their tokens; lowest first).
 * region_dev uint8, created_dev int32, access_dev int32: per logical token,
 * [n_seq][max_blocks * block_tokens] (token t of sequence a at
 * a * max_blocks * block_tokens + t); only t < seq_len[a] is read.
 * init / decay: host arrays of n_regions (1..16) finite non-negative floats.
 * Writes scores_dev (float [n_seq][max_blocks]: the mean score of each
 * logical block holding a stored token, +inf past the sequence's blocks) and,
 * for every sequence, the min(k_dev[a], blocks) lowest-scored logical blocks
 * (ties: the lower block index) in ascending order into victims_dev, with
 * offsets victims_off_dev int64 [n_seq + 1].  Scores are float32; a region id
 * >= n_regions scores 0 and sets KVS_DEVERR_JOB.  block_tokens <= 16. */
kvs_status kvs_evict_score(kvs_pool* pool, const uint8_t* region_dev, const int32_t* created_dev,
                           const int32_t* access_dev, const int32_t* seq_len_dev, int32_t n_seq, int32_t max_blocks,
                           const float* init, const float* decay, int32_t n_regions, int64_t step,
                           const int32_t* k_dev, float* scores_dev, int32_t* victims_dev, int64_t* victims_off_dev,
                           cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Block export / import ([Q4] §2.1: each agent's cache is kept as fixed-size
 * Q4 blocks in a persistent file and survives restarts; §2.2: the blocks are
 * loaded straight back into attention, without re-prefill; the file itself
 * is the caller's).  A packed record of one physical block holds, layer by
 * layer, its K then V bytes (Q4 pools: K codes, V codes, K scale/bias,
 * V scale/bias), each as stored in the slab; kvs_pool_block_bytes gives the
 * record size.  kvs_pool_export writes the records of blocks_dev[0 ..
 * n_blocks) to dst_dev in list order; kvs_pool_import writes records from
 * src_dev into those blocks (e.g. blocks taken off the free stack).  Buffers
 * are device memory, 16-byte aligned, >= n_blocks records; a block id out of
 * range sets KVS_DEVERR_BLOCK_ID and is skipped. */
kvs_status kvs_pool_block_bytes(const kvs_pool* pool, size_t* bytes);
kvs_status kvs_pool_export(kvs_pool* pool, const int32_t* blocks_dev, int32_t n_blocks, void* dst_dev,
                           size_t dst_bytes, cudaStream_t stream);
kvs_status kvs_pool_import(kvs_pool* pool, const int32_t* blocks_dev, int32_t n_blocks, const void* src_dev,
                           size_t src_bytes, cudaStream_t stream);

/* Test-only switches.  KVS_TEST_STALL_ONE_STAGE: the next kvs_decode_attn /
 * kvs_decode_attn_planned launch with a query group <= 8 leaves one ring
 * stage of one warp unarmed, so that warp's bounded wait runs out (about a
 * second); it records KVS_DEVERR_WAIT_TIMEOUT, waits briefly for its other
 * copies in flight and stops, leaving the CUDA context usable.  The flag is
 * consumed by that launch.  It exists to test the timeout path without a
 * device fault; nothing else sets it. */
#define KVS_TEST_STALL_ONE_STAGE 0x1u
/* KVS_TEST_TOKEN_MAJOR: while set, every kvs_decode_attn / kvs_decode_plan /
 * kvs_decode_attn_planned call with a query group <= 8 takes the planned
 * token-major path, also below the small-call bound (see kvs_decode_attn),
 * so that tests can run that path on small inputs.  It stays set until
 * kvs_pool_set_test_flags clears it.  Results agree between the two paths to
 * rounding. */
#define KVS_TEST_TOKEN_MAJOR 0x2u
kvs_status kvs_pool_set_test_flags(kvs_pool* pool, uint32_t flags);

/* Workspace bytes for an operation with the given call shape. */
#define KVS_OP_DEDUP 0
#define KVS_OP_DECODE_ATTN 1
#define KVS_OP_DECODE_ATTN_Q4 2
#define KVS_OP_SELECT 3
#define KVS_OP_MIRROR 4
#define KVS_OP_BLOCKS 5   /* n_seq = n_items = max(n_writes, n_seq); max_blocks unused */
kvs_status kvs_workspace_size(const kvs_pool* pool, int32_t op, int32_t n_seq,
                              int32_t max_blocks, int32_t n_q_heads, size_t* bytes);

/* Synchronise `stream`, read and clear the pool's device status word into
 * *flags (KVS_DEVERR_* bits).  Returns KVS_ERR_DEVICE_BOUNDS when any bit was
 * set, KVS_OK otherwise. */
kvs_status kvs_pool_check(kvs_pool* pool, cudaStream_t stream, uint32_t* flags);

/* Pool statistics from a dedup result: synchronises `stream`, copies the
 * refcounts back and reports unique (n_phys), shared (refcount > 1) blocks,
 * total references, and bytes a dense per-sequence layout would need versus
 * the pool — [INMS] §1.2 independent vs shared footprint. */
typedef struct {
  int64_t unique_blocks, shared_blocks, total_refs;
  int64_t pool_bytes, dense_bytes;
} kvs_stats;
kvs_status kvs_pool_stats(const kvs_pool* pool, const int32_t* refcount_dev,
                          const int32_t* n_phys_dev, cudaStream_t stream, kvs_stats* out);

/* Describes the last error raised on this host thread (never NULL). */
const char* kvs_last_error_string(void);

/* Number of kernels this library launched so far in this process. */
uint64_t kvs_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* KVS_H */
