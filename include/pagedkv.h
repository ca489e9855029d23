/*
 * pagedkv.h -- C ABI of libpagedkv.so: one engine step of attention over a
 * paged (block-tabled) KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The problem these calls solve is the one of a continuously batched serving
 * step.  The running requests form a ragged batch: each contributes one query
 * token (decode) or a chunk of query tokens (chunked prefill), flattened into
 * one [tokens, heads, head_dim] tensor with per-request offsets
 * (query_start_loc), the interface a variable-length attention kernel offers
 * (The Serving Playbook, "Continuous batching").  Each request's keys and
 * values live in fixed-size blocks of one shared pool, found through the
 * request's block table (The Serving Playbook, "Paged KV cache"; LLM 7 -
 * Efficient LLM Serving, sec. 3 "Paging the Cache").  A serving step first
 * writes this step's K/V into the cache through a slot mapping, then attends
 * (The Serving Playbook, "CUDA graphs and the CPU you forgot about", which
 * lists block tables and slot mappings among the preallocated step buffers).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Element type: bf16 for q, K/V rows, pools and out (pools hold e4m3 codes
 *   for pkv_append_fp8 / pkv_attention_fp8kv).  head_dim = 128 and
 *   block_size = 16 are the supported shapes; num_q_heads must be a multiple
 *   of num_kv_heads with a group size g = num_q_heads / num_kv_heads of 1..8.
 * - Layouts (row-major, contiguous):
 *     q, out        [num_q_tokens, num_q_heads, head_dim]
 *     k_new, v_new  [num_new_tokens, num_kv_heads, head_dim]
 *     k_pool,v_pool [num_blocks, num_kv_heads, block_size, head_dim]
 *                   -- one (block, KV head) pair is one contiguous 4 KiB tile
 *     block_tables  [num_reqs, max_blocks_per_req] int32
 *     seq_lens      [num_reqs] int32: L_r, INCLUDING this step's tokens
 *     query_start_loc [num_reqs + 1] int32: query rows of request r are
 *                   query_start_loc[r] .. query_start_loc[r+1]-1
 *     slot_mapping  [num_new_tokens] int64: block * block_size + offset
 * - Query head h reads KV head h / g.  Query i of request r (q_r queries)
 *   sits at position L_r - q_r + i and attends to keys 0 .. L_r - q_r + i.
 * - Ownership: every pointer is device memory owned by the caller; the
 *   library never frees or keeps it.  All calls are asynchronous on the given
 *   stream and never synchronise it (except pkv_get_device_error).
 * - All device pointers must be 16-byte aligned.
 * - Return codes: PKV_OK or a negative PKV_ERR_*; pkv_last_error() gives a
 *   message (thread-local).  Device-side violations (a block id outside the
 *   pool, inconsistent lengths) are skipped by the kernels and recorded in a
 *   per-device error word that pkv_get_device_error() reads and clears.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_OK 0
#define PKV_ERR_INVALID (-1)      /* null pointer, bad dims, misalignment */
#define PKV_ERR_UNSUPPORTED (-2)  /* head_dim, block_size, group size, too many requests */
#define PKV_ERR_WORKSPACE (-3)    /* workspace smaller than pkv_attention_workspace_size */
#define PKV_ERR_CUDA (-4)         /* a CUDA runtime call or launch failed */
#define PKV_ERR_DEVICE_BOUNDS (-5) /* reported later: block id or lengths out of range */
#define PKV_ERR_TIMEOUT (-6)      /* reported later: a bounded device wait ran out */

/* Upper bound on num_reqs for pkv_attention (every CTA scans the per-request
 * lengths to plan its share of the step). */
#define PKV_MAX_REQS 65536

typedef struct pkv_dims {
    int32_t num_reqs;           /* R */
    int32_t num_q_tokens;       /* Tq >= query_start_loc[R] (rows past it are padding) */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv */
    int32_t head_dim;           /* D, must be 128 */
    int32_t block_size;         /* bs, must be 16 */
    int32_t num_blocks;         /* physical blocks in each pool */
    int32_t max_blocks_per_req; /* columns of block_tables */
} pkv_dims;

/*
 * KV append (the step's cache write).  For each new token t with
 * slot_mapping[t] >= 0, copies k_new[t, :, :] into k_pool[slot / bs, :,
 * slot % bs, :] and v_new likewise, bit for bit.  Negative slots are padding
 * and are skipped.  A slot >= num_blocks * bs is skipped and recorded as
 * PKV_ERR_DEVICE_BOUNDS.  Duplicate slots are a caller error (the last writer
 * is unspecified).  Only dims->num_kv_heads, head_dim, block_size and
 * num_blocks are read.
 * Source: LLM 7 - Efficient LLM Serving, sec. 3 "What the Cache Stores" (the
 * new token's K and V join the cache each step); The Serving Playbook, "CUDA
 * graphs and the CPU you forgot about" (slot mappings as a step buffer).
 */
int pkv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping,
               void *k_pool, void *v_pool, int32_t num_new_tokens,
               const pkv_dims *dims, cudaStream_t stream);

/*
 * Whole-block copies between two pools of the same layout: for each pair i,
 * block pairs[2i] of (k_src, v_src) -- every KV head, K and V -- is copied to
 * block pairs[2i+1] of (k_dst, v_dst).  Source and destination may be the same
 * pool (copy-on-write of a shared block) or different pools; either side may
 * be pinned host memory that the device can address (swap out / swap in).
 * pairs: [num_pairs, 2] int64 in device-accessible memory.  Pairs naming a
 * block outside [0, src_num_blocks) / [0, dst_num_blocks) are skipped and
 * reported as PKV_ERR_DEVICE_BOUNDS; pairs must not overlap (no block is both
 * a source and a destination).  Only dims->num_kv_heads, head_dim and
 * block_size are read.
 * Source: LLM 7 - Efficient LLM Serving, sec. 3 "Sharing and Preemption"
 * (copy-on-write, swapping blocks to CPU memory); The Serving Playbook,
 * "Sharing is a reference count", "Preemption, where the folklore is wrong".
 */
int pkv_copy_blocks(const void *k_src, const void *v_src, void *k_dst, void *v_dst,
                    const int64_t *pairs, int32_t num_pairs, int32_t src_num_blocks,
                    int32_t dst_num_blocks, const pkv_dims *dims, cudaStream_t stream);

/*
 * Bytes of workspace pkv_attention needs for these dims (split-context
 * partial outputs, their log-sum-exp statistics and per-row merge counters).
 * Depends only on dims and the device's SM count, not on the lengths, so one
 * buffer serves every step of a captured CUDA graph.
 */
size_t pkv_attention_workspace_size(const pkv_dims *dims);

/*
 * Zeroes the merge counters at the head of a workspace (a stream-ordered
 * memset).  Call once after allocating a workspace, and again whenever the
 * workspace is reused with different num_q_tokens or num_kv_heads (the
 * counter region grows with them).  pkv_attention leaves the counters at zero
 * when it finishes, so calls with unchanged dims need no re-initialisation.
 * After a PKV_ERR_TIMEOUT report, initialise it again.
 */
int pkv_workspace_init(void *workspace, size_t workspace_bytes,
                       const pkv_dims *dims, cudaStream_t stream);

/*
 * Attention for one engine step.  For every request r and query i < q_r
 * (row t = query_start_loc[r] + i) and query head h:
 *     out[t, h, :] = sum_j softmax_j(scale * <q[t,h,:], K_r[j, h/g, :]>) V_r[j, h/g, :]
 * over keys j = 0 .. L_r - q_r + i, where K_r[j] = k_pool[block_tables[r,
 * j/bs], :, j%bs, :].  Computed with fp32 accumulation and an online softmax;
 * long contexts are split across CTAs and merged by log-sum-exp (Flash-
 * Decoding); prefill chunks, and decode rows of groups of 4 or more query
 * heads per KV head, run on tcgen05 tensor cores (their probabilities enter
 * the PV product in bf16).  out is written as
 * bf16 (round to nearest even).  Requests with q_r = 0 produce nothing.
 * Preconditions: query_start_loc[0] = 0, non-decreasing, last entry <=
 * num_q_tokens; 0 <= q_r <= L_r <= max_blocks_per_req * bs; table entries
 * b < ceil(L_r / bs) are in [0, num_blocks).  Violations found on the device
 * skip the affected work and are reported by pkv_get_device_error.
 * Padded (bucketed) steps: a CUDA graph captured for a bucket of R requests
 * and Tq query rows serves any step that fits in it, its buffers rewritten in
 * place between replays.  Pad the unused requests with q_r = 0 (their
 * query_start_loc entries repeat the last live one) and L_r = 0; their table
 * rows are not read.  Rows query_start_loc[R] .. num_q_tokens - 1 of out are
 * padding: no call writes them.  Give padding rows slot -1 in a slot mapping.
 * workspace: at least pkv_attention_workspace_size(dims) bytes, initialised
 * once with pkv_workspace_init; NULL makes the library use an internal
 * per-device buffer (allocated on first use: not capturable in a CUDA graph,
 * and not safe for concurrent calls on different streams).
 * Launch overlap: unless pkv_options.pdl is 0, the kernels are launched
 * with programmatic dependent launch and may start while the kernel before
 * them on the stream is still running.  They wait for it before touching q,
 * the pools, out or the workspace, but read seq_lens, query_start_loc and
 * (in the tensor-core decode) block_tables before that wait
 * (pkv_options.early_plan = 0 moves those reads after it).  So the kernel issued
 * immediately before this call must not write seq_lens, query_start_loc or
 * block_tables; pkv_append, which writes only pool slots, and host-to-device
 * copies may.
 * Source: The Serving Playbook, "The block table lives in the hottest kernel
 * in the system" (gather through the table, partial softmax per piece of the
 * cache, rescaling pass), "Kernel fusion, briefly" (Flash-Decoding splits the
 * KV axis), "Chunked prefill" (causal chunk over earlier chunks' KV); LLM 7,
 * sec. 2 "Online Softmax Makes Tiling Possible".
 */
int pkv_attention(const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *block_tables, const int32_t *seq_lens,
                  const int32_t *query_start_loc, float scale, void *out,
                  const pkv_dims *dims, void *workspace, size_t workspace_bytes,
                  cudaStream_t stream);

/*
 * One layer of an engine step: pkv_append of this step's dims->num_q_tokens
 * new tokens, then pkv_attention over the updated pools -- the same results
 * as the two calls in that order, with the same arguments, preconditions and
 * errors.  Additional precondition: slot_mapping[t] for t = query_start_loc[r]
 * + i is either negative (padding) or the slot of position L_r - q_r + i of
 * request r through its block table, i.e. the append writes no pool slot that
 * holds an earlier position.  Because of it the attention kernel does not
 * wait for the append before streaming the K/V tiles that hold only earlier
 * positions (nor before reading q and block_tables); it waits only before the
 * first tile of a row that holds one of the new tokens, so the append's
 * latency hides behind the gather (with pkv_options.pdl or .early_kv = 0 the
 * two run back to back instead).  pkv_options.early_trigger = 1 also lets the
 * attention kernel launch as soon as the append starts; it then reads q and writes
 * out and the workspace only after the append has finished, and the kernel
 * issued before this call must not write seq_lens, query_start_loc,
 * block_tables or pool slots of earlier positions either.
 * Source: LLM 7 - Efficient LLM Serving, sec. 3 "What the Cache Stores" (the
 * step appends each new token's K and V, then attends over the cache); The
 * Serving Playbook, "The block table lives in the hottest kernel in the
 * system".
 */
int pkv_append_attention(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                         void *k_pool, void *v_pool, const void *q,
                         const int32_t *block_tables, const int32_t *seq_lens,
                         const int32_t *query_start_loc, float scale, void *out,
                         const pkv_dims *dims, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * KV append into e4m3 pools (8-bit float: 1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits, largest finite magnitude 448).  Same slots, padding and
 * bounds rules as pkv_append; k_pool / v_pool are [num_blocks, Hkv, bs, 128]
 * bytes.  Element x of head h becomes the code nearest to x / k_scale[h]
 * (v_scale[h] for V), the quotient taken in fp32 with round to nearest even,
 * ties to the even code, magnitudes beyond 448 saturated to +-448.  k_scale /
 * v_scale: [num_kv_heads] positive finite fp32 in device memory (per layer:
 * pass that layer's scales).  k_new / v_new are bf16 as in pkv_append.
 * Source: The Serving Playbook, "Quantized serving" (an fp8 KV cache halves
 * the bytes decode reads); What Actually Runs the Model, "The KV cache".
 */
int pkv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                   void *k_pool, void *v_pool, const float *k_scale, const float *v_scale,
                   int32_t num_new_tokens, const pkv_dims *dims, cudaStream_t stream);

/*
 * pkv_attention over e4m3 pools written by pkv_append_fp8: the key of
 * position j, KV head kh, is decode(code) * k_scale[kh], the value
 * decode(code) * v_scale[kh]; everything else (q, out, lengths, tables,
 * workspace, errors) as in pkv_attention.  All rows, prefill chunks
 * included, run in the split-context decode kernels (the tensor-core prefill
 * kernel takes bf16 pools only); with 4 or more query heads per KV head that
 * is the tensor-core decode, which widens the codes to f16 in shared memory
 * and takes q and the probabilities in f16 (q rounded from bf16 to f16).
 * Source: as pkv_attention; The Serving Playbook, "Quantized serving".
 */
int pkv_attention_fp8kv(const void *q, const void *k_pool, const void *v_pool,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_tables, const int32_t *seq_lens,
                        const int32_t *query_start_loc, float scale, void *out,
                        const pkv_dims *dims, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/*
 * One layer of an engine step over e4m3 pools: pkv_append_fp8 of this step's
 * dims->num_q_tokens new tokens, then pkv_attention_fp8kv over the updated
 * pools -- the same results as the two calls in that order, with the same
 * arguments, preconditions and errors, and the slot-mapping precondition of
 * pkv_append_attention (slot_mapping[t] for t = query_start_loc[r] + i is
 * negative or the slot of position L_r - q_r + i of request r), under which
 * the attention streams the tiles holding only earlier positions before the
 * append finishes (pkv_options.early_kv, .early_trigger as there).
 * Source: as pkv_append_attention; The Serving Playbook, "Quantized serving".
 */
int pkv_append_attention_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             void *k_pool, void *v_pool, const float *k_scale,
                             const float *v_scale, const void *q,
                             const int32_t *block_tables, const int32_t *seq_lens,
                             const int32_t *query_start_loc, float scale, void *out,
                             const pkv_dims *dims, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/*
 * Bytes of workspace pkv_attention_cascade needs for these dims: the
 * pkv_attention workspace (same head, initialised the same way with
 * pkv_workspace_init), plus partial states for up to 8 chunks of each shared
 * prefix per (query token, query head), plus an int per request.
 */
size_t pkv_cascade_workspace_size(const pkv_dims *dims);

/*
 * pkv_attention for a batch whose requests share prompts (shared-prefix,
 * "cascade" attention).  The result is pkv_attention's; the shared blocks
 * are read once per batch instead of once per request.
 * Groups (device arrays, num_groups entries): group g is the requests
 * group_first_req[g] .. group_first_req[g] + group_num_reqs[g] - 1 (a
 * contiguous run; groups must not overlap), whose first
 * group_prefix_blocks[g] block-table entries name the same physical blocks.
 * Every member must have all of its query tokens after the shared prefix
 * (L_r - q_r >= 16 * group_prefix_blocks[g]); a member that does not reads
 * its whole context itself.  Entries naming requests outside [0, num_reqs)
 * are skipped and reported as PKV_ERR_DEVICE_BOUNDS.
 * How: one pass attends every member's query rows to the group's shared
 * blocks at once on the tensor cores (rows = the members' (token, head)
 * pairs; the shared keys split into up to 8 chunks of 128-key tiles, one
 * work item each) and keeps a partial state per row and chunk; the decode
 * then reads each row's remaining blocks and merges them by log-sum-exp.  Every row runs in the
 * decode path (no separate prefill kernel).  Sharing applies when the step
 * runs the tensor-core decode (bf16 pools, 4..8 query heads per KV head);
 * otherwise the call computes the same result without it.
 * workspace: caller-owned, at least pkv_cascade_workspace_size(dims) bytes.
 * Source: The Serving Playbook, "The tree changes what the scheduler should
 * do" (requests batched with a shared prefix read the same KV blocks, which
 * can then be fetched from HBM once per batch); LLM 7 - Efficient LLM
 * Serving, sec. 3 "Sharing and Preemption" (many block tables point at one
 * set of physical prefix blocks); sec. 2 "Online Softmax Makes Tiling
 * Possible" (merging partial softmax states).
 */
int pkv_attention_cascade(const void *q, const void *k_pool, const void *v_pool,
                          const int32_t *block_tables, const int32_t *seq_lens,
                          const int32_t *query_start_loc, const int32_t *group_first_req,
                          const int32_t *group_num_reqs, const int32_t *group_prefix_blocks,
                          int32_t num_groups, float scale, void *out, const pkv_dims *dims,
                          void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Size of the static scratch array behind pkv_attention_noalloc (4 MiB). */
#define PKV_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)

/*
 * pkv_attention without a workspace and without any allocation.  The paper
 * has no counterpart: this is a convenience of the library.
 *
 * For callers that cannot allocate device memory -- plugins whose host
 * framework owns all device memory through its own pool, serving loops that
 * forbid allocation after start-up -- and so cannot pass pkv_attention a
 * workspace.  Same arguments, results and error codes as pkv_attention; the
 * split-context scratch comes from a PKV_NOALLOC_SCRATCH_BYTES array compiled
 * into the library, which every GPU that loads the library holds until the
 * process exits.  Dims needing more scratch than that
 * (pkv_attention_workspace_size) return PKV_ERR_WORKSPACE.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Each call clears the head of the array (merge counters, prefill
 * work queue, plan cache) with a stream-ordered memset and leaves other
 * contents from earlier calls in place; so these calls make their plan
 * afresh every time, and the memset keeps the attention kernel from
 * overlapping the kernel before it.  All calls share the one array: calls
 * that overlap on the GPU (two streams, two host threads) race and must be
 * serialised by the caller.
 * Never calls cudaMalloc, cudaFree or any allocating routine.
 */
int pkv_attention_noalloc(const void *q, const void *k_pool, const void *v_pool,
                          const int32_t *block_tables, const int32_t *seq_lens,
                          const int32_t *query_start_loc, float scale, void *out,
                          const pkv_dims *dims, cudaStream_t stream);

/*
 * Launch and routing options (process-wide).  The defaults are the measured
 * best.  Each field can also be set by the environment variable named beside
 * it, read once, when a call of this library first needs the options; after
 * that, pkv_set_options is the only way to change them.  Every call takes a
 * copy of the options when it starts; change them only while no other host
 * thread is inside a call of this library.  None of them changes a result
 * beyond rounding: they choose kernels, launch overlap and work splits.
 */
typedef struct pkv_options {
    int32_t pdl;            /* PKV_PDL (1): programmatic dependent launch between the
                               library's kernels (see pkv_attention) */
    int32_t early_plan;     /* PKV_EARLY_PLAN (1): decode plans read seq_lens,
                               query_start_loc (and block_tables) before the launch wait */
    int32_t early_kv;       /* PKV_EARLY_KV (1): pkv_append_attention streams K/V tiles
                               without this step's tokens before the append finishes */
    int32_t early_trigger;  /* PKV_EARLY_TRIGGER (0): pkv_append_attention's append lets
                               the attention launch at once */
    int32_t plan_cache;     /* PKV_PLAN_CACHE (1): per-CTA plan cache in the workspace */
    int32_t decode_tc;      /* PKV_DECODE_TC (1): tensor-core decode for 4..8 query heads
                               per KV head (0: the SIMT decode for every group) */
    int32_t decode_tc_fp8;  /* PKV_DECODE_TC_FP8 (1): the same for e4m3 pools */
    int32_t prefill_min_q;  /* PKV_PREFILL_MIN_Q (16): requests with at least this many
                               query tokens run in the tensor-core prefill kernel
                               (0: none do); bf16 pools only */
    int32_t align;          /* PKV_ALIGN (1): with uniform row-groups, snap decode ranges
                               to row-group boundaries ... */
    int32_t align_slack;    /* PKV_ALIGN_SLACK (64): ... when that lengthens every range
                               by at most this many blocks */
    int32_t min_chunk;      /* PKV_MIN_CHUNK (4): smallest decode range per CTA, in
                               blocks (>= 1) */
    int32_t decode_grid;    /* PKV_DECODE_GRID (0): decode grid in CTAs (0: the
                               default for the kernel and group size; tuning only,
                               at most twice the SM count) */
    int32_t wait_limit_us;  /* PKV_WAIT_LIMIT_US (2000000): a bounded device wait gives
                               up after this many microseconds and reports
                               PKV_ERR_TIMEOUT (>= 1) */
    int32_t debug_withhold_q; /* testing only (0): the tensor-core decode never loads q,
                               so its waits run out after wait_limit_us; exercises
                               the timeout path.  Results are not computed. */
    int32_t rowgroup_cost;  /* PKV_ROWGROUP_COST (16): when the decode plan cuts the
                               step into equal per-CTA ranges, every (query row, KV
                               head) counts as its 16-token blocks plus this many,
                               the fixed cost of a piece (0..1024) */
} pkv_options;

/* Copies the current options into *opts. */
void pkv_get_options(pkv_options *opts);

/* Replaces the options; PKV_ERR_INVALID (nothing changed) if a field is out
 * of range. */
int pkv_set_options(const pkv_options *opts);

/* Message of the last failing call on this thread ("" if none). */
const char *pkv_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns PKV_OK, PKV_ERR_DEVICE_BOUNDS, PKV_ERR_TIMEOUT (a timeout
 * takes precedence) or PKV_ERR_CUDA.
 */
int pkv_get_device_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
