// pkv_internal.h -- kernel parameter blocks and launchers shared between the
// host ABI (pkv_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv_common.cuh"

struct pkv_dims;  // include/pagedkv.h

namespace pkv {

// Device ordinals the library keeps per-device state for (0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;

struct AppendParams {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int64_t* slot_mapping;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  int* err;
  int num_tokens;
  int num_kv_heads;
  int num_blocks;
  int pdl;  // launch with programmatic stream serialization
  // Let the next kernel (an attention kernel that reads only blocks without
  // these tokens before its own wait) launch before this one's wait.
  int early_trigger;
};

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// Whole-block copies between two pools (device or mapped host memory).
struct CopyParams {
  const __nv_bfloat16* k_src;
  const __nv_bfloat16* v_src;
  __nv_bfloat16* k_dst;
  __nv_bfloat16* v_dst;
  const int64_t* pairs;  // [num_pairs, 2]: (source block, destination block)
  int* err;
  int num_pairs;
  int num_kv_heads;
  long long src_blocks;
  long long dst_blocks;
  int pdl;
};

cudaError_t launch_copy_blocks(const CopyParams& p, int sm_count, cudaStream_t stream);

// Split-context decode: the device plan, the paged gather, the online
// softmax, and the log-sum-exp merge, in one launch.
struct DecodeParams {
  const __nv_bfloat16* q;
  const uint8_t* k_pool;   // bf16 or e4m3 elements, [num_blocks, Hkv, 16, 128]
  const uint8_t* v_pool;
  const float* k_scale;    // e4m3 pools: [Hkv] dequantisation scales (else unused)
  const float* v_scale;
  int kv_fp8;              // 1: the pools hold e4m3 codes
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  __nv_bfloat16* out;
  int* ws_cnt;    // [num_q_tokens * num_kv_heads] merge counters, zero between calls
  float* ws_ml;   // [num_slots, g, 2] (max, normaliser) of each partial piece, log2 domain
  float* ws_o;    // [num_slots, g, 128] normalised partial output of each piece
  int* err;
  int num_reqs;
  int num_q_tokens;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int max_blocks;
  float scale_log2;   // scale * log2(e)
  int prefill_min_q;  // requests with q_r >= this are left to the prefill kernel
  int num_slots;      // partial-piece slots in the workspace (>= 2 * grid)
  int min_chunk;      // smallest per-CTA range, in blocks
  int align;          // snap ranges to row-group boundaries when lengths are uniform
  int align_slack;    // ... if that lengthens the per-CTA range by at most this many blocks
  int early_plan;     // plan from seq_lens / query_start_loc before the PDL wait
  // If the step has at most this many blocks per CTA of half the grid, only
  // the first half of the grid takes work (0: the whole grid always does).
  int half_grid_blocks;
  // The kernel before this one on the stream is the append of exactly this
  // step's new tokens (positions L - q_r .. L - 1 of each request): q, the
  // block table and every K/V tile holding none of those positions are read
  // before the PDL wait, which is taken only before the first tile that does.
  int early_kv;
  // With early_kv: the append waited for its own predecessor before letting
  // this kernel launch, so q, out and the workspace are free as well (else
  // they wait for the append like the tiles with new tokens).
  int early_q;
  // Per-CTA plan cache in the workspace (see pkv_plan.cuh), or null.
  int* plan_cache;
  int plan_entries;
  // Shared-prefix (cascade) calls: the first table column each request reads
  // ([R], or null), and the prefix pass's partial states to merge
  // ([Tq, Hq, 128] normalised outputs and [Tq, Hq] (max, normaliser)).
  const int32_t* first_block;
  const float* pre_o;
  const float* pre_ml;
  int pdl;            // launch with programmatic stream serialization
  unsigned long long wait_limit_ns;  // bounded device waits give up after this long
  // Testing only: the tensor-core decode's producer arms the first piece's
  // q barrier but never issues its copy, so the waits on it run out.
  int debug_withhold_q;
  // Blocks' worth of work a piece costs beyond its blocks (its epilogue and
  // partial last tile): added to every row-group's length when the plan
  // cuts the CTAs' ranges.
  int rowgroup_cost;
};

// Workspace carve-up shared by the host code that sizes it and the launcher.
// Decode plans are cached for steps of up to kPlanCacheReqs requests, one
// entry of kPlanEntryWords int32 words per CTA index.
constexpr int kPlanCacheReqs = 256;
constexpr int kPlanEntryWords = 576;

struct WorkspaceLayout {
  size_t cnt_off, sched_off, plan_off, ml_off, o_off, total;
  int num_slots, plan_entries;
};

WorkspaceLayout decode_workspace_layout(int num_q_tokens, int num_kv_heads, int group,
                                        int sm_count);

int decode_grid(int sm_count, int group);

cudaError_t launch_decode(const DecodeParams& p, int group, int grid, cudaStream_t stream);
cudaError_t launch_decode_e4m3(const DecodeParams& p, int group, int grid, cudaStream_t stream);

// The same decode on tcgen05 tensor cores (bf16 pools, groups of 4..8).
struct DecodeTcLaunch {
  CUtensorMap qmap;  // q as [tokens][Hq][128], box (64, g, 1)
  CUtensorMap kmap;  // k_pool as [blocks*Hkv*16][128], box (64, 16), 128-byte swizzle
  CUtensorMap vmap;  // v_pool, same
  DecodeParams p;
  int grid;
};

cudaError_t launch_decode_tc(const DecodeTcLaunch& L, int group, cudaStream_t stream);

// Quantising KV append into e4m3 pools.
struct AppendFp8Params {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int64_t* slot_mapping;
  uint8_t* k_pool;
  uint8_t* v_pool;
  const float* k_scale;  // [Hkv]
  const float* v_scale;
  int* err;
  int num_tokens;
  int num_kv_heads;
  int num_blocks;
  int pdl;
  int early_trigger;  // as AppendParams::early_trigger
};

cudaError_t launch_append_fp8(const AppendFp8Params& p, cudaStream_t stream);

// Chunked-prefill attention on tcgen05 tensor cores (requests with
// q_r >= prefill_min_q).
struct PrefillParams {
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  __nv_bfloat16* out;
  int* err;
  int num_reqs;
  int num_q_tokens;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int max_blocks;
  float scale_log2;
  int prefill_min_q;
  int pdl;
  // Prefix pass of a shared-prefix (cascade) call: the work units are the
  // sharing groups -- all query tokens of a group's members (contiguous
  // requests) against the group's leading shared blocks, with no causal
  // mask -- and the output is each row's partial state, not `out`.
  int prefix_mode;
  const int32_t* grp_first;   // [num_groups] first member request
  const int32_t* grp_count;   // [num_groups] members
  const int32_t* grp_blocks;  // [num_groups] shared leading blocks
  int num_groups;
  float* pre_o;               // [Tq, Hq, 128] normalised partial outputs
  float* pre_ml;              // [Tq, Hq, 2] (max in log2 units, normaliser)
  // Work queue: [0] next item, [1] CTAs done; zero between launches (the
  // last CTA to finish resets both).
  unsigned long long* sched;
  unsigned long long wait_limit_ns;  // bounded device waits give up after this long
};

// Shared-prefix (cascade) prefix pass: a group's shared keys (L of them) are
// split into at most kPrefixSplits chunks of whole 128-key tiles, one work
// item each, so that a few groups still spread over many SMs; each chunk
// leaves its own partial state ([kPrefixSplits, Tq, Hq] slots).
#ifndef PKV_PREFIX_SPLITS
#define PKV_PREFIX_SPLITS 8
#endif
constexpr int kPrefixSplits = PKV_PREFIX_SPLITS;
constexpr int kPrefixTile = 128;
__host__ __device__ inline int prefix_chunk_tiles(int L) {
  const int tiles = (L + kPrefixTile - 1) / kPrefixTile;
  return (tiles + kPrefixSplits - 1) / kPrefixSplits;
}
__host__ __device__ inline int prefix_chunks(int L) {
  const int tiles = (L + kPrefixTile - 1) / kPrefixTile;
  return tiles > 0 ? (tiles + prefix_chunk_tiles(L) - 1) / prefix_chunk_tiles(L) : 1;
}

// Shared-prefix (cascade) set-up: per-request first unshared block.
struct CascadePrepParams {
  const int32_t* grp_first;
  const int32_t* grp_count;
  const int32_t* grp_blocks;
  int32_t* first_block;  // [num_reqs], cleared before the launch
  int* err;
  int num_groups;
  int num_reqs;
  int max_blocks;
  int pdl;
};

cudaError_t launch_cascade_prep(const CascadePrepParams& p, cudaStream_t stream);

struct PrefillLaunch {
  CUtensorMap qmap;  // q as [tokens][Hq][128], box (64, g, 128/g)
  CUtensorMap kmap;  // k_pool as [blocks*Hkv*16][128], box (64, 16), 128-byte swizzle
  CUtensorMap vmap;  // v_pool, same
  PrefillParams p;
  int grid;
};

int prefill_tokens_per_tile(int group);

#ifndef PKV_TRACE
#define PKV_TRACE 0
#endif
#if PKV_TRACE
cudaError_t decode_trace(void* host, size_t bytes);
#endif
#ifndef PKV_TC_TRACE
#define PKV_TC_TRACE 0
#endif
#if PKV_TC_TRACE
cudaError_t decode_tc_trace(void* host, size_t bytes);
#if PKV_TC_TRACE >= 3
cudaError_t append_trace(void* host, size_t bytes);
#endif
#endif
#ifndef PKV_PF_TRACE
#define PKV_PF_TRACE 0
#endif
#if PKV_PF_TRACE
cudaError_t prefill_trace(void* host, size_t bytes);
#endif

// Sets the thread's pkv_last_error() message.
void set_error_message(const char* msg);

// pkv_attention_workspace_size with its error code (message set on failure).
int attention_workspace_bytes(const ::pkv_dims* dims, size_t* bytes);

cudaError_t launch_prefill(const PrefillLaunch& L, int group, cudaStream_t stream);

}  // namespace pkv
