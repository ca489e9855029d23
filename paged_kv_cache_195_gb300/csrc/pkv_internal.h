// pkv_internal.h -- kernel parameter blocks and launchers shared between the
// host ABI (pkv_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv_common.cuh"

namespace pkv {

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
};

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// Split-context decode: the device plan, the paged gather, the online
// softmax, and the log-sum-exp merge, in one launch.
struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  __nv_bfloat16* out;
  int* ws_cnt;    // [num_q_tokens * num_kv_heads] merge counters, zero between calls
  float* ws_ml;   // [max_units, g, 2] (max, normaliser) of each split, log2 domain
  float* ws_o;    // [max_units, g, 128] normalised partial output of each split
  int* err;
  int num_reqs;
  int num_q_tokens;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int max_blocks;
  float scale_log2;   // scale * log2(e)
  int prefill_min_q;  // requests with q_r >= this are left to the prefill kernel
  int target_units;   // split policy: aim for about this many work units
  int max_units;      // workspace capacity in units
  int min_chunk;      // smallest split, in blocks
};

// Workspace carve-up shared by the host code that sizes it and the launcher.
struct WorkspaceLayout {
  size_t cnt_off, ml_off, o_off, total;
  int max_units;
};

WorkspaceLayout decode_workspace_layout(int num_q_tokens, int num_kv_heads, int group,
                                        int target_units);

// Returns the grid the decode launch will use (for workspace sizing).
int decode_target_units(int sm_count);

cudaError_t launch_decode(const DecodeParams& p, int group, int sm_count,
                          cudaStream_t stream);

}  // namespace pkv
