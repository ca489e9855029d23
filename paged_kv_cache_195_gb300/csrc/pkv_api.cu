// pkv_api.cu -- the C ABI of libpagedkv.so (declared in include/pagedkv.h):
// argument validation, per-device state, workspace carve-up and launches.
// No call allocates on the hot path (the NULL-workspace convenience path
// allocates once per device), none synchronises, so a whole step can be
// captured in a CUDA graph.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/pagedkv.h"
#include "pkv_internal.h"

static_assert(PKV_MAX_REQS == pkv::kMaxReqs, "request limit mismatch");

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The device error word lives in this translation unit; kernels get its
// address as an argument.
__device__ int g_device_error;

using pkv::kMaxDevices;

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int* err = nullptr;          // device address of g_device_error
  void* own_ws = nullptr;      // the NULL-workspace convenience buffer
  size_t own_ws_bytes = 0;
  size_t own_ws_cnt_bytes = 0; // counter bytes its last user needed zeroed
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Per-device set-up with that device current: SM count and the address of
// the error word.  Returns nullptr (and sets the message) on failure.
DeviceState* device_state() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    fail(PKV_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaDeviceGetAttribute");
      return nullptr;
    }
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err), g_device_error);
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaGetSymbolAddress(error word)");
      return nullptr;
    }
    st.ready = true;
  }
  return &st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_dims(const pkv_dims* d, bool for_attention) {
  if (d == nullptr) return fail(PKV_ERR_INVALID, "dims is NULL");
  if (d->head_dim != pkv::kHeadDim)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d unsupported (only 128)", d->head_dim);
  if (d->block_size != pkv::kBlockSize)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d unsupported (only 16)", d->block_size);
  if (d->num_kv_heads <= 0 || d->num_blocks < 0)
    return fail(PKV_ERR_INVALID, "num_kv_heads %d / num_blocks %d invalid", d->num_kv_heads,
                d->num_blocks);
  if ((long long)d->num_blocks * d->num_kv_heads * pkv::kBlockSize > (1ll << 40))
    return fail(PKV_ERR_INVALID, "pool too large");
  if (!for_attention) return PKV_OK;
  if (d->num_reqs < 0 || d->num_q_tokens < 0 || d->num_q_heads <= 0 ||
      d->max_blocks_per_req < 0)
    return fail(PKV_ERR_INVALID, "negative dims");
  if (d->num_q_heads % d->num_kv_heads != 0)
    return fail(PKV_ERR_INVALID, "num_q_heads %d not a multiple of num_kv_heads %d",
                d->num_q_heads, d->num_kv_heads);
  const int g = d->num_q_heads / d->num_kv_heads;
  if (g < 1 || g > 8) return fail(PKV_ERR_UNSUPPORTED, "group size %d unsupported (1..8)", g);
  if (d->num_reqs > pkv::kMaxReqs)
    return fail(PKV_ERR_UNSUPPORTED, "num_reqs %d beyond %d", d->num_reqs, pkv::kMaxReqs);
  if ((long long)d->max_blocks_per_req * pkv::kBlockSize > (1ll << 30))
    return fail(PKV_ERR_UNSUPPORTED, "max_blocks_per_req too large");
  return PKV_OK;
}

pkv::WorkspaceLayout layout_for(const pkv_dims* d, int sm_count) {
  return pkv::decode_workspace_layout(d->num_q_tokens, d->num_kv_heads,
                                      d->num_q_heads / d->num_kv_heads, sm_count);
}

// ----------------------------------------------------------------- options
// Process-wide launch and routing options: built-in defaults, overridden once
// by the environment when first needed, then only by pkv_set_options.  Every
// call works from one copy taken when it starts.
int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  return (v && *v) ? atoi(v) : dflt;
}

bool options_valid(const pkv_options& o) {
  return o.prefill_min_q >= 0 && o.align_slack >= 0 && o.min_chunk >= 1 && o.decode_grid >= 0 &&
         o.wait_limit_us >= 1 && o.rowgroup_cost >= 0 &&
         o.rowgroup_cost <= 1024;
}

pkv_options options_from_env() {
  pkv_options o{};
  o.pdl = env_int("PKV_PDL", 1);
  o.early_plan = env_int("PKV_EARLY_PLAN", 1);
  o.early_kv = env_int("PKV_EARLY_KV", 1);
  o.early_trigger = env_int("PKV_EARLY_TRIGGER", 0);
  o.plan_cache = env_int("PKV_PLAN_CACHE", 1);
  o.decode_tc = env_int("PKV_DECODE_TC", 1);
  o.decode_tc_fp8 = env_int("PKV_DECODE_TC_FP8", 1);
  o.prefill_min_q = env_int("PKV_PREFILL_MIN_Q", 16);
  o.align = env_int("PKV_ALIGN", 1);
  o.align_slack = env_int("PKV_ALIGN_SLACK", 64);
  o.min_chunk = env_int("PKV_MIN_CHUNK", 4);
  o.decode_grid = env_int("PKV_DECODE_GRID", 0);
  o.wait_limit_us = env_int("PKV_WAIT_LIMIT_US", (int)(pkv::kDefaultWaitLimitNs / 1000));
  o.debug_withhold_q = 0;  // never from the environment
  o.rowgroup_cost = env_int("PKV_ROWGROUP_COST", 16);
  // Out-of-range values from the environment fall back to the defaults.
  if (o.prefill_min_q < 0) o.prefill_min_q = 16;
  if (o.align_slack < 0) o.align_slack = 64;
  if (o.min_chunk < 1) o.min_chunk = 4;
  if (o.decode_grid < 0) o.decode_grid = 0;
  if (o.wait_limit_us < 1) o.wait_limit_us = (int)(pkv::kDefaultWaitLimitNs / 1000);
  if (o.rowgroup_cost < 0 || o.rowgroup_cost > 1024) o.rowgroup_cost = 16;
  return o;
}

std::mutex g_opts_mutex;
bool g_opts_ready = false;
pkv_options g_opts;

pkv_options current_options() {
  std::lock_guard<std::mutex> lock(g_opts_mutex);
  if (!g_opts_ready) {
    g_opts = options_from_env();
    g_opts_ready = true;
  }
  return g_opts;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 2-D map of a pool as [num_blocks * Hkv * 16 rows][128] bf16, 64 x 16 boxes.
// e4m3 pools: the same view in bytes, boxes of 16 rows x 128 codes.
int encode_pool_map_e4m3(CUtensorMap* m, const void* pool, const pkv_dims* d) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)pkv::kHeadDim,
                              (cuuint64_t)d->num_blocks * d->num_kv_heads * pkv::kBlockSize};
  const cuuint64_t strides[1] = {(cuuint64_t)pkv::kHeadDim};
  const cuuint32_t box[2] = {(cuuint32_t)pkv::kHeadDim, (cuuint32_t)pkv::kBlockSize};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "encode e4m3 pool tensor map: CUresult %d", (int)r);
  return PKV_OK;
}

int encode_pool_map(CUtensorMap* m, const void* pool, const pkv_dims* d) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)pkv::kHeadDim,
                              (cuuint64_t)d->num_blocks * d->num_kv_heads * pkv::kBlockSize};
  const cuuint64_t strides[1] = {(cuuint64_t)pkv::kHeadDim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)pkv::kBlockSize};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "encode pool tensor map: CUresult %d", (int)r);
  return PKV_OK;
}

// 3-D map of q as [Tq][Hq][128] bf16, boxes of (64 dims, g heads, `tokens` tokens).
int encode_q_map(CUtensorMap* m, const void* q, const pkv_dims* d, int group, int tokens) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[3] = {(cuuint64_t)pkv::kHeadDim, (cuuint64_t)d->num_q_heads,
                              (cuuint64_t)d->num_q_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)pkv::kHeadDim * 2,
                                 (cuuint64_t)d->num_q_heads * pkv::kHeadDim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)tokens};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "encode q tensor map: CUresult %d", (int)r);
  return PKV_OK;
}

}  // namespace

namespace pkv {
void set_error_message(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

int attention_workspace_bytes(const pkv_dims* dims, size_t* bytes) {
  *bytes = 0;
  const int rc = check_dims(dims, true);
  if (rc != PKV_OK) return rc;
  DeviceState* st = device_state();
  if (!st) return PKV_ERR_CUDA;
  *bytes = layout_for(dims, st->sm_count).total;
  return PKV_OK;
}
}  // namespace pkv

namespace {

int append_impl(const void* k_new, const void* v_new, const int64_t* slot_mapping, void* k_pool,
                void* v_pool, int32_t num_new_tokens, const pkv_dims* dims, cudaStream_t stream,
                bool early_trigger) {
  g_last_error[0] = '\0';
  int rc = check_dims(dims, false);
  if (rc != PKV_OK) return rc;
  if (num_new_tokens < 0) return fail(PKV_ERR_INVALID, "num_new_tokens < 0");
  if (num_new_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool)
    return fail(PKV_ERR_INVALID, "NULL pointer argument");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(PKV_ERR_INVALID, "bf16 buffers must be 16-byte aligned");
  DeviceState* st = device_state();
  if (!st) return PKV_ERR_CUDA;
  pkv::AppendParams p{};
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.slot_mapping = slot_mapping;
  p.k_pool = static_cast<__nv_bfloat16*>(k_pool);
  p.v_pool = static_cast<__nv_bfloat16*>(v_pool);
  p.err = st->err;
  p.num_tokens = num_new_tokens;
  p.num_kv_heads = dims->num_kv_heads;
  p.num_blocks = dims->num_blocks;
  p.pdl = current_options().pdl != 0;
  p.early_trigger = early_trigger && p.pdl;
  cudaError_t e = pkv::launch_append(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return PKV_OK;
}

int append_fp8_impl(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                    void* k_pool, void* v_pool, const float* k_scale, const float* v_scale,
                    int32_t num_new_tokens, const pkv_dims* dims, cudaStream_t stream,
                    bool early_trigger) {
  g_last_error[0] = '\0';
  int rc = check_dims(dims, false);
  if (rc != PKV_OK) return rc;
  if (num_new_tokens < 0) return fail(PKV_ERR_INVALID, "num_new_tokens < 0");
  if (num_new_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool || !k_scale || !v_scale)
    return fail(PKV_ERR_INVALID, "NULL pointer argument");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(PKV_ERR_INVALID, "k/v buffers and pools must be 16-byte aligned");
  DeviceState* st = device_state();
  if (!st) return PKV_ERR_CUDA;
  pkv::AppendFp8Params p{};
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.slot_mapping = slot_mapping;
  p.k_pool = static_cast<uint8_t*>(k_pool);
  p.v_pool = static_cast<uint8_t*>(v_pool);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = st->err;
  p.num_tokens = num_new_tokens;
  p.num_kv_heads = dims->num_kv_heads;
  p.num_blocks = dims->num_blocks;
  p.pdl = current_options().pdl != 0;
  p.early_trigger = early_trigger && p.pdl;
  cudaError_t e = pkv::launch_append_fp8(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "append_fp8 launch");
  return PKV_OK;
}

}  // namespace

extern "C" {

const char* pkv_last_error(void) { return g_last_error; }

int pkv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping, void* k_pool,
               void* v_pool, int32_t num_new_tokens, const pkv_dims* dims, cudaStream_t stream) {
  return append_impl(k_new, v_new, slot_mapping, k_pool, v_pool, num_new_tokens, dims, stream,
                     false);
}

int pkv_append_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                   void* k_pool, void* v_pool, const float* k_scale, const float* v_scale,
                   int32_t num_new_tokens, const pkv_dims* dims, cudaStream_t stream) {
  return append_fp8_impl(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale, v_scale,
                         num_new_tokens, dims, stream, false);
}

int pkv_copy_blocks(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                    const int64_t* pairs, int32_t num_pairs, int32_t src_num_blocks,
                    int32_t dst_num_blocks, const pkv_dims* dims, cudaStream_t stream) {
  g_last_error[0] = '\0';
  int rc = check_dims(dims, false);
  if (rc != PKV_OK) return rc;
  if (num_pairs < 0 || src_num_blocks < 0 || dst_num_blocks < 0)
    return fail(PKV_ERR_INVALID, "negative count");
  if (num_pairs == 0) return PKV_OK;
  if (!k_src || !v_src || !k_dst || !v_dst || !pairs)
    return fail(PKV_ERR_INVALID, "NULL pointer argument");
  if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_dst) || !aligned16(v_dst))
    return fail(PKV_ERR_INVALID, "pools must be 16-byte aligned");
  DeviceState* st = device_state();
  if (!st) return PKV_ERR_CUDA;
  pkv::CopyParams p{};
  p.k_src = static_cast<const __nv_bfloat16*>(k_src);
  p.v_src = static_cast<const __nv_bfloat16*>(v_src);
  p.k_dst = static_cast<__nv_bfloat16*>(k_dst);
  p.v_dst = static_cast<__nv_bfloat16*>(v_dst);
  p.pairs = pairs;
  p.err = st->err;
  p.num_pairs = num_pairs;
  p.num_kv_heads = dims->num_kv_heads;
  p.src_blocks = src_num_blocks;
  p.dst_blocks = dst_num_blocks;
  p.pdl = current_options().pdl != 0;
  cudaError_t e = pkv::launch_copy_blocks(p, st->sm_count, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return PKV_OK;
}

size_t pkv_attention_workspace_size(const pkv_dims* dims) {
  size_t bytes = 0;
  return pkv::attention_workspace_bytes(dims, &bytes) == PKV_OK ? bytes : 0;
}

int pkv_workspace_init(void* workspace, size_t workspace_bytes, const pkv_dims* dims,
                       cudaStream_t stream) {
  g_last_error[0] = '\0';
  int rc = check_dims(dims, true);
  if (rc != PKV_OK) return rc;
  DeviceState* st = device_state();
  if (!st) return PKV_ERR_CUDA;
  const pkv::WorkspaceLayout w = layout_for(dims, st->sm_count);
  if (workspace == nullptr || workspace_bytes < w.total)
    return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, w.total);
  cudaError_t e = cudaMemsetAsync(workspace, 0, w.ml_off, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace counters)");
  return PKV_OK;
}

}  // extern "C"

namespace {

// Sharing groups of a cascade call (device arrays).
struct CascadeArgs {
  const int32_t* grp_first;
  const int32_t* grp_count;
  const int32_t* grp_blocks;
  int num_groups;
};

// Regions a cascade call adds after the attention workspace.
struct CascadeLayout {
  size_t pre_o, pre_ml, first_block, total;
};

CascadeLayout cascade_layout(const pkv::WorkspaceLayout& w, const pkv_dims* d) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)pkv::kPrefixSplits * d->num_q_tokens * d->num_q_heads;
  CascadeLayout c;
  c.pre_o = up(w.total);
  c.pre_ml = c.pre_o + up(rows * pkv::kHeadDim * sizeof(float));
  c.first_block = c.pre_ml + up(rows * 2 * sizeof(float));
  c.total = c.first_block + up((size_t)d->num_reqs * sizeof(int32_t));
  return c;
}

// The attention entry points: bf16 pools (k_scale == nullptr) or e4m3 pools,
// optionally with shared-prefix groups.
int attention_impl(const void* q, const void* k_pool, const void* v_pool, const float* k_scale,
                   const float* v_scale, const int32_t* block_tables, const int32_t* seq_lens,
                   const int32_t* query_start_loc, float scale, void* out, const pkv_dims* dims,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream,
                   const CascadeArgs* cas = nullptr, bool after_append = false,
                   bool append_triggered_early = false) {
  g_last_error[0] = '\0';
  const bool fp8 = k_scale != nullptr;
  int rc = check_dims(dims, true);
  if (rc != PKV_OK) return rc;
  if (dims->num_reqs == 0 || dims->num_q_tokens == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !query_start_loc || !out)
    return fail(PKV_ERR_INVALID, "NULL pointer argument");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return fail(PKV_ERR_INVALID, "q, out and the pools must be 16-byte aligned");
  if (!(scale == scale) || scale == 0.f) return fail(PKV_ERR_INVALID, "scale must be finite, non-zero");
  if (cas) {
    if (cas->num_groups < 0) return fail(PKV_ERR_INVALID, "num_groups < 0");
    if (cas->num_groups > 0 && (!cas->grp_first || !cas->grp_count || !cas->grp_blocks))
      return fail(PKV_ERR_INVALID, "NULL group array");
  }
  DeviceState* st = device_state();
  if (!st) return PKV_ERR_CUDA;
  const pkv::WorkspaceLayout w = layout_for(dims, st->sm_count);
  const CascadeLayout cl = cascade_layout(w, dims);
  if (cas) {
    if (workspace == nullptr || workspace_bytes < cl.total)
      return fail(PKV_ERR_WORKSPACE, "cascade workspace %zu bytes, need %zu (caller-owned)",
                  workspace_bytes, cl.total);
  }
  if (workspace == nullptr) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (st->own_ws_bytes < w.total) {
      if (st->own_ws) cudaFree(st->own_ws);
      st->own_ws = nullptr;
      st->own_ws_bytes = 0;
      cudaError_t e = cudaMalloc(&st->own_ws, w.total);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
      e = cudaMemset(st->own_ws, 0, w.total);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(workspace)");
      st->own_ws_bytes = w.total;
      st->own_ws_cnt_bytes = w.ml_off;
    } else if (st->own_ws_cnt_bytes != w.ml_off) {
      // The counter region moved with the dims: zero it again.
      cudaError_t e = cudaMemsetAsync(st->own_ws, 0, w.ml_off, stream);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
      st->own_ws_cnt_bytes = w.ml_off;
    }
    workspace = st->own_ws;
    workspace_bytes = st->own_ws_bytes;
  }
  if (workspace_bytes < w.total)
    return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, w.total);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(PKV_ERR_INVALID, "workspace must be 256-byte aligned");

  const pkv_options opt = current_options();
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  pkv::DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.kv_fp8 = fp8 ? 1 : 0;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.ws_cnt = reinterpret_cast<int*>(ws + w.cnt_off);
  p.plan_cache = opt.plan_cache != 0 && dims->num_reqs <= pkv::kPlanCacheReqs
                     ? reinterpret_cast<int*>(ws + w.plan_off)
                     : nullptr;
  p.plan_entries = w.plan_entries;
  p.ws_ml = reinterpret_cast<float*>(ws + w.ml_off);
  p.ws_o = reinterpret_cast<float*>(ws + w.o_off);
  p.err = st->err;
  p.num_reqs = dims->num_reqs;
  p.num_q_tokens = dims->num_q_tokens;
  p.num_q_heads = dims->num_q_heads;
  p.num_kv_heads = dims->num_kv_heads;
  p.num_blocks = dims->num_blocks;
  p.max_blocks = dims->max_blocks_per_req;
  p.scale_log2 = scale * 1.4426950408889634f;
  // Requests with at least this many query tokens go to the tensor-core
  // prefill kernel (when the step has that many query tokens at all).
  int prefill_min_q = opt.prefill_min_q;
  if (prefill_min_q < 1) prefill_min_q = 0x7fffffff;
  // Launch it only when the step can hold such a request next to one query
  // for every other request; otherwise the decode kernel serves every row
  // (it is correct for any q_r, the prefill kernel is only faster).
  // e4m3 pools: every row runs in the decode kernel.
  const bool run_prefill =
      !fp8 && (long long)dims->num_q_tokens - dims->num_reqs + 1 >= (long long)prefill_min_q;
  p.prefill_min_q = run_prefill ? prefill_min_q : 0x7fffffff;
  p.num_slots = w.num_slots;
  p.pdl = opt.pdl != 0;
  p.min_chunk = opt.min_chunk;
  p.align = opt.align != 0;
  p.align_slack = opt.align_slack;
  p.early_plan = p.pdl && opt.early_plan != 0;
  p.wait_limit_ns = (unsigned long long)opt.wait_limit_us * 1000ull;
  p.debug_withhold_q = opt.debug_withhold_q != 0;
  p.rowgroup_cost = opt.rowgroup_cost;
  const int group = dims->num_q_heads / dims->num_kv_heads;
  int grid = pkv::decode_grid(st->sm_count, group);
  // tuning override, bounded by the workspace's slots
  if (opt.decode_grid > 0 && 2 * opt.decode_grid <= w.num_slots) grid = opt.decode_grid;
  // Groups of 4 or more query heads per KV head make the decode's FP32 FMA
  // work comparable to its HBM time; those run on the tensor cores, e4m3
  // pools included (their tiles widened to f16 in shared memory by two
  // converter warps; decode_tc_fp8 = 0 keeps them on the SIMT decode).
  const bool use_tc = group >= 4 && opt.decode_tc != 0 && (!fp8 || opt.decode_tc_fp8 != 0);
  cudaError_t e;
  // Shared prefixes are read once by the prefix pass when the tensor-core
  // decode serves the step; otherwise every row reads its whole context (the
  // same result, without the sharing).
  const bool cascade = cas && cas->num_groups > 0 && use_tc;
  if (cascade) {
    int32_t* first_block = reinterpret_cast<int32_t*>(ws + cl.first_block);
    e = cudaMemsetAsync(first_block, 0, (size_t)dims->num_reqs * sizeof(int32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(first blocks)");
    pkv::CascadePrepParams cp{};
    cp.grp_first = cas->grp_first;
    cp.grp_count = cas->grp_count;
    cp.grp_blocks = cas->grp_blocks;
    cp.first_block = first_block;
    cp.err = st->err;
    cp.num_groups = cas->num_groups;
    cp.num_reqs = dims->num_reqs;
    cp.max_blocks = dims->max_blocks_per_req;
    cp.pdl = p.pdl;
    e = pkv::launch_cascade_prep(cp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cascade set-up launch");
    // Prefix pass: every member's rows against the group's shared blocks.
    pkv::PrefillLaunch L{};
    rc = encode_q_map(&L.qmap, q, dims, group, pkv::prefill_tokens_per_tile(group));
    if (rc == PKV_OK) rc = encode_pool_map(&L.kmap, k_pool, dims);
    if (rc == PKV_OK) rc = encode_pool_map(&L.vmap, v_pool, dims);
    if (rc != PKV_OK) return rc;
    L.p.block_tables = block_tables;
    L.p.seq_lens = seq_lens;
    L.p.qsl = query_start_loc;
    L.p.out = p.out;
    L.p.err = st->err;
    L.p.num_reqs = dims->num_reqs;
    L.p.num_q_tokens = dims->num_q_tokens;
    L.p.num_q_heads = dims->num_q_heads;
    L.p.num_kv_heads = dims->num_kv_heads;
    L.p.num_blocks = dims->num_blocks;
    L.p.max_blocks = dims->max_blocks_per_req;
    L.p.scale_log2 = p.scale_log2;
    L.p.prefill_min_q = 1;
    L.p.pdl = p.pdl;
    L.p.prefix_mode = 1;
    L.p.grp_first = cas->grp_first;
    L.p.grp_count = cas->grp_count;
    L.p.grp_blocks = cas->grp_blocks;
    L.p.num_groups = cas->num_groups;
    L.p.pre_o = reinterpret_cast<float*>(ws + cl.pre_o);
    L.p.pre_ml = reinterpret_cast<float*>(ws + cl.pre_ml);
    L.p.sched = reinterpret_cast<unsigned long long*>(ws + w.sched_off);
    L.p.wait_limit_ns = p.wait_limit_ns;
    L.grid = st->sm_count;
    e = pkv::launch_prefill(L, group, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefix pass launch");
    // Decode of every row from its first unshared block, merging the prefix.
    p.first_block = first_block;
    p.pre_o = L.p.pre_o;
    p.pre_ml = L.p.pre_ml;
    p.prefill_min_q = 0x7fffffff;
    p.early_plan = 0;  // first_block comes from the set-up kernel, two launches back
  }
  // Right after the append of this step's tokens (pkv_append_attention), the
  // decode kernel streams every tile without a new token before waiting.
  p.early_kv = after_append && !cascade && p.pdl;
  p.early_q = !append_triggered_early;
  const bool do_prefill = run_prefill && !cascade;
  if (use_tc) {
    pkv::DecodeTcLaunch T{};
    rc = encode_q_map(&T.qmap, q, dims, group, 1);
    if (rc == PKV_OK) rc = fp8 ? encode_pool_map_e4m3(&T.kmap, k_pool, dims)
                               : encode_pool_map(&T.kmap, k_pool, dims);
    if (rc == PKV_OK) rc = fp8 ? encode_pool_map_e4m3(&T.vmap, v_pool, dims)
                               : encode_pool_map(&T.vmap, v_pool, dims);
    if (rc != PKV_OK) return rc;
    T.p = p;
    // Two CTAs per SM; steps with at most 8 tiles (64 blocks) per SM run on
    // one CTA per SM, so that the next launch's CTAs can prepare beside them.
    // When the dims alone bound the work that low (every decode row reads at
    // most max_blocks_per_req blocks per KV head) the grid is one CTA per SM;
    // otherwise the plan makes the choice on the device from the lengths.
    constexpr long long kHalfGridBlocks = 64;
    const long long bound = (long long)dims->num_q_tokens * dims->max_blocks_per_req * dims->num_kv_heads;
    const bool small = bound <= kHalfGridBlocks * st->sm_count;
    T.grid = small ? st->sm_count : 2 * st->sm_count;
    T.p.half_grid_blocks = small ? 0 : (int)kHalfGridBlocks;
    // tuning override, bounded by the workspace's slots
    if (opt.decode_grid > 0 && 2 * opt.decode_grid <= w.num_slots) {
      T.grid = opt.decode_grid;
      T.p.half_grid_blocks = 0;
    }
    e = pkv::launch_decode_tc(T, group, stream);
  } else {
    e = pkv::launch_decode(p, group, grid, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (do_prefill) {
    pkv::PrefillLaunch L{};
    rc = encode_q_map(&L.qmap, q, dims, group, pkv::prefill_tokens_per_tile(group));
    if (rc == PKV_OK) rc = encode_pool_map(&L.kmap, k_pool, dims);
    if (rc == PKV_OK) rc = encode_pool_map(&L.vmap, v_pool, dims);
    if (rc != PKV_OK) return rc;
    L.p.block_tables = block_tables;
    L.p.seq_lens = seq_lens;
    L.p.qsl = query_start_loc;
    L.p.out = p.out;
    L.p.err = st->err;
    L.p.num_reqs = dims->num_reqs;
    L.p.num_q_tokens = dims->num_q_tokens;
    L.p.num_q_heads = dims->num_q_heads;
    L.p.num_kv_heads = dims->num_kv_heads;
    L.p.num_blocks = dims->num_blocks;
    L.p.max_blocks = dims->max_blocks_per_req;
    L.p.scale_log2 = p.scale_log2;
    L.p.prefill_min_q = prefill_min_q;
    L.p.pdl = p.pdl;
    L.p.sched = reinterpret_cast<unsigned long long*>(ws + w.sched_off);
    L.p.wait_limit_ns = p.wait_limit_ns;
    L.grid = st->sm_count;
    e = pkv::launch_prefill(L, group, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_attention(const void* q, const void* k_pool, const void* v_pool,
                  const int32_t* block_tables, const int32_t* seq_lens,
                  const int32_t* query_start_loc, float scale, void* out, const pkv_dims* dims,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return attention_impl(q, k_pool, v_pool, nullptr, nullptr, block_tables, seq_lens,
                        query_start_loc, scale, out, dims, workspace, workspace_bytes, stream);
}

int pkv_append_attention(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                         void* k_pool, void* v_pool, const void* q, const int32_t* block_tables,
                         const int32_t* seq_lens, const int32_t* query_start_loc, float scale,
                         void* out, const pkv_dims* dims, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  g_last_error[0] = '\0';
  int rc = check_dims(dims, true);
  if (rc != PKV_OK) return rc;
  // The attention kernel reads K/V tiles without this step's tokens (and the
  // lengths and tables) before it waits for the append.  PKV_EARLY_TRIGGER=1
  // also lets it launch as soon as the append starts, before the kernel
  // ahead of the append has finished; q, out and the workspace then wait.
  const pkv_options opt = current_options();
  const bool pdl = opt.pdl != 0;
  const bool early = pdl && opt.early_kv != 0;
  const bool trigger = early && opt.early_trigger != 0;
  rc = append_impl(k_new, v_new, slot_mapping, k_pool, v_pool, dims->num_q_tokens, dims, stream,
                   trigger);
  if (rc != PKV_OK) return rc;
  return attention_impl(q, k_pool, v_pool, nullptr, nullptr, block_tables, seq_lens,
                        query_start_loc, scale, out, dims, workspace, workspace_bytes, stream,
                        nullptr, early, trigger);
}

int pkv_append_attention_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                             void* k_pool, void* v_pool, const float* k_scale,
                             const float* v_scale, const void* q, const int32_t* block_tables,
                             const int32_t* seq_lens, const int32_t* query_start_loc,
                             float scale, void* out, const pkv_dims* dims, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  g_last_error[0] = '\0';
  int rc = check_dims(dims, true);
  if (rc != PKV_OK) return rc;
  if (!k_scale || !v_scale) return fail(PKV_ERR_INVALID, "k_scale / v_scale is NULL");
  // As pkv_append_attention: tiles without this step's tokens are read
  // before the append finishes (early_kv), and with early_trigger the
  // attention launches as soon as the append starts.
  const pkv_options opt = current_options();
  const bool pdl = opt.pdl != 0;
  const bool early = pdl && opt.early_kv != 0;
  const bool trigger = early && opt.early_trigger != 0;
  rc = append_fp8_impl(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale, v_scale,
                       dims->num_q_tokens, dims, stream, trigger);
  if (rc != PKV_OK) return rc;
  return attention_impl(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                        query_start_loc, scale, out, dims, workspace, workspace_bytes, stream,
                        nullptr, early, trigger);
}

size_t pkv_cascade_workspace_size(const pkv_dims* dims) {
  if (check_dims(dims, true) != PKV_OK) return 0;
  DeviceState* st = device_state();
  if (!st) return 0;
  return cascade_layout(layout_for(dims, st->sm_count), dims).total;
}

int pkv_attention_cascade(const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_tables, const int32_t* seq_lens,
                          const int32_t* query_start_loc, const int32_t* group_first_req,
                          const int32_t* group_num_reqs, const int32_t* group_prefix_blocks,
                          int32_t num_groups, float scale, void* out, const pkv_dims* dims,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const CascadeArgs cas{group_first_req, group_num_reqs, group_prefix_blocks, num_groups};
  return attention_impl(q, k_pool, v_pool, nullptr, nullptr, block_tables, seq_lens,
                        query_start_loc, scale, out, dims, workspace, workspace_bytes, stream,
                        &cas);
}

int pkv_attention_fp8kv(const void* q, const void* k_pool, const void* v_pool,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        const int32_t* seq_lens, const int32_t* query_start_loc, float scale,
                        void* out, const pkv_dims* dims, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  if (!k_scale || !v_scale) {
    g_last_error[0] = '\0';
    return fail(PKV_ERR_INVALID, "k_scale / v_scale is NULL");
  }
  return attention_impl(q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                        query_start_loc, scale, out, dims, workspace, workspace_bytes, stream);
}

void pkv_get_options(pkv_options* opts) {
  if (opts) *opts = current_options();
}

int pkv_set_options(const pkv_options* opts) {
  g_last_error[0] = '\0';
  if (opts == nullptr) return fail(PKV_ERR_INVALID, "options is NULL");
  if (!options_valid(*opts)) return fail(PKV_ERR_INVALID, "an option is out of range");
  current_options();  // the environment is read once, before the first change
  std::lock_guard<std::mutex> lock(g_opts_mutex);
  g_opts = *opts;
  return PKV_OK;
}

int pkv_get_device_error(cudaStream_t stream) {
  g_last_error[0] = '\0';
  DeviceState* st = device_state();
  if (!st) return PKV_ERR_CUDA;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, st->err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  const int zero = 0;
  e = cudaMemcpy(st->err, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  if (word & pkv::kErrTimeout) return fail(PKV_ERR_TIMEOUT, "a device wait timed out (flags %d)", word);
  if (word & (pkv::kErrBounds | pkv::kErrCapacity))
    return fail(PKV_ERR_DEVICE_BOUNDS, "device bounds violation (flags %d)", word);
  return PKV_OK;
}

#if PKV_PF_TRACE
// Debug builds only: copies the prefill kernel's per-tile timeline.
int pkv_debug_pf_trace(void* host, size_t bytes) {
  return pkv::prefill_trace(host, bytes) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
#endif

#if PKV_TC_TRACE
// Debug builds only: copies the tensor-core decode's per-tile timeline.
int pkv_debug_tc_trace(void* host, size_t bytes) {
  return pkv::decode_tc_trace(host, bytes) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
#endif

#if PKV_TRACE
// Debug builds only: copies the decode kernel's per-CTA phase stamps.
int pkv_debug_trace(void* host, size_t bytes) {
  return pkv::decode_trace(host, bytes) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
#endif

}  // extern "C"
