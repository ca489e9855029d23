// pkv_noalloc.cu -- pkv_attention_noalloc: the attention step for callers
// that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: plugins hosted by a framework
// that owns every byte of device memory through its own pool, and serving
// loops that forbid allocation after start-up (an allocation there can stall
// on the driver or fail once memory is fragmented).  They also cannot hand
// pkv_attention a workspace of their own.  This entry point takes
// the split-context scratch (merge counters, partial outputs and their
// log-sum-exp statistics) from one fixed array compiled into the library.
//
// The array lives for the whole process on every GPU that loads the library.
// Its name, used in host code, is only a host-side stand-in for the symbol:
// the device address is fetched once per device with cudaGetSymbolAddress,
// with that device current, and passed to the kernels.  Every call shares the
// array, so calls that overlap on the GPU (two streams, or two host threads)
// race on it and must be serialised by the caller.  Each call clears the
// array's head (merge counters, prefill work queue and plan cache) with a
// stream-ordered memset, so these calls re-plan every time, and the decode
// kernel cannot overlap the kernel before the memset (programmatic dependent
// launch): a little slower than pkv_attention with a workspace.
#include <cstdio>
#include <mutex>

#include "../../include/pagedkv.h"
#include "pkv_internal.h"

namespace {

// The scratch: PKV_NOALLOC_SCRATCH_BYTES bytes per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

using pkv::kMaxDevices;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_fail(int code, const char* what) {
  char msg[200];
  snprintf(msg, sizeof msg, "pkv_attention_noalloc: %s", what);
  pkv::set_error_message(msg);
  return code;
}

}  // namespace

extern "C" int pkv_attention_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                     const int32_t* block_tables, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, float scale, void* out,
                                     const pkv_dims* dims, cudaStream_t stream) {
  pkv::set_error_message("");
  // Sizes first: dims the array cannot hold are an error, not an allocation.
  // (This also checks the dims and the current device, setting the message.)
  size_t need = 0;
  const int rc = pkv::attention_workspace_bytes(dims, &need);
  if (rc != PKV_OK) return rc;
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "pkv_attention_noalloc: these dims need %zu scratch bytes, more than the "
             "%d-byte static array (reduce num_q_tokens * num_kv_heads)",
             need, (int)PKV_NOALLOC_SCRATCH_BYTES);
    pkv::set_error_message(msg);
    return PKV_ERR_WORKSPACE;
  }
  // Once per device, with that device current: the array's device address.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return noalloc_fail(PKV_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(PKV_ERR_UNSUPPORTED, "device ordinal beyond the library's limit");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || ptr == nullptr)
        return noalloc_fail(PKV_ERR_CUDA, "cudaGetSymbolAddress of the scratch failed");
      g_noalloc_ptr[dev] = ptr;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // The array keeps the previous call's contents; its head (merge counters,
  // prefill work queue, plan cache) must start at zero: its extent moves with
  // the dims.
  int sm_count = 1;
  if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return noalloc_fail(PKV_ERR_CUDA, "cudaDeviceGetAttribute failed");
  const pkv::WorkspaceLayout w = pkv::decode_workspace_layout(
      dims->num_q_tokens, dims->num_kv_heads, dims->num_q_heads / dims->num_kv_heads, sm_count);
  if (w.ml_off > 0 && cudaMemsetAsync(scratch, 0, w.ml_off, stream) != cudaSuccess)
    return noalloc_fail(PKV_ERR_CUDA, "clearing the scratch counters failed");
  return pkv_attention(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc, scale, out,
                       dims, scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
