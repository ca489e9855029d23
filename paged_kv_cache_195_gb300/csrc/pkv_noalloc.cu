// pkv_noalloc.cu -- pkv_attention_noalloc: the attention step for callers
// that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code that runs while a CUDA
// graph is captured in global mode (where allocation is prohibited), plugins
// hosted by a framework that owns every byte of device memory through its own
// pool, and serving loops that forbid allocation after start-up.  They also
// cannot hand pkv_attention a workspace of their own.  This entry point takes
// the split-context scratch (merge counters, partial outputs and their
// log-sum-exp statistics) from one fixed array compiled into the library.
//
// The array lives for the whole process on every GPU that loads the library.
// Its name, used in host code, is only a host-side stand-in for the symbol:
// the device address is fetched once per device with cudaGetSymbolAddress,
// with that device current, and passed to the kernels.  Every call shares the
// array, so calls that overlap on the GPU (two streams, or two host threads)
// race on it and must be serialised by the caller.
#include <cstdio>
#include <mutex>

#include "../../include/pagedkv.h"
#include "pkv_internal.h"

namespace {

// The scratch: PKV_NOALLOC_SCRATCH_BYTES bytes per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

extern "C" int pkv_attention_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                     const int32_t* block_tables, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, float scale, void* out,
                                     const pkv_dims* dims, cudaStream_t stream) {
  // Sizes first: dims the array cannot hold are an error, not an allocation.
  const size_t need = pkv_attention_workspace_size(dims);  // 0: bad dims (message set)
  if (need == 0) return PKV_ERR_INVALID;
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
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || ptr == nullptr) {
        pkv::set_error_message("pkv_attention_noalloc: cudaGetSymbolAddress of the scratch failed");
        return PKV_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = ptr;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // The array keeps the previous call's contents; its head (merge counters,
  // prefill work queue, plan cache) must start at zero: its extent moves with
  // the dims.
  int sm_count = 1;
  if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    pkv::set_error_message("pkv_attention_noalloc: cudaDeviceGetAttribute failed");
    return PKV_ERR_CUDA;
  }
  const pkv::WorkspaceLayout w = pkv::decode_workspace_layout(
      dims->num_q_tokens, dims->num_kv_heads, dims->num_q_heads / dims->num_kv_heads, sm_count);
  if (w.ml_off > 0 && cudaMemsetAsync(scratch, 0, w.ml_off, stream) != cudaSuccess) {
    pkv::set_error_message("pkv_attention_noalloc: clearing the scratch counters failed");
    return PKV_ERR_CUDA;
  }
  return pkv_attention(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc, scale, out,
                       dims, scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
