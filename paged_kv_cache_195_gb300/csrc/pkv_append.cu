// pkv_append.cu -- KV append: scatter this step's K/V rows into pool slots.
//
// Each new token's key and value join the cache at the slot the block
// manager assigned (LLM 7 - Efficient LLM Serving, sec. 3 "What the Cache
// Stores"; The Serving Playbook, "CUDA graphs and the CPU you forgot about"
// for the slot mapping as a step buffer).  The work is a pure bit copy, bound
// by HBM: one warp moves one (token, KV head) pair, half a warp per tensor,
// 16 lanes x 16 bytes = one 256-byte row, fully coalesced on both sides.
#include "pkv_internal.h"

namespace pkv {

// Debug-only per-block timeline (entry, past the grid-dependency wait, row
// written by thread 0), read together with the decode kernel's.
#if PKV_TC_TRACE >= 3
constexpr int kApTrBlocks = 256, kApTrSlots = 32;
__device__ unsigned long long g_ap_trace[kApTrSlots][kApTrBlocks][4];
#define AP_TR(ev) do { if (threadIdx.x == 0 && blockIdx.x < kApTrBlocks) g_ap_trace[(uint32_t)((reinterpret_cast<uintptr_t>(p.k_new) >> 8) * 0x9E3779B1u) >> 27][blockIdx.x][ev] = global_timer_ns(); } while (0)
cudaError_t append_trace(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, g_ap_trace, bytes < sizeof(g_ap_trace) ? bytes : sizeof(g_ap_trace));
}
#else
#define AP_TR(ev) do { } while (0)
#endif

__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  AP_TR(0);
  if (p.early_trigger) allow_dependent_launch();
  grid_dependency_wait();  // inputs and pool may belong to the previous kernel
  if (!p.early_trigger) allow_dependent_launch();
  AP_TR(1);
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= p.num_tokens * p.num_kv_heads) return;
  const int t = warp / p.num_kv_heads;
  const int h = warp - t * p.num_kv_heads;
  const long long slot = p.slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= (long long)p.num_blocks * kBlockSize) {
    if (lane == 0) record_error(p.err, kErrBounds);
    return;
  }
  const long long blk = slot / kBlockSize;
  const int off = (int)(slot - blk * kBlockSize);
  const int half = lane >> 4;  // 0: K, 1: V
  const int c = lane & 15;     // 16-byte chunk of the 256-byte row
  const uint4* src = reinterpret_cast<const uint4*>(half ? p.v_new : p.k_new) +
                     ((long long)t * p.num_kv_heads + h) * (kHeadDim / 8) + c;
  uint4* dst = reinterpret_cast<uint4*>(half ? p.v_pool : p.k_pool) +
               ((blk * p.num_kv_heads + h) * kBlockSize + off) * (kHeadDim / 8) + c;
  *dst = __ldg(src);
  AP_TR(2);
}

// Quantising append into e4m3 pools (The Serving Playbook, "Quantized
// serving"): each element becomes the code nearest to x / scale[KV head]
// (round to nearest even on the fp32 quotient, saturated to +-448).  Same
// warp layout as the bf16 append; a lane reads 16 bytes and writes 8.
__global__ void __launch_bounds__(256) append_fp8_kernel(AppendFp8Params p) {
  if (p.early_trigger) allow_dependent_launch();
  grid_dependency_wait();  // inputs and pool may belong to the previous kernel
  if (!p.early_trigger) allow_dependent_launch();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= p.num_tokens * p.num_kv_heads) return;
  const int t = warp / p.num_kv_heads;
  const int h = warp - t * p.num_kv_heads;
  const long long slot = p.slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= (long long)p.num_blocks * kBlockSize) {
    if (lane == 0) record_error(p.err, kErrBounds);
    return;
  }
  const long long blk = slot / kBlockSize;
  const int off = (int)(slot - blk * kBlockSize);
  const int half = lane >> 4;  // 0: K, 1: V
  const int c = lane & 15;     // 8 elements of the 128-element row
  const float sc = __ldg((half ? p.v_scale : p.k_scale) + h);
  const uint4 w = __ldg(reinterpret_cast<const uint4*>(half ? p.v_new : p.k_new) +
                        ((long long)t * p.num_kv_heads + h) * (kHeadDim / 8) + c);
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t code[2] = {0u, 0u};
  #pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = bf16x2_to_float2(in[i]);
    const float2 y = make_float2(__fdiv_rn(x.x, sc), __fdiv_rn(x.y, sc));
    const uint32_t two = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
    code[i >> 1] |= two << (16 * (i & 1));
  }
  uint2* dst = reinterpret_cast<uint2*>(half ? p.v_pool : p.k_pool) +
               ((blk * p.num_kv_heads + h) * kBlockSize + off) * (kHeadDim / 8) + c;
  *dst = make_uint2(code[0], code[1]);
}

cudaError_t launch_append_fp8(const AppendFp8Params& p, cudaStream_t stream) {
  const long long warps = (long long)p.num_tokens * p.num_kv_heads;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, append_fp8_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const long long warps = (long long)p.num_tokens * p.num_kv_heads;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, append_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkv
