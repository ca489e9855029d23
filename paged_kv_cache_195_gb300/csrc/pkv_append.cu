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

__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  grid_dependency_wait();  // inputs and pool may belong to the previous kernel
  allow_dependent_launch();
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
