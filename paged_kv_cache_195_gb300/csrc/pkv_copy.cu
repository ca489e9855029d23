// pkv_copy.cu -- block copies: copy-on-write of a shared block and swapping
// blocks between the device pool and host memory.
//
// Several block tables may point at one physical block; when one sequence
// diverges it gets a private copy of that block (copy-on-write), and under
// memory pressure a scheduler may move blocks to CPU memory and back (LLM 7 -
// Efficient LLM Serving, sec. 3 "Sharing and Preemption"; The Serving
// Playbook, "Sharing is a reference count", "Preemption, where the folklore
// is wrong").  Both are the same operation on the [blocks, Hkv, 16, 128]
// layout: move whole blocks (all KV heads, K and V) from one pool to another.
// A pool may live in pinned host memory: on this system the GPU reads and
// writes it directly, so a swap is one gather/scatter kernel rather than one
// copy call per block.
#include "pkv_internal.h"

namespace pkv {

__global__ void __launch_bounds__(256) copy_blocks_kernel(CopyParams p) {
  grid_dependency_wait();
  allow_dependent_launch();
  const long long per_block = (long long)p.num_kv_heads * kTileBytes / 16;  // uint4 per tensor
  for (int i = blockIdx.x; i < p.num_pairs; i += gridDim.x) {
    const long long src = p.pairs[2 * i], dst = p.pairs[2 * i + 1];
    if (src < 0 || src >= p.src_blocks || dst < 0 || dst >= p.dst_blocks) {
      if (threadIdx.x == 0) record_error(p.err, kErrBounds);
      continue;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_src) + src * per_block;
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_src) + src * per_block;
    uint4* kd = reinterpret_cast<uint4*>(p.k_dst) + dst * per_block;
    uint4* vd = reinterpret_cast<uint4*>(p.v_dst) + dst * per_block;
    for (long long j = threadIdx.x; j < per_block; j += blockDim.x) {
      kd[j] = ks[j];
      vd[j] = vs[j];
    }
  }
}

cudaError_t launch_copy_blocks(const CopyParams& p, int sm_count, cudaStream_t stream) {
  if (p.num_pairs == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)min(p.num_pairs, sm_count * 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, copy_blocks_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkv
