// pkv_cascade.cu -- set-up of a shared-prefix (cascade) attention call.
//
// Requests batched together that share a prompt read the same KV blocks; the
// cascade reads those blocks once per batch (The Serving Playbook, "The tree
// changes what the scheduler should do").  A call names its sharing groups:
// contiguous runs of requests whose first few block-table entries are the
// same physical blocks.  The prefix pass (the prefill kernel in prefix mode)
// attends every member's query rows to the shared blocks at once and leaves
// a partial state per row; the decode kernel then reads each member's blocks
// from its first unshared one and merges the prefix partial by log-sum-exp.
//
// This file holds the small kernel that turns the group description into the
// per-request first block the decode plan reads.
#include "pkv_internal.h"

namespace pkv {
namespace {

// One warp per group: every member's first block is the group's shared
// block count.  first_block was cleared (all zero) before this launch.
__global__ void __launch_bounds__(256) cascade_prep_kernel(CascadePrepParams p) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int g = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (g >= p.num_groups) return;
  const int first = __ldg(p.grp_first + g), n = __ldg(p.grp_count + g);
  const int nb = __ldg(p.grp_blocks + g);
  if (first < 0 || n < 1 || (long long)first + n > p.num_reqs || nb < 0 || nb > p.max_blocks) {
    if (lane == 0) record_error(p.err, kErrBounds);
    return;
  }
  for (int i = lane; i < n; i += 32) p.first_block[first + i] = nb;
}

}  // namespace

cudaError_t launch_cascade_prep(const CascadePrepParams& p, cudaStream_t stream) {
  if (p.num_groups <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = ((long long)p.num_groups * 32 + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, cascade_prep_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pkv
