// pkv_decode.cu -- host side of the decode kernel (grid, workspace layout,
// dispatch by group size) and its bf16-pool instantiations.  The kernel
// itself is in pkv_decode_kernel.cuh; pkv_decode_fp8.cu instantiates it for
// e4m3 pools.
#include "pkv_decode_kernel.cuh"

namespace pkv {

#if PKV_TRACE
cudaError_t decode_trace(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace));
}
#endif

int decode_ctas_per_sm(int group) {
  switch (group) {
    case 1: return DecodeCfg<1>::kMinCtas;
    case 2: return DecodeCfg<2>::kMinCtas;
    case 3: return DecodeCfg<3>::kMinCtas;
    case 4: return DecodeCfg<4>::kMinCtas;
    case 5: return DecodeCfg<5>::kMinCtas;
    case 6: return DecodeCfg<6>::kMinCtas;
    case 7: return DecodeCfg<7>::kMinCtas;
    default: return DecodeCfg<8>::kMinCtas;
  }
}

int decode_grid(int sm_count, int group) { return sm_count * decode_ctas_per_sm(group); }

WorkspaceLayout decode_workspace_layout(int num_q_tokens, int num_kv_heads, int group,
                                        int sm_count) {
  WorkspaceLayout w;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  w.num_slots = 2 * sm_count * 2;  // two partial pieces per CTA, up to two CTAs per SM
  w.plan_entries = w.num_slots / 2;  // one per CTA index of the largest grid
  w.cnt_off = 0;
  // The prefill work queue and the plan cache sit inside the
  // zero-initialised head of the workspace.
  w.sched_off = up((size_t)num_q_tokens * num_kv_heads * sizeof(int));
  w.plan_off = w.sched_off + 256;
  w.ml_off = w.plan_off + up((size_t)w.plan_entries * kPlanEntryWords * sizeof(int));
  w.o_off = w.ml_off + up((size_t)w.num_slots * group * 2 * sizeof(float));
  w.total = w.o_off + up((size_t)w.num_slots * group * kHeadDim * sizeof(float));
  return w;
}

cudaError_t launch_decode(const DecodeParams& p, int group, int grid, cudaStream_t stream) {
  if (p.kv_fp8) return launch_decode_e4m3(p, group, grid, stream);
  switch (group) {
    case 1: return launch_decode_g<1, KvBf16>(p, grid, stream);
    case 2: return launch_decode_g<2, KvBf16>(p, grid, stream);
    case 3: return launch_decode_g<3, KvBf16>(p, grid, stream);
    case 4: return launch_decode_g<4, KvBf16>(p, grid, stream);
    case 5: return launch_decode_g<5, KvBf16>(p, grid, stream);
    case 6: return launch_decode_g<6, KvBf16>(p, grid, stream);
    case 7: return launch_decode_g<7, KvBf16>(p, grid, stream);
    case 8: return launch_decode_g<8, KvBf16>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
