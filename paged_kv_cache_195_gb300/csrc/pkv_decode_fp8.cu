// pkv_decode_fp8.cu -- the decode kernel (pkv_decode_kernel.cuh) instantiated
// for e4m3 pools with per-KV-head scales (What Actually Runs the Model, "The
// KV cache"; The Serving Playbook, "Quantized serving").  A translation unit
// of its own so that the two element types compile in parallel.
#include "pkv_decode_kernel.cuh"

namespace pkv {

cudaError_t launch_decode_e4m3(const DecodeParams& p, int group, int grid, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_g<1, KvE4m3>(p, grid, stream);
    case 2: return launch_decode_g<2, KvE4m3>(p, grid, stream);
    case 3: return launch_decode_g<3, KvE4m3>(p, grid, stream);
    case 4: return launch_decode_g<4, KvE4m3>(p, grid, stream);
    case 5: return launch_decode_g<5, KvE4m3>(p, grid, stream);
    case 6: return launch_decode_g<6, KvE4m3>(p, grid, stream);
    case 7: return launch_decode_g<7, KvE4m3>(p, grid, stream);
    case 8: return launch_decode_g<8, KvE4m3>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
