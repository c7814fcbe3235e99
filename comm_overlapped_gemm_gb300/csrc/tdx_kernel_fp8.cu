// e4m3 instantiations of the fused kernel (tcgen05.mma kind::f8f6f4, e4m3 inputs, fp32
// accumulate, per-tensor scales applied once in the output epilogue).
#include "tdx_kernel.cuh"

namespace tdx {

cudaError_t launch_fused_fp8(int op, int block_n, const KParams& p, int grid, cudaStream_t stream) {
  if (op != OP_AG) return cudaErrorInvalidValue;
  switch (block_n) {
    case 128: return launch_fused_t<128, true, OP_AG>(p, grid, stream);
    case 256: return launch_fused_t<256, true, OP_AG>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tdx
