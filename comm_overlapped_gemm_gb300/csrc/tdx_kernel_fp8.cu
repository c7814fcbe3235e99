// e4m3 instantiations of the fused kernel (tcgen05.mma kind::f8f6f4, e4m3 inputs, fp32
// accumulate, per-tensor scales applied once in the output epilogue).
#include "tdx_kernel.cuh"

namespace tdx {

cudaError_t launch_fused_fp8(int op, int block_n, int pm, const KParams& p, int grid, cudaStream_t stream) {
  if (op != OP_AG) return cudaErrorInvalidValue;
  if (pm != 0) {
    if (block_n != 256) return cudaErrorInvalidValue;
    return pm == 1 ? launch_fused_t<256, true, OP_AG, 1>(p, grid, stream)
                   : launch_fused_t<256, true, OP_AG, 2>(p, grid, stream);
  }
  switch (block_n) {
    case 128: return launch_fused_t<128, true, OP_AG, 0>(p, grid, stream);
    case 256: return launch_fused_t<256, true, OP_AG, 0>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int fused_max_grid_fp8(int op, int pm, int sms) {
  if (pm == 0 || op != OP_AG) return sms;
  return pm == 1 ? max_grid_t<256, true, OP_AG, 1>(sms) : max_grid_t<256, true, OP_AG, 2>(sms);
}

}  // namespace tdx
