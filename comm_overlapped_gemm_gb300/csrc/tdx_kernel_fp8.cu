// e4m3 instantiations of the fused kernel (tcgen05.mma kind::f8f6f4, e4m3 inputs, fp32
// accumulate; per-tensor scales applied once in the output epilogue for AllGather, and to each
// rank's partial before the fixed-order fold for ReduceScatter).
#include "tdx_kernel.cuh"

namespace tdx {

cudaError_t launch_fused_fp8(int op, int block_n, int pm, const KParams& p, int grid, cudaStream_t stream) {
  if (pm != 0) {
    if (pm != 2) return cudaErrorInvalidValue;
    if (block_n == 512)
      return op == OP_AG ? launch_fused_t<512, true, OP_AG, 2>(p, grid, stream)
                         : launch_fused_t<512, true, OP_RS, 2>(p, grid, stream);
    if (block_n != 256) return cudaErrorInvalidValue;
    return op == OP_AG ? launch_fused_t<256, true, OP_AG, 2>(p, grid, stream)
                       : launch_fused_t<256, true, OP_RS, 2>(p, grid, stream);
  }
  if (op == OP_AG) {
    switch (block_n) {
      case 128: return launch_fused_t<128, true, OP_AG, 0>(p, grid, stream);
      case 256: return launch_fused_t<256, true, OP_AG, 0>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (block_n) {
    case 128: return launch_fused_t<128, true, OP_RS, 0>(p, grid, stream);
    case 256: return launch_fused_t<256, true, OP_RS, 0>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int fused_max_grid_fp8(int op, int pm, int sms, int block_n) {
  if (pm == 0) return sms;
  if (pm != 2) return 0;
  if (block_n == 512)
    return op == OP_AG ? max_grid_t<512, true, OP_AG, 2>(sms) : max_grid_t<512, true, OP_RS, 2>(sms);
  return op == OP_AG ? max_grid_t<256, true, OP_AG, 2>(sms) : max_grid_t<256, true, OP_RS, 2>(sms);
}

}  // namespace tdx
