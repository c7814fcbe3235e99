// bf16 instantiations of the fused kernel (tcgen05.mma kind::f16, bf16 inputs, fp32 accumulate).
#include "tdx_kernel.cuh"

namespace tdx {

cudaError_t launch_fused_bf16(int op, int block_n, int pm, const KParams& p, int grid, cudaStream_t stream) {
  if (pm != 0) {
    if (pm != 2) return cudaErrorInvalidValue;
    if (block_n == 512)
      return op == OP_AG ? launch_fused_t<512, false, OP_AG, 2>(p, grid, stream)
                         : launch_fused_t<512, false, OP_RS, 2>(p, grid, stream);
    if (block_n != 256) return cudaErrorInvalidValue;
    return op == OP_AG ? launch_fused_t<256, false, OP_AG, 2>(p, grid, stream)
                       : launch_fused_t<256, false, OP_RS, 2>(p, grid, stream);
  }
  if (op == OP_AG) {
    switch (block_n) {
      case 64: return launch_fused_t<64, false, OP_AG, 0>(p, grid, stream);
      case 128: return launch_fused_t<128, false, OP_AG, 0>(p, grid, stream);
      case 256: return launch_fused_t<256, false, OP_AG, 0>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (block_n) {
    case 64: return launch_fused_t<64, false, OP_RS, 0>(p, grid, stream);
    case 128: return launch_fused_t<128, false, OP_RS, 0>(p, grid, stream);
    case 256: return launch_fused_t<256, false, OP_RS, 0>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int fused_max_grid_bf16(int op, int pm, int sms, int block_n) {
  if (pm == 0) return sms;
  if (pm != 2) return 0;
  if (block_n == 512)
    return op == OP_AG ? max_grid_t<512, false, OP_AG, 2>(sms) : max_grid_t<512, false, OP_RS, 2>(sms);
  return op == OP_AG ? max_grid_t<256, false, OP_AG, 2>(sms) : max_grid_t<256, false, OP_RS, 2>(sms);
}

// Zero-fill used for the degenerate K == 0 product (C = 0).
__global__ void tdx_fill_zero_kernel(uint4* dst, size_t n16, uint8_t* tail, size_t ntail) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
    dst[i] = make_uint4(0u, 0u, 0u, 0u);
  if (blockIdx.x == 0)
    for (size_t i = threadIdx.x; i < ntail; i += blockDim.x) tail[i] = 0;
}

cudaError_t launch_fill_zero(void* dst, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  const size_t n16 = bytes / 16;
  size_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks == 0) blocks = 1;
  tdx_fill_zero_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<uint4*>(dst), n16, reinterpret_cast<uint8_t*>(dst) + n16 * 16, bytes - n16 * 16);
  return cudaGetLastError();
}

int fused_smem_bytes(int block_n, bool fp8) {   // single-CTA configurations
  if (fp8) {
    switch (block_n) {
      case 128: return Cfg<128, true>::SMEM_BYTES;
      case 256: return Cfg<256, true>::SMEM_BYTES;
      default: return 0;
    }
  }
  switch (block_n) {
    case 64: return Cfg<64, false>::SMEM_BYTES;
    case 128: return Cfg<128, false>::SMEM_BYTES;
    case 256: return Cfg<256, false>::SMEM_BYTES;
    default: return 0;
  }
}

}  // namespace tdx
