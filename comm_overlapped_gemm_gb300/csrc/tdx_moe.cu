// Mixture-of-experts AllToAll dispatch + grouped GEMM and grouped GEMM + AllToAll combine: the
// routing-layout kernel and the instantiations of the fused kernel for OP_MOE (bf16, e4m3) and
// OP_MOE_COMBINE (bf16).
//
// The Triton-distributed article (cronfeed.work), section "DITRON adds three levels of tiling",
// lists AllToAll among the collectives split into chunks and paired with compute tiles, and notes
// that device-level tiles are dynamically sized because the tokens routed to each expert are known
// only at run time. Here the layout is computed on the device from the top-k expert ids: the
// receive buffer groups the routed rows by expert (experts ascending; inside an expert, source rank
// then token ascending), and the tile table cuts every expert's rows into 128-row GEMM tiles, so
// the GEMM's work list follows the routing without a round trip to the host.
#include "tdx_kernel.cuh"

namespace tdx {

namespace {

constexpr int kLayoutThreads = 1024;   // 32 warps: one (token, slot) pair per thread per round

// Exclusive prefix sum of one value per thread over the 1024-thread block; *total gets the sum.
// Every thread of the block must call it.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int res = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  if (total != nullptr) *total = warp_sums[31];
  __syncthreads();   // warp_sums may be reused by the next call
  return res;
}

// One CTA per source rank s. Every CTA counts the (rank, expert) table of all ranks (the same
// table in each), derives the expert offsets and its own rank's start inside every expert block,
// then gives its (token, slot) pairs their rows in pair order t*k + j: within a 1024-pair round a
// warp ranks equal experts with a match mask, per-warp counts are prefix-summed across warps per
// expert, and a running count per expert carries over rounds, so the order is stable. CTA 0 also
// writes the expert offsets and the tile table.
__global__ void __launch_bounds__(kLayoutThreads, 1) tdx_moe_layout_kernel(const __grid_constant__ MoeLayoutParams q) {
  extern __shared__ int lsm[];
  const int W = q.W, E = q.E;
  int* cnt = lsm;                 // [W][E] tokens of rank r routed to expert e
  int* wcnt = cnt + W * E;        // [32][E] per-warp counts of the current round
  int* run = wcnt + 32 * E;       // [E] pairs of this rank already placed per expert
  int* segb = run + E;            // [E] first row of this rank's pairs in expert e's block
  int* tot = segb + E;            // [E] pairs of the current round per expert
  __shared__ int warp_sums[32];
  __shared__ int bad_id;
  __shared__ int bad_flag;
  __shared__ int ntiles;
  const int s = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int pairs = q.T * q.k;

  for (int i = tid; i < W * E; i += kLayoutThreads) cnt[i] = 0;
  for (int i = tid; i < E; i += kLayoutThreads) run[i] = 0;
  if (tid == 0) {
    bad_flag = 0;
    bad_id = 0;
  }
  __syncthreads();
  for (int r = 0; r < W; ++r) {
    const int32_t* idx = q.topk[r];
    for (int i = tid; i < pairs; i += kLayoutThreads) {
      const int e = idx[i];
      if (e < 0 || e >= E) {
        if (atomicExch(&bad_flag, 1) == 0) bad_id = e;
        continue;
      }
      atomicAdd(&cnt[r * E + e], 1);
    }
  }
  __syncthreads();
  if (bad_flag) {
    // invalid routing: no tile, no copy; the fused kernel that follows does nothing
    if (s == 0 && tid == 0) {
      q.ntiles[0] = 0;
      q.ntiles[1] = 1;
      if (atomicCAS(&q.status[0], 0u, static_cast<uint32_t>(DEV_BAD_INPUT)) == 0u) {
        q.status[1] = ROLE_LAYOUT;
        q.status[2] = 0;
        q.status[3] = 0;
        q.status[4] = static_cast<uint32_t>(bad_id);
        q.status[5] = static_cast<uint32_t>(E);
        __threadfence();
      }
    }
    return;
  }
  // expert totals, offsets and this rank's start in every expert block
  int n_e = 0;
  if (tid < E)
    for (int r = 0; r < W; ++r) n_e += cnt[r * E + tid];
  int total_rows = 0;
  const int off_e = block_exclusive_scan(n_e, warp_sums, &total_rows);
  if (tid < E) {
    int b = off_e;
    for (int r = 0; r < s; ++r) b += cnt[r * E + tid];
    segb[tid] = b;
  }
  if (s == 0) {
    // expert offsets and the tile table: expert e's rows [off_e, off_e + n_e) in 128-row tiles
    int tc = (n_e + kBM - 1) / kBM;
    if (q.pair) tc = (tc + 1) & ~1;   // CTA pairs: an even count per expert (a padded tile stores nothing)
    const int toff = block_exclusive_scan(tc, warp_sums, &ntiles);
    if (tid < E) {
      q.offsets[tid] = off_e;
      if (q.user_offsets != nullptr) q.user_offsets[tid] = off_e;
      for (int i = 0; i < tc && toff + i < q.max_tiles; ++i)
        q.tiles[toff + i] = make_int4(off_e + i * kBM, off_e + n_e, tid, 0);
    }
    if (tid == 0) {
      q.offsets[E] = total_rows;
      if (q.user_offsets != nullptr) q.user_offsets[E] = total_rows;
      q.ntiles[0] = ntiles < q.max_tiles ? ntiles : q.max_tiles;
      q.ntiles[1] = 0;
    }
  }
  __syncthreads();
  // stable rows of this rank's pairs
  const int32_t* idx = q.topk[s];
  for (int base = 0; base < pairs; base += kLayoutThreads) {
    for (int i = tid; i < 32 * E; i += kLayoutThreads) wcnt[i] = 0;
    __syncthreads();
    const int pi = base + tid;
    const int e = pi < pairs ? idx[pi] : -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int lrank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && lrank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (tid < E) {
      int acc = 0;
      for (int w = 0; w < 32; ++w) {
        const int c = wcnt[w * E + tid];
        wcnt[w * E + tid] = acc;
        acc += c;
      }
      tot[tid] = acc;
    }
    __syncthreads();
    if (e >= 0) {
      const int row = segb[e] + run[e] + wcnt[warp * E + e] + lrank;
      q.dest[static_cast<size_t>(s) * pairs + pi] = row;
      q.src[row] = s * q.T + pi / q.k;
    }
    __syncthreads();
    if (tid < E) run[tid] += tot[tid];
  }
}

size_t layout_smem_bytes(int W, int E) { return static_cast<size_t>(W * E + 32 * E + 3 * E) * sizeof(int); }

}  // namespace

cudaError_t launch_moe_layout(const MoeLayoutParams& q, cudaStream_t stream) {
  if (q.W < 1 || q.W > kMaxW || q.E < 1 || q.E > kMoeMaxExperts) return cudaErrorInvalidValue;
  const size_t smem = layout_smem_bytes(q.W, q.E);
  static std::atomic<bool> attr_done[64];   // per device; calls may come from several host threads
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (!(dev >= 0 && dev < 64 && attr_done[dev].load(std::memory_order_relaxed))) {
    const cudaError_t e = cudaFuncSetAttribute(tdx_moe_layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(layout_smem_bytes(kMaxW, kMoeMaxExperts)));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_relaxed);
  }
  tdx_moe_layout_kernel<<<q.W, kLayoutThreads, smem, stream>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_fused_moe_bf16(int block_n, int pm, const KParams& p, int grid, cudaStream_t stream) {
  if (pm == 2)
    return block_n == 256   ? launch_fused_t<256, false, OP_MOE, 2>(p, grid, stream)
           : block_n == 512 ? launch_fused_t<512, false, OP_MOE, 2>(p, grid, stream)
                            : cudaErrorInvalidValue;
  switch (block_n) {
    case 64: return launch_fused_t<64, false, OP_MOE, 0>(p, grid, stream);
    case 128: return launch_fused_t<128, false, OP_MOE, 0>(p, grid, stream);
    case 256: return launch_fused_t<256, false, OP_MOE, 0>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fused_moe_combine_bf16(int block_n, int pm, const KParams& p, int grid, cudaStream_t stream) {
  if (pm == 2)
    return block_n == 256   ? launch_fused_t<256, false, OP_MOE_COMBINE, 2>(p, grid, stream)
           : block_n == 512 ? launch_fused_t<512, false, OP_MOE_COMBINE, 2>(p, grid, stream)
                            : cudaErrorInvalidValue;
  switch (block_n) {
    case 64: return launch_fused_t<64, false, OP_MOE_COMBINE, 0>(p, grid, stream);
    case 128: return launch_fused_t<128, false, OP_MOE_COMBINE, 0>(p, grid, stream);
    case 256: return launch_fused_t<256, false, OP_MOE_COMBINE, 0>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fused_moe_fp8(int block_n, int pm, const KParams& p, int grid, cudaStream_t stream) {
  if (pm == 2)
    return block_n == 256   ? launch_fused_t<256, true, OP_MOE, 2>(p, grid, stream)
           : block_n == 512 ? launch_fused_t<512, true, OP_MOE, 2>(p, grid, stream)
                            : cudaErrorInvalidValue;
  switch (block_n) {
    case 128: return launch_fused_t<128, true, OP_MOE, 0>(p, grid, stream);
    case 256: return launch_fused_t<256, true, OP_MOE, 0>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int fused_max_grid_moe(bool combine, int pm, int sms, bool fp8, int block_n) {
  if (pm != 2) return sms;
  if (block_n == 512)
    return combine ? max_grid_t<512, false, OP_MOE_COMBINE, 2>(sms)
                   : (fp8 ? max_grid_t<512, true, OP_MOE, 2>(sms) : max_grid_t<512, false, OP_MOE, 2>(sms));
  if (fp8) return max_grid_t<256, true, OP_MOE, 2>(sms);
  return combine ? max_grid_t<256, false, OP_MOE_COMBINE, 2>(sms) : max_grid_t<256, false, OP_MOE, 2>(sms);
}

}  // namespace tdx
