// Host side of the C ABI declared in include/tdx.h: argument validation, tiling choice, workspace
// carving (status word, chunk flags, gathered buffer, running-sum / partial-slot buffer, MoE layout
// tables and receive buffer), TMA tensor maps and the launches of the persistent fused kernel and
// of the MoE routing-layout kernel. No arithmetic of the operations happens here.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/tdx.h"
#include "tdx_internal.h"

using namespace tdx;

namespace {

constexpr uint32_t kVersion = (1u << 16) | 1u;   // 1.1: AllReduce, bf16 partials, MoE dispatch and combine

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elt_size(tdx_dtype d) { return d == TDX_BF16 ? 2 : d == TDX_FP8_E4M3 ? 1 : d == TDX_FP32 ? 4 : 0; }

tdx_opts defaults() {
  tdx_opts o;
  std::memset(&o, 0, sizeof(o));
  o.self_rank = 0;
  o.chunk_rows = 0;
  o.out_dtype = TDX_BF16;
  o.scale_a = nullptr;
  o.scale_b = nullptr;
  o.mode = TDX_FUSED;
  o.producer = TDX_PRODUCER_SM;
  o.epoch = 0;
  o.timeout_ns = 2000000000ull;
  o.perturb_seed = 0;
  o.trace = nullptr;
  o.num_sms = 0;
  o.split_k = 0;
  o.block_n = 0;
  o.reduce_mode = 0;
  o.cluster = 0;
  o.bf16_partials = 0;
  return o;
}

// Everything the launch needs that follows from shapes and options alone (no device queries),
// so that tdx_workspace_size and the calls carve the same layout.
struct Plan {
  int op = 0, W = 0, M = 0, M_local = 0, K = 0, N = 0, elt = 2;
  int allreduce = 0;     // op code 2: the ReduceScatter kernel writes every rank's full output
  int bf16_partials = 0; // slotted partials rounded to bf16
  int BN = 256, L = 1, tiles_m = 0, tiles_n = 0, T = 0, num_kb = 0;
  int chunk_rows = 0, n_chunks = 0;
  int reduce_last = 0;
  int CL = 1;            // CTAs per cluster (1 or 2)
  int PM = 0;            // pair mode: 0 single CTAs, 2 two-SM MMA pairs
  int group_n = 1;
  int rank_block = 1;    // RS: positions (in tile groups) per rank block
  int pull_a = 0;        // AG: tiles of whole small shards read A straight from the shards
  size_t off_chunk_flags = 0, off_chunk_cnt = 0, off_chain_flags = 0, off_tile_cnt = 0, off_tile_done = 0;
  size_t off_grid_bar = 0, ctrl_end = 0;
  int coop = 0;          // slotted fold: 0 last arriver, 1 per-tile cooperative, 2 grid-wide (see make_plan)
  size_t off_G = 0, off_S = 0, total = 0;
};

// 512-wide tiles run on 2-SM pairs only (checked with the pair choice below)
bool valid_bn(int bn, bool fp8) {
  return fp8 ? (bn == 128 || bn == 256 || bn == 512) : (bn == 64 || bn == 128 || bn == 256 || bn == 512);
}

int device_sms();

tdx_status make_plan(int op, int W, int Mx, int K, int N, tdx_dtype dtype, const tdx_opts& o, Plan* pl) {
  const bool allreduce = op == kOpAllReduce;
  if (allreduce) op = OP_RS;
  if (op != OP_AG && op != OP_RS) return TDX_ERR_INVALID_ARG;
  if (W < 1 || W > kMaxW || Mx < 0 || K < 0 || N < 0) return TDX_ERR_INVALID_ARG;
  if (dtype != TDX_BF16 && dtype != TDX_FP8_E4M3) return TDX_ERR_INVALID_ARG;
  const bool fp8 = dtype == TDX_FP8_E4M3;
  Plan p;
  p.op = op;
  p.allreduce = allreduce ? 1 : 0;
  p.W = W;
  p.K = K;
  p.N = N;
  p.elt = elt_size(dtype);
  if (op == OP_AG) {
    p.M_local = Mx;
    p.M = W * Mx;
    int cr = o.chunk_rows > 0 ? o.chunk_rows : (Mx < 128 ? Mx : 128);
    if (Mx > 0 && (cr <= 0 || Mx % cr != 0)) return TDX_ERR_INVALID_ARG;
    p.chunk_rows = Mx > 0 ? cr : 1;
    p.n_chunks = Mx > 0 ? Mx / cr : 0;
  } else {
    if (!allreduce && Mx % W != 0) return TDX_ERR_INVALID_ARG;
    p.M = Mx;
    p.M_local = allreduce ? Mx : Mx / W;
  }
  const int kb128 = (int)((static_cast<long long>(K) * p.elt + 127) / 128);   // 128-byte K blocks
  p.tiles_m = (p.M + kBM - 1) / kBM;
  // tile width
  int bn = o.block_n;
  if (bn != 0 && !valid_bn(bn, fp8)) return TDX_ERR_UNSUPPORTED;
  int L = 1;
  if (op == OP_AG) {
    const long long tiles256 = static_cast<long long>(p.tiles_m) * ((N + 255) / 256);
    const bool small = tiles256 * 2 <= kRefSMs && kb128 >= 2;
    if (bn == 0) {
      // small problems: 128-wide tiles with more K splits (a split's CTA re-reads fewer A bytes
      // per output column; 8 x 16 splits measured 15% faster than 16 x 9 splits of 64-wide tiles)
      if (small) bn = (fp8 || N > 64) ? 128 : 64;
      else bn = N > 128 ? 256 : (N > 64 || fp8 ? 128 : 64);
    }
    const long long tiles = static_cast<long long>(p.tiles_m) * ((N + bn - 1) / bn);
    if (o.split_k > 0) {
      L = o.split_k;
    } else if (small && tiles > 0) {
      // one wave of split-K items over the device's SMs (the CTAs of the persistent grid)
      int sms = device_sms();
      if (o.num_sms > 0 && (sms <= 0 || o.num_sms < sms)) sms = o.num_sms;
      if (sms <= 0) sms = kRefSMs;
      L = static_cast<int>(sms / tiles);
    }
    const int kb_bn = (int)((static_cast<long long>(K) * p.elt + k_slice_bytes(bn) - 1) / k_slice_bytes(bn));
    if (L > kMaxSplitK) L = kMaxSplitK;
    if (L > kb_bn) L = kb_bn;
    if (L < 1) L = 1;
  } else {
    if (bn == 0) {
      bn = N > 128 ? 256 : ((N > 64 || fp8) ? 128 : 64);
      // few output tiles: narrower tiles spread the ranks' partial reductions over more CTAs; not for
      // one or two M-tiles, where the run is bound by streaming B_r and 256-wide rows read it best
      // (small-M: 45.8 vs 49.0 us)
      if (bn == 256 && p.tiles_m > 2 && static_cast<long long>(p.tiles_m) * ((N + 255) / 256) < 2 * kRefSMs) bn = 128;
    }
    L = W;
  }
  p.BN = bn;
  p.L = L;
  p.num_kb = (int)((static_cast<long long>(K) * p.elt + k_slice_bytes(bn) - 1) / k_slice_bytes(bn));
  p.tiles_n = (N + bn - 1) / bn;
  p.T = p.tiles_m * p.tiles_n;
  p.group_n = op == OP_RS ? (p.tiles_n < kRsGroupN ? (p.tiles_n > 0 ? p.tiles_n : 1) : kRsGroupN) : p.tiles_n;
  // CTA pairs on vertically adjacent 128 x 256 tiles running one 2-SM MMA stream (cooperation mode
  // 3): large problems with 256-wide tiles and an even M-tile count. Mode 2 (pairs sharing B through
  // multicast loads) is not offered: every CTA loads only into its own shared memory.
  if (o.cluster < 0 || o.cluster > 3) return TDX_ERR_INVALID_ARG;
  if (o.cluster == 2) return TDX_ERR_UNSUPPORTED;
  if (o.reduce_mode < 0 || o.reduce_mode > 3) return TDX_ERR_INVALID_ARG;
  // the grid-wide fold runs on single CTAs
  if (o.reduce_mode == 3 && o.cluster == 3 && L > 1) return TDX_ERR_UNSUPPORTED;
  const bool pair_ok = (bn == 256 || bn == 512) && p.tiles_m % 2 == 0 && p.tiles_m > 0;
  if (o.cluster == 3) {
    if (!pair_ok) return TDX_ERR_UNSUPPORTED;
    p.PM = 2;
  } else if (o.cluster == 0 && pair_ok && static_cast<long long>(L) * p.T >= 4 * kRefSMs &&
             !(o.reduce_mode == 3 && L > 1)) {
    p.PM = 2;
  }
  if (bn == 512 && p.PM != 2) return TDX_ERR_UNSUPPORTED;   // one 512-column accumulator per CTA of a pair
  // Large AllGathers on pairs take 512-column tiles by default: 25% fewer operand bytes per MMA
  // (the large GEMMs are bound by operand bandwidth into the SMs), and the epilogue that the single
  // accumulator leaves exposed only stores C. Measured on GB300 (W=8, 8192 x 8192 x 3584 bf16):
  // fused 0.322 -> 0.313 ms, GEMM alone 0.297 -> 0.276 ms; e4m3 (16384 x 8192 x 8192) fused
  // 0.714 -> 0.693 ms. The ReduceScatter keeps 256 columns: its exposed running-sum epilogue made
  // 512 columns slower (2.28 -> 2.35 ms).
  if (op == OP_AG && o.block_n == 0 && p.PM == 2 && L == 1 && N >= 1024 &&
      static_cast<long long>(p.tiles_m / 2) * ((N + 511) / 512) >= kRefSMs) {
    bn = 512;
    p.BN = bn;
    p.tiles_n = (N + bn - 1) / bn;
    p.T = p.tiles_m * p.tiles_n;
    p.group_n = p.tiles_n;
  }
  p.CL = p.PM == 0 ? 1 : 2;
  {
    const int tg = (p.tiles_m / p.CL) * p.tiles_n;
    const int rb = kRsRankBlock / p.CL;
    p.rank_block = op == OP_RS ? (tg < rb ? (tg > 0 ? tg : 1) : rb) : (tg > 0 ? tg : 1);
  }
  // AllGather with shards smaller than a tile (whole shards per 128-row tile, 8-row aligned): the
  // consumers read A from the shards themselves instead of waiting for the gathered copy
  p.pull_a = (op == OP_AG && p.PM == 0 && Mx > 0 && Mx < kBM && kBM % Mx == 0 && Mx % 8 == 0) ? 1 : 0;
  // reduction of the L chain elements: slotted when a tile's elements run concurrently (K splits;
  // ReduceScatter with fewer than two waves of tiles per rank), else chained through one buffer
  if (o.bf16_partials < 0 || o.bf16_partials > 1) return TDX_ERR_INVALID_ARG;
  // bf16 partials: a rank's partial is rounded before the fold, which the slotted reduction does
  // (a chained running sum would be rounded at every hand-over instead); the grid-wide fold reads
  // fp32 slots only
  if (o.bf16_partials && (op != OP_RS || o.reduce_mode == 1 || o.reduce_mode == 3)) return TDX_ERR_UNSUPPORTED;
  p.bf16_partials = o.bf16_partials;
  if (L > 1) {
    if (o.reduce_mode == 1) p.reduce_last = 0;
    else if (o.reduce_mode >= 2 || p.bf16_partials) p.reduce_last = 1;
    else p.reduce_last = (op == OP_AG || p.T < 2 * kRefSMs) ? 1 : 0;
  }
  // slotted ReduceScatter may take a rank-inner order (blocks of one position) instead
  if (op == OP_RS && p.reduce_last && kSlottedRankInner) p.rank_block = 1;
  // cooperative fold (slotted, single CTAs, fp32 partials): every element of a tile waits for the
  // tile's L partials and folds 1/L of it, instead of the last arriver folding all of it. The wait
  // is safe only when a tile's elements are processed in the same wave of the persistent grid; it is
  // used when all work items fit one wave (a rank-inner order with the grid a multiple of L would
  // also qualify, but that order measured slower on the multi-wave small-M ReduceScatter).
  // (Spreading the folds of a multi-wave schedule over the CTAs that finished their items, as
  // deferred fold tasks, measured slower on the small-M ReduceScatter than the last arriver: with
  // the rank-outer order the tiles complete only at the end, while the last arriver's slots are
  // still in L2.)
  // Grid-wide fold (coop 2): when the work takes several waves but there are fewer tiles than CTAs,
  // the last arrivers of the few tiles would fold them alone at the end while the other CTAs idle.
  // Instead every CTA, once it has stored all its partials, arrives at a grid barrier (all CTAs are
  // resident: a cooperative launch), and then folds 1/grid of every tile's (row, 32-column) units.
  if (p.reduce_last && p.PM == 0 && !p.bf16_partials && L > 1) {
    int sms = device_sms();
    if (o.num_sms > 0 && (sms == 0 || o.num_sms < sms)) sms = o.num_sms;
    if (o.reduce_mode == 3) p.coop = 2;
    else if (sms > 0 && static_cast<long long>(L) * p.T <= sms) p.coop = 1;
    else if (sms > 0 && p.T < sms) p.coop = 2;
  }
  // workspace layout
  size_t off = kHeaderBytes;
  const size_t n_chunk_words = op == OP_AG ? static_cast<size_t>(W) * p.n_chunks : 0;
  p.off_chunk_flags = off;
  off += n_chunk_words * 4;
  p.off_chunk_cnt = off;
  off += n_chunk_words * 4;
  p.off_chain_flags = off;
  off += static_cast<size_t>(L > 1 && !p.reduce_last ? L - 1 : 0) * p.T * 4;
  p.off_tile_cnt = off;
  off += static_cast<size_t>(p.reduce_last ? p.T : 0) * 4;
  p.off_tile_done = off;   // cooperative fold: elements done folding per tile (reset by the last)
  off += static_cast<size_t>(p.reduce_last ? p.T : 0) * 4;
  p.off_grid_bar = off;    // grid-wide fold: CTAs arrived, CTAs departed (reset by the last to depart)
  off += p.reduce_last ? 8 : 0;
  off = align_up(off, 1024);
  p.ctrl_end = off;
  if (op == OP_AG) {
    p.off_G = off;
    off = align_up(off + static_cast<size_t>(p.M) * K * p.elt, 1024);
  }
  if (L > 1) {
    p.off_S = off;
    const size_t slots = p.reduce_last ? static_cast<size_t>(L) : 1;
    off = align_up(off + slots * static_cast<size_t>(p.T) * kBM * bn * (p.bf16_partials ? 2 : 4), 1024);
  }
  p.total = off;
  *pl = p;
  return TDX_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2D map over a row-major (rows x cols) matrix; box = box_cols x box_rows; 128- or 64-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, bool fp8, long long rows, long long cols, int box_cols,
              int box_rows, int swizzle_bytes = 128) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const int elt = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elt};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3D map with explicit byte strides of dimensions 1 and 2 (any order of sizes: a view may step a
// smaller distance in dimension 2 than in dimension 1); 128-byte swizzle, 128-byte box rows.
bool make_map_3d_strided(CUtensorMap* m, const void* base, bool fp8, long long d0, long long d1, long long d2,
                         long long stride1, long long stride2, int b0, int b1, int b2) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1), static_cast<cuuint64_t>(d2)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride1), static_cast<cuuint64_t>(stride2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(b0), static_cast<cuuint32_t>(b1), static_cast<cuuint32_t>(b2)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// B (K x N row-major) of a single-CTA plan as 128-byte column groups: dimension 0 the 128 bytes of
// one group, 1 the K rows, 2 the groups (128 bytes apart), so that one box holds a K slice across
// the whole tile width in the same shared-memory image as the tile's 2D boxes side by side. Only
// when N is whole groups: the last group of a ragged N would read past the matrix, where a 2D
// map fills zeros. Returns false (the caller keeps 2D maps) when the form does not apply.
bool make_b_groups_map(CUtensorMap* m, const void* B, const Plan& pl, int K, int N) {
  const int gn = 128 / pl.elt;
  if (pl.PM != 0 || N % gn != 0) return false;
  const int groups = pl.BN / gn;
  return make_map_3d_strided(m, B, pl.elt == 1, gn, K, N / gn, static_cast<long long>(N) * pl.elt, 128, gn,
                             k_slice_bytes(pl.BN) / pl.elt, groups);
}

int device_sms() {
  static std::atomic<int> cache[64];   // per device; calls may come from several host threads
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

tdx_status fill_zero(void* p, size_t bytes, cudaStream_t s) {
  return launch_fill_zero(p, bytes, s) == cudaSuccess ? TDX_OK : TDX_ERR_CUDA;
}

tdx_status launch(const Plan& pl, KParams& kp, bool fp8, int grid, cudaStream_t stream) {
  const cudaError_t e = fp8 ? launch_fused_fp8(pl.op, pl.BN, pl.PM, kp, grid, stream)
                            : launch_fused_bf16(pl.op, pl.BN, pl.PM, kp, grid, stream);
  if (e != cudaSuccess) {
    if (std::getenv("TDX_VERBOSE")) std::fprintf(stderr, "tdx: launch failed: %s\n", cudaGetErrorString(e));
    return TDX_ERR_CUDA;
  }
  return TDX_OK;
}

void fill_common(KParams& kp, const Plan& pl, const tdx_opts& o, uint8_t* ws) {
  kp.W = pl.W;
  kp.M = pl.M;
  kp.K = pl.K;
  kp.N = pl.N;
  kp.M_local = pl.M_local;
  kp.tiles_m = pl.tiles_m;
  kp.tiles_n = pl.tiles_n;
  kp.T = pl.T;
  kp.group_n = pl.group_n;
  kp.rank_block = pl.rank_block;
  kp.L = pl.L;
  kp.num_kb = pl.num_kb;
  kp.status = reinterpret_cast<uint32_t*>(ws);
  kp.chunk_flags = reinterpret_cast<uint32_t*>(ws + pl.off_chunk_flags);
  kp.chunk_cnt = reinterpret_cast<uint32_t*>(ws + pl.off_chunk_cnt);
  kp.chain_flags = reinterpret_cast<uint32_t*>(ws + pl.off_chain_flags);
  kp.sbuf = pl.L > 1 ? reinterpret_cast<float*>(ws + pl.off_S) : nullptr;
  kp.tile_cnt = reinterpret_cast<uint32_t*>(ws + pl.off_tile_cnt);
  kp.tile_done = reinterpret_cast<uint32_t*>(ws + pl.off_tile_done);
  kp.grid_bar = reinterpret_cast<uint32_t*>(ws + pl.off_grid_bar);
  kp.coop_fold = pl.coop;
  kp.reduce_last = pl.reduce_last;
  kp.trace = static_cast<uint32_t*>(o.trace);
  kp.epoch = o.epoch == 0 ? 1u : o.epoch;
  kp.dev_epoch = o.epoch == TDX_EPOCH_DEVICE ? reinterpret_cast<uint32_t*>(ws) + kDevEpochWord : nullptr;
  kp.timeout_ns = o.timeout_ns == 0 ? 2000000000ull : o.timeout_ns;
  kp.perturb = o.perturb_seed;
  kp.mode = o.mode;
  kp.row_bytes = static_cast<long long>(pl.K) * pl.elt;
  // an A tile is re-read by the other N-tiles of its M-tile, a B tile by the other M-tiles (pairs of
  // them with CTA pairs); with a single one of those the operand is read once and streamed
  kp.a_streamed = pl.tiles_n <= 1 ? 1 : 0;
  kp.b_streamed = pl.tiles_m / pl.CL <= 1 ? 1 : 0;
}

// Persistent grid: every CTA resident at once (one per SM; for pairs, the clusters that fit), capped
// by opts.num_sms and, when given, by the number of work items; a multiple of the cluster size.
int grid_for(const tdx_opts& o, const Plan& pl, bool fp8, int items_or_zero) {
  int sms = device_sms();
  if (sms <= 0) return 0;
  int g = fp8 ? fused_max_grid_fp8(pl.op, pl.PM, sms, pl.BN) : fused_max_grid_bf16(pl.op, pl.PM, sms, pl.BN);
  if (g <= 0) return 0;
  if (o.num_sms > 0 && o.num_sms < g) g = o.num_sms;
  if (items_or_zero > 0 && items_or_zero < g) g = items_or_zero;
  // grid-wide fold (several waves, fewer tiles than CTAs): as many CTAs as give every CTA the same
  // number of work items, so that the last wave leaves no CTA idle before the grid barrier. Small-M
  // ReduceScatter (W=8, 256 items): 128 CTAs instead of 152, 36.5 -> 35.6 us.
  if (pl.coop == 2) {
    const long long items = static_cast<long long>(pl.L) * pl.T;
    const long long waves = (items + g - 1) / g;
    if (waves > 1) g = static_cast<int>((items + waves - 1) / waves);
  }
  g -= g % pl.CL;
  return g;
}

// AllGather producer order. The first wave of the persistent grid takes the self rank's tiles (no
// wait) and then tiles of ranks self+1, self+2, ..., which wait for their chunks. The CTAs holding
// those tiles (kp.copy_lo on: the first wave's self tiles come first) copy the chunks those tiles
// wait for (release-order chunks 0..kp.copy_q1-1) themselves, through their operand ring, which is
// idle until then. Otherwise copy_q1 = 0 and every chunk goes round-robin in pieces.
void first_wave_chunks(KParams& kp, const Plan& pl, int grid, int self_rank, bool on) {
  kp.copy_lo = grid;
  kp.copy_q1 = 0;
  if (!on || pl.L != 1 || pl.M_local <= 0 || pl.n_chunks <= 0) return;
  const int CL = pl.CL;
  const int ncl = grid / CL;
  const int tiles_g = pl.tiles_m / CL;
  int start = (self_rank * pl.M_local + CL * kBM - 1) / (CL * kBM);
  if (start >= tiles_g) start = 0;
  const long long self_lo = static_cast<long long>(self_rank) * pl.M_local;
  const long long self_hi = self_lo + pl.M_local;
  int first_wait = -1;
  int q1 = 0;
  for (int pos = 0; pos < ncl && pos < tiles_g * pl.tiles_n; ++pos) {
    int mg = start + pos / pl.tiles_n;
    if (mg >= tiles_g) mg -= tiles_g;
    const long long r0 = static_cast<long long>(mg) * CL * kBM;
    const long long r1 = std::min(r0 + CL * kBM, static_cast<long long>(pl.M));
    if (r0 >= self_lo && r1 <= self_hi) {
      if (first_wait >= 0) return;   // a self tile after a waiting one: keep the round-robin order
      continue;
    }
    if (first_wait < 0) first_wait = pos;
    for (long long r = r0; r < r1; r += pl.chunk_rows) {
      const int j = static_cast<int>(r / pl.M_local);
      const int ck = static_cast<int>((r - static_cast<long long>(j) * pl.M_local) / pl.chunk_rows);
      const int rr = (j - self_rank - 1 + pl.W) % pl.W;   // release order of rank j's chunks
      q1 = std::max(q1, rr * pl.n_chunks + ck + 1);
    }
  }
  if (first_wait > 0 && q1 > 0 && q1 < pl.W * pl.n_chunks) {
    kp.copy_lo = first_wait * CL;
    kp.copy_q1 = q1;
  }
}

// Every host-side check of an AllGather+GEMM call that does not involve the workspace (arguments,
// options, tiling, alignment); fills the plan. Launches nothing.
tdx_status ag_check(const void* const* shards, const void* B, const void* C, int W, int M_local, int K, int N,
                    tdx_dtype dtype, const tdx_opts& o, Plan* pl) {
  if (shards == nullptr || B == nullptr || C == nullptr) return TDX_ERR_INVALID_ARG;
  if (W < 1 || W > kMaxW) return TDX_ERR_INVALID_ARG;
  for (int r = 0; r < W; ++r)
    if (shards[r] == nullptr) return TDX_ERR_INVALID_ARG;
  if (o.self_rank < 0 || o.self_rank >= W) return TDX_ERR_INVALID_ARG;
  if (o.out_dtype != TDX_BF16 && o.out_dtype != TDX_FP32) return TDX_ERR_INVALID_ARG;
  if (o.mode < TDX_FUSED || o.mode > TDX_CONSUMER_ONLY) return TDX_ERR_INVALID_ARG;
  if (o.producer != TDX_PRODUCER_SM && o.producer != TDX_PRODUCER_COPY_ENGINE) return TDX_ERR_INVALID_ARG;
  // The copy-engine producer is not offered: the consumer kernel would wait on copies issued
  // outside it, which need not run while the kernel holds every SM.
  if (o.producer == TDX_PRODUCER_COPY_ENGINE) return TDX_ERR_UNSUPPORTED;
  tdx_status s = make_plan(OP_AG, W, M_local, K, N, dtype, o, pl);
  if (s != TDX_OK) return s;
  const int out_elt = o.out_dtype == TDX_FP32 ? 4 : 2;
  for (int r = 0; r < W; ++r)
    if (!aligned16(shards[r])) return TDX_ERR_ALIGNMENT;
  if (!aligned16(B) || !aligned16(C)) return TDX_ERR_ALIGNMENT;
  if ((static_cast<long long>(K) * pl->elt) % 16 != 0 || (static_cast<long long>(N) * pl->elt) % 16 != 0 ||
      (static_cast<long long>(N) * out_elt) % 16 != 0)
    return TDX_ERR_ALIGNMENT;
  return TDX_OK;
}

// The launches of a checked AllGather+GEMM call on a workspace of at least pl.total bytes.
tdx_status ag_run(const void* const* shards, const void* B, void* C, uint8_t* ws, const Plan& pl, const tdx_opts& o,
                  cudaStream_t st) {
  const int W = pl.W, M_local = pl.M_local, K = pl.K;
  const bool fp8 = pl.elt == 1;
  const int out_elt = o.out_dtype == TDX_FP32 ? 4 : 2;
  if (M_local == 0 || pl.N == 0) return TDX_OK;
  if (K == 0) return fill_zero(C, static_cast<size_t>(pl.M) * pl.N * out_elt, st);
  static thread_local KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  fill_common(kp, pl, o, ws);
  kp.op = OP_AG;
  kp.self_rank = o.self_rank;
  kp.chunk_rows = pl.chunk_rows;
  kp.n_chunks = pl.n_chunks;
  kp.out_fp32 = o.out_dtype == TDX_FP32;
  kp.G = ws + pl.off_G;
  kp.out[0] = static_cast<uint8_t*>(C);
  for (int r = 0; r < W; ++r) {
    kp.shard[r] = static_cast<const uint8_t*>(shards[r]);
    const float sa = (fp8 && o.scale_a) ? o.scale_a[r] : 1.0f;
    const float sb = (fp8 && o.scale_b) ? o.scale_b[0] : 1.0f;
    kp.row_scale[r] = sa * sb;
  }
  kp.chunk_bytes = static_cast<long long>(pl.chunk_rows) * kp.row_bytes;
  kp.trace_chunks = W * pl.n_chunks;
  const int grid = grid_for(o, pl, fp8, 0);
  if (grid <= 0) return TDX_ERR_CUDA;
  // producer copy unit: about one piece per CTA, a multiple of 16 KiB, at most 64 KiB per release
  {
    const long long total = static_cast<long long>(W) * pl.n_chunks * kp.chunk_bytes;
    long long pb = (total / grid + kCopyRoundBytes - 1) / kCopyRoundBytes * kCopyRoundBytes;
    if (pb < kCopyRoundBytes) pb = kCopyRoundBytes;
    if (pb > kMaxPieceBytes) pb = kMaxPieceBytes;
    kp.piece_bytes = static_cast<int>(pb);
  }
  kp.ppc = static_cast<int>((kp.chunk_bytes + kp.piece_bytes - 1) / kp.piece_bytes);
  kp.total_pieces = W * pl.n_chunks * kp.ppc;
  const bool moving = o.mode == TDX_FUSED || o.mode == TDX_MOVE_ONLY;
  kp.copy_active = moving ? 1 : 0;
  kp.pull_a = pl.pull_a;
  kp.wait_flags = (!pl.pull_a && (o.mode == TDX_FUSED || o.mode == TDX_CONSUMER_ONLY)) ? 1 : 0;
  first_wave_chunks(kp, pl, grid, o.self_rank, o.mode == TDX_FUSED && kp.wait_flags);
  kp.total_pieces = (W * pl.n_chunks - kp.copy_q1) * kp.ppc;
  // A: K slices of k_slice_bytes(BN) bytes, 128 rows; B: 128-byte N rows, one K slice deep
  const int ks = k_slice_bytes(pl.BN);
  const int a_box = ks / pl.elt, b_box_n = 128 / pl.elt, b_box_k = ks / pl.elt;
  if (pl.pull_a) {
    // shards at one stride (a symmetric heap: rank r's buffer at base + r * pitch) are one 3D
    // tensor (K, row, rank) and a tile's shards one box; else one map per shard, a box of the whole
    // shard's M_local rows
    const long long pitch = W > 1 ? static_cast<long long>(reinterpret_cast<uintptr_t>(shards[1]) -
                                                            reinterpret_cast<uintptr_t>(shards[0]))
                                  : static_cast<long long>(M_local) * kp.row_bytes;
    bool one_stride = pitch >= static_cast<long long>(M_local) * kp.row_bytes && pitch % 16 == 0;
    for (int r = 2; r < W && one_stride; ++r)
      one_stride = reinterpret_cast<uintptr_t>(shards[r]) ==
                   reinterpret_cast<uintptr_t>(shards[0]) + static_cast<uintptr_t>(r) * static_cast<uintptr_t>(pitch);
    kp.pull_3d = one_stride && make_map_3d_strided(&kp.tm_a[0], shards[0], fp8, K, M_local, W, kp.row_bytes, pitch,
                                                   a_box, M_local, kBM / M_local)
                     ? 1
                     : 0;
    if (!kp.pull_3d)
      for (int r = 0; r < W; ++r)
        if (!make_map(&kp.tm_a[r], shards[r], fp8, M_local, K, a_box, M_local, ks)) return TDX_ERR_CUDA;
  } else if (!make_map(&kp.tm_a[0], kp.G, fp8, pl.M, K, a_box, kBM, ks) ||
             !make_map(&kp.tm_a[1], shards[o.self_rank], fp8, M_local, K, a_box, kBM, ks)) {
    return TDX_ERR_CUDA;
  }
  kp.b_groups = make_b_groups_map(&kp.tm_b[0], B, pl, K, pl.N) ? 1 : 0;
  if (!kp.b_groups && !make_map(&kp.tm_b[0], B, fp8, K, pl.N, b_box_n, b_box_k)) return TDX_ERR_CUDA;
  if (o.epoch == 0) {
    const tdx_status s = fill_zero(ws + pl.off_chunk_flags, pl.ctrl_end - pl.off_chunk_flags, st);
    if (s != TDX_OK) return s;
  }
  return launch(pl, kp, fp8, grid, st);
}

}  // namespace

extern "C" {

tdx_status tdx_opts_default(tdx_opts* opts) {
  if (opts == nullptr) return TDX_ERR_INVALID_ARG;
  *opts = defaults();
  return TDX_OK;
}

tdx_status tdx_workspace_size(int op, int W, int M_local_or_M, int K, int N, tdx_dtype dtype, const tdx_opts* opts,
                              size_t* bytes) {
  if (bytes == nullptr) return TDX_ERR_INVALID_ARG;
  const tdx_opts o = opts ? *opts : defaults();
  Plan pl;
  tdx_status s = make_plan(op, W, M_local_or_M, K, N, dtype, o, &pl);
  if (s != TDX_OK) return s;
  *bytes = pl.total;
  return TDX_OK;
}

tdx_status tdx_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TDX_ERR_WORKSPACE;
  return fill_zero(workspace, bytes, static_cast<cudaStream_t>(stream));
}

tdx_status tdx_ag_gemm(const void* const* shards, const void* B, void* C, void* workspace, size_t workspace_bytes,
                       int W, int M_local, int K, int N, tdx_dtype dtype, const tdx_opts* opts, void* stream) {
  const tdx_opts o = opts ? *opts : defaults();
  Plan pl;
  tdx_status s = ag_check(shards, B, C, W, M_local, K, N, dtype, o, &pl);
  if (s != TDX_OK) return s;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < pl.total)
    return TDX_ERR_WORKSPACE;
  return ag_run(shards, B, C, static_cast<uint8_t*>(workspace), pl, o, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// GEMM+ReduceScatter (allreduce = false: out[j] is output shard j) or GEMM+AllReduce (allreduce =
// true: out[r] is rank r's full M x N output).
tdx_status rs_call(const void* const* A_parts, const void* const* B_parts, void* const* out_shards, void* workspace,
                   size_t workspace_bytes, int W, int M, int K, int N, tdx_dtype dtype, const tdx_opts* opts,
                   void* stream, bool allreduce) {
  const tdx_opts o = opts ? *opts : defaults();
  if (A_parts == nullptr || B_parts == nullptr || out_shards == nullptr) return TDX_ERR_INVALID_ARG;
  if (W < 1 || W > kMaxW) return TDX_ERR_INVALID_ARG;
  for (int r = 0; r < W; ++r)
    if (A_parts[r] == nullptr || B_parts[r] == nullptr || out_shards[r] == nullptr) return TDX_ERR_INVALID_ARG;
  if (o.mode < TDX_FUSED || o.mode > TDX_MOVE_ONLY) return TDX_ERR_INVALID_ARG;
  if (o.out_dtype != TDX_BF16) return TDX_ERR_UNSUPPORTED;
  Plan pl;
  tdx_status s = make_plan(allreduce ? kOpAllReduce : OP_RS, W, M, K, N, dtype, o, &pl);
  if (s != TDX_OK) return s;
  const bool fp8 = dtype == TDX_FP8_E4M3;
  for (int r = 0; r < W; ++r)
    if (!aligned16(A_parts[r]) || !aligned16(B_parts[r]) || !aligned16(out_shards[r])) return TDX_ERR_ALIGNMENT;
  if ((static_cast<long long>(K) * pl.elt) % 16 != 0 || (static_cast<long long>(N) * pl.elt) % 16 != 0 ||
      (static_cast<long long>(N) * 2) % 16 != 0)
    return TDX_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < pl.total)
    return TDX_ERR_WORKSPACE;
  if (M == 0 || N == 0) return TDX_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    for (int r = 0; r < W; ++r) {
      s = fill_zero(out_shards[r], static_cast<size_t>(allreduce ? M : pl.M_local) * N * 2, st);
      if (s != TDX_OK) return s;
    }
    return TDX_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  static thread_local KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  fill_common(kp, pl, o, ws);
  kp.op = OP_RS;
  kp.allreduce = pl.allreduce;
  kp.bf16_partials = pl.bf16_partials;
  // B stays in 2D boxes here: one 4-group box per K slice measured slower on the 128-row
  // ReduceScatter (34.4 against 34.0 us per call)
  for (int r = 0; r < W; ++r) {
    kp.out[r] = static_cast<uint8_t*>(out_shards[r]);
    const int ks = k_slice_bytes(pl.BN);
    if (!make_map(&kp.tm_a[r], A_parts[r], fp8, M, K, ks / pl.elt, kBM, ks) ||
        !make_map(&kp.tm_b[r], B_parts[r], fp8, K, N, 128 / pl.elt, ks / pl.elt))
      return TDX_ERR_CUDA;
    const float sa = (fp8 && o.scale_a) ? o.scale_a[r] : 1.0f;
    const float sb = (fp8 && o.scale_b) ? o.scale_b[r] : 1.0f;
    kp.elem_scale[r] = sa * sb;
  }
  if (o.epoch == 0) {
    s = fill_zero(ws + pl.off_chunk_flags, pl.ctrl_end - pl.off_chunk_flags, st);
    if (s != TDX_OK) return s;
  }
  const int grid = grid_for(o, pl, fp8, pl.L * pl.T);
  if (grid <= 0) return TDX_ERR_CUDA;
  return launch(pl, kp, fp8, grid, st);
}

}  // namespace

extern "C" {

tdx_status tdx_gemm_rs(const void* const* A_parts, const void* const* B_parts, void* const* out_shards,
                       void* workspace, size_t workspace_bytes, int W, int M, int K, int N, tdx_dtype dtype,
                       const tdx_opts* opts, void* stream) {
  return rs_call(A_parts, B_parts, out_shards, workspace, workspace_bytes, W, M, K, N, dtype, opts, stream, false);
}

tdx_status tdx_gemm_ar(const void* const* A_parts, const void* const* B_parts, void* const* out_full, void* workspace,
                       size_t workspace_bytes, int W, int M, int K, int N, tdx_dtype dtype, const tdx_opts* opts,
                       void* stream) {
  return rs_call(A_parts, B_parts, out_full, workspace, workspace_bytes, W, M, K, N, dtype, opts, stream, true);
}

tdx_status tdx_read_device_status(const void* workspace, void* stream, tdx_status* out, uint32_t* detail) {
  if (workspace == nullptr || out == nullptr) return TDX_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t words[kStatusWords];
  if (cudaStreamSynchronize(st) != cudaSuccess) return TDX_ERR_CUDA;
  if (cudaMemcpy(words, workspace, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return TDX_ERR_CUDA;
  *out = static_cast<tdx_status>(words[0]);
  if (detail != nullptr) std::memcpy(detail, words, sizeof(words));
  return TDX_OK;
}

tdx_status tdx_plan_info(int op, int W, int M_local_or_M, int K, int N, tdx_dtype dtype, const tdx_opts* opts,
                         int64_t* info) {
  if (info == nullptr) return TDX_ERR_INVALID_ARG;
  const tdx_opts o = opts ? *opts : defaults();
  Plan pl;
  tdx_status s = make_plan(op, W, M_local_or_M, K, N, dtype, o, &pl);
  if (s != TDX_OK) return s;
  const int64_t v[22] = {pl.BN, pl.L, pl.tiles_m, pl.tiles_n, pl.T, pl.num_kb, pl.chunk_rows, pl.n_chunks,
                         (int64_t)pl.off_chunk_flags, (int64_t)pl.off_chunk_cnt, (int64_t)pl.off_chain_flags,
                         (int64_t)pl.off_G, (int64_t)pl.off_S, (int64_t)pl.total,
                         pl.L > 1 ? (pl.reduce_last ? 2 : 1) : 0, (int64_t)pl.off_tile_cnt, pl.PM + 1, pl.group_n, pl.rank_block, pl.pull_a,
                         pl.bf16_partials ? 2 : 4, pl.coop};
  std::memcpy(info, v, sizeof(v));
  return TDX_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Allocation-free AllGather+GEMM: the workspace is this file-scope device array, shared by every
// call on a device. Host code never dereferences or passes the symbol itself (on the host it is
// only a stand-in); its device address is looked up with cudaGetSymbolAddress, with the device
// current, at the first call on that device and cached together with the unique ID of the CUDA
// context it belongs to. A call made in another context (the device's context was re-created, for
// example after cudaDeviceReset) looks the address up again, so a stale address is never used.
static __device__ __align__(256) uint8_t g_tdx_noalloc_scratch[TDX_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique ID of the calling thread's current CUDA context (IDs are never reused within a process).
tdx_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_cur == nullptr || get_id == nullptr) return TDX_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return TDX_ERR_CUDA;
  return get_id(ctx, id) == CUDA_SUCCESS ? TDX_OK : TDX_ERR_CUDA;
}

tdx_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TDX_ERR_CUDA;
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx) == TDX_OK;   // false before the runtime made one current
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!have_ctx || g_noalloc_ptr[dev] == nullptr || g_noalloc_ctx[dev] != ctx) {
    // set-up: the lookup also makes the device's primary context current if none was
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tdx_noalloc_scratch) != cudaSuccess || p == nullptr) return TDX_ERR_CUDA;
    if (current_context_id(&ctx) != TDX_OK) return TDX_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return TDX_OK;
}

}  // namespace

extern "C" {

tdx_status tdx_ag_gemm_noalloc(const void* const* shards, const void* B, void* C, int W, int M_local, int K,
                               int N, tdx_dtype dtype, const tdx_opts* opts, uint32_t* device_status,
                               void* stream) {
  tdx_opts o = opts ? *opts : defaults();
  o.epoch = 0;   // the shared scratch is cleared by every call
  if (o.producer != TDX_PRODUCER_SM) return TDX_ERR_UNSUPPORTED;
  // every check comes before the first launch: a rejected call enqueues nothing on the shared array
  Plan pl;
  tdx_status s = ag_check(shards, B, C, W, M_local, K, N, dtype, o, &pl);
  if (s != TDX_OK) return s;
  if (pl.total > TDX_NOALLOC_SCRATCH_BYTES) {
    if (std::getenv("TDX_VERBOSE"))
      std::fprintf(stderr, "tdx_ag_gemm_noalloc: problem needs %zu bytes of scratch, the built-in scratch holds %u\n",
                   pl.total, TDX_NOALLOC_SCRATCH_BYTES);
    return TDX_ERR_WORKSPACE;
  }
  if (device_status != nullptr && !aligned16(device_status)) return TDX_ERR_ALIGNMENT;
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != TDX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // status word and details start at zero for this call (flags are cleared by the epoch-0 path)
  s = fill_zero(scratch, kStatusWords * sizeof(uint32_t), st);
  if (s != TDX_OK) return s;
  s = ag_run(shards, B, C, static_cast<uint8_t*>(scratch), pl, o, st);
  if (s != TDX_OK) return s;
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, scratch, kStatusWords * sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
    return TDX_ERR_CUDA;
  return TDX_OK;
}

size_t tdx_trace_size(int grid, int items, int chunks) {
  if (grid <= 0 || items < 0 || chunks < 0) return 0;
  const size_t per_cta = (static_cast<size_t>(items) + grid - 1) / grid;
  return 4 * (4 + kTraceStatWords * static_cast<size_t>(grid) + 1 + static_cast<size_t>(chunks) +
              static_cast<size_t>(grid) * per_cta);
}

const char* tdx_status_string(tdx_status s) {
  switch (s) {
    case TDX_OK: return "TDX_OK";
    case TDX_ERR_INVALID_ARG: return "TDX_ERR_INVALID_ARG: invalid argument";
    case TDX_ERR_UNSUPPORTED: return "TDX_ERR_UNSUPPORTED: request not implemented by the kernels";
    case TDX_ERR_ALIGNMENT: return "TDX_ERR_ALIGNMENT: pointer or row pitch not 16-byte aligned";
    case TDX_ERR_WORKSPACE: return "TDX_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case TDX_ERR_CUDA: return "TDX_ERR_CUDA: a CUDA call failed";
    case TDX_ERR_TIMEOUT: return "TDX_ERR_TIMEOUT: a bounded device wait ran out";
    case TDX_ERR_STALE_EPOCH: return "TDX_ERR_STALE_EPOCH: a flag held an epoch >= the call's epoch";
    default: return "unknown tdx_status";
  }
}

uint32_t tdx_version(void) { return kVersion; }

}  // extern "C"

// ================================================================================================
// Mixture-of-experts AllToAll dispatch + grouped GEMM
// ================================================================================================
namespace {

// Dispatch (combine = false): A = receive buffer (total x H, in the workspace), B = E x H x F, the
// GEMM's N = F. Combine (combine = true): A = the caller's dispatched rows (total x H, here H is the
// GEMM's K = the expert input width), B = E x H x F with F = the combined output width; the
// workspace holds the expert outputs Z (total x F bf16), the slot table and per-(token, N-tile)
// arrival counters instead of the receive buffer.
struct MoePlan {
  int W = 0, T = 0, H = 0, F = 0, E = 0, k = 0, BN = 0, tiles_n = 0, num_kb = 0;
  bool combine = false;
  long long total = 0;              // dispatched rows = W * T * k
  int n_chunks = 0, max_tiles = 0;  // 128-row chunks of the receive buffer; tile-table bound
  int PM = 0;                       // 0 single CTAs, 2 2-SM pairs on two tiles of one expert
  int elt = 2;                      // bytes per input element (bf16 2, e4m3 1)
  size_t off_flags = 0, off_cnt = 0, off_ntiles = 0, off_tokcnt = 0, ctrl_end = 0;
  size_t off_offsets = 0, off_src = 0, off_dest = 0, off_tiles = 0, off_R = 0, bytes = 0;
};

tdx_status make_moe_plan(int W, int T, int H, int F, int E, int k, tdx_dtype dtype, const tdx_opts& o, MoePlan* out,
                         bool combine = false) {
  if (W < 1 || W > kMaxW || T < 0 || H < 0 || F < 0 || E < 1 || k < 1 || k > E) return TDX_ERR_INVALID_ARG;
  if (E > kMoeMaxExperts || (combine && k > kMoeMaxTopk)) return TDX_ERR_UNSUPPORTED;
  if (dtype != TDX_BF16 && dtype != TDX_FP8_E4M3) return TDX_ERR_INVALID_ARG;
  const bool fp8 = dtype == TDX_FP8_E4M3;
  if (fp8 && combine) return TDX_ERR_UNSUPPORTED;
  if (o.split_k > 1 || o.cluster == 2 || o.cluster < 0 || o.cluster > 3 || o.bf16_partials != 0 ||
      o.out_dtype != TDX_BF16)
    return TDX_ERR_UNSUPPORTED;
  MoePlan p;
  p.combine = combine;
  p.elt = fp8 ? 1 : 2;
  p.W = W;
  p.T = T;
  p.H = H;
  p.F = F;
  p.E = E;
  p.k = k;
  p.total = static_cast<long long>(W) * T * k;
  if (p.total > (1ll << 30)) return TDX_ERR_INVALID_ARG;
  int bn = o.block_n;
  if (bn != 0 && bn != 64 && bn != 128 && bn != 256 && bn != 512) return TDX_ERR_UNSUPPORTED;
  if (fp8 && bn == 64) return TDX_ERR_UNSUPPORTED;   // e4m3 B boxes are 128 columns wide
  // 512-column tiles run on 2-SM pairs
  if (bn == 512 && o.cluster == 1) return TDX_ERR_UNSUPPORTED;
  if (bn == 0) bn = F > 128 ? 256 : ((F > 64 || fp8) ? 128 : 64);
  p.BN = bn;
  p.tiles_n = (F + bn - 1) / bn;
  p.num_kb = static_cast<int>((static_cast<long long>(H) * p.elt + 127) / 128);
  p.n_chunks = static_cast<int>((p.total + kBM - 1) / kBM);
  // 2-SM pairs (M = 256 per MMA, two tiles of one expert) when the experts average at least 8 tiles:
  // the tile table then pads every expert to an even tile count (at most one empty tile each). The
  // bf16 dispatch takes pairs from one tile per expert on: at 128 tokens per rank (W=8, top-8 of 64
  // experts, 7168 -> 2048) pairs of 256-wide tiles ran in 417 us against 434 us on single CTAs,
  // while e4m3 ran slower on pairs (230 against 220 us).
  const bool many_tiles = p.total >= 8LL * kBM * E;
  const bool bf16_dispatch_pairs = !fp8 && !combine && p.total >= static_cast<long long>(kBM) * E;
  if (o.cluster == 3 || bn == 512 || (o.cluster == 0 && bn == 256 && (many_tiles || bf16_dispatch_pairs))) {
    if (bn != 256 && bn != 512) return TDX_ERR_UNSUPPORTED;
    p.PM = 2;
  }
  // On pairs the dispatch's grouped GEMM takes 512-column tiles by default: 25% fewer operand bytes
  // per MMA, and it shares the SMs' load path with the dispatch copies. Measured on GB300 (moe_w8:
  // 262144 rows x 7168 -> 2048): fused 5.44 -> 5.02 ms, GEMM alone 4.35 -> 3.96 ms; e4m3 fused
  // 3.04 -> 2.84 ms. The combine keeps 256 (its token folds run in the epilogue, which one
  // accumulator would leave exposed).
  if (o.block_n == 0 && !combine && p.PM == 2 && F >= 1024 && many_tiles) {
    bn = 512;
    p.BN = bn;
    p.tiles_n = (F + bn - 1) / bn;
  }
  p.max_tiles = p.n_chunks + (p.PM == 2 ? 2 : 1) * E;   // a partial tile (and a pad) per expert
  size_t off = kHeaderBytes;
  p.off_flags = off;
  off += static_cast<size_t>(p.n_chunks) * 4;
  p.off_cnt = off;
  off += static_cast<size_t>(p.n_chunks) * 4;
  p.off_ntiles = off;
  off += 8;
  p.off_tokcnt = off;
  if (combine) off += static_cast<size_t>(W) * T * p.tiles_n * 4;
  p.ctrl_end = off = align_up(off, 1024);
  p.off_offsets = off;
  off = align_up(off + static_cast<size_t>(E + 1) * 4, 256);
  p.off_src = off;
  off = align_up(off + static_cast<size_t>(p.total) * 4, 256);
  p.off_dest = off;
  if (combine) off = align_up(off + static_cast<size_t>(p.total) * 4, 256);
  p.off_tiles = off;
  off = align_up(off + static_cast<size_t>(p.max_tiles) * 16, 1024);
  p.off_R = off;   // dispatch: receive buffer (total x H); combine: expert outputs Z (total x F)
  off = align_up(off + static_cast<size_t>(p.total) * (combine ? static_cast<size_t>(F) * 2 : static_cast<size_t>(H) * p.elt),
                 1024);
  p.bytes = off;
  *out = p;
  return TDX_OK;
}

// 3D map over a stack of `depth` row-major (rows x cols) bf16 matrices; box = box_cols x box_rows x 1,
// 128-byte swizzle (the same shared-memory image as the 2D box of one matrix).
bool make_map_3d(CUtensorMap* m, const void* base, long long depth, long long rows, long long cols, int box_cols,
                 int box_rows, bool fp8 = false) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const int elt = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(depth)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * elt, static_cast<cuuint64_t>(rows * cols) * elt};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                   dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

tdx_status tdx_moe_workspace_size(int W, int T, int H, int F, int E, int topk, tdx_dtype dtype, const tdx_opts* opts,
                                  size_t* bytes) {
  if (bytes == nullptr) return TDX_ERR_INVALID_ARG;
  const tdx_opts o = opts ? *opts : defaults();
  MoePlan pl;
  tdx_status s = make_moe_plan(W, T, H, F, E, topk, dtype, o, &pl);
  if (s != TDX_OK) return s;
  *bytes = pl.bytes;
  return TDX_OK;
}

tdx_status tdx_moe_plan_info(int W, int T, int H, int F, int E, int topk, tdx_dtype dtype, const tdx_opts* opts,
                             int64_t* info) {
  if (info == nullptr) return TDX_ERR_INVALID_ARG;
  const tdx_opts o = opts ? *opts : defaults();
  MoePlan pl;
  tdx_status s = make_moe_plan(W, T, H, F, E, topk, dtype, o, &pl);
  if (s != TDX_OK) return s;
  const int64_t v[16] = {pl.BN, pl.tiles_n, pl.max_tiles, pl.n_chunks, pl.total, (int64_t)pl.off_flags,
                         (int64_t)pl.off_ntiles, (int64_t)pl.off_offsets, (int64_t)pl.off_src, (int64_t)pl.off_tiles,
                         (int64_t)pl.off_R, (int64_t)pl.bytes, pl.num_kb, 0, 0, pl.PM == 2 ? 3 : 1};
  std::memcpy(info, v, sizeof(v));
  return TDX_OK;
}

tdx_status tdx_moe_combine_workspace_size(int W, int T, int F, int H, int E, int topk, tdx_dtype dtype,
                                          const tdx_opts* opts, size_t* bytes) {
  if (bytes == nullptr) return TDX_ERR_INVALID_ARG;
  const tdx_opts o = opts ? *opts : defaults();
  MoePlan pl;
  tdx_status s = make_moe_plan(W, T, F, H, E, topk, dtype, o, &pl, true);
  if (s != TDX_OK) return s;
  *bytes = pl.bytes;
  return TDX_OK;
}

tdx_status tdx_moe_combine_plan_info(int W, int T, int F, int H, int E, int topk, tdx_dtype dtype,
                                     const tdx_opts* opts, int64_t* info) {
  if (info == nullptr) return TDX_ERR_INVALID_ARG;
  const tdx_opts o = opts ? *opts : defaults();
  MoePlan pl;
  tdx_status s = make_moe_plan(W, T, F, H, E, topk, dtype, o, &pl, true);
  if (s != TDX_OK) return s;
  const int64_t v[16] = {pl.BN, pl.tiles_n, pl.max_tiles, pl.n_chunks, pl.total, (int64_t)pl.off_flags,
                         (int64_t)pl.off_ntiles, (int64_t)pl.off_offsets, (int64_t)pl.off_src, (int64_t)pl.off_tiles,
                         (int64_t)pl.off_R, (int64_t)pl.bytes, pl.num_kb, (int64_t)pl.off_tokcnt,
                         (int64_t)pl.off_dest, pl.PM == 2 ? 3 : 1};
  std::memcpy(info, v, sizeof(v));
  return TDX_OK;
}

tdx_status tdx_moe_gemm_combine(const void* Hd, const int32_t* const* topk_idx, const void* B_experts,
                                const float* const* gates, void* const* out, void* workspace, size_t workspace_bytes,
                                int W, int T, int F, int H, int E, int topk, tdx_dtype dtype, const tdx_opts* opts,
                                void* stream) {
  const tdx_opts o = opts ? *opts : defaults();
  if (Hd == nullptr || topk_idx == nullptr || B_experts == nullptr || gates == nullptr || out == nullptr)
    return TDX_ERR_INVALID_ARG;
  if (W < 1 || W > kMaxW) return TDX_ERR_INVALID_ARG;
  for (int s = 0; s < W; ++s)
    if (topk_idx[s] == nullptr || gates[s] == nullptr || out[s] == nullptr) return TDX_ERR_INVALID_ARG;
  if (o.mode < TDX_FUSED || o.mode > TDX_CONSUMER_ONLY) return TDX_ERR_INVALID_ARG;
  if (o.mode == TDX_CONSUMER_ONLY || o.producer != TDX_PRODUCER_SM) return TDX_ERR_UNSUPPORTED;
  MoePlan pl;
  tdx_status s = make_moe_plan(W, T, F, H, E, topk, dtype, o, &pl, true);
  if (s != TDX_OK) return s;
  for (int r = 0; r < W; ++r)
    if (!aligned16(out[r]) || (reinterpret_cast<uintptr_t>(topk_idx[r]) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(gates[r]) & 3u) != 0)
      return TDX_ERR_ALIGNMENT;
  if (!aligned16(Hd) || !aligned16(B_experts)) return TDX_ERR_ALIGNMENT;
  if ((static_cast<long long>(F) * 2) % 16 != 0 || (static_cast<long long>(H) * 2) % 16 != 0) return TDX_ERR_ALIGNMENT;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < pl.bytes)
    return TDX_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (pl.total == 0 || H == 0) return TDX_OK;
  if (o.epoch == 0) {
    s = fill_zero(ws + pl.off_flags, pl.ctrl_end - pl.off_flags, st);
    if (s != TDX_OK) return s;
  }
  // 1. routing layout on the device (the same as the dispatch's)
  static thread_local MoeLayoutParams lq;
  std::memset(&lq, 0, sizeof(lq));
  for (int r = 0; r < W; ++r) lq.topk[r] = topk_idx[r];
  lq.dest = reinterpret_cast<int32_t*>(ws + pl.off_dest);
  lq.src = reinterpret_cast<int32_t*>(ws + pl.off_src);
  lq.offsets = reinterpret_cast<int32_t*>(ws + pl.off_offsets);
  lq.user_offsets = nullptr;
  lq.tiles = reinterpret_cast<int4*>(ws + pl.off_tiles);
  lq.ntiles = reinterpret_cast<int32_t*>(ws + pl.off_ntiles);
  lq.status = reinterpret_cast<uint32_t*>(ws);
  lq.W = W;
  lq.T = T;
  lq.k = topk;
  lq.E = E;
  lq.max_tiles = pl.max_tiles;
  lq.pair = pl.PM == 2 ? 1 : 0;
  if (launch_moe_layout(lq, st) != cudaSuccess) return TDX_ERR_CUDA;
  if (F == 0) {
    for (int r = 0; r < W; ++r) {
      s = fill_zero(out[r], static_cast<size_t>(T) * H * 2, st);
      if (s != TDX_OK) return s;
    }
    return TDX_OK;
  }
  // 2. fused grouped GEMM + combine
  static thread_local KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.op = OP_MOE_COMBINE;
  kp.mode = o.mode;
  kp.W = W;
  kp.M = static_cast<int>(pl.total);
  kp.K = F;
  kp.N = H;
  kp.M_local = kp.M;
  kp.tiles_m = pl.n_chunks;
  kp.tiles_n = pl.tiles_n;
  kp.T = pl.max_tiles;
  kp.group_n = pl.tiles_n;
  kp.rank_block = 1;
  kp.L = 1;
  kp.num_kb = pl.num_kb;
  kp.status = reinterpret_cast<uint32_t*>(ws);
  kp.trace = static_cast<uint32_t*>(o.trace);
  kp.epoch = o.epoch == 0 ? 1u : o.epoch;
  kp.dev_epoch = o.epoch == TDX_EPOCH_DEVICE ? reinterpret_cast<uint32_t*>(ws) + kDevEpochWord : nullptr;
  kp.timeout_ns = o.timeout_ns == 0 ? 2000000000ull : o.timeout_ns;
  kp.perturb = o.perturb_seed;
  kp.row_bytes = static_cast<long long>(F) * 2;
  kp.G = ws + pl.off_R;
  for (int r = 0; r < W; ++r) {
    kp.out[r] = static_cast<uint8_t*>(out[r]);
    kp.moe_gates[r] = gates[r];
  }
  kp.moe_src = lq.src;
  kp.moe_tiles = lq.tiles;
  kp.moe_ntiles = lq.ntiles;
  kp.moe_T = T;
  kp.moe_k = topk;
  kp.moe_dest = lq.dest;
  kp.moe_cnt = reinterpret_cast<uint32_t*>(ws + pl.off_tokcnt);
  kp.copy_active = 0;
  kp.wait_flags = 0;
  int grid = fused_max_grid_moe(true, pl.PM, device_sms(), false, pl.BN);
  if (grid <= 0) return TDX_ERR_CUDA;
  if (o.num_sms > 0 && o.num_sms < grid) grid = o.num_sms;
  grid -= grid % (pl.PM == 2 ? 2 : 1);
  if (grid <= 0) return TDX_ERR_INVALID_ARG;
  if (!make_map(&kp.tm_a[0], Hd, false, pl.total, F, 64, kBM) || !make_map_3d(&kp.tm_b[0], B_experts, E, F, H, 64, 64))
    return TDX_ERR_CUDA;
  const cudaError_t e = launch_fused_moe_combine_bf16(pl.BN, pl.PM, kp, grid, st);
  if (e != cudaSuccess) {
    if (std::getenv("TDX_VERBOSE")) std::fprintf(stderr, "tdx: launch failed: %s\n", cudaGetErrorString(e));
    return TDX_ERR_CUDA;
  }
  return TDX_OK;
}

tdx_status tdx_moe_dispatch_gemm(const void* const* X, const int32_t* const* topk_idx, const void* B_experts, void* Y,
                                 int32_t* dest, int32_t* expert_offsets, void* workspace, size_t workspace_bytes, int W,
                                 int T, int H, int F, int E, int topk, tdx_dtype dtype, const tdx_opts* opts,
                                 void* stream) {
  const tdx_opts o = opts ? *opts : defaults();
  if (X == nullptr || topk_idx == nullptr || B_experts == nullptr || Y == nullptr || dest == nullptr)
    return TDX_ERR_INVALID_ARG;
  if (W < 1 || W > kMaxW) return TDX_ERR_INVALID_ARG;
  for (int s = 0; s < W; ++s)
    if (X[s] == nullptr || topk_idx[s] == nullptr) return TDX_ERR_INVALID_ARG;
  if (o.mode < TDX_FUSED || o.mode > TDX_CONSUMER_ONLY) return TDX_ERR_INVALID_ARG;
  if (o.mode == TDX_CONSUMER_ONLY || o.producer != TDX_PRODUCER_SM) return TDX_ERR_UNSUPPORTED;
  MoePlan pl;
  tdx_status s = make_moe_plan(W, T, H, F, E, topk, dtype, o, &pl);
  if (s != TDX_OK) return s;
  for (int r = 0; r < W; ++r)
    if (!aligned16(X[r]) || (reinterpret_cast<uintptr_t>(topk_idx[r]) & 3u) != 0) return TDX_ERR_ALIGNMENT;
  if (!aligned16(B_experts) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(dest) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) != 0)
    return TDX_ERR_ALIGNMENT;
  if ((static_cast<long long>(H) * pl.elt) % 16 != 0 || (static_cast<long long>(F) * pl.elt) % 16 != 0 ||
      (static_cast<long long>(F) * 2) % 16 != 0)
    return TDX_ERR_ALIGNMENT;
  const bool fp8 = pl.elt == 1;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < pl.bytes)
    return TDX_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (pl.total == 0) {
    return expert_offsets != nullptr ? fill_zero(expert_offsets, static_cast<size_t>(E + 1) * 4, st) : TDX_OK;
  }
  const uint32_t epoch = o.epoch == 0 ? 1u : o.epoch;
  if (o.epoch == 0) {
    s = fill_zero(ws + pl.off_flags, pl.ctrl_end - pl.off_flags, st);
    if (s != TDX_OK) return s;
  }
  // 1. routing layout on the device
  static thread_local MoeLayoutParams lq;
  std::memset(&lq, 0, sizeof(lq));
  for (int r = 0; r < W; ++r) lq.topk[r] = topk_idx[r];
  lq.dest = dest;
  lq.src = reinterpret_cast<int32_t*>(ws + pl.off_src);
  lq.offsets = reinterpret_cast<int32_t*>(ws + pl.off_offsets);
  lq.user_offsets = expert_offsets;
  lq.tiles = reinterpret_cast<int4*>(ws + pl.off_tiles);
  lq.ntiles = reinterpret_cast<int32_t*>(ws + pl.off_ntiles);
  lq.status = reinterpret_cast<uint32_t*>(ws);
  lq.W = W;
  lq.T = T;
  lq.k = topk;
  lq.E = E;
  lq.max_tiles = pl.max_tiles;
  lq.pair = pl.PM == 2 ? 1 : 0;
  if (launch_moe_layout(lq, st) != cudaSuccess) return TDX_ERR_CUDA;
  if (F == 0) return TDX_OK;
  if (H == 0) return fill_zero(Y, static_cast<size_t>(pl.total) * F * 2, st);

  // 2. fused dispatch + grouped GEMM
  static thread_local KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.op = OP_MOE;
  kp.mode = o.mode;
  kp.W = W;
  kp.M = static_cast<int>(pl.total);
  kp.K = H;
  kp.N = F;
  kp.M_local = kp.M;
  kp.tiles_m = pl.n_chunks;
  kp.tiles_n = pl.tiles_n;
  kp.T = pl.max_tiles;
  kp.group_n = pl.tiles_n;
  kp.rank_block = 1;
  kp.L = 1;
  kp.num_kb = pl.num_kb;
  kp.status = reinterpret_cast<uint32_t*>(ws);
  kp.chunk_flags = reinterpret_cast<uint32_t*>(ws + pl.off_flags);
  kp.chunk_cnt = reinterpret_cast<uint32_t*>(ws + pl.off_cnt);
  kp.trace = static_cast<uint32_t*>(o.trace);
  kp.epoch = epoch;
  kp.dev_epoch = o.epoch == TDX_EPOCH_DEVICE ? reinterpret_cast<uint32_t*>(ws) + kDevEpochWord : nullptr;
  kp.timeout_ns = o.timeout_ns == 0 ? 2000000000ull : o.timeout_ns;
  kp.perturb = o.perturb_seed;
  kp.row_bytes = static_cast<long long>(H) * pl.elt;
  kp.chunk_rows = kBM;
  kp.n_chunks = pl.n_chunks;
  kp.trace_chunks = pl.n_chunks;
  kp.chunk_bytes = kBM * kp.row_bytes;
  kp.G = ws + pl.off_R;
  kp.out[0] = static_cast<uint8_t*>(Y);
  for (int r = 0; r < W; ++r) {
    kp.shard[r] = static_cast<const uint8_t*>(X[r]);
    kp.row_scale[r] = (fp8 && o.scale_a) ? o.scale_a[r] : 1.0f;
  }
  for (int e = 0; e < E; ++e) kp.moe_bscale[e] = (fp8 && o.scale_b) ? o.scale_b[e] : 1.0f;
  kp.moe_src = lq.src;
  kp.moe_tiles = lq.tiles;
  kp.moe_ntiles = lq.ntiles;
  kp.moe_T = T;
  int grid = fused_max_grid_moe(false, pl.PM, device_sms(), fp8, pl.BN);
  if (grid <= 0) return TDX_ERR_CUDA;
  if (o.num_sms > 0 && o.num_sms < grid) grid = o.num_sms;
  grid -= grid % (pl.PM == 2 ? 2 : 1);
  if (grid <= 0) return TDX_ERR_INVALID_ARG;
  // producer: a CTA copies a whole 128-row chunk and releases its flag; with fewer chunks than CTAs
  // a chunk is cut into ppc pieces (at most 16) so that every CTA moves rows
  {
    int ppc = (grid + pl.n_chunks - 1) / pl.n_chunks;
    if (ppc < 1) ppc = 1;
    if (ppc > 16) ppc = 16;
    kp.ppc = ppc;
    kp.moe_rpp = (kBM + ppc - 1) / ppc;
    kp.total_pieces = pl.n_chunks * ppc;
  }
  const bool moving = o.mode == TDX_FUSED || o.mode == TDX_MOVE_ONLY;
  kp.copy_active = moving ? 1 : 0;
  kp.wait_flags = o.mode == TDX_FUSED ? 1 : 0;
  // A: 128-byte K slices of 128 rows; B: 128-byte N rows, one K slice deep, one expert
  const int box = 128 / pl.elt;
  if (!make_map(&kp.tm_a[0], kp.G, fp8, pl.total, H, box, kBM) ||
      !make_map_3d(&kp.tm_b[0], B_experts, E, H, F, box, box, fp8))
    return TDX_ERR_CUDA;
  const cudaError_t e = fp8 ? launch_fused_moe_fp8(pl.BN, pl.PM, kp, grid, st)
                            : launch_fused_moe_bf16(pl.BN, pl.PM, kp, grid, st);
  if (e != cudaSuccess) {
    if (std::getenv("TDX_VERBOSE")) std::fprintf(stderr, "tdx: launch failed: %s\n", cudaGetErrorString(e));
    return TDX_ERR_CUDA;
  }
  return TDX_OK;
}

}  // extern "C"
