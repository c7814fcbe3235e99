// Internal definitions shared by the host planner (tdx_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tdx {

constexpr int kMaxW = 16;
constexpr int kBM = 128;                 // rows of every output tile (one TMEM lane per row)
constexpr int kNumThreads = 384;         // 12 warps, roles below
constexpr int kTmaWarp = 0;              // lane 0 issues TMA loads (and waits on chunk flags)
constexpr int kMmaWarp = 1;              // lane 0 issues tcgen05.mma; the warp owns TMEM
constexpr int kCopyWarp0 = 2;            // warps 2-3: AllGather chunk producer
constexpr int kNumCopyWarps = 2;
constexpr int kEpiWarp0 = 4;             // warps 4-11: epilogue (TMEM -> registers -> global)
constexpr int kNumEpiWarps = 8;
constexpr int kEpiThreads = kNumEpiWarps * 32;
constexpr int kCopyThreads = kNumCopyWarps * 32;
constexpr int kCopyRoundBytes = 16384;   // producer: bytes in flight per CTA per round
constexpr int kMaxPieceBytes = 65536;    // producer: largest copy unit released at once
// Largest library-chosen K split of a small AllGather: 19 lets the 8 tiles of the small-M shape
// (W=8, 16-row shards, N=1024) fill the 152 SMs of a GB300 in one wave (15.8 -> 15.5 us per call
// against 16 splits).
constexpr int kMaxSplitK = 19;
// RS raster: N-tiles per group (a rank's tiles are taken group by group, M-tiles, then the group's
// N-tiles), so that a wave reads few columns of B_r while A_r is streamed once per group. Step
// throughput on GB300 (W=8 AG + RS) by group size 4 / 8 / 16 / 32: 1516 / 1538 / 1561 / 1513
// TFLOP/s.
#ifndef TDX_RS_GROUP_N
#define TDX_RS_GROUP_N 16
#endif
constexpr int kRsGroupN = TDX_RS_GROUP_N;
// RS order: tiles per rank block (divided by the CTAs per cluster to count positions); a block is
// processed for every rank before the next, so a tile's running sum is re-read by the next rank
// about one block later. Default: one block of every tile (rank-outer order), which measured
// fastest on GB300 (operand reuse across a rank's waves outweighs keeping running sums in L2;
// blocks of 74/148/296 tiles were 1.5-3% slower).
#ifndef TDX_RS_RANK_BLOCK
#define TDX_RS_RANK_BLOCK (1 << 30)
#endif
constexpr int kRsRankBlock = TDX_RS_RANK_BLOCK;
// Slotted ReduceScatter order: rank-inner (1) or the rank-outer order of the chained mode (0).
// Rank-outer measured faster on GB300 for the small-M case (48.6 vs 57.9 us).
#ifndef TDX_SLOTTED_RANK_INNER
#define TDX_SLOTTED_RANK_INNER 0
#endif
constexpr bool kSlottedRankInner = TDX_SLOTTED_RANK_INNER != 0;
constexpr int kRefSMs = 148;             // fixed SM count used only for the (host) tiling choice

// K bytes per shared-memory ring slot (host and device agree on it). 128 for every tile width: a
// 64-byte slice doubles the ring depth in the same shared memory but measured slower on GB300
// (per-slot barrier/commit overhead and a 64-byte-swizzled A operand cost more than the depth buys).
constexpr int k_slice_bytes(int /*block_n*/) { return 128; }

// OP_MOE: AllToAll dispatch + grouped GEMM; OP_MOE_COMBINE: grouped GEMM + AllToAll combine
enum Op { OP_AG = 0, OP_RS = 1, OP_MOE = 3, OP_MOE_COMBINE = 4 };
constexpr int kOpAllReduce = 2;          // API op code: GEMM+AllReduce (runs the OP_RS kernel)
constexpr int kMoeMaxExperts = 512;      // layout kernel: per-expert tables live in shared memory
constexpr int kMoeMaxTopk = 16;          // combine: a token's slots are held in registers
enum Mode { MODE_FUSED = 0, MODE_GEMM_ONLY = 1, MODE_MOVE_ONLY = 2, MODE_CONSUMER_ONLY = 3 };
enum FailRole { ROLE_FLAG = 1, ROLE_PIPE = 2, ROLE_CHAIN = 3, ROLE_PRODUCER = 4, ROLE_LAYOUT = 5 };
enum DevStatus { DEV_OK = 0, DEV_BAD_INPUT = 1, DEV_TIMEOUT = 6, DEV_STALE = 7 };

// Word offsets in the workspace header (first 4 KiB): the status word and its details, then the
// device-kept epoch (the last completed call's epoch) and the count of this call's CTAs that have
// read it (reset by the CTA that completes the count).
constexpr size_t kHeaderBytes = 4096;
constexpr int kStatusWords = 8;
constexpr int kDevEpochWord = 16;
// Trace: statistics words per CTA (see tdx_trace_size in include/tdx.h).
constexpr int kTraceStatWords = 12;

struct KParams {
  CUtensorMap tm_a[kMaxW];       // AG: [0] gathered buffer G, [1] self shard (pull mode: shard r). RS: A_r
  CUtensorMap tm_b[kMaxW];       // AG: [0] B. RS: B_r
  const uint8_t* shard[kMaxW];   // AG producer sources
  uint8_t* out[kMaxW];           // AG: [0] = C. RS: output shards. AllReduce: every rank's M x N output
  uint8_t* G;                    // AG gathered buffer
  uint32_t* status;              // kStatusWords words
  uint32_t* chunk_flags;         // AG: [W * n_chunks], flag of chunk (rank, c) at rank*n_chunks + c
  uint32_t* chunk_cnt;           // AG: pieces completed per chunk (reset by the last piece)
  uint32_t* chain_flags;         // [(L-1) * T]: running sum of chain elements 0..c done for tile
  float* sbuf;                   // chained: [T][kBM*BN] running sum; slotted: [L][T][kBM*BN] partials
  uint32_t* tile_cnt;            // slotted: partials stored per tile (reset by the last arriver)
  uint32_t* tile_done;           // cooperative fold: elements that folded their share (reset by the last)
  uint32_t* grid_bar;            // grid-wide fold: [0] CTAs arrived, [1] CTAs departed (reset by the last)
  int coop_fold;                 // slotted fold: 0 the last arriver folds the tile, 1 the L elements
                                 // of a tile fold 1/L each after all arrived (one wave of work),
                                 // 2 every CTA folds 1/grid of all tiles after a grid barrier
  int reduce_last;               // 1 = slotted (last arriver folds), 0 = chained running sum
  uint32_t* trace;               // optional
  int trace_chunks;              // chunk flags this call releases (size of the trace's producer section)
  float row_scale[kMaxW];        // AG e4m3: scale_a[r] * scale_b for rows of rank r
  float elem_scale[kMaxW];       // RS e4m3: scale_a[r] * scale_b[r] for rank r's partial
  int op, mode;
  int W, M, K, N;                // M = total rows (AG: W * M_local)
  int M_local;                   // AG: rows per shard. RS: rows per output shard (M / W)
  int self_rank;
  int chunk_rows, n_chunks;      // AG chunking (per rank)
  int tiles_m, tiles_n, T;       // T = tiles_m * tiles_n
  int group_n;                   // RS raster: N-tiles per group (1..tiles_n)
  int rank_block;                // RS order: positions per rank block (1..tiles per rank in groups)
  int L;                         // chain length: RS = W ranks, AG = split-K factor
  int num_kb;                    // K blocks of 128 bytes
  int out_fp32;
  int copy_active;               // producer warps copy chunks (AG, SM producer, fused/move)
  int wait_flags;                // consumers wait on chunk flags (AG fused / consumer-only)
  int pull_a;                    // AG small shards: tiles read A from the shards (tm_a[r]), no waits
  int pull_3d;                   // pull_a with shards at one stride: tm_a[0] is a 3D map (K, row, rank)
                                 // and a tile's shards are one box
  int b_groups;                  // AG single CTAs, N whole 128-byte groups: tm_b[0] is a 3D map
                                 // (128-byte column, K, column group) and a K slice of B is one box
                                 // across the tile width
  int a_streamed, b_streamed;    // operand read by one tile only: loaded evict_first (else evict_last)
  int allreduce;                 // RS kernel as GEMM+AllReduce: out[r] are full M x N outputs
  int bf16_partials;             // slotted RS/AR: partials rounded to bf16 in their slots (else fp32)
  const int32_t* moe_src;        // MoE: source token of every dispatched row, s * moe_T + t
  const int4* moe_tiles;         // MoE: tile table {first row, end row of its expert, expert, 0}
  const int32_t* moe_ntiles;     // MoE: [0] tiles in the table, [1] nonzero if the routing was invalid
  int moe_T;                     // MoE: tokens per rank
  int moe_rpp;                   // MoE producer: dispatched rows per piece
  int moe_k;                     // MoE combine: slots per token
  const int32_t* moe_dest;       // MoE combine: W x T x k dispatched row of every token slot
  const float* moe_gates[kMaxW]; // MoE combine: [W] T x k gate weights
  uint32_t* moe_cnt;             // MoE combine: arrivals per (token, N-tile), reset by the last
  float moe_bscale[kMoeMaxExperts];   // MoE e4m3: per-expert weight scale (row_scale: per source rank)
  uint32_t epoch;                // this call's epoch (unused when dev_epoch is set)
  uint32_t* dev_epoch;           // device-kept epochs: [0] last completed call's epoch, [1] CTAs that read it
  uint64_t timeout_ns;
  uint32_t perturb;
  int piece_bytes;               // producer copy unit (multiple of kCopyRoundBytes)
  int ppc;                       // pieces per chunk
  int total_pieces;              // AG: phase-2 pieces (chunks copy_q1.. in release order)
  int copy_lo, copy_q1;          // AG: chunks 0..copy_q1-1 (release order) are copied first by CTAs
                                 // copy_lo.. through their operand ring (copy_q1 = 0: none)
  long long row_bytes;           // K * element size
  long long chunk_bytes;
};

// Shared-memory footprint of one instantiation (host side, for the launch).
int fused_smem_bytes(int block_n, bool fp8);

// Launch the persistent fused kernel for (op, block_n, pair mode pm) on `grid` CTAs. pm: 0 single
// CTAs, 2 CTA pairs running one 2-SM MMA stream.
cudaError_t launch_fused_bf16(int op, int block_n, int pm, const KParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fused_fp8(int op, int block_n, int pm, const KParams& p, int grid, cudaStream_t stream);
// Largest grid whose CTAs are resident together (pairs: twice the 2-CTA clusters that fit).
int fused_max_grid_bf16(int op, int pm, int sms, int block_n);
int fused_max_grid_fp8(int op, int pm, int sms, int block_n);
cudaError_t launch_fill_zero(void* dst, size_t bytes, cudaStream_t stream);

// MoE: the fused dispatch + grouped GEMM kernel and the fused grouped GEMM + combine kernel
// (bf16, single CTAs).
// pm: 0 single CTAs, 2 2-SM pairs (tile width 256).
cudaError_t launch_fused_moe_bf16(int block_n, int pm, const KParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fused_moe_combine_bf16(int block_n, int pm, const KParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fused_moe_fp8(int block_n, int pm, const KParams& p, int grid, cudaStream_t stream);
int fused_max_grid_moe(bool combine, int pm, int sms, bool fp8, int block_n);

// MoE routing layout: from every rank's top-k expert ids, the dispatched row of every (rank, token,
// slot), the source of every dispatched row, the expert row offsets and the GEMM tile table.
struct MoeLayoutParams {
  const int32_t* topk[kMaxW];    // [W] T x k expert ids
  int32_t* dest;                 // W x T x k dispatched rows (output)
  int32_t* src;                  // total rows: s * T + t (output)
  int32_t* offsets;              // E + 1 expert row offsets (output)
  int32_t* user_offsets;         // optional copy of offsets for the caller (may be null)
  int4* tiles;                   // tile table (output)
  int32_t* ntiles;               // [0] tiles, [1] invalid routing (output)
  uint32_t* status;              // workspace status words
  int W, T, k, E, max_tiles;
  int pair;                      // pad every expert's tile count to even (CTA pairs)
};
cudaError_t launch_moe_layout(const MoeLayoutParams& q, cudaStream_t stream);

}  // namespace tdx
