// The persistent fused kernel: AllGather chunk producer + flag-gated tcgen05/TMEM GEMM, GEMM +
// rank-ordered ReduceScatter / AllReduce, and the mixture-of-experts AllToAll dispatch + grouped
// GEMM and grouped GEMM + combine, in one launch per call.
//
// Roles (one CTA per SM, 12 warps):
//   warp 0  lane 0  TMA issuer. For an AllGather (or MoE dispatch) tile it first acquire-waits the
//                   flags of every chunk the tile's rows fall in (unless the rows are the local
//                   shard), then streams 128-byte K slices of A and B into an S-stage ring.
//   warp 1  lane 0  MMA issuer: tcgen05.mma (bf16: kind::f16, e4m3: kind::f8f6f4) into one of two
//                   TMEM accumulators of 128 x BN fp32; tcgen05.commit frees ring slots and
//                   hands finished accumulators to the epilogue. Warp 1 allocates TMEM.
//   warps 2-3       producer: one thread moves shard chunks (AllGather) or gathered token rows
//                   (MoE dispatch) into the gathered / receive buffer with TMA bulk copies through
//                   a shared-memory staging ring (AllGather, first wave's chunks: through the
//                   operand ring of a CTA waiting for them); the copy that completes a chunk
//                   releases the chunk's flag (= epoch).
//   warps 4-11      epilogue: TMEM -> registers; either the output tile (rounded once) or, along
//                   a chain (RS ranks or AG K-splits) of L elements, the fixed-order fp32 sum
//                   ((P_0 + P_1) + P_2) + ... of the elements' partial tiles, in one of two ways:
//                   "chained": element c acquires flag (c-1, tile), adds its partial to the
//                   running sum of elements 0..c-1, stores it and releases flag (c, tile); the
//                   last element rounds and stores the output (large problems: the elements of a
//                   tile run far apart in time, one running-sum buffer). "slotted": every element
//                   stores its partial in its own slot and bumps the tile's arrival counter; the
//                   element that completes the count folds the slots in order 0..L-1, or, when
//                   all the work fits one wave, every element folds 1/L of the tile once all L
//                   arrived (small problems: the elements of a tile run concurrently). Either way
//                   the order is fixed, so results are bit-identical run to run. For the MoE
//                   combine the epilogue also counts each token's stored expert-output rows and
//                   folds the tokens it completes with their gates.
//
// The chunk/flag pipeline follows the Triton-distributed article (cronfeed.work), section "The
// first move was to expose the overlap" (chunks, compute on arrived chunks while others move,
// communication and computation blocks coordinated in one kernel through symmetric memory and
// signals) and section "DITRON adds three levels of tiling" (core-level tiles on tensor cores and
// TMA; collectives split into chunks paired with compute tiles, with synchronisation inserted).
//
// Every wait is bounded by p.timeout_ns (%globaltimer); a wait that runs out records an error in
// the workspace status word and sets a CTA-wide abort flag; all roles then stop issuing work, the
// MMA issuer waits for its in-flight MMAs, the TMA issuer for its in-flight loads, TMEM is freed and
// the kernel returns. Nothing traps.
#pragma once

#include <atomic>
#include <cuda_bf16.h>

#include "tdx_internal.h"
#include "tdx_ptx.cuh"

namespace tdx {

// Upper bound of the shared-memory ring depth (the budget below usually binds first); a build may
// lower it with -DTDX_MAX_STAGES=n to study how latency hiding scales with depth.
#ifndef TDX_MAX_STAGES
#define TDX_MAX_STAGES 12
#endif
// The TMA issuer prefetches into L2 the K slice this many slices ahead of the one it loads (0 = no
// prefetch), so that slices missing in L2 are on their way before their ring slot frees up.
#ifndef TDX_PREFETCH_AHEAD
#define TDX_PREFETCH_AHEAD 0
#endif
// L2 eviction policy of operand tile loads and of running-sum / output traffic: 0 = evict_first,
// 1 = evict_last, 2 = evict_normal.
#ifndef TDX_OPERAND_POLICY
#define TDX_OPERAND_POLICY 1
#endif
#ifndef TDX_SUM_POLICY
#define TDX_SUM_POLICY 0
#endif
// MoE dispatch producer: rows of the chunk ahead of the bulk copies that the producer threads
// prefetch into L2 (0 = none). Off: 16 and 48 rows ahead measured 3-5% slower on GB300 (the bulk
// loads already keep three segments in flight per SM).
#ifndef TDX_MOE_PREFETCH_ROWS
#define TDX_MOE_PREFETCH_ROWS 0
#endif
// Drop dead running-sum / partial-slot lines from L2 after their last read (1) or leave them (0).
// Measured neutral on GB300, so off: the workspace then keeps the last call's sums and partials.
#ifndef TDX_DISCARD_DEAD
#define TDX_DISCARD_DEAD 0
#endif

// MoE dispatch bulk copies: L2 policy of the token-row loads and of the receive-buffer stores
// (-1 = no hint, else as TDX_OPERAND_POLICY: 0 evict_first, 1 evict_last, 2 evict_normal). Token
// rows evict-first (each is re-read only by its other slots, far apart) and receive-buffer rows
// evict-last (the GEMM reads them next): fused dispatch + GEMM 5.54 -> 5.33 ms on GB300.
#ifndef TDX_MOE_LOAD_POLICY
#define TDX_MOE_LOAD_POLICY 0
#endif
#ifndef TDX_MOE_STORE_POLICY
#define TDX_MOE_STORE_POLICY 1
#endif
// MoE combine: L2 policy of the expert-output stores (read back by the combine): as above.
#ifndef TDX_COMBINE_Z_POLICY
#define TDX_COMBINE_Z_POLICY 1
#endif
// AllGather bulk producer: L2 policy of the gathered-buffer stores (as TDX_OPERAND_POLICY).
#ifndef TDX_AG_STORE_POLICY
#define TDX_AG_STORE_POLICY 1
#endif
// Largest MoE dispatch staging ring (KiB).
#ifndef TDX_MOE_STG_MAX_KB
#define TDX_MOE_STG_MAX_KB 32
#endif
// Grid-wide fold: float4 per slot a task loads (2: 8 columns; 4: 16 columns, which spilled
// registers and measured slower on the small-M ReduceScatter, 34.9 -> 36.3 us).
#ifndef TDX_GRID_FOLD_F4
#define TDX_GRID_FOLD_F4 2
#endif
// Programmatic dependent launch of the fused kernels (1 = on).
#ifndef TDX_PDL
#define TDX_PDL 1
#endif
// AllGather: GEMM ring budget and largest bulk-copy staging ring (KiB). 168 / 80 (three 2-SM pair
// stages of a 512-column tile, a 2.5x staging ring) copied faster alone (0.108 -> 0.089 ms) but
// slowed the GEMM, e4m3 most (fused 0.683 -> 0.731 ms).
#ifndef TDX_AG_RING_KB
#define TDX_AG_RING_KB 216
#endif
#ifndef TDX_AG_STG_MAX_KB
#define TDX_AG_STG_MAX_KB 32
#endif

// PAIR_MMA: the CTA is one half of a 2-SM MMA pair (tcgen05 cta_group::2). The pair computes a
// 256 x BN tile with one instruction stream issued by the leader; each CTA stages its own 128 rows
// of A and its half (BN/2 columns) of the B slice, and holds its 128 x BN accumulator in TMEM.
template <int BN, bool FP8, bool PAIR_MMA = false, int RING_KB = 216, int STG_MAX_KB = TDX_MOE_STG_MAX_KB>
struct Cfg {
  static constexpr int ELT = FP8 ? 1 : 2;
  // K bytes per ring slot (k_slice_bytes): A rows in a slot are KB bytes long; B keeps 128-byte MN
  // rows with KB/ELT K rows per box.
  static constexpr int KB = k_slice_bytes(BN);
  static constexpr int BK = KB / ELT;             // K elements per ring slot
  static constexpr int UMMA_K = 32 / ELT;         // K per tcgen05.mma (32 bytes)
  static constexpr int K_STEPS = BK / UMMA_K;     // 2 or 4
  static constexpr int A_BYTES = kBM * KB;        // 8 or 16 KiB
  static constexpr uint32_t A_SBO = 8 * KB;       // next group of 8 rows
  static constexpr uint32_t A_LAYOUT = KB == 128 ? 2u : 4u;   // descriptor swizzle: 128 B or 64 B
  static constexpr int B_BOX_N = 128 / ELT;       // N elements per B box (128 bytes)
  static constexpr int B_BOXES = BN / B_BOX_N;              // boxes across the tile width
  static constexpr int B_BOXES_CTA = PAIR_MMA ? B_BOXES / 2 : B_BOXES;   // boxes this CTA stages
  static constexpr int B_BOX_BYTES = BK * 128;
  // A tile wider than one MMA (512 columns, 2-SM pairs only) takes N_PARTS MMAs of MMA_N columns per
  // K step, part p on accumulator columns [p*MMA_N, (p+1)*MMA_N); this CTA's B boxes are stored part
  // by part (each part: its half of the part's columns in a pair)
  static constexpr int MMA_N = BN > 256 ? 256 : BN;
  static constexpr int N_PARTS = BN / MMA_N;
  static constexpr int BOXES_PART = MMA_N / B_BOX_N;
  static constexpr int BOXES_PART_CTA = PAIR_MMA ? BOXES_PART / 2 : BOXES_PART;
  static constexpr int B_PART_BYTES = BOXES_PART_CTA * B_BOX_BYTES;
  static constexpr int B_BYTES = B_BOXES_CTA * B_BOX_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_RAW = (RING_KB * 1024) / STAGE_BYTES;   // ring budget (216 KiB by default)
  static constexpr int STAGES = STAGES_RAW > TDX_MAX_STAGES ? TDX_MAX_STAGES : STAGES_RAW;
  // two accumulators (the epilogue drains one while the MMA fills the other) up to 256 columns;
  // a 512-column tile fills Tensor Memory with one accumulator
  static constexpr int ACC_BUFS = 2 * BN <= 512 ? 2 : 1;
  static constexpr int TMEM_COLS = (ACC_BUFS * BN < 32) ? 32 : ACC_BUFS * BN;   // 128 / 256 / 512
  static constexpr int NUM_BARS = 2 * STAGES + 5;   // ring full/empty, accumulators full/empty, drain
  // flags/decisions (64 B), MoE producer row sources (kBM ints) and staging barriers (8)
  static constexpr int MISC_BYTES = 64 + kBM * 4 + 8 * 8;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + MISC_BYTES;
  // staging ring for bulk copies (MoE dispatch, AllGather producer): what the GEMM ring leaves of
  // the 227 KiB, at most STG_MAX_KB, in whole KiB (at least 4 KiB)
  static constexpr int MOE_STG_RAW = 227 * 1024 - SMEM_BYTES - 128;
  static constexpr int MOE_STG = (MOE_STG_RAW > STG_MAX_KB * 1024 ? STG_MAX_KB * 1024 : MOE_STG_RAW) / 1024 * 1024;
  static constexpr int COLS_PER_WARP = BN / 2;    // 8 epilogue warps = 4 lane quarters x 2 halves
  static constexpr int CHUNKS = COLS_PER_WARP / 32;
  // Instruction descriptor: D fp32 (bits 4-5 = 1), A/B type (bits 7-9, 10-12: bf16 = 1,
  // e4m3 = 0), A K-major (bit 15 = 0), B MN-major (bit 16 = 1), N >> 3 (bits 17-22),
  // M >> 4 (bits 24-28).
  static constexpr int MMA_M = PAIR_MMA ? 2 * kBM : kBM;
  static constexpr uint32_t IDESC = (1u << 4) | ((FP8 ? 0u : 1u) << 7) | ((FP8 ? 0u : 1u) << 10) |
                                    (1u << 16) | (static_cast<uint32_t>(MMA_N >> 3) << 17) |
                                    (static_cast<uint32_t>(MMA_M >> 4) << 24);
  static_assert(BN % B_BOX_N == 0 && B_BOXES >= 1, "tile width must cover whole 128-byte boxes");
  static_assert(!PAIR_MMA || B_BOXES % 2 == 0, "a 2-SM pair splits B into two halves");
  static_assert(BN <= 256 || PAIR_MMA, "512-column tiles run on 2-SM pairs");
  static_assert(BN <= 512 && BN % MMA_N == 0 && (!PAIR_MMA || BOXES_PART % 2 == 0), "tile parts");
  static_assert(CHUNKS >= 1, "at least one 32-column chunk per epilogue warp");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// GEMM ring budget per op: the MoE dispatch may give part of it to its staging ring.
#ifndef TDX_MOE_RING_KB
#define TDX_MOE_RING_KB 216
#endif
constexpr int ring_kb(int op) { return op == OP_MOE ? TDX_MOE_RING_KB : op == OP_AG ? TDX_AG_RING_KB : 216; }
constexpr int stg_kb(int op) { return op == OP_AG ? TDX_AG_STG_MAX_KB : TDX_MOE_STG_MAX_KB; }
// Ops whose producer moves data with bulk copies through a shared-memory staging ring.
constexpr bool uses_staging(int op) { return op == OP_MOE || op == OP_AG; }



struct Item {
  int c;      // chain element (RS rank, or AG K split)
  int tile;   // tile id = mt * tiles_n + nt (MoE: the item index)
  int m0, n0;
  int mend;   // MoE: end row of the tile's expert (rows >= mend are not stored)
  int e;      // MoE: expert
};

// Work item `it` of a CTA whose rank in its cluster is `crank`. With CL CTAs per cluster, items
// index (chain element, group of CL consecutive M-tiles, N-tile) and the CTA of cluster rank r takes
// M-tile CL*group + r (the host keeps tiles_m a multiple of CL). AllGather groups are taken in the
// rank-swizzled arrival order: from the first group whose first row belongs to self_rank,
// wrapping around; N-tiles innermost.
template <int OP, int CL>
__device__ __forceinline__ Item decode_item(const KParams& p, int it, int BN, int crank) {
  Item r;
  if constexpr (OP == OP_MOE || OP == OP_MOE_COMBINE) {
    // MoE: the tile table lists each expert's 128-row tiles in dispatched-row order (experts
    // ascending), which is the order the producers fill the receive buffer in; N-tiles innermost.
    // With CTA pairs an item is a pair of consecutive tiles of one expert (the table pads every
    // expert to an even count) and the CTA of cluster rank r takes tile 2*pair + r.
    const int tp = it / p.tiles_n;
    const int4 ti = p.moe_tiles[tp * CL + crank];
    r.c = 0;
    r.tile = it;
    r.m0 = ti.x;
    r.mend = ti.y;
    r.e = ti.z;
    r.n0 = (it - tp * p.tiles_n) * BN;
    return r;
  }
  r.mend = 0;
  r.e = 0;
  const int tiles_g = p.tiles_m / CL;
  const int Tg = tiles_g * p.tiles_n;
  int pos;
  if constexpr (OP == OP_AG) {
    r.c = it / Tg;
    pos = it - r.c * Tg;
  } else {
    // ReduceScatter, rank-blocked: positions of a rank's tile order are taken in blocks of
    // rank_block; a block is done for ranks 0..L-1 before the next block starts, so the running sum
    // of a tile is handed to the next rank about one block (two waves) later, while it is in L2
    const int P = p.rank_block;
    const int nfull = Tg / P;
    const int full_items = nfull * p.L * P;
    if (it < full_items) {
      const int b = it / (p.L * P);
      const int rem = it - b * p.L * P;
      r.c = rem / P;
      pos = b * P + (rem - r.c * P);
    } else {
      const int Pl = Tg - nfull * P;
      const int rem = it - full_items;
      r.c = rem / Pl;
      pos = nfull * P + (rem - r.c * Pl);
    }
  }
  int mg, nt;
  if constexpr (OP == OP_AG) {
    int start = (p.self_rank * p.M_local + CL * kBM - 1) / (CL * kBM);
    if (start >= tiles_g) start = 0;
    mg = start + pos / p.tiles_n;
    if (mg >= tiles_g) mg -= tiles_g;
    nt = pos % p.tiles_n;
  } else {
    // ReduceScatter: within a rank, N-tiles in groups of group_n (the last group may be narrower);
    // group-outer, M groups, N-tiles of the group innermost, so that a wave of tiles touches few
    // rows of A_r and few columns of B_r
    const int gn = p.group_n;
    const int full = p.tiles_n / gn;
    const int per_group = tiles_g * gn;
    if (pos < full * per_group) {
      const int ng = pos / per_group;
      const int q = pos - ng * per_group;
      mg = q / gn;
      nt = ng * gn + (q - mg * gn);
    } else {
      const int rem = p.tiles_n - full * gn;
      const int q = pos - full * per_group;
      mg = q / rem;
      nt = full * gn + (q - mg * rem);
    }
  }
  const int mt = mg * CL + crank;
  r.tile = mt * p.tiles_n + nt;
  r.m0 = mt * kBM;
  r.n0 = nt * BN;
  return r;
}

// K blocks of one work item: an AllGather K split c covers [c*num_kb/L, (c+1)*num_kb/L); a
// ReduceScatter item (chain element = rank) covers all of K. The host keeps L <= num_kb, so every
// range is non-empty and the accumulator is always initialised.
template <int OP>
__device__ __forceinline__ void k_range(const KParams& p, const Item& w, int& kb0, int& kb1) {
  if constexpr (OP == OP_AG) {
    kb0 = static_cast<int>((static_cast<long long>(w.c) * p.num_kb) / p.L);
    kb1 = static_cast<int>((static_cast<long long>(w.c + 1) * p.num_kb) / p.L);
  } else {
    kb0 = 0;
    kb1 = p.num_kb;
  }
}

__device__ __forceinline__ void report_error(const KParams& p, uint32_t code, uint32_t role,
                                             uint32_t idx, uint32_t seen, uint32_t want) {
  if (atomicCAS(&p.status[0], 0u, code) == 0u) {
    p.status[1] = role;
    p.status[2] = blockIdx.x;
    p.status[3] = idx;
    p.status[4] = seen;
    p.status[5] = want;
    __threadfence();
  }
}

__device__ __forceinline__ uint32_t perturb_hash(uint32_t seed, uint32_t x) {
  uint32_t h = seed ^ (x * 0x9E3779B9u);
  h ^= h >> 16;
  h *= 0x7FEB352Du;
  h ^= h >> 15;
  return h;
}

// Producer trace: the k-th chunk flag released by this call (by any CTA) is recorded as its flag
// index in word 1 + k of the trace's producer section; word 0 of the section counts the releases and
// must be zero when the call starts.
__device__ __forceinline__ void trace_release(const KParams& p, int grid, uint32_t fi) {
  uint32_t* rel = p.trace + 4 + kTraceStatWords * grid;
  const uint32_t k = atomicAdd(rel, 1u);
  if (k < static_cast<uint32_t>(p.trace_chunks)) rel[1 + k] = fi;
}

// Bounded wait on an mbarrier phase. Gives up (false) when the CTA abort flag is raised or after
// 2 * p.timeout_ns; a timeout is recorded as DEV_TIMEOUT / ROLE_PIPE. Pipeline stages only wait on
// one another, so a stuck pipeline is normally caused by a flag wait upstream; the doubled bound
// lets that flag wait run out (and report itself) first.
static __device__ __noinline__ bool wait_mbar(const KParams& p, uint32_t bar, uint32_t parity,
                                       volatile int* abort_flag, uint32_t idx) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > 2 * p.timeout_ns) {
        report_error(p, DEV_TIMEOUT, ROLE_PIPE, idx, 0, parity);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Wait used while tearing down: ignores the abort flag, bounded by the timeout only.
static __device__ __noinline__ bool wait_mbar_drain(const KParams& p, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > p.timeout_ns) {
      report_error(p, DEV_TIMEOUT, ROLE_PIPE, 0xFFFFu, 0, parity);
      return false;
    }
  }
}

// Count `units` 16-byte units of AllGather chunk fi as copied (their stores completed and ordered
// before this); the copy that completes the chunk resets the count and releases the chunk's flag.
__device__ __forceinline__ void ag_chunk_done(const KParams& p, int fi, uint32_t units, uint32_t epoch, int grid) {
  __threadfence();
  const uint32_t total = static_cast<uint32_t>(p.chunk_bytes / 16);
  const uint32_t old = atomicAdd(p.chunk_cnt + fi, units);
  if (old + units == total) {
    p.chunk_cnt[fi] = 0u;
    const uint32_t prev = ld_relaxed_gpu(p.chunk_flags + fi);
    if (prev >= epoch) report_error(p, DEV_STALE, ROLE_PRODUCER, fi, prev, epoch);
    __threadfence();
    st_release_gpu(p.chunk_flags + fi, epoch);
    if (p.trace != nullptr) trace_release(p, grid, static_cast<uint32_t>(fi));
  }
}

// Copy `n` bytes (16-byte aligned addresses, n a multiple of 16) from src to dst with bulk copies
// through a staging ring: segments of `seg` bytes in `nb` (<= 8) ring buffers, nb - 1 loads in
// flight, each segment stored back as soon as it lands; returns once every store has completed and
// is ordered before later generic accesses. `g` rotates the buffers; bit b of `par` is the phase
// parity the next wait on barrier b expects (so that rings of different shapes may share the
// barriers). One thread.
static __device__ __noinline__ void bulk_copy_contig(const KParams& p, uint8_t* stg, uint64_t* bars, uint32_t seg, int nb,
                                                     uint32_t& g, uint32_t& par, const uint8_t* src, uint8_t* dst,
                                                     uint32_t n, uint64_t lpol, uint64_t spol) {
  const int nseg = static_cast<int>((n + seg - 1) / seg);
  auto issue = [&](int i) {
    const uint32_t off = static_cast<uint32_t>(i) * seg;
    const uint32_t m = n - off < seg ? n - off : seg;
    const uint32_t b = (g + static_cast<uint32_t>(i)) % static_cast<uint32_t>(nb);
    const uint32_t bar = smem_u32(bars + b);
    mbar_arrive_expect_tx(bar, m);
    bulk_load_g2s_hint(smem_u32(stg + b * seg), src + off, m, bar, lpol);
  };
  for (int i = 0; i < min(nb - 1, nseg); ++i) issue(i);
  for (int i = 0; i < nseg; ++i) {
    const int j = i + nb - 1;
    if (j < nseg) {
      bulk_wait_read_all();
      issue(j);
    }
    const uint32_t gi = g + static_cast<uint32_t>(i);
    const uint32_t b = gi % static_cast<uint32_t>(nb);
    wait_mbar_drain(p, smem_u32(bars + b), (par >> b) & 1u);
    par ^= 1u << b;
    const uint32_t off = static_cast<uint32_t>(i) * seg;
    const uint32_t m = n - off < seg ? n - off : seg;
    bulk_store_s2g_hint(dst + off, smem_u32(stg + b * seg), m, spol);
    bulk_commit();
  }
  g += static_cast<uint32_t>(nseg);
  bulk_wait_all();
  fence_proxy_async_global();
}

// One K slice of B for a single CTA's tile at column n0: the tile's 128-byte column boxes land one
// after another in shared memory. With `groups`, the map is 3D (128-byte column, K row, column
// group of 128 bytes) and one box covers every column group of the tile; else one 2D box per group.
template <class C>
static __device__ __forceinline__ void load_b_slice(uint8_t* dst, const CUtensorMap* map, uint32_t bar, int n0,
                                                    int kb, int groups, uint64_t pol) {
  if (groups) {
    tma_load_3d_hint(smem_u32(dst), map, bar, 0, kb * C::BK, n0 / C::B_BOX_N, pol);
    return;
  }
#pragma unroll
  for (int j = 0; j < C::B_BOXES; ++j)
    tma_load_2d_hint(smem_u32(dst + j * C::B_BOX_BYTES), map, bar, n0 + j * C::B_BOX_N, kb * C::BK, pol);
}

// Bounded wait until a shared-memory word set by another warp of the CTA is nonzero. Gives up
// (false) when the CTA abort flag is raised or after 2 * p.timeout_ns (recorded as DEV_TIMEOUT /
// ROLE_PIPE with index idx).
static __device__ __noinline__ bool wait_smem_flag(const KParams& p, const uint32_t* flag, volatile int* abort_flag,
                                                   uint32_t idx) {
  const volatile uint32_t* f = flag;
  if (*f != 0u) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (*f != 0u) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > 2 * p.timeout_ns) {
        report_error(p, DEV_TIMEOUT, ROLE_PIPE, idx, 0, 1);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded acquire-wait until *flag == epoch. A value above the epoch is a stale flag. Also gives
// up when any CTA has already recorded an error (status word != 0) or this CTA aborted.
static __device__ __noinline__ bool wait_flag(const KParams& p, uint32_t epoch, const uint32_t* flag, uint32_t role,
                                       uint32_t idx, volatile int* abort_flag, uint64_t* waited_ns) {
  uint32_t v = ld_acquire_gpu(flag);
  if (v == epoch) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (v > epoch) {
      report_error(p, DEV_STALE, role, idx, v, epoch);
      *abort_flag = 1;
      return false;
    }
    __nanosleep(32);
    v = ld_acquire_gpu(flag);
    if (v == epoch) {
      *waited_ns += globaltimer_ns() - t0;
      return true;
    }
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (ld_relaxed_gpu(p.status) != 0u) {
        *abort_flag = 1;
        return false;
      }
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        report_error(p, DEV_TIMEOUT, role, idx, v, epoch);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait until every chunk flag gc0..gc1 equals the epoch. The flags are polled with
// independent relaxed loads (one round trip for all of them, not one per flag), then a single
// acquire fence orders the data reads after them. Stale values and timeouts are reported like
// wait_flag's, for the first chunk not yet released.
static __device__ __noinline__ bool wait_flags_all(const KParams& p, uint32_t epoch, int gc0, int gc1,
                                                   volatile int* abort_flag, uint64_t* waited_ns) {
  constexpr int kBatch = 16;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    int pending = -1;
    uint32_t seen = 0;
    for (int b = gc0; b <= gc1 && pending < 0; b += kBatch) {
      uint32_t v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) v[j] = (b + j <= gc1) ? ld_relaxed_gpu(p.chunk_flags + b + j) : epoch;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (v[j] > epoch) {
          report_error(p, DEV_STALE, ROLE_FLAG, b + j, v[j], epoch);
          *abort_flag = 1;
          return false;
        }
        if (pending < 0 && v[j] != epoch) {
          pending = b + j;
          seen = v[j];
        }
      }
    }
    if (pending < 0) {
      fence_acq_rel_gpu();
      if (it > 0) *waited_ns += globaltimer_ns() - t0;
      return true;
    }
    if (it == 0) t0 = globaltimer_ns();
    __nanosleep(32);
    if ((it & 15u) == 15u) {
      if (*abort_flag) return false;
      if (ld_relaxed_gpu(p.status) != 0u) {
        *abort_flag = 1;
        return false;
      }
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        report_error(p, DEV_TIMEOUT, ROLE_FLAG, pending, seen, epoch);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// 32 fp32 values -> 32 bf16 (round to nearest even) packed in four 16-byte words.
__device__ __forceinline__ void pack_bf16x32(const float (&v)[32], uint4 (&pk)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 b0 = __floats2bfloat162_rn(v[8 * j + 0], v[8 * j + 1]);
    __nv_bfloat162 b1 = __floats2bfloat162_rn(v[8 * j + 2], v[8 * j + 3]);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * j + 4], v[8 * j + 5]);
    __nv_bfloat162 b3 = __floats2bfloat162_rn(v[8 * j + 6], v[8 * j + 7]);
    pk[j].x = *reinterpret_cast<uint32_t*>(&b0);
    pk[j].y = *reinterpret_cast<uint32_t*>(&b1);
    pk[j].z = *reinterpret_cast<uint32_t*>(&b2);
    pk[j].w = *reinterpret_cast<uint32_t*>(&b3);
  }
}

// 8 bf16 in a 16-byte word -> 8 fp32 (exact)
__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xFFFF0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xFFFF0000u);
  f[4] = __uint_as_float(u.z << 16);
  f[5] = __uint_as_float(u.z & 0xFFFF0000u);
  f[6] = __uint_as_float(u.w << 16);
  f[7] = __uint_as_float(u.w & 0xFFFF0000u);
}

// Store 32 fp32 values (columns col..col+31 of one row starting at orow) rounded once to the
// output type; columns >= N are skipped.
__device__ __forceinline__ void store_row_chunk(uint8_t* orow, const KParams& p, int col, const float (&v)[32],
                                                uint64_t pol) {
  if (p.out_fp32) {
    float* o = reinterpret_cast<float*>(orow) + col;
    if (col + 32 <= p.N) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_f4_hint(o + 4 * j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]), pol);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col + i < p.N) o[i] = v[i];
    }
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(orow) + col;
    if (col + 32 <= p.N) {
      uint4 pk[4];
      pack_bf16x32(v, pk);
#pragma unroll
      for (int j = 0; j < 4; ++j) st_v4_hint(o + 8 * j, pk[j], pol);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col + i < p.N) o[i] = __float2bfloat16_rn(v[i]);
    }
  }
}

// Round 32 consecutive fp32 values of one output row (columns col..col+31) once to the output type
// and store them: AllGather -> C (bf16 or fp32, e4m3 inputs scaled by scale_a[rank]*scale_b);
// ReduceScatter -> output shard row / (M/W); AllReduce -> row of every rank's full output (bf16).
// Rows >= M and columns >= N are skipped.
template <int OP, bool FP8>
__device__ __forceinline__ void store_out_chunk(const KParams& p, int row, int col, float (&v)[32], uint64_t pol) {
  if (row >= p.M) return;
  uint8_t* orow;
  if constexpr (OP == OP_AG) {
    if constexpr (FP8) {
      const float s = p.row_scale[row / p.M_local];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= s;
    }
    orow = p.out[0] + (size_t)row * p.N * (p.out_fp32 ? 4 : 2);
  } else if (p.allreduce) {
    // AllReduce: the reduced tile, rounded once, goes to every rank's full output (the fused
    // AllGather of the reduced shards)
    if (col + 32 <= p.N) {
      uint4 pk[4];
      pack_bf16x32(v, pk);
      for (int r = 0; r < p.W; ++r) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out[r] + (size_t)row * p.N * 2) + col;
#pragma unroll
        for (int j = 0; j < 4; ++j) st_v4_hint(o + 8 * j, pk[j], pol);
      }
      return;
    }
    for (int r = 1; r < p.W; ++r) store_row_chunk(p.out[r] + (size_t)row * p.N * 2, p, col, v, pol);
    orow = p.out[0] + (size_t)row * p.N * 2;
  } else if constexpr (OP == OP_MOE) {
    orow = p.out[0] + (size_t)row * p.N * 2;    // rows past the tile's expert arrive as row >= M
  } else if constexpr (OP == OP_MOE_COMBINE) {
    orow = p.G + (size_t)row * p.N * 2;         // expert outputs, dispatched order (bf16)
  } else {
    const int j = row / p.M_local;
    orow = p.out[j] + (size_t)(row - j * p.M_local) * p.N * 2;
  }
  store_row_chunk(orow, p, col, v, pol);
}

// Bounded acquire-wait until *ctr >= target (cooperative fold: all L partials of a tile stored).
static __device__ __noinline__ bool wait_count(const KParams& p, const uint32_t* ctr, uint32_t target,
                                               volatile int* abort_flag, uint32_t idx) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    __nanosleep(64);
    if ((it & 15u) == 15u) {
      if (*abort_flag) return false;
      if (ld_relaxed_gpu(p.status) != 0u) {
        *abort_flag = 1;
        return false;
      }
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        report_error(p, DEV_TIMEOUT, ROLE_CHAIN, idx, ld_relaxed_gpu(ctr), target);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Round 4 consecutive fp32 values (row, col..col+3) once to the output type and store them, like
// store_out_chunk (AllGather: C with the e4m3 row scale; ReduceScatter: output shard; AllReduce:
// every rank's output). Rows >= M and columns >= N are skipped.
template <int OP, bool FP8>
__device__ __forceinline__ void store_out_4(const KParams& p, int row, int col, float4 v) {
  if (row >= p.M) return;
  float a[4] = {v.x, v.y, v.z, v.w};
  if constexpr (OP == OP_AG) {
    if constexpr (FP8) {
      const float s = p.row_scale[row / p.M_local];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] *= s;
    }
    if (p.out_fp32) {
      float* o = reinterpret_cast<float*>(p.out[0] + (size_t)row * p.N * 4) + col;
      if (col + 4 <= p.N) {
        st_f4(o, make_float4(a[0], a[1], a[2], a[3]));
      } else {
        for (int i = 0; i < 4; ++i)
          if (col + i < p.N) o[i] = a[i];
      }
      return;
    }
  }
  __nv_bfloat162 b0 = __floats2bfloat162_rn(a[0], a[1]);
  __nv_bfloat162 b1 = __floats2bfloat162_rn(a[2], a[3]);
  const uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1));
  auto put = [&](uint8_t* orow) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(orow) + col;
    if (col + 4 <= p.N) {
      *reinterpret_cast<uint2*>(o) = pk;
    } else {
      for (int i = 0; i < 4; ++i)
        if (col + i < p.N) o[i] = __float2bfloat16_rn(a[i]);
    }
  };
  if constexpr (OP == OP_AG) {
    put(p.out[0] + (size_t)row * p.N * 2);
  } else {
    if (p.allreduce) {
      for (int r = 0; r < p.W; ++r) put(p.out[r] + (size_t)row * p.N * 2);
    } else {
      const int j = row / p.M_local;
      put(p.out[j] + (size_t)(row - j * p.M_local) * p.N * 2);
    }
  }
}

// Slots whose loads a cooperative-fold thread keeps in flight at once: 10 folds the 19 K splits of
// the small-M AllGather in two rounds of loads (12.96 -> 12.74 us per call against 8, three
// rounds); 20 spills registers.
#ifndef TDX_FOLD_GROUP
#define TDX_FOLD_GROUP 10
#endif
constexpr int kFoldGroup = TDX_FOLD_GROUP;

// Fold part `part` of `nparts` of tile `tile`: float4 blocks [part*per, (part+1)*per) of the slot
// layout (float4 f holds row f % 128, columns 32*(f/1024) + 4*((f/128) % 8) .. +3), every one of
// the L slots added in order 0..L-1, rounded once and stored. Called by all epilogue threads.
template <int OP, bool FP8, int BN>
__device__ __forceinline__ void fold_part(const KParams& p, int tile, int part, int nparts, int et, uint64_t pol) {
  constexpr int N4 = kBM * BN / 4;
  const int per = (N4 + nparts - 1) / nparts;
  const int f0 = part * per;
  const int f1 = min(N4, f0 + per);
  const size_t slot_f4 = (size_t)p.T * N4;
  const float4* base = reinterpret_cast<const float4*>(p.sbuf) + (size_t)tile * N4;
  const int m0 = (tile / p.tiles_n) * kBM;
  const int n0 = (tile % p.tiles_n) * BN;
#pragma unroll 1
  for (int f = f0 + et; f < f1; f += kEpiThreads) {
    // slots in groups of kFoldGroup: a group's loads are all in flight before the in-order adds
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
    for (int c0 = 0; c0 < p.L; c0 += kFoldGroup) {
      float4 sv[kFoldGroup];
#pragma unroll
      for (int c = 0; c < kFoldGroup; ++c)
        if (c0 + c < p.L) sv[c] = ld_cg_f4_hint(base + (size_t)(c0 + c) * slot_f4 + f, pol);
#pragma unroll
      for (int c = 0; c < kFoldGroup; ++c) {
        if (c0 + c < p.L) {
          if (c0 + c == 0) {
            acc = sv[c];
          } else {
            acc.x = acc.x + sv[c].x;
            acc.y = acc.y + sv[c].y;
            acc.z = acc.z + sv[c].z;
            acc.w = acc.w + sv[c].w;
          }
        }
      }
    }
    store_out_4<OP, FP8>(p, m0 + (f & 127), n0 + 32 * (f >> 10) + 4 * ((f >> 7) & 7), acc);
  }
}

// Fixed-order fold ((P_0 + P_1) + P_2) + ... of the L fp32 partial slots of one unit of tile `tile`:
// row i of the tile, columns col0..col0+31 (col0 a multiple of 32), two slots' loads in flight at a
// time; rounded once and stored. A warp's 32 lanes take 32 consecutive rows, so every load of the
// slot layout is 512 contiguous bytes.
template <int OP, bool FP8, int BN>
__device__ __forceinline__ void fold_unit_fp32(const KParams& p, int tile, int col0, int i, uint64_t pol) {
  const size_t off = ((size_t)(col0 >> 5) * 8 * kBM + i) * 4;
  const size_t slot = (size_t)p.T * (kBM * BN);
  const float* s0p = p.sbuf + (size_t)tile * (kBM * BN) + off;
  float v[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 s = ld_cg_f4_hint(s0p + j * kBM * 4, pol);
    v[4 * j + 0] = s.x;
    v[4 * j + 1] = s.y;
    v[4 * j + 2] = s.z;
    v[4 * j + 3] = s.w;
  }
  int c = 1;
#pragma unroll 1
  for (; c + 1 < p.L; c += 2) {
    const float* sp0 = s0p + (size_t)c * slot;
    const float* sp1 = sp0 + slot;
    float4 a0[8], a1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      a0[j] = ld_cg_f4_hint(sp0 + j * kBM * 4, pol);
      a1[j] = ld_cg_f4_hint(sp1 + j * kBM * 4, pol);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[4 * j + 0] = (v[4 * j + 0] + a0[j].x) + a1[j].x;
      v[4 * j + 1] = (v[4 * j + 1] + a0[j].y) + a1[j].y;
      v[4 * j + 2] = (v[4 * j + 2] + a0[j].z) + a1[j].z;
      v[4 * j + 3] = (v[4 * j + 3] + a0[j].w) + a1[j].w;
    }
  }
  if (c < p.L) {
    const float* sp = s0p + (size_t)c * slot;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 a = ld_cg_f4_hint(sp + j * kBM * 4, pol);
      v[4 * j + 0] = v[4 * j + 0] + a.x;
      v[4 * j + 1] = v[4 * j + 1] + a.y;
      v[4 * j + 2] = v[4 * j + 2] + a.z;
      v[4 * j + 3] = v[4 * j + 3] + a.w;
    }
  }
  store_out_chunk<OP, FP8>(p, (tile / p.tiles_n) * kBM + i, (tile % p.tiles_n) * BN + col0, v, pol);
}

// MoE combine, one warp: `count` units taken first, first + stride, ...; a unit is one token of the
// shared task list `tasks` at columns [col0, col0 + BN), or, without a list, the (token, N-tile)
// pair of index idx = token * tiles_n + N-tile. Units go two at a time (half h of the warp holds
// the k destination rows and gates of unit h, lane 16h + j for slot j), so the 2k expert-output
// loads of a lane (8 columns each, col0 + 8*lane) are in flight together, and the next pair's rows
// and gates are loaded while the current pair's outputs are. out_s[t] = sum_j g[s][t][j] *
// Z[dest[s][t][j]] in slot order j = 0..k-1 (fp32 fused multiply-adds), rounded once to bf16. The
// expert-output rows were written by other CTAs: read through L2.
__device__ __forceinline__ void moe_unit(const KParams& p, const int* tasks, long long idx, int col0, int BN, int& tok,
                                         int& c0) {
  if (tasks != nullptr) {
    tok = tasks[idx];
    c0 = col0;
  } else {
    tok = static_cast<int>(idx / p.tiles_n);
    c0 = static_cast<int>(idx - (long long)tok * p.tiles_n) * BN;
  }
}

static __device__ __forceinline__ void moe_combine_units(const KParams& p, const int* tasks, long long first,
                                                         long long stride, long long count, int col0, int BN,
                                                         int lane) {
  const int k = p.moe_k;
  const int half = lane >> 4;
  const int slot = lane & 15;
  const uint64_t once = policy_evict_first();
  // this lane's (destination row, gate) for unit 2q + half
  auto meta = [&](long long q, int& d, float& g) {
    d = 0;
    g = 0.0f;
    const long long u = 2 * q + half;
    if (u < count && slot < k) {
      int tok, c0;
      moe_unit(p, tasks, first + u * stride, col0, BN, tok, c0);
      const int s = tok / p.moe_T;
      d = p.moe_dest[(size_t)tok * k + slot];
      g = p.moe_gates[s][(size_t)(tok - s * p.moe_T) * k + slot];
    }
  };
  const long long npairs = (count + 1) / 2;
  int cd;
  float cg;
  meta(0, cd, cg);
#pragma unroll 1
  for (long long q = 0; q < npairs; ++q) {
    int nd = 0;
    float ng = 0.0f;
    if (q + 1 < npairs) meta(q + 1, nd, ng);
    // a warp covers 256 columns (8 per lane) at a time: tiles wider than that are walked in
    // 256-column blocks
#pragma unroll 1
    for (int cb = 0; cb < BN; cb += 256) {
      int tok[2], c[2];
      bool live[2], full[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const long long u = 2 * q + h;
        live[h] = u < count;
        tok[h] = 0;
        c[h] = 0;
        if (live[h]) {
          int c0;
          moe_unit(p, tasks, first + u * stride, col0, BN, tok[h], c0);
          c[h] = c0 + cb + 8 * lane;
          live[h] = cb + 8 * lane < BN && c[h] < p.N;
        }
        full[h] = c[h] + 8 <= p.N;
      }
      float acc[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
      // slots in groups of 8 per unit: a group's loads of both units are in flight together, the sum
      // keeps slot order
#pragma unroll 1
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint4 zr[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int j = j0 + jj;
            const int d = __shfl_sync(0xFFFFFFFFu, cd, 16 * h + (j & 15));
            zr[h][jj] = make_uint4(0u, 0u, 0u, 0u);
            if (j < k && live[h]) {
              const uint8_t* zp = p.G + (size_t)d * p.N * 2 + (size_t)c[h] * 2;
              if (full[h]) {
                zr[h][jj] = ld_cg_v4_hint(zp, once);
              } else {
                uint16_t hv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) hv[i] = c[h] + i < p.N ? reinterpret_cast<const uint16_t*>(zp)[i] : 0;
                zr[h][jj] = make_uint4(hv[0] | (uint32_t(hv[1]) << 16), hv[2] | (uint32_t(hv[3]) << 16),
                                       hv[4] | (uint32_t(hv[5]) << 16), hv[6] | (uint32_t(hv[7]) << 16));
              }
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int j = j0 + jj;
            const float g = __shfl_sync(0xFFFFFFFFu, cg, 16 * h + (j & 15));
            if (j < k) {
              float z[8];
              unpack_bf16x8(zr[h][jj], z);
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(g, z[i], acc[h][i]);
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!live[h]) continue;
        const int s = tok[h] / p.moe_T;
        const int t = tok[h] - s * p.moe_T;
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out[s] + (size_t)t * p.N * 2) + c[h];
        if (full[h]) {
          uint4 pk;
          __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[h][0], acc[h][1]);
          __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[h][2], acc[h][3]);
          __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[h][4], acc[h][5]);
          __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[h][6], acc[h][7]);
          pk.x = *reinterpret_cast<uint32_t*>(&b0);
          pk.y = *reinterpret_cast<uint32_t*>(&b1);
          pk.z = *reinterpret_cast<uint32_t*>(&b2);
          pk.w = *reinterpret_cast<uint32_t*>(&b3);
          st_v4(o, pk);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (c[h] + i < p.N) o[i] = __float2bfloat16_rn(acc[h][i]);
        }
      }
    }
    cd = nd;
    cg = ng;
  }
}

// PM (pair mode): 0 = single CTAs; 2 = CTA pairs running one 2-SM (cta_group::2) MMA stream. Every
// CTA loads only into its own shared memory (no multicast loads), so the same code serves buffers
// that live in another GPU's memory.
template <int BN, bool FP8, int OP, int PM>
__global__ void __launch_bounds__(kNumThreads, 1) tdx_fused_kernel(const __grid_constant__ KParams p) {
  static_assert(PM == 0 || PM == 2, "pair modes: 0 single CTAs, 2 two-SM MMA pairs");
  constexpr int CL = PM == 0 ? 1 : 2;      // CTAs per cluster
  static_assert(PM == 0 || Cfg<BN, FP8, PM == 2>::B_BOXES % 2 == 0, "pairs split B into two halves");
  using C = Cfg<BN, FP8, PM == 2, ring_kb(OP), stg_kb(OP)>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  // misc[0] TMEM base, misc[1] abort flag, misc[2] TMA k-blocks issued, misc[3] MMA k-blocks
  // consumed, misc[4] epilogue go/stop decision, misc[5] epilogue "last arriver" decision, misc[6]
  // MoE combine task count, misc[7] this call's epoch, misc[9] AllGather producer done with the
  // operand ring
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  // MoE dispatch: staging barriers after the row-source table, staging ring 128-byte aligned after them
  uint64_t* stg_bars = reinterpret_cast<uint64_t*>(misc + 16 + kBM);
  uint8_t* stg = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(stg_bars + 8) + 127) & ~static_cast<uintptr_t>(127));

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + C::STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * C::STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * C::STAGES + 2);
  const uint32_t drain_bar = smem_u32(bars + 2 * C::STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t t_entry = globaltimer_ns();

  // Device-kept epochs: every CTA reads the last completed call's epoch at its start and, once it
  // is in shared memory, counts itself in; the CTA whose count completes the grid knows that every
  // CTA has read it, and publishes this call's epoch at its end (the next call, stream-ordered after
  // this kernel, reads it at its start). An epilogue thread, idle until the first accumulator,
  // takes the count, so its round trip is off the kernel's critical path and its tail.
  uint32_t publish_old = 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, PM == 2 ? 2 : 1);   // PM 2: both CTAs' epilogues free the leader's
    }
    mbar_init(drain_bar, 1);
    if constexpr (uses_staging(OP))
      for (int b = 0; b < 8; ++b) mbar_init(smem_u32(stg_bars + b), 1);
    misc[1] = 0;
    misc[2] = 0;
    misc[3] = 0;
    misc[4] = 0;
    misc[5] = 0;
    misc[9] = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    if constexpr (PM == 2) {
      tmem_alloc_pair(smem_u32(&misc[0]), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&misc[0]), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  // Set-up above touches only this CTA's shared and Tensor Memory, so it may overlap the previous
  // kernel on the stream (programmatic dependent launch); everything below may read what that
  // kernel wrote.
  griddep_wait();
  if (threadIdx.x == 0) misc[7] = p.dev_epoch != nullptr ? ld_relaxed_gpu(p.dev_epoch) + 1u : p.epoch;
  if constexpr (CL > 1)
    cluster_sync_all();   // the peer's barriers are initialised before its loads or commits target them
  else
    __syncthreads();
  tc_fence_after();
  const uint64_t t_setup = globaltimer_ns();
  const uint32_t tmem_base = misc[0];
  const uint32_t epoch = misc[7];
  if (p.dev_epoch != nullptr && threadIdx.x == kEpiWarp0 * 32) publish_old = atomicAdd(p.dev_epoch + 1, 1u);
  const int crank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = crank == 0;           // PM 2: the CTA that issues the pair's MMAs
  const int cid = blockIdx.x / CL;          // cluster index
  const int ncl = gridDim.x / CL;           // clusters in the grid

  constexpr bool ag = OP == OP_AG;
  constexpr bool rs = OP == OP_RS;
  const bool ag_move_only = !rs && p.mode == MODE_MOVE_ONLY;   // AllGather / MoE: producer only
  const bool rs_move_only = rs && p.mode == MODE_MOVE_ONLY;
  int t_dyn = p.T;
  bool moe_bad = false;
  if constexpr (OP == OP_MOE || OP == OP_MOE_COMBINE) {
    // the count of 128-row tiles is known only on the device (written by the layout kernel before
    // this launch; never above the host's bound p.T); every one is cut into tiles_n N-tiles
    moe_bad = p.moe_ntiles[1] != 0;
    t_dyn = moe_bad ? 0 : min(p.moe_ntiles[0], p.T) * p.tiles_n;
  }
  const int items_all = ag_move_only ? 0 : p.L * t_dyn;   // (element, tile) work items
  const int items = items_all / CL;                       // items of one cluster-wide sequence
  const bool use_mma = !rs_move_only;  // RS move-only runs the chain on zero partials
  const bool chain = p.L > 1 && !(rs && p.mode == MODE_GEMM_ONLY);
  const int grid = gridDim.x;
  uint32_t* trace = p.trace;
  const int per_cta = (items_all + grid - 1) / grid;

  if (trace != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    trace[0] = grid;
    trace[1] = items_all;
    trace[2] = p.L;
    trace[3] = p.T;
  }

  if (warp == kTmaWarp) {
    // =============================================================== TMA issuer
    if (lane == 0 && use_mma) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      // operand tiles that other tiles re-read are kept in L2 (evict_last); an operand no other tile
      // reads (B of a single M-tile, A of a single N-tile) is streamed (evict_first) so that it does
      // not push out data that is reused, such as the partial slots folded at the end
      const uint64_t keep_a = p.a_streamed ? policy_evict_first() : policy_of(TDX_OPERAND_POLICY);
      const uint64_t keep_b = p.b_streamed ? policy_evict_first() : policy_of(TDX_OPERAND_POLICY);
      uint64_t flag_ns = 0;
      uint32_t n_waits = 0;
      uint64_t t_first = 0;
      bool stop = false;
      if (ag && p.copy_active && p.copy_q1 > 0 && static_cast<int>(blockIdx.x) >= p.copy_lo) {
        // this CTA's producer copies the first chunks through the operand ring: wait until it is done
        stop = !wait_smem_flag(p, misc + 9, abort_flag, 500);
        fence_proxy_async_shared();
      }
      for (int it = cid; it < items && !stop; it += ncl) {
        if (*abort_flag) break;
        const Item w = decode_item<OP, CL>(p, it, BN, crank);
        const CUtensorMap* map_a;
        const CUtensorMap* map_b;
        int arow = w.m0;
        int a_bytes = C::A_BYTES;   // A bytes this CTA loads per K slice
        int pull_r0 = 0, pull_nr = 0;
        if (ag && p.pull_a) {
          // remote data access: the tile's rows are whole shards (128/M_local of them); each is read
          // straight from its shard, so nothing waits on the gathered copy
          map_a = &p.tm_a[0];
          map_b = &p.tm_b[0];
          pull_r0 = w.m0 / p.M_local;
          pull_nr = min(kBM / p.M_local, p.W - pull_r0);
          // one 3D box counts its whole extent (ranks past W are zero-filled); per-shard boxes count
          // only the shards that exist
          a_bytes = p.pull_3d ? C::A_BYTES : pull_nr * p.M_local * 128;
        } else if (ag) {
          map_b = &p.tm_b[0];
          const int self_lo = p.self_rank * p.M_local;
          const bool self_tile = w.m0 >= self_lo && w.m0 + kBM <= self_lo + p.M_local;
          if (self_tile) {
            map_a = &p.tm_a[1];
            arow = w.m0 - self_lo;
          } else {
            map_a = &p.tm_a[0];
            if (p.wait_flags) {
              if (p.perturb) __nanosleep(perturb_hash(p.perturb, it) & 4095u);
              const int last_row = min(w.m0 + kBM, p.M) - 1;
              const int gc0 = w.m0 / p.chunk_rows;
              const int gc1 = last_row / p.chunk_rows;
              ++n_waits;
              if (!wait_flags_all(p, epoch, gc0, gc1, abort_flag, &flag_ns)) break;
              fence_proxy_async_global();
            }
          }
        } else if (OP == OP_MOE || OP == OP_MOE_COMBINE) {
          map_a = &p.tm_a[0];
          map_b = &p.tm_b[0];
          if (p.wait_flags) {
            // the 128-row chunks of the receive buffer holding this expert's rows of the tile; rows
            // past the expert's end are loaded too but never stored, so their chunk is not awaited
            if (p.perturb) __nanosleep(perturb_hash(p.perturb, it) & 4095u);
            ++n_waits;
            if (!wait_flags_all(p, epoch, w.m0 / kBM, (w.mend - 1) / kBM, abort_flag, &flag_ns)) break;
            fence_proxy_async_global();
          }
        } else {
          map_a = &p.tm_a[w.c];
          map_b = &p.tm_b[w.c];
        }
        int kb0, kb1;
        k_range<OP>(p, w, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_mbar(p, empty0 + 8 * stage, phase ^ 1u, abort_flag, 100 + stage)) {
            stop = true;
            break;
          }
          if constexpr (TDX_PREFETCH_AHEAD > 0 && PM != 2) {
            const int kp = kb + TDX_PREFETCH_AHEAD;
            if (kp < kb1) {
              tma_prefetch_2d(map_a, kp * C::BK, arow);
              if constexpr (CL == 1) {
#pragma unroll
                for (int j = 0; j < C::B_BOXES; ++j) tma_prefetch_2d(map_b, w.n0 + j * C::B_BOX_N, kp * C::BK);
              } else {
#pragma unroll
                for (int jj = 0; jj < C::B_BOXES / 2; ++jj)
                  tma_prefetch_2d(map_b, w.n0 + (crank * (C::B_BOXES / 2) + jj) * C::B_BOX_N, kp * C::BK);
              }
            }
          }
          const uint32_t fb = full0 + 8 * stage;
          if constexpr (PM == 0) {
            if (ag && p.pull_a) {
              mbar_arrive_expect_tx(fb, a_bytes + C::B_BYTES);
              if (p.pull_3d) {
                tma_load_3d_hint(smem_u32(sA + stage * C::A_BYTES), &p.tm_a[0], fb, kb * C::BK, 0, pull_r0, keep_a);
              } else {
                for (int q = 0; q < pull_nr; ++q)
                  tma_load_2d_hint(smem_u32(sA + stage * C::A_BYTES + q * p.M_local * 128), &p.tm_a[pull_r0 + q],
                                   fb, kb * C::BK, 0, keep_a);
              }
              load_b_slice<C>(sB + stage * C::B_BYTES, map_b, fb, w.n0, kb, p.b_groups, keep_b);
              goto issued_slice;
            }
          }
          if constexpr (PM == 2) {
            // both CTAs' slices count on the leader's slot barrier, armed once for the pair
            if (leader) mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);
            const uint32_t fbl = mapa_shared(fb, 0);
            tma_load_2d_pair_hint(smem_u32(sA + stage * C::A_BYTES), map_a, fbl, kb * C::BK, arow, keep_a);
#pragma unroll
            for (int jj = 0; jj < C::B_BOXES_CTA; ++jj) {
              // smem box jj = box j of part `part`: this CTA's columns of that MMA's B operand
              const int part = jj / C::BOXES_PART_CTA;
              const int j = jj - part * C::BOXES_PART_CTA;
              const int x = w.n0 + (part * C::BOXES_PART + crank * C::BOXES_PART_CTA + j) * C::B_BOX_N;
              if constexpr (OP == OP_MOE || OP == OP_MOE_COMBINE)
                tma_load_3d_pair_hint(smem_u32(sB + stage * C::B_BYTES + jj * C::B_BOX_BYTES), map_b, fbl,
                                      x, kb * C::BK, w.e, keep_b);
              else
                tma_load_2d_pair_hint(smem_u32(sB + stage * C::B_BYTES + jj * C::B_BOX_BYTES), map_b, fbl,
                                      x, kb * C::BK, keep_b);
            }
          } else {
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
            tma_load_2d_hint(smem_u32(sA + stage * C::A_BYTES), map_a, fb, kb * C::BK, arow, keep_a);
            if constexpr (OP == OP_MOE || OP == OP_MOE_COMBINE) {
#pragma unroll
              for (int j = 0; j < C::B_BOXES; ++j)
                tma_load_3d_hint(smem_u32(sB + stage * C::B_BYTES + j * C::B_BOX_BYTES), map_b, fb,
                                 w.n0 + j * C::B_BOX_N, kb * C::BK, w.e, keep_b);
            } else {
              load_b_slice<C>(sB + stage * C::B_BYTES, map_b, fb, w.n0, kb, p.b_groups, keep_b);
            }
          }
        issued_slice:
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (t_first == 0) t_first = globaltimer_ns();   // once per item, never inside the K loop
      }
      misc[2] = issued;
      if (trace != nullptr) {
        uint32_t* st = trace + 4 + kTraceStatWords * blockIdx.x;
        st[0] = static_cast<uint32_t>(flag_ns > 0xFFFFFFFFull ? 0xFFFFFFFFull : flag_ns);
        st[1] = n_waits;
        st[4] = static_cast<uint32_t>(t_entry);
        st[5] = static_cast<uint32_t>(t_setup);
        st[6] = static_cast<uint32_t>(t_first);
      }
    }
  } else if (warp == kMmaWarp) {
    // =============================================================== MMA issuer
    if (lane == 0 && use_mma && (PM != 2 || leader)) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t consumed = 0;
      int local = 0;
      uint64_t t_first_full = 0;
      bool stop = false;
      for (int it = cid; it < items && !stop; it += ncl, ++local) {
        const Item w = decode_item<OP, CL>(p, it, BN, crank);
        const int acc = C::ACC_BUFS == 2 ? (local & 1) : 0;
        const uint32_t aph = C::ACC_BUFS == 2 ? ((local >> 1) & 1) : (local & 1);
        if (!wait_mbar(p, tempty0 + 8 * acc, aph ^ 1u, abort_flag, 200 + acc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
        int kb0, kb1;
        k_range<OP>(p, w, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_mbar(p, full0 + 8 * stage, phase, abort_flag, 300 + stage)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < C::K_STEPS; ++k) {
            const uint64_t adesc = smem_desc(a_addr + k * 32, 16, C::A_SBO, C::A_LAYOUT);
            const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
#pragma unroll
            for (int part = 0; part < C::N_PARTS; ++part) {
              const uint64_t bdesc =
                  smem_desc(b_addr + part * C::B_PART_BYTES + k * C::UMMA_K * 128, C::B_BOX_BYTES, 1024, 2u);
              const uint32_t dp = d + static_cast<uint32_t>(part * C::MMA_N);
              if constexpr (PM == 2) {
                if constexpr (FP8)
                  umma_f8_pair(dp, adesc, bdesc, C::IDESC, accum);
                else
                  umma_bf16_pair(dp, adesc, bdesc, C::IDESC, accum);
              } else if constexpr (FP8) {
                umma_f8(dp, adesc, bdesc, C::IDESC, accum);
              } else {
                umma_bf16(dp, adesc, bdesc, C::IDESC, accum);
              }
            }
          }
          if constexpr (PM == 0)
            tc_commit(empty0 + 8 * stage);
          else
            tc_commit_pair_multicast(empty0 + 8 * stage, static_cast<uint16_t>(0x3));   // free it in both CTAs
          ++consumed;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
        if (t_first_full == 0) t_first_full = globaltimer_ns();   // once per item, never inside the K loop
        if constexpr (PM == 2)
          tc_commit_pair_multicast(tfull0 + 8 * acc, static_cast<uint16_t>(0x3));   // both halves ready
        else
          tc_commit(tfull0 + 8 * acc);
      }
      // every MMA issued by this thread has completed once the drain barrier flips
      if constexpr (PM == 2)
        tc_commit_pair(drain_bar);
      else
        tc_commit(drain_bar);
      wait_mbar_drain(p, drain_bar, 0);
      misc[3] = consumed;
      if (trace != nullptr) {
        trace[4 + kTraceStatWords * blockIdx.x + 7] = static_cast<uint32_t>(t_first_full);
        trace[4 + kTraceStatWords * blockIdx.x + 8] = static_cast<uint32_t>(globaltimer_ns());
      }
    }
  } else if (warp >= kCopyWarp0 && warp < kCopyWarp0 + kNumCopyWarps) {
    // =============================================================== AllGather producer
    if (ag && p.copy_active) {
      // One thread moves chunk bytes with bulk copies and counts them; the copy that completes a
      // chunk releases the chunk's flag. Chunks are numbered in release order (ranks self+1, ...,
      // self). Phase 1 (fused calls): the chunks the first wave's peer tiles wait for are split
      // evenly over the CTAs holding those tiles (copy_lo..), which copy their share through their
      // own operand ring (idle until those chunks arrive; seven 1/8-ring segments in flight) and
      // then hand the ring to the TMA warp. Phase 2: the other chunks, in pieces taken round-robin
      // by every CTA, through the staging ring after the operand ring.
      const int ct = threadIdx.x - kCopyWarp0 * 32;
      if (ct == 0) {
        const uint64_t lpol = policy_evict_first();   // each shard byte is read once
        const uint64_t spol = policy_of(TDX_AG_STORE_POLICY);   // the GEMM reads the gathered rows next
        uint32_t par = 0;   // staging barrier parities, shared by both rings
        auto copy_chunk_part = [&](int q, long long off, uint32_t n, uint8_t* ring, uint32_t seg, int nb, uint32_t& g) {
          const int rr = q / p.n_chunks;
          const int rank = (p.self_rank + 1 + rr) % p.W;
          const int ck = q - rr * p.n_chunks;
          if (n > 0)
            bulk_copy_contig(p, ring, stg_bars, seg, nb, g, par, p.shard[rank] + (long long)ck * p.chunk_bytes + off,
                             p.G + ((long long)rank * p.M_local + (long long)ck * p.chunk_rows) * p.row_bytes + off, n,
                             lpol, spol);
          ag_chunk_done(p, rank * p.n_chunks + ck, n / 16u, epoch, grid);
        };
        if (p.copy_q1 > 0 && static_cast<int>(blockIdx.x) >= p.copy_lo) {
          constexpr uint32_t kRing = static_cast<uint32_t>(C::STAGES * C::STAGE_BYTES);
          constexpr uint32_t kSeg1 = (kRing / 8) / 16 * 16;
          uint32_t g1 = 0;
          const long long region = (long long)p.copy_q1 * p.chunk_bytes;
          const int nw = grid - p.copy_lo;
          const int b = static_cast<int>(blockIdx.x) - p.copy_lo;
          const long long lo = (region * b / nw) & ~15LL;
          const long long hi = b == nw - 1 ? region : ((region * (b + 1) / nw) & ~15LL);
          if (p.perturb) __nanosleep(perturb_hash(p.perturb, 0x18000u + blockIdx.x) & 4095u);
          for (long long o = lo; o < hi;) {
            const int q = static_cast<int>(o / p.chunk_bytes);
            const long long off = o - (long long)q * p.chunk_bytes;
            const long long end = min(hi, (long long)(q + 1) * p.chunk_bytes);
            copy_chunk_part(q, off, static_cast<uint32_t>(end - o), smem, kSeg1, 8, g1);
            o = end;
          }
          // the operand ring is free: every bulk copy through it has completed
          __threadfence_block();
          *reinterpret_cast<volatile uint32_t*>(misc + 9) = 1u;
        }
        constexpr uint32_t kStg = static_cast<uint32_t>(C::MOE_STG);
        const uint32_t seg = (kStg / 4) / 16 * 16;
        const int nb = min(8, static_cast<int>(kStg / seg));
        uint32_t g2 = 0;
        for (int piece = blockIdx.x; piece < p.total_pieces; piece += grid) {
          const int q = p.copy_q1 + piece / p.ppc;
          const long long off = (long long)(piece % p.ppc) * p.piece_bytes;
          const long long rem = p.chunk_bytes - off;
          const uint32_t n = static_cast<uint32_t>(rem < p.piece_bytes ? rem : p.piece_bytes);
          if (p.perturb) __nanosleep(perturb_hash(p.perturb, 0x10000u + piece) & 4095u);
          copy_chunk_part(q, off, n, stg, seg, nb, g2);
        }
      }
    } else if (OP == OP_MOE && p.copy_active && !moe_bad) {
      // AllToAll dispatch: CTAs take pieces of the receive buffer's 128-row chunks in row order (a
      // whole chunk, or 1/ppc of it when there are fewer chunks than CTAs). The producer threads
      // stage the piece's row sources (row -> s * T + t) in shared memory; one thread moves the rows
      // with bulk copies through a ring of NB shared-memory segments (NB - 1 loads in flight, each
      // segment stored back as soon as it lands) and waits for its stores to complete; the chunk's
      // flag is released by its last piece (a per-chunk counter when ppc > 1).
      const int ct = threadIdx.x - kCopyWarp0 * 32;
      int* psrc = reinterpret_cast<int*>(misc + 16);         // [kBM] row sources of the chunk
      const int ntok = p.W * p.moe_T;
      const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
      // segment: a whole row if it fits a quarter of the ring, else a 16-byte multiple of that
      // quarter (at least four segments in the ring, three loads in flight)
      constexpr uint32_t kStg = static_cast<uint32_t>(C::MOE_STG);
      const uint32_t seg = rb <= kStg / 4 ? rb : (kStg / 4) / 16 * 16;
      const int nb = min(8, static_cast<int>(kStg / seg));
      const int spr = static_cast<int>((rb + seg - 1) / seg);   // segments per row
      uint32_t gseg = 0;                                        // segments issued by this CTA so far
      auto src_of = [&](int tok, uint32_t off) -> const uint8_t* {
        const int s = tok / p.moe_T;
        return p.shard[s] + (long long)(tok - s * p.moe_T) * p.row_bytes + off;
      };
      for (int piece = blockIdx.x; piece < p.total_pieces; piece += grid) {
        const int ck = piece / p.ppc;
        const int pc = piece - ck * p.ppc;
        const int r0 = ck * kBM + pc * p.moe_rpp;
        const int nrows = max(0, min(min(p.moe_rpp, kBM - pc * p.moe_rpp), p.M - r0));
        for (int i = ct; i < nrows; i += kCopyThreads) psrc[i] = p.moe_src[r0 + i];
        named_bar_sync(2, kCopyThreads);
        if (TDX_MOE_PREFETCH_ROWS > 0) {
          for (int i = ct; i < min(nrows, TDX_MOE_PREFETCH_ROWS); i += kCopyThreads) {
            const int tok = psrc[i];
            if (tok >= 0 && tok < ntok) prefetch_l2_bulk(src_of(tok, 0), rb);
          }
        }
        if (p.perturb && ct == 0) __nanosleep(perturb_hash(p.perturb, 0x10000u + piece) & 4095u);
        if (ct == 0) {
          const int nseg = nrows * spr;
          auto issue = [&](int i) {
            const int row = i / spr;
            const uint32_t off = static_cast<uint32_t>(i - row * spr) * seg;
            const uint32_t n = rb - off < seg ? rb - off : seg;
            const uint32_t g = gseg + static_cast<uint32_t>(i);
            const uint32_t b = g % static_cast<uint32_t>(nb);
            const int tok = psrc[row];
            const uint32_t bar = smem_u32(stg_bars + b);
            if (tok >= 0 && tok < ntok) {
              mbar_arrive_expect_tx(bar, n);
              if constexpr (TDX_MOE_LOAD_POLICY >= 0)
                bulk_load_g2s_hint(smem_u32(stg + b * seg), src_of(tok, off), n, bar, policy_of(TDX_MOE_LOAD_POLICY));
              else
                bulk_load_g2s(smem_u32(stg + b * seg), src_of(tok, off), n, bar);
            } else {
              mbar_arrive(bar);   // nothing to move for an invalid source; keep the phases in step
            }
            if (TDX_MOE_PREFETCH_ROWS > 0 && off == 0 && row + TDX_MOE_PREFETCH_ROWS < nrows) {
              const int t2 = psrc[row + TDX_MOE_PREFETCH_ROWS];
              if (t2 >= 0 && t2 < ntok) prefetch_l2_bulk(src_of(t2, 0), rb);
            }
          };
          for (int i = 0; i < min(nb - 1, nseg); ++i) issue(i);
          for (int i = 0; i < nseg; ++i) {
            const int j = i + nb - 1;
            if (j < nseg) {
              bulk_wait_read_all();   // the buffer of segment j held segment i - 1, stored just before
              issue(j);
            }
            const uint32_t g = gseg + static_cast<uint32_t>(i);
            const uint32_t b = g % static_cast<uint32_t>(nb);
            wait_mbar_drain(p, smem_u32(stg_bars + b), (g / static_cast<uint32_t>(nb)) & 1u);
            const int row = i / spr;
            const uint32_t off = static_cast<uint32_t>(i - row * spr) * seg;
            const uint32_t n = rb - off < seg ? rb - off : seg;
            const int tok = psrc[row];
            if (tok >= 0 && tok < ntok) {
              if constexpr (TDX_MOE_STORE_POLICY >= 0)
                bulk_store_s2g_hint(p.G + (long long)(r0 + row) * p.row_bytes + off, smem_u32(stg + b * seg), n,
                                    policy_of(TDX_MOE_STORE_POLICY));
              else
                bulk_store_s2g(p.G + (long long)(r0 + row) * p.row_bytes + off, smem_u32(stg + b * seg), n);
              bulk_commit();
            }
          }
          gseg += static_cast<uint32_t>(nseg);
          bulk_wait_all();            // the piece's rows are written
          fence_proxy_async_global();
          bool release = true;
          if (p.ppc > 1) {
            __threadfence();
            const uint32_t old = atomicAdd(p.chunk_cnt + ck, 1u);
            release = old == static_cast<uint32_t>(p.ppc - 1);
            if (release) p.chunk_cnt[ck] = 0u;
          }
          if (release) {
            const uint32_t prev = ld_relaxed_gpu(p.chunk_flags + ck);
            if (prev >= epoch) report_error(p, DEV_STALE, ROLE_PRODUCER, ck, prev, epoch);
            __threadfence();
            st_release_gpu(p.chunk_flags + ck, epoch);
            if (p.trace != nullptr) trace_release(p, grid, static_cast<uint32_t>(ck));
          }
        }
        named_bar_sync(2, kCopyThreads);   // psrc is rewritten for the next chunk
      }
    }
  } else {
    // =============================================================== epilogue
    const int e = warp - kEpiWarp0;           // 0..7
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int h = e >> 2;                     // column half
    const int row_in_tile = q * 32 + lane;
    const bool elected = threadIdx.x == kEpiWarp0 * 32;
    volatile uint32_t* decision = misc + 4;    // written before barrier 1, read after it
    volatile uint32_t* is_last = misc + 5;     // written between barriers 2 and 3, read after 3
    const bool rs_gemm_only = rs && p.mode == MODE_GEMM_ONLY;
    const bool chained = chain && !p.reduce_last;   // running sum handed from element to element
    const bool slotted = chain && p.reduce_last;    // own partial slot; the last arriver folds
    uint64_t chain_ns = 0;
    const uint64_t once = policy_of(TDX_SUM_POLICY);   // running sums and outputs
    const uint64_t keep_slot = policy_evict_last();     // slotted partials, folded soon after
    const uint64_t z_pol = policy_of(TDX_COMBINE_Z_POLICY);   // MoE expert outputs, combined soon after
    int local = 0;
    for (int it = cid; it < items; it += ncl, ++local) {
      const Item w = decode_item<OP, CL>(p, it, BN, crank);
      const int acc = C::ACC_BUFS == 2 ? (local & 1) : 0;
      const uint32_t aph = C::ACC_BUFS == 2 ? ((local >> 1) & 1) : (local & 1);
      const bool read_s = chained && w.c > 0;
      const bool write_s = (chained && w.c < p.L - 1) || slotted;
      // ReduceScatter GEMM-only: every rank's partial is computed and read out of TMEM, but only the
      // last rank's tile is stored (rounded, into the output): the GEMM without partial traffic
      const bool direct_out = (!chain && (!rs_gemm_only || w.c == p.L - 1)) || (chained && w.c == p.L - 1);
      if (elected) {
        bool ok = true;
        if (use_mma) ok = wait_mbar(p, tfull0 + 8 * acc, aph, abort_flag, 400 + acc);
        if (ok && read_s) {
          if (p.perturb) __nanosleep(perturb_hash(p.perturb, 0x20000u + it) & 4095u);
          ok = wait_flag(p, epoch, p.chain_flags + (size_t)(w.c - 1) * p.T + w.tile, ROLE_CHAIN,
                         (w.c - 1) * p.T + w.tile, abort_flag, &chain_ns);
        }
        if (*abort_flag) ok = false;
        *decision = ok ? 1u : 0u;
        if (trace != nullptr && ok)
          trace[4 + kTraceStatWords * grid + 1 + p.trace_chunks + blockIdx.x * per_cta + local] =
              (static_cast<uint32_t>(w.c) << 24) | static_cast<uint32_t>(w.tile);
      }
      named_bar_sync(1, kEpiThreads);
      if (*decision == 0u) break;
      tc_fence_after();

      const int row = w.m0 + row_in_tile;
      const size_t slot = slotted ? (size_t)w.c * p.T + w.tile : (size_t)w.tile;
      float moe_row_scale = 1.0f;
      if constexpr (FP8 && OP == OP_MOE) {
        if (row < w.mend) {
          const int tok = p.moe_src[row];
          if (tok >= 0 && tok < p.W * p.moe_T) moe_row_scale = p.row_scale[tok / p.moe_T] * p.moe_bscale[w.e];
        }
      }
      float* sb = p.sbuf + slot * (kBM * BN);
#pragma unroll 1
      for (int ch = 0; ch < C::CHUNKS; ++ch) {
        const int col0 = h * C::COLS_PER_WARP + ch * 32;   // column inside the tile
        float v[32];
        if (use_mma) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(acc * BN + col0),
                             r);
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          if constexpr (FP8 && OP == OP_RS) {
            // rank r's partial enters the fold dequantised: scale_a[r] * scale_b[r]
            const float s = p.elem_scale[w.c];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= s;
          }
          if constexpr (FP8 && OP == OP_MOE) {
            // dequantised by the token's source-rank scale and the expert's scale
            const float s = moe_row_scale;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= s;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
        // running-sum layout: element (row i, col 32*cc + 4*j + t) of a tile sits at float
        // ((cc*8 + j)*128 + i)*4 + t, so a warp's 32 rows read 512 contiguous bytes per vector
        float* sp = sb + ((size_t)(col0 >> 5) * 8 * kBM + row_in_tile) * 4;
        if (read_s) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 sv = ld_cg_f4_hint(sp + j * kBM * 4, once);
            v[4 * j + 0] = sv.x + v[4 * j + 0];
            v[4 * j + 1] = sv.y + v[4 * j + 1];
            v[4 * j + 2] = sv.z + v[4 * j + 2];
            v[4 * j + 3] = sv.w + v[4 * j + 3];
          }
        }
        if (write_s) {
          // slotted partials are folded soon after (keep them in L2); a chained running sum is read
          // by the next element much later
          const uint64_t pol = slotted ? keep_slot : once;
          if (p.bf16_partials) {
            // bf16 slot layout: element (row i, col 32*cc + 8*j + t) at bf16 ((cc*4 + j)*128 + i)*8 + t
            uint4 pk[4];
            pack_bf16x32(v, pk);
            uint8_t* bp = reinterpret_cast<uint8_t*>(p.sbuf) + slot * (kBM * BN * 2) +
                          ((size_t)(col0 >> 5) * 4 * kBM + row_in_tile) * 16;
#pragma unroll
            for (int j = 0; j < 4; ++j) st_v4_hint(bp + j * kBM * 16, pk[j], pol);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st_f4_hint(sp + j * kBM * 4, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]), pol);
          }
        }
        if (direct_out)
          store_out_chunk<OP, FP8>(p, ((OP == OP_MOE || OP == OP_MOE_COMBINE) && row >= w.mend) ? p.M : row,
                                   w.n0 + col0, v, OP == OP_MOE_COMBINE ? z_pol : once);
      }
      tc_fence_before();
      named_bar_sync(1, kEpiThreads);
      if (TDX_DISCARD_DEAD && chained && read_s && w.c == p.L - 1) {
        // the running sum of this tile is dead after the last element read it: drop it from L2
        const int et = threadIdx.x - kEpiWarp0 * 32;
        for (int l = et; l < 4 * BN; l += kEpiThreads) discard_l2_line(sb + (size_t)l * 32);
      }
      if (elected) {
        if (use_mma) {
          if constexpr (PM == 2) {
            if (leader)
              mbar_arrive(tempty0 + 8 * acc);
            else
              mbar_arrive_cluster(mapa_shared(tempty0 + 8 * acc, 0));   // free the leader's accumulator
          } else {
            mbar_arrive(tempty0 + 8 * acc);
          }
        }
        if (chained && write_s) {
          __threadfence();
          st_release_gpu(p.chain_flags + (size_t)w.c * p.T + w.tile, epoch);
        }
        if (slotted && p.coop_fold != 2) {
          // count this tile's stored partials; the element that completes the count folds them
          // (cooperative fold: every element waits for the count, then folds its share)
          if (p.perturb) __nanosleep(perturb_hash(p.perturb, 0x30000u + it) & 4095u);
          __threadfence();
          const uint32_t old = atomicAdd(p.tile_cnt + w.tile, 1u);
          if (p.coop_fold) {
            const bool ok = wait_count(p, p.tile_cnt + w.tile, static_cast<uint32_t>(p.L), abort_flag,
                                       static_cast<uint32_t>(w.tile));
            if (ok) fence_acq_rel_gpu();
            *is_last = ok ? 1u : 0u;
          } else {
            const bool last = old == static_cast<uint32_t>(p.L - 1);
            if (last) {
              p.tile_cnt[w.tile] = 0u;
              __threadfence();
            }
            *is_last = last ? 1u : 0u;
          }
        }
      }
      if constexpr (OP == OP_MOE_COMBINE) {
        if (p.mode == MODE_FUSED) {
          // count the stored expert-output rows of every token, per N-tile; tokens whose k rows are
          // now all stored are listed, and the epilogue warps fold them (two tokens per warp iteration)
          volatile int* task_n = reinterpret_cast<volatile int*>(misc + 6);
          int* tasks = reinterpret_cast<int*>(misc + 16);   // [kBM] tokens to combine
          const int et = threadIdx.x - kEpiWarp0 * 32;
          if (et == 0) *task_n = 0;
          named_bar_sync(1, kEpiThreads);
          if (h == 0 && row < w.mend) {
            const int tok = p.moe_src[row];
            if (tok >= 0) {
              if (p.perturb) __nanosleep(perturb_hash(p.perturb, 0x40000u + row) & 1023u);
              __threadfence();
              const size_t ci = (size_t)tok * p.tiles_n + w.n0 / BN;
              const uint32_t old = atomicAdd(p.moe_cnt + ci, 1u);
              if (old == static_cast<uint32_t>(p.moe_k - 1)) {
                p.moe_cnt[ci] = 0u;
                tasks[atomicAdd(const_cast<int*>(task_n), 1)] = tok;
              }
            }
          }
          named_bar_sync(1, kEpiThreads);
          const int nt_tasks = *task_n;
          if (nt_tasks > 0) {
            __threadfence();
            if (e < nt_tasks)
              moe_combine_units(p, tasks, e, kNumEpiWarps, (nt_tasks - e + kNumEpiWarps - 1) / kNumEpiWarps, w.n0, BN,
                                lane);
          }
        }
      }
      if (slotted && p.coop_fold == 1) {
        // cooperative fold: this element folds float4 block [c*per, (c+1)*per) of the tile's slot
        // layout (float4 f holds row f % 128, columns 32*(f/1024) + 4*((f/128) % 8) .. +3), all L
        // slots in order 0..L-1, and the element that completes the tile's done count resets both
        // counters for the next call
        named_bar_sync(1, kEpiThreads);
        if (*is_last) {
          fold_part<OP, FP8, BN>(p, w.tile, w.c, p.L, threadIdx.x - kEpiWarp0 * 32, once);
          named_bar_sync(1, kEpiThreads);
          if (elected) {
            const uint32_t done = atomicAdd(p.tile_done + w.tile, 1u);
            if (done == static_cast<uint32_t>(p.L - 1)) {
              p.tile_cnt[w.tile] = 0u;
              p.tile_done[w.tile] = 0u;
              __threadfence();
            }
          }
        }
      } else if (slotted && p.coop_fold == 0) {
        named_bar_sync(1, kEpiThreads);
        if (*is_last) {
          // fixed-order fold of the L partial slots: ((P_0 + P_1) + P_2) + ..., two slots' loads in
          // flight at a time
#pragma unroll 1
          for (int ch = 0; ch < C::CHUNKS && p.bf16_partials; ++ch) {
            // bf16 partials: widened exactly to fp32, folded in fp32
            const int col0 = h * C::COLS_PER_WARP + ch * 32;
            const size_t off = ((size_t)(col0 >> 5) * 4 * kBM + row_in_tile) * 16;
            const uint8_t* base = reinterpret_cast<const uint8_t*>(p.sbuf) + (size_t)w.tile * (kBM * BN * 2) + off;
            const size_t slot_stride = (size_t)p.T * (kBM * BN * 2);
            float v[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) unpack_bf16x8(ld_cg_v4_hint(base + j * kBM * 16, once), v + 8 * j);
            int c = 1;
#pragma unroll 1
            for (; c + 1 < p.L; c += 2) {
              const uint8_t* b0 = base + (size_t)c * slot_stride;
              uint4 u0[4], u1[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                u0[j] = ld_cg_v4_hint(b0 + j * kBM * 16, once);
                u1[j] = ld_cg_v4_hint(b0 + slot_stride + j * kBM * 16, once);
              }
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float f0[8], f1[8];
                unpack_bf16x8(u0[j], f0);
                unpack_bf16x8(u1[j], f1);
#pragma unroll
                for (int t = 0; t < 8; ++t) v[8 * j + t] = (v[8 * j + t] + f0[t]) + f1[t];
              }
            }
            if (c < p.L) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float f0[8];
                unpack_bf16x8(ld_cg_v4_hint(base + (size_t)c * slot_stride + j * kBM * 16, once), f0);
#pragma unroll
                for (int t = 0; t < 8; ++t) v[8 * j + t] = v[8 * j + t] + f0[t];
              }
            }
            store_out_chunk<OP, FP8>(p, row, w.n0 + col0, v, once);
          }
#pragma unroll 1
          for (int ch = 0; ch < C::CHUNKS && !p.bf16_partials; ++ch)
            fold_unit_fp32<OP, FP8, BN>(p, w.tile, h * C::COLS_PER_WARP + ch * 32, row_in_tile, once);
          if (TDX_DISCARD_DEAD) {
            // every slot of this tile is dead now: drop the lines from L2
            named_bar_sync(1, kEpiThreads);
            const int et = threadIdx.x - kEpiWarp0 * 32;
            const size_t sbytes = (size_t)kBM * BN * (p.bf16_partials ? 2 : 4);
            for (int c = 0; c < p.L; ++c)
              for (int l = et; l < (int)(sbytes / 128); l += kEpiThreads)
                discard_l2_line(reinterpret_cast<uint8_t*>(p.sbuf) + ((size_t)c * p.T + w.tile) * sbytes + (size_t)l * 128);
          }
        }
      }
    }
    const uint64_t t_items_done = globaltimer_ns();
    if constexpr (OP == OP_MOE_COMBINE) {
      if (p.mode == MODE_MOVE_ONLY && !moe_bad) {
        // the combine alone (expert outputs already in place): one (token, N-tile) per warp task
        const long long units = (long long)p.W * p.moe_T * p.tiles_n;
        const long long first = (long long)blockIdx.x * kNumEpiWarps + e;
        const long long stride = (long long)grid * kNumEpiWarps;
        if (first < units) moe_combine_units(p, nullptr, first, stride, (units - first + stride - 1) / stride, 0, BN, lane);
      }
    }
    if (elected && trace != nullptr) {
      uint32_t* st = trace + 4 + kTraceStatWords * blockIdx.x;
      st[2] = static_cast<uint32_t>(chain_ns > 0xFFFFFFFFull ? 0xFFFFFFFFull : chain_ns);
      st[3] = static_cast<uint32_t>(local);
      st[9] = static_cast<uint32_t>(t_items_done);
      st[10] = static_cast<uint32_t>(globaltimer_ns());
    }
  }

  // =============================================================== grid-wide fold
  if (PM == 0 && OP != OP_MOE && OP != OP_MOE_COMBINE && chain && p.reduce_last && p.coop_fold == 2) {   // single CTAs only
    // Every CTA arrives once all its partials are stored (a grid barrier; every CTA of the
    // cooperative launch is resident), then folds a contiguous 1/grid share of all tiles, cut into
    // units of 128 rows x 8 columns (4 KiB of a slot, contiguous in the slot layout), slots in order
    // 0..L-1. The last CTA to leave resets both counters.
    __syncthreads();
    volatile uint32_t* go = misc + 4;
    const uint64_t pol = policy_evict_first();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(p.grid_bar, 1u);
      bool ok = *abort_flag == 0;
      if (ok) ok = wait_count(p, p.grid_bar, static_cast<uint32_t>(grid), abort_flag, 0xFFFFFFu);
      if (ok) fence_acq_rel_gpu();
      *go = ok ? 1u : 0u;
    }
    __syncthreads();
    if (*go != 0u) {
      // a task is one row of one unit (kCols columns): the row's columns of up to 8 slots are loaded
      // at once (a warp's 32 lanes take 32 consecutive rows: 512 contiguous bytes per load), then
      // added in slot order; all 12 warps take tasks
      constexpr int kV = TDX_GRID_FOLD_F4;   // float4 of a slot per task
      constexpr int kCols = 4 * kV;
      const int units = p.T * (BN / kCols);
      const int per = (units + grid - 1) / grid;
      const int g0 = min(units, blockIdx.x * per);
      const int g1 = min(units, g0 + per);
      const size_t slot_f4 = (size_t)p.T * kBM * BN / 4;
#pragma unroll 1
      for (int task = threadIdx.x; task < (g1 - g0) * kBM; task += kNumThreads) {
        const int gu = g0 + (task >> 7);
        const int i = task & (kBM - 1);
        const int tile = gu / (BN / kCols);
        const int ru = gu - tile * (BN / kCols);
        const float4* base = reinterpret_cast<const float4*>(p.sbuf) + (size_t)gu * (kBM * kV) + i;
        float4 a[kV];
#pragma unroll 1
        for (int c0 = 0; c0 < p.L; c0 += 8) {
          float4 x[8][kV];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (c0 + c < p.L) {
#pragma unroll
              for (int v = 0; v < kV; ++v) x[c][v] = ld_cg_f4_hint(base + (size_t)(c0 + c) * slot_f4 + v * kBM, pol);
            }
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (c0 + c < p.L) {
#pragma unroll
              for (int v = 0; v < kV; ++v) {
                if (c0 + c == 0) {
                  a[v] = x[c][v];
                } else {
                  a[v].x = a[v].x + x[c][v].x;
                  a[v].y = a[v].y + x[c][v].y;
                  a[v].z = a[v].z + x[c][v].z;
                  a[v].w = a[v].w + x[c][v].w;
                }
              }
            }
          }
        }
        const int row = (tile / p.tiles_n) * kBM + i;
        const int col = (tile % p.tiles_n) * BN + ru * kCols;
#pragma unroll
        for (int v = 0; v < kV; ++v) store_out_4<OP, FP8>(p, row, col + 4 * v, a[v]);
      }
      if (threadIdx.x == 0 && *go != 0u) {
        __threadfence();
        if (atomicAdd(p.grid_bar + 1, 1u) == static_cast<uint32_t>(grid - 1)) {
          p.grid_bar[0] = 0u;
          p.grid_bar[1] = 0u;
          __threadfence();
        }
      }
    }
    if (trace != nullptr && threadIdx.x == 0)
      trace[4 + kTraceStatWords * blockIdx.x + 10] = static_cast<uint32_t>(globaltimer_ns());
  }

  // =============================================================== teardown
  // the next kernel on the stream may start its set-up on SMs this grid frees from here on
  griddep_launch_dependents();
  __syncthreads();
  if (PM == 2 && !leader && threadIdx.x == kTmaWarp * 32 && use_mma &&
      (*abort_flag || ld_relaxed_gpu(p.status) != 0u)) {
    // abort path of a pair's second CTA: its loads are counted on the leader's barriers, which this
    // CTA cannot observe; give any load still in flight ample time to land before leaving
    for (int i = 0; i < 64; ++i) __nanosleep(1000);
  }
  if (threadIdx.x == kTmaWarp * 32 && use_mma && (PM != 2 || leader)) {
    // loads issued but never consumed by the MMA issuer (abort path) must land before exit
    const uint32_t issued = misc[2];
    const uint32_t consumed = misc[3];
    uint32_t first = consumed;
    if (issued > static_cast<uint32_t>(C::STAGES) && first < issued - C::STAGES) first = issued - C::STAGES;
    for (uint32_t i = first; i < issued; ++i)
      wait_mbar_drain(p, full0 + 8 * (i % C::STAGES), (i / C::STAGES) & 1u);
  }
  tc_fence_before();
  if constexpr (CL > 1)
    cluster_sync_all();   // no CTA leaves while its peer may still load into it or arrive on it
  else
    __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    if constexpr (PM == 2)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (p.dev_epoch != nullptr && threadIdx.x == kEpiWarp0 * 32 && publish_old == gridDim.x - 1) {
    // the CTA that completed the start count publishes this call's epoch and resets the count
    p.dev_epoch[1] = 0u;
    p.dev_epoch[0] = epoch;
  }
}

template <int BN, bool FP8, int OP, int PM>
cudaError_t launch_fused_t(const KParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<BN, FP8, PM == 2, ring_kb(OP), stg_kb(OP)>;
  constexpr int CL = PM == 0 ? 1 : 2;
  // the staging ring / fold region (128-byte aligned) follows the GEMM's shared memory
  constexpr int kSmem = C::SMEM_BYTES + (uses_staging(OP) ? 128 + C::MOE_STG : 0);
  static_assert(!uses_staging(OP) || (C::MOE_STG >= 4096 && kSmem <= 227 * 1024), "staging ring budget");
  // the dynamic shared-memory limit is raised once per device for each instantiation (setting it
  // twice from two host threads is harmless; the flag only saves the call)
  static std::atomic<bool> attr_done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(tdx_fused_kernel<BN, FP8, OP, PM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  if constexpr (CL == 1) {
    // CTAs wait on flags other CTAs release: all of them must be resident at once
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    // pairs of CTAs; the host sizes the grid to the clusters that fit at once
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  }
  // programmatic dependent launch: the set-up may overlap the previous kernel's tail (the kernel
  // waits for that kernel's completion before reading any global memory)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = TDX_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tdx_fused_kernel<BN, FP8, OP, PM>, p);
}

// Largest grid whose CTAs are all resident at once: one CTA per SM, or for pairs twice the number
// of 2-CTA clusters the device can hold simultaneously.
template <int BN, bool FP8, int OP, int PM>
int max_grid_t(int sms) {
  constexpr int CL = PM == 0 ? 1 : 2;
  if constexpr (CL == 1) {
    return sms;
  } else {
    using C = Cfg<BN, FP8, PM == 2, ring_kb(OP), stg_kb(OP)>;
    constexpr int kSmem = C::SMEM_BYTES + (uses_staging(OP) ? 128 + C::MOE_STG : 0);
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
      const int c = cache[dev].load(std::memory_order_relaxed);
      if (c > 0) return c;
    }
    if (cudaFuncSetAttribute(tdx_fused_kernel<BN, FP8, OP, PM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sms, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tdx_fused_kernel<BN, FP8, OP, PM>, &cfg) != cudaSuccess) return 0;
    const int g = n * CL;
    if (dev >= 0 && dev < 64) cache[dev].store(g, std::memory_order_relaxed);
    return g;
  }
}

}  // namespace tdx
