/*
 * tdx.h -- C ABI of the tile-pipelined collective+GEMM library (sm_103a): AllGather+GEMM,
 * GEMM+ReduceScatter, GEMM+AllReduce and the mixture-of-experts AllToAll dispatch + grouped GEMM
 * and grouped GEMM + combine.
 *
 * What the operations are. The Triton-distributed article on cronfeed.work ("Triton-distributed
 * is turning communication into compiler territory"), section "The first move was to expose the
 * overlap", describes an AllGather that moves row shards into place feeding a GEMM, split into
 * chunks so that the GEMM computes on one chunk while another is still moving, and the mirror
 * operation GEMM-plus-ReduceScatter; communication and computation thread blocks of one kernel
 * are coordinated through symmetric memory and signals. Section "DITRON adds three levels of
 * tiling" adds that collectives such as AllGather and ReduceScatter are broken into chunks, paired
 * with compute tiles, and synchronised (AllToAll and AllReduce among them; the AllToAll entry
 * points are further down). This library implements these kernels for one GPU: the W ranks are
 * logical, i.e. W shard buffers (W partial products for ReduceScatter / AllReduce, W token sets
 * for the AllToAll) in one device's memory; the "network" is a chunk producer that copies shard
 * chunks into a symmetric gathered buffer and releases one flag per chunk, and the GEMM tiles
 * acquire those flags before they read a chunk.
 *
 * Conventions for every entry point:
 *  - Ownership: every tensor and the workspace are device memory owned by the caller. The library
 *    allocates nothing per call and keeps no pointer after a call returns.
 *  - Layout: all matrices are dense and row-major with no padding (row pitch = columns * element
 *    size). Each row pitch must be a multiple of 16 bytes and each pointer 16-byte aligned.
 *  - Asynchrony: calls are stream-ordered on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and return before the work runs. The returned status covers host-side validation and
 *    launch errors only. Errors found on the device (a bounded wait that timed out, a stale epoch)
 *    are recorded in the workspace's status word; read them with tdx_read_device_status. Kernels
 *    never trap: a failed wait makes the kernel stop issuing work, drain what it started and exit.
 *  - Threading: a workspace is used by one call at a time (calls that overlap on the GPU and share a
 *    workspace race). Different workspaces may be used concurrently.
 *  - No fallback: shapes the kernels cannot tile return TDX_ERR_UNSUPPORTED; nothing runs on the CPU.
 */
#ifndef TDX_H_
#define TDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TDX_OK = 0,
  TDX_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, W out of range, bad enum */
  TDX_ERR_UNSUPPORTED = 2,   /* valid request the kernels do not implement (dtype combination, tiling) */
  TDX_ERR_ALIGNMENT = 3,     /* pointer not 16-byte aligned or row pitch not a multiple of 16 bytes */
  TDX_ERR_WORKSPACE = 4,     /* workspace null, misaligned (256 B) or smaller than tdx_workspace_size */
  TDX_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed (launch, tensor map, memset) */
  TDX_ERR_TIMEOUT = 6,       /* device: a bounded wait on a flag or pipeline barrier ran out */
  TDX_ERR_STALE_EPOCH = 7    /* device: a flag already held an epoch >= the call's epoch */
} tdx_status;

typedef enum { TDX_BF16 = 0, TDX_FP8_E4M3 = 1, TDX_FP32 = 2 } tdx_dtype;

/* tdx_opts.epoch value selecting epochs kept on the device (see tdx_opts). */
#define TDX_EPOCH_DEVICE 0xFFFFFFFFu

typedef enum {
  TDX_FUSED = 0,          /* producer and consumer overlapped in one persistent kernel (default) */
  TDX_GEMM_ONLY = 1,      /* AG: GEMM on an already gathered buffer, no flag waits, no copies.
                             RS: every rank's partial tile computed and read out of Tensor Memory,
                             no partial buffer, no rank chain; only rank W-1's partial is stored,
                             rounded to bf16, into the output (the GEMM alone, for measurements) */
  TDX_MOVE_ONLY = 2,      /* AG: chunk copies and flag releases only. RS: the rank-order
                             read-add-write chain over the running-sum buffer with zero partials */
  TDX_CONSUMER_ONLY = 3   /* AG: consumers wait on flags that no producer releases (fault tests) */
} tdx_mode;

typedef enum {
  TDX_PRODUCER_SM = 0,          /* chunk copies by producer warps of the persistent kernel */
  TDX_PRODUCER_COPY_ENGINE = 1  /* not offered (TDX_ERR_UNSUPPORTED): copies issued outside the kernel
                                   that its consumers wait on need not run while it holds every SM */
} tdx_producer;

/* Per-call options. Pass NULL for all defaults; tdx_opts_default fills the same values. */
typedef struct tdx_opts {
  int self_rank;             /* AG: rank whose shard is local; arrival order self, self+1, ... (default 0) */
  int chunk_rows;            /* AG: rows per chunk and per flag; must divide M_local (default min(128, M_local)) */
  tdx_dtype out_dtype;       /* AG: TDX_BF16 (default) or TDX_FP32. RS: TDX_BF16 only */
  const float* scale_a;      /* host array [W]: per-shard (AG) / per-A_r (RS) / per source rank (MoE)
                                e4m3 dequantisation scales (NULL = 1) */
  const float* scale_b;      /* host array: AG [1] B's scale; RS [W] the B_r scales; MoE [E] the
                                experts' scales; e4m3 only (NULL = 1) */
  tdx_mode mode;             /* default TDX_FUSED */
  tdx_producer producer;     /* default TDX_PRODUCER_SM */
  uint32_t epoch;            /* 0: the library clears the flags on `stream` and uses epoch 1.
                                >0: flags are not cleared; the caller passes strictly increasing
                                epochs on one workspace (after tdx_workspace_init).
                                TDX_EPOCH_DEVICE: the epochs are kept in the workspace itself: a
                                call uses the epoch of the last completed call on that workspace
                                plus one and stores it when its kernel finishes. Nothing is cleared
                                and the host tracks nothing, so the same captured call replays
                                correctly in a CUDA graph. Start from a workspace zeroed by
                                tdx_workspace_init, and do not mix with caller epochs on one
                                workspace without re-initialising it (a flag left at a higher
                                epoch is reported as TDX_ERR_STALE_EPOCH). */
  uint64_t timeout_ns;       /* bound of every device-side wait (default 2e9 ns) */
  uint32_t perturb_seed;     /* test only: !=0 injects pseudo-random delays in producers/epilogues */
  void* trace;               /* optional device buffer of tdx_trace_size() bytes, or NULL */
  int num_sms;               /* largest persistent grid; 0 = every SM of the device (a plan with a
                                grid-wide fold takes as many CTAs as give each the same number of
                                work items; small AllGathers split K to fill this many CTAs) */
  int split_k;               /* AG: K splits reduced in fixed order (0 = library choice, 1 = none) */
  int block_n;               /* GEMM tile width 64/128/256, or 512 on 2-SM pairs (cluster 3; one
                                512-column accumulator per CTA, two MMAs per K step; bf16 and e4m3
                                AllGather / ReduceScatter / AllReduce). 0 = library choice */
  int reduce_mode;           /* fixed-order reduction of RS ranks / AG K splits: 0 = library choice,
                                1 = chained (element c adds its partial to the running sum of
                                elements 0..c-1 and hands it on), 2 = slotted (each element stores its
                                partial; the last to arrive folds them in order 0..L-1), 3 = slotted
                                with a grid-wide fold (once every CTA has stored its partials, all
                                CTAs fold 1/grid of every tile each, slots in order 0..L-1; single
                                CTAs and fp32 partials only). All give the same bits. */
  int cluster;               /* how CTAs cooperate on the GEMM: 0 = library choice, 1 = single CTAs,
                                3 = pairs running one 2-SM MMA stream on a 256 x 256 tile (each CTA
                                stages its 128 rows of A and half of B in its own shared memory;
                                needs tile width 256 and an even number of 128-row M-tiles).
                                2 (pairs sharing B through multicast loads) is not offered:
                                TDX_ERR_UNSUPPORTED. */
  int bf16_partials;         /* ReduceScatter / AllReduce: 0 (default) = each rank's partial enters
                                the fold in fp32; 1 = each partial is rounded once to bf16 (RNE, the
                                type a rank would send) before the fp32 fold, which halves the
                                partial-slot traffic. Needs the slotted reduction (reduce_mode 0 or 2);
                                AllGather: must be 0. */
} tdx_opts;

/* Fill *opts with the defaults above. Returns TDX_ERR_INVALID_ARG if opts is NULL. */
tdx_status tdx_opts_default(tdx_opts* opts);

/* Bytes of workspace needed by one call. op = 0: AllGather+GEMM (M_local_or_M = rows per shard);
 * op = 1: GEMM+ReduceScatter, op = 2: GEMM+AllReduce (M_local_or_M = rows of every A_r). The workspace holds the status
 * word, the chunk flags, the symmetric gathered buffer G (AG, (W*M_local) x K of `dtype`) and the
 * fp32 running-sum buffer with its rank-chain flags (RS, and AG with split K). Writes *bytes.
 * After a call the running-sum region holds the last call's fp32 sums (chained: ranks/splits
 * 0..L-2 of every tile) or partials (slotted: one slot per rank/split). */
tdx_status tdx_workspace_size(int op, int W, int M_local_or_M, int K, int N, tdx_dtype dtype,
                              const tdx_opts* opts, size_t* bytes);

/* Zero the control region of a workspace (status word, flags, counters) on `stream`. Call once
 * after allocating a workspace, and again after a call reported a device-side error. */
tdx_status tdx_workspace_init(void* workspace, size_t bytes, void* stream);

/* AllGather+GEMM: C = concat_r(shards[r]) @ B, the shards gathered in rank order 0..W-1.
 * (Triton-distributed article, section "The first move was to expose the overlap": the AllGather
 * moves shards into place, split into chunks, and the GEMM consumes each chunk once it has arrived.)
 *  shards     host array of W device pointers; shards[r] is M_local x K of `dtype`, row-major.
 *             Any addresses; shards at one stride (shards[r] = shards[0] + r * pitch, as in a
 *             symmetric heap) let tiles of small shards read them with fewer, larger loads (a
 *             performance difference only).
 *  B          device, K x N of `dtype`, row-major.
 *  C          device, (W*M_local) x N, row-major, of opts->out_dtype (bf16 or fp32). Row
 *             r*M_local + i of C is row i of shards[r] times B, whatever the arrival order.
 *  workspace  device, 256-byte aligned, workspace_bytes >= tdx_workspace_size(0, ...) with the
 *             same shapes and opts (else TDX_ERR_WORKSPACE). After the call its gathered buffer
 *             holds concat_r(shards[r]) and every chunk flag holds the epoch.
 *  W          logical ranks, 1..16. M_local, K, N >= 0 (M_local or N == 0: nothing is launched;
 *             K == 0: C is filled with zeros).
 *  dtype      TDX_BF16, or TDX_FP8_E4M3 with per-tensor scales: C = scale_a[r]*scale_b*(shard @ B).
 * Accumulation is fp32 on the tensor cores; the output is rounded once, to nearest even. */
tdx_status tdx_ag_gemm(const void* const* shards, const void* B, void* C, void* workspace,
                       size_t workspace_bytes, int W, int M_local, int K, int N, tdx_dtype dtype,
                       const tdx_opts* opts, void* stream);

/* GEMM+ReduceScatter: S = sum_{r=0}^{W-1} A_parts[r] @ B_parts[r], out_shards[j] = rows
 * [j*M/W, (j+1)*M/W) of S. (Same article and section: "GEMM-plus-ReduceScatter"; section "DITRON
 * adds three levels of tiling" lists ReduceScatter among the collectives split into chunks.)
 *  A_parts    host array of W device pointers, each M x K of `dtype`, row-major.
 *  B_parts    host array of W device pointers, each K x N of `dtype`, row-major.
 *  out_shards host array of W device pointers, each (M/W) x N bf16 row-major.
 *  workspace  device, 256-byte aligned, workspace_bytes >= tdx_workspace_size(1, ...) with the
 *             same shapes and opts (else TDX_ERR_WORKSPACE).
 *  W          1..16, and M must be a multiple of W.
 *  dtype      TDX_BF16, or TDX_FP8_E4M3 with per-rank scales: P_r = scale_a[r]*scale_b[r]*(A_r @ B_r).
 * Rank r's fp32 partial tile is added to the running sum of ranks 0..r-1 in that fixed order,
 * ((P_0 + P_1) + P_2) + ..., whatever the timing, so the result is identical run to run; the sum
 * is rounded once to bf16 (nearest even). */
tdx_status tdx_gemm_rs(const void* const* A_parts, const void* const* B_parts,
                       void* const* out_shards, void* workspace, size_t workspace_bytes,
                       int W, int M, int K, int N, tdx_dtype dtype,
                       const tdx_opts* opts, void* stream);

/* Size of the library's built-in scratch array used by tdx_ag_gemm_noalloc: 16 MiB per device. */
#define TDX_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* AllGather+GEMM for callers that cannot allocate device memory themselves: for example code that
 * runs inside a host framework which owns every device allocation and exposes no allocator to it
 * (a plugin of an inference runtime with a fixed memory budget), or a latency-critical caller that
 * cannot accept the device-wide synchronisation cudaMalloc may cause. The pages have no
 * counterpart of this entry point; it is a convenience of this library.
 *
 * Computes exactly what tdx_ag_gemm computes (same shards, B, C, W, M_local, K, N, dtype and opts
 * meaning), but instead of a caller-owned workspace it uses a scratch array that the library
 * declares statically in device memory: TDX_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 * library, held until the process exits. The call itself allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *  - Limit: problems whose tdx_workspace_size(0, W, M_local, K, N, dtype, opts) exceeds
 *    TDX_NOALLOC_SCRATCH_BYTES are rejected with TDX_ERR_WORKSPACE before anything is launched
 *    (the small-M and tiny AllGather shapes fit; W=8 x 1024 x 8192 bf16 does not).
 *  - First call on a device: it looks up the device address of the scratch array (with that
 *    device current) and caches it with the ID of the current CUDA context; make this first call
 *    before any stream capture. The cached address belongs to that context: after the device's
 *    context is destroyed and re-created (for example by cudaDeviceReset), the next call looks the
 *    address up again, and that call too should come before any stream capture.
 *  - Every argument is checked before anything is enqueued: a call that returns an error has
 *    launched nothing and left the scratch array untouched.
 *  - Shared state: every call on a device uses the same array, which keeps the previous call's
 *    contents. Each call clears, on `stream`, the status word and the flags that must start at
 *    zero (opts->epoch is ignored; epoch 1 is used). Calls that overlap on the GPU (different
 *    streams, or different host threads) race on the array: serialise them.
 *  - opts->producer must be TDX_PRODUCER_SM (else TDX_ERR_UNSUPPORTED).
 *  - device_status: optional device pointer to 8 uint32 words. If not NULL, the call copies the
 *    scratch's status word and details (see tdx_read_device_status) there on `stream` once the
 *    kernel has finished; if NULL, device-side errors of this call are not reported. */
tdx_status tdx_ag_gemm_noalloc(const void* const* shards, const void* B, void* C,
                               int W, int M_local, int K, int N, tdx_dtype dtype,
                               const tdx_opts* opts, uint32_t* device_status, void* stream);

/* GEMM+AllReduce: every rank r receives the whole S = sum_{r'} A_parts[r'] @ B_parts[r'] in
 * out_full[r]. (Triton-distributed article, section "DITRON adds three levels of tiling": AllReduce is
 * among the collectives broken into chunks and paired with compute tiles.) Realised as the chunked
 * ReduceScatter above fused with an AllGather: the element that completes a tile's fixed-order fold
 * ((P_0 + P_1) + ...) rounds the tile once to bf16 and writes it into every rank's output, so all W
 * outputs are bit-identical.
 *  A_parts, B_parts, workspace, dtype, scales: as tdx_gemm_rs (workspace sized with op = 2).
 *  out_full   host array of W device pointers, each M x N bf16 row-major. M need not be a multiple
 *             of W. */
tdx_status tdx_gemm_ar(const void* const* A_parts, const void* const* B_parts, void* const* out_full,
                       void* workspace, size_t workspace_bytes, int W, int M, int K, int N, tdx_dtype dtype,
                       const tdx_opts* opts, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Mixture-of-experts AllToAll dispatch + grouped GEMM.
 * (Triton-distributed article, section "DITRON adds three levels of tiling": AllToAll is among the
 * collectives broken into chunks and paired with compute tiles; the tokens routed to each expert of
 * a mixture-of-experts model are known only at run time, so its device-level tiles are sized
 * dynamically.)
 *
 * W ranks; rank s holds T tokens X[s] (T x H of `dtype`, row-major) and their routing topk_idx[s]
 * (T x topk int32 expert ids in [0, E)). Rank rho owns experts rho*E/W .. (rho+1)*E/W - 1. The
 * dispatch sends every (s, t, j) row X[s][t] to expert topk_idx[s][t][j]; the receive side (one
 * buffer for all ranks, in the workspace) groups the W*T*topk rows by expert, experts ascending,
 * and inside an expert by source rank then token, ascending. Expert e's rows are multiplied by its
 * weights B_experts[e] (H x F); Y keeps the dispatched row order:
 *   Y[dest[s][t][j]] = round_bf16(X[s][t] @ B_experts[topk_idx[s][t][j]]),
 * for e4m3 inputs multiplied first by scale_a[s] * scale_b[e] (fp32, in the epilogue).
 * The layout (counts, offsets, row of every pair, GEMM tile table) is computed on the device; the
 * dispatch copies the receive buffer in 128-row chunks, each released by a flag, while the GEMM
 * tiles of the experts whose rows have arrived already run.
 *  X              host array of W device pointers, each T x H of `dtype` (16-byte aligned).
 *  topk_idx       host array of W device pointers, each T x topk int32. Ids outside [0, E) make the
 *                 call do nothing further and record TDX_ERR_INVALID_ARG in the device status.
 *  B_experts      device pointer, E x H x F of `dtype` (expert e's weights at e*H*F).
 *  Y              device pointer, (W*T*topk) x F bf16 (for either input type), the dispatched order.
 *  dest           device pointer, W x T x topk int32 (output): the row of Y of every (s, t, j).
 *  expert_offsets optional device pointer, E + 1 int32 (output): expert e's rows are
 *                 [expert_offsets[e], expert_offsets[e+1]).
 *  workspace      caller-owned device memory of tdx_moe_workspace_size() bytes, 256-byte aligned,
 *                 zeroed once by tdx_workspace_init; it holds the status word, chunk flags, the
 *                 layout tables and the receive buffer ((W*T*topk) x H of `dtype`).
 *  dtype          TDX_BF16, or TDX_FP8_E4M3 with per-tensor scales: opts->scale_a host array [W]
 *                 (one per source rank's tokens), opts->scale_b host array [E] (one per expert's
 *                 weights); NULL = 1. e4m3 needs tile width 128 or 256.
 *  H and F rows of 16-byte multiples (bf16: multiples of 8; e4m3: H and F multiples of 16);
 *  1 <= topk <= E <= 512; W <= 16.
 *  opts: epoch, timeout_ns, perturb_seed, trace, num_sms, block_n and mode (TDX_FUSED, TDX_GEMM_ONLY:
 *  the receive buffer is assumed filled by an earlier call with the same routing, TDX_MOVE_ONLY:
 *  dispatch only) apply; other cooperation options must keep their defaults. */
tdx_status tdx_moe_workspace_size(int W, int T, int H, int F, int E, int topk, tdx_dtype dtype,
                                  const tdx_opts* opts, size_t* bytes);
tdx_status tdx_moe_dispatch_gemm(const void* const* X, const int32_t* const* topk_idx, const void* B_experts,
                                 void* Y, int32_t* dest, int32_t* expert_offsets, void* workspace,
                                 size_t workspace_bytes, int W, int T, int H, int F, int E, int topk,
                                 tdx_dtype dtype, const tdx_opts* opts, void* stream);
/* Plan of one MoE call (16 words to info): [0] tile width, [1] N-tiles, [2] tile-table capacity,
 * [3] 128-row chunks of the dispatched rows (one flag each), [4] dispatched rows W*T*topk, byte
 * offsets in the workspace of [5] chunk flags (uint32 per chunk), [6] tile count + invalid-routing
 * words, [7] expert offsets (int32 [E+1]), [8] source of every dispatched row (int32, s*T + t),
 * [9] tile table (int32x4 {first row, end row of the expert, expert, 0}), [10] receive buffer
 * (dispatch) / expert outputs Z (combine, (W*T*topk) x H bf16 in dispatched order), [11] total
 * workspace bytes, [12] 128-byte K blocks, [13] per-(token, N-tile) arrival counters (combine; 0
 * for the dispatch), [14] dispatched row of every token slot (combine, int32 W x T x topk; 0),
 * [15] CTA cooperation in use: 1 single CTAs, 3 2-SM pairs on two 128-row tiles of one expert
 * (chosen by default for tile width 256 when the experts average at least 8 tiles; the tile table
 * then pads every expert to an even count with an empty tile). opts.cluster: 0 library choice,
 * 1 single, 3 pairs (2: TDX_ERR_UNSUPPORTED). */
tdx_status tdx_moe_plan_info(int W, int T, int H, int F, int E, int topk, tdx_dtype dtype,
                             const tdx_opts* opts, int64_t* info);

/* ---------------------------------------------------------------------------------------------
 * Mixture-of-experts grouped GEMM + AllToAll combine (the reverse of the dispatch above; same
 * article section: AllToAll is chunked and paired with compute tiles).
 *
 * Hd holds the dispatched rows ((W*T*topk) x F bf16) in the order tdx_moe_dispatch_gemm lays out
 * for the same routing topk_idx (grouped by expert, then source rank, then token). Expert e's rows
 * are multiplied by B_experts[e] (F x H) into expert outputs Z, rounded once to bf16 (the type a
 * rank sends back), kept in the workspace in dispatched order; then every token is combined on its
 * source rank with its gates:
 *   out[s][t] = round_bf16( sum_{j=0}^{topk-1} gates[s][t][j] * Z[row of (s, t, j)] ),
 * the sum in slot order j (fp32 fused multiply-adds). A token's combine runs as soon as the tiles
 * holding all its rows are stored (an arrival counter per (token, N-tile); the last arriver folds),
 * so the combine overlaps the GEMM and the result does not depend on timing.
 *  Hd         device pointer, (W*T*topk) x F bf16 (16-byte aligned).
 *  topk_idx   host array of W device pointers, each T x topk int32 expert ids in [0, E).
 *  B_experts  device pointer, E x F x H bf16.
 *  gates      host array of W device pointers, each T x topk fp32.
 *  out        host array of W device pointers, each T x H bf16 (output).
 *  workspace  tdx_moe_combine_workspace_size() bytes, 256-byte aligned, zeroed once by
 *             tdx_workspace_init (layout tables, counters, Z).
 *  F, H multiples of 8; topk <= 16; 1 <= topk <= E <= 512; bf16 only. opts.mode: TDX_FUSED,
 *  TDX_GEMM_ONLY (Z only, no combine), TDX_MOVE_ONLY (combine only, from the Z of an earlier
 *  call with the same routing). */
tdx_status tdx_moe_combine_workspace_size(int W, int T, int F, int H, int E, int topk, tdx_dtype dtype,
                                          const tdx_opts* opts, size_t* bytes);
tdx_status tdx_moe_gemm_combine(const void* Hd, const int32_t* const* topk_idx, const void* B_experts,
                                const float* const* gates, void* const* out, void* workspace,
                                size_t workspace_bytes, int W, int T, int F, int H, int E, int topk,
                                tdx_dtype dtype, const tdx_opts* opts, void* stream);
/* Plan of one combine call: the 16 words of tdx_moe_plan_info, [10] = Z, [13] and [14] set. */
tdx_status tdx_moe_combine_plan_info(int W, int T, int F, int H, int E, int topk, tdx_dtype dtype,
                                     const tdx_opts* opts, int64_t* info);

/* Synchronise `stream`, then read the workspace's device status word into *out (TDX_OK, or the
 * first device-side error since tdx_workspace_init). If detail is not NULL it receives 8 words:
 * [0] status, [1] role that failed (1 flag wait, 2 pipeline wait, 3 chain wait, 4 producer,
 * 5 MoE routing layout: [4] the first invalid expert id seen, [5] E), [2] CTA index, [3] flag/barrier
 * index, [4] value observed, [5] value expected, [6..7] reserved. An invalid MoE routing is reported
 * as TDX_ERR_INVALID_ARG here (the ids are only read on the device). */
tdx_status tdx_read_device_status(const void* workspace, void* stream, tdx_status* out,
                                  uint32_t* detail);

/* Introspection for tests and tools: the tiling and workspace layout a call with these arguments
 * uses. Writes 22 words to info: [0] tile width BN, [1] chain length L (RS: W; AG: K splits),
 * [2] M-tiles, [3] N-tiles, [4] tiles T, [5] K blocks (128 bytes of K each, one ring slot),
 * [6] chunk rows, [7] chunks per rank,
 * byte offsets in the workspace of [8] chunk flags (uint32 [W * chunks], index rank*chunks + c),
 * [9] chunk piece counters, [10] chain flags (uint32 [(L-1) * T], index c*T + tile), [11] gathered
 * buffer G, [12] fp32 running-sum / partial-slot buffer, [13] total workspace bytes, [14] reduce
 * mode in use (1 chained, 2 slotted, 0 none), [15] offset of the per-tile arrival counters,
 * [16] CTA cooperation in use (1 single, 3 2-SM pair), [17] ReduceScatter
 * raster: N-tiles per group (within a rank the tiles are taken group by group, M-tiles, then the
 * group's N-tiles), [18] ReduceScatter rank block:
 * that many positions of a rank's tile order are processed for ranks 0..W-1 before the next block
 * (positions count tiles, or tile pairs when [16] >= 2), [19] 1 if AllGather tiles read A straight
 * from the shards (shards smaller than a 128-row tile: a tile covers 128/M_local whole shards, each
 * loaded from its own buffer, or all in one load when the shards sit at one stride, so no tile waits
 * on the gathered copy, which still completes G and its flags), else 0, [20] bytes per element of the running-sum / partial-slot buffer (4 fp32,
 * 2 bf16 partials), [21] how the slotted fold is shared (single CTAs, fp32 partials; depends on the
 * device's SM count and opts.num_sms): 0 the last arriver folds the tile; 1 every work item is in
 * one wave of the persistent grid, and each element of a tile waits for the tile's L partials and
 * folds 1/L of it; 2 several waves but fewer tiles than CTAs (or reduce_mode 3): after a grid
 * barrier every CTA folds 1/grid of all tiles. */
tdx_status tdx_plan_info(int op, int W, int M_local_or_M, int K, int N, tdx_dtype dtype,
                         const tdx_opts* opts, int64_t* info);

/* Bytes of the optional trace buffer (opts->trace) for a call on `grid` CTAs taking `items` work
 * items and releasing `chunks` chunk flags (AllGather: W * chunks per rank; MoE dispatch: the 128-row
 * chunks of the dispatched rows; 0 otherwise). Layout, in 32-bit words:
 *  [0..3]  {grid, items, chain length, tiles};
 *  then per CTA 12 statistics words {ns spent waiting on chunk flags, number of flag waits, ns
 *          spent waiting on rank-chain flags, items taken, then seven phase stamps, each the low 32
 *          bits of the GPU's nanosecond global timer: kernel entry, set-up done (barriers, Tensor
 *          Memory), all operand loads of the CTA's first item issued, all MMAs of its first item
 *          issued, last MMA completed, epilogue done with the CTA's own items, epilogue done (shared
 *          folds included); the MMA stamps are 0 for the second CTA of a 2-SM pair, the load and
 *          MMA stamps 0 for a CTA without items; then one word 0};
 *  then the producer section: one count of released chunks, then `chunks` words: word k holds the
 *          flag index (AllGather: rank * chunks per rank + chunk) of the k-th chunk released by the
 *          call, whichever CTA released it. The count must be zero when the call starts (pass a
 *          zero-filled buffer); every other word is written by the kernel;
 *  then per CTA, in order, the work items it took, one word each: (chain element << 24) | tile id,
 *          tile id = m_tile * N-tiles + n_tile. CTA b takes items b, b + grid, b + 2*grid, ... (CTA
 *          pairs: pair b/2 takes items b/2, b/2 + grid/2, ...). */
size_t tdx_trace_size(int grid, int items, int chunks);

/* Static description of a status code. Never NULL. */
const char* tdx_status_string(tdx_status s);

/* Library version, (major << 16) | minor. */
uint32_t tdx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TDX_H_ */
