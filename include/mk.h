/*
 * mk.h -- C ABI of the tile-pipelined fused collective + GEMM library for
 * GB300 (sm_103a).
 *
 * The operations are the fused kernels of the mKernel write-up
 * (news.chathome.org, "五种融合内核" table): AllGather + GEMM,
 * GEMM + ReduceScatter, GEMM + AllReduce and MoE Dispatch + GEMM.  The R
 * "ranks" are virtual: each rank's operands are separate device buffers (its
 * partition) in the memory of ONE GPU, and one persistent kernel per call
 * moves data between partitions with in-kernel copy / reduce roles while
 * its compute role runs TMA-fed tcgen05 (TMEM-accumulated) bf16 tiles.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Matrices are row-major.  A operands are [rows x k], B operands [k x n]
 *   (the x @ W convention); outputs are [rows x n].  bf16 inputs, fp32
 *   accumulation, output rounded once to bf16 (round-to-nearest-even) or
 *   written as fp32.
 * - Alignment: every device pointer must be 16-byte aligned; k and n must be
 *   multiples of 8 (16-byte row pitch for the tensor-memory-access engine).
 *   Row counts may be anything (ragged tiles are masked).
 * - Pointer arrays (`const void* const* a` etc.) are HOST arrays of R
 *   DEVICE pointers; the library copies them at call time.
 * - Ownership: the caller owns and allocates every buffer, including the
 *   workspace.  The library allocates no device memory.  It keeps only a
 *   per-device cache of SM count and kernel attributes, and a global call
 *   counter (the epoch) used to tag ready flags.
 * - Workspace: size it with mk_workspace_size() for the same op/shape/config
 *   and zero-fill it ONCE before its first use (cudaMemset); the library
 *   leaves it valid for later calls (flags are epoch-tagged, so no reset is
 *   needed between calls).  One workspace must not be used by two calls that
 *   may run at the same time.
 * - Epoch: every call of an entry point that takes a workspace draws a new
 *   epoch on the host and passes it to its kernels by value; the ready flags
 *   of that call are valid only for that epoch.  A CUDA graph that captured
 *   such a call would replay the epoch of the capture, which leaves stale
 *   flags looking ready, so these calls must not be captured into a graph.
 * - Asynchrony: every compute entry point only enqueues work on `stream`
 *   and returns.  Host-side argument errors return MK_ERR_INVALID /
 *   MK_ERR_UNSUPPORTED before anything is launched; a failed launch returns
 *   MK_ERR_CUDA.  Device-side errors (a ready-flag or pipeline wait that ran
 *   past mk_config.wait_limit_ns, a MoE capacity overflow) are recorded in a
 *   status word inside the workspace: read it with mk_get_device_status().
 *   A wait that times out never hangs the GPU: the kernel stops, releases its
 *   tensor memory and returns.
 * - No C++ exception crosses this interface.
 * - R is limited to MK_MAX_RANKS.
 */
#ifndef MK_H_
#define MK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_MAX_RANKS 16
#define MK_VERSION 1

/* Opaque CUDA stream (identical to cudaStream_t); NULL = legacy default stream. */
typedef struct CUstream_st *mk_stream_t;

typedef enum {
  MK_OK = 0,
  MK_ERR_INVALID = 1,      /* bad argument (NULL pointer, bad size, misaligned, R out of range) */
  MK_ERR_UNSUPPORTED = 2,  /* valid request the library cannot serve (e.g. no sm_103a device) */
  MK_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed                                 */
  MK_ERR_TIMEOUT = 4,      /* device: a bounded wait gave up (missing flag / stalled pipeline)  */
  MK_ERR_CAPACITY = 5      /* device: MoE rows for a rank exceeded cap_rows                     */
} mk_status;

typedef enum { MK_BF16 = 0, MK_F32 = 1 } mk_dtype;

typedef enum { MK_OP_AG_GEMM = 0, MK_OP_GEMM_RS = 1, MK_OP_GEMM_AR = 2, MK_OP_MOE = 3 } mk_op;

/* Execution mode: the fused single-launch path, or one of the two baselines
 * that the same library provides for measuring how much of the data movement
 * the fused path hides. */
typedef enum {
  MK_MODE_FUSED = 0,     /* one persistent launch: copy/reduce roles overlap the GEMM tiles */
  MK_MODE_GEMM_ONLY = 1, /* the same FLOPs with no data movement: AG reads a_gathered as
                            already filled; RS accumulates all ranks in tensor memory; AR
                            (few output tiles) runs one item per (tile, rank) and writes
                            rank r's own product A_r @ B_r to replica r (no reduction)    */
  MK_MODE_UNFUSED = 2    /* host-ordered: a copy launch then a GEMM launch (AG), or a
                            partial-GEMM launch then a reduce launch (RS/AR)               */
} mk_mode;

/* Tuning and test knobs.  Pass NULL, or zero a field, for the built-in choice. */
typedef struct {
  int n_copy_ctas;          /* AG / MoE: CTAs taking the copy-in role                  */
  int n_reduce_ctas;        /* RS / AR: CTAs taking the reduce role                    */
  int max_ctas;             /* cap on the persistent grid (default: one CTA per SM)    */
  int group_m;              /* tile raster: m-blocks per group (default per op)        */
  int split_k;              /* RS / AR: K slices per rank, each its own partial tile   */
  int mode;                 /* mk_mode                                                  */
  long long wait_limit_ns;  /* bound on every device-side wait (default 2e9 ns)        */
  int inject;               /* test only: 1 = one copy-in chunk never signals ready;
                               2 = one partial tile never signals ready                */
  int reduce;               /* RS / AR with n_reduce_ctas == 0: 0 = default: 4 for an AR
                                   with at most 2048 partial tiles (output tiles x R, i.e.
                                   256 MiB of staging) when wire == 0 and split_k <= 1,
                                   else 1,
                               1 = running sum forwarded in rank order by the epilogues,
                               2 = last arrival: every partial staged, the epilogue that
                                   completes a tile sums all of them in rank order,
                               3 = atomic: every partial added into one fp32 tile per
                                   output tile (red.global.add), the epilogue that
                                   completes a tile converts it.  The fp32 summation
                                   order is not fixed: results agree with the other
                                   modes within rounding (exactly when every partial
                                   sum is exact in fp32),
                               4 = sliced: every partial staged without waiting; once
                                   their own tiles are done, all epilogues sum 32-row x
                                   64-column slices of the tiles whose partials have all
                                   arrived, in rank order (the same bits as 1 and 2).  */
  int cta_pair;             /* GEMM tiles: 0 = default (pairs, except for an AR within the
                                   reduce = 4 size limit: one CTA per tile, in every mode),
                               1 = one CTA per 128 x 256 tile,
                               2 = CTA pairs (clusters of two SMs sharing a 256 x 256 tile
                                   through tcgen05 cta_group::2).  Pairs serve every launch
                                   without copy-role or reduce-role CTAs (MoE: 256-row
                                   tiles of each expert's rows); elsewhere, or where the
                                   device cannot co-schedule pairs, single CTAs run.
                                   Results are identical.                               */
  int wire;                 /* RS / AR running sum (reduce 0 or 1): 0 = the sum forwarded
                               from part to part is fp32; 1 = it is rounded to bf16
                               (round-to-nearest-even) at every forward, halving the
                               partial traffic.  Ignored by the other reductions.
                               The chained MLP takes neither reduce = 2, 3 nor wire.    */
  int operand;              /* AG / RS / AR operand type: 0 = bf16 A and B, B given as
                               [k x n] row-major; 1 = fp8 e4m3 A and B, B given as its
                               transpose B^T [n x k] row-major (both operands K-major,
                               the layout of the tensor cores' fp8 path); k % 16 == 0.
                               fp32 accumulation, bf16 / fp32 output as for bf16.  The
                               gathered A of AG is fp8 too.  MoE, combine, the MLP and
                               ring attention take bf16 only (MK_ERR_INVALID).           */
  int trace;                /* AG / RS / AR / MoE dispatch / chained MLP (fused or
                               GEMM-only): 1 = record per-item timestamps into a region
                               at the end of the workspace (see mk_trace_entries,
                               mk_moe_trace_entries, mk_mlp_trace_entries); 0 = off. */
} mk_config;

/* Bytes of workspace an op needs for this shape and config (0 on bad args).
 *   AG:  m = rows per shard (m_r), n, k.        RS / AR: m = rows of each A_r, n, k.
 *   MoE: m = tokens per rank T, n = N, k = H; R ranks; cfg->split_k is ignored.
 * For MoE the E_loc/topk/cap_rows that matter are passed to mk_moe_workspace_size. */
size_t mk_workspace_size(int op, int R, long long m, long long n, long long k,
                         const mk_config *cfg);

/* AllGather + GEMM (five-kernel table, row "AllGather + GEMM"): each rank
 * holds one row shard of A; the shards are gathered and every A tile is
 * consumed by the GEMM as soon as it has landed.  This call computes the
 * result of rank `local_rank`:
 *   a_gathered = [A_0; A_1; ...; A_{R-1}]   ([R*m_r x k] bf16, in rank order)
 *   c          = a_gathered @ b             ([R*m_r x n], c_dtype)
 * a_shards: R device pointers, each [m_r x k] bf16.  b: [k x n] bf16.
 * a_gathered: [R*m_r x k] bf16, written (it may alias a_shards[local_rank]
 * at row offset local_rank*m_r, in which case that shard is not copied).
 * The copy-in role moves the remote shards in ring order local+1, local+2, ...
 * and releases a ready flag per 128-row chunk; compute tiles of the local
 * shard start at once, the others after their chunk's flag.
 * With cfg->operand = 1 the shards, a_gathered and b are fp8 e4m3 and b is
 * B^T ([n x k]): c = a_gathered @ (b)^T.  The same holds for RS and AR. */
mk_status mk_ag_gemm(const void *const *a_shards, const void *b, void *a_gathered, void *c,
                     mk_dtype c_dtype, int R, int local_rank, long long m_r, long long n,
                     long long k, void *workspace, size_t ws_bytes, const mk_config *cfg,
                     mk_stream_t stream);

/* GEMM + ReduceScatter (five-kernel table, row "GEMM + ReduceScatter"):
 *   S = sum_r A_r @ B_r  (A_r [m x k], B_r [k x n], bf16; fp32 accumulation)
 *   c_blocks[o] = rows [o*m/R, (o+1)*m/R) of S   ([m/R x n], c_dtype)
 * m must be a multiple of R.  Every output tile's per-rank partial (fp32) is
 * staged in the owner's slot as soon as it is produced; the reduce role sums
 * the R partials of a tile in rank order 0..R-1 once all have been flagged
 * ready, and writes the owner's block. */
mk_status mk_gemm_rs(const void *const *a, const void *const *b, void *const *c_blocks,
                     mk_dtype c_dtype, int R, long long m, long long n, long long k,
                     void *workspace, size_t ws_bytes, const mk_config *cfg, mk_stream_t stream);

/* GEMM + AllReduce (five-kernel table, row "GEMM + AllReduce"):
 *   S = sum_r A_r @ B_r, and c_replicas[r] = S for every r  ([m x n], c_dtype).
 * Reduced exactly like mk_gemm_rs (rank order 0..R-1); the one reduced tile is
 * written to all R replica buffers, so the replicas are bit-identical. */
mk_status mk_gemm_ar(const void *const *a, const void *const *b, void *const *c_replicas,
                     mk_dtype c_dtype, int R, long long m, long long n, long long k,
                     void *workspace, size_t ws_bytes, const mk_config *cfg, mk_stream_t stream);

/* Workspace bytes for mk_moe_dispatch_gemm (0 on bad args). */
size_t mk_moe_workspace_size(int R, int E_loc, int topk, long long T, long long H, long long N,
                             long long cap_rows, const mk_config *cfg);

/* MoE Dispatch + grouped GEMM (five-kernel table, row "MoE Dispatch + GEMM"):
 * route every token of every rank to its top-k experts, move each
 * (token, expert) row to the rank that holds the expert, and multiply the rows
 * of each expert by that expert's weight, in one pipeline where a GEMM tile
 * starts as soon as its rows have landed.
 *   x[r]:      [T x H] bf16 tokens of rank r (device)
 *   logits[r]: [T x E] fp32 router logits, E = R*E_loc, finite (device)
 *   w[d]:      [E_loc x H x N] bf16 weights of the experts d*E_loc .. d*E_loc+E_loc-1
 * Routing: top-k logits per token, largest first, ties to the lower expert id.
 * Expert e is held by rank e / E_loc.  Rank d receives the rows routed to its
 * experts ordered by (local expert, global token id g = r*T + t).
 * Outputs (all device, int32 unless stated):
 *   topk_idx   [R*T x topk]   expert ids (row g = r*T + t)
 *   counts     [R x E]        counts[r*E + e] = rows of source rank r routed to e
 *   recv_src[d][cap_rows]     g*topk + slot of each received row
 *   recv_counts[R]            rows received by each rank
 *   recv_x[d]  [cap_rows x H] bf16 received rows (bit copies of x rows)
 *   y[d]       [cap_rows x N] bf16, y[d][j] = recv_x[d][j] @ w[d][local expert of j]
 * Rows past recv_counts[d] are left untouched.  If a rank would receive more
 * than cap_rows rows, nothing is dispatched for the call and the device status
 * becomes MK_ERR_CAPACITY.  Limits (else MK_ERR_INVALID, workspace size 0):
 * E = R*E_loc <= 256, 1 <= topk <= min(8, E), H and N multiples of 8,
 * R*T*topk, cap_rows, H and N below 2^31, cap_rows*H below 2^40. */
mk_status mk_moe_dispatch_gemm(const void *const *x, const float *const *logits,
                               const void *const *w, int R, int E_loc, int topk, long long T,
                               long long H, long long N, long long cap_rows, int *topk_idx,
                               int *counts, int *const *recv_src, int *recv_counts,
                               void *const *recv_x, void *const *y, void *workspace,
                               size_t ws_bytes, const mk_config *cfg, mk_stream_t stream);

/* Workspace bytes for mk_moe_combine (0 on bad args). */
size_t mk_moe_combine_workspace_size(int R, int E_loc, int topk, long long T, long long N,
                                     long long H, long long cap_rows, const mk_config *cfg);

/* MoE combine: the step after "MoE Dispatch + GEMM" (five-kernel table, row
 * "MoE Dispatch + GEMM", run in the return direction; the pages describe the
 * dispatch side only).  In one pipeline, every destination rank multiplies the
 * rows of each local expert by that expert's down-projection.  Each product
 * row returns to its token's source rank as soon as its tile is done.  The
 * last of a token's top-k rows to land (per 256-column block) forms the
 * gate-weighted sum.
 *   h[d]:       [cap_rows x N] bf16 expert hidden rows of rank d, in the order
 *               the dispatch delivered them (rows past recv_counts[d] unused)
 *   w2[d]:      [E_loc x N x H] bf16 down-projection of experts d*E_loc ..
 *   gates[r]:   [T x topk] fp32 gate weight of each (token, slot) of rank r
 *   recv_src[d]: [cap_rows] g*topk + slot of each received row (from the dispatch)
 *   counts:     [R x E] int32 rows of source rank r routed to expert e (from
 *               the dispatch; fixes each expert's row segment on its rank)
 *   All pointers are device pointers.
 * Outputs:
 *   ret[r]:  [T x topk x H] bf16; ret[r][t][k] = round_bf16(h[d][j] @ w2[d][l]),
 *            for the row j of rank d that holds (token g = r*T + t, slot k) and
 *            its local expert l (the returned expert rows)
 *   out[r]:  [T x H] bf16; out[r][t] = round_bf16(sum_k gates[r][t][k] * ret[r][t][k]),
 *            summed in fp32 in slot order k = 0..topk-1
 * Every (token, slot) must appear exactly once in the recv_src of the rank
 * that holds its expert; a recv_src entry outside [0, R*T*topk) is skipped and
 * sets the device status to MK_ERR_INVALID.  If a rank's rows (from counts)
 * exceed cap_rows, nothing is computed and the device status becomes
 * MK_ERR_CAPACITY.
 * mode: FUSED (one launch), GEMM_ONLY (the grouped GEMM and the return of the
 * rows; out is not written), UNFUSED (that launch, then a separate
 * weighted-sum launch).  N and H must be multiples of 8, 1 <= topk <= 8,
 * R*E_loc <= 256. */
mk_status mk_moe_combine(const void *const *h, const void *const *w2, const float *const *gates,
                         const int *const *recv_src, const int *counts, int R, int E_loc, int topk,
                         long long T, long long N, long long H, long long cap_rows,
                         void *const *ret, void *const *out, void *workspace, size_t ws_bytes,
                         const mk_config *cfg, mk_stream_t stream);

/* Ranks the chained MLP supports (it holds W1_r and W2_r tensor maps for every rank). */
#define MK_MLP_MAX_RANKS 8

/* Workspace bytes for mk_mlp_ag_rs (0 on bad args or an unsupported config). */
size_t mk_mlp_workspace_size(int R, long long m, long long h, long long f_r, const mk_config *cfg);

/* Chained tensor-parallel MLP layer: "AllGather + GEMM" -> ReLU -> "GEMM +
 * ReduceScatter" (five-kernel table, those two rows; chained in one
 * persistent kernel as the roadmap's multi-step kernel folds fused steps into
 * one launch), over R virtual ranks:
 *   x_gathered = [x_0; ...; x_{R-1}]                  ([R*m x h] bf16, written)
 *   hid[r]     = bf16(ReLU(x_gathered @ w1[r]))       ([R*m x f_r] bf16, written)
 *   S          = sum_r hid[r] @ w2[r]                 (fp32, ranks summed in order 0..R-1)
 *   y_blocks[o] = bf16(rows [o*m, (o+1)*m) of S)      ([m x h] bf16)
 * x_shards[r]: [m x h]; w1[r]: [h x f_r] (column shard of the up-projection);
 * w2[r]: [f_r x h] (row shard of the down-projection); all bf16, device.
 * In one launch, copy warps gather x, the up-projection tiles of every rank
 * start as their row chunk lands, and each down-projection tile starts once
 * the row block of hid[r] it reads is complete; its partial sums run through
 * the running-sum reduction of mk_gemm_rs.  The virtual ranks share one
 * gathered x (every rank's copy would hold the same rows).
 * R <= MK_MLP_MAX_RANKS; h and f_r multiples of 8.  mode: FUSED; GEMM_ONLY
 * (x_gathered as already filled, ranks summed in tensor memory); UNFUSED
 * (copy launch, up-projection launch, partial-tile launch, reduce launch).
 * Configs with split_k > 1, reduce = 2 or n_reduce_ctas > 0 are rejected
 * (MK_ERR_INVALID). */
mk_status mk_mlp_ag_rs(const void *const *x_shards, const void *const *w1, const void *const *w2,
                       int R, long long m, long long h, long long f_r, void *x_gathered,
                       void *const *hid, void *const *y_blocks, void *workspace, size_t ws_bytes,
                       const mk_config *cfg, mk_stream_t stream);

/* Workspace bytes for mk_ring_attention (0 on bad args). */
size_t mk_ring_attention_workspace_size(int R, int heads, long long s_r, int d, int causal,
                                        const mk_config *cfg);

/* Ring Attention (five-kernel table, row "Ring Attention") over R virtual
 * ranks, each holding a contiguous block of s_r positions of the sequence
 * (rank s: positions [s*s_r, (s+1)*s_r)) for every head:
 *   q[r], k[r], v[r]: [heads x s_r x d] bf16 (device), d = 128
 *   out[r] = softmax(scale * Q_r K^T (+ causal mask)) V over the whole
 *            sequence's K and V, [heads x s_r x d] bf16
 * The K/V blocks travel around the ring: at step j rank r receives the block
 * of rank (r - j) mod R into k_recv[r] / v_recv[r] ([(R-1) x heads x s_r x d]
 * bf16 each, step j at block j-1, written), and its query tiles consume each
 * 128-key tile as soon as it has landed, merging the partial softmax results
 * online in fp32 (P rounded to bf16 for the tensor cores).  causal != 0 masks
 * keys after the query position; then the blocks of later ranks are neither
 * moved nor read.  scale > 0 (usually 1/sqrt(d)).  R <= 8.
 * mode: FUSED (one launch); GEMM_ONLY (no ring: K/V read from the source
 * ranks, k_recv/v_recv unused and may be NULL); UNFUSED (a transfer launch,
 * then the attention launch reading the receive buffers). */
mk_status mk_ring_attention(const void *const *q, const void *const *k, const void *const *v, int R,
                            int heads, long long s_r, int d, int causal, float scale,
                            void *const *k_recv, void *const *v_recv, void *const *out,
                            void *workspace, size_t ws_bytes, const mk_config *cfg,
                            mk_stream_t stream);

/* Size of the library's own scratch array used by mk_ag_gemm_noalloc (bytes). */
#define MK_NOALLOC_SCRATCH_BYTES 65536

/* AllGather + GEMM for callers that cannot allocate device memory.
 * The paper has no counterpart for this entry point.
 * Same operation, arguments and results as mk_ag_gemm, but without a
 * workspace: the small scratch the kernel needs (ticket counter, status, one
 * ready flag per copied sub-chunk) lives in a fixed array of
 * MK_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the
 * library holds until the process exits.  It is meant for code that must not
 * call cudaMalloc: a plug-in running inside a host application that owns all
 * GPU memory through its own pool and does not let extensions allocate, or a
 * latency-critical path that may not allocate after start-up (an allocation
 * can synchronise the device and its size is not known in advance).
 *   - Limit: shapes whose scratch would exceed the array (about 1020 chunks of
 *     128 gathered rows, i.e. R*m_r up to 130560 rows) are rejected with
 *     MK_ERR_INVALID before anything is enqueued.
 *   - The first call on a device looks up the array's device address and
 *     zero-fills it on `stream` before its kernel.
 *   - Every call shares the one array and it keeps the previous call's
 *     contents; each call clears the part that must start at zero.  Two calls
 *     whose GPU work can overlap (different streams without ordering, or
 *     different host threads) race on the array: order them on one stream.
 *   - device_status: optional (may be NULL) caller-owned device int, 4-byte
 *     aligned, that receives this call's device status (MK_OK or
 *     MK_ERR_TIMEOUT) once the call's work on `stream` has finished.
 *   - cfg->trace must be 0 (MK_ERR_INVALID otherwise): the trace region would
 *     sit in the library's array, where the caller cannot read it.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
mk_status mk_ag_gemm_noalloc(const void *const *a_shards, const void *b, void *a_gathered, void *c,
                             mk_dtype c_dtype, int R, int local_rank, long long m_r, long long n,
                             long long k, int *device_status, const mk_config *cfg,
                             mk_stream_t stream);

/* In-kernel trace of an AG / RS / AR call made with cfg->trace = 1: the number
 * of records and (in *offset) their byte offset in the workspace; 0 records
 * when tracing is off or the arguments are bad.  Record 2*i + c (c = the CTA's
 * rank in its pair, 0 without pairs) belongs to work item i and holds eight
 * uint64, the first five %globaltimer (ns):
 *   [0] the TMA producer takes the item,
 *   [1] the item's inputs are ready (AG, MoE: its rows have landed;
 *       otherwise the same as [0]),
 *   [2] the producer has issued the item's last load,
 *   [3] the epilogue finds the accumulator complete,
 *   [4] the epilogue has stored (and published) the item;
 *   [5], [6] the SM's clock64 at [0] and at [3] (their ratio to [3] - [0] is
 *       the SM clock over the item);
 *   [7] (call epoch << 32) | (CTA index << 1) | c.
 * MK_TRACE_COPY_RECORDS records of the same size follow, one per copy warp of
 * the AllGather copy-in (record w for worker w = CTA * copy warps + warp):
 *   [0] start and [1] end (ns; the end follows its last chunk release),
 *   [2] pieces and [3] bytes it copied, [7] (call epoch << 32) | w.
 * Records of items a call did not run keep older contents (a lower epoch). */
#define MK_TRACE_COPY_RECORDS 1024
size_t mk_trace_entries(int op, int R, long long m, long long n, long long k, const mk_config *cfg,
                        size_t *offset);

/* The same for a MoE dispatch + grouped GEMM call (arguments as for
 * mk_moe_workspace_size): record 2*i + c belongs to entry i of the call's tile
 * table, with the words of mk_trace_entries ([1]: the tile's rows have been
 * dispatched).  The copy-warp records that follow are reserved (the dispatch
 * copy writes none). */
size_t mk_moe_trace_entries(int R, int E_loc, int topk, long long T, long long H, long long N,
                            long long cap_rows, const mk_config *cfg, size_t *offset);

/* The same for a chained MLP call (arguments as for mk_mlp_workspace_size;
 * MK_MODE_FUSED or MK_MODE_GEMM_ONLY): record 2*i + c belongs to work item i,
 * the up-projection tiles of every rank first, then the down-projection
 * items, with the words of mk_trace_entries ([1]: an up-projection tile's
 * gathered rows have landed; for a down-projection item, when its rows of
 * H_r are complete).  The copy-warp records that follow are those of the
 * AllGather copy-in. */
size_t mk_mlp_trace_entries(int R, long long m, long long h, long long f_r, const mk_config *cfg,
                            size_t *offset);

/* Synchronises `stream`, then reads and clears the device status word of a
 * workspace: MK_OK, MK_ERR_TIMEOUT or MK_ERR_CAPACITY (or MK_ERR_CUDA if the
 * stream itself reports an error).  `detail` (may be NULL) receives a code
 * saying which wait failed (role * 1e6 + item index), for diagnostics. */
mk_status mk_get_device_status(const void *workspace, mk_stream_t stream, long long *detail);

/* Static text for a status code. */
const char *mk_status_string(mk_status s);

/* MK_VERSION of the loaded library. */
int mk_version(void);

/* Number of SMs the library will use on the current device (0 if none). */
int mk_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MK_H_ */
