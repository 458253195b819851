// mk_internal.h -- definitions shared by the host launchers and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mk.h"

namespace mk {

// Tile shape of the compute role: one 128 x 256 fp32 accumulator per tile in
// tensor memory (two of them, double-buffered, fill all 512 TMEM columns),
// K consumed in 64-element (128-byte) slabs through a 4-stage smem ring.
constexpr int BM = 128;
constexpr int BN = 256;
#ifndef MK_BK
#define MK_BK 64
#endif
constexpr int BK = MK_BK;                      // 64 (128-B rows of A) or 32 (64-B rows)
static_assert(BK == 64 || BK == 32, "BK must be 64 or 32");
constexpr int STAGES = (BK == 64) ? 4 : 8;
constexpr int A_SWIZZLE_BYTES = BK * 2;        // A rows are one swizzle span wide
#ifndef MK_NTHREADS
#define MK_NTHREADS 384
#endif
// warp 0 TMA, warp 1 MMA, warps 2-5 epilogue, warps 6.. copy (AG / MoE copy-in)
constexpr int NTHREADS = MK_NTHREADS;
constexpr int N_COPY_WARPS = NTHREADS / 32 - 6;
static_assert(N_COPY_WARPS >= 1 && NTHREADS % 32 == 0, "need at least one copy warp");
constexpr int A_STAGE_BYTES = BM * BK * 2;    // K-major, BK*2-byte swizzle
constexpr int B_BOX_BYTES = BK * 64 * 2;      // BK K-rows x 64 N-cols, MN-major, 128-B swizzle
constexpr int B_STAGE_BYTES = BN * BK * 2;    // 4 boxes
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;   // 192 KiB, reused by copy/reduce roles
// CTA pairs (tcgen05 cta_group::2): a pair computes one 256 x 256 tile, each
// CTA holding its 128 rows of A and 128 of the 256 B columns per stage, so a
// stage is 32 KiB (BK = 64) and the same ring holds 6 of them.
constexpr int PSTAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES / 2;
constexpr int PSTAGES = RING_BYTES / PSTAGE_BYTES;
constexpr int MAX_STAGES = STAGES > PSTAGES ? STAGES : PSTAGES;
constexpr int BAR_BYTES = 256;
// MoE combine: ring of rows handed from the epilogue warps to the copy warps
// (16-byte entries after a 64-byte control block), placed after the barriers.
constexpr int CQ_CAP = 512;
constexpr int CQ_BYTES = 64 + 16 * CQ_CAP;
// Epilogue staging (after the combine ring): per epilogue warp 32 rows of 128
// bytes (rows 144 bytes apart, so that neither the row-wise writes nor the
// piece-wise reads of a quarter warp meet in a bank), used to turn the final
// output stores of the running-sum reduction into full 128-byte row segments.
constexpr int EPI_ROW_STRIDE = 144;
constexpr int EPI_WARP_BYTES = 32 * EPI_ROW_STRIDE;
constexpr int EPI_STAGE_BYTES = 4 * EPI_WARP_BYTES;
constexpr int SMEM_BYTES = 1024 + RING_BYTES + BAR_BYTES + CQ_BYTES + EPI_STAGE_BYTES;
static_assert(SMEM_BYTES <= 232448, "dynamic shared memory per block");
constexpr uint32_t TMEM_COLS = 512;
constexpr int TILE_F32 = BM * BN;              // floats in one partial tile
constexpr int MAX_PARTIALS = 16;               // staged partial tiles reduced per output tile
constexpr int MAX_CHAIN_PARTIALS = 128;        // partials per tile of the running-sum reduction
constexpr int COPY_SUB_MAX = 16;               // AG flag stride per 128-row chunk

// Workspace header words (uint32 each).
enum { HDR_TICKET = 0, HDR_ABORT = 1, HDR_STATUS = 2, HDR_DETAIL = 3, HDR_READY = 4, HDR_CLAIM = 5, HDR_WORDS = 64 };
constexpr size_t WS_HDR_BYTES = 256;

enum Op { OP_AG = 0, OP_RS = 1, OP_AR = 2, OP_MOE = 3, OP_MOE_COMBINE = 4, OP_MLP = 5 };

// Role codes used in the error detail word.
enum { WHERE_PRODUCER = 1, WHERE_MMA = 2, WHERE_EPILOGUE = 3, WHERE_COPY = 4, WHERE_REDUCE = 5,
       WHERE_DRAIN = 6, WHERE_MOE = 7, WHERE_BOUNDS = 8 };

// Bounds-checking build (MK_DEBUG_BOUNDS=1, built beside the library as
// libmk_debug.so): device-side index checks on tile coordinates, copy rows,
// MoE slots and received-row sources.  A failed check records MK_ERR_INVALID
// with detail WHERE_BOUNDS * 1e6 + check code * 1e4 + (index % 1e4), raises the
// abort word, skips the access and lets the kernel wind down like a timeout;
// it never traps.  With 0 (the default build) the checks compile to nothing.
#ifndef MK_DEBUG_BOUNDS
#define MK_DEBUG_BOUNDS 0
#endif
enum { BC_TILE = 1, BC_KRANGE = 2, BC_AG_COPY = 3, BC_MOE_COPY = 4, BC_MOE_SRC = 5, BC_MOE_TILE = 6,
       BC_OWNER = 7, BC_MOE_SCATTER = 8, BC_ATTN_TILE = 9, BC_ATTN_COPY = 10 };

struct FusedParams {
  CUtensorMap tmA[MK_MAX_RANKS];   // AG: [0] local shard, [1] gathered A; RS/AR: A_r; MoE: recv_x[d]
  CUtensorMap tmB[MK_MAX_RANKS];   // AG: [0] B; RS/AR: B_r; MoE: W[d] (3-D)
  const uint8_t* shard[MK_MAX_RANKS];
  void* out[MK_MAX_RANKS];
  uint8_t* gathered;
  uint32_t* flags;
  float* staging;
  uint32_t* hdr;
  const int* moe_tiles;            // MoE: tile table (see mk_moe.cu)
  const int* moe_ntiles;           // MoE: number of valid entries in the table
  long long wait_ns;
  uint32_t epoch;
  int op, mode, R, local;
  int M, N, K;
  int m_r;
  int n_mblk, n_nblk, n_kblk;
  int group_m;
  int split_k, kps;
  int P;
  int n_tiles, n_items;
  int n_copy, n_compute, n_reduce;
  int out_f32;
  int copy_local, ordered;
  int inject;
  int rows_per_owner;
  int n_copy_chunks;   // AG: 128-row chunks the copy-in role moves
  int copy_sub;        // AG: sub-chunks per chunk (each its own ready flag), power of 2 <= 16
  int chain;           // RS/AR: 1 = partials summed in rank order by the epilogues (running sum
                       //        forwarded tile by tile); 0 = staged partials + reduce-role CTAs
  int last_arrival;    // RS/AR: 1 = staged partials, the epilogue warp that completes a tile
                       //        quarter (32 rows) sums its partials (with chain = 0)
  int sliced;          // RS/AR with last_arrival: nobody sums on arrival; once its own tiles
                       //        are done, every epilogue warp sums 32-row x 64-column slices of
                       //        tiles whose partials have all arrived
  int pdl;             // launched as a programmatic dependent of the previous kernel on the stream
  int atomic;          // RS/AR: 1 = every partial added into one fp32 tile per output tile with
                       //        red.global.add; the warp that completes a quarter converts it
  int wire_bf16;       // RS/AR running sum: 1 = the sum forwarded between parts is bf16
  int fp8;             // AG/RS/AR: 1 = A and B are fp8 e4m3, B given as its transpose [n x k]
                       //           (both K-major); a k-block is 128 elements (128 bytes)
  int a_esz;           // bytes per A element (2 bf16, 1 fp8)
  unsigned long long* trace;   // per (item, pair rank) records of 8 x u64, or null
  int trace_cap;               // item records available (2 per item); then
                               // MK_TRACE_COPY_RECORDS copy-warp records
  uint32_t* zflags;    // atomic: one word per CTA, = epoch once its slice of the fp32 tiles is zero
  int group_tiles;     // RS/AR chain: tiles per scheduling group
  int copy_warps;      // AG: 1 = copy-in done by the copy warps of every compute CTA, one
                       //     piece counter per chunk (zeroed at kernel start by the CTA
                       //     with ticket 0); 0 = copy-role CTAs with per-sub-chunk flags
  int copy_rows;       // AG copy warps: gathered rows per piece (power of 2 dividing 128)
  int n_cw;            // copy warps per CTA that take part (1 .. N_COPY_WARPS)
  // MoE dispatch (copy warps) and grouped GEMM
  uint8_t* moe_recv_x[MK_MAX_RANKS];     // destination rows, [cap x H] per rank
  const int* moe_src[MK_MAX_RANKS];      // recv_src per rank: g*topk + slot of each row
  const int* moe_recv_counts;            // [R] rows received per rank
  const int* moe_fwd;                    // [R*T*topk] dispatch-order position of each (token, slot)
  const uint32_t* moe_rbase;             // [R] dispatch-order position of each rank's row 0
  const int* moe_ok;                     // 1 when no rank exceeds its capacity
  int moe_T, moe_topk, moe_nblk;         // tokens per rank, slots, 128-row blocks per rank
  int moe_rows_per_piece;                // destination rows per copy piece (divides 128)
  int moe_boost_waves;                   // waves of tiles whose rows every copy warp moves first
  // MoE combine (out[r] = combined rows of source rank r)
  uint8_t* moe_ret[MK_MAX_RANKS];        // [T x topk x N] bf16 returned expert rows per source rank
  const float* moe_gates[MK_MAX_RANKS];  // [T x topk] gate weights per source rank
  uint32_t* moe_cnt;                     // [R*T x n_nblk] slots landed per (token, 256-col block)
  // AG copy-in chunk counters (one per 128-row chunk, COPY_SUB_MAX words apart)
  uint32_t* chunk_cnt;
  // Chained MLP: phase 1 = up-projection tiles of every rank (items 0 .. mlp_n1-1),
  // phase 2 = the down-projection GEMM+ReduceScatter items after them
  uint8_t* mlp_hid[MK_MAX_RANKS];        // [M x mlp_f] bf16 hidden activations per rank
  uint32_t* mlp_cnt;                     // [R x n_mblk] phase-1 tiles done per (rank, row block)
  int mlp_n1, mlp_nb1, mlp_kb1, mlp_f;   // phase-1 items, n-blocks, k-blocks; hidden width
  int mlp_wait;                          // 1 = phase-2 tiles wait for their H_r row block
  int b_one_box;       // 1 = tmB maps are [64 cols, K, N/64 chunks (, experts)] views and a
                       //     stage's B tile (4 column chunks, 2 per CTA of a pair) is one TMA request
  int pair;            // 1 = launched as clusters of 2 CTAs sharing 256 x 256 tiles; items then
                       //     run over m-block pairs and n_compute counts pairs
  int n_mrow;          // m-positions of the raster: n_mblk, or ceil(n_mblk / 2) with pairs
  int n_sched;         // RS/AR: scheduled tiles (n_mrow * n_nblk)
};

// Workspace layout for the AG / RS / AR ops.
struct WsLayout {
  size_t flags_off, n_flags, staging_off, staging_bytes, total;
};

inline long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

// grid = CTAs (with pairs: 2 x pairs, launched as clusters of two).
cudaError_t launch_fused(const FusedParams& p, int grid, cudaStream_t stream);
// Clusters of two CTAs of the fused kernel that fit on the device at once (0 on error).
int max_pair_clusters();
constexpr int MOE_MAX_E = 256;        // experts in total (R * E_loc)
static_assert(2 * MK_MLP_MAX_RANKS <= MK_MAX_RANKS, "the MLP holds W1_r and W2_r maps");
constexpr int MOE_MAX_TOPK = 8;
int device_sm_count();
uint32_t next_epoch();
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// B-operand map over a row-major [k x n] matrix viewed as [64 cols, k, n/64 chunks]
// (n % 64 == 0): one box {64, BK, chunks} is a BK x (64 * chunks) stage tile
// (4 chunks: a single CTA's 256 columns; 2: one CTA's half of a pair's).
bool make_map_b_chunks(CUtensorMap* m, const void* base, uint64_t k, uint64_t n, uint32_t chunks = BN / 64);
// The same for the experts of a rank: [64 cols, H, N/64 chunks, E_loc].
bool make_map_w_chunks(CUtensorMap* m, const void* base, uint64_t h, uint64_t n, uint64_t experts,
                       uint32_t chunks = BN / 64);
// Grid cap for a call (SM count, or mk_config.max_ctas when smaller); 0 without a device.
int grid_cap(const mk_config* cfg);
// CTA pairs where mk_config.cta_pair allows them and at least one pair fits the grid cap.
bool use_pair(const mk_config* cfg, int sms);
// A-operand map: box BK x BM with the swizzle that matches BK.
bool make_map_a(CUtensorMap* m, const void* base, uint64_t k, uint64_t rows, uint64_t row_bytes);
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
                 uint32_t b2);
long long default_wait_ns(const mk_config* cfg);

// Launches kernel(a) as a programmatic dependent of the previous launch on s:
// the kernel must wait (griddepcontrol.wait) before it reads that launch's
// results, and its own launch overlaps that launch's end.
template <class Args>
cudaError_t launch_dependent(void (*kernel)(Args), dim3 grid, dim3 block, cudaStream_t s, const Args& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace mk
