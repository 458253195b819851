// mk_api.cu -- the C ABI for AllGather+GEMM, GEMM+ReduceScatter and
// GEMM+AllReduce: argument checks, workspace layout, tensor-map encoding,
// role split and the launch of the persistent fused kernel.
#include <atomic>
#include <cstring>

#include <cudaTypedefs.h>

#include "mk_internal.h"

namespace mk {

// ------------------------------------------------------------------ small utilities
static std::atomic<uint32_t> g_epoch{0};

uint32_t next_epoch() {
  uint32_t e = ++g_epoch;
  while (e == 0) e = ++g_epoch;  // 0 is the value of a zero-filled flag
  return e;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

long long default_wait_ns(const mk_config* cfg) {
  if (cfg && cfg->wait_limit_ns > 0) return cfg->wait_limit_ns;
  return 2000000000LL;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 2-D map over a row-major [outer x inner] matrix, 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                 uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_a(CUtensorMap* m, const void* base, uint64_t k, uint64_t rows, uint64_t row_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {k, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(BM)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  BK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp8 (byte) 2-D map over a row-major [rows x k] matrix, K-major boxes of
// 128 bytes x box_rows with 128-byte swizzle (A, and B given as B^T).
bool make_map_k8(CUtensorMap* m, const void* base, uint64_t k, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {k, rows};
  cuuint64_t strides[1] = {k};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_b_chunks(CUtensorMap* m, const void* base, uint64_t k, uint64_t n, uint32_t chunks) {
  auto fn = encode_fn();
  if (!fn || (n % 64)) return false;
  cuuint64_t dims[3] = {64, k, n / 64};
  cuuint64_t strides[2] = {n * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BK), chunks};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_w_chunks(CUtensorMap* m, const void* base, uint64_t h, uint64_t n, uint64_t experts,
                       uint32_t chunks) {
  auto fn = encode_fn();
  if (!fn || (n % 64)) return false;
  cuuint64_t dims[4] = {64, h, n / 64, experts};
  cuuint64_t strides[3] = {n * 2, 128, h * n * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(BK), chunks, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A buffer argument is valid when it is 16-byte aligned and, unless the
// buffer it describes is empty, not NULL (empty framework tensors may carry
// a NULL data pointer).
static inline bool buf_ok(const void* p, long long elems) {
  if (elems > 0 && !p) return false;
  return aligned16(p);
}

// Target size of one copy-warp piece of the gathered A (whole rows, power-of-two count).
#ifndef MK_AG_COPY_WARPS
#define MK_AG_COPY_WARPS 2   // copy warps per compute CTA for the AllGather copy-in
#endif
#ifndef MK_CW_PIECE_BYTES
#define MK_CW_PIECE_BYTES 16384
#endif

// SM count used for the device-independent parts of the plan (split-K), so
// that mk_workspace_size gives the same answer with or without a GPU.
constexpr int PLAN_SMS = 148;

// ------------------------------------------------------------------ planning
struct Plan {
  int op, mode, R;
  long long M, N, K, m_r;
  int n_mblk, n_nblk, n_kblk, n_tiles;
  int split_k, kps, P;
  int group_m;
  int chain, last, sliced, atomic, wire, fp8;
  int ar_single;   // AR small enough for the sliced reduction: single CTAs by default
  size_t flags_off, n_flags, staging_off, staging_bytes, total;
  size_t trace_off, trace_n;   // in-kernel trace records (8 x u64 each) at the end, or none
};
constexpr int ZFLAG_WORDS = 1024;   // atomic reduction: one zero-done word per CTA
constexpr long long SLICED_MAX_PARTIAL_TILES = 2048;   // 256 MiB of staged fp32 partial tiles

static bool plan_gemm(int op, int R, long long m, long long n, long long k, const mk_config* cfg,
                      Plan& pl) {
  if (R < 1 || R > MK_MAX_RANKS) return false;
  if (m < 0 || n < 0 || k < 0) return false;
  if ((n % 8) || (k % 8)) return false;
  const int mode = cfg ? cfg->mode : MK_MODE_FUSED;
  if (mode < MK_MODE_FUSED || mode > MK_MODE_UNFUSED) return false;
  pl.op = op;
  pl.mode = mode;
  pl.R = R;
  pl.m_r = m;
  pl.M = (op == OP_AG) ? m * R : m;
  pl.N = n;
  pl.K = k;
  if (pl.M >= (1LL << 31) || n >= (1LL << 31) || k >= (1LL << 31)) return false;
  if (op == OP_RS && R > 0 && (m % R)) return false;
  pl.n_mblk = static_cast<int>(ceil_div_ll(pl.M, BM));
  pl.n_nblk = static_cast<int>(ceil_div_ll(n, BN));
  pl.n_kblk = static_cast<int>(ceil_div_ll(k, BK));
  pl.n_tiles = pl.n_mblk * pl.n_nblk;
  pl.split_k = 1;
  pl.kps = pl.n_kblk;
  pl.P = 1;
  pl.group_m = (cfg && cfg->group_m > 0) ? cfg->group_m : 8;
  pl.flags_off = WS_HDR_BYTES;
  pl.n_flags = 0;
  pl.staging_bytes = 0;
  pl.chain = 0;
  pl.last = 0;
  pl.sliced = 0;
  pl.ar_single = 0;
  pl.atomic = 0;
  pl.wire = 0;
  const int want_reduce = cfg ? cfg->reduce : 0;
  const int want_wire = cfg ? cfg->wire : 0;
  if (want_reduce < 0 || want_reduce > 4 || want_wire < 0 || want_wire > 1) return false;
  // fp8 operands: 128-element k-blocks, and every row a whole number of 16-byte units
  pl.fp8 = cfg ? cfg->operand : 0;
  if (pl.fp8 < 0 || pl.fp8 > 1) return false;
  if (pl.fp8 && (k % 16)) return false;
  if (pl.fp8) pl.n_kblk = static_cast<int>(ceil_div_ll(k, 2 * BK));
  if (op == OP_AG) {
    pl.n_flags = static_cast<size_t>(pl.n_mblk) * COPY_SUB_MAX;
  } else {
    // Fused default: the partials of a tile are summed in rank order by the
    // compute epilogues (one running-sum tile per output tile).  With
    // n_reduce_ctas > 0, or in the unfused baseline, every partial is staged
    // in its own slot and reduce-role CTAs sum them (at most MAX_PARTIALS).
    // Without reduce-role CTAs the fused path reduces in the epilogues, either
    // as a running sum (the default for RS and large AllReduces), by slices
    // (below: the default for small AllReduces) or by last arrival (the warp
    // that completes a tile quarter sums all partials).
    // Two variants of the in-epilogue reduction trade the fixed rank order for
    // less partial traffic: the running sum forwarded in bf16 (wire = 1), and
    // red.global.add of every partial into one fp32 tile per output tile
    // (reduce = 3), converted by the warp that completes it.
    const bool in_epilogue = (mode == MK_MODE_FUSED && !(cfg && cfg->n_reduce_ctas > 0));
    // An AllReduce whose R partials per output tile fit in SLICED_MAX_PARTIAL_TILES
    // staged tiles (the decode shape: few output tiles) reduces by slices by
    // default: every part stages its partial without waiting, and once their own
    // tiles are done all epilogue warps sum 32-row x 64-column slices in rank
    // order -- the running sum's serial chain of R steps was the tail of the
    // launch.  Such AllReduces also run one CTA per tile by default (in every
    // mode, so the GEMM-only baseline has the same tiles): a pair's 256-row
    // tile is half empty at m = 128.
    pl.ar_single = (op == OP_AR && static_cast<long long>(pl.n_tiles) * R <= SLICED_MAX_PARTIAL_TILES) ? 1 : 0;
    int want = want_reduce;
    if (want == 0 && pl.ar_single && in_epilogue && want_wire == 0 && !(cfg && cfg->split_k > 1)) want = 4;
    pl.chain = (in_epilogue && want != 2 && want != 3 && want != 4) ? 1 : 0;
    pl.last = (in_epilogue && (want == 2 || want == 4)) ? 1 : 0;
    pl.sliced = (in_epilogue && want == 4) ? 1 : 0;
    pl.atomic = (in_epilogue && want == 3) ? 1 : 0;
    pl.wire = (pl.chain && want_wire == 1) ? 1 : 0;
    const int max_parts = in_epilogue ? MAX_CHAIN_PARTIALS : MAX_PARTIALS;
    int sk = (cfg && cfg->split_k > 0) ? cfg->split_k : 0;
    if (sk == 0) {
      sk = 1;
      const long long items = static_cast<long long>(pl.n_tiles) * R;
      // Split K only for the staged reduce-role path of a small-M AllReduce;
      // the running-sum reduction is fastest without it.
      if (op == OP_AR && cfg && cfg->n_reduce_ctas > 0 && items > 0 && items < 2LL * PLAN_SMS)
        sk = static_cast<int>(ceil_div_ll(2LL * PLAN_SMS, items));
    }
    sk = std::max(1, std::min(sk, max_parts / R));
    sk = std::min(sk, std::max(1, pl.n_kblk));
    pl.kps = static_cast<int>(ceil_div_ll(std::max(1, pl.n_kblk), sk));
    sk = static_cast<int>(ceil_div_ll(std::max(1, pl.n_kblk), pl.kps));  // drop empty slices
    pl.split_k = sk;
    pl.P = R * sk;
    if (pl.P > max_parts) return false;
    if (mode != MK_MODE_GEMM_ONLY) {
      // flags: one per (tile, partial); last arrival: four 64-bit counters per tile;
      // atomic: four counters per tile, then one zero-done word per CTA
      pl.n_flags = pl.last     ? static_cast<size_t>(pl.n_tiles) * 8
                   : pl.atomic ? static_cast<size_t>(pl.n_tiles) * 4 + ZFLAG_WORDS
                               : static_cast<size_t>(pl.n_tiles) * pl.P;
      const size_t slots = (pl.chain || pl.atomic) ? static_cast<size_t>(pl.n_tiles)
                                                   : static_cast<size_t>(pl.n_tiles) * pl.P;
      pl.staging_bytes = slots * TILE_F32 * sizeof(float);
    }
  }
  size_t off = pl.flags_off + pl.n_flags * sizeof(uint32_t);
  off = (off + 1023) & ~static_cast<size_t>(1023);
  pl.staging_off = off;
  pl.total = off + pl.staging_bytes;
  pl.trace_off = 0;
  pl.trace_n = 0;
  if (cfg && cfg->trace) {
    if (cfg->trace != 1) return false;
    // two records per work item (the CTAs of a pair); items <= tiles x partials
    pl.trace_n = static_cast<size_t>(std::max(pl.n_tiles, 1)) * std::max(pl.P, 1) * 2;
    pl.trace_off = (pl.total + 255) & ~static_cast<size_t>(255);
    pl.total = pl.trace_off + (pl.trace_n + MK_TRACE_COPY_RECORDS) * 64;
  }
  return true;
}

static void fill_common(FusedParams& p, const Plan& pl, uint8_t* ws, const mk_config* cfg,
                        mk_dtype c_dtype) {
  std::memset(&p, 0, sizeof(p));
  p.op = pl.op;
  p.mode = pl.mode;
  p.R = pl.R;
  p.M = static_cast<int>(pl.M);
  p.N = static_cast<int>(pl.N);
  p.K = static_cast<int>(pl.K);
  p.m_r = static_cast<int>(pl.m_r);
  p.n_mblk = pl.n_mblk;
  p.n_nblk = pl.n_nblk;
  p.n_kblk = pl.n_kblk;
  p.n_tiles = pl.n_tiles;
  p.n_mrow = pl.n_mblk;
  p.n_sched = pl.n_tiles;
  p.group_m = pl.group_m;
  p.split_k = pl.split_k;
  p.kps = pl.kps;
  p.P = pl.P;
  p.chain = pl.chain;
  p.last_arrival = pl.last;
  p.sliced = pl.sliced;
  p.atomic = pl.atomic;
  p.wire_bf16 = pl.wire;
  p.fp8 = pl.fp8;
  p.a_esz = pl.fp8 ? 1 : 2;
  p.trace = pl.trace_n ? reinterpret_cast<unsigned long long*>(ws + pl.trace_off) : nullptr;
  p.trace_cap = static_cast<int>(pl.trace_n);
  p.copy_sub = 1;
  p.out_f32 = (c_dtype == MK_F32) ? 1 : 0;
  p.hdr = reinterpret_cast<uint32_t*>(ws);
  p.flags = reinterpret_cast<uint32_t*>(ws + pl.flags_off);
  p.chunk_cnt = p.flags;
  p.staging = reinterpret_cast<float*>(ws + pl.staging_off);
  p.zflags = pl.atomic ? p.flags + static_cast<size_t>(pl.n_tiles) * 4 : nullptr;
  p.wait_ns = default_wait_ns(cfg);
  p.inject = cfg ? cfg->inject : 0;
  p.epoch = next_epoch();
}

static mk_status launch(FusedParams& p, int n_copy, int n_compute, int n_reduce, cudaStream_t s) {
  p.pair = 0;
  p.n_mrow = p.n_mblk;
  p.n_sched = p.n_tiles;
  p.n_copy = n_copy;
  p.n_compute = n_compute;
  p.n_reduce = n_reduce;
  const int grid = n_copy + n_compute + n_reduce;
  if (grid <= 0) return MK_OK;
  return launch_fused(p, grid, s) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

// CTA pairs where the config allows them (mk_config.cta_pair) and the device
// co-schedules at least one pair within the grid cap.
bool use_pair(const mk_config* cfg, int sms) {
  const int v = cfg ? cfg->cta_pair : 0;
  if (v == 1) return false;
  return std::min(max_pair_clusters(), sms / 2) > 0;
}

// Launch of compute CTAs only (no copy-role or reduce-role CTAs): CTA pairs
// on 256 x 256 tiles when wanted and the device co-schedules them, else one
// CTA per 128 x 256 tile.  Sets the item count for the chosen shape.
// Chained MLP: phases = 1 (up-projection items only), 2 (down-projection only), 3 (both).
static void set_items(FusedParams& p, int per, int mlp_phases) {
  p.n_items = p.n_sched * per;
  if (p.op != OP_MLP) return;
  p.mlp_n1 = (mlp_phases & 1) ? p.n_mrow * p.R * p.mlp_nb1 : 0;
  p.n_items = p.mlp_n1 + ((mlp_phases & 2) ? p.n_items : 0);
}

static mk_status launch_compute(FusedParams& p, bool pair, int sms, cudaStream_t s, int mlp_phases = 3) {
  // AR GEMM-only: one item per (tile, rank) (see decode); other GEMM-only
  // launches sum every rank of a tile in one item
  const int per = (p.op == OP_AG) ? 1
                  : (p.mode == MK_MODE_GEMM_ONLY) ? (p.op == OP_AR ? p.R : 1)
                                                  : p.P;
  if (pair && p.op != OP_MOE) {
    const int clusters = std::min(max_pair_clusters(), sms / 2);
    {
      p.pair = 1;
      p.n_mrow = (p.n_mblk + 1) / 2;
      p.n_sched = p.n_mrow * p.n_nblk;
      set_items(p, per, mlp_phases);
      const int n_pairs = std::min(clusters, p.n_items);
      if (n_pairs <= 0) return MK_OK;
      p.group_tiles = std::max(1, std::min(n_pairs, p.n_sched));
      p.n_copy = 0;
      p.n_compute = n_pairs;
      p.n_reduce = 0;
      if (p.atomic && 2 * n_pairs > ZFLAG_WORDS) return MK_ERR_UNSUPPORTED;
      return launch_fused(p, 2 * n_pairs, s) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
    }
  }
  p.pair = 0;
  p.n_mrow = p.n_mblk;
  p.n_sched = p.n_mblk * p.n_nblk;
  set_items(p, per, mlp_phases);
  const int n = std::min(sms, p.n_items);
  if (n <= 0) return MK_OK;
  if (p.atomic && n > ZFLAG_WORDS) return MK_ERR_UNSUPPORTED;
  p.group_tiles = std::max(1, std::min(n, p.n_sched));
  p.n_copy = 0;
  p.n_compute = n;
  p.n_reduce = 0;
  return launch_fused(p, n, s) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

int grid_cap(const mk_config* cfg) {
  int sms = device_sm_count();
  if (sms <= 0) return 0;
  if (cfg && cfg->max_ctas > 0) sms = std::min(sms, cfg->max_ctas);
  return sms;
}

static mk_status zero_outputs(void* const* outs, int nout, size_t bytes, cudaStream_t s) {
  for (int i = 0; i < nout; ++i)
    if (bytes && cudaMemsetAsync(outs[i], 0, bytes, s) != cudaSuccess) return MK_ERR_CUDA;
  return MK_OK;
}

}  // namespace mk

using namespace mk;

extern "C" {

int mk_version(void) { return MK_VERSION; }

int mk_device_sm_count(void) { return device_sm_count(); }

const char* mk_status_string(mk_status s) {
  switch (s) {
    case MK_OK: return "ok";
    case MK_ERR_INVALID: return "invalid argument";
    case MK_ERR_UNSUPPORTED: return "unsupported on this device or build";
    case MK_ERR_CUDA: return "CUDA error";
    case MK_ERR_TIMEOUT: return "device wait timed out (a ready flag or pipeline stage never arrived)";
    case MK_ERR_CAPACITY: return "MoE receive capacity exceeded";
  }
  return "unknown status";
}

size_t mk_workspace_size(int op, int R, long long m, long long n, long long k, const mk_config* cfg) {
  if (op == MK_OP_MOE) return 0;
  if (op < MK_OP_AG_GEMM || op > MK_OP_GEMM_AR) return 0;
  Plan pl;
  if (!plan_gemm(op, R, m, n, k, cfg, pl)) return 0;
  return pl.total;
}

size_t mk_trace_entries(int op, int R, long long m, long long n, long long k, const mk_config* cfg,
                        size_t* offset) {
  if (offset) *offset = 0;
  if (op < MK_OP_AG_GEMM || op > MK_OP_GEMM_AR) return 0;
  Plan pl;
  if (!plan_gemm(op, R, m, n, k, cfg, pl)) return 0;
  if (offset) *offset = pl.trace_off;
  return pl.trace_n;
}

mk_status mk_get_device_status(const void* workspace, mk_stream_t stream, long long* detail) {
  if (!workspace) return MK_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MK_ERR_CUDA;
  uint32_t h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MK_ERR_CUDA;
  if (detail) *detail = static_cast<long long>(static_cast<int32_t>(h[HDR_DETAIL]));
  if (h[HDR_STATUS] != 0) {
    uint32_t z[2] = {0, 0};
    if (cudaMemcpy(reinterpret_cast<uint8_t*>(const_cast<void*>(workspace)) + 4 * HDR_STATUS, z,
                   sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess)
      return MK_ERR_CUDA;
  }
  return static_cast<mk_status>(h[HDR_STATUS]);
}

mk_status mk_ag_gemm(const void* const* a_shards, const void* b, void* a_gathered, void* c,
                     mk_dtype c_dtype, int R, int local_rank, long long m_r, long long n, long long k,
                     void* workspace, size_t ws_bytes, const mk_config* cfg, mk_stream_t stream) {
  if (!a_shards || !workspace) return MK_ERR_INVALID;
  if (c_dtype != MK_BF16 && c_dtype != MK_F32) return MK_ERR_INVALID;
  if (R < 1 || R > MK_MAX_RANKS || local_rank < 0 || local_rank >= R) return MK_ERR_INVALID;
  if (m_r < 0 || n < 0 || k < 0) return MK_ERR_INVALID;
  for (int r = 0; r < R; ++r)
    if (!buf_ok(a_shards[r], m_r * k)) return MK_ERR_INVALID;
  if (!buf_ok(b, k * n) || !buf_ok(a_gathered, R * m_r * k) || !buf_ok(c, R * m_r * n) ||
      !aligned16(workspace))
    return MK_ERR_INVALID;
  Plan pl;
  if (!plan_gemm(OP_AG, R, m_r, n, k, cfg, pl)) return MK_ERR_INVALID;
  if (ws_bytes < pl.total) return MK_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (m_r == 0) return MK_OK;
  const int sms = grid_cap(cfg);
  if (sms <= 0) return MK_ERR_UNSUPPORTED;

  FusedParams p;
  fill_common(p, pl, static_cast<uint8_t*>(workspace), cfg, c_dtype);
  p.local = local_rank;
  p.b_one_box = (n % 64 == 0) ? 1 : 0;
  p.gathered = static_cast<uint8_t*>(a_gathered);
  for (int r = 0; r < R; ++r) p.shard[r] = static_cast<const uint8_t*>(a_shards[r]);
  p.out[0] = c;
  const size_t row_bytes = static_cast<size_t>(k) * p.a_esz;
  p.copy_local = (static_cast<const uint8_t*>(a_shards[local_rank]) !=
                  static_cast<uint8_t*>(a_gathered) + static_cast<size_t>(local_rank) * m_r * row_bytes)
                     ? 1 : 0;
  p.ordered = (m_r % BM == 0) ? 1 : 0;
  const int bps = static_cast<int>(m_r / BM);
  p.n_copy_chunks = p.ordered ? (p.copy_local ? R : R - 1) * bps : pl.n_mblk;
  const int n_items = (k > 0 && n > 0) ? pl.n_mblk * pl.n_nblk : 0;
  p.n_items = n_items;

  // Sub-chunks per 128-row chunk: as many as copy CTAs (a power of two,
  // <= 16), so that all copy CTAs move the same chunk at the same time.
  auto sub_for = [](int ncopy) {
    int S = 1;
    while (S * 2 <= std::min(ncopy, COPY_SUB_MAX)) S *= 2;
    return S;
  };
  if (k == 0 || n == 0) {
    // Nothing to multiply: C is all zeros (k == 0) or empty (n == 0); the
    // gathered A is still produced.
    if (n > 0) {
      mk_status st = zero_outputs(&c, 1, static_cast<size_t>(pl.M) * n * (c_dtype == MK_F32 ? 4 : 2), s);
      if (st != MK_OK) return st;
    }
    if (k == 0) return MK_OK;
    p.copy_sub = COPY_SUB_MAX;
    return launch(p, std::min(sms, std::max(1, p.n_copy_chunks * COPY_SUB_MAX)), 0, 0, s);
  }
  // CTA pairs for every compute-only launch (not with copy-role CTAs).
  const bool pair = use_pair(cfg, sms) && !(pl.mode == MK_MODE_FUSED && cfg && cfg->n_copy_ctas > 0);
  if (pl.fp8) {   // A shards / gathered A [rows x k] and B^T [n x k], all bytes
    if (!make_map_k8(&p.tmA[0], a_shards[local_rank], k, m_r, BM) ||
        !make_map_k8(&p.tmA[1], a_gathered, k, pl.M, BM) || !make_map_k8(&p.tmB[0], b, k, n, pair ? 128u : 256u))
      return MK_ERR_CUDA;
  } else if (!make_map_a(&p.tmA[0], a_shards[local_rank], k, m_r, row_bytes) ||
             !make_map_a(&p.tmA[1], a_gathered, k, pl.M, row_bytes) ||
             !(p.b_one_box ? make_map_b_chunks(&p.tmB[0], b, k, n, pair ? 2 : 4)
                           : make_map_2d(&p.tmB[0], b, n, k, static_cast<size_t>(n) * 2, 64, BK))) {
    return MK_ERR_CUDA;
  }
  if (pl.mode == MK_MODE_GEMM_ONLY) return launch_compute(p, pair, sms, s);
  if (pl.mode == MK_MODE_UNFUSED) {
    const uint32_t e = p.epoch;
    mk_status st = MK_OK;
    p.copy_sub = COPY_SUB_MAX;
    if (p.n_copy_chunks > 0) st = launch(p, std::min(sms, p.n_copy_chunks * COPY_SUB_MAX), 0, 0, s);
    if (st != MK_OK) return st;
    p.epoch = e;
    p.mode = MK_MODE_GEMM_ONLY;
    return launch_compute(p, pair, sms, s);
  }
  if (!(cfg && cfg->n_copy_ctas > 0)) {
    // Default: the copy-in is done by two spare warps of every compute CTA,
    // in pieces of about 16 KiB (rows of the gathered A), so every SM computes.
    int pr = 1;
    while (pr < BM && static_cast<long long>(pr) * row_bytes < MK_CW_PIECE_BYTES) pr *= 2;
    p.copy_warps = 1;
    p.copy_rows = pr;
    // two copy warps per CTA move the 7/8 of A in well under the GEMM's time;
    // more of them measured no faster and compete with the operand loads
    p.n_cw = std::min(MK_AG_COPY_WARPS, N_COPY_WARPS);
    return launch_compute(p, pair, sms, s);
  }
  int n_copy = cfg->n_copy_ctas;
  n_copy = std::min(n_copy, p.n_copy_chunks * COPY_SUB_MAX);
  n_copy = std::min(n_copy, sms - 1);
  n_copy = std::max(n_copy, 0);
  p.copy_sub = sub_for(std::max(1, n_copy));
  const int n_compute = std::min(sms - n_copy, n_items);
  return launch(p, n_copy, n_compute, 0, s);
}

static mk_status rs_ar_common(int op, const void* const* a, const void* const* b, void* const* outs,
                              mk_dtype c_dtype, int R, long long m, long long n, long long k,
                              void* workspace, size_t ws_bytes, const mk_config* cfg,
                              mk_stream_t stream) {
  if (!a || !b || !outs || !workspace) return MK_ERR_INVALID;
  if (c_dtype != MK_BF16 && c_dtype != MK_F32) return MK_ERR_INVALID;
  if (R < 1 || R > MK_MAX_RANKS) return MK_ERR_INVALID;
  if (m < 0 || n < 0 || k < 0) return MK_ERR_INVALID;
  const long long out_rows = (op == OP_RS) ? m / R : m;
  for (int r = 0; r < R; ++r) {
    if (!buf_ok(a[r], m * k) || !buf_ok(b[r], k * n) || !buf_ok(outs[r], out_rows * n))
      return MK_ERR_INVALID;
  }
  if (!aligned16(workspace)) return MK_ERR_INVALID;
  Plan pl;
  if (!plan_gemm(op, R, m, n, k, cfg, pl)) return MK_ERR_INVALID;
  if (ws_bytes < pl.total) return MK_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (m == 0 || n == 0) return MK_OK;
  const size_t esz = (c_dtype == MK_F32) ? 4 : 2;
  if (k == 0) {
    const size_t rows = (op == OP_RS) ? static_cast<size_t>(m / R) : static_cast<size_t>(m);
    return zero_outputs(outs, R, rows * n * esz, s);
  }
  const int sms = grid_cap(cfg);
  if (sms <= 0) return MK_ERR_UNSUPPORTED;

  FusedParams p;
  fill_common(p, pl, static_cast<uint8_t*>(workspace), cfg, c_dtype);
  p.rows_per_owner = static_cast<int>(m / R);
  if (op == OP_AR) p.rows_per_owner = static_cast<int>(m);
  p.b_one_box = (n % 64 == 0) ? 1 : 0;
  // CTA pairs for every compute-only launch (not with reduce-role CTAs).
  const bool pair = use_pair(cfg, sms) && (pl.mode != MK_MODE_FUSED || pl.chain || pl.last || pl.atomic) &&
                    !(pl.ar_single && !(cfg && cfg->cta_pair == 2));
  for (int r = 0; r < R; ++r) {
    p.out[r] = outs[r];
    if (pl.fp8) {   // A_r [m x k] and B_r^T [n x k], bytes
      if (!make_map_k8(&p.tmA[r], a[r], k, m, BM) || !make_map_k8(&p.tmB[r], b[r], k, n, pair ? 128u : 256u))
        return MK_ERR_CUDA;
    } else if (!make_map_a(&p.tmA[r], a[r], k, m, static_cast<size_t>(k) * 2) ||
               !(p.b_one_box ? make_map_b_chunks(&p.tmB[r], b[r], k, n, pair ? 2 : 4)
                             : make_map_2d(&p.tmB[r], b[r], n, k, static_cast<size_t>(n) * 2, 64, BK))) {
      return MK_ERR_CUDA;
    }
  }
  if (pl.mode == MK_MODE_GEMM_ONLY) return launch_compute(p, pair, sms, s);
  if (pl.mode == MK_MODE_UNFUSED) {
    const uint32_t e = p.epoch;
    mk_status st = launch_compute(p, pair, sms, s);
    if (st != MK_OK) return st;
    p.epoch = e;
    p.n_items = pl.n_tiles * pl.P;
    return launch(p, 0, 0, std::min(sms, pl.n_tiles), s);
  }
  if (pl.chain || pl.last || pl.atomic) return launch_compute(p, pair, sms, s);
  p.n_items = pl.n_tiles * pl.P;
  int n_red = cfg->n_reduce_ctas;
  n_red = std::min(n_red, pl.n_tiles);
  n_red = std::min(n_red, sms - 1);
  n_red = std::max(n_red, 1);
  const int n_compute = std::min(sms - n_red, p.n_items);
  return launch(p, 0, n_compute, n_red, s);
}

mk_status mk_gemm_rs(const void* const* a, const void* const* b, void* const* c_blocks, mk_dtype c_dtype,
                     int R, long long m, long long n, long long k, void* workspace, size_t ws_bytes,
                     const mk_config* cfg, mk_stream_t stream) {
  return rs_ar_common(OP_RS, a, b, c_blocks, c_dtype, R, m, n, k, workspace, ws_bytes, cfg, stream);
}

mk_status mk_gemm_ar(const void* const* a, const void* const* b, void* const* c_replicas,
                     mk_dtype c_dtype, int R, long long m, long long n, long long k, void* workspace,
                     size_t ws_bytes, const mk_config* cfg, mk_stream_t stream) {
  return rs_ar_common(OP_AR, a, b, c_replicas, c_dtype, R, m, n, k, workspace, ws_bytes, cfg, stream);
}

}  // extern "C"

namespace mk {
namespace {

// Workspace of the chained MLP: header | AG chunk counters | H_r row-block
// counters | the down-projection's GEMM+ReduceScatter flags and staging.
struct MlpLayout {
  Plan pl;
  size_t chunk_off, cnt_off, flags_off, staging_off, total;
  size_t trace_off, trace_n;   // in-kernel trace records at the end (cfg->trace = 1), or none
};

bool mlp_plan(int R, long long m, long long h, long long f_r, const mk_config* cfg, MlpLayout& L) {
  if (R < 1 || R > MK_MLP_MAX_RANKS || m < 0 || h < 0 || f_r < 0) return false;
  if ((h % 8) || (f_r % 8)) return false;
  if (cfg && (cfg->reduce >= 2 || cfg->wire != 0 || cfg->operand != 0 || cfg->trace < 0 || cfg->trace > 1 ||
              cfg->n_reduce_ctas > 0 || cfg->split_k > 1))
    return false;
  // the trace covers one launch: the fused call or its GEMM-only baseline
  if (cfg && cfg->trace && cfg->mode == MK_MODE_UNFUSED) return false;
  if (!plan_gemm(OP_RS, R, static_cast<long long>(R) * m, h, f_r, cfg, L.pl)) return false;
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t off = WS_HDR_BYTES;
  L.chunk_off = off;  off = al(off + static_cast<size_t>(L.pl.n_mblk) * COPY_SUB_MAX * 4);
  L.cnt_off = off;    off = al(off + static_cast<size_t>(R) * L.pl.n_mblk * 4);
  L.flags_off = off;  off = off + L.pl.n_flags * 4;
  off = (off + 1023) & ~static_cast<size_t>(1023);
  L.staging_off = off;
  L.total = off + L.pl.staging_bytes;
  L.trace_off = 0;
  L.trace_n = 0;
  if (cfg && cfg->trace) {
    // two records (the CTAs of a pair) per item, items counted for single CTAs
    // (the larger count): up-projection tiles of every rank, then down-projection
    // (tile, rank) parts
    const long long nb1 = ceil_div_ll(f_r, BN);
    const long long items = static_cast<long long>(L.pl.n_mblk) * R * nb1 +
                            static_cast<long long>(L.pl.n_mblk) * L.pl.n_nblk * R;
    L.trace_n = static_cast<size_t>(std::max(items, 1LL)) * 2;
    L.trace_off = al(L.total);
    L.total = L.trace_off + (L.trace_n + MK_TRACE_COPY_RECORDS) * 64;
  }
  return true;
}

}  // namespace
}  // namespace mk

extern "C" {

size_t mk_mlp_workspace_size(int R, long long m, long long h, long long f_r, const mk_config* cfg) {
  MlpLayout L;
  if (!mlp_plan(R, m, h, f_r, cfg, L)) return 0;
  return L.total;
}

size_t mk_mlp_trace_entries(int R, long long m, long long h, long long f_r, const mk_config* cfg,
                            size_t* offset) {
  if (offset) *offset = 0;
  MlpLayout L;
  if (!mlp_plan(R, m, h, f_r, cfg, L)) return 0;
  if (offset) *offset = L.trace_off;
  return L.trace_n;
}

mk_status mk_mlp_ag_rs(const void* const* x_shards, const void* const* w1, const void* const* w2, int R,
                       long long m, long long h, long long f_r, void* x_gathered, void* const* hid,
                       void* const* y_blocks, void* workspace, size_t ws_bytes, const mk_config* cfg,
                       mk_stream_t stream) {
  if (!x_shards || !w1 || !w2 || !hid || !y_blocks || !workspace) return MK_ERR_INVALID;
  MlpLayout L;
  if (!mlp_plan(R, m, h, f_r, cfg, L)) return MK_ERR_INVALID;
  if (ws_bytes < L.total || !aligned16(workspace)) return MK_ERR_INVALID;
  const long long M = static_cast<long long>(R) * m;
  for (int r = 0; r < R; ++r) {
    if (!buf_ok(x_shards[r], m * h) || !buf_ok(w1[r], h * f_r) || !buf_ok(w2[r], f_r * h) ||
        !buf_ok(hid[r], M * f_r) || !buf_ok(y_blocks[r], m * h))
      return MK_ERR_INVALID;
  }
  if (!buf_ok(x_gathered, M * h)) return MK_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (m == 0 || h == 0) return MK_OK;
  if (f_r == 0) {   // no hidden units: every output is zero, the gathered input is still produced
    mk_status st = zero_outputs(y_blocks, R, static_cast<size_t>(m) * h * 2, s);
    if (st != MK_OK) return st;
    for (int r = 0; r < R; ++r)
      if (cudaMemcpyAsync(static_cast<uint8_t*>(x_gathered) + static_cast<size_t>(r) * m * h * 2, x_shards[r],
                          static_cast<size_t>(m) * h * 2, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MK_ERR_CUDA;
    return MK_OK;
  }
  const int sms = grid_cap(cfg);
  if (sms <= 0) return MK_ERR_UNSUPPORTED;
  const Plan& pl = L.pl;
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  FusedParams p;
  fill_common(p, pl, ws, cfg, MK_BF16);
  p.op = OP_MLP;
  p.trace = L.trace_n ? reinterpret_cast<unsigned long long*>(ws + L.trace_off) : nullptr;
  p.trace_cap = static_cast<int>(L.trace_n);
  p.flags = reinterpret_cast<uint32_t*>(ws + L.flags_off);
  p.staging = reinterpret_cast<float*>(ws + L.staging_off);
  p.chunk_cnt = reinterpret_cast<uint32_t*>(ws + L.chunk_off);
  p.mlp_cnt = reinterpret_cast<uint32_t*>(ws + L.cnt_off);
  p.K = static_cast<int>(h);      // gathered row width (copy-in)
  p.N = static_cast<int>(h);      // down-projection output width
  p.m_r = static_cast<int>(m);
  p.rows_per_owner = static_cast<int>(m);
  p.mlp_f = static_cast<int>(f_r);
  p.mlp_nb1 = static_cast<int>(ceil_div_ll(f_r, BN));
  p.mlp_kb1 = static_cast<int>(ceil_div_ll(h, BK));
  p.mlp_wait = 1;
  p.gathered = static_cast<uint8_t*>(x_gathered);
  p.copy_local = 1;
  p.ordered = 0;
  p.n_copy_chunks = pl.n_mblk;
  for (int r = 0; r < R; ++r) {
    p.shard[r] = static_cast<const uint8_t*>(x_shards[r]);
    p.out[r] = y_blocks[r];
    p.mlp_hid[r] = static_cast<uint8_t*>(hid[r]);
  }
  const bool pair = use_pair(cfg, sms);
  p.b_one_box = (h % 64 == 0 && f_r % 64 == 0) ? 1 : 0;
  const uint32_t chunks = pair ? 2 : 4;
  if (!make_map_a(&p.tmA[0], x_gathered, h, M, static_cast<size_t>(h) * 2)) return MK_ERR_CUDA;
  for (int r = 0; r < R; ++r) {
    if (!make_map_a(&p.tmA[1 + r], hid[r], f_r, M, static_cast<size_t>(f_r) * 2)) return MK_ERR_CUDA;
    const bool ok1 = p.b_one_box ? make_map_b_chunks(&p.tmB[r], w1[r], h, f_r, chunks)
                                 : make_map_2d(&p.tmB[r], w1[r], f_r, h, static_cast<size_t>(f_r) * 2, 64, BK);
    const bool ok2 = p.b_one_box ? make_map_b_chunks(&p.tmB[R + r], w2[r], f_r, h, chunks)
                                 : make_map_2d(&p.tmB[R + r], w2[r], h, f_r, static_cast<size_t>(h) * 2, 64, BK);
    if (!ok1 || !ok2) return MK_ERR_CUDA;
  }
  int pr = 1;
  while (pr < BM && static_cast<long long>(pr) * h * 2 < MK_CW_PIECE_BYTES) pr *= 2;
  p.copy_rows = pr;
  p.n_cw = std::min(2, N_COPY_WARPS);

  if (pl.mode == MK_MODE_FUSED) {
    p.copy_warps = 1;
    return launch_compute(p, pair, sms, s, 3);
  }
  if (pl.mode == MK_MODE_GEMM_ONLY) {   // x_gathered as already filled; ranks summed in TMEM
    return launch_compute(p, pair, sms, s, 3);
  }
  // Unfused, host-ordered: copy-in launch, up-projection launch, then the
  // down-projection as partial tiles and a reduce launch.
  const uint32_t e = p.epoch;
  p.copy_sub = COPY_SUB_MAX;
  uint32_t* chain_flags = p.flags;
  p.flags = p.chunk_cnt;          // copy-role sub-chunk flags
  mk_status st = launch(p, std::min(sms, std::max(1, p.n_copy_chunks * COPY_SUB_MAX)), 0, 0, s);
  if (st != MK_OK) return st;
  p.flags = chain_flags;
  p.epoch = e;
  p.mode = MK_MODE_GEMM_ONLY;
  st = launch_compute(p, pair, sms, s, 1);
  if (st != MK_OK) return st;
  p.epoch = e;
  p.mode = MK_MODE_UNFUSED;
  p.mlp_wait = 0;                  // the hidden activations are complete
  st = launch_compute(p, pair, sms, s, 2);
  if (st != MK_OK) return st;
  p.epoch = e;
  p.mlp_n1 = 0;
  p.n_items = pl.n_tiles * pl.P;
  return launch(p, 0, 0, std::min(sms, pl.n_tiles), s);
}

}  // extern "C"
