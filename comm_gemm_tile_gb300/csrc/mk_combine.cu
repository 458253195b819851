// mk_combine.cu -- MoE combine, the return direction of the MoE row of the
// five-kernel table (mKernel write-up, news.chathome.org, "五种融合内核",
// row "MoE Dispatch + GEMM"): the down-projection of every expert's rows, the
// return of each product row to its token's source rank, and the gate-weighted
// sum over the token's top-k rows.
//
// Launch sequence on the caller's stream:
//   1. combine_plan_kernel (1 CTA): expert row totals from the dispatch counts,
//      each rank's expert segments, the capacity check, the tile-table prefix;
//   2. combine_tiles_kernel: the grouped-GEMM tile table and zeroed per-(token,
//      column block) slot counters;
//   3. the persistent fused kernel (op OP_MOE_COMBINE): tiles of each expert's
//      rows times its W2 slice; the epilogue returns the bf16 rows and the
//      last-arriving slot of a token forms the weighted sum (see
//      combine_epilogue in mk_fused.cu);
//   4. unfused baseline only: combine_sum_kernel after a GEMM-only launch.
#include <algorithm>
#include <cstring>

#include "mk_internal.h"
#include "mk_ptx.cuh"

namespace mk {

namespace {

enum { CMISC_NTILES = 0, CMISC_OK = 1, CMISC_WORDS = 64 };

struct CombineArgs {
  const int* counts;  // [R x E] rows of source rank r routed to expert e
  int* totals;        // [E]
  int* segoff;        // [R x (E_loc+1)] first row of each local expert's segment
  int* tprefix;       // [E + 1] tile-table prefix per (rank, local expert)
  int* tiles;         // [max_tiles x 5]
  uint32_t* misc;     // CMISC_* words
  uint32_t* cnt;      // [R*T x n_nblk] slot counters
  uint32_t* hdr;      // workspace header (status)
  int R, E_loc, E, T, n_nblk, tile_rows;
  long long cap;
};

// One CTA: expert totals, segment offsets, the capacity check and the
// tile-table prefix, with the small tables in shared memory and the prefixes
// taken by warp scans.
__global__ void __launch_bounds__(256) combine_plan_kernel(const __grid_constant__ CombineArgs a) {
  griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R, El = a.E_loc, E = a.E;
  __shared__ int s_tot[MOE_MAX_E];
  __shared__ int s_ok;
  if (tid == 0) s_ok = 1;
  for (int e = tid; e < E; e += 256) {
    int acc = 0;
    for (int r = 0; r < R; ++r) acc += a.counts[r * E + e];
    s_tot[e] = acc;
    a.totals[e] = acc;
  }
  __syncthreads();
  for (int d = warp; d < R; d += 256 / 32) {   // warp d: destination d's segments
    int* seg = a.segoff + d * (El + 1);
    const int tot = warp_exclusive_scan(
        El, [&](int l) { return s_tot[d * El + l]; }, [&](int l, int pre) { seg[l] = pre; });
    if (lane == 0) {
      seg[El] = tot;
      if (tot > a.cap) atomicExch(&s_ok, 0);
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int ok = s_ok;
    const int tr = a.tile_rows, nn = a.n_nblk;
    const int acc = warp_exclusive_scan(
        E, [&](int k) { return ok ? ((s_tot[k] + tr - 1) / tr) * nn : 0; },
        [&](int k, int pre) { a.tprefix[k] = pre; });
    if (lane == 0) {
      a.tprefix[E] = acc;
      a.misc[CMISC_NTILES] = static_cast<uint32_t>(acc);
      a.misc[CMISC_OK] = static_cast<uint32_t>(ok);
      if (!ok) atomicCAS(reinterpret_cast<int*>(&a.hdr[HDR_STATUS]), 0, MK_ERR_CAPACITY);
    }
  }
}

__global__ void __launch_bounds__(256) combine_tiles_kernel(const __grid_constant__ CombineArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long first = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long ncnt = static_cast<long long>(a.R) * a.T * a.n_nblk;
  for (long long q = first; q < ncnt; q += stride) a.cnt[q] = 0u;
  const int El = a.E_loc;
  const int ntiles = static_cast<int>(a.misc[CMISC_NTILES]);
  for (long long q = first; q < ntiles; q += stride) {
    int lo = 0, hi = a.E - 1;  // last k with tprefix[k] <= q
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (a.tprefix[mid] <= q) lo = mid;
      else hi = mid - 1;
    }
    const int k = lo;
    const int d = k / El, l = k - d * El;
    const int qq = static_cast<int>(q) - a.tprefix[k];
    const int mi = qq / a.n_nblk, nb = qq - mi * a.n_nblk;
    int* ent = a.tiles + 5 * q;
    ent[0] = d;
    ent[1] = l;
    ent[2] = a.segoff[d * (El + 1) + l] + mi * a.tile_rows;
    ent[3] = min(a.tile_rows, a.totals[k] - mi * a.tile_rows);
    ent[4] = nb;
  }
}

struct SumArgs {
  const uint8_t* ret[MK_MAX_RANKS];
  const float* gates[MK_MAX_RANKS];
  uint8_t* out[MK_MAX_RANKS];
  const uint32_t* ok;
  int R, T, topk, H;
};

// Unfused baseline: out[r][t] = sum_k gates[r][t][k] * ret[r][t][k], one thread per
// 8 columns of a token row (the same fp32 fused multiply-adds in slot order as
// the fused epilogue).
__global__ void __launch_bounds__(256) combine_sum_kernel(const __grid_constant__ SumArgs a) {
  if (*a.ok == 0u) return;
  const int g8 = a.H / 8;
  const long long n = static_cast<long long>(a.R) * a.T * g8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < n; u += stride) {
    const int c = static_cast<int>(u % g8);
    const long long rt = u / g8;
    const int r = static_cast<int>(rt / a.T), t = static_cast<int>(rt - static_cast<long long>(r) * a.T);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int q = 0; q < a.topk; ++q) {
      const float gq = a.gates[r][static_cast<size_t>(t) * a.topk + q];
      const uint4 w = ld_nc_v4(a.ret[r] + ((static_cast<size_t>(t) * a.topk + q) * a.H + 8 * c) * 2);
      const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(gq, __uint_as_float(w4[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(gq, __uint_as_float(w4[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
    st_global_v4(a.out[r] + (static_cast<size_t>(t) * a.H + 8 * c) * 2, pack_bf16x2(acc[0], acc[1]),
                 pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

struct CombineLayout {
  size_t misc_off, totals_off, segoff_off, tprefix_off, tiles_off, cnt_off, total;
  int n_nblk, max_tiles;
};

bool combine_layout(int R, int E_loc, int topk, long long T, long long N, long long H, long long cap,
                    CombineLayout& L) {
  if (R < 1 || R > MK_MAX_RANKS || E_loc < 1) return false;
  const long long E = static_cast<long long>(R) * E_loc;
  if (E > MOE_MAX_E || topk < 1 || topk > MOE_MAX_TOPK || topk > E) return false;
  if (T < 0 || N < 0 || H < 0 || cap < 0) return false;
  if ((N % 8) || (H % 8)) return false;
  const long long rows = static_cast<long long>(R) * T * topk;
  if (rows >= (1LL << 31) || cap >= (1LL << 31) || N >= (1LL << 31) || H >= (1LL << 31)) return false;
  if (cap * N >= (1LL << 40) || T * topk * H >= (1LL << 40)) return false;
  L.n_nblk = static_cast<int>(ceil_div_ll(H, BN));
  const long long max_tiles = (rows / BM + E) * L.n_nblk;
  if (max_tiles >= (1LL << 30)) return false;
  L.max_tiles = static_cast<int>(max_tiles);
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t off = WS_HDR_BYTES;
  L.misc_off = off;    off = al(off + CMISC_WORDS * 4);
  L.totals_off = off;  off = al(off + static_cast<size_t>(E) * 4);
  L.segoff_off = off;  off = al(off + static_cast<size_t>(R) * (E_loc + 1) * 4);
  L.tprefix_off = off; off = al(off + (static_cast<size_t>(E) + 1) * 4);
  L.tiles_off = off;   off = al(off + static_cast<size_t>(L.max_tiles) * 5 * 4);
  L.cnt_off = off;     off = al(off + static_cast<size_t>(R) * T * L.n_nblk * 4);
  L.total = off;
  return true;
}

inline bool okp(const void* p, long long elems, unsigned align) {
  if (elems > 0 && !p) return false;
  return (reinterpret_cast<uintptr_t>(p) & (align - 1)) == 0;
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" {

size_t mk_moe_combine_workspace_size(int R, int E_loc, int topk, long long T, long long N, long long H,
                                     long long cap_rows, const mk_config* cfg) {
  (void)cfg;
  CombineLayout L;
  if (!combine_layout(R, E_loc, topk, T, N, H, cap_rows, L)) return 0;
  return L.total;
}

mk_status mk_moe_combine(const void* const* h, const void* const* w2, const float* const* gates,
                         const int* const* recv_src, const int* counts, int R, int E_loc, int topk,
                         long long T, long long N, long long H, long long cap_rows, void* const* ret,
                         void* const* out, void* workspace, size_t ws_bytes, const mk_config* cfg,
                         mk_stream_t stream) {
  if (!h || !w2 || !gates || !recv_src || !ret || !out || !workspace) return MK_ERR_INVALID;
  CombineLayout L;
  if (!combine_layout(R, E_loc, topk, T, N, H, cap_rows, L)) return MK_ERR_INVALID;
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 15u)) return MK_ERR_INVALID;
  const int mode = cfg ? cfg->mode : MK_MODE_FUSED;
  if (mode < MK_MODE_FUSED || mode > MK_MODE_UNFUSED) return MK_ERR_INVALID;
  if (cfg && cfg->operand != 0) return MK_ERR_INVALID;   // bf16 operands only
  const long long E = static_cast<long long>(R) * E_loc;
  if (!okp(counts, R * E, 4)) return MK_ERR_INVALID;
  for (int r = 0; r < R; ++r) {
    if (!okp(h[r], cap_rows * N, 16) || !okp(w2[r], E_loc * N * H, 16) || !okp(gates[r], T * topk, 4) ||
        !okp(recv_src[r], cap_rows, 4) || !okp(ret[r], T * topk * H, 16) || !okp(out[r], T * H, 16))
      return MK_ERR_INVALID;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0 || H == 0) return MK_OK;
  if (N == 0) {
    // empty contraction: every returned row and every sum is zero
    for (int r = 0; r < R; ++r) {
      if (cudaMemsetAsync(ret[r], 0, static_cast<size_t>(T) * topk * H * 2, s) != cudaSuccess) return MK_ERR_CUDA;
      if (mode != MK_MODE_GEMM_ONLY &&
          cudaMemsetAsync(out[r], 0, static_cast<size_t>(T) * H * 2, s) != cudaSuccess)
        return MK_ERR_CUDA;
    }
    return MK_OK;
  }
  const int sms = grid_cap(cfg);
  if (sms <= 0) return MK_ERR_UNSUPPORTED;
  const bool pair = use_pair(cfg, sms);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CombineArgs a;
  std::memset(&a, 0, sizeof(a));
  a.counts = counts;
  a.totals = reinterpret_cast<int*>(ws + L.totals_off);
  a.segoff = reinterpret_cast<int*>(ws + L.segoff_off);
  a.tprefix = reinterpret_cast<int*>(ws + L.tprefix_off);
  a.tiles = reinterpret_cast<int*>(ws + L.tiles_off);
  a.misc = reinterpret_cast<uint32_t*>(ws + L.misc_off);
  a.cnt = reinterpret_cast<uint32_t*>(ws + L.cnt_off);
  a.hdr = reinterpret_cast<uint32_t*>(ws);
  a.R = R;
  a.E_loc = E_loc;
  a.E = static_cast<int>(E);
  a.T = static_cast<int>(T);
  a.n_nblk = L.n_nblk;
  a.tile_rows = pair ? 2 * BM : BM;
  a.cap = cap_rows;
  combine_plan_kernel<<<1, 256, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return MK_ERR_CUDA;
  const long long work = std::max(static_cast<long long>(R) * T * L.n_nblk, static_cast<long long>(L.max_tiles));
  const int tgrid = static_cast<int>(std::min<long long>(ceil_div_ll(work, 256), 4LL * device_sm_count()));
  // the tile kernel and the fused kernel launch as programmatic dependents of
  // the launch before them (each waits for its predecessor's results)
  if (launch_dependent(combine_tiles_kernel, dim3(std::max(1, tgrid)), dim3(256), s, a) != cudaSuccess)
    return MK_ERR_CUDA;

  FusedParams p;
  std::memset(&p, 0, sizeof(p));
  p.op = OP_MOE_COMBINE;
  p.mode = (mode == MK_MODE_FUSED) ? MK_MODE_FUSED : MK_MODE_GEMM_ONLY;
  p.R = R;
  p.M = static_cast<int>(cap_rows);
  p.N = static_cast<int>(H);
  p.K = static_cast<int>(N);
  p.n_nblk = L.n_nblk;
  p.n_kblk = static_cast<int>(ceil_div_ll(N, BK));
  p.n_mblk = 1;
  p.group_m = 1;
  p.split_k = 1;
  p.P = 1;
  p.n_items = L.max_tiles;
  p.moe_tiles = a.tiles;
  p.moe_ntiles = reinterpret_cast<const int*>(a.misc + CMISC_NTILES);
  p.moe_ok = reinterpret_cast<const int*>(a.misc + CMISC_OK);
  p.moe_T = static_cast<int>(T);
  p.moe_topk = topk;
  p.moe_cnt = a.cnt;
  p.b_one_box = (H % 64 == 0) ? 1 : 0;
  p.hdr = a.hdr;
  p.pdl = 1;
  p.wait_ns = default_wait_ns(cfg);
  p.inject = cfg ? cfg->inject : 0;
  p.epoch = next_epoch();
  for (int r = 0; r < R; ++r) {
    p.moe_src[r] = recv_src[r];
    p.out[r] = out[r];
    p.moe_ret[r] = static_cast<uint8_t*>(ret[r]);
    p.moe_gates[r] = gates[r];
    if (!make_map_a(&p.tmA[r], h[r], N, cap_rows, static_cast<size_t>(N) * 2) ||
        !(p.b_one_box ? make_map_w_chunks(&p.tmB[r], w2[r], N, H, E_loc, pair ? 2 : 4)
                      : make_map_3d(&p.tmB[r], w2[r], H, N, E_loc, static_cast<size_t>(H) * 2,
                                    static_cast<size_t>(N) * H * 2, 64, BK, 1)))
      return MK_ERR_CUDA;
  }
  int grid;
  if (pair) {
    const int n_pairs = std::max(1, std::min(std::min(max_pair_clusters(), sms / 2), L.max_tiles));
    p.pair = 1;
    p.n_compute = n_pairs;
    grid = 2 * n_pairs;
  } else {
    grid = std::max(1, std::min(sms, L.max_tiles));
    p.n_compute = grid;
  }
  if (launch_fused(p, grid, s) != cudaSuccess) return MK_ERR_CUDA;
  if (mode != MK_MODE_UNFUSED) return MK_OK;
  SumArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  for (int r = 0; r < R; ++r) {
    sa.ret[r] = static_cast<const uint8_t*>(ret[r]);
    sa.gates[r] = gates[r];
    sa.out[r] = static_cast<uint8_t*>(out[r]);
  }
  sa.ok = a.misc + CMISC_OK;
  sa.R = R;
  sa.T = static_cast<int>(T);
  sa.topk = topk;
  sa.H = static_cast<int>(H);
  const long long units = static_cast<long long>(R) * T * (H / 8);
  const int sgrid = static_cast<int>(std::min<long long>(ceil_div_ll(units, 256), 8LL * device_sm_count()));
  combine_sum_kernel<<<std::max(1, sgrid), 256, 0, s>>>(sa);
  return cudaGetLastError() == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

}  // extern "C"
