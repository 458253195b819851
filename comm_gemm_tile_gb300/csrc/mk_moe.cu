// mk_moe.cu -- MoE Dispatch + grouped GEMM (mKernel write-up,
// news.chathome.org, "五种融合内核" table, row "MoE Dispatch + GEMM": route
// tokens to their expert ranks, all-to-all dispatch, per-expert grouped GEMM,
// tokens processed on arrival).
//
// Four launches on the caller's stream:
//   1. route + rank (one CTA per chunk of 128 tokens of a source rank, one
//      thread per token): top-k
//      experts of every token, and for every (token, slot) its position among
//      the chunk's rows routed to the same expert (a stable block-level
//      multisplit), plus the chunk's per-expert counts;
//   2. offsets (one CTA): chunk prefixes and counts[r][e], expert totals,
//      per-destination segment offsets,
//      per-(rank, expert) bases, received-row counts, the capacity check, the
//      tile-table prefix, and zeroed per-block arrival counters;
//   3. scatter: recv_src (the destination-ordered inverse map) and the
//      grouped-GEMM tile table;
//   4. the persistent fused kernel: copy warps move token rows into recv_x in
//      destination order and count them per 128-row block; compute CTAs run
//      the tiles of each expert as soon as their blocks are complete.
// Launches 2-4 are programmatic dependents of the launch before them: each
// starts while its predecessor finishes and waits (griddepcontrol.wait) for
// its results before it reads them.
// Row order inside a destination rank d: local expert, then global token
// g = r*T + t; every (token, slot) pair is one row.
#include <algorithm>
#include <cstring>

#include "mk_internal.h"
#include "mk_ptx.cuh"

#ifndef MK_MOE_BOOST_WAVES
#define MK_MOE_BOOST_WAVES 2   // waves of tiles whose rows all copy warps move first
#endif
#ifndef MK_MOE_COPY_WARPS
#define MK_MOE_COPY_WARPS 3   // copy warps per compute CTA for the fused MoE dispatch
#endif

namespace mk {

namespace {

constexpr int RR_TOKENS = 128;                 // tokens per route/rank CTA, one thread each
constexpr int RR_THREADS = RR_TOKENS;
constexpr int RR_WARPS = RR_THREADS / 32;
constexpr int RR_COLS = 64;                    // experts staged in shared memory at a time
constexpr int RR_PITCH = RR_COLS + 1;          // padded row of the staged logits
constexpr int OF_THREADS = 1024;               // the offsets kernel's CTA
constexpr int OF_BATCH = 16;                   // chunk counts a thread loads at once
enum { MISC_NTILES = 0, MISC_OK = 1, MISC_RBASE = 16, MISC_WORDS = 64 };   // RBASE: R words
static_assert(MISC_RBASE + MK_MAX_RANKS <= MISC_WORDS, "misc words");

struct MoeArgs {
  const float* logits[MK_MAX_RANKS];
  int* recv_src[MK_MAX_RANKS];
  int* topk_idx;      // [R*T x topk]
  int* counts;        // [R x E]
  int* recv_counts;   // [R]
  int* pos;           // [R*T*topk] position among the chunk's rows of the same expert
  int* fwd;           // [R*T*topk] position of each (token, slot) row in the dispatch order
  int* hist;          // [R x C x E] per-chunk expert counts, turned into chunk prefixes
  int* base;          // [R x E]  rows of expert e from ranks before r
  int* totals;        // [E]
  int* segoff;        // [R x (E_loc+1)]
  int* tprefix;       // [R*E_loc + 1] tile-table prefix per (rank, local expert)
  int* tiles;         // [max_tiles x 5]
  uint32_t* misc;     // MISC_* words
  uint32_t* blocks;   // [R x nblk] arrival counters
  uint32_t* hdr;      // workspace header (status)
  int R, E_loc, E, topk, T, n_nblk, nblk, C;
  int tile_rows;      // rows per tile-table entry: 128, or 256 for CTA pairs
  long long cap;
};

#if MK_DEBUG_BOUNDS
// Bounds-checking build: a failed check records MK_ERR_INVALID with its detail
// (the first failure wins) and the caller skips the access.
__device__ __noinline__ void bounds_fail(const MoeArgs& a, int code, long long index) {
  int* st = reinterpret_cast<int*>(&a.hdr[HDR_STATUS]);
  if (atomicCAS(st, 0, MK_ERR_INVALID) == 0)
    atomicExch(reinterpret_cast<int*>(&a.hdr[HDR_DETAIL]),
               WHERE_BOUNDS * 1000000 + code * 10000 + static_cast<int>(index % 10000));
}
#endif

// Grid (C chunks, R ranks): CTA (c, r) routes tokens [c*RR_TOKENS, ...) of
// rank r, one thread per token, and ranks their (token, slot) pairs per expert
// inside the chunk.  The chunk's logits pass through shared memory in blocks
// of RR_COLS experts: copied row-contiguously (coalesced, all copies of a
// block in flight together by cp.async), then read by row
// (one token per thread; the padded pitch keeps the column reads conflict
// free).  A thread keeps its token's best KMAX (>= topk) experts as a list
// sorted by (logit descending, expert id ascending), branch free.
template <int KMAX>
__global__ void __launch_bounds__(RR_THREADS) moe_route_rank_kernel(const __grid_constant__ MoeArgs a) {
  griddep_launch_dependents();
  const int c = blockIdx.x, r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, T = a.T, K = a.topk;
  const int t0 = c * RR_TOKENS, t1 = min(T, t0 + RR_TOKENS), nt = t1 - t0;
  const float* lg = a.logits[r] + static_cast<size_t>(t0) * E;
  int* idx = a.topk_idx + static_cast<size_t>(r) * T * K;
  __shared__ float s_lg[RR_TOKENS * RR_PITCH];
  __shared__ int s_idx[RR_TOKENS * MOE_MAX_TOPK];
  __shared__ int wcnt[RR_WARPS * MOE_MAX_E];
  __shared__ int run[MOE_MAX_E];
  // ---- top-k per token.  Key of (logit v, expert e): the order-preserving
  // bits of v (-0 made +0, so that it ties with +0) above ~e, so that a larger
  // key is a larger logit or, on a tie, the lower expert id; 0 = empty.
  unsigned long long best[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) best[j] = 0ull;
  for (int e0 = 0; e0 < E; e0 += RR_COLS) {
    const int w = min(RR_COLS, E - e0);
    if (e0 > 0) __syncthreads();   // the previous block has been read
    {   // every copy of the block in flight at once
      const int ee = tid % RR_COLS;
      if (ee < w) {
        for (int tt = tid / RR_COLS; tt < nt; tt += RR_THREADS / RR_COLS)
          cp_async_4(smem_u32(&s_lg[tt * RR_PITCH + ee]), lg + static_cast<size_t>(tt) * E + e0 + ee);
      }
      cp_async_wait_all();
    }
    __syncthreads();
    if (tid < nt) {
#pragma unroll 8
      for (int ee = 0; ee < w; ++ee) {
        const float v = s_lg[tid * RR_PITCH + ee];
        const uint32_t b = __float_as_uint(v);
        const uint32_t u = (b << 1) == 0u ? 0u : b;   // -0 -> +0
        const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
        unsigned long long key = (static_cast<unsigned long long>(ord) << 32) | ~static_cast<uint32_t>(e0 + ee);
        // insert into the descending list: each slot keeps the larger key and
        // passes the smaller one on
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          const unsigned long long hi = key > best[j] ? key : best[j];
          key = key > best[j] ? best[j] : key;
          best[j] = hi;
        }
      }
    }
  }
  if (tid < nt) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K) {
        const int be = static_cast<int>(~static_cast<uint32_t>(best[j]));
        idx[static_cast<size_t>(t0 + tid) * K + j] = be;
        s_idx[tid * K + j] = be;
      }
  }
  for (int e = tid; e < E; e += RR_THREADS) run[e] = 0;
  __syncthreads();
  // ---- stable multisplit of the chunk's (token, slot) list by expert
  const int n = nt * K;
  const uint32_t lt = (1u << lane) - 1u;
  for (int b0 = 0; b0 < n; b0 += RR_THREADS) {
    for (int x = tid; x < RR_WARPS * E; x += RR_THREADS) wcnt[x] = 0;
    __syncthreads();
    const int ai = b0 + tid;
    const int e = (ai < n) ? s_idx[ai] : -1 - lane;   // distinct sentinels never group
    const uint32_t mask = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(mask & lt);
    if (ai < n && (__ffs(mask) - 1) == lane) wcnt[warp * E + e] = __popc(mask);
    __syncthreads();
    for (int ee = tid; ee < E; ee += RR_THREADS) {
      int acc = run[ee];
      for (int w = 0; w < RR_WARPS; ++w) {
        const int cnt = wcnt[w * E + ee];
        wcnt[w * E + ee] = acc;
        acc += cnt;
      }
      run[ee] = acc;
    }
    __syncthreads();
    if (ai < n) a.pos[static_cast<size_t>(r) * T * K + static_cast<size_t>(t0) * K + ai] = wcnt[warp * E + e] + rank_w;
    __syncthreads();
  }
  for (int e = tid; e < E; e += RR_THREADS)
    a.hist[(static_cast<size_t>(r) * a.C + c) * E + e] = run[e];
}

// One CTA.  Step 1: for every (rank r, expert e), the exclusive prefix of the
// chunk counts hist[r][c][e] over the chunks c (in place) and counts[r][e].
// A team of G threads shares a pair (G a power of two, G*R*E <= OF_THREADS):
// member m takes the m-th run of consecutive chunks, and consecutive threads
// take consecutive experts, so each load of a warp is one coalesced request and
// a thread has a whole batch of loads in flight.  Step 2 works in shared
// memory: expert totals, per-(rank, expert) bases, per-destination segment
// offsets, received-row counts, the capacity check and the tile-table prefix.
__global__ void __launch_bounds__(OF_THREADS) moe_offsets_kernel(const __grid_constant__ MoeArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int s_cnt[MK_MAX_RANKS * MOE_MAX_E];
  __shared__ int s_part[OF_THREADS];
  __shared__ int s_tot[MOE_MAX_E];
  __shared__ int s_rc[MK_MAX_RANKS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R, E = a.E, El = a.E_loc, C = a.C;
  const int P = R * E;
  int G = 1;
  while (2 * G * P <= OF_THREADS) G *= 2;
  const int span = (C + G - 1) / G;
  for (int x0 = 0; x0 < P * G; x0 += OF_THREADS) {   // more than one round only when G = 1
    const int x = x0 + tid;
    const bool act = x < P * G;
    const int pr = act ? x % P : 0, m = act ? x / P : 0;
    const int rr = pr / E, e = pr - rr * E;
    int* h = a.hist + static_cast<size_t>(rr) * C * E + e;
    const int c_lo = min(C, m * span), c_hi = act ? min(C, c_lo + span) : c_lo;
    int v[OF_BATCH];
    int sum = 0;
    for (int cb = c_lo; cb < c_hi; cb += OF_BATCH) {
#pragma unroll
      for (int u = 0; u < OF_BATCH; ++u) v[u] = (cb + u < c_hi) ? h[static_cast<size_t>(cb + u) * E] : 0;
#pragma unroll
      for (int u = 0; u < OF_BATCH; ++u) sum += v[u];
    }
    s_part[tid] = sum;
    __syncthreads();
    int acc = 0;   // the team's earlier members (G >= 2 means a single round, x0 = 0)
    for (int q = 0; q < m; ++q) acc += s_part[pr + q * P];
    if (act && m == G - 1) s_cnt[pr] = acc + sum;
    if (c_hi - c_lo <= OF_BATCH) {   // the run is still in registers
#pragma unroll
      for (int u = 0; u < OF_BATCH; ++u)
        if (c_lo + u < c_hi) {
          h[static_cast<size_t>(c_lo + u) * E] = acc;
          acc += v[u];
        }
    } else {
      for (int cb = c_lo; cb < c_hi; cb += OF_BATCH) {
#pragma unroll
        for (int u = 0; u < OF_BATCH; ++u) v[u] = (cb + u < c_hi) ? h[static_cast<size_t>(cb + u) * E] : 0;
#pragma unroll
        for (int u = 0; u < OF_BATCH; ++u)
          if (cb + u < c_hi) {
            h[static_cast<size_t>(cb + u) * E] = acc;
            acc += v[u];
          }
      }
    }
    __syncthreads();   // s_part is rewritten by the next round
  }
  for (int x = tid; x < P; x += OF_THREADS) a.counts[x] = s_cnt[x];
  for (int e = tid; e < E; e += OF_THREADS) {
    int acc = 0;
    for (int r = 0; r < R; ++r) {
      a.base[r * E + e] = acc;
      acc += s_cnt[r * E + e];
    }
    s_tot[e] = acc;
    a.totals[e] = acc;
  }
  __syncthreads();
  // warp d: segment offsets of destination d's local experts, and its received rows
  for (int d = warp; d < R; d += OF_THREADS / 32) {
    int* seg = a.segoff + d * (El + 1);
    const int tot = warp_exclusive_scan(
        El, [&](int l) { return s_tot[d * El + l]; }, [&](int l, int pre) { seg[l] = pre; });
    if (lane == 0) {
      seg[El] = tot;
      a.recv_counts[d] = tot;
      s_rc[d] = tot;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int ok = 1;
    for (int d = 0; d < R; ++d)
      if (s_rc[d] > a.cap) ok = 0;
    const int tr = a.tile_rows, nn = a.n_nblk;
    const int acc = warp_exclusive_scan(
        E, [&](int k) { return ok ? ((s_tot[k] + tr - 1) / tr) * nn : 0; },
        [&](int k, int pre) { a.tprefix[k] = pre; });
    if (lane == 0) {
      int rb = 0;   // first position of each destination's rows in the dispatch order
      for (int d = 0; d < R; ++d) {
        a.misc[MISC_RBASE + d] = static_cast<uint32_t>(rb);
        rb += s_rc[d];
      }
      a.tprefix[E] = acc;
      a.misc[MISC_NTILES] = static_cast<uint32_t>(acc);
      a.misc[MISC_OK] = static_cast<uint32_t>(ok);
      if (!ok) atomicCAS(reinterpret_cast<int*>(&a.hdr[HDR_STATUS]), 0, MK_ERR_CAPACITY);
    }
  }
  for (int x = tid; x < R * a.nblk; x += OF_THREADS) a.blocks[x] = 0u;
}

__global__ void __launch_bounds__(256) moe_scatter_kernel(const __grid_constant__ MoeArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int El = a.E_loc, E = a.E, K = a.topk, T = a.T;
  if (a.misc[MISC_OK] == 0u) return;
  const long long n = static_cast<long long>(a.R) * T * K;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long ai = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; ai < n; ai += stride) {
    const int r = static_cast<int>(ai / (static_cast<long long>(T) * K));
    const int aa = static_cast<int>(ai - static_cast<long long>(r) * T * K);
    const int t = aa / K, j = aa - t * K;
    const int e = a.topk_idx[ai];
#if MK_DEBUG_BOUNDS
    if (e < 0 || e >= E) {   // bounds-checking build: record and skip
      bounds_fail(a, BC_MOE_SCATTER, ai);
      continue;
    }
#endif
    const int d = e / El, l = e - d * El;
    const int c = t / RR_TOKENS;
    const int row = a.segoff[d * (El + 1) + l] + a.base[r * E + e] +
                    a.hist[(static_cast<size_t>(r) * a.C + c) * E + e] + a.pos[ai];
#if MK_DEBUG_BOUNDS
    if (row < 0 || row >= a.cap) {
      bounds_fail(a, BC_MOE_SCATTER, ai);
      continue;
    }
#endif
    a.recv_src[d][row] = (r * T + t) * K + j;
    a.fwd[ai] = static_cast<int>(a.misc[MISC_RBASE + d]) + row;
  }
  const int ntiles = static_cast<int>(a.misc[MISC_NTILES]);
  const int npairs = a.R * El;
  for (long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; q < ntiles; q += stride) {
    int lo = 0, hi = npairs - 1;  // last k with tprefix[k] <= q
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

struct MoeLayout {
  size_t blocks_off, misc_off, pos_off, fwd_off, hist_off, base_off, totals_off, segoff_off, tprefix_off, tiles_off;
  size_t trace_off, trace_n;   // in-kernel trace: item records (8 x u64), then copy-warp records
  size_t total;
  int nblk, n_nblk, max_tiles, C;
};

bool moe_layout(int R, int E_loc, int topk, long long T, long long H, long long N, long long cap,
                const mk_config* cfg, MoeLayout& L) {
  const int trace = cfg ? cfg->trace : 0;
  if (trace < 0 || trace > 1) return false;
  if (R < 1 || R > MK_MAX_RANKS || E_loc < 1) return false;
  const long long E = static_cast<long long>(R) * E_loc;
  if (E > MOE_MAX_E || topk < 1 || topk > MOE_MAX_TOPK || topk > E) return false;
  if (T < 0 || H < 0 || N < 0 || cap < 0) return false;
  if ((H % 8) || (N % 8)) return false;
  const long long rows = static_cast<long long>(R) * T * topk;
  if (rows >= (1LL << 31) || cap >= (1LL << 31) || H >= (1LL << 31) || N >= (1LL << 31)) return false;
  if (cap * H >= (1LL << 40)) return false;
  L.nblk = static_cast<int>(ceil_div_ll(cap, BM));
  L.n_nblk = static_cast<int>(ceil_div_ll(N, BN));
  const long long max_tiles = (rows / BM + E) * L.n_nblk;
  if (max_tiles >= (1LL << 30)) return false;
  L.max_tiles = static_cast<int>(max_tiles);
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t off = WS_HDR_BYTES;
  L.blocks_off = off;  off = al(off + static_cast<size_t>(R) * L.nblk * 4);
  L.misc_off = off;    off = al(off + MISC_WORDS * 4);
  L.pos_off = off;     off = al(off + static_cast<size_t>(rows) * 4);
  L.fwd_off = off;     off = al(off + static_cast<size_t>(rows) * 4);
  L.C = static_cast<int>(ceil_div_ll(std::max(T, 1LL), RR_TOKENS));
  L.hist_off = off;    off = al(off + static_cast<size_t>(R) * L.C * E * 4);
  L.base_off = off;    off = al(off + static_cast<size_t>(E) * R * 4);
  L.totals_off = off;  off = al(off + static_cast<size_t>(E) * 4);
  L.segoff_off = off;  off = al(off + static_cast<size_t>(R) * (E_loc + 1) * 4);
  L.tprefix_off = off; off = al(off + (static_cast<size_t>(E) + 1) * 4);
  L.tiles_off = off;   off = al(off + static_cast<size_t>(L.max_tiles) * 5 * 4);
  L.trace_off = 0;
  L.trace_n = 0;
  if (trace) {   // two records per tile-table entry (the CTAs of a pair)
    L.trace_n = static_cast<size_t>(std::max(L.max_tiles, 1)) * 2;
    L.trace_off = off;
    off = al(off + (L.trace_n + MK_TRACE_COPY_RECORDS) * 64);
  }
  L.total = off;
  return true;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool okp(const void* p, long long elems, unsigned align) {
  if (elems > 0 && !p) return false;
  return (reinterpret_cast<uintptr_t>(p) & (align - 1)) == 0;
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" {

size_t mk_moe_workspace_size(int R, int E_loc, int topk, long long T, long long H, long long N,
                             long long cap_rows, const mk_config* cfg) {
  MoeLayout L;
  if (!moe_layout(R, E_loc, topk, T, H, N, cap_rows, cfg, L)) return 0;
  return L.total;
}

size_t mk_moe_trace_entries(int R, int E_loc, int topk, long long T, long long H, long long N,
                            long long cap_rows, const mk_config* cfg, size_t* offset) {
  if (offset) *offset = 0;
  MoeLayout L;
  if (!moe_layout(R, E_loc, topk, T, H, N, cap_rows, cfg, L)) return 0;
  if (offset) *offset = L.trace_off;
  return L.trace_n;
}

mk_status mk_moe_dispatch_gemm(const void* const* x, const float* const* logits, const void* const* w,
                               int R, int E_loc, int topk, long long T, long long H, long long N,
                               long long cap_rows, int* topk_idx, int* counts, int* const* recv_src,
                               int* recv_counts, void* const* recv_x, void* const* y, void* workspace,
                               size_t ws_bytes, const mk_config* cfg, mk_stream_t stream) {
  if (!x || !logits || !w || !recv_src || !recv_x || !y || !workspace) return MK_ERR_INVALID;
  MoeLayout L;
  if (!moe_layout(R, E_loc, topk, T, H, N, cap_rows, cfg, L)) return MK_ERR_INVALID;
  if (cfg && cfg->operand != 0) return MK_ERR_INVALID;   // bf16 operands only
  if (ws_bytes < L.total || !al16(workspace)) return MK_ERR_INVALID;
  const long long E = static_cast<long long>(R) * E_loc;
  const long long rows = static_cast<long long>(R) * T * topk;
  if (!okp(topk_idx, rows, 4) || !okp(counts, R * E, 4) || !okp(recv_counts, R, 4)) return MK_ERR_INVALID;
  for (int r = 0; r < R; ++r) {
    if (!okp(x[r], T * H, 16) || !okp(logits[r], T * E, 4) || !okp(w[r], E_loc * H * N, 16) ||
        !okp(recv_src[r], cap_rows, 4) || !okp(recv_x[r], cap_rows * H, 16) || !okp(y[r], cap_rows * N, 16))
      return MK_ERR_INVALID;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int) * R * E, s) != cudaSuccess) return MK_ERR_CUDA;
    if (cudaMemsetAsync(recv_counts, 0, sizeof(int) * R, s) != cudaSuccess) return MK_ERR_CUDA;
    return MK_OK;
  }
  const int sms = grid_cap(cfg);
  if (sms <= 0) return MK_ERR_UNSUPPORTED;
  // CTA pairs take 256-row tiles of an expert's rows (one 128-row half each).
  const bool pair = use_pair(cfg, sms);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  MoeArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < R; ++r) {
    a.logits[r] = logits[r];
    a.recv_src[r] = recv_src[r];
  }
  a.topk_idx = topk_idx;
  a.counts = counts;
  a.recv_counts = recv_counts;
  a.pos = reinterpret_cast<int*>(ws + L.pos_off);
  a.fwd = reinterpret_cast<int*>(ws + L.fwd_off);
  a.hist = reinterpret_cast<int*>(ws + L.hist_off);
  a.C = L.C;
  a.base = reinterpret_cast<int*>(ws + L.base_off);
  a.totals = reinterpret_cast<int*>(ws + L.totals_off);
  a.segoff = reinterpret_cast<int*>(ws + L.segoff_off);
  a.tprefix = reinterpret_cast<int*>(ws + L.tprefix_off);
  a.tiles = reinterpret_cast<int*>(ws + L.tiles_off);
  a.misc = reinterpret_cast<uint32_t*>(ws + L.misc_off);
  a.blocks = reinterpret_cast<uint32_t*>(ws + L.blocks_off);
  a.hdr = reinterpret_cast<uint32_t*>(ws);
  a.R = R;
  a.E_loc = E_loc;
  a.E = static_cast<int>(E);
  a.topk = topk;
  a.T = static_cast<int>(T);
  a.n_nblk = L.n_nblk;
  a.nblk = L.nblk;
  a.cap = cap_rows;
  a.tile_rows = pair ? 2 * BM : BM;

  const dim3 rgrid(L.C, R);
  if (topk <= 2) moe_route_rank_kernel<2><<<rgrid, RR_THREADS, 0, s>>>(a);
  else moe_route_rank_kernel<MOE_MAX_TOPK><<<rgrid, RR_THREADS, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return MK_ERR_CUDA;
  // offsets, scatter and the fused kernel launch as programmatic dependents of
  // the kernel before them: each waits (griddepcontrol.wait) for its
  // predecessor's results, and its launch overlaps the predecessor's end.
  if (launch_dependent(moe_offsets_kernel, dim3(1), dim3(OF_THREADS), s, a) != cudaSuccess) return MK_ERR_CUDA;
  const long long work = std::max(rows, static_cast<long long>(L.max_tiles));
  const int sgrid = static_cast<int>(std::min<long long>(ceil_div_ll(work, 256), 4LL * sms));
  if (launch_dependent(moe_scatter_kernel, dim3(std::max(1, sgrid)), dim3(256), s, a) != cudaSuccess)
    return MK_ERR_CUDA;
  if (H == 0 || N == 0 || cap_rows == 0) return MK_OK;

  // ---- the persistent dispatch + grouped GEMM kernel
  FusedParams p;
  std::memset(&p, 0, sizeof(p));
  p.op = OP_MOE;
  p.mode = MK_MODE_FUSED;
  p.R = R;
  p.M = static_cast<int>(cap_rows);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(H);
  p.n_nblk = L.n_nblk;
  p.n_kblk = static_cast<int>(ceil_div_ll(H, BK));
  p.n_mblk = 1;
  p.group_m = 1;
  p.split_k = 1;
  p.P = 1;
  p.n_items = L.max_tiles;
  p.moe_tiles = a.tiles;
  p.moe_ntiles = reinterpret_cast<const int*>(a.misc + MISC_NTILES);
  p.moe_ok = reinterpret_cast<const int*>(a.misc + MISC_OK);
  p.moe_recv_counts = recv_counts;
  p.moe_fwd = a.fwd;
  p.moe_rbase = a.misc + MISC_RBASE;
  p.moe_T = static_cast<int>(T);
  p.moe_topk = topk;
  p.moe_nblk = L.nblk;
  int pr = 1;
  while (pr < BM && static_cast<long long>(pr) * 2 * H * 2 <= 32768) pr *= 2;
  p.moe_rows_per_piece = pr;
  // Fused: three copy warps per CTA move the rows at about the rate the tiles
  // consume them (measured: 6 warps front-load the copy and slow the tiles
  // that run beside it; 2 starve the tiles).  The unfused baseline's copy
  // launch runs alone and uses every copy warp.
  p.n_cw = std::max(1, std::min(MK_MOE_COPY_WARPS, N_COPY_WARPS));
  p.moe_boost_waves = MK_MOE_BOOST_WAVES;
  p.b_one_box = (N % 64 == 0) ? 1 : 0;
  p.flags = a.blocks;
  p.hdr = a.hdr;
  p.pdl = 1;
  p.wait_ns = default_wait_ns(cfg);
  p.inject = cfg ? cfg->inject : 0;
  p.epoch = next_epoch();
  p.trace = L.trace_n ? reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + L.trace_off)
                      : nullptr;
  p.trace_cap = static_cast<int>(L.trace_n);
  for (int r = 0; r < R; ++r) {
    p.shard[r] = static_cast<const uint8_t*>(x[r]);
    p.out[r] = y[r];
    p.moe_recv_x[r] = static_cast<uint8_t*>(recv_x[r]);
    p.moe_src[r] = recv_src[r];
    if (!make_map_a(&p.tmA[r], recv_x[r], H, cap_rows, static_cast<size_t>(H) * 2) ||
        !(p.b_one_box ? make_map_w_chunks(&p.tmB[r], w[r], H, N, E_loc, pair ? 2 : 4)
                      : make_map_3d(&p.tmB[r], w[r], N, H, E_loc, static_cast<size_t>(N) * 2,
                                    static_cast<size_t>(H) * N * 2, 64, BK, 1)))
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
  const int mode = cfg ? cfg->mode : MK_MODE_FUSED;
  if (mode == MK_MODE_UNFUSED) {
    // host-ordered baseline: the dispatch copy as one launch, then the grouped GEMM
    p.mode = MK_MODE_UNFUSED;
    p.n_cw = N_COPY_WARPS;
    if (launch_fused(p, grid, s) != cudaSuccess) return MK_ERR_CUDA;
    p.mode = MK_MODE_GEMM_ONLY;
  } else if (mode == MK_MODE_GEMM_ONLY) {
    p.mode = MK_MODE_GEMM_ONLY;   // baseline: recv_x as left by an earlier call
  }
  return launch_fused(p, grid, s) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

}  // extern "C"
