// mk_attn.cu -- ring attention (mKernel write-up, news.chathome.org,
// "五种融合内核" table, row "Ring Attention"): every rank holds a contiguous
// block of the sequence's Q, K and V; the K/V blocks travel around the ring
// while each rank attends its queries to every block that has arrived,
// merging the partial softmax results.
//
// One persistent launch of 384 threads per CTA, one CTA per SM.  A work item
// is a pair of 128-query tiles (Q0, Q1) of one (rank, head), so that every
// K/V tile brought into shared memory serves 256 query rows:
//   * warp 0 (TMA): the item's two Q tiles, then the K tiles, 128 keys each,
//     in ring order -- the rank's own block, then the blocks of ranks r-1,
//     r-2, ... as they land in its receive buffer; warp 11 (TMA): the V tiles;
//   * warp 1 (MMA, one elected lane issuing): per K/V tile, S_i = Q_i K^T
//     (i = 0, 1) into tensor memory, and O_i += P_i V with P_i read from
//     tensor memory (tcgen05, bf16 -> fp32), in the order PV_0(u-1), S_0(u),
//     PV_1(u-1), S_1(u), so that the product of one query tile runs while
//     the softmax works on the other;
//   * warps 2-9 (softmax): all eight on every S tile, S_0 then S_1; each
//     warp holds 16 query rows, each thread half a row (64 keys) in
//     registers; P = 2^(scale * log2(e) * s - m) is written as bf16 into
//     the row half's own columns of S_i; the exponentials are taken against
//     the running maximum, which moves only when it grows by more than 2^8
//     (O_i is then rescaled; the final division uses the same maximum for O
//     and the sum, so the result is unchanged); at the end of an item the
//     warps scale O_0 and O_1 by 1 / sum and store them;
//   * warp 10 (copy): the ring's transfers -- rank r receives the block
//     of rank (r - j) mod R at step j -- moved by the bulk-copy engine
//     through shared memory into its receive buffer, one counter per
//     (rank, step, head).
// Items run rank by rank, causal ones longest first, dealt to the CTAs in
// alternating directions so that every CTA's share of tiles is about equal.
// Causal attention skips the tiles after each query pair (and, in ring order,
// every block of a later rank: those blocks are not moved either).
#include <algorithm>
#include <cmath>
#include <cstring>

#include "mk_internal.h"
#include "mk_ptx.cuh"

namespace mk {

namespace {

constexpr int AT_D = 128;                    // head dimension
constexpr int AT_T = 128;                    // query rows / keys per tile
constexpr int AT_THREADS = 384;              // 12 warps: see the role list above
constexpr int AT_WARP_COPY = 10, AT_WARP_V = 11;
constexpr int AT_MAX_R = 8;
#ifndef MK_ATTN_KST
#define MK_ATTN_KST 2
#endif
constexpr int AT_KST = MK_ATTN_KST;          // K stages
constexpr int AT_VST = 2;                    // V stages
// shared memory (from the 1024-aligned base)
constexpr uint32_t AT_TILE = 32768;          // one 128 x 128 bf16 tile: 2 K-major atoms of [128 rows x 128 B]
constexpr uint32_t AT_Q = 0;                 // Q0, Q1
constexpr uint32_t AT_K = 2 * AT_TILE;       // K stages
constexpr uint32_t AT_V = AT_K + AT_KST * AT_TILE;   // V stages
constexpr uint32_t AT_CHUNK = 16384;         // the ring copy's staging: two buffers of this size
constexpr uint32_t AT_CBUF = AT_V + AT_VST * AT_TILE;
constexpr uint32_t AT_BARS = AT_CBUF + 2 * AT_CHUNK;
constexpr int AT_SMEM = 1024 + AT_BARS + 256;
static_assert(AT_SMEM <= 232448, "dynamic shared memory per block");
// barriers (byte offsets in the barrier block)
constexpr uint32_t B_QFULL = 0, B_QEMPTY = 8, B_KFULL = 16, B_KEMPTY = B_KFULL + 8 * AT_KST,
                   B_VFULL = B_KEMPTY + 8 * AT_KST, B_VEMPTY = B_VFULL + 8 * AT_VST,
                   B_SFULL = B_VEMPTY + 8 * AT_VST, B_GO = B_SFULL + 16, B_OFULL = B_GO + 16,
                   B_DRAIN = B_OFULL + 16, B_CFULL = B_DRAIN + 8, B_TMEM = B_CFULL + 16;
static_assert(B_TMEM + 4 <= 256, "barrier block");
constexpr uint32_t AT_TMEM_COLS = 512;       // S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512)
constexpr uint32_t AT_O_COL = 256;           // O_i at AT_O_COL + 128 i; S_i (and P_i) at 128 i
// S = Q K^T: both operands K-major; O += P V: P from tensor memory (K-major), V MN-major
constexpr uint32_t IDESC_S = idesc_bf16_f32(AT_T, AT_T, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(AT_T, AT_D, false, true);
constexpr float RESCALE_LOG2 = 8.f;          // rescale O when the maximum grows by more than 2^8
// Of every 16 pairs of exponentials in a row, this many are computed by the
// polynomial on the FMA pipe, the rest by the hardware ex2 (MUFU).
#ifndef MK_ATTN_POLY_PAIRS
#define MK_ATTN_POLY_PAIRS 0
#endif
constexpr int POLY_PAIRS = MK_ATTN_POLY_PAIRS;
// How P becomes bf16: 0 = cvt.rn.bf16x2.f32 (round to nearest even, on the
// conversion pipe); 1 = the exponentials are taken 2^-9 high (log2(1 + 2^-9)
// added to the argument), the two upper halves kept by one byte permute (which
// then rounds to within half a bf16 unit), and the row sum divided by the same
// 1 + 2^-9 at the end.
#ifndef MK_ATTN_PACK
#define MK_ATTN_PACK 0
#endif
static_assert(POLY_PAIRS >= 0 && POLY_PAIRS <= 16, "pairs per 16");

struct AttnParams {
  CUtensorMap tmQ[AT_MAX_R], tmK[AT_MAX_R], tmV[AT_MAX_R], tmKr[AT_MAX_R], tmVr[AT_MAX_R];
  uint8_t* out[AT_MAX_R];            // O_r [heads x s_r x d] bf16
  const uint8_t* ksrc[AT_MAX_R];     // K_r, V_r: the ring's sources
  const uint8_t* vsrc[AT_MAX_R];
  uint8_t* krecv[AT_MAX_R];          // [(R-1) x heads x s_r x d]: step j at block j-1
  uint8_t* vrecv[AT_MAX_R];
  uint32_t* cnt;                     // [R x (R-1) x heads] K/V pieces landed per step block
  uint32_t* hdr;
  long long wait_ns;
  uint32_t epoch;
  float scale_log2;                  // softmax scale * log2(e)
  int R, heads, s_r, nkt, nqt, npair, causal, n_items;
  int copy, use_recv, wait;          // ring copies by the copy warps; read them; wait for them
  int n_cw;
  int inject;                        // test only: 1 = one ring piece is never counted
};

// ------------------------------------------------------------------ waits (bounded)
__device__ __forceinline__ bool at_aborted(const AttnParams& p) {
  return ld_volatile(&p.hdr[HDR_ABORT]) == p.epoch;
}
__device__ __noinline__ void at_error(const AttnParams& p, int where, int item, int code = MK_ERR_TIMEOUT) {
  int* st = reinterpret_cast<int*>(&p.hdr[HDR_STATUS]);
  if (atomicCAS(st, 0, code) == 0)
    atomicExch(reinterpret_cast<int*>(&p.hdr[HDR_DETAIL]), where * 1000000 + (item % 1000000));
  __threadfence();
  atomicExch(&p.hdr[HDR_ABORT], p.epoch);
}
// Bounds check of the MK_DEBUG_BOUNDS build (compiled to true otherwise).
__device__ __forceinline__ bool at_bounds_ok(const AttnParams& p, bool cond, int code, long long index) {
#if MK_DEBUG_BOUNDS
  if (!cond) {
    at_error(p, WHERE_BOUNDS, code * 10000 + static_cast<int>(index % 10000), MK_ERR_INVALID);
    return false;
  }
#else
  (void)p; (void)cond; (void)code; (void)index;
#endif
  return true;
}
// The bounded wait loop.  SPIN: poll with the non-blocking test (the MMA
// warp's waits for K and V, which have almost always landed); otherwise
// try_wait, which suspends the warp until the phase completes or a time limit
// passes and leaves its issue slots to the other warps (the MMA warp's wait for
// the softmax: spinning there slowed the two softmax warps that share its SM
// sub-partition, and the slowest softmax warp sets the pace).
template <bool SPIN>
__device__ __noinline__ bool at_wait_loop(const AttnParams& p, uint32_t bar, uint32_t parity, int where, int item,
                                          bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (SPIN ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if ((++it & (SPIN ? 255u : 31u)) == 0) {
      if (honor_abort && at_aborted(p)) return false;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
        at_error(p, where, item);
        return false;
      }
    }
  }
}
// Bounded mbarrier wait.  The first test is inline: a call into the loop costs
// the issuing thread a few hundred cycles even when the phase has completed.
template <bool SPIN = false>
__device__ __forceinline__ bool at_wait_bar(const AttnParams& p, uint32_t bar, uint32_t parity, int where, int item,
                                            bool honor_abort = true) {
  if (SPIN ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  return at_wait_loop<SPIN>(p, bar, parity, where, item, honor_abort);
}
// The MMA warp's waits: every lane polls the barrier (one instruction for the
// warp, and no divergence: a lane-0 poll with a shuffle costs about four times
// as long) and the warp agrees by vote; lane 0 reports a timeout.
template <bool SPIN>
__device__ __noinline__ bool at_wait_warp_loop(const AttnParams& p, uint32_t bar, uint32_t parity, int where, int item,
                                               bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (__all_sync(0xffffffffu, SPIN ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))) return true;
    if ((++it & (SPIN ? 255u : 31u)) == 0) {
      int stop = 0;
      if ((threadIdx.x & 31) == 0) {
        if (honor_abort && at_aborted(p)) {
          stop = 1;
        } else if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
          at_error(p, where, item);
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0) != 0) return false;
    }
  }
}
template <bool SPIN = false>
__device__ __forceinline__ bool at_wait_warp(const AttnParams& p, uint32_t bar, uint32_t parity, int where, int item,
                                             bool honor_abort = true) {
  if (__all_sync(0xffffffffu, SPIN ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))) return true;
  return at_wait_warp_loop<SPIN>(p, bar, parity, where, item, honor_abort);
}
__device__ __noinline__ bool at_wait_value(const AttnParams& p, const uint32_t* f, uint32_t want, int where,
                                           int item) {
  if (ld_acquire_gpu(f) == want) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (ld_acquire_gpu(f) != want) {
    if ((++it & 7u) == 0) {
      if (at_aborted(p)) return false;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
        at_error(p, where, item);
        return false;
      }
    }
    __nanosleep(64);
  }
  return true;
}

// ------------------------------------------------------------------ work lists
struct AtItem {
  int r, h, qp, n;   // rank, head, query-tile pair (tiles 2qp, 2qp+1), K/V tiles to visit
};
// Items run rank by rank, the last rank first.  Causal items run longest first:
// a rank's later query pairs see more of its own block, so inside a rank the
// pairs go in descending order, the heads inside each pair (full attention:
// every item has the same length; heads outer, pairs inner).
__device__ __forceinline__ AtItem at_item(const AttnParams& p, int i) {
  AtItem it;
  const int per_r = p.heads * p.npair;
  it.r = p.R - 1 - i / per_r;
  const int rem = i - (p.R - 1 - it.r) * per_r;
  if (p.causal) {
    const int k = rem / p.heads;
    it.h = rem - k * p.heads;
    it.qp = p.npair - 1 - k;
  } else {
    it.h = rem / p.npair;
    it.qp = rem - it.h * p.npair;
  }
  it.n = p.causal ? min(2 * it.qp + 2, p.nkt) + it.r * p.nkt : p.R * p.nkt;
  return it;
}
// The CTA's round-j item: rounds of gridDim.x items, dealt in CTA order in even
// rounds and in reverse in odd ones, so that with items longest first every
// CTA's total stays near the mean (causal, 8 ranks x 4096 positions: the
// busiest CTA 2 % above it, against 17 % when every round is dealt in order).
// n_items or more: no item for this CTA in round j.  Every role walks the
// same sequence: for (j = 0; j * gridDim.x < n_items; ++j).
__device__ __forceinline__ int at_deal(int j) {
  const int g = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  return j * g + ((j & 1) ? g - 1 - b : b);
}
// Tile t of an item: ring step j (source rank s = r - j mod R) and key tile kt.
// Causal: the rank's own block up to the pair's second query tile, then the
// whole blocks of ranks r-1, r-2, ..., 0.
__device__ __forceinline__ void at_tile(const AttnParams& p, const AtItem& it, int t, int& j, int& s, int& kt) {
  if (p.causal) {
    const int own = min(2 * it.qp + 2, p.nkt);
    if (t < own) {
      j = 0;
      s = it.r;
      kt = t;
      return;
    }
    const int u = t - own;
    j = 1 + u / p.nkt;
    s = it.r - j;
    kt = u - (j - 1) * p.nkt;
    return;
  }
  j = t / p.nkt;
  kt = t - j * p.nkt;
  s = (it.r - j + p.R) % p.R;
}
// Pieces of rank r's step-j block of head h that have landed (K and V of
// every key tile: 2 * nkt when complete).  One acquire per step keeps the
// counter reads off the per-tile load path.
__device__ __forceinline__ uint32_t* at_counter(const AttnParams& p, int r, int j, int h) {
  return p.cnt + (static_cast<size_t>(r) * (p.R - 1) + (j - 1)) * p.heads + h;
}

// ------------------------------------------------------------------ roles
// The CTA's K/V tiles, counted over all its items, form one stream u = 0, 1, ...
// K(u) and V(u) go to stages u % AT_KST and u % AT_VST, each stage with a full
// barrier (the TMA bytes) and an empty barrier (the MMAs that read it), so a
// load is issued as soon as its stage is free.  GO_i phase u completes on the
// arrivals of the eight softmax warps once P_i(u) is written.
// The K / V maps have the block as their outer coordinate (head h of a
// rank's own K_r / V_r, or block (j-1) * heads + h of a receive buffer) and
// rows 0 .. s_r-1 inside it, so the rows of a ragged last tile past s_r read
// as zeros: never another block's rows, which in a receive buffer may not
// have arrived yet (and whatever they hold would enter P V even with P = 0,
// as 0 * NaN).
__device__ __forceinline__ bool at_src(const AttnParams& p, const AtItem& it, int t, bool is_v, int item,
                                       bool& ready, int& waited_j, const CUtensorMap*& m, int& row, int& blk) {
  int j, s, kt;
  at_tile(p, it, t, j, s, kt);
  if (!at_bounds_ok(p, j >= 0 && j < p.R && s >= 0 && s < p.R && kt >= 0 && kt < p.nkt && it.h >= 0 &&
                           it.h < p.heads && it.r >= 0 && it.r < p.R && 2 * it.qp < p.nqt,
                    BC_ATTN_TILE, item))
    return false;
  m = is_v ? &p.tmV[s] : &p.tmK[s];
  row = kt * AT_T;
  blk = it.h;
  if (j > 0 && p.use_recv) {
    if (p.wait && j != waited_j) {
      if (!ready) {
        if (!at_wait_value(p, &p.hdr[HDR_READY], p.epoch, WHERE_PRODUCER, item)) return false;
        ready = true;
      }
      if (!at_wait_value(p, at_counter(p, it.r, j, it.h), 2u * p.nkt, WHERE_PRODUCER, item)) return false;
      fence_proxy_async_global();
      waited_j = j;
    }
    m = is_v ? &p.tmVr[it.r] : &p.tmKr[it.r];
    blk = (j - 1) * p.heads + it.h;
  }
  return true;
}

// K producer (warp 0, one thread): each item's K tiles, and after the first of
// them its Q0 and Q1 (once the previous item's last S has completed).
__device__ void at_producer_k(const AttnParams& p, uint32_t bars, uint32_t base) {
  uint32_t q_ph = 0, e_ph = 0;
  int stage = 0;
  bool ready = false;
  for (int j = 0; j * static_cast<int>(gridDim.x) < p.n_items; ++j) {
    const int i = at_deal(j);
    if (i >= p.n_items) continue;
    const AtItem it = at_item(p, i);
    int waited_j = 0;
    for (int t = 0; t < it.n; ++t) {
      const CUtensorMap* m;
      int row, blk;
      if (!at_src(p, it, t, false, i, ready, waited_j, m, row, blk)) return;
      if (!at_wait_bar(p, bars + B_KEMPTY + 8u * stage, e_ph ^ 1u, WHERE_PRODUCER, i)) return;
      const uint32_t full = bars + B_KFULL + 8u * stage;
      const uint32_t dst = base + AT_K + static_cast<uint32_t>(stage) * AT_TILE;
      mbar_arrive_expect_tx(full, AT_TILE);
      tma_load_3d(dst, m, full, 0, row, blk);
      tma_load_3d(dst + 16384u, m, full, 64, row, blk);
      if (++stage == AT_KST) {
        stage = 0;
        e_ph ^= 1u;
      }
      if (t == 0) {   // the item's query tiles
        if (!at_wait_bar(p, bars + B_QEMPTY, q_ph ^ 1u, WHERE_PRODUCER, i)) return;
        q_ph ^= 1u;
        const int qrow = it.h * p.s_r + 2 * it.qp * AT_T;
        mbar_arrive_expect_tx(bars + B_QFULL, 2u * AT_TILE);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          tma_load_2d(base + AT_Q + q * AT_TILE, &p.tmQ[it.r], bars + B_QFULL, 0, qrow + q * AT_T);
          tma_load_2d(base + AT_Q + q * AT_TILE + 16384u, &p.tmQ[it.r], bars + B_QFULL, 64, qrow + q * AT_T);
        }
      }
    }
  }
}

// V producer (warp 11, one thread).
__device__ void at_producer_v(const AttnParams& p, uint32_t bars, uint32_t base) {
  uint32_t e_ph = 0;
  int stage = 0;
  bool ready = false;
  for (int j = 0; j * static_cast<int>(gridDim.x) < p.n_items; ++j) {
    const int i = at_deal(j);
    if (i >= p.n_items) continue;
    const AtItem it = at_item(p, i);
    int waited_j = 0;
    for (int t = 0; t < it.n; ++t) {
      const CUtensorMap* m;
      int row, blk;
      if (!at_src(p, it, t, true, i, ready, waited_j, m, row, blk)) return;
      if (!at_wait_bar(p, bars + B_VEMPTY + 8u * stage, e_ph ^ 1u, WHERE_PRODUCER, i)) return;
      const uint32_t full = bars + B_VFULL + 8u * stage;
      const uint32_t dst = base + AT_V + static_cast<uint32_t>(stage) * AT_TILE;
      mbar_arrive_expect_tx(full, AT_TILE);
      tma_load_4d(dst, m, full, 0, row, 0, blk);
      tma_load_4d(dst + 16384u, m, full, 0, row + 64, 0, blk);
      if (++stage == AT_VST) {
        stage = 0;
        e_ph ^= 1u;
      }
    }
  }
}

// S_i = Q_i K(u)^T into S_i (columns 128 i): 8 MMAs of K = 16.
__device__ __forceinline__ void at_s(uint32_t base, uint32_t tmem, int i, int kstage) {
  const uint32_t qb = base + AT_Q + static_cast<uint32_t>(i) * AT_TILE;
  const uint32_t kb = base + AT_K + static_cast<uint32_t>(kstage) * AT_TILE;
  // descriptors differ only in the start address field (address >> 4, low bits)
  const uint64_t dq = sdesc_swz(qb, 16u, 1024u, 2u), dk = sdesc_swz(kb, 16u, 1024u, 2u);
  if (elect_one_sync()) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = dq + ((16384u * a + 32u * k) >> 4);
        const uint64_t bd = dk + ((16384u * a + 32u * k) >> 4);
        tc_mma_bf16(tmem + static_cast<uint32_t>(i) * AT_T, ad, bd, IDESC_S, (a | k) ? 1u : 0u);
      }
  }
  __syncwarp();
}
// O_i (+)= P_i V(u): P_i from tensor memory (keys 2c, 2c+1 in column c for c < 32, keys
// 64 + 2c, 65 + 2c in column 64 + c), V MN-major
// (two 64-column atoms 8 KB apart, 8-key groups 1024 B apart).
__device__ __forceinline__ void at_pv(uint32_t base, uint32_t tmem, int i, int vstage, bool first) {
  const uint32_t vb = base + AT_V + static_cast<uint32_t>(vstage) * AT_TILE;
  const uint32_t pcol = tmem + static_cast<uint32_t>(i) * AT_T;
  const uint32_t obuf = tmem + AT_O_COL + static_cast<uint32_t>(i) * AT_T;
  const uint64_t dv = sdesc_sw128(vb, 8192u, 1024u);
  if (elect_one_sync()) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t bd = dv + ((16384u * a + 2048u * k) >> 4);
        tc_mma_bf16_ts(obuf, pcol + 64u * a + 8u * k, bd, IDESC_PV, (!first || a || k) ? 1u : 0u);
      }
  }
  __syncwarp();
}
// tcgen05.commit from the lane that issued the MMAs (elect.sync over the full
// warp chooses the same lane each time).
__device__ __forceinline__ void at_commit(uint32_t bar) {
  if (elect_one_sync()) tc_commit(bar);
  __syncwarp();
}

// MMA issuer (warp 1, converged: lane 0 waits, one elected lane issues the
// MMAs and commits, the descriptors are computed by the whole warp).
// Iteration u: [K(u), V(u-1) landed, GO_0 phase u-1] PV_0(u-1), S_0(u),
// [GO_1 phase u-1] PV_1(u-1), S_1(u).  A product of tile u-1 is
// issued before the S of tile u that overwrites its P: the tensor pipe runs a
// thread's MMAs in issue order.  Commits: S_i full after each S_i (for S_1
// also the K stage free), V stage free after PV_1, the query tiles free after
// an item's last S_1, O_i full after an item's last PV_i.
__device__ void at_mma(const AttnParams& p, uint32_t bars, uint32_t base, uint32_t tmem) {
  uint32_t q_ph = 0, go_ph = 0, k_ph = 0, v_ph = 0;
  uint32_t u = 0;
  int kst = 0, vst = 0;
  bool prev_first = false, prev_last = false;   // the pending tile u-1 opens / closes its item
  int item = -1;
  for (int j = 0; j * static_cast<int>(gridDim.x) < p.n_items; ++j) {
    const int i = at_deal(j);
    if (i >= p.n_items) continue;
    const AtItem it = at_item(p, i);
    item = i;
    for (int t = 0; t < it.n; ++t, ++u) {
      // the loads first (they have usually landed long before): every wait
      // costs the issuer time, and P_0(u-1) is the one the chain waits for
      if (t == 0) {
        if (!at_wait_warp(p, bars + B_QFULL, q_ph, WHERE_MMA, i)) goto done;
        q_ph ^= 1u;
      }
      if (!at_wait_warp<true>(p, bars + B_KFULL + 8u * kst, k_ph, WHERE_MMA, i)) goto done;
      if (u >= 1) {
        // V(u-1) landed and P_0(u-1) written
        if (!at_wait_warp<true>(p, bars + B_VFULL + 8u * vst, v_ph, WHERE_MMA, i)) goto done;
        if (!at_wait_warp<false>(p, bars + B_GO, go_ph, WHERE_MMA, i)) goto done;
        tc_fence_after();
        at_pv(base, tmem, 0, vst, prev_first);
        if (prev_last) at_commit(bars + B_OFULL);
      }
      tc_fence_after();
      at_s(base, tmem, 0, kst);
      at_commit(bars + B_SFULL);
      if (u >= 1) {
        if (!at_wait_warp<false>(p, bars + B_GO + 8u, go_ph, WHERE_MMA, i)) goto done;
        go_ph ^= 1u;
        tc_fence_after();
        at_pv(base, tmem, 1, vst, prev_first);
        at_commit(bars + B_VEMPTY + 8u * vst);   // V(u-1) read by both products
        if (prev_last) at_commit(bars + B_OFULL + 8u);
        if (++vst == AT_VST) {
          vst = 0;
          v_ph ^= 1u;
        }
      }
      at_s(base, tmem, 1, kst);
      at_commit(bars + B_SFULL + 8u);
      at_commit(bars + B_KEMPTY + 8u * kst);     // K(u) read by both S
      if (t == it.n - 1) at_commit(bars + B_QEMPTY);
      if (++kst == AT_KST) {
        kst = 0;
        k_ph ^= 1u;
      }
      prev_first = (t == 0);
      prev_last = (t == it.n - 1);
    }
  }
  if (u >= 1) {   // the products of the last tile
    if (!at_wait_warp<true>(p, bars + B_VFULL + 8u * vst, v_ph, WHERE_MMA, item)) goto done;
    if (!at_wait_warp<false>(p, bars + B_GO, go_ph, WHERE_MMA, item)) goto done;
    tc_fence_after();
    at_pv(base, tmem, 0, vst, prev_first);
    at_commit(bars + B_OFULL);
    if (!at_wait_warp<false>(p, bars + B_GO + 8u, go_ph, WHERE_MMA, item)) goto done;
    tc_fence_after();
    at_pv(base, tmem, 1, vst, prev_first);
    at_commit(bars + B_VEMPTY + 8u * vst);
    at_commit(bars + B_OFULL + 8u);
  }
done:
  at_commit(bars + B_DRAIN);
  at_wait_warp(p, bars + B_DRAIN, 0, WHERE_DRAIN, 0, false);
}

// 2^x for x <= 0 or -inf (the hardware approximation, flushing subnormals).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two fp32 lanes in one 64-bit register: a*b + c and a + b on both lanes at once.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Two values of 2^x on the FMA pipe, for -125 <= x <= 64 (smaller x are clamped:
// the result, <= 2^-125, is below anything a row keeps).  Range reduction:
// x = n + f with n = round(x) (adding 1.5 * 2^23 leaves n in the low mantissa
// bits) and |f| <= 1/2, then 2^f by a cubic 1 + f (c1 + f (c2 + f c3)) fitted to
// 2^f on [-1/2, 1/2] (relative error below 1.3e-4, far under bf16's 2^-9), and
// n added to the exponent field: the bits of 1.5 * 2^23 + n shifted left by 23
// are n << 23, since the constant's low nine bits are zero.
__device__ __forceinline__ void ex2_poly2(float x0, float x1, float& y0, float& y1) {
  constexpr float SHIFT = 12582912.f;            // 1.5 * 2^23
  const uint64_t xs = f2pack(fmaxf(x0, -125.f), fmaxf(x1, -125.f));
  const uint64_t t = f2add(xs, f2pack(SHIFT, SHIFT));
  const uint64_t n = f2add(t, f2pack(-SHIFT, -SHIFT));
  const uint64_t f = f2fma(n, f2pack(-1.f, -1.f), xs);   // exact: x - round(x)
  uint64_t q = f2fma(f, f2pack(0.05533514f, 0.05533514f), f2pack(0.24229739f, 0.24229739f));
  q = f2fma(q, f, f2pack(0.69322545f, 0.69322545f));
  q = f2fma(q, f, f2pack(1.f, 1.f));
  float q0, q1, t0, t1;
  f2unpack(q, q0, q1);
  f2unpack(t, t0, t1);
  uint32_t r0, r1;
  asm("mad.lo.u32 %0, %1, 8388608, %2;" : "=r"(r0) : "r"(__float_as_uint(t0)), "r"(__float_as_uint(q0)));
  asm("mad.lo.u32 %0, %1, 8388608, %2;" : "=r"(r1) : "r"(__float_as_uint(t1)), "r"(__float_as_uint(q1)));
  y0 = __uint_as_float(r0);
  y1 = __uint_as_float(r1);
}

// The reference the exponentials are taken against for running maximum m.
__device__ __forceinline__ float at_p_ref(float m) {
#if MK_ATTN_PACK
  return m - 0.0028150156f;   // log2(1 + 2^-9): the exponentials 2^-9 high
#else
  return m;
#endif
}
// Half a row: this thread's 64 keys of S_i (keys 64 kh + 0 .. 63, kh = the
// thread's half).  P = 2^(c*s - m_ref) (keys >= lim set to 0 when masked) is
// stored as bf16 pairs, keys 2q, 2q+1 (q = 0 .. 31 within the half) in
// column 64 kh + q of S_i, i.e. inside the half's own score columns; returns
// the half's sum of P.  MAX: also the maximum of the half's raw scores (of the
// keys below lim) into mx.
template <bool MAX>
__device__ __forceinline__ float at_emit_p(const uint32_t (&sv)[2][32], uint32_t sbase, float c, float m_ref,
                                           bool masked, int lim, int key0, float& mx) {
  const uint64_t c2 = f2pack(c, c), nm2 = f2pack(-m_ref, -m_ref);
  uint64_t l4[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
  float m4[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int cc = 0; cc < 2; ++cc)
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
      uint32_t pk[8];
#pragma unroll
      for (int qq = 0; qq < 8; ++qq) {
        const int q = 8 * h8 + qq;
        const int kk = key0 + 32 * cc + 2 * q;
        const float s0 = __uint_as_float(sv[cc][2 * q]), s1 = __uint_as_float(sv[cc][2 * q + 1]);
        if (MAX) {
          if (masked) {
            if (kk < lim) m4[cc] = fmaxf(m4[cc], s0);
            if (kk + 1 < lim) m4[cc] = fmaxf(m4[cc], s1);
          } else {
            m4[cc] = fmax3(m4[cc], s0, s1);
          }
        }
        float e0, e1, p0, p1;
        f2unpack(f2fma(f2pack(s0, s1), c2, nm2), e0, e1);
        if (((16 * cc + q) & 15) < POLY_PAIRS) {
          ex2_poly2(e0, e1, p0, p1);
        } else {
          p0 = ex2(e0);
          p1 = ex2(e1);
        }
        if (masked) {
          p0 = (kk < lim) ? p0 : 0.f;
          p1 = (kk + 1 < lim) ? p1 : 0.f;
        }
        l4[q & 1] = f2add(l4[q & 1], f2pack(p0, p1));
#if MK_ATTN_PACK
        pk[qq] = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x7632);
#else
        pk[qq] = pack_bf16x2(p0, p1);
#endif
      }
      tc_st_16x32bx2_x8_h64(sbase + 16u * cc + 8u * h8, pk);
    }
  if (MAX) mx = fmaxf(m4[0], m4[1]);
  float la, lb;
  f2unpack(f2add(l4[0], l4[1]), la, lb);
  return la + lb;
}

// Softmax (warps 2-9): all eight warps work on every S tile, S_0 then S_1 of
// each K/V tile.  Warp w takes 16 of the 32 TMEM lanes of its quarter (w % 4):
// lanes 32 (w % 4) + 16 ((w - 2) / 4) + 0 .. 15, one query row each; a row is
// split between threads t and t + 16 (keys 0 .. 63 and 64 .. 127), which
// combine its maximum and sum by one shuffle, so both halves of a row always
// hold the same running maximum.
__device__ void at_softmax(const AttnParams& p, uint32_t bars, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int lane16 = 32 * quarter + 16 * ((warp - 2) >> 2);  // first TMEM lane of this warp
  const int row = lane16 + (lane & 15);                      // query row within a tile
  const int kh = lane >> 4;                                  // which half of the row's keys
  const int key0 = 64 * kh;
  const uint32_t lane_off = static_cast<uint32_t>(lane16) << 16;
  const float c = p.scale_log2;
  uint32_t sf_ph = 0, of_ph = 0;                             // bit g: query tile g
  for (int j = 0; j * static_cast<int>(gridDim.x) < p.n_items; ++j) {
    const int i = at_deal(j);
    if (i >= p.n_items) continue;
    const AtItem it = at_item(p, i);
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    for (int t = 0; t < it.n; ++t) {
      int j, s, kt;
      at_tile(p, it, t, j, s, kt);
      const int valid = min(AT_T, p.s_r - kt * AT_T);       // keys of this tile inside the block
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int qt = 2 * it.qp + g;
        const uint32_t sbase = tmem + lane_off + static_cast<uint32_t>(g) * AT_T;
        int lim = valid;
        if (p.causal && j == 0) lim = (kt > qt) ? 0 : (kt == qt ? min(valid, row + 1) : valid);
        const bool masked = __any_sync(0xffffffffu, lim < AT_T);
        {
          const int ok = at_wait_bar(p, bars + B_SFULL + 8u * g, (sf_ph >> g) & 1u, WHERE_EPILOGUE, i) ? 1 : 0;
          if (!__all_sync(0xffffffffu, ok)) return;
        }
        sf_ph ^= 1u << g;
        tc_fence_after();
        uint32_t sv[2][32];
        tc_ld_16x32bx2_x32_h64(sbase, sv[0]);
        tc_ld_16x32bx2_x32_h64(sbase + 32u, sv[1]);
        tc_wait_ld_regs(sv[0]);
        reg_fence(sv[1]);
        float factor = 1.f, lsum, mx;
        if (t > 0 && !masked) {
          // P against the running maximum, the tile's maximum taken alongside:
          // the maximum moves only when it grows by more than 2^8, which the
          // check below catches (then the tile is done again)
          lsum = at_emit_p<true>(sv, sbase, c, at_p_ref(m_run[g]), false, AT_T, key0, mx);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[g], mx * c);
          const bool grow = m_new > m_run[g] + RESCALE_LOG2;
          if (__any_sync(0xffffffffu, grow)) {
            if (grow) {
              factor = ex2(m_run[g] - m_new);
              m_run[g] = m_new;
              l_run[g] *= factor;
            }
            tc_wait_st();
            lsum = at_emit_p<false>(sv, sbase, c, at_p_ref(m_run[g]), false, AT_T, key0, mx);
          }
        } else {
          // the row maximum first (scale > 0 keeps the order: taken unscaled)
          mx = -INFINITY;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if (!masked || key0 + 32 * cc + q < lim) mx = fmaxf(mx, __uint_as_float(sv[cc][q]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[g], mx * c);
          if (t == 0) {
            m_run[g] = m_new;
          } else if (m_new > m_run[g] + RESCALE_LOG2) {
            factor = ex2(m_run[g] - m_new);
            m_run[g] = m_new;
            l_run[g] *= factor;
          }
          lsum = at_emit_p<false>(sv, sbase, c, at_p_ref(m_run[g]), masked, lim, key0, mx);
        }
        l_run[g] += lsum;
        // S_g(u) complete implies the product of tile u-1 complete (issued
        // before it): O_g is settled until P_g(u) is published
        if (__any_sync(0xffffffffu, factor != 1.f)) {
          const uint32_t obase = tmem + lane_off + AT_O_COL + static_cast<uint32_t>(g) * AT_T;
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t v[32];
            tc_ld_16x32bx2_x32_h64(obase + 32u * cc, v);
            tc_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(__uint_as_float(v[q]) * factor);
            tc_st_16x32bx2_x32_h64(obase + 32u * cc, v);
          }
        }
        // P_g(u) (and any rescaled O_g) written: the products may read them
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + B_GO + 8u * g);
      }
    }
    // item done: the last product into each O_g has completed
    for (int g = 0; g < 2; ++g) {
      {
        const int ok = at_wait_bar(p, bars + B_OFULL + 8u * g, (of_ph >> g) & 1u, WHERE_EPILOGUE, i) ? 1 : 0;
        if (!__all_sync(0xffffffffu, ok)) return;
      }
      of_ph ^= 1u << g;
      tc_fence_after();
      const float l = l_run[g] + __shfl_xor_sync(0xffffffffu, l_run[g], 16);
#if MK_ATTN_PACK
      const float inv = (l > 0.f) ? 1.001953125f / l : 0.f;   // (1 + 2^-9) / sum
#else
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
#endif
      const int qpos = (2 * it.qp + g) * AT_T + row;          // position within rank r's block
      const bool row_ok = qpos < p.s_r;
      uint8_t* orow = p.out[it.r] + (static_cast<size_t>(it.h) * p.s_r + qpos) * AT_D * 2 + key0 * 2;
      const uint32_t obase = tmem + lane_off + AT_O_COL + static_cast<uint32_t>(g) * AT_T;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t v[32];
        tc_ld_16x32bx2_x32_h64(obase + 32u * cc, v);
        tc_wait_ld();
        if (!row_ok) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_v4(orow + (32 * cc + 8 * q) * 2,
                       pack_bf16x2(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv),
                       pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv),
                       pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv),
                       pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv));
      }
    }
    // O read out: the next item's first products may overwrite it once P of
    // that item's first tile is published (the waits before those products)
    tc_fence_before();
  }
}

// The ring's transfers: piece = (rank r, step j >= 1, head h, key tile kt, K or V),
// in the order the work list needs them (ranks as the items run, then step,
// head, tile).  Copy warp w takes pieces w, w + n_workers, ...  Lane 0 moves
// a piece with the bulk-copy engine in chunks of up to 16 KB through two
// shared-memory buffers (global -> shared on a barrier, shared -> global as a
// bulk group), the next chunk's load in flight while the current one is
// stored; once a piece's stores have completed it counts the piece in its
// (rank, step, head) counter.  (Row copies through registers cost the
// softmax and MMA warps more: their load/store stream competes with the
// barrier and tensor-memory traffic.)
__device__ void at_copy(const AttnParams& p, uint32_t bars, uint32_t base) {
  const int lane = threadIdx.x & 31;
  const int cw = (threadIdx.x >> 5) - AT_WARP_COPY;
  if (cw >= p.n_cw || lane != 0) return;
  const int worker = blockIdx.x * p.n_cw + cw;
  const int n_workers = gridDim.x * p.n_cw;
  if (!at_wait_value(p, &p.hdr[HDR_READY], p.epoch, WHERE_COPY, worker)) return;
  const long long per_r = static_cast<long long>(p.heads) * (p.R - 1) * p.nkt * 2;
  const long long total = per_r * p.R;
  bool skip_first = (p.inject == 1 && worker == 0);
  uint32_t n = 0;   // chunks whose load has been issued; chunk c uses buffer c & 1
  // the newest chunk: loaded (or landing) but not yet stored
  bool pend = false, pend_last = false;
  uint8_t* pend_dst = nullptr;
  uint32_t pend_bytes = 0;
  uint32_t* pend_counter = nullptr;
  // Store chunk n-1 once it has landed; after the last chunk of a piece, wait
  // until the piece's stores have completed and count it.
  auto store_pending = [&]() -> bool {
    const uint32_t pb = (n - 1) & 1u;
    if (!at_wait_bar(p, bars + B_CFULL + 8u * pb, ((n - 1) >> 1) & 1u, WHERE_COPY, worker)) return false;
    bulk_s2g(pend_dst, base + AT_CBUF + pb * AT_CHUNK, pend_bytes);
    bulk_commit();
    pend = false;
    if (pend_last) {
      bulk_wait<0>();
      fence_proxy_async_global();
      __threadfence();
      if (skip_first) skip_first = false;
      else atomicAdd(pend_counter, 1u);
    }
    return true;
  };
  for (long long q = worker; q < total; q += n_workers) {
    const int rr = static_cast<int>(q / per_r);
    long long rem = q - rr * per_r;
    const int r = p.R - 1 - rr;
    // step-major: the query tiles of a rank run in parallel and all need step j before j+1
    const int j = 1 + static_cast<int>(rem / (static_cast<long long>(p.heads) * p.nkt * 2));
    rem -= static_cast<long long>(j - 1) * p.heads * p.nkt * 2;
    const int h = static_cast<int>(rem / (p.nkt * 2));
    rem -= static_cast<long long>(h) * p.nkt * 2;
    const int kt = static_cast<int>(rem / 2), isv = static_cast<int>(rem & 1);
    const int s = (r - j + p.R) % p.R;
    if (p.causal && s > r) continue;            // a later rank's keys: never read
    if (at_aborted(p)) break;
    const int rows = min(AT_T, p.s_r - kt * AT_T);
    if (!at_bounds_ok(p, r >= 0 && r < p.R && j >= 1 && j < p.R && s >= 0 && s < p.R && h < p.heads && kt < p.nkt &&
                             rows > 0,
                      BC_ATTN_COPY, q))
      break;
    const size_t src_off = (static_cast<size_t>(h) * p.s_r + static_cast<size_t>(kt) * AT_T) * AT_D * 2;
    const size_t dst_off =
        ((static_cast<size_t>(j - 1) * p.heads + h) * p.s_r + static_cast<size_t>(kt) * AT_T) * AT_D * 2;
    const uint8_t* src = (isv ? p.vsrc[s] : p.ksrc[s]) + src_off;
    uint8_t* dst = (isv ? p.vrecv[r] : p.krecv[r]) + dst_off;
    const uint32_t bytes = static_cast<uint32_t>(rows) * AT_D * 2;   // a multiple of 256
    for (uint32_t off = 0; off < bytes; off += AT_CHUNK) {
      if (pend && !store_pending()) goto out;
      const uint32_t cb = min(AT_CHUNK, bytes - off);
      const uint32_t b = n & 1u;
      // buffer b was last read by the store of chunk n-2: only the newest
      // store (chunk n-1) may still be reading shared memory
      bulk_wait_read<1>();
      mbar_arrive_expect_tx(bars + B_CFULL + 8u * b, cb);
      bulk_g2s(base + AT_CBUF + b * AT_CHUNK, src + off, cb, bars + B_CFULL + 8u * b);
      ++n;
      pend = true;
      pend_dst = dst + off;
      pend_bytes = cb;
      pend_last = (off + cb >= bytes);
      pend_counter = at_counter(p, r, j, h);
    }
  }
  if (pend) store_pending();
out:
  bulk_wait<0>();   // no store may still read shared memory when the CTA exits
}

__global__ void __launch_bounds__(AT_THREADS, 1) mk_ring_attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = smem_u32(smem);
  const uint32_t bars = base + AT_BARS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + AT_BARS + B_TMEM);
  if (blockIdx.x == 0 && p.copy) {
    // zero this call's ring counters, then publish them
    const long long n = static_cast<long long>(p.R) * (p.R - 1) * p.heads;
    for (long long x = threadIdx.x; x < n; x += AT_THREADS) p.cnt[x] = 0u;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release_gpu(&p.hdr[HDR_READY], p.epoch);
  }
  if (warp == 0 && lane == 0) {
    mbar_init(bars + B_QFULL, 1);
    mbar_init(bars + B_QEMPTY, 1);
    for (int s = 0; s < AT_KST; ++s) {
      mbar_init(bars + B_KFULL + 8u * s, 1);
      mbar_init(bars + B_KEMPTY + 8u * s, 1);
    }
    for (int s = 0; s < AT_VST; ++s) {
      mbar_init(bars + B_VFULL + 8u * s, 1);
      mbar_init(bars + B_VEMPTY + 8u * s, 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(bars + B_SFULL + 8u * g, 1);
      mbar_init(bars + B_OFULL + 8u * g, 1);
    }
    mbar_init(bars + B_GO, 8);          // the softmax warps, for Q0
    mbar_init(bars + B_GO + 8u, 8);     // and for Q1
    mbar_init(bars + B_DRAIN, 1);       // MMA drain
    mbar_init(bars + B_CFULL, 1);       // the ring copy's two staging buffers
    mbar_init(bars + B_CFULL + 8u, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), AT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0 || warp == AT_WARP_V) {
    if (lane == 0) {
      if (warp == 0) at_producer_k(p, bars, base);
      else at_producer_v(p, bars, base);
    }
    __syncwarp();
  } else if (warp == 1) {
    at_mma(p, bars, base, tmem);
    __syncwarp();
  } else if (warp <= 9) {
    at_softmax(p, bars, tmem);
    __syncwarp();
  } else if (warp == AT_WARP_COPY && p.copy) {
    at_copy(p, bars, base);
    __syncwarp();
  }
  tc_fence_before();
  // after an abort, TMA loads whose barrier phases will never complete may
  // still be in flight: give them time to land before the CTA exits
  if (threadIdx.x == 0 && at_aborted(p)) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) __nanosleep(1000);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, AT_TMEM_COLS);
  }
}

struct AttnLayout {
  size_t cnt_off, total;
  int nkt, nqt;
};

bool attn_layout(int R, int heads, long long s_r, int d, AttnLayout& L) {
  if (R < 1 || R > AT_MAX_R || heads < 1 || s_r < 0 || d != AT_D) return false;
  if (static_cast<long long>(heads) * s_r >= (1LL << 31) / AT_D) return false;
  L.nkt = static_cast<int>(ceil_div_ll(s_r, AT_T));
  L.nqt = L.nkt;
  L.cnt_off = WS_HDR_BYTES;
  L.total = L.cnt_off + ((static_cast<size_t>(R) * std::max(R - 1, 0) * heads * 4 + 255) & ~size_t(255));
  return true;
}

cudaError_t attn_launch(const AttnParams& p, int grid, cudaStream_t s) {
  static int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(mk_ring_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  mk_ring_attn_kernel<<<grid, AT_THREADS, AT_SMEM, s>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" {

size_t mk_ring_attention_workspace_size(int R, int heads, long long s_r, int d, int causal,
                                        const mk_config* cfg) {
  (void)cfg;
  (void)causal;
  AttnLayout L;
  if (!attn_layout(R, heads, s_r, d, L)) return 0;
  return L.total;
}

mk_status mk_ring_attention(const void* const* q, const void* const* k, const void* const* v, int R, int heads,
                            long long s_r, int d, int causal, float scale, void* const* k_recv,
                            void* const* v_recv, void* const* out, void* workspace, size_t ws_bytes,
                            const mk_config* cfg, mk_stream_t stream) {
  if (!q || !k || !v || !out || !workspace) return MK_ERR_INVALID;
  AttnLayout L;
  if (!attn_layout(R, heads, s_r, d, L)) return MK_ERR_INVALID;
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 15u)) return MK_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MK_ERR_INVALID;
  const int mode = cfg ? cfg->mode : MK_MODE_FUSED;
  if (mode < MK_MODE_FUSED || mode > MK_MODE_UNFUSED) return MK_ERR_INVALID;
  if (cfg && cfg->operand != 0) return MK_ERR_INVALID;   // bf16 operands only
  const long long blk = static_cast<long long>(heads) * s_r * d;
  const bool need_recv = (R > 1 && mode != MK_MODE_GEMM_ONLY);
  if (need_recv && (!k_recv || !v_recv)) return MK_ERR_INVALID;
  for (int r = 0; r < R; ++r) {
    auto bad = [&](const void* ptr, long long elems) {
      return (elems > 0 && !ptr) || (reinterpret_cast<uintptr_t>(ptr) & 15u);
    };
    if (bad(q[r], blk) || bad(k[r], blk) || bad(v[r], blk) || bad(out[r], blk)) return MK_ERR_INVALID;
    if (need_recv && (bad(k_recv[r], blk * (R - 1)) || bad(v_recv[r], blk * (R - 1)))) return MK_ERR_INVALID;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (s_r == 0) return MK_OK;
  int sms = device_sm_count();
  if (sms <= 0) return MK_ERR_UNSUPPORTED;
  if (cfg && cfg->max_ctas > 0) sms = std::min(sms, cfg->max_ctas);

  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.R = R;
  p.heads = heads;
  p.s_r = static_cast<int>(s_r);
  p.nkt = L.nkt;
  p.nqt = L.nqt;
  p.npair = (L.nqt + 1) / 2;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.cnt = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + L.cnt_off);
  p.hdr = static_cast<uint32_t*>(workspace);
  p.wait_ns = default_wait_ns(cfg);
  p.inject = cfg ? cfg->inject : 0;
  p.epoch = next_epoch();
  p.n_cw = 1;   // warp 10
  const uint64_t rows = static_cast<uint64_t>(heads) * s_r;
  for (int r = 0; r < R; ++r) {
    p.out[r] = static_cast<uint8_t*>(out[r]);
    p.ksrc[r] = static_cast<const uint8_t*>(k[r]);
    p.vsrc[r] = static_cast<const uint8_t*>(v[r]);
    // K: [d, s_r, heads], boxes of 64 d x 128 rows; V: [64 d, s_r, 2 d halves,
    // heads], boxes of 64 rows x both halves (MN-major for P V)
    if (!make_map_a(&p.tmQ[r], q[r], AT_D, rows, AT_D * 2) ||
        !make_map_3d(&p.tmK[r], k[r], AT_D, s_r, heads, AT_D * 2, static_cast<uint64_t>(s_r) * AT_D * 2, 64, AT_T,
                     1) ||
        !make_map_w_chunks(&p.tmV[r], v[r], s_r, AT_D, heads, 2))
      return MK_ERR_CUDA;
    if (need_recv) {
      p.krecv[r] = static_cast<uint8_t*>(k_recv[r]);
      p.vrecv[r] = static_cast<uint8_t*>(v_recv[r]);
      const uint64_t blocks = static_cast<uint64_t>(heads) * (R - 1);
      if (!make_map_3d(&p.tmKr[r], k_recv[r], AT_D, s_r, blocks, AT_D * 2, static_cast<uint64_t>(s_r) * AT_D * 2, 64,
                       AT_T, 1) ||
          !make_map_w_chunks(&p.tmVr[r], v_recv[r], s_r, AT_D, blocks, 2))
        return MK_ERR_CUDA;
    }
  }
  const int n_items = R * heads * p.npair;
  const int grid = std::max(1, std::min(sms, n_items));
  if (mode == MK_MODE_GEMM_ONLY || R == 1) {   // K/V read from the source ranks: no ring
    p.n_items = n_items;
    return attn_launch(p, grid, s) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
  }
  if (mode == MK_MODE_FUSED) {
    p.copy = p.use_recv = p.wait = 1;
    p.n_items = n_items;
    return attn_launch(p, grid, s) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
  }
  // unfused: the ring's transfers as one launch, then the attention reading them
  p.copy = 1;
  p.n_items = 0;
  if (attn_launch(p, sms, s) != cudaSuccess) return MK_ERR_CUDA;
  p.copy = 0;
  p.use_recv = 1;
  p.n_items = n_items;
  return attn_launch(p, grid, s) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

}  // extern "C"
