// mk_fused.cu -- the persistent fused kernel behind mk_ag_gemm, mk_gemm_rs and
// mk_gemm_ar (and the grouped GEMM of mk_moe_dispatch_gemm).
//
// One launch, one CTA per SM.  Each CTA takes a ticket and with it a role
// (mKernel write-up, news.chathome.org, "mKernel的功能": CTAs assign
// themselves compute / communication / reduce roles, with the SM count per
// role tunable per shape):
//   * copy-in  (AllGather): moves remote row shards into the gathered A with
//     bulk async copies and releases one ready flag per 128-row chunk;
//   * compute: persistent tile loop, TMA -> 4-stage smem ring -> tcgen05.mma
//     into a double-buffered TMEM accumulator -> epilogue (bf16/fp32 store, or
//     an fp32 partial tile + ready flag);
//   * reduce (ReduceScatter / AllReduce): waits until all partial tiles of an
//     output tile are flagged, sums them in rank order and writes the owner's
//     block (or every replica).
// Tiles are consumed / reduced as soon as their inputs land ("五种融合内核"
// table: each A tile is consumed on arrival; each output tile is reduced and
// forwarded to its owner as soon as it is produced).
//
// Every wait (mbarrier phase, ready flag) is bounded by p.wait_ns of
// %globaltimer time; on expiry the CTA records MK_ERR_TIMEOUT in the
// workspace header, raises the abort word so that every other CTA stops at
// its next wait, drains its own copies in flight, frees its tensor memory and
// returns.
#include "mk_internal.h"
#include "mk_ptx.cuh"

namespace mk {

constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, true);
constexpr uint32_t IDESC_PAIR = idesc_bf16_f32(2 * BM, BN, false, true);   // M = 256 across the pair
constexpr uint32_t IDESC_F8 = idesc_e4m3_f32(BM, BN);                        // fp8: both operands K-major
constexpr uint32_t IDESC_F8_PAIR = idesc_e4m3_f32(2 * BM, BN);

// ------------------------------------------------------------------ errors / waits
__device__ __forceinline__ bool aborted(const FusedParams& p) {
  return ld_volatile(&p.hdr[HDR_ABORT]) == p.epoch;
}

__device__ __noinline__ void raise_error(const FusedParams& p, int code, int where, int item) {
  int* st = reinterpret_cast<int*>(&p.hdr[HDR_STATUS]);
  if (atomicCAS(st, 0, code) == 0) {
    atomicExch(reinterpret_cast<int*>(&p.hdr[HDR_DETAIL]), where * 1000000 + (item % 1000000));
  }
  __threadfence();
  atomicExch(&p.hdr[HDR_ABORT], p.epoch);
}

// Bounds check of the MK_DEBUG_BOUNDS build (true when the check passes; the
// default build compiles it to true).
__device__ __forceinline__ bool bounds_ok(const FusedParams& p, bool cond, int code, long long index) {
#if MK_DEBUG_BOUNDS
  if (!cond) {
    raise_error(p, MK_ERR_INVALID, WHERE_BOUNDS, code * 10000 + static_cast<int>(index % 10000));
    return false;
  }
#else
  (void)p; (void)cond; (void)code; (void)index;
#endif
  return true;
}

// Bounded mbarrier wait.  honor_abort = false is used only to drain copies
// that are known to be in flight (they complete on their own).  The first
// test is inline (wait_bar below): a call into this loop costs the calling
// thread a few hundred cycles even when the phase has already completed.
__device__ __noinline__ bool wait_bar_loop(const FusedParams& p, uint32_t bar, uint32_t parity, int where,
                                           int item, bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++it & 31u) == 0) {
      if (honor_abort && aborted(p)) return false;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
        raise_error(p, MK_ERR_TIMEOUT, where, item);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(const FusedParams& p, uint32_t bar, uint32_t parity, int where,
                                         int item, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_loop(p, bar, parity, where, item, honor_abort);
}

// The same wait by a whole warp that stays converged (the MMA warp): every
// lane tests the barrier and the warp agrees by vote -- cheaper for the issuing
// warp than one lane polling while the others wait -- and lane 0 reports a
// timeout.  Called by all 32 lanes.
__device__ __noinline__ bool wait_bar_warp_loop(const FusedParams& p, uint32_t bar, uint32_t parity, int where,
                                                int item, bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    if ((++it & 31u) == 0) {
      int stop = 0;
      if ((threadIdx.x & 31) == 0) {
        if (honor_abort && aborted(p)) {
          stop = 1;
        } else if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
          raise_error(p, MK_ERR_TIMEOUT, where, item);
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0) != 0) return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar_warp(const FusedParams& p, uint32_t bar, uint32_t parity, int where,
                                              int item, bool honor_abort = true) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  return wait_bar_warp_loop(p, bar, parity, where, item, honor_abort);
}

// Bounded wait until *f == epoch (acquire, gpu scope).  Single thread.  The
// first load is inline (wait_flag below).
__device__ __noinline__ bool wait_flag_loop(const FusedParams& p, const uint32_t* f, int where, int item) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (ld_acquire_gpu(f) != p.epoch) {
    if ((++it & 7u) == 0) {
      if (aborted(p)) return false;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
        raise_error(p, MK_ERR_TIMEOUT, where, item);
        return false;
      }
    }
    __nanosleep(100);
  }
  return true;
}

__device__ __forceinline__ bool wait_flag(const FusedParams& p, const uint32_t* f, int where, int item) {
  if (ld_acquire_gpu(f) == p.epoch) return true;
  return wait_flag_loop(p, f, where, item);
}

// AG copy warps: chunk mb is ready when its piece counter (the first word of
// the chunk's flag slot) reaches pieces(mb).  The CTA with ticket 0 zeroes
// the counters at kernel start and then releases hdr[HDR_READY] = epoch;
// nobody touches a counter before seeing that word.
__device__ __forceinline__ uint32_t* chunk_counter(const FusedParams& p, int mb) {
  return p.chunk_cnt + static_cast<size_t>(mb) * COPY_SUB_MAX;
}
__device__ __forceinline__ int chunk_pieces(const FusedParams& p, int mb) {
  const int rows = min(BM, p.M - mb * BM);
  return (rows + p.copy_rows - 1) / p.copy_rows;
}
// Bounded wait until the counter *c reaches `want` (single thread); the first
// load is inline (wait_count below).
__device__ __noinline__ bool wait_count_loop(const FusedParams& p, const uint32_t* c, uint32_t want, int item) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (ld_acquire_gpu(c) != want) {
    if ((++it & 7u) == 0) {
      if (aborted(p)) return false;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
        raise_error(p, MK_ERR_TIMEOUT, WHERE_PRODUCER, item);
        return false;
      }
    }
    __nanosleep(64);
  }
  return true;
}
__device__ __forceinline__ bool wait_count(const FusedParams& p, const uint32_t* c, uint32_t want, int item) {
  if (ld_acquire_gpu(c) == want) return true;
  return wait_count_loop(p, c, want, item);
}
__device__ __forceinline__ bool wait_chunk_count(const FusedParams& p, int mb, int item) {
  return wait_count(p, chunk_counter(p, mb), static_cast<uint32_t>(chunk_pieces(p, mb)), item);
}

// ------------------------------------------------------------------ work decoding
struct Item {
  int mb, nb;       // tile coordinates in the op's output space
  int arow;         // A row coordinate inside map tmA[amap]
  int amap, bmap;   // first maps; segment s uses amap+s / bmap+s
  int nseg;         // K segments (RS/AR GEMM-only: one per rank)
  int kb0, nkb;     // k-block range within each segment
  int wait_chunk;   // AG: chunk flag to wait for (-1 = none)
  int slot;         // RS/AR fused: partial slot index (-1 = write the output)
  int bz;           // MoE: local expert (3-D B map); -1 = 2-D B map
  int row_lo, row_hi;  // valid tile rows [row_lo, row_hi) (tile-relative)
  int out_row0;     // output row of tile row 0
  int phase;        // chained MLP: 1 = up-projection tile (of rank hid_r), 2 = down-projection; else 0
  int hid_r;
  int rep;          // AR GEMM-only: the one replica this item stores (-1: all of them)
};

// Grouped raster over (m-position, n-block): group_m m-positions per group,
// n-blocks outer inside a group.  An m-position is an m-block, or with CTA
// pairs the m-block pair {2q, 2q+1}.
__device__ __forceinline__ void raster(const FusedParams& p, int q, int& mb, int& nb) {
  const int gm = p.group_m;
  const int per_group = gm * p.n_nblk;
  const int g = q / per_group;
  const int first_m = g * gm;
  const int gsz = min(p.n_mrow - first_m, gm);
  const int r = q - g * per_group;
  mb = first_m + r % gsz;
  nb = r / gsz;
}

// AG: m-block processed at position `pos` of the compute order (local shard
// first, then remote shards in ring order local+1, local+2, ...).
__device__ __forceinline__ int ag_compute_mb(const FusedParams& p, int pos) {
  if (!p.ordered) return pos;
  const int bps = p.m_r / BM;
  const int q = pos / bps, i = pos - q * bps;
  const int s = (p.local + q) % p.R;
  return s * bps + i;
}
// AG: chunk copied at position `c` of the copy order (remote shards in ring
// order local+1, ..., then the local shard if it has to be copied).
__device__ __forceinline__ int ag_copy_mb(const FusedParams& p, int c) {
  if (!p.ordered) return c;
  const int bps = p.m_r / BM;
  const int q = c / bps, i = c - q * bps;
  const int s = (p.local + 1 + q) % p.R;
  return s * bps + i;
}
__device__ __forceinline__ bool ag_chunk_fully_local(const FusedParams& p, int mb) {
  const long long lo = static_cast<long long>(mb) * BM;
  const long long hi = min(lo + BM, static_cast<long long>(p.M));
  const long long l0 = static_cast<long long>(p.local) * p.m_r;
  return lo >= l0 && hi <= l0 + p.m_r;
}

// Item i of the work list, as seen by CTA `rank` of a pair (0 without pairs).
// With pairs an item covers two m-blocks; CTA r takes m-position 2q + r.  A
// half past the last m-block is empty: its loads read the zero fill beyond
// the matrix and it stores nothing and touches no flag.
__device__ __forceinline__ void empty_half(Item& it, int mb) {
  it.mb = mb;
  it.slot = -1;
  it.wait_chunk = -1;
  it.arow = mb * BM;
  it.out_row0 = mb * BM;
  it.row_hi = 0;
}

// Chained MLP up-projection: m-positions per raster group (see decode).
constexpr int MLP_GROUP_M = 8;

__device__ __forceinline__ bool decode(const FusedParams& p, int i, Item& it, int rank = 0) {
  it.bz = -1;
  it.slot = -1;
  it.wait_chunk = -1;
  it.nseg = 1;
  it.amap = 0;
  it.bmap = 0;
  it.kb0 = 0;
  it.nkb = p.n_kblk;
  it.row_lo = 0;
  it.row_hi = BM;
  it.phase = 0;
  it.hid_r = 0;
  it.rep = -1;
  if (p.op == OP_MLP && i < p.mlp_n1) {
    // up-projection of every rank in groups of MLP_GROUP_M m-positions: inside
    // a group rank-major, then n-block, then the group's m-positions, so that
    // a panel of W1_r is read once per group and reused from L2 by the group's
    // row blocks (row-block-major order streamed all of W1 once per row block)
    const int per_m = p.R * p.mlp_nb1;
    const int g = i / (MLP_GROUP_M * per_m);
    const int Gg = min(MLP_GROUP_M, p.n_mrow - g * MLP_GROUP_M);
    const int iin = i - g * MLP_GROUP_M * per_m;
    it.hid_r = iin / (Gg * p.mlp_nb1);
    const int rem = iin - it.hid_r * Gg * p.mlp_nb1;
    it.nb = rem / Gg;
    int pos = g * MLP_GROUP_M + (rem - it.nb * Gg);
    it.phase = 1;
    it.amap = 0;
    it.bmap = it.hid_r;
    it.nkb = p.mlp_kb1;
    if (p.pair) pos = 2 * pos + rank;
    if (pos >= p.n_mblk) {
      empty_half(it, pos);
      return true;
    }
    it.mb = pos;
    it.arow = pos * BM;
    it.out_row0 = pos * BM;
    it.row_hi = min(BM, p.M - it.out_row0);
    if (p.mode == MK_MODE_FUSED) it.wait_chunk = pos;
    return true;
  }
  if (p.op == OP_MLP) {
    i -= p.mlp_n1;
    it.phase = 2;
  }
  if (p.op == OP_AG) {
    int pos = i / p.n_nblk;
    it.nb = i - pos * p.n_nblk;
    if (p.pair) {
      pos = 2 * pos + rank;
      if (pos >= p.n_mblk) {
        it.amap = 1;
        empty_half(it, pos);
        return true;
      }
    }
    it.mb = ag_compute_mb(p, pos);
    it.out_row0 = it.mb * BM;
    if (p.mode == MK_MODE_FUSED && ag_chunk_fully_local(p, it.mb)) {
      it.amap = 0;
      it.arow = it.mb * BM - p.local * p.m_r;
    } else {
      it.amap = 1;
      it.arow = it.mb * BM;
      if (p.mode == MK_MODE_FUSED) it.wait_chunk = it.mb;
    }
    it.row_hi = min(BM, p.M - it.out_row0);
    return true;
  }
  if (p.op == OP_RS || p.op == OP_AR || p.op == OP_MLP) {
    if (p.mode == MK_MODE_GEMM_ONLY && p.op == OP_AR) {
      // AR baseline split over ranks, so that its few output tiles still fill
      // the chip: item (tile, rank) = that rank's product for the tile, in the
      // fused schedule's order, stored to that rank's replica (no reduction)
      const int G = p.group_tiles;
      const int g = i / (G * p.R);
      const int Gg = min(G, p.n_sched - g * G);
      const int iin = i - g * G * p.R;
      const int r = iin / Gg;
      raster(p, g * G + (iin - r * Gg), it.mb, it.nb);
      if (p.pair) it.mb = 2 * it.mb + rank;
      it.amap = r;
      it.bmap = r;
      it.rep = r;
    } else if (p.mode == MK_MODE_GEMM_ONLY) {
      raster(p, i, it.mb, it.nb);
      it.nseg = p.R;
      if (p.pair) it.mb = 2 * it.mb + rank;
    } else {
      int q, part;
      if (p.chain) {
        // Groups of group_tiles tiles; inside a group all tiles take part 0,
        // then part 1, ... so a tile's running sum moves on one part per round.
        const int G = p.group_tiles;
        const int g = i / (G * p.P);
        const int Gg = min(G, p.n_sched - g * G);
        const int iin = i - g * G * p.P;
        part = iin / Gg;
        q = g * G + (iin - part * Gg);
      } else {
        q = i / p.P;
        part = i - q * p.P;
      }
      raster(p, q, it.mb, it.nb);
      if (p.pair) it.mb = 2 * it.mb + rank;
      const int r = part / p.split_k, ks = part - r * p.split_k;
      it.amap = r;
      it.bmap = r;
      it.kb0 = ks * p.kps;
      it.nkb = min(p.kps, p.n_kblk - it.kb0);
      it.slot = (it.mb * p.n_nblk + it.nb) * p.P + part;
    }
    if (p.op == OP_MLP) {   // A = H_r (maps 1..R), B = W2_r (maps R..2R-1)
      it.amap += 1;
      it.bmap += p.R;
    }
    if (it.mb >= p.n_mblk) {
      empty_half(it, it.mb);
      return true;
    }
    it.arow = it.mb * BM;
    it.out_row0 = it.mb * BM;
    it.row_hi = min(BM, p.M - it.out_row0);
    return true;
  }
  // OP_MOE / OP_MOE_COMBINE: entry i of the tile table written by the routing kernel:
  // {dest rank d, local expert l, first row of the tile in recv_x[d], rows valid, n-block}.
  // With pairs an entry spans up to 256 rows; CTA r takes rows 128r .. 128r+127 of it.
  const int* e = p.moe_tiles + 5 * i;
  const int d = e[0];
  it.amap = d;
  it.bmap = d;
  it.bz = e[1];
  it.arow = e[2] + (p.pair ? BM * rank : 0);
  it.out_row0 = it.arow;
  it.row_hi = p.pair ? max(0, min(BM, e[3] - BM * rank)) : e[3];
  it.nb = e[4];
  it.mb = d;  // output buffer index
  return true;
}

// ------------------------------------------------------------------ compute role
// Barrier block of a compute CTA (8-byte mbarriers), then the TMEM base slot.
// With pairs, both CTAs lay it out alike: the leader's full and TMEM-empty
// barriers gate the pair, each CTA's empty and TMEM-full barriers are
// signalled by the leader's multicast commits.
constexpr uint32_t BAR_FULL = 0;
constexpr uint32_t BAR_EMPTY = BAR_FULL + 8u * MAX_STAGES;
constexpr uint32_t BAR_TFULL = BAR_EMPTY + 8u * MAX_STAGES;
constexpr uint32_t BAR_TEMPTY = BAR_TFULL + 16u;
constexpr uint32_t BAR_DRAIN = BAR_TEMPTY + 16u;
constexpr uint32_t BAR_PDONE = BAR_DRAIN + 8u;
constexpr uint32_t TMEM_SLOT = BAR_PDONE + 16u;
static_assert(TMEM_SLOT + 4 <= BAR_BYTES, "compute barriers exceed the barrier block");

// MoE combine queue: control words (u32 index) and entries (byte offset) in the queue block.
enum { CQ_TAIL = 0, CQ_CLAIM = 1, CQ_DONE = 2 };
constexpr uint32_t CQ_ENT = 64;

struct ComputeSmem {
  uint32_t ring;  // smem address of stage 0
  uint32_t bars;  // smem address of the barrier block
  uint32_t cq;    // smem address of the MoE combine queue block
  uint32_t* cq_ctl;   // the same block, generic pointer (control words)
  uint32_t epi;   // smem address of the epilogue staging (EPI_WARP_BYTES per epilogue warp)
  __device__ __forceinline__ uint32_t full(int s) const { return bars + BAR_FULL + 8u * s; }
  __device__ __forceinline__ uint32_t empty(int s) const { return bars + BAR_EMPTY + 8u * s; }
  __device__ __forceinline__ uint32_t tfull(int b) const { return bars + BAR_TFULL + 8u * b; }
  __device__ __forceinline__ uint32_t tempty(int b) const { return bars + BAR_TEMPTY + 8u * b; }
  __device__ __forceinline__ uint32_t drain() const { return bars + BAR_DRAIN; }
  __device__ __forceinline__ uint32_t pdone(int b) const { return bars + BAR_PDONE + 8u * b; }
};

// Ring geometry of the two compute variants.  With pairs a stage holds two
// consecutive k-blocks of a segment (each A + this CTA's half of B): the MMA
// issuer then waits once and commits once per 8 MMAs -- a satisfied mbarrier
// wait in the issuing thread costs on the order of a hundred cycles that the
// tensor pipe's short queue cannot hide.
template <bool PAIR>
struct Ring {
  static constexpr int kps = PAIR ? 2 : 1;                                   // k-blocks per stage
  static constexpr uint32_t kb_bytes = PAIR ? PSTAGE_BYTES : STAGE_BYTES;    // one k-block's part
  static constexpr int stages = (PAIR ? PSTAGES : STAGES) / kps;
  static constexpr uint32_t stage_bytes = kb_bytes * kps;
};

__device__ __forceinline__ int n_items_for(const FusedParams& p) {
  if (p.op == OP_MOE && p.mode == MK_MODE_UNFUSED) return 0;   // baseline: dispatch copy only
  if (p.op == OP_MOE || p.op == OP_MOE_COMBINE)
    return min(ld_acquire_gpu(reinterpret_cast<const uint32_t*>(p.moe_ntiles)),
               static_cast<uint32_t>(p.n_items));
  return p.n_items;
}

// In-kernel trace (mk_config.trace): word w of the record of (item i, pair rank).
// Words: 0 producer takes the item, 1 its inputs are ready, 2 its last load is
// issued, 3 accumulator ready, 4 epilogue done (all %globaltimer ns); 5 / 6 the
// SM's clock64 at 0 / 3; 7 epoch << 32 | CTA << 1 | pair rank.
constexpr int TRACE_WORDS = 8;
__device__ __forceinline__ void trace_put(const FusedParams& p, int i, uint32_t rank, int w,
                                          unsigned long long v) {
  const int idx = 2 * i + static_cast<int>(rank);
  if (p.trace != nullptr && idx < p.trace_cap)
    p.trace[static_cast<size_t>(idx) * TRACE_WORDS + w] = v;
}
// Copy-warp records follow the item records: record trace_cap + worker holds
// [0] start ns (after the kernel-start handshake), [1] end ns (last piece
// released), [2] pieces copied, [3] bytes copied, [7] epoch << 32 | worker.
__device__ __forceinline__ void trace_copy(const FusedParams& p, int worker, unsigned long long t0,
                                           unsigned long long pieces, unsigned long long bytes) {
  if (p.trace == nullptr || worker >= MK_TRACE_COPY_RECORDS) return;
  unsigned long long* r = p.trace + (static_cast<size_t>(p.trace_cap) + worker) * TRACE_WORDS;
  r[0] = t0;
  r[1] = globaltimer_ns();
  r[2] = pieces;
  r[3] = bytes;
  r[7] = (static_cast<unsigned long long>(p.epoch) << 32) | static_cast<unsigned long long>(worker);
}
__device__ __forceinline__ void trace_end(const FusedParams& p, int i, uint32_t rank) {
  if (p.trace == nullptr) return;
  trace_put(p, i, rank, 4, globaltimer_ns());
  trace_put(p, i, rank, 7, (static_cast<unsigned long long>(p.epoch) << 32) |
                               (static_cast<unsigned long long>(blockIdx.x) << 1) | rank);
}

// MoE dispatch: whether every row of the item has landed, from one round trip
// of relaxed loads (its block counters and the rank's row count, all in flight
// together, where acquire loads would go one after another); when they have,
// the acquire fence and the proxy fence that order the item's TMA loads after
// them are taken here.  false: not yet (or an entry out of range: the caller's
// bounds checks and bounded waits take over).
__device__ bool moe_rows_ready(const FusedParams& p, const Item& it) {
  const int d = it.amap;
  if (d < 0 || d >= p.R || it.arow < 0 || it.row_hi <= 0 || it.row_hi > BM || it.arow + it.row_hi > p.M) return false;
  const int b0 = it.arow / BM, b1 = (it.arow + it.row_hi - 1) / BM;   // b1 <= b0 + 1
  const uint32_t* cnt = p.flags + static_cast<size_t>(d) * p.moe_nblk;
  const uint32_t v0 = ld_relaxed_gpu(cnt + b0);
  const uint32_t v1 = (b1 > b0) ? ld_relaxed_gpu(cnt + b1) : 0u;
  const int rc = p.moe_recv_counts[d];
  const uint32_t w0 = static_cast<uint32_t>(min(BM, rc - b0 * BM));
  const uint32_t w1 = (b1 > b0) ? static_cast<uint32_t>(min(BM, rc - b1 * BM)) : 0u;
  if (v0 != w0 || v1 != w1) return false;
  fence_acq_rel_gpu();
  fence_proxy_async_global();
  return true;
}

// TMA producer (one thread).  With pairs each CTA loads its own 128 rows of A
// and its 128 of the tile's 256 B columns into its own ring, completing on
// the leader's full barrier, which the leader arms with both CTAs' bytes.
template <bool PAIR>
__device__ void producer(const FusedParams& p, const ComputeSmem& S, int cid, uint32_t rank) {
  constexpr int NST = Ring<PAIR>::stages;
  constexpr uint32_t SB = Ring<PAIR>::stage_bytes;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued_mask = 0, issued_par = 0;
  const int n_items = n_items_for(p);
  bool counters_ready = false;
  const bool moe_wait = (p.op == OP_MOE && p.mode == MK_MODE_FUSED);
  for (int i = cid; i < n_items; i += p.n_compute) {
    Item it;
    decode(p, i, it, static_cast<int>(rank));
    // the next item's tile-table entry (written by the routing kernels) into L1
    // while this item's loads are issued
    if ((p.op == OP_MOE || p.op == OP_MOE_COMBINE) && i + p.n_compute < n_items) {
      prefetch_l1(p.moe_tiles + 5 * (i + p.n_compute));
      prefetch_l1(p.moe_tiles + 5 * (i + p.n_compute) + 4);
    }
    if (p.trace != nullptr) {
      trace_put(p, i, rank, 0, globaltimer_ns());
      trace_put(p, i, rank, 5, clock64());
    }
    // the tile lies inside the output and the operands' k-blocks (MoE: inside
    // the receive buffer of a valid destination rank)
    if (!bounds_ok(p, it.row_hi >= 0 && it.row_hi <= BM && it.out_row0 >= 0 && it.arow >= 0 &&
                          (it.row_hi == 0 || it.out_row0 + it.row_hi <= p.M) && it.nb >= 0 &&
                          it.nb < (it.phase == 1 ? p.mlp_nb1 : p.n_nblk),
                   BC_TILE, i))
      goto done;
    if (!bounds_ok(p, it.kb0 >= 0 && it.nkb >= 0 && it.kb0 + it.nkb <= (it.phase == 1 ? p.mlp_kb1 : p.n_kblk) &&
                          it.amap >= 0 && it.amap + it.nseg <= MK_MAX_RANKS && it.bmap >= 0 &&
                          it.bmap + it.nseg <= MK_MAX_RANKS,
                   BC_KRANGE, i))
      goto done;
    if ((p.op == OP_MOE || p.op == OP_MOE_COMBINE) &&
        !bounds_ok(p, it.amap < p.R && it.bz >= 0 && (it.row_hi == 0 || it.arow + it.row_hi <= p.M),
                   BC_MOE_TILE, i))
      goto done;
    if (moe_wait && it.row_hi > 0 && !moe_rows_ready(p, it)) {
      // the tile's rows must have landed: every 128-row block of recv_x[d] it covers
      // (an empty pair half covers no rows and waits for nothing)
      const int d = it.amap;
      const int rc = p.moe_recv_counts[d];
      const int b0 = it.arow / BM, b1 = (it.arow + it.row_hi - 1) / BM;
      for (int b = b0; b <= b1; ++b) {
        const uint32_t want = static_cast<uint32_t>(min(BM, rc - b * BM));
        if (!wait_count(p, p.flags + static_cast<size_t>(d) * p.moe_nblk + b, want, i)) goto done;
      }
      fence_proxy_async_global();
    }
    if (it.wait_chunk >= 0 && p.copy_warps && !counters_ready) {
      if (!wait_flag(p, &p.hdr[HDR_READY], WHERE_PRODUCER, i)) goto done;
      counters_ready = true;
    }
    if (it.wait_chunk >= 0) {
      if (p.copy_warps) {
        if (!wait_chunk_count(p, it.wait_chunk, i)) goto done;
      } else {
        for (int j = 0; j < p.copy_sub; ++j)
          if (!wait_flag(p, p.flags + it.wait_chunk * COPY_SUB_MAX + j, WHERE_PRODUCER, i)) goto done;
      }
      fence_proxy_async_global();
    }
    if (p.trace != nullptr) trace_put(p, i, rank, 1, globaltimer_ns());
    for (int seg = 0; seg < it.nseg; ++seg) {
      const CUtensorMap* ma = &p.tmA[it.amap + seg];
      const CUtensorMap* mbm = &p.tmB[it.bmap + seg];
      if (it.phase == 2 && it.row_hi > 0 && p.mlp_wait) {
        // chained MLP: every up-projection tile of this row block of H_r has been stored
        if (!counters_ready) {
          if (!wait_flag(p, &p.hdr[HDR_READY], WHERE_PRODUCER, i)) goto done;
          counters_ready = true;
        }
        const int r = it.amap + seg - 1;
        if (!wait_count(p, p.mlp_cnt + static_cast<size_t>(r) * p.n_mblk + it.mb,
                        static_cast<uint32_t>(p.mlp_nb1), i))
          goto done;
        fence_proxy_async_global();
      }
      const int kend = it.kb0 + it.nkb;
      for (int kb0 = it.kb0; kb0 < kend; kb0 += Ring<PAIR>::kps) {
        if (!wait_bar(p, S.empty(stage), phase ^ 1u, WHERE_PRODUCER, i)) goto done;
        const int n0 = it.nb * BN;
        if constexpr (PAIR) {
          const int nk = min(Ring<PAIR>::kps, kend - kb0);   // k-blocks in this stage
          const uint32_t fb = mapa_shared(S.full(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(S.full(stage), 2u * PSTAGE_BYTES * static_cast<uint32_t>(nk));
          const int c0 = n0 / 64 + 2 * static_cast<int>(rank);   // this CTA's first column chunk
          for (int h = 0; h < nk; ++h) {
            const int kb = kb0 + h;
            const int kx = kb * (p.fp8 ? 2 * BK : BK);   // K coordinate (elements) of the k-block
            const uint32_t a_dst = S.ring + static_cast<uint32_t>(stage) * SB + static_cast<uint32_t>(h) * PSTAGE_BYTES;
            const uint32_t b_dst = a_dst + A_STAGE_BYTES;
            tma_load_2d_pair(a_dst, ma, fb, kx, it.arow);
            if (p.fp8) {   // B^T [n x k]: this CTA's 128 rows of the tile's 256
              tma_load_2d_pair(b_dst, mbm, fb, kx, n0 + 128 * static_cast<int>(rank));
            } else if (p.b_one_box) {
              if (it.bz < 0) tma_load_3d_pair(b_dst, mbm, fb, 0, kx, c0);
              else tma_load_4d_pair(b_dst, mbm, fb, 0, kx, c0, it.bz);
            } else if (it.bz < 0) {
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tma_load_2d_pair(b_dst + j * B_BOX_BYTES, mbm, fb, 64 * (c0 + j), kx);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tma_load_3d_pair(b_dst + j * B_BOX_BYTES, mbm, fb, 64 * (c0 + j), kx, it.bz);
            }
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        const int kb = kb0;
        const uint32_t a_dst = S.ring + static_cast<uint32_t>(stage) * SB;
        const uint32_t b_dst = a_dst + A_STAGE_BYTES;
        mbar_arrive_expect_tx(S.full(stage), STAGE_BYTES);
        if (p.fp8) {   // 128-element k-blocks; B^T [n x k]: the tile's 256 rows in one box
          tma_load_2d(a_dst, ma, S.full(stage), kb * 2 * BK, it.arow);
          tma_load_2d(b_dst, mbm, S.full(stage), kb * 2 * BK, n0);
        } else {
        tma_load_2d(a_dst, ma, S.full(stage), kb * BK, it.arow);
        if (p.b_one_box) {
          // the whole BK x 256 B tile in one request (4 column chunks of 64)
          if (it.bz < 0) tma_load_3d(b_dst, mbm, S.full(stage), 0, kb * BK, n0 / 64);
          else tma_load_4d(b_dst, mbm, S.full(stage), 0, kb * BK, n0 / 64, it.bz);
        } else if (it.bz < 0) {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(b_dst + j * B_BOX_BYTES, mbm, S.full(stage), n0 + 64 * j, kb * BK);
        } else {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_3d(b_dst + j * B_BOX_BYTES, mbm, S.full(stage), n0 + 64 * j, kb * BK, it.bz);
        }
        }
        issued_mask |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (p.trace != nullptr) trace_put(p, i, rank, 2, globaltimer_ns());
  }
done:
  // Every load issued must have landed before the CTA may exit.  With pairs
  // the leader's full barriers also count the peer's loads; the peer's own
  // loads of a stage the leader never armed (abort only) are waited out by
  // the pause before the pair's final cluster barrier.
  if (PAIR && rank != 0) return;
  for (int s = 0; s < NST; ++s)
    if (issued_mask & (1u << s))
      wait_bar(p, S.full(s), (issued_par >> s) & 1u, WHERE_DRAIN, s, /*honor_abort=*/false);
}

// MMA issuer (one thread; with pairs only the leader's).  A pair's MMA has
// M = 256: rows 0-127 from the leader's A stage, 128-255 from the peer's, and
// the B columns from both CTAs' halves; each CTA's TMEM receives its own rows.
template <bool PAIR, bool F8>
__device__ void mma_issuer(const FusedParams& p, const ComputeSmem& S, uint32_t tmem_base, int cid) {
  constexpr int NST = Ring<PAIR>::stages;
  constexpr uint32_t SB = Ring<PAIR>::stage_bytes;
  int stage = 0;
  uint32_t phase = 0;
  int buf = 0;
  uint32_t acc_phase = 0;
  const int n_items = n_items_for(p);
  for (int i = cid; i < n_items; i += p.n_compute) {
    Item it;
    decode(p, i, it);
    if (!wait_bar_warp(p, S.tempty(buf), acc_phase ^ 1u, WHERE_MMA, i)) goto done;
    tc_fence_after();
    {
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
      uint32_t acc = 0;
      for (int seg = 0; seg < it.nseg; ++seg) {
        for (int kb0 = 0; kb0 < it.nkb; kb0 += Ring<PAIR>::kps) {
          const int nk = min(Ring<PAIR>::kps, it.nkb - kb0);   // k-blocks in this stage
          if (!wait_bar_warp(p, S.full(stage), phase, WHERE_MMA, i)) goto done;
          tc_fence_after();
          if (elect_one_sync()) {
            for (int h = 0; h < nk; ++h) {
              const uint32_t a_addr =
                  S.ring + static_cast<uint32_t>(stage) * SB + static_cast<uint32_t>(h) * Ring<PAIR>::kb_bytes;
              const uint32_t b_addr = a_addr + A_STAGE_BYTES;
              if constexpr (F8) {
                // fp8: four K = 32 steps of 32 bytes; A and B^T both K-major, 128-byte
                // swizzle, 8-row groups 1024 B apart
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t ad = sdesc_swz(a_addr + 32u * k, 16u, 1024u, 2u);
                  const uint64_t bd = sdesc_swz(b_addr + 32u * k, 16u, 1024u, 2u);
                  if constexpr (PAIR) tc_mma_f8_pair(d_tmem, ad, bd, IDESC_F8_PAIR, acc);
                  else tc_mma_f8(d_tmem, ad, bd, IDESC_F8, acc);
                  acc = 1;
                }
                continue;
              }
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                // A: K-major, BK*2-byte swizzle, 8-row atoms 8*BK*2 B apart; +32 B per 16-wide K step.
                const uint64_t ad = sdesc_swz(a_addr + 32u * k, 16u, 8u * A_SWIZZLE_BYTES,
                                              A_SWIZZLE_BYTES == 128 ? 2u : 4u);
                // B: MN-major, 128-B swizzle; 64-column atoms 8 KiB apart (LBO),
                // 8-row K groups 1024 B apart (SBO); +2048 B per 16-row K step.
                const uint64_t bd = sdesc_sw128(b_addr + 2048u * k, static_cast<uint32_t>(B_BOX_BYTES), 1024u);
                if constexpr (PAIR) tc_mma_bf16_pair(d_tmem, ad, bd, IDESC_PAIR, acc);
                else tc_mma_bf16(d_tmem, ad, bd, IDESC, acc);
                acc = 1;
              }
            }
            if constexpr (PAIR) tc_commit_pair(S.empty(stage), 3);
            else tc_commit(S.empty(stage));
          }
          __syncwarp();
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    if (elect_one_sync()) {
      if constexpr (PAIR) tc_commit_pair(S.tfull(buf), 3);
      else tc_commit(S.tfull(buf));
    }
    __syncwarp();
    if (++buf == 2) {
      buf = 0;
      acc_phase ^= 1u;
    }
  }
done:
  // Every MMA issued must have completed before tensor memory is freed.
  if (elect_one_sync()) {
    if constexpr (PAIR) tc_commit_pair(S.drain(), 1);
    else tc_commit(S.drain());
  }
  __syncwarp();
  wait_bar_warp(p, S.drain(), 0, WHERE_DRAIN, 0, /*honor_abort=*/false);
}

__device__ __forceinline__ void store_row_chunk(void* dst, const uint32_t (&r)[32], int ncols_valid,
                                                bool f32) {
  // dst: first of 32 consecutive output columns of one row; ncols_valid in [0, 32], multiple of 8.
  if (f32) {
    float* d = reinterpret_cast<float*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (4 * q < ncols_valid) st_global_v4(d + 4 * q, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
  } else {
    uint16_t* d = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (8 * q < ncols_valid) {
        const uint32_t w0 = pack_bf16x2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
        const uint32_t w1 = pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
        const uint32_t w2 = pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
        const uint32_t w3 = pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
        st_global_v4(d + 8 * q, w0, w1, w2, w3);
      }
    }
  }
}

// Last-arrival reduction: one counter per (tile, 32-row quarter), zeroed at
// kernel start by the CTA with ticket 0 (published by hdr[HDR_READY]).
// Returns the number of partials of this quarter stored before this one.
__device__ __forceinline__ uint32_t bump_quarter(const FusedParams& p, int tile, int quarter) {
  return atomicAdd(p.flags + static_cast<size_t>(tile) * 4 + quarter, 1u);
}

// Rows of one warp quarter of a tile: sum of `nparts` staged fp32 tiles
// starting at `base`, in order, rounded and written to the owner block (RS)
// or every replica (AR).  nparts = 1 converts an accumulated tile.
__device__ void reduce_quarter(const FusedParams& p, const Item& it, const float* base, int nparts, int trow,
                               bool row_ok, int grow) {
  const size_t esz = p.out_f32 ? 4 : 2;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float4 acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      acc[q] = ld_global_cg_f4(base + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4);
    int part = 1;
    for (; part + 1 < nparts; part += 2) {
      float4 v0[8], v1[8];
      const float* s0 = base + static_cast<size_t>(part) * TILE_F32;
      const float* s1 = s0 + TILE_F32;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v0[q] = ld_global_cg_f4(s0 + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4);
        v1[q] = ld_global_cg_f4(s1 + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        acc[q].x += v0[q].x; acc[q].y += v0[q].y; acc[q].z += v0[q].z; acc[q].w += v0[q].w;
        acc[q].x += v1[q].x; acc[q].y += v1[q].y; acc[q].z += v1[q].z; acc[q].w += v1[q].w;
      }
    }
    if (part < nparts) {
      const float* s0 = base + static_cast<size_t>(part) * TILE_F32;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = ld_global_cg_f4(s0 + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4);
        acc[q].x += v.x; acc[q].y += v.y; acc[q].z += v.z; acc[q].w += v.w;
      }
    }
    const int col = it.nb * BN + 32 * c;
    const int nvalid = max(0, min(32, p.N - col));
    if (!row_ok || nvalid == 0) continue;
    uint32_t r[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      r[4 * q + 0] = __float_as_uint(acc[q].x);
      r[4 * q + 1] = __float_as_uint(acc[q].y);
      r[4 * q + 2] = __float_as_uint(acc[q].z);
      r[4 * q + 3] = __float_as_uint(acc[q].w);
    }
    if (p.op != OP_AR) {
      const int o = grow / p.rows_per_owner, lr = grow - o * p.rows_per_owner;
      uint8_t* ob = reinterpret_cast<uint8_t*>(p.out[o]);
      store_row_chunk(ob + (static_cast<size_t>(lr) * p.N + col) * esz, r, nvalid, p.out_f32);
    } else {
      for (int o = 0; o < p.R; ++o) {
        uint8_t* ob = reinterpret_cast<uint8_t*>(p.out[o]);
        store_row_chunk(ob + (static_cast<size_t>(grow) * p.N + col) * esz, r, nvalid, p.out_f32);
      }
    }
  }
}

// Final stores through the warp's staging: this lane's row piece (32 columns:
// 128 bytes of fp32 or 64 bytes of bf16, at byte `off` of the staged 128-byte
// row segment) goes to shared memory; flush_staged then writes the warp's 32
// rows x 128 bytes with lane l taking 16 bytes of row 4k + l/8, so each store
// instruction covers four whole 128-byte row segments (a lane per row would
// make 32 separate 16-byte writes of one instruction).
__device__ __forceinline__ void stage_piece(uint32_t stage, int lane, int off, const uint32_t (&r)[32], bool f32) {
  const uint32_t a = stage + static_cast<uint32_t>(lane * EPI_ROW_STRIDE + off);
  if (f32) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16u * q), "r"(r[4 * q]), "r"(r[4 * q + 1]),
                   "r"(r[4 * q + 2]), "r"(r[4 * q + 3]) : "memory");
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16u * q),
                   "r"(pack_bf16x2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]))),
                   "r"(pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]))),
                   "r"(pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]))),
                   "r"(pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7])))
                   : "memory");
  }
}
// The staged segment (columns col0 .. col0 + 128/esz - 1 of the warp's 32 rows,
// tile rows 32 quarter + 0 .. 31) to the output: every replica (AR) or the
// owner's row block (RS, the chained MLP).  Rows outside [row_lo, row_hi) and
// columns at or past N are skipped.
__device__ __forceinline__ void flush_staged(const FusedParams& p, const Item& it, uint32_t stage, int lane,
                                             int quarter, int col0) {
  const int esz = p.out_f32 ? 4 : 2;
  const int pc = col0 + (lane & 7) * (16 / esz);   // first column of this lane's 16-byte piece
  const bool col_ok = pc + 16 / esz <= p.N;
#pragma unroll 1
  for (int k = 0; k < 8; ++k) {
    const int row = 4 * k + (lane >> 3);
    const int trow = quarter * 32 + row;
    uint32_t v0, v1, v2, v3;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                 : "r"(stage + static_cast<uint32_t>(row * EPI_ROW_STRIDE + (lane & 7) * 16))
                 : "memory");
    if (!col_ok || trow < it.row_lo || trow >= it.row_hi) continue;
    const int grow = it.out_row0 + trow;
    if (p.op == OP_AR) {
      for (int o = 0; o < p.R; ++o)
        st_global_v4(reinterpret_cast<uint8_t*>(p.out[o]) + (static_cast<size_t>(grow) * p.N + pc) * esz, v0, v1,
                     v2, v3);
    } else {
      const int o = grow / p.rows_per_owner, lr = grow - o * p.rows_per_owner;
      st_global_v4(reinterpret_cast<uint8_t*>(p.out[o]) + (static_cast<size_t>(lr) * p.N + pc) * esz, v0, v1, v2,
                   v3);
    }
  }
}

// One 32-column chunk of the warp's 32 rows stored through its staging: lane
// l's piece goes to shared memory, and once a 128-byte segment of every row
// is staged (two bf16 chunks, one fp32 chunk) the warp writes it out, lane l
// taking 16 bytes of row 4j + l/8, so each store instruction covers four whole
// 128-byte row segments instead of 32 separate 16-byte pieces.  row_ptr: this
// lane's row (byte address of column 0), 0 to skip the row; columns at or
// past ncols are skipped.  Called by all 32 lanes, chunks c = 0, 1, ... in order.
__device__ __forceinline__ void staged_chunk(uint32_t stage, int lane, int c, const uint32_t (&r)[32], bool f32,
                                             unsigned long long row_ptr, int n0, int ncols) {
  const int per = f32 ? 1 : 2;   // chunks per staged 128-byte segment
  stage_piece(stage, lane, (c % per) * 64, r, f32);
  if (c % per != per - 1) return;
  __syncwarp();
  const int esz = f32 ? 4 : 2;
  const int pc = n0 + 32 * (c - per + 1) + (lane & 7) * (16 / esz);   // first column of this lane's piece
#pragma unroll 1
  for (int j = 0; j < 8; ++j) {
    const int row = 4 * j + (lane >> 3);
    const unsigned long long dst = __shfl_sync(0xffffffffu, row_ptr, row);
    uint32_t v0, v1, v2, v3;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                 : "r"(stage + static_cast<uint32_t>(row * EPI_ROW_STRIDE + (lane & 7) * 16))
                 : "memory");
    if (dst != 0ull && pc + 16 / esz <= ncols)
      st_global_v4(reinterpret_cast<uint8_t*>(dst) + static_cast<size_t>(pc) * esz, v0, v1, v2, v3);
  }
  __syncwarp();
}

// fp32 load through L2 (not L1) with an L2 eviction policy.
__device__ __forceinline__ float4 ld_cg_f4_pol(const float* ptr, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.cg.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}

// Sliced reduction (reduce = 4), after the warp's own tiles: job j = (tile,
// 32-row quarter, 64-column group).  An epilogue warp that has finished its own
// tiles claims the next job from a counter in the header, so the jobs go out
// in tile order (the order the tiles' partials complete in) to whichever warps
// are free first: warps of CTAs with fewer items sum the first tiles while the
// last wave still runs.  Once the quarter's arrival count shows all P partials
// staged, the warp sums its slice of them in rank order 0..P-1 (the running
// sum's order, so the result is the same bits) and writes it through its
// staging to every replica (AR) or the owner's block (RS).  The waits come after all of this CTA's own
// tiles, which wait for nothing, so every count is reached.  The partials were
// staged with an L2 evict_last policy (they stay in L2 while the operands
// stream past) and are read here with evict_first (each is read once).
__device__ void finalize_slices(const FusedParams& p, const Item& proto, uint32_t epi, int gw,
                                bool& counters_ready) {
  const int lane = threadIdx.x & 31;
  constexpr int GROUPS = BN / 64;
  const int n_jobs = p.n_tiles * 4 * GROUPS;
  const uint64_t pol_once = l2_policy_evict_first();
  while (true) {
    int j = 0;
    {
      int ok = 1;
      if (lane == 0) {
        // the claim counter is zeroed at kernel start, with the counts
        if (!counters_ready) {
          if (!wait_flag(p, &p.hdr[HDR_READY], WHERE_REDUCE, gw)) ok = 0;
          counters_ready = true;
        }
        if (ok) j = static_cast<int>(atomicAdd(&p.hdr[HDR_CLAIM], 1u));
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
      j = __shfl_sync(0xffffffffu, j, 0);
    }
    if (j >= n_jobs) break;
    const int tile = j / (4 * GROUPS), q = (j / GROUPS) % 4, g = j % GROUPS;
    const int mb = tile / p.n_nblk, nb = tile - mb * p.n_nblk;
    const int rows = min(BM, p.M - mb * BM);
    if (32 * q >= rows) continue;                   // no row of this quarter is an output row
    int ok = 1;
    if (lane == 0) {
      const uint32_t* cnt = p.flags + static_cast<size_t>(tile) * 4 + q;
      if (ok && ld_acquire_gpu(cnt) != static_cast<uint32_t>(p.P)) {
        const uint64_t t0 = globaltimer_ns();
        uint32_t it = 0;
        while (ld_acquire_gpu(cnt) != static_cast<uint32_t>(p.P)) {
          if ((++it & 7u) == 0) {
            if (aborted(p)) {
              ok = 0;
              break;
            }
            if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
              raise_error(p, MK_ERR_TIMEOUT, WHERE_REDUCE, j);
              ok = 0;
              break;
            }
          }
          __nanosleep(64);
        }
      }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    const int trow = 32 * q + lane;
    const float* base = p.staging + static_cast<size_t>(tile) * p.P * TILE_F32;
    Item it = proto;
    it.row_lo = 0;
    it.row_hi = rows;
    it.out_row0 = mb * BM;
    const int per = p.out_f32 ? 1 : 2;   // 32-column chunks per 128-byte staged segment
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * g + cc;
      float4 acc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        acc[u] = ld_cg_f4_pol(base + (static_cast<size_t>((c * 8 + u) * BM + trow)) * 4, pol_once);
      // two partials' loads in flight at a time, added in rank order
      int part = 1;
#pragma unroll 1
      for (; part + 1 < p.P; part += 2) {
        const float* s0 = base + static_cast<size_t>(part) * TILE_F32;
        const float* s1 = s0 + TILE_F32;
        float4 v0[8], v1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          v0[u] = ld_cg_f4_pol(s0 + (static_cast<size_t>((c * 8 + u) * BM + trow)) * 4, pol_once);
          v1[u] = ld_cg_f4_pol(s1 + (static_cast<size_t>((c * 8 + u) * BM + trow)) * 4, pol_once);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc[u].x += v0[u].x;
          acc[u].y += v0[u].y;
          acc[u].z += v0[u].z;
          acc[u].w += v0[u].w;
          acc[u].x += v1[u].x;
          acc[u].y += v1[u].y;
          acc[u].z += v1[u].z;
          acc[u].w += v1[u].w;
        }
      }
      if (part < p.P) {
        const float* s0 = base + static_cast<size_t>(part) * TILE_F32;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 v = ld_cg_f4_pol(s0 + (static_cast<size_t>((c * 8 + u) * BM + trow)) * 4, pol_once);
          acc[u].x += v.x;
          acc[u].y += v.y;
          acc[u].z += v.z;
          acc[u].w += v.w;
        }
      }
      uint32_t r[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        r[4 * u + 0] = __float_as_uint(acc[u].x);
        r[4 * u + 1] = __float_as_uint(acc[u].y);
        r[4 * u + 2] = __float_as_uint(acc[u].z);
        r[4 * u + 3] = __float_as_uint(acc[u].w);
      }
      stage_piece(epi, lane, (c % per) * 64, r, p.out_f32);
      if (c % per == per - 1) {
        __syncwarp();
        flush_staged(p, it, epi, lane, q, nb * BN + 32 * (c - per + 1));
        __syncwarp();
      }
    }
  }
}

// An epilogue warp is done reading TMEM buffer `buf`: arrive on the barrier
// that lets the MMA issuer overwrite it (the leader's, with pairs: it counts
// the four epilogue warps of both CTAs).
template <bool PAIR>
__device__ __forceinline__ void release_tmem(const ComputeSmem& S, int buf, uint32_t rank) {
  if (PAIR && rank != 0) mbar_arrive_cluster(mapa_shared(S.tempty(buf), 0));
  else mbar_arrive(S.tempty(buf));
}

// MoE combine epilogue of one warp (32 rows of a tile, 256 columns):
//  1. return: row j of destination rank d holds (token g, slot k) =
//     divmod(recv_src[d][j], topk); its bf16 product row goes to
//     ret[g / T][g % T][k] (columns n0 .. n0+255);
//  2. TMEM is released at once, so the next tile's MMAs may start;
//  3. last arrival: after a gpu-scope fence each lane counts its slot in the
//     (token, column block) counter; the lane that brings it to topk hands the
//     (token, column block) to the CTA's copy warps (combine_sum_role), which
//     form the gate-weighted sum while the epilogue moves on.
template <bool PAIR>
__device__ __forceinline__ void combine_epilogue(const FusedParams& p, const ComputeSmem& S, const Item& it,
                                                 uint32_t taddr, int buf, uint32_t rank, int lane, int trow,
                                                 bool row_ok, int grow, uint32_t epi) {
  const int topk = p.moe_topk, T = p.moe_T;
  const int n0 = it.nb * BN;
  int r = 0, t = 0, k = 0;
  if (row_ok) {
    const int src = p.moe_src[it.mb][grow];
    if (src < 0 || src >= p.R * T * topk) {   // not a (token, slot) of this call: skip the row
      raise_error(p, MK_ERR_INVALID, WHERE_EPILOGUE, grow);
      row_ok = false;
    } else {
      const int g = src / topk;
      k = src - g * topk;
      r = g / T;
      t = g - r * T;
    }
  }
  uint8_t* slot_row = p.moe_ret[r] + (static_cast<size_t>(t) * topk + k) * p.N * 2;
  const unsigned long long my_row = row_ok ? reinterpret_cast<unsigned long long>(slot_row) : 0ull;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t v[32];
    tc_ld_32x32b_x32(taddr + 32u * c, v);
    tc_wait_ld();
    staged_chunk(epi, lane, c, v, false, my_row, n0, p.N);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) release_tmem<PAIR>(S, buf, rank);
  if (p.mode != MK_MODE_FUSED || !row_ok) return;
  __threadfence();
  const uint32_t before = atomicAdd(p.moe_cnt + (static_cast<size_t>(r) * T + t) * p.n_nblk + it.nb, 1u);
  if (before != static_cast<uint32_t>(topk - 1)) return;
  __threadfence();   // every other slot's stores happened before its count
  // Hand (token row, column block) to the copy warps.  Entry s of the ring
  // (16 bytes: sequence word, unused, r*T + t, column block) is free for slot
  // s when its sequence word is 2s, full when it is 2s+1.
  const uint32_t slot = atomicAdd(S.cq_ctl + CQ_TAIL, 1u);
  const uint32_t e = S.cq + CQ_ENT + 16u * (slot % CQ_CAP);
  if (ld_acquire_cta_shared(e) != 2u * slot) {
    const uint64_t t0 = globaltimer_ns();
    uint32_t it2 = 0;
    while (ld_acquire_cta_shared(e) != 2u * slot) {
      if ((++it2 & 15u) == 0) {
        if (aborted(p)) return;
        if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
          raise_error(p, MK_ERR_TIMEOUT, WHERE_EPILOGUE, static_cast<int>(slot));
          return;
        }
      }
      __nanosleep(64);
    }
  }
  asm volatile("st.shared::cta.v2.u32 [%0], {%1, %2};" ::"r"(e + 8u),
               "r"(static_cast<uint32_t>(r * T + t)), "r"(static_cast<uint32_t>(it.nb)) : "memory");
  st_release_cta_shared(e, 2u * slot + 1u);
}

// MoE combine sums by the copy warps: each warp claims up to 8 handed-over rows
// at a time and sums them coalesced (lane l: columns n0 + 8l .. n0 + 8l + 7 of
// each row, 512 contiguous bytes per row and slot, 8 loads per slot in flight):
// out[r][t] = bf16(sum_k gates[r][t][k] * ret[r][t][k]) in fp32, slot order.
// A warp leaves when the four epilogue warps have finished and every
// handed-over row has been claimed (or on abort).
__device__ void combine_sum_role(const FusedParams& p, const ComputeSmem& S) {
  const int lane = threadIdx.x & 31;
  const int topk = p.moe_topk, T = p.moe_T;
  constexpr int CW = 8;
  const uint64_t t_start = globaltimer_ns();
  uint64_t t_idle = t_start;
  uint32_t spins = 0;
  while (true) {
    uint32_t c = 0, n = 0;
    int state = 0;   // 0 = nothing yet, 1 = claimed [c, c+n), 2 = leave
    if (lane == 0) {
      const uint32_t done = ld_acquire_cta_shared(S.cq + 4u * CQ_DONE);
      const uint32_t tail = ld_acquire_cta_shared(S.cq + 4u * CQ_TAIL);
      const uint32_t claim = ld_acquire_cta_shared(S.cq + 4u * CQ_CLAIM);
      if (claim < tail) {
        n = min(static_cast<uint32_t>(CW), tail - claim);
        if (atomicCAS(S.cq_ctl + CQ_CLAIM, claim, claim + n) == claim) {
          c = claim;
          state = 1;
        }
      } else if (done == 4u) {
        state = 2;
      }
      if (state == 0 && (++spins & 15u) == 0) {
        if (aborted(p)) state = 2;
        else if (globaltimer_ns() - t_idle > static_cast<uint64_t>(p.wait_ns)) {
          raise_error(p, MK_ERR_TIMEOUT, WHERE_COPY, static_cast<int>(claim));
          state = 2;
        }
      }
    }
    state = __shfl_sync(0xffffffffu, state, 0);
    if (state == 2) return;
    if (state == 0) {
      __nanosleep(128);
      continue;
    }
    c = __shfl_sync(0xffffffffu, c, 0);
    n = __shfl_sync(0xffffffffu, n, 0);
    if (lane == 0) t_idle = globaltimer_ns();
    // lane i < n takes entry c + i once it is full, then frees it for slot c + i + CQ_CAP
    int rt = -1, nb = 0, ok = 1;
    if (lane < static_cast<int>(n)) {
      const uint32_t slot = c + lane;
      const uint32_t e = S.cq + CQ_ENT + 16u * (slot % CQ_CAP);
      const uint64_t t0 = globaltimer_ns();
      uint32_t it2 = 0;
      while (ld_acquire_cta_shared(e) != 2u * slot + 1u) {
        if ((++it2 & 15u) == 0) {
          if (aborted(p)) { ok = 0; break; }
          if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
            raise_error(p, MK_ERR_TIMEOUT, WHERE_COPY, static_cast<int>(slot));
            ok = 0;
            break;
          }
        }
        __nanosleep(32);
      }
      if (ok) {
        uint32_t a, b;
        asm volatile("ld.shared::cta.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(e + 8u) : "memory");
        rt = static_cast<int>(a);
        nb = static_cast<int>(b);
        st_release_cta_shared(e, 2u * (slot + CQ_CAP));
      }
    }
    if (!__all_sync(0xffffffffu, ok)) return;
    int rr[CW], tt[CW], n0s[CW];
#pragma unroll
    for (int i = 0; i < CW; ++i) {
      const int x = __shfl_sync(0xffffffffu, rt, i);
      const int y = __shfl_sync(0xffffffffu, nb, i);
      const bool valid = i < static_cast<int>(n) && x >= 0 && x < p.R * T && y >= 0 && y < p.n_nblk;
      rr[i] = valid ? x / T : -1;
      tt[i] = valid ? x - (x / T) * T : 0;
      n0s[i] = valid ? y * BN : 0;
    }
    if (topk == 2) {
      // both slots of all rows in flight at once (16 loads per lane)
      uint4 v0[CW], v1[CW];
      float g0[CW], g1[CW];
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        v0[i] = v1[i] = make_uint4(0u, 0u, 0u, 0u);
        g0[i] = g1[i] = 0.f;
        const int col = n0s[i] + 8 * lane;
        if (rr[i] >= 0 && col < p.N) {
          const uint8_t* base = p.moe_ret[rr[i]] + (static_cast<size_t>(tt[i]) * 2 * p.N + col) * 2;
          const float4 f0 = ld_global_cg_f4(base);
          const float4 f1 = ld_global_cg_f4(base + static_cast<size_t>(p.N) * 2);
          v0[i] = make_uint4(__float_as_uint(f0.x), __float_as_uint(f0.y), __float_as_uint(f0.z),
                             __float_as_uint(f0.w));
          v1[i] = make_uint4(__float_as_uint(f1.x), __float_as_uint(f1.y), __float_as_uint(f1.z),
                             __float_as_uint(f1.w));
          const float* gp = p.moe_gates[rr[i]] + static_cast<size_t>(tt[i]) * 2;
          g0[i] = __ldg(gp);
          g1[i] = __ldg(gp + 1);
        }
      }
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        const int col = n0s[i] + 8 * lane;
        if (rr[i] < 0 || col >= p.N) continue;
        const uint32_t a4[4] = {v0[i].x, v0[i].y, v0[i].z, v0[i].w};
        const uint32_t b4[4] = {v1[i].x, v1[i].y, v1[i].z, v1[i].w};
        float o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // the same fused multiply-adds, in slot order, as the general path
          o[2 * j] = fmaf(g1[i], __uint_as_float(b4[j] << 16), fmaf(g0[i], __uint_as_float(a4[j] << 16), 0.f));
          o[2 * j + 1] = fmaf(g1[i], __uint_as_float(b4[j] & 0xFFFF0000u),
                              fmaf(g0[i], __uint_as_float(a4[j] & 0xFFFF0000u), 0.f));
        }
        uint8_t* dst = reinterpret_cast<uint8_t*>(p.out[rr[i]]) + (static_cast<size_t>(tt[i]) * p.N + col) * 2;
        st_global_v4(dst, pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                     pack_bf16x2(o[6], o[7]));
      }
      continue;
    }
    float acc[CW][8];
#pragma unroll
    for (int i = 0; i < CW; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int q = 0; q < topk; ++q) {
      uint4 v[CW];
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        const int col = n0s[i] + 8 * lane;
        if (rr[i] >= 0 && col < p.N) {
          const float4 f = ld_global_cg_f4(
              p.moe_ret[rr[i]] + ((static_cast<size_t>(tt[i]) * topk + q) * p.N + col) * 2);
          v[i] = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z),
                            __float_as_uint(f.w));
        }
      }
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        if (rr[i] < 0) continue;
        const float gq = __ldg(p.moe_gates[rr[i]] + static_cast<size_t>(tt[i]) * topk + q);
        const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][2 * j] = fmaf(gq, __uint_as_float(w4[j] << 16), acc[i][2 * j]);
          acc[i][2 * j + 1] = fmaf(gq, __uint_as_float(w4[j] & 0xFFFF0000u), acc[i][2 * j + 1]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < CW; ++i) {
      const int col = n0s[i] + 8 * lane;
      if (rr[i] < 0 || col >= p.N) continue;
      uint8_t* o = reinterpret_cast<uint8_t*>(p.out[rr[i]]) + (static_cast<size_t>(tt[i]) * p.N + col) * 2;
      st_global_v4(o, pack_bf16x2(acc[i][0], acc[i][1]), pack_bf16x2(acc[i][2], acc[i][3]),
                   pack_bf16x2(acc[i][4], acc[i][5]), pack_bf16x2(acc[i][6], acc[i][7]));
    }
  }
}

template <bool PAIR>
__device__ void epilogue(const FusedParams& p, const ComputeSmem& S, uint32_t tmem_base, int cid,
                         uint32_t rank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // TMEM lanes this warp may read: 32*quarter .. +31
  const int trow = quarter * 32 + lane;
  const size_t esz = p.out_f32 ? 4 : 2;
  const uint32_t epi = S.epi + static_cast<uint32_t>((warp - 2) * EPI_WARP_BYTES);   // this warp's staging
  int buf = 0;
  uint32_t acc_phase = 0;
  uint32_t pd_par = 0;           // phase bit of pdone(b) in bit b
  bool counters_ready = false;   // last-arrival counters published for this call
  bool zero_ready = false;       // atomic: every CTA's share of the fp32 tiles is zero
  const int n_items = n_items_for(p);
  for (int i = cid; i < n_items; i += p.n_compute) {
    Item it;
    decode(p, i, it, static_cast<int>(rank));
    // warp-uniform outcome: the tcgen05.ld below needs every lane of the warp
    const int landed = wait_bar(p, S.tfull(buf), acc_phase, WHERE_EPILOGUE, i) ? 1 : 0;
    if (!__all_sync(0xffffffffu, landed)) return;
#if MK_DEBUG_BOUNDS
    // the owner block of an RS / MLP output row exists (warp-uniform: the
    // tcgen05.ld below needs every lane)
    if ((p.op == OP_RS || p.op == OP_MLP) && it.phase != 1) {
      int ok = 1;
      if (lane == 0)
        ok = bounds_ok(p, it.row_hi == 0 || (it.out_row0 + it.row_hi - 1) / p.rows_per_owner < p.R, BC_OWNER, i)
                 ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    }
#endif
    if (p.trace != nullptr && warp == 2 && lane == 0) {
      trace_put(p, i, rank, 3, globaltimer_ns());
      trace_put(p, i, rank, 6, clock64());
    }
    tc_fence_after();
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(buf * BN);
    const bool row_ok = trow >= it.row_lo && trow < it.row_hi;
    const int grow = it.out_row0 + trow;
    const int n0 = it.nb * BN;
    if (it.slot >= 0 && p.chain) {
      // Running sum of this output tile, forwarded in rank order:
      //   sum_0 = P_0,  sum_j = sum_{j-1} + P_j,  output = round(sum_{P-1}).
      const int tile = it.slot / p.P, part = it.slot - tile * p.P;
      float* acc = p.staging + static_cast<size_t>(tile) * TILE_F32;
      if (part > 0) {
        // The running sum through part-1 must have been stored (acquire by
        // lane 0; __syncwarp orders the other lanes' loads after it).
        int ok = 1;
        if (lane == 0) ok = wait_flag(p, p.flags + it.slot - 1, WHERE_EPILOGUE, i) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return;
      }
      const bool last = (part == p.P - 1);
      // bf16 wire: the forwarded sum is a bf16 tile, uint4 (8 columns) at index
      // (32-column chunk * 4 + group) * BM + row
      uint8_t* accb = reinterpret_cast<uint8_t*>(p.staging) + static_cast<size_t>(tile) * TILE_F32 * 2;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + 32u * c, r);
        if (p.wire_bf16) {
          if (part > 0) {
            uint4 v[4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
              v[g] = ld_global_cg_u4(accb + (static_cast<size_t>((c * 4 + g) * BM + trow)) * 16);
            tc_wait_ld();
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t w[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                r[8 * g + 2 * e] = __float_as_uint(__uint_as_float(w[e] << 16) + __uint_as_float(r[8 * g + 2 * e]));
                r[8 * g + 2 * e + 1] =
                    __float_as_uint(__uint_as_float(w[e] & 0xffff0000u) + __uint_as_float(r[8 * g + 2 * e + 1]));
              }
            }
          } else {
            tc_wait_ld();
          }
          if (!last) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint8_t* d = accb + (static_cast<size_t>((c * 4 + g) * BM + trow)) * 16;
              st_global_v4(d, pack_bf16x2(__uint_as_float(r[8 * g]), __uint_as_float(r[8 * g + 1])),
                           pack_bf16x2(__uint_as_float(r[8 * g + 2]), __uint_as_float(r[8 * g + 3])),
                           pack_bf16x2(__uint_as_float(r[8 * g + 4]), __uint_as_float(r[8 * g + 5])),
                           pack_bf16x2(__uint_as_float(r[8 * g + 6]), __uint_as_float(r[8 * g + 7])));
            }
            continue;
          }
        } else if (part > 0) {
          float4 v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            v[q] = ld_global_cg_f4(acc + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4);
          tc_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            r[4 * q + 0] = __float_as_uint(v[q].x + __uint_as_float(r[4 * q + 0]));
            r[4 * q + 1] = __float_as_uint(v[q].y + __uint_as_float(r[4 * q + 1]));
            r[4 * q + 2] = __float_as_uint(v[q].z + __uint_as_float(r[4 * q + 2]));
            r[4 * q + 3] = __float_as_uint(v[q].w + __uint_as_float(r[4 * q + 3]));
          }
        } else {
          tc_wait_ld();
        }
        if (!last && !p.wire_bf16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float* d = acc + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4;
            st_global_v4(d, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
          }
        } else {
          // the final sum: through the warp's staging, as whole 128-byte row
          // segments (two 32-column chunks of bf16, one of fp32)
          const int per = p.out_f32 ? 1 : 2;
          stage_piece(epi, lane, (c % per) * 64, r, p.out_f32);
          if (c % per == per - 1) {
            __syncwarp();
            flush_staged(p, it, epi, lane, quarter, n0 + 32 * (c - per + 1));
            __syncwarp();
          }
        }
      }
    } else if (it.slot >= 0 && p.atomic) {
      // Add this partial into the tile's fp32 accumulator (zeroed by every CTA at
      // kernel start: wait once for all of them), then the warp whose count
      // completes its 32-row quarter (the P-th) converts and stores it.
      const int tile = it.slot / p.P;
      float* acc = p.staging + static_cast<size_t>(tile) * TILE_F32;
      if (!zero_ready) {
        int ok = 1;
        if (lane == 0)
          for (unsigned c = 0; c < gridDim.x && ok; ++c) ok = wait_flag(p, p.zflags + c, WHERE_EPILOGUE, i) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        zero_ready = true;
      }
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + 32u * c, r);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          red_add_v4_f32(acc + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4, r[4 * q], r[4 * q + 1],
                         r[4 * q + 2], r[4 * q + 3]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release_tmem<PAIR>(S, buf, rank);   // tensor memory is free again
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        if (!counters_ready) {
          if (!wait_flag(p, &p.hdr[HDR_READY], WHERE_EPILOGUE, i)) last = -1;
          counters_ready = true;
        }
        const bool skip = (p.inject == 2 && it.slot == 0);
        if (last == 0 && !skip)
          last = (bump_quarter(p, tile, quarter) == static_cast<uint32_t>(p.P - 1)) ? 1 : 0;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last < 0) return;
      if (last) {
        __threadfence();   // the other partials' additions happened before their counts
        reduce_quarter(p, it, acc, 1, trow, row_ok, grow);
      }
      if (warp == 2 && lane == 0) trace_end(p, i, rank);
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1u;
      }
      continue;
    } else if (it.slot >= 0 && p.last_arrival) {
      // Stage this partial, then the warp whose store completes its 32-row
      // quarter of the tile (the P-th arrival) sums all P partials in order.
      // Sliced: staged with L2 evict_last, so that they are still in L2 when
      // the slices are summed (measured: decode AR 0.1015 -> 0.0955 ms).
      float* slot = p.staging + static_cast<size_t>(it.slot) * TILE_F32;
      const uint64_t pol_keep = l2_policy_evict_last();
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + 32u * c, r);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float* d = slot + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4;
          if (p.sliced) st_global_v4_pol(d, make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]), pol_keep);
          else st_global_v4(d, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release_tmem<PAIR>(S, buf, rank);   // tensor memory is free again
      __threadfence();
      __syncwarp();
      const int tile = it.slot / p.P;
      int last = 0;
      if (lane == 0) {
        if (!counters_ready) {
          if (!wait_flag(p, &p.hdr[HDR_READY], WHERE_EPILOGUE, i)) last = -1;
          counters_ready = true;
        }
        const bool skip = (p.inject == 2 && it.slot == 0);
        if (last == 0 && !skip)
          last = (bump_quarter(p, tile, quarter) == static_cast<uint32_t>(p.P - 1)) ? 1 : 0;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last < 0) return;
      if (last && !p.sliced) {
        __threadfence();   // the other partials' stores happened before their counts
        reduce_quarter(p, it, p.staging + static_cast<size_t>(tile) * p.P * TILE_F32, p.P, trow, row_ok, grow);
      }
      if (warp == 2 && lane == 0) trace_end(p, i, rank);
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1u;
      }
      continue;
    } else if (p.op == OP_MOE_COMBINE) {
      combine_epilogue<PAIR>(p, S, it, taddr, buf, rank, lane, trow, row_ok, grow, epi);
      __syncwarp();   // lanes that handed a row over rejoin before the next tcgen05.ld
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1u;
      }
      continue;
    } else if (it.phase == 1) {
      // chained MLP up-projection: H_r = bf16(ReLU(acc)) into rank hid_r's hidden buffer
      uint8_t* hrow = p.mlp_hid[it.hid_r] + static_cast<size_t>(grow) * p.mlp_f * 2;
      const unsigned long long hptr = row_ok ? reinterpret_cast<unsigned long long>(hrow) : 0ull;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + 32u * c, r);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(fmaxf(__uint_as_float(r[q]), 0.f));
        staged_chunk(epi, lane, c, r, false, hptr, n0, p.mlp_f);
      }
    } else if (it.slot >= 0) {
      // Partial tile -> staging slot.  Layout: float4 (row, column group cg)
      // at index cg*BM + row, so a warp's 32 rows form 512 contiguous bytes.
      float* slot = p.staging + static_cast<size_t>(it.slot) * TILE_F32;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + 32u * c, r);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float* d = slot + (static_cast<size_t>((c * 8 + q) * BM + trow)) * 4;
          st_global_v4(d, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        }
      }
    } else if (p.op != OP_AR || it.rep >= 0) {
      // one destination row per lane: staged stores
      uint8_t* base;
      size_t orow;
      if (p.op == OP_AG || p.op == OP_MOE) {
        base = reinterpret_cast<uint8_t*>(p.out[p.op == OP_MOE ? it.mb : 0]);
        orow = static_cast<size_t>(grow);
      } else if (p.op == OP_RS || p.op == OP_MLP) {
        const int o = row_ok ? grow / p.rows_per_owner : 0;
        base = reinterpret_cast<uint8_t*>(p.out[o]);
        orow = static_cast<size_t>(row_ok ? grow - o * p.rows_per_owner : 0);
      } else {   // AR baseline: this rank's product to its replica
        base = reinterpret_cast<uint8_t*>(p.out[it.rep]);
        orow = static_cast<size_t>(grow);
      }
      const unsigned long long optr = row_ok ? reinterpret_cast<unsigned long long>(base + orow * p.N * esz) : 0ull;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + 32u * c, r);
        tc_wait_ld();
        staged_chunk(epi, lane, c, r, p.out_f32 != 0, optr, n0, p.N);
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + 32u * c, r);
        tc_wait_ld();
        const int col = n0 + 32 * c;
        const int nvalid = max(0, min(32, p.N - col));
        if (!row_ok || nvalid == 0) continue;
        for (int o = 0; o < p.R; ++o) {   // AR: the same bits to every replica
          uint8_t* base = reinterpret_cast<uint8_t*>(p.out[o]);
          store_row_chunk(base + (static_cast<size_t>(grow) * p.N + col) * esz, r, nvalid, p.out_f32);
        }
      }
    }
    // Tensor memory of this buffer may be overwritten by the next tile's MMAs.
    tc_fence_before();
    __syncwarp();
    // A tile that others wait for (a partial tile, an up-projection tile of
    // the chained MLP) is published once all four warps have stored it.  The
    // per-buffer barrier completes once per such tile, so it keeps its own
    // phase bit (items that publish nothing do not use it).
    const bool publish = it.slot >= 0 || (it.phase == 1 && it.row_hi > 0);
    if (lane == 0) {
      release_tmem<PAIR>(S, buf, rank);
      if (publish) mbar_arrive(S.pdone(buf));
    }
    if (publish && warp == 2 && lane == 0) {
      if (!wait_bar(p, S.pdone(buf), (pd_par >> buf) & 1u, WHERE_EPILOGUE, i)) return;
      if (it.phase == 1) {
        __threadfence();
        atomicAdd(p.mlp_cnt + static_cast<size_t>(it.hid_r) * p.n_mblk + it.mb, 1u);
      } else {
        const bool skip = (p.inject == 2 && it.slot == 0);
        if (!skip) {
          __threadfence();
          st_release_gpu(p.flags + it.slot, p.epoch);
        }
      }
    }
    if (publish) pd_par ^= 1u << buf;
    if (warp == 2 && lane == 0) trace_end(p, i, rank);
    if (++buf == 2) {
      buf = 0;
      acc_phase ^= 1u;
    }
  }
  if (p.sliced) {
    const int cta = PAIR ? 2 * cid + static_cast<int>(rank) : cid;
    Item proto{};
    finalize_slices(p, proto, epi, cta * 4 + (warp - 2), counters_ready);
  }
}

// The contiguous run at or after `row` below `hi`: rows of one shard,
// skipping the local shard's rows when it is not copied.
__device__ __forceinline__ bool copy_run(const FusedParams& p, long long& row, long long hi,
                                         long long& run_hi, int& s) {
  while (row < hi) {
    s = static_cast<int>(row / p.m_r);
    run_hi = min(hi, static_cast<long long>(s + 1) * p.m_r);
    if (s == p.local && !p.copy_local) {
      row = run_hi;
      continue;
    }
    return true;
  }
  return false;
}

// AG copy-in by the copy warps (6 and up) of every compute CTA.  The work list is (chunk in
// copy order, piece of copy_rows rows); worker w = n_cw*cta + (warp - 6) takes
// pieces w, w + n_cw*n_ctas, ... so all workers move neighbouring pieces of
// the same few chunks at a time.  Each lane streams 16-byte vectors, 16 loads
// in flight; after a piece every lane fences and lane 0 bumps the chunk's
// counter.  Copy warps never wait on anything, so they always progress.
#ifndef MK_CW_UNROLL
#define MK_CW_UNROLL 16
#endif
constexpr int CW_UNROLL = MK_CW_UNROLL;
#ifndef MK_MOE_CW_UNROLL
#define MK_MOE_CW_UNROLL MK_CW_UNROLL
#endif
constexpr int MOE_CW_UNROLL = MK_MOE_CW_UNROLL;   // 16-byte loads in flight per lane (MoE rows)
// MK_MOE_CW_HINT = 1: the dispatch copy reads token rows with an L2 evict_first
// policy and writes received rows with evict_last (the GEMM reads them next).
#ifndef MK_MOE_CW_HINT
#define MK_MOE_CW_HINT 0
#endif
// MK_CW_HINT = 1: shard reads marked L2 evict_first, gathered-A writes evict_last;
// 2: both evict_first.
#ifndef MK_CW_HINT
#define MK_CW_HINT 0
#endif

__device__ void copy_warps_role(const FusedParams& p, int cta, int n_ctas) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) - 6 >= p.n_cw) return;
  const int worker = cta * p.n_cw + ((threadIdx.x >> 5) - 6);
  const int n_workers = n_ctas * p.n_cw;
  const int pr = p.copy_rows;
  const int J = BM / pr;
  const long long n_pieces = static_cast<long long>(p.n_copy_chunks) * J;
  const size_t rb = static_cast<size_t>(p.K) * p.a_esz;   // bytes per gathered row
  bool skip_first = (p.inject == 1 && worker == 0);
#if MK_CW_HINT
  const uint64_t pol_src = l2_policy_evict_first();
  const uint64_t pol_dst = MK_CW_HINT == 2 ? l2_policy_evict_first() : l2_policy_evict_last();
#endif
  {
    int ok = 1;
    if (lane == 0) ok = wait_flag(p, &p.hdr[HDR_READY], WHERE_COPY, worker) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  }
  const unsigned long long t_start = p.trace != nullptr ? globaltimer_ns() : 0ull;
  unsigned long long n_done = 0, b_done = 0;
  for (long long pc = worker; pc < n_pieces; pc += n_workers) {
    const int c = static_cast<int>(pc / J), j = static_cast<int>(pc - static_cast<long long>(c) * J);
    const int mb = ag_copy_mb(p, c);
    if (j >= chunk_pieces(p, mb)) continue;  // past the end of a short last chunk
    int stop = 0;
    if (lane == 0) stop = aborted(p) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, stop, 0)) return;
    long long row = static_cast<long long>(mb) * BM + static_cast<long long>(j) * pr;
    const long long hi = min(row + pr, min(static_cast<long long>(mb + 1) * BM, static_cast<long long>(p.M)));
    long long run_hi;
    int s;
    while (copy_run(p, row, hi, run_hi, s)) {
      {
        const int ok = bounds_ok(p, row >= 0 && run_hi <= p.M && s >= 0 && s < p.R &&
                                        row >= static_cast<long long>(s) * p.m_r &&
                                        run_hi <= static_cast<long long>(s + 1) * p.m_r,
                                 BC_AG_COPY, row) ? 1 : 0;
        if (!__all_sync(0xffffffffu, ok)) return;
      }
      const uint8_t* src = p.shard[s] + static_cast<size_t>(row - static_cast<long long>(s) * p.m_r) * rb;
      uint8_t* dst = p.gathered + static_cast<size_t>(row) * rb;
      const size_t n16 = static_cast<size_t>(run_hi - row) * rb / 16;
      b_done += n16 * 16;
      for (size_t i0 = lane; i0 < n16; i0 += 32 * CW_UNROLL) {
        uint4 v[CW_UNROLL];
#pragma unroll
        for (int u = 0; u < CW_UNROLL; ++u) {
          const size_t idx = i0 + static_cast<size_t>(u) * 32;
#if MK_CW_HINT
          if (idx < n16) v[u] = ld_nc_v4_pol(src + idx * 16, pol_src);
#else
          if (idx < n16) v[u] = ld_nc_v4(src + idx * 16);
#endif
        }
#pragma unroll
        for (int u = 0; u < CW_UNROLL; ++u) {
          const size_t idx = i0 + static_cast<size_t>(u) * 32;
#if MK_CW_HINT
          if (idx < n16) st_global_v4_pol(dst + idx * 16, v[u], pol_dst);
#else
          if (idx < n16) st_global_v4(dst + idx * 16, v[u].x, v[u].y, v[u].z, v[u].w);
#endif
        }
      }
      row = run_hi;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      if (skip_first) skip_first = false;
      else atomicAdd(chunk_counter(p, mb), 1u);   // after this warp's fences: a release
    }
    __syncwarp();
    ++n_done;
  }
  if (p.trace != nullptr && lane == 0) trace_copy(p, worker, t_start, n_done, b_done);
}

// MoE dispatch by the copy warps of every compute CTA: destination rows of all
// ranks, rank-major (the dispatch order), in pieces of moe_rows_per_piece rows
// inside one 128-row block; row `row` of rank d is a bit copy of token
// g = recv_src[d][row] / topk (rank g / T, token g % T).  A token is read once:
// the copy of its slot that comes first in the dispatch order also writes the
// rows of its other slots (all later) and counts them in their blocks; the
// later rows are then skipped.  After a piece every lane fences and lane 0 adds
// the piece's own copied rows to the block's counter (zeroed by the offsets
// kernel), and the lanes holding forwarded rows add one each to theirs.
__device__ void moe_copy_warps_role(const FusedParams& p, int cta, int n_ctas) {
  const int lane = threadIdx.x & 31;
  const int wid = (threadIdx.x >> 5) - 6;   // copy warp of this CTA
  if (wid < 0 || wid >= N_COPY_WARPS) return;
  if (p.mode == MK_MODE_GEMM_ONLY) return;   // baseline: recv_x is already filled
  if (*reinterpret_cast<const volatile int*>(p.moe_ok) == 0) return;
  const int pr = p.moe_rows_per_piece;
  const int K = p.moe_topk;
  long long total = 0;
  for (int d = 0; d < p.R; ++d) total += (p.moe_recv_counts[d] + pr - 1) / pr;
  // The pieces of the first moe_boost_waves waves' tiles go to every copy warp
  // (those tiles wait for nothing else); the rest to the first n_cw warps of
  // every CTA, which keep ahead of the tiles without crowding out their loads.
  long long q_boost = 0;
  if (p.moe_boost_waves > 0) {
    const int nt = min(ld_acquire_gpu(reinterpret_cast<const uint32_t*>(p.moe_ntiles)),
                       static_cast<uint32_t>(p.n_items));
    const int ib = min(nt, p.moe_boost_waves * p.n_compute) - 1;
    if (ib >= 0) {
      const int* e = p.moe_tiles + 5 * ib;
      const int db = e[0], last = e[2] + e[3] - 1;   // the entry's destination rank and last row
      if (db >= 0 && db < p.R && last >= 0) {
        for (int d = 0; d < db; ++d) q_boost += (p.moe_recv_counts[d] + pr - 1) / pr;
        q_boost = min(total, q_boost + last / pr + 1);
      }
    }
  }
  const size_t rb = static_cast<size_t>(p.K) * 2;
  const size_t n16 = rb / 16;
  bool skip_first = (p.inject == 1 && cta == 0 && wid == 0);
#if MK_MOE_CW_HINT
  // token rows are read once per slot; received rows are read again by the GEMM
  const uint64_t pol_src = l2_policy_evict_first();
  const uint64_t pol_dst = l2_policy_evict_last();
#endif
  uint32_t* pend_w = nullptr;   // lane j < n_pend: block counter of the j-th forwarded row
  int n_pend = 0;
  // piece q of the dispatch order; false: stop (a bounds failure or an abort)
  auto copy_piece = [&](long long q) -> bool {
    int d = 0;
    long long j = q;
    int rc = p.moe_recv_counts[0];
    while (j >= (rc + pr - 1) / pr) {
      j -= (rc + pr - 1) / pr;
      ++d;
      rc = p.moe_recv_counts[d];
    }
    const int row0 = static_cast<int>(j) * pr;
    const int rows = min(pr, rc - row0);
    {
      const int ok = bounds_ok(p, d < p.R && row0 >= 0 && row0 + rows <= p.M, BC_MOE_COPY, q) ? 1 : 0;
      if (!__all_sync(0xffffffffu, ok)) return false;
    }
    const int base_d = static_cast<int>(p.moe_rbase[d]);
    int written = 0;
    for (int rr = 0; rr < rows; ++rr) {
      const int src = p.moe_src[d][row0 + rr];
      {
        const int ok = bounds_ok(p, src >= 0 && src < p.R * p.moe_T * K, BC_MOE_SRC, row0 + rr) ? 1 : 0;
        if (!__all_sync(0xffffffffu, ok)) return false;
      }
      const int g = src / K, slot = src - g * K;
      // dispatch-order positions of the token's other slots (lane l: slot l)
      const int self = base_d + row0 + rr;
      int pos = INT_MAX;
      if (lane < K && lane != slot) pos = p.moe_fwd[static_cast<size_t>(g) * K + lane];
      if (__any_sync(0xffffffffu, pos < self)) continue;   // copied and counted with an earlier slot
      uint8_t* xp = nullptr;    // lane l: slot l's destination row and its block counter
      uint32_t* xw = nullptr;
      int okx = 1;
      if (pos != INT_MAX) {
        int dd = 0;
        while (dd + 1 < p.R && static_cast<int>(p.moe_rbase[dd + 1]) <= pos) ++dd;
        const int rw = pos - static_cast<int>(p.moe_rbase[dd]);
        okx = bounds_ok(p, rw >= 0 && rw < p.moe_recv_counts[dd] && rw < p.M, BC_MOE_SRC, pos) ? 1 : 0;
        xp = p.moe_recv_x[dd] + static_cast<size_t>(rw) * rb;
        xw = p.flags + static_cast<size_t>(dd) * p.moe_nblk + rw / BM;
      }
      if (!__all_sync(0xffffffffu, okx)) return false;
      const uint32_t xmask = __ballot_sync(0xffffffffu, pos != INT_MAX);
      uint8_t* xd[MOE_MAX_TOPK];
#pragma unroll
      for (int l = 0; l < MOE_MAX_TOPK; ++l)
        xd[l] = reinterpret_cast<uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(xp), l));
      const int r = g / p.moe_T, t = g - r * p.moe_T;
      const uint8_t* sp = p.shard[r] + static_cast<size_t>(t) * rb;
      uint8_t* dp = p.moe_recv_x[d] + static_cast<size_t>(row0 + rr) * rb;
      for (size_t i0 = lane; i0 < n16; i0 += 32 * MOE_CW_UNROLL) {
        uint4 v[MOE_CW_UNROLL];
#pragma unroll
        for (int u = 0; u < MOE_CW_UNROLL; ++u) {
          const size_t idx = i0 + static_cast<size_t>(u) * 32;
#if MK_MOE_CW_HINT
          if (idx < n16) v[u] = ld_nc_v4_pol(sp + idx * 16, pol_src);
#else
          if (idx < n16) v[u] = ld_nc_v4(sp + idx * 16);
#endif
        }
#pragma unroll
        for (int u = 0; u < MOE_CW_UNROLL; ++u) {
          const size_t idx = i0 + static_cast<size_t>(u) * 32;
#if MK_MOE_CW_HINT
          if (idx < n16) st_global_v4_pol(dp + idx * 16, v[u], pol_dst);
#else
          if (idx < n16) st_global_v4(dp + idx * 16, v[u].x, v[u].y, v[u].z, v[u].w);
#endif
        }
#pragma unroll
        for (int l = 0; l < MOE_MAX_TOPK; ++l) {
          if (!((xmask >> l) & 1u)) continue;
#pragma unroll
          for (int u = 0; u < MOE_CW_UNROLL; ++u) {
            const size_t idx = i0 + static_cast<size_t>(u) * 32;
            if (idx < n16) st_global_v4(xd[l] + idx * 16, v[u].x, v[u].y, v[u].z, v[u].w);
          }
        }
      }
      ++written;
      // queue one count for each forwarded row (flushed with the piece's fence)
      for (uint32_t m = xmask; m != 0u; m &= m - 1u) {
        const int l = __ffs(m) - 1;
        uint32_t* w = reinterpret_cast<uint32_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(xw), l));
        if (n_pend == 32) {
          __threadfence();
          __syncwarp();
          atomicAdd(pend_w, 1u);
          n_pend = 0;
          __syncwarp();
        }
        if (lane == n_pend) pend_w = w;
        ++n_pend;
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0 && written > 0) {
      if (skip_first) skip_first = false;
      else atomicAdd(p.flags + static_cast<size_t>(d) * p.moe_nblk + row0 / BM, static_cast<uint32_t>(written));
    }
    if (lane < n_pend) atomicAdd(pend_w, 1u);
    n_pend = 0;
    __syncwarp();
    int stop = 0;
    if (lane == 0) stop = aborted(p) ? 1 : 0;
    return __shfl_sync(0xffffffffu, stop, 0) == 0;
  };
  for (long long q = static_cast<long long>(cta) * N_COPY_WARPS + wid; q < q_boost;
       q += static_cast<long long>(n_ctas) * N_COPY_WARPS)
    if (!copy_piece(q)) return;
  if (wid >= p.n_cw) return;
  for (long long q = q_boost + static_cast<long long>(cta) * p.n_cw + wid; q < total;
       q += static_cast<long long>(n_ctas) * p.n_cw)
    if (!copy_piece(q)) return;
}

// Compute CTA (cid = compute index; with pairs, the pair index).
// Atomic reduction: the spare warps of every CTA zero its share of the fp32
// accumulator tiles, then publish zflags[CTA] = epoch (all shares are waited
// for before the first addition into any tile).
__device__ void zero_role(const FusedParams& p) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) - 6;
  const size_t total4 = static_cast<size_t>(p.n_tiles) * TILE_F32 / 4;
  const size_t per = (total4 + gridDim.x - 1) / gridDim.x;
  const size_t lo = static_cast<size_t>(blockIdx.x) * per;
  const size_t hi = min(total4, lo + per);
  float* base = p.staging;
  for (size_t x = lo + static_cast<size_t>(w) * 32 + lane; x < hi; x += static_cast<size_t>(N_COPY_WARPS) * 32)
    st_global_v4(base + x * 4, 0u, 0u, 0u, 0u);
  __threadfence();
  asm volatile("barrier.sync 2, %0;" ::"n"(N_COPY_WARPS * 32) : "memory");   // the spare warps only
  if (w == 0 && lane == 0) st_release_gpu(p.zflags + blockIdx.x, p.epoch);
}

template <bool PAIR>
__device__ void compute_role(const FusedParams& p, uint8_t* smem, int cid) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  ComputeSmem S;
  S.ring = smem_u32(smem);
  S.bars = smem_u32(smem + RING_BYTES);
  S.cq = smem_u32(smem + RING_BYTES + BAR_BYTES);
  S.cq_ctl = reinterpret_cast<uint32_t*>(smem + RING_BYTES + BAR_BYTES);
  S.epi = smem_u32(smem + RING_BYTES + BAR_BYTES + CQ_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + RING_BYTES + TMEM_SLOT);
  if (p.op == OP_MOE_COMBINE) {
    // queue: control words zero, entry i free for slot i (sequence word 2i)
    if (threadIdx.x < 16) S.cq_ctl[threadIdx.x] = 0u;
    uint32_t* ent = S.cq_ctl + CQ_ENT / 4;
    for (int i = threadIdx.x; i < CQ_CAP; i += NTHREADS) ent[4 * i] = 2u * i;
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < Ring<PAIR>::stages; ++s) {
      mbar_init(S.full(s), 1);
      mbar_init(S.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(S.tfull(b), 1);
      mbar_init(S.tempty(b), PAIR ? 8 : 4);
    }
    mbar_init(S.drain(), 1);
    for (int b = 0; b < 2; ++b) mbar_init(S.pdone(b), 4);
    fence_mbar_init();
    for (int r = 0; r < MK_MAX_RANKS; ++r) {
      if (r < p.R || r < 2) {
        tma_prefetch_map(&p.tmA[r]);
        tma_prefetch_map(&p.tmB[r]);
      }
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();   // barriers of both CTAs initialised, TMEM allocated
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) producer<PAIR>(p, S, cid, rank);
    __syncwarp();
  } else if (warp == 1) {
    // the operand type picks the MMA loop once (the issuing warp's loop stays branch-free);
    // the warp runs it converged and one elected lane issues
    if (rank == 0) {
      if (p.fp8) mma_issuer<PAIR, true>(p, S, tmem_base, cid);
      else mma_issuer<PAIR, false>(p, S, tmem_base, cid);
    }
    __syncwarp();
  } else if (warp >= 2 && warp <= 5) {
    epilogue<PAIR>(p, S, tmem_base, cid, rank);
    __syncwarp();
    if (p.op == OP_MOE_COMBINE && lane == 0) {
      __threadfence_block();
      atomicAdd(S.cq_ctl + CQ_DONE, 1u);   // this warp hands over no more rows
    }
    __syncwarp();
  } else if (p.op == OP_MOE_COMBINE) {
    if (p.mode == MK_MODE_FUSED) combine_sum_role(p, S);
    __syncwarp();
  } else if (p.op == OP_MOE) {
    if constexpr (PAIR) moe_copy_warps_role(p, 2 * cid + static_cast<int>(rank), 2 * p.n_compute);
    else moe_copy_warps_role(p, cid, p.n_compute);
    __syncwarp();
  } else if (p.copy_warps) {
    if constexpr (PAIR) copy_warps_role(p, 2 * cid + static_cast<int>(rank), 2 * p.n_compute);
    else copy_warps_role(p, cid, p.n_compute);
    __syncwarp();
  } else if (p.atomic) {
    zero_role(p);
  }
  tc_fence_before();
  if constexpr (PAIR) {
    // After an abort a CTA of the pair may still have loads in flight into
    // its ring that the leader never armed; they land within microseconds.
    if (threadIdx.x == 0 && aborted(p)) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 50000ull) __nanosleep(1000);
    }
    __syncwarp();
    // Neither CTA leaves (or frees TMEM) while the leader's MMAs may still
    // read the peer's ring or write its tensor memory.
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ copy-in role (AG)
#ifndef MK_COPY_NBUF
#define MK_COPY_NBUF 3
#endif
#ifndef MK_COPY_BUF
#define MK_COPY_BUF 65536
#endif
#ifndef MK_COPY_WAITN
#define MK_COPY_WAITN 4
#endif
#ifndef MK_COPY_PFD
#define MK_COPY_PFD 0
#endif
// Copy-in pipeline: NBUF smem buffers of BUF bytes (bulk loads run NBUF-1
// pieces ahead, bulk stores drain them); a sub-chunk's flag is released once
// its stores are WAITN bulk groups old; pieces PFD ahead are prefetched to L2.
constexpr int COPY_NBUF = MK_COPY_NBUF;
constexpr uint32_t COPY_BUF = MK_COPY_BUF;
constexpr int COPY_WAITN = MK_COPY_WAITN;
constexpr int COPY_PFD = MK_COPY_PFD;
constexpr int COPY_PEND = 64;
static_assert(COPY_NBUF * COPY_BUF <= RING_BYTES, "copy buffers exceed the smem ring");
static_assert(104 + 8 * COPY_NBUF <= BAR_BYTES, "copy barriers exceed the barrier block");
static_assert(COPY_WAITN + 2 < COPY_PEND, "pending-release queue too small");

struct CopyIter {
  long long piece;   // index into the work list: (chunk position, sub-chunk)
  long long lo, hi;  // gathered rows of the current sub-chunk
  long long row;     // next row to copy
  long long off;     // byte offset inside the current contiguous run
  int flag;          // ready flag of the current sub-chunk
};

struct Piece {
  const uint8_t* src;
  uint8_t* dst;
  uint32_t bytes;
  int flag;
  bool last;  // last piece of its sub-chunk
};

// Rows [lo, hi) of the gathered A covered by work-list entry `piece`
// (sub-chunk `sub` of the chunk at copy-order position c).
__device__ __forceinline__ void sub_rows(const FusedParams& p, long long piece, CopyIter& st) {
  const int S = p.copy_sub;
  const int c = static_cast<int>(piece / S), sub = static_cast<int>(piece - static_cast<long long>(c) * S);
  const int mb = ag_copy_mb(p, c);
  const int rs = BM / S;
  st.lo = static_cast<long long>(mb) * BM + static_cast<long long>(sub) * rs;
  st.hi = min(st.lo + rs, min(static_cast<long long>(mb + 1) * BM, static_cast<long long>(p.M)));
  if (st.hi < st.lo) st.hi = st.lo;
  st.flag = mb * COPY_SUB_MAX + sub;
  st.row = st.lo;
  st.off = 0;
}

__device__ bool copy_next(const FusedParams& p, CopyIter& st, Piece& pc) {
  const size_t rb = static_cast<size_t>(p.K) * p.a_esz;   // bytes per gathered row
  const long long n_pieces = static_cast<long long>(p.n_copy_chunks) * p.copy_sub;
  if (st.piece >= n_pieces) return false;
  long long run_hi;
  int s;
  long long row = st.row;
  if (copy_run(p, row, st.hi, run_hi, s)) {
    const long long run_bytes = (run_hi - row) * static_cast<long long>(rb);
    const uint32_t n = static_cast<uint32_t>(min(run_bytes - st.off, static_cast<long long>(COPY_BUF)));
    pc.src = p.shard[s] + static_cast<size_t>(row - static_cast<long long>(s) * p.m_r) * rb + st.off;
    pc.dst = p.gathered + static_cast<size_t>(row) * rb + st.off;
    pc.bytes = n;
    pc.flag = st.flag;
    st.row = row;
    st.off += n;
    if (st.off == run_bytes) {
      st.row = run_hi;
      st.off = 0;
    }
    long long r2 = st.row, h2;
    int s2;
    pc.last = (st.off == 0) && !copy_run(p, r2, st.hi, h2, s2);
  } else {
    // a sub-chunk with nothing to copy (local rows only): signal it at once
    pc.src = nullptr;
    pc.dst = nullptr;
    pc.bytes = 0;
    pc.flag = st.flag;
    pc.last = true;
  }
  if (pc.last) {
    st.piece += p.n_copy;
    if (st.piece < n_pieces) sub_rows(p, st.piece, st);
  }
  return true;
}

__device__ void copy_role(const FusedParams& p, uint8_t* smem, int cid) {
  // One thread drives the pipeline: bulk loads (global -> smem) run
  // COPY_NBUF-1 pieces ahead; each landed piece is bulk-stored (smem ->
  // global); a sub-chunk's flag is released once its last store is complete.
  if (threadIdx.x != 0) return;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = smem_u32(smem + RING_BYTES) + 104u;
  for (int b = 0; b < COPY_NBUF; ++b) mbar_init(bars + 8u * b, 1);
  fence_mbar_init();

  const long long n_pieces = static_cast<long long>(p.n_copy_chunks) * p.copy_sub;
  CopyIter st;
  st.piece = cid;
  if (st.piece < n_pieces) sub_rows(p, st.piece, st);
  CopyIter pf = st;  // runs COPY_PFD pieces ahead, warming L2
  auto prefetch_one = [&]() {
    Piece x;
    if (COPY_PFD > 0 && copy_next(p, pf, x) && x.bytes) bulk_prefetch_l2(x.src, x.bytes);
  };
  for (int j = 0; j < COPY_PFD; ++j) prefetch_one();

  Piece q[COPY_NBUF];  // pieces whose loads are in flight, by buffer
  int pend_flag[COPY_PEND];
  long long pend_seq[COPY_PEND];
  int n_pend = 0;
  long long n_load = 0, n_store = 0;
  bool more = true, ok = true;
  const bool inject = (p.inject == 1 && cid == 0);
  bool injected = false;

  auto issue_load = [&](long long seq) -> bool {
    Piece pc;
    if (!copy_next(p, st, pc)) return false;
    prefetch_one();
    const int b = static_cast<int>(seq % COPY_NBUF);
    q[b] = pc;
    const uint32_t bar = bars + 8u * b;
    if (pc.bytes) {
      mbar_arrive_expect_tx(bar, pc.bytes);
      bulk_g2s(ring + static_cast<uint32_t>(b) * COPY_BUF, pc.src, pc.bytes, bar);
    } else {
      mbar_arrive(bar);
    }
    return true;
  };
  auto release = [&](int flag) {
    if (inject && !injected) {
      injected = true;
      return;
    }
    st_release_gpu(p.flags + flag, p.epoch);
  };

  for (; n_load < COPY_NBUF - 1 && more; ++n_load) more = issue_load(n_load);
  if (!more) --n_load;
  while (n_store < n_load) {
    const int b = static_cast<int>(n_store % COPY_NBUF);
    if (!wait_bar(p, bars + 8u * b, static_cast<uint32_t>((n_store / COPY_NBUF) & 1), WHERE_COPY,
                  q[b].flag)) {
      ok = false;
      break;
    }
    if (q[b].bytes) bulk_s2g(q[b].dst, ring + static_cast<uint32_t>(b) * COPY_BUF, q[b].bytes);
    bulk_commit();
    if (q[b].last) {
      pend_flag[n_pend] = q[b].flag;
      pend_seq[n_pend] = n_store;
      ++n_pend;
    }
    ++n_store;
    // Release sub-chunks whose stores are at least COPY_WAITN groups old (complete).
    bulk_wait<COPY_WAITN>();
    int keep = 0;
    for (int j = 0; j < n_pend; ++j) {
      if (pend_seq[j] <= n_store - 1 - COPY_WAITN) {
        fence_proxy_async_global();
        release(pend_flag[j]);
      } else {
        pend_flag[keep] = pend_flag[j];
        pend_seq[keep] = pend_seq[j];
        ++keep;
      }
    }
    n_pend = keep;
    if (n_pend >= COPY_PEND - 1) {  // bound the queue: wait for everything, release all
      bulk_wait<0>();
      fence_proxy_async_global();
      for (int j = 0; j < n_pend; ++j) release(pend_flag[j]);
      n_pend = 0;
    }
    // Refill the buffer whose store was issued one step ago.
    if (more) {
      bulk_wait_read<1>();
      if (issue_load(n_load)) ++n_load;
      else more = false;
    }
  }
  bulk_wait<0>();
  if (ok) {
    fence_proxy_async_global();
    for (int j = 0; j < n_pend; ++j) release(pend_flag[j]);
  }
  // Loads that were issued but not stored (abort path) must land before exit.
  for (long long s2 = n_store; s2 < n_load; ++s2) {
    const int b = static_cast<int>(s2 % COPY_NBUF);
    wait_bar(p, bars + 8u * b, static_cast<uint32_t>((s2 / COPY_NBUF) & 1), WHERE_DRAIN, 0, false);
  }
}

// ------------------------------------------------------------------ reduce role (RS / AR)
constexpr int RED_NSETS = 3;

__device__ void reduce_role(const FusedParams& p, uint8_t* smem, int rid) {
  const int tid = threadIdx.x;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = smem_u32(smem + RING_BYTES) + 104u;
  __shared__ int s_abort;
  const int P = p.P;
  const int pc = (P <= 8) ? 4 : 2;  // column groups (4 floats) per piece
  const uint32_t piece_bytes = static_cast<uint32_t>(pc * BM * 16);
  const uint32_t set_bytes = static_cast<uint32_t>(P) * piece_bytes;
  const int ppt = (BN / 4) / pc;  // pieces per tile
  const int my_tiles = (rid < p.n_tiles) ? (p.n_tiles - rid + p.n_reduce - 1) / p.n_reduce : 0;
  const long long total = static_cast<long long>(my_tiles) * ppt;
  if (tid == 0) {
    for (int b = 0; b < RED_NSETS; ++b) mbar_init(bars + 8u * b, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  __shared__ long long s_issued;
  auto issue = [&](long long seq) -> bool {  // thread 0 only
    const int t = static_cast<int>(seq / ppt), j = static_cast<int>(seq - static_cast<long long>(t) * ppt);
    const int q = rid + t * p.n_reduce;
    int mb, nb;
    raster(p, q, mb, nb);
    const int tile = mb * p.n_nblk + nb;
    if (j == 0) {
      for (int part = 0; part < P; ++part)
        if (!wait_flag(p, p.flags + static_cast<size_t>(tile) * P + part, WHERE_REDUCE, q)) return false;
      fence_proxy_async_global();
    }
    const int b = static_cast<int>(seq % RED_NSETS);
    const uint32_t bar = bars + 8u * b;
    mbar_arrive_expect_tx(bar, set_bytes);
    for (int part = 0; part < P; ++part) {
      const float* src = p.staging + (static_cast<size_t>(tile) * P + part) * TILE_F32 +
                         static_cast<size_t>(j) * pc * BM * 4;
      bulk_g2s(ring + b * (64u * 1024u) + part * piece_bytes, src, piece_bytes, bar);
    }
    return true;
  };

  if (tid == 0) {
    long long n = 0;
    for (; n < RED_NSETS - 1 && n < total; ++n)
      if (!issue(n)) {
        s_abort = 1;
        break;
      }
    s_issued = n;
  }
  __syncthreads();
  const size_t esz = p.out_f32 ? 4 : 2;
  long long seq = 0;
  for (; seq < total; ++seq) {
    // 1. keep RED_NSETS-1 sets in flight (the set refilled here was consumed
    //    in the previous iteration, which ended with a barrier)
    if (tid == 0 && !s_abort && s_issued == seq + RED_NSETS - 1 && s_issued < total) {
      if (issue(s_issued)) ++s_issued;
      else s_abort = 1;
    }
    __syncthreads();
    if (s_abort || seq >= s_issued) break;
    // 2. wait for this set's partial pieces
    const int b = static_cast<int>(seq % RED_NSETS);
    if (!wait_bar(p, bars + 8u * b, static_cast<uint32_t>((seq / RED_NSETS) & 1), WHERE_REDUCE,
                  static_cast<int>(seq)))
      s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    // 3. sum the P partials in fixed order and store
    const int t = static_cast<int>(seq / ppt), j = static_cast<int>(seq - static_cast<long long>(t) * ppt);
    const int qq = rid + t * p.n_reduce;
    int mb, nb;
    raster(p, qq, mb, nb);
    const uint8_t* buf = smem + b * (64 * 1024);
    const int units = BM * pc / 2;  // (row, pair of column groups)
    for (int u = tid; u < units; u += NTHREADS) {
      const int row = u % BM, cp = u / BM;
      float a[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) a[x] = 0.f;
      for (int part = 0; part < P; ++part) {
        const float4 v0 = *reinterpret_cast<const float4*>(buf + part * piece_bytes + ((2 * cp) * BM + row) * 16);
        const float4 v1 = *reinterpret_cast<const float4*>(buf + part * piece_bytes + ((2 * cp + 1) * BM + row) * 16);
        if (part == 0) {
          a[0] = v0.x; a[1] = v0.y; a[2] = v0.z; a[3] = v0.w;
          a[4] = v1.x; a[5] = v1.y; a[6] = v1.z; a[7] = v1.w;
        } else {
          a[0] += v0.x; a[1] += v0.y; a[2] += v0.z; a[3] += v0.w;
          a[4] += v1.x; a[5] += v1.y; a[6] += v1.z; a[7] += v1.w;
        }
      }
      const int grow = mb * BM + row;
      const int col = nb * BN + (j * pc + 2 * cp) * 4;
      if (grow >= p.M || col >= p.N) continue;
      const int nrep = (p.op == OP_AR) ? p.R : 1;
      for (int o = 0; o < nrep; ++o) {
        uint8_t* base;
        size_t off;
        if (p.op != OP_AR) {   // RS and the chained MLP: the owner's row block
          const int ow = grow / p.rows_per_owner;
          base = reinterpret_cast<uint8_t*>(p.out[ow]);
          off = (static_cast<size_t>(grow - ow * p.rows_per_owner) * p.N + col) * esz;
        } else {
          base = reinterpret_cast<uint8_t*>(p.out[o]);
          off = (static_cast<size_t>(grow) * p.N + col) * esz;
        }
        if (p.out_f32) {
          st_global_v4(base + off, __float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                       __float_as_uint(a[3]));
          st_global_v4(base + off + 16, __float_as_uint(a[4]), __float_as_uint(a[5]),
                       __float_as_uint(a[6]), __float_as_uint(a[7]));
        } else {
          st_global_v4(base + off, pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                       pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
        }
      }
    }
    __syncthreads();
  }
  __syncthreads();
  // Sets issued but not consumed (abort path) must land before the CTA exits.
  if (tid == 0) {
    for (long long s2 = seq; s2 < s_issued; ++s2) {
      const int b = static_cast<int>(s2 % RED_NSETS);
      wait_bar(p, bars + 8u * b, static_cast<uint32_t>((s2 / RED_NSETS) & 1), WHERE_DRAIN, 0, false);
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ the kernel
// PAIR = false: one CTA per SM, roles by ticket.  PAIR = true: launched as
// clusters of two; every CTA computes (no copy-role or reduce-role CTAs) and
// all tcgen05 work of the launch uses cta_group::2.
template <bool PAIR>
__global__ void __launch_bounds__(NTHREADS, 1) mk_fused_kernel(const __grid_constant__ FusedParams p) {
  // With p.pdl the launch overlaps the previous kernel's end (the MoE
  // bookkeeping); nothing here runs before that kernel's results are visible.
  griddep_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint32_t s_ticket;
  if constexpr (PAIR) {
    if (threadIdx.x == 0) s_ticket = blockIdx.x;
  } else {
    if (threadIdx.x == 0) {
      const uint32_t t = atomicAdd(&p.hdr[HDR_TICKET], 1u);
      if (t == gridDim.x - 1) atomicExch(&p.hdr[HDR_TICKET], 0u);
      s_ticket = t;
    }
  }
  __syncthreads();
  const int t = static_cast<int>(s_ticket);
  if (t == 0 && ((p.op == OP_AG && p.copy_warps) || p.last_arrival || p.atomic || p.op == OP_MLP)) {
    // Zero this call's counters (the workspace may hold anything from earlier
    // calls of any op), then publish them.
    if (p.op == OP_AG) {
      for (int mb = threadIdx.x; mb < p.n_mblk; mb += NTHREADS) *chunk_counter(p, mb) = 0u;
    } else if (p.op == OP_MLP) {
      if (p.copy_warps)
        for (int mb = threadIdx.x; mb < p.n_mblk; mb += NTHREADS) *chunk_counter(p, mb) = 0u;
      for (int x = threadIdx.x; x < p.R * p.n_mblk; x += NTHREADS) p.mlp_cnt[x] = 0u;
    } else {
      for (int x = threadIdx.x; x < p.n_tiles * 4; x += NTHREADS) p.flags[x] = 0u;
      if (threadIdx.x == 0) p.hdr[HDR_CLAIM] = 0u;   // the sliced reduction's next job
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release_gpu(&p.hdr[HDR_READY], p.epoch);
  }
  if constexpr (PAIR) {
    compute_role<true>(p, smem, t >> 1);
  } else {
    if (t < p.n_copy) {
      copy_role(p, smem, t);
    } else if (t < p.n_copy + p.n_compute) {
      compute_role<false>(p, smem, t - p.n_copy);
    } else {
      reduce_role(p, smem, t - p.n_copy - p.n_compute);
    }
  }
}

cudaError_t launch_fused(const FusedParams& p, int grid, cudaStream_t stream) {
  static int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(mk_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mk_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (p.pair) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = 2;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  if (p.pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  if (p.pair) return cudaLaunchKernelEx(&cfg, mk_fused_kernel<true>, p);
  return cudaLaunchKernelEx(&cfg, mk_fused_kernel<false>, p);
}

int max_pair_clusters() {
  static int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cached_dev == dev) return cached;
  if (cudaFuncSetAttribute(mk_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mk_fused_kernel<true>, &cfg) != cudaSuccess) n = 0;
  cached_dev = dev;
  cached = n;
  return n;
}

}  // namespace mk
