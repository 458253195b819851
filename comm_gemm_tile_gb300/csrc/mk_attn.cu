// mk_attn.cu -- ring attention (mKernel write-up, news.chathome.org,
// "五种融合内核" table, row "Ring Attention"): every rank holds a contiguous
// block of the sequence's Q, K and V; the K/V blocks travel around the ring
// while each rank attends its queries to every block that has arrived,
// merging the partial softmax results.
//
// One persistent launch of 416 threads per CTA, one CTA per SM:
//   * warps 0 and 12 (TMA): a 128-query tile of one (rank, head), then the K
//     (warp 0) and V (warp 12) tiles, 128 keys each, in ring order -- the
//     rank's own block, then the blocks of ranks r-1, r-2, ... as they land
//     in its receive buffer;
//   * warp 1 (MMA): S = Q K^T into one of two TMEM buffers, then O += P V
//     into one of two TMEM accumulators (tcgen05, bf16 -> fp32), with one
//     mbarrier wait and two commits per tile (see at_mma);
//   * warps 2-9 (softmax): online softmax in two groups of four warps, one
//     for the even tiles of the CTA's running tile count and one for the odd
//     ones (so a query tile's key tiles alternate between them), each
//     with its own running maximum, sum, P buffer (shared memory) and O
//     accumulator (TMEM), so that two tiles' softmax runs at once; P =
//     exp2(scale * log2(e) * s - m) as bf16; O is rescaled only when the
//     maximum grows by more than 2^8 (the final division uses the same stale
//     maximum for O and the sum, so the result is unchanged); at the end of a
//     query tile the two groups merge their maxima, sums and O;
//   * warps 10-11 (copy): the ring's transfers -- rank r receives the block
//     of rank (r - j) mod R at step j -- as row copies into its receive
//     buffer, one counter per (rank, step, head).
// Causal attention skips the tiles after each query tile (and, in ring order,
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
constexpr int AT_THREADS = 416;              // 13 warps: see the role list above
constexpr int AT_MAX_R = 8;
// shared memory (from the 1024-aligned base)
constexpr uint32_t AT_Q = 0;                 // Q tile: 2 K-major atoms of [128 rows x 128 B]
constexpr uint32_t AT_KV = 32768;            // 2 stages of K (32 KB) + V (32 KB)
constexpr uint32_t AT_KV_STAGE = 65536;
constexpr uint32_t AT_P = AT_KV + 2 * AT_KV_STAGE;   // two P tiles (same layout as Q), by tile parity
constexpr uint32_t AT_BARS = AT_P + 2 * 32768;
constexpr uint32_t AT_XCH = AT_BARS + 256;    // row maxima, then row sums, of the softmax warp pairs
constexpr int AT_SMEM = 1024 + AT_XCH + 2 * AT_T * 4;
// barriers (byte offsets in the barrier block)
constexpr uint32_t B_QFULL = 0, B_QEMPTY = 8, B_KFULL = 16, B_SFULL = 48, B_PFULL = 80,
                   B_PFREE = 96, B_OFREE = 112, B_TMEM = 120, B_DRAIN = 128, B_PAIR = 136;
constexpr uint32_t AT_TMEM_COLS = 512;       // S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512)
constexpr uint32_t AT_O_COL = 256;           // O of tile parity b at AT_O_COL + 128 b
// S = Q K^T: both operands K-major; O += P V: V MN-major
constexpr uint32_t IDESC_S = idesc_bf16_f32(AT_T, AT_T, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(AT_T, AT_D, false, true);
constexpr float RESCALE_LOG2 = 8.f;          // rescale O when the maximum grows by more than 2^8

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
  int R, heads, s_r, nkt, nqt, causal, n_items;
  int copy, use_recv, wait;          // ring copies by the copy warps; read them; wait for them
  int n_cw;
  int inject;                        // test only: 1 = one ring piece is never counted
};

// ------------------------------------------------------------------ waits (bounded)
__device__ __forceinline__ bool at_aborted(const AttnParams& p) {
  return ld_volatile(&p.hdr[HDR_ABORT]) == p.epoch;
}
__device__ __noinline__ void at_error(const AttnParams& p, int where, int item) {
  int* st = reinterpret_cast<int*>(&p.hdr[HDR_STATUS]);
  if (atomicCAS(st, 0, MK_ERR_TIMEOUT) == 0)
    atomicExch(reinterpret_cast<int*>(&p.hdr[HDR_DETAIL]), where * 1000000 + (item % 1000000));
  __threadfence();
  atomicExch(&p.hdr[HDR_ABORT], p.epoch);
}
__device__ __noinline__ bool at_wait_bar(const AttnParams& p, uint32_t bar, uint32_t parity, int where, int item,
                                         bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++it & 31u) == 0) {
      if (honor_abort && at_aborted(p)) return false;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.wait_ns)) {
        at_error(p, where, item);
        return false;
      }
    }
  }
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
  int r, h, qt, n;   // rank, head, query tile, K/V tiles to visit
};
// Items run longest first (causal: the last rank's queries see the most keys).
__device__ __forceinline__ AtItem at_item(const AttnParams& p, int i) {
  AtItem it;
  const int per_r = p.heads * p.nqt;
  it.r = p.R - 1 - i / per_r;
  const int rem = i - (p.R - 1 - it.r) * per_r;
  it.h = rem / p.nqt;
  it.qt = rem - it.h * p.nqt;
  it.n = p.causal ? (it.qt + 1) + it.r * p.nkt : p.R * p.nkt;
  return it;
}
// Tile t of an item: ring step j (source rank s = r - j mod R) and key tile kt.
__device__ __forceinline__ void at_tile(const AttnParams& p, const AtItem& it, int t, int& j, int& s, int& kt) {
  if (p.causal) {
    if (t <= it.qt) {
      j = 0;
      s = it.r;
      kt = t;
      return;
    }
    const int u = t - (it.qt + 1);
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
// TMA producers: warp 0 loads the Q tile of each item and the K tiles, warp 12
// the V tiles, each into its half of the two K/V stages.  Stage, S, P and O
// buffer of a tile are all the parity of the CTA's running tile count n.
// A K stage is free once S of tile n-2 is done (S full), a V stage once the
// product of tile n-2 is done (P free).  Both land on the P-full barrier of
// their buffer, V of tile n on the phase of tile n and K of tile n on the
// phase of tile n-2 (six arrivals: the four softmax warps', the V load's and
// the K load's, the loads with their bytes).  The MMA issuer's one wait per
// tile there, before S of tile n and the product of tile n-2, then covers
// K, P and V.  K of tiles 0 and 1, which have no tile two back, land on
// their own barriers; after the last tile the K producer still arrives,
// without bytes, on the two phases that no K tile follows.
template <bool IS_V>
__device__ void at_producer(const AttnParams& p, uint32_t bars, uint32_t base) {
  const uint32_t EMPTY = IS_V ? B_PFREE : B_SFULL;
  int stage = 0;
  uint32_t ph = 0, q_ph = 0;
  uint32_t count = 0;        // running tile count n of the next tile
  bool ready = false;
  for (int i = blockIdx.x; i < p.n_items; i += gridDim.x) {
    const AtItem it = at_item(p, i);
    if (!IS_V) {
      if (!at_wait_bar(p, bars + B_QEMPTY, q_ph ^ 1u, WHERE_PRODUCER, i)) return;
      q_ph ^= 1u;
      const int qrow = it.h * p.s_r + it.qt * AT_T;
      mbar_arrive_expect_tx(bars + B_QFULL, 2u * 16384u);
      tma_load_2d(base + AT_Q, &p.tmQ[it.r], bars + B_QFULL, 0, qrow);
      tma_load_2d(base + AT_Q + 16384u, &p.tmQ[it.r], bars + B_QFULL, 64, qrow);
    }
    int waited_j = 0;
    for (int t = 0; t < it.n; ++t) {
      int j, s, kt;
      at_tile(p, it, t, j, s, kt);
      if (!at_wait_bar(p, bars + EMPTY + 8u * stage, ph ^ 1u, WHERE_PRODUCER, i)) return;
      const CUtensorMap* m = IS_V ? &p.tmV[s] : &p.tmK[s];
      int row = it.h * p.s_r + kt * AT_T;
      if (j > 0 && p.use_recv) {
        if (p.wait && j != waited_j) {
          if (!ready) {
            if (!at_wait_value(p, &p.hdr[HDR_READY], p.epoch, WHERE_PRODUCER, i)) return;
            ready = true;
          }
          if (!at_wait_value(p, at_counter(p, it.r, j, it.h), 2u * p.nkt, WHERE_PRODUCER, i)) return;
          fence_proxy_async_global();
          waited_j = j;
        }
        m = IS_V ? &p.tmVr[it.r] : &p.tmKr[it.r];
        row = ((j - 1) * p.heads + it.h) * p.s_r + kt * AT_T;
      }
      const uint32_t dst = base + AT_KV + static_cast<uint32_t>(stage) * AT_KV_STAGE + (IS_V ? 32768u : 0u);
      const uint32_t full = bars + ((IS_V || count >= 2u) ? B_PFULL : B_KFULL) + 8u * stage;
      mbar_arrive_expect_tx(full, 32768u);
      if (IS_V) {
        tma_load_3d(dst, m, full, 0, row, 0);
        tma_load_3d(dst + 16384u, m, full, 0, row + 64, 0);
      } else {
        tma_load_2d(dst, m, full, 0, row);
        tma_load_2d(dst + 16384u, m, full, 64, row);
      }
      ++count;
      if (++stage == 2) {
        stage = 0;
        ph ^= 1u;
      }
    }
  }
  if (!IS_V) {
    // the phases of the last two tiles count a K arrival too: made once S of
    // those tiles is done, as a K load for the tiles after them would be
    for (uint32_t n = count; n < count + 2u; ++n) {
      if (n >= 2u) {
        if (!at_wait_bar(p, bars + B_SFULL + 8u * stage, ph ^ 1u, WHERE_PRODUCER, 0)) return;
        mbar_arrive(bars + B_PFULL + 8u * stage);
      }
      if (++stage == 2) {
        stage = 0;
        ph ^= 1u;
      }
    }
  }
}

// MMA issuer.  The CTA's n-th tile (counted over all its items) uses K/V
// stage, S, P and O buffers n & 1: the softmax of the even ones (warps 2-5)
// and of the odd ones (warps 6-9) each keep their own running maximum, sum
// and O for the item; they are merged when the item ends.
//
// Issue order: when the softmax of running tile n-2 has published P (one
// wait, which also covers V of that tile and frees S buffer n & 1), the
// issuer starts S of tile n first and then the product of tile n-2, so the
// softmax group's next S is not queued behind a product.  Per tile one
// mbarrier wait besides the K tile and two commits: S full (which also frees
// the K stage) and P free (which also frees the V stage and marks O
// updated).  Every wait and commit in this thread stalls the tensor pipe's
// short queue, so there are no others.
__device__ __forceinline__ void at_pv(const AttnParams& p, uint32_t bars, uint32_t base, uint32_t tmem, int pb,
                                      int tile) {
  const uint32_t vb = base + AT_KV + static_cast<uint32_t>(pb) * AT_KV_STAGE + 32768u;
  const uint32_t pbase = base + AT_P + 32768u * static_cast<uint32_t>(pb);
  const uint32_t obuf = tmem + AT_O_COL + static_cast<uint32_t>(pb) * AT_T;
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t ad = sdesc_swz(pbase + 16384u * a + 32u * k, 16u, 1024u, 2u);
      const uint64_t bd = sdesc_sw128(vb + 16384u * a + 2048u * k, 8192u, 1024u);
      // the first product of each O buffer in an item (tiles 0 and 1) overwrites it
      tc_mma_bf16(obuf, ad, bd, IDESC_PV, (tile >= 2 || a || k) ? 1u : 0u);
    }
  tc_commit(bars + B_PFREE + 8u * pb);   // P buffer and V stage free; O[pb] holds this product
}

__device__ void at_mma(const AttnParams& p, uint32_t bars, uint32_t base, uint32_t tmem) {
  uint32_t q_ph = 0, of_ph = 0;
  uint32_t pf_ph = 0;        // phase bits of the P-full barriers, bit b for buffer b
  int stage = 0;
  // products not yet issued: the tile two back (pend2) and one back (pend1),
  // as their tile index within their item (-1: none)
  int pend2 = -1, pend1 = -1;
  int item = -1;
  for (int i = blockIdx.x; i < p.n_items; i += gridDim.x) {
    const AtItem it = at_item(p, i);
    item = i;
    if (!at_wait_bar(p, bars + B_QFULL, q_ph, WHERE_MMA, i)) goto done;
    q_ph ^= 1u;
    for (int t = 0; t < it.n; ++t) {
      const int b = stage;
      if (pend2 >= 0) {
        // P and V of the tile two back (same buffer; S buffer b is free too)
        // and K of this tile
        if (!at_wait_bar(p, bars + B_PFULL + 8u * b, (pf_ph >> b) & 1u, WHERE_MMA, i)) goto done;
        pf_ph ^= 1u << b;
        if (pend2 == 0) {   // first product of an item: the previous item's O has been read out
          if (!at_wait_bar(p, bars + B_OFREE, of_ph ^ 1u, WHERE_MMA, i)) goto done;
          of_ph ^= 1u;
        }
      } else {
        // the CTA's first two tiles: K on its own barrier
        if (!at_wait_bar(p, bars + B_KFULL + 8u * b, 0u, WHERE_MMA, i)) goto done;
      }
      tc_fence_after();
      {
        const uint32_t kb = base + AT_KV + static_cast<uint32_t>(b) * AT_KV_STAGE;
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = sdesc_swz(base + AT_Q + 16384u * a + 32u * k, 16u, 1024u, 2u);
            const uint64_t bd = sdesc_swz(kb + 16384u * a + 32u * k, 16u, 1024u, 2u);
            tc_mma_bf16(tmem + static_cast<uint32_t>(b) * AT_T, ad, bd, IDESC_S, (a | k) ? 1u : 0u);
          }
        tc_commit(bars + B_SFULL + 8u * b);              // S ready; this K stage may be refilled
        if (t == it.n - 1) tc_commit(bars + B_QEMPTY);   // Q is read by no later MMA of this item
      }
      if (pend2 >= 0) at_pv(p, bars, base, tmem, b, pend2);
      pend2 = pend1;
      pend1 = t;
      if (++stage == 2) stage = 0;
    }
  }
  // the last two products (tiles two back and one back of the running count)
  for (int r = 0; r < 2; ++r) {
    if (pend2 >= 0) {
      const int b = stage;
      if (!at_wait_bar(p, bars + B_PFULL + 8u * b, (pf_ph >> b) & 1u, WHERE_MMA, item)) goto done;
      pf_ph ^= 1u << b;
      if (pend2 == 0) {
        if (!at_wait_bar(p, bars + B_OFREE, of_ph ^ 1u, WHERE_MMA, item)) goto done;
        of_ph ^= 1u;
      }
      tc_fence_after();
      at_pv(p, bars, base, tmem, b, pend2);
    }
    pend2 = pend1;
    pend1 = -1;
    if (++stage == 2) stage = 0;
  }
done:
  tc_commit(bars + B_DRAIN);
  at_wait_bar(p, bars + B_DRAIN, 0, WHERE_DRAIN, 0, false);
}

// P tile element (row, key): K-major, 128-byte swizzle, two 64-key atoms.
__device__ __forceinline__ uint32_t p_chunk_addr(uint32_t pbase, int row, int kchunk) {
  // kchunk: 8-key group 0..15
  const int atom = kchunk >> 3, c = kchunk & 7;
  return pbase + static_cast<uint32_t>(atom) * 16384u + static_cast<uint32_t>(row >> 3) * 1024u +
         static_cast<uint32_t>(row & 7) * 128u + static_cast<uint32_t>((c ^ (row & 7)) << 4);
}

// Softmax warps 2-9: warp w handles TMEM lanes 32*(w%4) .. +31 (query rows)
// and half (w-2)/4 of the 128 columns (keys of S, head dims of O).  The two
// warps of a row quarter exchange their row maxima and, at the end, their row
// sums through shared memory, meeting at a two-arrival mbarrier (a bounded
// wait, so that one warp leaving on an abort cannot strand the other).
__device__ __forceinline__ bool pair_sync(const AttnParams& p, uint32_t bar, uint32_t& ph, int item) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const int ok = at_wait_bar(p, bar, ph, WHERE_EPILOGUE, item) ? 1 : 0;
  ph ^= 1u;
  return __all_sync(0xffffffffu, ok) != 0;
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

__device__ void at_softmax(const AttnParams& p, uint32_t bars, uint32_t base, uint32_t tmem, float* xch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int grp = (warp - 2) >> 2;                           // 0: even tiles, 1: odd tiles (running count)
  const int row = quarter * 32 + lane;                       // query row within the tile
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t pbar = bars + B_PAIR + 8u * quarter;
  const uint32_t sbase = tmem + lane_off + static_cast<uint32_t>(grp) * AT_T;
  const uint32_t obase = tmem + lane_off + AT_O_COL;
  const uint32_t pbase = base + AT_P + 32768u * static_cast<uint32_t>(grp);
  const float c = p.scale_log2;
  uint32_t pair_ph = 0, sf_ph = 0, uses = 0;
  uint32_t count = 0;                                        // tiles of the CTA's earlier items
  for (int i = blockIdx.x; i < p.n_items; i += gridDim.x) {
    const AtItem it = at_item(p, i);
    const int qpos = it.qt * AT_T + row;                     // position within rank r's block
    const int par = static_cast<int>(count & 1u);
    const int t0 = grp ^ par;                                // this group's first tile of the item
    count += static_cast<uint32_t>(it.n);
    float m_run = -INFINITY, l_run = 0.f;
    for (int t = t0; t < it.n; t += 2) {
      int j, s, kt;
      at_tile(p, it, t, j, s, kt);
      const int valid = min(AT_T, p.s_r - kt * AT_T);       // keys of this tile inside the block
      const bool diag = p.causal && j == 0 && kt == it.qt;   // keys after the query are masked
      const int lim = diag ? min(valid, row + 1) : valid;
      const bool masked = __any_sync(0xffffffffu, lim < AT_T);
      {
        int ok = at_wait_bar(p, bars + B_SFULL + 8u * grp, sf_ph, WHERE_EPILOGUE, i) ? 1 : 0;
        if (!__all_sync(0xffffffffu, ok)) return;
      }
      sf_ph ^= 1u;
      tc_fence_after();
      // pass 1: the row maximum (scale > 0 keeps the order: taken unscaled); the
      // next 32 columns load while these are reduced
      float mx = -INFINITY;
      {
        uint32_t va[32], vb[32];
        tc_ld_32x32b_x32(sbase, va);
        tc_wait_ld_regs(va);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t (&cur)[32] = (cc & 1) ? vb : va;
          uint32_t (&nxt)[32] = (cc & 1) ? va : vb;
          if (cc < 3) tc_ld_32x32b_x32(sbase + 32u * (cc + 1), nxt);
          if (masked) {
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if (32 * cc + q < lim) mx = fmaxf(mx, __uint_as_float(cur[q]));
          } else {
#pragma unroll
            for (int q = 0; q < 32; q += 2) mx = fmax3(mx, __uint_as_float(cur[q]), __uint_as_float(cur[q + 1]));
          }
          if (cc < 3) tc_wait_ld_regs(nxt);
        }
      }
      const float m_new = fmaxf(m_run, mx * c);
      // the product that last read this P buffer (and wrote this O) has completed
      if (uses > 0u) {
        int ok = at_wait_bar(p, bars + B_PFREE + 8u * grp, (uses - 1u) & 1u, WHERE_EPILOGUE, i) ? 1 : 0;
        if (!__all_sync(0xffffffffu, ok)) return;
      }
      float factor = 1.f;
      if (t == t0) {
        m_run = m_new;
      } else if (m_new > m_run + RESCALE_LOG2) {
        factor = ex2(m_run - m_new);
        m_run = m_new;
        l_run *= factor;
      }
      if (__any_sync(0xffffffffu, factor != 1.f)) {
        tc_fence_after();
        const uint32_t ob = obase + static_cast<uint32_t>(grp) * AT_T;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tc_ld_32x32b_x32(ob + 32u * cc, v);
          tc_wait_ld();
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(__uint_as_float(v[q]) * factor);
          tc_st_32x32b_x32(ob + 32u * cc, v);
        }
        tc_wait_st();
      }
      // pass 2: P = 2^(c*s - m), the running sum, P as bf16 into shared memory
      // (two lanes per packed fp32 fused multiply-add / add)
      const uint64_t c2 = f2pack(c, c), nm2 = f2pack(-m_run, -m_run);
      uint64_t l2 = f2pack(0.f, 0.f);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tc_ld_32x32b_x32(sbase + 32u * cc, v);
        tc_wait_ld();
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {   // 8 keys per 16-byte chunk
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = 32 * cc + 8 * k8 + 2 * q;
            float e0, e1;
            f2unpack(f2fma(f2pack(__uint_as_float(v[8 * k8 + 2 * q]), __uint_as_float(v[8 * k8 + 2 * q + 1])), c2,
                           nm2),
                     e0, e1);
            float p0 = ex2(e0), p1 = ex2(e1);
            if (masked) {
              p0 = (kk < lim) ? p0 : 0.f;
              p1 = (kk + 1 < lim) ? p1 : 0.f;
            }
            l2 = f2add(l2, f2pack(p0, p1));
            pk[q] = pack_bf16x2(p0, p1);
          }
          const uint32_t a = p_chunk_addr(pbase, row, 4 * cc + k8);
          asm volatile("st.shared::cta.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[0]), "r"(pk[1]),
                       "r"(pk[2]), "r"(pk[3])
                       : "memory");
        }
      }
      {
        float la, lb;
        f2unpack(l2, la, lb);
        l_run += la + lb;
      }
      // S read out: the MMA may overwrite it; P written: the product may read it
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars + B_PFULL + 8u * grp);
      }
      ++uses;
    }
    // item done: this group's last product has completed
    if (t0 < it.n) {
      int ok = at_wait_bar(p, bars + B_PFREE + 8u * grp, (uses - 1u) & 1u, WHERE_EPILOGUE, i) ? 1 : 0;
      if (!__all_sync(0xffffffffu, ok)) return;
    }
    // merge the two groups' (maximum, sum, O): exchange maxima, then scaled sums
    xch[grp * AT_T + row] = m_run;
    if (!pair_sync(p, pbar, pair_ph, i)) return;
    const float m0 = xch[row], m1 = xch[AT_T + row];
    if (!pair_sync(p, pbar, pair_ph, i)) return;
    const bool h0 = par < it.n, h1 = (par ^ 1) < it.n;       // the group had tiles of this item
    const float m = h0 ? (h1 ? fmaxf(m0, m1) : m0) : m1;
    const float f0 = h0 ? ex2(m0 - m) : 0.f, f1 = h1 ? ex2(m1 - m) : 0.f;
    xch[grp * AT_T + row] = l_run * (grp ? f1 : f0);
    if (!pair_sync(p, pbar, pair_ph, i)) return;
    const float l_all = (h0 ? xch[row] : 0.f) + (h1 ? xch[AT_T + row] : 0.f);
    if (!pair_sync(p, pbar, pair_ph, i)) return;
    tc_fence_after();
    const float inv = (l_all > 0.f) ? 1.f / l_all : 0.f;
    const bool row_ok = qpos < p.s_r;
    const int c0 = 64 * grp;                                 // this group writes output columns c0 .. c0+63
    uint8_t* orow = p.out[it.r] + ((static_cast<size_t>(it.h) * p.s_r + qpos) * AT_D + c0) * 2;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v0[32], v1[32];
      tc_ld_32x32b_x32(obase + static_cast<uint32_t>(c0 + 32 * cc), v0);
      tc_ld_32x32b_x32(obase + AT_T + static_cast<uint32_t>(c0 + 32 * cc), v1);
      tc_wait_ld();
      if (!row_ok) continue;
      float o[32];
#pragma unroll
      for (int q = 0; q < 32; ++q)
        o[q] = (h0 ? (h1 ? fmaf(__uint_as_float(v0[q]), f0, __uint_as_float(v1[q]) * f1)
                         : __uint_as_float(v0[q]) * f0)
                   : __uint_as_float(v1[q]) * f1) * inv;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_global_v4(orow + (32 * cc + 8 * q) * 2, pack_bf16x2(o[8 * q], o[8 * q + 1]),
                     pack_bf16x2(o[8 * q + 2], o[8 * q + 3]), pack_bf16x2(o[8 * q + 4], o[8 * q + 5]),
                     pack_bf16x2(o[8 * q + 6], o[8 * q + 7]));
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + B_OFREE);
  }
}

// The ring's transfers: piece = (rank r, step j >= 1, head h, key tile kt, K or V),
// in the order the work list needs them (ranks as the items run, then step,
// head, tile).  Copy warp w takes pieces w, w + n_workers, ...; each lane
// streams 16-byte vectors, 16 loads in flight; after a piece every lane fences
// and lane 0 counts it in its (rank, step, head) counter.
__device__ void at_copy(const AttnParams& p) {
  const int lane = threadIdx.x & 31;
  const int cw = (threadIdx.x >> 5) - 10;
  if (cw >= p.n_cw) return;
  const int worker = blockIdx.x * p.n_cw + cw;
  const int n_workers = gridDim.x * p.n_cw;
  {
    int ok = 1;
    if (lane == 0) ok = at_wait_value(p, &p.hdr[HDR_READY], p.epoch, WHERE_COPY, worker) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  }
  const long long per_r = static_cast<long long>(p.heads) * (p.R - 1) * p.nkt * 2;
  const long long total = per_r * p.R;
  bool skip_first = (p.inject == 1 && worker == 0);
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
    int stop = 0;
    if (lane == 0) stop = at_aborted(p) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, stop, 0)) return;
    const int rows = min(AT_T, p.s_r - kt * AT_T);
    const size_t src_off = (static_cast<size_t>(h) * p.s_r + static_cast<size_t>(kt) * AT_T) * AT_D * 2;
    const size_t dst_off =
        ((static_cast<size_t>(j - 1) * p.heads + h) * p.s_r + static_cast<size_t>(kt) * AT_T) * AT_D * 2;
    const uint8_t* src = (isv ? p.vsrc[s] : p.ksrc[s]) + src_off;
    uint8_t* dst = (isv ? p.vrecv[r] : p.krecv[r]) + dst_off;
    const size_t n16 = static_cast<size_t>(rows) * AT_D * 2 / 16;
    constexpr int U = 16;
    for (size_t i0 = lane; i0 < n16; i0 += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t idx = i0 + static_cast<size_t>(u) * 32;
        if (idx < n16) v[u] = ld_nc_v4(src + idx * 16);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t idx = i0 + static_cast<size_t>(u) * 32;
        if (idx < n16) st_global_v4(dst + idx * 16, v[u].x, v[u].y, v[u].z, v[u].w);
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      if (skip_first) skip_first = false;
      else atomicAdd(at_counter(p, r, j, h), 1u);
    }
    __syncwarp();
  }
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars + B_KFULL + 8u * s, 1);
      mbar_init(bars + B_SFULL + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars + B_PFULL + 8u * b, 6);   // four softmax warps, the V load, the K load
      mbar_init(bars + B_PFREE + 8u * b, 1);
    }
    mbar_init(bars + B_OFREE, 8);
    mbar_init(bars + B_DRAIN, 1);       // MMA drain
    for (int qq = 0; qq < 4; ++qq) mbar_init(bars + B_PAIR + 8u * qq, 2);
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
  if (warp == 0 || warp == 12) {
    if (lane == 0) {
      if (warp == 0) at_producer<false>(p, bars, base);
      else at_producer<true>(p, bars, base);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) at_mma(p, bars, base, tmem);
    __syncwarp();
  } else if (warp <= 9) {
    at_softmax(p, bars, base, tmem, reinterpret_cast<float*>(smem + AT_XCH));
    __syncwarp();
  } else if (warp <= 11 && p.copy) {
    at_copy(p);
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
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.cnt = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + L.cnt_off);
  p.hdr = static_cast<uint32_t*>(workspace);
  p.wait_ns = default_wait_ns(cfg);
  p.inject = cfg ? cfg->inject : 0;
  p.epoch = next_epoch();
  p.n_cw = 2;   // warps 10-11
  const uint64_t rows = static_cast<uint64_t>(heads) * s_r;
  for (int r = 0; r < R; ++r) {
    p.out[r] = static_cast<uint8_t*>(out[r]);
    p.ksrc[r] = static_cast<const uint8_t*>(k[r]);
    p.vsrc[r] = static_cast<const uint8_t*>(v[r]);
    if (!make_map_a(&p.tmQ[r], q[r], AT_D, rows, AT_D * 2) || !make_map_a(&p.tmK[r], k[r], AT_D, rows, AT_D * 2) ||
        !make_map_b_chunks(&p.tmV[r], v[r], rows, AT_D, 2))
      return MK_ERR_CUDA;
    if (need_recv) {
      p.krecv[r] = static_cast<uint8_t*>(k_recv[r]);
      p.vrecv[r] = static_cast<uint8_t*>(v_recv[r]);
      const uint64_t rrows = rows * (R - 1);
      if (!make_map_a(&p.tmKr[r], k_recv[r], AT_D, rrows, AT_D * 2) ||
          !make_map_b_chunks(&p.tmVr[r], v_recv[r], rrows, AT_D, 2))
        return MK_ERR_CUDA;
    }
  }
  const int n_items = R * heads * L.nqt;
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
