// A CPU model of the signalling protocol of the fused kernels (test
// infrastructure; built and run by tests/test_protocol_cpu.py).
//
// CTAs are std::threads.  Every wait of the kernels is a bounded spin on a
// std::atomic, every publication the release that pairs with it, and the data
// they order (gathered rows, running sums, hidden activations) are plain ints,
// so ThreadSanitizer reports any access the protocol leaves unordered.  The
// work lists follow the kernels' own orders: the AllGather copy order (remote
// shards in ring order from local+1, local shard last), the compute order
// (local shard first), the grouped raster, the running-sum chain's
// part-major groups of one wave, the chained MLP's up-projection items ahead
// of its down-projection items, the MoE tile table in (rank, expert, row tile,
// column block) order, the combine's hand-over ring, ring attention's
// step-major transfers, and CTA pairs sharing one MMA issuer whose
// two accumulator buffers are freed by both CTAs' epilogues.
//
// Roles per CTA: a producer (waits for its item's inputs, then reads them), the
// pair's MMA issuer (one per pair: waits for both producers and for the
// accumulator buffer), an epilogue (waits for the accumulator and, in the
// running-sum chain, for the previous part; then publishes), and copy workers
// (never wait once started).  Each model launch runs twice with epochs 1 and
// 2 on the same flags, as back-to-back calls on one workspace do.
//
//   protocol_model ag  R m_r n_nblk n_pairs pair n_cw rows_per_piece local copy_local [bug]
//   protocol_model rs  R m n_nblk n_ctas pair group_m [bug]
//   protocol_model mlp R m f_nblk h_nblk n_ctas pair n_cw rows_per_piece
//   protocol_model moe R E_loc n_nblk n_units pair n_cw rows_per_piece seed
//   protocol_model combine R T topk n_nblk n_ctas n_cw ring_entries seed [bug]
//   protocol_model attn R heads key_tiles n_ctas n_cw causal
//   protocol_model rsv R m n_nblk n_ctas pair group_m atomic|last [bug]
// with an optional last argument wait=S (the wait bound, default 20 s).
// Prints "OK" and exits 0, or exits 2 on a wait that gives up (a deadlock in
// the modelled protocol) and 3 on wrong data.  Planted mistakes, for the
// tests that the model catches them: ag bug "relaxed" makes the copy workers
// publish with relaxed increments (the race a missing fence would be); rs bug
// "reversed" runs each group's parts in descending order (a chain that waits
// on work queued behind it); combine bug "earlyfree" frees a ring entry before
// reading it (a race with the next lap's writer); rsv bug "nozerowait" adds
// into the accumulators without waiting for the zero flags.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <string>
#include <thread>
#include <vector>

namespace {

constexpr int BM = 128;      // rows of a CTA's tile
constexpr int KW = 4;        // model words per matrix row
double g_wait_s = 20.0;        // bound of every wait (seconds; argument "wait=S")

std::atomic<int> g_fail{0};

// Bounded wait until pred() holds (the kernels bound every wait in time).
bool wait_until(const std::function<bool()>& pred, const char* what, long long who) {
  const auto t0 = std::chrono::steady_clock::now();
  while (!pred()) {
    if (g_fail.load(std::memory_order_relaxed)) return false;
    if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > g_wait_s) {
      std::fprintf(stderr, "wait gave up: %s (%lld)\n", what, who);
      g_fail.store(2);
      return false;
    }
    std::this_thread::yield();
  }
  return true;
}

void fail_data(const char* what, long long a, long long b) {
  std::fprintf(stderr, "wrong data: %s (%lld vs %lld)\n", what, a, b);
  int z = 0;
  g_fail.compare_exchange_strong(z, 3);
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Grouped raster over (m-position, n-block).
void raster(int q, int group_m, int n_mrow, int n_nblk, int& mb, int& nb) {
  const int per_group = group_m * n_nblk;
  const int g = q / per_group;
  const int first_m = g * group_m;
  const int gsz = std::min(n_mrow - first_m, group_m);
  const int r = q - g * per_group;
  mb = first_m + r % gsz;
  nb = r / gsz;
}

// One modelled launch: n_units CTA units (a pair or a single CTA), each with
// `halves` producer/epilogue threads, one MMA issuer, and copy workers.
struct Item {
  bool empty = false;
  std::function<bool()> inputs;     // producer: wait for and read the inputs
  std::function<bool()> epilogue;   // epilogue: chain wait, store, publish
};

struct Launch {
  int n_units = 1, halves = 1, n_items = 0, n_cw = 0;
  std::function<Item(int item, int half)> decode;
  std::function<void(int worker, int n_workers)> copy;      // copy worker body
  std::function<void()> prologue;                           // the ticket-0 CTA's counter reset

  void run(uint32_t epoch, std::atomic<uint32_t>& ready) {
    std::vector<std::thread> th;
    // per unit: items loaded per half, accumulators issued, epilogues done per half
    struct Unit {
      std::atomic<int> loaded[2];
      std::atomic<int> issued{0};
      std::atomic<int> done[2];
      Unit() { loaded[0] = loaded[1] = done[0] = done[1] = 0; }
    };
    std::vector<Unit> units(n_units);
    auto my_items = [&](int u) {
      std::vector<int> v;
      for (int i = u; i < n_items; i += n_units) v.push_back(i);
      return v;
    };
    for (int u = 0; u < n_units; ++u) {
      for (int h = 0; h < halves; ++h) {
        // producer
        th.emplace_back([&, u, h] {
          if (u == 0 && h == 0 && prologue) {
            prologue();
            ready.store(epoch, std::memory_order_release);
          }
          if (!wait_until([&] { return ready.load(std::memory_order_acquire) == epoch; }, "ready", u)) return;
          int k = 0;
          for (int i : my_items(u)) {
            // the operand ring holds less than an item: item k+1's loads start once
            // the MMAs of item k have been issued
            if (!wait_until([&] { return units[u].issued.load(std::memory_order_acquire) >= k; }, "ring", i))
              return;
            Item it = decode(i, h);
            if (!it.empty && it.inputs && !it.inputs()) return;
            units[u].loaded[h].store(++k, std::memory_order_release);
          }
        });
        // epilogue
        th.emplace_back([&, u, h] {
          int k = 0;
          for (int i : my_items(u)) {
            ++k;
            if (!wait_until([&] { return units[u].issued.load(std::memory_order_acquire) >= k; }, "accumulator", i))
              return;
            Item it = decode(i, h);
            if (!it.empty && it.epilogue && !it.epilogue()) return;
            units[u].done[h].store(k, std::memory_order_release);
          }
        });
      }
      // the unit's MMA issuer: both halves loaded, and the accumulator buffer of
      // two items back drained by both epilogues
      th.emplace_back([&, u] {
        int k = 0;
        for (int i : my_items(u)) {
          ++k;
          for (int h = 0; h < halves; ++h) {
            if (!wait_until([&] { return units[u].loaded[h].load(std::memory_order_acquire) >= k; }, "loads", i)) return;
            if (!wait_until([&] { return units[u].done[h].load(std::memory_order_acquire) >= k - 2; }, "tmem", i)) return;
          }
          units[u].issued.store(k, std::memory_order_release);
        }
      });
      // copy workers of the unit's CTAs
      for (int h = 0; h < halves && copy; ++h)
        for (int w = 0; w < n_cw; ++w)
          th.emplace_back([&, u, h, w] {
            if (!wait_until([&] { return ready.load(std::memory_order_acquire) == epoch; }, "ready", u)) return;
            copy((u * halves + h) * n_cw + w, n_units * halves * n_cw);
          });
    }
    for (auto& t : th) t.join();
  }
};

int arg(char** argv, int i) { return std::atoi(argv[i]); }

// ------------------------------------------------------------------ AllGather + GEMM
int run_ag(int argc, char** argv) {
  if (argc < 11) return 64;
  const int R = arg(argv, 2), m_r = arg(argv, 3), n_nblk = arg(argv, 4), n_units = arg(argv, 5);
  const int pair = arg(argv, 6), n_cw = arg(argv, 7), pr = arg(argv, 8), local = arg(argv, 9);
  const int copy_local = arg(argv, 10);
  const bool relaxed = argc > 11 && std::string(argv[11]) == "relaxed";
  const int M = R * m_r, n_mblk = ceil_div(M, BM);
  const bool ordered = m_r % BM == 0;
  const int bps = m_r / BM;
  const int n_chunks = ordered ? (copy_local ? R : R - 1) * bps : n_mblk;
  const int J = BM / pr;
  auto shard_val = [](int s, int row, int w) { return s * 1000003 + row * 131 + w; };
  std::vector<int> gathered(static_cast<size_t>(M) * KW, -1);
  auto reset_gathered = [&] {
    std::fill(gathered.begin(), gathered.end(), -1);
    if (!copy_local)   // the local block of the gathered A is the local shard itself
      for (int row = 0; row < m_r; ++row)
        for (int w = 0; w < KW; ++w)
          gathered[(static_cast<size_t>(local) * m_r + row) * KW + w] = shard_val(local, row, w);
  };
  std::vector<std::atomic<uint32_t>> cnt(n_mblk);
  std::vector<int> c_tiles(static_cast<size_t>(n_mblk) * n_nblk, 0);
  std::atomic<uint32_t> ready{0};
  auto copy_mb = [&](int c) { return ordered ? ((local + 1 + c / bps) % R) * bps + c % bps : c; };
  auto compute_mb = [&](int pos) { return ordered ? ((local + pos / bps) % R) * bps + pos % bps : pos; };
  auto pieces = [&](int mb) { return ceil_div(std::min(BM, M - mb * BM), pr); };
  auto fully_local = [&](int mb) {
    const int lo = mb * BM, hi = std::min(lo + BM, M);
    return lo >= local * m_r && hi <= (local + 1) * m_r;
  };
  Launch L;
  L.n_units = n_units;
  L.halves = pair ? 2 : 1;
  L.n_cw = n_cw;
  const int n_mrow = pair ? (n_mblk + 1) / 2 : n_mblk;
  L.n_items = n_mrow * n_nblk;
  L.prologue = [&] { for (auto& c : cnt) c.store(0, std::memory_order_relaxed); };
  L.copy = [&](int worker, int n_workers) {
    for (long long pc = worker; pc < static_cast<long long>(n_chunks) * J; pc += n_workers) {
      const int c = static_cast<int>(pc / J), j = static_cast<int>(pc % J);
      const int mb = copy_mb(c);
      if (j >= pieces(mb)) continue;
      const int lo = mb * BM + j * pr, hi = std::min({lo + pr, (mb + 1) * BM, M});
      for (int row = lo; row < hi; ++row) {
        const int s = row / m_r;
        if (s == local && !copy_local) continue;
        for (int w = 0; w < KW; ++w) gathered[static_cast<size_t>(row) * KW + w] = shard_val(s, row - s * m_r, w);
      }
      cnt[mb].fetch_add(1, relaxed ? std::memory_order_relaxed : std::memory_order_release);
    }
  };
  L.decode = [&](int i, int half) {
    Item it;
    int pos = i / n_nblk;
    const int nb = i % n_nblk;
    if (pair) pos = 2 * pos + half;
    if (pos >= n_mblk) {
      it.empty = true;
      return it;
    }
    const int mb = compute_mb(pos);
    it.inputs = [&, mb, i] {
      if (!fully_local(mb)) {
        const uint32_t want = static_cast<uint32_t>(pieces(mb));
        if (!wait_until([&] { return cnt[mb].load(std::memory_order_acquire) == want; }, "chunk", i)) return false;
      }
      for (int row = mb * BM; row < std::min((mb + 1) * BM, M); ++row) {
        const int s = row / m_r;
        for (int w = 0; w < KW; ++w) {
          const int got = fully_local(mb) ? shard_val(s, row - s * m_r, w) : gathered[static_cast<size_t>(row) * KW + w];
          if (got != shard_val(s, row - s * m_r, w)) {
            fail_data("gathered row", got, shard_val(s, row - s * m_r, w));
            return false;
          }
        }
      }
      return true;
    };
    it.epilogue = [&, mb, nb] {
      c_tiles[static_cast<size_t>(mb) * n_nblk + nb] += 1;
      return true;
    };
    return it;
  };
  for (uint32_t e = 1; e <= 2 && !g_fail.load(); ++e) {
    reset_gathered();
    L.run(e, ready);
  }
  for (size_t t = 0; t < c_tiles.size() && !g_fail.load(); ++t)
    if (c_tiles[t] != 2) fail_data("output tile stores", c_tiles[t], 2);
  return g_fail.load();
}

// ------------------------------------------------------------------ the running-sum chain
struct Chain {
  int P, n_mblk, n_nblk, n_mrow, n_sched, G, group_m, pair;
  std::vector<std::atomic<uint32_t>>* flags;
  std::vector<long long>* sums;
  std::vector<long long>* out;
  bool reversed = false;   // planted mistake: the parts of a group in descending order
  // item -> (mb, nb, part), or empty half
  bool decode(int i, int half, int& mb, int& nb, int& part) const {
    const int g = i / (G * P);
    const int Gg = std::min(G, n_sched - g * G);
    const int iin = i - g * G * P;
    part = iin / Gg;
    const int q_in = iin - part * Gg;
    if (reversed) part = P - 1 - part;
    const int q = g * G + q_in;
    raster(q, group_m, n_mrow, n_nblk, mb, nb);
    if (pair) mb = 2 * mb + half;
    return mb < n_mblk;
  }
  static long long partial(int tile, int part) { return 1000LL * tile + 7 * part + 1; }
  // epilogue of (tile, part): wait for part-1, add, store or forward, release
  bool epilogue(int mb, int nb, int part, uint32_t epoch, int item) const {
    const int tile = mb * n_nblk + nb;
    const size_t slot = static_cast<size_t>(tile) * P + part;
    if (part > 0 && !wait_until([&] { return (*flags)[slot - 1].load(std::memory_order_acquire) == epoch; },
                                "chain", item))
      return false;
    const long long s = (part > 0 ? (*sums)[tile] : 0) + partial(tile, part);
    if (part == P - 1) (*out)[tile] = s;
    else (*sums)[tile] = s;
    (*flags)[slot].store(epoch, std::memory_order_release);
    return true;
  }
  bool check() const {
    for (int t = 0; t < n_mblk * n_nblk; ++t) {
      long long want = 0;
      for (int p = 0; p < P; ++p) want += partial(t, p);
      if ((*out)[t] != want) {
        fail_data("reduced tile", (*out)[t], want);
        return false;
      }
    }
    return true;
  }
};

int run_rs(int argc, char** argv) {
  if (argc < 8) return 64;
  const int R = arg(argv, 2), m = arg(argv, 3), n_nblk = arg(argv, 4), n_ctas = arg(argv, 5);
  const int pair = arg(argv, 6), group_m = arg(argv, 7);
  const int n_mblk = ceil_div(m, BM);
  std::vector<std::atomic<uint32_t>> flags(static_cast<size_t>(n_mblk) * n_nblk * R);
  std::vector<long long> sums(static_cast<size_t>(n_mblk) * n_nblk), out(sums.size());
  Chain ch;
  ch.P = R;
  ch.n_mblk = n_mblk;
  ch.n_nblk = n_nblk;
  ch.pair = pair;
  ch.group_m = group_m;
  ch.n_mrow = pair ? (n_mblk + 1) / 2 : n_mblk;
  ch.n_sched = ch.n_mrow * n_nblk;
  const int n_units = pair ? std::max(1, n_ctas / 2) : n_ctas;
  ch.G = std::max(1, std::min(n_units, ch.n_sched));
  ch.flags = &flags;
  ch.sums = &sums;
  ch.out = &out;
  ch.reversed = argc > 8 && std::string(argv[8]) == "reversed";
  std::atomic<uint32_t> ready{0};
  Launch L;
  L.n_units = n_units;
  L.halves = pair ? 2 : 1;
  L.n_items = ch.n_sched * ch.P;
  L.prologue = [] {};
  uint32_t epoch = 0;
  L.decode = [&](int i, int half) {
    Item it;
    int mb, nb, part;
    if (!ch.decode(i, half, mb, nb, part)) {
      it.empty = true;
      return it;
    }
    it.epilogue = [&, mb, nb, part, i] { return ch.epilogue(mb, nb, part, epoch, i); };
    return it;
  };
  for (uint32_t e = 1; e <= 2 && !g_fail.load(); ++e) {
    epoch = e;
    std::fill(out.begin(), out.end(), 0);
    L.run(e, ready);
    if (!g_fail.load()) ch.check();
  }
  return g_fail.load();
}

// ------------------------------------------------------------------ RS / AR reduction variants
// Items (tile, part) with a tile's parts consecutive.  "atomic": the spare
// warps of every CTA zero their share of the fp32 accumulator tiles and then
// publish the CTA's zero flag; an epilogue waits once for every CTA's flag,
// adds its rows into the tile's accumulator (relaxed atomic adds), and counts
// each 32-row quarter (a release); the warp whose count completes a quarter
// reads the accumulator and stores the output rows.  "last": every partial is
// staged in its own slot (plain stores) and counted the same way; the warp that
// completes a quarter sums the slots in rank order.  The quarter counters are
// zeroed by the ticket-0 CTA before the ready word.
int run_rsv(int argc, char** argv) {
  if (argc < 9) return 64;
  const int R = arg(argv, 2), m = arg(argv, 3), n_nblk = arg(argv, 4), n_ctas = arg(argv, 5);
  const int pair = arg(argv, 6), group_m = arg(argv, 7);
  const bool atomic_mode = std::string(argv[8]) == "atomic";
  const bool skip_zero_wait = argc > 9 && std::string(argv[9]) == "nozerowait";
  const int n_mblk = ceil_div(m, BM), P = R, Q = 4, QR = 8;   // 4 quarters, 8 model rows each
  const int n_tiles = n_mblk * n_nblk;
  const int n_mrow = pair ? (n_mblk + 1) / 2 : n_mblk, n_sched = n_mrow * n_nblk;
  const int n_units = pair ? std::max(1, n_ctas / 2) : n_ctas, halves = pair ? 2 : 1;
  const int grid = n_units * halves;
  auto partial = [](int tile, int part, int row) { return 1000LL * tile + 37LL * part + row + 1; };
  std::vector<std::atomic<long long>> acc(static_cast<size_t>(n_tiles) * Q * QR);
  std::vector<long long> slots(static_cast<size_t>(n_tiles) * P * Q * QR, 0);
  std::vector<long long> out(static_cast<size_t>(n_tiles) * Q * QR, 0);
  std::vector<std::atomic<uint32_t>> qcnt(static_cast<size_t>(n_tiles) * Q), zflag(grid), zdone(grid);
  std::atomic<uint32_t> ready{0};
  uint32_t epoch = 0;
  Launch L;
  L.n_units = n_units;
  L.halves = halves;
  L.n_cw = atomic_mode ? 3 : 0;   // the spare warps zero the accumulators
  L.n_items = n_sched * P;
  L.prologue = [&] { for (auto& c : qcnt) c.store(0, std::memory_order_relaxed); };
  if (atomic_mode)
    L.copy = [&](int worker, int) {
      const int cta = worker / L.n_cw, w = worker % L.n_cw;
      const size_t total = acc.size(), per = (total + grid - 1) / grid;
      const size_t lo = std::min(total, static_cast<size_t>(cta) * per), hi = std::min(total, lo + per);
      for (size_t x = lo + w; x < hi; x += L.n_cw) acc[x].store(0, std::memory_order_relaxed);
      // the spare warps meet at a named barrier; one of them publishes the flag
      if (zdone[cta].fetch_add(1, std::memory_order_acq_rel) == static_cast<uint32_t>(L.n_cw - 1))
        zflag[cta].store(epoch, std::memory_order_release);
    };
  std::vector<int> zero_seen(grid, 0);
  L.decode = [&](int i, int half) {
    Item it;
    const int q = i / P, part = i % P;
    int mb, nb;
    raster(q, group_m, n_mrow, n_nblk, mb, nb);
    if (pair) mb = 2 * mb + half;
    if (mb >= n_mblk) {
      it.empty = true;
      return it;
    }
    const int tile = mb * n_nblk + nb;
    const int cta = (i % n_units) * halves + half;
    it.epilogue = [&, tile, part, cta, i] {
      if (atomic_mode && !zero_seen[cta] && !skip_zero_wait) {
        for (int c = 0; c < grid; ++c)
          if (!wait_until([&] { return zflag[c].load(std::memory_order_acquire) == epoch; }, "zero flags", i))
            return false;
        zero_seen[cta] = 1;
      }
      for (int qq = 0; qq < Q; ++qq) {
        for (int row = 0; row < QR; ++row) {
          const size_t x = (static_cast<size_t>(tile) * Q + qq) * QR + row;
          const long long v = partial(tile, part, qq * QR + row);
          if (atomic_mode) acc[x].fetch_add(v, std::memory_order_relaxed);
          else slots[((static_cast<size_t>(tile) * P + part) * Q + qq) * QR + row] = v;
        }
        const uint32_t before = qcnt[static_cast<size_t>(tile) * Q + qq].fetch_add(1, std::memory_order_acq_rel);
        if (before != static_cast<uint32_t>(P - 1)) continue;
        for (int row = 0; row < QR; ++row) {   // this warp completes the quarter
          const size_t x = (static_cast<size_t>(tile) * Q + qq) * QR + row;
          long long sum = 0;
          if (atomic_mode) sum = acc[x].load(std::memory_order_relaxed);
          else
            for (int p2 = 0; p2 < P; ++p2) sum += slots[((static_cast<size_t>(tile) * P + p2) * Q + qq) * QR + row];
          out[x] = sum;
        }
      }
      return true;
    };
    return it;
  };
  for (uint32_t e = 1; e <= 2 && !g_fail.load(); ++e) {
    epoch = e;
    std::fill(out.begin(), out.end(), 0);
    std::fill(zero_seen.begin(), zero_seen.end(), 0);
    for (auto& z : zdone) z.store(0, std::memory_order_relaxed);
    for (auto& a : acc) a.store(e == 1 ? 0 : 123456789, std::memory_order_relaxed);   // stale sums
    L.run(e, ready);
    for (int t = 0; t < n_tiles && !g_fail.load(); ++t)
      for (int r = 0; r < Q * QR; ++r) {
        long long want = 0;
        for (int p2 = 0; p2 < P; ++p2) want += partial(t, p2, r);
        if (out[static_cast<size_t>(t) * Q * QR + r] != want) {
          fail_data("reduced row", out[static_cast<size_t>(t) * Q * QR + r], want);
          break;
        }
      }
  }
  return g_fail.load();
}

// ------------------------------------------------------------------ the chained MLP
int run_mlp(int argc, char** argv) {
  if (argc < 10) return 64;
  const int R = arg(argv, 2), m = arg(argv, 3), f_nblk = arg(argv, 4), h_nblk = arg(argv, 5);
  const int n_ctas = arg(argv, 6), pair = arg(argv, 7), n_cw = arg(argv, 8), pr = arg(argv, 9);
  const int M = R * m, n_mblk = ceil_div(M, BM);
  const int n_mrow = pair ? (n_mblk + 1) / 2 : n_mblk;
  const int n_units = pair ? std::max(1, n_ctas / 2) : n_ctas;
  const int J = BM / pr;
  auto x_val = [](int row, int w) { return row * 17 + w + 5; };
  auto h_val = [](int r, int row, int nb) { return r * 7919 + row * 3 + nb; };
  std::vector<int> xg(static_cast<size_t>(M) * KW, -1);
  std::vector<int> hid(static_cast<size_t>(R) * M * f_nblk, -1);
  std::vector<std::atomic<uint32_t>> chunk(n_mblk), hcnt(static_cast<size_t>(R) * n_mblk);
  std::vector<std::atomic<uint32_t>> flags(static_cast<size_t>(n_mblk) * h_nblk * R);
  std::vector<long long> sums(static_cast<size_t>(n_mblk) * h_nblk), out(sums.size());
  auto pieces = [&](int mb) { return ceil_div(std::min(BM, M - mb * BM), pr); };
  Chain ch;
  ch.P = R;
  ch.n_mblk = n_mblk;
  ch.n_nblk = h_nblk;
  ch.pair = pair;
  ch.group_m = 8;
  ch.n_mrow = n_mrow;
  ch.n_sched = n_mrow * h_nblk;
  ch.G = std::max(1, std::min(n_units, ch.n_sched));
  ch.flags = &flags;
  ch.sums = &sums;
  ch.out = &out;
  const int n1 = n_mrow * R * f_nblk;
  std::atomic<uint32_t> ready{0};
  uint32_t epoch = 0;
  Launch L;
  L.n_units = n_units;
  L.halves = pair ? 2 : 1;
  L.n_cw = n_cw;
  L.n_items = n1 + ch.n_sched * ch.P;
  L.prologue = [&] {
    for (auto& c : chunk) c.store(0, std::memory_order_relaxed);
    for (auto& c : hcnt) c.store(0, std::memory_order_relaxed);
  };
  L.copy = [&](int worker, int n_workers) {
    for (long long pc = worker; pc < static_cast<long long>(n_mblk) * J; pc += n_workers) {
      const int mb = static_cast<int>(pc / J), j = static_cast<int>(pc % J);
      if (j >= pieces(mb)) continue;
      const int lo = mb * BM + j * pr, hi = std::min({lo + pr, (mb + 1) * BM, M});
      for (int row = lo; row < hi; ++row)
        for (int w = 0; w < KW; ++w) xg[static_cast<size_t>(row) * KW + w] = x_val(row, w);
      chunk[mb].fetch_add(1, std::memory_order_release);
    }
  };
  L.decode = [&](int i, int half) {
    Item it;
    if (i < n1) {   // up-projection: groups of 8 m-positions; inside one rank, n-block, m-position
      const int GM = 8, per_m = R * f_nblk;
      const int g = i / (GM * per_m);
      const int Gg = std::min(GM, n_mrow - g * GM);
      const int iin = i - g * GM * per_m;
      const int r = iin / (Gg * f_nblk);
      const int rem = iin - r * Gg * f_nblk;
      const int nb = rem / Gg;
      int pos = g * GM + (rem - nb * Gg);
      if (pair) pos = 2 * pos + half;
      if (pos >= n_mblk) {
        it.empty = true;
        return it;
      }
      const int mb = pos;
      it.inputs = [&, mb, i] {
        const uint32_t want = static_cast<uint32_t>(pieces(mb));
        if (!wait_until([&] { return chunk[mb].load(std::memory_order_acquire) == want; }, "x chunk", i)) return false;
        for (int row = mb * BM; row < std::min((mb + 1) * BM, M); ++row)
          if (xg[static_cast<size_t>(row) * KW] != x_val(row, 0)) {
            fail_data("gathered x", xg[static_cast<size_t>(row) * KW], x_val(row, 0));
            return false;
          }
        return true;
      };
      it.epilogue = [&, mb, r, nb] {
        for (int row = mb * BM; row < std::min((mb + 1) * BM, M); ++row)
          hid[(static_cast<size_t>(r) * M + row) * f_nblk + nb] = h_val(r, row, nb);
        hcnt[static_cast<size_t>(r) * n_mblk + mb].fetch_add(1, std::memory_order_release);
        return true;
      };
      return it;
    }
    int mb, nb, part;
    if (!ch.decode(i - n1, half, mb, nb, part)) {
      it.empty = true;
      return it;
    }
    const int r = part;   // one part per rank
    it.inputs = [&, mb, r, i] {
      if (!wait_until([&] {
            return hcnt[static_cast<size_t>(r) * n_mblk + mb].load(std::memory_order_acquire) ==
                   static_cast<uint32_t>(f_nblk);
          }, "hidden block", i))
        return false;
      for (int row = mb * BM; row < std::min((mb + 1) * BM, M); ++row)
        for (int fb = 0; fb < f_nblk; ++fb)
          if (hid[(static_cast<size_t>(r) * M + row) * f_nblk + fb] != h_val(r, row, fb)) {
            fail_data("hidden rows", hid[(static_cast<size_t>(r) * M + row) * f_nblk + fb], h_val(r, row, fb));
            return false;
          }
      return true;
    };
    it.epilogue = [&, mb, nb, part, i] { return ch.epilogue(mb, nb, part, epoch, i); };
    return it;
  };
  for (uint32_t e = 1; e <= 2 && !g_fail.load(); ++e) {
    epoch = e;
    std::fill(out.begin(), out.end(), 0);
    std::fill(hid.begin(), hid.end(), -1);
    std::fill(xg.begin(), xg.end(), -1);
    L.run(e, ready);
    if (!g_fail.load()) ch.check();
  }
  return g_fail.load();
}

// ------------------------------------------------------------------ MoE dispatch + grouped GEMM
// Expert segments of random sizes; the tile table lists, for each (rank d,
// local expert l) in order, its row tiles (128 rows, or 256 with CTA pairs)
// times the column blocks; copy workers move the received rows of every rank
// in pieces and count them per 128-row block; a tile waits until every block
// it covers holds all its rows.  The counters are zeroed by an earlier launch.
int run_moe(int argc, char** argv) {
  if (argc < 10) return 64;
  const int R = arg(argv, 2), E_loc = arg(argv, 3), n_nblk = arg(argv, 4), n_units = arg(argv, 5);
  const int pair = arg(argv, 6), n_cw = arg(argv, 7), pr = arg(argv, 8);
  unsigned seed = static_cast<unsigned>(arg(argv, 9));
  auto rnd = [&] { seed = seed * 1103515245u + 12345u; return (seed >> 8) % 1000u; };
  const int tile_rows = pair ? 2 * BM : BM;
  std::vector<int> seg(static_cast<size_t>(R) * E_loc), segoff(static_cast<size_t>(R) * (E_loc + 1));
  std::vector<int> rc(R, 0);
  for (int d = 0; d < R; ++d) {
    for (int l = 0; l < E_loc; ++l) {
      const unsigned u = rnd();
      seg[static_cast<size_t>(d) * E_loc + l] = u < 150 ? 0 : static_cast<int>(u % 700);   // some empty experts
      segoff[static_cast<size_t>(d) * (E_loc + 1) + l] = rc[d];
      rc[d] += seg[static_cast<size_t>(d) * E_loc + l];
    }
    segoff[static_cast<size_t>(d) * (E_loc + 1) + E_loc] = rc[d];
  }
  struct Ent { int d, first, rows, nb; };
  std::vector<Ent> table;
  for (int d = 0; d < R; ++d)
    for (int l = 0; l < E_loc; ++l) {
      const int tot = seg[static_cast<size_t>(d) * E_loc + l];
      for (int mi = 0; mi < ceil_div(tot, tile_rows); ++mi)
        for (int nb = 0; nb < n_nblk; ++nb)
          table.push_back({d, segoff[static_cast<size_t>(d) * (E_loc + 1) + l] + mi * tile_rows,
                           std::min(tile_rows, tot - mi * tile_rows), nb});
    }
  auto row_val = [](int d, int row) { return d * 100003 + row * 7 + 1; };
  std::vector<std::vector<int>> recv(R);
  std::vector<int> nblk(R);
  std::vector<std::vector<std::atomic<uint32_t>>> cnt(R);
  for (int d = 0; d < R; ++d) {
    recv[d].assign(static_cast<size_t>(std::max(rc[d], 1)), -1);
    nblk[d] = ceil_div(std::max(rc[d], 1), BM);
    cnt[d] = std::vector<std::atomic<uint32_t>>(nblk[d]);
  }
  std::vector<int> y(table.size() * 2, 0);
  long long total_pieces = 0;
  for (int d = 0; d < R; ++d) total_pieces += ceil_div(rc[d], pr);
  std::atomic<uint32_t> ready{0};
  Launch L;
  L.n_units = n_units;
  L.halves = pair ? 2 : 1;
  L.n_cw = n_cw;
  L.n_items = static_cast<int>(table.size());
  L.prologue = [] {};
  L.copy = [&](int worker, int n_workers) {
    for (long long q = worker; q < total_pieces; q += n_workers) {
      int d = 0;
      long long j = q;
      while (j >= ceil_div(rc[d], pr)) j -= ceil_div(rc[d++], pr);
      const int row0 = static_cast<int>(j) * pr, rows = std::min(pr, rc[d] - row0);
      for (int r = 0; r < rows; ++r) recv[d][row0 + r] = row_val(d, row0 + r);
      cnt[d][row0 / BM].fetch_add(static_cast<uint32_t>(rows), std::memory_order_release);
    }
  };
  L.decode = [&](int i, int half) {
    Item it;
    const Ent& e = table[i];
    const int first = e.first + half * BM, rows = std::min(BM, e.rows - half * BM);
    if (rows <= 0) {
      it.empty = true;
      return it;
    }
    const int d = e.d;
    it.inputs = [&, d, first, rows, i] {
      for (int b = first / BM; b <= (first + rows - 1) / BM; ++b) {
        const uint32_t want = static_cast<uint32_t>(std::min(BM, rc[d] - b * BM));
        if (!wait_until([&] { return cnt[d][b].load(std::memory_order_acquire) == want; }, "rows", i)) return false;
      }
      for (int r = first; r < first + rows; ++r)
        if (recv[d][r] != row_val(d, r)) {
          fail_data("received row", recv[d][r], row_val(d, r));
          return false;
        }
      return true;
    };
    it.epilogue = [&, i, half] {
      y[static_cast<size_t>(i) * 2 + half] += 1;
      return true;
    };
    return it;
  };
  for (uint32_t e = 1; e <= 2 && !g_fail.load(); ++e) {
    for (int d = 0; d < R; ++d) {   // the offsets launch zeroes the block counters
      for (auto& c : cnt[d]) c.store(0, std::memory_order_relaxed);
      std::fill(recv[d].begin(), recv[d].end(), -1);
    }
    ready.store(e, std::memory_order_release);
    L.run(e, ready);
  }
  for (size_t i = 0; i < table.size() && !g_fail.load(); ++i)
    for (int h = 0; h < L.halves; ++h)
      if (std::min(BM, table[i].rows - h * BM) > 0 && y[i * 2 + h] != 2) fail_data("expert tile stores", y[i * 2 + h], 2);
  return g_fail.load();
}

// ------------------------------------------------------------------ ring attention
// Items (rank, head, query tile), the last rank's first; an item visits its own
// block, then the blocks of ranks r-1, r-2, ... (step j), and before the first
// key tile of a remote step waits until the (rank, step, head) counter holds
// all 2 * nkt pieces (K and V of every key tile) that the copy workers move
// into the rank's receive buffer, step-major.  Causal: only earlier ranks'
// blocks and the diagonal block's first tiles.
int run_attn(int argc, char** argv) {
  if (argc < 8) return 64;
  const int R = arg(argv, 2), heads = arg(argv, 3), nkt = arg(argv, 4), n_units = arg(argv, 5);
  const int n_cw = arg(argv, 6), causal = arg(argv, 7);
  const int nqt = nkt;
  auto kv_val = [](int s, int h, int kt, int isv) { return ((s * 97 + h) * 89 + kt) * 2 + isv + 1; };
  auto rix = [&](int r, int j, int h, int kt, int isv) {
    return (((static_cast<size_t>(r) * R + j) * heads + h) * nkt + kt) * 2 + isv;
  };
  std::vector<int> recv(static_cast<size_t>(R) * R * heads * nkt * 2, -1);
  std::vector<std::atomic<uint32_t>> cnt(static_cast<size_t>(R) * R * heads);
  std::atomic<uint32_t> ready{0};
  const int per_r = heads * nqt;
  Launch L;
  L.n_units = n_units;
  L.halves = 1;
  L.n_cw = n_cw;
  L.n_items = R * per_r;
  L.prologue = [&] { for (auto& c : cnt) c.store(0, std::memory_order_relaxed); };
  L.copy = [&](int worker, int n_workers) {
    const long long per = static_cast<long long>(heads) * (R - 1) * nkt * 2;
    for (long long q = worker; q < per * R; q += n_workers) {
      const int r = R - 1 - static_cast<int>(q / per);
      long long rem = q % per;
      const int j = 1 + static_cast<int>(rem / (static_cast<long long>(heads) * nkt * 2));
      rem %= static_cast<long long>(heads) * nkt * 2;
      const int h = static_cast<int>(rem / (nkt * 2)), kt = static_cast<int>(rem % (nkt * 2)) / 2;
      const int isv = static_cast<int>(rem & 1);
      const int s = (r - j + R) % R;
      if (causal && s > r) continue;
      recv[rix(r, j, h, kt, isv)] = kv_val(s, h, kt, isv);
      cnt[(static_cast<size_t>(r) * R + j) * heads + h].fetch_add(1, std::memory_order_release);
    }
  };
  L.decode = [&](int i, int) {
    Item it;
    const int r = R - 1 - i / per_r, rem = i % per_r, h = rem / nqt, qt = rem % nqt;
    const int n = causal ? (qt + 1) + r * nkt : R * nkt;
    it.inputs = [&, r, h, qt, n, i] {
      int waited = 0;
      for (int t = 0; t < n; ++t) {
        int j, s, kt;
        if (causal && t <= qt) {
          j = 0; s = r; kt = t;
        } else if (causal) {
          const int u = t - (qt + 1);
          j = 1 + u / nkt; s = r - j; kt = u % nkt;
        } else {
          j = t / nkt; kt = t % nkt; s = (r - j + R) % R;
        }
        if (j == 0) continue;   // the rank's own block, read in place
        if (j != waited) {
          const uint32_t want = static_cast<uint32_t>(2 * nkt);
          if (!wait_until([&] { return cnt[(static_cast<size_t>(r) * R + j) * heads + h].load(std::memory_order_acquire) == want; },
                          "ring step", i))
            return false;
          waited = j;
        }
        for (int isv = 0; isv < 2; ++isv)
          if (recv[rix(r, j, h, kt, isv)] != kv_val(s, h, kt, isv)) {
            fail_data("received K/V tile", recv[rix(r, j, h, kt, isv)], kv_val(s, h, kt, isv));
            return false;
          }
      }
      return true;
    };
    return it;
  };
  for (uint32_t e = 1; e <= 2 && !g_fail.load(); ++e) {
    std::fill(recv.begin(), recv.end(), -1);
    L.run(e, ready);
  }
  return g_fail.load();
}

// ------------------------------------------------------------------ MoE combine
// Every (token, slot) row of every column block is produced by some tile's
// epilogue, which stores it into ret[r][t][slot] and counts it in the (token,
// column block) counter (a release after the stores); the row that completes
// a count hands (token, column block) to its CTA's copy warps through a ring
// of `cap` entries whose sequence word is 2s when entry s is free and 2s + 1
// when full.  A copy warp claims up to 8 entries at a time (tail / claim
// counters), frees each entry for the next lap, then sums the token's slots;
// it leaves when its CTA's epilogue is done and every entry is claimed.
int run_combine(int argc, char** argv) {
  if (argc < 9) return 64;
  const int R = arg(argv, 2), T = arg(argv, 3), topk = arg(argv, 4), n_nblk = arg(argv, 5);
  const int n_units = arg(argv, 6), n_cw = arg(argv, 7), cap = arg(argv, 8);
  unsigned seed = argc > 9 ? static_cast<unsigned>(arg(argv, 9)) : 1u;
  const bool early_free = argc > 10 && std::string(argv[10]) == "earlyfree";
  auto rnd = [&] { seed = seed * 1103515245u + 12345u; return seed >> 8; };
  const int n_tok = R * T, n_rows = n_tok * topk;
  std::vector<int> order(n_rows);   // the dispatch order of the (token, slot) rows
  for (int i = 0; i < n_rows; ++i) order[i] = i;
  for (int i = n_rows - 1; i > 0; --i) std::swap(order[i], order[rnd() % (i + 1)]);
  const int n_tiles = ceil_div(n_rows, BM);
  auto val = [](int g, int k, int nb) { return g * 31 + k * 7 + nb + 1; };
  std::vector<int> ret(static_cast<size_t>(n_rows) * n_nblk, 0), out(static_cast<size_t>(n_tok) * n_nblk, 0);
  std::vector<int> writes(out.size(), 0);
  std::vector<std::atomic<uint32_t>> cnt(out.size());
  struct Ring {
    std::vector<std::atomic<uint32_t>> seq;
    std::vector<int> payload;
    std::atomic<uint32_t> tail{0}, claim{0}, done{0};
  };
  std::vector<Ring> rings(n_units);
  for (auto& rg : rings) {
    rg.seq = std::vector<std::atomic<uint32_t>>(cap);
    rg.payload.assign(static_cast<size_t>(cap) * 2, 0);
  }
  Launch L;
  L.n_units = n_units;
  L.halves = 1;
  L.n_items = n_tiles * n_nblk;
  L.n_cw = n_cw;
  std::atomic<uint32_t> ready{0};
  std::vector<std::atomic<int>> epi_left(n_units);
  L.prologue = [] {};
  L.decode = [&](int i, int) {
    Item it;
    const int tile = i / n_nblk, nb = i % n_nblk;
    const int u = i % n_units;
    it.epilogue = [&, tile, nb, u, i] {
      Ring& rg = rings[u];
      for (int j = tile * BM; j < std::min((tile + 1) * BM, n_rows); ++j) {
        const int g = order[j] / topk, k = order[j] % topk;
        ret[static_cast<size_t>(order[j]) * n_nblk + nb] = val(g, k, nb);
        const uint32_t before = cnt[static_cast<size_t>(g) * n_nblk + nb].fetch_add(1, std::memory_order_acq_rel);
        if (before != static_cast<uint32_t>(topk - 1)) continue;
        const uint32_t slot = rg.tail.fetch_add(1, std::memory_order_acq_rel);
        if (!wait_until([&] { return rg.seq[slot % cap].load(std::memory_order_acquire) == 2u * slot; }, "ring free", i))
          return false;
        rg.payload[(slot % cap) * 2] = g;
        rg.payload[(slot % cap) * 2 + 1] = nb;
        rg.seq[slot % cap].store(2u * slot + 1u, std::memory_order_release);
      }
      if (epi_left[u].fetch_sub(1, std::memory_order_acq_rel) == 1) rg.done.store(1, std::memory_order_release);
      return true;
    };
    return it;
  };
  L.copy = [&](int worker, int) {
    Ring& rg = rings[worker / n_cw];
    const auto t0 = std::chrono::steady_clock::now();
    while (true) {
      const uint32_t done = rg.done.load(std::memory_order_acquire);
      const uint32_t tail = rg.tail.load(std::memory_order_acquire);
      uint32_t claim = rg.claim.load(std::memory_order_acquire);
      if (claim < tail) {
        const uint32_t n = std::min(8u, tail - claim);
        if (!rg.claim.compare_exchange_strong(claim, claim + n, std::memory_order_acq_rel)) continue;
        std::vector<std::pair<int, int>> got;
        for (uint32_t s = claim; s < claim + n; ++s) {
          if (!wait_until([&] { return rg.seq[s % cap].load(std::memory_order_acquire) == 2u * s + 1u; },
                          "ring full", static_cast<long long>(s)))
            return;
          if (early_free) rg.seq[s % cap].store(2u * (s + static_cast<uint32_t>(cap)), std::memory_order_release);
          got.emplace_back(rg.payload[(s % cap) * 2], rg.payload[(s % cap) * 2 + 1]);
          if (!early_free) rg.seq[s % cap].store(2u * (s + static_cast<uint32_t>(cap)), std::memory_order_release);
        }
        for (auto [g, nb] : got) {
          int sum = 0;
          for (int k = 0; k < topk; ++k) sum += ret[static_cast<size_t>(g * topk + k) * n_nblk + nb];
          out[static_cast<size_t>(g) * n_nblk + nb] = sum;
          writes[static_cast<size_t>(g) * n_nblk + nb] += 1;
        }
      } else if (done == 1) {
        return;
      } else if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > g_wait_s) {
        std::fprintf(stderr, "wait gave up: copy warp idle\n");
        g_fail.store(2);
        return;
      } else if (g_fail.load()) {
        return;
      } else {
        std::this_thread::yield();
      }
    }
  };
  for (uint32_t e = 1; e <= 2 && !g_fail.load(); ++e) {
    for (auto& c : cnt) c.store(0, std::memory_order_relaxed);   // zeroed by the plan launch
    std::fill(writes.begin(), writes.end(), 0);
    for (int u = 0; u < n_units; ++u) {
      Ring& rg = rings[u];
      for (int x = 0; x < cap; ++x) rg.seq[x].store(2u * x, std::memory_order_relaxed);
      rg.tail = 0;
      rg.claim = 0;
      rg.done = 0;
      int mine = 0;
      for (int i = u; i < L.n_items; i += n_units) ++mine;
      epi_left[u] = mine;
      if (mine == 0) rg.done = 1;
    }
    L.run(e, ready);
    for (int g = 0; g < n_tok && !g_fail.load(); ++g)
      for (int nb = 0; nb < n_nblk; ++nb) {
        int want = 0;
        for (int k = 0; k < topk; ++k) want += val(g, k, nb);
        const size_t x = static_cast<size_t>(g) * n_nblk + nb;
        if (writes[x] != 1) fail_data("combined rows written", writes[x], 1);
        else if (out[x] != want) fail_data("combined row", out[x], want);
      }
  }
  return g_fail.load();
}

}  // namespace

int main(int argc, char** argv) {
  // a trailing "wait=S" sets the wait bound
  if (argc > 2 && std::strncmp(argv[argc - 1], "wait=", 5) == 0) {
    g_wait_s = std::atof(argv[argc - 1] + 5);
    --argc;
  }
  if (argc < 2) return 64;
  const std::string op = argv[1];
  int rc = 64;
  if (op == "ag") rc = run_ag(argc, argv);
  else if (op == "rs") rc = run_rs(argc, argv);
  else if (op == "mlp") rc = run_mlp(argc, argv);
  else if (op == "moe") rc = run_moe(argc, argv);
  else if (op == "combine") rc = run_combine(argc, argv);
  else if (op == "attn") rc = run_attn(argc, argv);
  else if (op == "rsv") rc = run_rsv(argc, argv);
  if (rc == 0) std::printf("OK\n");
  return rc;
}
