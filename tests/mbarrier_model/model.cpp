// Host replay of the GEMM kernel's barrier protocol, for testing the
// pipeline's schedule without a GPU.
//
// The mbarrier is modelled exactly as the "mbarrier State and Operations"
// page defines it: init sets phase 0, pending = expected = count, tx = 0;
// arrive takes one off pending; arrive.expect_tx takes one off pending and
// adds bytes to tx; a finished copy takes its bytes off tx (complete_tx);
// tcgen05.commit arrives once when the earlier tensor-core operations are
// done; a phase completes when pending == 0 and tx == 0, which flips the
// parity and reloads pending from expected; try_wait(parity) only reads.
//
// The three roles of one CTA (TMA producer, MMA issuer, four epilogue
// warps) run as threads, but only one at a time: a seeded scheduler picks
// which runnable role, copy completion or tensor-core completion goes next,
// so every run is one reproducible interleaving.  The role loops use the
// same index and parity helpers as the device code (schedule.h).
//
// Checked on every interleaving:
//   * no deadlock (some role or event can always move until all finish);
//   * a stage is refilled only after the MMAs reading it completed;
//   * the MMA reads a stage only when all of its copies have landed, and it
//     holds the k-block the schedule says it should;
//   * an accumulator is overwritten only after all epilogue warps read it,
//     and the epilogue reads a complete accumulator of the right unit;
//   * no role arrives twice on one barrier phase (the double-arrive hazard
//     of the "Xe2 Nbarrier Pipelining" page);
//   * every barrier completes exactly as many phases as the schedule has
//     fills / releases (waits and arrivals balanced).
// With a fault unit, the copies of that unit's first stage are never
// issued: the replay must then stop with the MMA role blocked on exactly
// that stage's full barrier (the state the kernel's bounded wait escapes).
//
// Usage: model STAGES UNITS GRID CTA SPLIT_K KBLOCKS SEEDS [FAULT_UNIT]
// Prints "OK <n>" or "FAIL <reason>" / "DEADLOCK <where>".

#include <condition_variable>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <deque>
#include <functional>
#include <mutex>
#include <random>
#include <set>
#include <string>
#include <thread>
#include <vector>

#include "schedule.h"

using gf16::RingPos;

namespace {

constexpr uint32_t TX_A = 16384, TX_B = 8192, N_B_COPIES = 4;
constexpr uint32_t STAGE_TX = TX_A + N_B_COPIES * TX_B;
constexpr int EPI_WARPS = 4;

[[noreturn]] void fail(const std::string& why) {
  std::printf("FAIL %s\n", why.c_str());
  std::fflush(stdout);
  std::_Exit(1);
}

struct MBar {
  std::string name;
  uint32_t phase = 0;
  int expected = 0, pending = 0;
  int64_t tx = 0;
  int completions = 0;
  std::set<int> arrivers;  // roles that arrived in the current phase

  void init(const std::string& n, int count) {
    name = n;
    phase = 0;
    expected = pending = count;
    tx = 0;
    completions = 0;
    arrivers.clear();
  }
  void maybe_complete() {
    if (pending == 0 && tx == 0) {
      phase ^= 1u;
      pending = expected;
      ++completions;
      arrivers.clear();
    }
  }
  void note_arriver(int role) {
    if (role >= 0 && !arrivers.insert(role).second)
      fail("double arrive on " + name + " by role " + std::to_string(role));
  }
  void arrive(int role) {
    note_arriver(role);
    if (pending <= 0) fail("arrive with no pending arrival on " + name);
    --pending;
    maybe_complete();
  }
  void arrive_expect_tx(int role, uint32_t bytes) {
    note_arriver(role);
    if (pending <= 0) fail("arrive.expect_tx with no pending arrival on " + name);
    --pending;
    tx += bytes;
    maybe_complete();
  }
  void complete_tx(uint32_t bytes) {
    tx -= bytes;
    if (tx < 0) fail("tx count below zero on " + name);
    maybe_complete();
  }
  bool try_wait(uint32_t parity) const { return phase != parity; }
};

struct Params {
  int stages, units, grid, cta, split_k, kblocks, fault_unit;
};

enum StageState { FREE, FILLING, FULL, READING };

struct Sim {
  Params P;
  std::mt19937_64 rng;
  std::mutex mu;
  std::condition_variable cv;
  int turn = -1;  // which role thread may run; -1 = scheduler
  // roles: 0 producer, 1 mma, 2..5 epilogue warps
  static constexpr int NROLES = 2 + EPI_WARPS;
  bool done[NROLES] = {};
  std::function<bool()> waiting[NROLES];  // wait predicate, empty = runnable

  std::vector<MBar> full, empty;
  MBar tfull[2], tempty[2];
  std::vector<StageState> st;
  std::vector<std::pair<int, int>> tag;  // (unit, kb) loaded into the stage
  std::vector<int> landed;               // copies landed for the current fill
  // accumulator state
  int acc_unit[2] = {-1, -1}, acc_kbs[2] = {0, 0}, acc_reads[2] = {0, 0};
  bool acc_ready[2] = {false, false};

  // asynchronous events
  struct Copy { int stage; uint32_t bytes; };
  std::vector<Copy> copies;            // complete in any order
  std::deque<std::function<void()>> tc_queue;  // tensor-core ops complete in order

  void role_yield(int r) {  // give the token back and wait for it again
    std::unique_lock<std::mutex> lk(mu);
    turn = -1;
    cv.notify_all();
    cv.wait(lk, [&] { return turn == r; });
  }
  void wait_until(int r, std::function<bool()> pred) {
    while (!pred()) {
      waiting[r] = pred;
      role_yield(r);
      waiting[r] = nullptr;
    }
  }
  void finish(int r) {
    std::unique_lock<std::mutex> lk(mu);
    done[r] = true;
    turn = -1;
    cv.notify_all();
  }
  void start(int r) {
    std::unique_lock<std::mutex> lk(mu);
    cv.wait(lk, [&] { return turn == r; });
  }

  // ------------------------------------------------------------ roles
  void producer() {
    const int r = 0;
    start(r);
    RingPos pos{0, 0};
    for (int u = P.cta; u < P.units; u += P.grid) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t sg = pos.stage, par = gf16::producer_wait_parity(pos);
        wait_until(r, [&] { return empty[sg].try_wait(par); });
        if (st[sg] != FREE) fail("producer refills a stage that is still in use");
        full[sg].arrive_expect_tx(r, STAGE_TX);
        st[sg] = FILLING;
        tag[sg] = {u, kb};
        landed[sg] = 0;
        if (!(u == P.fault_unit && kb == kb0)) {
          copies.push_back({(int)sg, TX_A});
          for (uint32_t j = 0; j < N_B_COPIES; ++j) copies.push_back({(int)sg, TX_B});
        }
        gf16::ring_advance(pos, (uint32_t)P.stages);
        role_yield(r);
      }
    }
    finish(r);
  }

  void mma() {
    const int r = 1;
    start(r);
    RingPos pos{0, 0};
    uint32_t local = 0;
    for (int u = P.cta; u < P.units; u += P.grid) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      wait_until(r, [&] { return tempty[acc].try_wait(aph ^ 1u); });
      if (acc_unit[acc] != -1 && acc_reads[acc] != EPI_WARPS)
        fail("MMA overwrites an accumulator the epilogue has not read");
      acc_unit[acc] = u;
      acc_kbs[acc] = 0;
      acc_reads[acc] = 0;
      acc_ready[acc] = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t sg = pos.stage, par = gf16::consumer_wait_parity(pos);
        wait_until(r, [&] { return full[sg].try_wait(par); });
        if (st[sg] != FULL) fail("MMA reads a stage whose copies have not all landed");
        if (tag[sg] != std::make_pair(u, kb)) fail("MMA reads the wrong k-block");
        st[sg] = READING;
        const int a = (int)acc;
        tc_queue.push_back([this, a] { acc_kbs[a] += 1; });        // the MMAs
        tc_queue.push_back([this, sg] {                              // commit -> empty
          st[sg] = FREE;
          empty[sg].arrive(-1);
        });
        gf16::ring_advance(pos, (uint32_t)P.stages);
        role_yield(r);
      }
      const int a = (int)acc, want = kb1 - kb0;
      tc_queue.push_back([this, a, want] {  // commit -> tmem_full
        if (acc_kbs[a] != want) fail("accumulator handed over before its MMAs finished");
        acc_ready[a] = true;
        tfull[a].arrive(-1);
      });
      ++local;
      role_yield(r);
    }
    finish(r);
  }

  void epilogue(int w) {
    const int r = 2 + w;
    start(r);
    uint32_t local = 0;
    for (int u = P.cta; u < P.units; u += P.grid) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      wait_until(r, [&] { return tfull[acc].try_wait(aph); });
      if (!acc_ready[acc] || acc_unit[acc] != u || acc_kbs[acc] != kb1 - kb0)
        fail("epilogue reads an accumulator that is not this unit's finished tile");
      role_yield(r);  // the loads and stores take a while
      acc_reads[acc] += 1;
      tempty[acc].arrive(r);
      ++local;
      role_yield(r);
    }
    finish(r);
  }

  // ------------------------------------------------------------ scheduler
  // Returns 0 when all roles finished, 1 on deadlock.
  int run(std::string* where) {
    std::vector<std::thread> th;
    th.emplace_back([this] { producer(); });
    th.emplace_back([this] { mma(); });
    for (int w = 0; w < EPI_WARPS; ++w) th.emplace_back([this, w] { epilogue(w); });
    int rc = 0;
    while (true) {
      std::unique_lock<std::mutex> lk(mu);
      cv.wait(lk, [&] { return turn == -1; });
      std::vector<int> choices;  // role r, or NROLES + i for copy i, or -2 for tc
      for (int r = 0; r < NROLES; ++r)
        if (!done[r] && (!waiting[r] || waiting[r]())) choices.push_back(r);
      for (size_t i = 0; i < copies.size(); ++i) choices.push_back(NROLES + (int)i);
      if (!tc_queue.empty()) choices.push_back(-2);
      bool all_done = true;
      for (int r = 0; r < NROLES; ++r) all_done = all_done && done[r];
      if (choices.empty()) {
        if (!all_done) {
          rc = 1;
          *where = "";
          for (int r = 0; r < NROLES; ++r)
            if (!done[r]) *where += " role" + std::to_string(r);
        }
        break;
      }
      const int c = choices[rng() % choices.size()];
      if (c == -2) {
        auto f = tc_queue.front();
        tc_queue.pop_front();
        f();
      } else if (c >= NROLES) {
        const Copy cp = copies[c - NROLES];
        copies.erase(copies.begin() + (c - NROLES));
        landed[cp.stage] += 1;
        if (landed[cp.stage] == 1 + (int)N_B_COPIES) st[cp.stage] = FULL;
        full[cp.stage].complete_tx(cp.bytes);
      } else {
        turn = c;
        cv.notify_all();
      }
    }
    if (rc == 0) {
      for (auto& t : th) t.join();
    } else {
      for (auto& t : th) t.detach();  // blocked roles are abandoned; process exits
    }
    return rc;
  }
};

}  // namespace

int main(int argc, char** argv) {
  if (argc < 8) {
    std::fprintf(stderr, "usage: model STAGES UNITS GRID CTA SPLIT_K KBLOCKS SEEDS [FAULT_UNIT]\n");
    return 2;
  }
  Params P;
  P.stages = std::atoi(argv[1]);
  P.units = std::atoi(argv[2]);
  P.grid = std::atoi(argv[3]);
  P.cta = std::atoi(argv[4]);
  P.split_k = std::atoi(argv[5]);
  P.kblocks = std::atoi(argv[6]);
  const int seeds = std::atoi(argv[7]);
  P.fault_unit = argc > 8 ? std::atoi(argv[8]) : -1;
  for (int seed = 0; seed < seeds; ++seed) {
    Sim* sim = new Sim();  // leaked on deadlock (threads detached)
    sim->P = P;
    sim->rng.seed(0x9E3779B97F4A7C15ull * (uint64_t)(seed + 1));
    sim->full.resize(P.stages);
    sim->empty.resize(P.stages);
    for (int s = 0; s < P.stages; ++s) {
      sim->full[s].init("full[" + std::to_string(s) + "]", 1);
      sim->empty[s].init("empty[" + std::to_string(s) + "]", 1);
    }
    for (int a = 0; a < 2; ++a) {
      sim->tfull[a].init("tmem_full[" + std::to_string(a) + "]", 1);
      sim->tempty[a].init("tmem_empty[" + std::to_string(a) + "]", EPI_WARPS);
    }
    sim->st.assign(P.stages, FREE);
    sim->tag.assign(P.stages, {-1, -1});
    sim->landed.assign(P.stages, 0);
    std::string where;
    const int rc = sim->run(&where);
    // expected phase counts
    int fills = 0, my_units = 0;
    std::vector<int> per_stage(P.stages, 0);
    {
      RingPos pos{0, 0};
      for (int u = P.cta; u < P.units; u += P.grid) {
        int tpos, s, kb0, kb1;
        gf16::decode_unit(u, P.split_k, &tpos, &s);
        gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
        ++my_units;
        for (int kb = kb0; kb < kb1; ++kb) {
          per_stage[pos.stage] += 1;
          ++fills;
          gf16::ring_advance(pos, (uint32_t)P.stages);
        }
      }
    }
    if (P.fault_unit >= 0 && (P.fault_unit - P.cta) % P.grid == 0 && P.fault_unit >= P.cta &&
        P.fault_unit < P.units) {
      if (rc != 1) fail("fault injected but the replay finished");
      if (!sim->waiting[1]) fail("fault injected but the MMA role is not the one blocked");
      std::printf("DEADLOCK-AS-EXPECTED%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(0);
    }
    if (rc != 0) {
      std::printf("DEADLOCK%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(1);
    }
    for (int s = 0; s < P.stages; ++s) {
      if (sim->full[s].completions != per_stage[s]) fail("full barrier phase count mismatch");
      if (sim->empty[s].completions != per_stage[s]) fail("empty barrier phase count mismatch");
    }
    const int a0 = (my_units + 1) / 2, a1 = my_units / 2;
    if (sim->tfull[0].completions != a0 || sim->tfull[1].completions != a1 ||
        sim->tempty[0].completions != a0 || sim->tempty[1].completions != a1)
      fail("accumulator barrier phase count mismatch");
    if (!sim->copies.empty() || !sim->tc_queue.empty()) fail("work left in flight");
    (void)fills;
    delete sim;
  }
  std::printf("OK %d\n", seeds);
  return 0;
}
