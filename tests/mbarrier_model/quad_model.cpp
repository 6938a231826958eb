// Host replay of the cluster-of-four GEMM kernel's barrier protocol.
//
// Four CTAs (ranks 0-3); CTAs 2j and 2j+1 form pair j, the even one its
// leader.  CTA c holds the same A rows as CTA c ^ 2 of the other pair; per
// fill each of the two copies one half of those rows, multicast into both,
// and CTA c copies its own B half.  So a fill of stage s in CTA c is made of
// three pieces: its own A half, the counterpart's A half and its own B;
// each piece completes its bytes on the full barrier of the destination's
// pair leader.
//
// Roles: 0..3 producers (one per CTA), 4 and 5 the MMA issuers of the pair
// leaders 0 and 2, 6..21 epilogue warps (CTA c, warp w: 6 + 4 c + w).
// Barriers as in the kernel: full[L][s] in each pair leader L, one arrival
// (the leader producer's arrive.expect_tx for the pair's 64 KB), completed
// by the pieces landing in both CTAs of the pair; empty[c][s] in every CTA,
// two arrivals: both leaders' commits, each multicast to all four CTAs;
// tmem_full[c][a] in every CTA, arrived by its own leader's commit;
// tmem_empty[L][a] in each leader, eight arrivals (its pair's epilogue
// warps).  Each pair's tensor core completes in issue order, independently
// of the other pair's.
//
// Checked on every interleaving: no deadlock; a piece never lands in a
// stage whose previous fill a pair has not finished reading; the MMA reads a
// stage only when all pieces of its own k-block have landed in both of its
// CTAs; accumulator hand-over; double arrivals; balanced phase counts.
//
// Abort drain: with a fault unit (CTA 0 issues no copy for that unit's first
// fill) or with one producer stopped early (its timeout), the replay must
// deadlock; then all pending completions land, each leader's drain
// arithmetic runs exactly as in the kernel (its own missing arrival, the
// pair peer's bytes, the other pair's A halves for fills their producers
// never issued) and every phase the drains wait on must be complete --
// except the faulted fill's, whose bytes never come.
//
// Built with -DPLANT_OWN_PAIR_RELEASE, each leader's commit releases only its
// own pair's CTAs (empty barriers of one arrival): the other pair's
// producers may then multicast into a stage that is still being read, and
// the replay must catch it.  Built with -DPLANT_DRAIN_OWN_PAIR_ONLY, a
// leader's drain forgets the A halves the other pair's producers never
// copied: a stopped producer of the other pair must leave a phase open.
//
// Usage: quad_model STAGES UNITS NCLUSTERS CLUSTER SPLIT_K KBLOCKS SEEDS MODE [ARG [ARG2]]
//   MODE: normal | fault U | stop C X   (producer of CTA C stops after X fills)
// Prints "OK <n> deadlocks=<d>" or "FAIL <reason>" / "DEADLOCK <where>".

#include "mbar_model.h"
#include "schedule.h"

using gf16::RingPos;
using mbmodel::fail;
using mbmodel::MBar;

namespace {

constexpr uint32_t A_HALF = 8192, B_STAGE = 16384;
constexpr uint32_t OWN_TX = A_HALF + B_STAGE;         // bytes one CTA copies per fill
constexpr uint32_t STAGE_TX = 2 * (2 * A_HALF + B_STAGE);  // bytes landing per pair and fill
constexpr int EPI_WARPS = 4;
constexpr int NROLES = 4 + 2 + 4 * EPI_WARPS;
#ifdef PLANT_OWN_PAIR_RELEASE
constexpr int EMPTY_ARRIVALS = 1;
#else
constexpr int EMPTY_ARRIVALS = 2;
#endif

enum Mode { NORMAL, FAULT, STOP };

struct Params {
  int stages, units, nclusters, cluster, split_k, kblocks;
  Mode mode;
  int arg, arg2;
};

enum StageState { FREE, FILLING, FULL, READING };

int pair_of(int c) { return c >> 1; }

struct Sim {
  Params P;
  mbmodel::Scheduler sch{NROLES};
  std::vector<MBar> full[2];           // [pair] (in the pair's leader)
  std::vector<MBar> empty[4];          // [cta]
  MBar tfull[4][2];                    // [cta][acc]
  MBar tempty[2][2];                   // [pair][acc]
  std::vector<StageState> st[4];
  std::vector<std::pair<int, int>> tag[4];
  std::vector<int> landed[4];
  uint32_t issued[4] = {0, 0, 0, 0};
  int fault_fill = -1;                 // fill index whose CTA-0 copies were skipped
  int acc_unit[2][2] = {{-1, -1}, {-1, -1}}, acc_kbs[2][2] = {{0, 0}, {0, 0}};
  int acc_reads[2][2] = {{0, 0}, {0, 0}};
  bool acc_ready[2][2] = {{false, false}, {false, false}};
  std::deque<std::function<void()>>* tc[2] = {nullptr, nullptr};

  void unit_range(int u, int* kb0, int* kb1) {
    int tpos, s;
    gf16::decode_unit(u, P.split_k, &tpos, &s);
    gf16::split_range(P.kblocks, P.split_k, s, kb0, kb1);
  }

  // A piece of fill (u, kb) about to be written into CTA d's stage sg.
  void claim(int d, uint32_t sg, int u, int kb) {
    if (st[d][sg] == FULL || st[d][sg] == READING)
      fail("a copy lands in a stage whose previous fill is still being read");
    if (st[d][sg] == FREE) {
      st[d][sg] = FILLING;
      tag[d][sg] = {u, kb};
      landed[d][sg] = 0;
    } else if (tag[d][sg] != std::make_pair(u, kb)) {
      fail("two fills of one stage overlap");
    }
  }

  void land(int d, uint32_t sg, uint32_t bytes) {
    landed[d][sg] += 1;
    if (landed[d][sg] == 3) st[d][sg] = FULL;
    full[pair_of(d)][sg].complete_tx(bytes);
  }

  void producer(int c) {
    const int r = c;
    sch.start(r);
    RingPos pos{0, 0};
    bool stop = false;
    for (int u = P.cluster; u < P.units && !stop; u += P.nclusters) {
      int kb0, kb1;
      unit_range(u, &kb0, &kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (P.mode == STOP && c == P.arg && (int)issued[c] == P.arg2) {
          stop = true;  // this producer's wait timed out: it issues nothing more
          break;
        }
        const uint32_t sg = pos.stage, par = gf16::producer_wait_parity(pos);
        sch.wait_until(r, [&] { return empty[c][sg].try_wait(par); });
        if ((c & 1) == 0) full[pair_of(c)][sg].arrive_expect_tx(r, STAGE_TX);
        const bool skip = (P.mode == FAULT && c == 0 && u == P.arg && kb == kb0);
        if (skip) fault_fill = (int)issued[0];
        if (!skip) {
          const int o = c ^ 2;
          claim(c, sg, u, kb);
          claim(o, sg, u, kb);
          sch.copies.push_back({[this, c, sg] { land(c, sg, A_HALF); }});
          sch.copies.push_back({[this, o, sg] { land(o, sg, A_HALF); }});
          sch.copies.push_back({[this, c, sg] { land(c, sg, B_STAGE); }});
        }
        issued[c] += 1;
        gf16::ring_advance(pos, (uint32_t)P.stages);
        sch.role_yield(r);
      }
    }
    sch.finish(r);
  }

  void mma(int pj) {
    const int r = 4 + pj, L = 2 * pj;
    sch.start(r);
    RingPos pos{0, 0};
    uint32_t local = 0;
    for (int u = P.cluster; u < P.units; u += P.nclusters) {
      int kb0, kb1;
      unit_range(u, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      sch.wait_until(r, [&] { return tempty[pj][acc].try_wait(aph ^ 1u); });
      if (acc_unit[pj][acc] != -1 && acc_reads[pj][acc] != 2 * EPI_WARPS)
        fail("MMA overwrites an accumulator the epilogues have not read");
      acc_unit[pj][acc] = u;
      acc_kbs[pj][acc] = 0;
      acc_reads[pj][acc] = 0;
      acc_ready[pj][acc] = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t sg = pos.stage, par = gf16::consumer_wait_parity(pos);
        sch.wait_until(r, [&] { return full[pj][sg].try_wait(par); });
        for (int c = L; c < L + 2; ++c) {
          if (st[c][sg] != FULL) fail("MMA reads a stage whose pieces have not all landed");
          if (tag[c][sg] != std::make_pair(u, kb)) fail("MMA reads the wrong k-block");
          st[c][sg] = READING;
        }
        const int a = (int)acc;
        tc[pj]->push_back([this, pj, a] { acc_kbs[pj][a] += 1; });
        tc[pj]->push_back([this, pj, L, sg] {
          // commit: this pair has finished reading the stage in its CTAs;
          // the arrival goes to all four CTAs' empty barriers
          for (int c = L; c < L + 2; ++c) st[c][sg] = FREE;
#ifdef PLANT_OWN_PAIR_RELEASE
          for (int c = L; c < L + 2; ++c) empty[c][sg].arrive(-1);
#else
          for (int c = 0; c < 4; ++c) empty[c][sg].arrive(-1);
#endif
        });
        gf16::ring_advance(pos, (uint32_t)P.stages);
        sch.role_yield(r);
      }
      const int a = (int)acc, want = kb1 - kb0;
      tc[pj]->push_back([this, pj, L, a, want] {
        if (acc_kbs[pj][a] != want) fail("accumulator handed over before its MMAs finished");
        acc_ready[pj][a] = true;
        tfull[L][a].arrive(-1);
        tfull[L + 1][a].arrive(-1);
      });
      ++local;
      sch.role_yield(r);
    }
    sch.finish(r);
  }

  void epilogue(int c, int w) {
    const int r = 6 + c * EPI_WARPS + w, pj = pair_of(c);
    sch.start(r);
    uint32_t local = 0;
    for (int u = P.cluster; u < P.units; u += P.nclusters) {
      int kb0, kb1;
      unit_range(u, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      sch.wait_until(r, [&] { return tfull[c][acc].try_wait(aph); });
      if (!acc_ready[pj][acc] || acc_unit[pj][acc] != u || acc_kbs[pj][acc] != kb1 - kb0)
        fail("epilogue reads an accumulator that is not this unit's finished tile");
      sch.role_yield(r);
      acc_reads[pj][acc] += 1;
      tempty[pj][acc].arrive(r);
      ++local;
      sch.role_yield(r);
    }
    sch.finish(r);
  }

  // The kernel's leader_drain for leader L, on the model's barriers, after
  // every issued copy has landed.  Returns the number of phases left
  // incomplete; only the faulted fill's may stay open.
  int drain(int L) {
    const uint32_t S = (uint32_t)P.stages;
    uint32_t hi = 0;
    for (int c = 0; c < 4; ++c) hi = issued[c] > hi ? issued[c] : hi;
    const uint32_t lo = hi > S ? hi - S : 0u;
    int incomplete = 0;
    for (uint32_t j = lo; j < hi; ++j) {
      MBar& bar = full[pair_of(L)][j % S];
      if (j >= issued[L]) bar.arrive_expect_tx(-1, STAGE_TX - OWN_TX);
      if (j >= issued[L ^ 1]) bar.complete_tx(OWN_TX);
#ifndef PLANT_DRAIN_OWN_PAIR_ONLY
      if (j >= issued[L ^ 2]) bar.complete_tx(A_HALF);
      if (j >= issued[L ^ 3]) bar.complete_tx(A_HALF);
#endif
      if (!bar.try_wait((j / S) & 1u)) {
        if ((int)j != fault_fill) fail("drain leaves fill " + std::to_string(j) + " incomplete");
        ++incomplete;
      }
    }
    return incomplete;
  }
};

}  // namespace

int main(int argc, char** argv) {
  if (argc < 9) {
    std::fprintf(stderr, "usage: quad_model STAGES UNITS NCLUSTERS CLUSTER SPLIT_K KBLOCKS SEEDS "
                         "MODE [ARG [ARG2]]\n");
    return 2;
  }
  Params P;
  P.stages = std::atoi(argv[1]);
  P.units = std::atoi(argv[2]);
  P.nclusters = std::atoi(argv[3]);
  P.cluster = std::atoi(argv[4]);
  P.split_k = std::atoi(argv[5]);
  P.kblocks = std::atoi(argv[6]);
  const int seeds = std::atoi(argv[7]);
  const std::string mode = argv[8];
  P.arg = argc > 9 ? std::atoi(argv[9]) : -1;
  P.arg2 = argc > 10 ? std::atoi(argv[10]) : -1;
  P.mode = mode == "fault" ? FAULT : mode == "stop" ? STOP : NORMAL;
  int deadlocks = 0;
  for (int seed = 0; seed < seeds; ++seed) {
    Sim* sim = new Sim();  // leaked on deadlock (threads detached)
    sim->P = P;
    sim->sch.seed(0x9E3779B97F4A7C15ull * (uint64_t)(seed + 1));
    sim->tc[0] = &sim->sch.tc_queue;
    sim->tc[1] = &sim->sch.tc_queue_b;
    for (int pj = 0; pj < 2; ++pj) {
      sim->full[pj].resize(P.stages);
      for (int s = 0; s < P.stages; ++s)
        sim->full[pj][s].init("full[" + std::to_string(pj) + "][" + std::to_string(s) + "]", 1,
                              /*negative_tx_ok=*/true);
      for (int a = 0; a < 2; ++a) sim->tempty[pj][a].init("tmem_empty", 2 * EPI_WARPS);
    }
    for (int c = 0; c < 4; ++c) {
      sim->empty[c].resize(P.stages);
      for (int s = 0; s < P.stages; ++s)
        sim->empty[c][s].init("empty[" + std::to_string(c) + "][" + std::to_string(s) + "]",
                              EMPTY_ARRIVALS);
      for (int a = 0; a < 2; ++a) sim->tfull[c][a].init("tmem_full", 1);
      sim->st[c].assign(P.stages, FREE);
      sim->tag[c].assign(P.stages, {-1, -1});
      sim->landed[c].assign(P.stages, 0);
    }
    std::vector<std::function<void()>> roles;
    for (int c = 0; c < 4; ++c) roles.push_back([sim, c] { sim->producer(c); });
    for (int pj = 0; pj < 2; ++pj) roles.push_back([sim, pj] { sim->mma(pj); });
    for (int c = 0; c < 4; ++c)
      for (int w = 0; w < EPI_WARPS; ++w) roles.push_back([sim, c, w] { sim->epilogue(c, w); });
    std::string where;
    const int rc = sim->sch.run(roles, &where);
    if (P.mode == NORMAL) {
      if (rc != 0) {
        std::printf("DEADLOCK%s\n", where.c_str());
        std::fflush(stdout);
        std::_Exit(1);
      }
      std::vector<int> per_stage(P.stages, 0);
      int my_units = 0;
      RingPos pos{0, 0};
      for (int u = P.cluster; u < P.units; u += P.nclusters) {
        int kb0, kb1;
        sim->unit_range(u, &kb0, &kb1);
        ++my_units;
        for (int kb = kb0; kb < kb1; ++kb) {
          per_stage[pos.stage] += 1;
          gf16::ring_advance(pos, (uint32_t)P.stages);
        }
      }
      for (int s = 0; s < P.stages; ++s) {
        for (int pj = 0; pj < 2; ++pj)
          if (sim->full[pj][s].completions != per_stage[s]) fail("full phase count mismatch");
        for (int c = 0; c < 4; ++c)
          if (sim->empty[c][s].completions != per_stage[s]) fail("empty phase count mismatch");
      }
      const int a0 = (my_units + 1) / 2, a1 = my_units / 2;
      for (int c = 0; c < 4; ++c)
        if (sim->tfull[c][0].completions != a0 || sim->tfull[c][1].completions != a1)
          fail("tmem_full phase count mismatch");
      for (int pj = 0; pj < 2; ++pj)
        if (sim->tempty[pj][0].completions != a0 || sim->tempty[pj][1].completions != a1)
          fail("tmem_empty phase count mismatch");
      if (sim->drain(0) != 0 || sim->drain(2) != 0) fail("drain after a normal run is not a no-op");
      delete sim;
      continue;
    }
    // abort modes: a deadlock is what the kernel's bounded waits escape
    if (rc != 1) {
      if (sim->fault_fill >= 0) fail("fault injected but the replay finished");
      delete sim;
      continue;
    }
    ++deadlocks;
    // every issued copy lands before the drains (they wait for exactly that)
    while (!sim->sch.copies.empty()) {
      auto f = sim->sch.copies.back().land;
      sim->sch.copies.pop_back();
      f();
    }
    const int left = sim->drain(0) + sim->drain(2);
    // the faulted fill misses CTA 0's pieces in both pairs (its own A half
    // and B in pair 0, its A half in CTA 2 of pair 1)
    if (P.mode == FAULT && left != 2) fail("the faulted fill should stay incomplete in both pairs");
    if (P.mode != FAULT && left != 0) fail("drain left phases incomplete");
  }
  std::printf("OK %d deadlocks=%d\n", seeds, deadlocks);
  std::fflush(stdout);
  std::_Exit(0);
}
