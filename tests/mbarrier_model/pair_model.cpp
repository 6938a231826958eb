// Host replay of the CTA-pair GEMM kernel's barrier protocol.
//
// Roles: 0 leader producer, 1 peer producer, 2 MMA issuer (leader),
// 3..10 epilogue warps (3..6 leader, 7..10 peer).  Barriers as in the
// kernel: full[s] in the leader, one arrival (the leader producer's
// arrive.expect_tx for both CTAs' bytes), completed by three copies per
// CTA; empty[cta][s] and tmem_full[cta][a] in both CTAs, arrived by the
// leader's multicast commits; tmem_empty[a] in the leader, eight arrivals.
// The peer's copies may land before the leader expects them (a negative
// transaction count is allowed, as on the hardware).
//
// Checked on every interleaving, beyond the single-CTA replay's checks
// (deadlock, stage reuse, k-block identity, accumulator hand-over, double
// arrivals, balanced phase counts), for both CTAs' stages.
//
// Abort drain: with a fault unit (the leader issues no copy for that unit's
// first fill) or with one producer stopped early (its timeout), the replay
// must deadlock; then all pending completions land, the leader's drain
// arithmetic runs exactly as in the kernel (arrive for fills the leader
// never reached, complete_tx for the peer's bytes of fills the peer never
// issued), and every phase the drain waits on must be complete -- except
// the faulted fill's, whose own bytes never come.
//
// Usage: pair_model STAGES UNITS NPAIRS PAIR SPLIT_K KBLOCKS SEEDS MODE [ARG]
//   MODE: normal | fault U | stop_leader X | stop_peer Y
// Prints "OK <n>" or "FAIL <reason>" / "DEADLOCK <where>".

#include "mbar_model.h"
#include "schedule.h"

using gf16::RingPos;
using mbmodel::fail;
using mbmodel::MBar;

namespace {

constexpr uint32_t TX_A = 16384, TX_B = 8192;
constexpr uint32_t CTA_STAGE_TX = TX_A + 2 * TX_B;
constexpr int EPI_WARPS = 4;
constexpr int NROLES = 3 + 2 * EPI_WARPS;

enum Mode { NORMAL, FAULT, STOP_LEADER, STOP_PEER };

struct Params {
  int stages, units, npairs, pair, split_k, kblocks;
  Mode mode;
  int arg;
};

enum StageState { FREE, FILLING, FULL, READING };

struct Sim {
  Params P;
  mbmodel::Scheduler sch{NROLES};
  std::vector<MBar> full;              // leader
  std::vector<MBar> empty[2];          // per CTA
  MBar tfull[2][2];                    // [cta][acc]
  MBar tempty[2];                      // leader
  std::vector<StageState> st[2];
  std::vector<std::pair<int, int>> tag[2];
  std::vector<int> landed[2];
  uint32_t issued[2] = {0, 0};
  int fault_fill = -1;                 // fill index whose leader copies were skipped
  int acc_unit[2] = {-1, -1}, acc_kbs[2] = {0, 0}, acc_reads[2] = {0, 0};
  bool acc_ready[2] = {false, false};

  void producer(int cta) {
    const int r = cta;
    sch.start(r);
    RingPos pos{0, 0};
    bool stop = false;
    for (int u = P.pair; u < P.units && !stop; u += P.npairs) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        if ((P.mode == STOP_LEADER && cta == 0 && (int)issued[0] == P.arg) ||
            (P.mode == STOP_PEER && cta == 1 && (int)issued[1] == P.arg)) {
          stop = true;  // this producer's wait timed out: it issues nothing more
          break;
        }
        const uint32_t sg = pos.stage, par = gf16::producer_wait_parity(pos);
        sch.wait_until(r, [&] { return empty[cta][sg].try_wait(par); });
        if (st[cta][sg] != FREE) fail("producer refills a stage that is still in use");
        if (cta == 0) full[sg].arrive_expect_tx(r, 2 * CTA_STAGE_TX);
        st[cta][sg] = FILLING;
        tag[cta][sg] = {u, kb};
        landed[cta][sg] = 0;
        const bool skip = (P.mode == FAULT && cta == 0 && u == P.arg && kb == kb0);
        if (skip) fault_fill = (int)issued[0];
        if (!skip) {
          for (uint32_t bytes : {TX_A, TX_B, TX_B}) {
            sch.copies.push_back({[this, cta, sg, bytes] {
              landed[cta][sg] += 1;
              if (landed[cta][sg] == 3) st[cta][sg] = FULL;
              full[sg].complete_tx(bytes);
            }});
          }
        }
        issued[cta] += 1;
        gf16::ring_advance(pos, (uint32_t)P.stages);
        sch.role_yield(r);
      }
    }
    sch.finish(r);
  }

  void mma() {
    const int r = 2;
    sch.start(r);
    RingPos pos{0, 0};
    uint32_t local = 0;
    for (int u = P.pair; u < P.units; u += P.npairs) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      sch.wait_until(r, [&] { return tempty[acc].try_wait(aph ^ 1u); });
      if (acc_unit[acc] != -1 && acc_reads[acc] != 2 * EPI_WARPS)
        fail("MMA overwrites an accumulator the epilogues have not read");
      acc_unit[acc] = u;
      acc_kbs[acc] = 0;
      acc_reads[acc] = 0;
      acc_ready[acc] = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t sg = pos.stage, par = gf16::consumer_wait_parity(pos);
        sch.wait_until(r, [&] { return full[sg].try_wait(par); });
        for (int c = 0; c < 2; ++c) {
          if (st[c][sg] != FULL) fail("MMA reads a stage whose copies have not all landed");
          if (tag[c][sg] != std::make_pair(u, kb)) fail("MMA reads the wrong k-block");
          st[c][sg] = READING;
        }
        const int a = (int)acc;
        sch.tc_queue.push_back([this, a] { acc_kbs[a] += 1; });
        sch.tc_queue.push_back([this, sg] {  // commit, multicast to both CTAs
          for (int c = 0; c < 2; ++c) {
            st[c][sg] = FREE;
            empty[c][sg].arrive(-1);
          }
        });
        gf16::ring_advance(pos, (uint32_t)P.stages);
        sch.role_yield(r);
      }
      const int a = (int)acc, want = kb1 - kb0;
      sch.tc_queue.push_back([this, a, want] {
        if (acc_kbs[a] != want) fail("accumulator handed over before its MMAs finished");
        acc_ready[a] = true;
        tfull[0][a].arrive(-1);
        tfull[1][a].arrive(-1);
      });
      ++local;
      sch.role_yield(r);
    }
    sch.finish(r);
  }

  void epilogue(int cta, int w) {
    const int r = 3 + cta * EPI_WARPS + w;
    sch.start(r);
    uint32_t local = 0;
    for (int u = P.pair; u < P.units; u += P.npairs) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      sch.wait_until(r, [&] { return tfull[cta][acc].try_wait(aph); });
      if (!acc_ready[acc] || acc_unit[acc] != u || acc_kbs[acc] != kb1 - kb0)
        fail("epilogue reads an accumulator that is not this unit's finished tile");
      sch.role_yield(r);
      acc_reads[acc] += 1;
      tempty[acc].arrive(r);
      ++local;
      sch.role_yield(r);
    }
    sch.finish(r);
  }

  // The kernel's leader_drain, on the model's barriers, after every issued
  // copy has landed.  Returns the number of phases left incomplete.
  int drain() {
    const uint32_t mine = issued[0], peer = issued[1];
    const uint32_t S = (uint32_t)P.stages;
    const uint32_t hi = mine > peer ? mine : peer;
    const uint32_t lo = hi > S ? hi - S : 0u;
    int incomplete = 0;
    for (uint32_t j = lo; j < hi; ++j) {
      MBar& bar = full[j % S];
      if (j >= mine) bar.arrive_expect_tx(-1, CTA_STAGE_TX);
      if (j >= peer) bar.complete_tx(CTA_STAGE_TX);
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
    std::fprintf(stderr,
                 "usage: pair_model STAGES UNITS NPAIRS PAIR SPLIT_K KBLOCKS SEEDS MODE [ARG]\n");
    return 2;
  }
  Params P;
  P.stages = std::atoi(argv[1]);
  P.units = std::atoi(argv[2]);
  P.npairs = std::atoi(argv[3]);
  P.pair = std::atoi(argv[4]);
  P.split_k = std::atoi(argv[5]);
  P.kblocks = std::atoi(argv[6]);
  const int seeds = std::atoi(argv[7]);
  const std::string mode = argv[8];
  P.arg = argc > 9 ? std::atoi(argv[9]) : -1;
  P.mode = mode == "fault" ? FAULT : mode == "stop_leader" ? STOP_LEADER
         : mode == "stop_peer" ? STOP_PEER : NORMAL;
  int deadlocks = 0;
  for (int seed = 0; seed < seeds; ++seed) {
    Sim* sim = new Sim();  // leaked on deadlock (threads detached)
    sim->P = P;
    sim->sch.seed(0xD1B54A32D192ED03ull * (uint64_t)(seed + 1));
    sim->full.resize(P.stages);
    for (int s = 0; s < P.stages; ++s)
      sim->full[s].init("full[" + std::to_string(s) + "]", 1, /*negative_tx_ok=*/true);
    for (int c = 0; c < 2; ++c) {
      sim->empty[c].resize(P.stages);
      for (int s = 0; s < P.stages; ++s)
        sim->empty[c][s].init("empty[" + std::to_string(c) + "][" + std::to_string(s) + "]", 1);
      for (int a = 0; a < 2; ++a) sim->tfull[c][a].init("tmem_full", 1);
      sim->st[c].assign(P.stages, FREE);
      sim->tag[c].assign(P.stages, {-1, -1});
      sim->landed[c].assign(P.stages, 0);
    }
    for (int a = 0; a < 2; ++a) sim->tempty[a].init("tmem_empty", 2 * EPI_WARPS);
    std::vector<std::function<void()>> roles;
    roles.push_back([sim] { sim->producer(0); });
    roles.push_back([sim] { sim->producer(1); });
    roles.push_back([sim] { sim->mma(); });
    for (int c = 0; c < 2; ++c)
      for (int w = 0; w < EPI_WARPS; ++w) roles.push_back([sim, c, w] { sim->epilogue(c, w); });
    std::string where;
    const int rc = sim->sch.run(roles, &where);
    if (P.mode == NORMAL) {
      if (rc != 0) {
        std::printf("DEADLOCK%s\n", where.c_str());
        std::fflush(stdout);
        std::_Exit(1);
      }
      // phase counts: each stage's fills, each accumulator's units
      std::vector<int> per_stage(P.stages, 0);
      int my_units = 0;
      RingPos pos{0, 0};
      for (int u = P.pair; u < P.units; u += P.npairs) {
        int tpos, s, kb0, kb1;
        gf16::decode_unit(u, P.split_k, &tpos, &s);
        gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
        ++my_units;
        for (int kb = kb0; kb < kb1; ++kb) {
          per_stage[pos.stage] += 1;
          gf16::ring_advance(pos, (uint32_t)P.stages);
        }
      }
      for (int s = 0; s < P.stages; ++s) {
        if (sim->full[s].completions != per_stage[s]) fail("full phase count mismatch");
        for (int c = 0; c < 2; ++c)
          if (sim->empty[c][s].completions != per_stage[s]) fail("empty phase count mismatch");
      }
      const int a0 = (my_units + 1) / 2, a1 = my_units / 2;
      for (int c = 0; c < 2; ++c)
        if (sim->tfull[c][0].completions != a0 || sim->tfull[c][1].completions != a1)
          fail("tmem_full phase count mismatch");
      if (sim->tempty[0].completions != a0 || sim->tempty[1].completions != a1)
        fail("tmem_empty phase count mismatch");
      if (sim->drain() != 0) fail("drain after a normal run is not a no-op");
      delete sim;
      continue;
    }
    // abort modes: a deadlock is what the kernel's bounded waits escape
    if (rc != 1) {
      // a stop beyond this pair's work, or a fault unit of another pair
      if (sim->fault_fill >= 0) fail("fault injected but the replay finished");
      delete sim;
      continue;
    }
    ++deadlocks;
    const int left = sim->drain();
    if (P.mode == FAULT && left != 1) fail("the faulted fill should stay incomplete");
    if (P.mode != FAULT && left != 0) fail("drain left phases incomplete");
    // threads of this deadlocked replay are detached; start the next seed
  }
  std::printf("OK %d deadlocks=%d\n", seeds, deadlocks);
  std::fflush(stdout);
  std::_Exit(0);
}
