// Host replay of the single-CTA GEMM kernel's barrier protocol, for testing
// the pipeline's schedule without a GPU.
//
// The three roles of one CTA (TMA producer, MMA issuer, four epilogue
// warps) run one at a time under a seeded scheduler, interleaved with copy
// completions (any order) and tensor-core completions (issue order).  The
// role loops use the same index and parity helpers as the device code
// (schedule.h); the mbarrier follows the "mbarrier State and Operations"
// page (mbar_model.h).
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

#include "mbar_model.h"
#include "schedule.h"

using gf16::RingPos;
using mbmodel::fail;
using mbmodel::MBar;

namespace {

constexpr uint32_t TX_A = 16384, TX_B = 8192, N_B_COPIES = 4;
constexpr uint32_t STAGE_TX = TX_A + N_B_COPIES * TX_B;
constexpr int EPI_WARPS = 4;
constexpr int NROLES = 2 + EPI_WARPS;  // 0 producer, 1 mma, 2.. epilogue warps

struct Params {
  int stages, units, grid, cta, split_k, kblocks, fault_unit;
};

enum StageState { FREE, FILLING, FULL, READING };

struct Sim {
  Params P;
  mbmodel::Scheduler sch{NROLES};
  std::vector<MBar> full, empty;
  MBar tfull[2], tempty[2];
  std::vector<StageState> st;
  std::vector<std::pair<int, int>> tag;  // (unit, kb) loaded into the stage
  std::vector<int> landed;
  int acc_unit[2] = {-1, -1}, acc_kbs[2] = {0, 0}, acc_reads[2] = {0, 0};
  bool acc_ready[2] = {false, false};

  void producer() {
    const int r = 0;
    sch.start(r);
    RingPos pos{0, 0};
    for (int u = P.cta; u < P.units; u += P.grid) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t sg = pos.stage, par = gf16::producer_wait_parity(pos);
        sch.wait_until(r, [&] { return empty[sg].try_wait(par); });
        if (st[sg] != FREE) fail("producer refills a stage that is still in use");
        full[sg].arrive_expect_tx(r, STAGE_TX);
        st[sg] = FILLING;
        tag[sg] = {u, kb};
        landed[sg] = 0;
        if (!(u == P.fault_unit && kb == kb0)) {
          auto land = [this, sg](uint32_t bytes) {
            return mbmodel::Scheduler::Copy{[this, sg, bytes] {
              landed[sg] += 1;
              if (landed[sg] == 1 + (int)N_B_COPIES) st[sg] = FULL;
              full[sg].complete_tx(bytes);
            }};
          };
          sch.copies.push_back(land(TX_A));
          for (uint32_t j = 0; j < N_B_COPIES; ++j) sch.copies.push_back(land(TX_B));
        }
        gf16::ring_advance(pos, (uint32_t)P.stages);
        sch.role_yield(r);
      }
    }
    sch.finish(r);
  }

  void mma() {
    const int r = 1;
    sch.start(r);
    RingPos pos{0, 0};
    uint32_t local = 0;
    for (int u = P.cta; u < P.units; u += P.grid) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      sch.wait_until(r, [&] { return tempty[acc].try_wait(aph ^ 1u); });
      if (acc_unit[acc] != -1 && acc_reads[acc] != EPI_WARPS)
        fail("MMA overwrites an accumulator the epilogue has not read");
      acc_unit[acc] = u;
      acc_kbs[acc] = 0;
      acc_reads[acc] = 0;
      acc_ready[acc] = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t sg = pos.stage, par = gf16::consumer_wait_parity(pos);
        sch.wait_until(r, [&] { return full[sg].try_wait(par); });
        if (st[sg] != FULL) fail("MMA reads a stage whose copies have not all landed");
        if (tag[sg] != std::make_pair(u, kb)) fail("MMA reads the wrong k-block");
        st[sg] = READING;
        const int a = (int)acc;
        sch.tc_queue.push_back([this, a] { acc_kbs[a] += 1; });  // the MMAs
        sch.tc_queue.push_back([this, sg] {                        // commit -> empty
          st[sg] = FREE;
          empty[sg].arrive(-1);
        });
        gf16::ring_advance(pos, (uint32_t)P.stages);
        sch.role_yield(r);
      }
      const int a = (int)acc, want = kb1 - kb0;
      sch.tc_queue.push_back([this, a, want] {  // commit -> tmem_full
        if (acc_kbs[a] != want) fail("accumulator handed over before its MMAs finished");
        acc_ready[a] = true;
        tfull[a].arrive(-1);
      });
      ++local;
      sch.role_yield(r);
    }
    sch.finish(r);
  }

  void epilogue(int w) {
    const int r = 2 + w;
    sch.start(r);
    uint32_t local = 0;
    for (int u = P.cta; u < P.units; u += P.grid) {
      int tpos, s, kb0, kb1;
      gf16::decode_unit(u, P.split_k, &tpos, &s);
      gf16::split_range(P.kblocks, P.split_k, s, &kb0, &kb1);
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      sch.wait_until(r, [&] { return tfull[acc].try_wait(aph); });
      if (!acc_ready[acc] || acc_unit[acc] != u || acc_kbs[acc] != kb1 - kb0)
        fail("epilogue reads an accumulator that is not this unit's finished tile");
      sch.role_yield(r);  // the loads and stores take a while
      acc_reads[acc] += 1;
      tempty[acc].arrive(r);
      ++local;
      sch.role_yield(r);
    }
    sch.finish(r);
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
  const bool fault_here = P.fault_unit >= P.cta && P.fault_unit < P.units &&
                          (P.fault_unit - P.cta) % P.grid == 0;
  for (int seed = 0; seed < seeds; ++seed) {
    Sim* sim = new Sim();  // leaked on deadlock (threads detached)
    sim->P = P;
    sim->sch.seed(0x9E3779B97F4A7C15ull * (uint64_t)(seed + 1));
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
    std::vector<std::function<void()>> roles;
    roles.push_back([sim] { sim->producer(); });
    roles.push_back([sim] { sim->mma(); });
    for (int w = 0; w < EPI_WARPS; ++w) roles.push_back([sim, w] { sim->epilogue(w); });
    std::string where;
    const int rc = sim->sch.run(roles, &where);
    if (fault_here) {
      if (rc != 1) fail("fault injected but the replay finished");
      if (!sim->sch.blocked(1)) fail("fault injected but the MMA role is not blocked");
      std::printf("DEADLOCK-AS-EXPECTED%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(0);
    }
    if (rc != 0) {
      std::printf("DEADLOCK%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(1);
    }
    std::vector<int> per_stage(P.stages, 0);
    int my_units = 0;
    RingPos pos{0, 0};
    for (int u = P.cta; u < P.units; u += P.grid) {
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
      if (sim->full[s].completions != per_stage[s]) fail("full barrier phase count mismatch");
      if (sim->empty[s].completions != per_stage[s]) fail("empty barrier phase count mismatch");
    }
    const int a0 = (my_units + 1) / 2, a1 = my_units / 2;
    if (sim->tfull[0].completions != a0 || sim->tfull[1].completions != a1 ||
        sim->tempty[0].completions != a0 || sim->tempty[1].completions != a1)
      fail("accumulator barrier phase count mismatch");
    if (!sim->sch.copies.empty() || !sim->sch.tc_queue.empty()) fail("work left in flight");
    delete sim;
  }
  std::printf("OK %d\n", seeds);
  return 0;
}
