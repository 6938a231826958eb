// Host replay of the CTA-pair attention kernel's barrier protocol.
//
// Roles: 0 leader producer, 1 peer producer, 2 MMA issuer (leader), 3..6 the
// leader's softmax warps, 7..10 the peer's.  Barriers as in the kernel:
//   q_full, full[s]   leader: one arrive.expect_tx (both CTAs' bytes) by the
//                     leader producer, completed by each CTA's copy;
//   empty[c][s]       both CTAs: the MMA's multicast commit;
//   s_full[c]         both CTAs: multicast commit after S = Q K^T of a block
//                     (one S buffer);
//   s_free, p_full[b] leader: four arrive.expect_tx(16) by the leader's
//                     softmax warps, 16 bytes from each peer warp's
//                     signalling copy (which lands at any later time);
//                     s_free once all eight warps hold S_j in registers
//                     (not sent for the last block), p_full[b] once they
//                     wrote their rows of P_j into P buffer b;
//   o_done[c][b]      both CTAs: multicast commit after O += P V from P
//                     buffer b.
// Copies land in any order; tensor-core work and commits complete in issue
// order.  Checked on every interleaving:
//   * no deadlock;
//   * every wait for phase k of a barrier returns with exactly k + 1 phases
//     completed (a parity wait can neither run ahead of the barrier nor be
//     satisfied by a later phase);
//   * a ring slot is refilled only after the MMAs reading it completed, and
//     the MMA reads the tile (K_j or V_j) the schedule says, fully landed,
//     in both CTAs;
//   * S = Q K^T of block j overwrites the S buffer only after all eight
//     softmax warps read block j-1 from it; the softmax reads S_j only
//     after it was written;
//   * a softmax warp overwrites a P buffer only after O += P V that read it
//     completed; O += P V of block j runs only after all eight warps wrote
//     their rows of P_j;
//   * the compensation (O *= alpha, done by some warps in some blocks) runs
//     only after O += P V of block j-1 completed and before that of block j;
//     the epilogue reads O only after the last O += P V;
//   * no role arrives twice on a phase; phase counts balance at the end.
// With a fault (the leader issues no copy for its first ring fill) the
// replay must stop with the MMA role blocked on that fill.
//
// Usage: attn_pair_model RING NKV SEEDS [fault]
// Prints "OK <n>" or "FAIL <reason>" / "DEADLOCK <where>".

#include "mbar_model.h"
#include "schedule.h"

using gf16::RingPos;
using mbmodel::fail;
using mbmodel::MBar;

namespace {

constexpr uint32_t Q_BYTES = 65536, SLOT_BYTES = 32768, SIG = 16;
constexpr int WARPS = 4;                // softmax warps per CTA
constexpr int NROLES = 3 + 2 * WARPS;

enum SlotState { FREE, FILLING, FULL, READING };

struct Tile {
  bool is_k;
  int j;
  bool operator!=(const Tile& o) const { return is_k != o.is_k || j != o.j; }
};

struct Sim {
  int ring = 3, nkv = 1;
  bool fault = false;
  uint64_t seed = 1;
  mbmodel::Scheduler sch{NROLES};
  MBar q_full;
  std::vector<MBar> full;
  std::vector<MBar> empty[2];
  MBar s_full[2], s_free, p_full[2], o_done[2][2];
  std::vector<SlotState> st[2];
  std::vector<Tile> tag[2];
  // S buffer (per CTA): block held, warps that read it; P buffers (per CTA):
  // block written, warps done; O: last block accumulated, P V in flight.
  int s_block[2] = {-1, -1}, s_reads[2] = {0, 0};
  int p_block[2][2] = {{-1, -1}, {-1, -1}}, p_writes[2][2] = {{0, 0}, {0, 0}};
  int p_read_done[2][2] = {{-1, -1}, {-1, -1}};  // last block whose P V finished, per buffer
  int o_done_block = -1;                         // last block with O += P V completed
  int pv_started = -1;                           // last block whose P V began executing

  static bool rescale(uint64_t seed, int j, int warp) {
    const uint64_t h = (seed * 0x9E3779B97F4A7C15ull) ^ ((uint64_t)j * 0xBF58476D1CE4E5B9ull) ^
                       ((uint64_t)warp * 0x94D049BB133111EBull);
    return ((h >> 29) % 3) == 0;
  }

  // Wait for phase k of `bar` to complete; it must then be exactly k + 1.
  void wait_phase(int r, MBar& bar, int k) {
    sch.wait_until(r, [&] { return bar.try_wait((uint32_t)k & 1u); });
    if (bar.completions != k + 1)
      fail("parity wait on " + bar.name + " for phase " + std::to_string(k) + " returned with " +
           std::to_string(bar.completions) + " phases completed");
  }

  // The consumption order of the ring: K_0, then per block j: K_{j+1}, V_j.
  std::vector<Tile> order() const {
    std::vector<Tile> o{{true, 0}};
    for (int j = 0; j < nkv; ++j) {
      if (j + 1 < nkv) o.push_back({true, j + 1});
      o.push_back({false, j});
    }
    return o;
  }

  void producer(int cta) {
    const int r = cta;
    sch.start(r);
    if (cta == 0) q_full.arrive_expect_tx(r, 2 * Q_BYTES);
    sch.copies.push_back({[this] { q_full.complete_tx(Q_BYTES); }});
    RingPos pos{0, 0};
    int fill = 0;
    for (const Tile& t : order()) {
      const uint32_t s = pos.stage;
      const int k = (int)(fill / ring);  // this slot's use index
      if (k > 0) wait_phase(r, empty[cta][s], k - 1);
      if (st[cta][s] != FREE) fail("producer refills a slot still in use");
      if (cta == 0) full[s].arrive_expect_tx(r, 2 * SLOT_BYTES);
      st[cta][s] = FILLING;
      tag[cta][s] = t;
      if (!(fault && fill == 0 && cta == 0)) {
        sch.copies.push_back({[this, cta, s] {
          st[cta][s] = FULL;
          full[s].complete_tx(SLOT_BYTES);
        }});
      }
      ++fill;
      gf16::ring_advance(pos, (uint32_t)ring);
      sch.role_yield(r);
    }
    sch.finish(r);
  }

  void mma() {
    const int r = 2;
    sch.start(r);
    wait_phase(r, q_full, 0);
    RingPos pos{0, 0};
    int fill = 0;
    const std::vector<Tile> ord = order();
    auto consume = [&](const Tile& want) {
      const uint32_t s = pos.stage;
      wait_phase(r, full[s], fill / ring);
      for (int c = 0; c < 2; ++c) {
        if (st[c][s] != FULL) fail("MMA reads a slot whose copy has not landed");
        if (tag[c][s] != want) fail("MMA reads the wrong tile");
        st[c][s] = READING;
      }
      if (ord[fill] != want) fail("consumption order differs from the fill order");
      ++fill;
      gf16::ring_advance(pos, (uint32_t)ring);
      return s;
    };
    auto release = [&](uint32_t s) {
      sch.tc_queue.push_back([this, s] {
        for (int c = 0; c < 2; ++c) {
          st[c][s] = FREE;
          empty[c][s].arrive(-1);
        }
      });
    };
    auto issue_qk = [&](int j) {
      const uint32_t s = consume({true, j});
      sch.tc_queue.push_back([this, j] {  // S = Q K^T executes: writes the S buffer
        for (int c = 0; c < 2; ++c) {
          if (s_block[c] >= 0 && s_reads[c] != WARPS)
            fail("S = Q K^T overwrites the S buffer before the softmax read it");
          s_block[c] = j;
          s_reads[c] = 0;
        }
      });
      release(s);
      sch.tc_queue.push_back([this] {
        for (int c = 0; c < 2; ++c) s_full[c].arrive(-1);
      });
    };
    issue_qk(0);
    for (int j = 0; j < nkv; ++j) {
      if (j + 1 < nkv) {
#ifndef PLANT_SKIP_S_FREE_WAIT  // defined only by the test that plants this mistake
        wait_phase(r, s_free, j);
#endif
        issue_qk(j + 1);
      }
      const int pb = j & 1;
      wait_phase(r, p_full[pb], j >> 1);
      const uint32_t s = consume({false, j});
      sch.tc_queue.push_back([this, j, pb] {  // O += P V begins
        for (int c = 0; c < 2; ++c)
          if (p_block[c][pb] != j || p_writes[c][pb] != WARPS)
            fail("O += P V reads a P buffer not fully written for its block");
        if (o_done_block != j - 1) fail("O += P V out of order");
        pv_started = j;
      });
      sch.tc_queue.push_back([this, j, pb] {  // ... and ends
        o_done_block = j;
        for (int c = 0; c < 2; ++c) p_read_done[c][pb] = j;
      });
      release(s);
      sch.tc_queue.push_back([this, pb] {
        for (int c = 0; c < 2; ++c) o_done[c][pb].arrive(-1);
      });
      sch.role_yield(r);
    }
    sch.finish(r);
  }

  void softmax(int cta, int w) {
    const int r = 3 + cta * WARPS + w;
    sch.start(r);
    for (int j = 0; j < nkv; ++j) {
      const int pb = j & 1;
      wait_phase(r, s_full[cta], j);
      if (s_block[cta] != j) fail("softmax reads an S buffer that does not hold its block");
      s_reads[cta] += 1;
      if (j + 1 < nkv) {
        if (cta == 0)
          s_free.arrive_expect_tx(r, SIG);
        else
          sch.copies.push_back({[this] { s_free.complete_tx(SIG); }});
      }
      sch.role_yield(r);  // exp2, packing
      if (j >= 2) wait_phase(r, o_done[cta][pb], (j - 2) >> 1);
      if (p_block[cta][pb] != j) {  // the first warp to write P_j into this buffer
        if (p_block[cta][pb] >= 0 && p_read_done[cta][pb] != p_block[cta][pb])
          fail("softmax overwrites a P buffer that O += P V still reads");
        p_block[cta][pb] = j;
        p_writes[cta][pb] = 0;
      } else if (p_read_done[cta][pb] == j) {
        fail("softmax writes P rows after O += P V of their block ran");
      }
      p_writes[cta][pb] += 1;
      if (j > 0 && rescale(seed, j, cta * WARPS + w)) {
        wait_phase(r, o_done[cta][(j - 1) & 1], (j - 1) >> 1);
        if (o_done_block != j - 1 || pv_started >= j)
          fail("compensation while O += P V is not at block j-1");
        sch.role_yield(r);  // O *= alpha
      }
      if (cta == 0) {
        p_full[pb].arrive_expect_tx(r, SIG);
      } else {
        sch.copies.push_back({[this, pb] { p_full[pb].complete_tx(SIG); }});
      }
      sch.role_yield(r);  // the window: the sum update
    }
    wait_phase(r, o_done[cta][(nkv - 1) & 1], (nkv - 1) >> 1);
    if (o_done_block != nkv - 1) fail("epilogue reads O before the last O += P V");
    sch.finish(r);
  }
};

}  // namespace

int main(int argc, char** argv) {
  if (argc < 4) {
    std::fprintf(stderr, "usage: attn_pair_model RING NKV SEEDS [fault]\n");
    return 2;
  }
  const int ring = std::atoi(argv[1]), nkv = std::atoi(argv[2]), seeds = std::atoi(argv[3]);
  const bool fault = argc > 4 && std::string(argv[4]) == "fault";
  for (int seed = 0; seed < seeds; ++seed) {
    Sim* sim = new Sim();  // leaked on deadlock (threads detached)
    sim->ring = ring;
    sim->nkv = nkv;
    sim->fault = fault;
    sim->seed = (uint64_t)seed + 1;
    sim->sch.seed(0x9E3779B97F4A7C15ull * (uint64_t)(seed + 1));
    sim->q_full.init("q_full", 1, true);
    sim->full.resize(ring);
    for (int c = 0; c < 2; ++c) {
      sim->empty[c].resize(ring);
      sim->st[c].assign(ring, FREE);
      sim->tag[c].assign(ring, {false, -1});
    }
    for (int s = 0; s < ring; ++s) {
      sim->full[s].init("full[" + std::to_string(s) + "]", 1, true);
      for (int c = 0; c < 2; ++c)
        sim->empty[c][s].init("empty[" + std::to_string(c) + "][" + std::to_string(s) + "]", 1);
    }
    sim->s_free.init("s_free", WARPS, true);
    for (int c = 0; c < 2; ++c) sim->s_full[c].init("s_full[" + std::to_string(c) + "]", 1);
    for (int b = 0; b < 2; ++b) {
      sim->p_full[b].init("p_full[" + std::to_string(b) + "]", WARPS, true);
      for (int c = 0; c < 2; ++c)
        sim->o_done[c][b].init("o_done[" + std::to_string(c) + "][" + std::to_string(b) + "]", 1);
    }
    std::vector<std::function<void()>> roles;
    roles.push_back([sim] { sim->producer(0); });
    roles.push_back([sim] { sim->producer(1); });
    roles.push_back([sim] { sim->mma(); });
    for (int c = 0; c < 2; ++c)
      for (int w = 0; w < WARPS; ++w) roles.push_back([sim, c, w] { sim->softmax(c, w); });
    std::string where;
    const int rc = sim->sch.run(roles, &where);
    if (fault) {
      if (rc != 1) fail("fault injected but the replay finished");
      if (!sim->sch.blocked(2)) fail("fault injected but the MMA role is not blocked");
      std::printf("DEADLOCK-AS-EXPECTED%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(0);
    }
    if (rc != 0) {
      std::printf("DEADLOCK%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(1);
    }
    const int fills = 2 * nkv;
    for (int s = 0; s < ring; ++s) {
      const int uses = fills / ring + (s < fills % ring ? 1 : 0);
      if (sim->full[s].completions != uses) fail("full phase count mismatch");
      for (int c = 0; c < 2; ++c)
        if (sim->empty[c][s].completions != uses) fail("empty phase count mismatch");
    }
    for (int b = 0; b < 2; ++b) {
      const int uses = nkv / 2 + (b < nkv % 2 ? 1 : 0);
      if (sim->p_full[b].completions != uses) fail("p_full phase count mismatch");
      for (int c = 0; c < 2; ++c)
        if (sim->o_done[c][b].completions != uses) fail("o_done phase count mismatch");
    }
    for (int c = 0; c < 2; ++c)
      if (sim->s_full[c].completions != nkv) fail("s_full phase count mismatch");
    if (sim->s_free.completions != nkv - 1) fail("s_free phase count mismatch");
    if (sim->q_full.completions != 1) fail("q_full phase count mismatch");
    if (!sim->sch.copies.empty() || !sim->sch.tc_queue.empty()) fail("work left in flight");
    delete sim;
  }
  std::printf("OK %d\n", seeds);
  return 0;
}
