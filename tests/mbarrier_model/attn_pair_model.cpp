// Host replay of the CTA-pair attention kernel's barrier protocol, for one
// cluster that works through several units (a unit: 256 query rows and one
// range of their key blocks; with SPLITS ranges per item of NKV blocks, the
// ranges have ceil(NKV / SPLITS') blocks and the last one the rest, as in the
// kernel).  "Item" below means unit.
//
// Roles: 0 leader producer, 1 peer producer, 2 MMA issuer (leader), 3..10
// the softmax warps (CTA c, warp w: 3 + 4c + w), 11..18 the epilogue warps
// (11 + 4c + e).  Barriers as in the kernel:
//   q_full, full[s]   leader: one arrive.expect_tx (both CTAs' bytes) by the
//                     leader producer, completed by each CTA's copy;
//   q_empty[c]        both CTAs: the MMA's multicast commit after an item's
//                     last S = Q K^T;
//   empty[c][s]       both CTAs: the MMA's multicast commit;
//   s_full[c]         both CTAs: multicast commit after S = Q K^T of a block
//                     (one S buffer);
//   s_free, p_full[b], o_free
//                     leader: four arrive.expect_tx(16) by the leader's
//                     softmax (epilogue) warps, 16 bytes from each peer
//                     warp's signalling copy (which lands at any later time);
//                     s_free once all eight softmax warps hold S in registers
//                     (not sent after the cluster's last block), p_full[b]
//                     once they wrote their rows of P into P buffer b, o_free
//                     once all eight epilogue warps read O (not sent after
//                     the last item);
//   o_done[c][b]      both CTAs: multicast commit after O += P V from P
//                     buffer b;
//   l_ready[c], l_free[c]
//                     per CTA: four arrivals by the softmax (epilogue) warps
//                     handing an item's row sums over (l_free not after the
//                     last item).
// Copies land in any order; tensor-core work and commits complete in issue
// order.  Checked on every interleaving:
//   * no deadlock;
//   * every wait for phase k of a barrier returns with exactly k + 1 phases
//     completed (a parity wait can neither run ahead of the barrier nor be
//     satisfied by a later phase);
//   * a ring slot is refilled only after the MMAs reading it completed, and
//     the MMA reads the tile (item, K_j or V_j) the schedule says, fully
//     landed, in both CTAs; Q of an item is overwritten only after the last
//     S = Q K^T of the item before ran, and S reads the Q of its own item,
//     fully landed;
//   * S = Q K^T overwrites the S buffer only after all eight softmax warps
//     read the block before; the softmax reads S only after it was written;
//   * a softmax warp overwrites a P buffer only after O += P V that read it
//     completed; O += P V of a block runs only after all eight warps wrote
//     their rows of its P;
//   * the compensation (O *= alpha, done by some warps in some blocks) runs
//     only after O += P V of the item's previous block completed and before
//     that of the current block;
//   * the epilogue reads O of an item only after its last O += P V and
//     before the next item's first one, and the row sums of that item;
//     the softmax overwrites the row sums only after the epilogue read them;
//   * no role arrives twice on a phase; phase counts balance at the end.
// With a fault (the leader issues no copy for its first ring fill) the
// replay must stop with the MMA role blocked on that fill.
//
// Usage: attn_pair_model RING NKV ITEMS SPLITS SEEDS [fault]
// Prints "OK <n>" or "FAIL <reason>" / "DEADLOCK <where>".

#include "mbar_model.h"
#include "schedule.h"

using gf16::RingPos;
using mbmodel::fail;
using mbmodel::MBar;

namespace {

constexpr uint32_t Q_BYTES = 65536, SLOT_BYTES = 32768, SIG = 16;
constexpr int WARPS = 4;                // softmax (and epilogue) warps per CTA
constexpr int MMA_ROLE = 2;
constexpr int NROLES = 3 + 4 * WARPS;

enum SlotState { FREE, FILLING, FULL, READING };

struct Tile {
  int item;
  bool is_k;
  int j;
  bool operator!=(const Tile& o) const { return item != o.item || is_k != o.is_k || j != o.j; }
};

struct Sim {
  int ring = 4, nkv = 1, items = 1;
  std::vector<int> nbs, g0s;  // per unit: key blocks, global index of the first
  bool fault = false;
  uint64_t seed = 1;
  mbmodel::Scheduler sch{NROLES};
  MBar q_full, q_empty[2], s_full[2], s_free, p_full[2], o_free, l_ready[2], l_free[2];
  std::vector<MBar> full;
  std::vector<MBar> empty[2];
  MBar o_done[2][2];
  std::vector<SlotState> st[2];
  std::vector<Tile> tag[2];
  // Q buffer (per CTA): item held, copy landed; the item whose last S ran.
  int q_item[2] = {-1, -1};
  bool q_landed[2] = {false, false};
  int last_s_item_done = -1;
  // S buffer (per CTA): global block held, warps that read it.  P buffers
  // (per CTA): global block written, warps done, last global block whose
  // P V finished reading it.
  int s_block[2] = {-1, -1}, s_reads[2] = {0, 0};
  int p_block[2][2] = {{-1, -1}, {-1, -1}}, p_writes[2][2] = {{0, 0}, {0, 0}};
  int p_read_done[2][2] = {{-1, -1}, {-1, -1}};
  // O: item and block of the last O += P V that completed / began.
  int o_done_item = -1, o_done_j = -1, pv_started_item = -1, pv_started_j = -1;
  int o_read_item[2][WARPS] = {{-1, -1, -1, -1}, {-1, -1, -1, -1}};  // epilogue reads of O
  int l_item[2][WARPS] = {{-1, -1, -1, -1}, {-1, -1, -1, -1}};       // row sums written (softmax)
  int l_read_item[2][WARPS] = {{-1, -1, -1, -1}, {-1, -1, -1, -1}};  // row sums read (epilogue)

  static bool rescale(uint64_t seed, int g, int warp) {
    const uint64_t h = (seed * 0x9E3779B97F4A7C15ull) ^ ((uint64_t)g * 0xBF58476D1CE4E5B9ull) ^
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

  // A leader barrier counted in warps: the leader's warp arrives expecting
  // 16 bytes, the peer's sends them.
  void signal(int r, int cta, MBar& bar) {
    if (cta == 0)
      bar.arrive_expect_tx(r, SIG);
    else
      sch.copies.push_back({[&bar] { bar.complete_tx(SIG); }});
  }

  // The consumption order of the ring: per item K_0, then per block j:
  // K_{j+1}, V_j.
  std::vector<Tile> order() const {
    std::vector<Tile> o;
    for (int k = 0; k < items; ++k) {
      o.push_back({k, true, 0});
      for (int j = 0; j < nbs[k]; ++j) {
        if (j + 1 < nbs[k]) o.push_back({k, true, j + 1});
        o.push_back({k, false, j});
      }
    }
    return o;
  }

  void producer(int cta) {
    const int r = cta;
    sch.start(r);
    RingPos pos{0, 0};
    int fill = 0;
    const std::vector<Tile> ord = order();
    size_t next = 0;
    for (int k = 0; k < items; ++k) {
      if (k > 0) {
        wait_phase(r, q_empty[cta], k - 1);
        if (last_s_item_done != k - 1) fail("Q overwritten before the last S of its item ran");
      }
      if (cta == 0) q_full.arrive_expect_tx(r, 2 * Q_BYTES);
      q_item[cta] = k;
      q_landed[cta] = false;
      sch.copies.push_back({[this, cta] {
        q_landed[cta] = true;
        q_full.complete_tx(Q_BYTES);
      }});
      sch.role_yield(r);
      for (; next < ord.size() && ord[next].item == k; ++next) {
        const Tile t = ord[next];
        const uint32_t s = pos.stage;
        const int use = fill / ring;  // this slot's use index
        if (use > 0) wait_phase(r, empty[cta][s], use - 1);
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
    }
    sch.finish(r);
  }

  void mma() {
    const int r = MMA_ROLE;
    sch.start(r);
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
    // S of global block gs (item k, block j) into the S buffer.
    auto issue_qk = [&](int gs, int k, int j) {
#ifndef PLANT_SKIP_S_FREE_WAIT  // the PLANT_* switches are set only by tests planting a mistake
      if (gs > 0) wait_phase(r, s_free, gs - 1);
#endif
      const uint32_t s = consume({k, true, j});
      const bool last = j == nbs[k] - 1;
      sch.tc_queue.push_back([this, gs, k, last] {  // S = Q K^T executes
        for (int c = 0; c < 2; ++c) {
          if (q_item[c] != k || !q_landed[c]) fail("S = Q K^T reads a Q tile not of its item");
          if (s_block[c] >= 0 && s_reads[c] != WARPS)
            fail("S = Q K^T overwrites the S buffer before the softmax read it");
          s_block[c] = gs;
          s_reads[c] = 0;
        }
        if (last) last_s_item_done = k;
      });
      release(s);
      sch.tc_queue.push_back([this, last] {
        for (int c = 0; c < 2; ++c) {
          s_full[c].arrive(-1);
          if (last) q_empty[c].arrive(-1);
        }
      });
    };
    for (int k = 0; k < items; ++k) {
      const int g0 = g0s[k], nb = nbs[k];
      wait_phase(r, q_full, k);
      issue_qk(g0, k, 0);
      for (int j = 0; j < nb; ++j) {
        const int g = g0 + j;
        if (j + 1 < nb) issue_qk(g + 1, k, j + 1);
        const int pb = g & 1;
        wait_phase(r, p_full[pb], g >> 1);
        const uint32_t s = consume({k, false, j});
#ifndef PLANT_SKIP_O_FREE_WAIT
        if (j == 0 && k > 0) wait_phase(r, o_free, k - 1);
#endif
        sch.tc_queue.push_back([this, g, k, j, pb] {  // O += P V begins
          for (int c = 0; c < 2; ++c) {
            if (p_block[c][pb] != g || p_writes[c][pb] != WARPS)
              fail("O += P V reads a P buffer not fully written for its block");
            if (j == 0)
              for (int e = 0; e < WARPS; ++e)
                if (k > 0 && o_read_item[c][e] != k - 1)
                  fail("O += P V overwrites O before the epilogue read it");
          }
          if (j == 0 ? (o_done_item != k - 1 || (k > 0 && o_done_j != nbs[k - 1] - 1))
                     : (o_done_item != k || o_done_j != j - 1))
            fail("O += P V out of order");
          pv_started_item = k;
          pv_started_j = j;
        });
        sch.tc_queue.push_back([this, k, j, pb, g] {  // ... and ends
          o_done_item = k;
          o_done_j = j;
          for (int c = 0; c < 2; ++c) p_read_done[c][pb] = g;
        });
        release(s);
        sch.tc_queue.push_back([this, pb] {
          for (int c = 0; c < 2; ++c) o_done[c][pb].arrive(-1);
        });
        sch.role_yield(r);
      }
    }
    sch.finish(r);
  }

  void softmax(int cta, int w) {
    const int r = 3 + cta * WARPS + w;
    sch.start(r);
    for (int k = 0; k < items; ++k) {
      for (int j = 0; j < nbs[k]; ++j) {
        const int g = g0s[k] + j, pb = g & 1;
        wait_phase(r, s_full[cta], g);
        if (s_block[cta] != g) fail("softmax reads an S buffer that does not hold its block");
        s_reads[cta] += 1;
        if (j + 1 < nbs[k] || k + 1 < items) signal(r, cta, s_free);
        sch.role_yield(r);  // exp2, packing
        if (g >= 2) wait_phase(r, o_done[cta][pb], (g - 2) >> 1);
        if (p_block[cta][pb] != g) {  // the first warp to write this block's P here
          if (p_block[cta][pb] >= 0 && p_read_done[cta][pb] != p_block[cta][pb])
            fail("softmax overwrites a P buffer that O += P V still reads");
          p_block[cta][pb] = g;
          p_writes[cta][pb] = 0;
        } else if (p_read_done[cta][pb] == g) {
          fail("softmax writes P rows after O += P V of their block ran");
        }
        p_writes[cta][pb] += 1;
        if (j > 0 && rescale(seed, g, cta * WARPS + w)) {
          wait_phase(r, o_done[cta][(g - 1) & 1], (g - 1) >> 1);
          if (o_done_item != k || o_done_j != j - 1 ||
              (pv_started_item == k && pv_started_j >= j))
            fail("compensation while O += P V is not at the item's previous block");
          sch.role_yield(r);  // O *= alpha
        }
        signal(r, cta, p_full[pb]);
        sch.role_yield(r);  // the window: the sum update
      }
      // Row sums to the epilogue warps, once they took the previous ones.
      if (k > 0) {
#ifndef PLANT_SKIP_L_FREE_WAIT
        wait_phase(r, l_free[cta], k - 1);
#endif
        for (int e = 0; e < WARPS; ++e)
          if (l_read_item[cta][e] != k - 1) fail("row sums overwritten before the epilogue read them");
      }
      l_item[cta][w] = k;
      l_ready[cta].arrive(r);
    }
    sch.finish(r);
  }

  void epilogue(int cta, int e) {
    const int r = 3 + 2 * WARPS + cta * WARPS + e;
    sch.start(r);
    for (int k = 0; k < items; ++k) {
      const int g_last = g0s[k] + nbs[k] - 1;
      wait_phase(r, l_ready[cta], k);
      for (int w = 0; w < WARPS; ++w)
        if (l_item[cta][w] != k) fail("epilogue reads row sums not of its item");
      l_read_item[cta][e] = k;
      if (k + 1 < items) l_free[cta].arrive(r);
      wait_phase(r, o_done[cta][g_last & 1], g_last >> 1);
      if (o_done_item != k || o_done_j != nbs[k] - 1 || pv_started_item != k)
        fail("epilogue reads O that is not the finished O of its item");
      o_read_item[cta][e] = k;
      if (k + 1 < items) signal(r, cta, o_free);
      sch.role_yield(r);  // scale, stage, store
    }
    sch.finish(r);
  }
};

}  // namespace

int main(int argc, char** argv) {
  if (argc < 6) {
    std::fprintf(stderr, "usage: attn_pair_model RING NKV ITEMS SPLITS SEEDS [fault]\n");
    return 2;
  }
  const int ring = std::atoi(argv[1]), nkv = std::atoi(argv[2]), n_items = std::atoi(argv[3]);
  const int splits_req = std::atoi(argv[4]), seeds = std::atoi(argv[5]);
  const bool fault = argc > 6 && std::string(argv[6]) == "fault";
  // Key ranges as the kernel's host code makes them: bps blocks each, none empty.
  int splits = splits_req < 1 ? 1 : (splits_req > nkv ? nkv : splits_req);
  const int bps = (nkv + splits - 1) / splits;
  splits = (nkv + bps - 1) / bps;
  std::vector<int> nbs, g0s;
  for (int it = 0, g = 0; it < n_items; ++it)
    for (int sp = 0; sp < splits; ++sp) {
      const int nb = nkv - sp * bps < bps ? nkv - sp * bps : bps;
      nbs.push_back(nb);
      g0s.push_back(g);
      g += nb;
    }
  const int items = (int)nbs.size();  // units
  for (int seed = 0; seed < seeds; ++seed) {
    Sim* sim = new Sim();  // leaked on deadlock (threads detached)
    sim->ring = ring;
    sim->nkv = nkv;
    sim->items = items;
    sim->nbs = nbs;
    sim->g0s = g0s;
    sim->fault = fault;
    sim->seed = (uint64_t)seed + 1;
    sim->sch.seed(0x9E3779B97F4A7C15ull * (uint64_t)(seed + 1));
    sim->q_full.init("q_full", 1, true);
    sim->s_free.init("s_free", WARPS, true);
    sim->o_free.init("o_free", WARPS, true);
    sim->full.resize(ring);
    for (int c = 0; c < 2; ++c) {
      const std::string cs = "[" + std::to_string(c) + "]";
      sim->q_empty[c].init("q_empty" + cs, 1);
      sim->s_full[c].init("s_full" + cs, 1);
      sim->l_ready[c].init("l_ready" + cs, WARPS);
      sim->l_free[c].init("l_free" + cs, WARPS);
      sim->empty[c].resize(ring);
      sim->st[c].assign(ring, FREE);
      sim->tag[c].assign(ring, {-1, false, -1});
    }
    for (int s = 0; s < ring; ++s) {
      sim->full[s].init("full[" + std::to_string(s) + "]", 1, true);
      for (int c = 0; c < 2; ++c)
        sim->empty[c][s].init("empty[" + std::to_string(c) + "][" + std::to_string(s) + "]", 1);
    }
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
    for (int c = 0; c < 2; ++c)
      for (int e = 0; e < WARPS; ++e) roles.push_back([sim, c, e] { sim->epilogue(c, e); });
    std::string where;
    const int rc = sim->sch.run(roles, &where);
    if (fault) {
      if (rc != 1) fail("fault injected but the replay finished");
      if (!sim->sch.blocked(MMA_ROLE)) fail("fault injected but the MMA role is not blocked");
      std::printf("DEADLOCK-AS-EXPECTED%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(0);
    }
    if (rc != 0) {
      std::printf("DEADLOCK%s\n", where.c_str());
      std::fflush(stdout);
      std::_Exit(1);
    }
    int blocks = 0;
    for (int nb : nbs) blocks += nb;
    const int fills = 2 * blocks;
    for (int s = 0; s < ring; ++s) {
      const int uses = fills / ring + (s < fills % ring ? 1 : 0);
      if (sim->full[s].completions != uses) fail("full phase count mismatch");
      for (int c = 0; c < 2; ++c)
        if (sim->empty[c][s].completions != uses) fail("empty phase count mismatch");
    }
    for (int b = 0; b < 2; ++b) {
      const int uses = blocks / 2 + (b < blocks % 2 ? 1 : 0);
      if (sim->p_full[b].completions != uses) fail("p_full phase count mismatch");
      for (int c = 0; c < 2; ++c)
        if (sim->o_done[c][b].completions != uses) fail("o_done phase count mismatch");
    }
    for (int c = 0; c < 2; ++c) {
      if (sim->s_full[c].completions != blocks) fail("s_full phase count mismatch");
      if (sim->q_empty[c].completions != items) fail("q_empty phase count mismatch");
      if (sim->l_ready[c].completions != items || sim->l_free[c].completions != items - 1)
        fail("l_ready / l_free phase count mismatch");
    }
    if (sim->s_free.completions != blocks - 1) fail("s_free phase count mismatch");
    if (sim->o_free.completions != items - 1) fail("o_free phase count mismatch");
    if (sim->q_full.completions != items) fail("q_full phase count mismatch");
    if (!sim->sch.copies.empty() || !sim->sch.tc_queue.empty()) fail("work left in flight");
    delete sim;
  }
  std::printf("OK %d\n", seeds);
  return 0;
}
