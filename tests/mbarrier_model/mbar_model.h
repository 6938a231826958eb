// Shared pieces of the host replays of the kernels' barrier protocols: the
// mbarrier itself, modelled exactly as the "mbarrier State and Operations"
// page defines it, and a scheduler that runs role threads one at a time in
// a seeded random order, interleaved with asynchronous completions.
#pragma once

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

namespace mbmodel {

[[noreturn]] inline void fail(const std::string& why) {
  std::printf("FAIL %s\n", why.c_str());
  std::fflush(stdout);
  std::_Exit(1);
}

// init: phase 0, pending = expected = count, tx 0.  arrive: pending - 1.
// arrive.expect_tx: pending - 1, tx + bytes.  complete_tx: tx - bytes.
// A phase completes when pending == 0 and tx == 0: parity flips and pending
// is reloaded.  try_wait(parity) only reads: true once that phase is over.
// The transaction count is signed: bytes may land before they are expected.
struct MBar {
  std::string name;
  uint32_t phase = 0;
  int expected = 0, pending = 0;
  int64_t tx = 0;
  int completions = 0;
  bool allow_negative_tx = false;
  std::set<int> arrivers;  // roles that arrived in the current phase

  void init(const std::string& n, int count, bool negative_tx_ok = false) {
    name = n;
    phase = 0;
    expected = pending = count;
    tx = 0;
    completions = 0;
    allow_negative_tx = negative_tx_ok;
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
    if (tx < 0 && !allow_negative_tx) fail("tx count below zero on " + name);
    if (tx < -(int64_t)((1 << 20) - 1)) fail("tx count out of range on " + name);
    maybe_complete();
  }
  bool try_wait(uint32_t parity) const { return phase != parity; }
};

// Runs NROLES role threads one at a time.  A role gives the token back at
// every yield point and when it blocks in wait_until; the scheduler then
// picks, with its seeded generator, one runnable role, one pending copy
// completion (any order) or the oldest pending completion of a tensor core
// (in issue order; two independent tensor cores, `tc_queue` and
// `tc_queue_b`, for kernels with two MMA issuers).  No runnable choice left
// while roles are unfinished is a deadlock.
class Scheduler {
 public:
  struct Copy {
    std::function<void()> land;
  };

  explicit Scheduler(int nroles) : nroles_(nroles), done_(nroles, false), waiting_(nroles) {}

  void seed(uint64_t s) { rng_.seed(s); }
  std::vector<Copy> copies;
  std::deque<std::function<void()>> tc_queue;
  std::deque<std::function<void()>> tc_queue_b;

  void role_yield(int r) {
    std::unique_lock<std::mutex> lk(mu_);
    turn_ = -1;
    cv_.notify_all();
    cv_.wait(lk, [&] { return turn_ == r; });
  }
  void wait_until(int r, std::function<bool()> pred) {
    while (!pred()) {
      waiting_[r] = pred;
      role_yield(r);
      waiting_[r] = nullptr;
    }
  }
  void start(int r) {
    std::unique_lock<std::mutex> lk(mu_);
    cv_.wait(lk, [&] { return turn_ == r; });
  }
  void finish(int r) {
    std::unique_lock<std::mutex> lk(mu_);
    done_[r] = true;
    turn_ = -1;
    cv_.notify_all();
  }
  bool blocked(int r) const { return !done_[r] && waiting_[r] != nullptr; }

  // 0: all roles finished; 1: deadlock (blocked roles listed in *where).
  int run(const std::vector<std::function<void()>>& roles, std::string* where) {
    std::vector<std::thread> th;
    for (auto& f : roles) th.emplace_back(f);
    int rc = 0;
    while (true) {
      std::unique_lock<std::mutex> lk(mu_);
      cv_.wait(lk, [&] { return turn_ == -1; });
      std::vector<int> choices;  // role r, nroles + i = copy i, -2 / -3 = tensor core a / b
      for (int r = 0; r < nroles_; ++r)
        if (!done_[r] && (!waiting_[r] || waiting_[r]())) choices.push_back(r);
      for (size_t i = 0; i < copies.size(); ++i) choices.push_back(nroles_ + (int)i);
      if (!tc_queue.empty()) choices.push_back(-2);
      if (!tc_queue_b.empty()) choices.push_back(-3);
      bool all_done = true;
      for (int r = 0; r < nroles_; ++r) all_done = all_done && done_[r];
      if (choices.empty()) {
        if (!all_done) {
          rc = 1;
          where->clear();
          for (int r = 0; r < nroles_; ++r)
            if (!done_[r]) *where += " role" + std::to_string(r);
        }
        break;
      }
      const int c = choices[rng_() % choices.size()];
      if (c == -2) {
        auto f = tc_queue.front();
        tc_queue.pop_front();
        f();
      } else if (c == -3) {
        auto f = tc_queue_b.front();
        tc_queue_b.pop_front();
        f();
      } else if (c >= nroles_) {
        auto f = copies[c - nroles_].land;
        copies.erase(copies.begin() + (c - nroles_));
        f();
      } else {
        turn_ = c;
        cv_.notify_all();
      }
    }
    if (rc == 0) {
      for (auto& t : th) t.join();
    } else {
      for (auto& t : th) t.detach();  // blocked roles are abandoned; the process exits
    }
    return rc;
  }

 private:
  int nroles_;
  std::vector<bool> done_;
  std::vector<std::function<bool()>> waiting_;
  std::mt19937_64 rng_;
  std::mutex mu_;
  std::condition_variable cv_;
  int turn_ = -1;
};

}  // namespace mbmodel
