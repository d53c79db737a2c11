// Host planning on a worker thread (pkv_planner_*).
//
// A step's plan depends only on host data (lengths, block tables), while its
// KV append needs none, so a serving loop can queue the input copy and the
// append while the plan is being made.  One thread per planner runs the
// pkv_plan_step_ex calls posted to it; the caller polls for the result.  The
// hand-over is a single atomic state word: the poster writes the job and then
// publishes it (release), the worker reads it after seeing it (acquire), and
// the same pairing carries the result back.  Between jobs the worker polls for
// spin_us, then sleeps on a condition variable, so an idle planner costs no CPU.

#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdint>
#include <mutex>
#include <new>
#include <thread>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

enum : int { kIdle = 0, kPosted = 1, kDone = 2 };

struct Job {
  const int32_t *cu_q_lens, *context_lens, *block_tables;
  int32_t num_seqs, num_q_heads, num_sms, steps, max_blocks_per_seq, prefill_min_q;
  const pkv_pool_desc *desc;
  void *plan;
  int64_t plan_capacity;
  pkv_plan_info *info;
};

}  // namespace

struct pkv_planner {
  std::atomic<int> state{kIdle};
  std::atomic<bool> stop{false};
  Job job{};
  pkv_status result = PKV_OK;
  std::chrono::microseconds spin{0};
  std::mutex mu;
  std::condition_variable cv;
  std::thread worker;

  void run() {
    for (;;) {
      // poll for the next job for `spin`, then sleep until one is posted
      const auto t0 = std::chrono::steady_clock::now();
      while (state.load(std::memory_order_acquire) != kPosted &&
             !stop.load(std::memory_order_acquire)) {
        if (std::chrono::steady_clock::now() - t0 >= spin) {
          std::unique_lock<std::mutex> lk(mu);
          cv.wait(lk, [&] {
            return state.load(std::memory_order_acquire) == kPosted ||
                   stop.load(std::memory_order_acquire);
          });
        }
      }
      if (state.load(std::memory_order_acquire) != kPosted) return;  // stopped with no job
      const Job &j = job;
      result = pkv_plan_step_ex(j.cu_q_lens, j.context_lens, j.num_seqs, j.num_q_heads, j.desc,
                                j.num_sms, j.steps, j.block_tables, j.max_blocks_per_seq,
                                j.prefill_min_q, j.plan, j.plan_capacity, j.info);
      state.store(kDone, std::memory_order_release);
    }
  }
};

extern "C" pkv_status pkv_planner_create(int32_t spin_us, pkv_planner **out) {
  if (!out) return PKV_ERR_NULL;
  *out = nullptr;
  if (spin_us > 1000000) return PKV_ERR_RANGE;
  pkv_planner *p = new (std::nothrow) pkv_planner;
  if (!p) return PKV_ERR_HOST_MEMORY;
  p->spin = std::chrono::microseconds(spin_us > 0 ? spin_us : 0);
  try {
    p->worker = std::thread([p] { p->run(); });
  } catch (...) {
    delete p;
    return PKV_ERR_HOST_MEMORY;
  }
  *out = p;
  return PKV_OK;
}

extern "C" void pkv_planner_destroy(pkv_planner *p) {
  if (!p) return;
  {
    std::lock_guard<std::mutex> lk(p->mu);
    p->stop.store(true, std::memory_order_release);
  }
  p->cv.notify_one();
  if (p->worker.joinable()) p->worker.join();
  delete p;
}

extern "C" pkv_status pkv_planner_post(pkv_planner *p, const int32_t *cu_q_lens,
                                       const int32_t *context_lens, int32_t num_seqs,
                                       int32_t num_q_heads, const pkv_pool_desc *desc,
                                       int32_t num_sms, int32_t steps,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       int32_t prefill_min_q, void *plan, int64_t plan_capacity,
                                       pkv_plan_info *info) {
  if (!p) return PKV_ERR_NULL;
  if (p->state.load(std::memory_order_acquire) != kIdle) return PKV_ERR_STATE;
  if (num_sms <= 0) {
    // the caller's current device, not the worker thread's
    num_sms = pkv::device_sm_count();
    if (num_sms <= 0) return PKV_ERR_CUDA;
  }
  p->job = Job{cu_q_lens, context_lens, block_tables, num_seqs, num_q_heads, num_sms, steps,
               max_blocks_per_seq, prefill_min_q, desc, plan, plan_capacity, info};
  {
    // under the lock, so a worker about to sleep either sees the job or is woken
    std::lock_guard<std::mutex> lk(p->mu);
    p->state.store(kPosted, std::memory_order_release);
  }
  p->cv.notify_one();
  return PKV_OK;
}

extern "C" pkv_status pkv_planner_wait(pkv_planner *p) {
  if (!p) return PKV_ERR_NULL;
  int s = p->state.load(std::memory_order_acquire);
  if (s == kIdle) return PKV_ERR_STATE;
  while (s != kDone) s = p->state.load(std::memory_order_acquire);
  const pkv_status r = p->result;
  p->state.store(kIdle, std::memory_order_release);
  return r;
}
