// The cache object shared by the translation units of libmoecache.so.
#pragma once

#include "internal.cuh"

#include <cuda.h>

#include <vector>

// set the thread's last error message and return `st`
moe_status fail(moe_status st, const char* fmt, ...);

// Host-side fault injection for tests.  With MOE_INJECT_ALLOC_FAILURE=n in the
// environment, the n-th device or page-locked allocation (or host-pool
// registration) of one moe_cache_create or moe_cache_resize call reports out of
// memory instead of allocating (n >= 1; unset or 0: off).  The count starts over
// at each such call.  Every allocation of those calls goes through these.
void alloc_injection_begin();
cudaError_t moe_malloc(void** p, size_t bytes);
cudaError_t moe_host_alloc(void** p, size_t bytes, unsigned flags);
cudaError_t moe_host_register(void* p, size_t bytes, unsigned flags);
template <typename T> cudaError_t moe_malloc(T** p, size_t bytes) {
  return moe_malloc(reinterpret_cast<void**>(p), bytes);
}

#define CK(call)                                                                      \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess)                                                            \
      return fail(e_ == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "%s: %s", \
                  #call, cudaGetErrorString(e_));                                     \
  } while (0)

using namespace moe;

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// ---------------------------------------------------------------------------
// the cache object
// ---------------------------------------------------------------------------
struct moe_cache {
  moe_config cfg{};
  Shape sh{};
  int K = 0;
  uint64_t C = 0;
  int sms = 0;
  int gemv_grid = 0;
  int fill_ctas = 0;
  // how one-token calls run their resident experts: 0 a gate/up grid then a down +
  // combine grid, 1 one launch with a grid-wide barrier
  int resident_mode = 0;
  // host pool
  const uint8_t* host_pool = nullptr;
  const uint8_t* host_pool_dev = nullptr;
  uint64_t host_bytes = 0;
  bool registered_here = false;
  // device memory
  uint8_t* slots = nullptr;
  uint8_t* shared = nullptr;
  uint64_t* offsets = nullptr;
  CacheTables tab{};
  DecodeBufs b{};
  void* work = nullptr;            // one allocation behind DecodeBufs
  uint64_t dev_bytes = 0;
  int last_T = 0;
  // error word (page-locked, mapped)
  uint32_t* err_host = nullptr;
  uint32_t* err_dev = nullptr;
  // streams / events
  cudaStream_t fill_stream = nullptr;
  cudaEvent_t ev_ctrl = nullptr, ev_fill = nullptr;
  // CPU branch (moe_cache_set_cpu_branch): the registered function, its stream and
  // event, page-locked staging of what it reads and writes, the device copy of its
  // partial sums, and one host-node argument per (layer, T)
  struct CpuCall { moe_cache* c; int layer, T; };
  moe_cpu_branch_fn cpu_fn = nullptr;
  void* cpu_user = nullptr;
  cudaStream_t cpu_stream = nullptr;
  cudaEvent_t ev_cpu = nullptr;
  uint8_t* cpu_x_host = nullptr;
  int32_t* cpu_ids_host = nullptr;
  int32_t* cpu_sm_host = nullptr;
  float* cpu_part_host = nullptr;
  float* cpu_part_dev = nullptr;
  std::vector<CpuCall> cpu_calls;
  // prefill state (prefill.cu)
  void* prefill = nullptr;
  // kernel timing (moe_cache_profile)
  bool profiling = false;
  std::vector<cudaEvent_t> prof_events;     // pairs, created outside any capture
  std::vector<int> prof_kind;               // kind of each pair
  size_t prof_used = 0;
};

// The resident-expert path a call of T tokens takes (0 or 1 as resident_mode;
// only split-down shapes take 1, and only where the fused launch applies).
inline int resident_path(const moe_cache* c, int T) {
  if (!down_split_ok(c->sh, T, c->sms)) return 0;
  if (c->resident_mode == 1 && resident_fused_ok(c->sh, T, c->sms)) return 1;
  return 0;
}

// Record a start/stop event pair around a kernel group of `kind` when profiling.
struct ProfScope {
  moe_cache* c;
  cudaStream_t s;
  size_t idx = (size_t)-1;
  ProfScope(moe_cache* c_, cudaStream_t s_, int kind) : c(c_), s(s_) {
    if (!c->profiling) return;
    if (c->prof_used * 2 + 2 > c->prof_events.size()) {
      for (int i = 0; i < 256; ++i) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) { c->profiling = false; return; }
        c->prof_events.push_back(e);
      }
      c->prof_kind.resize(c->prof_events.size() / 2);
    }
    idx = c->prof_used++;
    c->prof_kind[idx] = kind;
    record(c->prof_events[2 * idx]);
  }
  ~ProfScope() {
    if (idx != (size_t)-1) record(c->prof_events[2 * idx + 1]);
  }
  // inside a stream capture a plain record only joins streams; an external record
  // becomes a real event node that every replay re-records
  void record(cudaEvent_t e) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &st);
    if (st == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else cudaEventRecord(e, s);
  }
};

namespace moe {
// prefill.cu
moe_status prefill_init(moe_cache* c);
void prefill_free(moe_cache* c);
}  // namespace moe

