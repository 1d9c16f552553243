// C ABI of libmoecache.so: cache lifetime, the decode call, state readout, resize.
//
// The cache is FreeToken's global expert-slot cache (snackonai deep dive
// "FreeToken, or why your laptop was never the bottleneck", sections "What It
// Actually Does" and "The Architecture, Unpacked"): the host copy of every
// expert is authoritative, GPU memory holds C complete expert blobs, and every
// table (where an expert lives, which slot goes next, what runs) is keyed by the
// flat id l*E+e.
//
// GB300 layout: the slot pool is one device allocation of C*S bytes (slot s at
// s*S, every blob 16-byte aligned); the residency tables are int32 arrays
// indexed by flat id and by slot, the recency stamps one uint64 per slot and a
// uint64 clock; per-call work buffers have fixed shapes sized by max_tokens so
// every launch has a fixed grid and the decode step can be captured in a CUDA
// graph.  The host pool stays where the caller put it, page-locked and mapped,
// and fills read it directly over the host link.
#include "internal.cuh"

#include <algorithm>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

namespace moe {
cudaError_t launch_resize_plan(int C_old, int C_new, int32_t* s2e, uint64_t* stamp, int32_t* new_s2e,
                               uint64_t* new_stamp, int32_t* new2old, int32_t* n_keep,
                               cudaStream_t s);
cudaError_t launch_resize_copy(const int32_t* new2old, const int32_t* n_keep, int C_new,
                               const uint8_t* old_slots, uint8_t* new_slots, uint64_t S, cudaStream_t s);
cudaError_t launch_rebuild_e2s(int n_flat, int C_new, const int32_t* new_s2e, int32_t* e2s, cudaStream_t s);
}  // namespace moe

using namespace moe;

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
static thread_local std::string g_last_error;

moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}


#include "cache.cuh"

#include <cstdlib>

static thread_local int g_inject_at = 0;      // the allocation that fails (0: none)
static thread_local int g_alloc_seen = 0;     // allocations so far in this create / resize call

void alloc_injection_begin() {
  const char* e = getenv("MOE_INJECT_ALLOC_FAILURE");
  g_inject_at = e ? atoi(e) : 0;
  g_alloc_seen = 0;
}
static bool injected_failure() { return g_inject_at > 0 && ++g_alloc_seen == g_inject_at; }
cudaError_t moe_malloc(void** p, size_t bytes) {
  if (injected_failure()) return cudaErrorMemoryAllocation;
  return cudaMalloc(p, bytes);
}
cudaError_t moe_host_alloc(void** p, size_t bytes, unsigned flags) {
  if (injected_failure()) return cudaErrorMemoryAllocation;
  return cudaHostAlloc(p, bytes, flags);
}
cudaError_t moe_host_register(void* p, size_t bytes, unsigned flags) {
  if (injected_failure()) return cudaErrorMemoryAllocation;
  return cudaHostRegister(p, bytes, flags);
}

static moe_status check_err_word(moe_cache* c) {
  const uint32_t e = *reinterpret_cast<volatile uint32_t*>(c->err_host);
  if (e == 0) return MOE_OK;
  *reinterpret_cast<volatile uint32_t*>(c->err_host) = 0;
  return fail(MOE_EDEVICE, "device flagged an earlier call: %s%s%s%s%s",
              (e & kErrBadExpertId) ? "expert id out of range; " : "",
              (e & kErrMissingCpuPart) ? "CPU-assigned pair without CPU partial sums; " : "",
              (e & kErrCapacity) ? "prefill capacity; " : "",
              (e & kErrClock) ? "recency clock overflow; " : "",
              (e & kErrTimeout) ? "device wait timed out; " : "");
}

static void free_cpu_branch(moe_cache* c) {
  if (c->ev_cpu) cudaEventDestroy(c->ev_cpu);
  if (c->cpu_stream) cudaStreamDestroy(c->cpu_stream);
  if (c->cpu_x_host) cudaFreeHost(c->cpu_x_host);
  if (c->cpu_ids_host) cudaFreeHost(c->cpu_ids_host);
  if (c->cpu_sm_host) cudaFreeHost(c->cpu_sm_host);
  if (c->cpu_part_host) cudaFreeHost(c->cpu_part_host);
  cudaFree(c->cpu_part_dev);
  c->ev_cpu = nullptr; c->cpu_stream = nullptr; c->cpu_x_host = nullptr; c->cpu_ids_host = nullptr;
  c->cpu_sm_host = nullptr; c->cpu_part_host = nullptr; c->cpu_part_dev = nullptr;
  c->cpu_fn = nullptr; c->cpu_user = nullptr;
  c->cpu_calls.clear();
}

static void destroy_impl(moe_cache* c) {
  if (!c) return;
  DeviceGuard g(c->cfg.device);
  cudaDeviceSynchronize();
  moe::prefill_free(c);
  free_cpu_branch(c);
  if (c->ev_ctrl) cudaEventDestroy(c->ev_ctrl);
  if (c->ev_fill) cudaEventDestroy(c->ev_fill);
  if (c->fill_stream) cudaStreamDestroy(c->fill_stream);
  cudaFree(c->slots);
  cudaFree(c->shared);
  cudaFree(c->offsets);
  cudaFree(c->tab.e2s);
  cudaFree(c->tab.s2e);
  cudaFree(c->tab.stamp);
  cudaFree(c->tab.clock);
  cudaFree(c->tab.counters);
  cudaFree(c->tab.pool);
  cudaFree(c->work);
  if (c->err_host) cudaFreeHost(c->err_host);
  if (c->registered_here) cudaHostUnregister(const_cast<uint8_t*>(c->host_pool));
  delete c;
}

static bool valid_dtype(int d) { return d == MOE_F32 || d == MOE_BF16 || d == MOE_FP8E4M3_B128 || d == MOE_NVFP4 ||
                                         d == MOE_MXFP4; }

static moe_status alloc_tables(moe_cache* c, uint64_t C) {
  const uint64_t nflat = (uint64_t)c->sh.L * c->sh.E;
  CK(moe_malloc(&c->tab.s2e, C * sizeof(int32_t)));
  CK(moe_malloc(&c->tab.stamp, C * sizeof(uint64_t)));
  CK(cudaMemset(c->tab.s2e, 0xff, C * sizeof(int32_t)));
  CK(cudaMemset(c->tab.stamp, 0, C * sizeof(uint64_t)));
  (void)nflat;
  return MOE_OK;
}

extern "C" moe_status moe_cache_create(const moe_config* cfg, const void* host_pool, uint64_t host_pool_bytes,
                                       const uint64_t* blob_offsets, const void* shared_host, uint64_t n_slots,
                                       moe_cache** out) {
  if (!cfg || !out) return fail(MOE_EINVAL, "cfg and out must not be NULL");
  *out = nullptr;
  alloc_injection_begin();
  const moe_config& k = *cfg;
  if (k.n_layers < 1 || k.n_experts < 1 || k.n_experts > kMaxExperts)
    return fail(MOE_EINVAL, "need 1 <= L and 1 <= E <= %d", kMaxExperts);
  if (k.top_k < 1 || k.top_k > k.n_experts) return fail(MOE_EINVAL, "need 1 <= top_k <= E");
  if (k.max_tokens < 1 || k.max_tokens > kMaxDecodeTokens)
    return fail(MOE_EINVAL, "need 1 <= max_tokens <= %d", kMaxDecodeTokens);
  if (!valid_dtype(k.wdtype) || (k.adtype != MOE_F32 && k.adtype != MOE_BF16))
    return fail(MOE_EINVAL, "bad wdtype/adtype");
  if (k.hidden < 8 || k.inter < 8 || k.hidden % 8 || k.inter % 8)
    return fail(MOE_EINVAL, "H and I must be positive multiples of 8");
  if (k.wdtype == MOE_FP8E4M3_B128 && (k.hidden % 128 || k.inter % 128))
    return fail(MOE_EINVAL, "fp8 block-scaled weights need H and I multiples of 128");
  if ((k.wdtype == MOE_NVFP4 || k.wdtype == MOE_MXFP4) && (k.hidden % 32 || k.inter % 32))
    return fail(MOE_EINVAL, "fp4 weights need H and I multiples of 32");
  // every slot and host blob starts on a 16-byte boundary (the kernels move 16-byte chunks)
  if (blob_bytes(k.wdtype, k.hidden, k.inter) % 16)
    return fail(MOE_EINVAL, "blob size S = %llu is not a multiple of 16 bytes (fp8: the scale count "
                "(2I/128)(H/128) + (H/128)(I/128) must be a multiple of 4)",
                (unsigned long long)blob_bytes(k.wdtype, k.hidden, k.inter));
  if (k.n_shared != 0 && k.n_shared != 1) return fail(MOE_EINVAL, "n_shared must be 0 or 1");
  if (k.n_shared && !shared_host) return fail(MOE_EINVAL, "n_shared = 1 needs shared_host");
  if ((uint64_t)k.bw_pcie_mbps + k.bw_cpu_mbps == 0) return fail(MOE_EINVAL, "B_pcie + B_cpu must be > 0");
  if (n_slots < 1 || n_slots >= kMaxSlots) return fail(MOE_EINVAL, "need 1 <= n_slots < 2^20");
  if (!host_pool) return fail(MOE_EINVAL, "host_pool must not be NULL");
  if (reinterpret_cast<uintptr_t>(host_pool) % 16) return fail(MOE_EINVAL, "host_pool must be 16-byte aligned");
  if (k.max_prefill_tokens < 0) return fail(MOE_EINVAL, "max_prefill_tokens must be >= 0");

  int ndev = 0;
  CK(cudaGetDeviceCount(&ndev));
  if (k.device < 0 || k.device >= ndev) return fail(MOE_EINVAL, "device %d out of range", k.device);
  DeviceGuard guard(k.device);

  moe_cache* c = new moe_cache();
  c->cfg = k;
  c->sh.L = k.n_layers; c->sh.E = k.n_experts; c->sh.H = k.hidden; c->sh.I = k.inter; c->sh.k = k.top_k;
  c->sh.wdtype = k.wdtype; c->sh.adtype = k.adtype; c->sh.n_shared = k.n_shared;
  c->sh.S = blob_bytes(k.wdtype, k.hidden, k.inter);
  const uint64_t S = c->sh.S;
  const uint64_t nflat = (uint64_t)k.n_layers * k.n_experts;
  c->K = k.max_fetch < 0 ? std::min(k.n_experts, k.max_tokens * k.top_k) : std::min(k.max_fetch, kMaxExperts);
  c->C = n_slots;
  c->host_pool = static_cast<const uint8_t*>(host_pool);
  c->host_bytes = host_pool_bytes;

  auto bail = [&](moe_status st) { destroy_impl(c); return st; };

  // offsets
  std::vector<uint64_t> offs(nflat);
  for (uint64_t f = 0; f < nflat; ++f) {
    offs[f] = blob_offsets ? blob_offsets[f] : f * S;
    if (offs[f] % 16 || offs[f] + S > host_pool_bytes) {
      moe_status st = fail(MOE_EINVAL, "blob %llu: offset %llu not 16-aligned or past the pool",
                           (unsigned long long)f, (unsigned long long)offs[f]);
      return bail(st);
    }
  }

  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, k.device) != cudaSuccess) return bail(fail(MOE_ECUDA, "device properties"));
  c->sms = prop.multiProcessorCount;
  c->gemv_grid = 2 * c->sms;
  c->fill_ctas = c->sms / 2;
  {
    // The resident experts of a decode call run as a gate/up grid then a down +
    // combine grid (the default, "grids"), or, for one-token calls, chosen by
    // MOE_DECODE_RESIDENT when the cache is created: "fused" = one launch with a
    // grid-wide barrier between the two (also MOE_DECODE_FUSED=1).  Both give the
    // same outputs bit for bit.
    const char* er = getenv("MOE_DECODE_RESIDENT");
    const char* ef = getenv("MOE_DECODE_FUSED");
    c->resident_mode = 0;
    if (ef && ef[0] == '1') c->resident_mode = 1;
    if (er && strcmp(er, "grids") == 0) c->resident_mode = 0;
    else if (er && strcmp(er, "fused") == 0) c->resident_mode = 1;
    else if (er && er[0]) return bail(fail(MOE_EINVAL, "MOE_DECODE_RESIDENT must be grids or fused"));
  }

  // host pool: page-lock (mapped) unless it already is
  cudaPointerAttributes attr;
  cudaError_t ae = cudaPointerGetAttributes(&attr, host_pool);
  if (ae != cudaSuccess) cudaGetLastError();
  if (ae != cudaSuccess || attr.type != cudaMemoryTypeHost) {
    cudaError_t re = moe_host_register(const_cast<void*>(host_pool), host_pool_bytes,
                                       cudaHostRegisterMapped | cudaHostRegisterReadOnly);
    if (re != cudaSuccess && re != cudaErrorMemoryAllocation) {   // read-only mapping refused: plain mapped
      cudaGetLastError();
      re = cudaHostRegister(const_cast<void*>(host_pool), host_pool_bytes, cudaHostRegisterMapped);
    }
    if (re != cudaSuccess) return bail(fail(MOE_ENOMEM, "cudaHostRegister of the pool: %s", cudaGetErrorString(re)));
    c->registered_here = true;
  }
  void* dptr = nullptr;
  if (cudaHostGetDevicePointer(&dptr, const_cast<void*>(host_pool), 0) != cudaSuccess)
    return bail(fail(MOE_ECUDA, "host pool has no device mapping"));
  c->host_pool_dev = static_cast<const uint8_t*>(dptr);

  moe_status st;
#define CKB(call)                                                                             \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess)                                                                    \
      return bail(fail(e_ == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "%s: %s", #call, \
                       cudaGetErrorString(e_)));                                              \
  } while (0)

  CKB(setup_control_kernels());
  CKB(setup_gemv_kernels());
  CKB(moe_malloc(&c->offsets, nflat * sizeof(uint64_t)));
  CKB(cudaMemcpy(c->offsets, offs.data(), nflat * sizeof(uint64_t), cudaMemcpyHostToDevice));
  CKB(moe_malloc(&c->slots, c->C * S));
  CKB(moe_malloc(&c->tab.e2s, nflat * sizeof(int32_t)));
  CKB(cudaMemset(c->tab.e2s, 0xff, nflat * sizeof(int32_t)));
  if ((st = alloc_tables(c, c->C)) != MOE_OK) return bail(st);
  CKB(moe_malloc(&c->tab.clock, sizeof(uint64_t)));
  CKB(cudaMemset(c->tab.clock, 0, sizeof(uint64_t)));
  CKB(moe_malloc(&c->tab.counters, 8 * sizeof(uint64_t)));
  CKB(cudaMemset(c->tab.counters, 0, 8 * sizeof(uint64_t)));
  CKB(moe_malloc(&c->tab.pool, (kPoolN + 1) * sizeof(uint64_t)));
  CKB(cudaMemset(c->tab.pool, 0, (kPoolN + 1) * sizeof(uint64_t)));   // count 0: rebuilt at the first call
  if (k.n_shared) {
    CKB(moe_malloc(&c->shared, (uint64_t)k.n_layers * S));
    CKB(cudaMemcpy(c->shared, shared_host, (uint64_t)k.n_layers * S, cudaMemcpyHostToDevice));
  }
  // work buffers
  {
    const int umax = std::min(k.n_experts, k.max_tokens * k.top_k);
    const int max_gpu = umax + k.n_shared;
    const uint64_t max_pairs = (uint64_t)k.max_tokens * k.top_k + (uint64_t)k.max_tokens * k.n_shared;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) & ~size_t(255); return o; };
    const size_t o_plan = take(P_COUNT * 4), o_vict = take((size_t)std::max(c->K, 1) * 4),
                 o_fill = take((size_t)std::max(c->K, 1) * 8), o_cpu = take((size_t)umax * 4),
                 o_sm = take((size_t)k.max_tokens * k.top_k * 4), o_goff = take((size_t)(max_gpu + 1) * 4),
                 o_gp = take(max_pairs * 4), o_gw = take((size_t)max_gpu * 8),
                 o_h = take(max_pairs * k.inter * 4), o_y = take(max_pairs * k.hidden * 4),
                 o_arr = take((size_t)k.hidden * 4), o_fb = take(8), o_ns = take(4);
    CKB(moe_malloc(&c->work, off));
    CKB(cudaMemset(c->work, 0, off));
    uint8_t* w = static_cast<uint8_t*>(c->work);
    c->b.plan = reinterpret_cast<int32_t*>(w + o_plan);
    c->b.victims = reinterpret_cast<int32_t*>(w + o_vict);
    c->b.fills = reinterpret_cast<int32_t*>(w + o_fill);
    c->b.cpu = reinterpret_cast<int32_t*>(w + o_cpu);
    c->b.slot_map = reinterpret_cast<int32_t*>(w + o_sm);
    c->b.gpu_off = reinterpret_cast<int32_t*>(w + o_goff);
    c->b.gpu_pairs = reinterpret_cast<int32_t*>(w + o_gp);
    c->b.gpu_w = reinterpret_cast<const uint8_t**>(w + o_gw);
    c->b.h = reinterpret_cast<float*>(w + o_h);
    c->b.y = reinterpret_cast<float*>(w + o_y);
    c->b.arrive = reinterpret_cast<uint32_t*>(w + o_arr);
    c->b.fused_bar = reinterpret_cast<unsigned long long*>(w + o_fb);
    // A test of the bounded waits (MOE_TEST_UNSET_WAIT=1 when the cache is created):
    // the resident experts' down kernel also waits for a word nothing writes,
    // gives up after 20 ms, flags the timeout and returns; the next call reports
    // MOE_EDEVICE.  Off unless set.
    CKB(cudaMemset(w + o_ns, 0xff, 4));
    c->b.never_set = reinterpret_cast<const float*>(w + o_ns);
    {
      const char* tw = getenv("MOE_TEST_UNSET_WAIT");
      c->b.test_wait = (tw && tw[0] == '1') ? 1 : 0;
    }
    c->dev_bytes = off;
  }
  c->dev_bytes += c->C * S + nflat * 12 + c->C * 12 + (k.n_shared ? (uint64_t)k.n_layers * S : 0);
  CKB(moe_host_alloc(reinterpret_cast<void**>(&c->err_host), sizeof(uint32_t), cudaHostAllocMapped));
  *c->err_host = 0;
  CKB(cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->err_dev), c->err_host, 0));
  {
    // fills gate the filled experts' GEMV: give their CTAs first pick of free SM slots
    int least = 0, greatest = 0;
    CKB(cudaDeviceGetStreamPriorityRange(&least, &greatest));
    CKB(cudaStreamCreateWithPriority(&c->fill_stream, cudaStreamNonBlocking, greatest));
  }
  CKB(cudaEventCreateWithFlags(&c->ev_ctrl, cudaEventDisableTiming));
  CKB(cudaEventCreateWithFlags(&c->ev_fill, cudaEventDisableTiming));
  if (k.max_prefill_tokens > 0) {
    if ((st = moe::prefill_init(c)) != MOE_OK) return bail(st);
  }
  CKB(cudaDeviceSynchronize());
#undef CKB
  *out = c;
  g_last_error.clear();
  return MOE_OK;
}

extern "C" moe_status moe_cache_destroy(moe_cache* c) {
  destroy_impl(c);
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// CPU branch
// ---------------------------------------------------------------------------
// The host node of a decode call's CPU branch (runs on a CUDA driver thread).
static void CUDART_CB cpu_branch_host(void* p) {
  const moe_cache::CpuCall* a = static_cast<const moe_cache::CpuCall*>(p);
  moe_cache* c = a->c;
  c->cpu_fn(c->cpu_user, a->layer, a->T, c->cpu_x_host, c->cpu_ids_host, c->cpu_sm_host, c->cpu_part_host);
}

// The exact merge once both branches are done: y of the GPU pairs, the CPU
// branch's partial sums, top-k order (+ shared expert).
static moe_status combine_after_cpu_branch(moe_cache* c, int T, const float* w, float* out, cudaStream_t s) {
  CK(cudaStreamWaitEvent(s, c->ev_cpu, 0));
  ProfScope p(c, s, PROF_DOWN_COMBINE);
  CK(launch_combine(c->sh, T, w, c->cpu_part_dev, c->b, out, c->err_dev, s));
  return MOE_OK;
}

extern "C" moe_status moe_cache_set_cpu_branch(moe_cache* c, moe_cpu_branch_fn fn, void* user) {
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  DeviceGuard guard(c->cfg.device);
  CK(cudaDeviceSynchronize());
  free_cpu_branch(c);
  if (!fn) return MOE_OK;
  const size_t T = (size_t)c->cfg.max_tokens, k = (size_t)c->sh.k, H = (size_t)c->sh.H;
  const size_t xb = T * H * (c->sh.adtype == MOE_F32 ? 4 : 2);
  cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&c->cpu_x_host), xb, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&c->cpu_ids_host), T * k * 4, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&c->cpu_sm_host), T * k * 4, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&c->cpu_part_host), T * k * H * 4, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&c->cpu_part_dev), T * k * H * 4);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->cpu_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_cpu, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_cpu_branch(c);
    return fail(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "CPU branch set-up: %s", cudaGetErrorString(e));
  }
  memset(c->cpu_part_host, 0, T * k * H * 4);
  c->cpu_calls.resize((size_t)c->sh.L * T);
  for (int l = 0; l < c->sh.L; ++l)
    for (size_t t = 0; t < T; ++t) c->cpu_calls[(size_t)l * T + t] = {c, l, (int)t + 1};
  c->cpu_fn = fn;
  c->cpu_user = user;
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// decode: control -> side stream: fill + gate/up of the filled experts, then
//                    their down projection
//                 -> gate/up of the resident experts, then their down projection
//                 -> the second of the two down grids to finish a row block
//                    forms its combine; the call ends with the streams joined.
// Shapes whose h or down rows do not fit the split kernels run the down
// projection of every GPU expert after the fills instead.
// ---------------------------------------------------------------------------
extern "C" moe_status moe_layer_decode(moe_cache* c, int32_t layer, int32_t T, const void* x,
                                       const int32_t* ids, const float* w, const float* cpu_part,
                                       float* out, int32_t* slot_map, void* stream) {
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  moe_status st = check_err_word(c);
  if (st != MOE_OK) return st;
  if (layer < 0 || layer >= c->sh.L) return fail(MOE_EINVAL, "layer %d out of range", layer);
  if (T < 0 || T > c->cfg.max_tokens) return fail(MOE_EINVAL, "T = %d outside [0, max_tokens]", T);
  if (T == 0) return MOE_OK;
  if (!x || !ids || !w || !out) return fail(MOE_EINVAL, "x, topk_ids, topk_w and out must not be NULL");
  if (!aligned_to(x, 16) || !aligned_to(out, 16) || (cpu_part && !aligned_to(cpu_part, 16)))
    return fail(MOE_EINVAL, "x, out and cpu_part must be 16-byte aligned");
  if (!aligned_to(ids, 4) || !aligned_to(w, 4) || (slot_map && !aligned_to(slot_map, 4)))
    return fail(MOE_EINVAL, "topk_ids, topk_w and slot_map must be 4-byte aligned");
  DeviceGuard guard(c->cfg.device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_T = T;
  const bool split = down_split_ok(c->sh, T, c->sms);
  const int path = resident_path(c, T);
  // with a CPU branch the down kernels only store y; one combine kernel follows both branches
  const bool branch = c->cpu_fn != nullptr;
  DecodeBufs b = c->b;
  b.defer_combine = branch ? 1 : 0;
  if (branch) cpu_part = nullptr;
  {
    ProfScope p(c, s, PROF_CONTROL);
    CK(launch_decode_control(c->sh, layer, T, (int)c->C, c->K, c->cfg.bw_pcie_mbps, c->cfg.bw_cpu_mbps, ids,
                             c->tab, b, slot_map, c->slots, c->shared, c->err_dev, s));
  }
  CK(cudaEventRecord(c->ev_ctrl, s));
  CK(cudaStreamWaitEvent(c->fill_stream, c->ev_ctrl, 0));
  if (branch) {
    // The CPU branch: what the CPU-assigned experts read goes to the host, the
    // registered function computes their partial sums, and those come back
    const size_t kT = (size_t)T * c->sh.k;
    const size_t xb = (size_t)T * c->sh.H * (c->sh.adtype == MOE_F32 ? 4 : 2);
    CK(cudaStreamWaitEvent(c->cpu_stream, c->ev_ctrl, 0));
    CK(cudaMemcpyAsync(c->cpu_x_host, x, xb, cudaMemcpyDeviceToHost, c->cpu_stream));
    CK(cudaMemcpyAsync(c->cpu_ids_host, ids, kT * 4, cudaMemcpyDeviceToHost, c->cpu_stream));
    CK(cudaMemcpyAsync(c->cpu_sm_host, c->b.slot_map, kT * 4, cudaMemcpyDeviceToHost, c->cpu_stream));
    CK(cudaLaunchHostFunc(c->cpu_stream, cpu_branch_host,
                          &c->cpu_calls[(size_t)layer * c->cfg.max_tokens + (T - 1)]));
    CK(cudaMemcpyAsync(c->cpu_part_dev, c->cpu_part_host, kT * c->sh.H * 4, cudaMemcpyHostToDevice, c->cpu_stream));
    CK(cudaEventRecord(c->ev_cpu, c->cpu_stream));
  }
  {
    // fills, and the gate/up GEMV of the filled experts on the way through
    ProfScope p(c, c->fill_stream, PROF_FILL);
    CK(launch_fill_gate_up(c->sh, T, x, b, c->host_pool_dev, c->offsets, c->slots, c->fill_ctas, c->fill_stream));
  }
  if (split) {
    // Beside the fused resident launch, whose CTAs wait on one another at its grid
    // barrier, the filled-expert grid is a plain launch: launched early, its CTAs
    // would sit on SMs for the whole fill and could keep some fused CTAs off the GPU.
    ProfScope p(c, c->fill_stream, PROF_DOWN_FILLED);
    CK(launch_down_split(c->sh, 1, T, w, cpu_part, b, out, c->err_dev, c->sms, c->fill_stream, path == 0));
  }
  CK(cudaEventRecord(c->ev_fill, c->fill_stream));
  if (split) {
    {
      // one timed group: the two grids run back to back under a programmatic dependency
      ProfScope p(c, s, PROF_GEMV_RESIDENT);
      if (path == 1) {
        CK(launch_resident_fused(c->sh, T, x, w, cpu_part, b, out, c->err_dev, c->sms, s));
      } else {
        CK(launch_gate_up(c->sh, 0, T, x, b, c->sms, s, c->err_dev));
        CK(launch_down_split(c->sh, 0, T, w, cpu_part, b, out, c->err_dev, c->sms, s));
      }
    }
    CK(cudaStreamWaitEvent(s, c->ev_fill, 0));
    return branch ? combine_after_cpu_branch(c, T, w, out, s) : MOE_OK;
  }
  {
    ProfScope p(c, s, PROF_GEMV_RESIDENT);
    CK(launch_gate_up(c->sh, 0, T, x, b, c->sms, s, c->err_dev));
  }
  CK(cudaStreamWaitEvent(s, c->ev_fill, 0));
  {
    ProfScope p(c, s, PROF_DOWN_COMBINE);
    CK(launch_down_combine(c->sh, T, w, cpu_part, b, out, c->err_dev, c->sms, s));
  }
  return branch ? combine_after_cpu_branch(c, T, w, out, s) : MOE_OK;
}

// ---------------------------------------------------------------------------
// readout
// ---------------------------------------------------------------------------
extern "C" moe_status moe_cache_get_state(moe_cache* c, int32_t* s2e, uint64_t* stamps, int32_t* e2s,
                                          uint64_t* counters, uint64_t* clock) {
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  DeviceGuard guard(c->cfg.device);
  CK(cudaDeviceSynchronize());
  if (s2e) CK(cudaMemcpy(s2e, c->tab.s2e, c->C * 4, cudaMemcpyDeviceToHost));
  if (stamps) CK(cudaMemcpy(stamps, c->tab.stamp, c->C * 8, cudaMemcpyDeviceToHost));
  if (e2s) CK(cudaMemcpy(e2s, c->tab.e2s, (size_t)c->sh.L * c->sh.E * 4, cudaMemcpyDeviceToHost));
  if (counters) CK(cudaMemcpy(counters, c->tab.counters, 64, cudaMemcpyDeviceToHost));
  if (clock) CK(cudaMemcpy(clock, c->tab.clock, 8, cudaMemcpyDeviceToHost));
  return check_err_word(c);
}

extern "C" moe_status moe_cache_get_plan(moe_cache* c, int32_t* scalars, int32_t* victims, int32_t* fills,
                                         float* y) {
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  DeviceGuard guard(c->cfg.device);
  CK(cudaDeviceSynchronize());
  if (scalars) {
    int32_t p[P_COUNT];
    CK(cudaMemcpy(p, c->b.plan, sizeof(p), cudaMemcpyDeviceToHost));
    scalars[0] = p[P_LAYER]; scalars[1] = p[P_U]; scalars[2] = p[P_H]; scalars[3] = p[P_M];
    scalars[4] = p[P_Q]; scalars[5] = p[P_NCPU]; scalars[6] = p[P_NGPU]; scalars[7] = 0;
  }
  if (victims && c->K) CK(cudaMemcpy(victims, c->b.victims, (size_t)c->K * 4, cudaMemcpyDeviceToHost));
  if (fills && c->K) CK(cudaMemcpy(fills, c->b.fills, (size_t)c->K * 8, cudaMemcpyDeviceToHost));
  if (y) CK(cudaMemcpy(y, c->b.y, (size_t)c->last_T * c->sh.k * c->sh.H * 4, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

extern "C" moe_status moe_cache_info(moe_cache* c, uint64_t* info) {
  if (!c || !info) return fail(MOE_EINVAL, "NULL argument");
  info[0] = c->sh.S; info[1] = c->C; info[2] = (uint64_t)c->K; info[3] = (uint64_t)c->sh.L * c->sh.E;
  info[4] = c->dev_bytes; info[5] = c->host_bytes; info[7] = 0;
  {
    const int T = c->cfg.max_tokens;
    info[7] = (uint64_t)resident_path(c, T);
  }
  {
    // control + fill + resident experts (one fused launch, or gate/up + down) + filled-expert down,
    // or control + fill + gate/up + the down/combine kernels where the split ones do not fit
    const int T = c->cfg.max_tokens;
    if (down_split_ok(c->sh, T, c->sms))
      info[6] = resident_path(c, T) != 0 ? 4 : 5;
    else
      info[6] = 3 + (uint64_t)down_combine_launches(c->sh, T, c->sms);
    if (c->cpu_fn) info[6] += 1;   // the combine kernel after the CPU branch
  }
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// resize (safe point): plan survivors on the device, copy them into a new pool
// ---------------------------------------------------------------------------
extern "C" moe_status moe_cache_resize(moe_cache* c, uint64_t n_slots) {
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  if (n_slots < 1 || n_slots >= kMaxSlots) return fail(MOE_EINVAL, "need 1 <= n_slots < 2^20");
  moe_status st = check_err_word(c);
  if (st != MOE_OK) return st;
  DeviceGuard guard(c->cfg.device);
  CK(cudaDeviceSynchronize());
  const uint64_t S = c->sh.S;
  uint8_t* new_slots = nullptr;
  int32_t *new_s2e = nullptr, *new2old = nullptr;
  uint64_t* new_stamp = nullptr;
  auto cleanup = [&]() { cudaFree(new_slots); cudaFree(new_s2e); cudaFree(new2old); cudaFree(new_stamp); };
  alloc_injection_begin();
  cudaError_t e = moe_malloc(&new_slots, n_slots * S);
  if (e == cudaSuccess) e = moe_malloc(&new_s2e, n_slots * 4);
  if (e == cudaSuccess) e = moe_malloc(&new_stamp, n_slots * 8);
  if (e == cudaSuccess) e = moe_malloc(&new2old, (n_slots + 1) * 4);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cleanup();
    return fail(MOE_ENOMEM, "resize to %llu slots: %s (the old pool is kept)", (unsigned long long)n_slots,
                cudaGetErrorString(e));
  }
  cudaStream_t s = c->fill_stream;
  int32_t* n_keep = new2old + n_slots;
  e = launch_resize_plan((int)c->C, (int)n_slots, c->tab.s2e, c->tab.stamp, new_s2e, new_stamp, new2old, n_keep, s);
  if (e == cudaSuccess) e = launch_resize_copy(new2old, n_keep, (int)n_slots, c->slots, new_slots, S, s);
  if (e == cudaSuccess) e = launch_rebuild_e2s(c->sh.L * c->sh.E, (int)n_slots, new_s2e, c->tab.e2s, s);
  // new slots enter empty (stamp 0, below every kept candidate): drop the decode candidate pool
  if (e == cudaSuccess) e = cudaMemsetAsync(c->tab.pool + kPoolN, 0, sizeof(uint64_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cleanup();
    return fail(MOE_ECUDA, "resize: %s", cudaGetErrorString(e));
  }
  cudaFree(c->slots);
  cudaFree(c->tab.s2e);
  cudaFree(c->tab.stamp);
  c->dev_bytes = c->dev_bytes - c->C * (S + 12) + n_slots * (S + 12);
  c->slots = new_slots;
  c->tab.s2e = new_s2e;
  c->tab.stamp = new_stamp;
  c->C = n_slots;
  cudaFree(new2old);
  return MOE_OK;
}

extern "C" moe_status moe_cache_profile(moe_cache* c, int32_t mode, double* ms_host, uint64_t* launches_host) {
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  if (mode < 0 || mode > 3) return fail(MOE_EINVAL, "profile mode must be 0..3");
  DeviceGuard guard(c->cfg.device);
  if (mode == 1) {            // start: reset and record; pre-create events so capture never creates any
    while (c->prof_events.size() < 2 * 4096) {
      cudaEvent_t e;
      CK(cudaEventCreate(&e));
      c->prof_events.push_back(e);
    }
    c->prof_kind.resize(c->prof_events.size() / 2);
    c->prof_used = 0;
    c->profiling = true;
    return MOE_OK;
  }
  if (mode == 3) {            // pause: keep the recorded pairs, record no new ones
    c->profiling = false;
    return MOE_OK;
  }
  // 0 = stop + read + reset, 2 = read only
  if (mode == 0) c->profiling = false;
  CK(cudaDeviceSynchronize());
  double ms[PROF_KINDS] = {0};
  uint64_t n[PROF_KINDS] = {0};
  for (size_t i = 0; i < c->prof_used; ++i) {
    float t = 0.f;
    CK(cudaEventElapsedTime(&t, c->prof_events[2 * i], c->prof_events[2 * i + 1]));
    ms[c->prof_kind[i]] += t;
    n[c->prof_kind[i]] += 1;
  }
  for (int k = 0; k < PROF_KINDS; ++k) {
    if (ms_host) ms_host[k] = ms[k];
    if (launches_host) launches_host[k] = n[k];
  }
  if (mode == 0) c->prof_used = 0;
  return MOE_OK;
}

extern "C" const char* moe_last_error(void) { return g_last_error.c_str(); }
