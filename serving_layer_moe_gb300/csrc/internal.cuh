// Internal declarations of libmoecache.so (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe_cache.h"

namespace moe {

// ---------------------------------------------------------------------------
// limits
// ---------------------------------------------------------------------------
constexpr int kMaxExperts = 4096;          // E: routed-expert bitmap of 128 words
constexpr int kMaxDecodeTokens = 1024;
constexpr int kSlotBits = 20;              // slot index field of an LRU key
constexpr uint64_t kMaxSlots = 1ull << kSlotBits;
constexpr int kCtrlThreads = 512;
// one shared-memory carveout (percent) for every decode kernel: no L1/shared
// reconfiguration between the kernels of a layer
constexpr int kDecodeCarveout = 100;

// error word bits (device -> host through page-locked mapped memory)
enum : uint32_t {
  kErrBadExpertId = 1u,
  kErrMissingCpuPart = 2u,
  kErrCapacity = 4u,
  kErrClock = 8u,
  kErrTimeout = 16u,
};

// ---------------------------------------------------------------------------
// plan scalars written by the decode control kernel, read by the GEMV / fill
// ---------------------------------------------------------------------------
enum PlanIdx : int {
  P_LAYER = 0, P_U = 1, P_H = 2, P_M = 3, P_Q = 4, P_NCPU = 5, P_NGPU = 6,
  P_NFIRST = 7,     // GPU experts in the first (resident) pass: hits + shared
  P_COUNT = 8,
};

// kernel groups timed by moe_cache_profile
enum ProfKind : int {
  PROF_CONTROL = 0, PROF_FILL = 1, PROF_GEMV_RESIDENT = 2, PROF_DOWN_FILLED = 3, PROF_DOWN_COMBINE = 4,
  PROF_PREFILL_CONTROL = 5, PROF_PREFILL_LOAD = 6, PROF_PREFILL_GEMM = 7, PROF_KINDS = 8,
};

// Everything the decode kernels of one call need, by value.
struct DecodeBufs {
  int32_t* plan;          // [P_COUNT]
  int32_t* victims;       // [K]
  int32_t* fills;         // [2K]  (flat id, slot)
  int32_t* cpu;           // [max unique]
  int32_t* slot_map;      // [max_tokens * k]  internal copy
  int32_t* gpu_off;       // [max_gpu + 1]  pair-list offsets per GPU expert
  int32_t* gpu_pairs;     // [max_pairs]    pair ids grouped by GPU expert
  const uint8_t** gpu_w;  // [max_gpu]      weight blob of each GPU expert
  float* h;               // [max_pairs, I] SwiGLU activations
  float* y;               // [max_pairs, H] expert outputs (unweighted)
  uint32_t* arrive;       // [H] arrivals of the two split down kernels per row block (parity = who combines)
  unsigned long long* fused_bar;   // grid-barrier arrivals of the fused resident kernel (only grows)
  // test of the bounded waits: with test_wait set, the resident down kernel (pass 0)
  // also waits (20 ms at most) for *never_set, which nothing writes
  const float* never_set;
  int test_wait;
  // This call's combine runs later, as its own kernel (a registered CPU branch
  // supplies the CPU partial sums): the down kernels only store y.
  int defer_combine;
};


struct CacheTables {
  int32_t* e2s;           // [L*E]
  int32_t* s2e;           // [C]
  uint64_t* stamp;        // [C]
  uint64_t* clock;        // [1]
  uint64_t* counters;     // [8]
  uint64_t* pool;         // [kPoolN + 1]: oldest LRU keys at the last rebuild, ascending; [kPoolN] = count
};

// Decode victim candidates kept between calls (K <= kPoolMaxK): the n smallest
// LRU keys as of the last full selection, n = pool_size(K, C) <= kPoolN.
constexpr int kPoolN = 512;
constexpr int kPoolMaxK = 128;
constexpr int kWarpPathMaxK = 16;   // the control kernel's one-warp path
__host__ __device__ constexpr int pool_size(int K, int C) {
  const int want = 4 * K < 64 ? 64 : (4 * K > kPoolN ? kPoolN : 4 * K);
  return C < want ? C : want;
}

struct Shape {
  int L, E, H, I, k;
  int wdtype, adtype;
  int n_shared;
  uint64_t S;             // blob bytes
};

// ---------------------------------------------------------------------------
// kernels (launch wrappers; all enqueue only)
// ---------------------------------------------------------------------------
// control.cu
cudaError_t launch_decode_control(const Shape& sh, int layer, int T, int C, int K, uint32_t bp,
                                  uint32_t bc, const int32_t* ids, CacheTables tab, DecodeBufs b,
                                  int32_t* slot_map_out, const uint8_t* slots_base,
                                  const uint8_t* shared_base, uint32_t* err, cudaStream_t s);

cudaError_t setup_control_kernels();  // once per device, before the first launch
cudaError_t setup_gemv_kernels();     // once per device, before the first launch

// expert_gemv.cu
cudaError_t launch_fill(const Shape& sh, const int32_t* plan, const int32_t* fills,
                        const uint8_t* host_pool_dev, const uint64_t* offsets, uint8_t* slots,
                        int n_ctas, cudaStream_t s);
cudaError_t launch_copy_blobs(const int32_t* count, const int32_t* skip, const int32_t* list,
                              const uint8_t* host_pool_dev, const uint64_t* offsets, uint8_t* slots,
                              uint64_t S, int n_ctas, cudaStream_t s);
// Prefill with NVFP4 / MXFP4 experts: the active experts of the layer that have
// routed rows (active[e] != 0, offsets[e + 1] > offsets[e], slot wslot[e]) decoded
// from their slots to bf16 blobs at staging + e * 3IH.
cudaError_t launch_fp4_to_bf16(const Shape& sh, const int32_t* wslot, const int32_t* active, const int32_t* offsets,
                               const uint8_t* slots, uint16_t* staging, int sms, cudaStream_t s);
cudaError_t launch_expert_gemv(const Shape& sh, int pass, int T, const void* x, DecodeBufs b,
                               int sms, cudaStream_t s);
// dynamic shared memory launch_expert_gemv's gate/up kernel needs for T tokens,
// and the most setup_gemv_kernels() allows it (a call above that cannot launch)
size_t expert_gemv_smem(const Shape& sh, int T);
size_t expert_gemv_smem_limit();
cudaError_t launch_fill_gate_up(const Shape& sh, int T, const void* x, DecodeBufs b, const uint8_t* host_pool_dev,
                                const uint64_t* offsets, uint8_t* slots, int n_ctas, cudaStream_t s);
cudaError_t launch_gate_up(const Shape& sh, int pass, int T, const void* x, DecodeBufs b, int sms, cudaStream_t s,
                           uint32_t* err);
cudaError_t launch_down_combine(const Shape& sh, int T, const float* w, const float* cpu_part, DecodeBufs b,
                                float* out, uint32_t* err, int sms, cudaStream_t s);
bool down_combine_fits(const Shape& sh, int T);
// Split down projection: pass 0 = resident experts (main stream, after their
// gate/up), pass 1 = filled experts (fill stream, after the fill); the second
// of the two CTAs of each row block to finish forms that block's combine.
bool down_split_ok(const Shape& sh, int T, int sms);
// pdl = false: a plain launch, whose CTAs hold no SM while the predecessor runs.
cudaError_t launch_down_split(const Shape& sh, int pass, int T, const float* w, const float* cpu_part, DecodeBufs b,
                              float* out, uint32_t* err, int sms, cudaStream_t s, bool pdl = true);
cudaError_t launch_combine(const Shape& sh, int T, const float* w, const float* cpu_part,
                           DecodeBufs b, float* out, uint32_t* err, cudaStream_t s);
// Gate/up + down + combine of the resident experts in one launch with a grid-wide
// barrier between them (bf16, one token, up to 8 resident experts, no shared
// expert): can replace launch_gate_up(pass 0) + launch_down_split(pass 0).
bool resident_fused_ok(const Shape& sh, int T, int sms);
cudaError_t launch_resident_fused(const Shape& sh, int T, const void* x, const float* w, const float* cpu_part,
                                  DecodeBufs b, float* out, uint32_t* err, int sms, cudaStream_t s);
int down_combine_launches(const Shape& sh, int T, int sms);   // kernels of launch_down_combine
int gemv_block_threads();

// Programmatic dependent launch: a kernel launched this way may start while its
// predecessor in the stream is still running.  It must call pdl_wait() before
// touching anything the predecessor writes (and always calls it, so that its own
// completion implies the predecessor's), and calls pdl_trigger() only after that
// wait, so the guarantee chains from kernel to kernel.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// pointer alignment the kernels' vector loads and bulk copies assume
inline bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// blob geometry
inline uint64_t blob_bytes(int wdtype, int H, int I) {
  uint64_t HI = (uint64_t)H * (uint64_t)I;
  if (wdtype == MOE_F32) return 12ull * HI;
  if (wdtype == MOE_BF16) return 6ull * HI;
  if (wdtype == MOE_NVFP4) return 3ull * HI / 2 + 3ull * HI / 16 + 16;
  if (wdtype == MOE_MXFP4) return 3ull * HI / 2 + 3ull * HI / 32;
  uint64_t ns = (uint64_t)(2 * I / 128) * (H / 128) + (uint64_t)(H / 128) * (I / 128);
  return 3ull * HI + 4ull * ns;
}

}  // namespace moe
