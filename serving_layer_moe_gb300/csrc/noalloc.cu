// moe_layer_ffn_noalloc: the expert SwiGLU + combine of one MoE layer for
// callers that cannot allocate GPU memory.
//
// Some callers may not call cudaMalloc at all: code that runs inside another
// framework's memory pool or arena, a host that reserved all GPU memory up
// front, or a runtime that forbids allocation after start-up (to keep memory
// use fixed).  For them this entry point takes the caller's inputs and
// outputs and keeps every intermediate (routing lists, per-pair activations
// and outputs) in one file-scope device array of fixed size, so a call
// allocates nothing.
//
// It computes what moe_layer_decode computes when every routed expert of the
// layer is already resident (no cache, no fills, no CPU-assigned pairs): the
// caller hands over the layer's E expert blobs back to back in device memory.
// It reuses the decode GEMV and combine kernels unchanged; only the routing
// step that builds their work lists is new, and it writes those lists into the
// static array instead of into a cache's allocated buffers.
#include "cache.cuh"

#include <mutex>

namespace moe {

namespace {

// Scratch shared by every call of moe_layer_ffn_noalloc on a device.  Every GPU
// that loads this library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
// Routed pairs (T * top_k) of one call, at most: the gate/up kernel stages the
// pair lists in shared memory, and this many always fit what set-up allows it.
constexpr int kNoAllocMaxPairs = 9216;
std::mutex g_setup_mu;
uint8_t* g_scratch_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device
int g_sms[kMaxDevices] = {};

struct NoAllocLayout {
  size_t plan, slot_map, gpu_off, gpu_pairs, gpu_w, err, h, y, total;
};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

NoAllocLayout layout_for(int T, int k, int E, int H, int I) {
  NoAllocLayout l{};
  const size_t pairs = (size_t)T * k;
  const size_t umax = (size_t)(E < T * k ? E : T * k);
  size_t o = 0;
  l.plan = o; o = up256(o + P_COUNT * 4);
  l.slot_map = o; o = up256(o + pairs * 4);
  l.gpu_off = o; o = up256(o + (umax + 1) * 4);
  l.gpu_pairs = o; o = up256(o + pairs * 4);
  l.gpu_w = o; o = up256(o + umax * 8);
  l.err = o; o = up256(o + 4);
  l.h = o; o = up256(o + pairs * (size_t)I * 4);
  l.y = o; o = up256(o + pairs * (size_t)H * 4);
  l.total = o;
  return l;
}

// One CTA: routed experts -> GPU expert list (ascending e), per-expert pair
// lists, weight pointers into the caller's expert blobs, slot map, plan.
// Every field the GEMV and combine read is rewritten here on every call, so
// nothing carries over from the previous call.
__global__ void __launch_bounds__(1024, 1)
noalloc_route_kernel(int T, int k, int E, uint64_t S, const int32_t* __restrict__ ids,
                     const uint8_t* __restrict__ experts, DecodeBufs b, uint32_t* err) {
  __shared__ uint32_t bits[kMaxExperts / 32];
  __shared__ int base[kMaxExperts / 32 + 1];
  __shared__ int cursor[kMaxExperts];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  const int NW = (E + 31) >> 5, P = T * k;
  for (int i = tid; i < NW; i += nt) bits[i] = 0u;
  for (int i = tid; i < E; i += nt) cursor[i] = 0;
  if (tid == 0) *err = 0u;
  __syncthreads();
  for (int p = tid; p < P; p += nt) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E) {
      atomicOr(&bits[e >> 5], 1u << (e & 31));
      atomicAdd(&cursor[e], 1);     // pair count per expert for now
    }
  }
  __syncthreads();
  if (tid < 32) {  // exclusive popcount prefix over the bitmap words
    int running = 0;
    for (int w0 = 0; w0 < NW; w0 += 32) {
      const int w = w0 + lane;
      const int c = w < NW ? __popc(bits[w]) : 0;
      int incl = c;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (w < NW) base[w] = running + incl - c;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) base[NW] = running;
  }
  __syncthreads();
  const int u = base[NW];
  if (tid < 32) {  // pair-list offsets of the GPU experts, in ascending e
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool on = e < E && (bits[e >> 5] & (1u << (e & 31)));
      const int c = on ? cursor[e] : 0;
      int incl = c;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (on) {
        const int g = base[e >> 5] + __popc(bits[e >> 5] & ((1u << (e & 31)) - 1u));
        b.gpu_off[g] = running + incl - c;
        cursor[e] = running + incl - c;
        b.gpu_w[g] = experts + (size_t)e * S;
      }
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) b.gpu_off[u] = running;
  }
  __syncthreads();
  for (int p = tid; p < P; p += nt) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E) {
      b.gpu_pairs[atomicAdd(&cursor[e], 1)] = p;
      b.slot_map[p] = e;
    } else {
      b.slot_map[p] = -1;   // contributes nothing (the combine gets no CPU partial sums)
    }
  }
  if (tid == 0) {
    int32_t* pl = b.plan;
    pl[P_LAYER] = 0; pl[P_U] = u; pl[P_H] = u; pl[P_M] = 0; pl[P_Q] = 0;
    pl[P_NCPU] = 0; pl[P_NGPU] = u; pl[P_NFIRST] = u;
  }
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_layer_ffn_noalloc(int32_t n_experts, int32_t hidden, int32_t inter, int32_t top_k,
                                            int32_t wdtype, int32_t adtype, const void* experts_dev, int32_t T,
                                            const void* x_dev, const int32_t* topk_ids_dev,
                                            const float* topk_w_dev, float* out_dev, void* stream) {
  if (n_experts < 1 || n_experts > kMaxExperts || top_k < 1 || top_k > n_experts)
    return fail(MOE_EINVAL, "need 1 <= E <= %d and 1 <= top_k <= E", kMaxExperts);
  if (wdtype != MOE_F32 && wdtype != MOE_BF16 && wdtype != MOE_FP8E4M3_B128) return fail(MOE_EINVAL, "bad wdtype");
  if (adtype != MOE_F32 && adtype != MOE_BF16) return fail(MOE_EINVAL, "bad adtype");
  if (hidden < 8 || inter < 8 || hidden % 8 || inter % 8)
    return fail(MOE_EINVAL, "H and I must be positive multiples of 8");
  if (wdtype == MOE_FP8E4M3_B128 && (hidden % 128 || inter % 128))
    return fail(MOE_EINVAL, "fp8 block-scaled weights need H and I multiples of 128");
  if (blob_bytes(wdtype, hidden, inter) % 16)   // expert e starts at e * S, read in 16-byte chunks
    return fail(MOE_EINVAL, "blob size S = %llu is not a multiple of 16 bytes (fp8: the scale count "
                "(2I/128)(H/128) + (H/128)(I/128) must be a multiple of 4)",
                (unsigned long long)blob_bytes(wdtype, hidden, inter));
  if (T < 0) return fail(MOE_EINVAL, "T must be >= 0");
  if (T == 0) return MOE_OK;
  if (!experts_dev || !x_dev || !topk_ids_dev || !topk_w_dev || !out_dev)
    return fail(MOE_EINVAL, "experts, x, topk_ids, topk_w and out must not be NULL");
  if (reinterpret_cast<uintptr_t>(experts_dev) % 16) return fail(MOE_EINVAL, "experts_dev must be 16-byte aligned");
  if (!aligned_to(x_dev, 16) || !aligned_to(out_dev, 16)) return fail(MOE_EINVAL, "x and out must be 16-byte aligned");
  if (!aligned_to(topk_ids_dev, 4) || !aligned_to(topk_w_dev, 4))
    return fail(MOE_EINVAL, "topk_ids and topk_w must be 4-byte aligned");
  const NoAllocLayout lay = layout_for(T, top_k, n_experts, hidden, inter);
  if (lay.total > kNoAllocScratchBytes)
    return fail(MOE_ECAPACITY, "T * top_k * (H + I) needs %zu bytes of scratch; the fixed scratch holds %zu",
                lay.total, kNoAllocScratchBytes);
  if ((int64_t)T * top_k > kNoAllocMaxPairs)
    return fail(MOE_ECAPACITY, "T * top_k = %lld routed pairs; one call takes at most %d",
                (long long)T * top_k, kNoAllocMaxPairs);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(MOE_ECUDA, "no current CUDA device (or ordinal >= %d)", kMaxDevices);
  uint8_t* scratch = nullptr;
  int sms = 0;
  {
    // first call on this device: let the GEMV kernels use the shared memory they
    // stage into (a process may call this without ever creating a cache), then
    // look up the device address of the static array
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
      const cudaError_t ke = setup_gemv_kernels();
      if (ke != cudaSuccess) {
        cudaGetLastError();
        return fail(MOE_ECUDA, "setting up the GEMV kernels: %s", cudaGetErrorString(ke));
      }
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return fail(MOE_ECUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
      }
      int n = 0;
      if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return fail(MOE_ECUDA, "cannot read the SM count of device %d", dev);
      }
      g_sms[dev] = n;
      g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
    }
    scratch = g_scratch_ptr[dev];
    sms = g_sms[dev];
  }

  Shape sh{};
  sh.L = 1; sh.E = n_experts; sh.H = hidden; sh.I = inter; sh.k = top_k;
  sh.wdtype = wdtype; sh.adtype = adtype; sh.n_shared = 0;
  sh.S = blob_bytes(wdtype, hidden, inter);
  if (expert_gemv_smem(sh, T) > expert_gemv_smem_limit())   // not reached within kNoAllocMaxPairs
    return fail(MOE_ECAPACITY, "the call's pair lists need %zu bytes of shared memory; at most %zu",
                expert_gemv_smem(sh, T), expert_gemv_smem_limit());
  DecodeBufs b{};
  b.plan = reinterpret_cast<int32_t*>(scratch + lay.plan);
  b.slot_map = reinterpret_cast<int32_t*>(scratch + lay.slot_map);
  b.gpu_off = reinterpret_cast<int32_t*>(scratch + lay.gpu_off);
  b.gpu_pairs = reinterpret_cast<int32_t*>(scratch + lay.gpu_pairs);
  b.gpu_w = reinterpret_cast<const uint8_t**>(scratch + lay.gpu_w);
  b.h = reinterpret_cast<float*>(scratch + lay.h);
  b.y = reinterpret_cast<float*>(scratch + lay.y);
  uint32_t* err = reinterpret_cast<uint32_t*>(scratch + lay.err);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  noalloc_route_kernel<<<1, 1024, 0, s>>>(T, top_k, n_experts, sh.S, topk_ids_dev,
                                          static_cast<const uint8_t*>(experts_dev), b, err);
  CK(cudaGetLastError());
  CK(launch_expert_gemv(sh, 0, T, x_dev, b, sms, s));
  CK(launch_combine(sh, T, topk_w_dev, nullptr, b, out_dev, err, s));
  return MOE_OK;
}
