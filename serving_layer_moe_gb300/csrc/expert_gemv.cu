// Decode-side expert work: the slot fill copy, the grouped SwiGLU GEMV over
// resident slots, and the fixed-order combine.
//
// Follows the snackonai deep dive "FreeToken, or why your laptop was never the
// bottleneck", section "The split policy itself" (closing note: on the GPU
// side a miss means updating the cache, copying the experts in as a batch and
// evaluating them grouped) and section "What It Actually Does" (the GPU and CPU
// partial sums are merged without approximation); the
// dev.to summary "FreeToken runs frontier-scale MoE models ...", section "When
// it misses": RAM -> link -> VRAM -> GPU execute.
//
// Expert (not written out on the pages; the SwiGLU of the Qwen3 / DeepSeek-V3
// MoE families): h = silu(W_gate x) * (W_up x) in fp32, y = W_down h in fp32.
//
// GB300 design: decode is a matrix-vector product per expert (a handful of
// tokens per expert), so it is bound by HBM bandwidth, not by tensor cores.
//   * Resident experts: gate_up_bulk_kernel gives every warp a ring of
//     shared-memory stages that cp.async.bulk fills with whole gate/up row
//     pairs (mbarrier completion), so each SM keeps ~200 KB of weights in
//     flight while the warp computes from the previous stage; it also has L2
//     fetch the same experts' W_down.  down_bulk_kernel then streams W_down
//     row blocks the same way, one wave of CTAs with R = ceil(H / SMs) rows
//     each, and fuses the fixed-order combine.
//   * Filled experts: fill_gate_up_kernel copies each blob from page-locked
//     host memory (an SM copy over NVLink-C2C, since the fill list is decided
//     on the device) and computes gate/up on the rows as they pass; a second
//     down grid on the fill stream takes those experts.  The resident and
//     filled-expert down grids count their arrivals per row block, and the
//     second to arrive combines.
//   * Each pair's y is formed in the same per-lane order and reduction tree on
//     the ring, no-ring and fused paths, so it is the same bit for bit whichever
//     of those grids computes it.
//   * Register-staged gate_up_kernel / down_kernel / down_combine_kernel take
//     the calls whose x (gate/up) or ring (down) does not fit in shared memory.
//   * Launch shapes depend only on the cache's shape, never on the plan (the
//     control kernel publishes it in device memory), so a decode step can be
//     captured in a CUDA graph.
#include <vector>

#include "internal.cuh"

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>

#include <algorithm>

namespace moe {

namespace {

constexpr int kGemvThreads = 512;
constexpr int kChunksPerLane = 4;

// ---- weight formats: one 16-byte chunk -> V floats ---------------------------
template <int WT> struct WFmt;
// row(n): bytes of n elements; sgu_off / sd_off / g_off: offsets of the scale
// arrays (and NVFP4's matrix scales) inside a blob of the format
template <> struct WFmt<MOE_F32> {
  static constexpr int V = 4;
  __host__ __device__ static constexpr size_t row(size_t n) { return n * 4; }
  __host__ __device__ static constexpr size_t sd_off(size_t, size_t) { return 0; }
  __device__ static void unpack(const uint4& w, float* f) {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
  }
};
template <> struct WFmt<MOE_BF16> {
  static constexpr int V = 8;
  __host__ __device__ static constexpr size_t row(size_t n) { return n * 2; }
  __host__ __device__ static constexpr size_t sd_off(size_t, size_t) { return 0; }
  __device__ static void unpack(const uint4& w, float* f) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(v[i] << 16);
      f[2 * i + 1] = __uint_as_float(v[i] & 0xffff0000u);
    }
  }
};
template <> struct WFmt<MOE_FP8E4M3_B128> {
  static constexpr int V = 16;
  __host__ __device__ static constexpr size_t row(size_t n) { return n; }
  __host__ __device__ static constexpr size_t sd_off(size_t H, size_t I) {
    return 3 * I * H + 4 * (2 * I / 128) * (H / 128);
  }
  __device__ static void unpack(const uint4& w, float* f) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v[i] & 0xffffu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v[i] >> 16), __NV_E4M3);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      f[4 * i] = a.x; f[4 * i + 1] = a.y; f[4 * i + 2] = b.x; f[4 * i + 3] = b.y;
    }
  }
};

// The e2m1 code layout of the two 4-bit formats: 32 values per 16-byte chunk,
// element 2j from the low nibble of byte j.
struct E2M1Codes {
  static constexpr int V = 32;   // two elements per byte
  __host__ __device__ static constexpr size_t row(size_t n) { return n / 2; }
  __device__ static void unpack(const uint4& w, float* f) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((v[i] >> (8 * b)) & 0xffu), __NV_E2M1);
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&h));
        f[8 * i + 2 * b] = p.x;
        f[8 * i + 2 * b + 1] = p.y;
      }
  }
};

// NVFP4: one e4m3 scale per 16 row elements, one fp32 scale per matrix (g_off).
template <> struct WFmt<MOE_NVFP4> : E2M1Codes {
  using scale_t = uint16_t;   // the two e4m3 block scales of one 32-value chunk
  __host__ __device__ static constexpr size_t sgu_off(size_t H, size_t I) { return 3 * I * H / 2; }
  __host__ __device__ static constexpr size_t sd_off(size_t H, size_t I) { return 3 * I * H / 2 + 2 * I * H / 16; }
  __host__ __device__ static constexpr size_t g_off(size_t H, size_t I) { return sd_off(H, I) + H * I / 16; }
  // One chunk (two 16-element blocks; s2 = their e4m3 scale codes, the first
  // block's in the low byte) against 32 activations: (sum of the first 16
  // products) * scale_0 + (sum of the last 16) * scale_1.  Every NVFP4 path
  // uses this, so a row's value does not depend on the kernel.
  __device__ static __forceinline__ float dot(const uint4& w, uint32_t s2, const float* x) {
    float f[32];
    unpack(w, f);
    float lo = 0.f, hi = 0.f;
#pragma unroll
    for (int v = 0; v < 16; ++v) lo = fmaf(f[v], x[v], lo);
#pragma unroll
    for (int v = 0; v < 16; ++v) hi = fmaf(f[16 + v], x[16 + v], hi);
    const __half2_raw sr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(s2 & 0xffffu), __NV_E4M3);
    const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&sr));
    return fmaf(hi, sf.y, lo * sf.x);
  }
  // the chunk's 32 weights: e2m1 * block scale * g (g = the matrix's fp32 scale)
  __device__ static __forceinline__ void decode32(const uint4& w, uint32_t s2, float g, float* f) {
    unpack(w, f);
    const __half2_raw sr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(s2 & 0xffffu), __NV_E4M3);
    const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&sr));
    const float a = sf.x * g, b = sf.y * g;
#pragma unroll
    for (int v = 0; v < 16; ++v) { f[v] *= a; f[16 + v] *= b; }
  }
};

// OCP MX E8M0 scale: 2^(code - 127), code 255 NaN.  Codes 1..254 are the fp32
// exponent field itself; code 0 (2^-127) is the fp32 subnormal 0x00400000.
__device__ __forceinline__ float e8m0_to_f32(uint32_t code) {
  return code == 0 ? __uint_as_float(0x00400000u) : code == 255 ? __uint_as_float(0x7fc00000u) : __uint_as_float(code << 23);
}

// MXFP4 (OCP Microscaling): one e8m0 scale per 32 row elements, i.e. per chunk;
// no matrix scale.
template <> struct WFmt<MOE_MXFP4> : E2M1Codes {
  using scale_t = uint8_t;    // the chunk's e8m0 block scale
  __host__ __device__ static constexpr size_t sgu_off(size_t H, size_t I) { return 3 * I * H / 2; }
  __host__ __device__ static constexpr size_t sd_off(size_t H, size_t I) { return 3 * I * H / 2 + 2 * I * H / 32; }
  // One chunk against 32 activations: (two 16-product partial sums, added) * scale.
  __device__ static __forceinline__ float dot(const uint4& w, uint32_t s, const float* x) {
    float f[32];
    unpack(w, f);
    float lo = 0.f, hi = 0.f;
#pragma unroll
    for (int v = 0; v < 16; ++v) lo = fmaf(f[v], x[v], lo);
#pragma unroll
    for (int v = 0; v < 16; ++v) hi = fmaf(f[16 + v], x[16 + v], hi);
    return (lo + hi) * e8m0_to_f32(s & 0xffu);
  }
  // the chunk's 32 weights: e2m1 * 2^(scale - 127), exact in fp32 and in bf16
  __device__ static __forceinline__ void decode32(const uint4& w, uint32_t s, float, float* f) {
    unpack(w, f);
    const float sc = e8m0_to_f32(s & 0xffu);
#pragma unroll
    for (int v = 0; v < 32; ++v) f[v] *= sc;
  }
};

template <int WT> constexpr bool kFp4 = WT == MOE_NVFP4 || WT == MOE_MXFP4;

// ---- activations: V consecutive values as floats --------------------------
template <int AT, int V> __device__ __forceinline__ void load_act(const void* x, size_t off, float* f);
template <int V> __device__ __forceinline__ void load_act_f32(const float* p, float* f) {
#pragma unroll
  for (int i = 0; i < V; i += 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p + i));
    f[i] = v.x; f[i + 1] = v.y; f[i + 2] = v.z; f[i + 3] = v.w;
  }
}
template <> __device__ __forceinline__ void load_act<MOE_F32, 4>(const void* x, size_t off, float* f) {
  load_act_f32<4>(reinterpret_cast<const float*>(x) + off, f);
}
template <> __device__ __forceinline__ void load_act<MOE_F32, 8>(const void* x, size_t off, float* f) {
  load_act_f32<8>(reinterpret_cast<const float*>(x) + off, f);
}
template <> __device__ __forceinline__ void load_act<MOE_F32, 16>(const void* x, size_t off, float* f) {
  load_act_f32<16>(reinterpret_cast<const float*>(x) + off, f);
}
template <> __device__ __forceinline__ void load_act<MOE_F32, 32>(const void* x, size_t off, float* f) {
  load_act_f32<32>(reinterpret_cast<const float*>(x) + off, f);
}
template <int V> __device__ __forceinline__ void load_act_bf16(const uint16_t* p, float* f) {
#pragma unroll
  for (int i = 0; i < V; i += 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p + i));
    WFmt<MOE_BF16>::unpack(v, f + i);
  }
}
template <> __device__ __forceinline__ void load_act<MOE_BF16, 8>(const void* x, size_t off, float* f) {
  load_act_bf16<8>(reinterpret_cast<const uint16_t*>(x) + off, f);
}
template <> __device__ __forceinline__ void load_act<MOE_BF16, 16>(const void* x, size_t off, float* f) {
  load_act_bf16<16>(reinterpret_cast<const uint16_t*>(x) + off, f);
}
template <> __device__ __forceinline__ void load_act<MOE_BF16, 32>(const void* x, size_t off, float* f) {
  load_act_bf16<32>(reinterpret_cast<const uint16_t*>(x) + off, f);
}
template <> __device__ __forceinline__ void load_act<MOE_BF16, 4>(const void* x, size_t off, float* f) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(x) + off));
  f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
}

// Weights are read once per step: stream them past L1 and mark them first to
// leave L2, so the kernels' code, the residency tables and the activations
// stay cached between layers.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ld_stream(const uint4* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// acc + w.lo * x.lo, then + w.hi * x.hi, on bf16 pairs with an f32 accumulator:
// the products of two bf16 values are exact in f32, so each step rounds once,
// exactly like fmaf on the widened operands.
__device__ __forceinline__ float fma_bf16x2(uint32_t w, uint32_t x, float acc) {
  asm("{\n .reg .b16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %1;\n mov.b32 {xl, xh}, %2;\n"
      " fma.rn.f32.bf16 %0, wl, xl, %0;\n fma.rn.f32.bf16 %0, wh, xh, %0;\n}"
      : "+f"(acc) : "r"(w), "r"(x));
  return acc;
}

struct GemvArgs {
  int H, I, k, T, P;             // P = T * k (pair ids >= P are shared-expert rows)
  int pass;                      // 0: hits + shared, 1: fills, 2: every GPU expert
  int n_shared;
  int max_g, max_p;              // bounds of the GPU-expert and pair lists of this call
  int x_smem;                    // stage x in shared memory
  const void* x;
  DecodeBufs b;
};

// The plan the control kernel published, staged once per CTA in shared memory:
// weight pointer and pair-list offsets of every GPU expert, pair ids and their
// tokens.  One parallel round trip instead of a chain of dependent global reads
// per expert.
struct StagedPlan {
  const uint8_t** w;   // [max_g]
  int* off;            // [max_g + 1]
  int* pid;            // [max_p]
  int* tok;            // [max_p]
  size_t bytes;
};

__host__ __device__ inline size_t staged_plan_bytes(int max_g, int max_p) {
  return ((size_t)max_g * 8 + (size_t)(max_g + 1) * 4 + (size_t)max_p * 8 + 15) & ~size_t(15);
}

__device__ __forceinline__ StagedPlan stage_plan(uint8_t* smem, const GemvArgs& a) {
  StagedPlan sp;
  sp.w = reinterpret_cast<const uint8_t**>(smem);
  sp.off = reinterpret_cast<int*>(sp.w + a.max_g);
  sp.pid = sp.off + a.max_g + 1;
  sp.tok = sp.pid + a.max_p;
  sp.bytes = staged_plan_bytes(a.max_g, a.max_p);
  for (int i = threadIdx.x; i < a.max_g; i += blockDim.x) sp.w[i] = a.b.gpu_w[i];
  for (int i = threadIdx.x; i <= a.max_g; i += blockDim.x) sp.off[i] = a.b.gpu_off[i];
  for (int i = threadIdx.x; i < a.max_p; i += blockDim.x) {
    const int p = a.b.gpu_pairs[i];
    sp.pid[i] = p;
    sp.tok[i] = p < a.P ? p / a.k : p - a.P;
  }
  return sp;
}

// x values from shared or global memory (generic loads)
template <int AT, int V> __device__ __forceinline__ void load_x(const void* x, size_t off, float* f) {
  if (AT == MOE_F32) {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + off);
#pragma unroll
    for (int i = 0; i < V / 4; ++i) {
      const float4 v = p[i];
      f[4 * i] = v.x; f[4 * i + 1] = v.y; f[4 * i + 2] = v.z; f[4 * i + 3] = v.w;
    }
  } else if (V >= 8) {
    const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(x) + off);
#pragma unroll
    for (int i = 0; i < V / 8; ++i) WFmt<MOE_BF16>::unpack(p[i], f + 8 * i);
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(x) + off);
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
  }
}

__device__ __forceinline__ void pass_range(const GemvArgs& a, int& g0, int& g1) {
  const int* plan = a.b.plan;
  g0 = a.pass == 1 ? plan[P_NFIRST] : 0;
  g1 = a.pass == 0 ? plan[P_NFIRST] : plan[P_NGPU];
}

__device__ __forceinline__ int token_of(int pid, int k, int P) { return pid < P ? pid / k : pid - P; }

// ---- phase 1: h[pair, i] = silu(gate_i . x_t) * (up_i . x_t) ------------------
template <int WT, int AT, int kTokGroup>
__global__ void __launch_bounds__(kGemvThreads, kTokGroup == 1 ? 2 : 1) gate_up_kernel(GemvArgs a) {
  using F = WFmt<WT>;
  constexpr int V = F::V;
  extern __shared__ __align__(16) uint8_t gsm[];
  pdl_wait();
  pdl_trigger();
  const StagedPlan sp = stage_plan(gsm, a);
  const int H = a.H, I = a.I;
  const void* xs = a.x;
  if (a.x_smem) {   // stage x [T, H] next to the plan
    uint4* dst = reinterpret_cast<uint4*>(gsm + sp.bytes);
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    const int n16 = (int)(((size_t)a.T * H * (AT == MOE_F32 ? 4 : 2)) >> 4);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
    xs = dst;
  }
  int g0, g1;
  pass_range(a, g0, g1);
  __syncthreads();
  const long rows = (long)(g1 - g0) * I;
  const int lane = threadIdx.x & 31;
  const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  const long wid = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int NCH = H / V;                       // 16-byte chunks per row
  const size_t row_bytes = F::row(H);
  const int HB = H / 128;                      // fp8 scale columns
  const uint64_t pol = evict_first_policy();

  for (long r = wid; r < rows; r += nwarps) {
    const int g = g0 + (int)(r / I);
    const int i = (int)(r % I);
    const uint8_t* wb = sp.w[g];
    const uint4* gate = reinterpret_cast<const uint4*>(wb + (size_t)i * row_bytes);
    const uint4* up = reinterpret_cast<const uint4*>(wb + (size_t)(I + i) * row_bytes);
    const float* sgu = reinterpret_cast<const float*>(wb + 3ull * (size_t)I * row_bytes);
    const int pb = sp.off[g], pe = sp.off[g + 1];
    for (int tp = pb; tp < pe; tp += kTokGroup) {
      const int nt = min(kTokGroup, pe - tp);
      int tok[kTokGroup];
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) tok[n] = n < nt ? sp.tok[tp + n] : 0;
      float ag[kTokGroup], au[kTokGroup];
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) { ag[n] = 0.f; au[n] = 0.f; }
      for (int seg = 0; seg < NCH; seg += 32 * kChunksPerLane) {
        uint4 wg[kChunksPerLane], wu[kChunksPerLane];
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j) {
          const int c = seg + j * 32 + lane;
          if (c < NCH) { wg[j] = ld_stream(gate + c, pol); wu[j] = ld_stream(up + c, pol); }
        }
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j) {
          const int c = seg + j * 32 + lane;
          if (c < NCH) {
            if constexpr (kFp4<WT>) {   // the chunk dot product of every 4-bit path, with its block scales
              const auto* srow = reinterpret_cast<const typename F::scale_t*>(wb + F::sgu_off(H, I));
              const uint32_t s2g = __ldg(srow + (size_t)i * (H / 32) + c);
              const uint32_t s2u = __ldg(srow + (size_t)(I + i) * (H / 32) + c);
#pragma unroll
              for (int n = 0; n < kTokGroup; ++n) {
                if (n < nt) {
                  float xv[V];
                  load_x<AT, V>(xs, (size_t)tok[n] * H + (size_t)c * V, xv);
                  ag[n] += F::dot(wg[j], s2g, xv);
                  au[n] += F::dot(wu[j], s2u, xv);
                }
              }
            } else {
              float fg[V], fu[V];
              F::unpack(wg[j], fg);
              F::unpack(wu[j], fu);
              float scg = 1.f, scu = 1.f;
              if (WT == MOE_FP8E4M3_B128) {
                const int cb = (c * V) >> 7;
                scg = __ldg(sgu + (size_t)(i >> 7) * HB + cb);
                scu = __ldg(sgu + (size_t)((I + i) >> 7) * HB + cb);
              }
#pragma unroll
              for (int n = 0; n < kTokGroup; ++n) {
                if (n < nt) {
                  float xv[V];
                  load_x<AT, V>(xs, (size_t)tok[n] * H + (size_t)c * V, xv);
                  float dg = 0.f, du = 0.f;
#pragma unroll
                  for (int v = 0; v < V; ++v) { dg = fmaf(fg[v], xv[v], dg); du = fmaf(fu[v], xv[v], du); }
                  ag[n] = fmaf(dg, scg, ag[n]);
                  au[n] = fmaf(du, scu, au[n]);
                }
              }
            }
          }
        }
      }
      float gg = 1.f;
      if constexpr (WT == MOE_NVFP4) gg = __ldg(reinterpret_cast<const float*>(wb + F::g_off(H, I)));   // W_gu's scale
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) {
        if (n < nt) {
          float sg = warp_sum(ag[n]);
          float su = warp_sum(au[n]);
          if constexpr (WT == MOE_NVFP4) { sg *= gg; su *= gg; }
          if (lane == 0) a.b.h[(size_t)sp.pid[tp + n] * I + i] = silu(sg) * su;
        }
      }
    }
  }
}

// ---- fill fused with the gate/up GEMV of the filled experts -----------------------
// The fill path of decode.  For each filled expert (flat id f -> victim slot s):
// every gate/up row pair is streamed from page-locked host memory over the host
// link, written into the slot, and dotted with the expert's tokens on the way
// through (h of its pairs, like gate_up_kernel); the rest of the blob (W_down
// and, for fp8, the scales) is copied in 4 KB pieces with default stores, so the
// down projection that follows finds them in L2.  The bytes cross the link
// once and the filled experts need no separate gate/up pass.
constexpr int kFillThreads = 256;   // small CTAs: they share SMs with the resident-expert GEMV

template <int WT, int AT, int kTokGroup>
__global__ void __launch_bounds__(kFillThreads, 2)
fill_gate_up_kernel(GemvArgs a, const int32_t* __restrict__ fills, const uint8_t* __restrict__ host,
                    const uint64_t* __restrict__ offs, uint8_t* __restrict__ slots, uint64_t S) {
  using F = WFmt<WT>;
  constexpr int V = F::V;
  pdl_trigger();   // the filled-expert down grid may stage its plan meanwhile; it waits for this grid to finish
  const int* plan = a.b.plan;
  const int q = plan[P_Q];
  if (q == 0) return;
  const int nfirst = plan[P_NFIRST];
  const int H = a.H, I = a.I;
  const int lane = threadIdx.x & 31;
  const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  const long wid = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int NCH = H / V;
  const size_t row_bytes = F::row(H);
  const int HB = H / 128;
  const size_t down_off = 2ull * (size_t)I * row_bytes;
  const uint64_t tail16 = (S - down_off) >> 4;             // 16-byte chunks after W_gu
  constexpr int kPiece = 256;                               // 16-byte chunks per copy item (4 KB)
  const long pieces = (long)((tail16 + kPiece - 1) / kPiece);
  const long row_items = (long)q * I;
  const long items = row_items + (long)q * pieces;

  for (long it = wid; it < items; it += nwarps) {
    if (it >= row_items) {  // plain copy of a piece of W_down (+ scales)
      const long k = it - row_items;
      const int fi = (int)(k / pieces);
      const uint64_t c0 = (uint64_t)(k % pieces) * kPiece;
      const uint4* src = reinterpret_cast<const uint4*>(host + offs[fills[2 * fi]] + down_off);
      uint4* dst = reinterpret_cast<uint4*>(slots + (size_t)fills[2 * fi + 1] * S + down_off);
      const uint64_t c1 = min(tail16, c0 + kPiece);
      uint4 v[kPiece / 32];
#pragma unroll
      for (int j = 0; j < kPiece / 32; ++j) {
        const uint64_t c = c0 + (uint64_t)j * 32 + lane;
        if (c < c1) v[j] = src[c];
      }
#pragma unroll
      for (int j = 0; j < kPiece / 32; ++j) {
        const uint64_t c = c0 + (uint64_t)j * 32 + lane;
        if (c < c1) dst[c] = v[j];   // default policy: the down projection reads these next, from L2
      }
      continue;
    }
    const int fi = (int)(it / I);
    const int i = (int)(it % I);
    const int g = nfirst + fi;
    const uint8_t* sb = host + offs[fills[2 * fi]];
    uint8_t* db = slots + (size_t)fills[2 * fi + 1] * S;
    const uint4* gate = reinterpret_cast<const uint4*>(sb + (size_t)i * row_bytes);
    const uint4* up = reinterpret_cast<const uint4*>(sb + (size_t)(I + i) * row_bytes);
    uint4* dgate = reinterpret_cast<uint4*>(db + (size_t)i * row_bytes);
    uint4* dup = reinterpret_cast<uint4*>(db + (size_t)(I + i) * row_bytes);
    const float* sgu = reinterpret_cast<const float*>(sb + 3ull * (size_t)I * row_bytes);
    const int pb = a.b.gpu_off[g], pe = a.b.gpu_off[g + 1];
    int tok[kTokGroup];
    float ag[kTokGroup], au[kTokGroup];
    for (int tp = pb; tp < pe || tp == pb; tp += kTokGroup) {
      const int nt = max(0, min(kTokGroup, pe - tp));
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) {
        tok[n] = n < nt ? token_of(a.b.gpu_pairs[tp + n], a.k, a.P) : 0;
        ag[n] = 0.f;
        au[n] = 0.f;
      }
      for (int seg = 0; seg < NCH; seg += 32 * kChunksPerLane) {
        uint4 wg[kChunksPerLane], wu[kChunksPerLane];
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j) {
          const int c = seg + j * 32 + lane;
          if (c < NCH) { wg[j] = gate[c]; wu[j] = up[c]; }
        }
        if (tp == pb) {   // the first token group writes the rows into the slot
#pragma unroll
          for (int j = 0; j < kChunksPerLane; ++j) {
            const int c = seg + j * 32 + lane;
            if (c < NCH) { __stcs(dgate + c, wg[j]); __stcs(dup + c, wu[j]); }
          }
        }
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j) {
          const int c = seg + j * 32 + lane;
          if (c < NCH) {
            if constexpr (kFp4<WT>) {   // scales straight from the host blob
              const auto* srow = reinterpret_cast<const typename F::scale_t*>(sb + F::sgu_off(H, I));
              const uint32_t sg2 = srow[(size_t)i * (H / 32) + c], su2 = srow[(size_t)(I + i) * (H / 32) + c];
#pragma unroll
              for (int n = 0; n < kTokGroup; ++n) {
                if (n < nt) {
                  float xv[V];
                  load_act<AT, V>(a.x, (size_t)tok[n] * H + (size_t)c * V, xv);
                  ag[n] += F::dot(wg[j], sg2, xv);
                  au[n] += F::dot(wu[j], su2, xv);
                }
              }
            } else {
              float fg[V], fu[V];
              F::unpack(wg[j], fg);
              F::unpack(wu[j], fu);
              float scg = 1.f, scu = 1.f;
              if (WT == MOE_FP8E4M3_B128) {
                const int cb = (c * V) >> 7;
                scg = sgu[(size_t)(i >> 7) * HB + cb];
                scu = sgu[(size_t)((I + i) >> 7) * HB + cb];
              }
#pragma unroll
              for (int n = 0; n < kTokGroup; ++n) {
                if (n < nt) {
                  float xv[V];
                  load_act<AT, V>(a.x, (size_t)tok[n] * H + (size_t)c * V, xv);
                  float dg = 0.f, du = 0.f;
#pragma unroll
                  for (int v = 0; v < V; ++v) { dg = fmaf(fg[v], xv[v], dg); du = fmaf(fu[v], xv[v], du); }
                  ag[n] = fmaf(dg, scg, ag[n]);
                  au[n] = fmaf(du, scu, au[n]);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) {
        if (n < nt) {
          float sg = warp_sum(ag[n]);
          float su = warp_sum(au[n]);
          if constexpr (WT == MOE_NVFP4) {
            const float gg = *reinterpret_cast<const float*>(sb + F::g_off(H, I));
            sg *= gg;
            su *= gg;
          }
          if (lane == 0) a.b.h[(size_t)a.b.gpu_pairs[tp + n] * I + i] = silu(sg) * su;
        }
      }
      if (pe <= pb) break;
    }
  }
}

// ---- phase 2: y[pair, r] = down_r . h[pair] ------------------------------------
template <int WT, int kTokGroup>
__global__ void __launch_bounds__(kGemvThreads, kTokGroup == 1 ? 2 : 1) down_kernel(GemvArgs a) {
  using F = WFmt<WT>;
  constexpr int V = F::V;
  int g0, g1;
  pass_range(a, g0, g1);
  const int H = a.H, I = a.I;
  const long rows = (long)(g1 - g0) * H;
  const int lane = threadIdx.x & 31;
  const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  const long wid = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int NCH = I / V;
  const size_t row_bytes = F::row(I);
  const size_t down_off = 2ull * (size_t)I * F::row(H);
  const size_t sd_off = F::sd_off(H, I);
  const int IB = I / 128;
  const uint64_t pol = evict_first_policy();

  for (long r = wid; r < rows; r += nwarps) {
    const int g = g0 + (int)(r / H);
    const int row = (int)(r % H);
    const uint8_t* wb = a.b.gpu_w[g];
    const uint4* wrow = reinterpret_cast<const uint4*>(wb + down_off + (size_t)row * row_bytes);
    const float* sd = reinterpret_cast<const float*>(wb + sd_off);
    const int pb = a.b.gpu_off[g], pe = a.b.gpu_off[g + 1];
    for (int tp = pb; tp < pe; tp += kTokGroup) {
      const int nt = min(kTokGroup, pe - tp);
      int pid[kTokGroup];
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) pid[n] = n < nt ? a.b.gpu_pairs[tp + n] : 0;
      float acc[kTokGroup];
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) acc[n] = 0.f;
      for (int seg = 0; seg < NCH; seg += 32 * kChunksPerLane) {
        uint4 w[kChunksPerLane];
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j) {
          const int c = seg + j * 32 + lane;
          if (c < NCH) w[j] = ld_stream(wrow + c, pol);
        }
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j) {
          const int c = seg + j * 32 + lane;
          if (c < NCH) {
            if constexpr (kFp4<WT>) {   // the chunk dot product of every 4-bit path, with its block scales
              const auto* srow = reinterpret_cast<const typename F::scale_t*>(wb + sd_off);
              const uint32_t s2 = __ldg(srow + (size_t)row * (I / 32) + c);
#pragma unroll
              for (int n = 0; n < kTokGroup; ++n) {
                if (n < nt) {
                  float hv[V];
                  load_act_f32<V>(a.b.h + (size_t)pid[n] * I + (size_t)c * V, hv);
                  acc[n] += F::dot(w[j], s2, hv);
                }
              }
            } else {
              float fw[V];
              F::unpack(w[j], fw);
              float sc = 1.f;
              if (WT == MOE_FP8E4M3_B128) sc = __ldg(sd + (size_t)(row >> 7) * IB + ((c * V) >> 7));
#pragma unroll
              for (int n = 0; n < kTokGroup; ++n) {
                if (n < nt) {
                  float hv[V];
                  load_act_f32<V>(a.b.h + (size_t)pid[n] * I + (size_t)c * V, hv);
                  float d = 0.f;
#pragma unroll
                  for (int v = 0; v < V; ++v) d = fmaf(fw[v], hv[v], d);
                  acc[n] = fmaf(d, sc, acc[n]);
                }
              }
            }
          }
        }
      }
      float gd = 1.f;
      if constexpr (WT == MOE_NVFP4) gd = __ldg(reinterpret_cast<const float*>(wb + F::g_off(H, I)) + 1);   // W_d's scale
#pragma unroll
      for (int n = 0; n < kTokGroup; ++n) {
        if (n < nt) {
          float s = warp_sum(acc[n]);
          if constexpr (WT == MOE_NVFP4) s *= gd;
          if (lane == 0) a.b.y[(size_t)pid[n] * H + row] = s;
        }
      }
    }
  }
}

// ---- down projection fused with the combine -------------------------------------
// One warp per output row r: it streams row r of every GPU expert's W_down
// (kDCGroup experts' rows in flight at once), dots it with the h of each of the
// expert's pairs into a per-warp shared buffer y[pair], then forms
// out[t, r] = sum_j w[t,j] * (slot >= 0 ? y[t,j] : cpu_part[t,j,r]) in j order,
// plus the shared expert.  The h of every pair is staged once per CTA in shared
// memory when it fits (the first expert group's weight loads are already in
// flight meanwhile), so no dot product waits on a second global round trip.
// Used when all pairs fit the per-warp buffer and a down row fits one pass of
// kDCChunks 16-byte chunks per lane.
constexpr int kDCWarps = 8;
constexpr int kDCGroup = 4;
constexpr int kDCChunks = 4;
constexpr int kDCMaxPairs = 1024;
constexpr size_t kDCHSmem = 96 * 1024;    // h staged in shared memory up to this size

template <int WT>
__global__ void __launch_bounds__(kDCWarps * 32) down_combine_kernel(GemvArgs a, const float* __restrict__ w,
                                                                     const float* __restrict__ cpu,
                                                                     float* __restrict__ out, uint32_t* err) {
  using F = WFmt<WT>;
  constexpr int V = F::V;
  extern __shared__ __align__(16) uint8_t dsm8[];
  pdl_wait();
  pdl_trigger();
  const StagedPlan sp = stage_plan(dsm8, a);
  int* s_slot = reinterpret_cast<int*>(dsm8 + sp.bytes);                  // [P] slot map
  float* s_wt = reinterpret_cast<float*>(s_slot + a.P);                   // [P] gates
  for (int i = threadIdx.x; i < a.P; i += blockDim.x) { s_slot[i] = a.b.slot_map[i]; s_wt[i] = w[i]; }
  float* dsm = reinterpret_cast<float*>(dsm8 + sp.bytes + (((size_t)a.P * 8 + 15) & ~size_t(15)));
  const int NP = a.P + a.T * a.n_shared;
  const int H = a.H, I = a.I;
  const bool h_smem = (size_t)NP * I * sizeof(float) <= kDCHSmem;
  float* hs = dsm;                                            // [NP, I] if staged
  float* ys = dsm + (h_smem ? (size_t)NP * I : 0) + (threadIdx.x >> 5) * NP;
  const float* hsrc = h_smem ? hs : a.b.h;
  const int lane = threadIdx.x & 31;
  const int ngpu = a.b.plan[P_NGPU];
  __syncthreads();   // staged plan visible
  const int NCH = I / V;
  const size_t row_bytes = F::row(I);
  const size_t down_off = 2ull * (size_t)I * F::row(H);
  const size_t sd_off = F::sd_off(H, I);
  const int IB = I / 128;
  const int nwarps = gridDim.x * kDCWarps;
  const uint64_t pol = evict_first_policy();
  bool missing = false;

  int r = blockIdx.x * kDCWarps + (threadIdx.x >> 5);
  uint4 wv[kDCGroup][kDCChunks];
  auto load_group = [&](int row, int g0) {
#pragma unroll
    for (int gi = 0; gi < kDCGroup; ++gi) {
      if (g0 + gi < ngpu) {
        const uint4* wrow = reinterpret_cast<const uint4*>(sp.w[g0 + gi] + down_off + (size_t)row * row_bytes);
#pragma unroll
        for (int j = 0; j < kDCChunks; ++j) {
          const int c = j * 32 + lane;
          if (c < NCH) wv[gi][j] = ld_stream(wrow + c, pol);
        }
      }
    }
  };
  if (r < H) load_group(r, 0);
  if (h_smem) {   // stage every pair's h while the first weight rows are in flight
    const float4* src = reinterpret_cast<const float4*>(a.b.h);
    float4* dst = reinterpret_cast<float4*>(hs);
    const int n4 = NP * I / 4;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = src[i];
    __syncthreads();
  }
  for (; r < H; r += nwarps) {
    for (int g0 = 0; g0 < ngpu; g0 += kDCGroup) {
      if (g0 > 0) load_group(r, g0);
#pragma unroll
      for (int gi = 0; gi < kDCGroup; ++gi) {
        const int g = g0 + gi;
        if (g >= ngpu) break;
        const float* sd = reinterpret_cast<const float*>(sp.w[g] + sd_off);
        const int pb = sp.off[g], pe = sp.off[g + 1];
        for (int tp = pb; tp < pe; ++tp) {
          const int pid = sp.pid[tp];
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < kDCChunks; ++j) {
            const int c = j * 32 + lane;
            if (c < NCH) {
              float fw[V], hv[V];
              F::unpack(wv[gi][j], fw);
              const float4* hp = reinterpret_cast<const float4*>(hsrc + (size_t)pid * I + (size_t)c * V);
#pragma unroll
              for (int v = 0; v < V; v += 4) {
                const float4 q = hp[v / 4];
                hv[v] = q.x; hv[v + 1] = q.y; hv[v + 2] = q.z; hv[v + 3] = q.w;
              }
              float d = 0.f;
#pragma unroll
              for (int v = 0; v < V; ++v) d = fmaf(fw[v], hv[v], d);
              if (WT == MOE_FP8E4M3_B128) d *= __ldg(sd + (size_t)(r >> 7) * IB + ((c * V) >> 7));
              acc += d;
            }
          }
          acc = warp_sum(acc);
          if (lane == 0) {
            ys[pid] = acc;
            a.b.y[(size_t)pid * H + r] = acc;   // per-pair output stays readable (moe_cache_get_plan)
          }
        }
      }
    }
    __syncwarp();
    for (int t = lane; !a.b.defer_combine && t < a.T; t += 32) {
      float acc = 0.f;
      for (int j = 0; j < a.k; ++j) {
        const int p = t * a.k + j;
        float v;
        if (s_slot[p] >= 0) {
          v = ys[p];
        } else if (cpu != nullptr) {
          v = __ldg(cpu + (size_t)p * H + r);
        } else {
          v = 0.f;
          missing = true;
        }
        acc = fmaf(s_wt[p], v, acc);
      }
      if (a.n_shared) acc += ys[a.P + t];
      out[(size_t)t * H + r] = acc;
    }
    __syncwarp();
    if (r + nwarps < H) load_group(r + nwarps, 0);
  }
  if (__any_sync(0xffffffffu, missing) && lane == 0) atomicOr_system(err, kErrMissingCpuPart);
}

// ---- TMA-bulk-streamed GEMVs ------------------------------------------------------
// Weight bytes go global -> shared memory by cp.async.bulk, so a CTA holds far
// more bytes in flight than registers could stage.  Every warp owns a ring of
// shared-memory stages with one mbarrier each: its lane 0 keeps the next items'
// copies in flight while the warp computes the current one, and nothing but the
// warp's own barrier orders its stream.  Every wait is bounded by the global
// timer (2 s): on timeout the kernel flags the error word, lets its own copies
// land and returns.
constexpr unsigned long long kBulkWaitNs = 2000000000ull;
constexpr unsigned long long kTestWaitNs = 20000000ull;   // the test wait's limit (20 ms)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool bar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
  if (bar_test(bar, parity)) return true;
  const unsigned long long t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (bar_test(bar, parity)) return true;
    if ((i & 255u) == 0u && gtime() - t0 > kBulkWaitNs) return false;
  }
}
// one bulk copy global -> shared, counted on `bar` (whose expect_tx covers it)
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
// asks L2 to fetch [p, p + bytes) from HBM (16-byte aligned, 16-byte multiple); no completion
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// the same without an L2 eviction hint (data that other CTAs read too)
__device__ __forceinline__ void bulk_copy_keep(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void bar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Sums 16 per-lane values over the warp: 16 shuffles instead of 16 x 5.  Each
// step halves the values a lane holds, exchanging the other half with the lane
// `off` away; afterwards lane l holds the full sum of value (l >> 1).
__device__ __forceinline__ float reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool hi = lane & 16;
    const float send = hi ? v[j] : v[j + 8];
    v[j] = (hi ? v[j + 8] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool hi = lane & 8;
    const float send = hi ? v[j] : v[j + 4];
    v[j] = (hi ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const bool hi = lane & 4;
    const float send = hi ? v[j] : v[j + 2];
    v[j] = (hi ? v[j + 2] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  {
    const bool hi = lane & 2;
    const float send = hi ? v[0] : v[1];
    v[0] = (hi ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// The same for 8 values: afterwards lane l holds the full sum of value (l >> 2) & 7.
// The pairing of lanes (16, 8, 4, 2, 1) is that of warp_sum and reduce16, so a
// row's sum is the same bit for bit whichever of them forms it.
__device__ __forceinline__ float reduce8(float (&v)[8], int lane) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool hi = lane & 16;
    const float send = hi ? v[j] : v[j + 4];
    v[j] = (hi ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const bool hi = lane & 8;
    const float send = hi ? v[j] : v[j + 2];
    v[j] = (hi ? v[j + 2] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const bool hi = lane & 4;
    const float send = hi ? v[0] : v[1];
    v[0] = (hi ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

constexpr int kDownRows = 16;   // output rows per CTA of the bulk down kernel, at most
constexpr size_t kPrefetchPiece = 32 * 1024;
// dynamic shared memory the bulk kernels may ask for (the down kernel also has a few static bytes)
constexpr int kBulkSmemAttr = 224 * 1024;

struct BulkGeom {
  int R;        // down: output rows per CTA
  int NS;       // ring stages per warp (< 2: the shape does not fit)
  int NW;       // warps per CTA
  int h_smem;   // down: h of every pair staged in shared memory
  int pf_down;  // gate/up: have L2 fetch the experts' W_down behind the rows (it fits there)
  int RS, nsb;  // down: rows per ring stage, and sub-blocks of RS rows per CTA's R rows
  int grid;     // CTAs
  size_t SB;    // bytes per stage
  size_t ring_off, plan_off, extra_off, smem;
};

// Gate/up of the resident experts (pass 0).  A work item is one (expert, row i)
// pair: gate row i and up row I + i, 2 H weight elements; warp w of the grid
// takes items w, w + warps, ...  x is staged per CTA in shared memory while
// the first items are in flight.
template <int WT, int AT, int kJX>
__global__ void __launch_bounds__(256) gate_up_bulk_kernel(GemvArgs a, BulkGeom geo, uint32_t* err) {
  using F = WFmt<WT>;
  constexpr int V = F::V;
  extern __shared__ __align__(128) uint8_t sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm) + warp * geo.NS;
  uint8_t* ring = sm + geo.ring_off + (size_t)warp * geo.NS * geo.SB;
  if (lane == 0) {
    for (int i = 0; i < geo.NS; ++i) bar_init(&bars[i]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  const StagedPlan sp = stage_plan(sm + geo.plan_off, a);
  const int H = a.H, I = a.I;
  uint8_t* xsm = sm + geo.extra_off;
  const int ng = a.b.plan[P_NFIRST];   // pass 0: hits and the shared expert
  __syncthreads();
  const long items = (long)ng * I;
  const long nwarps = (long)gridDim.x * geo.NW;
  const long w0 = (long)blockIdx.x * geo.NW + warp;
  const size_t row_bytes = F::row(H);
  const uint64_t pol = evict_first_policy();
  long last_issued[4] = {-1, -1, -1, -1};
  auto issue = [&](long it, int st) {   // lane 0 only
    const int g = (int)(it / I), i = (int)(it % I);
    last_issued[st] = it;
    bar_expect(&bars[st], (uint32_t)(2 * row_bytes));
    uint8_t* dst = ring + (size_t)st * geo.SB;
    bulk_copy(dst, sp.w[g] + (size_t)i * row_bytes, (uint32_t)row_bytes, &bars[st], pol);
    bulk_copy(dst + row_bytes, sp.w[g] + (size_t)(I + i) * row_bytes, (uint32_t)row_bytes, &bars[st], pol);
  };
  // W_down of these experts is read by the down grid right after this one: once a
  // warp has issued its last row copy it asks L2 to fetch its share of those bytes
  // (32 KB pieces, piece p to warp p mod warps), so they queue behind the rows.
  const size_t wd_bytes = (size_t)H * F::row(I);
  const long pf_per = (long)((wd_bytes + kPrefetchPiece - 1) / kPrefetchPiece);
  auto prefetch_down = [&]() {   // lane 0 only
    for (long p = w0; p < (long)ng * pf_per; p += nwarps) {
      const int g = (int)(p / pf_per);
      const size_t o = (size_t)(p % pf_per) * kPrefetchPiece;
      const size_t n = wd_bytes - o < kPrefetchPiece ? wd_bytes - o : kPrefetchPiece;
      bulk_prefetch_l2(sp.w[g] + 2ull * (size_t)I * row_bytes + o, (uint32_t)n);
    }
  };
  const long n_mine = items > w0 ? (items - w0 + nwarps - 1) / nwarps : 0;
  if (lane == 0) {
    for (int k = 0; k < geo.NS; ++k) {
      const long it = w0 + (long)k * nwarps;
      if (it < items) issue(it, k);
    }
    if (geo.pf_down && n_mine <= geo.NS) prefetch_down();
  }
  {
    uint4* dst = reinterpret_cast<uint4*>(xsm);
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    const int n16 = (int)(((size_t)a.T * H * (AT == MOE_F32 ? 4 : 2)) >> 4);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const int NCH = H / V;
  const int HB = H / 128;
  // kJX > 0: one bf16 token, bf16 weights, NCH = 32 kJX: a lane's x chunks stay in
  // registers and each weight pair feeds one mixed-precision FMA
  uint4 xr[kJX > 0 ? kJX : 1];
  if (kJX > 0) {
#pragma unroll
    for (int j = 0; j < kJX; ++j) xr[j] = reinterpret_cast<const uint4*>(xsm)[j * 32 + lane];
  }
  bool ok = true;
  int k = 0;
  for (long it = w0; it < items; it += nwarps, ++k) {
    const int st = k % geo.NS;
    if (!__all_sync(0xffffffffu, bar_wait(&bars[st], (uint32_t)((k / geo.NS) & 1)))) { ok = false; break; }
    const int g = (int)(it / I), i = (int)(it % I);
    const uint4* gate = reinterpret_cast<const uint4*>(ring + (size_t)st * geo.SB);
    const uint4* up = reinterpret_cast<const uint4*>(ring + (size_t)st * geo.SB + row_bytes);
    const float* sgu = reinterpret_cast<const float*>(sp.w[g] + 3ull * (size_t)I * row_bytes);
    const int pb = sp.off[g], pe = sp.off[g + 1];
    if (kJX > 0) {   // same per-chunk partials and order as the generic loop below
      float ag = 0.f, au = 0.f;
#pragma unroll
      for (int j = 0; j < kJX; ++j) {
        const uint4 wg = gate[j * 32 + lane], wu = up[j * 32 + lane];
        float pg = 0.f, pu = 0.f;
        pg = fma_bf16x2(wg.x, xr[j].x, pg); pu = fma_bf16x2(wu.x, xr[j].x, pu);
        pg = fma_bf16x2(wg.y, xr[j].y, pg); pu = fma_bf16x2(wu.y, xr[j].y, pu);
        pg = fma_bf16x2(wg.z, xr[j].z, pg); pu = fma_bf16x2(wu.z, xr[j].z, pu);
        pg = fma_bf16x2(wg.w, xr[j].w, pg); pu = fma_bf16x2(wu.w, xr[j].w, pu);
        ag += pg;
        au += pu;
      }
      ag = warp_sum(ag);
      au = warp_sum(au);
      if (lane == 0)
        for (int tp = pb; tp < pe; ++tp) a.b.h[(size_t)sp.pid[tp] * I + i] = silu(ag) * au;
    }
    for (int tp = pb; kJX == 0 && tp < pe; ++tp) {
      const int t = sp.tok[tp];
      float ag = 0.f, au = 0.f;
      // unrolled: four chunks' independent FMA chains in flight; the sums keep
      // their order, so h is the same bit for bit as the fill's
#pragma unroll 4
      for (int c = lane; c < NCH; c += 32) {
        float dg = 0.f, du = 0.f;
        if constexpr (kFp4<WT>) {
          float xv[V];
          load_x<AT, V>(xsm, (size_t)t * H + (size_t)c * V, xv);
          const auto* srow = reinterpret_cast<const typename F::scale_t*>(sp.w[g] + F::sgu_off(H, I));
          dg = F::dot(gate[c], __ldg(srow + (size_t)i * (H / 32) + c), xv);
          du = F::dot(up[c], __ldg(srow + (size_t)(I + i) * (H / 32) + c), xv);
        } else {
          float fg[V], fu[V], xv[V];
          F::unpack(gate[c], fg);
          F::unpack(up[c], fu);
          load_x<AT, V>(xsm, (size_t)t * H + (size_t)c * V, xv);
#pragma unroll
          for (int v = 0; v < V; ++v) { dg = fmaf(fg[v], xv[v], dg); du = fmaf(fu[v], xv[v], du); }
          if (WT == MOE_FP8E4M3_B128) {
            const int cb = (c * V) >> 7;
            dg *= __ldg(sgu + (size_t)(i >> 7) * HB + cb);
            du *= __ldg(sgu + (size_t)((I + i) >> 7) * HB + cb);
          }
        }
        ag += dg;
        au += du;
      }
      ag = warp_sum(ag);
      au = warp_sum(au);
      if constexpr (WT == MOE_NVFP4) {   // the gate/up matrix's fp32 scale
        const float gg = __ldg(reinterpret_cast<const float*>(sp.w[g] + F::g_off(H, I)));
        ag *= gg;
        au *= gg;
      }
      if (lane == 0) a.b.h[(size_t)sp.pid[tp] * I + i] = silu(ag) * au;
    }
    __syncwarp();
    if (lane == 0 && it + (long)geo.NS * nwarps < items) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(it + (long)geo.NS * nwarps, st);
      if (geo.pf_down && k == n_mine - geo.NS - 1) prefetch_down();   // that was this warp's last row copy
    }
  }
  if (!ok && lane == 0) {  // flag the timeout; this warp's copies land before it exits
    atomicOr_system(err, kErrTimeout);
    for (int s2 = 0; s2 < geo.NS; ++s2) {
      if (last_issued[s2] < 0) continue;
      const long kk = (last_issued[s2] - w0) / nwarps;
      const uint32_t par = (uint32_t)((kk / geo.NS) & 1);
      const unsigned long long t0 = gtime();
      while (!bar_test(&bars[s2], par) && gtime() - t0 < kBulkWaitNs) {
      }
    }
  }
}

// Down projection fused with the combine.  A CTA owns output rows [r0, r0 + R),
// R <= 16, of the GPU experts of its pass (0: resident, 1: filled, 2: all).
// Warp w takes experts g0 + w, g0 + w + NW, ...  With kRing, their row blocks
// (R rows x I) stream through the warp's ring of shared-memory stages by bulk
// copy; without it (the filled experts, just written by the fill and still in
// L2) the rows are loaded directly.  Per pair, each lane holds its columns of h
// in registers and accumulates all R rows; one 16-value warp reduction leaves
// row (lane >> 1) in lane pairs.  The weight copies need only the control
// kernel's plan and the slot contents, both complete before this grid starts
// (a fill is a full dependency), so they are issued before the wait on the
// gate/up grid; h comes by bulk copy (pair rows) after it.
//
// Combine, out[t, r] = sum_j w[t,j] * (slot >= 0 ? y : cpu_part) in j order
// (+ shared): pass 2 forms it from shared memory after one barrier.  Passes 0
// and 1 are two grids over the same row blocks: each publishes its y, counts
// itself in arrive[block], and the second of the two (odd count before its
// increment) forms the block's combine from y in global memory.
template <int WT, bool kRing, int kJN, bool kPair = false, bool kR8 = false>
__global__ void __launch_bounds__((kRing && !kPair) || (!kRing && kJN > 0) ? 256 : 512) down_bulk_kernel(GemvArgs a, BulkGeom geo,
                                                        const float* __restrict__ w,
                                                        const float* __restrict__ cpu, float* __restrict__ out,
                                                        uint32_t* err) {
  // kPair: two warps per ring stage (one expert each pair), each taking 8 of its rows;
  // kR8: ring items of at most 8 rows, each warp accumulating 8 rows
  static_assert(!kPair || (kRing && kJN > 0), "pair mode is the straight-line ring path");
  static_assert(!kR8 || (kRing && !kPair), "8-row items are a ring form");
  using F = WFmt<WT>;
  constexpr int V = F::V;
  constexpr int J = 32 / V;   // 16-byte chunks per lane per column segment (32 h values in registers)
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint32_t s_second;
  // Split passes: when one of the two expert sets is empty the other grid combines
  // alone (no arrival is counted) and the empty grid leaves at once; with both
  // empty (every pair on the CPU) the resident grid combines.
  const bool split = a.pass != 2;
  bool alone = !split;
  if (split) {
    const int nfirst = a.b.plan[P_NFIRST], ngpu = a.b.plan[P_NGPU];
    if (a.pass == 1 ? ngpu == nfirst : (nfirst == 0 && ngpu > 0)) return;
    alone = a.pass == 0 ? ngpu == nfirst : nfirst == 0;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rw = kPair ? (warp >> 1) : warp;      // owner of the ring stages this warp reads
  const int half = kPair ? (warp & 1) : 0;        // pair mode: rows [8 half, 8 half + 8)
  const bool owner = !kPair || half == 0;         // issues and re-arms the stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm) + rw * geo.NS;
  uint64_t* hbar = reinterpret_cast<uint64_t*>(sm) + 31;   // ring barriers use at most 8 x 2
  uint8_t* ring = sm + geo.ring_off + (size_t)rw * geo.NS * geo.SB;
  if (lane == 0) {
    if (kRing && owner)
      for (int i = 0; i < geo.NS; ++i) bar_init(&bars[i]);
    if (warp == 0) bar_init(hbar);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const StagedPlan sp = stage_plan(sm + geo.plan_off, a);
  const int H = a.H, I = a.I;
  const int NP = a.P + a.T * a.n_shared;
  int* s_slot = reinterpret_cast<int*>(sm + geo.extra_off);
  float* s_wt = reinterpret_cast<float*>(s_slot + a.P);
  float* ys = reinterpret_cast<float*>(sm + geo.extra_off + (((size_t)a.P * 8 + 127) & ~size_t(127)));
  float* hs = ys + ((((size_t)geo.R * NP * 4 + NP + 127) & ~size_t(127)) >> 2);
  for (int i = threadIdx.x; i < a.P; i += blockDim.x) { s_slot[i] = a.b.slot_map[i]; s_wt[i] = w[i]; }
  const float* hsrc = geo.h_smem ? hs : a.b.h;
  int g0, g1;
  pass_range(a, g0, g1);
  uint8_t* s_mine = reinterpret_cast<uint8_t*>(ys + (size_t)geo.R * NP);   // [NP] pairs of this grid's experts
  __syncthreads();   // staged plan visible
  for (int i = threadIdx.x; i < NP; i += blockDim.x) s_mine[i] = 0;
  __syncthreads();
  for (int tp = sp.off[g0] + threadIdx.x; tp < sp.off[g1]; tp += blockDim.x) s_mine[sp.pid[tp]] = 1;
  const int r0 = blockIdx.x * geo.R;
  const int nr = min(geo.R, H - r0);
  const size_t row_bytes = F::row(I);
  const size_t down_off = 2ull * (size_t)I * F::row(H);
  const size_t sd_off = F::sd_off(H, I);
  const uint64_t pol = evict_first_policy();
  const bool h_copy = geo.h_smem && g1 > g0;
  __syncthreads();
  // Ring items: (expert g, sub-block sb of RS rows) of this pass's experts, expert
  // major; this CTA's nr rows (fewer than R in the last CTA) take ceil(nr / RS)
  // sub-blocks of 1..RS rows.  Each ring owner takes an even, contiguous share of
  // the items, so consecutive items of a warp mostly keep the same expert (and its
  // h in registers) and no warp has more than one item above another.
  const int nsb = (nr + geo.RS - 1) / geo.RS;
  const int n_all = (g1 - g0) * nsb;
  const int k_base = n_all * rw / geo.NW;
  const int n_wi = n_all * (rw + 1) / geo.NW - k_base;
  auto item_g = [&](int k) { return g0 + (k_base + k) / nsb; };
  auto item_sb = [&](int k) { return (k_base + k) % nsb; };
  auto item_rows = [&](int sb) { return min(geo.RS, nr - sb * geo.RS); };
  int last_issued[2] = {-1, -1};
  auto issue = [&](int k, int st) {   // lane 0 only
    last_issued[st] = k;
    const int sb = item_sb(k);
    const uint32_t bytes = (uint32_t)(item_rows(sb) * row_bytes);
    bar_expect(&bars[st], bytes);
    bulk_copy(ring + (size_t)st * geo.SB, sp.w[item_g(k)] + down_off + (size_t)(r0 + sb * geo.RS) * row_bytes, bytes,
              &bars[st], pol);
  };
  if (kRing && lane == 0 && owner)
    for (int k = 0; k < geo.NS && k < n_wi; ++k) issue(k, k);
  pdl_wait();   // h of the resident experts is complete from here on
  pdl_trigger();
  if (h_copy && threadIdx.x == 0) {   // the h rows (I floats, a 16-byte multiple) of this pass's pairs
    const int pb = sp.off[g0], pe = sp.off[g1];
    bar_expect(hbar, (uint32_t)((size_t)(pe - pb) * I * 4));
    for (int tp = pb; tp < pe; ++tp) {
      const size_t o = (size_t)sp.pid[tp] * I;
      bulk_copy_keep(hs + o, a.b.h + o, (uint32_t)(I * 4), hbar);
    }
  }
  const int NCH = I / V;
  const int IB = I / 128;
  bool ok = true;
  if (!kRing && kJN > 0) {
    // NCH = 32 kJN, no ring: items of (expert, kG rows) over all warps.  Every
    // 16-byte chunk of the kG rows is loaded before the first is used, so a warp
    // has kG x kJN loads in flight (the rows come from L2 right after their fill);
    // rows past nr repeat the last one.  The per-lane chunk order, its grouping by
    // J and the butterfly are those of the other paths, so y is the same bit for bit.
    constexpr int kG = 4;
    const int ngr = (nr + kG - 1) / kG;
    const int n_items = (g1 - g0) * ngr;
    float hn[kJN > 0 ? kJN : 1][V];
    int hn_pid = -1;
    for (int item = warp; item < n_items; item += geo.NW) {
      const int g = g0 + item / ngr, rb = (item % ngr) * kG;
      const int nrr = min(kG, nr - rb);
      const uint8_t* base = sp.w[g] + down_off + (size_t)(r0 + rb) * row_bytes;
      const float* sd = reinterpret_cast<const float*>(sp.w[g] + sd_off);
      uint4 wv[kG][kJN > 0 ? kJN : 1];
#pragma unroll
      for (int r = 0; r < kG; ++r) {
        const uint4* wrow = reinterpret_cast<const uint4*>(base + (size_t)(r < nrr ? r : nrr - 1) * row_bytes);
#pragma unroll
        for (int j = 0; j < kJN; ++j) wv[r][j] = wrow[j * 32 + lane];
      }
      for (int tp = sp.off[g]; tp < sp.off[g + 1]; ++tp) {
        const int pid = sp.pid[tp];
        if (pid != hn_pid) {
#pragma unroll
          for (int j = 0; j < kJN; ++j) {
            const float4* hp = reinterpret_cast<const float4*>(hsrc + (size_t)pid * I + (size_t)(j * 32 + lane) * V);
#pragma unroll
            for (int v = 0; v < V; v += 4) {
              const float4 q = hp[v / 4];
              hn[j][v] = q.x; hn[j][v + 1] = q.y; hn[j][v + 2] = q.z; hn[j][v + 3] = q.w;
            }
          }
          hn_pid = pid;
        }
#pragma unroll
        for (int r = 0; r < kG; ++r) {
          const int rr = r < nrr ? r : nrr - 1;
          float s = 0.f, d = 0.f;
#pragma unroll
          for (int j = 0; j < kJN; ++j) {
            float fw[V];
            F::unpack(wv[r][j], fw);
            float dj = 0.f;
#pragma unroll
            for (int v = 0; v < V; ++v) dj = fmaf(fw[v], hn[j][v], dj);
            if (WT == MOE_FP8E4M3_B128) dj *= __ldg(sd + (size_t)((r0 + rb + rr) >> 7) * IB + (((j * 32 + lane) * V) >> 7));
            d += dj;
            if ((j + 1) % J == 0 || j + 1 == kJN) {
              s += d;
              d = 0.f;
            }
          }
          float acc = 0.f;
          acc += s;
          acc = warp_sum(acc);
          if (lane == 0 && r < nrr) {
            ys[(size_t)(rb + r) * NP + pid] = acc;
            a.b.y[(size_t)pid * H + r0 + rb + r] = acc;
          }
        }
      }
    }
  }
  if (!kRing && kJN == 0) {   // (expert, row) items over all warps; the per-lane sums and the butterfly match the ring path
    if (h_copy && !__all_sync(0xffffffffu, bar_wait(hbar, 0))) ok = false;
    const int n_items = (g1 - g0) * nr;
    for (int item = warp; ok && item < n_items; item += geo.NW) {
      const int g = g0 + item / nr, r = item % nr;
      const uint4* wrow = reinterpret_cast<const uint4*>(sp.w[g] + down_off + (size_t)(r0 + r) * row_bytes);
      const float* sd = reinterpret_cast<const float*>(sp.w[g] + sd_off);
      if (item + geo.NW < n_items && lane == 0) {   // the warp's next row: on its way to L1 meanwhile
        const int g2 = g0 + (item + geo.NW) / nr, r2 = (item + geo.NW) % nr;
        const uint8_t* nx = sp.w[g2] + down_off + (size_t)(r0 + r2) * row_bytes;
        for (size_t o = 0; o < row_bytes; o += 128) asm volatile("prefetch.global.L1 [%0];" ::"l"(nx + o));
      }
      for (int tp = sp.off[g]; tp < sp.off[g + 1]; ++tp) {
        const int pid = sp.pid[tp];
        float acc = 0.f;
        for (int c0 = 0; c0 < NCH; c0 += 32 * J) {
          float d = 0.f;
#pragma unroll
          for (int j = 0; j < J; ++j) {
            const int c = c0 + j * 32 + lane;
            if (c < NCH) {
              const float4* hp = reinterpret_cast<const float4*>(hsrc + (size_t)pid * I + (size_t)c * V);
              float dj = 0.f;
              if constexpr (kFp4<WT>) {
                float hv[V];
#pragma unroll
                for (int v = 0; v < V; v += 4) {
                  const float4 q = hp[v / 4];
                  hv[v] = q.x; hv[v + 1] = q.y; hv[v + 2] = q.z; hv[v + 3] = q.w;
                }
                const auto* srow = reinterpret_cast<const typename F::scale_t*>(sp.w[g] + sd_off);
                dj = F::dot(wrow[c], __ldg(srow + (size_t)(r0 + r) * (I / 32) + c), hv);
              } else {
                float fw[V];
                F::unpack(wrow[c], fw);
#pragma unroll
                for (int v = 0; v < V; v += 4) {
                  const float4 q = hp[v / 4];
                  dj = fmaf(fw[v], q.x, dj);
                  dj = fmaf(fw[v + 1], q.y, dj);
                  dj = fmaf(fw[v + 2], q.z, dj);
                  dj = fmaf(fw[v + 3], q.w, dj);
                }
                if (WT == MOE_FP8E4M3_B128) dj *= __ldg(sd + (size_t)((r0 + r) >> 7) * IB + ((c * V) >> 7));
              }
              d += dj;
            }
          }
          acc += d;
        }
        acc = warp_sum(acc);
        if constexpr (WT == MOE_NVFP4) acc *= __ldg(reinterpret_cast<const float*>(sp.w[g] + F::g_off(H, I)) + 1);
        if (lane == 0) {
          ys[(size_t)r * NP + pid] = acc;
          a.b.y[(size_t)pid * H + r0 + r] = acc;
        }
      }
    }
  }
  float hv[kJN > 0 ? kJN : 1][V];   // the straight-line path's h of pair hv_pid
  int hv_pid = -1;
  for (int k = 0; kRing && k < n_wi; ++k) {
    const int st = k % geo.NS;
    if (k == 0 && h_copy && !__all_sync(0xffffffffu, bar_wait(hbar, 0))) { ok = false; break; }
    if (!__all_sync(0xffffffffu, bar_wait(&bars[st], (uint32_t)((k / geo.NS) & 1)))) { ok = false; break; }
    const uint8_t* blk = ring + (size_t)st * geo.SB;
    const int g = item_g(k), sb = item_sb(k);
    const int rsb = sb * geo.RS;             // this sub-block's first row within the CTA's R rows
    const int nrs = item_rows(sb);           // and its rows
    const float* sd = reinterpret_cast<const float*>(sp.w[g] + sd_off);
    const int pb = sp.off[g], pe = sp.off[g + 1];
    constexpr int kRW = (kPair || kR8) ? 8 : kDownRows;   // rows this warp accumulates
    const int rbase = kPair ? 8 * half : 0;
    for (int tp = pb; tp < pe; ++tp) {
      const int pid = sp.pid[tp];
      float acc[kRW];
#pragma unroll
      for (int r = 0; r < kRW; ++r) acc[r] = 0.f;
      if (kJN > 0) {
        // NCH = 32 kJN: one column segment, no guards; rows past nr repeat the
        // last row (their sums are never stored), so the whole block is one
        // straight run of independent chains.  h stays in registers while the
        // warp's items keep the same pair.
        if (pid != hv_pid) {
#pragma unroll
          for (int j = 0; j < kJN; ++j) {
            const float4* hp = reinterpret_cast<const float4*>(hsrc + (size_t)pid * I + (size_t)(j * 32 + lane) * V);
#pragma unroll
            for (int v = 0; v < V; v += 4) {
              const float4 q = hp[v / 4];
              hv[j][v] = q.x; hv[j][v + 1] = q.y; hv[j][v + 2] = q.z; hv[j][v + 3] = q.w;
            }
          }
          hv_pid = pid;
        }
#pragma unroll
        for (int r = 0; r < kRW; ++r) {
          const int rr = rbase + r < nrs ? rbase + r : nrs - 1;
          const uint4* wrow = reinterpret_cast<const uint4*>(blk + (size_t)rr * row_bytes);
          // chunk sums grouped J at a time, as the guarded path below adds them
          float s = 0.f, d = 0.f;
#pragma unroll
          for (int j = 0; j < kJN; ++j) {
            float fw[V];
            F::unpack(wrow[j * 32 + lane], fw);
            float dj = 0.f;
#pragma unroll
            for (int v = 0; v < V; ++v) dj = fmaf(fw[v], hv[j][v], dj);
            if (WT == MOE_FP8E4M3_B128) dj *= __ldg(sd + (size_t)((r0 + rsb + rr) >> 7) * IB + (((j * 32 + lane) * V) >> 7));
            d += dj;
            if ((j + 1) % J == 0 || j + 1 == kJN) {
              s += d;
              d = 0.f;
            }
          }
          acc[r] += s;
        }
      }
      for (int c0 = 0; kJN == 0 && c0 < NCH; c0 += 32 * J) {
        float hv[J][V];
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int c = c0 + j * 32 + lane;
          if (c < NCH) {
            const float4* hp = reinterpret_cast<const float4*>(hsrc + (size_t)pid * I + (size_t)c * V);
#pragma unroll
            for (int v = 0; v < V; v += 4) {
              const float4 q = hp[v / 4];
              hv[j][v] = q.x; hv[j][v + 1] = q.y; hv[j][v + 2] = q.z; hv[j][v + 3] = q.w;
            }
          } else {
#pragma unroll
            for (int v = 0; v < V; ++v) hv[j][v] = 0.f;
          }
        }
#pragma unroll
        for (int r = 0; r < kRW; ++r) {
          if (r < nrs) {
            const uint4* wrow = reinterpret_cast<const uint4*>(blk + (size_t)r * row_bytes);
            float d = 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) {
              const int c = c0 + j * 32 + lane;
              if (c < NCH) {
                float dj = 0.f;
                if constexpr (kFp4<WT>) {
                  const auto* srow = reinterpret_cast<const typename F::scale_t*>(sp.w[g] + sd_off);
                  dj = F::dot(wrow[c], __ldg(srow + (size_t)(r0 + rsb + r) * (I / 32) + c), hv[j]);
                } else {
                  float fw[V];
                  F::unpack(wrow[c], fw);
#pragma unroll
                  for (int v = 0; v < V; ++v) dj = fmaf(fw[v], hv[j][v], dj);
                  if (WT == MOE_FP8E4M3_B128) dj *= __ldg(sd + (size_t)((r0 + rsb + r) >> 7) * IB + ((c * V) >> 7));
                }
                d += dj;
              }
            }
            acc[r] += d;
          }
        }
      }
      float v;
      int r;
      bool mine;
      if constexpr (kPair || kR8) {
        v = reduce8(acc, lane);
        r = rbase + ((lane >> 2) & 7);
        mine = (lane & 3) == 0;
      } else {
        v = reduce16(acc, lane);
        r = lane >> 1;
        mine = (lane & 1) == 0;
      }
      if constexpr (WT == MOE_NVFP4) v *= __ldg(reinterpret_cast<const float*>(sp.w[g] + F::g_off(H, I)) + 1);
      if (mine && r < nrs) {
        ys[(size_t)(rsb + r) * NP + pid] = v;
        a.b.y[(size_t)pid * H + r0 + rsb + r] = v;   // per-pair output stays readable (moe_cache_get_plan)
      }
    }
    __syncwarp();
    if (lane == 0 && owner && k + geo.NS < n_wi) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(k + geo.NS, st);
    }
  }
  if (!ok && lane == 0) {   // flag the timeout; this warp's copies land before the CTA exits
    atomicOr_system(err, kErrTimeout);
    if (kRing)
      for (int s2 = 0; s2 < geo.NS; ++s2) {
        if (last_issued[s2] < 0) continue;
        const int kk = last_issued[s2];   // the item index of the copy that stage holds
        const uint32_t par = (uint32_t)((kk / geo.NS) & 1);
        const unsigned long long t0 = gtime();
        while (!bar_test(&bars[s2], par) && gtime() - t0 < kBulkWaitNs) {
        }
      }
  }
  if (h_copy && threadIdx.x == 0) {   // the h copy has landed before the CTA may exit
    const unsigned long long t0 = gtime();
    while (!bar_test(hbar, 0) && gtime() - t0 < kBulkWaitNs) {
    }
  }
  if (a.b.test_wait && a.pass == 0 && threadIdx.x == 0) {
    // a test of the bounded waits: a word nothing writes, given up on after 20 ms
    const unsigned long long t0 = gtime();
    bool set = false;
    for (uint32_t n = 0; !set; ++n) {
      set = __float_as_uint(*reinterpret_cast<const volatile float*>(a.b.never_set)) != 0xFFFFFFFFu;
      if ((n & 15u) == 15u && gtime() - t0 > kTestWaitNs) break;
    }
    if (!set) {
      ok = false;
      atomicOr_system(err, kErrTimeout);
    }
  }
  const bool all_ok = __syncthreads_and(ok);
  if (a.b.defer_combine) return;   // y is stored; the combine runs after the CPU branch
  if (!alone) {
    // Publish y and count this grid's arrival: the barrier orders every thread's y
    // stores before thread 0's gpu-scope acquire-release increment; the grid that
    // sees an odd count arrives second and combines.  It takes the other grid's
    // pairs from global memory (gathered in one parallel round trip into ys).
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t old;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.b.arrive + blockIdx.x) : "memory");
      s_second = old & 1u;
    }
    __syncthreads();
    if (!s_second) return;
    for (int idx = threadIdx.x; idx < nr * NP; idx += blockDim.x) {
      const int r = idx / NP, p = idx % NP;
      const bool gpu = p >= a.P || s_slot[p] >= 0;
      if (gpu && !s_mine[p]) ys[(size_t)r * NP + p] = __ldcg(a.b.y + (size_t)p * H + r0 + r);
    }
    __syncthreads();
  } else if (!all_ok) {
    return;
  }
  // (alone: every GPU pair of the call is this grid's own, in ys)
  bool missing = false;
  for (int idx = threadIdx.x; idx < nr * a.T; idx += blockDim.x) {
    const int r = idx / a.T, t = idx % a.T;
    float acc = 0.f;
    for (int j = 0; j < a.k; ++j) {
      const int p = t * a.k + j;
      float v;
      if (s_slot[p] >= 0) {
        v = ys[(size_t)r * NP + p];
      } else if (cpu != nullptr) {
        v = __ldg(cpu + (size_t)p * H + r0 + r);
      } else {
        v = 0.f;
        missing = true;
      }
      acc = fmaf(s_wt[p], v, acc);
    }
    if (a.n_shared) acc += ys[(size_t)r * NP + a.P + t];
    out[(size_t)t * H + r0 + r] = acc;
  }
  if (missing) atomicOr_system(err, kErrMissingCpuPart);
}

constexpr size_t kFusedSmemMax = 226 * 1024;   // dynamic shared memory of one CTA, at most

// ---- resident experts: the gate/up grid and its down projection in one launch ------
// One bf16 token, at most 8 resident experts (no shared expert).  Phase 1 is
// gate_up_bulk_kernel unchanged: per-warp rings of row pairs, and once a warp
// has issued its last row copy it has L2 fetch its share of the experts' W_down
// (cp.async.bulk.prefetch.L2), bytes in flight that need no shared memory.
// Then one grid-wide barrier (every h written), and phase 2 is the down
// projection + combine of down_bulk_kernel pass 0 by the same CTAs: warp g
// reads expert g's R x I block of W_down (from L2 by now) into the shared
// memory the rings used and its pair's h into registers (loads at L2), and the
// combine follows the split protocol (the resident and filled-expert grids
// count their arrivals per row block; the second combines).  Compared with two
// grids this saves the second grid's launch, its wait for the first grid's CTAs
// to leave their SMs, and its plan staging.
//
// The barrier needs every CTA of the grid on the GPU at once: one CTA per SM,
// and no kernel that could keep an SM waits on this one (the fill and the
// filled-expert down grid never do).  Its count only grows: a CTA's arrival
// number tells it which launch it belongs to.  The wait is bounded by the
// global timer; a timeout flags the error word.
constexpr int kFusedWarps = 8;

struct FusedGeom {
  int NS;             // gate/up ring stages per warp
  int R, nblk;        // down: rows per CTA, CTAs with rows
  size_t SBG, SBD;    // stage bytes: one gate/up row pair, one down row block
  size_t ring_off, plan_off, x_off, extra_off, smem;
};

template <int kJX, int kJN>
__global__ void __launch_bounds__(kFusedWarps * 32, 2) resident_fused_kernel(GemvArgs a, FusedGeom geo,
                                                                             const float* __restrict__ w,
                                                                             const float* __restrict__ cpu,
                                                                             float* __restrict__ out, uint32_t* err) {
  using F = WFmt<MOE_BF16>;
  constexpr int V = 8;
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint32_t s_second;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm) + warp * geo.NS;                 // phase 1
  uint64_t* dbar = reinterpret_cast<uint64_t*>(sm) + kFusedWarps * geo.NS + warp;   // phase 2
  if (lane == 0) {
    for (int i = 0; i < geo.NS; ++i) bar_init(&bars[i]);
    bar_init(dbar);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  const StagedPlan sp = stage_plan(sm + geo.plan_off, a);
  const int H = a.H, I = a.I;
  const int nfirst = a.b.plan[P_NFIRST], ngpu = a.b.plan[P_NGPU];
  const bool skip = nfirst == 0 && ngpu > 0;   // only filled experts: their grid combines alone
  const bool alone = ngpu == nfirst;           // no filled expert: this grid combines alone
  const int ng = skip ? 0 : nfirst;
  uint8_t* ring = sm + geo.ring_off;
  uint8_t* xsm = sm + geo.x_off;
  __syncthreads();

  // ---- phase 1: h = silu(gate . x) * (up . x), the gate_up_bulk_kernel stream ----------
  const long items = (long)ng * I;
  const long nwarps = (long)gridDim.x * kFusedWarps;
  const long w0 = (long)blockIdx.x * kFusedWarps + warp;
  const size_t row_h = F::row(H), row_i = F::row(I);
  const size_t down_off = 2ull * (size_t)I * row_h;
  const uint64_t pol = evict_first_policy();
  long last_issued[4] = {-1, -1, -1, -1};
  auto issue = [&](long it, int st) {   // lane 0 only
    const int g = (int)(it / I), i = (int)(it % I);
    last_issued[st] = it;
    bar_expect(&bars[st], (uint32_t)(2 * row_h));
    uint8_t* dst = ring + ((size_t)warp * geo.NS + st) * geo.SBG;
    bulk_copy(dst, sp.w[g] + (size_t)i * row_h, (uint32_t)row_h, &bars[st], pol);
    bulk_copy(dst + row_h, sp.w[g] + (size_t)(I + i) * row_h, (uint32_t)row_h, &bars[st], pol);
  };
  const size_t wd_bytes = (size_t)H * row_i;
  const long pf_per = (long)((wd_bytes + kPrefetchPiece - 1) / kPrefetchPiece);
  auto prefetch_down = [&]() {   // lane 0 only: this warp's share of the experts' W_down into L2
    for (long p = w0; p < (long)ng * pf_per; p += nwarps) {
      const int g = (int)(p / pf_per);
      const size_t o = (size_t)(p % pf_per) * kPrefetchPiece;
      const size_t n = wd_bytes - o < kPrefetchPiece ? wd_bytes - o : kPrefetchPiece;
      bulk_prefetch_l2(sp.w[g] + down_off + o, (uint32_t)n);
    }
  };
  const long n_mine = items > w0 ? (items - w0 + nwarps - 1) / nwarps : 0;
  if (lane == 0) {
    for (int k = 0; k < geo.NS; ++k) {
      const long it = w0 + (long)k * nwarps;
      if (it < items) issue(it, k);
    }
    if (n_mine <= geo.NS) prefetch_down();
  }
  {
    uint4* dst = reinterpret_cast<uint4*>(xsm);
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    const int n16 = (int)(((size_t)H * 2) >> 4);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  uint4 xr[kJX];
#pragma unroll
  for (int j = 0; j < kJX; ++j) xr[j] = reinterpret_cast<const uint4*>(xsm)[j * 32 + lane];
  bool ok = true;
  int k = 0;
  for (long it = w0; it < items; it += nwarps, ++k) {
    const int st = k % geo.NS;
    if (!__all_sync(0xffffffffu, bar_wait(&bars[st], (uint32_t)((k / geo.NS) & 1)))) { ok = false; break; }
    const int g = (int)(it / I), i = (int)(it % I);
    const uint4* gate = reinterpret_cast<const uint4*>(ring + ((size_t)warp * geo.NS + st) * geo.SBG);
    const uint4* up = reinterpret_cast<const uint4*>(ring + ((size_t)warp * geo.NS + st) * geo.SBG + row_h);
    float ag = 0.f, au = 0.f;   // the per-chunk partials and order of gate_up_bulk_kernel
#pragma unroll
    for (int j = 0; j < kJX; ++j) {
      const uint4 wg = gate[j * 32 + lane], wu = up[j * 32 + lane];
      float pg = 0.f, pu = 0.f;
      pg = fma_bf16x2(wg.x, xr[j].x, pg); pu = fma_bf16x2(wu.x, xr[j].x, pu);
      pg = fma_bf16x2(wg.y, xr[j].y, pg); pu = fma_bf16x2(wu.y, xr[j].y, pu);
      pg = fma_bf16x2(wg.z, xr[j].z, pg); pu = fma_bf16x2(wu.z, xr[j].z, pu);
      pg = fma_bf16x2(wg.w, xr[j].w, pg); pu = fma_bf16x2(wu.w, xr[j].w, pu);
      ag += pg;
      au += pu;
    }
    ag = warp_sum(ag);
    au = warp_sum(au);
    if (lane == 0)
      for (int tp = sp.off[g]; tp < sp.off[g + 1]; ++tp) a.b.h[(size_t)sp.pid[tp] * I + i] = silu(ag) * au;
    __syncwarp();
    if (lane == 0 && it + (long)geo.NS * nwarps < items) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(it + (long)geo.NS * nwarps, st);
      if (k == n_mine - geo.NS - 1) prefetch_down();   // that was this warp's last row copy
    }
  }
  if (!ok && lane == 0) {   // flag the timeout; this warp's copies land before the ring is reused
    atomicOr_system(err, kErrTimeout);
    for (int s2 = 0; s2 < geo.NS; ++s2) {
      if (last_issued[s2] < 0) continue;
      const long kk = (last_issued[s2] - w0) / nwarps;
      const uint32_t par = (uint32_t)((kk / geo.NS) & 1);
      const unsigned long long t0 = gtime();
      while (!bar_test(&bars[s2], par) && gtime() - t0 < kBulkWaitNs) {
      }
    }
  }

  // ---- this CTA's W_down blocks, then the grid-wide barrier (every CTA's h written) ------
  // The blocks do not depend on h: they head for the rings as soon as this CTA's
  // warps are done with them, and land while the CTA waits at the barrier.
  const int r0 = blockIdx.x * geo.R;
  const int nr = blockIdx.x < geo.nblk ? min(geo.R, H - r0) : 0;
  __syncthreads();
  if (lane == 0 && warp < ng && nr > 0) {   // warp g: expert g's row block
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bytes = (uint32_t)(nr * row_i);
    bar_expect(dbar, bytes);
    bulk_copy(ring + (size_t)warp * geo.SBD, sp.w[warp] + down_off + (size_t)r0 * row_i, bytes, dbar, pol);
  }
  if (threadIdx.x == 0) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(a.b.fused_bar) : "memory");
    const unsigned long long target = (old / gridDim.x + 1ull) * gridDim.x;
    const unsigned long long t0 = gtime();
    for (uint32_t it = 0;; ++it) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.b.fused_bar) : "memory");
      if (v >= target) break;
      if ((it & 15u) == 15u && gtime() - t0 > kBulkWaitNs) { atomicOr_system(err, kErrTimeout); break; }
      __nanosleep(32);
    }
  }
  __syncthreads();

  // ---- phase 2: down rows [r0, r0 + nr) of the resident experts, then the combine ----------
  if (nr == 0 || skip) return;   // the same for the whole CTA
  const int NP = a.P;
  int* s_slot = reinterpret_cast<int*>(sm + geo.extra_off);
  float* s_wt = reinterpret_cast<float*>(s_slot + a.P);
  float* ys = reinterpret_cast<float*>(sm + geo.extra_off + (((size_t)a.P * 8 + 127) & ~size_t(127)));
  uint8_t* s_mine = reinterpret_cast<uint8_t*>(ys + (size_t)geo.R * NP);
  for (int i = threadIdx.x; i < a.P; i += blockDim.x) { s_slot[i] = a.b.slot_map[i]; s_wt[i] = w[i]; s_mine[i] = 0; }
  __syncthreads();
  for (int tp = sp.off[0] + threadIdx.x; tp < sp.off[ng]; tp += blockDim.x) s_mine[sp.pid[tp]] = 1;
  bool dok = true;
  if (warp < ng) {   // one token: expert `warp` has exactly one pair
    const uint8_t* blk = ring + (size_t)warp * geo.SBD;
    const int pid = sp.pid[sp.off[warp]];
    // the lane's h values of the pair, written by every CTA before the barrier:
    // all 2 kJN loads at L2 in flight together, ahead of the wait for the block
    float hv[kJN][V];
#pragma unroll
    for (int j = 0; j < kJN; ++j) {
      const float4* hp = reinterpret_cast<const float4*>(a.b.h + (size_t)pid * I + (size_t)(j * 32 + lane) * V);
      const float4 q0 = __ldcg(hp), q1 = __ldcg(hp + 1);
      hv[j][0] = q0.x; hv[j][1] = q0.y; hv[j][2] = q0.z; hv[j][3] = q0.w;
      hv[j][4] = q1.x; hv[j][5] = q1.y; hv[j][6] = q1.z; hv[j][7] = q1.w;
    }
    dok = __all_sync(0xffffffffu, bar_wait(dbar, 0u));
    if (dok) {
      // the straight-line row block of down_bulk_kernel: rows past nr repeat the last
      // row (never stored), per-lane sums in the same order, then the 16-value butterfly
      float acc[kDownRows];
#pragma unroll
      for (int r = 0; r < kDownRows; ++r) {
        const int rr = r < nr ? r : nr - 1;
        const uint4* wrow = reinterpret_cast<const uint4*>(blk + (size_t)rr * row_i);
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < kJN; ++j) {
          float fw[V];
          F::unpack(wrow[j * 32 + lane], fw);
          float dj = 0.f;
#pragma unroll
          for (int v = 0; v < V; ++v) dj = fmaf(fw[v], hv[j][v], dj);
          d += dj;
        }
        acc[r] = 0.f + d;
      }
      const float v = reduce16(acc, lane);
      const int r = lane >> 1;
      if ((lane & 1) == 0 && r < nr) {
        ys[(size_t)r * NP + pid] = v;
        a.b.y[(size_t)pid * H + r0 + r] = v;   // per-pair output stays readable (moe_cache_get_plan)
      }
    }
    if (!dok && lane == 0) {   // flag the timeout; the block lands before the CTA exits
      atomicOr_system(err, kErrTimeout);
      const unsigned long long t0 = gtime();
      while (!bar_test(dbar, 0u) && gtime() - t0 < kBulkWaitNs) {
      }
    }
  }
  __syncthreads();
  if (a.b.defer_combine) return;   // y is stored; the combine runs after the CPU branch
  if (!alone) {   // the split protocol of down_bulk_kernel
    if (threadIdx.x == 0) {
      uint32_t old;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.b.arrive + blockIdx.x) : "memory");
      s_second = old & 1u;
    }
    __syncthreads();
    if (!s_second) return;
    for (int idx = threadIdx.x; idx < nr * NP; idx += blockDim.x) {
      const int r = idx / NP, p = idx % NP;
      if (s_slot[p] >= 0 && !s_mine[p]) ys[(size_t)r * NP + p] = __ldcg(a.b.y + (size_t)p * H + r0 + r);
    }
    __syncthreads();
  }
  bool missing = false;
  for (int r = threadIdx.x; r < nr; r += blockDim.x) {   // one token
    float acc = 0.f;
    for (int j = 0; j < a.k; ++j) {
      float v;
      if (s_slot[j] >= 0) {
        v = ys[(size_t)r * NP + j];
      } else if (cpu != nullptr) {
        v = __ldg(cpu + (size_t)j * H + r0 + r);
      } else {
        v = 0.f;
        missing = true;
      }
      acc = fmaf(s_wt[j], v, acc);
    }
    out[r0 + r] = acc;
  }
  if (missing) atomicOr_system(err, kErrMissingCpuPart);
}

// ---- combine: out[t] = sum_j w[t,j] * (slot >= 0 ? y : cpu_part) in j order (+ shared) --
__global__ void combine_kernel(int T, int H, int k, int n_shared, const float* __restrict__ w,
                               const int32_t* __restrict__ sm, const float* __restrict__ y,
                               const float* __restrict__ cpu, float* __restrict__ out, uint32_t* err) {
  const int H4 = H >> 2;
  const long n = (long)T * H4;
  const int P = T * k;
  bool missing = false;
  for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / H4);
    const int c = (int)(idx % H4) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int p = t * k + j;
      const float wt = __ldg(w + p);
      float4 v;
      if (sm[p] >= 0) {
        v = __ldg(reinterpret_cast<const float4*>(y + (size_t)p * H + c));
      } else if (cpu != nullptr) {
        v = __ldg(reinterpret_cast<const float4*>(cpu + (size_t)p * H + c));
      } else {
        v = make_float4(0.f, 0.f, 0.f, 0.f);
        missing = true;
      }
      acc.x = fmaf(wt, v.x, acc.x); acc.y = fmaf(wt, v.y, acc.y);
      acc.z = fmaf(wt, v.z, acc.z); acc.w = fmaf(wt, v.w, acc.w);
    }
    if (n_shared) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(y + (size_t)(P + t) * H + c));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    *reinterpret_cast<float4*>(out + (size_t)t * H + c) = acc;
  }
  if (__any_sync(0xffffffffu, missing) && (threadIdx.x & 31) == 0) atomicOr_system(err, kErrMissingCpuPart);
}

// ---- blob copy: complete experts host pool -> slots ---------------------------------
// Prefill with 4-bit experts: every active expert e of the layer that has routed
// rows (offsets[e + 1] > offsets[e]), read from its slot wslot[e], is written as a bf16 blob of the bank layout (W_gu [2I, H], then
// W_d [H, I]) at staging + e * 3IH, which the grouped GEMMs read.  One thread per
// 16-byte chunk of codes (32 weights); the chunks of W_gu and W_d are contiguous in
// the slot, and so are their scale entries (one scale_t per chunk).
template <int WT>
__global__ void __launch_bounds__(256) fp4_to_bf16_kernel(const int32_t* __restrict__ wslot,
                                                          const int32_t* __restrict__ active,
                                                          const int32_t* __restrict__ offsets, int E, int H, int I,
                                                          const uint8_t* __restrict__ slots, uint64_t S,
                                                          uint16_t* __restrict__ staging) {
  using F = WFmt<WT>;
  const long n_gu = (long)2 * I * H / 32;               // chunks of W_gu
  const long per = n_gu + (long)H * I / 32;             // chunks per expert
  const long total = (long)E * per;
  for (long it = (long)blockIdx.x * blockDim.x + threadIdx.x; it < total; it += (long)gridDim.x * blockDim.x) {
    const int e = (int)(it / per);
    const int slot = wslot[e];
    if (!active[e] || slot < 0 || offsets[e + 1] <= offsets[e]) continue;
    const long c = it - (long)e * per;
    const uint8_t* b = slots + (size_t)slot * S;
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(b) + c);
    const uint32_t sc = reinterpret_cast<const typename F::scale_t*>(b + F::sgu_off(H, I))[c];
    float g = 1.f;
    if constexpr (WT == MOE_NVFP4) g = reinterpret_cast<const float*>(b + F::g_off(H, I))[c < n_gu ? 0 : 1];
    float f[32];
    F::decode32(w, sc, g, f);
    uint4 o[4];
    uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * v], f[2 * v + 1]);
      ow[v] = *reinterpret_cast<const uint32_t*>(&p);
    }
    uint4* dst = reinterpret_cast<uint4*>(staging + (size_t)e * 3 * (size_t)I * H + (size_t)c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = o[q];
  }
}

// list = (flat id, slot) pairs; the copy starts at pair *skip (if skip) and takes *count
// pairs.  Every CTA copies its 1/gridDim share of every blob, so one launch spreads
// any number of blobs over the whole grid with 16-byte loads, 4 in flight per thread.
__global__ void __launch_bounds__(512) copy_blobs_kernel(const int32_t* __restrict__ count,
                                                         const int32_t* __restrict__ skip,
                                                         const int32_t* __restrict__ list,
                                                         const uint8_t* __restrict__ host,
                                                         const uint64_t* __restrict__ offs,
                                                         uint8_t* __restrict__ slots, uint64_t S) {
  constexpr int U = 4;
  const int n = *count;
  const int32_t* pairs = list + (skip ? 2 * (*skip) : 0);
  const uint64_t n16 = S >> 4;
  const uint64_t per = (n16 + gridDim.x - 1) / gridDim.x;
  const uint64_t c0 = per * blockIdx.x;
  const uint64_t c1 = min(n16, c0 + per);
  for (int i = 0; i < n; ++i) {
    const int f = pairs[2 * i];
    const int s = pairs[2 * i + 1];
    const uint4* src = reinterpret_cast<const uint4*>(host + offs[f]);
    uint4* dst = reinterpret_cast<uint4*>(slots + (size_t)s * S);
    uint64_t c = c0 + threadIdx.x;
    for (; c + (U - 1) * blockDim.x < c1; c += U * blockDim.x) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = src[c + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < U; ++u) __stcs(dst + c + u * blockDim.x, v[u]);
    }
    for (; c < c1; c += blockDim.x) __stcs(dst + c, src[c]);
  }
}

constexpr size_t kXSmem = 64 * 1024;      // x staged in shared memory up to this size

GemvArgs make_args(const Shape& sh, int pass, int T, const void* x, const DecodeBufs& b) {
  GemvArgs a;
  a.H = sh.H; a.I = sh.I; a.k = sh.k; a.T = T; a.P = T * sh.k; a.pass = pass; a.n_shared = sh.n_shared;
  a.max_g = (sh.E < T * sh.k ? sh.E : T * sh.k) + sh.n_shared;
  a.max_p = T * sh.k + T * sh.n_shared;
  a.x_smem = (size_t)T * sh.H * (sh.adtype == MOE_F32 ? 4 : 2) <= kXSmem ? 1 : 0;
  a.x = x; a.b = b;
  return a;
}

size_t gate_up_smem(const GemvArgs& a, int adtype) {
  return staged_plan_bytes(a.max_g, a.max_p) +
         (a.x_smem ? (size_t)a.T * a.H * (adtype == MOE_F32 ? 4 : 2) : 0);
}

template <int WT, int AT>
cudaError_t launch_gemv_typed(const GemvArgs& a, int sms, cudaStream_t s) {
  if (a.T == 1) {
    gate_up_kernel<WT, AT, 1><<<2 * sms, kGemvThreads, gate_up_smem(a, AT), s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    down_kernel<WT, 1><<<2 * sms, kGemvThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
  gate_up_kernel<WT, AT, 4><<<sms, kGemvThreads, gate_up_smem(a, AT), s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  down_kernel<WT, 4><<<sms, kGemvThreads, 0, s>>>(a);
  return cudaGetLastError();
}

// A plain launch (not programmatic): launched early, its CTAs would hold every
// SM's registers while waiting and keep the fill of the same layer off the GPU.
template <int WT, int AT>
cudaError_t launch_gate_up_typed(const GemvArgs& a, int sms, cudaStream_t s) {
  const size_t smem = gate_up_smem(a, AT);
  if (a.T == 1) gate_up_kernel<WT, AT, 1><<<2 * sms, kGemvThreads, smem, s>>>(a);
  else gate_up_kernel<WT, AT, 4><<<sms, kGemvThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int WT>
cudaError_t launch_down_typed(const GemvArgs& a, int sms, cudaStream_t s) {
  if (a.T == 1) down_kernel<WT, 1><<<2 * sms, kGemvThreads, 0, s>>>(a);
  else down_kernel<WT, 4><<<sms, kGemvThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int WT>
cudaError_t launch_down_combine_typed(const GemvArgs& a, const float* w, const float* cpu, float* out,
                                      uint32_t* err, int sms, cudaStream_t s) {
  const size_t np = (size_t)(a.P + a.T * a.n_shared);
  const size_t hbytes = np * a.I * sizeof(float);
  const size_t smem = staged_plan_bytes(a.max_g, a.max_p) + (((size_t)a.P * 8 + 15) & ~size_t(15)) +
                      (size_t)kDCWarps * np * sizeof(float) + (hbytes <= kDCHSmem ? hbytes : 0);
  const int blocks = (a.H + kDCWarps - 1) / kDCWarps;
  return launch_pdl(down_combine_kernel<WT>, dim3(blocks < 4 * sms ? blocks : 4 * sms), dim3(kDCWarps * 32), smem, s,
                    a, w, cpu, out, err);
}


}  // namespace

int gemv_block_threads() { return kGemvThreads; }

// The register-staged gate/up kernel stages the plan (and x, up to kXSmem) in
// dynamic shared memory; setup_gemv_kernels() allows it at most this much.
size_t expert_gemv_smem(const Shape& sh, int T) {
  return gate_up_smem(make_args(sh, 0, T, nullptr, DecodeBufs{}), sh.adtype);
}
size_t expert_gemv_smem_limit() { return kXSmem + staged_plan_bytes(4096 + 1, 1024 * 8 + 1024); }

template <int WT, int AT>
cudaError_t carveout_typed() {
  const void* ks[] = {(const void*)gate_up_kernel<WT, AT, 1>, (const void*)gate_up_kernel<WT, AT, 4>,
                      (const void*)fill_gate_up_kernel<WT, AT, 1>, (const void*)fill_gate_up_kernel<WT, AT, 4>};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kDecodeCarveout);
    if (e != cudaSuccess) return e;
  }
  std::vector<const void*> bulk = {(const void*)gate_up_bulk_kernel<WT, AT, 0>};
  if constexpr (WT == MOE_BF16 && AT == MOE_BF16) {
    bulk.push_back((const void*)gate_up_bulk_kernel<WT, AT, 4>);
    bulk.push_back((const void*)gate_up_bulk_kernel<WT, AT, 8>);
  }
  for (const void* k : bulk) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmemAttr);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kDecodeCarveout);
    if (e != cudaSuccess) return e;
  }
  // x (up to kXSmem) plus the staged plan of up to 1024 tokens x top-8 pairs
  const int gu_smem = (int)expert_gemv_smem_limit();
  for (const void* k : {(const void*)gate_up_kernel<WT, AT, 1>, (const void*)gate_up_kernel<WT, AT, 4>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, gu_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t setup_gemv_kernels() {
  const int smem = (int)(kDCHSmem + (size_t)kDCWarps * kDCMaxPairs * sizeof(float) +
                         staged_plan_bytes(4096 + 1, kDCMaxPairs) + (size_t)kDCMaxPairs * 8);
  for (const void* k : {(const void*)down_bulk_kernel<MOE_F32, true, 0>, (const void*)down_bulk_kernel<MOE_BF16, true, 0>,
                        (const void*)down_bulk_kernel<MOE_BF16, true, 3>, (const void*)down_bulk_kernel<MOE_BF16, true, 4>,
                        (const void*)down_bulk_kernel<MOE_BF16, true, 3, true>,
                        (const void*)down_bulk_kernel<MOE_BF16, true, 4, true>,
                        (const void*)down_bulk_kernel<MOE_FP8E4M3_B128, true, 0>,
                        (const void*)down_bulk_kernel<MOE_FP8E4M3_B128, true, 3, false, true>,
                        (const void*)down_bulk_kernel<MOE_FP8E4M3_B128, true, 4, false, true>,
                        (const void*)down_bulk_kernel<MOE_F32, false, 0>, (const void*)down_bulk_kernel<MOE_BF16, false, 0>,
                        (const void*)down_bulk_kernel<MOE_BF16, false, 3>, (const void*)down_bulk_kernel<MOE_BF16, false, 4>,
                        (const void*)down_bulk_kernel<MOE_FP8E4M3_B128, false, 3>,
                        (const void*)down_bulk_kernel<MOE_FP8E4M3_B128, false, 4>,
                        (const void*)down_bulk_kernel<MOE_FP8E4M3_B128, false, 0>,
                        (const void*)down_bulk_kernel<MOE_NVFP4, true, 0>, (const void*)down_bulk_kernel<MOE_NVFP4, false, 0>,
                        (const void*)gate_up_bulk_kernel<MOE_NVFP4, MOE_F32, 0>,
                        (const void*)gate_up_bulk_kernel<MOE_NVFP4, MOE_BF16, 0>,
                        (const void*)down_bulk_kernel<MOE_MXFP4, true, 0>, (const void*)down_bulk_kernel<MOE_MXFP4, false, 0>,
                        (const void*)gate_up_bulk_kernel<MOE_MXFP4, MOE_F32, 0>,
                        (const void*)gate_up_bulk_kernel<MOE_MXFP4, MOE_BF16, 0>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmemAttr);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kDecodeCarveout);
    if (e != cudaSuccess) return e;
  }
  for (const void* k : {(const void*)resident_fused_kernel<8, 3>, (const void*)resident_fused_kernel<8, 4>,
                        (const void*)resident_fused_kernel<4, 3>, (const void*)resident_fused_kernel<4, 4>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedSmemMax);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kDecodeCarveout);
    if (e != cudaSuccess) return e;
  }
  const void* dc[] = {(const void*)down_combine_kernel<MOE_F32>, (const void*)down_combine_kernel<MOE_BF16>,
                      (const void*)down_combine_kernel<MOE_FP8E4M3_B128>};
  for (const void* k : dc) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kDecodeCarveout);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = carveout_typed<MOE_F32, MOE_F32>();
  if (e == cudaSuccess) e = carveout_typed<MOE_F32, MOE_BF16>();
  if (e == cudaSuccess) e = carveout_typed<MOE_BF16, MOE_F32>();
  if (e == cudaSuccess) e = carveout_typed<MOE_BF16, MOE_BF16>();
  if (e == cudaSuccess) e = carveout_typed<MOE_FP8E4M3_B128, MOE_F32>();
  if (e == cudaSuccess) e = carveout_typed<MOE_FP8E4M3_B128, MOE_BF16>();
  if (e == cudaSuccess) e = carveout_typed<MOE_NVFP4, MOE_F32>();
  if (e == cudaSuccess) e = carveout_typed<MOE_NVFP4, MOE_BF16>();
  if (e == cudaSuccess) e = carveout_typed<MOE_MXFP4, MOE_F32>();
  if (e == cudaSuccess) e = carveout_typed<MOE_MXFP4, MOE_BF16>();
  return e;
}

template <int WT, int AT>
cudaError_t launch_fill_gate_up_typed(const GemvArgs& a, const int32_t* fills, const uint8_t* host,
                                      const uint64_t* offs, uint8_t* slots, uint64_t S, int n_ctas, cudaStream_t s) {
  if (a.T == 1) fill_gate_up_kernel<WT, AT, 1><<<n_ctas, kFillThreads, 0, s>>>(a, fills, host, offs, slots, S);
  else fill_gate_up_kernel<WT, AT, 4><<<n_ctas, kFillThreads, 0, s>>>(a, fills, host, offs, slots, S);
  return cudaGetLastError();
}

cudaError_t launch_fill_gate_up(const Shape& sh, int T, const void* x, DecodeBufs b, const uint8_t* host_pool_dev,
                                const uint64_t* offsets, uint8_t* slots, int n_ctas, cudaStream_t s) {
  const GemvArgs a = make_args(sh, 1, T, x, b);
  const int32_t* f = b.fills;
  switch (sh.wdtype * 2 + sh.adtype) {
    case MOE_F32 * 2 + MOE_F32:
      return launch_fill_gate_up_typed<MOE_F32, MOE_F32>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_F32 * 2 + MOE_BF16:
      return launch_fill_gate_up_typed<MOE_F32, MOE_BF16>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_BF16 * 2 + MOE_F32:
      return launch_fill_gate_up_typed<MOE_BF16, MOE_F32>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_BF16 * 2 + MOE_BF16:
      return launch_fill_gate_up_typed<MOE_BF16, MOE_BF16>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_FP8E4M3_B128 * 2 + MOE_F32:
      return launch_fill_gate_up_typed<MOE_FP8E4M3_B128, MOE_F32>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_FP8E4M3_B128 * 2 + MOE_BF16:
      return launch_fill_gate_up_typed<MOE_FP8E4M3_B128, MOE_BF16>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_NVFP4 * 2 + MOE_F32:
      return launch_fill_gate_up_typed<MOE_NVFP4, MOE_F32>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_NVFP4 * 2 + MOE_BF16:
      return launch_fill_gate_up_typed<MOE_NVFP4, MOE_BF16>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_MXFP4 * 2 + MOE_F32:
      return launch_fill_gate_up_typed<MOE_MXFP4, MOE_F32>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
    case MOE_MXFP4 * 2 + MOE_BF16:
      return launch_fill_gate_up_typed<MOE_MXFP4, MOE_BF16>(a, f, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
  }
  return cudaErrorInvalidValue;
}

// bytes of n weight elements
size_t wrow(int wdtype, size_t n) {
  return wdtype == MOE_F32 ? 4 * n : wdtype == MOE_BF16 ? 2 * n : (wdtype == MOE_NVFP4 || wdtype == MOE_MXFP4) ? n / 2 : n;
}
size_t up128(size_t x) { return (x + 127) & ~size_t(127); }

// Ring geometry and shared-memory layout of the bulk-streamed kernels; NS = 0
// (gate/up: NS < 2) means the shape does not fit and the register-staged
// kernel runs instead.
constexpr size_t kRingBudget = 220 * 1024;
constexpr size_t kPrefetchDownMax = 40ull << 20;   // W_down bytes the gate/up grid has L2 fetch, at most

// Gate/up: one CTA per SM, up to 8 warps with up to 3 stages of one row pair each
// (about 200 KB for the Qwen3 shape: the stream is bound by the bytes each SM has
// in flight; the fill and the filled-expert down grid still fit beside it).
BulkGeom gate_up_geom(const GemvArgs& a, int wdtype, int adtype, int sms) {
  BulkGeom g{};
  g.grid = sms;
  const size_t row = wrow(wdtype, (size_t)a.H);
  const size_t xbytes = (size_t)a.T * a.H * (adtype == MOE_F32 ? 4 : 2);
  const size_t plan = up128(staged_plan_bytes(a.max_g, a.max_p));
  g.SB = up128(2 * row);
  const size_t fixed = 256 + plan + up128(xbytes);
  if (xbytes > kXSmem || fixed >= kRingBudget) return g;
  const size_t room = kRingBudget - fixed;
  for (g.NW = 8; g.NW >= 2; --g.NW) {
    g.NS = (int)std::min<size_t>(3, room / ((size_t)g.NW * g.SB));
    if (g.NS >= 2) break;
  }
  if (g.NS < 2) { g.NS = 0; return g; }
  g.ring_off = 256;
  g.plan_off = g.ring_off + (size_t)g.NW * g.NS * g.SB;
  g.extra_off = g.plan_off + plan;
  g.smem = g.extra_off + up128(xbytes);
  // W_down of the call's experts fetched into L2 behind the gate/up rows helps only
  // if it stays there until the down grid reads it: beside a full-rate stream that
  // holds for a few tens of MB (8 Qwen3-shaped experts: 25 MB), not for 132 MB
  // (the DeepSeek-V3 slice) or 200 MB (16 tokens over ~66 experts), which L2 evicts
  // first and the down grid reads from HBM again.
  g.pf_down = (size_t)a.max_g * a.H * wrow(wdtype, (size_t)a.I) <= kPrefetchDownMax ? 1 : 0;
  return g;
}

// Down: R = ceil(H / sms) output rows per CTA, so the grid is one wave; the ring
// streams them in sub-blocks of RS <= 16 rows (one sub-block when R <= 16, as for
// the Qwen3 shapes; 4 of up to 13 rows for the DeepSeek-V3 slice's R = 48), with
// one stage for each of 8 warps when there are at most 8 GPU experts, else
// two-stage rings of at least four warps; fewer rows per stage when that does not
// fit.  (Shrinking R instead would take several waves of CTAs, each filling its
// ring from cold.)
BulkGeom down_geom(const GemvArgs& a, int wdtype, int sms) {
  BulkGeom g{};
  const size_t row = wrow(wdtype, (size_t)a.I);
  const size_t np = (size_t)(a.P + a.T * a.n_shared);
  const size_t hbytes = np * a.I * 4;
  const size_t plan = up128(staged_plan_bytes(a.max_g, a.max_p));
  g.h_smem = hbytes <= 64 * 1024 ? 1 : 0;
  const int R = (a.H + sms - 1) / sms;
  const size_t extra = up128((size_t)a.P * 8) + up128((size_t)R * np * 4 + np) + (g.h_smem ? hbytes : 0);
  const size_t fixed = 256 + plan + up128(extra);
  if (fixed >= kRingBudget) { g.NS = 0; return g; }
  const size_t room = kRingBudget - fixed;
  // fp8 rows stream in items of at most 8 rows (the straight-line 8-row form;
  // with 16 the DeepSeek-V3 slice got sub-blocks of 12 rows on 4 warps)
  const int rs_max = wdtype == MOE_FP8E4M3_B128 ? 8 : kDownRows;
  for (int RS = std::min(R, rs_max); RS >= 1; --RS) {
    g.SB = up128((size_t)RS * row);
    if (a.max_g <= 8 && 8 * g.SB <= room) {
      g.NS = 1;
      g.NW = 8;
    } else {
      g.NS = 2;
      g.NW = (int)std::min<size_t>(8, room / (2 * g.SB));
    }
    if (g.NW >= 4) {
      g.R = R;
      g.RS = RS;
      g.nsb = (R + RS - 1) / RS;
      g.grid = (a.H + R - 1) / R;
      g.ring_off = 256;
      g.plan_off = g.ring_off + (size_t)g.NW * g.NS * g.SB;
      g.extra_off = g.plan_off + plan;
      g.smem = g.extra_off + up128(extra);
      return g;
    }
  }
  g.NS = 0;
  return g;
}

template <int WT, int AT>
cudaError_t launch_gate_up_bulk(const GemvArgs& a, const BulkGeom& geo, uint32_t* err, cudaStream_t s) {
  // one bf16 token over bf16 rows of 4 or 8 16-byte chunks per lane: the register-x path
  if constexpr (WT == MOE_BF16 && AT == MOE_BF16) {
    const int jx = (a.T == 1 && (a.H / 8) % 32 == 0) ? a.H / 8 / 32 : 0;
    if (jx == 8)
      return launch_pdl(gate_up_bulk_kernel<WT, AT, 8>, dim3(geo.grid), dim3(geo.NW * 32), geo.smem, s, a, geo, err);
    if (jx == 4)
      return launch_pdl(gate_up_bulk_kernel<WT, AT, 4>, dim3(geo.grid), dim3(geo.NW * 32), geo.smem, s, a, geo, err);
  }
  return launch_pdl(gate_up_bulk_kernel<WT, AT, 0>, dim3(geo.grid), dim3(geo.NW * 32), geo.smem, s, a, geo, err);
}

cudaError_t launch_gate_up(const Shape& sh, int pass, int T, const void* x, DecodeBufs b, int sms, cudaStream_t s,
                           uint32_t* err) {
  const GemvArgs a = make_args(sh, pass, T, x, b);
  if (pass == 0 && err != nullptr) {
    const BulkGeom geo = gate_up_geom(a, sh.wdtype, sh.adtype, sms);
    if (geo.NS >= 2) {
      switch (sh.wdtype * 2 + sh.adtype) {
        case MOE_F32 * 2 + MOE_F32: return launch_gate_up_bulk<MOE_F32, MOE_F32>(a, geo, err, s);
        case MOE_F32 * 2 + MOE_BF16: return launch_gate_up_bulk<MOE_F32, MOE_BF16>(a, geo, err, s);
        case MOE_BF16 * 2 + MOE_F32: return launch_gate_up_bulk<MOE_BF16, MOE_F32>(a, geo, err, s);
        case MOE_BF16 * 2 + MOE_BF16: return launch_gate_up_bulk<MOE_BF16, MOE_BF16>(a, geo, err, s);
        case MOE_FP8E4M3_B128 * 2 + MOE_F32: return launch_gate_up_bulk<MOE_FP8E4M3_B128, MOE_F32>(a, geo, err, s);
        case MOE_FP8E4M3_B128 * 2 + MOE_BF16: return launch_gate_up_bulk<MOE_FP8E4M3_B128, MOE_BF16>(a, geo, err, s);
        case MOE_NVFP4 * 2 + MOE_F32: return launch_gate_up_bulk<MOE_NVFP4, MOE_F32>(a, geo, err, s);
        case MOE_NVFP4 * 2 + MOE_BF16: return launch_gate_up_bulk<MOE_NVFP4, MOE_BF16>(a, geo, err, s);
        case MOE_MXFP4 * 2 + MOE_F32: return launch_gate_up_bulk<MOE_MXFP4, MOE_F32>(a, geo, err, s);
        case MOE_MXFP4 * 2 + MOE_BF16: return launch_gate_up_bulk<MOE_MXFP4, MOE_BF16>(a, geo, err, s);
      }
    }
  }
  switch (sh.wdtype * 2 + sh.adtype) {   // register-staged kernels
    case MOE_NVFP4 * 2 + MOE_F32: return launch_gate_up_typed<MOE_NVFP4, MOE_F32>(a, sms, s);
    case MOE_NVFP4 * 2 + MOE_BF16: return launch_gate_up_typed<MOE_NVFP4, MOE_BF16>(a, sms, s);
    case MOE_MXFP4 * 2 + MOE_F32: return launch_gate_up_typed<MOE_MXFP4, MOE_F32>(a, sms, s);
    case MOE_MXFP4 * 2 + MOE_BF16: return launch_gate_up_typed<MOE_MXFP4, MOE_BF16>(a, sms, s);
    case MOE_F32 * 2 + MOE_F32: return launch_gate_up_typed<MOE_F32, MOE_F32>(a, sms, s);
    case MOE_F32 * 2 + MOE_BF16: return launch_gate_up_typed<MOE_F32, MOE_BF16>(a, sms, s);
    case MOE_BF16 * 2 + MOE_F32: return launch_gate_up_typed<MOE_BF16, MOE_F32>(a, sms, s);
    case MOE_BF16 * 2 + MOE_BF16: return launch_gate_up_typed<MOE_BF16, MOE_BF16>(a, sms, s);
    case MOE_FP8E4M3_B128 * 2 + MOE_F32: return launch_gate_up_typed<MOE_FP8E4M3_B128, MOE_F32>(a, sms, s);
    case MOE_FP8E4M3_B128 * 2 + MOE_BF16: return launch_gate_up_typed<MOE_FP8E4M3_B128, MOE_BF16>(a, sms, s);
  }
  return cudaErrorInvalidValue;
}

bool down_combine_fits(const Shape& sh, int T) {
  const int V = sh.wdtype == MOE_F32 ? 4 : sh.wdtype == MOE_BF16 ? 8 : 16;
  return T * sh.k + T * sh.n_shared <= kDCMaxPairs && sh.I / V <= 32 * kDCChunks;
}

template <int WT>
cudaError_t launch_down_bulk(const GemvArgs& a, const BulkGeom& geo, bool ring, bool pdl, const float* w,
                             const float* cpu, float* out, uint32_t* err, cudaStream_t s) {
  if (!ring) {   // same rows per CTA, no ring and h read through L1: a few KB of shared memory
    BulkGeom d = geo;
    d.NS = 0;
    d.NW = 16;
    const size_t shift = geo.plan_off - geo.ring_off;
    d.plan_off -= shift;
    d.extra_off -= shift;
    d.smem -= shift;
    if (d.h_smem) {
      d.smem -= (size_t)(a.P + a.T * a.n_shared) * a.I * 4;
      d.h_smem = 0;
    }
    auto go1 = [&](auto kern) -> cudaError_t {
      if (pdl) return launch_pdl(kern, dim3(d.grid), dim3(d.NW * 32), d.smem, s, a, d, w, cpu, out, err);
      kern<<<d.grid, d.NW * 32, d.smem, s>>>(a, d, w, cpu, out, err);
      return cudaGetLastError();
    };
    // bf16 or fp8 rows of 3 or 4 16-byte chunks per lane: the straight-line variant,
    // 8 warps (measured against 4 warps, and against plain launches of both, on the
    // DeepSeek-V3 slice: 3593 layer-steps/s against 3546-3576; the guarded path 3459)
    if constexpr (WT == MOE_BF16 || WT == MOE_FP8E4M3_B128) {
      const int nch = (int)(a.I / WFmt<WT>::V);
      d.NW = 8;
      if (nch == 96) return go1(down_bulk_kernel<WT, false, 3>);
      if (nch == 128) return go1(down_bulk_kernel<WT, false, 4>);
      d.NW = 16;
    }
    return go1(down_bulk_kernel<WT, false, 0>);
  }
  auto go = [&](auto kern, int threads) -> cudaError_t {
    if (pdl) return launch_pdl(kern, dim3(geo.grid), dim3(threads), geo.smem, s, a, geo, w, cpu, out, err);
    kern<<<geo.grid, threads, geo.smem, s>>>(a, geo, w, cpu, out, err);
    return cudaGetLastError();
  };
  if constexpr (WT == MOE_FP8E4M3_B128) {   // the same for fp8 rows of 3 or 4 chunks per lane
    const int nch = a.I / 16;
    if (geo.RS <= 8 && nch == 96) return go(down_bulk_kernel<WT, true, 3, false, true>, geo.NW * 32);
    if (geo.RS <= 8 && nch == 128) return go(down_bulk_kernel<WT, true, 4, false, true>, geo.NW * 32);
  }
  if constexpr (WT == MOE_BF16) {   // rows of 3 or 4 chunks per lane: the unguarded straight-line path
    const int nch = a.I / 8;
    // one stage per expert for at most 8 experts: two warps per stage, 8 rows each
    const bool pair = geo.NS == 1 && geo.NW == 8 && a.max_g <= 8 && geo.R <= 16 && geo.nsb == 1;
    if (nch == 96)
      return pair ? go(down_bulk_kernel<WT, true, 3, true>, 512) : go(down_bulk_kernel<WT, true, 3>, geo.NW * 32);
    if (nch == 128)
      return pair ? go(down_bulk_kernel<WT, true, 4, true>, 512) : go(down_bulk_kernel<WT, true, 4>, geo.NW * 32);
  }
  return go(down_bulk_kernel<WT, true, 0>, geo.NW * 32);
}

cudaError_t launch_down_bulk_any(const Shape& sh, const GemvArgs& a, const BulkGeom& geo, bool ring, bool pdl,
                                 const float* w, const float* cpu, float* out, uint32_t* err, cudaStream_t s) {
  if (sh.wdtype == MOE_F32) return launch_down_bulk<MOE_F32>(a, geo, ring, pdl, w, cpu, out, err, s);
  if (sh.wdtype == MOE_BF16) return launch_down_bulk<MOE_BF16>(a, geo, ring, pdl, w, cpu, out, err, s);
  if (sh.wdtype == MOE_NVFP4) return launch_down_bulk<MOE_NVFP4>(a, geo, ring, pdl, w, cpu, out, err, s);
  if (sh.wdtype == MOE_MXFP4) return launch_down_bulk<MOE_MXFP4>(a, geo, ring, pdl, w, cpu, out, err, s);
  return launch_down_bulk<MOE_FP8E4M3_B128>(a, geo, ring, pdl, w, cpu, out, err, s);
}


// The bulk down kernel runs when its ring fits and every pair's h fits in
// shared memory, or, for one token, when only the ring fits: each warp then
// reads its pair's h through L1 (the DeepSeek-V3 shape: 9 pairs x 2048 fp32 =
// 72 KB of h).  The split into resident / filled grids rides on it.
bool down_split_ok(const Shape& sh, int T, int sms) {
  const GemvArgs a = make_args(sh, 2, T, nullptr, DecodeBufs{});
  const BulkGeom geo = down_geom(a, sh.wdtype, sms);
  return geo.NS >= 1 && (geo.h_smem || T == 1);
}

cudaError_t launch_down_split(const Shape& sh, int pass, int T, const float* w, const float* cpu_part, DecodeBufs b,
                              float* out, uint32_t* err, int sms, cudaStream_t s, bool pdl) {
  if (pass != 0 && pass != 1) return cudaErrorInvalidValue;
  const GemvArgs a = make_args(sh, pass, T, nullptr, b);
  const BulkGeom geo = down_geom(a, sh.wdtype, sms);
  // pass 0 follows its gate/up grid, pass 1 the fill, as programmatic dependencies
  // unless `pdl` is false
  return launch_down_bulk_any(sh, a, geo, pass == 0, pdl, w, cpu_part, out, err, s);
}


int down_combine_launches(const Shape& sh, int T, int sms) {
  const GemvArgs a = make_args(sh, 2, T, nullptr, DecodeBufs{});
  const BulkGeom geo = down_geom(a, sh.wdtype, sms);
  if (geo.NS >= 1) return 1;
  if (down_combine_fits(sh, T) && sh.wdtype != MOE_NVFP4 && sh.wdtype != MOE_MXFP4) return 1;
  return 2;
}

// Geometry of resident_fused_kernel, or NS = 0 when the call does not take it: bf16
// weights and activations, one token, no shared expert, at most 8 resident
// experts (one down stage per warp), gate/up rows of 4 or 8 16-byte chunks per
// lane, W_down rows of 3 or 4, and the row blocks of the split down kernels.
FusedGeom fused_geom(const GemvArgs& a, int wdtype, int adtype, int sms) {
  FusedGeom f{};
  if (wdtype != MOE_BF16 || adtype != MOE_BF16 || a.T != 1 || a.n_shared != 0 || a.max_g > kFusedWarps) return f;
  if (a.H % 256 != 0 || (a.H / 256 != 4 && a.H / 256 != 8) || a.I % 256 != 0 || (a.I / 256 != 3 && a.I / 256 != 4))
    return f;
  const BulkGeom dg = down_geom(a, wdtype, sms);
  if (dg.NS < 1 || !dg.h_smem || dg.grid > sms || dg.R < 1 || dg.R > kDownRows) return f;
  f.R = dg.R;
  f.nblk = dg.grid;
  f.SBG = up128(2 * wrow(MOE_BF16, (size_t)a.H));
  f.SBD = up128((size_t)f.R * wrow(MOE_BF16, (size_t)a.I));
  const size_t np = (size_t)a.P;
  const size_t plan = up128(staged_plan_bytes(a.max_g, a.max_p));
  const size_t xb = up128((size_t)a.H * 2);
  const size_t extra = up128(np * 8) + up128((size_t)f.R * np * 4 + np);
  f.NS = 2;
  const size_t ring = std::max((size_t)kFusedWarps * f.NS * f.SBG, (size_t)kFusedWarps * f.SBD);
  f.ring_off = 256;
  f.plan_off = f.ring_off + ring;
  f.x_off = f.plan_off + plan;
  f.extra_off = f.x_off + xb;
  f.smem = f.extra_off + extra;
  if (f.smem > kFusedSmemMax) f.NS = 0;
  return f;
}

bool resident_fused_ok(const Shape& sh, int T, int sms) {
  const GemvArgs a = make_args(sh, 0, T, nullptr, DecodeBufs{});
  return fused_geom(a, sh.wdtype, sh.adtype, sms).NS > 0;
}

cudaError_t launch_resident_fused(const Shape& sh, int T, const void* x, const float* w, const float* cpu_part,
                                  DecodeBufs b, float* out, uint32_t* err, int sms, cudaStream_t s) {
  const GemvArgs a = make_args(sh, 0, T, x, b);
  const FusedGeom g = fused_geom(a, sh.wdtype, sh.adtype, sms);
  if (g.NS == 0 || b.fused_bar == nullptr) return cudaErrorInvalidValue;
  const dim3 grid(sms), block(kFusedWarps * 32);
  const int jx = a.H / 256, jn = a.I / 256;
  if (jx == 8 && jn == 3) return launch_pdl(resident_fused_kernel<8, 3>, grid, block, g.smem, s, a, g, w, cpu_part, out, err);
  if (jx == 8 && jn == 4) return launch_pdl(resident_fused_kernel<8, 4>, grid, block, g.smem, s, a, g, w, cpu_part, out, err);
  if (jx == 4 && jn == 3) return launch_pdl(resident_fused_kernel<4, 3>, grid, block, g.smem, s, a, g, w, cpu_part, out, err);
  return launch_pdl(resident_fused_kernel<4, 4>, grid, block, g.smem, s, a, g, w, cpu_part, out, err);
}



cudaError_t launch_down_combine(const Shape& sh, int T, const float* w, const float* cpu_part, DecodeBufs b,
                                float* out, uint32_t* err, int sms, cudaStream_t s) {
  {
    // The bulk down kernel whenever its ring fits.  When not every pair's h fits in
    // shared memory (more than two tokens at the Qwen3 shape) each warp reads the
    // h of its item's pairs through L1, once per item of up to kDownRows rows;
    // down_combine_kernel reads it once per row.
    const GemvArgs a = make_args(sh, 2, T, nullptr, b);
    const BulkGeom geo = down_geom(a, sh.wdtype, sms);
    if (geo.NS >= 1) return launch_down_bulk_any(sh, a, geo, true, true, w, cpu_part, out, err, s);
  }
  if (down_combine_fits(sh, T) && sh.wdtype != MOE_NVFP4 && sh.wdtype != MOE_MXFP4) {
    const GemvArgs a = make_args(sh, 2, T, nullptr, b);
    if (sh.wdtype == MOE_F32) return launch_down_combine_typed<MOE_F32>(a, w, cpu_part, out, err, sms, s);
    if (sh.wdtype == MOE_BF16) return launch_down_combine_typed<MOE_BF16>(a, w, cpu_part, out, err, sms, s);
    return launch_down_combine_typed<MOE_FP8E4M3_B128>(a, w, cpu_part, out, err, sms, s);
  }
  // large batches: down projection of every GPU expert, then the separate combine
  const GemvArgs a = make_args(sh, 2, T, nullptr, b);
  cudaError_t e;
  if (sh.wdtype == MOE_F32) e = launch_down_typed<MOE_F32>(a, sms, s);
  else if (sh.wdtype == MOE_BF16) e = launch_down_typed<MOE_BF16>(a, sms, s);
  else if (sh.wdtype == MOE_NVFP4) e = launch_down_typed<MOE_NVFP4>(a, sms, s);
  else if (sh.wdtype == MOE_MXFP4) e = launch_down_typed<MOE_MXFP4>(a, sms, s);
  else e = launch_down_typed<MOE_FP8E4M3_B128>(a, sms, s);
  if (e != cudaSuccess || b.defer_combine) return e;   // deferred: the combine follows the CPU branch
  return launch_combine(sh, T, w, cpu_part, b, out, err, s);
}

cudaError_t launch_fill(const Shape& sh, const int32_t* plan, const int32_t* fills,
                        const uint8_t* host_pool_dev, const uint64_t* offsets, uint8_t* slots,
                        int n_ctas, cudaStream_t s) {
  return launch_copy_blobs(plan + P_Q, nullptr, fills, host_pool_dev, offsets, slots, sh.S, n_ctas, s);
}

cudaError_t launch_copy_blobs(const int32_t* count, const int32_t* skip, const int32_t* list,
                              const uint8_t* host_pool_dev, const uint64_t* offsets, uint8_t* slots,
                              uint64_t S, int n_ctas, cudaStream_t s) {
  copy_blobs_kernel<<<n_ctas, 512, 0, s>>>(count, skip, list, host_pool_dev, offsets, slots, S);
  return cudaGetLastError();
}

cudaError_t launch_fp4_to_bf16(const Shape& sh, const int32_t* wslot, const int32_t* active, const int32_t* offsets,
                               const uint8_t* slots, uint16_t* staging, int sms, cudaStream_t s) {
  // Two 256-thread blocks per SM leave thread slots for the next layer's copy
  // CTAs, which run beside this pass (MXFP4 chunk of 8192 tokens: 84.1-84.4 ms
  // wall against 90.8-91.7 with 8 blocks per SM and 93.9-94.1 with 1).
  const int grid = sms * 2;
  if (sh.wdtype == MOE_NVFP4)
    fp4_to_bf16_kernel<MOE_NVFP4><<<grid, 256, 0, s>>>(wslot, active, offsets, sh.E, sh.H, sh.I, slots, sh.S, staging);
  else if (sh.wdtype == MOE_MXFP4)
    fp4_to_bf16_kernel<MOE_MXFP4><<<grid, 256, 0, s>>>(wslot, active, offsets, sh.E, sh.H, sh.I, slots, sh.S, staging);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_expert_gemv(const Shape& sh, int pass, int T, const void* x, DecodeBufs b,
                               int sms, cudaStream_t s) {
  const GemvArgs a = make_args(sh, pass, T, x, b);
  if (sh.wdtype == MOE_F32 && sh.adtype == MOE_F32) return launch_gemv_typed<MOE_F32, MOE_F32>(a, sms, s);
  if (sh.wdtype == MOE_F32 && sh.adtype == MOE_BF16) return launch_gemv_typed<MOE_F32, MOE_BF16>(a, sms, s);
  if (sh.wdtype == MOE_BF16 && sh.adtype == MOE_F32) return launch_gemv_typed<MOE_BF16, MOE_F32>(a, sms, s);
  if (sh.wdtype == MOE_BF16 && sh.adtype == MOE_BF16) return launch_gemv_typed<MOE_BF16, MOE_BF16>(a, sms, s);
  if (sh.wdtype == MOE_FP8E4M3_B128 && sh.adtype == MOE_F32)
    return launch_gemv_typed<MOE_FP8E4M3_B128, MOE_F32>(a, sms, s);
  if (sh.wdtype == MOE_FP8E4M3_B128 && sh.adtype == MOE_BF16)
    return launch_gemv_typed<MOE_FP8E4M3_B128, MOE_BF16>(a, sms, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const Shape& sh, int T, const float* w, const float* cpu_part,
                           DecodeBufs b, float* out, uint32_t* err, cudaStream_t s) {
  const long n = (long)T * (sh.H / 4);
  const int threads = 256;
  const long want = (n + threads - 1) / threads;
  const int grid = (int)(want < 152L * 8 ? want : 152L * 8);
  combine_kernel<<<grid, threads, 0, s>>>(T, sh.H, sh.k, sh.n_shared, w, b.slot_map, b.y, cpu_part, out, err);
  return cudaGetLastError();
}

}  // namespace moe
