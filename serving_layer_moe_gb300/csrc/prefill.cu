// Full-layer double-buffered prefill over the shared slot pool, with a
// TMA-fed tcgen05 grouped GEMM.
//
// Follows the ai.thesatyajit.com article "FreeToken: a 753B model on one GPU,
// and the two bandwidths that decide everything", section "Prefill: hide the
// pool behind the wire" (the decode cache's slot pool lends room for two whole
// layers; as the GPU computes layer l, a copy stream brings in every expert of
// layer l+1, before l+1's routing exists; the experts left resident after the
// prefill are where decode starts), the snackonai deep dive "FreeToken, or why
// your laptop was never the bottleneck", section "The Architecture, Unpacked",
// decision two (one pool for both; when it is too small for two whole layers,
// experts load as they are needed), and the signalovernoise
// newsletter "FreeToken: treat the whole PC as one" (same mechanism).
//
// Readings:
//   * a "buffer" is the set of E pool slots holding one layer; experts of the
//     layer that are already resident stay where they are; the missing ones
//     are loaded into LRU victims that exclude every slot of layers l and l+1.
//   * the call for layer l loads what is missing of l (normally nothing: the
//     previous call prefetched it), starts loading all missing experts of l+1
//     on the transfer stream, runs the grouped GEMM of l on the caller's
//     stream, and marks all E experts of l used (ascending e), then the
//     prefetched experts of l+1 (ascending e).
//   * on-demand mode (C < 2E): the routed experts of l in ascending order, in
//     groups of at most C; each group is loaded into victims that exclude its
//     own resident slots, computed, and marked used.
//   * without the second buffer (moe_cache_set_prefill_prefetch(cache, 0), the
//     ablation both pages quote: 19 % at 4k, 25 % at 8k, 26 % at 16k tokens on
//     their 5090): the call for layer l loads only what is missing of l, into
//     victims that exclude the slots of l, and computes once those loads are
//     done, so loads and computation run one after the other.
//
// The expert is the SwiGLU of the decode path: h = silu(x W_gate^T) * (x W_up^T)
// stored as bf16, y = h W_down^T in fp32, out[t] = sum_j w[t,j] y[t,j].
//
// GB300 design of the GEMM (one CTA per SM, persistent):
//   rows of x are gathered per expert into a contiguous bf16 matrix, and each
//   expert's rows are cut into 128-row tiles (the last one partial: its
//   epilogue keeps only the expert's own rows); tiles of 128 rows x 256
//   columns x 64-deep K slices are staged by TMA (128-byte swizzle) into a
//   shared-memory ring (4 stages for GEMM 1, 3 for GEMM 2), multiplied by
//   tcgen05.mma (kind::f16, bf16 in, fp32 accumulate, M=128 N=256 K=16) issued
//   by one thread into a double-buffered TMEM accumulator (2 x 256 columns),
//   and drained with tcgen05.ld by 8 (GEMM 1) or 16 (GEMM 2) epilogue warps,
//   several per 32-lane TMEM quarter, while the next tile's MMAs run.  The
//   expert's weights are read straight out of its pool slot through one tensor
//   map over the whole pool (the slot picks the row coordinate).
//   GEMM 1 (gate|up, N = 128 gate + 128 up columns of the same rows) fuses
//   SwiGLU into its epilogue and writes h as bf16; GEMM 2 (down) multiplies by
//   the router gate in its epilogue and adds its rows into out with bulk
//   reductions (cp.reduce.async.bulk .add.f32 of 128-byte row pieces): the k
//   contributions of a token arrive from k different experts, so their order
//   varies from run to run.
//   4-bit experts (NVFP4, MXFP4) are first decoded to a bf16 staging area by
//   fp4_to_bf16_kernel and the GEMMs read that instead of the pool.
//   Every wait on an mbarrier is bounded by the GPU global timer; on timeout
//   the kernel flags the error word, drains its own copies and frees TMEM.
#include "cache.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <vector>

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int GEMM_THREADS = 320;             // GEMM 1: warp 0 TMA, warp 1 MMA, warps 2-9 epilogue (two per TMEM lane quarter)
constexpr int GEMM2_THREADS = 576;            // GEMM 2: warps 2-17 epilogue (four per TMEM lane quarter)
constexpr int GEMM2_STAGES = 3;               // GEMM 2's short K (I) needs fewer stages; the room goes to staging
constexpr int TMEM_COLS = 512;                // two 128 x 256 fp32 accumulators
constexpr size_t GEMM_SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256;
constexpr size_t GEMM2_SMEM = (size_t)GEMM2_STAGES * STAGE_BYTES + 1024 + 256 +
                              (size_t)(GEMM2_THREADS - 64) * 144;   // + a 128-byte reduce staging buffer per epilogue thread
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s bound on any wait

struct PrefillState {
  int P_max = 0, max_mtiles = 0;
  uint16_t* xs = nullptr;       // [P_max, H] bf16 rows of x, grouped by expert
  uint16_t* hs = nullptr;       // [P_max, I] bf16 SwiGLU activations
  int32_t* ibuf = nullptr;      // one allocation for the int32 arrays below
  int32_t* perm = nullptr;      // [P_max] pair id of each grouped row
  int32_t* counts = nullptr;    // [E]
  int32_t* offsets = nullptr;   // [E + 1]
  int32_t* cursor = nullptr;    // [E]
  int32_t* mtiles = nullptr;    // [max_mtiles * 4] (expert, row begin, row end, 0)
  int32_t* n_mtiles = nullptr;  // [1]
  int32_t* wslot = nullptr;     // [E] slot of each expert of the layer (-1 = not loaded)
  int32_t* active = nullptr;    // [E] expert computed in this round
  int32_t* loads = nullptr;     // [2 * 2E] (flat id, slot): this layer's loads, then prefetch
  int32_t* n_loads = nullptr;   // [2] loads of this layer, prefetched loads of the next
  uint16_t* wbf = nullptr;      // 4-bit experts: [E, 3IH] bf16 blobs the GEMMs read, expert e at e * 3IH
  int32_t* ident = nullptr;     // 4-bit experts: [E] = 0..E-1, the GEMMs' "slot" of expert e in wbf
  CUtensorMap tm_a1, tm_a2, tm_b1, tm_b2;
  const void* b_maps_pool = nullptr;  // pool the B maps were built for
  uint64_t b_maps_C = 0;
  cudaEvent_t ev_ctrl = nullptr, ev_cur = nullptr;
  bool prefetch_next = true;    // full-layer mode: the second buffer (next layer loads during this one)
};

PrefillState* state_of(moe_cache* c) { return static_cast<PrefillState*>(c->prefill); }

// ---------------------------------------------------------------------------
// small PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait on the phase of the given parity; false on timeout or abort
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > kWaitNs) return false;
    }
  }
}
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major, M x N
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// the grouped GEMM
// ---------------------------------------------------------------------------
struct GemmArgs {
  const int32_t* mtiles;
  const int32_t* n_mtiles;
  const int32_t* wslot;
  int n_ntiles;           // N tiles per expert
  int kblocks;            // K / 64
  int b_rows_per_slot;    // rows of the pool view per slot
  int b_row_off;          // first row of this matrix inside a slot
  int b_half_off;         // row offset of the second 128-row half of a B tile
  int b_n_step;           // rows per N tile
  // epilogue 0 (SwiGLU -> bf16)
  uint16_t* hs;
  int I;
  // epilogue 1 (gate-weighted accumulate)
  const int32_t* perm;
  const float* w;
  float* out;
  int H, k;
  uint32_t* err;
};

template <int EPI>
__global__ void __launch_bounds__(EPI == 0 ? GEMM_THREADS : GEMM2_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs a) {
  constexpr int STAGES = EPI == 0 ? ::moe::STAGES : GEMM2_STAGES;
  constexpr int NEPI = EPI == 0 ? 8 : 16;         // epilogue warps; NEPI / 4 of them share a TMEM lane quarter
  constexpr int CSPLIT = NEPI / 4;                // ... and split its columns
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], 32 * NEPI); }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = *a.n_mtiles * a.n_ntiles;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int armed_stage[STAGES], armed_phase[STAGES], narmed = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const int mt = tile / a.n_ntiles, nt = tile % a.n_ntiles;
      const int e = a.mtiles[4 * mt], r0 = a.mtiles[4 * mt + 1];
      const int brow = a.wslot[e] * a.b_rows_per_slot + a.b_row_off + nt * a.b_n_step;
      for (int kb = 0; kb < a.kblocks; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        mbar_expect_tx(&full[stage], STAGE_BYTES);
        tma_load_2d(&tmA, &full[stage], sa, kb * BK, r0);
        tma_load_2d(&tmB, &full[stage], sb, kb * BK, brow);
        tma_load_2d(&tmB, &full[stage], sb + B_BYTES / 2, kb * BK, brow + a.b_half_off);
        armed_stage[narmed % STAGES] = stage;
        armed_phase[narmed % STAGES] = (int)phase;
        ++narmed;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr_system(a.err, kErrTimeout);
      // let our own copies land before the CTA exits
      const int n = narmed < STAGES ? narmed : STAGES;
      for (int i = 0; i < n; ++i) {
        const int j = (narmed - 1 - i) % STAGES;
        const unsigned long long t0 = gtimer();
        while (!mbar_test(&full[armed_stage[j]], (uint32_t)armed_phase[j]) && gtimer() - t0 < kWaitNs) {
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
      fence_after();
      const uint32_t d = tmem + (uint32_t)(acc * BN);
      for (int kb = 0; kb < a.kblocks; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
        fence_after();
        const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16(d, sdesc(sa + kk * 32), sdesc(sb + kk * 32), (kb | kk) != 0 ? 1u : 0u);
        umma_commit(&empty[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      umma_commit(&tfull[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) { *abort_flag = 1; atomicOr_system(a.err, kErrTimeout); }
  } else if (warp >= 2) {
    // ---------------- epilogue: 4 warps, one TMEM lane (= tile row) per thread ----------------
    const int sub = warp & 3;
    const int part = (warp - 2) >> 2;   // which column share of the lane quarter
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
        *abort_flag = 1;
        atomicOr_system(a.err, kErrTimeout);
        break;
      }
      fence_after();
      const int mt = tile / a.n_ntiles, nt = tile % a.n_ntiles;
      const int r0 = a.mtiles[4 * mt + 1], r1 = a.mtiles[4 * mt + 2];
      const int row = r0 + 32 * sub + lane;
      const bool valid = row < r1;
      const uint32_t tbase = tmem + ((uint32_t)(32 * sub) << 16) + (uint32_t)(acc * BN);
      if (EPI == 0) {
        uint16_t* dst = a.hs + (size_t)row * a.I + (size_t)nt * (BN / 2);
#pragma unroll 1
        for (int c = part * (BN / 2 / CSPLIT); c < (part + 1) * (BN / 2 / CSPLIT); c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c, g);
          tmem_ld32(tbase + BN / 2 + c, u);
          tmem_ld_wait();
          if (valid) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float h0 = g0 / (1.0f + expf(-g0)) * __uint_as_float(u[2 * i]);
              const float h1 = g1 / (1.0f + expf(-g1)) * __uint_as_float(u[2 * i + 1]);
              const __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
              packed[i] = *reinterpret_cast<const uint32_t*>(&hb);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
          }
        }
      } else {
        int t = 0;
        float wt = 0.f;
        if (valid) {
          const int p = a.perm[row];
          t = p / a.k;
          wt = a.w[p];
        }
        // Each row's 32 gated columns go through this thread's 128-byte staging
        // buffer into one bulk reduce-add on the row of out: the TMA unit does the
        // fp32 adds in L2 as one contiguous 128-byte request, and the thread moves
        // on (it only waits for the buffer to have been read before refilling it).
        float* dst = a.out + (size_t)t * a.H + (size_t)nt * BN;
        // (thread stride 144 B: the eight 16-byte stores of a warp spread over all banks)
        float4* stg = reinterpret_cast<float4*>(smem + STAGES * STAGE_BYTES + 256) + (threadIdx.x - 64) * 9;
#pragma unroll 1
        for (int c = part * (BN / CSPLIT); c < (part + 1) * (BN / CSPLIT); c += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          tmem_ld_wait();
          if (valid) {
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 8; ++i)
              stg[i] = make_float4(wt * __uint_as_float(v[4 * i]), wt * __uint_as_float(v[4 * i + 1]),
                                   wt * __uint_as_float(v[4 * i + 2]), wt * __uint_as_float(v[4 * i + 3]));
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 128;" ::"l"(dst + c),
                         "r"(smem_u32(stg))
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      }
      fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (EPI == 1) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // every reduce has landed
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// routing: group the T*k (token, expert) pairs by expert
// ---------------------------------------------------------------------------
__global__ void route_count_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ counts,
                                   uint32_t* err) {
  bool bad = false;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E) atomicAdd(&counts[e], 1);
    else bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr_system(err, kErrBadExpertId);
}

__global__ void route_scan_kernel(const int32_t* __restrict__ counts, int E, int32_t* __restrict__ offsets,
                                  int32_t* __restrict__ cursor) {
  // one warp: exclusive scan over E counts
  const int lane = threadIdx.x;
  int running = 0;
  for (int b = 0; b < E; b += 32) {
    const int e = b + lane;
    const int c = e < E ? counts[e] : 0;
    int incl = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (e < E) { offsets[e] = running + incl - c; cursor[e] = running + incl - c; }
    running += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) offsets[E] = running;
}

__global__ void route_scatter_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ cursor,
                                     int32_t* __restrict__ perm) {
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E) perm[atomicAdd(&cursor[e], 1)] = p;
  }
}

// xs[row] = x[token of perm[row]], one warp per row, 16-byte moves
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ offsets, int E, int H, int k,
                                   uint16_t* __restrict__ xs) {
  const int rows = offsets[E];
  const int lane = threadIdx.x & 31;
  const int n16 = H / 8;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += (gridDim.x * blockDim.x) >> 5) {
    const int t = perm[r] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)r * H);
    for (int c = lane; c < n16; c += 32) dst[c] = __ldg(src + c);
  }
}

// m-tiles of the active experts: (expert, first row, end row)
__global__ void tiles_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ active, int E,
                             int32_t* __restrict__ mtiles, int32_t* __restrict__ n_mtiles) {
  const int lane = threadIdx.x;
  int running = 0;
  for (int b = 0; b < E; b += 32) {
    const int e = b + lane;
    int nt = 0, r0 = 0, r1 = 0;
    if (e < E && active[e]) {
      r0 = offsets[e];
      r1 = offsets[e + 1];
      nt = (r1 - r0 + BM - 1) / BM;
    }
    int incl = nt;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int base = running + incl - nt;
    for (int i = 0; i < nt; ++i) {
      int* m = mtiles + 4 * (base + i);
      m[0] = e;
      m[1] = r0 + i * BM;
      m[2] = r1;
      m[3] = 0;
    }
    running += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) *n_mtiles = running;
}

// ---------------------------------------------------------------------------
// prefill control: which experts to load where, recency, per-expert slots
// ---------------------------------------------------------------------------
struct PCtrlArgs {
  int layer, L, E, C, T, k, full_layer, round;
  int prefetch_next;              // full-layer mode: also load layer + 1 (the second buffer)
  const int32_t* ids;
  CacheTables tab;
  int32_t* loads;
  int32_t* n_loads;
  int32_t* wslot;
  int32_t* active;
  uint32_t* err;
};

struct PCtrlScalars {
  int n_cur, n_nxt, u, g0, g1, digit, kth, ncand;
  unsigned long long clock0;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// One CTA.  Shared memory: need flags/lists over 2E experts, routed bitmap, radix histogram, candidates.
__global__ void __launch_bounds__(1024, 1) prefill_control_kernel(PCtrlArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ PCtrlScalars sc;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  const int E = a.E, NW = (E + 31) >> 5;
  uint32_t* ebits = reinterpret_cast<uint32_t*>(smem);           // [NW] routed (on-demand mode)
  uint32_t* ebase = ebits + NW;                                    // [NW + 1]
  int32_t* need = reinterpret_cast<int32_t*>(ebase + NW + 1);      // [2E] flat ids to load, in order
  int32_t* grp = need + 2 * E;                                     // [E] flat ids of the group (on-demand)
  uint32_t* hist = reinterpret_cast<uint32_t*>(grp + E);           // [256]
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(
      (reinterpret_cast<uintptr_t>(hist + 256) + 7) & ~uintptr_t(7));  // [2E]

  const int fbase = a.layer * E;
  const bool has_next = a.full_layer && a.prefetch_next && (a.layer + 1 < a.L);
  int32_t* e2s = a.tab.e2s;
  int32_t* s2e = a.tab.s2e;
  uint64_t* stamp = a.tab.stamp;

  if (tid == 0) { sc.clock0 = *a.tab.clock; sc.ncand = 0; }
  for (int i = tid; i < NW; i += nt) ebits[i] = 0u;
  for (int e = tid; e < E; e += nt) { a.wslot[e] = -1; a.active[e] = 0; }
  __syncthreads();

  // ---- which experts: full layer (l, then l+1) or this round's group of routed experts ----
  int lo = 0, hi = 0;  // flat-id range protected from eviction (full-layer mode)
  if (a.full_layer) {
    if (tid < 32) {  // missing experts of l, then of l+1, each in ascending e
      int base = 0;
      for (int half = 0; half < (has_next ? 2 : 1); ++half) {
        const int f0 = fbase + half * E;
        for (int c0 = 0; c0 < E; c0 += 32) {
          const int i = c0 + lane;
          const bool miss = i < E && e2s[f0 + i] < 0;
          const uint32_t bm = __ballot_sync(0xffffffffu, miss);
          if (miss) need[base + __popc(bm & lanemask_lt())] = f0 + i;
          base += __popc(bm);
        }
        if (half == 0 && lane == 0) sc.n_cur = base;
      }
      if (lane == 0) sc.n_nxt = base - sc.n_cur;
    }
    lo = fbase;
    hi = fbase + (has_next ? 2 * E : E);
    for (int e = tid; e < E; e += nt) a.active[e] = 1;
  } else {
    const int P = a.T * a.k;
    for (int p = tid; p < P; p += nt) {
      const int e = a.ids[p];
      if ((unsigned)e < (unsigned)E) atomicOr(&ebits[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (tid < 32) {
      int running = 0;
      for (int w0 = 0; w0 < NW; w0 += 32) {
        const int w = w0 + lane;
        const int c = w < NW ? __popc(ebits[w]) : 0;
        int incl = c;
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (w < NW) ebase[w] = running + incl - c;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        sc.u = running;
        sc.g0 = min(running, a.round * a.C);
        sc.g1 = min(running, (a.round + 1) * a.C);
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) {
      const uint32_t wb = ebits[e >> 5];
      if (wb & (1u << (e & 31))) {
        const int idx = ebase[e >> 5] + __popc(wb & ((1u << (e & 31)) - 1u));
        if (idx >= sc.g0 && idx < sc.g1) { grp[idx - sc.g0] = fbase + e; a.active[e] = 1; }
      }
    }
    __syncthreads();
    if (tid < 32) {
      int base = 0;
      const int ng = sc.g1 - sc.g0;
      for (int c0 = 0; c0 < ng; c0 += 32) {
        const int i = c0 + lane;
        const bool miss = i < ng && e2s[grp[i]] < 0;
        const uint32_t bm = __ballot_sync(0xffffffffu, miss);
        if (miss) need[base + __popc(bm & lanemask_lt())] = grp[i];
        base += __popc(bm);
      }
      if (lane == 0) { sc.n_cur = base; sc.n_nxt = 0; }
    }
  }
  __syncthreads();
  const int n_cur = sc.n_cur, n_nxt = sc.n_nxt, nneed = n_cur + n_nxt;

  // ---- victims: the nneed smallest (stamp, slot) keys among unprotected slots ----
  auto key_of = [&](int s) -> unsigned long long {
    const int f = s2e[s];
    if (a.full_layer) {
      if (f >= lo && f < hi) return ~0ull;
    } else if (f >= fbase && f < fbase + E && a.active[f - fbase]) {
      return ~0ull;
    }
    return ((unsigned long long)stamp[s] << kSlotBits) | (unsigned long long)s;
  };
  if (nneed > 0) {
    const unsigned long long maxkey = (sc.clock0 << kSlotBits) | (kMaxSlots - 1);
    const int top = 63 - __clzll((long long)maxkey);
    unsigned long long prefix = 0ull, maskhi = 0ull;
    int kth = nneed;
    for (int shift = (top / 8) * 8; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += nt) hist[i] = 0u;
      __syncthreads();
      for (int s = tid; s < a.C; s += nt) {
        const unsigned long long key = key_of(s);
        if ((key & maskhi) == prefix) atomicAdd(&hist[(key >> shift) & 255ull], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        int c = 0;
        for (int j = 0; j < 8; ++j) c += (int)hist[lane * 8 + j];
        int incl = c;
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const int excl = incl - c;
        if (excl < kth && kth <= incl) {
          int run = excl, d = lane * 8;
          for (int j = 0; j < 8; ++j) {
            const int hj = (int)hist[lane * 8 + j];
            if (run + hj >= kth) { d = lane * 8 + j; break; }
            run += hj;
          }
          sc.digit = d;
          sc.kth = kth - run;
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)sc.digit << shift;
      maskhi |= 255ull << shift;
      kth = sc.kth;
      __syncthreads();
    }
    for (int s = tid; s < a.C; s += nt) {
      const unsigned long long key = key_of(s);
      if (key <= prefix) {
        const int i = atomicAdd(&sc.ncand, 1);
        if (i < nneed) cand[i] = key;
      }
    }
    __syncthreads();
    // rank, then assign need[r] -> victim of rank r
    for (int i = tid; i < nneed; i += nt) {
      const unsigned long long ki = cand[i];
      int r = 0;
      for (int j = 0; j < nneed; ++j) r += (cand[j] < ki);
      const int v = (int)(ki & (kMaxSlots - 1));
      a.loads[2 * r] = need[r];
      a.loads[2 * r + 1] = v;
    }
    __syncthreads();  // loads[] complete (global, same CTA)
    for (int r = tid; r < nneed; r += nt) {
      const int v = a.loads[2 * r + 1];
      const int old = s2e[v];
      if (old >= 0) e2s[old] = -1;
    }
    __syncthreads();
    for (int r = tid; r < nneed; r += nt) {
      const int f = a.loads[2 * r];
      const int v = a.loads[2 * r + 1];
      s2e[v] = f;
      e2s[f] = v;
    }
  }
  __syncthreads();

  // ---- recency, per-expert slots, counters ----------------------------------------
  const unsigned long long c0 = sc.clock0;
  if (a.full_layer) {
    for (int e = tid; e < E; e += nt) {
      const int s = e2s[fbase + e];
      stamp[s] = c0 + (unsigned long long)e + 1ull;
      a.wslot[e] = s;
    }
    for (int r = tid; r < n_nxt; r += nt) stamp[a.loads[2 * (n_cur + r) + 1]] = c0 + (unsigned long long)(E + r) + 1ull;
    if (tid == 0) *a.tab.clock = c0 + (unsigned long long)(E + n_nxt);
  } else {
    const int ng = sc.g1 - sc.g0;
    for (int i = tid; i < ng; i += nt) {
      const int f = grp[i];
      const int s = e2s[f];
      stamp[s] = c0 + (unsigned long long)i + 1ull;
      a.wslot[f - fbase] = s;
    }
    if (tid == 0) *a.tab.clock = c0 + (unsigned long long)ng;
  }
  if (tid == 0) {
    a.n_loads[0] = n_cur;
    a.n_loads[1] = n_nxt;
    a.tab.counters[7] += (uint64_t)nneed;
    if (nneed > 0 && sc.ncand < nneed) atomicOr_system(a.err, kErrCapacity);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D bf16 map over rows of `cols` elements, box 64 x 128, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {BK, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool fp4_weights(const moe_cache* c) { return c->sh.wdtype == MOE_NVFP4 || c->sh.wdtype == MOE_MXFP4; }

// The B maps view bf16 expert blobs as rows: the slot pool itself, or for 4-bit
// experts the bf16 staging area (fixed; built once).
moe_status refresh_b_maps(moe_cache* c) {
  PrefillState* ps = state_of(c);
  const uint64_t H = c->sh.H, I = c->sh.I;
  if (fp4_weights(c)) {
    if (ps->b_maps_pool == ps->wbf) return MOE_OK;
    const uint64_t E = c->sh.E;
    if (!make_map(&ps->tm_b1, ps->wbf, H, E * 3 * I) || !make_map(&ps->tm_b2, ps->wbf, I, E * 3 * H))
      return fail(MOE_ECUDA, "cuTensorMapEncodeTiled failed for the bf16 staging area");
    ps->b_maps_pool = ps->wbf;
    return MOE_OK;
  }
  if (ps->b_maps_pool == c->slots && ps->b_maps_C == c->C) return MOE_OK;
  if (!make_map(&ps->tm_b1, c->slots, H, c->C * 3 * I) || !make_map(&ps->tm_b2, c->slots, I, c->C * 3 * H))
    return fail(MOE_ECUDA, "cuTensorMapEncodeTiled failed for the slot pool");
  ps->b_maps_pool = c->slots;
  ps->b_maps_C = c->C;
  return MOE_OK;
}

}  // namespace

moe_status prefill_init(moe_cache* c) {
  const moe_config& k = c->cfg;
  if ((k.wdtype != MOE_BF16 && k.wdtype != MOE_NVFP4 && k.wdtype != MOE_MXFP4) || k.adtype != MOE_BF16)
    return fail(MOE_EINVAL, "prefill needs bf16, nvfp4 or mxfp4 weights and bf16 activations");
  if (k.hidden % BN || k.inter % 128)
    return fail(MOE_EINVAL, "prefill needs H a multiple of 256 and I a multiple of 128");
  if (!get_encode()) return fail(MOE_ECUDA, "cuTensorMapEncodeTiled is not available");
  PrefillState* ps = new PrefillState();
  c->prefill = ps;
  const int E = k.n_experts;
  ps->P_max = k.max_prefill_tokens * k.top_k;
  ps->max_mtiles = (ps->P_max + BM - 1) / BM + E;
  CK(moe_malloc(&ps->xs, (size_t)ps->P_max * k.hidden * 2));
  CK(moe_malloc(&ps->hs, (size_t)ps->P_max * k.inter * 2));
  const size_t ints = (size_t)ps->P_max + E + (E + 1) + E + (size_t)ps->max_mtiles * 4 + 1 + E + E + 4 * E + 2;
  CK(moe_malloc(&ps->ibuf, ints * 4));
  CK(cudaMemset(ps->ibuf, 0, ints * 4));
  int32_t* p = ps->ibuf;
  ps->perm = p; p += ps->P_max;
  ps->counts = p; p += E;
  ps->offsets = p; p += E + 1;
  ps->cursor = p; p += E;
  ps->mtiles = p; p += (size_t)ps->max_mtiles * 4;
  ps->n_mtiles = p; p += 1;
  ps->wslot = p; p += E;
  ps->active = p; p += E;
  ps->loads = p; p += 4 * E;
  ps->n_loads = p; p += 2;
  c->dev_bytes += (size_t)ps->P_max * (k.hidden + k.inter) * 2 + ints * 4;
  if (fp4_weights(c)) {
    const size_t wb = (size_t)E * 3 * k.inter * k.hidden * 2;
    CK(moe_malloc(&ps->wbf, wb));
    CK(moe_malloc(&ps->ident, (size_t)E * 4));
    std::vector<int32_t> id(E);
    for (int e = 0; e < E; ++e) id[e] = e;
    CK(cudaMemcpy(ps->ident, id.data(), (size_t)E * 4, cudaMemcpyHostToDevice));
    c->dev_bytes += wb + (size_t)E * 4;
  }
  if (!make_map(&ps->tm_a1, ps->xs, k.hidden, ps->P_max) || !make_map(&ps->tm_a2, ps->hs, k.inter, ps->P_max))
    return fail(MOE_ECUDA, "cuTensorMapEncodeTiled failed for the activation buffers");
  CK(cudaEventCreateWithFlags(&ps->ev_ctrl, cudaEventDisableTiming));
  CK(cudaEventCreateWithFlags(&ps->ev_cur, cudaEventDisableTiming));
  CK(cudaFuncSetAttribute(grouped_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GEMM_SMEM));
  CK(cudaFuncSetAttribute(grouped_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GEMM2_SMEM));
  CK(cudaFuncSetAttribute(prefill_control_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
  return refresh_b_maps(c);
}

void prefill_free(moe_cache* c) {
  PrefillState* ps = state_of(c);
  if (!ps) return;
  cudaFree(ps->xs);
  cudaFree(ps->hs);
  cudaFree(ps->ibuf);
  cudaFree(ps->wbf);
  cudaFree(ps->ident);
  if (ps->ev_ctrl) cudaEventDestroy(ps->ev_ctrl);
  if (ps->ev_cur) cudaEventDestroy(ps->ev_cur);
  delete ps;
  c->prefill = nullptr;
}

// the two GEMMs of one round over the m-tiles of the active experts
static moe_status run_gemms(moe_cache* c, int T, const float* w, float* out, cudaStream_t s) {
  PrefillState* ps = state_of(c);
  const Shape& sh = c->sh;
  GemmArgs g{};
  g.mtiles = ps->mtiles;
  g.n_mtiles = ps->n_mtiles;
  g.wslot = fp4_weights(c) ? ps->ident : ps->wslot;
  g.hs = ps->hs;
  g.I = sh.I;
  g.perm = ps->perm;
  g.w = w;
  g.out = out;
  g.H = sh.H;
  g.k = sh.k;
  g.err = c->err_dev;
  (void)T;
  // GEMM 1: [rows, H] x W_gu^T; a 256-wide N tile = 128 gate rows + the 128 up rows I further on
  g.n_ntiles = sh.I / (BN / 2);
  g.kblocks = sh.H / BK;
  g.b_rows_per_slot = 3 * sh.I;
  g.b_row_off = 0;
  g.b_half_off = sh.I;
  g.b_n_step = BN / 2;
  grouped_gemm_kernel<0><<<c->sms, GEMM_THREADS, GEMM_SMEM, s>>>(ps->tm_a1, ps->tm_b1, g);
  CK(cudaGetLastError());
  // GEMM 2: [rows, I] x W_d^T; W_d rows start 2H rows into a slot (rows of I elements)
  g.n_ntiles = sh.H / BN;
  g.kblocks = sh.I / BK;
  g.b_rows_per_slot = 3 * sh.H;
  g.b_row_off = 2 * sh.H;
  g.b_half_off = BN / 2;
  g.b_n_step = BN;
  grouped_gemm_kernel<1><<<c->sms, GEMM2_THREADS, GEMM2_SMEM, s>>>(ps->tm_a2, ps->tm_b2, g);
  CK(cudaGetLastError());
  return MOE_OK;
}

}  // namespace moe

extern "C" moe_status moe_cache_set_prefill_prefetch(moe_cache* c, int32_t on) {
  using namespace moe;
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  PrefillState* ps = state_of(c);
  if (!ps) return fail(MOE_EINVAL, "prefill is disabled (max_prefill_tokens = 0)");
  if (on != 0 && on != 1) return fail(MOE_EINVAL, "on must be 0 or 1");
  ps->prefetch_next = on != 0;
  return MOE_OK;
}

extern "C" moe_status moe_layer_prefill(moe_cache* c, int32_t layer, int32_t T, const void* x, const int32_t* ids,
                                        const float* w, float* out, void* stream) {
  using namespace moe;
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  PrefillState* ps = state_of(c);
  if (!ps) return fail(MOE_EINVAL, "prefill is disabled (max_prefill_tokens = 0)");
  if (layer < 0 || layer >= c->sh.L) return fail(MOE_EINVAL, "layer %d out of range", layer);
  if (T < 0 || T > c->cfg.max_prefill_tokens) return fail(MOE_EINVAL, "T = %d outside [0, max_prefill_tokens]", T);
  if (*reinterpret_cast<volatile uint32_t*>(c->err_host)) {
    const uint32_t e = *reinterpret_cast<volatile uint32_t*>(c->err_host);
    *reinterpret_cast<volatile uint32_t*>(c->err_host) = 0;
    return fail(MOE_EDEVICE, "device flagged an earlier call (bits 0x%x)", e);
  }
  if (T == 0) return MOE_OK;
  if (!x || !ids || !w || !out) return fail(MOE_EINVAL, "x, topk_ids, topk_w and out must not be NULL");
  if (!aligned_to(x, 16) || !aligned_to(out, 16)) return fail(MOE_EINVAL, "x and out must be 16-byte aligned");
  if (!aligned_to(ids, 4) || !aligned_to(w, 4)) return fail(MOE_EINVAL, "topk_ids and topk_w must be 4-byte aligned");
  DeviceGuard guard(c->cfg.device);
  moe_status st = refresh_b_maps(c);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Shape& sh = c->sh;
  const int E = sh.E, P = T * sh.k;
  const bool full = c->C >= 2ull * (uint64_t)E;
  const int rounds = full ? 1 : (int)((E + c->C - 1) / c->C);

  {
    ProfScope p(c, s, PROF_PREFILL_CONTROL);
    CK(cudaMemsetAsync(out, 0, (size_t)T * sh.H * sizeof(float), s));
    // prefill rewrites slots and stamps by its own rules: the decode candidate pool is rebuilt afterwards
    CK(cudaMemsetAsync(c->tab.pool + kPoolN, 0, sizeof(uint64_t), s));
    CK(cudaMemsetAsync(ps->counts, 0, (size_t)E * 4, s));
    const int g = std::max(1, std::min(c->sms * 4, (P + 255) / 256));
    route_count_kernel<<<g, 256, 0, s>>>(ids, P, E, ps->counts, c->err_dev);
    route_scan_kernel<<<1, 32, 0, s>>>(ps->counts, E, ps->offsets, ps->cursor);
    route_scatter_kernel<<<g, 256, 0, s>>>(ids, P, E, ps->cursor, ps->perm);
    gather_rows_kernel<<<c->sms * 4, 256, 0, s>>>(static_cast<const uint16_t*>(x), ps->perm, ps->offsets, E,
                                                   sh.H, sh.k, ps->xs);
    CK(cudaGetLastError());
  }
  const int NW = (E + 31) / 32;
  const size_t csmem = (size_t)(2 * NW + 1) * 4 + (size_t)3 * E * 4 + 256 * 4 + 16 + (size_t)2 * E * 8 + 16;
  for (int r = 0; r < rounds; ++r) {
    {
      ProfScope p(c, s, PROF_PREFILL_CONTROL);
      PCtrlArgs a{};
      a.layer = layer; a.L = sh.L; a.E = E; a.C = (int)c->C; a.T = T; a.k = sh.k; a.full_layer = full ? 1 : 0;
      a.round = r; a.prefetch_next = ps->prefetch_next ? 1 : 0; a.ids = ids; a.tab = c->tab; a.loads = ps->loads; a.n_loads = ps->n_loads; a.wslot = ps->wslot;
      a.active = ps->active; a.err = c->err_dev;
      prefill_control_kernel<<<1, 1024, csmem, s>>>(a);
      CK(cudaGetLastError());
      tiles_kernel<<<1, 32, 0, s>>>(ps->offsets, ps->active, E, ps->mtiles, ps->n_mtiles);
      CK(cudaGetLastError());
    }
    CK(cudaEventRecord(ps->ev_ctrl, s));
    CK(cudaStreamWaitEvent(c->fill_stream, ps->ev_ctrl, 0));
    {
      ProfScope p(c, c->fill_stream, PROF_PREFILL_LOAD);
      CK(launch_copy_blobs(ps->n_loads, nullptr, ps->loads, c->host_pool_dev, c->offsets, c->slots, sh.S,
                           c->fill_ctas, c->fill_stream));
    }
    CK(cudaEventRecord(ps->ev_cur, c->fill_stream));
    if (full) {
      // start the next layer's full load; it overlaps this layer's GEMMs
      ProfScope p(c, c->fill_stream, PROF_PREFILL_LOAD);
      CK(launch_copy_blobs(ps->n_loads + 1, ps->n_loads, ps->loads, c->host_pool_dev, c->offsets, c->slots, sh.S,
                           c->fill_ctas, c->fill_stream));
    }
    CK(cudaStreamWaitEvent(s, ps->ev_cur, 0));
    {
      ProfScope p(c, s, PROF_PREFILL_GEMM);
      if (fp4_weights(c))   // this round's experts, now resident, decoded to bf16 for the GEMMs
        CK(launch_fp4_to_bf16(sh, ps->wslot, ps->active, ps->offsets, c->slots, ps->wbf, c->sms, s));
      st = run_gemms(c, T, w, out, s);
      if (st != MOE_OK) return st;
    }
  }
  return MOE_OK;
}
