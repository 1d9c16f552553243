// Runtime cache reconfiguration: rebuild the slot pool for a new slot count.
//
// Follows the snackonai deep dive "FreeToken, or why your laptop was never the
// bottleneck", section "Resizing the cache without a restart" (rebuild the
// expert cache to a new slot count; safe because the host copy of every expert
// is authoritative: a smaller cache only costs speed) and the
// ai.thesatyajit.com article, section "Elastic memory, because the machine is
// not yours" (the rebuild happens between steps, and the host pool is not
// loaded again).
//
// Reading: keep the min(C_new, resident) most recently used experts, packed
// into slots 0.. in ascending old-slot order, each with its recency stamp;
// the remaining new slots are empty.
//
// The survivor choice runs on the device in one CTA: count resident slots,
// radix-select the N-th largest stamp (stamps of resident slots are unique),
// then a block-wide scan gives each survivor its new index.  A copy kernel
// moves the survivors' blobs into the new pool and a scatter rebuilds the
// flat-id -> slot table.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kThreads = 1024;

struct ResizeScalars {
  int resident, digit, kth;
};

__global__ void __launch_bounds__(kThreads, 1)
resize_plan_kernel(int C_old, int C_new, const int32_t* __restrict__ s2e, const uint64_t* __restrict__ stamp,
                   int32_t* __restrict__ new_s2e, uint64_t* __restrict__ new_stamp,
                   int32_t* __restrict__ new2old, int32_t* __restrict__ n_keep) {
  __shared__ ResizeScalars sc;
  __shared__ unsigned int hist[256];
  __shared__ int part[kThreads];
  const int tid = threadIdx.x, lane = tid & 31, nt = blockDim.x;
  if (tid == 0) sc.resident = 0;
  __syncthreads();
  int mine = 0;
  unsigned long long maxst = 0ull;
  for (int s = tid; s < C_old; s += nt) {
    if (s2e[s] >= 0) { ++mine; maxst = max(maxst, (unsigned long long)stamp[s]); }
  }
  atomicAdd(&sc.resident, mine);
  // the largest stamp bounds the digits to scan
  __shared__ unsigned long long smax;
  if (tid == 0) smax = 0ull;
  __syncthreads();
  atomicMax(&smax, maxst);
  __syncthreads();
  const int R = sc.resident;
  const int N = min(C_new, R);
  // threshold: the N-th largest stamp = the (R - N + 1)-th smallest among resident slots
  unsigned long long thr = 0ull;
  if (N > 0 && N < R) {
    const int top = smax ? 63 - __clzll((long long)smax) : 0;
    unsigned long long prefix = 0ull, maskhi = 0ull;
    int kth = R - N + 1;
    for (int shift = (top / 8) * 8; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += nt) hist[i] = 0u;
      __syncthreads();
      for (int s = tid; s < C_old; s += nt) {
        if (s2e[s] < 0) continue;
        const unsigned long long key = stamp[s];
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
    thr = prefix;
  }
  // survivors in ascending old slot: contiguous ranges per thread + block scan
  const int per = (C_old + nt - 1) / nt;
  const int s0 = min(C_old, tid * per), s1 = min(C_old, s0 + per);
  auto survives = [&](int s) { return s2e[s] >= 0 && (N == R || (N > 0 && stamp[s] >= thr)); };
  int cnt = 0;
  for (int s = s0; s < s1; ++s) cnt += survives(s) ? 1 : 0;
  part[tid] = cnt;
  __syncthreads();
  if (tid < 32) {  // exclusive scan of 1024 partial counts by one warp
    int running = 0;
    for (int b = 0; b < nt; b += 32) {
      const int v = part[b + lane];
      int incl = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      part[b + lane] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  int j = part[tid];
  for (int s = s0; s < s1; ++s) {
    if (survives(s)) {
      new_s2e[j] = s2e[s];
      new_stamp[j] = stamp[s];
      new2old[j] = s;
      ++j;
    }
  }
  for (int i = N + tid; i < C_new; i += nt) { new_s2e[i] = -1; new_stamp[i] = 0ull; }
  if (tid == 0) *n_keep = N;
}

__global__ void __launch_bounds__(512) resize_copy_kernel(const int32_t* __restrict__ new2old,
                                                          const int32_t* __restrict__ n_keep,
                                                          const uint8_t* __restrict__ old_slots,
                                                          uint8_t* __restrict__ new_slots, uint64_t S) {
  const int n = *n_keep;
  const uint64_t n16 = S >> 4;
  const uint64_t per = (n16 + gridDim.x - 1) / gridDim.x;
  const uint64_t c0 = per * blockIdx.x, c1 = min(n16, c0 + per);
  for (int j = 0; j < n; ++j) {
    const uint4* src = reinterpret_cast<const uint4*>(old_slots + (size_t)new2old[j] * S);
    uint4* dst = reinterpret_cast<uint4*>(new_slots + (size_t)j * S);
    for (uint64_t c = c0 + threadIdx.x; c < c1; c += blockDim.x) dst[c] = src[c];
  }
}

__global__ void rebuild_e2s_kernel(int C_new, const int32_t* __restrict__ new_s2e, int32_t* __restrict__ e2s) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < C_new; j += gridDim.x * blockDim.x) {
    const int f = new_s2e[j];
    if (f >= 0) e2s[f] = j;
  }
}

}  // namespace

cudaError_t launch_resize_plan(int C_old, int C_new, int32_t* s2e, uint64_t* stamp, int32_t* new_s2e,
                               uint64_t* new_stamp, int32_t* new2old, int32_t* n_keep, cudaStream_t s) {
  resize_plan_kernel<<<1, kThreads, 0, s>>>(C_old, C_new, s2e, stamp, new_s2e, new_stamp, new2old, n_keep);
  return cudaGetLastError();
}

cudaError_t launch_resize_copy(const int32_t* new2old, const int32_t* n_keep, int C_new,
                               const uint8_t* old_slots, uint8_t* new_slots, uint64_t S, cudaStream_t s) {
  (void)C_new;
  resize_copy_kernel<<<4 * 152, 512, 0, s>>>(new2old, n_keep, old_slots, new_slots, S);
  return cudaGetLastError();
}

cudaError_t launch_rebuild_e2s(int n_flat, int C_new, const int32_t* new_s2e, int32_t* e2s, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(e2s, 0xff, (size_t)n_flat * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  rebuild_e2s_kernel<<<(C_new + 255) / 256, 256, 0, s>>>(C_new, new_s2e, e2s);
  return cudaGetLastError();
}

}  // namespace moe
