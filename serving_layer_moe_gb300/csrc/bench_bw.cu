// Bandwidth calibration: B_P (host -> GPU expert transfer) and B_H (host-side
// expert read), and the hybrid recommendation.
//
// Follows the snackonai deep dive "FreeToken, or why your laptop was never the
// bottleneck", section "The Code, Annotated", subsection "Calibration decides
// the backend, not the GPU": measure the two bandwidths once per machine on
// the deployed expert shapes (not spec-sheet numbers) and recommend hybrid
// when B_H > 2 x B_P (threshold 2.0); and the ai.thesatyajit.com article,
// section "Decode: the one equation" (B_P = pinned expert-transfer bandwidth,
// B_H = host-side expert-processing bandwidth).
//
// Readings: B_P is timed through the library's own fill path (the SM copy
// kernel reading page-locked host memory) on expert-sized blobs; B_H is the
// rate at which all host threads can stream expert blobs out of host memory,
// the bytes an in-place CPU expert has to read.  (The CPU expert executor
// itself is not part of this library.)
#include "internal.cuh"

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstring>
#include <thread>
#include <vector>

extern "C" moe_status bench_bw(int32_t device, uint64_t expert_bytes, double* b_pcie_gbs, double* b_host_gbs,
                               int32_t* recommend_hybrid);

namespace {

double host_read_gbs(const uint8_t* buf, size_t bytes) {
  unsigned nthreads = std::max(1u, std::thread::hardware_concurrency());
  std::vector<std::thread> th;
  std::vector<uint64_t> sink(nthreads * 8, 0);
  double best = 0.0;
  for (int rep = 0; rep < 3; ++rep) {
    std::atomic<int> ready{0};
    std::atomic<bool> go{false};
    th.clear();
    std::vector<double> t0(nthreads), t1(nthreads);
    for (unsigned t = 0; t < nthreads; ++t) {
      th.emplace_back([&, t]() {
        const size_t per = (bytes / 64 / nthreads) * 64;
        const uint64_t* p = reinterpret_cast<const uint64_t*>(buf + per * t);
        const size_t n = per / 8;
        ready.fetch_add(1);
        while (!go.load(std::memory_order_acquire)) {
        }
        uint64_t a0 = 0, a1 = 0, a2 = 0, a3 = 0, a4 = 0, a5 = 0, a6 = 0, a7 = 0;
        for (size_t i = 0; i + 8 <= n; i += 8) {
          a0 ^= p[i]; a1 ^= p[i + 1]; a2 ^= p[i + 2]; a3 ^= p[i + 3];
          a4 ^= p[i + 4]; a5 ^= p[i + 5]; a6 ^= p[i + 6]; a7 ^= p[i + 7];
        }
        sink[t * 8] = a0 ^ a1 ^ a2 ^ a3 ^ a4 ^ a5 ^ a6 ^ a7;
      });
    }
    while (ready.load() < (int)nthreads) {
    }
    auto s = std::chrono::steady_clock::now();
    go.store(true, std::memory_order_release);
    for (auto& x : th) x.join();
    auto e = std::chrono::steady_clock::now();
    const double sec = std::chrono::duration<double>(e - s).count();
    const size_t moved = (bytes / 64 / nthreads) * 64 * nthreads;
    best = std::max(best, (double)moved / sec / 1e9);
  }
  volatile uint64_t keep = sink[0];
  (void)keep;
  return best;
}

}  // namespace

extern "C" moe_status bench_bw(int32_t device, uint64_t expert_bytes, double* b_pcie_gbs, double* b_host_gbs,
                               int32_t* recommend_hybrid) {
  if (expert_bytes == 0) return MOE_EINVAL;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MOE_EINVAL;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(device);
  const uint64_t S = (expert_bytes + 15) & ~uint64_t(15);
  // at least 1 GiB of distinct blobs, larger than the host's last-level cache
  const int nblob = (int)std::max<uint64_t>(8, ((1ull << 30) + S - 1) / S);
  const uint64_t total = S * (uint64_t)nblob;
  uint8_t* host = nullptr;
  uint8_t* dev = nullptr;
  int32_t* dplan = nullptr;
  int32_t* dfills = nullptr;
  uint64_t* doffs = nullptr;
  cudaStream_t st = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  moe_status rc = MOE_OK;
  double bp = 0.0, bh = 0.0;
  do {
    if (cudaHostAlloc(reinterpret_cast<void**>(&host), total, cudaHostAllocMapped) != cudaSuccess) { rc = MOE_ENOMEM; break; }
    for (uint64_t i = 0; i < total; i += 4096) host[i] = (uint8_t)(i >> 12);
    if (cudaMalloc(&dev, total) != cudaSuccess) { rc = MOE_ENOMEM; break; }
    std::vector<int32_t> plan(moe::P_COUNT, 0), fills(2 * nblob);
    std::vector<uint64_t> offs(nblob);
    plan[moe::P_Q] = nblob;
    for (int i = 0; i < nblob; ++i) { fills[2 * i] = i; fills[2 * i + 1] = i; offs[i] = (uint64_t)i * S; }
    if (cudaMalloc(&dplan, plan.size() * 4) != cudaSuccess || cudaMalloc(&dfills, fills.size() * 4) != cudaSuccess ||
        cudaMalloc(&doffs, offs.size() * 8) != cudaSuccess) { rc = MOE_ENOMEM; break; }
    cudaMemcpy(dplan, plan.data(), plan.size() * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dfills, fills.data(), fills.size() * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(doffs, offs.data(), offs.size() * 8, cudaMemcpyHostToDevice);
    void* hdev = nullptr;
    cudaHostGetDevicePointer(&hdev, host, 0);
    cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaDeviceProp prop;
    cudaGetDeviceProperties(&prop, device);
    moe::Shape sh{};
    sh.S = S;
    float best_ms = 1e30f;
    for (int rep = 0; rep < 4; ++rep) {
      cudaEventRecord(e0, st);
      moe::launch_fill(sh, dplan, dfills, static_cast<const uint8_t*>(hdev), doffs, dev, prop.multiProcessorCount / 2, st);
      cudaEventRecord(e1, st);
      if (cudaEventSynchronize(e1) != cudaSuccess) { rc = MOE_ECUDA; break; }
      float ms = 0.f;
      cudaEventElapsedTime(&ms, e0, e1);
      if (rep > 0) best_ms = std::min(best_ms, ms);
    }
    if (rc != MOE_OK) break;
    bp = (double)total / (best_ms * 1e-3) / 1e9;
    bh = host_read_gbs(host, total);
  } while (false);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (st) cudaStreamDestroy(st);
  cudaFree(dplan);
  cudaFree(dfills);
  cudaFree(doffs);
  cudaFree(dev);
  if (host) cudaFreeHost(host);
  cudaSetDevice(prev);
  if (rc != MOE_OK) return rc;
  if (b_pcie_gbs) *b_pcie_gbs = bp;
  if (b_host_gbs) *b_host_gbs = bh;
  if (recommend_hybrid) *recommend_hybrid = (bh > 2.0 * bp) ? 1 : 0;
  return MOE_OK;
}
