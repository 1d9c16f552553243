// Routing-control kernel of one decode MoE layer (one CTA, no host sync).
//
// Follows the snackonai deep dive "FreeToken, or why your laptop was never the
// bottleneck", section "The Architecture, Unpacked" (decision three: for each
// MoE layer a single kernel removes duplicate routed ids, looks them up in the
// residency table, computes q, chooses victims and maps every id to a slot or
// to the CPU; the victims, the K slots used longest ago, come out of a single
// pass) and section "The split policy itself"
// (q* = round(m B_P / B_H), clamp max(1, min(q, m)), the first q misses fill).
// Recency follows ai.thesatyajit.com "FreeToken: a 753B model on one GPU ...",
// section "Residency that follows the router": a hit makes an expert the most
// recent, a fill brings one in, an eviction drops the one unused longest.
//
// Readings (the pages leave these open):
//   * B_H = B_pcie + B_cpu, so q* = round_half_even(m B_pcie / (B_pcie + B_cpu))
//     in exact integer arithmetic; the clamp applies when m > 0; q is then
//     capped by K and by the evictable slots V = C - hits.
//   * Misses fill in ascending flat id; the i-th fill takes the i-th victim.
//   * LRU key of a slot = (stamp, slot); an empty slot has stamp 0; slots that
//     hold one of this call's hits are not evictable.  Victims = the K
//     smallest keys, ascending.
//   * After the rewrite every expert that runs on the GPU (hits, fills) is
//     stamped in ascending flat id with the next values of one global clock;
//     CPU-assigned experts are not touched.
//
// Design for one SM: everything the decision needs (the routed ids, this
// layer's slice of the flat-id -> slot table, every slot's LRU key, the clock)
// is loaded into shared memory in one parallel pass, so the critical path has
// a single global-memory round trip; the rest runs out of shared memory.  The
// routed set is a bitmap over E experts (dedup = atomicOr, order = popcount
// prefix), hit/miss ranks come from warp ballots (one thread per expert when
// the layer's experts fit the CTA).  Victims: for K <= kPoolMaxK the kernel
// keeps, between calls, the min(C, max(64, 4K)) smallest keys of its last full
// selection.  Keys only grow, so the first valid entries of that pool that are
// not this call's hits are the victims; the pool is rebuilt only when it runs
// short, and if even the rebuilt pool is short (more of this call's hits among
// its slots than it has room for) the call selects over all slots.  Above
// kPoolMaxK every call selects over all slots.  Both selections are an MSB
// radix select with 8-bit digits (keys held in registers up to 8 slots per
// thread), then a sort of the selected keys.  Calls of at most 32 routed pairs with K <= 16 (decode at
// small batch) take every step in one warp with ballots, match and warp
// barriers, after one block barrier that makes the loaded tables visible:
// 2.6 us less per call than the block-wide steps with their block barriers.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kSmemKeyCap = 12288;   // slots whose keys are cached in shared memory
constexpr size_t kCtrlSmemLimit = 200 * 1024;

struct CtrlArgs {
  int layer, T, k, E, C, K, n_shared;
  uint32_t bp, bc;
  uint64_t S;
  const int32_t* ids;
  CacheTables tab;
  DecodeBufs b;
  int32_t* slot_map_out;
  const uint8_t* slots_base;
  const uint8_t* shared_blob;   // this layer's shared expert, or null
  uint32_t* err;
  int umax;                     // min(E, T*k)
  int cache_keys;               // keys of all C slots fit in shared memory
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// round_half_even(m * bp / (bp + bc)) on integers (bp + bc > 0)
__device__ __forceinline__ uint32_t q_star(uint32_t m, uint32_t bp, uint32_t bc) {
  const uint64_t num = (uint64_t)m * bp;
  const uint64_t den = (uint64_t)bp + bc;
  uint64_t q, r;
  if ((num >> 32) == 0 && (den >> 32) == 0) {   // the 32-bit divide (the 64-bit one is a long routine)
    const uint32_t n32 = (uint32_t)num, d32 = (uint32_t)den;
    q = n32 / d32;
    r = n32 - (uint32_t)q * d32;
  } else {
    q = num / den;
    r = num - q * den;
  }
  if (2 * r > den) q += 1;
  else if (2 * r == den) q += (q & 1);
  return (uint32_t)q;
}


// LRU key of slot s for this call: (stamp << 20) | s, or all ones when s holds
// one of this call's routed experts (a hit: not evictable)
__device__ __forceinline__ unsigned long long key_of_fast(const CtrlArgs& a, const int32_t* slotf,
                                                          const unsigned long long* rawkey, const uint32_t* ebits,
                                                          int fbase, int E, int s) {
  const int f = a.cache_keys ? slotf[s] : a.tab.s2e[s];
  if (f >= fbase && f < fbase + E) {
    const int e = f - fbase;
    if (ebits[e >> 5] & (1u << (e & 31))) return ~0ull;
  }
  return a.cache_keys ? rawkey[s] : (((unsigned long long)a.tab.stamp[s] << kSlotBits) | (unsigned long long)s);
}

// shared scalars of the control CTA
struct CtrlScalars {
  int bad, u, h, m, q, keff, ncand, read_hits, read_misses, pool_n, enough;
  int rdigit[2], rkth[2], rstop[2];   // radix select: one result per pass, double-buffered
  unsigned long long clock0;
};

// kSel: 1 = radix select over all slots on every call (K > kPoolMaxK), 2 = K <=
// kPoolMaxK from the kept candidate pool (rebuilt by radix select when it runs short)
template <int kSel>
__global__ void __launch_bounds__(kCtrlThreads, 1) decode_control_kernel(CtrlArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ CtrlScalars sc;
  __shared__ unsigned long long wcand[2 * (kCtrlThreads / 32)];   // per-warp key minimum and maximum
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, NW = (E + 31) >> 5;
  const int P = a.T * a.k;
  const int U = a.umax;
  const int C = a.C;

  // shared layout (8-byte arrays first)
  unsigned long long* rawkey = reinterpret_cast<unsigned long long*>(smem);        // [C] if cached
  int32_t* slotf = reinterpret_cast<int32_t*>(rawkey + (a.cache_keys ? C : 0));   // [C] if cached
  int32_t* lslot = slotf + (a.cache_keys ? C : 0);                                 // [E] slot of each e of layer
  int32_t* pid = lslot + E;                                                        // [P] routed ids
  uint32_t* ebits = reinterpret_cast<uint32_t*>(pid + P);                          // [NW]
  uint32_t* ebase = ebits + NW;                                                    // [NW + 1]
  int32_t* uniq_e = reinterpret_cast<int32_t*>(ebase + NW + 1);                    // [U]
  int32_t* uniq_slot = uniq_e + U;                                                 // [U]
  int32_t* uniq_rank = uniq_slot + U;                                              // [U]
  int32_t* uniq_cls = uniq_rank + U;                                               // [U] 0 hit, 1 fill, 2 cpu
  int32_t* miss_list = uniq_cls + U;                                               // [U]
  int32_t* gcnt = miss_list + U;                                                   // [U + 2]
  int32_t* ecnt = gcnt + U + 2;                                                    // [E] routed pairs per expert
  int32_t* vict = ecnt + E;                                                        // [K]
  uint32_t* hist = reinterpret_cast<uint32_t*>(vict + a.K);                        // [2][256]
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(
      (reinterpret_cast<uintptr_t>(hist + 512) + 7) & ~uintptr_t(7));               // [max(K, kPoolN)]
  unsigned long long* s_pool = cand + (a.K > kPoolN ? a.K : kPoolN);               // [kPoolN]
  const int cand_cap = a.K > kPoolN ? a.K : kPoolN;

  int32_t* s2e = a.tab.s2e;
  uint64_t* stamp = a.tab.stamp;
  const int fbase = a.layer * E;

  // ---- 0. one parallel load of everything the decision reads ----------------
  // The residency tables were written by an earlier control kernel, not by the
  // kernel this one may overlap: they are loaded before waiting on the
  // predecessor.  Every thread issues all its loads (kB slots at a time) before
  // its first shared-memory store, so the preload costs one memory round trip
  // rather than one per loop iteration (2.3 us -> see the control section).
  {
    static_assert(kPoolN <= kCtrlThreads, "one pool entry per thread");
    constexpr int kB = 8;
    const int ncs = a.cache_keys ? C : 0;
    const unsigned long long clk = tid == 0 ? (unsigned long long)*a.tab.clock : 0ull;
    const int ls = tid < E ? a.tab.e2s[fbase + tid] : -1;
    unsigned long long pv = 0ull;
    int pn = 0;
    if (kSel == 2) {
      if (tid < pool_size(a.K, C)) pv = a.tab.pool[tid];   // the cache's pool size, not the capacity
      if (tid == 0) pn = (int)a.tab.pool[kPoolN];
    }
    int sv[kB];
    unsigned long long tv[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = tid + u * nt;
      if (i < ncs) { sv[u] = s2e[i]; tv[u] = stamp[i]; }
    }
    if (tid == 0) {
      sc.bad = 0; sc.ncand = 0; sc.read_hits = 0; sc.read_misses = 0;
      sc.clock0 = clk;
      if (kSel == 2) sc.pool_n = pn;
    }
    for (int i = tid; i < NW; i += nt) ebits[i] = 0u;
    for (int i = tid; i < U + 2; i += nt) gcnt[i] = 0;
    for (int i = tid; i < E; i += nt) ecnt[i] = 0;
    if (tid < E) lslot[tid] = ls;
    for (int e = tid + nt; e < E; e += nt) lslot[e] = a.tab.e2s[fbase + e];   // E above the CTA's threads
    if (kSel == 2 && tid < pool_size(a.K, C)) s_pool[tid] = pv;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = tid + u * nt;
      if (i < ncs) { slotf[i] = sv[u]; rawkey[i] = (tv[u] << kSlotBits) | (unsigned long long)i; }
    }
    for (int b0 = tid + kB * nt; b0 < ncs; b0 += kB * nt) {   // more than kB slots per thread
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int i = b0 + u * nt;
        if (i < ncs) { sv[u] = s2e[i]; tv[u] = stamp[i]; }
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int i = b0 + u * nt;
        if (i < ncs) { slotf[i] = sv[u]; rawkey[i] = (tv[u] << kSlotBits) | (unsigned long long)i; }
      }
    }
  }
  pdl_wait();       // the routed ids may come from the preceding kernel
  pdl_trigger();
  if (kSel == 2 && a.K <= kWarpPathMaxK && P + a.n_shared <= 32 && NW <= 32) {
    // ---- one warp for calls of at most 32 routed pairs ---------------------------
    // The steps below for a handful of pairs, in warp 0 with ballots and warp
    // barriers instead of block barriers.  Two block barriers remain: one makes
    // the tables loaded above visible to warp 0, the other publishes whether the
    // kept candidate pool holds enough victims.  If it does not, the pool must be
    // rebuilt with the whole CTA: every warp then runs the general path below
    // from its start (what warp 0 wrote here is rewritten or unchanged by it).
    __shared__ int s_fast;
    const uint32_t FULL = 0xffffffffu;
    const int e = lane < P ? a.ids[lane] : -1;   // in flight across the barrier
    __syncthreads();
    // per-lane state of warp 0: routed pair `lane`, unique expert `lane` (ascending)
    bool valid = false, hasu = false;
    int idx = -1, u = 0, h = 0, m = 0, q = 0, keff = 0, cls = 2, slot = -1, rank = 0;
    if (warp == 0) {
      valid = lane < P && (unsigned)e < (unsigned)E;
      if (valid) atomicOr(&ebits[e >> 5], 1u << (e & 31));
      __syncwarp();
      const uint32_t wb = lane < NW ? ebits[lane] : 0u;
      const int c = __popc(wb);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += v;
      }
      u = __shfl_sync(FULL, incl, 31);
      if (lane < NW) ebase[lane] = incl - c;
      if (lane == 0) ebase[NW] = u;
      __syncwarp();
      if (valid) {
        const uint32_t wbits = ebits[e >> 5];
        idx = ebase[e >> 5] + __popc(wbits & ((1u << (e & 31)) - 1u));
      }
      // the lowest lane of each routed expert writes its unique entry
      const uint32_t same = __match_any_sync(FULL, valid ? e : -1 - lane);
      if (valid && __ffs(same) - 1 == lane) { uniq_e[idx] = e; uniq_slot[idx] = lslot[e]; }
      __syncwarp();
      // classes and ranks in ascending flat id; the split q; the evictable count
      hasu = lane < u;
      const int usl = hasu ? uniq_slot[lane] : -1;
      const bool hit = hasu && usl >= 0, miss = hasu && usl < 0;
      const uint32_t bh = __ballot_sync(FULL, hit), bm = __ballot_sync(FULL, miss);
      h = __popc(bh);
      m = __popc(bm);
      rank = hit ? __popc(bh & lanemask_lt()) : __popc(bm & lanemask_lt());
      cls = hit ? 0 : 2;
      slot = usl;
      const int V = C - h;
      if (m > 0 && lane == 0) {
        q = (int)q_star((uint32_t)m, a.bp, a.bc);
        q = max(1, min(q, m));
        q = max(min(q, min(a.K, V)), 0);
      }
      q = __shfl_sync(FULL, q, 0);
      keff = max(0, min(a.K, V));
      // the keff smallest evictable keys: the first valid, non-hit entries of the pool
      int taken = 0;
      const int pn = sc.pool_n;
      for (int i0 = 0; i0 < pn && keff > 0; i0 += 32) {
        const int i = i0 + lane;
        const unsigned long long k = i < pn ? s_pool[i] : ~0ull;
        const bool ok = i < pn && key_of_fast(a, slotf, rawkey, ebits, fbase, E, (int)(k & (kMaxSlots - 1))) == k;
        const uint32_t bal = __ballot_sync(FULL, ok);
        const int r = taken + __popc(bal & lanemask_lt());
        if (ok && r < keff) vict[r] = (int)(k & (kMaxSlots - 1));
        taken += __popc(bal);
      }
      if (lane == 0) s_fast = taken >= keff;
    }
    __syncthreads();
    if (s_fast) {
      if (warp != 0) return;
      const int ns = a.n_shared;
      const int nfirst = h + ns;
      const int ngpu = nfirst + q;
      // victims, and the rewrite: the r-th miss (ascending flat id) fills victim r if r < q
      if (lane < a.K) a.b.victims[lane] = lane < keff ? vict[lane] : -1;
      if (hasu && cls == 2) {
        const int f = fbase + uniq_e[lane];
        if (rank < q) {
          const int v = vict[rank];
          const int old = a.cache_keys ? slotf[v] : s2e[v];
          if (old >= 0) a.tab.e2s[old] = -1;
          s2e[v] = f;
          a.tab.e2s[f] = v;
          slot = v;
          cls = 1;
          a.b.fills[2 * rank] = f;
          a.b.fills[2 * rank + 1] = v;
        } else {
          a.b.cpu[rank - q] = f;
        }
      }
      // recency: the GPU-run experts in ascending flat id take the next clock values
      const bool touched = hasu && cls < 2;
      const uint32_t bt = __ballot_sync(FULL, touched);
      const unsigned long long clock0 = sc.clock0;
      if (touched) stamp[slot] = clock0 + (unsigned long long)__popc(bt & lanemask_lt()) + 1ull;
      const int tb = __popc(bt);
      // GPU expert index: hits 0..h-1, the shared expert h, fills after
      const int g = cls == 0 ? rank : cls == 1 ? nfirst + rank : -1;
      if (g >= 0) a.b.gpu_w[g] = a.slots_base + (size_t)slot * a.S;
      if (ns && lane == 0) a.b.gpu_w[h] = a.shared_blob;
      if (hasu) { uniq_cls[lane] = cls; uniq_slot[lane] = slot; uniq_rank[lane] = g; }
      __syncwarp();
      // slot map, read counts, and the pair lists (ascending pair id within an expert)
      int pcls = 2, pslot = -1, pg = -1;
      if (valid) { pcls = uniq_cls[idx]; pslot = uniq_slot[idx]; pg = uniq_rank[idx]; }
      const int smv = pcls < 2 ? pslot : -1;
      if (lane < P) {
        a.b.slot_map[lane] = smv;
        if (a.slot_map_out) a.slot_map_out[lane] = smv;
      }
      const int read_hits = __popc(__ballot_sync(FULL, lane < P && pcls == 0));
      const uint32_t grp = __match_any_sync(FULL, pcls < 2 ? pg : -1 - lane);
      if (pcls < 2 && __ffs(grp) - 1 == lane) gcnt[pg] = __popc(grp);
      if (ns && lane == 0) gcnt[h] = a.T;
      __syncwarp();
      const int cg = lane < ngpu ? gcnt[lane] : 0;
      int incl = cg;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane < ngpu) a.b.gpu_off[lane] = incl - cg;
      if (lane == ngpu - 1) a.b.gpu_off[ngpu] = incl;
      if (ngpu == 0 && lane == 0) a.b.gpu_off[0] = 0;
      __syncwarp();
      if (lane < ngpu) gcnt[lane] = incl - cg;
      __syncwarp();
      if (pcls < 2) a.b.gpu_pairs[gcnt[pg] + __popc(grp & lanemask_lt())] = lane;
      if (ns && lane < a.T) a.b.gpu_pairs[gcnt[h] + lane] = P + lane;
      // plan scalars, counters, error word
      const bool bad_id = __ballot_sync(FULL, lane < P && !valid) != 0;
      if (lane == 0) {
        *a.tab.clock = clock0 + (unsigned long long)tb;
        int32_t* pl = a.b.plan;
        pl[P_LAYER] = a.layer; pl[P_U] = u; pl[P_H] = h; pl[P_M] = m; pl[P_Q] = q;
        pl[P_NCPU] = m - q; pl[P_NGPU] = ngpu; pl[P_NFIRST] = nfirst;
        unsigned long long* cn = reinterpret_cast<unsigned long long*>(a.tab.counters);
        atomicAdd(cn + 0, (unsigned long long)h);
        atomicAdd(cn + 1, (unsigned long long)m);
        atomicAdd(cn + 2, (unsigned long long)q);
        atomicAdd(cn + 3, (unsigned long long)(m - q));
        atomicAdd(cn + 4, (unsigned long long)read_hits);
        atomicAdd(cn + 5, (unsigned long long)(P - read_hits));
        atomicAdd(cn + 6, 1ull);
        uint32_t err = 0;
        if (bad_id) err |= kErrBadExpertId;
        if (((clock0 + tb) >> (64 - kSlotBits)) != 0ull) err |= kErrClock;
        if (err) atomicOr_system(a.err, err);
      }
      return;
    }
  }
  for (int p = tid; p < P; p += nt) pid[p] = a.ids[p];
  __syncthreads();

  // ---- 1. dedup: routed-expert bitmap and routed pairs per expert ---------
  for (int p = tid; p < P; p += nt) {
    const int e = pid[p];
    if ((unsigned)e >= (unsigned)E) {
      atomicOr(&sc.bad, 1);
    } else {
      atomicOr(&ebits[e >> 5], 1u << (e & 31));
      atomicAdd(&ecnt[e], 1);
    }
  }
  __syncthreads();
  int u, h, m, q, keff;
  // One thread per expert of the layer when E fits the CTA: thread e holds
  // whether e is routed, a hit or a miss, and its ranks among them in ascending
  // flat id (a ballot prefix over the warps), and takes every later step of e.
  const bool by_expert = E <= nt;
  __shared__ int s_wc[3][kCtrlThreads / 32];
  bool e_hit = false, e_miss = false, e_fill = false;
  int e_slot = -1, e_hrank = 0, e_mrank = 0, e_g = -1;
  if (by_expert) {
    // ---- 2. classification and ranks, one thread per expert ---------------
    const int e = tid;
    const bool present = e < E && ((ebits[e >> 5] >> (e & 31)) & 1u);
    e_slot = present ? lslot[e] : -1;
    e_hit = present && e_slot >= 0;
    e_miss = present && e_slot < 0;
    const uint32_t bpr = __ballot_sync(0xffffffffu, present);
    const uint32_t bht = __ballot_sync(0xffffffffu, e_hit);
    const uint32_t bms = __ballot_sync(0xffffffffu, e_miss);
    if (lane == 0) { s_wc[0][warp] = __popc(bpr); s_wc[1][warp] = __popc(bht); s_wc[2][warp] = __popc(bms); }
    __syncthreads();
    int pb = 0;
    u = 0; h = 0; m = 0;
#pragma unroll
    for (int w2 = 0; w2 < kCtrlThreads / 32; ++w2) {
      const int c0 = s_wc[0][w2], c1 = s_wc[1][w2], c2 = s_wc[2][w2];
      if (w2 < warp) { pb += c0; e_hrank += c1; e_mrank += c2; }
      u += c0; h += c1; m += c2;
    }
    const uint32_t lt = lanemask_lt();
    const int uidx = pb + __popc(bpr & lt);
    e_hrank += __popc(bht & lt);   // hits before e
    e_mrank += __popc(bms & lt);   // misses before e
    // ---- 3. the split q (every thread) -----------------------------------------
    const int V = C - h;  // slots this call may evict
    q = 0;
    if (m > 0) {
      q = (int)q_star((uint32_t)m, a.bp, a.bc);
      q = max(1, min(q, m));
      q = min(q, min(a.K, V));
      q = max(q, 0);
    }
    keff = max(0, min(a.K, V));
    if (present) {
      uniq_e[uidx] = e;
      if (e_miss) miss_list[e_mrank] = uidx;
    }
    if (e < E) lslot[e] = present ? uidx : -1;   // from here on: e -> its unique index
  } else {   // more experts than threads: the unique list from the bitmap's word prefix
    if (tid < 32) {  // exclusive popcount prefix over the bitmap words
      int running = 0;
      for (int w0 = 0; w0 < NW; w0 += 32) {
        const int w = w0 + lane;
        const int c = (w < NW) ? __popc(ebits[w]) : 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (w < NW) ebase[w] = running + incl - c;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) { ebase[NW] = running; sc.u = running; }
    }
    __syncthreads();
    u = sc.u;
    // ---- 2. unique list (ascending flat id) and classification --------------
    for (int e = tid; e < E; e += nt) {
      const uint32_t wbits = ebits[e >> 5];
      if (wbits & (1u << (e & 31))) {
        const int idx = ebase[e >> 5] + __popc(wbits & ((1u << (e & 31)) - 1u));
        uniq_e[idx] = e;
        uniq_slot[idx] = lslot[e];
      }
    }
    __syncthreads();
    if (tid < 32) {  // hit / miss ranks in ascending flat id
      int hb = 0, mb = 0;
      for (int c0 = 0; c0 < u; c0 += 32) {
        const int i = c0 + lane;
        const bool valid = i < u;
        const bool hit = valid && uniq_slot[i] >= 0;
        const bool miss = valid && !hit;
        const uint32_t bh = __ballot_sync(0xffffffffu, hit);
        const uint32_t bm = __ballot_sync(0xffffffffu, miss);
        if (hit) { uniq_rank[i] = hb + __popc(bh & lanemask_lt()); uniq_cls[i] = 0; }
        if (miss) {
          const int r = mb + __popc(bm & lanemask_lt());
          uniq_rank[i] = r;
          miss_list[r] = i;
          uniq_cls[i] = 2;
        }
        hb += __popc(bh);
        mb += __popc(bm);
      }
      if (lane == 0) {
        sc.h = hb;
        sc.m = mb;
        // ---- 3. the split q ----------------------------------------------------
        const int V = C - hb;  // slots this call may evict
        int q = 0;
        if (mb > 0) {
          q = (int)q_star((uint32_t)mb, a.bp, a.bc);
          q = max(1, min(q, mb));
          q = min(q, min(a.K, V));
          q = max(q, 0);
        }
        sc.q = q;
        sc.keff = max(0, min(a.K, V));
      }
    }
    __syncthreads();
    h = sc.h; m = sc.m; q = sc.q; keff = sc.keff;
  }

  // ---- 4. the K least-recently-used evictable slots, one pass ----------------
  // key(s) = (stamp << 20) | s, or all-ones when s holds one of this call's hits
  auto key_of = [&](int s) -> unsigned long long {
    const int f = a.cache_keys ? slotf[s] : s2e[s];
    if (f >= fbase && f < fbase + E) {
      const int e = f - fbase;
      if (ebits[e >> 5] & (1u << (e & 31))) return ~0ull;
    }
    return a.cache_keys ? rawkey[s] : (((unsigned long long)stamp[s] << kSlotBits) | (unsigned long long)s);
  };
  // The n_want smallest keys (keyfn; keys unique among the finite ones, n_want <=
  // number of finite keys), emitted ascending as emit(rank, key): MSB radix select
  // with 8-bit digits, then a rank sort of the candidates.
  //   * A thread keeps the keys of its slots in registers (C <= 8 threads' worth).
  //   * Each pass has two block barriers: the histograms and the per-pass results
  //     are double-buffered, and the next pass's histogram is cleared by warps
  //     1.. while warp 0 scans this one.
  //   * It stops as soon as the bucket holding the n_want-th key is needed whole:
  //     stamps are unique (only empty slots share stamp 0), so after the stamp's
  //     digits the buckets hold single keys.  The selected keys are then every key
  //     <= prefix | (bits below the last digit).
  auto radix_smallest = [&](int n_want, auto keyfn, auto emit) {
    constexpr int KPT = 8;
    const bool in_regs = C <= KPT * nt;
    unsigned long long mk[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int s = tid + j * nt;
      mk[j] = (in_regs && s < C) ? keyfn(s) : ~0ull;
    }
    const unsigned long long maxkey = (sc.clock0 << kSlotBits) | (kMaxSlots - 1);
    const int top = 63 - __clzll((long long)maxkey);
    // The bits above the highest bit where the smallest and the largest finite key
    // differ are the same for every finite key: the first digit is the 8 bits
    // ending at that bit (so the first pass spreads the keys over 256 buckets
    // instead of the few a byte-aligned top digit would use), the last digit may
    // be narrower.  (Keys in registers only; otherwise the top byte.)
    int hib = (top / 8) * 8 + 7;   // highest bit of the first digit
    unsigned long long prefix = 0ull, maskhi = 0ull;
    if (in_regs) {
      unsigned long long lo = ~0ull, hi = 0ull;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const unsigned long long key = mk[j];
        if (tid + j * nt < C && key != ~0ull) { lo = key < lo ? key : lo; hi = key > hi ? key : hi; }
      }
      const unsigned lhi = __reduce_min_sync(0xffffffffu, (unsigned)(lo >> 32));
      const unsigned llo = __reduce_min_sync(0xffffffffu, (unsigned)(lo >> 32) == lhi ? (unsigned)lo : ~0u);
      const unsigned hhi = __reduce_max_sync(0xffffffffu, (unsigned)(hi >> 32));
      const unsigned hlo = __reduce_max_sync(0xffffffffu, (unsigned)(hi >> 32) == hhi ? (unsigned)hi : 0u);
      if (lane == 0) { wcand[2 * warp] = ((unsigned long long)lhi << 32) | llo; wcand[2 * warp + 1] = ((unsigned long long)hhi << 32) | hlo; }
    }
    for (int i = tid; i < 256; i += nt) hist[i] = 0u;
    if (tid == 0) sc.ncand = 0;
    __syncthreads();
    if (in_regs) {
      unsigned long long lo = ~0ull, hi = 0ull;
      for (int w = 0; w < (nt >> 5); ++w) {
        lo = wcand[2 * w] < lo ? wcand[2 * w] : lo;
        hi = wcand[2 * w + 1] > hi ? wcand[2 * w + 1] : hi;
      }
      if (lo <= hi) {   // some finite key (always: n_want >= 1 finite keys)
        const unsigned long long diff = lo ^ hi;
        hib = diff ? 63 - __clzll((long long)diff) : 0;
        maskhi = hib + 1 >= 64 ? 0ull : ~((1ull << (hib + 1)) - 1ull);
        prefix = lo & maskhi;
      }
    }
    int kth = n_want;  // 1-based rank still to find below the current prefix
    int last_shift = 0;
    int pass = 0;
    for (int lo_bit = hib - 7;; lo_bit -= 8, ++pass) {
      const int shift = lo_bit > 0 ? lo_bit : 0;
      const unsigned long long dmask = (1ull << (lo_bit >= 0 ? 8 : 8 + lo_bit)) - 1ull;   // digit bits
      uint32_t* hc = hist + (pass & 1) * 256;
      uint32_t* hn = hist + ((pass + 1) & 1) * 256;
      if (in_regs) {
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
          const unsigned long long key = mk[j];
          if (tid + j * nt < C && (key & maskhi) == prefix) atomicAdd(&hc[(key >> shift) & dmask], 1u);
        }
      } else {
        for (int s = tid; s < C; s += nt) {
          const unsigned long long key = keyfn(s);
          if ((key & maskhi) == prefix) atomicAdd(&hc[(key >> shift) & dmask], 1u);
        }
      }
      if (warp != 0)
        for (int i = tid - 32; i < 256; i += nt - 32) hn[i] = 0u;
      __syncthreads();
      if (warp == 0) {
        int c = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) c += (int)hc[lane * 8 + j];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const int excl = incl - c;
        if ((excl < kth) && (kth <= incl)) {
          int run = excl, d = lane * 8;
          for (int j = 0; j < 8; ++j) {
            const int hj = (int)hc[lane * 8 + j];
            if (run + hj >= kth) { d = lane * 8 + j; break; }
            run += hj;
          }
          sc.rdigit[pass & 1] = d;
          sc.rkth[pass & 1] = kth - run;
          sc.rstop[pass & 1] = (int)hc[d] == kth - run;
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)sc.rdigit[pass & 1] << shift;
      maskhi |= dmask << shift;
      kth = sc.rkth[pass & 1];
      last_shift = shift;
      if (sc.rstop[pass & 1] || shift == 0) break;
    }
    // exactly n_want keys are <= thr
    const unsigned long long thr = prefix | ((1ull << last_shift) - 1ull);
    auto collect = [&](bool valid, unsigned long long key) {   // warp-uniform call
      const bool in = valid && key <= thr;
      const uint32_t bal = __ballot_sync(0xffffffffu, in);
      int base = 0;
      if (bal && lane == 0) base = atomicAdd(&sc.ncand, __popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      const int i = base + __popc(bal & lanemask_lt());
      if (in && i < n_want) cand[i] = key;
    };
    if (in_regs) {   // every ballot first, then one shared atomic per warp
      uint32_t bals[KPT];
      int tot = 0;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        bals[j] = __ballot_sync(0xffffffffu, tid + j * nt < C && mk[j] <= thr);
        tot += __popc(bals[j]);
      }
      int base = 0;
      if (lane == 0 && tot) base = atomicAdd(&sc.ncand, tot);
      base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        if ((bals[j] >> lane) & 1u) {
          const int i = base + __popc(bals[j] & lanemask_lt());
          if (i < n_want) cand[i] = mk[j];
        }
        base += __popc(bals[j]);
      }
    } else {
      for (int s0 = warp * 32; s0 < C; s0 += nt) {
        const int s = s0 + lane;
        collect(s < C, s < C ? keyfn(s) : ~0ull);
      }
    }
    __syncthreads();
    if (n_want > 128 && n_want <= nt && nt <= cand_cap) {
      // many candidates (a pool rebuild): bitonic sort of nt keys, one per thread,
      // the tail padded with all-ones keys.  Exchanges between lanes of a warp go
      // by shuffles; the 10 of 45 steps (for 512) between warps go through
      // shared memory.
      unsigned long long v = tid < n_want ? cand[tid] : ~0ull;
      for (int kk = 2; kk <= nt; kk <<= 1)
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
          unsigned long long pv;
          if (jj < 32) {
            pv = __shfl_xor_sync(0xffffffffu, v, jj);
          } else {
            __syncthreads();
            cand[tid] = v;
            __syncthreads();
            pv = cand[tid ^ jj];
          }
          const bool keep_min = ((tid & jj) == 0) == ((tid & kk) == 0);
          v = keep_min ? (v < pv ? v : pv) : (v > pv ? v : pv);
        }
      if (tid < n_want) emit(tid, v);
    } else {
      // ranks: four threads per candidate, each over a quarter of the list
      const int sub = tid & 3;
      for (int i0 = 0; i0 < n_want; i0 += nt >> 2) {   // uniform trip count
        const int i = i0 + (tid >> 2);
        const unsigned long long ki = i < n_want ? cand[i] : 0ull;
        int r = 0;
#pragma unroll 8
        for (int j = sub; j < n_want; j += 4) r += (cand[j] < ki);
        r += __shfl_xor_sync(0xffffffffu, r, 1);
        r += __shfl_xor_sync(0xffffffffu, r, 2);
        if (i < n_want && sub == 0) emit(r, ki);
      }
    }
    __syncthreads();
  };
  auto raw_key = [&](int s) -> unsigned long long {
    return a.cache_keys ? rawkey[s] : (((unsigned long long)stamp[s] << kSlotBits) | (unsigned long long)s);
  };
  if (kSel == 2 && keff > 0) {
    // Every slot outside the pool had a larger key than the pool's largest at the
    // rebuild, and a slot's key only changes by a new stamp from the clock, which
    // is larger still; so the valid entries (key unchanged) are exactly the slots
    // below that bound and the keff smallest evictable keys are the first keff
    // valid entries that are not this call's hits, whenever there are that many.
    // One entry per thread (n <= kPoolN = the CTA's threads); its rank among the
    // valid entries is a ballot prefix over the warps.
    __shared__ int s_wcnt[kCtrlThreads / 32];
    bool enough = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
      const int pn = sc.pool_n;
      const unsigned long long k = tid < pn ? s_pool[tid] : ~0ull;
      const bool ok = tid < pn && key_of((int)(k & (kMaxSlots - 1))) == k;
      const uint32_t bal = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) s_wcnt[warp] = __popc(bal);
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll
      for (int w2 = 0; w2 < kCtrlThreads / 32; ++w2) {
        const int c = s_wcnt[w2];
        before += w2 < warp ? c : 0;
        total += c;
      }
      const int r = before + __popc(bal & lanemask_lt());
      if (ok && r < keff) vict[r] = (int)(k & (kMaxSlots - 1));
      enough = total >= keff;   // the same in every thread
      if (enough || attempt == 1) break;
      // rebuild: the n smallest keys over all slots (hits included)
      const int n = pool_size(a.K, C);
      radix_smallest(n, raw_key, [&](int r2, unsigned long long key) {
        s_pool[r2] = key;
        a.tab.pool[r2] = key;
      });
      if (tid == 0) {
        sc.pool_n = n;
        a.tab.pool[kPoolN] = (uint64_t)n;
      }
      __syncthreads();
    }
    // More of this call's hits among the n oldest slots than n - keff: the exact
    // selection over all slots for this call
    if (!enough)
      radix_smallest(keff, key_of, [&](int r2, unsigned long long key) { vict[r2] = (int32_t)(key & (kMaxSlots - 1)); });
  } else if (kSel == 1 && keff > 0) {   // K above the pool's reach: the exact selection every call
    radix_smallest(keff, key_of, [&](int r, unsigned long long key) { vict[r] = (int32_t)(key & (kMaxSlots - 1)); });
  }
  for (int i = keff + tid; i < a.K; i += nt) vict[i] = -1;
  __syncthreads();

  // ---- 5.-6. rewrite, recency, GPU expert index -----------------------------
  // fills take victims in order, the rest go to the CPU; hits and fills in
  // ascending flat id take the next clock values; GPU expert index: hits
  // 0..h-1, the shared expert h, fills after
  const int ns = a.n_shared;
  const int nfirst = h + ns;
  for (int i = tid; i < a.K; i += nt) a.b.victims[i] = vict[i];
  if (by_expert) {
    const int e = tid;
    e_fill = e_miss && e_mrank < q;
    int slot = e_slot;
    if (e_fill) {
      const int f = fbase + e;
      const int v = vict[e_mrank];
      const int old = a.cache_keys ? slotf[v] : s2e[v];
      if (old >= 0) a.tab.e2s[old] = -1;
      s2e[v] = f;
      a.tab.e2s[f] = v;
      a.b.fills[2 * e_mrank] = f;
      a.b.fills[2 * e_mrank + 1] = v;
      slot = v;
    } else if (e_miss) {
      a.b.cpu[e_mrank - q] = fbase + e;
    }
    // e_hrank hits and min(e_mrank, q) fills come before e
    if (e_hit || e_fill) stamp[slot] = sc.clock0 + (unsigned long long)(e_hrank + min(e_mrank, q)) + 1ull;
    if (tid == 0) {
      *a.tab.clock = sc.clock0 + (unsigned long long)(h + q);
      if (((sc.clock0 + (unsigned long long)(h + q)) >> (64 - kSlotBits)) != 0ull) atomicOr(&sc.bad, 2);
    }
    e_g = e_hit ? e_hrank : e_fill ? nfirst + e_mrank : -1;
    if (e_g >= 0) a.b.gpu_w[e_g] = a.slots_base + (size_t)slot * a.S;
    const int ui = e < E ? lslot[e] : -1;
    if (ui >= 0) {
      uniq_cls[ui] = e_hit ? 0 : e_fill ? 1 : 2;
      uniq_slot[ui] = slot;
      uniq_rank[ui] = e_g;
    }
  } else {
    // ---- 5. rewrite: fills take victims in order, the rest go to the CPU ------
    for (int r = tid; r < m; r += nt) {
      const int i = miss_list[r];
      const int f = fbase + uniq_e[i];
      if (r < q) {
        const int v = vict[r];
        const int old = a.cache_keys ? slotf[v] : s2e[v];
        if (old >= 0) a.tab.e2s[old] = -1;
        s2e[v] = f;
        a.tab.e2s[f] = v;
        uniq_slot[i] = v;
        uniq_cls[i] = 1;
        a.b.fills[2 * r] = f;
        a.b.fills[2 * r + 1] = v;
      } else {
        a.b.cpu[r - q] = f;
      }
    }
    __syncthreads();

    // ---- 6. recency: stamp GPU-run experts in ascending flat id ---------------
    if (tid < 32) {
      int tb = 0;
      for (int c0 = 0; c0 < u; c0 += 32) {
        const int i = c0 + lane;
        const bool touched = (i < u) && uniq_cls[i] < 2;
        const uint32_t bt = __ballot_sync(0xffffffffu, touched);
        if (touched) stamp[uniq_slot[i]] = sc.clock0 + (unsigned long long)(tb + __popc(bt & lanemask_lt())) + 1ull;
        tb += __popc(bt);
      }
      if (lane == 0) {
        *a.tab.clock = sc.clock0 + (unsigned long long)tb;
        if (((sc.clock0 + tb) >> (64 - kSlotBits)) != 0ull) atomicOr(&sc.bad, 2);
      }
    }
    // GPU expert index of each unique: hits 0..h-1, shared expert h, fills after
    for (int i = tid; i < u; i += nt) {
      const int cls = uniq_cls[i];
      int g = -1;
      if (cls == 0) g = uniq_rank[i];
      else if (cls == 1) g = nfirst + uniq_rank[i];
      uniq_rank[i] = g;  // reuse: GPU expert index (or -1)
      if (g >= 0) a.b.gpu_w[g] = a.slots_base + (size_t)uniq_slot[i] * a.S;
    }
  }
  if (ns && tid == 0) a.b.gpu_w[h] = a.shared_blob;
  __syncthreads();

  // ---- 7. slot map and pair lists ---------------------------------------------
  const int ngpu = nfirst + q;
  if (by_expert) {
    // Pair counts of the hits and fills, exclusive prefix in GPU-index order
    // (hits in ascending flat id, the shared expert, fills in ascending flat id):
    // a warp scan per count and one block barrier; thread e keeps its expert's
    // offset as the write cursor of its pairs.  The order of an expert's pairs
    // within its list is not fixed (as in the other block-wide form): each pair's
    // values are formed on their own.
    const int e = tid;
    const int c = (e_hit || e_fill) ? ecnt[e] : 0;
    const int vh = e_hit ? c : 0, vf = e_fill ? c : 0;
    int ih = vh, iff = vf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, ih, o);
      const int y = __shfl_up_sync(0xffffffffu, iff, o);
      if (lane >= o) { ih += x; iff += y; }
    }
    if (lane == 31) { s_wc[0][warp] = ih; s_wc[1][warp] = iff; }
    __syncthreads();
    int bh = 0, bf = 0, th = 0, tf = 0;
#pragma unroll
    for (int w2 = 0; w2 < kCtrlThreads / 32; ++w2) {
      const int x = s_wc[0][w2], y = s_wc[1][w2];
      if (w2 < warp) { bh += x; bf += y; }
      th += x;
      tf += y;
    }
    const int fill_base = th + ns * a.T;   // the shared expert's pairs follow the hits'
    if (e_g >= 0) {
      const int off = e_hit ? bh + ih - vh : fill_base + bf + iff - vf;
      a.b.gpu_off[e_g] = off;
      ecnt[e] = off;
    }
    if (ns && tid == 0) a.b.gpu_off[h] = th;
    if (tid == 0) a.b.gpu_off[ngpu] = fill_base + tf;
    __syncthreads();
    int my_hits = 0, my_misses = 0;
    for (int p = tid; p < P; p += nt) {
      const int e2 = pid[p];
      int slot = -1;
      if ((unsigned)e2 < (unsigned)E) {
        const int i = lslot[e2];
        const int cls = uniq_cls[i];
        if (cls == 0) ++my_hits; else ++my_misses;
        if (cls < 2) {
          slot = uniq_slot[i];
          a.b.gpu_pairs[atomicAdd(&ecnt[e2], 1)] = p;
        }
      } else {
        ++my_misses;
      }
      a.b.slot_map[p] = slot;
      if (a.slot_map_out) a.slot_map_out[p] = slot;
    }
    if (my_hits) atomicAdd(&sc.read_hits, my_hits);
    if (my_misses) atomicAdd(&sc.read_misses, my_misses);
    if (ns)
      for (int t = tid; t < a.T; t += nt) a.b.gpu_pairs[th + t] = P + t;   // shared pairs after routed hits
  } else {
    int my_hits = 0, my_misses = 0;
    for (int p = tid; p < P; p += nt) {
      const int e = pid[p];
      int slot = -1;
      if ((unsigned)e < (unsigned)E) {
        const uint32_t wbits = ebits[e >> 5];
        const int i = by_expert ? lslot[e] : ebase[e >> 5] + __popc(wbits & ((1u << (e & 31)) - 1u));
        const int cls = uniq_cls[i];
        if (cls == 0) ++my_hits; else ++my_misses;
        if (cls < 2) {
          slot = uniq_slot[i];
          atomicAdd(&gcnt[uniq_rank[i]], 1);
        }
      } else {
        ++my_misses;
      }
      a.b.slot_map[p] = slot;
      if (a.slot_map_out) a.slot_map_out[p] = slot;
    }
    if (my_hits) atomicAdd(&sc.read_hits, my_hits);
    if (my_misses) atomicAdd(&sc.read_misses, my_misses);
    if (ns && tid == 0) gcnt[h] = a.T;
    __syncthreads();
    if (tid < 32) {  // exclusive scan of pair counts -> offsets (gcnt becomes write cursors)
      int running = 0;
      for (int c0 = 0; c0 < ngpu; c0 += 32) {
        const int g = c0 + lane;
        const int c = g < ngpu ? gcnt[g] : 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (g < ngpu) { a.b.gpu_off[g] = running + incl - c; gcnt[g] = running + incl - c; }
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) a.b.gpu_off[ngpu] = running;
    }
    __syncthreads();
    for (int p = tid; p < P; p += nt) {
      const int e = pid[p];
      if ((unsigned)e < (unsigned)E) {
        const uint32_t wbits = ebits[e >> 5];
        const int i = by_expert ? lslot[e] : ebase[e >> 5] + __popc(wbits & ((1u << (e & 31)) - 1u));
        if (uniq_cls[i] < 2) a.b.gpu_pairs[atomicAdd(&gcnt[uniq_rank[i]], 1)] = p;
      }
    }
    if (ns) {
      for (int t = tid; t < a.T; t += nt) a.b.gpu_pairs[gcnt[h] + t] = P + t;  // shared pairs after routed ones
    }
  }

  // ---- 8. plan scalars, counters, error word ------------------------------------
  __syncthreads();
  if (tid == 0) {
    int32_t* pl = a.b.plan;
    pl[P_LAYER] = a.layer; pl[P_U] = u; pl[P_H] = h; pl[P_M] = m; pl[P_Q] = q;
    pl[P_NCPU] = m - q; pl[P_NGPU] = ngpu; pl[P_NFIRST] = nfirst;
    // reductions, not read-modify-writes: nothing waits for the old values
    unsigned long long* c = reinterpret_cast<unsigned long long*>(a.tab.counters);
    atomicAdd(c + 0, (unsigned long long)h); atomicAdd(c + 1, (unsigned long long)m);
    atomicAdd(c + 2, (unsigned long long)q); atomicAdd(c + 3, (unsigned long long)(m - q));
    atomicAdd(c + 4, (unsigned long long)sc.read_hits); atomicAdd(c + 5, (unsigned long long)sc.read_misses);
    atomicAdd(c + 6, 1ull);
    uint32_t e = 0;
    if (sc.bad & 1) e |= kErrBadExpertId;
    if (sc.bad & 2) e |= kErrClock;
    if (e) atomicOr_system(a.err, e);
  }
}

}  // namespace

cudaError_t launch_decode_control(const Shape& sh, int layer, int T, int C, int K, uint32_t bp,
                                  uint32_t bc, const int32_t* ids, CacheTables tab, DecodeBufs b,
                                  int32_t* slot_map_out, const uint8_t* slots_base,
                                  const uint8_t* shared_base, uint32_t* err, cudaStream_t s) {
  CtrlArgs a;
  a.layer = layer; a.T = T; a.k = sh.k; a.E = sh.E; a.C = C; a.K = K; a.n_shared = sh.n_shared;
  a.bp = bp; a.bc = bc; a.S = sh.S; a.ids = ids; a.tab = tab; a.b = b;
  a.slot_map_out = slot_map_out; a.slots_base = slots_base;
  a.shared_blob = sh.n_shared ? shared_base + (size_t)layer * sh.S : nullptr;
  a.err = err;
  a.umax = min(sh.E, T * sh.k);
  const int NW = (sh.E + 31) / 32;
  const size_t base = (size_t)sh.E * 4 + (size_t)T * sh.k * 4 + (size_t)(2 * NW + 1) * 4 +
                      (size_t)(6 * a.umax + 2) * 4 + (size_t)sh.E * 4 + (size_t)K * 4 + 512 * 4 + 8 +
                      (size_t)(K > kPoolN ? K : kPoolN) * 8 + (size_t)kPoolN * 8 + 16;
  a.cache_keys = (C <= kSmemKeyCap && base + (size_t)C * 12 <= kCtrlSmemLimit) ? 1 : 0;
  const size_t smem = base + (a.cache_keys ? (size_t)C * 12 : 0);
  if (smem > kCtrlSmemLimit) return cudaErrorInvalidConfiguration;
  if (K <= kPoolMaxK) return launch_pdl(decode_control_kernel<2>, dim3(1), dim3(kCtrlThreads), smem, s, a);
  return launch_pdl(decode_control_kernel<1>, dim3(1), dim3(kCtrlThreads), smem, s, a);
}

cudaError_t setup_control_kernels() {
  for (auto k : {decode_control_kernel<1>, decode_control_kernel<2>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCtrlSmemLimit);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kDecodeCarveout);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
