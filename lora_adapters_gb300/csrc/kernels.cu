// CUDA-core kernels of the heterogeneous-batch LoRA path (sm_103a):
//   build_segments  -- stable grouping of the batch's tokens by adapter, and
//                      the work lists of the apply kernel
//   apply_cc        -- one launch: shrink v[j, k] = x[perm[j], :] . A_a[:, k],
//                      a grid barrier, then expand
//                      y[perm[j], n] += s * sum_k v[j, k] B_a[k, n]
//   scatter         -- adapter load: staged rows -> their pool pages
//
// The method ("S-LoRA: Serving Thousands of Concurrent LoRA Adapters";
// dongaigc.com summary, section 2 "heterogeneous batching"; nubint.ai review,
// method list) batches the LoRA part of tokens that use different adapters of
// different ranks in one pass, reading adapter weights directly from
// non-contiguous pool pages.  At decode shapes the arithmetic intensity is
// below 2 flop/byte, so shrink and expand are organised around HBM traffic:
// persistent CTAs (one per SM) in which one producer warp streams whole page
// rows into a shared-memory ring with 1-D bulk copies (TMA engine, mbarrier
// completion) while eight consumer warps compute from shared memory.  Every
// distinct adapter row leaves HBM once per token tile.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include "internal.h"

namespace slora {
namespace {

// ---- 16-bit element helpers ----------------------------------------------------
struct F16 {
  static constexpr bool kBf16 = false;
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return __half22float2(h);
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
};
struct BF16 {
  static constexpr bool kBf16 = true;
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    __nv_bfloat162 h;
    memcpy(&h, &u, 4);
    return __bfloat1622float2(h);
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
  }
};

template <class D>
__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  float2 a = D::unpack(v.x), b = D::unpack(v.y), c = D::unpack(v.z), e = D::unpack(v.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = e.x; f[7] = e.y;
}

// Block-wide exclusive scan of K ints per thread; sh holds 33*K ints.  The
// second level scans the K per-warp totals in K warps at once.
template <int K>
__device__ __forceinline__ void block_scan_excl(int (&v)[K], int (&total)[K], int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  static_assert(K <= 32, "one warp per scanned value");
  int inc[K];
#pragma unroll
  for (int k = 0; k < K; ++k) inc[k] = v[k];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      int n = __shfl_up_sync(0xffffffffu, inc[k], off);
      if (lane >= off) inc[k] += n;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int k = 0; k < K; ++k) sh[warp * K + k] = inc[k];
  }
  __syncthreads();
  for (int k = warp; k < K; k += nw) {   // warp k scans value k over the warps
    int w = lane < nw ? sh[lane * K + k] : 0;
    int ws = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, ws, off);
      if (lane >= off) ws += n;
    }
    if (lane < nw) sh[lane * K + k] = ws - w;
    if (lane == 31) sh[32 * K + k] = ws;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    v[k] = inc[k] - v[k] + sh[warp * K + k];
    total[k] = sh[32 * K + k];
  }
  __syncthreads();
}

// ---- bulk copies, mbarriers and programmatic dependent launch ------------------
// A wait gives up after kWaitLimit polls (each poll may itself block briefly);
// the kernel then records SLORA_ERR_TIMEOUT in the error word and leaves its
// loop instead of spinning forever.
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kErrTimeout = -8;  // SLORA_ERR_TIMEOUT

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase of the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Programmatic dependent launch: wait for the preceding kernel's results /
// let the next kernel's CTAs start their prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void report(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Position q (in work order) of work unit `item`: the largest q with
// off[q] <= item, searched in shared memory when the prefix array fits there.
__device__ __forceinline__ int find_pos(const int32_t* s_off, const int32_t* g_off, bool in_smem, int S,
                                        int item) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int v = in_smem ? s_off[mid] : __ldg(g_off + mid);
    if (v <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Selects a[i] for a runtime index i without local memory.
template <int N>
__device__ __forceinline__ int pick(const int (&a)[N], int i) {
  int v = a[0];
#pragma unroll
  for (int m = 1; m < N; ++m)
    if (i == m) v = a[m];
  return v;
}

// ---- build_segments ----------------------------------------------------------------
// One CTA of 1024 threads.
//  (1) histogram of adapter ids in shared memory (ids out of range or not
//      resident are left out and reported); every adapter's rank is read
//      into shared memory first when it fits;
//  (2) one block scan over the histogram (each thread owns a run of adapter
//      ids) -> one segment per adapter present, in ascending id;
//  (3) stable scatter of token indices.  A batch of several tiles whose
//      tokens come in few runs of one adapter (prefill: a run per request) is
//      placed run by run: the runs are listed with one block scan, one warp
//      gives each run its first position (the adapter's running start plus
//      the earlier runs of that adapter), and every thread places its own
//      contiguous tokens.  Otherwise tokens are visited in order, 1024 at a
//      time; each warp groups its tokens by adapter (match_any), one warp
//      then gives every (warp, adapter) group its first position by walking
//      the warps in order, and a token's position is its group's first
//      position + its rank inside the group;
//  (4) work order: segments by rank, largest first (so that the persistent
//      apply kernels hand out the longest work units first), then the
//      per-position work-unit counts and their prefix sums.  Ties between
//      equal ranks are broken by shared-memory atomics: the order of equal-
//      rank segments, and so which CTA computes which unit, may differ from
//      run to run; every output element is still computed by exactly one unit
//      in a fixed order, so results do not change.
// Only step (1) reads global memory; the segment arrays are built in shared
// memory when they fit (flag kSegInSmem) and written out at the end.
constexpr int kCachedTiles = 4;  // token keys of the first 4096 tokens stay in registers

__global__ void __launch_bounds__(kSegThreads) build_segments_kernel(const SegBuildArgs args) {
  extern __shared__ int32_t smem_i[];
  __shared__ int32_t grp_key[32][32];
  __shared__ int32_t grp_cnt[32][32];
  __shared__ int32_t grp_base[32][32];
  __shared__ int32_t ngrp[32];
  __shared__ int32_t scan_sh[33 * 6];
  __shared__ int32_t rcount[kMaxRank + 1];
  __shared__ int32_t s_bad, s_err;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int A = args.max_adapters, T = args.T;
  const SegDev& sd = args.seg;
  const bool rank_smem = (args.smem_flags & kRankInSmem) != 0;
  const bool seg_smem = (args.smem_flags & kSegInSmem) != 0;
  int32_t* hist = smem_i;                                        // [A]
  int32_t* rank_s = rank_smem ? smem_i + A : nullptr;            // [A]
  int32_t* sbase = smem_i + (rank_smem ? 2 * A : A);
  const int cap = args.seg_cap;
  int32_t* s_adapter = seg_smem ? sbase : sd.seg_adapter;        // [cap]
  int32_t* s_start = seg_smem ? sbase + cap : sd.seg_start;      // [cap + 1]
  int32_t* s_rank = seg_smem ? sbase + 2 * cap + 1 : sd.seg_rank;
  int32_t* s_order = seg_smem ? sbase + 3 * cap + 1 : sd.seg_order;
  const bool keys_smem = (args.smem_flags & kKeysInSmem) != 0;
  int32_t* skeys = sbase + (seg_smem ? 4 * cap + 1 : 0);         // [T] when keys_smem
  // The apply kernels may start their prologue now; they wait for this
  // kernel's results (griddepcontrol.wait) before reading any of them.
  pdl_trigger();

  // Zero the histogram and, with independent loads in flight together, bring
  // in every adapter's rank (when the cache fits) and the batch's keys (when
  // they fit): no dependent round trip per token.
  for (int a = tid; a < A; a += nthr) {
    hist[a] = 0;
    if (rank_smem) rank_s[a] = args.rank[a];
  }
  if (keys_smem) {
    // kKeyBatch independent loads in flight per thread, then their stores
    constexpr int kKeyBatch = 8;
    for (int base = 0; base < T; base += kKeyBatch * nthr) {
      int kv[kKeyBatch];
#pragma unroll
      for (int u = 0; u < kKeyBatch; ++u) {
        const int i = base + u * nthr + tid;
        kv[u] = i < T ? args.token_adapter[i] : 0;
      }
#pragma unroll
      for (int u = 0; u < kKeyBatch; ++u) {
        const int i = base + u * nthr + tid;
        if (i < T) skeys[i] = kv[u];
      }
    }
  }
  for (int r = tid; r <= kMaxRank; r += nthr) rcount[r] = 0;
  if (tid == 0) {
    s_bad = 0;
    s_err = 0;
    // No apply kernel runs now (this kernel is not launched early), so the
    // apply kernel's barrier count can be reset: a call that gave up part-way
    // cannot leave later calls a stale count.
    if (args.grid_sync) args.grid_sync[kSyncCount] = 0;
  }
  __syncthreads();

  // (1) histogram; keys of the first tiles are kept for (3)
  // Whole warps call this (inactive lanes pass i >= T); equal keys within a
  // warp are counted with one shared-memory atomic (prefill batches hold long
  // runs of one adapter, which would otherwise serialise on one address).
  auto classify = [&](int i) -> int {
    int key = -1;
    if (i < T) {
      const int a = args.token_adapter[i];
      if (a >= 0 && a < A) {
        const int r = rank_smem ? rank_s[a] : args.rank[a];
        if (r > 0) {
          key = a;
        } else {
          atomicAdd(&s_bad, 1);
          atomicCAS(&s_err, 0, -4 /* SLORA_ERR_NOT_RESIDENT */);
        }
      } else if (a != -1) {
        atomicAdd(&s_bad, 1);
        atomicCAS(&s_err, 0, -1 /* SLORA_ERR_INVALID */);
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (peers & ((1u << lane) - 1u)) == 0u) atomicAdd(&hist[key], __popc(peers));
    return key;
  };
  int keys[kCachedTiles];
  if (keys_smem) {
    // all keys were staged in shared memory above; validated and counted in
    // one pass (whole warps take part in every iteration for match_any)
    for (int base = 0; base < T; base += nthr) {
      const int i = base + tid;
      const int a = i < T ? skeys[i] : -1;
      int key = -1;
      if (a >= 0 && a < A) {
        const int r = rank_smem ? rank_s[a] : args.rank[a];
        if (r > 0) {
          key = a;
        } else {
          atomicAdd(&s_bad, 1);
          atomicCAS(&s_err, 0, -4 /* SLORA_ERR_NOT_RESIDENT */);
        }
      } else if (a != -1) {
        atomicAdd(&s_bad, 1);
        atomicCAS(&s_err, 0, -1 /* SLORA_ERR_INVALID */);
      }
      if (i < T) skeys[i] = key;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      if (key >= 0 && (peers & ((1u << lane) - 1u)) == 0u) atomicAdd(&hist[key], __popc(peers));
    }
  } else {
#pragma unroll
    for (int c = 0; c < kCachedTiles; ++c) keys[c] = classify(c * nthr + tid);
    for (int base = kCachedTiles * nthr; base < T; base += nthr) classify(base + tid);
  }
  __syncthreads();

  // (2) segments in ascending adapter id; hist[a] becomes a's running start
  int segs, total_pos;
  {
    const int m = (A + nthr - 1) / nthr;
    const int lo = min(A, tid * m), hi = min(A, lo + m);
    int cnt = 0, ns = 0;
    for (int a = lo; a < hi; ++a) {
      const int c = hist[a];
      cnt += c;
      ns += c > 0;
    }
    int v[2] = {cnt, ns}, tot[2];
    block_scan_excl<2>(v, tot, scan_sh);
    int pos = v[0], s = v[1];
    for (int a = lo; a < hi; ++a) {
      const int c = hist[a];
      if (c > 0) {
        s_adapter[s] = a;
        s_start[s] = pos;
        const int r = rank_smem ? rank_s[a] : args.rank[a];
        s_rank[s] = r;
        atomicAdd(&rcount[r], 1);   // (4a) folded in: segments per rank
        hist[a] = pos;
        pos += c;
        ++s;
      }
    }
    total_pos = tot[0];
    segs = tot[1];
  }
  if (tid == 0) {
    s_start[segs] = total_pos;
    sd.counts[kNumSegs] = segs;
    sd.counts[kNSorted] = total_pos;
    sd.counts[kBadTokens] = s_bad;
    if (s_err != 0) atomicCAS(args.error, 0, s_err);
  }
  __syncthreads();

  // (3a) stable scatter by runs: warp w owns tokens [wlo, whi), its lanes
  // taking consecutive tokens (so the stores of a warp are consecutive
  // positions of a run); a run starts wherever the key changes (runs of
  // invalid tokens are listed too and placed nowhere)
  bool scattered = false;
  if (keys_smem && T > nthr) {
    const int nwarps = nthr >> 5;
    const int per_warp = ((T + nwarps - 1) / nwarps + 31) & ~31;
    const int wlo = min(T, warp * per_warp), whi = min(T, wlo + per_warp);
    const unsigned below = (1u << lane) - 1u;
    auto starts_run = [&](int i) -> bool { return i == 0 || skeys[i - 1] != skeys[i]; };
    int cnt = 0;
    for (int i = wlo + lane; i < whi; i += 32) cnt += starts_run(i) ? 1 : 0;
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    int v[1] = {lane == 0 ? cnt : 0}, tot[1];
    block_scan_excl<1>(v, tot, scan_sh);
    const int wbase = __shfl_sync(0xffffffffu, v[0], 0);   // runs starting before wlo
    const int R = tot[0];
    // worth it only for few, long runs; the run list lives in the group arrays
    if (R < 32 * 32 && 8 * R <= T) {
      int* run_start = &grp_cnt[0][0];   // [R + 1]
      int* run_key = &grp_key[0][0];     // [R]
      int* run_base = &grp_base[0][0];   // [R]
      int q = wbase;
      for (int i0 = wlo; i0 < whi; i0 += 32) {
        const int i = i0 + lane;
        const bool st = i < whi && starts_run(i);
        const unsigned b = __ballot_sync(0xffffffffu, st);
        if (st) {
          run_start[q + __popc(b & below)] = i;
          run_key[q + __popc(b & below)] = skeys[i];
        }
        q += __popc(b);
      }
      if (tid == 0) run_start[R] = T;
      __syncthreads();
      if (warp == 0) {
        // 32 runs at a time, in token order: a run's first position is its
        // adapter's running start plus the earlier runs of that adapter in
        // this chunk; the last of them moves the running start on
        for (int c0 = 0; c0 < R; c0 += 32) {
          const int qr = c0 + lane;
          const int k = qr < R ? run_key[qr] : -1;
          const int kk = k >= 0 ? k : -1 - lane;   // invalid runs match nothing
          const int len = k >= 0 ? run_start[qr + 1] - run_start[qr] : 0;
          int before = 0;
          bool last = true;
          for (int j = 0; j < 32; ++j) {
            const int kj = __shfl_sync(0xffffffffu, kk, j), lj = __shfl_sync(0xffffffffu, len, j);
            if (kj == kk) {
              if (j < lane) before += lj;
              if (j > lane) last = false;
            }
          }
          const int b = k >= 0 ? hist[k] : 0;
          __syncwarp();
          if (k >= 0) {
            run_base[qr] = b + before;
            if (last) hist[k] = b + before + len;
          }
          __syncwarp();
        }
      }
      __syncthreads();
      // the run holding token wlo (token 0 always starts one), then each
      // lane moves forward to the run holding its own token
      int cur = wbase - 1 + (wlo < whi && starts_run(wlo) ? 1 : 0);
      for (int i = wlo + lane; i < whi; i += 32) {
        while (run_start[cur + 1] <= i) ++cur;
        if (skeys[i] >= 0) sd.perm[run_base[cur] + (i - run_start[cur])] = i;
      }
      scattered = true;
    }
  }
  // (3b) stable scatter, one tile of 1024 tokens at a time, in token order
  const unsigned lt = (1u << lane) - 1u;
  for (int c = 0, base = 0; base < T && !scattered; ++c, base += nthr) {
    const int i = base + tid;
    int key = -1;
    if (keys_smem) {
      key = i < T ? skeys[i] : -1;
    } else if (c < kCachedTiles) {
      key = pick(keys, c);
    } else if (i < T) {
      const int a = args.token_adapter[i];
      if (a >= 0 && a < A && (rank_smem ? rank_s[a] : args.rank[a]) > 0) key = a;
    }
    const bool valid = key >= 0;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank_w = __popc(peers & lt);
    const bool leader = (peers & lt) == 0u;
    const unsigned lead_mask = __ballot_sync(0xffffffffu, valid && leader);
    // my group's slot in this warp's list: the slot of my group's leader
    const int slot = __shfl_sync(0xffffffffu, __popc(lead_mask & lt), valid ? __ffs(peers) - 1 : 0);
    if (valid && leader) {
      grp_key[warp][slot] = key;
      grp_cnt[warp][slot] = __popc(peers);
    }
    if (lane == 0) ngrp[warp] = __popc(lead_mask);
    __syncthreads();
    // One warp hands every (warp, adapter) group its first position, in
    // token order: the adapter's running start plus the tokens of that
    // adapter in earlier warps of this tile; the running start then moves
    // past this tile.  When every warp holds at most two groups (long runs of
    // one adapter, as in prefill batches of several tiles) lane w takes warp
    // w's groups and all bases come from one round of shuffles; otherwise the warps are walked
    // one by one (the groups of one warp have distinct adapters, so its
    // lanes update distinct running starts).
    if (warp == 0) {
      const int nw = min(nthr, T - base + 31) >> 5;   // warps with tokens in this tile
      const int ng_l = lane < nw ? ngrp[lane] : 0;
      if (T > nthr && __all_sync(0xffffffffu, ng_l <= 2)) {   // batches of several tiles
        // lane w holds warp w's (at most two) groups; empty slots match nothing
        const int k0 = ng_l > 0 ? grp_key[lane][0] : -1 - 2 * lane;
        const int c0 = ng_l > 0 ? grp_cnt[lane][0] : 0;
        const int k1 = ng_l > 1 ? grp_key[lane][1] : -2 - 2 * lane;
        const int c1 = ng_l > 1 ? grp_cnt[lane][1] : 0;
        int before0 = 0, before1 = 0;
        bool last0 = true, last1 = true;
        for (int j = 0; j < 32; ++j) {
          const int kj0 = __shfl_sync(0xffffffffu, k0, j), cj0 = __shfl_sync(0xffffffffu, c0, j);
          const int kj1 = __shfl_sync(0xffffffffu, k1, j), cj1 = __shfl_sync(0xffffffffu, c1, j);
          // the two groups of one warp have distinct adapters
          const int m0 = (kj0 == k0 ? cj0 : 0) + (kj1 == k0 ? cj1 : 0);
          const int m1 = (kj0 == k1 ? cj0 : 0) + (kj1 == k1 ? cj1 : 0);
          if (j < lane) {
            before0 += m0;
            before1 += m1;
          }
          if (j > lane) {
            last0 = last0 && m0 == 0;
            last1 = last1 && m1 == 0;
          }
        }
        const int b0 = ng_l > 0 ? hist[k0] : 0;
        const int b1 = ng_l > 1 ? hist[k1] : 0;
        __syncwarp();
        if (ng_l > 0) {
          grp_base[lane][0] = b0 + before0;
          if (last0) hist[k0] = b0 + before0 + c0;
        }
        if (ng_l > 1) {
          grp_base[lane][1] = b1 + before1;
          if (last1) hist[k1] = b1 + before1 + c1;
        }
      } else {
        for (int w = 0; w < nw; ++w) {
          const int ng = ngrp[w];
          if (lane < ng) {
            const int k = grp_key[w][lane];
            const int b = hist[k];
            grp_base[w][lane] = b;
            hist[k] = b + grp_cnt[w][lane];
          }
          __syncwarp();
        }
      }
    }
    __syncthreads();
    if (valid) sd.perm[grp_base[warp][slot] + rank_w] = i;
  }

  // (4b) start of each rank's run, largest rank first (warp 0; 9 ranks per lane)
  if (warp == 0) {
    int run = 0;
    for (int j = 0; j < 9; ++j) {
      const int d = lane * 9 + j;
      if (d <= kMaxRank) run += rcount[kMaxRank - d];
    }
    int inc = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += n;
    }
    int base = inc - run;
    for (int j = 0; j < 9; ++j) {
      const int d = lane * 9 + j;
      if (d <= kMaxRank) {
        const int c = rcount[kMaxRank - d];
        rcount[kMaxRank - d] = base;
        base += c;
      }
    }
  }
  __syncthreads();
  // (4c) place every segment in work order
  for (int s = tid; s < segs; s += nthr) s_order[atomicAdd(&rcount[s_rank[s]], 1)] = s;
  __syncthreads();
  // (4d) work units per position and their prefix sums (each thread owns a run of positions)
  {
    const int m = (segs + nthr - 1) / nthr;
    const int lo = min(segs, tid * m), hi = min(segs, lo + m);
    auto units = [&](int q, int (&u)[6]) {
      const int s = s_order[q];
      const int len = s_start[s + 1] - s_start[s];
      const int r = s_rank[s];
      const int ntt = (len + kTT - 1) / kTT;
      const int nrc = (r + kShrinkRows - 1) / kShrinkRows;
      const int nmt = (len + kTcM - 1) / kTcM;
      const bool is_short = len < args.tc_threshold;
      u[0] = ntt * nrc;
      u[1] = ntt;
      u[2] = is_short ? ntt * nrc : 0;
      u[3] = is_short ? ntt : 0;
      u[4] = nmt;
      u[5] = is_short ? 0 : nmt;
    };
    int sum[6] = {0, 0, 0, 0, 0, 0};
    for (int q = lo; q < hi; ++q) {
      int u[6];
      units(q, u);
#pragma unroll
      for (int k = 0; k < 6; ++k) sum[k] += u[k];
    }
    int tot[6];
    block_scan_excl<6>(sum, tot, scan_sh);
    for (int q = lo; q < hi; ++q) {
      sd.cc_shrink_all[q] = sum[0];
      sd.cc_tile_all[q] = sum[1];
      sd.cc_shrink_short[q] = sum[2];
      sd.cc_tile_short[q] = sum[3];
      sd.tc_tile_all[q] = sum[4];
      sd.tc_tile_long[q] = sum[5];
      int u[6];
      units(q, u);
#pragma unroll
      for (int k = 0; k < 6; ++k) sum[k] += u[k];
    }
    if (tid == 0) {
      sd.cc_shrink_all[segs] = tot[0];
      sd.cc_tile_all[segs] = tot[1];
      sd.cc_shrink_short[segs] = tot[2];
      sd.cc_tile_short[segs] = tot[3];
      sd.tc_tile_all[segs] = tot[4];
      sd.tc_tile_long[segs] = tot[5];
      sd.counts[kCcShrinkAll] = tot[0];
      sd.counts[kCcTileAll] = tot[1];
      sd.counts[kCcShrinkShort] = tot[2];
      sd.counts[kCcTileShort] = tot[3];
      sd.counts[kTcTileAll] = tot[4];
      sd.counts[kTcTileLong] = tot[5];
    }
  }
  // (5) the per-position descriptors; segment arrays built in shared memory
  // go out to global memory
  for (int q = tid; q < segs; q += nthr) {
    const int s = s_order[q];
    sd.seg_desc[q] = make_int4(s_adapter[s], s_rank[s], s_start[s], s_start[s + 1]);
  }
  if (seg_smem) {
    for (int s = tid; s < segs; s += nthr) {
      sd.seg_adapter[s] = s_adapter[s];
      sd.seg_rank[s] = s_rank[s];
      sd.seg_order[s] = s_order[s];
    }
    for (int s = tid; s <= segs; s += nthr) sd.seg_start[s] = s_start[s];
  }
}

// ---- build_segments for batches of at most 1024 tokens ---------------------------
// One CTA, one token per thread, no histogram over the adapter ids: a decode
// batch is short, and this kernel sits on its critical path, so it is built
// from few block-wide steps, each a handful of instructions.
//  (1) every thread reads its token's id and the adapter's rank (every rank
//      comes into shared memory first when there are few adapters) and forms
//      the composite key (id << 10) | token, unique per token; tokens that
//      are base-only or invalid get a key above every valid one;
//  (2) a token's sorted position is the number of keys below its own
//      (block_rank: sorted runs of 32 keys, binary searches): ascending id,
//      token order within an id;
//  (3) segment heads are the sorted positions whose id differs from the
//      previous one; a ballot scan numbers them;
//  (4) the work order -- segments by rank, largest first, ties by id -- is
//      the same ranking of (256 - rank, segment) keys, so it does not depend
//      on scheduling;
//  (5) work units per work-order position and their prefix sums (shuffle
//      scans), then the segment arrays go out.
constexpr int kSmallSegMax = 1024;

// Exclusive block scan of K ints per thread and their totals: shuffle scans
// inside each warp, one warp scans the warp totals.
template <int K>
__device__ __forceinline__ void small_block_scan(int (&v)[K], int (&excl)[K], int (&total)[K], int (*wtot)[K]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc[K];
#pragma unroll
  for (int k = 0; k < K; ++k) inc[k] = v[k];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1)
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int n = __shfl_up_sync(0xffffffffu, inc[k], off);
      if (lane >= off) inc[k] += n;
    }
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < K; ++k) wtot[warp][k] = inc[k];
  __syncthreads();
  if (warp == 0) {   // row nw of wtot receives the totals
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int t = lane < nw ? wtot[lane][k] : 0;
      int x = t;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += n;
      }
      __syncwarp();
      if (lane < nw) wtot[lane][k] = x - t;
      if (lane == 31) wtot[32][k] = x;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    excl[k] = wtot[warp][k] + inc[k] - v[k];
    total[k] = wtot[32][k];
  }
}

// Rank of every thread's key among the block's keys (keys unique, at most
// blockDim of them; absent keys = INT_MAX): each warp sorts its 32 keys with
// a bitonic network in registers and lays them out as a sorted run in
// `runs`; a thread's rank is the sum over the runs of the keys below its own,
// found by binary search, four runs' searches at a time.  Only the first
// `live` warps may hold present keys (the other runs are all INT_MAX and
// count nothing), so only their runs are searched.  Ends with the block
// synchronised.
__device__ __forceinline__ int block_rank(int key, int* runs, int live) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = key;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool keep_min = ((lane & j) == 0) == ((lane & k) == 0);
      v = keep_min ? min(v, o) : max(v, o);
    }
  runs[warp * 32 + lane] = v;
  __syncthreads();
  int rank = 0;
#pragma unroll 4
  for (int w = 0; w < live; ++w) {
    const int* r = runs + w * 32;
    int c = 0;   // keys of run w below `key`
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
      if (r[c + step - 1] < key) c += step;
    if (c == 31 && r[31] < key) c = 32;
    rank += c;
  }
  __syncthreads();
  return rank;
}

__global__ void __launch_bounds__(kSmallSegMax) build_segments_small_kernel(const SegBuildArgs args) {
  __shared__ int32_t s_rank_all[4 * kSmallSegMax];   // every adapter's rank, when there are few
  __shared__ __align__(16) int32_t s_key[kSmallSegMax];   // composite keys, then work-order keys
  __shared__ int32_t s_kr[kSmallSegMax];             // sorted position -> id | rank << 16
  __shared__ int32_t s_start[kSmallSegMax + 1], s_adapter[kSmallSegMax], s_rnk[kSmallSegMax];
  __shared__ int32_t s_order[kSmallSegMax];
  __shared__ int32_t s_wcnt[32];
  __shared__ int32_t s_wtot[33][6];
  __shared__ int32_t s_bad, s_err;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int A = args.max_adapters, T = args.T;
  const SegDev& sd = args.seg;
  pdl_trigger();

  // (1) ids and ranks: one round of independent loads when the ranks fit
  const bool rank_smem = A <= 4 * nthr;
  const int key = tid < T ? args.token_adapter[tid] : -1;
  if (rank_smem)
    for (int a = tid; a < A; a += nthr) s_rank_all[a] = args.rank[a];
  if (tid == 0) {
    s_bad = 0;
    s_err = 0;
    // No apply kernel runs now, so the apply kernel's barrier count can be
    // reset: a call that gave up part-way cannot leave later calls a stale count.
    if (args.grid_sync) args.grid_sync[kSyncCount] = 0;
  }
  __syncthreads();
  const bool in_range = key >= 0 && key < A;
  const int r = in_range ? (rank_smem ? s_rank_all[key] : __ldg(args.rank + key)) : 0;
  const bool valid = in_range && r > 0;
  if (tid < T && !valid && key != -1) {
    atomicAdd(&s_bad, 1);
    atomicCAS(&s_err, 0, in_range ? -4 /* SLORA_ERR_NOT_RESIDENT */ : -1 /* SLORA_ERR_INVALID */);
  }
  const int ckey = valid ? (key << 10) | tid : 0x7fffffff;
  const int n_sorted = __syncthreads_count(valid);

  // (2) sorted position = keys below this one
  const int pos = block_rank(ckey, s_key, nthr >> 5);
  if (valid) {
    s_kr[pos] = key | (r << 16);
    sd.perm[pos] = tid;
  }
  __syncthreads();

  // (3) segment heads in sorted order, numbered by a ballot scan
  const int kr = tid < n_sorted ? s_kr[tid] : 0;
  const bool head = tid < n_sorted && (tid == 0 || (s_kr[tid - 1] & 0xffff) != (kr & 0xffff));
  const unsigned hb = __ballot_sync(0xffffffffu, head);
  if (lane == 0) s_wcnt[warp] = __popc(hb);
  __syncthreads();
  int seg_base = 0, S = 0;
  for (int w = 0; w < (nthr >> 5); ++w) {
    const int c = s_wcnt[w];
    if (w < warp) seg_base += c;
    S += c;
  }
  if (head) {
    const int sg = seg_base + __popc(hb & ((1u << lane) - 1u));
    s_start[sg] = tid;
    s_adapter[sg] = kr & 0xffff;
    s_rnk[sg] = kr >> 16;
  }
  if (tid == 0) {
    s_start[S] = n_sorted;
    sd.counts[kNumSegs] = S;
    sd.counts[kNSorted] = n_sorted;
    sd.counts[kBadTokens] = s_bad;
    if (s_err != 0) atomicCAS(args.error, 0, s_err);
  }
  __syncthreads();

  // (4) work order: (256 - rank, segment) keys, ranked like (2)
  const int wkey = tid < S ? ((kMaxRank - s_rnk[tid]) << 10) | tid : 0x7fffffff;
  const int q = block_rank(wkey, s_key, (S + 31) >> 5);
  if (tid < S) s_order[q] = tid;
  __syncthreads();

  // (5) work units per work-order position, their prefix sums, descriptors
  int u[6] = {0, 0, 0, 0, 0, 0};
  int sg = 0, len = 0, rk = 0;
  if (tid < S) {
    sg = s_order[tid];
    len = s_start[sg + 1] - s_start[sg];
    rk = s_rnk[sg];
    const int ntt = (len + kTT - 1) / kTT;
    const int nrc = (rk + kShrinkRows - 1) / kShrinkRows;
    const int nmt = (len + kTcM - 1) / kTcM;
    const bool is_short = len < args.tc_threshold;
    u[0] = ntt * nrc;
    u[1] = ntt;
    u[2] = is_short ? ntt * nrc : 0;
    u[3] = is_short ? ntt : 0;
    u[4] = nmt;
    u[5] = is_short ? 0 : nmt;
  }
  int ex[6], tot[6];
  small_block_scan<6>(u, ex, tot, s_wtot);
  int32_t* const pre[6] = {sd.cc_shrink_all, sd.cc_tile_all, sd.cc_shrink_short, sd.cc_tile_short,
                           sd.tc_tile_all, sd.tc_tile_long};
  if (tid < S) {
#pragma unroll
    for (int k = 0; k < 6; ++k) pre[k][tid] = ex[k];
    sd.seg_desc[tid] = make_int4(s_adapter[sg], rk, s_start[sg], s_start[sg] + len);
    sd.seg_order[tid] = sg;
    sd.seg_adapter[tid] = s_adapter[tid];
    sd.seg_rank[tid] = s_rnk[tid];
  }
  if (tid < S) sd.seg_start[tid] = s_start[tid];
  if (tid == 0) {
    sd.seg_start[S] = s_start[S];   // S may equal the block size
    constexpr int idx[6] = {kCcShrinkAll, kCcTileAll, kCcShrinkShort, kCcTileShort, kTcTileAll, kTcTileLong};
#pragma unroll
    for (int k = 0; k < 6; ++k) {
      pre[k][S] = tot[k];
      sd.counts[idx[k]] = tot[k];
    }
  }
}

// ---- the CUDA-core apply kernel: shrink, grid barrier, expand (one launch) --------
// Persistent CTA per SM (grid = number of SMs, all CTAs resident at once):
// warps 0-7 consume; warp 8 plans the stages and warp 9 issues their copies.
// Every CTA first runs its shrink units, then its expand units; both kinds
// stream through the same 4-deep ring of 48 KB shared-memory stages.  The
// planner claims a free stage, writes its metadata, announces its bytes on the
// stage's mbarrier and lists its copies (one per lane: a whole row chunk,
// source and place in the stage); the issuer turns the list into 1-D bulk
// copies (TMA engine).  Issuing a stage's bulk copies holds a warp for about
// as long as planning the next stage does, so the two run side by side.
//
// Shrink unit = (segment position q, token tile of <= kTT tokens, chunk of 8
// rank rows, projection); projection varies fastest.  Per K chunk of <=
// kShrinkK elements (never crossing a page) a stage holds the 8 A rows, read
// straight from their pool pages, and the tile's x rows, each row 16 bytes
// longer than the chunk.  The eight consumer warps split the chunk's K range
// in 16-element steps; a step is one ldmatrix (8 A rows and the tile's x rows
// at once) and one warp-level m16n8k16 MMA (16-bit inputs, fp32 accumulation;
// rank rows on M, tokens on N).  Its M and N are mostly padding, but one MMA
// replaces the 512 conversions and multiply-adds the CUDA cores would issue
// for those 16 K values, which is what bounds this phase: the HBM bytes of a
// stage arrive in about 1,500 cycles.  At the unit's end the warps' partial
// sums meet in shared memory and one warp writes v (fp32).
//
// Between the phases the CTAs meet once (a grid barrier on two counters in
// global memory): the expand phase reads v rows that any CTA may have written.
// The producer does not wait for it before streaming the expand phase's B and
// y rows; only the v rows of an expand unit are held back until the barrier
// has opened, and they land on a separate mbarrier per v buffer.
//
// Expand unit = (segment position q, token tile, projection, column tile of
// <= kExpandCols columns inside one page); projection and column tile vary
// fastest.  Stages carry kExpandRKBig B rows each (a whole stage), and the
// unit's last stage at most kExpandRK B rows together with the tile's y rows.  Each consumer thread owns 8 adjacent columns:
// fp32 accumulation over the unit's rank rows for every token of the tile,
// then y + s * acc, one rounding, a 16-byte store.  (Warp-level MMAs were
// measured here too: with 4 of 8 token slots used and the legacy MMA path's
// rate on this GPU they took twice as long per stage as the FMAs.)
//
// The producer resolves units 32 at a time (one per lane), so page-table and
// segment lookups of a whole batch of units cost one round of loads, and it
// fetches the next expand unit's page indices while it streams the current one.
constexpr int kStages = 4;                             // ring depth (also the v item-ring depth)
constexpr int kShrinkK = 2048;                         // K chunk (elements) of a shrink stage
// Shrink rows are kShrinkPitch elements apart: 16 bytes past the chunk, so
// the 8 rows one ldmatrix phase reads sit in 8 different 16-byte bank groups.
constexpr int kShrinkPitch = kShrinkK + 8;
constexpr int kExpandRK = 8;                           // B rows of a unit's last expand stage (which also carries y)
constexpr int kExpandRKBig = 12;                       // B rows of its other stages (a whole 48 KB stage)
constexpr int kStageElems = (kShrinkRows + kTT) * kShrinkPitch;   // 48.2 KB of 16-bit elements
constexpr int kRowsOff = kShrinkRows * kShrinkK;       // y rows of an expand stage start here
static_assert((kShrinkPitch * 2) % 16 == 0 && (kStageElems * 2) % 16 == 0, "bulk copies need 16-byte rows");
constexpr int kPagesPerLane = kMaxRank / 32;           // B-row page indices one lane prefetches
static_assert(kExpandRK * kExpandCols <= kRowsOff, "B rows of a stage must fit before the x/y rows");
static_assert(kExpandRK % 4 == 0, "a full expand stage reads v four ranks at a time");
static_assert(kExpandRK <= kExpandRKBig, "the last stage takes at most as many rows as the others");
static_assert(kTT * kExpandCols <= kStageElems - kRowsOff, "y rows of a stage must fit");
static_assert(kExpandRKBig * kExpandCols <= kStageElems, "a stage of B rows must fit");
static_assert(kExpandRKBig <= 32, "a stage's B rows come from distinct lanes");
static_assert(kExpandRKBig % 4 == 0, "a full expand stage reads v four ranks at a time");

enum : int { kKindShrink = 0, kKindExpand = 1 };
// A stage's copy list: at most kCpMax copies; entry = source address and
// (byte offset in the stage << 13 | bytes), 0 = no copy for that lane.
constexpr int kCpMax = 12;
static_assert(kExpandRKBig <= kCpMax, "a stage's B rows must fit its copy list");
static_assert(kShrinkRows + kTT <= kCpMax && kExpandRK + kTT <= kCpMax, "a stage's copies must fit its list");
static_assert(kStageElems * 2 < (1 << 19) && kShrinkK * 2 < (1 << 13) && kExpandCols * 2 < (1 << 13),
              "stage offsets and copy sizes must fit the packed copy entry");
__device__ __forceinline__ uint32_t cp_entry(uint32_t off_bytes, uint32_t bytes) { return off_bytes << 13 | bytes; }
struct __align__(16) StageMeta {
  int kind, ntok, p, len, last;
  int j0, k0, nrows;                // shrink
  float sa;                         // shrink: the adapter's scale, applied to v
  int col0, nk, buf, vph;           // expand (k0 = first B row of the stage)
  int rows[kTT];
};
struct VPending {                   // an expand unit whose v rows wait for the grid barrier
  int buf, vph, p, j0, ntok, r;
};
struct ApplySmem {
  uint16_t st[kStages][kStageElems];
  float V[kStages][kTT][kMaxRank];
  // Shrink: the consumer warps' partial sums of a unit (8 rank rows x 4
  // tokens each), summed by one warp (unit u: warp u % 8, so that the extra
  // work goes round).  Unit u uses buffer u % kRedBufs: a warp can run at
  // most kStages stages (so kStages units) ahead of any other, so the summing
  // warp has read a buffer before any warp writes it again.
  float red[kStages + 1][kCcConsumerWarps][32];
  uint64_t redbar[kStages + 1];
  StageMeta meta[kStages];
  VPending pend[kStages];
  uint64_t full[kStages], empty[kStages], vfull[kStages];
  uint64_t issue[kStages];                 // the planner has listed the stage's copies (32 arrivals)
  const void* cp_src[kStages][kCpMax];
  uint32_t cp_desc[kStages][kCpMax];
  int32_t cp_stop[kStages];                // 1: no more stages (the issuer leaves)
  int32_t off_s[kSegSmem], off_e[kSegSmem];
  int32_t gen0;
};
constexpr int kRedBufs = kStages + 1;
static_assert(sizeof(ApplySmem) <= 232448, "apply kernel shared memory exceeds 227 KB");

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ua, ub, uc, r;
  memcpy(&ua, &a, 8);
  memcpy(&ub, &b, 8);
  memcpy(&uc, &c, 8);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(ua), "l"(ub), "l"(uc));
  float2 o;
  memcpy(&o, &r, 8);
  return o;
}
template <class D>
__device__ __forceinline__ void unpack4x2(uint4 v, float2 (&f)[4]) {
  f[0] = D::unpack(v.x);
  f[1] = D::unpack(v.y);
  f[2] = D::unpack(v.z);
  f[3] = D::unpack(v.w);
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ldmatrix: four (or two) 8 x 8 matrices of 16-bit elements; lane l gives
// the address of row l % 8 of matrix l / 8.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
// Warp-level MMA, fp32 accumulation: D[16 x 8] += A[16 x 16] B[16 x 8] with
// A rows 8..15 zero (a1 = a3 = 0), and the 8-deep form for a K tail.
template <bool BF>
__device__ __forceinline__ void mma_k16(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  if constexpr (BF)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
template <bool BF>
__device__ __forceinline__ void mma_k8(float (&c)[4], uint32_t a0, uint32_t b0) {
  if constexpr (BF)
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(0u), "r"(b0));
  else
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(0u), "r"(b0));
}

// 1-D bulk copy global -> shared through the TMA engine; completion is
// counted in bytes on the mbarrier.  Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// v rows (fp32, `n` floats, a multiple of 4) of one expand unit onto the unit's
// v-buffer barrier: lane 0 announces the bytes, lanes 0..ntok-1 copy a row each.
__device__ __forceinline__ void load_vrows(float (*dst)[kMaxRank], const float* src, int64_t ld, int ntok, int n,
                                           uint64_t* bar, int lane) {
  if (lane == 0) mbar_expect_tx(bar, (uint32_t)ntok * (uint32_t)n * 4u);
  __syncwarp();
  if (lane < ntok) bulk_load(&dst[lane][0], src + (int64_t)lane * ld, (uint32_t)n * 4u, bar);
}

// Column tile ct of a row of h_out elements stored in pages of H: tiles never
// cross a page; returns the page chunk c, the offset o inside it and the length.
__device__ __forceinline__ void col_tile(int ct, int h_out, int H, int& c, int& o, int& len) {
  for (c = 0;; ++c) {
    const int lenc = min(H, h_out - c * H);
    const int nt = (lenc + kExpandCols - 1) / kExpandCols;
    if (ct < nt) {
      o = ct * kExpandCols;
      len = min(kExpandCols, lenc - o);
      return;
    }
    ct -= nt;
  }
}

// Page indices of B rows lane, lane+32, ... of (adapter a, rank r, projection
// p, page chunk c).
__device__ __forceinline__ void load_b_pages(const ApplyDev& d, int a, int r, int p, int c,
                                             int (&pg)[kPagesPerLane], int lane) {
  const ProjDev& P = d.proj[p];
  const int32_t* ptB = d.page_table + (int64_t)a * d.pt_stride + (int64_t)r * (P.rows_before + P.ppi) + c;
#pragma unroll
  for (int m = 0; m < kPagesPerLane; ++m) {
    const int row = lane + 32 * m;
    pg[m] = row < r ? dbg_index(__ldg(ptB + (int64_t)row * P.ppo), d.num_pages, d.error) : 0;
  }
}

// Expand compute of NK B rows (a multiple of 4): the rows' pieces and the
// tokens' NK v values are loaded first, then the multiply-adds run, so that
// shared-memory latency is paid once per group rather than once per row.
template <class D, int NT, int NK>
__device__ __forceinline__ void expand_rows(const uint16_t* brows, const float (*V)[kMaxRank], int k0, int col,
                                            float2 (&acc)[kTT][4]) {
  uint4 b[NK];
#pragma unroll
  for (int k = 0; k < NK; ++k) b[k] = *reinterpret_cast<const uint4*>(brows + k * kExpandCols + col);
  float4 v[NT][NK / 4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int q = 0; q < NK / 4; ++q) v[t][q] = *reinterpret_cast<const float4*>(&V[t][k0 + 4 * q]);
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    float2 fb[4];
    unpack4x2<D>(b[k], fb);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float4 vq = v[t][k >> 2];
      const float vv = (k & 3) == 0 ? vq.x : (k & 3) == 1 ? vq.y : (k & 3) == 2 ? vq.z : vq.w;
      const float2 v2 = make_float2(vv, vv);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = ffma2(v2, fb[e], acc[t][e]);
    }
  }
}
// Expand stage compute of the consumer threads, specialised on the tile's
// token count so that no issue slot goes to absent tokens; whole stages
// (kExpandRKBig or kExpandRK rows) in groups of 8 and 4 rows.
template <class D, int NT>
__device__ __forceinline__ void expand_stage(const uint16_t* brows, const float (*V)[kMaxRank], int k0, int nk,
                                             int col, float2 (&acc)[kTT][4]) {
  if (nk == kExpandRKBig || nk == kExpandRK) {   // k0 is a multiple of 4 (the planner's split)
    expand_rows<D, NT, 8>(brows, V, k0, col, acc);
    if (nk == kExpandRKBig) expand_rows<D, NT, kExpandRKBig - 8>(brows + 8 * kExpandCols, V, k0 + 8, col, acc);
    return;
  }
#pragma unroll 2
  for (int k = 0; k < nk; ++k) {
    float2 fb[4];
    unpack4x2<D>(*reinterpret_cast<const uint4*>(brows + k * kExpandCols + col), fb);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float vv = V[t][k0 + k];
      const float2 v2 = make_float2(vv, vv);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = ffma2(v2, fb[e], acc[t][e]);
    }
  }
}

template <class D>
__global__ void __launch_bounds__(kCcThreads, 1) apply_cc_kernel(const __grid_constant__ ApplyDev d) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ApplySmem& sm = *reinterpret_cast<ApplySmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCcConsumerWarps);
      mbar_init(&sm.vfull[s], 1);
      mbar_init(&sm.issue[s], 32);
    }
    for (int s = 0; s < kRedBufs; ++s) mbar_init(&sm.redbar[s], kCcConsumerWarps);
    mbar_fence_init();
  }
  pdl_wait();  // the work lists come from the segment kernel; an earlier apply has finished
  // The barrier generation before this launch's CTAs arrive: it changes only
  // once every CTA of this launch has arrived, and this CTA has not.
  if (threadIdx.x == 0) sm.gen0 = ld_acquire(d.grid_sync + kSyncGen);
  // The work-list prefixes are loaded for as many positions as the batch can
  // have segments (d.off_n, set by the host), together with the counts, so
  // that the prologue costs one round of loads.
  for (int i = threadIdx.x; i < d.off_n; i += blockDim.x) {
    sm.off_s[i] = d.shrink_off[i];
    sm.off_e[i] = d.tile_off[i];
  }
  const int units_s = d.counts[d.shrink_total_idx];
  const int tiles = d.counts[d.tile_total_idx];
  const int S = d.counts[kNumSegs];
  const bool off_smem = S + 1 <= d.off_n;
  __syncthreads();
  pdl_trigger();
  int per_tile = 0;  // expand units of one token tile: (projection, column tile)
  for (int p = 0; p < d.nproj; ++p) per_tile += d.proj[p].ncol_tiles;
  const int64_t Gs = (int64_t)units_s * d.nproj;
  const int64_t Ge = (int64_t)tiles * per_tile;
  // Units in "snake" order: round i gives CTA b unit i * G + b on even rounds
  // and i * G + (G - 1 - b) on odd rounds.  The lists run largest work first,
  // so the CTA that drew a larger unit in one round draws a smaller one in the
  // next, and the CTAs' totals stay close.
  const int64_t G = gridDim.x, b = blockIdx.x;
  auto snake_unit = [&](int64_t i) -> int64_t { return i * G + ((i & 1) ? G - 1 - b : b); };
  auto snake_count = [&](int64_t total) -> int64_t {
    const int64_t R = total / G, rem = total - R * G;
    return R + (((R & 1) ? G - 1 - b : b) < rem ? 1 : 0);
  };
  const int64_t ns = snake_count(Gs), ne = snake_count(Ge);   // this CTA's units
  // Polls of a wait on other warps (or CTAs) before this kernel gives up;
  // the waits for its own copies in flight before it exits keep kWaitLimit.
  const uint32_t lim = d.wait_limit ? d.wait_limit : kWaitLimit;

  // slots (bit s) with copies issued, and the parity of that phase: what a
  // warp that gives up must wait for before the CTA exits
  auto mark = [](uint32_t& set, uint32_t& par, int s2, uint32_t ph) {
    set |= 1u << s2;
    par = (par & ~(1u << s2)) | (ph << s2);
  };
  if (warp == kCcConsumerWarps) {  // ============================= planner warp
    uint32_t stage = 0, phase = 0, nitem = 0;
    bool ok = true;
    bool opened = false;  // the grid barrier has opened (v rows may be read)
    int npend = 0;        // expand units whose v rows wait for it
    uint32_t vissued = 0, vpar = 0;   // v-row copies issued here
    // The stage's copy list, one entry per lane (src NULL: none), handed to
    // the issuer warp; every lane arrives on the stage's issue barrier.
    auto post = [&](const void* src, uint32_t off_bytes, uint32_t bytes) {
      if (lane < kCpMax) {
        sm.cp_src[stage][lane] = src;
        sm.cp_desc[stage][lane] = src ? cp_entry(off_bytes, bytes) : 0u;
      }
      if (lane == 0) sm.cp_stop[stage] = 0;
      mbar_arrive(&sm.issue[stage]);
    };
    const int gen0 = sm.gen0;
    // v rows of the units held back, once the barrier has opened
    auto release_pending = [&]() {
      for (int i = 0; i < npend; ++i) {
        const VPending e = sm.pend[i];
        load_vrows(sm.V[e.buf], d.proj[e.p].v + (int64_t)e.j0 * d.v_ld, d.v_ld, e.ntok, (e.r + 3) & ~3,
                   &sm.vfull[e.buf], lane);
        mark(vissued, vpar, e.buf, (uint32_t)e.vph);
      }
      npend = 0;
    };
    // Has the grid barrier opened?  Every lane reads the generation with
    // acquire semantics, so that each lane's later copies of v rows are
    // ordered after the other CTAs' writes of them.
    auto barrier_open = [&]() -> bool {
      const bool o = __all_sync(0xffffffffu, ld_acquire(d.grid_sync + kSyncGen) != gen0);
      if (o) asm volatile("fence.proxy.async.global;" ::: "memory");
      return o;
    };
    // Next stage slot.  While expand units wait for v rows, the wait for a
    // free slot also watches the grid barrier (the consumers cannot free a
    // slot before those v rows arrive), without blocking on the slot.
    auto acquire = [&]() -> bool {
      for (uint32_t it = 0; it < lim; ++it) {
        int got = 0;
        if (lane == 0)
          got = (npend > 0 ? mbar_test_wait(&sm.empty[stage], phase ^ 1) : mbar_try_wait(&sm.empty[stage], phase ^ 1))
                    ? 1 : 0;
        if (__shfl_sync(0xffffffffu, got, 0)) return true;
        if (npend > 0 && barrier_open()) {
          opened = true;
          release_pending();
        }
      }
      return false;
    };
    // ---- shrink units
    for (int64_t i0 = 0; i0 < ns && ok; i0 += 32) {
      const int64_t gl = snake_unit(i0 + lane);   // lane l resolves this CTA's unit i0 + l
      const int nb = (int)min((int64_t)32, ns - i0);
      int m_p = 0, m_j0 = 0, m_ntok = 0, m_k0 = 0, m_nrows = 0, m_r = 0, m_a = 0;
      float m_sa = 1.f;
      int pg[kShrinkRows], xt[kTT];
#pragma unroll
      for (int i = 0; i < kShrinkRows; ++i) pg[i] = 0;
#pragma unroll
      for (int t = 0; t < kTT; ++t) xt[t] = 0;
      if (lane < nb) {
        const int unit = (int)(gl / d.nproj);
        m_p = (int)(gl - (int64_t)unit * d.nproj);
        const int q = find_pos(sm.off_s, d.shrink_off, off_smem, S, unit);
        const int local = unit - (off_smem ? sm.off_s[q] : __ldg(d.shrink_off + q));
        const int4 sd = __ldg(d.seg_desc + q);   // adapter, rank, start, end
        m_a = sd.x;
        m_r = sd.y;
        if (d.scale) m_sa = __ldg(d.scale + m_a);
        const int nrc = (m_r + kShrinkRows - 1) / kShrinkRows;
        const int tt = local / nrc, rc = local - tt * nrc;
        m_j0 = sd.z + tt * kTT;
        m_ntok = min(kTT, sd.w - m_j0);
        m_k0 = rc * kShrinkRows;
        m_nrows = min(kShrinkRows, m_r - m_k0);
        const ProjDev& P = d.proj[m_p];
        const int32_t* pt = d.page_table + (int64_t)m_a * d.pt_stride + (int64_t)m_r * P.rows_before +
                            (int64_t)m_k0 * P.ppi;
#pragma unroll
        for (int i = 0; i < kShrinkRows; ++i)
          if (i < m_nrows) pg[i] = dbg_index(__ldg(pt + (int64_t)i * P.ppi), d.num_pages, d.error);
#pragma unroll
        for (int t = 0; t < kTT; ++t)
          if (t < m_ntok) xt[t] = dbg_index(__ldg(d.perm + m_j0 + t), d.T, d.error);
      }
      for (int l = 0; l < nb && ok; ++l) {
        const int p = __shfl_sync(0xffffffffu, m_p, l);
        const int j0 = __shfl_sync(0xffffffffu, m_j0, l);
        const int ntok = __shfl_sync(0xffffffffu, m_ntok, l);
        const int k0 = __shfl_sync(0xffffffffu, m_k0, l);
        const int nrows = __shfl_sync(0xffffffffu, m_nrows, l);
        const int r = __shfl_sync(0xffffffffu, m_r, l);
        const int a = __shfl_sync(0xffffffffu, m_a, l);
        const float sa = __shfl_sync(0xffffffffu, m_sa, l);
        // lane i < nrows holds A row k0 + i's page, lane 8 + t token t of the tile
        int my = 0;
#pragma unroll
        for (int i = 0; i < kShrinkRows; ++i) {
          const int v = __shfl_sync(0xffffffffu, pg[i], l);
          if (lane == i) my = v;
        }
#pragma unroll
        for (int t = 0; t < kTT; ++t) {
          const int v = __shfl_sync(0xffffffffu, xt[t], l);
          if (lane == kShrinkRows + t) my = v;
        }
        const ProjDev& P = d.proj[p];
        const bool has_row = lane < nrows;
        const int32_t* pt_row = d.page_table + (int64_t)a * d.pt_stride + (int64_t)r * P.rows_before +
                                (int64_t)(k0 + lane) * P.ppi;
        const uint16_t* xbase = static_cast<const uint16_t*>(P.x);
        for (int c = 0; c < P.ppi && ok; ++c) {
          const int lenc = min(d.H, P.h_in - c * d.H);
          // the next page of this lane's row, fetched while this one streams
          const int next = (has_row && c + 1 < P.ppi) ? dbg_index(__ldg(pt_row + c + 1), d.num_pages, d.error) : 0;
          for (int o = 0; o < lenc; o += kShrinkK) {
            const int len = min(kShrinkK, lenc - o);
            const int last = (c == P.ppi - 1) && (o + len >= lenc);
            if (!acquire()) {
              ok = false;
              break;
            }
            if (lane == 0) {
              StageMeta& m = sm.meta[stage];
              m.kind = kKindShrink;
              m.ntok = ntok;
              m.p = p;
              m.len = len;
              m.last = last;
              m.j0 = j0;
              m.k0 = k0;
              m.nrows = nrows;
              m.sa = sa;
              mbar_expect_tx(&sm.full[stage], (uint32_t)(nrows + ntok) * (uint32_t)len * 2u);
            }
            // A row i and token row t at rows i and kShrinkRows + t of the stage
            const uint16_t* src = nullptr;
            if (lane < nrows) src = d.pool + (int64_t)my * d.H + o;
            else if (lane >= kShrinkRows && lane < kShrinkRows + ntok)
              src = xbase + (int64_t)my * P.ldx + (int64_t)c * d.H + o;
            post(src, (uint32_t)(lane * kShrinkPitch) * 2u, (uint32_t)len * 2u);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (lane < kShrinkRows) my = next;
        }
      }
    }
    // ---- expand units
    for (int64_t i0 = 0; i0 < ne && ok; i0 += 32) {
      const int64_t gl = snake_unit(i0 + lane);   // lane l resolves this CTA's unit i0 + l
      const int nb = (int)min((int64_t)32, ne - i0);
      int m_p = 0, m_j0 = 0, m_ntok = 0, m_r = 0, m_a = 0, m_c = 0, m_o = 0, m_len = 0;
      int rws[kTT];
#pragma unroll
      for (int t = 0; t < kTT; ++t) rws[t] = 0;
      if (lane < nb) {
        const int tile = (int)(gl / per_tile);
        int ct = (int)(gl - (int64_t)tile * per_tile);
        while (ct >= d.proj[m_p].ncol_tiles) ct -= d.proj[m_p++].ncol_tiles;
        const int q = find_pos(sm.off_e, d.tile_off, off_smem, S, tile);
        const int tt = tile - (off_smem ? sm.off_e[q] : __ldg(d.tile_off + q));
        const int4 sd = __ldg(d.seg_desc + q);   // adapter, rank, start, end
        m_a = sd.x;
        m_r = sd.y;
        m_j0 = sd.z + tt * kTT;
        m_ntok = min(kTT, sd.w - m_j0);
        col_tile(ct, d.proj[m_p].h_out, d.H, m_c, m_o, m_len);
#pragma unroll
        for (int t = 0; t < kTT; ++t)
          if (t < m_ntok) rws[t] = dbg_index(__ldg(d.perm + m_j0 + t), d.T, d.error);
      }
      int pg[kPagesPerLane];
      load_b_pages(d, __shfl_sync(0xffffffffu, m_a, 0), __shfl_sync(0xffffffffu, m_r, 0),
                   __shfl_sync(0xffffffffu, m_p, 0), __shfl_sync(0xffffffffu, m_c, 0), pg, lane);
      for (int l = 0; l < nb && ok; ++l, ++nitem) {
        const int p = __shfl_sync(0xffffffffu, m_p, l);
        const int j0 = __shfl_sync(0xffffffffu, m_j0, l);
        const int ntok = __shfl_sync(0xffffffffu, m_ntok, l);
        const int r = __shfl_sync(0xffffffffu, m_r, l);
        const int o = __shfl_sync(0xffffffffu, m_o, l);
        const int c = __shfl_sync(0xffffffffu, m_c, l);
        const int len = __shfl_sync(0xffffffffu, m_len, l);
        int rows[kTT];
#pragma unroll
        for (int t = 0; t < kTT; ++t) rows[t] = __shfl_sync(0xffffffffu, rws[t], l);
        // prefetch the next unit's page indices
        int pgn[kPagesPerLane];
        const int ln = l + 1 < nb ? l + 1 : l;
        load_b_pages(d, __shfl_sync(0xffffffffu, m_a, ln), __shfl_sync(0xffffffffu, m_r, ln),
                     __shfl_sync(0xffffffffu, m_p, ln), __shfl_sync(0xffffffffu, m_c, ln), pgn, lane);
        const ProjDev& P = d.proj[p];
        const int col0 = c * d.H + o;
        const int buf = (int)(nitem % kStages);
        const int vph = (int)((nitem / kStages) & 1);
        // the unit's rows: stages of at most kExpandRKBig rows (a multiple of
        // 4, so that every stage starts at a multiple of 4 and its v values
        // load as float4), then a last stage of at most kExpandRK rows
        // together with the tile's y rows
        for (int k0 = 0, nk = 0; k0 < r; k0 += nk) {
          nk = r - k0 <= kExpandRK ? r - k0 : min(kExpandRKBig, (r - k0 - 1) & ~3);
          const bool first = k0 == 0;
          const int last = k0 + nk >= r;
          if (!acquire()) {
            ok = false;
            break;
          }
          if (first) {
            // v rows of the unit: now if the barrier has opened, else held back
            if (!opened) opened = barrier_open();
            if (opened) {
              if (npend > 0) release_pending();
              load_vrows(sm.V[buf], P.v + (int64_t)j0 * d.v_ld, d.v_ld, ntok, (r + 3) & ~3, &sm.vfull[buf], lane);
              mark(vissued, vpar, buf, (uint32_t)vph);
            } else {
              if (lane == 0) sm.pend[npend] = VPending{buf, vph, p, j0, ntok, r};
              __syncwarp();
              ++npend;
            }
          }
          // B row k0 + i's page is held by lane (k0 + i) % 32, slot (k0 + i) / 32:
          // each lane offers the row of the window k0 .. k0 + 31 it holds
          const int offer = pick(pg, (k0 + ((lane - k0) & 31)) >> 5);
          const int page_i = __shfl_sync(0xffffffffu, offer, (k0 + lane) & 31);
          if (lane == 0) {
            StageMeta& m = sm.meta[stage];
            m.kind = kKindExpand;
            m.ntok = ntok;
            m.p = p;
            m.len = len;
            m.last = last;
            m.k0 = k0;
            m.col0 = col0;
            m.nk = nk;
            m.buf = buf;
            m.vph = vph;
#pragma unroll
            for (int t = 0; t < kTT; ++t) m.rows[t] = rows[t];
            uint32_t bytes = (uint32_t)nk * (uint32_t)len * 2u;
            if (last) bytes += (uint32_t)ntok * (uint32_t)len * 2u;
            mbar_expect_tx(&sm.full[stage], bytes);
          }
          const uint16_t* src = nullptr;
          uint32_t off = 0;
          if (lane < nk) {
            src = d.pool + (int64_t)page_i * d.H + o;
            off = (uint32_t)(lane * kExpandCols) * 2u;
          } else if (last && lane >= kExpandRK && lane < kExpandRK + ntok) {
            src = static_cast<const uint16_t*>(P.y) + (int64_t)pick(rows, lane - kExpandRK) * P.ldy + col0;
            off = (uint32_t)(kRowsOff + (lane - kExpandRK) * kExpandCols) * 2u;
          }
          post(src, off, (uint32_t)len * 2u);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
#pragma unroll
        for (int m = 0; m < kPagesPerLane; ++m) pg[m] = pgn[m];
      }
    }
    // v rows still held back (a CTA whose ring never filled up): wait for the
    // barrier here
    if (ok && npend > 0) {
      bool open = false;
      for (uint32_t it = 0; it < lim && !open; ++it) open = barrier_open();
      if (open) release_pending();
      else ok = false;
    }
    // Tell the issuer that no stage follows: one more free slot, marked as
    // the end (a planner that gave up sends nothing; the issuer's own wait
    // then runs out).
    if (ok) {
      if (acquire()) {
        if (lane == 0) sm.cp_stop[stage] = 1;
        mbar_arrive(&sm.issue[stage]);
      } else {
        ok = false;
      }
    }
    // No copy may still be landing when the CTA exits: wait (with the
    // built-in limit) for the last phase issued on each v buffer.  On the
    // normal path the consumers have already waited for every v buffer and
    // these waits return at once; they matter when the consumers gave up,
    // which they can do while the planner never had to.
    if (lane == 0)
      for (int s2 = 0; s2 < kStages; ++s2)
        if (vissued >> s2 & 1u) (void)mbar_wait(&sm.vfull[s2], vpar >> s2 & 1u);
    if (!ok && lane == 0) report(d.error, kErrTimeout);
  } else if (warp == kCcConsumerWarps + 1) {  // ===================== issuer warp
    // Stages in ring order: wait until the planner has listed the copies,
    // then issue them (one bulk copy per lane) onto the stage's barrier.
    uint32_t stage = 0, phase = 0, issued = 0, ipar = 0;
    bool ok = true;
    for (;;) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.issue[stage], phase, lim))) {
        ok = false;
        break;
      }
      if (sm.cp_stop[stage]) break;
      if (lane < kCpMax) {
        const uint32_t e = sm.cp_desc[stage][lane];
        if (e)
          bulk_load(reinterpret_cast<unsigned char*>(&sm.st[stage][0]) + (e >> 13), sm.cp_src[stage][lane],
                    e & 0x1fffu, &sm.full[stage]);
      }
      mark(issued, ipar, stage, phase);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    // No copy issued here may still be landing when the CTA exits.
    if (lane == 0)
      for (int s2 = 0; s2 < kStages; ++s2)
        if (issued >> s2 & 1u) (void)mbar_wait(&sm.full[s2], ipar >> s2 & 1u);
    if (!ok && lane == 0) report(d.error, kErrTimeout);
  } else {  // ====================================================== consumer warps
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    // ---- shrink units: warp w takes the 16-element K steps w, w + 8, ... of
    // every stage; per step one ldmatrix.x4 brings A rows 0-7 (k, k + 8) and
    // the tile's token rows (k, k + 8): lanes 0-15 address the A rows, lanes
    // 16-31 the token rows (rows 4-7 of the MMA's N side repeat tokens 0-3;
    // those accumulator columns are never read).
    {
      const int lq = lane >> 3, lr = lane & 7;
      const int lrow = lq < 2 ? lr : kShrinkRows + (lr & 3);
      const uint32_t lofs = (uint32_t)(lrow * kShrinkPitch + (lq & 1) * 8) * 2u;
      // the K tail of 8 (m16n8k8): lanes 0-7 A rows, lanes 8-15 token rows
      const uint32_t lofs8 = (uint32_t)((lane < 8 ? lane : kShrinkRows + (lane & 3)) * kShrinkPitch) * 2u;
      uint32_t rb = 0, rph = 0;   // partial-sum buffer of this unit and its phase
      for (int64_t i = 0; i < ns && ok; ++i) {
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        float acc2[4] = {0.f, 0.f, 0.f, 0.f}, acc3[4] = {0.f, 0.f, 0.f, 0.f};
        while (true) {
          if (!mbar_wait(&sm.full[stage], phase, lim)) {
            ok = false;
            break;
          }
          const StageMeta& ms = sm.meta[stage];
          const int ntok = ms.ntok, len = ms.len, nrows = ms.nrows, last = ms.last;
          const int p = ms.p, j0 = ms.j0, k0 = ms.k0;
          const float sa = ms.sa;
          const uint32_t sbase = smem_addr(&sm.st[stage][0]);
          const int nk16 = len >> 4;
          int ks = warp;
          for (; ks + 3 * kCcConsumerWarps < nk16; ks += 4 * kCcConsumerWarps) {   // four chains in flight
            uint32_t r0[4], r1[4], r2[4], r3[4];
            ldsm_x4(r0, sbase + lofs + (uint32_t)ks * 32u);
            ldsm_x4(r1, sbase + lofs + (uint32_t)(ks + kCcConsumerWarps) * 32u);
            ldsm_x4(r2, sbase + lofs + (uint32_t)(ks + 2 * kCcConsumerWarps) * 32u);
            ldsm_x4(r3, sbase + lofs + (uint32_t)(ks + 3 * kCcConsumerWarps) * 32u);
            mma_k16<D::kBf16>(acc0, r0[0], r0[1], r0[2], r0[3]);
            mma_k16<D::kBf16>(acc1, r1[0], r1[1], r1[2], r1[3]);
            mma_k16<D::kBf16>(acc2, r2[0], r2[1], r2[2], r2[3]);
            mma_k16<D::kBf16>(acc3, r3[0], r3[1], r3[2], r3[3]);
          }
          for (; ks < nk16; ks += kCcConsumerWarps) {
            uint32_t r0[4];
            ldsm_x4(r0, sbase + lofs + (uint32_t)ks * 32u);
            mma_k16<D::kBf16>(acc0, r0[0], r0[1], r0[2], r0[3]);
          }
          if ((len & 15) && warp == nk16 % kCcConsumerWarps) {   // chunk lengths are multiples of 8
            uint32_t r0[2];
            ldsm_x2(r0, sbase + lofs8 + (uint32_t)nk16 * 32u);
            mma_k8<D::kBf16>(acc1, r0[0], r0[1]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
          if (last) {
            // lane (g, c) holds rank row g = lane / 4, tokens 2c and 2c + 1
            float* red = &sm.red[rb][0][0];
            if ((lane & 3) < 2) {
              red[warp * 32 + (lane >> 2) * kTT + 2 * (lane & 3)] = (acc0[0] + acc1[0]) + (acc2[0] + acc3[0]);
              red[warp * 32 + (lane >> 2) * kTT + 2 * (lane & 3) + 1] = (acc0[1] + acc1[1]) + (acc2[1] + acc3[1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.redbar[rb]);
            if (warp == (int)(i % kCcConsumerWarps)) {   // the eight partial sums, in warp order
              bool got = true;
              if (lane == 0) got = mbar_wait(&sm.redbar[rb], rph, lim);
              if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
                ok = false;
                break;
              }
              const int row = lane / kTT, t = lane % kTT;
              float tot = 0.f;
#pragma unroll
              for (int w = 0; w < kCcConsumerWarps; ++w) tot += red[w * 32 + lane];
              if (row < nrows && t < ntok) d.proj[p].v[(int64_t)(j0 + t) * d.v_ld + k0 + row] = sa * tot;
            }
            if (++rb == kRedBufs) {
              rb = 0;
              rph ^= 1;
            }
            break;
          }
        }
      }
    }
    // ---- grid barrier: this CTA's v rows are written.  The CTA barrier
    // orders every consumer warp's v stores before thread 0's release add,
    // which makes them visible at GPU scope with it.
    asm volatile("bar.sync 1, %0;" ::"n"(kCcConsumerWarps * 32) : "memory");
    if (threadIdx.x == 0) {
      int prev;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(d.grid_sync + kSyncCount) : "memory");
      if (prev == (int)gridDim.x - 1) {
        // the last CTA to arrive opens the barrier, then resets the count for
        // the next launch (whose CTAs arrive only after this grid has ended)
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(d.grid_sync + kSyncGen) : "memory");
        d.grid_sync[kSyncCount] = 0;
      }
    }
    // ---- expand units: thread owns 8 adjacent columns of the unit's tile
    const int col = threadIdx.x * 8;  // threads 0..255
    for (int64_t i = 0; i < ne && ok; ++i) {
      float2 acc[kTT][4];
#pragma unroll
      for (int t = 0; t < kTT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = make_float2(0.f, 0.f);
      bool first = true;
      while (true) {
        if (!mbar_wait(&sm.full[stage], phase, lim)) {
          ok = false;
          break;
        }
        const StageMeta& me = sm.meta[stage];
        const int ntok = me.ntok, len = me.len, nk = me.nk, k0 = me.k0, buf = me.buf, last = me.last;
        if (first) {
          first = false;
          if (!mbar_wait(&sm.vfull[buf], (uint32_t)me.vph, lim)) {
            ok = false;
            break;
          }
        }
        if (col < len) {
          const uint16_t* brows = &sm.st[stage][0];
          switch (ntok) {
            case 1: expand_stage<D, 1>(brows, sm.V[buf], k0, nk, col, acc); break;
            case 2: expand_stage<D, 2>(brows, sm.V[buf], k0, nk, col, acc); break;
            case 3: expand_stage<D, 3>(brows, sm.V[buf], k0, nk, col, acc); break;
            default: expand_stage<D, 4>(brows, sm.V[buf], k0, nk, col, acc); break;
          }
          if (last) {
            // the tile's y rows arrived with this stage; finish before releasing it
            const ProjDev& P = d.proj[me.p];
#pragma unroll
            for (int t = 0; t < kTT; ++t) {
              if (t < ntok) {
                float2 fy[4];
                unpack4x2<D>(*reinterpret_cast<const uint4*>(&sm.st[stage][kRowsOff + t * kExpandCols + col]), fy);
                uint4 out;
                out.x = D::pack(fy[0].x + d.s * acc[t][0].x, fy[0].y + d.s * acc[t][0].y);
                out.y = D::pack(fy[1].x + d.s * acc[t][1].x, fy[1].y + d.s * acc[t][1].y);
                out.z = D::pack(fy[2].x + d.s * acc[t][2].x, fy[2].y + d.s * acc[t][2].y);
                out.w = D::pack(fy[3].x + d.s * acc[t][3].x, fy[3].y + d.s * acc[t][3].y);
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.y) + (int64_t)me.rows[t] * P.ldy + me.col0 + col) =
                    out;
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (last) break;
      }
    }
    if (!ok && lane == 0) report(d.error, kErrTimeout);
  }
}

// ---- per-adapter scale: one value, ordered on a stream -------------------------
__global__ void set_f32_kernel(float* p, float v) { *p = v; }

// ---- adapter load: staging -> pages ---------------------------------------------
// One CTA per page-table entry: copies that row chunk (<= H elements) from the
// packed staging copy to its page and zero-fills the rest of the page.  The
// entry's projection q is the last one whose entries start at or before it
// (entries of q start at rank * rows_before[q]; a binary search over the
// pool's projection table).
__global__ void __launch_bounds__(128) scatter_kernel(const __grid_constant__ ScatterDev d) {
  for (int e = blockIdx.x; e < d.n_entries; e += gridDim.x) {
    int lo = 0, hi = d.nproj - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (d.rank * __ldg(&d.proj[mid].rows_before) <= e) lo = mid;
      else hi = mid - 1;
    }
    const ProjLayout L = d.proj[lo];
    int local = e - d.rank * L.rows_before;
    const int64_t src_base = (int64_t)d.rank * L.elems_before;
    const int na = d.rank * L.ppi;
    const uint16_t* src;
    int len;
    if (local < na) {
      const int k = local / L.ppi, c = local - k * L.ppi;
      src = d.staging + src_base + (int64_t)k * L.h_in + (int64_t)c * d.H;
      len = min(d.H, L.h_in - c * d.H);
    } else {
      local -= na;
      const int k = local / L.ppo, c = local - k * L.ppo;
      src = d.staging + src_base + (int64_t)d.rank * L.h_in + (int64_t)k * L.h_out + (int64_t)c * d.H;
      len = min(d.H, L.h_out - c * d.H);
    }
    uint16_t* dst = d.pool + (int64_t)d.pages[e] * d.H;
    for (int v = threadIdx.x; v < d.H / 8; v += blockDim.x) {
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (v * 8 < len) val = *reinterpret_cast<const uint4*>(src + v * 8);
      *reinterpret_cast<uint4*>(dst + v * 8) = val;
    }
  }
}

}  // namespace

// Programmatic dependent launch; `cooperative` also asks for every CTA of
// the grid to be resident at once (the apply kernel's CTAs wait on one
// another at its grid barrier).
template <typename Kern>
cudaError_t launch_pdl(Kern kernel, int grid, int block, size_t smem, cudaStream_t st, const ApplyDev& a,
                       bool cooperative) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

cudaError_t prepare_kernels(int /*device*/) {
  cudaError_t e = cudaFuncSetAttribute(build_segments_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSegSmemMax);
  if (e != cudaSuccess) return e;
  const int as = (int)sizeof(ApplySmem);
  if ((e = cudaFuncSetAttribute(apply_cc_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, as))) return e;
  return cudaFuncSetAttribute(apply_cc_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, as);
}

cudaError_t launch_build_segments(const SegBuildArgs& in, cudaStream_t st) {
  if (in.T <= kSmallSegMax) {
    // one token per thread; whole warps, at least two
    const int threads = in.T <= 64 ? 64 : (in.T + 31) / 32 * 32;
    build_segments_small_kernel<<<1, threads, 0, st>>>(in);
    return cudaGetLastError();
  }
  // Shared memory: the histogram, then (if they fit) the rank cache and the
  // segment arrays; anything that does not fit stays in global memory.
  SegBuildArgs a = in;
  const size_t hist = sizeof(int32_t) * (size_t)a.max_adapters;
  const size_t seg_arrays = sizeof(int32_t) * (4 * (size_t)a.seg_cap + 1);
  size_t smem = hist;
  a.smem_flags = 0;
  if (smem + hist <= (size_t)kSegSmemMax) {
    smem += hist;
    a.smem_flags |= kRankInSmem;
  }
  if (smem + seg_arrays <= (size_t)kSegSmemMax) {
    smem += seg_arrays;
    a.smem_flags |= kSegInSmem;
    const size_t keys = sizeof(int32_t) * (size_t)a.T;
    if (smem + keys <= (size_t)kSegSmemMax) {
      smem += keys;
      a.smem_flags |= kKeysInSmem;
    }
  }
  // Small batches take a smaller block: its barriers are cheaper.
  const int threads = a.T <= 256 ? 256 : a.T <= 512 ? 512 : kSegThreads;
  build_segments_kernel<<<1, threads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_apply_cc(const ApplyDev& a, int dtype, int grid, cudaStream_t st) {
  if (dtype == 0) return launch_pdl(apply_cc_kernel<F16>, grid, kCcThreads, sizeof(ApplySmem), st, a, true);
  return launch_pdl(apply_cc_kernel<BF16>, grid, kCcThreads, sizeof(ApplySmem), st, a, true);
}

cudaError_t launch_set_f32(float* p, float v, cudaStream_t st) {
  set_f32_kernel<<<1, 1, 0, st>>>(p, v);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const ScatterDev& a, cudaStream_t st) {
  if (a.n_entries <= 0) return cudaSuccess;
  int grid = a.n_entries < 1216 ? a.n_entries : 1216;
  scatter_kernel<<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace slora
