// CUDA-core kernels of the heterogeneous-batch LoRA path (sm_103a):
//   build_segments  -- stable grouping of the batch's tokens by adapter
//   shrink_cc       -- v[j, k] = x[perm[j], :] . A_a[:, k]   (gather, HBM-bound)
//   expand_cc       -- y[perm[j], n] += s * sum_k v[j, k] B_a[k, n]
//   scatter         -- adapter load: staged rows -> their pool pages
//
// The method ("S-LoRA: Serving Thousands of Concurrent LoRA Adapters";
// dongaigc.com summary, section 2 "heterogeneous batching"; nubint.ai review,
// method list) batches the LoRA part of tokens that use different adapters of
// different ranks in one pass, reading adapter weights directly from
// non-contiguous pool pages.  At decode shapes the arithmetic intensity is
// below 2 flop/byte, so these kernels are organised around HBM traffic: each
// distinct adapter's page rows are streamed once per token tile with 128-bit
// loads, x and y rows are touched once per rank chunk / column tile, and
// persistent grids walk flattened work lists built by build_segments.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include "internal.h"

namespace slora {
namespace {

// ---- 16-bit element helpers ------------------------------------------------
struct F16 {
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

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

template <class D>
__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  float2 a = D::unpack(v.x), b = D::unpack(v.y), c = D::unpack(v.z), e = D::unpack(v.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = e.x; f[7] = e.y;
}

template <class D>
__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  float fa[8], fb[8];
  unpack8<D>(a, fa);
  unpack8<D>(b, fb);
#pragma unroll
  for (int e = 0; e < 8; ++e) acc = fmaf(fa[e], fb[e], acc);
  return acc;
}

// Largest s in [0, S) with off[s] <= item; off is a non-decreasing prefix
// array with off[S] > item, so segment s holds work unit `item`.
__device__ __forceinline__ int find_seg(const int32_t* off, int S, int item) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Block-wide exclusive scan of K ints per thread; sh holds 33*K ints.
template <int K>
__device__ __forceinline__ void block_scan_excl(int (&v)[K], int (&total)[K], int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
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
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
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
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    v[k] = inc[k] - v[k] + sh[warp * K + k];
    total[k] = sh[32 * K + k];
  }
  __syncthreads();
}

// ---- build_segments ----------------------------------------------------------
// One CTA of 1024 threads.  (1) histogram of adapter ids in shared memory,
// (2) exclusive scan -> segment starts in ascending adapter id, (3) stable
// scatter of token indices: tokens are visited in order, 1024 at a time; a
// token's position is its adapter's running start + the number of earlier
// tokens of the same adapter in this tile (same warp: match_any + popc;
// earlier warps: their per-warp (adapter, count) groups), (4) per-segment
// work-unit counts and their prefix sums for the apply kernels.
__global__ void __launch_bounds__(kSegThreads) build_segments_kernel(const SegBuildArgs args) {
  extern __shared__ int32_t hist[];  // [max_adapters]
  __shared__ int32_t grp_key[32][32];
  __shared__ int32_t grp_cnt[32][32];
  __shared__ int32_t ngrp[32];
  __shared__ int32_t scan_sh[33 * 6];
  __shared__ int32_t s_bad, s_err;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int A = args.max_adapters, T = args.T;
  const SegDev& sd = args.seg;

  for (int a = tid; a < A; a += blockDim.x) hist[a] = 0;
  if (tid == 0) {
    s_bad = 0;
    s_err = 0;
  }
  __syncthreads();

  // (1) histogram; ids that are out of range or not resident are left out
  for (int i = tid; i < T; i += blockDim.x) {
    const int a = args.token_adapter[i];
    if (a == -1) continue;
    if (a < -1 || a >= A) {
      atomicAdd(&s_bad, 1);
      atomicCAS(&s_err, 0, -1 /* SLORA_ERR_INVALID */);
      continue;
    }
    if (args.rank[a] <= 0) {
      atomicAdd(&s_bad, 1);
      atomicCAS(&s_err, 0, -4 /* SLORA_ERR_NOT_RESIDENT */);
      continue;
    }
    atomicAdd(&hist[a], 1);
  }
  __syncthreads();

  // (2) segments in ascending adapter id; hist[a] becomes a's running start
  int segs = 0, pos = 0;
  for (int base = 0; base < A; base += blockDim.x) {
    const int a = base + tid;
    const int c = a < A ? hist[a] : 0;
    int v[2] = {c, c > 0 ? 1 : 0}, tot[2];
    block_scan_excl<2>(v, tot, scan_sh);
    if (c > 0) {
      sd.seg_adapter[segs + v[1]] = a;
      sd.seg_start[segs + v[1]] = pos + v[0];
      hist[a] = pos + v[0];
    }
    pos += tot[0];
    segs += tot[1];
  }
  if (tid == 0) {
    sd.seg_start[segs] = pos;
    sd.counts[kNumSegs] = segs;
    sd.counts[kNSorted] = pos;
    sd.counts[kBadTokens] = s_bad;
    if (s_err != 0) atomicCAS(args.error, 0, s_err);
  }
  __syncthreads();

  // (3) stable scatter, one tile of 1024 tokens at a time, in token order
  const unsigned lt = (1u << lane) - 1u;
  for (int base = 0; base < T; base += blockDim.x) {
    const int i = base + tid;
    int key = -1;
    bool valid = false;
    if (i < T) {
      key = args.token_adapter[i];
      valid = key >= 0 && key < A && args.rank[key] > 0;
    }
    const int k2 = valid ? key : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, k2);
    const int rank_w = __popc(peers & lt);
    const bool leader = (peers & lt) == 0u;
    const unsigned lead_mask = __ballot_sync(0xffffffffu, valid && leader);
    if (valid && leader) {
      const int slot = __popc(lead_mask & lt);
      grp_key[warp][slot] = key;
      grp_cnt[warp][slot] = __popc(peers);
    }
    if (lane == 0) ngrp[warp] = __popc(lead_mask);
    __syncthreads();
    if (valid) {
      int p = hist[key] + rank_w;
      for (int w = 0; w < warp; ++w) {
        const int ng = ngrp[w];
        for (int g = 0; g < ng; ++g)
          if (grp_key[w][g] == key) p += grp_cnt[w][g];
      }
      sd.perm[p] = i;
    }
    __syncthreads();
    if (valid && leader) atomicAdd(&hist[key], __popc(peers));
    __syncthreads();
  }

  // (4) work units per segment and their prefix sums
  int carry[6] = {0, 0, 0, 0, 0, 0};
  for (int base = 0; base < segs; base += blockDim.x) {
    const int s = base + tid;
    int q[6] = {0, 0, 0, 0, 0, 0};
    if (s < segs) {
      const int len = sd.seg_start[s + 1] - sd.seg_start[s];
      const int r = args.rank[sd.seg_adapter[s]];
      sd.seg_rank[s] = r;
      const int ntt = (len + kTT - 1) / kTT;
      const int nrc = (r + kShrinkRows - 1) / kShrinkRows;
      const int nmt = (len + kTcM - 1) / kTcM;
      const bool is_short = len < args.tc_threshold;
      q[0] = ntt * nrc;
      q[1] = ntt;
      q[2] = is_short ? ntt * nrc : 0;
      q[3] = is_short ? ntt : 0;
      q[4] = nmt;
      q[5] = is_short ? 0 : nmt;
    }
    int tot[6];
    block_scan_excl<6>(q, tot, scan_sh);
    if (s < segs) {
      sd.cc_shrink_all[s] = carry[0] + q[0];
      sd.cc_tile_all[s] = carry[1] + q[1];
      sd.cc_shrink_short[s] = carry[2] + q[2];
      sd.cc_tile_short[s] = carry[3] + q[3];
      sd.tc_tile_all[s] = carry[4] + q[4];
      sd.tc_tile_long[s] = carry[5] + q[5];
    }
#pragma unroll
    for (int k = 0; k < 6; ++k) carry[k] += tot[k];
  }
  if (tid == 0) {
    sd.cc_shrink_all[segs] = carry[0];
    sd.cc_tile_all[segs] = carry[1];
    sd.cc_shrink_short[segs] = carry[2];
    sd.cc_tile_short[segs] = carry[3];
    sd.tc_tile_all[segs] = carry[4];
    sd.tc_tile_long[segs] = carry[5];
    sd.counts[kCcShrinkAll] = carry[0];
    sd.counts[kCcTileAll] = carry[1];
    sd.counts[kCcShrinkShort] = carry[2];
    sd.counts[kCcTileShort] = carry[3];
    sd.counts[kTcTileAll] = carry[4];
    sd.counts[kTcTileLong] = carry[5];
  }
}

// ---- shrink: v = x A (CUDA cores) -----------------------------------------------
// Work unit = (projection, segment, token tile of <= kTT tokens, chunk of 8
// rank rows).  Warp w owns rank row k = chunk*8 + w: it streams that A row
// (one page per H elements) once with 16-byte loads and dots it against the
// tile's x rows (which the CTA's 8 warps share through L1), then reduces the
// per-lane partial sums with shuffles.
template <class D>
__global__ void __launch_bounds__(kShrinkThreads) shrink_cc_kernel(const __grid_constant__ ApplyDev d) {
  const int total = d.counts[d.shrink_total_idx];
  const int S = d.counts[kNumSegs];
  const int64_t G = (int64_t)total * d.nproj;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t g = blockIdx.x; g < G; g += gridDim.x) {
    const int p = (int)(g / total);
    const int item = (int)(g - (int64_t)p * total);
    const ProjDev& P = d.proj[p];
    const int s = find_seg(d.shrink_off, S, item);
    const int local = item - __ldg(d.shrink_off + s);
    const int r = __ldg(d.seg_rank + s);
    const int nrc = (r + kShrinkRows - 1) / kShrinkRows;
    const int tt = local / nrc, rc = local - tt * nrc;
    const int j0 = __ldg(d.seg_start + s) + tt * kTT;
    const int ntok = min(kTT, __ldg(d.seg_start + s + 1) - j0);
    const int k = rc * kShrinkRows + warp;
    if (k >= r) continue;
    const int a = __ldg(d.seg_adapter + s);
    const int32_t* pt = d.page_table + (int64_t)a * d.pt_stride +
                        (int64_t)r * P.rows_before + (int64_t)k * P.ppi;
    const uint16_t* xr[kTT];
#pragma unroll
    for (int t = 0; t < kTT; ++t)
      xr[t] = static_cast<const uint16_t*>(P.x) +
              (int64_t)__ldg(d.perm + j0 + min(t, ntok - 1)) * P.ldx;
    float acc[kTT];
#pragma unroll
    for (int t = 0; t < kTT; ++t) acc[t] = 0.f;

    for (int chunk = 0; chunk < P.ppi; ++chunk) {
      const uint16_t* page = d.pool + (int64_t)__ldg(pt + chunk) * d.H;
      const int c0 = chunk * d.H;
      const int n8 = min(d.H, P.h_in - c0) >> 3;  // 16-byte vectors in this chunk
      for (int v0 = lane; v0 < n8; v0 += 32 * 4) {
        uint4 av[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int vv = v0 + u * 32;
          av[u] = vv < n8 ? ldg16(page + vv * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int t = 0; t < kTT; ++t) {
          if (t < ntok) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int vv = v0 + u * 32;
              if (vv < n8) acc[t] = dot8<D>(av[u], ldg16(xr[t] + c0 + vv * 8), acc[t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kTT; ++t) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    }
    float mine = acc[0];
#pragma unroll
    for (int t = 1; t < kTT; ++t)
      if (lane == t) mine = acc[t];
    if (lane < ntok) P.v[(int64_t)(j0 + lane) * d.v_ld + k] = mine;
  }
}

// ---- expand: y += s v B (CUDA cores) ------------------------------------------
// Work unit = (projection, segment, token tile, column tile of 1024).  The
// tile's v rows go to shared memory; each thread owns 8 adjacent output
// columns (one 16-byte vector), streams the adapter's B rows for them
// (8 rows in flight), accumulates in fp32 for every token of the tile, then
// reads y once, adds s * acc, rounds once and writes y back.
template <class D>
__global__ void __launch_bounds__(kExpandThreads) expand_cc_kernel(const __grid_constant__ ApplyDev d) {
  __shared__ float vt[kTT][kMaxRank];
  const int tiles = d.counts[d.tile_total_idx];
  const int S = d.counts[kNumSegs];
  int64_t G = 0;
  for (int p = 0; p < d.nproj; ++p) G += (int64_t)tiles * d.proj[p].ncol_tiles;
  for (int64_t g = blockIdx.x; g < G; g += gridDim.x) {
    int p = 0;
    int64_t gg = g;
    while (gg >= (int64_t)tiles * d.proj[p].ncol_tiles) {
      gg -= (int64_t)tiles * d.proj[p].ncol_tiles;
      ++p;
    }
    const ProjDev& P = d.proj[p];
    const int tile = (int)(gg / P.ncol_tiles);
    const int ct = (int)(gg - (int64_t)tile * P.ncol_tiles);
    const int s = find_seg(d.tile_off, S, tile);
    const int tt = tile - __ldg(d.tile_off + s);
    const int j0 = __ldg(d.seg_start + s) + tt * kTT;
    const int ntok = min(kTT, __ldg(d.seg_start + s + 1) - j0);
    const int r = __ldg(d.seg_rank + s);
    const int a = __ldg(d.seg_adapter + s);
    __syncthreads();  // vt of the previous unit is no longer read
    for (int e = threadIdx.x; e < ntok * r; e += blockDim.x) {
      const int t = e / r, k = e - t * r;
      vt[t][k] = P.v[(int64_t)(j0 + t) * d.v_ld + k];
    }
    __syncthreads();
    const int col = ct * kExpandCols + threadIdx.x * 8;
    if (col >= P.h_out) continue;
    const int chunk = col / d.H, off = col - chunk * d.H;
    const int32_t* ptB = d.page_table + (int64_t)a * d.pt_stride +
                         (int64_t)r * (P.rows_before + P.ppi) + chunk;
    float acc[kTT][8];
#pragma unroll
    for (int t = 0; t < kTT; ++t)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;

    constexpr int U = 8;
    int k = 0;
    for (; k + U <= r; k += U) {
      uint4 b[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        b[u] = ldg16(d.pool + (int64_t)__ldg(ptB + (int64_t)(k + u) * P.ppo) * d.H + off);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float bf[8];
        unpack8<D>(b[u], bf);
#pragma unroll
        for (int t = 0; t < kTT; ++t) {
          if (t < ntok) {
            const float vv = vt[t][k + u];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[t][e] = fmaf(vv, bf[e], acc[t][e]);
          }
        }
      }
    }
    for (; k < r; ++k) {
      float bf[8];
      unpack8<D>(ldg16(d.pool + (int64_t)__ldg(ptB + (int64_t)k * P.ppo) * d.H + off), bf);
#pragma unroll
      for (int t = 0; t < kTT; ++t) {
        if (t < ntok) {
          const float vv = vt[t][k];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[t][e] = fmaf(vv, bf[e], acc[t][e]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kTT; ++t) {
      if (t < ntok) {
        const int row = __ldg(d.perm + j0 + t);
        uint4* yp = reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.y) + (int64_t)row * P.ldy + col);
        uint4 yv = *yp;
        float yf[8];
        unpack8<D>(yv, yf);
#pragma unroll
        for (int e = 0; e < 8; ++e) yf[e] = yf[e] + d.s * acc[t][e];
        yv.x = D::pack(yf[0], yf[1]);
        yv.y = D::pack(yf[2], yf[3]);
        yv.z = D::pack(yf[4], yf[5]);
        yv.w = D::pack(yf[6], yf[7]);
        *yp = yv;
      }
    }
  }
}

// ---- adapter load: staging -> pages ---------------------------------------------
// One CTA per page-table entry: copies that row chunk (<= H elements) from the
// packed staging copy to its page and zero-fills the rest of the page.
__global__ void __launch_bounds__(128) scatter_kernel(const __grid_constant__ ScatterDev d) {
  for (int e = blockIdx.x; e < d.n_entries; e += gridDim.x) {
    int q = 0;
    while (q + 1 < d.nproj && e >= d.entry_base[q + 1]) ++q;
    int local = e - d.entry_base[q];
    const int na = d.rank * d.ppi[q];
    const uint16_t* src;
    int len;
    if (local < na) {
      const int k = local / d.ppi[q], c = local - k * d.ppi[q];
      src = d.staging + d.src_base[q] + (int64_t)k * d.h_in[q] + (int64_t)c * d.H;
      len = min(d.H, d.h_in[q] - c * d.H);
    } else {
      local -= na;
      const int k = local / d.ppo[q], c = local - k * d.ppo[q];
      src = d.staging + d.src_base[q] + (int64_t)d.rank * d.h_in[q] + (int64_t)k * d.h_out[q] +
            (int64_t)c * d.H;
      len = min(d.H, d.h_out[q] - c * d.H);
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

cudaError_t prepare_kernels(int /*device*/) {
  return cudaFuncSetAttribute(build_segments_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(sizeof(int32_t) * kMaxAdapters));
}

cudaError_t launch_build_segments(const SegBuildArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(int32_t) * (size_t)a.max_adapters;
  build_segments_kernel<<<1, kSegThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_shrink_cc(const ApplyDev& a, int dtype, int grid, cudaStream_t st) {
  if (dtype == 0) shrink_cc_kernel<F16><<<grid, kShrinkThreads, 0, st>>>(a);
  else shrink_cc_kernel<BF16><<<grid, kShrinkThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_expand_cc(const ApplyDev& a, int dtype, int grid, cudaStream_t st) {
  if (dtype == 0) expand_cc_kernel<F16><<<grid, kExpandThreads, 0, st>>>(a);
  else expand_cc_kernel<BF16><<<grid, kExpandThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const ScatterDev& a, cudaStream_t st) {
  if (a.n_entries <= 0) return cudaSuccess;
  int grid = a.n_entries < 1216 ? a.n_entries : 1216;
  scatter_kernel<<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

int occupancy_shrink_cc(int dtype) {
  int n = 0;
  if (dtype == 0) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, shrink_cc_kernel<F16>, kShrinkThreads, 0);
  else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, shrink_cc_kernel<BF16>, kShrinkThreads, 0);
  return n > 0 ? n : 1;
}

int occupancy_expand_cc(int dtype) {
  int n = 0;
  if (dtype == 0) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, expand_cc_kernel<F16>, kExpandThreads, 0);
  else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, expand_cc_kernel<BF16>, kExpandThreads, 0);
  return n > 0 ? n : 1;
}

}  // namespace slora
