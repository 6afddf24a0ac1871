// The "traditional batched matmul" variant of the LoRA delta, kept as a
// comparator for the paged kernels ("S-LoRA: Serving Thousands of Concurrent
// LoRA Adapters", dongaigc.com summary, section "S-LoRA的性能评估", the
// comparison of S-LoRA with its own variants: one without unified memory and
// one using traditional batched matrix multiplication).
//
// Every token's adapter rows are gathered out of the pool into dense
// tensors padded to one rank r_pad (rows past the adapter's rank are zero),
// then two batched GEMMs (cuBLAS, fp32 accumulation, v kept in fp32) give
// delta_t = (x_t A_a(t)) B_a(t), and an epilogue adds s * s_a * delta_t into
// y_t with one rounding.  Tokens without an adapter get zero rows.  These
// kernels are the gather, the token map and the epilogue; the GEMMs are
// library calls made by the host.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace slora {
namespace {

template <class E>
struct Cvt;
template <>
struct Cvt<__half> {
  static __device__ __forceinline__ float to(uint16_t b) { return __half2float(__ushort_as_half(b)); }
  static __device__ __forceinline__ uint16_t from(float v) { return __half_as_ushort(__float2half_rn(v)); }
};
template <>
struct Cvt<__nv_bfloat16> {
  static __device__ __forceinline__ float to(uint16_t b) { return __bfloat162float(__ushort_as_bfloat16(b)); }
  static __device__ __forceinline__ uint16_t from(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
};

constexpr int kBmmThreads = 256;

// tok_seg[token] = segment of the token (the caller set every entry to -1).
__global__ void __launch_bounds__(kBmmThreads) bmm_map_kernel(const __grid_constant__ BmmDev d) {
  const int n = d.counts[kNSorted], S = d.counts[kNumSegs];
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x) {
    int lo = 0, hi = S - 1;   // last segment whose start is <= j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (d.seg_start[mid] <= j) lo = mid;
      else hi = mid - 1;
    }
    d.tok_seg[dbg_index(d.perm[j], d.T, d.error)] = lo;
  }
}

// One block per (token, padded rank row): A row k into a_pad[t][k][0..h_in)
// (16-bit, as stored) and B row k into b_pad[t][k][0..h_out) (fp32); zeros
// for rows at or past the adapter's rank and for tokens without an adapter.
template <class E>
__global__ void __launch_bounds__(kBmmThreads) bmm_gather_kernel(const __grid_constant__ BmmDev d) {
  const int64_t rows = (int64_t)d.T * d.r_pad;
  for (int64_t b = blockIdx.x; b < rows; b += gridDim.x) {
    const int t = (int)(b / d.r_pad), k = (int)(b - (int64_t)t * d.r_pad);
    const int s = d.tok_seg[t];
    const int a = s >= 0 ? d.seg_adapter[s] : 0;
    const int r = s >= 0 ? d.seg_rank[s] : 0;
    uint16_t* arow = d.a_pad + b * d.h_in;
    float* brow = d.b_pad + b * d.h_out;
    const int32_t* pt = d.page_table + (int64_t)a * d.pt_stride;
    for (int c8 = threadIdx.x; c8 < d.h_in / 8; c8 += blockDim.x) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (k < r) {
        const int e = c8 * 8, chunk = e / d.H;
        const int page = dbg_index(pt[(int64_t)r * d.rows_before + (int64_t)k * d.ppi + chunk], d.num_pages, d.error);
        v = *reinterpret_cast<const uint4*>(d.pool + (int64_t)page * d.H + (e - chunk * d.H));
      }
      *reinterpret_cast<uint4*>(arow + c8 * 8) = v;
    }
    for (int c8 = threadIdx.x; c8 < d.h_out / 8; c8 += blockDim.x) {
      float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (k < r) {
        const int e = c8 * 8, chunk = e / d.H;
        const int page =
            dbg_index(pt[(int64_t)r * (d.rows_before + d.ppi) + (int64_t)k * d.ppo + chunk], d.num_pages, d.error);
        const uint4 v = *reinterpret_cast<const uint4*>(d.pool + (int64_t)page * d.H + (e - chunk * d.H));
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = Cvt<E>::to(h[i]);
      }
      float4* dst = reinterpret_cast<float4*>(brow + c8 * 8);
      dst[0] = make_float4(f[0], f[1], f[2], f[3]);
      dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
}

// y_t += s * s_a * delta_t, one rounding, for tokens with an adapter.
template <class E>
__global__ void __launch_bounds__(kBmmThreads) bmm_epilogue_kernel(const __grid_constant__ BmmDev d) {
  const int n8 = d.h_out / 8;
  const int64_t total = (int64_t)d.T * n8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / n8), c = (int)(i - (int64_t)t * n8) * 8;
    const int s = d.tok_seg[t];
    if (s < 0) continue;
    const float f = d.s * (d.scale ? d.scale[d.seg_adapter[s]] : 1.f);
    uint16_t* yp = static_cast<uint16_t*>(d.y) + (int64_t)t * d.ldy + c;
    const float* dp = d.delta + (int64_t)t * d.h_out + c;
    uint4 v = *reinterpret_cast<const uint4*>(yp);
    uint16_t* h = reinterpret_cast<uint16_t*>(&v);
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = Cvt<E>::from(Cvt<E>::to(h[e]) + f * dp[e]);
    *reinterpret_cast<uint4*>(yp) = v;
  }
}

}  // namespace

cudaError_t launch_bmm_gather(const BmmDev& d, int dtype, int grid, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(d.tok_seg, 0xff, sizeof(int32_t) * (size_t)d.T, st);
  if (e != cudaSuccess) return e;
  bmm_map_kernel<<<grid, kBmmThreads, 0, st>>>(d);
  if (dtype == 0) bmm_gather_kernel<__half><<<16 * grid, kBmmThreads, 0, st>>>(d);
  else bmm_gather_kernel<__nv_bfloat16><<<16 * grid, kBmmThreads, 0, st>>>(d);
  return cudaGetLastError();
}

cudaError_t launch_bmm_epilogue(const BmmDev& d, int dtype, int grid, cudaStream_t st) {
  if (dtype == 0) bmm_epilogue_kernel<__half><<<8 * grid, kBmmThreads, 0, st>>>(d);
  else bmm_epilogue_kernel<__nv_bfloat16><<<8 * grid, kBmmThreads, 0, st>>>(d);
  return cudaGetLastError();
}

}  // namespace slora
