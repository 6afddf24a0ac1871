// Tensor-core (tcgen05) kernels of the LoRA delta for long segments (prefill).
//
// A segment of many tokens on one adapter turns the per-token products into
// dense contractions ("S-LoRA: Serving Thousands of Concurrent LoRA
// Adapters": heterogeneous batching runs custom kernels directly on the
// non-contiguous pool; the pages give no kernel internals).  Tiles of one
// segment are multiplied on the 5th-generation tensor cores, fp16/bf16
// operands from shared memory, fp32 accumulators in TMEM:
//
//   tc_shrink:  V^T[r x 256] = A[r x H_in] . X^T   (A rows = pages; rank on M, tokens on N)
//   tc_combine: V = s_a (sum of tc_shrink's K parts), written as V_hi and V_lo
//   tc_expand:  Y[128 x 128] += s * (V_hi + V_lo)[128 x r] . B[r x 128]
//
// tc_shrink copies token rows of x and adapter rows of A with cp.async into
// the 128-byte-swizzled layout the MMA reads; tc_expand gathers B rows with
// the TMA engine (`tile::gather4` over the page pool viewed as a [pages x H]
// matrix) and loads v and y tiles as 2-D boxes or row gathers.  V is carried
// as two 16-bit halves, V_hi = round(v) and V_lo = round(v - V_hi), so the
// expand multiplies with ~fp32 accuracy on 16-bit tensor cores.
//
// tc_shrink and tc_expand are persistent (one CTA per SM) and warp-
// specialised: copy warps fill a ring of shared-memory stages, warp 1 owns
// TMEM and issues the MMAs (one thread), the epilogue warps drain TMEM
// accumulators (more than one, so the epilogue of one tile overlaps the MMAs
// of the next) and write partial sums of v or y.  Every wait is bounded
// (SLORA_ERR_TIMEOUT on give-up).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace slora {
namespace {

using namespace ptx;

constexpr int kTcThreads = 6 * 32;
constexpr int kRowBytes = kTcK * 2;  // one 64-element K (or N) row of a swizzle atom = 128 bytes

__device__ __forceinline__ void report_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Largest q with off[q] <= item (prefix array, shared memory when it fits).
__device__ __forceinline__ int find_pos_tc(const int32_t* s_off, const int32_t* g_off, bool in_smem, int S,
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

template <class T>
struct Elem;
template <>
struct Elem<__half> {
  static __device__ __forceinline__ uint16_t from(float f) { return __half_as_ushort(__float2half_rn(f)); }
  static __device__ __forceinline__ float to(uint16_t u) { return __half2float(__ushort_as_half(u)); }
  // a pair packed in 32 bits (first value in the low half)
  static __device__ __forceinline__ uint32_t from2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 to2(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ uint16_t from(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
  static __device__ __forceinline__ float to(uint16_t u) { return __bfloat162float(__ushort_as_bfloat16(u)); }
  static __device__ __forceinline__ uint32_t from2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 to2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  }
};

// ================================================================ tc_shrink
// v^T = A_a x^T, one unit per (token tile, projection, K part).  The
// adapter's A rows are the MMA's M side (128 rows, the rank padded) and the
// tile's tokens its N side (up to 256).  A tcgen05 MMA of 128 x N x 16 costs
// the same for every N up to 256, so this way round each MMA covers up to 256
// tokens instead of the rank's 8..128 columns.  Ranks above 128 take two M
// blocks (two accumulators) and tiles of 128 tokens.
//
// Warps: 1 issues the MMAs, 2-5 drain TMEM, 6-13 copy each stage's token
// rows (x) and adapter rows (A); warp 0 has no role.  Rows go through the
// load/store unit: each loader thread copies one 16-byte chunk column of every
// 32nd row with cp.async, straight to its 128-byte-swizzled place, and has the
// copies themselves arrive on the stage's barrier when they land
// (cp.async.mbarrier.arrive), so a loader runs up to the whole ring ahead
// without waiting for its own copies; the MMA warp fences the async proxy
// after its wait, before the tensor cores read the stage.
//
// The K range of (tile, projection) is split into up to kShParts parts (units
// of their own, so that a short list of tiles still spreads over the CTAs).
// Each part writes its fp32 partial sums; tc_combine then adds the parts in
// order and writes s_a v as its 16-bit hi and lo halves.
constexpr int kShrinkTcStages = 4;
constexpr int kShrinkLoaderWarps = 8;
constexpr int kShrinkLoaders = kShrinkLoaderWarps * 32;
constexpr int kShrinkTcThreads = kTcThreads + kShrinkLoaders;
constexpr int kLoaderRowStep = kShrinkLoaders / (kRowBytes / 16);   // 32 rows between one thread's rows
constexpr int kShTokWide = 256;                                     // tokens per unit when r <= 128
constexpr int kShTokNarrow = 128;                                   // tokens per unit when r > 128
constexpr int kShStageBytes = (kShTokWide + kTcM) * kRowBytes;      // 48 KB: x rows, then A rows
static_assert((kShTokNarrow + 2 * kTcM) * kRowBytes == kShStageBytes, "both stage layouts fill a stage");
constexpr int kShParts = kTcShrinkParts;
constexpr int kShTmemCols = 2 * kShTokWide;                          // two accumulator buffers
constexpr int kShMaxRows = kShTokWide / kLoaderRowStep;              // x or A rows one loader thread covers
struct TcShrinkSmem {
  uint8_t st[kShrinkTcStages][kShStageBytes];
  uint64_t full[kShrinkTcStages], empty[kShrinkTcStages], tfull[2], tempty[2];
  uint32_t tmem_slot;
  int32_t off[kSegSmem];    // tensor-core 128-token tile list (prefix per work-order position)
  int32_t uoff[kSegSmem];   // unit tiles per position (256 tokens when r <= 128, else 128)
};

__device__ __forceinline__ void cp16_shared(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// The first `bytes` (0..16) of the chunk from global memory, the rest zeros.
__device__ __forceinline__ void cp16_shared_zfill(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// Shrink unit g: part fastest, then projection, then unit tile.
struct ShUnit {
  int tile, p, part, nparts, kb_lo, kb_hi;
  int j0, ntok, tok, r, a;   // tok: the tile's token capacity (kShTokWide or kShTokNarrow)
  bool skip;
};
__device__ __forceinline__ ShUnit sh_unit(const TcDev& t, const int32_t* uoff, bool wide_ok, int S, int64_t g) {
  const ApplyDev& d = t.a;
  ShUnit s;
  s.part = (int)(g % kShParts);
  const int64_t tp = g / kShParts;
  s.tile = (int)(tp / d.nproj);
  s.p = (int)(tp - (int64_t)s.tile * d.nproj);
  const int nkb = (d.proj[s.p].h_in + kTcK - 1) / kTcK;
  s.nparts = min(kShParts, nkb);
  s.skip = s.part >= s.nparts;
  s.kb_lo = nkb * s.part / s.nparts;
  s.kb_hi = nkb * (s.part + 1) / s.nparts;
  const int q = find_pos_tc(uoff, t.tc_off, wide_ok, S, s.tile);
  const int mt = s.tile - (wide_ok ? uoff[q] : __ldg(t.tc_off + q));
  const int4 sd = __ldg(d.seg_desc + q);   // adapter, rank, start, end
  s.a = sd.x;
  s.r = sd.y;
  s.tok = wide_ok && s.r <= kTcM ? kShTokWide : kShTokNarrow;
  s.j0 = sd.z + mt * s.tok;
  s.ntok = min(s.tok, sd.w - s.j0);
  return s;
}

template <class E>
__global__ void __launch_bounds__(kShrinkTcThreads, 1) tc_shrink_kernel(const __grid_constant__ TcDev t) {
  extern __shared__ uint8_t smem_raw[];
  TcShrinkSmem& sm = *reinterpret_cast<TcShrinkSmem*>(smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const ApplyDev& d = t.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 1) tmem_alloc(&sm.tmem_slot, kShTmemCols);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kShrinkTcStages; ++s) {
      mbar_init(&sm.full[s], kShrinkLoaders);   // every loader thread
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], 4);
    }
    mbar_fence_init();
  }
  pdl_wait();
  const int tiles = d.counts[t.tc_total_idx];
  const int S = d.counts[kNumSegs];
  // Wide unit tiles need the per-position list of unit tiles, built here in
  // shared memory when it fits; otherwise every unit tile is a 128-token tile.
  const bool wide_ok = S + 1 <= kSegSmem;
  if (wide_ok)
    for (int i = threadIdx.x; i <= S; i += blockDim.x) sm.off[i] = t.tc_off[i];
  __syncthreads();
  if (wide_ok && warp == 0) {
    const int per = (S + 31) >> 5;   // positions per lane
    const int lo = min(S, lane * per), hi = min(S, lo + per);
    auto units = [&](int q) -> int {
      const int n = sm.off[q + 1] - sm.off[q];
      return __ldg(d.seg_desc + q).y <= kTcM ? (n + 1) >> 1 : n;
    };
    int sum = 0;
    for (int q = lo; q < hi; ++q) sum += units(q);
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    int run = inc - sum;
    for (int q = lo; q < hi; ++q) {
      sm.uoff[q] = run;
      run += units(q);
    }
    if (lane == 31) sm.uoff[S] = inc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = sm.tmem_slot;
  const int utiles = wide_ok ? sm.uoff[S] : tiles;
  const int64_t G = (int64_t)utiles * d.nproj * kShParts;
  constexpr bool bf16 = std::is_same<E, __nv_bfloat16>::value;
  bool ok = true;

  if (warp == 0) {
    // no role
  } else if (warp == 1) {  // ----------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0;
    int n = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const ShUnit su = sh_unit(t, sm.uoff, wide_ok, S, g);
      if (su.skip) continue;
      const int ab = n & 1;
      bool got = true;
      if (lane == 0) got = mbar_wait(&sm.tempty[ab], ((n >> 1) & 1) ^ 1);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int nmb = su.r > kTcM ? 2 : 1;   // M blocks of 128 rank rows
      const uint32_t idesc = umma_idesc_f16(kTcM, (su.ntok + 15) & ~15, bf16, false);
      const uint32_t dtm = tmem + (uint32_t)(ab * kShTokWide);
      for (int kb = su.kb_lo; kb < su.kb_hi; ++kb) {
        if (lane == 0) got = mbar_wait(&sm.full[stage], phase);
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the loaders' cp.async writes (generic proxy), ordered before this
        // point by the barrier, become visible to the MMAs' async-proxy reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) {
          const uint32_t xa = smem_addr(sm.st[stage]), aa = xa + (uint32_t)su.tok * kRowBytes;
#pragma unroll
          for (int ks = 0; ks < kTcK / 16; ++ks)
            for (int mb = 0; mb < nmb; ++mb)
              umma_f16(dtm + (uint32_t)(mb * kShTokNarrow), umma_desc_sw128(aa + mb * kTcM * kRowBytes + ks * 32, 16, 1024),
                       umma_desc_sw128(xa + ks * 32, 16, 1024), idesc, (kb != su.kb_lo || ks) ? 1u : 0u);
          umma_commit(&sm.empty[stage]);  // the stage is free once these MMAs have read it
        }
        __syncwarp();
        if (++stage == kShrinkTcStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&sm.tfull[ab]);
      __syncwarp();
      ++n;
    }
  } else if (warp >= 6) {  // ------------------------------------ x-row and A-row loaders
    const int lt = threadIdx.x - 6 * 32;    // 0 .. kShrinkLoaders - 1
    const int ch = lt & 7;                  // 16-byte chunk column of the 128-byte row
    const int row0 = lt >> 3;               // rows row0, row0 + kLoaderRowStep, ...
    uint32_t stage = 0, phase = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const ShUnit su = sh_unit(t, sm.uoff, wide_ok, S, g);
      if (su.skip) continue;
      const ProjDev& P = d.proj[su.p];
      const int32_t* pt = d.page_table + (int64_t)su.a * d.pt_stride + (int64_t)su.r * P.rows_before;
      const int nrow = (su.r - row0 + kLoaderRowStep - 1) / kLoaderRowStep;    // my A rows below r
      const int nxr = (su.ntok - row0 + kLoaderRowStep - 1) / kLoaderRowStep;  // my x rows below ntok
      // my x rows (rows past the tile's end are not loaded: those
      // accumulator columns are never read)
      const uint16_t* xrow[kShMaxRows];
#pragma unroll
      for (int j = 0; j < kShMaxRows; ++j)
        xrow[j] = j < nxr ? static_cast<const uint16_t*>(P.x) +
                                (int64_t)dbg_index(__ldg(d.perm + su.j0 + row0 + kLoaderRowStep * j), d.T, d.error) *
                                    P.ldx
                          : nullptr;
      int chunk = -1;
      int pg[kShMaxRows];
      for (int kb = su.kb_lo; kb < su.kb_hi; ++kb) {
        const int k0 = kb * kTcK, c = k0 / d.H, o = k0 - c * d.H;
        if (c != chunk) {  // pages of my rows for this page chunk
          chunk = c;
#pragma unroll
          for (int j = 0; j < kShMaxRows; ++j)
            pg[j] = j < nrow ? dbg_index(__ldg(pt + (int64_t)(row0 + kLoaderRowStep * j) * P.ppi + c), d.num_pages, d.error)
                             : 0;
        }
        if (!mbar_wait(&sm.empty[stage], phase ^ 1)) {
          ok = false;
          break;
        }
        const uint32_t xbase = smem_addr(sm.st[stage]), abase = xbase + (uint32_t)su.tok * kRowBytes;
#pragma unroll
        for (int j = 0; j < kShMaxRows; ++j) {
          if (j < nrow) {
            const int row = row0 + kLoaderRowStep * j;
            cp16_shared(abase + row * kRowBytes + ((ch ^ (row & 7)) << 4), d.pool + (int64_t)pg[j] * d.H + o + ch * 8);
          }
        }
        // x: columns past h_in are zero-filled (A's are zero in its pages)
        const int e = k0 + ch * 8;
        const uint32_t xbytes = (uint32_t)min(16, max(0, 2 * (P.h_in - e)));
#pragma unroll
        for (int j = 0; j < kShMaxRows; ++j) {
          if (j < nxr) {
            const int m = row0 + kLoaderRowStep * j;
            cp16_shared_zfill(xbase + m * kRowBytes + ((ch ^ (m & 7)) << 4), xrow[j] + (xbytes ? e : 0), xbytes);
          }
        }
        // one of the stage's kShrinkLoaders arrivals, made when all of this
        // thread's copies so far have landed
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&sm.full[stage])) : "memory");
        if (++stage == kShrinkTcStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {  // ------------------------------------------------- epilogue (warps 2-5)
    // Warp w owns TMEM lanes 32 (w % 4) .. +31: rank rows k (and k + 128 in
    // the second M block); accumulator columns are the tile's tokens.  For
    // each token the warp's 32 lanes write 32 consecutive ranks of its
    // part's partial row.
    const int quarter = warp & 3;
    int n = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const ShUnit su = sh_unit(t, sm.uoff, wide_ok, S, g);
      if (su.skip) continue;
      const int ab = n & 1;
      bool got = true;
      if (lane == 0) got = mbar_wait(&sm.tfull[ab], (n >> 1) & 1);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      ++n;
      tc_fence_after();
      const int nmb = su.r > kTcM ? 2 : 1;
      const uint32_t tacc = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(ab * kShTokWide);
      // this warp's partial rows (rank rows below r)
      if (32 * quarter < su.r || nmb == 2) {
        float* part = t.vpart + (int64_t)su.part * t.vpart_part + (int64_t)su.p * t.vpart_proj;
        for (int mb = 0; mb < nmb; ++mb) {
          const int k = mb * kTcM + 32 * quarter + lane;
          for (int c00 = 0; c00 < su.ntok; c00 += 32) {
            uint32_t raw[32];
            tmem_ld32_nowait(tacc + (uint32_t)(mb * kShTokNarrow + c00), raw);
            tmem_wait_ld(raw);
            if (k < su.r) {
              float* dst = part + (int64_t)(su.j0 + c00) * d.v_ld + k;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c00 + i < su.ntok) dst[(int64_t)i * d.v_ld] = __uint_as_float(raw[i]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tempty[ab]);
    }
  }
  if (!ok && lane == 0) report_err(d.error, kErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kShTmemCols);
  }
}

// ================================================================ tc_combine
// v of the tensor-core tiles from tc_shrink's K parts: their fp32 partial rows
// added in part order, times s_a, written as 16-bit hi and lo halves (zeros
// from r up to the next multiple of 16, which tc_expand reads as K padding).
// Block = 32 tokens of a 128-token tile and one projection; consecutive
// threads take consecutive ranks of a token row, and each thread loads
// kCombineUnroll elements' partial sums before it adds any of them.
constexpr int kCombineThreads = 256;
constexpr int kCombineTokens = 32;
constexpr int kCombineUnroll = 4;
template <class E>
__global__ void __launch_bounds__(kCombineThreads) tc_combine_kernel(const __grid_constant__ TcDev t) {
  __shared__ int32_t s_off[kSegSmem];   // the tile list's prefix, searched here when it fits
  const ApplyDev& d = t.a;
  pdl_wait();
  const int tiles = d.counts[t.tc_total_idx];
  const int S = d.counts[kNumSegs];
  pdl_trigger();
  const bool off_smem = S + 1 <= kSegSmem;
  if (off_smem)
    for (int i = threadIdx.x; i <= S; i += kCombineThreads) s_off[i] = __ldg(t.tc_off + i);
  __syncthreads();
  constexpr int kGroups = kTcM / kCombineTokens;
  const int64_t nblk = (int64_t)tiles * d.nproj * kGroups;
  for (int64_t b = blockIdx.x; b < nblk; b += gridDim.x) {
    const int tile = (int)(b / (d.nproj * kGroups));
    const int rem = (int)(b - (int64_t)tile * d.nproj * kGroups);
    const int p = rem / kGroups, grp = rem - p * kGroups;
    const int q = find_pos_tc(s_off, t.tc_off, off_smem, S, tile);
    const int4 sd = __ldg(d.seg_desc + q);   // adapter, rank, start, end
    const int j0 = sd.z + (tile - (off_smem ? s_off[q] : __ldg(t.tc_off + q))) * kTcM + grp * kCombineTokens;
    const int ntok = min(kCombineTokens, sd.w - j0);
    if (ntok <= 0) continue;
    const int r = sd.y, r16 = (r + 15) & ~15;
    const int nparts = min(kTcShrinkParts, (d.proj[p].h_in + kTcK - 1) / kTcK);
    const float sa = d.scale ? __ldg(d.scale + sd.x) : 1.f;
    const float* part0 = t.vpart + (int64_t)p * t.vpart_proj;
    uint16_t* hbase = t.vhi[p];
    uint16_t* lbase = t.vlo[p];
    const int total = ntok * r16;
    for (int base = threadIdx.x; base < total; base += kCombineUnroll * kCombineThreads) {
      float acc[kCombineUnroll][kTcShrinkParts];
#pragma unroll
      for (int u = 0; u < kCombineUnroll; ++u) {
        const int idx = base + u * kCombineThreads;
        const int m = idx / r16, k = idx - m * r16;
        const bool live = idx < total && k < r;
#pragma unroll
        for (int o = 0; o < kTcShrinkParts; ++o)
          acc[u][o] = live && o < nparts ? part0[(int64_t)o * t.vpart_part + (int64_t)(j0 + m) * d.v_ld + k] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kCombineUnroll; ++u) {
        const int idx = base + u * kCombineThreads;
        if (idx < total) {
          const int m = idx / r16, k = idx - m * r16;
          float x = 0.f;
#pragma unroll
          for (int o = 0; o < kTcShrinkParts; ++o) x += acc[u][o];
          x *= sa;
          const int64_t j = j0 + m;
          const uint16_t hi = Elem<E>::from(x);
          hbase[j * t.v16_ld + k] = hi;
          lbase[j * t.v16_ld + k] = Elem<E>::from(x - Elem<E>::to(hi));
        }
      }
    }
  }
}

// ================================================================ tc_expand
// Work unit = (segment in work order, projection, column tile of <= kTcNe
// columns inside one page).  The adapter's B rows for the column tile are
// gathered once per unit (all rank rows, N-major) and reused by every 128-token
// tile of the segment.  Units of rank <= 128 alternate between the two halves
// of the B area, so the next unit's rows load while this one computes; a unit
// of larger rank takes the whole area.  Per token tile the producer loads the tile's v halves
// (2-D boxes, rows consecutive in sorted order) and its y rows (2-D boxes when
// the tile is a run of consecutive tokens, row gathers otherwise) into
// double-buffered stages, so the epilogue reads y from shared memory and its
// global stores are fire-and-forget.
constexpr int kTcNe = 128;                        // expand column tile
constexpr int kEAtoms = kTcNe / 64;               // 64-column swizzle atoms per tile
constexpr int kEKBlocks = kMaxRank / kTcK;        // B row blocks of 64 ranks
constexpr int kEBufs = 3;                         // y tiles and TMEM accumulators in flight
// warps: 0 y tiles and B rows, 1 MMAs, 2-5 epilogue, 6 v halves, 7 y stores
constexpr int kExpandTcThreads = kTcThreads + 64;
constexpr int kETmemCols = 512;                   // power of two >= kEBufs * kTcNe
static_assert(kEBufs * kTcNe <= kETmemCols, "accumulators must fit the TMEM allocation");
struct TcExpandSmem {
  uint8_t B[kEKBlocks][kEAtoms][kTcK * kRowBytes];   // <= 256 rank rows x 128 columns, N-major (64 KB)
  uint8_t Vhi[2][kTcM * kRowBytes];                  // 128 tokens x 64 ranks (16 KB)
  uint8_t Vlo[2][kTcM * kRowBytes];
  uint8_t Y[kEBufs][kEAtoms][kTcM * kRowBytes];      // 128 tokens x 128 columns (32 KB)
  uint64_t b_full[2], b_empty[2], v_full[2], v_empty[2];
  uint64_t y_full[kEBufs], y_empty[kEBufs], tfull[kEBufs], tempty[kEBufs], epi_done[kEBufs];
  uint32_t tmem_slot;
};

// Unit g of the expand list: segment position q (any segment; those with no
// tensor-core tile do nothing), projection and column tile
// (tc_eunit_raw / tc_eunit_done below).
struct TcEUnit {
  int p, start, len, r, a, c, o, ncols, ntm;  // ntm = 128-token tiles (0: skip)
};
// The loads of unit g's descriptor, kept apart from the arithmetic on them
// (tc_eunit_done), so that a warp can have the next unit's loads in flight
// while it works on this one.  g >= G: no unit (ntm 0), nothing loaded.
struct TcERaw {
  int p, c, o, ncols;
  int off0, off1;
  int4 sd;
};
__device__ __forceinline__ TcERaw tc_eunit_raw(const TcDev& t, int64_t g, int per_seg, int64_t G) {
  const ApplyDev& d = t.a;
  TcERaw w{};
  if (g >= G) return w;
  const int q = (int)(g / per_seg);
  int nt = (int)(g - (int64_t)q * per_seg);
  while (nt >= t.tc_ncol[w.p]) nt -= t.tc_ncol[w.p++];
  for (w.c = 0;; ++w.c) {  // column tile within one page chunk
    const int lenc = min(d.H, d.proj[w.p].h_out - w.c * d.H);
    const int n = (lenc + kTcNe - 1) / kTcNe;
    if (nt < n) {
      w.o = nt * kTcNe;
      w.ncols = min(kTcNe, lenc - w.o);
      break;
    }
    nt -= n;
  }
  w.off0 = __ldg(t.tc_off + q);
  w.off1 = __ldg(t.tc_off + q + 1);
  w.sd = __ldg(d.seg_desc + q);   // adapter, rank, start, end
  return w;
}
__device__ __forceinline__ TcEUnit tc_eunit_done(const TcERaw& w) {
  TcEUnit u;
  u.p = w.p;
  u.c = w.c;
  u.o = w.o;
  u.ncols = w.ncols;
  u.ntm = w.off1 - w.off0;
  u.start = w.sd.z;
  u.len = w.sd.w - w.sd.z;
  u.r = w.sd.y;
  u.a = w.sd.x;
  return u;
}

template <class E>
__global__ void __launch_bounds__(kExpandTcThreads, 1) tc_expand_kernel(const __grid_constant__ TcDev t) {
  extern __shared__ uint8_t smem_raw[];
  TcExpandSmem& sm = *reinterpret_cast<TcExpandSmem*>(smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const ApplyDev& d = t.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 1) tmem_alloc(&sm.tmem_slot, kETmemCols);
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.b_full[b], 1);
      mbar_init(&sm.b_empty[b], 1);
      mbar_init(&sm.v_full[b], 1);
      mbar_init(&sm.v_empty[b], 1);
    }
    for (int b = 0; b < kEBufs; ++b) {
      mbar_init(&sm.y_full[b], 1);
      mbar_init(&sm.y_empty[b], 1);   // epilogue warp 2 lane 0, after the four warps are done
      mbar_init(&sm.epi_done[b], 4);  // each epilogue warp, done with the y tile
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], 4);
    }
    mbar_fence_init();
  }
  pdl_wait();
  const int S = d.counts[kNumSegs];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = sm.tmem_slot;
  int per_seg = 0;
  for (int p = 0; p < d.nproj; ++p) per_seg += t.tc_ncol[p];
  const int64_t G = (int64_t)S * per_seg;
  constexpr bool bf16 = std::is_same<E, __nv_bfloat16>::value;
  bool ok = true;
  auto wait_lane0 = [&](uint64_t* bar, uint32_t parity) -> bool {
    bool got = true;
    if (lane == 0) got = mbar_wait(bar, parity);
    return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
  };

  if (warp == 0) {  // ------------------------------------------ producer
    uint32_t bu0 = 0, bu1 = 0, ny = 0;  // B uses per half, y tiles issued
    int bsel = 0;
    TcERaw rw = tc_eunit_raw(t, blockIdx.x, per_seg, G);   // one unit ahead
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const TcEUnit u = tc_eunit_done(rw);
      rw = tc_eunit_raw(t, g + gridDim.x, per_seg, G);
      if (u.ntm == 0) continue;
      const ProjDev& P = d.proj[u.p];
      const int r16 = (u.r + 15) & ~15;
      const int nkb = (r16 + kTcK - 1) / kTcK;
      const int natoms = (u.ncols + 63) >> 6;
      const int col0 = u.c * d.H + u.o;
      // B rows of this column tile, all rank blocks (rows >= r: row 0 again;
      // the matching v columns are zero), into half bsel of the B area, or
      // into the whole area for ranks above 128
      const bool whole = nkb > kEKBlocks / 2;
      const int hb = whole ? 0 : bsel;
      if (!wait_lane0(&sm.b_empty[hb], ((hb ? bu1 : bu0) & 1) ^ 1)) { ok = false; break; }
      if (hb) ++bu1; else ++bu0;
      if (whole) {
        if (!wait_lane0(&sm.b_empty[1], (bu1 & 1) ^ 1)) { ok = false; break; }
        ++bu1;
      } else {
        bsel ^= 1;
      }
      if (lane == 0) {
        mbar_expect_tx(&sm.b_full[hb], (uint32_t)(natoms * r16) * kRowBytes);
        if (whole) mbar_arrive(&sm.b_full[1]);
      }
      __syncwarp();
      const int kb0 = hb * (kEKBlocks / 2);   // first rank block of this half
      const int32_t* ptB = d.page_table + (int64_t)u.a * d.pt_stride + (int64_t)u.r * (P.rows_before + P.ppi) + u.c;
      for (int k4 = lane; 4 * k4 < r16; k4 += 32) {
        int pg[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = 4 * k4 + i;
          pg[i] = dbg_index(__ldg(ptB + (int64_t)(row < u.r ? row : 0) * P.ppo), d.num_pages, d.error);
        }
        const int kb = kb0 + (4 * k4) / kTcK, kr = (4 * k4) % kTcK;
        for (int nb = 0; nb < natoms; ++nb)
          tma_gather4(&sm.B[kb][nb][kr * kRowBytes], &t.pool_map, u.o + 64 * nb, pg[0], pg[1], pg[2], pg[3],
                      &sm.b_full[hb]);
      }
      for (int mt = 0; mt < u.ntm && ok; ++mt) {
        const int j0 = u.start + mt * kTcM;
        const int len = min(kTcM, u.start + u.len - j0);
        int tok[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = 4 * lane + i;
          tok[i] = dbg_index(__ldg(d.perm + j0 + (m < len ? m : 0)), d.T, d.error);
        }
        const int t_first = __shfl_sync(0xffffffffu, tok[0], 0);
        const bool run = dbg_index(__ldg(d.perm + j0 + len - 1), d.T, d.error) - t_first == len - 1;
        const int n16 = (len + 15) >> 4, nx4 = (len + 3) >> 2;
        // y tile
        const int yb = (int)(ny % kEBufs);
        if (!wait_lane0(&sm.y_empty[yb], ((ny / kEBufs) & 1) ^ 1)) { ok = false; break; }
        ++ny;
        const uint32_t ybytes = (uint32_t)natoms * (run ? (len == kTcM ? kTcM : 16 * n16) : 4 * nx4) * kRowBytes;
        if (lane == 0) mbar_expect_tx(&sm.y_full[yb], ybytes);
        __syncwarp();
        for (int nb = 0; nb < natoms; ++nb) {
          if (run && len == kTcM) {
            if (lane == 0) tma_load_2d(sm.Y[yb][nb], &t.y128_map[u.p], col0 + 64 * nb, t_first, &sm.y_full[yb]);
          } else if (run) {
            if (lane < n16)
              tma_load_2d(&sm.Y[yb][nb][16 * lane * kRowBytes], &t.y16_map[u.p], col0 + 64 * nb, t_first + 16 * lane,
                          &sm.y_full[yb]);
          } else if (lane < nx4) {
            tma_gather4(&sm.Y[yb][nb][4 * lane * kRowBytes], &t.y_map[u.p], col0 + 64 * nb, tok[0], tok[1], tok[2],
                        tok[3], &sm.y_full[yb]);
          }
        }
      }
    }
  } else if (warp == 6) {  // ------------------------------------ v halves
    // In the MMA warp's order: per unit, per token tile, per 64-rank block,
    // the tile's v hi and lo halves into one of the two v stages.  Apart from
    // the producer, so that they do not queue behind the y and B copies.
    uint32_t nv = 0;
    TcERaw rw = tc_eunit_raw(t, blockIdx.x, per_seg, G);   // one unit ahead
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const TcEUnit u = tc_eunit_done(rw);
      rw = tc_eunit_raw(t, g + gridDim.x, per_seg, G);
      if (u.ntm == 0) continue;
      const int nkb = (((u.r + 15) & ~15) + kTcK - 1) / kTcK;
      for (int mt = 0; mt < u.ntm && ok; ++mt) {
        const int j0 = u.start + mt * kTcM;
        for (int kb = 0; kb < nkb; ++kb) {
          const int vb = nv & 1;
          if (!wait_lane0(&sm.v_empty[vb], ((nv >> 1) & 1) ^ 1)) { ok = false; break; }
          ++nv;
          if (lane == 0) {
            mbar_expect_tx(&sm.v_full[vb], 2u * kTcM * kRowBytes);
            tma_load_2d(sm.Vhi[vb], &t.vhi_map[u.p], kb * kTcK, j0, &sm.v_full[vb]);
            tma_load_2d(sm.Vlo[vb], &t.vlo_map[u.p], kb * kTcK, j0, &sm.v_full[vb]);
          }
          __syncwarp();
        }
      }
    }
  } else if (warp == 1) {  // ----------------------------------- MMA issuer
    // The next unit's descriptor loads are in flight while this unit's MMAs
    // are issued (this warp is on the path from the copies to the epilogue).
    uint32_t bu0 = 0, bu1 = 0, nv = 0, nt = 0;
    int bsel = 0;
    TcERaw rw = tc_eunit_raw(t, blockIdx.x, per_seg, G);
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const TcEUnit u = tc_eunit_done(rw);
      rw = tc_eunit_raw(t, g + gridDim.x, per_seg, G);
      const int ntm = u.ntm;
      if (ntm == 0) continue;
      const int r = u.r;
      const int ncols = u.ncols;
      const int r16 = (r + 15) & ~15;
      const int nkb = (r16 + kTcK - 1) / kTcK;
      const uint32_t idesc = umma_idesc_f16(kTcM, (ncols + 15) & ~15, bf16, true);
      const bool whole = nkb > kEKBlocks / 2;
      const int hb = whole ? 0 : bsel;
      if (!wait_lane0(&sm.b_full[hb], (hb ? bu1 : bu0) & 1)) { ok = false; break; }
      if (hb) ++bu1; else ++bu0;
      if (whole) {
        if (!wait_lane0(&sm.b_full[1], bu1 & 1)) { ok = false; break; }
        ++bu1;
      } else {
        bsel ^= 1;
      }
      const int kb0 = hb * (kEKBlocks / 2);
      tc_fence_after();
      for (int mt = 0; mt < ntm && ok; ++mt) {
        const int ab = (int)(nt % kEBufs);
        if (!wait_lane0(&sm.tempty[ab], ((nt / kEBufs) & 1) ^ 1)) { ok = false; break; }
        ++nt;
        tc_fence_after();
        const uint32_t dtm = tmem + (uint32_t)(ab * kTcNe);
        for (int kb = 0; kb < nkb; ++kb) {
          const int vb = nv & 1;
          if (!wait_lane0(&sm.v_full[vb], (nv >> 1) & 1)) { ok = false; break; }
          ++nv;
          tc_fence_after();
          if (lane == 0) {
            const int nk = min(kTcK, r16 - kb * kTcK);
            const uint32_t ha = smem_addr(sm.Vhi[vb]), la = smem_addr(sm.Vlo[vb]);
            const uint32_t ba = smem_addr(sm.B[kb0 + kb][0]);
            for (int ks = 0; ks < nk / 16; ++ks) {
              // B is N-major: 64-column atoms kTcK rows apart, 8-row groups 1 KB apart
              const uint64_t bdesc = umma_desc_sw128(ba + ks * 16 * kRowBytes, kTcK * kRowBytes, 1024);
              umma_f16(dtm, umma_desc_sw128(ha + ks * 32, 16, 1024), bdesc, idesc, (kb | ks) ? 1u : 0u);
              umma_f16(dtm, umma_desc_sw128(la + ks * 32, 16, 1024), bdesc, idesc, 1u);
            }
            umma_commit(&sm.v_empty[vb]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) umma_commit(&sm.tfull[ab]);
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {  // B free once this unit's MMAs are done
        umma_commit(&sm.b_empty[hb]);
        if (whole) umma_commit(&sm.b_empty[1]);
      }
      __syncwarp();
    }
  } else if (warp < 6) {  // --------------------------------------- epilogue (warps 2-5)
    // Per token tile: 64 accumulator columns per TMEM round trip; the TMEM
    // buffer is released as soon as it has been read.  A tile of 128
    // consecutive tokens and 128 columns (the common prefill case) is written
    // back into its y tile in shared memory and stored by the TMA engine in
    // whole 128-byte rows; other tiles store their 16-byte pieces directly.
    const int quarter = warp & 3;
    const int m = 32 * quarter + lane;
    uint32_t nt = 0;
    TcERaw rw = tc_eunit_raw(t, blockIdx.x, per_seg, G);   // one unit ahead
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const TcEUnit u = tc_eunit_done(rw);
      rw = tc_eunit_raw(t, g + gridDim.x, per_seg, G);
      if (u.ntm == 0) continue;
      const ProjDev& P = d.proj[u.p];
      const int col0 = u.c * d.H + u.o;
      const int natoms = (u.ncols + 63) >> 6;
      for (int mt = 0; mt < u.ntm && ok; ++mt) {
        const int j0 = u.start + mt * kTcM;
        const int len = min(kTcM, u.start + u.len - j0);
        const int token = m < len ? dbg_index(__ldg(d.perm + j0 + m), d.T, d.error) : 0;
        const int t_first = dbg_index(__ldg(d.perm + j0), d.T, d.error);
        const bool tma_out = len == kTcM && u.ncols == kTcNe &&
                             dbg_index(__ldg(d.perm + j0 + kTcM - 1), d.T, d.error) - t_first == kTcM - 1;
        const int ab = (int)(nt % kEBufs);
        const uint32_t ph = (nt / kEBufs) & 1;
        if (!wait_lane0(&sm.tfull[ab], ph) || !wait_lane0(&sm.y_full[ab], ph)) {
          ok = false;
          break;
        }
        ++nt;
        tc_fence_after();
        uint16_t* yrow = static_cast<uint16_t*>(P.y) + (int64_t)token * P.ldy + col0;
        for (int at = 0; at < natoms; ++at) {
          uint32_t r0[32], r1[32];
          const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(ab * kTcNe + 64 * at);
          tmem_ld32_nowait(ta, r0);
          tmem_ld32_nowait(ta + 32, r1);
          tmem_wait_ld(r0);
          tmem_wait_ld(r1);
          if (at == natoms - 1) {  // this warp is done with the TMEM buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tempty[ab]);
          }
          if (m < len) {
            uint8_t* ytile = sm.Y[ab][at] + m * kRowBytes;
            const int nch = min(8, (u.ncols - 64 * at) >> 3);   // 8-column chunks in this atom
            // every chunk of the row first: the stores below could otherwise
            // hold each load back (the compiler cannot tell the chunks apart)
            uint4 yin[8];
#pragma unroll
            for (int h = 0; h < 8; ++h)
              if (h < nch) yin[h] = *reinterpret_cast<const uint4*>(ytile + ((h ^ (m & 7)) << 4));
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              if (h < nch) {
                uint8_t* py = ytile + ((h ^ (m & 7)) << 4);   // swizzled 16-byte chunk
                uint4 yv = yin[h];
                uint32_t w[4];
                memcpy(w, &yv, 16);
#pragma unroll
                for (int i = 0; i < 4; ++i) {   // pairs of columns: one unpack, two FMAs, one packing rounding
                  const uint32_t b0 = h < 4 ? r0[8 * h + 2 * i] : r1[8 * (h - 4) + 2 * i];
                  const uint32_t b1 = h < 4 ? r0[8 * h + 2 * i + 1] : r1[8 * (h - 4) + 2 * i + 1];
                  const float2 yy = Elem<E>::to2(w[i]);
                  w[i] = Elem<E>::from2(yy.x + d.s * __uint_as_float(b0), yy.y + d.s * __uint_as_float(b1));
                }
                memcpy(&yv, w, 16);
                if (tma_out) *reinterpret_cast<uint4*>(py) = yv;
                else *reinterpret_cast<uint4*>(yrow + 64 * at + 8 * h) = yv;
              }
            }
          }
        }
        if (tma_out) fence_async_shared();   // the tile's new values, for the TMA engine
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.epi_done[ab]);
      }
    }
  } else {  // ------------------------------------------------------------ y stores
    // Once the four epilogue warps are done with a y tile: store it (TMA,
    // whole 128-byte rows) and, when the stores have read it, hand the
    // buffer back to the producer; a tile stored piecewise by the epilogue
    // goes back at once.  Apart from the epilogue warps, so that they start
    // the next tile while the stores read this one.
    uint32_t nt = 0;
    TcERaw rw = tc_eunit_raw(t, blockIdx.x, per_seg, G);   // one unit ahead
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const TcEUnit u = tc_eunit_done(rw);
      rw = tc_eunit_raw(t, g + gridDim.x, per_seg, G);
      if (u.ntm == 0) continue;
      const int col0 = u.c * d.H + u.o;
      for (int mt = 0; mt < u.ntm && ok; ++mt) {
        const int j0 = u.start + mt * kTcM;
        const int len = min(kTcM, u.start + u.len - j0);
        const int t_first = dbg_index(__ldg(d.perm + j0), d.T, d.error);
        const bool tma_out = len == kTcM && u.ncols == kTcNe &&
                             dbg_index(__ldg(d.perm + j0 + kTcM - 1), d.T, d.error) - t_first == kTcM - 1;
        const int ab = (int)(nt % kEBufs);
        const uint32_t ph = (nt / kEBufs) & 1;
        ++nt;
        if (!wait_lane0(&sm.epi_done[ab], ph)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (tma_out) {
#pragma unroll
            for (int at = 0; at < kEAtoms; ++at)
              tma_store_2d(&t.y128_map[u.p], col0 + 64 * at, t_first, sm.Y[ab][at]);
            bulk_commit();
            bulk_wait_read();   // the y tile may be refilled once the stores have read it
          }
          mbar_arrive(&sm.y_empty[ab]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // stores complete
  }
  if (!ok && lane == 0) report_err(d.error, kErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kETmemCols);
  }
}

template <typename Kern>
cudaError_t launch_pdl_tc(Kern kernel, int grid, int threads, size_t smem, cudaStream_t st, const TcDev& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

constexpr size_t kShrinkTcSmem = sizeof(TcShrinkSmem) + 1024;
constexpr size_t kExpandTcSmem = sizeof(TcExpandSmem) + 1024;

}  // namespace

cudaError_t prepare_tc_kernels() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(tc_shrink_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kShrinkTcSmem)))
    return e;
  if ((e = cudaFuncSetAttribute(tc_shrink_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kShrinkTcSmem)))
    return e;
  if ((e = cudaFuncSetAttribute(tc_expand_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kExpandTcSmem)))
    return e;
  return cudaFuncSetAttribute(tc_expand_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kExpandTcSmem);
}

cudaError_t launch_tc_shrink(const TcDev& a, int dtype, int grid, cudaStream_t st) {
  cudaError_t e = dtype == 0 ? launch_pdl_tc(tc_shrink_kernel<__half>, grid, kShrinkTcThreads, kShrinkTcSmem, st, a)
                             : launch_pdl_tc(tc_shrink_kernel<__nv_bfloat16>, grid, kShrinkTcThreads, kShrinkTcSmem, st, a);
  if (e != cudaSuccess) return e;
  // the K parts' sums: eight small blocks per SM
  return dtype == 0 ? launch_pdl_tc(tc_combine_kernel<__half>, 8 * grid, kCombineThreads, 0, st, a)
                    : launch_pdl_tc(tc_combine_kernel<__nv_bfloat16>, 8 * grid, kCombineThreads, 0, st, a);
}

cudaError_t launch_tc_expand(const TcDev& a, int dtype, int grid, cudaStream_t st) {
  if (dtype == 0) return launch_pdl_tc(tc_expand_kernel<__half>, grid, kExpandTcThreads, kExpandTcSmem, st, a);
  return launch_pdl_tc(tc_expand_kernel<__nv_bfloat16>, grid, kExpandTcThreads, kExpandTcSmem, st, a);
}

int32_t tc_col_tiles(int32_t h_out, int32_t H) {
  int32_t n = 0;
  for (int32_t c = 0; c * H < h_out; ++c) {
    const int32_t len = (h_out - c * H) < H ? (h_out - c * H) : H;
    n += (len + kTcNe - 1) / kTcNe;
  }
  return n;
}

}  // namespace slora
