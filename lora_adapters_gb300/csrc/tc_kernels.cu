// Tensor-core (tcgen05) kernels of the LoRA delta for long segments (prefill).
//
// A segment of many tokens on one adapter turns the per-token products into
// dense contractions ("S-LoRA: Serving Thousands of Concurrent LoRA
// Adapters": heterogeneous batching runs custom kernels directly on the
// non-contiguous pool; the pages give no kernel internals).  Per work unit a
// 128-token tile of one segment is multiplied on the 5th-generation tensor
// cores, fp16/bf16 operands from shared memory, fp32 accumulators in TMEM:
//
//   tc_shrink:  V[128 x r] = X[128 x H_in] . A^T   (A rows = pages, K-major)
//   tc_expand:  Y[128 x 256] += s * (V_hi + V_lo)[128 x r] . B[r x 256]
//
// Operands are gathered by the TMA engine straight from where they live:
// token rows of x by `tile::gather4` through the segment's sorted token list,
// adapter rows by `gather4` over the page pool viewed as a [pages x H] matrix,
// v rows (consecutive in sorted order) by 2-D tiles; all land in shared
// memory in the 128-byte-swizzled layout the MMA reads.  V is carried as two
// 16-bit halves, V_hi = round(v) and V_lo = round(v - V_hi), so the expand
// multiplies with ~fp32 accuracy on 16-bit tensor cores.
//
// Each kernel is persistent (one CTA per SM) and warp-specialised: warp 0
// issues copies into a ring of shared-memory stages, warp 1 owns TMEM and
// issues the MMAs (one thread), warps 2-5 drain a TMEM accumulator (two of
// them, so the epilogue of one unit overlaps the MMAs of the next) and write
// v or y.  Every wait is bounded (SLORA_ERR_TIMEOUT on give-up).
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

struct TcUnit {
  int p, j0, len, r, a, seg;
};

// Tile `tile` of the long-segment list: segment (in work order) and row range.
__device__ __forceinline__ TcUnit tc_tile(const TcDev& t, const int32_t* s_off, bool in_smem, int S, int tile,
                                          int p) {
  const ApplyDev& d = t.a;
  TcUnit u;
  const int q = find_pos_tc(s_off, t.tc_off, in_smem, S, tile);
  const int mt = tile - (in_smem ? s_off[q] : __ldg(t.tc_off + q));
  const int s = __ldg(d.seg_order + q);
  const int start = __ldg(d.seg_start + s), end = __ldg(d.seg_start + s + 1);
  u.p = p;
  u.j0 = start + mt * kTcM;
  u.len = min(kTcM, end - u.j0);
  u.r = __ldg(d.seg_rank + s);
  u.a = __ldg(d.seg_adapter + s);
  u.seg = s;
  return u;
}

template <class T>
struct Elem;
template <>
struct Elem<__half> {
  static __device__ __forceinline__ uint16_t from(float f) { return __half_as_ushort(__float2half_rn(f)); }
  static __device__ __forceinline__ float to(uint16_t u) { return __half2float(__ushort_as_half(u)); }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ uint16_t from(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
  static __device__ __forceinline__ float to(uint16_t u) { return __bfloat162float(__ushort_as_bfloat16(u)); }
};

// ================================================================ tc_shrink
// Warps: 0 loads x tiles (TMA), 1 issues the MMAs, 2-5 drain TMEM, 6-9 copy
// the adapter's rows.  Adapter rows go through the load/store unit rather
// than the TMA engine: a K block needs r rows of 128 bytes, and a TMA op per
// four rows made the copy engine's op rate the limit.  Each loader thread
// copies one 16-byte chunk column of every 16th row with cp.async, straight
// to its 128-byte-swizzled place, then (once its copies have landed) fences
// them for the tensor cores' async proxy and arrives on the stage.
constexpr int kShrinkTcStages = 4;
constexpr int kShrinkLoaderWarps = 4;
constexpr int kShrinkLoaders = kShrinkLoaderWarps * 32;
constexpr int kShrinkTcThreads = kTcThreads + kShrinkLoaders;
constexpr int kRowsPerLoader = kMaxRank * (kRowBytes / 16) / kShrinkLoaders;   // rows one loader thread covers
struct TcShrinkSmem {
  uint8_t X[kShrinkTcStages][kTcM * kRowBytes];     // 128 token rows x 64 K, swizzled (16 KB)
  uint8_t B[kShrinkTcStages][kMaxRank * kRowBytes]; // <= 256 adapter rows x 64 K (32 KB)
  uint64_t full[kShrinkTcStages], empty[kShrinkTcStages], tfull[2], tempty[2];
  uint32_t tmem_slot;
  int32_t off[kSegSmem];
};

__device__ __forceinline__ void cp16_shared(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Shrink unit g: the K range of (tile, projection) is split in two halves
// (units 2u and 2u+1), so that the short list of 128-token tiles spreads over
// twice as many units.  A projection with fewer than two K blocks is not
// split (its second half is skipped).
struct ShUnit {
  int tile, p, kb_lo, kb_hi;
  bool split, skip;
  int half;
};
__device__ __forceinline__ ShUnit sh_unit(const ApplyDev& d, int64_t g) {
  ShUnit s;
  s.half = (int)(g & 1);
  const int64_t tp = g >> 1;
  s.tile = (int)(tp / d.nproj);
  s.p = (int)(tp - (int64_t)s.tile * d.nproj);
  const int nkb = (d.proj[s.p].h_in + kTcK - 1) / kTcK;
  s.split = nkb >= 2;
  s.skip = !s.split && s.half == 1;
  const int mid = nkb / 2;
  s.kb_lo = s.split && s.half ? mid : 0;
  s.kb_hi = s.split && !s.half ? mid : nkb;
  return s;
}

template <class E>
__global__ void __launch_bounds__(kShrinkTcThreads, 1) tc_shrink_kernel(const __grid_constant__ TcDev t) {
  extern __shared__ uint8_t smem_raw[];
  TcShrinkSmem& sm = *reinterpret_cast<TcShrinkSmem*>(smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const ApplyDev& d = t.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 1) tmem_alloc(&sm.tmem_slot, 2 * kTcN);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kShrinkTcStages; ++s) {
      mbar_init(&sm.full[s], 1 + kShrinkLoaders);   // x bytes (warp 0) + every loader thread
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
  const bool off_smem = S + 1 <= kSegSmem;
  if (off_smem)
    for (int i = threadIdx.x; i <= S; i += blockDim.x) sm.off[i] = t.tc_off[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = sm.tmem_slot;
  const int64_t G = (int64_t)tiles * d.nproj * 2;   // K halves
  constexpr bool bf16 = std::is_same<E, __nv_bfloat16>::value;
  bool ok = true;

  if (warp == 0) {  // ------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const ShUnit su = sh_unit(d, g);
      if (su.skip) continue;
      const TcUnit u = tc_tile(t, sm.off, off_smem, S, su.tile, su.p);
      const int r16 = (u.r + 15) & ~15;
      const int nx4 = (u.len + 3) >> 2;  // gather4 ops for the token rows
      const int nb4 = r16 >> 2;          // gather4 ops for the adapter rows
      int tok[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = 4 * lane + i;
        tok[i] = __ldg(d.perm + u.j0 + (m < u.len ? m : 0));
      }
      // Tokens of a segment are in increasing order, so the tile is one run
      // of consecutive rows of x exactly when its last token is first + len - 1
      // (prefill requests): then 2-D boxes replace the row gathers.
      const int t_first = __shfl_sync(0xffffffffu, tok[0], 0);
      const int t_last = __ldg(d.perm + u.j0 + u.len - 1);
      const bool run = t_last - t_first == u.len - 1;
      const int n16 = (u.len + 15) >> 4;  // 16-row boxes of a partial run tile
      const uint32_t x_bytes = run ? (u.len == kTcM ? (uint32_t)kTcM * kRowBytes : (uint32_t)n16 * 16 * kRowBytes)
                                   : (uint32_t)(4 * nx4) * kRowBytes;
      (void)nb4;
      for (int kb = su.kb_lo; kb < su.kb_hi; ++kb) {
        const int k0 = kb * kTcK;
        bool got = true;
        if (lane == 0) got = mbar_wait(&sm.empty[stage], phase ^ 1);
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_expect_tx(&sm.full[stage], x_bytes);
        __syncwarp();
        if (!run) {
          if (lane < nx4)
            tma_gather4(&sm.X[stage][4 * lane * kRowBytes], &t.x_map[u.p], k0, tok[0], tok[1], tok[2], tok[3],
                        &sm.full[stage]);
        } else if (u.len == kTcM) {
          if (lane == 0) tma_load_2d(sm.X[stage], &t.x128_map[u.p], k0, t_first, &sm.full[stage]);
        } else if (lane < n16) {
          tma_load_2d(&sm.X[stage][16 * lane * kRowBytes], &t.x16_map[u.p], k0, t_first + 16 * lane, &sm.full[stage]);
        }
        if (++stage == kShrinkTcStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {  // ----------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0;
    int n = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const ShUnit su = sh_unit(d, g);
      if (su.skip) continue;
      const int tile = su.tile, p = su.p;
      int r = 0;
      if (lane == 0) r = tc_tile(t, sm.off, off_smem, S, tile, p).r;
      r = __shfl_sync(0xffffffffu, r, 0);
      const int r16 = (r + 15) & ~15;
      const int ab = n & 1;
      bool got = true;
      if (lane == 0) got = mbar_wait(&sm.tempty[ab], ((n >> 1) & 1) ^ 1);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t idesc = umma_idesc_f16(kTcM, r16, bf16, false);
      const uint32_t dtm = tmem + (uint32_t)(ab * kTcN);
      for (int kb = su.kb_lo; kb < su.kb_hi; ++kb) {
        if (lane == 0) got = mbar_wait(&sm.full[stage], phase);
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t xa = smem_addr(sm.X[stage]), ba = smem_addr(sm.B[stage]);
#pragma unroll
          for (int ks = 0; ks < kTcK / 16; ++ks)
            umma_f16(dtm, umma_desc_sw128(xa + ks * 32, 16, 1024), umma_desc_sw128(ba + ks * 32, 16, 1024), idesc,
                     (kb != su.kb_lo || ks) ? 1u : 0u);
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
  } else if (warp >= 6) {  // ------------------------------------ adapter-row loaders
    const int lt = threadIdx.x - 6 * 32;    // 0 .. kShrinkLoaders - 1
    const int ch = lt & 7;                  // 16-byte chunk column of the 128-byte row
    const int row0 = lt >> 3;               // rows row0, row0 + 16, ...
    uint32_t stage = 0, phase = 0;
    int pending = -1;                       // stage whose copies are committed, not yet announced
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const ShUnit su = sh_unit(d, g);
      if (su.skip) continue;
      const TcUnit u = tc_tile(t, sm.off, off_smem, S, su.tile, su.p);
      const ProjDev& P = d.proj[u.p];
      const int32_t* pt = d.page_table + (int64_t)u.a * d.pt_stride + (int64_t)u.r * P.rows_before;
      const int nrow = (u.r - row0 + 15) >> 4;   // my rows below r (rows past r are never read back)
      int chunk = -1;
      int pg[kRowsPerLoader];
      for (int kb = su.kb_lo; kb < su.kb_hi; ++kb) {
        const int k0 = kb * kTcK, c = k0 / d.H, o = k0 - c * d.H;
        if (c != chunk) {  // pages of my rows for this page chunk
          chunk = c;
#pragma unroll
          for (int j = 0; j < kRowsPerLoader; ++j)
            pg[j] = j < nrow ? __ldg(pt + (int64_t)(row0 + 16 * j) * P.ppi + c) : 0;
        }
        if (!mbar_wait(&sm.empty[stage], phase ^ 1)) {
          ok = false;
          break;
        }
        const uint32_t base = smem_addr(sm.B[stage]);
#pragma unroll
        for (int j = 0; j < kRowsPerLoader; ++j) {
          if (j < nrow) {
            const int row = row0 + 16 * j;
            cp16_shared(base + row * kRowBytes + ((ch ^ (row & 7)) << 4),
                        d.pool + (int64_t)pg[j] * d.H + o + ch * 8);
          }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (pending >= 0) {
          // the previous stage's copies have landed: make them visible to the
          // tensor cores' async proxy, then announce them
          asm volatile("cp.async.wait_group 1;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&sm.full[pending]);
        }
        pending = (int)stage;
        if (++stage == kShrinkTcStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (pending >= 0 && ok) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&sm.full[pending]);
    }
  } else {  // ------------------------------------------------- epilogue (warps 2-5)
    // A split unit writes its partial sums (fp32) to its half's scratch
    // rows; the half that finishes second (per warp: per 32 rows) adds the
    // other half's rows to its own accumulator and writes s_a v and its
    // 16-bit halves.  Neither half waits for the other.
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int m = 32 * quarter + lane;
    int n = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const ShUnit su = sh_unit(d, g);
      if (su.skip) continue;
      const TcUnit u = tc_tile(t, sm.off, off_smem, S, su.tile, su.p);
      const int r16 = (u.r + 15) & ~15;
      const int ab = n & 1;
      bool got = true;
      if (lane == 0) got = mbar_wait(&sm.tfull[ab], (n >> 1) & 1);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      ++n;
      tc_fence_after();
      const int j = u.j0 + m;
      const uint32_t tacc = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(ab * kTcN);
      bool finish = true;            // this warp writes the final v rows
      const float* other = nullptr;  // the other half's partial row
      if (su.split) {
        float* mine = t.vpart + (int64_t)su.half * t.vpart_half + (int64_t)u.p * t.vpart_proj + (int64_t)j * d.v_ld;
        for (int c00 = 0; c00 < r16; c00 += 32) {
          uint32_t raw[32];
          tmem_ld32_nowait(tacc + (uint32_t)c00, raw);
          tmem_wait_ld(raw);
          if (m < u.len) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              if (c00 + i < u.r)
                *reinterpret_cast<float4*>(mine + c00 + i) =
                    make_float4(__uint_as_float(raw[i]), __uint_as_float(raw[i + 1]), __uint_as_float(raw[i + 2]),
                                __uint_as_float(raw[i + 3]));
          }
        }
        __threadfence();   // my partial rows, before the count says they are there
        __syncwarp();
        int old = 0;
        int32_t* cnt = t.combine + ((int64_t)su.tile * d.nproj + u.p) * 4 + quarter;
        if (lane == 0) old = atomicAdd(cnt, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        finish = old == 1;
        if (finish) {
          __threadfence();   // the other half's partial rows are visible now
          other = t.vpart + (int64_t)(1 - su.half) * t.vpart_half + (int64_t)u.p * t.vpart_proj + (int64_t)j * d.v_ld;
          if (lane == 0) *cnt = 0;   // both halves are in: ready for the next call
        }
      }
      if (finish) {
        const float sa = d.scale ? __ldg(d.scale + u.a) : 1.f;   // the adapter's scale, applied to v
        float* vrow = d.proj[u.p].v + (int64_t)j * d.v_ld;
        uint16_t* hrow = t.vhi[u.p] + (int64_t)j * t.v16_ld;
        uint16_t* lrow = t.vlo[u.p] + (int64_t)j * t.v16_ld;
        // 32 accumulator columns per TMEM round trip
        for (int c00 = 0; c00 < r16; c00 += 32) {
          uint32_t raw[32];
          tmem_ld32_nowait(tacc + (uint32_t)c00, raw);
          tmem_wait_ld(raw);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int c0 = c00 + 16 * hh;
            if (m < u.len && c0 < r16) {
              float v[16];
              uint16_t hi[16], lo[16];
              if (other) {
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                  const float4 o4 = c0 + i < u.r ? *reinterpret_cast<const float4*>(other + c0 + i)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                  v[i] = o4.x;
                  v[i + 1] = o4.y;
                  v[i + 2] = o4.z;
                  v[i + 3] = o4.w;
                }
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float x = c0 + i < u.r ? sa * (__uint_as_float(raw[16 * hh + i]) + v[i]) : 0.f;
                v[i] = x;
                hi[i] = Elem<E>::from(x);
                lo[i] = Elem<E>::from(x - Elem<E>::to(hi[i]));
              }
              // fp32 v: 16-byte stores up to the row's last multiple of 4 columns
              // (the v row stride is a multiple of 4 floats, past r only padding)
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                if (c0 + i < u.r)
                  *reinterpret_cast<float4*>(vrow + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
              uint4 h0, h1, l0, l1;
              memcpy(&h0, hi, 16);
              memcpy(&h1, hi + 8, 16);
              memcpy(&l0, lo, 16);
              memcpy(&l1, lo + 8, 16);
              *reinterpret_cast<uint4*>(hrow + c0) = h0;
              *reinterpret_cast<uint4*>(hrow + c0 + 8) = h1;
              *reinterpret_cast<uint4*>(lrow + c0) = l0;
              *reinterpret_cast<uint4*>(lrow + c0 + 8) = l1;
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
    tmem_dealloc(tmem, 2 * kTcN);
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
// tensor-core tile do nothing), projection and column tile.
struct TcEUnit {
  int p, start, len, r, a, c, o, ncols, ntm;  // ntm = 128-token tiles (0: skip)
};
__device__ __forceinline__ TcEUnit tc_eunit(const TcDev& t, int64_t g, int per_seg) {
  const ApplyDev& d = t.a;
  TcEUnit u;
  const int q = (int)(g / per_seg);
  int nt = (int)(g - (int64_t)q * per_seg);
  u.p = 0;
  while (nt >= t.tc_ncol[u.p]) nt -= t.tc_ncol[u.p++];
  u.ntm = __ldg(t.tc_off + q + 1) - __ldg(t.tc_off + q);
  const int s = __ldg(d.seg_order + q);
  u.start = __ldg(d.seg_start + s);
  u.len = __ldg(d.seg_start + s + 1) - u.start;
  u.r = __ldg(d.seg_rank + s);
  u.a = __ldg(d.seg_adapter + s);
  for (u.c = 0;; ++u.c) {  // column tile within one page chunk
    const int lenc = min(d.H, d.proj[u.p].h_out - u.c * d.H);
    const int n = (lenc + kTcNe - 1) / kTcNe;
    if (nt < n) {
      u.o = nt * kTcNe;
      u.ncols = min(kTcNe, lenc - u.o);
      break;
    }
    nt -= n;
  }
  return u;
}

template <class E>
__global__ void __launch_bounds__(kTcThreads, 1) tc_expand_kernel(const __grid_constant__ TcDev t) {
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
    uint32_t bu0 = 0, bu1 = 0, nv = 0, ny = 0;  // B uses per half, v stages, y tiles issued
    int bsel = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const TcEUnit u = tc_eunit(t, g, per_seg);
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
          pg[i] = __ldg(ptB + (int64_t)(row < u.r ? row : 0) * P.ppo);
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
          tok[i] = __ldg(d.perm + j0 + (m < len ? m : 0));
        }
        const int t_first = __shfl_sync(0xffffffffu, tok[0], 0);
        const bool run = __ldg(d.perm + j0 + len - 1) - t_first == len - 1;
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
        // v halves, one 64-rank block per stage
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
    uint32_t bu0 = 0, bu1 = 0, nv = 0, nt = 0;
    int bsel = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      TcEUnit u;
      if (lane == 0) u = tc_eunit(t, g, per_seg);
      const int ntm = __shfl_sync(0xffffffffu, lane == 0 ? u.ntm : 0, 0);
      if (ntm == 0) continue;
      const int r = __shfl_sync(0xffffffffu, lane == 0 ? u.r : 0, 0);
      const int ncols = __shfl_sync(0xffffffffu, lane == 0 ? u.ncols : 0, 0);
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
  } else {  // ------------------------------------------------- epilogue (warps 2-5)
    // Per token tile: 64 accumulator columns per TMEM round trip; the TMEM
    // buffer is released as soon as it has been read.  A tile of 128
    // consecutive tokens and 128 columns (the common prefill case) is written
    // back into its y tile in shared memory and stored by the TMA engine in
    // whole 128-byte rows; other tiles store their 16-byte pieces directly.
    const int quarter = warp & 3;
    const int m = 32 * quarter + lane;
    uint32_t nt = 0;
    for (int64_t g = blockIdx.x; g < G && ok; g += gridDim.x) {
      const TcEUnit u = tc_eunit(t, g, per_seg);
      if (u.ntm == 0) continue;
      const ProjDev& P = d.proj[u.p];
      const int col0 = u.c * d.H + u.o;
      const int natoms = (u.ncols + 63) >> 6;
      for (int mt = 0; mt < u.ntm && ok; ++mt) {
        const int j0 = u.start + mt * kTcM;
        const int len = min(kTcM, u.start + u.len - j0);
        const int token = m < len ? __ldg(d.perm + j0 + m) : 0;
        const int t_first = __ldg(d.perm + j0);
        const bool tma_out =
            len == kTcM && u.ncols == kTcNe && __ldg(d.perm + j0 + kTcM - 1) - t_first == kTcM - 1;
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
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              if (h < nch) {
                uint8_t* py = ytile + ((h ^ (m & 7)) << 4);   // swizzled 16-byte chunk
                uint4 yv = *reinterpret_cast<const uint4*>(py);
                uint16_t e[8];
                memcpy(e, &yv, 16);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const uint32_t bits = h < 4 ? r0[8 * h + i] : r1[8 * (h - 4) + i];
                  e[i] = Elem<E>::from(Elem<E>::to(e[i]) + d.s * __uint_as_float(bits));
                }
                memcpy(&yv, e, 16);
                if (tma_out) *reinterpret_cast<uint4*>(py) = yv;
                else *reinterpret_cast<uint4*>(yrow + 64 * at + 8 * h) = yv;
              }
            }
          }
        }
        if (tma_out) fence_async_shared();   // the tile's new values, for the TMA engine
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.epi_done[ab]);
        if (warp == 2 && lane == 0) {
          // once the four warps are done with the y tile: store it (TMA) or
          // just hand it back to the producer
          if (!mbar_wait(&sm.epi_done[ab], ph)) {
            ok = false;
          } else {
            if (tma_out) {
#pragma unroll
              for (int at = 0; at < kEAtoms; ++at)
                tma_store_2d(&t.y128_map[u.p], col0 + 64 * at, t_first, sm.Y[ab][at]);
              bulk_commit();
              bulk_wait_read();   // the y tile may be refilled once the stores have read it
            }
            mbar_arrive(&sm.y_empty[ab]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
    if (warp == 2 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // stores complete
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
  if (dtype == 0) return launch_pdl_tc(tc_shrink_kernel<__half>, grid, kShrinkTcThreads, kShrinkTcSmem, st, a);
  return launch_pdl_tc(tc_shrink_kernel<__nv_bfloat16>, grid, kShrinkTcThreads, kShrinkTcSmem, st, a);
}

cudaError_t launch_tc_expand(const TcDev& a, int dtype, int grid, cudaStream_t st) {
  if (dtype == 0) return launch_pdl_tc(tc_expand_kernel<__half>, grid, kTcThreads, kExpandTcSmem, st, a);
  return launch_pdl_tc(tc_expand_kernel<__nv_bfloat16>, grid, kTcThreads, kExpandTcSmem, st, a);
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
