// slora_lora_apply_noalloc: the LoRA delta for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they need the LoRA
// delta: a serving runtime that hands all GPU memory to its own arena (the
// unified page pool, the KV cache, activations) and forbids any further
// allocation, or code that must not change the device memory footprint while
// it serves requests.  The pool-based entry points allocate their scratch when
// the pool is created; this entry point needs no pool at all.  The caller
// passes the page pool, page table, ranks, token assignments, x and y as
// device pointers it already owns, and the scratch this path needs (the token
// grouping and the fp32 shrink result v) lives in one file-scope __device__
// array below, which every GPU that loads this library holds until the
// process exits.
//
// The paper has no counterpart of this entry point: it only changes where the
// scratch memory comes from.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/slora.h"
#include "internal.h"

using namespace slora;

namespace {

// Limits of the static scratch (see SLORA_NOALLOC_* in slora.h).
constexpr int kNaMaxTokens = 2048;
constexpr int kNaMaxSegs = kNaMaxTokens;
constexpr int kNaMaxAdapters = kMaxAdapters;
constexpr size_t kNaIntsSeg =
    4 * (size_t)(kNaMaxSegs + 1) + kNumCounts + kNaMaxTokens + 10 * (size_t)(kNaMaxSegs + 1) + 1 + kGridSyncInts;
constexpr size_t kNaIntsRank = kNaMaxAdapters;
constexpr size_t kNaIntBytes = ((kNaIntsSeg + kNaIntsRank) * sizeof(int32_t) + 255) / 256 * 256;
constexpr size_t kNaVFloats = (size_t)kNaMaxTokens * kMaxRank;
constexpr size_t kNaBytes = kNaIntBytes + kNaVFloats * sizeof(float);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_dev[kMaxDevices] = {};   // device address of g_noalloc_scratch per device
int g_grid[kMaxDevices] = {};

// Failures are reported through slora_last_error_string(), like every call.
int na_fail(int code, const char* msg, cudaError_t e = cudaSuccess) {
  char buf[384];
  if (e != cudaSuccess) snprintf(buf, sizeof buf, "%s: %s", msg, cudaGetErrorString(e));
  else snprintf(buf, sizeof buf, "%s", msg);
  set_last_error(buf);
  return code;
}

// Copy of the caller's ranks with every value outside [1, rmax] set to 0
// (treated as "not resident").  rmax = min(SLORA_MAX_RANK, pt_stride /
// entries per unit of rank): no rank can index past the rows of the static v
// buffer, nor past its adapter's own stretch of the page table.
__global__ void sanitize_ranks_kernel(const int32_t* in, int32_t* out, int n, int32_t rmax) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int32_t r = in[i];
    out[i] = (r >= 1 && r <= rmax) ? r : 0;
  }
}

// Once per device, with that device current: the device address of the
// scratch array (in host code its name is only a host-side stand-in) and the
// persistent grid sizes.
int setup_device(int dev, unsigned char** base) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_dev[dev]) {
    *base = g_scratch_dev[dev];
    return SLORA_OK;
  }
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "cudaGetSymbolAddress(scratch)", e);
  e = prepare_kernels(dev);
  if (e != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "kernel attribute set-up", e);
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "cudaDeviceGetAttribute", e);
  g_grid[dev] = sms;   // one persistent CTA per SM
  g_scratch_dev[dev] = static_cast<unsigned char*>(ptr);
  *base = g_scratch_dev[dev];
  return SLORA_OK;
}

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" int slora_lora_apply_noalloc(const void* d_pool, int32_t page_elems, int32_t dtype,
                                        const int32_t* d_page_table, int64_t pt_stride,
                                        const int32_t* d_rank, int32_t max_adapters, int32_t num_proj,
                                        const int32_t* proj_in, const int32_t* proj_out, int32_t proj,
                                        const int32_t* d_token_adapter, int32_t T, const void* d_x,
                                        int64_t ldx, void* d_y, int64_t ldy, float s, void* stream,
                                        int32_t* status) {
  if (!d_pool || !d_page_table || !d_rank || !proj_in || !proj_out)
    return na_fail(SLORA_ERR_INVALID, "NULL pool, page table, ranks or projection dims");
  if (page_elems <= 0 || page_elems % 8 || page_elems > 65536)
    return na_fail(SLORA_ERR_INVALID, "page_elems must be a positive multiple of 8, <= 65536");
  if (dtype != SLORA_F16 && dtype != SLORA_BF16) return na_fail(SLORA_ERR_INVALID, "dtype");
  if (max_adapters <= 0 || max_adapters > kNaMaxAdapters)
    return na_fail(SLORA_ERR_INVALID, "max_adapters out of [1, SLORA_MAX_ADAPTERS]");
  if (num_proj <= 0 || num_proj > kMaxPoolProj || proj < 0 || proj >= num_proj)
    return na_fail(SLORA_ERR_INVALID, "projection index or count out of range");
  if (T < 0 || T > kNaMaxTokens)
    return na_fail(SLORA_ERR_INVALID, "T exceeds SLORA_NOALLOC_MAX_TOKENS (the static scratch holds 2048 tokens)");
  int64_t before = 0, per_rank = 0;
  for (int q = 0; q < num_proj; ++q) {
    if (proj_in[q] <= 0 || proj_out[q] <= 0 || proj_in[q] % 8 || proj_out[q] % 8)
      return na_fail(SLORA_ERR_INVALID, "projection dims must be positive multiples of 8");
    if (q < proj) before += ceil_div64(proj_in[q], page_elems) + ceil_div64(proj_out[q], page_elems);
    per_rank += ceil_div64(proj_in[q], page_elems) + ceil_div64(proj_out[q], page_elems);
  }
  if (pt_stride < per_rank)
    return na_fail(SLORA_ERR_INVALID, "pt_stride smaller than one adapter's page-table entries");
  // the largest rank whose entries fit in an adapter's stretch of the table
  const int64_t rfit = pt_stride / per_rank;
  const int32_t rmax = rfit < kMaxRank ? (int32_t)rfit : kMaxRank;
  if (T > 0) {
    if (!d_token_adapter || !d_x || !d_y) return na_fail(SLORA_ERR_INVALID, "NULL tokens, x or y");
    if ((reinterpret_cast<uintptr_t>(d_x) | reinterpret_cast<uintptr_t>(d_y) |
         reinterpret_cast<uintptr_t>(d_pool)) & 15)
      return na_fail(SLORA_ERR_INVALID, "pool, x and y must be 16-byte aligned");
    if (ldx < proj_in[proj] || ldx % 8 || ldy < proj_out[proj] || ldy % 8)
      return na_fail(SLORA_ERR_INVALID, "row strides must be multiples of 8 and cover the row");
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return na_fail(SLORA_ERR_INVALID, "device index above 63");
  unsigned char* base = nullptr;
  if (int rc = setup_device(dev, &base)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Carve the static scratch: segment arrays, sanitised ranks, then v.
  int32_t* ints = reinterpret_cast<int32_t*>(base);
  SegDev sd{};
  int32_t* q = ints;
  const int64_t S1 = kNaMaxSegs + 1;
  sd.seg_desc = reinterpret_cast<int4*>(q); q += 4 * S1;   // 16-byte aligned: first in the array
  sd.counts = q; q += kNumCounts;
  sd.perm = q; q += kNaMaxTokens;
  sd.seg_start = q; q += S1;
  sd.seg_adapter = q; q += S1;
  sd.seg_rank = q; q += S1;
  sd.seg_order = q; q += S1;
  sd.cc_shrink_all = q; q += S1;
  sd.cc_tile_all = q; q += S1;
  sd.cc_shrink_short = q; q += S1;
  sd.cc_tile_short = q; q += S1;
  sd.tc_tile_all = q; q += S1;
  sd.tc_tile_long = q; q += S1;
  int32_t* err = q; q += 1;
  // the apply kernel's grid barrier: zero when the module loads; the
  // segment kernel resets its arrival count on every call
  int32_t* grid_sync = q; q += kGridSyncInts;
  int32_t* rank_c = ints + kNaIntsSeg;
  float* v = reinterpret_cast<float*>(base + kNaIntBytes);

  // The error word must start at zero on every call; everything else is
  // fully rewritten by the kernels before it is read.
  e = cudaMemsetAsync(err, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "cudaMemsetAsync(error word)", e);
  // The call's device status, once its kernels are done, into the caller's
  // word (device memory or pinned host memory; no allocation).
  auto copy_status = [&]() -> int {
    if (!status) return SLORA_OK;
    cudaError_t e2 = cudaMemcpyAsync(status, err, sizeof(int32_t), cudaMemcpyDefault, st);
    if (e2 != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "cudaMemcpyAsync(status)", e2);
    return SLORA_OK;
  };
  if (T == 0) return copy_status();
  sanitize_ranks_kernel<<<(max_adapters + 255) / 256, 256, 0, st>>>(d_rank, rank_c, max_adapters, rmax);
  if ((e = cudaGetLastError()) != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "rank copy launch", e);

  SegBuildArgs b{};
  b.token_adapter = d_token_adapter;
  b.T = T;
  b.seg_cap = T < max_adapters ? T : max_adapters;
  b.rank = rank_c;
  b.max_adapters = max_adapters;
  b.tc_threshold = 1 << 30;                 // every segment on the CUDA-core kernels
  b.seg = sd;
  b.error = err;
  b.grid_sync = grid_sync;
  if ((e = launch_build_segments(b, st)) != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "segment build launch", e);

  ApplyDev d{};
  d.nproj = 1;
  d.H = page_elems;
  d.pool = static_cast<const uint16_t*>(d_pool);
  d.page_table = d_page_table;
  d.pt_stride = pt_stride;
  d.perm = sd.perm;
  d.seg_start = sd.seg_start;
  d.seg_adapter = sd.seg_adapter;
  d.seg_rank = sd.seg_rank;
  d.seg_order = sd.seg_order;
  d.counts = sd.counts;
  d.shrink_off = sd.cc_shrink_all;
  d.tile_off = sd.cc_tile_all;
  d.shrink_total_idx = kCcShrinkAll;
  d.tile_total_idx = kCcTileAll;
  d.v_ld = kMaxRank;
  d.s = s;
  d.error = err;
  d.num_pages = 0;   // the caller's pool size is not known here: page indices are not checked
  d.T = T;
  ProjDev& P = d.proj[0];
  P.x = d_x;
  P.ldx = ldx;
  P.y = d_y;
  P.ldy = ldy;
  P.h_in = proj_in[proj];
  P.h_out = proj_out[proj];
  P.ppi = (int32_t)ceil_div64(proj_in[proj], page_elems);
  P.ppo = (int32_t)ceil_div64(proj_out[proj], page_elems);
  P.rows_before = (int32_t)before;
  P.ncol_tiles = expand_col_tiles(P.h_out, page_elems);
  P.v = v;
  d.grid_sync = grid_sync;
  d.seg_desc = sd.seg_desc;
  d.off_n = (T < max_adapters ? T : max_adapters) + 1 < kSegSmem ? (T < max_adapters ? T : max_adapters) + 1 : kSegSmem;
  if ((e = launch_apply_cc(d, dtype, g_grid[dev], st)) != cudaSuccess) return na_fail(SLORA_ERR_CUDA, "apply launch", e);
  return copy_status();
}

static_assert(kNaBytes == SLORA_NOALLOC_SCRATCH_BYTES, "SLORA_NOALLOC_SCRATCH_BYTES must describe the array");
static_assert(kNaMaxTokens == SLORA_NOALLOC_MAX_TOKENS, "SLORA_NOALLOC_MAX_TOKENS must describe the array");
