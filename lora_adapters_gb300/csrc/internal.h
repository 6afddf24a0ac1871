// Internal interface between the host pool (pool.cpp) and the kernels
// (kernels.cu).  Not installed; the public ABI is include/slora.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace slora {

constexpr int kMaxProj = 8;            // == SLORA_MAX_PROJ_PER_CALL: projections of one apply call
constexpr int kMaxPoolProj = 128;      // == SLORA_MAX_PROJ: projections a pool's adapters carry
constexpr int kMaxRank = 256;          // == SLORA_MAX_RANK
constexpr int kMaxAdapters = 32768;    // == SLORA_MAX_ADAPTERS (segment kernel keeps a histogram in smem)

// CUDA-core (gather) kernels: persistent, one CTA per SM, 8 consumer warps
// and one producer warp that feeds a shared-memory ring with bulk copies.
constexpr int kTT = 4;                 // tokens per tile
constexpr int kShrinkRows = 8;         // rank rows per shrink work unit (one per consumer warp)
constexpr int kCcConsumerWarps = 8;
constexpr int kCcThreads = (kCcConsumerWarps + 2) * 32;   // + the planner and the issuer warp
constexpr int kExpandCols = kCcConsumerWarps * 32 * 8;  // 8 output columns (16 bytes) per thread
constexpr int kSegSmem = 1536;         // work-list prefix entries searched in shared memory
constexpr int kSegThreads = 1024;

// Tensor-core (tcgen05) kernels: 128-token tiles of the work lists (the M
// side of tc_expand, half a tc_shrink tile), K block (one 128-byte swizzle row
// of 16-bit elements).
constexpr int kTcM = 128;
constexpr int kTcK = 64;
constexpr int kTcShrinkParts = 3;        // K parts of one tc_shrink (tile, projection)

// Indices into SegDev::counts.
enum CountIdx {
  kNumSegs = 0,
  kNSorted = 1,
  kBadTokens = 2,
  kCcShrinkAll = 3,
  kCcTileAll = 4,
  kCcShrinkShort = 5,
  kCcTileShort = 6,
  kTcTileAll = 7,
  kTcTileLong = 8,
  kNumCounts = 16
};

// Device arrays written by the segment kernel.  Prefix arrays have
// max_segs + 1 entries over work-order positions: prefix[q] = work units of
// the segments seg_order[0..q-1].
struct SegDev {
  int4* seg_desc;           // [max_segs] by work-order position: {adapter, rank, start, end}
  int32_t* perm;            // [max_tokens]
  int32_t* seg_start;       // [max_segs + 1]
  int32_t* seg_adapter;     // [max_segs]
  int32_t* seg_rank;        // [max_segs]
  int32_t* seg_order;       // [max_segs] work order: segments by rank, largest first
  int32_t* counts;          // [kNumCounts]
  int32_t* cc_shrink_all;   // shrink items (token tile x rank-row chunk), every segment
  int32_t* cc_tile_all;     // token tiles, every segment
  int32_t* cc_shrink_short; // the same, only segments below the tensor-core threshold
  int32_t* cc_tile_short;
  int32_t* tc_tile_all;     // 128-token M tiles, every segment
  int32_t* tc_tile_long;    // 128-token M tiles, only segments at/above the threshold
};

// Shared memory of the segment kernel (its own static arrays take ~10 KB).
constexpr int kSegSmemMax = 200 * 1024;
constexpr int32_t kRankInSmem = 1, kSegInSmem = 2, kKeysInSmem = 4;

struct SegBuildArgs {
  const int32_t* token_adapter;  // [T]
  int32_t T;
  int32_t seg_cap;               // segments this batch can have: min(T, max_adapters)
  int32_t smem_flags;            // set by the launcher
  const int32_t* rank;           // [max_adapters], 0 = not resident
  int32_t max_adapters;
  int32_t tc_threshold;
  SegDev seg;
  int32_t* error;                // first device error (0 = none)
  int32_t* grid_sync;            // the apply kernel's grid barrier: arrival count reset here
};

// One projection of an apply call.
struct ProjDev {
  const void* x;
  int64_t ldx;
  void* y;
  int64_t ldy;
  int32_t h_in, h_out;
  int32_t ppi, ppo;              // pages per A row / per B row
  int32_t rows_before;           // page chunks per unit of rank in earlier projections
  int32_t ncol_tiles;            // expand column tiles of kExpandCols
  float* v;                      // shrink result [max_tokens][v_ld], sorted-position rows
};

struct ApplyDev {
  ProjDev proj[kMaxProj];
  int32_t nproj;
  int32_t H;
  const uint16_t* pool;
  const int32_t* page_table;     // adapter a's entries start at a * pt_stride
  int64_t pt_stride;
  const int32_t* perm;
  const int32_t* seg_start;
  const int32_t* seg_adapter;
  const int32_t* seg_rank;
  const int32_t* seg_order;
  const int32_t* counts;
  const int32_t* shrink_off;     // prefix array of the chosen work list
  const int32_t* tile_off;
  int32_t off_n;                 // prefix entries the kernel may stage in shared memory:
                                 // min(kSegSmem, segments this batch can have + 1)
  int32_t shrink_total_idx;      // counts[] index of the list's totals
  int32_t tile_total_idx;
  int32_t v_ld;                  // multiple of 4 (v rows are bulk-copied)
  float s;
  int32_t* error;                // first device error (0 = none)
  const int4* seg_desc;          // per work-order position: {adapter, rank, start, end}
  const float* scale;            // per adapter id: s_a, applied to v (NULL: 1 for every adapter)
  // The grid barrier between the apply kernel's shrink and expand phases:
  // [kSyncCount] CTAs arrived (back to 0 when the last arrives; the segment
  // kernel also zeroes it), [kSyncGen] generation (incremented when the
  // barrier opens).  Zero-initialised with the pool.
  int32_t* grid_sync;
  uint32_t wait_limit;           // polls of a wait on other warps before it gives up (0: kWaitLimit)
  int64_t num_pages;             // pages of the pool (0: unknown, page indices not checked)
  int32_t T;                     // tokens of the batch
};
enum : int { kSyncCount = 0, kSyncGen = 1, kGridSyncInts = 2 };

// Bounds checks of the SLORA_DEBUG build (no code in other builds): an index
// read from a page table or a token order and used to address memory is
// checked against its range (bound <= 0: no range known); one outside it is
// reported in the device error word as SLORA_ERR_DEVICE_ASSERT and replaced
// by 0, so that the access stays in bounds and every copy a barrier expects
// still arrives.  No trap.
constexpr int32_t kErrDeviceAssert = -9;   // == SLORA_ERR_DEVICE_ASSERT
#ifdef __CUDACC__
__device__ __forceinline__ int dbg_index(int v, int64_t bound, int32_t* err) {
#ifdef SLORA_DEBUG
  if (bound > 0 && (v < 0 || (int64_t)v >= bound)) {
    if (err) atomicCAS(err, 0, kErrDeviceAssert);
    return 0;
  }
#else
  (void)bound;
  (void)err;
#endif
  return v;
}
#endif

// Column tiles of a row of h_out elements over pages of H: tiles of at most
// kExpandCols columns that never cross a page boundary.
inline int32_t expand_col_tiles(int32_t h_out, int32_t H) {
  int32_t n = 0;
  for (int32_t c = 0; c * H < h_out; ++c) {
    const int32_t len = (h_out - c * H) < H ? (h_out - c * H) : H;
    n += (len + kExpandCols - 1) / kExpandCols;
  }
  return n;
}

// Tensor-core path of one apply call (long segments).
struct TcDev {
  ApplyDev a;                        // projections, segments, v (fp32), error word
  CUtensorMap pool_map;              // pool as [num_pages x H], box {64, 1} (gather4 rows)
  CUtensorMap y_map[kMaxProj];       // y of each projection as [T x h_out], box {64, 1}
  CUtensorMap y128_map[kMaxProj];    // box {64, 128}
  CUtensorMap y16_map[kMaxProj];     // box {64, 16}
  CUtensorMap vhi_map[kMaxProj];     // v halves as [max_tokens x v16_ld], box {64, 128}
  CUtensorMap vlo_map[kMaxProj];
  uint16_t* vhi[kMaxProj];
  uint16_t* vlo[kMaxProj];
  int32_t v16_ld;                    // multiple of kTcK
  // tc_shrink splits each (tile, projection)'s K range into up to
  // kTcShrinkParts parts; their partial sums (fp32, rows like v) wait here
  // for tc_combine
  float* vpart;                      // tc_shrink's partial sums, [kTcShrinkParts][kMaxProj][rows][v_ld] (by call position)
  int64_t vpart_part, vpart_proj;    // strides in floats
  int32_t tc_ncol[kMaxProj];         // expand column tiles per projection (tc_col_tiles)
  const int32_t* tc_off;             // prefix array of the tensor-core tile list
  int32_t tc_total_idx;
};

// Layout of one of a pool's projections, for the adapter-load kernel (a
// device table written when the pool is created).
struct ProjLayout {
  int32_t h_in, h_out, ppi, ppo;
  int32_t rows_before;           // page chunks per unit of rank in earlier projections
  int32_t pad;
  int64_t elems_before;          // elements per unit of rank in earlier projections (staging layout)
};

// Adapter load: staging -> pages.
struct ScatterDev {
  const uint16_t* staging;       // packed: per projection, A rows then B rows
  uint16_t* pool;
  int32_t H;
  const int32_t* pages;          // the adapter's page-table entries (device)
  int32_t n_entries;
  int32_t rank;
  int32_t nproj;
  const ProjLayout* proj;        // [nproj] (device)
};

// The padded batched-matmul comparator (bmm.cu): one projection.
struct BmmDev {
  const uint16_t* pool;
  const int32_t* page_table;
  int64_t pt_stride;
  int32_t H;
  const int32_t* perm;
  const int32_t* seg_start;
  const int32_t* seg_adapter;
  const int32_t* seg_rank;
  const int32_t* counts;
  const float* scale;            // per adapter id: s_a (NULL: 1)
  int32_t T;                     // tokens of the batch
  int32_t r_pad;                 // every adapter padded to this rank
  int32_t h_in, h_out, ppi, ppo, rows_before;
  int32_t* tok_seg;              // [T] segment of each token, -1: none
  uint16_t* a_pad;               // [T][r_pad][h_in], as stored
  float* b_pad;                  // [T][r_pad][h_out]
  float* delta;                  // [T][h_out] = (x A) B per token (cuBLAS)
  void* y;
  int64_t ldy;
  float s;
  int64_t num_pages;             // pages of the pool (bounds checks of the SLORA_DEBUG build)
  int32_t* error;                // device error word
};
cudaError_t launch_bmm_gather(const BmmDev& d, int dtype, int grid, cudaStream_t st);
cudaError_t launch_bmm_epilogue(const BmmDev& d, int dtype, int grid, cudaStream_t st);

// Launchers (kernels.cu).  dtype: 0 = fp16, 1 = bf16.
cudaError_t launch_build_segments(const SegBuildArgs& a, cudaStream_t st);
// The CUDA-core apply (shrink units, grid barrier, expand units); grid = SMs,
// every CTA resident at once.
cudaError_t launch_apply_cc(const ApplyDev& a, int dtype, int grid, cudaStream_t st);
cudaError_t launch_scatter(const ScatterDev& a, cudaStream_t st);
// *p = v, ordered on the stream (one thread).
cudaError_t launch_set_f32(float* p, float v, cudaStream_t st);
cudaError_t prepare_kernels(int device);   // opt-in shared memory sizes
// Tensor-core kernels (tc_kernels.cu); the page size must be a multiple of kTcK.
cudaError_t prepare_tc_kernels();
cudaError_t launch_tc_shrink(const TcDev& a, int dtype, int grid, cudaStream_t st);
cudaError_t launch_tc_expand(const TcDev& a, int dtype, int grid, cudaStream_t st);
int32_t tc_col_tiles(int32_t h_out, int32_t H);
// Sets the message slora_last_error_string() returns on this thread (pool.cpp).
void set_last_error(const char* msg);

}  // namespace slora
