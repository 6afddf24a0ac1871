// Internal interface between the host pool (pool.cpp) and the kernels
// (kernels.cu).  Not installed; the public ABI is include/slora.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace slora {

constexpr int kMaxProj = 8;            // == SLORA_MAX_PROJ
constexpr int kMaxRank = 256;          // == SLORA_MAX_RANK
constexpr int kMaxAdapters = 32768;    // == SLORA_MAX_ADAPTERS (segment kernel keeps a histogram in smem)

// CUDA-core (gather) kernels: token tile and shrink row chunk.
constexpr int kTT = 8;                 // tokens per tile
constexpr int kShrinkThreads = 256;    // 8 warps, one rank row per warp
constexpr int kShrinkRows = kShrinkThreads / 32;
constexpr int kExpandThreads = 128;    // 8 output columns (16 bytes) per thread
constexpr int kExpandCols = kExpandThreads * 8;
constexpr int kSegThreads = 1024;

// Tensor-core (tcgen05) kernels: M tile of tokens.
constexpr int kTcM = 128;

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
// max_segs + 1 entries: prefix[s] = work units of segments < s.
struct SegDev {
  int32_t* perm;            // [max_tokens]
  int32_t* seg_start;       // [max_segs + 1]
  int32_t* seg_adapter;     // [max_segs]
  int32_t* seg_rank;        // [max_segs]
  int32_t* counts;          // [kNumCounts]
  int32_t* cc_shrink_all;   // shrink items (token tile x rank-row chunk), every segment
  int32_t* cc_tile_all;     // token tiles, every segment
  int32_t* cc_shrink_short; // the same, only segments below the tensor-core threshold
  int32_t* cc_tile_short;
  int32_t* tc_tile_all;     // 128-token M tiles, every segment
  int32_t* tc_tile_long;    // 128-token M tiles, only segments at/above the threshold
};

struct SegBuildArgs {
  const int32_t* token_adapter;  // [T]
  int32_t T;
  const int32_t* rank;           // [max_adapters], 0 = not resident
  int32_t max_adapters;
  int32_t tc_threshold;
  SegDev seg;
  int32_t* error;                // first device error (0 = none)
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
  const int32_t* counts;
  const int32_t* shrink_off;     // prefix array of the chosen work list
  const int32_t* tile_off;
  int32_t shrink_total_idx;      // counts[] index of the list's totals
  int32_t tile_total_idx;
  int32_t v_ld;
  float s;
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
  int32_t h_in[kMaxProj], h_out[kMaxProj];
  int32_t ppi[kMaxProj], ppo[kMaxProj];
  int64_t src_base[kMaxProj];    // element offset of projection q's A rows in staging
  int32_t entry_base[kMaxProj];  // first page-table entry of projection q
};

// Launchers (kernels.cu).  dtype: 0 = fp16, 1 = bf16.
cudaError_t launch_build_segments(const SegBuildArgs& a, cudaStream_t st);
cudaError_t launch_shrink_cc(const ApplyDev& a, int dtype, int grid, cudaStream_t st);
cudaError_t launch_expand_cc(const ApplyDev& a, int dtype, int grid, cudaStream_t st);
cudaError_t launch_scatter(const ScatterDev& a, cudaStream_t st);
cudaError_t prepare_kernels(int device);   // opt-in shared memory sizes
// Sets the message slora_last_error_string() returns on this thread (pool.cpp).
void set_last_error(const char* msg);
// Resident CTAs per SM of each persistent kernel (for grid sizing).
int occupancy_shrink_cc(int dtype);
int occupancy_expand_cc(int dtype);

}  // namespace slora
