// Host side of libslora: the unified page pool (allocator + page tables), the
// asynchronous adapter loader, and the C ABI declared in include/slora.h.
//
// Unified Paging ("S-LoRA: Serving Thousands of Concurrent LoRA Adapters",
// nubint.ai review, abstract; dongaigc.com summary, section 1): one pool of
// H-element pages holds adapter rows of every rank and KV slots of every
// length.  The allocator always hands out the lowest-numbered free pages
// (all or nothing), which makes every page table reproducible call by call.
// Adapters live in host memory and are fetched on demand (nubint.ai review,
// abstract): one cudaMemcpyAsync per weight block into a device staging
// buffer on the copy stream, then a scatter kernel that writes each row chunk
// to its page; the compute stream waits on the load's event before using it.
#include <cublas_v2.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/slora.h"
#include "internal.h"

using namespace slora;

namespace {

thread_local std::string g_err;

// An NVTX range around every call of the C ABI, named after the call, so a
// timeline profiler shows where the host spends its time per call.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
#define SLORA_RANGE(name) NvtxRange nvtx_range_(name)

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CUDA_TRY(call)                                                                    \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return fail(SLORA_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));         \
  } while (0)

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int32_t kOwnerFree = -1;
constexpr int32_t kOwnerKV = -2;
constexpr int32_t kOwnerPending = -3;

enum TimerKind { kTBuild = 0, kTApplyCC, kTShrinkTC, kTExpandTC, kTScatter, kTLoadWait, kTNum };
// load_wait is not a kernel: the time the compute stream waited for adapter
// copies before a segment build (recorded only when it had to wait)
const char* kTimerNames[kTNum] = {"build_segments", "apply_cc", "shrink_tc", "expand_tc", "scatter", "load_wait"};

}  // namespace

struct slora_pool {
  // configuration
  int64_t num_pages = 0;
  int32_t H = 0, dtype = 0, max_adapters = 0, max_rank = 0, max_tokens = 0, num_proj = 0;
  int32_t max_segs = 0;
  int32_t proj_in[kMaxPoolProj] = {}, proj_out[kMaxPoolProj] = {};
  int32_t ppi[kMaxPoolProj] = {}, ppo[kMaxPoolProj] = {}, rows_before[kMaxPoolProj] = {};
  ProjLayout* d_layout = nullptr;        // the projections' layout for the load kernel
  int64_t chunks_per_rank = 0;   // page-table entries per unit of rank
  int64_t pt_stride = 0;         // entries reserved per adapter id
  int64_t staging_elems = 0;
  bool planning = true;
  // AUTO mode: segments of at least tc_threshold tokens on the tensor cores,
  // in batches of at least tc_min_batch tokens (smaller batches: CUDA cores)
  int32_t tc_threshold = 8;
  int32_t tc_min_batch = 2048;

  // allocator
  std::vector<int32_t> owner;    // per page: -1 free, -2 KV, else adapter id
  std::vector<uint64_t> free_bits;
  int64_t free_count = 0;
  int64_t hint_word = 0;         // no free page below word hint_word
  std::vector<int32_t> rank_h;
  std::vector<int64_t> npages_h; // page-table entries per resident adapter
  int32_t* pt_h = nullptr;       // host page-table mirror (pinned unless planning)
  int32_t* rank_pin = nullptr;   // pinned rank mirror (source of the rank H2D copies)

  // device
  uint16_t* d_pool = nullptr;
  cudaStream_t compute = nullptr, copy = nullptr;
  int device = 0;
  int32_t* d_pt = nullptr;
  int32_t* d_rank = nullptr;
  float* d_scale = nullptr;              // per adapter: s_a (1 after a load)
  int32_t* d_error = nullptr;
  int32_t* d_seg_mem = nullptr;
  SegDev seg{};
  float* d_v = nullptr;
  int32_t* d_grid_sync = nullptr;        // the apply kernel's grid barrier
  uint16_t* d_staging = nullptr;
  std::vector<cudaEvent_t> load_event;   // per adapter id (created lazily)
  std::vector<char> load_pending;        // load event recorded, maybe not yet complete
  std::vector<int32_t> pending;          // ids with load_pending set
  cudaEvent_t order_event = nullptr;
  uint64_t seg_generation = 0;
  int32_t seg_T = 0;
  int num_sms = 0;
  int grid_cc = 0;
  // tensor-core path (page size a multiple of kTcK)
  bool tc_ok = false;
  // padded batched-matmul comparator: cuBLAS handle and scratch, made on first use
  cublasHandle_t cublas = nullptr;
  void* d_bmm = nullptr;
  size_t bmm_bytes = 0;
  int32_t v16_ld = 0;            // row stride of the 16-bit v halves
  uint16_t* d_v16 = nullptr;     // v_hi then v_lo, [kMaxProj][max_tokens][v16_ld] each
  float* d_vpart = nullptr;      // tc_shrink's K-part partial sums, [kTcShrinkParts][kMaxProj][rows][v_ld]
  CUtensorMap pool_map{};
  CUtensorMap vhi_map[kMaxProj]{}, vlo_map[kMaxProj]{};

  // fault injection on the host (slora_debug_set_fault / SLORA_FAULT):
  // countdown to the failing event per kind, 0 = disarmed
  int64_t fault_left[3] = {0, 0, 0};
  uint32_t wait_limit = 0;       // polls of the apply kernel's bounded waits (0: the built-in limit)

  // timing
  bool timing = false;
  struct Rec {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> spare_events;
  double t_ms[kTNum] = {};
  int64_t t_launches[kTNum] = {};
};

namespace {

// ---- allocator ------------------------------------------------------------------
void bits_set_free(slora_pool* p, int64_t page, bool is_free) {
  uint64_t m = 1ull << (page & 63);
  if (is_free) p->free_bits[page >> 6] |= m;
  else p->free_bits[page >> 6] &= ~m;
}

// The n lowest-numbered free pages, ascending; caller checked n <= free_count.
void take_lowest(slora_pool* p, int64_t n, int32_t owner, int32_t* out) {
  int64_t got = 0;
  int64_t w = p->hint_word;
  const int64_t nw = (int64_t)p->free_bits.size();
  while (got < n && w < nw) {
    uint64_t bits = p->free_bits[w];
    while (bits && got < n) {
      const int b = __builtin_ctzll(bits);
      bits &= bits - 1;
      const int64_t page = (w << 6) + b;
      out[got++] = (int32_t)page;
      p->owner[page] = owner;
      bits_set_free(p, page, false);
    }
    if (p->free_bits[w] == 0) ++w;
    else break;
  }
  p->hint_word = w;
  // skip words that became full
  while (p->hint_word < nw && p->free_bits[p->hint_word] == 0) ++p->hint_word;
  p->free_count -= n;
}

void give_back(slora_pool* p, int64_t n, const int32_t* pages) {
  for (int64_t i = 0; i < n; ++i) {
    const int64_t page = pages[i];
    p->owner[page] = kOwnerFree;
    bits_set_free(p, page, true);
    p->hint_word = std::min<int64_t>(p->hint_word, page >> 6);
  }
  p->free_count += n;
}

// Row stride of the fp32 shrink scratch: a multiple of 4 floats, so that
// every row starts on a 16-byte boundary for the bulk copies that read it.
int32_t v_ld(const slora_pool* p) { return (p->max_rank + 3) & ~3; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// A 2-D map of 16-bit elements, 128-byte swizzle: `cols` x `rows` with a
// row stride of `row_bytes`, box of box_cols x box_rows.
int encode_2d(CUtensorMap* m, const void* base, int dtype, uint64_t cols, uint64_t rows, uint64_t row_bytes,
              uint32_t box_cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return fail(SLORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dtype == SLORA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SLORA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SLORA_OK;
}

int check_pool(const slora_pool* p) {
  if (!p) return fail(SLORA_ERR_INVALID, "pool is NULL");
  return SLORA_OK;
}

int check_device_pool(const slora_pool* p) {
  if (!p) return fail(SLORA_ERR_INVALID, "pool is NULL");
  if (p->planning) return fail(SLORA_ERR_INVALID, "planning pool (no device buffer): no GPU work");
  return SLORA_OK;
}

// ---- fault injection ----------------------------------------------------------
// True when this event is the one the armed fault of `kind` names (it then
// disarms).  The caller fails the call as the real failure would.
bool fault_fires(slora_pool* p, int kind) {
  int64_t& left = p->fault_left[kind];
  if (left <= 0) return false;
  return --left == 0;
}

// SLORA_FAULT="alloc:N" or "copy:N" arms the fault of slora_debug_set_fault
// for every pool the process creates.
void arm_fault_from_env(slora_pool* p) {
  const char* env = std::getenv("SLORA_FAULT");
  if (!env) return;
  long long n = 0;
  if (std::sscanf(env, "alloc:%lld", &n) == 1 && n > 0) p->fault_left[SLORA_FAULT_PAGE_ALLOC] = n;
  else if (std::sscanf(env, "copy:%lld", &n) == 1 && n > 0) p->fault_left[SLORA_FAULT_COPY] = n;
}

// ---- timing ---------------------------------------------------------------------
cudaEvent_t get_event(slora_pool* p) {
  if (!p->spare_events.empty()) {
    cudaEvent_t e = p->spare_events.back();
    p->spare_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct Timed {
  slora_pool* p;
  int kind;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  Timed(slora_pool* p_, int kind_, cudaStream_t st_) : p(p_), kind(kind_), st(st_) {
    if (p->timing) {
      a = get_event(p);
      if (a) cudaEventRecord(a, st);
    }
  }
  void done() {
    if (!a) return;
    cudaEvent_t b = get_event(p);
    if (!b) return;
    cudaEventRecord(b, st);
    p->recs.push_back({kind, a, b});
    a = nullptr;
  }
};

// Make the compute stream wait for adapter loads that may still be running:
// every one of them, or (h_ids not NULL) only those of the adapters the T
// host ids name.  *waits: the waits enqueued.
int wait_pending_loads(slora_pool* p, const int32_t* h_ids, int32_t T, int* waits) {
  *waits = 0;
  if (h_ids) {
    for (int32_t i = 0; i < T; ++i) {
      const int32_t a = h_ids[i];
      if (a < 0 || a >= p->max_adapters || !p->load_pending[a]) continue;
      cudaError_t q = cudaEventQuery(p->load_event[a]);
      if (q == cudaErrorNotReady) {
        // still copying: the compute stream waits for it; the load stays
        // pending (a reload of the id must still wait for its copies)
        (void)cudaGetLastError();
        CUDA_TRY(cudaStreamWaitEvent(p->compute, p->load_event[a], 0));
        ++*waits;
      } else if (q == cudaSuccess) {
        p->load_pending[a] = 0;
      } else {
        return fail(SLORA_ERR_CUDA, "cudaEventQuery: %s", cudaGetErrorString(q));
      }
    }
    return SLORA_OK;
  }
  std::vector<int32_t> still;
  for (int32_t a : p->pending) {
    if (!p->load_pending[a]) continue;
    cudaError_t q = cudaEventQuery(p->load_event[a]);
    if (q == cudaSuccess) {
      p->load_pending[a] = 0;
      continue;
    }
    if (q != cudaErrorNotReady) return fail(SLORA_ERR_CUDA, "cudaEventQuery: %s", cudaGetErrorString(q));
    (void)cudaGetLastError();  // clear the sticky-free not-ready status
    CUDA_TRY(cudaStreamWaitEvent(p->compute, p->load_event[a], 0));
    ++*waits;
    still.push_back(a);
  }
  p->pending.swap(still);
  return SLORA_OK;
}

// cuBLAS, opened on first use of the comparator only: the library itself
// does not depend on it.
struct CublasApi {
  bool ok = false;
  cublasStatus_t (*create)(cublasHandle_t*) = nullptr;
  cublasStatus_t (*destroy)(cublasHandle_t) = nullptr;
  cublasStatus_t (*set_stream)(cublasHandle_t, cudaStream_t) = nullptr;
  cublasStatus_t (*gemm_sb)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void*,
                            const void*, cudaDataType, int, long long, const void*, cudaDataType, int, long long,
                            const void*, void*, cudaDataType, int, long long, int, cublasComputeType_t,
                            cublasGemmAlgo_t) = nullptr;
};
const CublasApi& cublas_api() {
  static CublasApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* names[] = {"libcublas.so.13", "libcublas.so", "/usr/local/cuda/lib64/libcublas.so.13",
                           "/usr/local/cuda/lib64/libcublas.so"};
    void* h = nullptr;
    for (const char* n : names)
      if ((h = dlopen(n, RTLD_NOW | RTLD_GLOBAL)) != nullptr) break;
    if (!h) return;
    api.create = reinterpret_cast<decltype(api.create)>(dlsym(h, "cublasCreate_v2"));
    api.destroy = reinterpret_cast<decltype(api.destroy)>(dlsym(h, "cublasDestroy_v2"));
    api.set_stream = reinterpret_cast<decltype(api.set_stream)>(dlsym(h, "cublasSetStream_v2"));
    api.gemm_sb = reinterpret_cast<decltype(api.gemm_sb)>(dlsym(h, "cublasGemmStridedBatchedEx"));
    api.ok = api.create && api.destroy && api.set_stream && api.gemm_sb;
  });
  return api;
}

void free_device(slora_pool* p) {
  if (p->planning) {
    std::free(p->pt_h);
    std::free(p->rank_pin);
    return;
  }
  for (auto& r : p->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : p->spare_events) cudaEventDestroy(e);
  for (auto e : p->load_event)
    if (e) cudaEventDestroy(e);
  if (p->order_event) cudaEventDestroy(p->order_event);
  cudaFree(p->d_layout);
  cudaFree(p->d_pt);
  cudaFree(p->d_rank);
  cudaFree(p->d_scale);
  cudaFree(p->d_error);
  cudaFree(p->d_seg_mem);
  cudaFree(p->d_v);
  cudaFree(p->d_grid_sync);
  cudaFree(p->d_v16);
  cudaFree(p->d_vpart);
  cudaFree(p->d_staging);
  cudaFree(p->d_bmm);
  if (p->cublas) cublas_api().destroy(p->cublas);
  if (p->pt_h) cudaFreeHost(p->pt_h);
  if (p->rank_pin) cudaFreeHost(p->rank_pin);
}

}  // namespace

void slora::set_last_error(const char* msg) { g_err = msg ? msg : ""; }

// =================================================================================
extern "C" {

const char* slora_last_error_string(void) { return g_err.c_str(); }

int slora_pool_create(slora_pool** out, void* d_pool, int64_t num_pages, int32_t page_elems,
                      int32_t dtype, int32_t max_adapters, int32_t max_rank, int32_t max_tokens,
                      int32_t num_proj, const int32_t* proj_in, const int32_t* proj_out,
                      void* compute_stream, void* copy_stream) {
  SLORA_RANGE("slora_pool_create");
  if (!out) return fail(SLORA_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (num_pages <= 0 || num_pages >= (1ll << 31))
    return fail(SLORA_ERR_INVALID, "num_pages %lld out of range", (long long)num_pages);
  if (page_elems <= 0 || page_elems % 8 != 0 || page_elems > 65536)
    return fail(SLORA_ERR_INVALID, "page_elems %d must be a positive multiple of 8, <= 65536", page_elems);
  if (dtype != SLORA_F16 && dtype != SLORA_BF16) return fail(SLORA_ERR_INVALID, "dtype %d", dtype);
  if (max_adapters <= 0 || max_adapters > kMaxAdapters)
    return fail(SLORA_ERR_INVALID, "max_adapters %d not in [1, %d]", max_adapters, kMaxAdapters);
  if (max_rank <= 0 || max_rank > kMaxRank)
    return fail(SLORA_ERR_INVALID, "max_rank %d not in [1, %d]", max_rank, kMaxRank);
  if (max_tokens < 0 || max_tokens > (1 << 24)) return fail(SLORA_ERR_INVALID, "max_tokens %d", max_tokens);
  if (num_proj <= 0 || num_proj > kMaxPoolProj || !proj_in || !proj_out)
    return fail(SLORA_ERR_INVALID, "num_proj %d not in [1, %d]", num_proj, kMaxPoolProj);
  if (d_pool && (reinterpret_cast<uintptr_t>(d_pool) & 15))
    return fail(SLORA_ERR_INVALID, "d_pool must be 16-byte aligned");

  slora_pool* p = new (std::nothrow) slora_pool();
  if (!p) return fail(SLORA_ERR_OOM, "host allocation failed");
  p->num_pages = num_pages;
  p->H = page_elems;
  p->dtype = dtype;
  p->max_adapters = max_adapters;
  p->max_rank = max_rank;
  p->max_tokens = max_tokens;
  p->num_proj = num_proj;
  p->max_segs = std::max(1, std::min(max_tokens, max_adapters));
  int64_t before = 0;
  for (int q = 0; q < num_proj; ++q) {
    if (proj_in[q] <= 0 || proj_out[q] <= 0 || proj_in[q] % 8 || proj_out[q] % 8) {
      delete p;
      return fail(SLORA_ERR_INVALID, "projection %d dims %d x %d must be positive multiples of 8", q,
                  proj_in[q], proj_out[q]);
    }
    p->proj_in[q] = proj_in[q];
    p->proj_out[q] = proj_out[q];
    p->ppi[q] = (int32_t)ceil_div(proj_in[q], page_elems);
    p->ppo[q] = (int32_t)ceil_div(proj_out[q], page_elems);
    p->rows_before[q] = (int32_t)before;
    before += p->ppi[q] + p->ppo[q];
    p->staging_elems += (int64_t)max_rank * (proj_in[q] + proj_out[q]);
  }
  p->chunks_per_rank = before;
  p->pt_stride = (int64_t)max_rank * before;
  const int64_t pt_entries = (int64_t)max_adapters * p->pt_stride;

  p->owner.assign((size_t)num_pages, kOwnerFree);
  p->free_bits.assign((size_t)ceil_div(num_pages, 64), ~0ull);
  if (num_pages % 64) p->free_bits.back() = (1ull << (num_pages % 64)) - 1;
  p->free_count = num_pages;
  p->rank_h.assign((size_t)max_adapters, 0);
  p->npages_h.assign((size_t)max_adapters, 0);
  p->planning = (d_pool == nullptr);
  arm_fault_from_env(p);

  if (p->planning) {
    p->pt_h = static_cast<int32_t*>(std::malloc(sizeof(int32_t) * (size_t)pt_entries));
    p->rank_pin = static_cast<int32_t*>(std::calloc((size_t)max_adapters, sizeof(int32_t)));
    if (!p->pt_h || !p->rank_pin) {
      free_device(p);
      delete p;
      return fail(SLORA_ERR_OOM, "host allocation failed");
    }
    std::fill(p->pt_h, p->pt_h + pt_entries, -1);
    *out = p;
    return SLORA_OK;
  }

  p->d_pool = static_cast<uint16_t*>(d_pool);
  p->compute = static_cast<cudaStream_t>(compute_stream);
  p->copy = static_cast<cudaStream_t>(copy_stream);
  int rc = SLORA_OK;
  auto setup = [&]() -> int {
    CUDA_TRY(cudaGetDevice(&p->device));
    CUDA_TRY(cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device));
    CUDA_TRY(prepare_kernels(p->device));
    CUDA_TRY(cudaMallocHost(&p->pt_h, sizeof(int32_t) * (size_t)pt_entries));
    CUDA_TRY(cudaMallocHost(&p->rank_pin, sizeof(int32_t) * (size_t)max_adapters));
    std::fill(p->pt_h, p->pt_h + pt_entries, -1);
    std::fill(p->rank_pin, p->rank_pin + max_adapters, 0);
    CUDA_TRY(cudaMalloc(&p->d_pt, sizeof(int32_t) * (size_t)pt_entries));
    CUDA_TRY(cudaMalloc(&p->d_rank, sizeof(int32_t) * (size_t)max_adapters));
    CUDA_TRY(cudaMalloc(&p->d_scale, sizeof(float) * (size_t)max_adapters));
    {
      const std::vector<float> ones((size_t)max_adapters, 1.0f);
      CUDA_TRY(cudaMemcpy(p->d_scale, ones.data(), sizeof(float) * (size_t)max_adapters, cudaMemcpyHostToDevice));
    }
    CUDA_TRY(cudaMalloc(&p->d_error, sizeof(int32_t)));
    // segment arrays: per-position descriptors (16-byte aligned, first),
    // counts, perm, seg_start, seg_adapter, seg_rank, seg_order, 6 prefix arrays
    const int64_t S1 = p->max_segs + 1;
    const int64_t seg_ints = 4 * S1 + std::max<int64_t>(max_tokens, 1) + S1 * 10 + kNumCounts;
    CUDA_TRY(cudaMalloc(&p->d_seg_mem, sizeof(int32_t) * (size_t)seg_ints));
    int32_t* q = p->d_seg_mem;
    p->seg.seg_desc = reinterpret_cast<int4*>(q); q += 4 * S1;
    p->seg.counts = q; q += kNumCounts;
    p->seg.perm = q; q += std::max<int64_t>(max_tokens, 1);
    p->seg.seg_start = q; q += S1;
    p->seg.seg_adapter = q; q += S1;
    p->seg.seg_rank = q; q += S1;
    p->seg.seg_order = q; q += S1;
    p->seg.cc_shrink_all = q; q += S1;
    p->seg.cc_tile_all = q; q += S1;
    p->seg.cc_shrink_short = q; q += S1;
    p->seg.cc_tile_short = q; q += S1;
    p->seg.tc_tile_all = q; q += S1;
    p->seg.tc_tile_long = q; q += S1;
    CUDA_TRY(cudaMalloc(&p->d_v, sizeof(float) * (size_t)kMaxProj * std::max(max_tokens, 1) * v_ld(p)));
    CUDA_TRY(cudaMalloc(&p->d_staging, sizeof(uint16_t) * (size_t)p->staging_elems));
    {
      std::vector<ProjLayout> lay((size_t)num_proj);
      int64_t elems = 0;
      for (int q = 0; q < num_proj; ++q) {
        lay[q] = ProjLayout{p->proj_in[q], p->proj_out[q], p->ppi[q], p->ppo[q], p->rows_before[q], 0, elems};
        elems += p->proj_in[q] + p->proj_out[q];
      }
      CUDA_TRY(cudaMalloc(&p->d_layout, sizeof(ProjLayout) * (size_t)num_proj));
      CUDA_TRY(cudaMemcpy(p->d_layout, lay.data(), sizeof(ProjLayout) * (size_t)num_proj, cudaMemcpyHostToDevice));
    }
    CUDA_TRY(cudaMalloc(&p->d_grid_sync, kGridSyncInts * sizeof(int32_t)));
    CUDA_TRY(cudaMemsetAsync(p->d_grid_sync, 0, kGridSyncInts * sizeof(int32_t), p->compute));
    CUDA_TRY(cudaMemsetAsync(p->d_pt, 0xff, sizeof(int32_t) * (size_t)pt_entries, p->compute));
    CUDA_TRY(cudaMemsetAsync(p->d_rank, 0, sizeof(int32_t) * (size_t)max_adapters, p->compute));
    CUDA_TRY(cudaMemsetAsync(p->d_error, 0, sizeof(int32_t), p->compute));
    CUDA_TRY(cudaMemsetAsync(p->d_seg_mem, 0, sizeof(int32_t) * (size_t)seg_ints, p->compute));
    CUDA_TRY(cudaEventCreateWithFlags(&p->order_event, cudaEventDisableTiming));
    CUDA_TRY(cudaStreamSynchronize(p->compute));
    p->load_event.assign((size_t)max_adapters, nullptr);
    p->load_pending.assign((size_t)max_adapters, 0);
    p->grid_cc = p->num_sms;   // one persistent CTA per SM
    // Tensor-core path: needs pages of whole 64-element K blocks.
    p->tc_ok = page_elems % kTcK == 0;
    if (p->tc_ok) {
      p->v16_ld = (max_rank + kTcK - 1) / kTcK * kTcK;
      const int64_t rows = std::max(max_tokens, kTcM);   // at least one 128-row box
      const size_t half_elems = (size_t)kMaxProj * rows * p->v16_ld;
      CUDA_TRY(cudaMalloc(&p->d_v16, sizeof(uint16_t) * 2 * half_elems));
      CUDA_TRY(cudaMemsetAsync(p->d_v16, 0, sizeof(uint16_t) * 2 * half_elems, p->compute));
      CUDA_TRY(cudaMalloc(&p->d_vpart, sizeof(float) * kTcShrinkParts * (size_t)kMaxProj * rows * v_ld(p)));
      if (int rc = encode_2d(&p->pool_map, p->d_pool, dtype, (uint64_t)page_elems, (uint64_t)num_pages,
                             (uint64_t)page_elems * 2, kTcK, 1))
        return rc;
      for (int i = 0; i < kMaxProj; ++i) {
        uint16_t* hi = p->d_v16 + (size_t)i * rows * p->v16_ld;
        uint16_t* lo = hi + half_elems;
        if (int rc = encode_2d(&p->vhi_map[i], hi, dtype, p->v16_ld, rows, (uint64_t)p->v16_ld * 2, kTcK, kTcM))
          return rc;
        if (int rc = encode_2d(&p->vlo_map[i], lo, dtype, p->v16_ld, rows, (uint64_t)p->v16_ld * 2, kTcK, kTcM))
          return rc;
      }
      CUDA_TRY(prepare_tc_kernels());
    } else {
      p->tc_threshold = INT32_MAX;   // every segment stays on the CUDA-core kernels
    }
    return SLORA_OK;
  };
  rc = setup();
  if (rc != SLORA_OK) {
    std::string why = g_err;
    free_device(p);
    delete p;
    g_err = why;
    return rc;
  }
  *out = p;
  return SLORA_OK;
}

int slora_pool_destroy(slora_pool* p) {
  SLORA_RANGE("slora_pool_destroy");
  if (!p) return fail(SLORA_ERR_INVALID, "pool is NULL");
  int rc = SLORA_OK;
  if (!p->planning) {
    cudaError_t e1 = cudaStreamSynchronize(p->copy);
    cudaError_t e2 = cudaStreamSynchronize(p->compute);
    if (e1 != cudaSuccess || e2 != cudaSuccess)
      rc = fail(SLORA_ERR_CUDA, "stream synchronize at destroy: %s",
                cudaGetErrorString(e1 != cudaSuccess ? e1 : e2));
  }
  free_device(p);
  delete p;
  return rc;
}

int slora_pages_alloc(slora_pool* p, int64_t n, int32_t* out_pages) {
  SLORA_RANGE("slora_pages_alloc");
  if (int rc = check_pool(p)) return rc;
  if (n < 0 || (n > 0 && !out_pages)) return fail(SLORA_ERR_INVALID, "bad count or NULL output");
  if (n > p->free_count)
    return fail(SLORA_ERR_OOM, "need %lld pages, %lld free", (long long)n, (long long)p->free_count);
  if (fault_fires(p, SLORA_FAULT_PAGE_ALLOC)) return fail(SLORA_ERR_OOM, "injected page-allocation failure");
  take_lowest(p, n, kOwnerKV, out_pages);
  return SLORA_OK;
}

int slora_pages_free(slora_pool* p, int64_t n, const int32_t* pages) {
  SLORA_RANGE("slora_pages_free");
  if (int rc = check_pool(p)) return rc;
  if (n < 0 || (n > 0 && !pages)) return fail(SLORA_ERR_INVALID, "bad count or NULL pages");
  int64_t i = 0;
  int rc = SLORA_OK;
  for (; i < n; ++i) {  // validate, marking pages pending to catch duplicates
    const int64_t pg = pages[i];
    if (pg < 0 || pg >= p->num_pages) { rc = fail(SLORA_ERR_INVALID, "page %lld out of range", (long long)pg); break; }
    if (p->owner[pg] != kOwnerKV) {
      rc = fail(SLORA_ERR_INVALID, "page %lld is not a KV page (owner %d)", (long long)pg, p->owner[pg]);
      break;
    }
    p->owner[pg] = kOwnerPending;
  }
  if (rc != SLORA_OK) {
    for (int64_t j = 0; j < i; ++j) p->owner[pages[j]] = kOwnerKV;
    return rc;
  }
  give_back(p, n, pages);
  return SLORA_OK;
}

int slora_pool_info(const slora_pool* p, int64_t* free_pages, int64_t* num_pages, int32_t* page_elems,
                    int64_t* pages_per_rank) {
  SLORA_RANGE("slora_pool_info");
  if (int rc = check_pool(p)) return rc;
  if (free_pages) *free_pages = p->free_count;
  if (num_pages) *num_pages = p->num_pages;
  if (page_elems) *page_elems = p->H;
  if (pages_per_rank) *pages_per_rank = p->chunks_per_rank;
  return SLORA_OK;
}

int slora_adapter_load(slora_pool* p, int32_t a, int32_t rank, const void* const* h_A,
                       const void* const* h_B, void** done) {
  SLORA_RANGE("slora_adapter_load");
  if (int rc = check_pool(p)) return rc;
  if (done) *done = nullptr;
  if (a < 0 || a >= p->max_adapters) return fail(SLORA_ERR_INVALID, "adapter id %d out of range", a);
  if (rank < 1 || rank > p->max_rank) return fail(SLORA_ERR_INVALID, "rank %d not in [1, %d]", rank, p->max_rank);
  if (p->rank_h[a] != 0) return fail(SLORA_ERR_EXISTS, "adapter %d already resident", a);
  if (!p->planning) {
    if (!h_A || !h_B) return fail(SLORA_ERR_INVALID, "NULL weight arrays");
    for (int q = 0; q < p->num_proj; ++q)
      if (!h_A[q] || !h_B[q]) return fail(SLORA_ERR_INVALID, "NULL weights of projection %d", q);
  }
  const int64_t n = (int64_t)rank * p->chunks_per_rank;
  if (n > p->free_count)
    return fail(SLORA_ERR_OOM, "adapter %d needs %lld pages, %lld free", a, (long long)n, (long long)p->free_count);
  if (fault_fires(p, SLORA_FAULT_PAGE_ALLOC)) return fail(SLORA_ERR_OOM, "injected page-allocation failure");

  if (!p->planning && p->load_pending[a]) {
    // The previous load of this id may still read its page-table mirror.
    CUDA_TRY(cudaEventSynchronize(p->load_event[a]));
    p->load_pending[a] = 0;
  }
  int32_t* tab = p->pt_h + (int64_t)a * p->pt_stride;
  take_lowest(p, n, a, tab);
  p->rank_h[a] = rank;
  p->npages_h[a] = n;
  if (p->planning) return SLORA_OK;

  // A failed enqueue: the pages go back and the host state is as before the
  // call.  Work already queued on the copy stream (staging copies, the page
  // table, the scatter into the pages) is waited for first, so that nothing
  // writes the pages once another owner may hold them; the id's device rank
  // stays 0, so nothing reads what it wrote.  This wait is the error path's
  // only blocking call.
  auto rollback = [&](int code) {
    const std::string why = g_err;
    (void)cudaStreamSynchronize(p->copy);
    (void)cudaGetLastError();
    give_back(p, n, tab);
    std::fill(tab, tab + n, -1);
    p->rank_h[a] = 0;
    p->npages_h[a] = 0;
    p->rank_pin[a] = 0;
    g_err = why;
    return code;
  };
  auto enqueue = [&]() -> int {
    if (!p->load_event[a]) CUDA_TRY(cudaEventCreateWithFlags(&p->load_event[a], cudaEventDisableTiming));
    // Order the copies after everything queued on the compute stream so far:
    // pages released by earlier evicts / KV frees are no longer being read,
    // and an evict's rank clear of this id lands before the new rank.
    CUDA_TRY(cudaEventRecord(p->order_event, p->compute));
    CUDA_TRY(cudaStreamWaitEvent(p->copy, p->order_event, 0));
    p->rank_pin[a] = rank;
    // every copy or kernel the load enqueues is one event of SLORA_FAULT_COPY
    auto injected = [&]() { return fault_fires(p, SLORA_FAULT_COPY); };
    if (injected()) return fail(SLORA_ERR_CUDA, "injected failure of a copy enqueue");
    CUDA_TRY(cudaMemcpyAsync(p->d_pt + (int64_t)a * p->pt_stride, tab, sizeof(int32_t) * (size_t)n,
                             cudaMemcpyHostToDevice, p->copy));
    int64_t off = 0;
    ScatterDev sd{};
    sd.staging = p->d_staging;
    sd.pool = p->d_pool;
    sd.H = p->H;
    sd.pages = p->d_pt + (int64_t)a * p->pt_stride;
    sd.n_entries = (int32_t)n;
    sd.rank = rank;
    sd.nproj = p->num_proj;
    sd.proj = p->d_layout;
    // The staging buffer takes projection by projection the A rows, then the
    // B rows.  Host blocks that follow each other in host memory as they do
    // in staging go in one copy: an adapter stored contiguously (per layer,
    // or whole) moves in a few large copies instead of two per projection.
    const char* run_src = nullptr;
    size_t run_bytes = 0;
    int64_t run_dst = 0;
    auto flush = [&]() -> int {
      if (run_bytes == 0) return SLORA_OK;
      if (injected()) return fail(SLORA_ERR_CUDA, "injected failure of a copy enqueue");
      CUDA_TRY(cudaMemcpyAsync(p->d_staging + run_dst, run_src, run_bytes, cudaMemcpyHostToDevice, p->copy));
      run_bytes = 0;
      return SLORA_OK;
    };
    for (int q = 0; q < p->num_proj; ++q) {
      for (int half = 0; half < 2; ++half) {
        const char* src = static_cast<const char*>(half == 0 ? h_A[q] : h_B[q]);
        const size_t bytes = sizeof(uint16_t) * (size_t)rank * (half == 0 ? p->proj_in[q] : p->proj_out[q]);
        if (run_bytes > 0 && src != run_src + run_bytes)
          if (int rc = flush()) return rc;
        if (run_bytes == 0) {
          run_src = src;
          run_dst = off;
        }
        run_bytes += bytes;
        off += (int64_t)(bytes / sizeof(uint16_t));
      }
    }
    if (int rc = flush()) return rc;
    {
      Timed tm(p, kTScatter, p->copy);
      if (injected()) return fail(SLORA_ERR_CUDA, "injected failure of a copy enqueue");
      CUDA_TRY(launch_scatter(sd, p->copy));
      tm.done();
    }
    if (injected()) return fail(SLORA_ERR_CUDA, "injected failure of a copy enqueue");
    CUDA_TRY(launch_set_f32(p->d_scale + a, 1.0f, p->copy));   // a fresh adapter: s_a = 1
    if (injected()) return fail(SLORA_ERR_CUDA, "injected failure of a copy enqueue");
    CUDA_TRY(cudaMemcpyAsync(p->d_rank + a, p->rank_pin + a, sizeof(int32_t), cudaMemcpyHostToDevice,
                             p->copy));
    CUDA_TRY(cudaEventRecord(p->load_event[a], p->copy));
    return SLORA_OK;
  };
  int rc = enqueue();
  if (rc != SLORA_OK) return rollback(rc);
  p->load_pending[a] = 1;
  p->pending.push_back(a);
  if (done) *done = p->load_event[a];
  return SLORA_OK;
}

int slora_adapter_evict(slora_pool* p, int32_t a) {
  SLORA_RANGE("slora_adapter_evict");
  if (int rc = check_pool(p)) return rc;
  if (a < 0 || a >= p->max_adapters || p->rank_h[a] == 0)
    return fail(SLORA_ERR_NOT_RESIDENT, "adapter %d is not resident", a);
  if (!p->planning) {
    // A load of this adapter still copying writes its pages: later work on
    // the compute stream (which may reuse them) waits for it.
    if (p->load_pending[a]) CUDA_TRY(cudaStreamWaitEvent(p->compute, p->load_event[a], 0));
    // Work queued before this call still sees the adapter; later work does not.
    CUDA_TRY(cudaMemsetAsync(p->d_rank + a, 0, sizeof(int32_t), p->compute));
  }
  int32_t* tab = p->pt_h + (int64_t)a * p->pt_stride;
  give_back(p, p->npages_h[a], tab);
  std::fill(tab, tab + p->npages_h[a], -1);
  p->rank_h[a] = 0;
  p->npages_h[a] = 0;
  // Segment handles carry the ranks seen when they were built; a reload of
  // this id with another rank would make them index the wrong entries.
  p->seg_generation++;
  return SLORA_OK;
}

int slora_adapter_set_scale(slora_pool* p, int32_t a, float scale) {
  SLORA_RANGE("slora_adapter_set_scale");
  if (int rc = check_device_pool(p)) return rc;
  if (a < 0 || a >= p->max_adapters || p->rank_h[a] == 0)
    return fail(SLORA_ERR_NOT_RESIDENT, "adapter %d is not resident", a);
  if (!std::isfinite(scale)) return fail(SLORA_ERR_INVALID, "scale of adapter %d is not finite", a);
  // after the adapter's own load (which sets s_a = 1), before later applies
  if (p->load_pending[a]) CUDA_TRY(cudaStreamWaitEvent(p->compute, p->load_event[a], 0));
  CUDA_TRY(launch_set_f32(p->d_scale + a, scale, p->compute));
  return SLORA_OK;
}

int slora_adapter_ready(slora_pool* p, int32_t a, int32_t* ready) {
  SLORA_RANGE("slora_adapter_ready");
  if (int rc = check_pool(p)) return rc;
  if (!ready) return fail(SLORA_ERR_INVALID, "ready is NULL");
  if (a < 0 || a >= p->max_adapters || p->rank_h[a] == 0)
    return fail(SLORA_ERR_NOT_RESIDENT, "adapter %d is not resident", a);
  *ready = 1;
  if (!p->planning && p->load_pending[a]) {
    const cudaError_t q = cudaEventQuery(p->load_event[a]);
    if (q == cudaSuccess) {
      p->load_pending[a] = 0;
    } else if (q == cudaErrorNotReady) {
      (void)cudaGetLastError();
      *ready = 0;
    } else {
      return fail(SLORA_ERR_CUDA, "cudaEventQuery: %s", cudaGetErrorString(q));
    }
  }
  return SLORA_OK;
}

int slora_adapter_pages(const slora_pool* p, int32_t a, int32_t* out_pages, int64_t capacity, int64_t* n) {
  SLORA_RANGE("slora_adapter_pages");
  if (int rc = check_pool(p)) return rc;
  if (a < 0 || a >= p->max_adapters || p->rank_h[a] == 0)
    return fail(SLORA_ERR_NOT_RESIDENT, "adapter %d is not resident", a);
  const int64_t cnt = p->npages_h[a];
  if (n) *n = cnt;
  if (out_pages) {
    if (capacity < cnt) return fail(SLORA_ERR_INVALID, "capacity %lld < %lld", (long long)capacity, (long long)cnt);
    std::memcpy(out_pages, p->pt_h + (int64_t)a * p->pt_stride, sizeof(int32_t) * (size_t)cnt);
  }
  return SLORA_OK;
}

int slora_build_segments(slora_pool* p, const int32_t* d_ta, int32_t T, slora_segments* out) {
  SLORA_RANGE("slora_build_segments");
  return slora_build_segments_for(p, d_ta, T, nullptr, out);
}

int slora_build_segments_for(slora_pool* p, const int32_t* d_ta, int32_t T, const int32_t* h_ta,
                             slora_segments* out) {
  SLORA_RANGE("slora_build_segments_for");
  if (int rc = check_device_pool(p)) return rc;
  if (!out) return fail(SLORA_ERR_INVALID, "out is NULL");
  if (T < 0 || T > p->max_tokens) return fail(SLORA_ERR_INVALID, "T=%d not in [0, %d]", T, p->max_tokens);
  if (T > 0 && !d_ta) return fail(SLORA_ERR_INVALID, "token_adapter is NULL");
  {
    // the waits, timed when timing is on and a wait was enqueued
    cudaEvent_t w0 = p->timing ? get_event(p) : nullptr;
    if (w0) cudaEventRecord(w0, p->compute);
    int waits = 0;
    if (int rc = wait_pending_loads(p, h_ta, T, &waits)) return rc;
    if (w0) {
      cudaEvent_t w1 = waits ? get_event(p) : nullptr;
      if (w1) {
        cudaEventRecord(w1, p->compute);
        p->recs.push_back({kTLoadWait, w0, w1});
      } else {
        p->spare_events.push_back(w0);
      }
    }
  }
  SegBuildArgs args{};
  args.token_adapter = d_ta;
  args.T = T;
  args.seg_cap = std::max(1, std::min(T, p->max_adapters));
  args.rank = p->d_rank;
  args.max_adapters = p->max_adapters;
  args.tc_threshold = p->tc_threshold;
  args.seg = p->seg;
  args.error = p->d_error;
  args.grid_sync = p->d_grid_sync;
  {
    Timed tm(p, kTBuild, p->compute);
    CUDA_TRY(launch_build_segments(args, p->compute));
    tm.done();
  }
  p->seg_generation++;
  p->seg_T = T;
  out->T = T;
  out->max_segs = p->max_segs;
  out->perm = p->seg.perm;
  out->seg_start = p->seg.seg_start;
  out->seg_adapter = p->seg.seg_adapter;
  out->counts = p->seg.counts;
  out->generation = p->seg_generation;
  return SLORA_OK;
}

int slora_lora_apply_multi(slora_pool* p, const slora_segments* seg, int32_t n, const int32_t* projs,
                           const void* const* d_x, const int64_t* ldx, void* const* d_y,
                           const int64_t* ldy, float s, int32_t mode) {
  SLORA_RANGE("slora_lora_apply_multi");
  if (int rc = check_device_pool(p)) return rc;
  if (!seg || seg->generation != p->seg_generation || seg->generation == 0)
    return fail(SLORA_ERR_INVALID, "segments are missing or stale (rebuild them after every build call)");
  if (n < 1 || n > kMaxProj || !projs || !d_x || !ldx || !d_y || !ldy)
    return fail(SLORA_ERR_INVALID, "n=%d projections (1..%d) and non-NULL arrays required", n, kMaxProj);
  if (mode < SLORA_MODE_AUTO || mode > SLORA_MODE_PREFILL) return fail(SLORA_ERR_INVALID, "mode %d", mode);
  ApplyDev d{};
  d.nproj = n;
  d.H = p->H;
  d.pool = p->d_pool;
  d.page_table = p->d_pt;
  d.pt_stride = p->pt_stride;
  d.perm = p->seg.perm;
  d.seg_start = p->seg.seg_start;
  d.seg_adapter = p->seg.seg_adapter;
  d.seg_rank = p->seg.seg_rank;
  d.seg_order = p->seg.seg_order;
  d.counts = p->seg.counts;
  d.v_ld = v_ld(p);
  d.error = p->d_error;
  d.grid_sync = p->d_grid_sync;
  d.seg_desc = p->seg.seg_desc;
  d.scale = p->d_scale;
  d.off_n = std::min<int32_t>(kSegSmem, std::max(1, std::min(p->seg_T, p->max_adapters)) + 1);
  d.s = s;
  d.wait_limit = p->wait_limit;
  d.num_pages = p->num_pages;
  d.T = p->seg_T;
  for (int i = 0; i < n; ++i) {
    const int q = projs[i];
    if (q < 0 || q >= p->num_proj) return fail(SLORA_ERR_INVALID, "projection %d out of range", q);
    if (p->seg_T > 0 && (!d_x[i] || !d_y[i])) return fail(SLORA_ERR_INVALID, "NULL x or y");
    if ((reinterpret_cast<uintptr_t>(d_x[i]) | reinterpret_cast<uintptr_t>(d_y[i])) & 15)
      return fail(SLORA_ERR_INVALID, "x and y must be 16-byte aligned");
    if (ldx[i] < p->proj_in[q] || ldx[i] % 8 || ldy[i] < p->proj_out[q] || ldy[i] % 8)
      return fail(SLORA_ERR_INVALID, "row strides must be multiples of 8 and cover the row");
    ProjDev& P = d.proj[i];
    P.x = d_x[i];
    P.ldx = ldx[i];
    P.y = d_y[i];
    P.ldy = ldy[i];
    P.h_in = p->proj_in[q];
    P.h_out = p->proj_out[q];
    P.ppi = p->ppi[q];
    P.ppo = p->ppo[q];
    P.rows_before = p->rows_before[q];
    P.ncol_tiles = expand_col_tiles(P.h_out, p->H);
    P.v = p->d_v + (int64_t)i * std::max(p->max_tokens, 1) * v_ld(p);
  }
  if (p->seg_T == 0) return SLORA_OK;
  // PREFILL: every segment on the tensor cores.  AUTO: the long segments of a
  // large batch; a small batch (decode) has too few long segments to fill the
  // tensor-core kernels, which are then bound by latency, not bandwidth.
  const bool use_tc = p->tc_ok && (mode == SLORA_MODE_PREFILL ||
                                   (mode == SLORA_MODE_AUTO && p->seg_T >= p->tc_min_batch));
  if (use_tc) {
    // short segments on the CUDA-core kernels, long ones on the tensor cores
    d.shrink_off = p->seg.cc_shrink_short;
    d.tile_off = p->seg.cc_tile_short;
    d.shrink_total_idx = kCcShrinkShort;
    d.tile_total_idx = kCcTileShort;
  } else {
    d.shrink_off = p->seg.cc_shrink_all;
    d.tile_off = p->seg.cc_tile_all;
    d.shrink_total_idx = kCcShrinkAll;
    d.tile_total_idx = kCcTileAll;
  }
  if (use_tc) {
    TcDev t;
    memset(&t, 0, sizeof t);
    t.a = d;
    t.pool_map = p->pool_map;
    t.v16_ld = p->v16_ld;
    const int64_t rows = std::max(p->max_tokens, kTcM);
    const size_t half_elems = (size_t)kMaxProj * rows * p->v16_ld;
    for (int i = 0; i < n; ++i) {
      const ProjDev& P = d.proj[i];
      for (int b = 0; b < 3; ++b) {   // y maps of tc_expand (x rows are copied with cp.async)
        const uint32_t box_rows = b == 0 ? 1 : b == 1 ? kTcM : 16;
        CUtensorMap* my = b == 0 ? &t.y_map[i] : b == 1 ? &t.y128_map[i] : &t.y16_map[i];
        if (int rc = encode_2d(my, P.y, p->dtype, (uint64_t)P.h_out, (uint64_t)p->seg_T, (uint64_t)P.ldy * 2, kTcK,
                               box_rows))
          return rc;
      }
      t.vhi_map[i] = p->vhi_map[i];
      t.vlo_map[i] = p->vlo_map[i];
      t.vhi[i] = p->d_v16 + (size_t)i * rows * p->v16_ld;
      t.vlo[i] = t.vhi[i] + half_elems;
      t.tc_ncol[i] = tc_col_tiles(P.h_out, p->H);
    }
    t.vpart = p->d_vpart;
    t.vpart_proj = rows * v_ld(p);
    t.vpart_part = (int64_t)kMaxProj * rows * v_ld(p);
    if (!t.vpart) return fail(SLORA_ERR_INVALID, "tensor-core scratch is missing");
    if (mode == SLORA_MODE_PREFILL) {
      // every segment on the tensor cores; no CUDA-core launch
      t.tc_off = p->seg.tc_tile_all;
      t.tc_total_idx = kTcTileAll;
    } else {
      t.tc_off = p->seg.tc_tile_long;
      t.tc_total_idx = kTcTileLong;
      Timed tm(p, kTApplyCC, p->compute);
      CUDA_TRY(launch_apply_cc(d, p->dtype, p->grid_cc, p->compute));
      tm.done();
    }
    {
      Timed tm(p, kTShrinkTC, p->compute);
      CUDA_TRY(launch_tc_shrink(t, p->dtype, p->grid_cc, p->compute));
      tm.done();
    }
    {
      Timed tm(p, kTExpandTC, p->compute);
      CUDA_TRY(launch_tc_expand(t, p->dtype, p->grid_cc, p->compute));
      tm.done();
    }
  } else {
    Timed tm(p, kTApplyCC, p->compute);
    CUDA_TRY(launch_apply_cc(d, p->dtype, p->grid_cc, p->compute));
    tm.done();
  }
  return SLORA_OK;
}

int slora_lora_apply(slora_pool* p, const slora_segments* seg, int32_t proj, const void* d_x, int64_t ldx,
                     void* d_y, int64_t ldy, float s, int32_t mode) {
  SLORA_RANGE("slora_lora_apply");
  const void* xs[1] = {d_x};
  void* ys[1] = {d_y};
  return slora_lora_apply_multi(p, seg, 1, &proj, xs, &ldx, ys, &ldy, s, mode);
}

int slora_lora_apply_bmm(slora_pool* p, const slora_segments* seg, int32_t proj, const void* d_x, int64_t ldx,
                         void* d_y, int64_t ldy, float s) {
  SLORA_RANGE("slora_lora_apply_bmm");
  if (int rc = check_device_pool(p)) return rc;
  if (!seg || seg->generation != p->seg_generation || seg->generation == 0)
    return fail(SLORA_ERR_INVALID, "segments are missing or stale (rebuild them after every build call)");
  if (proj < 0 || proj >= p->num_proj) return fail(SLORA_ERR_INVALID, "projection %d out of range", proj);
  if (p->seg_T > 0 && (!d_x || !d_y)) return fail(SLORA_ERR_INVALID, "NULL x or y");
  if ((reinterpret_cast<uintptr_t>(d_x) | reinterpret_cast<uintptr_t>(d_y)) & 15)
    return fail(SLORA_ERR_INVALID, "x and y must be 16-byte aligned");
  if (ldx < p->proj_in[proj] || ldx % 8 || ldy < p->proj_out[proj] || ldy % 8)
    return fail(SLORA_ERR_INVALID, "row strides must be multiples of 8 and cover the row");
  if (p->seg_T == 0) return SLORA_OK;
  const CublasApi& cb = cublas_api();
  if (!cb.ok) return fail(SLORA_ERR_CUDA, "cuBLAS could not be opened");
  const int T = p->seg_T, r_pad = p->max_rank;
  const int h_in = p->proj_in[proj], h_out = p->proj_out[proj];
  if (!p->d_bmm) {   // sized for the largest batch and projection of the pool
    int32_t mi = 0, mo = 0;
    for (int q = 0; q < p->num_proj; ++q) {
      mi = std::max(mi, p->proj_in[q]);
      mo = std::max(mo, p->proj_out[q]);
    }
    const size_t Tm = (size_t)std::max(p->max_tokens, 1);
    const size_t bytes = Tm * r_pad * mi * 2 + Tm * r_pad * mo * 4 + Tm * r_pad * 4 + Tm * mo * 4 + Tm * 4 + 64;
    if (cudaMalloc(&p->d_bmm, bytes) != cudaSuccess) {
      p->d_bmm = nullptr;
      cudaGetLastError();
      return fail(SLORA_ERR_OOM, "comparator scratch of %zu bytes", bytes);
    }
    p->bmm_bytes = bytes;
  }
  if (!p->cublas) {
    if (cb.create(&p->cublas) != CUBLAS_STATUS_SUCCESS) {
      p->cublas = nullptr;
      return fail(SLORA_ERR_CUDA, "cublasCreate failed");
    }
  }
  if (cb.set_stream(p->cublas, p->compute) != CUBLAS_STATUS_SUCCESS) return fail(SLORA_ERR_CUDA, "cublasSetStream failed");
  BmmDev d{};
  d.pool = p->d_pool;
  d.page_table = p->d_pt;
  d.pt_stride = p->pt_stride;
  d.H = p->H;
  d.perm = p->seg.perm;
  d.seg_start = p->seg.seg_start;
  d.seg_adapter = p->seg.seg_adapter;
  d.seg_rank = p->seg.seg_rank;
  d.counts = p->seg.counts;
  d.scale = p->d_scale;
  d.T = T;
  d.r_pad = r_pad;
  d.num_pages = p->num_pages;
  d.error = p->d_error;
  d.h_in = h_in;
  d.h_out = h_out;
  d.ppi = p->ppi[proj];
  d.ppo = p->ppo[proj];
  d.rows_before = p->rows_before[proj];
  char* q = static_cast<char*>(p->d_bmm);
  d.a_pad = reinterpret_cast<uint16_t*>(q); q += (size_t)T * r_pad * h_in * 2;
  d.b_pad = reinterpret_cast<float*>(q); q += (size_t)T * r_pad * h_out * 4;
  float* v = reinterpret_cast<float*>(q); q += (size_t)T * r_pad * 4;
  d.delta = reinterpret_cast<float*>(q); q += (size_t)T * h_out * 4;
  d.tok_seg = reinterpret_cast<int32_t*>(q);
  d.y = d_y;
  d.ldy = ldy;
  d.s = s;
  CUDA_TRY(launch_bmm_gather(d, p->dtype, p->grid_cc, p->compute));
  const cudaDataType t16 = p->dtype == SLORA_F16 ? CUDA_R_16F : CUDA_R_16BF;
  const float one = 1.f, zero = 0.f;
  // v_t[r_pad] = A_t (x_t): a_pad[t] is [r_pad][h_in] row-major, i.e. h_in x r_pad column-major
  if (cb.gemm_sb(p->cublas, CUBLAS_OP_T, CUBLAS_OP_N, r_pad, 1, h_in, &one, d.a_pad, t16, h_in,
                 (long long)r_pad * h_in, d_x, t16, (int)ldx, (long long)ldx, &zero, v, CUDA_R_32F, r_pad,
                 (long long)r_pad, T, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return fail(SLORA_ERR_CUDA, "batched GEMM (x A) failed");
  // delta_t[h_out] = B_t^T v_t: b_pad[t] is [r_pad][h_out] row-major, i.e. h_out x r_pad column-major
  if (cb.gemm_sb(p->cublas, CUBLAS_OP_N, CUBLAS_OP_N, h_out, 1, r_pad, &one, d.b_pad, CUDA_R_32F, h_out,
                 (long long)r_pad * h_out, v, CUDA_R_32F, r_pad, (long long)r_pad, &zero, d.delta, CUDA_R_32F,
                 h_out, (long long)h_out, T, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return fail(SLORA_ERR_CUDA, "batched GEMM (v B) failed");
  CUDA_TRY(launch_bmm_epilogue(d, p->dtype, p->grid_cc, p->compute));
  return SLORA_OK;
}

int slora_bmm_scratch_bytes(const slora_pool* p, size_t* bytes) {
  SLORA_RANGE("slora_bmm_scratch_bytes");
  if (int rc = check_pool(p)) return rc;
  if (!bytes) return fail(SLORA_ERR_INVALID, "bytes is NULL");
  *bytes = p->bmm_bytes;
  return SLORA_OK;
}

int slora_device_status(slora_pool* p, int32_t* status) {
  SLORA_RANGE("slora_device_status");
  if (int rc = check_device_pool(p)) return rc;
  if (!status) return fail(SLORA_ERR_INVALID, "status is NULL");
  int32_t v = 0;
  CUDA_TRY(cudaMemcpyAsync(&v, p->d_error, sizeof v, cudaMemcpyDeviceToHost, p->compute));
  CUDA_TRY(cudaMemsetAsync(p->d_error, 0, sizeof(int32_t), p->compute));
  CUDA_TRY(cudaStreamSynchronize(p->compute));
  if (v == SLORA_ERR_TIMEOUT) {
    // A call that gave up may have left the apply kernel's grid barrier
    // part-way; clear it so that the next call starts clean.
    CUDA_TRY(cudaMemsetAsync(p->d_grid_sync, 0, kGridSyncInts * sizeof(int32_t), p->compute));
    CUDA_TRY(cudaStreamSynchronize(p->compute));
  }
  *status = v;
  return SLORA_OK;
}

int slora_pool_snapshot(const slora_pool* p, void* buf, size_t* len) {
  SLORA_RANGE("slora_pool_snapshot");
  if (int rc = check_pool(p)) return rc;
  if (!len) return fail(SLORA_ERR_INVALID, "len is NULL");
  const size_t need = 2 * sizeof(int64_t) + 2 * sizeof(int32_t) +
                      sizeof(int32_t) * ((size_t)p->num_pages + (size_t)p->max_adapters +
                                         (size_t)p->max_adapters * (size_t)p->pt_stride);
  if (!buf) {
    *len = need;
    return SLORA_OK;
  }
  if (*len < need) return fail(SLORA_ERR_INVALID, "buffer of %zu bytes < %zu", *len, need);
  char* c = static_cast<char*>(buf);
  const int64_t hdr64[2] = {p->num_pages, p->free_count};
  const int32_t hdr32[2] = {p->max_adapters, (int32_t)p->pt_stride};
  std::memcpy(c, hdr64, sizeof hdr64);
  c += sizeof hdr64;
  std::memcpy(c, hdr32, sizeof hdr32);
  c += sizeof hdr32;
  std::memcpy(c, p->owner.data(), sizeof(int32_t) * (size_t)p->num_pages);
  c += sizeof(int32_t) * (size_t)p->num_pages;
  std::memcpy(c, p->rank_h.data(), sizeof(int32_t) * (size_t)p->max_adapters);
  c += sizeof(int32_t) * (size_t)p->max_adapters;
  std::memcpy(c, p->pt_h, sizeof(int32_t) * (size_t)p->max_adapters * (size_t)p->pt_stride);
  *len = need;
  return SLORA_OK;
}

int slora_timing_enable(slora_pool* p, int32_t enable) {
  SLORA_RANGE("slora_timing_enable");
  if (int rc = check_device_pool(p)) return rc;
  p->timing = enable != 0;
  return SLORA_OK;
}

int slora_timing_read(slora_pool* p, int32_t capacity, const char** names, double* ms, int64_t* launches,
                      int32_t* n) {
  SLORA_RANGE("slora_timing_read");
  if (int rc = check_device_pool(p)) return rc;
  for (auto& r : p->recs) {
    CUDA_TRY(cudaEventSynchronize(r.b));
    float t = 0.f;
    CUDA_TRY(cudaEventElapsedTime(&t, r.a, r.b));
    p->t_ms[r.kind] += t;
    p->t_launches[r.kind] += 1;
    p->spare_events.push_back(r.a);
    p->spare_events.push_back(r.b);
  }
  p->recs.clear();
  const int k = std::min<int>(capacity, kTNum);
  for (int i = 0; i < k; ++i) {
    if (names) names[i] = kTimerNames[i];
    if (ms) ms[i] = p->t_ms[i];
    if (launches) launches[i] = p->t_launches[i];
  }
  for (int i = 0; i < kTNum; ++i) {
    p->t_ms[i] = 0;
    p->t_launches[i] = 0;
  }
  if (n) *n = k;
  return SLORA_OK;
}

int slora_set_tc_threshold(slora_pool* p, int32_t min_tokens) {
  SLORA_RANGE("slora_set_tc_threshold");
  if (int rc = check_pool(p)) return rc;
  if (min_tokens < 0) return fail(SLORA_ERR_INVALID, "threshold %d", min_tokens);
  if (p->tc_ok || p->planning) p->tc_threshold = min_tokens;
  return SLORA_OK;
}

int slora_debug_set_fault(slora_pool* p, int32_t kind, int64_t nth) {
  SLORA_RANGE("slora_debug_set_fault");
  if (int rc = check_pool(p)) return rc;
  if (kind < SLORA_FAULT_NONE || kind > SLORA_FAULT_COPY || nth < 0)
    return fail(SLORA_ERR_INVALID, "fault kind %d, count %lld", kind, (long long)nth);
  for (int64_t& f : p->fault_left) f = 0;
  if (kind != SLORA_FAULT_NONE) p->fault_left[kind] = nth;
  return SLORA_OK;
}

int slora_debug_poke_page_table(slora_pool* p, int64_t entry, int32_t value, int32_t* old) {
  SLORA_RANGE("slora_debug_poke_page_table");
  if (int rc = check_device_pool(p)) return rc;
#ifdef SLORA_DEBUG
  if (!old) return fail(SLORA_ERR_INVALID, "old is NULL");
  if (entry < 0 || entry >= (int64_t)p->max_adapters * p->pt_stride)
    return fail(SLORA_ERR_INVALID, "entry %lld outside the page table", (long long)entry);
  CUDA_TRY(cudaStreamSynchronize(p->compute));
  CUDA_TRY(cudaMemcpy(old, p->d_pt + entry, sizeof(int32_t), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemcpy(p->d_pt + entry, &value, sizeof(int32_t), cudaMemcpyHostToDevice));
  return SLORA_OK;
#else
  (void)entry;
  (void)value;
  (void)old;
  return fail(SLORA_ERR_INVALID, "slora_debug_poke_page_table exists only in the SLORA_DEBUG build");
#endif
}

int slora_debug_set_wait_limit(slora_pool* p, uint32_t polls) {
  SLORA_RANGE("slora_debug_set_wait_limit");
  if (int rc = check_pool(p)) return rc;
  p->wait_limit = polls;
  return SLORA_OK;
}

int slora_set_tc_min_batch(slora_pool* p, int32_t min_tokens) {
  SLORA_RANGE("slora_set_tc_min_batch");
  if (int rc = check_pool(p)) return rc;
  if (min_tokens < 0) return fail(SLORA_ERR_INVALID, "minimum batch %d", min_tokens);
  p->tc_min_batch = min_tokens;
  return SLORA_OK;
}

}  // extern "C"
