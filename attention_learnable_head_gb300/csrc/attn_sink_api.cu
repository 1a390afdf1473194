// Host side of libattn_sink.so: argument validation, TMA tensor-map encoding,
// launch configuration and workspace carving for the C ABI in attn_sink.h.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "attn_sink.h"
#include "bwd_dq_kernel.cuh"
#include "bwd_kernel.cuh"
#include "decode_kernel.cuh"
#include "fwd_band_kernel.cuh"
#include "fwd_kernel.cuh"
#include "merge_kernel.cuh"
#include "schedule_kernel.cuh"

// Device word a kernel sets when it gives up on a bounded wait.
__device__ int g_attn_sink_device_error = 0;

// Scratch of attn_sink_fwd_noalloc (the fp16 copy of v), one per device, held
// for the life of the process.  In host code this name is only a host-side
// stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_SINK_NOALLOC_SCRATCH_BYTES];

namespace {

using namespace attn_sink;

constexpr int kMaxDevices = 64;

// Kernels this library has launched in this process (successful launches).
std::atomic<unsigned long long> g_launches{0};

// The most recent CUDA error a call of this library ran into (0 = none).
std::atomic<int> g_last_cuda_error{0};

inline bool launched() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    g_last_cuda_error.store((int)e, std::memory_order_relaxed);
    return false;
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return true;
}

// Optional per-launch timing of the library's main kernels (attn_sink_kernel_timing):
// an event pair recorded on the launching stream around each launch, read back
// and summed by attn_sink_kernel_time.  Events are reused through a pool.
struct TimedLaunch {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_timing_mutex;
std::atomic<bool> g_timing_on{false};
std::vector<TimedLaunch> g_timing_pending;
std::vector<cudaEvent_t> g_timing_pool;
double g_timing_ms[ATTN_SINK_KERNEL_COUNT] = {0.0};
unsigned long long g_timing_count[ATTN_SINK_KERNEL_COUNT] = {0};

cudaEvent_t timing_event() {
  if (!g_timing_pool.empty()) {
    cudaEvent_t e = g_timing_pool.back();
    g_timing_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
}

// Records the start event of a timed launch; returns the pending record (or
// kernel = -1 when timing is off or no event could be had).
TimedLaunch timing_begin(int kernel, cudaStream_t s) {
  TimedLaunch t{-1, nullptr, nullptr};
  if (!g_timing_on.load(std::memory_order_relaxed)) return t;
  std::lock_guard<std::mutex> lock(g_timing_mutex);
  t.start = timing_event();
  t.stop = timing_event();
  if (t.start == nullptr || t.stop == nullptr || cudaEventRecord(t.start, s) != cudaSuccess) {
    if (t.start) g_timing_pool.push_back(t.start);
    if (t.stop) g_timing_pool.push_back(t.stop);
    return TimedLaunch{-1, nullptr, nullptr};
  }
  t.kernel = kernel;
  return t;
}

void timing_end(const TimedLaunch& t, cudaStream_t s, bool ok) {
  if (t.kernel < 0) return;
  std::lock_guard<std::mutex> lock(g_timing_mutex);
  if (ok && cudaEventRecord(t.stop, s) == cudaSuccess) {
    g_timing_pending.push_back(t);
  } else {
    g_timing_pool.push_back(t.start);
    g_timing_pool.push_back(t.stop);
  }
}

#ifdef ATTN_SINK_TEST_HOOKS
// Test build only: tiles the next launches withhold (see attn_sink_test_withhold).
std::atomic<int> g_test_skip_k_tile{-1};
std::atomic<int> g_test_skip_q_step{-1};
#endif

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

std::mutex g_dev_mutex;
int g_sm_count[kMaxDevices] = {0};
int* g_err_ptr[kMaxDevices] = {nullptr};
bool g_attr_set[kMaxDevices] = {false};

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Per-device state: SM count, address of the error word, kernel attributes.
int device_state(int* sm_count, int** err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return ATTN_SINK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return ATTN_SINK_ERR_CUDA;
    void* e = nullptr;
    if (cudaGetSymbolAddress(&e, g_attn_sink_device_error) != cudaSuccess)
      return ATTN_SINK_ERR_CUDA;
    g_sm_count[dev] = n;
    g_err_ptr[dev] = static_cast<int*>(e);
  }
  if (!g_attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_sink_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFwdSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(attn_sink_fwd_band_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBandSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(attn_sink_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kDqSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(attn_sink_bwd_main_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBwdSmemBytes) != cudaSuccess)
      return ATTN_SINK_ERR_CUDA;
    g_attr_set[dev] = true;
  }
  *sm_count = g_sm_count[dev];
  *err = g_err_ptr[dev];
  return ATTN_SINK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// An NVTX range around one entry point's host work (validation, tensor maps,
// launches), so that a profiler's timeline names the library's calls.  NVTX is
// header-only here: without a profiler attached a range costs a branch.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Problem geometry resolved from the params (dense or packed).
struct Geometry {
  bool varlen;
  int num_seqs;
  int total_q, total_k;
  int max_q, max_k;
  int group;
};

int validate(const attn_sink_params* p, const int* cu_q, const int* cu_k, Geometry* g) {
  if (p == nullptr) return ATTN_SINK_ERR_INVALID_ARG;
  if (p->head_dim != kHeadDim) return ATTN_SINK_ERR_UNSUPPORTED;
  if (p->heads_q <= 0 || p->heads_kv <= 0 || p->heads_q % p->heads_kv != 0)
    return ATTN_SINK_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return ATTN_SINK_ERR_INVALID_ARG;
  if (p->window > 0 && !p->causal) return ATTN_SINK_ERR_INVALID_ARG;
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale > 0.0f))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (p->grad_dtype != 0 && p->grad_dtype != 1) return ATTN_SINK_ERR_INVALID_ARG;
  if ((cu_q == nullptr) != (cu_k == nullptr)) return ATTN_SINK_ERR_INVALID_ARG;
  // One mode at a time: packed (cu_seqlens given, batch = 0) or dense (num_seqs = 0).
  if (cu_q == nullptr && p->num_seqs > 0) return ATTN_SINK_ERR_INVALID_ARG;
  if (cu_q != nullptr && p->batch > 0) return ATTN_SINK_ERR_INVALID_ARG;
  g->varlen = cu_q != nullptr;
  g->group = p->heads_q / p->heads_kv;
  if (g->varlen) {
    if (p->num_seqs < 0 || p->total_q < 0 || p->total_k < 0 || p->max_seqlen_q < 0 ||
        p->max_seqlen_k < 0)
      return ATTN_SINK_ERR_INVALID_ARG;
    if (p->num_seqs > 0 && (p->max_seqlen_q > p->total_q || p->max_seqlen_k > p->total_k))
      return ATTN_SINK_ERR_INVALID_ARG;
    g->num_seqs = p->num_seqs;
    g->total_q = p->total_q;
    g->total_k = p->total_k;
    g->max_q = p->max_seqlen_q;
    g->max_k = p->max_seqlen_k;
  } else {
    if (p->batch < 0 || p->seqlen_q < 0 || p->seqlen_k < 0) return ATTN_SINK_ERR_INVALID_ARG;
    const long long tq = (long long)p->batch * p->seqlen_q;
    const long long tk = (long long)p->batch * p->seqlen_k;
    if (tq > INT32_MAX || tk > INT32_MAX) return ATTN_SINK_ERR_INVALID_ARG;
    g->num_seqs = p->batch;
    g->total_q = (int)tq;
    g->total_k = (int)tk;
    g->max_q = p->seqlen_q;
    g->max_k = p->seqlen_k;
  }
  // Launch-grid limits (tiles in grid.y, sequences in grid.z).
  if (g->num_seqs > 65535) return ATTN_SINK_ERR_UNSUPPORTED;
  if ((g->max_q + kBlockM - 1) / kBlockM > 65535 || (g->max_k + kBlockN - 1) / kBlockN > 65535)
    return ATTN_SINK_ERR_UNSUPPORTED;
  return ATTN_SINK_OK;
}

// 3-D map over a [tokens][heads][64] tensor with a (128 bytes) x box_heads x
// box_rows box and 128-byte swizzle: 64 columns of a 16-bit type, or 32 of fp32.
int encode_rows(CUtensorMap* m, const void* ptr, long long tokens, int heads,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                int box_rows = kBlockM, int box_heads = 1) {
  if (!load_encode()) return ATTN_SINK_ERR_CUDA;
  const cuuint64_t esize = dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * esize, (cuuint64_t)heads * kHeadDim * esize};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, dtype, 3, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_SINK_OK : ATTN_SINK_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Entries of the tile-order table of a packed batch of several sequences
// (schedule_kernel.cuh; query tiles, or key tiles with by_keys): at least the
// number of 128-row tiles; 0 where the dense (tile, sequence) grid is used.
int order_slots(const Geometry& g, bool by_keys) {
  if (!g.varlen || g.num_seqs < 2) return 0;
  const long long total = by_keys ? g.total_k : g.total_q;
  const long long slots = (total + kBlockM - 1) / kBlockM + g.num_seqs;
  return slots <= 65535 ? (int)slots : 0;
}

// Launches the sort of a packed batch's tiles into `table` (see order_slots).
bool launch_order(const attn_sink_params* p, const Geometry& g, const int* cu_q,
                  const int* cu_k, bool by_keys, bool chunk, int q_pos0, int slots,
                  uint32_t* table, cudaStream_t stream) {
  SchedParams sp;
  sp.cu_q = cu_q;
  sp.cu_k = cu_k;
  sp.num_seqs = g.num_seqs;
  sp.causal = p->causal;
  sp.window = p->window > 0 ? p->window : 0;
  sp.chunk = chunk ? 1 : 0;
  sp.q_pos0 = chunk ? q_pos0 : 0;
  sp.by_keys = by_keys ? 1 : 0;
  sp.n_slots = slots;
  sp.table = table;
  attn_sink_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(sp);
  return launched();
}

// Forward workspace: the fp16 copy of v, then the tile-order table.
size_t fwd_v16_bytes(const attn_sink_params* p, const Geometry& g) {
  return align256((size_t)g.total_k * p->heads_kv * kHeadDim * 2);
}
size_t fwd_workspace_bytes(const attn_sink_params* p, const Geometry& g) {
  return fwd_v16_bytes(p, g) + align256((size_t)order_slots(g, false) * sizeof(uint32_t));
}

// How many CTAs share one (kv head, key tile) in the backward pass.  Splitting
// the GQA group shortens the longest CTA when there are too few key tiles to
// fill the GPU; the split partials are summed in a fixed order afterwards.  The
// group is split until the longest CTA carries no more steps than an SM's
// share of the total: every further split only adds per-CTA set-up and
// partial-sum traffic (measured on the 4096-token GPT-OSS layer: split 2 beats
// 1, 4 and 8).
int choose_split(const attn_sink_params* p, const Geometry& g, int sm_count) {
  const int qt = (g.max_q + kBlockM - 1) / kBlockM;
  const int kt = (g.max_k + kBlockN - 1) / kBlockN;
  if (qt == 0 || kt == 0 || g.num_seqs == 0) return 1;
  double total, longest;           // in units of (query head, query tile, key tile) steps
  int q_per_key;                   // query tiles a key tile meets at most
  if (p->causal && p->window > 0) {
    q_per_key = std::min(qt, (p->window + kBlockM - 1) / kBlockM + 1);
    total = (double)g.num_seqs * p->heads_q * qt * q_per_key;
  } else if (p->causal) {
    q_per_key = qt;
    total = (double)g.num_seqs * p->heads_q * qt * (kt + 1) * 0.5;
  } else {
    q_per_key = qt;
    total = (double)g.num_seqs * p->heads_q * qt * kt;
  }
  int split = 1;
  while (split < g.group && g.group % (split * 2) == 0) {
    longest = (double)(g.group / split) * q_per_key;
    if (longest * sm_count <= total) break;
    split *= 2;
  }
  return split;
}

struct BwdLayout {
  size_t off_D, off_part, off_dq, off_dk, off_dv, off_q16, off_do16, off_k16, off_v16, off_work,
      total;
  int slots;   // entries of the key-tile order table (0: dense grid)
  int n_blocks;
  int split;
};

BwdLayout bwd_layout(const attn_sink_params* p, const Geometry& g, int sm_count) {
  BwdLayout L;
  L.n_blocks = (g.total_q + kPreRows - 1) / kPreRows;
  L.split = choose_split(p, g, sm_count);
  size_t off = 0;
  L.off_D = off;
  off += align256((size_t)p->heads_q * g.total_q * sizeof(float2));
  L.off_part = off;
  off += align256((size_t)p->heads_q * std::max(L.n_blocks, 1) * sizeof(float));
  L.off_dq = off;
  if (p->grad_dtype == 0) off += align256((size_t)g.total_q * p->heads_q * kHeadDim * sizeof(float));
  const size_t kv_part = (size_t)L.split * g.total_k * p->heads_kv * kHeadDim * sizeof(float);
  L.off_dk = off;
  if (L.split > 1) off += align256(kv_part);
  L.off_dv = off;
  if (L.split > 1) off += align256(kv_part);
  const size_t q16 = (size_t)g.total_q * p->heads_q * kHeadDim * 2;
  const size_t k16 = (size_t)g.total_k * p->heads_kv * kHeadDim * 2;
  L.off_q16 = off;
  off += align256(q16);
  L.off_do16 = off;
  off += align256(q16);
  L.off_k16 = off;
  off += align256(k16);
  L.off_v16 = off;
  off += align256(k16);
  L.slots = order_slots(g, true);
  L.off_work = off;
  off += align256((size_t)L.slots * sizeof(uint32_t));
  L.total = off;
  return L;
}

int sm_count_or_default() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    return n;
  cudaGetLastError();
  return 148;
}

}  // namespace

extern "C" {

const char* attn_sink_status_string(int status) {
  switch (status) {
    case ATTN_SINK_OK: return "ok";
    case ATTN_SINK_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_SINK_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_SINK_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_SINK_ERR_CUDA: return "CUDA error";
    case ATTN_SINK_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

// The band kernel's launch (fwd_band_kernel.cuh): items of 128 / G tokens x the
// G query heads of a kv group, a window of n_cols keys each; persistent grid of
// two CTAs per SM.  v16 is the fp16 copy of v already written by the caller.
int fwd_band(const attn_sink_params* params, const Geometry& g, const void* q, const void* k,
             const void* v16, const void* sink, const int* cu_seqlens_q,
             const int* cu_seqlens_k, void* out, void* out_residual, float* lse, void* stream,
             bool chunk, int q_pos0, bool sink_bf16, int tokens, int n_cols, int sms, int* err) {
  FwdBandParams bp;
  std::memset(&bp, 0, sizeof(bp));
  int st;
  if ((st = encode_rows(&bp.tm_q, q, g.total_q, params->heads_q,
                        CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tokens, g.group)) != ATTN_SINK_OK)
    return st;
  if ((st = encode_rows(&bp.tm_k, k, g.total_k, params->heads_kv,
                        CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n_cols)) != ATTN_SINK_OK)
    return st;
  if ((st = encode_rows(&bp.tm_v, v16, g.total_k, params->heads_kv,
                        CU_TENSOR_MAP_DATA_TYPE_FLOAT16, n_cols)) != ATTN_SINK_OK)
    return st;
  if ((st = encode_rows(&bp.tm_out, out, g.total_q, params->heads_q,
                        CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tokens, g.group)) != ATTN_SINK_OK)
    return st;
  if ((st = encode_rows(&bp.tm_out_lo, out_residual ? out_residual : out, g.total_q,
                        params->heads_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tokens, g.group)) !=
      ATTN_SINK_OK)
    return st;
  const long long n_tb = (g.max_q + tokens - 1) / tokens;
  const long long n_items = (long long)g.num_seqs * n_tb * params->heads_kv;
  if (n_items >= (1ll << 30)) return ATTN_SINK_ERR_UNSUPPORTED;
  if (n_items == 0) return ATTN_SINK_OK;
  bp.cu_q = cu_seqlens_q;
  bp.cu_k = cu_seqlens_k;
  bp.sink = sink_bf16 ? nullptr : static_cast<const float*>(sink);
  bp.sink_bf16 = sink_bf16 ? static_cast<const __nv_bfloat16*>(sink) : nullptr;
  bp.out = static_cast<__nv_bfloat16*>(out);
  bp.out_lo = static_cast<__nv_bfloat16*>(out_residual);
  bp.lse = lse;
  bp.err = err;
  bp.seqlen_q = g.varlen ? 0 : params->seqlen_q;
  bp.seqlen_k = g.varlen ? 0 : params->seqlen_k;
  bp.total_q = g.total_q;
  bp.heads_q = params->heads_q;
  bp.heads_kv = params->heads_kv;
  bp.group = g.group;
  bp.log2_group = 0;
  while ((1 << bp.log2_group) < g.group) ++bp.log2_group;
  bp.tokens = tokens;
  bp.n_cols = n_cols;
  bp.half0_cols = 16 * ((n_cols / 16 + 1) / 2);
  bp.window = params->window;
  bp.scale_log2 = params->softmax_scale * kLog2e;
  bp.chunk = chunk ? 1 : 0;
  bp.q_pos0 = chunk ? q_pos0 : 0;
  bp.n_tb = (int)n_tb;
  bp.n_items = (int)n_items;
  fast_div_init(params->heads_kv, &bp.div_hkv_mul, &bp.div_hkv_shift);
  fast_div_init(bp.n_tb, &bp.div_tb_mul, &bp.div_tb_shift);
#ifdef ATTN_SINK_TEST_HOOKS
  bp.skip_k_tile = g_test_skip_k_tile.load();
#endif
  // At least 80 KB, so that no SM holds a third CTA (two fill its 512 TMEM
  // columns; a third would wait in its allocation until one of them ends).
  const int smem = std::max(80 * 1024, band_smem_bytes(n_cols));
  const int grid = (int)std::min<long long>(n_items, (long long)kBandCtasPerSm * sms);
  const TimedLaunch t = timing_begin(ATTN_SINK_KERNEL_FWD, static_cast<cudaStream_t>(stream));
  attn_sink_fwd_band_kernel<<<grid, kBandThreads, smem, static_cast<cudaStream_t>(stream)>>>(bp);
  const bool ok = launched();
  timing_end(t, static_cast<cudaStream_t>(stream), ok);
  return ok ? ATTN_SINK_OK : ATTN_SINK_ERR_CUDA;
}

// The forward, with or without the sink; `chunk` selects key-chunk mode (no
// sink, query row i at key position i + q_pos0 in every sequence).
int fwd_impl(const attn_sink_params* params, const void* q, const void* k, const void* v,
             const void* sink, const int* cu_seqlens_q, const int* cu_seqlens_k, void* out,
             void* out_residual, float* lse, void* workspace, size_t workspace_bytes,
             void* stream, bool chunk, int q_pos0, bool sink_bf16) {
  NvtxRange range(chunk ? "attn_sink_fwd_chunk" : "attn_sink_fwd");
  Geometry g;
  int st = validate(params, cu_seqlens_q, cu_seqlens_k, &g);
  if (st != ATTN_SINK_OK) return st;
  if (g.num_seqs == 0 || g.total_q == 0) return ATTN_SINK_OK;   // nothing to compute
  const size_t ws_bytes = fwd_workspace_bytes(params, g);
  if (ws_bytes > 0 && (workspace == nullptr || workspace_bytes < ws_bytes ||
                       (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return ATTN_SINK_ERR_WORKSPACE;
  if (q == nullptr || (!chunk && sink == nullptr) || out == nullptr || lse == nullptr)
    return ATTN_SINK_ERR_INVALID_ARG;
  if (g.total_k > 0 && (k == nullptr || v == nullptr)) return ATTN_SINK_ERR_INVALID_ARG;
  if (chunk && (q_pos0 > (1 << 30) || q_pos0 < -(1 << 30))) return ATTN_SINK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(out_residual))
    return ATTN_SINK_ERR_INVALID_ARG;
  int sms = 0;
  int* err = nullptr;
  if ((st = device_state(&sms, &err)) != ATTN_SINK_OK) return st;

  FwdParams fp;
  std::memset(&fp, 0, sizeof(fp));
  // An empty key tensor is never read (every tile has no key); its map only
  // needs a valid address.
  const void* kp = g.total_k > 0 ? k : q;
  const void* vp = g.total_k > 0 ? workspace : q;
  const int tk = g.total_k > 0 ? g.total_k : 1;
  const int hk = g.total_k > 0 ? params->heads_kv : 1;
  if ((st = encode_rows(&fp.tm_q, q, g.total_q, params->heads_q)) != ATTN_SINK_OK) return st;
  if ((st = encode_rows(&fp.tm_k, kp, tk, hk)) != ATTN_SINK_OK) return st;
  if ((st = encode_rows(&fp.tm_v, vp, tk, hk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != ATTN_SINK_OK)
    return st;
  if ((st = encode_rows(&fp.tm_out, out, g.total_q, params->heads_q)) != ATTN_SINK_OK ||
      (st = encode_rows(&fp.tm_out_lo, out_residual ? out_residual : out, g.total_q,
                        params->heads_q)) != ATTN_SINK_OK)
    return st;
  if (g.total_k > 0) {
    // fp16 copy of v for the P V products
    const size_t n8 = (size_t)g.total_k * params->heads_kv * kHeadDim / 8;
    const int blocks = (int)std::min<size_t>((n8 + 255) / 256, (size_t)sms * 8);
    attn_sink_convert_f16_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(v), static_cast<uint16_t*>(workspace), n8, err);
    if (!launched()) return ATTN_SINK_ERR_CUDA;
  }
  // Sliding-window layers whose item window (128 / G tokens + W - 1 keys) fits
  // one product go to the band kernel.
  const int band_tokens = (kBlockM % g.group == 0) ? kBlockM / g.group : 0;
  const long long band_cols =
      band_tokens > 0 ? ((long long)band_tokens + params->window - 1 + 15) / 16 * 16 : 0;
  if (params->causal && params->window > 0 && g.total_k > 0 && band_tokens > 0 &&
      band_cols <= kBandMaxCols)
    return fwd_band(params, g, q, k, workspace, sink, cu_seqlens_q, cu_seqlens_k, out,
                    out_residual, lse, stream, chunk, q_pos0, sink_bf16, band_tokens,
                    (int)band_cols, sms, err);
  fp.cu_q = cu_seqlens_q;
  fp.cu_k = cu_seqlens_k;
  fp.sink = sink_bf16 ? nullptr : static_cast<const float*>(sink);
  fp.sink_bf16 = sink_bf16 ? static_cast<const __nv_bfloat16*>(sink) : nullptr;
  fp.out = static_cast<__nv_bfloat16*>(out);
  fp.out_lo = static_cast<__nv_bfloat16*>(out_residual);
  fp.lse = lse;
  fp.err = err;
  fp.seqlen_q = g.varlen ? 0 : params->seqlen_q;
  fp.seqlen_k = g.varlen ? 0 : params->seqlen_k;
  fp.total_q = g.total_q;
  fp.heads_q = params->heads_q;
  fp.group = g.group;
  fp.causal = params->causal;
  fp.window = params->window > 0 ? params->window : 0;
  fp.scale_log2 = params->softmax_scale * kLog2e;
  fp.chunk = chunk ? 1 : 0;
  fp.q_pos0 = chunk ? q_pos0 : 0;
  fp.n_qtiles = (g.max_q + kBlockM - 1) / kBlockM;
#ifdef ATTN_SINK_TEST_HOOKS
  fp.skip_k_tile = g_test_skip_k_tile.load();
#endif
  if (fp.n_qtiles == 0) return ATTN_SINK_OK;
  dim3 grid(params->heads_q, fp.n_qtiles, g.num_seqs);
  const int slots = order_slots(g, false);
  if (slots > 0) {
    uint32_t* table =
        reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + fwd_v16_bytes(params, g));
    if (!launch_order(params, g, cu_seqlens_q, cu_seqlens_k, false, chunk, q_pos0, slots, table,
                      static_cast<cudaStream_t>(stream)))
      return ATTN_SINK_ERR_CUDA;
    fp.work = table;
    grid = dim3(params->heads_q, slots, 1);
  }
  const TimedLaunch t = timing_begin(ATTN_SINK_KERNEL_FWD, static_cast<cudaStream_t>(stream));
  attn_sink_fwd_kernel<<<grid, kFwdThreads, kFwdSmemBytes, static_cast<cudaStream_t>(stream)>>>(fp);
  const bool ok = launched();
  timing_end(t, static_cast<cudaStream_t>(stream), ok);
  return ok ? ATTN_SINK_OK : ATTN_SINK_ERR_CUDA;
}

}  // namespace

extern "C" {

int attn_sink_fwd(const attn_sink_params* params, const void* q, const void* k, const void* v,
                  const float* sink, const int* cu_seqlens_q, const int* cu_seqlens_k,
                  void* out, void* out_residual, float* lse, void* workspace,
                  size_t workspace_bytes, void* stream) {
  return fwd_impl(params, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                  workspace, workspace_bytes, stream, false, 0, false);
}

int attn_sink_fwd_ex(const attn_sink_params* params, int flags, const void* q, const void* k,
                     const void* v, const void* sink, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, void* out, void* out_residual, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if ((flags & ~ATTN_SINK_FLAG_SINK_BF16) != 0) return ATTN_SINK_ERR_INVALID_ARG;
  return fwd_impl(params, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                  workspace, workspace_bytes, stream, false, 0,
                  (flags & ATTN_SINK_FLAG_SINK_BF16) != 0);
}

int attn_sink_fwd_chunk(const attn_sink_params* params, int q_pos0, const void* q,
                        const void* k, const void* v, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, void* out, void* out_residual, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(params, q, k, v, nullptr, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                  workspace, workspace_bytes, stream, true, q_pos0, false);
}

int attn_sink_merge(int num_chunks, int total_q, int heads_q, int head_dim, const void* o_parts,
                    const void* o_residual_parts, const float* lse_parts, const float* sink,
                    void* out, void* out_residual, float* lse, void* stream) {
  NvtxRange range("attn_sink_merge");
  if (num_chunks < 1 || total_q < 0 || heads_q < 1) return ATTN_SINK_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return ATTN_SINK_ERR_UNSUPPORTED;
  if (total_q == 0) return ATTN_SINK_OK;
  if (o_parts == nullptr || lse_parts == nullptr || sink == nullptr || out == nullptr ||
      lse == nullptr)
    return ATTN_SINK_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o_residual_parts) || !aligned16(out) ||
      !aligned16(out_residual))
    return ATTN_SINK_ERR_INVALID_ARG;
  int sms = 0;
  int* err = nullptr;
  int st;
  if ((st = device_state(&sms, &err)) != ATTN_SINK_OK) return st;
  MergeParams mp;
  mp.o_parts = static_cast<const __nv_bfloat16*>(o_parts);
  mp.res_parts = static_cast<const __nv_bfloat16*>(o_residual_parts);
  mp.lse_parts = lse_parts;
  mp.sink = sink;
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.out_lo = static_cast<__nv_bfloat16*>(out_residual);
  mp.lse = lse;
  mp.num_chunks = num_chunks;
  mp.total_q = total_q;
  mp.heads_q = heads_q;
  const size_t pairs = (size_t)total_q * heads_q;
  const int blocks = (int)std::min<size_t>((pairs + 31) / 32, (size_t)sms * 8);
  const TimedLaunch t = timing_begin(ATTN_SINK_KERNEL_MERGE, static_cast<cudaStream_t>(stream));
  attn_sink_merge_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(mp);
  const bool ok = launched();
  timing_end(t, static_cast<cudaStream_t>(stream), ok);
  return ok ? ATTN_SINK_OK : ATTN_SINK_ERR_CUDA;
}

}  // extern "C"

namespace {

// query heads per kv head that the decode kernel is built for
bool decode_group_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

struct DecodeLayout {
  int splits;
  size_t off_lo, off_lse, off_done, total;
};

// Key splits: enough (batch x kv head x split) CTAs for about eight waves of
// the five decode CTAs an SM holds at once (fewer waves leave a part-filled
// last wave and too few copies in flight: measured, 40 x SMs beat 2, 8 and 20
// x SMs), each split at least 256 keys of the longest possible sequence, at
// most 64.
bool decode_layout(const attn_sink_decode_params* p, int sm_count, DecodeLayout* L) {
  if (p == nullptr || p->batch < 0 || p->heads_kv < 1 || p->heads_q < 1 ||
      p->heads_q % p->heads_kv != 0 || !decode_group_ok(p->heads_q / p->heads_kv) ||
      p->page_size < 1 || p->num_pages < 0 || p->max_pages < 0 ||
      !(p->softmax_scale > 0.0f) || !std::isfinite(p->softmax_scale))
    return false;
  const long long cap = (long long)p->max_pages * p->page_size;
  if (cap > (1ll << 30)) return false;
  const long long ctas = (long long)p->batch * p->heads_kv;
  const long long keys = (p->window > 0) ? std::min<long long>(cap, p->window) : cap;
  long long s = 1;
  if (ctas > 0) s = std::max<long long>(1, (40ll * sm_count + ctas - 1) / ctas);
  s = std::min<long long>(s, std::max<long long>(1, (keys + 255) / 256));
  s = std::min<long long>(s, 64);
  L->splits = (int)s;
  const size_t o = (size_t)s * p->batch * p->heads_q * 64 * 2;   // bf16
  L->off_lo = align256(o);
  L->off_lse = L->off_lo + align256(o);
  L->off_done = L->off_lse + align256((size_t)s * p->heads_q * p->batch * sizeof(float));
  L->total = L->off_done + align256((size_t)p->batch * p->heads_kv * sizeof(int));
  return true;
}

}  // namespace

extern "C" {

size_t attn_sink_decode_workspace_size(const attn_sink_decode_params* params) {
  DecodeLayout L;
  if (params == nullptr || params->head_dim != kHeadDim || params->batch == 0 ||
      params->batch > 65535 || params->heads_kv > 65535 ||
      !decode_layout(params, sm_count_or_default(), &L))
    return 0;
  return L.total;
}

int attn_sink_decode(const attn_sink_decode_params* params, const void* q, const void* k_cache,
                     const void* v_cache, const int* block_table, const int* seq_lens,
                     const float* sink, void* out, void* out_residual, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange range("attn_sink_decode");
  if (params == nullptr) return ATTN_SINK_ERR_INVALID_ARG;
  if (params->head_dim != kHeadDim) return ATTN_SINK_ERR_UNSUPPORTED;
  // launch-grid limits: kv heads in grid.y, sequences in grid.z
  if (params->batch > 65535 || params->heads_kv > 65535) return ATTN_SINK_ERR_UNSUPPORTED;
  DecodeLayout L;
  if (!decode_layout(params, sm_count_or_default(), &L)) {
    if (params->heads_kv >= 1 && params->heads_q >= 1 &&
        params->heads_q % params->heads_kv == 0 &&
        !decode_group_ok(params->heads_q / params->heads_kv))
      return ATTN_SINK_ERR_UNSUPPORTED;
    return ATTN_SINK_ERR_INVALID_ARG;
  }
  if (params->batch == 0) return ATTN_SINK_OK;
  if (q == nullptr || sink == nullptr || out == nullptr || lse == nullptr ||
      seq_lens == nullptr || (params->max_pages > 0 && block_table == nullptr) ||
      (params->num_pages > 0 && (k_cache == nullptr || v_cache == nullptr)))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(out_residual))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return ATTN_SINK_ERR_WORKSPACE;
  int sms = 0;
  int* err = nullptr;
  int st;
  if ((st = device_state(&sms, &err)) != ATTN_SINK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams dp;
  dp.q = static_cast<const __nv_bfloat16*>(q);
  dp.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  dp.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  dp.block_table = block_table;
  dp.seq_lens = seq_lens;
  dp.o_part = reinterpret_cast<__nv_bfloat16*>(ws);
  dp.o_part_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.off_lo);
  dp.lse_part = reinterpret_cast<float*>(ws + L.off_lse);
  dp.done = reinterpret_cast<int*>(ws + L.off_done);
  dp.sink = sink;
  dp.out = static_cast<__nv_bfloat16*>(out);
  dp.out_lo = static_cast<__nv_bfloat16*>(out_residual);
  dp.lse = lse;
  dp.err = err;
  dp.batch = params->batch;
  dp.heads_q = params->heads_q;
  dp.heads_kv = params->heads_kv;
  dp.page_size = params->page_size;
  dp.num_pages = params->num_pages;
  dp.max_pages = params->max_pages;
  dp.window = params->window > 0 ? params->window : 0;
  dp.splits = L.splits;
  dp.scale_log2 = params->softmax_scale * kLog2e;
  // Whole pages by TMA for power-of-two page sizes of 8 keys or more (and a
  // pool whose rows fit the copy coordinates); per-thread copies otherwise.
  const long long rows = (long long)params->num_pages * params->page_size;
  const bool tma = decode_tma_page(params->page_size) && rows > 0 && rows < (1ll << 31);
  dp.log2_page = 0;
  while ((1 << dp.log2_page) < params->page_size) ++dp.log2_page;
  if (tma) {
    const int box = std::min(params->page_size, kDecKeys);
    if ((st = encode_rows(&dp.tm_k, k_cache, rows, params->heads_kv,
                          CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, box)) != ATTN_SINK_OK ||
        (st = encode_rows(&dp.tm_v, v_cache, rows, params->heads_kv,
                          CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, box)) != ATTN_SINK_OK)
      return st;
  }
  // the per-(sequence, kv head) completion counters start at zero
  if (cudaMemsetAsync(dp.done, 0, (size_t)params->batch * params->heads_kv * sizeof(int), s) !=
      cudaSuccess)
    return ATTN_SINK_ERR_CUDA;
  const dim3 grid(L.splits, params->heads_kv, params->batch);
  switch ((params->heads_q / params->heads_kv) * 2 + (tma ? 1 : 0)) {
    case 2: attn_sink_decode_kernel<1, false><<<grid, kDecThreads, 0, s>>>(dp); break;
    case 3: attn_sink_decode_kernel<1, true><<<grid, kDecThreads, 0, s>>>(dp); break;
    case 4: attn_sink_decode_kernel<2, false><<<grid, kDecThreads, 0, s>>>(dp); break;
    case 5: attn_sink_decode_kernel<2, true><<<grid, kDecThreads, 0, s>>>(dp); break;
    case 8: attn_sink_decode_kernel<4, false><<<grid, kDecThreads, 0, s>>>(dp); break;
    case 9: attn_sink_decode_kernel<4, true><<<grid, kDecThreads, 0, s>>>(dp); break;
    case 16: attn_sink_decode_kernel<8, false><<<grid, kDecThreads, 0, s>>>(dp); break;
    default: attn_sink_decode_kernel<8, true><<<grid, kDecThreads, 0, s>>>(dp); break;
  }
  return launched() ? ATTN_SINK_OK : ATTN_SINK_ERR_CUDA;
}

size_t attn_sink_fwd_workspace_size(const attn_sink_params* params) {
  if (params == nullptr) return 0;
  static const int kMarker = 0;
  const bool packed = params->num_seqs > 0;
  Geometry g;
  if (validate(params, packed ? &kMarker : nullptr, packed ? &kMarker : nullptr, &g) !=
      ATTN_SINK_OK)
    return 0;
  return fwd_workspace_bytes(params, g);
}

size_t attn_sink_bwd_workspace_size(const attn_sink_params* params) {
  if (params == nullptr) return 0;
  // Packed fields are used when num_seqs > 0, the dense fields otherwise.
  static const int kMarker = 0;
  const bool packed = params->num_seqs > 0;
  Geometry g;
  if (validate(params, packed ? &kMarker : nullptr, packed ? &kMarker : nullptr, &g) !=
      ATTN_SINK_OK)
    return 0;
  return bwd_layout(params, g, sm_count_or_default()).total;
}

}  // extern "C"

namespace {

// The backward; `deterministic` computes dQ with the query-stationary kernel
// (fixed summation order) instead of reduce-adds from the main kernel.
int bwd_impl(const attn_sink_params* params, const void* q, const void* k, const void* v,
             const void* sink, const int* cu_seqlens_q, const int* cu_seqlens_k,
             const void* out, const void* out_residual, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, void* dsink, void* workspace,
             size_t workspace_bytes, void* stream, int flags) {
  const bool deterministic = (flags & ATTN_SINK_FLAG_DETERMINISTIC) != 0;
  NvtxRange range(deterministic ? "attn_sink_bwd_deterministic" : "attn_sink_bwd");
  const bool sink_bf16 = (flags & ATTN_SINK_FLAG_SINK_BF16) != 0;
  const bool accumulate = (flags & ATTN_SINK_FLAG_ACCUMULATE_DSINK) != 0;
  Geometry g;
  int st = validate(params, cu_seqlens_q, cu_seqlens_k, &g);
  if (st != ATTN_SINK_OK) return st;
  if (sink == nullptr || dsink == nullptr) return ATTN_SINK_ERR_INVALID_ARG;
  if (g.total_q > 0 && (q == nullptr || out == nullptr || lse == nullptr || dout == nullptr ||
                        dq == nullptr))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (g.total_k > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(out_residual))
    return ATTN_SINK_ERR_INVALID_ARG;
  int sms = 0;
  int* err = nullptr;
  if ((st = device_state(&sms, &err)) != ATTN_SINK_OK) return st;
  const BwdLayout L = bwd_layout(params, g, sms);
  if (L.total > 0 && (workspace == nullptr || workspace_bytes < L.total ||
                      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return ATTN_SINK_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float2* LD = reinterpret_cast<float2*>(ws + L.off_D);
  float* partials = reinterpret_cast<float*>(ws + L.off_part);
  float* dq_acc = params->grad_dtype == 1 ? static_cast<float*>(dq)
                                          : reinterpret_cast<float*>(ws + L.off_dq);
  const float scale = params->softmax_scale;
  uint16_t* q16 = reinterpret_cast<uint16_t*>(ws + L.off_q16);
  uint16_t* do16 = reinterpret_cast<uint16_t*>(ws + L.off_do16);
  uint16_t* k16 = reinterpret_cast<uint16_t*>(ws + L.off_k16);
  uint16_t* v16 = reinterpret_cast<uint16_t*>(ws + L.off_v16);

  // 1. D, dsink partials, fp16 operand copies, zero the dq accumulator
  if (g.total_q > 0) {
    PreParams pp;
    pp.q = static_cast<const __nv_bfloat16*>(q);
    pp.out_lo = static_cast<const __nv_bfloat16*>(out_residual);
    pp.q16 = q16;
    pp.do16 = do16;
    pp.err = err;
    pp.out = static_cast<const __nv_bfloat16*>(out);
    pp.dout = static_cast<const __nv_bfloat16*>(dout);
    pp.lse = lse;
    pp.sink = sink_bf16 ? nullptr : static_cast<const float*>(sink);
    pp.sink_bf16 = sink_bf16 ? static_cast<const __nv_bfloat16*>(sink) : nullptr;
    pp.LD = LD;
    pp.partials = partials;
    pp.dq_acc = deterministic ? nullptr : dq_acc;
    pp.total_q = g.total_q;
    pp.heads_q = params->heads_q;
    pp.n_blocks = L.n_blocks;
    attn_sink_bwd_pre_kernel<<<dim3(L.n_blocks, params->heads_q), 256, 0, s>>>(pp);
    if (!launched()) return ATTN_SINK_ERR_CUDA;
  }
  if (g.total_k > 0) {
    const size_t n8 = (size_t)g.total_k * params->heads_kv * kHeadDim / 8;
    const int blocks = (int)std::min<size_t>((n8 + 255) / 256, (size_t)sms * 8);
    attn_sink_kv_convert_kernel<<<blocks, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), k16, v16, n8,
        err);
    if (!launched()) return ATTN_SINK_ERR_CUDA;
  }
  // 2. main loop: dK, dV (and their split partials), dQ accumulation
  const int n_ktiles = (g.max_k + kBlockN - 1) / kBlockN;
  if (g.total_k > 0 && g.num_seqs > 0 && n_ktiles > 0) {
    BwdParams bp;
    std::memset(&bp, 0, sizeof(bp));
    // An empty query tensor is never read (no key tile has a query); its maps
    // only need a valid address.
    const void* qp = g.total_q > 0 ? (const void*)q16 : (const void*)k16;
    const void* op = g.total_q > 0 ? (const void*)do16 : (const void*)k16;
    const int tq = g.total_q > 0 ? g.total_q : 1;
    const int hq = g.total_q > 0 ? params->heads_q : 1;
    const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if ((st = encode_rows(&bp.tm_q, qp, tq, hq, f16)) != ATTN_SINK_OK) return st;
    if ((st = encode_rows(&bp.tm_do, op, tq, hq, f16)) != ATTN_SINK_OK) return st;
    if ((st = encode_rows(&bp.tm_k, k16, g.total_k, params->heads_kv, f16)) != ATTN_SINK_OK)
      return st;
    if ((st = encode_rows(&bp.tm_v, v16, g.total_k, params->heads_kv, f16)) != ATTN_SINK_OK)
      return st;
    const void* dqp = g.total_q > 0 ? (const void*)dq_acc : (const void*)k16;
    if ((st = encode_rows(&bp.tm_dq, dqp, tq, hq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)) !=
        ATTN_SINK_OK)
      return st;
    bp.cu_q = cu_seqlens_q;
    bp.cu_k = cu_seqlens_k;
    bp.LD = LD;
    bp.dq_acc = dq_acc;
    bp.dk = dk;
    bp.dv = dv;
    bp.dk_part = reinterpret_cast<float*>(ws + L.off_dk);
    bp.dv_part = reinterpret_cast<float*>(ws + L.off_dv);
    bp.err = err;
    bp.seqlen_q = g.varlen ? 0 : params->seqlen_q;
    bp.seqlen_k = g.varlen ? 0 : params->seqlen_k;
    bp.total_q = g.total_q;
    bp.total_k = g.total_k;
    bp.heads_q = params->heads_q;
    bp.heads_kv = params->heads_kv;
    bp.group = g.group;
    bp.split = L.split;
    bp.causal = params->causal;
    bp.window = params->window > 0 ? params->window : 0;
    bp.scale = scale;
    bp.scale_log2 = scale * kLog2e;
    bp.n_ktiles = n_ktiles;
    bp.grad_fp32 = params->grad_dtype;
    bp.skip_dq = deterministic ? 1 : 0;
#ifdef ATTN_SINK_TEST_HOOKS
    bp.skip_q_step = g_test_skip_q_step.load();
#endif
    dim3 grid(params->heads_kv * L.split, n_ktiles, g.num_seqs);
    if (L.slots > 0) {
      uint32_t* table = reinterpret_cast<uint32_t*>(ws + L.off_work);
      if (!launch_order(params, g, cu_seqlens_q, cu_seqlens_k, true, false, 0, L.slots, table, s))
        return ATTN_SINK_ERR_CUDA;
      bp.work = table;
      grid = dim3(params->heads_kv * L.split, L.slots, 1);
    }
    const TimedLaunch t = timing_begin(ATTN_SINK_KERNEL_BWD_MAIN, s);
    attn_sink_bwd_main_kernel<<<grid, kBwdThreads, kBwdSmemBytes, s>>>(bp);
    const bool ok = launched();
    timing_end(t, s, ok);
    if (!ok) return ATTN_SINK_ERR_CUDA;
    if (L.split > 1) {
      const size_t n4 = (size_t)g.total_k * params->heads_kv * kHeadDim / 4;
      const int blocks = (int)std::min<size_t>((n4 + 255) / 256, (size_t)sms * 8);
      attn_sink_dkdv_reduce_kernel<<<blocks, 256, 0, s>>>(bp.dk_part, bp.dv_part, L.split, n4,
                                                          scale, dk, dv, params->grad_dtype);
      if (!launched()) return ATTN_SINK_ERR_CUDA;
    }
  }
  // 3. deterministic dQ, written directly in the requested dtype
  if (deterministic && g.total_q > 0 && g.num_seqs > 0) {
    const int n_qtiles = (g.max_q + kBlockM - 1) / kBlockM;
    DqParams dp;
    std::memset(&dp, 0, sizeof(dp));
    const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // An empty key tensor is never read (every tile has no key); its maps only
    // need a valid address.
    const void* kp = g.total_k > 0 ? (const void*)k16 : (const void*)q16;
    const void* vp = g.total_k > 0 ? (const void*)v16 : (const void*)q16;
    const int tk = g.total_k > 0 ? g.total_k : 1;
    const int hk = g.total_k > 0 ? params->heads_kv : 1;
    if ((st = encode_rows(&dp.tm_q, q16, g.total_q, params->heads_q, f16)) != ATTN_SINK_OK)
      return st;
    if ((st = encode_rows(&dp.tm_do, do16, g.total_q, params->heads_q, f16)) != ATTN_SINK_OK)
      return st;
    // K and V come in steps of kDqKeys keys
    if ((st = encode_rows(&dp.tm_k, kp, tk, hk, f16, kDqKeys)) != ATTN_SINK_OK) return st;
    if ((st = encode_rows(&dp.tm_v, vp, tk, hk, f16, kDqKeys)) != ATTN_SINK_OK) return st;
    dp.cu_q = cu_seqlens_q;
    dp.cu_k = cu_seqlens_k;
    dp.LD = LD;
    dp.dq = dq;
    dp.err = err;
    dp.seqlen_q = g.varlen ? 0 : params->seqlen_q;
    dp.seqlen_k = g.varlen ? 0 : params->seqlen_k;
    dp.total_q = g.total_q;
    dp.heads_q = params->heads_q;
    dp.group = g.group;
    dp.causal = params->causal;
    dp.window = params->window > 0 ? params->window : 0;
    dp.scale = scale;
    dp.scale_log2 = scale * kLog2e;
    dp.n_qtiles = n_qtiles;
    dp.grad_fp32 = params->grad_dtype;
    const TimedLaunch t = timing_begin(ATTN_SINK_KERNEL_BWD_DQ, s);
    attn_sink_bwd_dq_kernel<<<dim3(params->heads_q, g.num_seqs, n_qtiles), kDqThreads,
                              kDqSmemBytes, s>>>(dp);
    const bool ok = launched();
    timing_end(t, s, ok);
    if (!ok) return ATTN_SINK_ERR_CUDA;
  }
  // 3'. dq (bf16) from the fp32 accumulator
  if (!deterministic && g.total_q > 0 && params->grad_dtype == 0) {
    const size_t n8 = (size_t)g.total_q * params->heads_q * kHeadDim / 8;
    const int blocks = (int)std::min<size_t>((n8 + 255) / 256, (size_t)sms * 8);
    attn_sink_dq_convert_kernel<<<blocks, 256, 0, s>>>(dq_acc, static_cast<__nv_bfloat16*>(dq),
                                                       n8);
    if (!launched()) return ATTN_SINK_ERR_CUDA;
  }
  // 4. dsink
  if (g.total_q > 0) {
    attn_sink_dsink_reduce_kernel<<<params->heads_q, 256, 0, s>>>(
        partials, L.n_blocks, dsink, sink_bf16 ? 1 : 0, accumulate ? 1 : 0);
    return launched() ? ATTN_SINK_OK : ATTN_SINK_ERR_CUDA;
  }
  // no query row: the gradient is zero (nothing to add when accumulating)
  if (!accumulate && cudaMemsetAsync(dsink, 0, (sink_bf16 ? 2 : 4) * (size_t)params->heads_q,
                                     s) != cudaSuccess)
    return ATTN_SINK_ERR_CUDA;
  return ATTN_SINK_OK;
}

}  // namespace

extern "C" {

int attn_sink_bwd(const attn_sink_params* params, const void* q, const void* k, const void* v,
                  const float* sink, const int* cu_seqlens_q, const int* cu_seqlens_k,
                  const void* out, const void* out_residual, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, float* dsink,
                  void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(params, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                  dout, dq, dk, dv, dsink, workspace, workspace_bytes, stream, 0);
}

int attn_sink_bwd_deterministic(const attn_sink_params* params, const void* q, const void* k,
                                const void* v, const float* sink, const int* cu_seqlens_q,
                                const int* cu_seqlens_k, const void* out,
                                const void* out_residual, const float* lse, const void* dout,
                                void* dq, void* dk, void* dv, float* dsink, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return bwd_impl(params, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                  dout, dq, dk, dv, dsink, workspace, workspace_bytes, stream,
                  ATTN_SINK_FLAG_DETERMINISTIC);
}

int attn_sink_bwd_ex(const attn_sink_params* params, int flags, const void* q, const void* k,
                     const void* v, const void* sink, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, const void* out, const void* out_residual,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     void* dsink, void* workspace, size_t workspace_bytes, void* stream) {
  if ((flags & ~(ATTN_SINK_FLAG_SINK_BF16 | ATTN_SINK_FLAG_ACCUMULATE_DSINK |
                 ATTN_SINK_FLAG_DETERMINISTIC)) != 0)
    return ATTN_SINK_ERR_INVALID_ARG;
  return bwd_impl(params, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                  dout, dq, dk, dv, dsink, workspace, workspace_bytes, stream, flags);
}

// Caller entry point that allocates nothing: the workspace of attn_sink_fwd is
// the static device array above.  Per device, the array's device address is
// looked up once (with that device current) and cached.
int attn_sink_fwd_noalloc(const attn_sink_params* params, const void* q, const void* k,
                          const void* v, const float* sink, const int* cu_seqlens_q,
                          const int* cu_seqlens_k, void* out, void* out_residual, float* lse,
                          void* stream) {
  static std::mutex scratch_mutex;
  static void* scratch_ptr[kMaxDevices] = {nullptr};
  if (params == nullptr) return ATTN_SINK_ERR_INVALID_ARG;
  const bool packed = params->num_seqs > 0;
  Geometry g;
  const int st = validate(params, packed ? cu_seqlens_q : nullptr,
                          packed ? cu_seqlens_k : nullptr, &g);
  if (st != ATTN_SINK_OK) return st;
  // Too large for the static scratch: a clear error, nothing launched.
  if (fwd_workspace_bytes(params, g) > (size_t)ATTN_SINK_NOALLOC_SCRATCH_BYTES)
    return ATTN_SINK_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return ATTN_SINK_ERR_CUDA;
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(scratch_mutex);
    if (scratch_ptr[dev] == nullptr) {
      void* a = nullptr;
      if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || a == nullptr)
        return ATTN_SINK_ERR_CUDA;
      scratch_ptr[dev] = a;
    }
    ptr = scratch_ptr[dev];
  }
  return attn_sink_fwd(params, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                       ptr, (size_t)ATTN_SINK_NOALLOC_SCRATCH_BYTES, stream);
}

#ifdef ATTN_SINK_TEST_HOOKS
// Test build only (not in attn_sink.h): from the next launch on, the forward's
// producer withholds K tile `fwd_k_tile` of every CTA and the backward's
// producer the Q/dO tiles of step `bwd_q_step` (-1: none), so that the waits
// for them run out and the bounded-wait path returns an error code.
int attn_sink_test_withhold(int fwd_k_tile, int bwd_q_step) {
  g_test_skip_k_tile.store(fwd_k_tile);
  g_test_skip_q_step.store(bwd_q_step);
  return ATTN_SINK_OK;
}
#endif

int attn_sink_kernel_timing(int on) {
  g_timing_on.store(on != 0, std::memory_order_relaxed);
  return ATTN_SINK_OK;
}

int attn_sink_kernel_time(int kernel, double* total_ms, unsigned long long* launches) {
  if (kernel < 0 || kernel >= ATTN_SINK_KERNEL_COUNT || total_ms == nullptr || launches == nullptr)
    return ATTN_SINK_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_timing_mutex);
  int status = ATTN_SINK_OK;
  for (const TimedLaunch& t : g_timing_pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(t.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, t.start, t.stop) == cudaSuccess) {
      g_timing_ms[t.kernel] += ms;
      g_timing_count[t.kernel] += 1;
    } else {
      status = ATTN_SINK_ERR_CUDA;
    }
    g_timing_pool.push_back(t.start);
    g_timing_pool.push_back(t.stop);
  }
  g_timing_pending.clear();
  *total_ms = g_timing_ms[kernel];
  *launches = g_timing_count[kernel];
  g_timing_ms[kernel] = 0.0;
  g_timing_count[kernel] = 0;
  return status;
}

int attn_sink_last_cuda_error(void) { return g_last_cuda_error.load(std::memory_order_relaxed); }

unsigned long long attn_sink_launch_count(void) {
  return g_launches.load(std::memory_order_relaxed);
}

int attn_sink_device_error(void* stream, int* code) {
  if (code == nullptr) return ATTN_SINK_ERR_INVALID_ARG;
  *code = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_SINK_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_sink_device_error, sizeof(int)) != cudaSuccess)
    return ATTN_SINK_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_attn_sink_device_error, &zero, sizeof(int)) != cudaSuccess)
      return ATTN_SINK_ERR_CUDA;
  }
  *code = v;
  // a kernel that gave up on a bounded wait (0x1xx forward, 0x2xx backward)
  const int kind = v & 0xF00;
  return (kind == DEVERR_TIMEOUT_FWD || kind == DEVERR_TIMEOUT_BWD) ? ATTN_SINK_ERR_TIMEOUT
                                                                   : ATTN_SINK_OK;
}

}  // extern "C"
