// C ABI of the fused linear selected-token log-probability: argument checks,
// workspace layout, tensor-memory-copy descriptors and the launch sequence.
// Declarations and the contract are in include/linear_logp.h.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "fused_logp.h"
#include "linear_logp.h"
#include "llp_internal.h"
#include "sm103_ptx.cuh"

// Code of the last failed CUDA call made by this library on the calling thread,
// the last failed driver call's result, and the source line of the check that
// turned a failure into LLP_ERR_CUDA.
thread_local int g_last_cuda_error = 0;
thread_local int g_last_driver_result = 0;
thread_local int g_last_failure_line = 0;

int fail_cuda(int line) {
  g_last_failure_line = line;
  return LLP_ERR_CUDA;
}

namespace llp {
cudaError_t note_cuda(cudaError_t e) {
  if (e != cudaSuccess) g_last_cuda_error = static_cast<int>(e);
  return e;
}
}  // namespace llp

namespace {

// Kernel status word: a kernel that gives up on a bounded wait records why here.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceInit {
  bool done = false;
  int status = LLP_OK;
  int num_sms = 0;
  unsigned int* status_ptr = nullptr;
  llp::LaunchCaps caps = {};
};

std::mutex g_mu;
DeviceInit g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;

// Tensor-map encoding is a driver call and needs a current context on the
// calling thread.  A thread whose only CUDA work so far went through an
// allocator's cache (an autograd worker, say) may have none yet: bind the
// current device's primary context then (cudaSetDevice does, since CUDA 12),
// and leave a context the caller made current alone.
int ensure_context(int dev) {
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  CUcontext ctx = nullptr;
  if (g_ctx_get_current != nullptr && g_ctx_get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr) return LLP_OK;
  return llp::note_cuda(cudaSetDevice(dev)) == cudaSuccess ? LLP_OK : fail_cuda(__LINE__);
}

int load_encode_fn() {
  static std::once_flag once;
  static int st = LLP_OK;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
      st = fail_cuda(__LINE__);
    } else {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  });
  return st;
}

// Per-device one-time set-up with that device current: architecture check,
// shared-memory opt-in for every kernel, SM count, status-word address.
int init_device(DeviceInit** out) {
  // A pending, non-sticky error left on this thread by an earlier, unrelated
  // CUDA call would otherwise be read back after our first launch and taken
  // for this call's failure; a sticky (context) error persists and is reported.
  (void)cudaGetLastError();
  int dev = 0;
  if (llp::note_cuda(cudaGetDevice(&dev)) != cudaSuccess) return fail_cuda(__LINE__);
  if (dev < 0 || dev >= kMaxDevices) return LLP_ERR_UNSUPPORTED_DEVICE;
  if (ensure_context(dev) != LLP_OK) return LLP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInit& d = g_dev[dev];
  if (!d.done) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return fail_cuda(__LINE__);
    }
    if (major != 10 || minor != 3) {
      d.status = LLP_ERR_UNSUPPORTED_DEVICE;
    } else if (llp::fwd_setup(&d.caps) != cudaSuccess || llp::bwd_setup(&d.caps) != cudaSuccess ||
               llp::small_grad_hidden_setup() != cudaSuccess ||
               cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status_ptr), g_status_word) != cudaSuccess) {
      d.status = fail_cuda(__LINE__);
    } else {
      d.status = LLP_OK;
    }
    d.num_sms = sms;
    d.done = true;
  }
  *out = &d;
  return d.status;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

constexpr int64_t kLim31 = (int64_t(1) << 31) - 1;
constexpr int64_t kLim62 = int64_t(1) << 62;

bool product_ok(int64_t a, int64_t b) { return a == 0 || b <= kLim62 / a; }

int check_shapes(int64_t N, int64_t D, int64_t V) {
  if (N < 0 || D < 1 || V < 1 || (D % 8) != 0) return LLP_ERR_BAD_SHAPE;
  if (N > kLim31 || D > kLim31 || V > kLim31) return LLP_ERR_BAD_SHAPE;
  if (!product_ok(N, D) || !product_ok(V, D) || !product_ok(N, round_up(V, 64))) return LLP_ERR_BAD_SHAPE;
  // every work-unit count and tile index must fit a 32-bit int
  const int64_t num_m = cdiv(N, llp::kUnitM);
  const int64_t num_vt = cdiv(V, llp::kTileN);
  const int64_t num_d = cdiv(D, llp::kTileN);
  if (num_m * num_vt > kLim31) return LLP_ERR_BAD_SHAPE;
  if (cdiv(V, llp::kKSegment) * num_m * num_d > kLim31) return LLP_ERR_BAD_SHAPE;
  if (cdiv(N, llp::kKSegment) * cdiv(V, llp::kUnitM) * num_d > kLim31) return LLP_ERR_BAD_SHAPE;
  return LLP_OK;
}

int check_inputs(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                 const float* temperature, int64_t N, int64_t D, int64_t V) {
  if (hidden == nullptr || weight == nullptr || targets == nullptr) return LLP_ERR_NULL_POINTER;
  const int s = check_shapes(N, D, V);
  if (s != LLP_OK) return s;
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(targets, 8)) return LLP_ERR_MISALIGNED;
  if (bias != nullptr && !aligned(bias, 4)) return LLP_ERR_MISALIGNED;
  if (temperature != nullptr && !aligned(temperature, 4)) return LLP_ERR_MISALIGNED;
  return LLP_OK;
}

// Workspace carving: each region starts on a 256-byte boundary from the base.
struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  }
};

struct FwdLayout {
  size_t part_m, part_s, zt, total;
};

FwdLayout fwd_layout(int64_t N, int64_t V) {
  const size_t S = static_cast<size_t>(cdiv(V, llp::kSplitWidth));
  Carver c;
  FwdLayout L;
  L.part_m = c.take(S * N * sizeof(float));
  L.part_s = c.take(S * N * sizeof(float));
  L.zt = c.take(N * sizeof(float));
  L.total = c.off;
  return L;
}

struct BwdLayout {
  size_t sched, dz, gb_part, dh_part, dw_part, total;
  bool has_gb, has_dh, has_dw;
};

BwdLayout bwd_layout(int64_t N, int64_t D, int64_t V, bool bias, bool want_dh, bool want_dw) {
  const size_t V_pad = round_up(static_cast<size_t>(V), 64);
  const size_t num_m = static_cast<size_t>(cdiv(N, llp::kUnitM));
  const size_t nseg_v = static_cast<size_t>(cdiv(V, llp::kKSegment));
  const size_t nseg_n = static_cast<size_t>(cdiv(N, llp::kKSegment));
  Carver c;
  BwdLayout L;
  L.sched = c.take(llp::kNumSchedCounters * sizeof(int));
  L.dz = c.take(static_cast<size_t>(N) * V_pad * 2);
  L.has_gb = bias;
  L.gb_part = bias ? c.take(num_m * (llp::kUnitM / 32) * static_cast<size_t>(V) * sizeof(float)) : 0;
  L.has_dh = want_dh && nseg_v > 1;
  L.dh_part = L.has_dh ? c.take(nseg_v * static_cast<size_t>(N) * D * sizeof(float)) : 0;
  L.has_dw = want_dw && nseg_n > 1;
  L.dw_part = L.has_dw ? c.take(nseg_n * static_cast<size_t>(V) * D * sizeof(float)) : 0;
  L.total = c.off;
  return L;
}

// 2-D map of a 16-bit matrix: bf16, or IEEE fp16 when f16.
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
             uint32_t box_inner, uint32_t box_outer, bool f16 = false) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                              const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) g_last_driver_result = static_cast<int>(r);
  return r == CUDA_SUCCESS ? LLP_OK : fail_cuda(__LINE__);
}

// 3-D map of a row-major 16-bit matrix [rows][cols] (row pitch pitch_bytes) seen
// as its 64-column chunks: {64, rows, cols / 64} with strides {pitch, 128 B}.  A
// box {64, box_rows, box_chunks} lands in shared memory as box_chunks 2-D
// {64, box_rows} boxes back to back.  cols must be a multiple of 64 (chunks never
// straddle a row end).
int make_map_chunked(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch_bytes,
                     uint32_t box_rows, uint32_t box_chunks, bool f16) {
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {pitch_bytes, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                              const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) g_last_driver_result = static_cast<int>(r);
  return r == CUDA_SUCCESS ? LLP_OK : fail_cuda(__LINE__);
}

// Output map of fp32 segment partials [nseg][rows][cols], box {32, 32, 1}:
// a store clips at `rows` inside each segment.
int make_map_part(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t nseg) {
  cuuint64_t dims[3] = {cols, rows, nseg};
  cuuint64_t strides[2] = {cols * 4, rows * cols * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) g_last_driver_result = static_cast<int>(r);
  return r == CUDA_SUCCESS ? LLP_OK : fail_cuda(__LINE__);
}

// Output map of a gradient [rows][D] (bf16) or of its segment partials.
int make_map_grad_out(CUtensorMap* m, const llp::GradGemmParams& p) {
  if (p.nseg == 1 && !p.f32_out)
    return make_map(m, p.out, p.D, p.rows, static_cast<uint64_t>(p.D) * 2, 64, 32, p.f16 != 0);
  return make_map_part(m, p.part, p.D, p.rows, p.nseg);
}

// ----------------------------------------------------------------------------
// Optional launch recorder (see linear_logp_profile_start in the header).
// ----------------------------------------------------------------------------
enum KernelId {
  kKFwdPartials = 0,
  kKFwdMerge,
  kKDlogits,
  kKGradHidden,
  kKGradWeight,
  kKSegSumHidden,
  kKSegSumWeight,
  kKBiasSum,
  kKNumKernels
};

const char* const kKernelNames[kKNumKernels] = {"fwd_partials",  "fwd_merge",          "dlogits",
                                                "grad_hidden",   "grad_weight",        "segment_sum_hidden",
                                                "segment_sum_weight", "bias_sum"};

struct Recorder {
  std::mutex mu;
  bool on = false;
  int launch_cap = 0;
  int launches = 0;
  int used = 0;
  std::vector<cudaEvent_t> events;
  std::vector<int> ids;  // -1: call start; otherwise the kernel id launched just before
};

Recorder g_rec;

void rec_mark(cudaStream_t s, int id) {
  if (!g_rec.on) return;
  std::lock_guard<std::mutex> lock(g_rec.mu);
  if (!g_rec.on || g_rec.used >= static_cast<int>(g_rec.events.size())) return;
  if (id >= 0) {
    if (g_rec.launches >= g_rec.launch_cap) return;
    ++g_rec.launches;
  }
  cudaEventRecord(g_rec.events[g_rec.used], s);
  g_rec.ids[g_rec.used] = id;
  ++g_rec.used;
}

// Row tiling of the two token-row GEMMs (forward logits, dlogits) for a batch of
// N rows.  A batch that fits in one 128-row tile runs on single CTAs: in a CTA
// pair the second CTA's 128 rows would all be padding, and single CTAs put
// every SM on the weight stream.  Both tilings accumulate every element over the
// same 16-deep K steps in the same order (cta_group::1 M=128 or cta_group::2
// M=256 instructions), and a row's results are bitwise the same under both.
struct RowTiling {
  bool single;
  int unit_rows;   // rows per unit: kTileM single, kUnitM pair
  int w_box_rows;  // rows of a weight tile each CTA loads
};
RowTiling row_tiling(int64_t N) {
  const bool single = N <= llp::kTileM;
  return {single, single ? llp::kTileM : llp::kUnitM, single ? llp::kTileN : llp::kBRows};
}

// K-blocks per pipeline stage of the forward / dlogits GEMMs: two (one 3-D copy
// per operand per stage) on CTA pairs when the hidden size is whole 64-column
// chunks.  The single-CTA tiling of small batches streams the weight from HBM
// and keeps one-k-block stages: with 128-row hidden boxes two double stages
// would leave only one in flight while the MMAs read the other, and with
// 32-row boxes three double stages ran no faster than six single ones.
int k_blocks_per_stage(int64_t D, bool single) { return ((LLP_KPS2 & 1) && !single && (D % 64) == 0) ? 2 : 1; }

// Tensor maps of the two K-major operands of the forward / dlogits GEMMs, the
// hidden states (box rows kTileM) and the weight (box rows w_box_rows): 2-D with
// a 64-wide K box, or, with kps == 2, 3-D over 64-column K chunks, two chunks per box.
int make_kmajor_maps(CUtensorMap* tm_h, CUtensorMap* tm_w, const void* hidden, const void* weight, int64_t N,
                     int64_t D, int64_t V, int w_box_rows, int kps, bool f16, int h_box_rows = llp::kTileM) {
  if (kps == 2) {
    if (make_map_chunked(tm_h, hidden, D, N, D * 2, h_box_rows, 2, f16) != LLP_OK) return LLP_ERR_CUDA;
    return make_map_chunked(tm_w, weight, D, V, D * 2, w_box_rows, 2, f16);
  }
  if (make_map(tm_h, hidden, D, N, D * 2, llp::kTileK, h_box_rows, f16) != LLP_OK) return LLP_ERR_CUDA;
  return make_map(tm_w, weight, D, V, D * 2, llp::kTileK, w_box_rows, f16);
}

// Forward launch sequence on validated arguments (N > 0, workspace sized by fwd_layout).
// With sh_max set, `weight` is a vocab shard whose row 0 is global id vocab_start,
// and the shard's (max, sum, target logit) triple is written instead of logp / lse.
int fwd_core(DeviceInit* dev, const void* hidden, const void* weight, const float* bias, const int64_t* targets,
             const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index, float* out_logp,
             float* out_lse, uint8_t* ws, cudaStream_t s, int64_t vocab_start = 0, float* sh_max = nullptr,
             float* sh_se = nullptr, float* sh_tl = nullptr, bool f16 = false) {
  const FwdLayout L = fwd_layout(N, V);
  const RowTiling T = row_tiling(N);
  CUtensorMap tm_h, tm_w;
  const int kps = k_blocks_per_stage(D, T.single);
  if (make_kmajor_maps(&tm_h, &tm_w, hidden, weight, N, D, V, T.w_box_rows, kps, f16,
                       llp::hidden_box_rows(N, T.single)) != LLP_OK)
    return fail_cuda(__LINE__);
  llp::FwdParams p;
  p.N = static_cast<int>(N);
  p.D = static_cast<int>(D);
  p.V = static_cast<int>(V);
  p.num_m = static_cast<int>(cdiv(N, T.unit_rows));
  p.num_vt = static_cast<int>(cdiv(V, llp::kTileN));
  p.num_splits = static_cast<int>(cdiv(V, llp::kSplitWidth));
  p.group_m = llp::kGroupM;
  p.bias = bias;
  p.targets = reinterpret_cast<const long long*>(targets);
  p.temperature = temperature;
  p.ignore_index = ignore_index;
  p.part_m = reinterpret_cast<float*>(ws + L.part_m);
  p.part_s = reinterpret_cast<float*>(ws + L.part_s);
  p.zt = reinterpret_cast<float*>(ws + L.zt);
  p.err = dev->status_ptr;
  p.vocab_start = vocab_start;
  p.global_V = V;
  p.f16 = f16 ? 1 : 0;
  p.kps = kps;
  const int64_t units = static_cast<int64_t>(p.num_m) * p.num_splits;
  rec_mark(s, -1);
  if (llp::launch_fwd_partials(tm_h, tm_w, p, units, dev->caps, s, T.single) != cudaSuccess) return fail_cuda(__LINE__);
  rec_mark(s, kKFwdPartials);
  if (sh_max != nullptr) {
    if (llp::launch_shard_stats(p, sh_max, sh_se, sh_tl, s) != cudaSuccess) return fail_cuda(__LINE__);
  } else {
    if (llp::launch_fwd_merge(p, out_logp, out_lse, s) != cudaSuccess) return fail_cuda(__LINE__);
  }
  rec_mark(s, kKFwdMerge);
  return LLP_OK;
}

// LINEAR_LOGP_SCHEDULE=static (read once per process) makes every GEMM take its
// units round-robin.  A diagnostic: results are the same under either schedule.
bool force_static_schedule() {
  static const bool v = [] {
    const char* e = std::getenv("LINEAR_LOGP_SCHEDULE");
    return e != nullptr && std::strcmp(e, "static") == 0;
  }();
  return v;
}

// LINEAR_LOGP_SMALL_GRAD_HIDDEN=0 (read once per process) sends batches of at
// most kSmallGhMaxN rows through the CTA-pair grad_hidden GEMM instead of the
// swapped-operand kernel.  A diagnostic: both give the same results.
bool use_small_grad_hidden() {
  static const bool v = [] {
    const char* e = std::getenv("LINEAR_LOGP_SMALL_GRAD_HIDDEN");
    return LLP_SMALL_GH != 0 && !(e != nullptr && std::strcmp(e, "0") == 0);
  }();
  return v;
}

// K-blocks of a gradient GEMM's longest unit (a full K segment, or all of K
// when it is shorter).  The long units carry the work and the L2 reuse that
// in-order claiming protects; a short last segment rides along.
int64_t max_unit_kblocks(const llp::GradGemmParams& p) {
  const int64_t total = cdiv(p.K, llp::kTileK);
  return total < p.kseg_blocks ? total : p.kseg_blocks;
}

// Backward launch sequence on validated arguments (N > 0, workspace sized by bwd_layout).
// For a vocab shard: `weight` starts at global id vocab_start, targets are valid
// against global_V, and grad_hidden_f32 (fp32 [N, D]) receives this shard's
// contribution dz_local . W_local instead of a bf16 grad_hidden.
int bwd_core(DeviceInit* dev, const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
             const float* bias, const int64_t* targets, const float* temperature, int64_t N, int64_t D, int64_t V,
             int64_t ignore_index, void* grad_hidden, void* grad_weight, float* grad_bias, uint8_t* ws,
             cudaStream_t s, int64_t vocab_start = 0, int64_t global_V = -1, float* grad_hidden_f32 = nullptr,
             bool f16 = false) {
  if (global_V < 0) global_V = V;
  const bool want_gb = grad_bias != nullptr;
  const bool want_gh = grad_hidden != nullptr || grad_hidden_f32 != nullptr;
  const BwdLayout L = bwd_layout(N, D, V, bias != nullptr, want_gh, grad_weight != nullptr);
  const int64_t V_pad = static_cast<int64_t>(round_up(static_cast<size_t>(V), 64));
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(ws + L.dz);
  int* sched = reinterpret_cast<int*>(ws + L.sched);  // zeroed by the dlogits kernel

  // B1: dlogits (+ grad_bias partials)
  const RowTiling T = row_tiling(N);
  {
    CUtensorMap tm_h, tm_w;
    const int kps = k_blocks_per_stage(D, T.single);
    if (make_kmajor_maps(&tm_h, &tm_w, hidden, weight, N, D, V, T.w_box_rows, kps, f16,
                         llp::hidden_box_rows(N, T.single)) != LLP_OK)
      return fail_cuda(__LINE__);
    llp::DzParams p;
    p.N = static_cast<int>(N);
    p.D = static_cast<int>(D);
    p.V = static_cast<int>(V);
    p.V_pad = static_cast<int>(V_pad);
    p.num_m = static_cast<int>(cdiv(N, T.unit_rows));
    p.num_vt = static_cast<int>(cdiv(V, llp::kTileN));
    p.group_m = llp::kGroupM;
    p.bias = bias;
    p.targets = reinterpret_cast<const long long*>(targets);
    p.temperature = temperature;
    p.ignore_index = ignore_index;
    p.grad_logp = grad_logp;
    p.lse = saved_lse;
    p.dz = dz;
    p.gb_part = want_gb ? reinterpret_cast<float*>(ws + L.gb_part) : nullptr;
    p.err = dev->status_ptr;
    p.vocab_start = vocab_start;
    p.global_V = global_V;
    p.sched_reset = sched;
    p.f16 = f16 ? 1 : 0;
    p.kps = kps;
    const int64_t units = static_cast<int64_t>(p.num_m) * p.num_vt;
    rec_mark(s, -1);
    // dz [N][V_pad], written in 64 x 32 slabs; the columns [V, V_pad) of the last
    // slab are zeros, so readers may treat every row as V_pad long
    CUtensorMap tm_dz_out;
    if (make_map(&tm_dz_out, dz, V_pad, N, V_pad * 2, 64, 32, f16) != LLP_OK) return fail_cuda(__LINE__);
    if (llp::launch_dlogits(tm_h, tm_w, tm_dz_out, p, units, dev->caps, s, T.single) != cudaSuccess)
      return fail_cuda(__LINE__);
    rec_mark(s, kKDlogits);
  }

  // B2: grad_hidden = dz . W over fixed vocab segments
  if (want_gh) {
    const int nseg = static_cast<int>(cdiv(V, llp::kKSegment));
    const bool f32_out = grad_hidden_f32 != nullptr;
    // fp32 segment partials, or (one segment) a shard's fp32 contribution written directly
    float* part = L.has_dh ? reinterpret_cast<float*>(ws + L.dh_part) : (f32_out ? grad_hidden_f32 : nullptr);
    llp::GhSmallParams sp;
    if (use_small_grad_hidden() && llp::small_grad_hidden_plan(static_cast<int>(N), &sp)) {
      // a batch of at most kSmallGhMaxN rows: tokens on the MMA's N side, weight streamed in tall boxes
      CUtensorMap tm_w_rows, tm_dz_tok;
      sp.w_chunked = (D % 128) == 0 ? 1 : 0;
      if (sp.w_chunked) {
        if (make_map_chunked(&tm_w_rows, weight, D, V, D * 2, llp::kSmallGhRows, 2, f16) != LLP_OK)
          return fail_cuda(__LINE__);
      } else if (make_map(&tm_w_rows, weight, D, V, D * 2, 64, llp::kSmallGhRows, f16) != LLP_OK) {
        return fail_cuda(__LINE__);
      }
      // dz's padding columns [V, V_pad) are zero (written by the dlogits kernel)
      if (make_map_chunked(&tm_dz_tok, dz, V_pad, N, V_pad * 2, sp.BN, llp::kSmallGhRows / 64 * sp.b_span, f16) !=
          LLP_OK)
        return fail_cuda(__LINE__);
      sp.D = static_cast<int>(D);
      sp.V = static_cast<int>(V);
      sp.nseg = nseg;
      sp.num_dt = static_cast<int>(cdiv(D, 128));
      sp.part = part;
      sp.out = static_cast<__nv_bfloat16*>(grad_hidden);
      sp.f16 = f16 ? 1 : 0;
      sp.err = dev->status_ptr;
      if (llp::launch_small_grad_hidden(tm_w_rows, tm_dz_tok, sp, dev->num_sms, s) != cudaSuccess)
        return fail_cuda(__LINE__);
    } else {
      CUtensorMap tm_dz, tm_w_mn;
      const bool w_chunked = LLP_CHUNKED_MN && !LLP_HALF_TILE && (D % 64) == 0;  // half tiles load one chunk
      // dz rows are V_pad long with zero padding columns: whole 64-column K chunks
      const int kps = ((LLP_KPS2 & 2) && w_chunked) ? 2 : 1;
      if (kps == 2) {
        if (make_map_chunked(&tm_dz, dz, V_pad, N, V_pad * 2, llp::kTileM, 2, f16) != LLP_OK)
          return fail_cuda(__LINE__);
      } else if (make_map(&tm_dz, dz, V, N, V_pad * 2, llp::kTileK, llp::kTileM, f16) != LLP_OK) {
        return fail_cuda(__LINE__);
      }
      if (w_chunked) {
        if (make_map_chunked(&tm_w_mn, weight, D, V, D * 2, llp::kTileK * kps, llp::kBRows / 64, f16) != LLP_OK)
          return fail_cuda(__LINE__);
      } else if (make_map(&tm_w_mn, weight, D, V, D * 2, 64, llp::kTileK, f16) != LLP_OK) {
        return fail_cuda(__LINE__);
      }
      llp::GradGemmParams p;
      p.a_chunked = 0;
      p.b_chunked = w_chunked ? 1 : 0;
      p.kps = kps;
      p.rows = static_cast<int>(N);
      p.D = static_cast<int>(D);
      p.K = static_cast<int>(V);
      p.num_m = static_cast<int>(cdiv(N, llp::kUnitM));
      p.num_d = static_cast<int>(cdiv(D, llp::kTileN));
      p.nseg = nseg;
      p.kseg_blocks = llp::kKSegment / llp::kTileK;
      p.out = static_cast<__nv_bfloat16*>(grad_hidden);
      p.part = part;
      p.err = dev->status_ptr;
      p.f32_out = f32_out ? 1 : 0;
      p.f16 = f16 ? 1 : 0;
      p.sched = !force_static_schedule() && max_unit_kblocks(p) >= llp::kDynMinKBlocks ? sched + 0 : nullptr;
      p.progress = (LLP_LOCKSTEP > 0 && (LLP_LOCKSTEP_MASK & 1) && p.sched != nullptr)
                       ? reinterpret_cast<unsigned int*>(sched + 2)
                       : nullptr;
      const int64_t units = static_cast<int64_t>(p.nseg) * p.num_m * p.num_d;
      CUtensorMap tm_out;
      if (make_map_grad_out(&tm_out, p) != LLP_OK) return fail_cuda(__LINE__);
      if (llp::launch_grad_hidden(tm_dz, tm_w_mn, tm_out, p, units, dev->caps, s) != cudaSuccess)
        return fail_cuda(__LINE__);
    }
    rec_mark(s, kKGradHidden);
    if (nseg > 1) {
      const cudaError_t e =
          f32_out ? llp::launch_segment_sum_f32(part, nseg, static_cast<long long>(N) * D, grad_hidden_f32,
                                                dev->num_sms, s)
                  : llp::launch_segment_sum(part, nseg, static_cast<long long>(N) * D,
                                            static_cast<__nv_bfloat16*>(grad_hidden), dev->num_sms, s, f16 ? 1 : 0);
      if (e != cudaSuccess) return fail_cuda(__LINE__);
      rec_mark(s, kKSegSumHidden);
    }
  }

  // B3: grad_weight = dz^T . h over fixed token segments
  if (grad_weight != nullptr) {
    CUtensorMap tm_dz_mn, tm_h_mn;
    // dz rows are V_pad long with zero padding columns: whole 64-column chunks
    const bool dz_chunked = LLP_CHUNKED_MN != 0;
    const bool h_chunked = LLP_CHUNKED_MN && !LLP_HALF_TILE && (D % 64) == 0;
    // a unit's K is at most one token segment: with few tokens the second
    // k-block of a stage would mostly be padding
    const int kps = ((LLP_KPS2 & 4) && dz_chunked && h_chunked && N >= 1024) ? 2 : 1;
    if (dz_chunked) {
      if (make_map_chunked(&tm_dz_mn, dz, V_pad, N, V_pad * 2, llp::kTileK * kps, llp::kTileM / 64, f16) != LLP_OK)
        return fail_cuda(__LINE__);
    } else if (make_map(&tm_dz_mn, dz, V, N, V_pad * 2, 64, llp::kTileK, f16) != LLP_OK) {
      return fail_cuda(__LINE__);
    }
    if (h_chunked) {
      if (make_map_chunked(&tm_h_mn, hidden, D, N, D * 2, llp::kTileK * kps, llp::kBRows / 64, f16) != LLP_OK)
        return fail_cuda(__LINE__);
    } else if (make_map(&tm_h_mn, hidden, D, N, D * 2, 64, llp::kTileK, f16) != LLP_OK) {
      return fail_cuda(__LINE__);
    }
    llp::GradGemmParams p;
    p.a_chunked = dz_chunked ? 1 : 0;
    p.b_chunked = h_chunked ? 1 : 0;
    p.kps = kps;
    p.rows = static_cast<int>(V);
    p.D = static_cast<int>(D);
    p.K = static_cast<int>(N);
    p.num_m = static_cast<int>(cdiv(V, llp::kUnitM));
    p.num_d = static_cast<int>(cdiv(D, llp::kTileN));
    p.nseg = static_cast<int>(cdiv(N, llp::kKSegment));
    p.kseg_blocks = llp::kKSegment / llp::kTileK;
    p.out = static_cast<__nv_bfloat16*>(grad_weight);
    p.part = L.has_dw ? reinterpret_cast<float*>(ws + L.dw_part) : nullptr;
    p.f32_out = 0;
    p.f16 = f16 ? 1 : 0;
    p.err = dev->status_ptr;
    p.sched = !force_static_schedule() && max_unit_kblocks(p) >= llp::kDynMinKBlocks ? sched + 1 : nullptr;
    p.progress = (LLP_LOCKSTEP > 0 && (LLP_LOCKSTEP_MASK & 2) && p.sched != nullptr)
                     ? reinterpret_cast<unsigned int*>(sched + 3)
                     : nullptr;
    const int64_t units = static_cast<int64_t>(p.nseg) * p.num_m * p.num_d;
    CUtensorMap tm_out;
    if (make_map_grad_out(&tm_out, p) != LLP_OK) return fail_cuda(__LINE__);
    if (llp::launch_grad_weight(tm_dz_mn, tm_h_mn, tm_out, p, units, dev->caps, s) != cudaSuccess)
      return fail_cuda(__LINE__);
    rec_mark(s, kKGradWeight);
    if (p.nseg > 1) {
      if (llp::launch_segment_sum(p.part, p.nseg, static_cast<long long>(V) * D, p.out, dev->num_sms, s, p.f16) !=
          cudaSuccess)
        return fail_cuda(__LINE__);
      rec_mark(s, kKSegSumWeight);
    }
  }

  // B4: grad_bias
  if (want_gb) {
    // the 32-row blocks the dlogits units covered (padding rows give zero sums)
    const int nblocks = static_cast<int>(cdiv(N, T.unit_rows) * (T.unit_rows / 32));
    if (llp::launch_bias_sum(reinterpret_cast<const float*>(ws + L.gb_part), nblocks, static_cast<int>(V), grad_bias,
                             s) != cudaSuccess)
      return fail_cuda(__LINE__);
    rec_mark(s, kKBiasSum);
  }
  return LLP_OK;
}


}  // namespace

extern "C" {

size_t linear_logp_fwd_workspace_bytes(int64_t N, int64_t D, int64_t V) {
  if (N <= 0 || check_shapes(N, D, V) != LLP_OK) return 0;
  return fwd_layout(N, V).total;
}

size_t linear_logp_bwd_workspace_bytes(int64_t N, int64_t D, int64_t V, int has_bias) {
  if (N <= 0 || check_shapes(N, D, V) != LLP_OK) return 0;
  return bwd_layout(N, D, V, has_bias != 0, true, true).total;
}

const char* linear_logp_status_string(int status) {
  switch (status) {
    case LLP_OK: return "ok";
    case LLP_ERR_NULL_POINTER: return "a required pointer is NULL";
    case LLP_ERR_BAD_SHAPE: return "unsupported shape (need N >= 0, D >= 1, V >= 1, D % 8 == 0, sizes in range)";
    case LLP_ERR_MISALIGNED: return "misaligned pointer";
    case LLP_ERR_UNSUPPORTED_DEVICE: return "current device is not an sm_103 GPU";
    case LLP_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case LLP_ERR_CUDA: return "CUDA call or kernel launch failed";
    case LLP_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
    case LLP_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than linear_logp_fwd_noalloc's fixed 16 MiB array holds";
    default: return "unknown status";
  }
}

// hidden / weight are bf16, or IEEE fp16 when f16.
static int fwd_entry(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                     const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                     float* out_logp, float* out_lse, void* workspace, size_t workspace_bytes, void* stream, bool f16) {
  int st = check_shapes(N, D, V);
  if (st != LLP_OK) return st;
  if (N == 0) return LLP_OK;  // nothing to compute; per-token pointers may be NULL
  st = check_inputs(hidden, weight, bias, targets, temperature, N, D, V);
  if (st != LLP_OK) return st;
  if (out_logp == nullptr || out_lse == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(out_logp, 4) || !aligned(out_lse, 4)) return LLP_ERR_MISALIGNED;
  const FwdLayout L = fwd_layout(N, V);
  if (workspace == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(workspace, 16)) return LLP_ERR_MISALIGNED;
  if (workspace_bytes < L.total) return LLP_ERR_WORKSPACE_TOO_SMALL;

  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  if ((st = load_encode_fn()) != LLP_OK) return st;
  return fwd_core(dev, hidden, weight, bias, targets, temperature, N, D, V, ignore_index, out_logp, out_lse,
                  static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream), 0, nullptr, nullptr, nullptr,
                  f16);
}

int linear_logp_fwd(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                    const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                    float* out_logp, float* out_lse, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_entry(hidden, weight, bias, targets, temperature, N, D, V, ignore_index, out_logp, out_lse, workspace,
                   workspace_bytes, stream, false);
}

int linear_logp_fwd_f16(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                        const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                        float* out_logp, float* out_lse, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_entry(hidden, weight, bias, targets, temperature, N, D, V, ignore_index, out_logp, out_lse, workspace,
                   workspace_bytes, stream, true);
}

// hidden / weight / grad_hidden / grad_weight are bf16, or IEEE fp16 when f16.
static int bwd_entry(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                     const float* bias, const int64_t* targets, const float* temperature, int64_t N, int64_t D,
                     int64_t V, int64_t ignore_index, void* grad_hidden, void* grad_weight, float* grad_bias,
                     void* workspace, size_t workspace_bytes, void* stream, bool f16) {
  int st = check_shapes(N, D, V);
  if (st != LLP_OK) return st;
  if (grad_bias != nullptr && bias == nullptr) return LLP_ERR_NULL_POINTER;
  if ((grad_hidden && !aligned(grad_hidden, 16)) || (grad_weight && !aligned(grad_weight, 16)) ||
      (grad_bias && !aligned(grad_bias, 4)))
    return LLP_ERR_MISALIGNED;
  if (grad_hidden == nullptr && grad_weight == nullptr && grad_bias == nullptr) return LLP_OK;

  DeviceInit* dev = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    // Sums over an empty set of tokens: the weight and bias gradients are zero.
    // The per-token pointers (hidden, targets, grad_logp, saved_lse) may be NULL.
    if ((st = init_device(&dev)) != LLP_OK) return st;
    if (grad_weight && cudaMemsetAsync(grad_weight, 0, static_cast<size_t>(V) * D * 2, s) != cudaSuccess)
      return fail_cuda(__LINE__);
    if (grad_bias && cudaMemsetAsync(grad_bias, 0, static_cast<size_t>(V) * sizeof(float), s) != cudaSuccess)
      return fail_cuda(__LINE__);
    return LLP_OK;
  }
  st = check_inputs(hidden, weight, bias, targets, temperature, N, D, V);
  if (st != LLP_OK) return st;
  if (grad_logp == nullptr || saved_lse == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(grad_logp, 4) || !aligned(saved_lse, 4)) return LLP_ERR_MISALIGNED;
  const BwdLayout L = bwd_layout(N, D, V, bias != nullptr, grad_hidden != nullptr, grad_weight != nullptr);
  if (workspace == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(workspace, 16)) return LLP_ERR_MISALIGNED;
  if (workspace_bytes < L.total) return LLP_ERR_WORKSPACE_TOO_SMALL;

  if ((st = init_device(&dev)) != LLP_OK) return st;
  if ((st = load_encode_fn()) != LLP_OK) return st;
  return bwd_core(dev, grad_logp, saved_lse, hidden, weight, bias, targets, temperature, N, D, V, ignore_index,
                  grad_hidden, grad_weight, grad_bias, static_cast<uint8_t*>(workspace), s, 0, -1, nullptr, f16);
}

int linear_logp_bwd(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                    const float* bias, const int64_t* targets, const float* temperature, int64_t N, int64_t D,
                    int64_t V, int64_t ignore_index, void* grad_hidden, void* grad_weight, float* grad_bias,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_entry(grad_logp, saved_lse, hidden, weight, bias, targets, temperature, N, D, V, ignore_index,
                   grad_hidden, grad_weight, grad_bias, workspace, workspace_bytes, stream, false);
}

int linear_logp_bwd_f16(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                        const float* bias, const int64_t* targets, const float* temperature, int64_t N, int64_t D,
                        int64_t V, int64_t ignore_index, void* grad_hidden, void* grad_weight, float* grad_bias,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_entry(grad_logp, saved_lse, hidden, weight, bias, targets, temperature, N, D, V, ignore_index,
                   grad_hidden, grad_weight, grad_bias, workspace, workspace_bytes, stream, true);
}

// ----------------------------------------------------------------------------
// Row-subset (indexed) variants: select -> gather a compact problem of
// Kc = min(K, N) rows (padding slots carry an ignored target) -> the plain
// launch sequence on it -> scatter back.  Every launch size is known on the host.
// ----------------------------------------------------------------------------
struct IdxLayout {
  size_t sel, c_hidden, c_targets, c_temp, c_a, c_b, c_gh, inner, total;
  int64_t Kc;
};

static IdxLayout idx_layout(int64_t N, int64_t D, int64_t V, int64_t K, bool bwd, bool bias) {
  IdxLayout L;
  L.Kc = K < N ? K : N;
  const size_t Kc = static_cast<size_t>(L.Kc);
  Carver c;
  L.sel = c.take(llp::select_workspace_bytes(N, K));
  L.c_hidden = c.take(Kc * D * 2);
  L.c_targets = c.take(Kc * 8);
  L.c_temp = c.take(Kc * 4);
  L.c_a = c.take(Kc * 4);  // forward: compact logp; backward: compact grad_logp
  L.c_b = c.take(Kc * 4);  // compact lse
  L.c_gh = bwd ? c.take(Kc * D * 2) : 0;
  L.inner = c.take(L.Kc > 0 ? (bwd ? bwd_layout(L.Kc, D, V, bias, true, true).total
                                   : fwd_layout(L.Kc, V).total)
                            : 0);
  L.total = c.off;
  return L;
}

size_t linear_logp_fwd_indexed_workspace_bytes(int64_t N, int64_t D, int64_t V, int64_t K) {
  if (N <= 0 || K <= 0 || check_shapes(N, D, V) != LLP_OK) return 0;
  return idx_layout(N, D, V, K, false, false).total;
}

size_t linear_logp_bwd_indexed_workspace_bytes(int64_t N, int64_t D, int64_t V, int64_t K, int has_bias) {
  if (N <= 0 || K <= 0 || check_shapes(N, D, V) != LLP_OK) return 0;
  return idx_layout(N, D, V, K, true, has_bias != 0).total;
}

// hidden / weight bf16, or IEEE fp16 when f16 (the row copies move raw 16-bit values).
static int fwd_indexed_entry(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                             const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                             const int64_t* indices, int64_t K, float* out_logp, float* out_lse, void* workspace,
                             size_t workspace_bytes, void* stream, bool f16) {
  int st = check_shapes(N, D, V);
  if (st != LLP_OK) return st;
  if (K < 0 || K > kLim31) return LLP_ERR_BAD_SHAPE;
  if (N == 0 || K == 0) return LLP_OK;  // nothing selected: outputs untouched
  if (indices == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(indices, 8)) return LLP_ERR_MISALIGNED;
  st = check_inputs(hidden, weight, bias, targets, temperature, N, D, V);
  if (st != LLP_OK) return st;
  if (out_logp == nullptr || out_lse == nullptr || workspace == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(out_logp, 4) || !aligned(out_lse, 4) || !aligned(workspace, 16)) return LLP_ERR_MISALIGNED;
  const IdxLayout L = idx_layout(N, D, V, K, false, false);
  if (workspace_bytes < L.total) return LLP_ERR_WORKSPACE_TOO_SMALL;
  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  if ((st = load_encode_fn()) != LLP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  llp::RowSelection sel;
  if (llp::build_row_selection(reinterpret_cast<const long long*>(indices), K, static_cast<int>(N), ws + L.sel, &sel,
                               s) != cudaSuccess)
    return fail_cuda(__LINE__);
  auto* c_hidden = reinterpret_cast<__nv_bfloat16*>(ws + L.c_hidden);
  auto* c_targets = reinterpret_cast<long long*>(ws + L.c_targets);
  float* c_temp = temperature ? reinterpret_cast<float*>(ws + L.c_temp) : nullptr;
  if (llp::gather_selected_rows(sel, static_cast<int>(D), static_cast<const __nv_bfloat16*>(hidden),
                                reinterpret_cast<const long long*>(targets), temperature, nullptr, nullptr,
                                ignore_index, c_hidden, c_targets, c_temp, nullptr, nullptr, s) != cudaSuccess)
    return fail_cuda(__LINE__);
  float* c_logp = reinterpret_cast<float*>(ws + L.c_a);
  float* c_lse = reinterpret_cast<float*>(ws + L.c_b);
  st = fwd_core(dev, c_hidden, weight, bias, reinterpret_cast<const int64_t*>(c_targets), c_temp, L.Kc, D, V,
                ignore_index, c_logp, c_lse, ws + L.inner, s, 0, nullptr, nullptr, nullptr, f16);
  if (st != LLP_OK) return st;
  return llp::scatter_selected_outputs(sel, c_logp, c_lse, out_logp, out_lse, s) == cudaSuccess ? LLP_OK : fail_cuda(__LINE__);
}

int linear_logp_fwd_indexed(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                            const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                            const int64_t* indices, int64_t K, float* out_logp, float* out_lse, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return fwd_indexed_entry(hidden, weight, bias, targets, temperature, N, D, V, ignore_index, indices, K, out_logp,
                           out_lse, workspace, workspace_bytes, stream, false);
}

int linear_logp_fwd_indexed_f16(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                                const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                                const int64_t* indices, int64_t K, float* out_logp, float* out_lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return fwd_indexed_entry(hidden, weight, bias, targets, temperature, N, D, V, ignore_index, indices, K, out_logp,
                           out_lse, workspace, workspace_bytes, stream, true);
}

static int bwd_indexed_entry(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                             const float* bias, const int64_t* targets, const float* temperature, int64_t N,
                             int64_t D, int64_t V, int64_t ignore_index, const int64_t* indices, int64_t K,
                             void* grad_hidden, void* grad_weight, float* grad_bias, void* workspace,
                             size_t workspace_bytes, void* stream, bool f16) {
  int st = check_shapes(N, D, V);
  if (st != LLP_OK) return st;
  if (K < 0 || K > kLim31) return LLP_ERR_BAD_SHAPE;
  if (grad_bias != nullptr && bias == nullptr) return LLP_ERR_NULL_POINTER;
  if ((grad_hidden && !aligned(grad_hidden, 16)) || (grad_weight && !aligned(grad_weight, 16)) ||
      (grad_bias && !aligned(grad_bias, 4)))
    return LLP_ERR_MISALIGNED;
  if (grad_hidden == nullptr && grad_weight == nullptr && grad_bias == nullptr) return LLP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceInit* dev = nullptr;
  if (N == 0 || K == 0) {  // nothing selected: every gradient is zero
    if ((st = init_device(&dev)) != LLP_OK) return st;
    if (grad_hidden && N > 0 && cudaMemsetAsync(grad_hidden, 0, static_cast<size_t>(N) * D * 2, s) != cudaSuccess)
      return fail_cuda(__LINE__);
    if (grad_weight && cudaMemsetAsync(grad_weight, 0, static_cast<size_t>(V) * D * 2, s) != cudaSuccess)
      return fail_cuda(__LINE__);
    if (grad_bias && cudaMemsetAsync(grad_bias, 0, static_cast<size_t>(V) * 4, s) != cudaSuccess)
      return fail_cuda(__LINE__);
    return LLP_OK;
  }
  if (indices == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(indices, 8)) return LLP_ERR_MISALIGNED;
  st = check_inputs(hidden, weight, bias, targets, temperature, N, D, V);
  if (st != LLP_OK) return st;
  if (grad_logp == nullptr || saved_lse == nullptr || workspace == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(grad_logp, 4) || !aligned(saved_lse, 4) || !aligned(workspace, 16)) return LLP_ERR_MISALIGNED;
  const IdxLayout L = idx_layout(N, D, V, K, true, bias != nullptr);
  if (workspace_bytes < L.total) return LLP_ERR_WORKSPACE_TOO_SMALL;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  if ((st = load_encode_fn()) != LLP_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  llp::RowSelection sel;
  if (llp::build_row_selection(reinterpret_cast<const long long*>(indices), K, static_cast<int>(N), ws + L.sel, &sel,
                               s) != cudaSuccess)
    return fail_cuda(__LINE__);
  auto* c_hidden = reinterpret_cast<__nv_bfloat16*>(ws + L.c_hidden);
  auto* c_targets = reinterpret_cast<long long*>(ws + L.c_targets);
  float* c_temp = temperature ? reinterpret_cast<float*>(ws + L.c_temp) : nullptr;
  float* c_grad = reinterpret_cast<float*>(ws + L.c_a);
  float* c_lse = reinterpret_cast<float*>(ws + L.c_b);
  if (llp::gather_selected_rows(sel, static_cast<int>(D), static_cast<const __nv_bfloat16*>(hidden),
                                reinterpret_cast<const long long*>(targets), temperature, grad_logp, saved_lse,
                                ignore_index, c_hidden, c_targets, c_temp, c_grad, c_lse, s) != cudaSuccess)
    return fail_cuda(__LINE__);
  auto* c_gh = grad_hidden ? reinterpret_cast<__nv_bfloat16*>(ws + L.c_gh) : nullptr;
  st = bwd_core(dev, c_grad, c_lse, c_hidden, weight, bias, reinterpret_cast<const int64_t*>(c_targets), c_temp,
                L.Kc, D, V, ignore_index, c_gh, grad_weight, grad_bias, ws + L.inner, s, 0, -1, nullptr, f16);
  if (st != LLP_OK) return st;
  if (grad_hidden &&
      llp::scatter_selected_grad_hidden(sel, static_cast<int>(N), static_cast<int>(D), c_gh,
                                        static_cast<__nv_bfloat16*>(grad_hidden), s) != cudaSuccess)
    return fail_cuda(__LINE__);
  return LLP_OK;
}

int linear_logp_bwd_indexed(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                            const float* bias, const int64_t* targets, const float* temperature, int64_t N,
                            int64_t D, int64_t V, int64_t ignore_index, const int64_t* indices, int64_t K,
                            void* grad_hidden, void* grad_weight, float* grad_bias, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return bwd_indexed_entry(grad_logp, saved_lse, hidden, weight, bias, targets, temperature, N, D, V, ignore_index,
                           indices, K, grad_hidden, grad_weight, grad_bias, workspace, workspace_bytes, stream, false);
}

int linear_logp_bwd_indexed_f16(const float* grad_logp, const float* saved_lse, const void* hidden,
                                const void* weight, const float* bias, const int64_t* targets,
                                const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                                const int64_t* indices, int64_t K, void* grad_hidden, void* grad_weight,
                                float* grad_bias, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_indexed_entry(grad_logp, saved_lse, hidden, weight, bias, targets, temperature, N, D, V, ignore_index,
                           indices, K, grad_hidden, grad_weight, grad_bias, workspace, workspace_bytes, stream, true);
}

// ----------------------------------------------------------------------------
// Vocab-parallel shards.
// ----------------------------------------------------------------------------
// hidden / weight_local bf16, or IEEE fp16 when f16.
static int fwd_shard_entry(const void* hidden, const void* weight_local, const float* bias_local,
                           const int64_t* targets, const float* temperature, int64_t N, int64_t D, int64_t V_local,
                           int64_t vocab_start, int64_t ignore_index, float* out_max, float* out_sumexp,
                           float* out_target_logit, void* workspace, size_t workspace_bytes, void* stream, bool f16) {
  int st = check_shapes(N, D, V_local);
  if (st != LLP_OK) return st;
  if (vocab_start < 0 || vocab_start > kLim31 - V_local) return LLP_ERR_BAD_SHAPE;
  if (N == 0) return LLP_OK;
  st = check_inputs(hidden, weight_local, bias_local, targets, temperature, N, D, V_local);
  if (st != LLP_OK) return st;
  if (out_max == nullptr || out_sumexp == nullptr || out_target_logit == nullptr || workspace == nullptr)
    return LLP_ERR_NULL_POINTER;
  if (!aligned(out_max, 4) || !aligned(out_sumexp, 4) || !aligned(out_target_logit, 4) || !aligned(workspace, 16))
    return LLP_ERR_MISALIGNED;
  if (workspace_bytes < fwd_layout(N, V_local).total) return LLP_ERR_WORKSPACE_TOO_SMALL;
  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  if ((st = load_encode_fn()) != LLP_OK) return st;
  return fwd_core(dev, hidden, weight_local, bias_local, targets, temperature, N, D, V_local, ignore_index, nullptr,
                  nullptr, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream), vocab_start, out_max,
                  out_sumexp, out_target_logit, f16);
}

int linear_logp_fwd_shard(const void* hidden, const void* weight_local, const float* bias_local,
                          const int64_t* targets, const float* temperature, int64_t N, int64_t D, int64_t V_local,
                          int64_t vocab_start, int64_t ignore_index, float* out_max, float* out_sumexp,
                          float* out_target_logit, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_shard_entry(hidden, weight_local, bias_local, targets, temperature, N, D, V_local, vocab_start,
                         ignore_index, out_max, out_sumexp, out_target_logit, workspace, workspace_bytes, stream,
                         false);
}

int linear_logp_fwd_shard_f16(const void* hidden, const void* weight_local, const float* bias_local,
                              const int64_t* targets, const float* temperature, int64_t N, int64_t D,
                              int64_t V_local, int64_t vocab_start, int64_t ignore_index, float* out_max,
                              float* out_sumexp, float* out_target_logit, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return fwd_shard_entry(hidden, weight_local, bias_local, targets, temperature, N, D, V_local, vocab_start,
                         ignore_index, out_max, out_sumexp, out_target_logit, workspace, workspace_bytes, stream,
                         true);
}

int linear_logp_merge_shards(const float* shard_max, const float* shard_sumexp, const float* shard_target_logit,
                             int64_t R, int64_t N, const int64_t* targets, int64_t global_V, int64_t ignore_index,
                             float* out_logp, float* out_lse, void* stream) {
  if (R < 1 || N < 0 || global_V < 1 || N > kLim31 || global_V > kLim31 || !product_ok(R, N) || R * N > kLim62)
    return LLP_ERR_BAD_SHAPE;
  if (N == 0) return LLP_OK;
  if (!shard_max || !shard_sumexp || !shard_target_logit || !targets || !out_logp || !out_lse)
    return LLP_ERR_NULL_POINTER;
  if (!aligned(shard_max, 4) || !aligned(shard_sumexp, 4) || !aligned(shard_target_logit, 4) ||
      !aligned(targets, 8) || !aligned(out_logp, 4) || !aligned(out_lse, 4))
    return LLP_ERR_MISALIGNED;
  DeviceInit* dev = nullptr;
  const int st = init_device(&dev);
  if (st != LLP_OK) return st;
  return llp::launch_merge_shards(shard_max, shard_sumexp, shard_target_logit, static_cast<int>(R),
                                  static_cast<int>(N), reinterpret_cast<const long long*>(targets), global_V,
                                  ignore_index, out_logp, out_lse, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LLP_OK : fail_cuda(__LINE__);
}

static int bwd_shard_entry(const float* grad_logp, const float* lse, const void* hidden, const void* weight_local,
                           const float* bias_local, const int64_t* targets, const float* temperature, int64_t N,
                           int64_t D, int64_t V_local, int64_t vocab_start, int64_t global_V, int64_t ignore_index,
                           float* grad_hidden_partial, void* grad_weight_local, float* grad_bias_local,
                           void* workspace, size_t workspace_bytes, void* stream, bool f16) {
  int st = check_shapes(N, D, V_local);
  if (st != LLP_OK) return st;
  if (vocab_start < 0 || global_V < 1 || global_V > kLim31 || vocab_start > global_V - V_local)
    return LLP_ERR_BAD_SHAPE;
  if (grad_bias_local != nullptr && bias_local == nullptr) return LLP_ERR_NULL_POINTER;
  if ((grad_hidden_partial && !aligned(grad_hidden_partial, 16)) ||
      (grad_weight_local && !aligned(grad_weight_local, 16)) || (grad_bias_local && !aligned(grad_bias_local, 4)))
    return LLP_ERR_MISALIGNED;
  if (!grad_hidden_partial && !grad_weight_local && !grad_bias_local) return LLP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceInit* dev = nullptr;
  if (N == 0) {
    if ((st = init_device(&dev)) != LLP_OK) return st;
    if (grad_weight_local && cudaMemsetAsync(grad_weight_local, 0, static_cast<size_t>(V_local) * D * 2, s))
      return fail_cuda(__LINE__);
    if (grad_bias_local && cudaMemsetAsync(grad_bias_local, 0, static_cast<size_t>(V_local) * 4, s))
      return fail_cuda(__LINE__);
    return LLP_OK;
  }
  st = check_inputs(hidden, weight_local, bias_local, targets, temperature, N, D, V_local);
  if (st != LLP_OK) return st;
  if (grad_logp == nullptr || lse == nullptr || workspace == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(grad_logp, 4) || !aligned(lse, 4) || !aligned(workspace, 16)) return LLP_ERR_MISALIGNED;
  const BwdLayout L = bwd_layout(N, D, V_local, bias_local != nullptr, grad_hidden_partial != nullptr,
                                 grad_weight_local != nullptr);
  if (workspace_bytes < L.total) return LLP_ERR_WORKSPACE_TOO_SMALL;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  if ((st = load_encode_fn()) != LLP_OK) return st;
  return bwd_core(dev, grad_logp, lse, hidden, weight_local, bias_local, targets, temperature, N, D, V_local,
                  ignore_index, nullptr, grad_weight_local, grad_bias_local, static_cast<uint8_t*>(workspace), s,
                  vocab_start, global_V, grad_hidden_partial, f16);
}

int linear_logp_bwd_shard(const float* grad_logp, const float* lse, const void* hidden, const void* weight_local,
                          const float* bias_local, const int64_t* targets, const float* temperature, int64_t N,
                          int64_t D, int64_t V_local, int64_t vocab_start, int64_t global_V, int64_t ignore_index,
                          float* grad_hidden_partial, void* grad_weight_local, float* grad_bias_local,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_shard_entry(grad_logp, lse, hidden, weight_local, bias_local, targets, temperature, N, D, V_local,
                         vocab_start, global_V, ignore_index, grad_hidden_partial, grad_weight_local,
                         grad_bias_local, workspace, workspace_bytes, stream, false);
}

int linear_logp_bwd_shard_f16(const float* grad_logp, const float* lse, const void* hidden,
                              const void* weight_local, const float* bias_local, const int64_t* targets,
                              const float* temperature, int64_t N, int64_t D, int64_t V_local, int64_t vocab_start,
                              int64_t global_V, int64_t ignore_index, float* grad_hidden_partial,
                              void* grad_weight_local, float* grad_bias_local, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return bwd_shard_entry(grad_logp, lse, hidden, weight_local, bias_local, targets, temperature, N, D, V_local,
                         vocab_start, global_V, ignore_index, grad_hidden_partial, grad_weight_local,
                         grad_bias_local, workspace, workspace_bytes, stream, true);
}

static int sum_partials_entry(const float* parts, int64_t R, int64_t count, void* out_bf16, void* stream,
                              bool f16) {
  if (R < 1 || count < 0 || (count % 4) != 0 || !product_ok(R, count)) return LLP_ERR_BAD_SHAPE;
  if (count == 0) return LLP_OK;
  if (parts == nullptr || out_bf16 == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(parts, 16) || !aligned(out_bf16, 8)) return LLP_ERR_MISALIGNED;
  DeviceInit* dev = nullptr;
  const int st = init_device(&dev);
  if (st != LLP_OK) return st;
  return llp::launch_segment_sum(parts, static_cast<int>(R), count, static_cast<__nv_bfloat16*>(out_bf16),
                                 dev->num_sms, static_cast<cudaStream_t>(stream), f16 ? 1 : 0) == cudaSuccess
             ? LLP_OK : fail_cuda(__LINE__);
}

int linear_logp_sum_partials(const float* parts, int64_t R, int64_t count, void* out_bf16, void* stream) {
  return sum_partials_entry(parts, R, count, out_bf16, stream, false);
}

int linear_logp_sum_partials_f16(const float* parts, int64_t R, int64_t count, void* out_f16, void* stream) {
  return sum_partials_entry(parts, R, count, out_f16, stream, true);
}

// ----------------------------------------------------------------------------
// Logits-input fused log-prob (include/fused_logp.h).
// ----------------------------------------------------------------------------
static int fused_check(const void* logits, int dtype, int64_t N, int64_t V, const int64_t* targets) {
  if (dtype != FUSED_LOGP_DTYPE_BF16 && dtype != FUSED_LOGP_DTYPE_F32 && dtype != FUSED_LOGP_DTYPE_F16)
    return LLP_ERR_BAD_SHAPE;
  if (N < 0 || V < 1 || N > kLim31 || V > kLim31 || !product_ok(N, V)) return LLP_ERR_BAD_SHAPE;
  if (N * cdiv(V, llp::kLogitsSplit) > kLim31) return LLP_ERR_BAD_SHAPE;
  if (N == 0) return LLP_OK;
  if (logits == nullptr || targets == nullptr) return LLP_ERR_NULL_POINTER;
  const uintptr_t es = dtype == FUSED_LOGP_DTYPE_F32 ? 4 : 2;
  if (!aligned(logits, es) || !aligned(targets, 8)) return LLP_ERR_MISALIGNED;
  return LLP_OK;
}

static bool fused_vec_ok(const void* p, int dtype, int64_t V) {
  const int64_t es = dtype == FUSED_LOGP_DTYPE_F32 ? 4 : 2;
  return aligned(p, 16) && ((V * es) % 16) == 0;
}

size_t fused_logp_workspace_bytes(int64_t N, int64_t V) {
  if (N <= 0 || V < 1 || N > kLim31 || V > kLim31) return 0;
  return static_cast<size_t>(2 * cdiv(V, llp::kLogitsSplit) * N) * sizeof(float);
}

int fused_logp_fwd(const void* logits, int dtype, int64_t N, int64_t V, const int64_t* targets,
                   int64_t ignore_index, float* out_logp, float* out_row_max, float* out_log_sum, void* workspace,
                   size_t workspace_bytes, void* stream) {
  int st = fused_check(logits, dtype, N, V, targets);
  if (st != LLP_OK) return st;
  if (N == 0) return LLP_OK;
  if (out_logp == nullptr || out_row_max == nullptr || out_log_sum == nullptr || workspace == nullptr)
    return LLP_ERR_NULL_POINTER;
  if (!aligned(out_logp, 4) || !aligned(out_row_max, 4) || !aligned(out_log_sum, 4) || !aligned(workspace, 16))
    return LLP_ERR_MISALIGNED;
  if (workspace_bytes < fused_logp_workspace_bytes(N, V)) return LLP_ERR_WORKSPACE_TOO_SMALL;
  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  const cudaError_t e = llp::launch_logits_fwd(
      logits, dtype, static_cast<int>(N), nullptr, static_cast<int>(V), reinterpret_cast<const long long*>(targets),
      ignore_index, static_cast<float*>(workspace), out_logp, out_row_max, out_log_sum,
      fused_vec_ok(logits, dtype, V), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LLP_OK : fail_cuda(__LINE__);
}

int fused_logp_bwd(const float* grad_logp, const float* row_max, const float* log_sum, const void* logits, int dtype,
                   int64_t N, int64_t V, const int64_t* targets, int64_t ignore_index, void* grad_logits,
                   void* stream) {
  int st = fused_check(logits, dtype, N, V, targets);
  if (st != LLP_OK) return st;
  if (N == 0) return LLP_OK;
  if (grad_logp == nullptr || row_max == nullptr || log_sum == nullptr || grad_logits == nullptr)
    return LLP_ERR_NULL_POINTER;
  const uintptr_t es = dtype == FUSED_LOGP_DTYPE_F32 ? 4 : 2;
  if (!aligned(grad_logp, 4) || !aligned(row_max, 4) || !aligned(log_sum, 4) || !aligned(grad_logits, es))
    return LLP_ERR_MISALIGNED;
  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  const bool vec = fused_vec_ok(logits, dtype, V) && fused_vec_ok(grad_logits, dtype, V);
  const cudaError_t e = llp::launch_logits_bwd(
      logits, dtype, static_cast<int>(N), static_cast<int>(V), reinterpret_cast<const long long*>(targets),
      ignore_index, grad_logp, row_max, log_sum, nullptr, grad_logits, vec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LLP_OK : fail_cuda(__LINE__);
}

// Row-subset forms: the index list becomes a byte mask and an ascending list
// of distinct selected rows (padded with -1 to min(K, N) slots).
static size_t fused_sel_bytes(int64_t N, int64_t K) {
  return round_up(llp::select_workspace_bytes(N, K), 256);
}

size_t fused_logp_fwd_indexed_workspace_bytes(int64_t N, int64_t V, int64_t K) {
  if (N <= 0 || K <= 0 || V < 1 || N > kLim31 || V > kLim31 || K > kLim31) return 0;
  const int64_t Kc = K < N ? K : N;
  return fused_sel_bytes(N, K) + static_cast<size_t>(2 * cdiv(V, llp::kLogitsSplit) * Kc) * sizeof(float);
}

size_t fused_logp_bwd_indexed_workspace_bytes(int64_t N, int64_t K) {
  if (N <= 0 || N > kLim31 || K < 0 || K > kLim31) return 0;
  return fused_sel_bytes(N, K);
}

int fused_logp_fwd_indexed(const void* logits, int dtype, int64_t N, int64_t V, const int64_t* targets,
                           int64_t ignore_index, const int64_t* indices, int64_t K, float* out_logp,
                           float* out_row_max, float* out_log_sum, void* workspace, size_t workspace_bytes,
                           void* stream) {
  int st = fused_check(logits, dtype, N, V, targets);
  if (st != LLP_OK) return st;
  if (K < 0 || K > kLim31) return LLP_ERR_BAD_SHAPE;
  if (N == 0 || K == 0) return LLP_OK;  // nothing selected: outputs untouched
  if (indices == nullptr || out_logp == nullptr || out_row_max == nullptr || out_log_sum == nullptr ||
      workspace == nullptr)
    return LLP_ERR_NULL_POINTER;
  if (!aligned(indices, 8) || !aligned(out_logp, 4) || !aligned(out_row_max, 4) || !aligned(out_log_sum, 4) ||
      !aligned(workspace, 16))
    return LLP_ERR_MISALIGNED;
  if (workspace_bytes < fused_logp_fwd_indexed_workspace_bytes(N, V, K)) return LLP_ERR_WORKSPACE_TOO_SMALL;
  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  llp::RowSelection sel;
  if (llp::build_row_selection(reinterpret_cast<const long long*>(indices), K, static_cast<int>(N), ws, &sel, s) !=
      cudaSuccess)
    return fail_cuda(__LINE__);
  const cudaError_t e = llp::launch_logits_fwd(
      logits, dtype, sel.K, sel.rows, static_cast<int>(V), reinterpret_cast<const long long*>(targets), ignore_index,
      reinterpret_cast<float*>(ws + fused_sel_bytes(N, K)), out_logp, out_row_max, out_log_sum,
      fused_vec_ok(logits, dtype, V), s);
  return e == cudaSuccess ? LLP_OK : fail_cuda(__LINE__);
}

int fused_logp_bwd_indexed(const float* grad_logp, const float* row_max, const float* log_sum, const void* logits,
                           int dtype, int64_t N, int64_t V, const int64_t* targets, int64_t ignore_index,
                           const int64_t* indices, int64_t K, void* grad_logits, void* workspace,
                           size_t workspace_bytes, void* stream) {
  int st = fused_check(logits, dtype, N, V, targets);
  if (st != LLP_OK) return st;
  if (K < 0 || K > kLim31) return LLP_ERR_BAD_SHAPE;
  if (N == 0) return LLP_OK;
  if (grad_logp == nullptr || row_max == nullptr || log_sum == nullptr || grad_logits == nullptr ||
      workspace == nullptr || (K > 0 && indices == nullptr))
    return LLP_ERR_NULL_POINTER;
  const uintptr_t es = dtype == FUSED_LOGP_DTYPE_F32 ? 4 : 2;
  if (!aligned(grad_logp, 4) || !aligned(row_max, 4) || !aligned(log_sum, 4) || !aligned(grad_logits, es) ||
      !aligned(workspace, 16) || (K > 0 && !aligned(indices, 8)))
    return LLP_ERR_MISALIGNED;
  if (workspace_bytes < fused_logp_bwd_indexed_workspace_bytes(N, K)) return LLP_ERR_WORKSPACE_TOO_SMALL;
  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  llp::RowSelection sel;
  if (llp::build_row_selection(reinterpret_cast<const long long*>(indices), K, static_cast<int>(N), workspace, &sel,
                               s) != cudaSuccess)
    return fail_cuda(__LINE__);
  const bool vec = fused_vec_ok(logits, dtype, V) && fused_vec_ok(grad_logits, dtype, V);
  const cudaError_t e = llp::launch_logits_bwd(logits, dtype, static_cast<int>(N), static_cast<int>(V),
                                               reinterpret_cast<const long long*>(targets), ignore_index, grad_logp,
                                               row_max, log_sum, sel.mask, grad_logits, vec, s);
  return e == cudaSuccess ? LLP_OK : fail_cuda(__LINE__);
}

// One thread waits, with the production wait code, on a barrier that nothing
// ever completes; the bounded wait must give up after limit_ns and record the
// self-test code instead of hanging.
static __global__ void wait_timeout_probe_kernel(unsigned int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  llp::mbar_init(&bar, 1);
  abort_flag = 0;
  llp::fence_mbarrier_init();
  llp::mbar_wait(&bar, 0, &abort_flag, err, llp::kDevTimeoutSelfTest, limit_ns);
}

int linear_logp_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns < 1 || limit_ns > 1000000000ull) return LLP_ERR_BAD_SHAPE;
  DeviceInit* dev = nullptr;
  const int st = init_device(&dev);
  if (st != LLP_OK) return st;
  wait_timeout_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(dev->status_ptr, limit_ns);
  return llp::launch_result() == cudaSuccess ? LLP_OK : fail_cuda(__LINE__);
}

int linear_logp_last_cuda_error(void) { return g_last_cuda_error; }

int linear_logp_last_failure(int* cuda_error, int* driver_result, int* site) {
  if (cuda_error) *cuda_error = g_last_cuda_error;
  if (driver_result) *driver_result = g_last_driver_result;
  if (site) *site = g_last_failure_line;
  return LLP_OK;
}

const char* linear_logp_cuda_error_name(int code) { return cudaGetErrorName(static_cast<cudaError_t>(code)); }

int linear_logp_device_status(void* stream, unsigned int* device_code) {
  DeviceInit* dev = nullptr;
  const int st = init_device(&dev);
  if (st != LLP_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return fail_cuda(__LINE__);
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return fail_cuda(__LINE__);
  if (device_code != nullptr) *device_code = v;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return fail_cuda(__LINE__);
    return LLP_ERR_DEVICE_TIMEOUT;
  }
  return LLP_OK;
}

// ----------------------------------------------------------------------------
// Forward without a caller workspace (linear_logp_fwd_noalloc in the header):
// for callers that cannot allocate device memory themselves.  Its scratch is
// this fixed file-scope array; host code only ever uses the device address
// obtained from cudaGetSymbolAddress, never the array's name.
// ----------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[LINEAR_LOGP_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[kMaxDevices] = {};

// One-time per-device look-up of the scratch array's device address, with that
// device current.  Returns LLP_OK and the address, or LLP_ERR_CUDA.
static int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail_cuda(__LINE__);
  if (dev < 0 || dev >= kMaxDevices) return LLP_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return fail_cuda(__LINE__);
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return LLP_OK;
}

int linear_logp_fwd_noalloc(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                            const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                            float* out_logp, float* out_lse, void* stream) {
  int st = check_shapes(N, D, V);
  if (st != LLP_OK) return st;
  if (N == 0) return LLP_OK;
  st = check_inputs(hidden, weight, bias, targets, temperature, N, D, V);
  if (st != LLP_OK) return st;
  if (out_logp == nullptr || out_lse == nullptr) return LLP_ERR_NULL_POINTER;
  if (!aligned(out_logp, 4) || !aligned(out_lse, 4)) return LLP_ERR_MISALIGNED;
  const FwdLayout L = fwd_layout(N, V);
  if (L.total > static_cast<size_t>(LINEAR_LOGP_NOALLOC_SCRATCH_BYTES)) return LLP_ERR_SCRATCH_LIMIT;

  DeviceInit* dev = nullptr;
  if ((st = init_device(&dev)) != LLP_OK) return st;
  if ((st = load_encode_fn()) != LLP_OK) return st;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != LLP_OK) return st;
  // the same launch sequence as linear_logp_fwd, with the fixed array as its workspace
  return fwd_core(dev, hidden, weight, bias, targets, temperature, N, D, V, ignore_index, out_logp, out_lse,
                  static_cast<uint8_t*>(scratch), static_cast<cudaStream_t>(stream));
}

int linear_logp_profile_start(int capacity) {
  if (capacity < 1) return LLP_ERR_BAD_SHAPE;
  std::lock_guard<std::mutex> lock(g_rec.mu);
  const size_t need = static_cast<size_t>(capacity) * 2 + 2;
  while (g_rec.events.size() < need) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return fail_cuda(__LINE__);
    g_rec.events.push_back(e);
  }
  g_rec.ids.assign(g_rec.events.size(), -1);
  g_rec.launch_cap = capacity;
  g_rec.launches = 0;
  g_rec.used = 0;
  g_rec.on = true;
  return LLP_OK;
}

int linear_logp_profile_stop(int* kernel_ids, float* ms, int capacity) {
  std::lock_guard<std::mutex> lock(g_rec.mu);
  g_rec.on = false;
  if (g_rec.used == 0) return 0;
  if (cudaEventSynchronize(g_rec.events[g_rec.used - 1]) != cudaSuccess) return fail_cuda(__LINE__);
  int n = 0;
  for (int i = 1; i < g_rec.used; ++i) {
    if (g_rec.ids[i] < 0) continue;
    if (n < capacity && kernel_ids != nullptr && ms != nullptr) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, g_rec.events[i - 1], g_rec.events[i]) != cudaSuccess) return fail_cuda(__LINE__);
      kernel_ids[n] = g_rec.ids[i];
      ms[n] = t;
    }
    ++n;
  }
  return n;
}

const char* linear_logp_kernel_name(int kernel_id) {
  if (kernel_id < 0 || kernel_id >= kKNumKernels) return "unknown";
  return kKernelNames[kernel_id];
}

}  // extern "C"
