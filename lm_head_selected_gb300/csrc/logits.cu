// Logits-input fused log-probability ("Fused LogP": the logits [N, V] are
// already materialised; "add backward support for fused logp CUDA kernels",
// Summary and Implementation details).
//
//   forward   per (row, 16384-wide vocab split) CTA: stream the split once with
//             16-byte loads, keep a per-thread (max, sum of exp) pair, merge the
//             pairs in a fixed tree order -> partial (m_s, s_s);
//             then per row: merge the splits in ascending order, read z[t] once,
//             row_max = M, log_sum = log S, logp = (z[t] - M) - log S.
//   backward  per (row, split) CTA: grad[v] = g * (onehot(t)[v] - exp((z[v] -
//             row_max) - log_sum)) written in the logits' dtype, zero rows for
//             invalid targets; no probability tensor is formed.
//
// Both are bound by HBM bandwidth (every logit read once; the backward also
// writes every gradient once).  The split width and the reduction trees depend
// on V only, so a row's results are the same for every N and every run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "llp_internal.h"
#include "sm103_ptx.cuh"

namespace llp {

namespace {

constexpr int kLThreads = 256;
constexpr float kLog2eL = 1.4426950408889634f;
// Split-kernel shape, from a sweep at N=16384, V=131072, bf16 (0.712 ms for
// the split pass against 1.09 ms with 8-vector chunks at 3 CTAs per SM):
// 4 vectors per load batch, registers bounded so that 8 CTAs fit on an SM.
constexpr int kLChunk = 4;  // the same in the aligned and the element-wise path: a row's
                             // summation order must not depend on its address
#ifndef LLP_PACKED_MAX
#define LLP_PACKED_MAX 1  // chunk maximum on packed 16-bit pairs
#endif
constexpr int kLMinBlocks = 8;



__device__ __forceinline__ bool tgt_ok(long long t, int V, long long ignore_index) {
  return t != ignore_index && t >= 0 && t < static_cast<long long>(V);
}

// 16-byte vector of logits converted to fp32.
template <int DT>
struct Vec;
template <>
struct Vec<kDtypeBF16> {
  static constexpr int W = 8;
  using T = __nv_bfloat16;
  static __device__ __forceinline__ void load(const T* p, float (&v)[W]) {
    const uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ float load1(const T* p) { return __bfloat162float(*p); }
  // The W elements at p as stored, elements at or past n_valid reading as -inf.
  // One 16-byte load only when `vec` (p is 16-byte aligned) and all W are valid;
  // otherwise element-wise 2-byte loads.
  static __device__ __forceinline__ uint4 load_raw(const T* p, int n_valid, bool vec) {
    if (vec && n_valid >= W) return __ldg(reinterpret_cast<const uint4*>(p));
    uint32_t w[4];
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (2 * i < n_valid) ? q[2 * i] : 0xFF80u;
      const uint32_t hi = (2 * i + 1 < n_valid) ? q[2 * i + 1] : 0xFF80u;
      w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ void unpack(const uint4& r, float (&v)[W]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void store(T* p, const float (&v)[W]) {
    uint4 r;
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]),
                   c = __floats2bfloat162_rn(v[4], v[5]), d = __floats2bfloat162_rn(v[6], v[7]);
    r.x = *reinterpret_cast<uint32_t*>(&a);
    r.y = *reinterpret_cast<uint32_t*>(&b);
    r.z = *reinterpret_cast<uint32_t*>(&c);
    r.w = *reinterpret_cast<uint32_t*>(&d);
    *reinterpret_cast<uint4*>(p) = r;
  }
  static __device__ __forceinline__ void store1(T* p, float v) { *p = __float2bfloat16_rn(v); }
  // Maximum of n packed vectors, taken on bf16 pairs (exact: the result is one of the elements).
  template <int NV>
  static __device__ __forceinline__ float max_of(const uint4 (&r)[NV]) {
    __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162*>(&r[0].x);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
#pragma unroll
      for (int k = (i == 0 ? 1 : 0); k < 4; ++k) m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    }
    return fmaxf(__low2float(m), __high2float(m));
  }
};
template <>
struct Vec<kDtypeF32> {
  static constexpr int W = 4;
  using T = float;
  static __device__ __forceinline__ void load(const T* p, float (&v)[W]) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = r.x;
    v[1] = r.y;
    v[2] = r.z;
    v[3] = r.w;
  }
  static __device__ __forceinline__ float load1(const T* p) { return __ldg(p); }
  static __device__ __forceinline__ uint4 load_raw(const T* p, int n_valid, bool vec) {
    if (vec && n_valid >= W) return __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t ninf = __float_as_uint(-INFINITY);
    return make_uint4(n_valid > 0 ? __float_as_uint(p[0]) : ninf, n_valid > 1 ? __float_as_uint(p[1]) : ninf,
                      n_valid > 2 ? __float_as_uint(p[2]) : ninf, n_valid > 3 ? __float_as_uint(p[3]) : ninf);
  }
  static __device__ __forceinline__ void unpack(const uint4& r, float (&v)[W]) {
    v[0] = __uint_as_float(r.x);
    v[1] = __uint_as_float(r.y);
    v[2] = __uint_as_float(r.z);
    v[3] = __uint_as_float(r.w);
  }
  static __device__ __forceinline__ void store(T* p, const float (&v)[W]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  static __device__ __forceinline__ void store1(T* p, float v) { *p = v; }
  template <int NV>
  static __device__ __forceinline__ float max_of(const uint4 (&r)[NV]) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NV; ++i) m = fmaxf(fmaxf(fmaxf(m, __uint_as_float(r[i].x)), __uint_as_float(r[i].y)),
                                           fmaxf(__uint_as_float(r[i].z), __uint_as_float(r[i].w)));
    return m;
  }
};

template <>
struct Vec<kDtypeF16> {
  static constexpr int W = 8;
  using T = __half;
  static __device__ __forceinline__ float load1(const T* p) { return __half2float(*p); }
  // As the bf16 form; fp16 -inf is 0xFC00.
  static __device__ __forceinline__ uint4 load_raw(const T* p, int n_valid, bool vec) {
    if (vec && n_valid >= W) return __ldg(reinterpret_cast<const uint4*>(p));
    uint32_t w[4];
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (2 * i < n_valid) ? q[2 * i] : 0xFC00u;
      const uint32_t hi = (2 * i + 1 < n_valid) ? q[2 * i + 1] : 0xFC00u;
      w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ void unpack(const uint4& r, float (&v)[W]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void load(const T* p, float (&v)[W]) {
    unpack(__ldg(reinterpret_cast<const uint4*>(p)), v);
  }
  static __device__ __forceinline__ void store(T* p, const float (&v)[W]) {
    uint4 r;
    __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]), c = __floats2half2_rn(v[4], v[5]),
            d = __floats2half2_rn(v[6], v[7]);
    r.x = *reinterpret_cast<uint32_t*>(&a);
    r.y = *reinterpret_cast<uint32_t*>(&b);
    r.z = *reinterpret_cast<uint32_t*>(&c);
    r.w = *reinterpret_cast<uint32_t*>(&d);
    *reinterpret_cast<uint4*>(p) = r;
  }
  static __device__ __forceinline__ void store1(T* p, float v) { *p = __float2half_rn(v); }
  template <int NV>
  static __device__ __forceinline__ float max_of(const uint4 (&r)[NV]) {
    __half2 m = *reinterpret_cast<const __half2*>(&r[0].x);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
#pragma unroll
      for (int k = (i == 0 ? 1 : 0); k < 4; ++k) m = __hmax2(m, *reinterpret_cast<const __half2*>(&w[k]));
    }
    return fmaxf(__low2float(m), __high2float(m));
  }
};

// Merge (m, s) pairs: s is a sum of exp(x - m).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  s = s * exp2f((m - mn) * kLog2eL) + s2 * exp2f((m2 - mn) * kLog2eL);
  m = mn;
}

// Fixed-order block reduction of the per-thread pairs (butterfly within warps,
// then warp 0 over the warps in ascending order).
__device__ __forceinline__ void block_merge(float& m, float& s, float* sm_m, float* sm_s) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    merge_ms(m, s, m2, s2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm_m[warp] = m;
    sm_s[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = sm_m[0], S = sm_s[0];
    for (int w = 1; w < kLThreads / 32; ++w) merge_ms(M, S, sm_m[w], sm_s[w]);
    sm_m[0] = M;
    sm_s[0] = S;
  }
  __syncthreads();
  m = sm_m[0];
  s = sm_s[0];
}

// Each thread owns elements [split0 + (it * kLThreads + tid) * W, + W) for it = 0..ITERS-1,
// loaded kLChunk vectors at a time and kept packed until they are folded into
// the thread's (max, sum) pair, so few registers are live and 8 CTAs per SM
// keep many loads in flight.
template <int DT, bool VEC>
// Items are (slot, split) over P row slots: slot j is row rows[j] (row j when
// rows is null; a slot of -1 is padding and does nothing); partials go to
// [split][j].
__global__ void __launch_bounds__(kLThreads, kLMinBlocks) logits_split_kernel(const typename Vec<DT>::T* __restrict__ z,
                                                                    int V, int S, int P, const int* __restrict__ rows,
                                                                    float* __restrict__ part_m,
                                                                    float* __restrict__ part_s) {
  using VV = Vec<DT>;
  constexpr int W = VV::W;
  constexpr int ITERS = kLogitsSplit / (kLThreads * W);
  constexpr int CHUNK = ITERS < kLChunk ? ITERS : kLChunk;
  __shared__ float sm_m[kLThreads / 32], sm_s[kLThreads / 32];
  const long long cta = blockIdx.x;
  const int j = static_cast<int>(cta / S);
  const int split = static_cast<int>(cta - static_cast<long long>(j) * S);
  const int row = rows != nullptr ? rows[j] : j;
  if (row < 0) return;  // padding slot (block-uniform)
  const int v0 = split * kLogitsSplit;
  const typename VV::T* zr = z + static_cast<size_t>(row) * V;
  float m = -INFINITY, s = 0.f;
#pragma unroll
  for (int c0 = 0; c0 < ITERS; c0 += CHUNK) {
    uint4 raw[CHUNK];
#pragma unroll
    for (int i = 0; i < CHUNK; ++i) {
      const int v = v0 + ((c0 + i) * kLThreads + threadIdx.x) * W;
      // n_valid <= 0: nothing is read and every element is -inf
      raw[i] = VV::load_raw(zr + (v < V ? v : 0), V - v, VEC);
    }
    float cm;
    if (LLP_PACKED_MAX) {
      cm = VV::template max_of<CHUNK>(raw);
    } else {
      cm = -INFINITY;
#pragma unroll
      for (int i = 0; i < CHUNK; ++i) {
        float x[W];
        VV::unpack(raw[i], x);
#pragma unroll
        for (int k = 0; k < W; ++k) cm = fmaxf(cm, x[k]);
      }
    }
    if (cm == -INFINITY) continue;
    // x - cm first (exact near the maximum), so a large constant logit shift
    // costs no precision; the exponent of a logit far below the chunk maximum
    // may flush to zero, which changes the sum by less than one fp32 ulp
    float cs = 0.f;
#pragma unroll
    for (int i = 0; i < CHUNK; ++i) {
      float x[W];
      VV::unpack(raw[i], x);
#pragma unroll
      for (int k = 0; k < W; ++k) cs += ex2_approx((x[k] - cm) * kLog2eL);
    }
    merge_ms(m, s, cm, cs);
  }
  block_merge(m, s, sm_m, sm_s);
  if (threadIdx.x == 0) {
    part_m[static_cast<size_t>(split) * P + j] = m;
    part_s[static_cast<size_t>(split) * P + j] = s;
  }
}

template <int DT>
__global__ void __launch_bounds__(256) logits_merge_kernel(const typename Vec<DT>::T* __restrict__ z, int P, int V,
                                                           int S, const int* __restrict__ rows,
                                                           const long long* __restrict__ targets,
                                                           long long ignore_index, const float* __restrict__ part_m,
                                                           const float* __restrict__ part_s, float* __restrict__ logp,
                                                           float* __restrict__ row_max, float* __restrict__ log_sum) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= P) return;
  const int n = rows != nullptr ? rows[j] : j;
  if (n < 0) return;  // padding slot
  const long long t = targets[n];
  if (!tgt_ok(t, V, ignore_index)) {
    logp[n] = 0.f;
    row_max[n] = -INFINITY;
    log_sum[n] = 0.f;
    return;
  }
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, part_m[static_cast<size_t>(s) * P + j]);
  float Ssum = 0.f;
  for (int s = 0; s < S; ++s) {
    const size_t i = static_cast<size_t>(s) * P + j;
    Ssum += part_s[i] * exp2f((part_m[i] - M) * kLog2eL);
  }
  const float ls = logf(Ssum);
  const float zt = Vec<DT>::load1(z + static_cast<size_t>(n) * V + t);
  row_max[n] = M;
  log_sum[n] = ls;
  logp[n] = (zt - M) - ls;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kLThreads) logits_grad_kernel(const typename Vec<DT>::T* __restrict__ z, int N,
                                                                int V, int S, const long long* __restrict__ targets,
                                                                long long ignore_index,
                                                                const float* __restrict__ grad_logp,
                                                                const float* __restrict__ row_max,
                                                                const float* __restrict__ log_sum,
                                                                const unsigned char* __restrict__ mask,
                                                                typename Vec<DT>::T* __restrict__ grad) {
  using VV = Vec<DT>;
  constexpr int W = VV::W;
  constexpr int ITERS = kLogitsSplit / (kLThreads * W);
  const long long cta = blockIdx.x;
  const int row = static_cast<int>(cta / S);
  const int split = static_cast<int>(cta - static_cast<long long>(row) * S);
  const int v0 = split * kLogitsSplit;
  const typename VV::T* zr = z + static_cast<size_t>(row) * V;
  typename VV::T* gr = grad + static_cast<size_t>(row) * V;
  const long long t = targets[row];
  // a row outside the selection (mask given and 0) gets a zero gradient row
  const bool ok = tgt_ok(t, V, ignore_index) && (mask == nullptr || mask[row] != 0);
  const float g = ok ? grad_logp[row] : 0.f;
  const float m = ok ? row_max[row] : 0.f;
  const float ls = ok ? log_sum[row] : 0.f;
#pragma unroll 2
  for (int it = 0; it < ITERS; ++it) {
    const int v = v0 + (it * kLThreads + threadIdx.x) * W;
    if (v >= V) break;
    float x[W];
    const bool vec = VEC && v + W <= V;
    if (vec) {
      VV::load(zr + v, x);
    } else {
#pragma unroll
      for (int k = 0; k < W; ++k) x[k] = (v + k < V) ? VV::load1(zr + v + k) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const float p = ex2_approx(((x[k] - m) - ls) * kLog2eL);
      const float oh = (static_cast<long long>(v + k) == t) ? 1.f : 0.f;
      x[k] = ok ? g * (oh - p) : 0.f;
    }
    if (vec) {
      VV::store(gr + v, x);
    } else {
#pragma unroll
      for (int k = 0; k < W; ++k)
        if (v + k < V) VV::store1(gr + v + k, x[k]);
    }
  }
}

template <int DT>
cudaError_t launch_fwd_dt(const void* z, int P, const int* rows, int V, const long long* targets,
                          long long ignore_index, float* part, float* logp, float* row_max, float* log_sum, bool vec,
                          cudaStream_t s) {
  using T = typename Vec<DT>::T;
  const int S = (V + kLogitsSplit - 1) / kLogitsSplit;
  float* pm = part;
  float* ps = part + static_cast<size_t>(S) * P;
  const long long items = static_cast<long long>(P) * S;
  if (vec)
    logits_split_kernel<DT, true><<<static_cast<unsigned>(items), kLThreads, 0, s>>>(static_cast<const T*>(z), V, S,
                                                                                    P, rows, pm, ps);
  else
    logits_split_kernel<DT, false><<<static_cast<unsigned>(items), kLThreads, 0, s>>>(static_cast<const T*>(z), V, S,
                                                                                     P, rows, pm, ps);
  cudaError_t e = launch_result();
  if (e != cudaSuccess) return e;
  logits_merge_kernel<DT><<<(P + 255) / 256, 256, 0, s>>>(static_cast<const T*>(z), P, V, S, rows, targets,
                                                          ignore_index, pm, ps, logp, row_max, log_sum);
  return launch_result();
}

template <int DT>
cudaError_t launch_bwd_dt(const void* z, int N, int V, const long long* targets, long long ignore_index,
                          const float* grad_logp, const float* row_max, const float* log_sum,
                          const unsigned char* mask, void* grad, bool vec, cudaStream_t s) {
  using T = typename Vec<DT>::T;
  const int S = (V + kLogitsSplit - 1) / kLogitsSplit;
  const long long ctas = static_cast<long long>(N) * S;
  if (vec)
    logits_grad_kernel<DT, true><<<static_cast<unsigned>(ctas), kLThreads, 0, s>>>(
        static_cast<const T*>(z), N, V, S, targets, ignore_index, grad_logp, row_max, log_sum, mask,
        static_cast<T*>(grad));
  else
    logits_grad_kernel<DT, false><<<static_cast<unsigned>(ctas), kLThreads, 0, s>>>(
        static_cast<const T*>(z), N, V, S, targets, ignore_index, grad_logp, row_max, log_sum, mask,
        static_cast<T*>(grad));
  return launch_result();
}

}  // namespace

cudaError_t launch_logits_fwd(const void* z, int dtype, int P, const int* rows, int V, const long long* targets,
                              long long ignore_index, float* part, float* logp, float* row_max, float* log_sum,
                              bool vec, cudaStream_t s) {
  if (dtype == kDtypeF16)
    return launch_fwd_dt<kDtypeF16>(z, P, rows, V, targets, ignore_index, part, logp, row_max, log_sum, vec, s);
  return dtype == kDtypeBF16 ? launch_fwd_dt<kDtypeBF16>(z, P, rows, V, targets, ignore_index, part, logp, row_max,
                                                         log_sum, vec, s)
                             : launch_fwd_dt<kDtypeF32>(z, P, rows, V, targets, ignore_index, part, logp, row_max,
                                                        log_sum, vec, s);
}

cudaError_t launch_logits_bwd(const void* z, int dtype, int N, int V, const long long* targets,
                              long long ignore_index, const float* grad_logp, const float* row_max,
                              const float* log_sum, const unsigned char* mask, void* grad, bool vec,
                              cudaStream_t s) {
  if (dtype == kDtypeF16)
    return launch_bwd_dt<kDtypeF16>(z, N, V, targets, ignore_index, grad_logp, row_max, log_sum, mask, grad, vec, s);
  return dtype == kDtypeBF16 ? launch_bwd_dt<kDtypeBF16>(z, N, V, targets, ignore_index, grad_logp, row_max, log_sum,
                                                         mask, grad, vec, s)
                             : launch_bwd_dt<kDtypeF32>(z, N, V, targets, ignore_index, grad_logp, row_max, log_sum,
                                                        mask, grad, vec, s);
}

}  // namespace llp
