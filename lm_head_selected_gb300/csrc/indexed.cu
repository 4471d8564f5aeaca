// Row-subset ("indexed") support: only the rows named by an index list are
// computed ("recursive deterministic LogP autograd on B200", What: indexed
// semantics keep the full output row shape, duplicate indices are idempotent,
// out-of-range indices are ignored, unselected rows have zero derivatives;
// "add backward support for fused logp CUDA kernels", Implementation details:
// exactly zero gradients for rows omitted by indexed variants).
//
// The index list becomes a byte mask over the N rows (duplicates set the same
// byte), then a deterministic compaction lists the selected rows in ascending
// order: per-block counts, one exclusive scan, per-block placement.  The list is
// padded to K slots with -1, so every later launch has a size known on the host
// (no device-to-host read).
#include <cuda_bf16.h>

#include "llp_internal.h"

namespace llp {

namespace {

constexpr int kScanBlock = 1024;  // rows per compaction block

__global__ void mark_rows_kernel(const long long* __restrict__ idx, long long K, long long N,
                                 unsigned char* __restrict__ mask) {
  const long long k = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (k >= K) return;
  const long long i = idx[k];
  if (i >= 0 && i < N) mask[i] = 1;  // duplicates write the same byte
}

__global__ void __launch_bounds__(kScanBlock) count_rows_kernel(const unsigned char* __restrict__ mask, int N,
                                                                int* __restrict__ counts) {
  __shared__ int warp_sums[kScanBlock / 32];
  const int i = blockIdx.x * kScanBlock + threadIdx.x;
  const int v = (i < N) ? mask[i] : 0;
  const int w = __popc(__ballot_sync(0xffffffffu, v != 0));
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = w;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int k = 0; k < kScanBlock / 32; ++k) s += warp_sums[k];
    counts[blockIdx.x] = s;
  }
}

// Exclusive scan of the block counts in one CTA (ascending block order); the
// total number of selected rows goes to *total.
__global__ void __launch_bounds__(1024) scan_counts_kernel(int* __restrict__ counts, int nblocks,
                                                           int* __restrict__ total) {
  __shared__ int carry;
  __shared__ int warp_sums[32];
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < nblocks; base += 1024) {
    const int i = base + threadIdx.x;
    const int v = (i < nblocks) ? counts[i] : 0;
    int x = v;  // inclusive scan within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if ((threadIdx.x & 31) >= off) x += y;
    }
    if ((threadIdx.x & 31) == 31) warp_sums[threadIdx.x >> 5] = x;
    __syncthreads();
    if (threadIdx.x < 32) {
      int ws = warp_sums[threadIdx.x];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, ws, off);
        if (threadIdx.x >= off) ws += y;
      }
      warp_sums[threadIdx.x] = ws;  // inclusive
    }
    __syncthreads();
    const int warp_off = (threadIdx.x >> 5) ? warp_sums[(threadIdx.x >> 5) - 1] : 0;
    if (i < nblocks) counts[i] = carry + warp_off + x - v;  // exclusive
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sums[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) *total = carry;
}

__global__ void __launch_bounds__(kScanBlock) place_rows_kernel(const unsigned char* __restrict__ mask, int N,
                                                                const int* __restrict__ offsets,
                                                                int* __restrict__ rows) {
  __shared__ int warp_sums[kScanBlock / 32];
  const int i = blockIdx.x * kScanBlock + threadIdx.x;
  const int v = (i < N) ? mask[i] : 0;
  const unsigned bal = __ballot_sync(0xffffffffu, v != 0);
  const int lane = threadIdx.x & 31;
  const int before_in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_sums[threadIdx.x >> 5] = __popc(bal);
  __syncthreads();
  int warp_off = 0;
  for (int k = 0; k < (threadIdx.x >> 5); ++k) warp_off += warp_sums[k];
  if (v) rows[offsets[blockIdx.x] + warp_off + before_in_warp] = i;
}

// Slots j >= total get row -1.
__global__ void pad_rows_kernel(int* __restrict__ rows, int K, const int* __restrict__ total) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < K && j >= *total) rows[j] = -1;
}

// Compact copies of the per-row inputs; padded slots get an ignored target.
__global__ void gather_rows_kernel(const int* __restrict__ rows, int K, int D, const __nv_bfloat16* __restrict__ hidden,
                                   const long long* __restrict__ targets, const float* __restrict__ temperature,
                                   const float* __restrict__ grad_logp, const float* __restrict__ lse,
                                   long long ignore_index, __nv_bfloat16* __restrict__ c_hidden,
                                   long long* __restrict__ c_targets, float* __restrict__ c_temperature,
                                   float* __restrict__ c_grad, float* __restrict__ c_lse) {
  const int j = blockIdx.x;
  const int r = rows[j];
  const int vecs = D / 8;  // D % 8 == 0: rows are whole 16-byte vectors
  uint4* dst = reinterpret_cast<uint4*>(c_hidden + static_cast<size_t>(j) * D);
  if (r >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(r) * D);
    for (int k = threadIdx.x; k < vecs; k += blockDim.x) dst[k] = src[k];
  } else {
    for (int k = threadIdx.x; k < vecs; k += blockDim.x) dst[k] = make_uint4(0, 0, 0, 0);
  }
  if (threadIdx.x == 0) {
    c_targets[j] = (r >= 0) ? targets[r] : ignore_index;
    if (c_temperature) c_temperature[j] = (r >= 0 && temperature) ? temperature[r] : 1.f;
    if (c_grad) c_grad[j] = (r >= 0) ? grad_logp[r] : 0.f;
    if (c_lse) c_lse[j] = (r >= 0) ? lse[r] : 0.f;
  }
}

__global__ void scatter_outputs_kernel(const int* __restrict__ rows, int K, const float* __restrict__ c_logp,
                                       const float* __restrict__ c_lse, float* __restrict__ logp,
                                       float* __restrict__ lse) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  const int r = rows[j];
  if (r < 0) return;
  logp[r] = c_logp[j];
  lse[r] = c_lse[j];
}

// grad_hidden [N, D]: selected rows from the compact result, all other rows zero.
__global__ void scatter_grad_hidden_kernel(const unsigned char* __restrict__ mask, const int* __restrict__ slot_of,
                                           int N, int D, const __nv_bfloat16* __restrict__ c_gh,
                                           __nv_bfloat16* __restrict__ gh) {
  const int r = blockIdx.x;
  const int vecs = D / 8;
  uint4* dst = reinterpret_cast<uint4*>(gh + static_cast<size_t>(r) * D);
  if (mask[r]) {
    const uint4* src = reinterpret_cast<const uint4*>(c_gh + static_cast<size_t>(slot_of[r]) * D);
    for (int k = threadIdx.x; k < vecs; k += blockDim.x) dst[k] = src[k];
  } else {
    for (int k = threadIdx.x; k < vecs; k += blockDim.x) dst[k] = make_uint4(0, 0, 0, 0);
  }
}

__global__ void slot_of_kernel(const int* __restrict__ rows, int K, int* __restrict__ slot_of) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  const int r = rows[j];
  if (r >= 0) slot_of[r] = j;
}

}  // namespace

size_t select_workspace_bytes(long long N, long long K) {
  const long long nb = (N + kScanBlock - 1) / kScanBlock;
  const long long Kc = K < N ? K : N;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(static_cast<size_t>(N)) + up(static_cast<size_t>(nb + 1) * 4) + up(static_cast<size_t>(Kc) * 4) +
         up(static_cast<size_t>(N) * 4);
}

cudaError_t build_row_selection(const long long* idx, long long K, int N, void* ws, RowSelection* sel,
                                 cudaStream_t s) {
  const int nb = (N + kScanBlock - 1) / kScanBlock;
  const long long Kc = K < N ? K : N;  // at most N distinct rows can be selected
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* p = static_cast<uint8_t*>(ws);
  sel->mask = p;
  p += up(static_cast<size_t>(N));
  int* counts = reinterpret_cast<int*>(p);
  sel->total = counts + nb;
  p += up(static_cast<size_t>(nb + 1) * 4);
  sel->rows = reinterpret_cast<int*>(p);
  p += up(static_cast<size_t>(Kc) * 4);
  sel->slot_of = reinterpret_cast<int*>(p);
  sel->K = static_cast<int>(Kc);
  cudaError_t e = cudaMemsetAsync(sel->mask, 0, static_cast<size_t>(N), s);
  if (e != cudaSuccess) return e;
  if (K > 0) {
    mark_rows_kernel<<<static_cast<unsigned>((K + 255) / 256), 256, 0, s>>>(idx, K, N, sel->mask);
    if ((e = launch_result()) != cudaSuccess) return e;
  }
  count_rows_kernel<<<nb, kScanBlock, 0, s>>>(sel->mask, N, counts);
  if ((e = launch_result()) != cudaSuccess) return e;
  scan_counts_kernel<<<1, 1024, 0, s>>>(counts, nb, sel->total);
  if ((e = launch_result()) != cudaSuccess) return e;
  place_rows_kernel<<<nb, kScanBlock, 0, s>>>(sel->mask, N, counts, sel->rows);
  if ((e = launch_result()) != cudaSuccess) return e;
  if (K > 0) {
    pad_rows_kernel<<<(sel->K + 255) / 256, 256, 0, s>>>(sel->rows, sel->K, sel->total);
    if ((e = launch_result()) != cudaSuccess) return e;
    slot_of_kernel<<<(sel->K + 255) / 256, 256, 0, s>>>(sel->rows, sel->K, sel->slot_of);
    e = launch_result();
  }
  return e;
}

cudaError_t gather_selected_rows(const RowSelection& sel, int D, const __nv_bfloat16* hidden,
                                 const long long* targets, const float* temperature, const float* grad_logp,
                                 const float* lse, long long ignore_index, __nv_bfloat16* c_hidden,
                                 long long* c_targets, float* c_temperature, float* c_grad, float* c_lse,
                                 cudaStream_t s) {
  if (sel.K == 0) return cudaSuccess;
  gather_rows_kernel<<<sel.K, 128, 0, s>>>(sel.rows, sel.K, D, hidden, targets, temperature, grad_logp, lse,
                                           ignore_index, c_hidden, c_targets, c_temperature, c_grad, c_lse);
  return launch_result();
}

cudaError_t scatter_selected_outputs(const RowSelection& sel, const float* c_logp, const float* c_lse, float* logp,
                                     float* lse, cudaStream_t s) {
  if (sel.K == 0) return cudaSuccess;
  scatter_outputs_kernel<<<(sel.K + 255) / 256, 256, 0, s>>>(sel.rows, sel.K, c_logp, c_lse, logp, lse);
  return launch_result();
}

cudaError_t scatter_selected_grad_hidden(const RowSelection& sel, int N, int D, const __nv_bfloat16* c_gh,
                                         __nv_bfloat16* gh, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  scatter_grad_hidden_kernel<<<N, 128, 0, s>>>(sel.mask, sel.slot_of, N, D, c_gh, gh);
  return launch_result();
}

}  // namespace llp
