// grad_hidden for small batches (at most kSmallGhMaxN = 96 token rows), with the
// operands of the contraction swapped:
//
//     grad_hidden^T [D, N] = W^T [D, V] . dz^T [V, N]
//
// so that the hidden dimension sits on the MMA's M side (128 rows per CTA) and
// the few tokens on its N side (rounded up to 16).  The CTA-pair GEMM puts the
// tokens on M instead, so at N = 32 a 256-row tile holds 224 padding rows and
// the tensor pipe, not the weight stream, sets the pace.  Here no padding rows
// are multiplied, and the kernel is a pure stream of the weight.
//
// The vocab reduction keeps the fixed segments of the CTA-pair GEMM (32768
// vocab rows, partials summed afterwards in ascending order by the segment-sum
// kernel), and within a segment every output element accumulates the same
// 16-wide vocab slices in the same ascending order, in fp32 TMEM, starting from
// zero; only the roles of the two operands in each tcgen05.mma differ.  A unit
// is one (segment, 128-column hidden tile) pair: 4 x 21 = 84 units for the
// Nemotron head, one per SM.
//
// How the weight is streamed decides the speed.  An SM issues only about four
// tensor copies per microsecond from HBM whatever their size, so with 64 x 64
// boxes (8 KB, the CTA-pair GEMM's weight tiles) it pulls about 36 GB/s, and
// 84 SMs reach half the HBM bandwidth.  Here every stage of the weight is one
// 3-D copy of 128 vocab rows x 128 hidden columns (32 KB: the 64-column chunks
// of the row-major weight are the map's third dimension), and the ring holds
// as many stages as shared memory allows (six for up to 64 tokens), because
// past the copy count the bytes in flight set the rate.  dz (a few MB at these
// sizes, L2-resident) comes through a shallower ring of its own, also one copy
// per stage.
//
// Roles (224 threads): warp 0 = TMA producer of the weight, warp 6 = TMA
// producer of dz (each ring fills on its own, so the weight ring keeps all of
// its stages in flight however shallow the dz ring is), warp 1 = TMEM owner
// and MMA issuer, warps 2..5 = epilogue (warp w reads TMEM lanes
// 32 * (w % 4) + 0..31, one hidden column per thread, and stores one token per
// instruction: 32 consecutive fp32 columns, a coalesced 128-byte row segment).
// Every wait is bounded, as in the CTA-pair GEMM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "llp_internal.h"
#include "sm103_ptx.cuh"

namespace llp {

namespace {

constexpr int kSmThreads = 224;
constexpr int kSmTmemCols = 256;  // two accumulators of up to 128 token columns
constexpr int kSmBarBytes = 512;  // 4 rings of up to kSmallGhMaxStages barriers, 5 more, 2 words

// Per stage the weight ring holds kSmallGhRows vocab rows x 128 hidden columns
// (two 64-column chunks of kSmallGhRows x 128 bytes); a dz slot holds b_span stages' worth of
// vocab rows for all BN tokens.
__host__ __device__ inline int sm_a_box(const GhSmallParams&) { return kSmallGhRows * 128; }
__host__ __device__ inline int sm_a_stage(const GhSmallParams&) { return 2 * kSmallGhRows * 128; }

struct SmLayout {
  int a_off, b_off, bar_off, total;
};

__host__ __device__ inline SmLayout sm_layout(const GhSmallParams& p) {
  SmLayout L;
  L.a_off = 0;
  L.b_off = p.stages_a * sm_a_stage(p);
  L.bar_off = L.b_off + p.stages_b * p.b_slot_bytes;
  L.total = L.bar_off + kSmBarBytes + 1024;  // + alignment slack of the dynamic base
  return L;
}

__device__ __forceinline__ int sm_units(const GhSmallParams& p) { return p.nseg * p.num_dt; }

// weight stages of segment seg
__device__ __forceinline__ int sm_groups(const GhSmallParams& p, int seg) {
  const int len = min(kKSegment, p.V - seg * kKSegment);
  return (len + kSmallGhRows - 1) / kSmallGhRows;
}

__global__ void __launch_bounds__(kSmThreads, 1)
    gh_small_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_dz,
                    const GhSmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmLayout L = sm_layout(p);
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty_a = full_a + kSmallGhMaxStages;
  uint64_t* full_b = empty_a + kSmallGhMaxStages;
  uint64_t* empty_b = full_b + kSmallGhMaxStages;
  uint64_t* tmem_full = empty_b + kSmallGhMaxStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages_a; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&empty_a[s], 1);
    }
    for (int s = 0; s < p.stages_b; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 4);  // one arrive per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_dz);
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(tmem_slot, kSmTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int units = sm_units(p);
  const int a_stage = sm_a_stage(p);
  const int chunk_bytes = p.BN * 128;  // one 64-row vocab chunk of dz in a slot

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ---------------- producers: the weight (warp 0), dz (warp 6) ----------------
      // One copy per stage and operand: an SM issues only a handful of tensor
      // copies per microsecond from HBM, whatever their size.  A 3-D box lands
      // as its 64-column chunks one after another, exactly the layout of
      // separate 2-D boxes placed back to back.
      const bool weight = warp == 0;
      const uint64_t pol = weight ? l2_policy_evict_first()   // streamed once
                                  : l2_policy_evict_last();   // re-read by every hidden tile
      const int depth = weight ? p.stages_a : p.stages_b;
      const int rows = weight ? kSmallGhRows : kSmallGhRows * p.b_span;  // vocab rows per copy
      uint64_t* full = weight ? full_a : full_b;
      uint64_t* empty = weight ? empty_a : empty_b;
      int ga = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int seg = u / p.num_dt;
        const int dt = u - seg * p.num_dt;
        const int ng = sm_groups(p, seg);
        const int nc = weight ? ng : (ng + p.b_span - 1) / p.b_span;
        for (int g = 0; g < nc; ++g, ++ga) {
          const int sl = ga % depth;
          const uint32_t ph = static_cast<uint32_t>(ga / depth) & 1u;
          if (!mbar_wait(&empty[sl], ph ^ 1u, abort_flag, p.err, kDevTimeoutEmpty)) {
            ok = false;
            break;
          }
          const int v0 = seg * kKSegment + g * rows;
          if (weight) {
            const uint32_t sA = smem_u32(smem + L.a_off + sl * a_stage);
            mbar_arrive_expect_tx(&full[sl], static_cast<uint32_t>(a_stage));
            if (p.w_chunked) {
              tma_load_3d(sA, &tm_w, &full[sl], 0, v0, 2 * dt, pol);
            } else {
              tma_load_2d(sA, &tm_w, &full[sl], dt * 128, v0, pol);
              tma_load_2d(sA + sm_a_box(p), &tm_w, &full[sl], dt * 128 + 64, v0, pol);
            }
          } else {
            const uint32_t sB = smem_u32(smem + L.b_off + sl * p.b_slot_bytes);
            mbar_arrive_expect_tx(&full[sl], static_cast<uint32_t>(p.b_slot_bytes));
            tma_load_3d(sB, &tm_dz, &full[sl], 0, 0, v0 / 64, pol);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      // This thread's issue rate bounds the kernel: each 16-deep step of a
      // segment is one tcgen05.mma, and a segment's 2048 steps run one after
      // another on one SM.  So the loop keeps per-step work to two descriptor
      // additions (the start address is the low field, and no address here
      // carries out of it) and per-stage work to counter updates.
      const uint32_t idesc = make_idesc_16_f32(128, p.BN, /*a_mn=*/true, /*b_mn=*/false, p.f16 != 0);
      const uint64_t b_chunk = static_cast<uint64_t>(chunk_bytes >> 4);  // next 64-row chunk of dz
      int sa = 0, sb = 0, sub = 0;
      uint32_t pa = 0, pb = 0;
      uint32_t acc_i = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x, ++acc_i) {
        const int seg = u / p.num_dt;
        const int ng = sm_groups(p, seg);
        const uint32_t buf = acc_i & 1u;
        if (!mbar_wait(&tmem_empty[buf], ((acc_i >> 1) & 1u) ^ 1u, abort_flag, p.err, kDevTimeoutTmemEmpty))
          break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * 128;
        bool ok = true;
        for (int g = 0; g < ng; ++g) {
          if (!mbar_wait(&full_a[sa], pa, abort_flag, p.err, kDevTimeoutFull) ||
              (sub == 0 && !mbar_wait(&full_b[sb], pb, abort_flag, p.err, kDevTimeoutFull))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // A (weight, MN-major): 16 vocab rows = 2 KB further per step; the
          // second 64-column chunk is kSmallGhRows x 128 bytes on.  B (dz, K-major):
          // 64-row vocab chunks of BN token rows, 32 bytes per 16-wide step
          // inside a chunk.
          const uint64_t ad0 =
              make_smem_desc_sw128(smem_u32(smem + L.a_off + sa * a_stage), static_cast<uint32_t>(sm_a_box(p)), 1024);
          const uint64_t bd0 = make_smem_desc_sw128(
              smem_u32(smem + L.b_off + sb * p.b_slot_bytes) + sub * (kSmallGhRows / 64) * chunk_bytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kSmallGhRows / 16; ++kk) {
            const uint64_t ad = ad0 + static_cast<uint64_t>(kk * (2048 >> 4));
            const uint64_t bd = bd0 + static_cast<uint64_t>(kk >> 2) * b_chunk + static_cast<uint64_t>((kk & 3) * 2);
            umma_bf16_f32(d_tmem, ad, bd, idesc, (g > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty_a[sa]);
          if (++sa == p.stages_a) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sub == p.b_span || g == ng - 1) {  // the last stage that reads this dz slot
            umma_commit(&empty_b[sb]);
            sub = 0;
            if (++sb == p.stages_b) {
              sb = 0;
              pb ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit(&tmem_full[buf]);
      }
      umma_commit(drain);
      if (!mbar_wait_drain(drain, 0, 100000000ull)) atomicCAS(p.err, 0u, kDevTimeoutDrain);
    }
  } else if (warp <= 5) {
    // ---------------- epilogue ----------------
    const int lg = warp & 3;  // TMEM lane group of this warp
    uint32_t acc_i = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++acc_i) {
      const int seg = u / p.num_dt;
      const int dt = u - seg * p.num_dt;
      const uint32_t buf = acc_i & 1u;
      if (!mbar_wait(&tmem_full[buf], (acc_i >> 1) & 1u, abort_flag, p.err, kDevTimeoutTmemFull)) break;
      tc_fence_after_sync();
      const int d = dt * 128 + lg * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + buf * 128;
      for (int c0 = 0; c0 < p.N; c0 += 32) {
        float a[32];
        tmem_load_32cols(taddr + c0, a);
        if (d < p.D) {
          if (p.part != nullptr) {
            float* dst = p.part + (static_cast<size_t>(seg) * p.N + c0) * p.D + d;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < p.N) dst[static_cast<size_t>(j) * p.D] = a[j];
          } else {
            __nv_bfloat16* dst = p.out + static_cast<size_t>(c0) * p.D + d;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < p.N) {
                const float x = a[j];
                uint16_t bits;
                if (p.f16) {
                  const __half hv = __float2half_rn(x);
                  bits = *reinterpret_cast<const uint16_t*>(&hv);
                } else {
                  const __nv_bfloat16 bv = __float2bfloat16_rn(x);
                  bits = *reinterpret_cast<const uint16_t*>(&bv);
                }
                reinterpret_cast<uint16_t*>(dst)[static_cast<size_t>(j) * p.D] = bits;
              }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[buf]);
    }
  }

  tc_fence_before_sync();
  __syncwarp();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kSmTmemCols);
}

}  // namespace

bool small_grad_hidden_plan(int N, GhSmallParams* p) {
  if (N < 1 || N > kSmallGhMaxN) return false;
  p->N = N;
  p->BN = (N + 15) / 16 * 16;
  p->b_span = 1;
  p->b_slot_bytes = p->BN * 2 * kSmallGhRows * p->b_span;
  // dz: two slots where they leave room for two weight stages, else one; the
  // weight: as many stages as the rest of shared memory holds, since the bytes
  // in flight set the stream rate
  for (p->stages_b = 2; p->stages_b >= 1; --p->stages_b) {
    const int room = kSmallGhSmemLimit - kSmBarBytes - 1024 - p->stages_b * p->b_slot_bytes;
    p->stages_a = room / sm_a_stage(*p);
    if (p->stages_a > kSmallGhMaxStages) p->stages_a = kSmallGhMaxStages;
    if (p->stages_a >= 2) break;
  }
  return p->stages_b >= 1 && p->stages_a >= 2 && sm_layout(*p).total <= kSmallGhSmemLimit;
}

cudaError_t small_grad_hidden_setup() {
  return cudaFuncSetAttribute(gh_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallGhSmemLimit);
}

cudaError_t launch_small_grad_hidden(const CUtensorMap& tm_w, const CUtensorMap& tm_dz, const GhSmallParams& p,
                                     int num_sms, cudaStream_t s) {
  const int units = p.nseg * p.num_dt;
  const int grid = units < num_sms ? units : num_sms;
  gh_small_kernel<<<grid, kSmThreads, sm_layout(p).total, s>>>(tm_w, tm_dz, p);
  return launch_result();
}

}  // namespace llp
