// Warp-specialised, persistent tcgen05 GEMM core shared by every contraction
// of the fused linear log-prob path.
//
//   warp 0      : TMA producer (one elected lane) streaming A/B k-blocks into a
//                 ring of shared-memory stages, completion on mbarriers.
//   warp 1      : TMEM owner + MMA issuer (one elected lane): tcgen05.mma
//                 128 x BN x 16 bf16 -> fp32 into one of two TMEM accumulators.
//   warps 2..5  : epilogue; warp w reads TMEM lanes 32*(w%4)..+31, so each
//                 thread owns one accumulator row.  The epilogue of tile i
//                 overlaps the MMAs of tile i+1 (double-buffered TMEM).
//
// A unit of work is a run of `ntiles` consecutive BM x BN output tiles that
// share A rows (the forward's vocab split) or a single tile with a K range
// (a fixed K segment of the gradient GEMMs).  CTAs take units round-robin;
// which CTA runs a unit never changes any arithmetic, so results do not
// depend on the grid size, and every per-row / per-element reduction runs
// in a fixed order.
//
// Operand layouts (both 128-byte swizzled, as TMA writes them):
//   K-major  : box {64 K, R rows}; row pitch 128 B; 8-row groups 1024 B apart.
//   MN-major : R/64 boxes {64 MN, 64 K}, each 8 KB; 8-K-row groups 1024 B apart,
//              64-element MN chunks 8 KB apart.
#pragma once

#include "llp_internal.h"
#include "sm103_ptx.cuh"

namespace llp {

constexpr int BM = kTileM;
constexpr int BK = kTileK;
constexpr int UMMA_K = 16;
constexpr int kNumThreads = 192;
constexpr int kNumEpiThreads = 128;
constexpr int kTmemCols = 512;

struct UnitInfo {
  int m0;      // first A row (M coordinate) of the unit
  int n0;      // N coordinate of the unit's first tile
  int ntiles;  // tiles along N, each BN wide
  int kb0;     // first k-block (BK elements each)
  int nkb;     // k-blocks per tile
};

template <int BN_, int STAGES_, int EXTRA_>
struct SmemPlan {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN_ * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TILES_BYTES = STAGES_ * STAGE_BYTES;
  static constexpr int BAR_OFFSET = TILES_BYTES + EXTRA_;
  static constexpr int BAR_BYTES = 256;
  static constexpr int TOTAL = BAR_OFFSET + BAR_BYTES + 1024;  // + alignment slack
  static_assert(TOTAL <= 232448, "shared memory budget exceeded");
};

struct SharedState {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tmem_full;
  uint64_t* tmem_empty;
  uint64_t* drain;
  volatile int* abort;
  unsigned int* err;
  uint8_t* tiles;
  uint8_t* extra;
  uint32_t tmem_base;
};

// ----------------------------------------------------------------------------
// Producer: one lane of warp 0.
// ----------------------------------------------------------------------------
template <class Cfg>
__device__ __forceinline__ void run_producer(const SharedState& st, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                             const typename Cfg::Params& p) {
  using Plan = SmemPlan<Cfg::BN, Cfg::STAGES, Cfg::EXTRA_SMEM>;
  const uint64_t polA = Cfg::policy_a();
  const uint64_t polB = Cfg::policy_b();
  int stage = 0;
  uint32_t phase = 0;
  const int num_units = Cfg::num_units(p);
  for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
    const UnitInfo ui = Cfg::unit(p, u);
    for (int j = 0; j < ui.ntiles; ++j) {
      const int n0 = ui.n0 + j * Cfg::BN;
      for (int kb = 0; kb < ui.nkb; ++kb) {
        if (!mbar_wait(&st.empty[stage], phase ^ 1u, st.abort, st.err, kDevTimeoutEmpty)) return;
        const uint32_t sA = smem_u32(st.tiles + stage * Plan::STAGE_BYTES);
        const uint32_t sB = sA + Plan::A_BYTES;
        mbar_arrive_expect_tx(&st.full[stage], Plan::STAGE_BYTES);
        const int kx = (ui.kb0 + kb) * BK;
        if (!Cfg::A_MN) {
          tma_load_2d(sA, tmA, &st.full[stage], kx, ui.m0, polA);
        } else {
#pragma unroll
          for (int i = 0; i < BM / 64; ++i) tma_load_2d(sA + i * 8192, tmA, &st.full[stage], ui.m0 + 64 * i, kx, polA);
        }
        if (!Cfg::B_MN) {
          tma_load_2d(sB, tmB, &st.full[stage], kx, n0, polB);
        } else {
#pragma unroll
          for (int i = 0; i < Cfg::BN / 64; ++i) tma_load_2d(sB + i * 8192, tmB, &st.full[stage], n0 + 64 * i, kx, polB);
        }
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
}

// ----------------------------------------------------------------------------
// MMA issuer: one lane of warp 1.
// ----------------------------------------------------------------------------
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
  // K-major: advancing K by 16 bf16 = 32 bytes inside the 128-byte swizzle row.
  // MN-major: advancing K by 16 rows = 16 * 128 bytes; MN chunks 8 KB apart.
  return MN ? make_smem_desc_sw128(base + kk * (UMMA_K * 128), 8192, 1024)
            : make_smem_desc_sw128(base + kk * (UMMA_K * 2), 16, 1024);
}

template <class Cfg>
__device__ __forceinline__ void run_mma(const SharedState& st, const typename Cfg::Params& p) {
  using Plan = SmemPlan<Cfg::BN, Cfg::STAGES, Cfg::EXTRA_SMEM>;
  constexpr uint32_t idesc = make_idesc_bf16_f32(BM, Cfg::BN, Cfg::A_MN, Cfg::B_MN);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t acc_i = 0;
  const int num_units = Cfg::num_units(p);
  for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
    const UnitInfo ui = Cfg::unit(p, u);
    for (int j = 0; j < ui.ntiles; ++j, ++acc_i) {
      const uint32_t buf = acc_i & 1u;
      const uint32_t acc_phase = (acc_i >> 1) & 1u;
      if (!mbar_wait(&st.tmem_empty[buf], acc_phase ^ 1u, st.abort, st.err, kDevTimeoutTmemEmpty)) return;
      tc_fence_after_sync();
      const uint32_t d_tmem = st.tmem_base + buf * Cfg::BN;
      for (int kb = 0; kb < ui.nkb; ++kb) {
        if (!mbar_wait(&st.full[stage], phase, st.abort, st.err, kDevTimeoutFull)) return;
        tc_fence_after_sync();
        const uint32_t sA = smem_u32(st.tiles + stage * Plan::STAGE_BYTES);
        const uint32_t sB = sA + Plan::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          umma_bf16_f32(d_tmem, operand_desc<Cfg::A_MN>(sA, kk), operand_desc<Cfg::B_MN>(sB, kk), idesc,
                        (kb > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&st.empty[stage]);  // frees the stage once these MMAs have read it
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      umma_commit(&st.tmem_full[buf]);  // accumulator ready for the epilogue
    }
  }
}

// ----------------------------------------------------------------------------
// Epilogue: warps 2..5.
// ----------------------------------------------------------------------------
template <class Cfg>
__device__ __forceinline__ void run_epilogue(const SharedState& st, const typename Cfg::Params& p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = warp & 3;          // TMEM lane group this warp may access
  const int row = g * 32 + lane;   // accumulator row owned by this thread
  uint32_t acc_i = 0;
  const int num_units = Cfg::num_units(p);
  for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
    const UnitInfo ui = Cfg::unit(p, u);
    typename Cfg::RowState rs;
    Cfg::unit_begin(p, ui, u, row, rs);
    for (int j = 0; j < ui.ntiles; ++j, ++acc_i) {
      const uint32_t buf = acc_i & 1u;
      const uint32_t acc_phase = (acc_i >> 1) & 1u;
      if (!mbar_wait(&st.tmem_full[buf], acc_phase, st.abort, st.err, kDevTimeoutTmemFull)) return;
      tc_fence_after_sync();
      const uint32_t taddr = st.tmem_base + (static_cast<uint32_t>(g * 32) << 16) + buf * Cfg::BN;
      Cfg::tile(p, ui, u, j, row, g, lane, taddr, rs);
      tc_fence_before_sync();
      mbar_arrive(&st.tmem_empty[buf]);
    }
    Cfg::unit_end(p, ui, u, row, rs);
  }
}

template <class Cfg>
__global__ void __launch_bounds__(kNumThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const typename Cfg::Params p) {
  using Plan = SmemPlan<Cfg::BN, Cfg::STAGES, Cfg::EXTRA_SMEM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  SharedState st;
  st.tiles = smem;
  st.extra = smem + Plan::TILES_BYTES;
  st.full = reinterpret_cast<uint64_t*>(smem + Plan::BAR_OFFSET);
  st.empty = st.full + Cfg::STAGES;
  st.tmem_full = st.empty + Cfg::STAGES;
  st.tmem_empty = st.tmem_full + 2;
  st.drain = st.tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(st.drain + 1);
  st.abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  st.err = p.err;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&st.tmem_full[b], 1);
      mbar_init(&st.tmem_empty[b], kNumEpiThreads);
    }
    mbar_init(st.drain, 1);
    *st.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  st.tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) run_producer<Cfg>(st, &tmA, &tmB, p);
  } else if (warp == 1) {
    if (lane == 0) {
      run_mma<Cfg>(st, p);
      // Every MMA this thread issued must have finished before TMEM is freed,
      // also when a role gave up early.
      umma_commit(st.drain);
      if (!mbar_wait_drain(st.drain, 0, 100000000ull)) atomicCAS(st.err, 0u, kDevTimeoutDrain);
    }
  } else {
    run_epilogue<Cfg>(st, p);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(st.tmem_base, kTmemCols);
}

}  // namespace llp
