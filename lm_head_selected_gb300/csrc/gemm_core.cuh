// Warp-specialised, persistent tcgen05 GEMM core shared by every contraction
// of the fused linear log-prob path.
//
//   warp 0      : TMA producer (one lane) streaming A/B k-blocks into a ring of
//                 shared-memory stages, completion on mbarriers.
//   warp 1      : TMEM owner; one lane issues tcgen05.mma 16-deep steps into one
//                 of two fp32 TMEM accumulators (256 columns each).
//   warps 2..5  : epilogue; warp w reads TMEM lanes 32*(w%4)..+31, so each
//                 thread owns one accumulator row.  The epilogue of tile i
//                 overlaps the MMAs of tile i+1 (double-buffered TMEM).
//
// Two modes, chosen per configuration at compile time:
//   single CTA (PAIR = false): a CTA computes 128 x BN tiles on its own SM.
//   CTA pair   (PAIR = true) : a 2-CTA cluster computes 256 x BN tiles with
//       tcgen05.mma.cta_group::2 issued by the even CTA.  Each CTA loads its
//       own 128 rows of A and half (BN/2 rows) of B, so per CTA the shared
//       memory and L2 operand traffic per MMA falls by a third.  Both CTAs'
//       TMA loads complete on the even CTA's stage barrier; its commits are
//       multicast to both CTAs; the odd CTA's epilogue warps release an
//       accumulator with a remote arrive on the even CTA's barrier.
//
// A unit of work is a run of `ntiles` consecutive output tiles that share A
// rows (the forward's vocab split) or a single tile with a K range (a fixed K
// segment of the gradient GEMMs).  CTAs (or pairs) take units either
// round-robin (static) or, for configurations with DYNAMIC set and a launch
// given a ticket counter, in ascending order from that counter (the host gives
// one only when units are long enough to repay the hand-off, about a
// microsecond per unit): the pair's producer draws the ticket and
// hands the unit id to every other role through a small ring of slots in
// shared memory.  In-order claiming keeps the units that share operands
// running at the same time, so their operands are re-used from L2 instead of
// drifting apart over the launch.  Which CTA runs a unit never changes any
// arithmetic, so results do not depend on the grid size or on the schedule,
// and every per-row / per-element reduction runs in a fixed order.
//
// A unit's tiles are BN wide, or BN/2 (`UnitInfo::bn`, MN-major B only) for a
// last column tile with no more than BN/2 columns when LLP_HALF_TILE is set.
// It is off by default: the half-width MMA halves the compute per stage while
// the copy latency stays, and the stalls cost more than the padding saves.
//
// Operand layouts (both 128-byte swizzled, as TMA writes them):
//   K-major  : box {64 K, R rows}; row pitch 128 B; 8-row groups 1024 B apart.
//   MN-major : R/64 boxes {64 MN, 64 K}, each 8 KB; 8-K-row groups 1024 B apart,
//              64-element MN chunks 8 KB apart.  When the MN extent is a whole
//              number of 64-element chunks the operand comes as one 3-D copy
//              {64, 64 K, R/64 chunks} (the map's third dimension steps over
//              the chunks of a row), which lands in exactly that layout: an SM
//              issues only so many tensor copies per microsecond.
#pragma once

#include "llp_internal.h"
#include "sm103_ptx.cuh"

namespace llp {

// exp2 of the epilogues' softmax terms
__device__ __forceinline__ float epi_exp2(float x) { return LLP_EPI_FASTEXP ? ex2_approx(x) : exp2f(x); }

constexpr int BM = kTileM;  // accumulator rows per CTA
constexpr int BK = kTileK;
constexpr int UMMA_K = 16;
constexpr int kNumThreads = 192;
constexpr int kTmemCols = 512;

struct UnitInfo {
  int m0;      // first A row (M coordinate) of the unit (of the pair in pair mode)
  int n0;      // N coordinate of the unit's first tile
  int ntiles;  // tiles along N, each BN wide
  int kb0;     // first k-block (BK elements each)
  int nkb;     // k-blocks per tile
  int bn;      // MMA N of the unit's tiles: Cfg::BN, or Cfg::BN / 2 for a ragged last column tile
};

constexpr int kSchedDepth = 4;  // unit-id slots between the ticket drawer and the other roles
constexpr int kLockChunk = 16;                     // k-blocks between progress reports (advisory lockstep)
constexpr unsigned long long kLockMaxWaitNs = 20000;  // longest nap per report

template <class Cfg>
struct Plan {
  static constexpr bool PAIR = Cfg::PAIR;
  static constexpr int NCTA = PAIR ? 2 : 1;
  static constexpr int UM = NCTA * BM;                         // unit rows (M) per tile
  static constexpr int B_ROWS = PAIR ? Cfg::BN / 2 : Cfg::BN;  // B rows each CTA loads
  static constexpr int A_BYTES = Cfg::A_ROWS * BK * 2;  // A rows loaded per k-block (the MMA reads BM)
  static_assert(Cfg::A_ROWS == BM || (!PAIR && !Cfg::A_MN && A_BYTES + Cfg::BN * BK * 2 >= BM * BK * 2),
                "short A boxes: single CTA, K-major A, and the MMA's BM rows must stay inside the stage");
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TX_BYTES = NCTA * STAGE_BYTES;  // bytes landing per stage on the MMA's barrier
  static constexpr int TILES_BYTES = Cfg::STAGES * STAGE_BYTES;
  static constexpr int BAR_OFFSET = TILES_BYTES + Cfg::EXTRA_SMEM;
  static constexpr int BAR_BYTES = 256;
  static constexpr int TOTAL = BAR_OFFSET + BAR_BYTES + 1024;  // + alignment slack
  static constexpr int EPI_ARRIVALS = 4 * NCTA;                // one per epilogue warp of the pair
  // readers of a unit-id slot: MMA lane + 4 epilogue warps (+ the odd CTA's producer and 4 epilogue warps)
  static constexpr int SCHED_READERS = PAIR ? 10 : 5;
  static constexpr int BAR_USED = (2 * Cfg::STAGES + 5 + 2 * kSchedDepth) * 8 + 8 + 4 * kSchedDepth;
  static_assert(BAR_USED <= BAR_BYTES, "barrier region overflow");
  static_assert(TOTAL <= 232448, "shared memory budget exceeded");
  static_assert(B_ROWS % 64 == 0 && B_ROWS <= 256, "B half must be whole 64-row swizzle atoms");
};

struct SharedState {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tmem_full;
  uint64_t* tmem_empty;
  uint64_t* drain;
  uint64_t* sched_full;   // [kSchedDepth], this CTA: a unit id is in the slot
  uint64_t* sched_empty;  // [kSchedDepth], even CTA: every reader has taken the slot
  int* sched_slot;        // [kSchedDepth], this CTA
  volatile int* abort;
  unsigned int* err;
  uint8_t* tiles;
  uint8_t* extra;
  uint32_t tmem_base;
  uint32_t rank;    // CTA rank inside the pair (0 in single-CTA mode)
  int unit_first;   // first unit of this CTA (or pair)
  int unit_stride;  // number of CTAs (or pairs) in the grid
};

// ----------------------------------------------------------------------------
// Epilogue output path: each epilogue warp stages 32-row x 128-byte slabs of
// its accumulator rows in shared memory (two 4 KB buffers, 128-byte swizzled
// exactly as the store's tensor map expects: 16-byte chunk c of row r sits at
// chunk c ^ (r % 8)) and writes them with TMA tensor stores, so global writes
// leave the SM as whole lines instead of 32 scattered 16-byte pieces.
// ----------------------------------------------------------------------------
constexpr int kEpiStageBytes = 4096;
constexpr int kEpiSmemBytes = 4 * 2 * kEpiStageBytes;  // 4 epilogue warps x 2 buffers

struct EpiStore {
  const CUtensorMap* map;
  uint32_t buf0;  // this warp's first staging buffer (shared address, 1024-aligned)
  uint32_t next;  // buffer the next slab goes to
  int lane;
};

// Returns the staging buffer for the next slab once its previous store has read it.
__device__ __forceinline__ uint32_t epi_slab_begin(EpiStore& es) {
  if (es.lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  return es.buf0 + es.next * kEpiStageBytes;
}

// This lane's 16-byte chunk c (0..7) of its slab row.
__device__ __forceinline__ void epi_slab_put(uint32_t buf, int lane, int c, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  const uint32_t addr = buf + lane * 128 + ((static_cast<uint32_t>(c) ^ (lane & 7)) << 4);
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void epi_slab_store_2d(EpiStore& es, uint32_t buf, int x, int y) {
  fence_proxy_async_smem();
  __syncwarp();
  if (es.lane == 0) {
    tma_store_2d(es.map, buf, x, y);
    bulk_commit_group();
  }
  es.next ^= 1u;
}

// As epi_slab_store_2d, with an L2 eviction-priority hint (a createpolicy
// value): evict-first for an output that is streamed once through L2 (the bf16
// dlogits of a large batch), so it does not push out the operand tiles that the
// running units still re-read; evict-last for one that the next kernel re-reads
// from L2 (the dlogits of a small batch).
__device__ __forceinline__ void epi_slab_store_2d_hint(EpiStore& es, uint32_t buf, int x, int y, uint64_t policy) {
  fence_proxy_async_smem();
  __syncwarp();
  if (es.lane == 0) {
    tma_store_2d_hint(es.map, buf, x, y, policy);
    bulk_commit_group();
  }
  es.next ^= 1u;
}

__device__ __forceinline__ void epi_slab_store_3d(EpiStore& es, uint32_t buf, int x, int y, int z) {
  fence_proxy_async_smem();
  __syncwarp();
  if (es.lane == 0) {
    tma_store_3d(es.map, buf, x, y, z);
    bulk_commit_group();
  }
  es.next ^= 1u;
}

// ----------------------------------------------------------------------------
// Unit schedule.  The k-th unit of this CTA (pair) is >= 0 a unit id, -1 no
// more units, -2 a wait gave up (the caller returns).
// ----------------------------------------------------------------------------
// Even CTA's producer: publish unit `u` (or -1) as this pair's k-th unit.
template <class Cfg>
__device__ __forceinline__ int publish_unit(const SharedState& st, int k, int u) {
  const int s = k % kSchedDepth;
  const uint32_t ph = static_cast<uint32_t>(k / kSchedDepth) & 1u;
  if (!mbar_wait_cluster(&st.sched_empty[s], ph ^ 1u, st.abort, st.err, kDevTimeoutSched)) return -2;
  st.sched_slot[s] = u;
  mbar_arrive(&st.sched_full[s]);
  if (Plan<Cfg>::PAIR) {
    st_shared_cluster_u32(map_to_cta(smem_u32(&st.sched_slot[s]), 1), static_cast<uint32_t>(u));
    mbar_arrive_cluster(map_to_cta(smem_u32(&st.sched_full[s]), 1));  // release: orders the store above
  }
  return u;
}

// Any other role: take the k-th unit id from this CTA's slot and release the slot.
// With warp_wide, every lane of the warp calls it: lane 0 waits, reads and
// releases, and the id reaches the other lanes by shuffle.
template <class Cfg>
__device__ __forceinline__ int receive_unit(const SharedState& st, int k, bool warp_wide) {
  int u = -2;
  if (!warp_wide || (threadIdx.x & 31) == 0) {
    const int s = k % kSchedDepth;
    const uint32_t ph = static_cast<uint32_t>(k / kSchedDepth) & 1u;
    if (mbar_wait_cluster(&st.sched_full[s], ph, st.abort, st.err, kDevTimeoutSched)) {
      u = *reinterpret_cast<volatile int*>(&st.sched_slot[s]);
      if (Plan<Cfg>::PAIR)
        mbar_arrive_cluster(map_to_cta(smem_u32(&st.sched_empty[s]), 0));
      else
        mbar_arrive(&st.sched_empty[s]);
    }
  }
  if (warp_wide) u = __shfl_sync(0xffffffffu, u, 0);
  return u;
}

template <class Cfg>
__device__ __forceinline__ int static_unit(const SharedState& st, const typename Cfg::Params& p, int k) {
  const int u = st.unit_first + k * st.unit_stride;
  return u < Cfg::num_units(p) ? u : -1;
}

// ----------------------------------------------------------------------------
// Producer: one lane of warp 0 in every CTA.
// ----------------------------------------------------------------------------
// kps: k-blocks per stage, 1, or 2 when both operands come as 3-D copies of two
// k-blocks each (one copy per operand per stage; same bytes in flight).  A
// template parameter, so that each form compiles to straight-line code.
template <class Cfg, int kps>
__device__ __forceinline__ void run_producer_k(const SharedState& st, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                               const typename Cfg::Params& p) {
  using P = Plan<Cfg>;
  const uint64_t polA = Cfg::policy_a();
  const uint64_t polB = Cfg::policy_b();
  const bool leader = st.rank == 0;
  constexpr int nstages = Cfg::STAGES / kps;
  constexpr int stage_bytes = P::STAGE_BYTES * kps;
  int stage = 0;
  uint32_t phase = 0;
  const int num_units = Cfg::num_units(p);
  const bool dyn = Cfg::DYNAMIC && Cfg::sched_counter(p) != nullptr;
  int ticket = 0;
  if (dyn && leader) ticket = atomicAdd(Cfg::sched_counter(p), 1);
  // Advisory lockstep of in-order units: every kLockChunk k-blocks the pair adds
  // them to a shared progress counter and, while it is more than the window
  // ahead of the mean over all pairs, naps (at most kLockMaxWaitNs per check,
  // then goes on regardless).  Units that share operands then stream the same
  // K window at the same time and meet in L2.  Scheduling only: no wait here
  // decides anything about the arithmetic.
  unsigned int* const prog = dyn && leader ? Cfg::progress_counter(p) : nullptr;
  const unsigned int npairs = gridDim.x / P::NCTA;
  unsigned int mine = 0;
  for (int k = 0;; ++k) {
    int u;
    if (dyn)
      u = leader ? publish_unit<Cfg>(st, k, ticket < num_units ? ticket : -1) : receive_unit<Cfg>(st, k, false);
    else
      u = static_unit<Cfg>(st, p, k);
    if (u < 0) return;
    const UnitInfo ui = Cfg::unit(p, u);
    const int a_row = ui.m0 + static_cast<int>(st.rank) * BM;
    // B rows this CTA loads per k-block: half of the unit's N in pair mode
    const int b_rows = P::PAIR ? ui.bn / 2 : ui.bn;
    const uint32_t tx = static_cast<uint32_t>(P::NCTA * (P::A_BYTES + b_rows * BK * 2) * kps);
    // draw the next ticket a few k-blocks before the unit ends, so its latency
    // hides behind the loads still to issue
    const int draw_at = ui.nkb > 4 ? ui.nkb - 4 : 0;
    for (int j = 0; j < ui.ntiles; ++j) {
      const int b_row = ui.n0 + j * Cfg::BN + static_cast<int>(st.rank) * b_rows;
      for (int kb = 0; kb < ui.nkb; kb += kps) {
        if (dyn && leader && j == ui.ntiles - 1 && kb <= draw_at && draw_at < kb + kps)
          ticket = atomicAdd(Cfg::sched_counter(p), 1);
        if (prog != nullptr && ((kb + kps) % kLockChunk) == 0) {
          mine += kLockChunk;
          unsigned int total = atomicAdd(prog, static_cast<unsigned int>(kLockChunk)) + kLockChunk;
          // the last wave runs free: pairs without units stop reporting
          if (u + static_cast<int>(npairs) < num_units) {
            const unsigned long long t0 = global_timer_ns();
            const unsigned int win = static_cast<unsigned int>(LLP_LOCKSTEP);
            while (static_cast<unsigned long long>(mine) * npairs >
                   static_cast<unsigned long long>(total) + static_cast<unsigned long long>(win) * npairs) {
              if (global_timer_ns() - t0 > kLockMaxWaitNs) break;
              __nanosleep(256);
              total = *reinterpret_cast<volatile unsigned int*>(prog);
            }
          }
        }
        if (!mbar_wait(&st.empty[stage], phase ^ 1u, st.abort, st.err, kDevTimeoutEmpty)) return;
        const uint32_t sA = smem_u32(st.tiles + stage * stage_bytes);
        const uint32_t sB = sA + P::A_BYTES * kps;
        const int kx = (ui.kb0 + kb) * BK;
        // K-major with kps == 2: the 3-D map's third dimension steps over 64-wide
        // K chunks; MN-major chunked: over 64-wide MN chunks, K rows in the box
        if (P::PAIR) {
          if (leader) mbar_arrive_expect_tx(&st.full[stage], tx);
          const uint32_t bar = map_to_cta(smem_u32(&st.full[stage]), 0);
          if (!Cfg::A_MN) {
            if (kps == 2)
              tma_load_3d_pair(sA, tmA, bar, 0, a_row, kx / 64, polA);
            else
              tma_load_2d_pair(sA, tmA, bar, kx, a_row, polA);
          } else if (Cfg::a_chunked(p)) {
            tma_load_3d_pair(sA, tmA, bar, 0, kx, a_row / 64, polA);
          } else {
#pragma unroll
            for (int i = 0; i < BM / 64; ++i) tma_load_2d_pair(sA + i * 8192, tmA, bar, a_row + 64 * i, kx, polA);
          }
          if (!Cfg::B_MN) {
            if (kps == 2)
              tma_load_3d_pair(sB, tmB, bar, 0, b_row, kx / 64, polB);
            else
              tma_load_2d_pair(sB, tmB, bar, kx, b_row, polB);
          } else if (Cfg::b_chunked(p)) {
            tma_load_3d_pair(sB, tmB, bar, 0, kx, b_row / 64, polB);
          } else {
            for (int i = 0; i < b_rows / 64; ++i) tma_load_2d_pair(sB + i * 8192, tmB, bar, b_row + 64 * i, kx, polB);
          }
        } else {
          mbar_arrive_expect_tx(&st.full[stage], tx);
          if (!Cfg::A_MN) {
            if (kps == 2)
              tma_load_3d(sA, tmA, &st.full[stage], 0, a_row, kx / 64, polA);
            else
              tma_load_2d(sA, tmA, &st.full[stage], kx, a_row, polA);
          } else if (Cfg::a_chunked(p)) {
            tma_load_3d(sA, tmA, &st.full[stage], 0, kx, a_row / 64, polA);
          } else {
#pragma unroll
            for (int i = 0; i < BM / 64; ++i)
              tma_load_2d(sA + i * 8192, tmA, &st.full[stage], a_row + 64 * i, kx, polA);
          }
          if (!Cfg::B_MN) {
            if (kps == 2)
              tma_load_3d(sB, tmB, &st.full[stage], 0, b_row, kx / 64, polB);
            else
              tma_load_2d(sB, tmB, &st.full[stage], kx, b_row, polB);
          } else if (Cfg::b_chunked(p)) {
            tma_load_3d(sB, tmB, &st.full[stage], 0, kx, b_row / 64, polB);
          } else {
            for (int i = 0; i < b_rows / 64; ++i)
              tma_load_2d(sB + i * 8192, tmB, &st.full[stage], b_row + 64 * i, kx, polB);
          }
        }
        if (++stage == nstages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
}

template <class Cfg>
__device__ __forceinline__ void run_producer(const SharedState& st, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                             const typename Cfg::Params& p) {
  if (Cfg::kps(p) == 2)  // STAGES / 2 double stages (an odd last buffer goes unused)
    run_producer_k<Cfg, 2>(st, tmA, tmB, p);
  else
    run_producer_k<Cfg, 1>(st, tmA, tmB, p);
}

// ----------------------------------------------------------------------------
// MMA issuer: one lane of warp 1 (of the even CTA in pair mode).
// ----------------------------------------------------------------------------
// Descriptor of a stage's operand at its first 16-deep step.  K-major: rows of
// 128 bytes, 8-row groups 1024 B apart.  MN-major: 8-K-row groups 1024 B apart,
// 64-element MN chunks (64 * kps K rows of 128 B each) further on.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kps) {
  return MN ? make_smem_desc_sw128(base, 8192u * static_cast<uint32_t>(kps), 1024)
            : make_smem_desc_sw128(base, 16, 1024);
}

// How far the start-address field (16-byte units) moves for step kk (0..3) of
// the stage's k-block c: K-major, 32 bytes per step inside the swizzle row and
// a whole k-block tile (rows x 128 B) per k-block; MN-major, 16 K rows of 128 B
// per step.
template <bool MN>
__device__ __forceinline__ uint32_t operand_offset(int c, int kk, int rows) {
  return MN ? static_cast<uint32_t>(((c * 4 + kk) * UMMA_K * 128) >> 4)
            : static_cast<uint32_t>((c * rows * 128 + kk * UMMA_K * 2) >> 4);
}

template <class Cfg, int kps>
__device__ __forceinline__ void run_mma_k(const SharedState& st, const typename Cfg::Params& p) {
  using P = Plan<Cfg>;
  // both operands have the same 16-bit type (the params' f16 flag)
  const uint32_t idesc_full = make_idesc_16_f32(P::UM, Cfg::BN, Cfg::A_MN, Cfg::B_MN, p.f16 != 0);
  const uint32_t idesc_half = make_idesc_16_f32(P::UM, Cfg::BN / 2, Cfg::A_MN, Cfg::B_MN, p.f16 != 0);
  constexpr int nstages = Cfg::STAGES / kps;
  constexpr int stage_bytes = P::STAGE_BYTES * kps;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t acc_i = 0;
  const bool dyn = Cfg::DYNAMIC && Cfg::sched_counter(p) != nullptr;
  for (int k = 0;; ++k) {
    int u;
    if (dyn)
      u = receive_unit<Cfg>(st, k, false);
    else
      u = static_unit<Cfg>(st, p, k);
    if (u < 0) return;
    const UnitInfo ui = Cfg::unit(p, u);
    const uint32_t idesc = ui.bn == Cfg::BN ? idesc_full : idesc_half;
    for (int j = 0; j < ui.ntiles; ++j, ++acc_i) {
      const uint32_t buf = acc_i & 1u;
      const uint32_t acc_phase = (acc_i >> 1) & 1u;
      if (!mbar_wait(&st.tmem_empty[buf], acc_phase ^ 1u, st.abort, st.err, kDevTimeoutTmemEmpty)) return;
      tc_fence_after_sync();
      const uint32_t d_tmem = st.tmem_base + buf * Cfg::BN;
      for (int kb = 0; kb < ui.nkb; kb += kps) {
        if (!mbar_wait(&st.full[stage], phase, st.abort, st.err, kDevTimeoutFull)) return;
        tc_fence_after_sync();
        const uint32_t sA = smem_u32(st.tiles + stage * stage_bytes);
        const uint32_t sB = sA + P::A_BYTES * kps;
        // descriptors of the stage's first step; each further step only moves
        // the start address (the low field, which no address here carries out of)
        const uint64_t ad0 = operand_desc<Cfg::A_MN>(sA, kps);
        const uint64_t bd0 = operand_desc<Cfg::B_MN>(sB, kps);
#pragma unroll
        for (int c = 0; c < kps; ++c) {
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t ad = ad0 + operand_offset<Cfg::A_MN>(c, kk, Cfg::A_ROWS);
            const uint64_t bd = bd0 + operand_offset<Cfg::B_MN>(c, kk, P::B_ROWS);
            const uint32_t acc = (kb > 0 || c > 0 || kk > 0) ? 1u : 0u;
            if (P::PAIR)
              umma_bf16_f32_pair(d_tmem, ad, bd, idesc, acc);
            else
              umma_bf16_f32(d_tmem, ad, bd, idesc, acc);
          }
        }
        // frees the stage (in both CTAs) once these MMAs have read it
        if (P::PAIR)
          umma_commit_pair_multicast(&st.empty[stage], 0x3);
        else
          umma_commit(&st.empty[stage]);
        if (++stage == nstages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // accumulator ready for the epilogue (of both CTAs)
      if (P::PAIR)
        umma_commit_pair_multicast(&st.tmem_full[buf], 0x3);
      else
        umma_commit(&st.tmem_full[buf]);
    }
  }
}

template <class Cfg>
__device__ __forceinline__ void run_mma(const SharedState& st, const typename Cfg::Params& p) {
  if (Cfg::kps(p) == 2)
    run_mma_k<Cfg, 2>(st, p);
  else
    run_mma_k<Cfg, 1>(st, p);
}

// ----------------------------------------------------------------------------
// Epilogue: warps 2..5 of every CTA.
// ----------------------------------------------------------------------------
template <class Cfg>
__device__ __forceinline__ void run_epilogue(const SharedState& st, const CUtensorMap* tmC,
                                             const typename Cfg::Params& p) {
  using P = Plan<Cfg>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = warp & 3;                                          // TMEM lane group of this warp
  const int row = static_cast<int>(st.rank) * BM + g * 32 + lane;  // accumulator row within the unit
  EpiStore es;
  es.map = tmC;
  es.buf0 = smem_u32(st.extra) + static_cast<uint32_t>(g) * 2u * kEpiStageBytes;
  es.next = 0;
  es.lane = lane;
  uint32_t acc_i = 0;
  bool ok = true;
  const bool dyn = Cfg::DYNAMIC && Cfg::sched_counter(p) != nullptr;
  for (int k = 0; ok; ++k) {
    int u;
    if (dyn)
      u = receive_unit<Cfg>(st, k, true);
    else
      u = static_unit<Cfg>(st, p, k);
    if (u < 0) break;
    const UnitInfo ui = Cfg::unit(p, u);
    typename Cfg::RowState rs;
    Cfg::unit_begin(p, ui, u, row, rs);
    for (int j = 0; j < ui.ntiles; ++j, ++acc_i) {
      const uint32_t buf = acc_i & 1u;
      const uint32_t acc_phase = (acc_i >> 1) & 1u;
      if (!mbar_wait(&st.tmem_full[buf], acc_phase, st.abort, st.err, kDevTimeoutTmemFull)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t taddr = st.tmem_base + (static_cast<uint32_t>(g * 32) << 16) + buf * Cfg::BN;
      Cfg::tile(p, ui, u, j, row, lane, taddr, rs, es);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (P::PAIR)
          // CTA-scope arrive: the tcgen05 fence above orders the TMEM reads; a
          // cluster-scope release here was the top stall of short-unit launches
          mbar_arrive_remote(map_to_cta(smem_u32(&st.tmem_empty[buf]), 0));
        else
          mbar_arrive(&st.tmem_empty[buf]);
      }
    }
    if (ok) Cfg::unit_end(p, ui, u, row, rs);
  }
  // every tensor store of this warp must be complete before the CTA exits
  if (lane == 0) bulk_wait_group_all();
  __syncwarp();
}

template <class Cfg>
__global__ void __launch_bounds__(kNumThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const typename Cfg::Params p) {
  using P = Plan<Cfg>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  SharedState st;
  st.tiles = smem;
  st.extra = smem + P::TILES_BYTES;
  st.full = reinterpret_cast<uint64_t*>(smem + P::BAR_OFFSET);
  st.empty = st.full + Cfg::STAGES;
  st.tmem_full = st.empty + Cfg::STAGES;
  st.tmem_empty = st.tmem_full + 2;
  st.drain = st.tmem_empty + 2;
  st.sched_full = st.drain + 1;
  st.sched_empty = st.sched_full + kSchedDepth;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(st.sched_empty + kSchedDepth);
  st.abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  st.sched_slot = reinterpret_cast<int*>(tmem_slot + 2);
  st.err = p.err;
  st.rank = P::PAIR ? cluster_ctarank() : 0u;
  st.unit_first = static_cast<int>(blockIdx.x) / P::NCTA;
  st.unit_stride = static_cast<int>(gridDim.x) / P::NCTA;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&st.tmem_full[b], 1);
      mbar_init(&st.tmem_empty[b], P::EPI_ARRIVALS);
    }
    mbar_init(st.drain, 1);
    for (int s = 0; s < kSchedDepth; ++s) {
      mbar_init(&st.sched_full[s], 1);
      mbar_init(&st.sched_empty[s], P::SCHED_READERS);
    }
    *st.abort = 0;
    fence_mbarrier_init();
    if (blockIdx.x == 0) Cfg::on_launch(p);
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Cfg::EXTRA_SMEM > 0) tma_prefetch_desc(&tmC);
  }
  __syncwarp();  // the .aligned barriers and tcgen05 allocation below need converged warps
  if (warp == 1) {
    if (P::PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_alloc_permit_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish_alloc_permit();
    }
  }
  tc_fence_before_sync();
  // the peer's TMA loads and arrives target this CTA's barriers: both CTAs
  // must have initialised them before either starts
  if (P::PAIR)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after_sync();
  st.tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) run_producer<Cfg>(st, &tmA, &tmB, p);
  } else if (warp == 1) {
    if (lane == 0 && st.rank == 0) {
      run_mma<Cfg>(st, p);
      // Every MMA this thread issued must have finished before TMEM is freed,
      // also when a role gave up early.
      if (P::PAIR)
        umma_commit_pair(st.drain);
      else
        umma_commit(st.drain);
      if (!mbar_wait_drain(st.drain, 0, 100000000ull)) atomicCAS(st.err, 0u, kDevTimeoutDrain);
    }
  } else {
    run_epilogue<Cfg>(st, &tmC, p);
  }

  tc_fence_before_sync();
  __syncwarp();  // lanes that skipped a role wait here for the one that ran it
  // neither CTA of a pair may free TMEM or exit while the other can still
  // touch its shared memory or TMEM
  if (P::PAIR)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    if (P::PAIR)
      tmem_dealloc_pair(st.tmem_base, kTmemCols);
    else
      tmem_dealloc(st.tmem_base, kTmemCols);
  }
}

// Launch helper: pair configurations run as 2-CTA clusters.
template <class Cfg>
inline cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                               const typename Cfg::Params& p, int grid, cudaStream_t s) {
  using P = Plan<Cfg>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = P::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P::NCTA;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return note_cuda(cudaLaunchKernelEx(&cfg, tc_gemm_kernel<Cfg>, a, b, c, p));
}

// One-time set-up per kernel: shared-memory opt-in and the number of clusters
// (CTAs in single mode) that can be resident at once, which bounds the grid of
// the persistent kernel so that no CTA waits for a second wave.
template <class Cfg>
inline cudaError_t setup_gemm(int* resident_groups) {
  using P = Plan<Cfg>;
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, P::TOTAL);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P::NCTA, 1, 1);
  cfg.blockDim = dim3(kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = P::TOTAL;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P::NCTA;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int groups = 0;
  e = cudaOccupancyMaxActiveClusters(&groups, tc_gemm_kernel<Cfg>, &cfg);
  if (e != cudaSuccess) return e;
  if (groups < 1) return cudaErrorInvalidConfiguration;
  *resident_groups = groups;
  return cudaSuccess;
}

}  // namespace llp
