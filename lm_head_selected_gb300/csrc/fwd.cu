// Forward of the fused linear selected-token log-probability on tcgen05.
//
//   F1  per (128-token tile, 512-column vocab split):
//         acc = h_tile . W_tile^T on the tensor cores (bf16 in, fp32 in TMEM),
//         z = (acc + b[v]) * (1/tau_n), folded into a per-row online max/sum,
//         with z[t_n] captured as the tile holding t_n passes.  Only the
//         per-split (max, sum) pair and the target logit leave the SM; the
//         [N, V] logits never reach global memory.
//   F2  per row: merge the splits in ascending order,
//         M = max_s m_s,  S = sum_s s_s * exp(m_s - M),
//         lse = M + log S,  logp = (z_t - M) - log S.
//
// Semantics follow "Fused Linear LogP" (Reference Semantics, Tensor Contract):
// logp = z[target] - logsumexp(z); the per-row temperature of "Feat/nemotron h
// lm head logprob cuda" divides the biased logit; invalid targets (ignore index
// or outside [0, V)) give logp = 0 and lse = -inf ("recursive deterministic
// LogP autograd on B200", Summary), without any read at the target index.
// The final expression keeps target - max - log(sum) apart, as the
// deterministic forward in "recursive deterministic LogP autograd on B200"
// (Prior art table) does.
#include "gemm_core.cuh"

namespace llp {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool target_valid(long long t, int V, long long ignore_index) {
  return t != ignore_index && t >= 0 && t < static_cast<long long>(V);
}

// PAIRED = false: single CTAs with 128-row tiles, used when the whole batch fits
// in one of them (a pair's second CTA would hold only padding rows).  AROWS:
// hidden rows loaded per stage (kSmallARows for a batch that small).
template <bool HAS_BIAS, bool PAIRED = kPairMMA, int AROWS = kTileM>
struct FwdCfg {
  static constexpr bool A_MN = false;
  static constexpr bool B_MN = false;
  static constexpr bool PAIR = PAIRED;
  static constexpr int BN = kTileN;
  static constexpr int A_ROWS = AROWS;
  static constexpr int STAGES = PAIR ? kPairStages : (AROWS < kTileM ? kSmallAFwdStages : 4);
  static constexpr int EXTRA_SMEM = 0;
  static constexpr int TPS = kTilesPerSplit;
  static constexpr int UM = PAIR ? kUnitM : kTileM;
  using Params = FwdParams;

  struct RowState {
    float m;        // running max over the split
    float s;        // running sum of exp(z - m)
    float zt;       // captured target logit
    float inv_tau;  // 1 / tau for this row
    int tloc;       // target column relative to the unit's first column (may be out of range)
    int n;          // token row
  };

  static __device__ __forceinline__ uint64_t policy_a() { return l2_policy_evict_last(); }
  static __device__ __forceinline__ uint64_t policy_b() { return l2_policy_evict_normal(); }
  static constexpr bool DYNAMIC = false;
  static __device__ __forceinline__ int* sched_counter(const Params&) { return nullptr; }
  static __device__ __forceinline__ unsigned int* progress_counter(const Params&) { return nullptr; }
  static __device__ __forceinline__ bool a_chunked(const Params&) { return false; }
  static __device__ __forceinline__ bool b_chunked(const Params&) { return false; }
  static __device__ __forceinline__ int kps(const Params& p) { return p.kps; }
  static __device__ __forceinline__ void on_launch(const Params&) {}

  static __device__ __forceinline__ int num_units(const Params& p) { return p.num_m * p.num_splits; }

  // Raster: groups of group_m token tiles; inside a group the vocab split is the
  // slow index, so concurrently running CTAs share the same weight tiles in L2.
  static __device__ __forceinline__ UnitInfo unit(const Params& p, int u) {
    const int gsize = p.group_m * p.num_splits;
    const int grp = u / gsize;
    const int r = u - grp * gsize;
    const int gm = min(p.group_m, p.num_m - grp * p.group_m);
    const int split = r / gm;
    const int mt = grp * p.group_m + (r - split * gm);
    UnitInfo ui;
    ui.m0 = mt * UM;
    ui.n0 = split * TPS * BN;
    ui.ntiles = min(TPS, p.num_vt - split * TPS);
    ui.kb0 = 0;
    ui.nkb = (p.D + BK - 1) / BK;
    ui.bn = BN;
    return ui;
  }

  static __device__ __forceinline__ void unit_begin(const Params& p, const UnitInfo& ui, int, int row, RowState& rs) {
    rs.n = ui.m0 + row;
    rs.m = -INFINITY;
    rs.s = 0.f;
    rs.zt = 0.f;
    rs.inv_tau = 1.f;
    rs.tloc = -1;
    if (rs.n < p.N) {
      // local vocab id of the target (this weight may be a vocab shard starting at vocab_start)
      const long long t = p.targets[rs.n];
      const long long tl = t - p.vocab_start;
      if (t != p.ignore_index && tl >= 0 && tl < static_cast<long long>(p.V)) rs.tloc = static_cast<int>(tl - ui.n0);
      if (p.temperature != nullptr) rs.inv_tau = __frcp_rn(p.temperature[rs.n]);
    }
  }

  static __device__ __forceinline__ void tile(const Params& p, const UnitInfo& ui, int, int j, int, int,
                                              uint32_t taddr, RowState& rs, EpiStore&) {
    const int v0 = ui.n0 + j * BN;
    const bool full = (v0 + BN) <= p.V;
    // a bias slice (a vocab shard's) may start at any float: vector loads only when 16-byte aligned
    const bool bias_vec = full && (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0;
    const int tl = rs.tloc - j * BN;
    const bool mine = (tl >= 0) && (tl < BN);
    const bool any_t = __any_sync(0xffffffffu, mine);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float z[32];
      tmem_load_32cols(taddr + c * 32, z);
      const int vc = v0 + c * 32;
      if (HAS_BIAS) {
        if (bias_vec) {
          const float4* b4 = reinterpret_cast<const float4*>(p.bias + vc);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 b = __ldg(b4 + q);
            z[4 * q + 0] += b.x;
            z[4 * q + 1] += b.y;
            z[4 * q + 2] += b.z;
            z[4 * q + 3] += b.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] += (vc + i < p.V) ? __ldg(p.bias + vc + i) : 0.f;
        }
      }
      float cm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        z[i] *= rs.inv_tau;
        if (!full && vc + i >= p.V) z[i] = -INFINITY;
        cm = fmaxf(cm, z[i]);
      }
      if (any_t) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (tl == c * 32 + i) rs.zt = z[i];
      }
      const float mn = fmaxf(rs.m, cm);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        a0 += epi_exp2((z[i + 0] - mn) * kLog2e);
        a1 += epi_exp2((z[i + 1] - mn) * kLog2e);
        a2 += epi_exp2((z[i + 2] - mn) * kLog2e);
        a3 += epi_exp2((z[i + 3] - mn) * kLog2e);
      }
      rs.s = rs.s * epi_exp2((rs.m - mn) * kLog2e) + ((a0 + a1) + (a2 + a3));
      rs.m = mn;
    }
  }

  static __device__ __forceinline__ void unit_end(const Params& p, const UnitInfo& ui, int, int, RowState& rs) {
    if (rs.n >= p.N) return;
    const int split = ui.n0 / (TPS * BN);
    const size_t idx = static_cast<size_t>(split) * p.N + rs.n;
    p.part_m[idx] = rs.m;
    p.part_s[idx] = rs.s;
    if (rs.tloc >= 0 && rs.tloc < ui.ntiles * BN) p.zt[rs.n] = rs.zt;
  }
};

// A block merges 32 rows: lane l of every warp serves row n0 + l, and warp w
// holds a contiguous run of kMergeHeld splits of each round of kMergeRound
// splits in registers, so every partial load is a coalesced 128-byte row
// segment and all of a warp's loads are in flight at once.  The maximum is
// combined across warps (exact in any order).  The sum is one chain of fused
// multiply-adds in ascending split order: warp 0 folds its run, hands the
// running sum to warp 1 through shared memory, and so on, so a row's sum is the
// same sequence of roundings whatever N or the grid is.  At small N a single
// block does all the work, and its time is the number of dependent round trips
// to memory: one per round (two when the splits need more than one round).
constexpr int kMergeRows = 32;                           // rows per 256-thread block
constexpr int kMergeWarps = 8;                           // warps sharing a row's splits
constexpr int kMergeHeld = 32;                           // splits a warp holds per round
constexpr int kMergeRound = kMergeWarps * kMergeHeld;  // splits per round

struct MergeSmem {
  float red[kMergeWarps][kMergeRows];
  float carry[kMergeRows];
};

// Loads warp w's run of round r0: m (and s when `with_s`) of splits
// r0 + w * kMergeHeld + k; splits past the end read as m = -inf, s = 0.
__device__ __forceinline__ void merge_load_run(const FwdParams& p, int n, int r0, int w, bool with_s,
                                               float (&mv)[kMergeHeld], float (&sv)[kMergeHeld]) {
#pragma unroll
  for (int k = 0; k < kMergeHeld; ++k) {
    const int s = r0 + w * kMergeHeld + k;
    const size_t i = static_cast<size_t>(s) * p.N + n;
    mv[k] = s < p.num_splits ? p.part_m[i] : -INFINITY;
    if (with_s) sv[k] = s < p.num_splits ? p.part_s[i] : 0.f;
  }
}

// Returns (M, S) of row n in every thread of lane n - n0 (all warps).  All
// threads of the block must call it.
__device__ __forceinline__ void merge_splits_block(const FwdParams& p, int n, MergeSmem& sm, float& M, float& S) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const bool valid = n < p.N;
  const int ns = p.num_splits;
  const bool held = ns <= kMergeRound;  // one round: the first loads serve both passes
  float mv[kMergeHeld], sv[kMergeHeld];
  float mx = -INFINITY;
  for (int r0 = 0; r0 < ns; r0 += kMergeRound) {
    if (valid) {
      merge_load_run(p, n, r0, w, held, mv, sv);
#pragma unroll
      for (int k = 0; k < kMergeHeld; ++k) mx = fmaxf(mx, mv[k]);
    }
  }
  sm.red[w][lane] = mx;
  if (w == 0) sm.carry[lane] = 0.f;
  __syncthreads();
  M = sm.red[0][lane];
#pragma unroll
  for (int k = 1; k < kMergeWarps; ++k) M = fmaxf(M, sm.red[k][lane]);
  for (int r0 = 0; r0 < ns; r0 += kMergeRound) {
    if (valid) {
      if (!held) merge_load_run(p, n, r0, w, true, mv, sv);
#pragma unroll
      for (int k = 0; k < kMergeHeld; ++k) mv[k] = exp2f((mv[k] - M) * kLog2e);
    }
    for (int ww = 0; ww < kMergeWarps; ++ww) {
      if (w == ww && valid) {
        float acc = sm.carry[lane];
#pragma unroll
        for (int k = 0; k < kMergeHeld; ++k)
          if (r0 + ww * kMergeHeld + k < ns) acc = __fmaf_rn(sv[k], mv[k], acc);
        sm.carry[lane] = acc;
      }
      __syncthreads();
    }
  }
  S = sm.carry[lane];
}

__global__ void __launch_bounds__(256) fwd_merge_kernel(FwdParams p, float* __restrict__ out_logp,
                                                        float* __restrict__ out_lse) {
  __shared__ MergeSmem sm;
  const int n = blockIdx.x * kMergeRows + (threadIdx.x & 31);
  const bool mine = threadIdx.x < 32 && n < p.N;
  // issued before the merge so that their latency overlaps it; zt is used only for valid targets
  const long long t = mine ? p.targets[n] : 0;
  const float zt = mine ? p.zt[n] : 0.f;
  float M, S;
  merge_splits_block(p, n, sm, M, S);
  if (!mine) return;
  if (!target_valid(t, p.V, p.ignore_index)) {
    out_logp[n] = 0.f;
    out_lse[n] = -INFINITY;
    return;
  }
  const float ls = logf(S);
  out_lse[n] = M + ls;
  out_logp[n] = (zt - M) - ls;
}

// Vocab-parallel shard statistics ("Fused Linear LogP", Tensor Parallel Vocab
// Shards: each rank computes local online-softmax state that collectives then
// merge): per row the shard's max, its sum of exp(z - max) (splits merged in
// ascending order) and the target logit when the target lies in the shard,
// else -inf.
__global__ void __launch_bounds__(256) shard_stats_kernel(FwdParams p, float* __restrict__ out_max,
                                                          float* __restrict__ out_se, float* __restrict__ out_tl) {
  __shared__ MergeSmem sm;
  const int n = blockIdx.x * kMergeRows + (threadIdx.x & 31);
  float M, S;
  merge_splits_block(p, n, sm, M, S);
  if (threadIdx.x >= 32 || n >= p.N) return;
  const long long t = p.targets[n];
  const long long tl = t - p.vocab_start;
  const bool local = t != p.ignore_index && tl >= 0 && tl < static_cast<long long>(p.V);
  out_max[n] = M;
  out_se[n] = S;
  out_tl[n] = local ? p.zt[n] : -INFINITY;
}

// Merge of R shards' (max, sum, target logit) in ascending rank order, then the
// same final expression as the unsharded merge.  Exactly one shard holds a
// valid target, so the target logit is the largest of the R entries.
__global__ void __launch_bounds__(256) merge_shards_kernel(const float* __restrict__ mx, const float* __restrict__ se,
                                                           const float* __restrict__ tl, int R, int N,
                                                           const long long* __restrict__ targets, long long global_V,
                                                           long long ignore_index, float* __restrict__ out_logp,
                                                           float* __restrict__ out_lse) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const long long t = targets[n];
  if (t == ignore_index || t < 0 || t >= global_V) {
    out_logp[n] = 0.f;
    out_lse[n] = -INFINITY;
    return;
  }
  float M = -INFINITY, zt = -INFINITY;
  for (int r = 0; r < R; ++r) {
    M = fmaxf(M, mx[static_cast<size_t>(r) * N + n]);
    zt = fmaxf(zt, tl[static_cast<size_t>(r) * N + n]);
  }
  float S = 0.f;
  for (int r = 0; r < R; ++r) {
    const size_t i = static_cast<size_t>(r) * N + n;
    S += se[i] * exp2f((mx[i] - M) * kLog2e);
  }
  const float ls = logf(S);
  out_lse[n] = M + ls;
  out_logp[n] = (zt - M) - ls;
}

cudaError_t launch_shard_stats(const FwdParams& p, float* out_max, float* out_sumexp, float* out_tlogit,
                               cudaStream_t s) {
  shard_stats_kernel<<<(p.N + kMergeRows - 1) / kMergeRows, 256, 0, s>>>(p, out_max, out_sumexp, out_tlogit);
  return launch_result();
}

cudaError_t launch_merge_shards(const float* mx, const float* se, const float* tl, int R, int N,
                                const long long* targets, long long global_V, long long ignore_index, float* out_logp,
                                float* out_lse, cudaStream_t s) {
  merge_shards_kernel<<<(N + 255) / 256, 256, 0, s>>>(mx, se, tl, R, N, targets, global_V, ignore_index, out_logp,
                                                      out_lse);
  return launch_result();
}

cudaError_t fwd_setup(LaunchCaps* caps) {
  cudaError_t e = setup_gemm<FwdCfg<false>>(&caps->fwd_groups[0]);
  if (e == cudaSuccess) e = setup_gemm<FwdCfg<true>>(&caps->fwd_groups[1]);
  if (e == cudaSuccess) e = setup_gemm<FwdCfg<false, false>>(&caps->fwd_single[0]);
  if (e == cudaSuccess) e = setup_gemm<FwdCfg<true, false>>(&caps->fwd_single[1]);
  if (e == cudaSuccess) e = setup_gemm<FwdCfg<false, false, kSmallARows>>(&caps->fwd_small[0]);
  if (e == cudaSuccess) e = setup_gemm<FwdCfg<true, false, kSmallARows>>(&caps->fwd_small[1]);
  return e;
}

template <class Cfg>
static cudaError_t launch_units(const CUtensorMap& a, const CUtensorMap& b, const typename Cfg::Params& p,
                                long long units, int groups, cudaStream_t s) {
  const long long g = units < groups ? units : groups;
  return launch_gemm<Cfg>(a, b, a, p, static_cast<int>(g) * Plan<Cfg>::NCTA, s);  // no tensor stores
}

cudaError_t launch_fwd_partials(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const FwdParams& p,
                                long long units, const LaunchCaps& caps, cudaStream_t s, bool single) {
  if (single && hidden_box_rows(p.N, true) == kSmallARows)
    return p.bias ? launch_units<FwdCfg<true, false, kSmallARows>>(tm_h, tm_w, p, units, caps.fwd_small[1], s)
                  : launch_units<FwdCfg<false, false, kSmallARows>>(tm_h, tm_w, p, units, caps.fwd_small[0], s);
  if (single)
    return p.bias ? launch_units<FwdCfg<true, false>>(tm_h, tm_w, p, units, caps.fwd_single[1], s)
                  : launch_units<FwdCfg<false, false>>(tm_h, tm_w, p, units, caps.fwd_single[0], s);
  return p.bias ? launch_units<FwdCfg<true>>(tm_h, tm_w, p, units, caps.fwd_groups[1], s)
                : launch_units<FwdCfg<false>>(tm_h, tm_w, p, units, caps.fwd_groups[0], s);
}

cudaError_t launch_fwd_merge(const FwdParams& p, float* out_logp, float* out_lse, cudaStream_t s) {
  fwd_merge_kernel<<<(p.N + kMergeRows - 1) / kMergeRows, 256, 0, s>>>(p, out_logp, out_lse);
  return launch_result();
}

}  // namespace llp
