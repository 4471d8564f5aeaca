// Backward of the fused linear selected-token log-probability on tcgen05.
//
//   B1  dlogits: recompute each 128 x 256 logit tile exactly as the forward
//       does, then  dz = (g_n / tau_n) * (onehot(t_n) - exp(z - lse_n)),
//       selected to 0 on invalid rows (so a NaN upstream gradient there cannot
//       leak), written as bf16 into a [N, V_pad] workspace.  With a bias, each
//       warp also reduces its 32 rows of dz per column in a fixed butterfly
//       order into a [N/32, V] fp32 partial for grad_bias.
//   B2  grad_hidden = dz . W        (M = tokens, N = hidden, K = vocab)
//   B3  grad_weight = dz^T . h      (M = vocab,  N = hidden, K = tokens)
//       Both are tcgen05 GEMMs over fixed K segments of kKSegment; with more
//       than one segment the fp32 segment partials are summed in ascending
//       order and rounded once to bf16.
//   B4  grad_bias[v] = sum of the 32-row partials in ascending row order.
//
// The formula is the one of "add backward support for fused logp CUDA
// kernels" (Implementation details: grad_out * (one_hot - softmax) from saved
// softmax statistics, no logits-sized probability tensor); the 1/tau factor
// is the chain rule through the temperature of "Feat/nemotron h lm head
// logprob cuda".  The fixed ascending K segments with fp32 partials follow
// the same page's fix for reductions longer than 32768 ("split into <= 32768
// segments whose FP32 partials are summed in a fixed ascending order"); here
// fp32 accumulation in TMEM has no length limit, the segments only fix the
// reduction order and spread the long vocab reduction over more SMs.
#include "gemm_core.cuh"

namespace llp {

constexpr float kLog2eB = 1.4426950408889634f;

__device__ __forceinline__ bool target_ok(long long t, int V, long long ignore_index) {
  return t != ignore_index && t >= 0 && t < static_cast<long long>(V);
}

// Column sums of a 32 x 32 block held one row per lane: on return lane l holds
// the sum over the 32 lanes of column l.  Butterfly order, fixed.
__device__ __forceinline__ float warp_column_sums(float (&x)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? x[i] : x[i + off];
      const float keep = upper ? x[i + off] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return x[0];
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two floats rounded to the path's 16-bit type (fp16 when f16, else bf16).
__device__ __forceinline__ uint32_t pack16x2(bool f16, float a, float b) {
  return f16 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
}

// ----------------------------------------------------------------------------
// B1: dlogits
// ----------------------------------------------------------------------------
// PAIRED = false: single CTAs with 128-row tiles, for a batch that fits in one.
// AROWS: hidden rows loaded per stage (kSmallARows for a batch that small).
template <bool HAS_BIAS, bool PAIRED = kPairMMA, int AROWS = kTileM>
struct DzCfg {
  static constexpr bool A_MN = false;
  static constexpr bool B_MN = false;
  static constexpr bool PAIR = PAIRED;
  static constexpr int BN = kTileN;
  static constexpr int A_ROWS = AROWS;
  static constexpr int STAGES = PAIR ? kPairStages : (AROWS < kTileM ? kSmallADzStages : 4);
  static constexpr int EXTRA_SMEM = kEpiSmemBytes;
  static constexpr int UM = PAIR ? kUnitM : kTileM;
  using Params = DzParams;

  struct RowState {
    float inv_tau, gs, lse;
    int t;
    int n;
    bool valid;
  };

  static __device__ __forceinline__ uint64_t policy_a() { return l2_policy_evict_last(); }
  static __device__ __forceinline__ uint64_t policy_b() { return l2_policy_evict_normal(); }
  static constexpr bool DYNAMIC = false;
  static __device__ __forceinline__ int* sched_counter(const Params&) { return nullptr; }
  static __device__ __forceinline__ unsigned int* progress_counter(const Params&) { return nullptr; }
  static __device__ __forceinline__ bool a_chunked(const Params&) { return false; }
  static __device__ __forceinline__ bool b_chunked(const Params&) { return false; }
  static __device__ __forceinline__ int kps(const Params& p) { return p.kps; }
  // the gradient GEMMs that follow on the stream start from ticket 0
  static __device__ __forceinline__ void on_launch(const Params& p) {
    if (p.sched_reset != nullptr)
      for (int i = 0; i < kNumSchedCounters; ++i) p.sched_reset[i] = 0;
  }

  static __device__ __forceinline__ int num_units(const Params& p) { return p.num_m * p.num_vt; }

  static __device__ __forceinline__ UnitInfo unit(const Params& p, int u) {
    const int gsize = p.group_m * p.num_vt;
    const int grp = u / gsize;
    const int r = u - grp * gsize;
    const int gm = min(p.group_m, p.num_m - grp * p.group_m);
    const int vt = r / gm;
    const int mt = grp * p.group_m + (r - vt * gm);
    UnitInfo ui;
    ui.m0 = mt * UM;
    ui.n0 = vt * BN;
    ui.ntiles = 1;
    ui.kb0 = 0;
    ui.nkb = (p.D + BK - 1) / BK;
    ui.bn = BN;
    return ui;
  }

  static __device__ __forceinline__ void unit_begin(const Params& p, const UnitInfo& ui, int, int row, RowState& rs) {
    rs.n = ui.m0 + row;
    rs.valid = false;
    rs.inv_tau = 1.f;
    rs.gs = 0.f;
    rs.lse = 0.f;
    rs.t = -1;
    if (rs.n < p.N) {
      // validity is global; the one-hot column is the target's local id in this
      // (possibly vocab-sharded) weight, outside [0, V) when another shard holds it
      const long long t = p.targets[rs.n];
      if (target_ok(t, static_cast<int>(p.global_V), p.ignore_index)) {
        rs.valid = true;
        rs.t = static_cast<int>(t - p.vocab_start);
        if (p.temperature != nullptr) rs.inv_tau = __frcp_rn(p.temperature[rs.n]);
        rs.gs = p.grad_logp[rs.n] * rs.inv_tau;
        rs.lse = p.lse[rs.n];
      }
    }
  }

  static __device__ __forceinline__ void tile(const Params& p, const UnitInfo& ui, int, int, int row, int lane,
                                              uint32_t taddr, RowState& rs, EpiStore& es) {
    const int v0 = ui.n0;
    const bool full = (v0 + BN) <= p.V;
    const bool bias_vec = full && (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0;
    const int blk = (ui.m0 + row) >> 5;  // 32-row block of this warp
    const bool f16 = p.f16 != 0;
    const int row0 = ui.m0 + row - lane;  // first token row of this warp's slab
#pragma unroll 1
    for (int q = 0; q < BN / 64; ++q) {  // 64-column slabs of dz, one TMA store each
      if (v0 + 64 * q >= p.V) break;     // warp-uniform
      const uint32_t sbuf = epi_slab_begin(es);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int vc = v0 + 64 * q + 32 * h;
        float z[32];
        tmem_load_32cols(taddr + 64 * q + 32 * h, z);
        if (HAS_BIAS) {
          if (bias_vec) {
            const float4* b4 = reinterpret_cast<const float4*>(p.bias + vc);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float4 b = __ldg(b4 + k);
              z[4 * k + 0] += b.x;
              z[4 * k + 1] += b.y;
              z[4 * k + 2] += b.z;
              z[4 * k + 3] += b.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] += (vc + i < p.V) ? __ldg(p.bias + vc + i) : 0.f;
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float zz = z[i] * rs.inv_tau;
          const float pr = epi_exp2((zz - rs.lse) * kLog2eB);
          const float oh = (vc + i == rs.t) ? 1.f : 0.f;
          float d = rs.gs * (oh - pr);
          if (!rs.valid || (!full && vc + i >= p.V)) d = 0.f;
          z[i] = d;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
          epi_slab_put(sbuf, lane, 4 * h + k, pack16x2(f16, z[8 * k + 0], z[8 * k + 1]),
                       pack16x2(f16, z[8 * k + 2], z[8 * k + 3]), pack16x2(f16, z[8 * k + 4], z[8 * k + 5]),
                       pack16x2(f16, z[8 * k + 6], z[8 * k + 7]));
        if (HAS_BIAS && p.gb_part != nullptr) {  // warp-uniform
          const float colsum = warp_column_sums(z, lane);
          const int v = vc + lane;
          if (v < p.V) p.gb_part[static_cast<size_t>(blk) * p.V + v] = colsum;
        }
      }
      // rows >= N and columns >= V are clipped by the store's tensor map; a slab
      // that starts past the last row is not stored at all (warp-uniform)
      if (row0 < p.N) {
        // a large batch's dz (GBs) streams through L2 once per gradient GEMM; a
        // batch of at most 128 rows (single CTAs) has a few MB of dz, which the
        // grad_hidden kernel right after re-reads for every hidden tile: keep it
        if (!PAIR)
          epi_slab_store_2d_hint(es, sbuf, v0 + 64 * q, row0, l2_policy_evict_last());
        else if (LLP_DZ_STREAM)
          epi_slab_store_2d_hint(es, sbuf, v0 + 64 * q, row0, l2_policy_evict_first());
        else
          epi_slab_store_2d(es, sbuf, v0 + 64 * q, row0);
      }
    }
  }

  static __device__ __forceinline__ void unit_end(const Params&, const UnitInfo&, int, int, RowState&) {}
};

// ----------------------------------------------------------------------------
// B2 / B3: gradient GEMMs with fixed K segments.
// ----------------------------------------------------------------------------
template <bool A_MN_, bool B_MN_>
struct GradCfg {
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
  static_assert(B_MN, "half-width column tiles load B in 64-row MN-major boxes");
  static constexpr bool PAIR = kPairMMA;
  static constexpr int BN = kTileN;
  static constexpr int A_ROWS = BM;
  static constexpr int STAGES = PAIR ? kPairStages : 4;
  static constexpr int EXTRA_SMEM = kEpiSmemBytes;
  static constexpr int UM = kUnitM;
  using Params = GradGemmParams;

  struct RowState {
    int r;
  };

  static __device__ __forceinline__ uint64_t policy_a() { return l2_policy_evict_normal(); }
  // grad_weight's B, the hidden states, is re-read by every unit
  static __device__ __forceinline__ uint64_t policy_b() {
    return (A_MN && LLP_GW_H_EVICT_LAST) ? l2_policy_evict_last() : l2_policy_evict_normal();
  }
  // units are claimed in ascending order from a ticket counter, so the tiles
  // that share A rows or a K window of B run together
  static constexpr bool DYNAMIC = (LLP_DYNAMIC_SCHED & (A_MN ? 2 : 1)) != 0;
  static __device__ __forceinline__ int* sched_counter(const Params& p) { return p.sched; }
  static __device__ __forceinline__ unsigned int* progress_counter(const Params& p) { return p.progress; }
  static __device__ __forceinline__ bool a_chunked(const Params& p) { return p.a_chunked != 0; }
  static __device__ __forceinline__ bool b_chunked(const Params& p) { return p.b_chunked != 0; }
  static __device__ __forceinline__ int kps(const Params& p) { return p.kps; }
  // grad_weight's B is the hidden states
  static __device__ __forceinline__ void on_launch(const Params&) {}

  static __device__ __forceinline__ int num_units(const Params& p) { return p.nseg * p.num_m * p.num_d; }

  // Segment is the slowest index, then M tile, then the output column tile, so the
  // CTAs that run together share A rows and the same K window of B.
  static __device__ __forceinline__ UnitInfo unit(const Params& p, int u) {
    const int per_seg = p.num_m * p.num_d;
    const int seg = u / per_seg;
    const int r = u - seg * per_seg;
    const int mt = r / p.num_d;
    const int dt = r - mt * p.num_d;
    const int total_kb = (p.K + BK - 1) / BK;
    UnitInfo ui;
    ui.m0 = mt * UM;
    ui.n0 = dt * BN;
    ui.ntiles = 1;
    ui.kb0 = seg * p.kseg_blocks;
    ui.nkb = min(p.kseg_blocks, total_kb - ui.kb0);
    ui.bn = (LLP_HALF_TILE && p.D - ui.n0 <= BN / 2) ? BN / 2 : BN;  // ragged last column tile: half-width MMA
    return ui;
  }

  static __device__ __forceinline__ void unit_begin(const Params&, const UnitInfo& ui, int, int row, RowState& rs) {
    rs.r = ui.m0 + row;
  }

  // Output through 32-row slabs and TMA stores: bf16 [rows][D] with one
  // segment, else the fp32 partial of this segment in [nseg][rows][D] (a 3-D
  // tensor map, so rows past `rows` are clipped inside the segment).
  static __device__ __forceinline__ void tile(const Params& p, const UnitInfo& ui, int u, int, int row, int lane,
                                              uint32_t taddr, RowState&, EpiStore& es) {
    const int seg = u / (p.num_m * p.num_d);
    const int row0 = ui.m0 + row - lane;
    if (row0 >= p.rows) return;  // this warp's rows are all past the end (warp-uniform)
    if (p.nseg == 1 && !p.f32_out) {
      const bool f16 = p.f16 != 0;
#pragma unroll 1
      for (int q = 0; q < BN / 64; ++q) {
        const int d0 = ui.n0 + 64 * q;
        if (d0 >= p.D) break;  // warp-uniform
        const uint32_t sbuf = epi_slab_begin(es);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float a[32];
          tmem_load_32cols(taddr + 64 * q + 32 * h, a);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            epi_slab_put(sbuf, lane, 4 * h + k, pack16x2(f16, a[8 * k + 0], a[8 * k + 1]),
                         pack16x2(f16, a[8 * k + 2], a[8 * k + 3]), pack16x2(f16, a[8 * k + 4], a[8 * k + 5]),
                         pack16x2(f16, a[8 * k + 6], a[8 * k + 7]));
        }
        epi_slab_store_2d(es, sbuf, d0, row0);
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int d0 = ui.n0 + 32 * c;
        if (d0 >= p.D) break;  // warp-uniform
        const uint32_t sbuf = epi_slab_begin(es);
        float a[32];
        tmem_load_32cols(taddr + 32 * c, a);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          epi_slab_put(sbuf, lane, k, __float_as_uint(a[4 * k + 0]), __float_as_uint(a[4 * k + 1]),
                       __float_as_uint(a[4 * k + 2]), __float_as_uint(a[4 * k + 3]));
        epi_slab_store_3d(es, sbuf, d0, row0, seg);
      }
    }
  }

  static __device__ __forceinline__ void unit_end(const Params&, const UnitInfo&, int, int, RowState&) {}
};

// out[i] = bf16 (fp16 when f16) of sum_{s ascending} part[s][i], 4 elements per thread step.
__global__ void __launch_bounds__(256) segment_sum_kernel(const float* __restrict__ part, int nseg, long long count,
                                                          __nv_bfloat16* __restrict__ out, int f16) {
  const long long n4 = count / 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(part)[i];
    for (int s = 1; s < nseg; ++s) {
      const float4 v = reinterpret_cast<const float4*>(part + static_cast<size_t>(s) * count)[i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    uint2 w;
    w.x = pack16x2(f16 != 0, acc.x, acc.y);
    w.y = pack16x2(f16 != 0, acc.z, acc.w);
    reinterpret_cast<uint2*>(out)[i] = w;
  }
}

// out[i] = sum_{s ascending} part[s][i], kept in fp32.
__global__ void __launch_bounds__(256) segment_sum_f32_kernel(const float* __restrict__ part, int nseg,
                                                              long long count, float* __restrict__ out) {
  const long long n4 = count / 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(part)[i];
    for (int s = 1; s < nseg; ++s) {
      const float4 v = reinterpret_cast<const float4*>(part + static_cast<size_t>(s) * count)[i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    reinterpret_cast<float4*>(out)[i] = acc;
  }
}

// grad_bias[v] = sum over 32-row blocks in ascending order.
__global__ void __launch_bounds__(256) bias_sum_kernel(const float* __restrict__ gb_part, int nblocks, int V,
                                                       float* __restrict__ out) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= V) return;
  float acc = 0.f;
  for (int b = 0; b < nblocks; ++b) acc += gb_part[static_cast<size_t>(b) * V + v];
  out[v] = acc;
}

template <class Cfg>
static cudaError_t launch_units(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                                const typename Cfg::Params& p, long long units, int groups, cudaStream_t s) {
  const long long g = units < groups ? units : groups;
  return launch_gemm<Cfg>(a, b, c, p, static_cast<int>(g) * Plan<Cfg>::NCTA, s);
}

cudaError_t bwd_setup(LaunchCaps* caps) {
  cudaError_t e;
  if ((e = setup_gemm<DzCfg<false>>(&caps->dz_groups[0])) != cudaSuccess) return e;
  if ((e = setup_gemm<DzCfg<true>>(&caps->dz_groups[1])) != cudaSuccess) return e;
  if ((e = setup_gemm<DzCfg<false, false>>(&caps->dz_single[0])) != cudaSuccess) return e;
  if ((e = setup_gemm<DzCfg<true, false>>(&caps->dz_single[1])) != cudaSuccess) return e;
  if ((e = setup_gemm<DzCfg<false, false, kSmallARows>>(&caps->dz_small[0])) != cudaSuccess) return e;
  if ((e = setup_gemm<DzCfg<true, false, kSmallARows>>(&caps->dz_small[1])) != cudaSuccess) return e;
  if ((e = setup_gemm<GradCfg<false, true>>(&caps->gh_groups)) != cudaSuccess) return e;
  return setup_gemm<GradCfg<true, true>>(&caps->gw_groups);
}

cudaError_t launch_dlogits(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const CUtensorMap& tm_dz_out,
                           const DzParams& p, long long units, const LaunchCaps& caps, cudaStream_t s, bool single) {
  if (single && hidden_box_rows(p.N, true) == kSmallARows)
    return p.bias ? launch_units<DzCfg<true, false, kSmallARows>>(tm_h, tm_w, tm_dz_out, p, units, caps.dz_small[1], s)
                  : launch_units<DzCfg<false, false, kSmallARows>>(tm_h, tm_w, tm_dz_out, p, units, caps.dz_small[0],
                                                                   s);
  if (single)
    return p.bias ? launch_units<DzCfg<true, false>>(tm_h, tm_w, tm_dz_out, p, units, caps.dz_single[1], s)
                  : launch_units<DzCfg<false, false>>(tm_h, tm_w, tm_dz_out, p, units, caps.dz_single[0], s);
  return p.bias ? launch_units<DzCfg<true>>(tm_h, tm_w, tm_dz_out, p, units, caps.dz_groups[1], s)
                : launch_units<DzCfg<false>>(tm_h, tm_w, tm_dz_out, p, units, caps.dz_groups[0], s);
}

cudaError_t launch_grad_hidden(const CUtensorMap& tm_dz, const CUtensorMap& tm_w_mn, const CUtensorMap& tm_out,
                               const GradGemmParams& p, long long units, const LaunchCaps& caps, cudaStream_t s) {
  return launch_units<GradCfg<false, true>>(tm_dz, tm_w_mn, tm_out, p, units, caps.gh_groups, s);
}

cudaError_t launch_grad_weight(const CUtensorMap& tm_dz_mn, const CUtensorMap& tm_h_mn, const CUtensorMap& tm_out,
                               const GradGemmParams& p, long long units, const LaunchCaps& caps, cudaStream_t s) {
  return launch_units<GradCfg<true, true>>(tm_dz_mn, tm_h_mn, tm_out, p, units, caps.gw_groups, s);
}

// Grid-stride kernels: enough blocks to fill the device (16 per SM), never more than the work.
static long long segment_sum_blocks(long long count, int threads, int num_sms) {
  long long blocks = (count / 4 + threads - 1) / threads;
  const long long cap = 16LL * (num_sms > 0 ? num_sms : 1);
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : blocks;
}

cudaError_t launch_segment_sum(const float* part, int nseg, long long count, __nv_bfloat16* out, int num_sms,
                               cudaStream_t s, int f16) {
  const int threads = 256;
  const long long blocks = segment_sum_blocks(count, threads, num_sms);
  segment_sum_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(part, nseg, count, out, f16);
  return launch_result();
}

cudaError_t launch_segment_sum_f32(const float* part, int nseg, long long count, float* out, int num_sms,
                                   cudaStream_t s) {
  const int threads = 256;
  const long long blocks = segment_sum_blocks(count, threads, num_sms);
  segment_sum_f32_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(part, nseg, count, out);
  return launch_result();
}

cudaError_t launch_bias_sum(const float* gb_part, int nblocks, int V, float* out, cudaStream_t s) {
  const int threads = 256;
  bias_sum_kernel<<<(V + threads - 1) / threads, threads, 0, s>>>(gb_part, nblocks, V, out);
  return launch_result();
}

}  // namespace llp
