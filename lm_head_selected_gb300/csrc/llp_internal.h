// Internal (non-exported) declarations shared by the kernel translation units
// and the C-ABI layer.  Plain structs only: they are kernel parameters.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace llp {

// Fixed tiling.  None of these depend on N, so each token row sees the same
// vocab tiles, vocab splits, K order and merge order at every batch size.
constexpr int kTileM = 128;           // tokens (or vocab rows for grad_weight) per tile
constexpr int kTileN = 256;           // vocab (or hidden) columns per tile
constexpr int kTileK = 64;            // K elements per pipeline stage
constexpr int kTilesPerSplit = 2;     // forward vocab split = 512 columns
constexpr int kSplitWidth = kTileN * kTilesPerSplit;
constexpr int kKSegment = 32768;      // fixed K segment of the gradient GEMMs
constexpr bool kPairMMA = true;       // 2-CTA (cta_group::2) tiles: 256 rows per unit
constexpr int kUnitM = kPairMMA ? 2 * kTileM : kTileM;  // unit rows (M) per tile
constexpr int kBRows = kPairMMA ? kTileN / 2 : kTileN;  // rows of a K-major B tile each CTA loads
// Compile-time tuning knobs (defaults are the tuned values).
#ifndef LLP_GROUP_M
#define LLP_GROUP_M 32     // L2 raster group in unit M tiles (256 rows); scheduling only
#endif
constexpr int kGroupM = LLP_GROUP_M;
#ifndef LLP_PAIR_STAGES
#define LLP_PAIR_STAGES 6  // shared-memory pipeline stages in pair mode (32 KB each)
#endif
constexpr int kPairStages = LLP_PAIR_STAGES;
#ifndef LLP_DYNAMIC_SCHED
#define LLP_DYNAMIC_SCHED 3  // bit 0: grad_hidden, bit 1: grad_weight claim units in order from a ticket counter
#endif
#ifndef LLP_DZ_STREAM
#define LLP_DZ_STREAM 1      // store the bf16 dlogits with L2 evict-first priority
#endif
#ifndef LLP_DYN_MIN_KB
#define LLP_DYN_MIN_KB 128   // in-order claiming only when full units span at least this many k-blocks
#endif
constexpr int kDynMinKBlocks = LLP_DYN_MIN_KB;
#ifndef LLP_EPI_FASTEXP
#define LLP_EPI_FASTEXP 1    // GEMM epilogues: the ex2.approx.ftz instruction instead of exp2f
#endif
#ifndef LLP_LOCKSTEP
#define LLP_LOCKSTEP 0       // gradient GEMMs: pairs report progress and wait when too far ahead (k-block window, 0 = off)
#endif
#ifndef LLP_LOCKSTEP_MASK
#define LLP_LOCKSTEP_MASK 3  // bit 0: grad_hidden, bit 1: grad_weight take part in the lockstep
#endif
#ifndef LLP_CHUNKED_MN
#define LLP_CHUNKED_MN 1     // MN-major GEMM operands as one 3-D copy per stage (when MN % 64 == 0)
#endif
#ifndef LLP_KPS2
#define LLP_KPS2 5           // two k-blocks per pipeline stage (one 3-D copy per operand) where the maps allow,
                             // bit 0: forward / dlogits on CTA pairs, 1: grad_hidden, 2: grad_weight (>= 1024 tokens)
#endif
#ifndef LLP_HALF_TILE
#define LLP_HALF_TILE 0      // half-width MMA for a last column tile with <= 128 columns
#endif

#ifndef LLP_SMALL_GH
#define LLP_SMALL_GH 1       // grad_hidden of batches of at most kSmallGhMaxN rows on the swapped-operand kernel
#endif

// grad_hidden of small batches with the hidden dimension on the MMA's M side
// and the tokens on its N side (gh_small.cu).
// Largest batch it takes (tokens padded to a multiple of 16).  Above 96 tokens
// a dz slot (256 vocab rows x tokens) is so large that only one fits beside two
// weight stages, and the two-CTA GEMM is faster (N=112: 220 vs 160 us).
constexpr int kSmallGhMaxN = 96;
constexpr int kSmallGhRows = 256;        // vocab rows per weight stage (height of the weight boxes)
constexpr int kSmallGhMaxStages = 8;     // deepest ring of either operand
constexpr int kSmallGhSmemLimit = 232448;  // dynamic shared memory the kernel may use

struct GhSmallParams {
  int N, D, V;
  int BN;            // MMA N: N rounded up to 16
  int nseg, num_dt;  // vocab segments of kKSegment rows; 128-column hidden tiles
  int b_span;        // weight stages of kSmallGhRows vocab rows per dz slot
  int stages_a, stages_b, b_slot_bytes;  // ring depths (weight, dz) and bytes of one dz slot
  int w_chunked;     // the weight map is 3-D {64, V, D/64}: one copy per stage (D % 128 == 0), else 2-D
  float* part;          // fp32 [nseg][N][D] (segment partials, or a shard's contribution); nullptr: `out`
  __nv_bfloat16* out;   // [N][D] bf16 (fp16 when f16), with one segment and part == nullptr
  int f16;
  unsigned int* err;
};
// Fills N, BN, the ring depths and slot size; false when the batch is too large for the kernel.
bool small_grad_hidden_plan(int N, GhSmallParams* p);
cudaError_t small_grad_hidden_setup();
// tm_w: the weight [V][D] as 64-column chunks, {64, V, D/64} with box {64, kSmallGhRows, 2}
// (w_chunked), else 2-D {D, V} with box {64, kSmallGhRows}; tm_dz: dz [N][V_pad] as 64-column
// chunks, {64, N, V_pad/64} with box {64, BN, kSmallGhRows/64 * b_span} (its padding columns
// must be zero).
cudaError_t launch_small_grad_hidden(const CUtensorMap& tm_w, const CUtensorMap& tm_dz, const GhSmallParams& p,
                                     int num_sms, cudaStream_t s);

#ifndef LLP_GW_H_EVICT_LAST
#define LLP_GW_H_EVICT_LAST 1  // grad_weight loads the hidden states with an L2 evict-last hint
                               // (every unit re-reads them; at small N all pairs read the same few lines)
#endif

#ifndef LLP_SMALL_A
#define LLP_SMALL_A 1        // single-CTA forward / dlogits of <= kSmallARows rows load only those hidden rows
#endif
// A batch of at most kSmallARows rows (single-CTA tiles) loads a kSmallARows-row
// hidden box per stage instead of a kTileM-row one.  The MMA still reads kTileM
// rows: the rest fall on the stage's weight tile and feed only accumulator rows
// past the batch, which no epilogue writes.  The bytes saved hold more weight
// stages (a 2% faster weight stream in these HBM-bound kernels).
constexpr int kSmallARows = 32;
constexpr int kSmallAFwdStages = 6;  // 6 x 36 KB
constexpr int kSmallADzStages = 5;   // 5 x 36 KB + the epilogue's 32 KB of store buffers
// Rows of the hidden-state box that the forward / dlogits maps use for N rows.
inline int hidden_box_rows(long long N, bool single) {
  return (LLP_SMALL_A && single && N <= kSmallARows) ? kSmallARows : kTileM;
}

// Resident work groups (CTA pairs, or CTAs in single mode) per GEMM kernel,
// found once per device; the persistent grids never exceed them.
struct LaunchCaps {
  int fwd_groups[2];  // [has_bias]
  int fwd_single[2];  // [has_bias], single-CTA forward for batches of at most kTileM rows
  int fwd_small[2];   // [has_bias], single-CTA forward with kSmallARows-row hidden boxes
  int dz_groups[2];   // [has_bias]
  int dz_single[2];   // [has_bias], single-CTA dlogits for batches of at most kTileM rows
  int dz_small[2];    // [has_bias], single-CTA dlogits with kSmallARows-row hidden boxes
  int gh_groups;
  int gw_groups;
};

struct FwdParams {
  int N, D, V;
  int num_m, num_splits, num_vt, group_m;
  const float* bias;
  const long long* targets;
  const float* temperature;
  long long ignore_index;
  float* part_m;   // [num_splits][N] running max of each split
  float* part_s;   // [num_splits][N] sum of exp(z - part_m) over the split
  float* zt;       // [N] target logit (written by the split that holds the target)
  unsigned int* err;
  long long vocab_start;  // global id of local vocab row 0 (vocab-parallel shards; 0 otherwise)
  long long global_V;     // global vocab size (== V unless sharded)
  int f16;                // hidden / weight are IEEE fp16 (else bf16)
  int kps;                // k-blocks per pipeline stage: 2 with 3-D chunked maps (D % 64 == 0), else 1
};

struct DzParams {
  int N, D, V, V_pad;
  int num_m, num_vt, group_m;
  const float* bias;
  const long long* targets;
  const float* temperature;
  long long ignore_index;
  const float* grad_logp;
  const float* lse;
  __nv_bfloat16* dz;  // [N][V_pad], bf16 (or fp16 when f16; the two operands of a GEMM share one type)
  float* gb_part;     // [num_m*4][V]: per 32-row block column sums of dz (bias only)
  unsigned int* err;
  long long vocab_start;  // global id of local vocab row 0 (vocab-parallel shards; 0 otherwise)
  long long global_V;     // global vocab size: decides which targets are valid
  int* sched_reset;       // [kNumSchedCounters] ticket counters of the gradient GEMMs, zeroed at launch
  int f16;                // hidden / weight / dz are IEEE fp16 (else bf16)
  int kps;                // k-blocks per pipeline stage: 2 with 3-D chunked maps (D % 64 == 0), else 1
};

// Ticket counters of the in-order scheduled gradient GEMMs (one per GEMM of a
// backward) and their progress counters, held in the backward workspace and
// zeroed by the dlogits kernel that precedes them on the stream.
constexpr int kNumSchedCounters = 4;

struct GradGemmParams {
  int rows;          // M extent: N for grad_hidden, V for grad_weight
  int D;             // output columns
  int K;             // reduction extent: V for grad_hidden, N for grad_weight
  int num_m, num_d, nseg, kseg_blocks;
  __nv_bfloat16* out;  // [rows][D] bf16 (fp16 when f16) when nseg == 1 and !f32_out
  float* part;         // [nseg][rows][D] fp32 partials when nseg > 1 or f32_out
  unsigned int* err;
  int f32_out;         // 1: always write fp32 partials (a vocab shard's grad_hidden contribution)
  int* sched;          // ticket counter, 0 at launch; nullptr: round-robin units
  unsigned int* progress;  // k-blocks issued by all pairs, 0 at launch (advisory lockstep); nullptr: off
  int a_chunked, b_chunked;  // the MN-major operand's map is 3-D {64, K, MN/64}: one copy per stage
  int kps;             // k-blocks per pipeline stage: 2 when every operand map is 3-D, else 1
  int f16;             // operands and the 16-bit output are IEEE fp16 (else bf16)
};

// Records a failed CUDA call's code for linear_logp_last_cuda_error (per calling
// thread) and returns it unchanged.
cudaError_t note_cuda(cudaError_t e);
// The error of the launch just made on this thread (cudaGetLastError, recorded).
inline cudaError_t launch_result() { return note_cuda(cudaGetLastError()); }

// Launchers (return the launch error, never synchronise).  `units` is the
// number of work units; the grid is min(units, resident groups) groups.
cudaError_t fwd_setup(LaunchCaps* caps);
// single: 128-row single-CTA tiles (p.num_m counted in kTileM rows, W map box
// kTileN rows) instead of 256-row CTA-pair tiles (kUnitM rows, box kBRows rows).
cudaError_t launch_fwd_partials(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const FwdParams& p,
                                long long units, const LaunchCaps& caps, cudaStream_t s, bool single);
cudaError_t launch_fwd_merge(const FwdParams& p, float* out_logp, float* out_lse, cudaStream_t s);
// Vocab-parallel shards: per-row (max, sum of exp(z - max), target logit or -inf)
// of this shard, and the ascending-rank merge of R shards' triples.
cudaError_t launch_shard_stats(const FwdParams& p, float* out_max, float* out_sumexp, float* out_tlogit,
                               cudaStream_t s);
cudaError_t launch_merge_shards(const float* mx, const float* se, const float* tl, int R, int N,
                                const long long* targets, long long global_V, long long ignore_index, float* out_logp,
                                float* out_lse, cudaStream_t s);
// num_sms: the device's SM count (the grid is at most 16 blocks per SM).
cudaError_t launch_segment_sum_f32(const float* part, int nseg, long long count, float* out, int num_sms,
                                   cudaStream_t s);

cudaError_t bwd_setup(LaunchCaps* caps);
// The third tensor map is the output the epilogue stores through: dz (bf16,
// box 64 x 32), or the gradient (bf16, box 64 x 32) / its fp32 segment
// partials ([nseg][rows][D], box 32 x 32 x 1).
cudaError_t launch_dlogits(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const CUtensorMap& tm_dz_out,
                           const DzParams& p, long long units, const LaunchCaps& caps, cudaStream_t s,
                           bool single);
cudaError_t launch_grad_hidden(const CUtensorMap& tm_dz, const CUtensorMap& tm_w_mn, const CUtensorMap& tm_out,
                               const GradGemmParams& p, long long units, const LaunchCaps& caps, cudaStream_t s);
cudaError_t launch_grad_weight(const CUtensorMap& tm_dz_mn, const CUtensorMap& tm_h_mn, const CUtensorMap& tm_out,
                               const GradGemmParams& p, long long units, const LaunchCaps& caps, cudaStream_t s);
// Logits-input fused log-prob (logits.cu).  dtype: kDtypeBF16, kDtypeF32 or kDtypeF16.
// The forward works on P row slots: slot j is row rows[j] (row j when rows is
// null; -1 = padding); `part` holds 2 * ceil(V / kLogitsSplit) * P floats.  The
// backward writes all N rows, a zero row where `mask` (optional) is 0.  `vec` =
// rows are 16-byte aligned (base and row pitch), so 16-byte loads and stores may be used.
constexpr int kDtypeBF16 = 0;
constexpr int kDtypeF32 = 1;
constexpr int kDtypeF16 = 2;
constexpr int kLogitsSplit = 16384;  // vocab elements per CTA (fixed: depends on nothing)
cudaError_t launch_logits_fwd(const void* z, int dtype, int P, const int* rows, int V, const long long* targets,
                              long long ignore_index, float* part, float* logp, float* row_max, float* log_sum,
                              bool vec, cudaStream_t s);
cudaError_t launch_logits_bwd(const void* z, int dtype, int N, int V, const long long* targets,
                              long long ignore_index, const float* grad_logp, const float* row_max,
                              const float* log_sum, const unsigned char* mask, void* grad, bool vec, cudaStream_t s);

// Row selection for the indexed variants (indexed.cu): the index list becomes a
// byte mask over N rows and the selected rows, in ascending order, padded with
// -1 up to K = min(#indices, N) slots.  `total` (device) = number of rows selected.
struct RowSelection {
  unsigned char* mask;  // [N]
  int* rows;            // [K]
  int* slot_of;         // [N], valid where mask != 0
  int* total;           // device scalar
  int K;
};
size_t select_workspace_bytes(long long N, long long K);
cudaError_t build_row_selection(const long long* idx, long long K, int N, void* ws, RowSelection* sel,
                                cudaStream_t s);
cudaError_t gather_selected_rows(const RowSelection& sel, int D, const __nv_bfloat16* hidden,
                                 const long long* targets, const float* temperature, const float* grad_logp,
                                 const float* lse, long long ignore_index, __nv_bfloat16* c_hidden,
                                 long long* c_targets, float* c_temperature, float* c_grad, float* c_lse,
                                 cudaStream_t s);
cudaError_t scatter_selected_outputs(const RowSelection& sel, const float* c_logp, const float* c_lse, float* logp,
                                     float* lse, cudaStream_t s);
cudaError_t scatter_selected_grad_hidden(const RowSelection& sel, int N, int D, const __nv_bfloat16* c_gh,
                                         __nv_bfloat16* gh, cudaStream_t s);

// out: bf16, or fp16 when f16 != 0; num_sms: the device's SM count (the grid
// is at most 16 blocks per SM).
cudaError_t launch_segment_sum(const float* part, int nseg, long long count, __nv_bfloat16* out, int num_sms,
                               cudaStream_t s, int f16 = 0);
cudaError_t launch_bias_sum(const float* gb_part, int nblocks, int V, float* out, cudaStream_t s);

}  // namespace llp
