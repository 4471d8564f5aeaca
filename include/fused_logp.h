/*
 * fused_logp.h -- C ABI of the logits-input fused log-probability on GB300
 * (sm_103a), in the same library as linear_logp.h.
 *
 * The logits z [N, V] are already materialised ("Fused Linear LogP" docs page:
 * Fused LogP takes already-materialized logits as input).  Forward:
 *
 *     row_max[n] = max_v z[n, v]
 *     log_sum[n] = log sum_v exp(z[n, v] - row_max[n])
 *     logp[n]    = (z[n, t_n] - row_max[n]) - log_sum[n]
 *
 * with row_max and log_sum returned separately so that the backward rebuilds
 * probabilities without losing precision under large constant logit shifts,
 * and backward from those saved statistics, without forming a probability
 * tensor ("add backward support for fused logp CUDA kernels", Summary and
 * Implementation details):
 *
 *     grad_z[n, v] = grad_logp[n] * (onehot(t_n)[v] - exp((z[n, v] - row_max[n]) - log_sum[n]))
 *
 * A row whose target equals ignore_index or lies outside [0, V) gives logp = 0,
 * row_max = -inf, log_sum = 0 (so lse = row_max + log_sum = -inf) and a zero
 * gradient row ("recursive deterministic LogP autograd on B200", Summary).
 *
 * Conventions as in linear_logp.h: device pointers, caller-owned buffers, work
 * enqueued on `stream`, arguments checked before anything is enqueued, the same
 * LLP_* status codes.  z is contiguous row-major [N, V] in bf16 (dtype 0),
 * fp32 (dtype 1) or fp16 (dtype 2); grad_z has the same dtype.  Per-row results do not depend on
 * N and are identical across runs.  16-byte aligned rows (z base and V * element
 * size multiples of 16) take the vectorised path; other layouts still work.
 */
#ifndef FUSED_LOGP_H_
#define FUSED_LOGP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FUSED_LOGP_DTYPE_BF16 0
#define FUSED_LOGP_DTYPE_F32 1
#define FUSED_LOGP_DTYPE_F16 2

/* Workspace bytes fused_logp_fwd needs (per-row, per-vocab-split max / sum pairs). */
size_t fused_logp_workspace_bytes(int64_t N, int64_t V);

/* Forward: out_logp, out_row_max, out_log_sum are fp32 [N] (all required). */
int fused_logp_fwd(const void* logits, int dtype, int64_t N, int64_t V, const int64_t* targets,
                   int64_t ignore_index, float* out_logp, float* out_row_max, float* out_log_sum, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Backward: grad_logp, row_max, log_sum fp32 [N] from the forward on the same
 * logits; grad_logits [N, V] in `dtype` (overwritten, not accumulated). */
int fused_logp_bwd(const float* grad_logp, const float* row_max, const float* log_sum, const void* logits, int dtype,
                   int64_t N, int64_t V, const int64_t* targets, int64_t ignore_index, void* grad_logits,
                   void* stream);

/*
 * Row-subset (indexed) forms ("recursive deterministic LogP autograd on B200",
 * Indexed semantics: full output row shape, duplicate indices idempotent,
 * out-of-range indices ignored, zero derivatives for rows not selected).
 * `indices` [K] int64 (device) names the rows.
 *   fused_logp_fwd_indexed writes out_logp / out_row_max / out_log_sum for each
 *     selected row (bitwise what fused_logp_fwd gives that row) and leaves the
 *     other entries untouched.  Workspace: fused_logp_fwd_indexed_workspace_bytes.
 *   fused_logp_bwd_indexed writes the full grad_logits [N, V]: selected rows as
 *     fused_logp_bwd computes them, every other row zero.  row_max / log_sum /
 *     grad_logp are read on selected rows only.  Workspace:
 *     fused_logp_bwd_indexed_workspace_bytes (K = 0 selects nothing).
 */
size_t fused_logp_fwd_indexed_workspace_bytes(int64_t N, int64_t V, int64_t K);
size_t fused_logp_bwd_indexed_workspace_bytes(int64_t N, int64_t K);
int fused_logp_fwd_indexed(const void* logits, int dtype, int64_t N, int64_t V, const int64_t* targets,
                           int64_t ignore_index, const int64_t* indices, int64_t K, float* out_logp,
                           float* out_row_max, float* out_log_sum, void* workspace, size_t workspace_bytes,
                           void* stream);
int fused_logp_bwd_indexed(const float* grad_logp, const float* row_max, const float* log_sum, const void* logits,
                           int dtype, int64_t N, int64_t V, const int64_t* targets, int64_t ignore_index,
                           const int64_t* indices, int64_t K, void* grad_logits, void* workspace,
                           size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FUSED_LOGP_H_ */
