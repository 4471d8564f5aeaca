/*
 * linear_logp.h -- C ABI of the fused linear selected-token log-probability
 * on GB300 (sm_103a).
 *
 * The operation ("Fused Linear LogP", Reference Semantics and Tensor Contract;
 * per-row temperature from "Feat/nemotron h lm head logprob cuda", summary):
 *
 *     z[n, v]  = (hidden[n, :] . weight[v, :] + bias[v]) / temperature[n]
 *     lse[n]   = log sum_v exp(z[n, v])
 *     logp[n]  = z[n, targets[n]] - lse[n]
 *
 * and its gradients ("add backward support for fused logp CUDA kernels",
 * Implementation details):
 *
 *     dz[n, v]        = grad_logp[n] / temperature[n] * (onehot(targets[n])[v] - exp(z[n, v] - lse[n]))
 *     grad_hidden     = dz . weight          [N, D]
 *     grad_weight     = dz^T . hidden        [V, D]
 *     grad_bias       = sum_n dz[n, :]       [V]
 *
 * The [N, V] logits never reach global memory in the forward.  A row whose
 * target equals ignore_index or lies outside [0, V) is invalid: logp = 0,
 * lse = -inf, and it contributes nothing to any gradient; its target,
 * temperature and grad_logp entries are never used in arithmetic
 * ("recursive deterministic LogP autograd on B200", Summary: invalid token
 * ids give zero log-probability and -inf log-sum-exp).
 *
 * Determinism: every reduction runs in a fixed order that depends only on
 * (D, V) for per-row results, so logp / lse / grad_hidden rows are bitwise
 * identical for any batch size N and across runs; grad_weight / grad_bias are
 * bitwise reproducible across runs for a given input.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers into the current device's
 *     memory, row-major and contiguous.  16-bit tensors (bf16; IEEE fp16 for
 *     the *_f16 entry points) are passed as raw storage (void*).  The caller
 *     owns every buffer; the library allocates nothing and keeps no per-call
 *     state (the one exception, linear_logp_fwd_noalloc, says so below).
 *   - `stream` is a cudaStream_t of the current device (NULL = legacy default
 *     stream).  Work is enqueued on it; the library never synchronises.  A
 *     thread with no current context gets the current device's primary one.
 *   - Alignment: hidden, weight, grad_hidden, grad_weight and workspace must be
 *     16-byte aligned; bias and other float arrays 4-byte aligned;
 *     targets 8-byte aligned.
 *   - Shapes: N >= 0, 1 <= D, D % 8 == 0 (16-byte rows for the tensor-memory
 *     copies), 1 <= V, and N, D, V < 2^31 with N*D, V*D and N*V < 2^62.
 *   - N == 0: the forward is a no-op and the backward writes zeros into
 *     grad_weight / grad_bias (sums over no tokens); per-token pointers may
 *     then be NULL.  Both return LLP_OK.
 *   - Invalid arguments are reported BEFORE anything is enqueued; the outputs
 *     are then untouched.  There is no fallback path.
 *   - temperature values must be finite and > 0 (not checked on the device).
 */
#ifndef LINEAR_LOGP_H_
#define LINEAR_LOGP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  LLP_OK = 0,
  LLP_ERR_NULL_POINTER = -1,        /* a required pointer is NULL */
  LLP_ERR_BAD_SHAPE = -2,           /* N < 0, D < 1, V < 1, D % 8 != 0, or too large */
  LLP_ERR_MISALIGNED = -3,          /* a pointer violates the alignment rules above */
  LLP_ERR_UNSUPPORTED_DEVICE = -4,  /* the current device is not an sm_103 GPU */
  LLP_ERR_WORKSPACE_TOO_SMALL = -5, /* workspace_bytes below the *_workspace_bytes() query */
  LLP_ERR_CUDA = -6,                /* a CUDA runtime / driver call or launch failed */
  LLP_ERR_DEVICE_TIMEOUT = -7,      /* a kernel gave up on a wait (see linear_logp_device_status) */
  LLP_ERR_SCRATCH_LIMIT = -8        /* problem too large for linear_logp_fwd_noalloc's fixed scratch */
};

/* Scheduling note: the gradient GEMMs hand out their work units in ascending
 * order from a counter in the backward workspace when the units are long, and
 * round-robin otherwise.  Which SM computes a unit never changes the
 * arithmetic, so results are bitwise the same either way; setting the
 * environment variable LINEAR_LOGP_SCHEDULE=static before the library's first
 * call forces round-robin everywhere (a diagnostic, read once per process).
 *
 * Kernel-choice note: the backward of a batch of at most 96 rows computes
 * grad_hidden with the hidden dimension on the tensor-core MMA's M side and the
 * tokens on its N side (no padding rows are multiplied); larger batches use the
 * two-CTA GEMM with the tokens on M.  Both accumulate every element over the
 * same 16-wide vocab slices in the same order, so the results are bitwise the
 * same; LINEAR_LOGP_SMALL_GRAD_HIDDEN=0 before the first call sends small
 * batches through the two-CTA GEMM too (a diagnostic, read once per process). */

/* Bytes of workspace linear_logp_fwd needs for an N x D x V problem
 * (0 when N == 0).  The workspace holds the per-vocab-split (max, sum) pairs
 * and the captured target logits. */
size_t linear_logp_fwd_workspace_bytes(int64_t N, int64_t D, int64_t V);

/* Bytes of workspace linear_logp_bwd needs: two work-ticket counters of the
 * gradient GEMMs (set by the library itself; the workspace need not be
 * zeroed), the bf16 dlogits buffer [N, round_up(V, 64)], the grad_bias
 * partials when has_bias != 0, and the fp32 K-segment partials of grad_hidden
 * (V > 32768) and grad_weight (N > 32768). */
size_t linear_logp_bwd_workspace_bytes(int64_t N, int64_t D, int64_t V, int has_bias);

/*
 * Forward.
 *   hidden       [N, D] bf16            (required)
 *   weight       [V, D] bf16            (required)
 *   bias         [V] fp32 or NULL
 *   targets      [N] int64              (required)
 *   temperature  [N] fp32 or NULL (NULL = 1)
 *   ignore_index   target value that marks an ignored row (e.g. -100)
 *   out_logp     [N] fp32  (required; overwritten)
 *   out_lse      [N] fp32  (required; overwritten; the backward needs it)
 *   workspace    device scratch of at least linear_logp_fwd_workspace_bytes()
 * Returns LLP_OK or a negative LLP_ERR_* code.
 */
int linear_logp_fwd(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                    const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                    float* out_logp, float* out_lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward that allocates nothing and takes no workspace.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory on their own: a plugin inside a host
 * program that owns all device memory through its own allocator and hands
 * none out, a service that has already reserved the whole device (weights,
 * caches) and forbids further allocation, or a latency-critical loop where
 * cudaMalloc is not allowed because it is slow and may synchronise the device.
 *
 * Same arguments, results and checks as linear_logp_fwd, minus the workspace.
 * The scratch (per-split max / sum pairs and target logits) lives in one
 * file-scope device array of LINEAR_LOGP_NOALLOC_SCRATCH_BYTES (16 MiB) inside
 * the library; every GPU that loads the library holds it until the process
 * exits.  The problem needs about N * (8 * ceil(V / 512) + 4) bytes of it (plus
 * 256-byte alignment of each region): up to about 8000 tokens at V = 131072.
 * Larger problems return LLP_ERR_SCRATCH_LIMIT before anything is enqueued.
 *   - No cudaMalloc / cudaFree or any allocating call is made.
 *   - The first call on a device performs a one-time set-up with that device
 *     current (it looks up the array's device address); make that first call
 *     before any stream capture.  The address it keeps (like the library's
 *     other per-device set-up: kernel attributes, the status word) belongs to
 *     that device's context: after the host program destroys the context
 *     (cudaDeviceReset), unload and reload the library before calling it again.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it has to start at zero, because every call writes each
 *     scratch entry it later reads.  Calls whose work overlaps on the GPU
 *     (different streams or threads without ordering between them) race on
 *     the array and give undefined results: order them on one stream or with
 *     events.
 */
#define LINEAR_LOGP_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int linear_logp_fwd_noalloc(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                            const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                            float* out_logp, float* out_lse, void* stream);

/*
 * Backward.  Same inputs as the forward plus
 *   grad_logp    [N] fp32  upstream gradient of logp (required)
 *   saved_lse    [N] fp32  out_lse of the forward on the same inputs (required)
 * Outputs (each may be NULL to skip it; all NULL is a no-op):
 *   grad_hidden  [N, D] bf16  (overwritten, not accumulated)
 *   grad_weight  [V, D] bf16  (overwritten)
 *   grad_bias    [V] fp32     (overwritten; requires bias != NULL)
 *   workspace    device scratch of at least linear_logp_bwd_workspace_bytes()
 */
int linear_logp_bwd(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                    const float* bias, const int64_t* targets, const float* temperature, int64_t N, int64_t D,
                    int64_t V, int64_t ignore_index, void* grad_hidden, void* grad_weight, float* grad_bias,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * fp16 inputs ("Fused Linear LogP", Tensor Contract: hidden and lm_head_weight
 * may be bf16 or fp16).  Same arguments, workspaces, checks and results as
 * linear_logp_fwd / linear_logp_bwd, except that hidden and weight are IEEE
 * fp16 [N, D] / [V, D] and grad_hidden / grad_weight are written in fp16.  The
 * dlogits workspace then holds fp16 too, since both operands of a tensor-core
 * product have one type; every accumulation stays fp32.  fp16 cannot hold a
 * dlogit above 65504 in magnitude: |grad_logp / temperature| must stay below
 * that.  fp32 inputs are not accepted by any entry point (the Python wrapper
 * refuses them).  The row-subset variants have fp16 forms too
 * (linear_logp_fwd_indexed_f16 / linear_logp_bwd_indexed_f16).
 */
int linear_logp_fwd_f16(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                        const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                        float* out_logp, float* out_lse, void* workspace, size_t workspace_bytes, void* stream);
int linear_logp_bwd_f16(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                        const float* bias, const int64_t* targets, const float* temperature, int64_t N, int64_t D,
                        int64_t V, int64_t ignore_index, void* grad_hidden, void* grad_weight, float* grad_bias,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Row-subset (indexed) variants ("recursive deterministic LogP autograd on
 * B200", What: indexed semantics; "add backward support for fused logp CUDA
 * kernels", Implementation details: zero gradients for rows omitted by indexed
 * variants).  `indices` [K] int64 (device) names the token rows to compute;
 * duplicates count once, entries outside [0, N) are ignored.
 *   linear_logp_fwd_indexed writes out_logp[i] / out_lse[i] for each selected
 *     row i (bitwise the values linear_logp_fwd gives that row) and leaves every
 *     other entry of out_logp / out_lse untouched.
 *   linear_logp_bwd_indexed returns the gradients of sum over selected rows i of
 *     grad_logp[i] * logp[i]: grad_hidden is written for all N rows (zero for
 *     rows not selected); grad_weight / grad_bias sum over the selected rows.
 * Same arguments, checks and conventions as the plain calls otherwise; the
 * workspace is sized by the *_indexed_workspace_bytes queries (K = len(indices)).
 */
size_t linear_logp_fwd_indexed_workspace_bytes(int64_t N, int64_t D, int64_t V, int64_t K);
size_t linear_logp_bwd_indexed_workspace_bytes(int64_t N, int64_t D, int64_t V, int64_t K, int has_bias);
int linear_logp_fwd_indexed(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                            const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                            const int64_t* indices, int64_t K, float* out_logp, float* out_lse, void* workspace,
                            size_t workspace_bytes, void* stream);
int linear_logp_bwd_indexed(const float* grad_logp, const float* saved_lse, const void* hidden, const void* weight,
                            const float* bias, const int64_t* targets, const float* temperature, int64_t N,
                            int64_t D, int64_t V, int64_t ignore_index, const int64_t* indices, int64_t K,
                            void* grad_hidden, void* grad_weight, float* grad_bias, void* workspace,
                            size_t workspace_bytes, void* stream);
/* fp16 forms of the two row-subset variants: IEEE fp16 hidden / weight /
 * grad_hidden / grad_weight, otherwise as above (see linear_logp_fwd_f16). */
int linear_logp_fwd_indexed_f16(const void* hidden, const void* weight, const float* bias, const int64_t* targets,
                                const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                                const int64_t* indices, int64_t K, float* out_logp, float* out_lse, void* workspace,
                                size_t workspace_bytes, void* stream);
int linear_logp_bwd_indexed_f16(const float* grad_logp, const float* saved_lse, const void* hidden,
                                const void* weight, const float* bias, const int64_t* targets,
                                const float* temperature, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                                const int64_t* indices, int64_t K, void* grad_hidden, void* grad_weight,
                                float* grad_bias, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Vocab-parallel shards ("Fused Linear LogP", Tensor Parallel Vocab Shards: each
 * rank holds a contiguous weight shard [V_local, D] starting at global vocab id
 * vocab_start, computes local online-softmax state, and collectives merge the
 * global max, sum and target logit; hidden.grad is summed over ranks, the weight
 * and bias gradients stay local).  The collectives themselves belong to the
 * caller (e.g. torch.distributed all-gathers); these calls are the device work
 * around them, and every merge runs in ascending rank order so the results do
 * not depend on collective timing.
 *   linear_logp_fwd_shard: per row, the shard's max, its sum of exp(z - max) and
 *     the target logit if the (global) target lies in this shard, else -inf.
 *     Workspace: linear_logp_fwd_workspace_bytes(N, D, V_local).
 *   linear_logp_merge_shards: R shards' triples laid out [R][N] each (rank
 *     order) -> logp, lse exactly as the unsharded forward defines them; targets
 *     are valid against global_V.  The shards must partition [0, global_V).
 *   linear_logp_bwd_shard: with the merged lse, this shard's dz; writes its
 *     contribution dz_local . W_local to grad_hidden_partial (fp32 [N, D],
 *     16-byte aligned, may be NULL), and the local grad_weight / grad_bias.
 *     Workspace: linear_logp_bwd_workspace_bytes(N, D, V_local, has_bias).
 *   linear_logp_sum_partials: out (bf16, `count` elements) = sum over r = 0..R-1
 *     in ascending order of parts[r] (fp32, R x count, count % 4 == 0).
 */
int linear_logp_fwd_shard(const void* hidden, const void* weight_local, const float* bias_local,
                          const int64_t* targets, const float* temperature, int64_t N, int64_t D, int64_t V_local,
                          int64_t vocab_start, int64_t ignore_index, float* out_max, float* out_sumexp,
                          float* out_target_logit, void* workspace, size_t workspace_bytes, void* stream);
int linear_logp_merge_shards(const float* shard_max, const float* shard_sumexp, const float* shard_target_logit,
                             int64_t R, int64_t N, const int64_t* targets, int64_t global_V, int64_t ignore_index,
                             float* out_logp, float* out_lse, void* stream);
int linear_logp_bwd_shard(const float* grad_logp, const float* lse, const void* hidden, const void* weight_local,
                          const float* bias_local, const int64_t* targets, const float* temperature, int64_t N,
                          int64_t D, int64_t V_local, int64_t vocab_start, int64_t global_V, int64_t ignore_index,
                          float* grad_hidden_partial, void* grad_weight_local, float* grad_bias_local,
                          void* workspace, size_t workspace_bytes, void* stream);
int linear_logp_sum_partials(const float* parts, int64_t R, int64_t count, void* out_bf16, void* stream);
/* fp16 forms of the shard entry points: hidden / weight_local /
 * grad_weight_local in IEEE fp16 and an fp16 sum of the partials; otherwise as
 * above (see linear_logp_fwd_f16). */
int linear_logp_fwd_shard_f16(const void* hidden, const void* weight_local, const float* bias_local,
                              const int64_t* targets, const float* temperature, int64_t N, int64_t D,
                              int64_t V_local, int64_t vocab_start, int64_t ignore_index, float* out_max,
                              float* out_sumexp, float* out_target_logit, void* workspace, size_t workspace_bytes,
                              void* stream);
int linear_logp_bwd_shard_f16(const float* grad_logp, const float* lse, const void* hidden,
                              const void* weight_local, const float* bias_local, const int64_t* targets,
                              const float* temperature, int64_t N, int64_t D, int64_t V_local, int64_t vocab_start,
                              int64_t global_V, int64_t ignore_index, float* grad_hidden_partial,
                              void* grad_weight_local, float* grad_bias_local, void* workspace,
                              size_t workspace_bytes, void* stream);
int linear_logp_sum_partials_f16(const float* parts, int64_t R, int64_t count, void* out_f16, void* stream);

/* Human-readable name of a status code (static storage). */
const char* linear_logp_status_string(int status);

/*
 * Optional launch recorder (a measurement aid; off by default, not
 * thread-safe against concurrent calls).  While it is on, every forward /
 * backward call records one CUDA event on its stream when it starts and one
 * after each kernel it launches, so the time between consecutive events is the
 * device time of one launch.
 *   linear_logp_profile_start(capacity): clears the record and turns it on for
 *     at most `capacity` launches (creates the events on first use).
 *   linear_logp_profile_stop(kernel_ids, ms, capacity): turns it off,
 *     synchronises the recorded events, writes up to `capacity` (kernel id,
 *     milliseconds) pairs in launch order and returns how many launches were
 *     recorded (or a negative LLP_ERR_* code).
 *   linear_logp_kernel_name(id): name of a kernel id.
 */
int linear_logp_profile_start(int capacity);
int linear_logp_profile_stop(int* kernel_ids, float* ms, int capacity);
const char* linear_logp_kernel_name(int kernel_id);

/* Diagnostic: checks that a bounded wait in device code gives up and reports
 * instead of hanging.  Enqueues on `stream` one single-thread kernel that waits
 * on a barrier nothing will ever complete, with a limit of `limit_ns`
 * nanoseconds (1 .. 10^9); when the limit passes the kernel records
 * LINEAR_LOGP_DEVICE_SELFTEST_CODE in the status word and returns normally, so
 * the context stays usable.  Read the outcome with linear_logp_device_status.
 * Returns LLP_OK, LLP_ERR_BAD_SHAPE for a limit out of range, or an error. */
#define LINEAR_LOGP_DEVICE_SELFTEST_CODE 6u
int linear_logp_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/* Synchronises `stream`, then reads and clears the current device's kernel
 * status word.  Returns LLP_OK if no kernel gave up on a wait since the last
 * call, LLP_ERR_DEVICE_TIMEOUT if one did (the detailed code goes to
 * *device_code when it is not NULL), or LLP_ERR_CUDA.  Detailed codes: 1 a
 * tensor-core issuer waited for an operand stage, 2 a loader waited for a free
 * stage, 3 an epilogue waited for an accumulator, 4 the issuer waited for a
 * drained accumulator, 5 in-flight tensor-core work did not finish at
 * teardown, 6 the self-test below, 7 a role waited for its next work-unit id. */
int linear_logp_device_status(void* stream, unsigned int* device_code);

/* The cudaError_t code of the last CUDA call of this library that failed on the
 * calling thread (the cause behind an LLP_ERR_CUDA), 0 if none, and its name.
 * Entry points clear a pending non-sticky error that an unrelated earlier CUDA
 * call left on the calling thread, so it is not reported as theirs. */
int linear_logp_last_cuda_error(void);
const char* linear_logp_cuda_error_name(int code);
/* Diagnostic detail of the calling thread's last LLP_ERR_CUDA: the CUDA error
 * code (0 if the failing call was not a runtime call), the CUresult of a failed
 * tensor-map encoding (0 if none), and the library source line of the check
 * that failed.  Pointers may be NULL.  Returns LLP_OK. */
int linear_logp_last_failure(int* cuda_error, int* driver_result, int* site);

#ifdef __cplusplus
}
#endif

#endif /* LINEAR_LOGP_H_ */
