/*
 * h3attn.h -- C ABI of the batch-invariant MiniMax-H3 attention core (sm_103a).
 *
 * The library computes, for a packed sequence of independent samples,
 *
 *   q^ = RoPE(RMSNorm(q) * q_norm_w),  k^ = RoPE(RMSNorm(k) * k_norm_w)
 *   out_i = sum_j softmax_j(scale * q^_i . k^_j) v_j     (j in i's sample only)
 *
 * and its gradients.  The operations are the q_norm/k_norm, rope_q/rope_k and
 * attention nodes of one MiniMax-H3 transformer block as bound on the
 * "ws1_one_h3_block" page of RL-Kernel (PR #539), Bindings table: RMSNorm on
 * the 128-wide heads with a 128-element weight, partial 3-axis multimodal RoPE
 * from packed (t, h, w) position ids, non-causal attention per packed sample.
 * The numerical contract follows the strict mode of the "ws1_full_h3_transformer"
 * page (PR #571), Scope / Known limitations: no TF32, no fast-math, no split-K,
 * FP32 accumulation, and unsupported shapes, dtypes and devices are rejected
 * with an error instead of falling back.  Each sample's results are bitwise
 * identical whether it runs alone or packed with other samples, and from run
 * to run (same page, rollout-vs-train control).
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Tensors are caller-owned DEVICE memory on the current CUDA device, except
 *   where a comment says otherwise.  The library never frees them.
 * - bf16 tensors q, k, v, out, dout, dq, dk, dv are token-major and contiguous:
 *   element (token i, head h, channel c) sits at index (i * H + h) * 128 + c.
 *   Every tensor pointer must be 16-byte aligned.
 * - pos_ids[0..2] are int32 [total_tokens] arrays of the t, h and w position of
 *   each token.  seg_offsets is int32 [num_samples + 1]: 0, then strictly
 *   increasing sample ends, the last equal to total_tokens.  Sample s owns
 *   tokens [seg_offsets[s], seg_offsets[s + 1]).  Both are read on the device.
 * - lse is float32 [H, total_tokens]: lse[h * S + i] = log sum_j exp(scale q^_i.k^_j).
 * - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and is asynchronous.  A handle must not be used by two streams at
 *   the same time (it owns one workspace).
 * - Errors found on the host (bad arguments, capacity, unsupported config)
 *   return immediately and enqueue nothing.  Errors found on the device (an
 *   invalid seg_offsets array, a bounded wait that timed out) are recorded in
 *   the handle and returned by h3attn_device_status().
 */
#ifndef H3ATTN_H
#define H3ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct h3attn_ctx *h3attn_t;

/* IEEE bfloat16 bit pattern. */
typedef uint16_t h3attn_bf16;

typedef enum {
    H3ATTN_OK = 0,
    H3ATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad sizes, bad offsets */
    H3ATTN_ERR_UNSUPPORTED = 2,  /* head_dim != 128, unsupported RoPE layout, device not sm_103 */
    H3ATTN_ERR_CAPACITY = 3,     /* total_tokens > max_tokens or num_samples > max_samples */
    H3ATTN_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    H3ATTN_ERR_TIMEOUT = 5       /* a bounded on-device wait expired (kernel returned early) */
} h3attn_status;

typedef struct {
    int num_heads;         /* H, heads of q, k and v (no grouped heads), >= 1           */
    int head_dim;          /* must be 128                                               */
    float eps;             /* RMSNorm epsilon, added to the mean square inside the sqrt */
    float rope_theta;      /* RoPE base, e.g. 10000                                     */
    int rope_sections[3];  /* rotary channels of the t, h, w axes, in that order from
                              channel 0; each a multiple of 8, sum <= 128; channels
                              past the sum are not rotated.  e.g. {16, 24, 24}         */
    int rope_pairing;      /* 0 = rotate-half inside each section (the only one)        */
    float softmax_scale;   /* 0 -> 1/sqrt(128)                                          */
    int max_tokens;        /* capacity: largest total_tokens of any call                */
    int max_samples;       /* capacity: largest num_samples of any call                 */
    int key_order;         /* H3ATTN_KEY_ORDER_PACKED (0) or H3ATTN_KEY_ORDER_CANONICAL */
    int store_ds;          /* 1: the dK/dV kernel also writes dS to the workspace and dQ
                              is one product per block (faster; workspace H * ceil(T/128)
                              * (ceil(T/128) + max_samples) * 32 KB, T = max_tokens);
                              0: the dQ kernel recomputes S and dP.  Both are
                              deterministic and identical alone vs packed; dq may
                              differ between them in the last bits (dS comes from the
                              transposed product in the first)                        */
    int reuse_qk_hat;      /* 1: h3attn_backward skips the q/k norm + RoPE pass when the
                              handle's last forward (h3attn_forward or
                              h3attn_qkv_forward, packed key order) computed the
                              rotated rows from the same q, k, norm-weight, position
                              and offset pointers and sizes: the workspace still
                              holds them.  The caller promises that the contents of
                              those tensors did not change in between (as a training
                              step's saved tensors do not); results are bitwise those
                              of the recomputation.  0: always recompute.           */
} h3attn_config;

/*
 * Order in which a call sums over a sample's tokens.
 *
 * PACKED: keys (forward, dq) and queries (dk, dv, weight gradients) are summed
 * in the order the tokens sit in memory.  Results are bitwise repeatable and
 * identical alone vs packed, but permuting a sample's rows (with their
 * positions) changes output bits: control H-C3 in the Results of the
 * "ws1_one_h3_block" page of RL-Kernel (PR #539).
 *
 * CANONICAL: every call first sorts each sample's tokens by
 *   1. position (t, h, w) as signed integers, t first;
 *   2. the k row, then the v row, then the q row (and in the backward the dout
 *      row), each over all heads in memory order, as sequences of bf16 bit
 *      patterns compared as unsigned 16-bit integers;
 *   3. packed index (tokens equal up to here are identical in every input);
 * gathers its per-token inputs into that order, runs the same kernels and
 * scatters the outputs back.  Every output bit is then also independent of how
 * each sample's tokens are permuted in memory.  Cost: an O(L^2) rank count per
 * sample of L tokens and HBM-bound row copies (forward: v in, out back;
 * backward: v, dout in, dv back; q, k, out, dq and dk are read or written in
 * place through the order), and four more [max_tokens, H, 128] bf16 buffers in
 * the workspace.
 */
#define H3ATTN_KEY_ORDER_PACKED 0
#define H3ATTN_KEY_ORDER_CANONICAL 1

/*
 * Creates a handle on the current CUDA device and allocates its workspace
 * (rotated q^/k^ buffers of max_tokens * H * 128 fp16 each, the backward's FP32
 * dq^/dk^ rows of max_tokens * H * 128 floats each, a max_tokens * 256-float
 * rotary cos/sin table, softmax row terms,
 * weight-gradient partials, a small per-call plan, 16 bytes of sort key per
 * token for the canonical order).  The workspace is bounded by the config,
 * never by the inputs.  *out receives the handle.  With
 * key_order CANONICAL it also allocates the order's buffers: a permutation and
 * positions (4 * max_tokens int32), row terms (H * max_tokens floats) and four
 * max_tokens * H * 128 bf16 row copies.
 * With store_ds = 1 it also allocates the stored dS blocks (see store_ds).
 * Errors: INVALID_ARG (null pointer, sizes < 1, key_order, store_ds or
 * reuse_qk_hat not 0 or 1), UNSUPPORTED (head_dim, pairing, sections, device not sm_103),
 * CAPACITY (the stored dS would exceed 2^31 rows of 128 values), CUDA
 * (allocation failed).
 */
h3attn_status h3attn_create(const h3attn_config *cfg, h3attn_t *out);

/* Frees the workspace and the handle (synchronises the device first). NULL is OK. */
h3attn_status h3attn_destroy(h3attn_t h);

/*
 * Forward: out = attention(RoPE(RMSNorm(q) w_q), RoPE(RMSNorm(k) w_k), v) per sample.
 * q, k, v: bf16 [S, H, 128]; q_norm_w, k_norm_w: float32 [128]; out: bf16 [S, H, 128]
 * (written for every token); lse: float32 [H, S] or NULL (not needed for
 * inference, required by h3attn_backward).
 * total_tokens == 0 is a no-op.  Errors: INVALID_ARG, CAPACITY, CUDA.
 */
h3attn_status h3attn_forward(h3attn_t h,
                             const h3attn_bf16 *q, const h3attn_bf16 *k, const h3attn_bf16 *v,
                             const float *q_norm_w, const float *k_norm_w,
                             const int32_t *const pos_ids[3], const int32_t *seg_offsets,
                             int num_samples, int total_tokens,
                             h3attn_bf16 *out, float *lse, void *stream);

/*
 * Backward of sum(out * dout) through attention, RoPE and RMSNorm.
 * Inputs as in h3attn_forward plus out (bf16 [S, H, 128]) and lse (float32
 * [H, S]) from the forward of the same inputs, and dout (bf16 [S, H, 128]).
 * Outputs: dq, dk, dv bf16 [S, H, 128]; dq_norm_w, dk_norm_w float32 [128]
 * (overwritten with the sum over all tokens and heads, samples added in index
 * order); dq_norm_w_per_sample, dk_norm_w_per_sample float32 [num_samples, 128]
 * or NULL (per-sample sums; these, like dq/dk/dv, are identical whether a sample
 * runs alone or packed).  All reductions run in a fixed order, no atomics: the
 * weight gradients per (sample, head) over 128-token tiles, then per sample over
 * heads, then over samples, each in ascending order (see the head-sharded runs
 * below).
 * With key_order CANONICAL the order of every sum is the canonical one (see
 * H3ATTN_KEY_ORDER_CANONICAL), including the dout rows in the sort.
 * Errors: INVALID_ARG, CAPACITY, CUDA.
 */
h3attn_status h3attn_backward(h3attn_t h,
                              const h3attn_bf16 *q, const h3attn_bf16 *k, const h3attn_bf16 *v,
                              const float *q_norm_w, const float *k_norm_w,
                              const int32_t *const pos_ids[3], const int32_t *seg_offsets,
                              int num_samples, int total_tokens,
                              const h3attn_bf16 *out, const float *lse, const h3attn_bf16 *dout,
                              h3attn_bf16 *dq, h3attn_bf16 *dk, h3attn_bf16 *dv,
                              float *dq_norm_w, float *dk_norm_w,
                              float *dq_norm_w_per_sample, float *dk_norm_w_per_sample,
                              void *stream);

/*
 * Waits for `stream`, then returns and clears the errors the device recorded
 * since the last call: INVALID_ARG (seg_offsets not 0 / increasing / ending at
 * total_tokens; or a finite rotated q^/k^ value beyond the fp16 range of the
 * tensor-core operands, |x| > 65504; or a non-finite dq/dk row, which from
 * finite inputs means the fp16 softmax gradient dS overflowed; outputs of that
 * call are unspecified), TIMEOUT (a bounded wait
 * expired; outputs unspecified), CUDA (an asynchronous CUDA error), else OK.
 */
h3attn_status h3attn_device_status(h3attn_t h, void *stream);

/*
 * The canonical order itself (see H3ATTN_KEY_ORDER_CANONICAL), for callers
 * that want to store or check it; usable with a handle of either key order.
 * Inputs as in h3attn_forward; dout (bf16 [S, H, 128]) may be NULL, and when
 * given joins the sort after q, as in the backward.  perm: device int32
 * [total_tokens], caller-owned, receives for every canonical slot c the packed
 * index of the token placed there; the slots of sample s are seg_offsets[s] ..
 * seg_offsets[s + 1] - 1, so perm only moves tokens within their sample.
 * Integer work only: perm is exact.  total_tokens == 0 is a no-op.
 * Errors: INVALID_ARG, CAPACITY, CUDA (host); an invalid seg_offsets array is
 * reported by h3attn_device_status and leaves perm unspecified.
 */
/*
 * The QKV projection and the attention forward in one call:
 *   [q | k | v] = x w_qkv^T (+ b_qkv), rounded once to bf16,
 *   then out, lse = h3attn_forward(q, k, v, ...).
 * The projection is the block's QKV node ("ws1_one_h3_block" page of
 * RL-Kernel, PR #539, Bindings table) and its epilogue also performs the q/k
 * RMSNorm + RoPE while each row is on chip (the separate prologue pass of
 * h3attn_forward is skipped).  x: bf16 [total_tokens, in_features];
 * w_qkv: bf16 [3 * H * 128, in_features], rows = the q heads, then the k
 * heads, then the v heads (each 128 rows, head-major); b_qkv: float32
 * [3 * H * 128] or NULL.  q, k, v: bf16 [total_tokens, H, 128], written (the
 * backward takes them); out, lse as in h3attn_forward.  Other inputs as in
 * h3attn_forward.  Results are bitwise those of h3attn_linear on the same x,
 * w_qkv, b_qkv, split into q, k, v, followed by h3attn_forward.
 * Requires in_features % 64 == 0 and a handle with the packed key order,
 * else UNSUPPORTED.  total_tokens == 0 is a no-op.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY, CUDA.
 */
h3attn_status h3attn_qkv_forward(h3attn_t h, const h3attn_bf16 *x, int in_features,
                                 const h3attn_bf16 *w_qkv, const float *b_qkv,
                                 const float *q_norm_w, const float *k_norm_w,
                                 const int32_t *const pos_ids[3], const int32_t *seg_offsets,
                                 int num_samples, int total_tokens,
                                 h3attn_bf16 *q, h3attn_bf16 *k, h3attn_bf16 *v,
                                 h3attn_bf16 *out, float *lse, void *stream);

h3attn_status h3attn_canonical_order(h3attn_t h,
                                     const h3attn_bf16 *q, const h3attn_bf16 *k, const h3attn_bf16 *v,
                                     const h3attn_bf16 *dout,
                                     const int32_t *const pos_ids[3], const int32_t *seg_offsets,
                                     int num_samples, int total_tokens,
                                     int32_t *perm, void *stream);

/*
 * Per-stage GPU time, for profiling (instrumentation; not part of the method).
 * When enabled, every launch of a stage is bracketed by CUDA events on the call's
 * stream (about 2 x 7 events per forward + backward; up to 4096 per handle,
 * later launches are not timed).  h3attn_stage_times() waits for those events,
 * writes the summed milliseconds and launch counts of each stage (arrays of
 * n_stages, stage order below) and resets the record.  Events are created on
 * first use.  Errors: INVALID_ARG, CUDA.
 */
enum {
    H3ATTN_STAGE_PLAN = 0,      /* seg_offsets check + sample order            */
    H3ATTN_STAGE_PROLOGUE = 1,  /* q/k RMSNorm + RoPE -> q^, k^                */
    H3ATTN_STAGE_FWD = 2,       /* QK^T, online softmax, PV, lse               */
    H3ATTN_STAGE_BWD_DELTA = 3, /* rowsum(dO * O)                              */
    H3ATTN_STAGE_BWD_DKDV = 4,  /* dK (through RoPE/RMSNorm), dV               */
    H3ATTN_STAGE_BWD_DQ = 5,    /* dQ (through RoPE/RMSNorm)                   */
    H3ATTN_STAGE_BWD_DW = 6,    /* fixed-order norm-weight gradient reduction  */
    H3ATTN_STAGE_BWD_ROWS = 7,  /* RoPE^-1 + RMSNorm backward of dq^, dk^ rows */
    H3ATTN_STAGE_ORDER = 8,     /* canonical order: rank count per sample      */
    H3ATTN_STAGE_PERMUTE = 9,   /* canonical order: row gathers and scatters   */
    H3ATTN_STAGE_QKV = 10,      /* fused QKV projection + q/k norm and RoPE    */
    H3ATTN_NUM_STAGES = 11
};
h3attn_status h3attn_set_stage_timing(h3attn_t h, int enable);
h3attn_status h3attn_stage_times(h3attn_t h, float *total_ms, int *launches, int n_stages);

/*
 * h3attn_forward_static: the forward for callers that cannot allocate device
 * memory (there is no counterpart on the pages; it is a deployment aid).
 *
 * Hosts such as inference servers that hand a plugin a fixed memory pool, or
 * processes that run under a device-memory budget, may not call cudaMalloc once
 * they are serving; h3attn_create's workspace is then out of reach.  This entry
 * point takes no handle and allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library call): its scratch - rotated q^/k^ rows, the sample plan
 * and an error word, 64 MiB + 64 KiB in all - is one static __device__ array
 * of the library, which every GPU that loads the library holds until the
 * process exits.
 *
 * Arguments are those of h3attn_forward with the configuration passed directly
 * (cfg->max_tokens, cfg->max_samples and cfg->store_ds are ignored), plus device_error_flags:
 * a device uint32 (may be NULL) that receives this call's device-side error
 * bits (0 = none; 1 = invalid seg_offsets, 2 = a bounded wait timed out, 4 = a
 * value beyond the fp16 operand range), written on `stream` after the kernels.
 * Limits: total_tokens * num_heads <= H3ATTN_STATIC_MAX_TOKEN_HEADS and
 * num_samples <= H3ATTN_STATIC_MAX_SAMPLES, else H3ATTN_ERR_CAPACITY.
 * The first call on a device resolves the array's device address and prepares
 * the kernels for that device (make that first call before any stream
 * capture).  Every call on a device shares the one array and leaves its
 * contents behind; the call clears what must start at zero.  Two calls whose
 * work overlaps on the GPU (different streams, or different host threads)
 * race on the array: serialise them.  Results are bitwise those of
 * h3attn_forward for the same inputs.  Only the packed key order is offered
 * (the canonical order's row copies do not fit the static scratch):
 * cfg->key_order != H3ATTN_KEY_ORDER_PACKED returns UNSUPPORTED.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY, CUDA.
 */
#define H3ATTN_STATIC_MAX_TOKEN_HEADS 131072
#define H3ATTN_STATIC_MAX_SAMPLES 2048
h3attn_status h3attn_forward_static(const h3attn_config *cfg,
                                    const h3attn_bf16 *q, const h3attn_bf16 *k, const h3attn_bf16 *v,
                                    const float *q_norm_w, const float *k_norm_w,
                                    const int32_t *const pos_ids[3], const int32_t *seg_offsets,
                                    int num_samples, int total_tokens,
                                    h3attn_bf16 *out, float *lse, uint32_t *device_error_flags,
                                    void *stream);

/*
 * The projection either side of the attention core (the block's QKV
 * projection feeding the q/k norms, and its output projection; "ws1_one_h3_block"
 * page of RL-Kernel, PR #539, Bindings table and Prior art): y = x W^T (+ b).
 *   x  bf16 [rows, in_features] row-major;  w bf16 [out_features, in_features]
 *      row-major (a linear layer's [out, in] weight);  bias FP32 [out_features]
 *      or NULL;  y bf16 [rows, out_features] row-major.  Caller-owned device
 *      memory, 16-byte aligned.  The q, k and v of the attention are three calls
 *      (or one call with the three weights stacked and the outputs split after).
 *   FP32 accumulation over in_features in ascending order, one rounding to bf16
 *   after the bias: each output row's bits depend only on that row of x and on
 *   w and bias (the same whatever the number of rows or the row's position).
 *   device_error_flags: device uint32, required; the call clears it on `stream`
 *   and sets bit 2 if an on-device wait timed out (outputs then unspecified).
 * Needs in_features % 64 == 0 and out_features % 32 == 0 (UNSUPPORTED
 * otherwise).  rows == 0 is a no-op.  Asynchronous on `stream`; allocates
 * nothing.  Errors: INVALID_ARG (sizes < 0, null or misaligned pointers),
 * UNSUPPORTED (shapes, device not sm_103), CAPACITY, CUDA.
 */
h3attn_status h3attn_linear(const h3attn_bf16 *x, int rows, int in_features,
                            const h3attn_bf16 *w, int out_features, const float *bias,
                            h3attn_bf16 *y, uint32_t *device_error_flags, void *stream);

/*
 * Head-sharded runs.  The path has no exchange step between heads: a layer's
 * heads can be split across GPUs, each GPU running its own heads (q, k, v,
 * dout as contiguous [S, H_g, 128] tensors) through a handle of H_g heads, and
 * its out, lse, dq, dk and dv are bitwise those of a one-GPU run of all heads.
 * The norm weights are shared by all heads, so their gradient needs the other
 * GPUs' heads; it is reduced in a fixed order that does not depend on how the
 * heads are split: per (sample, head) over the sample's 128-token tiles in
 * ascending order, then per sample over heads in ascending order, then over
 * samples in ascending order (h3attn_backward itself reduces this way).  A
 * head-sharded run gathers every GPU's (sample, head) partials in head order
 * and reduces them with h3attn_combine_norm_weight_grads: the result is
 * bitwise the one-GPU result for every split.  (The pages' precedent is the
 * WS2 parallel layer, ws2_comm.py in the changed-file list of the
 * "ws1_full_h3_transformer" page, PR #571.)
 *
 * h3attn_norm_weight_grad_partials: copies the per-(sample, head) partials of
 * the handle's last h3attn_backward call, float32 [num_samples, H, 128] each
 * for q_norm_w and k_norm_w, into caller-owned device memory, on `stream`
 * (call it on the backward's stream, before the next backward on the handle).
 * Nothing is copied before the first backward or after an empty one.
 * Errors: INVALID_ARG (null handle or pointer, other device), CUDA.
 *
 * h3attn_combine_norm_weight_grads: partials float32 [num_samples,
 * num_heads, 128] (device, heads in global order) -> per_sample float32
 * [num_samples, 128] (device, required: the total is summed from it) and
 * total float32 [128] (device).  Allocates nothing; asynchronous on `stream`.
 * num_samples == 0 zeroes total.  Errors: INVALID_ARG (sizes, null or
 * misaligned pointers), UNSUPPORTED (device not sm_103), CUDA.
 */
h3attn_status h3attn_norm_weight_grad_partials(h3attn_t h, float *dq_norm_w_partials, float *dk_norm_w_partials,
                                               void *stream);
h3attn_status h3attn_combine_norm_weight_grads(const float *partials, int num_samples, int num_heads,
                                               float *per_sample, float *total, void *stream);

/*
 * A 64-bit fingerprint of `bytes` bytes of device memory at `data`, computed on
 * the GPU and written to the device uint64 *fingerprint on `stream`, so that
 * runs can be compared without copying their outputs to the host (the
 * "ws1_full_h3_transformer" page, PR #571, Status: GPU-side checksum
 * fingerprints of the provider and candidate runs).  Definition: the bytes as
 * little-endian 64-bit words w_0 .. w_{m-1} (the last zero-padded), mix() the
 * splitmix64 finaliser (shifts 30, 27, 31; multipliers 0xbf58476d1ce4e5b9 and
 * 0x94d049bb133111eb), G = 0x9e3779b97f4a7c15:
 *   fingerprint = mix( sum_i mix(w_i + (i + 1) G) + bytes )   (mod 2^64).
 * The sum is an integer sum, so the value is a pure function of the bytes
 * (no dependence on the GPU's thread order).  data must be 8-byte aligned (may
 * be NULL when bytes == 0), fingerprint 8-byte aligned.  Allocates nothing.
 * Errors: INVALID_ARG, UNSUPPORTED (device not sm_103), CUDA.
 */
h3attn_status h3attn_fingerprint(const void *data, uint64_t bytes, uint64_t *fingerprint, void *stream);

/*
 * Test hook for the bounded waits (instrumentation; no counterpart on the
 * pages, which ask that a failure close rather than fall back: the strict mode
 * of the "ws1_full_h3_transformer" page, PR #571, Scope / Known limitations).
 * The next h3attn_forward, h3attn_backward or h3attn_qkv_forward call on this
 * handle makes one role of one kernel wait once, early in its first work item,
 * on an on-device barrier that nothing completes.  That wait gives up after
 * budget_cycles SM clock cycles, as every wait of the library does after its
 * own budget: the kernel records TIMEOUT, its other warps leave their loops,
 * it waits for the bulk copies and tensor-core products it already issued,
 * releases its tensor memory and returns.  h3attn_device_status() then
 * returns H3ATTN_ERR_TIMEOUT (outputs of that call are unspecified) and the
 * following call is an ordinary one.  The request is cleared by the call that
 * reads it, whether or not that call launches the named kernel.
 * kernel: H3ATTN_STALL_FWD (attention forward), H3ATTN_STALL_DKDV,
 * H3ATTN_STALL_DQ (whichever dQ kernel the handle runs), H3ATTN_STALL_QKV (the
 * fused QKV projection of h3attn_qkv_forward), or 0 to cancel a request;
 * role: H3ATTN_STALL_PRODUCER (the TMA producer warp), H3ATTN_STALL_MMA (the
 * tensor-core issuer), H3ATTN_STALL_CONSUMER (a softmax or epilogue warp).
 * Errors: INVALID_ARG (null handle, unknown kernel or role, budget_cycles < 1).
 */
#define H3ATTN_STALL_FWD 1
#define H3ATTN_STALL_DKDV 2
#define H3ATTN_STALL_DQ 3
#define H3ATTN_STALL_QKV 4
#define H3ATTN_STALL_PRODUCER 1
#define H3ATTN_STALL_MMA 2
#define H3ATTN_STALL_CONSUMER 3
h3attn_status h3attn_debug_stall(h3attn_t h, int kernel, int role, long long budget_cycles);

/*
 * Test hook (instrumentation; no counterpart on the pages): y[i] = 2^x[i] by
 * one of the attention kernels' two exponential paths, path 0 = the SFU
 * instruction (ex2.approx.ftz.f32), path 1 = the FMA-pipe polynomial the
 * softmax uses for a fixed share of its columns (range reduction to
 * x = n + f, f in [0, 1), a degree-5 minimax polynomial for 2^f, 2^n through
 * the exponent field; results below 2^-126 are 0; valid for x <= 127).
 * x, y: device float32 [n].  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
h3attn_status h3attn_debug_exp2(const float *x, float *y, int n, int path, void *stream);

/* Static, human-readable name of a status code. */
const char *h3attn_status_string(h3attn_status s);

#ifdef __cplusplus
}
#endif

#endif /* H3ATTN_H */
