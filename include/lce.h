/*
 * lce.h — C ABI of the fused output-projection + cross-entropy library
 * (liblce.so, sm_103a).
 *
 * Operation. For hidden states H[N,d], a vocabulary matrix W[V,d] (tied to the
 * input embedding or not) and integer targets t[N] in which ignore_index marks
 * padding, with I = { i : t_i != ignore_index } and Nv = |I|:
 *
 *   loss    = (1/Nv) * sum_{i in I} ( logsumexp_v(h_i . w_v) - h_i . w_{t_i} )
 *   dH[i,:] = sum_v g_iv W[v,:]  for i in I, and 0 for ignored rows
 *   dW[v,:] = sum_{i in I} g_iv H[i,:]
 *   g_iv    = ( softmax_v(h_i . W^T)_v - [v == t_i] ) / Nv
 *
 * This is the output projection and loss computed in streamed chunks with
 * padding tokens skipped, so that no N x V logits buffer ever exists
 * ("OjasX 0.6.1: Training a 1B-Parameter LLM in 6.35GB of RAM", section
 * "Core Technology", the zero-byte vocabulary logits item), with the logits
 * recomputed in backward rather than kept ("6GB显卡预训练11亿参数模型：全是已发表
 * 技术，实测需375天", section "关键参数说明", --chunked-loss 512, and section
 * "内存实际花在哪里"). The row normaliser is the streaming (online) softmax
 * recurrence, which reaches the same value as the two-pass one (OjasX page,
 * "Online Softmax" note). Padding is removed by an on-device compaction into a
 * dense index list ("为什么26万词表会卡死16GB显卡", section 2.3 稀疏索引引擎).
 *
 * Conventions shared by every entry point.
 *  - All tensor arguments are DEVICE pointers owned by the caller, row-major
 *    and contiguous; the library never frees or retains them after the call.
 *  - H, W (and dH) are bf16 for lce_forward / lce_forward_backward, or the
 *    dtype given in lce_args_t; dW, loss and lse are fp32.
 *  - H, W, dH, dW base pointers must be 16-byte aligned and d % 8 == 0:
 *    W and the compacted H are read by the Tensor Memory Accelerator in rows
 *    of 16-byte multiples.
 *  - bf16 inputs run on bf16 tensor cores with fp32 accumulation. fp32
 *    inputs are split into bf16 pairs x = hi + lo and every product is formed
 *    as hi.hi + hi.lo + lo.hi (three times the tensor work, relative error
 *    about 2^-16); that path also holds a bf16 split copy of W (4*V*d bytes)
 *    in its workspace.
 *  - 1 <= N < 2^31, 1 <= d <= 65536, 1 <= V < 2^31.
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *    call returns without synchronising. Scratch memory is stream-ordered
 *    (cudaMallocAsync/cudaFreeAsync) unless a workspace is passed.
 *  - Host-detectable problems (null pointers, shapes, alignment, device)
 *    return an error code synchronously and enqueue nothing. Problems only the
 *    device can see (a non-ignored target outside [0, V), a bounded wait that
 *    gave up) never trap: they set bits in a per-device status word that
 *    lce_get_device_status reads; the loss is then NaN and the gradients are
 *    unspecified.
 *  - Nv == 0 gives loss = NaN (a mean over no tokens) and zero dH and dW.
 *  - Results are deterministic: the same inputs give bitwise-identical
 *    outputs (no floating-point atomics).
 *  - The library runs on sm_103 devices only (LCE_ERR_DEVICE otherwise).
 */
#ifndef LCE_H
#define LCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *lce_stream_t;

typedef enum {
    LCE_OK = 0,
    LCE_ERR_NULL = 1,         /* a required pointer is NULL */
    LCE_ERR_SHAPE = 2,        /* N, d, V or vocab_chunk out of range */
    LCE_ERR_ALIGN = 3,        /* base pointer or row stride not 16-byte aligned */
    LCE_ERR_DTYPE = 4,        /* unknown dtype */
    LCE_ERR_CUDA = 5,         /* a CUDA call failed; see lce_last_cuda_error() */
    LCE_ERR_WORKSPACE = 6,    /* workspace_bytes below lce_workspace_size() */
    LCE_ERR_TARGET_RANGE = 7, /* device: a non-ignored target outside [0, V) */
    LCE_ERR_TIMEOUT = 8,      /* device: a bounded wait inside a kernel gave up */
    LCE_ERR_DEVICE = 9,       /* current device is not sm_103 */
    LCE_ERR_ARG = 10          /* an option value or combination that is not supported */
} lce_status_t;

typedef enum { LCE_BF16 = 0, LCE_FP32 = 1 } lce_dtype_t;

/* Bits of the device status word (lce_get_device_status). */
#define LCE_DEV_TARGET_RANGE 0x1  /* a non-ignored target was outside [0, V) */
#define LCE_DEV_TIMEOUT      0x2  /* a pipeline wait gave up; that kernel returned early */

/*
 * Forward only: writes the mean loss to the device scalar `loss`.
 * H [N,d] bf16, W [V,d] bf16, targets [N] int64.
 */
lce_status_t lce_forward(const void *H, const void *W, const int64_t *targets,
                         int64_t ignore_index, int64_t N, int64_t d, int64_t V,
                         float *loss, lce_stream_t stream);

/*
 * Forward and backward in one call: loss (device fp32 scalar), dH [N,d] bf16
 * (overwritten; ignored rows are zero) and dW [V,d] fp32 (overwritten).
 * H, W and targets as in lce_forward. dW is fp32 so a tied W's gradient can be
 * added to the input-embedding gradient without a rounding step.
 */
lce_status_t lce_forward_backward(const void *H, const void *W, const int64_t *targets,
                                  int64_t ignore_index, int64_t N, int64_t d, int64_t V,
                                  float *loss, void *dH, float *dW, lce_stream_t stream);

/*
 * Valid-token compaction alone (the first step of every call): idx[0..Nv)
 * receives the ascending positions whose target is not ignore_index, inv[i]
 * the compacted row of position i or -1, counts[0] = Nv and counts[1] = the
 * number of non-ignored targets outside [0, V). idx and inv hold N int32
 * each, counts 2 int32; all device pointers. One CTA sweeps the targets with
 * warp ballots and a block scan; the list is exact (integer) and ascending.
 * Padding-aware valid mask of "为什么26万词表会卡死16GB显卡", section 2.3
 * 稀疏索引引擎.
 */
lce_status_t lce_compact(const int64_t *targets, int64_t N, int64_t ignore_index, int64_t V,
                         int32_t *idx, int32_t *inv, int32_t *counts, lce_stream_t stream);

/*
 * Optimizer step on W fused into the backward (lce_args_t.optim): the
 * gradient of W is consumed where it is produced, in the epilogue of each dW
 * tile, and never stored — no V x d gradient buffer exists, the "zero-byte
 * persistent .grad buffers" item of "OjasX 0.6.1: Training a 1B-Parameter LLM
 * in 6.35GB of RAM" (section "Core Technology"; its usage listing attaches an
 * "adamw" or "sgd" optimizer that updates weights in place during backward).
 * The pages do not define the two rules; these follow PyTorch's SGD and AdamW
 * (no dampening, no Nesterov, no amsgrad), with g the gradient of W
 * (grad_scale and grad_loss applied):
 *   SGD:   g += weight_decay * w; with momentum != 0: b = g on step 1, else
 *          b = momentum * b + g, and g = b (b in exp_avg); w -= lr * g.
 *   AdamW: w *= 1 - lr * weight_decay; m = beta1*m + (1-beta1)*g;
 *          v = beta2*v + (1-beta2)*g^2;
 *          w -= lr/(1-beta1^step) * m / (sqrt(v)/sqrt(1-beta2^step) + eps)
 *          (m in exp_avg, v in exp_avg_sq).
 * W is updated in place in its own dtype (bf16 rounded to nearest), or, for
 * bf16 W with master_W given, the fp32 master copy is updated and W is
 * rewritten as its bf16 rounding. Every W row is updated exactly once per
 * call, after the last read of its old value (loss, lse and dH are those of
 * the old W). State arrays are fp32 [V,d], device, 16-byte aligned, owned by
 * the caller; with state_bf16 they are bf16 [V,d] instead, as torch.optim
 * keeps them for a bf16 parameter: each is read, updated in fp32 (the update
 * of w uses the fp32 values) and stored rounded to the nearest bf16, which
 * halves their memory and traffic (12 instead of 20 bytes moved per W
 * element for AdamW on a bf16 W). Requirements (else LCE_ERR_ARG /
 * LCE_ERR_NULL): dH given and
 * dW NULL, accumulate_dW 0, one token chunk, step >= 1, lr >= 0,
 * weight_decay >= 0, 0 <= beta1, beta2 < 1, eps > 0, master_W only for bf16.
 */
typedef enum { LCE_OPT_NONE = 0, LCE_OPT_SGD = 1, LCE_OPT_ADAMW = 2 } lce_optim_kind_t;
typedef struct {
    lce_optim_kind_t kind;
    float lr;
    float weight_decay;
    float momentum;           /* SGD */
    float beta1, beta2, eps;  /* AdamW */
    int64_t step;             /* 1-based number of this update */
    float *master_W;          /* optional fp32 [V,d] master weights of a bf16 W */
    void *exp_avg;            /* [V,d] fp32 (bf16 with state_bf16): AdamW first moment, SGD momentum buffer */
    void *exp_avg_sq;         /* [V,d] fp32 (bf16 with state_bf16): AdamW second moment */
    int state_bf16;           /* nonzero: exp_avg / exp_avg_sq are bf16 */
} lce_optim_t;

/* Full argument set for lce_run. Zero-initialise, then fill. */
typedef struct {
    lce_dtype_t dtype;        /* element type of H, W and dH */
    const void *H;            /* [N,d] */
    const void *W;            /* [V,d]; written only by a fused optimizer step (optim) */
    const int64_t *targets;   /* [N] */
    int64_t ignore_index;
    int64_t N, d, V;
    float *loss;              /* device fp32 scalar; required unless lse_in is given */
    void *dH;                 /* [N,d] of dtype, or NULL for forward only */
    void *dW;                 /* [V,d] fp32 (bf16 with dW_bf16), or NULL for forward only (NULL iff dH
                                 is NULL, except that dW is NULL with a fused optimizer) */
    int accumulate_dW;        /* nonzero: dW += gradient; zero: dW = gradient */
    float grad_scale;         /* multiplies dH and dW (0 is read as 1) */
    float *lse;               /* optional [N] fp32: per-row logsumexp (natural log), NaN on ignored rows */
    void *workspace;          /* optional device scratch; NULL = stream-ordered allocation */
    size_t workspace_bytes;   /* size of `workspace` */
    int64_t vocab_chunk;      /* vocab rows per backward chunk; 0 = default (6144-row chunks, evened out over V); else a multiple of 256 */
    lce_stream_t stream;
    const float *lse_in;      /* optional [N] fp32 per-row logsumexp from an earlier forward (the `lse`
                                 output of lce_run): the forward pass is skipped, only dH/dW are
                                 computed (dH and dW required, loss may be NULL) */
    const float *grad_loss;   /* optional device fp32 scalar: upstream gradient of the loss,
                                 multiplies dH and dW (read on the device, no host sync) */
    int64_t token_chunk;      /* 0 = all N rows at once; else the rows are processed token_chunk
                                 positions at a time (scratch O(token_chunk*(d + vocab_chunk)),
                                 dW accumulated across chunks in a fixed order): the chunked loss
                                 of "6GB显卡预训练11亿参数模型", section "关键参数说明" (--chunked-loss 512) */
    const lce_optim_t *optim; /* optional: optimizer step on W fused into the backward (W is written) */
    int row_gather;           /* nonzero: the GEMMs read H's valid rows through the compaction index
                                 with TMA gather4 loads instead of from a compacted copy (no
                                 N*d*2-byte copy in the workspace; bf16 and d % 256 == 0 only, else
                                 LCE_ERR_ARG). Same results; slower on sm_103 (32 gather4 of 512
                                 bytes per pipeline stage against one tiled load). The dense index
                                 list of "为什么26万词表会卡死16GB显卡", section 2.3 稀疏索引引擎,
                                 used directly as the operand's row map. */
    int dW_bf16;              /* nonzero: dW is bf16 [V,d] (the fp32 accumulator of each element
                                 rounded to nearest once), for a bf16 W whose gradient is kept in
                                 its own dtype; half the dW bytes. bf16 inputs only, not with
                                 accumulate_dW or token chunks (else LCE_ERR_ARG). */
} lce_args_t;

/* Forward, or forward + backward when dH/dW are given, or backward alone
 * from a stored lse (lse_in), with every option. */
lce_status_t lce_run(const lce_args_t *args);

/*
 * Backward alone, for a training loop that runs the forward and backward
 * passes at different times: dH [N,d] bf16 and dW [V,d] fp32 (overwritten)
 * from the per-row lse [N] fp32 that a forward stored (lce_run with
 * args.lse), times the device scalar *grad_loss (NULL = 1). The logits are
 * recomputed from H and W ("6GB显卡预训练11亿参数模型", section "关键参数说明":
 * the chunked loss recomputes logits in backward instead of keeping them).
 * H, W, targets and ignore_index must be those of the forward.
 */
lce_status_t lce_backward(const void *H, const void *W, const int64_t *targets, int64_t ignore_index,
                          int64_t N, int64_t d, int64_t V, const float *lse, const float *grad_loss,
                          void *dH, float *dW, lce_stream_t stream);

/*
 * Bytes of scratch lce_run needs for these sizes (what the library allocates
 * itself when no workspace is passed). Grows as O(N*(d + vocab_chunk)), never
 * with N*V. Returns 0 for invalid arguments.
 */
size_t lce_workspace_size(int64_t N, int64_t d, int64_t V, lce_dtype_t dtype, int64_t vocab_chunk);

/* Bytes of scratch lce_run needs for exactly these arguments (all options,
 * token_chunk included); 0 for invalid arguments. Pointers are not read. */
size_t lce_workspace_size_args(const lce_args_t *args);

/*
 * Synchronises `stream`, then returns in *bits the current device's status
 * word (LCE_DEV_* bits accumulated since the last read) and clears it.
 * Returns LCE_ERR_TARGET_RANGE or LCE_ERR_TIMEOUT when the matching bit is
 * set, LCE_OK when the word is clear.
 */
lce_status_t lce_get_device_status(lce_stream_t stream, int32_t *bits);

/* Static string naming a status code. */
const char *lce_status_string(lce_status_t status);

/* cudaError_t value of the last CUDA failure seen by this thread (0 = none). */
int lce_last_cuda_error(void);

/* Number of kernels this library has launched in this process. */
int64_t lce_launch_count(void);

/*
 * Phase timing for profiling. While enabled (on the calling thread), every
 * call records CUDA events on its stream around each phase:
 *   0 compaction + gather of valid rows, 1 logits + online log-sum-exp,
 *   2 log-sum-exp merge + loss, 3 backward (recomputed logits -> G, dW = G^T H,
 *   dH += G W, one launch per vocab chunk), 4 scatter of dH to the caller's rows.
 * lce_profile_end synchronises those events and returns, per phase, the summed
 * milliseconds and the number of kernel launches; it then disables timing.
 * n is the length of both output arrays (at most LCE_PROFILE_PHASES used).
 */
#define LCE_PROFILE_PHASES 5
lce_status_t lce_profile_begin(void);
lce_status_t lce_profile_end(double *ms, int64_t *launches, int n);

/*
 * Forward loss like lce_forward, for callers that must not allocate device
 * memory: real-time or long-running loops whose memory budget is fixed up
 * front (an allocation can stall the device or fail from fragmentation at an
 * arbitrary point), and hosts that forbid device allocation after start-up.
 * It calls no cudaMalloc, cudaFree or other allocating routine; the pages
 * have no counterpart of this entry point.
 *
 * Scratch lives in one fixed 21 MiB device array inside the library, which
 * every GPU that loads liblce.so holds until the process exits. Limits:
 * N <= 4096 and d <= 2048 (LCE_ERR_SHAPE beyond them); bf16 H and W; other
 * arguments, layout and errors as in lce_forward. The first call on each
 * device looks up the array's device address (with that device current); make
 * that first call before any stream capture. All calls share the one array:
 * calls that overlap on the GPU (different streams, or different host threads
 * on one device) race and corrupt each other's results; serialise them.
 */
lce_status_t lce_forward_noalloc(const void *H, const void *W, const int64_t *targets,
                                 int64_t ignore_index, int64_t N, int64_t d, int64_t V,
                                 float *loss, lce_stream_t stream);

/*
 * Failure-path self-test: launches one thread that waits on a pipeline
 * barrier nothing completes, using the same bounded wait as the GEMM kernels
 * but with a limit of `cycles` SM clocks (1 .. 2^34). The wait gives up,
 * sets LCE_DEV_TIMEOUT in the device status word and the kernel returns, so
 * the context stays usable; *gave_up (device int32) receives 1. Read the
 * status with lce_get_device_status.
 */
lce_status_t lce_selftest_wait_timeout(int64_t cycles, int32_t *gave_up, lce_stream_t stream);

/*
 * Input-embedding lookup that skips padding, for a vocabulary matrix W shared
 * by the input lookup and the output projection ("6GB显卡预训练11亿参数模型",
 * section "关键参数说明", --tie-embeddings):
 *   E[i,:] = W[tokens[i],:] where tokens[i] != pad_id, a zero row where it is.
 * The valid mask and the lookup run in one kernel with no host
 * synchronisation ("为什么26万词表会卡死16GB显卡", section 2.3 稀疏索引引擎).
 * W [V,d] and E [N,d] are device arrays of `dtype`; tokens [N] int64.
 * A non-padding token outside [0, V) gets a zero row and sets
 * LCE_DEV_TARGET_RANGE in the device status word. Same shape, alignment and
 * error rules as lce_run (d % 8 == 0, 16-byte aligned W and E).
 */
lce_status_t lce_embedding_forward(lce_dtype_t dtype, const void *W, const int64_t *tokens, int64_t pad_id,
                                   int64_t N, int64_t d, int64_t V, void *E, lce_stream_t stream);

/*
 * Gradient of lce_embedding_forward with respect to W:
 *   dW[v,:] (+)= sum of dE[i,:] over the positions i with tokens[i] == v,
 * for tokens that are not pad_id and lie in [0, V) (others are skipped and
 * flagged as in the forward). dE [N,d] of `dtype`, dW [V,d] fp32 (device).
 * accumulate = 0 overwrites dW (rows of tokens that do not occur become 0);
 * nonzero adds into it, so for a tied W the output projection's dW (lce_run)
 * and this gradient sum into one buffer. The positions are grouped by token
 * on the device and each row's sum is taken in ascending position order (the
 * batch's per-token gradients aggregated after backward, same page, section
 * 2.2, without atomics): results are reproducible bit for bit.
 * The grouping is a stable radix sort of the valid positions by token over
 * several CTAs; the sorted list is cut into fixed chunks of 32, each token's
 * rows in a chunk are summed in order and a token whose rows span chunks
 * gets its chunk sums added in chunk order. Scratch: lce_embedding_workspace_size(N, d) bytes of
 * `workspace` (device, 16-byte aligned), or NULL for a stream-ordered
 * allocation.
 */
size_t lce_embedding_workspace_size(int64_t N, int64_t d);
lce_status_t lce_embedding_backward(lce_dtype_t dtype, const void *dE, const int64_t *tokens, int64_t pad_id,
                                    int64_t N, int64_t d, int64_t V, float *dW, int accumulate, void *workspace,
                                    size_t workspace_bytes, lce_stream_t stream);

/*
 * The same gradient written as bf16 [V,d] (dW, device, 16-byte aligned):
 * every row sum is taken in fp32 exactly as above and rounded to nearest once
 * when it is stored, so the result equals lce_embedding_backward's fp32 dW
 * rounded to bf16. For a bf16 W whose gradient is kept in its own dtype; dW
 * is overwritten (no accumulation: a second rounding would follow).
 */
lce_status_t lce_embedding_backward_bf16(lce_dtype_t dtype, const void *dE, const int64_t *tokens, int64_t pad_id,
                                         int64_t N, int64_t d, int64_t V, void *dW, void *workspace,
                                         size_t workspace_bytes, lce_stream_t stream);

/* ABI version: major*10000 + minor*100 + patch. */
int lce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LCE_H */
