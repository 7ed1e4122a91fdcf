/*
 * nc.h -- C ABI of the nanochat pretraining step on one B300 (sm_103a).
 *
 * The step is the one the nanochat pages describe for pretraining: the
 * depth-dialled decoder-only GPT (nanochat explainer, "Architecture Choices"
 * and "How dimensions are derived") run forward, scored with the mean
 * next-token cross-entropy (same page, "The Full Pipeline" / "Pretraining":
 * given tokens 1..N predict N+1), and differentiated analytically w.r.t.
 * every parameter.
 *
 * Model: untied token embedding wte[V,d]; `depth` pre-norm blocks, each
 *   xn1 = rmsnorm(x); q,k,v = split(xn1 W_qkv^T);
 *   q,k <- rope(rmsnorm_per_head(q,k)) (QK-norm + RoPE, half-split pairs,
 *          angle pos * 10000^(-j/64));
 *   o = causal softmax(q k^T / sqrt(128)) v;  x += o W_o^T;
 *   xn2 = rmsnorm(x); x += relu(xn2 W_fc^T)^2 W_proj^T;
 * then hf = rmsnorm(x), logits = hf lm_head^T. RMSNorm is parameter-free,
 * y = z / sqrt(mean(z^2) + 1e-6). Loss = mean over all B*T positions of
 * logsumexp(logits) - logit[target], in nats.
 *
 * Conventions shared by every call:
 *  - Every call returns nc_status; no C++ exception crosses the ABI.
 *    nc_last_error() gives a message for the calling thread's last failure.
 *  - Device pointers are plain CUDA device addresses owned by the caller; the
 *    library never frees them. The library itself allocates only a small
 *    RoPE cos/sin table and a device status word (at nc_configure).
 *  - All work is enqueued on the stream given to nc_configure (0 = legacy
 *    default stream) and is asynchronous unless stated otherwise.
 *  - Kernels never trap. A device-side failure (token id out of range, a
 *    pipeline wait that exceeded its iteration limit) sets the status word;
 *    the next synchronising call returns NC_ERR_DEVICE or NC_ERR_TIMEOUT.
 */
#ifndef NC_H
#define NC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct nc_ctx nc_ctx;

typedef enum {
  NC_OK = 0,
  NC_ERR_ARG = 1,         /* bad shape, null pointer, misaligned buffer */
  NC_ERR_STATE = 2,       /* call out of order (e.g. backward before forward) */
  NC_ERR_CUDA = 3,        /* a CUDA runtime call failed (message has the code) */
  NC_ERR_TIMEOUT = 4,     /* a device pipeline wait exceeded its limit */
  NC_ERR_DEVICE = 5,      /* device-side check failed (e.g. token id >= vocab) */
  NC_ERR_UNSUPPORTED = 6  /* valid request the library does not serve     */
} nc_status;

/* Precision modes for nc_configure. */
enum {
  NC_BF16 = 0,       /* bf16 params and stored activations, fp32 accumulate,
                        tcgen05 tensor-core kernels */
  NC_FP32_DEBUG = 1  /* fp32 params and activations, plain fp32 FMA kernels */
};

/* Create a context for one model shape. Host only; touches no GPU.
 * depth >= 1; d_model == 128 * n_head (head_dim is fixed at 128, nanochat
 * explainer "How dimensions are derived"); vocab % 128 == 0 and
 * 128 <= vocab <= 2^20; seq_len >= 1. d_model = 64 * depth is the pages'
 * rule but is not enforced, so that a depth-2 model of width 128 exists.
 * On success *out owns the context (free with nc_destroy). */
nc_status nc_create(int depth, int d_model, int n_head, int seq_len, int vocab, nc_ctx** out);

/* Fix the batch size and precision and bind a CUDA stream (a cudaStream_t,
 * may be NULL). Uses the current CUDA device. Allocates the RoPE table
 * (fp32 [seq_len, 64], angles formed in float64 on the host) and the status
 * word. NC_BF16 requires seq_len % 128 == 0 and d_model % 128 == 0.
 * Can be called again to change batch or precision; the workspace must then
 * be set again. */
nc_status nc_configure(nc_ctx* ctx, int batch, int precision, void* cuda_stream);

/* Number of parameters: 2*V*d + 12*depth*d^2. */
size_t nc_param_count(const nc_ctx* ctx);

/* Layout of the flat parameter (and gradient) vector, in elements.
 * index 0 = wte[V,d]; for layer l, 1+4l = w_qkv[3d,d] (rows: q, then k,
 * then v; row h*128+j is dim j of head h), 2+4l = w_o[d,d],
 * 3+4l = w_fc[4d,d], 4+4l = w_proj[d,4d]; index 1+4*depth = lm_head[V,d].
 * Matrices are row-major [out, in]; every offset is a multiple of 128. */
nc_status nc_param_offset(const nc_ctx* ctx, int index, size_t* offset, int* rows, int* cols);

/* Bytes of device workspace the configured step needs (activation stash
 * for the backward pass plus scratch). 0 before nc_configure. */
size_t nc_workspace_bytes(const nc_ctx* ctx);

/* Hand the context a caller-owned device buffer of at least
 * nc_workspace_bytes() bytes, 1024-byte aligned. The buffer must outlive
 * every later call that uses it. */
nc_status nc_set_workspace(nc_ctx* ctx, void* dev_ptr, size_t bytes);

/* Forward pass + mean next-token cross-entropy.
 * params: device, nc_param_count() elements, bf16 (NC_BF16) or fp32
 *   (NC_FP32_DEBUG), layout of nc_param_offset.
 * tokens, targets: device int32 [batch, seq_len] row-major, ids in
 *   [0, vocab); an id out of range makes the step return NC_ERR_DEVICE.
 *   A target of -1 masks its position (the supervised fine-tuning variant
 *   of the nanochat explainer, "Supervised Fine-Tuning (SFT)": the loss is
 *   taken on the response tokens only): it adds no loss and no gradient,
 *   and the loss is the mean over the other positions (0 if none).
 * loss: HOST float*; the call synchronises the stream and writes the loss.
 * The context keeps params/tokens/targets pointers for nc_backward: the
 * caller must not change those buffers (or the workspace) in between. */
nc_status nc_forward_loss(nc_ctx* ctx, const void* params, const int32_t* tokens,
                          const int32_t* targets, float* loss);

/* As nc_forward_loss but writes the loss to DEVICE memory d_loss (one
 * float) and does not synchronise. */
nc_status nc_forward_loss_async(nc_ctx* ctx, const void* params, const int32_t* tokens,
                                const int32_t* targets, float* d_loss);

/* Backward pass of the last forward: writes the gradient of the mean loss
 * w.r.t. every parameter as fp32 into grads (device, nc_param_count()
 * floats, same layout as params; overwritten, not accumulated). Rows of
 * wte that no token uses get exactly 0. NC_ERR_STATE without a preceding
 * successful forward. Asynchronous. */
nc_status nc_backward(nc_ctx* ctx, float* grads);

/* Gradient accumulation over micro-batches (the pages' training loop sums
 * the gradients of several micro-batches before one optimizer step): as
 * nc_backward, but ADDS scale * d(loss)/d(params) to grads instead of
 * overwriting them. The loss of each micro-batch is its own mean over its
 * unmasked targets, so with scale = 1/n the sum over n calls is the gradient
 * of the mean of the n micro-batch losses (for micro-batches with equal
 * unmasked counts, the gradient of the whole batch's mean loss). grads must
 * hold finite values (zero them before the first micro-batch). NC_ERR_ARG
 * for a non-finite scale, NC_ERR_STATE without a preceding successful
 * forward. Asynchronous. */
nc_status nc_backward_accumulate(nc_ctx* ctx, float* grads, float scale);

/* Forward + loss from packed uint16 token ids, the shard format of the
 * pages' data loader (ids of a 65,536-entry vocabulary fit 16 bits): packed
 * is a DEVICE array [batch, seq_len + 1] row-major; row b's ids 0..T-1 are
 * the inputs and its ids 1..T the next-token targets (no masked targets).
 * The ids are widened into the context's own token/target buffers, which
 * the following backward uses; ids >= vocab report NC_ERR_DEVICE as in
 * nc_forward_loss. The loss goes to DEVICE memory d_loss; asynchronous. */
nc_status nc_forward_loss_u16(nc_ctx* ctx, const void* params, const uint16_t* packed, float* d_loss);

/* One training step from HOST packed uint16 rows [batch, seq_len + 1]
 * (ideally pinned; batch*(seq_len+1)*2 bytes are copied to the device):
 * forward, loss and backward into grads (device, overwritten), the loss to
 * *h_loss. Synchronises the stream. */
nc_status nc_train_step_host_u16(nc_ctx* ctx, const void* params, const uint16_t* h_packed, float* grads,
                                 float* h_loss);

/* One training step from HOST token buffers: copies tokens and targets
 * (host int32 [batch, seq_len], ideally pinned) to the device, runs the
 * forward and backward on device-resident params/grads, and copies the loss
 * back to *h_loss. Synchronises the stream. */
nc_status nc_train_step_host(nc_ctx* ctx, const void* params, const int32_t* h_tokens,
                             const int32_t* h_targets, float* grads, float* h_loss);

/* Per-position results of the last forward, copied device-to-device:
 * d_lse, d_nll: fp32 [batch*seq_len]; d_argmax: int32 [batch*seq_len]
 * (lowest vocabulary index among ties); d_nll is 0 at masked positions.
 * Any pointer may be NULL. */
nc_status nc_get_token_outputs(nc_ctx* ctx, float* d_lse, float* d_nll, int32_t* d_argmax);

/* Greedy next-token prediction of the last forward (nanochat explainer,
 * "Pretraining": the model predicts token N+1 from tokens 1..N): d_argmax
 * (device int32 [batch*seq_len]) receives, per position, the vocabulary index
 * of the largest logit, the lowest index among ties. Copied device to device
 * on the context's stream (asynchronous). NC_ERR_ARG for a NULL d_argmax,
 * NC_ERR_STATE without a preceding successful forward. nc_get_token_outputs
 * returns the same ids together with lse and nll. */
nc_status nc_get_argmax(nc_ctx* ctx, int32_t* d_argmax);

/* Final hidden state of the last forward (the RMS-normalised input of
 * lm_head), copied device-to-device into d_hf: elem [batch*seq_len, d_model]
 * (bf16 in NC_BF16, fp32 in NC_FP32_DEBUG). */
nc_status nc_get_hidden(nc_ctx* ctx, void* d_hf);

/* Synchronise the stream and report a pending device-side failure. */
nc_status nc_sync(nc_ctx* ctx);

/* ---- measurement ----
 * Kernel families for nc_profile_read. */
enum {
  NC_FAM_GEMM = 0,      /* tensor-core (or fp32 debug) GEMMs; work = 2*M*N*K FLOPs */
  NC_FAM_ATTN_FWD = 1,  /* causal attention forward; work = 2*128*T*(T+1)*B*H FLOPs */
  NC_FAM_ATTN_BWD = 2,  /* attention backward; work = 2x the forward's FLOPs */
  NC_FAM_ROWS = 3,      /* norms, embedding, QK-norm/RoPE, CE reductions; work = bytes */
  NC_FAM_OPT_NS = 4,    /* optimizer: Newton-Schulz GEMMs of Muon; work = FLOPs */
  NC_FAM_OPT_ELEM = 5,  /* optimizer: norm, AdamW and Muon element passes; work = bytes */
  NC_FAM_DEC_GEMM = 6,  /* generation: weight-streaming products; work = weight bytes */
  NC_FAM_DEC_ATTN = 7,  /* generation: attention over the KV cache; work = cache bytes read */
  NC_FAM_DEC_ROWS = 8,  /* generation: norms, embedding, QK-norm/RoPE, head reductions; bytes */
  NC_FAM_COUNT = 9
};

/* Number of kernels the context has launched since nc_create. */
unsigned long long nc_launch_count(const nc_ctx* ctx);

/* Turn per-launch CUDA-event timing on (1) or off (0) and clear the record.
 * With it on, every launch is bracketed by events on the context's stream. */
nc_status nc_profile_enable(nc_ctx* ctx, int enable);

/* Synchronise and sum, over the launches recorded since the last reset, the
 * device time (ms), the number of launches and their algorithmic work. */
nc_status nc_profile_read(nc_ctx* ctx, int family, double* ms, long long* launches, double* work);

/* Synchronise and clear the recorded launches (profiling stays as set). */
nc_status nc_profile_reset(nc_ctx* ctx);

/* Test hook for the failure path: set the time limit (ns) of every pipeline
 * wait (TMA stage, accumulator and softmax hand-offs) of the tensor-core
 * kernels launched afterwards on the current device, for every context; 0
 * restores the default of 2 s. Below 1000 ns a wait gives up at its first
 * unsuccessful poll, so a launch reports NC_ERR_TIMEOUT at the next
 * synchronising call (its kernels unwind: the waits for the copies and
 * products already in flight keep the default limit, and TMEM is freed).
 * Only the attention kernels and GEMMs of at most 128 rows may run under a
 * short limit: a GEMM of more rows runs in CTA pairs, whose unwinding waits
 * only for the copies of the phases the even CTA of the pair armed.
 * Synchronises the device. */
nc_status nc_set_pipeline_wait_limit(unsigned long long ns);

/* Message for the calling thread's last failing call ("" if none). */
const char* nc_last_error(const nc_ctx* ctx);

/* Free the context and what the library allocated. NULL is allowed. */
void nc_destroy(nc_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* NC_H */
