/*
 * nc_optim.h -- the optimizer step that completes a nanochat pretraining
 * step: global gradient clipping, AdamW on the embedding and unembedding,
 * Muon on every 2-D block matrix, and the learning-rate schedule.
 *
 * The nanochat explainer ("The Full Pipeline" / "Pretraining") names Muon for
 * the matrix (2-D) weights plus AdamW for the embedding and unembedding, a
 * cosine learning-rate schedule with warmup, gradient clipping at 1.0 and
 * weight decay 0.1; the topaiproduct article ("What the Community Is Saying")
 * names Muon as Bernstein's optimizer in Keller Jordan's implementation. The
 * pages give no further constants, so this library takes:
 *
 *   clip     every gradient times k = min(1, max_norm / (||g||_2 + 1e-6)),
 *            ||g||_2 over all parameters (summed in a fixed order: deterministic)
 *   AdamW    m <- b1 m + (1-b1) g ; v <- b2 v + (1-b2) g^2 ;
 *            p <- p (1 - lr wd) - lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)
 *            (defaults b1 0.9, b2 0.999, eps 1e-8)
 *   Muon     buf <- mu buf + g ; u = g + mu buf (Nesterov, mu 0.95);
 *            X = u / (||u||_F + 1e-7), then ns_steps (5) quintic Newton-Schulz
 *            steps X <- a X + (b A + c A A) X, A = X X^T, (a, b, c) =
 *            (3.4445, -4.7750, 2.0315), on the wide orientation of the matrix;
 *            p <- p (1 - lr wd) - lr sqrt(max(1, rows/cols)) X
 *
 * Each w_qkv, w_o, w_fc and w_proj of each layer is one Muon matrix as stored.
 * In NC_BF16 the Newton-Schulz products run on the tensor cores in bf16 with
 * fp32 accumulation (every iterate rounded to bf16); in NC_FP32_DEBUG in fp32.
 * The optimizer keeps fp32 master weights in its state; after a step the
 * parameter buffer holds their image in the element type (bf16 rounded to
 * nearest even, or fp32).
 *
 * Memory: the state is one caller-owned device buffer of
 * nc_optim_state_bytes() bytes, laid out as fp32 master [P] | AdamW m [2 V d]
 * | AdamW v [2 V d] | Muon momentum [12 L d^2] (AdamW moments for wte then
 * lm_head; momentum in the flat order of the block matrices). The step uses
 * the context's workspace as scratch, so it ends the saved forward: call
 * nc_backward before nc_optim_step, never after. Calls are asynchronous on the
 * context's stream and return nc_status; nothing is allocated.
 */
#ifndef NC_OPTIM_H
#define NC_OPTIM_H

#include "nc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of optimizer state for the context's model (0 before nc_configure). */
size_t nc_optim_state_bytes(const nc_ctx* ctx);

/* Start a run: master <- params (elem -> fp32), moments and momentum <- 0.
 * params: device, elem, flat layout (nc.h); state: device, 16-byte aligned,
 * nc_optim_state_bytes() bytes. NC_ERR_ARG on null or misaligned pointers. */
nc_status nc_optim_init(nc_ctx* ctx, const void* params, void* state);

/* Hyper-parameters that stay fixed over a run. NC_ERR_ARG unless
 * 0 <= beta1, beta2, momentum < 1, eps > 0 and 1 <= ns_steps <= 32. */
nc_status nc_optim_set_hparams(nc_ctx* ctx, float beta1, float beta2, float eps, float momentum, int ns_steps);

/* One optimizer step at 1-based step number t (AdamW's bias correction):
 * reads grads (device fp32, flat layout, as nc_backward wrote them), updates
 * state and writes the new params (device, elem). lr_adamw and lr_muon are
 * this step's learning rates (see nc_lr_at); weight_decay applies to both
 * groups; max_grad_norm is the clipping threshold. stats (device float[2],
 * may be NULL) receives the pre-clip gradient norm and the clip factor.
 * grads is not modified. NC_ERR_STATE without a workspace; NC_ERR_ARG on
 * t < 1, a negative rate, decay or threshold, or null / misaligned pointers. */
nc_status nc_optim_step(nc_ctx* ctx, void* params, const float* grads, void* state, int t, float lr_adamw,
                        float lr_muon, float weight_decay, float max_grad_norm, float* stats);

/* Learning rate at 0-based step `step`: peak * (step + 1) / warmup while
 * step < warmup, then a half cosine from peak down to final_frac * peak at
 * step `total` (held there after). Host-only, pure. */
double nc_lr_at(long long step, long long warmup, long long total, double peak, double final_frac);

#ifdef __cplusplus
}
#endif

#endif /* NC_OPTIM_H */
