/*
 * nc_ops.h -- op-level entry points of the nanochat step (one call per step
 * of the path), for parity tests and for callers that assemble their own
 * step. All take a context that nc_configure has set up (its precision,
 * stream, batch, shapes and RoPE table are used) and, where stated, its
 * workspace for scratch. Element type ("elem") is bf16 for NC_BF16 and fp32
 * for NC_FP32_DEBUG. Pointers are device pointers owned by the caller.
 * Every call is asynchronous on the context's stream and returns nc_status
 * (NC_ERR_STATE when the context is not configured or has no workspace).
 * A call here invalidates the context's saved forward (nc_backward then
 * returns NC_ERR_STATE until the next nc_forward_loss).
 */
#ifndef NC_OPS_H
#define NC_OPS_H

#include "nc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogue codes for nc_op_gemm. */
enum {
  NC_EPI_STORE = 0,      /* C (elem) = alpha * acc                                  */
  NC_EPI_STORE_F32 = 1,  /* C (fp32) = alpha * acc + beta * C                       */
  NC_EPI_RELU2 = 2,      /* C (elem) = u = alpha * acc ; C2 (elem) = max(u, 0)^2    */
  NC_EPI_RELU2_BWD = 3,  /* C (elem) = alpha * acc * 2 * sqrt(a), a = max(u, 0)^2
                            read from C2 (relu(u) recovered from the stored a)      */
  NC_EPI_CE_BWD = 4,     /* C (elem) = exp(alpha*acc - row_f[m]) - (n == row_i[m])  */
  NC_EPI_QKNORM_ROPE = 6, /* NC_BF16 only; the QKV projection with QK-norm + RoPE:
                            M = batch*seq_len, N = 3*d_model; C (elem [M, 3d]) gets
                            q, k heads RMS-normalised and rotated (position m % seq_len)
                            and v heads as computed; C2 = fp32 rqk [M, 2H]          */
  NC_EPI_AXPBY = 7,      /* C (elem) = alpha * acc + beta * C2 (elem, ldc2)          */
  NC_EPI_RELU2A = 8      /* C (elem) = max(alpha * acc, 0)^2 (a alone, no u)         */
};

/* Linear-layer contraction of the step (the QKV, out-projection, MLP and
 * lm_head matmuls and their backward products):
 *   acc[m,n] = sum_k A(m,k) B(n,k), m < M, n < N, k < K,
 *   A(m,k) = a_kmajor ? A[m*lda + k] : A[k*lda + m]   (elem)
 *   B(n,k) = b_kmajor ? B[n*ldb + k] : B[k*ldb + n]   (elem)
 * then the epilogue above writes C[m*ldc + n] (and C2[m*ldc2 + n]).
 * With a workspace set, fp32-output products with many k-blocks and few
 * output tiles (the weight gradients) are split along K into partial sums
 * in the workspace and reduced in a fixed order (deterministic).
 * The ReLU^2 epilogues follow the nanochat explainer's "ReLU^2 Sparsity";
 * the CE_BWD epilogue forms softmax(logits) - onehot(target) of
 * "Pretraining"'s cross-entropy. In NC_BF16 the operands' leading
 * dimensions must be multiples of 8 elements and the base addresses 16-byte
 * aligned (tensor-core path); NC_ERR_UNSUPPORTED otherwise. */
nc_status nc_op_gemm(nc_ctx* ctx, int M, int N, int K, const void* A, long long lda, int a_kmajor,
                     const void* B, long long ldb, int b_kmajor, int epi, float alpha, float beta,
                     void* C, long long ldc, void* C2, long long ldc2, const float* row_f,
                     const int32_t* row_i);

/* A batch of independent contractions of the same shape whose operands are
 * stacked along their outer (row) dimension: problem i uses
 * A + i*a_brows*lda, B + i*b_brows*ldb, C + i*c_brows*ldc and
 * C2 + i*c_brows*ldc2, each as in nc_op_gemm. This is the shape of Muon's
 * Newton-Schulz products over the same-shaped matrices of every layer
 * (nc_optim.h); epi is NC_EPI_STORE or NC_EPI_AXPBY. In NC_BF16, M must be a
 * multiple of 128, a_brows >= (a_kmajor ? M : K), b_brows >= (b_kmajor ? N : K),
 * c_brows >= M, and an operand stacked along k (not k-major) needs a multiple
 * of 64 rows per problem; NC_ERR_UNSUPPORTED otherwise. */
nc_status nc_op_gemm_batched(nc_ctx* ctx, int batch, int M, int N, int K, const void* A, long long lda,
                             int a_kmajor, long long a_brows, const void* B, long long ldb, int b_kmajor,
                             long long b_brows, int epi, float alpha, float beta, void* C, long long ldc,
                             void* C2, long long ldc2, long long c_brows);

/* Fused lm_head + softmax cross-entropy forward over M = batch*seq_len rows
 * (nanochat explainer, "Pretraining": cross-entropy between the predicted
 * logits and the next tokens). hf: elem [M, d]; w_lm: elem [V, d];
 * tgt: int32 [M] (-1 masks a row: nll 0 there). Outputs lse, nll: fp32 [M];
 * argmax: int32 [M] (lowest index among ties). The full [M, V] logits are
 * never stored; scratch comes from the context's workspace. */
nc_status nc_op_lmhead_ce_fwd(nc_ctx* ctx, const void* hf, const void* w_lm, const int32_t* tgt,
                              float* lse, float* nll, int32_t* argmax);

/* Backward of the mean cross-entropy w.r.t. hf and w_lm, recomputing the
 * logits: g = (softmax - onehot(tgt)) / n on the n rows whose target is not
 * -1 and 0 on the masked rows; dhf = g w_lm (fp32 [M, d]); dw_lm = g^T hf
 * (fp32 [V, d], overwritten). lse from nc_op_lmhead_ce_fwd. */
nc_status nc_op_lmhead_ce_bwd(nc_ctx* ctx, const void* hf, const void* w_lm, const int32_t* tgt,
                              const float* lse, float* dhf, float* dw_lm);

/* Causal multi-head attention forward (nanochat explainer, "Multi-Head
 * Attention (what nanochat uses)"), scale 1/sqrt(128).
 * qkv: elem [B*T, 3d], columns q_hat | k_hat | v, head h at h*128 (q_hat,
 * k_hat already QK-normed and rotated). o: elem [B*T, d]; lse: fp32 [B, H, T]. */
nc_status nc_op_attention_fwd(nc_ctx* ctx, const void* qkv, void* o, float* lse);

/* Attention backward. dout: elem [B*T, d]; lse from the forward.
 * dqk: fp32 [2, B*T, d] receives the dq_hat plane then the dk_hat plane;
 * dqkv: elem [B*T, 3d] receives dv in its v columns (q,k columns untouched).
 * Scratch (the softmax-backward row sums) from the workspace. NC_BF16 needs
 * seq_len % 128 == 0 (tensor-core kernels). */
nc_status nc_op_attention_bwd(nc_ctx* ctx, const void* qkv, const void* o, const void* dout,
                              const float* lse, float* dqk, void* dqkv);

/* QK-norm + RoPE in place on the q and k columns of qkv (elem [B*T, 3d]):
 * per head, q <- rope(q / sqrt(mean(q^2) + 1e-6)), half-split pairs (j, j+64),
 * angle pos * 10000^(-j/64) (nanochat explainer, "RoPE Intuition").
 * rqk: fp32 [B*T, 2H], the per-head reciprocal RMS of q heads then k heads. */
nc_status nc_op_qk_norm_rope_fwd(nc_ctx* ctx, void* qkv, float* rqk);

/* Parameter-free RMSNorm of the fp32 residual stream x [B*T, d]:
 * y (elem) = x * r, r (fp32 [B*T]) = 1/sqrt(mean(x^2) + 1e-6). */
nc_status nc_op_rmsnorm_fwd(nc_ctx* ctx, const float* x, void* y, float* r);

/* Backward of the parameter-free RMSNorm y = z * r (nanochat explainer,
 * "Architecture Choices": RMSNorm; the gradient follows from y = z / rms(z)):
 * dz = r * (dy - y * mean(dy * y)) per row of M = batch*seq_len rows of
 * d_model. dy, y: elem [M, d]; r: fp32 [M] from the forward. dx: fp32 [M, d]
 * receives dz, or dx + dz when accumulate is non-zero (the residual stream's
 * gradient adds the branch's); dx_e (elem [M, d], may be NULL) gets a copy of
 * the new dx in the element type. */
nc_status nc_op_rmsnorm_bwd(nc_ctx* ctx, const void* dy, const void* y, const float* r, float* dx, void* dx_e,
                            int accumulate);

/* Token embedding lookup (nanochat explainer, "Architecture Choices": untied
 * token embedding): x[m, :] = wte[tok[m], :] as fp32 (the residual stream),
 * no scaling or normalisation. tok: int32 [M] in [0, vocab); wte: elem [V, d];
 * x: fp32 [M, d]. An id out of range writes a zero row and sets the status
 * word (the next nc_sync returns NC_ERR_DEVICE). */
nc_status nc_op_embed_fwd(nc_ctx* ctx, const int32_t* tok, const void* wte, float* x);

/* Backward of the lookup: dwte (fp32 [V, d], overwritten) gets, in row id,
 * the sum of dx[m, :] (fp32 [M, d]) over the positions m with tok[m] = id;
 * the rows of ids that no position holds are exactly 0. The sums are formed
 * by atomic adds, so their order (and the last bits) may vary between runs. */
nc_status nc_op_embed_bwd(nc_ctx* ctx, const int32_t* tok, const float* dx, float* dwte);

/* Backward of the QK-norm + RoPE of nc_op_qk_norm_rope_fwd, for the q and the
 * k heads: with q_hat = R_pos q / rms(q) (nanochat explainer, "RoPE
 * Intuition"), dq = r * (dq_n - q_n * mean(dq_n * q_n)) where dq_n = R_pos^T
 * dq_hat and q_n = R_pos^T q_hat. dqk: fp32 [2, M, d], the dq_hat plane then
 * the dk_hat plane (as nc_op_attention_bwd writes them); qkv: elem [M, 3d],
 * the forward's output (q_hat, k_hat, v); rqk: fp32 [M, 2H] from the forward.
 * dq and dk go to the q and k columns of dqkv (elem [M, 3d]); its v columns
 * are left as they are. */
nc_status nc_op_qk_norm_rope_bwd(nc_ctx* ctx, const float* dqk, const void* qkv, const float* rqk, void* dqkv);

/* Fused lm_head + cross-entropy forward that allocates no device memory.
 * The nanochat pages have no counterpart of this call; it exists for callers
 * that must not call cudaMalloc where they need the loss (code inside another
 * framework's memory pool or allocation budget). It computes what
 * nc_op_lmhead_ce_fwd computes, in bf16 only, with no context:
 * hf: bf16 [M, d]; w_lm: bf16 [V, d] (both 16-byte aligned); tgt: int32 [M];
 * lse, nll: fp32 [M]; argmax: int32 [M] (lowest index among ties);
 * d_status: optional device int32, set to 0, or to 1 if a target id is out of
 * range, or to 2 if a pipeline wait timed out. With d_status NULL neither
 * failure is reported anywhere: the call still returns NC_OK, and a row whose
 * target id is out of range gets nll = lse (its target logit reads as 0), so
 * pass d_status unless the targets are known to be valid; cuda_stream: a cudaStream_t
 * (NULL = legacy default stream). d and V must be multiples of 8.
 * Scratch is a 16 MiB array in the library's static device memory, held by
 * every GPU that loads the library until the process exits; a call needs
 * M * (12 * ceil(V/128) + 4) bytes of it (at V = 65536: at most 2728 rows per
 * call), larger requests return NC_ERR_UNSUPPORTED with a message. The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress)
 * and caches it, so make that first call before any stream capture. Calls
 * share the one array: calls that overlap on the GPU (on different streams,
 * or on different host threads) race and give wrong results. Asynchronous;
 * nothing is allocated and no allocating library routine is called. */
nc_status nc_lmhead_ce_fwd_static(const void* hf, const void* w_lm, const int32_t* tgt, int M, int d, int V,
                                  float* lse, float* nll, int32_t* argmax, int32_t* d_status,
                                  void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* NC_OPS_H */
