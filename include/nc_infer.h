/*
 * nc_infer.h -- generation with a KV cache: prefill of a prompt, then one
 * token per decode step (nanochat explainer, "Inference & KV Cache": the
 * prefill processes the whole prompt in parallel and fills the cache with
 * the keys and values of every layer and position; each decode step then
 * computes attention of the new token against the cached keys and values).
 *
 * The context's batch B and seq_len T fix the shapes: a prompt is B
 * sequences of exactly T tokens, and each decode step takes one new token
 * per sequence. Keys are cached after QK-norm and RoPE (as attention uses
 * them); the next token is the argmax of the position's logits (lowest
 * index on ties), i.e. greedy decoding.
 *
 * KV cache: one caller-owned device buffer of nc_kv_cache_bytes(ctx,
 * max_len) bytes, 256-byte aligned, laid out as, per layer, K then V, each
 * elem [B][H][max_len][128] (elem = bf16 in NC_BF16, fp32 in
 * NC_FP32_DEBUG), followed by the RoPE table for max_len positions and the
 * scratch of one decode step. nc_prefill fills positions 0..T-1 and the
 * table; nc_decode_step at position pos writes position pos and reads
 * 0..pos, so positions before pos must hold the cache of earlier tokens of
 * the same sequences. The context's workspace is scratch for both calls
 * (they end the saved forward of the training step). Calls are
 * asynchronous on the context's stream except where stated; nothing is
 * allocated on the device.
 */
#ifndef NC_INFER_H
#define NC_INFER_H

#include "nc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of KV cache for the configured batch and max_len positions (0 on a
 * bad context or max_len < 1). */
size_t nc_kv_cache_bytes(const nc_ctx* ctx, int max_len);

/* Prefill: run tokens (device int32 [B, T], ids in [0, vocab)) through the
 * model, write positions 0..T-1 of the cache and the RoPE table, and the
 * greedy next token of every sequence into next_tokens (device int32 [B]).
 * last_logits (device fp32 [B, vocab], may be NULL) receives the logits of
 * position T-1. Requires T <= max_len <= 65536. The first call with a given
 * max_len builds the RoPE table on the host and keeps it on the device (one
 * stream synchronisation); later calls copy it into the cache on the device
 * and do not synchronise. NC_ERR_DEVICE for an id out of range. */
nc_status nc_prefill(nc_ctx* ctx, const void* params, const int32_t* tokens, void* kv_cache, int max_len,
                     int32_t* next_tokens, float* last_logits);

/* Decode step at position pos (0 <= pos < max_len): tokens (device int32
 * [B]) are the tokens at position pos; their keys/values are appended to
 * the cache and next_tokens (device int32 [B]) receives the greedy token
 * for position pos + 1; logits (device fp32 [B, vocab], may be NULL) its
 * logits. */
nc_status nc_decode_step(nc_ctx* ctx, const void* params, const int32_t* tokens, int pos, void* kv_cache,
                         int max_len, int32_t* next_tokens, float* logits);

/* As nc_decode_step, with the position read from device memory (*d_pos, an
 * int32) and advanced by one after the step, so the call's launches do not
 * depend on the position: a caller can capture one step in a CUDA graph and
 * replay it for every position (the attention grid covers max_len; chunks
 * past the position exit at once). A position outside [0, max_len) makes
 * the step write nothing to the cache and report NC_ERR_DEVICE at the next
 * synchronising call. The first call must not be made during capture (it
 * sets up kernel attributes). */
nc_status nc_decode_step_dev(nc_ctx* ctx, const void* params, const int32_t* tokens, int32_t* d_pos, void* kv_cache,
                             int max_len, int32_t* next_tokens, float* logits);

#ifdef __cplusplus
}
#endif

#endif /* NC_INFER_H */
