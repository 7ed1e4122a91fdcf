// Context, workspace layout and launch sequence of the nanochat pretraining
// step (forward, mean next-token cross-entropy, analytic backward) behind the
// C ABI of include/nc.h and include/nc_ops.h.
//
// The step follows the nanochat explainer: pre-norm decoder blocks with
// parameter-free RMSNorm, QK-norm + RoPE attention, ReLU^2 MLP
// ("Architecture Choices", "RoPE Intuition", "ReLU^2 Sparsity"), untied
// embedding / lm_head, and the cross-entropy of "Pretraining".
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <string>
#include <vector>

#include "../../include/nc.h"
#include "../../include/nc_ops.h"
#include "../../include/nc_optim.h"
#include "../../include/nc_infer.h"
#include "ops.cuh"

using namespace nc;

namespace {

thread_local std::string g_err;

nc_status fail(nc_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
nc_status fail(nc_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

#define CK(expr)                                                                              \
  do {                                                                                        \
    cudaError_t e_ = (expr);                                                                  \
    if (e_ != cudaSuccess)                                                                    \
      return fail(NC_ERR_CUDA, "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), __FILE__, \
                  __LINE__);                                                                  \
  } while (0)

#define CKS(expr)                          \
  do {                                     \
    nc_status s_ = (expr);                 \
    if (s_ != NC_OK) return s_;            \
  } while (0)

constexpr size_t kAlign = 1024;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace

namespace nc {
// Record a message for nc_last_error from other translation units.
nc_status set_last_error(nc_status st, const char* msg) {
  g_err = msg;
  return st;
}
}  // namespace nc

struct nc_ctx {
  // model shape
  int L = 0, d = 0, H = 0, T = 0, V = 0, F = 0;
  // configuration
  int B = 0, M = 0, prec = -1, esz = 0;
  cudaStream_t stream = nullptr;
  int device = -1;
  int sms = 148;            // SM count of the configured device
  bool use_tc = false;      // tensor-core GEMMs for the bf16 mode
  float* rope_cos = nullptr;   // [T][64]
  float* rope_sin = nullptr;
  float* rope_cos4 = nullptr;  // the same angles, angle-major [16][T][4] (GEMM and attention epilogues)
  float* rope_sin4 = nullptr;
  float* dec_rope = nullptr;   // decode RoPE table for dec_rope_len positions: cos [len][64] then sin
  int dec_rope_len = 0;
  int* status = nullptr;    // device status word
  int* tile_done = nullptr;  // kGemmTileCap split-K tile counters of the GEMM (0 between launches)
  // workspace
  char* ws = nullptr;
  size_t ws_bytes = 0, ws_need = 0;
  int ce_rows = 0;          // rows per lm_head / cross-entropy chunk
  int ce_tiles = 0;         // 128-wide vocabulary tiles (tensor-core CE partials)
  size_t partial_bytes = 0; // split-K partial sums of the weight-gradient GEMMs
  struct Off {
    size_t xn1, r1, qkv, rqk, o, lse_att, xn2, r2, a;  // per-layer stash (stride below)
    size_t layer_stride;
    size_t x, hf, rf, lse, nll, amax, loss, pmax, psum, parg, ptgt, chunk;
    size_t dx, dxe, dy, du, dout, dqkv, dqk, drow, tok, tgt, partial, inv_count, grad_scale, packed;
  } off{};
  // optimizer scratch: overlays the step's workspace from offset 0 (the
  // stash is dead once the backward has run)
  struct OptOff {
    size_t stats, part_norm, part_muon, inv_norm, x_all, pong, gram, poly;
  } opt{};
  // decode scratch (one token per sequence), after the step's layout
  struct DecOff {
    size_t x, r, xn, qkv, o, u, a, hf, lse, nll, tgt, cep;
  } dec{};
  // optimizer hyper-parameters fixed per context (nc_optim_set_hparams)
  float opt_b1 = 0.9f, opt_b2 = 0.999f, opt_eps = 1e-8f, opt_mu = 0.95f;
  int opt_ns = 5;
  int gemm_fam = NC_FAM_GEMM;  // family the GEMM launches are timed under
  // launch accounting and optional per-family event timing
  unsigned long long launches = 0;
  bool prof = false;
  struct Rec { cudaEvent_t a, b; int fam; double work; };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  size_t pool_next = 0;
  // last forward
  const void* params = nullptr;
  const int* tok = nullptr;
  const int* tgt = nullptr;
  bool have_fwd = false;
};

namespace {

template <typename P>
P* wsp(nc_ctx* c, size_t off) { return reinterpret_cast<P*>(c->ws + off); }

// ------------------------------------------------------------------ accounting

nc_status next_event(nc_ctx* c, cudaEvent_t* ev) {
  if (c->pool_next == c->pool.size()) {
    cudaEvent_t e;
    CK(cudaEventCreate(&e));
    c->pool.push_back(e);
  }
  *ev = c->pool[c->pool_next++];
  return NC_OK;
}

nc_status prof_begin(nc_ctx* c, cudaEvent_t* a) {
  if (!c->prof) return NC_OK;
  CKS(next_event(c, a));
  CK(cudaEventRecord(*a, c->stream));
  return NC_OK;
}

nc_status prof_end(nc_ctx* c, cudaEvent_t a, int fam, double work, int n) {
  c->launches += (unsigned long long)n;
  if (!c->prof) return NC_OK;
  cudaEvent_t b;
  CKS(next_event(c, &b));
  CK(cudaEventRecord(b, c->stream));
  c->recs.push_back({a, b, fam, work});
  return NC_OK;
}

// Launch `expr` (a launcher returning cudaError_t that starts `n` kernels),
// counting it and, when profiling, timing it under family `fam` with
// algorithmic work `work` (FLOPs or bytes).
#define KL(fam, work, n, expr)                                                                  \
  do {                                                                                          \
    cudaEvent_t ev_a_ = nullptr;                                                                \
    CKS(prof_begin(c, &ev_a_));                                                                 \
    cudaError_t e_ = (expr);                                                                    \
    if (e_ != cudaSuccess) return fail(NC_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));  \
    CKS(prof_end(c, ev_a_, (fam), (double)(work), (n)));                                        \
  } while (0)

size_t param_offset(const nc_ctx* c, int index, int* rows, int* cols) {
  size_t d = c->d, V = c->V, F = c->F;
  size_t per_layer = 3 * d * d + d * d + F * d + d * F;
  if (index == 0) { *rows = c->V; *cols = c->d; return 0; }
  if (index == 1 + 4 * c->L) { *rows = c->V; *cols = c->d; return V * d + (size_t)c->L * per_layer; }
  int l = (index - 1) / 4, k = (index - 1) % 4;
  size_t base = V * d + (size_t)l * per_layer;
  switch (k) {
    case 0: *rows = 3 * c->d; *cols = c->d; return base;
    case 1: *rows = c->d; *cols = c->d; return base + 3 * d * d;
    case 2: *rows = c->F; *cols = c->d; return base + 4 * d * d;
    default: *rows = c->d; *cols = c->F; return base + 4 * d * d + F * d;
  }
}

void plan_workspace(nc_ctx* c) {
  size_t M = c->M, d = c->d, F = c->F, H = c->H, V = c->V, e = c->esz;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += align_up(bytes); return r; };
  auto& f = c->off;
  f.xn1 = take(M * d * e);
  f.r1 = take(M * 4);
  f.qkv = take(M * 3 * d * e);
  f.rqk = take(M * 2 * H * 4);
  f.o = take(M * d * e);
  f.lse_att = take(M * H * 4);
  f.xn2 = take(M * d * e);
  f.r2 = take(M * 4);
  f.a = take(M * F * e);
  f.layer_stride = o;
  o = f.layer_stride * c->L;
  f.x = take(M * d * 4);
  f.hf = take(M * d * e);
  f.rf = take(M * 4);
  f.lse = take(M * 4);
  f.nll = take(M * 4);
  f.amax = take(M * 4);
  f.loss = take(4);
  c->ce_tiles = (int)((V + 127) / 128);
  f.pmax = take((size_t)c->ce_tiles * M * 4);
  f.psum = take((size_t)c->ce_tiles * M * 4);
  f.parg = take((size_t)c->ce_tiles * M * 4);
  f.ptgt = take(M * 4);
  // rows per lm_head / cross-entropy backward chunk: in bf16 the whole batch up to 32,768 rows (g is 2 B per
  // logit, 4.3 GB at 32,768 x 65,536), so the input- and weight-gradient GEMMs each run once over every row
  // instead of eight times on a 4096-row slice that fills 1.08 waves of the SMs; the fp32 debug mode
  // materialises logits, 4096 rows at a time
  c->ce_rows = (int)(c->prec == NC_BF16 ? (M < 32768 ? M : 32768) : (M < 4096 ? M : 4096));
  f.chunk = take((size_t)c->ce_rows * V * e);  // fp32 logits (debug) or bf16 g
  f.dx = take(M * d * 4);
  f.dxe = take(M * d * e);
  f.dy = take(M * d * 4);
  f.du = take(M * F * e);
  f.dout = take(M * d * e);
  f.dqkv = take(M * 3 * d * e);
  f.dqk = take(M * 2 * d * 4);
  f.drow = take(2 * M * H * 4);  // D rows, then the negated base-2 lse rows of the bf16 attention backward
  f.tok = take(M * 4);
  f.tgt = take(M * 4);
  // up to 8 k-splits of the largest weight gradient (4d x d), at least 64 MiB
  c->partial_bytes = 8 * 4 * d * d * 4;
  if (c->partial_bytes < (size_t(64) << 20)) c->partial_bytes = size_t(64) << 20;
  f.partial = take(c->partial_bytes);
  f.inv_count = take(4);  // 1 / number of unmasked targets of the last forward
  f.grad_scale = take(4);  // inv_count times an accumulating backward's scale
  f.packed = take((size_t)c->B * (c->T + 1) * 2);  // host uint16 token rows staged by nc_train_step_host_u16
  // decode scratch: B rows of the step's activations
  {
    const size_t Bn = c->B;
    auto& q = c->dec;
    q.x = take(Bn * d * 4);
    q.r = take(Bn * 4);
    q.xn = take(Bn * d * e);
    q.qkv = take(Bn * 3 * d * 4);
    q.o = take(Bn * d * e);
    q.u = take(Bn * F * 4);  // fp32 up-projection when ReLU^2 is not fused into it
    q.a = take(Bn * F * e);
    q.hf = take(Bn * d * e);
    q.lse = take(Bn * 4);
    q.nll = take(Bn * 4);
    q.tgt = take(Bn * 4);
    q.cep = take(Bn * kCeMaxSegments * 16);  // cross-entropy row segments of the greedy head
  }
  c->ws_need = o;
  // optimizer scratch, from offset 0
  o = 0;
  const size_t d2 = d * d, L = c->L, nb = 12 * L * d2;
  auto& q = c->opt;
  q.stats = take(2 * 4);
  q.part_norm = take(kNormBlocks * 8);
  q.part_muon = take(nb / kMuonChunk * 8);
  q.inv_norm = take(4 * L * 4);
  q.x_all = take(nb * e);          // Newton-Schulz input / iterate, stacked per kind
  q.pong = take(4 * L * d2 * e);   // second iterate buffer (largest kind)
  q.gram = take(L * d2 * e);       // X X^T per matrix
  q.poly = take(L * d2 * e);       // b A + c A A per matrix
  if (o > c->ws_need) c->ws_need = o;
}

nc_status check_ready(nc_ctx* c) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  if (c->prec < 0) return fail(NC_ERR_STATE, "nc_configure has not been called");
  if (!c->ws) return fail(NC_ERR_STATE, "nc_set_workspace has not been called");
  int dev = -1;
  CK(cudaGetDevice(&dev));
  if (dev != c->device) return fail(NC_ERR_STATE, "current device %d differs from the configured %d", dev, c->device);
  return NC_OK;
}

nc_status read_status(nc_ctx* c) {
  int st = 0;
  CK(cudaMemcpyAsync(&st, c->status, sizeof(int), cudaMemcpyDeviceToHost, c->stream));
  CK(cudaStreamSynchronize(c->stream));
  if (st == DEV_OK) return NC_OK;
  CK(cudaMemsetAsync(c->status, 0, sizeof(int), c->stream));
  // a GEMM that gave up may have left split-K tile counters part-way
  if (st == DEV_TIMEOUT && c->tile_done) CK(cudaMemsetAsync(c->tile_done, 0, kGemmTileCap * sizeof(int), c->stream));
  CK(cudaStreamSynchronize(c->stream));
  if (st == DEV_TIMEOUT) return fail(NC_ERR_TIMEOUT, "a device pipeline wait exceeded its iteration limit");
  if (st == DEV_BAD_TOKEN) return fail(NC_ERR_DEVICE, "a token or target id is outside [0, vocab)");
  return fail(NC_ERR_DEVICE, "device status %d", st);
}

// ------------------------------------------------------------------ GEMM dispatch

nc_status gemm(nc_ctx* c, GemmArgs g) {
  g.status = c->status;
  cudaError_t e;
  cudaEvent_t ev_a = nullptr;
  CKS(prof_begin(c, &ev_a));
  if (c->prec == NC_FP32_DEBUG) {
    e = gemm_simt<float>(g, c->stream);
  } else if (c->use_tc) {
    if (g.epi == EPI_STORE_F32 && c->ws) {
      const int sp = gemm_tc_pick_splits(g);
      if (sp > 1 && (size_t)sp * g.M * g.N * 4 <= c->partial_bytes) {
        g.splits = sp;
        g.partial = wsp<float>(c, c->off.partial);
        g.tile_done = c->tile_done;  // in-kernel ordered reduction where it applies
      }
    }
    if (!gemm_tc_supports(g))
      return fail(NC_ERR_UNSUPPORTED, "tensor-core GEMM cannot serve M=%d N=%d K=%d epi=%d", g.M, g.N, g.K, g.epi);
    e = gemm_tc(g, c->stream);
  } else {
    e = gemm_simt<bf16>(g, c->stream);
  }
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "gemm M=%d N=%d K=%d epi=%d: %s", g.M, g.N, g.K, g.epi, cudaGetErrorString(e));
  // a split-K reduction kernel, where one follows, counts as a second launch
  int n = c->use_tc && c->prec != NC_FP32_DEBUG ? gemm_tc_launches(g) : ((g.M > 0 && g.N > 0) ? 1 : 0);
  // decode GEMMs stream their weights: their work is counted in bytes
  const double work = c->gemm_fam == NC_FAM_DEC_GEMM ? (double)g.N * g.K * c->esz
                                                     : 2.0 * g.M * g.N * (double)g.K * g.batch;
  return prof_end(c, ev_a, c->gemm_fam, work, n);
}

GemmArgs mk(int M, int N, int K, const void* A, long long lda, int ak, const void* B, long long ldb,
            int bk, int epi, void* C, long long ldc, float alpha = 1.f, float beta = 0.f) {
  GemmArgs g;
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.a_kmajor = ak;
  g.B = B; g.ldb = ldb; g.b_kmajor = bk;
  g.epi = epi; g.C = C; g.ldc = ldc; g.alpha = alpha; g.beta = beta;
  return g;
}

// Algorithmic FLOPs of one causal attention forward over the configured
// batch: QK^T and PV over the lower triangle, 2*D*T*(T+1) per (b, h).
double attn_fwd_flops(const nc_ctx* c) {
  return 2.0 * kHeadDim * (double)c->T * (c->T + 1) * c->B * c->H;
}

// Causal attention: tcgen05 kernels for bf16, fp32 FMA kernels for the fp32
// debug mode. dqk is the planar fp32 [2, M, d] (dq_hat, dk_hat) scratch.
template <typename T>
cudaError_t attn_fwd(nc_ctx* c, const T* qkv, T* o, float* lse) {
  if constexpr (sizeof(T) == 2)
    return attn_fwd_tc(qkv, o, lse, c->B, c->T, c->H, c->status, c->stream);
  else
    return attn_fwd_simt<T>(qkv, o, lse, c->B, c->T, c->H, c->stream);
}

// With rqk (the step), the tensor-core kernel also finishes the k half of the
// QK-norm + RoPE backward; without it (the op-level call) it leaves dk_hat.
template <typename T>
cudaError_t attn_bwd(nc_ctx* c, const T* qkv, const T* dout, const float* lse, const float* drow, float* dqk,
                     T* dqkv, const float* rqk = nullptr) {
  if constexpr (sizeof(T) == 2)  // the tensor-core kernel reads the negated base-2 lse written after drow
    return attn_bwd_tc(qkv, dout, drow + (size_t)c->M * c->H, drow, dqk, dqk + (size_t)c->M * c->d, dqkv, c->B,
                       c->T, c->H, c->status, c->stream, rqk, rqk ? c->rope_cos4 : nullptr,
                       rqk ? c->rope_sin4 : nullptr);
  else
    return attn_bwd_simt<T>(qkv, dout, lse, drow, dqk, dqkv, c->B, c->T, c->H, c->stream);
}

// ------------------------------------------------------------------ step pieces

template <typename T>
nc_status lmhead_ce_forward(nc_ctx* c, const T* hf, const T* wlm, const int* tgt, int M, float* lse,
                            float* nll, int* amax) {
  int d = c->d, V = c->V;
  if (c->prec == NC_BF16 && c->use_tc) {
    GemmArgs g = mk(M, V, d, hf, d, 1, wlm, d, 1, EPI_CE_FWD, nullptr, 0);
    g.row_i = tgt;
    g.p_max = wsp<float>(c, c->off.pmax);
    g.p_sum = wsp<float>(c, c->off.psum);
    g.p_arg = wsp<int>(c, c->off.parg);
    g.p_tgt = wsp<float>(c, c->off.ptgt);
    CKS(gemm(c, g));
    KL(NC_FAM_ROWS, 12.0 * c->ce_tiles * M + 16.0 * M, 1,
       ce_reduce_partials(g.p_max, g.p_sum, g.p_arg, g.p_tgt, tgt, c->ce_tiles, lse, nll, amax, M, c->stream));
    return NC_OK;
  }
  float* logits = wsp<float>(c, c->off.chunk);
  for (int r0 = 0; r0 < M; r0 += c->ce_rows) {
    int rows = M - r0 < c->ce_rows ? M - r0 : c->ce_rows;
    CKS(gemm(c, mk(rows, V, d, hf + (size_t)r0 * d, d, 1, wlm, d, 1, EPI_STORE_F32, logits, V)));
    KL(NC_FAM_ROWS, 8.0 * rows * V, rows > 0 ? 1 : 0,
       ce_rows_from_logits(logits, tgt + r0, lse + r0, nll + r0, amax + r0, rows, V, c->status, c->stream));
  }
  return NC_OK;
}

// g = softmax - onehot per chunk; dhf = g W_lm / M ; dW_lm = g^T hf / M.
// dhf is written in DT (the element type inside the step, fp32 for the op).
template <typename T, typename DT>
nc_status lmhead_ce_backward(nc_ctx* c, const T* hf, const T* wlm, const int* tgt, const float* lse,
                             int M, const float* d_inv_count, DT* dhf, float* dwlm, bool accumulate = false) {
  int d = c->d, V = c->V;
  T* g = wsp<T>(c, c->off.chunk);
  for (int r0 = 0; r0 < M; r0 += c->ce_rows) {
    int rows = M - r0 < c->ce_rows ? M - r0 : c->ce_rows;
    GemmArgs a = mk(rows, V, d, hf + (size_t)r0 * d, d, 1, wlm, d, 1, EPI_CE_BWD, g, V);
    a.row_f = lse + r0;
    a.row_i = tgt + r0;
    a.dscale = d_inv_count;  // g = (softmax - onehot) / (unmasked rows), 0 on masked rows
    CKS(gemm(c, a));
    CKS(gemm(c, mk(rows, d, V, g, V, 1, wlm, d, 0, sizeof(DT) == 4 ? EPI_STORE_F32 : EPI_STORE,
                   dhf + (size_t)r0 * d, d)));
    CKS(gemm(c, mk(V, d, rows, g, V, 0, hf + (size_t)r0 * d, d, 0, EPI_STORE_F32, dwlm, d, 1.f,
                   r0 == 0 && !accumulate ? 0.f : 1.f)));
  }
  return NC_OK;
}

template <typename T>
nc_status forward_blocks(nc_ctx* c, const T* P, const int* tok) {
  int M = c->M, d = c->d, H = c->H, F = c->F, V = c->V, Tn = c->T;
  cudaStream_t s = c->stream;
  KL(NC_FAM_ROWS, 4.0 * M, 1, check_ids(tok, M, 0, V, c->status, s));
  float* x = wsp<float>(c, c->off.x);
  int rows, cols;
  KL(NC_FAM_ROWS, (double)M * d * (sizeof(T) + 4) + 4.0 * M, 1, embed_fwd<T>(tok, P, x, M, d, V, c->status, s));
  for (int l = 0; l < c->L; ++l) {
    size_t lb = (size_t)l * c->off.layer_stride;
    T* xn1 = wsp<T>(c, lb + c->off.xn1);
    float* r1 = wsp<float>(c, lb + c->off.r1);
    T* qkv = wsp<T>(c, lb + c->off.qkv);
    float* rqk = wsp<float>(c, lb + c->off.rqk);
    T* o = wsp<T>(c, lb + c->off.o);
    float* lse_att = wsp<float>(c, lb + c->off.lse_att);
    T* xn2 = wsp<T>(c, lb + c->off.xn2);
    float* r2 = wsp<float>(c, lb + c->off.r2);
    T* a = wsp<T>(c, lb + c->off.a);
    const T* Wqkv = P + param_offset(c, 1 + 4 * l, &rows, &cols);
    const T* Wo = P + param_offset(c, 2 + 4 * l, &rows, &cols);
    const T* Wfc = P + param_offset(c, 3 + 4 * l, &rows, &cols);
    const T* Wproj = P + param_offset(c, 4 + 4 * l, &rows, &cols);

    KL(NC_FAM_ROWS, (double)M * d * (4 + sizeof(T)) + 4.0 * M, 1, rmsnorm_fwd<T>(x, xn1, r1, M, d, s));
    if (c->use_tc) {
      // QK-norm + RoPE fused into the QKV GEMM epilogue
      GemmArgs gq = mk(M, 3 * d, d, xn1, d, 1, Wqkv, d, 1, EPI_QKNORM_ROPE, qkv, 3 * d);
      gq.rope_cos = c->rope_cos4; gq.rope_sin = c->rope_sin4; gq.rqk = rqk;
      gq.seq_len = Tn; gq.d_model = d;
      CKS(gemm(c, gq));
    } else {
      CKS(gemm(c, mk(M, 3 * d, d, xn1, d, 1, Wqkv, d, 1, EPI_STORE, qkv, 3 * d)));
      KL(NC_FAM_ROWS, 4.0 * M * d * sizeof(T) + 8.0 * M * H, 1, qk_norm_rope_fwd<T>(qkv, rqk, c->rope_cos, c->rope_sin, M, Tn, H, s));
    }
    KL(NC_FAM_ATTN_FWD, attn_fwd_flops(c), 1, attn_fwd<T>(c, qkv, o, lse_att));
    CKS(gemm(c, mk(M, d, d, o, d, 1, Wo, d, 1, EPI_STORE_F32, x, d, 1.f, 1.f)));
    KL(NC_FAM_ROWS, (double)M * d * (4 + sizeof(T)) + 4.0 * M, 1, rmsnorm_fwd<T>(x, xn2, r2, M, d, s));
    // a = relu(u)^2 only: the backward recovers relu(u) as sqrt(a)
    CKS(gemm(c, mk(M, F, d, xn2, d, 1, Wfc, d, 1, EPI_RELU2A, a, F)));
    CKS(gemm(c, mk(M, d, F, a, F, 1, Wproj, F, 1, EPI_STORE_F32, x, d, 1.f, 1.f)));
  }
  T* hf = wsp<T>(c, c->off.hf);
  float* rf = wsp<float>(c, c->off.rf);
  KL(NC_FAM_ROWS, (double)M * d * (4 + sizeof(T)) + 4.0 * M, 1, rmsnorm_fwd<T>(x, hf, rf, M, d, s));
  return NC_OK;
}

template <typename T>
nc_status forward_impl(nc_ctx* c, const T* P, const int* tok, const int* tgt, float* d_loss) {
  const int M = c->M, V = c->V;
  cudaStream_t s = c->stream;
  KL(NC_FAM_ROWS, 4.0 * M, 1, check_ids(tgt, M, -1, V, c->status, s));  // -1: masked target
  CKS(forward_blocks<T>(c, P, tok));
  T* hf = wsp<T>(c, c->off.hf);
  int rows, cols;
  const T* Wlm = P + param_offset(c, 1 + 4 * c->L, &rows, &cols);
  CKS(lmhead_ce_forward<T>(c, hf, Wlm, tgt, M, wsp<float>(c, c->off.lse), wsp<float>(c, c->off.nll),
                           wsp<int>(c, c->off.amax)));
  KL(NC_FAM_ROWS, 8.0 * M, 1, mean_loss(wsp<float>(c, c->off.nll), tgt, M, d_loss, wsp<float>(c, c->off.inv_count), s));
  return NC_OK;
}

// G = d(loss)/d(params), or with accumulate G += scale * d(loss)/d(params):
// the scale enters once, in the loss gradient (every other gradient is linear
// in it), and every parameter gradient is then added instead of stored.
template <typename T>
nc_status backward_impl(nc_ctx* c, const T* P, const int* tok, const int* tgt, float* G, bool accumulate = false,
                        float scale = 1.f) {
  int M = c->M, d = c->d, H = c->H, F = c->F, V = c->V, Tn = c->T;
  cudaStream_t s = c->stream;
  const float gb = accumulate ? 1.f : 0.f;  // beta of every parameter-gradient GEMM
  const float* gscale = wsp<float>(c, c->off.inv_count);
  if (scale != 1.f) {
    CK(scale_scalar(gscale, scale, wsp<float>(c, c->off.grad_scale), s));
    gscale = wsp<float>(c, c->off.grad_scale);
  }
  int rows, cols;
  float* dx = wsp<float>(c, c->off.dx);
  T* dxe = wsp<T>(c, c->off.dxe);
  T* dy = wsp<T>(c, c->off.dy);  // gradient into each RMSNorm, element type
  T* du = wsp<T>(c, c->off.du);
  T* dout = wsp<T>(c, c->off.dout);
  T* dqkv = wsp<T>(c, c->off.dqkv);
  float* dqk = wsp<float>(c, c->off.dqk);
  float* drow = wsp<float>(c, c->off.drow);
  const T* hf = wsp<T>(c, c->off.hf);
  size_t o_lm = param_offset(c, 1 + 4 * c->L, &rows, &cols);
  CKS((lmhead_ce_backward<T, T>(c, hf, P + o_lm, tgt, wsp<float>(c, c->off.lse), M, gscale, dy, G + o_lm,
                                accumulate)));
  KL(NC_FAM_ROWS, (double)M * d * (4 + 3 * sizeof(T)) + 4.0 * M, 1, rmsnorm_bwd<T>(dy, hf, wsp<float>(c, c->off.rf), dx, dxe, M, d, 0, s));
  for (int l = c->L - 1; l >= 0; --l) {
    size_t lb = (size_t)l * c->off.layer_stride;
    const T* xn1 = wsp<T>(c, lb + c->off.xn1);
    const float* r1 = wsp<float>(c, lb + c->off.r1);
    const T* qkv = wsp<T>(c, lb + c->off.qkv);
    const float* rqk = wsp<float>(c, lb + c->off.rqk);
    const T* o = wsp<T>(c, lb + c->off.o);
    const float* lse_att = wsp<float>(c, lb + c->off.lse_att);
    const T* xn2 = wsp<T>(c, lb + c->off.xn2);
    const float* r2 = wsp<float>(c, lb + c->off.r2);
    const T* a = wsp<T>(c, lb + c->off.a);
    size_t oq = param_offset(c, 1 + 4 * l, &rows, &cols);
    size_t oo = param_offset(c, 2 + 4 * l, &rows, &cols);
    size_t of = param_offset(c, 3 + 4 * l, &rows, &cols);
    size_t op = param_offset(c, 4 + 4 * l, &rows, &cols);
    // MLP: x += relu2(xn2 Wfc^T) Wproj^T
    CKS(gemm(c, mk(d, F, M, dxe, d, 0, a, F, 0, EPI_STORE_F32, G + op, F, 1.f, gb)));
    GemmArgs g1 = mk(M, F, d, dxe, d, 1, P + op, F, 0, EPI_RELU2_BWD, du, F);
    g1.C2 = const_cast<T*>(a); g1.ldc2 = F;  // relu(u) = sqrt(a)
    CKS(gemm(c, g1));
    CKS(gemm(c, mk(F, d, M, du, F, 0, xn2, d, 0, EPI_STORE_F32, G + of, d, 1.f, gb)));
    CKS(gemm(c, mk(M, d, F, du, F, 1, P + of, d, 0, sizeof(T) == 4 ? EPI_STORE_F32 : EPI_STORE, dy, d)));
    KL(NC_FAM_ROWS, (double)M * d * (8 + 3 * sizeof(T)) + 4.0 * M, 1, rmsnorm_bwd<T>(dy, xn2, r2, dx, dxe, M, d, 1, s));
    // attention: x += attn(xn1) Wo^T
    CKS(gemm(c, mk(d, d, M, dxe, d, 0, o, d, 0, EPI_STORE_F32, G + oo, d, 1.f, gb)));
    if (sizeof(T) == 2 && c->use_tc && c->prec == NC_BF16) {
      // dout with the attention backward's row terms in its epilogue: D = rowsum(dout o) per head
      // and the negated base-2 lse rows, with o loaded by tensor copies beside the accumulator
      GemmArgs gd = mk(M, d, d, dxe, d, 1, P + oo, d, 0, EPI_ROWDOT, dout, d);
      gd.C2 = const_cast<T*>(o);
      gd.ldc2 = d;
      gd.seq_len = Tn;
      gd.rd_D = drow;
      gd.rd_L2 = drow + (size_t)M * H;
      gd.rd_lse = lse_att;
      CKS(gemm(c, gd));
    } else {
      CKS(gemm(c, mk(M, d, d, dxe, d, 1, P + oo, d, 0, EPI_STORE, dout, d)));
      KL(NC_FAM_ROWS, 2.0 * M * d * sizeof(T) + (sizeof(T) == 2 ? 12.0 : 4.0) * M * H, 1,
         attn_rowdot<T>(dout, o, drow, c->B, Tn, H, s, sizeof(T) == 2 ? lse_att : nullptr,
                        sizeof(T) == 2 ? drow + (size_t)M * H : nullptr));
    }
    const bool fused_k = c->prec == NC_BF16;  // k half of the QK-norm/RoPE backward inside the kernel
    KL(NC_FAM_ATTN_BWD, 2.0 * attn_fwd_flops(c), fused_k ? 1 : 2,
       attn_bwd<T>(c, qkv, dout, lse_att, drow, dqk, dqkv, fused_k ? rqk : nullptr));
    KL(NC_FAM_ROWS, (fused_k ? 1.0 : 2.0) * M * d * (4 + 2 * sizeof(T)) + 8.0 * M * H, 1,
       qk_norm_rope_bwd<T>(dqk, qkv, rqk, c->rope_cos, c->rope_sin, dqkv, M, Tn, H, s, fused_k ? 1 : 2));
    CKS(gemm(c, mk(3 * d, d, M, dqkv, 3 * d, 0, xn1, d, 0, EPI_STORE_F32, G + oq, d, 1.f, gb)));
    CKS(gemm(c, mk(M, d, 3 * d, dqkv, 3 * d, 1, P + oq, d, 0, sizeof(T) == 4 ? EPI_STORE_F32 : EPI_STORE, dy, d)));
    KL(NC_FAM_ROWS, (double)M * d * (8 + 3 * sizeof(T)) + 4.0 * M, 1, rmsnorm_bwd<T>(dy, xn1, r1, dx, dxe, M, d, 1, s));
  }
  if (!accumulate) CK(cudaMemsetAsync(G, 0, (size_t)V * d * sizeof(float), s));
  // deterministic scatter: sort keys in the D-row buffer, run sums in the dq/dk plane (both dead here)
  KL(NC_FAM_ROWS, 8.0 * M * d + 4.0 * M, embed_bwd_launches(M, d, V, true),
     embed_bwd<T>(tok, nullptr, dx, G, M, d, V, s, reinterpret_cast<unsigned*>(drow), dqk));
  return NC_OK;
}

nc_status forward_any(nc_ctx* c, const void* params, const int32_t* tok, const int32_t* tgt, float* d_loss) {
  if (!params || !tok || !tgt || !d_loss) return fail(NC_ERR_ARG, "null pointer argument");
  CKS(check_ready(c));
  c->have_fwd = false;
  nc_status st = c->prec == NC_BF16
                     ? forward_impl<bf16>(c, static_cast<const bf16*>(params), tok, tgt, d_loss)
                     : forward_impl<float>(c, static_cast<const float*>(params), tok, tgt, d_loss);
  if (st != NC_OK) return st;
  c->params = params; c->tok = tok; c->tgt = tgt; c->have_fwd = true;
  return NC_OK;
}


// ------------------------------------------------------------------ optimizer

// Quintic Newton-Schulz coefficients of Muon as Keller Jordan published it.
constexpr float kNsA = 3.4445f, kNsB = -4.7750f, kNsC = 2.0315f;

// Matrix kinds of a layer in flat order: rows, cols (in units of d) and the
// offset inside the layer (units of d^2).
struct Kind { int r, c, pre; };
constexpr Kind kKinds[4] = {{3, 1, 0}, {1, 1, 3}, {4, 1, 4}, {1, 4, 8}};

// ns_steps Newton-Schulz iterations on the stacked matrices of one kind
// (all L layers per launch). X holds the normalised start; Y, A, Bp are
// scratch; *out gets whichever of X / Y holds the result. Wide matrices
// (rows <= cols) iterate X <- a X + Bp X with A = X X^T; tall ones iterate the
// transpose Y = X^T directly: A = Y^T Y and Y <- a Y + Y Bp^T, which is the
// same iteration read transposed, with no transpose in memory.
template <typename T>
nc_status newton_schulz(nc_ctx* c, int kind, T* X, T* Y, T* A, T* Bp, T** out) {
  const long long d = c->d, r = kKinds[kind].r * d, cc = kKinds[kind].c * d;
  const bool tall = r > cc;
  const long long s = tall ? cc : r;
  const int L = c->L;
  T* cur = X;
  T* nxt = Y;
  for (int it = 0; it < c->opt_ns; ++it) {
    GemmArgs g1 = tall ? mk((int)s, (int)s, (int)r, cur, cc, 0, cur, cc, 0, EPI_STORE, A, s)
                       : mk((int)s, (int)s, (int)cc, cur, cc, 1, cur, cc, 1, EPI_STORE, A, s);
    g1.batch = L; g1.a_brows = r; g1.b_brows = r; g1.c_brows = s;
    CKS(gemm(c, g1));
    GemmArgs g2 = mk((int)s, (int)s, (int)s, A, s, 1, A, s, 0, EPI_AXPBY, Bp, s, kNsC, kNsB);
    g2.C2 = A; g2.ldc2 = s;
    g2.batch = L; g2.a_brows = s; g2.b_brows = s; g2.c_brows = s;
    CKS(gemm(c, g2));
    GemmArgs g3 = tall ? mk((int)r, (int)cc, (int)cc, cur, cc, 1, Bp, s, 1, EPI_AXPBY, nxt, cc, 1.f, kNsA)
                       : mk((int)r, (int)cc, (int)r, Bp, s, 1, cur, cc, 0, EPI_AXPBY, nxt, cc, 1.f, kNsA);
    g3.C2 = cur; g3.ldc2 = cc;
    g3.batch = L; g3.a_brows = tall ? r : s; g3.b_brows = tall ? s : r; g3.c_brows = r;
    CKS(gemm(c, g3));
    T* t = cur; cur = nxt; nxt = t;
  }
  *out = cur;
  return NC_OK;
}

template <typename T>
nc_status optim_step(nc_ctx* c, T* param, const float* grads, float* state, int t, float lr_a, float lr_m, float wd,
                     float max_norm, float* stats_out) {
  const long long d = c->d, V = c->V, L = c->L, d2 = d * d;
  const long long P = 2 * V * d + 12 * L * d2, Vd = V * d, nb = 12 * L * d2;
  const size_t e = sizeof(T);
  float* master = state;
  float* m1 = master + P;
  float* m2 = m1 + 2 * Vd;
  float* buf = m2 + 2 * Vd;
  auto& q = c->opt;
  float* stats = wsp<float>(c, q.stats);
  double* part_norm = wsp<double>(c, q.part_norm);
  double* part_muon = wsp<double>(c, q.part_muon);
  float* inv_norm = wsp<float>(c, q.inv_norm);
  T* x_all = wsp<T>(c, q.x_all);
  T* pong = wsp<T>(c, q.pong);
  T* gram = wsp<T>(c, q.gram);
  T* poly = wsp<T>(c, q.poly);
  const float b1 = c->opt_b1, b2 = c->opt_b2;
  const float inv_bc1 = (float)(1.0 / (1.0 - pow((double)b1, t)));
  const float inv_bc2 = (float)(1.0 / (1.0 - pow((double)b2, t)));
  KL(NC_FAM_OPT_ELEM, 4.0 * P, 2, grad_norm(grads, P, max_norm, part_norm, stats, stats_out, c->stream));
  KL(NC_FAM_OPT_ELEM, 2.0 * Vd * (7 * 4 + e), 1,
     adamw_update<T>(master, param, grads, m1, m2, Vd, P - Vd, stats, lr_a, b1, b2, c->opt_eps, wd, inv_bc1, inv_bc2,
                     c->stream));
  KL(NC_FAM_OPT_ELEM, 12.0 * nb, 1, muon_momentum(grads + Vd, buf, nb, stats, c->opt_mu, part_muon, c->stream));
  KL(NC_FAM_OPT_ELEM, (8.0 + e) * nb, 2,
     muon_normalize<T>(grads + Vd, buf, stats, c->opt_mu, part_muon, inv_norm, (int)L, (int)d, x_all, c->stream));
  for (int k = 0; k < 4; ++k) {
    const Kind& kd = kKinds[k];
    const long long msize = (long long)kd.r * kd.c * d2;
    T* fin = nullptr;
    c->gemm_fam = NC_FAM_OPT_NS;
    nc_status st = newton_schulz<T>(c, k, x_all + (long long)kd.pre * L * d2, pong, gram, poly, &fin);
    c->gemm_fam = NC_FAM_GEMM;
    CKS(st);
    const float scale = (float)sqrt(fmax(1.0, (double)kd.r / kd.c));
    KL(NC_FAM_OPT_ELEM, (double)L * msize * (2 * e + 8), 1,
       muon_apply<T>(master + Vd, param + Vd, fin, (int)L, msize, 12 * d2, (long long)kd.pre * d2, 1.f - lr_m * wd,
                     lr_m * scale, c->stream));
  }
  return NC_OK;
}


// ------------------------------------------------------------------ generation

// KV cache buffer: per layer K then V, each [B][H][max_len][128] elem; then the
// RoPE table for max_len positions (cos, sin fp32 [max_len, 64]); then the
// attention partials of one decode step.
struct KvLayout {
  size_t per, rc, rs, part, cnt, skp, skc, total;
};
KvLayout kv_layout(const nc_ctx* c, int max_len) {
  KvLayout k;
  const size_t Bn = c->B, H = c->H, L = c->L, ml = max_len;
  k.per = align_up(Bn * H * ml * 128 * c->esz);
  size_t o = 2 * L * k.per;
  k.rc = o;
  o += align_up(ml * 64 * 4);
  k.rs = o;
  o += align_up(ml * 64 * 4);
  k.part = o;
  const size_t nch = (ml + kDecodeChunk - 1) / kDecodeChunk;
  o += align_up(Bn * H * nch * kDecodePartFloats * 4);
  k.cnt = o;  // per (sequence, head): chunks of the decode attention done (0 between calls)
  o += align_up(Bn * H * 4);
  // k-range partial sums and per-column-block counters of the weight-streaming products
  size_t skf = 0, skn = 0;
  const int d = c->d, F = c->F, V = c->V;
  const int shapes[5][2] = {{3 * d, d}, {d, d}, {F, d}, {d, F}, {V, d}};
  for (const auto& nk : shapes) {
    skf = std::max(skf, skinny_scratch_floats(nk[0], nk[1]));
    skn = std::max(skn, (size_t)skinny_counters(nk[0]));
  }
  k.skp = o;
  o += align_up(skf * 4);
  k.skc = o;
  o += align_up(skn * 4);
  k.total = o;
  return k;
}

// One product of the decode step, C (fp32 [B, N]) = A W^T (+ beta C) with A
// (elem [B, K]) one row per sequence: the weight-streaming kernel in bf16 for
// up to 16 rows, the step's GEMM otherwise. Timed as decode GEMM work, counted
// in weight bytes streamed.
// With relu2 given the product leaves as relu2 = relu(A W^T)^2 (elem [B, N]):
// fused into the weight-streaming kernel, else through C and a row kernel.
// With xres given (the fp32 residual rows), A is their RMSNorm: formed inside
// the weight-streaming kernel, else written to A by the row kernel first (r
// receives the row scales). kv: the KV cache buffer, whose scratch holds the
// weight-streaming kernel's k-range partial sums and counters.
template <typename T>
nc_status dec_gemm(nc_ctx* c, char* kv, const KvLayout& kl, int N, int K, const T* A, const T* W, float* C,
                   float beta, T* relu2 = nullptr, const float* xres = nullptr, float* r = nullptr) {
  const int Bn = c->B;
  if constexpr (sizeof(T) == 2) {
    if (skinny_gemm_supports(Bn, N, K, K, K, A, W) &&
        (!xres || ((reinterpret_cast<uintptr_t>(xres) & 15) == 0 && skinny_gemm_norm_ok(N, K)))) {
      KL(NC_FAM_DEC_GEMM, (double)N * K * sizeof(T), 1,
         skinny_gemm(A, K, W, K, C, N, Bn, N, K, 1.f, beta, c->sms, c->stream, relu2,
                     reinterpret_cast<float*>(kv + kl.skp), reinterpret_cast<int*>(kv + kl.skc), c->status, xres));
      return NC_OK;
    }
  }
  if (xres)
    KL(NC_FAM_DEC_ROWS, (double)Bn * K * (4 + c->esz), 1,
       rmsnorm_fwd<T>(xres, const_cast<T*>(A), r, Bn, K, c->stream));
  c->gemm_fam = NC_FAM_DEC_GEMM;
  nc_status st = gemm(c, mk(Bn, N, K, A, K, 1, W, K, 1, EPI_STORE_F32, C, N, 1.f, beta));
  c->gemm_fam = NC_FAM_GEMM;
  CKS(st);
  if (relu2) KL(NC_FAM_DEC_ROWS, (double)Bn * N * (4 + c->esz), 1, relu2_rows<T>(C, relu2, (long long)Bn * N, c->stream));
  return NC_OK;
}

// Greedy head over B rows of final hidden state: argmax (lowest index on
// ties) into next; fp32 logits too when requested. With the weight-streaming
// product the logits of the B rows are formed in fp32 (in the caller's buffer
// when given, else in the workspace) and reduced per row.
template <typename T>
nc_status decode_head(nc_ctx* c, char* kv, const KvLayout& kl, const T* P, const T* hf, int32_t* next,
                      float* logits, const float* xres = nullptr, float* r = nullptr) {
  const int Bn = c->B, d = c->d, V = c->V;
  int rows, cols;
  const T* Wlm = P + param_offset(c, 1 + 4 * c->L, &rows, &cols);
  const int* tgt = wsp<int>(c, c->dec.tgt);  // all -1 (set by the caller): only lse and argmax
  if (c->prec == NC_BF16 && skinny_gemm_supports(Bn, V, d, d, d, hf, Wlm)) {
    float* lg = logits ? logits : wsp<float>(c, c->off.chunk);
    CKS(dec_gemm<T>(c, kv, kl, V, d, hf, Wlm, lg, 0.f, nullptr, xres, r));
    KL(NC_FAM_DEC_ROWS, 4.0 * Bn * V, 1,
       ce_rows_from_logits(lg, tgt, wsp<float>(c, c->dec.lse), wsp<float>(c, c->dec.nll), next, Bn, V, c->status,
                           c->stream, wsp<float>(c, c->dec.cep), c->status + 3, c->sms));
    return NC_OK;
  }
  if (xres)
    KL(NC_FAM_DEC_ROWS, (double)Bn * d * (4 + c->esz), 1, rmsnorm_fwd<T>(xres, const_cast<T*>(hf), r, Bn, d, c->stream));
  c->gemm_fam = NC_FAM_DEC_GEMM;
  nc_status st = lmhead_ce_forward<T>(c, hf, Wlm, tgt, Bn, wsp<float>(c, c->dec.lse), wsp<float>(c, c->dec.nll), next);
  if (st == NC_OK && logits) st = gemm(c, mk(Bn, V, d, hf, d, 1, Wlm, d, 1, EPI_STORE_F32, logits, V));
  c->gemm_fam = NC_FAM_GEMM;
  return st;
}

void rope_table(int n, std::vector<float>& hc, std::vector<float>& hs) {
  hc.resize((size_t)n * kHalf);
  hs.resize((size_t)n * kHalf);
  for (int t = 0; t < n; ++t)
    for (int j = 0; j < kHalf; ++j) {
      const double ang = (double)t * pow(10000.0, -(double)j / (double)kHalf);
      hc[(size_t)t * kHalf + j] = (float)cos(ang);
      hs[(size_t)t * kHalf + j] = (float)sin(ang);
    }
}

template <typename T>
nc_status prefill_impl(nc_ctx* c, const T* P, const int* tok, char* kv, int max_len, int32_t* next, float* logits) {
  const KvLayout kl = kv_layout(c, max_len);
  // the table for max_len positions is built on the host once per length and
  // kept on the device; each prefill copies it into the cache device to device
  if (c->dec_rope_len != max_len) {
    if (c->dec_rope) { cudaFree(c->dec_rope); c->dec_rope = nullptr; c->dec_rope_len = 0; }
    std::vector<float> hc, hs;
    rope_table(max_len, hc, hs);
    CK(cudaMalloc(&c->dec_rope, 2 * hc.size() * 4));
    CK(cudaMemcpyAsync(c->dec_rope, hc.data(), hc.size() * 4, cudaMemcpyHostToDevice, c->stream));
    CK(cudaMemcpyAsync(c->dec_rope + hc.size(), hs.data(), hs.size() * 4, cudaMemcpyHostToDevice, c->stream));
    CK(cudaStreamSynchronize(c->stream));  // the host tables go out of scope
    c->dec_rope_len = max_len;
  }
  const size_t tab = (size_t)max_len * kHalf;
  CK(cudaMemcpyAsync(kv + kl.rc, c->dec_rope, tab * 4, cudaMemcpyDeviceToDevice, c->stream));
  CK(cudaMemcpyAsync(kv + kl.rs, c->dec_rope + tab, tab * 4, cudaMemcpyDeviceToDevice, c->stream));
  CK(cudaMemsetAsync(kv + kl.cnt, 0, (size_t)c->B * c->H * 4, c->stream));
  CK(cudaMemsetAsync(kv + kl.skc, 0, kl.total - kl.skc, c->stream));
  CKS(forward_blocks<T>(c, P, tok));
  for (int l = 0; l < c->L; ++l) {
    const T* qkv = wsp<T>(c, (size_t)l * c->off.layer_stride + c->off.qkv);
    T* K = reinterpret_cast<T*>(kv + (size_t)2 * l * kl.per);
    T* Vc = reinterpret_cast<T*>(kv + (size_t)(2 * l + 1) * kl.per);
    KL(NC_FAM_DEC_ROWS, 4.0 * c->M * c->d * c->esz, 1, kv_from_qkv<T>(qkv, K, Vc, c->B, c->T, c->H, max_len, c->stream));
  }
  T* hl = wsp<T>(c, c->dec.hf);
  KL(NC_FAM_DEC_ROWS, 2.0 * c->B * c->d * c->esz, 1, gather_last<T>(wsp<T>(c, c->off.hf), hl, c->B, c->T, c->d, c->stream));
  CK(cudaMemsetAsync(wsp<int>(c, c->dec.tgt), 0xff, (size_t)c->B * sizeof(int), c->stream));
  return decode_head<T>(c, kv, kl, P, hl, next, logits);
}

// pos: the step's position, or -1 with d_pos: read it from device memory and
// advance it after the step (graph-replayable: no host decision depends on it)
template <typename T>
nc_status decode_impl(nc_ctx* c, const T* P, const int* tok, int pos, int* d_pos, char* kv, int max_len, int32_t* next,
                      float* logits) {
  const KvLayout kl = kv_layout(c, max_len);
  const int Bn = c->B, d = c->d, H = c->H, F = c->F, V = c->V;
  cudaStream_t s = c->stream;
  const double e = c->esz;
  float* x = wsp<float>(c, c->dec.x);
  float* r = wsp<float>(c, c->dec.r);
  T* xn = wsp<T>(c, c->dec.xn);
  float* qkv = wsp<float>(c, c->dec.qkv);
  T* o = wsp<T>(c, c->dec.o);
  float* u = wsp<float>(c, c->dec.u);
  T* a = wsp<T>(c, c->dec.a);
  T* hf = wsp<T>(c, c->dec.hf);
  const float* rc = reinterpret_cast<const float*>(kv + kl.rc);
  const float* rs = reinterpret_cast<const float*>(kv + kl.rs);
  float* part = reinterpret_cast<float*>(kv + kl.part);
  int* cnt = reinterpret_cast<int*>(kv + kl.cnt);
  // the greedy head's targets: -1 (no target, only lse and argmax)
  CK(cudaMemsetAsync(wsp<int>(c, c->dec.tgt), 0xff, (size_t)Bn * sizeof(int), s));
  KL(NC_FAM_DEC_ROWS, (double)Bn * d * (e + 4) + 4.0 * Bn, 1, embed_fwd<T>(tok, P, x, Bn, d, V, c->status, s));
  int rows, cols;
  for (int l = 0; l < c->L; ++l) {
    const T* Wqkv = P + param_offset(c, 1 + 4 * l, &rows, &cols);
    const T* Wo = P + param_offset(c, 2 + 4 * l, &rows, &cols);
    const T* Wfc = P + param_offset(c, 3 + 4 * l, &rows, &cols);
    const T* Wproj = P + param_offset(c, 4 + 4 * l, &rows, &cols);
    T* K = reinterpret_cast<T*>(kv + (size_t)2 * l * kl.per);
    T* Vc = reinterpret_cast<T*>(kv + (size_t)(2 * l + 1) * kl.per);
    // each RMSNorm rides in the product that consumes it (the kernel normalises x itself)
    CKS(dec_gemm<T>(c, kv, kl, 3 * d, d, xn, Wqkv, qkv, 0.f, nullptr, x, r));
    KL(NC_FAM_DEC_ATTN, 2.0 * Bn * d * ((d_pos ? max_len : pos) + 1) * e, 1,
       attn_decode<T>(qkv, rc, rs, K, Vc, part, cnt, o, Bn, H, pos, d_pos, max_len, kDecodeChunk, c->status, s));
    CKS(dec_gemm<T>(c, kv, kl, d, d, o, Wo, x, 1.f));
    CKS(dec_gemm<T>(c, kv, kl, F, d, xn, Wfc, u, 0.f, a, x, r));
    CKS(dec_gemm<T>(c, kv, kl, d, F, a, Wproj, x, 1.f));
  }
  CKS(decode_head<T>(c, kv, kl, P, hf, next, logits, x, r));
  if (d_pos) KL(NC_FAM_DEC_ROWS, 8.0, 1, advance_pos(d_pos, s));
  return NC_OK;
}

}  // namespace

// ====================================================================== ABI

extern "C" {

nc_status nc_create(int depth, int d_model, int n_head, int seq_len, int vocab, nc_ctx** out) {
  if (!out) return fail(NC_ERR_ARG, "out is null");
  *out = nullptr;
  if (depth < 1 || depth > 512) return fail(NC_ERR_ARG, "depth %d outside [1, 512]", depth);
  if (n_head < 1 || d_model != 128 * n_head)
    return fail(NC_ERR_ARG, "d_model (%d) must equal 128 * n_head (%d): head_dim is 128", d_model, n_head);
  if (vocab < 128 || vocab > (1 << 20) || vocab % 128 != 0)
    return fail(NC_ERR_ARG, "vocab %d must be a multiple of 128 in [128, 2^20]", vocab);
  if (seq_len < 1 || seq_len > (1 << 16)) return fail(NC_ERR_ARG, "seq_len %d outside [1, 65536]", seq_len);
  nc_ctx* c = new (std::nothrow) nc_ctx();
  if (!c) return fail(NC_ERR_ARG, "out of host memory");
  c->L = depth; c->d = d_model; c->H = n_head; c->T = seq_len; c->V = vocab; c->F = 4 * d_model;
  *out = c;
  g_err.clear();
  return NC_OK;
}

nc_status nc_configure(nc_ctx* c, int batch, int precision, void* stream) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  if (batch < 1) return fail(NC_ERR_ARG, "batch %d < 1", batch);
  if ((long long)batch * c->T > (1LL << 22)) return fail(NC_ERR_ARG, "batch*seq_len too large");
  if (precision != NC_BF16 && precision != NC_FP32_DEBUG) return fail(NC_ERR_ARG, "unknown precision %d", precision);
  if (precision == NC_BF16 && c->T % 128 != 0)
    return fail(NC_ERR_ARG, "NC_BF16 needs seq_len %% 128 == 0 (got %d)", c->T);
  int dev = -1;
  CK(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3)
    return fail(NC_ERR_UNSUPPORTED, "this library is built for sm_103a (B300); device is sm_%d%d", prop.major, prop.minor);
  if (c->rope_cos) { cudaFree(c->rope_cos); c->rope_cos = nullptr; }
  if (c->rope_sin) { cudaFree(c->rope_sin); c->rope_sin = nullptr; }
  if (c->rope_cos4) { cudaFree(c->rope_cos4); c->rope_cos4 = nullptr; }
  if (c->rope_sin4) { cudaFree(c->rope_sin4); c->rope_sin4 = nullptr; }
  // the decode table is rebuilt on the (possibly different) device by the next prefill
  if (c->dec_rope) { cudaFree(c->dec_rope); c->dec_rope = nullptr; }
  c->dec_rope_len = 0;
  // device words: [0] status, [1] and [2] work counters of the persistent attention backward and forward,
  // [3] the finished-CTA count of the split cross-entropy rows (left at 0 by each launch).
  // A context configured again on another device gets them anew there, like the tables above.
  if (c->status && c->device >= 0 && c->device != dev) {
    cudaFree(c->status);
    c->status = nullptr;
    if (c->tile_done) cudaFree(c->tile_done);
    c->tile_done = nullptr;
  }
  if (!c->status) CK(cudaMalloc(&c->status, 16 * sizeof(int)));
  if (!c->tile_done) CK(cudaMalloc(&c->tile_done, kGemmTileCap * sizeof(int)));
  // RoPE table: angle pos * 10000^(-j/64) formed in float64, stored fp32.
  // Also stored angle-major in groups of four angles, [16][T][4], for the
  // epilogues whose threads each own one position: consecutive threads then
  // read consecutive 16-byte pieces.
  std::vector<float> hc((size_t)c->T * kHalf), hs((size_t)c->T * kHalf);
  std::vector<float> hc4((size_t)c->T * kHalf), hs4((size_t)c->T * kHalf);
  for (int t = 0; t < c->T; ++t)
    for (int j = 0; j < kHalf; ++j) {
      double ang = (double)t * pow(10000.0, -(double)j / (double)kHalf);
      hc[(size_t)t * kHalf + j] = (float)cos(ang);
      hs[(size_t)t * kHalf + j] = (float)sin(ang);
      const size_t i4 = ((size_t)(j / 4) * c->T + t) * 4 + j % 4;
      hc4[i4] = hc[(size_t)t * kHalf + j];
      hs4[i4] = hs[(size_t)t * kHalf + j];
    }
  CK(cudaMalloc(&c->rope_cos, hc.size() * sizeof(float)));
  CK(cudaMalloc(&c->rope_sin, hs.size() * sizeof(float)));
  CK(cudaMalloc(&c->rope_cos4, hc4.size() * sizeof(float)));
  CK(cudaMalloc(&c->rope_sin4, hs4.size() * sizeof(float)));
  c->stream = static_cast<cudaStream_t>(stream);
  CK(cudaMemcpyAsync(c->rope_cos, hc.data(), hc.size() * sizeof(float), cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->rope_sin, hs.data(), hs.size() * sizeof(float), cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->rope_cos4, hc4.data(), hc4.size() * sizeof(float), cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->rope_sin4, hs4.data(), hs4.size() * sizeof(float), cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemsetAsync(c->status, 0, 16 * sizeof(int), c->stream));
  CK(cudaMemsetAsync(c->tile_done, 0, kGemmTileCap * sizeof(int), c->stream));
  CK(cudaStreamSynchronize(c->stream));
  c->device = dev;
  c->sms = prop.multiProcessorCount > 0 ? prop.multiProcessorCount : 148;
  c->B = batch; c->M = batch * c->T; c->prec = precision;
  c->esz = precision == NC_BF16 ? 2 : 4;
  c->use_tc = precision == NC_BF16;
  plan_workspace(c);
  c->ws = nullptr; c->ws_bytes = 0; c->have_fwd = false;
  return NC_OK;
}

size_t nc_param_count(const nc_ctx* c) {
  if (!c) return 0;
  return 2 * (size_t)c->V * c->d + 12 * (size_t)c->L * c->d * c->d;
}

nc_status nc_param_offset(const nc_ctx* c, int index, size_t* offset, int* rows, int* cols) {
  if (!c || !offset || !rows || !cols) return fail(NC_ERR_ARG, "null argument");
  if (index < 0 || index > 1 + 4 * c->L) return fail(NC_ERR_ARG, "index %d outside [0, %d]", index, 1 + 4 * c->L);
  *offset = param_offset(c, index, rows, cols);
  return NC_OK;
}

size_t nc_workspace_bytes(const nc_ctx* c) { return c && c->prec >= 0 ? c->ws_need : 0; }

nc_status nc_set_workspace(nc_ctx* c, void* p, size_t bytes) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  if (c->prec < 0) return fail(NC_ERR_STATE, "nc_configure has not been called");
  if (!p) return fail(NC_ERR_ARG, "null workspace");
  if (reinterpret_cast<uintptr_t>(p) % kAlign) return fail(NC_ERR_ARG, "workspace must be %zu-byte aligned", kAlign);
  if (bytes < c->ws_need) return fail(NC_ERR_ARG, "workspace has %zu bytes, needs %zu", bytes, c->ws_need);
  c->ws = static_cast<char*>(p);
  c->ws_bytes = bytes;
  c->have_fwd = false;
  return NC_OK;
}

nc_status nc_forward_loss_async(nc_ctx* c, const void* params, const int32_t* tok, const int32_t* tgt, float* d_loss) {
  return forward_any(c, params, tok, tgt, d_loss);
}

nc_status nc_forward_loss(nc_ctx* c, const void* params, const int32_t* tok, const int32_t* tgt, float* loss) {
  if (!loss) return fail(NC_ERR_ARG, "loss is null");
  CKS(check_ready(c));
  float* dl = wsp<float>(c, c->off.loss);
  CKS(forward_any(c, params, tok, tgt, dl));
  CK(cudaMemcpyAsync(loss, dl, sizeof(float), cudaMemcpyDeviceToHost, c->stream));
  nc_status st = read_status(c);
  if (st != NC_OK) c->have_fwd = false;
  return st;
}

nc_status nc_backward(nc_ctx* c, float* grads) {
  if (!grads) return fail(NC_ERR_ARG, "grads is null");
  CKS(check_ready(c));
  if (!c->have_fwd) return fail(NC_ERR_STATE, "nc_backward needs a successful forward first");
  return c->prec == NC_BF16
             ? backward_impl<bf16>(c, static_cast<const bf16*>(c->params), c->tok, c->tgt, grads)
             : backward_impl<float>(c, static_cast<const float*>(c->params), c->tok, c->tgt, grads);
}

nc_status nc_backward_accumulate(nc_ctx* c, float* grads, float scale) {
  if (!grads) return fail(NC_ERR_ARG, "grads is null");
  if (!std::isfinite(scale)) return fail(NC_ERR_ARG, "scale must be finite");
  CKS(check_ready(c));
  if (!c->have_fwd) return fail(NC_ERR_STATE, "nc_backward_accumulate needs a successful forward first");
  return c->prec == NC_BF16
             ? backward_impl<bf16>(c, static_cast<const bf16*>(c->params), c->tok, c->tgt, grads, true, scale)
             : backward_impl<float>(c, static_cast<const float*>(c->params), c->tok, c->tgt, grads, true, scale);
}

nc_status nc_forward_loss_u16(nc_ctx* c, const void* params, const uint16_t* packed, float* d_loss) {
  if (!params || !packed || !d_loss) return fail(NC_ERR_ARG, "null pointer argument");
  CKS(check_ready(c));
  int* dt = wsp<int>(c, c->off.tok);
  int* dg = wsp<int>(c, c->off.tgt);
  CK(unpack_u16(packed, c->B, c->T, dt, dg, c->stream));
  return forward_any(c, params, dt, dg, d_loss);
}

nc_status nc_train_step_host_u16(nc_ctx* c, const void* params, const uint16_t* h_packed, float* grads,
                                 float* h_loss) {
  if (!params || !h_packed || !grads || !h_loss) return fail(NC_ERR_ARG, "null pointer argument");
  CKS(check_ready(c));
  uint16_t* dp = wsp<uint16_t>(c, c->off.packed);
  CK(cudaMemcpyAsync(dp, h_packed, (size_t)c->B * (c->T + 1) * 2, cudaMemcpyHostToDevice, c->stream));
  float* dl = wsp<float>(c, c->off.loss);
  CKS(nc_forward_loss_u16(c, params, dp, dl));
  CKS(nc_backward(c, grads));
  CK(cudaMemcpyAsync(h_loss, dl, sizeof(float), cudaMemcpyDeviceToHost, c->stream));
  return read_status(c);
}

nc_status nc_train_step_host(nc_ctx* c, const void* params, const int32_t* h_tok, const int32_t* h_tgt,
                             float* grads, float* h_loss) {
  if (!params || !h_tok || !h_tgt || !grads || !h_loss) return fail(NC_ERR_ARG, "null pointer argument");
  CKS(check_ready(c));
  int* dt = wsp<int>(c, c->off.tok);
  int* dg = wsp<int>(c, c->off.tgt);
  CK(cudaMemcpyAsync(dt, h_tok, (size_t)c->M * 4, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(dg, h_tgt, (size_t)c->M * 4, cudaMemcpyHostToDevice, c->stream));
  float* dl = wsp<float>(c, c->off.loss);
  CKS(forward_any(c, params, dt, dg, dl));
  CKS(nc_backward(c, grads));
  CK(cudaMemcpyAsync(h_loss, dl, sizeof(float), cudaMemcpyDeviceToHost, c->stream));
  return read_status(c);
}

nc_status nc_get_token_outputs(nc_ctx* c, float* d_lse, float* d_nll, int32_t* d_argmax) {
  CKS(check_ready(c));
  if (!c->have_fwd) return fail(NC_ERR_STATE, "no forward has run");
  size_t n = (size_t)c->M * 4;
  if (d_lse) CK(cudaMemcpyAsync(d_lse, c->ws + c->off.lse, n, cudaMemcpyDeviceToDevice, c->stream));
  if (d_nll) CK(cudaMemcpyAsync(d_nll, c->ws + c->off.nll, n, cudaMemcpyDeviceToDevice, c->stream));
  if (d_argmax) CK(cudaMemcpyAsync(d_argmax, c->ws + c->off.amax, n, cudaMemcpyDeviceToDevice, c->stream));
  return NC_OK;
}

nc_status nc_get_argmax(nc_ctx* c, int32_t* d_argmax) {
  if (!d_argmax) return fail(NC_ERR_ARG, "d_argmax is null");
  return nc_get_token_outputs(c, nullptr, nullptr, d_argmax);
}

nc_status nc_get_hidden(nc_ctx* c, void* d_hf) {
  CKS(check_ready(c));
  if (!c->have_fwd) return fail(NC_ERR_STATE, "no forward has run");
  if (!d_hf) return fail(NC_ERR_ARG, "d_hf is null");
  CK(cudaMemcpyAsync(d_hf, c->ws + c->off.hf, (size_t)c->M * c->d * c->esz, cudaMemcpyDeviceToDevice, c->stream));
  return NC_OK;
}

nc_status nc_sync(nc_ctx* c) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  if (c->prec < 0) return fail(NC_ERR_STATE, "nc_configure has not been called");
  CK(cudaStreamSynchronize(c->stream));
  return read_status(c);
}

unsigned long long nc_launch_count(const nc_ctx* c) { return c ? c->launches : 0; }

nc_status nc_profile_enable(nc_ctx* c, int enable) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  c->prof = enable != 0;
  c->recs.clear();
  c->pool_next = 0;
  return NC_OK;
}

nc_status nc_profile_read(nc_ctx* c, int family, double* ms, long long* launches, double* work) {
  if (!c || !ms || !launches || !work) return fail(NC_ERR_ARG, "null argument");
  if (family < 0 || family >= NC_FAM_COUNT) return fail(NC_ERR_ARG, "family %d unknown", family);
  CK(cudaStreamSynchronize(c->stream));
  double t = 0, w = 0;
  long long n = 0;
  for (auto& r : c->recs) {
    if (r.fam != family) continue;
    float x = 0.f;
    CK(cudaEventElapsedTime(&x, r.a, r.b));
    t += x;
    w += r.work;
    ++n;
  }
  *ms = t; *launches = n; *work = w;
  return NC_OK;
}

nc_status nc_profile_reset(nc_ctx* c) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  CK(cudaStreamSynchronize(c->stream));
  c->recs.clear();
  c->pool_next = 0;
  return NC_OK;
}

nc_status nc_set_pipeline_wait_limit(unsigned long long ns) {
  CK(cudaDeviceSynchronize());  // no kernel of this library may be running while the limit changes
  CK(gemm_tc_set_wait_limit(ns));
  CK(attn_tc_set_wait_limit(ns));
  CK(cudaDeviceSynchronize());
  return NC_OK;
}

const char* nc_last_error(const nc_ctx*) { return g_err.c_str(); }

void nc_destroy(nc_ctx* c) {
  if (!c) return;
  for (auto e : c->pool) cudaEventDestroy(e);
  if (c->rope_cos) cudaFree(c->rope_cos);
  if (c->rope_sin) cudaFree(c->rope_sin);
  if (c->rope_cos4) cudaFree(c->rope_cos4);
  if (c->rope_sin4) cudaFree(c->rope_sin4);
  if (c->dec_rope) cudaFree(c->dec_rope);
  if (c->status) cudaFree(c->status);
  if (c->tile_done) cudaFree(c->tile_done);
  delete c;
}

// ---------------------------------------------------------------- op-level entry points

nc_status nc_op_gemm(nc_ctx* c, int M, int N, int K, const void* A, long long lda, int a_kmajor,
                     const void* B, long long ldb, int b_kmajor, int epi, float alpha, float beta,
                     void* C, long long ldc, void* C2, long long ldc2, const float* row_f,
                     const int32_t* row_i) {
  if (!c || c->prec < 0) return fail(NC_ERR_STATE, "context not configured");
  if (M < 0 || N < 0 || K < 0) return fail(NC_ERR_ARG, "negative size");
  if (epi < EPI_STORE || epi > EPI_RELU2A || epi == EPI_CE_FWD)
    return fail(NC_ERR_ARG, "epilogue %d not available here", epi);
  if (epi == EPI_QKNORM_ROPE && (!c->use_tc || N != 3 * c->d || M != c->M || !C2))
    return fail(NC_ERR_ARG, "the QK-norm + RoPE epilogue needs NC_BF16, N = 3*d_model, M = batch*seq_len and C2 = rqk");
  if (!A || !B || !C) return fail(NC_ERR_ARG, "null operand");
  if ((epi == EPI_RELU2 || epi == EPI_RELU2_BWD || epi == EPI_AXPBY) && !C2) return fail(NC_ERR_ARG, "epilogue needs C2");
  if (epi == EPI_CE_BWD && (!row_f || !row_i)) return fail(NC_ERR_ARG, "epilogue needs row_f/row_i");
  GemmArgs g = mk(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, epi, C, ldc, alpha, beta);
  g.C2 = C2; g.ldc2 = ldc2; g.row_f = row_f; g.row_i = row_i;
  if (epi == EPI_QKNORM_ROPE) {
    g.C2 = nullptr;
    g.rqk = static_cast<float*>(C2);
    g.rope_cos = c->rope_cos4; g.rope_sin = c->rope_sin4; g.seq_len = c->T; g.d_model = c->d;
  }
  return gemm(c, g);
}

nc_status nc_op_lmhead_ce_fwd(nc_ctx* c, const void* hf, const void* w_lm, const int32_t* tgt,
                              float* lse, float* nll, int32_t* argmax) {
  CKS(check_ready(c));
  if (!hf || !w_lm || !tgt || !lse || !nll || !argmax) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  return c->prec == NC_BF16
             ? lmhead_ce_forward<bf16>(c, (const bf16*)hf, (const bf16*)w_lm, tgt, c->M, lse, nll, argmax)
             : lmhead_ce_forward<float>(c, (const float*)hf, (const float*)w_lm, tgt, c->M, lse, nll, argmax);
}

nc_status nc_op_lmhead_ce_bwd(nc_ctx* c, const void* hf, const void* w_lm, const int32_t* tgt,
                              const float* lse, float* dhf, float* dw_lm) {
  CKS(check_ready(c));
  if (!hf || !w_lm || !tgt || !lse || !dhf || !dw_lm) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  float* inv = wsp<float>(c, c->off.inv_count);  // 1 / (unmasked targets)
  KL(NC_FAM_ROWS, 4.0 * c->M, 1, mean_loss(nullptr, tgt, c->M, nullptr, inv, c->stream));
  return c->prec == NC_BF16
             ? lmhead_ce_backward<bf16, float>(c, (const bf16*)hf, (const bf16*)w_lm, tgt, lse, c->M, inv, dhf, dw_lm)
             : lmhead_ce_backward<float, float>(c, (const float*)hf, (const float*)w_lm, tgt, lse, c->M, inv, dhf, dw_lm);
}

nc_status nc_op_attention_fwd(nc_ctx* c, const void* qkv, void* o, float* lse) {
  CKS(check_ready(c));
  if (!qkv || !o || !lse) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  if (c->prec == NC_BF16) CK(attn_fwd<bf16>(c, (const bf16*)qkv, (bf16*)o, lse));
  else CK(attn_fwd<float>(c, (const float*)qkv, (float*)o, lse));
  return NC_OK;
}

nc_status nc_op_attention_bwd(nc_ctx* c, const void* qkv, const void* o, const void* dout,
                              const float* lse, float* dqk, void* dqkv) {
  CKS(check_ready(c));
  if (!qkv || !o || !dout || !lse || !dqk || !dqkv) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  float* drow = wsp<float>(c, c->off.drow);
  if (c->prec == NC_BF16) {
    CK(attn_rowdot<bf16>((const bf16*)dout, (const bf16*)o, drow, c->B, c->T, c->H, c->stream, lse,
                         drow + (size_t)c->M * c->H));
    CK(attn_bwd<bf16>(c, (const bf16*)qkv, (const bf16*)dout, lse, drow, dqk, (bf16*)dqkv));
  } else {
    CK(attn_rowdot<float>((const float*)dout, (const float*)o, drow, c->B, c->T, c->H, c->stream));
    CK(attn_bwd<float>(c, (const float*)qkv, (const float*)dout, lse, drow, dqk, (float*)dqkv));
  }
  return NC_OK;
}

nc_status nc_op_qk_norm_rope_fwd(nc_ctx* c, void* qkv, float* rqk) {
  CKS(check_ready(c));
  if (!qkv || !rqk) return fail(NC_ERR_ARG, "null pointer argument");
  if (c->prec == NC_BF16) CK(qk_norm_rope_fwd<bf16>((bf16*)qkv, rqk, c->rope_cos, c->rope_sin, c->M, c->T, c->H, c->stream));
  else CK(qk_norm_rope_fwd<float>((float*)qkv, rqk, c->rope_cos, c->rope_sin, c->M, c->T, c->H, c->stream));
  return NC_OK;
}

nc_status nc_op_rmsnorm_fwd(nc_ctx* c, const float* x, void* y, float* r) {
  CKS(check_ready(c));
  if (!x || !y || !r) return fail(NC_ERR_ARG, "null pointer argument");
  if (c->prec == NC_BF16) CK(rmsnorm_fwd<bf16>(x, (bf16*)y, r, c->M, c->d, c->stream));
  else CK(rmsnorm_fwd<float>(x, (float*)y, r, c->M, c->d, c->stream));
  return NC_OK;
}

nc_status nc_op_rmsnorm_bwd(nc_ctx* c, const void* dy, const void* y, const float* r, float* dx, void* dx_e,
                            int accumulate) {
  CKS(check_ready(c));
  if (!dy || !y || !r || !dx) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  const double bytes = (double)c->M * c->d * (4.0 * (accumulate ? 2 : 1) + c->esz * (dx_e ? 3 : 2)) + 4.0 * c->M;
  if (c->prec == NC_BF16)
    KL(NC_FAM_ROWS, bytes, 1, rmsnorm_bwd<bf16>((const bf16*)dy, (const bf16*)y, r, dx, (bf16*)dx_e, c->M, c->d,
                                                accumulate ? 1 : 0, c->stream));
  else
    KL(NC_FAM_ROWS, bytes, 1, rmsnorm_bwd<float>((const float*)dy, (const float*)y, r, dx, (float*)dx_e, c->M, c->d,
                                                 accumulate ? 1 : 0, c->stream));
  return NC_OK;
}

nc_status nc_op_embed_fwd(nc_ctx* c, const int32_t* tok, const void* wte, float* x) {
  CKS(check_ready(c));
  if (!tok || !wte || !x) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  const double bytes = (double)c->M * c->d * (c->esz + 4) + 4.0 * c->M;
  if (c->prec == NC_BF16)
    KL(NC_FAM_ROWS, bytes, 1, embed_fwd<bf16>(tok, (const bf16*)wte, x, c->M, c->d, c->V, c->status, c->stream));
  else
    KL(NC_FAM_ROWS, bytes, 1, embed_fwd<float>(tok, (const float*)wte, x, c->M, c->d, c->V, c->status, c->stream));
  return NC_OK;
}

nc_status nc_op_embed_bwd(nc_ctx* c, const int32_t* tok, const float* dx, float* dwte) {
  CKS(check_ready(c));
  if (!tok || !dx || !dwte) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  CK(cudaMemsetAsync(dwte, 0, (size_t)c->V * c->d * sizeof(float), c->stream));
  KL(NC_FAM_ROWS, 8.0 * c->M * c->d + 4.0 * c->M, embed_bwd_launches(c->M, c->d, c->V, true),
     embed_bwd<bf16>(tok, nullptr, dx, dwte, c->M, c->d, c->V, c->stream, wsp<unsigned>(c, c->off.drow),
                     wsp<float>(c, c->off.dqk)));
  return NC_OK;
}

nc_status nc_op_qk_norm_rope_bwd(nc_ctx* c, const float* dqk, const void* qkv, const float* rqk, void* dqkv) {
  CKS(check_ready(c));
  if (!dqk || !qkv || !rqk || !dqkv) return fail(NC_ERR_ARG, "null pointer argument");
  c->have_fwd = false;
  const double bytes = 2.0 * c->M * c->d * (4 + 2 * c->esz) + 8.0 * c->M * c->H;
  if (c->prec == NC_BF16)
    KL(NC_FAM_ROWS, bytes, 1, qk_norm_rope_bwd<bf16>(dqk, (const bf16*)qkv, rqk, c->rope_cos, c->rope_sin,
                                                     (bf16*)dqkv, c->M, c->T, c->H, c->stream, 2));
  else
    KL(NC_FAM_ROWS, bytes, 1, qk_norm_rope_bwd<float>(dqk, (const float*)qkv, rqk, c->rope_cos, c->rope_sin,
                                                      (float*)dqkv, c->M, c->T, c->H, c->stream, 2));
  return NC_OK;
}

// ------------------------------------------------------------------ optimizer

size_t nc_optim_state_bytes(const nc_ctx* c) {
  if (!c || c->prec < 0) return 0;
  const size_t P = nc_param_count(c), Vd = (size_t)c->V * c->d;
  return 4 * (P + 4 * Vd + 12 * (size_t)c->L * c->d * c->d);
}

nc_status nc_optim_init(nc_ctx* c, const void* params, void* state) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  if (c->prec < 0) return fail(NC_ERR_STATE, "nc_configure has not been called");
  if (!params || !state) return fail(NC_ERR_ARG, "null pointer argument");
  if ((reinterpret_cast<uintptr_t>(params) | reinterpret_cast<uintptr_t>(state)) & 15)
    return fail(NC_ERR_ARG, "params and state must be 16-byte aligned");
  const long long P = (long long)nc_param_count(c);
  float* master = static_cast<float*>(state);
  KL(NC_FAM_OPT_ELEM, (double)P * (4 + c->esz), 1,
     c->prec == NC_BF16 ? upcast<bf16>(static_cast<const bf16*>(params), master, P, c->stream)
                        : upcast<float>(static_cast<const float*>(params), master, P, c->stream));
  CK(cudaMemsetAsync(master + P, 0, nc_optim_state_bytes(c) - 4 * (size_t)P, c->stream));
  return NC_OK;
}

nc_status nc_optim_set_hparams(nc_ctx* c, float beta1, float beta2, float eps, float momentum, int ns_steps) {
  if (!c) return fail(NC_ERR_ARG, "null context");
  if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) || !(momentum >= 0.f && momentum < 1.f))
    return fail(NC_ERR_ARG, "beta1, beta2 and momentum must lie in [0, 1)");
  if (!(eps > 0.f)) return fail(NC_ERR_ARG, "eps must be positive");
  if (ns_steps < 1 || ns_steps > 32) return fail(NC_ERR_ARG, "ns_steps %d outside [1, 32]", ns_steps);
  c->opt_b1 = beta1; c->opt_b2 = beta2; c->opt_eps = eps; c->opt_mu = momentum; c->opt_ns = ns_steps;
  return NC_OK;
}

nc_status nc_optim_step(nc_ctx* c, void* params, const float* grads, void* state, int t, float lr_adamw,
                        float lr_muon, float weight_decay, float max_grad_norm, float* stats) {
  CKS(check_ready(c));
  if (!params || !grads || !state) return fail(NC_ERR_ARG, "null pointer argument");
  if ((reinterpret_cast<uintptr_t>(params) | reinterpret_cast<uintptr_t>(grads) |
       reinterpret_cast<uintptr_t>(state)) & 15)
    return fail(NC_ERR_ARG, "params, grads and state must be 16-byte aligned");
  if (t < 1) return fail(NC_ERR_ARG, "step number t = %d must be >= 1", t);
  if (!(lr_adamw >= 0.f) || !(lr_muon >= 0.f) || !(weight_decay >= 0.f) || !(max_grad_norm > 0.f))
    return fail(NC_ERR_ARG, "learning rates and weight decay must be >= 0 and max_grad_norm > 0");
  c->have_fwd = false;  // the workspace is scratch from here on
  return c->prec == NC_BF16
             ? optim_step<bf16>(c, static_cast<bf16*>(params), grads, static_cast<float*>(state), t, lr_adamw,
                                lr_muon, weight_decay, max_grad_norm, stats)
             : optim_step<float>(c, static_cast<float*>(params), grads, static_cast<float*>(state), t, lr_adamw,
                                 lr_muon, weight_decay, max_grad_norm, stats);
}

double nc_lr_at(long long step, long long warmup, long long total, double peak, double final_frac) {
  if (step < warmup) return peak * (double)(step + 1) / (double)warmup;
  double span = (double)(total - warmup);
  if (span < 1.0) span = 1.0;
  double prog = (double)(step - warmup) / span;
  if (prog > 1.0) prog = 1.0;
  if (prog < 0.0) prog = 0.0;
  return peak * (final_frac + (1.0 - final_frac) * 0.5 * (1.0 + cos(M_PI * prog)));
}

nc_status nc_op_gemm_batched(nc_ctx* c, int batch, int M, int N, int K, const void* A, long long lda,
                             int a_kmajor, long long a_brows, const void* B, long long ldb, int b_kmajor,
                             long long b_brows, int epi, float alpha, float beta, void* C, long long ldc,
                             void* C2, long long ldc2, long long c_brows) {
  if (!c || c->prec < 0) return fail(NC_ERR_STATE, "context not configured");
  if (batch < 1 || M < 0 || N < 0 || K < 0) return fail(NC_ERR_ARG, "batch < 1 or negative size");
  if (epi != EPI_STORE && epi != EPI_AXPBY) return fail(NC_ERR_ARG, "batched epilogue must be STORE or AXPBY");
  if (!A || !B || !C || (epi == EPI_AXPBY && !C2)) return fail(NC_ERR_ARG, "null operand");
  if (a_brows < 0 || b_brows < 0 || c_brows < 0) return fail(NC_ERR_ARG, "negative batch stride");
  GemmArgs g = mk(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, epi, C, ldc, alpha, beta);
  g.C2 = C2; g.ldc2 = ldc2;
  g.batch = batch; g.a_brows = a_brows; g.b_brows = b_brows; g.c_brows = c_brows;
  return gemm(c, g);
}

// ------------------------------------------------------------------ generation

size_t nc_kv_cache_bytes(const nc_ctx* c, int max_len) {
  if (!c || c->prec < 0 || max_len < 1) return 0;
  return kv_layout(c, max_len).total;
}

static nc_status check_kv(nc_ctx* c, const void* kv, int max_len) {
  if (!kv) return fail(NC_ERR_ARG, "null KV cache");
  if (reinterpret_cast<uintptr_t>(kv) % 256) return fail(NC_ERR_ARG, "the KV cache must be 256-byte aligned");
  if (max_len < c->T || max_len > (1 << 16))
    return fail(NC_ERR_ARG, "max_len %d outside [seq_len = %d, 65536]", max_len, c->T);
  return NC_OK;
}

nc_status nc_prefill(nc_ctx* c, const void* params, const int32_t* tokens, void* kv_cache, int max_len,
                     int32_t* next_tokens, float* last_logits) {
  CKS(check_ready(c));
  if (!params || !tokens || !next_tokens) return fail(NC_ERR_ARG, "null pointer argument");
  CKS(check_kv(c, kv_cache, max_len));
  c->have_fwd = false;
  char* kv = static_cast<char*>(kv_cache);
  return c->prec == NC_BF16
             ? prefill_impl<bf16>(c, static_cast<const bf16*>(params), tokens, kv, max_len, next_tokens, last_logits)
             : prefill_impl<float>(c, static_cast<const float*>(params), tokens, kv, max_len, next_tokens,
                                   last_logits);
}

nc_status nc_decode_step(nc_ctx* c, const void* params, const int32_t* tokens, int pos, void* kv_cache, int max_len,
                         int32_t* next_tokens, float* logits) {
  CKS(check_ready(c));
  if (!params || !tokens || !next_tokens) return fail(NC_ERR_ARG, "null pointer argument");
  CKS(check_kv(c, kv_cache, max_len));
  if (pos < 0 || pos >= max_len) return fail(NC_ERR_ARG, "position %d outside [0, max_len = %d)", pos, max_len);
  c->have_fwd = false;
  char* kv = static_cast<char*>(kv_cache);
  return c->prec == NC_BF16
             ? decode_impl<bf16>(c, static_cast<const bf16*>(params), tokens, pos, nullptr, kv, max_len, next_tokens,
                                 logits)
             : decode_impl<float>(c, static_cast<const float*>(params), tokens, pos, nullptr, kv, max_len, next_tokens,
                                  logits);
}

nc_status nc_decode_step_dev(nc_ctx* c, const void* params, const int32_t* tokens, int32_t* d_pos, void* kv_cache,
                             int max_len, int32_t* next_tokens, float* logits) {
  CKS(check_ready(c));
  if (!params || !tokens || !next_tokens || !d_pos) return fail(NC_ERR_ARG, "null pointer argument");
  CKS(check_kv(c, kv_cache, max_len));
  c->have_fwd = false;
  char* kv = static_cast<char*>(kv_cache);
  return c->prec == NC_BF16
             ? decode_impl<bf16>(c, static_cast<const bf16*>(params), tokens, -1, d_pos, kv, max_len, next_tokens,
                                 logits)
             : decode_impl<float>(c, static_cast<const float*>(params), tokens, -1, d_pos, kv, max_len, next_tokens,
                                  logits);
}

}  // extern "C"
