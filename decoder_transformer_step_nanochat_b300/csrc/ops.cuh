// Internal launch API of the step kernels. Every launcher enqueues on
// `stream` and returns the cudaError_t of the launch.
#pragma once

#include "common.cuh"

namespace nc {

// ------------------------------------------------------------------ GEMM
// C[m,n] = alpha * sum_k A(m,k) B(n,k), then an epilogue.
//   A(m,k) = a_kmajor ? A[m*lda + k] : A[k*lda + m]
//   B(n,k) = b_kmajor ? B[n*ldb + k] : B[k*ldb + n]
enum Epi : int {
  EPI_STORE = 0,       // C (elem) = alpha*acc
  EPI_STORE_F32 = 1,   // C (f32)  = alpha*acc + beta*C
  EPI_RELU2 = 2,       // C (elem) = u = alpha*acc ; C2 (elem) = max(u,0)^2
  EPI_RELU2_BWD = 3,   // C (elem) = alpha*acc * 2*sqrt(a), a = relu(u)^2 read from C2
  EPI_CE_BWD = 4,      // C (elem) = (exp(alpha*acc - row_f[m]) - (n == row_i[m])) * s, s = *dscale (0 if row_i[m] < 0)
  EPI_CE_FWD = 5,      // per (row, 128-column tile) softmax partials (tensor-core path)
  EPI_QKNORM_ROPE = 6, // C (elem) = qkv with per-head RMSNorm + RoPE on the q,k columns
  EPI_AXPBY = 7,       // C (elem) = alpha*acc + beta*C2 (C2 elem, same shape as C)
  EPI_RELU2A = 8,      // C (elem) = max(alpha*acc, 0)^2 only (the step keeps a, not u)
  EPI_ROWDOT = 9,      // C (elem) = alpha*acc; rd_D[b,h,t] = sum over head h's 128 columns of C (as stored) * C2,
                       // rd_L2 = -(rd_lse * log2(e) + 3.5) (tensor-core path; rows m = b*seq_len + t)
};

struct GemmArgs {
  int M = 0, N = 0, K = 0;
  const void* A = nullptr; long long lda = 0; int a_kmajor = 1;
  const void* B = nullptr; long long ldb = 0; int b_kmajor = 1;
  int epi = EPI_STORE;
  float alpha = 1.f, beta = 0.f;
  void* C = nullptr; long long ldc = 0;
  void* C2 = nullptr; long long ldc2 = 0;
  const float* row_f = nullptr;  // CE bwd: lse per row
  const int* row_i = nullptr;    // CE fwd/bwd: target id per row (negative: masked row)
  const float* dscale = nullptr; // CE bwd: device scalar the unmasked rows are scaled by (null: 1)
  // CE forward partials, [n_tiles][M] each, one tile per 128 vocabulary columns
  float* p_max = nullptr; float* p_sum = nullptr; int* p_arg = nullptr;
  float* p_tgt = nullptr;        // [M]: logit of the target column
  // QK-norm + RoPE epilogue
  // angle-major RoPE table [16][seq_len][4]: entry (g, t, u) is angle 4g + u
  // at position t, so 32 consecutive rows read 512 contiguous bytes
  const float* rope_cos = nullptr; const float* rope_sin = nullptr;
  float* rqk = nullptr;          // [M, 2H] rstd of q heads then k heads
  int seq_len = 0, d_model = 0;
  // row dot of the attention backward (EPI_ROWDOT): [B, N/128, seq_len] fp32 each
  float* rd_D = nullptr; float* rd_L2 = nullptr; const float* rd_lse = nullptr;
  // split-K (EPI_STORE_F32 only): splits > 1 writes alpha*partial sums to
  // `partial` ([splits, M, N] fp32) and a reduction kernel forms C.
  int splits = 1;
  float* partial = nullptr;
  // with tile_done (kGemmTileCap zeroed ints) and beta 0 or 1, the splits are
  // instead added into C in split order inside the kernel (no partial slabs,
  // no reduction launch); each launch leaves the counters at 0
  int* tile_done = nullptr;
  // batched problems (EPI_STORE / EPI_AXPBY, M % 128 == 0 on the tensor
  // cores): `batch` independent GEMMs whose operands are stacked along their
  // outer (row) dimension; problem i reads A rows from i*a_brows, B rows from
  // i*b_brows and writes C (and reads C2) rows from i*c_brows.
  int batch = 1;
  long long a_brows = 0, b_brows = 0, c_brows = 0;
  int* status = nullptr;
};

// Number of k-splits the tensor-core GEMM would use for this problem (1 = none).
int gemm_tc_pick_splits(const GemmArgs& g);
// C[m*ldc+n] = sum_s partial[s][m][n] + beta * C[m*ldc+n]   (fp32)
cudaError_t splitk_reduce(const float* partial, int splits, float* C, long long ldc, int M, int N, float beta,
                          cudaStream_t s);

// Plain fp32-FMA tiled GEMM (any majorness, any sizes). elem = float or bf16.
template <typename T> cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t s);

// tcgen05 / TMEM / TMA GEMM for bf16 operands. Returns cudaErrorNotSupported
// for shapes it cannot serve (the caller treats that as a hard error).
cudaError_t gemm_tc(const GemmArgs& g, cudaStream_t s);
constexpr int kGemmTileCap = 16384;  // 128 x 256 output tiles with an in-kernel split-K counter
// launches gemm_tc makes for g: 2 when a split-K reduction kernel follows
int gemm_tc_launches(const GemmArgs& g);
bool gemm_tc_supports(const GemmArgs& g);

// Weight-streaming product of the decode step: C (fp32) = alpha * A W^T (+ beta * C)
// for M <= 16 rows of A (bf16 [M, K], K-major) and W (bf16 [N, K], K-major),
// K a multiple of 32, 16-byte aligned operands; one launch, deterministic.
// sms: the device's SM count (the persistent grid). With relu2 given, the
// product u = alpha * A W^T leaves as relu2[m, n] = bf16(max(u, 0)^2) (row
// stride ldc) and C is not touched. K longer than 2048 runs in k-ranges whose
// partial sums need part (skinny_scratch_floats(N, K) floats) and cnt
// (skinny_counters(N) ints, 0 before the first call; each call leaves them 0).
// A wait past its limit sets DEV_TIMEOUT in *status. With xres (fp32 [M, K],
// row stride lda) the kernel forms A itself as bf16(xres * r), r the row's
// RMSNorm scale 1/sqrt(mean(xres^2) + eps) (the sum of squares in another
// order than rmsnorm_fwd's), when skinny_gemm_norm_ok(N, K).
bool skinny_gemm_supports(int M, int N, int K, long long lda, long long ldw, const void* A, const void* W);
size_t skinny_scratch_floats(int N, int K);
// xres (the fused RMSNorm) needs the whole row in one k-range: K <= 2048
bool skinny_gemm_norm_ok(int N, int K);
int skinny_counters(int N);
cudaError_t skinny_gemm(const bf16* A, long long lda, const bf16* W, long long ldw, float* C, long long ldc, int M,
                        int N, int K, float alpha, float beta, int sms, cudaStream_t s, bf16* relu2, float* part,
                        int* cnt, int* status, const float* xres = nullptr);

// ------------------------------------------------------------------ rows
template <typename T>
cudaError_t embed_fwd(const int* tok, const T* wte, float* x, int M, int d, int V, int* status,
                      cudaStream_t s);
// dwte[tok[m]] += dx[m] (dwte zeroed first unless accumulating). With keys
// (M uint32) and part (M x d fp32) scratch, the sum per id runs in ascending
// position order with a fixed grouping (deterministic) when d % 4 == 0, the
// position and id bit counts fit 32 bits and M <= 1024 * kEmbMaxChunks;
// otherwise by float atomics.
constexpr int kEmbMaxChunks = 1024;
template <typename T>
cudaError_t embed_bwd(const int* tok, const T* dx_unused, const float* dx, float* dwte, int M,
                      int d, int V, cudaStream_t s, unsigned* keys = nullptr, float* part = nullptr);
int embed_bwd_launches(int M, int d, int V, bool scratch);
template <typename T>
cudaError_t rmsnorm_fwd(const float* x, T* y, float* r, int M, int d, cudaStream_t s);
// dx (f32) = (accumulate ? dx : 0) + r*(dy - y*mean(dy*y)); also dx_e = elem copy (if non-null)
template <typename T>
cudaError_t rmsnorm_bwd(const T* dy, const T* y, const float* r, float* dx, T* dx_e, int M,
                        int d, int accumulate, cudaStream_t s);
template <typename T>
cudaError_t qk_norm_rope_fwd(T* qkv, float* rqk, const float* cs, const float* sn, int M, int T_,
                             int H, cudaStream_t s);
// heads = 2 (q and k heads) or 1 (q heads only: k was finished elsewhere)
template <typename T>
cudaError_t qk_norm_rope_bwd(const float* dqk, const T* qkv, const float* rqk, const float* cs,
                             const float* sn, T* dqkv, int M, int T_, int H, cudaStream_t s, int heads = 2);

// ------------------------------------------------------------------ attention
template <typename T>
cudaError_t attn_fwd_simt(const T* qkv, T* o, float* lse, int B, int T_, int H, cudaStream_t s);
template <typename T>
cudaError_t attn_rowdot(const T* dout, const T* o, float* Drow, int B, int T_, int H,
                        cudaStream_t s, const float* lse = nullptr, float* L2 = nullptr);
// dqk is planar fp32 [2, B*T, d]: dq_hat plane, then dk_hat plane.
template <typename T>
cudaError_t attn_bwd_simt(const T* qkv, const T* dout, const float* lse, const float* Drow,
                          float* dqk, T* dqkv, int B, int T_, int H, cudaStream_t s);

// Limit (ns) of the pipeline waits of the kernels launched after the call
// (0: the default of 2 s), one setter per kernel file. A test hook: the
// teardown waits keep the default, and CTA pairs (GEMMs of more than 128 rows)
// must not run under a short limit (a pair's unwinding waits for the copies of
// the phases the even CTA armed, not for copies the odd CTA started alone).
cudaError_t gemm_tc_set_wait_limit(uint64_t ns);
cudaError_t attn_tc_set_wait_limit(uint64_t ns);

// tcgen05 flash attention (bf16, T % 128 == 0).
bool attn_tc_supports(int T);
// status points at three device words: the status word, the backward's work
// counter and the forward's (reset here before the launch).
cudaError_t attn_fwd_tc(const bf16* qkv, bf16* o, float* lse, int B, int T, int H, int* status, cudaStream_t s);
// dq (zeroed here, then accumulated) is fp32 [B*T, d]; dv goes to dqkv's v columns. Without rqk,
// dk_hat goes to the fp32 plane dk; with rqk (+ the RoPE table) the k half of the QK-norm + RoPE
// backward runs in the kernel and the final dk goes to dqkv's k columns.
// status points at two device words: the status word and, after it, a counter
// the kernel schedules its work units with (reset here before the launch).
// L2row is the forward's lse in the negated, base-2, score-scale-folded form
// that attn_rowdot writes next to Drow when given lse. rope_cos / rope_sin
// are the angle-major tables [16][T][4] (as in GemmArgs).
cudaError_t attn_bwd_tc(const bf16* qkv, const bf16* dout, const float* L2row, const float* Drow, float* dq,
                        float* dk, bf16* dqkv, int B, int T, int H, int* status, cudaStream_t s,
                        const float* rqk = nullptr, const float* rope_cos = nullptr,
                        const float* rope_sin = nullptr);

// out = *in * scale (one device float).
cudaError_t scale_scalar(const float* in, float scale, float* out, cudaStream_t s);
// Packed uint16 token rows [B, T+1] -> int32 inputs tok [B, T] (ids 0..T-1 of
// each row) and targets tgt [B, T] (ids 1..T).
cudaError_t unpack_u16(const uint16_t* packed, int B, int T_, int32_t* tok, int32_t* tgt, cudaStream_t s);

// ------------------------------------------------------------------ loss
// part (16 bytes x kCeMaxSegments per row) and counter (a device int at 0)
// may be null; given, rows are split over more CTAs when there are few of them
constexpr int kCeMaxSegments = 512;
cudaError_t ce_rows_from_logits(const float* logits, const int* tgt, float* lse, float* nll, int* amax, int M, int V,
                                int* status, cudaStream_t s, float* part = nullptr, int* counter = nullptr,
                                int sms = 148);
// rows whose target is negative (masked) get nll 0
cudaError_t ce_reduce_partials(const float* p_max, const float* p_sum, const int* p_arg,
                               const float* p_tgt, const int* tgt, int n_tiles, float* lse, float* nll,
                               int* amax, int M, cudaStream_t s);
// loss = mean of nll over unmasked rows (tgt >= 0), inv_count = 1/their number (0 if none);
// nll, loss and inv_count may be null
cudaError_t mean_loss(const float* nll, const int* tgt, int M, float* loss, float* inv_count, cudaStream_t s);
// status DEV_BAD_TOKEN unless lo <= id < V for every id
cudaError_t check_ids(const int* ids, int n, int lo, int V, int* status, cudaStream_t s);

// ------------------------------------------------------------------ generation (KV cache)
// cache layout per layer: K and V each [B][H][max_len][128] (elem)
template <typename T>
cudaError_t kv_from_qkv(const T* qkv, T* K, T* Vc, int B, int Tn, int H, int max_len, cudaStream_t s);
// Decode attention of one layer: from qkv fp32 [B, 3d] of the step's token,
// k_hat and v go into the cache at pos and o elem [B, d] = attention of q_hat
// over cached positions 0..pos. The position is pos, or *d_pos when d_pos is
// not null (graph-replayable launches); one outside [0, max_len) sets
// DEV_BAD_TOKEN and writes nothing. part holds B*H*ceil(span/chunk) partials
// of 132 floats (span = max_len with d_pos, else pos + 1); cnt holds B*H ints
// that must be 0 before the first call (each call leaves them at 0).
constexpr int kDecodeChunk = 256;
constexpr int kDecodePartFloats = 132;
template <typename T>
cudaError_t attn_decode(const float* qkv, const float* rc, const float* rs, T* K, T* Vc, float* part, int* cnt, T* out,
                        int B, int H, int pos, const int* d_pos, int max_len, int chunk, int* status, cudaStream_t s);
// *d_pos += 1 (one thread)
cudaError_t advance_pos(int* d_pos, cudaStream_t s);
template <typename T>
cudaError_t relu2_rows(const float* u, T* a, long long n, cudaStream_t s);
template <typename T>
cudaError_t gather_last(const T* hf, T* out, int B, int Tn, int d, cudaStream_t s);

// ------------------------------------------------------------------ optimizer
// Chunk of the Muon passes (every block matrix holds a whole number of them:
// d^2 is a multiple of 16384 when d is a multiple of 128) and the fixed block
// count of the gradient-norm reduction.
constexpr int kMuonChunk = 8192;
constexpr int kNormBlocks = 1184;
// stats[0] = ||g||_2 over n fp32 gradients, stats[1] = min(1, max_norm / (norm + 1e-6));
// part = kNormBlocks fp64 partials. stats_out (may be null) gets a copy.
cudaError_t grad_norm(const float* g, long long n, float max_norm, double* part, float* stats, float* stats_out,
                      cudaStream_t s);
// AdamW on two segments of seg elements each: parameter offsets [0, seg) and [off2, off2 + seg)
template <typename T>
cudaError_t adamw_update(float* master, T* param, const float* grad, float* m, float* v, long long seg, long long off2,
                         const float* stats, float lr, float b1, float b2, float eps, float wd, float inv_bc1,
                         float inv_bc2, cudaStream_t s);
// buf <- mu buf + k g over n block-matrix elements; part[chunk] = sum of u^2, u = k g + mu buf
cudaError_t muon_momentum(const float* grad, float* buf, long long n, const float* stats, float mu, double* part,
                          cudaStream_t s);
// per-matrix 1/(||u||+1e-7), then X[kind][l] = u * inv (stacked per kind: w_qkv, w_o, w_fc, w_proj)
template <typename T>
cudaError_t muon_normalize(const float* grad, const float* buf, const float* stats, float mu, const double* part,
                           float* inv_norm, int L, int d, T* X, cudaStream_t s);
// master <- master*decay - step*X ; param <- master, for one kind's stack [L, msize]
template <typename T>
cudaError_t muon_apply(float* master, T* param, const T* X, int L, long long msize, long long layer, long long pre,
                       float decay, float step, cudaStream_t s);
template <typename T>
cudaError_t upcast(const T* p, float* master, long long n, cudaStream_t s);

}  // namespace nc
