// Causal multi-head attention with plain fp32 FMA (fp32 debug mode).
//
// Forward: flash-style online softmax over 32-key tiles staged in shared
// memory; one warp per query row, lane L scores key kb+L and owns output
// dims L, L+32, L+64, L+96. Backward: the two-kernel split of the
// flash-attention backward (dq by query rows, dk/dv by key rows), softmax
// probabilities recomputed from the forward's logsumexp, no atomics.
//
// qkv is [B*T, 3d] holding q_hat (QK-normed and rotated), k_hat, v; o is
// [B*T, d]; lse and D are [B, H, T]; scale is 1/sqrt(128). The backward
// writes dq_hat and dk_hat as two fp32 [B*T, d] planes of dqk.
#include "ops.cuh"

namespace nc {

namespace {

constexpr int kRows = 8;   // query (or key) rows per CTA, one per warp
constexpr int kTile = 32;  // keys (or queries) per shared-memory tile

template <typename T>
__global__ void __launch_bounds__(256) attn_fwd_simt_k(const T* __restrict__ qkv, T* __restrict__ o,
                                                       float* __restrict__ lse, int Tlen, int H) {
  __shared__ float Qs[kRows][kHeadDim];
  __shared__ float Ks[kTile][kHeadDim + 1];
  __shared__ float Vs[kTile][kHeadDim];
  int w = threadIdx.x / 32, lane = threadIdx.x & 31;
  int h = blockIdx.y, b = blockIdx.z;
  int t0 = blockIdx.x * kRows, t = t0 + w;
  int d = H * kHeadDim;
  size_t ld = 3 * (size_t)d;
  const T* base = qkv + (size_t)b * Tlen * ld;
  for (int i = threadIdx.x; i < kRows * kHeadDim; i += 256) {
    int r = i / kHeadDim, e = i % kHeadDim, tt = t0 + r;
    Qs[r][e] = tt < Tlen ? ldf(base + tt * ld + h * kHeadDim + e) : 0.f;
  }
  const float scale = rsqrtf((float)kHeadDim);
  float m_i = -INFINITY, l_i = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  int kend = min(Tlen, t0 + kRows);
  for (int kb = 0; kb < kend; kb += kTile) {
    __syncthreads();
    for (int i = threadIdx.x; i < kTile * kHeadDim; i += 256) {
      int r = i / kHeadDim, e = i % kHeadDim, j = kb + r;
      Ks[r][e] = j < Tlen ? ldf(base + j * ld + d + h * kHeadDim + e) : 0.f;
      Vs[r][e] = j < Tlen ? ldf(base + j * ld + 2 * d + h * kHeadDim + e) : 0.f;
    }
    __syncthreads();
    if (t < Tlen) {
      int j = kb + lane;
      float s = -INFINITY;
      if (j <= t) {
        float a = 0.f;
#pragma unroll 16
        for (int e = 0; e < kHeadDim; ++e) a = fmaf(Qs[w][e], Ks[lane][e], a);
        s = a * scale;
      }
      float m_new = fmaxf(m_i, warp_max(s));
      float p = (j <= t) ? expf(s - m_new) : 0.f;
      float alpha = expf(m_i - m_new);
      l_i = l_i * alpha + warp_sum(p);
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] *= alpha;
      for (int jj = 0; jj < kTile; ++jj) {
        float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = fmaf(pj, Vs[jj][lane + 32 * c], acc[c]);
      }
      m_i = m_new;
    }
  }
  if (t < Tlen) {
    T* orow = o + ((size_t)b * Tlen + t) * d + h * kHeadDim;
    float inv = 1.f / l_i;
#pragma unroll
    for (int c = 0; c < 4; ++c) stf(orow + lane + 32 * c, acc[c] * inv);
    if (lane == 0) lse[((size_t)b * H + h) * Tlen + t] = m_i + logf(l_i);
  }
}

// dq_hat[t] = scale * sum_{j<=t} p_tj (dp_tj - D_t) k_j, p recomputed from lse.
template <typename T>
__global__ void __launch_bounds__(256) attn_bwd_dq_simt_k(const T* __restrict__ qkv, const T* __restrict__ dout,
                                                          const float* __restrict__ lse,
                                                          const float* __restrict__ Drow,
                                                          float* __restrict__ dqk, int Tlen, int H) {
  __shared__ float Qs[kRows][kHeadDim];
  __shared__ float Gs[kRows][kHeadDim];
  __shared__ float Ks[kTile][kHeadDim + 1];
  __shared__ float Vs[kTile][kHeadDim + 1];
  int w = threadIdx.x / 32, lane = threadIdx.x & 31;
  int h = blockIdx.y, b = blockIdx.z;
  int t0 = blockIdx.x * kRows, t = t0 + w;
  int d = H * kHeadDim;
  size_t ld = 3 * (size_t)d;
  const T* base = qkv + (size_t)b * Tlen * ld;
  const T* gbase = dout + (size_t)b * Tlen * d;
  for (int i = threadIdx.x; i < kRows * kHeadDim; i += 256) {
    int r = i / kHeadDim, e = i % kHeadDim, tt = t0 + r;
    Qs[r][e] = tt < Tlen ? ldf(base + tt * ld + h * kHeadDim + e) : 0.f;
    Gs[r][e] = tt < Tlen ? ldf(gbase + (size_t)tt * d + h * kHeadDim + e) : 0.f;
  }
  const float scale = rsqrtf((float)kHeadDim);
  size_t bh = ((size_t)b * H + h) * Tlen;
  float L = t < Tlen ? lse[bh + t] : 0.f;
  float Dt = t < Tlen ? Drow[bh + t] : 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  int kend = min(Tlen, t0 + kRows);
  for (int kb = 0; kb < kend; kb += kTile) {
    __syncthreads();
    for (int i = threadIdx.x; i < kTile * kHeadDim; i += 256) {
      int r = i / kHeadDim, e = i % kHeadDim, j = kb + r;
      Ks[r][e] = j < Tlen ? ldf(base + j * ld + d + h * kHeadDim + e) : 0.f;
      Vs[r][e] = j < Tlen ? ldf(base + j * ld + 2 * d + h * kHeadDim + e) : 0.f;
    }
    __syncthreads();
    if (t < Tlen) {
      int j = kb + lane;
      float ds = 0.f;
      if (j <= t) {
        float a = 0.f, dp = 0.f;
#pragma unroll 16
        for (int e = 0; e < kHeadDim; ++e) {
          a = fmaf(Qs[w][e], Ks[lane][e], a);
          dp = fmaf(Gs[w][e], Vs[lane][e], dp);
        }
        float p = expf(a * scale - L);
        ds = p * (dp - Dt);
      }
      for (int jj = 0; jj < kTile; ++jj) {
        float dj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = fmaf(dj, Ks[jj][lane + 32 * c], acc[c]);
      }
    }
  }
  if (t < Tlen) {
    float* row = dqk + ((size_t)b * Tlen + t) * d + h * kHeadDim;  // dq_hat plane
#pragma unroll
    for (int c = 0; c < 4; ++c) row[lane + 32 * c] = acc[c] * scale;
  }
}

// dv[j] = sum_{i>=j} p_ij do_i ; dk_hat[j] = scale * sum_{i>=j} p_ij (dp_ij - D_i) q_i.
template <typename T>
__global__ void __launch_bounds__(256) attn_bwd_dkv_simt_k(const T* __restrict__ qkv, const T* __restrict__ dout,
                                                           const float* __restrict__ lse,
                                                           const float* __restrict__ Drow,
                                                           float* __restrict__ dqk, T* __restrict__ dqkv,
                                                           int Tlen, int H) {
  __shared__ float Ks[kRows][kHeadDim];
  __shared__ float Vs[kRows][kHeadDim];
  __shared__ float Qs[kTile][kHeadDim + 1];
  __shared__ float Gs[kTile][kHeadDim + 1];
  __shared__ float Ls[kTile], Ds[kTile];
  int w = threadIdx.x / 32, lane = threadIdx.x & 31;
  int h = blockIdx.y, b = blockIdx.z;
  int j0 = blockIdx.x * kRows, j = j0 + w;
  int d = H * kHeadDim;
  size_t ld = 3 * (size_t)d;
  const T* base = qkv + (size_t)b * Tlen * ld;
  const T* gbase = dout + (size_t)b * Tlen * d;
  for (int i = threadIdx.x; i < kRows * kHeadDim; i += 256) {
    int r = i / kHeadDim, e = i % kHeadDim, jj = j0 + r;
    Ks[r][e] = jj < Tlen ? ldf(base + jj * ld + d + h * kHeadDim + e) : 0.f;
    Vs[r][e] = jj < Tlen ? ldf(base + jj * ld + 2 * d + h * kHeadDim + e) : 0.f;
  }
  const float scale = rsqrtf((float)kHeadDim);
  size_t bh = ((size_t)b * H + h) * Tlen;
  float dk[4] = {0.f, 0.f, 0.f, 0.f}, dv[4] = {0.f, 0.f, 0.f, 0.f};
  for (int qb = (j0 / kTile) * kTile; qb < Tlen; qb += kTile) {
    __syncthreads();
    for (int i = threadIdx.x; i < kTile * kHeadDim; i += 256) {
      int r = i / kHeadDim, e = i % kHeadDim, ii = qb + r;
      Qs[r][e] = ii < Tlen ? ldf(base + ii * ld + h * kHeadDim + e) : 0.f;
      Gs[r][e] = ii < Tlen ? ldf(gbase + (size_t)ii * d + h * kHeadDim + e) : 0.f;
    }
    if (threadIdx.x < kTile) {
      int ii = qb + threadIdx.x;
      Ls[threadIdx.x] = ii < Tlen ? lse[bh + ii] : 0.f;
      Ds[threadIdx.x] = ii < Tlen ? Drow[bh + ii] : 0.f;
    }
    __syncthreads();
    if (j < Tlen) {
      int i = qb + lane;
      float p = 0.f, ds = 0.f;
      if (i >= j && i < Tlen) {
        float a = 0.f, dp = 0.f;
#pragma unroll 16
        for (int e = 0; e < kHeadDim; ++e) {
          a = fmaf(Qs[lane][e], Ks[w][e], a);
          dp = fmaf(Gs[lane][e], Vs[w][e], dp);
        }
        p = expf(a * scale - Ls[lane]);
        ds = p * (dp - Ds[lane]);
      }
      for (int ii = 0; ii < kTile; ++ii) {
        float pi = __shfl_sync(0xffffffffu, p, ii);
        float di = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          dv[c] = fmaf(pi, Gs[ii][lane + 32 * c], dv[c]);
          dk[c] = fmaf(di, Qs[ii][lane + 32 * c], dk[c]);
        }
      }
    }
  }
  if (j < Tlen) {
    size_t m = (size_t)b * Tlen + j;
    float* krow = dqk + (size_t)gridDim.z * Tlen * d + m * d + h * kHeadDim;  // dk_hat plane
    T* vrow = dqkv + m * 3 * d + 2 * d + h * kHeadDim;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      krow[lane + 32 * c] = dk[c] * scale;
      stf(vrow + lane + 32 * c, dv[c]);
    }
  }
}

}  // namespace

template <typename T>
cudaError_t attn_fwd_simt(const T* qkv, T* o, float* lse, int B, int T_, int H, cudaStream_t s) {
  if (B * T_ == 0) return cudaSuccess;
  dim3 grid((T_ + kRows - 1) / kRows, H, B);
  attn_fwd_simt_k<T><<<grid, 256, 0, s>>>(qkv, o, lse, T_, H);
  return cudaGetLastError();
}

template <typename T>
cudaError_t attn_bwd_simt(const T* qkv, const T* dout, const float* lse, const float* Drow,
                          float* dqk, T* dqkv, int B, int T_, int H, cudaStream_t s) {
  if (B * T_ == 0) return cudaSuccess;
  dim3 grid((T_ + kRows - 1) / kRows, H, B);
  attn_bwd_dq_simt_k<T><<<grid, 256, 0, s>>>(qkv, dout, lse, Drow, dqk, T_, H);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dkv_simt_k<T><<<grid, 256, 0, s>>>(qkv, dout, lse, Drow, dqk, dqkv, T_, H);
  return cudaGetLastError();
}

template cudaError_t attn_fwd_simt<float>(const float*, float*, float*, int, int, int, cudaStream_t);
template cudaError_t attn_fwd_simt<bf16>(const bf16*, bf16*, float*, int, int, int, cudaStream_t);
template cudaError_t attn_bwd_simt<float>(const float*, const float*, const float*, const float*,
                                          float*, float*, int, int, int, cudaStream_t);
template cudaError_t attn_bwd_simt<bf16>(const bf16*, const bf16*, const float*, const float*,
                                         float*, bf16*, int, int, int, cudaStream_t);

}  // namespace nc
