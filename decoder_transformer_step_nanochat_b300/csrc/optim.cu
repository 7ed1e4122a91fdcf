// Element-wise and reduction kernels of the optimizer step (the matrix work
// of Muon, the Newton-Schulz iterations, runs on the batched GEMM):
//
//   grad_sumsq   global L2 norm of every gradient, in a fixed summation order
//                (per-block fp64 partials over fixed ranges, one block sums them)
//   adamw        AdamW with decoupled weight decay on wte and lm_head
//   muon_*       Nesterov momentum, per-matrix Frobenius normalisation into the
//                Newton-Schulz buffer, and the final scaled update
//
// The pages (nanochat explainer, "The Full Pipeline" / "Pretraining"; the
// topaiproduct article, "What the Community Is Saying") name Muon for the
// block matrices, AdamW for the embedding and unembedding, clipping at 1.0
// and weight decay 0.1. All passes stream fp32 state with 16-byte accesses:
// they are bound by HBM bandwidth. The optimizer keeps fp32 master weights;
// the parameters the step reads are written as their rounded image.
#include "ops.cuh"

namespace nc {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ double block_sum_d(double v, double* sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x / 32, l = threadIdx.x & 31;
  if (l == 0) sh[w] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kThreads / 32; ++i) t += sh[i];  // fixed order
  __syncthreads();
  return t;
}

__device__ __forceinline__ float sq4(float4 a) { return a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w; }

// Block b sums the squares of float4 indices [b*per, min(n4, (b+1)*per)):
// runs of 16 float4 per thread in fp32, folded into an fp64 sum.
__global__ void __launch_bounds__(kThreads) grad_sumsq_k(const float4* __restrict__ g, long long n4, long long per,
                                                         double* __restrict__ part) {
  __shared__ double sh[kThreads / 32];
  const long long b0 = (long long)blockIdx.x * per;
  const long long b1 = min(n4, b0 + per);
  double acc = 0.0;
  for (long long i0 = b0 + threadIdx.x; i0 < b1; i0 += 16LL * kThreads) {
    float s = 0.f;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
      const long long i = i0 + (long long)j * kThreads;
      if (i < b1) s += sq4(__ldcs(g + i));
    }
    acc += (double)s;
  }
  const double t = block_sum_d(acc, sh);
  if (threadIdx.x == 0) part[blockIdx.x] = t;
}

// One block: sum of the partials in a fixed order, norm and clip factor.
__global__ void __launch_bounds__(kThreads) grad_norm_finish_k(const double* __restrict__ part, int n, float max_norm,
                                                               float* __restrict__ stats, float* __restrict__ stats_out) {
  __shared__ double sh[kThreads / 32];
  double acc = 0.0;
  for (int i = threadIdx.x; i < n; i += kThreads) acc += part[i];
  const double t = block_sum_d(acc, sh);
  if (threadIdx.x == 0) {
    const double norm = sqrt(t);
    const double k = fmin(1.0, (double)max_norm / (norm + 1e-6));
    stats[0] = (float)norm;
    stats[1] = (float)k;
    if (stats_out) {
      stats_out[0] = (float)norm;
      stats_out[1] = (float)k;
    }
  }
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<bf16>(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void adamw1(float g, float& m, float& v, float& p, float b1, float b2, float eps,
                                       float lr, float decay, float inv_bc1, float inv_bc2) {
  m = b1 * m + (1.f - b1) * g;
  v = b2 * v + (1.f - b2) * g * g;
  p = p * decay - lr * (m * inv_bc1) / (sqrtf(v * inv_bc2) + eps);
}

// AdamW over the two tables of the group: moment index i < seg covers wte
// (parameter offset i), i >= seg covers lm_head (parameter offset off2 + i - seg).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    adamw_k(float* __restrict__ master, T* __restrict__ param, const float* __restrict__ grad, float* __restrict__ mom1,
            float* __restrict__ mom2, long long seg4, long long off2, const float* __restrict__ stats, float lr, float b1,
            float b2, float eps, float wd, float inv_bc1, float inv_bc2) {
  const float k = stats[1];
  const float decay = 1.f - lr * wd;
  const long long n4 = 2 * seg4;
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < n4; i += (long long)gridDim.x * kThreads) {
    const long long po = 4 * ((i < seg4) ? i : off2 / 4 + (i - seg4));
    const float4 g4 = __ldcs(reinterpret_cast<const float4*>(grad + po));
    float4 m4 = reinterpret_cast<float4*>(mom1)[i];
    float4 v4 = reinterpret_cast<float4*>(mom2)[i];
    float4 p4 = *reinterpret_cast<float4*>(master + po);
    adamw1(g4.x * k, m4.x, v4.x, p4.x, b1, b2, eps, lr, decay, inv_bc1, inv_bc2);
    adamw1(g4.y * k, m4.y, v4.y, p4.y, b1, b2, eps, lr, decay, inv_bc1, inv_bc2);
    adamw1(g4.z * k, m4.z, v4.z, p4.z, b1, b2, eps, lr, decay, inv_bc1, inv_bc2);
    adamw1(g4.w * k, m4.w, v4.w, p4.w, b1, b2, eps, lr, decay, inv_bc1, inv_bc2);
    reinterpret_cast<float4*>(mom1)[i] = m4;
    reinterpret_cast<float4*>(mom2)[i] = v4;
    *reinterpret_cast<float4*>(master + po) = p4;
    store4<T>(param + po, p4);
  }
}

// Muon momentum over the block matrices (flat layout, chunks of kMuonChunk
// elements, each inside one matrix): buf <- mu buf + k g; the squares of the
// Nesterov direction u = k g + mu buf are summed per chunk.
__global__ void __launch_bounds__(kThreads)
    muon_momentum_k(const float* __restrict__ grad, float* __restrict__ buf, const float* __restrict__ stats, float mu,
                    double* __restrict__ part) {
  __shared__ double sh[kThreads / 32];
  const float k = stats[1];
  const long long base = (long long)blockIdx.x * kMuonChunk;
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kMuonChunk / (4 * kThreads); ++j) {
    const long long e = base + 4LL * (threadIdx.x + j * kThreads);
    const float4 g4 = __ldcs(reinterpret_cast<const float4*>(grad + e));
    float4 b4 = *reinterpret_cast<const float4*>(buf + e);
    b4.x = mu * b4.x + k * g4.x;
    b4.y = mu * b4.y + k * g4.y;
    b4.z = mu * b4.z + k * g4.z;
    b4.w = mu * b4.w + k * g4.w;
    *reinterpret_cast<float4*>(buf + e) = b4;
    const float4 u = make_float4(k * g4.x + mu * b4.x, k * g4.y + mu * b4.y, k * g4.z + mu * b4.z, k * g4.w + mu * b4.w);
    s += sq4(u);
  }
  const double t = block_sum_d((double)s, sh);
  if (threadIdx.x == 0) part[blockIdx.x] = t;
}

// Where chunk c of the block-matrix region lives: layer l, kind (0 w_qkv,
// 1 w_o, 2 w_fc, 3 w_proj) and its element offset inside the matrix. A layer
// is 12 d^2 elements: 3 d^2, d^2, 4 d^2, 4 d^2.
__device__ __forceinline__ void chunk_place(long long c, long long cpd2, int& l, int& kind, long long& inner) {
  const long long per_layer = 12 * cpd2;  // chunks per layer
  l = (int)(c / per_layer);
  long long r = c - l * per_layer;
  if (r < 3 * cpd2) kind = 0;
  else if (r < 4 * cpd2) kind = 1, r -= 3 * cpd2;
  else if (r < 8 * cpd2) kind = 2, r -= 4 * cpd2;
  else kind = 3, r -= 8 * cpd2;
  inner = r * kMuonChunk;
}

__device__ __forceinline__ long long kind_d2(int kind) { return kind == 0 ? 3 : (kind == 1 ? 1 : 4); }

// Per matrix (l, kind): fixed-order sum of its chunks' partials, then
// inv_norm = 1 / (||u||_F + 1e-7).
__global__ void __launch_bounds__(kThreads) muon_norms_k(const double* __restrict__ part, long long cpd2,
                                                         float* __restrict__ inv_norm) {
  __shared__ double sh[kThreads / 32];
  const int l = blockIdx.x / 4, kind = blockIdx.x % 4;
  const long long pre = kind == 0 ? 0 : (kind == 1 ? 3 : (kind == 2 ? 4 : 8));
  const long long c0 = l * 12 * cpd2 + pre * cpd2, n = kind_d2(kind) * cpd2;
  double acc = 0.0;
  for (long long i = threadIdx.x; i < n; i += kThreads) acc += part[c0 + i];
  const double t = block_sum_d(acc, sh);
  if (threadIdx.x == 0) inv_norm[blockIdx.x] = (float)(1.0 / (sqrt(t) + 1e-7));
}

// X (elem) = u * inv_norm, written per kind as stacked [L, rows, cols].
template <typename T>
__global__ void __launch_bounds__(kThreads)
    muon_normalize_k(const float* __restrict__ grad, const float* __restrict__ buf, const float* __restrict__ stats,
                     float mu, const float* __restrict__ inv_norm, long long cpd2, int L, T* __restrict__ X) {
  const float k = stats[1];
  int l, kind;
  long long inner;
  chunk_place(blockIdx.x, cpd2, l, kind, inner);
  const long long d2 = cpd2 * kMuonChunk;
  const long long kbase = (kind == 0 ? 0 : (kind == 1 ? 3 : (kind == 2 ? 4 : 8))) * d2 * L;  // kind's stack
  T* dst = X + kbase + (long long)l * kind_d2(kind) * d2 + inner;
  const float inv = inv_norm[l * 4 + kind];
  const long long base = (long long)blockIdx.x * kMuonChunk;
#pragma unroll
  for (int j = 0; j < kMuonChunk / (4 * kThreads); ++j) {
    const long long e = 4LL * (threadIdx.x + j * kThreads);
    const float4 g4 = __ldcs(reinterpret_cast<const float4*>(grad + base + e));
    const float4 b4 = *reinterpret_cast<const float4*>(buf + base + e);
    store4<T>(dst + e, make_float4((k * g4.x + mu * b4.x) * inv, (k * g4.y + mu * b4.y) * inv,
                                   (k * g4.z + mu * b4.z) * inv, (k * g4.w + mu * b4.w) * inv));
  }
}

// Final update of one kind: master <- master (1 - lr wd) - lr scale X, param
// <- rounded master. Chunk c covers elements [c*chunk, ...) of the kind's
// stack [L, msize]; the matrix of layer l sits at l*layer + pre in the
// block-matrix region.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    muon_apply_k(float* __restrict__ master, T* __restrict__ param, const T* __restrict__ X, long long msize,
                 long long layer, long long pre, float decay, float step) {
  const long long base = (long long)blockIdx.x * kMuonChunk;
  const long long l = base / msize, inner = base - l * msize;
  const long long po = l * layer + pre + inner;
#pragma unroll
  for (int j = 0; j < kMuonChunk / (4 * kThreads); ++j) {
    const long long e = 4LL * (threadIdx.x + j * kThreads);
    const float4 x4 = load4<T>(X + base + e);
    float4 p4 = *reinterpret_cast<const float4*>(master + po + e);
    p4.x = p4.x * decay - step * x4.x;
    p4.y = p4.y * decay - step * x4.y;
    p4.z = p4.z * decay - step * x4.z;
    p4.w = p4.w * decay - step * x4.w;
    *reinterpret_cast<float4*>(master + po + e) = p4;
    store4<T>(param + po + e, p4);
  }
}

// master (fp32) <- params (elem), the optimizer's starting point.
template <typename T>
__global__ void __launch_bounds__(kThreads) upcast_k(const T* __restrict__ p, float* __restrict__ master, long long n4) {
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < n4; i += (long long)gridDim.x * kThreads)
    reinterpret_cast<float4*>(master)[i] = load4<T>(p + 4 * i);
}

int grid_for(long long n4, int sms) {
  long long g = (n4 + kThreads - 1) / kThreads;
  const long long cap = 8LL * (sms > 0 ? sms : 148);
  return (int)(g < cap ? (g < 1 ? 1 : g) : cap);
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

cudaError_t grad_norm(const float* g, long long n, float max_norm, double* part, float* stats, float* stats_out,
                      cudaStream_t s) {
  const long long n4 = n / 4;
  const long long per = (n4 + kNormBlocks - 1) / kNormBlocks;
  grad_sumsq_k<<<kNormBlocks, kThreads, 0, s>>>(reinterpret_cast<const float4*>(g), n4, per, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  grad_norm_finish_k<<<1, kThreads, 0, s>>>(part, kNormBlocks, max_norm, stats, stats_out);
  return cudaGetLastError();
}

template <typename T>
cudaError_t adamw_update(float* master, T* param, const float* grad, float* m, float* v, long long seg, long long off2,
                         const float* stats, float lr, float b1, float b2, float eps, float wd, float inv_bc1,
                         float inv_bc2, cudaStream_t s) {
  const long long n4 = 2 * (seg / 4);
  adamw_k<T><<<grid_for(n4, num_sms()), kThreads, 0, s>>>(master, param, grad, m, v, seg / 4, off2, stats, lr, b1, b2,
                                                         eps, wd, inv_bc1, inv_bc2);
  return cudaGetLastError();
}

cudaError_t muon_momentum(const float* grad, float* buf, long long n, const float* stats, float mu, double* part,
                          cudaStream_t s) {
  const long long chunks = n / kMuonChunk;
  muon_momentum_k<<<(unsigned)chunks, kThreads, 0, s>>>(grad, buf, stats, mu, part);
  return cudaGetLastError();
}

template <typename T>
cudaError_t muon_normalize(const float* grad, const float* buf, const float* stats, float mu, const double* part,
                           float* inv_norm, int L, int d, T* X, cudaStream_t s) {
  const long long cpd2 = (long long)d * d / kMuonChunk;
  muon_norms_k<<<4 * L, kThreads, 0, s>>>(part, cpd2, inv_norm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  muon_normalize_k<T><<<(unsigned)(12LL * L * cpd2), kThreads, 0, s>>>(grad, buf, stats, mu, inv_norm, cpd2, L, X);
  return cudaGetLastError();
}

template <typename T>
cudaError_t muon_apply(float* master, T* param, const T* X, int L, long long msize, long long layer, long long pre,
                       float decay, float step, cudaStream_t s) {
  muon_apply_k<T><<<(unsigned)(L * msize / kMuonChunk), kThreads, 0, s>>>(master, param, X, msize, layer, pre, decay,
                                                                         step);
  return cudaGetLastError();
}

template <typename T>
cudaError_t upcast(const T* p, float* master, long long n, cudaStream_t s) {
  upcast_k<T><<<grid_for(n / 4, num_sms()), kThreads, 0, s>>>(p, master, n / 4);
  return cudaGetLastError();
}

template cudaError_t adamw_update<float>(float*, float*, const float*, float*, float*, long long, long long,
                                         const float*, float, float, float, float, float, float, float, cudaStream_t);
template cudaError_t adamw_update<bf16>(float*, bf16*, const float*, float*, float*, long long, long long,
                                        const float*, float, float, float, float, float, float, float, cudaStream_t);
template cudaError_t muon_normalize<float>(const float*, const float*, const float*, float, const double*, float*, int,
                                           int, float*, cudaStream_t);
template cudaError_t muon_normalize<bf16>(const float*, const float*, const float*, float, const double*, float*, int,
                                          int, bf16*, cudaStream_t);
template cudaError_t muon_apply<float>(float*, float*, const float*, int, long long, long long, long long, float,
                                       float, cudaStream_t);
template cudaError_t muon_apply<bf16>(float*, bf16*, const bf16*, int, long long, long long, long long, float, float,
                                      cudaStream_t);
template cudaError_t upcast<float>(const float*, float*, long long, cudaStream_t);
template cudaError_t upcast<bf16>(const bf16*, float*, long long, cudaStream_t);

}  // namespace nc
