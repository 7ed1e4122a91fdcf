// Kernels of generation with a KV cache (nanochat explainer, "Inference &
// KV Cache": prefill fills the cache with every layer's keys and values;
// decode then produces one token at a time, its query attending to the
// cached keys and values).
//
//   kv_from_qkv      prefill: copy k_hat and v of one layer's stash into the
//                    cache layout [B][H][max_len][128]
//   decode_qkv       decode: per-head RMSNorm + RoPE of q and k at the step's
//                    position; q_hat out, k_hat and v appended to the cache
//   attn_decode      flash-decoding: each CTA scores one chunk of cached
//                    positions of one (sequence, head) and leaves a partial
//                    (max, sum, o); attn_decode_combine merges the chunks
//   relu2_rows       a = max(u, 0)^2 from the fp32 up-projection
//   gather_last      prefill: the last position's hidden row of each sequence
//
// Decode is bound by HBM bandwidth: the weights and the cached keys/values
// are read once per step; every kernel here streams with 8- or 16-byte
// accesses.
#include "ops.cuh"

namespace nc {

namespace {

constexpr float kLog2eD = 1.4426950408889634f;
// a chunk partial: m, l, two pad words, o[128] (o starts 16-byte aligned)
constexpr int kPart = 132;

__device__ __forceinline__ float4 ld4e(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4e(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4e(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4e(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// one thread per 4 elements of a (row m, head h, k-or-v) 128-element slice
template <typename T>
__global__ void kv_from_qkv_k(const T* __restrict__ qkv, T* __restrict__ K, T* __restrict__ Vc, int B, int Tn, int H,
                              int max_len) {
  const int d = H * 128;
  const long long total = (long long)B * Tn * H * 2 * 32;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int c4 = (int)(i & 31);
    long long r = i >> 5;
    const int kv = (int)(r & 1);
    r >>= 1;
    const int h = (int)(r % H);
    const long long m = r / H;
    const int b = (int)(m / Tn), t = (int)(m % Tn);
    const T* src = qkv + m * 3 * d + (1 + kv) * d + h * 128 + c4 * 4;
    T* dst = (kv ? Vc : K) + (((long long)b * H + h) * max_len + t) * 128 + c4 * 4;
    st4e(dst, ld4e(src));
  }
}

// One warp per (sequence b, head h, kind): kind 0 = q, 1 = k (normed and
// rotated at position pos), 2 = v. Lane L holds dims 4L..4L+3; the RoPE
// partner of dim j < 64 is j + 64, held by lane L ^ 16.
template <typename T>
__global__ void decode_qkv_k(const float* __restrict__ qkv, T* __restrict__ qh, T* __restrict__ K, T* __restrict__ Vc,
                             const float* __restrict__ rc, const float* __restrict__ rs, int B, int H, int pos_arg,
                             const int* __restrict__ d_pos, int max_len, int* status) {
  const int pos = d_pos ? *d_pos : pos_arg;
  if (pos < 0 || pos >= max_len) {  // a device position past the cache: report, touch nothing
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, DEV_BAD_TOKEN);
    return;
  }
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= B * H * 3) return;
  const int kind = wid % 3, bh = wid / 3, b = bh / H, h = bh % H;
  const int d = H * 128;
  float4 v = ld4e(qkv + (size_t)b * 3 * d + kind * d + h * 128 + lane * 4);
  const size_t cache_row = (((size_t)b * H + h) * max_len + pos) * 128 + lane * 4;
  if (kind == 2) {
    st4e(Vc + cache_row, v);
    return;
  }
  float ss = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  ss = warp_sum(ss);
  const float r = rsqrtf(ss * (1.f / 128.f) + kEps);
  v.x *= r; v.y *= r; v.z *= r; v.w *= r;
  // partner values (dims j +- 64)
  float4 w;
  w.x = __shfl_xor_sync(0xffffffffu, v.x, 16);
  w.y = __shfl_xor_sync(0xffffffffu, v.y, 16);
  w.z = __shfl_xor_sync(0xffffffffu, v.z, 16);
  w.w = __shfl_xor_sync(0xffffffffu, v.w, 16);
  const int j0 = (lane & 15) * 4;  // rotation pair index of .x
  const float4 c = ld4e(rc + (size_t)pos * 64 + j0);
  const float4 s = ld4e(rs + (size_t)pos * 64 + j0);
  float4 o;
  if (lane < 16) {  // first half: x1 c - x2 s
    o.x = v.x * c.x - w.x * s.x; o.y = v.y * c.y - w.y * s.y;
    o.z = v.z * c.z - w.z * s.z; o.w = v.w * c.w - w.w * s.w;
  } else {          // second half: x1 s + x2 c (x1 is the partner)
    o.x = w.x * s.x + v.x * c.x; o.y = w.y * s.y + v.y * c.y;
    o.z = w.z * s.z + v.z * c.z; o.w = w.w * s.w + v.w * c.w;
  }
  if (kind == 0) st4e(qh + (size_t)b * d + h * 128 + lane * 4, o);
  else st4e(K + cache_row, o);
}

constexpr int kDecWarps = 4;

// Partial attention of one chunk of cached positions [c*chunk, min(...,
// pos + 1)) for one (b, h): each warp walks a quarter of the chunk, four
// positions at a time, keeping an online softmax in the log2 domain; the
// warps then merge through shared memory. Partial = (m, l, -, -, o[128]).
template <typename T>
__global__ void __launch_bounds__(32 * kDecWarps)
    attn_decode_k(const T* __restrict__ qh, const T* __restrict__ K, const T* __restrict__ Vc,
                  float* __restrict__ part, int H, int pos_arg, const int* __restrict__ d_pos, int max_len, int chunk,
                  int nchunks) {
  __shared__ float sm_m[kDecWarps], sm_l[kDecWarps];
  __shared__ float sm_o[kDecWarps][128];
  const int bh = blockIdx.x, c = blockIdx.y;
  const int pos = d_pos ? *d_pos : pos_arg;
  if (pos < 0 || pos >= max_len) return;  // reported by decode_qkv
  if (c * chunk > pos) return;  // a fixed grid (device position): chunks past pos are unused
  const int b = bh / H, h = bh % H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = H * 128;
  const int t0 = c * chunk, t1 = min(t0 + chunk, pos + 1);
  const float sc = kLog2eD * rsqrtf(128.f);
  float4 q = ld4e(qh + (size_t)b * d + h * 128 + lane * 4);
  q.x *= sc; q.y *= sc; q.z *= sc; q.w *= sc;
  const T* Kb = K + ((size_t)b * H + h) * max_len * 128 + lane * 4;
  const T* Vb = Vc + ((size_t)b * H + h) * max_len * 128 + lane * 4;
  float m = -INFINITY, l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  // this warp's positions: t0 + warp*4 + 16*i + u, u in 0..3
  for (int tb = t0 + warp * 4; tb < t1; tb += 4 * kDecWarps) {
    float s4[4];
    float4 v4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tb + u;
      if (t < t1) {
        const float4 k = ld4e(Kb + (size_t)t * 128);
        v4[u] = ld4e(Vb + (size_t)t * 128);
        s4[u] = q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w;
      } else {
        v4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        s4[u] = 0.f;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int u = 0; u < 4; ++u) s4[u] += __shfl_xor_sync(0xffffffffu, s4[u], off);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (tb + u >= t1) s4[u] = -INFINITY;
    }
    const float mx = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
    const float m_new = fmaxf(m, mx);
    const float corr = exp2f(m - m_new);  // 0 while m = -inf
    l *= corr;
    o.x *= corr; o.y *= corr; o.z *= corr; o.w *= corr;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float pr = exp2f(s4[u] - m_new);
      l += pr;
      o.x += pr * v4[u].x; o.y += pr * v4[u].y; o.z += pr * v4[u].z; o.w += pr * v4[u].w;
    }
    m = m_new;
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  sm_o[warp][lane * 4 + 0] = o.x;
  sm_o[warp][lane * 4 + 1] = o.y;
  sm_o[warp][lane * 4 + 2] = o.z;
  sm_o[warp][lane * 4 + 3] = o.w;
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w]);
    float L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float f = sm_m[w] == -INFINITY ? 0.f : exp2f(sm_m[w] - M);
      L += f * sm_l[w];
      O.x += f * sm_o[w][lane * 4 + 0];
      O.y += f * sm_o[w][lane * 4 + 1];
      O.z += f * sm_o[w][lane * 4 + 2];
      O.w += f * sm_o[w][lane * 4 + 3];
    }
    float* pp = part + ((size_t)bh * nchunks + c) * kPart;
    if (lane == 0) {
      pp[0] = M;
      pp[1] = L;
    }
    st4e(pp + 4 + lane * 4, O);
  }
}

// One warp per (b, h): merge the chunk partials into o = sum_c w_c O_c / sum_c w_c L_c.
template <typename T>
__global__ void attn_decode_combine_k(const float* __restrict__ part, T* __restrict__ out, int BH, int H,
                                      int nchunks_grid, const int* __restrict__ d_pos, int chunk) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= BH) return;
  // partials are laid out with the grid's chunk count; only the chunks up to pos hold data
  const int pd = d_pos ? *d_pos : 0;
  const int nchunks = d_pos ? min(nchunks_grid, (max(pd, 0) + chunk) / chunk) : nchunks_grid;
  const int stride = nchunks_grid;
  const float* pp = part + (size_t)wid * stride * kPart;
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c) M = fmaxf(M, pp[(size_t)c * kPart]);
  float L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = 0; c < nchunks; ++c) {
    const float mc = pp[(size_t)c * kPart];
    const float f = mc == -INFINITY ? 0.f : exp2f(mc - M);
    L += f * pp[(size_t)c * kPart + 1];
    const float4 oc = ld4e(pp + (size_t)c * kPart + 4 + lane * 4);
    O.x += f * oc.x; O.y += f * oc.y; O.z += f * oc.z; O.w += f * oc.w;
  }
  const float inv = 1.f / L;
  const int b = wid / H, h = wid % H;
  st4e(out + (size_t)b * H * 128 + h * 128 + lane * 4, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
}

template <typename T>
__global__ void relu2_rows_k(const float* __restrict__ u, T* __restrict__ a, long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    float4 v = ld4e(u + 4 * i);
    v.x = fmaxf(v.x, 0.f); v.y = fmaxf(v.y, 0.f); v.z = fmaxf(v.z, 0.f); v.w = fmaxf(v.w, 0.f);
    st4e(a + 4 * i, make_float4(v.x * v.x, v.y * v.y, v.z * v.z, v.w * v.w));
  }
}

template <typename T>
__global__ void gather_last_k(const T* __restrict__ hf, T* __restrict__ out, int B, int Tn, int d) {
  const long long n4 = (long long)B * d / 4;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const long long e = 4 * i;
    const int b = (int)(e / d), c = (int)(e % d);
    st4e(out + e, ld4e(hf + ((size_t)b * Tn + Tn - 1) * d + c));
  }
}

inline int blocks_for(long long work, int per_block) {
  long long g = (work + per_block - 1) / per_block;
  if (g > 148LL * 32) g = 148LL * 32;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

template <typename T>
cudaError_t kv_from_qkv(const T* qkv, T* K, T* Vc, int B, int Tn, int H, int max_len, cudaStream_t s) {
  const long long total = (long long)B * Tn * H * 2 * 32;
  kv_from_qkv_k<T><<<blocks_for(total, 256), 256, 0, s>>>(qkv, K, Vc, B, Tn, H, max_len);
  return cudaGetLastError();
}

template <typename T>
cudaError_t decode_qkv(const float* qkv, T* qh, T* K, T* Vc, const float* rc, const float* rs, int B, int H, int pos,
                       const int* d_pos, int max_len, int* status, cudaStream_t s) {
  const int warps = B * H * 3;
  decode_qkv_k<T><<<(warps + 7) / 8, 256, 0, s>>>(qkv, qh, K, Vc, rc, rs, B, H, pos, d_pos, max_len, status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t attn_decode(const T* qh, const T* K, const T* Vc, float* part, T* out, int B, int H, int pos,
                        const int* d_pos, int max_len, int chunk, cudaStream_t s) {
  // with a device position the grid covers max_len (a graph replays it at any position)
  const int span = d_pos ? max_len : pos + 1;
  const int nchunks = (span + chunk - 1) / chunk;
  attn_decode_k<T><<<dim3(B * H, nchunks), 32 * kDecWarps, 0, s>>>(qh, K, Vc, part, H, pos, d_pos, max_len, chunk,
                                                                   nchunks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_decode_combine_k<T><<<(B * H + 7) / 8, 256, 0, s>>>(part, out, B * H, H, nchunks, d_pos, chunk);
  return cudaGetLastError();
}

namespace {
__global__ void advance_pos_k(int* d_pos) { *d_pos += 1; }
}  // namespace

cudaError_t advance_pos(int* d_pos, cudaStream_t s) {
  advance_pos_k<<<1, 1, 0, s>>>(d_pos);
  return cudaGetLastError();
}

template <typename T>
cudaError_t relu2_rows(const float* u, T* a, long long n, cudaStream_t s) {
  relu2_rows_k<T><<<blocks_for(n / 4, 256), 256, 0, s>>>(u, a, n / 4);
  return cudaGetLastError();
}

template <typename T>
cudaError_t gather_last(const T* hf, T* out, int B, int Tn, int d, cudaStream_t s) {
  gather_last_k<T><<<blocks_for((long long)B * d / 4, 256), 256, 0, s>>>(hf, out, B, Tn, d);
  return cudaGetLastError();
}

#define NC_DEC_INST(T)                                                                                         \
  template cudaError_t kv_from_qkv<T>(const T*, T*, T*, int, int, int, int, cudaStream_t);                   \
  template cudaError_t decode_qkv<T>(const float*, T*, T*, T*, const float*, const float*, int, int, int,     \
                                     const int*, int, int*, cudaStream_t);                                   \
  template cudaError_t attn_decode<T>(const T*, const T*, const T*, float*, T*, int, int, int, const int*, int, \
                                      int, cudaStream_t);                                                    \
  template cudaError_t relu2_rows<T>(const float*, T*, long long, cudaStream_t);                               \
  template cudaError_t gather_last<T>(const T*, T*, int, int, int, cudaStream_t);
NC_DEC_INST(float)
NC_DEC_INST(bf16)
#undef NC_DEC_INST

}  // namespace nc
