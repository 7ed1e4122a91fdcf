// Kernels of generation with a KV cache (nanochat explainer, "Inference &
// KV Cache": prefill fills the cache with every layer's keys and values;
// decode then produces one token at a time, its query attending to the
// cached keys and values).
//
//   kv_from_qkv      prefill: copy k_hat and v of one layer's stash into the
//                    cache layout [B][H][max_len][128]
//   attn_decode      decode, one launch per layer: q_hat and k_hat of the
//                    step's token (per-head RMSNorm + RoPE at its position)
//                    from the fp32 qkv row, k_hat and v appended to the cache,
//                    then flash-decoding: each CTA scores one chunk of cached
//                    positions of one (sequence, head), and the last CTA of
//                    the (sequence, head) to finish merges the chunks
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

// RMSNorm over one head's 128 dims, then the rotation by the angles of
// position pos (first half x1 c - x2 s, second half x1 s + x2 c), on one warp:
// lane L holds dims 4L..4L+3 and the partner of dim j < 64, j + 64, sits in
// lane L ^ 16.
__device__ __forceinline__ float4 head_norm_rope(float4 v, const float* __restrict__ rc,
                                                 const float* __restrict__ rs, int pos, int lane) {
  float ss = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  ss = warp_sum(ss);
  const float r = rsqrtf(ss * (1.f / 128.f) + kEps);
  v.x *= r; v.y *= r; v.z *= r; v.w *= r;
  float4 w;
  w.x = __shfl_xor_sync(0xffffffffu, v.x, 16);
  w.y = __shfl_xor_sync(0xffffffffu, v.y, 16);
  w.z = __shfl_xor_sync(0xffffffffu, v.z, 16);
  w.w = __shfl_xor_sync(0xffffffffu, v.w, 16);
  const int j0 = (lane & 15) * 4;  // rotation pair index of .x
  const float4 c = ld4e(rc + (size_t)pos * 64 + j0);
  const float4 s = ld4e(rs + (size_t)pos * 64 + j0);
  float4 o;
  if (lane < 16) {
    o.x = v.x * c.x - w.x * s.x; o.y = v.y * c.y - w.y * s.y;
    o.z = v.z * c.z - w.z * s.z; o.w = v.w * c.w - w.w * s.w;
  } else {  // x1 is the partner
    o.x = w.x * s.x + v.x * c.x; o.y = w.y * s.y + v.y * c.y;
    o.z = w.z * s.z + v.z * c.z; o.w = w.w * s.w + v.w * c.w;
  }
  return o;
}

// the value as the cache element type holds it
__device__ __forceinline__ float4 as_elem(float4 v, const float*) { return v; }
__device__ __forceinline__ float4 as_elem(float4 v, const bf16*) {
  const float2 a = __bfloat1622float2(__floats2bfloat162_rn(v.x, v.y));
  const float2 b = __bfloat1622float2(__floats2bfloat162_rn(v.z, v.w));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 ld4cg(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 ld4cg(const bf16* p) {
  const uint2 u = __ldcg(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

constexpr int kDecWarps = 4;

// Attention of the step's token for one (sequence b, head h) over one chunk
// of cached positions [c*chunk, min(c*chunk + chunk, pos + 1)), from the fp32
// qkv row of the token:
//  - every warp forms q_hat = RoPE(RMSNorm(q)) of the head (rounded to the
//    cache element type, as the prefill's attention reads it);
//  - the CTA of the chunk holding pos first appends k_hat and v of the token
//    to the cache at pos (warps 0 and 1), so it reads them back like any
//    other position;
//  - each warp walks a quarter of the chunk, four positions at a time, with
//    an online softmax in the log2 domain; the warps merge through shared
//    memory into the chunk's (max, sum, o[128]);
//  - with one chunk the CTA writes o; otherwise it leaves its partial in part
//    and the CTA that counts itself last for this (b, h) on cnt[b H + h]
//    merges the chunks in chunk order (so the result does not depend on
//    scheduling), writes o and sets the counter back to 0.
// A position outside [0, max_len) sets DEV_BAD_TOKEN and touches nothing.
// The cache is read through L2 only (ld.global.cg): this launch writes it.
template <typename T>
__global__ void __launch_bounds__(32 * kDecWarps)
    attn_decode_k(const float* __restrict__ qkv, const float* __restrict__ rc, const float* __restrict__ rs, T* K,
                  T* Vc, float* part, int* cnt, T* __restrict__ out, int H, int pos_arg, const int* __restrict__ d_pos,
                  int max_len, int chunk, int nchunks, int* status) {
  __shared__ float sm_m[kDecWarps], sm_l[kDecWarps];
  __shared__ float sm_o[kDecWarps][128];
  __shared__ int is_last;
  const int bh = blockIdx.x, c = blockIdx.y;
  const int pos = d_pos ? *d_pos : pos_arg;
  if (pos < 0 || pos >= max_len) {
    if (bh == 0 && c == 0 && threadIdx.x == 0) set_status(status, DEV_BAD_TOKEN);
    return;
  }
  if (c * chunk > pos) return;  // a fixed grid (device position): chunks past pos are unused
  const int n_act = pos / chunk + 1;
  const int b = bh / H, h = bh % H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = H * 128;
  const float* qrow = qkv + (size_t)b * 3 * d + h * 128 + lane * 4;
  T* Kb = K + ((size_t)b * H + h) * max_len * 128 + lane * 4;
  T* Vb = Vc + ((size_t)b * H + h) * max_len * 128 + lane * 4;
  const int t0 = c * chunk, t1 = min(t0 + chunk, pos + 1);
  {
    // the cache rows of this warp's first two rounds start towards L2 while
    // q_hat (and, in the last chunk, k_hat and v) are formed: one line per lane
    const int t = t0 + warp * 4 + (lane & 3) + ((lane >> 4) & 1) * 4 * kDecWarps;
    const size_t off = (size_t)t * 128 * sizeof(T) + ((lane >> 2) & 1) * 128;
    if (t < t1 && off < 128 * sizeof(T) * (size_t)(t + 1)) {
      const char* base = reinterpret_cast<const char*>((lane & 8) ? Vb - lane * 4 : Kb - lane * 4);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(base + off));
    }
  }
  if (c == n_act - 1) {  // this chunk holds pos: append the token's k_hat and v
    if (warp == 0) st4e(Kb + (size_t)pos * 128, head_norm_rope(ld4e(qrow + d), rc, rs, pos, lane));
    else if (warp == 1) st4e(Vb + (size_t)pos * 128, ld4e(qrow + 2 * d));
    __syncthreads();
  }
  const float sc = kLog2eD * rsqrtf(128.f);
  float4 q = as_elem(head_norm_rope(ld4e(qrow), rc, rs, pos, lane), static_cast<const T*>(nullptr));
  q.x *= sc; q.y *= sc; q.z *= sc; q.w *= sc;
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
        const float4 k = ld4cg(Kb + (size_t)t * 128);
        v4[u] = ld4cg(Vb + (size_t)t * 128);
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
  T* orow = out + (size_t)b * d + h * 128 + lane * 4;
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
    if (n_act == 1) {
      const float inv = 1.f / L;
      st4e(orow, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
    } else {
      float* pp = part + ((size_t)bh * nchunks + c) * kPart;
      if (lane == 0) {
        pp[0] = M;
        pp[1] = L;
      }
      st4e(pp + 4 + lane * 4, O);
      __threadfence();
      __syncwarp();
      if (lane == 0) is_last = atomicAdd(cnt + bh, 1) == n_act - 1;
      __syncwarp();
      if (is_last) {  // every chunk's partial is in part: merge them in chunk order
        __threadfence();
        const float* pb = part + (size_t)bh * nchunks * kPart;
        float Mx = -INFINITY;
        for (int k = 0; k < n_act; ++k) Mx = fmaxf(Mx, __ldcg(pb + (size_t)k * kPart));
        float Lt = 0.f;
        float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < n_act; ++k) {
          const float mk = __ldcg(pb + (size_t)k * kPart);
          const float f = mk == -INFINITY ? 0.f : exp2f(mk - Mx);
          Lt += f * __ldcg(pb + (size_t)k * kPart + 1);
          const float4 ok = ld4cg(pb + (size_t)k * kPart + 4 + lane * 4);
          Ot.x += f * ok.x; Ot.y += f * ok.y; Ot.z += f * ok.z; Ot.w += f * ok.w;
        }
        const float inv = 1.f / Lt;
        st4e(orow, make_float4(Ot.x * inv, Ot.y * inv, Ot.z * inv, Ot.w * inv));
        if (lane == 0) cnt[bh] = 0;
      }
    }
  }
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
cudaError_t attn_decode(const float* qkv, const float* rc, const float* rs, T* K, T* Vc, float* part, int* cnt, T* out,
                        int B, int H, int pos, const int* d_pos, int max_len, int chunk, int* status, cudaStream_t s) {
  // with a device position the grid covers max_len (a graph replays it at any position)
  const int span = d_pos ? max_len : pos + 1;
  const int nchunks = (span + chunk - 1) / chunk;
  attn_decode_k<T><<<dim3(B * H, nchunks), 32 * kDecWarps, 0, s>>>(qkv, rc, rs, K, Vc, part, cnt, out, H, pos, d_pos,
                                                                   max_len, chunk, nchunks, status);
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
  template cudaError_t attn_decode<T>(const float*, const float*, const float*, T*, T*, float*, int*, T*, int, \
                                      int, int, const int*, int, int, int*, cudaStream_t);                     \
  template cudaError_t relu2_rows<T>(const float*, T*, long long, cudaStream_t);                               \
  template cudaError_t gather_last<T>(const T*, T*, int, int, int, cudaStream_t);
NC_DEC_INST(float)
NC_DEC_INST(bf16)
#undef NC_DEC_INST

}  // namespace nc
