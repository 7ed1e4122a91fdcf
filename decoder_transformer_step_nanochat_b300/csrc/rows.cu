// Row-wise, memory-bound kernels of the step: embedding gather/scatter,
// parameter-free RMSNorm forward/backward, per-head QK-norm + RoPE forward
// and backward, softmax cross-entropy row reductions and the mean loss.
//
// One warp owns one row (or one 128-wide head row); lanes stride the row so
// every warp-wide access is coalesced, and reductions use warp shuffles.
#include "ops.cuh"

namespace nc {

namespace {

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const bf16* p) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld2(const bf16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st2(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void st2(bf16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

constexpr int kRowWarps = 8;  // warps per CTA in the one-warp-per-row kernels

// x[m,:] = wte[tok[m],:] (fp32 residual stream). The embedding is used as is:
// no scaling and no normalisation after the lookup.
template <typename T>
__global__ void embed_fwd_k(const int* __restrict__ tok, const T* __restrict__ wte,
                            float* __restrict__ x, int M, int d, int V, int* status) {
  int m = blockIdx.x * kRowWarps + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (m >= M) return;
  int id = tok[m];
  float* xr = x + (size_t)m * d;
  if (id < 0 || id >= V) {
    if (lane == 0) set_status(status, DEV_BAD_TOKEN);
    for (int c = lane * 4; c < d; c += 128) st4(xr + c, make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const T* wr = wte + (size_t)id * d;
  for (int c = lane * 4; c < d; c += 128) st4(xr + c, ld4(wr + c));
}

// dwte[tok[m],:] += dx[m,:]; dwte must be zeroed first. Rows of ids that no
// position holds stay exactly zero.
__global__ void embed_bwd_k(const int* __restrict__ tok, const float* __restrict__ dx,
                            float* __restrict__ dwte, int M, int d, int V) {
  int m = blockIdx.x * kRowWarps + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (m >= M) return;
  int id = tok[m];
  if (id < 0 || id >= V) return;
  const float* g = dx + (size_t)m * d;
  float* w = dwte + (size_t)id * d;
  for (int c = lane * 4; c < d; c += 128) {
    float4 v = ld4(g + c);
    atomicAdd(reinterpret_cast<float4*>(w + c), v);
  }
}

// Deterministic embedding gradient, dwte[id] += sum of dx[m] over the
// positions m holding id, in ascending m with a fixed grouping, so the
// result does not depend on scheduling (float atomics would add in arrival
// order). Three launches:
//  1. keys (id << mbits) | m, unique per position, sorted: chunks of 1024
//     positions in shared memory, then each key placed by its rank across
//     the chunks; out-of-range ids become the largest key and are dropped.
//     Sorted by key is sorted by (id, m).
//  2. embed_piece_k: the sorted list is cut into pieces of kEmbPiece
//     entries; a warp sums, for one piece and one 512-column block, the dx
//     rows of each run of equal ids in order, and leaves the run's sum in
//     part at the row of the run's first sorted entry in the piece.
//  3. embed_gather_k: the warps of an id's first sorted entry (one per 128
//     columns) add the id's piece sums in piece order (its own, then the one
//     at each later piece start the run still covers) into dwte[id].
constexpr int kEmbPiece = 32;
constexpr int kEmbCols = 512;  // columns per warp task: 4 float4 per lane
constexpr unsigned kEmbNone = 0xffffffffu;

// 1a. each CTA sorts one chunk of kEmbChunk consecutive positions' keys
// (bitonic network in shared memory, one key per thread)
constexpr int kEmbChunk = 1024;
constexpr size_t kEmbRankSmem = 192 * 1024;  // the rank pass stages up to 48 sorted chunks
__global__ void __launch_bounds__(kEmbChunk) embed_sort_chunk_k(const int* __restrict__ tok, int M, int V, int mbits,
                                                               unsigned* __restrict__ chunks) {
  __shared__ unsigned sk[kEmbChunk];
  const int i = threadIdx.x;
  const int m = blockIdx.x * kEmbChunk + i;
  unsigned key = kEmbNone;
  if (m < M) {
    const int id = tok[m];
    if (id >= 0 && id < V) key = ((unsigned)id << mbits) | (unsigned)m;
  }
  sk[i] = key;
  __syncthreads();
  for (int k = 2; k <= kEmbChunk; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int pj = i ^ j;
      if (pj > i) {
        const unsigned a = sk[i], b = sk[pj];
        if ((a > b) == ((i & k) == 0)) {  // ascending where bit k of i is clear
          sk[i] = b;
          sk[pj] = a;
        }
      }
      __syncthreads();
    }
  chunks[(size_t)blockIdx.x * kEmbChunk + i] = sk[i];
}

// 1b. a key's place in the whole sorted list is its index in its sorted chunk
// plus, for every other chunk, the number of that chunk's keys below it
// (binary search); the keys are unique, so the places are a permutation.
// keys[] beyond the valid keys must hold kEmbNone already.
template <bool SMEM>
__global__ void __launch_bounds__(1024) embed_rank_k(const unsigned* __restrict__ chunks, int nchunks,
                                                     unsigned* __restrict__ keys) {
  extern __shared__ unsigned sc[];  // every sorted chunk, when they fit
  const unsigned* src = chunks;
  if (SMEM) {
    for (int i = threadIdx.x; i < nchunks * kEmbChunk; i += blockDim.x) sc[i] = chunks[i];
    __syncthreads();
    src = sc;
  }
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= nchunks * kEmbChunk) return;
  const unsigned key = src[e];
  if (key == kEmbNone) return;
  const int c = e / kEmbChunk;
  int rank = e - c * kEmbChunk;
  for (int c2 = 0; c2 < nchunks; ++c2) {
    if (c2 == c) continue;
    const unsigned* s = src + (size_t)c2 * kEmbChunk;
    int lo = 0, n = kEmbChunk;  // first index with s[index] >= key
    while (n > 0) {
      const int h = n >> 1;
      if (s[lo + h] < key) {
        lo += h + 1;
        n -= h + 1;
      } else {
        n = h;
      }
    }
    rank += lo;
  }
  keys[rank] = key;
}

__device__ __forceinline__ void emb_add_row(float4* acc, const float* row, int c0, int d, int lane) {
#pragma unroll
  for (int q = 0; q < kEmbCols / 128; ++q) {
    const int c = c0 + q * 128 + lane * 4;
    if (c < d) {
      const float4 v = ld4(row + c);
      acc[q].x += v.x; acc[q].y += v.y; acc[q].z += v.z; acc[q].w += v.w;
    }
  }
}
__device__ __forceinline__ void emb_put_row(float* row, const float4* acc, int c0, int d, int lane) {
#pragma unroll
  for (int q = 0; q < kEmbCols / 128; ++q) {
    const int c = c0 + q * 128 + lane * 4;
    if (c < d) st4(row + c, acc[q]);
  }
}

// warp task w = piece * ncb + column block
__global__ void embed_piece_k(const unsigned* __restrict__ keys, const float* __restrict__ dx, float* __restrict__ part,
                              int M, int d, int mbits, int ncb) {
  const long long w = (long long)blockIdx.x * kRowWarps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const long long tasks = (long long)((M + kEmbPiece - 1) / kEmbPiece) * ncb;
  if (w >= tasks) return;
  const int piece = (int)(w / ncb), c0 = (int)(w % ncb) * kEmbCols;
  const int i0 = piece * kEmbPiece, i1 = min(M, i0 + kEmbPiece);
  const unsigned mmask = (1u << mbits) - 1;
  float4 acc[kEmbCols / 128];
#pragma unroll
  for (int q = 0; q < kEmbCols / 128; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  int run = i0;
  unsigned cur = keys[i0] == kEmbNone ? kEmbNone : keys[i0] >> mbits;
  for (int i = i0; i < i1; ++i) {
    const unsigned key = keys[i];
    if (key == kEmbNone) break;  // the rest of the list is out-of-range ids
    const unsigned id = key >> mbits;
    if (id != cur) {  // a new run: leave the finished one's sum
      emb_put_row(part + (size_t)run * d, acc, c0, d, lane);
#pragma unroll
      for (int q = 0; q < kEmbCols / 128; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      run = i;
      cur = id;
    }
    emb_add_row(acc, dx + (size_t)(key & mmask) * d, c0, d, lane);
  }
  if (cur != kEmbNone) emb_put_row(part + (size_t)run * d, acc, c0, d, lane);
}

// warp task w = sorted entry * ncg + 128-column group; only an id's first
// entry works. The piece starts the run still covers are checked 32 at a
// time (one per lane); their sums are then added in piece order, 16 rows'
// loads in flight before the adds (a long run of a frequent id would
// otherwise be a chain of dependent loads).
constexpr int kEmbGatherRows = 16;
__global__ void embed_gather_k(const unsigned* __restrict__ keys, const float* __restrict__ part,
                               float* __restrict__ dwte, int M, int d, int mbits, int ncg) {
  const long long w = (long long)blockIdx.x * kRowWarps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)M * ncg) return;
  const int i = (int)(w / ncg);
  const int c = (int)(w % ncg) * 128 + lane * 4;
  const unsigned key = keys[i];
  if (key == kEmbNone) return;
  const unsigned id = key >> mbits;
  if (i > 0 && (keys[i - 1] >> mbits) == id && keys[i - 1] != kEmbNone) return;
  const bool col = c < d;
  float4 acc = col ? ld4(part + (size_t)i * d + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = (i / kEmbPiece + 1) * kEmbPiece; q0 < M; q0 += 32 * kEmbPiece) {
    const int q = q0 + lane * kEmbPiece;
    const unsigned kq = q < M ? keys[q] : kEmbNone;
    const unsigned same = __ballot_sync(0xffffffffu, kq != kEmbNone && (kq >> mbits) == id);
    const int n = same == 0xffffffffu ? 32 : __ffs(~same) - 1;  // the run is contiguous
    for (int t0 = 0; t0 < n; t0 += kEmbGatherRows) {
      if (!col) continue;
      float4 r[kEmbGatherRows];
#pragma unroll
      for (int t = 0; t < kEmbGatherRows; ++t)  // rows past the run repeat its last one (not added)
        r[t] = ld4(part + (size_t)(q0 + min(t0 + t, n - 1) * kEmbPiece) * d + c);
#pragma unroll
      for (int t = 0; t < kEmbGatherRows; ++t)
        if (t0 + t < n) { acc.x += r[t].x; acc.y += r[t].y; acc.z += r[t].z; acc.w += r[t].w; }
    }
    if (n < 32) break;
  }
  if (col) {
    float* row = dwte + (size_t)id * d + c;
    const float4 o = ld4(row);
    st4(row, make_float4(o.x + acc.x, o.y + acc.y, o.z + acc.z, o.w + acc.w));
  }
}

// y = x * r, r = 1/sqrt(mean(x^2) + eps).
template <typename T>
__global__ void rmsnorm_fwd_k(const float* __restrict__ x, T* __restrict__ y, float* __restrict__ r,
                              int M, int d) {
  int m = blockIdx.x * kRowWarps + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (m >= M) return;
  const float* xr = x + (size_t)m * d;
  float ss = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float4 v = ld4(xr + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  float rr = rsqrtf(ss / (float)d + kEps);
  T* yr = y + (size_t)m * d;
  for (int c = lane * 4; c < d; c += 128) {
    float4 v = ld4(xr + c);
    st4(yr + c, make_float4(v.x * rr, v.y * rr, v.z * rr, v.w * rr));
  }
  if (lane == 0) r[m] = rr;
}

// dx = [dx +] r * (dy - y * mean(dy * y)); optional copy in the element type.
// dy arrives in the element type (bf16 in the bf16 mode); dx stays fp32.
template <typename T>
__global__ void rmsnorm_bwd_k(const T* __restrict__ dy, const T* __restrict__ y,
                              const float* __restrict__ r, float* __restrict__ dx, T* __restrict__ dxe,
                              int M, int d, int accumulate) {
  int m = blockIdx.x * kRowWarps + threadIdx.x / 32;
  int lane = threadIdx.x & 31;
  if (m >= M) return;
  const T* g = dy + (size_t)m * d;
  const T* yr = y + (size_t)m * d;
  float dot = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float4 a = ld4(g + c), b = ld4(yr + c);
    dot += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
  }
  dot = warp_sum(dot) / (float)d;
  float rr = r[m];
  float* o = dx + (size_t)m * d;
  T* oe = dxe ? dxe + (size_t)m * d : nullptr;
  for (int c = lane * 4; c < d; c += 128) {
    float4 a = ld4(g + c), b = ld4(yr + c);
    float4 v = make_float4(rr * (a.x - b.x * dot), rr * (a.y - b.y * dot), rr * (a.z - b.z * dot),
                           rr * (a.w - b.w * dot));
    if (accumulate) {
      float4 p = ld4(o + c);
      v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
    }
    st4(o + c, v);
    if (oe) st4(oe + c, v);
  }
}

// Per-head QK-norm then RoPE, in place on the q and k columns of qkv[M,3d].
// Lane L owns head dims L, L+32, L+64, L+96, so the RoPE partners (j, j+64)
// sit in the same lane. rqk[m, which*H + h] = 1/sqrt(mean(q^2)+eps).
template <typename T>
__global__ void qk_norm_rope_fwd_k(T* __restrict__ qkv, float* __restrict__ rqk,
                                   const float* __restrict__ cs, const float* __restrict__ sn,
                                   int M, int Tlen, int H) {
  int w = blockIdx.x * kRowWarps + threadIdx.x / 32;  // (m, which, h)
  int lane = threadIdx.x & 31;
  if (w >= M * 2 * H) return;
  int m = w / (2 * H), wh = w % (2 * H);
  int d = H * kHeadDim;
  T* p = qkv + (size_t)m * 3 * d + (size_t)wh * kHeadDim;  // q heads then k heads
  float v[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) v[c] = ldf(p + lane + 32 * c);
  float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
  float rr = rsqrtf(ss / (float)kHeadDim + kEps);
  int t = m % Tlen;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    int j = lane + 32 * c;
    float co = cs[t * kHalf + j], si = sn[t * kHalf + j];
    float a = v[c] * rr, b = v[c + 2] * rr;
    stf(p + j, a * co - b * si);
    stf(p + j + kHalf, a * si + b * co);
  }
  if (lane == 0) rqk[(size_t)m * 2 * H + wh] = rr;
}

// Backward of q_hat = rope(rmsnorm(q)): dq_n = R^T dq_hat, q_n = R^T q_hat,
// dq = r * (dq_n - q_n * mean(dq_n * q_n)). dqk is fp32 [2, M, d] (dq_hat
// plane, then dk_hat plane); results go to the q,k columns of dqkv[M,3d].
// One warp per (token, q or k): the position's rotation angles are read once
// and the token's heads are taken four at a time, with all their loads issued
// before the arithmetic (a warp-per-head layout kept too few bytes in flight).
// Lane L owns the rotation pairs j = 2L, 2L+1 (partners j+64), so every access
// is a coalesced 2-element vector; heads = 1 covers only the q heads.
template <typename T>
__global__ void qk_norm_rope_bwd_k(const float* __restrict__ dqk, const T* __restrict__ qkv,
                                   const float* __restrict__ rqk, const float* __restrict__ cs,
                                   const float* __restrict__ sn, T* __restrict__ dqkv, int M,
                                   int Tlen, int H, int heads) {
  const int w = blockIdx.x * kRowWarps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= M * heads) return;
  const int m = w / heads, which = w % heads;
  const int d = H * kHeadDim;
  const int t = m % Tlen, j = 2 * lane;
  const float2 co = *reinterpret_cast<const float2*>(cs + t * kHalf + j);
  const float2 si = *reinterpret_cast<const float2*>(sn + t * kHalf + j);
  const float c2[2] = {co.x, co.y}, s2[2] = {si.x, si.y};
  const float* gbase = dqk + (size_t)which * M * d + (size_t)m * d;
  const T* qbase = qkv + (size_t)m * 3 * d + (size_t)which * d;
  T* obase = dqkv + (size_t)m * 3 * d + (size_t)which * d;
  const float* rbase = rqk + (size_t)m * 2 * H + (size_t)which * H;
  for (int h0 = 0; h0 < H; h0 += 4) {
    float2 g1[4], g2[4], qa[4], qb[4];
    float rr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int h = h0 + i;
      if (h < H) {
        const float* g = gbase + h * kHeadDim;
        const T* q = qbase + h * kHeadDim;
        g1[i] = *reinterpret_cast<const float2*>(g + j);
        g2[i] = *reinterpret_cast<const float2*>(g + j + kHalf);
        qa[i] = ld2(q + j);
        qb[i] = ld2(q + j + kHalf);
        rr[i] = rbase[h];
      } else {
        g1[i] = g2[i] = qa[i] = qb[i] = make_float2(0.f, 0.f);
        rr[i] = 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float q1[2] = {qa[i].x, qa[i].y}, q2[2] = {qb[i].x, qb[i].y};
      const float a1[2] = {g1[i].x, g1[i].y}, a2[2] = {g2[i].x, g2[i].y};
      float gn[4], qn[4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        gn[u] = a1[u] * c2[u] + a2[u] * s2[u];
        gn[u + 2] = -a1[u] * s2[u] + a2[u] * c2[u];
        qn[u] = q1[u] * c2[u] + q2[u] * s2[u];
        qn[u + 2] = -q1[u] * s2[u] + q2[u] * c2[u];
      }
      const float dot = warp_sum(gn[0] * qn[0] + gn[1] * qn[1] + gn[2] * qn[2] + gn[3] * qn[3]) / (float)kHeadDim;
      const int h = h0 + i;
      if (h < H) {
        T* o = obase + h * kHeadDim;
        st2(o + j, make_float2(rr[i] * (gn[0] - qn[0] * dot), rr[i] * (gn[1] - qn[1] * dot)));
        st2(o + j + kHalf, make_float2(rr[i] * (gn[2] - qn[2] * dot), rr[i] * (gn[3] - qn[3] * dot)));
      }
    }
  }
}

__device__ __forceinline__ void ld8(const bf16* p, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}
__device__ __forceinline__ void ld8(const float* p, float* f) {
  const float4 a = ld4(p), b = ld4(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// D[b,h,t] = sum_e dout[m, h*128+e] * o[m, h*128+e]  (softmax backward term).
// With lse given, also nL2[b,h,t] = -(lse * log2(e) + 3.5): the row's negated
// logsumexp in base-2 units, offset so that exp2(s * log2(e) / sqrt(128) + nL2)
// is the probability already multiplied by the 1/sqrt(128) = 2^-3.5 score
// scale. One warp per token row and all its heads: the warp's halves take
// heads 2i and 2i+1, a lane 8 consecutive dims, and the loads of four head
// pairs are issued before any sum (one warp per (token, head) kept 512 bytes
// in flight per warp).
template <typename T>
__global__ void attn_rowdot_k(const T* __restrict__ dout, const T* __restrict__ o,
                              float* __restrict__ Drow, int B, int Tlen, int H,
                              const float* __restrict__ lse, float* __restrict__ L2) {
  const int m = blockIdx.x * kRowWarps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int M = B * Tlen;
  if (m >= M) return;
  const int half = lane >> 4, l16 = lane & 15;
  const int b = m / Tlen, t = m % Tlen;
  const size_t row = (size_t)m * H * kHeadDim + l16 * 8;
  // head pairs per round: six in bf16 (the d20 model's ten heads in one round,
  // raw 16-byte loads all issued first), four in fp32
  constexpr int RP = sizeof(T) == 2 ? 6 : 4;
  for (int h0 = 0; h0 < H; h0 += 2 * RP) {
    float lsev[RP];
#pragma unroll
    for (int i = 0; i < RP; ++i) {  // the lse rows early, off the end of the chain
      const int h = h0 + 2 * i + half;
      lsev[i] = (L2 && l16 == 0 && h < H) ? lse[((size_t)b * H + h) * Tlen + t] : 0.f;
    }
    uint4 ru[RP], rv[RP];
    float u[RP][8], v[RP][8];
    if constexpr (sizeof(T) == 2) {
#pragma unroll
      for (int i = 0; i < RP; ++i) {
        const int h = h0 + 2 * i + half;
        ru[i] = h < H ? *reinterpret_cast<const uint4*>(dout + row + (size_t)h * kHeadDim) : make_uint4(0, 0, 0, 0);
        rv[i] = h < H ? *reinterpret_cast<const uint4*>(o + row + (size_t)h * kHeadDim) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < RP; ++i) {
        const uint32_t wu[4] = {ru[i].x, ru[i].y, ru[i].z, ru[i].w}, wv[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wu[q]));
          const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[q]));
          u[i][2 * q] = a.x; u[i][2 * q + 1] = a.y;
          v[i][2 * q] = c.x; v[i][2 * q + 1] = c.y;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < RP; ++i) {
        const int h = h0 + 2 * i + half;
        if (h < H) {
          ld8(dout + row + (size_t)h * kHeadDim, u[i]);
          ld8(o + row + (size_t)h * kHeadDim, v[i]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) u[i][e] = v[i][e] = 0.f;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RP; ++i) {
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += u[i][e] * v[i][e];
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      const int h = h0 + 2 * i + half;
      if (l16 == 0 && h < H) {
        const size_t idx = ((size_t)b * H + h) * Tlen + t;
        Drow[idx] = sum;
        if (L2) L2[idx] = -fmaf(lsev[i], 1.4426950408889634f, 3.5f);
      }
    }
  }
}

// out = in * s for one device float (the loss-gradient scale of an
// accumulating backward: 1 / unmasked count times the caller's scale).
__global__ void scale_scalar_k(const float* __restrict__ in, float s, float* __restrict__ out) { *out = *in * s; }

// Packed uint16 token rows [B, T+1] -> inputs tok[b, t] = row[b][t] and
// targets tgt[b, t] = row[b][t + 1] (int32, [B, T]).
__global__ void unpack_u16_k(const uint16_t* __restrict__ packed, int B, int Tlen, int32_t* __restrict__ tok,
                             int32_t* __restrict__ tgt) {
  const long long n = (long long)B * Tlen;
  for (long long m = blockIdx.x * (long long)blockDim.x + threadIdx.x; m < n; m += (long long)gridDim.x * blockDim.x) {
    const long long b = m / Tlen, t = m - b * Tlen;
    const uint16_t* row = packed + b * (Tlen + 1);
    tok[m] = row[t];
    tgt[m] = row[t + 1];
  }
}

// Combine the per-tile cross-entropy partials of each row: lse = max + log(sum
// of sum-exp rescaled to that max), argmax (lowest column among ties: the
// tiles are in column order and a later tile only wins with a strictly
// larger maximum), nll = lse - target logit. A block covers 32 consecutive
// rows (one per lane, so every load is one 128-byte row segment); its 8 warps
// each take a contiguous eighth of the tiles in one online pass, and the 8
// results are combined in tile order.
constexpr int kCeWarps = 8;
__device__ __forceinline__ void ce_merge(float& mx, float& s, int& arg, float m2, float s2, int a2) {
  if (m2 > mx) {
    s = s * expf(mx - m2) + s2;  // mx = -inf: s is 0 and so is the product
    mx = m2;
    arg = a2;
  } else if (m2 != -INFINITY) {
    s += s2 * expf(m2 - mx);
  }
}
__global__ void __launch_bounds__(32 * kCeWarps)
    ce_reduce_k(const float* __restrict__ pm, const float* __restrict__ ps, const int* __restrict__ pa,
                const float* __restrict__ pt, const int* __restrict__ tgt, int nt, float* __restrict__ lse,
                float* __restrict__ nll, int* __restrict__ amax, int M) {
  __shared__ float smx[kCeWarps][32], ss[kCeWarps][32];
  __shared__ int sarg[kCeWarps][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int m = blockIdx.x * 32 + lane;
  const int per = (nt + kCeWarps - 1) / kCeWarps;
  const int t0 = w * per, t1 = min(nt, t0 + per);
  float mx = -INFINITY, s = 0.f;
  int arg = 0;
  if (m < M)
    for (int t = t0; t < t1; ++t) {
      const size_t i = (size_t)t * M + m;
      const float v = pm[i];
      if (v > mx) {
        s = s * expf(mx - v) + ps[i];
        mx = v;
        arg = pa[i];
      } else if (v != -INFINITY) {
        s += ps[i] * expf(v - mx);
      }
    }
  smx[w][lane] = mx;
  ss[w][lane] = s;
  sarg[w][lane] = arg;
  __syncthreads();
  if (w == 0 && m < M) {
    for (int k = 1; k < kCeWarps; ++k) ce_merge(mx, s, arg, smx[k][lane], ss[k][lane], sarg[k][lane]);
    const float l = mx + logf(s);
    lse[m] = l;
    nll[m] = tgt[m] < 0 ? 0.f : l - pt[m];  // a masked position carries no loss
    amax[m] = arg;
  }
}

// Two running (maximum, sum of exp(x - maximum), argmax) states of column
// sets in no particular order: the argmax tie goes to the lower column.
__device__ __forceinline__ void ce_merge_any(float& mx, float& s, int& arg, float m2, float s2, int a2) {
  if (m2 == -INFINITY) return;
  if (mx == -INFINITY) { mx = m2; s = s2; arg = a2; return; }
  const float nm = fmaxf(mx, m2);
  s = s * expf(mx - nm) + s2 * expf(m2 - nm);
  if (m2 > mx || (m2 == mx && a2 < arg)) arg = a2;
  mx = nm;
}

// Cross-entropy rows of a materialised fp32 logits block [M, V]: logsumexp,
// loss lse - logit[target] (0 for a masked target -1), argmax (lowest column
// among ties). CTA (seg, m) reads columns [seg L, min(V, seg L + L)) of row m
// once, each thread keeping a running maximum and the sum of exp(x - maximum)
// (rescaled when the maximum grows) over its 16-byte pieces, four in flight.
// With one segment per row the CTA finishes its row. With S > 1 segments
// (few rows: the segments spread a row over many SMs) each CTA leaves its
// (maximum, sum, argmax, target logit) in part[m S + seg], and the CTA that
// counts itself last on *counter merges every row's segments in column order
// (the result does not depend on scheduling) and sets the counter back to 0.
constexpr int kCeRowThreads = 256;
__global__ void __launch_bounds__(kCeRowThreads)
    ce_rows_k(const float* __restrict__ logits, const int* __restrict__ tgt, float* __restrict__ lse,
              float* __restrict__ nll, int* __restrict__ amax, int M, int V, int L, int S, float4* part, int* counter,
              int* status) {
  __shared__ float smx[kCeRowThreads / 32], ssum[kCeRowThreads / 32];
  __shared__ int sarg[kCeRowThreads / 32];
  __shared__ int is_last;
  const int seg = blockIdx.x, m = blockIdx.y;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const float* row = logits + (size_t)m * V;
  const int lo = seg * L, hi = min(V, lo + L);
  float mx = -INFINITY, s = 0.f;
  int arg = 0x7fffffff;
  if ((V & 3) == 0) {  // L is a multiple of 4: every piece is whole and aligned
    constexpr int kStep = 4 * kCeRowThreads;
    for (int n0 = lo + 4 * threadIdx.x; n0 < hi; n0 += 4 * kStep) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int n = n0 + u * kStep;
        v[u] = n < hi ? ld4(row + n) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int n = n0 + u * kStep;
        if (n >= hi) break;
        const float gm = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
        if (gm > mx) {
          s *= expf(mx - gm);  // 0 while mx = -inf
          mx = gm;
          arg = v[u].x == gm ? n : v[u].y == gm ? n + 1 : v[u].z == gm ? n + 2 : n + 3;
        }
        s += expf(v[u].x - mx) + expf(v[u].y - mx) + expf(v[u].z - mx) + expf(v[u].w - mx);
      }
    }
  } else {
    for (int n = lo + threadIdx.x; n < hi; n += kCeRowThreads) {
      const float x = row[n];
      if (x > mx) {
        s *= expf(mx - x);
        mx = x;
        arg = n;
      }
      s += expf(x - mx);
    }
  }
  // this CTA's state: warps, then warp 0 over the warps
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mx, o), os = __shfl_xor_sync(0xffffffffu, s, o);
    const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
    ce_merge_any(mx, s, arg, om, os, oa);
  }
  if (lane == 0) {
    smx[wid] = mx;
    ssum[wid] = s;
    sarg[wid] = arg;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kCeRowThreads / 32; ++w) ce_merge_any(mx, s, arg, smx[w], ssum[w], sarg[w]);
    const int t = tgt[m];
    if (S == 1) {
      const float l = mx + logf(s);
      lse[m] = l;
      amax[m] = arg;
      if (t == -1) {
        nll[m] = 0.f;  // masked position: no loss
      } else if (t < 0 || t >= V) {
        set_status(status, DEV_BAD_TOKEN);
        nll[m] = 0.f;
      } else {
        nll[m] = l - row[t];
      }
    } else {
      const float tl = (t >= lo && t < hi) ? row[t] : 0.f;
      part[(size_t)m * S + seg] = make_float4(mx, s, __int_as_float(arg), tl);
      __threadfence();
      is_last = atomicAdd(counter, 1) == S * M - 1;
    }
  }
  if (S == 1) return;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int r = threadIdx.x; r < M; r += kCeRowThreads) {
    float rm = -INFINITY, rs = 0.f;
    int ra = 0;
    for (int k = 0; k < S; ++k) {  // column order: a later segment wins a tie only with a larger maximum
      const float4 q = __ldcg(part + (size_t)r * S + k);
      ce_merge(rm, rs, ra, q.x, q.y, __float_as_int(q.z));
    }
    const float l = rm + logf(rs);
    const int t = tgt[r];
    lse[r] = l;
    amax[r] = ra;
    if (t == -1) {
      nll[r] = 0.f;
    } else if (t < 0 || t >= V) {
      set_status(status, DEV_BAD_TOKEN);
      nll[r] = 0.f;
    } else {
      nll[r] = l - __ldcg(part + (size_t)r * S + t / L).w;
    }
  }
  if (threadIdx.x == 0) *counter = 0;
}

// loss = mean of nll over the positions whose target is not masked (-1),
// 0 when every position is masked; inv_count = 1 / that count (0 if none).
// Fixed summation order (one CTA, float64 partials). nll may be null: then
// only inv_count is formed.
__global__ void mean_loss_k(const float* __restrict__ nll, const int* __restrict__ tgt, int M,
                            float* __restrict__ loss, float* __restrict__ inv_count) {
  __shared__ double sh[1024];
  __shared__ int shn[1024];
  double s = 0.0;
  int n = 0;
  for (int i = threadIdx.x; i < M; i += blockDim.x) {
    if (tgt[i] >= 0) {
      if (nll) s += (double)nll[i];
      ++n;
    }
  }
  sh[threadIdx.x] = s;
  shn[threadIdx.x] = n;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) {
      sh[threadIdx.x] += sh[threadIdx.x + w];
      shn[threadIdx.x] += shn[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int cnt = shn[0];
    if (loss) *loss = cnt > 0 ? (float)(sh[0] / (double)cnt) : 0.f;
    if (inv_count) *inv_count = cnt > 0 ? (float)(1.0 / (double)cnt) : 0.f;
  }
}

__global__ void check_ids_k(const int* __restrict__ ids, int n, int lo, int V, int* status) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    int v = ids[i];
    if (v < lo || v >= V) set_status(status, DEV_BAD_TOKEN);
  }
}

// C[m, n] = sum_s partial[s, m, n] + beta * C[m, n]; the split order is fixed,
// so the result does not depend on scheduling.
__global__ void splitk_reduce_k(const float* __restrict__ part, int splits, float* __restrict__ C, long long ldc,
                                int M, int N, float beta) {
  const long long n4 = (long long)N / 4;
  const long long total = (long long)M * n4;
  const size_t plane = (size_t)M * N;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const long long m = i / n4, c = (i % n4) * 4;
    const float* src = part + (size_t)m * N + c;
    float4 a = ld4(src);
    for (int s = 1; s < splits; ++s) {
      float4 b = ld4(src + s * plane);
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    float* dst = C + (size_t)m * ldc + c;
    if (beta != 0.f) {
      float4 o = ld4(dst);
      a.x += beta * o.x; a.y += beta * o.y; a.z += beta * o.z; a.w += beta * o.w;
    }
    st4(dst, a);
  }
}

inline int row_blocks(long long rows) { return (int)((rows + kRowWarps - 1) / kRowWarps); }

}  // namespace

template <typename T>
cudaError_t embed_fwd(const int* tok, const T* wte, float* x, int M, int d, int V, int* status,
                      cudaStream_t s) {
  embed_fwd_k<T><<<row_blocks(M), 32 * kRowWarps, 0, s>>>(tok, wte, x, M, d, V, status);
  return cudaGetLastError();
}

namespace {
struct EmbPlan {
  int mbits, nchunks;
  bool sorted;
};
EmbPlan emb_plan(int M, int d, int V, bool scratch) {
  EmbPlan pl;
  int vbits = 1;
  pl.mbits = 1;
  while ((1LL << pl.mbits) < M) ++pl.mbits;
  while ((1LL << vbits) < V) ++vbits;
  pl.nchunks = (M + kEmbChunk - 1) / kEmbChunk;
  pl.sorted = scratch && d % 4 == 0 && pl.mbits + vbits <= 32 && pl.nchunks <= kEmbMaxChunks;
  return pl;
}
}  // namespace

int embed_bwd_launches(int M, int d, int V, bool scratch) {
  if (M == 0) return 0;
  return emb_plan(M, d, V, scratch).sorted ? 4 : 1;
}

template <typename T>
cudaError_t embed_bwd(const int* tok, const T*, const float* dx, float* dwte, int M, int d, int V,
                      cudaStream_t s, unsigned* keys, float* part) {
  if (M == 0) return cudaSuccess;
  const EmbPlan pl = emb_plan(M, d, V, keys && part);
  const int mbits = pl.mbits, nch = pl.nchunks;
  if (!pl.sorted) {  // float atomics: the summation order follows arrival
    embed_bwd_k<<<row_blocks(M), 32 * kRowWarps, 0, s>>>(tok, dx, dwte, M, d, V);
    return cudaGetLastError();
  }
  // the sorted chunks sit in part (dead until the run sums), keys fill from kEmbNone
  unsigned* chunks = reinterpret_cast<unsigned*>(part);
  cudaError_t e = cudaMemsetAsync(keys, 0xff, (size_t)M * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  embed_sort_chunk_k<<<nch, kEmbChunk, 0, s>>>(tok, M, V, mbits, chunks);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t rank_smem = (size_t)nch * kEmbChunk * sizeof(unsigned);
  if (rank_smem <= kEmbRankSmem) {
    e = cudaFuncSetAttribute(embed_rank_k<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEmbRankSmem);
    if (e != cudaSuccess) return e;
    embed_rank_k<true><<<nch, kEmbChunk, rank_smem, s>>>(chunks, nch, keys);
  } else {
    embed_rank_k<false><<<nch, kEmbChunk, 0, s>>>(chunks, nch, keys);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int ncb = (d + kEmbCols - 1) / kEmbCols;
  const long long pt = (long long)((M + kEmbPiece - 1) / kEmbPiece) * ncb;
  embed_piece_k<<<(int)((pt + kRowWarps - 1) / kRowWarps), 32 * kRowWarps, 0, s>>>(keys, dx, part, M, d, mbits, ncb);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int ncg = (d + 127) / 128;
  const long long gt = (long long)M * ncg;
  embed_gather_k<<<(int)((gt + kRowWarps - 1) / kRowWarps), 32 * kRowWarps, 0, s>>>(keys, part, dwte, M, d, mbits,
                                                                                    ncg);
  return cudaGetLastError();
}

template <typename T>
cudaError_t rmsnorm_fwd(const float* x, T* y, float* r, int M, int d, cudaStream_t s) {
  rmsnorm_fwd_k<T><<<row_blocks(M), 32 * kRowWarps, 0, s>>>(x, y, r, M, d);
  return cudaGetLastError();
}

template <typename T>
cudaError_t rmsnorm_bwd(const T* dy, const T* y, const float* r, float* dx, T* dx_e, int M,
                        int d, int accumulate, cudaStream_t s) {
  rmsnorm_bwd_k<T><<<row_blocks(M), 32 * kRowWarps, 0, s>>>(dy, y, r, dx, dx_e, M, d, accumulate);
  return cudaGetLastError();
}

template <typename T>
cudaError_t qk_norm_rope_fwd(T* qkv, float* rqk, const float* cs, const float* sn, int M, int T_,
                             int H, cudaStream_t s) {
  qk_norm_rope_fwd_k<T><<<row_blocks((long long)M * 2 * H), 32 * kRowWarps, 0, s>>>(qkv, rqk, cs, sn, M, T_, H);
  return cudaGetLastError();
}

template <typename T>
cudaError_t qk_norm_rope_bwd(const float* dqk, const T* qkv, const float* rqk, const float* cs,
                             const float* sn, T* dqkv, int M, int T_, int H, cudaStream_t s, int heads) {
  qk_norm_rope_bwd_k<T><<<row_blocks((long long)M * heads), 32 * kRowWarps, 0, s>>>(dqk, qkv, rqk, cs, sn, dqkv, M,
                                                                                T_, H, heads);
  return cudaGetLastError();
}

template <typename T>
cudaError_t attn_rowdot(const T* dout, const T* o, float* Drow, int B, int T_, int H,
                        cudaStream_t s, const float* lse, float* L2) {
  attn_rowdot_k<T><<<row_blocks((long long)B * T_), 32 * kRowWarps, 0, s>>>(dout, o, Drow, B, T_, H, lse, L2);
  return cudaGetLastError();
}

cudaError_t ce_rows_from_logits(const float* logits, const int* tgt, float* lse, float* nll, int* amax, int M, int V,
                                int* status, cudaStream_t s, float* part, int* counter, int sms) {
  if (M == 0) return cudaSuccess;
  if (M > 65535 || V < 1) return cudaErrorInvalidValue;
  // segments per row: enough CTAs for two per SM, at least 1024 columns each
  int S = 1;
  if (part && counter && M < 2 * sms) {
    S = (2 * sms + M - 1) / M;
    if (S > kCeMaxSegments) S = kCeMaxSegments;
    if (S > V / 1024) S = V / 1024 > 1 ? V / 1024 : 1;
  }
  const int L = ((V + S - 1) / S + 3) & ~3;
  S = (V + L - 1) / L;  // no empty segment
  ce_rows_k<<<dim3(S, M), kCeRowThreads, 0, s>>>(logits, tgt, lse, nll, amax, M, V, L, S,
                                                 reinterpret_cast<float4*>(part), counter, status);
  return cudaGetLastError();
}

cudaError_t ce_reduce_partials(const float* p_max, const float* p_sum, const int* p_arg,
                               const float* p_tgt, const int* tgt, int n_tiles, float* lse, float* nll, int* amax,
                               int M, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  ce_reduce_k<<<(M + 31) / 32, 32 * kCeWarps, 0, s>>>(p_max, p_sum, p_arg, p_tgt, tgt, n_tiles, lse, nll, amax, M);
  return cudaGetLastError();
}

cudaError_t scale_scalar(const float* in, float scale, float* out, cudaStream_t s) {
  scale_scalar_k<<<1, 1, 0, s>>>(in, scale, out);
  return cudaGetLastError();
}

cudaError_t unpack_u16(const uint16_t* packed, int B, int T_, int32_t* tok, int32_t* tgt, cudaStream_t s) {
  const long long n = (long long)B * T_;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 148 * 8) blocks = 148 * 8;
  unpack_u16_k<<<(int)blocks, 256, 0, s>>>(packed, B, T_, tok, tgt);
  return cudaGetLastError();
}

cudaError_t splitk_reduce(const float* partial, int splits, float* C, long long ldc, int M, int N, float beta,
                          cudaStream_t s) {
  long long total = (long long)M * (N / 4);
  if (total == 0) return cudaSuccess;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 148 * 16) blocks = 148 * 16;
  splitk_reduce_k<<<blocks, 256, 0, s>>>(partial, splits, C, ldc, M, N, beta);
  return cudaGetLastError();
}

cudaError_t mean_loss(const float* nll, const int* tgt, int M, float* loss, float* inv_count, cudaStream_t s) {
  mean_loss_k<<<1, 1024, 0, s>>>(nll, tgt, M, loss, inv_count);
  return cudaGetLastError();
}

cudaError_t check_ids(const int* ids, int n, int lo, int V, int* status, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  check_ids_k<<<(n + 255) / 256, 256, 0, s>>>(ids, n, lo, V, status);
  return cudaGetLastError();
}

#define NC_INST(T)                                                                               \
  template cudaError_t embed_fwd<T>(const int*, const T*, float*, int, int, int, int*,          \
                                    cudaStream_t);                                               \
  template cudaError_t embed_bwd<T>(const int*, const T*, const float*, float*, int, int, int,  \
                                    cudaStream_t, unsigned*, float*);                            \
  template cudaError_t rmsnorm_fwd<T>(const float*, T*, float*, int, int, cudaStream_t);         \
  template cudaError_t rmsnorm_bwd<T>(const T*, const T*, const float*, float*, T*, int,         \
                                      int, int, cudaStream_t);                                   \
  template cudaError_t qk_norm_rope_fwd<T>(T*, float*, const float*, const float*, int, int,     \
                                           int, cudaStream_t);                                   \
  template cudaError_t qk_norm_rope_bwd<T>(const float*, const T*, const float*, const float*,   \
                                           const float*, T*, int, int, int, cudaStream_t, int);  \
  template cudaError_t attn_rowdot<T>(const T*, const T*, float*, int, int, int, cudaStream_t, const float*, float*);
NC_INST(float)
NC_INST(bf16)
#undef NC_INST

}  // namespace nc
