// Weight-streaming products of the decode step: C[m, n] = alpha * sum_k A[m, k] W[n, k]
// (+ beta * C) for at most 16 rows m (one token per sequence), bf16 operands,
// fp32 output, or relu(.)^2 in bf16 for the MLP up-projection. The product is
// bound by streaming W once from HBM (2 bytes per weight for 2 * rows FLOPs).
//
// Work items are (k-range, 16-column block) pairs, k-range-major; persistent
// CTAs (one per SM) take items round robin. The 16 W rows x k-range of an
// item are brought into shared memory by 16 untiled bulk copies (one per row)
// that complete on the item's mbarrier, in a ring of up to 4 stages, so an
// SM keeps the next items' weight reads (100+ KB) in flight while it works on
// the current one. (Per-thread 16-byte loads kept too few requests in flight:
// each warp load touched eight half lines, and the products ran at 1.2-1.4
// TB/s.) A staged row is padded by 64 bytes, so the 16-byte fragment reads of
// a warp's eight rows fall in distinct banks.
//
// The sum runs on the warp-level tensor-core MMA (m16n8k16, fp32 accumulate):
// a lane reads 8 consecutive k of one W row, which form the two k16 fragments
// of a 32-wide k chunk under a fixed permutation of k inside the chunk (the
// sum over k does not depend on its order); the A rows use the same
// permutation and stay in registers across the items of one k-range. The 16
// warps take the chunks of the k-range round robin; their partial sums are
// added in shared memory in warp order. With one k-range per product the CTA
// writes the outputs; with several, each item leaves its partial sums and the
// CTA that completes a column block last (a counter per block, left at zero)
// adds the k-ranges in order. Every result is independent of scheduling.
#include "ops.cuh"
#include "tc_ptx.cuh"

namespace nc {
namespace {

constexpr int SK_WARPS = 16;
constexpr int SK_THREADS = 32 * SK_WARPS;
constexpr int SK_CW = 16;                          // columns per item: two n8 tiles
constexpr int SK_KCH = 4;                          // k chunks per warp and item, at most
constexpr int SK_KC_MAX = SK_WARPS * SK_KCH * 32;  // longest k-range: 2048
constexpr int SK_PAD = 64;                         // bytes after each staged row
constexpr int SK_RED_BYTES = 2 * SK_WARPS * 16 * SK_CW * 4;  // double-buffered warp partials
constexpr int SK_SMEM_MAX = 227 * 1024 - 1024;  // dynamic part, leaving room for the static words
constexpr uint64_t kSkWaitNs = 2000000000ull;

struct SkParams {
  const bf16* A;
  const float* xres;  // if set, A = bf16(xres * r) with r the row's RMSNorm scale (A unused)
  const bf16* W;
  float* C;
  bf16* relu2;
  float* part;  // [nks][16][N] partial sums (nks > 1)
  int* cnt;     // [ncb] finished k-ranges per column block (nks > 1)
  int* status;
  long long lda, ldw, ldc;
  int M, N, K;
  float alpha, beta;
  int ncb, nks, KC, items, ns, row_bytes, stage_bytes;
  int whole;  // one k-range and rows packed (ldw == K): an item is one contiguous copy
};

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// eight fp32 values times a scale, as packed bf16
__device__ __forceinline__ uint4 pack8s(const float* v, float r) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0] * r, v[1] * r), h1 = __floats2bfloat162_rn(v[2] * r, v[3] * r);
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[4] * r, v[5] * r), h3 = __floats2bfloat162_rn(v[6] * r, v[7] * r);
  return make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                    *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
}

// the output value as stored: fp32 C (alpha, beta) or bf16 relu(alpha v)^2
__device__ __forceinline__ void sk_store(const SkParams& p, int m, int n, float v) {
  const size_t o = (size_t)m * p.ldc + n;
  if (p.relu2) {
    const float u = fmaxf(p.alpha * v, 0.f);
    p.relu2[o] = __float2bfloat16_rn(u * u);
  } else {
    p.C[o] = p.beta != 0.f ? p.alpha * v + p.beta * p.C[o] : p.alpha * v;
  }
}

// thread 0: the bulk copies of item i into stage s
__device__ __forceinline__ void sk_issue(const SkParams& p, uint8_t* stages, uint64_t* full, int i, int s) {
  const int kr = i / p.ncb, cb = i - kr * p.ncb;
  const int k0 = kr * p.KC, kn = min(p.KC, p.K - k0);
  const int n0 = cb * SK_CW, rows = min(SK_CW, p.N - n0);
  tc::mbar_arrive_expect_tx(full + s, (uint32_t)(rows * kn * 2));
  uint8_t* dst = stages + (size_t)s * p.stage_bytes;
  if (p.whole) {
    tc::bulk_load(dst, p.W + (size_t)n0 * p.ldw, (uint32_t)(rows * kn * 2), full + s);
    return;
  }
  for (int r = 0; r < rows; ++r)
    tc::bulk_load(dst + (size_t)r * p.row_bytes, p.W + (size_t)(n0 + r) * p.ldw + k0, (uint32_t)(kn * 2), full + s);
}

__global__ void __launch_bounds__(SK_THREADS, 1) skinny_gemm_k(const SkParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)p.ns * p.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.ns * p.stage_bytes + SK_RED_BYTES);
  __shared__ int s_last;
  __shared__ float s_ss[SK_WARPS][16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int first = blockIdx.x, step = gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.ns; ++s) tc::mbar_init(full + s, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int j = 0; j < p.ns; ++j) {
      const int i = first + j * step;
      if (i < p.items) sk_issue(p, stages, full, i, j);
    }
  // A fragments of this warp's chunks (rows g and g + 8, zero past M) for the k-range a_kr
  uint4 af[SK_KCH][2];
  int a_kr = -1;
  const bool a0ok = g < p.M, a1ok = g + 8 < p.M;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  if (p.xres) {
    // A = bf16(x r), r = 1/sqrt(mean(x^2) + eps) per row, from the fp32
    // residual rows (one k-range covers the row): each warp loads its
    // chunks' x once, the rows' sums of squares are added warp by warp in
    // warp order through shared memory, then the fragments are scaled
    float xf[SK_KCH][2][8];
    float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
    for (int u = 0; u < SK_KCH; ++u) {
      const int c = warp + SK_WARPS * u;
      const bool in = c * 32 < p.K;
      const size_t k = (size_t)c * 32 + 8 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool ok = in && (h ? a1ok : a0ok);
        const float* xr = p.xres + (size_t)(g + 8 * h) * p.lda + k;
        const float4 lo = ok ? *reinterpret_cast<const float4*>(xr) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 hi = ok ? *reinterpret_cast<const float4*>(xr + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        xf[u][h][0] = lo.x; xf[u][h][1] = lo.y; xf[u][h][2] = lo.z; xf[u][h][3] = lo.w;
        xf[u][h][4] = hi.x; xf[u][h][5] = hi.y; xf[u][h][6] = hi.z; xf[u][h][7] = hi.w;
      }
    }
#pragma unroll
    for (int u = 0; u < SK_KCH; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ss0 += xf[u][0][e] * xf[u][0][e];
        ss1 += xf[u][1][e] * xf[u][1][e];
      }
    ss0 += __shfl_xor_sync(0xffffffffu, ss0, 1);
    ss1 += __shfl_xor_sync(0xffffffffu, ss1, 1);
    ss0 += __shfl_xor_sync(0xffffffffu, ss0, 2);
    ss1 += __shfl_xor_sync(0xffffffffu, ss1, 2);
    if (t == 0) {
      s_ss[warp][g] = ss0;
      s_ss[warp][g + 8] = ss1;
    }
    __syncthreads();
    float tot0 = 0.f, tot1 = 0.f;
#pragma unroll
    for (int w = 0; w < SK_WARPS; ++w) {
      tot0 += s_ss[w][g];
      tot1 += s_ss[w][g + 8];
    }
    const float r0 = rsqrtf(tot0 / (float)p.K + kEps), r1 = rsqrtf(tot1 / (float)p.K + kEps);
#pragma unroll
    for (int u = 0; u < SK_KCH; ++u) {
      af[u][0] = pack8s(xf[u][0], r0);
      af[u][1] = pack8s(xf[u][1], r1);
    }
    a_kr = 0;
  }
  int it = 0;
  for (int i = first; i < p.items; i += step, ++it) {
    const int s = it % p.ns;
    const uint32_t ph = (uint32_t)(it / p.ns) & 1;
    const int kr = i / p.ncb, cb = i - kr * p.ncb;
    const int k0 = kr * p.KC, nch = min(p.KC, p.K - k0) / 32;
    const int n0 = cb * SK_CW;
    if (kr != a_kr) {
#pragma unroll
      for (int u = 0; u < SK_KCH; ++u) {
        const int c = warp + SK_WARPS * u;
        const bool in = c < nch;
        const size_t k = (size_t)k0 + c * 32 + 8 * t;
        af[u][0] = (in && a0ok) ? __ldg(reinterpret_cast<const uint4*>(p.A + (size_t)g * p.lda + k)) : zero;
        af[u][1] = (in && a1ok) ? __ldg(reinterpret_cast<const uint4*>(p.A + (size_t)(g + 8) * p.lda + k)) : zero;
      }
      a_kr = kr;
    }
    const bool ok = tc::mbar_wait(full + s, ph, nullptr, kSkWaitNs);
    if (__syncthreads_or(!ok)) {
      // give up: report, and let the copies already issued land before the CTA leaves
      if (threadIdx.x == 0) {
        set_status(p.status, DEV_TIMEOUT);
        for (int j = 0; j < p.ns; ++j) {
          const int ij = i + j * step;
          if (ij < p.items) tc::mbar_wait(full + (it + j) % p.ns, (uint32_t)((it + j) / p.ns) & 1, nullptr, kSkWaitNs);
        }
      }
      __syncthreads();
      return;
    }
    const uint8_t* sw = stages + (size_t)s * p.stage_bytes;
    float acc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
    for (int u = 0; u < SK_KCH; ++u) {
      const int c = warp + SK_WARPS * u;
      if (c >= nch) break;
      // k16 step 0 takes physical k 8t..8t+3 of the chunk, step 1 takes 8t+4..8t+7:
      // fragment registers {k 2t,2t+1} <- pieces .x/.z, {k 2t+8,2t+9} <- .y/.w
      const uint32_t a_s0[4] = {af[u][0].x, af[u][1].x, af[u][0].y, af[u][1].y};
      const uint32_t a_s1[4] = {af[u][0].z, af[u][1].z, af[u][0].w, af[u][1].w};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint4 wv = *reinterpret_cast<const uint4*>(sw + (size_t)(8 * j + g) * p.row_bytes + (c * 32 + 8 * t) * 2);
        const uint32_t b_s0[2] = {wv.x, wv.y};
        const uint32_t b_s1[2] = {wv.z, wv.w};
        mma16816(acc[j], a_s0, b_s0);
        mma16816(acc[j], a_s1, b_s1);
      }
    }
    // D fragment: rows g, g+8; columns 2t, 2t+1 of each n8 tile
    float* rb = red + (size_t)(it & 1) * SK_WARPS * 16 * SK_CW;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float* r0 = rb + ((size_t)warp * 16 + g) * SK_CW + 8 * j + 2 * t;
      float* r1 = rb + ((size_t)warp * 16 + g + 8) * SK_CW + 8 * j + 2 * t;
      r0[0] = acc[j][0];
      r0[1] = acc[j][1];
      r1[0] = acc[j][2];
      r1[1] = acc[j][3];
    }
    __syncthreads();
    // the stage is free: it takes item i + ns * step
    if (threadIdx.x == 0) {
      const int ni = i + p.ns * step;
      if (ni < p.items) sk_issue(p, stages, full, ni, s);
    }
    // the 16 warps' partial sums in warp order, one output per thread
    const int m = threadIdx.x / SK_CW, nn = threadIdx.x % SK_CW, n = n0 + nn;
    float v = 0.f;
    if (threadIdx.x < 16 * SK_CW) {
#pragma unroll
      for (int w = 0; w < SK_WARPS; ++w) v += rb[((size_t)w * 16 + m) * SK_CW + nn];
    }
    if (p.nks == 1) {
      if (threadIdx.x < 16 * SK_CW && m < p.M && n < p.N) sk_store(p, m, n, v);
      continue;
    }
    if (threadIdx.x < 16 * SK_CW && n < p.N) p.part[((size_t)kr * 16 + m) * p.N + n] = v;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.cnt + cb, 1) == p.nks - 1;
    __syncthreads();
    if (s_last) {  // every k-range of this column block is in part: add them in order
      __threadfence();
      if (threadIdx.x < 16 * SK_CW && m < p.M && n < p.N) {
        float sum = 0.f;
        for (int r = 0; r < p.nks; ++r) sum += __ldcg(p.part + ((size_t)r * 16 + m) * p.N + n);
        sk_store(p, m, n, sum);
      }
      if (threadIdx.x == 0) p.cnt[cb] = 0;
    }
  }
}

struct SkShape {
  int ncb, nks, KC, row_bytes, stage_bytes, ns, whole;
};

// whole: packed rows (ldw == K) in a single k-range, staged as one copy per
// item with unpadded rows (the fragment reads then meet 2-way bank conflicts
// when 2K is a multiple of 128, a few per item; one copy per item costs far
// less than sixteen)
SkShape sk_shape(int N, int K, long long ldw) {
  SkShape sh;
  sh.ncb = (N + SK_CW - 1) / SK_CW;
  sh.nks = (K + SK_KC_MAX - 1) / SK_KC_MAX;
  sh.KC = ((K + sh.nks - 1) / sh.nks + 63) / 64 * 64;
  if (sh.KC > SK_KC_MAX) sh.KC = SK_KC_MAX;
  sh.whole = sh.nks == 1 && ldw == K;
  sh.row_bytes = sh.whole ? 2 * K : 2 * sh.KC + SK_PAD;
  sh.stage_bytes = SK_CW * sh.row_bytes;
  sh.ns = (SK_SMEM_MAX - SK_RED_BYTES - 256) / sh.stage_bytes;
  if (sh.ns > 4) sh.ns = 4;
  return sh;
}

}  // namespace

bool skinny_gemm_supports(int M, int N, int K, long long lda, long long ldw, const void* A, const void* W) {
  return M >= 1 && M <= 16 && N >= 1 && K >= 32 && K % 32 == 0 && lda % 8 == 0 && ldw % 8 == 0 &&
         (reinterpret_cast<uintptr_t>(A) & 15) == 0 && (reinterpret_cast<uintptr_t>(W) & 15) == 0;
}

size_t skinny_scratch_floats(int N, int K) {
  const SkShape sh = sk_shape(N, K, K);
  return sh.nks > 1 ? (size_t)sh.nks * 16 * N : 0;
}

int skinny_counters(int N) { return (N + SK_CW - 1) / SK_CW; }

bool skinny_gemm_norm_ok(int N, int K) { return sk_shape(N, K, K).nks == 1; }

cudaError_t skinny_gemm(const bf16* A, long long lda, const bf16* W, long long ldw, float* C, long long ldc, int M,
                        int N, int K, float alpha, float beta, int sms, cudaStream_t s, bf16* relu2, float* part,
                        int* cnt, int* status, const float* xres) {
  const SkShape sh = sk_shape(N, K, ldw);
  if (sh.ns < 1) return cudaErrorNotSupported;
  if (sh.nks > 1 && (!part || !cnt)) return cudaErrorInvalidValue;
  if (xres && sh.nks > 1) return cudaErrorNotSupported;  // the row norm needs the whole row in one k-range
  SkParams p;
  p.A = A; p.xres = xres; p.W = W; p.C = C; p.relu2 = relu2; p.part = part; p.cnt = cnt; p.status = status;
  p.lda = lda; p.ldw = ldw; p.ldc = ldc;
  p.M = M; p.N = N; p.K = K; p.alpha = alpha; p.beta = beta;
  p.ncb = sh.ncb; p.nks = sh.nks; p.KC = sh.KC; p.items = sh.ncb * sh.nks;
  p.ns = sh.ns; p.row_bytes = sh.row_bytes; p.stage_bytes = sh.stage_bytes; p.whole = sh.whole;
  const int smem = sh.ns * sh.stage_bytes + SK_RED_BYTES + 8 * sh.ns;
  // the dynamic shared-memory limit is a per-device function attribute: raised
  // when a launch needs more than the device's setting so far
  static int attr_dev = -1, attr_bytes = 0;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev != attr_dev || smem > attr_bytes) {
    e = cudaFuncSetAttribute(skinny_gemm_k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
    attr_bytes = smem;
  }
  const int grid = p.items < sms ? p.items : sms;
  skinny_gemm_k<<<grid, SK_THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace nc
