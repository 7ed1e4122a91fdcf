// Weight-streaming products of the decode step: C[m, n] = alpha * sum_k A[m, k] W[n, k]
// (+ beta * C) for at most 16 rows m (one token per sequence), bf16 operands,
// fp32 output. The product is bound by streaming W once from HBM (2 bytes per
// weight for 2 * rows FLOPs), so it runs on the warp-level tensor-core MMA
// (m16n8k16, fp32 accumulate) with W read straight from global memory in
// 16-byte pieces: a lane loads 8 consecutive k of one W row, which form the
// two k16 fragments of one 32-wide k chunk under a fixed permutation of k
// inside the chunk (the sum over k does not depend on its order); the rows of
// A use the same permutation. A CTA owns 8 * NT columns (NT n8 tiles) and its
// 16 warps take the 32-wide k chunks round robin; the warps' partial sums are
// added in shared memory in a fixed order (deterministic), so each product is
// one launch. NT is chosen per product so that the CTAs cover the SMs. The
// MLP up-projection may leave as relu(u)^2 in bf16 directly.
#include "ops.cuh"

namespace nc {
namespace {

constexpr int SK_WARPS = 16;
constexpr int SK_UNROLL = 4;  // 32-wide k chunks per round (loads in flight)

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <int NT>
__global__ void __launch_bounds__(32 * SK_WARPS)
    skinny_gemm_k(const bf16* __restrict__ A, long long lda, const bf16* __restrict__ W, long long ldw, float* C,
                  long long ldc, int M, int N, int K, float alpha, float beta, bf16* __restrict__ relu2) {
  constexpr int CW = 8 * NT;  // columns of this CTA
  __shared__ float red[SK_WARPS][16][CW];
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.x * CW;
  const int nchunks = K / 32;
  // this lane's W rows (one per n8 tile) and A rows (g, g + 8; zero beyond M)
  const bf16* wrow[NT];
  bool wok[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int n = n0 + 8 * j + g;
    wok[j] = n < N;
    wrow[j] = W + (size_t)(wok[j] ? n : 0) * ldw;
  }
  const bool a0ok = g < M, a1ok = g + 8 < M;
  const bf16* arow0 = A + (size_t)(a0ok ? g : 0) * lda;
  const bf16* arow1 = A + (size_t)(a1ok ? g + 8 : 0) * lda;
  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int c0 = warp; c0 < nchunks; c0 += SK_WARPS * SK_UNROLL) {
    uint4 wv[SK_UNROLL][NT], av[SK_UNROLL][2];
#pragma unroll
    for (int u = 0; u < SK_UNROLL; ++u) {
      const int ch = c0 + u * SK_WARPS;
      const bool in = ch < nchunks;
      const int k = ch * 32 + 8 * t;
#pragma unroll
      for (int j = 0; j < NT; ++j)
        wv[u][j] = (in && wok[j]) ? __ldg(reinterpret_cast<const uint4*>(wrow[j] + k)) : zero;
      av[u][0] = (in && a0ok) ? __ldg(reinterpret_cast<const uint4*>(arow0 + k)) : zero;
      av[u][1] = (in && a1ok) ? __ldg(reinterpret_cast<const uint4*>(arow1 + k)) : zero;
    }
#pragma unroll
    for (int u = 0; u < SK_UNROLL; ++u) {
      // k16 step 0 takes physical k 8t..8t+3 of the chunk, step 1 takes 8t+4..8t+7:
      // fragment registers {k 2t,2t+1} <- pieces .x/.z, {k 2t+8,2t+9} <- .y/.w
      const uint32_t a_s0[4] = {av[u][0].x, av[u][1].x, av[u][0].y, av[u][1].y};
      const uint32_t a_s1[4] = {av[u][0].z, av[u][1].z, av[u][0].w, av[u][1].w};
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const uint32_t b_s0[2] = {wv[u][j].x, wv[u][j].y};
        const uint32_t b_s1[2] = {wv[u][j].z, wv[u][j].w};
        mma16816(acc[j], a_s0, b_s0);
        mma16816(acc[j], a_s1, b_s1);
      }
    }
  }
  // D fragment: rows g, g+8; columns 2t, 2t+1 of each n8 tile
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    red[warp][g][8 * j + 2 * t] = acc[j][0];
    red[warp][g][8 * j + 2 * t + 1] = acc[j][1];
    red[warp][g + 8][8 * j + 2 * t] = acc[j][2];
    red[warp][g + 8][8 * j + 2 * t + 1] = acc[j][3];
  }
  __syncthreads();
  // the 16 warps' partial sums in warp order, one output per thread
  for (int i = threadIdx.x; i < 16 * CW; i += 32 * SK_WARPS) {
    const int m = i / CW, nn = i % CW, n = n0 + nn;
    if (m >= M || n >= N) continue;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < SK_WARPS; ++w) s += red[w][m][nn];
    if (relu2) {
      const float u = fmaxf(alpha * s, 0.f);
      relu2[(size_t)m * ldc + n] = __float2bfloat16_rn(u * u);
      continue;
    }
    float* c = C + (size_t)m * ldc + n;
    *c = beta != 0.f ? alpha * s + beta * *c : alpha * s;
  }
}

}  // namespace

bool skinny_gemm_supports(int M, int N, int K, long long lda, long long ldw, const void* A, const void* W) {
  return M >= 1 && M <= 16 && N >= 1 && K >= 32 && K % 32 == 0 && lda % 8 == 0 && ldw % 8 == 0 &&
         (reinterpret_cast<uintptr_t>(A) & 15) == 0 && (reinterpret_cast<uintptr_t>(W) & 15) == 0;
}

cudaError_t skinny_gemm(const bf16* A, long long lda, const bf16* W, long long ldw, float* C, long long ldc, int M,
                        int N, int K, float alpha, float beta, int sms, cudaStream_t s, bf16* relu2) {
  // the widest column group that still gives every SM a CTA
  const int nt = (N + 31) / 32 >= sms ? 4 : ((N + 15) / 16 >= sms ? 2 : 1);
  const int cw = 8 * nt;
  const int blocks = (N + cw - 1) / cw;
  if (nt == 4)
    skinny_gemm_k<4><<<blocks, 32 * SK_WARPS, 0, s>>>(A, lda, W, ldw, C, ldc, M, N, K, alpha, beta, relu2);
  else if (nt == 2)
    skinny_gemm_k<2><<<blocks, 32 * SK_WARPS, 0, s>>>(A, lda, W, ldw, C, ldc, M, N, K, alpha, beta, relu2);
  else
    skinny_gemm_k<1><<<blocks, 32 * SK_WARPS, 0, s>>>(A, lda, W, ldw, C, ldc, M, N, K, alpha, beta, relu2);
  return cudaGetLastError();
}

}  // namespace nc
