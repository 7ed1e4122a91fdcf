// Plain fp32-FMA tiled GEMM: C = alpha * A B^T with either majorness for A
// and B, any sizes, and the step's epilogues. It serves the fp32 debug mode
// (every linear layer, lm_head and its backward) and is the reference shape
// of the epilogue semantics the tensor-core kernel implements.
//
// 128x128 output tile, 8-deep k slices, 256 threads, 8x8 outputs per thread
// laid out with a stride of 16 rows/columns so that shared-memory reads are
// conflict-free and epilogue stores are coalesced.
#include "ops.cuh"

namespace nc {

namespace {

constexpr int BM = 128, BN = 128, BK = 8;

template <typename T>
__device__ __forceinline__ float load_op(const T* p, long long ld, int kmajor, int r, int k, int R,
                                         int K) {
  if (r >= R || k >= K) return 0.f;
  return kmajor ? ldf(p + (size_t)r * ld + k) : ldf(p + (size_t)k * ld + r);
}

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_k(GemmArgs g) {
  __shared__ float As[BK][BM];
  __shared__ float Bs[BK][BN];
  // blockIdx.z selects one problem of a stacked batch
  const size_t bz = blockIdx.z;
  const T* A = static_cast<const T*>(g.A) + bz * g.a_brows * g.lda;
  const T* B = static_cast<const T*>(g.B) + bz * g.b_brows * g.ldb;
  const size_t c_off = bz * g.c_brows * g.ldc, c2_off = bz * g.c_brows * g.ldc2;
  int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < g.K; k0 += BK) {
    // each thread stages 4 elements of the A slice and 4 of the B slice
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int idx = threadIdx.x + 256 * e;  // 0..1023
      int r, k;
      if (g.a_kmajor) { r = idx / BK; k = idx % BK; } else { k = idx / BM; r = idx % BM; }
      As[k][r] = load_op(A, g.lda, g.a_kmajor, m0 + r, k0 + k, g.M, g.K);
      if (g.b_kmajor) { r = idx / BK; k = idx % BK; } else { k = idx / BN; r = idx % BN; }
      Bs[k][r] = load_op(B, g.ldb, g.b_kmajor, n0 + r, k0 + k, g.N, g.K);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[8], b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 8; ++j) b[j] = Bs[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int m = m0 + ty + 16 * i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int n = n0 + tx + 16 * j;
      if (n >= g.N) continue;
      float v = g.alpha * acc[i][j];
      size_t ci = c_off + (size_t)m * g.ldc + n;
      switch (g.epi) {
        case EPI_STORE:
          stf(static_cast<T*>(g.C) + ci, v);
          break;
        case EPI_STORE_F32: {
          float* c = static_cast<float*>(g.C) + ci;
          *c = (g.beta != 0.f) ? v + g.beta * *c : v;
          break;
        }
        case EPI_RELU2: {
          stf(static_cast<T*>(g.C) + ci, v);
          float u = fmaxf(v, 0.f);
          stf(static_cast<T*>(g.C2) + c2_off + (size_t)m * g.ldc2 + n, u * u);
          break;
        }
        case EPI_RELU2_BWD: {  // C2 holds a = relu(u)^2, so relu(u) = sqrt(a)
          float a = ldf(static_cast<const T*>(g.C2) + c2_off + (size_t)m * g.ldc2 + n);
          stf(static_cast<T*>(g.C) + ci, v * 2.f * sqrtf(fmaxf(a, 0.f)));
          break;
        }
        case EPI_RELU2A: {
          float u = fmaxf(v, 0.f);
          stf(static_cast<T*>(g.C) + ci, u * u);
          break;
        }
        case EPI_CE_BWD: {
          const int t = g.row_i[m];
          const float sc = t < 0 ? 0.f : (g.dscale ? *g.dscale : 1.f);  // masked rows: no gradient
          float p = expf(v - g.row_f[m]);
          stf(static_cast<T*>(g.C) + ci, (p - (n == t ? 1.f : 0.f)) * sc);
          break;
        }
        case EPI_AXPBY: {
          float c2 = ldf(static_cast<const T*>(g.C2) + c2_off + (size_t)m * g.ldc2 + n);
          stf(static_cast<T*>(g.C) + ci, v + g.beta * c2);
          break;
        }
        default:
          break;
      }
    }
  }
}

}  // namespace

template <typename T>
cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t s) {
  if (g.epi == EPI_CE_FWD || g.epi == EPI_QKNORM_ROPE) return cudaErrorNotSupported;
  if (g.batch < 1 || g.batch > 65535) return cudaErrorNotSupported;
  if (g.batch > 1 && (g.epi == EPI_CE_BWD || g.splits > 1)) return cudaErrorNotSupported;
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, g.batch);
  gemm_simt_k<T><<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

template cudaError_t gemm_simt<float>(const GemmArgs&, cudaStream_t);
template cudaError_t gemm_simt<bf16>(const GemmArgs&, cudaStream_t);

}  // namespace nc
