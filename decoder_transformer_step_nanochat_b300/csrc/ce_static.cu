// Fused lm_head + cross-entropy forward that allocates no device memory.
//
// Who needs it: callers that may not call cudaMalloc at the point where they
// need the loss -- code running inside another framework's memory pool or
// under a strict memory budget, or code that must not trigger allocation on
// its hot path. nc_op_lmhead_ce_fwd takes its scratch (the per-vocabulary-tile
// softmax partials) from a context workspace, and setting up a context
// allocates (nc_configure); this entry point needs neither.
//
// Its scratch is the file-scope device array below: every GPU that loads the
// library holds these 16 MiB until the process exits. Host code must not pass
// the array's name to a kernel (on the host it is a stand-in symbol, not a
// device address); the device address is looked up once per device with
// cudaGetSymbolAddress and cached.
#include <mutex>

#include "../../include/nc.h"
#include "../../include/nc_ops.h"
#include "ops.cuh"

namespace nc {
nc_status set_last_error(nc_status st, const char* msg);

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_ce_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_ce_scratch on the current device (set-up on first use).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ce_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace nc

using namespace nc;

extern "C" nc_status nc_lmhead_ce_fwd_static(const void* hf, const void* w_lm, const int32_t* tgt, int M, int d,
                                             int V, float* lse, float* nll, int32_t* argmax, int32_t* d_status,
                                             void* cuda_stream) {
  if (!hf || !w_lm || !tgt || !lse || !nll || !argmax)
    return set_last_error(NC_ERR_ARG, "nc_lmhead_ce_fwd_static: null pointer argument");
  if (M < 0 || d < 1 || V < 1 || d % 8 != 0 || V % 8 != 0)
    return set_last_error(NC_ERR_ARG, "nc_lmhead_ce_fwd_static: need M >= 0 and d, V positive multiples of 8");
  if (M == 0) return NC_OK;
  const size_t tiles = (size_t)(V + 127) / 128;
  const size_t part = align256((size_t)M * tiles * 4);
  const size_t need = 3 * part + align256((size_t)M * 4);
  if (need > kStaticScratchBytes)
    return set_last_error(NC_ERR_UNSUPPORTED,
                          "nc_lmhead_ce_fwd_static: M * (12 * ceil(V/128) + 4) bytes of scratch exceed the "
                          "16 MiB static buffer (at V = 65536 at most 2728 rows per call)");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess)
    return set_last_error(NC_ERR_CUDA, "nc_lmhead_ce_fwd_static: cudaGetSymbolAddress of the static scratch failed");
  char* b = static_cast<char*>(base);
  GemmArgs g;
  g.M = M; g.N = V; g.K = d;
  g.A = hf; g.lda = d; g.a_kmajor = 1;
  g.B = w_lm; g.ldb = d; g.b_kmajor = 1;
  g.epi = EPI_CE_FWD;
  g.row_i = tgt;
  g.p_max = reinterpret_cast<float*>(b);
  g.p_sum = reinterpret_cast<float*>(b + part);
  g.p_arg = reinterpret_cast<int*>(b + 2 * part);
  g.p_tgt = reinterpret_cast<float*>(b + 3 * part);
  g.status = d_status;
  if (!gemm_tc_supports(g))
    return set_last_error(NC_ERR_UNSUPPORTED, "nc_lmhead_ce_fwd_static: hf and w_lm must be 16-byte aligned");
  // The target logit is written only by the tile that holds the target; clear
  // it so that an out-of-range target cannot pick up a previous call's value.
  if (cudaMemsetAsync(g.p_tgt, 0, (size_t)M * 4, s) != cudaSuccess ||
      (d_status && cudaMemsetAsync(d_status, 0, sizeof(int32_t), s) != cudaSuccess) ||
      check_ids(tgt, M, 0, V, d_status, s) != cudaSuccess || gemm_tc(g, s) != cudaSuccess ||
      ce_reduce_partials(g.p_max, g.p_sum, g.p_arg, g.p_tgt, tgt, (int)tiles, lse, nll, argmax, M, s) != cudaSuccess)
    return set_last_error(NC_ERR_CUDA, "nc_lmhead_ce_fwd_static: a kernel launch failed");
  return NC_OK;
}
