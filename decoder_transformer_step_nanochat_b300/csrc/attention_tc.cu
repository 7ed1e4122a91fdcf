// Causal flash attention, forward and backward, on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), bf16 operands, fp32 softmax and accumulation.
//
// Layout: qkv is [B*T, 3d] (q_hat | k_hat | v, head h at columns h*128), o and
// dout are [B*T, d], lse and D are [B, H, T]. T % 128 == 0. Scale 1/sqrt(128).
//
// Every 128x128 bf16 tile sits in shared memory as two 64-column halves of
// 128 rows x 128 bytes with the 128-byte swizzle TMA applies, so one tile
// serves as a K-major operand (rows = M/N index) or as an MN-major operand
// (rows = K index) by choosing the descriptor. Softmax threads own one row
// each (TMEM lane = row) and write P / dS tiles in the same swizzled layout.
//
// Forward, one CTA per (b, h, 128-query tile): S = Q K^T into one of two TMEM
// buffers, online softmax in registers (log2 domain), P (bf16) to shared
// memory, O += P V accumulated in TMEM. Backward, one CTA per
// (b, h, 128-key tile): per query tile S^T = K Q^T and dP^T = V dO^T, then
// P^T, dS^T = P^T (dP^T - D) to shared memory, dV += P^T dO and dK += dS^T Q
// accumulate in TMEM, dQ = dS K goes to TMEM and is added to an fp32 global
// buffer with vector atomics. All waits are bounded (DEV_TIMEOUT on expiry).
#include <cudaTypedefs.h>

#include <mutex>

#include "ops.cuh"
#include "tc_ptx.cuh"

namespace nc {

namespace {

constexpr int TILE = 128;
constexpr int HALF_BYTES = TILE * 128;        // 128 rows x 128 B
constexpr int TILE_BYTES = 2 * HALF_BYTES;    // 32 KB
constexpr int NTHREADS = 192;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kstep) {
  return tc::sdesc_sw128(base + (kstep >> 2) * HALF_BYTES + (kstep & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kstep) {
  return tc::sdesc_sw128(base + kstep * 2048, HALF_BYTES, 1024);
}

// Store 8 consecutive bf16 (columns c8*8 .. c8*8+7, c8 in 0..15) of row r of a
// swizzled 128x128 tile.
__device__ __forceinline__ void st_tile8(uint8_t* tile, int r, int c8, uint4 v) {
  int half = c8 >> 3, chunk = c8 & 7;
  uint8_t* p = tile + half * HALF_BYTES + r * 128 + ((chunk ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(p) = v;
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 r;
  uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return r;
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a, bool a_mn, uint32_t b, bool b_mn,
                                         uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int k = 0; k < TILE / 16; ++k) {
    uint64_t ad = a_mn ? desc_mn(a, k) : desc_k(a, k);
    uint64_t bd = b_mn ? desc_mn(b, k) : desc_k(b, k);
    tc::mma_bf16(d_tmem, ad, bd, idesc, (accumulate || k > 0) ? 1u : 0u);
  }
}

struct AttnParams {
  int B, T, H, nq;
  bf16* o;        // forward output
  float* lse;     // forward output / backward input
  const float* Drow;
  float* dq;      // backward: fp32 [B*T, d], accumulated with atomics (pre-zeroed)
  float* dk;      // backward: fp32 [B*T, d]
  bf16* dqkv;     // backward: dv goes to its v columns
  int* status;
};

// ============================================================== forward
//
// MMA issue order per CTA: S_0, S_1, PV_0, S_2, PV_1, ... : S_{j+1} (into the
// other TMEM S buffer) runs while the softmax threads work on S_j, and PV_j
// accumulates straight into the TMEM output O. The softmax keeps, per row, a
// reference maximum m (log2 units) and exponentiates against it; only when a
// tile's maximum exceeds m by more than 8 (so p could exceed 2^8) does the
// warp move m up and rescale its rows of O and the running sum l, after the
// previous PV has landed. P_j goes to shared-memory buffer j % 2; PV_{j-2}
// (the last reader of that buffer) finished before S_j's completion fired.

constexpr float kRescaleLog2 = 8.f;

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd_tc_k(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + TILE_BYTES;          // 2 stages
  uint8_t* sV = sK + 2 * TILE_BYTES;      // 2 stages
  uint8_t* sP = sV + 2 * TILE_BYTES;      // 2 buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * TILE_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;    // [2]
  uint64_t* pv_done = bars + 9;
  uint64_t* o_full = bars + 10;
  uint64_t* drain = bars + 11;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int qt = p.nq - 1 - (int)(blockIdx.x / BH);  // heaviest query tiles first
  const int bh = blockIdx.x % BH, b = bh / p.H, h = bh % p.H;
  const int d = p.H * 128;
  const int row0 = b * p.T + qt * TILE;
  const int nkv = qt + 1;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(kv_full + s, 1);
      tc::mbar_init(kv_empty + s, 1);
      tc::mbar_init(s_full + s, 1);
      tc::mbar_init(p_full + s, 128);
    }
    tc::mbar_init(pv_done, 1);
    tc::mbar_init(o_full, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tO = tmem + 256;  // S buffers at columns 0 and 128
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tqkv);
      tc::mbar_arrive_expect_tx(q_full, TILE_BYTES);
      tc::tma_load_2d(sQ, &tqkv, h * 128, row0, q_full);
      tc::tma_load_2d(sQ + HALF_BYTES, &tqkv, h * 128 + 64, row0, q_full);
      bool issued[2] = {false, false};
      uint32_t iphase[2] = {0, 0};
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!tc::mbar_wait(kv_empty + s, ph ^ 1, abort_flag, kWaitNs)) { failed = true; break; }
        const int kr = b * p.T + j * TILE;
        tc::mbar_arrive_expect_tx(kv_full + s, 2 * TILE_BYTES);
        tc::tma_load_2d(sK + s * TILE_BYTES, &tqkv, d + h * 128, kr, kv_full + s);
        tc::tma_load_2d(sK + s * TILE_BYTES + HALF_BYTES, &tqkv, d + h * 128 + 64, kr, kv_full + s);
        tc::tma_load_2d(sV + s * TILE_BYTES, &tqkv, 2 * d + h * 128, kr, kv_full + s);
        tc::tma_load_2d(sV + s * TILE_BYTES + HALF_BYTES, &tqkv, 2 * d + h * 128 + 64, kr, kv_full + s);
        issued[s] = true;
        iphase[s] = ph;
      }
      if (failed) {
        *abort_flag = 1;
        tc::mbar_wait(q_full, 0, nullptr, kWaitNs);
        for (int s = 0; s < 2; ++s)
          if (issued[s]) tc::mbar_wait(kv_full + s, iphase[s], nullptr, kWaitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t idesc_pv = tc::idesc_bf16(128, 128, 0, 1);
      const uint32_t aQ = tc::smem_u32(sQ);
      bool any = false;
      if (!tc::mbar_wait(q_full, 0, abort_flag, kWaitNs)) failed = true;
      // PV_i = P_i V_i accumulated into O, once the softmax threads released P_i
      auto issue_pv = [&](int i) -> bool {
        const int s = i & 1;
        if (!tc::mbar_wait(p_full + s, (i >> 1) & 1, abort_flag, kWaitNs)) return false;
        tc::tc_fence_after();
        mma_tile(tO, tc::smem_u32(sP + s * TILE_BYTES), false, tc::smem_u32(sV + s * TILE_BYTES), true, idesc_pv,
                 i > 0);
        tc::mma_commit(pv_done);
        tc::mma_commit(kv_empty + s);
        return true;
      };
      for (int j = 0; j < nkv && !failed; ++j) {
        const int s = j & 1;
        if (!tc::mbar_wait(kv_full + s, (j >> 1) & 1, abort_flag, kWaitNs)) { failed = true; break; }
        tc::tc_fence_after();
        // S_j into buffer s: its previous reader (softmax of S_{j-2}) released
        // it before PV_{j-2} was issued.
        mma_tile(tmem + s * 128, aQ, false, tc::smem_u32(sK + s * TILE_BYTES), false, idesc, false);
        tc::mma_commit(s_full + s);
        any = true;
        if (j > 0 && !issue_pv(j - 1)) { failed = true; break; }
      }
      if (!failed && !issue_pv(nkv - 1)) failed = true;
      if (!failed) tc::mma_commit(o_full);
      if (failed) {
        *abort_flag = 1;
        if (any) {
          tc::mma_commit(drain);
          tc::mbar_wait(drain, 0, nullptr, kWaitNs);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = kLog2e * rsqrtf(128.f);
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nkv; ++j) {
      const int s = j & 1;
      bool ok = tc::mbar_wait(s_full + s, (j >> 1) & 1, abort_flag, kWaitNs);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      tc::tc_fence_after();
      const bool diag = (j == qt);
      float v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(tmem + s * 128 + lane_off + c * 32, v + c * 32);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        v[i] *= sl2;
        if (!diag || i <= r) mx = fmaxf(mx, v[i]);
      }
      const bool grow = mx > m + kRescaleLog2;
      if (__any_sync(0xffffffffu, grow)) {
        // move this warp's reference maxima up; rows of O that already hold
        // partial sums are rescaled once the previous PV has landed
        const float m_new = grow ? mx : m;
        const float alpha = exp2f(m - m_new);  // 0 for the first tile (m = -inf)
        l *= alpha;
        m = m_new;
        if (j > 0) {
          ok = tc::mbar_wait(pv_done, (j - 1) & 1, abort_flag, kWaitNs);
          if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float o[32];
            tc::tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tc::tmem_st32(tO + lane_off + c * 32, o);
          }
        }
      }
      float rs = 0.f;
      uint8_t* pbuf = sP + s * TILE_BYTES;
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        float e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int k = g * 8 + i;
          e[i] = (!diag || k <= r) ? exp2f(v[k] - m) : 0.f;
          rs += e[i];
        }
        st_tile8(pbuf, r, g, pack8(e));
      }
      l += rs;
      fence_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(p_full + s);
    }
    if (!failed) {
      bool ok = tc::mbar_wait(o_full, 0, abort_flag, kWaitNs);
      if (!__all_sync(0xffffffffu, ok)) failed = true;
    }
    if (!failed) {
      tc::tc_fence_after();
      const float inv = 1.f / l;
      bf16* orow = p.o + (size_t)(row0 + r) * d + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tc::tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float w8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w8[i] = o[g * 8 + i] * inv;
          *reinterpret_cast<uint4*>(orow + c * 32 + g * 8) = pack8(w8);
        }
      }
      p.lse[((size_t)b * p.H + h) * p.T + qt * TILE + r] = (m + log2f(l)) * kLn2;
    } else {
      *abort_flag = 1;
    }
  }

  if (failed) set_status(p.status, DEV_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ============================================================== backward

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_tc_k(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + TILE_BYTES;
  uint8_t* sQ = sV + TILE_BYTES;
  uint8_t* sdO = sQ + TILE_BYTES;
  uint8_t* sPt = sdO + TILE_BYTES;
  uint8_t* sdSt = sPt + TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sdSt + TILE_BYTES);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = bars + 2;
  uint64_t* st_full = bars + 3;
  uint64_t* p_full = bars + 4;
  uint64_t* dq_full = bars + 5;
  uint64_t* tm_free = bars + 6;
  uint64_t* acc_full = bars + 7;
  uint64_t* drain = bars + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 9);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int kt = (int)(blockIdx.x / BH);  // key tile; small kt has the most query tiles
  const int bh = blockIdx.x % BH, b = bh / p.H, h = bh % p.H;
  const int d = p.H * 128;
  const int krow0 = b * p.T + kt * TILE;
  const int nit = p.nq - kt;  // query tiles qt = kt .. nq-1

  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    tc::mbar_init(st_full, 1);
    tc::mbar_init(p_full, 128);
    tc::mbar_init(dq_full, 1);
    tc::mbar_init(tm_free, 128);
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
  const uint32_t tdQ = tS;  // S^T is consumed before dQ is formed
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tqkv);
      tc::prefetch_tmap(&tdo);
      tc::mbar_arrive_expect_tx(kv_full, 2 * TILE_BYTES);
      tc::tma_load_2d(sK, &tqkv, d + h * 128, krow0, kv_full);
      tc::tma_load_2d(sK + HALF_BYTES, &tqkv, d + h * 128 + 64, krow0, kv_full);
      tc::tma_load_2d(sV, &tqkv, 2 * d + h * 128, krow0, kv_full);
      tc::tma_load_2d(sV + HALF_BYTES, &tqkv, 2 * d + h * 128 + 64, krow0, kv_full);
      int last = -1;
      for (int it = 0; it < nit; ++it) {
        if (!tc::mbar_wait(q_empty, (it & 1) ^ 1, abort_flag, kWaitNs)) { failed = true; break; }
        const int qr = b * p.T + (kt + it) * TILE;
        tc::mbar_arrive_expect_tx(q_full, 2 * TILE_BYTES);
        tc::tma_load_2d(sQ, &tqkv, h * 128, qr, q_full);
        tc::tma_load_2d(sQ + HALF_BYTES, &tqkv, h * 128 + 64, qr, q_full);
        tc::tma_load_2d(sdO, &tdo, h * 128, qr, q_full);
        tc::tma_load_2d(sdO + HALF_BYTES, &tdo, h * 128 + 64, qr, q_full);
        last = it;
      }
      if (failed) {
        *abort_flag = 1;
        tc::mbar_wait(kv_full, 0, nullptr, kWaitNs);
        if (last >= 0) tc::mbar_wait(q_full, last & 1, nullptr, kWaitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_kk = tc::idesc_bf16(128, 128, 0, 0);   // both K-major
      const uint32_t id_kmn = tc::idesc_bf16(128, 128, 0, 1);  // B MN-major
      const uint32_t id_mnmn = tc::idesc_bf16(128, 128, 1, 1); // A and B MN-major
      const uint32_t aK = tc::smem_u32(sK), aV = tc::smem_u32(sV), aQ = tc::smem_u32(sQ);
      const uint32_t adO = tc::smem_u32(sdO), aPt = tc::smem_u32(sPt), adSt = tc::smem_u32(sdSt);
      bool any = false;
      if (!tc::mbar_wait(kv_full, 0, abort_flag, kWaitNs)) failed = true;
      for (int it = 0; it < nit && !failed; ++it) {
        if (!tc::mbar_wait(q_full, it & 1, abort_flag, kWaitNs)) { failed = true; break; }
        if (it > 0 && !tc::mbar_wait(tm_free, (it - 1) & 1, abort_flag, kWaitNs)) { failed = true; break; }
        tc::tc_fence_after();
        mma_tile(tS, aK, false, aQ, false, id_kk, false);     // S^T  = K Q^T
        mma_tile(tdP, aV, false, adO, false, id_kk, false);   // dP^T = V dO^T
        tc::mma_commit(st_full);
        any = true;
        if (!tc::mbar_wait(p_full, it & 1, abort_flag, kWaitNs)) { failed = true; break; }
        tc::tc_fence_after();
        mma_tile(tdV, aPt, false, adO, true, id_kmn, it > 0);   // dV += P^T dO
        mma_tile(tdK, adSt, false, aQ, true, id_kmn, it > 0);   // dK += dS^T Q
        mma_tile(tdQ, adSt, true, aK, true, id_mnmn, false);    // dQ  = dS K
        tc::mma_commit(dq_full);
        tc::mma_commit(q_empty);
      }
      if (!failed) tc::mma_commit(acc_full);
      if (failed) {
        *abort_flag = 1;
        if (any) {
          tc::mma_commit(drain);
          tc::mbar_wait(drain, 0, nullptr, kWaitNs);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax / epilogue warps
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // key row of this CTA (and query row of the dQ tile)
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = kLog2e * rsqrtf(128.f);
    const float scale = rsqrtf(128.f);
    const size_t bhT = ((size_t)b * p.H + h) * p.T;
    for (int it = 0; it < nit; ++it) {
      const int qt = kt + it;
      const float* Lq = p.lse + bhT + qt * TILE;   // same 128 values for every thread: L1 broadcast
      const float* Dq = p.Drow + bhT + qt * TILE;
      bool ok = tc::mbar_wait(st_full, it & 1, abort_flag, kWaitNs);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      tc::tc_fence_after();
      const bool diag = (it == 0);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float sv[32], dp[32];
        tc::tmem_ld32(tS + lane_off + c * 32, sv);
        tc::tmem_ld32(tdP + lane_off + c * 32, dp);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 l0 = __ldg(reinterpret_cast<const float4*>(Lq + c * 32 + g * 8));
          const float4 l1 = __ldg(reinterpret_cast<const float4*>(Lq + c * 32 + g * 8 + 4));
          const float4 d0 = __ldg(reinterpret_cast<const float4*>(Dq + c * 32 + g * 8));
          const float4 d1 = __ldg(reinterpret_cast<const float4*>(Dq + c * 32 + g * 8 + 4));
          const float Lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
          const float Dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int qc = c * 32 + g * 8 + i;  // query column within the tile
            const bool keep = !diag || (qc >= r);
            const float pr = keep ? exp2f(fmaf(sv[g * 8 + i], sl2, -Lv[i] * kLog2e)) : 0.f;
            sv[g * 8 + i] = pr;
            dp[g * 8 + i] = pr * (dp[g * 8 + i] - Dv[i]);
          }
          st_tile8(sPt, r, c * 4 + g, pack8(sv + 8 * g));
          st_tile8(sdSt, r, c * 4 + g, pack8(dp + 8 * g));
        }
      }
      fence_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(p_full);
      ok = tc::mbar_wait(dq_full, it & 1, abort_flag, kWaitNs);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      tc::tc_fence_after();
      // dQ tile row r (query qt*128 + r): add scale * dQ into the fp32 buffer
      float* dqrow = p.dq + (size_t)(b * p.T + qt * TILE + r) * d + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tc::tmem_ld32(tdQ + lane_off + c * 32, v);
#pragma unroll
        for (int g = 0; g < 8; ++g)
          atomicAdd(reinterpret_cast<float4*>(dqrow + c * 32 + g * 4),
                    make_float4(v[g * 4] * scale, v[g * 4 + 1] * scale, v[g * 4 + 2] * scale, v[g * 4 + 3] * scale));
      }
      tc::tc_fence_before();
      tc::mbar_arrive(tm_free);
    }
    if (!failed) {
      bool ok = tc::mbar_wait(acc_full, 0, abort_flag, kWaitNs);
      if (!__all_sync(0xffffffffu, ok)) failed = true;
    }
    if (!failed) {
      tc::tc_fence_after();
      const size_t m = (size_t)krow0 + r;
      float* dkrow = p.dk + m * d + h * 128;
      bf16* dvrow = p.dqkv + m * 3 * d + 2 * d + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tc::tmem_ld32(tdK + lane_off + c * 32, v);
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<float4*>(dkrow + c * 32 + g * 4) =
              make_float4(v[g * 4] * scale, v[g * 4 + 1] * scale, v[g * 4 + 2] * scale, v[g * 4 + 3] * scale);
        tc::tmem_ld32(tdV + lane_off + c * 32, v);
#pragma unroll
        for (int g = 0; g < 4; ++g) *reinterpret_cast<uint4*>(dvrow + c * 32 + g * 8) = pack8(v + 8 * g);
      }
    } else {
      *abort_flag = 1;
    }
  }

  if (failed) set_status(p.status, DEV_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ============================================================== host side

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;

bool encoder() {
  std::call_once(g_enc_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_enc != nullptr;
}

bool map_rows(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int FWD_SMEM = 7 * TILE_BYTES + 1024 + 256;
constexpr int BWD_SMEM = 6 * TILE_BYTES + 1024 + 256;

}  // namespace

bool attn_tc_supports(int T) { return T > 0 && T % TILE == 0; }

cudaError_t attn_fwd_tc(const bf16* qkv, bf16* o, float* lse, int B, int T, int H, int* status, cudaStream_t s) {
  if (!attn_tc_supports(T)) return cudaErrorNotSupported;
  if (B * T == 0) return cudaSuccess;
  if (!encoder()) return cudaErrorNotSupported;
  CUtensorMap tq;
  if (!map_rows(&tq, qkv, 3ull * H * 128, (uint64_t)B * T)) return cudaErrorInvalidValue;
  AttnParams p{};
  p.B = B; p.T = T; p.H = H; p.nq = T / TILE;
  p.o = o; p.lse = lse; p.status = status;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_k, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
  if (e != cudaSuccess) return e;
  attn_fwd_tc_k<<<B * H * p.nq, NTHREADS, FWD_SMEM, s>>>(tq, p);
  return cudaGetLastError();
}

cudaError_t attn_bwd_tc(const bf16* qkv, const bf16* dout, const float* lse, const float* Drow, float* dq,
                        float* dk, bf16* dqkv, int B, int T, int H, int* status, cudaStream_t s) {
  if (!attn_tc_supports(T)) return cudaErrorNotSupported;
  if (B * T == 0) return cudaSuccess;
  if (!encoder()) return cudaErrorNotSupported;
  CUtensorMap tq, tdo;
  if (!map_rows(&tq, qkv, 3ull * H * 128, (uint64_t)B * T)) return cudaErrorInvalidValue;
  if (!map_rows(&tdo, dout, 1ull * H * 128, (uint64_t)B * T)) return cudaErrorInvalidValue;
  AttnParams p{};
  p.B = B; p.T = T; p.H = H; p.nq = T / TILE;
  p.lse = const_cast<float*>(lse); p.Drow = Drow; p.dq = dq; p.dk = dk; p.dqkv = dqkv; p.status = status;
  cudaError_t e = cudaMemsetAsync(dq, 0, (size_t)B * T * H * 128 * sizeof(float), s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_tc_k, cudaFuncAttributeMaxDynamicSharedMemorySize, BWD_SMEM);
  if (e != cudaSuccess) return e;
  attn_bwd_tc_k<<<B * H * p.nq, NTHREADS, BWD_SMEM, s>>>(tq, tdo, p);
  return cudaGetLastError();
}

}  // namespace nc
