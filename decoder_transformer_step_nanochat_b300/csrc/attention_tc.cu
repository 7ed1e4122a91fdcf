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
constexpr uint64_t kWaitNs = 2000000000ull;
// Limit of the pipeline waits (those an abort can end), in ns; kWaitNs
// unless a test lowers it through the setter below. Teardown waits (for the
// copies and products a CTA has in flight) always use kWaitNs.
__device__ uint64_t g_pipe_wait_ns = kWaitNs;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSqrt128 = 11.313708498984761f;

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

__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

// One 32-bit column of this thread's TMEM lane: store (then wait) and load.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(__float_as_uint(v)) : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
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
  const bf16* qkv;  // backward: k_hat rows for the in-kernel QK-norm/RoPE backward of k
  bf16* o;        // forward output
  float* lse;     // forward output
  const float* L2row;  // backward: -(lse * log2(e) + 3.5) per (b, h, t) (base 2, score scale folded in)
  const float* Drow;
  float* dq;      // backward: fp32 [B*T, d], accumulated with atomics (pre-zeroed)
  float* dk;      // backward: fp32 [B*T, d] (dk_hat), unless the k half is finished in-kernel
  bf16* dqkv;     // backward: dv goes to its v columns (and dk to its k columns when finished)
  // finishing the k half in-kernel (QK-norm + RoPE backward of k): needs rstd of
  // the k heads (rqk [B*T, 2H]) and the RoPE table (angle-major [16][T][4] cos / sin)
  const float* rqk;
  const float* rope_cos;
  const float* rope_sin;
  int* sched;     // backward: unit counter, zero at launch (dynamic scheduling)
  int* status;
};

// ============================================================== forward
//
// Persistent: two CTAs per SM, each taking work items (b, h, 128-query tile)
// from a global counter in (batch, head)-major order, heaviest query tile
// first within a head. The tensor cores interleave the independent products
// of the SM's two CTAs, which a single accumulator chain cannot keep busy (a
// 128x128x16 MMA issued back to back into one accumulator runs at about 58%
// of the tensor rate; two chains reach it). Eight warps: warp 0 draws the
// items and loads Q and K, warp 2 loads V, one thread of warp 1 issues the
// MMAs, warps 4-7 run the softmax with one thread per query row (TMEM lane =
// row), so a row's max and sum never leave its thread, and write O. TMEM (256
// columns per CTA, allocated once): S [0,128), with P written back over its
// first 64 columns as packed bf16 that O += P V reads straight from TMEM, and O
// [128,256). Shared memory: Q and single K and V buffers (96 KB).
//
// MMA order per item: S(0), then per key tile j >= 1: PV(j-1), S(j), then the
// last PV. A commit covers every MMA issued before it, so once S(j) is seen
// complete PV(j-1) has landed too: O is quiescent while the softmax may
// rescale it, and P(j-1) was read before S(j) overwrote it. The softmax keeps
// per row a reference maximum m (log2 units); only when a tile's maximum
// exceeds m by more than 8 does it move m up and rescale the row of O and the
// running sum. Between items: the next Q and first K load once the last S(j)
// has read Q and K, and the next item's S(0) runs while the softmax warps
// read O out; its first PV waits until they have (o_free).

constexpr float kRescaleLog2 = 8.f;
constexpr int FWD_WARPS = 8;
constexpr int FWD_THREADS = 32 * FWD_WARPS;
constexpr int FWD_SOFT = 128;
// Registers: 128 per thread at launch (two CTAs of 256 threads per SM); the
// load/MMA warpgroup drops to 56 and the softmax warpgroup rises to 200.
constexpr int FWD_REG_LAUNCH = 128, FWD_REG_LOW = 56, FWD_REG_HIGH = 200;
static_assert(128 * FWD_REG_LOW + 128 * FWD_REG_HIGH <= FWD_THREADS * FWD_REG_LAUNCH, "register split");
constexpr int FWD_KST = 1, FWD_VST = 1;

struct FwdItem {
  int b, h, qt, row0;
};
__device__ __forceinline__ FwdItem fwd_item(const AttnParams& p, int v) {
  FwdItem it;
  const int bh = v / p.nq;
  it.b = bh / p.H;
  it.h = bh % p.H;
  it.qt = p.nq - 1 - v % p.nq;
  it.row0 = it.b * p.T + it.qt * TILE;
  return it;
}

__global__ void __launch_bounds__(FWD_THREADS, 2)
    attn_fwd_tc_k(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint64_t wait_ns = g_pipe_wait_ns;
  if (tc::smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0) set_status(p.status, DEV_BAD_LAUNCH);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + TILE_BYTES;
  uint8_t* sV = sK + TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + TILE_BYTES);
  uint64_t* q_full = bars + 0;   // Q of an item landed (and the item announced)
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 2;
  uint64_t* v_full = bars + 3;
  uint64_t* v_empty = bars + 4;
  uint64_t* s_full = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* o_full = bars + 7;   // the item's last PV done
  uint64_t* drain = bars + 8;
  uint64_t* q_empty = bars + 9;  // the item's last S done (Q free)
  uint64_t* o_free = bars + 10;  // O read out (one arrival per softmax warp)
  // the V loader and each softmax warp have read the item's announcement: an
  // item's q_full phase may complete before a role that lags (behind an O
  // read-out) polls it, so the next phase waits for all of them
  uint64_t* q_seen = bars + 11;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // item index of this CTA's i-th item at slot i % 4 (-1: no more items),
  // written before the arrival that completes that item's q_full phase
  volatile int* item_ring = reinterpret_cast<volatile int*>(tmem_holder + 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int d = p.H * 128;
  const int nitems = p.B * p.H * p.nq;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    tc::mbar_init(k_full, 1);
    tc::mbar_init(k_empty, 1);
    tc::mbar_init(v_full, 1);
    tc::mbar_init(v_empty, 1);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, FWD_SOFT / 32);  // one arrival per softmax warp
    tc::mbar_init(o_full, 1);
    tc::mbar_init(drain, 1);
    tc::mbar_init(q_empty, 1);
    tc::mbar_init(o_free, FWD_SOFT / 32);
    tc::mbar_init(q_seen, 1 + FWD_SOFT / 32);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool failed = false;
  if (warp < 4) {
    tc::setmaxnreg_dec<FWD_REG_LOW>();
    if (warp == 0 && lane == 0) {
      // ---- items, Q and K
      tc::prefetch_tmap(&tqkv);
      int jg = 0;                 // key tiles issued over all items
      int q_last = -1;            // last item whose Q load was issued
      for (int i = 0;; ++i) {
        int v = atomicAdd(p.sched, 1);
        if (v >= nitems) v = -1;
        // Q is free once the previous item's last S product is done, and the
        // next announcement waits until every role has read the previous one
        if (i > 0 && !tc::mbar_wait(q_empty, (i - 1) & 1, abort_flag, wait_ns)) { failed = true; break; }
        if (i > 0 && !tc::mbar_wait(q_seen, (i - 1) & 1, abort_flag, wait_ns)) { failed = true; break; }
        item_ring[i & 3] = v;
        if (v < 0) {
          tc::mbar_arrive(q_full);  // the end marker, on the phase every role waits on next
          break;
        }
        const FwdItem it = fwd_item(p, v);
        tc::mbar_arrive_expect_tx(q_full, TILE_BYTES);
        tc::tma_load_2d(sQ, &tqkv, it.h * 128, it.row0, q_full);
        tc::tma_load_2d(sQ + HALF_BYTES, &tqkv, it.h * 128 + 64, it.row0, q_full);
        q_last = i;
        for (int j = 0; j <= it.qt; ++j, ++jg) {
          if (!tc::mbar_wait(k_empty, (jg & 1) ^ 1, abort_flag, wait_ns)) { failed = true; break; }
          const int kr = it.b * p.T + j * TILE;
          tc::mbar_arrive_expect_tx(k_full, TILE_BYTES);
          tc::tma_load_2d(sK, &tqkv, d + it.h * 128, kr, k_full);
          tc::tma_load_2d(sK + HALF_BYTES, &tqkv, d + it.h * 128 + 64, kr, k_full);
        }
        if (failed) break;
      }
      if (failed) {
        *abort_flag = 1;
        // the copies this thread started land before the CTA exits (one Q and
        // one K buffer: only the last of each can be in flight)
        if (q_last >= 0) tc::mbar_wait(q_full, q_last & 1, nullptr, kWaitNs);
        if (jg > 0) tc::mbar_wait(k_full, (jg - 1) & 1, nullptr, kWaitNs);
      }
    } else if (warp == 2 && lane == 0) {
      // ---- V
      int jg = 0;
      for (int i = 0;; ++i) {
        if (!tc::mbar_wait(q_full, i & 1, abort_flag, wait_ns)) { failed = true; break; }
        const int v = item_ring[i & 3];
        if (v < 0) break;
        tc::mbar_arrive(q_seen);
        const FwdItem it = fwd_item(p, v);
        for (int j = 0; j <= it.qt; ++j, ++jg) {
          if (!tc::mbar_wait(v_empty, (jg & 1) ^ 1, abort_flag, wait_ns)) { failed = true; break; }
          const int kr = it.b * p.T + j * TILE;
          tc::mbar_arrive_expect_tx(v_full, TILE_BYTES);
          tc::tma_load_2d(sV, &tqkv, 2 * d + it.h * 128, kr, v_full);
          tc::tma_load_2d(sV + HALF_BYTES, &tqkv, 2 * d + it.h * 128 + 64, kr, v_full);
        }
        if (failed) break;
      }
      if (failed) {
        *abort_flag = 1;
        if (jg > 0) tc::mbar_wait(v_full, (jg - 1) & 1, nullptr, kWaitNs);
      }
    } else if (warp == 1 && lane == 0) {
      // ---- MMA issuer
      const uint32_t idesc = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t idesc_pv = tc::idesc_bf16(128, 128, 0, 1);
      bool any = false;
      int jg = 0;  // key tiles over all items (the s_full / p_full / K / V phases)
      for (int i = 0;; ++i) {
        if (!tc::mbar_wait(q_full, i & 1, abort_flag, wait_ns)) { failed = true; break; }
        const int v = item_ring[i & 3];
        if (v < 0) break;
        const int nkv = fwd_item(p, v).qt + 1;
        const int j0 = jg;  // global index of this item's first key tile
        for (int j = 0; j <= nkv && !failed; ++j) {
          if (j > 0) {  // O += P(j-1) V(j-1), P read from the first 64 columns of S
            const int gi = j0 + j - 1;
            if (!tc::mbar_wait(v_full, gi & 1, abort_flag, wait_ns)) { failed = true; break; }
            if (!tc::mbar_wait(p_full, gi & 1, abort_flag, wait_ns)) { failed = true; break; }
            // the item's first PV overwrites O: the previous item's O must be read out
            if (j == 1 && i > 0 && !tc::mbar_wait(o_free, (i - 1) & 1, abort_flag, wait_ns)) {
              failed = true;
              break;
            }
            tc::tc_fence_after();
            const uint32_t aV = tc::smem_u32(sV);
#pragma unroll
            for (int k = 0; k < TILE / 16; ++k)
              tc::mma_bf16_tmem_a(tmem + 128, tmem + k * 8, desc_mn(aV, k), idesc_pv, (j > 1 || k > 0) ? 1u : 0u);
            any = true;
            tc::mma_commit(v_empty);
          }
          if (j < nkv) {
            const int gi = j0 + j;
            if (!tc::mbar_wait(k_full, gi & 1, abort_flag, wait_ns)) { failed = true; break; }
            tc::tc_fence_after();
            mma_tile(tmem, tc::smem_u32(sQ), false, tc::smem_u32(sK), false, idesc, false);
            any = true;
            tc::mma_commit(s_full);
            tc::mma_commit(k_empty);
            if (j == nkv - 1) tc::mma_commit(q_empty);  // Q no longer read
          }
        }
        if (failed) break;
        jg = j0 + nkv;
        tc::mma_commit(o_full);
      }
      if (failed) {
        *abort_flag = 1;
        if (any) {
          tc::mma_commit(drain);
          tc::mbar_wait(drain, 0, nullptr, kWaitNs);
        }
      }
    }
  } else {
    tc::setmaxnreg_inc<FWD_REG_HIGH>();
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off, tO = tmem + 128 + lane_off;
    const float sl2 = kLog2e * rsqrtf(128.f);
    int jg = 0;
    for (int i = 0;; ++i) {
      {
        const bool ok = tc::mbar_wait(q_full, i & 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      }
      const int v = item_ring[i & 3];
      if (v < 0) break;
      tc::mbar_arrive_warp(q_seen);
      const FwdItem it = fwd_item(p, v);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j <= it.qt; ++j, ++jg) {
        bool ok = tc::mbar_wait(s_full, jg & 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        tc::tc_fence_after();
        float v128[128];
        tc::tmem_ld32x4(tS, tS + 32, tS + 64, tS + 96, v128, v128 + 32, v128 + 64, v128 + 96);
        if (j == it.qt) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > r) v128[c] = -INFINITY;
        }
        // row maximum: four chains of three-input maxima
        float mx4[4] = {v128[0], v128[1], v128[2], v128[3]};
#pragma unroll
        for (int c = 4; c < 128; c += 8) {
          mx4[0] = tc::fmax3(mx4[0], v128[c], v128[c + 4]);
          mx4[1] = tc::fmax3(mx4[1], v128[c + 1], v128[c + 5]);
          mx4[2] = tc::fmax3(mx4[2], v128[c + 2], v128[c + 6]);
          mx4[3] = tc::fmax3(mx4[3], v128[c + 3], v128[c + 7]);
        }
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
        const bool grow = mx > m + kRescaleLog2;
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? mx : m;
          const float alpha = exp2f(m - m_new);
          l *= alpha;
          m = m_new;
          if (j > 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float o[32];
              tc::tmem_ld32(tO + c * 32, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tc::tmem_st32(tO + c * 32, o);
            }
          }
        }
        // P = exp2(S * log2(e)/sqrt(128) - m) on fp32 pairs; the row sum in
        // two paired accumulators
        const uint64_t sl2x2 = tc::f2pack(sl2, sl2), nm2 = tc::f2pack(-m, -m);
        uint64_t rs2[2] = {tc::f2pack(0.f, 0.f), tc::f2pack(0.f, 0.f)};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 x = tc::f2unpack(tc::ffma2(tc::f2pack(v128[2 * c], v128[2 * c + 1]), sl2x2, nm2));
          const float e0 = tc::ex2(x.x), e1 = tc::ex2(x.y);
          rs2[c & 1] = tc::fadd2(rs2[c & 1], tc::f2pack(e0, e1));
          __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
          pk[c] = *reinterpret_cast<uint32_t*>(&h2);
        }
        const float2 ra = tc::f2unpack(rs2[0]), rb = tc::f2unpack(rs2[1]);
        l += (ra.x + ra.y) + (rb.x + rb.y);
        tc::tmem_st32(tS, reinterpret_cast<const float*>(pk));
        tc::tmem_st32(tS + 32, reinterpret_cast<const float*>(pk + 32));
        tc::tc_fence_before();
        tc::mbar_arrive_warp(p_full);
      }
      if (failed) break;
      // ---- O of this item: normalise and store; then O may take the next item's products
      bool ok = tc::mbar_wait(o_full, i & 1, abort_flag, wait_ns);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      tc::tc_fence_after();
      const float inv = 1.f / l;
      bf16* orow = p.o + (size_t)(it.row0 + r) * d + it.h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tc::tmem_ld32(tO + c * 32, o);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float w8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w8[e] = o[g * 8 + e] * inv;
          *reinterpret_cast<uint4*>(orow + c * 32 + g * 8) = pack8(w8);
        }
      }
      p.lse[((size_t)it.b * p.H + it.h) * p.T + it.qt * TILE + r] = (m + log2f(l)) * kLn2;
      tc::tc_fence_before();
      tc::mbar_arrive_warp(o_free);
    }
    if (failed) *abort_flag = 1;
  }

  if (failed) set_status(p.status, DEV_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 256);
  }
}

// ============================================================== backward
//
// Persistent: one CTA per SM takes work units (b, h, 128-key tile) from a
// global counter in (batch, head)-major order, heaviest key tile first within
// a head, so the CTAs running together share a few heads' Q, dO and dq rows
// in L2 and finish together. The producer thread draws each unit and hands
// its index to the other roles through a shared-memory ring. 10 warps: TMA
// producer, MMA issuer and eight softmax/epilogue warps; warps 2-5 work on
// query columns 0-63 of each query tile and warps 6-9 on columns 64-127, one
// key row per thread (TMEM lane).
//
// TMEM: S^T [0,128) and dP^T [128,256) of one 128-query tile; the P^T of
// query half h is written back packed (bf16 pairs) over columns 64h..64h+31
// of S^T and feeds dV from TMEM; dQ^T (= K^T dS^T, head dimension in the
// TMEM lane) replaces dP^T; dV [256,384) and dK [384,512) accumulate over the
// unit. Shared memory: K, V, two Q/dO stages (the next query tile loads while
// this one computes, across units too) and dS^T. Once a tile's products are
// complete its Q/dO stage (64 KB) stages the tile's dQ for the reduce-adds,
// and the softmax warps, not the tensor cores, hand the stage back to the
// producer when those have read it.
//
// Per query tile: S^T = K Q^T and dP^T = V dO^T, two accumulator chains of
// 128x128x16 products interleaved; P'^T = exp2(S^T log2(e)/sqrt(128) - L2)
// and dS'^T = P'^T (dP^T - D) by the softmax warps (paired fp32 arithmetic),
// where L2 = lse log2(e) + 3.5 (stored negated) makes P' = P/sqrt(128), so dS' = dS/sqrt(128) already carries the score
// scale of dQ and dK (dV, accumulated from P', is multiplied back by sqrt(128)
// once per unit); then dQ^T = K^T dS'^T interleaved with the first halves
// of dV += P'^T dO and dK += dS'^T Q, and the second halves of dV and dK as
// two chains while dQ^T is read out. The tensor cores keep a single
// accumulator chain of small products far below their rate (each product
// waits on the previous one), so every phase runs two or three independent
// chains of N = 128 products. dQ^T is read out (its TMEM columns released at
// once), staged transposed and added to the fp32 dq plane with one bulk tensor
// reduce-add per warp, without waiting for it. The tensor memory accelerator
// serves both these reduce-adds and the Q/dO loads; an 8 KB reduce-add reads
// its staging block only after a few thousand cycles.
// Between units, the next K/V load as soon as the finished unit's products are
// done and its first query tile runs while the epilogue warps drain dV/dK;
// only its first dV/dK products wait for that drain.

// Warm L2 with a tile the kernel will load later (no shared memory written,
// nothing to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

constexpr int BWD_WARPS = 10;
constexpr int BWD_THREADS = 32 * BWD_WARPS;
constexpr int BWD_SOFT = 32 * (BWD_WARPS - 2);  // 256 softmax threads

struct BwdUnit {
  int b, h, kt, nit, krow0;
};
__device__ __forceinline__ BwdUnit bwd_unit(const AttnParams& p, int v) {
  BwdUnit u;
  const int bh = v / p.nq;
  u.b = bh / p.H;
  u.h = bh % p.H;
  u.kt = v % p.nq;  // within a head the key tiles with the most query tiles come first
  u.nit = p.nq - u.kt;
  u.krow0 = u.b * p.T + u.kt * TILE;
  return u;
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_tc_k(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdkv,
                  const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint64_t wait_ns = g_pipe_wait_ns;
  if (tc::smem_u32(smem_raw) & 1023) {  // see the forward kernel
    if (threadIdx.x == 0) set_status(p.status, DEV_BAD_LAUNCH);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem;
  uint8_t* sV = sK + TILE_BYTES;
  uint8_t* sQ = sV + TILE_BYTES;      // 2 stages
  uint8_t* sdO = sQ + 2 * TILE_BYTES; // 2 stages
  uint8_t* sdSt = sdO + 2 * TILE_BYTES;
  float* sLD = reinterpret_cast<float*>(sdSt + TILE_BYTES);  // [stage][lse 128 | D 128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sLD + 2 * 2 * TILE);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;    // [2]
  uint64_t* q_empty = bars + 4;   // [2]: the stage's dq staging was read (one arrival per softmax warp)
  uint64_t* st_full = bars + 6;   // S^T and dP^T of the query tile complete
  uint64_t* p_full = bars + 8;    // P^T in TMEM and dS^T in shared memory (every softmax warp)
  uint64_t* dq_full = bars + 10;  // dQ^T of the tile complete
  uint64_t* tm_free = bars + 12;  // dQ^T read out of TMEM (every softmax warp)
  uint64_t* acc_full = bars + 14;
  uint64_t* acc_free = bars + 15;
  uint64_t* drain = bars + 16;
  uint64_t* tile_done = bars + 17;  // every product of the tile complete (its Q/dO stage unread)
  uint64_t* pair = bars + 22;       // [4]: the two warps (one per warpgroup) of a 32-row block
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // unit index of this CTA's ul-th unit at slot ul % 4 (-1: no more units); it
  // is written before the arrive that completes that unit's kv_full phase
  // (and, for the end marker, a q_full phase), so a waiter on those sees it
  volatile int* unit_ring = reinterpret_cast<volatile int*>(tmem_holder + 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int d = p.H * 128;
  const int nunits = p.B * p.H * p.nq;

  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    tc::mbar_init(kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(q_full + s, 1);
      tc::mbar_init(q_empty + s, BWD_SOFT / 32);
    }
    tc::mbar_init(st_full, 1);
    tc::mbar_init(p_full, BWD_SOFT / 32);  // one arrival per softmax warp
    tc::mbar_init(dq_full, 1);
    tc::mbar_init(tm_free, BWD_SOFT / 32);
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(acc_free, BWD_SOFT / 32);
    tc::mbar_init(drain, 1);
    tc::mbar_init(tile_done, 1);
    for (int q = 0; q < 4; ++q) tc::mbar_init(pair + q, 2);  // one arrival per warp
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
  // S^T and dP^T: query column c at column c of each region; the P^T of
  // query half h (columns 64h..64h+63) is packed over columns 64h..64h+31 of
  // S^T; dQ^T (head dimension in the lane, query in the column) replaces dP^T
  // once the softmax has read it
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
  bool failed = false;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&tqkv);
      tc::prefetch_tmap(&tdo);
      int g = 0, ul = 0;                 // query tiles and units issued so far
      int kv_last = -1;                  // unit whose K/V were issued last
      for (;; ++ul) {
        int v = atomicAdd(p.sched, 1);
        if (v >= nunits) v = -1;
        if (v >= 0) {
          // the unit's K and V head for L2 now; their loads follow once the
          // previous unit's last products have released the buffers
          const BwdUnit un = bwd_unit(p, v);
          tma_prefetch_2d(&tqkv, d + un.h * 128, un.krow0);
          tma_prefetch_2d(&tqkv, d + un.h * 128 + 64, un.krow0);
          tma_prefetch_2d(&tqkv, 2 * d + un.h * 128, un.krow0);
          tma_prefetch_2d(&tqkv, 2 * d + un.h * 128 + 64, un.krow0);
        }
        // K and V of the previous unit are free once its last products finished
        // (and by then every role has read the older ring slots)
        if (ul > 0 && !tc::mbar_wait(kv_empty, (ul - 1) & 1, abort_flag, wait_ns)) { failed = true; break; }
        unit_ring[ul & 3] = v;
        if (v < 0) {
          // end marker: complete the phases the MMA thread (kv_full) and the
          // softmax warps (q_full of the next tile) wait on next; that query
          // stage's previous phase must be over first (its tile consumed)
          tc::mbar_arrive(kv_full);
          if (g >= 2 && !tc::mbar_wait(q_empty + (g & 1), ((g >> 1) & 1) ^ 1, abort_flag, wait_ns)) {
            failed = true;
            break;
          }
          tc::mbar_arrive(q_full + (g & 1));
          break;
        }
        const BwdUnit u = bwd_unit(p, v);
        tc::mbar_arrive_expect_tx(kv_full, 2 * TILE_BYTES);
        tc::tma_load_2d(sK, &tqkv, d + u.h * 128, u.krow0, kv_full);
        tc::tma_load_2d(sK + HALF_BYTES, &tqkv, d + u.h * 128 + 64, u.krow0, kv_full);
        tc::tma_load_2d(sV, &tqkv, 2 * d + u.h * 128, u.krow0, kv_full);
        tc::tma_load_2d(sV + HALF_BYTES, &tqkv, 2 * d + u.h * 128 + 64, u.krow0, kv_full);
        kv_last = ul;
        for (int it = 0; it < u.nit; ++it, ++g) {
          const int s = g & 1;
          const uint32_t ph = (g >> 1) & 1;
          if (!tc::mbar_wait(q_empty + s, ph ^ 1, abort_flag, wait_ns)) { failed = true; break; }
          const int qr = u.b * p.T + (u.kt + it) * TILE;
          const size_t lrow = ((size_t)u.b * p.H + u.h) * p.T + (size_t)(u.kt + it) * TILE;
          tc::mbar_arrive_expect_tx(q_full + s, 2 * TILE_BYTES + 2 * TILE * 4);
          tc::bulk_load(sLD + s * 2 * TILE, p.L2row + lrow, TILE * 4, q_full + s);
          tc::bulk_load(sLD + s * 2 * TILE + TILE, p.Drow + lrow, TILE * 4, q_full + s);
          tc::tma_load_2d(sQ + s * TILE_BYTES, &tqkv, u.h * 128, qr, q_full + s);
          tc::tma_load_2d(sQ + s * TILE_BYTES + HALF_BYTES, &tqkv, u.h * 128 + 64, qr, q_full + s);
          tc::tma_load_2d(sdO + s * TILE_BYTES, &tdo, u.h * 128, qr, q_full + s);
          tc::tma_load_2d(sdO + s * TILE_BYTES + HALF_BYTES, &tdo, u.h * 128 + 64, qr, q_full + s);
        }
        if (failed) break;
      }
      if (failed) {
        *abort_flag = 1;
        // every copy this thread started lands before the CTA exits: the last
        // K/V (unit ul) and the last two query stages
        if (kv_last >= 0) tc::mbar_wait(kv_full, kv_last & 1, nullptr, kWaitNs);
        for (int gg = (g - 2 > 0 ? g - 2 : 0); gg < g; ++gg)
          tc::mbar_wait(q_full + (gg & 1), (gg >> 1) & 1, nullptr, kWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_kk = tc::idesc_bf16(128, 128, 0, 0);    // S^T, dP^T: both K-major
      const uint32_t id_kmn = tc::idesc_bf16(128, 128, 0, 1);   // dV, dK: B MN-major
      const uint32_t id_mnmn = tc::idesc_bf16(128, 128, 1, 1);  // dQ^T: A and B MN-major
      const uint32_t aK = tc::smem_u32(sK), aV = tc::smem_u32(sV), adSt = tc::smem_u32(sdSt);
      bool any = false;
      int g = 0, ul = 0;
      for (;; ++ul) {
        if (!tc::mbar_wait(kv_full, ul & 1, abort_flag, wait_ns)) { failed = true; break; }
        const int v = unit_ring[ul & 3];
        if (v < 0) break;
        const BwdUnit u = bwd_unit(p, v);
        for (int it = 0; it < u.nit; ++it, ++g) {
          const int s = g & 1;
          const uint32_t aQ = tc::smem_u32(sQ + s * TILE_BYTES), adO = tc::smem_u32(sdO + s * TILE_BYTES);
          if (!tc::mbar_wait(q_full + s, (g >> 1) & 1, abort_flag, wait_ns)) { failed = true; break; }
          // dP^T replaces dQ^T of the previous tile: wait until it was read out
          // (S^T replaces P^T, whose reader dV was issued before, and tcgen05
          // products of one thread run in issue order)
          if (g > 0 && !tc::mbar_wait(tm_free, (g - 1) & 1, abort_flag, wait_ns)) { failed = true; break; }
          tc::tc_fence_after();
          // S^T = K Q^T and dP^T = V dO^T over the whole 128-query tile: two
          // independent accumulator chains, interleaved
#pragma unroll
          for (int k = 0; k < TILE / 16; ++k) {
            tc::mma_bf16(tS, desc_k(aK, k), desc_k(aQ, k), id_kk, k > 0 ? 1u : 0u);
            tc::mma_bf16(tdP, desc_k(aV, k), desc_k(adO, k), id_kk, k > 0 ? 1u : 0u);
          }
          any = true;
          tc::mma_commit(st_full);
          if (!tc::mbar_wait(p_full, g & 1, abort_flag, wait_ns)) { failed = true; break; }
          // the first dV/dK of a unit overwrite the accumulators of the previous
          // one: wait until the epilogue warps have read them out
          if (it == 0 && ul > 0 && !tc::mbar_wait(acc_free, (ul - 1) & 1, abort_flag, wait_ns)) {
            failed = true;
            break;
          }
          tc::tc_fence_after();
          // dQ^T = K^T dS^T (into the dP^T columns; k-steps of 16 keys) with the
          // first half of dV += P^T dO (P^T from TMEM) and dK += dS^T Q (k-steps
          // of 16 queries), three chains interleaved; then the second halves of
          // dV and dK, two chains, which run while dQ^T is read out
          const bool acc0 = it > 0;
#pragma unroll
          for (int k = 0; k < TILE / 16; ++k) {
            if (k < 4) {
              tc::mma_bf16_tmem_a(tdV, tS + k * 8, desc_mn(adO, k), id_kmn, (acc0 || k > 0) ? 1u : 0u);
              tc::mma_bf16(tdK, desc_k(adSt, k), desc_mn(aQ, k), id_kmn, (acc0 || k > 0) ? 1u : 0u);
            }
            tc::mma_bf16(tdP, desc_mn(aK, k), desc_mn(adSt, k), id_mnmn, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(dq_full);
          // the unit's last tile: nothing after dQ^T reads K or V (dV and dK read
          // P^T, dO, dS^T and Q), so the next unit's K/V may load now
          if (it + 1 == u.nit) tc::mma_commit(kv_empty);
#pragma unroll
          for (int k = 4; k < TILE / 16; ++k) {
            tc::mma_bf16_tmem_a(tdV, tS + 64 + (k & 3) * 8, desc_mn(adO, k), id_kmn, 1u);
            tc::mma_bf16(tdK, desc_k(adSt, k), desc_mn(aQ, k), id_kmn, 1u);
          }
          tc::mma_commit(tile_done);
        }
        if (failed) break;
        tc::mma_commit(acc_full);  // dV, dK of this unit complete
      }
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
    const int ch = (warp - 2) >> 2;  // the 64-query half this warp works on
    const int r = q4 * 32 + lane;    // key row of this CTA (TMEM lane; a head dimension for dQ^T)
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = kLog2e * rsqrtf(128.f);
    // this warp's 8 KB staging block for its dQ bulk reduce-add: [64 queries
    // x 32 dims] fp32 in the query tile's own Q (ch = 0) or dO (ch = 1) stage,
    // which the tile's products no longer read once dQ^T is complete
    const uint32_t stg_off = (ch ? 2 * TILE_BYTES : 0) + q4 * 8192;
    int g = 0, ul = 0;
    for (;; ++ul) {
      // the first query tile of the next unit (or the end marker) is announced
      // on that tile's q_full phase
      {
        const bool ok = tc::mbar_wait(q_full + (g & 1), (g >> 1) & 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      }
      const int v = unit_ring[ul & 3];
      if (v < 0) break;
      const BwdUnit u = bwd_unit(p, v);
      for (int it = 0; it < u.nit; ++it, ++g) {
        const int qt = u.kt + it;
        const int s = g & 1;
        const float* Lq = sLD + s * 2 * TILE + ch * 64;        // negated base-2 lse of this half's 64 query columns
        const float* Dq = sLD + s * 2 * TILE + TILE + ch * 64; // D of the same columns
        bool ok = tc::mbar_wait(st_full, g & 1, abort_flag, wait_ns);
        // the lse / D rows arrived with this tile's Q (already complete here)
        ok = ok && tc::mbar_wait(q_full + s, (g >> 1) & 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        tc::tc_fence_after();
        const bool diag = (it == 0);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float sv[32], dp[32];
          tc::tmem_ld32x2(tS + lane_off + ch * 64 + c * 32, tdP + lane_off + ch * 64 + c * 32, sv, dp);
          // P' = exp2(S * log2(e)/sqrt(128) + nL2) = P / sqrt(128): the score
          // scale rides on P' into dS' = P' (dP - D) = dS / sqrt(128); the
          // arithmetic runs on fp32 pairs
          const uint64_t sl2x2 = tc::f2pack(sl2, sl2);
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const float4 l0 = *reinterpret_cast<const float4*>(Lq + c * 32 + gq * 8);
            const float4 l1 = *reinterpret_cast<const float4*>(Lq + c * 32 + gq * 8 + 4);
            const uint64_t nl[4] = {tc::f2pack(l0.x, l0.y), tc::f2pack(l0.z, l0.w), tc::f2pack(l1.x, l1.y),
                                    tc::f2pack(l1.z, l1.w)};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i = gq * 8 + 2 * k;
              const float2 x = tc::f2unpack(tc::ffma2(tc::f2pack(sv[i], sv[i + 1]), sl2x2, nl[k]));
              sv[i] = tc::ex2(x.x);
              sv[i + 1] = tc::ex2(x.y);
            }
          }
          if (diag) {  // the diagonal tile: query q sees key r only if q >= r
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (ch * 64 + c * 32 + i < r) sv[i] = 0.f;
          }
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const float4 d0 = *reinterpret_cast<const float4*>(Dq + c * 32 + gq * 8);
            const float4 d1 = *reinterpret_cast<const float4*>(Dq + c * 32 + gq * 8 + 4);
            const uint64_t dd[4] = {tc::f2pack(d0.x, d0.y), tc::f2pack(d0.z, d0.w), tc::f2pack(d1.x, d1.y),
                                    tc::f2pack(d1.z, d1.w)};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i = gq * 8 + 2 * k;
              const float2 w = tc::f2unpack(
                  tc::fmul2(tc::f2pack(sv[i], sv[i + 1]), tc::fsub2(tc::f2pack(dp[i], dp[i + 1]), dd[k])));
              dp[i] = w.x;
              dp[i + 1] = w.y;
            }
            st_tile8(sdSt, r, ch * 8 + c * 4 + gq, pack8(dp + 8 * gq));
          }
          // P'^T of these 32 query columns -> 16 packed bf16 pairs in TMEM
          float pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(sv[2 * i], sv[2 * i + 1]);
            pk[i] = __uint_as_float(*reinterpret_cast<uint32_t*>(&h2));
          }
          tc::tmem_st16(tS + lane_off + ch * 64 + c * 16, pk);
        }
        fence_async_smem();
        tc::tc_fence_before();
        tc::mbar_arrive_warp(p_full);
        // while the tensor cores run this tile's dV/dK/dQ: the previous tile's
        // stage may take new Q/dO once this warp's dq reduce-add has read its
        // staging block there
        if (g > 0 && lane == 0) {
          tc::bulk_wait_read();
          tc::mbar_arrive(q_empty + (s ^ 1));
        }
        ok = tc::mbar_wait(dq_full, g & 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        tc::tc_fence_after();
        // dQ^T of this half: TMEM lane = head dim 32*q4 + lane, column = query
        float vq[64];
        tc::tmem_ld32x2(tdP + lane_off + ch * 64, tdP + lane_off + ch * 64 + 32, vq, vq + 32);
        // dQ^T is in registers: its TMEM columns may take the next dP^T at once,
        // while the staging and reduce-add below proceed off that path
        tc::tc_fence_before();
        tc::mbar_arrive_warp(tm_free);
        // [64 queries x 32 dims] staged transposed (128-byte swizzle) and added
        // to the dq plane by one bulk tensor reduce-add, once the tile's last
        // products no longer read its Q/dO stage
        ok = tc::mbar_wait(tile_done, g & 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        uint8_t* blk = sQ + s * TILE_BYTES + stg_off;
#pragma unroll
        for (int q = 0; q < 64; ++q)
          *reinterpret_cast<float*>(blk + q * 128 + ((((lane >> 2) ^ q) & 7) << 4) + (lane & 3) * 4) = vq[q];
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::tma_reduce_add_2d(&tdq, blk, u.h * 128 + q4 * 32, u.b * p.T + qt * TILE + ch * 64);
          tc::bulk_commit();
        }
      }
      if (failed) break;
      // ---- this unit's dK / dV, read out while the next unit's first query
      // tile already runs on the tensor cores
      bool ok = tc::mbar_wait(acc_full, ul & 1, abort_flag, wait_ns);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      tc::tc_fence_after();
      const size_t m = (size_t)u.krow0 + r;
      const int h = u.h;
      if (p.rqk) {
        // dk_hat = acc (dS' carried the score scale). With R the RoPE rotation
        // of the row's position, k_n = R^T k_hat and dk_n = R^T dk_hat, the
        // RMSNorm backward dk = rk (dk_n - k_n mean(dk_n k_n)) equals
        // rk R^T (dk_hat - k_hat mean(dk_hat k_hat)): a rotation keeps dot
        // products, so the mean needs neither the table nor a rotation.
        // Warpgroup ch finishes the rotation pairs (j, j + 64) with j in
        // [32 ch, 32 ch + 32) and dv dims [64 ch, 64 ch + 64). Both leave
        // through the idle dS^T buffer, staged bf16 in the tile layout and
        // written by tensor copies of 32 rows x 64 dims (lane 1 issues them,
        // so their completion is tracked apart from lane 0's dq reduce-adds):
        // first each warp's dV block; then, once both warps of the row block
        // have seen their dV blocks read, the dK rows of the block. The two
        // warps of a row block (one per warpgroup) meet on pair[q4] four
        // times per unit; their partial row dots pass through TMEM, each in
        // the first dV column that its writer has already read.
        const int t = u.kt * TILE + r;
        const int j0 = 32 * ch;
        const bf16* krow = p.qkv + m * 3 * d + d + h * 128;
        const uint32_t tk = tdK + lane_off;
        uint64_t* pb = pair + q4;
        const int yblk = u.krow0 + 32 * q4;  // first row of this warp's block
        uint4 klo[4], khi[4];  // k_hat dims j0..j0+31 and 64+j0..64+j0+31
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          klo[q8] = __ldg(reinterpret_cast<const uint4*>(krow + j0) + q8);
          khi[q8] = __ldg(reinterpret_cast<const uint4*>(krow + 64 + j0) + q8);
        }
        const float rk = p.rqk[m * 2 * p.H + p.H + h];
        // dV first: it needs no loads, so the k_hat row and rk arrive meanwhile
        {
          float a[32], bb[32];
          tc::tmem_ld32x2(tdV + lane_off + 64 * ch, tdV + lane_off + 64 * ch + 32, a, bb);
#pragma unroll
          for (int i = 0; i < 32; ++i) {  // dV accumulated P' = P / sqrt(128)
            a[i] *= kSqrt128;
            bb[i] *= kSqrt128;
          }
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            st_tile8(sdSt, r, 8 * ch + gq, pack8(a + 8 * gq));
            st_tile8(sdSt, r, 8 * ch + 4 + gq, pack8(bb + 8 * gq));
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 1) {
          tc::tma_store_2d(&tdkv, sdSt + ch * HALF_BYTES + q4 * 32 * 128, 2 * d + h * 128 + 64 * ch, yblk);
          tc::bulk_commit();
        }
        float glo[32], ghi[32];
        tc::tmem_ld32x2(tk + j0, tk + 64 + j0, glo, ghi);
        float part = 0.f;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float k1[8], k2[8];
          unpack8(klo[q8], k1);
          unpack8(khi[q8], k2);
#pragma unroll
          for (int i = 0; i < 8; ++i) part += glo[q8 * 8 + i] * k1[i] + ghi[q8 * 8 + i] * k2[i];
        }
        tmem_st1(tdV + lane_off + 64 * ch, part);
        tc::tc_fence_before();
        tc::mbar_arrive_warp(pb);
        ok = tc::mbar_wait(pb, 0, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        tc::tc_fence_after();
        const float po = tmem_ld1(tdV + lane_off + 64 * (1 - ch));
        // every TMEM read of the unit is done: dV/dK may take the next unit's products
        tc::tc_fence_before();
        tc::mbar_arrive_warp(acc_free);
        const float dot = ch == 0 ? part + po : po + part;
        const float dmean = dot * (1.f / 128.f);
        // the dK rows go where both warps' dV blocks were: once those are read
        if (lane == 1) tc::bulk_wait_read();
        __syncwarp();
        tc::mbar_arrive_warp(pb);
        ok = tc::mbar_wait(pb, 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        // angle-major tables [16][T][4]: angles j0..j0+31 are groups j0/4..j0/4+7,
        // and the warp's 32 positions read 512 contiguous bytes per group
        const float4* cs4 = reinterpret_cast<const float4*>(p.rope_cos) + t;
        const float4* sn4 = reinterpret_cast<const float4*>(p.rope_sin) + t;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {  // 8 rotation pairs at a time
          const float4 ca = __ldg(cs4 + (size_t)(j0 / 4 + 2 * q8) * p.T);
          const float4 cb = __ldg(cs4 + (size_t)(j0 / 4 + 2 * q8 + 1) * p.T);
          const float4 sa = __ldg(sn4 + (size_t)(j0 / 4 + 2 * q8) * p.T);
          const float4 sb = __ldg(sn4 + (size_t)(j0 / 4 + 2 * q8 + 1) * p.T);
          const float cc[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
          const float ss[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
          float k1[8], k2[8], o1[8], o2[8];
          unpack8(klo[q8], k1);
          unpack8(khi[q8], k2);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float w1 = glo[q8 * 8 + i] - k1[i] * dmean, w2 = ghi[q8 * 8 + i] - k2[i] * dmean;
            o1[i] = rk * (w1 * cc[i] + w2 * ss[i]);
            o2[i] = rk * (-w1 * ss[i] + w2 * cc[i]);
          }
          st_tile8(sdSt, r, 4 * ch + q8, pack8(o1));       // dims j0 + 8 q8 .. (first half)
          st_tile8(sdSt, r, 8 + 4 * ch + q8, pack8(o2));   // dims 64 + j0 + 8 q8 .. (second half)
        }
        fence_async_smem();
        tc::mbar_arrive_warp(pb);
        ok = tc::mbar_wait(pb, 0, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        if (ch == 0 && lane == 1) {
          tc::tma_store_2d(&tdkv, sdSt + q4 * 32 * 128, d + h * 128, yblk);
          tc::tma_store_2d(&tdkv, sdSt + HALF_BYTES + q4 * 32 * 128, d + h * 128 + 64, yblk);
          tc::bulk_commit();
          tc::bulk_wait_read();
        }
        __syncwarp();
        // the block's staging is read: the buffer may take the next dS^T
        tc::mbar_arrive_warp(pb);
        ok = tc::mbar_wait(pb, 1, abort_flag, wait_ns);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      } else {
        float* dkrow = p.dk + m * d + h * 128 + ch * 64;
        bf16* dvrow = p.dqkv + m * 3 * d + 2 * d + h * 128 + ch * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float vk[32], w[32];
          tc::tmem_ld32x2(tdK + lane_off + ch * 64 + c * 32, tdV + lane_off + ch * 64 + c * 32, vk, w);
#pragma unroll
          for (int gq = 0; gq < 8; ++gq)
            *reinterpret_cast<float4*>(dkrow + c * 32 + gq * 4) =
                make_float4(vk[gq * 4], vk[gq * 4 + 1], vk[gq * 4 + 2], vk[gq * 4 + 3]);
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] *= kSqrt128;
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) *reinterpret_cast<uint4*>(dvrow + c * 32 + gq * 8) = pack8(w + 8 * gq);
        }
        // dV/dK may take the next unit's products
        tc::tc_fence_before();
        tc::mbar_arrive_warp(acc_free);
      }
    }
    if (lane <= 1) tc::bulk_wait_all();  // this warp's dQ reduce-adds and dK/dV stores have landed
    __syncwarp();
    if (failed) *abort_flag = 1;
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

}  // namespace

cudaError_t attn_tc_set_wait_limit(uint64_t ns) {
  const uint64_t v = ns ? ns : kWaitNs;
  return cudaMemcpyToSymbol(g_pipe_wait_ns, &v, sizeof(v));
}

namespace {

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

constexpr int FWD_SMEM = (1 + FWD_KST + FWD_VST) * TILE_BYTES + 256;  // Q, K, V, barriers
constexpr int BWD_SMEM = 7 * TILE_BYTES + 2 * 2 * TILE * 4 + 256;

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
  // persistent: two CTAs per SM (at most one per item), items drawn from a
  // counter (the third device word) that starts at zero
  p.sched = status + 2;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_k, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.sched, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int items = B * H * p.nq;
  attn_fwd_tc_k<<<items < 2 * sms ? items : 2 * sms, FWD_THREADS, FWD_SMEM, s>>>(tq, p);
  return cudaGetLastError();
}

cudaError_t attn_bwd_tc(const bf16* qkv, const bf16* dout, const float* L2row, const float* Drow, float* dq,
                        float* dk, bf16* dqkv, int B, int T, int H, int* status, cudaStream_t s, const float* rqk,
                        const float* rope_cos, const float* rope_sin) {
  if (!attn_tc_supports(T)) return cudaErrorNotSupported;
  if (B * T == 0) return cudaSuccess;
  if (!encoder()) return cudaErrorNotSupported;
  CUtensorMap tq, tdo, tdq;
  if (!map_rows(&tq, qkv, 3ull * H * 128, (uint64_t)B * T)) return cudaErrorInvalidValue;
  if (!map_rows(&tdo, dout, 1ull * H * 128, (uint64_t)B * T)) return cudaErrorInvalidValue;
  {
    // dq fp32 [B*T, d]: 32-dim x 64-query boxes, 128-byte swizzle (the staging layout)
    cuuint64_t dims[2] = {(uint64_t)H * 128, (uint64_t)B * T};
    cuuint64_t strides[1] = {(uint64_t)H * 128 * 4};
    cuuint32_t box[2] = {32, 64};
    cuuint32_t es[2] = {1, 1};
    if (g_enc(&tdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, dq, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // dqkv bf16 [B*T, 3d]: 64-dim x 32-row boxes, 128-byte swizzle (the tile
  // layout), for the k and v gradients of the fused QK-norm/RoPE path
  CUtensorMap tdkv = tq;
  if (rqk) {
    cuuint64_t dims[2] = {3ull * H * 128, (uint64_t)B * T};
    cuuint64_t strides[1] = {3ull * H * 128 * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t es[2] = {1, 1};
    if (g_enc(&tdkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dqkv, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  AttnParams p{};
  p.B = B; p.T = T; p.H = H; p.nq = T / TILE;
  p.qkv = qkv;
  p.L2row = L2row; p.Drow = Drow; p.dq = dq; p.dk = dk; p.dqkv = dqkv; p.status = status;
  p.rqk = rqk; p.rope_cos = rope_cos; p.rope_sin = rope_sin;
  int* sched = status + 1;
  p.sched = sched;
  cudaError_t e = cudaMemsetAsync(dq, 0, (size_t)B * T * H * 128 * sizeof(float), s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_tc_k, cudaFuncAttributeMaxDynamicSharedMemorySize, BWD_SMEM);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (at most one per work unit), units drawn from
  // a counter that starts at zero
  e = cudaMemsetAsync(sched, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int units = B * H * p.nq;
  attn_bwd_tc_k<<<units < sms ? units : sms, BWD_THREADS, BWD_SMEM, s>>>(tq, tdo, tdq, tdkv, p);
  return cudaGetLastError();
}

}  // namespace nc
