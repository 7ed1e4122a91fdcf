// bf16 GEMM on the 5th-generation tensor cores (tcgen05, sm_103a) with the
// step's fused epilogues: plain store, fp32 store/accumulate, ReLU^2 (u and
// relu(u)^2, or relu(u)^2 alone), ReLU^2 backward (dA * 2 sqrt(a), a loaded
// by TMA), QKV with per-head RMSNorm + RoPE, cross-entropy forward partials
// (per-row max / sum-exp / argmax / target logit over each 128-column
// vocabulary half-tile, so the logits are never written), cross-entropy
// backward (softmax - onehot), alpha acc + beta C2 (the optimizer) and the
// attention backward's row terms beside dout (rowsum(dout o) per head, o loaded
// by TMA, and the negated base-2 lse rows).
//
// Structure: persistent CTAs (one per SM), 128x256 output tiles, 64-deep k
// slices of bf16 staged by TMA into 128-byte-swizzled shared memory in an
// mbarrier ring (4 stages for single CTAs, 6 for CTA pairs); warp 0 issues TMA, one thread of warp 1 issues
// tcgen05.mma into a TMEM accumulator (two 256-column buffers, so the
// epilogue of tile i overlaps the main loop of tile i+1), warps 2..9 read the
// accumulator with tcgen05.ld (one thread per output row and 128-column half)
// and run the epilogue. Weight-gradient shapes (few output tiles, K = tokens)
// split K across CTAs; where one split's units fill the SMs the splits are
// added into C inside the kernel in split order (per-tile counters), else
// into fp32 partial slabs that a reduction kernel sums.
// CTAs run as 2-CTA clusters on vertically adjacent tiles with 2-SM products
// (tcgen05 cta_group::2): one thread of the even CTA issues 256x256x16 MMAs
// whose A rows come half from each CTA's shared memory and whose B tile is
// split by columns between them, so each SM stages and reads 32 KB per k-slice
// instead of 48 KB; each CTA's TMEM receives its own 128 rows. Both CTAs' TMA
// loads complete on the even CTA's barriers, its commits release the stages
// and accumulators in both, and the odd CTA's epilogue warps arrive on its
// accumulator-free barriers. Every wait is bounded; on timeout the kernel
// records DEV_TIMEOUT, unwinds, frees its TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "ops.cuh"
#include "tc_ptx.cuh"

namespace nc {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int NEPI_WARPS = 8;           // two per TMEM lane quadrant, each half the columns
constexpr int NTHREADS = 64 + 32 * NEPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;    // two 256-column fp32 accumulators
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait before giving up
// Limit of the pipeline waits (those an abort can end), in ns; kWaitNs
// unless a test lowers it through the setter below. Teardown waits (for the
// copies and products a CTA has in flight) always use kWaitNs.
__device__ uint64_t g_pipe_wait_ns = kWaitNs;
constexpr int STAGING_BYTES = 4096;  // per epilogue warp: 32 rows x 128 B, 128B-swizzled

// Pipeline shape per CTA: single CTAs stage A and the whole B tile (4 x 48 KB);
// a CTA pair running 2-SM products stages its own A rows and its half of B
// (6 x 32 KB).
template <int CL>
struct Pipe {
  static constexpr int STAGES = CL == 2 ? 6 : 4;
  static constexpr int B_STAGE = CL == 2 ? B_BYTES / 2 : B_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_STAGE;
};
constexpr int RING_BYTES = 6 * (A_BYTES + B_BYTES / 2);
static_assert(RING_BYTES == 4 * (A_BYTES + B_BYTES), "both pipelines use the same ring");
constexpr int SMEM_BYTES = RING_BYTES + NEPI_WARPS * STAGING_BYTES + 1024 + 256;

struct TcParams {
  GemmArgs g;
  int num_m, num_n, num_kb, total;  // total = tiles * splits work units
  int splits, kb_per_split;
  // k-splits added into C in split order inside the kernel (no partial slabs):
  // split 0 stores (or adds, beta = 1), split s > 0 adds once the tile's
  // counter shows every warp of splits 0..s-1 done; the counter of a 128-row
  // tile is left at 0 by its last writer
  int ordered;
  int* tile_done;
};

// Work unit v of a CTA (CL = 1) or of a CTA pair (CL = 2: the two CTAs of a
// cluster take vertically adjacent 128-row blocks that share the B tile):
// problem bt of a batch, row offset m0, column block nb, k-split and its
// k-blocks [kb0, kb1). Order, for L2 reuse of the operand panels: split-major
// (the units running together share one k-range), then problem, then groups
// of kGroupRows row blocks (or row pairs) that sweep every column block
// together, rows fastest. With about 74 pairs running at once, 8 rows per
// group keep the set of tiles in flight near square on the wide products
// (QKV, MLP up, lm_head), so fewer A and B panels stream at once: measured on
// the d20 step, GEMM time 74.8 ms with 16 rows, 74.3 with 8, 75.1 with 6 or 10,
// 75.2 with 32, 78.1 with 64.
constexpr int kGroupRows = 8;

template <int CL>
__device__ __forceinline__ void unit_of(const TcParams& p, int v, int rank, int& bt, int& m0, int& nb, int& split,
                                        int& kb0, int& kb1) {
  const int rows = (CL == 1) ? p.num_m : (p.num_m + 1) / 2;  // row blocks or row-block pairs
  const int tiles = rows * p.num_n;
  const int slab = v / tiles;
  split = slab / p.g.batch;
  bt = slab - split * p.g.batch;
  const int t = v % tiles;
  const int per_group = kGroupRows * p.num_n;
  const int g0 = (t / per_group) * kGroupRows;
  const int gsize = min(kGroupRows, rows - g0);
  const int w = t % per_group;
  const int r = g0 + w % gsize;
  nb = w / gsize;
  m0 = ((CL == 1) ? r : 2 * r + rank) * BM;
  kb0 = split * p.kb_per_split;
  kb1 = min(p.num_kb, kb0 + p.kb_per_split);
  if (kb1 < kb0) kb1 = kb0;
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 r;
  uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return r;
}

__device__ __forceinline__ void unpack8_bf16(uint4 r, float* v) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    float2 f = __bfloat1622float2(h);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// Epilogue for one 32-column chunk of one row. v holds alpha*acc.
template <int EPI>
__device__ __forceinline__ void epi_chunk(const GemmArgs& g, int m, int nc0, float* v) {
  if (EPI == EPI_STORE || EPI == EPI_RELU2) {
    bf16* c = static_cast<bf16*>(g.C) + (size_t)m * g.ldc + nc0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (nc0 + 8 * j < g.N) *reinterpret_cast<uint4*>(c + 8 * j) = pack8_bf16(v + 8 * j);
    if (EPI == EPI_RELU2) {
      bf16* c2 = static_cast<bf16*>(g.C2) + (size_t)m * g.ldc2 + nc0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float u = fmaxf(v[8 * j + i], 0.f);
          a[i] = u * u;
        }
        if (nc0 + 8 * j < g.N) *reinterpret_cast<uint4*>(c2 + 8 * j) = pack8_bf16(a);
      }
    }
  } else if (EPI == EPI_STORE_F32) {
    float* c = static_cast<float*>(g.C) + (size_t)m * g.ldc + nc0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (nc0 + 4 * j < g.N) {
        float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        if (g.beta != 0.f) {
          float4 p = *reinterpret_cast<const float4*>(c + 4 * j);
          o.x += g.beta * p.x; o.y += g.beta * p.y; o.z += g.beta * p.z; o.w += g.beta * p.w;
        }
        *reinterpret_cast<float4*>(c + 4 * j) = o;
      }
    }
  } else if (EPI == EPI_RELU2_BWD) {
    const bf16* u = static_cast<const bf16*>(g.C2) + (size_t)m * g.ldc2 + nc0;
    bf16* c = static_cast<bf16*>(g.C) + (size_t)m * g.ldc + nc0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (nc0 + 8 * j < g.N) {
        float uf[8], o[8];
        unpack8_bf16(*reinterpret_cast<const uint4*>(u + 8 * j), uf);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = v[8 * j + i] * 2.f * tc::sqrt_approx(fmaxf(uf[i], 0.f));
        *reinterpret_cast<uint4*>(c + 8 * j) = pack8_bf16(o);
      }
    }
  }
}

// One 32-row x 128-byte chunk of an epilogue warp goes out through its
// staging buffer: each lane writes its row's 8 16-byte pieces in the
// 128-byte swizzle the output tensor map expects, then lane 0 issues one
// bulk tensor store (or fp32 reduce-add). The buffer is reused only after the
// previous store has read it.
struct Stager {
  uint8_t* buf;
  int lane;
  __device__ __forceinline__ void begin() {
    if (lane == 0) tc::bulk_wait_read();
    __syncwarp();
  }
  __device__ __forceinline__ void put(int j, uint4 v) {
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
  }
  __device__ __forceinline__ void store(const CUtensorMap* map, int x, int y, bool add) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      if (add) tc::tma_reduce_add_2d(map, buf, x, y);
      else tc::tma_store_2d(map, buf, x, y);
      tc::bulk_commit();
    }
  }
  __device__ __forceinline__ void store3(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                       reinterpret_cast<uint64_t>(map)),
                   "r"(tc::smem_u32(buf)), "r"(x), "r"(y), "r"(z)
                   : "memory");
      tc::bulk_commit();
    }
  }
};

// Poll a tile counter (acquire, device scope) until it reaches target; gives
// up like the pipeline waits (limit or abort flag).
__device__ __forceinline__ bool wait_count(const int* ctr, int target, volatile int* abort, uint64_t limit_ns) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
  if (v >= target) return true;
  const uint64_t t0 = tc::globaltimer();
  for (uint32_t it = 1;; ++it) {
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (limit_ns < 1000 || (it & 63) == 0) {
      if (abort && *abort) return false;
      if (tc::globaltimer() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ uint4 f4u(float a, float b, float c, float d) {
  return make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c), __float_as_uint(d));
}

template <int EPI, int A_MN, int B_MN, int CL>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_k(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
              const __grid_constant__ CUtensorMap tc_, const __grid_constant__ CUtensorMap tc2,
              const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int STAGES = Pipe<CL>::STAGES, B_STAGE = Pipe<CL>::B_STAGE, STAGE_BYTES = Pipe<CL>::STAGE_BYTES;
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sStage = smem + RING_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + NEPI_WARPS * STAGING_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* c2bar = drain + 1;  // per epilogue warp: its staging buffer holds the C2 chunk it loaded
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(c2bar + NEPI_WARPS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const GemmArgs& g = p.g;
  const uint64_t wait_ns = g_pipe_wait_ns;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int rank = (CL == 2) ? (int)tc::cluster_ctarank() : 0;
  const int v_first = (CL == 2) ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const int v_step = (CL == 2) ? (int)gridDim.x / 2 : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tfull + b, 1);
      tc::mbar_init(tempty + b, CL * NEPI_WARPS);  // one arrival per epilogue warp (of both CTAs)
    }
    tc::mbar_init(drain, 1);
    for (int w = 0; w < NEPI_WARPS; ++w) tc::mbar_init(c2bar + w, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&ta);
    tc::prefetch_tmap(&tb);
  }
  if (warp == 1) {
    if (CL == 2) {
      tc::tmem_alloc_pair(tmem_holder, TMEM_COLS);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(tmem_holder, TMEM_COLS);
      tc::tmem_relinquish();
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (CL == 2) tc::cluster_sync();  // the peer's barriers exist before any load or commit reaches them
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  bool failed = false;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[STAGES];
      bool issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = false, issued_phase[s] = 0;
      for (int v = v_first; v < p.total && !failed; v += v_step) {
        int bt, m0, nb, split, kb0, kb1;
        unit_of<CL>(p, v, rank, bt, m0, nb, split, kb0, kb1);
        const int n0 = nb * BN;
        const int a_off = (int)(bt * g.a_brows), b_off = (int)(bt * g.b_brows);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(empty + stage, phase ^ 1, abort_flag, wait_ns)) { failed = true; break; }
          const int k0 = kb * BK;
          uint8_t* a = sA + stage * A_BYTES;
          uint8_t* b = sB + stage * B_STAGE;
          if (CL == 2) {
            // own A rows and own half of the B columns; both CTAs' bytes
            // complete on the even CTA's barrier, which expects them all
            if (rank == 0) tc::mbar_arrive_expect_tx(full + stage, 2 * STAGE_BYTES);
            const uint32_t bar = tc::cluster_addr(full + stage, 0);
            if (A_MN) {
              tc::tma_load_2d_pair(a, &ta, m0, k0 + a_off, bar);
              tc::tma_load_2d_pair(a + 8192, &ta, m0 + 64, k0 + a_off, bar);
            } else {
              tc::tma_load_2d_pair(a, &ta, k0, m0 + a_off, bar);
            }
            const int nh = n0 + (BN / 2) * rank;
            if (B_MN) {
              tc::tma_load_2d_pair(b, &tb, nh, k0 + b_off, bar);
              tc::tma_load_2d_pair(b + 8192, &tb, nh + 64, k0 + b_off, bar);
            } else {
              tc::tma_load_2d_pair(b, &tb, k0, nh + b_off, bar);
            }
            issued[stage] = true;
            issued_phase[stage] = phase;
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
            continue;
          }
          tc::mbar_arrive_expect_tx(full + stage, STAGE_BYTES);
          if (A_MN) {
            tc::tma_load_2d(a, &ta, m0, k0 + a_off, full + stage);
            tc::tma_load_2d(a + 8192, &ta, m0 + 64, k0 + a_off, full + stage);
          } else {
            tc::tma_load_2d(a, &ta, k0, m0 + a_off, full + stage);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < 4; ++j) tc::tma_load_2d(b + j * 8192, &tb, n0 + 64 * j, k0 + b_off, full + stage);
          } else {
            tc::tma_load_2d(b, &tb, k0, n0 + b_off, full + stage);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (failed) {
        *abort_flag = 1;
        // let every copy this CTA's barriers track land before it exits (the
        // odd CTA of a pair has none: its copies complete on the peer's)
        if (CL == 1 || rank == 0)
          for (int s = 0; s < STAGES; ++s)
            if (issued[s]) tc::mbar_wait(full + s, issued_phase[s], nullptr, kWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // (in a CTA pair, the even CTA's thread issues the 2-SM products for both)
    if (lane == 0 && (CL == 1 || rank == 0)) {
      const uint32_t idesc = tc::idesc_bf16(CL * BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int cnt = 0;
      bool any_mma = false;
      for (int v = v_first; v < p.total && !failed; v += v_step, ++cnt) {
        int bt, m0, nb, split, kb0, kb1;
        unit_of<CL>(p, v, rank, bt, m0, nb, split, kb0, kb1);
        const int ab = cnt & 1;
        const uint32_t aph = (cnt >> 1) & 1;
        if (!tc::mbar_wait(tempty + ab, aph ^ 1, abort_flag, wait_ns)) { failed = true; break; }
        tc::tc_fence_after();
        const uint32_t dtm = tmem_base + ab * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(full + stage, phase, abort_flag, wait_ns)) { failed = true; break; }
          tc::tc_fence_after();
          const uint32_t a_addr = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = tc::smem_u32(sB + stage * B_STAGE);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = A_MN ? tc::sdesc_sw128(a_addr + k * 2048, 8192, 1024)
                                     : tc::sdesc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? tc::sdesc_sw128(b_addr + k * 2048, 8192, 1024)
                                     : tc::sdesc_sw128(b_addr + k * 32, 16, 1024);
            if (CL == 2) tc::mma_bf16_pair(dtm, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            else tc::mma_bf16(dtm, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          if (CL == 2) tc::mma_commit_pair_multicast(empty + stage, 0x3);  // frees the stage in both CTAs
          else tc::mma_commit(empty + stage);
          any_mma = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (failed) break;
        if (CL == 2) tc::mma_commit_pair_multicast(tfull + ab, 0x3);  // both CTAs' accumulators
        else tc::mma_commit(tfull + ab);
      }
      if (failed) {
        *abort_flag = 1;
        if (any_mma) {
          // wait for the MMAs already issued before the TMEM is released
          if (CL == 2) tc::mma_commit_pair(drain);
          else tc::mma_commit(drain);
          tc::mbar_wait(drain, 0, nullptr, kWaitNs);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue warps
    const int q = warp & 3;            // TMEM lane quadrant this warp may read
    const int ch = (warp - 2) >> 2;    // which 128-column half of the tile
    const int row = q * 32 + lane;
    Stager stg{sStage + (warp - 2) * STAGING_BYTES, lane};
    uint32_t c2n = 0;  // C2 chunks this warp has loaded (its barrier's phase)
    int cnt = 0;
    for (int v = v_first; v < p.total && !failed; v += v_step, ++cnt) {
      int bt, m0, nb, split, kb0, kb1;
      unit_of<CL>(p, v, rank, bt, m0, nb, split, kb0, kb1);
      const int ab = cnt & 1;
      const uint32_t aph = (cnt >> 1) & 1;
      const int n0 = nb * BN + ch * (BN / 2);
      const bool ok = tc::mbar_wait(tfull + ab, aph, abort_flag, wait_ns);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; *abort_flag = 1; break; }
      tc::tc_fence_after();
      const int m = m0 + row;
      const bool row_ok = m < g.M;
      const bool have_acc = kb1 > kb0;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + ab * BN + ch * (BN / 2);
      if (EPI == EPI_CE_FWD) {
        float mx = -INFINITY, sum = 0.f, tl = 0.f;
        int arg = 0;
        const int t = row_ok ? g.row_i[m] : -1;
        for (int c = 0; c < BN / 64; ++c) {
          float v[32];
          if (have_acc) tc::tmem_ld32(taddr + c * 32, v);
          else
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          const int nc0 = n0 + c * 32;
          if (nc0 >= g.N) continue;
          float lm = -INFINITY;
          int la = nc0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x = v[i] * g.alpha;
            v[i] = x;
            if (nc0 + i < g.N && x > lm) { lm = x; la = nc0 + i; }
            if (nc0 + i == t) tl = x;
          }
          if (lm > mx) {
            sum *= __expf(mx - lm);
            mx = lm;
            arg = la;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (nc0 + i < g.N) sum += __expf(v[i] - mx);
        }
        if (row_ok && n0 < g.N) {
          const size_t pi = (size_t)(nb * 2 + ch) * g.M + m;
          g.p_max[pi] = mx;
          g.p_sum[pi] = sum;
          g.p_arg[pi] = arg;
          if (t >= n0 && t < n0 + BN / 2) g.p_tgt[m] = tl;
        }
      } else {
        // ---- outputs leave through the staging buffer as bulk tensor stores
        const int rblk_local = m0 + q * 32;  // first row of this warp's 32-row block
        const bool blk_ok = rblk_local < g.M;
        const int rblk = rblk_local + (int)(bt * g.c_brows);  // in the stacked output
        if (EPI == EPI_STORE_F32) {
          const bool direct = (p.splits == 1 && g.beta != 0.f && g.beta != 1.f);
          int* ctr = p.ordered ? p.tile_done + (m0 / BM) * p.num_n + nb : nullptr;
          if (p.ordered && split > 0) {
            // the tile's earlier splits (all NEPI_WARPS warps each) are in C
            bool got = true;
            if (lane == 0) got = wait_count(ctr, split * NEPI_WARPS, abort_flag, wait_ns);
            if (!__all_sync(0xffffffffu, __shfl_sync(0xffffffffu, got, 0))) { failed = true; *abort_flag = 1; break; }
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          for (int c = 0; c < 4; ++c) {
            float v[32];
            if (have_acc) tc::tmem_ld32(taddr + c * 32, v);
            else
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.f;
            const int nc0 = n0 + c * 32;
            if (!blk_ok || nc0 >= g.N) continue;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= g.alpha;
            if (direct) {  // general beta: read-modify-write from registers
              if (row_ok) epi_chunk<EPI>(g, m, nc0, v);
              continue;
            }
            stg.begin();
#pragma unroll
            for (int j = 0; j < 8; ++j) stg.put(j, f4u(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            if (p.ordered) stg.store(&tc_, nc0, rblk, split > 0 || g.beta == 1.f);  // in split order
            else if (p.splits > 1) stg.store3(&tc2, nc0, rblk, split);    // this split's partial slab
            else stg.store(&tc_, nc0, rblk, g.beta == 1.f);               // C = acc, or C += acc
          }
          if (p.ordered) {
            // this warp's part of the tile is in C: count it (the last writer resets the counter)
            if (lane == 0) {
              tc::bulk_wait_all();
              asm volatile("fence.proxy.async.global;" ::: "memory");
              __threadfence();
              if (atomicAdd(ctr, 1) == p.splits * NEPI_WARPS - 1) atomicExch(ctr, 0);
            }
            __syncwarp();
          }
        } else {
          // bf16 outputs: two chunks of 64 columns
          float v[128];
          if (EPI == EPI_QKNORM_ROPE) {
            if (have_acc) tc::tmem_ld32x4(taddr, taddr + 32, taddr + 64, taddr + 96, v, v + 32, v + 64, v + 96);
            else
#pragma unroll
              for (int i = 0; i < 128; ++i) v[i] = 0.f;
            if (row_ok && n0 < g.N) {
              // this warp's 128 columns are one head of q, k or v for its row:
              // q and k heads get RMSNorm (eps 1e-6) then the half-split
              // rotation by the position's angles; v heads pass through
              float ss = 0.f;
#pragma unroll
              for (int i = 0; i < 128; ++i) {
                v[i] *= g.alpha;
                ss += v[i] * v[i];
              }
              if (n0 < 2 * g.d_model) {
                const float rr = rsqrtf(ss * (1.f / 128.f) + kEps);
                const int t = m % g.seq_len;
                // angle-major table: the warp's 32 positions read 512 contiguous bytes
                const float4* cs4 = reinterpret_cast<const float4*>(g.rope_cos) + t;
                const float4* sn4 = reinterpret_cast<const float4*>(g.rope_sin) + t;
#pragma unroll
                for (int j4 = 0; j4 < 16; ++j4) {
                  const float4 c4 = __ldg(cs4 + (size_t)j4 * g.seq_len);
                  const float4 s4 = __ldg(sn4 + (size_t)j4 * g.seq_len);
                  const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                  for (int u = 0; u < 4; ++u) {
                    const int j = j4 * 4 + u;
                    const float a = v[j] * rr, b = v[j + 64] * rr;
                    v[j] = a * cc[u] - b * sv[u];
                    v[j + 64] = a * sv[u] + b * cc[u];
                  }
                }
                g.rqk[(size_t)m * (2 * g.d_model / 128) + n0 / 128] = rr;
              }
            }
          }
          float rdot = 0.f;  // EPI_ROWDOT: this row's dot over the warp's head
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            float* w = v + h2 * 64;
            const int nc0 = n0 + h2 * 64;
            const bool chunk_ok = blk_ok && nc0 < g.N;
            if ((EPI == EPI_RELU2_BWD || EPI == EPI_ROWDOT) && chunk_ok) {
              // this warp's 32 rows x 64 columns of C2 land in its staging
              // buffer by one tensor load (rows past M and columns past N read
              // as 0) while the accumulator is read: coalesced, where a row
              // per thread would cost a wavefront per 16 bytes
              stg.begin();
              if (lane == 0) {
                tc::mbar_arrive_expect_tx(c2bar + (warp - 2), 32 * 128);
                tc::tma_load_2d(stg.buf, &tc2, nc0, rblk, c2bar + (warp - 2));
              }
            }
            if (EPI != EPI_QKNORM_ROPE) {
              if (have_acc) tc::tmem_ld32x2(taddr + h2 * 64, taddr + h2 * 64 + 32, w, w + 32);
              else
#pragma unroll
                for (int i = 0; i < 64; ++i) w[i] = 0.f;
#pragma unroll
              for (int i = 0; i < 64; ++i) w[i] *= g.alpha;
            }
            if (!chunk_ok) continue;
            if (EPI == EPI_RELU2_BWD || EPI == EPI_ROWDOT) {
              const bool got = tc::mbar_wait(c2bar + (warp - 2), c2n & 1, abort_flag, wait_ns);
              ++c2n;
              if (!__all_sync(0xffffffffu, got)) {
                failed = true;
                *abort_flag = 1;
                // the tile load this warp started lands before the CTA can leave
                if (!got) tc::mbar_wait(c2bar + (warp - 2), (c2n - 1) & 1, nullptr, kWaitNs);
              }
            }
            if (EPI == EPI_ROWDOT) {
              // the row's dot of C, as it is stored (bf16), with its C2 (o) row over this head
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float of[8];
                unpack8_bf16(*reinterpret_cast<const uint4*>(stg.buf + lane * 128 + ((j ^ (lane & 7)) << 4)), of);
#pragma unroll
                for (int i = 0; i < 8; ++i) rdot += __bfloat162float(__float2bfloat16_rn(w[8 * j + i])) * of[i];
              }
            }
            if (EPI == EPI_RELU2_BWD) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float uf[8];
                unpack8_bf16(*reinterpret_cast<const uint4*>(stg.buf + lane * 128 + ((j ^ (lane & 7)) << 4)), uf);
#pragma unroll
                // C2 holds a = relu(u)^2, so relu(u) = sqrt(a)
                for (int i = 0; i < 8; ++i) w[8 * j + i] *= 2.f * tc::sqrt_approx(fmaxf(uf[i], 0.f));
              }
            } else if (EPI == EPI_RELU2A) {
#pragma unroll
              for (int i = 0; i < 64; ++i) {
                const float uu = fmaxf(w[i], 0.f);
                w[i] = uu * uu;
              }
            } else if (EPI == EPI_CE_BWD) {
              if (row_ok) {
                const float l = g.row_f[m];
                const int t = g.row_i[m];
                const float sc = t < 0 ? 0.f : (g.dscale ? *g.dscale : 1.f);  // masked rows: no gradient
#pragma unroll
                for (int i = 0; i < 64; ++i) w[i] = (__expf(w[i] - l) - (nc0 + i == t ? 1.f : 0.f)) * sc;
              }
            } else if (EPI == EPI_AXPBY) {
              if (row_ok) {
                const bf16* c2 = static_cast<const bf16*>(g.C2) + (size_t)(bt * g.c_brows + m) * g.ldc2 + nc0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  if (nc0 + 8 * j < g.N) {
                    float cf[8];
                    unpack8_bf16(*reinterpret_cast<const uint4*>(c2 + 8 * j), cf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[8 * j + i] += g.beta * cf[i];
                  }
                }
              }
            }
            stg.begin();
#pragma unroll
            for (int j = 0; j < 8; ++j) stg.put(j, pack8_bf16(w + 8 * j));
            stg.store(&tc_, nc0, rblk, false);
            if (EPI == EPI_RELU2) {  // second output a = relu(u)^2
              float a8[8];
              stg.begin();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float uu = fmaxf(w[8 * j + i], 0.f);
                  a8[i] = uu * uu;
                }
                stg.put(j, pack8_bf16(a8));
              }
              stg.store(&tc2, nc0, rblk, false);
            }
          }
          if (EPI == EPI_ROWDOT && row_ok && n0 < g.N) {  // the warp's 128 columns are one head
            const int H = g.N / 128, bq = m / g.seq_len, t = m - bq * g.seq_len;
            const size_t idx = ((size_t)bq * H + n0 / 128) * g.seq_len + t;
            g.rd_D[idx] = rdot;
            if (g.rd_L2) g.rd_L2[idx] = -fmaf(g.rd_lse[idx], 1.4426950408889634f, 3.5f);
          }
        }
      }
      tc::tc_fence_before();
      if (CL == 2) tc::mbar_arrive_warp_cluster(tc::cluster_addr(tempty + ab, 0));  // the even CTA's barrier
      else tc::mbar_arrive_warp(tempty + ab);
    }
    if (lane == 0) tc::bulk_wait_all();  // this warp's stores have landed
    __syncwarp();
  }

  if (failed) {
    set_status(g.status, DEV_TIMEOUT);
    *abort_flag = 1;
  }
  tc::tc_fence_before();
  __syncthreads();
  // neither CTA of a pair may leave (or free the TMEM) while the other can
  // still arrive on its barriers or its products still run
  if (CL == 2) tc::cluster_sync();
  if (warp == 1) {
    tc::tc_fence_after();
    if (CL == 2) tc::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

cudaError_t gemm_tc_set_wait_limit(uint64_t ns) {
  const uint64_t v = ns ? ns : kWaitNs;
  return cudaMemcpyToSymbol(g_pipe_wait_ns, &v, sizeof(v));
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
int g_num_sms = 0;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  });
  return g_encode != nullptr;
}

// 2-D bf16 tensor map: inner (contiguous) extent, outer extent, row pitch in
// elements, box of box_inner x box_outer, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t pitch,
              uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

typedef void (*KernFn)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcParams);

// Output maps: 32-row x 128-byte boxes, 128-byte swizzle (the staging layout).
bool make_out_map(CUtensorMap* m, const void* ptr, bool f32, uint64_t cols, uint64_t rows, uint64_t pitch) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch * (f32 ? 4 : 2)};
  cuuint32_t box[2] = {f32 ? 32u : 64u, 32u};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                  dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [splits, M, N] partial slabs: a 3-D map so a box is clipped at M per split.
bool make_partial_map(CUtensorMap* m, const void* ptr, uint64_t N, uint64_t M, uint64_t splits) {
  cuuint64_t dims[3] = {N, M, splits};
  cuuint64_t strides[2] = {N * 4, N * M * 4};
  cuuint32_t box[3] = {32u, 32u, 1u};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, int CL>
KernFn pick(int a_mn, int b_mn) {
  if (!a_mn && !b_mn) return gemm_tc_k<EPI, 0, 0, CL>;
  if (!a_mn && b_mn) return gemm_tc_k<EPI, 0, 1, CL>;
  if (a_mn && !b_mn) return gemm_tc_k<EPI, 1, 0, CL>;
  return gemm_tc_k<EPI, 1, 1, CL>;
}

template <int CL>
KernFn pick_kernel(int epi, int a_mn, int b_mn) {
  switch (epi) {
    case EPI_STORE: return pick<EPI_STORE, CL>(a_mn, b_mn);
    case EPI_STORE_F32: return pick<EPI_STORE_F32, CL>(a_mn, b_mn);
    case EPI_RELU2: return pick<EPI_RELU2, CL>(a_mn, b_mn);
    case EPI_RELU2_BWD: return pick<EPI_RELU2_BWD, CL>(a_mn, b_mn);
    case EPI_CE_BWD: return pick<EPI_CE_BWD, CL>(a_mn, b_mn);
    case EPI_CE_FWD: return pick<EPI_CE_FWD, CL>(a_mn, b_mn);
    case EPI_QKNORM_ROPE: return pick<EPI_QKNORM_ROPE, CL>(a_mn, b_mn);
    case EPI_AXPBY: return pick<EPI_AXPBY, CL>(a_mn, b_mn);
    case EPI_RELU2A: return pick<EPI_RELU2A, CL>(a_mn, b_mn);
    case EPI_ROWDOT: return pick<EPI_ROWDOT, CL>(a_mn, b_mn);
    default: return nullptr;
  }
}

// Most 2-CTA clusters of a kernel that can be resident at once (cached).
std::mutex g_cl_mu;
std::unordered_map<const void*, int> g_cl_max;

int max_clusters(KernFn fn) {
  std::lock_guard<std::mutex> lock(g_cl_mu);
  auto it = g_cl_max.find(reinterpret_cast<const void*>(fn));
  if (it != g_cl_max.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (g_num_sms / 2));
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) n = g_num_sms / 2;
  g_cl_max[reinterpret_cast<const void*>(fn)] = n;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// k-splits summed into C inside the kernel, in split order (see TcParams).
// Only where one split's work units fill the resident CTA pairs: then split
// s of a tile runs a wave after split s - 1 and finds it done. With fewer
// tiles the splits of a tile run side by side and their epilogues would
// queue one behind the other (measured: the 256-wide model's step 1.8 ->
// 2.3 ms), so those keep the partial slabs and the reduction kernel.
bool split_in_kernel(const GemmArgs& g, int splits) {
  if (splits < 2 || !g.tile_done || g.batch != 1 || (g.beta != 0.f && g.beta != 1.f)) return false;
  const long long rows = (g.M + BM - 1) / BM, cols = (g.N + BN - 1) / BN;
  if (rows * cols > kGemmTileCap) return false;
  const long long units = (g.M > BM ? (rows + 1) / 2 : rows) * cols;  // CTA-pair units of one split
  return units >= (g_num_sms > 0 ? g_num_sms : 148) / 2;
}

}  // namespace

bool gemm_tc_supports(const GemmArgs& g) {
  if (g.M < 0 || g.N < 0 || g.K < 0) return false;
  if (g.N % 8 || g.lda % 8 || g.ldb % 8) return false;
  if (!aligned16(g.A) || !aligned16(g.B)) return false;
  if (g.batch < 1) return false;
  if (g.batch > 1) {
    // stacked problems: whole 128-row blocks per problem so no tile's rows
    // reach into the next problem's output; 64-deep k slices per problem
    // for operands stacked along k (the MN-major ones)
    if (g.epi != EPI_STORE && g.epi != EPI_AXPBY) return false;
    if (g.splits > 1 || g.M % BM) return false;
    if (g.c_brows < g.M) return false;
    if (g.a_brows < (g.a_kmajor ? g.M : g.K) || g.b_brows < (g.b_kmajor ? g.N : g.K)) return false;
    if ((!g.a_kmajor && g.a_brows % BK) || (!g.b_kmajor && g.b_brows % BK)) return false;
    const long long rows_max = 0x7fffffffLL;
    if ((long long)g.batch * g.a_brows > rows_max || (long long)g.batch * g.b_brows > rows_max ||
        (long long)g.batch * g.c_brows > rows_max)
      return false;
  }
  if (g.epi == EPI_AXPBY && (!g.C2 || g.ldc2 % 8 || !aligned16(g.C2))) return false;
  if (g.epi == EPI_CE_FWD) return g.p_max && g.p_sum && g.p_arg && g.p_tgt && g.row_i;
  if (g.splits > 1 && (g.epi != EPI_STORE_F32 || (!g.partial && !g.tile_done) || g.N % 4)) return false;
  if (g.ldc % 8 || !aligned16(g.C)) return false;
  if ((g.epi == EPI_RELU2 || g.epi == EPI_RELU2_BWD || g.epi == EPI_ROWDOT) && (!g.C2 || g.ldc2 % 8 || !aligned16(g.C2)))
    return false;
  if (g.epi == EPI_ROWDOT &&
      (g.N % 128 || g.seq_len < 1 || g.M % g.seq_len || !g.rd_D || (g.rd_L2 == nullptr) != (g.rd_lse == nullptr)))
    return false;
  if (g.epi == EPI_CE_BWD && (!g.row_f || !g.row_i)) return false;
  if (g.epi == EPI_QKNORM_ROPE &&
      (!g.rope_cos || !g.rope_sin || !g.rqk || g.seq_len < 1 || g.d_model % 128 || g.N != 3 * g.d_model))
    return false;
  return g.epi >= EPI_STORE && g.epi <= EPI_ROWDOT;
}

cudaError_t gemm_tc(const GemmArgs& g, cudaStream_t s) {
  if (!gemm_tc_supports(g)) return cudaErrorNotSupported;
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (!get_encode()) return cudaErrorNotSupported;
  // CTA pairs sharing the B tile whenever there are at least two row blocks
  // (in a batch: an even number per problem, so no pair spans two problems)
  const int CLn = (g.M > BM && (g.batch == 1 || (g.M / BM) % 2 == 0)) ? 2 : 1;
  CUtensorMap ta, tb;
  // TMA needs an extent of at least one element; an empty K reads nothing.
  uint64_t K = g.K > 0 ? (uint64_t)g.K : 1;
  // outer extents cover every stacked problem
  const uint64_t a_outer = g.batch > 1 ? (uint64_t)g.batch * g.a_brows : (g.a_kmajor ? (uint64_t)g.M : K);
  const uint64_t b_outer = g.batch > 1 ? (uint64_t)g.batch * g.b_brows : (g.b_kmajor ? (uint64_t)g.N : K);
  const uint64_t c_rows = g.batch > 1 ? (uint64_t)g.batch * g.c_brows : (uint64_t)g.M;
  bool ok = g.a_kmajor ? make_map(&ta, g.A, K, a_outer, g.lda, 64, 128) : make_map(&ta, g.A, g.M, a_outer, g.lda, 64, 64);
  ok = ok && (g.b_kmajor ? make_map(&tb, g.B, K, b_outer, g.ldb, 64, CLn == 2 ? 128 : 256)
                         : make_map(&tb, g.B, g.N, b_outer, g.ldb, 64, 64));
  if (!ok) return cudaErrorInvalidValue;
  CUtensorMap tcm = ta, tcm2 = ta;  // unused maps stay valid copies
  const bool f32out = g.epi == EPI_STORE_F32;
  if (g.epi != EPI_CE_FWD) ok = make_out_map(&tcm, g.C, f32out, g.N, c_rows, g.ldc);
  // RELU2's second output a, or RELU2_BWD's input a (loaded in 32 x 64 chunks)
  if (ok && (g.epi == EPI_RELU2 || g.epi == EPI_RELU2_BWD || g.epi == EPI_ROWDOT))
    ok = make_out_map(&tcm2, g.C2, false, g.N, g.M, g.ldc2);
  if (!ok) return cudaErrorInvalidValue;
  TcParams p;
  p.g = g;
  p.num_m = (g.M + BM - 1) / BM;
  p.num_n = (g.N + BN - 1) / BN;
  p.num_kb = (g.K + BK - 1) / BK;
  p.splits = (g.splits > 1 && g.epi == EPI_STORE_F32 && (g.partial || g.tile_done)) ? g.splits : 1;
  p.kb_per_split = (p.num_kb + p.splits - 1) / p.splits;
  p.ordered = split_in_kernel(g, p.splits);
  p.tile_done = p.ordered ? g.tile_done : nullptr;
  if (p.splits > 1 && !p.ordered && !make_partial_map(&tcm2, g.partial, g.N, g.M, p.splits))
    return cudaErrorInvalidValue;
  KernFn fn = CLn == 2 ? pick_kernel<2>(g.epi, !g.a_kmajor, !g.b_kmajor) : pick_kernel<1>(g.epi, !g.a_kmajor, !g.b_kmajor);
  if (!fn) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (CLn == 2) {
    // work units are pairs of row blocks; one 2-CTA cluster per unit at a time
    p.total = ((p.num_m + 1) / 2) * p.num_n * p.splits * g.batch;
    int clusters = max_clusters(fn);
    if (clusters > p.total) clusters = p.total;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, ta, tb, tcm, tcm2, p);
  } else {
    p.total = p.num_m * p.num_n * p.splits * g.batch;
    int grid = p.total < g_num_sms ? p.total : g_num_sms;
    fn<<<grid, NTHREADS, SMEM_BYTES, s>>>(ta, tb, tcm, tcm2, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || p.splits == 1 || p.ordered) return e;
  return splitk_reduce(g.partial, p.splits, static_cast<float*>(g.C), g.ldc, g.M, g.N, g.beta, s);
}

int gemm_tc_launches(const GemmArgs& g) {
  if (g.M == 0 || g.N == 0) return 0;
  const int splits = (g.splits > 1 && g.epi == EPI_STORE_F32 && (g.partial || g.tile_done)) ? g.splits : 1;
  return (splits > 1 && !split_in_kernel(g, splits)) ? 2 : 1;
}

// Choose k-splits for fp32-output GEMMs whose output tiles underfill the SMs
// (the weight gradients, K = tokens): minimise the estimated time of
// ceil(units / SMs) waves of ceil(kblocks / splits) k-blocks each, plus the
// partial-sum traffic (write + read of splits * M * N fp32).
int gemm_tc_pick_splits(const GemmArgs& g) {
  if (g.epi != EPI_STORE_F32 || g.M == 0 || g.N == 0) return 1;
  get_encode();
  const long long tiles = (long long)((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
  const long long kb = (g.K + BK - 1) / BK;
  if (kb < 16 || tiles >= 4LL * g_num_sms) return 1;
  const double t_kb = 0.28e-6;                 // one 128x256x64 k-block per SM, seconds
  const double bw = 6.0e12;                    // bytes/s for the partial-sum round trip
  int best = 1;
  double best_t = 1e30;
  for (int s = 1; s <= 8; ++s) {
    const long long per = (kb + s - 1) / s;
    const long long waves = (tiles * s + g_num_sms - 1) / g_num_sms;
    const double t = waves * per * t_kb + (s > 1 ? 8.0 * s * g.M * (double)g.N / bw : 0.0);
    if (t < best_t * 0.97) { best_t = t; best = s; }
  }
  return best;
}

}  // namespace nc
