// Relative-position memory attention backward on sm_103a tensor cores.
//
// With P_ij = exp(scale*A_ij - lse_i) on allowed pairs, D_i = dO_i.O_i and
// dA_ij = scale * P_ij (dO_i.V_j - D_i) (chain rule of "Dimension
// Walkthrough"; stop-gradient of "Why Stop Gradient": nothing is written to
// the cached rows, their K/V gradients are returned like any other row):
//   dV_j = sum_i P_ij dO_i             dK_j = sum_i dA_ij (q_i+u)
//   dQ_i = sum_j dA_ij (k_j + r_{i-j})  dR_d = sum_b sum_{i-j=d} dA_ij (q_i+v)
//   du   = sum dA_ij k_j               dv   = sum dA_ij r_{i-j}
//
// Kernels (all on the caller's stream):
//   zero   : dR <- 0; dK/dV rows of ring slots without valid memory <- 0
//   prep   : the forward kernel in preparation mode: D_i from the fp32 O, and
//            the bf16 (Q+u), (Q+v) rows the two kernels below load by TMA
//   kv     : one CTA per (b, h, 128-key tile), loops over query tiles:
//            S, G -> P (skewed, masked), dP = dO V^T -> dA;
//            dV += P^T dO and dK += dA^T (Q+u) accumulate in TMEM
//   q      : one CTA per (b, h, 128-query tile), loops over key tiles:
//            S, G -> P, dP -> dA, and the sheared dG[ii][t] = dA[ii][ii+127-t];
//            dQ_content += dA K and dQ_position += dG Rband accumulate in TMEM;
//            dR_band = dG^T (Q+v) per tile pair, added into dR (fp32 atomics).
//            The position products run in fp16 (dG scaled by a CTA-wide power
//            of two, R band and (Q+v) converted in place): R rows are several
//            times larger than K rows, and bf16 rounding of dA in that term
//            alone can exceed 1% of max|dQ| on short contexts.
//   finish : du, dv = fixed-order sums of the per-CTA column sums of the two
//            dQ parts
// Both main kernels keep the score tile in TMEM (lanes = query rows), so the
// skewed read of the position scores is the one the forward uses.
#include <math.h>

#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace rxl {
namespace {

using namespace sm103;
using namespace tc;

constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant, each owning 64 of a row's keys
constexpr int kThreads = (kSoftmaxWarps + 1) * 32;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_G = idesc_bf16(128, 256, false, false);
constexpr uint32_t IDESC_MN_MN = idesc_bf16(128, 64, true, true);   // A^T . B, both d/row-major tiles
constexpr uint32_t IDESC_K_MN = idesc_bf16(128, 64, false, true);
constexpr uint32_t IDESC_K_MN_F16 = idesc_f16(128, 64, false, true);
constexpr uint32_t IDESC_MN_MN_F16 = idesc_f16(128, 64, true, true);
constexpr float kLog2e = 1.4426950408889634f;

__device__ int g_bwd_error;

struct BwdParams {
  int B, H, L, cap, m, head, nq, kv_rows, nkt;
  float scale, scale_log2;
  const float *lse, *delta;
  __nv_bfloat16 *dq, *dk, *dv;
  float *dr;        // [H][kv_rows][64], zeroed by the zero kernel
  float *duv_part;  // [B*H][nq][2][64]
};

// K-major operand: 128-byte swizzled [rows][64] tile, k-step kk of 16 elements.
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
// MN-major operand: [K rows][MN] tiles of 64 MN columns (16 KB apart), k-step of 16 rows.
__device__ __forceinline__ uint64_t mndesc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, 16384, 1024);
}

// 64 fp32 values (keys 64*hf ..) of row ii as bf16 into column block hf of a
// [128][128] K-major 128-byte-swizzled tile pair (blocks 16 KB apart).
__device__ __forceinline__ void store_half_bf16(uint32_t base, int ii, int hf, const float (&a)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(base + hf * 16384 + sw128_offset(ii, c), pack_bf16(a[8 * c + 0], a[8 * c + 1]),
                 pack_bf16(a[8 * c + 2], a[8 * c + 3]), pack_bf16(a[8 * c + 4], a[8 * c + 5]),
                 pack_bf16(a[8 * c + 6], a[8 * c + 7]));
}

// Bounded rendezvous of the two warps of a lane quadrant (mbarrier, count 2).
__device__ __forceinline__ bool pair_sync(uint32_t bar, int lane, uint32_t &phase,
                                          volatile int *abort_flag) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, phase & 1, abort_flag));
  ++phase;
  return ok;
}

// Output chunk D of the sheared dG row ii: columns 32*quad + 32*D + y hold
// v[ii + 127 - col] = w1[y + u] with w1[z] = v[158 - 32D - z] and u = 31 - lane
// (5-stage barrel shift), stored as fp16 into a [128][256] K-major tile set
// (four 16 KB column blocks).
__device__ __forceinline__ void shear_put(uint32_t base, int ii, int quad, int lane, int D,
                                          float (&w1)[63]) {
  const int u = 31 - lane;
#pragma unroll
  for (int b = 4; b >= 0; --b) {
    const int sh = 1 << b;
    const bool take = (u >> b) & 1;
#pragma unroll
    for (int e = 0; e < 62; ++e)
      if (e < 32 + sh - 1 && e + sh < 63) w1[e] = take ? w1[e + sh] : w1[e];
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int col = 32 * (quad + D) + 8 * e;
    st_shared_v4(base + (col >> 6) * 16384 + sw128_offset(ii, (col & 63) >> 3),
                 pack_f16(w1[8 * e + 0], w1[8 * e + 1]), pack_f16(w1[8 * e + 2], w1[8 * e + 3]),
                 pack_f16(w1[8 * e + 4], w1[8 * e + 5]), pack_f16(w1[8 * e + 6], w1[8 * e + 7]));
  }
}

// Half 0 of a row writes chunks D = 2, 3, 4 from its keys 0..63 (y) and keys
// 64..95 received from half 1 (xk, already scaled); half 1 writes D = 0, 1
// from its keys 64..127. Values are scaled by sig (a power of two).
template <int D>
__device__ __forceinline__ void shear_chunk_lo(uint32_t base, int ii, int quad, int lane,
                                               const float (&y)[64], const float (&xk)[32], float sig) {
  float w1[63];
#pragma unroll
  for (int z = 0; z < 63; ++z) {
    const int key = 158 - 32 * D - z;
    w1[z] = (key >= 0 && key < 64) ? sig * y[(key >= 0 && key < 64) ? key : 0]
            : (key >= 64 && key < 96) ? xk[(key >= 64 && key < 96) ? key - 64 : 0]
                                      : 0.f;
  }
  shear_put(base, ii, quad, lane, D, w1);
}
template <int D>
__device__ __forceinline__ void shear_chunk_hi(uint32_t base, int ii, int quad, int lane,
                                               const float (&y)[64], float sig) {
  float w1[63];
#pragma unroll
  for (int z = 0; z < 63; ++z) {
    const int key = 158 - 32 * D - z;
    w1[z] = (key >= 64 && key < 128) ? sig * y[(key >= 64 && key < 128) ? key - 64 : 0] : 0.f;
  }
  shear_put(base, ii, quad, lane, D, w1);
}

// ------------------------------------------------------------- dK / dV kernel

constexpr uint32_t KV_K = 0, KV_V = 16384, KV_QU = 32768, KV_QV = 49152, KV_DO = 65536;
constexpr uint32_t KV_R = 81920, KV_P = 114688, KV_DA = 147456, KV_BAR = 180224;
constexpr uint32_t KV_SMEM = KV_BAR + 128 + 1024;
constexpr uint32_t TM_S = 0, TM_G = 128, TM_A = 384, TM_B = 448;  // A/B: dV/dK or dQc/dQp

__global__ void __launch_bounds__(kThreads, 1)
rxl_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_qu,
                  const __grid_constant__ CUtensorMap tm_qv, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.nkt, kt = blockIdx.x % p.nkt;
  const int h = bh % p.H;
  const KeyTiles tiles(p.m, p.cap, p.head, p.L);
  const KeyTile x = tiles.get(kt);
  const int qlo = x.jlog0 >= 0 ? x.jlog0 / BQ : 0;
  const int NQ = p.nq - qlo;

  const uint32_t bar_kv = sb + KV_BAR, bar_q = bar_kv + 8, bar_sg = bar_kv + 16, bar_p = bar_kv + 24;
  const uint32_t bar_dp = bar_kv + 32, bar_ds = bar_kv + 40, bar_pair = bar_kv + 48;
  const uint32_t bar_drain = bar_kv + 56;
  uint32_t *tmem_slot = (uint32_t *)(smem + KV_BAR + 64);
  volatile int *abort_flag = (volatile int *)(smem + KV_BAR + 72);
  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1); mbar_init(bar_q, 1); mbar_init(bar_sg, 1);
    mbar_init(bar_p, kSoftmaxWarps * 32); mbar_init(bar_dp, 1);
    mbar_init(bar_ds, kSoftmaxWarps * 32); mbar_init(bar_pair, 1); mbar_init(bar_drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kProducerWarp) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int q_issued = 0;
      auto issue_q = [&](int n) {
        const int i0 = (qlo + n) * BQ;
        mbar_expect_tx(bar_q, 3 * 16384 + 32768);
        tma_load_3d(sb + KV_QU, &tm_qu, 0, i0, bh, bar_q);
        tma_load_3d(sb + KV_QV, &tm_qv, 0, i0, bh, bar_q);
        tma_load_3d(sb + KV_DO, &tm_do, 0, i0, bh, bar_q);
        tma_load_3d(sb + KV_R, &tm_r, 0, i0 - x.jlog0 - (BK - 1), h, bar_q);
        ++q_issued;
      };
      bool ok = true;
      mbar_expect_tx(bar_kv, 2 * 16384);
      tma_load_3d(sb + KV_K, &tm_k, 0, x.phys0, bh, bar_kv);
      tma_load_3d(sb + KV_V, &tm_v, 0, x.phys0, bh, bar_kv);
      issue_q(0);
      ok = mbar_wait(bar_kv, 0, abort_flag);
      for (int n = 0; ok && n < NQ; ++n) {
        if (!(ok = mbar_wait(bar_q, n & 1, abort_flag))) break;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_S, kdesc(sb + KV_QU, k), kdesc(sb + KV_K, k), IDESC_S, k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_G, kdesc(sb + KV_QV, k), kdesc(sb + KV_R, k), IDESC_G, k > 0);
        mma_commit(bar_sg);
        if (!(ok = mbar_wait(bar_p, n & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_S, kdesc(sb + KV_DO, k), kdesc(sb + KV_V, k), IDESC_S, k > 0);
        mma_commit(bar_dp);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16(tmem + TM_A, mndesc(sb + KV_P, k), mndesc(sb + KV_DO, k), IDESC_MN_MN,
                   (n > 0 || k > 0) ? 1u : 0u);
        if (!(ok = mbar_wait(bar_ds, n & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16(tmem + TM_B, mndesc(sb + KV_DA, k), mndesc(sb + KV_QU, k), IDESC_MN_MN,
                   (n > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_pair);
        if (n + 1 < NQ) {
          if (!(ok = mbar_wait(bar_pair, n & 1, abort_flag))) break;
          issue_q(n + 1);
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        mbar_wait(bar_kv, 0, &no_abort);
        if (q_issued > 0) mbar_wait(bar_q, (q_issued - 1) & 1, &no_abort);
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, &no_abort);
        atomicExch(&g_bwd_error, 1);
      }
    }
    __syncwarp();
  } else {
    const int quad = warp & 3, hf = warp >> 2;
    const int ii = quad * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    for (int n = 0; n < NQ; ++n) {
      const int i = (qlo + n) * BQ + ii;
      const bool row_ok = i < p.L;
      const size_t row = (size_t)bh * p.L + (row_ok ? i : 0);
      const float lse2 = row_ok ? p.lse[row] * kLog2e : 0.f;
      const float Di = row_ok ? p.delta[row] : 0.f;
      ok = mbar_wait(bar_sg, n & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      float y[64];
      half_tile_logits<true>(trow, TM_S, TM_G, quad, lane, hf, i, x, p.scale_log2, y);
#pragma unroll
      for (int k = 0; k < 64; ++k) y[k] = row_ok ? ex2(y[k] - lse2) : 0.f;  // P
      store_half_bf16(sb + KV_P, ii, hf, y);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_p);
      ok = mbar_wait(bar_dp, n & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dp[32];
        tmem_ld32(trow + TM_S + 64 * hf + 32 * cc, dp);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float pv = y[32 * cc + k];
          y[32 * cc + k] = pv != 0.f ? p.scale * pv * (__uint_as_float(dp[k]) - Di) : 0.f;  // dA
        }
      }
      store_half_bf16(sb + KV_DA, ii, hf, y);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_ds);
    }
    if (ok && NQ > 0) ok = mbar_wait(bar_pair, (NQ - 1) & 1, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      // TMEM lanes of the dV / dK accumulators are key rows; half 0 writes
      // dV, half 1 dK
      tc_fence_after();
      const int kk = ii;
      const size_t krow = (size_t)bh * p.kv_rows + x.phys0 + (kk < x.nvalid ? kk : 0);
      __nv_bfloat16 *dst = (hf ? p.dk : p.dv) + krow * DH;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t g[32];
        tmem_ld32(trow + (hf ? TM_B : TM_A) + 32 * c, g);
        tmem_wait_ld();
        if (kk < x.nvalid) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ((uint4 *)dst)[4 * c + e] = make_uint4(
                pack_bf16(__uint_as_float(g[8 * e + 0]), __uint_as_float(g[8 * e + 1])),
                pack_bf16(__uint_as_float(g[8 * e + 2]), __uint_as_float(g[8 * e + 3])),
                pack_bf16(__uint_as_float(g[8 * e + 4]), __uint_as_float(g[8 * e + 5])),
                pack_bf16(__uint_as_float(g[8 * e + 6]), __uint_as_float(g[8 * e + 7])));
        }
      }
    } else {
      atomicExch(&g_bwd_error, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------- dQ / dR / du / dv kernel

constexpr uint32_t Q_QU = 0, Q_QV = 16384, Q_DO = 32768, Q_K = 49152, Q_V = 65536;
constexpr uint32_t Q_R = 81920, Q_DA = 114688, Q_DG = 147456, Q_X = 212992, Q_BAR = 221184;
constexpr uint32_t Q_SMEM = Q_BAR + 256 + 1024;  // barriers, TMEM slot, flags, [2][8] warp maxima

__global__ void __launch_bounds__(kThreads, 1)
rxl_bwd_q_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_qu,
                 const __grid_constant__ CUtensorMap tm_qv, const __grid_constant__ CUtensorMap tm_do,
                 const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = p.nq - 1 - (int)(blockIdx.x % p.nq);
  const int bh = (int)(blockIdx.x / p.nq);
  const int h = bh % p.H;
  const int i0 = qt * BQ;
  const KeyTiles tiles(p.m, p.cap, p.head, min(i0 + BQ, p.L));
  const int T = tiles.count();

  const uint32_t bar_q = sb + Q_BAR, bar_k = bar_q + 8, bar_sg = bar_q + 16, bar_p = bar_q + 24;
  const uint32_t bar_dp = bar_q + 32, bar_ds = bar_q + 40, bar_dr = bar_q + 48, bar_fl = bar_q + 56;
  const uint32_t bar_drain = bar_q + 64, bar_red = bar_q + 72, bar_x0 = bar_q + 80;  // + 4 pair barriers
  uint32_t *tmem_slot = (uint32_t *)(smem + Q_BAR + 112);
  volatile int *abort_flag = (volatile int *)(smem + Q_BAR + 116);
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1); mbar_init(bar_k, 1); mbar_init(bar_sg, 1);
    mbar_init(bar_p, kSoftmaxWarps * 32); mbar_init(bar_dp, 1);
    mbar_init(bar_ds, kSoftmaxWarps * 32); mbar_init(bar_dr, 1);
    mbar_init(bar_fl, kSoftmaxWarps * 32); mbar_init(bar_drain, 1);
    mbar_init(bar_red, kSoftmaxWarps);
    for (int q = 0; q < 4; ++q) mbar_init(bar_x0 + 8 * q, 2);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kProducerWarp) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int k_issued = 0;
      auto issue_k = [&](int t) {
        const KeyTile x = tiles.get(t);
        // (Q+v) is reloaded with every key tile: the previous copy was
        // converted to fp16 in place
        mbar_expect_tx(bar_k, 3 * 16384 + 32768);
        tma_load_3d(sb + Q_K, &tm_k, 0, x.phys0, bh, bar_k);
        tma_load_3d(sb + Q_V, &tm_v, 0, x.phys0, bh, bar_k);
        tma_load_3d(sb + Q_R, &tm_r, 0, i0 - x.jlog0 - (BK - 1), h, bar_k);
        tma_load_3d(sb + Q_QV, &tm_qv, 0, i0, bh, bar_k);
        ++k_issued;
      };
      bool ok = true;
      mbar_expect_tx(bar_q, 2 * 16384);
      tma_load_3d(sb + Q_QU, &tm_qu, 0, i0, bh, bar_q);
      tma_load_3d(sb + Q_DO, &tm_do, 0, i0, bh, bar_q);
      issue_k(0);
      ok = mbar_wait(bar_q, 0, abort_flag);
      for (int t = 0; ok && t < T; ++t) {
        if (!(ok = mbar_wait(bar_k, t & 1, abort_flag))) break;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_S, kdesc(sb + Q_QU, k), kdesc(sb + Q_K, k), IDESC_S, k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_G, kdesc(sb + Q_QV, k), kdesc(sb + Q_R, k), IDESC_G, k > 0);
        mma_commit(bar_sg);
        if (!(ok = mbar_wait(bar_p, t & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_S, kdesc(sb + Q_DO, k), kdesc(sb + Q_V, k), IDESC_S, k > 0);
        mma_commit(bar_dp);
        if (!(ok = mbar_wait(bar_ds, t & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)   // dQ_content += dA . K
          mma_bf16(tmem + TM_A, kdesc(sb + Q_DA, k), mndesc(sb + Q_K, k), IDESC_K_MN,
                   (t > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 16; ++k)  // dQ_position += dG . Rband (fp16)
          mma_bf16(tmem + TM_B, kdesc(sb + Q_DG, k), mndesc(sb + Q_R, k), IDESC_K_MN_F16,
                   (t > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)  // dR band = dG^T . (Q+v), two 128-distance blocks (fp16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16(tmem + TM_G + 64 * mb, mndesc(sb + Q_DG + 2 * mb * 16384, k),
                     mndesc(sb + Q_QV, k), IDESC_MN_MN_F16, k > 0);
        mma_commit(bar_dr);
        if (!(ok = mbar_wait(bar_fl, t & 1, abort_flag))) break;
        if (t + 1 < T) issue_k(t + 1);
      }
      if (!ok) {
        volatile int no_abort = 0;
        mbar_wait(bar_q, 0, &no_abort);
        if (k_issued > 0) mbar_wait(bar_k, (k_issued - 1) & 1, &no_abort);
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, &no_abort);
        atomicExch(&g_bwd_error, 4);
      }
    }
    __syncwarp();
  } else {
    const int quad = warp & 3, hf = warp >> 2;
    const int ii = quad * 32 + lane;
    const int i = i0 + ii;
    const bool row_ok = i < p.L;
    const size_t row = (size_t)bh * p.L + (row_ok ? i : 0);
    const float lse2 = row_ok ? p.lse[row] * kLog2e : 0.f;
    const float Di = row_ok ? p.delta[row] : 0.f;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t bar_x = bar_x0 + 8 * quad;
    volatile float *wmax = (volatile float *)(smem + Q_BAR + 96 + 32);  // [2][8] in the slack
    uint32_t xphase = 0;
    float sig = 1.0e30f;  // fp16 scale of the position products (power of two, non-increasing)
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const KeyTile x = tiles.get(t);
      ok = mbar_wait(bar_sg, t & 1, abort_flag) && mbar_wait(bar_k, t & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      // S and G are done with the bf16 R band and (Q+v): convert them to fp16
      // for the position-gradient products of this tile pair
#pragma unroll
      for (int c = 0; c < 8; ++c) chunk_bf16_to_f16(sb + Q_R + hf * 16384 + sw128_offset(ii, c));
#pragma unroll
      for (int c = 0; c < 4; ++c) chunk_bf16_to_f16(sb + Q_QV + sw128_offset(ii, 4 * hf + c));
      float y[64];
      half_tile_logits<true>(trow, TM_S, TM_G, quad, lane, hf, i, x, p.scale_log2, y);
#pragma unroll
      for (int k = 0; k < 64; ++k) y[k] = row_ok ? ex2(y[k] - lse2) : 0.f;  // P
      tc_fence_before();
      mbar_arrive(bar_p);
      ok = mbar_wait(bar_dp, t & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dp[32];
        tmem_ld32(trow + TM_S + 64 * hf + 32 * cc, dp);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float pv = y[32 * cc + k];
          y[32 * cc + k] = pv != 0.f ? p.scale * pv * (__uint_as_float(dp[k]) - Di) : 0.f;  // dA
        }
      }
      store_half_bf16(sb + Q_DA, ii, hf, y);
      // CTA-wide max |dA| of this tile pair -> power-of-two fp16 scale
      float am = 0.f;
#pragma unroll
      for (int k = 0; k < 64; ++k) am = fmaxf(am, fabsf(y[k]));
      am = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(am)));
      if (lane == 0) {
        wmax[(t & 1) * 8 + warp] = am;
        mbar_arrive(bar_red);
      }
      ok = mbar_wait(bar_red, t & 1, abort_flag);  // bounded, unlike a named barrier
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      am = 0.f;
#pragma unroll
      for (int w = 0; w < kSoftmaxWarps; ++w) am = fmaxf(am, wmax[(t & 1) * 8 + w]);
      if (am > 0.f) {
        const float want = exp2f(14.f - ceilf(log2f(am)));  // max |scaled dA| <= 2^14
        if (want < sig) {
          if (t > 0) {
            // rescale this half's columns of the fp16-scaled dQ_position accumulator
            const float f = want / sig;
            uint32_t g[32];
            tmem_ld32(trow + TM_B + 32 * hf, g);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) g[e] = __float_as_uint(__uint_as_float(g[e]) * f);
            tmem_st32(trow + TM_B + 32 * hf, g);
            tmem_wait_st();
          }
          sig = want;
        }
      }
      // sheared dG (fp16, scaled by sig): half 1 hands keys 64..95 to half 0
      const uint32_t xrow = sb + Q_X + ii * 64;
      if (hf == 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          st_shared_v4(xrow + 16 * e, pack_f16(sig * y[8 * e + 0], sig * y[8 * e + 1]),
                       pack_f16(sig * y[8 * e + 2], sig * y[8 * e + 3]),
                       pack_f16(sig * y[8 * e + 4], sig * y[8 * e + 5]),
                       pack_f16(sig * y[8 * e + 6], sig * y[8 * e + 7]));
      }
      if (!(ok = pair_sync(bar_x, lane, xphase, abort_flag))) break;
      // column chunks outside [32*quad, 32*quad + 160) are zero for every lane
      for (int C = 0; C < 8; ++C) {
        if (hf == 0 ? C < quad : C > quad + 4) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = 32 * C + 8 * e;
            st_shared_v4(sb + Q_DG + (col >> 6) * 16384 + sw128_offset(ii, (col & 63) >> 3), 0, 0, 0, 0);
          }
        }
      }
      if (hf == 0) {
        float xk[32];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t a, b, c, d;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                       : "r"(xrow + 16 * e));
          const uint32_t w[4] = {a, b, c, d};
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const __half2 hv = *reinterpret_cast<const __half2 *>(&w[f]);
            const float2 fv = __half22float2(hv);
            xk[8 * e + 2 * f] = fv.x;
            xk[8 * e + 2 * f + 1] = fv.y;
          }
        }
        shear_chunk_lo<2>(sb + Q_DG, ii, quad, lane, y, xk, sig);
        shear_chunk_lo<3>(sb + Q_DG, ii, quad, lane, y, xk, sig);
        shear_chunk_lo<4>(sb + Q_DG, ii, quad, lane, y, xk, sig);
      } else {
        shear_chunk_hi<0>(sb + Q_DG, ii, quad, lane, y, sig);
        shear_chunk_hi<1>(sb + Q_DG, ii, quad, lane, y, sig);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_ds);
      ok = mbar_wait(bar_dr, t & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      // dR rows of this tile pair: TMEM lane = band row, half hf reads block hf
      const int d0 = i0 - x.jlog0 - (BK - 1);
      {
        const int d = d0 + 128 * hf + ii;
        float *dst = p.dr + ((size_t)h * p.kv_rows + (d >= 0 ? d : 0)) * DH;
        const float f = 1.f / sig;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t g[32];
          tmem_ld32(trow + TM_G + 64 * hf + 32 * c, g);
          tmem_wait_ld();
          if (d >= 0 && d < p.m + p.L) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              red_add_v4(dst + 32 * c + 4 * e, f * __uint_as_float(g[4 * e]), f * __uint_as_float(g[4 * e + 1]),
                         f * __uint_as_float(g[4 * e + 2]), f * __uint_as_float(g[4 * e + 3]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_fl);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      // dQ = content + position parts; du, dv partials = column sums of the
      // parts. This thread owns columns 32*hf .. 32*hf+31 of its row.
      float *red = (float *)(smem + Q_DG);  // [2][128][64] fp32, reuses the dG tile
      uint4 *qrow = (uint4 *)(p.dq + row * DH);
      uint32_t a[32], b[32];
      tmem_ld32(trow + TM_A + 32 * hf, a);
      tmem_ld32(trow + TM_B + 32 * hf, b);
      tmem_wait_ld();
      const float f = sig < 1.0e29f ? 1.f / sig : 0.f;  // undo the fp16 scale
#pragma unroll
      for (int e = 0; e < 32; ++e) b[e] = __float_as_uint(__uint_as_float(b[e]) * f);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        red[ii * 64 + 32 * hf + e] = __uint_as_float(a[e]);
        red[128 * 64 + ii * 64 + 32 * hf + e] = __uint_as_float(b[e]);
      }
      if (row_ok) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float s8[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) s8[g] = __uint_as_float(a[8 * e + g]) + __uint_as_float(b[8 * e + g]);
          qrow[4 * hf + e] = make_uint4(pack_bf16(s8[0], s8[1]), pack_bf16(s8[2], s8[3]),
                                        pack_bf16(s8[4], s8[5]), pack_bf16(s8[6], s8[7]));
        }
      }
    } else {
      atomicExch(&g_bwd_error, 8);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the softmax warps only
    if (ok && threadIdx.x < 128) {
      const float *red = (const float *)(smem + Q_DG);
      const int part = threadIdx.x >> 6, col = threadIdx.x & 63;  // (part, column)
      float acc = 0.f;
      for (int r = 0; r < BQ; ++r) acc += red[part * 128 * 64 + r * 64 + col];
      p.duv_part[(((size_t)bh * p.nq + qt) * 2 + part) * DH + col] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------- small kernels

__global__ void bwd_zero_kernel(float *dr, size_t n_dr, __nv_bfloat16 *dk, __nv_bfloat16 *dv,
                                int BH, int cap, int m, int head, int kv_rows) {
  const size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t e = tid; e < n_dr / 4; e += stride) ((float4 *)dr)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  // dK/dV rows of ring slots that hold no valid memory: 8 x 16 B per row
  const int empty = cap - m;
  const size_t n_rows = (size_t)BH * empty * 8;
  for (size_t e = tid; e < n_rows; e += stride) {
    const int c = (int)(e & 7);
    const size_t r = e >> 3;
    const int bh = (int)(r / empty), t = m + (int)(r % empty);  // logical slot t >= m
    int pr = head + t;
    if (pr >= cap) pr -= cap;
    const size_t off = ((size_t)bh * kv_rows + pr) * DH;
    ((uint4 *)(dk + off))[c] = make_uint4(0, 0, 0, 0);
    ((uint4 *)(dv + off))[c] = make_uint4(0, 0, 0, 0);
  }
}

// Streaming preparation when the forward kept the low part of O: per row,
// (Q+u) and (Q+v) in bf16 and D_i = dO_i . (o_i + o_lo_i). Eight threads
// per row, 16 bytes each.
__global__ void __launch_bounds__(256) bwd_light_prep_kernel(
    long long rows, int L, int H, const __nv_bfloat16 *__restrict__ q,
    const __nv_bfloat16 *__restrict__ u, const __nv_bfloat16 *__restrict__ vb,
    const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ o_lo,
    const __nv_bfloat16 *__restrict__ dout, __nv_bfloat16 *__restrict__ qu,
    __nv_bfloat16 *__restrict__ qv, float *__restrict__ delta) {
  const int sub = threadIdx.x & 7;
  for (long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 3; row < rows;
       row += ((long long)gridDim.x * blockDim.x) >> 3) {
    const int h = (int)((row / L) % H);
    const size_t off = (size_t)row * DH;
    const uint4 q4 = ((const uint4 *)(q + off))[sub];
    const uint4 u4 = ((const uint4 *)(u + (size_t)h * DH))[sub];
    const uint4 v4 = ((const uint4 *)(vb + (size_t)h * DH))[sub];
    const uint4 o4 = ((const uint4 *)(o + off))[sub];
    const uint4 l4 = ((const uint4 *)(o_lo + off))[sub];
    const uint4 d4 = ((const uint4 *)(dout + off))[sub];
    const uint32_t qw[4] = {q4.x, q4.y, q4.z, q4.w}, uw[4] = {u4.x, u4.y, u4.z, u4.w};
    const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w}, ow[4] = {o4.x, o4.y, o4.z, o4.w};
    const uint32_t lw[4] = {l4.x, l4.y, l4.z, l4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
    auto lo = [](uint32_t x) { return __uint_as_float(x << 16); };
    auto hi = [](uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); };
    uint32_t a[4], b[4];
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a[e] = pack_bf16(lo(qw[e]) + lo(uw[e]), hi(qw[e]) + hi(uw[e]));
      b[e] = pack_bf16(lo(qw[e]) + lo(vw[e]), hi(qw[e]) + hi(vw[e]));
      acc += lo(dw[e]) * (lo(ow[e]) + lo(lw[e])) + hi(dw[e]) * (hi(ow[e]) + hi(lw[e]));
    }
    ((uint4 *)(qu + off))[sub] = make_uint4(a[0], a[1], a[2], a[3]);
    ((uint4 *)(qv + off))[sub] = make_uint4(b[0], b[1], b[2], b[3]);
#pragma unroll
    for (int w = 4; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (sub == 0) delta[row] = acc;
  }
}

__global__ void bwd_finish_kernel(const float *duv_part, float *du, float *dvb, int B, int H, int nq) {
  const int h = blockIdx.x, part = threadIdx.x >> 6, c = threadIdx.x & 63;
  float acc = 0.f;
  for (int b = 0; b < B; ++b)
    for (int q = 0; q < nq; ++q)
      acc += duv_part[((((size_t)b * H + h) * nq + q) * 2 + part) * DH + c];
  (part ? dvb : du)[h * DH + c] = acc;
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}

bool make_map(CUtensorMap *m, const void *base, int planes, int rows, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {128, (cuuint64_t)rows * 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

BwdWorkspace tc_bwd_workspace(const AttnShape &s) {
  const size_t rows = (size_t)s.B * s.H * s.L;
  const int nq = (s.L + BQ - 1) / BQ;
  BwdWorkspace w;
  w.d_off = 0;                                              // D [B,H,L] f32
  w.dqu_off = up256(rows * 4);                              // (Q+u) bf16
  w.dqv_off = w.dqu_off + up256(rows * DH * 2);             // (Q+v) bf16
  const size_t duv_off = w.dqv_off + up256(rows * DH * 2);  // du/dv partials
  w.total = duv_off + up256((size_t)s.B * s.H * nq * 2 * DH * 4);
  return w;
}

cudaError_t launch_tc_bwd(const AttnShape &s, const void *q, const void *k, const void *v,
                          const void *r, const void *u, const void *vb, const void *o,
                          const void *o_lo, const float *lse,
                          const void *dout, void *dq, void *dk, void *dv, float *dr, float *du,
                          float *dvb, void *ws, cudaStream_t st, int *launches) {
  const BwdWorkspace w = tc_bwd_workspace(s);
  float *delta = (float *)((char *)ws + w.d_off);
  void *qu = (char *)ws + w.dqu_off;
  void *qv = (char *)ws + w.dqv_off;
  float *duv = (float *)((char *)ws + w.dqv_off + up256((size_t)s.B * s.H * s.L * DH * 2));
  const int nq = (s.L + BQ - 1) / BQ;

  CUtensorMap tk, tv, tr, tqu, tqv, tdo;
  if (!make_map(&tk, k, s.B * s.H, s.kv_rows, BK) || !make_map(&tv, v, s.B * s.H, s.kv_rows, BK) ||
      !make_map(&tr, r, s.H, s.kv_rows, NB) || !make_map(&tqu, qu, s.B * s.H, s.L, BQ) ||
      !make_map(&tqv, qv, s.B * s.H, s.L, BQ) || !make_map(&tdo, dout, s.B * s.H, s.L, BQ))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(rxl_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KV_SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(rxl_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Q_SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;

  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t n_dr = (size_t)s.H * s.kv_rows * DH;
  bwd_zero_kernel<<<sms * 4, 256, 0, st>>>(dr, n_dr, (__nv_bfloat16 *)dk, (__nv_bfloat16 *)dv,
                                           s.B * s.H, s.cap, s.m, s.head, s.kv_rows);
  ++*launches;
  if (o_lo) {
    const long long rows = (long long)s.B * s.H * s.L;
    long long blocks = (rows * 8 + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    bwd_light_prep_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        rows, s.L, s.H, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)u,
        (const __nv_bfloat16 *)vb, (const __nv_bfloat16 *)o, (const __nv_bfloat16 *)o_lo,
        (const __nv_bfloat16 *)dout, (__nv_bfloat16 *)qu, (__nv_bfloat16 *)qv, delta);
    ++*launches;
  } else {
    cudaError_t e = launch_tc_bwd_prep(s, q, k, v, r, u, vb, dout, delta, qu, qv, st, launches);
    if (e != cudaSuccess) return e;
  }

  BwdParams p;
  p.B = s.B; p.H = s.H; p.L = s.L; p.cap = s.cap; p.m = s.m; p.head = s.head; p.nq = nq;
  p.kv_rows = s.kv_rows;
  {
    // key tiles per (b,h): ring runs A and B, then the current rows
    const int lenA = s.m < s.cap - s.head ? s.m : s.cap - s.head;
    const int lenB = s.m - lenA;
    p.nkt = (lenA + BK - 1) / BK + (lenB + BK - 1) / BK + (s.L + BK - 1) / BK;
  }
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.lse = lse; p.delta = delta;
  p.dq = (__nv_bfloat16 *)dq; p.dk = (__nv_bfloat16 *)dk; p.dv = (__nv_bfloat16 *)dv;
  p.dr = dr; p.duv_part = duv;
  rxl_bwd_kv_kernel<<<(unsigned)(s.B * s.H * p.nkt), kThreads, KV_SMEM, st>>>(tk, tv, tr, tqu, tqv, tdo, p);
  ++*launches;
  rxl_bwd_q_kernel<<<(unsigned)(s.B * s.H * nq), kThreads, Q_SMEM, st>>>(tk, tv, tr, tqu, tqv, tdo, p);
  ++*launches;
  bwd_finish_kernel<<<s.H, 128, 0, st>>>(duv, du, dvb, s.B, s.H, nq);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t tc_bwd_read_error(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_bwd_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof(int));
  return e;
}

}  // namespace rxl
