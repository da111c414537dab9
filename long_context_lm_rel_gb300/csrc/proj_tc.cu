// Projection front-end on sm_103a tensor cores ("Segment-Level Recurrence":
// Q = H W^Q, K = [SG(M); H] W^K, V = [SG(M); H] W^V; "Batched Tensor
// Contract" for the shapes).
//
// The memory holds the layer's input hidden states in a ring of M rows per
// batch row (the same ring layout as K/V: logical memory row t at physical
// row (head + t) mod M). Ring slot p projects to physical row p of K and V
// and the current rows to rows M .. M+L-1, so the projected K/V are already
// in the attention's ring layout. Only ring slots holding valid memory are
// projected (their rows are walked as the attention walks its key tiles);
// rows of empty slots are not written.
//
// An output block is 128 hidden-state rows of one batch row times up to 4
// heads (N <= 256 columns) of one of Q, K, V, with the hidden width d
// streamed in 64-wide steps through a 5-stage TMA pipeline:
//   A = hidden rows [128][64] bf16 (K-major, 128-byte swizzle)
//   B = W rows [64][N] bf16 (MN-major: 64x64 swizzled boxes, 8 KB apart;
//       each CTA of a pair holds its two heads' boxes)
//   D = TMEM [128 lanes][N] fp32; four epilogue warps write bf16 rows of
//   64 columns per head.
// The kernel runs on persistent CTA pairs (tcgen05 cta_group::2: one
// M = 256, N = 256 MMA per k-step over two blocks that share their W columns,
// each SM loading its own rows and half of the columns), with one producer
// warp, one MMA warp and two accumulators, so pipeline fill and epilogue of
// one unit overlap the main loop of the next; the epilogue stages each head's
// 32 rows per warp as a 128-byte-swizzled box and writes it with one TMA
// store.
#include <math.h>

#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace rxl {
namespace {

using namespace sm103;
using namespace tc;

constexpr int P_STAGES = 5;
// warps 0-3 epilogue (TMEM lane quadrants), warp 4 TMA producer, warp 5 MMA
// issuer (first CTA of the pair; TMEM allocation only in the second)
constexpr int P_THREADS = 192;
constexpr uint32_t P_A_BYTES = 128 * 64 * 2;     // 16 KB: this CTA's 128 rows
constexpr uint32_t P_B_BYTES = 2 * 64 * 64 * 2;  // 16 KB: this CTA's 128 of the pair's 256 columns
constexpr uint32_t P_STAGE = P_A_BYTES + P_B_BYTES;
constexpr uint32_t P_BAR = P_STAGES * P_STAGE;
// epilogue staging: 4 warps x 2 buffers x 32 rows x 128 B, 1024-byte aligned
// (the layout of a 128-byte-swizzled TMA box)
constexpr uint32_t P_STG = P_BAR + 1024;
constexpr uint32_t P_SMEM = P_STG + 4 * 8192 + 1024;

__device__ int g_proj_error;

struct ProjParams {
  int B, H, L, cap, m, head, d;
  int NT;              // column tiles of up to 4 heads
  int Tq, Tkv;         // row tiles of Q and of K/V per batch row
  int pairs_q, pairs_kv;  // pairs of row tiles of Q and of K (or V), over all batch rows
  __nv_bfloat16 *out[3];  // q, k, v
};

// One CTA's output block of a pair unit: which of Q, K, V, its batch row,
// heads and rows; `store` is false for the second CTA of a pair whose list
// has an odd number of row tiles (it repeats the first CTA's rows).
struct ProjItem {
  const CUtensorMap *amap, *wmap, *omap;
  __nv_bfloat16 *out;
  int b, h0, nh, arow, orow0, nvalid, orows;
  bool store, kv;
};

// Unit u = (column tile nt, pair of row tiles): the row tiles of Q over all
// batch rows in order, then those of K, then those of V, two per unit, so
// both CTAs of a pair use the same W columns.
__device__ __forceinline__ ProjItem proj_item(const ProjParams &p, int u, int rank, const CUtensorMap *tm_hmem,
                                              const CUtensorMap *tm_hcur, const CUtensorMap *tm_wq,
                                              const CUtensorMap *tm_wk, const CUtensorMap *tm_wv,
                                              const CUtensorMap *tm_oq, const CUtensorMap *tm_ok,
                                              const CUtensorMap *tm_ov) {
  ProjItem it;
  const int nt = u % p.NT;
  int q = u / p.NT;
  int which, T;
  if (q < p.pairs_q) {
    which = 0;
    T = p.Tq;
  } else {
    q -= p.pairs_q;
    which = 1 + q / p.pairs_kv;
    q %= p.pairs_kv;
    T = p.Tkv;
  }
  int idx = 2 * q + rank;
  it.store = idx < p.B * T;
  if (!it.store) idx = 2 * q;
  it.b = idx / T;
  const int tile = idx % T;
  it.h0 = 4 * nt;
  it.nh = min(4, p.H - it.h0);
  it.amap = tm_hcur;
  if (which == 0) {
    it.arow = tile * BQ;
    it.orow0 = it.arow;
    it.nvalid = min(BQ, p.L - it.arow);
    it.orows = p.L;
  } else {
    const KeyTiles tiles(p.m, p.cap, p.head, p.L);
    const KeyTile x = tiles.get(tile);
    const bool mem = x.jlog0 < 0;
    it.amap = mem ? tm_hmem : tm_hcur;
    it.arow = mem ? x.phys0 : x.jlog0;
    it.orow0 = x.phys0;
    it.nvalid = x.nvalid;
    it.orows = p.cap + p.L;
  }
  it.wmap = which == 0 ? tm_wq : (which == 1 ? tm_wk : tm_wv);
  it.omap = which == 0 ? tm_oq : (which == 1 ? tm_ok : tm_ov);
  it.kv = which != 0;
  it.out = p.out[which];
  return it;
}

// Persistent CTA pairs (clusters of two): pair c takes units c, c + P, ...
// (P pairs) as one stream of 64-wide k-steps through the stage ring. Each
// CTA loads its own 128 hidden-state rows and its half (two heads) of the
// unit's W columns; the first CTA issues one M = 256, N = 256 MMA chain per
// unit into TMEM columns 256 (j & 1) .. +255 of both CTAs, so the epilogue
// of unit j runs while the MMAs of unit j+1 do. Heads past H load a valid
// head's columns and are not stored.
__global__ void __launch_bounds__(P_THREADS, 1)
rxl_proj_kernel(const __grid_constant__ CUtensorMap tm_hmem, const __grid_constant__ CUtensorMap tm_hcur,
                const __grid_constant__ CUtensorMap tm_wq, const __grid_constant__ CUtensorMap tm_wk,
                const __grid_constant__ CUtensorMap tm_wv, const __grid_constant__ CUtensorMap tm_oq,
                const __grid_constant__ CUtensorMap tm_ok, const __grid_constant__ CUtensorMap tm_ov,
                const ProjParams p, int nunits) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)(blockIdx.x & 1), pair = (int)(blockIdx.x >> 1), P = (int)(gridDim.x >> 1);
  const int nj = pair < nunits ? (nunits - 1 - pair) / P + 1 : 0;
  auto item = [&](int j) {
    return proj_item(p, pair + j * P, rank, &tm_hmem, &tm_hcur, &tm_wq, &tm_wk, &tm_wv, &tm_oq, &tm_ok, &tm_ov);
  };

  const uint32_t bar_full = sb + P_BAR;                // [S] (first CTA) the stage landed in both CTAs
  const uint32_t bar_empty = bar_full + 8 * P_STAGES;  // [S] the stage's MMAs are done
  const uint32_t bar_accf = bar_empty + 8 * P_STAGES;  // [2] accumulator written
  const uint32_t bar_acce = bar_accf + 16;             // [2] (first CTA) accumulator read by 8 warps
  const uint32_t bar_drain = bar_acce + 16;            // MMAs drained after an abort
  uint32_t *tmem_slot = (uint32_t *)(smem + P_BAR + 16 * P_STAGES + 40);
  volatile int *abort_flag = (volatile int *)(smem + P_BAR + 16 * P_STAGES + 44);
  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_accf + 8 * a, 1);
      mbar_init(bar_acce + 8 * a, 8);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 5) tmem_alloc_pair(smem_u32(tmem_slot), 512);
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers and TMEM are ready
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // inputs written by the previous kernel on the stream
  griddep_launch_dependents();
  const int nk = p.d / 64;
  const int total = nj * nk;  // k-steps of this pair

  if (warp == 4) {
    // ---- producer: k-step g of the pair's stream goes to stage g % P_STAGES
    // of both CTAs; every copy counts on the first CTA's full barrier, which
    // expects both CTAs' bytes
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(bar_full, 0);
      int issued[P_STAGES] = {};
      bool ok = true;
      int lj = -1;
      ProjItem li;
      for (int g = 0; g < total; ++g) {
        const int j = g / nk, kt = g - j * nk, s = g % P_STAGES;
        // the stage's previous k-step must have been consumed by the pair's MMAs
        if (g >= P_STAGES &&
            !(ok = mbar_wait_cluster(bar_empty + 8 * s, ((g / P_STAGES) - 1) & 1, abort_flag)))
          break;
        if (j != lj) {
          li = item(j);
          lj = j;
        }
        const uint32_t a = sb + s * P_STAGE, bb = a + P_A_BYTES;
        if (rank == 0) mbar_expect_tx(bar_full + 8 * s, 2 * P_STAGE);
        tma_load_3d_pair(a, li.amap, kt * 64, li.arow, li.b, full0 + 8 * s);
        for (int jj = 0; jj < 2; ++jj) {
          const int h = min(li.h0 + 2 * rank + jj, p.H - 1);
          tma_load_3d_pair(bb + jj * 8192, li.wmap, h * 64, kt * 64, 0, full0 + 8 * s);
        }
        ++issued[s];
      }
      // the last stages' releases arrive before the pair may exit
      for (int g = total > P_STAGES ? total - P_STAGES : 0; ok && g < total; ++g)
        ok = mbar_wait_cluster(bar_empty + 8 * (g % P_STAGES), (g / P_STAGES) & 1, abort_flag);
      if (!ok) {
        // let in-flight copies land before shared memory is released: the
        // first CTA sees its full barriers complete (they count both CTAs'
        // bytes); the second CTA, which has no barrier of its own to watch,
        // gives its copies a bounded grace period
        volatile int no_abort = 0;
        if (rank == 0) {
          for (int s = 0; s < P_STAGES; ++s)
            if (issued[s] > 0) mbar_wait(bar_full + 8 * s, (issued[s] - 1) & 1, &no_abort);
        } else {
          const long long t0 = clock64();
          while (clock64() - t0 < 20000000LL) {
          }
        }
        atomicExch(&g_proj_error, 1);
      }
    }
    __syncwarp();
  } else if (warp == 5 && rank == 0) {
    // ---- first CTA: MMA issuer for the pair
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(256, 256, false, true);
      bool ok = true;
      for (int j = 0; ok && j < nj; ++j) {
        const uint32_t acc = tmem + 256 * (j & 1);
        // the accumulator last held unit j-2: both epilogues must have read it
        if (j >= 2 && !(ok = mbar_wait_cluster(bar_acce + 8 * (j & 1), ((j >> 1) - 1) & 1, abort_flag)))
          break;
        tc_fence_after();
        for (int kt = 0; kt < nk; ++kt) {
          const int g = j * nk + kt, s = g % P_STAGES;
          if (!(ok = mbar_wait_cluster(bar_full + 8 * s, (g / P_STAGES) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t a = sb + s * P_STAGE, bb = a + P_A_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_pair(acc, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(bb + k * 2048, 8192, 1024), idesc,
                          (kt > 0 || k > 0) ? 1u : 0u);
          mma_commit_pair(bar_empty + 8 * s, 3);
        }
        if (ok) mma_commit_pair(bar_accf + 8 * (j & 1), 3);
      }
      if (!ok) {  // the MMAs in flight finish before TMEM and shared memory are released
        volatile int no_abort = 0;
        mma_commit_pair(bar_drain, 1);
        mbar_wait(bar_drain, 0, &no_abort);
        atomicExch(&g_proj_error, 1);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---- epilogue: TMEM lane = row of this CTA's block. Each warp turns its
    // 32 rows of a head around in shared memory (16-byte chunks xor-swizzled
    // by row: a 128-byte-swizzled box) and one lane stores the box with the
    // TMA; two buffers per warp, so a head is staged while the previous
    // head's box is read out. A K/V box that reaches past the block's valid
    // rows (their successors belong to another block) is stored row by row.
    const uint32_t stg0 = sb + P_STG + warp * 8192;
    const uint32_t acce0 = mapa_shared(bar_acce, 0);
    const int rr0 = lane >> 3, c = lane & 7;
    int nst = 0;  // boxes this warp handed to the TMA
    bool ok = true;
    for (int j = 0; j < nj; ++j) {
      const ProjItem it = item(j);
      const uint32_t trow = tmem + 256 * (j & 1) + ((uint32_t)(warp * 32) << 16);
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar_accf + 8 * (j & 1), (j >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      // Q rows past the block are past L (the box is clipped); K/V rows are not
      const bool any = warp * 32 < it.nvalid;
      const bool by_tma = any && (!it.kv || warp * 32 + 32 <= it.nvalid);
      for (int hh = 0; hh < it.nh; ++hh) {
        uint32_t lo[32], hi[32];
        tmem_ld32(trow + 64 * hh, lo);
        tmem_ld32(trow + 64 * hh + 32, hi);
        tmem_wait_ld();
        if (hh == it.nh - 1) {  // the accumulator may take unit j+2
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acce0 + 8 * (j & 1));
        }
        if (!it.store || !any) continue;
        const uint32_t stg = stg0 + (nst & 1) * 4096, srow = stg + lane * 128;
        // the box stored from this buffer two boxes ago has been read
        if (lane == 0) bulk_wait_read_but_latest();
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          st_shared_v4(srow + ((e ^ (lane & 7)) << 4),
                       pack_bf16(__uint_as_float(lo[8 * e]), __uint_as_float(lo[8 * e + 1])),
                       pack_bf16(__uint_as_float(lo[8 * e + 2]), __uint_as_float(lo[8 * e + 3])),
                       pack_bf16(__uint_as_float(lo[8 * e + 4]), __uint_as_float(lo[8 * e + 5])),
                       pack_bf16(__uint_as_float(lo[8 * e + 6]), __uint_as_float(lo[8 * e + 7])));
          st_shared_v4(srow + (((4 + e) ^ (lane & 7)) << 4),
                       pack_bf16(__uint_as_float(hi[8 * e]), __uint_as_float(hi[8 * e + 1])),
                       pack_bf16(__uint_as_float(hi[8 * e + 2]), __uint_as_float(hi[8 * e + 3])),
                       pack_bf16(__uint_as_float(hi[8 * e + 4]), __uint_as_float(hi[8 * e + 5])),
                       pack_bf16(__uint_as_float(hi[8 * e + 6]), __uint_as_float(hi[8 * e + 7])));
        }
        if (by_tma) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(it.omap, 0, it.orow0 + warp * 32, it.b * p.H + it.h0 + hh, stg);
            bulk_commit();
          }
          ++nst;
        } else {
          __syncwarp();
          __nv_bfloat16 *obase =
              it.out + (((size_t)it.b * p.H + it.h0 + hh) * it.orows + it.orow0 + warp * 32) * DH + c * 8;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + rr0;
            const uint4 v = ld_shared_v4(stg + rr * 128 + ((c ^ (rr & 7)) << 4));
            if (warp * 32 + rr < it.nvalid) *(uint4 *)(obase + rr * DH) = v;
          }
          __syncwarp();
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // every box written before the CTA leaves
    __syncwarp();
    if (!ok) atomicExch(&g_proj_error, 2);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still touch its shared memory or TMEM
  tc_fence_after();
  if (warp == 5) tmem_dealloc_pair(tmem, 512);
}

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

// bf16 [planes][rows][inner], boxes of 64 x box_rows, 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, int planes, int rows, int inner, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)rows * inner * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc_proj(const AttnShape &s, int d, const void *h_mem, const void *h_cur,
                           const void *wq, const void *wk, const void *wv, void *q, void *k, void *v,
                           cudaStream_t st, int *launches) {
  CUtensorMap thm, thc, twq, twk, twv, toq, tok, tov;
  const int n = s.H * DH;
  if (!make_map(&toq, q, s.B * s.H, s.L, DH, 32) || !make_map(&tok, k, s.B * s.H, s.cap + s.L, DH, 32) ||
      !make_map(&tov, v, s.B * s.H, s.cap + s.L, DH, 32) || !make_map(&thc, h_cur, s.B, s.L, d, BQ) ||
      !make_map(&thm, s.cap > 0 ? h_mem : h_cur, s.B, s.cap > 0 ? s.cap : s.L, d, BQ) ||
      !make_map(&twq, wq, 1, d, n, 64) || !make_map(&twk, wk, 1, d, n, 64) ||
      !make_map(&twv, wv, 1, d, n, 64))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(rxl_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  ProjParams p;
  p.B = s.B; p.H = s.H; p.L = s.L; p.cap = s.cap; p.m = s.m; p.head = s.head; p.d = d;
  p.NT = (s.H + 3) / 4;
  p.Tq = (s.L + BQ - 1) / BQ;
  {
    const int lenA = s.m < s.cap - s.head ? s.m : s.cap - s.head;
    const int lenB = s.m - lenA;
    p.Tkv = (lenA + BK - 1) / BK + (lenB + BK - 1) / BK + (s.L + BK - 1) / BK;
  }
  p.pairs_q = (s.B * p.Tq + 1) / 2;
  p.pairs_kv = (s.B * p.Tkv + 1) / 2;
  p.out[0] = (__nv_bfloat16 *)q; p.out[1] = (__nv_bfloat16 *)k; p.out[2] = (__nv_bfloat16 *)v;
  const long long units = (long long)p.NT * (p.pairs_q + 2LL * p.pairs_kv);
  if (units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = P_SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent pairs: as many as can be resident at once
  static std::once_flag occ_once;
  static int max_pairs = 0;
  std::call_once(occ_once, [&] {
    cudaLaunchConfig_t one = cfg;
    one.gridDim = dim3(2);
    if (cudaOccupancyMaxActiveClusters(&max_pairs, rxl_proj_kernel, &one) != cudaSuccess) max_pairs = 0;
  });
  if (max_pairs <= 0) return cudaErrorLaunchOutOfResources;
  const long long pairs = units < max_pairs ? units : max_pairs;
  cudaError_t e = launch_ex(rxl_proj_kernel, dim3((unsigned)(2 * pairs)), dim3(P_THREADS), P_SMEM, st, 2, thm, thc,
                            twq, twk, twv, toq, tok, tov, p, (int)units);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t tc_proj_read_error(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_proj_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_proj_error, &zero, sizeof(int));
  return e;
}

}  // namespace rxl
