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
// One CTA computes one output block: 128 hidden-state rows of one batch row
// times up to 4 heads (N <= 256 columns) of one of Q, K, V, with the hidden
// width d streamed in 64-wide steps through a 4-stage TMA pipeline:
//   A = hidden rows [128][64] bf16 (K-major, 128-byte swizzle)
//   B = W rows [64][N] bf16 (MN-major: 64x64 swizzled boxes, 8 KB apart)
//   D = TMEM [128 lanes][N] fp32; four epilogue warps write bf16 rows of
//   64 columns per head.
#include <math.h>

#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace rxl {
namespace {

using namespace sm103;
using namespace tc;

constexpr int P_STAGES = 4;
constexpr int P_THREADS = 160;  // warps 0-3 epilogue (TMEM lane quadrants), warp 4 TMA + MMA
constexpr uint32_t P_A_BYTES = 128 * 64 * 2;  // 16 KB
constexpr uint32_t P_B_BYTES = 4 * 64 * 64 * 2;  // 32 KB (up to four 64-column boxes)
constexpr uint32_t P_STAGE = P_A_BYTES + P_B_BYTES;
constexpr uint32_t P_BAR = P_STAGES * P_STAGE;
constexpr uint32_t P_SMEM = P_BAR + 128 + 1024;

__device__ int g_proj_error;

struct ProjParams {
  int B, H, L, cap, m, head, d;
  int NT;        // column tiles of up to 4 heads
  int Tq, Tkv;   // row tiles of Q and of K/V per batch row
  __nv_bfloat16 *out[3];  // q, k, v
};

__global__ void __launch_bounds__(P_THREADS, 1)
rxl_proj_kernel(const __grid_constant__ CUtensorMap tm_hmem, const __grid_constant__ CUtensorMap tm_hcur,
                const __grid_constant__ CUtensorMap tm_wq, const __grid_constant__ CUtensorMap tm_wk,
                const __grid_constant__ CUtensorMap tm_wv, const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which output block
  const int per_b = p.NT * (p.Tq + 2 * p.Tkv);
  const int b = blockIdx.x / per_b;
  int rest = blockIdx.x % per_b;
  const int nt = rest % p.NT;
  rest /= p.NT;
  int which, tile;  // 0 q, 1 k, 2 v
  if (rest < p.Tq) {
    which = 0;
    tile = rest;
  } else {
    rest -= p.Tq;
    which = 1 + rest / p.Tkv;
    tile = rest % p.Tkv;
  }
  const int h0 = 4 * nt, nh = min(4, p.H - h0), N = 64 * nh;
  // source rows and output rows of the block
  const CUtensorMap *amap = &tm_hcur;
  int arow, orow0, nvalid, orows;
  if (which == 0) {
    arow = tile * BQ;
    orow0 = arow;
    nvalid = min(BQ, p.L - arow);
    orows = p.L;
  } else {
    const KeyTiles tiles(p.m, p.cap, p.head, p.L);
    const KeyTile x = tiles.get(tile);
    const bool mem = x.jlog0 < 0;
    amap = mem ? &tm_hmem : &tm_hcur;
    arow = mem ? x.phys0 : x.jlog0;
    orow0 = x.phys0;
    nvalid = x.nvalid;
    orows = p.cap + p.L;
  }
  const CUtensorMap *wmap = which == 0 ? &tm_wq : (which == 1 ? &tm_wk : &tm_wv);
  __nv_bfloat16 *out = p.out[which];

  const uint32_t bar_full = sb + P_BAR, bar_empty = bar_full + 8 * P_STAGES;
  const uint32_t bar_done = bar_empty + 8 * P_STAGES;
  uint32_t *tmem_slot = (uint32_t *)(smem + P_BAR + 16 * P_STAGES + 8);
  volatile int *abort_flag = (volatile int *)(smem + P_BAR + 16 * P_STAGES + 12);
  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 4) tmem_alloc(smem_u32(tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nk = p.d / 64;

  if (warp == 4) {
    if (lane == 0) {
      int issued[P_STAGES] = {0, 0, 0, 0};
      auto load = [&](int kt) {
        const int s = kt % P_STAGES;
        const uint32_t a = sb + s * P_STAGE, bb = a + P_A_BYTES;
        mbar_expect_tx(bar_full + 8 * s, P_A_BYTES + nh * 8192);
        tma_load_3d(a, amap, kt * 64, arow, b, bar_full + 8 * s);
        for (int j = 0; j < nh; ++j)
          tma_load_3d(bb + j * 8192, wmap, (h0 + j) * 64, kt * 64, 0, bar_full + 8 * s);
        ++issued[s];
      };
      const uint32_t idesc = idesc_bf16(128, N, false, true);
      bool ok = true;
      for (int kt = 0; kt < nk && kt < P_STAGES; ++kt) load(kt);
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % P_STAGES;
        if (!(ok = mbar_wait(bar_full + 8 * s, (kt / P_STAGES) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t a = sb + s * P_STAGE, bb = a + P_A_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(bb + k * 2048, 8192, 1024), idesc,
                   (kt > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_empty + 8 * s);
        // refill the previous k-step's stage once its MMAs are done: they
        // finish while this step's are queued, so the tensor pipe does not
        // run dry during the wait
        const int kp = kt - 1;
        if (kp >= 0 && kp + P_STAGES < nk) {
          const int sp = kp % P_STAGES;
          if (!(ok = mbar_wait(bar_empty + 8 * sp, (kp / P_STAGES) & 1, abort_flag))) break;
          load(kp + P_STAGES);
        }
      }
      if (!ok) {
        // let in-flight copies land before shared memory is released
        volatile int no_abort = 0;
        for (int s = 0; s < P_STAGES; ++s)
          if (issued[s] > 0) mbar_wait(bar_full + 8 * s, (issued[s] - 1) & 1, &no_abort);
        atomicExch(&g_proj_error, 1);
      }
      mma_commit(bar_done);
      if (!ok) {  // the epilogue gives up at once: wait for the MMAs here
        volatile int no_abort = 0;
        mbar_wait(bar_done, 0, &no_abort);
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: TMEM lane = row of the block
    const int r = warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_done, 0, abort_flag));
    if (ok) {
      tc_fence_after();
      for (int hh = 0; hh < nh; ++hh) {
        uint32_t lo[32], hi[32];
        tmem_ld32(trow + 64 * hh, lo);
        tmem_ld32(trow + 64 * hh + 32, hi);
        tmem_wait_ld();
        if (r < nvalid) {
          uint4 *dst = (uint4 *)(out + (((size_t)b * p.H + h0 + hh) * orows + orow0 + r) * DH);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dst[e] = make_uint4(pack_bf16(__uint_as_float(lo[8 * e]), __uint_as_float(lo[8 * e + 1])),
                                pack_bf16(__uint_as_float(lo[8 * e + 2]), __uint_as_float(lo[8 * e + 3])),
                                pack_bf16(__uint_as_float(lo[8 * e + 4]), __uint_as_float(lo[8 * e + 5])),
                                pack_bf16(__uint_as_float(lo[8 * e + 6]), __uint_as_float(lo[8 * e + 7])));
            dst[4 + e] = make_uint4(pack_bf16(__uint_as_float(hi[8 * e]), __uint_as_float(hi[8 * e + 1])),
                                    pack_bf16(__uint_as_float(hi[8 * e + 2]), __uint_as_float(hi[8 * e + 3])),
                                    pack_bf16(__uint_as_float(hi[8 * e + 4]), __uint_as_float(hi[8 * e + 5])),
                                    pack_bf16(__uint_as_float(hi[8 * e + 6]), __uint_as_float(hi[8 * e + 7])));
          }
        }
      }
    } else {
      atomicExch(&g_proj_error, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 256);
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
  CUtensorMap thm, thc, twq, twk, twv;
  const int n = s.H * DH;
  if (!make_map(&thc, h_cur, s.B, s.L, d, BQ) ||
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
  p.out[0] = (__nv_bfloat16 *)q; p.out[1] = (__nv_bfloat16 *)k; p.out[2] = (__nv_bfloat16 *)v;
  const long long blocks = (long long)s.B * p.NT * (p.Tq + 2 * p.Tkv);
  rxl_proj_kernel<<<(unsigned)blocks, P_THREADS, P_SMEM, st>>>(thm, thc, twq, twk, twv, p);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t tc_proj_read_error(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_proj_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_proj_error, &zero, sizeof(int));
  return e;
}

}  // namespace rxl
