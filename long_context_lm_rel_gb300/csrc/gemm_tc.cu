// Dense layers of the Transformer-XL block on sm_103a tensor cores:
//   out[b, i, :] = act(A[b, i, :] . W + bias) + residual[b, i, :]
// with bf16 operands, fp32 accumulation in TMEM and a bf16 result.
//
// The rows are B groups of R rows (a batch row's R positions); a 128-row tile
// never straddles two groups. A is either a row-major [B, R, K] activation or
// the attention output O [B, H, R, 64] read as [B, R, H*64] (heads merged by
// the TMA box coordinates, no copy). W is [K, N] row-major. One CTA computes a
// 128 x 256 output block (128 x 128 when the 256-wide blocks would leave half
// the SMs idle) with K streamed in 64-wide steps through a 4-stage
// TMA pipeline (the structure of the projection kernel), then four epilogue
// warps add the bias, apply ReLU, add the residual and store bf16 rows.
// With at most a quarter as many output blocks as SMs (few rows: short
// segments) the K range is split over S CTAs per block: each stores its fp32 partial block
// and a finalize kernel sums the S partials before bias, ReLU and residual.
#include <math.h>

#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace rxl {
namespace {

using namespace sm103;
using namespace tc;

constexpr int G_STAGES = 4;
constexpr int G_THREADS = 160;  // warps 0-3 epilogue, warp 4 TMA + MMA
constexpr uint32_t G_A_BYTES = 128 * 64 * 2;
constexpr uint32_t G_B_BYTES = 4 * 64 * 64 * 2;
constexpr uint32_t G_STAGE = G_A_BYTES + G_B_BYTES;
constexpr uint32_t G_BAR = G_STAGES * G_STAGE;
constexpr uint32_t G_SMEM = G_BAR + 128 + 1024;

__device__ int g_gemm_error;

struct GemmParams {
  int B, R, K, N;
  int Tr, Tn;  // row tiles per group, column tiles of TN columns
  int TN;      // 256, or 128 when the 256-wide blocks would fill at most half the SMs
  int splits;       // K split over this many CTAs per output block (1: no split)
  float *partials;  // splits > 1: [splits][B * R][N] fp32 partial sums
  const __nv_bfloat16 *bias;      // [N] or null
  const __nv_bfloat16 *residual;  // [B, R, N] or null
  __nv_bfloat16 *out;             // [B, R, N]
  int relu;
};

template <bool A_HEADS>
__global__ void __launch_bounds__(G_THREADS, 1)
rxl_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = p.B * p.Tr * p.Tn;
  const int z = blockIdx.x / tiles, tile = blockIdx.x % tiles;  // K split, output block
  const int nt = tile % p.Tn;
  const int rt = (tile / p.Tn) % p.Tr;
  const int b = tile / (p.Tn * p.Tr);
  const int row0 = rt * 128, nrows = min(128, p.R - row0);
  const int col0 = nt * p.TN, ncols = min(p.TN, p.N - col0), nbox = (ncols + 63) / 64;

  const uint32_t bar_full = sb + G_BAR, bar_empty = bar_full + 8 * G_STAGES;
  const uint32_t bar_done = bar_empty + 8 * G_STAGES;
  uint32_t *tmem_slot = (uint32_t *)(smem + G_BAR + 16 * G_STAGES + 8);
  volatile int *abort_flag = (volatile int *)(smem + G_BAR + 16 * G_STAGES + 12);
  if (threadIdx.x == 0) {
    for (int s = 0; s < G_STAGES; ++s) {
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
  griddep_wait();  // inputs written by the previous kernel on the stream
  griddep_launch_dependents();
  // this CTA's 64-wide k-steps [kb, ke)
  const int nk_all = p.K / 64;
  const int kb = z * nk_all / p.splits, ke = (z + 1) * nk_all / p.splits, nk = ke - kb;

  if (warp == 4) {
    if (lane == 0) {
      int issued[G_STAGES] = {0, 0, 0, 0};
      auto load = [&](int kt) {  // kt counts from kb
        const int s = kt % G_STAGES;
        const int kg = kb + kt;
        const uint32_t a = sb + s * G_STAGE, bb = a + G_A_BYTES;
        mbar_expect_tx(bar_full + 8 * s, G_A_BYTES + nbox * 8192);
        if (A_HEADS)  // k-step kg is head kg of O [B, H, R, 64]
          tma_load_4d(a, &tm_a, 0, row0, kg, b, bar_full + 8 * s);
        else
          tma_load_3d(a, &tm_a, kg * 64, row0, b, bar_full + 8 * s);
        for (int j = 0; j < nbox; ++j)
          tma_load_3d(bb + j * 8192, &tm_w, col0 + 64 * j, kg * 64, 0, bar_full + 8 * s);
        ++issued[s];
      };
      const uint32_t idesc = idesc_bf16(128, 64 * nbox, false, true);
      bool ok = true;
      for (int kt = 0; kt < nk && kt < G_STAGES; ++kt) load(kt);
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % G_STAGES;
        if (!(ok = mbar_wait(bar_full + 8 * s, (kt / G_STAGES) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t a = sb + s * G_STAGE, bb = a + G_A_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(bb + k * 2048, 8192, 1024), idesc,
                   (kt > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_empty + 8 * s);
        // refill the previous k-step's stage once its MMAs are done: they
        // finish while this step's are queued, so the tensor pipe does not
        // run dry during the wait
        const int kp = kt - 1;
        if (kp >= 0 && kp + G_STAGES < nk) {
          const int sp = kp % G_STAGES;
          if (!(ok = mbar_wait(bar_empty + 8 * sp, (kp / G_STAGES) & 1, abort_flag))) break;
          load(kp + G_STAGES);
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int s = 0; s < G_STAGES; ++s)
          if (issued[s] > 0) mbar_wait(bar_full + 8 * s, (issued[s] - 1) & 1, &no_abort);
        atomicExch(&g_gemm_error, 1);
      }
      mma_commit(bar_done);
      if (!ok) {
        volatile int no_abort = 0;
        mbar_wait(bar_done, 0, &no_abort);
      }
    }
    __syncwarp();
  } else {
    const int r = warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_done, 0, abort_flag));
    if (ok) {
      tc_fence_after();
      const size_t orow = ((size_t)b * p.R + row0 + r) * p.N + col0;
      for (int c = 0; c < 2 * nbox; ++c) {  // 32-column chunks
        uint32_t acc[32];
        tmem_ld32(trow + 32 * c, acc);
        tmem_wait_ld();
        if (r >= nrows || 32 * c >= ncols) continue;
        if (p.splits > 1) {  // this split's fp32 partial; the finalize kernel does the rest
          float4 *dst = (float4 *)(p.partials + (size_t)z * p.B * p.R * p.N + orow + 32 * c);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(acc[4 * q]), __uint_as_float(acc[4 * q + 1]),
                                 __uint_as_float(acc[4 * q + 2]), __uint_as_float(acc[4 * q + 3]));
          continue;
        }
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(acc[e]);
        if (p.bias) {
          const uint4 *bp = (const uint4 *)(p.bias + col0 + 32 * c);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w = bp[q];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              f[8 * q + 2 * t] += __uint_as_float(ww[t] << 16);
              f[8 * q + 2 * t + 1] += __uint_as_float(ww[t] & 0xFFFF0000u);
            }
          }
        }
        if (p.relu) {
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = fmaxf(f[e], 0.f);
        }
        if (p.residual) {
          const uint4 *rp = (const uint4 *)(p.residual + orow + 32 * c);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w = rp[q];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              f[8 * q + 2 * t] += __uint_as_float(ww[t] << 16);
              f[8 * q + 2 * t + 1] += __uint_as_float(ww[t] & 0xFFFF0000u);
            }
          }
        }
        uint4 *dst = (uint4 *)(p.out + orow + 32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pack_bf16(f[8 * q], f[8 * q + 1]), pack_bf16(f[8 * q + 2], f[8 * q + 3]),
                              pack_bf16(f[8 * q + 4], f[8 * q + 5]), pack_bf16(f[8 * q + 6], f[8 * q + 7]));
      }
    } else {
      atomicExch(&g_gemm_error, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 256);
}

// Split K: out = act(sum of the partials + bias) + residual, 8 columns per thread.
__global__ void __launch_bounds__(256) gemm_finalize_kernel(const float *__restrict__ partials, int splits,
                                                            long long rows, int N,
                                                            const __nv_bfloat16 *__restrict__ bias, int relu,
                                                            const __nv_bfloat16 *__restrict__ residual,
                                                            __nv_bfloat16 *__restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const long long n8 = rows * (N / 8), plane = rows * N;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n8;
       e += (long long)gridDim.x * blockDim.x) {
    const long long off = e * 8;
    const int col = (int)(off % N);
    float f[8];
    {
      const float4 a = *(const float4 *)(partials + off), b = *(const float4 *)(partials + off + 4);
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
#pragma unroll
    for (int zz = 1; zz < 8; ++zz) {  // splits <= 8: every load of the row group in flight at once
      if (zz >= splits) break;
      const float4 a = *(const float4 *)(partials + zz * plane + off);
      const float4 b = *(const float4 *)(partials + zz * plane + off + 4);
      f[0] += a.x; f[1] += a.y; f[2] += a.z; f[3] += a.w; f[4] += b.x; f[5] += b.y; f[6] += b.z; f[7] += b.w;
    }
    if (bias) {
      const uint4 w = *(const uint4 *)(bias + col);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        f[2 * t] += __uint_as_float(ww[t] << 16);
        f[2 * t + 1] += __uint_as_float(ww[t] & 0xFFFF0000u);
      }
    }
    if (relu) {
#pragma unroll
      for (int t = 0; t < 8; ++t) f[t] = fmaxf(f[t], 0.f);
    }
    if (residual) {
      const uint4 w = *(const uint4 *)(residual + off);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        f[2 * t] += __uint_as_float(ww[t] << 16);
        f[2 * t + 1] += __uint_as_float(ww[t] & 0xFFFF0000u);
      }
    }
    *(uint4 *)(out + off) = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                                       pack_bf16(f[6], f[7]));
  }
}

// Split K followed by the block's LayerNorm, one CTA per row and 8 columns
// per thread (N / 8 <= 1024 threads, so a row is read once and stays in
// registers): x = act(sum of the partials + bias) + residual, rounded to
// bf16 (what the separate pass would store), then y = LayerNorm(x) with fp32
// statistics: mean, then the mean squared deviation, each summed per thread,
// per warp and over the CTA.
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();  // red may still be read from the previous sum
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < nw; ++w) s += red[w];
  return s;
}

__global__ void __launch_bounds__(1024) gemm_finalize_ln_kernel(const float *__restrict__ partials, int splits,
                                                                long long rows, int N,
                                                                const __nv_bfloat16 *__restrict__ bias, int relu,
                                                                const __nv_bfloat16 *__restrict__ residual,
                                                                const __nv_bfloat16 *__restrict__ gamma,
                                                                const __nv_bfloat16 *__restrict__ beta, float eps,
                                                                __nv_bfloat16 *__restrict__ y) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[32];
  const long long row = blockIdx.x;
  const int c = threadIdx.x;  // 16-byte chunk of the row; blockDim.x == N / 8
  const long long plane = rows * N, off = row * N + 8 * c;
  float f[8];
  {
    const float4 a = *(const float4 *)(partials + off), b = *(const float4 *)(partials + off + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
#pragma unroll
  for (int zz = 1; zz < 8; ++zz) {  // splits <= 8: every load of the row group in flight at once
    if (zz >= splits) break;
    const float4 a = *(const float4 *)(partials + zz * plane + off);
    const float4 b = *(const float4 *)(partials + zz * plane + off + 4);
    f[0] += a.x; f[1] += a.y; f[2] += a.z; f[3] += a.w; f[4] += b.x; f[5] += b.y; f[6] += b.z; f[7] += b.w;
  }
  if (bias) {
    const uint4 w = *(const uint4 *)(bias + 8 * c);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      f[2 * t] += __uint_as_float(ww[t] << 16);
      f[2 * t + 1] += __uint_as_float(ww[t] & 0xFFFF0000u);
    }
  }
  if (relu) {
#pragma unroll
    for (int t = 0; t < 8; ++t) f[t] = fmaxf(f[t], 0.f);
  }
  if (residual) {
    const uint4 w = *(const uint4 *)(residual + off);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      f[2 * t] += __uint_as_float(ww[t] << 16);
      f[2 * t + 1] += __uint_as_float(ww[t] & 0xFFFF0000u);
    }
  }
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {  // the bf16 value the separate pass would read
    const uint32_t w = pack_bf16(f[2 * t], f[2 * t + 1]);
    f[2 * t] = __uint_as_float(w << 16);
    f[2 * t + 1] = __uint_as_float(w & 0xFFFF0000u);
    s += f[2 * t] + f[2 * t + 1];
  }
  const float mean = block_sum(s, red) / N;
  float v = 0.f;
#pragma unroll
  for (int t = 0; t < 8; ++t) v += (f[t] - mean) * (f[t] - mean);
  const float rstd = rsqrtf(block_sum(v, red) / N + eps);
  const uint4 g = *(const uint4 *)(gamma + 8 * c), bt = *(const uint4 *)(beta + 8 * c);
  const uint32_t gg[4] = {g.x, g.y, g.z, g.w}, bb[4] = {bt.x, bt.y, bt.z, bt.w};
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    o[t] = pack_bf16((f[2 * t] - mean) * rstd * __uint_as_float(gg[t] << 16) + __uint_as_float(bb[t] << 16),
                     (f[2 * t + 1] - mean) * rstd * __uint_as_float(gg[t] & 0xFFFF0000u) +
                         __uint_as_float(bb[t] & 0xFFFF0000u));
  *(uint4 *)(y + off) = make_uint4(o[0], o[1], o[2], o[3]);
}

// LayerNorm over the last dimension (one warp per row, statistics in fp32):
// y = (x - mean) / sqrt(var + eps) * gamma + beta, var the biased variance.
__global__ void __launch_bounds__(256) layernorm_kernel(const __nv_bfloat16 *__restrict__ x,
                                                        const __nv_bfloat16 *__restrict__ gamma,
                                                        const __nv_bfloat16 *__restrict__ beta,
                                                        __nv_bfloat16 *__restrict__ y, long long rows,
                                                        int d, float eps) {
  griddep_wait();
  griddep_launch_dependents();
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4 *xr = (const uint4 *)(x + row * d);
  const int chunks = d / 8;  // 16-byte chunks, d % 256 == 0 -> a multiple of 32
  float s = 0.f;
  for (int c = lane; c < chunks; c += 32) {
    const uint4 w = xr[c];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) s += __uint_as_float(ww[t] << 16) + __uint_as_float(ww[t] & 0xFFFF0000u);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s / d;
  float v = 0.f;
  for (int c = lane; c < chunks; c += 32) {
    const uint4 w = xr[c];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float a = __uint_as_float(ww[t] << 16) - mean, bb = __uint_as_float(ww[t] & 0xFFFF0000u) - mean;
      v += a * a + bb * bb;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const float rstd = rsqrtf(v / d + eps);
  uint4 *yr = (uint4 *)(y + row * d);
  const uint4 *gr = (const uint4 *)gamma, *br = (const uint4 *)beta;
  for (int c = lane; c < chunks; c += 32) {
    const uint4 w = xr[c], g = gr[c], bt = br[c];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w}, gg[4] = {g.x, g.y, g.z, g.w}, bb[4] = {bt.x, bt.y, bt.z, bt.w};
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float a = (__uint_as_float(ww[t] << 16) - mean) * rstd * __uint_as_float(gg[t] << 16) +
                      __uint_as_float(bb[t] << 16);
      const float c2 = (__uint_as_float(ww[t] & 0xFFFF0000u) - mean) * rstd *
                           __uint_as_float(gg[t] & 0xFFFF0000u) +
                       __uint_as_float(bb[t] & 0xFFFF0000u);
      o[t] = pack_bf16(a, c2);
    }
    yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
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

// bf16 tensor of `rank` dims (innermost first), 64 x box_rows boxes, 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t strides[4];
  cuuint64_t acc = dims[0] * 2;
  for (int i = 1; i < rank; ++i) {
    strides[i - 1] = acc;
    acc *= dims[i];
  }
  const cuuint32_t box[5] = {64, (cuuint32_t)box_rows, 1, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc_gemm(int B, int R, int K, int N, const void *a, bool a_heads, const void *w,
                           const void *bias, const void *residual, bool relu, void *out,
                           float *partials, size_t partial_floats, const void *ln_gamma, const void *ln_beta,
                           float ln_eps, void *ln_out, cudaStream_t st, int *launches) {
  CUtensorMap ta, tw;
  bool ok;
  if (a_heads) {  // O [B, K/64, R, 64]
    const cuuint64_t dims[4] = {64, (cuuint64_t)R, (cuuint64_t)(K / 64), (cuuint64_t)B};
    ok = make_map(&ta, a, 4, dims, 128);
  } else {
    const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)R, (cuuint64_t)B};
    ok = make_map(&ta, a, 3, dims, 128);
  }
  const cuuint64_t wdims[3] = {(cuuint64_t)N, (cuuint64_t)K, 1};
  if (!ok || !make_map(&tw, w, 3, wdims, 64)) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(rxl_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(rxl_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  GemmParams p;
  p.B = B; p.R = R; p.K = K; p.N = N;
  p.Tr = (R + 127) / 128;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // 128-column blocks when the 256-column ones would fill at most half the
  // SMs: twice the CTAs, each streaming a third less per k-step
  p.TN = 2LL * B * p.Tr * ((N + 255) / 256) <= sms ? 128 : 256;
  p.Tn = (N + p.TN - 1) / p.TN;
  p.bias = (const __nv_bfloat16 *)bias;
  p.residual = (const __nv_bfloat16 *)residual;
  p.out = (__nv_bfloat16 *)out;
  p.relu = relu ? 1 : 0;
  const long long tiles = (long long)B * p.Tr * p.Tn;
  // split K when the blocks fill at most a quarter of the SMs: as many
  // splits as fit the SMs, at least two k-steps each, at most 8, within the
  // partial budget; fewer than 4 splits do not repay the finalize pass
  const long long per_split = (long long)B * R * N;
  long long S = 1;
  if (partials && 4 * tiles <= sms) {
    S = sms / tiles;
    if (S > K / 128) S = K / 128;
    if (S > 8) S = 8;
    if (S > (long long)(partial_floats / per_split)) S = (long long)(partial_floats / per_split);
    if (S < 4) S = 1;
  }
  p.splits = (int)S;
  p.partials = partials;
  const unsigned grid = (unsigned)(tiles * S);
  const long long rows = (long long)B * R;
  cudaError_t e = a_heads ? launch_ex(rxl_gemm_kernel<true>, dim3(grid), dim3(G_THREADS), G_SMEM, st, 1, ta, tw, p)
                          : launch_ex(rxl_gemm_kernel<false>, dim3(grid), dim3(G_THREADS), G_SMEM, st, 1, ta, tw, p);
  ++*launches;
  if (e != cudaSuccess) return e;
  const __nv_bfloat16 *bias16 = (const __nv_bfloat16 *)bias, *res16 = (const __nv_bfloat16 *)residual;
  const __nv_bfloat16 *g16 = (const __nv_bfloat16 *)ln_gamma, *b16 = (const __nv_bfloat16 *)ln_beta;
  const bool fused_ln = ln_out && S > 1 && N / 8 <= 1024;
  if (S > 1) {
    long long blocks = (per_split / 8 + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    if (fused_ln)  // the sum of the partials and the LayerNorm in one pass over the rows
      e = launch_ex(gemm_finalize_ln_kernel, dim3((unsigned)rows), dim3((unsigned)(N / 8)), 0, st, 1,
                    (const float *)partials, (int)S, rows, N, bias16, relu ? 1 : 0, res16, g16, b16, ln_eps,
                    (__nv_bfloat16 *)ln_out);
    else
      e = launch_ex(gemm_finalize_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, (const float *)partials,
                    (int)S, rows, N, bias16, relu ? 1 : 0, res16, (__nv_bfloat16 *)out);
    ++*launches;
    if (e != cudaSuccess) return e;
  }
  if (ln_out && !fused_ln) {
    e = launch_ex(layernorm_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, st, 1,
                  (const __nv_bfloat16 *)out, g16, b16, (__nv_bfloat16 *)ln_out, rows, N, ln_eps);
    ++*launches;
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t tc_gemm_read_error(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_gemm_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
  return e;
}

}  // namespace rxl
