// CUDA-core (FFMA) relative-position memory attention, forward and backward.
//
// This is the float32 path (exact fp32 arithmetic for the 1e-5 tolerance
// that tensor-core TF32 cannot meet). One warp owns one output row; each
// lane owns two of the 64 head-width columns, so every row read (K, V, R,
// dO) is one coalesced 256-byte (fp32) transaction.
//
// Math (Transformer-XL page, "Relative Positional Encoding" and "Dimension
// Walkthrough"): A_ij = (q_i+u).k_j + (q_i+v).r_{i-j}, logits scale*A_ij
// where allow(i,j) ("Causal Mask With Memory"), softmax, times V. The
// backward is the chain rule of that expression with stop-gradient on the
// cache ("Why Stop Gradient"): memory rows get dK/dV, the cache is never
// written. Every reduction runs in a fixed order, so results are
// bit-reproducible run to run.
#include <math.h>

#include "internal.cuh"

namespace rxl {
namespace {

template <typename T>
__device__ __forceinline__ float2 ld2(const T *p);
template <>
__device__ __forceinline__ float2 ld2<float>(const float *p) {
  return *reinterpret_cast<const float2 *>(p);
}
template <>
__device__ __forceinline__ float2 ld2<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
template <typename T>
__device__ __forceinline__ void st2(T *p, float2 x);
template <>
__device__ __forceinline__ void st2<float>(float *p, float2 x) {
  *reinterpret_cast<float2 *>(p) = x;
}
template <>
__device__ __forceinline__ void st2<__nv_bfloat16>(__nv_bfloat16 *p, float2 x) {
  *reinterpret_cast<__nv_bfloat162 *>(p) = __float22bfloat162_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ float dot2(float2 a, float2 b) { return a.x * b.x + a.y * b.y; }

// Physical K/V row of logical key position j in [-m, L).
__device__ __forceinline__ int phys_row(const AttnShape &s, int j) {
  if (j >= 0) return s.cap + j;
  int t = s.head + s.m + j;  // logical memory row m+j, rotated by head
  return t >= s.cap ? t - s.cap : t;
}

// Memory rows batch row b sees: all m, or under a per-row document reset its
// newest mvis[b] (clamped into [0, m]); they are logical positions -mb..-1.
__device__ __forceinline__ int row_m(const AttnShape &s, long long b) {
  if (!s.mvis) return s.m;
  const int mb = s.mvis[b];
  return mb < 0 ? 0 : (mb > s.m ? s.m : mb);
}

constexpr int kDh = 64;
constexpr int kWarps = 4;

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_fwd_kernel(
    AttnShape s, const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ r, const T *__restrict__ u, const T *__restrict__ vb,
    T *__restrict__ o, float *__restrict__ lse) {
  const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)s.B * s.H * s.L) return;
  const int i = (int)(row % s.L);
  const long long bh = row / s.L;
  const int h = (int)(bh % s.H);
  const float2 qq = ld2(q + row * kDh + 2 * lane);
  const float2 uu = ld2(u + h * kDh + 2 * lane), vv = ld2(vb + h * kDh + 2 * lane);
  const float2 qu = make_float2(qq.x + uu.x, qq.y + uu.y);
  const float2 qv = make_float2(qq.x + vv.x, qq.y + vv.y);
  const T *kb = k + bh * s.kv_rows * kDh, *vbase = v + bh * s.kv_rows * kDh;
  const T *rh = r + (long long)h * s.kv_rows * kDh;
  float mx = -INFINITY, l = 0.f;
  float2 acc = make_float2(0.f, 0.f);
  for (int j = -row_m(s, bh / s.H); j <= i; ++j) {
    const long long pr = phys_row(s, j);
    const float a = warp_sum(dot2(qu, ld2(kb + pr * kDh + 2 * lane)) +
                             dot2(qv, ld2(rh + (long long)(i - j) * kDh + 2 * lane)));
    const float z = a * s.scale;
    const float mnew = fmaxf(mx, z);
    const float corr = expf(mx - mnew);
    const float p = expf(z - mnew);
    const float2 vj = ld2(vbase + pr * kDh + 2 * lane);
    l = l * corr + p;
    acc.x = acc.x * corr + p * vj.x;
    acc.y = acc.y * corr + p * vj.y;
    mx = mnew;
  }
  const float inv = 1.f / l;
  st2(o + row * kDh + 2 * lane, make_float2(acc.x * inv, acc.y * inv));
  if (lane == 0) lse[row] = mx + logf(l);
}

// D_i = dO_i . O_i with O_i recomputed in fp32: D_i = sum_j P_ij (dO_i . V_j).
// The stored O is rounded to the input type; taking D from it would put that
// rounding error into every dS_ij of the row.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_d_kernel(
    AttnShape s, const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ r, const T *__restrict__ u, const T *__restrict__ vb,
    const float *__restrict__ lse, const T *__restrict__ dout, float *__restrict__ D) {
  const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)s.B * s.H * s.L) return;
  const int i = (int)(row % s.L);
  const long long bh = row / s.L;
  const int h = (int)(bh % s.H);
  const float2 qq = ld2(q + row * kDh + 2 * lane);
  const float2 uu = ld2(u + h * kDh + 2 * lane), vv = ld2(vb + h * kDh + 2 * lane);
  const float2 qu = make_float2(qq.x + uu.x, qq.y + uu.y);
  const float2 qv = make_float2(qq.x + vv.x, qq.y + vv.y);
  const float2 dO = ld2(dout + row * kDh + 2 * lane);
  const float lse_i = lse[row];
  const T *kb = k + bh * s.kv_rows * kDh, *vbase = v + bh * s.kv_rows * kDh;
  const T *rh = r + (long long)h * s.kv_rows * kDh;
  float2 acc = make_float2(0.f, 0.f);
  for (int j = -row_m(s, bh / s.H); j <= i; ++j) {
    const long long pr = phys_row(s, j);
    const float a = warp_sum(dot2(qu, ld2(kb + pr * kDh + 2 * lane)) +
                             dot2(qv, ld2(rh + (long long)(i - j) * kDh + 2 * lane)));
    const float p = expf(a * s.scale - lse_i);
    const float2 vj = ld2(vbase + pr * kDh + 2 * lane);
    acc.x += p * vj.x;
    acc.y += p * vj.y;
  }
  const float d = warp_sum(acc.x * dO.x + acc.y * dO.y);
  if (lane == 0) D[row] = d;
}

// Recomputes dA_ij for one (row i, key j) pair; all lanes return the value.
template <typename T>
__device__ __forceinline__ float recompute_dA(const AttnShape &s, float2 qu, float2 qv, float2 dO,
                                              float lse_i, float D_i, const T *krow,
                                              const T *vrow, const T *rrow, int lane,
                                              float *p_out) {
  const float a = warp_sum(dot2(qu, ld2(krow + 2 * lane)) + dot2(qv, ld2(rrow + 2 * lane)));
  const float p = expf(a * s.scale - lse_i);
  const float dp = warp_sum(dot2(dO, ld2(vrow + 2 * lane)));
  *p_out = p;
  return s.scale * p * (dp - D_i);
}

// dq (and the per-row content/position parts used for du, dv) per query row.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_dq_kernel(
    AttnShape s, const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ r, const T *__restrict__ u, const T *__restrict__ vb,
    const float *__restrict__ lse, const T *__restrict__ dout, const float *__restrict__ D,
    T *__restrict__ dq, float *__restrict__ dqu, float *__restrict__ dqv) {
  const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)s.B * s.H * s.L) return;
  const int i = (int)(row % s.L);
  const long long bh = row / s.L;
  const int h = (int)(bh % s.H);
  const float2 qq = ld2(q + row * kDh + 2 * lane);
  const float2 uu = ld2(u + h * kDh + 2 * lane), vv = ld2(vb + h * kDh + 2 * lane);
  const float2 qu = make_float2(qq.x + uu.x, qq.y + uu.y);
  const float2 qv = make_float2(qq.x + vv.x, qq.y + vv.y);
  const float2 dO = ld2(dout + row * kDh + 2 * lane);
  const float lse_i = lse[row], D_i = D[row];
  const T *kb = k + bh * s.kv_rows * kDh, *vbase = v + bh * s.kv_rows * kDh;
  const T *rh = r + (long long)h * s.kv_rows * kDh;
  float2 gu = make_float2(0.f, 0.f), gv = make_float2(0.f, 0.f);
  for (int j = -row_m(s, bh / s.H); j <= i; ++j) {
    const long long pr = phys_row(s, j);
    const T *rrow = rh + (long long)(i - j) * kDh;
    float p;
    const float dA = recompute_dA(s, qu, qv, dO, lse_i, D_i, kb + pr * kDh, vbase + pr * kDh,
                                  rrow, lane, &p);
    const float2 kj = ld2(kb + pr * kDh + 2 * lane), rd = ld2(rrow + 2 * lane);
    gu.x += dA * kj.x; gu.y += dA * kj.y;
    gv.x += dA * rd.x; gv.y += dA * rd.y;
  }
  st2(dq + row * kDh + 2 * lane, make_float2(gu.x + gv.x, gu.y + gv.y));
  *reinterpret_cast<float2 *>(dqu + row * kDh + 2 * lane) = gu;
  *reinterpret_cast<float2 *>(dqv + row * kDh + 2 * lane) = gv;
}

// dk, dv per physical key row (ring rows without valid memory get zeros).
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_dkv_kernel(
    AttnShape s, const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ r, const T *__restrict__ u, const T *__restrict__ vb,
    const float *__restrict__ lse, const T *__restrict__ dout, const float *__restrict__ D,
    T *__restrict__ dk, T *__restrict__ dv) {
  const long long krow = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (krow >= (long long)s.B * s.H * s.kv_rows) return;
  const int pr = (int)(krow % s.kv_rows);
  const long long bh = krow / s.kv_rows;
  const int h = (int)(bh % s.H);
  int j;
  if (pr < s.cap) {
    int t = pr - s.head;
    if (t < 0) t += s.cap;
    // ring rows that hold no valid memory, or that this batch row's document
    // reset masks, get zeros
    if (t >= s.m || t - s.m < -row_m(s, bh / s.H)) {
      st2(dk + krow * kDh + 2 * lane, make_float2(0.f, 0.f));
      st2(dv + krow * kDh + 2 * lane, make_float2(0.f, 0.f));
      return;
    }
    j = t - s.m;
  } else {
    j = pr - s.cap;
  }
  const float2 uu = ld2(u + h * kDh + 2 * lane), vv = ld2(vb + h * kDh + 2 * lane);
  const T *rh = r + (long long)h * s.kv_rows * kDh;
  float2 gk = make_float2(0.f, 0.f), gvv = make_float2(0.f, 0.f);
  for (int i = j < 0 ? 0 : j; i < s.L; ++i) {
    const long long qrow = bh * s.L + i;
    const float2 qq = ld2(q + qrow * kDh + 2 * lane);
    const float2 qu = make_float2(qq.x + uu.x, qq.y + uu.y);
    const float2 qv = make_float2(qq.x + vv.x, qq.y + vv.y);
    const float2 dO = ld2(dout + qrow * kDh + 2 * lane);
    float p;
    const float dA = recompute_dA(s, qu, qv, dO, lse[qrow], D[qrow], k + krow * kDh,
                                  v + krow * kDh, rh + (long long)(i - j) * kDh, lane, &p);
    gvv.x += p * dO.x; gvv.y += p * dO.y;
    gk.x += dA * qu.x; gk.y += dA * qu.y;
  }
  st2(dk + krow * kDh + 2 * lane, gk);
  st2(dv + krow * kDh + 2 * lane, gvv);
}

// dr_d per (head, distance): sum over b, then i, in fixed order.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) simt_bwd_dr_kernel(
    AttnShape s, const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ r, const T *__restrict__ u, const T *__restrict__ vb,
    const float *__restrict__ lse, const T *__restrict__ dout, const float *__restrict__ D,
    float *__restrict__ dr) {
  const long long w = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= (long long)s.H * s.kv_rows) return;
  const int d = (int)(w % s.kv_rows);
  const int h = (int)(w / s.kv_rows);
  float2 g = make_float2(0.f, 0.f);
  if (d < s.m + s.L) {
    const float2 uu = ld2(u + h * kDh + 2 * lane), vv = ld2(vb + h * kDh + 2 * lane);
    const T *rrow = r + ((long long)h * s.kv_rows + d) * kDh;
    for (int b = 0; b < s.B; ++b) {
      const long long bh = (long long)b * s.H + h;
      const T *kb = k + bh * s.kv_rows * kDh, *vbase = v + bh * s.kv_rows * kDh;
      const int mb = row_m(s, b);  // keys j = i - d >= -mb
      for (int i = d - mb > 0 ? d - mb : 0; i < s.L; ++i) {
        const int j = i - d;
        const long long qrow = bh * s.L + i;
        const long long pr = phys_row(s, j);
        const float2 qq = ld2(q + qrow * kDh + 2 * lane);
        const float2 qu = make_float2(qq.x + uu.x, qq.y + uu.y);
        const float2 qv = make_float2(qq.x + vv.x, qq.y + vv.y);
        float p;
        const float dA = recompute_dA(s, qu, qv, ld2(dout + qrow * kDh + 2 * lane), lse[qrow],
                                      D[qrow], kb + pr * kDh, vbase + pr * kDh, rrow, lane, &p);
        g.x += dA * qv.x; g.y += dA * qv.y;
      }
    }
  }
  *reinterpret_cast<float2 *>(dr + w * kDh + 2 * lane) = g;
}

// du[h], dv[h]: fixed-order sums of the per-row content/position parts of dq.
__global__ void simt_bwd_duv_kernel(AttnShape s, const float *__restrict__ dqu,
                                    const float *__restrict__ dqv, float *__restrict__ du,
                                    float *__restrict__ dvb) {
  const int h = blockIdx.x, c = threadIdx.x;  // 64 threads
  float a = 0.f, b2 = 0.f;
  for (int b = 0; b < s.B; ++b)
    for (int i = 0; i < s.L; ++i) {
      const long long row = ((long long)b * s.H + h) * s.L + i;
      a += dqu[row * kDh + c];
      b2 += dqv[row * kDh + c];
    }
  du[h * kDh + c] = a;
  dvb[h * kDh + c] = b2;
}

inline unsigned blocks_for(long long warps) { return (unsigned)((warps + kWarps - 1) / kWarps); }

template <typename T>
cudaError_t fwd_impl(const AttnShape &s, const void *q, const void *k, const void *v,
                     const void *r, const void *u, const void *vb, void *o, float *lse,
                     cudaStream_t st, int *launches) {
  const long long rows = (long long)s.B * s.H * s.L;
  simt_fwd_kernel<T><<<blocks_for(rows), kWarps * 32, 0, st>>>(
      s, (const T *)q, (const T *)k, (const T *)v, (const T *)r, (const T *)u, (const T *)vb,
      (T *)o, lse);
  ++*launches;
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_impl(const AttnShape &s, const void *q, const void *k, const void *v,
                     const void *r, const void *u, const void *vb, const void *o,
                     const float *lse, const void *dout, void *dq, void *dk, void *dv, float *dr,
                     float *du, float *dvb, void *ws, cudaStream_t st, int *launches) {
  const BwdWorkspace w = simt_bwd_workspace(s);
  float *D = (float *)((char *)ws + w.d_off);
  float *dqu = (float *)((char *)ws + w.dqu_off);
  float *dqv = (float *)((char *)ws + w.dqv_off);
  const long long rows = (long long)s.B * s.H * s.L;
  const T *Q = (const T *)q, *K = (const T *)k, *V = (const T *)v, *R = (const T *)r;
  const T *U = (const T *)u, *VB = (const T *)vb, *DO = (const T *)dout;
  simt_bwd_d_kernel<T><<<blocks_for(rows), kWarps * 32, 0, st>>>(s, Q, K, V, R, U, VB, lse, DO, D);
  simt_bwd_dq_kernel<T><<<blocks_for(rows), kWarps * 32, 0, st>>>(s, Q, K, V, R, U, VB, lse, DO,
                                                                 D, (T *)dq, dqu, dqv);
  simt_bwd_dkv_kernel<T><<<blocks_for((long long)s.B * s.H * s.kv_rows), kWarps * 32, 0, st>>>(
      s, Q, K, V, R, U, VB, lse, DO, D, (T *)dk, (T *)dv);
  simt_bwd_dr_kernel<T><<<blocks_for((long long)s.H * s.kv_rows), kWarps * 32, 0, st>>>(
      s, Q, K, V, R, U, VB, lse, DO, D, dr);
  simt_bwd_duv_kernel<<<s.H, kDh, 0, st>>>(s, dqu, dqv, du, dvb);
  *launches += 5;
  return cudaGetLastError();
}

}  // namespace

BwdWorkspace simt_bwd_workspace(const AttnShape &s) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)s.B * s.H * s.L;
  BwdWorkspace w;
  w.d_off = 0;
  w.dqu_off = up(rows * sizeof(float));
  w.dqv_off = w.dqu_off + up(rows * kDh * sizeof(float));
  w.total = w.dqv_off + up(rows * kDh * sizeof(float));
  return w;
}

cudaError_t launch_simt_fwd(const AttnShape &s, rxl_dtype dt, const void *q, const void *k,
                            const void *v, const void *r, const void *u, const void *vb,
                            void *o, float *lse, cudaStream_t st, int *launches) {
  if (dt == RXL_DTYPE_F32) return fwd_impl<float>(s, q, k, v, r, u, vb, o, lse, st, launches);
  return fwd_impl<__nv_bfloat16>(s, q, k, v, r, u, vb, o, lse, st, launches);
}

cudaError_t launch_simt_bwd(const AttnShape &s, rxl_dtype dt, const void *q, const void *k,
                            const void *v, const void *r, const void *u, const void *vb,
                            const void *o, const float *lse, const void *dout, void *dq,
                            void *dk, void *dv, float *dr, float *du, float *dvb, void *ws,
                            cudaStream_t st, int *launches) {
  if (dt == RXL_DTYPE_F32)
    return bwd_impl<float>(s, q, k, v, r, u, vb, o, lse, dout, dq, dk, dv, dr, du, dvb, ws, st,
                           launches);
  return bwd_impl<__nv_bfloat16>(s, q, k, v, r, u, vb, o, lse, dout, dq, dk, dv, dr, du, dvb, ws,
                                 st, launches);
}

}  // namespace rxl
