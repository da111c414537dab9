// C ABI of librxl: argument validation, dispatch and status reporting.
// See include/rxl.h for the contract of every entry point.
#include <math.h>
#include <stdint.h>

#include <initializer_list>

#include "internal.cuh"

namespace rxl {
std::atomic<int> g_fail_next_launch{0};
}  // namespace rxl

namespace {

thread_local int g_last_cuda_error = 0;
thread_local int g_last_launches = 0;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

rxl_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RXL_OK;
  g_last_cuda_error = (int)e;
  return RXL_ERR_CUDA;
}

// Checks the descriptor; on success fills the kernel-side shape.
rxl_status check_desc(const rxl_attn_desc *d, rxl::AttnShape *s) {
  if (!d) return RXL_ERR_INVALID_ARGUMENT;
  if (d->B < 1 || d->H < 1 || d->L < 1 || d->dh < 1) return RXL_ERR_INVALID_ARGUMENT;
  if (d->mem_cap < 0 || d->mem_len < 0 || d->mem_len > d->mem_cap) return RXL_ERR_INVALID_ARGUMENT;
  if (d->mem_cap == 0 ? d->mem_head != 0 : (d->mem_head < 0 || d->mem_head >= d->mem_cap))
    return RXL_ERR_INVALID_ARGUMENT;
  if (!isfinite(d->scale)) return RXL_ERR_INVALID_ARGUMENT;
  // int32 row indexing inside the kernels: keep every per-(b,h) extent and
  // the grid sizes far from overflow
  const long long rows = (long long)d->mem_cap + d->L;
  if (rows > (1LL << 24) || (long long)d->B * d->H > (1LL << 24) ||
      (long long)d->B * d->H * rows > (1LL << 34))
    return RXL_ERR_INVALID_ARGUMENT;
  if (d->dtype != RXL_DTYPE_F32 && d->dtype != RXL_DTYPE_BF16) return RXL_ERR_UNSUPPORTED;
  if (d->dh != 64) return RXL_ERR_UNSUPPORTED;
  s->B = d->B; s->H = d->H; s->L = d->L;
  s->cap = d->mem_cap; s->m = d->mem_len; s->head = d->mem_head;
  s->scale = d->scale;
  s->kv_rows = d->mem_cap + d->L;
  return RXL_OK;
}

rxl_status check_ptrs(std::initializer_list<const void *> ps) {
  for (const void *p : ps)
    if (!p) return RXL_ERR_INVALID_ARGUMENT;
  for (const void *p : ps)
    if (!aligned16(p)) return RXL_ERR_MISALIGNED;
  return RXL_OK;
}

}  // namespace

extern "C" {

const char *rxl_status_string(rxl_status s) {
  switch (s) {
    case RXL_OK: return "RXL_OK";
    case RXL_ERR_INVALID_ARGUMENT: return "RXL_ERR_INVALID_ARGUMENT";
    case RXL_ERR_UNSUPPORTED: return "RXL_ERR_UNSUPPORTED";
    case RXL_ERR_MISALIGNED: return "RXL_ERR_MISALIGNED";
    case RXL_ERR_WORKSPACE_TOO_SMALL: return "RXL_ERR_WORKSPACE_TOO_SMALL";
    case RXL_ERR_CUDA: return "RXL_ERR_CUDA";
  }
  return "RXL_ERR_UNKNOWN";
}

int rxl_last_cuda_error(void) { return g_last_cuda_error; }

int rxl_last_launch_count(void) { return g_last_launches; }

void rxl_test_fail_next_launch(int cuda_error) { rxl::g_fail_next_launch.store(cuda_error); }

int rxl_test_forward_wait_timeout(long long wait_cycles, int withhold) {
  return (int)rxl::tc_fwd_test_hooks(wait_cycles, withhold);
}

int rxl_device_error_flags(void) {
  int fwd = 0, bwd = 0, proj = 0, gemm = 0, range_b = 0, range_f = 0;
  if (rxl::tc_fwd_read_error(&fwd) != cudaSuccess || rxl::tc_bwd_read_error(&bwd) != cudaSuccess ||
      rxl::tc_proj_read_error(&proj) != cudaSuccess || rxl::tc_gemm_read_error(&gemm) != cudaSuccess ||
      rxl::tc_bwd_read_range(&range_b) != cudaSuccess || rxl::tc_fwd_read_range(&range_f) != cudaSuccess)
    return -1;
  return (fwd ? 1 : 0) | (bwd ? 2 : 0) | (proj ? 4 : 0) | (gemm ? 8 : 0) | ((range_b || range_f) ? 16 : 0);
}

namespace {
struct LayerWs {
  size_t q, k, v, o, lse, x1, x1n, z, x2, part, part_floats, total;
};
size_t up256_(size_t x) { return (x + 255) & ~(size_t)255; }
LayerWs layer_ws(const rxl::AttnShape &s, int d, int dff) {
  const size_t rows = (size_t)s.B * s.L, bh = (size_t)s.B * s.H;
  LayerWs w;
  w.q = 0;
  w.k = w.q + up256_(bh * s.L * 64 * 2);
  w.v = w.k + up256_(bh * s.kv_rows * 64 * 2);
  w.o = w.v + up256_(bh * s.kv_rows * 64 * 2);
  w.lse = w.o + up256_(bh * s.L * 64 * 2);
  w.x1 = w.lse + up256_(bh * s.L * 4);
  w.x1n = w.x1 + up256_(rows * d * 2);
  w.z = w.x1n + up256_(rows * d * 2);
  w.x2 = w.z + up256_(rows * dff * 2);
  // fp32 partial sums of the dense layers when their K range is split
  // (short segments): up to 8 splits of a [rows][d] output
  w.part = w.x2 + up256_(rows * d * 2);
  w.part_floats = rows * 8 * (size_t)d;
  w.total = w.part + up256_(w.part_floats * 4);
  return w;
}
rxl_status check_layer(const rxl_attn_desc *desc, int d, int dff, rxl::AttnShape *s) {
  rxl_status st = check_desc(desc, s);
  if (st != RXL_OK) return st;
  if (desc->dtype != RXL_DTYPE_BF16) return RXL_ERR_UNSUPPORTED;
  if (d < 256 || d % 256 != 0 || d > (1 << 16) || dff < 64 || dff % 64 != 0 || dff > (1 << 17))
    return RXL_ERR_UNSUPPORTED;
  return RXL_OK;
}
}  // namespace

size_t rxl_layer_fwd_workspace_bytes(const rxl_attn_desc *desc, int d_model, int d_ff) {
  rxl::AttnShape s;
  if (check_layer(desc, d_model, d_ff, &s) != RXL_OK) return 0;
  return layer_ws(s, d_model, d_ff).total;
}

rxl_status rxl_layer_fwd(const rxl_attn_desc *desc, int d_model, int d_ff, const rxl_layer_weights *w,
                         const void *h_mem, const void *h_in, void *h_out, void *workspace,
                         size_t workspace_bytes, rxl_stream_t stream) {
  rxl::AttnShape s;
  rxl_status st = check_layer(desc, d_model, d_ff, &s);
  if (st != RXL_OK) return st;
  if (!w) return RXL_ERR_INVALID_ARGUMENT;
  if ((st = check_ptrs({w->w_q, w->w_k, w->w_v, w->w_o, w->r, w->u, w->vbias, w->ln1_gamma,
                        w->ln1_beta, w->w_1, w->b_1, w->w_2, w->b_2, w->ln2_gamma, w->ln2_beta,
                        h_in, h_out, workspace})) != RXL_OK)
    return st;
  if (s.cap > 0 && (st = check_ptrs({h_mem})) != RXL_OK) return st;
  const LayerWs lw = layer_ws(s, d_model, d_ff);
  if (workspace_bytes < lw.total) return RXL_ERR_WORKSPACE_TOO_SMALL;
  char *ws = (char *)workspace;
  void *q = ws + lw.q, *k = ws + lw.k, *v = ws + lw.v, *o = ws + lw.o;
  float *lse = (float *)(ws + lw.lse);
  void *x1 = ws + lw.x1, *x1n = ws + lw.x1n, *z = ws + lw.z, *x2 = ws + lw.x2;
  float *part = (float *)(ws + lw.part);
  cudaStream_t cs = (cudaStream_t)stream;
  int launches = 0;
  cudaError_t e = rxl::launch_tc_proj(s, d_model, h_mem, h_in, w->w_q, w->w_k, w->w_v, q, k, v, cs,
                                      &launches);
  if (e == cudaSuccess)
    e = rxl::launch_tc_fwd(s, q, k, v, w->r, w->u, w->vbias, o, nullptr, lse, cs, &launches);
  if (e == cudaSuccess)  // x1n = LayerNorm(h + attention . W_O) (heads merged by the A operand's layout)
    e = rxl::launch_tc_gemm(s.B, s.L, s.H * 64, d_model, o, true, w->w_o, nullptr, h_in, false, x1,
                            part, lw.part_floats, w->ln1_gamma, w->ln1_beta, 1e-5f, x1n, cs, &launches);
  if (e == cudaSuccess)  // z = ReLU(x1n . W_1 + b_1)
    e = rxl::launch_tc_gemm(s.B, s.L, d_model, d_ff, x1n, false, w->w_1, w->b_1, nullptr, true, z,
                            part, lw.part_floats, nullptr, nullptr, 0.f, nullptr, cs, &launches);
  if (e == cudaSuccess)  // h_out = LayerNorm(x1n + z . W_2 + b_2)
    e = rxl::launch_tc_gemm(s.B, s.L, d_ff, d_model, z, false, w->w_2, w->b_2, x1n, false, x2,
                            part, lw.part_floats, w->ln2_gamma, w->ln2_beta, 1e-5f, h_out, cs, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

rxl_status rxl_qkv_proj(const rxl_attn_desc *desc, int d_model, const void *h_mem,
                        const void *h_cur, const void *w_q, const void *w_k, const void *w_v,
                        void *q, void *k, void *v, rxl_stream_t stream) {
  rxl::AttnShape s;
  rxl_status st = check_desc(desc, &s);
  if (st != RXL_OK) return st;
  if (desc->dtype != RXL_DTYPE_BF16) return RXL_ERR_UNSUPPORTED;
  if (d_model < 64 || d_model % 64 != 0 || d_model > (1 << 16)) return RXL_ERR_UNSUPPORTED;
  if ((st = check_ptrs({h_cur, w_q, w_k, w_v, q, k, v})) != RXL_OK) return st;
  if (s.cap > 0 && (st = check_ptrs({h_mem})) != RXL_OK) return st;
  int launches = 0;
  const cudaError_t e = rxl::launch_tc_proj(s, d_model, h_mem, h_cur, w_q, w_k, w_v, q, k, v,
                                            (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

}  // extern "C"

namespace {

// The forward with an optional per-row document reset (mvis: device int32 [B]).
rxl_status attn_fwd(const rxl_attn_desc *desc, const int32_t *mvis, const void *q, const void *k,
                    const void *v, const void *r, const void *u, const void *vbias, void *o,
                    void *o_lo, float *lse, rxl_stream_t stream) {
  rxl::AttnShape s;
  rxl_status st = check_desc(desc, &s);
  if (st != RXL_OK) return st;
  s.mvis = mvis;
  if ((st = check_ptrs({q, k, v, r, u, vbias, o, lse})) != RXL_OK) return st;
  if (o_lo && desc->dtype != RXL_DTYPE_BF16) return RXL_ERR_INVALID_ARGUMENT;
  if (o_lo && !aligned16(o_lo)) return RXL_ERR_MISALIGNED;
  int launches = 0;
  const cudaError_t e =
      desc->dtype == RXL_DTYPE_BF16
          ? rxl::launch_tc_fwd(s, q, k, v, r, u, vbias, o, o_lo, lse, (cudaStream_t)stream, &launches)
          : rxl::launch_simt_fwd(s, desc->dtype, q, k, v, r, u, vbias, o, lse,
                                 (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

}  // namespace

extern "C" {

rxl_status rxl_attn_fwd_ex(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                           const void *r, const void *u, const void *vbias, void *o, void *o_lo,
                           float *lse, rxl_stream_t stream) {
  return attn_fwd(desc, nullptr, q, k, v, r, u, vbias, o, o_lo, lse, stream);
}

rxl_status rxl_attn_fwd_reset(const rxl_attn_desc *desc, const int32_t *mem_visible, const void *q,
                              const void *k, const void *v, const void *r, const void *u,
                              const void *vbias, void *o, void *o_lo, float *lse,
                              rxl_stream_t stream) {
  if (!mem_visible) return RXL_ERR_INVALID_ARGUMENT;
  if ((uintptr_t)mem_visible % 4) return RXL_ERR_MISALIGNED;
  return attn_fwd(desc, mem_visible, q, k, v, r, u, vbias, o, o_lo, lse, stream);
}

rxl_status rxl_attn_fwd(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                        const void *r, const void *u, const void *vbias, void *o, float *lse,
                        rxl_stream_t stream) {
  return rxl_attn_fwd_ex(desc, q, k, v, r, u, vbias, o, nullptr, lse, stream);
}

size_t rxl_attn_bwd_workspace_bytes(const rxl_attn_desc *desc) {
  rxl::AttnShape s;
  if (check_desc(desc, &s) != RXL_OK) return 0;
  return desc->dtype == RXL_DTYPE_BF16 ? rxl::tc_bwd_workspace(s).total
                                       : rxl::simt_bwd_workspace(s).total;
}

}  // extern "C"

namespace {

// The backward with an optional per-row document reset (mvis: device int32 [B]).
rxl_status attn_bwd(const rxl_attn_desc *desc, const int32_t *mvis, const void *q, const void *k,
                    const void *v, const void *r, const void *u, const void *vbias, const void *o,
                    const void *o_lo, const float *lse, const void *dout, void *dq, void *dk,
                    void *dv, float *dr, float *du, float *dvbias, void *workspace,
                    size_t workspace_bytes, rxl_stream_t stream) {
  rxl::AttnShape s;
  rxl_status st = check_desc(desc, &s);
  if (st != RXL_OK) return st;
  s.mvis = mvis;
  if (o_lo && desc->dtype != RXL_DTYPE_BF16) return RXL_ERR_INVALID_ARGUMENT;
  if (o_lo && !aligned16(o_lo)) return RXL_ERR_MISALIGNED;
  if ((st = check_ptrs({q, k, v, r, u, vbias, o, lse, dout, dq, dk, dv, dr, du, dvbias,
                        workspace})) != RXL_OK)
    return st;
  const bool tc = desc->dtype == RXL_DTYPE_BF16;
  if (workspace_bytes < (tc ? rxl::tc_bwd_workspace(s).total : rxl::simt_bwd_workspace(s).total))
    return RXL_ERR_WORKSPACE_TOO_SMALL;
  int launches = 0;
  const cudaError_t e =
      tc ? rxl::launch_tc_bwd(s, q, k, v, r, u, vbias, o, o_lo, lse, dout, dq, dk, dv, dr, du,
                              dvbias, workspace, (cudaStream_t)stream, &launches)
         : rxl::launch_simt_bwd(s, desc->dtype, q, k, v, r, u, vbias, o, lse, dout, dq, dk, dv, dr,
                                du, dvbias, workspace, (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

}  // namespace

extern "C" {

rxl_status rxl_attn_bwd_ex(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                           const void *r, const void *u, const void *vbias, const void *o,
                           const void *o_lo, const float *lse, const void *dout, void *dq,
                           void *dk, void *dv, float *dr, float *du, float *dvbias,
                           void *workspace, size_t workspace_bytes, rxl_stream_t stream) {
  return attn_bwd(desc, nullptr, q, k, v, r, u, vbias, o, o_lo, lse, dout, dq, dk, dv, dr, du,
                  dvbias, workspace, workspace_bytes, stream);
}

rxl_status rxl_attn_bwd_reset(const rxl_attn_desc *desc, const int32_t *mem_visible, const void *q,
                              const void *k, const void *v, const void *r, const void *u,
                              const void *vbias, const void *o, const void *o_lo, const float *lse,
                              const void *dout, void *dq, void *dk, void *dv, float *dr, float *du,
                              float *dvbias, void *workspace, size_t workspace_bytes,
                              rxl_stream_t stream) {
  if (!mem_visible) return RXL_ERR_INVALID_ARGUMENT;
  if ((uintptr_t)mem_visible % 4) return RXL_ERR_MISALIGNED;
  return attn_bwd(desc, mem_visible, q, k, v, r, u, vbias, o, o_lo, lse, dout, dq, dk, dv, dr, du,
                  dvbias, workspace, workspace_bytes, stream);
}

rxl_status rxl_attn_bwd(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                        const void *r, const void *u, const void *vbias, const void *o,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv,
                        float *dr, float *du, float *dvbias, void *workspace,
                        size_t workspace_bytes, rxl_stream_t stream) {
  return rxl_attn_bwd_ex(desc, q, k, v, r, u, vbias, o, nullptr, lse, dout, dq, dk, dv, dr, du,
                         dvbias, workspace, workspace_bytes, stream);
}

rxl_status rxl_mem_update_rings(rxl_ring *const *rings, const void *const *srcs,
                                const long long *src_plane_strides, int n, int L, rxl_stream_t stream) {
  if (!rings || !srcs || !src_plane_strides || L < 0) return RXL_ERR_INVALID_ARGUMENT;
  if (n < 1 || n > rxl::kMaxRingsPerUpdate) return RXL_ERR_INVALID_ARGUMENT;
  for (int r = 0; r < n; ++r)
    if (!rings[r]) return RXL_ERR_INVALID_ARGUMENT;
  const rxl_ring &g = *rings[0];  // the shared geometry
  if (g.dtype != RXL_DTYPE_F32 && g.dtype != RXL_DTYPE_BF16) return RXL_ERR_UNSUPPORTED;
  if (g.planes < 1 || g.cap < 0 || g.D < 1) return RXL_ERR_INVALID_ARGUMENT;
  if (g.len < 0 || g.len > g.cap) return RXL_ERR_INVALID_ARGUMENT;
  if (g.cap == 0 ? g.head != 0 : (g.head < 0 || g.head >= g.cap)) return RXL_ERR_INVALID_ARGUMENT;
  const int es = g.dtype == RXL_DTYPE_F32 ? 4 : 2;
  for (int r = 0; r < n; ++r) {
    const rxl_ring &x = *rings[r];
    if (x.planes != g.planes || x.cap != g.cap || x.D != g.D || x.dtype != g.dtype || x.head != g.head ||
        x.len != g.len)
      return RXL_ERR_INVALID_ARGUMENT;
    for (int t = 0; t < r; ++t)
      if (rings[t] == rings[r]) return RXL_ERR_INVALID_ARGUMENT;  // each ring advances once
    if (x.plane_stride < (long long)x.cap * x.D) return RXL_ERR_INVALID_ARGUMENT;
    if (src_plane_strides[r] < (long long)L * x.D) return RXL_ERR_INVALID_ARGUMENT;
  }
  g_last_launches = 0;
  if (g.cap == 0 || L == 0) return RXL_OK;  // nothing kept / nothing appended
  for (int r = 0; r < n; ++r) {
    const rxl_ring &x = *rings[r];
    if (!x.data || !srcs[r]) return RXL_ERR_INVALID_ARGUMENT;
    if (!aligned16(x.data) || !aligned16(srcs[r]) || ((long long)x.D * es) % 16 != 0 ||
        (x.plane_stride * es) % 16 != 0 || (src_plane_strides[r] * es) % 16 != 0)
      return RXL_ERR_MISALIGNED;
  }
  const int cap = g.cap;
  const int nwrite = L < cap ? L : cap;          // only the last min(L, cap) rows survive
  rxl::MemUpdateArgs a;
  for (int r = 0; r < n; ++r) {
    a.data[r] = rings[r]->data;
    a.src[r] = srcs[r];
    a.plane_stride[r] = rings[r]->plane_stride;
    a.src_plane_stride[r] = src_plane_strides[r];
  }
  a.nrings = n;
  a.planes = g.planes;
  a.cap = cap;
  a.D = g.D;
  a.elem_bytes = es;
  a.src_row0 = L - nwrite;
  a.nrows = nwrite;
  a.dst_row0 = (int)(((long long)g.head + g.len + a.src_row0) % cap);
  int launches = 0;
  const cudaError_t e = rxl::launch_mem_update(a, (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  if (e != cudaSuccess) return cuda_status(e);
  const long long total = (long long)g.len + L;
  int head = g.head, len;
  if (total > cap) {
    head = (int)(((long long)g.head + total - cap) % cap);
    len = cap;
  } else {
    len = (int)total;
  }
  for (int r = 0; r < n; ++r) {
    rings[r]->head = head;
    rings[r]->len = len;
  }
  return RXL_OK;
}

rxl_status rxl_mem_update(rxl_ring *ring, const void *src, long long src_plane_stride, int L,
                          rxl_stream_t stream) {
  return rxl_mem_update_rings(&ring, &src, &src_plane_stride, 1, L, stream);
}

}  // extern "C"
