// Internal declarations shared by the translation units of librxl.
// Not part of the public ABI (include/rxl.h is).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/rxl.h"

namespace rxl {

// Launches k (optionally as clusters of `cluster` CTAs) with programmatic
// dependent launch allowed: its CTAs may start their setup while the previous
// kernel on the stream finishes; the kernels wait for it (griddep_wait)
// before their first global-memory access.
// Testing hook: a non-zero value is returned, once, by the next launch_ex
// instead of launching (rxl_test_fail_next_launch).
extern std::atomic<int> g_fail_next_launch;

template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             unsigned cluster, Args... args) {
  if (const int injected = g_fail_next_launch.exchange(0)) return (cudaError_t)injected;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  unsigned n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

// Opt-in device timing (rxl_kernel_timing): timing_begin records a start event
// on st and returns a slot (-1 when timing is off or full); timing_end records
// the matching stop event.
// 0: forward kernel, 1: backward main kernel, 2: backward prep launches (zero and
// operand prep), 3: backward finish kernel
constexpr int kTimedKernels = 4;
bool timing_enabled();
int timing_begin(int kernel, cudaStream_t st);
void timing_end(int kernel, int slot, cudaStream_t st);

// Validated shape of one attention call, as the kernels see it.
struct AttnShape {
  int B, H, L;
  int cap;        // M: memory rows reserved in K/V
  int m;          // valid memory rows
  int head;       // physical row of the oldest memory row
  float scale;
  int kv_rows;    // cap + L
  // per-row document reset (nullable device pointer, B entries): batch row b
  // sees only its newest mvis[b] memory rows (clamped into [0, m])
  const int *mvis = nullptr;
};

// Workspace layout of the backward (offsets in bytes from the base).
struct BwdWorkspace {
  size_t d_off, dqu_off, dqv_off, total;
};
BwdWorkspace simt_bwd_workspace(const AttnShape &s);

// Launchers return cudaSuccess or the launch error; `launches` is
// incremented by the number of kernels put on the stream.
// One FIFO update of up to kMaxRingsPerUpdate rings of the same geometry
// (planes, cap, D, element size, head, len): rows src_row0 .. src_row0+nrows-1
// of every source plane go to ring rows dst_row0 .. (mod cap).
constexpr int kMaxRingsPerUpdate = 8;
struct MemUpdateArgs {
  void *data[kMaxRingsPerUpdate];
  const void *src[kMaxRingsPerUpdate];
  long long plane_stride[kMaxRingsPerUpdate];      // elements
  long long src_plane_stride[kMaxRingsPerUpdate];  // elements
  int nrings, planes, cap, D, elem_bytes;
  int src_row0, nrows, dst_row0;
};
cudaError_t launch_mem_update(const MemUpdateArgs &a, cudaStream_t st, int *launches);

cudaError_t launch_simt_fwd(const AttnShape &s, rxl_dtype dt, const void *q, const void *k,
                            const void *v, const void *r, const void *u, const void *vb,
                            void *o, float *lse, cudaStream_t st, int *launches);

cudaError_t launch_simt_bwd(const AttnShape &s, rxl_dtype dt, const void *q, const void *k,
                            const void *v, const void *r, const void *u, const void *vb,
                            const void *o, const float *lse, const void *dout, void *dq,
                            void *dk, void *dv, float *dr, float *du, float *dvb, void *ws,
                            cudaStream_t st, int *launches);

// sm_103a tensor-core forward (bf16).
// o_lo (nullable) receives O - bf16(O) in bf16.
cudaError_t launch_tc_fwd(const AttnShape &s, const void *q, const void *k, const void *v,
                          const void *r, const void *u, const void *vb, void *o, void *o_lo,
                          float *lse, cudaStream_t st, int *launches);
// Reads and clears the forward kernel's wait-timeout flag (synchronous).
cudaError_t tc_fwd_read_error(int *flag);
// Testing hook of the forward kernel: its bounded waits give up after
// wait_cycles (<= 0: the default), and with withhold != 0 its softmax warps
// withhold the arrival that tells the producer a new item's query tiles are
// ready, so that the producer's wait on it runs out.
cudaError_t tc_fwd_test_hooks(long long wait_cycles, int withhold);

// Forward kernel in backward-preparation mode: D = dO.O (fp32 O) and the
// (Q+u) rows in bf16 and (Q+v) rows in fp16.
cudaError_t launch_tc_bwd_prep(const AttnShape &s, const void *q, const void *k, const void *v,
                               const void *r, const void *u, const void *vb, const void *dout,
                               float *delta, void *qu_out, void *qv_out, cudaStream_t st,
                               int *launches);

// sm_103a tensor-core backward (bf16).
BwdWorkspace tc_bwd_workspace(const AttnShape &s);
// With o_lo (nullable), D comes from dO.(o + o_lo) in a streaming pass;
// without it the forward is recomputed to obtain D from the fp32 O.
cudaError_t launch_tc_bwd(const AttnShape &s, const void *q, const void *k, const void *v,
                          const void *r, const void *u, const void *vb, const void *o,
                          const void *o_lo, const float *lse,
                          const void *dout, void *dq, void *dk, void *dv, float *dr, float *du,
                          float *dvb, void *ws, cudaStream_t st, int *launches);
cudaError_t tc_bwd_read_error(int *flag);
// Read and clear the fp16 range words (an R or q + v element beyond 65504 in
// magnitude reached the backward's fp16 position products and was clamped).
cudaError_t tc_bwd_read_range(int *flag);
cudaError_t tc_fwd_read_range(int *flag);

// Projection front-end (bf16): q, k, v from the hidden-state memory ring and
// the current hidden states.
cudaError_t launch_tc_proj(const AttnShape &s, int d, const void *h_mem, const void *h_cur,
                           const void *wq, const void *wk, const void *wv, void *q, void *k, void *v,
                           cudaStream_t st, int *launches);

// Dense layer out = act(A . W + bias) + residual over B groups of R rows
// (bf16); A is [B, R, K] or, with a_heads, the attention output [B, K/64, R, 64].
// partials (nullable): fp32 scratch of partial_floats floats that lets the
// K range be split over several CTAs per output block when there are few
// blocks (each split needs B * R * N floats).
// ln_out (nullable): the result then goes on through the LayerNorm
// (ln_gamma, ln_beta, ln_eps) into ln_out; out is written only when K is not
// split (the split's finalize pass applies the LayerNorm itself).
cudaError_t launch_tc_gemm(int B, int R, int K, int N, const void *a, bool a_heads, const void *w,
                           const void *bias, const void *residual, bool relu, void *out,
                           float *partials, size_t partial_floats, const void *ln_gamma, const void *ln_beta,
                           float ln_eps, void *ln_out, cudaStream_t st, int *launches);

cudaError_t tc_proj_read_error(int *flag);
cudaError_t tc_gemm_read_error(int *flag);

}  // namespace rxl
