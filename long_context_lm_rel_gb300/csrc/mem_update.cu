// FIFO memory update: the last min(L, cap) source rows of every plane are
// copied into the ring at consecutive physical rows (mod cap).
//
// Transformer-XL page, eq. Tail_M and update_mems ("Batched Tensor
// Contract"): M_{t+1} = last M rows of [M_t; H_t]. Held as a ring, only the
// appended rows move; the Polish glossary page describes the same FIFO buffer
// on the GPU with the oldest entries overwritten.
//
// HBM-bound copy: every thread moves one 16-byte vector; consecutive threads
// move consecutive vectors of a row, so each warp reads and writes whole
// 128-byte lines. The grid is a grid-stride loop sized to the SM count.
#include "internal.cuh"
#include "sm103.cuh"

namespace rxl {

__global__ void __launch_bounds__(256) mem_update_kernel(
    int4 *__restrict__ data, long long plane_stride_v, int cap, int vpr,
    const int4 *__restrict__ src, long long src_plane_stride_v, int src_row0, int nrows,
    int dst_row0, long long total_v) {
  sm103::griddep_wait();
  sm103::griddep_launch_dependents();
  const long long per_plane = (long long)nrows * vpr;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total_v;
       e += (long long)gridDim.x * blockDim.x) {
    const long long p = e / per_plane;
    const int rem = (int)(e - p * per_plane);
    const int row = rem / vpr;
    const int c = rem - row * vpr;
    int dst_row = dst_row0 + row;
    if (dst_row >= cap) dst_row -= cap;  // dst_row0 < cap and row < cap
    const int4 val = __ldg(src + p * src_plane_stride_v + (long long)(src_row0 + row) * vpr + c);
    data[p * plane_stride_v + (long long)dst_row * vpr + c] = val;
  }
}

cudaError_t launch_mem_update(void *data, int planes, int cap, int D, long long plane_stride,
                              int elem_bytes, const void *src, long long src_plane_stride,
                              int src_row0, int nrows, int dst_row0, cudaStream_t st,
                              int *launches) {
  const int vpr = D * elem_bytes / 16;
  const long long total = (long long)planes * nrows * vpr;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap_blocks = (long long)sms * 8;  // 8 resident 256-thread blocks per SM
  if (blocks > cap_blocks) blocks = cap_blocks;
  const cudaError_t e = launch_ex(mem_update_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, (int4 *)data,
                                  (long long)(plane_stride * elem_bytes / 16), cap, vpr, (const int4 *)src,
                                  (long long)(src_plane_stride * elem_bytes / 16), src_row0, nrows, dst_row0,
                                  total);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rxl
