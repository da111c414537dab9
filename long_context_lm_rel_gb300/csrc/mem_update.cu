// FIFO memory update: the last min(L, cap) source rows of every plane are
// copied into the ring at consecutive physical rows (mod cap).
//
// Transformer-XL page, eq. Tail_M and update_mems ("Batched Tensor
// Contract"): M_{t+1} = last M rows of [M_t; H_t]. Held as a ring, only the
// appended rows move; the Polish glossary page describes the same FIFO buffer
// on the GPU with the oldest entries overwritten.
//
// HBM-bound copy of 16-byte vectors. Per plane the copied source rows are one
// contiguous block and so are their destination rows, except for one wrap of
// the ring: with the plane's vectors numbered f = 0 .. n-1, the destination
// is dst0 + f, minus cap_v once f reaches the wrap point. No division per
// element and 64-bit offsets throughout. Blocks take (ring, plane) pairs
// along y and split a plane's vectors along x; each thread keeps four
// coalesced 16-byte loads in flight before it stores them. Several rings
// of one geometry (the K and V rings of a layer) go in one launch.
#include "internal.cuh"
#include "sm103.cuh"

namespace rxl {

struct RingCopy {
  int4 *data[kMaxRingsPerUpdate];
  const int4 *src[kMaxRingsPerUpdate];
  long long plane_v[kMaxRingsPerUpdate];      // vectors between planes of the ring
  long long src_plane_v[kMaxRingsPerUpdate];  // vectors between planes of the source
  int nrings, planes;
  long long n_v;       // vectors copied per plane: nrows * vectors per row
  long long src0_v;    // first copied source vector of a plane (src_row0 * vpr)
  long long dst0_v;    // its destination (dst_row0 * vpr)
  long long wrap_v;    // f >= wrap_v wraps to the start of the ring: (cap - dst_row0) * vpr
  long long cap_v;     // cap * vpr
};

constexpr int kVecPerThread = 4;
constexpr int kThreadsPerBlock = 256;

__global__ void __launch_bounds__(kThreadsPerBlock) mem_update_kernel(const __grid_constant__ RingCopy rc) {
  sm103::griddep_wait();
  sm103::griddep_launch_dependents();
  const long long chunk = (long long)kThreadsPerBlock * kVecPerThread;
  for (int pp = blockIdx.y; pp < rc.nrings * rc.planes; pp += gridDim.y) {
    const int ring = pp / rc.planes, p = pp - ring * rc.planes;
    const int4 *src = rc.src[ring] + (long long)p * rc.src_plane_v[ring] + rc.src0_v;
    int4 *dst = rc.data[ring] + (long long)p * rc.plane_v[ring];
    for (long long base = blockIdx.x * chunk; base < rc.n_v; base += (long long)gridDim.x * chunk) {
      int4 val[kVecPerThread];
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const long long f = base + threadIdx.x + (long long)k * kThreadsPerBlock;
        if (f < rc.n_v) val[k] = __ldcs(src + f);  // streamed: read once
      }
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const long long f = base + threadIdx.x + (long long)k * kThreadsPerBlock;
        if (f < rc.n_v) dst[rc.dst0_v + f - (f >= rc.wrap_v ? rc.cap_v : 0)] = val[k];
      }
    }
  }
}

cudaError_t launch_mem_update(const MemUpdateArgs &a, cudaStream_t st, int *launches) {
  const long long vpr = (long long)a.D * a.elem_bytes / 16;
  const long long n_v = (long long)a.nrows * vpr;
  if (n_v == 0 || a.nrings == 0) return cudaSuccess;
  RingCopy rc;
  for (int r = 0; r < a.nrings; ++r) {
    rc.data[r] = (int4 *)a.data[r];
    rc.src[r] = (const int4 *)a.src[r];
    rc.plane_v[r] = a.plane_stride[r] * a.elem_bytes / 16;
    rc.src_plane_v[r] = a.src_plane_stride[r] * a.elem_bytes / 16;
  }
  rc.nrings = a.nrings;
  rc.planes = a.planes;
  rc.n_v = n_v;
  rc.src0_v = (long long)a.src_row0 * vpr;
  rc.dst0_v = (long long)a.dst_row0 * vpr;
  rc.wrap_v = (long long)(a.cap - a.dst_row0) * vpr;
  rc.cap_v = (long long)a.cap * vpr;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long pairs = (long long)a.nrings * a.planes;
  const unsigned gy = (unsigned)(pairs < 65535 ? pairs : 65535);
  // enough blocks along x to cover a plane, within ~8 resident blocks per SM overall
  const long long chunk = (long long)kThreadsPerBlock * kVecPerThread;
  long long gx = (n_v + chunk - 1) / chunk;
  long long gx_cap = ((long long)sms * 8 + gy - 1) / gy;
  if (gx_cap < 1) gx_cap = 1;
  if (gx > gx_cap) gx = gx_cap;
  const cudaError_t e = launch_ex(mem_update_kernel, dim3((unsigned)gx, gy), dim3(kThreadsPerBlock), 0, st, 1, rc);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rxl
