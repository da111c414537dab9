// rxl_attn_bwd_noalloc: the backward for callers that cannot allocate.
//
// Some callers hold nothing but their input and output buffers when they run
// the backward: plugin-style interfaces that hand the library pre-allocated
// tensors and no allocator, or latency-critical loops where a cudaMalloc (which
// may synchronise the device and is slow) is not acceptable. This entry point
// runs the same kernels as rxl_attn_bwd, but its scratch is a fixed array
// compiled into the library instead of a caller workspace.
//
// Costs and limits:
//  * every GPU that loads the library holds kScratchBytes for this array
//    until the process exits;
//  * shapes whose backward needs more scratch than that are rejected;
//  * all calls share the one array per device, so calls that overlap on the
//    GPU (different streams, or different host threads) race on it.
#include <mutex>

#include "internal.cuh"

namespace {

// 16 MiB: enough for B*H*L up to about 32,000 query rows (the backward needs
// about 520 bytes of scratch per query row, plus 128 bytes per head and K/V
// row for an fp16 copy of R).
constexpr size_t kScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device. The name is only a
// host-side stand-in for the array, so the address is looked up once per
// device, with that device current, and cached.
cudaError_t scratch_on_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t rxl_attn_bwd_noalloc_max_scratch_bytes(void) { return kScratchBytes; }

rxl_status rxl_attn_bwd_noalloc(const rxl_attn_desc *desc, const void *q, const void *k,
                                const void *v, const void *r, const void *u, const void *vbias,
                                const void *o, const float *lse, const void *dout, void *dq,
                                void *dk, void *dv, float *dr, float *du, float *dvbias,
                                rxl_stream_t stream) {
  const size_t need = rxl_attn_bwd_workspace_bytes(desc);
  if (need > kScratchBytes) return RXL_ERR_WORKSPACE_TOO_SMALL;  // shape too large for the array
  void *scratch = nullptr;
  // No part of the scratch has to start at zero: every byte the backward
  // reads from its workspace is written earlier in the same call.
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) return RXL_ERR_CUDA;
  return rxl_attn_bwd(desc, q, k, v, r, u, vbias, o, lse, dout, dq, dk, dv, dr, du, dvbias, scratch,
                      kScratchBytes, stream);
}

}  // extern "C"
