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
#include <cuda.h>

#include <mutex>

#include "internal.cuh"

namespace {

// 16 MiB. The backward's scratch is, with rows = B*H*L query rows and
// kv = M+L key rows per head (bf16; the f32 path needs only the first term):
//   516*rows + 384*H*kv + 32,768*H bytes (+ at most 2 KB of alignment),
// i.e. per query row D (4 B), (Q+u) and (Q+v) (2 x 128 B) and the fp32 dQ
// accumulator (256 B); per head and key row the fp16 copy of R (128 B) and
// the fp32 dR accumulator (256 B, with 128 extra rows per head). Long memory
// reaches the limit well before many query rows do: B4 H16 L128 with 1600
// memory rows already needs about 15.4 MiB.
constexpr size_t kScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
struct Cached {
  unsigned long long ctx_id;  // the context the address belongs to (0: none yet)
  void *addr;
};
Cached g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
  void *f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return (Fn)f;
  return nullptr;
}

// Unique id of the calling thread's current context, 0 if unknown.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_bwd_scratch on the current device. The array's name is
// only a host-side stand-in, so the address is looked up with the device
// current, at the first call on that device, and cached. The cache is keyed
// by the context's unique id as well: after a device reset the module is
// loaded again in a new context, the array may move, and the next call looks
// the address up again instead of using a stale one. (When the id cannot be
// read, e.g. before the runtime has made a context current, the address is
// looked up on every call.)
cudaError_t scratch_on_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  Cached &c = g_scratch[dev];
  if (!c.addr || id == 0 || c.ctx_id != id) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    c.addr = p;
    c.ctx_id = current_context_id();  // the lookup made the device's context current
  }
  *out = c.addr;
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
