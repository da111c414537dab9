/*
 * rxl.h -- C ABI of librxl: Transformer-XL relative-position memory attention
 * on one GB300 (sm_103a).
 *
 * The operation (Transformer-XL page, zty624.github.io ch4_transformer/xl.html):
 *   - "Segment-Level Recurrence": the L queries of the current segment attend
 *     over [SG(memory); current]; keys/values have memory+current rows,
 *     queries only the current ones ("Batched Tensor Contract").
 *   - "Causal Mask With Memory", eq. allow: key positions -m..-1 (memory)
 *     are always visible, current key j is visible to query i iff j <= i.
 *   - "Relative Positional Encoding", four-term score:
 *        A_ij = (q_i + u).k_j + (q_i + v).r_{i-j}
 *     (the regrouped form is printed on the iopencloud page, section 2.2).
 *   - "Dimension Walkthrough": O = softmax((A + M_causal)/sqrt(d_h)) V; the
 *     scale applies to the whole of A; R has (M+L) rows, one per distance.
 *   - "Why Stop Gradient": gradients reach the K/V rows of the memory block
 *     (and R, u, v) but nothing flows back into the cached states.
 *   - eq. Tail_M and update_mems ("Batched Tensor Contract"): after each
 *     segment every layer keeps the last M states; the Polish glossary page
 *     (robocikowo.com) describes it as a FIFO buffer on the GPU whose oldest
 *     entries are overwritten.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller. The
 *     library allocates no device memory and keeps no device state between
 *     calls; a call only reads its inputs and writes its outputs/workspace.
 *   - Row-major, contiguous, d_h innermost. Element type = desc.dtype for
 *     q, k, v, r, u, vbias, o, dout, dq, dk, dv; float32 for lse, dr, du,
 *     dvbias and workspace.
 *   - Every pointer must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     and never synchronise. Arguments are checked before anything is
 *     launched; on any error nothing is launched and no output is touched.
 *     Device faults surface at the caller's next synchronisation.
 *   - Stream order is kept. The sm_103a kernels are launched with
 *     programmatic dependent launch: a kernel may start its on-chip setup
 *     while the previous kernel on the stream finishes, and touches no
 *     device memory before that kernel has completed.
 *   - Thread safety: calls may be made from several host threads; the only
 *     shared host state is a cache of TMA descriptors guarded by a mutex.
 */
#ifndef RXL_H
#define RXL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *rxl_stream_t;

typedef enum {
  RXL_OK = 0,
  RXL_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative or inconsistent size */
  RXL_ERR_UNSUPPORTED = 2,        /* a valid request the library does not implement (d_h != 64, dtype) */
  RXL_ERR_MISALIGNED = 3,         /* pointer or row stride not 16-byte aligned */
  RXL_ERR_WORKSPACE_TOO_SMALL = 4,
  RXL_ERR_CUDA = 5                /* a CUDA call or launch failed (see rxl_last_cuda_error) */
} rxl_status;

typedef enum { RXL_DTYPE_F32 = 0, RXL_DTYPE_BF16 = 1 } rxl_dtype;

/*
 * Shape of one attention call.
 *   B, H, L   batch, heads, current-segment rows (queries), all >= 1
 *   dh        head width; must be 64
 *   mem_cap   M: rows reserved for memory in K/V (>= 0)
 *   mem_len   m: valid memory rows, 0 <= m <= M (memory fills up over the
 *             first segments of a stream)
 *   mem_head  physical row of the OLDEST memory row, 0 <= head < M (0 if M==0)
 *   scale     multiplies the whole score A (1/sqrt(dh) in the paper)
 *
 * K and V have M+L rows per (b,h): rows [0, M) are the memory ring, and
 * logical memory row t (t = 0 oldest, t < m) lives at physical row
 * (mem_head + t) mod M; rows [M, M+L) are the current segment. Logical key
 * position of memory row t is t - m; of current row i it is i. R has M+L rows
 * per head; row d embeds the distance d; rows 0..m+L-1 are read.
 */
typedef struct {
  int B, H, L, dh;
  int mem_cap;
  int mem_len;
  int mem_head;
  float scale;
  rxl_dtype dtype;
} rxl_attn_desc;

/*
 * Forward (Transformer-XL page, "Relative Positional Encoding" and
 * "Dimension Walkthrough"):
 *   O_i   = sum_j softmax_j(scale * A_ij | allow(i,j)) V_j
 *   lse_i = log sum_j exp(scale * A_ij)   (natural log, allowed j only)
 * q [B,H,L,dh]; k, v [B,H,M+L,dh]; r [H,M+L,dh]; u, vbias [H,dh];
 * o [B,H,L,dh] (written); lse [B,H,L] float32 (written).
 * The L x (m+L) score matrix is never written to memory.
 */
rxl_status rxl_attn_fwd(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                        const void *r, const void *u, const void *vbias, void *o, float *lse,
                        rxl_stream_t stream);

/* Workspace bytes rxl_attn_bwd needs for this shape (0 on invalid desc). */
size_t rxl_attn_bwd_workspace_bytes(const rxl_attn_desc *desc);

/*
 * Backward of the forward above for upstream gradient dout [B,H,L,dh], given
 * the forward's o and lse. With dA_ij = scale * P_ij (dout_i.V_j - D_i) and
 * D_i = dout_i . o_i:
 *   dq_i  = sum_j dA_ij (k_j + r_{i-j})            [B,H,L,dh]
 *   dk_j  = sum_i dA_ij (q_i + u)                  [B,H,M+L,dh]
 *   dv_j  = sum_i P_ij dout_i                      [B,H,M+L,dh]
 *   dr_d  = sum_b sum_{i-j=d} dA_ij (q_i + v)      [H,M+L,dh] float32
 *   du    = sum_{b,i,j} dA_ij k_j                  [H,dh]     float32
 *   dvbias= sum_{b,i,j} dA_ij r_{i-j}              [H,dh]     float32
 * dk/dv use the physical row layout of k/v: memory rows get their K/V
 * gradient (stop-gradient stops only the path into the cached states, which
 * this call never writes); ring rows that hold no valid memory get zeros, as
 * do dr rows d >= m+L. k and v are read-only here.
 * workspace: device scratch of at least rxl_attn_bwd_workspace_bytes(desc)
 * bytes (16-byte aligned), owned by the caller; contents on entry ignored.
 * Range (bf16): the position products run on fp16 operands, so r and
 * q + vbias must stay within |x| <= 65504; larger elements are clamped and
 * reported through bit 4 of rxl_device_error_flags().
 * The fp32 sums over tiles (dq, dr, du, dvbias) are accumulated with
 * hardware reductions in an order that varies from run to run: results agree
 * to rounding, not bit for bit (dk, dv and the forward are reproducible).
 */
rxl_status rxl_attn_bwd(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                        const void *r, const void *u, const void *vbias, const void *o,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv,
                        float *dr, float *du, float *dvbias, void *workspace,
                        size_t workspace_bytes, rxl_stream_t stream);

/*
 * rxl_attn_bwd_noalloc -- rxl_attn_bwd without a caller-supplied workspace.
 * The paper has no counterpart: this is a deployment convenience.
 *
 * For callers that cannot allocate device memory when they run the backward:
 * plugin-style hosts that pass in only pre-allocated inputs and outputs and
 * provide no allocator, or latency-critical loops that must not pay for a
 * cudaMalloc. The scratch is a fixed array inside the library
 * (rxl_attn_bwd_noalloc_max_scratch_bytes() bytes, 16 MiB), held on every GPU
 * that loads the library until the process exits; this call itself allocates
 * nothing.
 *  - Same arguments, outputs and checks as rxl_attn_bwd minus the workspace.
 *  - Shapes whose backward needs more than the fixed scratch
 *    (rxl_attn_bwd_workspace_bytes(desc) > max) return
 *    RXL_ERR_WORKSPACE_TOO_SMALL without launching anything. In bf16 the
 *    need is about 516*B*H*L + 384*H*(M+L) + 32768*H bytes, so long memory
 *    reaches the limit first (B=4, H=16, L=128, M=1600 needs ~15.4 MiB);
 *    in f32 it is about 516*B*H*L bytes.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it per context; make that first call
 *    before any stream capture. After a device reset the next call looks the
 *    address up again.
 *  - All calls share the one array per device and it keeps the last call's
 *    contents (nothing in it has to start at zero). Calls that overlap on the
 *    GPU, e.g. on two streams, race on it: serialise them.
 */
rxl_status rxl_attn_bwd_noalloc(const rxl_attn_desc *desc, const void *q, const void *k,
                                const void *v, const void *r, const void *u, const void *vbias,
                                const void *o, const float *lse, const void *dout, void *dq,
                                void *dk, void *dv, float *dr, float *du, float *dvbias,
                                rxl_stream_t stream);

/* Size in bytes of the fixed scratch rxl_attn_bwd_noalloc uses. */
size_t rxl_attn_bwd_noalloc_max_scratch_bytes(void);

/*
 * Training pair: the same forward and backward, with one more output of the
 * forward that the backward consumes. o_lo [B,H,L,dh] (bf16 only; NULL for
 * f32, where O is exact) receives O - o, i.e. what rounding O to bf16
 * dropped, itself rounded to bf16. With it the backward takes
 * D_i = dout_i . (o_i + o_lo_i) from a streaming pass; with o_lo == NULL
 * (also what rxl_attn_fwd / rxl_attn_bwd do) the backward recomputes the
 * forward to obtain D from the unrounded O. D enters every dA_ij of the row,
 * so it must be more accurate than a bf16 O. Other arguments, outputs and
 * checks as in rxl_attn_fwd / rxl_attn_bwd.
 */
rxl_status rxl_attn_fwd_ex(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                           const void *r, const void *u, const void *vbias, void *o, void *o_lo,
                           float *lse, rxl_stream_t stream);

rxl_status rxl_attn_bwd_ex(const rxl_attn_desc *desc, const void *q, const void *k, const void *v,
                           const void *r, const void *u, const void *vbias, const void *o,
                           const void *o_lo, const float *lse, const void *dout, void *dq,
                           void *dk, void *dv, float *dr, float *du, float *dvbias,
                           void *workspace, size_t workspace_bytes, rxl_stream_t stream);

/*
 * Per-row document reset (Transformer-XL page, "Causal Mask With Memory",
 * the note after the mask picture, and "Batched Streams": a batch row that
 * has just entered a new document must not take the previous document as
 * its context, and the reset is per row, not per batch).
 *   mem_visible  DEVICE int32 [B] (4-byte aligned): batch row b attends only
 *                to its newest mem_visible[b] memory rows, i.e. logical
 *                memory rows m - mem_visible[b] .. m-1 (key positions
 *                -mem_visible[b] .. -1); the older ones are masked as if
 *                absent. A row that starts a new document passes 0 and its
 *                count grows again as that document's segments arrive.
 *                Values are clamped into [0, mem_len] on the device.
 * The ring itself is shared by all rows (rxl_mem_update is unchanged). In
 * the backward, the masked memory rows of a batch row get dk = dv = 0 and
 * contribute nothing to dr, du, dvbias. All other arguments, outputs and
 * checks as in rxl_attn_fwd_ex / rxl_attn_bwd_ex (o_lo may be NULL).
 */
rxl_status rxl_attn_fwd_reset(const rxl_attn_desc *desc, const int32_t *mem_visible, const void *q,
                              const void *k, const void *v, const void *r, const void *u,
                              const void *vbias, void *o, void *o_lo, float *lse,
                              rxl_stream_t stream);

rxl_status rxl_attn_bwd_reset(const rxl_attn_desc *desc, const int32_t *mem_visible, const void *q,
                              const void *k, const void *v, const void *r, const void *u,
                              const void *vbias, const void *o, const void *o_lo, const float *lse,
                              const void *dout, void *dq, void *dk, void *dv, float *dr, float *du,
                              float *dvbias, void *workspace, size_t workspace_bytes,
                              rxl_stream_t stream);

/*
 * Projection front-end (Transformer-XL page, "Segment-Level Recurrence":
 * Q = H W^Q, K = [SG(M); H] W^K, V = [SG(M); H] W^V; shapes as in "Batched
 * Tensor Contract"). The memory holds the layer's input hidden states, as the
 * pages define it, in a ring with the same mapping as K/V.
 *   d_model   hidden width d: a multiple of 64 (bf16 only)
 *   h_mem     [B, M, d] hidden-state ring: logical memory row t at physical
 *             row (mem_head + t) mod M; NULL allowed when M == 0
 *   h_cur     [B, L, d] the current segment's hidden states
 *   w_q, w_k, w_v  [d, H*dh] row-major; column h*dh + e feeds element e of head h
 *   q         [B, H, L, dh] written
 *   k, v      [B, H, M+L, dh] written in the attention's layout: ring slot p
 *             of h_mem projects to physical row p, current row i to row M+i.
 *             Rows of ring slots without valid memory are not written.
 * The ring of hidden states is advanced with rxl_mem_update (D = d_model).
 * Errors: RXL_ERR_UNSUPPORTED for f32 or a width that is not a multiple of
 * 64; the usual argument, alignment and device-error rules otherwise.
 */
rxl_status rxl_qkv_proj(const rxl_attn_desc *desc, int d_model, const void *h_mem,
                        const void *h_cur, const void *w_q, const void *w_k, const void *w_v,
                        void *q, void *k, void *v, rxl_stream_t stream);

/*
 * One Transformer-XL layer for evaluation streams (forward only): the
 * attention sublayer over [SG(memory); current] (projections, the
 * relative-position attention above, output projection) and a feed-forward
 * sublayer. The pages define the attention and the memory; they leave the
 * rest of the layer open ("obtain the layer's new representation"). Read
 * here as the original post-norm block:
 *   x1  = h_in + Attn([SG(h_mem); h_in]) . W_O
 *   x1n = LayerNorm1(x1)
 *   x2  = x1n + ReLU(x1n . W_1 + b_1) . W_2 + b_2
 *   h_out = LayerNorm2(x2)           (LayerNorm: biased variance, eps 1e-5)
 * Weights (bf16, row-major, device): w_q, w_k, w_v [d, H*dh]; w_o [H*dh, d];
 * r [H, M+L, dh], u, vbias [H, dh] as for the attention; w_1 [d, d_ff], b_1
 * [d_ff]; w_2 [d_ff, d], b_2 [d]; ln*_gamma, ln*_beta [d].
 *   h_mem  [B, M, d] the layer's hidden-state memory ring (as in rxl_qkv_proj)
 *   h_in   [B, L, d] the layer's input; h_out [B, L, d] written
 *   workspace  rxl_layer_fwd_workspace_bytes(desc, d_model, d_ff) bytes:
 *              projected Q/K/V, the attention output, the sublayer
 *              intermediates and fp32 partial sums of the dense layers (when
 *              few output blocks split their K range over several CTAs)
 * The caller advances the memory afterwards with rxl_mem_update(ring over
 * h_mem with D = d, src = h_in): the layer's input states are what the next
 * segment's layer attends to (eq. Tail_M). bf16 only; d_model a multiple of
 * 256, d_ff a multiple of 64 (else RXL_ERR_UNSUPPORTED).
 */
typedef struct {
  const void *w_q, *w_k, *w_v, *w_o;
  const void *r, *u, *vbias;
  const void *ln1_gamma, *ln1_beta;
  const void *w_1, *b_1, *w_2, *b_2;
  const void *ln2_gamma, *ln2_beta;
} rxl_layer_weights;

size_t rxl_layer_fwd_workspace_bytes(const rxl_attn_desc *desc, int d_model, int d_ff);

rxl_status rxl_layer_fwd(const rxl_attn_desc *desc, int d_model, int d_ff, const rxl_layer_weights *w,
                         const void *h_mem, const void *h_in, void *h_out, void *workspace,
                         size_t workspace_bytes, rxl_stream_t stream);

/*
 * FIFO memory ring (eq. Tail_M; update_mems with mem_len == cap).
 *   data         device pointer to plane 0, row 0
 *   planes       independent rings (e.g. B*H), >= 1
 *   cap          capacity M in rows (>= 0; 0 keeps nothing)
 *   D            elements per row (D * elem_size must be a multiple of 16)
 *   plane_stride elements between planes (>= cap*D, 16-byte multiple)
 *   head, len    oldest row's physical index and number of valid rows;
 *                logical row t lives at physical (head + t) mod cap
 */
typedef struct {
  void *data;
  int planes, cap, D;
  long long plane_stride;
  rxl_dtype dtype;
  int head, len;
} rxl_ring;

/*
 * Append L rows per plane and keep the last cap rows:
 *   ring <- Tail_cap([ring_logical; src]).
 * src plane p starts at src + p * src_plane_stride (elements) and holds L
 * contiguous rows of D elements; src must not overlap the rows written.
 * Only the last min(L, cap) rows of src are copied (bit-exact); nothing
 * else in the ring moves. On success ring->head and ring->len are advanced
 * on the host (the struct is caller-owned host memory); on error the ring
 * struct and the device data are unchanged.
 */
rxl_status rxl_mem_update(rxl_ring *ring, const void *src, long long src_plane_stride, int L,
                          rxl_stream_t stream);

/*
 * The same update for n rings (1 <= n <= 8) in one launch, e.g. the K and V
 * rings of a layer, which the recurrence advances together (eq. Tail_M is
 * applied per layer to the states it caches). rings[r] is appended the L rows
 * of srcs[r] (plane stride src_plane_strides[r] elements). All rings must
 * share planes, cap, D, dtype, head and len (else RXL_ERR_INVALID_ARGUMENT)
 * and be distinct structs; data pointers and strides may differ. On success
 * every ring's head and len advance as in rxl_mem_update; on any error
 * nothing is launched and no ring changes.
 */
rxl_status rxl_mem_update_rings(rxl_ring *const *rings, const void *const *srcs,
                                const long long *src_plane_strides, int n, int L,
                                rxl_stream_t stream);

/* Static, human-readable name of a status code. */
const char *rxl_status_string(rxl_status status);

/* The CUDA error code behind the most recent RXL_ERR_CUDA on this thread. */
int rxl_last_cuda_error(void);

/* Number of kernels the most recent successful call on this thread launched. */
int rxl_last_launch_count(void);

/*
 * Device-side failure report. Every wait inside the tensor-core kernels is
 * bounded (about two seconds); a kernel that gives up records it in a device
 * word instead of hanging, drains its in-flight copies, frees its tensor
 * memory and exits with its outputs undefined. This call synchronises the
 * current device, returns the recorded bits (bit 0: forward kernel, bit 1:
 * backward kernels, bit 2: projection kernel, bit 3: dense-layer kernel) and
 * clears them; -1 if the device could not be read.
 * Bit 4 is a range report, not a wait timeout: the bf16 backward runs its
 * position products (dq's r_{i-j} term and dr) on fp16 operands: r, q + vbias
 * and dA (the latter scaled by a power of two so that it stays in range). An
 * r or q + vbias element beyond the fp16 range (|x| > 65504) is clamped to
 * +-65504 and sets bit 4; the gradients of that call are then inexact.
 */
int rxl_device_error_flags(void);

/*
 * Measurement hook (no counterpart in the paper). With timing enabled, every
 * launch of the forward kernel (kernel 0: rxl_attn_fwd*, not the backward's
 * recomputation), of the backward's main kernel (kernel 1: the fused pass
 * over the (query tile, key tile) pairs), of the backward's preparation
 * (kernel 2: zeroing and the (Q+u), (Q+v), D operands, one or two launches)
 * and of the backward's finish kernel (kernel 3) is bracketed by a CUDA event
 * pair recorded on the call's stream; up to 1024 launches per kernel are kept.
 * rxl_kernel_timing_read waits for the recorded events, returns the summed
 * device time in milliseconds and the number of timed launches, and clears
 * them. Launches captured into a CUDA graph are not timed. The events sit
 * between kernels, so a timed launch does not overlap the previous kernel's
 * tail (programmatic dependent launch): timing is for measurement runs, off
 * by default. Both return 0 or a cudaError_t value.
 */
int rxl_kernel_timing(int enable);
int rxl_kernel_timing_read(int kernel, double *total_ms, int *launches);

/*
 * Testing hooks (no counterpart in the paper): they let a test exercise the
 * failure paths above without faulting, trapping or hanging a GPU.
 *
 * rxl_test_fail_next_launch: the next kernel launch of any entry point (on
 * any thread) is not made; it reports cuda_error instead (a cudaError_t
 * value, 0 disarms), so that call returns RXL_ERR_CUDA with
 * rxl_last_cuda_error() == cuda_error. One-shot.
 *
 * rxl_test_forward_wait_timeout: every bounded wait of the forward kernel
 * gives up after wait_cycles SM clock cycles (<= 0 restores the default,
 * about two seconds), and with withhold != 0 the kernel's softmax warps do
 * not signal that the first item's query tiles are ready, so the producer's
 * wait for it runs out: the kernel drains its copies, frees its tensor memory,
 * exits and sets bit 0 of rxl_device_error_flags(). Stays in force until
 * called again with (0, 0). Synchronous; returns 0 or a cudaError_t value.
 */
void rxl_test_fail_next_launch(int cuda_error);
int rxl_test_forward_wait_timeout(long long wait_cycles, int withhold);

#ifdef __cplusplus
}
#endif

#endif /* RXL_H */
