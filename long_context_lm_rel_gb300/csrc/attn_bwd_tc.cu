// Relative-position memory attention backward on sm_103a tensor cores.
//
// With P_ij = exp(scale*A_ij - lse_i) on allowed pairs, D_i = dO_i.O_i and
// dA_ij = scale * P_ij (dO_i.V_j - D_i) (chain rule of "Dimension
// Walkthrough"; stop-gradient of "Why Stop Gradient": nothing is written to
// the cached rows, their K/V gradients are returned like any other row):
//   dV_j = sum_i P_ij dO_i             dK_j = sum_i dA_ij (q_i+u)
//   dQ_i = sum_j dA_ij (k_j + r_{i-j})  dR_d = sum_b sum_{i-j=d} dA_ij (q_i+v)
//   du   = sum dA_ij k_j               dv   = sum dA_ij r_{i-j}
//
// One pass over the visible (query tile, key tile) pairs computes every
// gradient; the logits are formed once per pair. Internally the softmax
// carries scale * P (log2(scale) folded into the exponent), so dA is one
// product away and dV is divided by scale once per item.
//
// Kernels (all on the caller's stream):
//   zero   : dR, the fp32 dQ accumulator and the du/dv outputs <- 0; dK/dV rows
//            of ring slots without valid memory <- 0; R -> fp16 copy
//   prep   : D_i and the (Q+u) (bf16) and (Q+v) (fp16) rows, either from
//            dO.(o + o_lo) in a streaming pass or, without o_lo, from the
//            forward kernel recomputing the fp32 O
//   main   : persistent; a CTA takes one (b, h, 128-key tile) item at a time
//            and loops over the query tiles that see it:
//              S = (Q+u)K^T, G = (Q+v)Rband^T    -> P (skewed G, masked)
//              dP = dO V^T, dV += P^T dO         -> dA, sheared dG
//              dK += dA^T (Q+u), dQc = dA K, dQp = dG Rband, dRband = dG^T (Q+v)
//            dV, dK stay in TMEM for the whole item; the pair's dQc + dQp
//            and its two 128-distance dR blocks are staged in fp32 in the
//            shared buffers its MMAs no longer need and added into fp32
//            global accumulators by TMA tensor reductions, issued by a warp of
//            their own while the next pair proceeds. The column sums of dQp over
//            the rows give dv (added into dvbias, subtracted from du);
//            du = (column sums of dQ) - dv.
//            The position products run in fp16 with dG scaled by a power of
//            two chosen per pair from max |dA|: R rows are several times
//            larger than K rows, and bf16 rounding of dA in that term alone
//            can exceed 1% of max|dQ| on short contexts.
//   finish : dQ -> bf16 with per-head column sums (added into du), dR
//            copied out
// (zero and prep share one launch when the forward kept the low part of O)
#include <math.h>

#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace rxl {
namespace {

using namespace sm103;
using namespace tc;

constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant, each owning 64 of a row's keys
constexpr int kProducerWarp = kSoftmaxWarps;   // TMA loads and MMA issue
constexpr int kStoreWarp = kSoftmaxWarps + 1;  // TMA reductions of the staged dQ / dR rows
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_G_F16 = idesc_f16(128, 128, false, false);  // one 128-distance half of G
constexpr uint32_t IDESC_MN_MN = idesc_bf16(128, 64, true, true);   // A^T . B, both d/row-major tiles
constexpr uint32_t IDESC_K_MN = idesc_bf16(128, 64, false, true);
constexpr uint32_t IDESC_K_MN_F16 = idesc_f16(128, 64, false, true);
constexpr uint32_t IDESC_MN_MN_F16 = idesc_f16(128, 64, true, true);
constexpr float kLog2e = 1.4426950408889634f;

__device__ int g_bwd_error;
// set when an operand converted to fp16 for the position products (R, Q+v)
// was beyond the fp16 range and clamped (reported, not silent)
__device__ int g_bwd_range;

struct BwdParams {
  int B, H, L, cap, m, head, nq, kv_rows, nitems;
  const int *mvis;  // per-row document reset (nullable): newest memory rows per batch row
  float scale, scale_log2;
  const float *lse, *delta;
  __nv_bfloat16 *dk, *dv;
  // [H][64] outputs, zeroed: dvb += the column sums of the position part of
  // dQ, du -= them (the finish kernel adds the column sums of dQ into du)
  float *du, *dvb;
  FastDiv fd_bh, fd_h;  // division by B*H and by H
};

// dR accumulates in [H][kDrPad + kv_rows][64] fp32 with kDrPad leading rows,
// so that every 32-row box of a band starts at a non-negative row (the bands
// start at distance >= -127; their rows below 0 only ever receive zeros).
constexpr int kDrPad = 128;

// K-major operand: 128-byte swizzled [rows][64] tile, k-step kk of 16 elements
// (kk >= 4: the next [rows][64] tile, 16 KB on). kd0 = kdesc0(tile base).
__device__ __forceinline__ uint64_t kdesc0(uint32_t base) { return sdesc_sw128(base, 16, 1024); }
__device__ __forceinline__ uint64_t kdesc(uint64_t kd0, int kk) {
  return sdesc_add(kd0, (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32));
}
// MN-major operand: [K rows][MN] tiles of 64 MN columns (16 KB apart), k-step
// of 16 rows. md0 = mndesc0(tile base).
__device__ __forceinline__ uint64_t mndesc0(uint32_t base) { return sdesc_sw128(base, 16384, 1024); }
__device__ __forceinline__ uint64_t mndesc(uint64_t md0, int kk) { return sdesc_add(md0, (uint32_t)(kk * 2048)); }

// 64 fp32 values (keys 64*hf ..) of row ii as bf16 into column block hf of a
// [128][128] K-major 128-byte-swizzled tile pair; row = sw128_row(block hf, ii).
__device__ __forceinline__ void store_half_bf16(uint32_t row, const float (&a)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(sw128_at(row, c), pack_bf16(a[8 * c + 0], a[8 * c + 1]),
                 pack_bf16(a[8 * c + 2], a[8 * c + 3]), pack_bf16(a[8 * c + 4], a[8 * c + 5]),
                 pack_bf16(a[8 * c + 6], a[8 * c + 7]));
}

// Bounded rendezvous of the two warps of a lane quadrant (mbarrier, count 2).
__device__ __forceinline__ bool pair_sync(uint32_t bar, int lane, uint32_t &phase,
                                          volatile int *abort_flag) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, phase & 1, abort_flag));
  ++phase;
  return ok;
}

// ------------------------------------------------------------ main kernel

// Shared memory: K, V, (Q+u), two (Q+v) buffers (the next pair's rows load
// while the current pair still reads its own), three 16 KB slots that hold
// dO and the two 128-row halves of the R band in turn, P/dA (bf16, then the
// pair's dQ staging), dG (fp16, then its dR staging), barriers.
constexpr uint32_t F_K = 0, F_V = 16384, F_QU = 32768, F_QV0 = 49152, F_QV1 = 65536, F_SLOT = 81920;
constexpr uint32_t F_PA = 131072, F_DG = 163840, F_BAR = 229376;
constexpr uint32_t F_SMEM = F_BAR + 512 + 1024;
// TMEM columns: dV, dK accumulators; S (then dP); G (then dQc, dQp, dR blocks)
constexpr uint32_t TM_DV = 0, TM_DK = 64, TM_S = 128, TM_G = 256;
constexpr uint32_t TM_QC = 256, TM_QP = 320, TM_R0 = 384;

// A work item is one (b, h, key tile); items are numbered key tile major, so
// that the memory tiles and the early current tiles (seen by the most query
// tiles) come first. CTA c of G takes one item per round, snake order. Under
// a per-row document reset a batch row may have fewer key tiles than the
// item numbering allows for; its surplus items are empty (NQ = 0).
struct FItem {
  int bh, h, qlo, NQ;
  KeyTile x;
};

__device__ __forceinline__ FItem fitem(const BwdParams &p, int w) {
  FItem it;
  const int t = (int)p.fd_bh.div((uint32_t)w);  // w = t * B*H + bh
  it.bh = w - t * (int)p.fd_bh.d;
  const int b = (int)p.fd_h.div((uint32_t)it.bh);
  it.h = it.bh - b * (int)p.fd_h.d;
  const RowMemory rm = row_memory(p.mvis, b, p.m, p.cap, p.head);
  const KeyTiles tiles(rm.m, p.cap, rm.head, p.L);
  if (t >= tiles.count()) {
    it.x.phys0 = it.x.jlog0 = it.x.nvalid = 0;
    it.qlo = it.NQ = 0;
    return it;
  }
  it.x = tiles.get(t);
  it.qlo = it.x.jlog0 >= 0 ? it.x.jlog0 / BQ : 0;
  it.NQ = p.nq - it.qlo;
  return it;
}

// Walks this CTA's (item, query tile) pairs: r counts rounds, k the items
// with work, n the query tiles of the current item.
struct PairCursor {
  int r, k, n;
  bool valid;
  FItem it;
  __device__ __forceinline__ static int item_of_round(int r) {
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((r & 1) ? G - 1 - c : c);
  }
  // from round r on, the first item that has work
  __device__ void seek(const BwdParams &p) {
    for (;; ++r) {
      const int w = item_of_round(r);
      valid = w < p.nitems;
      if (!valid) return;
      it = fitem(p, w);
      if (it.NQ > 0) return;
    }
  }
  __device__ void init(const BwdParams &p) {
    r = 0;
    k = 0;
    n = 0;
    seek(p);
  }
  __device__ void next(const BwdParams &p) {
    if (++n == it.NQ) {
      n = 0;
      ++k;
      ++r;
      seek(p);
    }
  }
  __device__ int i0() const { return (it.qlo + n) * BQ; }
};

__global__ void __launch_bounds__(kThreads, 1)
rxl_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_r16, const __grid_constant__ CUtensorMap tm_qu,
                    const __grid_constant__ CUtensorMap tm_qv16, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dr,
                    const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t b0 = sb + F_BAR;
  // TMA: (Q+v), the R band and, for an item's first pair, V of pair g
  // complete one phase of bar_nx0 / bar_nx1 (by the parity of g), so that the
  // producer waits once per pair for them; dO of a pair; (Q+u) of a pair,
  // with K for an item's first pair
  const uint32_t bar_nx0 = b0 + 8, bar_nx1 = b0 + 16;
  const uint32_t bar_do = b0 + 32, bar_qu = b0 + 40;
  // MMA commits: S and G; dP; dV; dK and dQc; dQp; dR (the pair's last)
  const uint32_t bar_sg = b0 + 48, bar_dp = b0 + 56, bar_dv = b0 + 64, bar_f0 = b0 + 72;
  const uint32_t bar_dq = b0 + 80, bar_fin = b0 + 88, bar_drain = b0 + 96;
  // softmax warps (256 arrivals): P, dA, dG written; TMEM G columns read;
  // dV/dK of an item read
  const uint32_t bar_p = b0 + 104, bar_da = b0 + 112, bar_ds = b0 + 120, bar_fl = b0 + 128;
  const uint32_t bar_acc = b0 + 136;
  const uint32_t bar_red = b0 + 144;     // max |dA| of each softmax warp (8)
  const uint32_t bar_x0 = b0 + 152;      // 4 lane-quadrant rendezvous (2 each)
  const uint32_t bar_stq = b0 + 184;     // each softmax warp staged its dQ rows (8)
  const uint32_t bar_str = b0 + 192;     // each softmax warp staged its dR rows (8)
  const uint32_t bar_sfree = b0 + 200;   // the dQ staging has been read (1)
  const uint32_t bar_gfree = b0 + 208;   // the dR staging has been read (1)
  const uint32_t bar_sread = b0 + 288;   // each softmax warp read its S / G columns (8)
  const uint32_t bar_rlo = b0 + 296;     // MMA commit: dQp's products with the band's lower half
  uint32_t *tmem_slot = (uint32_t *)(smem + F_BAR + 216);
  volatile int *abort_flag = (volatile int *)(smem + F_BAR + 220);
  volatile float *wmax = (volatile float *)(smem + F_BAR + 224);  // [2][8]
  if (threadIdx.x == 0) {
    mbar_init(bar_nx0, 1); mbar_init(bar_nx1, 1); mbar_init(bar_do, 1); mbar_init(bar_qu, 1);
    mbar_init(bar_sg, 1); mbar_init(bar_dp, 1); mbar_init(bar_dv, 1); mbar_init(bar_f0, 1);
    mbar_init(bar_dq, 1); mbar_init(bar_fin, 1); mbar_init(bar_drain, 1);
    mbar_init(bar_p, kSoftmaxWarps * 32); mbar_init(bar_da, kSoftmaxWarps * 32);
    mbar_init(bar_ds, kSoftmaxWarps * 32); mbar_init(bar_fl, kSoftmaxWarps * 32);
    mbar_init(bar_acc, kSoftmaxWarps * 32);
    mbar_init(bar_red, kSoftmaxWarps);
    for (int q = 0; q < 4; ++q) mbar_init(bar_x0 + 8 * q, 2);
    mbar_init(bar_stq, kSoftmaxWarps); mbar_init(bar_str, kSoftmaxWarps);
    mbar_init(bar_sfree, 1); mbar_init(bar_gfree, 1); mbar_init(bar_sread, kSoftmaxWarps);
    mbar_init(bar_rlo, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    if (lane == 0) {
      tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v); tma_prefetch_desc(&tm_r16);
      tma_prefetch_desc(&tm_qu); tma_prefetch_desc(&tm_qv16); tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_dq); tma_prefetch_desc(&tm_dr);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // inputs written by the previous kernel on the stream
  griddep_launch_dependents();

  if (warp == kProducerWarp) {
    // ------------------------------------------------ producer / MMA issuer
    // Pair g reads (Q+v) buffer g & 1. Each operand is reloaded as soon as
    // its last reader of the previous pair is done: (Q+u), and K and V of a
    // new item, once dK and dQc are; dO and the R band by the slot rotation
    // below; the next pair's (Q+v) goes into the other buffer right after
    // this pair's G is issued. So the next pair's S is issued right behind
    // this pair's dR, for a new item too, and the tensor pipe does not idle
    // between items.
    // The whole warp runs the schedule (uniform control flow, so that the
    // descriptors stay in uniform registers); one elected thread issues.
    // A phase of bar_nx{b} is opened by the first copy issued without
    // arrival ((Q+v)) and closed by the last one (an R half), which arrives;
    // the phase then completes when all of its bytes have landed.
    int n_do = 0, n_qu = 0, nx_closed0 = 0, nx_closed1 = 0;
    bool nx_open0 = false, nx_open1 = false;
    // (the polling loop out of line: the producer's code is the part of the
    // kernel whose size costs time, while the softmax warps' waits stay
    // inline, as a call there forces register saves)
    auto wait = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait_lean(bar, parity, abort_flag));
    };
    // The R band of a pair is two 128-row halves (distances d0 .. d0+127 and
    // d0+128 .. d0+255). The next query tile of the same item needs
    // d0+128 .. d0+383: its lower half is this pair's upper half, already
    // resident. Three slots rotate among dO and the two halves, each refilled
    // as soon as its last reader is done: dO's once dV is done, the lower
    // half's once dQp's products with it are, the upper half's once dQp is.
    //   same item: next upper half -> dO's slot, next dO -> lower half's
    //   new item : next lower half -> dO's slot, next upper half -> lower
    //              half's, next dO -> upper half's
    // s_lo, s_hi, s_do: slot of each operand.
    int s_do = 0, s_lo = 1, s_hi = 2;
    auto slot = [](int k) { return F_SLOT + (uint32_t)k * 16384u; };
    auto load_do = [&](const PairCursor &c, int k) {
      if (elect_one()) {
        mbar_expect_tx(bar_do, 16384);
        tma_load_3d(sb + slot(k), &tm_do, 0, c.i0(), c.it.bh, bar_do);
      }
      __syncwarp();
      ++n_do;
    };
    // (Q+u) of a pair, with K for the first pair of an item (S reads both)
    auto load_qu = [&](const PairCursor &c) {
      const bool with_k = c.n == 0;
      if (elect_one()) {
        mbar_expect_tx(bar_qu, with_k ? 2 * 16384 : 16384);
        tma_load_3d(sb + F_QU, &tm_qu, 0, c.i0(), c.it.bh, bar_qu);
        if (with_k) tma_load_3d(sb + F_K, &tm_k, 0, c.it.x.phys0, c.it.bh, bar_qu);
      }
      __syncwarp();
      ++n_qu;
    };
    // one 16 KB tile into the phase of bar_nx{pb} (pb: the parity of the
    // pair it is for); the phase's last copy closes it (arrives)
    auto load_nx = [&](uint32_t dst, const CUtensorMap *tm, int y, int z, int pb, bool close) {
      if (elect_one()) {
        const uint32_t bar = pb ? bar_nx1 : bar_nx0;
        if (close)
          mbar_expect_tx(bar, 16384);
        else
          mbar_expect_tx_noarrive(bar, 16384);
        tma_load_3d(dst, tm, 0, y, z, bar);
      }
      __syncwarp();
      bool &open = pb ? nx_open1 : nx_open0;
      if (close) {
        open = false;
        ++(pb ? nx_closed1 : nx_closed0);
      } else {
        open = true;
      }
    };
    auto load_qv = [&](const PairCursor &c, int pb) {
      load_nx(sb + (pb ? F_QV1 : F_QV0), &tm_qv16, c.i0(), c.it.bh, pb, false);
    };
    auto band0 = [](const PairCursor &c) { return c.i0() - c.it.x.jlog0 - (BK - 1); };
    // operand descriptors: two bases built once (K-major and MN-major
    // layouts at the start of shared memory); a tile, k-step or buffer is
    // a constant added to them
    const uint64_t kb = kdesc0(sb), mb0 = mndesc0(sb);
    const uint64_t k_qu = sdesc_add(kb, F_QU), k_k = sdesc_add(kb, F_K), k_slot = sdesc_add(kb, F_SLOT);
    const uint64_t k_v = sdesc_add(kb, F_V), k_pa = sdesc_add(kb, F_PA), k_dg = sdesc_add(kb, F_DG);
    const uint64_t m_pa = sdesc_add(mb0, F_PA), m_slot = sdesc_add(mb0, F_SLOT), m_qu = sdesc_add(mb0, F_QU);
    const uint64_t m_k = sdesc_add(mb0, F_K), m_dg = sdesc_add(mb0, F_DG);
    bool ok = true;
    PairCursor c;
    c.init(p);
    if (c.valid) {
      load_qv(c, 0);
      load_qu(c);
      load_do(c, s_do);
      load_nx(sb + F_V, &tm_v, c.it.x.phys0, c.it.bh, 0, false);
      load_nx(sb + slot(s_lo), &tm_r16, band0(c), c.it.h, 0, false);
      load_nx(sb + slot(s_hi), &tm_r16, band0(c) + 128, c.it.h, 0, true);
    }
    // S of pair g, once its (Q+u) (and an item's K) have landed, into the S
    // columns (free since the previous pair's dA was formed)
    auto issue_s = [&](int g) {
      if (!(ok = wait(bar_qu, g & 1))) return;
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_S, kdesc(k_qu, k), kdesc(k_k, k), IDESC_S, k > 0);
      }
      __syncwarp();
    };
    // G of pair g, once its (Q+v), R band (and an item's V) have landed and
    // the previous pair's flush has released the G columns; commits S and G
    auto issue_g = [&](int g) {
      if (!(ok = wait((g & 1) ? bar_nx1 : bar_nx0, (g >> 1) & 1))) return;
      if (g > 0 && !(ok = wait(bar_fl, (g - 1) & 1))) return;
      const uint64_t k_qv = sdesc_add(kb, (g & 1) ? F_QV1 : F_QV0);
      const uint64_t k_rlo = sdesc_add(k_slot, s_lo * 16384), k_rhi = sdesc_add(k_slot, s_hi * 16384);
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // G columns 0-127 from the lower half, 128-255 from the upper
          mma_bf16(tmem + TM_G, kdesc(k_qv, k), kdesc(k_rlo, k), IDESC_G_F16, k > 0);
          mma_bf16(tmem + TM_G + 128, kdesc(k_qv, k), kdesc(k_rhi, k), IDESC_G_F16, k > 0);
        }
        mma_commit(bar_sg);
      }
      __syncwarp();
    };
    // after G of pair g: (Q+v) of the pair after it (cursor n2) into the
    // other buffer, last read by pair g-1's dR, which completed before pair
    // g-1's flush released the G columns; n2's other operands come from HBM
    // on first touch (about 2.5k cycles): pulled into L2 now, ahead of their
    // loads
    auto after_g = [&](int g, const PairCursor &n2) {
      if (!n2.valid) return;
      load_qv(n2, (g + 1) & 1);
      if (elect_one()) {
        const int i0n = n2.i0(), d0n = band0(n2);
        tma_prefetch_l2_3d(&tm_qu, 0, i0n, n2.it.bh);
        tma_prefetch_l2_3d(&tm_do, 0, i0n, n2.it.bh);
        tma_prefetch_l2_3d(&tm_r16, 0, d0n + 128, n2.it.h);
        if (n2.n == 0) {
          tma_prefetch_l2_3d(&tm_r16, 0, d0n, n2.it.h);
          tma_prefetch_l2_3d(&tm_k, 0, n2.it.x.phys0, n2.it.bh);
          tma_prefetch_l2_3d(&tm_v, 0, n2.it.x.phys0, n2.it.bh);
        }
      }
      __syncwarp();
    };
    PairCursor nx = c;
    nx.next(p);
    if (c.valid) {
      issue_s(0);
      if (ok) issue_g(0);
      if (ok) after_g(0, nx);
    }
    // Pair g's S and G were issued at the end of the previous iteration (by
    // the prologue for the first pair), right behind pair g-1's dR, so that
    // only the latency of G lies between a pair's flush and the next pair's
    // softmax.
    for (int g = 0; ok && c.valid; ++g) {
      const bool first = c.n == 0;
      const int buf = g & 1;
      const uint64_t m_qv = sdesc_add(mb0, buf ? F_QV1 : F_QV0);
      const uint64_t m_rlo = sdesc_add(m_slot, s_lo * 16384), m_rhi = sdesc_add(m_slot, s_hi * 16384);
      const uint64_t k_do = sdesc_add(k_slot, s_do * 16384), m_do = sdesc_add(m_slot, s_do * 16384);
      // dP into the S columns as soon as the softmax warps have read S: it
      // runs while they form P
      if (!(ok = wait(bar_sread, g & 1))) break;
      if (!(ok = wait(bar_do, g & 1))) break;
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_S, kdesc(k_do, k), kdesc(k_v, k), IDESC_S, k > 0);
        mma_commit(bar_dp);  // dA needs only dP
      }
      __syncwarp();
      if (!(ok = wait(bar_p, g & 1))) break;
      // the first dV of an item overwrites the accumulators: the previous
      // item's epilogue must have read them
      if (first && c.k > 0 && !(ok = wait(bar_acc, (c.k - 1) & 1))) break;
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)  // dV += P^T dO
          mma_bf16(tmem + TM_DV, mndesc(m_pa, k), mndesc(m_do, k), IDESC_MN_MN, (!first || k > 0) ? 1u : 0u);
        mma_commit(bar_dv);
      }
      __syncwarp();
      // dO's slot is free once dP and dV are done: the next pair's upper
      // half (same item; the last copy of its phase) or lower half (new item)
      const bool same = nx.valid && nx.n != 0;
      if (nx.valid) {
        if (!(ok = wait(bar_dv, g & 1))) break;
        load_nx(sb + slot(s_do), &tm_r16, band0(nx) + (same ? 128 : 0), nx.it.h, buf ^ 1, same);
      }
      // dK and dQc as soon as dA is written, while the softmax warps
      // shear dG; then dQp and the dR blocks
      if (!(ok = wait(bar_da, g & 1))) break;
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)  // dK += dA^T (Q+u)
          mma_bf16(tmem + TM_DK, mndesc(m_pa, k), mndesc(m_qu, k), IDESC_MN_MN, (!first || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 8; ++k)  // dQc = dA K
          mma_bf16(tmem + TM_QC, kdesc(k_pa, k), mndesc(m_k, k), IDESC_K_MN, k > 0);
        mma_commit(bar_f0);
      }
      __syncwarp();
      if (nx.valid) {  // (Q+u), K and V are free once dK and dQc are done
        if (!(ok = wait(bar_f0, g & 1))) break;
        load_qu(nx);
        if (!same) load_nx(sb + F_V, &tm_v, nx.it.x.phys0, nx.it.bh, buf ^ 1, false);
      }
      if (!(ok = wait(bar_ds, g & 1))) break;
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)  // dQp = dG Rband (fp16), band rows 16k .. 16k+15: lower half
          mma_bf16(tmem + TM_QP, kdesc(k_dg, k), mndesc(m_rlo, k), IDESC_K_MN_F16, k > 0);
        mma_commit(bar_rlo);
#pragma unroll
        for (int k = 8; k < 16; ++k)  // upper half
          mma_bf16(tmem + TM_QP, kdesc(k_dg, k), mndesc(m_rhi, k & 7), IDESC_K_MN_F16, 1u);
        mma_commit(bar_dq);
      }
      __syncwarp();
      if (elect_one()) {
        // dR right behind dQp (it does not read the R band): the tensor pipe
        // runs the two chains back to back
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)  // dR band = dG^T (Q+v), two 128-distance blocks (fp16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16(tmem + TM_R0 + 64 * mb, mndesc(sdesc_add(m_dg, 2 * mb * 16384), k), mndesc(m_qv, k),
                     IDESC_MN_MN_F16, k > 0);
        mma_commit(bar_fin);
      }
      __syncwarp();
      if (!nx.valid) break;
      // The lower half's slot is free once dQp's products with it are done
      // (and with them every earlier product of the pair): the next dO (same
      // item) or the next upper half (new item; the last copy of its phase).
      // The slots rotate: the next pair's lower half is this pair's upper
      // half (same item) or the band loaded into dO's slot (new item).
      const int old_lo = s_lo;
      if (same) {
        s_lo = s_hi;
        s_hi = s_do;
        s_do = old_lo;
      } else {
        if (!(ok = wait(bar_rlo, g & 1))) break;
        load_nx(sb + slot(old_lo), &tm_r16, band0(nx) + 128, nx.it.h, buf ^ 1, true);
        s_lo = s_do;
        s_do = s_hi;
        s_hi = old_lo;
      }
      // the next pair's S and G (same item: nothing they read is still on
      // its way, so they go first)
      issue_s(g + 1);
      if (!ok) break;
      issue_g(g + 1);
      if (!ok) break;
      if (same) {
        if (!(ok = wait(bar_rlo, g & 1))) break;
        load_do(nx, s_do);
      }
      PairCursor n2 = nx;
      n2.next(p);
      after_g(g + 1, n2);
      // new item: the next dO into the old upper half's slot once dQp is done
      if (!same) {
        if (!(ok = wait(bar_dq, g & 1))) break;
        load_do(nx, s_do);
      }
      c = nx;
      nx = n2;
    }
    if (!ok) {
      // wind down: let in-flight copies and MMAs land before TMEM and
      // shared memory are released
      // (the latest copy of each barrier; an earlier one completed before
      // the latest was issued, and a completed phase returns at once)
      if (elect_one()) {
        volatile int no_abort = 0;
        // a phase whose closing copy was not issued yet is closed here, so
        // that it completes once the copies issued for it have landed
        if (nx_open0) mbar_arrive(bar_nx0);
        if (nx_open1) mbar_arrive(bar_nx1);
        const int ph0 = nx_closed0 + (nx_open0 ? 1 : 0), ph1 = nx_closed1 + (nx_open1 ? 1 : 0);
        if (ph0 > 0) mbar_wait_lean(bar_nx0, (ph0 - 1) & 1, &no_abort);
        if (ph1 > 0) mbar_wait_lean(bar_nx1, (ph1 - 1) & 1, &no_abort);
        if (n_do > 0) mbar_wait_lean(bar_do, (n_do - 1) & 1, &no_abort);
        if (n_qu > 0) mbar_wait_lean(bar_qu, (n_qu - 1) & 1, &no_abort);
        mma_commit(bar_drain);
        mbar_wait_lean(bar_drain, 0, &no_abort);
        atomicExch(&g_bwd_error, 1);
      }
      __syncwarp();
    }
  } else if (warp == kStoreWarp) {
    // --------------------------------------------------- reduction issuer
    if (lane == 0) {
      bool ok = true;
      PairCursor c;
      c.init(p);
      for (int g = 0; c.valid; ++g) {
        const int i0 = c.i0();
        const int d0 = kDrPad + i0 - c.it.x.jlog0 - (BK - 1);  // >= 1
        // warp (quad, hf) staged its dQ box in the P/dA buffer and its dR
        // block-hf rows in dG atoms 2hf, 2hf+1; dQ is staged first (while
        // the dR MMAs run)
        if (!(ok = mbar_wait(bar_stq, g & 1, abort_flag))) break;
#pragma unroll 1
        for (int w = 0; w < kSoftmaxWarps; ++w) {
          const int quad = w & 3, hf = w >> 2;
          const int qrow = i0 + 32 * quad;
          if (qrow < p.L)
            tma_reduce_add_3d(&tm_dq, 32 * hf, qrow, c.it.bh, sb + F_PA + hf * 16384 + quad * 4096);
        }
        bulk_commit();
        if (!(ok = mbar_wait(bar_str, g & 1, abort_flag))) break;
#pragma unroll 1
        for (int w = 0; w < kSoftmaxWarps; ++w) {
          const int quad = w & 3, hf = w >> 2;
          const int drow = d0 + 128 * hf + 32 * quad;
          if (drow < kDrPad + p.kv_rows) {
            tma_reduce_add_3d(&tm_dr, 0, drow, c.it.h, sb + F_DG + 2 * hf * 16384 + quad * 4096);
            tma_reduce_add_3d(&tm_dr, 32, drow, c.it.h, sb + F_DG + (2 * hf + 1) * 16384 + quad * 4096);
          }
        }
        bulk_commit();
        bulk_wait_read_but_latest();
        mbar_arrive(bar_sfree);
        bulk_wait_read();
        mbar_arrive(bar_gfree);
        c.next(p);
      }
      // the reductions must be complete before shared memory goes away
      bulk_wait_all();
      if (!ok) atomicExch(&g_bwd_error, 4);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------- softmax warps
    const int quad = warp & 3, hf = warp >> 2;
    const int ii = quad * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t bar_x = bar_x0 + 8 * quad;
    const int c0 = ii >> 3;  // first 16-byte chunk of row ii's sheared values
    // row ii in the P/dA block hf (also dQ staging), in the dG tile (chunk C
    // at sw128_at(row_dg, C & 7) + (C >> 3) * 16384) and in dR staging atom 2hf
    const uint32_t row_pa = sw128_row(sb + F_PA + hf * 16384, ii);
    const uint32_t row_dg = sw128_row(sb + F_DG, ii);
    const uint32_t row_dr = sw128_row(sb + F_DG + 2 * hf * 16384, ii);
    uint32_t xphase = 0;
    // this thread's dQp row values summed over the pairs of the item
    // (columns 32*hf ..); summed over the warp's rows once per item
    float dva[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) dva[e] = 0.f;
    // the exponent bias carries log2(scale): the softmax handles scale * P
    // throughout (dA = (scale P)(dP - D) in two packed ops); the P tile of
    // the dV product holds scale * P, so dV is divided by scale at the end
    const float log2_scale = log2f(p.scale), inv_scale = 1.f / p.scale;
    bool ok = true;
    PairCursor c;
    c.init(p);
    // lse and D of row ii of a pair's query tile, loaded a pair ahead (for
    // a new (b, h) they come from HBM); rows past L: lse = +inf makes P = 0
    // without a select per key
    float lse_n = INFINITY, d_n = 0.f;
    auto load_stats = [&](const PairCursor &cc) {
      const int i = cc.i0() + ii;
      if (i < p.L) {
        const size_t row = (size_t)cc.it.bh * p.L + i;
        lse_n = p.lse[row];
        d_n = p.delta[row];
      } else {
        lse_n = INFINITY;
        d_n = 0.f;
      }
    };
    if (c.valid) load_stats(c);
    for (int g = 0; c.valid; ++g) {
      const FItem it = c.it;
      const int i0 = c.i0();
      const int i = i0 + ii;
      const float lse2 = lse_n * kLog2e;
      const float Di = d_n;
      ok = mbar_wait(bar_sg, g & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      if (c.n == 0 && ii >= it.x.nvalid) {
        // rows of K and V past the run hold another run's (or junk) data:
        // zero them so that 0 * junk cannot leak into dP or dQc (the
        // logits of those keys are masked, the S products of later pairs
        // then read zeros)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          st_shared_v4(sb + F_K + sw128_offset(ii, 4 * hf + cc), 0, 0, 0, 0);
          st_shared_v4(sb + F_V + sw128_offset(ii, 4 * hf + cc), 0, 0, 0, 0);
        }
      }
      float y[64];
      half_tile_exponents(trow, TM_S, TM_G, quad, lane, hf, i, it.x, p.scale_log2, log2_scale - lse2, y);
      // S is read: dP may take its columns (and read the zeroed V rows)
      if (c.n == 0 && it.x.nvalid < BK) fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sread);
#pragma unroll
      for (int k = 0; k < 64; ++k) y[k] = ex2(y[k]);  // scale * P
      // the P/dA buffer held the previous pair's dQ staging
      if (g > 0) {
        ok = mbar_wait(bar_sfree, (g - 1) & 1, abort_flag);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
      }
      store_half_bf16(row_pa, y);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_p);
      ok = mbar_wait(bar_dp, g & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dp[32];
        tmem_ld32(trow + TM_S + 64 * hf + 32 * cc, dp);
        tmem_wait_ld();
        const float2 ndi2 = make_float2(-Di, -Di);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {  // dA (P = 0 and finite dP off the allowed pairs)
          const float2 d = __fadd2_rn(make_float2(__uint_as_float(dp[k]), __uint_as_float(dp[k + 1])), ndi2);
          const float2 t = __fmul2_rn(make_float2(y[32 * cc + k], y[32 * cc + k + 1]), d);
          y[32 * cc + k] = t.x;
          y[32 * cc + k + 1] = t.y;
        }
      }
      // CTA-wide max |dA| of this pair -> power-of-two fp16 scale of dG;
      // this warp's part is published while the dV product may still run
      float am = 0.f;
#pragma unroll
      for (int k = 0; k < 64; k += 2) am = fmax3(am, fabsf(y[k]), fabsf(y[k + 1]));
      am = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(am)));
      if (lane == 0) {
        wmax[(g & 1) * 8 + warp] = am;
        mbar_arrive(bar_red);
      }
      // P is no longer read once dV is done
      ok = mbar_wait(bar_dv, g & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      store_half_bf16(row_pa, y);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_da);
      ok = mbar_wait(bar_red, g & 1, abort_flag);  // bounded, unlike a named barrier
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      am = 0.f;
#pragma unroll
      for (int w = 0; w < kSoftmaxWarps; ++w) am = fmaxf(am, wmax[(g & 1) * 8 + w]);
      // sig = 2^(14 - ceil(log2 max|dA|)), so max |sig dA| <= 2^14, and
      // inv = 1/sig, both read off the exponent bits of max|dA| (1 for 0)
      float sig, inv;
      {
        const uint32_t ab = __float_as_uint(am);
        int ce = (int)(ab >> 23) - 127 + ((ab & 0x7FFFFFu) != 0u);  // ceil(log2 am), am normal
        int e = am > 0.f ? 14 - ce : 0;
        e = e < -126 ? -126 : (e > 126 ? 126 : e);
        sig = __uint_as_float((uint32_t)(e + 127) << 23);
        inv = __uint_as_float((uint32_t)(127 - e) << 23);
      }
      // the dG buffer held the previous pair's dR staging
      if (g > 0) {
        ok = mbar_wait(bar_gfree, (g - 1) & 1, abort_flag);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
      }
      // Sheared dG row ii: key jj sits at column ii + 127 - jj. This half's
      // keys fill columns s .. s+63 (s = ii + 64 - 64 hf) in reverse key
      // order; shifted right by s mod 8 = ii mod 8 elements they line up
      // with 16-byte chunks (s >> 3) .. (s >> 3) + 8. w holds them as fp16
      // pairs (element x in half x & 1 of word x >> 1).
      {
        const int r = ii & 7;
        uint32_t w[36];
        const float2 sig2 = make_float2(sig, sig);
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const float2 t = __fmul2_rn(make_float2(y[63 - 2 * m], y[62 - 2 * m]), sig2);
          w[m] = pack_f16(t.x, t.y);
        }
#pragma unroll
        for (int m = 32; m < 36; ++m) w[m] = 0u;
        // odd part of the shift: element x <- x - 1 by a byte permute of
        // neighbouring words; then whole words by 2 and 1
        const uint32_t sel = (r & 1) ? 0x5432u : 0x7654u;
#pragma unroll
        for (int m = 35; m >= 0; --m) w[m] = __byte_perm(m > 0 ? w[m > 0 ? m - 1 : 0] : 0u, w[m], sel);
#pragma unroll
        for (int b = 2; b >= 1; b >>= 1) {
          const bool take = ((r >> 1) & b) != 0;
#pragma unroll
          for (int m = 35; m >= 0; --m) w[m] = take ? (m >= b ? w[m >= b ? m - b : 0] : 0u) : w[m];
        }
        const int cbase = c0 + (hf ? 0 : 8);
        // columns outside [ii, ii + 127] are zero (staging overwrote them)
        if (hf == 1) {
#pragma unroll
          for (int C = 0; C < 15; ++C)
            if (C < c0) st_shared_v4(sw128_at(row_dg, C & 7) + (C >> 3) * 16384, 0, 0, 0, 0);
        } else {
#pragma unroll
          for (int C = 17; C < 32; ++C)
            if (C > c0 + 16) st_shared_v4(sw128_at(row_dg, C & 7) + (C >> 3) * 16384, 0, 0, 0, 0);
        }
        // chunk c0 + 8 is shared by the two halves: the upper half (hf 1)
        // writes its part there (zeros in the other half's positions), the
        // lower half ORs its part in after the rendezvous
        const uint32_t shared_chunk = sw128_at(row_dg, (c0 + 8) & 7) + ((c0 + 8) >> 3) * 16384;
        if (hf == 1) {
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int C = cbase + t;
            st_shared_v4(sw128_at(row_dg, C & 7) + (C >> 3) * 16384, w[4 * t],
                         w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
          }
          st_shared_v4(shared_chunk, w[32], w[33], w[34], w[35]);
        } else {
#pragma unroll
          for (int t = 1; t < 9; ++t) {
            const int C = cbase + t;
            st_shared_v4(sw128_at(row_dg, C & 7) + (C >> 3) * 16384, w[4 * t],
                         w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
          }
        }
        if (!(ok = pair_sync(bar_x, lane, xphase, abort_flag))) break;
        if (hf == 0) {
          // the two halves' values occupy complementary positions of the
          // shared chunk (+0 elsewhere): OR merges them exactly
          const uint4 o = ld_shared_v4(shared_chunk);
          st_shared_v4(shared_chunk, o.x | w[0], o.y | w[1], o.z | w[2], o.w | w[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_ds);
      float v[32];
      ok = mbar_wait(bar_dq, g & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      {
        // flush, dQ part (while the dR MMAs run): this half's 32 dQ columns
        // of row ii staged in fp32 (a 128-byte swizzled 32-column box) in the
        // P/dA buffer, whose dA the finished dK/dQc products no longer read
        uint32_t qc[32], qp[32];
        tmem_ld32(trow + TM_QC + 32 * hf, qc);
        tmem_ld32(trow + TM_QP + 32 * hf, qp);
        tmem_wait_ld();
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 t = __fmul2_rn(make_float2(__uint_as_float(qp[e]), __uint_as_float(qp[e + 1])), inv2);
          v[e] = t.x;
          v[e + 1] = t.y;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 lo = __fadd2_rn(make_float2(__uint_as_float(qc[4 * e]), __uint_as_float(qc[4 * e + 1])),
                                       make_float2(v[4 * e], v[4 * e + 1]));
          const float2 hi = __fadd2_rn(make_float2(__uint_as_float(qc[4 * e + 2]), __uint_as_float(qc[4 * e + 3])),
                                       make_float2(v[4 * e + 2], v[4 * e + 3]));
          st_shared_v4(sw128_at(row_pa, e), __float_as_uint(lo.x),
                       __float_as_uint(lo.y), __float_as_uint(hi.x), __float_as_uint(hi.y));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_stq);
      }
      ok = mbar_wait(bar_fin, g & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      {
        // flush, dR part: row ii of dR block hf, staged in fp32 in dG atoms
        // 2hf, 2hf+1 (the dG products are done)
        uint32_t ra[32], rb[32];
        tmem_ld32(trow + TM_R0 + 64 * hf, ra);
        tmem_ld32(trow + TM_R0 + 64 * hf + 32, rb);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_fl);  // the G columns may take the next pair's logits
        const float2 inv2 = make_float2(inv, inv);
        auto scaled = [&](const uint32_t(&src)[32], int e) {
          return __fmul2_rn(make_float2(__uint_as_float(src[e]), __uint_as_float(src[e + 1])), inv2);
        };
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 a0 = scaled(ra, 4 * e), a1 = scaled(ra, 4 * e + 2);
          const float2 b0 = scaled(rb, 4 * e), b1 = scaled(rb, 4 * e + 2);
          st_shared_v4(sw128_at(row_dr, e), __float_as_uint(a0.x),
                       __float_as_uint(a0.y), __float_as_uint(a1.x), __float_as_uint(a1.y));
          st_shared_v4(sw128_at(row_dr, e) + 16384, __float_as_uint(b0.x),
                       __float_as_uint(b0.y), __float_as_uint(b1.x), __float_as_uint(b1.y));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_str);
      }
      {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 t = __fadd2_rn(make_float2(dva[e], dva[e + 1]), make_float2(v[e], v[e + 1]));
          dva[e] = t.x;
          dva[e + 1] = t.y;
        }
      }
      c.next(p);
      if (c.valid) load_stats(c);
      if (c.valid && c.n != 0) continue;
      // ---- end of the item: dV (half 0) and dK (half 1) rows, dv sums.
      // Thread ii holds row ii (128 bytes); stored as they are, each store
      // instruction would write 32 partial sectors, which slows the whole SM
      // down. An 8 x 8 transpose of 16-byte chunks within each group of 8
      // lanes (three shuffle butterflies) leaves lane 8k + r with chunk r of
      // the group's rows 8k .. 8k+7, so that each store instruction writes
      // four whole 128-byte rows (a key tile's rows are consecutive in dK /
      // dV: it never straddles the ring's wrap).
      {
        uint32_t ga[32], gb[32];
        tmem_ld32(trow + (hf ? TM_DK : TM_DV), ga);
        tmem_ld32(trow + (hf ? TM_DK : TM_DV) + 32, gb);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_acc);
        const float gs = hf ? 1.f : inv_scale;  // dV accumulated (scale P)^T dO
        auto f = [&](const uint32_t(&a)[32], int e) { return __uint_as_float(a[e]) * gs; };
        auto pack8 = [&](const uint32_t(&a)[32], int e) {
          return make_uint4(pack_bf16(f(a, 8 * e + 0), f(a, 8 * e + 1)), pack_bf16(f(a, 8 * e + 2), f(a, 8 * e + 3)),
                            pack_bf16(f(a, 8 * e + 4), f(a, 8 * e + 5)), pack_bf16(f(a, 8 * e + 6), f(a, 8 * e + 7)));
        };
        uint4 m[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          m[e] = pack8(ga, e);
          m[4 + e] = pack8(gb, e);
        }
#pragma unroll
        for (int sx = 4; sx >= 1; sx >>= 1) {
          const bool up = (lane & sx) != 0;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            if (cc & sx) continue;
            const uint4 snd = up ? m[cc] : m[cc + sx];
            uint4 rcv;
            rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, sx);
            rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, sx);
            rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, sx);
            rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, sx);
            if (up)
              m[cc] = rcv;
            else
              m[cc + sx] = rcv;
          }
        }
        const int r0 = quad * 32 + 8 * (lane >> 3);  // the lane group's first row of the tile
        uint4 *out = (uint4 *)((hf ? p.dk : p.dv) + ((size_t)it.bh * p.kv_rows + it.x.phys0 + r0) * DH) + (lane & 7);
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (r0 + t < it.x.nvalid) out[t * (DH / 8)] = m[t];
        // column sums of dQp over the warp's 32 rows (recursive halving):
        // afterwards lane l holds column 32*hf + l
#pragma unroll
        for (int h2 = 16; h2 >= 1; h2 >>= 1) {
          const bool upper = (lane & h2) != 0;
          if (h2 == 1) {
            const float send = upper ? dva[0] : dva[1];
            const float keep = upper ? dva[1] : dva[0];
            dva[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
          } else {
#pragma unroll
            for (int k = 0; k < h2; k += 2) {  // pairs of columns through the packed add
              const float s0 = upper ? dva[k] : dva[k + h2], s1 = upper ? dva[k + 1] : dva[k + 1 + h2];
              const float k0 = upper ? dva[k + h2] : dva[k], k1 = upper ? dva[k + 1 + h2] : dva[k + 1];
              const float2 t = __fadd2_rn(make_float2(k0, k1),
                                          make_float2(__shfl_xor_sync(0xffffffffu, s0, h2),
                                                      __shfl_xor_sync(0xffffffffu, s1, h2)));
              dva[k] = t.x;
              dva[k + 1] = t.y;
            }
          }
        }
        atomicAdd(p.dvb + it.h * DH + 32 * hf + lane, dva[0]);
        atomicAdd(p.du + it.h * DH + 32 * hf + lane, -dva[0]);
#pragma unroll
        for (int e = 0; e < 32; ++e) dva[e] = 0.f;
      }
    }
    if (!ok) atomicExch(&g_bwd_error, 2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------- small kernels

// The dR and dQ accumulators and the du/dv outputs (sums of atomic adds) <-
// 0; dK/dV rows of ring slots that hold no valid memory <- 0; R16 <- fp16(R)
// (satfinite).
struct ZeroArgs {
  float *dr;
  size_t n_dr;
  float *dq_acc;
  size_t n_dq;
  float *du, *dvb;  // [H][64] each
  int n_hd;
  __nv_bfloat16 *dk, *dv;
  int BH, H, cap, m, head, kv_rows;
  const __nv_bfloat16 *r;
  __half *r16;
  size_t n_r;
  const int *mvis;
};

__device__ void zero_work(const ZeroArgs &z, size_t tid, size_t stride) {
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t e = tid; e < z.n_dr / 4; e += stride) ((float4 *)z.dr)[e] = z4;
  for (size_t e = tid; e < z.n_dq / 4; e += stride) ((float4 *)z.dq_acc)[e] = z4;
  for (size_t e = tid; e < (size_t)z.n_hd; e += stride) {
    z.du[e] = 0.f;
    z.dvb[e] = 0.f;
  }
  float rmax = 0.f;  // largest |R| converted by this thread
  for (size_t e = tid; e < z.n_r / 8; e += stride) {
    const uint4 a = ((const uint4 *)z.r)[e];
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t o[4];
#pragma unroll
    for (int f = 0; f < 4; ++f) {
      const float lo = __uint_as_float(w[f] << 16), hi = __uint_as_float(w[f] & 0xFFFF0000u);
      rmax = fmax3(rmax, fabsf(lo), fabsf(hi));
      o[f] = pack_f16(lo, hi);
    }
    ((uint4 *)z.r16)[e] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (__any_sync(0xffffffffu, rmax > 65504.f) && (threadIdx.x & 31) == 0) atomicOr(&g_bwd_range, 1);
  // ring slots whose rows the row does not see: logical slots t < m - mb
  // (masked by a document reset) and t >= m (no valid memory); 8 x 16 B per
  // row. Without a reset only t >= m: the walk covers those slots alone (none
  // when the ring is full)
  const int t_lo = z.mvis ? 0 : z.m, n_t = z.cap - t_lo;
  if (n_t <= 0) return;
  const size_t n_rows = (size_t)z.BH * n_t * 8;
  for (size_t e = tid; e < n_rows; e += stride) {
    const int c = (int)(e & 7);
    const size_t rr = e >> 3;
    const int bh = (int)(rr / n_t), t = t_lo + (int)(rr % n_t);
    const int mb = row_memory(z.mvis, bh / z.H, z.m, z.cap, z.head).m;
    if (t >= z.m - mb && t < z.m) continue;
    int pr = z.head + t;
    if (pr >= z.cap) pr -= z.cap;
    const size_t off = ((size_t)bh * z.kv_rows + pr) * DH;
    ((uint4 *)(z.dk + off))[c] = make_uint4(0, 0, 0, 0);
    ((uint4 *)(z.dv + off))[c] = make_uint4(0, 0, 0, 0);
  }
}

__global__ void bwd_zero_kernel(const ZeroArgs z) {
  griddep_wait();
  griddep_launch_dependents();
  zero_work(z, blockIdx.x * (size_t)blockDim.x + threadIdx.x, (size_t)gridDim.x * blockDim.x);
}

// Streaming preparation when the forward kept the low part of O: per row,
// (Q+u) in bf16, (Q+v) in fp16 and D_i = dO_i . (o_i + o_lo_i), eight
// threads per row, 16 bytes each; then the zeroing above, in the same launch.
__global__ void __launch_bounds__(256) bwd_light_prep_kernel(
    const ZeroArgs z, long long rows, int L, int H, const __nv_bfloat16 *__restrict__ q,
    const __nv_bfloat16 *__restrict__ u, const __nv_bfloat16 *__restrict__ vb,
    const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ o_lo,
    const __nv_bfloat16 *__restrict__ dout, __nv_bfloat16 *__restrict__ qu,
    __half *__restrict__ qv, float *__restrict__ delta) {
  griddep_wait();
  griddep_launch_dependents();
  const int sub = threadIdx.x & 7;
  float qvmax = 0.f;  // largest |q + v| converted to fp16 by this thread
  for (long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 3; row < rows;
       row += ((long long)gridDim.x * blockDim.x) >> 3) {
    // the row's head (32-bit division whenever the row count allows)
    const int h = rows < (1ll << 32) ? (int)(((unsigned)row / (unsigned)L) % (unsigned)H) : (int)((row / L) % H);
    const size_t off = (size_t)row * DH;
    const uint4 q4 = ((const uint4 *)(q + off))[sub];
    const uint4 u4 = ((const uint4 *)(u + (size_t)h * DH))[sub];
    const uint4 v4 = ((const uint4 *)(vb + (size_t)h * DH))[sub];
    const uint4 o4 = ((const uint4 *)(o + off))[sub];
    const uint4 l4 = ((const uint4 *)(o_lo + off))[sub];
    const uint4 d4 = ((const uint4 *)(dout + off))[sub];
    const uint32_t qw[4] = {q4.x, q4.y, q4.z, q4.w}, uw[4] = {u4.x, u4.y, u4.z, u4.w};
    const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w}, ow[4] = {o4.x, o4.y, o4.z, o4.w};
    const uint32_t lw[4] = {l4.x, l4.y, l4.z, l4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
    auto lo = [](uint32_t x) { return __uint_as_float(x << 16); };
    auto hi = [](uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); };
    uint32_t a[4], b[4];
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a[e] = pack_bf16(lo(qw[e]) + lo(uw[e]), hi(qw[e]) + hi(uw[e]));
      const float v0 = lo(qw[e]) + lo(vw[e]), v1 = hi(qw[e]) + hi(vw[e]);
      qvmax = fmax3(qvmax, fabsf(v0), fabsf(v1));
      b[e] = pack_f16(v0, v1);
      acc += lo(dw[e]) * (lo(ow[e]) + lo(lw[e])) + hi(dw[e]) * (hi(ow[e]) + hi(lw[e]));
    }
    ((uint4 *)(qu + off))[sub] = make_uint4(a[0], a[1], a[2], a[3]);
    ((uint4 *)(qv + off))[sub] = make_uint4(b[0], b[1], b[2], b[3]);
    // the row's 8 lanes (a warp's last rows may leave other groups outside
    // the loop, so the mask names this group only)
    const unsigned group = 0xFFu << (threadIdx.x & 24);
#pragma unroll
    for (int w = 4; w > 0; w >>= 1) acc += __shfl_xor_sync(group, acc, w);
    if (sub == 0) delta[row] = acc;
  }
  if (__any_sync(0xffffffffu, qvmax > 65504.f) && (threadIdx.x & 31) == 0) atomicOr(&g_bwd_range, 1);
  zero_work(z, blockIdx.x * (size_t)blockDim.x + threadIdx.x, (size_t)gridDim.x * blockDim.x);
}

// dq = bf16(dQ accumulator); the per-head column sums of dQ are added into
// du (which the main kernel's atomics already hold -dv in), and the dR rows
// are copied out of the padded accumulator. Block (bh, chunk) covers 128 rows
// of one (b, h) plane: 8 threads per row, 8 columns each. No block waits on
// another: every load is issued first, then the stores and the atomics.
__global__ void __launch_bounds__(256) bwd_dq_finish_kernel(
    const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dq, float *du,
    const float *__restrict__ dr_acc, float *__restrict__ dr, int L, int H, int kv_rows, int chunks) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float part[8][64];  // column sums of each warp's rows
  const int bh = blockIdx.x / chunks, ch = blockIdx.x % chunks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = threadIdx.x & 7, slot = threadIdx.x >> 3;
  const int r_end = min(L, (ch + 1) * 128);
  // the thread's four rows (slot, slot + 32, ..): all loads in flight first
  float4 a[4], b[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int i = ch * 128 + slot + 32 * t;
    a[t] = b[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < r_end) {
      const size_t off = ((size_t)bh * L + i) * DH + 8 * sub;
      a[t] = *(const float4 *)(dq_acc + off);
      b[t] = *(const float4 *)(dq_acc + off + 4);
    }
  }
  {
    // the block's share of the dR rows (16-byte chunks past the padding)
    const size_t per_h = (size_t)kv_rows * (DH / 4), n = (size_t)H * per_h;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
      const size_t h = e / per_h, o = e - h * per_h;
      ((float4 *)dr)[e] = ((const float4 *)(dr_acc + (h * (kv_rows + kDrPad) + kDrPad) * DH))[o];
    }
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int i = ch * 128 + slot + 32 * t;
    acc[0] += a[t].x; acc[1] += a[t].y; acc[2] += a[t].z; acc[3] += a[t].w;
    acc[4] += b[t].x; acc[5] += b[t].y; acc[6] += b[t].z; acc[7] += b[t].w;
    if (i < r_end) {
      const size_t off = ((size_t)bh * L + i) * DH + 8 * sub;
      *(uint4 *)(dq + off) = make_uint4(pack_bf16(a[t].x, a[t].y), pack_bf16(a[t].z, a[t].w),
                                        pack_bf16(b[t].x, b[t].y), pack_bf16(b[t].z, b[t].w));
    }
  }
  // lanes l, l+8, l+16, l+24 hold the same 8 columns: fold them, then the
  // warps' partials through shared memory
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 8);
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
  }
  if (lane < 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) part[warp][8 * lane + e] = acc[e];
  }
  __syncthreads();
  if (threadIdx.x < 64) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += part[w][threadIdx.x];
    atomicAdd(du + (bh % H) * DH + threadIdx.x, sum);
  }
}

// ------------------------------------------------------------------ host side

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

bool make_map(CUtensorMap *m, const void *base, int planes, int rows, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {128, (cuuint64_t)rows * 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [planes][rows][64] with 32-row x 32-column boxes, 128-byte swizzle
// (the reduction targets of the main kernel).
bool make_map_f32(CUtensorMap *m, const void *base, int planes, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {256, (cuuint64_t)rows * 256};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// Workspace: D [rows] f32 | (Q+u) [rows][64] bf16 | (Q+v) [rows][64] fp16 |
// R fp16 [H][kv_rows][64] | dQ accumulator [rows][64] f32 |
// dR accumulator [H][kDrPad + kv_rows][64] f32
BwdWorkspace tc_bwd_workspace(const AttnShape &s) {
  const size_t rows = (size_t)s.B * s.H * s.L;
  BwdWorkspace w;
  w.d_off = 0;
  w.dqu_off = up256(rows * 4);
  w.dqv_off = w.dqu_off + up256(rows * DH * 2);
  const size_t r16_off = w.dqv_off + up256(rows * DH * 2);
  const size_t dq_off = r16_off + up256((size_t)s.H * s.kv_rows * DH * 2);
  const size_t dr_off = dq_off + up256(rows * DH * 4);
  w.total = dr_off + up256((size_t)s.H * (kDrPad + s.kv_rows) * DH * 4);
  return w;
}

cudaError_t launch_tc_bwd(const AttnShape &s, const void *q, const void *k, const void *v,
                          const void *r, const void *u, const void *vb, const void *o,
                          const void *o_lo, const float *lse,
                          const void *dout, void *dq, void *dk, void *dv, float *dr, float *du,
                          float *dvb, void *ws, cudaStream_t st, int *launches) {
  const BwdWorkspace w = tc_bwd_workspace(s);
  const size_t rows = (size_t)s.B * s.H * s.L;
  float *delta = (float *)((char *)ws + w.d_off);
  void *qu = (char *)ws + w.dqu_off;
  void *qv = (char *)ws + w.dqv_off;
  const size_t r16_off = w.dqv_off + up256(rows * DH * 2);
  __half *r16 = (__half *)((char *)ws + r16_off);
  const size_t dq_off = r16_off + up256((size_t)s.H * s.kv_rows * DH * 2);
  float *dq_acc = (float *)((char *)ws + dq_off);
  float *dr_acc = (float *)((char *)ws + dq_off + up256(rows * DH * 4));
  const size_t n_dr_acc = (size_t)s.H * (kDrPad + s.kv_rows) * DH;
  const int nq = (s.L + BQ - 1) / BQ;

  CUtensorMap tk, tv, tr16, tqu, tqv, tdo, tdq, tdr;
  if (!make_map(&tk, k, s.B * s.H, s.kv_rows, BK) || !make_map(&tv, v, s.B * s.H, s.kv_rows, BK) ||
      !make_map(&tr16, r16, s.H, s.kv_rows, 128) || !make_map(&tqu, qu, s.B * s.H, s.L, BQ) ||
      !make_map(&tqv, qv, s.B * s.H, s.L, BQ) || !make_map(&tdo, dout, s.B * s.H, s.L, BQ) ||
      !make_map_f32(&tdq, dq_acc, s.B * s.H, s.L) ||
      !make_map_f32(&tdr, dr_acc, s.H, kDrPad + s.kv_rows))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(rxl_bwd_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    F_SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;

  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  ZeroArgs z;
  z.dr = dr_acc; z.n_dr = n_dr_acc; z.dq_acc = dq_acc; z.n_dq = rows * DH;
  z.du = du; z.dvb = dvb; z.n_hd = s.H * DH;
  z.dk = (__nv_bfloat16 *)dk; z.dv = (__nv_bfloat16 *)dv;
  z.BH = s.B * s.H; z.H = s.H; z.cap = s.cap; z.m = s.m; z.head = s.head; z.kv_rows = s.kv_rows;
  z.r = (const __nv_bfloat16 *)r; z.r16 = r16; z.n_r = (size_t)s.H * s.kv_rows * DH;
  z.mvis = s.mvis;
  const int prep_slot = timing_begin(2, st);
  if (o_lo) {
    long long blocks = ((long long)rows * 8 + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    if (blocks < (long long)sms * 4) blocks = (long long)sms * 4;  // enough for the zeroing
    const cudaError_t e = launch_ex(
        bwd_light_prep_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, z, (long long)rows, s.L, s.H,
        (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)u, (const __nv_bfloat16 *)vb, (const __nv_bfloat16 *)o,
        (const __nv_bfloat16 *)o_lo, (const __nv_bfloat16 *)dout, (__nv_bfloat16 *)qu, (__half *)qv, delta);
    ++*launches;
    if (e != cudaSuccess) {
      timing_end(2, prep_slot, st);
      return e;
    }
  } else {
    cudaError_t e = launch_ex(bwd_zero_kernel, dim3((unsigned)(sms * 4)), dim3(256), 0, st, 1, z);
    ++*launches;
    if (e != cudaSuccess) {
      timing_end(2, prep_slot, st);
      return e;
    }
    e = launch_tc_bwd_prep(s, q, k, v, r, u, vb, dout, delta, qu, qv, st, launches);
    if (e != cudaSuccess) {
      timing_end(2, prep_slot, st);
      return e;
    }
  }
  timing_end(2, prep_slot, st);

  BwdParams p;
  p.B = s.B; p.H = s.H; p.L = s.L; p.cap = s.cap; p.m = s.m; p.head = s.head; p.nq = nq;
  p.kv_rows = s.kv_rows;
  p.mvis = s.mvis;
  p.fd_bh.init((uint32_t)(s.B * s.H));
  p.fd_h.init((uint32_t)s.H);
  {
    // key tiles per (b,h): ring runs A and B, then the current rows
    const int lenA = s.m < s.cap - s.head ? s.m : s.cap - s.head;
    const int lenB = s.m - lenA;
    const int nkt = (lenA + BK - 1) / BK + (lenB + BK - 1) / BK + (s.L + BK - 1) / BK;
    p.nitems = s.B * s.H * nkt;
  }
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.lse = lse; p.delta = delta;
  p.dk = (__nv_bfloat16 *)dk; p.dv = (__nv_bfloat16 *)dv;
  p.du = du; p.dvb = dvb;
  const unsigned grid = (unsigned)(p.nitems < sms ? p.nitems : sms);
  const int slot = timing_begin(1, st);
  cudaError_t e = launch_ex(rxl_bwd_main_kernel, dim3(grid), dim3(kThreads), F_SMEM, st, 1, tk, tv, tr16, tqu, tqv,
                            tdo, tdq, tdr, p);
  timing_end(1, slot, st);
  ++*launches;
  if (e != cudaSuccess) return e;
  const int chunks = (s.L + 127) / 128;
  const int fin_slot = timing_begin(3, st);
  e = launch_ex(bwd_dq_finish_kernel, dim3((unsigned)(s.B * s.H * chunks)), dim3(256), 0, st, 1,
                (const float *)dq_acc, (__nv_bfloat16 *)dq, du, (const float *)dr_acc, dr, s.L, s.H,
                s.kv_rows, chunks);
  timing_end(3, fin_slot, st);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t tc_bwd_read_range(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_bwd_range, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bwd_range, &zero, sizeof(int));
  return e;
}

cudaError_t tc_bwd_read_error(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_bwd_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof(int));
  return e;
}

}  // namespace rxl
