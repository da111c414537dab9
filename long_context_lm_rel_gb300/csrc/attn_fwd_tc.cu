// Fused relative-position memory attention forward on sm_103a tensor cores.
//
// Math (Transformer-XL page, "Relative Positional Encoding", "Dimension
// Walkthrough", "Causal Mask With Memory"):
//   A_ij = (q_i+u).k_j + (q_i+v).r_{i-j},  O_i = softmax_j(scale*A_ij | allow) V
// The L x (m+L) score matrix never leaves the SM.
//
// One CTA owns (b, h, 128 query rows). It walks the visible keys in tiles of
// 128 physically contiguous K/V rows (the ring's two runs and the current
// block; a tile never straddles the ring's wrap). For every key tile:
//   * TMA loads K, V (128 x 64) and the band of 256 R rows the tile needs:
//     distances d0 .. d0+255 with d0 = i0 - j0 - 127 (rows outside R read as
//     zero and are masked anyway);
//   * tcgen05: S = (Q+u) K^T   -> TMEM cols [0,128)     (M=128, N=128)
//              G = (Q+v) Rb^T  -> TMEM cols [128,384)   (M=128, N=256)
//     so G[ii][t] = (q_ii+v).r_{d0+t}; the relative shift the pages do by
//     pad/reshape/slice is an index skew here: S_p[ii][jj] = G[ii][ii-jj+127];
//     (Q+u) and (Q+v) are stored prescaled by scale*log2(e), so S + S_p is
//     already the base-2 logit;
//   * 8 softmax warps, two per TMEM lane quadrant: the thread of (row ii,
//     half hf) handles keys 64*hf .. 64*hf+63 of row ii. It loads S and its
//     skewed G window, masks, and runs the fp32 online softmax (exp2) over
//     its half on its own: each half keeps its own exponent reference, sum
//     and O accumulator, so the two warps of a row never wait on each other
//     within an item. P goes to shared memory (bf16). A half's running
//     maximum, used as its exponent reference, only moves when the half's
//     max grows by more than 2^8 (then its O is rescaled in TMEM), so
//     P <= 256;
//   * tcgen05: O_h += P_h V_h -> TMEM cols [384,448), [448,512) for the key
//     halves h (M=128, N=64, K=64 each); the epilogue combines the halves
//     with their references (one exchange through shared memory per item)
//     and writes O (and its low part) by per-warp TMA stores staged in the
//     free P buffer
// Warp 8 is the producer: the whole warp runs the schedule and one elected
// thread issues each TMA load (two stages ahead, across items) and each MMA;
// tcgen05.commit signals completion through mbarriers.
//
// Few items (at most half as many as SMs: short segments, few heads): the
// kernel runs as clusters of two CTAs per item instead of persistently, each
// CTA over half of the item's key tiles. Rank 1 hands its O (fp32,
// relative to its own reference), reference and sum to rank 0 through
// distributed shared memory once rank 0 has finished with its K/V stages;
// rank 0 merges the two and writes the output. Every cross-CTA wait is a
// bounded mbarrier wait. All waits here probe inline once and poll out of
// line (mbar_wait_lean): the smaller code fetches faster.
//
// The skew: thread of row ii = 32*quad + lane needs G columns ii..ii+127. For
// its 64 keys it loads one warp-uniform 96-column window and shifts it by its
// lane with a 5-stage predicated barrel shift.
#include <math.h>
#include <stdio.h>

#include <cstring>
#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace rxl {
namespace {

using namespace sm103;
using tc::BQ;
using tc::BK;
using tc::DH;
using tc::NB;
using tc::KeyTile;
using tc::KeyTiles;
using tc::RowMemory;
using tc::lane_shift_window96;
using tc::row_memory;
using tc::FastDiv;

constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarps + 1) * 32;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr uint32_t SM_QU = 0;                  // [128][64] bf16, sw128
constexpr uint32_t SM_QV = 16384;
constexpr uint32_t SM_K = 32768;               // 2 stages x 16 KB
constexpr uint32_t SM_V = 65536;               // 2 stages x 16 KB
constexpr uint32_t SM_R = 98304;               // 2 stages x 32 KB
constexpr uint32_t SM_P = 163840;              // 2 x [128][64] bf16 (keys 0-63, 64-127)
constexpr uint32_t SM_BAR = 196608;            // mbarriers, TMEM slot, abort flag
constexpr uint32_t SM_X = SM_BAR + 256;        // row-half exchange: [2][2][128] floats
constexpr uint32_t SM_QRAW = 199680;           // the next item's Q rows [128][64] bf16 (TMA, sw128)
constexpr uint32_t SM_UV = SM_QRAW + 16384;     // and its head's u and v rows (2 x 128 B)
constexpr uint32_t SMEM_BYTES = SM_UV + 256 + 1024;  // + alignment slack
constexpr float kRescaleThreshold = 8.f;       // log2 units
// O accumulators: keys 0-63 of every tile into TM_O, keys 64-127 into TM_O + 64
constexpr uint32_t TM_S = 0, TM_G = 128, TM_O = 384, TM_COLS = 512;

constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_G = idesc_bf16(128, 256, false, false);
constexpr uint32_t IDESC_O = idesc_bf16(128, 64, false, true);   // V is MN-major (d contiguous)

__device__ int g_fwd_error;
// set when the backward preparation mode converted a (q + v) element beyond
// the fp16 range (clamped)
__device__ int g_fwd_range;
// Testing hook (tc_fwd_test_hooks): non-zero makes the softmax warps withhold
// their arrival on bar_qready for the CTA's first item.
__device__ int g_fwd_withhold;

struct Params {
  int B, H, L, cap, m, head, nq;
  float scale_log2;  // scale * log2(e)
  const __nv_bfloat16 *q, *u, *vb;
  __nv_bfloat16 *o;
  __nv_bfloat16 *o_lo;  // optional: O - bf16(O), rounded to bf16 (exact D in the backward)
  float *lse;
  // backward preparation (kPrep): dO in, D = dO.O (fp32 O) and the bf16
  // (Q+u), (Q+v) rows (unscaled) out
  const __nv_bfloat16 *dout;
  float *delta;
  __nv_bfloat16 *qu_out;
  __half *qv_out;  // (Q+v) rows in fp16 for the backward's position products
  const int *mvis;  // per-row document reset (nullable): newest memory rows per batch row
  FastDiv fd_bh, fd_h;  // division by B*H and by H
};

constexpr int kFwd = 0, kPrep = 1;

// Exchange of one float per row between the two warps of a lane quadrant
// (bounded wait): returns the partner's value.
__device__ __forceinline__ bool pair_exchange(float mine, float *out, volatile float *xbuf,
                                              uint32_t bar, int hf, int ii, int lane,
                                              uint32_t &phase, volatile int *abort_flag) {
  volatile float *slot = xbuf + (phase & 1) * 256;
  slot[hf * 128 + ii] = mine;
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait_lean(bar, phase & 1, abort_flag));
  ++phase;
  *out = slot[(1 - hf) * 128 + ii];
  return ok;
}

// A work item is one (b, h, 128-query tile). Items are numbered so that the
// longest query tiles (most keys) come first. CTA c of G takes one item per
// round r, in snake order: item r*G + c on even rounds, r*G + G-1-c on odd
// ones, so that the CTAs' total key-tile counts stay within about one tile.
struct Item {
  int bh, h, i0, T;
  int m, head;  // the memory this batch row sees (all of it unless reset)
};

template <bool RESET>
__device__ __forceinline__ Item item_at(const Params &p, int w) {
  Item it;
  const uint32_t t = p.fd_bh.div((uint32_t)w);  // w = t * B*H + bh
  it.bh = w - (int)(t * p.fd_bh.d);
  const uint32_t b = p.fd_h.div((uint32_t)it.bh);
  it.h = it.bh - (int)(b * p.fd_h.d);
  it.i0 = (p.nq - 1 - (int)t) * BQ;
  if (RESET) {
    const RowMemory rm = row_memory(p.mvis, (int)b, p.m, p.cap, p.head);
    it.m = rm.m;
    it.head = rm.head;
  } else {
    it.m = p.m;
    it.head = p.head;
  }
  it.T = KeyTiles(it.m, p.cap, it.head, min(it.i0 + BQ, p.L)).count();
  return it;
}

// Walks this CTA's tiles across its items: k counts the CTA's items, t the
// key tiles of the current item, which this CTA takes from t0 up to t1.
// SPLIT: a cluster of two CTAs per item, the first (rank 0) taking the first
// half of its key tiles, rank 1 the rest; one item per cluster.
template <bool RESET, bool SPLIT>
struct Cursor {
  int k, w, t, t0, t1, nitems;
  bool valid;
  Item it;
  __device__ __forceinline__ int item_of_round(int r) const {
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((r & 1) ? G - 1 - c : c);
  }
  __device__ void init(const Params &p, int n) {
    nitems = n;
    k = 0;
    w = SPLIT ? (int)(blockIdx.x >> 1) : item_of_round(0);
    valid = w < nitems;
    if (!valid) return;
    it = item_at<RESET>(p, w);
    t0 = 0;
    t1 = it.T;
    if (SPLIT) {
      const int half = (it.T + 1) >> 1;
      if (blockIdx.x & 1) t0 = half; else t1 = half;
      valid = t0 < t1;
    }
    t = t0;
  }
  __device__ void next(const Params &p) {
    if (++t == t1) {
      if (SPLIT) {
        valid = false;
        return;
      }
      t = 0;
      ++k;
      w = item_of_round(k);
      valid = w < nitems;
      if (valid) {
        it = item_at<RESET>(p, w);
        t0 = 0;
        t1 = it.T;
      }
    }
  }
};

// (Q+u)*c and (Q+v)*c in bf16, c = scale*log2(e), as 128-byte swizzled
// K-major tiles for the item's query rows, from the raw Q tile the producer
// loaded ahead; the row's two warps split its 8 chunks. In kPrep mode the unscaled rows also go to global memory ((Q+v) in fp16).
template <int MODE>
__device__ __forceinline__ void q_prep(const Params &p, const Item &it, uint32_t sbase, int quad,
                                       int hf, int lane) {
  const int ii = quad * 32 + lane;
  const int i = it.i0 + ii;
  const float c2 = p.scale_log2;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * hf + cc;
    // the raw Q rows were loaded by TMA (rows past L read as zero), the
    // head's u and v rows with them
    uint4 qv4;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(qv4.x), "=r"(qv4.y), "=r"(qv4.z), "=r"(qv4.w)
                 : "r"(sbase + SM_QRAW + sw128_offset(ii, c)));
    const uint4 u4 = ld_shared_v4(sbase + SM_UV + 16 * c), v4 = ld_shared_v4(sbase + SM_UV + 128 + 16 * c);
    const uint32_t qw[4] = {qv4.x, qv4.y, qv4.z, qv4.w};
    const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
    const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w};
    uint32_t a[4], b[4], a1[4], b1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float q0 = __uint_as_float(qw[e] << 16), q1 = __uint_as_float(qw[e] & 0xFFFF0000u);
      const float u0 = __uint_as_float(uw[e] << 16), u1 = __uint_as_float(uw[e] & 0xFFFF0000u);
      const float v0 = __uint_as_float(vw[e] << 16), v1 = __uint_as_float(vw[e] & 0xFFFF0000u);
      a[e] = pack_bf16((q0 + u0) * c2, (q1 + u1) * c2);
      b[e] = pack_bf16((q0 + v0) * c2, (q1 + v1) * c2);
      a1[e] = pack_bf16(q0 + u0, q1 + u1);
      b1[e] = pack_f16(q0 + v0, q1 + v1);
      if (MODE == kPrep && fmaxf(fabsf(q0 + v0), fabsf(q1 + v1)) > 65504.f) atomicOr(&g_fwd_range, 1);
    }
    st_shared_v4(sbase + SM_QU + sw128_offset(ii, c), a[0], a[1], a[2], a[3]);
    st_shared_v4(sbase + SM_QV + sw128_offset(ii, c), b[0], b[1], b[2], b[3]);
    if (MODE == kPrep && i < p.L) {
      const size_t off = ((size_t)it.bh * p.L + i) * DH;
      ((uint4 *)(p.qu_out + off))[c] = make_uint4(a1[0], a1[1], a1[2], a1[3]);
      ((uint4 *)(p.qv_out + off))[c] = make_uint4(b1[0], b1[1], b1[2], b1[3]);
    }
  }
}

// Persistent kernel: gridDim.x CTAs walk all work items. Per CTA, tiles are
// numbered g = 0, 1, ... across its items; every barrier phase follows g
// (tile barriers) or the item counter k (q_ready, o_free).
template <int MODE, bool RESET, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
rxl_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_olo,
                  const Params p, int nitems) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = tc::align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t b0 = sbase + SM_BAR;
  // TMA per stage: K and R of a tile (bar_kr*), its V (bar_v*)
  const uint32_t bar_kr0 = b0, bar_kr1 = b0 + 8, bar_v0 = b0 + 152, bar_v1 = b0 + 160;
  const uint32_t bar_sg = b0 + 16;       // S/G MMAs of a tile done (commit)
  const uint32_t bar_sgfree = b0 + 24;   // softmax finished reading S/G of a tile (256)
  const uint32_t bar_pr = b0 + 32;       // softmax finished a tile: P written (256)
  const uint32_t bar_pv = b0 + 40;       // P.V of a tile done (commit)
  const uint32_t bar_qready = b0 + 48;   // Q tiles of an item written (256)
  const uint32_t bar_ofree = b0 + 56;    // epilogue of an item read O (256)
  const uint32_t bar_drain = b0 + 64;
  const uint32_t bar_x0 = b0 + 72;       // 4 quadrant exchange barriers
  // SPLIT: rank 0's K/V stages are free for rank 1's half (rank 1, count 1);
  // rank 1's half has landed in them (rank 0, count 1 + the copy's bytes);
  // rank 1's softmax warps staged their part in its own stages (rank 1, 256)
  const uint32_t bar_peer = b0 + 112, bar_data = b0 + 120, bar_staged = b0 + 136;
  const uint32_t bar_q = b0 + 128;  // TMA: the raw Q rows of the next item
  const uint32_t bar_gread = b0 + 144;   // softmax finished reading G of a tile (256)
  uint32_t *tmem_slot = (uint32_t *)(smem + SM_BAR + 104);
  volatile int *abort_flag = (volatile int *)(smem + SM_BAR + 108);
  volatile float *xbuf = (volatile float *)(smem + SM_X);

  if (threadIdx.x == 0) {
    mbar_init(bar_kr0, 1);
    mbar_init(bar_kr1, 1);
    mbar_init(bar_v0, 1);
    mbar_init(bar_v1, 1);
    mbar_init(bar_sg, 1);
    mbar_init(bar_sgfree, kSoftmaxWarps * 32);
    mbar_init(bar_gread, kSoftmaxWarps * 32);
    mbar_init(bar_pr, kSoftmaxWarps * 32);
    mbar_init(bar_pv, 1);
    mbar_init(bar_qready, kSoftmaxWarps * 32);
    mbar_init(bar_ofree, kSoftmaxWarps * 32);
    mbar_init(bar_drain, 1);
    mbar_init(bar_q, 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar_x0 + 8 * q, 2);
    if (SPLIT) {
      mbar_init(bar_peer, 1);
      mbar_init(bar_data, 1);
      mbar_init(bar_staged, kSoftmaxWarps * 32);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  // the peer CTA arrives on this CTA's barriers: they must be initialised first
  if (SPLIT) cluster_sync();
  if (warp == kProducerWarp) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_r);
      tma_prefetch_desc(&tm_q);
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
    // The whole warp runs the schedule (uniform control flow, so that the
    // descriptors stay in uniform registers); one elected thread issues.
    // Stage s of tile g = g & 1 holds its K and R (bar_kr{s}) and its V
    // (bar_v{s}): K and R are reloaded for tile g+2 as soon as the S/G
    // products of tile g are done, V once its P.V is, so each copy has about
    // two tiles of lead.
    {
      int n_kr0 = 0, n_kr1 = 0, n_v0 = 0, n_v1 = 0;  // copies issued per barrier
      Cursor<RESET, SPLIT> kc, vc;  // next tile whose K/R, whose V to load
      kc.init(p, nitems);
      vc.init(p, nitems);
      int g_kr = 0, g_v = 0;
      auto wait = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait_lean(bar, parity, abort_flag));
      };
      auto issue_kr = [&]() {
        const int s = g_kr & 1;
        const KeyTile x = KeyTiles(kc.it.m, p.cap, kc.it.head, min(kc.it.i0 + BQ, p.L)).get(kc.t);
        if (elect_one()) {
          const uint32_t bar = s ? bar_kr1 : bar_kr0;
          mbar_expect_tx(bar, 16384 + 32768);
          tma_load_3d(sbase + SM_K + s * 16384, &tm_k, 0, x.phys0, kc.it.bh, bar);
          tma_load_3d(sbase + SM_R + s * 32768, &tm_r, 0, kc.it.i0 - x.jlog0 - (BK - 1), kc.it.h, bar);
        }
        __syncwarp();
        if (s) ++n_kr1; else ++n_kr0;
        ++g_kr;
        kc.next(p);
      };
      auto issue_v = [&]() {
        const int s = g_v & 1;
        const KeyTile x = KeyTiles(vc.it.m, p.cap, vc.it.head, min(vc.it.i0 + BQ, p.L)).get(vc.t);
        if (elect_one()) {
          const uint32_t bar = s ? bar_v1 : bar_v0;
          mbar_expect_tx(bar, 16384);
          tma_load_3d(sbase + SM_V + s * 16384, &tm_v, 0, x.phys0, vc.it.bh, bar);
        }
        __syncwarp();
        if (s) ++n_v1; else ++n_v0;
        ++g_v;
        vc.next(p);
      };
      // operand descriptors, built once; a k-step or a stage is an add
      const uint64_t d_qu = sdesc_sw128(sbase + SM_QU, 16, 1024), d_qv = sdesc_sw128(sbase + SM_QV, 16, 1024);
      const uint64_t d_k = sdesc_sw128(sbase + SM_K, 16, 1024), d_r = sdesc_sw128(sbase + SM_R, 16, 1024);
      const uint64_t d_p = sdesc_sw128(sbase + SM_P, 16, 1024), d_v = sdesc_sw128(sbase + SM_V, 16, 1024);
      // G of a tile (two thirds of its S/G work) goes as soon as the softmax
      // has read the previous tile's G, while it still skews it; S once it
      // has read S; one commit covers both
      auto issue_g = [&](int g) {
        const uint64_t dr_s = sdesc_add(d_r, (g & 1) * 32768);
        if (elect_one()) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(tmem + TM_G, sdesc_add(d_qv, k * 32), sdesc_add(dr_s, k * 32), IDESC_G, k > 0);
        }
        __syncwarp();
      };
      auto issue_s_commit = [&](int g) {
        const uint64_t dk_s = sdesc_add(d_k, (g & 1) * 16384);
        if (elect_one()) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(tmem + TM_S, sdesc_add(d_qu, k * 32), sdesc_add(dk_s, k * 32), IDESC_S, k > 0);
          mma_commit(bar_sg);
        }
        __syncwarp();
      };
      auto wait_kr = [&](int g) { return wait((g & 1) ? bar_kr1 : bar_kr0, (g >> 1) & 1); };
      auto wait_v = [&](int g) { return wait((g & 1) ? bar_v1 : bar_v0, (g >> 1) & 1); };
      // the raw Q rows of this CTA's item k (round k of the item order)
      int nq_loads = 0;
      auto load_q = [&](int k) {
        int w;
        if (SPLIT) {
          if (k > 0) return;
          w = (int)(blockIdx.x >> 1);
        } else {
          const int G = gridDim.x, c = blockIdx.x;
          w = k * G + ((k & 1) ? G - 1 - c : c);
        }
        if (w >= nitems) return;
        const Item qi = item_at<RESET>(p, w);
        if (elect_one()) {
          mbar_expect_tx(bar_q, 16384 + 256);
          tma_load_3d(sbase + SM_QRAW, &tm_q, 0, qi.i0, qi.bh, bar_q);
          bulk_load(sbase + SM_UV, p.u + (size_t)qi.h * DH, 128, bar_q);
          bulk_load(sbase + SM_UV + 128, p.vb + (size_t)qi.h * DH, 128, bar_q);
        }
        __syncwarp();
        ++nq_loads;
      };
      bool ok = true;
      Cursor<RESET, SPLIT> mc;  // tile whose P.V is next
      mc.init(p, nitems);
      if (mc.valid) load_q(0);
      for (int t = 0; t < 2 && kc.valid; ++t) {
        issue_kr();
        issue_v();
      }
      // later V copies: the one of tile g+1 during tile g (g >= 1)
      if (mc.valid) {
        ok = wait(bar_qready, 0) && wait_kr(0);
        if (ok) {
          load_q(1);  // the softmax has read item 0's raw rows
          issue_g(0);
          issue_s_commit(0);
        }
      }
      for (int g = 0; ok && mc.valid; ++g) {
        Cursor<RESET, SPLIT> nx = mc;
        nx.next(p);
        const bool new_item = nx.valid && nx.t == nx.t0;
        // S/G of tile g+1 as soon as the softmax released S/G of tile g
        // (same item: the Q tiles are unchanged)
        if (nx.valid && !new_item) {
          if (!(ok = wait(bar_gread, g & 1) && wait_kr(g + 1))) break;
          issue_g(g + 1);
        }
        if (g > 0 && vc.valid) {
          // the V stage of tile g-1 is free once its P.V completed: tile g+1
          if (!(ok = wait(bar_pv, (g - 1) & 1))) break;
          issue_v();
        }
        if (nx.valid && !new_item) {
          if (!(ok = wait(bar_sgfree, g & 1))) break;
          issue_s_commit(g + 1);
          // the S/G products of tile g are done (the softmax has read them):
          // its K and R stage takes tile g+2
          if (kc.valid) issue_kr();
        }
        if (!(ok = wait(bar_pr, g & 1) && wait_v(g))) break;
        // the first P.V of an item overwrites O: its epilogue must have read it
        if (mc.t == mc.t0 && mc.k > 0 && !(ok = wait(bar_ofree, (mc.k - 1) & 1))) break;
        const int s = g & 1;
        const uint64_t dv_s = sdesc_add(d_v, s * 16384);
        const uint32_t acc0 = mc.t > mc.t0 ? 1u : 0u;
        if (elect_one()) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)  // O_h += P_h V_h for the key halves h = k / 4
            mma_bf16(tmem + TM_O + 64 * (k >> 2), sdesc_add(d_p, (k >> 2) * 16384 + (k & 3) * 32),
                     sdesc_add(dv_s, k * 2048), IDESC_O, ((k & 3) > 0) ? 1u : acc0);
          mma_commit(bar_pv);
        }
        __syncwarp();
        if (new_item) {
          // next item: its Q tiles are written once the softmax finished
          // this item's last tile; its S/G first, then the copies
          if (!(ok = wait(bar_sgfree, g & 1) && wait(bar_qready, nx.k & 1) && wait_kr(g + 1))) break;
          issue_g(g + 1);
          issue_s_commit(g + 1);
          load_q(nx.k + 1);  // the softmax has read item nx.k's raw rows
          if (kc.valid) issue_kr();  // tile g's S/G are done (read by the softmax)
        }
        mc = nx;
      }
      if (!ok) {
        // wind down: let in-flight copies and MMAs land before TMEM and
        // shared memory are released (the latest copy of each barrier; an
        // earlier one completed before it, and a completed phase returns at once)
        if (elect_one()) {
          volatile int no_abort = 0;
          if (n_kr0 > 0) mbar_wait_lean(bar_kr0, (n_kr0 - 1) & 1, &no_abort);
          if (n_kr1 > 0) mbar_wait_lean(bar_kr1, (n_kr1 - 1) & 1, &no_abort);
          if (n_v0 > 0) mbar_wait_lean(bar_v0, (n_v0 - 1) & 1, &no_abort);
          if (n_v1 > 0) mbar_wait_lean(bar_v1, (n_v1 - 1) & 1, &no_abort);
          if (nq_loads > 0) mbar_wait_lean(bar_q, (nq_loads - 1) & 1, &no_abort);
          mma_commit(bar_drain);
          mbar_wait_lean(bar_drain, 0, &no_abort);
          atomicExch(&g_fwd_error, 1);
        }
        __syncwarp();
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------- softmax warps
    const int quad = warp & 3, hf = warp >> 2;
    const int ii = quad * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t row_p = sw128_row(sbase + SM_P + hf * 16384, ii);  // row ii of P block hf
    const uint32_t bar_x = bar_x0 + 8 * quad;
    uint32_t xphase = 0;
    float m_run = -INFINITY, l_run = 0.f;  // l_run: this half's part of the row sum
    bool ok = true;
    Cursor<RESET, SPLIT> cur;
    cur.init(p, nitems);
    if (cur.valid) {
      ok = __all_sync(0xffffffffu, mbar_wait_lean(bar_q, 0, abort_flag));
      if (ok) {
        q_prep<MODE>(p, cur.it, sbase, quad, hf, lane);
        fence_proxy_async_smem();
        if (!*(volatile int *)&g_fwd_withhold) mbar_arrive(bar_qready);
      } else {
        cur.valid = false;
      }
    }
    for (int g = 0; cur.valid; ++g) {
      const Item it = cur.it;
      const int t = cur.t, t0 = cur.t0, t1 = cur.t1;
      const int i = it.i0 + ii;
      const int s = g & 1;
      ok = mbar_wait_lean(bar_sg, g & 1, abort_flag);
      // tcgen05.ld/st below are warp-collective: keep every decision warp-uniform
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      const KeyTile x = KeyTiles(it.m, p.cap, it.head, min(it.i0 + BQ, p.L)).get(t);
      float y[64];
      {
        // One 96-column window of G serves both 32-key chunks of this half:
        // chunk 2hf reads columns W .. W+63 and chunk 2hf+1 columns W-32 ..
        // W+31 (W = 32 quad + 96 - 64 hf). Shifted left by the lane, the
        // keys 32 c + k sit at win[63 - k] (c = 2hf) and win[31 - k] (2hf+1).
        float win[96];
        {
          uint32_t w0[32], w1[32], w2[32];
          const uint32_t gcol = TM_G + 32 * quad + 64 - 64 * hf;
          tmem_ld32(trow + gcol, w0);
          tmem_ld32(trow + gcol + 32, w1);
          tmem_ld32(trow + gcol + 64, w2);
          tmem_wait_ld();
          // done reading G: the next tile's G products may start
          tc_fence_before();
          mbar_arrive(bar_gread);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            win[e] = __uint_as_float(w0[e]);
            win[32 + e] = __uint_as_float(w1[e]);
            win[64 + e] = __uint_as_float(w2[e]);
          }
        }
        lane_shift_window96(win, lane);  // win[x] <- win[x + lane]
        uint32_t s0[32], s1[32];
        tmem_ld32(trow + TM_S + 64 * hf, s0);
        tmem_ld32(trow + TM_S + 64 * hf + 32, s1);
        tmem_wait_ld();
        // done reading S: the next tile's S products may start
        tc_fence_before();
        mbar_arrive(bar_sgfree);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 a0 = __fadd2_rn(make_float2(__uint_as_float(s0[k]), __uint_as_float(s0[k + 1])),
                                       make_float2(win[63 - k], win[62 - k]));
          const float2 a1 = __fadd2_rn(make_float2(__uint_as_float(s1[k]), __uint_as_float(s1[k + 1])),
                                       make_float2(win[31 - k], win[30 - k]));
          y[k] = a0.x;
          y[k + 1] = a0.y;
          y[32 + k] = a1.x;
          y[32 + k + 1] = a1.y;
        }
        // key jj = 32c + k is visible iff jj < nvalid and jlog0 + jj <= i;
        // the warp skips the mask where all 32 keys are visible to all its rows
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int lim = min(x.nvalid - 1, i - x.jlog0) - 32 * (2 * hf + cc);
          if (!__all_sync(0xffffffffu, lim >= 31)) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (k > lim) y[32 * cc + k] = -INFINITY;
          }
        }
      }
      float mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < 64; k += 2) mt = fmax3(mt, y[k], y[k + 1]);
      // this half's exponent reference only moves when its max outgrows it
      // by 2^8 (each half keeps its own reference, sum and O accumulator)
      const bool move = mt > m_run + kRescaleThreshold;
      const float m_new = move ? mt : m_run;
      const float ref = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = move ? ex2(m_run - ref) : 1.f;  // 0 on the first visible tile
      float2 sum2 = make_float2(0.f, 0.f);
      const float2 nref2 = make_float2(-ref, -ref);
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const float2 e = __fadd2_rn(make_float2(y[k], y[k + 1]), nref2);
        const float2 pp = make_float2(ex2(e.x), ex2(e.y));
        sum2 = __fadd2_rn(sum2, pp);
        pk[k / 2] = pack_bf16(pp.x, pp.y);
      }
      const float sum = sum2.x + sum2.y;
      l_run = l_run * alpha + sum;
      m_run = m_new;
      // the P buffer and O: P.V(g-1), which ran while this tile's logits
      // were formed, must be done
      if (g > 0) {
        ok = mbar_wait_lean(bar_pv, (g - 1) & 1, abort_flag);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();
      }
      // the warp's part of the P buffer held the previous item's O rows on
      // their way out
      if (MODE != kPrep && !SPLIT && t == t0 && cur.k > 0) {
        if (lane == 0) bulk_wait_read();
        __syncwarp();
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(sw128_at(row_p, c), pk[4 * c], pk[4 * c + 1],
                     pk[4 * c + 2], pk[4 * c + 3]);
      // rows of V past the run hold another run's (or junk) data: zero them
      // so that 0 * junk cannot leak into O (once the tile's V has landed)
      if (x.nvalid < BK) {
        ok = __all_sync(0xffffffffu, mbar_wait_lean(s ? bar_v1 : bar_v0, (g >> 1) & 1, abort_flag));
        if (!ok) break;
      }
      if (ii >= x.nvalid) {
        const uint32_t vrow = sbase + SM_V + s * 16384 + ii * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) st_shared_v4(vrow + 16 * (4 * hf + c), 0, 0, 0, 0);
      }
      if (__any_sync(0xffffffffu, t > t0 && alpha != 1.f)) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          tmem_ld32(trow + TM_O + 64 * hf + 32 * cc, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(trow + TM_O + 64 * hf + 32 * cc, o);
          tmem_wait_st();
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_pr);

      cur.next(p);
      if (t + 1 < t1) continue;
      // ---- last tile of the item: Q tiles of the next item, then epilogue
      if (cur.valid) {
        // the S/G MMAs of this item are all done (bar_sg waited above)
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_lean(bar_q, cur.k & 1, abort_flag)))) break;
        q_prep<MODE>(p, cur.it, sbase, quad, hf, lane);
        fence_proxy_async_smem();
        mbar_arrive(bar_qready);
      }
      ok = __all_sync(0xffffffffu, mbar_wait_lean(bar_pv, g & 1, abort_flag));
      // the two halves' references and sums; O_h and l_h are relative to
      // 2^(reference of half h), which is -inf for a half that saw no key
      float m_other = -INFINITY, l_other = 0.f;
      if (ok) ok = pair_exchange(m_run, &m_other, xbuf, bar_x, hf, ii, lane, xphase, abort_flag);
      if (ok) ok = pair_exchange(l_run, &l_other, xbuf, bar_x, hf, ii, lane, xphase, abort_flag);
      if (!ok) break;
      tc_fence_after();
      float m_row = fmaxf(m_run, m_other);
      const float a_own = m_run == -INFINITY ? 0.f : ex2(m_run - m_row);
      const float a_oth = m_other == -INFINITY ? 0.f : ex2(m_other - m_row);
      float l_row = l_run * a_own + l_other * a_oth;
      uint32_t o[32];
      {
        // this warp's 32 output columns: both halves' accumulators, scaled
        uint32_t o1[32];
        tmem_ld32(trow + TM_O + 32 * hf, o);
        tmem_ld32(trow + TM_O + 64 + 32 * hf, o1);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_ofree);
        const float a0 = hf ? a_oth : a_own, a1 = hf ? a_own : a_oth;
#pragma unroll
        for (int e = 0; e < 32; ++e)
          o[e] = __float_as_uint(__uint_as_float(o[e]) * a0 + __uint_as_float(o1[e]) * a1);
      }
      if (SPLIT) {
        // rank 1 hands its part of the item (O relative to 2^m_row, m_row,
        // l_row) to rank 0: it stages the O rows in its own K stages
        // ([128][64] fp32, 16-byte chunks swizzled by row) and m, l in its V
        // stage, then one thread moves the 33 KB into the same places of rank
        // 0 with one bulk copy over distributed shared memory (per-thread
        // remote stores took 2.1 us at the cfg5 shape); rank 0 merges the two
        const uint32_t orow = ii * 256 + hf * 128;
        constexpr uint32_t kHandBytes = 32768, kMlBytes = 1024;
        if (blockIdx.x & 1) {
          // this CTA's stages were last read by its final P.V (done above)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(sbase + SM_K + orow + ((c ^ (ii & 7)) << 4), o[4 * c], o[4 * c + 1], o[4 * c + 2],
                         o[4 * c + 3]);
          if (hf == 0) {
            *(volatile float *)(smem + SM_V + 4 * ii) = m_row;
            *(volatile float *)(smem + SM_V + 512 + 4 * ii) = l_row;
          }
          fence_proxy_async_smem();
          mbar_arrive(bar_staged);
          if (warp == 0) {
            if (lane == 0) {
              ok = mbar_wait_lean(bar_staged, 0, abort_flag) && mbar_wait_cluster(bar_peer, 0, abort_flag);
              if (ok) {
                const uint32_t bar0 = mapa_shared(bar_data, 0);
                bulk_copy_to_cluster(mapa_shared(sbase + SM_K, 0), sbase + SM_K, kHandBytes, bar0);
                bulk_copy_to_cluster(mapa_shared(sbase + SM_V, 0), sbase + SM_V, kMlBytes, bar0);
                bulk_commit();
                bulk_wait_read();  // the source stays valid until the copy has read it
              }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          }
          break;  // this CTA's only item is done
        }
        if (it.T >= 2) {  // rank 1 has tiles: its stages were read (P.V done above)
          if (threadIdx.x == 0) {
            mbar_expect_tx(bar_data, kHandBytes + kMlBytes);  // the arrival of this phase
            mbar_arrive_remote(mapa_shared(bar_peer, 1));
          }
          ok = __all_sync(0xffffffffu, mbar_wait_lean(bar_data, 0, abort_flag));
          if (!ok) break;
          const float m1 = *(volatile float *)(smem + SM_V + 4 * ii);
          const float l1 = *(volatile float *)(smem + SM_V + 512 + 4 * ii);
          const float mm = fmaxf(m_row, m1);
          const float as = m_row == -INFINITY ? 0.f : ex2(m_row - mm);
          const float ap = m1 == -INFINITY ? 0.f : ex2(m1 - mm);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t a, b, cc, d;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(a), "=r"(b), "=r"(cc), "=r"(d)
                         : "r"(sbase + SM_K + orow + ((c ^ (ii & 7)) << 4)));
            const uint32_t w[4] = {a, b, cc, d};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              o[4 * c + e] = __float_as_uint(__uint_as_float(o[4 * c + e]) * as + __uint_as_float(w[e]) * ap);
          }
          l_row = l_row * as + l1 * ap;
          m_row = mm;
        }
      }
      const float inv = 1.f / l_row;
      if (MODE == kPrep) {
        // D_i = dO_i . O_i with O_i still in fp32
        const uint4 *drow = (const uint4 *)(p.dout + ((size_t)it.bh * p.L + (i < p.L ? i : 0)) * DH);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 d4 = drow[4 * hf + e];
          const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int f = 0; f < 4; ++f)
            acc += __uint_as_float(o[8 * e + 2 * f]) * __uint_as_float(dw[f] << 16) +
                   __uint_as_float(o[8 * e + 2 * f + 1]) * __uint_as_float(dw[f] & 0xFFFF0000u);
        }
        float acc_other = 0.f;
        if (!(ok = pair_exchange(acc, &acc_other, xbuf, bar_x, hf, ii, lane, xphase, abort_flag))) break;
        if (hf == 0 && i < p.L) p.delta[(size_t)it.bh * p.L + i] = (acc + acc_other) * inv;
      } else {
        if (hf == 0 && i < p.L)
          p.lse[(size_t)it.bh * p.L + i] = (m_row + log2f(l_row)) * 0.69314718055994531f;
        // this thread's half row of O as four 16-byte chunks (and of the low
        // part), then a 4 x 4 transpose of chunks within each group of 4
        // lanes (two shuffle butterflies): lane 4k + r holds chunk r of the
        // group's rows 4k .. 4k+3, so that each store instruction writes
        // whole 32-byte sectors (64 contiguous bytes of 8 rows) instead of
        // 32 half sectors
        uint4 mh[4], ml[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float f[8];
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int g2 = 0; g2 < 8; ++g2) f[g2] = __uint_as_float(o[8 * e + g2]) * inv;
#pragma unroll
          for (int g2 = 0; g2 < 4; ++g2) {
            hi[g2] = pack_bf16(f[2 * g2], f[2 * g2 + 1]);
            // low part: what bf16 rounding of O dropped, itself in bf16
            lo[g2] = pack_bf16(f[2 * g2] - __uint_as_float(hi[g2] << 16),
                               f[2 * g2 + 1] - __uint_as_float(hi[g2] & 0xFFFF0000u));
          }
          mh[e] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          ml[e] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        if (SPLIT) {
          // one item per CTA (2-CTA clusters): a 4 x 4 transpose of 16-byte
          // chunks within each group of 4 lanes (two shuffle butterflies),
          // so that each store writes whole 32-byte sectors; here the TMA
          // stores below came out slower (their issue waits on the busy TMA
          // engine and nothing follows to hide it)
          auto xchg = [&](uint4 &a, uint4 &b, bool up, int sx) {  // up: send a, receive into a
            const uint4 snd = up ? a : b;
            uint4 rcv;
            rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, sx);
            rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, sx);
            rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, sx);
            rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, sx);
            if (up)
              a = rcv;
            else
              b = rcv;
          };
#pragma unroll
          for (int sx = 2; sx >= 1; sx >>= 1) {
            const bool up = (lane & sx) != 0;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              if (cc & sx) continue;
              xchg(mh[cc], mh[cc + sx], up, sx);
              if (p.o_lo) xchg(ml[cc], ml[cc + sx], up, sx);
            }
          }
          const int r0 = it.i0 + quad * 32 + 4 * (lane >> 2);  // the lane group's first row
          const size_t c0 = ((size_t)it.bh * p.L + r0) * (DH / 8) + 4 * hf + (lane & 3);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (r0 + t < p.L) {
              ((uint4 *)p.o)[c0 + t * (DH / 8)] = mh[t];
              if (p.o_lo) ((uint4 *)p.o_lo)[c0 + t * (DH / 8)] = ml[t];
            }
          }
        } else {
          // this warp's 32 rows x 32 columns of O (and of its low part) leave
          // by TMA stores from the warp's own 4 KB of the P buffer (the last
          // P.V has read P): 64-byte swizzled boxes, 2 KB each, so that the
          // row-per-thread staging stores hit every bank; rows past L are
          // clipped by the copy. The warp's next P store waits for the copies
          // to have read the box.
          const uint32_t obox = sbase + SM_P + hf * 16384 + quad * 4096;
          const uint32_t orow = obox + lane * 64;
          const int osw = (lane >> 1) & 3;  // 64-byte swizzle: chunk ^= (row >> 1) & 3
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            st_shared_v4(orow + ((e ^ osw) << 4), mh[e].x, mh[e].y, mh[e].z, mh[e].w);
            if (p.o_lo) st_shared_v4(orow + 2048 + ((e ^ osw) << 4), ml[e].x, ml[e].y, ml[e].z, ml[e].w);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && it.i0 + 32 * quad < p.L) {
            tma_store_3d(&tm_o, 32 * hf, it.i0 + 32 * quad, it.bh, obox);
            if (p.o_lo) tma_store_3d(&tm_olo, 32 * hf, it.i0 + 32 * quad, it.bh, obox + 2048);
            bulk_commit();
          }
        }
      }
      m_run = -INFINITY;
      l_run = 0.f;
    }
    // the O stores must have completed before shared memory goes away
    if (MODE != kPrep && !SPLIT) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
    if (!ok) atomicExch(&g_fwd_error, 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp) tmem_dealloc(tmem, TM_COLS);
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

// [planes][rows][64] bf16 output tensor, 32 x 32 boxes, 64-byte swizzle (the
// O stores of the epilogue).
bool make_map_out(CUtensorMap *m, const void *base, int planes, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {128, (cuuint64_t)rows * 128};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [planes][rows][64] bf16 tensor, box of `box_rows` rows, 128-byte swizzle.
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

template <int MODE>
cudaError_t launch_mode(const AttnShape &s, const void *q, const void *k, const void *v,
                        const void *r, const void *u, const void *vb, void *o, void *o_lo, float *lse,
                        const void *dout, float *delta, void *qu_out, void *qv_out,
                        cudaStream_t st, int *launches) {
  CUtensorMap tk, tv, tr, tq, to, tolo;
  if (!make_map(&tk, k, s.B * s.H, s.kv_rows, BK) || !make_map(&tv, v, s.B * s.H, s.kv_rows, BK) ||
      !make_map(&tr, r, s.H, s.kv_rows, NB) || !make_map(&tq, q, s.B * s.H, s.L, BQ))
    return cudaErrorInvalidValue;
  // the outputs' maps (the preparation pass writes no O: its maps are unused)
  memset(&to, 0, sizeof(to));
  memset(&tolo, 0, sizeof(tolo));
  if (MODE == kFwd && (!make_map_out(&to, o, s.B * s.H, s.L) || (o_lo && !make_map_out(&tolo, o_lo, s.B * s.H, s.L))))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    const void *fns[4] = {(const void *)rxl_fwd_tc_kernel<MODE, false, false>,
                          (const void *)rxl_fwd_tc_kernel<MODE, true, false>,
                          (const void *)rxl_fwd_tc_kernel<MODE, false, true>,
                          (const void *)rxl_fwd_tc_kernel<MODE, true, true>};
    for (int f = 0; f < 4 && attr_err == cudaSuccess; ++f)
      attr_err = cudaFuncSetAttribute(fns[f], cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  Params p;
  p.dout = (const __nv_bfloat16 *)dout; p.delta = delta;
  p.qu_out = (__nv_bfloat16 *)qu_out; p.qv_out = (__half *)qv_out;
  p.B = s.B; p.H = s.H; p.L = s.L; p.cap = s.cap; p.m = s.m; p.head = s.head;
  p.mvis = s.mvis;
  p.nq = (s.L + BQ - 1) / BQ;
  p.fd_bh.init((uint32_t)(s.B * s.H));
  p.fd_h.init((uint32_t)s.H);
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.q = (const __nv_bfloat16 *)q; p.u = (const __nv_bfloat16 *)u; p.vb = (const __nv_bfloat16 *)vb;
  p.o = (__nv_bfloat16 *)o; p.o_lo = (__nv_bfloat16 *)o_lo; p.lse = lse;
  const int nitems = s.B * s.H * p.nq;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // the per-row reset is a separate instantiation: the plain call pays nothing for it
  if (MODE == kFwd && 2 * nitems <= sms) {
    // few items (short segments, few heads): two CTAs per item, each over
    // half of its key tiles, merged through distributed shared memory
    const int slot = timing_begin(0, st);
    cudaError_t e =
        s.mvis ? launch_ex(rxl_fwd_tc_kernel<MODE, true, true>, dim3((unsigned)(2 * nitems)), dim3(kThreads),
                           SMEM_BYTES, st, 2, tk, tv, tr, tq, to, tolo, p, nitems)
               : launch_ex(rxl_fwd_tc_kernel<MODE, false, true>, dim3((unsigned)(2 * nitems)), dim3(kThreads),
                           SMEM_BYTES, st, 2, tk, tv, tr, tq, to, tolo, p, nitems);
    timing_end(0, slot, st);
    ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const unsigned grid = (unsigned)(nitems < sms ? nitems : sms);
  const int slot = MODE == kFwd ? timing_begin(0, st) : -1;
  const cudaError_t e =
      s.mvis ? launch_ex(rxl_fwd_tc_kernel<MODE, true, false>, dim3(grid), dim3(kThreads), SMEM_BYTES, st, 1, tk, tv,
                         tr, tq, to, tolo, p, nitems)
             : launch_ex(rxl_fwd_tc_kernel<MODE, false, false>, dim3(grid), dim3(kThreads), SMEM_BYTES, st, 1, tk,
                         tv, tr, tq, to, tolo, p, nitems);
  timing_end(0, slot, st);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_fwd(const AttnShape &s, const void *q, const void *k, const void *v,
                          const void *r, const void *u, const void *vb, void *o, void *o_lo,
                          float *lse, cudaStream_t st, int *launches) {
  return launch_mode<kFwd>(s, q, k, v, r, u, vb, o, o_lo, lse, nullptr, nullptr, nullptr, nullptr, st,
                           launches);
}

cudaError_t launch_tc_bwd_prep(const AttnShape &s, const void *q, const void *k, const void *v,
                               const void *r, const void *u, const void *vb, const void *dout,
                               float *delta, void *qu_out, void *qv_out, cudaStream_t st,
                               int *launches) {
  return launch_mode<kPrep>(s, q, k, v, r, u, vb, nullptr, nullptr, nullptr, dout, delta, qu_out, qv_out,
                            st, launches);
}

cudaError_t tc_fwd_test_hooks(long long wait_cycles, int withhold) {
  const long long cycles = wait_cycles > 0 ? wait_cycles : sm103::kWaitCycles;
  const int w = withhold ? 1 : 0;
  cudaError_t e = cudaMemcpyToSymbol(sm103::g_wait_cycles, &cycles, sizeof(cycles));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fwd_withhold, &w, sizeof(w));
  return e;
}

cudaError_t tc_fwd_read_range(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_fwd_range, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fwd_range, &zero, sizeof(int));
  return e;
}

cudaError_t tc_fwd_read_error(int *flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_fwd_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fwd_error, &zero, sizeof(int));
  return e;
}

}  // namespace rxl
