// Shared pieces of the sm_103a attention kernels: key-tile enumeration over
// the memory ring, the skewed position-score read-out and small TMEM helpers.
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "sm103.cuh"

namespace rxl {
namespace tc {

using namespace sm103;

constexpr int BQ = 128, BK = 128, DH = 64, NB = 256;

// Unsigned division by a divisor fixed for a launch, for n, d < 2^31: with
// s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1 (computed on the
// host), floor(n / d) = (umulhi(n, m) + n) >> s — the round-up reciprocal of
// Granlund and Montgomery, "Division by invariant integers using
// multiplication" (1994). The work cursors split item numbers with it.
struct FastDiv {
  uint32_t d, mul, shift;
  __host__ void init(uint32_t divisor) {
    d = divisor;
    shift = 0;
    while ((1ull << shift) < d) ++shift;
    mul = (uint32_t)((((1ull << 32) * ((1ull << shift) - d)) / d) + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, mul) + n) >> shift; }
  __device__ __forceinline__ uint32_t mod(uint32_t n) const { return n - div(n) * d; }
};

// A run of 128 physically contiguous K/V rows.
struct KeyTile {
  int phys0;   // first physical K/V row
  int jlog0;   // logical key position of that row (-m .. L-1)
  int nvalid;  // rows of the tile that belong to this run
};

// Key tiles over ring run A (head .. cap), ring run B (0 .. ), then the
// current rows 0 .. lenC. A tile never straddles the ring's wrap, so its
// rows are consecutive logical keys and one R band serves the whole tile.
struct KeyTiles {
  int m, cap, head, lenA, lenB, lenC, nA, nB, nC;
  __device__ KeyTiles(int m_, int cap_, int head_, int lenC_) {
    m = m_; cap = cap_; head = head_;
    lenA = min(m, cap - head);
    lenB = m - lenA;
    lenC = lenC_;
    nA = (lenA + BK - 1) / BK;
    nB = (lenB + BK - 1) / BK;
    nC = (lenC + BK - 1) / BK;
  }
  __device__ int count() const { return nA + nB + nC; }
  __device__ KeyTile get(int t) const {
    KeyTile x;
    if (t < nA) {
      x.phys0 = head + t * BK;
      x.jlog0 = -m + t * BK;
      x.nvalid = min(BK, lenA - t * BK);
    } else if (t < nA + nB) {
      const int u = t - nA;
      x.phys0 = u * BK;
      x.jlog0 = -m + lenA + u * BK;
      x.nvalid = min(BK, lenB - u * BK);
    } else {
      const int u = t - nA - nB;
      x.phys0 = cap + u * BK;
      x.jlog0 = u * BK;
      x.nvalid = min(BK, lenC - u * BK);
    }
    return x;
  }
};

// Memory seen by batch row b under a per-row document reset: its newest
// mb = clamp(mvis[b], 0, m) rows, which are themselves a ring run starting
// at physical row (head + m - mb) mod cap. mvis == nullptr: all m rows.
struct RowMemory {
  int m, head;
};
__device__ __forceinline__ RowMemory row_memory(const int *mvis, int b, int m, int cap, int head) {
  RowMemory r{m, head};
  if (mvis) {
    int mb = mvis[b];
    mb = mb < 0 ? 0 : (mb > m ? m : mb);
    r.m = mb;
    r.head = cap > 0 ? (head + m - mb) % cap : 0;
  }
  return r;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return (uint8_t *)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// win[x] <- win[x + lane] for x = 0..63: a 96-value window (serving two
// adjacent 32-key chunks) shifted left by the lane index in 5 predicated
// stages, largest shift first. Two of every three pairs of a stage are
// selects on the ALU pipe and the third goes through the FMA pipe as
// take * t + keep * (1 - t) with t in {0, 1}, which is exact for finite
// values (the window holds position logits of finite operands): the stages
// are the ALU pipe's main load, and this split measured fastest (all on the
// ALU, half or a quarter on the FMA pipe were slower).
__device__ __forceinline__ void lane_shift_window96(float (&win)[96], int lane) {
#pragma unroll
  for (int b = 4; b >= 0; --b) {
    const int sh = 1 << b;
    const bool take = (lane >> b) & 1;
    const float t = take ? 1.f : 0.f;
    const float2 t2 = make_float2(t, t), nt2 = make_float2(1.f - t, 1.f - t);
    const int n = 64 + sh - 1;  // window entries this stage still needs
#pragma unroll
    for (int e = 0; e < 95; e += 2) {
      if (e >= n) continue;
      if ((e >> 1) % 3 == 2 && e + 1 < n) {
        const float2 keep = make_float2(win[e], win[e + 1]);
        const float2 tk = make_float2(win[e + sh], win[e + 1 + sh]);
        const float2 r = __ffma2_rn(tk, t2, __fmul2_rn(keep, nt2));
        win[e] = r.x;
        win[e + 1] = r.y;
      } else {
        win[e] = take ? win[e + sh] : win[e];
        if (e + 1 < n) win[e + 1] = take ? win[e + 1 + sh] : win[e + 1];
      }
    }
  }
}

// Base-2 exponents of P for half a 128x128 tile, two warps per TMEM lane
// quadrant: the calling thread (quadrant `quad`, half `hf`) produces, for
// keys jj = 64*hf + k (k = 0..63) of its row ii = 32*quad + lane,
// y[k] = (S + G_skewed) * scale + bias, -inf where masked. One 96-column G
// window serves both 32-key chunks of the half: chunk 2hf reads columns W ..
// W+63 and chunk 2hf+1 columns W-32 .. W+31 (W = 32 quad + 96 - 64 hf), so
// after the lane shift keys 32c + k sit at win[63 - k] (c = 2hf) and
// win[31 - k] (c = 2hf+1). Pairs of keys go through the packed fp32x2 add
// and fma.
__device__ __forceinline__ void half_tile_exponents(uint32_t trow, uint32_t s_col, uint32_t g_col,
                                                    int quad, int lane, int hf, int i,
                                                    const KeyTile &x, float scale, float bias,
                                                    float (&y)[64]) {
  const float2 scale2 = make_float2(scale, scale), bias2 = make_float2(bias, bias);
  float win[96];
  {
    uint32_t w0[32], w1[32], w2[32];
    const uint32_t gcol = g_col + 32 * quad + 64 - 64 * hf;
    tmem_ld32(trow + gcol, w0);
    tmem_ld32(trow + gcol + 32, w1);
    tmem_ld32(trow + gcol + 64, w2);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      win[e] = __uint_as_float(w0[e]);
      win[32 + e] = __uint_as_float(w1[e]);
      win[64 + e] = __uint_as_float(w2[e]);
    }
  }
  lane_shift_window96(win, lane);
  uint32_t s0[32], s1[32];
  tmem_ld32(trow + s_col + 64 * hf, s0);
  tmem_ld32(trow + s_col + 64 * hf + 32, s1);
  tmem_wait_ld();
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    const float2 a0 = __fadd2_rn(make_float2(__uint_as_float(s0[k]), __uint_as_float(s0[k + 1])),
                                 make_float2(win[63 - k], win[62 - k]));
    const float2 a1 = __fadd2_rn(make_float2(__uint_as_float(s1[k]), __uint_as_float(s1[k + 1])),
                                 make_float2(win[31 - k], win[30 - k]));
    const float2 t0 = __ffma2_rn(a0, scale2, bias2), t1 = __ffma2_rn(a1, scale2, bias2);
    y[k] = t0.x;
    y[k + 1] = t0.y;
    y[32 + k] = t1.x;
    y[32 + k + 1] = t1.y;
  }
  // key jj = 32c + k is visible iff jj < nvalid and jlog0 + jj <= i; the
  // warp skips the mask where all 32 keys are visible to all its rows
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

}  // namespace tc
}  // namespace rxl
