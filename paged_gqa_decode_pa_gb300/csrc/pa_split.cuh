// pa_split.cuh -- phase 1 of paged GQA decode: the persistent split kernel.
//
// One CTA per SM, W warps (8).  Each CTA walks the pieces the schedule
// (pa_sched.cuh) gives it; a piece is a run of physical blocks of one
// (sequence b, kv head j) segment, cut into 16-token tiles.  Tile t of a
// piece belongs to warp t % W.
//
// Every warp runs its own pipeline: a ring of R shared-memory stages, each
// holding the K and V rows (kv head j) of one 16-token tile.  The warp loads
// the tile's physical block id from the block table (32 ids per warp-wide
// load, "Paged Attention Kernel Architecture for BI-V100", section 3: the
// table indirection), checks it, and lane 0 issues the tile's 5-D TMA tensor
// copy (64 dims x 16 rows x d/64 chunks, 128-byte swizzle; one copy for K and
// V when one tensor map spans both pools, else one each) that completes on
// the stage's mbarrier.  After computing tile n the warp refills the same
// stage with tile n + R, so loads of R tiles are always in flight per warp.
//
// A warp keeps the online-softmax state (running max, exp-sum, weighted-V
// accumulator; "v10_triton_paged_gqa", Core Principle) of ALL G query heads
// of kv head j: each K/V byte is read from HBM once for the whole group (the
// BI-V100 design, section 4).  At the end of a piece the W warp states are
// folded with the (max, exp-sum, weighted-V) combine op (section 2, Levels
// 1-2) and written as the final output or as a partial state for the merge
// kernel (section 2, Level 3).
//
// Scores are kept in log2 units (times scale*log2(e)) so every exponential
// is one ex2 instruction; the merge kernel uses the same units.
//
// Tensor-core variant (kMma): per 16-token tile, S^T[16 tokens x 8 heads] =
// K[16 x d] . q^T[d x 8] (the raw 16-bit q, exact; the fp32 scores then take
// the factor scale*log2(e)) and O^T[d x 8] += V^T[d x 16] . P^T[16 x 8] with
// mma.sync m16n8k16 (fp32 accumulate).  P is split into a high and a low
// 16-bit part (p = hi + lo) so that the product keeps ~16 significant bits;
// heads beyond G are zero columns.
// CUDA-core variant (kSimt): lane <-> token for q.k (fp32 FMA), lane <->
// dimension pair for p.V.
#pragma once

#include <math.h>

#include <type_traits>

#include "pa_kernels.cuh"
#include "pa_ptx.cuh"

namespace pa {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: a stuck pipeline, never expected
constexpr uint32_t kStatusBadBlock = 0x1u;
constexpr uint32_t kStatusBadSeqlen = 0x2u;
constexpr uint32_t kStatusTimeout = 0x4u;
constexpr uint32_t kStatusNoSlot = 0x8u;
constexpr uint32_t kInfoBad = 0x10000u;

// Byte offset of the 16-byte unit `unit` (0..7) of row `row` inside one
// 128B-swizzled [rows][64] chunk tile written by TMA (tile base 1024-aligned).
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t unit) {
  return row * 128u + ((unit ^ (row & 7u)) << 4);
}

// ------------------------------------------------------------------ prologue

// Prefix sums of the per-row counts into pre[0..B] (shared memory).
template <class LenOf>
__device__ __forceinline__ void build_prefix(const SplitArgs& a, const LenOf& len_of, int32_t* pre,
                                             int32_t* scratch) {
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  const int per = (a.B + T - 1) / T;
  const int b0 = min(a.B, tid * per), b1 = min(a.B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b)
    local += seq_count(seq_blocks(len_of(b), a.bs, a.maxblk), a.part_blocks, a.piece_k);
  // inclusive scan of `local` over the block
  const int lane = tid & 31, warp = tid >> 5;
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < T / 32; ++w) {
      int t = scratch[w];
      scratch[w] = run;
      run += t;
    }
    pre[a.B] = run;
  }
  __syncthreads();
  int run = scratch[warp] + x - local;
  for (int b = b0; b < b1; ++b) {
    pre[b] = run;
    run += seq_count(seq_blocks(len_of(b), a.bs, a.maxblk), a.part_blocks, a.piece_k);
  }
  __syncthreads();
}

// ------------------------------------------------------------- consumer state

template <typename T, int D, int NB, bool kQ>
struct MmaState {
  uint32_t qf[NB][D / 16][2];  // B fragments of q (the 16-bit values, exact)
  float qsc;                   // scale * log2(e), applied to the fp32 scores
  float o[NB][D / 16][4];                         // O^T accumulators
  float m[NB][2], l[NB][2];                       // columns 8nb + 2t, 8nb + 2t + 1 of this lane
  int32_t lim[NB][2];                             // kQ: key limit of those columns
  bool bad;

  // B fragments of q for the 8 NB columns, from the CTA's shared fp32 copy
  // qs [C][D+4] of the 16-bit values (columns >= C are zero); packing them
  // back to 16 bits is exact, so the scores K.q come out of the mma with fp32
  // accumulation and only then take the factor scale * log2(e).  kQ: also the
  // columns' key limits (tokens t < lim are visible).
  __device__ __forceinline__ void load_q(const float* qs, int C, const int32_t* qlim, float qscale) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    qsc = qscale;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int col = nb * 8 + g;
      const bool live = col < C;
      const float* qrow = qs + (live ? col : 0) * (D + 4);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v = 0;
          if (live) {
            const float2 x = *reinterpret_cast<const float2*>(qrow + ks * 16 + half * 8 + 2 * t);
            v = Cvt<T>::pack(x.x, x.y);
          }
          qf[nb][ks][half] = v;
        }
      }
      if constexpr (kQ) {
        lim[nb][0] = qlim[nb * 8 + 2 * t];
        lim[nb][1] = qlim[nb * 8 + 2 * t + 1];
      }
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[nb][i][c] = 0.f;
      m[nb][0] = m[nb][1] = -INFINITY;
      l[nb][0] = l[nb][1] = 0.f;
    }
    bad = false;
  }

  // One 16-token tile, `valid` (1..16) of its rows real, tok0 = index of its
  // first token in the sequence; K chunks at kb, V chunks at vb, each chunk a
  // 128B-swizzled [16][64] tile of 2 KB.
  //
  // ldmatrix takes one row address per lane, so two kinds of rows are read
  // from outside the TMA stage (which no thread ever writes): V rows past the
  // sequence end read the CTA's zero row, and row `new_r` (the token being
  // appended, or -1) reads the warp's copy of the new K/V rows at nk / nv.
  // Those buffers are unswizzled: 64-dim chunk c, unit u at c*128 + u*16.
  // Each K and V fragment feeds the NB column blocks.
  __device__ __forceinline__ void tile(uint32_t kb, uint32_t vb, int valid, int tok0, int new_r,
                                       uint32_t nk, uint32_t nv, uint32_t zrow) {
    const int lane = threadIdx.x & 31;
    constexpr uint32_t chunk = kTile * 128u;
    // ---- S^T = K . q^T  (rows: the 16 tokens, cols: query columns); four
    // independent accumulator chains per block (k-step mod 4)
    float acc4[NB][4][4] = {};
    {
      const uint32_t tok = (lane & 7) + ((lane >> 3) & 1) * 8;
      const uint32_t uh = (uint32_t)(lane >> 4);
      const bool knew = (int)tok == new_r;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        const uint32_t unit = 2u * (ks & 3) + uh;
        const uint32_t addr = knew ? nk + (uint32_t)(ks >> 2) * 128u + unit * 16u
                                   : kb + (uint32_t)(ks >> 2) * chunk + swz(tok, unit);
        ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          mma_16816<T>(acc4[nb][ks & 3], a0, a1, a2, a3, qf[nb][ks][0], qf[nb][ks][1]);
        }
      }
    }
    const int tr = lane >> 2;
    uint32_t bh0[NB], bh1[NB], bl0[NB], bl1[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float s0 = ((acc4[nb][0][0] + acc4[nb][1][0]) + (acc4[nb][2][0] + acc4[nb][3][0])) * qsc;
      float s1 = ((acc4[nb][0][1] + acc4[nb][1][1]) + (acc4[nb][2][1] + acc4[nb][3][1])) * qsc;
      float s2 = ((acc4[nb][0][2] + acc4[nb][1][2]) + (acc4[nb][2][2] + acc4[nb][3][2])) * qsc;
      float s3 = ((acc4[nb][0][3] + acc4[nb][1][3]) + (acc4[nb][2][3] + acc4[nb][3][3])) * qsc;
      if constexpr (kQ) {
        // per-column visibility: token tok0 + row is seen by a column only
        // below its limit; with the tile's real rows, rows [0, vis) count
        const int vis0 = min(valid, lim[nb][0] - tok0), vis1 = min(valid, lim[nb][1] - tok0);
        if (tr >= vis0) s0 = -INFINITY;
        if (tr >= vis1) s1 = -INFINITY;
        if (tr + 8 >= vis0) s2 = -INFINITY;
        if (tr + 8 >= vis1) s3 = -INFINITY;
      } else {
        if (tr >= valid) s0 = s1 = -INFINITY;
        if (tr + 8 >= valid) s2 = s3 = -INFINITY;
      }
      // ---- online softmax update for the lane's two columns
      float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
      }
      // Lazy running max: a column's max moves only when the tile's max is
      // above it by more than kLazyMax (log2 units).  Otherwise p is taken
      // against the stale max and stays below 2^kLazyMax, and the
      // accumulator is not rescaled; the state (m, l, o) is consistent for
      // any m, so the folds downstream are unchanged.
      const float n0 = (x0 > m[nb][0] + kLazyMax) ? x0 : m[nb][0];
      const float n1 = (x1 > m[nb][1] + kLazyMax) ? x1 : m[nb][1];
      const float u0 = (n0 == -INFINITY) ? 0.f : n0;
      const float u1 = (n1 == -INFINITY) ? 0.f : n1;
      const float al0 = ex2(m[nb][0] - u0), al1 = ex2(m[nb][1] - u1);
      const float p0 = ex2(s0 - u0), p1 = ex2(s1 - u1), p2 = ex2(s2 - u0), p3 = ex2(s3 - u1);
      l[nb][0] = l[nb][0] * al0 + (p0 + p2);
      l[nb][1] = l[nb][1] * al1 + (p1 + p3);
      m[nb][0] = n0;
      m[nb][1] = n1;
      // rescale the accumulator only when some running max moved
      if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
          o[nb][dt][0] *= al0;
          o[nb][dt][1] *= al1;
          o[nb][dt][2] *= al0;
          o[nb][dt][3] *= al1;
        }
      }
      // ---- P^T fragments (k = tokens, n = columns), hi + lo parts
      const uint32_t h01 = Cvt<T>::pack(p0, p1), h23 = Cvt<T>::pack(p2, p3);
      const uint32_t e01 = Cvt<T>::pack(p0 - Cvt<T>::low(h01), p1 - Cvt<T>::high(h01));
      const uint32_t e23 = Cvt<T>::pack(p2 - Cvt<T>::low(h23), p3 - Cvt<T>::high(h23));
      bh0[nb] = movmatrix_trans(h01);
      bh1[nb] = movmatrix_trans(h23);
      bl0[nb] = movmatrix_trans(e01);
      bl1[nb] = movmatrix_trans(e23);
    }
    // ---- O^T += V^T . P^T  (rows past the end read zeros, so p = 0 adds 0
    // even where the pool holds NaN)
    {
      const uint32_t tok = (lane & 7) + (lane >> 4) * 8;
      const uint32_t uh = (uint32_t)((lane >> 3) & 1);
      const bool vplain = (int)tok == new_r || (int)tok >= valid;
      const uint32_t vrow = (int)tok == new_r ? nv : zrow;
#pragma unroll
      for (int dt = 0; dt < D / 16; ++dt) {
        uint32_t a0, a1, a2, a3;
        const uint32_t unit = 2u * (dt & 3) + uh;
        const uint32_t addr = vplain ? vrow + (uint32_t)(dt >> 2) * 128u + unit * 16u
                                     : vb + (uint32_t)(dt >> 2) * chunk + swz(tok, unit);
        ldmatrix_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          mma_16816<T>(o[nb][dt], a0, a1, a2, a3, bh0[nb], bh1[nb]);
          mma_16816<T>(o[nb][dt], a0, a1, a2, a3, bl0[nb], bl1[nb]);
        }
      }
    }
  }

  // Publish this warp's state for the CTA-level combine: its C columns, in
  // a slot of `stride` columns.
  __device__ __forceinline__ void publish(uint8_t* smem, const SmemLayout& L, int w, int C,
                                          int stride) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    float* mm = reinterpret_cast<float*>(smem + L.mm) + w * kColMax;
    float* ml = reinterpret_cast<float*>(smem + L.ml) + w * kColMax;
    float* mo = reinterpret_cast<float*>(smem + L.mo) + (size_t)w * stride * (D + 4);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float l0 = l[nb][0], l1 = l[nb][1];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      const int c0 = nb * 8 + 2 * t, c1 = c0 + 1;
      if (g == 0) {
        mm[c0] = m[nb][0];
        mm[c1] = m[nb][1];
        ml[c0] = l0;
        ml[c1] = l1;
      }
#pragma unroll
      for (int dt = 0; dt < D / 16; ++dt) {
        const int dim = dt * 16 + g;
        if (c0 < C) {
          mo[c0 * (D + 4) + dim] = o[nb][dt][0];
          mo[c0 * (D + 4) + dim + 8] = o[nb][dt][2];
        }
        if (c1 < C) {
          mo[c1 * (D + 4) + dim] = o[nb][dt][1];
          mo[c1 * (D + 4) + dim + 8] = o[nb][dt][3];
        }
      }
    }
    if (lane == 0) reinterpret_cast<int*>(smem + L.mbad)[w] = bad ? 1 : 0;
  }
};

// Rows of up to kRowCols (token, head) columns held by one warp, the columns
// as the mma's M dimension (m-tile mt holds columns 16 mt .. 16 mt + 15):
//   S[16 columns x 16 tokens] = q . K^T   (per m-tile; K is the B operand)
//   O[16 columns x D]        += P . V     (P the A operand, V the B operand)
// The C fragment of S -- row g / g + 8, tokens 2t, 2t+1 of each 8-token
// n-block -- is already P's A fragment once packed to 16 bits, so no
// transposes; each K and V fragment feeds both m-tiles.  q's A fragments are
// read from the 16-bit copy in shared memory at every k-step (registers hold
// the 2 x D/8 x 4 accumulators instead).  Each lane's exp-sums cover its own
// tokens; the quad's are added when the state is published.
template <typename T, int D>
struct MmaWState {
  static constexpr int MT = 2;      // m-tiles of 16 columns
  static constexpr int NT = D / 8;  // n-blocks of 8 dims of O
  float o[MT][NT][4];     // rows g, g+8 of each m-tile: [0,1] row g dims 2t, 2t+1; [2,3] row g+8
  float m[MT][2], l[MT][2];
  int32_t lim[MT][2];     // key limit of rows g, g+8 (tokens t < lim are visible)
  float qsc;              // scale * log2(e), applied to the fp32 scores
  bool bad;

  __device__ __forceinline__ void load_lim(const int32_t* qlim, float qscale) {
    const int g = (threadIdx.x & 31) >> 2;
    qsc = qscale;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      lim[mt][0] = qlim[mt * 16 + g];
      lim[mt][1] = qlim[mt * 16 + g + 8];
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[mt][n][c] = 0.f;
      m[mt][0] = m[mt][1] = -INFINITY;
      l[mt][0] = l[mt][1] = 0.f;
    }
    bad = false;
  }

  // One 16-token tile (see MmaState::tile for kb, vb, valid, tok0, zrow);
  // qa: the row's 16-bit q, [kRowCols][D + 8].
  __device__ __forceinline__ void tile(uint32_t kb, uint32_t vb, int valid, int tok0, uint32_t zrow,
                                       uint32_t qa) {
    const int lane = threadIdx.x & 31;
    const int t = lane & 3;
    constexpr uint32_t chunk = kTile * 128u;
    constexpr uint32_t qstride = wide_q_stride(D);
    // ---- S = q . K^T: eight independent accumulator chains (m-tile x
    // n-block x k-step parity)
    float acc2[MT][2][2][4] = {};
    {
      // K, non-transposed: matrices (tokens 0-7 | 8-15) x (dims lo | hi of
      // the k-step) give b0, b1 of n-block 0 and b0, b1 of n-block 1
      const uint32_t ktok = (lane & 7) + (lane >> 4) * 8;
      const uint32_t kuh = (uint32_t)((lane >> 3) & 1);
      // q: matrices (columns 0-7 | 8-15) x (dims lo | hi) give a0 .. a3
      const uint32_t qrow = (lane & 7) + ((lane >> 3) & 1) * 8;
      const uint32_t qoff = qa + qrow * qstride + (uint32_t)(lane >> 4) * 16u;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kb + (uint32_t)(ks >> 2) * chunk + swz(ktok, 2u * (ks & 3) + kuh), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(qoff + (uint32_t)mt * 16u * qstride + (uint32_t)ks * 32u, a0, a1, a2, a3);
          mma_16816<T>(acc2[mt][0][ks & 1], a0, a1, a2, a3, b0, b1);
          mma_16816<T>(acc2[mt][1][ks & 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    // ---- online softmax per row, both m-tiles before any branch (so that
    // their chains interleave); one vote for the rescale; then P's A
    // fragments (high and low parts)
    float x[MT][2][4];  // [m-tile][row g, g+8][tokens 2t, 2t+1, 8+2t, 9+2t]
    float al[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          x[mt][0][2 * nb + e] = (acc2[mt][nb][0][e] + acc2[mt][nb][1][e]) * qsc;
          x[mt][1][2 * nb + e] = (acc2[mt][nb][0][2 + e] + acc2[mt][nb][1][2 + e]) * qsc;
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        // tokens [0, vis) of the tile are real and below the row's key limit
        const int vis = min(valid, lim[mt][r] - tok0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tk = (i >> 1) * 8 + 2 * t + (i & 1);
          if (tk >= vis) x[mt][r][i] = -INFINITY;
        }
        float mx = fmaxf(fmaxf(x[mt][r][0], x[mt][r][1]), fmaxf(x[mt][r][2], x[mt][r][3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // lazy running max, as in MmaState::tile
        const float nm = (mx > m[mt][r] + kLazyMax) ? mx : m[mt][r];
        const float u = (nm == -INFINITY) ? 0.f : nm;
        al[mt][r] = ex2(m[mt][r] - u);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[mt][r][i] = ex2(x[mt][r][i] - u);
          sum += x[mt][r][i];
        }
        l[mt][r] = l[mt][r] * al[mt][r] + sum;
        m[mt][r] = nm;
      }
    }
    if (__any_sync(0xffffffffu, al[0][0] != 1.f || al[0][1] != 1.f || al[1][0] != 1.f ||
                                    al[1][1] != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[mt][n][0] *= al[mt][0];
          o[mt][n][1] *= al[mt][0];
          o[mt][n][2] *= al[mt][1];
          o[mt][n][3] *= al[mt][1];
        }
    }
    uint32_t ph[MT][4], pl[MT][4];
    auto split = [](float p0, float p1, uint32_t& hi, uint32_t& lo) {
      hi = Cvt<T>::pack(p0, p1);
      lo = Cvt<T>::pack(p0 - Cvt<T>::low(hi), p1 - Cvt<T>::high(hi));
    };
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      // a0: row g tokens 2t, 2t+1; a1: row g+8; a2, a3: tokens 8 + 2t, 9 + 2t
      split(x[mt][0][0], x[mt][0][1], ph[mt][0], pl[mt][0]);
      split(x[mt][1][0], x[mt][1][1], ph[mt][1], pl[mt][1]);
      split(x[mt][0][2], x[mt][0][3], ph[mt][2], pl[mt][2]);
      split(x[mt][1][2], x[mt][1][3], ph[mt][3], pl[mt][3]);
    }
    // ---- O += P . V  (V transposed by ldmatrix; rows past the end read
    // the zero row, so p = 0 adds 0 even where the pool holds NaN)
    {
      // matrices (tokens 0-7 | 8-15) x (dims of n-block 2p | 2p + 1)
      const uint32_t vtok = (lane & 7) + ((lane >> 3) & 1) * 8;
      const uint32_t vuh = (uint32_t)(lane >> 4);
      const bool vzero = (int)vtok >= valid;
#pragma unroll
      for (int p = 0; p < D / 16; ++p) {
        uint32_t b0, b1, b2, b3;
        const uint32_t unit = 2u * (p & 3) + vuh;
        const uint32_t addr = vzero ? zrow + (uint32_t)(p >> 2) * 128u + unit * 16u
                                    : vb + (uint32_t)(p >> 2) * chunk + swz(vtok, unit);
        ldmatrix_x4_trans(addr, b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_16816<T>(o[mt][2 * p], ph[mt][0], ph[mt][1], ph[mt][2], ph[mt][3], b0, b1);
          mma_16816<T>(o[mt][2 * p + 1], ph[mt][0], ph[mt][1], ph[mt][2], ph[mt][3], b2, b3);
          mma_16816<T>(o[mt][2 * p], pl[mt][0], pl[mt][1], pl[mt][2], pl[mt][3], b0, b1);
          mma_16816<T>(o[mt][2 * p + 1], pl[mt][0], pl[mt][1], pl[mt][2], pl[mt][3], b2, b3);
        }
      }
    }
  }

  // Publish m-tile MTI (columns 16 MTI .. 16 MTI + 15) of this warp's state
  // for the CTA-level combine, as a 16-column state.
  template <int MTI>
  __device__ __forceinline__ void publish(uint8_t* smem, const SmemLayout& L, int w) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    float* mm = reinterpret_cast<float*>(smem + L.mm) + w * kColMax;
    float* ml = reinterpret_cast<float*>(smem + L.ml) + w * kColMax;
    float* mo = reinterpret_cast<float*>(smem + L.mo) + (size_t)w * kColMax * (D + 4);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float lr = l[MTI][r];
      lr += __shfl_xor_sync(0xffffffffu, lr, 1);
      lr += __shfl_xor_sync(0xffffffffu, lr, 2);
      const int lc = g + 8 * r;
      if (t == 0) {
        mm[lc] = m[MTI][r];
        ml[lc] = lr;
      }
#pragma unroll
      for (int n = 0; n < NT; ++n)
        *reinterpret_cast<float2*>(mo + lc * (D + 4) + n * 8 + 2 * t) =
            make_float2(o[MTI][n][2 * r], o[MTI][n][2 * r + 1]);
    }
    if (lane == 0) reinterpret_cast<int*>(smem + L.mbad)[w] = bad ? 1 : 0;
  }
};

template <typename T, int D>
struct SimtState {
  float acc[kGMax][D / 32];  // dims c*64 + 2*lane + e, e in {0,1}, chunk c
  float m[kGMax], l[kGMax];  // m: warp-uniform; l: this lane's tokens only
  bool bad;

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[g][i] = 0.f;
      m[g] = -INFINITY;
      l[g] = 0.f;
    }
    bad = false;
  }

  // One 16-token tile, `valid` (1..16) rows real.  qs: shared [G][D] fp32
  // q*scale*log2e.  ps: this warp's [16][8] fp32 buffer.  Lanes 0-15 and
  // 16-31 take the same 16 tokens for the two halves of the G heads.
  // Rows as in MmaState::tile: row new_r (or -1) is read from nk / nv.
  __device__ __forceinline__ void tile(uint32_t kb, uint32_t vb, int valid, const float* qs,
                                       float* ps, int G, int new_r, uint32_t nk, uint32_t nv) {
    const int lane = threadIdx.x & 31;
    constexpr uint32_t chunk = kTile * 128u;
    // ---------------- q . k : lane <-> token
    const int GH = (G + 1) >> 1;
    const int h0 = (lane >> 4) * GH;
    const int h1 = min(G, h0 + GH);
    const int tt = lane & 15;
    float s[kGMax];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) s[g] = 0.f;
#pragma unroll 4
    for (int c8 = 0; c8 < D / 8; ++c8) {
      const uint4 kr = lds128(tt == new_r ? nk + (uint32_t)(c8 >> 3) * 128u + (uint32_t)(c8 & 7) * 16u
                                          : kb + (uint32_t)(c8 >> 3) * chunk + swz(tt, c8 & 7));
      float kf[8];
      kf[0] = Cvt<T>::low(kr.x);
      kf[1] = Cvt<T>::high(kr.x);
      kf[2] = Cvt<T>::low(kr.y);
      kf[3] = Cvt<T>::high(kr.y);
      kf[4] = Cvt<T>::low(kr.z);
      kf[5] = Cvt<T>::high(kr.z);
      kf[6] = Cvt<T>::low(kr.w);
      kf[7] = Cvt<T>::high(kr.w);
#pragma unroll
      for (int g = 0; g < kGMax; ++g) {
        if (g >= h0 && g < h1) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + g * (D + 4) + c8 * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + g * (D + 4) + c8 * 8 + 4);
          float v = s[g];
          v = fmaf(qa.x, kf[0], v);
          v = fmaf(qa.y, kf[1], v);
          v = fmaf(qa.z, kf[2], v);
          v = fmaf(qa.w, kf[3], v);
          v = fmaf(qb.x, kf[4], v);
          v = fmaf(qb.y, kf[5], v);
          v = fmaf(qb.z, kf[6], v);
          v = fmaf(qb.w, kf[7], v);
          s[g] = v;
        }
      }
    }
    const bool live = tt < valid;
    float mx[kGMax];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
      const bool mine = g >= h0 && g < h1;
      if (!mine || !live) s[g] = -INFINITY;
      mx[g] = s[g];
    }
    // tile max per head, made warp-uniform (other half's heads are -inf here)
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], off));
    }
    float alpha[kGMax];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
      const float n = fmaxf(m[g], mx[g]);
      const float mu = (n == -INFINITY) ? 0.f : n;
      alpha[g] = ex2(m[g] - mu);
      m[g] = n;
      const bool mine = g >= h0 && g < h1;
      const float p = (mine && live) ? ex2(s[g] - mu) : 0.f;
      l[g] = l[g] * alpha[g] + p;
      if (mine) ps[tt * kGMax + g] = p;
    }
    __syncwarp();
    // ---------------- p . V : lane <-> dimension pair
#pragma unroll
    for (int g = 0; g < kGMax; ++g)
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[g][i] *= alpha[g];
    const uint32_t col = (uint32_t)((lane & 3) * 4);
    const uint32_t unit = (uint32_t)(lane >> 2);
    for (int t = 0; t < valid; ++t) {
      const float4 pa = *reinterpret_cast<const float4*>(ps + t * kGMax);
      const float4 pb = *reinterpret_cast<const float4*>(ps + t * kGMax + 4);
      const float p[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const uint32_t v = lds32(t == new_r ? nv + (uint32_t)c * 128u + unit * 16u + col
                                            : vb + (uint32_t)c * chunk + swz(t, unit) + col);
        const float v0 = Cvt<T>::low(v), v1 = Cvt<T>::high(v);
#pragma unroll
        for (int g = 0; g < kGMax; ++g) {
          if (g < G) {
            acc[g][2 * c] = fmaf(p[g], v0, acc[g][2 * c]);
            acc[g][2 * c + 1] = fmaf(p[g], v1, acc[g][2 * c + 1]);
          }
        }
      }
    }
    __syncwarp();
  }

  __device__ __forceinline__ void publish(uint8_t* smem, const SmemLayout& L, int w, int G) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
    }
    float* mm = reinterpret_cast<float*>(smem + L.mm) + w * kColMax;
    float* ml = reinterpret_cast<float*>(smem + L.ml) + w * kColMax;
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < kGMax; ++g) {
        mm[g] = m[g];
        ml[g] = l[g];
      }
    }
    float* mo = reinterpret_cast<float*>(smem + L.mo) + (size_t)w * G * (D + 4);
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
      if (g < G) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          float2 v = make_float2(acc[g][2 * c], acc[g][2 * c + 1]);
          *reinterpret_cast<float2*>(mo + g * (D + 4) + c * 64 + 2 * lane) = v;
        }
      }
    }
    if (lane == 0) reinterpret_cast<int*>(smem + L.mbad)[w] = bad ? 1 : 0;
  }
};

// Where column c of a piece's row goes: its output row (or -1 when the
// column holds no query) -- decode: head j*G + c of sequence b; several
// query tokens: token g*tq + c/G of the row's sequence, head j*G + c%G.
template <bool kQ>
__device__ __forceinline__ int64_t column_out(const SplitArgs& a, int row, int j, int c, int q0,
                                              int nq) {
  if constexpr (!kQ) {
    return (int64_t)row * a.H + (int64_t)j * a.G + c;
  } else {
    const int g = row % a.nqg;
    const int tok = g * a.tq + c / a.G;
    if (tok >= nq) return -1;
    return (int64_t)(q0 + tok) * a.H + (int64_t)j * a.G + c % a.G;
  }
}

// CTA-level combine of the W warp states of one piece (all threads).  A
// column that saw no key (l = 0: a query token whose causal limit is 0)
// gets 0, as an empty sequence does.
// q0, nq: the query rows of the piece's sequence (several query tokens).
// kPair: warp pairs, warps [0, W/2) hold columns [0, cw) and warps
// [W/2, W) columns [cw, C), each state with cw columns; otherwise every warp
// holds all C columns.
//
// Two passes, one barrier between them: first one thread per column folds
// the warps' maxima and sums into the column's weights (e_w = 2^(m_w - M),
// divided by the column's sum when the piece's result is final); then every
// thread takes 4 consecutive dims of one column at a time, weighs the warps'
// accumulators with float4 shared loads and writes a float4.  The fold order
// over the warps is fixed, so the result is deterministic.
// c0, nc, ns (not kPair): fold columns [c0, c0 + nc) of the row, published
// by every warp as states of ns columns (a wide row's m-tiles, one at a
// time: ns = 16); by default the whole row, ns = nc = C.
template <int D, int W, bool kQ, bool kPair>
__device__ __forceinline__ void combine_piece(const SplitArgs& a, uint8_t* smem, const SmemLayout& L,
                                              const Piece& pc, int q0, int nq, int cw, int c0 = 0,
                                              int nc = -1, int ns = -1) {
  const int C = a.C;
  if (nc < 0) nc = C;
  if (ns < 0) ns = nc;
  const int stride = kPair ? cw : ns;  // columns of one published warp state
  constexpr int NW = kPair ? W / 2 : W;  // warps holding a column
  constexpr int WS = kMaxWarps + 2;      // floats per column in the weight table
  const float* mm = reinterpret_cast<const float*>(smem + L.mm);
  const float* ml = reinterpret_cast<const float*>(smem + L.ml);
  const float* mo = reinterpret_cast<const float*>(smem + L.mo);
  const int* mbad = reinterpret_cast<const int*>(smem + L.mbad);
  float* cwt = reinterpret_cast<float*>(smem + L.cwt);
  bool bad = false;
#pragma unroll
  for (int w = 0; w < W; ++w) bad |= (mbad[w] != 0);
  const float qnan = __int_as_float(0x7fc00000);
  const bool final_out = pc.slot < 0;
  // the warps holding column c, and its index in their states
  auto col_warps = [&](int c, int& w0, int& lc) {
    w0 = 0;
    lc = c - c0;
    if constexpr (kPair) {
      const int cg = c >= cw ? 1 : 0;
      w0 = cg * NW;
      lc = c - cg * cw;
    }
  };
  if (threadIdx.x < nc) {
    const int c = c0 + threadIdx.x;
    int w0, lc;
    col_warps(c, w0, lc);
    float mw[NW];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      mw[w] = mm[(w0 + w) * kColMax + lc];
      M = fmaxf(M, mw[w]);
    }
    float e[NW];
    float Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      e[w] = (mw[w] == -INFINITY) ? 0.f : ex2(mw[w] - M);
      Lsum = fmaf(e[w], ml[(w0 + w) * kColMax + lc], Lsum);
    }
    const float inv = final_out ? (Lsum == 0.f ? 0.f : 1.f / Lsum) : 1.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) cwt[c * WS + w] = e[w] * inv;
    if (!final_out) {
      a.ws_ml[((int64_t)pc.slot * C + c) * 2 + 0] = M;
      a.ws_ml[((int64_t)pc.slot * C + c) * 2 + 1] = bad ? qnan : Lsum;
    }
  }
  named_bar_sync(2, blockDim.x);
  constexpr int DV = D / 4;  // float4s per column
  for (int v = threadIdx.x; v < nc * DV; v += blockDim.x) {
    const int c = c0 + v / DV, d4 = (v % DV) * 4;
    int w0, lc;
    col_warps(c, w0, lc);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float ew = cwt[c * WS + w];
      const float4 x = *reinterpret_cast<const float4*>(mo + ((w0 + w) * stride + lc) * (D + 4) + d4);
      o.x = fmaf(ew, x.x, o.x);
      o.y = fmaf(ew, x.y, o.y);
      o.z = fmaf(ew, x.z, o.z);
      o.w = fmaf(ew, x.w, o.w);
    }
    if (bad) o = make_float4(qnan, qnan, qnan, qnan);
    if (final_out) {
      const int64_t r = column_out<kQ>(a, pc.b, pc.j, c, q0, nq);
      if (r >= 0) *reinterpret_cast<float4*>(a.out + r * D + d4) = o;
    } else {
      *reinterpret_cast<float4*>(a.ws_acc + ((int64_t)pc.slot * C + c) * D + d4) = o;
    }
  }
}

// Tiles of stream s of S in a piece: tiles s, s + S, ...
__device__ __forceinline__ int stream_tiles(const Piece& pc, int sl, int s, int S) {
  const int nt = (pc.blk1 - pc.blk0) << sl;
  return nt > s ? (nt - s + S - 1) / S : 0;
}

// The issuing side of one warp's pipeline: walks the warp's tile stream (all
// pieces of the CTA, tiles w, w+W, ... of each) R tiles ahead of the
// computing side and loads each tile into the ring slot the computing side
// has just freed.  Block-table entries are read 32 tiles at a time, one
// window ahead.
template <class LenOf>
struct IssuerT {
  PieceIterT<LenOf> it;
  Piece pc;
  int i, cnt;        // next tile index (of this warp) in pc, and their count
  int win;           // first tile index of the current table window
  int32_t entry;     // this lane's entry of the current window (tile win + lane)
  int32_t entry_next;  // ... of the next window (tile win + 32 + lane)
  int32_t len;       // the length row pc.b attends to
  int32_t seq;       // the row's sequence (its block-table row)
  uint32_t issued;   // tiles issued so far
  bool done;
};

// Block-table entry of the ii-th tile of stream s (of S) in piece pc.
__device__ __forceinline__ int32_t table_entry(const SplitArgs& a, const Piece& pc, int seq, int cnt,
                                               int ii, int sl, int s, int S) {
  if (ii >= cnt) return 0;
  const int t = s + S * ii;
  return __ldg(a.table + (int64_t)seq * a.maxblk + pc.blk0 + (t >> sl));
}

// a: the arguments in the constant bank (read for every tile); pa: their
// shared-memory copy (read when the issuer moves to the next piece).
// s: the warp's tile stream, of S (one per warp, or one per warp pair).
template <int D, class LenOf>
__device__ __forceinline__ void issue_next(IssuerT<LenOf>& is, const SplitArgs& a,
                                           const SplitArgs& pa, const CUtensorMap* tmk,
                                           const CUtensorMap* tmv, uint32_t base,
                                           const SmemLayout& L, int s, int S, uint32_t slot,
                                           int sl) {
  const int lane = threadIdx.x & 31;
  while (!is.done && is.i >= is.cnt) {
    if (!is.it.next(is.pc)) {
      is.done = true;
      break;
    }
    is.i = 0;
    is.cnt = stream_tiles(is.pc, sl, s, S);
    is.win = 0;
    is.len = is.it.len_of(is.pc.b);
    is.seq = pa.nqg > 1 ? is.pc.b / pa.nqg : is.pc.b;
    is.entry = table_entry(pa, is.pc, is.seq, is.cnt, lane, sl, s, S);
    is.entry_next = table_entry(pa, is.pc, is.seq, is.cnt, 32 + lane, sl, s, S);
    // the piece after this one: its length and first window of table
    // entries are brought into L1 now, so that the next move finds them
    // there instead of waiting an L2 round trip behind the K/V stream
    int32_t nb, nblk0;
    if (is.it.peek_start(nb, nblk0)) {
      const int32_t nseq = pa.nqg > 1 ? nb / pa.nqg : nb;
      const int32_t blk = nblk0 + ((s + S * lane) >> sl);
      if (blk < pa.maxblk) prefetch_l1(pa.table + (int64_t)nseq * pa.maxblk + blk);
      if (lane == 0) prefetch_l1(pa.seqlens + nseq);
    }
  }
  if (is.done) return;
  if (is.i >= is.win + 32) {
    is.win += 32;
    is.entry = is.entry_next;
    is.entry_next = table_entry(pa, is.pc, is.seq, is.cnt, is.win + 32 + lane, sl, s, S);
  }
  const int32_t phys = __shfl_sync(0xffffffffu, is.entry, is.i - is.win);
  if (lane == 0) {
    const int t = s + S * is.i;
    const int blk = is.pc.blk0 + (t >> sl), h = t & ((1 << sl) - 1);
    const int valid = max(0, min(kTile, is.len - blk * a.bs - h * kTile));
    const bool bad = phys < 0 || phys >= a.P;
    const uint32_t gslot = (uint32_t)s * a.ring + slot;
    const uint32_t full = base + L.full + 8 * gslot;
    sts64(base + L.info + 8 * gslot,
          ((uint64_t)(uint32_t)phys << 32) | (uint32_t)valid | (bad ? kInfoBad : 0u));
    if (bad || valid == 0) {
      if (bad && h == 0) atomicOr(a.status, kStatusBadBlock);
      mbar_arrive(full);
    } else {
      constexpr uint32_t chunk = kTile * 128u;
      const uint64_t pol = l2_evict_first_policy();  // K/V rows are read once per step
      mbar_arrive_expect_tx(full, L.stage_bytes);
      const uint32_t kdst = base + L.stage + gslot * L.stage_bytes;
      if (a.kv_fused) {
        // one copy: (64 dims, 16 rows, D/64 chunks, one (block, kv head) slot, K and V)
        tma_load_5d(kdst, tmk, full, 0, h * kTile, 0, phys * a.bs * a.Hkv + is.pc.j, 0, pol);
      } else {
        tma_load_5d(kdst, tmk, full, 0, h * kTile, 0, is.pc.j, phys, pol);
        tma_load_5d(kdst + (D / 64) * chunk, tmv, full, 0, h * kTile, 0, is.pc.j, phys, pol);
      }
    }
  }
  ++is.i;
  ++is.issued;
}

// The next piece's q, fetched while the current piece runs: its raw 16-bit
// values are copied (cp.async) into the shared staging buffer qraw -- at
// the start of the current piece in decode, after its tiles with several
// query tokens (whose rows need the sequence's query span first) -- and at
// the piece boundary `finish` widens them to fp32 in the buffer qs (times
// scale * log2(e) on the CUDA-core path; the tensor-core path applies that
// factor to the scores).  kQ: column c is token g*tq + c/G (head c%G) of the
// row's sequence; `finish` also writes each column's key limit and the
// row's query span.
template <int D, bool kQ>
struct QStage {
  int32_t len;          // stored cache_seqlens of the piece's sequence
  int32_t q0, nq, grp;  // kQ: the sequence's query rows, the row's group

  __device__ __forceinline__ void start(const SplitArgs& a, const Piece& pc, uint32_t qraw) {
    if constexpr (!kQ) {
      len = __ldg(a.seqlens + pc.b);
      const char* src =
          reinterpret_cast<const char*>(a.q + ((int64_t)pc.b * a.H + (int64_t)pc.j * a.G) * D);
      const int chunks = a.C * D / 8;  // 16-byte pieces of G contiguous rows
      for (int i = threadIdx.x; i < chunks; i += blockDim.x)
        cp_async16(qraw + 16u * i, src + 16 * (int64_t)i, 16u);
      cp_async_commit();
    } else {
      const int seq = pc.b / a.nqg;
      grp = pc.b - seq * a.nqg;
      len = __ldg(a.seqlens + seq);
      query_span(a.cu_q, seq, a.total_q, a.max_q, q0, nq);
    }
  }

  // kQ: the copies, once the span is known (columns without a query are
  // zero-filled).
  __device__ __forceinline__ void issue_copies(const SplitArgs& a, const Piece& pc, uint32_t qraw) {
    constexpr int per_col = D / 8;
    const int chunks = a.C * per_col;
    for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
      const int c = i / per_col, k = i - c * per_col;
      const int tok = grp * a.tq + c / a.G;
      const bool valid = tok < nq;
      const char* src =
          valid ? reinterpret_cast<const char*>(
                      a.q + ((int64_t)(q0 + tok) * a.H + (int64_t)pc.j * a.G + c % a.G) * D) +
                      16 * k
                : reinterpret_cast<const char*>(a.q);
      cp_async16(qraw + 16u * i, src, valid ? 16u : 0u);
    }
    cp_async_commit();
  }

  // After every thread's copies are complete and a barrier.  kWide: qs
  // takes the raw 16-bit values, [kRowCols][D + 8] (columns >= C zero),
  // instead of fp32.
  template <typename T, bool kScaled, bool kWide = false>
  __device__ __forceinline__ void finish(const SplitArgs& a, uint32_t qraw, float* qs, int32_t* info,
                                         int32_t* qlim) {
    if (threadIdx.x == 0) {
      info[1] = len;
      if constexpr (kQ) {
        info[2] = q0;
        info[3] = nq;
      }
    }
    if constexpr (kQ) {
      // the key limit of every column: tokens t < limit are visible; columns
      // that hold no query see everything (their q is zero)
      const int c = threadIdx.x;
      if (c < kRowCols) {
        int32_t lim = 0x7fffffff;
        const int tok = grp * a.tq + c / a.G;
        if (c < a.C && tok < nq && a.causal) lim = max(0, min(len, len - nq + tok + 1));
        qlim[c] = lim;
      }
    }
    if constexpr (kWide) {
      constexpr int per_col = D / 8;  // 16-byte units of a column
      const uint32_t qa = smem_u32(qs);
      for (int i = threadIdx.x; i < kRowCols * per_col; i += blockDim.x) {
        const int c = i / per_col, k = i - c * per_col;
        const uint4 v = c < a.C ? lds128(qraw + 16u * i) : make_uint4(0u, 0u, 0u, 0u);
        sts128(qa + (uint32_t)c * wide_q_stride(D) + 16u * k, v);
      }
      return;
    }
    const int nw = a.C * D / 2;
    for (int i = threadIdx.x; i < nw; i += blockDim.x) {
      const int c = (2 * i) / D, d = (2 * i) % D;
      const uint32_t v = lds32(qraw + 4u * i);
      float2 x;
      x.x = Cvt<T>::low(v);
      x.y = Cvt<T>::high(v);
      if constexpr (kScaled) {
        x.x *= a.qscale;
        x.y *= a.qscale;
      }
      *reinterpret_cast<float2*>(qs + c * (D + 4) + d) = x;
    }
  }
};

// Prologue of a split CTA after the prefix sums (all threads): rows with no
// key to read get out = 0, rows with an invalid length NaN + a status bit
// (with the fused append also "no slot": nothing is written for them); CTA 0
// stores the prefix sums (only the fixed split's merge reads them), and every
// CTA stores the descriptor of the segment that begins in it and continues
// past it (balanced split).
template <int D, bool kQ, class LenOf>
__device__ __forceinline__ void rows_without_keys_and_descriptors(const SplitArgs& a,
                                                                  const LenOf& len_of,
                                                                  const int32_t* pre,
                                                                  const SchedShape& sched, int cta) {
  const int tid = threadIdx.x;
  for (int b = cta; b < a.B; b += gridDim.x) {
    if (pre[b + 1] != pre[b]) continue;  // has blocks: no global read needed
    const int32_t len = len_of(b);
    const bool ok = len >= 0;
    const float v = ok ? 0.f : __int_as_float(0x7fc00000);
    if constexpr (!kQ) {
      float* row = a.out + (int64_t)b * a.H * D;
      for (int i = tid; i < a.H * D; i += blockDim.x) row[i] = v;
      if (!ok && tid == 0) atomicOr(a.status, kStatusBadSeqlen | (a.len_add ? kStatusNoSlot : 0u));
    } else {
      // the row's query tokens are consecutive packed rows of out
      const int seq = b / a.nqg, grp = b - seq * a.nqg;
      int32_t q0, nq;
      const bool span = query_span(a.cu_q, seq, a.total_q, a.max_q, q0, nq);
      if ((!span || !ok) && grp == 0 && tid == 0) atomicOr(a.status, kStatusBadSeqlen);
      const int first = grp * a.tq;
      if (!span || first >= nq) continue;
      const int cnt = min(a.tq, nq - first);
      float* rows = a.out + (int64_t)(q0 + first) * a.H * D;
      for (int i = tid; i < cnt * a.H * D; i += blockDim.x) rows[i] = v;
    }
  }
  if (cta == 0 && a.part_blocks > 0)
    for (int b = tid; b <= a.B; b += blockDim.x) a.ws_pre[b] = pre[b];
  if (tid == 0) {
    if (a.part_blocks == 0) {
      int32_t b, j, c_last, slot;
      int4 desc = make_int4(-1, 0, 0, 0);
      if (balanced_split_segment(pre, sched, cta, b, j, c_last, slot)) desc = make_int4(b, j, c_last, slot);
      a.ws_desc[cta] = desc;
    }
  }
}

template <typename T, int D, int MODE>
__global__ void __launch_bounds__(32 * split_warps(D, MODE), 1)
    pa_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ SplitArgs a) {
  constexpr int W = split_warps(D, MODE);
  constexpr bool kQ = several_tokens(MODE);
  constexpr bool kPair = MODE == kMmaP;
  constexpr int NB = mma_blocks(D, MODE);
  using RowLen = typename std::conditional<kQ, MultiLen, DecodeLen>::type;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x;
  // The code that runs once per piece reads the arguments -- and the layout
  // offsets derived from them -- from this shared copy: read from the
  // constant bank after a long run of tiles, they miss in the constant cache
  // and wait microseconds behind the HBM stream.
  SplitArgs* sa = reinterpret_cast<SplitArgs*>(smem + kArgsOffset);
  for (int i = tid; i < (int)(sizeof(SplitArgs) / 4); i += blockDim.x)
    reinterpret_cast<uint32_t*>(sa)[i] = reinterpret_cast<const uint32_t*>(&a)[i];
  __syncthreads();
  const SplitArgs& A = *sa;
  const int R = a.ring;  // ring slots per tile stream
  // tile streams: one per warp, or one per warp pair
  constexpr int S = split_streams(W, MODE);
  const SmemLayout L = split_smem_layout(D, A.C, A.B, W, A.ring, MODE);

  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  int32_t* pre = reinterpret_cast<int32_t*>(smem + L.pre);
  float* qs = reinterpret_cast<float*>(smem + L.qs);
  int32_t* piece_info = reinterpret_cast<int32_t*>(smem + L.abort_flag);  // [1] len, [2] q0, [3] nq
  int32_t* qlim = reinterpret_cast<int32_t*>(smem + L.qlim);
  __shared__ int32_t scan_scratch[kMaxWarps];

  RowLen len_of;
  if constexpr (kQ) {
    len_of = MultiLen{a.seqlens, a.cu_q, a.nqg, a.tq, a.causal, a.total_q, a.max_q, a.bs, a.maxblk};
  } else {
    len_of = DecodeLen{a.seqlens, a.len_add, a.bs, a.maxblk};
  }

  if (tid == 0) {
    for (int s = 0; s < S * R; ++s) {
      mbar_init(base + L.full + 8 * s, 1);
      if (kPair) mbar_init(base + L.empty + 8 * s, 1);
    }
    if (a.stall_test) mbar_init(base + kStallOffset, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  const uint64_t wait_ns = a.wait_us > 0 ? (uint64_t)a.wait_us * 1000ull : kWaitLimitNs;
  for (int i = tid; i < D / 8; i += blockDim.x) sts128(base + L.zrow + 16u * i, make_uint4(0u, 0u, 0u, 0u));
  if (lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  // Launched as a programmatic dependent of the kernel before it on the
  // stream, this grid may be resident while that kernel finishes: nothing
  // above touches global memory; from here on, that kernel's writes (q,
  // tables, lengths, the pools; the previous merge's reads of the workspace
  // are done) are complete and visible.  Without such a launch this returns
  // at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  build_prefix(a, len_of, pre, scan_scratch);  // contains __syncthreads
  // The merge kernel may be scheduled now; it waits for this grid to finish.
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const SchedShape sched{a.B,           a.Hkv,      a.bs,     a.maxblk,
                         a.part_blocks, (int32_t)gridDim.x, a.len_add, a.piece_k};
  const int cta = blockIdx.x;

  const int w = warp;
  // the warp's tile stream and column group: with warp pairs, warps w and
  // w + W/2 take the same tiles, the lower one issuing their copies
  const int sw = kPair ? w % S : w, cg = kPair ? w / S : 0;
  const bool issuer = !kPair || cg == 0;
  const int cw = warp_columns(D, A.C, MODE);           // columns of a warp state
  const int cl = kPair ? min(cw, A.C - cg * cw) : A.C;  // columns this warp computes
  const int sl = a.bs == 16 ? 0 : (a.bs == 32 ? 1 : 2);  // log2(16-token tiles per block)
  constexpr int NC = D / 64;
  constexpr uint32_t chunk = kTile * 128u;

  // ---- the first piece's q: its copy starts first, so that its latency
  // overlaps the block-table reads of the ring's first tiles
  PieceIterT<RowLen> it;
  it.init(pre, len_of, sched, cta);
  Piece pc;
  bool have = it.next(pc);
  const uint32_t qraw = base + L.qraw;
  QStage<D, kQ> qn;
  if (have) {
    qn.start(*sa, pc, qraw);
    if constexpr (kQ) qn.issue_copies(*sa, pc, qraw);
  }

  // ---- the warp's issuing side: prime the ring with the first R tiles
  IssuerT<RowLen> is;
  is.it.init(pre, len_of, sched, cta);
  is.i = is.cnt = 0;
  is.win = 0;
  is.entry = is.entry_next = 0;
  is.len = 0;
  is.seq = 0;
  is.issued = 0;
  is.done = false;
  if (issuer)
    for (int r = 0; r < R; ++r) issue_next<D>(is, a, *sa, &tmk, &tmv, base, L, sw, S, (uint32_t)r, sl);

  // outputs of rows without keys, and the merge kernel's descriptors: after
  // the first copies are on their way (nothing above depends on them)
  rows_without_keys_and_descriptors<D, kQ>(a, len_of, pre, sched, cta);

  // ---- the computing side
  if (have) cp_async_wait_all();
  __syncthreads();
  if (have) qn.template finish<T, MODE == kSimt, MODE == kMmaW>(*sa, qraw, qs, piece_info, qlim);
  __syncthreads();
  uint32_t slot = 0, phase = 0;  // ring slot to consume next; per-slot parity bits
  uint32_t ephase = 0;           // warp pairs, issuer: per-slot parity of the "empty" barriers
  uint32_t consumed = 0;
  // the first of this warp's tiles whose wait gave up: from there on, copies
  // it issued may still be in flight when the loop ends (see the drain)
  int64_t first_fail = -1;
  bool stall = a.stall_test && w == 0;
  typename std::conditional<MODE == kMmaW, MmaWState<T, D>, MmaState<T, D, NB, kQ>>::type mst;
  SimtState<T, D> sst;
  float* ps = reinterpret_cast<float*>(smem + L.ps) + w * kTile * kGMax;
  while (have) {
    if constexpr (MODE == kMmaW) {
      mst.load_lim(qlim, A.qscale);
      mst.reset();
    } else if constexpr (MODE != kSimt) {
      if constexpr (kPair)
        mst.load_q(qs + cg * cw * (D + 4), cl, qlim + cg * cw, A.qscale);
      else
        mst.load_q(qs, A.C, qlim, A.qscale);
      mst.reset();
    } else {
      sst.reset();
    }
    // the next piece's q starts on its way now
    Piece next;
    bool more;
    {
      PieceIterT<RowLen> peek = it;
      more = peek.next(next);
    }
    if (more) qn.start(*sa, next, qraw);
    bool bad = false;
    const int cnt = stream_tiles(pc, sl, sw, S);
    // fused append: the position of this sequence's new token; the warp
    // whose tile holds it loads the new K/V row now, ahead of that tile
    int32_t new_pos = -1;
    uint4 nk = make_uint4(0u, 0u, 0u, 0u), nv = nk;
    if (a.len_add) {
      const int32_t p0 = *reinterpret_cast<volatile int32_t*>(piece_info + 1);
      const int rel = p0 - pc.blk0 * a.bs;
      if (rel >= 0 && rel < (pc.blk1 - pc.blk0) * a.bs && ((rel >> 4) % S) == sw) {
        new_pos = p0;
        const int64_t src = ((int64_t)pc.b * a.Hkv + pc.j) * D;
        if (lane < D / 8) {
          nk = __ldg(reinterpret_cast<const uint4*>(a.k_new + src) + lane);
          nv = __ldg(reinterpret_cast<const uint4*>(a.v_new + src) + lane);
        }
      }
    }
    for (int i = 0; i < cnt; ++i) {
      const uint32_t gslot = (uint32_t)sw * R + slot;
      // the timeout-path test waits on a barrier nothing completes instead
      const uint32_t wbar = stall ? base + kStallOffset : base + L.full + 8 * gslot;
      const uint32_t wpar = stall ? 0u : (phase >> slot) & 1u;
      stall = false;
      // lanes poll on their own: a give-up seen by one lane counts for the
      // warp, so the warp-wide mma below runs on all lanes or on none
      const bool ok =
          __all_sync(0xffffffffu, mbar_wait_bounded(wbar, wpar, abort_flag, wait_ns));
      if (!ok && first_fail < 0) first_fail = consumed;
      const uint64_t info64 = lds64(base + L.info + 8 * gslot);
      const uint32_t info = (uint32_t)info64;
      const int valid = (int)(info & 0xffffu);
      if (!ok || (info & kInfoBad)) {
        bad = true;
        if (!ok) {
          if (lane == 0) atomicOr(a.status, kStatusTimeout);
          is.done = true;  // stop issuing after a timeout
        }
      } else if (valid > 0) {
        const uint32_t sb = base + L.stage + gslot * L.stage_bytes;
        const uint32_t kb = sb + (a.kv_swap ? NC * chunk : 0u);
        const uint32_t vb = sb + (a.kv_swap ? 0u : NC * chunk);
        const int t = sw + S * i;
        const int tok0 = (pc.blk0 + (t >> sl)) * a.bs + (t & ((1 << sl) - 1)) * kTile;
        int new_r = -1;
        const uint32_t nkr = base + L.nrow + (uint32_t)w * 4u * D, nvr = nkr + 2u * D;
        if (new_pos >= 0) {
          // The tile holding the new token: its row comes from the warp's
          // copy of k_new/v_new, which also goes to the pool slot (no other
          // CTA reads this row).
          const int r = new_pos - tok0;
          if (r >= 0 && r < kTile) {
            const int32_t phys = (int32_t)(info64 >> 32);
            const int64_t dst = (((int64_t)phys * a.bs + (new_pos % a.bs)) * a.Hkv + pc.j) * D;
            if (lane < D / 8) {
              sts128(nkr + lane * 16u, nk);
              sts128(nvr + lane * 16u, nv);
              reinterpret_cast<uint4*>(a.k_pool + dst)[lane] = nk;
              reinterpret_cast<uint4*>(a.v_pool + dst)[lane] = nv;
            }
            __syncwarp();
            new_r = r;
          }
        }
        if constexpr (MODE == kMmaW) {
          mst.tile(kb, vb, valid, tok0, base + L.zrow, base + L.qs);
        } else if constexpr (MODE != kSimt) {
          mst.tile(kb, vb, valid, tok0, new_r, nkr, nvr, base + L.zrow);
        } else {
          sst.tile(kb, vb, valid, qs, ps, a.G, new_r, nkr, nvr);
        }
      }
      __syncwarp();
      phase ^= 1u << slot;
      ++consumed;
      if (issuer) {
        if constexpr (kPair) {
          // the partner warp must be done with this slot before it is refilled
          const bool freed = __all_sync(
              0xffffffffu, mbar_wait_bounded(base + L.empty + 8 * gslot, (ephase >> slot) & 1u,
                                             abort_flag, wait_ns));
          ephase ^= 1u << slot;
          if (!freed) {
            if (lane == 0) atomicOr(a.status, kStatusTimeout);
            is.done = true;  // stop issuing
          }
        }
        issue_next<D>(is, a, *sa, &tmk, &tmv, base, L, sw, S, slot, sl);
      } else if (lane == 0) {
        mbar_arrive(base + L.empty + 8 * gslot);  // this warp is done with the slot
      }
      slot = (slot + 1 == (uint32_t)R) ? 0u : slot + 1;
    }
    if constexpr (kQ) {
      if (more) qn.issue_copies(*sa, next, qraw);
    }
    if constexpr (MODE == kMmaW) {
      mst.bad |= bad;
      mst.template publish<0>(smem, L, w);
    } else if constexpr (MODE != kSimt) {
      mst.bad |= bad;
      if constexpr (kPair)
        mst.publish(smem, L, w, cl, cw);
      else
        mst.publish(smem, L, w, A.C, A.C);
    } else {
      sst.bad |= bad;
      sst.publish(smem, L, w, a.G);
    }
    // this piece's query span, read before the next piece's `finish` may
    // overwrite it
    const int q0 = kQ ? piece_info[2] : 0, nq = kQ ? piece_info[3] : 0;
    cp_async_wait_all();  // this thread's copies of the next q have landed
    named_bar_sync(1, blockDim.x);
    if constexpr (MODE == kMmaW) {
      // a wide row's two m-tiles, folded one after the other through the
      // same 16-column state buffers
      combine_piece<D, W, kQ, false>(*sa, smem, L, pc, q0, nq, 0, 0, min(kColMax, A.C), kColMax);
      if (A.C > kColMax) {
        named_bar_sync(1, blockDim.x);  // m-tile 0's states are read
        mst.template publish<1>(smem, L, w);
        named_bar_sync(1, blockDim.x);
        combine_piece<D, W, kQ, false>(*sa, smem, L, pc, q0, nq, 0, kColMax, A.C - kColMax,
                                       kColMax);
      }
    } else {
      combine_piece<D, W, kQ, kPair>(*sa, smem, L, pc, q0, nq, kPair ? cw : 0);
    }
    if (more) qn.template finish<T, MODE == kSimt, MODE == kMmaW>(*sa, qraw, qs, piece_info, qlim);
    named_bar_sync(1, blockDim.x);
    have = it.next(pc);
  }
  if (first_fail >= 0 && lane == 0) {
    // Drain: wait (bounded, ignoring the abort flag) for this warp's copies
    // that may still be in flight before the CTA may exit.  Tile n of the
    // warp's stream sits in ring slot n % R in phase (n / R) & 1.  Before
    // the first give-up every issued tile was waited for; after it nothing
    // more was issued, so tiles first_fail .. issued-1 (at most R, one per
    // slot) are the ones to wait for -- each slot's phase completes once
    // more at most, so waiting on a tile already consumed returns at once.
    volatile int never = 0;
    for (int64_t kk = first_fail; kk < (int64_t)is.issued; ++kk)
      mbar_wait_bounded(base + L.full + 8 * ((uint32_t)sw * R + (uint32_t)(kk % R)),
                        (uint32_t)((kk / R) & 1), &never, kWaitLimitNs / 4);
  }
}

template <typename T, int D, int MODE>
cudaError_t launch_split(const CUtensorMap& tmk, const CUtensorMap& tmv, const SplitArgs& a,
                         int grid, int threads, size_t smem, cudaStream_t stream) {
  // a programmatic dependent of the previous kernel on the stream: its CTAs
  // may be scheduled (and run up to griddepcontrol.wait) while that kernel
  // drains, which hides the launch gap between consecutive decode steps
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pa_split_kernel<T, D, MODE>, tmk, tmv, a);
}

template <typename T, int D, int MODE>
const void* split_kernel_ptr() {
  return reinterpret_cast<const void*>(&pa_split_kernel<T, D, MODE>);
}

}  // namespace pa

#define PA_INSTANTIATE_SPLIT(T, D, MODE)                                                     \
  template cudaError_t pa::launch_split<T, D, MODE>(const CUtensorMap&, const CUtensorMap&,  \
                                                    const pa::SplitArgs&, int, int, size_t,  \
                                                    cudaStream_t);                           \
  template const void* pa::split_kernel_ptr<T, D, MODE>();
