// pa_split_tc.cuh -- phase 1 on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory), head dimension 128.
//
// Same schedule, pieces, partial states and outputs as pa_split.cuh; the
// tiles are 128 tokens and the products run as tcgen05.mma issued by one
// thread:
//   S[128 tokens x 16 columns]  = K[128 x 128] . q^T          (TMEM, fp32)
//   O^T[128 dims x 16 columns] += V^T[128 x 128] . P^T         (TMEM, fp32)
// with K and V straight from the TMA stage (K as a K-major operand, V as an
// MN-major one), q and P (high and low 16-bit parts) written to shared
// memory by the softmax threads.  A column is a query head (decode) or a
// (query token, head) pair of one sequence (several query tokens).
//
// Warps 0-3 (128 threads) own the 128 TMEM lanes: thread t holds token t of
// a tile's scores and dimension t of the accumulator.  Warps 4 and 6 issue
// the TMA copies of K and of V (one per block and 64-dim chunk) into two
// rings: a K slot is free again as soon as the tile's scores are computed,
// a V slot only after the O update, so the V ring is the deeper one.  Warp
// 5 issues the MMAs.
//
// Online softmax per column ("v10_triton_paged_gqa", Core Principle) in log2
// units with a lazy running max: the max moves only when a tile's scores
// exceed it by more than tc_lazy_max, so the column maxima over the 128 tokens
// (a cross-thread reduction) and the rescale of the accumulator in TMEM are
// needed only then; each thread keeps its own part of every column's
// exp-sum, reduced once per piece.
#pragma once

#include "pa_kernels.cuh"
#include "pa_ptx.cuh"
#include "pa_split.cuh"

namespace pa {

// Slack of the running max (log2 units).  The accumulator lives in tensor
// memory, where a rescale costs a round trip and a wait for the previous
// products, so the max moves only on large jumps: p stays below 2^24 with
// bf16 operands (the high + low split keeps ~16 significant bits at any
// magnitude, and an exp-sum of up to 2^20 such terms stays far inside fp32)
// and below 2^14 with fp16 ones (whose largest finite value is ~2^16).
template <typename T>
__device__ __forceinline__ constexpr float tc_lazy_max() {
  return std::is_same<T, __nv_bfloat16>::value ? 24.f : 14.f;
}

// Offset of the 16-bit element (row, col) of a [rows][128] operand stored
// as two 128B-swizzled [rows][64] chunks of rows*128 bytes each.
__device__ __forceinline__ uint32_t tc_op_offset(int row, int col, uint32_t chunk_bytes) {
  const int c = col & 63;
  return (uint32_t)(col >> 6) * chunk_bytes + swz((uint32_t)row, (uint32_t)(c >> 3)) +
         (uint32_t)(c & 7) * 2u;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// The 128-token tiles of a piece.  bs divides 128, so rounding the piece's
// blocks up to tiles gives the same count as rounding its tokens (which end
// at the row's length inside the last block): the producers and the MMA
// thread need no length.
__device__ __forceinline__ int tc_tiles(const Piece& pc, int bs) {
  return ((pc.blk1 - pc.blk0) * bs + kTcTile - 1) / kTcTile;
}

// The columns of one piece: where their q rows come from (and their
// outputs go), and up to which key each one sees.
template <bool kQ>
struct TcColumns {
  int32_t len;      // the sequence's stored key length
  int32_t row_len;  // keys the row reads: the length, or the limit of its last token
  int32_t q0, nq;   // several query tokens: the sequence's query rows
  int32_t grp;      // several query tokens: the row's group

  __device__ __forceinline__ void setup(const SplitArgs& a, const Piece& pc) {
    if constexpr (!kQ) {
      len = __ldg(a.seqlens + pc.b);
      row_len = len;
      q0 = 0;
      nq = 1;
      grp = 0;
    } else {
      const int seq = pc.b / a.nqg;
      grp = pc.b - seq * a.nqg;
      len = __ldg(a.seqlens + seq);
      query_span(a.cu_q, seq, a.total_q, a.max_q, q0, nq);
      // as MultiLen: the row's pieces exist only for a valid length and span
      const int first = grp * a.tq, last = min(nq, first + a.tq) - 1;
      row_len = a.causal ? max(0, min(len, len - nq + last + 1)) : len;
    }
  }

  // Row of q and out ([rows][H] index) of column c, or -1: no query there.
  __device__ __forceinline__ int64_t row(const SplitArgs& a, const Piece& pc, int c) const {
    if (c >= a.C) return -1;
    if constexpr (!kQ) {
      return (int64_t)pc.b * a.H + (int64_t)pc.j * a.G + c;
    } else {
      const int tok = grp * a.tq + c / a.G;
      if (tok >= nq) return -1;
      return (int64_t)(q0 + tok) * a.H + (int64_t)pc.j * a.G + c % a.G;
    }
  }

  // Keys t < limit are visible to column c.
  __device__ __forceinline__ int32_t limit(const SplitArgs& a, int c) const {
    if constexpr (!kQ) {
      return 0x7fffffff;
    } else {
      const int tok = grp * a.tq + c / a.G;
      if (c >= a.C || tok >= nq || !a.causal) return 0x7fffffff;
      return max(0, min(len, len - nq + tok + 1));
    }
  }
};

// q of the piece's 16 columns (zero where a column holds no query), 256
// units of 8 dims, two per softmax thread: loaded into registers early,
// stored later into the K-major B operand at qdst.
template <bool kQ>
__device__ __forceinline__ void tc_load_q(const SplitArgs& a, const Piece& pc,
                                          const TcColumns<kQ>& cols, uint4 (&v)[2]) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int u = (int)threadIdx.x + 128 * k;
    const int c = u >> 4, d8 = (u & 15) * 8;
    const int64_t r = cols.row(a, pc, c);
    v[k] = make_uint4(0u, 0u, 0u, 0u);
    if (r >= 0) v[k] = __ldg(reinterpret_cast<const uint4*>(a.q + r * kTcD + d8));
  }
}

__device__ __forceinline__ void tc_store_q(const uint4 (&v)[2], uint32_t qdst) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int u = (int)threadIdx.x + 128 * k;
    const int c = u >> 4, d8 = (u & 15) * 8;
    sts128(qdst + (uint32_t)(d8 >> 6) * (kTcOpBytes / 2) + swz((uint32_t)c, (uint32_t)((d8 & 63) >> 3)),
           v[k]);
  }
}

// ---------------------------------------------------------------- producers

// Warp 4 (K) and warp 6 (V): walk the CTA's pieces and tiles and load each
// tile's K (or V) rows into the next slot of their ring once the products
// that used it are done (the scores for K, the O update for V).  Lane
// i < 128/bs reads the table entry of the tile's i-th block and issues its
// two copies (one per 64-dim chunk), each bs rows landing at row i*bs of the
// slot's [128][64] chunks.  Blocks with a bad entry are skipped and flagged;
// their rows are never used (the softmax flags the piece from the same
// entries); the K producer sets the status bit.
template <bool kQ, bool kV, class LenOf>
__device__ __forceinline__ void tc_producer(const SplitArgs& A, PieceIterT<LenOf> it,
                                            const CUtensorMap* map, uint32_t base, const TcLayout& L,
                                            int NV, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first_policy();  // K/V rows are read once per step
  const int bs = A.bs, bpt = kTcTile / bs;
  const int N = kV ? NV : kTcKStages;
  const uint32_t bars = base + L.bars;
  const uint32_t ring = base + (kV ? L.v : L.k);
  uint32_t i = 0;
  bool ok = true;
  Piece pc;
  while (ok && it.next(pc)) {
    const int seq = kQ ? pc.b / A.nqg : pc.b;
    const int ntiles = tc_tiles(pc, bs);
    for (int t = 0; t < ntiles; ++t, ++i) {
      const int s = (int)(i % (uint32_t)N);
      if (i >= (uint32_t)N) {
        int w = 1;
        if (lane == 0)
          w = mbar_wait_bounded(bars + (kV ? TcBars::empty_v(s) : TcBars::empty_k(s)), ((i / N) - 1) & 1u,
                                abort_flag, kWaitLimitNs);
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) break;
      }
      const int blk = pc.blk0 + t * bpt;
      const int nb = min(bpt, pc.blk1 - blk);
      int32_t phys = 0;
      if (lane < nb) phys = __ldg(A.table + (int64_t)seq * A.maxblk + blk + lane);
      const bool bad = lane < nb && (phys < 0 || phys >= A.P);
      const unsigned badm = __ballot_sync(0xffffffffu, bad);
      const unsigned goodm = __ballot_sync(0xffffffffu, lane < nb && !bad);
      const uint32_t full = bars + (kV ? TcBars::full_v(s) : TcBars::full_k(s));
      if (lane == 0) {
        if (!kV && badm) atomicOr(A.status, kStatusBadBlock);
        const uint32_t bytes = (uint32_t)__popc(goodm) * 2u * (uint32_t)bs * 128u;
        if (bytes)
          mbar_arrive_expect_tx(full, bytes);
        else
          mbar_arrive(full);
      }
      __syncwarp();
      if (lane < nb && !bad) {
        const uint32_t st = ring + (uint32_t)s * kTcHalfBytes + (uint32_t)(lane * bs) * 128u;
#pragma unroll
        for (int c = 0; c < kTcD / 64; ++c)
          tma_load_5d(st + (uint32_t)c * kTcChunk, map, full, 0, 0, c, pc.j, phys, pol);
      }
    }
  }
  // Normally nothing is pending here; after a timeout the copies of the last
  // N tiles must still land (bounded wait) before the CTA may exit.
  if (lane == 0) {
    volatile int never = 0;
    for (uint32_t k = i > (uint32_t)N ? i - N : 0; k < i; ++k)
      mbar_wait_bounded(bars + (kV ? TcBars::full_v((int)(k % N)) : TcBars::full_k((int)(k % N))),
                        (k / N) & 1u, &never, kWaitLimitNs / 4);
  }
}

// ------------------------------------------------------------- MMA issuer

// One thread of warp 5.  S(k) = K . q^T goes into S buffer k%2 once K slot
// k%2 has landed and the softmax has read that buffer's previous scores;
// it is issued one tile ahead, so the tensor cores compute the next tile's
// scores while the softmax works on this one.  Once the softmax has written
// P, [O_hi O_lo]^T += V^T . [P_hi P_lo]^T (the first product of a piece
// overwrites O, after the previous piece's O has been read).  Completion is
// signalled with tcgen05.commit: S ready and K slot free, V slot and P
// buffer free.
// tcgen05.mma without a memory clobber: the MMA thread touches shared memory
// only through the mbarrier operations, which keep their own ordering.  A
// descriptor's start address (bits 0-13, in 16-byte units) advances by a
// constant per k-step, so the loops add to one descriptor instead of
// rebuilding it (addresses stay below 2^18 bytes: no carry out of the field).
__device__ __forceinline__ void tc_umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}

template <typename T, class LenOf>
__device__ __forceinline__ void tc_mma(const SplitArgs& A, PieceIterT<LenOf> it, uint32_t base,
                                       const TcLayout& L, int NV, uint32_t tmem,
                                       volatile int* abort_flag) {
  constexpr int bf = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
  constexpr uint32_t idS = idesc_f16(bf, 0, 0, kTcTile, kTcN);  // A = K tile, K-major
  // A = V^T, MN-major; B = P with its high and low parts as 32 columns, so
  // one product per k-step accumulates O_hi and O_lo side by side
  constexpr uint32_t idO = idesc_f16(bf, 1, 0, kTcTile, 2 * kTcN);
  constexpr uint32_t opc = kTcOpBytes / 2;                      // chunk of a q operand
  const uint32_t bars = base + L.bars;
  auto issue_s = [&](uint32_t k, uint32_t qop) -> bool {
    const int s = (int)(k % (uint32_t)kTcKStages), sb = (int)(k & 1u);
    if (!mbar_wait_bounded(bars + TcBars::full_k(s), (k / kTcKStages) & 1u, abort_flag, kWaitLimitNs))
      return false;
    if (k >= 2 &&
        !mbar_wait_bounded(bars + TcBars::s_free(sb), ((k - 2) / 2) & 1u, abort_flag, kWaitLimitNs))
      return false;
    tc_fence_after();
    const uint32_t kst = base + L.k + (uint32_t)s * kTcHalfBytes;
    const uint64_t a0 = sdesc_sw128(kst, 16, 1024), b0 = sdesc_sw128(qop, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < kTcD / 16; ++ks)  // 32 bytes per k-step, 64 dims per chunk
      tc_umma(tmem + 16u * sb, a0 + (uint64_t)((ks >> 2) * (kTcChunk >> 4) + (ks & 3) * 2),
              b0 + (uint64_t)((ks >> 2) * (opc >> 4) + (ks & 3) * 2), idS, ks > 0);
    umma_commit(bars + TcBars::s_full(sb));
    umma_commit(bars + TcBars::empty_k(s));
    return true;
  };
  auto issue_pv = [&](uint32_t k, bool first) -> bool {
    const int s = (int)(k % (uint32_t)NV), sb = (int)(k & 1u);
    if (!mbar_wait_bounded(bars + TcBars::full_v(s), (k / NV) & 1u, abort_flag, kWaitLimitNs)) return false;
    if (!mbar_wait_bounded(bars + TcBars::p_full(sb), (k / 2) & 1u, abort_flag, kWaitLimitNs)) return false;
    tc_fence_after();
    const uint32_t vst = base + L.v + (uint32_t)s * kTcHalfBytes;
    const uint32_t pb = base + L.p + (uint32_t)sb * kTcPBytes;
    // V^T: 64-dim blocks one chunk apart, 8-token groups 1 KB apart
    const uint64_t a0 = sdesc_sw128(vst, kTcChunk, 1024), b0 = sdesc_sw128(pb, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < kTcTile / 16; ++ks)
      tc_umma(tmem + 32u, a0 + (uint64_t)(ks * (2048 >> 4)),
              b0 + (uint64_t)((ks >> 2) * ((kTcPBytes / 2) >> 4) + (ks & 3) * 2), idO,
              (first && ks == 0) ? 0u : 1u);
    umma_commit(bars + TcBars::empty_v(s));
    umma_commit(bars + TcBars::p_free(sb));
    return true;
  };
  uint32_t i = 0, piece = 0;
  bool ok = true;
  Piece pc;
  while (ok && it.next(pc)) {
    const int ntiles = tc_tiles(pc, A.bs);
    ok = mbar_wait_bounded(bars + TcBars::q_ready(), piece & 1u, abort_flag, kWaitLimitNs);
    if (ok) {
      tc_fence_after();
      const uint32_t qop = base + L.q + (piece & 1u) * kTcOpBytes;
      ok = issue_s(i, qop);
      for (int t = 0; t < ntiles && ok; ++t, ++i) {
        if (t + 1 < ntiles) ok = issue_s(i + 1, qop);
        if (ok && t == 0 && piece > 0)
          ok = mbar_wait_bounded(bars + TcBars::o_free(), (piece - 1) & 1u, abort_flag, kWaitLimitNs);
        if (ok) ok = issue_pv(i, t == 0);
        if (!ok) break;
      }
    }
    ++piece;
  }
  // every product issued has completed before the tensor memory is released
  umma_commit(bars + TcBars::drain());
  volatile int never = 0;
  mbar_wait_bounded(bars + TcBars::drain(), 0, &never, kWaitLimitNs / 4);
}

// ---------------------------------------------------------------- softmax

// Warps 0-3.  Per piece: stage q, then per tile read S (thread t = token t),
// scale and mask, update the lazy running max (column maxima over the tile
// only when some score is above max + tc_lazy_max), write p = 2^(s - m) as the
// P operands (high and low parts), and zero the V rows past the valid
// tokens so that p = 0 never meets stale data.  At the piece end, read O
// (thread t = dimension t), reduce the exp-sums and write the output or the
// partial state.
// NC: the columns that can hold a query (C <= NC <= kTcN); the P rows of
// the others are zeroed once and never written again.
template <typename T, bool kQ, int NC, class LenOf>
__device__ __forceinline__ void tc_softmax(const SplitArgs& A, PieceIterT<LenOf> it, uint32_t base,
                                           uint8_t* smem, const TcLayout& L, int NV, uint32_t tmem,
                                           volatile int* abort_flag) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t bars = base + L.bars;
  const uint32_t lanes = tmem + ((uint32_t)(32 * warp) << 16);  // this warp's TMEM lanes
  float* red = reinterpret_cast<float*>(smem + L.red);
  const float qscale = A.qscale;
  const int C = A.C;
  const float qnan = __int_as_float(0x7fc00000);
  uint32_t i = 0, piece = 0;
  Piece pc;
  TcColumns<kQ> cols;
  if constexpr (NC < kTcN) {
    // both P buffers start at zero: the rows of columns >= NC stay so
    for (uint32_t off = 16u * (uint32_t)t; off < 2u * kTcPBytes; off += 16u * 128u)
      sts128(base + L.p + off, make_uint4(0u, 0u, 0u, 0u));
  }
  bool have = it.next(pc);
  if (have) {
    cols.setup(A, pc);
    uint4 qv[2];
    tc_load_q<kQ>(A, pc, cols, qv);
    tc_store_q(qv, base + L.q);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (have && lane == 0) mbar_arrive(bars + TcBars::q_ready());
  while (have) {
    // the next piece; its q is loaded during this piece's first tile and
    // stored after the last one, so its score products need not wait for
    // this piece's epilogue
    PieceIterT<LenOf> nit = it;
    Piece nx;
    const bool more = nit.next(nx);
    TcColumns<kQ> ncols;
    uint4 nqv[2];
    int32_t lim[NC];
    float m[NC], lp[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      lim[c] = cols.limit(A, c);
      m[c] = -INFINITY;
      lp[c] = 0.f;
    }
    bool bad = false;
    const int ntiles = tc_tiles(pc, A.bs);
    const int tok_begin = pc.blk0 * A.bs;
    const int tok_end = min(pc.blk1 * A.bs, cols.row_len);
    const int bpt = kTcTile / A.bs;
    const int seq = kQ ? pc.b / A.nqg : pc.b;
    int32_t phys_pend = 0;  // the previous tile's table entry of this thread's block
    int nb_pend = 0;
    for (int tt = 0; tt < ntiles; ++tt, ++i) {
      const int sb = (int)(i & 1u);
      // The tile's tokens, and its blocks' table entries (checked one tile
      // later, or at the piece's end, so the load's latency is hidden).  No
      // wait on the K slot here: a K slot is reloaded as soon as the scores
      // are computed, so its barrier may run two phases ahead of this thread.
      const int tok0 = tok_begin + tt * kTcTile;
      const int valid = max(0, min(kTcTile, tok_end - tok0));
      const int blk = pc.blk0 + tt * bpt, nb = min(bpt, pc.blk1 - blk);
      int32_t phys = 0;
      if (t < nb) phys = __ldg(A.table + (int64_t)seq * A.maxblk + blk + t);
      bool ok = mbar_wait_bounded(bars + TcBars::s_full(sb), (i / 2) & 1u, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      float sc[kTcN];
      if (ok) {
        tc_fence_after();
        tmem_ld16(lanes + 16u * sb, sc);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + TcBars::s_free(sb));
      if (!ok) bad = true;
      const bool in = t < valid;
      const int tok = tok0 + t;
      bool need = false;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float x = ok ? sc[c] * qscale : -INFINITY;
        if (!in || tok >= lim[c]) x = -INFINITY;
        sc[c] = x;
        need |= x > m[c] + tc_lazy_max<T>();
      }
      if (named_bar_or(1, 128, need)) {
        // the tile's column maxima: warp trees, then the four warps in order
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          float v = sc[c];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
          if (lane == 0) red[warp * kTcN + c] = v;
        }
        named_bar_sync(2, 128);
        float al[NC];
        bool moved = false;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float tm = fmaxf(fmaxf(red[c], red[kTcN + c]), fmaxf(red[2 * kTcN + c], red[3 * kTcN + c]));
          const float nm = tm > m[c] + tc_lazy_max<T>() ? tm : m[c];
          al[c] = (m[c] == -INFINITY) ? 0.f : ex2(m[c] - nm);
          moved |= al[c] != 1.f;
          lp[c] *= al[c];
          m[c] = nm;
        }
        if (moved && tt > 0) {
          // O holds this piece's earlier tiles: rescale it in TMEM once the
          // previous tile's products are complete
          const uint32_t pi = i - 1;
          bool ok2 = mbar_wait_bounded(bars + TcBars::p_free((int)(pi & 1u)), (pi / 2) & 1u, abort_flag,
                                       kWaitLimitNs);
          ok2 = __all_sync(0xffffffffu, ok2);
          if (ok2) {
            tc_fence_after();
            float oh[kTcN], ol[kTcN];
            tmem_ld16(lanes + 32u, oh);
            tmem_ld16(lanes + 48u, ol);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              oh[c] *= al[c];
              ol[c] *= al[c];
            }
            tmem_st16(lanes + 32u, oh);
            tmem_st16(lanes + 48u, ol);
            tmem_st_wait();
            tc_fence_before();
          } else {
            bad = true;
          }
        }
      }
      // P buffer sb is free once the products of tile i - 2 are complete
      if (i >= 2) {
        bool ok3 = mbar_wait_bounded(bars + TcBars::p_free(sb), ((i - 2) / 2) & 1u, abort_flag, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok3)) bad = true;
      }
      const uint32_t pbuf = base + L.p + (uint32_t)sb * kTcPBytes;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const float u = (m[c] == -INFINITY) ? 0.f : m[c];
        const float pv = ex2(sc[c] - u);
        lp[c] += pv;
        const uint32_t hi = Cvt<T>::pack(pv, 0.f) & 0xffffu;
        const uint32_t lo = Cvt<T>::pack(pv - Cvt<T>::low(hi), 0.f) & 0xffffu;
        sts16(pbuf + tc_op_offset(c, t, kTcPBytes / 2), (uint16_t)hi);
        sts16(pbuf + tc_op_offset(kTcN + c, t, kTcPBytes / 2), (uint16_t)lo);
      }
      if (valid < kTcTile) {
        // V rows past the valid tokens are zeroed once the tile's V has
        // landed (the same for every thread: valid is the tile's)
        const int sv = (int)(i % (uint32_t)NV);
        bool okv = mbar_wait_bounded(bars + TcBars::full_v(sv), (i / NV) & 1u, abort_flag, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, okv)) bad = true;
        if (!in) {
          const uint32_t vrow = base + L.v + (uint32_t)sv * kTcHalfBytes + (uint32_t)t * 128u;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              sts128(vrow + (uint32_t)c2 * kTcChunk + 16u * u, make_uint4(0u, 0u, 0u, 0u));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + TcBars::p_full(sb));
      if (t < nb_pend && (phys_pend < 0 || phys_pend >= A.P)) bad = true;
      phys_pend = phys;
      nb_pend = nb;
      if (tt == 0 && more) {
        ncols.setup(A, nx);
        tc_load_q<kQ>(A, nx, ncols, nqv);
      }
      if (tt == ntiles - 1 && more) {
        // the buffer's previous reader, the score products of piece - 1, has
        // completed (their scores were all read)
        tc_store_q(nqv, base + L.q + ((piece + 1) & 1u) * kTcOpBytes);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + TcBars::q_ready());
      }
    }
    // ---- the piece's result: O (thread t = dimension t) over the exp-sums
    if (t < nb_pend && (phys_pend < 0 || phys_pend >= A.P)) bad = true;
    const uint32_t last = i - 1;
    bool ok = mbar_wait_bounded(bars + TcBars::p_free((int)(last & 1u)), (last / 2) & 1u, abort_flag,
                                kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    float o[kTcN], ol[kTcN];
    if (ok) {
      tc_fence_after();
      tmem_ld16(lanes + 32u, o);
      tmem_ld16(lanes + 48u, ol);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < NC; ++c) o[c] += ol[c];
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + TcBars::o_free());  // the next piece may overwrite O
    named_bar_sync(2, 128);  // every thread is done with the maxima scratch
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float v = lp[c];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) red[warp * kTcN + c] = v;
    }
    const bool any_bad = named_bar_or(1, 128, bad || !ok);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      if (c >= C) continue;
      const float l = (red[c] + red[kTcN + c]) + (red[2 * kTcN + c] + red[3 * kTcN + c]);
      const int64_t r = cols.row(A, pc, c);
      if (r < 0) continue;
      if (pc.slot < 0) {
        A.out[r * kTcD + t] = any_bad ? qnan : (l == 0.f ? 0.f : o[c] / l);
      } else {
        A.ws_acc[((int64_t)pc.slot * C + c) * kTcD + t] = any_bad ? qnan : o[c];
        if (t == 0) {
          A.ws_ml[((int64_t)pc.slot * C + c) * 2 + 0] = m[c];
          A.ws_ml[((int64_t)pc.slot * C + c) * 2 + 1] = any_bad ? qnan : l;
        }
      }
    }
    it = nit;
    pc = nx;
    cols = ncols;
    have = more;
    ++piece;
  }
}

// ------------------------------------------------------------------ kernel

template <typename T, bool kQ, int NC>
__global__ void __launch_bounds__(kTcThreads, 1)
    pa_split_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ SplitArgs a) {
  using RowLen = typename std::conditional<kQ, MultiLen, DecodeLen>::type;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NV = a.ring;  // V slots
  const TcLayout L = tc_smem_layout(a.B, NV);
  // the arguments, read by the once-per-piece code, from shared memory
  SplitArgs* sa = reinterpret_cast<SplitArgs*>(smem + L.args);
  for (int i = tid; i < (int)(sizeof(SplitArgs) / 4); i += blockDim.x)
    reinterpret_cast<uint32_t*>(sa)[i] = reinterpret_cast<const uint32_t*>(&a)[i];
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  int32_t* pre = reinterpret_cast<int32_t*>(smem + L.pre);
  __shared__ int32_t scan_scratch[kMaxWarps];
  RowLen len_of;
  if constexpr (kQ) {
    len_of = MultiLen{a.seqlens, a.cu_q, a.nqg, a.tq, a.causal, a.total_q, a.max_q, a.bs, a.maxblk};
  } else {
    len_of = DecodeLen{a.seqlens, 0, a.bs, a.maxblk};
  }
  const uint32_t bars = base + L.bars;
  if (tid == 0) {
    for (int s = 0; s < kTcKStages; ++s) {
      mbar_init(bars + TcBars::full_k(s), 1);
      mbar_init(bars + TcBars::empty_k(s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bars + TcBars::full_v(s), 1);
      mbar_init(bars + TcBars::empty_v(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars + TcBars::s_full(b), 1);
      mbar_init(bars + TcBars::s_free(b), 4);
      mbar_init(bars + TcBars::p_full(b), 4);
      mbar_init(bars + TcBars::p_free(b), 1);
    }
    mbar_init(bars + TcBars::q_ready(), 4);
    mbar_init(bars + TcBars::o_free(), 4);
    mbar_init(bars + TcBars::drain(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(base + L.tbase, kTcTmemCols);
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  tc_fence_before();
  // a programmatic dependent of the previous kernel on the stream: nothing
  // above touches global memory
  asm volatile("griddepcontrol.wait;" ::: "memory");
  build_prefix(a, len_of, pre, scan_scratch);  // contains __syncthreads
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L.tbase);
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const SchedShape sched{a.B, a.Hkv, a.bs, a.maxblk, a.part_blocks, (int32_t)gridDim.x, 0, a.piece_k};
  const int cta = blockIdx.x;
  rows_without_keys_and_descriptors<kTcD, kQ>(a, len_of, pre, sched, cta);
  PieceIterT<RowLen> it;
  it.init(pre, len_of, sched, cta);
  const SplitArgs& A = *sa;
  if (warp < 4) {
    tc_softmax<T, kQ, NC>(A, it, base, smem, L, NV, tmem, abort_flag);
  } else if (warp == 4) {
    tc_producer<kQ, false>(A, it, &tmk, base, L, NV, abort_flag);
  } else if (warp == 6) {
    tc_producer<kQ, true>(A, it, &tmv, base, L, NV, abort_flag);
  } else if (lane == 0) {
    tc_mma<T>(A, it, base, L, NV, tmem, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) atomicOr(a.status, kStatusTimeout);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// The softmax's live columns for C query columns: several query tokens fill
// all 16; decode takes 4 or 8 (C = G).
PA_HD constexpr int tc_live_columns(bool several, int C) {
  return several ? kTcN : (C <= 4 ? 4 : (C <= 8 ? 8 : kTcN));
}

template <typename T, bool kQ>
cudaError_t launch_split_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const SplitArgs& a,
                            int grid, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (tc_live_columns(kQ, a.C)) {
    case 4: return cudaLaunchKernelEx(&cfg, pa_split_tc_kernel<T, kQ, kQ ? kTcN : 4>, tmk, tmv, a);
    case 8: return cudaLaunchKernelEx(&cfg, pa_split_tc_kernel<T, kQ, kQ ? kTcN : 8>, tmk, tmv, a);
    default: return cudaLaunchKernelEx(&cfg, pa_split_tc_kernel<T, kQ, kTcN>, tmk, tmv, a);
  }
}

template <typename T, bool kQ>
const void* split_tc_kernel_ptr(int C) {
  switch (tc_live_columns(kQ, C)) {
    case 4: return reinterpret_cast<const void*>(&pa_split_tc_kernel<T, kQ, kQ ? kTcN : 4>);
    case 8: return reinterpret_cast<const void*>(&pa_split_tc_kernel<T, kQ, kQ ? kTcN : 8>);
    default: return reinterpret_cast<const void*>(&pa_split_tc_kernel<T, kQ, kTcN>);
  }
}

}  // namespace pa

#define PA_INSTANTIATE_SPLIT_TC(T, KQ)                                                         \
  template cudaError_t pa::launch_split_tc<T, KQ>(const CUtensorMap&, const CUtensorMap&,     \
                                                  const pa::SplitArgs&, int, size_t,          \
                                                  cudaStream_t);                              \
  template const void* pa::split_tc_kernel_ptr<T, KQ>(int);
