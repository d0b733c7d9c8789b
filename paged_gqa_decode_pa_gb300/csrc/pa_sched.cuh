// pa_sched.cuh -- how the persistent split kernel divides one decode step's
// work among its CTAs, and how the merge kernel finds the pieces again.
// Compiled for host and device so that pa_plan_pieces (host) and the kernels
// run the very same code.
//
// Work unit: one physical block of one (row b, kv head j) "segment".
// Segment (b, j) holds nblk_b = ceil(len_b / bs) units.  A row is one
// sequence in decode; with several query tokens per sequence it is one
// group of a sequence's query tokens, and len_b the keys that group reads.
//
// Balanced split (partition_tokens == 0): every non-empty segment is
// charged K extra "overhead units" ahead of its blocks -- a piece costs a
// fixed amount (publishing, folding and writing the warp states, loading the
// next q) on top of its blocks, so a CTA that holds many short segments must
// get fewer blocks.  Units are ordered (b, j, [K overhead units, blocks]);
// CTA c of C_eff owns units [floor(V c / C_eff), floor(V (c+1) / C_eff)),
// V = Hkv * sum_b (nblk_b + K [nblk_b > 0]), and processes the blocks in its
// range.  A CTA's range cuts at most two segments (its first and its last
// piece), so each CTA writes at most two partial states: slot 2c (its first
// piece, when that continues a segment begun in an earlier CTA) and slot
// 2c+1 (its last piece, when that begins here and continues past the range).
// A segment that lies inside one CTA is finished there and written straight
// to `out`.
//
// Fixed split (partition_tokens > 0, part_blocks = partition_tokens / bs):
// segment (b, j) has np_b = ceil(nblk_b / part_blocks) partitions; items are
// ordered (b, partition, j) so the Hkv sibling heads of one partition are
// adjacent and CTAs c, c+1, ... read the same physical blocks together.
// CTA c takes items c, c + C, c + 2C, ...; item i writes partial slot i
// (or `out` directly when np_b == 1).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define PA_HD __host__ __device__ __forceinline__
#else
#define PA_HD inline
#endif

namespace pa {

// Fewest units (blocks) a CTA of the balanced split is given: avoids
// spreading tiny steps over many CTAs whose fixed costs would dominate.
constexpr int kMinUnitsPerCta = 4;

struct SchedShape {
  int32_t B, Hkv, bs, maxblk;
  int32_t part_blocks;  // 0 = balanced
  int32_t num_ctas;     // launched persistent grid
  int32_t len_add;      // 1 when the step also appends each sequence's new token
  int32_t K;            // balanced split: overhead units charged per segment
};

// Overhead units per segment of the balanced split: a piece's fixed cost in
// units of one block of one kv head (4 bs D bytes of K and V).  Measured
// best on GB300 at about 200 KB worth (sweeps of 60 to 320 KB on the serving
// and prefix-sharing steps; long context does not move).  With several query
// tokens per sequence a piece's fold and q cover up to 16 columns and cost
// more: measured best at about 360 KB (sweeps of 120 to 600 KB on the 4-token
// serving step and the 2-token prefix-sharing step; on one box the 4-token
// serving split took 510.7 us at 360 against 519.6 at 300, 513.8 at 340,
// 512.2 at 380, 523.2 at 460 and 537.1 at 220, and 2-token prefix sharing
// 186.6 against 185.9 at 300).  Rows of warp pairs (up
// to 32 columns) spend twice the compute on every block, so the same piece
// cost is fewer blocks' worth: best at about 220 KB (sweep of 40 to 440 KB on
// the 8-token serving step: 906 us against 990 at 440 KB).  Wide rows (one
// warp per row of up to 32 columns, folded in two halves) are best at about
// 380 KB (8-token serving split on one box: 653.8 us, against 656.0 at 350,
// 659.5 at 410, 665.6 at 320, 666.7 at 440, 682.5 at 520 and 694.0 at 260;
// the 6-token step and 4-token prefix sharing agree).
constexpr int32_t kPieceKb = 200;
constexpr int32_t kPieceKbMulti = 360;
constexpr int32_t kPieceKbPair = 220;
constexpr int32_t kPieceKbWide = 380;
PA_HD int32_t piece_units(int32_t bs, int32_t D, int32_t kb = kPieceKb) {
  const int32_t unit = 4 * bs * D;
  const int32_t k = (kb * 1024 + unit / 2) / unit;
  return k < 1 ? 1 : k;
}

// Blocks of a sequence; lengths outside [0, maxblk*bs] count as empty (the
// kernels flag them separately).
PA_HD int32_t seq_blocks(int32_t len, int32_t bs, int32_t maxblk) {
  if (len <= 0 || (int64_t)len > (int64_t)maxblk * bs) return 0;
  return (len + bs - 1) / bs;
}

PA_HD bool seq_len_valid(int32_t len, int32_t bs, int32_t maxblk) {
  return len >= 0 && (int64_t)len <= (int64_t)maxblk * bs;
}

// The length a step attends to: the stored length plus `add` (1 when the
// step also appends the new token), or -1 when that is not a valid length.
PA_HD int32_t eff_len(int32_t stored, int32_t add, int32_t bs, int32_t maxblk) {
  if (stored < 0) return -1;
  const int64_t e = (int64_t)stored + add;
  return e > (int64_t)maxblk * bs ? -1 : (int32_t)e;
}

// Per-row count that the prefix sums run over: partitions (fixed split), or
// blocks plus the K overhead units of a non-empty segment (balanced split).
PA_HD int32_t seq_count(int32_t nblk, int32_t part_blocks, int32_t K) {
  if (part_blocks > 0) return (nblk + part_blocks - 1) / part_blocks;
  return nblk > 0 ? nblk + K : 0;
}

// Largest b in [0, B) with mult * pre[b] <= x, for x < mult * pre[B]
// (pre is non-decreasing with pre[0] == 0).
PA_HD int32_t find_seq(const int32_t* pre, int32_t B, int64_t mult, int64_t x) {
  int32_t lo = 0, hi = B;
  while (hi - lo > 1) {
    int32_t mid = (lo + hi) >> 1;
    if (mult * (int64_t)pre[mid] <= x)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- balanced

PA_HD int32_t balanced_ctas(int64_t U, int32_t C) {
  int64_t want = (U + kMinUnitsPerCta - 1) / kMinUnitsPerCta;
  if (want < 1) want = 1;
  return (int32_t)(want < C ? want : C);
}

PA_HD int64_t balanced_begin(int64_t U, int32_t Ce, int32_t c) {
  return (U * (int64_t)c) / Ce;
}

// The CTA whose range holds unit u (0 <= u < U).
PA_HD int32_t balanced_cta_of(int64_t U, int32_t Ce, int64_t u) {
  return (int32_t)(((u + 1) * (int64_t)Ce - 1) / U);
}

struct Piece {
  int32_t b, j, blk0, blk1;  // blocks [blk0, blk1) of segment (b, j)
  int32_t slot;              // partial-state slot, or -1 = whole segment
};

// Row lengths from a host array of stored lengths (plus `add`).
struct HostLens {
  const int32_t* lens;
  int32_t add, bs, maxblk;
  PA_HD int32_t operator()(int32_t b) const { return eff_len(lens[b], add, bs, maxblk); }
};

// Iterates the pieces one CTA processes, in processing order.  LenOf maps a
// row to the length it attends to (the fixed split needs nblk per row).
template <class LenOf>
struct PieceIterT {
  const int32_t* pre;     // [B+1] prefix sums of seq_count
  LenOf len_of;
  SchedShape s;
  int32_t cta;
  // balanced state
  int64_t U, u, u_end, u_begin;
  int32_t Ce;
  // fixed state
  int64_t item, items;

  PA_HD void init(const int32_t* pre_, const LenOf& len_of_, const SchedShape& s_,
                  int32_t cta_) {
    pre = pre_;
    len_of = len_of_;
    s = s_;
    cta = cta_;
    if (s.part_blocks == 0) {
      U = (int64_t)s.Hkv * pre[s.B];
      Ce = balanced_ctas(U, s.num_ctas);
      if (cta < Ce && U > 0) {
        u_begin = balanced_begin(U, Ce, cta);
        u_end = balanced_begin(U, Ce, cta + 1);
      } else {
        u_begin = u_end = 0;
      }
      u = u_begin;
      items = item = 0;
    } else {
      items = (int64_t)s.Hkv * pre[s.B];
      item = cta;
      U = u = u_end = u_begin = 0;
      Ce = s.num_ctas;
    }
  }

  // The row and first block of the piece next() would return, without
  // advancing (false when there is none).  Only reads the iterator.
  PA_HD bool peek_start(int32_t& b, int32_t& blk0) const {
    if (s.part_blocks == 0) {
      if (u >= u_end) return false;
      b = find_seq(pre, s.B, s.Hkv, u);
      const int32_t n = pre[b + 1] - pre[b];
      const int32_t r = (int32_t)(u - (int64_t)s.Hkv * pre[b]);
      const int32_t off = r - (r / n) * n;
      blk0 = off < s.K ? 0 : off - s.K;
      return true;
    }
    if (item >= items) return false;
    b = find_seq(pre, s.B, s.Hkv, item);
    const int64_t r = item - (int64_t)s.Hkv * pre[b];
    blk0 = (int32_t)(r / s.Hkv) * s.part_blocks;
    return true;
  }

  // Next piece; false when the CTA has no more work.
  PA_HD bool next(Piece& p) {
    if (s.part_blocks == 0) {
      if (u >= u_end) return false;
      int32_t b = find_seq(pre, s.B, s.Hkv, u);
      int32_t n = pre[b + 1] - pre[b];  // K + blocks of each segment of row b
      // r < Hkv * n fits in 32 bits (the counts of one row), so the division
      // is a 32-bit one
      const int32_t r = (int32_t)(u - (int64_t)s.Hkv * pre[b]);
      int32_t j = r / n;
      int32_t off = r - j * n;
      if (off < s.K) {  // the segment's overhead units: on to its first block
        u += s.K - off;
        off = s.K;
        if (u >= u_end) return false;
      }
      const int32_t nb = n - s.K;
      const int32_t blk0 = off - s.K;
      int64_t avail = u_end - u;
      int32_t cnt = (int64_t)(nb - blk0) < avail ? (nb - blk0) : (int32_t)avail;
      p.b = b;
      p.j = j;
      p.blk0 = blk0;
      p.blk1 = blk0 + cnt;
      const bool cont = blk0 > 0;          // begun in an earlier CTA
      const bool past = blk0 + cnt < nb;   // continues in a later one
      p.slot = (cont || past) ? 2 * cta + (cont ? 0 : 1) : -1;
      u += cnt;
      return true;
    }
    if (item >= items) return false;
    int32_t b = find_seq(pre, s.B, s.Hkv, item);
    int64_t r = item - (int64_t)s.Hkv * pre[b];
    int32_t part = (int32_t)(r / s.Hkv);
    int32_t j = (int32_t)(r % s.Hkv);
    int32_t nb = seq_blocks(len_of(b), s.bs, s.maxblk);
    int32_t np = pre[b + 1] - pre[b];
    p.b = b;
    p.j = j;
    p.blk0 = part * s.part_blocks;
    p.blk1 = (part + 1) * s.part_blocks < nb ? (part + 1) * s.part_blocks : nb;
    p.slot = (np == 1) ? -1 : (int32_t)item;
    item += s.num_ctas;
    return true;
  }
};

using PieceIter = PieceIterT<HostLens>;

// Balanced split: the segment that begins inside CTA c and continues past
// its range, if any.  Returns false when CTA c has none.  On success gives
// the segment, the last CTA holding one of its pieces, and the slot of the
// piece in CTA c.  Every such segment has exactly one such CTA, so merging
// it there (and only there) merges every split segment once.
PA_HD bool balanced_split_segment(const int32_t* pre, const SchedShape& s, int32_t c,
                                  int32_t& b, int32_t& j, int32_t& c_last, int32_t& slot) {
  int64_t U = (int64_t)s.Hkv * pre[s.B];
  if (U <= 0) return false;
  int32_t Ce = balanced_ctas(U, s.num_ctas);
  if (c >= Ce) return false;
  int64_t u0 = balanced_begin(U, Ce, c);
  int64_t u1 = balanced_begin(U, Ce, c + 1);
  if (u1 <= u0) return false;
  int64_t last = u1 - 1;
  b = find_seq(pre, s.B, s.Hkv, last);
  int32_t n = pre[b + 1] - pre[b];
  int64_t r = last - (int64_t)s.Hkv * pre[b];
  j = (int32_t)(r / n);
  int64_t seg_begin = (int64_t)s.Hkv * pre[b] + (int64_t)j * n;
  int64_t first_blk = seg_begin + s.K;  // unit of the segment's first block
  int64_t seg_end = seg_begin + n;
  if (seg_end <= u1) return false;     // finishes inside c
  if (first_blk < u0 || first_blk >= u1) return false;  // its blocks do not begin in c
  c_last = balanced_cta_of(U, Ce, seg_end - 1);
  slot = 2 * c + 1;
  return true;
}

// The pieces merge index `seg` combines: balanced split -- the segment that
// begins in split CTA seg and continues past it (desc as written by the split
// kernel from balanced_split_segment); fixed split -- segment (b, j) =
// (seg / Hkv, seg % Hkv) when it has more than one partition.
struct MergeSeg {
  int32_t b, j, np;   // np = number of pieces (0: nothing to merge)
  int32_t seg, Hkv;
  int32_t balanced;
  int64_t slot0;      // balanced: slot of piece 0
  int64_t fbase;      // fixed: slot of partition 0

  PA_HD int64_t slot(int32_t p) const {
    if (balanced) return p == 0 ? slot0 : 2 * (int64_t)(seg + p);  // slot0 = 2 seg + 1
    return fbase + (int64_t)p * Hkv;
  }
};

// desc = (b, j, c_last, slot) or b < 0.  pre only read for the fixed split.
PA_HD MergeSeg merge_segment(const SchedShape& s, int32_t seg, int32_t db, int32_t dj,
                             int32_t dlast, int32_t dslot, const int32_t* pre) {
  MergeSeg m;
  m.seg = seg;
  m.Hkv = s.Hkv;
  m.balanced = s.part_blocks == 0;
  m.np = 0;
  m.b = m.j = 0;
  m.slot0 = m.fbase = 0;
  if (m.balanced) {
    if (db < 0) return m;
    m.b = db;
    m.j = dj;
    m.np = dlast - seg + 1;
    m.slot0 = dslot;
  } else {
    m.b = seg / s.Hkv;
    m.j = seg % s.Hkv;
    const int32_t n = pre[m.b + 1] - pre[m.b];
    if (n <= 1) return m;
    m.np = n;
    m.fbase = (int64_t)s.Hkv * pre[m.b] + m.j;
  }
  return m;
}

}  // namespace pa
