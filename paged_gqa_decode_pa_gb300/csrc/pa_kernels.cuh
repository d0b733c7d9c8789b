// pa_kernels.cuh -- internal interface between the host API (pa_api.cu) and
// the kernels: argument blocks, the shared-memory carve-up of the split
// kernel (computed identically on host and device), and launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_sched.cuh"

namespace pa {

constexpr int kMaxWarps = 8;   // warps per split CTA (each runs its own TMA ring)

constexpr int kMaxSlots = 64;  // warps x ring slots
constexpr int kGMax = 8;       // query heads per kv head handled by one CTA
constexpr int kColMax = 16;    // query columns (token, head) of a warp state: two mma n-blocks
constexpr int kRowCols = 32;   // query columns of a row: a warp pair's two states
constexpr int kTile = 16;      // tokens per pipeline stage (one mma row tile)
constexpr int kMergeThreads = 128;
// Slack of the lazy running max in the tensor-core tile (log2 units): p <= 2^8.
constexpr float kLazyMax = 8.f;

// kSimt / kMma: one query token per sequence (decode).  kMmaQ: several query
// tokens per sequence; a row is a group of one sequence's query tokens whose
// (token, head) pairs fill up to mma_blocks(D) x 8 columns.  kMmaP: the same
// with warp pairs -- warps w and w + W/2 consume the same tiles (stream
// w % (W/2)), each for its own half of the row's columns ([0, 8 NB) and
// [8 NB, C)), so a row of up to 16 NB columns reads its K/V once; the lower
// warp loads the tiles, the upper one releases each ring slot through the
// slot's "empty" mbarrier.  kMmaW: rows of up to kRowCols columns held by
// one warp, with the columns as the mma's M dimension (two m-tiles of 16):
// the scores come out in the layout the P.V product takes them in, and each
// tile's K/V fragments feed all the row's columns (head_dim <= 128).
enum Mode { kSimt = 1, kMma = 2, kMmaQ = 3, kTc = 4, kMmaP = 5, kMmaW = 6 };  // kTc: pa_split_tc.cuh

// Warps per split CTA for a head dimension (and kernel mode): 8, or 4 for
// d = 256 so that each warp can keep three 16 KB stages in flight within the
// shared memory; kWideWarps for wide rows, with kWideRing slots each.
constexpr int kWideWarps = 8;
constexpr int kWideRing = 2;
PA_HD constexpr int split_warps(int D, int mode = kMma) {
  return D == 256 ? 4 : (mode == kMmaW ? kWideWarps : kMaxWarps);
}

PA_HD constexpr bool several_tokens(int mode) {
  return mode == kMmaQ || mode == kMmaP || mode == kMmaW;
}

// mma n-blocks of 8 query columns a warp keeps (registers allow two below
// d = 256).
PA_HD constexpr int mma_blocks(int D, int mode) { return (several_tokens(mode) && D <= 128) ? 2 : 1; }

struct SplitArgs {
  const uint16_t* q;        // [B, H, D] raw 16-bit patterns
  const int32_t* table;     // [B, maxblk]
  const int32_t* seqlens;   // [B]
  float* out;               // [B, H, D]
  float* ws_ml;             // [slots][G][2] (max in log2 units, exp-sum)
  float* ws_acc;            // [slots][G][D] unnormalised weighted V
  int32_t* ws_pre;          // [B + 1] prefix sums of the per-sequence count
  int4* ws_desc;            // [grid] balanced split: segment beginning in CTA c
  uint32_t* status;         // sticky PA_STATUS_* bits
  int32_t B, H, Hkv, G, bs, maxblk, P;
  int32_t part_blocks;      // 0 = balanced split
  int32_t piece_k;          // balanced split: overhead units per segment (pa_sched.cuh)
  int32_t warps;            // warps per CTA (= blockDim.x / 32)
  int32_t ring;             // TMA ring slots per warp
  float qscale;             // scale * log2(e): scores are kept in log2 units
  // fused append: each sequence's new K/V row (k_new/v_new [B, Hkv, D]) is
  // written to position cache_seqlens[b] of the pool and attended to
  int32_t len_add;          // 0, or 1 with the fused append
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_pool;         // the pools, writable (fused append only)
  uint16_t* v_pool;
  // columns of one row: G heads in decode; tq tokens x G heads with several
  // query tokens per sequence
  int32_t C;
  // 1: one tensor map covers both pools (its last dimension, extent 2, steps
  // from one pool to the other), so a tile's K and V rows come in one copy;
  // kv_swap: the map starts at the V pool (V lands first in the stage)
  int32_t kv_fused, kv_swap;
  // several query tokens per sequence (kMmaQ): B counts rows = sequences x
  // nqg groups of tq tokens; q and out are packed [total_q, H, D] rows and
  // sequence s owns rows cu_q[s] .. cu_q[s+1]-1
  const int32_t* cu_q;
  int32_t nqg, tq, causal, total_q, max_q;
  // the longest a pipeline wait may take before the step gives up (us; 0 =
  // kWaitLimitNs), and the timeout-path test: 1 = warp 0 of every CTA waits
  // for its first tile on a barrier that nothing completes
  int32_t wait_us, stall_test;
  // the cluster kernel (pa_cluster.cuh), host-buffer calls: once every CTA
  // has counted itself in `done` (a workspace word, zero between calls), the
  // last one copies *status to *status_out and clears both words
  uint32_t* status_out;
  uint32_t* done;
};

// Query rows [q0, q0 + nq) of sequence s, or false when cu_q is not a valid
// span there (then nothing of s is read or written).
__device__ __forceinline__ bool query_span(const int32_t* cu_q, int32_t s, int32_t total_q,
                                           int32_t max_q, int32_t& q0, int32_t& nq) {
  const int32_t a = __ldg(cu_q + s), b = __ldg(cu_q + s + 1);
  const bool ok = a >= 0 && a <= b && b <= total_q && b - a <= max_q;
  q0 = ok ? a : 0;
  nq = ok ? b - a : 0;
  return ok;
}

// Decode rows: the stored length (plus the appended token).
struct DecodeLen {
  const int32_t* seqlens;
  int32_t add, bs, maxblk;
  __device__ __forceinline__ int32_t operator()(int32_t b) const {
    return eff_len(__ldg(seqlens + b), add, bs, maxblk);
  }
};

// Rows of several query tokens: row r = group r % nqg of sequence r / nqg.
// The group's tokens are the sequence's query tokens [g*tq, g*tq + tq); a
// query token i of nq sees keys t < k_len - nq + i + 1 (causal) or all k_len
// keys, so the row reads up to the limit of its last token.  -1: the
// sequence's key length is invalid; 0: nothing to read.
struct MultiLen {
  const int32_t* seqlens;
  const int32_t* cu_q;
  int32_t nqg, tq, causal, total_q, max_q, bs, maxblk;
  __device__ __forceinline__ int32_t operator()(int32_t r) const {
    const int32_t s = r / nqg, g = r - s * nqg;
    const int32_t klen = __ldg(seqlens + s);
    if (!seq_len_valid(klen, bs, maxblk)) return -1;
    int32_t q0, nq;
    if (!query_span(cu_q, s, total_q, max_q, q0, nq)) return 0;
    const int32_t first = g * tq;
    if (first >= nq) return 0;
    if (!causal) return klen;
    const int32_t last = min(nq, first + tq) - 1;
    return max(0, min(klen, klen - nq + last + 1));
  }
};

// Shared-memory room for a copy of SplitArgs, at a fixed offset after the
// mbarriers and stage infos.
constexpr uint32_t kArgsBytes = 256;
constexpr uint32_t kArgsOffset = 1024;
static_assert(sizeof(SplitArgs) <= kArgsBytes && sizeof(SplitArgs) % 4 == 0, "SplitArgs copy");
// Warp pairs: one "empty" mbarrier per ring slot, after the SplitArgs copy.
constexpr uint32_t kEmptyOffset = kArgsOffset + kArgsBytes;
static_assert(kEmptyOffset + 8u * kMaxSlots <= 2048u, "empty barriers below the stages");
// The timeout-path test's barrier (initialised, never arrived on).
constexpr uint32_t kStallOffset = kEmptyOffset + 8u * kMaxSlots;
static_assert(kStallOffset + 8u <= 2048u, "stall barrier below the stages");

struct MergeArgs {
  const int32_t* seqlens;
  float* out;
  const float* ws_ml;
  const float* ws_acc;
  const int32_t* ws_pre;
  const int4* ws_desc;
  int32_t B, H, Hkv, G, D, bs, maxblk;
  int32_t part_blocks;
  int32_t num_ctas;  // grid of the split kernel
  int32_t C;         // columns per row (G in decode)
  const int32_t* cu_q;  // non-null: rows of several query tokens (see SplitArgs)
  int32_t nqg, tq, total_q, max_q;
  // status_out non-null: once the split grid is done, CTA 0 copies the status
  // word the split kernel accumulated (*status) to *status_out and clears it
  uint32_t* status;
  uint32_t* status_out;
};

// Host-to-device staging by the SMs: n parts of `words` 4-byte words each,
// read from page-locked host memory the device maps (src) and written to
// device memory (dst); `status`, if not null, is cleared first.
struct StageArgs {
  const uint32_t* src[4];
  uint32_t* dst[4];
  int64_t words[4];
  int32_t n;
  uint32_t* status;
};

struct AppendArgs {
  const uint16_t* k_new;  // [B, Hkv, D]
  const uint16_t* v_new;
  uint16_t* k_cache;      // [P, bs, Hkv, D]
  uint16_t* v_cache;
  const int32_t* table;
  const int32_t* seqlens;
  uint32_t* status;
  int32_t B, Hkv, D, bs, maxblk, P;
};

// Byte offsets inside the split kernel's dynamic shared memory, relative to
// a 1024-byte aligned base.
struct SmemLayout {
  uint32_t full, info, abort_flag;  // per slot: mbarrier, (phys << 32 | bad | valid rows)
  uint32_t empty;                   // per slot (warp pairs): released by the upper warp
  uint32_t stage;                   // [streams][R] stages: K chunks | V chunks, 16 rows each
  uint32_t stage_bytes;
  uint32_t mo, mm, ml, mbad;        // per-warp partial states for the CTA combine
  uint32_t cwt;                     // [kRowCols][kMaxWarps + 2] fp32 combine weights, max, sum
  uint32_t qs;                      // [C][D+4] fp32 q of the current piece (x scale*log2(e): CUDA cores; kMmaW: 16-bit)
  uint32_t qlim;                    // [kRowCols] int32 key limit per column (several tokens)
  uint32_t qraw;                    // [C][D] raw 16-bit q of the next piece (cp.async target)
  uint32_t args;                    // a copy of the SplitArgs, read by the once-per-piece code
  uint32_t zrow;                    // one all-zero K/V row (D x 2 bytes)
  uint32_t nrow;                    // per warp: the appended token's K and V rows
  uint32_t ps;                      // CUDA-core path: p per warp
  uint32_t pre;                     // [B + 1] prefix sums
  uint32_t total;                   // bytes to request (incl. alignment slack)
};

PA_HD uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Tile streams of a CTA: one per warp, or one per warp pair (kMmaP).
PA_HD constexpr int split_streams(int W, int mode) { return mode == kMmaP ? W / 2 : W; }

// Columns of the row a warp publishes at once (the stride of its published
// state): its half of a pair's row, a wide row's 16-column m-tile, or the
// whole row.
PA_HD constexpr int warp_columns(int D, int C, int mode) {
  return mode == kMmaP ? 8 * mma_blocks(D, mode) : (mode == kMmaW ? kColMax : C);
}

// Row stride (bytes) of a wide row's 16-bit q copy: 16-byte rows for
// ldmatrix, 8 rows landing in distinct bank groups.
PA_HD constexpr uint32_t wide_q_stride(int D) { return (uint32_t)(D + 8) * 2u; }

// C = query columns per row (G in decode), B = rows, R = ring slots per
// tile stream.
PA_HD SmemLayout split_smem_layout(int D, int C, int B, int W, int R, int mode) {
  SmemLayout L;
  L.full = 0;
  L.info = 8 * kMaxSlots;
  L.args = kArgsOffset;  // fixed, so it can be filled before the layout is known
  L.empty = kEmptyOffset;
  L.stage = 2048;
  L.stage_bytes = 4u * (uint32_t)D * (uint32_t)kTile;  // K + V tiles, 2 bytes each
  uint32_t off = L.stage + (uint32_t)(split_streams(W, mode) * R) * L.stage_bytes;
  L.mo = off;
  off += (uint32_t)(W * warp_columns(D, C, mode) * (D + 4)) * 4u;
  L.mm = off;
  off += (uint32_t)W * kColMax * 4u;
  L.ml = off;
  off += (uint32_t)W * kColMax * 4u;
  L.mbad = off;
  off += (uint32_t)W * 4u;
  L.cwt = off;
  off += (uint32_t)kRowCols * (kMaxWarps + 2) * 4u;
  L.abort_flag = off;  // followed by the current piece's stored length, q0, nq
  off += 16u;
  L.qlim = off;
  off += (uint32_t)kRowCols * 4u;
  off = align_up(off, 16);
  L.qs = off;  // kMmaW: the row's q as 16-bit [kRowCols][D + 8] (columns >= C zero)
  off += mode == kMmaW ? (uint32_t)kRowCols * wide_q_stride(D) : (uint32_t)(C * (D + 4)) * 4u;
  L.qraw = off;
  off += (uint32_t)(C * D) * 2u;
  L.zrow = off;
  off += (uint32_t)D * 2u;
  L.nrow = off;  // the fused append only (one query token per sequence)
  off += several_tokens(mode) ? 0u : (uint32_t)(W * 2 * D) * 2u;
  if (mode == kSimt) {
    L.ps = off;
    off += (uint32_t)(W * kTile * kGMax) * 4u;
  } else {
    L.ps = 0;
  }
  L.pre = off;
  off += (uint32_t)(B + 1) * 4u;
  off = align_up(off, 16);
  L.total = off + 1024;  // slack to align the base to 1024 bytes
  return L;
}

// ---- the tcgen05 split kernel (pa_split_tc.cuh): constants and shared-memory
// layout, computed identically on host and device.

constexpr int kTcTile = 128;                        // tokens per tile (MMA M)
constexpr int kTcD = 128;                           // head dimension of this kernel
constexpr int kTcN = 16;                            // MMA N: query columns (C <= 16)
constexpr int kTcThreads = 224;                     // 4 softmax warps, K producer, MMA, V producer
constexpr uint32_t kTcChunk = kTcTile * 128u;       // [128 rows][64 dims] swizzled: 16 KB
constexpr uint32_t kTcHalfBytes = 2u * kTcChunk;    // a tile's K (or V): 2 chunks, 32 KB
constexpr uint32_t kTcOpBytes = kTcN * 128u * 2u;   // q: [16 rows][128] 16-bit, two 2 KB chunks
constexpr uint32_t kTcPBytes = 2u * kTcOpBytes;     // P: [32 rows (high, low)][128], two 4 KB chunks
constexpr uint32_t kTcTmemCols = 64;                // S0 at 0, S1 at 16, O (high, low) at 32, 48
constexpr int kTcKStages = 2;                       // K slots: freed when the scores are done
constexpr int kTcMaxVStages = 4;                    // V slots: freed when O is updated

// Byte offsets in the kernel's dynamic shared memory (base 1024-aligned).
struct TcLayout {
  uint32_t k;       // [kTcKStages] K slots
  uint32_t v;       // [NV] V slots
  uint32_t p;       // [2 buffers] P operands (rows 0-15 high parts, 16-31 low)
  uint32_t q;       // [2] q operands (piece parity)
  uint32_t bars;    // mbarriers (see TcBars)
  uint32_t red;     // [4 warps][16] fp32 reduction scratch
  uint32_t tbase;   // TMEM base address (written by tcgen05.alloc)
  uint32_t abort_flag;
  uint32_t args;    // the SplitArgs copy
  uint32_t pre;     // [rows + 1] prefix sums
  uint32_t total;
};

// mbarrier offsets inside TcLayout::bars (8 bytes each).
struct TcBars {
  static PA_HD uint32_t full_k(int s) { return 8u * (uint32_t)s; }
  static PA_HD uint32_t empty_k(int s) { return 8u * (uint32_t)(kTcKStages + s); }
  static PA_HD uint32_t full_v(int s) { return 8u * (uint32_t)(2 * kTcKStages + s); }
  static PA_HD uint32_t empty_v(int s) { return 8u * (uint32_t)(2 * kTcKStages + kTcMaxVStages + s); }
  static constexpr int kRest = 2 * kTcKStages + 2 * kTcMaxVStages;
  static PA_HD uint32_t s_full(int b) { return 8u * (uint32_t)(kRest + b); }
  static PA_HD uint32_t s_free(int b) { return 8u * (uint32_t)(kRest + 2 + b); }
  static PA_HD uint32_t p_full(int b) { return 8u * (uint32_t)(kRest + 4 + b); }
  static PA_HD uint32_t p_free(int b) { return 8u * (uint32_t)(kRest + 6 + b); }
  static PA_HD uint32_t q_ready() { return 8u * (uint32_t)(kRest + 8); }
  static PA_HD uint32_t o_free() { return 8u * (uint32_t)(kRest + 9); }
  static PA_HD uint32_t drain() { return 8u * (uint32_t)(kRest + 10); }
  static constexpr uint32_t kBytes = 8u * (kRest + 11);
};

// NV: V slots.
PA_HD TcLayout tc_smem_layout(int rows, int NV) {
  TcLayout L;
  uint32_t off = 0;
  L.k = off;
  off += (uint32_t)kTcKStages * kTcHalfBytes;
  L.v = off;
  off += (uint32_t)NV * kTcHalfBytes;
  L.p = off;
  off += 2u * kTcPBytes;
  L.q = off;
  off += 2u * kTcOpBytes;
  L.bars = off;
  off += TcBars::kBytes;
  L.red = align_up(off, 16);
  off = L.red;
  off += 4u * kTcN * 4u;
  L.tbase = off;
  off += 16u;
  L.abort_flag = off;
  off += 16u;
  L.args = off;
  off += kArgsBytes;
  L.pre = off;
  off += (uint32_t)(rows + 1) * 4u;
  L.total = align_up(off, 16) + 1024;  // slack to align the base to 1024 bytes
  return L;
}

// V slots that fit next to everything else (>= 2 needed), at most kTcMaxVStages.
PA_HD int tc_stages(int rows, int max_smem) {
  for (int nv = kTcMaxVStages; nv >= 2; --nv)
    if ((int)tc_smem_layout(rows, nv).total <= max_smem) return nv;
  return 0;
}

// ---- the cluster kernel (pa_cluster.cuh): small steps, one thread-block
// cluster of up to kMaxCluster CTAs per (sequence, kv head) segment.

constexpr int kMaxCluster = 8;
constexpr int kClusterMaxTable = 4096;  // block-table entries staged in shared memory

// Shared memory: the split kernel's carve-up for one row (rings, warp states,
// q), then the segment's block-table row, the CTA's folded state and the
// weights of the cluster's states.
struct ClusterLayout {
  SmemLayout s;
  uint32_t table;   // [maxblk] int32
  uint32_t st_acc;  // [C][D] fp32: the CTA's accumulator, relative to st_ml's max
  uint32_t st_ml;   // [C][2] fp32: max (log2 units), exp-sum
  uint32_t wts;     // [C][kMaxCluster] fp32
  uint32_t total;
};

PA_HD ClusterLayout cluster_layout(int D, int C, int W, int R, int maxblk) {
  ClusterLayout L;
  L.s = split_smem_layout(D, C, 0, W, R, kMma);
  uint32_t off = align_up(L.s.total - 1024, 16);
  L.table = off;
  off = align_up(off + (uint32_t)maxblk * 4u, 16);
  L.st_acc = off;
  off += (uint32_t)(C * D) * 4u;
  L.st_ml = off;
  off += (uint32_t)C * 8u;
  L.wts = off;
  off += (uint32_t)(C * kMaxCluster) * 4u;
  L.total = align_up(off, 16) + 1024;  // slack to align the base to 1024 bytes
  return L;
}

// Launchers (explicitly instantiated in pa_split_*.cu, pa_cluster_*.cu).
template <typename T, int D, int MODE>
cudaError_t launch_split(const CUtensorMap& tmk, const CUtensorMap& tmv, const SplitArgs& a,
                         int grid, int threads, size_t smem, cudaStream_t stream);

template <typename T, int D, int MODE>
const void* split_kernel_ptr();

// The tcgen05 split kernel (pa_split_tc.cuh; head_dim 128; kQ: several
// query tokens per sequence), instantiated in pa_split_tc_*.cu.
template <typename T, bool kQ>
cudaError_t launch_split_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const SplitArgs& a,
                            int grid, size_t smem, cudaStream_t stream);

template <typename T, bool kQ>
const void* split_tc_kernel_ptr(int C);  // the variant for C query columns

// The cluster kernel: grid (cs, segs), clusters of cs CTAs along x.
template <typename T, int D>
cudaError_t launch_cluster(const CUtensorMap& tmk, const CUtensorMap& tmv, const SplitArgs& a, int cs,
                           int segs, size_t smem, cudaStream_t stream);

// Clusters of cs CTAs with `smem` bytes each that can be resident at once.
template <typename T, int D>
int cluster_capacity(int cs, size_t smem, int max_smem);

}  // namespace pa
