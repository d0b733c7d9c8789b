// pa_api.cu -- the C ABI of libpagedgqa.so (see include/pagedgqa.h): argument
// checks, per-device setup, TMA tensor maps, and the phase-2 merge and cache
// append kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "pa_kernels.cuh"
#include "pa_ptx.cuh"
#include "pagedgqa.h"

using namespace pa;

namespace {

// ------------------------------------------------------------------ merge

// Phase 2: combine the partial states of every segment the split kernel cut
// across CTAs (balanced split) or partitions (fixed split).  A block folds
// one column (a query head, or a (token, head) pair) of one merge index
// (pa_sched.cuh, merge_segment): with the balanced split, block i takes
// column i % C of the (i / C)-th segment that has pieces to merge
// (find_segment); with the fixed split, block (seg, g) takes column g of
// segment seg.  The fold uses the combine op ("Paged Attention Kernel
// Architecture for BI-V100", section 2, Level 1 binary op / Level 3): warp w
// of NW folds pieces w, w+NW, ... in order, each lane holding D/32 of the
// dims; the NW warp states are then folded in a fixed order, so the result is
// deterministic.  The loads of up to kMergeBatch pieces are issued before
// any of them is folded, so a segment of many pieces costs few round trips.
constexpr int kMergeBatch = 16;

template <int V>
struct Vec {
  float v[V];
};

template <int V>
__device__ __forceinline__ Vec<V> load_vec(const float* p) {
  Vec<V> r;
  if constexpr (V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 4) {
      const float4 x = *reinterpret_cast<const float4*>(p + i);
      r.v[i] = x.x;
      r.v[i + 1] = x.y;
      r.v[i + 2] = x.z;
      r.v[i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; i += 2) {
      const float2 x = *reinterpret_cast<const float2*>(p + i);
      r.v[i] = x.x;
      r.v[i + 1] = x.y;
    }
  }
  return r;
}

template <int D, int NW>
__device__ __forceinline__ void merge_column(const MergeArgs& a, const MergeSeg& ms, int g,
                                             int64_t out_row) {
  constexpr int V = D / 32;  // dims per lane
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  __shared__ float wm[NW], wl[NW];
  __shared__ __align__(16) float wacc[NW][D];
  float m = -INFINITY, l = 0.f;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  for (int p0 = w; p0 < ms.np; p0 += NW * kMergeBatch) {
    float mp[kMergeBatch], lp[kMergeBatch];
    Vec<V> x[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int p = p0 + u * NW;
      mp[u] = -INFINITY;
      lp[u] = 0.f;
      if (p < ms.np) {
        const int64_t s = ms.slot(p);
        mp[u] = a.ws_ml[(s * a.C + g) * 2];
        lp[u] = a.ws_ml[(s * a.C + g) * 2 + 1];
        x[u] = load_vec<V>(a.ws_acc + (s * a.C + g) * D + lane * V);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) x[u].v[i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      // an empty state (m = -inf) gets weight 0: the identity, except that a
      // NaN it carries (a bad piece) still reaches the result
      const float nm = fmaxf(m, mp[u]);
      const float sa = (m == -INFINITY) ? 0.f : ex2(m - nm);
      const float sb = (mp[u] == -INFINITY) ? 0.f : ex2(mp[u] - nm);
      l = l * sa + lp[u] * sb;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = acc[i] * sa + x[u].v[i] * sb;
      m = nm;
    }
  }
  if (lane == 0) {
    wm[w] = m;
    wl[w] = l;
  }
#pragma unroll
  for (int i = 0; i < V; ++i) wacc[w][lane * V + i] = acc[i];
  __syncthreads();
  // warp 0 folds the NW warp states in order and writes the column
  if (w == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int v = 0; v < NW; ++v) M = fmaxf(M, wm[v]);
    float L = 0.f;
    float o[V];
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = 0.f;
#pragma unroll
    for (int v = 0; v < NW; ++v) {
      const float e = (wm[v] == -INFINITY) ? 0.f : ex2(wm[v] - M);
      L = fmaf(e, wl[v], L);
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] = fmaf(e, wacc[v][lane * V + i], o[i]);
    }
    // a column that saw no key (causal limit 0) gets 0; NaN passes through.
    // Each lane's V dims go out as 16- (or 8-) byte stores, so the warp
    // writes whole lines: out may be page-locked host memory, where strided
    // 4-byte stores become partial-line writes across the chip link.
    float* dst = a.out + out_row * D + lane * V;
    float r[V];
#pragma unroll
    for (int i = 0; i < V; ++i) r[i] = L == 0.f ? 0.f : o[i] / L;
    if constexpr (V % 4 == 0) {
#pragma unroll
      for (int i = 0; i < V; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(r[i], r[i + 1], r[i + 2], r[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < V; i += 2) *reinterpret_cast<float2*>(dst + i) = make_float2(r[i], r[i + 1]);
    }
  }
}

// Balanced split: which segment merge CTA `blockIdx.x` takes.  The segments
// with more than one piece are the split CTAs whose descriptor is set; the
// CTA takes the k-th of them in CTA order, k = blockIdx.x / C, so the CTAs
// that have work are the first ones of the grid and start in its first wave.
// Returns false when fewer than k + 1 segments have pieces to merge.
template <int NW>
__device__ __forceinline__ bool find_segment(const MergeArgs& a, int k, int& seg, int4& desc) {
  constexpr int kThreads = NW * 32;
  constexpr int kPre = 4;  // descriptor chunks loaded before the scan
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  __shared__ int wcount[NW];
  __shared__ int found_seg;
  __shared__ int4 found_desc;
  if (tid == 0) found_seg = -1;
  int4 pre[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int c = i * kThreads + tid;
    pre[i] = c < a.num_ctas ? a.ws_desc[c] : make_int4(-1, 0, 0, 0);
  }
  int base = 0;  // segments found in the chunks before
  for (int i = 0; i * kThreads < a.num_ctas; ++i) {
    const int c = i * kThreads + tid;
    int4 d = make_int4(-1, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kPre; ++u)
      if (u == i) d = pre[u];
    if (i >= kPre && c < a.num_ctas) d = a.ws_desc[c];
    const bool has = d.x >= 0;
    const unsigned bal = __ballot_sync(0xffffffffu, has);
    if (lane == 0) wcount[w] = __popc(bal);
    __syncthreads();
    int before = base, total = 0;
#pragma unroll
    for (int v = 0; v < NW; ++v) {
      before += v < w ? wcount[v] : 0;
      total += wcount[v];
    }
    if (has && before + __popc(bal & ((1u << lane) - 1u)) == k) {
      found_seg = c;
      found_desc = d;
    }
    __syncthreads();  // found_* written; wcount free for the next chunk
    base += total;
    if (base > k) break;  // uniform over the block
  }
  seg = found_seg;
  desc = found_desc;
  return seg >= 0;
}

// Balanced split whose segments have few pieces (typically at most
// kMergeBatch: many more rows than split CTAs): CTA i takes column group
// i mod ng (kColGroup columns, one per warp) of the segment that split CTA
// i / ng begins and cuts, if any.  Each warp folds its column's pieces in
// piece order, a batch of loads at a time, and writes the column; no warp
// waits for another.
constexpr int kColGroup = 4;
constexpr int kColBatch = 4;
template <int D>
__global__ void __launch_bounds__(kColGroup * 32) pa_merge_cols_kernel(const MergeArgs a) {
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (a.status_out && blockIdx.x == 0 && threadIdx.x == 0) {
    volatile uint32_t* st = a.status;
    *a.status_out = *st;
    *st = 0u;
  }
  const int ng = (a.C + kColGroup - 1) / kColGroup;
  const SchedShape sched{a.B, a.Hkv, a.bs, a.maxblk, a.part_blocks, a.num_ctas, 0, 0};
  // the descriptor of split CTA seg: the segment that begins in it and
  // continues past it, if any (the grid fits in one wave, so CTAs without
  // work cost no dispatch round)
  const int seg = blockIdx.x / ng;
  const int4 desc = a.ws_desc[seg];
  if (desc.x < 0) return;
  const MergeSeg ms = merge_segment(sched, seg, desc.x, desc.y, desc.z, desc.w, a.ws_pre);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = (blockIdx.x % ng) * kColGroup + w;
  if (ms.np == 0 || g >= a.C) return;
  int64_t out_row = (int64_t)ms.b * a.H + (int64_t)ms.j * a.G + g;
  if (a.cu_q) {
    const int sq = ms.b / a.nqg, grp = ms.b - sq * a.nqg;
    int32_t q0, nq;
    query_span(a.cu_q, sq, a.total_q, a.max_q, q0, nq);
    const int tok = grp * a.tq + g / a.G;
    if (tok >= nq) return;  // the column holds no query
    out_row = (int64_t)(q0 + tok) * a.H + (int64_t)ms.j * a.G + g % a.G;
  }
  constexpr int V = D / 32;  // dims per lane
  float m = -INFINITY, l = 0.f;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  // batches of kColBatch pieces: segments here have two or three pieces as
  // a rule, and few registers keep the whole grid in one wave; a long
  // segment among short ones can span many more split CTAs
  for (int p0 = 0; p0 < ms.np; p0 += kColBatch) {
    float mp[kColBatch], lp[kColBatch];
    Vec<V> x[kColBatch];
#pragma unroll
    for (int u = 0; u < kColBatch; ++u) {
      mp[u] = -INFINITY;
      lp[u] = 0.f;
      if (p0 + u < ms.np) {
        const int64_t sl = ms.slot(p0 + u);
        mp[u] = a.ws_ml[(sl * a.C + g) * 2];
        lp[u] = a.ws_ml[(sl * a.C + g) * 2 + 1];
        x[u] = load_vec<V>(a.ws_acc + (sl * a.C + g) * D + lane * V);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) x[u].v[i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kColBatch; ++u) {
      // an empty state (m = -inf) gets weight 0; a NaN it carries (a bad
      // piece) still reaches the result
      const float nm = fmaxf(m, mp[u]);
      const float sa = (m == -INFINITY) ? 0.f : ex2(m - nm);
      const float sb = (mp[u] == -INFINITY) ? 0.f : ex2(mp[u] - nm);
      l = l * sa + lp[u] * sb;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = acc[i] * sa + x[u].v[i] * sb;
      m = nm;
    }
  }
  // a column that saw no key gets 0; NaN passes through; whole-line stores
  float* dst = a.out + out_row * D + lane * V;
  float r[V];
#pragma unroll
  for (int i = 0; i < V; ++i) r[i] = l == 0.f ? 0.f : acc[i] / l;
  if constexpr (V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 4)
      *reinterpret_cast<float4*>(dst + i) = make_float4(r[i], r[i + 1], r[i + 2], r[i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < V; i += 2) *reinterpret_cast<float2*>(dst + i) = make_float2(r[i], r[i + 1]);
  }
}

// Staging of a host-buffer call's inputs by the SMs (see StageArgs): each
// thread moves 16-byte chunks, four in flight, then the parts' 4-byte tails.
// Dependents (the split kernel) may be scheduled at once; they wait for this
// grid before reading what it writes.  Launched as a programmatic dependent
// of the kernel before it (the asynchronous host-buffer calls), the grid
// fills its staging slot -- which no kernel still running reads: the calls
// alternate between two slots -- while that kernel finishes, and waits for
// it only at the end, so its own dependents still see everything before it
// complete.  Launched plainly, the wait returns at once.
constexpr int kStageThreads = 256;
__global__ void __launch_bounds__(kStageThreads) pa_stage_in_kernel(const StageArgs s) {
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * blockDim.x;
  if (tid == 0 && s.status) *s.status = 0u;
#pragma unroll
  for (int p = 0; p < 4; ++p) {  // unrolled: the parameter arrays stay in the constant bank
    if (p >= s.n) break;
    const int64_t n16 = s.words[p] / 4;
    const uint4* src = reinterpret_cast<const uint4*>(s.src[p]);
    uint4* dst = reinterpret_cast<uint4*>(s.dst[p]);
    int64_t i = tid;
    for (; i + 3 * nth < n16; i += 4 * nth) {
      const uint4 x0 = src[i], x1 = src[i + nth], x2 = src[i + 2 * nth], x3 = src[i + 3 * nth];
      dst[i] = x0;
      dst[i + nth] = x1;
      dst[i + 2 * nth] = x2;
      dst[i + 3 * nth] = x3;
    }
    for (; i < n16; i += nth) dst[i] = src[i];
    for (int64_t k = 4 * n16 + tid; k < s.words[p]; k += nth) s.dst[p][k] = s.src[p][k];
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// NW warps per CTA: 4, or 8 where a segment may have many pieces (one
// round of loads covers kMergeBatch pieces per warp).
template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) pa_merge_kernel(const MergeArgs a) {
  // The next kernel on the stream (the next step's split kernel) may be
  // scheduled now: it waits for this grid to finish before touching memory.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // With programmatic dependent launch this grid may start while the split
  // kernel is finishing: wait until its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (a.status_out && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    volatile uint32_t* st = a.status;
    *a.status_out = *st;
    *st = 0u;
  }
  const SchedShape sched{a.B, a.Hkv, a.bs, a.maxblk, a.part_blocks, a.num_ctas, 0, 0};
  int seg, g;
  int4 desc = make_int4(-1, 0, 0, 0);
  if (a.part_blocks == 0) {
    g = blockIdx.x % a.C;
    if (!find_segment<NW>(a, blockIdx.x / a.C, seg, desc)) return;
  } else {
    seg = blockIdx.x;  // segment (b, j) = (seg / Hkv, seg % Hkv)
    g = blockIdx.y;
  }
  const MergeSeg ms = merge_segment(sched, seg, desc.x, desc.y, desc.z, desc.w, a.ws_pre);
  if (ms.np == 0) return;
  // the output row of column g: head j*G + g of sequence b (decode), or
  // token grp*tq + g/G, head j*G + g%G of the row's sequence
  int64_t out_row = (int64_t)ms.b * a.H + (int64_t)ms.j * a.G + g;
  if (a.cu_q) {
    const int seq = ms.b / a.nqg, grp = ms.b - seq * a.nqg;
    int32_t q0, nq;
    query_span(a.cu_q, seq, a.total_q, a.max_q, q0, nq);
    const int tok = grp * a.tq + g / a.G;
    if (tok >= nq) return;  // the column holds no query (uniform over the block)
    out_row = (int64_t)(q0 + tok) * a.H + (int64_t)ms.j * a.G + g % a.G;
  }
  merge_column<D, NW>(a, ms, g, out_row);
}

// --------------------------------------------------------------- append

// Copy k_new / v_new rows of sequence b = blockIdx.x into the slot of
// position cache_seqlens[b] ("Paged attention", decoding path example).
__global__ void pa_append_kernel(const AppendArgs a) {
  const int b = blockIdx.x;
  const int32_t pos = __ldg(a.seqlens + b);
  bool ok = pos >= 0 && (int64_t)pos < (int64_t)a.maxblk * a.bs;
  int32_t phys = -1;
  if (ok) phys = __ldg(a.table + (int64_t)b * a.maxblk + pos / a.bs);
  ok = ok && phys >= 0 && phys < a.P;
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(a.status, PA_STATUS_NO_SLOT);
    return;
  }
  const int row = pos % a.bs;
  const int units = a.D / 8;  // 16-byte units per row
  for (int u = threadIdx.x; u < a.Hkv * units; u += blockDim.x) {
    const int j = u / units, e = u % units;
    const int64_t dst = (((int64_t)phys * a.bs + row) * a.Hkv + j) * a.D + (int64_t)e * 8;
    const int64_t src = ((int64_t)b * a.Hkv + j) * a.D + (int64_t)e * 8;
    *reinterpret_cast<uint4*>(a.k_cache + dst) = __ldg(reinterpret_cast<const uint4*>(a.k_new + src));
    *reinterpret_cast<uint4*>(a.v_cache + dst) = __ldg(reinterpret_cast<const uint4*>(a.v_new + src));
  }
}

// ----------------------------------------------------------- host helpers

constexpr int kMaxDevices = 64;
constexpr size_t kHeaderBytes = 256;
// Workspace header: the status word at 0; the cluster kernel's CTA count.
constexpr size_t kDoneOffset = 16;
constexpr int kMaxDynamicSmem = 227 * 1024 - 64;  // minus the kernel's static shared memory

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

struct FuncCache {
  const void* fn;
  int dev;
  size_t smem;
  int occ;
};
constexpr int kFuncCacheSize = 256;
FuncCache g_funcs[kFuncCacheSize];
int g_nfuncs = 0;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const pa_shape* s) {
  if (!s) return PA_ERR_NULL;
  if (s->batch < 0 || s->batch > PA_MAX_BATCH) return PA_ERR_SHAPE;
  if (s->num_heads < 1 || s->num_kv_heads < 1) return PA_ERR_SHAPE;
  if (s->num_heads % s->num_kv_heads != 0) return PA_ERR_SHAPE;
  const int G = s->num_heads / s->num_kv_heads;
  if (G > kGMax) return PA_ERR_SHAPE;
  if (s->head_dim != 64 && s->head_dim != 128 && s->head_dim != 256) return PA_ERR_SHAPE;
  if (s->block_size != 16 && s->block_size != 32 && s->block_size != 64) return PA_ERR_SHAPE;
  if (s->max_blocks_per_seq < 1 || s->num_blocks < 1) return PA_ERR_SHAPE;
  if ((int64_t)s->max_blocks_per_seq * s->block_size > INT32_MAX) return PA_ERR_SHAPE;
  if ((int64_t)s->batch * s->max_blocks_per_seq > INT32_MAX) return PA_ERR_SHAPE;
  // the balanced schedule counts a row's (kv head, block) units in 32 bits
  if ((int64_t)s->num_kv_heads * (s->max_blocks_per_seq + 64) > INT32_MAX) return PA_ERR_SHAPE;
  if (s->dtype != PA_F16 && s->dtype != PA_BF16) return PA_ERR_SHAPE;
  return PA_OK;
}

int check_options(const pa_shape* s, const pa_options* o) {
  if (!o) return PA_OK;
  if (o->partition_tokens < 0) return PA_ERR_OPTION;
  if (o->partition_tokens > 0 && o->partition_tokens % s->block_size != 0) return PA_ERR_OPTION;
  if (o->compute < PA_COMPUTE_AUTO || o->compute > PA_COMPUTE_TC) return PA_ERR_OPTION;
  if (o->num_ctas < 0 || o->num_ctas > (1 << 20)) return PA_ERR_OPTION;
  if (o->stages < 0 || o->stages > kMaxSlots / kMaxWarps) return PA_ERR_OPTION;
  if (o->phase < PA_PHASE_BOTH || o->phase > PA_PHASE_MERGE) return PA_ERR_OPTION;
  if (o->wait_limit_us < 0) return PA_ERR_OPTION;
  if (o->stall_test < 0 || o->stall_test > 1) return PA_ERR_OPTION;
  if (o->stall_test && o->compute == PA_COMPUTE_TC) return PA_ERR_OPTION;
  return PA_OK;
}

struct Plan {
  int D, G, bs, mode, warps, ring;  // kTc: ring = the CTA's 128-token stages
  int multi;          // several query tokens per sequence
  int C;              // query columns per row (G in decode)
  int rows;           // rows of the schedule (B in decode, B * nqg with several tokens)
  int nqg, tq;        // several query tokens: groups per sequence, tokens per group
  int part_blocks;
  int grid;  // split kernel CTAs
  size_t smem;
  int64_t slots;
  size_t off_pre, off_desc, off_ml, off_acc, total;
  // > 0: the step runs as one cluster kernel (pa_cluster.cuh) with clusters
  // of `cluster` CTAs, rings of `cring` slots per warp and `csmem` bytes of
  // shared memory; the merge phase is then empty
  int cluster, cring;
  size_t csmem;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

int choose_mode(const pa_options* o) {
  const int c = o ? o->compute : PA_COMPUTE_AUTO;
  return c == PA_COMPUTE_SIMT ? kSimt : (c == PA_COMPUTE_TC ? kTc : kMma);
}

// Ring slots per tile stream: 2 by default (measured best for every head
// dimension: one tile computing, one in flight), 4 for a warp pair's stream
// (the same stages per CTA), fewer when shared memory does not hold them; at
// most what fits in the per-block limit.
int choose_ring(const pa_shape* s, const pa_options* o, int mode, int W, int C, int rows) {
  const int streams = split_streams(W, mode);
  const SmemLayout L0 = split_smem_layout(s->head_dim, C, rows, W, 0, mode);
  int fit = (kMaxDynamicSmem - (int)L0.total) / (streams * (int)L0.stage_bytes);
  if (fit > kMaxSlots / streams) fit = kMaxSlots / streams;
  if (o && o->stages > 0) return o->stages <= fit ? o->stages : -1;
  const int want = mode == kMmaP ? 4 : (mode == kMmaW ? kWideRing : 2);
  return fit < want ? fit : want;
}

// The wide-row kernel exists for head_dim <= 128 only.
template <typename T, int DD>
const void* wide_kernel_ptr() {
  if constexpr (DD <= 128) return split_kernel_ptr<T, DD, kMmaW>();
  return nullptr;
}

template <typename T, int DD>
cudaError_t launch_wide(const CUtensorMap& tmk, const CUtensorMap& tmv, const SplitArgs& a, int grid,
                        int threads, size_t smem, cudaStream_t stream) {
  if constexpr (DD <= 128) return launch_split<T, DD, kMmaW>(tmk, tmv, a, grid, threads, smem, stream);
  return cudaErrorInvalidValue;
}

const void* kernel_for(int dtype, int D, int mode, int multi, int C) {
  if (mode == kTc) {
    if (D != kTcD) return nullptr;
    if (dtype == PA_BF16)
      return multi ? split_tc_kernel_ptr<__nv_bfloat16, true>(C)
                   : split_tc_kernel_ptr<__nv_bfloat16, false>(C);
    return multi ? split_tc_kernel_ptr<__half, true>(C) : split_tc_kernel_ptr<__half, false>(C);
  }
#define PA_PICK(T, DD)                                                                 \
  if (D == DD) return mode == kSimt ? split_kernel_ptr<T, DD, kSimt>()                \
                      : mode == kMmaQ ? split_kernel_ptr<T, DD, kMmaQ>()              \
                      : mode == kMmaP ? split_kernel_ptr<T, DD, kMmaP>()              \
                      : mode == kMmaW ? wide_kernel_ptr<T, DD>()                      \
                                      : split_kernel_ptr<T, DD, kMma>();
  if (dtype == PA_BF16) {
    PA_PICK(__nv_bfloat16, 64)
    PA_PICK(__nv_bfloat16, 128)
    PA_PICK(__nv_bfloat16, 256)
  } else {
    PA_PICK(__half, 64)
    PA_PICK(__half, 128)
    PA_PICK(__half, 256)
  }
#undef PA_PICK
  return nullptr;
}

// Occupancy of the split kernel for this smem size on device `dev`; also
// raises the kernel's dynamic shared-memory limit (once).
int occupancy(const void* fn, int dev, size_t smem, int threads, int* occ_out) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_nfuncs; ++i) {
    if (g_funcs[i].fn == fn && g_funcs[i].dev == dev && g_funcs[i].smem == smem) {
      *occ_out = g_funcs[i].occ;
      return PA_OK;
    }
  }
  bool attr_set = false;
  for (int i = 0; i < g_nfuncs; ++i)
    if (g_funcs[i].fn == fn && g_funcs[i].dev == dev) attr_set = true;
  if (!attr_set && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kMaxDynamicSmem) != cudaSuccess)
    return PA_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem) != cudaSuccess)
    return PA_ERR_CUDA;
  if (occ < 1) return PA_ERR_SHAPE;
  if (g_nfuncs < kFuncCacheSize) g_funcs[g_nfuncs++] = FuncCache{fn, dev, smem, occ};
  *occ_out = occ;
  return PA_OK;
}

int device_sms(int* dev_out, int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[dev].ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    g_dev[dev].sms = sms;
    g_dev[dev].ready = true;
  }
  *dev_out = dev;
  *sms_out = g_dev[dev].sms;
  return PA_OK;
}

// Clusters of the cluster kernel that can be resident at once, cached per
// (device, dtype, head dimension, cluster size, shared memory).
struct ClusterCap {
  int dev, dtype, D, cs;
  size_t smem;
  int n;
};
constexpr int kClusterCapCache = 64;
ClusterCap g_ccap[kClusterCapCache];
int g_nccap = 0;

int cluster_cap(int dev, int dtype, int D, int cs, size_t smem) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_nccap; ++i) {
      const ClusterCap& e = g_ccap[i];
      if (e.dev == dev && e.dtype == dtype && e.D == D && e.cs == cs && e.smem == smem) return e.n;
    }
  }
  int n = 0;
#define PA_CAP(T, DD) \
  if (D == DD) n = cluster_capacity<T, DD>(cs, smem, kMaxDynamicSmem);
  if (dtype == PA_BF16) {
    PA_CAP(__nv_bfloat16, 64)
    PA_CAP(__nv_bfloat16, 128)
    PA_CAP(__nv_bfloat16, 256)
  } else {
    PA_CAP(__half, 64)
    PA_CAP(__half, 128)
    PA_CAP(__half, 256)
  }
#undef PA_CAP
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_nccap < kClusterCapCache) g_ccap[g_nccap++] = ClusterCap{dev, dtype, D, cs, smem, n};
  return n;
}

// The cluster kernel's plan for a decode step, or cluster = 0 when the
// persistent split kernel (with the merge kernel) is the better choice.
// Chosen from the shape and options only, so a captured graph stays valid:
// one query token per sequence on the mma.sync path with the balanced split
// and the library's grid; a small step (at most 64 MB of K/V even with
// every table row full: above that the persistent grid's even split of the
// bytes wins); a table row that fits in shared memory.  The ring is as deep
// as shared memory allows (up to 8 slots per warp).  The cluster is the
// smallest (1 to 8 CTAs) whose CTAs each hold their share of the longest
// possible segment in one ring load -- every tile then is in flight at once
// and the fold across the cluster stays short -- else the largest that fits;
// all B * Hkv clusters must be resident at once.
void plan_cluster(const pa_shape* s, const pa_options* o, int dev, int sms, Plan* p) {
  p->cluster = 0;
  p->cring = 0;
  p->csmem = 0;
  if (p->multi || p->mode != kMma || p->part_blocks != 0) return;
  if (o && (o->num_ctas > 0 || o->stall_test)) return;
  const int64_t segs = (int64_t)s->batch * s->num_kv_heads;
  const int64_t worst = (int64_t)s->batch * s->max_blocks_per_seq * s->block_size *
                        s->num_kv_heads * s->head_dim * 4;
  if (segs < 1 || segs > sms || worst > (64ll << 20) || s->max_blocks_per_seq > kClusterMaxTable)
    return;
  const int W = split_warps(p->D);
  int ring = 0;
  size_t smem = 0;
  for (int r = (o && o->stages > 0) ? o->stages : kMaxSlots / W; r >= 1; --r) {
    if (W * r > kMaxSlots) continue;
    const size_t t = cluster_layout(p->D, p->C, W, r, s->max_blocks_per_seq).total;
    if (t <= (size_t)kMaxDynamicSmem) {
      ring = r;
      smem = t;
      break;
    }
    if (o && o->stages > 0) return;  // the asked-for depth does not fit
  }
  if (ring == 0) return;
  const int64_t tiles = (int64_t)s->max_blocks_per_seq * (s->block_size / kTile);
  const int64_t want64 = (tiles + (int64_t)W * ring - 1) / ((int64_t)W * ring);
  const int want = (int)std::min<int64_t>(std::max<int64_t>(want64, 1), kMaxCluster);
  auto fits = [&](int cs) {
    return segs * cs <= sms && cluster_cap(dev, s->dtype, p->D, cs, smem) >= segs;
  };
  int cs = 0;
  for (int c = want; c <= kMaxCluster && !cs; ++c)
    if (fits(c)) cs = c;
  for (int c = want - 1; c >= 1 && !cs; --c)
    if (fits(c)) cs = c;
  if (!cs) return;
  p->cluster = cs;
  p->cring = ring;
  p->csmem = smem;
}

// Sizes and offsets of everything one call needs.  `need_device` = false
// only when options->num_ctas fixes the grid (pure host computation).
// max_q > 0: several query tokens per sequence, at most max_q each.
int make_plan(const pa_shape* s, const pa_options* o, bool setup_kernel, Plan* p, int max_q = 0) {
  int rc = check_shape(s);
  if (rc) return rc;
  rc = check_options(s, o);
  if (rc) return rc;
  p->D = s->head_dim;
  p->G = s->num_heads / s->num_kv_heads;
  p->bs = s->block_size;
  p->mode = choose_mode(o);
  if (p->mode == kTc && p->D != kTcD) return PA_ERR_OPTION;
  p->warps = p->mode == kTc ? kTcThreads / 32 : split_warps(p->D);
  p->C = p->G;
  p->rows = s->batch;
  p->nqg = 1;
  p->tq = 1;
  p->multi = max_q > 0;
  if (max_q > 0) {
    if (max_q > PA_MAX_QUERY_TOKENS) return PA_ERR_SHAPE;
    if (p->mode == kSimt) return PA_ERR_OPTION;  // tensor-core path only
    // groups of (token, head) columns: a warp keeps cw = 8 x mma_blocks of
    // them; rows wider than that (2 cw columns, one read of the K/V) go to
    // wide rows (one warp, columns as the mma's M; head_dim <= 128) or warp
    // pairs.  The tcgen05 kernel keeps groups of N = 16.
    const int cw = 8 * mma_blocks(p->D, kMmaQ);
    if (p->mode != kTc)
      p->mode = (int64_t)max_q * p->G > cw ? (p->D <= 128 ? kMmaW : kMmaP) : kMmaQ;
    p->tq = (p->mode == kTc ? kTcN : (p->mode == kMmaP || p->mode == kMmaW ? 2 * cw : cw)) / p->G;
    p->nqg = (max_q + p->tq - 1) / p->tq;
    p->C = p->tq * p->G;
    if ((int64_t)s->batch * p->nqg > PA_MAX_BATCH) return PA_ERR_SHAPE;
    p->rows = s->batch * p->nqg;
  }
  if (p->mode == kTc) {
    const int fit = tc_stages(p->rows, kMaxDynamicSmem);
    if (fit < 2) return PA_ERR_SHAPE;
    if (o && o->stages > 0) {
      if (o->stages < 2 || o->stages > fit) return PA_ERR_OPTION;
      p->ring = o->stages;
    } else {
      p->ring = fit;  // V slots: as many as fit (4 at 256 rows)
    }
    p->smem = tc_smem_layout(p->rows, p->ring).total;
  } else {
    p->warps = split_warps(p->D, p->mode);
    p->ring = choose_ring(s, o, p->mode, p->warps, p->C, p->rows);
    if (p->mode == kMmaW && p->ring < 2 && !(o && o->stages > 0)) {
      // too many rows for two slots per warp next to the wide states: the
      // same rows on warp pairs
      p->mode = kMmaP;
      p->warps = split_warps(p->D, p->mode);
      p->ring = choose_ring(s, o, p->mode, p->warps, p->C, p->rows);
    }
    if (p->ring < 1) return (o && o->stages > 0) ? PA_ERR_OPTION : PA_ERR_SHAPE;
    const SmemLayout L = split_smem_layout(p->D, p->C, p->rows, p->warps, p->ring, p->mode);
    p->smem = L.total;
  }
  p->part_blocks = (o && o->partition_tokens > 0) ? o->partition_tokens / s->block_size : 0;
  if (p->smem > (size_t)kMaxDynamicSmem) return PA_ERR_SHAPE;
  const bool fixed_grid = o && o->num_ctas > 0;
  if (fixed_grid) p->grid = o->num_ctas;
  if (setup_kernel || !fixed_grid) {
    int dev, sms, occ;
    rc = device_sms(&dev, &sms);
    if (rc) return rc;
    const void* fn = kernel_for(s->dtype, p->D, p->mode, p->multi, p->C);
    if (!fn) return PA_ERR_SHAPE;
    rc = occupancy(fn, dev, p->smem, 32 * p->warps, &occ);
    if (rc) return rc;
    if (!fixed_grid) p->grid = sms * occ;
    plan_cluster(s, o, dev, sms, p);
  } else {
    p->cluster = 0;
    p->cring = 0;
    p->csmem = 0;
  }
  if (p->part_blocks == 0) {
    p->slots = 2 * (int64_t)p->grid;
  } else {
    const int64_t nparts = (s->max_blocks_per_seq + p->part_blocks - 1) / p->part_blocks;
    p->slots = (int64_t)p->rows * s->num_kv_heads * nparts;
  }
  size_t off = kHeaderBytes;
  p->off_pre = off;
  off = round256(off + sizeof(int32_t) * (size_t)(p->rows + 1));
  p->off_desc = off;
  off = round256(off + sizeof(int4) * (size_t)p->grid);
  p->off_ml = off;
  off = round256(off + sizeof(float) * 2 * (size_t)p->slots * p->C);
  p->off_acc = off;
  off = round256(off + sizeof(float) * (size_t)p->slots * p->C * p->D);
  p->total = off;
  return PA_OK;
}

int get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return PA_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return PA_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PA_OK;
}

// 5-D map over a [P, bs, Hkv, D] pool: dims (64, bs, D/64, Hkv, P) with
// element, row, 64-dim chunk, kv head and block strides; box (64, 16, D/64,
// 1, 1), 128-byte swizzle.  One box = 16 rows of one kv head of one physical
// block, landing in shared memory as D/64 chunk tiles of [16][64].
// One pool as (64 dims, bs rows, D/64 chunks, Hkv, P).  The box is a 16-row
// tile of all chunks of one kv head, or (tc) all bs rows of one 64-dim chunk
// of one block, for the tcgen05 kernel's 128-row stage chunks.
int make_pool_map(CUtensorMap* map, const void* pool, const pa_shape* s, bool tc) {
  const uint64_t D = (uint64_t)s->head_dim, Hkv = (uint64_t)s->num_kv_heads;
  const uint64_t bs = (uint64_t)s->block_size, P = (uint64_t)s->num_blocks;
  cuuint64_t dims[5] = {64, bs, D / 64, Hkv, P};
  cuuint64_t strides[4] = {Hkv * D * 2, 128, D * 2, bs * Hkv * D * 2};
  cuuint32_t box[5] = {64, tc ? (cuuint32_t)bs : (cuuint32_t)kTile, tc ? 1u : (cuuint32_t)(D / 64), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUtensorMapDataType dt =
      s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(map, dt, 5, const_cast<void*>(pool), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// One 5-D map over both pools, for one copy per tile: dims (64, bs, D/64,
// P*bs*Hkv, 2) with strides (row Hkv*D*2, chunk 128, "slot" D*2, pool
// distance).  Coordinate (0, row, 0, phys*bs*Hkv + j, 0) with box (64, 16,
// D/64, 1, 2) lands 16 rows of kv head j of block phys from the lower pool,
// then the same rows from the other one -- the K chunks then the V chunks
// of a stage, or V then K when the V pool has the lower address (*swap).
// The slot and row dimensions alias (slot index phys*bs*Hkv + j plus row *
// Hkv is the row's index in the pool), which only addresses rows of the
// pools.  PA_ERR_SHAPE when the pools cannot be described this way (the
// same buffer, a distance of 2^40 bytes or more, a slot index past int32).
int make_kv_map(CUtensorMap* map, const void* k_pool, const void* v_pool, const pa_shape* s,
                int* swap) {
  const uint64_t D = (uint64_t)s->head_dim, Hkv = (uint64_t)s->num_kv_heads;
  const uint64_t bs = (uint64_t)s->block_size, P = (uint64_t)s->num_blocks;
  const uintptr_t k = reinterpret_cast<uintptr_t>(k_pool), v = reinterpret_cast<uintptr_t>(v_pool);
  if (k == v) return PA_ERR_SHAPE;
  const uint64_t dist = k < v ? v - k : k - v;
  if (dist % 16 != 0 || dist >= (1ull << 40)) return PA_ERR_SHAPE;
  if (P * bs * Hkv >= (1ull << 31)) return PA_ERR_SHAPE;
  *swap = v < k ? 1 : 0;
  cuuint64_t dims[5] = {64, bs, D / 64, P * bs * Hkv, 2};
  cuuint64_t strides[4] = {Hkv * D * 2, 128, D * 2, dist};
  cuuint32_t box[5] = {64, (cuuint32_t)kTile, (cuuint32_t)(D / 64), 1, 2};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUtensorMapDataType dt =
      s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(map, dt, 5, reinterpret_cast<void*>(k < v ? k : v), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_SHAPE;
}

struct Call {
  Plan plan;
  SplitArgs sa;
  MergeArgs ma;
};

int prepare(const pa_shape* s, const pa_options* o, const void* q, const void* k_cache,
            const void* v_cache, const int32_t* block_table, const int32_t* cache_seqlens,
            float scale, float* out, void* workspace, size_t workspace_bytes, bool need_kv,
            Call* c, int max_q = 0) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (!block_table || !cache_seqlens || !out || !workspace) return PA_ERR_NULL;
  if (need_kv && (!q || !k_cache || !v_cache)) return PA_ERR_NULL;
  if (!aligned16(block_table) || !aligned16(cache_seqlens) || !aligned16(out) ||
      !aligned16(workspace))
    return PA_ERR_ALIGN;
  if (need_kv && (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)))
    return PA_ERR_ALIGN;
  if (!(scale == scale)) return PA_ERR_SHAPE;  // NaN scale
  rc = make_plan(s, o, false, &c->plan, max_q);
  if (rc) return rc;
  if (workspace_bytes < c->plan.total) return PA_ERR_WORKSPACE;
  if (need_kv) {
    // kernel attributes (dynamic shared memory limit) before the first launch
    rc = make_plan(s, o, true, &c->plan, max_q);
    if (rc) return rc;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const Plan& p = c->plan;
  SplitArgs& a = c->sa;
  a.q = static_cast<const uint16_t*>(q);
  a.table = block_table;
  a.seqlens = cache_seqlens;
  a.out = out;
  a.ws_ml = reinterpret_cast<float*>(ws + p.off_ml);
  a.ws_acc = reinterpret_cast<float*>(ws + p.off_acc);
  a.ws_pre = reinterpret_cast<int32_t*>(ws + p.off_pre);
  a.ws_desc = reinterpret_cast<int4*>(ws + p.off_desc);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.B = p.rows;
  a.H = s->num_heads;
  a.Hkv = s->num_kv_heads;
  a.G = p.G;
  a.bs = s->block_size;
  a.maxblk = s->max_blocks_per_seq;
  a.P = s->num_blocks;
  a.part_blocks = p.part_blocks;
  a.piece_k = p.part_blocks == 0
                  ? piece_units(s->block_size, s->head_dim,
                                !p.multi ? kPieceKb
                                         : (p.mode == kMmaW   ? kPieceKbWide
                                            : p.mode == kMmaP ? kPieceKbPair
                                                              : kPieceKbMulti))
                  : 0;
  a.warps = p.warps;
  a.ring = p.ring;
  a.qscale = scale * 1.4426950408889634f;  // log2(e)
  a.len_add = 0;
  a.k_new = a.v_new = nullptr;
  a.k_pool = a.v_pool = nullptr;
  a.C = p.C;
  a.cu_q = nullptr;
  a.nqg = p.nqg;
  a.tq = p.tq;
  a.causal = 0;
  a.total_q = 0;
  a.max_q = max_q;
  a.wait_us = o ? o->wait_limit_us : 0;
  a.stall_test = o ? o->stall_test : 0;
  a.status_out = nullptr;
  a.done = reinterpret_cast<uint32_t*>(ws + kDoneOffset);
  MergeArgs& m = c->ma;
  m.seqlens = cache_seqlens;
  m.out = out;
  m.ws_ml = a.ws_ml;
  m.ws_acc = a.ws_acc;
  m.ws_pre = a.ws_pre;
  m.ws_desc = a.ws_desc;
  m.B = a.B;
  m.H = a.H;
  m.Hkv = a.Hkv;
  m.G = a.G;
  m.D = p.D;
  m.bs = a.bs;
  m.maxblk = a.maxblk;
  m.part_blocks = a.part_blocks;
  m.num_ctas = p.grid;
  m.C = p.C;
  m.cu_q = nullptr;
  m.nqg = p.nqg;
  m.tq = p.tq;
  m.total_q = 0;
  m.max_q = max_q;
  m.status = a.status;
  m.status_out = nullptr;
  return PA_OK;
}

// Encoded pool maps are cached by (pool address, shape): encoding is host
// work of a few microseconds per map, and a decode loop reuses its pools.
struct MapEntry {
  const void* pool;
  const void* pool2;  // the other pool of a map over both (nullptr: one pool)
  int32_t D, Hkv, bs, P, dtype;
  int32_t tc;         // the tcgen05 kernel's box (make_pool_map)
  int32_t rc, swap;   // encode result (a map over both pools may be impossible)
  alignas(64) CUtensorMap map;
};
constexpr int kMapCache = 32;
MapEntry g_maps[kMapCache];
int g_nmaps = 0, g_next_map = 0;

// pool2 == nullptr: the map of one pool; otherwise the map over both pools
// (make_kv_map), whose result code is cached too.
int pool_map(CUtensorMap* out, const void* pool, const void* pool2, const pa_shape* s,
             int* swap, bool tc = false) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_nmaps; ++i) {
    const MapEntry& e = g_maps[i];
    if (e.pool == pool && e.pool2 == pool2 && e.D == s->head_dim && e.Hkv == s->num_kv_heads &&
        e.bs == s->block_size && e.P == s->num_blocks && e.dtype == s->dtype && e.tc == (int)tc) {
      if (e.rc == PA_OK) {
        *out = e.map;
        if (swap) *swap = e.swap;
      }
      return e.rc;
    }
  }
  MapEntry e;
  e.pool = pool;
  e.pool2 = pool2;
  e.D = s->head_dim;
  e.Hkv = s->num_kv_heads;
  e.bs = s->block_size;
  e.P = s->num_blocks;
  e.dtype = s->dtype;
  e.tc = tc;
  e.swap = 0;
  e.rc = pool2 ? make_kv_map(&e.map, pool, pool2, s, &e.swap) : make_pool_map(&e.map, pool, s, tc);
  if (e.rc != PA_OK && e.rc != PA_ERR_SHAPE) return e.rc;  // encoder failure: not cached
  const int slot = g_nmaps < kMapCache ? g_nmaps++ : (g_next_map++ % kMapCache);
  g_maps[slot] = e;
  if (e.rc == PA_OK) {
    *out = e.map;
    if (swap) *swap = e.swap;
  }
  return e.rc;
}

int launch_split_phase(const pa_shape* s, const void* k_cache, const void* v_cache, Call* c,
                       cudaStream_t stream) {
  int rc = get_encoder();
  if (rc) return rc;
  alignas(64) CUtensorMap tmk;
  alignas(64) CUtensorMap tmv;
  const Plan& p = c->plan;
  if (p.mode == kTc) {
    rc = pool_map(&tmk, k_cache, nullptr, s, nullptr, true);
    if (rc) return rc;
    rc = pool_map(&tmv, v_cache, nullptr, s, nullptr, true);
    if (rc) return rc;
    c->sa.kv_fused = 0;
    c->sa.kv_swap = 0;
    cudaError_t e;
    if (s->dtype == PA_BF16)
      e = p.multi ? launch_split_tc<__nv_bfloat16, true>(tmk, tmv, c->sa, p.grid, p.smem, stream)
                  : launch_split_tc<__nv_bfloat16, false>(tmk, tmv, c->sa, p.grid, p.smem, stream);
    else
      e = p.multi ? launch_split_tc<__half, true>(tmk, tmv, c->sa, p.grid, p.smem, stream)
                  : launch_split_tc<__half, false>(tmk, tmv, c->sa, p.grid, p.smem, stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  int swap = 0;
  if (p.cluster > 0) {
    // the whole step in one kernel (pa_cluster.cuh)
    if (pool_map(&tmk, k_cache, v_cache, s, &swap) == PA_OK) {
      c->sa.kv_fused = 1;
      c->sa.kv_swap = swap;
      tmv = tmk;
    } else {
      c->sa.kv_fused = 0;
      c->sa.kv_swap = 0;
      rc = pool_map(&tmk, k_cache, nullptr, s, nullptr);
      if (rc) return rc;
      rc = pool_map(&tmv, v_cache, nullptr, s, nullptr);
      if (rc) return rc;
    }
    SplitArgs a = c->sa;
    a.ring = p.cring;
    const int segs = s->batch * s->num_kv_heads;
    cudaError_t e = cudaErrorInvalidValue;
#define PA_LAUNCH_CL(T, DD) \
  if (p.D == DD) e = launch_cluster<T, DD>(tmk, tmv, a, p.cluster, segs, p.csmem, stream);
    if (s->dtype == PA_BF16) {
      PA_LAUNCH_CL(__nv_bfloat16, 64)
      PA_LAUNCH_CL(__nv_bfloat16, 128)
      PA_LAUNCH_CL(__nv_bfloat16, 256)
    } else {
      PA_LAUNCH_CL(__half, 64)
      PA_LAUNCH_CL(__half, 128)
      PA_LAUNCH_CL(__half, 256)
    }
#undef PA_LAUNCH_CL
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  if (pool_map(&tmk, k_cache, v_cache, s, &swap) == PA_OK) {
    // one copy per tile for K and V
    c->sa.kv_fused = 1;
    c->sa.kv_swap = swap;
    tmv = tmk;
  } else {
    c->sa.kv_fused = 0;
    c->sa.kv_swap = 0;
    rc = pool_map(&tmk, k_cache, nullptr, s, nullptr);
    if (rc) return rc;
    rc = pool_map(&tmv, v_cache, nullptr, s, nullptr);
    if (rc) return rc;
  }
  cudaError_t e = cudaErrorInvalidValue;
#define PA_LAUNCH(T, DD)                                                                        \
  if (p.D == DD)                                                                                \
    e = p.mode == kSimt                                                                         \
            ? launch_split<T, DD, kSimt>(tmk, tmv, c->sa, p.grid, 32 * p.warps, p.smem, stream)     \
        : p.mode == kMmaQ                                                                       \
            ? launch_split<T, DD, kMmaQ>(tmk, tmv, c->sa, p.grid, 32 * p.warps, p.smem, stream)     \
        : p.mode == kMmaP                                                                       \
            ? launch_split<T, DD, kMmaP>(tmk, tmv, c->sa, p.grid, 32 * p.warps, p.smem, stream)     \
        : p.mode == kMmaW                                                                       \
            ? launch_wide<T, DD>(tmk, tmv, c->sa, p.grid, 32 * p.warps, p.smem, stream)             \
            : launch_split<T, DD, kMma>(tmk, tmv, c->sa, p.grid, 32 * p.warps, p.smem, stream);
  if (s->dtype == PA_BF16) {
    PA_LAUNCH(__nv_bfloat16, 64)
    PA_LAUNCH(__nv_bfloat16, 128)
    PA_LAUNCH(__nv_bfloat16, 256)
  } else {
    PA_LAUNCH(__half, 64)
    PA_LAUNCH(__half, 128)
    PA_LAUNCH(__half, 256)
  }
#undef PA_LAUNCH
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// `overlap`: launch as a programmatic dependent of the split kernel that was
// just enqueued on the same stream (its CTAs may be scheduled while the
// split kernel drains; griddepcontrol.wait orders the reads).
int launch_merge_phase(Call* c, cudaStream_t stream, bool overlap) {
  const Plan& p = c->plan;
  if (p.cluster > 0) return PA_OK;  // the cluster kernel merged already
  // balanced split: one CTA per (segment with pieces to merge, column); such
  // segments continue past a split CTA, so there are fewer than the split
  // CTAs and at most one per row.  Fixed split: one per (row, column).
  const int rows = c->sa.B * c->sa.Hkv;
  // the most pieces a segment can have: its partitions (fixed split), or
  // about the split CTAs per (row, kv head) (balanced split)
  const int64_t pieces =
      p.part_blocks > 0
          ? ((int64_t)c->sa.maxblk + p.part_blocks - 1) / p.part_blocks
          : (int64_t)p.grid / std::max(1, rows) + 2;
  // 8 warps (two rounds of loads fewer): long context, 38 pieces per
  // column, 68.8 -> 68.0 us per step; nothing changes where segments have
  // two or three pieces
  const bool wide = pieces > 2 * kMergeBatch;
  // few pieces per segment (balanced split): column groups, a warp per
  // column.  Same box, step times against the per-column grid: 8-token
  // serving 668.2 -> 654.9 us, 4-token prefix sharing 250.9 -> 238.4,
  // 4-token serving 515.2 -> 510.5, prefix sharing (G = 8) 180.8 -> 178.8,
  // the serving mix 479.4 -> 477.8
  const bool cols = p.part_blocks == 0 && pieces <= kMergeBatch;
  const int ng = (p.C + kColGroup - 1) / kColGroup;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = cols ? dim3(p.grid * ng, 1, 1)
                : p.part_blocks == 0 ? dim3(std::min(p.grid, rows) * p.C, 1, 1)
                                     : dim3(rows, p.C, 1);
  cfg.blockDim = dim3(cols ? 32 * kColGroup : (wide ? 2 * kMergeThreads : kMergeThreads));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  cudaError_t e = cudaErrorInvalidValue;
  if (cols) {
    if (p.D == 64) e = cudaLaunchKernelEx(&cfg, pa_merge_cols_kernel<64>, c->ma);
    if (p.D == 128) e = cudaLaunchKernelEx(&cfg, pa_merge_cols_kernel<128>, c->ma);
    if (p.D == 256) e = cudaLaunchKernelEx(&cfg, pa_merge_cols_kernel<256>, c->ma);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  constexpr int NW = kMergeThreads / 32;
  if (p.D == 64) e = wide ? cudaLaunchKernelEx(&cfg, pa_merge_kernel<64, 2 * NW>, c->ma)
                          : cudaLaunchKernelEx(&cfg, pa_merge_kernel<64, NW>, c->ma);
  if (p.D == 128) e = wide ? cudaLaunchKernelEx(&cfg, pa_merge_kernel<128, 2 * NW>, c->ma)
                           : cudaLaunchKernelEx(&cfg, pa_merge_kernel<128, NW>, c->ma);
  if (p.D == 256) e = wide ? cudaLaunchKernelEx(&cfg, pa_merge_kernel<256, 2 * NW>, c->ma)
                           : cudaLaunchKernelEx(&cfg, pa_merge_kernel<256, NW>, c->ma);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Both phases (the merge as a programmatic dependent of the split), or the
// one options->phase names.
int run_phases(const pa_shape* s, const pa_options* o, const void* k_cache, const void* v_cache,
               Call* c, cudaStream_t st) {
  const int phase = o ? o->phase : PA_PHASE_BOTH;
  if (phase != PA_PHASE_MERGE) {
    const int rc = launch_split_phase(s, k_cache, v_cache, c, st);
    if (rc) return rc;
  }
  if (phase == PA_PHASE_SPLIT) return PA_OK;
  return launch_merge_phase(c, st, phase == PA_PHASE_BOTH);
}

// Device staging that the host-buffer calls add after a plan's workspace:
// the step's block table, lengths, query offsets, the call's status words
// (accumulated, published), then out and q for `rows` query rows (last, so a
// call with fewer rows than the workspace was sized for still fits).
struct HostLayout {
  size_t table, lens, cu, status, out, q, total;
  size_t table_bytes, lens_bytes, cu_bytes, out_bytes, q_bytes;
};

// slot: which of the asynchronous calls' two staging areas (0 for the
// synchronous calls, which have one); `total` covers the slots 0..slot.
HostLayout host_layout(const Plan& p, const pa_shape* s, int64_t rows, bool multi, int slot = 0) {
  HostLayout h;
  const size_t B = (size_t)s->batch, row = (size_t)s->num_heads * s->head_dim;
  h.table_bytes = sizeof(int32_t) * B * (size_t)s->max_blocks_per_seq;
  h.lens_bytes = sizeof(int32_t) * B;
  h.cu_bytes = multi ? sizeof(int32_t) * (B + 1) : 0;
  h.out_bytes = sizeof(float) * (size_t)rows * row;
  h.q_bytes = 2 * (size_t)rows * row;
  // one slot's bytes, laid out as below
  size_t one = round256(h.table_bytes) + round256(h.lens_bytes) + round256(h.cu_bytes) +
               round256(2 * sizeof(uint32_t)) + round256(h.out_bytes) + round256(h.q_bytes);
  size_t off = round256(p.total) + (size_t)slot * one;
  h.table = off;
  off = round256(off + h.table_bytes);
  h.lens = off;
  off = round256(off + h.lens_bytes);
  h.cu = off;
  off = round256(off + h.cu_bytes);
  h.status = off;
  off = round256(off + 2 * sizeof(uint32_t));
  h.out = off;
  off = round256(off + h.out_bytes);
  h.q = off;
  h.total = off + h.q_bytes;
  return h;
}

// The address at which this device's kernels can use `p` directly, if `p`
// is page-locked host memory the device maps (cudaHostAlloc,
// cudaHostRegister) or memory of the current device, and that address is
// aligned to `align` bytes; otherwise null (pageable memory, another
// device's memory: the caller copies instead).
void* mapped_host(const void* p, uintptr_t align) {
  if (!p || (reinterpret_cast<uintptr_t>(p) & (align - 1))) return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != at.device) return nullptr;
  } else if (at.type != cudaMemoryTypeHost) {
    return nullptr;
  }
  if (!at.devicePointer || (reinterpret_cast<uintptr_t>(at.devicePointer) & (align - 1)))
    return nullptr;
  return at.devicePointer;
}

struct HostBuffers {
  const void* q;
  const int32_t* cu;  // several query tokens only
  const int32_t* table;
  const int32_t* lens;
  float* out;
  uint32_t* status;
};

// Where the kernels write out: the caller's buffer itself when the device
// maps it, else the staging (copied back at the end).
float* host_out_target(const HostLayout& h, uint8_t* ws, float* out_host) {
  void* d = mapped_host(out_host, 16);
  return d ? static_cast<float*>(d) : reinterpret_cast<float*>(ws + h.out);
}

// One step from host buffers, after every argument check has passed: stage
// the inputs (by the SMs from page-locked memory the device maps, by copies
// otherwise), run both phases, bring out and the call's status back, wait
// for the stream.  `c` was prepared on the staged inputs and on the output
// target host_out_target chose.
int run_host_step(const pa_shape* s, const pa_options* o, const HostLayout& h, uint8_t* ws,
                  const HostBuffers& hb, const void* k_cache, const void* v_cache, Call* c,
                  cudaStream_t st, bool async = false) {
  // The cluster kernel reads the length, the table row and q once, in its
  // first round trip: when all three sit in page-locked memory the device
  // maps, it reads them there directly and the staging kernel is skipped.
  if (c->plan.cluster > 0 && !hb.cu) {
    const void* dq = mapped_host(hb.q, 16);
    const void* dt = mapped_host(hb.table, 16);
    const void* dl = mapped_host(hb.lens, 16);
    if (dq && dt && dl) {
      uint32_t* slot = reinterpret_cast<uint32_t*>(ws + h.status);
      c->sa.q = static_cast<const uint16_t*>(dq);
      c->sa.table = static_cast<const int32_t*>(dt);
      c->sa.seqlens = static_cast<const int32_t*>(dl);
      uint32_t* published = nullptr;
      if (hb.status) {
        // this call's bits: the slot's word (left at zero by the kernel that
        // published the previous call's), published by the last CTA
        c->sa.status = slot;
        published = static_cast<uint32_t*>(mapped_host(hb.status, 4));
        c->sa.status_out = published ? published : slot + 1;
      }
      int rc = launch_split_phase(s, k_cache, v_cache, c, st);
      if (rc) return rc;
      if (c->sa.out == reinterpret_cast<float*>(ws + h.out) &&
          cudaMemcpyAsync(hb.out, ws + h.out, h.out_bytes, cudaMemcpyDefault, st) != cudaSuccess)
        return PA_ERR_CUDA;
      if (hb.status && !published &&
          cudaMemcpyAsync(hb.status, slot + 1, sizeof(uint32_t), cudaMemcpyDefault, st) !=
              cudaSuccess)
        return PA_ERR_CUDA;
      if (async) return PA_OK;
      return cudaStreamSynchronize(st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
  }
  StageArgs sa = {};
  auto part = [&](const void* host, size_t off, size_t bytes) {
    if (bytes == 0) return PA_OK;
    const void* d = mapped_host(host, 16);
    if (d && bytes % 4 == 0) {
      sa.src[sa.n] = static_cast<const uint32_t*>(d);
      sa.dst[sa.n] = reinterpret_cast<uint32_t*>(ws + off);
      sa.words[sa.n] = (int64_t)(bytes / 4);
      ++sa.n;
      return PA_OK;
    }
    return cudaMemcpyAsync(ws + off, host, bytes, cudaMemcpyDefault, st) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
  };
  int rc = part(hb.q, h.q, h.q_bytes);
  if (!rc) rc = part(hb.table, h.table, h.table_bytes);
  if (!rc) rc = part(hb.lens, h.lens, h.lens_bytes);
  if (!rc && hb.cu) rc = part(hb.cu, h.cu, h.cu_bytes);
  if (rc) return rc;
  uint32_t* slot = reinterpret_cast<uint32_t*>(ws + h.status);
  uint32_t* published = nullptr;
  if (hb.status) {
    // this call's bits: a fresh word, published by the merge kernel
    sa.status = slot;
    c->sa.status = slot;
    c->ma.status = slot;
    published = static_cast<uint32_t*>(mapped_host(hb.status, 4));
    c->ma.status_out = published ? published : slot + 1;
    c->sa.status_out = c->ma.status_out;  // the cluster kernel publishes it itself
  }
  int64_t vec = 0;
  for (int i = 0; i < sa.n; ++i) vec += sa.words[i] / 4;
  const int64_t want = (vec + kStageThreads * 4 - 1) / (kStageThreads * 4);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, 2 * (int64_t)c->plan.grid));
  if (async) {
    // a programmatic dependent of the previous step's merge: fills this
    // call's slot while that kernel finishes (pa_stage_in_kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStageThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, pa_stage_in_kernel, sa) != cudaSuccess) return PA_ERR_CUDA;
  } else {
    pa_stage_in_kernel<<<grid, kStageThreads, 0, st>>>(sa);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  rc = run_phases(s, o, k_cache, v_cache, c, st);
  if (rc) return rc;
  const cudaMemcpyKind back = cudaMemcpyDefault;
  if (c->sa.out == reinterpret_cast<float*>(ws + h.out) &&
      cudaMemcpyAsync(hb.out, ws + h.out, h.out_bytes, back, st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (hb.status && !published &&
      cudaMemcpyAsync(hb.status, slot + 1, sizeof(uint32_t), back, st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (async) return PA_OK;
  return cudaStreamSynchronize(st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

int pa_version(void) { return 100; }

int pa_workspace_size(const pa_shape* shape, const pa_options* options, size_t* bytes) {
  if (!shape || !bytes) return PA_ERR_NULL;
  Plan p;
  int rc = make_plan(shape, options, false, &p);
  if (rc) return rc;
  *bytes = p.total;
  return PA_OK;
}

int pa_launch_plan(const pa_shape* shape, const pa_options* options, int32_t max_q,
                   int32_t* info) {
  if (!shape || !info) return PA_ERR_NULL;
  if (max_q < 0) return PA_ERR_SHAPE;
  Plan p;
  const int rc = make_plan(shape, options, true, &p, max_q);
  if (rc) return rc;
  info[0] = p.cluster > 0 ? 1 : 2;
  info[1] = p.cluster > 0 ? p.cluster * shape->batch * shape->num_kv_heads : p.grid;
  info[2] = p.cluster;
  info[3] = p.cluster > 0 ? p.cring : p.ring;
  return PA_OK;
}

int pa_decode_split(const pa_shape* shape, const pa_options* options, const void* q,
                    const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* cache_seqlens, float scale, float* out, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
  if (shape && shape->batch == 0 && check_shape(shape) == PA_OK) return PA_OK;
  Call c;
  int rc = prepare(shape, options, q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                   workspace, workspace_bytes, true, &c);
  if (rc) return rc;
  return launch_split_phase(shape, k_cache, v_cache, &c, reinterpret_cast<cudaStream_t>(stream));
}

int pa_decode_merge(const pa_shape* shape, const pa_options* options, const void* q,
                    const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* cache_seqlens, float scale, float* out, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
  if (shape && shape->batch == 0 && check_shape(shape) == PA_OK) return PA_OK;
  Call c;
  int rc = prepare(shape, options, q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                   workspace, workspace_bytes, false, &c);
  if (rc) return rc;
  return launch_merge_phase(&c, reinterpret_cast<cudaStream_t>(stream), false);
}

int pa_decode(const pa_shape* shape, const pa_options* options, const void* q,
              const void* k_cache, const void* v_cache, const int32_t* block_table,
              const int32_t* cache_seqlens, float scale, float* out, void* workspace,
              size_t workspace_bytes, pa_stream_t stream) {
  if (shape && shape->batch == 0 && check_shape(shape) == PA_OK) return PA_OK;
  Call c;
  int rc = prepare(shape, options, q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                   workspace, workspace_bytes, true, &c);
  if (rc) return rc;
  return run_phases(shape, options, k_cache, v_cache, &c, reinterpret_cast<cudaStream_t>(stream));
}

int pa_decode_append(const pa_shape* shape, const pa_options* options, const void* q,
                     const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const int32_t* block_table, const int32_t* cache_seqlens, float scale,
                     float* out, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (shape && shape->batch == 0 && check_shape(shape) == PA_OK) return PA_OK;
  if (!k_new || !v_new) return PA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new)) return PA_ERR_ALIGN;
  if (options && options->compute == PA_COMPUTE_TC) return PA_ERR_OPTION;  // not with the append
  Call c;
  int rc = prepare(shape, options, q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                   workspace, workspace_bytes, true, &c);
  if (rc) return rc;
  c.plan.cluster = 0;  // the appended row is written by the split kernel
  c.sa.len_add = 1;
  c.sa.k_new = static_cast<const uint16_t*>(k_new);
  c.sa.v_new = static_cast<const uint16_t*>(v_new);
  c.sa.k_pool = static_cast<uint16_t*>(k_cache);
  c.sa.v_pool = static_cast<uint16_t*>(v_cache);
  return run_phases(shape, options, k_cache, v_cache, &c, reinterpret_cast<cudaStream_t>(stream));
}

int pa_workspace_size_multi(const pa_shape* shape, const pa_options* options, int32_t max_q,
                            size_t* bytes) {
  if (!shape || !bytes) return PA_ERR_NULL;
  if (max_q < 1) return PA_ERR_SHAPE;
  Plan p;
  int rc = make_plan(shape, options, false, &p, max_q);
  if (rc) return rc;
  *bytes = p.total;
  return PA_OK;
}

int pa_decode_multi(const pa_shape* shape, const pa_options* options, const void* q,
                    const int32_t* cu_seqlens_q, int32_t total_q, int32_t max_q, int32_t causal,
                    const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* cache_seqlens, float scale, float* out, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
  if (max_q < 1 || total_q < 0) return PA_ERR_SHAPE;
  if (shape && shape->batch == 0 && check_shape(shape) == PA_OK) return PA_OK;
  if (!cu_seqlens_q) return PA_ERR_NULL;
  if (!aligned16(cu_seqlens_q)) return PA_ERR_ALIGN;
  if (total_q == 0) return PA_OK;
  Call c;
  int rc = prepare(shape, options, q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
                   workspace, workspace_bytes, true, &c, max_q);
  if (rc) return rc;
  c.sa.cu_q = cu_seqlens_q;
  c.sa.causal = causal ? 1 : 0;
  c.sa.total_q = total_q;
  c.ma.cu_q = cu_seqlens_q;
  c.ma.total_q = total_q;
  return run_phases(shape, options, k_cache, v_cache, &c, reinterpret_cast<cudaStream_t>(stream));
}

int pa_workspace_size_host(const pa_shape* shape, const pa_options* options, size_t* bytes) {
  if (!shape || !bytes) return PA_ERR_NULL;
  Plan p;
  int rc = make_plan(shape, options, false, &p);
  if (rc) return rc;
  *bytes = host_layout(p, shape, shape->batch, false).total;
  return PA_OK;
}

int pa_workspace_size_host_async(const pa_shape* shape, const pa_options* options,
                                 size_t* bytes) {
  if (!shape || !bytes) return PA_ERR_NULL;
  Plan p;
  int rc = make_plan(shape, options, false, &p);
  if (rc) return rc;
  *bytes = host_layout(p, shape, shape->batch, false, 1).total;
  return PA_OK;
}

}  // extern "C"

namespace {

// pa_decode_host and pa_decode_host_async: slot < 0 waits for the stream.
int decode_host(const pa_shape* shape, const pa_options* options, const void* q_host,
                const void* k_cache, const void* v_cache, const int32_t* block_table_host,
                const int32_t* cache_seqlens_host, float scale, float* out_host,
                uint32_t* status_host, int slot, void* workspace, size_t workspace_bytes,
                pa_stream_t stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (options && options->phase != PA_PHASE_BOTH) return PA_ERR_OPTION;
  if (slot > 1) return PA_ERR_OPTION;
  if (shape->batch == 0) {  // a no-op, as for pa_decode
    if (status_host) *status_host = 0;
    return PA_OK;
  }
  if (!q_host || !block_table_host || !cache_seqlens_host || !out_host || !workspace)
    return PA_ERR_NULL;
  Plan p;
  rc = make_plan(shape, options, false, &p);
  if (rc) return rc;
  const HostLayout h = host_layout(p, shape, shape->batch, false, slot < 0 ? 0 : slot);
  if (workspace_bytes < h.total) return PA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Call c;
  rc = prepare(shape, options, ws + h.q, k_cache, v_cache,
               reinterpret_cast<const int32_t*>(ws + h.table),
               reinterpret_cast<const int32_t*>(ws + h.lens), scale,
               host_out_target(h, ws, out_host), workspace, p.total, true, &c);
  if (rc) return rc;
  const HostBuffers hb{q_host, nullptr, block_table_host, cache_seqlens_host, out_host,
                       status_host};
  return run_host_step(shape, options, h, ws, hb, k_cache, v_cache, &c,
                       reinterpret_cast<cudaStream_t>(stream), slot >= 0);
}

int decode_multi_host(const pa_shape* shape, const pa_options* options, const void* q_host,
                      const int32_t* cu_seqlens_q_host, int32_t total_q, int32_t max_q,
                      int32_t causal, const void* k_cache, const void* v_cache,
                      const int32_t* block_table_host, const int32_t* cache_seqlens_host,
                      float scale, float* out_host, uint32_t* status_host, int slot,
                      void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (max_q < 1 || total_q < 0) return PA_ERR_SHAPE;
  int rc = check_shape(shape);
  if (rc) return rc;
  if (options && options->phase != PA_PHASE_BOTH) return PA_ERR_OPTION;
  if (slot > 1) return PA_ERR_OPTION;
  if (shape->batch == 0 || total_q == 0) {  // nothing to attend
    if (status_host) *status_host = 0;
    return PA_OK;
  }
  if (!q_host || !cu_seqlens_q_host || !block_table_host || !cache_seqlens_host || !out_host ||
      !workspace)
    return PA_ERR_NULL;
  Plan p;
  rc = make_plan(shape, options, false, &p, max_q);
  if (rc) return rc;
  const HostLayout h = host_layout(p, shape, total_q, true, slot < 0 ? 0 : slot);
  if (workspace_bytes < h.total) return PA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Call c;
  rc = prepare(shape, options, ws + h.q, k_cache, v_cache,
               reinterpret_cast<const int32_t*>(ws + h.table),
               reinterpret_cast<const int32_t*>(ws + h.lens), scale,
               host_out_target(h, ws, out_host), workspace, p.total, true, &c, max_q);
  if (rc) return rc;
  const int32_t* cu = reinterpret_cast<const int32_t*>(ws + h.cu);
  c.sa.cu_q = cu;
  c.sa.causal = causal ? 1 : 0;
  c.sa.total_q = total_q;
  c.ma.cu_q = cu;
  c.ma.total_q = total_q;
  const HostBuffers hb{q_host, cu_seqlens_q_host, block_table_host, cache_seqlens_host, out_host,
                       status_host};
  return run_host_step(shape, options, h, ws, hb, k_cache, v_cache, &c,
                       reinterpret_cast<cudaStream_t>(stream), slot >= 0);
}

}  // namespace

extern "C" {

int pa_decode_host(const pa_shape* shape, const pa_options* options, const void* q_host,
                   const void* k_cache, const void* v_cache, const int32_t* block_table_host,
                   const int32_t* cache_seqlens_host, float scale, float* out_host,
                   uint32_t* status_host, void* workspace, size_t workspace_bytes,
                   pa_stream_t stream) {
  return decode_host(shape, options, q_host, k_cache, v_cache, block_table_host,
                     cache_seqlens_host, scale, out_host, status_host, -1, workspace,
                     workspace_bytes, stream);
}

int pa_decode_host_async(const pa_shape* shape, const pa_options* options, const void* q_host,
                         const void* k_cache, const void* v_cache,
                         const int32_t* block_table_host, const int32_t* cache_seqlens_host,
                         float scale, float* out_host, uint32_t* status_host, int32_t slot,
                         void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (slot < 0) return PA_ERR_OPTION;
  return decode_host(shape, options, q_host, k_cache, v_cache, block_table_host,
                     cache_seqlens_host, scale, out_host, status_host, slot, workspace,
                     workspace_bytes, stream);
}

int pa_workspace_size_multi_host(const pa_shape* shape, const pa_options* options, int32_t max_q,
                                 int32_t max_total_q, size_t* bytes) {
  if (!shape || !bytes) return PA_ERR_NULL;
  if (max_q < 1 || max_total_q < 0) return PA_ERR_SHAPE;
  Plan p;
  int rc = make_plan(shape, options, false, &p, max_q);
  if (rc) return rc;
  *bytes = host_layout(p, shape, max_total_q, true).total;
  return PA_OK;
}

int pa_workspace_size_multi_host_async(const pa_shape* shape, const pa_options* options,
                                       int32_t max_q, int32_t max_total_q, size_t* bytes) {
  if (!shape || !bytes) return PA_ERR_NULL;
  if (max_q < 1 || max_total_q < 0) return PA_ERR_SHAPE;
  Plan p;
  int rc = make_plan(shape, options, false, &p, max_q);
  if (rc) return rc;
  *bytes = host_layout(p, shape, max_total_q, true, 1).total;
  return PA_OK;
}

int pa_decode_multi_host(const pa_shape* shape, const pa_options* options, const void* q_host,
                         const int32_t* cu_seqlens_q_host, int32_t total_q, int32_t max_q,
                         int32_t causal, const void* k_cache, const void* v_cache,
                         const int32_t* block_table_host, const int32_t* cache_seqlens_host,
                         float scale, float* out_host, uint32_t* status_host, void* workspace,
                         size_t workspace_bytes, pa_stream_t stream) {
  return decode_multi_host(shape, options, q_host, cu_seqlens_q_host, total_q, max_q, causal,
                           k_cache, v_cache, block_table_host, cache_seqlens_host, scale,
                           out_host, status_host, -1, workspace, workspace_bytes, stream);
}

int pa_decode_multi_host_async(const pa_shape* shape, const pa_options* options,
                               const void* q_host, const int32_t* cu_seqlens_q_host,
                               int32_t total_q, int32_t max_q, int32_t causal,
                               const void* k_cache, const void* v_cache,
                               const int32_t* block_table_host,
                               const int32_t* cache_seqlens_host, float scale, float* out_host,
                               uint32_t* status_host, int32_t slot, void* workspace,
                               size_t workspace_bytes, pa_stream_t stream) {
  if (slot < 0) return PA_ERR_OPTION;
  return decode_multi_host(shape, options, q_host, cu_seqlens_q_host, total_q, max_q, causal,
                           k_cache, v_cache, block_table_host, cache_seqlens_host, scale,
                           out_host, status_host, slot, workspace, workspace_bytes, stream);
}

int pa_cache_append(const pa_shape* shape, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* block_table, const int32_t* cache_seqlens,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !cache_seqlens || !workspace)
    return PA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(block_table) || !aligned16(cache_seqlens) || !aligned16(workspace))
    return PA_ERR_ALIGN;
  if (workspace_bytes < kHeaderBytes) return PA_ERR_WORKSPACE;
  if (shape->batch == 0) return PA_OK;
  AppendArgs a;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_cache = static_cast<uint16_t*>(k_cache);
  a.v_cache = static_cast<uint16_t*>(v_cache);
  a.table = block_table;
  a.seqlens = cache_seqlens;
  a.status = static_cast<uint32_t*>(workspace);
  a.B = shape->batch;
  a.Hkv = shape->num_kv_heads;
  a.D = shape->head_dim;
  a.bs = shape->block_size;
  a.maxblk = shape->max_blocks_per_seq;
  a.P = shape->num_blocks;
  pa_append_kernel<<<shape->batch, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_read_status(void* workspace, uint32_t* flags, pa_stream_t stream) {
  if (!workspace || !flags) return PA_ERR_NULL;
  if (!aligned16(workspace)) return PA_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof v, st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  *flags = v;
  return PA_OK;
}

const char* pa_status_string(int code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_SHAPE: return "unsupported or inconsistent shape or dtype";
    case PA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case PA_ERR_WORKSPACE: return "workspace smaller than pa_workspace_size";
    case PA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case PA_ERR_OPTION: return "invalid pa_options value";
    case PA_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the built-in static buffer "
             "(PA_STATIC_SCRATCH_BYTES) of pa_decode_noalloc holds";
    case PA_ERR_STATE: return "block manager: invalid handle, id, index or request";
    case PA_ERR_NO_BLOCKS: return "block manager: not enough free blocks";
    default: break;
  }
  if (code > 0) {
    if (code & PA_STATUS_TIMEOUT) return "device: a pipeline wait gave up";
    if (code & PA_STATUS_BAD_SEQLEN) return "device: cache_seqlens entry out of range";
    if (code & PA_STATUS_BAD_BLOCK) return "device: block_table entry unmapped or out of range";
    if (code & PA_STATUS_NO_SLOT) return "device: appended token has no cache slot";
  }
  return "unknown code";
}

int pa_plan_pieces(const pa_shape* shape, const pa_options* options,
                   const int32_t* cache_seqlens_host, int32_t num_ctas, int32_t cta,
                   int32_t* pieces, int32_t max_pieces) {
  int rc = check_shape(shape);
  if (rc) return rc;
  rc = check_options(shape, options);
  if (rc) return rc;
  if (!cache_seqlens_host || (!pieces && max_pieces > 0)) return PA_ERR_NULL;
  if (num_ctas < 1 || cta < 0 || cta >= num_ctas) return PA_ERR_OPTION;
  const int B = shape->batch;
  const int part_blocks =
      (options && options->partition_tokens > 0) ? options->partition_tokens / shape->block_size : 0;
  const int K = part_blocks == 0 ? piece_units(shape->block_size, shape->head_dim) : 0;
  int32_t* pre = new int32_t[B + 1];
  pre[0] = 0;
  for (int b = 0; b < B; ++b)
    pre[b + 1] = pre[b] + seq_count(seq_blocks(cache_seqlens_host[b], shape->block_size,
                                               shape->max_blocks_per_seq),
                                    part_blocks, K);
  const SchedShape sched{B,           shape->num_kv_heads, shape->block_size, shape->max_blocks_per_seq,
                         part_blocks, num_ctas,            0,                 K};
  PieceIter it;
  it.init(pre, HostLens{cache_seqlens_host, 0, shape->block_size, shape->max_blocks_per_seq},
          sched, cta);
  Piece pc;
  int n = 0;
  while (it.next(pc)) {
    if (n < max_pieces) {
      pieces[5 * n + 0] = pc.b;
      pieces[5 * n + 1] = pc.j;
      pieces[5 * n + 2] = pc.blk0;
      pieces[5 * n + 3] = pc.blk1;
      pieces[5 * n + 4] = pc.slot;
    }
    ++n;
  }
  delete[] pre;
  return n;
}

int pa_plan_merge(const pa_shape* shape, const pa_options* options,
                  const int32_t* cache_seqlens_host, int32_t num_ctas, int32_t seg,
                  int32_t* b_j, int32_t* slots, int32_t max_slots) {
  int rc = check_shape(shape);
  if (rc) return rc;
  rc = check_options(shape, options);
  if (rc) return rc;
  if (!cache_seqlens_host || !b_j || (!slots && max_slots > 0)) return PA_ERR_NULL;
  if (num_ctas < 1 || seg < 0) return PA_ERR_OPTION;
  const int B = shape->batch;
  const int part_blocks =
      (options && options->partition_tokens > 0) ? options->partition_tokens / shape->block_size : 0;
  const int nseg = part_blocks == 0 ? num_ctas : B * shape->num_kv_heads;
  if (seg >= nseg) return PA_ERR_OPTION;
  const int K = part_blocks == 0 ? piece_units(shape->block_size, shape->head_dim) : 0;
  int32_t* pre = new int32_t[B + 1];
  pre[0] = 0;
  for (int b = 0; b < B; ++b)
    pre[b + 1] = pre[b] + seq_count(seq_blocks(cache_seqlens_host[b], shape->block_size,
                                               shape->max_blocks_per_seq),
                                    part_blocks, K);
  const SchedShape sched{B,           shape->num_kv_heads, shape->block_size, shape->max_blocks_per_seq,
                         part_blocks, num_ctas,            0,                 K};
  int32_t db = -1, dj = 0, dlast = 0, dslot = 0;
  if (part_blocks == 0 && !balanced_split_segment(pre, sched, seg, db, dj, dlast, dslot)) db = -1;
  const MergeSeg ms = merge_segment(sched, seg, db, dj, dlast, dslot, pre);
  b_j[0] = ms.np > 0 ? ms.b : -1;
  b_j[1] = ms.np > 0 ? ms.j : -1;
  for (int p = 0; p < ms.np && p < max_slots; ++p) slots[p] = (int32_t)ms.slot(p);
  delete[] pre;
  return ms.np;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without any caller-provided or library-allocated workspace.
//
// Some callers cannot allocate device memory where they run a decode step:
// a plugin whose host framework owns every device allocation, or a serving
// loop that fixes its memory at start-up and may not call cudaMalloc (which
// can also synchronise the device) on its hot path.  For them the scratch the
// split and merge kernels need (status word, prefix sums, merge descriptors,
// partial states) lives in one file-scope device array of a fixed size,
// reserved on every GPU that loads this library for as long as the process
// runs.  Nothing here calls cudaMalloc, cudaFree or an allocating library
// routine.

static __device__ __align__(256) uint8_t g_pa_static_scratch[PA_STATIC_SCRATCH_BYTES];

namespace {

void* g_static_ptr[kMaxDevices];

// Once per device, with that device current: the array's device address.
// (In host code the array's name is only a host-side stand-in.)  The first
// call also zeroes the array's header (status word and the split kernel's
// work counters, which must start at zero) on the caller's stream, so the
// zeroing is ordered before that call's kernels.
int static_scratch(void** ptr, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_static_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, kHeaderBytes, stream) != cudaSuccess) return PA_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(const pa_shape* shape, const pa_options* options, const void* q,
                                 const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* cache_seqlens,
                                 float scale, float* out, uint32_t* status, pa_stream_t stream) {
  if (shape && shape->batch == 0 && check_shape(shape) == PA_OK) return PA_OK;
  int rc = check_shape(shape);
  if (rc) return rc;
  rc = check_options(shape, options);
  if (rc) return rc;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return PA_ERR_ALIGN;
  // both phases always run here: the scratch is not the caller's to carry
  // from a split-only call to a merge-only one
  if (options && options->phase != PA_PHASE_BOTH) return PA_ERR_OPTION;
  Plan plan;
  rc = make_plan(shape, options, false, &plan);
  if (rc) return rc;
  if (plan.total > (size_t)PA_STATIC_SCRATCH_BYTES) return PA_ERR_SCRATCH_LIMIT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  rc = static_scratch(&scratch, st);
  if (rc) return rc;
  Call c;
  rc = prepare(shape, options, q, k_cache, v_cache, block_table, cache_seqlens, scale, out,
               scratch, (size_t)PA_STATIC_SCRATCH_BYTES, true, &c);
  if (rc) return rc;
  if (status) c.sa.status = status;
  rc = launch_split_phase(shape, k_cache, v_cache, &c, st);
  if (rc) return rc;
  return launch_merge_phase(&c, st, true);
}
