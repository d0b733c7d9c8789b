// pa_cluster.cuh -- one decode step in one kernel for steps with few
// (sequence, kv head) segments: each segment is handled by one thread-block
// cluster of CS CTAs (CS <= 8), and the CTAs fold their partial states
// through distributed shared memory.
//
// The persistent split kernel (pa_split.cuh) spreads a small step over all
// SMs by cutting segments across CTAs, which then needs the length prefix
// sums, partial states in the workspace and a second (merge) kernel: at a
// few MB of K/V those dependent round trips, not the bytes, set the time.
// Here the launch shape comes from the shape alone (grid CS x B*Hkv), so:
//   - no prefix sums: CTA rank r of cluster (b, j) takes blocks
//     [r n / CS, (r+1) n / CS) of the n = ceil(len_b / bs) blocks;
//   - one round trip brings the length, the whole block-table row (into
//     shared memory) and q, before the length is known;
//   - the K/V tiles stream through the same per-warp TMA rings and the same
//     tensor-core tile (MmaState) as the split kernel; the CTA then folds its
//     warps' states with the same combine op (combine_piece) into its own
//     shared memory;
//   - the cluster's CS states are folded with that combine op ("Paged
//     Attention Kernel Architecture for BI-V100", section 2, Levels 1-3),
//     in rank order, each CTA reading its peers' shared memory for its share
//     of the (column, 4 dims) outputs -- no workspace, no merge kernel.
#pragma once

#include "pa_split.cuh"

namespace pa {

template <typename T, int D>
__global__ void __launch_bounds__(32 * split_warps(D), 1)
    pa_cluster_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ SplitArgs a) {
  constexpr int W = split_warps(D);
  constexpr int NC = D / 64;
  constexpr uint32_t chunk = kTile * 128u;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int R = a.ring;
  const int C = a.C;
  const ClusterLayout CL = cluster_layout(D, C, W, R, a.maxblk);
  const SmemLayout& L = CL.s;
  const uint32_t CS = gridDim.x;  // the cluster spans the grid's x extent
  const uint32_t rank = cluster_ctarank();
  const int seg = blockIdx.y, b = seg / a.Hkv, j = seg - b * a.Hkv;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  int32_t* tab = reinterpret_cast<int32_t*>(smem + CL.table);
  float* qs = reinterpret_cast<float*>(smem + L.qs);
  const uint32_t qraw = base + L.qraw;
  // the argument copy the CTA-level combine reads, with its partial-state
  // pointers aimed at this CTA's shared memory (slot 0)
  SplitArgs* sa = reinterpret_cast<SplitArgs*>(smem + kArgsOffset);
  for (int i = tid; i < (int)(sizeof(SplitArgs) / 4); i += blockDim.x)
    reinterpret_cast<uint32_t*>(sa)[i] = reinterpret_cast<const uint32_t*>(&a)[i];
  if (tid == 0) {
    for (int s = 0; s < W * R; ++s) mbar_init(base + L.full + 8 * s, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < D / 8; i += blockDim.x) sts128(base + L.zrow + 16u * i, make_uint4(0u, 0u, 0u, 0u));
  if (lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncthreads();
  if (tid == 0) {
    sa->ws_acc = reinterpret_cast<float*>(smem + CL.st_acc);
    sa->ws_ml = reinterpret_cast<float*>(smem + CL.st_ml);
  }
  const uint64_t wait_ns = a.wait_us > 0 ? (uint64_t)a.wait_us * 1000ull : kWaitLimitNs;
  // As a programmatic dependent of the kernel before it, the grid may be
  // resident while that kernel finishes; from here on its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- one round trip: the length, the whole table row, q.  Plain loads:
  // with the host-buffer calls these three may be page-locked host memory
  // the device maps, read here directly.
  const int32_t stored = a.seqlens[b];
  for (int i = tid; i < a.maxblk; i += blockDim.x) tab[i] = a.table[(int64_t)b * a.maxblk + i];
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.H + (int64_t)j * a.G) * D);
    for (int i = tid; i < C * D / 8; i += blockDim.x) sts128(qraw + 16u * i, src[i]);
  }
  const int32_t len = eff_len(stored, 0, a.bs, a.maxblk);  // -1: not a valid length
  const int nblk = len >= 0 ? seq_blocks(len, a.bs, a.maxblk) : 0;
  const int blk0 = (int)((int64_t)nblk * rank / CS), blk1 = (int)((int64_t)nblk * (rank + 1) / CS);
  const int sl = a.bs == 16 ? 0 : (a.bs == 32 ? 1 : 2);  // log2(16-token tiles per block)
  const int nt = (blk1 - blk0) << sl;
  const int cnt = nt > w ? (nt - w + W - 1) / W : 0;  // this warp's tiles: w, w + W, ...
  if (len < 0 && rank == 0 && tid == 0) atomicOr(a.status, kStatusBadSeqlen);
  __syncthreads();  // the table row, q and the argument copy are in place
  // ---- the CTA's tiles through the warps' rings
  auto issue = [&](int n, uint32_t slot) {
    if (lane == 0) {
      const int t = w + W * n;
      const int blk = blk0 + (t >> sl), h = t & ((1 << sl) - 1);
      const int32_t phys = tab[blk];
      const int valid = max(0, min(kTile, len - blk * a.bs - h * kTile));
      const bool bad = phys < 0 || phys >= a.P;
      const uint32_t gslot = (uint32_t)w * R + slot;
      const uint32_t full = base + L.full + 8 * gslot;
      sts64(base + L.info + 8 * gslot,
            ((uint64_t)(uint32_t)phys << 32) | (uint32_t)valid | (bad ? kInfoBad : 0u));
      if (bad || valid == 0) {
        if (bad && h == 0) atomicOr(a.status, kStatusBadBlock);
        mbar_arrive(full);
      } else {
        const uint64_t pol = l2_evict_first_policy();
        mbar_arrive_expect_tx(full, L.stage_bytes);
        const uint32_t kdst = base + L.stage + gslot * L.stage_bytes;
        if (a.kv_fused) {
          tma_load_5d(kdst, &tmk, full, 0, h * kTile, 0, phys * a.bs * a.Hkv + j, 0, pol);
        } else {
          tma_load_5d(kdst, &tmk, full, 0, h * kTile, 0, j, phys, pol);
          tma_load_5d(kdst + NC * chunk, &tmv, full, 0, h * kTile, 0, j, phys, pol);
        }
      }
    }
  };
  // the ring's first copies go out before q is widened: they need only
  // the table row and the length
  int issued = 0;
  for (int r = 0; r < R && r < cnt; ++r, ++issued) issue(r, (uint32_t)r);
  for (int i = tid; i < C * D / 2; i += blockDim.x) {
    const int c = (2 * i) / D, d = (2 * i) % D;
    const uint32_t v = lds32(qraw + 4u * i);
    *reinterpret_cast<float2*>(qs + c * (D + 4) + d) = make_float2(Cvt<T>::low(v), Cvt<T>::high(v));
  }
  __syncthreads();

  MmaState<T, D, 1, false> mst;
  mst.load_q(qs, C, nullptr, a.qscale);
  mst.reset();
  bool bad = len < 0, stop = false;
  int first_fail = -1;
  uint32_t slot = 0, phase = 0;
  for (int n = 0; n < cnt; ++n) {
    const uint32_t gslot = (uint32_t)w * R + slot;
    const bool ok = __all_sync(
        0xffffffffu, mbar_wait_bounded(base + L.full + 8 * gslot, (phase >> slot) & 1u, abort_flag, wait_ns));
    if (!ok && first_fail < 0) first_fail = n;
    const uint64_t info64 = lds64(base + L.info + 8 * gslot);
    const uint32_t info = (uint32_t)info64;
    const int valid = (int)(info & 0xffffu);
    if (!ok || (info & kInfoBad)) {
      bad = true;
      if (!ok) {
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        stop = true;
      }
    } else if (valid > 0) {
      const uint32_t sb = base + L.stage + gslot * L.stage_bytes;
      const uint32_t kb = sb + (a.kv_swap ? NC * chunk : 0u);
      const uint32_t vb = sb + (a.kv_swap ? 0u : NC * chunk);
      const int t = w + W * n;
      const int tok0 = (blk0 + (t >> sl)) * a.bs + (t & ((1 << sl) - 1)) * kTile;
      mst.tile(kb, vb, valid, tok0, -1, 0u, 0u, base + L.zrow);
    }
    __syncwarp();
    phase ^= 1u << slot;
    if (!stop && n + R < cnt) {
      issue(n + R, slot);
      ++issued;
    }
    slot = (slot + 1 == (uint32_t)R) ? 0u : slot + 1;
  }
  if (first_fail >= 0 && lane == 0) {
    // as in the split kernel: wait (bounded, ignoring the abort flag) for
    // the copies this warp may still have in flight -- tile n sits in slot
    // n % R in phase (n / R) & 1
    volatile int never = 0;
    for (int kk = first_fail; kk < issued; ++kk)
      mbar_wait_bounded(base + L.full + 8 * ((uint32_t)w * R + (uint32_t)(kk % R)),
                        (uint32_t)((kk / R) & 1), &never, kWaitLimitNs / 4);
  }

  // ---- the CTA's state: its warps folded (into shared memory, slot 0)
  mst.bad |= bad;
  mst.publish(smem, L, w, C, C);
  __syncthreads();
  const Piece pc{b, j, blk0, blk1, 0};
  combine_piece<D, W, false, false>(*sa, smem, L, pc, 0, 0, 0);

  // ---- the cluster's states, folded in rank order (the cluster barrier
  // also orders this CTA's own threads: no separate CTA barrier)
  cluster_sync();
  float* wts = reinterpret_cast<float*>(smem + CL.wts);
  const uint32_t ml_addr = base + CL.st_ml, acc_addr = base + CL.st_acc;
  if (tid < C) {
    const int c = tid;
    float mr[kMaxCluster], lr[kMaxCluster];
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      mr[r] = -INFINITY;
      lr[r] = 0.f;
      if (r < (int)CS) {
        mr[r] = ld_dsmem_f32(dsmem_addr(ml_addr + 8u * c, r));
        lr[r] = ld_dsmem_f32(dsmem_addr(ml_addr + 8u * c + 4u, r));
        M = fmaxf(M, mr[r]);
      }
    }
    float e[kMaxCluster];
    float Lsum = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      // an empty state (m = -inf) gets weight 0; a NaN it carries (a bad
      // piece or length) still reaches the result through 0 * NaN
      e[r] = (mr[r] == -INFINITY) ? 0.f : ex2(mr[r] - M);
      Lsum = fmaf(e[r], lr[r], Lsum);
    }
    // a column that saw no key (an empty sequence) gets 0
    const float inv = Lsum == 0.f ? 0.f : 1.f / Lsum;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) wts[c * kMaxCluster + r] = e[r] * inv;
  }
  __syncthreads();
  constexpr int DV = D / 4;
  const int nvec = C * DV;
  const int v0 = (int)((int64_t)nvec * rank / CS), v1 = (int)((int64_t)nvec * (rank + 1) / CS);
  for (int v = v0 + tid; v < v1; v += blockDim.x) {
    const int c = v / DV, d4 = (v - c * DV) * 4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint32_t r = 0; r < CS; ++r) {
      const float wr = wts[c * kMaxCluster + r];
      const float4 x = ld_dsmem_f32x4(dsmem_addr(acc_addr + 4u * (uint32_t)(c * D + d4), r));
      o.x = fmaf(wr, x.x, o.x);
      o.y = fmaf(wr, x.y, o.y);
      o.z = fmaf(wr, x.z, o.z);
      o.w = fmaf(wr, x.w, o.w);
    }
    *reinterpret_cast<float4*>(a.out + ((int64_t)b * a.H + (int64_t)j * a.G + c) * D + d4) = o;
  }
  // this thread is done reading the others' shared memory
  cluster_arrive();
  if (a.status_out) {
    // this thread's status bits and outputs, before the count below
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      // host-buffer calls: the last CTA to finish publishes the call's status
      if (atomicAdd(a.done, 1u) == gridDim.x * gridDim.y - 1) {
        __threadfence();
        volatile uint32_t* st = a.status;
        *a.status_out = *st;
        *st = 0u;
        *reinterpret_cast<volatile uint32_t*>(a.done) = 0u;
      }
    }
  }
  // no CTA leaves while another still reads its shared memory
  cluster_wait();
}

template <typename T, int D>
cudaError_t launch_cluster(const CUtensorMap& tmk, const CUtensorMap& tmv, const SplitArgs& a, int cs,
                           int segs, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, segs, 1);
  cfg.blockDim = dim3(32 * split_warps(D));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, pa_cluster_kernel<T, D>, tmk, tmv, a);
}

// Clusters of `cs` CTAs with this much shared memory that can be resident
// at once (0 on error); also raises the kernel's shared-memory limit.
template <typename T, int D>
int cluster_capacity(int cs, size_t smem, int max_smem) {
  const void* fn = reinterpret_cast<const void*>(&pa_cluster_kernel<T, D>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, 1, 1);
  cfg.blockDim = dim3(32 * split_warps(D));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace pa

#define PA_INSTANTIATE_CLUSTER(T, D)                                                          \
  template cudaError_t pa::launch_cluster<T, D>(const CUtensorMap&, const CUtensorMap&,       \
                                                const pa::SplitArgs&, int, int, size_t,       \
                                                cudaStream_t);                                \
  template int pa::cluster_capacity<T, D>(int, size_t, int);
