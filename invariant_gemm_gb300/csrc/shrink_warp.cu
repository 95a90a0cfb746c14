// LoRA shrink for small ranks: Z = scale * X A_i^T with a Split-K reduction,
// the partials on the warp-level tensor cores (shrink_core.cuh).
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction":
//   Eq. 3 / Fig. 1  S thread blocks per output tile, block s sums over the
//                   s-th contiguous K partition;
//   Algorithm 1     DET: FP32 partial -> scratch, gpu fence, block barrier,
//                   acq_rel integer increment of the tile's counter; the block
//                   that saw S-1 sums scratch[t][0..S-1] in increasing order,
//                   multiplies by the scale, writes the tile and zeroes the
//                   counter;
//   sec. 4.1        ATOMIC: FP32 atomic add of scale * partial into zeroed Z;
//   sec. 4.2        UNSPLIT: S = 1, one block over the whole of K;
//   sec. 4.3        DET_TREE: partials only, combined by reduce_tree.cu.
//
// Block = BN/4 warps, tile = up to 8 token rows of one adapter (one entry of
// the token map's tile table) x BN rank columns, one K partition; thread o
// ends with the output of token row o / BN, rank o % BN. The A rows of the
// partition are streamed through shared memory in k-blocks of 256 elements
// by TMA copies (completion counted on an mbarrier), four stages deep; x goes
// from global memory straight into registers (shrink_core.cuh).
//
// Latency: the tile entry is read before griddep_wait() (the token map is
// complete before this kernel starts); with IG_FLAG_STATIC_WEIGHTS the A
// rows of the first stages are requested before it too, so only the x rows
// wait for the previous kernel; L2 is asked for those early as well.
//
// Reduction order inside a partition (shrink_core.cuh): 64-element groups
// dealt round-robin to the warps, each warp's groups accumulated in
// increasing k by bf16 MMAs into two FP32 accumulators, then the warp sums
// added in warp order. It depends only on K/S and BN.
#include <map>
#include <mutex>

#include "shrink_core.cuh"

namespace ig {

namespace {

template <int BN>
struct ShrinkSmem {
  static constexpr int kStagesOff = 1024;                          // mbarriers + info
  static constexpr int kRedOff = kStagesOff + kShrinkStages * PartialRing<BN>::kStageBytes;
  // + 1024: the base is aligned to 1024 bytes (128-byte swizzle atoms)
  static constexpr int kBytes = 1024 + kRedOff + PartialRing<BN>::kRedBytes;
};

// CL (IG_MODE_DET only): the S partition blocks of a tile form a cluster;
// block s owns outputs [s TB/S, (s+1) TB/S) of the tile and receives their S
// partials by asynchronous remote stores counted on its mbarrier, then sums
// them from FP32 zero in increasing partition order (the counter protocol's
// order, so the same bits) without the workspace round trip.
template <int BN, int MODE, bool CL>
__global__ void __launch_bounds__(ShrinkGeo<BN>::THREADS)
    shrink_warp_kernel(const __grid_constant__ ShrinkParams p) {
  // the next kernel may be scheduled now: it reads nothing of ours before
  // its own griddep_wait(), which waits for this grid to complete
  griddep_launch();
  using SM = ShrinkSmem<BN>;
  constexpr int kThreads = ShrinkGeo<BN>::THREADS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* bar_recv = bars + kShrinkStages;                 // cluster combine
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 64);    // tile entry (kTileInts)
  int32_t* info = reinterpret_cast<int32_t*>(smem + 192);
  float* recv = reinterpret_cast<float*>(smem + 256);        // [S][TB/S] (TB floats)
  constexpr int TB = ShrinkGeo<BN>::TB;
  uint8_t* stages = smem + SM::kStagesOff;
  float* red = reinterpret_cast<float*>(smem + SM::kRedOff);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int S = p.S;

  uint32_t bid = blockIdx.x;
  const int s = (int)next_digit(bid, (uint32_t)S);
  const int jb = (int)next_digit(bid, (uint32_t)p.jblocks);
  const int sl = (int)next_digit(bid, (uint32_t)p.slices);
  const int64_t t = bid;

  // Tile entry: [g, nrows, consecutive, 0, rows[8]]; complete before this kernel began.
  if (tid < kTileInts) ent_s[tid] = p.tiles[t * kTileInts + tid];
  if (tid == 0) {
    for (int i = 0; i < kShrinkStages; ++i) mbar_init(&bars[i], 1);
    if (CL) mbar_init(bar_recv, 1);
    fence_mbar_init();
    if (CL) mbar_arrive_expect_tx(bar_recv, (uint32_t)(TB * 4));
  }
  __syncthreads();
  const int g = ent_s[0];
  const int nrows = ent_s[1];
  const int32_t* rows_s = ent_s + 4;
  const int64_t r = p.r;
  const int64_t M = p.M;
  if (nrows <= 0) return;

  if (g == p.L) {
    // tokens without an adapter: their Z rows are zero (ATOMIC zeroed Z already)
    griddep_wait();
    if (MODE != IG_MODE_ATOMIC && s == 0) {
      for (int i = tid; i < nrows * BN; i += kThreads) {
        const int row = i / BN, j = i % BN;
        p.z[((int64_t)sl * M + rows_s[row]) * r + jb * BN + j] = 0.0f;
      }
    }
    return;
  }

  // every block of the cluster has initialised and armed its mbarrier once
  // the matching cluster_wait returns
  if (CL) cluster_arrive_relaxed();
  const int64_t k0 = (int64_t)s * p.Ks;
  const bool early_a = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;
  PartialArgs pa;
  pa.rows = rows_s;
  pa.status = p.status;
  pa.Ks = (int)p.Ks;
  pa.nrows = nrows;
  pa.x = p.x;
  pa.K = p.K;
  pa.tm_a = &p.tm_a;
  pa.tm_a3 = p.has_a3 ? &p.tm_a3 : nullptr;
  pa.k0 = (int)k0;
  pa.a_row = (int)(((int64_t)g * p.slices + sl) * r + (int64_t)jb * BN);
  pa.first_budget = first_copy_budget(p.flags);
  PartialRing<BN> ring;
  ring.stages = stages;
  ring.bars = bars;
  ring.nst = kShrinkStages;
  ring.nkb = (int)((p.Ks + kShrinkKB - 1) / kShrinkKB);

  const int first = min(ring.nkb, kShrinkStages);
  if (warp == 0) {
    for (int b = 0; b < first; ++b) {
      ring.expect(pa, b);
      if (early_a) ring.issue_a(pa, b);
    }
  } else if (warp == 1 && (threadIdx.x & 31) < nrows) {
    // L2 prefetch of the x rows (no effect on the values read after the wait)
    bulk_prefetch_l2(p.x + (int64_t)rows_s[threadIdx.x & 31] * p.K + k0, (uint32_t)(p.Ks * 2));
  }
  // static weights and a short partition: A chunks into registers before
  // the wait (shrink_core.cuh)
  const __nv_bfloat16* xrow = ring.x_row(pa);
  const bool fast = ring.fast(early_a);
  typename PartialRing<BN>::ARegs ar[PartialRing<BN>::kFastKB];
  const bool a_ok = fast ? ring.fast_prologue(pa, ar) : true;
  griddep_wait();
  if (warp == 0 && !early_a)
    for (int b = 0; b < first; ++b) ring.issue_a(pa, b);
  float v;
  const bool ok = fast ? ring.fast_run(pa, xrow, ar, a_ok, red, v, []() {})
                       : ring.run(pa, xrow, red, v, []() {});
  if (CL) {
    // Send output tid's partial to its owner; every block sends on every
    // path (zeros after a failed copy), so every owner receives TB * 4 bytes.
    const int per = TB / S;
    cluster_wait();
    const int owner = tid / per;
    st_async_f32(map_rank(recv + s * per + tid % per, (uint32_t)owner), ok ? v : 0.0f,
                 map_rank(bar_recv, (uint32_t)owner));
    // The wait outlasts any sender's bounded waits, so the block never leaves
    // while a partial is still on its way to it.
    const bool got = mbar_wait_bounded(bar_recv, 0, p.status, 1ll << 36);
    if (got && tid < per) {
      const int o = s * per + tid;
      const int row = o / BN, j = o % BN;
      if (row < nrows) {
        float total = 0.0f;
        for (int q = 0; q < S; ++q) total += recv[q * per + tid];
        p.z[((int64_t)sl * M + rows_s[row]) * r + jb * BN + j] = total * p.scale;
      }
    }
    return;
  }
  if (!ok) return;
  const int rrow = tid / BN;                 // this thread's output
  const int j0 = tid % BN;

  if (MODE == IG_MODE_UNSPLIT || MODE == IG_MODE_ATOMIC) {
    if (rrow < nrows) {
      float* zp = p.z + ((int64_t)sl * M + rows_s[rrow]) * r + jb * BN + j0;
      if (MODE == IG_MODE_UNSPLIT) *zp = v * p.scale;
      else atomicAdd(zp, v * p.scale);
    }
    return;
  }

  // DET: publish the partial, then the completion-counter protocol.
  // DET_TREE: publish the partial only; a second kernel combines.
  const int64_t slot = (t * p.slices + sl) * p.jblocks + jb;
  float* part = p.partials + (slot * S) * (kTileRows * BN);
  part[(int64_t)s * (kTileRows * BN) + rrow * BN + j0] = v;
  if (MODE == IG_MODE_DET_TREE) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atom_add_acq_rel_gpu(p.counters + slot, 1u);
    info[0] = (int)prev;
    if (prev >= (uint32_t)S) atomicOr(p.status, kStatusCorrupt);
  }
  __syncthreads();
  const uint32_t prev = (uint32_t)info[0];
  if (prev != (uint32_t)(S - 1)) return;
  __threadfence();
  for (int o = tid; o < kTileRows * BN; o += kThreads) {
    const int row = o / BN, j = o % BN;
    if (row >= nrows) continue;
    float total = 0.0f;
    for (int q = 0; q < S; ++q) total += __ldcg(part + (int64_t)q * (kTileRows * BN) + o);
    p.z[((int64_t)sl * M + rows_s[row]) * r + jb * BN + j] = total * p.scale;
  }
  if (tid == 0) p.counters[slot] = 0u;
}

template <int BN, int MODE>
cudaError_t launch_one(const ShrinkParams& p, int64_t tiles_max, cudaStream_t st) {
  using SM = ShrinkSmem<BN>;
  auto kern = shrink_warp_kernel<BN, MODE, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SM::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = tiles_max * p.slices * p.jblocks * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(ShrinkGeo<BN>::THREADS), SM::kBytes, st, p);
}

// Deterministic combine inside a cluster of the S partition blocks (same
// bits as the counter protocol). Returns cudaErrorNotSupported when such a
// cluster cannot be resident, for the caller to use the counter protocol.
template <int BN>
cudaError_t launch_cluster(const ShrinkParams& p, int64_t tiles_max, cudaStream_t st) {
  using SM = ShrinkSmem<BN>;
  auto kern = shrink_warp_kernel<BN, IG_MODE_DET, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SM::kBytes);
  if (e != cudaSuccess) return e;
  if (p.S > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const int64_t grid = tiles_max * p.slices * p.jblocks * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(ShrinkGeo<BN>::THREADS);
  cfg.dynamicSmemBytes = SM::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    // can one such cluster be resident? (cached per S)
    static std::mutex mu;
    static std::map<int, bool> fits;
    std::lock_guard<std::mutex> lock(mu);
    auto it = fits.find(p.S);
    if (it == fits.end()) {
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3((unsigned)p.S);
      int n = 0;
      const bool ok = cudaOccupancyMaxActiveClusters(&n, kern, &q) == cudaSuccess && n >= 1;
      cudaGetLastError();
      it = fits.emplace(p.S, ok).first;
    }
    if (!it->second) return cudaErrorNotSupported;
  }
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BN>
cudaError_t launch_det(const ShrinkParams& p, int64_t tiles_max, cudaStream_t st) {
  constexpr int TB = ShrinkGeo<BN>::TB;
  if (!(p.flags & IG_FLAG_UNFUSED) && p.S <= 16 && TB % p.S == 0) {
    const cudaError_t e = launch_cluster<BN>(p, tiles_max, st);
    if (e != cudaErrorNotSupported) return e;
  }
  return launch_one<BN, IG_MODE_DET>(p, tiles_max, st);
}

}  // namespace

cudaError_t launch_shrink_warp(const ShrinkParams& p, int mode, int bn, int64_t tiles_max,
                              cudaStream_t st) {
  if (bn == 16) {
    if (mode == IG_MODE_DET_TREE) return launch_one<16, IG_MODE_DET_TREE>(p, tiles_max, st);
    if (mode == IG_MODE_DET) return launch_det<16>(p, tiles_max, st);
    if (mode == IG_MODE_ATOMIC) return launch_one<16, IG_MODE_ATOMIC>(p, tiles_max, st);
    return launch_one<16, IG_MODE_UNSPLIT>(p, tiles_max, st);
  }
  if (mode == IG_MODE_DET_TREE) return launch_one<8, IG_MODE_DET_TREE>(p, tiles_max, st);
  if (mode == IG_MODE_DET) return launch_det<8>(p, tiles_max, st);
  if (mode == IG_MODE_ATOMIC) return launch_one<8, IG_MODE_ATOMIC>(p, tiles_max, st);
  return launch_one<8, IG_MODE_UNSPLIT>(p, tiles_max, st);
}

}  // namespace ig
