// LoRA shrink on CUDA cores (IG_PATH_FMA): Z = scale * X A_i^T with a
// Split-K reduction.
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
// Block = BN/4 warps (warp w: rank columns 4w .. 4w+3 of all rows), tile =
// up to 8 token rows of one adapter (one entry of the token
// map's tile table) x BN rank columns, one K partition. The partition
// is streamed through shared memory in k-blocks of 256 elements by TMA
// copies (one tiled copy for the A block, one row gather per 4 token rows,
// completion counted on an mbarrier), four stages deep.
//
// Latency: the tile entry is read before griddep_wait() (the token map is
// complete before this kernel starts); with IG_FLAG_STATIC_WEIGHTS the A
// rows of the first stages are requested before it too, so only the x rows
// wait for the previous kernel.
//
// Reduction order inside a partition, identical for every row and every M:
//   lane l owns the 8-element chunks l, l+32, l+64, ... of the partition and
//   accumulates their elements in increasing k with FMA into one FP32
//   register per output; the 32 lane sums are then combined by a fixed
//   butterfly (xor 16, 8, 4, 2, 1), done as a reduce-scatter so each lane
//   ends with NV/32 finished outputs. It depends only on K/S.
#include "fma_core.cuh"

namespace ig {

namespace {

template <int BN>
struct ShrinkSmem {
  static constexpr int kStagesOff = 256;                           // mbarriers + info
  static constexpr int kBytes = kStagesOff + kShrinkStages * FmaRing<BN>::kStageBytes;
};

template <int BN, int MODE>
__global__ void __launch_bounds__(FmaGeo<BN>::THREADS)
    shrink_fma_kernel(const __grid_constant__ ShrinkParams p) {
  using SM = ShrinkSmem<BN>;
  constexpr int kThreads = FmaGeo<BN>::THREADS;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 64);    // tile entry (kTileInts)
  int32_t* info = reinterpret_cast<int32_t*>(smem + 192);
  uint8_t* stages = smem + SM::kStagesOff;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    fence_mbar_init();
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
    griddep_launch();
    if (MODE != IG_MODE_ATOMIC && s == 0) {
      for (int i = tid; i < nrows * BN; i += kThreads) {
        const int row = i / BN, j = i % BN;
        p.z[((int64_t)sl * M + rows_s[row]) * r + jb * BN + j] = 0.0f;
      }
    }
    return;
  }

  const int64_t K = p.K;
  const int64_t k0 = (int64_t)s * p.Ks;
  const bool early_a = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;
  FmaArgs pa;
  pa.x = p.x + k0;
  pa.A = p.A + (((int64_t)g * p.slices + sl) * r + (int64_t)jb * BN) * K + k0;
  pa.rows = rows_s;
  pa.status = p.status;
  pa.K = K;
  pa.Ks = p.Ks;
  pa.nrows = nrows;
  pa.tm_x = &p.tm_x;
  pa.tm_a = &p.tm_a;
  pa.k0 = (int)k0;
  pa.a_row = (int)(((int64_t)g * p.slices + sl) * r + (int64_t)jb * BN);
  FmaRing<BN> ring;
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
  }
  griddep_wait();
  griddep_launch();
  if (warp == 0) {
    for (int b = 0; b < first; ++b) {
      if (!early_a) ring.issue_a(pa, b);
      ring.issue_x(pa, b);
    }
  }

  float v;
  if (!ring.run(pa, v)) return;
  const int rrow = lane / 4;                 // this lane's output
  const int j0 = warp * FmaGeo<BN>::JPW + lane % 4;

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
  auto kern = shrink_fma_kernel<BN, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SM::kBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = tiles_max * p.slices * p.jblocks * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(FmaGeo<BN>::THREADS), SM::kBytes, st, p);
}

}  // namespace

cudaError_t launch_shrink_fma(const ShrinkParams& p, int mode, int bn, int64_t tiles_max,
                              cudaStream_t st) {
  if (bn == 16) {
    if (mode == IG_MODE_DET_TREE) return launch_one<16, IG_MODE_DET_TREE>(p, tiles_max, st);
    if (mode == IG_MODE_DET) return launch_one<16, IG_MODE_DET>(p, tiles_max, st);
    if (mode == IG_MODE_ATOMIC) return launch_one<16, IG_MODE_ATOMIC>(p, tiles_max, st);
    return launch_one<16, IG_MODE_UNSPLIT>(p, tiles_max, st);
  }
  if (mode == IG_MODE_DET_TREE) return launch_one<8, IG_MODE_DET_TREE>(p, tiles_max, st);
  if (mode == IG_MODE_DET) return launch_one<8, IG_MODE_DET>(p, tiles_max, st);
  if (mode == IG_MODE_ATOMIC) return launch_one<8, IG_MODE_ATOMIC>(p, tiles_max, st);
  return launch_one<8, IG_MODE_UNSPLIT>(p, tiles_max, st);
}

}  // namespace ig
