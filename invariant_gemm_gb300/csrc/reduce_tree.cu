// Second-launch Split-K combine with a fixed pairwise tree (IG_MODE_DET_TREE).
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// sec. 4.3: before the single-kernel design of Algorithm 1 the authors
// computed the Split-K partials in parallel and combined them in a separate
// kernel with a fixed pairwise reduction tree; deterministic, but the extra
// launch costs time on small decode workloads. This kernel is that combine:
// the shrink kernels store their FP32 partials exactly as in IG_MODE_DET
// (without the counter protocol), then one block per partial slot sums the S
// partials of each output element with the tree
//     level 0: P_0 .. P_{S-1};
//     level i+1: (v_0 + v_1), (v_2 + v_3), ..., and an odd last value carried;
// until one value is left, multiplies by the scale and writes Z. For S = 8:
// ((P0 + P1) + (P2 + P3)) + ((P4 + P5) + (P6 + P7)).
#include "ig_common.cuh"

namespace ig {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxS = 64;

__device__ __forceinline__ float tree_sum(float (&v)[kMaxS], int n) {
  while (n > 1) {
    const int h = n / 2;
    for (int i = 0; i < h; ++i) v[i] = v[2 * i] + v[2 * i + 1];
    if (n & 1) v[h] = v[n - 1];
    n = h + (n & 1);
  }
  return v[0];
}

__global__ void __launch_bounds__(kThreads) reduce_tree_kernel(TreeParams p) {
  // the next kernel may be scheduled now: it reads nothing of ours before
  // its own griddep_wait(), which waits for this grid to complete
  griddep_launch();
  uint32_t bid = blockIdx.x;
  const int jb = (int)next_digit(bid, (uint32_t)p.jblocks);
  const int sl = (int)next_digit(bid, (uint32_t)p.slices);
  const int64_t t = bid;
  const int ents = 4 + p.tile_rows;
  const int32_t* ent = p.tiles + t * ents;
  const int g = ent[0];
  const int nrows = ent[1];
  griddep_wait();
  if (nrows <= 0 || g < 0 || g >= p.L) return;  // no-adapter rows were zeroed by the shrink
  const int64_t slot = (t * p.slices + sl) * p.jblocks + jb;
  const int64_t per = (int64_t)p.tile_rows * p.bn;     // partial values per split
  const float* part = p.partials + slot * p.S * per;
  for (int o = threadIdx.x; o < nrows * p.bn; o += kThreads) {
    float v[kMaxS];
    for (int q = 0; q < p.S; ++q) v[q] = __ldcg(part + (int64_t)q * per + o);
    const float total = tree_sum(v, p.S);
    const int row = o / p.bn, j = o % p.bn;
    p.z[((int64_t)sl * p.M + ent[4 + row]) * p.r + (int64_t)jb * p.bn + j] = total * p.scale;
  }
}

}  // namespace

cudaError_t launch_reduce_tree(const TreeParams& p, int64_t tiles_max, cudaStream_t st) {
  if (p.S > kMaxS) return cudaErrorInvalidValue;
  const int64_t grid = tiles_max * p.slices * p.jblocks;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(reduce_tree_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, p);
}

}  // namespace ig
