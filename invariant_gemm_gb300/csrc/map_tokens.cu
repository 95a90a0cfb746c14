// Token grouping: a stable counting sort of the per-token adapter index.
//
// The pages pass "mapping information" along with the shrink inputs
// ("Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// sec. 5.2); the kernels need each output tile to use one adapter's A_i and
// B_i, so tokens are grouped by adapter first. Group g < L holds the tokens
// of adapter g, group L the tokens without an adapter (index -1) and, flagged
// in the status word, any out-of-range index.
//
// Integer work only, and deterministic: the order inside a group is the
// original token order, whatever the thread schedule.
//
// One CTA of 1024 threads. The M rows are cut into 32 contiguous segments,
// one per warp. Pass 1 counts each warp's rows per group into hist[warp][g]
// (warp-synchronous, via __match_any_sync); the CTA then turns the counts
// into global start positions (exclusive scan over warps, then over groups);
// pass 2 re-walks the segments and writes each row to
// start[warp][g] + (rank among equal groups within the 32-row step).
//
// Finally it writes the tile table the shrink and expand kernels read: group
// g is cut into ceil(count_g / T) tiles of at most T consecutive rows of the
// grouped order (T = 8 for the warp-path and FMA-path kernels, 128 for the tcgen05
// kernels); tile entries hold [g, nrows, contiguous, 0, rows[T]] so that a block
// learns its adapter and its token rows with one contiguous load.
// `contiguous` is 1 when the rows are consecutive token indices (then a
// tile can be copied as one box instead of row by row). Tiles of
// adapters 0..L-1 come first (in adapter order), then the no-adapter group,
// then empty entries (nrows = 0) up to tiles_max.
//
// This kernel is launched without programmatic dependent launch and never
// releases its dependents early, so every later kernel on the stream starts
// after the map is complete and may read it before its own griddep_wait().
#include "ig_common.cuh"

namespace ig {

namespace {

constexpr int kMapThreads = 1024;
constexpr int kMapWarps = kMapThreads / 32;

__device__ __forceinline__ int group_of(const int32_t* idx, int64_t m, int L, uint32_t* status) {
  int a = idx[m];
  if (a >= 0 && a < L) return a;
  if (a != -1) atomicOr(status, kStatusAdapterRange);
  return L;
}

__global__ void __launch_bounds__(kMapThreads) map_tokens_kernel(MapParams p) {
  extern __shared__ int32_t hist[];  // [kMapWarps][G], total[G], cntg[G], tstart[G+1]
  const int G = p.L + 1;
  int32_t* total = hist + kMapWarps * G;
  int32_t* cntg = total + G;
  int32_t* tstart = cntg + G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t M = p.M;
  const int64_t seg = (M + kMapWarps - 1) / kMapWarps;
  const int64_t lo = min(M, (int64_t)warp * seg);
  const int64_t hi = min(M, lo + seg);
  const unsigned lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < kMapWarps * G; i += kMapThreads) hist[i] = 0;
  __syncthreads();

  // pass 1: per-warp group counts
  int32_t* h = hist + warp * G;
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t m = base + lane;
    const bool valid = m < hi;
    const int g = valid ? group_of(p.idx, m, p.L, p.status) : -1;
    const unsigned act = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const unsigned peers = __match_any_sync(act, g);
      if ((peers & lt_mask) == 0) h[g] += __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();

  // per group: exclusive scan over warps, and the group total
  for (int g = tid; g < G; g += kMapThreads) {
    int32_t run = 0;
    for (int w = 0; w < kMapWarps; ++w) {
      const int32_t c = hist[w * G + g];
      hist[w * G + g] = run;
      run += c;
    }
    total[g] = run;
  }
  __syncthreads();

  // exclusive scan over groups (warp 0, 32 groups per step)
  if (warp == 0) {
    int32_t carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      const int32_t c = g < G ? total[g] : 0;
      int32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < G) {
        cntg[g] = c;
        total[g] = carry + incl - c;  // now the group's start
        p.offsets[g] = carry + incl - c;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) p.offsets[G] = carry;
  }
  __syncthreads();

  // tile starts per group: exclusive scan of ceil(count_g / kTileRows)
  __syncthreads();
  if (warp == 0) {
    int32_t carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      const int32_t c = g < G ? (cntg[g] + p.tile_rows - 1) / p.tile_rows : 0;
      int32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < G) tstart[g] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tstart[G] = carry;
  }
  for (int i = tid; i < kMapWarps * G; i += kMapThreads) hist[i] += total[i % G];
  __syncthreads();

  // pass 2: stable placement
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t m = base + lane;
    const bool valid = m < hi;
    int g = -1;
    if (valid) {
      const int a = p.idx[m];
      g = (a >= 0 && a < p.L) ? a : p.L;
    }
    const unsigned act = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const unsigned peers = __match_any_sync(act, g);
      const int rank = __popc(peers & lt_mask);
      p.perm[h[g] + rank] = (int32_t)m;
      __syncwarp(act);
      if ((peers & lt_mask) == 0) h[g] += __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();

  // tile table: one warp per tile
  const int T = p.tile_rows;
  const int ents = 4 + T;
  const int64_t ntiles = tstart[G];
  for (int64_t t = warp; t < p.tiles_max; t += kMapWarps) {
    int32_t* ent = p.tiles + t * ents;
    if (t >= ntiles) {
      for (int i = lane; i < ents; i += 32) ent[i] = i == 0 ? -1 : 0;
      continue;
    }
    int lo_g = 0, hi_g = G - 1;  // last group with tstart[g] <= t
    while (lo_g < hi_g) {
      const int mid = (lo_g + hi_g + 1) >> 1;
      if (tstart[mid] <= t) lo_g = mid; else hi_g = mid - 1;
    }
    const int g = lo_g;
    const int q = (int)(t - tstart[g]);
    const int first = total[g] + q * T;                   // total[] holds group starts
    const int cnt = min(T, total[g] + cntg[g] - first);
    const int r0 = p.perm[first];
    bool consec = true;
    for (int i = lane; i < T; i += 32) {
      const int v = i < cnt ? p.perm[first + i] : 0;
      ent[4 + i] = v;
      if (i < cnt && v != r0 + i) consec = false;
    }
    consec = __all_sync(0xffffffffu, consec);
    if (lane == 0) ent[0] = g;
    if (lane == 1) ent[1] = cnt;
    if (lane == 2) ent[2] = consec ? 1 : 0;
    if (lane == 3) ent[3] = 0;
  }
}

}  // namespace

cudaError_t launch_map_tokens(const MapParams& p, cudaStream_t st) {
  const int G = p.L + 1;
  const size_t smem = ((size_t)(kMapWarps + 3) * G + 1) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(map_tokens_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  map_tokens_kernel<<<1, kMapThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ig
