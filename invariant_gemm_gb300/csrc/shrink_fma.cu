// LoRA shrink on CUDA cores: Z = scale * X A_i^T with a Split-K reduction.
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
//   sec. 4.2        UNSPLIT: S = 1, one block over the whole of K.
//
// Block = 8 warps, tile = 32 token rows (one adapter) x BN rank columns,
// one K partition. The partition is streamed through shared memory in
// k-blocks of 256 elements by 1-D bulk async copies (one per token row and
// one per A row, completion counted on an mbarrier), four stages deep.
//
// Reduction order inside a partition, identical for every row and every M:
//   lane l owns the 8-element chunks l, l+32, l+64, ... of the partition and
//   accumulates their elements in increasing k with FMA into one FP32
//   register per output; the 32 lane sums are then combined by a fixed
//   butterfly (xor 16, 8, 4, 2, 1), done as a reduce-scatter so each lane
//   ends with NV/32 finished outputs. It depends only on K/S.
#include "ig_common.cuh"

namespace ig {

namespace {

constexpr int kThreads = kShrinkWarps * 32;

template <int BN>
struct ShrinkSmem {
  static constexpr int kRowBytes = kShrinkKB * 2;                  // 512
  static constexpr int kStageBytes = (kShrinkBM + BN) * kRowBytes;
  static constexpr int kHeader = 256;                              // mbarriers + info
  static constexpr int kRowsOff = kHeader;                         // int32[BM]
  static constexpr int kStagesOff = kHeader + 256;
  static constexpr int kBytes = kStagesOff + kShrinkStages * kStageBytes;
};

template <int BN, int MODE>
__global__ void __launch_bounds__(kThreads) shrink_fma_kernel(ShrinkParams p) {
  using SM = ShrinkSmem<BN>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  int32_t* info = reinterpret_cast<int32_t*>(smem + 128);
  int32_t* rows_s = reinterpret_cast<int32_t*>(smem + SM::kRowsOff);
  uint8_t* stages = smem + SM::kStagesOff;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;

  int64_t bid = blockIdx.x;
  const int s = (int)(bid % S);
  bid /= S;
  const int jb = (int)(bid % p.jblocks);
  bid /= p.jblocks;
  const int sl = (int)(bid % p.slices);
  const int64_t t = bid / p.slices;

  if (warp == 0) {
    int g = 0, row0 = 0, nrows = 0;
    const bool ok = find_tile(p.offsets, p.L + 1, kShrinkBM, t, &g, &row0, &nrows);
    if (lane == 0) {
      info[0] = ok ? 1 : 0;
      info[1] = g;
      info[2] = row0;
      info[3] = nrows;
    }
  }
  __syncthreads();
  if (info[0] == 0) return;
  const int g = info[1];
  const int nrows = info[3];
  const int32_t* perm_t = p.perm + p.offsets[g] + info[2];
  const int64_t r = p.r;
  const int64_t M = p.M;

  if (g == p.L) {
    // tokens without an adapter: their Z rows are zero (ATOMIC zeroed Z already)
    if (MODE != IG_MODE_ATOMIC && s == 0) {
      for (int i = tid; i < nrows * BN; i += kThreads) {
        const int row = i / BN, j = i % BN;
        p.z[((int64_t)sl * M + perm_t[row]) * r + jb * BN + j] = 0.0f;
      }
    }
    return;
  }

  if (tid < kShrinkBM) rows_s[tid] = tid < nrows ? perm_t[tid] : 0;
  if (tid == 0) {
    for (int i = 0; i < kShrinkStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int64_t K = p.K;
  const int64_t k0 = (int64_t)s * p.Ks;
  const int nkb = (int)((p.Ks + kShrinkKB - 1) / kShrinkKB);
  const __nv_bfloat16* Ablk =
      p.A + (((int64_t)g * p.slices + sl) * r + (int64_t)jb * BN) * K + k0;
  const __nv_bfloat16* xbase = p.x + k0;

  // Producer: warp 0 issues the copies of k-block b into stage b % stages.
  auto issue = [&](int b) {
    const int st = b % kShrinkStages;
    const int64_t kofs = (int64_t)b * kShrinkKB;
    const int64_t klen = min((int64_t)kShrinkKB, p.Ks - kofs);
    const uint32_t bytes = (uint32_t)(klen * 2);
    uint8_t* sx = stages + st * SM::kStageBytes;
    uint8_t* sa = sx + kShrinkBM * SM::kRowBytes;
    if (lane == 0) mbar_arrive_expect_tx(&bars[st], bytes * (uint32_t)(nrows + BN));
    __syncwarp();
    for (int i = lane; i < nrows + BN; i += 32) {
      if (i < nrows) {
        bulk_g2s(sx + i * SM::kRowBytes, xbase + (int64_t)rows_s[i] * K + kofs, bytes, &bars[st]);
      } else {
        const int j = i - nrows;
        bulk_g2s(sa + j * SM::kRowBytes, Ablk + (int64_t)j * K + kofs, bytes, &bars[st]);
      }
    }
  };

  if (warp == 0) {
    for (int b = 0; b < nkb && b < kShrinkStages; ++b) issue(b);
  }

  float acc[kShrinkRowsPerWarp][BN];
#pragma unroll
  for (int rr = 0; rr < kShrinkRowsPerWarp; ++rr)
#pragma unroll
    for (int j = 0; j < BN; ++j) acc[rr][j] = 0.0f;

  // Blocks [0, issued) have had their copies issued; block b is consumed in
  // iteration b and block b + stages is issued right after it.
  int issued = min(nkb, kShrinkStages);
  int fail_b = -1;
  for (int b = 0; b < nkb; ++b) {
    const int st = b % kShrinkStages;
    const uint32_t parity = (uint32_t)((b / kShrinkStages) & 1);
    const bool ok = mbar_wait_bounded(&bars[st], parity, p.status);
    if (__syncthreads_or(!ok)) { fail_b = b; break; }
    const int64_t klen = min((int64_t)kShrinkKB, p.Ks - (int64_t)b * kShrinkKB);
    if ((int64_t)lane * 8 < klen) {
      const uint8_t* sx = stages + st * SM::kStageBytes;
      const uint8_t* sa = sx + kShrinkBM * SM::kRowBytes;
      float xv[kShrinkRowsPerWarp][8];
#pragma unroll
      for (int rr = 0; rr < kShrinkRowsPerWarp; ++rr) {
        const int row = warp * kShrinkRowsPerWarp + rr;
        if (row < nrows) {
          const uint4 u = *reinterpret_cast<const uint4*>(sx + row * SM::kRowBytes + lane * 16);
          unpack8(u, xv[rr]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) xv[rr][e] = 0.0f;
        }
      }
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        const uint4 u = *reinterpret_cast<const uint4*>(sa + j * SM::kRowBytes + lane * 16);
        float av[8];
        unpack8(u, av);
#pragma unroll
        for (int rr = 0; rr < kShrinkRowsPerWarp; ++rr)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[rr][j] = fmaf(xv[rr][e], av[e], acc[rr][j]);
      }
    }
    __syncthreads();
    if (b + kShrinkStages < nkb) {
      if (warp == 0) issue(b + kShrinkStages);
      issued = b + kShrinkStages + 1;
    }
  }
  if (fail_b >= 0) {
    // A wait expired (recorded in the status word). Before the block exits,
    // wait, again bounded, for every copy it still has in flight.
    if (tid == 0) {
      for (int bb = fail_b; bb < issued; ++bb)
        mbar_wait_bounded(&bars[bb % kShrinkStages],
                          (uint32_t)((bb / kShrinkStages) & 1), p.status);
    }
    __syncthreads();
    return;
  }

  // Reduce-scatter across the warp: NV values per lane -> NV/32 per lane,
  // lane l ending with values [l*NV/32, (l+1)*NV/32).
  constexpr int NV = kShrinkRowsPerWarp * BN;
  static_assert(NV % 32 == 0, "rows x BN must be a multiple of 32");
  float v[NV];
#pragma unroll
  for (int rr = 0; rr < kShrinkRowsPerWarp; ++rr)
#pragma unroll
    for (int j = 0; j < BN; ++j) v[rr * BN + j] = acc[rr][j];
#pragma unroll
  for (int lvl = 0; lvl < 5; ++lvl) {
    const int off = 16 >> lvl;
    const int half = NV >> (lvl + 1);
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = keep + recv;
    }
  }
  constexpr int PER = NV / 32;
  const int vbase = lane * PER;  // index rr*BN + j of v[0]
  const int rrow = warp * kShrinkRowsPerWarp + vbase / BN;
  const int j0 = vbase % BN;  // PER consecutive columns of one row

  if (MODE == IG_MODE_UNSPLIT || MODE == IG_MODE_ATOMIC) {
    if (rrow < nrows) {
      float* zp = p.z + ((int64_t)sl * M + rows_s[rrow]) * r + jb * BN + j0;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        if (MODE == IG_MODE_UNSPLIT) zp[i] = v[i] * p.scale;
        else atomicAdd(zp + i, v[i] * p.scale);
      }
    }
    return;
  }

  // DET: publish the partial, then the completion-counter protocol.
  const int64_t slot = (t * p.slices + sl) * p.jblocks + jb;
  float* part = p.partials + (slot * S) * (kShrinkBM * BN);
  {
    float* dst = part + (int64_t)s * (kShrinkBM * BN) + rrow * BN + j0;
#pragma unroll
    for (int i = 0; i < PER; ++i) dst[i] = v[i];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atom_add_acq_rel_gpu(p.counters + slot, 1u);
    info[4] = (int)prev;
    if (prev >= (uint32_t)S) atomicOr(p.status, kStatusCorrupt);
  }
  __syncthreads();
  const uint32_t prev = (uint32_t)info[4];
  if (prev != (uint32_t)(S - 1)) return;
  __threadfence();
  for (int o = tid; o < kShrinkBM * BN; o += kThreads) {
    const int row = o / BN, j = o % BN;
    if (row >= nrows) continue;
    float total = 0.0f;
    for (int q = 0; q < S; ++q) total += __ldcg(part + (int64_t)q * (kShrinkBM * BN) + o);
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
  kern<<<(unsigned)grid, kThreads, SM::kBytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_shrink_fma(const ShrinkParams& p, int mode, int bn, int64_t tiles_max,
                              cudaStream_t st) {
  if (bn == 16) {
    if (mode == IG_MODE_DET) return launch_one<16, IG_MODE_DET>(p, tiles_max, st);
    if (mode == IG_MODE_ATOMIC) return launch_one<16, IG_MODE_ATOMIC>(p, tiles_max, st);
    return launch_one<16, IG_MODE_UNSPLIT>(p, tiles_max, st);
  }
  if (mode == IG_MODE_DET) return launch_one<8, IG_MODE_DET>(p, tiles_max, st);
  if (mode == IG_MODE_ATOMIC) return launch_one<8, IG_MODE_ATOMIC>(p, tiles_max, st);
  return launch_one<8, IG_MODE_UNSPLIT>(p, tiles_max, st);
}

}  // namespace ig
