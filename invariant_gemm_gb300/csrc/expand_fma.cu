// LoRA expand on CUDA cores: y += bf16(Z) B_i^T, in place, one rounding.
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// Eq. 1 (the expand multiplies the r-wide shrink output by B in
// R^{Hout x r}) and sec. 6.2 / Fig. 5 (the FP32 shrink output reaches the
// next operation as BF16, rounded to nearest).
//
// For each output element:
//   acc = 0; for j = 0..r-1: acc = fma(bf16_rn(z[j]), B[n][j], acc)
//   y   = bf16_rn(f32(y) + acc)
// The j order is fixed and every element is computed by one thread, so the
// result does not depend on the tiling, on M or on the other rows.
//
// Block = 8 warps, tile = 32 token rows of one adapter x 256 output columns of
// one slice. Lane l owns columns n0 + 8l .. n0 + 8l + 7 (one 16-byte vector of
// y per row, so a warp reads and writes 512 contiguous bytes of a row); warp w
// owns rows 4w .. 4w+3. The bf16-rounded Z rows of the tile sit in shared
// memory; B is read straight into registers in chunks of 8 rank elements.
#include "ig_common.cuh"

namespace ig {

namespace {

constexpr int kThreads = kExpandWarps * 32;
constexpr int kMaxRank = 256;

__global__ void __launch_bounds__(kThreads) expand_fma_kernel(ExpandParams p) {
  extern __shared__ __align__(16) float zs[];  // [kExpandBM][r]
  __shared__ int32_t info[4];
  __shared__ int32_t rows_s[kExpandBM];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int64_t bid = blockIdx.x;
  const int nt = (int)(bid % p.ntiles);
  bid /= p.ntiles;
  const int sl = (int)(bid % p.slices);
  const int64_t t = bid / p.slices;

  if (warp == 0) {
    int g = 0, row0 = 0, nrows = 0;
    const bool ok = find_tile(p.offsets, p.L, kExpandBM, t, &g, &row0, &nrows);
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
  const int r = (int)p.r;
  const int64_t M = p.M;
  if (tid < kExpandBM) rows_s[tid] = tid < nrows ? p.perm[p.offsets[g] + info[2] + tid] : 0;
  __syncthreads();

  for (int i = tid; i < nrows * r; i += kThreads) {
    const int row = i / r, j = i % r;
    zs[i] = bf16_round_f32(p.z[((int64_t)sl * M + rows_s[row]) * r + j]);
  }
  __syncthreads();

  const int64_t N = p.N;
  const int64_t n = (int64_t)nt * kExpandBN + lane * 8;
  if (n >= N) return;
  const __nv_bfloat16* Bp = p.B + (((int64_t)g * p.slices + sl) * N + n) * r;

  float acc[kExpandRowsPerWarp][8];
#pragma unroll
  for (int rr = 0; rr < kExpandRowsPerWarp; ++rr)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[rr][i] = 0.0f;

  const int row_base = warp * kExpandRowsPerWarp;
  for (int jc = 0; jc < r; jc += kExpandJC) {
    float b[8][kExpandJC];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(Bp + (int64_t)i * r + jc));
      unpack8(u, b[i]);
    }
#pragma unroll
    for (int rr = 0; rr < kExpandRowsPerWarp; ++rr) {
      const int row = row_base + rr;
      if (row >= nrows) break;
      const float* zr = zs + row * r + jc;
#pragma unroll
      for (int j = 0; j < kExpandJC; ++j) {
        const float zb = zr[j];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[rr][i] = fmaf(zb, b[i][j], acc[rr][i]);
      }
    }
  }

  const int64_t ld = (int64_t)p.slices * N;
#pragma unroll
  for (int rr = 0; rr < kExpandRowsPerWarp; ++rr) {
    const int row = row_base + rr;
    if (row >= nrows) break;
    __nv_bfloat16* yp = p.y + (int64_t)rows_s[row] * ld + (int64_t)sl * N + n;
    const uint4 u = *reinterpret_cast<const uint4*>(yp);
    float yv[8];
    unpack8(u, yv);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = f32_to_bf16_bits(yv[i] + acc[rr][i]);
    uint4 w;
    w.x = o[0] | (o[1] << 16);
    w.y = o[2] | (o[3] << 16);
    w.z = o[4] | (o[5] << 16);
    w.w = o[6] | (o[7] << 16);
    *reinterpret_cast<uint4*>(yp) = w;
  }
}

}  // namespace

cudaError_t launch_expand_fma(const ExpandParams& p, int64_t tiles_max, cudaStream_t st) {
  if (p.r > kMaxRank) return cudaErrorInvalidValue;
  const int64_t grid = tiles_max * p.slices * p.ntiles;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)kExpandBM * p.r * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(expand_fma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  expand_fma_kernel<<<(unsigned)grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ig
