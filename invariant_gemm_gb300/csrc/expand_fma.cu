// LoRA expand on CUDA cores (IG_PATH_FMA): y += bf16(Z) B_i^T, in place, one
// rounding.
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
// Block = 4 warps, tile = up to 8 token rows of one adapter (one entry of
// the token map's tile table) x 256 output columns of one slice. Lane l owns
// columns n0 + 8l .. n0 + 8l + 7 (one 16-byte vector of y per row, so a warp
// reads and writes 512 contiguous bytes of a row); warp w owns rows 2w and
// 2w+1. B is read straight into registers, 16 rank elements at a time.
//
// Latency: the tile entry is read before griddep_wait(); with
// IG_FLAG_STATIC_WEIGHTS the block's B slice is also requested into L2 before
// it. After the wait each lane issues its y, z and B loads together, then
// computes and stores.
#include "ig_common.cuh"

namespace ig {

namespace {

constexpr int kThreads = kExpandWarps * 32;
constexpr int kMaxRank = 256;
constexpr int RW = 2;                 // token rows per warp (4 warps x 2 = kTileRows)
constexpr int kExpandJC = 16;         // rank elements per register chunk
static_assert(kExpandWarps * RW == kTileRows, "tile rows");

// JC = rank elements per register chunk: 16, or 8 when r is an odd multiple
// of 8. The chunking does not change the order of the j sum.
template <int JC>
__global__ void __launch_bounds__(kThreads, 2) expand_fma_kernel(ExpandParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint8_t* sB = smem + 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint32_t bid = blockIdx.x;
  const int nt = (int)next_digit(bid, (uint32_t)p.ntiles);
  const int sl = (int)next_digit(bid, (uint32_t)p.slices);
  const int64_t t = bid;

  // Tile entry [g, nrows, consecutive, 0, rows[8]]; complete before this kernel began.
  const int32_t* ent = p.tiles + t * kTileInts;
  const int g = ent[0];
  const int nrows = ent[1];
  if (g < 0 || g >= p.L || nrows <= 0) return;
  const int row0 = warp * RW;
  int m[RW];
#pragma unroll
  for (int i = 0; i < RW; ++i) m[i] = (row0 + i < nrows) ? ent[4 + row0 + i] : -1;

  const int64_t N = p.N;
  const int64_t n0 = (int64_t)nt * kExpandBN;
  const int groups = (int)min((int64_t)(kExpandBN / 8), (N - n0) / 8);  // 8-column groups
  const int r = (int)p.r;
  const int lbs = 16 * r + 16;  // smem stride of one 8-column group
  const bool early_b = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue_b = [&]() {
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(groups * 16 * r));
    __syncwarp();
    const __nv_bfloat16* src = p.B + (((int64_t)g * p.slices + sl) * N + n0) * r;
    if (lane < groups) bulk_g2s(sB + lane * lbs, src + (int64_t)lane * 8 * r, 16 * r, bar);
  };
  if (early_b && warp == 0) issue_b();

  griddep_wait();
  griddep_launch();
  if (!early_b && warp == 0) issue_b();
  const bool active = lane < groups && row0 < nrows;
  const int64_t n = n0 + lane * 8;

  const int64_t M = p.M;
  const int64_t ld = (int64_t)p.slices * N;
  uint4 yv[RW];
#pragma unroll
  for (int i = 0; i < RW; ++i)
    if (active && m[i] >= 0)
      yv[i] = *reinterpret_cast<const uint4*>(p.y + (int64_t)m[i] * ld + (int64_t)sl * N + n);
  // The tile's Z rows for one rank chunk, rounded to bf16 (as FP32 values;
  // with IG_FLAG_Z_FP32 left as stored). Every lane loads the same
  // addresses: one transaction per warp; L2 only, Z was written by the
  // previous kernel.
  const bool zf32 = (p.flags & IG_FLAG_Z_FP32) != 0;
  float zf[RW][JC];
  auto load_z = [&](int jc) {
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      if (!active || m[i] < 0) continue;
      const float4* zsrc =
          reinterpret_cast<const float4*>(p.z + ((int64_t)sl * M + m[i]) * r + jc);
#pragma unroll
      for (int q = 0; q < JC / 4; ++q) {
        const float4 f = __ldcg(zsrc + q);
        zf[i][4 * q + 0] = zf32 ? f.x : bf16_round_f32(f.x);
        zf[i][4 * q + 1] = zf32 ? f.y : bf16_round_f32(f.y);
        zf[i][4 * q + 2] = zf32 ? f.z : bf16_round_f32(f.z);
        zf[i][4 * q + 3] = zf32 ? f.w : bf16_round_f32(f.w);
      }
    }
  };
  load_z(0);
  // every thread waits for the B slice, so the block never exits with copies
  // in flight; after an expired wait, once more (bounded) before it leaves
  if (!mbar_wait_bounded(bar, 0, p.status)) {
    mbar_wait_bounded(bar, 0, p.status);
    return;
  }
  if (!active) return;

  float acc[RW][8];
#pragma unroll
  for (int i = 0; i < RW; ++i)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[i][c] = 0.0f;

  for (int jc = 0; jc < r; jc += JC) {
    if (jc > 0) load_z(jc);
#pragma unroll
    for (int q = 0; q < JC / 8; ++q) {
      uint4 bq[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        bq[c] = *reinterpret_cast<const uint4*>(sB + lane * lbs + (c * r + jc + 8 * q) * 2);
      float zq[RW][8];
#pragma unroll
      for (int i = 0; i < RW; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) zq[i][e] = zf[i][8 * q + e];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float bf[8];
        unpack8(bq[c], bf);
#pragma unroll
        for (int i = 0; i < RW; ++i) {
          if (m[i] < 0) continue;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][c] = fmaf(zq[i][e], bf[e], acc[i][c]);
        }
      }
    }
  }

#pragma unroll
  for (int i = 0; i < RW; ++i) {
    if (m[i] < 0) continue;
    float yf[8];
    unpack8(yv[i], yf);
    uint4 w;
    w.x = f32x2_to_bf16x2_bits(yf[0] + acc[i][0], yf[1] + acc[i][1]);
    w.y = f32x2_to_bf16x2_bits(yf[2] + acc[i][2], yf[3] + acc[i][3]);
    w.z = f32x2_to_bf16x2_bits(yf[4] + acc[i][4], yf[5] + acc[i][5]);
    w.w = f32x2_to_bf16x2_bits(yf[6] + acc[i][6], yf[7] + acc[i][7]);
    *reinterpret_cast<uint4*>(p.y + (int64_t)m[i] * ld + (int64_t)sl * N + n) = w;
  }
}

}  // namespace

cudaError_t launch_expand_fma(const ExpandParams& p, int64_t tiles_max, cudaStream_t st) {
  if (p.r > kMaxRank || p.r % 8 != 0) return cudaErrorInvalidValue;
  const int64_t grid = tiles_max * p.slices * p.ntiles;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = 128 + (size_t)(kExpandBN / 8) * (16 * p.r + 16);
  if (p.r % kExpandJC == 0) {
    auto kern = expand_fma_kernel<kExpandJC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, p);
  }
  auto kern = expand_fma_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, p);
}

}  // namespace ig
