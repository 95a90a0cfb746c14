// LoRA expand on the tcgen05 tensor cores: y += bf16(Z) B_i^T, in place, one
// rounding; for ranks where the token x output x rank tile is a real dense
// contraction (prefill).
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// Eq. 1 (the expand multiplies the r-wide shrink output by B in R^{Hout x r})
// and sec. 6.2 / Fig. 5 (the FP32 shrink output reaches the next operation as
// BF16, rounded to nearest).
//
// Block = 4 warps, tile = up to 128 token rows of one adapter (128-row tile
// table) x 128 output columns of one slice (64 KB of shared memory at r = 64,
// so that three blocks share an SM and overlap their copies and epilogues). The A operand of the MMA is the
// tile's Z rows rounded to bf16, written by the threads straight into the
// 128-byte-swizzled K-major layout; the B operand is B_i's 128 rows x r,
// brought by tiled TMA copies (64 rank columns each; columns past r read as
// zero). The y tile (128 rows x 128 columns) is copied by TMA (one box per 64
// columns when the tile's tokens are consecutive, else row gathers) into
// swizzled shared memory while the MMA runs. tcgen05.mma, M = 128, N = 128,
// K = 16 per instruction, r/16 of them,
// FP32 in tensor memory. Each thread then reads its row of the accumulator,
// adds it to y in FP32 and rounds once to bf16 in shared memory; a final pass
// writes y back with whole rows per warp.
//
// Arithmetic, fixed by r: the tensor core's FP32 sum over j, then
// bf16_rn(f32(y) + sum). A row's value depends only on that row.
#include "umma.cuh"

namespace ig {

namespace {

constexpr int kThreads = 128;
constexpr int kBN = kMmaExpandCols;              // output columns per block (128)
constexpr int kYBlocks = kBN / 64;               // 64-column blocks of the y tile
constexpr int kYBlockBytes = kMmaTileRows * 128; // one 64-column block of the y tile

struct Ctl {
  uint64_t bar_b;   // B copies
  uint64_t bar_y;   // y copies
  uint64_t done;    // MMAs
  uint32_t tmem;
  int32_t fail;     // the B copies never arrived
};

// layout (offsets from the 1024-aligned base): ctl 1024, tile entry 1024,
// then zb [r/64][128 rows][128 B], B [r/64][128 rows][128 B], y [2][128][128 B]
constexpr int kBAtomBytes = kBN * 128;
// (with FP32 Z: zb holds the hi atoms, then the lo atoms)
__host__ __device__ inline size_t off_zb() { return 2048; }
__host__ __device__ inline size_t off_b(int r, bool zf32) {
  return off_zb() + (size_t)((r + 63) / 64) * 16384 * (zf32 ? 2 : 1);
}
__host__ __device__ inline size_t off_y(int r, bool zf32) {
  return off_b(r, zf32) + (size_t)((r + 63) / 64) * kBAtomBytes;
}
__host__ __device__ inline size_t mma_expand_smem(int r, bool zf32) {
  return 1024 + off_y(r, zf32) + kYBlocks * kYBlockBytes;
}

__global__ void __launch_bounds__(kThreads)
    expand_mma_kernel(const __grid_constant__ MmaExpandParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 1024);
  const int r = (int)p.r;
  const bool zf32 = (p.flags & IG_FLAG_Z_FP32) != 0;
  uint8_t* s_zb = smem + off_zb();
  uint8_t* s_b = smem + off_b(r, zf32);
  uint8_t* s_y = smem + off_y(r, zf32);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int64_t bid = blockIdx.x;
  const int nt = (int)(bid % p.ntiles);
  bid /= p.ntiles;
  const int sl = (int)(bid % p.slices);
  const int64_t t = bid / p.slices;

  for (int i = tid; i < kMmaTileInts; i += kThreads) ent_s[i] = p.tiles[t * kMmaTileInts + i];
  if (tid == 0) {
    mbar_init(&ctl->bar_b, 1);
    mbar_init(&ctl->bar_y, 1);
    mbar_init(&ctl->done, 1);
    ctl->fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, kBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const int g = ent_s[0];
  const int nrows = ent_s[1];
  const int32_t* rows_s = ent_s + 4;
  auto teardown = [&]() {
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kBN);
  };
  if (g < 0 || g >= p.L || nrows <= 0) {
    teardown();
    return;
  }

  const int64_t N = p.N, M = p.M;
  const int64_t n0 = (int64_t)nt * kBN;
  const int ka = (r + 63) / 64;                       // 64-column atoms of the rank
  const int b_row = (int)(((int64_t)g * p.slices + sl) * N + n0);
  const int y_col = (int)((int64_t)sl * N + n0);
  const int groups4 = (nrows + 3) / 4;
  const bool contiguous = ent_s[2] != 0;   // rows are consecutive tokens: one box
  const bool early_b = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;

  auto issue_b = [&]() {
    for (int a = 0; a < ka; ++a)
      tma_load_2d(s_b + a * kBAtomBytes, &p.tm_b, a * 64, b_row, &ctl->bar_b);
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(&ctl->bar_b, (uint32_t)ka * kBAtomBytes);
    mbar_arrive_expect_tx(&ctl->bar_y, contiguous ? (uint32_t)kYBlocks * kYBlockBytes
                                                  : (uint32_t)groups4 * 4 * 128 * kYBlocks);
    if (early_b) issue_b();
  }
  griddep_wait();
  griddep_launch();
  if (tid == 0 && !early_b) issue_b();
  // y tile: 64-column blocks, each one box (consecutive tokens) or row
  // gathers spread over the lanes of warp 0
  if (warp == 0 && contiguous) {
    if (lane < kYBlocks)
      tma_load_2d(s_y + lane * kYBlockBytes, &p.tm_yt, y_col + lane * 64, rows_s[0], &ctl->bar_y);
  } else if (warp == 0) {
    const int last = nrows - 1;
    for (int q = lane; q < groups4 * kYBlocks; q += 32) {
      const int cb = q / groups4, g4 = q % groups4;
      tma_gather4(s_y + cb * kYBlockBytes + g4 * 512, &p.tm_y, y_col + cb * 64,
                  rows_s[min(4 * g4, last)], rows_s[min(4 * g4 + 1, last)],
                  rows_s[min(4 * g4 + 2, last)], rows_s[min(4 * g4 + 3, last)], &ctl->bar_y);
    }
  }

  // A operand: this thread's Z row (token row `tid` of the tile), rounded to
  // bf16, into the swizzled K-major layout (16-byte chunk c of a 128-byte row
  // m sits at chunk c ^ (m % 8)). With FP32 Z also the remainder
  // lo = bf16_rn(z - hi), in atoms after the hi ones.
  {
    const int m = tid;
    const bool valid = m < nrows;
    const float* zr = p.z + ((int64_t)sl * M + (valid ? rows_s[m] : 0)) * r;
    for (int a = 0; a < ka; ++a) {
      uint8_t* rowp = s_zb + a * 16384 + m * 128;
      uint8_t* lowp = s_zb + (ka + a) * 16384 + m * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) hi[e] = lo[e] = 0;
        if (valid && a * 64 + c * 8 < r) {
          const float4 f0 = __ldcg(reinterpret_cast<const float4*>(zr + a * 64 + c * 8));
          const float4 f1 = __ldcg(reinterpret_cast<const float4*>(zr + a * 64 + c * 8 + 4));
          const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            hi[e] = f32_to_bf16_bits(f[e]);
            if (zf32) lo[e] = f32_to_bf16_bits(f[e] - __uint_as_float(hi[e] << 16));
          }
        }
        const int pc = (c ^ (m & 7)) * 16;
        *reinterpret_cast<uint4*>(rowp + pc) = make_uint4(
            hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16), hi[4] | (hi[5] << 16), hi[6] | (hi[7] << 16));
        if (zf32)
          *reinterpret_cast<uint4*>(lowp + pc) = make_uint4(
              lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16), lo[4] | (lo[5] << 16), lo[6] | (lo[7] << 16));
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (warp == 1 && lane == 0) {
    if (mbar_wait_bounded(&ctl->bar_b, 0, p.status)) {
      tc_fence_after();
      const uint32_t idesc = umma_idesc_bf16_f32(kMmaTileRows, kBN);
      for (int k = 0; k < r / 16; ++k) {
        const int a = k / 4, kk = k % 4;
        const uint64_t bdesc = umma_desc_sw128(smem_u32(s_b + a * kBAtomBytes) + kk * 32);
        umma_bf16(tmem, umma_desc_sw128(smem_u32(s_zb + a * 16384) + kk * 32), bdesc, idesc,
                  k > 0);
        if (zf32)
          umma_bf16(tmem, umma_desc_sw128(smem_u32(s_zb + (ka + a) * 16384) + kk * 32), bdesc,
                    idesc, true);
      }
    } else {
      ctl->fail = 1;
    }
    umma_commit(&ctl->done);
  }
  __syncwarp();
  const bool y_ok = mbar_wait_bounded(&ctl->bar_y, 0, p.status);
  const bool acc_ok = mbar_wait_bounded(&ctl->done, 0, p.status) &&
                      *reinterpret_cast<volatile int32_t*>(&ctl->fail) == 0;
  tc_fence_after();

  // epilogue 1: this thread's row: y = bf16_rn(f32(y) + acc), in shared memory
  {
    const int m = tid;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c = 0; c < kBN; c += 32) {
      float v[32];
      tmem_ld32(trow + c, v);
      if (!(acc_ok && y_ok) || m >= nrows) continue;
      const int cb = c / 64;
      uint8_t* rowp = s_y + cb * kYBlockBytes + m * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int chunk = ((c % 64) / 8) + q;            // logical 16-byte chunk in the row
        uint4* cp = reinterpret_cast<uint4*>(rowp + ((chunk ^ (m & 7)) * 16));
        uint4 u = *cp;
        float yf[8];
        unpack8(u, yf);
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = f32_to_bf16_bits(yf[e] + v[8 * q + e]);
        u.x = o[0] | (o[1] << 16);
        u.y = o[2] | (o[3] << 16);
        u.z = o[4] | (o[5] << 16);
        u.w = o[6] | (o[7] << 16);
        *cp = u;
      }
    }
  }
  __syncthreads();

  // epilogue 2: two whole rows (256 bytes each) per warp-instruction back to
  // global memory
  if (acc_ok && y_ok) {
    const int64_t ld = (int64_t)p.slices * N;
    const int64_t ncols = min((int64_t)kBN, N - n0);
    for (int m0 = 2 * warp; m0 < nrows; m0 += 8) {
      const int m = m0 + lane / 16;
      const int ch = lane % 16;            // 16-byte chunk of the 256-byte row
      if (m >= nrows || (int64_t)ch * 8 >= ncols) continue;
      const int cb = ch / 8, c = ch % 8;
      const uint4 u =
          *reinterpret_cast<const uint4*>(s_y + cb * kYBlockBytes + m * 128 + ((c ^ (m & 7)) * 16));
      *reinterpret_cast<uint4*>(p.y + (int64_t)rows_s[m] * ld + y_col + ch * 8) = u;
    }
  }
  if (!(acc_ok && y_ok)) {
    if (tid == 0) {
      mbar_wait_bounded(&ctl->bar_b, 0, p.status);
      mbar_wait_bounded(&ctl->bar_y, 0, p.status);
    }
  }
  teardown();
}

}  // namespace

cudaError_t launch_expand_mma(const MmaExpandParams& p, int64_t tiles_max, cudaStream_t st) {
  const size_t smem = mma_expand_smem((int)p.r, (p.flags & IG_FLAG_Z_FP32) != 0);
  cudaError_t e = cudaFuncSetAttribute(expand_mma_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = tiles_max * p.slices * p.ntiles;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(expand_mma_kernel, dim3((unsigned)grid), dim3(kThreads), smem, st, p);
}

size_t expand_mma_smem_bytes(int r) { return mma_expand_smem(r, false); }

}  // namespace ig
