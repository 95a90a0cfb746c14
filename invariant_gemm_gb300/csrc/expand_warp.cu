// LoRA expand for small ranks: y += bf16(Z) B_i^T, in place, one rounding,
// on the warp-level tensor cores.
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// Eq. 1 (the expand multiplies the r-wide shrink output by B in
// R^{Hout x r}) and sec. 6.2 / Fig. 5 (the FP32 shrink output reaches the
// next operation as BF16, rounded to nearest).
//
// For each output element:
//   D = tensor-core sum over j of bf16_rn(z[j]) * B[n][j]   (FP32)
//   y = bf16_rn(f32(y) + D)
// with the MMA sequence of warp_mma.cuh: 16-element j chunks in increasing
// order (m16n8k16, then m16n8k8 for a last 8), D rows = 16 output
// columns, D columns = the tile's 8 token rows. Every element comes from one MMA of
// one warp, so the result does not depend on the tiling, on M or on the
// other rows, and it is the same as the fused decode kernel's.
//
// Block = 4 warps, tile = up to 8 token rows of one adapter (one entry of
// the token map's tile table) x 256 output columns of one slice. The
// block's B columns are copied by TMA as 128-byte rows (128-byte swizzle);
// the tile's Z rows are read from global memory once, rounded (or split
// into three bf16 parts with IG_FLAG_Z_FP32) into shared memory. The
// block's columns form 8 groups of 32: warp w takes the groups w and w + 4,
// and lane 4g + t updates columns 4g .. 4g+3 of each in the rows of tokens
// 2t and 2t + 1, with one 8-byte load and store of y per row and group.
//
// Latency: the tile entry is read before griddep_wait(); with
// IG_FLAG_STATIC_WEIGHTS the block's B copy is issued before it too. After
// the wait each lane issues its y loads, then Z is read and the MMAs run.
#include <type_traits>

#include "warp_mma.cuh"

namespace ig {

namespace {

constexpr int kThreads = kExpandWarps * 32;
constexpr int kMaxRank = 256;
constexpr int kGW = kExpandBN / 32 / kExpandWarps;   // 32-column groups per warp (2)

struct ExpandLayout {
  int box_rows, nbox;
  size_t zb_off, b_off, bytes;
};

__host__ __device__ inline ExpandLayout expand_layout(int r, int64_t N) {
  ExpandLayout L;
  const int cols = (int)(N < kExpandBN ? N : kExpandBN);
  const int brows = cols * r / 64;   // 128-byte B rows of a full block
  L.box_rows = brows < 256 ? brows : 256;
  L.nbox = (brows + L.box_rows - 1) / L.box_rows;
  L.zb_off = 64;
  L.b_off = (L.zb_off + (size_t)3 * kTileRows * r * 2 + 1023) / 1024 * 1024;
  // room for whole 32-column groups (rows past the block's columns are read
  // by the MMAs of a partial last group, never used)
  const int rows_alloc = (cols + 31) / 32 * 32 * r / 64;
  const int rows_loaded = L.nbox * L.box_rows;
  L.bytes = L.b_off + (size_t)(rows_loaded > rows_alloc ? rows_loaded : rows_alloc) * 128;
  return L;
}

__global__ void __launch_bounds__(kThreads, 2)
    expand_warp_kernel(const __grid_constant__ ExpandParams p) {
  // the next kernel may be scheduled now: it reads nothing of ours before
  // its own griddep_wait(), which waits for this grid to complete
  griddep_launch();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int r = (int)p.r;
  const ExpandLayout lay = expand_layout(r, p.N);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint16_t* zb = reinterpret_cast<uint16_t*>(smem + lay.zb_off);   // [3][8][r]
  uint8_t* sB = smem + lay.b_off;
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

  const int64_t N = p.N;
  const int64_t n0 = (int64_t)nt * kExpandBN;
  const int ncols = (int)min((int64_t)kExpandBN, N - n0);
  const int brows = ncols * r / 64;
  const int nbox = (brows + lay.box_rows - 1) / lay.box_rows;
  const bool early_b = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;
  const int b_row0 = (int)((((int64_t)g * p.slices + sl) * N + n0) * r / 64);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, (uint32_t)(nbox * lay.box_rows * 128));
  }
  __syncthreads();
  auto issue_b = [&]() {
    if (tid == 0)
      for (int bi = 0; bi < nbox; ++bi)
        tma_load_2d(sB + (size_t)bi * lay.box_rows * 128, &p.tm_b, 0, b_row0 + bi * lay.box_rows,
                    bar);
  };
  if (early_b) issue_b();

  griddep_wait();
  if (!early_b) issue_b();

  const int64_t M = p.M;
  // lane 4g + t updates columns 4g .. 4g+3 of each of its groups in the rows
  // of tokens 2t and 2t + 1 (warp_mma.cuh)
  const int gq = lane >> 2, tq = lane & 3;
  const bool has0 = 2 * tq < nrows, has1 = 2 * tq + 1 < nrows;
  const int64_t ld = (int64_t)p.slices * N;
  __nv_bfloat16* yrow0 = p.y + (int64_t)ent[4 + min(2 * tq, nrows - 1)] * ld + (int64_t)sl * N +
                         n0 + 4 * gq;
  __nv_bfloat16* yrow1 = p.y + (int64_t)ent[4 + min(2 * tq + 1, nrows - 1)] * ld +
                         (int64_t)sl * N + n0 + 4 * gq;
  auto col_ok = [&](int cb) { return cb + 4 * gq < ncols; };
  uint2 ypre[kGW][2];
#pragma unroll
  for (int i = 0; i < kGW; ++i) {
    const int cb = 32 * (warp + i * kExpandWarps);
    ypre[i][0] = has0 && col_ok(cb) ? ldg_cg_v2(yrow0 + cb) : make_uint2(0u, 0u);
    ypre[i][1] = has1 && col_ok(cb) ? ldg_cg_v2(yrow1 + cb) : make_uint2(0u, 0u);
  }

  // The tile's Z rows -> bf16 parts in shared memory (rows past nrows zero).
  // L2 only: Z was written by the previous kernel.
  const bool zf32 = (p.flags & IG_FLAG_Z_FP32) != 0;
  for (int o = tid; o < kTileRows * r; o += kThreads) {
    const int row = o / r;
    uint16_t hi = 0, mid = 0, lo = 0;
    if (row < nrows) split_z(__ldcg(p.z + ((int64_t)sl * M + ent[4 + row]) * r + o % r), zf32,
                             hi, mid, lo);
    zb[o] = hi;
    zb[kTileRows * r + o] = mid;
    zb[2 * kTileRows * r + o] = lo;
  }
  __syncthreads();
  // every thread waits for the B slice, so the block never exits with copies
  // in flight; after an expired wait, once more (bounded) before it leaves
  if (!mbar_wait_bounded(bar, 0, p.status)) {
    mbar_wait_bounded(bar, 0, p.status);
    return;
  }

  const uint32_t sB_addr = smem_u32(sB);
  const int parts = zf32 ? 3 : 1;
  const int cmax = ncols - 1;
  auto store = [&](int cb, const uint2 (&yv)[2], const float (&v)[8]) {
    if (!col_ok(cb)) return;
    if (has0) *reinterpret_cast<uint2*>(yrow0 + cb) = y_add4(yv[0], v[0], v[1], v[2], v[3]);
    if (has1) *reinterpret_cast<uint2*>(yrow1 + cb) = y_add4(yv[1], v[4], v[5], v[6], v[7]);
  };
  if (!zf32 && (r == 16 || r == 8)) {
    // A operands of the warp's groups, then their MMAs, then the y updates
    // (the same MMAs as expand_group_mma)
    auto run = [&](auto rank) {
      constexpr int R = decltype(rank)::value;
      ExpandFrag<R> zf;
      zf.load_z(zb, lane);
      uint32_t bq[kGW][2][4];
      uint32_t off[2];
      ExpandFrag<R>::lane_offsets(lane, warp & 1, off);
#pragma unroll
      for (int i = 0; i < kGW; ++i) {
        const int grp = warp + i * kExpandWarps;   // whole warp: groups past ncols skipped
        if (32 * grp < ncols)
          ExpandFrag<R>::load_b_at(sB_addr + (uint32_t)(grp >> 1) * (128u * R), off, bq[i]);
      }
      float v[kGW][8];
#pragma unroll
      for (int i = 0; i < kGW; ++i) zf.mma(v[i], bq[i]);
#pragma unroll
      for (int i = 0; i < kGW; ++i) store(32 * (warp + i * kExpandWarps), ypre[i], v[i]);
    };
    if (r == 16) run(std::integral_constant<int, 16>());
    else run(std::integral_constant<int, 8>());
    return;
  }
#pragma unroll
  for (int i = 0; i < kGW; ++i) {
    const int cb = 32 * (warp + i * kExpandWarps);
    if (cb >= ncols) break;
    float v[8];
    expand_group_mma(v, sB_addr, cb, cmax, r, zb, parts, lane);
    store(cb, ypre[i], v);
  }
}

}  // namespace

size_t expand_warp_smem_bytes(int r, int64_t N) { return 1024 + expand_layout(r, N).bytes; }
int expand_warp_box_rows(int r, int64_t N) { return expand_layout(r, N).box_rows; }

cudaError_t launch_expand_warp(const ExpandParams& p, int64_t tiles_max, cudaStream_t st) {
  if (p.r > kMaxRank || p.r % 8 != 0) return cudaErrorInvalidValue;
  const int64_t grid = tiles_max * p.slices * p.ntiles;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = expand_warp_smem_bytes((int)p.r, p.N);
  cudaError_t e = cudaFuncSetAttribute(expand_warp_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(expand_warp_kernel, dim3((unsigned)grid), dim3(kThreads), smem, st, p);
}

}  // namespace ig
