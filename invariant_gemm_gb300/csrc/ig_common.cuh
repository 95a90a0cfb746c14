// Internal definitions shared by the kernels and the host core of the
// invariant_gemm library: workspace layout, device status bits, launch
// parameter blocks, and small device helpers (bf16 conversion, mbarrier and
// bulk-copy wrappers, bounded waits).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/invariant_gemm.h"

namespace ig {

// ---------------------------------------------------------------------------
// workspace layout
//
//   [0, 256)                      status words (u32 status at offset 0)
//   [256, 256 + 4*kMaxCounters)   per-tile completion counters (u32)
//   [kMapOffset, ...)             token map: perm[M] int32, offsets[G+1]
//                                 int32, tile table [tiles_max][kTileInts]
//                                 int32 (each at a 256-byte boundary)
//   [partials, ...)               FP32 partials [slots][S][BM*BN] (DET only)
//
// The counters sit at a fixed place whatever the shape, so one
// ig_workspace_init makes a workspace valid for every later call that fits
// in it: counters are only ever left at zero (Algorithm 1: the last arriver resets its counter).
// ---------------------------------------------------------------------------
constexpr int64_t kMaxCounters = 65536;
constexpr size_t kStatusBytes = 256;
constexpr size_t kCountersOffset = kStatusBytes;
constexpr size_t kMapOffset = kCountersOffset + 4 * kMaxCounters;
constexpr int kMaxAdapters = 1023;  // token-map groups G = L + 1 <= 1024

constexpr uint32_t kStatusAdapterRange = 1u << 0;
constexpr uint32_t kStatusCorrupt = 1u << 1;
constexpr uint32_t kStatusTimeout = 1u << 2;

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) {
  return (v + a - 1) / a * a;
}

// Small-rank (warp-MMA) path geometry (fixed: part of the determinism key
// where it sets the arithmetic order).
constexpr int kTileRows = 8;           // token rows per tile of the tile table (the MMA's N)
constexpr int kTileInts = 4 + kTileRows;  // [g, nrows, consecutive, 0, rows[8]] = 48 bytes
constexpr int kShrinkKB = 256;        // elements per k-block (4 swizzled sub-blocks of 64)
constexpr int kShrinkStages = 4;
constexpr int kExpandWarps = 4;
constexpr int kExpandBN = 256;        // output columns per expand block: 4 warps x 2 groups of 32
// Revision of the arithmetic of the kernels; part of the determinism key.
constexpr int kArithRevision = 4;
// tensor-core path: 128-row tiles (the MMA's M)
constexpr int kMmaTileRows = 128;
// Z operand of the tcgen05 expand for one (tile, slice): the tile's 128 rows
// of Z as bf16 (three parts hi, mid, lo with FP32 Z), each part ceil(r / 64)
// atoms of [128 rows][128 bytes], 128-byte swizzled (16-byte chunk c of row m
// at chunk c ^ (m % 8)). Written by the shrink inside lora_apply, so that the
// expand copies it instead of building it from z.
__host__ __device__ inline size_t zt_entry_bytes(int64_t r, bool z_fp32) {
  return (size_t)((r + 63) / 64) * 16384u * (z_fp32 ? 3u : 1u);
}
constexpr int kMmaTileInts = 4 + kMmaTileRows;
constexpr int kMmaExpandCols = 1024;   // most output columns per tensor-core expand block
constexpr int kMmaExpandBN = 64;       // output columns per MMA (N) of that block

// Tile count over token groups: sum over groups g of ceil(count_g / bm),
// bounded by floor(M / bm) + (number of non-empty groups).
inline int64_t tiles_upper_bound(int64_t M, int64_t groups, int64_t bm) {
  if (M <= 0) return 0;
  int64_t ne = groups < M ? groups : M;
  return M / bm + ne;
}

struct MapParams {
  const int32_t* idx;
  int32_t* perm;
  int32_t* offsets;
  int32_t* tiles;      // tile table [tiles_max][kTileInts]
  uint32_t* status;
  int64_t M;
  int64_t tiles_max;
  int32_t L;
  int32_t tile_rows;   // 8 (warp and FMA paths) or 128 (tcgen05 path)
};

struct ShrinkParams {
  CUtensorMap tm_x;     // x [M][K], box 256 x 1, no swizzle (FMA path row gathers)
  CUtensorMap tm_a;     // A_stack as [L*slices*r][K], box 64 x BN, 128-byte swizzle
  CUtensorMap tm_a3;    // the same as {64, rows, K/64}, box {64, BN, 4} (when has_a3)
  const __nv_bfloat16* x;
  const __nv_bfloat16* A;
  const int32_t* tiles;
  float* z;
  float* partials;
  uint32_t* counters;
  uint32_t* status;
  int64_t M, K, r, Ks;
  int32_t slices, L, S, jblocks, flags;
  int32_t has_a3;       // K and K/S multiples of 64: one 3-D copy per k-block of A
  float scale;
};

struct ExpandParams {
  CUtensorMap tm_b;     // B_stack as rows of 64 elements, box 64 x box_rows, 128-byte swizzle
  const float* z;
  const __nv_bfloat16* B;
  const int32_t* tiles;
  __nv_bfloat16* y;
  uint32_t* status;
  int64_t M, N, r;
  int32_t slices, L, ntiles, flags;
};

// 2-D bf16 tensor map [rows][cols] with the given row stride; box
// box_cols x box_rows; swizzle is a CUtensorMapSwizzle value. IG_OK or
// IG_ERR_CUDA (driver entry point missing or encode rejected).
int encode_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                  uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows, int swizzle);
// A_stack [rows][K] (K % 64 == 0) seen as a 3-D bf16 tensor {64, rows, K / 64}
// with strides {K * 2, 128} bytes: a box {64, box_rows, 4} brings 4
// consecutive 64-element sub-blocks of box_rows rows, stored sub-block by
// sub-block, 128-byte swizzled. IG_OK or IG_ERR_CUDA.
int encode_map_a3(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K,
                  uint32_t box_rows);

struct FusedParams {
  CUtensorMap tm_x;     // x [M][K], box 256 x 1, no swizzle (FMA path row gathers)
  CUtensorMap tm_a;     // A_stack as [L*slices*r][K], box 64 x r, 128-byte swizzle
  CUtensorMap tm_a3;    // the same as {64, rows, K/64}, box {64, r, 4} (when has_a3)
  CUtensorMap tm_b;     // B_stack as rows of 64 elements (64/r output columns
                        // x r), box 64 x b_box_rows, 128-byte swizzle
  const __nv_bfloat16* x;
  const __nv_bfloat16* A;
  const __nv_bfloat16* B;
  const int32_t* tiles;
  float* z;
  __nv_bfloat16* y;
  uint32_t* status;
  int64_t M, K, N, Ks;
  int32_t slices, L, S, flags;
  int32_t b_box_rows;
  int32_t has_a3;
  float scale;
};

struct MmaShrinkParams {
  CUtensorMap tm_x;     // x [M][K], box 64 x 1, 128-byte swizzle (row gathers)
  CUtensorMap tm_xt;    // x [M][K], box 64 x 128, 128-byte swizzle (contiguous tiles)
  CUtensorMap tm_a;     // A_stack as [L*slices*r][K], box 64 x (stack*r), 128-byte swizzle
  const int32_t* tiles; // 128-row tile table
  float* z;
  float* partials;
  uint32_t* counters;
  uint32_t* status;
  int64_t M, K, r, Ks;
  int32_t slices, L, S, flags;
  int32_t stack;        // slices per block (1, or all slices: MMA N = slices x r)
  float scale;
  uint8_t* zt;          // Z operand tiles for the expand (entry t * slices + slice), or null
};

struct MmaExpandParams {
  CUtensorMap tm_b;     // B_stack as [L*slices*N][r], box 64 x 64, 128-byte swizzle
  CUtensorMap tm_yt;    // y [M][slices*N], box 64 x 128, 128-byte swizzle (contiguous tiles)
  const float* z;
  const int32_t* tiles; // 128-row tile table
  __nv_bfloat16* y;
  uint32_t* status;
  int64_t M, N, r;
  int32_t slices, L, ntiles, flags;
  int32_t nb;           // 64-column blocks per thread block (columns per block / 64)
  const uint8_t* zt;    // Z operand tiles written by the shrink, or null: build from z
};

struct TreeParams {
  const float* partials;
  const int32_t* tiles;
  float* z;
  int64_t M, r;
  int32_t tile_rows, bn, jblocks, slices, L, S;
  float scale;
};

// Launchers (defined in the .cu files); they return cudaGetLastError().
cudaError_t launch_map_tokens(const MapParams& p, cudaStream_t st);
cudaError_t launch_shrink_warp(const ShrinkParams& p, int mode, int bn,
                              int64_t tiles_max, cudaStream_t st);
cudaError_t launch_expand_warp(const ExpandParams& p, int64_t tiles_max,
                              cudaStream_t st);
cudaError_t launch_fused_warp(const FusedParams& p, int bn, int64_t tiles_max, cudaStream_t st);
size_t fused_smem_bytes(int bn, int64_t Ks, int64_t N, int S);
int fused_b_box_rows(int bn, int64_t Ks, int64_t N, int S);
size_t expand_warp_smem_bytes(int r, int64_t N);
// IG_PATH_FMA (CUDA cores): the same kernel roles with FP32 FMA arithmetic
cudaError_t launch_shrink_fma(const ShrinkParams& p, int mode, int bn, int64_t tiles_max,
                              cudaStream_t st);
cudaError_t launch_expand_fma(const ExpandParams& p, int64_t tiles_max, cudaStream_t st);
cudaError_t launch_fused_fma(const FusedParams& p, int bn, int64_t tiles_max, cudaStream_t st);
size_t fused_fma_smem_bytes(int bn, int64_t Ks, int64_t N, int S);
int fused_fma_b_box_rows(int bn, int64_t Ks, int64_t N, int S);
int expand_warp_box_rows(int r, int64_t N);
cudaError_t launch_shrink_mma(const MmaShrinkParams& p, int mode, int64_t tiles_max,
                              cudaStream_t st);
cudaError_t launch_expand_mma(const MmaExpandParams& p, int64_t tiles_max, cudaStream_t st);
size_t expand_mma_smem_bytes(int r, bool z_fp32);
cudaError_t launch_reduce_tree(const TreeParams& p, int64_t tiles_max, cudaStream_t st);

// Launch helper: programmatic dependent launch on `st` (see griddep_wait).
template <typename Kern, typename P>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const P& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

#ifdef __CUDACC__
// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x);
  f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z);
  f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

// FP32 -> BF16 bits, round to nearest, ties to even (cvt.rn.bf16.f32).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Two values in one conversion (cvt.rn.bf16x2.f32): lo -> bits 0..15, hi ->
// bits 16..31. Where values come in pairs this is the cheapest rounding on
// GB300: half the conversion instructions of the scalar form, and fewer
// issue slots than rounding on the integer pipes.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return (uint32_t)__bfloat16_as_ushort(h.x) | ((uint32_t)__bfloat16_as_ushort(h.y) << 16);
}
__device__ __forceinline__ float bf16_round_f32(float f) {
  return __uint_as_float(f32_to_bf16_bits(f) << 16);
}

// Programmatic dependent launch. A kernel launched with
// cudaLaunchAttributeProgrammaticStreamSerialization may start before the
// previous kernel on the stream has finished; griddep_wait() blocks until that
// kernel has completed and its memory is visible. Every kernel here reads
// activations, z, y and workspace state, and writes anything, only after
// griddep_wait(). griddep_launch() lets the next kernel start launching:
// the warp-level tensor-core kernels (and the pairwise-tree combine) call it
// first thing, so that the next layer's blocks are resident and through
// their prologue (tile entry, weight copies) by the time this grid
// completes; the tcgen05 kernels call it only after their wait, so that no
// early block of the next kernel can hold tensor memory that a block of
// this one still has to allocate, and so do the CUDA-core FMA kernels (their
// decode layer measured 20% slower with the early release).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Next digit of a block index, in 32-bit unsigned arithmetic (grids stay
// below 2^31 blocks, and the divisors are small): v becomes v / d, the
// remainder is returned. A 64-bit division by a runtime value costs every
// thread a long instruction sequence; this one a few instructions.
__device__ __forceinline__ uint32_t next_digit(uint32_t& v, uint32_t d) {
  const uint32_t q = v / d;
  const uint32_t rem = v - q * d;
  v = q;
  return rem;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Non-blocking check of an mbarrier phase (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase. Gives up after ~2^31 SM clocks (about a
// second), records kStatusTimeout and returns false. A budget of 0 or less
// checks the phase once without waiting (IG_FLAG_TEST_COPY_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t* status,
                                                  long long budget = 1ll << 31) {
  if (budget <= 0) {
    if (mbar_test_wait(bar, parity)) return true;
    atomicOr(status, kStatusTimeout);
    return false;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// --- thread-block clusters ------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Split cluster barrier. The arrive carries no memory ordering: it only
// tells the other blocks that this block's mbarriers are initialised (made
// visible to the cluster by fence.mbarrier_init before it).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in block `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  return remote;
}
// Asynchronous 4-byte store into another block's shared memory; its bytes
// are counted (complete_tx) on that block's mbarrier `remote_bar`.
__device__ __forceinline__ void st_async_f32(uint32_t remote, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               ::"r"(remote), "r"(__float_as_uint(v)), "r"(remote_bar) : "memory");
}
// Asynchronous 16-byte store into another block's shared memory, counted on
// that block's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t remote, float4 v, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(remote), "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)),
        "r"(__float_as_uint(v.z)), "r"(__float_as_uint(v.w)), "r"(remote_bar) : "memory");
}
// Full cluster barrier: every block's earlier memory operations are visible
// to the cluster afterwards.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Z split for the expand's A operand: hi = bf16(z); with full FP32 Z also
// mid = bf16(z - hi) and lo = bf16(z - hi - mid), each difference exact, so
// that hi + mid + lo == z exactly (24 significant bits = 3 x 8).
__device__ __forceinline__ void split_z(float z, bool fp32, uint16_t& hi, uint16_t& mid,
                                        uint16_t& lo) {
  const uint32_t h = f32_to_bf16_bits(z);
  hi = (uint16_t)h;
  if (!fp32) {
    mid = lo = 0;
    return;
  }
  const float r1 = z - __uint_as_float(h << 16);
  const uint32_t m = f32_to_bf16_bits(r1);
  const float r2 = r1 - __uint_as_float(m << 16);
  mid = (uint16_t)m;
  lo = (uint16_t)f32_to_bf16_bits(r2);
}

// Fetch a kernel-parameter tensor map into the descriptor cache early.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Tiled 2-D tensor copy global -> shared (box of the tensor map at
// coordinates {c0 = column, c1 = row}); c0 * 2 bytes must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
        "r"(smem_u32(bar)) : "memory");
}
// Tiled 3-D tensor copy global -> shared (box at coordinates {c0, c1, c2},
// innermost first); c0 * 2 bytes must be a multiple of 16.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
        "r"(smem_u32(bar)) : "memory");
}
// Row gather: four rows r0..r3 of a 2-D tensor map whose box is one row high,
// columns [c0, c0 + box), written one after the other to dst.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, int c0, int r0,
                                            int r1, int r2, int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r0), "r"(r1),
        "r"(r2), "r"(r3), "r"(smem_u32(bar)) : "memory");
}

// One-dimensional bulk copy global -> shared, completion counted in bytes on
// the mbarrier. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// 8-byte global load cached in L2 only, issued where it stands (see below).
__device__ __forceinline__ uint2 ldg_cg_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
// 16-byte global load cached in L2 only, issued where it stands: volatile,
// so that the compiler neither sinks it towards its first use (a load meant
// to be in flight during other work) nor merges it away.
__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Ask for `bytes` (a multiple of 16, from a 16-byte aligned address) to be
// brought into L2; no destination, no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

#endif  // __CUDACC__

}  // namespace ig
