// Host core of the invariant_gemm C ABI: argument validation, the plan (a
// function of K, r, N, slices, split_k, mode and path, never of M), the
// workspace layout, and the launch sequence of each entry point.
#include <cstdio>
#include <cstring>
#include <mutex>

#include <algorithm>
#include <map>

#include "ig_common.cuh"

namespace ig {
namespace {

struct Plan {
  int path;          // IG_PATH_WARP / IG_PATH_MMA
  int mode;
  int S;             // partitions
  int64_t Ks;        // K / S
  int bn;            // shrink rank columns per tile
  int jblocks;       // r / bn
  int stack;         // tcgen05 shrink: slices per block (1, or all: MMA N = slices x r)
  int tile_rows;     // rows per tile: 8 (warp and FMA paths) or 128 (tcgen05)
  int64_t tiles;     // tile-table entries: upper bound on tiles (groups 0..L)
  int ntiles;        // expand column tiles per slice
  size_t off_perm, off_offsets, off_tiles, off_partials, off_zt, zt_bytes, total;
  bool fused;        // lora_apply runs the one-launch cluster kernel
  uint64_t key;
};

uint64_t fnv1a(uint64_t h, int64_t v) {
  for (int i = 0; i < 8; ++i) {
    h ^= (uint64_t)((v >> (8 * i)) & 0xff);
    h *= 1099511628211ull;
  }
  return h;
}

int make_plan(const ig_shape* sh, Plan* pl) {
  if (!sh || !pl) return IG_ERR_ARG;
  if ((sh->flags & ~(IG_FLAG_STATIC_WEIGHTS | IG_FLAG_UNFUSED | IG_FLAG_Z_FP32 |
                     IG_FLAG_TEST_COPY_TIMEOUT | IG_FLAG_INPUT_READY)) != 0)
    return IG_ERR_ARG;
  if (sh->mode < IG_MODE_DET || sh->mode > IG_MODE_DET_TREE) return IG_ERR_ARG;
  if (sh->path < IG_PATH_AUTO || sh->path > IG_PATH_FMA) return IG_ERR_ARG;
  const int64_t M = sh->M, K = sh->K, N = sh->N, r = sh->r;
  if (M < 0 || K < 8 || N < 8 || r < 8) return IG_ERR_SHAPE;
  if (K % 8 || N % 8 || r % 8) return IG_ERR_SHAPE;
  if (sh->slices < 1 || sh->num_adapters < 1) return IG_ERR_SHAPE;
  const int64_t lim = (int64_t)1 << 40;
  // K and N: 32-bit tensor-map coordinates and column indices in the kernels
  if (M > (1ll << 31) - 1 || K > (1ll << 31) - 1 || N > (1ll << 31) - 1 || r > 256)
    return IG_ERR_UNSUPPORTED;
  if (M * K > ((int64_t)1 << 46) || (int64_t)sh->slices * N * r > lim) return IG_ERR_UNSUPPORTED;
  if (sh->num_adapters > kMaxAdapters) return IG_ERR_UNSUPPORTED;
  int S = sh->mode == IG_MODE_UNSPLIT ? 1 : sh->split_k;
  if (S < 1) return IG_ERR_SHAPE;
  if ((K / 8) % S) return IG_ERR_SHAPE;
  // Tensor cores where the token x rank x K tile is a dense contraction:
  // ranks of 32 and more (prefill-class adapters). Decided from r and K/S,
  // never from M.
  // With FP32 Z the tcgen05 expand keeps three bf16 parts of the tile's Z in
  // shared memory, which for r = 256 no longer fits beside its copy stages.
  const bool mma_ok = r % 16 == 0 && (K / S) % 16 == 0 && r <= 256 &&
                      expand_mma_smem_bytes((int)r, (sh->flags & IG_FLAG_Z_FP32) != 0) <=
                          227 * 1024;
  int path = sh->path;
  if (path == IG_PATH_AUTO) path = (mma_ok && r >= 32) ? IG_PATH_MMA : IG_PATH_WARP;
  if (path == IG_PATH_MMA && !mma_ok) return IG_ERR_UNSUPPORTED;

  pl->path = path;
  pl->mode = sh->mode;
  pl->S = S;
  pl->Ks = K / S;
  const bool mma = path == IG_PATH_MMA;
  pl->bn = mma ? (int)r : ((r % 16 == 0) ? 16 : 8);
  pl->jblocks = mma ? 1 : (int)(r / pl->bn);
  // The tcgen05 shrink runs all slices of a tile in one block (one x tile
  // read, one MMA of N = slices x r) where N fits one MMA; not for the
  // pairwise-tree mode, whose second launch reads one slice per block.
  pl->stack = (mma && sh->slices > 1 && sh->slices * r <= 256 &&
               sh->mode != IG_MODE_DET_TREE) ? sh->slices : 1;
  pl->tile_rows = mma ? kMmaTileRows : kTileRows;
  const int L = sh->num_adapters;
  pl->tiles = tiles_upper_bound(M, L + 1, pl->tile_rows);
  pl->ntiles = (int)((N + kExpandBN - 1) / kExpandBN);
  const int64_t slots = pl->tiles * sh->slices * pl->jblocks;
  const bool partials = sh->mode == IG_MODE_DET || sh->mode == IG_MODE_DET_TREE;
  if (sh->mode == IG_MODE_DET && slots > kMaxCounters) return IG_ERR_UNSUPPORTED;
  if (sh->mode == IG_MODE_DET_TREE && S > 64) return IG_ERR_UNSUPPORTED;

  pl->off_perm = kMapOffset;
  pl->off_offsets = align_up(pl->off_perm + 4 * (size_t)M, 256);
  pl->off_tiles = align_up(pl->off_offsets + 4 * (size_t)(L + 2), 256);
  pl->off_partials =
      align_up(pl->off_tiles + 4 * (size_t)(4 + pl->tile_rows) * pl->tiles, 256);
  size_t part = 0;
  if (partials) part = (size_t)slots * S * pl->tile_rows * pl->bn * sizeof(float);
  // the tcgen05 expand's Z operand, written by the shrink inside lora_apply
  // where one block writes each final z value (DET, UNSPLIT)
  pl->off_zt = align_up(pl->off_partials + part, 1024);
  pl->zt_bytes = (mma && (sh->mode == IG_MODE_DET || sh->mode == IG_MODE_UNSPLIT))
                     ? (size_t)pl->tiles * sh->slices *
                           zt_entry_bytes(r, (sh->flags & IG_FLAG_Z_FP32) != 0)
                     : 0;
  pl->total = align_up(pl->off_zt + pl->zt_bytes, 256);

  // The fused kernel expands N/S columns per block; past 1024 the two-kernel
  // path (256-column expand blocks) is faster. Both give the same bits.
  const size_t fsmem = path == IG_PATH_FMA ? fused_fma_smem_bytes(pl->bn, pl->Ks, N, S)
                                           : fused_smem_bytes(pl->bn, pl->Ks, N, S);
  pl->fused = sh->mode == IG_MODE_DET && (path == IG_PATH_WARP || path == IG_PATH_FMA) &&
              (r == 8 || r == 16) && pl->bn == r && S <= 16 && (N + S - 1) / S <= 1024 &&
              !(sh->flags & IG_FLAG_UNFUSED) && fsmem <= 200 * 1024;

  uint64_t h = 1469598103934665603ull;
  const int64_t fields[] = {IG_ABI_VERSION, kArithRevision, path, sh->mode, S, pl->Ks, K, r, N,
                            sh->slices, pl->bn, mma ? 64 : kShrinkKB, pl->stack,
                            sh->flags & IG_FLAG_Z_FP32};
  for (int64_t f : fields) h = fnv1a(h, f);
  pl->key = h;
  return IG_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// SMs of the current device (cached per device; 152 on GB300).
int sm_count() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  cache[dev] = n;
  return n;
}

int check_ws(const Plan& pl, void* ws, size_t ws_bytes) {
  if (!ws) return IG_ERR_ARG;
  if (!aligned16(ws)) return IG_ERR_ALIGN;
  if (ws_bytes < pl.total) return IG_ERR_WS_SMALL;
  return IG_OK;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return IG_OK;
  return IG_ERR_CUDA;
}

int run_map(const ig_shape* sh, const Plan& pl, const int32_t* idx, uint8_t* ws,
            cudaStream_t st) {
  MapParams mp;
  mp.idx = idx;
  mp.perm = reinterpret_cast<int32_t*>(ws + pl.off_perm);
  mp.offsets = reinterpret_cast<int32_t*>(ws + pl.off_offsets);
  mp.tiles = reinterpret_cast<int32_t*>(ws + pl.off_tiles);
  mp.status = reinterpret_cast<uint32_t*>(ws);
  mp.M = sh->M;
  mp.tiles_max = pl.tiles;
  mp.tile_rows = pl.tile_rows;
  mp.L = sh->num_adapters;
  return cuda_status(launch_map_tokens(mp, st));
}

int run_shrink_mma(const ig_shape* sh, const Plan& pl, const void* x, const void* A,
                   float scale, float* z, uint8_t* ws, cudaStream_t st, uint8_t* zt) {
  MmaShrinkParams p;
  int rc = encode_map_2d(&p.tm_x, x, (uint64_t)sh->M, (uint64_t)sh->K, (uint64_t)sh->K * 2, 64,
                         1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != IG_OK) return rc;
  rc = encode_map_2d(&p.tm_xt, x, (uint64_t)sh->M, (uint64_t)sh->K, (uint64_t)sh->K * 2, 64,
                     kMmaTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != IG_OK) return rc;
  rc = encode_map_2d(&p.tm_a, A, (uint64_t)sh->num_adapters * sh->slices * sh->r,
                     (uint64_t)sh->K, (uint64_t)sh->K * 2, 64, (uint32_t)(pl.stack * sh->r),
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != IG_OK) return rc;
  p.tiles = reinterpret_cast<const int32_t*>(ws + pl.off_tiles);
  p.z = z;
  p.partials = reinterpret_cast<float*>(ws + pl.off_partials);
  p.counters = reinterpret_cast<uint32_t*>(ws + kCountersOffset);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.M = sh->M;
  p.K = sh->K;
  p.r = sh->r;
  p.Ks = pl.Ks;
  p.slices = sh->slices;
  p.L = sh->num_adapters;
  p.S = pl.S;
  p.stack = pl.stack;
  p.flags = sh->flags;
  p.scale = scale;
  p.zt = zt;
  return cuda_status(launch_shrink_mma(p, pl.mode, pl.tiles, st));
}

int run_expand_mma(const ig_shape* sh, const Plan& pl, const float* z, const void* B, void* y,
                   uint8_t* ws, cudaStream_t st, const uint8_t* zt) {
  MmaExpandParams p;
  int rc = encode_map_2d(&p.tm_b, B, (uint64_t)sh->num_adapters * sh->slices * sh->N,
                         (uint64_t)sh->r, (uint64_t)sh->r * 2, 64, kMmaExpandBN,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != IG_OK) return rc;
  rc = encode_map_2d(&p.tm_yt, y, (uint64_t)sh->M, (uint64_t)sh->slices * sh->N,
                     (uint64_t)sh->slices * sh->N * 2, 64, kMmaTileRows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != IG_OK) return rc;
  p.z = z;
  p.tiles = reinterpret_cast<const int32_t*>(ws + pl.off_tiles);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.M = sh->M;
  p.N = sh->N;
  p.r = sh->r;
  p.slices = sh->slices;
  p.L = sh->num_adapters;
  // column blocks of 64 per thread block: enough blocks for about three per
  // SM, each streaming at least 2 and at most 16 column blocks
  const int64_t nblk = (sh->N + kMmaExpandBN - 1) / kMmaExpandBN;
  const int64_t units = pl.tiles * sh->slices * nblk;
  const int64_t target = 3 * (int64_t)sm_count();
  p.nb = (int)std::min<int64_t>(kMmaExpandCols / kMmaExpandBN,
                                std::max<int64_t>(2, (units + target - 1) / target));
  p.ntiles = (int)((nblk + p.nb - 1) / p.nb);
  p.flags = sh->flags;
  p.zt = zt;
  return cuda_status(launch_expand_mma(p, pl.tiles, st));
}

int run_tree(const ig_shape* sh, const Plan& pl, float scale, float* z, uint8_t* ws,
             cudaStream_t st) {
  TreeParams p;
  p.partials = reinterpret_cast<const float*>(ws + pl.off_partials);
  p.tiles = reinterpret_cast<const int32_t*>(ws + pl.off_tiles);
  p.z = z;
  p.M = sh->M;
  p.r = sh->r;
  p.tile_rows = pl.tile_rows;
  p.bn = pl.bn;
  p.jblocks = pl.jblocks;
  p.slices = sh->slices;
  p.L = sh->num_adapters;
  p.S = pl.S;
  p.scale = scale;
  return cuda_status(launch_reduce_tree(p, pl.tiles, st));
}

int run_shrink_only(const ig_shape* sh, const Plan& pl, const void* x, const void* A,
                    float scale, float* z, uint8_t* ws, cudaStream_t st, uint8_t* zt = nullptr);

// zt: where the tcgen05 shrink also writes the expand's Z operand (lora_apply)
int run_shrink(const ig_shape* sh, const Plan& pl, const void* x, const void* A, float scale,
               float* z, uint8_t* ws, cudaStream_t st, uint8_t* zt = nullptr) {
  const int rc = run_shrink_only(sh, pl, x, A, scale, z, ws, st, zt);
  if (rc != IG_OK || pl.mode != IG_MODE_DET_TREE) return rc;
  return run_tree(sh, pl, scale, z, ws, st);
}

int run_shrink_only(const ig_shape* sh, const Plan& pl, const void* x, const void* A,
                    float scale, float* z, uint8_t* ws, cudaStream_t st, uint8_t* zt) {
  if (pl.mode == IG_MODE_ATOMIC) {
    cudaError_t e = cudaMemsetAsync(z, 0, sizeof(float) * sh->slices * sh->M * sh->r, st);
    if (e != cudaSuccess) return IG_ERR_CUDA;
  }
  if (pl.path == IG_PATH_MMA) return run_shrink_mma(sh, pl, x, A, scale, z, ws, st, zt);
  ShrinkParams p;
  const bool fma = pl.path == IG_PATH_FMA;
  // x (FMA path only; the warp path loads x into registers): 256-element
  // rows, no swizzle; A: warp path 64-element boxes, 128-byte swizzle, FMA
  // path 256, no swizzle
  const uint32_t kbox = fma ? kShrinkKB : 64;
  const int swz = fma ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  int rc = IG_OK;
  if (fma) {
    rc = encode_map_2d(&p.tm_x, x, (uint64_t)sh->M, (uint64_t)sh->K, (uint64_t)sh->K * 2,
                       kShrinkKB, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != IG_OK) return rc;
  }
  rc = encode_map_2d(&p.tm_a, A, (uint64_t)sh->num_adapters * sh->slices * sh->r,
                     (uint64_t)sh->K, (uint64_t)sh->K * 2, kbox, (uint32_t)pl.bn, swz);
  if (rc != IG_OK) return rc;
  p.has_a3 = !fma && sh->K % 64 == 0 && pl.Ks % 64 == 0;
  if (p.has_a3) {
    rc = encode_map_a3(&p.tm_a3, A, (uint64_t)sh->num_adapters * sh->slices * sh->r,
                       (uint64_t)sh->K, (uint32_t)pl.bn);
    if (rc != IG_OK) return rc;
  }
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.A = static_cast<const __nv_bfloat16*>(A);
  p.tiles = reinterpret_cast<const int32_t*>(ws + pl.off_tiles);
  p.z = z;
  p.partials = reinterpret_cast<float*>(ws + pl.off_partials);
  p.counters = reinterpret_cast<uint32_t*>(ws + kCountersOffset);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.M = sh->M;
  p.K = sh->K;
  p.r = sh->r;
  p.Ks = pl.Ks;
  p.slices = sh->slices;
  p.L = sh->num_adapters;
  p.S = pl.S;
  p.jblocks = pl.jblocks;
  p.flags = sh->flags;
  p.scale = scale;
  if (fma) return cuda_status(launch_shrink_fma(p, pl.mode, pl.bn, pl.tiles, st));
  return cuda_status(launch_shrink_warp(p, pl.mode, pl.bn, pl.tiles, st));
}

int run_fused(const ig_shape* sh, const Plan& pl, const void* x, const void* A, const void* B,
              float scale, float* z, void* y, uint8_t* ws, cudaStream_t st) {
  FusedParams p;
  const bool fma = pl.path == IG_PATH_FMA;
  // FMA path: x rows gathered 4 at a time (box 256 x 1; the warp path loads
  // x into registers); A blocks are r rows high
  const uint32_t kbox = fma ? kShrinkKB : 64;
  const int swz = fma ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  int rc = IG_OK;
  if (fma) {
    rc = encode_map_2d(&p.tm_x, x, (uint64_t)sh->M, (uint64_t)sh->K, (uint64_t)sh->K * 2,
                       kShrinkKB, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != IG_OK) return rc;
  }
  rc = encode_map_2d(&p.tm_a, A, (uint64_t)sh->num_adapters * sh->slices * sh->r,
                     (uint64_t)sh->K, (uint64_t)sh->K * 2, kbox, (uint32_t)sh->r, swz);
  if (rc != IG_OK) return rc;
  p.has_a3 = !fma && sh->K % 64 == 0 && pl.Ks % 64 == 0;
  if (p.has_a3) {
    rc = encode_map_a3(&p.tm_a3, A, (uint64_t)sh->num_adapters * sh->slices * sh->r,
                       (uint64_t)sh->K, (uint32_t)sh->r);
    if (rc != IG_OK) return rc;
  }
  // B as rows of 64 elements (64 / r output columns x r ranks), 128-byte
  // swizzled boxes of b_box_rows rows
  p.b_box_rows = fma ? fused_fma_b_box_rows(pl.bn, pl.Ks, sh->N, pl.S)
                     : fused_b_box_rows(pl.bn, pl.Ks, sh->N, pl.S);
  rc = encode_map_2d(&p.tm_b, B, (uint64_t)sh->num_adapters * sh->slices * sh->N * sh->r / 64,
                     64, 128, 64, (uint32_t)p.b_box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != IG_OK) return rc;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.A = static_cast<const __nv_bfloat16*>(A);
  p.B = static_cast<const __nv_bfloat16*>(B);
  p.tiles = reinterpret_cast<const int32_t*>(ws + pl.off_tiles);
  p.z = z;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.M = sh->M;
  p.K = sh->K;
  p.N = sh->N;
  p.Ks = pl.Ks;
  p.slices = sh->slices;
  p.L = sh->num_adapters;
  p.S = pl.S;
  p.flags = sh->flags;
  p.scale = scale;
  if (fma) return cuda_status(launch_fused_fma(p, pl.bn, pl.tiles, st));
  return cuda_status(launch_fused_warp(p, pl.bn, pl.tiles, st));
}

// zt: the Z operand the shrink wrote (lora_apply), or null: built from z
int run_expand(const ig_shape* sh, const Plan& pl, const float* z, const void* B, void* y,
               uint8_t* ws, cudaStream_t st, const uint8_t* zt = nullptr) {
  if (pl.path == IG_PATH_MMA) return run_expand_mma(sh, pl, z, B, y, ws, st, zt);
  ExpandParams p;
  if (pl.path != IG_PATH_FMA) {   // the FMA expand copies B with 1-D bulk copies
    int rc = encode_map_2d(&p.tm_b, B,
                           (uint64_t)sh->num_adapters * sh->slices * sh->N * sh->r / 64, 64, 128,
                           64, (uint32_t)expand_warp_box_rows((int)sh->r, sh->N),
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != IG_OK) return rc;
  }
  p.z = z;
  p.B = static_cast<const __nv_bfloat16*>(B);
  p.tiles = reinterpret_cast<const int32_t*>(ws + pl.off_tiles);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.M = sh->M;
  p.N = sh->N;
  p.r = sh->r;
  p.slices = sh->slices;
  p.L = sh->num_adapters;
  p.ntiles = pl.ntiles;
  p.flags = sh->flags;
  if (pl.path == IG_PATH_FMA) return cuda_status(launch_expand_fma(p, pl.tiles, st));
  return cuda_status(launch_expand_warp(p, pl.tiles, st));
}

}  // namespace

// Workspace bytes lora_shrink itself touches: everything before the expand's
// Z operand, which only lora_apply writes. 0 for an invalid shape.
size_t shrink_ws_bytes(const ig_shape* sh) {
  Plan pl;
  if (make_plan(sh, &pl) != IG_OK) return 0;
  return pl.zt_bytes ? pl.off_zt : pl.total;
}

// lora_shrink with the workspace checked against shrink_ws_bytes when
// `full` is false (the built-in scratch of lora_shrink_noalloc).
int lora_shrink_ws(const ig_shape* shape, const void* x, const void* A_stack,
                   const int32_t* adapter_idx, float scale, float* z, void* ws,
                   size_t ws_bytes, void* stream, bool full) {
  Plan pl;
  int rc = make_plan(shape, &pl);
  if (rc != IG_OK) return rc;
  if (shape->M == 0) return IG_OK;
  rc = check_ws(pl, ws, ws_bytes);
  if (rc == IG_ERR_WS_SMALL && !full && ws_bytes >= shrink_ws_bytes(shape)) rc = IG_OK;
  if (rc != IG_OK) return rc;
  if (!x || !A_stack || !z) return IG_ERR_ARG;
  if (!aligned16(x) || !aligned16(A_stack) || !aligned16(z) ||
      (adapter_idx && !aligned16(adapter_idx)))
    return IG_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (adapter_idx) {
    rc = run_map(shape, pl, adapter_idx, w, st);
    if (rc != IG_OK) return rc;
  }
  return run_shrink(shape, pl, x, A_stack, scale, z, w, st);
}

}  // namespace ig

using namespace ig;

extern "C" {

const char* ig_version(void) { return "invariant_gemm 0.1 (sm_103a)"; }

const char* ig_status_string(int s) {
  switch (s) {
    case IG_OK: return "ok";
    case IG_ERR_ARG: return "invalid argument (null pointer or enum value)";
    case IG_ERR_SHAPE: return "invalid shape";
    case IG_ERR_ALIGN: return "pointer not 16-byte aligned";
    case IG_ERR_WS_SMALL: return "workspace too small";
    case IG_ERR_CUDA: return "CUDA runtime error";
    case IG_ERR_WS_CORRUPT: return "completion counter corrupt";
    case IG_ERR_ADAPTER_RANGE: return "adapter index out of range";
    case IG_ERR_TIMEOUT: return "bounded device wait expired";
    case IG_ERR_UNSUPPORTED: return "unsupported by this build";
    default: return "unknown status";
  }
}

size_t ig_workspace_bytes(const ig_shape* shape) {
  Plan pl;
  if (make_plan(shape, &pl) != IG_OK) return 0;
  return pl.total;
}

int ig_plan_query(const ig_shape* shape, ig_plan_info* out) {
  if (!out) return IG_ERR_ARG;
  Plan pl;
  int rc = make_plan(shape, &pl);
  if (rc != IG_OK) return rc;
  memset(out, 0, sizeof(*out));
  out->path = pl.path;
  out->split_k = pl.S;
  out->k_split = pl.Ks;
  out->shrink_bm = pl.tile_rows;
  out->shrink_bn = pl.bn;
  out->expand_bm = pl.tile_rows;
  out->expand_bn = pl.path == IG_PATH_MMA ? kMmaExpandCols : kExpandBN;
  out->shrink_tiles_max = pl.tiles;
  out->shrink_ctas_max = pl.tiles * (shape->slices / pl.stack) * pl.jblocks * pl.S;
  out->workspace_bytes = (int64_t)pl.total;
  out->determinism_key = pl.key;
  out->apply_kernels = pl.fused ? 1 : 2;
  return IG_OK;
}

int ig_workspace_init(void* ws, size_t ws_bytes, const ig_shape* shape, void* stream) {
  Plan pl;
  int rc = make_plan(shape, &pl);
  if (rc != IG_OK) return rc;
  rc = check_ws(pl, ws, ws_bytes);
  if (rc != IG_OK) return rc;
  cudaError_t e = cudaMemsetAsync(ws, 0, kMapOffset, static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

int ig_map_tokens(const ig_shape* shape, const int32_t* adapter_idx, void* ws, size_t ws_bytes,
                  void* stream) {
  Plan pl;
  int rc = make_plan(shape, &pl);
  if (rc != IG_OK) return rc;
  if (shape->M == 0) return IG_OK;
  rc = check_ws(pl, ws, ws_bytes);
  if (rc != IG_OK) return rc;
  if (!adapter_idx) return IG_ERR_ARG;
  if (!aligned16(adapter_idx)) return IG_ERR_ALIGN;
  return run_map(shape, pl, adapter_idx, static_cast<uint8_t*>(ws),
                 static_cast<cudaStream_t>(stream));
}

int lora_shrink(const ig_shape* shape, const void* x, const void* A_stack,
                const int32_t* adapter_idx, float scale, float* z, void* ws, size_t ws_bytes,
                void* stream) {
  return lora_shrink_ws(shape, x, A_stack, adapter_idx, scale, z, ws, ws_bytes, stream, true);
}

int lora_expand(const ig_shape* shape, const float* z, const void* B_stack,
                const int32_t* adapter_idx, void* y, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  int rc = make_plan(shape, &pl);
  if (rc != IG_OK) return rc;
  if (shape->M == 0) return IG_OK;
  rc = check_ws(pl, ws, ws_bytes);
  if (rc != IG_OK) return rc;
  if (!z || !B_stack || !y) return IG_ERR_ARG;
  if (!aligned16(z) || !aligned16(B_stack) || !aligned16(y) ||
      (adapter_idx && !aligned16(adapter_idx)))
    return IG_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (adapter_idx) {
    rc = run_map(shape, pl, adapter_idx, w, st);
    if (rc != IG_OK) return rc;
  }
  return run_expand(shape, pl, z, B_stack, y, w, st);
}

int lora_apply(const ig_shape* shape, const void* x, void* y, const int32_t* adapter_idx,
               const void* A_stack, const void* B_stack, float scale, float* z, void* ws,
               size_t ws_bytes, void* stream) {
  Plan pl;
  int rc = make_plan(shape, &pl);
  if (rc != IG_OK) return rc;
  if (shape->M == 0) return IG_OK;
  rc = check_ws(pl, ws, ws_bytes);
  if (rc != IG_OK) return rc;
  if (!x || !y || !A_stack || !B_stack || !z) return IG_ERR_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(A_stack) || !aligned16(B_stack) ||
      !aligned16(z) || (adapter_idx && !aligned16(adapter_idx)))
    return IG_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (adapter_idx) {
    rc = run_map(shape, pl, adapter_idx, w, st);
    if (rc != IG_OK) return rc;
  }
  if (pl.fused) return run_fused(shape, pl, x, A_stack, B_stack, scale, z, y, w, st);
  uint8_t* zt = pl.zt_bytes ? w + pl.off_zt : nullptr;
  rc = run_shrink(shape, pl, x, A_stack, scale, z, w, st, zt);
  if (rc != IG_OK) return rc;
  return run_expand(shape, pl, z, B_stack, y, w, st, zt);
}

int ig_check_status(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return IG_ERR_ARG;
  if (ws_bytes < kMapOffset) return IG_ERR_WS_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return IG_ERR_CUDA;
  uint32_t status = 0;
  if (cudaMemcpy(&status, ws, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
    return IG_ERR_CUDA;
  if (status == 0) return IG_OK;
  // Clear the word; after a corrupt counter or an abandoned tile, zero the
  // counters too so that the workspace is usable again.
  size_t clear = (status & (kStatusCorrupt | kStatusTimeout)) ? kMapOffset : sizeof(uint32_t);
  if (cudaMemsetAsync(ws, 0, clear, st) != cudaSuccess) return IG_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return IG_ERR_CUDA;
  if (status & kStatusTimeout) return IG_ERR_TIMEOUT;
  if (status & kStatusCorrupt) return IG_ERR_WS_CORRUPT;
  return IG_ERR_ADAPTER_RANGE;
}

}  // extern "C"
