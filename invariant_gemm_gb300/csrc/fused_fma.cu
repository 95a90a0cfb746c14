// Fused decode LoRA layer on CUDA cores (IG_PATH_FMA): deterministic Split-K
// shrink and expand in one launch, with the S partition blocks of a tile
// forming one thread-block cluster.
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// sec. 4.3 / Algorithm 1 / Fig. 2: S blocks compute FP32 partials of one
// output tile, and the partials are summed in increasing partition order
// starting from FP32 zero, then multiplied by the scale. The pages keep the
// partials in global scratch and pick the block that finishes last with an
// integer counter, and they run the expand as a separate kernel; they name
// the extra launch as the cost of the earlier two-kernel design (sec. 4.3)
// and leave the expand to vLLM (Eq. 1). On GB300 the S blocks of a tile can
// be one cluster: each block sends its partial into slot s of every block's
// shared memory with asynchronous remote stores that count their bytes on
// the receiving block's mbarrier, so a block starts its combine as soon as
// the S partials have landed in its own shared memory, with no cluster-wide
// barrier on the way. Every block then sums the S partials in the same fixed
// order. No scratch, no counter, and the expand of the tile's rows follows
// in the same launch, each block taking 1/S of the output columns.
//
// Bit-for-bit the same results as the two-kernel path (shrink kernel with
// the counter protocol, then the expand kernel): the partials come from the
// same code (shrink_core.cuh), the combine adds them in the same order, and
// the expand keeps the same j order and single rounding.
//
// Block = r/4 warps; cluster = S blocks (rank s = K partition s); tile = up
// to 8 token rows of one adapter (tile-table entry) x all r rank columns
// (r = 8 or 16). Copies: the A block of each k-block by one tiled TMA copy,
// the token rows of x by row-gather TMA copies (4 rows each), the block's B
// column slice by tiled TMA copies of 128-byte rows (64/r columns x r ranks
// each, 128-byte swizzled so that the rows read by 8 neighbouring lanes sit
// in 8 distinct bank groups); the y values of a thread's first expand unit
// are loaded into registers right after griddep_wait, so they arrive while
// the shrink computes.
#include <type_traits>

#include "fma_core.cuh"

namespace ig {

namespace {

template <int BN>
struct FusedGeo {
  static constexpr int CU = 64 / BN;   // output columns per expand unit (128 bytes of B)
  static constexpr int CP = CU / 2;    // column pairs per unit
  static constexpr int TB = kTileRows * BN;   // partial values per block
};

struct FusedLayout {
  int nst;           // ring depth
  int cols;          // output columns per block (multiple of 8)
  int units;         // expand units per block (cols / CU), one 128-byte B row each
  int box_rows;      // B rows per TMA box (<= 256)
  int nbox;          // B boxes per block
  size_t ring_off, part_off, zd_off, b_off, bytes;   // from the 1024-aligned base
};

template <int BN>
__host__ __device__ inline FusedLayout fused_layout(int64_t Ks, int64_t N, int S) {
  using F = FusedGeo<BN>;
  FusedLayout L;
  const int nkb = (int)((Ks + kShrinkKB - 1) / kShrinkKB);
  L.nst = nkb < kShrinkStages ? nkb : kShrinkStages;
  L.cols = (((int)N + S - 1) / S + 7) / 8 * 8;   // N < 2^31: 32-bit division
  L.units = L.cols / F::CU;
  L.box_rows = L.units < 256 ? L.units : 256;
  L.nbox = (L.units + L.box_rows - 1) / L.box_rows;
  L.ring_off = 256;
  L.part_off = L.ring_off + (size_t)L.nst * FmaRing<BN>::kStageBytes;
  L.zd_off = L.part_off + (size_t)S * F::TB * 4;
  L.b_off = (L.zd_off + (size_t)F::TB * 8 + 1023) / 1024 * 1024;
  L.bytes = L.b_off + (size_t)L.nbox * L.box_rows * 128;
  return L;
}

template <int BN>
__global__ void __launch_bounds__(FmaGeo<BN>::THREADS)
    fused_fma_kernel(const __grid_constant__ FusedParams p) {
  constexpr int kThreads = FmaGeo<BN>::THREADS;
  using F = FusedGeo<BN>;
  constexpr int CU = F::CU, CP = F::CP, TB = F::TB;
  using YV = typename std::conditional<CU == 4, uint2, uint4>::type;   // CU bf16 of y
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const FusedLayout lay = fused_layout<BN>(p.Ks, p.N, p.S);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);            // ring bars [0, 4)
  uint64_t* bar_b = bars + kShrinkStages;                        // B copies
  uint64_t* bar_part = bars + kShrinkStages + 1;                 // incoming partials
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 64);        // tile entry
  float* part = reinterpret_cast<float*>(smem + lay.part_off);   // [S][8][BN]
  float2* zd = reinterpret_cast<float2*>(smem + lay.zd_off);     // [8][BN] (z, z)
  uint8_t* sB = smem + lay.b_off;                                // [units][128 B], swizzled

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;
  const int s = (int)cluster_rank();
  uint32_t cl = blockIdx.x / (uint32_t)S;
  const int sl = (int)next_digit(cl, (uint32_t)p.slices);
  const int64_t t = cl;

  if (tid < kTileInts) ent_s[tid] = p.tiles[t * kTileInts + tid];
  if (tid == 0) {
    prefetch_tensormap(&p.tm_x);
    prefetch_tensormap(&p.tm_a);
    prefetch_tensormap(&p.tm_b);
    for (int i = 0; i < lay.nst; ++i) mbar_init(&bars[i], 1);
    mbar_init(bar_b, 1);
    mbar_init(bar_part, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_part, (uint32_t)(S * TB * 4));
  }
  __syncthreads();
  const int g = ent_s[0];
  const int nrows = ent_s[1];
  const int32_t* rows_s = ent_s + 4;
  const int64_t M = p.M, N = p.N, K = p.K;
  const int r = BN;
  if (nrows <= 0) return;  // the whole cluster shares the tile: all exit

  if (g == p.L) {
    // tokens without an adapter: zero Z rows, y untouched
    griddep_wait();
    griddep_launch();
    if (s == 0)
      for (int i = tid; i < nrows * r; i += kThreads)
        p.z[((int64_t)sl * M + rows_s[i / r]) * r + i % r] = 0.0f;
    return;
  }
  // every block of the cluster has initialised and armed its mbarriers once
  // the matching cluster_wait returns
  cluster_arrive_relaxed();

  // this block's output columns [c0, c0 + ncols) of slice sl
  const int64_t c0 = (int64_t)s * lay.cols;
  const int ncols = (int)max((int64_t)0, min((int64_t)lay.cols, N - c0));
  const int nunits = ncols / CU;
  const bool early_w = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;

  FmaArgs pa;
  pa.x = p.x + (int64_t)s * p.Ks;
  pa.A = p.A + ((int64_t)g * p.slices + sl) * r * K + (int64_t)s * p.Ks;
  pa.rows = rows_s;
  pa.status = p.status;
  pa.K = K;
  pa.Ks = p.Ks;
  pa.nrows = nrows;
  pa.tm_x = &p.tm_x;
  pa.tm_a = &p.tm_a;
  pa.k0 = (int)((int64_t)s * p.Ks);
  pa.a_row = (int)(((int64_t)g * p.slices + sl) * r);
  FmaRing<BN> ring;
  ring.stages = smem + lay.ring_off;
  ring.bars = bars;
  ring.nst = lay.nst;
  ring.nkb = (int)((p.Ks + kShrinkKB - 1) / kShrinkKB);
  const int first = min(ring.nkb, lay.nst);

  // B rows of this block: 128-byte row u holds columns c0 + CU*u .. + CU-1
  const int b_row0 = (int)((((int64_t)g * p.slices + sl) * N + c0) / CU);
  auto issue_b = [&]() {
    if (lane == 0 && ncols > 0)
      for (int bi = 0; bi < lay.nbox; ++bi)
        tma_load_2d(sB + (size_t)bi * lay.box_rows * 128, &p.tm_b, 0,
                    b_row0 + bi * lay.box_rows, bar_b);
  };
  const int64_t ldy = (int64_t)p.slices * N;

  if (warp == 0) {
    if (lane == 0)
      mbar_arrive_expect_tx(bar_b, ncols > 0 ? (uint32_t)(lay.nbox * lay.box_rows * 128) : 0u);
    __syncwarp();
    for (int b = 0; b < first; ++b) {
      ring.expect(pa, b);
      if (early_w) ring.issue_a(pa, b);
    }
    if (early_w) issue_b();
  }
  griddep_wait();
  griddep_launch();
  if (warp == 0) {
    for (int b = 0; b < first; ++b) {
      if (!early_w) ring.issue_a(pa, b);
      ring.issue_x(pa, b);
    }
    if (!early_w) issue_b();
  }

  // y of the thread's first expand unit (all tile rows), loaded now so that
  // it arrives during the shrink
  YV ypre[kTileRows];
  if (tid < nunits) {
#pragma unroll
    for (int rr = 0; rr < kTileRows; ++rr)
      if (rr < nrows)
        ypre[rr] = *reinterpret_cast<const YV*>(p.y + (int64_t)rows_s[rr] * ldy +
                                                (int64_t)sl * N + c0 + CU * tid);
  }

  float v;
  const bool ok = ring.run(pa, v);

  // Send this block's partial P_s to slot s of every block of the cluster
  // (its own included). Every block sends on every path (zeros after a
  // failed copy), so every block receives exactly S * TB * 4 bytes.
  cluster_wait();
  {
    const int o = (lane / 4) * BN + warp * FmaGeo<BN>::JPW + lane % 4;
    const float pv = ok ? v : 0.0f;
    for (int q = 0; q < S; ++q)
      st_async_f32(map_rank(part + s * TB + o, (uint32_t)q), pv, map_rank(bar_part, (uint32_t)q));
  }
  // The wait outlasts any sender's own bounded waits, so a block never
  // leaves while a partial is still on its way to it.
  const bool got = mbar_wait_bounded(bar_part, 0, p.status, 1ll << 36);

  // Combine (Algorithm 1 order): total = 0; total += P_q for q = 0..S-1.
  for (int o = tid; o < nrows * BN; o += kThreads) {
    float total = 0.0f;
    for (int q = 0; q < S; ++q) total += part[q * TB + o];
    const float zv = total * p.scale;
    const float zb = (p.flags & IG_FLAG_Z_FP32) ? zv : bf16_round_f32(zv);
    zd[o] = make_float2(zb, zb);
    if (s == 0) p.z[((int64_t)sl * M + rows_s[o / BN]) * r + o % BN] = zv;
  }
  __syncthreads();   // zd complete

  // Expand this block's columns: y = bf16_rn(f32(y) + sum_j zb_j B_nj), the
  // j sum a chain of FMAs in increasing j (two columns per f32x2 FMA). A unit
  // is CU consecutive columns for all rows of the tile: its B values are
  // converted once and used for every row. Every element is computed by one
  // thread, so the split does not change any result.
  const bool copies_ok = mbar_wait_bounded(bar_b, 0, p.status);
  if (copies_ok && got) {
    for (int u = tid, k = 0; u < nunits; u += kThreads, ++k) {
      float2 bp[CP][BN];   // (B[c][j], B[c+1][j]) for column pair c = 2cp
      {
        const uint8_t* row = sB + (size_t)u * 128;
        const int sw = u & 7;   // 128-byte swizzle: 16-byte chunk i sits at i ^ (row % 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 w = *reinterpret_cast<const uint4*>(row + ((i ^ sw) << 4));
          float f[8];
          unpack8(w, f);
          const int cc = (8 * i) / BN, jb = (8 * i) % BN;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (cc % 2 == 0) bp[cc / 2][jb + e].x = f[e];
            else bp[cc / 2][jb + e].y = f[e];
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < kTileRows; ++rr) {
        if (rr >= nrows) break;
        __nv_bfloat16* yp = p.y + (int64_t)rows_s[rr] * ldy + (int64_t)sl * N + c0 + CU * u;
        const YV yv = k == 0 ? ypre[rr] : *reinterpret_cast<const YV*>(yp);
        float2 acc[CP];
#pragma unroll
        for (int cp = 0; cp < CP; ++cp) acc[cp] = make_float2(0.0f, 0.0f);
        const float4* zr = reinterpret_cast<const float4*>(zd + rr * BN);
#pragma unroll
        for (int jj = 0; jj < BN / 2; ++jj) {
          const float4 z2 = zr[jj];   // (z_j, z_j, z_j+1, z_j+1)
#pragma unroll
          for (int cp = 0; cp < CP; ++cp)
            acc[cp] = __ffma2_rn(make_float2(z2.x, z2.y), bp[cp][2 * jj], acc[cp]);
#pragma unroll
          for (int cp = 0; cp < CP; ++cp)
            acc[cp] = __ffma2_rn(make_float2(z2.z, z2.w), bp[cp][2 * jj + 1], acc[cp]);
        }
        const uint32_t* yw = reinterpret_cast<const uint32_t*>(&yv);
        YV out;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
        for (int cp = 0; cp < CP; ++cp)
          ow[cp] = f32x2_to_bf16x2_bits(bf16lo(yw[cp]) + acc[cp].x, bf16hi(yw[cp]) + acc[cp].y);
        *reinterpret_cast<YV*>(yp) = out;
      }
    }
  }
  // a copy that never completed: wait for it once more (bounded) before the
  // block's shared memory goes away
  if (!copies_ok) mbar_wait_bounded(bar_b, 0, p.status);
}

}  // namespace

size_t fused_fma_smem_bytes(int bn, int64_t Ks, int64_t N, int S) {
  // + 1024: the kernel aligns its base to 1024 bytes (128-byte swizzle atoms)
  return 1024 + (bn == 16 ? fused_layout<16>(Ks, N, S).bytes : fused_layout<8>(Ks, N, S).bytes);
}

int fused_fma_b_box_rows(int bn, int64_t Ks, int64_t N, int S) {
  return bn == 16 ? fused_layout<16>(Ks, N, S).box_rows : fused_layout<8>(Ks, N, S).box_rows;
}

cudaError_t launch_fused_fma(const FusedParams& p, int bn, int64_t tiles_max, cudaStream_t st) {
  const int64_t grid = tiles_max * p.slices * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = fused_fma_smem_bytes(bn, p.Ks, p.N, p.S);
  void (*kern)(FusedParams) = bn == 16 ? fused_fma_kernel<16> : fused_fma_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  if (p.S > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(bn == 16 ? FmaGeo<16>::THREADS : FmaGeo<8>::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ig
