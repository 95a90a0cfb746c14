// Fused decode LoRA layer: deterministic Split-K shrink and expand in one
// launch, with the S partition blocks of a tile forming one thread-block
// cluster.
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// sec. 4.3 / Algorithm 1 / Fig. 2: S blocks compute FP32 partials of one
// output tile, and the partials are summed in increasing partition order
// starting from FP32 zero, then multiplied by the scale. The pages keep the
// partials in global scratch and pick the block that finishes last with an
// integer counter, and they run the expand as a separate kernel; they name
// the extra launch as the cost of the earlier two-kernel design (sec. 4.3)
// and leave the expand to vLLM (Eq. 1). On GB300 the S blocks of a tile can
// be one cluster: each block stores its partial into every block's shared
// memory (distributed shared memory), one cluster barrier publishes them,
// and every block sums the S partials in the same fixed order. No scratch, no
// counter, and the expand of the tile's rows follows in the same launch,
// each block taking 1/S of the output columns.
//
// Bit-for-bit the same results as the two-kernel path (shrink kernel with
// the counter protocol, then the expand kernel): the partials come from the
// same code (shrink_core.cuh), the combine adds them in the same order, and
// the expand keeps the same j order and single rounding.
//
// Block = r/4 warps; cluster = S blocks (rank s = K
// partition s); tile = up to 8 token rows of one adapter (tile-table entry)
// x all r rank columns (r = 8 or 16). Copies: the A block of each k-block by
// one tiled TMA copy, the token rows of x by row-gather TMA copies (4 rows
// each), the block's B column slice (contiguous in B_stack) by one bulk copy;
// the y values a thread will update are loaded into registers right after
// griddep_wait, so they arrive while the shrink computes.
#include "shrink_core.cuh"

namespace ig {

namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store into the same offset of block `rank`'s shared memory.
__device__ __forceinline__ void st_dsmem_f32(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

struct FusedLayout {
  int nst;           // ring depth
  int cols;          // output columns per block (multiple of 8)
  size_t ring_off, part_off, zs_off, b_off, bytes;
};

template <int BN>
struct ZsStride {
  static constexpr int v = BN + 4;  // padded row: 8 rows hit 8 distinct bank groups
};

template <int BN>
__host__ __device__ inline FusedLayout fused_layout(int64_t Ks, int64_t N, int S) {
  FusedLayout L;
  const int nkb = (int)((Ks + kShrinkKB - 1) / kShrinkKB);
  L.nst = nkb < kShrinkStages ? nkb : kShrinkStages;
  L.cols = (int)(((N + S - 1) / S + 7) / 8 * 8);
  L.ring_off = 256;
  L.part_off = L.ring_off + (size_t)L.nst * PartialRing<BN>::kStageBytes;
  L.zs_off = L.part_off + (size_t)S * kTileRows * BN * 4;
  L.b_off = L.zs_off + kTileRows * ZsStride<BN>::v * 4;
  L.bytes = L.b_off + (size_t)L.cols * BN * 2;
  return L;
}

template <int BN>
__global__ void __launch_bounds__(ShrinkGeo<BN>::THREADS)
    fused_fma_kernel(const __grid_constant__ FusedParams p) {
  constexpr int kThreads = ShrinkGeo<BN>::THREADS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const FusedLayout lay = fused_layout<BN>(p.Ks, p.N, p.S);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);            // ring bars [0, 4)
  uint64_t* bar_by = bars + kShrinkStages;                       // B and y copies
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 64);        // tile entry
  float* part = reinterpret_cast<float*>(smem + lay.part_off);   // [S][rows][BN]
  float* zs = reinterpret_cast<float*>(smem + lay.zs_off);       // [16][BN + 4]
  uint8_t* sB = smem + lay.b_off;                                // [cols][BN] bf16

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;
  const int s = (int)cluster_rank();
  const int64_t cl = blockIdx.x / S;
  const int sl = (int)(cl % p.slices);
  const int64_t t = cl / p.slices;

  if (tid < kTileInts) ent_s[tid] = p.tiles[t * kTileInts + tid];
  if (tid == 0) {
    for (int i = 0; i < lay.nst; ++i) mbar_init(&bars[i], 1);
    mbar_init(bar_by, 1);
    fence_mbar_init();
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

  // this block's output columns [c0, c0 + ncols) of slice sl
  const int64_t c0 = (int64_t)s * lay.cols;
  const int ncols = (int)max((int64_t)0, min((int64_t)lay.cols, N - c0));
  const int groups = ncols / 8;
  constexpr int ZS = ZsStride<BN>::v;
  const bool early_w = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;

  PartialArgs pa;
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
  PartialRing<BN> ring;
  ring.stages = smem + lay.ring_off;
  ring.bars = bars;
  ring.nst = lay.nst;
  ring.nkb = (int)((p.Ks + kShrinkKB - 1) / kShrinkKB);
  const int first = min(ring.nkb, lay.nst);

  const __nv_bfloat16* Bsrc = p.B + (((int64_t)g * p.slices + sl) * N + c0) * r;
  const uint32_t b_bytes = (uint32_t)ncols * r * 2;
  const int64_t ldy = (int64_t)p.slices * N;

  if (warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(bar_by, b_bytes);
    __syncwarp();
    for (int b = 0; b < first; ++b) {
      ring.expect(pa, b);
      if (early_w) ring.issue_a(pa, b);
    }
    if (early_w && lane == 0 && b_bytes) bulk_g2s(sB, Bsrc, b_bytes, bar_by);
  }
  griddep_wait();
  griddep_launch();
  if (warp == 0) {
    for (int b = 0; b < first; ++b) {
      if (!early_w) ring.issue_a(pa, b);
      ring.issue_x(pa, b);
    }
    if (!early_w && lane == 0 && b_bytes) bulk_g2s(sB, Bsrc, b_bytes, bar_by);
  }

  // Expand work units: (pair of rows rp, 8-column group q), rp varying
  // fastest so that the 8 lanes of a shared-memory phase read the same B
  // group (broadcast) and rows of Z that sit in distinct banks. The y values
  // of a thread's first two units are loaded now and arrive during the
  // shrink.
  const int pairs = (nrows + 1) / 2;
  const int units = pairs * groups;
  uint4 ypre[2][2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int u = tid + k * kThreads;
    if (u < units) {
      const int rp = u % pairs, q = u / pairs;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = min(2 * rp + i, nrows - 1);
        ypre[k][i] = *reinterpret_cast<const uint4*>(p.y + (int64_t)rows_s[row] * ldy +
                                                     (int64_t)sl * N + c0 + q * 8);
      }
    }
  }

  // This block's partial P_s goes to slot s of every block of the cluster
  // (its own included), so that after one cluster barrier each block sums
  // the S partials from its own shared memory.
  float v;
  const bool ok = ring.run(pa, v);
  {
    constexpr int TB = kTileRows * BN;
    const int o = (lane / 4) * BN + warp * ShrinkGeo<BN>::JPW + lane % 4;
    for (int q = 0; q < S; ++q) st_dsmem_f32(part + s * TB + o, (uint32_t)q, ok ? v : 0.0f);
  }

  // Every block of the cluster reaches the cluster barrier on every path;
  // after it no block touches another block's shared memory.
  cluster_sync();

  // Combine (Algorithm 1 order): total = 0; total += P_q for q = 0..S-1.
  for (int o = tid; o < nrows * BN; o += kThreads) {
    float total = 0.0f;
    for (int q = 0; q < S; ++q) total += part[q * kTileRows * BN + o];
    const float zv = total * p.scale;
    zs[(o / BN) * ZS + o % BN] = (p.flags & IG_FLAG_Z_FP32) ? zv : bf16_round_f32(zv);
    if (s == 0) p.z[((int64_t)sl * M + rows_s[o / BN]) * r + o % BN] = zv;
  }
  __syncthreads();   // zs complete

  // Expand this block's columns: y = bf16_rn(f32(y) + sum_j zb_j B_nj), the
  // j sum a chain of FMAs in increasing j (two columns per f32x2 FMA). Work
  // units are (pair of rows, 8-column group), spread over all threads of
  // the block; every element is computed by one thread, so the split does
  // not change any result.
  const bool copies_ok = mbar_wait_bounded(bar_by, 0, p.status);
  if (copies_ok) {
    for (int k = 0; tid + k * kThreads < units; ++k) {
      const int u = tid + k * kThreads;
      const int rp = u % pairs, q = u / pairs;
      const int ra = 2 * rp, rb = 2 * rp + 1;
      const bool has_b = rb < nrows;
      uint4 yv[2];
      if (k == 0) {
        yv[0] = ypre[0][0];
        yv[1] = ypre[0][1];
      } else if (k == 1) {
        yv[0] = ypre[1][0];
        yv[1] = ypre[1][1];
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          yv[i] = *reinterpret_cast<const uint4*>(p.y + (int64_t)rows_s[min(ra + i, nrows - 1)] *
                                                  ldy + (int64_t)sl * N + c0 + q * 8);
      }
      float2 acc[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) acc[i][cp] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int h = 0; h < BN / 8; ++h) {
        float za[8], zb[8];
        {
          const float4 a0 = *reinterpret_cast<const float4*>(zs + ra * ZS + 8 * h);
          const float4 a1 = *reinterpret_cast<const float4*>(zs + ra * ZS + 8 * h + 4);
          const float4 b0 = *reinterpret_cast<const float4*>(zs + (has_b ? rb : ra) * ZS + 8 * h);
          const float4 b1 =
              *reinterpret_cast<const float4*>(zs + (has_b ? rb : ra) * ZS + 8 * h + 4);
          za[0] = a0.x; za[1] = a0.y; za[2] = a0.z; za[3] = a0.w;
          za[4] = a1.x; za[5] = a1.y; za[6] = a1.z; za[7] = a1.w;
          zb[0] = b0.x; zb[1] = b0.y; zb[2] = b0.z; zb[3] = b0.w;
          zb[4] = b1.x; zb[5] = b1.y; zb[6] = b1.z; zb[7] = b1.w;
        }
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
          const uint4 u0 =
              *reinterpret_cast<const uint4*>(sB + ((q * 8 + 2 * cp) * r + 8 * h) * 2);
          const uint4 u1 =
              *reinterpret_cast<const uint4*>(sB + ((q * 8 + 2 * cp + 1) * r + 8 * h) * 2);
          float b0[8], b1[8];
          unpack8(u0, b0);
          unpack8(u1, b1);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 bb = make_float2(b0[e], b1[e]);
            acc[0][cp] = __ffma2_rn(make_float2(za[e], za[e]), bb, acc[0][cp]);
            acc[1][cp] = __ffma2_rn(make_float2(zb[e], zb[e]), bb, acc[1][cp]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = ra + i;
        if (row >= nrows) break;
        float yf[8];
        unpack8(yv[i], yf);
        uint32_t o[8];
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
          o[2 * cp] = f32_to_bf16_bits(yf[2 * cp] + acc[i][cp].x);
          o[2 * cp + 1] = f32_to_bf16_bits(yf[2 * cp + 1] + acc[i][cp].y);
        }
        uint4 w;
        w.x = o[0] | (o[1] << 16);
        w.y = o[2] | (o[3] << 16);
        w.z = o[4] | (o[5] << 16);
        w.w = o[6] | (o[7] << 16);
        *reinterpret_cast<uint4*>(p.y + (int64_t)rows_s[row] * ldy + (int64_t)sl * N + c0 +
                                  q * 8) = w;
      }
    }
  }
  // a copy that never completed: wait for it once more (bounded) before the
  // block's shared memory goes away
  if (!copies_ok) mbar_wait_bounded(bar_by, 0, p.status);
}

}  // namespace

size_t fused_smem_bytes(int bn, int64_t Ks, int64_t N, int S) {
  return bn == 16 ? fused_layout<16>(Ks, N, S).bytes : fused_layout<8>(Ks, N, S).bytes;
}

cudaError_t launch_fused_fma(const FusedParams& p, int bn, int64_t tiles_max, cudaStream_t st) {
  const int64_t grid = tiles_max * p.slices * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = fused_smem_bytes(bn, p.Ks, p.N, p.S);
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
  cfg.blockDim = dim3(bn == 16 ? ShrinkGeo<16>::THREADS : ShrinkGeo<8>::THREADS);
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
