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
// the expand keeps the same j order and single rounding (warp_mma.cuh).
//
// Block = r/4 warps; cluster = S blocks (rank s = K partition s); tile = up
// to 8 token rows of one adapter (tile-table entry) x all r rank columns
// (r = 8 or 16). Copies: the A rows of the partition by TMA (128-byte
// swizzled, one 3-D copy per 256 elements), and the block's B column slice
// by tiled TMA copies of 128-byte rows (64/r columns x r ranks each), both
// issued before griddep_wait when the weights are static (and then, for a
// partition of at most two k-blocks, this lane's A chunks are read into
// registers before the wait too); x and y go straight from global memory
// into registers right after the wait, x in 16-byte and y in 8-byte loads
// (L2 was asked for the block's x and y rows before it), so that y arrives
// while the shrink computes. Both the shrink partial and the expand run on
// the warp-level tensor cores.
#include "shrink_core.cuh"

namespace ig {

namespace {


template <int BN>
struct FusedGeo {
  static constexpr int CU = 64 / BN;   // output columns per 128-byte B row
  static constexpr int TB = kTileRows * BN;   // partial values per block
};

struct FusedLayout {
  int nst;           // ring depth
  int cols;          // output columns per block (multiple of 8)
  int box_rows;      // B rows (128 bytes) per TMA box (<= 256)
  int nbox;          // B boxes per block
  size_t ring_off, part_off, red_off, zb_off, b_off, bytes;   // from the 1024-aligned base
};

template <int BN>
__host__ __device__ inline FusedLayout fused_layout(int64_t Ks, int64_t N, int S) {
  using F = FusedGeo<BN>;
  FusedLayout L;
  const int nkb = (int)((Ks + kShrinkKB - 1) / kShrinkKB);
  L.nst = nkb < kShrinkStages ? nkb : kShrinkStages;
  L.cols = (((int)N + S - 1) / S + 7) / 8 * 8;   // N < 2^31: 32-bit division
  const int brows = L.cols / F::CU;
  L.box_rows = brows < 256 ? brows : 256;
  L.nbox = (brows + L.box_rows - 1) / L.box_rows;
  L.ring_off = 1024;
  L.part_off = L.ring_off + (size_t)L.nst * PartialRing<BN>::kStageBytes;
  L.red_off = L.part_off + (size_t)S * F::TB * 4;
  L.zb_off = L.red_off + PartialRing<BN>::kRedBytes;
  L.b_off = (L.zb_off + (size_t)3 * F::TB * 2 + 1023) / 1024 * 1024;
  // room for whole 32-column groups (the rows past the block's columns are
  // read by the expand's MMAs of a partial last group, never used)
  const int rows_alloc = (L.cols + 31) / 32 * 32 / F::CU;
  const int rows_loaded = L.nbox * L.box_rows;
  L.bytes = L.b_off + (size_t)(rows_loaded > rows_alloc ? rows_loaded : rows_alloc) * 128;
  return L;
}

// At least four blocks per SM (at most 128 registers a thread for BN = 16),
// so that the next layer's blocks fit beside this layer's and run their
// prologue early.
template <int BN>
__global__ void __launch_bounds__(ShrinkGeo<BN>::THREADS, 4)
    fused_warp_kernel(const __grid_constant__ FusedParams p) {
  // the next kernel may be scheduled now: it reads nothing of ours before
  // its own griddep_wait(), which waits for this grid to complete
  griddep_launch();
  constexpr int kThreads = ShrinkGeo<BN>::THREADS;
  constexpr int W = ShrinkGeo<BN>::WARPS;
  constexpr int TB = FusedGeo<BN>::TB;
  constexpr int CU = FusedGeo<BN>::CU;
  constexpr int kGB = 4;   // 32-column groups per warp whose y is loaded together
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const FusedLayout lay = fused_layout<BN>(p.Ks, p.N, p.S);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);            // ring bars [0, 4)
  uint64_t* bar_b = bars + kShrinkStages;                        // B copies
  uint64_t* bar_part = bars + kShrinkStages + 1;                 // incoming partials
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 64);        // tile entry
  float* part = reinterpret_cast<float*>(smem + lay.part_off);   // [S][8][BN]
  float* red = reinterpret_cast<float*>(smem + lay.red_off);     // warp sums
  uint16_t* zb = reinterpret_cast<uint16_t*>(smem + lay.zb_off); // [3][8][BN] bf16 parts of Z
  uint8_t* sB = smem + lay.b_off;                                // 128-byte rows, swizzled

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;
  const int s = (int)cluster_rank();
  uint32_t cl = blockIdx.x / (uint32_t)S;
  const int sl = (int)next_digit(cl, (uint32_t)p.slices);
  const int64_t t = cl;

  if (tid < kTileInts) ent_s[tid] = p.tiles[t * kTileInts + tid];
  if (tid == 0) {
    prefetch_tensormap(p.has_a3 ? &p.tm_a3 : &p.tm_a);
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
  const int64_t M = p.M, N = p.N;
  const int r = BN;
  if (nrows <= 0) return;  // the whole cluster shares the tile: all exit

  if (g == p.L) {
    // tokens without an adapter: zero Z rows, y untouched
    griddep_wait();
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
  const bool early_w = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;

  PartialArgs pa;
  pa.rows = rows_s;
  pa.status = p.status;
  pa.x = p.x;
  pa.K = p.K;
  pa.Ks = (int)p.Ks;
  pa.nrows = nrows;
  pa.tm_a = &p.tm_a;
  pa.tm_a3 = p.has_a3 ? &p.tm_a3 : nullptr;
  pa.k0 = (int)((int64_t)s * p.Ks);
  pa.a_row = (int)(((int64_t)g * p.slices + sl) * r);
  pa.first_budget = first_copy_budget(p.flags);
  PartialRing<BN> ring;
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

  if (warp == 0) {
    if (lane == 0)
      mbar_arrive_expect_tx(bar_b, ncols > 0 ? (uint32_t)(lay.nbox * lay.box_rows * 128) : 0u);
    __syncwarp();
    for (int b = 0; b < first; ++b) {
      ring.expect(pa, b);
      if (early_w) ring.issue_a(pa, b);
    }
    if (early_w) issue_b();
  } else if (warp == 1) {
    // Ask L2 for this block's x and y rows now. A prefetch has no effect on
    // the values read: the loads after griddep_wait() see the previous
    // kernel's writes, L2 being where they land.
    if (lane < nrows)
      bulk_prefetch_l2(p.x + (int64_t)rows_s[lane] * p.K + pa.k0, (uint32_t)(p.Ks * 2));
    else if (lane >= 8 && lane - 8 < nrows && ncols > 0)
      bulk_prefetch_l2(p.y + (int64_t)rows_s[lane - 8] * ((int64_t)p.slices * N) +
                           (int64_t)sl * N + c0,
                       (uint32_t)(ncols * 2));
  }
  // Everything that depends only on the token map is computed before the
  // wait: this lane's x row, and the expand geometry. The block's columns
  // form groups of 32 (the last one may be partial); warp w takes the groups
  // w, w + W, ...; lane 4g + t updates columns 4g .. 4g+3 of each in the rows
  // of tokens 2t and 2t + 1 (warp_mma.cuh). The y of its first kGB groups is
  // loaded right after the x loads and arrives during the shrink.
  const __nv_bfloat16* xrow = ring.x_row(pa);
  uint32_t boff[2];
  ExpandFrag<BN>::lane_offsets(lane, warp & 1, boff);
  const int gq = lane >> 2, tq = lane & 3;
  const bool has0 = 2 * tq < nrows, has1 = 2 * tq + 1 < nrows;
  const int64_t ld = (int64_t)p.slices * N;
  __nv_bfloat16* yrow0 = p.y + (int64_t)rows_s[min(2 * tq, nrows - 1)] * ld + (int64_t)sl * N +
                         c0 + 4 * gq;
  __nv_bfloat16* yrow1 = p.y + (int64_t)rows_s[min(2 * tq + 1, nrows - 1)] * ld +
                         (int64_t)sl * N + c0 + 4 * gq;
  const int ngroups = (ncols + 31) / 32;
  auto col_ok = [&](int grp) { return grp < ngroups && 32 * grp + 4 * gq < ncols; };
  auto load_y = [&](int h, uint2 (&yq)[kGB][2]) {
#pragma unroll
    for (int i = 0; i < kGB; ++i) {
      const int grp = warp + (h + i) * W;
      const bool ok = col_ok(grp);
      yq[i][0] = ok && has0 ? ldg_cg_v2(yrow0 + 32 * grp) : make_uint2(0u, 0u);
      yq[i][1] = ok && has1 ? ldg_cg_v2(yrow1 + 32 * grp) : make_uint2(0u, 0u);
    }
  };
  // Static weights and a short partition: this lane's A chunks go into
  // registers now, while the previous kernel still runs.
  const bool fast = ring.fast(early_w);
  typename PartialRing<BN>::ARegs ar[PartialRing<BN>::kFastKB];
  const bool a_ok = fast ? ring.fast_prologue(pa, ar) : true;

  // With IG_FLAG_INPUT_READY (and static weights) x is not written by the
  // kernel before this one on the stream: the shrink, the partial exchange
  // and the combine run before the dependency wait, and only the z store and
  // the y update (reads included) follow it.
  const bool pre = early_w && (p.flags & IG_FLAG_INPUT_READY) != 0;
  if (!pre) griddep_wait();
  if (warp == 0 && !early_w) {
    for (int b = 0; b < first; ++b) ring.issue_a(pa, b);
    issue_b();
  }
  uint2 ypre[kGB][2];
  float v;
  const bool ok = fast ? ring.fast_run(pa, xrow, ar, a_ok, red, v,
                                       [&]() { if (!pre) load_y(0, ypre); })
                       : ring.run(pa, xrow, red, v, [&]() { if (!pre) load_y(0, ypre); });

  // Send this block's partial P_s to slot s of every block of the cluster
  // (its own included). Every block sends on every path (zeros after a
  // failed copy), so every block receives exactly S * TB * 4 bytes.
  cluster_wait();
  {
    const float pv = ok ? v : 0.0f;
    for (int q = 0; q < S; ++q)
      st_async_f32(map_rank(part + s * TB + tid, (uint32_t)q), pv,
                   map_rank(bar_part, (uint32_t)q));
  }
  // While the partials travel: the B operands of this warp's first kGB
  // column groups (one Z part), from the slice that landed during the shrink.
  const bool zf32 = (p.flags & IG_FLAG_Z_FP32) != 0;
  const bool copies_ok = mbar_wait_bounded(bar_b, 0, p.status);
  const uint32_t sB_addr = smem_u32(sB);
  const int cmax = ncols - 1;
  uint32_t bq[kGB][2][4];
  // group g's B rows start at sB + (g / 2) * 128 * BN; this warp's groups all
  // have the parity of the warp (W is even)
  // (only groups that exist: the buffer holds ngroups whole groups)
  auto load_bq = [&](int h) {
#pragma unroll
    for (int i = 0; i < kGB; ++i) {
      const int grp = warp + (h + i) * W;
      if (grp < ngroups)
        ExpandFrag<BN>::load_b_at(sB_addr + (uint32_t)(grp >> 1) * (128u * BN), boff, bq[i]);
    }
  };
  if (copies_ok && !zf32 && warp < ngroups) load_bq(0);
  // The wait outlasts any sender's own bounded waits, so a block never
  // leaves while a partial is still on its way to it.
  const bool got = mbar_wait_bounded(bar_part, 0, p.status, 1ll << 36);

  // Combine (Algorithm 1 order): total = 0; total += P_q for q = 0..S-1.
  // Thread o owns output o (token row o / r, rank o % r).
  float zv = 0.0f;
  {
    const int o = tid;
    uint16_t hi = 0, mid = 0, lo = 0;
    if (o < nrows * BN) {
      // the S partials loaded together (S <= 16), then added in order
      float pq[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) pq[q] = q < S ? part[q * TB + o] : 0.0f;
      float total = 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q < S) total += pq[q];
      zv = total * p.scale;
      split_z(zv, zf32, hi, mid, lo);
    }
    zb[o] = hi;
    zb[TB + o] = mid;
    zb[2 * TB + o] = lo;
  }
  if (pre) {
    griddep_wait();
    load_y(0, ypre);
  }
  if (s == 0 && tid < nrows * BN) p.z[((int64_t)sl * M + rows_s[tid / BN]) * r + tid % BN] = zv;
  __syncthreads();   // zb complete

  // Expand this block's columns: y = bf16_rn(f32(y) + D), D the tensor-core
  // sum over j of bf16(z_j) B_nj (the same MMAs as the two-kernel expand).
  // Every element is computed by one MMA of one warp, so the split over
  // warps and blocks does not change any result. Batches of kGB of the
  // warp's groups (B operands of the first batch loaded above); the y of the
  // next batch is loaded before the current one is computed.
  if (copies_ok && got) {
    ExpandFrag<BN> zf;
    zf.load_z(zb, lane);
    for (int h = 0; warp + h * W < ngroups; h += kGB) {
      uint2 ynext[kGB][2];
      const bool more = warp + (h + kGB) * W < ngroups;
      if (more) load_y(h + kGB, ynext);
      if (h > 0 && !zf32) load_bq(h);
#pragma unroll
      for (int i = 0; i < kGB; ++i) {
        const int grp = warp + (h + i) * W;
        float vv[8];
        if (!zf32) zf.mma(vv, bq[i]);
        else expand_group_mma(vv, sB_addr, 32 * grp, cmax, BN, zb, 3, lane);
        if (col_ok(grp)) {
          if (has0)
            *reinterpret_cast<uint2*>(yrow0 + 32 * grp) = y_add4(ypre[i][0], vv[0], vv[1], vv[2], vv[3]);
          if (has1)
            *reinterpret_cast<uint2*>(yrow1 + 32 * grp) = y_add4(ypre[i][1], vv[4], vv[5], vv[6], vv[7]);
        }
      }
      if (more) {
#pragma unroll
        for (int i = 0; i < kGB; ++i) {
          ypre[i][0] = ynext[i][0];
          ypre[i][1] = ynext[i][1];
        }
      }
    }
  }
  // a copy that never completed: wait for it once more (bounded) before the
  // block's shared memory goes away
  if (!copies_ok) mbar_wait_bounded(bar_b, 0, p.status);
}

}  // namespace

size_t fused_smem_bytes(int bn, int64_t Ks, int64_t N, int S) {
  // + 1024: the kernel aligns its base to 1024 bytes (128-byte swizzle atoms)
  return 1024 + (bn == 16 ? fused_layout<16>(Ks, N, S).bytes : fused_layout<8>(Ks, N, S).bytes);
}

int fused_b_box_rows(int bn, int64_t Ks, int64_t N, int S) {
  return bn == 16 ? fused_layout<16>(Ks, N, S).box_rows : fused_layout<8>(Ks, N, S).box_rows;
}

cudaError_t launch_fused_warp(const FusedParams& p, int bn, int64_t tiles_max, cudaStream_t st) {
  const int64_t grid = tiles_max * p.slices * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = fused_smem_bytes(bn, p.Ks, p.N, p.S);
  void (*kern)(FusedParams) = bn == 16 ? fused_warp_kernel<16> : fused_warp_kernel<8>;
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
  cudaLaunchAttribute attr[3];
  // With IG_FLAG_INPUT_READY the shrink, exchange and combine run beside the
  // previous layer, and letting the hardware balance the clusters' blocks
  // over the SMs took such a chain from 3.43 to 3.13 us per layer; without
  // the flag the same policy made the chain slower (3.69 -> 4.12 us), so
  // it keeps the default placement.
  attr[2].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[2].val.clusterSchedulingPolicyPreference =
      (p.flags & IG_FLAG_INPUT_READY) ? cudaClusterSchedulingPolicyLoadBalancing
                                      : cudaClusterSchedulingPolicyDefault;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 3;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ig
