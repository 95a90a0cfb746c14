// LoRA expand on the tcgen05 tensor cores: y += bf16(Z) B_i^T, in place, one
// rounding; for ranks where the token x output x rank tile is a real dense
// contraction (prefill).
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction",
// Eq. 1 (the expand multiplies the r-wide shrink output by B in R^{Hout x r})
// and sec. 6.2 / Fig. 5 (the FP32 shrink output reaches the next operation as
// BF16, rounded to nearest).
//
// Block = 8 warps (two warpgroups), work = one 128-row tile of one adapter (128-row tile
// table) x one slice x nb column blocks of 64 (2 <= nb <= 16, chosen on the
// host so that the grid fills the GPU about three blocks per SM; it does not
// change any result). The A operand of the MMA, the tile's Z rows rounded to bf16,
// is built once per block (coalesced loads, written by the threads straight
// into the 128-byte-swizzled K-major layout), or, inside lora_apply, copied
// in that layout from where the shrink wrote it (one bulk copy per 16 KB
// atom), and serves all its column blocks. Per column block: the B operand (64 rows of B_i x r) and the y tile
// (128 rows x 64 columns: one TMA box when the tile's tokens are
// consecutive, else 16-byte asynchronous copies by every thread) come into
// one of two stages, so the copies of
// block i+2 are in flight while block i is computed; tcgen05.mma, M = 128,
// N = 64, K = 16 per instruction, r/16 of them, FP32 into one of two TMEM
// accumulators. Each thread then reads half a row of the accumulator (warp w:
// rows 32 (w % 4) .., columns 32 (w / 4) ..), adds it to y in FP32 and rounds
// once to bf16 in shared memory; the tile goes back by
// one TMA store when it is 128 consecutive tokens, else by whole-row stores.
//
// Arithmetic, fixed by r: the tensor core's FP32 sum over j, then
// bf16_rn(f32(y) + sum). A row's value depends only on that row.
#include "umma.cuh"

namespace ig {

namespace {

constexpr int kBN = kMmaExpandBN;                // output columns per column block
constexpr int kYB = kBN / 64;                    // 64-column y boxes per column block
constexpr int kYBox = kMmaTileRows * 128;        // one y box: 128 rows x 64 columns (16 KB)
constexpr int kYBytes = kYB * kYBox;             // y tile of one column block
constexpr int kBAtom = kBN * 128;                // B rows of one column block, per 64 ranks

constexpr int kMaxStages = 2;

struct Ctl {
  uint64_t full_b[kMaxStages];   // B copies of a stage
  uint64_t full_y[kMaxStages];   // y copies of a stage
  uint64_t done[2];              // MMAs of an accumulator
  uint64_t zbar;                 // the Z operand copy (Z written by the shrink)
  uint32_t tmem;
  int32_t fail;                  // a B copy never arrived
};

// Copy stages. Two: a third stage costs the third block per SM at r = 64,
// which measured slower (84 us against 52.5 us on the QKV prefill shape),
// and at r = 128 three to five stages leave one block per SM, 60% slower
// (a block's epilogues, not its copies in flight, set the pace).
__host__ __device__ inline int expand_stages(int) { return 2; }

// layout (offsets from the 1024-aligned base): ctl 0, tile entry 128,
// zb [parts][r/64][128 rows][128 B] at 1024, then the stages, each
// {B [r/64][64 rows][128 B], y [128 rows][128 B]}
__host__ __device__ inline size_t off_zb() { return 1024; }
__host__ __device__ inline size_t stage_bytes(int r) {
  return (size_t)((r + 63) / 64) * kBAtom + kYBytes;
}
__host__ __device__ inline size_t off_stage(int r, bool zf32, int s) {
  return off_zb() + (size_t)((r + 63) / 64) * 16384 * (zf32 ? 3 : 1) + s * stage_bytes(r);
}
__host__ __device__ inline size_t mma_expand_smem(int r, bool zf32) {
  return 1024 + off_stage(r, zf32, expand_stages(r));
}

// 16-byte asynchronous copy global -> shared (L2 only), and the arrival on
// an mbarrier once every earlier such copy of this thread has landed.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1,
                                             const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the shared-memory sources of this thread's bulk stores have been read
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// WG warpgroups per block: one where shared memory leaves room for three
// blocks per SM (at most 168 registers a thread), two where it leaves room
// for two (at most 128), so that either way 12 or 16 warps share an SM.
template <int NS, int WG>
__global__ void __launch_bounds__(128 * WG, WG == 1 ? 3 : 2)
    expand_mma_kernel(const __grid_constant__ MmaExpandParams p) {
  constexpr int kThreads = 128 * WG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 128);
  const int r = (int)p.r;
  const bool zf32 = (p.flags & IG_FLAG_Z_FP32) != 0;
  const int ka = (r + 63) / 64;                       // 64-column atoms of the rank
  uint8_t* s_zb = smem + off_zb();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t bid = blockIdx.x;
  const int nt = (int)next_digit(bid, (uint32_t)p.ntiles);
  const int sl = (int)next_digit(bid, (uint32_t)p.slices);
  const int64_t t = bid;

  for (int i = tid; i < kMmaTileInts; i += kThreads) ent_s[i] = p.tiles[t * kMmaTileInts + i];
  if (tid == 0) {
    // y of a tile of consecutive tokens comes by one TMA box (one arrival
    // with its byte count); of scattered tokens, by 16-byte copies from
    // every thread (one arrival each)
    const bool contig = p.tiles[t * kMmaTileInts + 2] != 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&ctl->full_b[i], 1);
      mbar_init(&ctl->full_y[i], contig ? 1 : kThreads);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&ctl->done[i], 1);
    mbar_init(&ctl->zbar, 1);
    ctl->fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 2 * kBN);
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
    if (warp == 1) tmem_dealloc(tmem, 2 * kBN);
  };
  if (g < 0 || g >= p.L || nrows <= 0) {
    teardown();
    return;
  }

  const int64_t N = p.N, M = p.M;
  const int64_t n0 = (int64_t)nt * p.nb * kBN;
  const int nb = (int)min((int64_t)p.nb, (N - n0 + kBN - 1) / kBN);   // column blocks here
  const int b_row = (int)(((int64_t)g * p.slices + sl) * N + n0);
  const int y_col = (int)((int64_t)sl * N + n0);
  const bool contiguous = ent_s[2] != 0;   // rows are consecutive tokens: one box
  const bool full_box = contiguous && nrows == kMmaTileRows;
  const bool early_b = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;
  const uint32_t y_tx = kYB * (uint32_t)kYBox;

  // column block i: stage i % NS (phase (i / NS) & 1), accumulator i % 2
  // (phase (i / 2) & 1)
  auto stage = [&](int i) { return smem + off_stage(r, zf32, i % NS); };
  auto sph = [&](int i) { return (uint32_t)((i / NS) & 1); };
  auto issue_b = [&](int i) {   // thread 0
    mbar_arrive_expect_tx(&ctl->full_b[i % NS], (uint32_t)ka * kBAtom);
    for (int a = 0; a < ka; ++a)
      tma_load_2d(stage(i) + a * kBAtom, &p.tm_b, a * 64, b_row + i * kBN, &ctl->full_b[i % NS]);
  };
  // y tile of column block i into its stage, 128-byte swizzled (16-byte
  // chunk c of row m at chunk c ^ (m % 8)). Consecutive tokens: one TMA box
  // per 64 columns, thread 0. Scattered tokens: every thread copies 16-byte
  // chunks (a warp instruction covers 4 rows x 128 bytes; columns past the
  // block's ncols are not read) and arrives once its copies have landed; row
  // gathers by TMA measured slower for scattered rows.
  const int64_t ld = (int64_t)p.slices * N;
  // Row copies (scattered tokens) and row stores (any tile not stored as one
  // box): thread t moves the 16-byte chunk t % 8 of tile rows
  // m_k = t / 8 + 32k (k = 0..3) in every column block, so the rows' global
  // offsets (column block 0; -1 past nrows) and the swizzled place of the
  // chunk (the same for every k, 32k being a multiple of 8) are computed once
  // per block.
  static_assert(kYB == 1, "one 64-column y box per column block");
  constexpr int kRowSets = kMmaTileRows * 8 / kThreads;   // rows per thread
  const int ych = tid & 7;
  const int ym = tid >> 3;
  const uint32_t ys_off = (uint32_t)ym * 128u + ((uint32_t)(ych ^ (ym & 7)) << 4);
  constexpr uint32_t kRowSetBytes = (kThreads / 8) * 128;
  int64_t yoff[kRowSets];
#pragma unroll
  for (int k = 0; k < kRowSets; ++k) {
    const int m = ym + (kThreads / 8) * k;
    yoff[k] = m < nrows ? (int64_t)rows_s[m] * ld + y_col + ych * 8 : -1;
  }
  auto issue_y = [&](int i) {   // thread 0 (consecutive tokens) or every thread
    uint8_t* sy = stage(i) + ka * kBAtom;
    if (contiguous) {
      if (tid == 0) {
        mbar_arrive_expect_tx(&ctl->full_y[i % NS], y_tx);
        for (int yb = 0; yb < kYB; ++yb)
          tma_load_2d(sy + yb * kYBox, &p.tm_yt, y_col + i * kBN + yb * 64, rows_s[0],
                      &ctl->full_y[i % NS]);
      }
      return;
    }
    const int nc = (int)min((int64_t)kBN, N - n0 - (int64_t)i * kBN);
    if (ych * 8 < nc) {
      const __nv_bfloat16* yi = p.y + (int64_t)i * kBN;
#pragma unroll
      for (int k = 0; k < kRowSets; ++k)
        if (yoff[k] >= 0) cp_async16(sy + ys_off + kRowSetBytes * k, yi + yoff[k]);
    }
    cp_async_mbar_arrive(&ctl->full_y[i % NS]);
  };

  if (tid == 0 && early_b)
    for (int i = 0; i < min(nb, NS); ++i) issue_b(i);
  // Inside lora_apply (the shrink wrote the Z operand) the first y copies
  // start before the dependency wait: the shrink writes no y, and it lets
  // this grid start only after its own dependency wait, by which time every
  // earlier kernel on the stream (the last writer of y among them) has
  // completed and its writes are visible.
  const bool y_early = p.zt != nullptr;
  if (y_early)
    for (int i = 0; i < min(nb, NS); ++i) issue_y(i);
  griddep_wait();
  griddep_launch();
  // Z written by the shrink as this tile's operand: one bulk copy per atom
  const uint32_t zt_bytes = (uint32_t)zt_entry_bytes(r, zf32);
  if (p.zt && tid == 0) {
    const uint8_t* src = p.zt + ((size_t)t * p.slices + sl) * zt_bytes;
    mbar_arrive_expect_tx(&ctl->zbar, zt_bytes);
    for (uint32_t o = 0; o < zt_bytes; o += 16384) bulk_g2s(s_zb + o, src + o, 16384, &ctl->zbar);
  }
  for (int i = 0; i < min(nb, NS); ++i) {
    if (tid == 0 && !early_b) issue_b(i);
    if (!y_early) issue_y(i);
  }

  // A operand: the tile's Z rows rounded to bf16 into the swizzled K-major
  // layout (16-byte chunk c of a 128-byte row m sits at chunk c ^ (m % 8)),
  // rows past nrows zero. Each warp loads its 128 / warps rows, r/4 lanes per row
  // (4 values each, coalesced), 16 loads in flight per lane before any is
  // used (one at a time, each load's latency under the copies in flight
  // added up to most of the block's life). With FP32 Z also
  // mid = bf16_rn(z - hi) and lo = bf16_rn(z - hi - mid) (hi + mid + lo == z
  // exactly), in atoms after the hi ones.
  if (p.zt) {
    // a copy that never lands fails the block's first accumulator wait
    if (!mbar_wait_bounded(&ctl->zbar, 0, p.status)) ctl->fail = 1;
  } else {
    constexpr int kWRows = kMmaTileRows / (kThreads / 32);   // rows per warp
    const int per_row = r / 4;
    const int total = kWRows * per_row;       // float4 of the warp's rows
    for (int b0 = 0; b0 < total; b0 += 16 * 32) {
      float4 f4[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int idx = b0 + lane + 32 * k;
        const int m = warp * kWRows + idx / per_row;
        f4[k] = idx < total && m < nrows
                    ? __ldcg(reinterpret_cast<const float4*>(
                          p.z + ((int64_t)sl * M + rows_s[m]) * r + 4 * (idx % per_row)))
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int idx = b0 + lane + 32 * k;
        if (idx >= total) continue;
        const int m = warp * kWRows + idx / per_row;
        const int j = 4 * (idx % per_row);
        const float fv[4] = {f4[k].x, f4[k].y, f4[k].z, f4[k].w};
        uint32_t pt[3][4];   // bf16 parts hi, mid, lo
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint16_t h, md, l;
          split_z(fv[e], zf32, h, md, l);
          pt[0][e] = h;
          pt[1][e] = md;
          pt[2][e] = l;
        }
        const int a = j / 64, c = (j % 64) / 8;
        const size_t off = (size_t)a * 16384 + m * 128 + ((c ^ (m & 7)) << 4) + (j % 8) * 2;
        for (int q = 0; q < (zf32 ? 3 : 1); ++q)
          *reinterpret_cast<uint2*>(s_zb + (size_t)q * ka * 16384 + off) =
              make_uint2(pt[q][0] | (pt[q][1] << 16), pt[q][2] | (pt[q][3] << 16));
      }
    }
    // rank columns past r inside the last atom are zero
    if (r % 64) {
      for (int idx = tid; idx < kMmaTileRows * ((64 - r % 64) / 8); idx += kThreads) {
        const int m = idx / ((64 - r % 64) / 8);
        const int c = (r % 64) / 8 + idx % ((64 - r % 64) / 8);
        const size_t off = (size_t)(ka - 1) * 16384 + m * 128 + ((c ^ (m & 7)) << 4);
        for (int q = 0; q < (zf32 ? 3 : 1); ++q)
          *reinterpret_cast<uint4*>(s_zb + (size_t)q * ka * 16384 + off) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  const uint32_t idesc = umma_idesc_bf16_f32(kMmaTileRows, kBN);
  // MMAs of column block i into accumulator i % 2 (thread 32); the B copy
  // of the block has been waited for, or the wait is bounded here
  auto issue_mma = [&](int i, bool b_ready) {
    const uint32_t acc = tmem + (uint32_t)((i & 1) * kBN);
    if (b_ready || mbar_wait_bounded(&ctl->full_b[i % NS], sph(i), p.status)) {
      tc_fence_after();
      const uint32_t sb = smem_u32(stage(i));
      for (int k = 0; k < r / 16; ++k) {
        const int a = k / 4, kk = k % 4;
        const uint64_t bdesc = umma_desc_sw128(sb + a * kBAtom + kk * 32);
        umma_bf16(acc, umma_desc_sw128(smem_u32(s_zb + a * 16384) + kk * 32), bdesc, idesc,
                  k > 0);
        if (zf32)   // mid and lo parts of FP32 Z, same k step
          for (int q = 1; q < 3; ++q)
            umma_bf16(acc, umma_desc_sw128(smem_u32(s_zb + (q * ka + a) * 16384) + kk * 32),
                      bdesc, idesc, true);
      }
    } else {
      ctl->fail = 1;
    }
    umma_commit(&ctl->done[i & 1]);
  };
  int next_mma = 0;   // thread 32: first block whose MMAs are not issued yet
  if (tid == 32) issue_mma(next_mma++, false);

  int issued = min(nb, NS);   // column blocks whose copies have been issued
  int i = 0;
  bool ok = true;
  for (; i < nb; ++i) {
    // the next block's MMAs overlap this block's epilogue (other
    // accumulator) when its B copy is already there; else they follow the
    // epilogue
    if (tid == 32 && next_mma == i + 1 && next_mma < nb &&
        mbar_try_wait(&ctl->full_b[next_mma % NS], sph(next_mma)))
      issue_mma(next_mma++, true);
    __syncwarp();
    const bool y_ok = mbar_wait_bounded(&ctl->full_y[i % NS], sph(i), p.status);
    const bool acc_ok = mbar_wait_bounded(&ctl->done[i & 1], (uint32_t)((i >> 1) & 1), p.status) &&
                        *reinterpret_cast<volatile int32_t*>(&ctl->fail) == 0;
    tc_fence_after();
    // a thread whose own wait expired writes nothing; the block agrees on
    // the failure at the barrier after the epilogue
    const bool mine = y_ok && acc_ok;
    uint8_t* sy = stage(i) + ka * kBAtom;

    // epilogue 1: y = bf16_rn(f32(y) + acc), in shared memory. Warp w reads
    // accumulator rows 32 (w % 4) .. + 31 (the lanes of tensor memory it may
    // access); warpgroup g the 32-column halves g, g + WG, ... of them
    const int m = 32 * (warp & 3) + lane;
    const uint32_t trow = tmem + (uint32_t)((i & 1) * kBN) + ((uint32_t)(32 * (warp & 3)) << 16);
    static_assert(kBN == 64, "two 32-column halves per column block");
    for (int c = 32 * (warp >> 2); c < kBN; c += 32 * WG) {
      float v[32];
      tmem_ld32(trow + c, v);
      if (m < nrows && mine) {
        uint8_t* rowp = sy + m * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = c / 8 + q;                       // logical 16-byte chunk
          uint4* cp = reinterpret_cast<uint4*>(rowp + ((chunk ^ (m & 7)) * 16));
          uint4 u = *cp;
          float yf[8];
          unpack8(u, yf);
          u.x = f32x2_to_bf16x2_bits(yf[0] + v[8 * q + 0], yf[1] + v[8 * q + 1]);
          u.y = f32x2_to_bf16x2_bits(yf[2] + v[8 * q + 2], yf[3] + v[8 * q + 3]);
          u.z = f32x2_to_bf16x2_bits(yf[4] + v[8 * q + 4], yf[5] + v[8 * q + 5]);
          u.w = f32x2_to_bf16x2_bits(yf[6] + v[8 * q + 6], yf[7] + v[8 * q + 7]);
          *cp = u;
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    if (__syncthreads_or(!mine)) {
      ok = false;
      break;
    }

    // epilogue 2: back to global memory. A full tile of consecutive tokens
    // goes by one TMA store that only thread 0 issues, so thread 0 alone
    // frees the stage (after the store has read it) and refills it, with no
    // block barrier; row stores read the stage from every thread, and a
    // barrier follows them.
    const int ncols = (int)min((int64_t)kBN, N - n0 - (int64_t)i * kBN);
    const bool tma_store = full_box && ncols == kBN;
    if (tma_store) {
      if (tid == 0) {
        for (int yb = 0; yb < kYB; ++yb)
          tma_store_2d(&p.tm_yt, y_col + i * kBN + yb * 64, rows_s[0], sy + yb * kYBox);
        bulk_commit();
      }
    } else {
      // four rows (128 bytes each) per warp-instruction, the rows and chunk
      // of the scattered-token copies above
      if (ych * 8 < ncols) {
        __nv_bfloat16* yi = p.y + (int64_t)i * kBN;
#pragma unroll
        for (int k = 0; k < kRowSets; ++k)
          if (yoff[k] >= 0)
            *reinterpret_cast<uint4*>(yi + yoff[k]) =
                *reinterpret_cast<const uint4*>(sy + ys_off + kRowSetBytes * k);
      }
      __syncthreads();
    }
    // stage i % NS is free once the store has read it: copies of block i + NS
    if (i + NS < nb) {
      if (tid == 0) {
        bulk_wait_read0();
        issue_b(i + NS);
      }
      issue_y(i + NS);
      issued = i + NS + 1;
    }
    if (tid == 32 && next_mma == i + 1 && next_mma < nb) issue_mma(next_mma++, false);
  }
  if (tid == 0) bulk_wait_read0();
  if (!ok) {
    // drain (bounded) what may still be in flight before the block leaves:
    // the copies of blocks i .. issued-1 and the MMAs issued for blocks >= i
    if (tid == 0)
      for (int b = i; b < issued; ++b) {
        mbar_wait_bounded(&ctl->full_b[b % NS], sph(b), p.status);
        mbar_wait_bounded(&ctl->full_y[b % NS], sph(b), p.status);
      }
    if (tid == 32)
      for (int b = i; b < next_mma; ++b)
        mbar_wait_bounded(&ctl->done[b & 1], (uint32_t)((b >> 1) & 1), p.status);
    if (tid == 0 && p.zt) mbar_wait_bounded(&ctl->zbar, 0, p.status);
  }
  teardown();
}

}  // namespace

cudaError_t launch_expand_mma(const MmaExpandParams& p, int64_t tiles_max, cudaStream_t st) {
  const size_t smem = mma_expand_smem((int)p.r, (p.flags & IG_FLAG_Z_FP32) != 0);
  // shared memory of one SM; each resident block also takes 1 KB of it
  static const int sm_smem = [] {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    return v;
  }();
  const int wg = 3 * (smem + 1024) <= (size_t)sm_smem ? 1 : 2;
  void (*kern)(MmaExpandParams) = wg == 1 ? expand_mma_kernel<2, 1> : expand_mma_kernel<2, 2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = tiles_max * p.slices * p.ntiles;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(128 * wg), smem, st, p);
}

size_t expand_mma_smem_bytes(int r, bool z_fp32) { return mma_expand_smem(r, z_fp32); }

}  // namespace ig
