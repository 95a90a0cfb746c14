// LoRA shrink on the tcgen05 tensor cores: Z = scale * X A_i^T with a Split-K
// reduction, for ranks where the token x rank x K tile is a real dense
// contraction (prefill).
//
// "Reproducible LoRA Inference Through Deterministic Split-K Reduction":
//   Eq. 3 / Fig. 1  S thread blocks per output tile, block s over the s-th
//                   contiguous K partition;
//   Algorithm 1     DET: FP32 partial -> scratch, gpu fence, block barrier,
//                   acq_rel integer increment of the tile's counter; the block
//                   that saw S-1 sums scratch[t][0..S-1] in increasing order,
//                   multiplies by the scale, writes the tile, zeroes the
//                   counter;
//   sec. 4.1        ATOMIC: FP32 atomic add of scale * partial into zeroed Z;
//   sec. 4.2        UNSPLIT: S = 1;
//   sec. 4.3        DET_TREE: partials only, combined by reduce_tree.cu.
//
// DET with S dividing 128 and S <= 16 (when such a cluster can be resident):
// the S blocks of a tile are one thread-block cluster, and block s owns tile
// rows [s 128/S, (s+1) 128/S). Every block writes its FP32 partial to slot s
// of the tile's workspace area (staged in shared memory, half the columns at
// a time, so that the global stores are coalesced), then a cluster barrier,
// then each owner sums the S partials of its rows from FP32 zero in
// increasing partition order (16 loads in flight per thread) and scales
// them: the counter protocol's order, so the same bits, with no counter and
// the combine spread over the S blocks. The owner then drops the partial
// lines it read from L2 without a write-back. (Exchanging the partials
// through distributed shared memory measured slower: 84 KB per block at the
// QKV shape took 7.8 us against 4.8 us through L2.)
//
// Block = 8 warps, tile = up to 128 token rows of one adapter (one entry of
// the token map's 128-row tile table) x all r rank columns of one slice, or of
// all slices at once where slices x r <= 256 (the slices' A rows are
// consecutive in A_stack, so one tiled copy and one MMA of N = slices x r
// serve them, and the x tile is read once instead of once per slice). Warp 0
// issues the TMA copies: per k-step of 64 elements, x as one 128-row box
// when the tile's tokens are consecutive (else row gathers, 4 rows each,
// only the tile's rows, from the lanes of warps 0 and 2) and one tiled copy
// of the A block (r rows), all 128-byte swizzled, into a 2- to 4-deep ring.
// One thread of warp 1 issues per k-step four tcgen05.mma (M = 128 tokens,
// N = r, K = 16) into an FP32 accumulator in tensor memory and commits each
// stage back to the producer. The last k-step of a partition that is not a
// multiple of 64 issues only the MMAs inside the partition. All 8 warps then
// read the accumulator (warp w: token rows 32 (w % 4) .. + 31, one row per
// thread, every other 32 columns from column 32 (w / 4)).
//
// Inside lora_apply (DET and UNSPLIT) the block that writes a final z value
// also writes its bf16 parts into the expand's Z operand for the tile
// (zt_entry_bytes layout), and zeroes the operand's rows past the tile's
// tokens and ranks past r, so that the expand copies the operand instead of
// building it; the rounding is the expand's own, so the bits are the same.
//
// Arithmetic order, fixed by K/S and r only: the tensor core's FP32
// accumulation of the K-steps in order within the partition, then the
// partitions summed in increasing order. A row's value depends only on that
// row, its adapter and the plan.
#include <map>
#include <mutex>
#include <utility>

#include "umma.cuh"

namespace ig {

namespace {

constexpr int kThreads = 256;   // two warpgroups: both read the accumulator
constexpr int kMaxStages = 4;
// Copy ring depth: 4 stages up to r = 64, 3 at r = 128, 2 at r = 256, so that
// two blocks share an SM (one per SM leaves 16-block clusters short of SMs).
__host__ __device__ inline int shrink_stages(int r) {
  const int stage = kMmaTileRows * 128 + r * 128;
  const int n = (110 * 1024) / stage;
  return n < 2 ? 2 : (n > kMaxStages ? kMaxStages : n);
}
constexpr int kKStep = 64;                      // elements per k-step (128 bytes)
constexpr int kXTileBytes = kMmaTileRows * 128;  // 16 KB

struct Ctl {                       // control block at the start of shared memory
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t done;
  uint32_t tmem;
  int32_t info[4];
};

// nc = accumulator columns (stacked slices x r). The cluster combine stages
// its partial, [128][nc / 2 + 4] FP32, in the ring, which is sized to hold
// it.
__host__ __device__ inline size_t mma_ring_bytes(int nc, bool cl) {
  const size_t ring = (size_t)shrink_stages(nc) * (kXTileBytes + (size_t)nc * 128);
  const size_t stage = (size_t)kMmaTileRows * (nc / 2 + 4) * 4;   // cluster combine staging
  return cl && stage > ring ? stage : ring;
}
__host__ __device__ inline size_t mma_shrink_smem(int nc, bool cl) {
  return 1024 /*align slack*/ + 1024 /*ctl*/ + (size_t)kMmaTileInts * 4 +
         mma_ring_bytes(nc, cl) + 1024;
}

__host__ __device__ inline uint32_t tmem_cols_for(int r) {
  uint32_t c = 32;
  while (c < (uint32_t)r) c <<= 1;
  return c;
}

// The expand's Z operand (zt_entry_bytes layout): ranks j .. j+3 (j % 4 == 0)
// of tile row m, bf16 parts of the final z values as the expand would round
// or split them.
__device__ __forceinline__ void zt_put4(uint8_t* ent, int ka, bool zf32, int m, int j,
                                        float4 zv) {
  const float f[4] = {zv.x, zv.y, zv.z, zv.w};
  uint32_t pt[3][4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint16_t h, md, l;
    split_z(f[e], zf32, h, md, l);
    pt[0][e] = h;
    pt[1][e] = md;
    pt[2][e] = l;
  }
  const size_t off = (size_t)(j / 64) * 16384 + (size_t)m * 128 +
                     ((((j % 64) / 8) ^ (m & 7)) << 4) + (j % 8) * 2;
  for (int q = 0; q < (zf32 ? 3 : 1); ++q)
    *reinterpret_cast<uint2*>(ent + (size_t)q * ka * 16384 + off) =
        make_uint2(pt[q][0] | (pt[q][1] << 16), pt[q][2] | (pt[q][3] << 16));
}

// Zero, in every part, the 16-byte chunks of tile rows [m0, m1) from rank
// column cfrom on (a multiple of 8): rows past the tile's tokens (cfrom = 0)
// and the ranks past r in the last atom, which the expand's MMAs read.
__device__ __forceinline__ void zt_zero(uint8_t* ent, int ka, int parts, int m0, int m1,
                                        int cfrom, int tid, int nthr) {
  const int c0 = cfrom / 8, nch = ka * 8 - c0, nr = m1 - m0;
  if (nch <= 0 || nr <= 0) return;
  for (int i = tid; i < parts * nr * nch; i += nthr) {
    const int q = i / (nr * nch), rem = i % (nr * nch);
    const int m = m0 + rem / nch, cc = c0 + rem % nch;
    *reinterpret_cast<uint4*>(ent + (size_t)(q * ka + cc / 8) * 16384 + (size_t)m * 128 +
                              (((cc % 8) ^ (m & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// CL (IG_MODE_DET only): the S partition blocks of a tile are one cluster and
// combine there instead of through scratch and the counter.
template <int MODE, bool CL>
__global__ void __launch_bounds__(kThreads)
    shrink_mma_kernel(const __grid_constant__ MmaShrinkParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned working area (128-byte swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  int32_t* ent_s = reinterpret_cast<int32_t*>(smem + 1024);
  uint8_t* ring = smem + 1024 + ((kMmaTileInts * 4 + 1023) / 1024) * 1024;
  const int r = (int)p.r;
  const int ns = p.stack;                 // slices of this block
  const int nc = ns * r;                  // accumulator columns: slice sl0 + c / r, rank c % r
  const int stage_bytes = kXTileBytes + nc * 128;
  const int nst = shrink_stages(nc);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;
  const int ngroups = p.slices / ns;
  uint32_t bid = blockIdx.x;
  const int s = (int)next_digit(bid, (uint32_t)S);
  const int sg = (int)next_digit(bid, (uint32_t)ngroups);
  const int sl0 = sg * ns;
  const int64_t t = bid;
  // z address of accumulator column c (four columns never straddle a slice:
  // r is a multiple of 16)
  auto zrow = [&](int c, int tok) -> float* {
    return p.z + ((int64_t)(sl0 + c / r) * p.M + tok) * r + c % r;
  };
  // the expand's Z operand (lora_apply): entry of slice sl0 + c / r
  const bool zf32 = (p.flags & IG_FLAG_Z_FP32) != 0;
  const int zka = (r + 63) / 64;
  const size_t zt_bytes = zt_entry_bytes(r, zf32);
  auto zt_ent = [&](int sl) -> uint8_t* {
    return p.zt + ((size_t)t * p.slices + sl) * zt_bytes;
  };

  for (int i = tid; i < kMmaTileInts; i += kThreads) ent_s[i] = p.tiles[t * kMmaTileInts + i];
  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], 1);
    }
    mbar_init(&ctl->done, 1);
    fence_mbar_init();
  }
  const uint32_t ncols = tmem_cols_for(nc);
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const int g = ent_s[0];
  const int nrows = ent_s[1];
  const int32_t* rows_s = ent_s + 4;
  // cluster combine: block s owns tile rows [s R, s R + R), R = 128 / S, and
  // receives the S partials of its valid rows
  const int R = kMmaTileRows / S;
  const int own_rows = max(0, min(R, nrows - s * R));
  // zero the rows [m0, m1) past nrows and the ranks past r of rows
  // [m0, min(m1, nrows)) in the block's slices
  auto zt_pad = [&](int m0, int m1) {
    for (int k = 0; k < ns; ++k) {
      zt_zero(zt_ent(sl0 + k), zka, zf32 ? 3 : 1, max(m0, nrows), m1, 0, tid, kThreads);
      if (r % 64) zt_zero(zt_ent(sl0 + k), zka, zf32 ? 3 : 1, m0, min(m1, nrows), r, tid, kThreads);
    }
  };

  auto teardown = [&]() {
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, ncols);
  };

  if (nrows <= 0) {
    teardown();
    return;
  }
  if (g == p.L) {
    griddep_wait();
    griddep_launch();
    if (MODE != IG_MODE_ATOMIC && s == 0)
      for (int i = tid; i < nrows * nc; i += kThreads) *zrow(i % nc, rows_s[i / nc]) = 0.0f;
    teardown();
    return;
  }

  const int64_t Ks = p.Ks;
  const int k0 = (int)((int64_t)s * Ks);
  const int nk = (int)((Ks + kKStep - 1) / kKStep);      // k-steps
  const int a_row = (int)(((int64_t)g * p.slices + sl0) * r);
  const int groups4 = (nrows + 3) / 4;
  const bool contiguous = ent_s[2] != 0;   // rows are consecutive tokens: one box
  const uint32_t stage_tx =
      (contiguous ? (uint32_t)kXTileBytes : (uint32_t)groups4 * 4 * 128) + (uint32_t)nc * 128;
  const bool early_a = (p.flags & IG_FLAG_STATIC_WEIGHTS) != 0;
  const int first = min(nk, nst);

  auto issue_a = [&](int b) {
    uint8_t* st = ring + (b % nst) * stage_bytes;
    tma_load_2d(st + kXTileBytes, &p.tm_a, k0 + b * kKStep, a_row, &ctl->full[b % nst]);
  };
  // x of k-step b: lane 0 copies the box of a tile of consecutive tokens;
  // the rows of a scattered tile are gathered four at a time, the gathers
  // spread over the 32 lanes of a warp, warp 0 for the even k-steps and
  // warp 2 for the odd ones (one thread issuing all of them held a
  // scattered-token shrink at 40% of the copy bandwidth, one warp at 49%,
  // two warps at 58%, three warps at 55%)
  auto issue_x = [&](int b) {
    uint8_t* st = ring + (b % nst) * stage_bytes;
    if (contiguous) {
      if (lane == 0) tma_load_2d(st, &p.tm_xt, k0 + b * kKStep, rows_s[0], &ctl->full[b % nst]);
      return;
    }
    const int last = nrows - 1;
    for (int q = lane; q < groups4; q += 32)
      tma_gather4(st + q * 4 * 128, &p.tm_x, k0 + b * kKStep, rows_s[min(4 * q, last)],
                  rows_s[min(4 * q + 1, last)], rows_s[min(4 * q + 2, last)],
                  rows_s[min(4 * q + 3, last)], &ctl->full[b % nst]);
  };

  bool failed = false;
  if (warp == 0 && lane == 0) {
    for (int b = 0; b < first; ++b) {
      mbar_arrive_expect_tx(&ctl->full[b], stage_tx);
      if (early_a) issue_a(b);
    }
  }
  griddep_wait();
  griddep_launch();

  if (warp == 0) {
    // producer warp: lane 0 waits for a free stage, arms it with the stage's
    // byte count and copies A; the x copies follow (the arming may come
    // after a lane's gather has landed: the stage cannot complete before
    // lane 0's arrival)
    for (int b = 0; b < nk; ++b) {
      int ok = 1;
      if (lane == 0) {
        if (b >= first) {
          const int st = b % nst;
          if (mbar_wait_bounded(&ctl->empty[st], (uint32_t)(((b / nst) - 1) & 1), p.status)) {
            mbar_arrive_expect_tx(&ctl->full[st], stage_tx);
            issue_a(b);
          } else {
            ok = 0;
          }
        } else if (!early_a) {
          issue_a(b);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        failed = true;
        break;
      }
      if (contiguous || (b & 1) == 0) issue_x(b);
    }
  } else if (warp == 2 && !contiguous) {
    // second gather warp of a scattered tile: the x rows of the odd k-steps,
    // once their stage is free (lane 0 of warp 0 arms it)
    for (int b = 1; b < nk; b += 2) {
      int ok = 1;
      if (lane == 0 && b >= first)
        ok = mbar_wait_bounded(&ctl->empty[b % nst], (uint32_t)(((b / nst) - 1) & 1), p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        failed = true;
        break;
      }
      issue_x(b);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = umma_idesc_bf16_f32(kMmaTileRows, nc);
    for (int b = 0; b < nk; ++b) {
      const int st = b % nst;
      if (!mbar_wait_bounded(&ctl->full[st], (uint32_t)((b / nst) & 1), p.status)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint32_t xs = smem_u32(ring + st * stage_bytes);
      const uint32_t as = xs + kXTileBytes;
      const int64_t rem = Ks - (int64_t)b * kKStep;
      const int ksub = (int)min((int64_t)4, (rem + 15) / 16);
      for (int kk = 0; kk < ksub; ++kk)
        umma_bf16(tmem, umma_desc_sw128(xs + kk * 32), umma_desc_sw128(as + kk * 32), idesc,
                  b > 0 || kk > 0);
      umma_commit(&ctl->empty[st]);
    }
    umma_commit(&ctl->done);  // also after a failure: tracks everything issued
  }
  __syncwarp();

  // epilogue: wait for the accumulator
  const bool acc_ok = mbar_wait_bounded(&ctl->done, 0, p.status);
  tc_fence_after();
  // warp w reads accumulator rows 32 (w % 4) .. + 31 (the lanes of tensor
  // memory it may access), warpgroup cg = w / 4 every other 32 columns
  const int row = 32 * (warp & 3) + lane;
  const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const int cg = warp >> 2;
  if (CL) {
    // This block's partial -> slot s of the tile's workspace area, staged in
    // shared memory (the ring: every MMA of this block has completed) half
    // the columns at a time, rows padded by 16 bytes, then stored with
    // consecutive threads on consecutive 16-byte pieces of a row.
    const int64_t slot = t * ngroups + sg;
    float* part = p.partials + slot * (int64_t)S * (kMmaTileRows * nc);
    const int cw = nc / 2;                        // nc is a multiple of 16
    const int rowf = cw + 4;                      // padded staged row, floats
    float* stg = reinterpret_cast<float*>(ring);  // [128][rowf]
    for (int h = 0; h < 2; ++h) {
      for (int c = 32 * cg; c < cw; c += 64) {
        float v[32];
        tmem_ld32(trow + h * cw + c, v);
        const int nv = acc_ok ? min(32, cw - c) : 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (4 * i < nv)
            *reinterpret_cast<float4*>(stg + row * rowf + c + 4 * i) =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
      __syncthreads();
      const int q4 = cw / 4;
      float* dst = part + (int64_t)s * (kMmaTileRows * nc) + h * cw;
      for (int o = tid; acc_ok && o < nrows * q4; o += kThreads) {
        const int m = o / q4, c4 = o % q4;
        *reinterpret_cast<float4*>(dst + (int64_t)m * nc + 4 * c4) =
            *reinterpret_cast<const float4*>(stg + m * rowf + 4 * c4);
      }
      __syncthreads();
    }
    // every block's partial is in L2 and visible to the cluster
    __threadfence();
    cluster_sync_all();
    // Combine (Algorithm 1 order) of the owned rows: total = 0; total += P_q
    // for q = 0..S-1; z = total * scale. Four columns per step; 16 loads in
    // flight per thread (two steps of up to 8 partitions, or one of 16).
    const int n4 = own_rows * nc / 4;
    const int64_t own4 = (int64_t)s * R * nc / 4;
    const int64_t pstride4 = (int64_t)kMmaTileRows * nc / 4;
    const float4* p4 = reinterpret_cast<const float4*>(part) + own4;
    const int per = S <= 8 ? 2 : 1;               // steps per thread per round
    for (int b0 = 0; acc_ok && b0 < n4; b0 += per * kThreads) {
      float4 v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int k = per == 2 ? i / 8 : 0, q = per == 2 ? i % 8 : i;
        const int o4 = b0 + k * kThreads + tid;
        v[i] = (o4 < n4 && q < S) ? __ldcg(p4 + q * pstride4 + o4)
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
      for (int k = 0; k < per; ++k) {
        const int o4 = b0 + k * kThreads + tid;
        if (o4 >= n4) continue;
        float4 total = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int i = k * 8 + q;
          if (q < S && (per == 1 || q < 8)) {
            const float4 w = v[per == 2 ? i : q];
            total.x += w.x;
            total.y += w.y;
            total.z += w.z;
            total.w += w.w;
          }
        }
        const int o = 4 * o4;
        const float4 zv = make_float4(total.x * p.scale, total.y * p.scale,
                                      total.z * p.scale, total.w * p.scale);
        *reinterpret_cast<float4*>(zrow(o % nc, rows_s[s * R + o / nc])) = zv;
        if (p.zt) zt_put4(zt_ent(sl0 + (o % nc) / r), zka, zf32, s * R + o / nc, (o % nc) % r, zv);
      }
    }
    if (p.zt && acc_ok) zt_pad(s * R, s * R + R);
    // The owned rows' partial lines are read and dead (the next call writes
    // them again before reading them): drop them from L2 without writing them
    // back. Each owner's R rows of a slot are whole 128-byte lines.
    __syncthreads();
    {
      const int lines = R * nc * 4 / 128;
      for (int i = tid; i < S * lines; i += kThreads) {
        const int q = i / lines, l = i % lines;
        const char* a = reinterpret_cast<const char*>(p4 + q * pstride4) + l * 128;
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(a) : "memory");
      }
    }
    if (failed || !acc_ok) {
      if (tid == 0)
        for (int st = 0; st < nst; ++st) mbar_wait_bounded(&ctl->full[st], 0, p.status);
    }
    teardown();
    return;
  }
  const int64_t slot = t * ngroups + sg;
  float* part = p.partials + slot * (int64_t)S * (kMmaTileRows * nc);
  for (int c = 32 * cg; c < nc; c += 64) {
    float v[32];
    tmem_ld32(trow + c, v);
    if (!acc_ok || row >= nrows) continue;
    const int nv = min(32, nc - c);   // nc is a multiple of 16
    if (MODE == IG_MODE_DET || MODE == IG_MODE_DET_TREE) {
      float4* dst = reinterpret_cast<float4*>(part + (int64_t)s * (kMmaTileRows * nc) +
                                              (int64_t)row * nc + c);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (4 * i < nv) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else if (MODE == IG_MODE_UNSPLIT) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (4 * i < nv) {
          const float4 zv = make_float4(v[4 * i] * p.scale, v[4 * i + 1] * p.scale,
                                        v[4 * i + 2] * p.scale, v[4 * i + 3] * p.scale);
          *reinterpret_cast<float4*>(zrow(c + 4 * i, rows_s[row])) = zv;
          if (p.zt) zt_put4(zt_ent(sl0 + (c + 4 * i) / r), zka, zf32, row, (c + 4 * i) % r, zv);
        }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nv) atomicAdd(zrow(c + i, rows_s[row]), v[i] * p.scale);
    }
  }

  if (MODE == IG_MODE_UNSPLIT && p.zt && acc_ok) zt_pad(0, kMmaTileRows);
  if (MODE == IG_MODE_DET) {
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const uint32_t prev = atom_add_acq_rel_gpu(p.counters + slot, 1u);
      ctl->info[0] = (int)prev;
      if (prev >= (uint32_t)S) atomicOr(p.status, kStatusCorrupt);
    }
    __syncthreads();
    if ((uint32_t)ctl->info[0] == (uint32_t)(S - 1)) {
      __threadfence();
      // Each thread owns up to kPer float4 outputs (four consecutive columns
      // of one row) and adds the partitions q = 0..S-1 in order; the kPer
      // loads of one partition are in flight together (2048 per block).
      constexpr int kPer = 2048 / kThreads;
      const int n4 = nrows * nc / 4;
      for (int base = 0; base < n4; base += kPer * kThreads) {
        float4 tot[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) tot[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int q = 0; q < S; ++q) {
          const float4* src =
              reinterpret_cast<const float4*>(part + (int64_t)q * (kMmaTileRows * nc));
          float4 v[kPer];
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int o4 = base + i * kThreads + tid;
            v[i] = o4 < n4 ? __ldcg(src + o4) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          }
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            tot[i].x += v[i].x;
            tot[i].y += v[i].y;
            tot[i].z += v[i].z;
            tot[i].w += v[i].w;
          }
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int o4 = base + i * kThreads + tid;
          if (o4 >= n4) continue;
          const int o = 4 * o4;
          const float4 zv = make_float4(tot[i].x * p.scale, tot[i].y * p.scale,
                                        tot[i].z * p.scale, tot[i].w * p.scale);
          *reinterpret_cast<float4*>(zrow(o % nc, rows_s[o / nc])) = zv;
          if (p.zt) zt_put4(zt_ent(sl0 + (o % nc) / r), zka, zf32, o / nc, (o % nc) % r, zv);
        }
      }
      if (p.zt) zt_pad(0, kMmaTileRows);
      if (tid == 0) p.counters[slot] = 0u;
    }
  }

  if (failed || !acc_ok) {
    // drain (bounded) the copies of stages that were issued and not consumed
    if (tid == 0)
      for (int st = 0; st < nst; ++st)
        mbar_wait_bounded(&ctl->full[st], 0, p.status);
  }
  teardown();
}

template <int MODE>
cudaError_t launch_mode(const MmaShrinkParams& p, int64_t tiles_max, cudaStream_t st) {
  auto kern = shrink_mma_kernel<MODE, false>;
  const size_t smem = mma_shrink_smem((int)(p.stack * p.r), false);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = tiles_max * (p.slices / p.stack) * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, p);
}

// Can a cluster of S blocks with this footprint be resident? Cached per
// (S, accumulator columns).
bool cluster_fits(int S, int nc) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, bool> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(S, nc);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  auto kern = shrink_mma_kernel<IG_MODE_DET, true>;
  const size_t smem = mma_shrink_smem(nc, true);
  bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) == cudaSuccess;
  if (ok && S > 8)
    ok = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
         cudaSuccess;
  int n = 0;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1;
  }
  cudaGetLastError();   // clear a refused query
  cache[key] = ok;
  return ok;
}

cudaError_t launch_cluster(const MmaShrinkParams& p, int64_t tiles_max, cudaStream_t st) {
  auto kern = shrink_mma_kernel<IG_MODE_DET, true>;
  const size_t smem = mma_shrink_smem((int)(p.stack * p.r), true);
  // per launch: the attribute is per function, and other ranks set it too
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  if (p.S > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const int64_t grid = tiles_max * (p.slices / p.stack) * p.S;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
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

}  // namespace

cudaError_t launch_shrink_mma(const MmaShrinkParams& p, int mode, int64_t tiles_max,
                              cudaStream_t st) {
  if (mode == IG_MODE_DET) {
    // the cluster combine and the counter protocol give the same bits
    // (rows are dealt to the S blocks in equal shares, S must divide 128; the
    // received partials, 128 rows x nc FP32, share the ring's memory, and the
    // footprint must leave two blocks per SM)
    const int nc = (int)(p.stack * p.r);
    if (!(p.flags & IG_FLAG_UNFUSED) && p.S <= 16 && kMmaTileRows % p.S == 0 &&
        mma_ring_bytes(nc, true) <= 110 * 1024 && cluster_fits(p.S, nc))
      return launch_cluster(p, tiles_max, st);
    return launch_mode<IG_MODE_DET>(p, tiles_max, st);
  }
  if (mode == IG_MODE_DET_TREE) return launch_mode<IG_MODE_DET_TREE>(p, tiles_max, st);
  if (mode == IG_MODE_ATOMIC) return launch_mode<IG_MODE_ATOMIC>(p, tiles_max, st);
  return launch_mode<IG_MODE_UNSPLIT>(p, tiles_max, st);
}

}  // namespace ig
