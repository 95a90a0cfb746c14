// The shrink partial of one tile over one K partition, on the warp-level
// tensor cores. Shared by the Split-K shrink kernel and the fused decode
// kernel so that both compute bit-identical partials.
//
// Tile: up to 8 token rows x BN rank columns (BN = 8 or 16); the block has
// BN/4 warps (4 or 2) and ends with one output per thread: thread o holds
// the partial of token row o / BN, rank o % BN. The partition [k0, k0 + Ks)
// is streamed through a ring of `nst` shared-memory stages of 256 elements:
// the BN A rows as four 64-element sub-blocks, 128-byte swizzled (one 3-D
// TMA copy when K and K/S are multiples of 64, else one 2-D copy per
// sub-block), and the token rows of x unswizzled, 512 bytes each (one row
// gather per 4 tokens; a last group of one token by a tiled copy); completion
// is counted in bytes on one mbarrier per stage, and warp 0 issues the copies.
// The x operand rows of the MMA past nrows read the tile's last row (the same
// address: a broadcast). Full tiles of large batches take x swizzled instead
// (64-element sub-blocks: conflict-free ldmatrix, four copies per k-block);
// at small batches the one-copy layout's shorter latency wins. Either way the
// operand values, and so the results, are the same.
//
// Order of the sum, identical for every row and every M ("Reproducible LoRA
// Inference Through Deterministic Split-K Reduction" leaves the order inside
// a partition to the kernel, sec. 4.3): the partition is cut into 16-element
// steps (an 8-element step last when Ks % 16 == 8); step i of a 256-element
// block belongs to warp i % W. Each warp accumulates its steps in increasing
// k with bf16 tensor-core MMAs into FP32 (m16n8k16: 16 ranks x 8 tokens x 16
// k per instruction; ranks 8..15 are zero when BN = 8). The W warp sums are
// then added in warp order: ((D0 + D1) + D2) + D3. A token's value depends
// only on its own x row: the MMA's columns are independent.
#pragma once

#include "warp_mma.cuh"

namespace ig {

template <int BN>
struct ShrinkGeo {
  static constexpr int WARPS = BN / 4;            // 4 for BN = 16, 2 for BN = 8
  static constexpr int THREADS = WARPS * 32;
  static constexpr int TB = kTileRows * BN;       // outputs per tile = threads
  static_assert(TB == THREADS, "one output per thread");
};

struct PartialArgs {
  const int32_t* rows;        // token rows of the tile (shared memory)
  uint32_t* status;
  int64_t Ks;                 // partition length
  int nrows;
  const CUtensorMap* tm_x;    // x [M][K], box 256 x 1, no swizzle
  const CUtensorMap* tm_xs;   // x [M][K], box 64 x 1, 128-byte swizzle (wide tiles)
  const CUtensorMap* tm_a;    // A as [rows][K], box 64 x BN, 128-byte swizzle
  const CUtensorMap* tm_a3;   // A as {64, rows, K/64}, box {64, BN, 4}, or null
  int k0;                     // partition start (column coordinate)
  int a_row;                  // row coordinate of the tile's first A row
  int wide_rows;              // tiles of this many tokens or more: swizzled x
};

template <int BN>
struct PartialRing {
  using G = ShrinkGeo<BN>;
  static constexpr int kSub = kShrinkKB / 64;                 // 64-element sub-blocks
  static constexpr int kXBytes = kTileRows * kShrinkKB * 2;   // [8 rows][512 B]
  static constexpr int kABytes = kSub * BN * 128;             // [sub][BN rows][128 B]
  static constexpr int kStageBytes = kXBytes + kABytes;       // multiple of 1024
  static constexpr int kRowBytes = kShrinkKB * 2;             // x row (512 B)
  uint8_t* stages;   // 1024-aligned
  uint64_t* bars;
  int nst;      // ring depth
  int nkb;      // k-blocks in the partition

  __device__ __forceinline__ int klen(const PartialArgs& a, int b) const {
    return (int)min((int64_t)kShrinkKB, a.Ks - (int64_t)b * kShrinkKB);
  }
  __device__ __forceinline__ int nsub(const PartialArgs& a, int b) const {
    return (klen(a, b) + 63) / 64;
  }
  // x rows copied: 4 per row gather; a last group holding one row is copied
  // by a one-row tiled load instead (no repeated rows)
  __device__ __forceinline__ static int x_rows_copied(int nrows) {
    return (nrows / 4) * 4 + (nrows % 4 == 1 ? 1 : (nrows % 4 ? 4 : 0));
  }
  // Tiles of at least a.wide_rows tokens take x in 64-element,
  // 128-byte-swizzled sub-blocks (conflict-free ldmatrix, four copies per
  // k-block); smaller tiles take unswizzled 512-byte rows (one copy per
  // k-block). Same operand values, same results: the host picks the
  // threshold from the batch size.
  __device__ __forceinline__ static bool wide(const PartialArgs& a) {
    return a.nrows >= a.wide_rows;
  }
  // warp 0: arm stage b % nst for all copies of k-block b
  __device__ __forceinline__ void expect(const PartialArgs& a, int b) const {
    const uint32_t xb = wide(a) ? (uint32_t)nsub(a, b) * 128u * x_rows_copied(a.nrows)
                                : (uint32_t)kRowBytes * x_rows_copied(a.nrows);
    const uint32_t bytes = (uint32_t)nsub(a, b) * 128u * BN + xb;
    if ((threadIdx.x & 31) == 0) mbar_arrive_expect_tx(&bars[b % nst], bytes);
    __syncwarp();
  }
  __device__ __forceinline__ void issue_a(const PartialArgs& a, int b) const {
    if ((threadIdx.x & 31) != 0) return;
    const int st = b % nst;
    uint8_t* sa = stages + st * kStageBytes + kXBytes;
    const int ns = nsub(a, b);
    if (a.tm_a3 && ns == kSub) {   // the four sub-blocks in one copy (same layout)
      tma_load_3d(sa, a.tm_a3, 0, a.a_row, (a.k0 + b * kShrinkKB) / 64, &bars[st]);
      return;
    }
    for (int q = 0; q < ns; ++q)
      tma_load_2d(sa + q * BN * 128, a.tm_a, a.k0 + b * kShrinkKB + q * 64, a.a_row, &bars[st]);
  }
  __device__ __forceinline__ void issue_x(const PartialArgs& a, int b) const {
    const int lane = threadIdx.x & 31;
    const int st = b % nst;
    uint8_t* sx = stages + st * kStageBytes;
    const int groups4 = (a.nrows + 3) / 4;
    const int last = a.nrows - 1;
    if (wide(a)) {
      // one lane per (sub-block, group of 4 rows), 128-byte swizzled
      if (lane < nsub(a, b) * groups4) {
        const int q = lane / groups4, gq = lane % groups4;
        uint8_t* dst = sx + q * 1024 + gq * 512;
        const int kc = a.k0 + b * kShrinkKB + q * 64;
        if (4 * gq == last)
          tma_load_2d(dst, a.tm_xs, kc, a.rows[last], &bars[st]);
        else
          tma_gather4(dst, a.tm_xs, kc, a.rows[4 * gq], a.rows[min(4 * gq + 1, last)],
                      a.rows[min(4 * gq + 2, last)], a.rows[min(4 * gq + 3, last)], &bars[st]);
      }
      return;
    }
    // one lane per group of 4 rows; in a group of 2 or 3 rows the last row
    // repeats (loaded, never used); a group of one row is one tiled copy
    if (lane < groups4) {
      uint8_t* dst = sx + lane * 4 * kRowBytes;
      const int kc = a.k0 + b * kShrinkKB;
      if (4 * lane == last)
        tma_load_2d(dst, a.tm_x, kc, a.rows[last], &bars[st]);
      else
        tma_gather4(dst, a.tm_x, kc, a.rows[4 * lane], a.rows[min(4 * lane + 1, last)],
                    a.rows[min(4 * lane + 2, last)], a.rows[min(4 * lane + 3, last)], &bars[st]);
    }
  }

  // The MMAs of k-block b (stage st, kl elements) for this warp, accumulated
  // into d: 16-element steps kk = warp, warp + W, ... in increasing order, the
  // last 8 elements (kl % 16 == 8) by the warp whose turn it is.
  __device__ __forceinline__ void mma_kblock(const PartialArgs& a, int st, int kl,
                                             float (&d)[4]) const {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // ldmatrix row addresses of this lane: A (ranks) rows and x (tokens) rows
    const int arow = (lane & 7) + (BN == 16 ? 8 * ((lane >> 3) & 1) : 0);
    const int achunk = BN == 16 ? (lane >> 4) : ((lane >> 3) & 1);
    const int xrow = min(lane & 7, a.nrows - 1);   // this lane's token row
    const int xchunk = (lane >> 3) & 1;
    const bool wd = wide(a);
    const int n16 = kl / 16;
    const uint32_t sx = smem_u32(stages + st * kStageBytes);
    const uint32_t sa = sx + kXBytes;
    // operands of step kk (16 elements): A fragment (ranks) and x fragment (tokens)
    auto frag = [&](int kk, uint32_t (&af)[4], uint32_t (&bf)[2]) {
      const int q = kk >> 2, c16 = (kk & 3) * 2;    // sub-block, first 16-byte chunk
      if (BN == 16) {
        ldsm_x4(sa + q * BN * 128 + arow * 128 + (((c16 + achunk) ^ (arow & 7)) << 4),
                af[0], af[1], af[2], af[3]);
      } else {
        ldsm_x2(sa + q * BN * 128 + arow * 128 + (((c16 + achunk) ^ (arow & 7)) << 4),
                af[0], af[2]);
        af[1] = af[3] = 0u;
      }
      if (wd)
        ldsm_x2(sx + q * 1024 + xrow * 128 + (((c16 + xchunk) ^ xrow) << 4), bf[0], bf[1]);
      else
        ldsm_x2(sx + xrow * kRowBytes + kk * 32 + xchunk * 16, bf[0], bf[1]);
    };
    if (kl == kShrinkKB) {
      // full k-block: this warp's 16 / W steps, all operands first, then the
      // MMAs in step order (the same sequence as the loop below)
      constexpr int NS = 16 / G::WARPS;
      uint32_t af[NS][4], bf[NS][2];
#pragma unroll
      for (int i = 0; i < NS; ++i) frag(warp + i * G::WARPS, af[i], bf[i]);
#pragma unroll
      for (int i = 0; i < NS; ++i)
        mma_16816(d, af[i][0], af[i][1], af[i][2], af[i][3], bf[i][0], bf[i][1]);
    } else {
      for (int kk = warp; kk < n16; kk += G::WARPS) {
        uint32_t af[4], bf[2];
        frag(kk, af, bf);
        mma_16816(d, af[0], af[1], af[2], af[3], bf[0], bf[1]);
      }
    }
    if ((kl & 15) && warp == n16 % G::WARPS) {
      // the last 8 elements of the partition
      const int q = n16 >> 2, c = (n16 & 3) * 2;
      uint32_t a0, a1, b0;
      if (BN == 16) {
        ldsm_x2(sa + q * BN * 128 + arow * 128 + ((c ^ (arow & 7)) << 4), a0, a1);
      } else {
        ldsm_x1(sa + q * BN * 128 + arow * 128 + ((c ^ (arow & 7)) << 4), a0);
        a1 = 0u;
      }
      if (wd)
        ldsm_x1(sx + q * 1024 + xrow * 128 + ((c ^ xrow) << 4), b0);
      else
        ldsm_x1(sx + xrow * kRowBytes + n16 * 32, b0);
      mma_1688(d, a0, a1, b0);
    }
  }

  // Warp sums -> shared memory (stage 0: no copy in flight and every warp
  // done reading the stages), then thread o adds the W values of output o in
  // warp order.
  __device__ __forceinline__ void reduce_warps(const float (&d)[4], float& out) const {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* red = reinterpret_cast<float*>(stages);
    const int g = lane >> 2, t = lane & 3;
    red[warp * G::TB + (2 * t) * BN + g] = d[0];
    red[warp * G::TB + (2 * t + 1) * BN + g] = d[1];
    if (BN == 16) {
      red[warp * G::TB + (2 * t) * BN + g + 8] = d[2];
      red[warp * G::TB + (2 * t + 1) * BN + g + 8] = d[3];
    }
    __syncthreads();
    float v = red[tid];
#pragma unroll
    for (int w = 1; w < G::WARPS; ++w) v += red[w * G::TB + tid];
    out = v;
  }

  // All threads. The first min(nkb, nst) k-blocks must already be armed and
  // issued. On return `out` is this thread's output:
  // token row tid / BN, rank tid % BN (not yet scaled). Returns false if a
  // copy wait expired (after draining, bounded, every copy still in flight).
  __device__ __forceinline__ bool run(const PartialArgs& a, float& out) const {
    const int tid = threadIdx.x, warp = tid >> 5;
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int issued = min(nkb, nst);
    int fail_b = -1;
    for (int b = 0; b < nkb; ++b) {
      const int st = b % nst;
      const uint32_t parity = (uint32_t)((b / nst) & 1);
      const bool ok = mbar_wait_bounded(&bars[st], parity, a.status);
      if (__syncthreads_or(!ok)) { fail_b = b; break; }
      mma_kblock(a, st, klen(a, b), d);
      __syncthreads();
      if (b + nst < nkb) {
        if (warp == 0) {
          expect(a, b + nst);
          issue_a(a, b + nst);
          issue_x(a, b + nst);
        }
        issued = b + nst + 1;
      }
    }
    if (fail_b >= 0) {
      if (tid == 0)
        for (int bb = fail_b; bb < issued; ++bb)
          mbar_wait_bounded(&bars[bb % nst], (uint32_t)((bb / nst) & 1), a.status);
      __syncthreads();
      return false;
    }
    reduce_warps(d, out);
    return true;
  }
};

}  // namespace ig
