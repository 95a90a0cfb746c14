// The shrink partial of one tile over one K partition on CUDA cores (FP32
// FMA, warp-shuffle reduction): IG_PATH_FMA, the CUDA-core alternative to the
// warp-level tensor-core path (shrink_core.cuh). Shared by the Split-K shrink
// kernel and the fused decode kernel of this path (shrink_fma.cu,
// fused_fma.cu) so that both compute bit-identical partials.
//
// Tile: up to 8 token rows x BN rank columns (BN = 8 or 16). The block has
// BN/4 warps; warp w computes rank columns 4w .. 4w+3 for all 8 rows (32
// outputs), so every lane ends with exactly one finished output and every
// warp has work however few rows the tile holds. The partition [k0, k0 + Ks) is streamed through a ring of
// `nst` shared-memory stages, k-blocks of 256 elements, completion counted in
// bytes on one mbarrier per stage; warp 0 issues the copies. Two ways to
// copy: with tensor maps, one tiled TMA copy brings the A block (BN rows)
// and one row-gather TMA copy per 4 token rows brings x (boxes are always
// 256 wide; columns past the partition are loaded but not used); without,
// one 1-D bulk copy per row.
//
// Order of the sum, identical for every row and every M ("Reproducible LoRA
// Inference Through Deterministic Split-K Reduction" leaves the order inside
// a partition to the kernel, sec. 4.3): lane l owns the 8-element chunks
// l, l+32, ... of the partition and accumulates them in increasing k with FMA
// (two independent FMAs per packed f32x2 instruction, each rounded like
// fmaf); the 32 lane sums are then combined by a fixed xor butterfly
// (16, 8, 4, 2, 1) as a reduce-scatter. Neither the number of rows a warp
// holds nor which warp holds a row changes a row's arithmetic.
#pragma once

#include "ig_common.cuh"

namespace ig {

template <int BN>
struct FmaGeo {
  static constexpr int JPW = 4;                   // rank columns per warp
  static constexpr int WARPS = BN / JPW;          // 4 for BN = 16, 2 for BN = 8
  static constexpr int THREADS = WARPS * 32;
  static_assert(kTileRows * JPW == 32 && WARPS * JPW == BN, "shrink geometry");
};

struct FmaArgs {
  const __nv_bfloat16* x;     // x + k0
  const __nv_bfloat16* A;     // first A row of the tile's column block, + k0
  const int32_t* rows;        // token rows of the tile (shared memory)
  uint32_t* status;
  int64_t K;                  // row stride of x and A, in elements
  int64_t Ks;                 // partition length
  int nrows;
  // tensor-map copies (both null: 1-D bulk copies)
  const CUtensorMap* tm_x;    // x [M][K], box 256 x 1
  const CUtensorMap* tm_a;    // A as [rows][K], box 256 x BN
  int k0;                     // partition start (column coordinate)
  int a_row;                  // row coordinate of the tile's first A row
};

template <int BN>
struct FmaRing {
  using G = FmaGeo<BN>;
  static constexpr int kRowBytes = kShrinkKB * 2;                  // 512
  static constexpr int kStageBytes = (kTileRows + BN) * kRowBytes;
  uint8_t* stages;
  uint64_t* bars;
  int nst;      // ring depth
  int nkb;      // k-blocks in the partition

  __device__ __forceinline__ uint32_t block_bytes(const FmaArgs& a, int b) const {
    return (uint32_t)(min((int64_t)kShrinkKB, a.Ks - (int64_t)b * kShrinkKB) * 2);
  }
  // warp 0: arm stage b % nst for all copies of k-block b
  __device__ __forceinline__ void expect(const FmaArgs& a, int b) const {
    uint32_t bytes;
    if (a.tm_x) bytes = (uint32_t)kRowBytes * (BN + 4 * ((a.nrows + 3) / 4));
    else bytes = block_bytes(a, b) * (uint32_t)(a.nrows + BN);
    if ((threadIdx.x & 31) == 0) mbar_arrive_expect_tx(&bars[b % nst], bytes);
    __syncwarp();
  }
  __device__ __forceinline__ void issue_a(const FmaArgs& a, int b) const {
    const int lane = threadIdx.x & 31;
    const int st = b % nst;
    uint8_t* sa = stages + st * kStageBytes + kTileRows * kRowBytes;
    if (a.tm_a) {
      if (lane == 0) tma_load_2d(sa, a.tm_a, a.k0 + b * kShrinkKB, a.a_row, &bars[st]);
      return;
    }
    const uint32_t bytes = block_bytes(a, b);
    for (int j = lane; j < BN; j += 32)
      bulk_g2s(sa + j * kRowBytes, a.A + (int64_t)j * a.K + (int64_t)b * kShrinkKB, bytes,
               &bars[st]);
  }
  __device__ __forceinline__ void issue_x(const FmaArgs& a, int b) const {
    const int lane = threadIdx.x & 31;
    const int st = b % nst;
    uint8_t* sx = stages + st * kStageBytes;
    if (a.tm_x) {
      // rows past nrows repeat the last row: loaded, never used
      if (4 * lane < a.nrows) {
        const int last = a.nrows - 1;
        tma_gather4(sx + 4 * lane * kRowBytes, a.tm_x, a.k0 + b * kShrinkKB,
                    a.rows[min(4 * lane, last)], a.rows[min(4 * lane + 1, last)],
                    a.rows[min(4 * lane + 2, last)], a.rows[min(4 * lane + 3, last)], &bars[st]);
      }
      return;
    }
    const uint32_t bytes = block_bytes(a, b);
    for (int i = lane; i < a.nrows; i += 32)
      bulk_g2s(sx + i * kRowBytes, a.x + (int64_t)a.rows[i] * a.K + (int64_t)b * kShrinkKB,
               bytes, &bars[st]);
  }

  // All threads. The first min(nkb, nst) k-blocks must already be armed and
  // issued. On return `out` is this lane's output: row lane/4, column
  // 4*warp + lane%4 (not yet scaled). Returns false if a copy wait expired
  // (after draining, bounded, every copy still in flight).
  __device__ __forceinline__ bool run(const FmaArgs& a, float& out) const {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = warp * G::JPW;
    float2 acc[kTileRows][2];   // [row][column pair]
#pragma unroll
    for (int rr = 0; rr < kTileRows; ++rr) acc[rr][0] = acc[rr][1] = make_float2(0.0f, 0.0f);

    int issued = min(nkb, nst);
    int fail_b = -1;
    for (int b = 0; b < nkb; ++b) {
      const int st = b % nst;
      const uint32_t parity = (uint32_t)((b / nst) & 1);
      const bool ok = mbar_wait_bounded(&bars[st], parity, a.status);
      if (__syncthreads_or(!ok)) { fail_b = b; break; }
      const int64_t klen = min((int64_t)kShrinkKB, a.Ks - (int64_t)b * kShrinkKB);
      if ((int64_t)lane * 8 < klen) {
        const uint8_t* sx = stages + st * kStageBytes;
        const uint8_t* sa = sx + kTileRows * kRowBytes;
        float2 aa[2][8];   // columns (j0, j0+1) and (j0+2, j0+3), element e
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          const uint4 u0 = *reinterpret_cast<const uint4*>(sa + (j0 + 2 * jp) * kRowBytes + lane * 16);
          const uint4 u1 = *reinterpret_cast<const uint4*>(sa + (j0 + 2 * jp + 1) * kRowBytes + lane * 16);
          float a0[8], a1[8];
          unpack8(u0, a0);
          unpack8(u1, a1);
#pragma unroll
          for (int e = 0; e < 8; ++e) aa[jp][e] = make_float2(a0[e], a1[e]);
        }
#pragma unroll
        for (int rr = 0; rr < kTileRows; ++rr) {
          if (rr >= a.nrows) break;
          const uint4 u = *reinterpret_cast<const uint4*>(sx + rr * kRowBytes + lane * 16);
          float xv[8];
          unpack8(u, xv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 xx = make_float2(xv[e], xv[e]);
            acc[rr][0] = __ffma2_rn(xx, aa[0][e], acc[rr][0]);
            acc[rr][1] = __ffma2_rn(xx, aa[1][e], acc[rr][1]);
          }
        }
      }
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

    // Reduce-scatter: 32 values per lane (row-major rr*4 + j) -> one per lane.
    float v[32];
#pragma unroll
    for (int rr = 0; rr < kTileRows; ++rr) {
      v[rr * 4 + 0] = acc[rr][0].x;
      v[rr * 4 + 1] = acc[rr][0].y;
      v[rr * 4 + 2] = acc[rr][1].x;
      v[rr * 4 + 3] = acc[rr][1].y;
    }
#pragma unroll
    for (int lvl = 0; lvl < 5; ++lvl) {
      const int off = 16 >> lvl;
      const int half = 32 >> (lvl + 1);
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        const float recv = __shfl_xor_sync(0xffffffffu, send, off);
        v[i] = keep + recv;
      }
    }
    out = v[0];
    return true;
  }
};

}  // namespace ig
