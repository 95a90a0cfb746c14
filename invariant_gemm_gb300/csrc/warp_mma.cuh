// Warp-level tensor-core helpers for the small-rank (decode) path: ldmatrix
// loads and the bf16 mma.sync shapes m16n8k16 / m16n8k8 with FP32
// accumulation, plus the 128-byte-swizzled shared-memory addressing that the
// TMA copies of the path produce.
//
// Why warp-level MMA here and tcgen05 on the prefill path: a decode tile is
// 8 tokens x 8 or 16 ranks. tcgen05.mma needs M >= 64 with both operands in
// shared memory, so most of what it would read would be padding; m16n8k16 is
// exactly 16 ranks x 8 tokens x 16 k (or 16 columns x 8 tokens x 16 ranks in
// the expand), with its operands in registers.
//
// Fragment layouts (PTX ISA, mma.m16n8k16 / m16n8k8 with .bf16, .row.col),
// lane = 4 g + t:
//   A (16 x 16): reg0 (row g, k 2t..2t+1), reg1 (row g+8, k 2t..),
//                reg2 (row g, k 2t+8..),  reg3 (row g+8, k 2t+8..)
//   A (16 x 8):  reg0 (row g, k 2t..),    reg1 (row g+8, k 2t..)
//   B (16 x 8):  reg0 (k 2t..2t+1, col g), reg1 (k 2t+8.., col g)
//   B (8 x 8):   reg0 (k 2t..2t+1, col g)
//   D (16 x 8):  d0 (row g, col 2t), d1 (row g, col 2t+1),
//                d2 (row g+8, col 2t), d3 (row g+8, col 2t+1)
// ldmatrix .m8n8 gives lane 4g + t the elements 2t, 2t+1 of row g of each
// 8 x 8 matrix; lanes 8i .. 8i+7 supply the row addresses of matrix i.
#pragma once

#include "ig_common.cuh"

namespace ig {

// Byte offset of element e (a multiple of 8) in a buffer of 128-byte rows of
// 64 bf16 written by a TMA copy with 128-byte swizzle (buffer 1024-aligned):
// the 16-byte chunk q of row R sits at chunk position q ^ (R % 8).
__device__ __forceinline__ uint32_t swz128(uint32_t e) {
  const uint32_t R = e >> 6, q = (e >> 3) & 7;
  return (R << 7) | ((q ^ (R & 7)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x1(uint32_t addr, uint32_t& r0) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x1.shared.b16 {%0}, [%1];" : "=r"(r0) : "r"(addr));
}

// d = A B + d, A 16 x 16, B 16 x 8 (bf16), d FP32 (registers only: not
// volatile, so the compiler may schedule it; the ldmatrix loads stay volatile
// to keep them behind the waits that publish their shared memory)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// d = A B + d, A 16 x 8, B 8 x 8 (bf16), d FP32
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5}, {%6}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// Round-to-nearest-even bf16 bits of an FP32 value, as the low half.
__device__ __forceinline__ uint32_t bf16_bits(float f) { return f32_to_bf16_bits(f); }

// The expand on the tensor cores, one group of 32 output columns at a time:
//   D[c][m] = sum over j of B[c][j] * Zb[m][j]   (c: 16 columns, m: 8 tokens)
// one m16n8k16 per 16 columns and 16-element j chunk (m16n8k8 for a last 8),
// the B rows as the A operand (ldmatrix from the swizzled B slice) and the
// tile's Zb rows as the B operand (registers); j chunks in increasing order,
// with three Z parts (FP32 Z) the hi, mid and lo MMAs of a chunk follow each
// other. A group is 2 MMAs (h = 0, 1): MMA row g of MMA h is the group's
// column 4g + 2h and row g + 8 its column 4g + 2h + 1, so that lane 4g + t
// ends with columns 4g .. 4g+3 of tokens 2t (v[0..3]) and 2t + 1 (v[4..7]),
// all four accumulator registers used, and updates them in y with one 8-byte
// load and store per token. Which MMA computes a column does not change its
// value: every element is one dot product over all of j, in the same order.
// Under the 128-byte swizzle the 8 column addresses of one 8x8 matrix fall
// in 8 distinct bank groups for r = 8 and r = 16.
// zb: bf16 [parts][8][r] in shared memory; sB: the block's B columns,
// column c at elements c * r .. c * r + r - 1 of a 128-byte-swizzled buffer
// (see swz128); cb: the group's first column; columns past cmax are read as
// column cmax (their results are not used).
__device__ __forceinline__ void expand_group_mma(float (&v)[8], uint32_t sB_addr, int cb,
                                                 int cmax, int r, const uint16_t* zb,
                                                 int parts, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;    // the 8x8 matrix and row this lane addresses
  const uint32_t* z32 = reinterpret_cast<const uint32_t*>(zb);
  const int zrow = g * (r / 2);               // token g's Z row, in bf16 pairs
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int c = min(cb + 4 * rr + (mi & 1) + 2 * h, cmax);
    int j = 0;
    for (; j + 16 <= r; j += 16) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sB_addr + swz128((uint32_t)(c * r + j + (mi >> 1) * 8)), a0, a1, a2, a3);
#pragma unroll 1
      for (int q = 0; q < parts; ++q) {
        const uint32_t* zp = z32 + q * 4 * r + zrow + j / 2 + t;
        mma_16816(d, a0, a1, a2, a3, zp[0], zp[4]);
      }
    }
    if (j < r) {   // last 8 elements
      uint32_t a0, a1;
      ldsm_x2(sB_addr + swz128((uint32_t)(c * r + j)), a0, a1);
#pragma unroll 1
      for (int q = 0; q < parts; ++q) {
        const uint32_t* zp = z32 + q * 4 * r + zrow + j / 2 + t;
        mma_1688(d, a0, a1, zp[0]);
      }
    }
    v[2 * h] = d[0];
    v[2 * h + 1] = d[2];
    v[4 + 2 * h] = d[1];
    v[5 + 2 * h] = d[3];
  }
}

// The same MMAs as expand_group_mma for r = R (16 or 8) and one Z part,
// split into operand loads and MMAs, with the ldmatrix addresses computed
// once per lane.
template <int R>
struct ExpandFrag {
  uint32_t zb0, zb1;   // Zb fragment: token g, j 2t..2t+1 and j 2t+8..2t+9 (R = 16)
  __device__ __forceinline__ void load_z(const uint16_t* zb, int lane) {
    const uint32_t* z32 = reinterpret_cast<const uint32_t*>(zb) + (lane >> 2) * (R / 2) +
                          (lane & 3);
    zb0 = z32[0];
    zb1 = R == 16 ? z32[4] : 0u;
  }
  // Byte offsets, from the start of a pair of groups in the B buffer, of the
  // B rows this lane addresses in the 2 MMAs of a group of parity `par`:
  // two groups span 64 columns x R elements = R 128-byte rows, a multiple of
  // 8, so the swizzle pattern repeats from one pair to the next.
  __device__ __forceinline__ static void lane_offsets(int lane, int par, uint32_t (&off)[2]) {
    const int mi = lane >> 3, rr = lane & 7;
    const int jsel = R == 16 ? (mi >> 1) * 8 : 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      off[h] = swz128((uint32_t)((32 * par + 4 * rr + (mi & 1) + 2 * h) * R + jsel));
  }
  // A operands of the group whose pair starts at byte `base` of the B buffer
  // (group g: base = sB + (g / 2) * 128 * R, offsets of parity g % 2); the
  // buffer holds whole groups, so no column needs clamping.
  __device__ __forceinline__ static void load_b_at(uint32_t base, const uint32_t (&off)[2],
                                                   uint32_t (&a)[2][4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (R == 16) {
        ldsm_x4(base + off[h], a[h][0], a[h][1], a[h][2], a[h][3]);
      } else {
        ldsm_x2(base + off[h], a[h][0], a[h][1]);
        a[h][2] = a[h][3] = 0u;
      }
    }
  }
  __device__ __forceinline__ void mma(float (&v)[8], const uint32_t (&a)[2][4]) const {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (R == 16) mma_16816(d, a[h][0], a[h][1], a[h][2], a[h][3], zb0, zb1);
      else mma_1688(d, a[h][0], a[h][1], zb0);
      v[2 * h] = d[0];
      v[2 * h + 1] = d[2];
      v[4 + 2 * h] = d[1];
      v[5 + 2 * h] = d[3];
    }
  }
};

// y = bf16_rn(f32(y) + v) for 4 consecutive bf16 values (one rounding each).
__device__ __forceinline__ uint2 y_add4(const uint2& y, float v0, float v1, float v2, float v3) {
  uint2 o;
  o.x = f32x2_to_bf16x2_bits(bf16lo(y.x) + v0, bf16hi(y.x) + v1);
  o.y = f32x2_to_bf16x2_bits(bf16lo(y.y) + v2, bf16hi(y.y) + v3);
  return o;
}

}  // namespace ig
