// The shrink partial of one tile over one K partition, on the warp-level
// tensor cores. Shared by the Split-K shrink kernel and the fused decode
// kernel so that both compute bit-identical partials.
//
// Tile: up to 8 token rows x BN rank columns (BN = 8 or 16); the block has
// W = BN/4 warps (4 or 2) and ends with one output per thread: thread o holds
// the partial of token row o / BN, rank o % BN.
//
// Operands. The partition [k0, k0 + Ks) is cut into 64-element groups. The
// BN A rows stream through a ring of `nst` shared-memory stages of 256
// elements (4 groups), 128-byte swizzled by TMA (one 3-D copy per stage when
// K and K/S are multiples of 64, else one 2-D copy per group); completion is
// counted in bytes on one mbarrier per stage. x does not go through shared
// memory: lane 4g + t loads the 16-byte chunks 2t and 2t+1 of a group of its
// token row g straight into registers (the rows past nrows repeat the tile's
// last row; never used), and reads the same two chunks of A rows g and g + 8
// with 16-byte shared-memory loads (under the swizzle the 8 chunks that a
// quarter warp reads sit in 8 distinct bank groups). With static weights and
// a partition of at most two k-blocks (decode), the A chunks are read into
// registers before the dependency wait, so that after it only the x loads
// and the MMAs remain.
//
// The contraction of a group is 4 bf16 MMAs m16n8k16 (16 ranks x 8 tokens
// x 16 k), u = 0..3: in MMA u the k slots 2t, 2t+1 hold the group's elements
// 16t + 2u, 16t + 2u + 1 and the slots 2t + 8, 2t + 9 hold 16t + 8 + 2u,
// 16t + 9 + 2u. A and x use the same slot map, so the 4 MMAs add each of the
// group's 64 products exactly once. Elements past the partition end are zero
// in both operands (ranks 8..15 are zero when BN = 8).
//
// Order of the sum, identical for every row and every M ("Reproducible LoRA
// Inference Through Deterministic Split-K Reduction" leaves the order inside
// a partition to the kernel, sec. 4.3): group G belongs to warp G % W; a warp
// takes its groups in increasing G and accumulates MMAs u = 0, 2 into FP32
// accumulator E and u = 1, 3 into accumulator O, then D = E + O; the W warp
// sums are added in warp order: ((D0 + D1) + D2) + D3. A token's value
// depends only on its own x row: the MMA's columns are independent.
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
  const __nv_bfloat16* x;     // x [M][K]
  int64_t K;                  // row stride of x, in elements
  int Ks;                     // partition length (K < 2^31)
  int nrows;
  const CUtensorMap* tm_a;    // A as [rows][K], box 64 x BN, 128-byte swizzle
  const CUtensorMap* tm_a3;   // A as {64, rows, K/64}, box {64, BN, 4}, or null
  int k0;                     // partition start (column coordinate)
  int a_row;                  // row coordinate of the tile's first A row
  long long first_budget;     // budget of the first A-copy wait (clocks; <= 0:
                              // one check, IG_FLAG_TEST_COPY_TIMEOUT)
};

// Budget of a block's first A-copy wait for the given ig_shape flags.
__host__ __device__ inline long long first_copy_budget(int flags) {
  return (flags & IG_FLAG_TEST_COPY_TIMEOUT) ? 0ll : (1ll << 31);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

template <int BN>
struct PartialRing {
  using G = ShrinkGeo<BN>;
  static constexpr int W = G::WARPS;
  static constexpr int kGroups = kShrinkKB / 64;          // 64-element groups per k-block
  static constexpr int NGW = kGroups / W;                 // groups per warp per k-block
  static constexpr int kStageBytes = kGroups * BN * 128;  // [group][BN rows][128 B]
  static constexpr int kRedBytes = W * G::TB * 4;         // warp sums for the reduce
  static constexpr int kAF = BN == 16 ? 4 : 2;            // A chunks of a group per lane
  // Register-resident path: with static weights and a partition of at most
  // kFastKB k-blocks, every A chunk a lane needs is loaded into registers
  // before the dependency wait (A is not written by the previous kernel).
  static constexpr int kFastKB = 2;
  uint8_t* stages;   // 1024-aligned
  uint64_t* bars;
  int nst;      // ring depth
  int nkb;      // k-blocks in the partition

  using XRegs = uint4[NGW][2];     // x chunks 2t, 2t+1 of the warp's groups in one k-block
  using ARegs = uint4[NGW][kAF];   // A chunks (rows g, g + 8) of the same groups

  __device__ __forceinline__ int klen(const PartialArgs& a, int b) const {
    return min(kShrinkKB, a.Ks - b * kShrinkKB);
  }
  __device__ __forceinline__ int nsub(const PartialArgs& a, int b) const {
    return (klen(a, b) + 63) / 64;
  }
  __device__ __forceinline__ bool fast(bool static_weights) const {
    return static_weights && nkb <= kFastKB && nkb <= nst;
  }
  // warp 0: arm stage b % nst for the A copies of k-block b
  __device__ __forceinline__ void expect(const PartialArgs& a, int b) const {
    if ((threadIdx.x & 31) == 0)
      mbar_arrive_expect_tx(&bars[b % nst], (uint32_t)nsub(a, b) * 128u * BN);
    __syncwarp();
  }
  __device__ __forceinline__ void issue_a(const PartialArgs& a, int b) const {
    if ((threadIdx.x & 31) != 0) return;
    const int st = b % nst;
    uint8_t* sa = stages + st * kStageBytes;
    const int ns = nsub(a, b);
    if (a.tm_a3 && ns == kGroups) {   // the four groups in one copy (same layout)
      tma_load_3d(sa, a.tm_a3, 0, a.a_row, (a.k0 + b * kShrinkKB) / 64, &bars[st]);
      return;
    }
    for (int q = 0; q < ns; ++q)
      tma_load_2d(sa + q * BN * 128, a.tm_a, a.k0 + b * kShrinkKB + q * 64, a.a_row, &bars[st]);
  }

  // This lane's x row from the partition start (token row g; rows past
  // nrows repeat the tile's last row).
  __device__ __forceinline__ const __nv_bfloat16* x_row(const PartialArgs& a) const {
    const int g = (threadIdx.x & 31) >> 2;
    return a.x + (int64_t)a.rows[min(g, a.nrows - 1)] * a.K + a.k0;
  }
  // This lane's x chunks of k-block b: for each of the warp's groups, chunks
  // 2t and 2t+1 (zero past the partition). L2 only: x may have been written
  // by the previous kernel.
  __device__ __forceinline__ void load_x(const __nv_bfloat16* xrow, const PartialArgs& a, int b,
                                         XRegs& xr) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = lane & 3;
#pragma unroll
    for (int i = 0; i < NGW; ++i) {
      const int e = (kGroups * b + warp + W * i) * 64 + 16 * t;
      xr[i][0] = e < a.Ks ? ldg_cg_v4(xrow + e) : make_uint4(0u, 0u, 0u, 0u);
      xr[i][1] = e + 8 < a.Ks ? ldg_cg_v4(xrow + e + 8) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // This lane's A chunks of k-block b from stage st: chunks 2t, 2t+1 of rows
  // g (and g + 8), zero past the partition. Under the 128-byte swizzle chunk
  // c of row R sits at position c ^ (R % 8); rows g and g + 8 share it.
  __device__ __forceinline__ void load_a(const PartialArgs& a, int st, int b, ARegs& ar) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t sa = smem_u32(stages + st * kStageBytes);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < NGW; ++i) {
      const int q = warp + W * i;                    // group within the k-block
      const int e = (kGroups * b + q) * 64 + 16 * t;
      const bool vlo = e < a.Ks, vhi = e + 8 < a.Ks;
      const uint32_t row = sa + q * BN * 128 + g * 128;
      const uint32_t clo = (uint32_t)(((2 * t) ^ g) << 4), chi = (uint32_t)(((2 * t + 1) ^ g) << 4);
      ar[i][0] = vlo ? lds128(row + clo) : zero;
      ar[i][1] = vhi ? lds128(row + chi) : zero;
      if (BN == 16) {
        ar[i][kAF - 2] = vlo ? lds128(row + 8 * 128 + clo) : zero;
        ar[i][kAF - 1] = vhi ? lds128(row + 8 * 128 + chi) : zero;
      }
    }
  }
  // The 4 MMAs of each of the warp's groups of k-block b: u = 0, 2 into dE,
  // u = 1, 3 into dO (groups past the partition skipped, whole warp).
  __device__ __forceinline__ void mma(const PartialArgs& a, int b, const ARegs& ar,
                                      const XRegs& xr, float (&dE)[4], float (&dO)[4]) const {
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < NGW; ++i) {
      if ((kGroups * b + warp + W * i) * 64 >= a.Ks) continue;
      const uint4& lo = ar[i][0];
      const uint4& hi = ar[i][1];
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      const uint4& lo8 = BN == 16 ? ar[i][kAF - 2] : zero;
      const uint4& hi8 = BN == 16 ? ar[i][kAF - 1] : zero;
      const uint4& xl = xr[i][0];
      const uint4& xh = xr[i][1];
      mma_16816(dE, lo.x, lo8.x, hi.x, hi8.x, xl.x, xh.x);
      mma_16816(dO, lo.y, lo8.y, hi.y, hi8.y, xl.y, xh.y);
      mma_16816(dE, lo.z, lo8.z, hi.z, hi8.z, xl.z, xh.z);
      mma_16816(dO, lo.w, lo8.w, hi.w, hi8.w, xl.w, xh.w);
    }
  }

  // Warp sums -> shared memory, then thread o adds the W values of output o
  // in warp order. `failed` must be uniform over the block or false; ok is
  // this thread's own. On failure thread 0 waits (bounded) for the last
  // k-block issued on each stage, the only phase that may be outstanding.
  __device__ __forceinline__ bool finish(const PartialArgs& a, const float (&dE)[4],
                                         const float (&dO)[4], bool ok, bool failed, int issued,
                                         float* red, float& out) const {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    float* rw = red + warp * G::TB;
    rw[(2 * t) * BN + g] = dE[0] + dO[0];
    rw[(2 * t + 1) * BN + g] = dE[1] + dO[1];
    if (BN == 16) {
      rw[(2 * t) * BN + g + 8] = dE[2] + dO[2];
      rw[(2 * t + 1) * BN + g + 8] = dE[3] + dO[3];
    }
    if (!failed) failed = __syncthreads_or(!ok);
    if (failed) {
      if (tid == 0)
        for (int bb = max(0, issued - nst); bb < issued; ++bb)
          mbar_wait_bounded(&bars[bb % nst], (uint32_t)((bb / nst) & 1), a.status);
      __syncthreads();
      return false;
    }
    float v = red[tid];
#pragma unroll
    for (int w = 1; w < W; ++w) v += red[w * G::TB + tid];
    out = v;
    return true;
  }

  // Register-resident path, before the dependency wait (all threads): wait
  // for the A copies of every k-block (armed and issued) and load this lane's
  // chunks. Returns false if a wait expired.
  __device__ __forceinline__ bool fast_prologue(const PartialArgs& a,
                                                ARegs (&ar)[kFastKB]) const {
    bool ok = true;
#pragma unroll
    for (int b = 0; b < kFastKB; ++b) {
      if (b < nkb && ok)
        ok = mbar_wait_bounded(&bars[b], 0u, a.status, b == 0 ? a.first_budget : 1ll << 31);
      if (b < nkb && ok) load_a(a, b, b, ar[b]);
    }
    return ok;
  }
  // Register-resident path, after the dependency wait: x loads, then
  // `after_x` (the fused kernel issues its y loads there), then the MMAs.
  template <typename F>
  __device__ __forceinline__ bool fast_run(const PartialArgs& a, const __nv_bfloat16* xrow,
                                           const ARegs (&ar)[kFastKB], bool ok, float* red,
                                           float& out, F&& after_x) const {
    XRegs xr[kFastKB];
#pragma unroll
    for (int b = 0; b < kFastKB; ++b)
      if (b < nkb) load_x(xrow, a, b, xr[b]);
    after_x();
    float dE[4] = {0.0f, 0.0f, 0.0f, 0.0f}, dO[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int b = 0; b < kFastKB; ++b)
      if (b < nkb && ok) mma(a, b, ar[b], xr[b], dE, dO);
    return finish(a, dE, dO, ok, false, nkb, red, out);
  }

  // Streaming path (all threads): the A copies of the first min(nkb, nst)
  // k-blocks must already be armed (and issued, or issued by warp 0 before
  // any wait could time out); later k-blocks are refilled into their stage
  // once every warp is done with it. `after_first_x` runs once, right after
  // this lane's x loads of the first k-blocks are issued. `red` holds
  // kRedBytes of shared memory used by nothing else meanwhile. On return
  // `out` is this thread's output: token row tid / BN, rank tid % BN (not yet
  // scaled). Returns false if a copy wait expired (after draining, bounded,
  // every copy still in flight).
  template <typename F>
  __device__ __forceinline__ bool run(const PartialArgs& a, const __nv_bfloat16* xrow, float* red,
                                      float& out, F&& after_first_x) const {
    const int warp = threadIdx.x >> 5;
    float dE[4] = {0.0f, 0.0f, 0.0f, 0.0f}, dO[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    XRegs xc, xn;
    load_x(xrow, a, 0, xc);
    int issued = min(nkb, nst);   // k-blocks whose A copies are armed and issued
    bool ok = true, failed = false;
    for (int b = 0; b < nkb; ++b) {
      if (b + 1 < nkb) load_x(xrow, a, b + 1, xn);
      if (b == 0) after_first_x();
      const int st = b % nst;
      if (ok)
        ok = mbar_wait_bounded(&bars[st], (uint32_t)((b / nst) & 1), a.status,
                               b == 0 ? a.first_budget : 1ll << 31);
      if (ok) {
        ARegs ar;
        load_a(a, st, b, ar);
        mma(a, b, ar, xc, dE, dO);
      }
      if (b + nst < nkb) {
        // stage st is refilled: every warp must be done reading it
        if (__syncthreads_or(!ok)) { failed = true; break; }
        if (warp == 0) {
          expect(a, b + nst);
          issue_a(a, b + nst);
        }
        issued = b + nst + 1;
      }
#pragma unroll
      for (int i = 0; i < NGW; ++i) {
        xc[i][0] = xn[i][0];
        xc[i][1] = xn[i][1];
      }
    }
    return finish(a, dE, dO, ok, failed, issued, red, out);
  }
};

}  // namespace ig
