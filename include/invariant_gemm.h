/*
 * invariant_gemm — multi-adapter LoRA shrink / expand with a deterministic
 * Split-K reduction, for NVIDIA GB300 (sm_103a).
 *
 * The operations follow "Reproducible LoRA Inference Through Deterministic
 * Split-K Reduction" (Balusamy & Mohan):
 *   - Eq. 1: a LoRA linear layer computes Y = X W^T + s (X A^T) B^T with
 *     A in R^{r x H} and B in R^{Hout x r}. The shrink is Z = s X A^T (narrow,
 *     r columns); the expand adds Z B^T to Y.
 *   - Eq. 3 / Fig. 1: Split-K partitions the reduction index H into S parts,
 *     one thread block per (output tile, part).
 *   - Algorithm 1 / Fig. 2 / sec. 4.3: each block stores an FP32 partial into
 *     scratch, fences, and bumps a per-tile integer counter; the block that
 *     sees the previous value S-1 sums the S partials in increasing partition
 *     order, multiplies by the scale, writes the tile and resets the counter.
 *   - sec. 4.1: the atomic Split-K baseline adds partials with FP32 atomics.
 *   - sec. 4.2: the unsplit baseline (Split-K = 1) uses one block per tile.
 *   - sec. 4.3: an earlier deterministic design combined the partials in a
 *     separate kernel with a fixed pairwise tree (IG_MODE_DET_TREE).
 *   - sec. 6.2 / Fig. 5: the FP32 shrink output is rounded to BF16
 *     (round-to-nearest, ties to even) where the next operation reads it.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers, owned by the caller, and must
 *     stay valid until the work queued on `stream` has finished. The library
 *     allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call only enqueues work; none synchronises, except
 *     ig_check_status.
 *   - Layouts are dense row-major with the last index contiguous. bf16 is
 *     IEEE binary32 with the low 16 bits dropped, stored as 2 bytes.
 *       x        bf16  [M][K]
 *       A_stack  bf16  [L][slices][r][K]      (L = num_adapters)
 *       B_stack  bf16  [L][slices][N][r]
 *       z        f32   [slices][M][r]
 *       y        bf16  [M][slices*N]          (updated in place)
 *       adapter_idx int32 [M]; value a in [0, L) selects adapter a, -1 means
 *                the token has no adapter (its z row is 0 and its y row is
 *                left untouched). Any other value is an error: the row is
 *                treated as -1 and the device status word records
 *                IG_ERR_ADAPTER_RANGE (see ig_check_status).
 *   - Every pointer must be 16-byte aligned; K, N and r must be multiples of
 *     8 (so rows are whole 16-byte vectors).
 *   - Return value: IG_OK, or a negative ig_status. Argument errors are
 *     detected on the host before anything is enqueued. IG_ERR_CUDA reports
 *     a failed launch (cudaGetLastError).
 *   - Overlap: shrink and expand kernels are launched with programmatic
 *     dependent launch. A kernel may start while the previous kernel on the
 *     stream finishes, but it reads activations, z, y and the workspace
 *     (other than the token map) and writes anything only after that kernel
 *     has completed; only the token map (which is always complete before any
 *     later kernel starts) and, with IG_FLAG_STATIC_WEIGHTS, A_stack/B_stack
 *     are read earlier.
 *   - Determinism: in IG_MODE_DET, IG_MODE_DET_TREE and IG_MODE_UNSPLIT the
 *     bits of each z row
 *     and y row are a function of that row's inputs, its adapter and the plan
 *     only. The plan (ig_plan_query) is a function of
 *     (K, r, N, slices, split_k, mode, path) and never of M, so results do not
 *     depend on the batch size, the other rows of the batch, the row's
 *     position, or the run. IG_MODE_ATOMIC has no such property.
 */
#ifndef INVARIANT_GEMM_H
#define INVARIANT_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IG_ABI_VERSION 1

typedef enum ig_status {
  IG_OK = 0,
  IG_ERR_ARG = -1,           /* null pointer or invalid enum value */
  IG_ERR_SHAPE = -2,         /* sizes invalid or not divisible as required */
  IG_ERR_ALIGN = -3,         /* a pointer is not 16-byte aligned */
  IG_ERR_WS_SMALL = -4,      /* workspace smaller than ig_workspace_bytes */
  IG_ERR_CUDA = -5,          /* a CUDA runtime call failed */
  IG_ERR_WS_CORRUPT = -6,    /* device: a completion counter held a value >= S */
  IG_ERR_ADAPTER_RANGE = -7, /* device: an adapter index outside [-1, L) */
  IG_ERR_TIMEOUT = -8,       /* device: a bounded wait expired */
  IG_ERR_UNSUPPORTED = -9    /* valid request outside this build's limits */
} ig_status;

/* Reduction variant of the shrink (sec. 4.1-4.3). */
typedef enum ig_mode {
  IG_MODE_DET = 0,     /* Split-K with FP32 partials in the workspace and a
                          last-arriver fixed-order combine (Algorithm 1) */
  IG_MODE_ATOMIC = 1,  /* Split-K with FP32 atomic adds into a zeroed z */
  IG_MODE_UNSPLIT = 2, /* Split-K = 1: one block per output tile */
  IG_MODE_DET_TREE = 3 /* Split-K with FP32 partials in the workspace, summed by
                          a second kernel with a fixed pairwise tree
                          ((P0+P1)+(P2+P3))+...: the earlier deterministic
                          design the pages describe in sec. 4.3 */
} ig_mode;

/* Arithmetic path. It is part of the determinism key: the same request on
 * another path gives results within tolerance but not bit-equal. */
typedef enum ig_path {
  IG_PATH_AUTO = 0,  /* chosen from (K, r, N, slices, flags) only, never
                        from M: IG_PATH_MMA for r >= 32 where it applies,
                        else IG_PATH_WARP */
  IG_PATH_WARP = 1,  /* small ranks: 8-token tiles on the warp-level tensor
                        cores (bf16 mma.sync m16n8k16, FP32 accumulation) */
  IG_PATH_MMA = 2,   /* 128-token tiles on the tcgen05 tensor cores, FP32
                        accumulation in TMEM; needs r and K/S multiples of
                        16, and r <= 192 with IG_FLAG_Z_FP32
                        (IG_ERR_UNSUPPORTED otherwise) */
  IG_PATH_FMA = 3    /* small ranks on CUDA cores: 8-token tiles, FP32 FMA in
                        increasing k per lane, warp-shuffle butterfly across
                        lanes; never chosen by IG_PATH_AUTO (the warp path
                        measured faster), kept as the CUDA-core baseline */
} ig_path;

typedef struct ig_shape {
  int64_t M;            /* tokens: rows of x, z and y; 0 is a valid no-op */
  int64_t K;            /* hidden size H: reduction length of the shrink
                           (< 2^31) */
  int64_t N;            /* output features per slice (Hout, < 2^31) */
  int64_t r;            /* adapter rank */
  int32_t slices;       /* stacked projections that share x, e.g. 3 for QKV */
  int32_t num_adapters; /* L: adapters held in A_stack and B_stack */
  int32_t split_k;      /* S: partitions of K; (K/8) % S == 0. Ignored (1)
                           in IG_MODE_UNSPLIT */
  int32_t mode;         /* ig_mode */
  int32_t path;         /* ig_path */
  int32_t flags;        /* 0 or IG_FLAG_* bits */
} ig_shape;

/* ig_shape.flags bits. */
#define IG_FLAG_STATIC_WEIGHTS 1 /* A_stack and B_stack are not written by any
                                    work still running on `stream` when the
                                    call is enqueued (true for inference
                                    weights). Lets a kernel start reading
                                    them while the previous kernel on the
                                    stream is still finishing. */
#define IG_FLAG_UNFUSED 2        /* IG_MODE_DET combines through the
                                    workspace with the completion counter
                                    (Algorithm 1) even where a cluster
                                    combine applies: lora_apply runs the
                                    Split-K shrink and the expand as two
                                    kernels instead of the fused one-launch
                                    kernel, and the tcgen05 shrink does not
                                    combine inside a thread-block cluster.
                                    Both give the same bits. */
#define IG_FLAG_Z_FP32 4         /* The expand reads Z in FP32 instead of
                                    rounding it to bf16 first (sec. 6.2 shows
                                    the bf16 boundary turning tiny FP32
                                    differences into visible ones). Tensor-
                                    core paths: Z = hi + mid + lo exactly,
                                    hi = bf16_rn(Z), mid = bf16_rn(Z - hi),
                                    lo = bf16_rn(Z - hi - mid), three MMAs
                                    per step of the rank sum; FMA path: Z
                                    used as stored. */

#define IG_FLAG_INPUT_READY 16   /* With IG_FLAG_STATIC_WEIGHTS: x is not written
                                    by any work still running on `stream`
                                    when the call is enqueued (true when x is
                                    the input of a base GEMM that runs just
                                    before the LoRA call, or comes from an
                                    earlier layer). The fused decode kernel
                                    of the warp path (lora_apply with
                                    ig_plan_info.apply_kernels == 1, not
                                    IG_PATH_FMA) then runs its shrink,
                                    partial exchange and combine while the
                                    previous kernel on the stream is still
                                    finishing; z and y are still read and
                                    written only after it has completed.
                                    Other kernels ignore the flag. Same
                                    results; not part of the determinism
                                    key. */
#define IG_FLAG_TEST_COPY_TIMEOUT 8 /* For testing the timeout path only; never
                                    set it in production. Warp-path shrink
                                    kernels (lora_shrink, and lora_apply's
                                    fused kernel) give their first A-copy wait
                                    no time at all: each block checks that
                                    copy once, right after issuing it, finds it
                                    still in flight, records IG_ERR_TIMEOUT,
                                    waits (bounded) for its own copies to land
                                    and leaves. The call's z and y are then
                                    unspecified, and ig_check_status reports
                                    IG_ERR_TIMEOUT and re-zeroes the counters.
                                    Not part of the determinism key. */

/* The resolved plan. Everything that fixes the arithmetic is in
 * determinism_key, which never depends on M. */
typedef struct ig_plan_info {
  int32_t path;             /* IG_PATH_WARP, IG_PATH_MMA or IG_PATH_FMA */
  int32_t split_k;          /* S used (1 for IG_MODE_UNSPLIT) */
  int64_t k_split;          /* K / S: elements per partition */
  int32_t shrink_bm;        /* shrink output tile: token rows ... */
  int32_t shrink_bn;        /* ... x rank columns */
  int32_t expand_bm;        /* expand tile: token rows ... */
  int32_t expand_bn;        /* ... x output columns */
  int64_t shrink_tiles_max; /* upper bound on shrink output tiles for this M */
  int64_t shrink_ctas_max;  /* shrink grid size for this M */
  int64_t workspace_bytes;  /* same as ig_workspace_bytes */
  uint64_t determinism_key; /* hash of the arithmetic-defining plan fields */
  int32_t apply_kernels;    /* kernels lora_apply launches after the token
                               map: 1 = fused shrink+expand (IG_MODE_DET,
                               r = 8 or 16, S <= 16, warp or FMA path), 2 = shrink
                               then expand */
  int32_t reserved;
} ig_plan_info;

/* Library version string and a message for a status code. Host only. */
const char* ig_version(void);
const char* ig_status_string(int status);

/* Bytes of device workspace a call with this shape needs: status word,
 * per-tile completion counters, the token map (rows grouped by adapter),
 * for IG_MODE_DET and IG_MODE_DET_TREE the FP32 partials [tiles][S][BM x BN],
 * and on the tcgen05 path in IG_MODE_DET and IG_MODE_UNSPLIT the expand's Z
 * operand that the shrink of lora_apply writes (bf16 z per tile, slice and
 * bf16 part). Returns 0 for an invalid shape. Host only. */
size_t ig_workspace_bytes(const ig_shape* shape);

/* Resolve the plan for a shape without touching the GPU. IG_OK or an
 * argument error. */
int ig_plan_query(const ig_shape* shape, ig_plan_info* out);

/* Zero the workspace's status word and completion counters (enqueued on
 * stream). Call once after allocating a workspace: afterwards the counters
 * reset themselves (Algorithm 1: the last block writes 0 back). */
int ig_workspace_init(void* ws, size_t ws_bytes, const ig_shape* shape, void* stream);

/* Group the tokens by adapter: a stable counting sort of adapter_idx[0..M)
 * written into the workspace's token map. lora_shrink, lora_expand and
 * lora_apply build the map themselves when given a non-NULL adapter_idx;
 * calling this once and then passing adapter_idx = NULL to several calls
 * with the same M, num_adapters and workspace reuses it (one map per batch,
 * shared by every LoRA layer of a forward pass). Supports num_adapters up to
 * 1023. */
int ig_map_tokens(const ig_shape* shape, const int32_t* adapter_idx,
                  void* ws, size_t ws_bytes, void* stream);

/* Shrink (Eq. 1, Eq. 3, Algorithm 1):
 *   z[sl][m][j] = scale * sum_k x[m][k] * A_stack[a_m][sl][j][k]
 * with FP32 accumulation of exact bf16 x bf16 products. The reduction over k
 * follows shape->mode; in IG_MODE_DET the S partials of a tile are summed in
 * increasing partition order by the last block to finish, then multiplied by
 * scale. IG_MODE_ATOMIC zeroes z (cudaMemsetAsync) and then adds
 * scale * partial with FP32 atomics. adapter_idx may be NULL to reuse the
 * token map already in ws (see ig_map_tokens). */
int lora_shrink(const ig_shape* shape, const void* x, const void* A_stack,
                const int32_t* adapter_idx, float scale, float* z,
                void* ws, size_t ws_bytes, void* stream);

/* Expand (Eq. 1, sec. 6.2):
 *   y[m][sl*N + n] = bf16_rn( f32(y[m][sl*N+n])
 *                             + sum_{j<r} bf16_rn(z[sl][m][j]) * B_stack[a_m][sl][n][j] )
 * (with IG_FLAG_Z_FP32: z[sl][m][j] itself instead of bf16_rn(z); the
 * tensor-core paths feed it as three bf16 parts that sum to it exactly)
 * The sum over j is an FP32 sum whose order is fixed by r and the path, not
 * by M: on the tensor-core paths (IG_PATH_WARP, IG_PATH_MMA) the rank axis
 * is taken in chunks of 16 in increasing order, one MMA per chunk, each
 * adding its 16 products into the FP32 accumulator inside the tensor core;
 * on IG_PATH_FMA a sequential FMA chain in increasing j. y is rounded once.
 * Rows with adapter -1 are not written. adapter_idx may be NULL to reuse the
 * token map in ws. */
int lora_expand(const ig_shape* shape, const float* z, const void* B_stack,
                const int32_t* adapter_idx, void* y,
                void* ws, size_t ws_bytes, void* stream);

/* Token map (if adapter_idx != NULL), shrink into z, then expand into y, all
 * on `stream`. z is caller-owned scratch of slices*M*r floats and holds the
 * shrink output afterwards. In IG_MODE_DET with r = 8 or 16 and S <= 16 the
 * shrink and expand run as one launch: the S partition blocks of a tile form
 * a thread-block cluster, sum their partials over distributed shared memory
 * in the same increasing partition order, and expand the tile's rows
 * (ig_plan_info.apply_kernels == 1; IG_FLAG_UNFUSED turns this off). On
 * the tcgen05 path (IG_PATH_MMA) in IG_MODE_DET and IG_MODE_UNSPLIT the
 * shrink also writes the expand's bf16 Z operand into ws, the expand copies
 * it instead of building it from z, and it starts its first y copies before
 * its dependency wait (the shrink writes no y). The results are
 * bit-identical to lora_shrink followed by lora_expand. */
int lora_apply(const ig_shape* shape, const void* x, void* y,
               const int32_t* adapter_idx, const void* A_stack,
               const void* B_stack, float scale, float* z,
               void* ws, size_t ws_bytes, void* stream);

/* lora_shrink without a caller-provided workspace. The paper has no
 * counterpart: it exists for callers that cannot allocate device memory
 * where they run the shrink (code that must not risk the device-wide
 * synchronisation an allocation can bring, runtimes that plan all memory
 * ahead and give libraries no allocator, plugin hosts that own every
 * allocation).
 *
 * Same arguments, arithmetic and results as lora_shrink (adapter_idx must be
 * non-NULL), but the token map, counters, status word and partials live in
 * a 4 MiB array inside the library, held by every GPU that loads it until
 * the process exits. This call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *   - Shapes whose shrink needs more than 4 MiB of workspace are rejected
 *     with IG_ERR_WS_SMALL before anything is enqueued. That is
 *     ig_workspace_bytes without the expand's Z operand, which only
 *     lora_apply writes.
 *   - The first call on a device looks up the array's device address (with
 *     that device current). Make that first call before any stream capture.
 *   - Every call shares the one array and it keeps the previous call's
 *     contents; each call clears the status word and the counters it uses
 *     (a memset on `stream`). Calls that overlap on the GPU (other streams,
 *     other threads) race on the array and give wrong results: serialise
 *     them.
 *   - Device-side status (out-of-range adapter index, expired wait) is not
 *     reported; validate adapter_idx beforehand. */
int lora_shrink_noalloc(const ig_shape* shape, const void* x, const void* A_stack,
                        const int32_t* adapter_idx, float scale, float* z, void* stream);

/* Synchronise `stream`, read and clear the workspace status word, and return
 * the most severe device-side error recorded since the last check
 * (IG_ERR_TIMEOUT, IG_ERR_WS_CORRUPT, IG_ERR_ADAPTER_RANGE) or IG_OK. After
 * IG_ERR_WS_CORRUPT or IG_ERR_TIMEOUT the completion counters are zeroed
 * again, so the workspace is usable for the next call. After IG_ERR_TIMEOUT
 * the z and y written by the calls since the last check are unspecified
 * (a block whose wait expired contributed nothing, or zeros); every block
 * still waited, bounded, for its own copies before it left. */
int ig_check_status(void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* INVARIANT_GEMM_H */
