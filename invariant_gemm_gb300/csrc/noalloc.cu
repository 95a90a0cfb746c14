// lora_shrink_noalloc: the shrink with its scratch memory built into the
// library, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the shrink: code that must not trigger the implicit device-wide
// synchronisation an allocation can cause (latency-critical serving loops),
// runtimes that hand out memory only from a budget planned ahead of time
// and give a kernel library no allocator, and plugin hosts that own every
// allocation. This entry point takes the same inputs and output as
// lora_shrink but needs no workspace from the caller: the token map,
// completion counters, status word and Split-K partials live in one
// file-scope device array of fixed size, which every GPU that loads the
// library holds until the process exits.
#include <mutex>

#include "ig_common.cuh"

namespace ig {

// api.cu: lora_shrink's own share of the workspace (the expand's Z operand,
// which only lora_apply writes, left out), and lora_shrink checking the
// workspace against it
size_t shrink_ws_bytes(const ig_shape* sh);
int lora_shrink_ws(const ig_shape* shape, const void* x, const void* A_stack,
                   const int32_t* adapter_idx, float scale, float* z, void* ws,
                   size_t ws_bytes, void* stream, bool full);

namespace {

// 4 MiB: the fixed counter area plus room for decode-sized token maps and
// partials (e.g. M = 1024, r = 32, 32 adapters, Split-K = 8 needs ~1.6 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current). In host code the array's name only
// stands for the symbol; its device address must come from the runtime.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return IG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return IG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return IG_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return IG_OK;
}

}  // namespace
}  // namespace ig

extern "C" int lora_shrink_noalloc(const ig_shape* shape, const void* x, const void* A_stack,
                                   const int32_t* adapter_idx, float scale, float* z,
                                   void* stream) {
  using namespace ig;
  ig_plan_info info;
  int rc = ig_plan_query(shape, &info);
  if (rc != IG_OK) return rc;
  if (shape->M == 0) return IG_OK;
  if (!adapter_idx) return IG_ERR_ARG;  // no map survives between calls by contract
  // The argument checks lora_shrink makes, made here before the clear below
  // is enqueued: a rejected call enqueues nothing.
  if (!x || !A_stack || !z) return IG_ERR_ARG;
  auto aligned16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (!aligned16(x) || !aligned16(A_stack) || !aligned16(z) || !aligned16(adapter_idx))
    return IG_ERR_ALIGN;
  if (shrink_ws_bytes(shape) > kNoAllocScratchBytes) return IG_ERR_WS_SMALL;
  void* ws = nullptr;
  rc = scratch_for_current_device(&ws);
  if (rc != IG_OK) return rc;
  // The array keeps whatever the previous call left. The status word and the
  // counters this call uses must start at zero; clear them on the stream.
  const int64_t slots = info.shrink_ctas_max / info.split_k;
  const size_t clear = kCountersOffset + 4 * (size_t)slots;
  if (cudaMemsetAsync(ws, 0, clear, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return IG_ERR_CUDA;
  return lora_shrink_ws(shape, x, A_stack, adapter_idx, scale, z, ws, kNoAllocScratchBytes,
                        stream, false);
}
