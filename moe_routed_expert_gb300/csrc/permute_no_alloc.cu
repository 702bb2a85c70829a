// moe_permute_no_alloc: the token permute for callers that cannot allocate
// device memory -- code that runs where cudaMalloc is off limits (inside a
// framework whose allocator owns all device memory, a plugin or embedded
// runtime with a fixed memory budget, a path that must never block on the
// driver's allocator) and therefore cannot hand moe_permute a workspace.
//
// The permute's only scratch (per-chunk expert counts, 1024 slots per chunk)
// lives instead in one file-scope device array of fixed size, created when the
// library's module is loaded on a device and kept there until the process
// exits.  Host code must not pass the array's name to a kernel: on the host it
// names a host-side stand-in, not device memory.  Its device address is looked
// up with cudaGetSymbolAddress, with the device current, on the first call in
// each CUDA context of that device: a context rebuilt after cudaDeviceReset
// gets the address of its own copy of the array, never a stale one.
//
// Nothing in the array has to start at zero: every call writes all the counts
// it later reads.  Calls share the array, so two calls whose kernels overlap on
// the GPU (other streams, other host threads) race; order them on one stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "moe_gmm.h"

namespace moe {
namespace {

// 512 KiB of int32 counters: ceil(T*k / 1024) * E must not exceed this.
constexpr int64_t kNoAllocCounters = 131072;

static __device__ __align__(256) int32_t g_permute_counts[kNoAllocCounters];

constexpr int kMaxDevices = 64;

// The calling thread's current CUDA context (driver call, looked up through the
// runtime so the library needs no link to libcuda); nullptr if unavailable.
CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(ptr);
  });
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_permute_counts in the current device's current context,
// looked up on the first call in that context (nullptr if the lookup fails).
void* counts_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  static CUcontext ctx[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CUcontext c = current_context();  // null until the runtime has made a context current
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || c == nullptr || ctx[dev] != c) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_counts) != cudaSuccess) return nullptr;  // sets up the context
    if ((c = current_context()) == nullptr) return nullptr;
    addr[dev] = p;
    ctx[dev] = c;
  }
  return addr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_permute_no_alloc(const moe_bf16* x, const int32_t* topk_ids, int64_t T, int64_t H,
                                             int64_t k, int64_t E, moe_bf16* x_perm, int64_t* group_list,
                                             int32_t* row_id_map, int32_t* sorted_flat, uint32_t* device_status,
                                             moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_permute_args(x, topk_ids, T, H, k, E, x_perm, group_list, row_id_map, sorted_flat);
  if (st != MOE_OK) return st;
  if (reinterpret_cast<uintptr_t>(device_status) & 3u) return MOE_ERR_INVALID;  // an atomically updated word
  if (T == 0)  // nothing routed: every expert gets zero rows
    return cudaMemsetAsync(group_list, 0, E * sizeof(int64_t), reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
  const int64_t chunks = (T * k + 1023) / 1024;
  if (chunks * E > kNoAllocCounters) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* counts = counts_address();
  if (counts == nullptr) return MOE_ERR_CUDA;
  return launch_permute(x, topk_ids, T, x ? H : 0, k, E, x_perm, group_list, row_id_map, sorted_flat,
                        device_status, counts, reinterpret_cast<cudaStream_t>(stream));
}
