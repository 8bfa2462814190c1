// sr_noalloc.cu -- chunk attention for callers that cannot allocate device memory.
//
// sr_chunk_attention can split the key range of a chunk's last query block
// into several work units, which exchange partial results through a scratch
// area, and runs persistent CTAs that take units from a counter there; the
// scratch is normally the session's caller-owned workspace. Some callers cannot
// provide one: code that runs where cudaMalloc is off limits (inside a
// framework's memory pool with a fixed budget, in a plugin that must not touch
// the allocator, or in a process that only receives a stream and a few
// tensors). sr_chunk_attention_noalloc serves them: its scratch is a fixed
// array compiled into this library, so the call allocates nothing.
//
// The array is a file-scope __device__ object of kScratchBytes; every GPU that
// loads the library holds it until the process exits. In host code its name is
// only a host-side stand-in, never a device address: the device address is
// obtained once per device with cudaGetSymbolAddress (with that device
// current; again if the device's context has been replaced, e.g. after
// cudaDeviceReset) and handed to the kernels as a pointer. Every call shares the
// array and finds the previous call's contents in it, so the arrival counters
// that must start at zero are cleared on the stream before each launch, and
// calls that overlap on the GPU (on different streams, or sessions used
// concurrently) race on it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "sr.h"
#include "sr_kernels.h"

namespace {

// Room for a session of up to 62 heads at head_dim 128 (4 key parts per head).
constexpr uint64_t kScratchBytes = 16ull << 20;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

// The launch-wide unit counter and the per-head arrival counters sit at the
// start of the scratch.
__global__ void clear_arrival_counters(int n) {
  int32_t* ctr = reinterpret_cast<int32_t*>(g_attn_scratch);
  for (int i = threadIdx.x; i < n; i += blockDim.x) ctr[i] = 0;
}

constexpr int kMaxDevices = 64;

// The current context's process-unique id (cuCtxGetId), or 0 if the driver
// cannot say. A context torn down and created again (cudaDeviceReset, then
// more work on the device) gets a new id, and the array a new address.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array in the current device's context. The
// set-up looks it up with cudaGetSymbolAddress once per device (with that
// device current) and again only if the device's context was replaced since;
// nullptr if the lookup fails.
void* scratch_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices];
  static unsigned long long ctx_id[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long id = current_context_id();   // 0: no context yet, or no id
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr || id == 0 || id != ctx_id[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
    ctx_id[dev] = current_context_id();   // the lookup has made the context current
  }
  return addr[dev];
}

}  // namespace

extern "C" {

sr_status sr_chunk_attention_noalloc(sr_session* s, int32_t step, const void* q, const void* k, const void* v,
                                     void* o, float* lse, void* stream) {
  sr_status st = sr::attention_scratch_check(s, step, q, k, v, o, lse, kScratchBytes);
  if (st != SR_OK) return st;
  void* scratch = scratch_address();
  if (scratch == nullptr) return SR_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (sr::launch_plain(clear_arrival_counters, 1, 256, cs,
                       static_cast<int>(sr::kWsUnitCtrBytes / 4) + sr::session_heads(s)) != cudaSuccess)
    return SR_ERR_CUDA;
  return sr::attention_into_scratch(s, step, q, k, v, o, lse, stream, scratch);
}

}  // extern "C"
