// moe_permute_static_scratch: the grouping step (moe_permute) for callers
// that cannot allocate device memory.
//
// The grouping kernels need one scratch buffer besides their inputs and
// outputs: a table of per-chunk, per-expert counts (ceil(T*top_k/1024) x E
// int32, chunks of kPermuteChunk = 1024 assignments).  moe_permute takes it from the caller's workspace.  This variant
// keeps it in a fixed array in the library's own device memory instead, so
// the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds its 256 KB + 256 bytes until the process exits.
// Its host-side name is only a stand-in for the symbol, never a device
// address; the device address is looked up with cudaGetSymbolAddress on the
// first call made with that device current and cached together with the
// unique id of the CUDA context it belongs to.  A device reset destroys that
// context and the module with it; the next call runs in a context with a new
// id and looks the address up again instead of using a stale one.
//
// Every call uses the same array.  The count kernel rewrites every table
// entry it later reads, so the table needs no clearing; the status word in
// the array's first bytes is cleared at the start of each call.  Two calls
// whose work overlaps on the GPU (different streams, no ordering between
// them) race on the array and may produce wrong results.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kMaxTableEntries = 65536;  // chunks x experts, int32 each
constexpr size_t kScratchBytes = kStatusBytes + kMaxTableEntries * sizeof(int32_t);

static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

struct CachedAddress {
  void* ptr;
  unsigned long long ctx_id;  // 0: none cached
};
std::mutex g_addr_mu;
CachedAddress g_addr[64] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (ids are never
// reused within a process), or 0 when there is none or it cannot be read.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_scratch on the current device, looked up on the
// first call in each context (with that device current) and cached for it.
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && g_addr[dev].ctx_id == ctx) {
    *out = g_addr[dev].ptr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);  // makes the context current if needed
  if (e != cudaSuccess) return e;
  g_addr[dev] = CachedAddress{p, current_context_id()};
  *out = p;
  return cudaSuccess;
}

moe_status_t reject(moe_status_t st, const std::string& msg) {
  set_last_error(msg);
  return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_permute_static_scratch(const int32_t* topk_ids, const moe_bf16* x,
                                                   int T, int d, int E, int top_k,
                                                   int32_t* expert_counts,
                                                   int32_t* expert_offsets, int32_t* perm,
                                                   int32_t* slot_pos, moe_bf16* x_perm,
                                                   uint32_t* device_status,
                                                   moe_stream_t stream) {
  if (T < 0 || d <= 0 || E <= 0 || top_k <= 0)
    return reject(MOE_ERR_INVALID_ARG, "T must be >= 0 and d, E, top_k > 0");
  if (d % 64) return reject(MOE_ERR_UNSUPPORTED, "d must be a multiple of 64");
  if (E > kMaxExperts) return reject(MOE_ERR_UNSUPPORTED, "at most 256 experts");
  if (top_k > E || top_k > kMaxTopK) return reject(MOE_ERR_INVALID_ARG, "top_k must be <= min(E, 8)");
  const long long n = static_cast<long long>(T) * top_k;
  const long long chunks = (n + kPermuteChunk - 1) / kPermuteChunk;
  if (chunks * E > static_cast<long long>(kMaxTableEntries)) {
    char buf[200];
    std::snprintf(buf, sizeof buf,
                  "moe_permute_static_scratch: ceil(T*top_k/%d)*E = %lld exceeds its fixed "
                  "table of %zu entries (e.g. T*top_k <= %zu with E = 256); use moe_permute",
                  kPermuteChunk, chunks * E, kMaxTableEntries,
                  kMaxTableEntries / kMaxExperts * kPermuteChunk);
    return reject(MOE_ERR_UNSUPPORTED, buf);
  }
  if (T == 0) return MOE_OK;
  if (!topk_ids || !expert_counts || !expert_offsets || !perm || !slot_pos)
    return reject(MOE_ERR_INVALID_ARG, "moe_permute_static_scratch: null pointer");
  if (x && (!x_perm || !aligned16(x) || !aligned16(x_perm)))
    return reject(MOE_ERR_INVALID_ARG,
                  "moe_permute_static_scratch: x and x_perm must be 16-byte aligned");
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return reject(MOE_ERR_CUDA, "moe_permute_static_scratch: cannot query the device");
  if (major != 10 || minor != 3)
    return reject(MOE_ERR_UNSUPPORTED, "this library is built for sm_103a");

  void* scratch = nullptr;
  cudaError_t e = static_scratch_address(&scratch);
  if (e != cudaSuccess)
    return reject(MOE_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned* status = device_status ? reinterpret_cast<unsigned*>(device_status)
                                   : static_cast<unsigned*>(scratch);
  if (!device_status) {
    e = cudaMemsetAsync(scratch, 0, sizeof(unsigned), s);
    if (e != cudaSuccess)
      return reject(MOE_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  }
  int32_t* table = reinterpret_cast<int32_t*>(static_cast<char*>(scratch) + kStatusBytes);
  e = launch_permute(s, topk_ids, x, T, d, E, top_k, expert_counts, expert_offsets, perm,
                     slot_pos, x_perm, table, status);
  if (e != cudaSuccess)
    return reject(MOE_ERR_CUDA, std::string("permute launch: ") + cudaGetErrorString(e));
  return MOE_OK;
}
