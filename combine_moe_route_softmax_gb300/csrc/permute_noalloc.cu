// moe_permute_noalloc: moe_permute for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: plugins embedded in an inference engine
// that owns every device allocation (their enqueue step must not allocate), code that
// runs while its stream is being captured into a CUDA graph (a synchronous allocation
// there breaks the capture), and real-time serving paths with a fixed device-memory
// budget.  moe_permute needs a small index scratch (per-block, per-expert counts) that
// those callers would otherwise have to provide.  This entry point takes it instead from
// a file-scope static __device__ array of a fixed size, which exists on every GPU that
// loads the library until the process exits.
//
// The array's name in host code is only a host-side stand-in for the symbol, not a
// device address: the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached together with the CUDA
// context it belongs to.  That set-up happens on the first call on each device, so that
// first call should be made before any stream capture begins.  A device reset
// (cudaDeviceReset) ends the context and may move the array; the next call sees a new
// current context and looks the address up again, so it too belongs outside a capture.
//
// Every call on a device shares the one array.  Nothing in it has to start at zero: the
// count kernel writes every entry the later kernels read.  Two calls whose kernels
// overlap on the GPU (different streams without ordering between them) race on the
// array and produce garbage; calls on one stream, or otherwise ordered, are safe.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace moe {
constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
}

// The scratch itself: one copy per GPU that loads the library, alive until exit.
static __device__ __align__(256) unsigned char g_permute_scratch[moe::kStaticScratchBytes];

namespace moe {
namespace {

constexpr int kMaxDevices = 64;

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// cuCtxGetCurrent from the CUDA driver, looked up once (the library links only the runtime).
PFN_cuCtxGetCurrent_v4000 ctx_get_fn() {
  static const PFN_cuCtxGetCurrent_v4000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    return static_cast<PFN_cuCtxGetCurrent_v4000>(nullptr);
  }();
  return fn;
}

// Device address of g_permute_scratch on the current device: looked up once per device
// and context (a device reset gives the device a new context, and the lookup is redone).
moe_status_t static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  const PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_get_fn();
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (ctx == nullptr || !g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
    // (the lookup also makes the device's primary context current when none is yet)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_permute_noalloc_max_scratch_bytes(void) { return moe::kStaticScratchBytes; }

extern "C" moe_status_t moe_permute_noalloc(const int32_t* topk_idx, int T, int K, int E, int with_shared,
                                            const uint16_t* x, int H, moe_dtype_t out_dtype, void* xp,
                                            float* xp_scales, int32_t* cu_seqlens, int32_t* src_row,
                                            int32_t* inv_map, int32_t* shared_map, int32_t* dev_status,
                                            void* stream) {
  const size_t need = moe_permute_workspace_bytes(T, K, E, with_shared);
  if (need > moe::kStaticScratchBytes) return MOE_ERR_WORKSPACE;  // shape too large for the static scratch
  void* scratch = nullptr;
  const moe_status_t st = moe::static_scratch(&scratch);
  if (st != MOE_OK) return st;
  return moe_permute(topk_idx, T, K, E, with_shared, x, H, out_dtype, xp, xp_scales, cu_seqlens, src_row, inv_map,
                     shared_map, scratch, moe::kStaticScratchBytes, dev_status, stream);
}
