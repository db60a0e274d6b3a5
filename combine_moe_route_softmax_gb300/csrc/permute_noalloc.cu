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
// cudaGetSymbolAddress (with that device current) and cached.  That set-up happens on the
// first call on each device, so that first call should be made before any stream capture
// begins.
//
// Every call on a device shares the one array.  Nothing in it has to start at zero: the
// count kernel writes every entry the later kernels read.  Two calls whose kernels
// overlap on the GPU (different streams without ordering between them) race on the
// array and produce garbage; calls on one stream, or otherwise ordered, are safe.
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

// Device address of g_permute_scratch on the current device (looked up once per device).
moe_status_t static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
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
