// gdn_proj_noalloc.cu - the input projections with the split of x kept in a
// fixed scratch array compiled into the library, for callers that hand the
// library no workspace. The projection itself is launch_in_proj, unchanged:
// only where its workspace lives differs.

#include <mutex>

#include "gdn_launch.h"

namespace gdn {

constexpr size_t kStaticScratchBytes = size_t(48) << 20;  // 48 MiB per device

// One instance per device, zero-initialised at module load; never freed.
static __device__ __align__(256) unsigned char g_proj_scratch[kStaticScratchBytes];

namespace {
std::mutex g_mutex;
void* g_scratch_ptr[64] = {nullptr};
}  // namespace

size_t proj_static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t launch_in_proj_static(const ProjArgs& args, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_scratch_ptr[dev] == nullptr) {
            e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_proj_scratch);
            if (e != cudaSuccess) {
                g_scratch_ptr[dev] = nullptr;
                return e;
            }
        }
        scratch = g_scratch_ptr[dev];
    }
    ProjArgs a = args;
    a.workspace = scratch;
    return launch_in_proj(a, stream);
}

}  // namespace gdn
