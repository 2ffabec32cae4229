// la_noalloc.cu -- la_decode_step_noalloc: the decode step for callers that must not
// allocate device memory.
//
// la_decode_step_ex keeps its fp32 pre-norm y, the per-head sums of squares and the
// per-sequence arrival counters in a workspace it allocates with cudaMalloc on first
// use.  Some callers cannot let a library do that: a serving engine that has reserved
// all of HBM for its own pool (a stray cudaMalloc would fail or eat into the pool), or
// a latency-critical loop where the implicit device synchronisation of
// cudaMalloc/cudaFree is not acceptable.  This entry point runs the same decode kernel
// with its scratch taken from a fixed array in the library's own device data instead.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchFloats 4-byte words
// (8.13 MiB), which every device that loads this library holds until the process
// exits.  Host code cannot use the array's name as a device address (on the host it
// names a host-side shadow), so the first call on each device looks the address up
// with cudaGetSymbolAddress while that device is current and caches it.
//
// The CUDA runtime loads a library's device code lazily by default, so the array is
// most likely materialised on a device by that first lookup, not when the library is
// loaded.  A caller that reserves all free device memory for its own pool should make
// its first call on each device before reserving the pool (or run with
// CUDA_MODULE_LOADING=EAGER, which materialises the array when the library loads).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/lightning_attn.h"
#include "la_internal.h"

namespace la {
namespace {

// y [B*H][d] fp32, then ss [B*H] fp32, then one arrival counter per sequence (B <= B*H),
// for up to LA_NOALLOC_MAX_HEADS heads.  The counters start at zero (static storage)
// and every call leaves them at zero.
constexpr size_t kNoAllocScratchFloats =
    size_t(LA_NOALLOC_MAX_HEADS) * kHeadDim + 2 * size_t(LA_NOALLOC_MAX_HEADS);

__device__ __align__(256) float g_decode_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
float* g_scratch_addr[kMaxDevices];  // device address of g_decode_scratch, per device

// Device address of the scratch array on the current device (looked up once per
// device), or nullptr if the lookup failed.
float* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    return g_scratch_addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace la

using namespace la;

extern "C" int la_decode_step_noalloc(float* kv_state, const void* q, const void* k,
                                      const void* v, const void* g, void* out, int B, int H,
                                      int d, int dtype, float eps, void* cuda_stream) {
    if (B <= 0 || H <= 0 || d <= 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 && dtype != LA_F32) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (d != kHeadDim) return LA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > LA_NOALLOC_MAX_HEADS) return LA_ERR_SCRATCH_LIMIT;
    if (!kv_state || !q || !k || !v || !g || !out) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {kv_state, q, k, v, g, out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return LA_ERR_MISALIGNED;
    const bool bf16 = dtype == LA_BF16;
    const size_t io_bytes = (size_t)B * H * d * (bf16 ? 2 : 4);
    const size_t state_bytes = (size_t)B * H * d * d * sizeof(float);
    const void* ins[] = {q, k, v, g};
    for (const void* p : ins) {
        if (overlaps(out, io_bytes, p, io_bytes)) return LA_ERR_INVALID_ARG;
        if (overlaps(kv_state, state_bytes, p, io_bytes)) return LA_ERR_INVALID_ARG;
    }
    if (overlaps(kv_state, state_bytes, out, io_bytes)) return LA_ERR_INVALID_ARG;

    float* scratch = scratch_on_current_device();
    if (!scratch) return LA_ERR_CUDA;
    // The kernel writes every y and ss entry it later reads, and returns each counter it
    // uses to zero, so the scratch needs no clearing between calls.
    float* y = scratch;
    float* ss = scratch + (size_t)LA_NOALLOC_MAX_HEADS * kHeadDim;
    unsigned* cnt = reinterpret_cast<unsigned*>(ss + LA_NOALLOC_MAX_HEADS);
    return launch_decode(kv_state, q, k, v, g, out, y, ss, cnt, B, H, eps, bf16,
                         reinterpret_cast<cudaStream_t>(cuda_stream));
}
