// la_internal.h -- declarations shared by the translation units of liblightning_attn.so.
// Not installed; the public surface is include/lightning_attn.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

constexpr int kHeadDim = 128;  // the only head size the kernels cover (64 x 128 heads)

// Per-device scratch owned by the library (see la_api.cu).
struct Workspace {
    void* base = nullptr;   // grown on demand
    size_t bytes = 0;
    int* status = nullptr;  // device status word (LA_OK / LA_ERR_TIMEOUT)
};

// Returns LA_OK and a workspace of at least `bytes` for the current device.
int workspace_acquire(size_t bytes, Workspace* ws);

// Launch accounting behind la_launch_count().
void note_launches(int n);

// ---- CUDA-core kernels (la_simt.cu) ----------------------------------------------
// Prefill: y (fp32 [B][N][H][d]) and the final state; then the norm/gate pass.
int launch_prefill_simt(const void* q, const void* k, const void* v, const float* S_in,
                        float* y, float* S_out, int B, int H, int64_t N, bool bf16,
                        cudaStream_t st);
int launch_norm_gate_rows(const float* y, const void* g, void* out, int64_t rows, int width,
                          float eps, bool bf16, cudaStream_t st);
// Decode: state update + y = q S (y fp32 [B][H][d], per-(b,h) sum of squares), then norm.
int launch_decode(float* S, const void* q, const void* k, const void* v, const void* g,
                  void* out, float* y, float* ss, int B, int H, float eps, bool bf16,
                  cudaStream_t st);
int launch_zero_state(float* S, int64_t n, cudaStream_t st);

// ---- tensor-core prefill (la_prefill_tc.cu) --------------------------------------
// Returns LA_ERR_UNSUPPORTED when the shape is outside what the kernel covers.
int prefill_tc_supported(int B, int H, int64_t N);
size_t prefill_tc_workspace_bytes(int B, int H, int64_t N);
int launch_prefill_tc(const void* q, const void* k, const void* v, const void* g, void* out,
                      const float* S_in, float* S_out, float* y_debug, int B, int H, int64_t N,
                      float eps, const Workspace& ws, cudaStream_t st);

}  // namespace la
