// la_internal.h -- declarations shared by the translation units of liblightning_attn.so.
// Not installed; the public surface is include/lightning_attn.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

constexpr int kHeadDim = 128;  // the only head size the kernels cover (64 x 128 heads)

// Arrival counters of the tensor-core prefill's cross-head exchange: two banks, one
// counter per (sequence, chunk).  A launch uses one bank and zeroes the other for the
// next launch, so no separate reset is needed between calls.
constexpr int kTcCounterSlots = 1 << 17;
constexpr size_t kTcCounterBytes = size_t(kTcCounterSlots) * sizeof(unsigned);
// Per-sequence arrival counters of the decode step (one per sequence b, B <= 65535).
constexpr int kDecodeCounterSlots = 65536;

// Per-device scratch owned by the library (see la_api.cu).
struct Workspace {
    void* base = nullptr;      // grown on demand
    size_t bytes = 0;
    int* status = nullptr;     // device status word (LA_OK / LA_ERR_TIMEOUT)
    unsigned* banks = nullptr; // 2 x kTcCounterSlots counters, zeroed at allocation
    unsigned* dec_cnt = nullptr; // kDecodeCounterSlots decode counters, zero between calls
    unsigned bank = 0;         // the bank the next tensor-core prefill uses
};

// Returns LA_OK and a workspace of at least `bytes` for the current device.  On the
// first call for a device the status word and the counter banks are allocated and
// zeroed on `st`.
int workspace_acquire(size_t bytes, cudaStream_t st, Workspace* ws);
// The tensor-core prefill just launched on the current bank: the next one uses the other.
void workspace_switch_bank();

// Launch accounting behind la_launch_count().
void note_launches(int n);

// ---- CUDA-core kernels (la_simt.cu) ----------------------------------------------
// Prefill: y (fp32 [B][N][H][d]) and the final state; then the norm/gate pass.
int launch_prefill_simt(const void* q, const void* k, const void* v, const float* S_in,
                        float* y, float* S_out, int B, int H, int64_t N, bool bf16,
                        cudaStream_t st);
int launch_norm_gate_rows(const float* y, const void* g, void* out, int64_t rows, int width,
                          float eps, bool bf16, cudaStream_t st);
// Decode: state update + y = q S (y fp32 [B][H][d], per-(b,h) sum of squares), and the
// norm + gate by the last head of each sequence to arrive on cnt[b] (cnt: B counters,
// zero on entry and left zero).
int launch_decode(float* S, const void* q, const void* k, const void* v, const void* g,
                  void* out, float* y, float* ss, unsigned* cnt, int B, int H, float eps,
                  bool bf16, cudaStream_t st);
int launch_zero_state(float* S, int64_t n, cudaStream_t st);

// ---- tensor-core prefill (la_prefill_tc.cu) --------------------------------------
// Returns LA_ERR_UNSUPPORTED when the shape is outside what the kernel covers.
int prefill_tc_supported(int B, int H, int64_t N);
size_t prefill_tc_workspace_bytes(int B, int H, int64_t N);
int launch_prefill_tc(const void* q, const void* k, const void* v, const void* g, void* out,
                      const float* S_in, float* S_out, float* y_debug, int B, int H, int64_t N,
                      float eps, const Workspace& ws, cudaStream_t st);

}  // namespace la
