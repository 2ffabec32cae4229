// la_internal.h -- declarations shared by the translation units of liblightning_attn.so.
// Not installed; the public surface is include/lightning_attn.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

constexpr int kHeadDim = 128;  // the only head size the kernels cover (64 x 128 heads)

// Per-sequence arrival counters of the decode step (one per sequence b, B <= 65535).
constexpr int kDecodeCounterSlots = 65536;

// Bit pattern of an exchange slot not yet written: a negative float, which a sum of
// squares never is.
constexpr uint32_t kXchEmpty = 0x80808080u;

// Per-device scratch owned by the library (see la_api.cu).
struct Workspace {
    void* base = nullptr;        // grown on demand
    size_t bytes = 0;
    int* status = nullptr;       // device status word (LA_OK / LA_ERR_TIMEOUT)
    unsigned* dec_cnt = nullptr; // kDecodeCounterSlots decode counters, zero between calls
};

// Returns LA_OK and a workspace of at least `bytes` for the current device.  On the
// first call for a device the status word and the decode counters are allocated and
// zeroed on `st`.
int workspace_acquire(size_t bytes, cudaStream_t st, Workspace* ws);

// The cross-head exchange of the tensor-core prefill.  Per chunk: the per-token sums of
// squares of every head half ("partials", written before they are read, never reset; a
// ring of 16 chunks whose slot a head half reuses once the norm factors of the chunk
// that held it are published) and the chunk's arrival counter and per-token norm
// factors ("flags", 129 words per chunk), which live in two banks whose every word holds
// kXchEmpty until written.  A launch writes one flag
// bank and resets, in the other, the words that the previous launch wrote there; so
// every flag bank is all-empty again one launch after its use and nothing runs between
// calls.
struct XchLease {
    float* use = nullptr;        // the flag bank this launch writes (all words empty)
    uint32_t* clear = nullptr;   // the other flag bank
    size_t clear_words = 0;      // its words [0, clear_words) to reset to kXchEmpty
    unsigned bank = 0;
    float* part = nullptr;       // the partials
};
// A lease with at least `flag_words` words per flag bank and `part_floats` partials for
// the current device.
int xch_acquire(size_t flag_words, size_t part_floats, cudaStream_t st, XchLease* out);
// The launch of `lease` was enqueued and will write `words_used` words of its flag bank.
void xch_commit(const XchLease& lease, size_t words_used);

// Launch accounting behind la_launch_count().
void note_launches(int n);

// ---- CUDA-core kernels (la_simt.cu) ----------------------------------------------
// Prefill: y (fp32 [B][N][H][d]) and the final state; then the norm/gate pass.
// activated: q, k, v are already SiLU-activated (step 2 is skipped).
int launch_prefill_simt(const void* q, const void* k, const void* v, const float* S_in,
                        float* y, float* S_out, int B, int H, int64_t N, bool bf16,
                        bool activated, cudaStream_t st);
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
// (sequence, chunk) items of a batch of B sequences of N tokens
int prefill_tc_items(int B, int64_t N);
size_t prefill_tc_flag_words(int items);
// The partials: a ring of chunks per segment, independent of the length.
size_t prefill_tc_part_floats(int H, int nseg);
// Segment-parallel plan for B sequences of N tokens: the number of segments (1: the
// serial chunk chain), their length in chunks (seg_items) and the state-pass pieces per
// segment (fine).  Only B == 1 is cut, and only when H leaves SMs idle.
int prefill_tc_segment_plan(int B, int H, int64_t N, int* seg_items, int* fine);
// nseg > 1: segment s of seg_items chunks starts from S_seg[s] ([nseg][H][d][d], B == 1).
int launch_prefill_tc(const void* q, const void* k, const void* v, const void* g, void* out,
                      const float* S_in, float* S_out, float* y_debug, int B, int H, int64_t N,
                      float eps, bool activated, const Workspace& ws, const XchLease& xl,
                      cudaStream_t st, int nseg = 1, int seg_items = 0,
                      const float* S_seg = nullptr);
// A packed batch of T tokens: items (device, `total` of them) = {first row, valid rows,
// sequence, first chunk of its sequence}, chunks of 128 tokens in order.
int launch_prefill_tc_varlen(const void* q, const void* k, const void* v, const void* g,
                             void* out, const float* S_in, float* S_out, float* y_debug, int H,
                             int64_t T, int total, const int4* items, float eps,
                             bool activated, const Workspace& ws, const XchLease& xl,
                             cudaStream_t st);
// Chunk length of the tensor-core prefill (the items' granularity).
constexpr int kTcChunk = 128;
// The [B][N][H*d] bf16 tensor map of the tensor-core kernels (64-feature x 128-token
// boxes, 128B swizzle); false if the driver's encoder is unavailable or refuses.
bool encode_io_map_bf16(CUtensorMap* m, const void* base, int B, int H, int64_t N);

// ---- state-only pass (la_state_tc.cu) ------------------------------------------------
// Segments per (b, h) for a state pass over N tokens (whole 128-token chunks each).
int state_segments(int B, int H, int64_t N);
// Partial states part[nseg][B][H][d][d] of the segments (bf16 k, v; activated: already
// SiLU-activated).
int launch_state_tc(const void* k, const void* v, float* part, int B, int H, int64_t N,
                    int nseg, bool activated, int* status, cudaStream_t st);
// out[j] = (base ? base[j] : 0) + sum_{i < count} parts[i * n + j] in the order of i.
int launch_sum_rows(const float* parts, int count, int64_t n, const float* base, float* out,
                    cudaStream_t st);
// out[s] = (base or 0) + sum_{i < s * per} parts[i] for s < nout, one running sum in the
// order of i (each equal to launch_sum_rows with count = s * per).
int launch_prefix_rows(const float* parts, int per, int nout, int64_t n, const float* base,
                       float* out, cudaStream_t st);

}  // namespace la
