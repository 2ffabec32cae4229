/*
 * lightning_attn.h -- C ABI of liblightning_attn.so, the B300 (sm_103a) forward pass
 * of the Lightning Attention layer (causal linear attention with an RMSNorm output
 * and a sigmoid gate).
 *
 * The operation (MiniMax-01 deep dive, Hugging Face blog, "Hybrid Modeling", the
 * four-step mechanism of the 7/8 linear-attention layers):
 *   q^ = SiLU(q), k^ = SiLU(k), v^ = SiLU(v)                       (step 2)
 *   S_t = S_{t-1} + k^_t^T v^_t ,  y_t = q^_t S_t   (causal, s <= t) (step 3, the
 *         O(d^2 n) right-product route the same section contrasts with O(n^2 d))
 *   out_t = y_t / sqrt(mean(y_t^2) + eps) * sigmoid(g_t)           (step 4)
 * The mean runs over all H*d features of a token; the RMSNorm weight is one; g is
 * the gate input and gets no SiLU; there is no 1/sqrt(d) scale and no decay.
 * Head count and head size come from the MiniMax-Text-01 architecture list
 * (64 heads of size 128); this library requires d == 128.
 *
 * Layouts (all row-major, no padding):
 *   prefill q, k, v, g, out, y_debug : [B][N][H][d]   (= [B*N][H*d])
 *   decode  q, k, v, g, out          : [B][H][d]
 *   state   kv_state                 : [B][H][d][d] fp32, S[i][j] = sum_s k^_s[i] v^_s[j]
 *
 * Ownership and memory: every pointer is a DEVICE pointer owned by the caller
 * (16-byte aligned).  Inputs are read only and are not modified; out must not alias
 * an input.  The library owns one internal per-device workspace (exchange buffers,
 * status word), grown on demand under a mutex and freed at unload.  The prefill's
 * exchange holds 1 MiB at H = 64 for any length plus 2 x 516 bytes per 128-token chunk.
 *
 * Execution: calls enqueue kernels on the given CUDA stream (NULL = legacy default
 * stream) and return without synchronising.  Calls on one device share the
 * workspace, so calls that may run concurrently on different streams of the same
 * device must be ordered by the caller.  Argument errors are detected on the
 * host before anything is launched and nothing is written.  A kernel that gives up
 * a bounded wait records LA_ERR_TIMEOUT in the device status word, which
 * la_get_device_status() reads.  Nothing in the library prints, exits or traps.
 */
#ifndef LIGHTNING_ATTN_H
#define LIGHTNING_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1, /* NULL pointer, B/H/N out of range, eps < 0, aliasing   */
    LA_ERR_UNSUPPORTED = 2, /* d != 128, or a shape the kernels do not cover          */
    LA_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned                       */
    LA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed            */
    LA_ERR_NOMEM = 5,       /* the workspace could not be grown                       */
    LA_ERR_TIMEOUT = 6,     /* a kernel gave up a bounded cross-CTA wait              */
    LA_ERR_SCRATCH_LIMIT = 7 /* B*H above LA_NOALLOC_MAX_HEADS (la_decode_step_noalloc) */
} la_status;

typedef enum {
    LA_BF16 = 0, /* bf16 inputs/outputs, fp32 state and accumulation */
    LA_F32 = 1   /* fp32 inputs/outputs, fp32 everywhere              */
} la_dtype;

/* Flags for the _ex entry points. */
#define LA_FLAG_SIMT 1u /* prefill: run the CUDA-core kernel instead of the
                           tensor-core kernel (the only kernel for LA_F32) */
#define LA_FLAG_ACTIVATED 2u /* prefill: q, k, v are already SiLU-activated (as
                                la_qkvg_projection writes them with LA_PROJ_SILU);
                                the kernels skip step 2.  g is raw either way. */
#define LA_FLAG_SERIAL 4u /* prefill: keep one chunk chain per head even where the
                             segment-parallel mode would run (see la_prefill_path) */

/*
 * Prefill of B sequences of N tokens ("Hybrid Modeling", mechanism steps 2-4).
 * bf16 I/O, eps = 1e-6, zero initial state, legacy default stream.
 *   q, k, v, g    in  [B][N][H][d] bf16, pre-activation projections
 *   out           out [B][N][H][d] bf16
 *   kv_state_out  out [B][H][d][d] fp32, the state after token N-1 (may be NULL)
 * N == 0 is legal: kv_state_out receives zeros and out is untouched.
 * Returns an la_status.
 */
int la_prefill(const void* q, const void* k, const void* v, const void* g, void* out,
               float* kv_state_out, int B, int H, int64_t N, int d);

/*
 * One decode step for B sequences: for each (b,h), S += k^T v (in place), then
 * y = q S; out = RMSNorm over the H*d features of each b, times sigmoid(g).
 * bf16 I/O, eps = 1e-6, legacy default stream.
 *   kv_state  in/out [B][H][d][d] fp32
 *   q,k,v,g   in     [B][H][d] bf16;  out  out [B][H][d] bf16
 */
int la_decode_step(float* kv_state, const void* q, const void* k, const void* v,
                   const void* g, void* out, int B, int H, int d);

/*
 * Extended prefill.  bf16 runs the tensor-core kernel (LA_ERR_UNSUPPORTED for a shape it
 * does not cover, see la_prefill_path); LA_F32, or LA_FLAG_SIMT, the CUDA-core kernel.
 *   kv_state_in  in  [B][H][d][d] fp32 initial state, or NULL for zeros; lets a long
 *                    sequence be processed in pieces (the state is the resume point)
 *   kv_state_out out [B][H][d][d] fp32 or NULL; may equal kv_state_in
 *   y_debug      out [B][N][H][d] fp32 pre-norm y, or NULL
 *   dtype        la_dtype of q, k, v, g, out
 *   eps          RMSNorm epsilon (>= 0)
 *   flags        LA_FLAG_* bits
 *   cuda_stream  cudaStream_t to enqueue on (NULL = legacy default stream)
 */
int la_prefill_ex(const void* q, const void* k, const void* v, const void* g, void* out,
                  float* kv_state_out, const float* kv_state_in, float* y_debug, int B,
                  int H, int64_t N, int d, int dtype, float eps, unsigned flags,
                  void* cuda_stream);

/*
 * Packed ("varlen") prefill of num_seqs sequences of different lengths, stored back to
 * back without padding -- the padding optimisation the MiniMax-01 deep dive lists
 * among its training-infrastructure improvements ("Post Training and Infra"), for the
 * same layer ("Hybrid Modeling", mechanism steps 2-4).  Each sequence is its own
 * causal recurrence (its own state, starting from kv_state_in[b] or zeros); the
 * RMSNorm is per token as in la_prefill.
 *   cu_seqlens   HOST array of num_seqs + 1 int64 token offsets: cu_seqlens[0] = 0,
 *                non-decreasing; sequence b is tokens [cu_seqlens[b], cu_seqlens[b+1])
 *                (empty sequences are allowed).  T = cu_seqlens[num_seqs].
 *   q, k, v, g   in  [T][H][d] (dtype);  out  out [T][H][d]
 *   kv_state_out out [num_seqs][H][d][d] fp32 or NULL (may equal kv_state_in)
 *   kv_state_in  in  [num_seqs][H][d][d] fp32 or NULL (zeros)
 *   y_debug      out [T][H][d] fp32 pre-norm y, or NULL
 * The chunk table is uploaded from host memory on the stream, which waits for the
 * stream's earlier work first.  Errors as for la_prefill_ex; additionally
 * LA_ERR_INVALID_ARG for a cu_seqlens that does not start at 0 or decreases.
 */
int la_prefill_varlen_ex(const void* q, const void* k, const void* v, const void* g, void* out,
                         float* kv_state_out, const float* kv_state_in, float* y_debug,
                         const int64_t* cu_seqlens, int num_seqs, int H, int d, int dtype,
                         float eps, unsigned flags, void* cuda_stream);

/* la_prefill_varlen_ex with bf16 I/O, zero initial states, no y_debug, eps = 1e-6 and
   the legacy default stream. */
int la_prefill_varlen(const void* q, const void* k, const void* v, const void* g, void* out,
                      float* kv_state_out, const int64_t* cu_seqlens, int num_seqs, int H,
                      int d);

/* Extended decode step: as la_decode_step with dtype, eps, an optional fp32 pre-norm
   y_debug [B][H][d] (or NULL; it must not overlap any other argument) and a stream. */
int la_decode_step_ex(float* kv_state, const void* q, const void* k, const void* v,
                      const void* g, void* out, float* y_debug, int B, int H, int d,
                      int dtype, float eps, void* cuda_stream);

/* Which prefill kernel la_prefill_ex would run for this shape on the current device:
   0 = tensor-core kernel, 1 = CUDA-core kernel, 2 = tensor-core kernel in the
   segment-parallel mode, or -(la_status) if la_prefill_ex would refuse the call.
   The segment-parallel mode is the blockwise route's prefix over the d x d states
   ("Hybrid Modeling": the O(d^2 n) form) spread over the SMs that a few heads leave
   idle.  It runs for one sequence (B == 1) when the device holds at least twice H
   head pairs plus a reducer pair (H <= 36 on a 148-SM B300) and N spans at least
   2 x 64 chunks of 128 tokens (N > 16256), unless LA_FLAG_SERIAL is set: the tokens are cut into segments of whole 128-token chunks,
   the state-only pass (as la_state_pass) sums K^T V^ over the tokens before each
   segment, the per-segment states are added in a fixed order, and then every segment
   runs its own head pairs from its prefix state, all segments in one launch.  It reads
   k and v once more for all but the last segment.  The result is deterministic and
   differs from the serial chain only in the order of fp32 additions of the state.  bf16 I/O runs the tensor-core kernel, and LA_F32 or LA_FLAG_SIMT
   the CUDA-core kernel; there is no silent switch between them: bf16 without
   LA_FLAG_SIMT on a shape the tensor-core kernel does not cover gives
   -LA_ERR_UNSUPPORTED (and la_prefill_ex returns LA_ERR_UNSUPPORTED).  The tensor-core
   kernel covers d = 128, H smaller than the number of two-CTA clusters the device holds
   at once (73 on a 148-SM B300: it keeps every head resident for the cross-head RMSNorm,
   runs the B sequences one after another, and needs at least one more cluster for the
   norm's reducers), N <= 2^30 and B * ceil(N / 128) <= 2^23.  The kernel's cross-CTA
   waits assume its CTAs run together: a concurrent kernel on another stream that
   holds SMs can delay it, and one that holds them past the 4 s wait bound makes the
   prefill record LA_ERR_TIMEOUT. */
int la_prefill_path(int B, int H, int64_t N, int d, int dtype, unsigned flags);

/*
 * Decode step that allocates nothing.  The paper has no counterpart: this entry point
 * exists for callers that cannot let a library call cudaMalloc -- for example a
 * serving engine that has reserved all device memory for its own pool, or a
 * latency-critical loop that cannot take the device synchronisation of
 * cudaMalloc/cudaFree.  It computes exactly what la_decode_step_ex computes (same
 * kernel, y_debug not offered), with the kernel's scratch (fp32 pre-norm y, per-head
 * sums of squares and per-sequence arrival counters) in a fixed array inside the
 * library's device data:
 *   - the array holds LA_NOALLOC_MAX_HEADS * (d + 2) 4-byte words (8.13 MiB), and every
 *     GPU that loads the library keeps it until the process exits;
 *   - B * H above LA_NOALLOC_MAX_HEADS returns LA_ERR_SCRATCH_LIMIT before any launch;
 *   - the first call on a device looks the array's device address up (one
 *     cudaGetSymbolAddress with that device current) and caches it; make that first
 *     call before any stream capture on that device;
 *   - the runtime loads device code lazily by default, so that first call is also
 *     when the array most likely takes its device memory: make it before reserving
 *     the rest of the device's memory for a pool (or set CUDA_MODULE_LOADING=EAGER,
 *     which places the array when the library is loaded);
 *   - all calls on a device share the one array and it keeps the last call's
 *     contents: calls whose kernels may overlap on the GPU (different streams with
 *     no ordering between them) race on it and must be ordered by the caller.
 * The kernel writes every scratch entry it reads and returns each counter it uses to
 * zero, so nothing is cleared between calls.  Arguments, layouts, dtype and eps are as for la_decode_step_ex; argument
 * errors are returned before any launch.
 */
#define LA_NOALLOC_MAX_HEADS 16384 /* B * H, e.g. 256 sequences x 64 heads */
int la_decode_step_noalloc(float* kv_state, const void* q, const void* k, const void* v,
                           const void* g, void* out, int B, int H, int d, int dtype,
                           float eps, void* cuda_stream);

/*
 * State of a run of tokens without its outputs ("Hybrid Modeling", MiniMax-01 deep dive,
 * Hugging Face blog: step 2's SiLU on K and V and step 3's K^T V, the d x d state of the
 * O(d^2 n) route):
 *     kv_state_out[b][h] = kv_state_in[b][h] + sum_t SiLU(k[b][t][h])^T SiLU(v[b][t][h])
 * i.e. the state la_prefill reaches after the same N tokens, at two fifths of its memory
 * traffic (k and v are read; q, g and out are not touched).  A rank of a
 * sequence-sharded prefill takes the states of the ranks before it from this.
 *   k, v          in  [B][N][H][d] bf16, pre-activation (or activated with
 *                     LA_FLAG_ACTIVATED in flags)
 *   kv_state_in   in  [B][H][d][d] fp32, or NULL for zeros
 *   kv_state_out  out [B][H][d][d] fp32; may equal kv_state_in, must not overlap k or v
 * bf16 only (LA_ERR_UNSUPPORTED for LA_F32), d = 128.  N = 0 copies (or zeroes) the
 * state.  The tokens of each (b, h) are split into segments summed on tensor cores and
 * the segments' fp32 states are added in a fixed order (deterministic); the segment
 * states live in the library's per-device workspace.  Device pointers, 16-byte aligned;
 * argument errors are returned before any launch; a bounded device wait that gives up
 * records LA_ERR_TIMEOUT.
 */
int la_state_pass(const void* k, const void* v, float* kv_state_out, const float* kv_state_in,
                  int B, int H, int64_t N, int d, int dtype, unsigned flags, void* cuda_stream);

/*
 * Fixed-order sum of fp32 arrays, for the state prefix of a sequence-sharded prefill
 * (the state a rank continues from is the sum of the states of the ranks before it):
 *     out[j] = (base ? base[j] : 0) + parts[0][j] + parts[1][j] + ... + parts[count-1][j]
 * added left to right, so every rank that sums the same arrays gets the same bits.
 *   parts  in  [count][n] fp32 (count >= 0);  base in [n] fp32 or NULL;  out out [n] fp32
 * n a multiple of 4; out may equal base and must not overlap parts.  Device pointers,
 * 16-byte aligned.  Argument errors are returned before any launch.
 */
int la_state_sum(const float* parts, int count, const float* base, float* out, int64_t n,
                 void* cuda_stream);

/* Static text for an la_status value. */
const char* la_status_string(int status);

/* Synchronises cuda_stream, returns and clears the device status word of the current
   device (LA_OK or LA_ERR_TIMEOUT), or LA_ERR_CUDA if synchronisation failed. */
int la_get_device_status(void* cuda_stream);

/*
 * Input projection of the layer on tensor cores: the step before the path
 * ("Hybrid Modeling", MiniMax-01 deep dive: step 1 "Input X", step 2 "Q, K, V =
 * SiLU(X)", the projections being the part the printed step leaves out; hidden size
 * 6144 in MiniMax-Text-01, the model card's "Model Architecture" list):
 *     [q | k | v | g] = x W^T,  then SiLU on q, k, v when flags has LA_PROJ_SILU
 *   x        in  [T][hidden] bf16, row-major
 *   w        in  [4*H*d][hidden] bf16, row-major: rows [0, Hd) make q, [Hd, 2Hd) k,
 *                [2Hd, 3Hd) v, [3Hd, 4Hd) g (a fused bias-free linear layer's weight)
 *   q,k,v,g  out [T][H][d] bf16 each: the layout la_prefill reads.  g is never
 *                activated (the layer applies sigmoid to it after the norm).
 *   flags    0 or LA_PROJ_SILU; with it the outputs are la_prefill_ex's
 *            LA_FLAG_ACTIVATED inputs, without it la_prefill's raw inputs
 * fp32 accumulation; each output element is rounded once to bf16 (RNE).  d must be 128
 * and H even (H*d a multiple of 256), hidden a multiple of 8 (LA_ERR_UNSUPPORTED
 * otherwise).  All pointers are device pointers, 16-byte aligned; the caller owns them;
 * no output may overlap x, w or another output.  T = 0 does nothing.  Argument errors
 * are returned before any launch; a bounded device wait that gives up records
 * LA_ERR_TIMEOUT in the device status word.
 */
#define LA_PROJ_SILU 1u
int la_qkvg_projection(const void* x, const void* w, void* q, void* k, void* v, void* g,
                       int64_t T, int hidden, int H, int d, unsigned flags, void* cuda_stream);

/*
 * The softmax layer of the hybrid stack: partial RoPE, then causal softmax attention.
 * MiniMax-Text-01 puts one such layer after every seven Lightning Attention layers
 * ("Hybrid Modeling", MiniMax-01 deep dive: RoPE on half of the head dimension); the
 * model card's "Model Architecture" list gives 64 heads of size 128 and RoPE base
 * 10,000,000.
 *     q', k' = RoPE(q), RoPE(k): features [0, 64) of each head rotated as pairs
 *              (i, i + 32) by the angle t * rope_base^(-i/32) at token t (t from 0 in
 *              every sequence); features [64, 128) unchanged
 *     out_t  = sum_{s <= t} softmax_s(q'_t . k'_s / sqrt(d)) v_s
 *   q, k, v  in  [B][N][H][d] bf16 (one key/value head per query head)
 *   out      out [B][N][H][d] bf16; must not overlap q, k or v
 *   rope_base    > 1 (1e7 for MiniMax-Text-01)
 * d must be 128 (LA_ERR_UNSUPPORTED otherwise), N <= 2^30; N = 0 does nothing.  The
 * rotated copies of q and k live in the library's per-device workspace (grown on
 * demand; 2 * B*N*H*d*2 bytes).  The cos/sin table (N*256 bytes) is cached per device
 * and rebuilt when a call needs more tokens or another base; that call waits for the
 * rebuild on its stream, so make it before any stream capture.  Scores, the softmax and
 * P*V run in fp32 with bf16 MMA operands; each output is rounded once to bf16.  Device
 * pointers, 16-byte aligned, owned by the caller.  Argument errors are returned before
 * any launch; a bounded device wait that gives up records LA_ERR_TIMEOUT.
 */
int la_softmax_attention(const void* q, const void* k, const void* v, void* out, int B, int H,
                         int64_t N, int d, double rope_base, void* cuda_stream);

/* Library version, major*10000 + minor*100 + patch. */
int la_version(void);

/* Number of kernels this library has launched in this process (all devices), for
   launch accounting by benchmarks.  Counts launches, not completed work. */
int64_t la_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LIGHTNING_ATTN_H */
