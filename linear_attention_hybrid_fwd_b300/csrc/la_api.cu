// la_api.cu -- the C ABI of liblightning_attn.so (declared in include/lightning_attn.h):
// argument validation, the per-device workspace, and launch sequencing on the
// caller's stream.  Every numeric step runs in the CUDA kernels of la_simt.cu and
// la_prefill_tc.cu; nothing here computes on the host.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/lightning_attn.h"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int64_t> g_launches{0};
std::mutex g_ws_mutex;
Workspace g_ws[kMaxDevices];

struct XchState {
    float* base = nullptr;   // 2 flag banks of `words` words
    size_t words = 0;
    unsigned bank = 0;       // the bank the next launch writes
    size_t dirty[2] = {0, 0};
    float* part = nullptr;   // partials
    size_t part_floats = 0;
};
XchState g_xch[kMaxDevices];

struct ItemBuf {
    int4* dev = nullptr;     // chunk table of the last packed-batch launch
    size_t cap = 0;
};
ItemBuf g_items[kMaxDevices];

struct WorkspaceReaper {
    ~WorkspaceReaper() {
        // Process teardown: the driver may already be gone; ignore errors.
        for (auto& x : g_xch) {
            if (x.base) cudaFree(x.base);
            if (x.part) cudaFree(x.part);
        }
        for (auto& i : g_items)
            if (i.dev) cudaFree(i.dev);
        for (auto& w : g_ws) {
            if (w.base) cudaFree(w.base);
            if (w.status) cudaFree(w.status);
            if (w.dec_cnt) cudaFree(w.dec_cnt);
        }
    }
} g_reaper;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

// Failure-detection test hook: with LA_TEST_WITHHOLD_ARRIVAL=1 in the environment, a
// tensor-core prefill starts with one cross-CTA arrival counter off its sentinel, so
// one chunk never gathers all its head halves.  Every wait in the kernel is bounded, so
// the launch ends with LA_ERR_TIMEOUT in the status word and the context stays usable.
bool withhold_requested() {
    const char* e = getenv("LA_TEST_WITHHOLD_ARRIVAL");
    return e && e[0] == '1';
}

}  // namespace

void note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int workspace_acquire(size_t bytes, cudaStream_t st, Workspace* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace& w = g_ws[dev];
    if (!w.status) {
        int* status = nullptr;
        unsigned* cnt = nullptr;
        if (cudaMalloc(&status, 256) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_NOMEM;
        }
        const size_t cbytes = size_t(kDecodeCounterSlots) * sizeof(unsigned);
        if (cudaMalloc(&cnt, cbytes) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(status);
            return LA_ERR_NOMEM;
        }
        if (cudaMemsetAsync(status, 0, 256, st) != cudaSuccess ||
            cudaMemsetAsync(cnt, 0, cbytes, st) != cudaSuccess) {
            cudaFree(status);
            cudaFree(cnt);
            return LA_ERR_CUDA;
        }
        w.status = status;
        w.dec_cnt = cnt;
    }
    if (bytes > w.bytes) {
        // cudaFree waits for work already queued on the device, so a smaller
        // workspace still in use by an earlier call is not released under it.
        if (w.base) cudaFree(w.base);
        w.base = nullptr;
        w.bytes = 0;
        const size_t want = (bytes + (size_t(1) << 21) - 1) & ~((size_t(1) << 21) - 1);
        if (cudaMalloc(&w.base, want) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_NOMEM;
        }
        w.bytes = want;
    }
    *out = w;
    return LA_OK;
}

int xch_acquire(size_t flag_words, size_t part_floats, cudaStream_t st, XchLease* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    XchState& x = g_xch[dev];
    if (flag_words > x.words) {
        if (x.base) cudaFree(x.base);  // waits for work already queued on the device
        x.base = nullptr;
        x.words = 0;
        const size_t want = (flag_words + (size_t(1) << 16) - 1) & ~((size_t(1) << 16) - 1);
        if (cudaMalloc(&x.base, 2 * want * sizeof(float)) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_NOMEM;
        }
        // every word starts empty (kXchEmpty is the byte 0x80 repeated)
        if (cudaMemsetAsync(x.base, 0x80, 2 * want * sizeof(float), st) != cudaSuccess) {
            cudaFree(x.base);
            x.base = nullptr;
            return LA_ERR_CUDA;
        }
        x.words = want;
        x.bank = 0;
        x.dirty[0] = x.dirty[1] = 0;
    }
    if (part_floats > x.part_floats) {
        if (x.part) cudaFree(x.part);
        x.part = nullptr;
        x.part_floats = 0;
        const size_t want = (part_floats + (size_t(1) << 18) - 1) & ~((size_t(1) << 18) - 1);
        if (cudaMalloc(&x.part, want * sizeof(float)) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_NOMEM;
        }
        x.part_floats = want;
    }
    out->bank = x.bank;
    out->use = x.base + x.bank * x.words;
    out->clear = reinterpret_cast<uint32_t*>(x.base + (x.bank ^ 1u) * x.words);
    out->clear_words = x.dirty[x.bank ^ 1u];
    out->part = x.part;
    return LA_OK;
}

void xch_commit(const XchLease& lease, size_t words_used) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    XchState& x = g_xch[dev];
    x.dirty[lease.bank] = words_used;
    x.dirty[lease.bank ^ 1u] = 0;
    x.bank = lease.bank ^ 1u;
}

// Uploads a packed batch's chunk table into the device's table buffer (grown on demand)
// on `st`.  The copy is from pageable memory, so it waits for the stream's earlier work.
int items_upload(const std::vector<int4>& items, cudaStream_t st, const int4** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    ItemBuf& b = g_items[dev];
    if (items.size() > b.cap) {
        if (b.dev) cudaFree(b.dev);
        b.dev = nullptr;
        b.cap = 0;
        const size_t want = (items.size() + 4095) & ~size_t(4095);
        if (cudaMalloc(&b.dev, want * sizeof(int4)) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_NOMEM;
        }
        b.cap = want;
    }
    if (cudaMemcpyAsync(b.dev, items.data(), items.size() * sizeof(int4), cudaMemcpyHostToDevice,
                        st) != cudaSuccess)
        return LA_ERR_CUDA;
    *out = b.dev;
    return LA_OK;
}

}  // namespace la

using namespace la;

extern "C" {

const char* la_status_string(int s) {
    switch (s) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument";
        case LA_ERR_UNSUPPORTED: return "unsupported shape (head size must be 128)";
        case LA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case LA_ERR_CUDA: return "CUDA error";
        case LA_ERR_NOMEM: return "out of device memory for the workspace";
        case LA_ERR_TIMEOUT: return "a kernel gave up a bounded cross-CTA wait";
        case LA_ERR_SCRATCH_LIMIT:
            return "B*H exceeds the fixed scratch of la_decode_step_noalloc";
        default: return "unknown status";
    }
}

int la_version(void) { return 200; }  // 0.2.0: + varlen, projection, softmax layer

int64_t la_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int la_prefill_ex(const void* q, const void* k, const void* v, const void* g, void* out,
                  float* kv_state_out, const float* kv_state_in, float* y_debug, int B, int H,
                  int64_t N, int d, int dtype, float eps, unsigned flags, void* cuda_stream) {
    // ---- host-side validation: nothing is launched or written on failure ----
    if (B <= 0 || H <= 0 || N < 0 || d <= 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 && dtype != LA_F32) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (flags & ~(LA_FLAG_SIMT | LA_FLAG_ACTIVATED | LA_FLAG_SERIAL)) return LA_ERR_INVALID_ARG;
    if (d != kHeadDim) return LA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 4096) return LA_ERR_UNSUPPORTED;
    // element counts: B*N*H*d must stay well inside int64 (the kernels index in int64)
    if (N > (int64_t(1) << 40) / ((int64_t)B * H * d)) return LA_ERR_INVALID_ARG;
    const bool bf16 = dtype == LA_BF16;
    const size_t esz = bf16 ? 2 : 4;
    const int64_t nelem = (int64_t)B * N * H * d;
    const size_t io_bytes = (size_t)nelem * esz;
    const size_t state_bytes = (size_t)B * H * d * d * sizeof(float);
    if (N > 0 && (!q || !k || !v || !g || !out)) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, out, kv_state_out, kv_state_in, y_debug};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    if (N > 0) {
        const void* ins[] = {q, k, v, g};
        for (const void* p : ins)
            if (overlaps(out, io_bytes, p, io_bytes)) return LA_ERR_INVALID_ARG;
        if (overlaps(kv_state_out, state_bytes, out, io_bytes)) return LA_ERR_INVALID_ARG;
        if (y_debug && overlaps(y_debug, (size_t)nelem * 4, out, io_bytes))
            return LA_ERR_INVALID_ARG;
    }
    if (kv_state_in && kv_state_out && kv_state_in != kv_state_out &&
        overlaps(kv_state_in, state_bytes, kv_state_out, state_bytes))
        return LA_ERR_INVALID_ARG;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (N == 0) {
        if (kv_state_out && kv_state_out != kv_state_in) {
            if (kv_state_in)
                return cuda_status(cudaMemcpyAsync(kv_state_out, kv_state_in, state_bytes,
                                                   cudaMemcpyDeviceToDevice, st));
            return launch_zero_state(kv_state_out, (int64_t)B * H * d * d, st);
        }
        return LA_OK;
    }

    // bf16 runs on the tensor-core kernel unless the caller asks for the CUDA-core one;
    // a shape the tensor-core kernel does not cover is refused, not switched silently
    const bool use_tc = bf16 && !(flags & LA_FLAG_SIMT);
    if (use_tc && prefill_tc_supported(B, H, N) != LA_OK) return LA_ERR_UNSUPPORTED;
    if (use_tc) {
        // one long sequence with few heads: segments run side by side from prefix states
        int seg_items = 0, fine = 1;
        const int nseg = (flags & LA_FLAG_SERIAL) ? 1
                                                  : prefill_tc_segment_plan(B, H, N, &seg_items, &fine);
        const size_t set_floats = (size_t)H * d * d;  // one state per head (B == 1)
        const size_t seg_floats = nseg > 1 ? ((size_t)(nseg - 1) * fine + nseg) * set_floats : 0;
        Workspace ws;
        int rc = workspace_acquire(seg_floats * sizeof(float), st, &ws);
        if (rc != LA_OK) return rc;
        XchLease xl;
        const int items = prefill_tc_items(B, N);
        rc = xch_acquire(prefill_tc_flag_words(items), prefill_tc_part_floats(H, nseg), st, &xl);
        if (rc != LA_OK) return rc;
        if (withhold_requested()) {
            // failure-detection test: chunk 0's arrival counter starts off its sentinel,
            // as if one head half's arrival were lost; the launch's waits run out
            // (bounded) and the status word reads LA_ERR_TIMEOUT
            if (cudaMemsetAsync(xl.use, 0, sizeof(unsigned), st) != cudaSuccess)
                return LA_ERR_CUDA;
        }
        const bool act = (flags & LA_FLAG_ACTIVATED) != 0;
        const float* S_seg = nullptr;
        if (nseg > 1) {
            // the state of the tokens before each segment: K^T V^ of fixed pieces (the
            // state pass), then prefix[s] = S_in + the pieces before segment s, in order
            float* pieces = static_cast<float*>(ws.base);
            float* prefix = pieces + (size_t)(nseg - 1) * fine * set_floats;
            const int64_t Np = (int64_t)(nseg - 1) * seg_items * 128;
            rc = launch_state_tc(k, v, pieces, 1, H, Np, (nseg - 1) * fine, act, ws.status, st);
            if (rc == LA_OK)
                rc = launch_prefix_rows(pieces, fine, nseg, (int64_t)set_floats, kv_state_in,
                                        prefix, st);
            if (rc != LA_OK) return rc;
            S_seg = prefix;
        }
        return launch_prefill_tc(q, k, v, g, out, kv_state_in, kv_state_out, y_debug, B, H, N,
                                 eps, act, ws, xl, st, nseg, seg_items, S_seg);
    }
    // CUDA-core kernel: y in fp32 (into y_debug when given), then the norm/gate pass.
    float* y = y_debug;
    if (!y) {
        Workspace ws;
        int rc = workspace_acquire((size_t)nelem * sizeof(float), st, &ws);
        if (rc != LA_OK) return rc;
        y = static_cast<float*>(ws.base);
    }
    int rc = launch_prefill_simt(q, k, v, kv_state_in, y, kv_state_out, B, H, N, bf16,
                                 (flags & LA_FLAG_ACTIVATED) != 0, st);
    if (rc != LA_OK) return rc;
    return launch_norm_gate_rows(y, g, out, (int64_t)B * N, H * d, eps, bf16, st);
}

int la_prefill_path(int B, int H, int64_t N, int d, int dtype, unsigned flags) {
    if (B <= 0 || H <= 0 || N < 0 || d <= 0) return -LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 && dtype != LA_F32) return -LA_ERR_INVALID_ARG;
    if (flags & ~(LA_FLAG_SIMT | LA_FLAG_ACTIVATED | LA_FLAG_SERIAL)) return -LA_ERR_INVALID_ARG;
    if (d != kHeadDim) return -LA_ERR_UNSUPPORTED;
    if (dtype != LA_BF16 || (flags & LA_FLAG_SIMT)) return 1;
    if (N == 0) return 0;  // nothing is launched
    if (prefill_tc_supported(B, H, N) != LA_OK) return -LA_ERR_UNSUPPORTED;
    int seg_items = 0, fine = 1;
    if (!(flags & LA_FLAG_SERIAL) && prefill_tc_segment_plan(B, H, N, &seg_items, &fine) > 1)
        return 2;
    return 0;
}

int la_prefill(const void* q, const void* k, const void* v, const void* g, void* out,
               float* kv_state_out, int B, int H, int64_t N, int d) {
    return la_prefill_ex(q, k, v, g, out, kv_state_out, nullptr, nullptr, B, H, N, d, LA_BF16,
                         1e-6f, 0u, nullptr);
}

int la_prefill_varlen_ex(const void* q, const void* k, const void* v, const void* g, void* out,
                         float* kv_state_out, const float* kv_state_in, float* y_debug,
                         const int64_t* cu_seqlens, int num_seqs, int H, int d, int dtype,
                         float eps, unsigned flags, void* cuda_stream) {
    // ---- host-side validation: nothing is launched or written on failure ----
    if (num_seqs <= 0 || H <= 0 || d <= 0 || !cu_seqlens) return LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 && dtype != LA_F32) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    // a packed batch always runs one chunk chain per (sequence, head): LA_FLAG_SERIAL
    // is accepted and changes nothing
    if (flags & ~(LA_FLAG_SIMT | LA_FLAG_ACTIVATED | LA_FLAG_SERIAL)) return LA_ERR_INVALID_ARG;
    if (d != kHeadDim) return LA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || H > 4096) return LA_ERR_UNSUPPORTED;
    if (cu_seqlens[0] != 0) return LA_ERR_INVALID_ARG;
    for (int b = 0; b < num_seqs; ++b)
        if (cu_seqlens[b + 1] < cu_seqlens[b]) return LA_ERR_INVALID_ARG;
    const int64_t T = cu_seqlens[num_seqs];
    if (T > (int64_t(1) << 30) / H) return LA_ERR_INVALID_ARG;
    const bool bf16 = dtype == LA_BF16;
    const size_t esz = bf16 ? 2 : 4;
    const size_t io_bytes = (size_t)T * H * d * esz;
    const size_t state_bytes = (size_t)num_seqs * H * d * d * sizeof(float);
    if (T > 0 && (!q || !k || !v || !g || !out)) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, out, kv_state_out, kv_state_in, y_debug};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    if (T > 0) {
        const void* ins[] = {q, k, v, g};
        for (const void* p : ins)
            if (overlaps(out, io_bytes, p, io_bytes)) return LA_ERR_INVALID_ARG;
        if (overlaps(kv_state_out, state_bytes, out, io_bytes)) return LA_ERR_INVALID_ARG;
        if (y_debug && overlaps(y_debug, (size_t)T * H * d * 4, out, io_bytes))
            return LA_ERR_INVALID_ARG;
    }
    if (kv_state_in && kv_state_out && kv_state_in != kv_state_out &&
        overlaps(kv_state_in, state_bytes, kv_state_out, state_bytes))
        return LA_ERR_INVALID_ARG;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    const size_t head_state = (size_t)H * d * d;  // floats per sequence
    // sequences without tokens: their final state is their initial state
    if (kv_state_out && kv_state_out != kv_state_in) {
        for (int b = 0; b < num_seqs; ++b) {
            if (cu_seqlens[b + 1] != cu_seqlens[b]) continue;
            int rc = kv_state_in ? cuda_status(cudaMemcpyAsync(
                                       kv_state_out + b * head_state, kv_state_in + b * head_state,
                                       head_state * sizeof(float), cudaMemcpyDeviceToDevice, st))
                                 : launch_zero_state(kv_state_out + b * head_state,
                                                     (int64_t)head_state, st);
            if (rc != LA_OK) return rc;
        }
    }
    if (T == 0) return LA_OK;

    const bool use_tc = bf16 && !(flags & LA_FLAG_SIMT);
    if (use_tc && prefill_tc_supported(1, H, T) != LA_OK) return LA_ERR_UNSUPPORTED;
    if (use_tc) {
        std::vector<int4> items;
        for (int b = 0; b < num_seqs; ++b) {
            const int64_t n = cu_seqlens[b + 1] - cu_seqlens[b];
            for (int64_t c0 = 0; c0 < n; c0 += kTcChunk) {
                const int64_t nv = n - c0 < kTcChunk ? n - c0 : kTcChunk;
                items.push_back(make_int4(static_cast<int>(cu_seqlens[b] + c0),
                                          static_cast<int>(nv), b, c0 == 0 ? 1 : 0));
            }
        }
        Workspace ws;
        int rc = workspace_acquire(0, st, &ws);
        if (rc != LA_OK) return rc;
        const int total = static_cast<int>(items.size());
        XchLease xl;
        rc = xch_acquire(prefill_tc_flag_words(total), prefill_tc_part_floats(H, 1), st, &xl);
        if (rc != LA_OK) return rc;
        const int4* dev_items = nullptr;
        rc = items_upload(items, st, &dev_items);
        if (rc != LA_OK) return rc;
        return launch_prefill_tc_varlen(q, k, v, g, out, kv_state_in, kv_state_out, y_debug, H,
                                        T, total, dev_items, eps, (flags & LA_FLAG_ACTIVATED) != 0, ws,
                                        xl, st);
    }
    // CUDA-core kernel (fp32 I/O, or on request): one prefill per sequence
    const size_t row = (size_t)H * d;  // elements per token
    for (int b = 0; b < num_seqs; ++b) {
        const int64_t r0 = cu_seqlens[b], n = cu_seqlens[b + 1] - r0;
        if (n == 0) continue;
        const size_t off = (size_t)r0 * row * esz;
        auto at = [&](const void* p) {
            return static_cast<const void*>(static_cast<const char*>(p) + off);
        };
        int rc = la_prefill_ex(at(q), at(k), at(v), at(g), static_cast<char*>(out) + off,
                               kv_state_out ? kv_state_out + b * head_state : nullptr,
                               kv_state_in ? kv_state_in + b * head_state : nullptr,
                               y_debug ? y_debug + (size_t)r0 * row : nullptr, 1, H, n, d, dtype,
                               eps, flags, cuda_stream);
        if (rc != LA_OK) return rc;
    }
    return LA_OK;
}

int la_prefill_varlen(const void* q, const void* k, const void* v, const void* g, void* out,
                      float* kv_state_out, const int64_t* cu_seqlens, int num_seqs, int H,
                      int d) {
    return la_prefill_varlen_ex(q, k, v, g, out, kv_state_out, nullptr, nullptr, cu_seqlens,
                                num_seqs, H, d, LA_BF16, 1e-6f, 0u, nullptr);
}

int la_decode_step_ex(float* kv_state, const void* q, const void* k, const void* v,
                      const void* g, void* out, float* y_debug, int B, int H, int d, int dtype,
                      float eps, void* cuda_stream) {
    if (B <= 0 || H <= 0 || d <= 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 && dtype != LA_F32) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (d != kHeadDim) return LA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535 || (int64_t)B * H > (int64_t(1) << 31) - 1)
        return LA_ERR_UNSUPPORTED;
    if (!kv_state || !q || !k || !v || !g || !out) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {kv_state, q, k, v, g, out, y_debug};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    const bool bf16 = dtype == LA_BF16;
    const size_t io_bytes = (size_t)B * H * d * (bf16 ? 2 : 4);
    const size_t state_bytes = (size_t)B * H * d * d * sizeof(float);
    const void* ins[] = {q, k, v, g};
    for (const void* p : ins) {
        if (overlaps(out, io_bytes, p, io_bytes)) return LA_ERR_INVALID_ARG;
        if (overlaps(kv_state, state_bytes, p, io_bytes)) return LA_ERR_INVALID_ARG;
    }
    if (overlaps(kv_state, state_bytes, out, io_bytes)) return LA_ERR_INVALID_ARG;
    if (y_debug) {  // fp32 [B][H][d], written by the kernel
        const size_t y_bytes = (size_t)B * H * d * sizeof(float);
        for (const void* p : ins)
            if (overlaps(y_debug, y_bytes, p, io_bytes)) return LA_ERR_INVALID_ARG;
        if (overlaps(y_debug, y_bytes, out, io_bytes) ||
            overlaps(y_debug, y_bytes, kv_state, state_bytes))
            return LA_ERR_INVALID_ARG;
    }

    const size_t ny = (size_t)B * H * d;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    Workspace ws;
    int rc = workspace_acquire((ny + (size_t)B * H) * sizeof(float) + 256, st, &ws);
    if (rc != LA_OK) return rc;
    float* y = y_debug ? y_debug : static_cast<float*>(ws.base);
    float* ss = static_cast<float*>(ws.base) + ny;
    return launch_decode(kv_state, q, k, v, g, out, y, ss, ws.dec_cnt, B, H, eps, bf16, st);
}

int la_decode_step(float* kv_state, const void* q, const void* k, const void* v,
                   const void* g, void* out, int B, int H, int d) {
    return la_decode_step_ex(kv_state, q, k, v, g, out, nullptr, B, H, d, LA_BF16, 1e-6f,
                             nullptr);
}

int la_state_pass(const void* k, const void* v, float* kv_state_out, const float* kv_state_in,
                  int B, int H, int64_t N, int d, int dtype, unsigned flags, void* cuda_stream) {
    // ---- host-side validation: nothing is launched or written on failure ----
    if (B <= 0 || H <= 0 || N < 0 || d <= 0 || !kv_state_out) return LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 && dtype != LA_F32) return LA_ERR_INVALID_ARG;
    if (flags & ~LA_FLAG_ACTIVATED) return LA_ERR_INVALID_ARG;
    if (d != kHeadDim || dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return LA_ERR_UNSUPPORTED;
    if (N > (int64_t(1) << 40) / ((int64_t)B * H * d)) return LA_ERR_INVALID_ARG;
    if (N > 0 && (!k || !v)) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {k, v, kv_state_out, kv_state_in};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    const size_t io_bytes = (size_t)B * N * H * d * 2;
    const size_t state_bytes = (size_t)B * H * d * d * sizeof(float);
    if (N > 0 && (overlaps(kv_state_out, state_bytes, k, io_bytes) ||
                  overlaps(kv_state_out, state_bytes, v, io_bytes)))
        return LA_ERR_INVALID_ARG;
    if (kv_state_in && kv_state_in != kv_state_out &&
        overlaps(kv_state_in, state_bytes, kv_state_out, state_bytes))
        return LA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    const int64_t n = (int64_t)B * H * d * d;
    if (N == 0) {
        if (kv_state_in == kv_state_out) return LA_OK;
        if (kv_state_in)
            return cuda_status(cudaMemcpyAsync(kv_state_out, kv_state_in, state_bytes,
                                               cudaMemcpyDeviceToDevice, st));
        return launch_zero_state(kv_state_out, n, st);
    }
    const int nseg = state_segments(B, H, N);
    Workspace ws;
    int rc = workspace_acquire((size_t)nseg * state_bytes, st, &ws);
    if (rc != LA_OK) return rc;
    float* part = static_cast<float*>(ws.base);
    rc = launch_state_tc(k, v, part, B, H, N, nseg, (flags & LA_FLAG_ACTIVATED) != 0, ws.status,
                         st);
    if (rc != LA_OK) return rc;
    return launch_sum_rows(part, nseg, n, kv_state_in, kv_state_out, st);
}

int la_state_sum(const float* parts, int count, const float* base, float* out, int64_t n,
                 void* cuda_stream) {
    if (count < 0 || n < 0 || !out || (n % 4) != 0) return LA_ERR_INVALID_ARG;
    if (count > 0 && !parts) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {parts, base, out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    const size_t bytes = (size_t)n * sizeof(float);
    if (count > 0 && overlaps(out, bytes, parts, (size_t)count * bytes)) return LA_ERR_INVALID_ARG;
    if (base && base != out && overlaps(base, bytes, out, bytes)) return LA_ERR_INVALID_ARG;
    if (n == 0) return LA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    return launch_sum_rows(parts, count, n, base, out, st);
}

int la_get_device_status(void* cuda_stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return LA_ERR_CUDA;
    Workspace ws;
    int rc = workspace_acquire(0, st, &ws);
    if (rc != LA_OK) return rc;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LA_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, ws.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LA_ERR_CUDA;
    if (h != 0 && cudaMemset(ws.status, 0, sizeof(int)) != cudaSuccess) return LA_ERR_CUDA;
    return h == 0 ? LA_OK : h;
}

}  // extern "C"
