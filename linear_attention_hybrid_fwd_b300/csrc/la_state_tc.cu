// la_state_tc.cu -- the state of a run of tokens without its outputs (sm_103a).
//
// What it computes ("Hybrid Modeling", MiniMax-01 deep dive, Hugging Face blog: step 2
// K, V = SiLU(X) and step 3's K^T V, the d x d state of the O(d^2 n) route):
//     S_out = S_in + sum_t SiLU(k_t)^T SiLU(v_t)        per (sequence b, head h),
// which is where the token recurrence S_t = S_{t-1} + k^_t^T v^_t ends after the run.
// A rank of a sequence-sharded prefill needs exactly this of the ranks before it, and
// reads k and v only (two of the five tensors a prefill moves).
//
// Design (k_state_tc):
//  * The N tokens of each (b, h) are cut into nseg contiguous segments of whole
//    128-token chunks; one CTA per (segment, head, sequence) sums its segment's
//    K^T V into a 128 x 128 fp32 TMEM accumulator with tcgen05 MMAs (M = d_k, N = d_v,
//    K = 16 tokens per instruction, both operands MN-major straight from the token-major
//    tiles), and writes it to a partial slot.  nseg is chosen so that the grid covers
//    the SMs once (one CTA per SM, a single wave).
//  * k and v arrive by TMA in 128B-swizzled 64-feature x 128-token boxes, three chunks
//    in flight; sixteen warps apply SiLU in shared memory (tanh approximation, one SFU
//    operation per element), then one thread issues the chunk's 8 MMAs.  Rows past N
//    are the tensor map's zero fill, and SiLU(0) = 0.
//  * k_sum_rows adds the partial slots in segment order to S_in (deterministic), which
//    is also the fixed-order sum la_state_sum exposes.
//  * Every wait is bounded; a CTA that gives up records LA_ERR_TIMEOUT in the status
//    word, drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lightning_attn.h"
#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace {

using namespace sm100;

constexpr int D = kHeadDim;
constexpr int CH = 128;                      // tokens per chunk
constexpr int kThreadsS = 640;               // 20 warps
constexpr int kStages = 3;
constexpr uint32_t HALF = 16384;             // 128 tokens x 64 features, bf16
constexpr uint32_t STAGE = 4 * HALF;         // k (two halves) + v (two halves)
constexpr uint32_t SMEM_DYN_S = kStages * STAGE + 1024;
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr uint32_t IDESC_KV = idesc_bf16_f32(128, 128, 1, 1);  // A, B MN-major

struct SParams {
    float* part;      // [nseg][B][H][d][d] fp32 partial states
    int* status;
    int B, H, Nc, nseg, cps;  // chunks per sequence, segments, chunks per segment
};

struct SShared {
    uint64_t full[kStages], act[kStages], empty[kStages], done;
    uint32_t tmem_base;
    int abort_flag;
    int verdict;
};

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// SiLU of both bf16 halves: with h = x/2 (exact on the packed pair), SiLU(x) = h (1 + tanh h).
__device__ __forceinline__ uint32_t silu_bf16x2(uint32_t u) {
    uint32_t hh;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hh) : "r"(u), "r"(0x3F003F00u));
    const float h0 = __uint_as_float(hh << 16), h1 = __uint_as_float(hh & 0xFFFF0000u);
    return pack_bf16x2(fmaf(h0, tanh_approx(h0), h0), fmaf(h1, tanh_approx(h1), h1));
}
__device__ __forceinline__ uint4 silu_chunk(uint4 v) {
    return make_uint4(silu_bf16x2(v.x), silu_bf16x2(v.y), silu_bf16x2(v.z), silu_bf16x2(v.w));
}
// Byte offset of the 16-byte chunk `c` (0..7) of row `r` in a 128B-swizzled block.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}
// MN-major operand over two 64-element blocks HALF apart; k-step ks covers 16 tokens.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int ks) {
    return smem_desc_sw128(base + ks * 2048, HALF, 1024);
}

__device__ __forceinline__ bool abort_set(SShared& sh) {
    return *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0;
}
__device__ bool wait_bar(SShared& sh, int* status, uint64_t* bar, uint32_t parity,
                         bool honor_abort = true, uint64_t limit_ns = kTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (honor_abort && abort_set(sh)) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
                atomicExch(status, LA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
// Leader waits (bounded), the group syncs on named barrier `id`, every thread then
// observes the phase itself; returns the leader's verdict.
__device__ bool group_wait(SShared& sh, int* status, uint64_t* bar, uint32_t parity, bool leader,
                           uint32_t id, uint32_t n) {
    if (leader) sh.verdict = wait_bar(sh, status, bar, parity) ? 1 : 0;
    named_bar_sync(id, n);
    const bool ok = *reinterpret_cast<volatile int*>(&sh.verdict) != 0;
    if (ok)
        while (!mbar_try_wait(bar, parity)) {
        }
    named_bar_sync(id, n);
    return ok;
}

template <bool kAct>
__global__ void __launch_bounds__(kThreadsS, 1)
    k_state_tc(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
               const SParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ SShared sh;
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int c0 = seg * p.cps;
    const int c1 = c0 + p.cps < p.Nc ? c0 + p.cps : p.Nc;
    const int n = c1 > c0 ? c1 - c0 : 0;  // chunks of this CTA

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.act[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.done, 1);
        sh.abort_flag = 0;
        sh.verdict = 0;
        fence_mbar_init();
    }
    if (warp == 2) tmem_alloc(&sh.tmem_base, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------- TMA producer: k and v
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int s = i % kStages;
                const uint32_t ph = static_cast<uint32_t>(i / kStages) & 1u;
                if (!wait_bar(sh, p.status, &sh.empty[s], ph ^ 1u)) break;
                uint8_t* st = sm + s * STAGE;
                const int y = (c0 + i) * CH;
                mbar_arrive_expect_tx(&sh.full[s], STAGE);
                tma_load_3d(st, &tk, h * D, y, b, &sh.full[s]);
                tma_load_3d(st + HALF, &tk, h * D + 64, y, b, &sh.full[s]);
                tma_load_3d(st + 2 * HALF, &tv, h * D, y, b, &sh.full[s]);
                tma_load_3d(st + 3 * HALF, &tv, h * D + 64, y, b, &sh.full[s]);
                issued = i + 1;
            }
            for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
                wait_bar(sh, p.status, &sh.full[i % kStages],
                         static_cast<uint32_t>(i / kStages) & 1u, false, kDrainNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer: S += K^T V
        if (lane == 0) {
            for (int i = 0; i < n; ++i) {
                const int s = i % kStages;
                if (!wait_bar(sh, p.status, &sh.act[s], static_cast<uint32_t>(i / kStages) & 1u))
                    break;
                tc_fence_after();
                const uint32_t ka = sbase + s * STAGE, va = ka + 2 * HALF;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tm, desc_mnmajor(ka, ks), desc_mnmajor(va, ks), IDESC_KV,
                           (i > 0 || ks > 0) ? 1u : 0u);
                mma_commit(&sh.empty[s]);
            }
            mma_commit(&sh.done);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ SiLU (sixteen warps), then the
        // epilogue (warps 4-7: the four TMEM lane quadrants)
        const int u = tid - 128;                     // 0..511
        const int t = u & 127, sel = u >> 7;         // token row; (tile, feature half)
        const bool leader = u == 0;
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            const int s = i % kStages;
            if (!group_wait(sh, p.status, &sh.full[s], static_cast<uint32_t>(i / kStages) & 1u,
                            leader, 1, 512)) {
                ok = false;
                break;
            }
            if (!kAct) {
                // block sel: k half 0, k half 1, v half 0, v half 1
                uint8_t* blk = sm + s * STAGE + sel * HALF;
#pragma unroll
                for (int g4 = 0; g4 < 2; ++g4) {
                    uint4 x[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        x[j] = *reinterpret_cast<const uint4*>(blk + swz(t, 4 * g4 + j));
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(blk + swz(t, 4 * g4 + j)) = silu_chunk(x[j]);
                }
                fence_proxy_async_smem();
            }
            named_bar_sync(1, 512);
            if (leader) mbar_arrive(&sh.act[s]);
        }
        if (warp < 8) {
            // the partial state of this segment: TMEM lane t = row d_k of S
            const int q4 = warp & 3;
            const int r = q4 * 32 + lane;
            const bool lead4 = r == 0;
            bool fine = ok;
            if (lead4) sh.verdict = fine && wait_bar(sh, p.status, &sh.done, 0) ? 1 : 0;
            named_bar_sync(2, 128);
            fine = *reinterpret_cast<volatile int*>(&sh.verdict) != 0;
            if (fine) {
                while (!mbar_try_wait(&sh.done, 0)) {
                }
                tc_fence_after();
                float* dst = p.part +
                             ((((static_cast<size_t>(seg) * p.B + b) * p.H + h) * D + r) * D);
                const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    LA_TMEM_LD32(lb + 32 * c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + 32 * c + j) = make_float4(
                            n > 0 ? __uint_as_float(v[j]) : 0.f,
                            n > 0 ? __uint_as_float(v[j + 1]) : 0.f,
                            n > 0 ? __uint_as_float(v[j + 2]) : 0.f,
                            n > 0 ? __uint_as_float(v[j + 3]) : 0.f);
                }
            }
        }
    }

    // ---------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (tid == 32)  // the MMAs issued (on any path) complete before TMEM is freed
        wait_bar(sh, p.status, &sh.done, 0, false, kDrainNs);
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tm, 128);
}

// out[j] = (base ? base[j] : 0) + sum_{i < count} parts[i * n + j], in the order of i;
// n a multiple of 4, 16-byte aligned arrays.
__global__ void __launch_bounds__(256) k_sum_rows(const float* __restrict__ parts, int count,
                                                  int64_t n, const float* base, float* out) {
    const int64_t n4 = n / 4;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n4;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 acc = base ? reinterpret_cast<const float4*>(base)[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < count; ++i) {
            const float4 x = __ldcs(reinterpret_cast<const float4*>(parts + static_cast<size_t>(i) * n) + j);
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
        }
        reinterpret_cast<float4*>(out)[j] = acc;
    }
}

// The prefixes of a segment-parallel prefill in one pass: out[s][j] = (base ? base[j] :
// 0) + sum_{i < s * per} parts[i][j] for s = 0 .. nout - 1, each the same running sum,
// in the order of i, that k_sum_rows forms for count = s * per (bitwise the same).
__global__ void __launch_bounds__(256) k_prefix_rows(const float* __restrict__ parts, int per,
                                                     int nout, int64_t n, const float* base,
                                                     float* out) {
    const int64_t n4 = n / 4;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n4;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 acc = base ? reinterpret_cast<const float4*>(base)[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < nout; ++s) {
            reinterpret_cast<float4*>(out + static_cast<size_t>(s) * n)[j] = acc;
            if (s + 1 == nout) break;
            for (int i = s * per; i < (s + 1) * per; ++i) {
                const float4 x =
                    __ldcs(reinterpret_cast<const float4*>(parts + static_cast<size_t>(i) * n) + j);
                acc.x += x.x;
                acc.y += x.y;
                acc.z += x.z;
                acc.w += x.w;
            }
        }
    }
}

int g_num_sms[64];

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!g_num_sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        g_num_sms[dev] = v;
    }
    return g_num_sms[dev];
}

}  // namespace

int state_segments(int B, int H, int64_t N) {
    // one CTA per SM at most (one wave): as many segments per (b, h) as fit the SMs
    const int64_t Nc = (N + CH - 1) / CH;
    const int64_t want = static_cast<int64_t>(num_sms()) / (static_cast<int64_t>(B) * H);
    int64_t nseg = want < 1 ? 1 : want;
    if (nseg > Nc) nseg = Nc;
    if (nseg > 65535) nseg = 65535;
    return static_cast<int>(nseg < 1 ? 1 : nseg);
}

int launch_sum_rows(const float* parts, int count, int64_t n, const float* base, float* out,
                    cudaStream_t st) {
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = 8 * static_cast<int64_t>(num_sms());
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_sum_rows<<<static_cast<unsigned>(blocks), 256, 0, st>>>(parts, count, n, base, out);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    note_launches(1);
    return LA_OK;
}

int launch_prefix_rows(const float* parts, int per, int nout, int64_t n, const float* base,
                       float* out, cudaStream_t st) {
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = 8 * static_cast<int64_t>(num_sms());
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_prefix_rows<<<static_cast<unsigned>(blocks), 256, 0, st>>>(parts, per, nout, n, base, out);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    note_launches(1);
    return LA_OK;
}

int launch_state_tc(const void* k, const void* v, float* part, int B, int H, int64_t N,
                    int nseg, bool activated, int* status, cudaStream_t st) {
    CUtensorMap mk, mv;
    if (!encode_io_map_bf16(&mk, k, B, H, N) || !encode_io_map_bf16(&mv, v, B, H, N))
        return LA_ERR_UNSUPPORTED;
    auto fn = activated ? k_state_tc<true> : k_state_tc<false>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_DYN_S)) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    SParams prm;
    prm.part = part;
    prm.status = status;
    prm.B = B;
    prm.H = H;
    prm.Nc = static_cast<int>((N + CH - 1) / CH);
    prm.nseg = nseg;
    prm.cps = (prm.Nc + nseg - 1) / nseg;
    fn<<<dim3(static_cast<unsigned>(nseg), static_cast<unsigned>(H), static_cast<unsigned>(B)),
         kThreadsS, SMEM_DYN_S, st>>>(mk, mv, prm);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    note_launches(1);
    return LA_OK;
}

}  // namespace la
