// la_simt.cu -- CUDA-core kernels of the Lightning Attention forward.
//
//  * k_prefill_simt: chunked causal linear attention in fp32 FFMA.  Within a chunk
//    of C tokens it forms the masked block (Q^ K^T * M) V^ and adds Q^ S_prefix; the
//    state then absorbs K^T V of the chunk -- the blockwise, flash-like route with
//    O(d^2 n) cost named in "Hybrid Modeling" (MiniMax-01 deep dive, Hugging Face
//    blog).  This is the kernel of the fp32 I/O mode; for bf16 it is the
//    CUDA-core alternative to the tensor-core kernel.
//  * k_norm_gate_rows: step 4 of the mechanism, RMSNorm over the H*d features of a
//    token times sigmoid(g), one CTA per token row.
//  * k_decode_step: one-token decode against the carried state, with the norm over
//    all heads of a sequence fused in (the last head of each sequence applies it).
//
// All accumulation is fp32; SiLU and sigmoid use the accurate expf.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lightning_attn.h"
#include "la_internal.h"

namespace la {
namespace {

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

template <typename T> __device__ __forceinline__ float ldf(const T* p, int64_t i);
template <> __device__ __forceinline__ float ldf<float>(const float* p, int64_t i) {
    return p[i];
}
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p,
                                                                  int64_t i) {
    return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ void stf(T* p, int64_t i, float x);
template <> __device__ __forceinline__ void stf<float>(float* p, int64_t i, float x) { p[i] = x; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, int64_t i,
                                                               float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Four consecutive elements at element offset i (a multiple of 4: 16- or 8-byte aligned).
__device__ __forceinline__ float4 ld4(const float* p, int64_t i) {
    return *reinterpret_cast<const float4*>(p + i);
}
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p, int64_t i) {
    const uint2 u = *reinterpret_cast<const uint2*>(p + i);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
__device__ __forceinline__ void st4(float* p, int64_t i, float4 v) {
    *reinterpret_cast<float4*>(p + i) = v;
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, int64_t i, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p + i) = u;
}

constexpr int D = kHeadDim;
constexpr int C = 64;        // tokens per chunk
constexpr int DV = 32;       // d_v columns per CTA (grid.y = D / DV)
constexpr int LDQ = D + 4;   // padded row pitch of the Q^/K^ tiles
constexpr int LDA = C + 4;   // padded row pitch of the masked score tile
constexpr size_t kSimtSmem =
    sizeof(float) * (size_t(C) * LDQ * 2 + size_t(C) * DV + size_t(C) * LDA + size_t(D) * DV);

// One CTA per (b, h, d_v slice of 32).  256 threads.
template <typename T>
__global__ void __launch_bounds__(256) k_prefill_simt(const T* __restrict__ q,
                                                      const T* __restrict__ k,
                                                      const T* __restrict__ v,
                                                      const float* __restrict__ S_in,
                                                      float* __restrict__ y,
                                                      float* __restrict__ S_out, int H,
                                                      int64_t N, int activated) {
    // step 2 (SiLU) unless the inputs arrive activated
    auto act = [activated](float x) { return activated ? x : silu_f(x); };
    extern __shared__ float smem[];
    float* Qs = smem;              // [C][LDQ]  q^ rows of the chunk
    float* Ks = Qs + C * LDQ;      // [C][LDQ]  k^ rows
    float* Vs = Ks + C * LDQ;      // [C][DV]   v^ slice
    float* As = Vs + C * DV;       // [C][LDA]  masked scores
    float* Ss = As + C * LDA;      // [D][DV]   state slice S[:, j0:j0+DV]
    const int tid = threadIdx.x;
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / H, h = bh % H;
    const int j0 = blockIdx.y * DV;

    for (int idx = tid; idx < D * DV; idx += 256) {
        const int i = idx / DV, j = idx % DV;
        Ss[idx] = S_in ? S_in[(bh * D + i) * D + j0 + j] : 0.0f;
    }

    for (int64_t c0 = 0; c0 < N; c0 += C) {
        const int nc = (int)((N - c0) < C ? (N - c0) : C);
        __syncthreads();
        for (int idx = tid; idx < C * D; idx += 256) {
            const int t = idx / D, i = idx % D;
            float qv = 0.f, kv = 0.f;
            if (t < nc) {
                const int64_t off = ((b * N + c0 + t) * H + h) * D + i;
                qv = act(ldf(q, off));
                kv = act(ldf(k, off));
            }
            Qs[t * LDQ + i] = qv;
            Ks[t * LDQ + i] = kv;
        }
        for (int idx = tid; idx < C * DV; idx += 256) {
            const int t = idx / DV, j = idx % DV;
            float vv = 0.f;
            if (t < nc) vv = act(ldf(v, ((b * N + c0 + t) * H + h) * D + j0 + j));
            Vs[idx] = vv;
        }
        __syncthreads();
        // A = Q^ K^T masked to s <= t: each thread a 4 x 4 block.
        {
            const int ty = tid / 16, tx = tid % 16;
            float acc[4][4] = {};
            for (int i = 0; i < D; i += 4) {
                float4 qa[4], kb[4];
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    qa[a] = *reinterpret_cast<const float4*>(&Qs[(ty * 4 + a) * LDQ + i]);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    kb[c] = *reinterpret_cast<const float4*>(&Ks[(tx * 4 + c) * LDQ + i]);
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc[a][c] += qa[a].x * kb[c].x + qa[a].y * kb[c].y +
                                     qa[a].z * kb[c].z + qa[a].w * kb[c].w;
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int t = ty * 4 + a, s = tx * 4 + c;
                    As[t * LDA + s] = (s <= t) ? acc[a][c] : 0.0f;
                }
        }
        __syncthreads();
        // y[t, j] = q^_t S_prefix[:, j] + sum_{s<=t} A[t, s] v^_s[j]
        {
            const int t = tid / 4, jg = (tid % 4) * 8;
            float acc[8] = {};
            for (int i = 0; i < D; ++i) {
                const float qv = Qs[t * LDQ + i];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) acc[jj] += qv * Ss[i * DV + jg + jj];
            }
            for (int s = 0; s <= t; ++s) {
                const float a = As[t * LDA + s];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) acc[jj] += a * Vs[s * DV + jg + jj];
            }
            if (t < nc) {
                float* yr = y + ((b * N + c0 + t) * H + h) * D + j0 + jg;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) yr[jj] = acc[jj];
            }
        }
        __syncthreads();
        // S[:, slice] += K^T V over the chunk (rows past the tail are zero).
        {
            const int i = tid / 2, jh = (tid % 2) * 16;
            float acc[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) acc[jj] = Ss[i * DV + jh + jj];
            for (int s = 0; s < nc; ++s) {
                const float kv = Ks[s * LDQ + i];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) acc[jj] += kv * Vs[s * DV + jh + jj];
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) Ss[i * DV + jh + jj] = acc[jj];
        }
    }
    __syncthreads();
    if (S_out)
        for (int idx = tid; idx < D * DV; idx += 256) {
            const int i = idx / DV, j = idx % DV;
            S_out[(bh * D + i) * D + j0 + j] = Ss[idx];
        }
}

__device__ __forceinline__ float block_sum_256(float x, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    __syncthreads();
    if (l == 0) red[w] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += red[i];  // fixed order: deterministic
    return s;
}

// One CTA per token row of width H*d: out = y / sqrt(mean(y^2) + eps) * sigmoid(g).
template <typename T>
__global__ void __launch_bounds__(256) k_norm_gate_rows(const float* __restrict__ y,
                                                        const T* __restrict__ g,
                                                        T* __restrict__ out, int width,
                                                        float eps) {
    __shared__ float red[8];
    const int64_t base = (int64_t)blockIdx.x * width;
    float ss = 0.f;
    for (int c = threadIdx.x; c < width; c += 256) {
        const float yv = y[base + c];
        ss += yv * yv;
    }
    ss = block_sum_256(ss, red);
    const float r = rsqrtf(ss / (float)width + eps);
    for (int c = threadIdx.x; c < width; c += 256)
        stf(out, base + c, y[base + c] * r * sigmoid_f(ldf(g, base + c)));
}

// Decode: one CTA per (b,h), 256 threads; thread (rg, jc) streams rows i = rg + 8 r of
// the 128 x 128 fp32 state as float4 columns 4 jc .. 4 jc + 3, updates them in place
// (S += k^T v) and accumulates y = q S.  The CTA then publishes y and its sum of squares
// and bumps the arrival counter of sequence b; the last of the H heads of b to arrive
// applies the norm over all H*d features of b and the gate (no CTA ever waits, so the
// order in which CTAs run does not matter).  The last CTA also resets the counter, so
// the counters are zero between calls.
template <typename T>
__global__ void __launch_bounds__(256, 3) k_decode_step(float* __restrict__ S,
                                                     const T* __restrict__ q,
                                                     const T* __restrict__ k,
                                                     const T* __restrict__ v,
                                                     const T* __restrict__ g,
                                                     T* __restrict__ out, float* __restrict__ y,
                                                     float* __restrict__ ss,
                                                     unsigned* __restrict__ cnt, int H,
                                                     float eps) {
    __shared__ float qs[D], ks[D];
    __shared__ __align__(16) float vs[D];
    __shared__ float4 red[8][32];
    __shared__ float rsh[8];
    __shared__ int last;
    const int tid = threadIdx.x;
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / H;
    if (tid < D) {
        const int64_t off = bh * D + tid;
        qs[tid] = silu_f(ldf(q, off));
        ks[tid] = silu_f(ldf(k, off));
        vs[tid] = silu_f(ldf(v, off));
    }
    __syncthreads();
    const int jc = tid % 32, rg = tid / 32;
    const float4 vv = reinterpret_cast<const float4*>(vs)[jc];
    float4* Sp = reinterpret_cast<float4*>(S + bh * D * D);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 sv[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) sv[r] = Sp[(rg + 8 * r) * 32 + jc];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int i = rg + 8 * r;
        const float kk = ks[i], qq = qs[i];
        float4 s = sv[r];
        s.x += kk * vv.x; s.y += kk * vv.y; s.z += kk * vv.z; s.w += kk * vv.w;
        Sp[i * 32 + jc] = s;
        acc.x += qq * s.x; acc.y += qq * s.y; acc.z += qq * s.z; acc.w += qq * s.w;
    }
    red[rg][jc] = acc;
    __syncthreads();
    if (tid < 32) {
        float4 t = red[0][tid];
#pragma unroll
        for (int r = 1; r < 8; ++r) {
            const float4 u = red[r][tid];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        reinterpret_cast<float4*>(y + bh * D)[tid] = t;
        float p = t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
        if (tid == 0) ss[bh] = p;
        __threadfence();  // y and ss are visible device-wide before the arrival below
    }
    __syncthreads();
    if (tid == 0) last = atomicAdd(cnt + b, 1u) == static_cast<unsigned>(H - 1);
    __syncthreads();
    if (!last) return;
    // ---- the last head of sequence b: norm over the H*d features, then the gate
    __threadfence();
    float part = 0.f;
    for (int i = tid; i < H; i += 256) part += __ldcg(ss + b * H + i);
    // fixed-order reduction (deterministic): warp tree, then the 8 warps in order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((tid & 31) == 0) rsh[tid >> 5] = part;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += rsh[w];
    const float r = rsqrtf(tot / static_cast<float>(H * D) + eps);
    const int64_t base = b * H * D;
    // 4 consecutive features per thread and step; 4 steps' loads are issued together
    const int n4 = H * (D / 4);
    for (int k0 = tid; k0 < n4; k0 += 256 * 4) {
        float4 yv[4];
        float4 gv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = k0 + 256 * j;
            if (k < n4) {
                yv[j] = __ldcg(reinterpret_cast<const float4*>(y + base) + k);
                gv[j] = ld4(g, base + 4 * static_cast<int64_t>(k));
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = k0 + 256 * j;
            if (k < n4)
                st4(out, base + 4 * static_cast<int64_t>(k),
                    make_float4(yv[j].x * r * sigmoid_f(gv[j].x), yv[j].y * r * sigmoid_f(gv[j].y),
                                yv[j].z * r * sigmoid_f(gv[j].z), yv[j].w * r * sigmoid_f(gv[j].w)));
        }
    }
    if (tid == 0) cnt[b] = 0u;
}

__global__ void k_zero(float* p, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = 0.f;
}

}  // namespace

int launch_prefill_simt(const void* q, const void* k, const void* v, const float* S_in,
                        float* y, float* S_out, int B, int H, int64_t N, bool bf16,
                        bool activated, cudaStream_t st) {
    dim3 grid((unsigned)((int64_t)B * H), D / DV);
    if (bf16) {
        auto kern = k_prefill_simt<__nv_bfloat16>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSimtSmem) != cudaSuccess)
            return LA_ERR_CUDA;
        kern<<<grid, 256, kSimtSmem, st>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                           (const __nv_bfloat16*)v, S_in, y, S_out, H, N,
                                           activated ? 1 : 0);
    } else {
        auto kern = k_prefill_simt<float>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSimtSmem) != cudaSuccess)
            return LA_ERR_CUDA;
        kern<<<grid, 256, kSimtSmem, st>>>((const float*)q, (const float*)k, (const float*)v,
                                           S_in, y, S_out, H, N, activated ? 1 : 0);
    }
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int launch_norm_gate_rows(const float* y, const void* g, void* out, int64_t rows, int width,
                          float eps, bool bf16, cudaStream_t st) {
    if (rows <= 0) return LA_OK;
    // grid.x holds up to 2^31-1 rows; 1M tokens x B stays far below that
    if (bf16)
        k_norm_gate_rows<__nv_bfloat16><<<(unsigned)rows, 256, 0, st>>>(
            y, (const __nv_bfloat16*)g, (__nv_bfloat16*)out, width, eps);
    else
        k_norm_gate_rows<float><<<(unsigned)rows, 256, 0, st>>>(y, (const float*)g,
                                                                (float*)out, width, eps);
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int launch_decode(float* S, const void* q, const void* k, const void* v, const void* g,
                  void* out, float* y, float* ss, unsigned* cnt, int B, int H, float eps,
                  bool bf16, cudaStream_t st) {
    const unsigned nbh = (unsigned)((int64_t)B * H);
    if (bf16)
        k_decode_step<__nv_bfloat16><<<nbh, 256, 0, st>>>(
            S, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
            (const __nv_bfloat16*)g, (__nv_bfloat16*)out, y, ss, cnt, H, eps);
    else
        k_decode_step<float><<<nbh, 256, 0, st>>>(S, (const float*)q, (const float*)k,
                                                  (const float*)v, (const float*)g,
                                                  (float*)out, y, ss, cnt, H, eps);
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int launch_zero_state(float* S, int64_t n, cudaStream_t st) {
    if (n <= 0) return LA_OK;
    k_zero<<<592, 256, 0, st>>>(S, n);
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace la
