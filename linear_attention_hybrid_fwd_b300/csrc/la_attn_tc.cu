// la_attn_tc.cu -- the softmax layer of the hybrid stack on tensor cores (sm_103a):
// partial RoPE, then causal softmax attention.
//
// What it computes.  MiniMax-Text-01 places one softmax attention layer after every
// seven Lightning Attention layers ("Hybrid Modeling", MiniMax-01 deep dive); it
// applies RoPE to half of the head dimension, with base frequency 10,000,000 (the
// model card's "Model Architecture" list; 64 heads of size 128).  Here:
//     q', k' = RoPE(q), RoPE(k):  features [0, 64) of a head rotated as pairs
//              (i, i + 32), angle t * base^(-i/32) at token t; [64, 128) unchanged
//     o_t    = sum_{s <= t} softmax_s(q'_t . k'_s / sqrt(d)) v_s
// with q, k, v, o laid out [B][N][H][d] bf16 like the linear layer's tensors.
//
// Design:
//  * k_rope_table writes cos/sin of every (token, pair) angle in fp32, each computed
//    in fp64 (angles reach 1e6 rad at 1M tokens); the table is cached per device.
//    k_rope rotates q and k into library-owned copies (one RNE rounding to bf16),
//    eight threads per row with 16-byte accesses.
//  * k_attn_fwd: one CTA per (pair of 128-query tiles, head, sequence), head-major,
//    the pairs with the most key tiles first.  Warp 0 lane 0 loads both query tiles
//    once and the key/value tiles of the causal range into two stages by TMA (128B
//    swizzle); the two query tiles share every key/value tile.  Warp 1 lane 0 issues
//    tcgen05 MMAs: S_t = Q_t K_j^T (128 x 128, fp32) into query tile t's TMEM score
//    buffer, and O_t += P_t V_j (P in TMEM, bf16) as one N = 128 chain, followed at
//    once by S_t of the next key tile.  Warps 4-7 (tile 0) and 8-11 (tile 1) own one
//    query row per thread: they read S_t from TMEM, mask it (causal, keys past N),
//    keep the running max m and sum l of the online softmax in base 2, write P_t as
//    bf16 over the first 64 columns of the score buffer, and rescale O_t in TMEM when
//    a row's max moved.  While one tile's softmax runs, the tensor pipe works on the
//    other tile.  At the end they divide O_t by l and store bf16 rows.
//  * Every wait is bounded (%globaltimer); a CTA that gives up records LA_ERR_TIMEOUT
//    in the status word, lets its copies and MMAs finish, frees TMEM and exits.
//
// TMEM columns: [0, 128) S / P of query tile 0 | [128, 256) of tile 1 |
//               [256, 384) O of tile 0 | [384, 512) O of tile 1.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/lightning_attn.h"
#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace {

using namespace sm100;

constexpr int D = kHeadDim;            // 128
constexpr int BQ = 128;                // queries per tile (TMEM lanes)
constexpr int BKV = 128;               // keys per tile
constexpr int kPairs = D / 4;          // rotated pairs: features [0, 64) of a head
constexpr int kThreads = 384;          // 12 warps
constexpr uint32_t HALF = 16384;       // 128 rows x 64 bf16, one 128B-swizzled block
constexpr uint32_t TILE = 2 * HALF;    // 128 rows x 128 bf16
constexpr uint32_t OFF_Q = 0;                   // 2 query tiles
constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;    // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE;    // 2 stages
constexpr uint32_t SMEM_USED = OFF_V + 2 * TILE;      // 192 KiB
constexpr uint32_t SMEM_DYN = SMEM_USED + 1024;       // + alignment slack
static_assert(SMEM_DYN + 1024 <= 227 * 1024, "shared memory budget");
constexpr uint32_t TM_S = 0, TM_O = 256;
constexpr uint32_t IDESC_S = idesc_bf16_f32(BQ, BKV, 0, 0);   // Q K-major, K K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BQ, D, 0, 1);    // P (TMEM), V MN-major, N = 128
constexpr float kMaxSlack = 8.0f;      // base-2 growth of a row's max before O rescales
constexpr uint64_t kTimeoutNs = 4000000000ull;  // 4 s
constexpr uint64_t kDrainNs = 200000000ull;     // 0.2 s

struct AttnParams {
    __nv_bfloat16* out;
    int* status;
    int B, H, N;
    int Qt;            // query tiles per sequence
    int Qp;            // pairs of query tiles per sequence (a CTA each)
    float scale_log2;  // log2(e) / sqrt(d)
};

struct Shared {
    // sfull, pfull, pvdone: one per query tile of the pair
    uint64_t qfull, kfull[2], kempty[2], vfull[2], vempty[2], sfull[2], pfull[2], pvdone[2],
        mmadone;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ bool abort_set(Shared& sh) {
    return *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0;
}
// Bounded wait for the phase of `bar` with `parity`; false when the CTA is aborting
// (honor_abort) or after `limit_ns`, in which case it raises the abort itself.
__device__ bool wait_bar(Shared& sh, int* status, uint64_t* bar, uint32_t parity,
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

// Smem descriptors (128B swizzle).  K-major operand of 128 x 128 bf16 stored as two
// 64-wide halves; k-step ks (16 elements = 32 bytes).  MN-major operand (rows = K,
// one 64-wide MN block): k-step ks covers 16 rows (2048 bytes).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int ks) {
    return smem_desc_sw128(base + (ks >> 2) * HALF + (ks & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int ks) {
    return smem_desc_sw128(base + ks * 2048, HALF, 1024);
}

// ------------------------------------------------------------------ RoPE
// cs[t][i] = (cos, sin) of t * base^(-i / kPairs), the angle and both functions in fp64.
__global__ void k_rope_table(float2* __restrict__ cs, int N, double base) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(N) * kPairs) return;
    const int t = static_cast<int>(idx / kPairs), i = static_cast<int>(idx % kPairs);
    const double ang = static_cast<double>(t) * pow(base, -static_cast<double>(i) / kPairs);
    double s, c;
    sincos(ang, &s, &c);
    cs[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
}

// Eight threads per (token, head) row of q (blockIdx.y = 0) or k (1); rows are
// [B][N][H].  Thread c < 4 rotates the pairs (8c + e, 8c + e + 32), e < 8, by the row's
// token angles; thread c >= 4 copies features [64 + 16(c - 4), + 16).  16-byte accesses.
__global__ void k_rope(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       __nv_bfloat16* __restrict__ qr, __nv_bfloat16* __restrict__ kr,
                       const float2* __restrict__ cs, int64_t rows, int H, int N) {
    const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
    if (row >= rows) return;
    const int c = threadIdx.x & 7;
    const uint4* src = reinterpret_cast<const uint4*>((blockIdx.y == 0 ? q : k) + row * D);
    uint4* dst = reinterpret_cast<uint4*>((blockIdx.y == 0 ? qr : kr) + row * D);
    if (c >= 4) {
        const int o = 8 + 2 * (c - 4);  // 16-byte chunk index of feature 64 + 16(c - 4)
        dst[o] = src[o];
        dst[o + 1] = src[o + 1];
        return;
    }
    const int64_t t = (row / H) % N;  // token position within its sequence
    const uint4 a4 = src[c], b4 = src[c + 4];
    const uint32_t* a = reinterpret_cast<const uint32_t*>(&a4);
    const uint32_t* b = reinterpret_cast<const uint32_t*>(&b4);
    const float4* cs4 = reinterpret_cast<const float4*>(cs + t * kPairs + 8 * c);
    uint4 ra4, rb4;
    uint32_t* ra = reinterpret_cast<uint32_t*>(&ra4);
    uint32_t* rb = reinterpret_cast<uint32_t*>(&rb4);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float4 r = cs4[e];  // (cos, sin) of pairs 8c + 2e and 8c + 2e + 1
        const float a0 = __uint_as_float(a[e] << 16), a1 = __uint_as_float(a[e] & 0xFFFF0000u);
        const float b0 = __uint_as_float(b[e] << 16), b1 = __uint_as_float(b[e] & 0xFFFF0000u);
        ra[e] = pack_bf16x2(a0 * r.x - b0 * r.y, a1 * r.z - b1 * r.w);
        rb[e] = pack_bf16x2(a0 * r.y + b0 * r.x, a1 * r.w + b1 * r.z);
    }
    dst[c] = ra4;
    dst[c + 4] = rb4;
}

// ------------------------------------------------------------------ attention
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Shared sh;
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // head-major order, the tile pairs of a head with the most key tiles first: CTAs
    // running together share their heads' key/value tiles in L2
    const int bh = static_cast<int>(blockIdx.x / p.Qp);
    const int q0 = 2 * (p.Qp - 1 - static_cast<int>(blockIdx.x % p.Qp));  // first query tile
    const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
    const int ntile = q0 + 1 < p.Qt ? 2 : 1;
    const int nkv = q0 + ntile;  // causal: key tiles 0 .. q0 + ntile - 1

    if (tid == 0) {
        mbar_init(&sh.qfull, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.kfull[s], 1);
            mbar_init(&sh.kempty[s], 1);
            mbar_init(&sh.vfull[s], 1);
            mbar_init(&sh.vempty[s], 1);
            mbar_init(&sh.sfull[s], 1);
            mbar_init(&sh.pfull[s], 4);  // one arrival per softmax warp of the tile
            mbar_init(&sh.pvdone[s], 1);
        }
        mbar_init(&sh.mmadone, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) tmem_alloc(&sh.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const int col = h * D;
            mbar_arrive_expect_tx(&sh.qfull, ntile * TILE);
            for (int t = 0; t < ntile; ++t) {
                tma_load_3d(sm + OFF_Q + t * TILE, &tq, col, (q0 + t) * BQ, b, &sh.qfull);
                tma_load_3d(sm + OFF_Q + t * TILE + HALF, &tq, col + 64, (q0 + t) * BQ, b,
                            &sh.qfull);
            }
            int issued = 0;
            for (int j = 0; j < nkv; ++j) {
                const int s = j & 1;
                const uint32_t ph = static_cast<uint32_t>(j >> 1) & 1u;
                if (!wait_bar(sh, p.status, &sh.kempty[s], ph ^ 1u)) break;
                mbar_arrive_expect_tx(&sh.kfull[s], TILE);
                tma_load_3d(sm + OFF_K + s * TILE, &tk, col, j * BKV, b, &sh.kfull[s]);
                tma_load_3d(sm + OFF_K + s * TILE + HALF, &tk, col + 64, j * BKV, b, &sh.kfull[s]);
                if (!wait_bar(sh, p.status, &sh.vempty[s], ph ^ 1u)) {
                    issued = -(j + 1);  // K_j issued, V_j not
                    break;
                }
                mbar_arrive_expect_tx(&sh.vfull[s], TILE);
                tma_load_3d(sm + OFF_V + s * TILE, &tv, col, j * BKV, b, &sh.vfull[s]);
                tma_load_3d(sm + OFF_V + s * TILE + HALF, &tv, col + 64, j * BKV, b, &sh.vfull[s]);
                issued = j + 1;
            }
            // drain: every load issued lands before this CTA may exit
            wait_bar(sh, p.status, &sh.qfull, 0, false, kDrainNs);
            const int nk = issued < 0 ? -issued : issued;   // K tiles issued
            const int nv = issued < 0 ? -issued - 1 : issued;
            for (int j = nk - 2 < 0 ? 0 : nk - 2; j < nk; ++j)
                wait_bar(sh, p.status, &sh.kfull[j & 1], static_cast<uint32_t>(j >> 1) & 1u,
                         false, kDrainNs);
            for (int j = nv - 2 < 0 ? 0 : nv - 2; j < nv; ++j)
                wait_bar(sh, p.status, &sh.vfull[j & 1], static_cast<uint32_t>(j >> 1) & 1u,
                         false, kDrainNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            // Query tile t, key tile j: S_t = Q_t K_j^T into t's score buffer; once t's
            // softmax has written P_t there, O_t += P_t V_j, and right after that product
            // S_t for key tile j + 1.  While one tile's softmax runs, the tensor pipe
            // works on the other tile.
            bool ok = wait_bar(sh, p.status, &sh.qfull, 0);
            auto issue_s = [&](int t, int j) {
                const uint32_t qa = sbase + OFF_Q + t * TILE;
                const uint32_t ka = sbase + OFF_K + (j & 1) * TILE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tm + TM_S + t * BKV, desc_kmajor(qa, ks), desc_kmajor(ka, ks), IDESC_S,
                           ks > 0 ? 1u : 0u);
                mma_commit(&sh.sfull[t]);
            };
            if (ok) ok = wait_bar(sh, p.status, &sh.kfull[0], 0);
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < ntile; ++t) issue_s(t, 0);
                mma_commit(&sh.kempty[0]);
            }
            for (int j = 0; j < nkv && ok; ++j) {
                const int s = j & 1;
                if (!wait_bar(sh, p.status, &sh.vfull[s], static_cast<uint32_t>(j >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                const uint32_t va = sbase + OFF_V + s * TILE;
                const bool next = j + 1 < nkv;
                if (next && !wait_bar(sh, p.status, &sh.kfull[(j + 1) & 1],
                                      static_cast<uint32_t>((j + 1) >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                for (int t = 0; t < ntile && ok; ++t) {
                    if (j > q0 + t) continue;  // past tile t's causal range
                    if (!wait_bar(sh, p.status, &sh.pfull[t], static_cast<uint32_t>(j) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < BKV / 16; ++ks)
                        mma_ts(tm + TM_O + t * BKV, tm + TM_S + t * BKV + ks * 8,
                               desc_mnmajor(va, ks), IDESC_PV, (j > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&sh.pvdone[t]);
                    if (j + 1 <= q0 + t) {
                        // the score buffer holds P_t until this product is done
                        if (!wait_bar(sh, p.status, &sh.pvdone[t], static_cast<uint32_t>(j) & 1u)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_s(t, j + 1);
                    }
                }
                if (!ok) break;
                mma_commit(&sh.vempty[s]);
                if (next) mma_commit(&sh.kempty[(j + 1) & 1]);
            }
            mma_commit(&sh.mmadone);
            wait_bar(sh, p.status, &sh.mmadone, 0, false, kDrainNs);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax rows
        const int t = (warp - 4) >> 2;              // query tile of this warpgroup
        const int quarter = warp & 3;               // TMEM lanes 32 quarter .. + 31
        if (t < ntile) {
            const int qi = q0 + t;
            const int nkv_t = qi + 1;
            const int r = quarter * 32 + lane;      // query row of the tile
            const int qrow = qi * BQ + r;           // token position
            const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
            const uint32_t sa = tm + TM_S + t * BKV + lane_off;
            const uint32_t oa = tm + TM_O + t * BKV + lane_off;
            float m = -INFINITY, l = 0.0f;
            bool ok = true;
            for (int j = 0; j < nkv_t; ++j) {
                if (!__all_sync(0xffffffffu, wait_bar(sh, p.status, &sh.sfull[t],
                                                      static_cast<uint32_t>(j) & 1u))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t xu[BKV];
#pragma unroll
                for (int c = 0; c < BKV / 32; ++c) LA_TMEM_LD32(sa + c * 32, (xu + c * 32));
                tmem_wait_ld();
                // keys after the query or past N are masked; a tile below the diagonal
                // and inside N (the same for every row of the tile) needs no mask
                const int k0 = j * BKV;
                if (!(j < qi && k0 + BKV <= p.N)) {
                    const int kmax = min(qrow, p.N - 1) - k0;  // last allowed key here
#pragma unroll
                    for (int c = 0; c < BKV; ++c)
                        if (c > kmax) xu[c] = __float_as_uint(-INFINITY);
                }
                // the row max on raw scores (the scale is positive), four chains
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < BKV; ++c)
                    mx4[c & 3] = fmaxf(mx4[c & 3], __uint_as_float(xu[c]));
                const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                // The reference max moves only when the row's max grows by more than
                // kMaxSlack (base 2): probabilities stay below 2^kMaxSlack, and O and l
                // need no rescale (and the softmax no wait on O) in most key tiles.
                const float m_row = mx * p.scale_log2;                  // base-2 units
                const bool move = m_row > m + kMaxSlack;
                float alpha = 1.0f;
                if (move) {
                    alpha = ex2_approx(m - m_row);  // 0 for the first key tile (m = -inf)
                    m = m_row;
                }
                const bool rescale = __any_sync(0xffffffffu, move) && j > 0;
                const float m_use = m == -INFINITY ? 0.0f : m;          // no key yet
                float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int c = 0; c < BKV / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = ex2_approx(
                            fmaf(__uint_as_float(xu[c * 32 + 2 * e]), p.scale_log2, -m_use));
                        const float p1 = ex2_approx(
                            fmaf(__uint_as_float(xu[c * 32 + 2 * e + 1]), p.scale_log2, -m_use));
                        sum4[e & 3] += p0 + p1;
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    LA_TMEM_ST16(sa + c * 16, pk);  // P over the first 64 columns
                }
                l = l * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
                tmem_wait_st();
                if (rescale) {
                    // O holds the products up to key tile j - 1 once the last is done;
                    // rescale the rows whose reference max moved (alpha = 1 elsewhere)
                    if (!__all_sync(0xffffffffu,
                                    wait_bar(sh, p.status, &sh.pvdone[t],
                                             static_cast<uint32_t>(j - 1) & 1u))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t u[32];
                        LA_TMEM_LD32(oa + c * 32, u);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
                        LA_TMEM_ST32(oa + c * 32, u);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.pfull[t]);
            }
            // -------------------------------------------------------- epilogue
            if (ok && __all_sync(0xffffffffu,
                                 wait_bar(sh, p.status, &sh.pvdone[t],
                                          static_cast<uint32_t>(nkv_t - 1) & 1u))) {
                tc_fence_after();
                const float inv = 1.0f / l;
                __nv_bfloat16* dst =
                    p.out + ((static_cast<int64_t>(b) * p.N + qrow) * p.H + h) * D;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t u[32];
                    LA_TMEM_LD32(oa + c * 32, u);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(u[2 * e]) * inv,
                                            __uint_as_float(u[2 * e + 1]) * inv);
                    if (qrow < p.N) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2],
                                               pk[4 * e + 3]);
                    }
                }
            }
        }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::mutex g_attr_mutex;
bool g_attr_set[64];  // per device: the kernel's shared-memory attribute is set

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode;
}

// [B][N][H*d] bf16 as a 3-D tensor (feature, token, sequence), boxes of 64 features x
// 128 tokens, 128B swizzle; reads past N give zeros.
bool encode_io_map(CUtensorMap* m, const void* base, int B, int H, int64_t N) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * D * 2,
                             static_cast<cuuint64_t>(N) * H * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prepare_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (!g_attr_set[dev]) {
        if (cudaFuncSetAttribute(k_attn_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SMEM_DYN)) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        g_attr_set[dev] = true;
    }
    return true;
}

// The cos/sin table of the current device for at least N tokens and this base, built
// on `st` when it grows or the base changes (the host then waits for it once, so calls
// on other streams find it complete).
struct RopeTable {
    float2* cs = nullptr;
    int64_t n = 0;
    double base = 0.0;
};
RopeTable g_tables[64];
std::mutex g_table_mutex;

struct TableReaper {
    ~TableReaper() {
        // Process teardown: the driver may already be gone; ignore errors.
        for (auto& t : g_tables)
            if (t.cs) cudaFree(t.cs);
    }
} g_table_reaper;

int rope_table(int64_t N, double base, cudaStream_t st, const float2** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_table_mutex);
    RopeTable& tb = g_tables[dev];
    if (tb.cs && tb.n >= N && tb.base == base) {
        *out = tb.cs;
        return LA_OK;
    }
    const int64_t n = N > tb.n ? N : tb.n;
    if (n > tb.n) {
        if (tb.cs) cudaFree(tb.cs);  // waits for work already queued on the device
        tb.cs = nullptr;
        tb.n = 0;
        if (cudaMalloc(&tb.cs, static_cast<size_t>(n) * kPairs * sizeof(float2)) != cudaSuccess) {
            cudaGetLastError();
            tb.cs = nullptr;
            return LA_ERR_NOMEM;
        }
    }
    const int64_t nt = n * kPairs;
    k_rope_table<<<static_cast<unsigned>((nt + 255) / 256), 256, 0, st>>>(tb.cs, static_cast<int>(n),
                                                                         base);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) {
        tb.n = 0;
        return LA_ERR_CUDA;
    }
    note_launches(1);
    tb.n = n;
    tb.base = base;
    *out = tb.cs;
    return LA_OK;
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

extern "C" int la_softmax_attention(const void* q, const void* k, const void* v, void* out,
                                    int B, int H, int64_t N, int d, double rope_base,
                                    void* cuda_stream) {
    if (B <= 0 || H <= 0 || N < 0 || d <= 0) return LA_ERR_INVALID_ARG;
    if (!(rope_base > 1.0) || !isfinite(rope_base)) return LA_ERR_INVALID_ARG;
    if (d != D) return LA_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, out};
    for (const void* x : ptrs)
        if (!aligned16(x)) return LA_ERR_MISALIGNED;
    if (N > (int64_t(1) << 30)) return LA_ERR_UNSUPPORTED;
    const int64_t Qt = (N + BQ - 1) / BQ;
    if (Qt * B * H > (int64_t(1) << 31) - 1 || static_cast<int64_t>(B) * H > (1 << 24))
        return LA_ERR_UNSUPPORTED;
    const size_t bytes = static_cast<size_t>(B) * N * H * D * 2;
    if (overlaps(out, bytes, q, bytes) || overlaps(out, bytes, k, bytes) ||
        overlaps(out, bytes, v, bytes))
        return LA_ERR_INVALID_ARG;
    if (N == 0) return LA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (!prepare_device()) return LA_ERR_CUDA;
    // workspace: rotated q and k (bf16); the cos/sin table is cached per device
    Workspace ws;
    int rc = workspace_acquire(2 * bytes, st, &ws);
    if (rc != LA_OK) return rc;
    auto* qr = static_cast<__nv_bfloat16*>(ws.base);
    auto* kr = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws.base) + bytes);
    const float2* cs = nullptr;
    rc = rope_table(N, rope_base, st, &cs);
    if (rc != LA_OK) return rc;
    const int64_t rows = static_cast<int64_t>(B) * N * H;
    k_rope<<<dim3(static_cast<unsigned>((rows * 8 + 255) / 256), 2), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), qr, kr, cs,
        rows, H, static_cast<int>(N));
    CUtensorMap mq, mk, mv;
    if (!encode_io_map(&mq, qr, B, H, N) || !encode_io_map(&mk, kr, B, H, N) ||
        !encode_io_map(&mv, v, B, H, N))
        return LA_ERR_UNSUPPORTED;
    AttnParams prm;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.status = ws.status;
    prm.B = B;
    prm.H = H;
    prm.N = static_cast<int>(N);
    prm.Qt = static_cast<int>(Qt);
    prm.Qp = static_cast<int>((Qt + 1) / 2);
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(D)));
    k_attn_fwd<<<static_cast<unsigned>(static_cast<int64_t>(prm.Qp) * B * H), kThreads, SMEM_DYN,
                 st>>>(mq, mk, mv, prm);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    note_launches(2);
    return LA_OK;
}
