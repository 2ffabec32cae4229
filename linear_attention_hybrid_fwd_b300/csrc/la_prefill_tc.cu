// la_prefill_tc.cu -- tensor-core prefill of the Lightning Attention layer (sm_103a).
//
// What it computes ("Hybrid Modeling", MiniMax-01 deep dive, Hugging Face blog,
// mechanism steps 2-4): q^,k^,v^ = SiLU(q,k,v); y_t = q^_t sum_{s<=t} k^_s^T v^_s;
// out = y / sqrt(mean over the H*d features of y^2 + eps) * sigmoid(g).  The causal
// product takes the blockwise O(d^2 n) route of the same section: per chunk c of 128
// tokens
//     Y_c = Q^_c S_{<c} + (Q^_c K^_c^T * M) V^_c ,    S_{<c+1} = S_{<c} + K^_c^T V^_c
// with M the inclusive lower-triangular mask.
//
// Design (one B300 SM per CTA, 224 KiB shared memory, all 512 TMEM columns):
//  * A cluster of two CTAs owns one (sequence b, head h).  CTA r takes the chunks
//    c = r, r+2, r+4, ... and keeps the partial state S_r = sum of K^T V over ITS
//    chunks in TMEM (fp32).  S_{<c} = S_0 + S_1 is applied as two MMAs, Q^ S_own and
//    Q^ S_peer; after each chunk a CTA converts its S_own to bf16 and bulk-copies it
//    into the peer's shared memory.  Only a d x d state crosses the pair, and the
//    pair has no redundant loads or activations.
//  * Warp roles: warp 0 issues TMA loads (q, k, v tiles, 128B-swizzled), warp 1 issues
//    tcgen05 MMAs, warp 2 owns TMEM, warps 4-7 apply SiLU (q into TMEM as the A
//    operand; k, v in place in shared memory), mask the score tile and convert the
//    state, warps 8-15 run the epilogue.
//  * The RMSNorm spans all heads of a token, so the epilogue exchanges per-token
//    partial sums of squares through global memory: every head's CTA for chunk c
//    writes its 128 partials, bumps a counter and waits (bounded) until all H have
//    arrived, then sums the H partials in a fixed order (deterministic).  All CTAs of
//    the grid must be co-resident; the host checks that before launching.
//  * Every wait is bounded (%globaltimer); a CTA that gives up records LA_ERR_TIMEOUT
//    in the status word, drains its in-flight copies and MMAs, frees TMEM and exits.
//
// TMEM columns: [0,128) S_own fp32 | [128,256) scores A fp32 | [256,384) Y fp32 |
//               [384,448) Q^ bf16x2 (A operand) | [448,512) P = mask(A) bf16x2.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/lightning_attn.h"
#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace {

using namespace sm100;

constexpr int D = kHeadDim;
constexpr int CH = 128;               // tokens per chunk
constexpr int kThreads = 512;
constexpr uint32_t TILE = 32768;      // 128 x 128 bf16 = two swizzled 128 x 64 halves
constexpr uint32_t HALF = 16384;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE;        // two stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE;    // two stages
constexpr uint32_t OFF_SOWN = OFF_V + 2 * TILE;
constexpr uint32_t OFF_SPEER = OFF_SOWN + TILE;
constexpr uint32_t SMEM_USED = OFF_SPEER + TILE;  // 224 KiB
constexpr uint32_t SMEM_DYN = SMEM_USED + 1024;   // + alignment slack
constexpr uint32_t TM_S = 0, TM_A = 128, TM_Y = 256, TM_Q = 384, TM_P = 448;
constexpr uint64_t kTimeoutNs = 4000000000ull;    // 4 s
constexpr uint64_t kDrainNs = 200000000ull;       // 0.2 s

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, 0, 0);  // A K-major, B K-major
constexpr uint32_t IDESC_XB = idesc_bf16_f32(128, 128, 0, 1);  // A K-major, B MN-major
constexpr uint32_t IDESC_KV = idesc_bf16_f32(128, 128, 1, 1);  // A MN-major, B MN-major

struct Params {
    const __nv_bfloat16* g;
    __nv_bfloat16* out;
    const float* S_in;
    float* S_out;
    float* y_dbg;
    float* xch;      // [B][Nc][128][H] per-token, per-head partial sums of squares
    unsigned* cnt;   // [B][Nc] arrival counters (zeroed before launch)
    int* status;
    int B, H;
    int64_t N;
    int Nc;
    float eps;
    float inv_width;  // 1 / (H * d)
};

struct Shared {
    uint64_t qfull, qempty, kvfull[2], kvready[2], kvempty[2], qhfull, qhempty, afull, pfull,
        sdone, sownfull, speerfull, peercons, yfull, yempty, mmadone;
    uint32_t tmem_base;
    int abort_flag;
    int verdict[2];   // group-uniform wait results (WG1, WG2)
    float red[2][CH];
    float rnorm[CH];
};

// ------------------------------------------------------------------ numerics
// sigmoid(x) = 1 / (1 + e^-x) and SiLU(x) = x sigmoid(x), with the fast CUDA
// intrinsics (relative error ~1e-6 over the input range; the bf16 rounding of the
// result, 2^-9, dominates).
__device__ __forceinline__ float sigmoid_fast(float x) {
    return __fdividef(1.0f, 1.0f + __expf(-x));
}
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t silu_bf16x2(uint32_t u) {
    return pack_bf16x2(silu_fast(bf_lo(u)), silu_fast(bf_hi(u)));
}
__device__ __forceinline__ uint4 silu_chunk(uint4 v) {
    return make_uint4(silu_bf16x2(v.x), silu_bf16x2(v.y), silu_bf16x2(v.z), silu_bf16x2(v.w));
}

// Byte offset of the 16-byte chunk `c` (0..7) of row `r` in a 128B-swizzled half tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ bounded waits
__device__ __forceinline__ bool abort_set(Shared& sh) {
    return *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0;
}
__device__ __forceinline__ void raise_abort(Shared& sh, int* status) {
    *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
    atomicExch(status, LA_ERR_TIMEOUT);
}
// Waits for the phase of `bar` with `parity` to complete.  Gives up (false) when the
// CTA is aborting (honor_abort) or after `limit_ns`, raising the abort itself.
__device__ bool wait_bar(Shared& sh, int* status, uint64_t* bar, uint32_t parity,
                         bool honor_abort = true, uint64_t limit_ns = kTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (honor_abort && abort_set(sh)) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                raise_abort(sh, status);
                return false;
            }
        }
    }
}
// Group-uniform wait: thread `leader` waits (bounded), the group of `n` threads syncs on
// named barrier `id`, then every thread observes the completed phase itself.
__device__ bool group_wait(Shared& sh, int* status, uint64_t* bar, uint32_t parity, bool leader,
                           uint32_t id, uint32_t n, int slot) {
    if (leader) sh.verdict[slot] = wait_bar(sh, status, bar, parity) ? 1 : 0;
    named_bar_sync(id, n);
    const bool ok = *reinterpret_cast<volatile int*>(&sh.verdict[slot]) != 0;
    if (ok)
        while (!mbar_try_wait(bar, parity)) {
        }
    named_bar_sync(id, n);  // verdict slot may be rewritten only after everyone read it
    return ok;
}

// Write 32 fp32 values (columns 32*part .. +31 of row r) as bf16 into an MN-major
// 128B-swizzled 128 x 128 tile (two 128-column halves of 64).
__device__ __forceinline__ void store_row_bf16(uint8_t* tile, int r, int part,
                                               const uint32_t (&v)[32]) {
    uint8_t* half = tile + (part >> 1) * HALF;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(v[8 * cc + 0]), __uint_as_float(v[8 * cc + 1]));
        w.y = pack_bf16x2(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3]));
        w.z = pack_bf16x2(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5]));
        w.w = pack_bf16x2(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7]));
        *reinterpret_cast<uint4*>(half + swz(r, (part & 1) * 4 + cc)) = w;
    }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 1)
    k_prefill_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Shared sh;
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int item = blockIdx.x >> 1;  // b * H + h
    const int b = item / p.H, h = item % p.H;
    const int Nc = p.Nc;
    const int n_own = (Nc - static_cast<int>(rank) + 1) / 2;
    const int n_peer = (Nc - static_cast<int>(peer) + 1) / 2;

    if (tid == 0) {
        mbar_init(&sh.qfull, 1);
        mbar_init(&sh.qempty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.kvfull[s], 1);
            mbar_init(&sh.kvready[s], 1);
            mbar_init(&sh.kvempty[s], 1);
        }
        mbar_init(&sh.qhfull, 1);
        mbar_init(&sh.qhempty, 1);
        mbar_init(&sh.afull, 1);
        mbar_init(&sh.pfull, 1);
        mbar_init(&sh.sdone, 1);
        mbar_init(&sh.sownfull, 1);
        mbar_init(&sh.speerfull, 1);
        mbar_init(&sh.peercons, 1);
        mbar_init(&sh.yfull, 1);
        mbar_init(&sh.yempty, 1);
        mbar_init(&sh.mmadone, 1);
        sh.abort_flag = 0;
        sh.verdict[0] = sh.verdict[1] = 0;
        fence_mbar_init();
        // the first bf16 state from the peer lands here; armed before the peer can send
        if (n_own > 0) mbar_arrive_expect_tx(&sh.speerfull, TILE);
    }
    if (warp == 2) tmem_alloc(&sh.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tm = sh.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < n_own; ++i) {
                const int c = 2 * i + static_cast<int>(rank);
                const int row0 = c * CH;
                const int s = i & 1;
                const uint32_t u = static_cast<uint32_t>(i >> 1);
                if (!wait_bar(sh, p.status, &sh.kvempty[s], (u & 1u) ^ 1u)) break;
                mbar_arrive_expect_tx(&sh.kvfull[s], 2 * TILE);
                uint8_t* kt = sm + OFF_K + s * TILE;
                uint8_t* vt = sm + OFF_V + s * TILE;
                tma_load_3d(kt, &tk, h * D, row0, b, &sh.kvfull[s]);
                tma_load_3d(kt + HALF, &tk, h * D + 64, row0, b, &sh.kvfull[s]);
                tma_load_3d(vt, &tv, h * D, row0, b, &sh.kvfull[s]);
                tma_load_3d(vt + HALF, &tv, h * D + 64, row0, b, &sh.kvfull[s]);
                issued = i + 1;
                if (!wait_bar(sh, p.status, &sh.qempty, static_cast<uint32_t>(i & 1) ^ 1u)) {
                    issued = -issued;  // the q tile of this index was not issued
                    break;
                }
                mbar_arrive_expect_tx(&sh.qfull, TILE);
                tma_load_3d(sm + OFF_Q, &tq, h * D, row0, b, &sh.qfull);
                tma_load_3d(sm + OFF_Q + HALF, &tq, h * D + 64, row0, b, &sh.qfull);
            }
            // drain: every issued copy lands before this CTA may exit
            const bool q_last_missing = issued < 0;
            const int n_kv = issued < 0 ? -issued : issued;
            for (int i = n_kv - 2 < 0 ? 0 : n_kv - 2; i < n_kv; ++i)
                wait_bar(sh, p.status, &sh.kvfull[i & 1], static_cast<uint32_t>(i >> 1) & 1u,
                         false, kDrainNs);
            const int n_q = q_last_missing ? n_kv - 1 : n_kv;
            if (n_q > 0)
                wait_bar(sh, p.status, &sh.qfull, static_cast<uint32_t>(n_q - 1) & 1u, false,
                         kDrainNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t speer = sbase + OFF_SPEER, sown = sbase + OFF_SOWN;
            for (int i = 0; i < n_own; ++i) {
                const int s = i & 1;
                const uint32_t u = static_cast<uint32_t>(i >> 1);
                const uint32_t ph = static_cast<uint32_t>(i) & 1u;
                if (!wait_bar(sh, p.status, &sh.kvready[s], u & 1u)) break;
                if (!wait_bar(sh, p.status, &sh.qhfull, ph)) break;
                tc_fence_after();
                const uint32_t ka = sbase + OFF_K + s * TILE, va = sbase + OFF_V + s * TILE;
                // scores A = Q^ K^T
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ts(tm + TM_A, tm + TM_Q + ks * 8,
                           smem_desc_sw128(ka + (ks >> 2) * HALF + (ks & 3) * 32, 16, 1024),
                           IDESC_QK, ks > 0);
                mma_commit(&sh.afull);
                if (!wait_bar(sh, p.status, &sh.yempty, ph ^ 1u)) break;
                if (!wait_bar(sh, p.status, &sh.sownfull, ph)) break;
                tc_fence_after();
                // Y = Q^ S_own
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ts(tm + TM_Y, tm + TM_Q + ks * 8,
                           smem_desc_sw128(sown + ks * 2048, HALF, 1024), IDESC_XB, ks > 0);
                // S_own += K^T V
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tm + TM_S, smem_desc_sw128(ka + ks * 2048, HALF, 1024),
                           smem_desc_sw128(va + ks * 2048, HALF, 1024), IDESC_KV, 1u);
                mma_commit(&sh.sdone);
                if (!wait_bar(sh, p.status, &sh.speerfull, ph)) break;
                if (i + 1 < n_own) mbar_arrive_expect_tx(&sh.speerfull, TILE);
                tc_fence_after();
                // Y += Q^ S_peer
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ts(tm + TM_Y, tm + TM_Q + ks * 8,
                           smem_desc_sw128(speer + ks * 2048, HALF, 1024), IDESC_XB, 1u);
                mma_commit_multicast(&sh.peercons, static_cast<uint16_t>(1u << peer));
                mma_commit(&sh.qhempty);
                if (!wait_bar(sh, p.status, &sh.pfull, ph)) break;
                tc_fence_after();
                // Y += mask(A) V^
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ts(tm + TM_Y, tm + TM_P + ks * 8,
                           smem_desc_sw128(va + ks * 2048, HALF, 1024), IDESC_XB, 1u);
                mma_commit(&sh.yfull);
                mma_commit(&sh.kvempty[s]);
            }
            mma_commit(&sh.mmadone);
            wait_bar(sh, p.status, &sh.mmadone, 0, false, kDrainNs);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ transform warpgroup
        const int q4 = warp - 4;
        const int t = q4 * 32 + lane;  // token row (q, k, v, A, P) or d_k row (S)
        const bool leader = t == 0;
        const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
        // initial state: S_in for rank 0 (or zeros), zeros for rank 1
        {
            const float* src =
                (rank == 0 && p.S_in) ? p.S_in + (static_cast<size_t>(item) * D + t) * D : nullptr;
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float4 f = src ? *reinterpret_cast<const float4*>(src + 32 * part + j)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    r[j] = __float_as_uint(f.x);
                    r[j + 1] = __float_as_uint(f.y);
                    r[j + 2] = __float_as_uint(f.z);
                    r[j + 3] = __float_as_uint(f.w);
                }
                LA_TMEM_ST32(lb + TM_S + 32 * part, r);
                store_row_bf16(sm + OFF_SOWN, t, part, r);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 128);
        int sends = 0, consumed = 0;
        const uint32_t peer_speer = map_to_rank(sbase + OFF_SPEER, peer);
        const uint32_t peer_bar = map_to_rank(smem_addr(&sh.speerfull), peer);
        if (leader) {
            mbar_arrive(&sh.sownfull);
            if (rank == 1 && n_peer > 0)
                bulk_copy_to_peer(peer_speer, sbase + OFF_SOWN, TILE, peer_bar);
        }
        if (rank == 1 && n_peer > 0) sends = 1;

        for (int i = 0; i < n_own; ++i) {
            const int s = i & 1;
            const uint32_t u = static_cast<uint32_t>(i >> 1);
            const uint32_t ph = static_cast<uint32_t>(i) & 1u;
            // (1) q -> SiLU -> TMEM (A operand of the score and state products)
            if (!group_wait(sh, p.status, &sh.qfull, ph, leader, 1, 128, 0)) break;
            if (!group_wait(sh, p.status, &sh.qhempty, ph ^ 1u, leader, 1, 128, 0)) break;
            tc_fence_after();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t r[32];
                const uint8_t* tile = sm + OFF_Q + hf * HALF;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 v = silu_chunk(*reinterpret_cast<const uint4*>(tile + swz(t, cc)));
                    r[4 * cc] = v.x;
                    r[4 * cc + 1] = v.y;
                    r[4 * cc + 2] = v.z;
                    r[4 * cc + 3] = v.w;
                }
                LA_TMEM_ST32(lb + TM_Q + 32 * hf, r);
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(1, 128);
            if (leader) {
                mbar_arrive(&sh.qhfull);
                mbar_arrive(&sh.qempty);
            }
            // (2) k, v -> SiLU in place (operands of the score, state and P V products)
            if (!group_wait(sh, p.status, &sh.kvfull[s], u & 1u, leader, 1, 128, 0)) break;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                uint8_t* tile = sm + (m == 0 ? OFF_K : OFF_V) + s * TILE;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        uint4* pch = reinterpret_cast<uint4*>(tile + hf * HALF + swz(t, cc));
                        *pch = silu_chunk(*pch);
                    }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) mbar_arrive(&sh.kvready[s]);
            // (3) P = A masked to s <= t, packed bf16 into TMEM
            if (!group_wait(sh, p.status, &sh.afull, ph, leader, 1, 128, 0)) break;
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                uint32_t r[32];
                LA_TMEM_LD32(lb + TM_A + 32 * part, r);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int s0 = 32 * part + 2 * j;
                    const float lo = s0 <= t ? __uint_as_float(r[2 * j]) : 0.f;
                    const float hi = s0 + 1 <= t ? __uint_as_float(r[2 * j + 1]) : 0.f;
                    pk[j] = pack_bf16x2(lo, hi);
                }
                LA_TMEM_ST16(lb + TM_P + 16 * part, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(1, 128);
            if (leader) mbar_arrive(&sh.pfull);
            // (4) bf16 copy of S_own for the next own chunk and for the peer
            const bool send = rank == 0 ? (i < n_peer) : (i + 1 < n_peer);
            if (i + 1 < n_own || send) {
                if (!group_wait(sh, p.status, &sh.sdone, ph, leader, 1, 128, 0)) break;
                if (sends > consumed) {
                    if (!group_wait(sh, p.status, &sh.peercons,
                                    static_cast<uint32_t>(consumed) & 1u, leader, 1, 128, 0))
                        break;
                    ++consumed;
                }
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t r[32];
                    LA_TMEM_LD32(lb + TM_S + 32 * part, r);
                    tmem_wait_ld();
                    store_row_bf16(sm + OFF_SOWN, t, part, r);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(1, 128);
                if (leader) {
                    mbar_arrive(&sh.sownfull);
                    if (send) bulk_copy_to_peer(peer_speer, sbase + OFF_SOWN, TILE, peer_bar);
                }
                if (send) ++sends;
            }
        }
        // the peer must have consumed our last copy before either CTA exits
        if (sends > consumed && leader)
            wait_bar(sh, p.status, &sh.peercons, static_cast<uint32_t>(consumed) & 1u,
                     !abort_set(sh), abort_set(sh) ? kDrainNs : kTimeoutNs);
    } else if (warp >= 8) {
        // ------------------------------------------------ epilogue (8 warps)
        const int e = warp - 8;
        const int q4 = e & 3, hf = e >> 2;  // TMEM lane quarter, column half
        const int t = q4 * 32 + lane;
        const int et = tid - 256;
        const bool leader = et == 0;
        const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
        for (int i = 0; i < n_own; ++i) {
            const int c = 2 * i + static_cast<int>(rank);
            const int64_t row0 = static_cast<int64_t>(c) * CH;
            const int64_t rem = p.N - row0;
            const int nc = rem < CH ? static_cast<int>(rem) : CH;
            const bool valid = t < nc;
            const size_t grow =
                ((static_cast<size_t>(b) * p.N + row0 + t) * p.H + h) * D + hf * 64;
            if (!group_wait(sh, p.status, &sh.yfull, static_cast<uint32_t>(i) & 1u, leader, 2,
                            256, 1))
                break;
            tc_fence_after();
            uint32_t y[64];
            LA_TMEM_LD32(lb + TM_Y + 64 * hf, y);
            LA_TMEM_LD32(lb + TM_Y + 64 * hf + 32, (y + 32));
            uint4 gv[8];
            if (valid) {
                const uint4* gp = reinterpret_cast<const uint4*>(p.g + grow);
#pragma unroll
                for (int j = 0; j < 8; ++j) gv[j] = __ldg(gp + j);
            }
            tmem_wait_ld();
            tc_fence_before();
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j)
                ss = fmaf(__uint_as_float(y[j]), __uint_as_float(y[j]), ss);
            sh.red[hf][t] = ss;
            named_bar_sync(2, 256);
            if (leader) mbar_arrive(&sh.yempty);
            // partial sums of squares of chunk c: [token t][head], H floats per token
            float* slot = p.xch + (static_cast<size_t>(b) * Nc + c) * CH * p.H;
            if (hf == 0) {
                slot[static_cast<size_t>(t) * p.H + h] = sh.red[0][t] + sh.red[1][t];
                __threadfence();
            }
            // while the other heads arrive: debug copy of y, then y *= sigmoid(g)
            if (valid) {
                if (p.y_dbg) {
                    float4* yp = reinterpret_cast<float4*>(p.y_dbg + grow);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        yp[j] = make_float4(__uint_as_float(y[4 * j]), __uint_as_float(y[4 * j + 1]),
                                            __uint_as_float(y[4 * j + 2]),
                                            __uint_as_float(y[4 * j + 3]));
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t gw[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        y[8 * j + 2 * k2] = __float_as_uint(__uint_as_float(y[8 * j + 2 * k2]) *
                                                            sigmoid_fast(bf_lo(gw[k2])));
                        y[8 * j + 2 * k2 + 1] = __float_as_uint(
                            __uint_as_float(y[8 * j + 2 * k2 + 1]) * sigmoid_fast(bf_hi(gw[k2])));
                    }
                }
            }
            named_bar_sync(2, 256);
            if (leader) {
                unsigned* cp = p.cnt + static_cast<size_t>(b) * Nc + c;
                red_release_gpu_add(cp, 1u);
                int ok = 1;
                uint64_t t0 = 0;
                for (uint32_t it = 0;; ++it) {
                    if (ld_acquire_gpu(cp) >= static_cast<unsigned>(p.H)) break;
                    if ((it & 63u) == 63u) {
                        if (abort_set(sh)) { ok = 0; break; }
                        const uint64_t now = global_timer_ns();
                        if (t0 == 0) t0 = now;
                        else if (now - t0 > kTimeoutNs) { raise_abort(sh, p.status); ok = 0; break; }
                    }
                }
                sh.verdict[1] = ok;
            }
            named_bar_sync(2, 256);
            if (!*reinterpret_cast<volatile int*>(&sh.verdict[1])) break;
            {
                // half hf sums heads [hh0, hh1) of token t; the loads are issued together
                const int hh0 = hf * (p.H / 2), hh1 = hf == 0 ? p.H / 2 : p.H;
                const float* src = slot + static_cast<size_t>(t) * p.H;
                float acc = 0.f;
                if ((p.H & 7) == 0) {
                    const float4* s4 = reinterpret_cast<const float4*>(src + hh0);
                    const int n4 = (hh1 - hh0) >> 2;
                    for (int base = 0; base < n4; base += 8) {
                        float4 v[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            v[j] = base + j < n4 ? __ldcg(s4 + base + j)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc += ((v[j].x + v[j].y) + (v[j].z + v[j].w));
                    }
                } else {
                    for (int base = hh0; base < hh1; base += 16) {
                        float v[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = base + j < hh1 ? __ldcg(src + base + j) : 0.f;
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc += v[j];
                    }
                }
                sh.red[hf][t] = acc;
            }
            named_bar_sync(2, 256);
            if (hf == 0) sh.rnorm[t] = rsqrtf((sh.red[0][t] + sh.red[1][t]) * p.inv_width + p.eps);
            named_bar_sync(2, 256);
            const float rn = sh.rnorm[t];
            if (valid) {
                uint4* op = reinterpret_cast<uint4*>(p.out + grow);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t ow[4];
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2)
                        ow[k2] = pack_bf16x2(__uint_as_float(y[8 * j + 2 * k2]) * rn,
                                             __uint_as_float(y[8 * j + 2 * k2 + 1]) * rn);
                    op[j] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                }
            }
        }
    }

    // ---------------------------------------------------- final state S_0 + S_1
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool ok_all = !abort_set(sh);
    const bool combine = p.S_out != nullptr;
    if (combine && rank == 1 && warp >= 4 && warp < 8) {
        const int q4 = warp - 4, t = q4 * 32 + lane;
        const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
        float* row = reinterpret_cast<float*>(sm + OFF_K + t * 512);
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            uint32_t r[32];
            LA_TMEM_LD32(lb + TM_S + 32 * part, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(row + 32 * part + j) =
                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        }
    }
    cluster_sync();
    if (combine && ok_all && rank == 0 && warp >= 4 && warp < 8) {
        const int q4 = warp - 4, t = q4 * 32 + lane;
        const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
        const uint32_t prow = map_to_rank(sbase + OFF_K + t * 512, peer);
        float* dst = p.S_out + (static_cast<size_t>(item) * D + t) * D;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            uint32_t r[32];
            LA_TMEM_LD32(lb + TM_S + 32 * part, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 o = ld_cluster_f4(prow + (32 * part + j) * 4);
                *reinterpret_cast<float4*>(dst + 32 * part + j) =
                    make_float4(__uint_as_float(r[j]) + o.x, __uint_as_float(r[j + 1]) + o.y,
                                __uint_as_float(r[j + 2]) + o.z, __uint_as_float(r[j + 3]) + o.w);
            }
        }
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::mutex g_occ_mutex;
int g_max_clusters[64];  // per device; 0 = not queried yet, -1 = unavailable

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

// [B][N][H*d] bf16 as a 3-D tensor (x = feature, y = token, z = sequence); boxes of
// 64 features x 128 tokens, 128B swizzle; tokens past N read as zero.
bool encode_io_map(CUtensorMap* m, const void* base, int B, int H, int64_t N) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * D * 2,
                             static_cast<cuuint64_t>(N) * H * D * 2};
    cuuint32_t box[3] = {64, CH, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int max_active_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    if (g_max_clusters[dev] != 0) return g_max_clusters[dev];
    int n = -1;
    if (cudaFuncSetAttribute(k_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_DYN)) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = SMEM_DYN;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int m = 0;
        if (cudaOccupancyMaxActiveClusters(&m, k_prefill_tc, &cfg) == cudaSuccess) n = m;
    }
    cudaGetLastError();
    g_max_clusters[dev] = n > 0 ? n : -1;
    return g_max_clusters[dev];
}

}  // namespace

int prefill_tc_supported(int B, int H, int64_t N) {
    if (N <= 0 || N > (int64_t(1) << 30)) return LA_ERR_UNSUPPORTED;
    if (!encoder()) return LA_ERR_UNSUPPORTED;
    const int mc = max_active_clusters();
    // every (b, h) pair must be resident at once for the cross-head exchange
    if (mc <= 0 || static_cast<int64_t>(B) * H > mc) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

size_t prefill_tc_workspace_bytes(int B, int H, int64_t N) {
    const int64_t Nc = (N + CH - 1) / CH;
    const size_t xch = static_cast<size_t>(B) * Nc * H * CH * sizeof(float);
    const size_t cnt = (static_cast<size_t>(B) * Nc * sizeof(unsigned) + 255) & ~size_t(255);
    return xch + cnt;
}

int launch_prefill_tc(const void* q, const void* k, const void* v, const void* g, void* out,
                      const float* S_in, float* S_out, float* y_debug, int B, int H, int64_t N,
                      float eps, const Workspace& ws, cudaStream_t st) {
    const int64_t Nc = (N + CH - 1) / CH;
    CUtensorMap mq, mk, mv;
    if (!encode_io_map(&mq, q, B, H, N) || !encode_io_map(&mk, k, B, H, N) ||
        !encode_io_map(&mv, v, B, H, N))
        return LA_ERR_UNSUPPORTED;
    Params prm;
    prm.g = static_cast<const __nv_bfloat16*>(g);
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.S_in = S_in;
    prm.S_out = S_out;
    prm.y_dbg = y_debug;
    const size_t xch_bytes = static_cast<size_t>(B) * Nc * H * CH * sizeof(float);
    prm.xch = static_cast<float*>(ws.base);
    prm.cnt = reinterpret_cast<unsigned*>(static_cast<char*>(ws.base) + xch_bytes);
    prm.status = ws.status;
    prm.B = B;
    prm.H = H;
    prm.N = N;
    prm.Nc = static_cast<int>(Nc);
    prm.eps = eps;
    prm.inv_width = 1.0f / static_cast<float>(H * D);
    if (cudaMemsetAsync(prm.cnt, 0, static_cast<size_t>(B) * Nc * sizeof(unsigned), st) !=
        cudaSuccess)
        return LA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * B * H), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM_DYN;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_prefill_tc, mq, mk, mv, prm) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    note_launches(1);
    return LA_OK;
}

}  // namespace la
