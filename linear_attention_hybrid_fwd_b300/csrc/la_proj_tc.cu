// la_proj_tc.cu -- the input projection of the Lightning Attention layer on tensor cores
// (sm_103a).
//
// What it computes ("Hybrid Modeling", MiniMax-01 deep dive, Hugging Face blog: step 1
// "Input X" and step 2 "Q, K, V = SiLU(X)", with the projections that the printed step
// leaves out):
//     [q~ | k~ | v~ | g] = x W^T      x: [T][hidden] bf16, W: [4*H*d][hidden] bf16
//     q, k, v = SiLU(q~), SiLU(k~), SiLU(v~) (or the raw values), g raw
// into four [T][H][d] bf16 tensors: exactly the inputs la_prefill reads.  The rows of W
// are the q, k, v and g output features in that order (a fused nn.Linear weight).
//
// Design (two-CTA clusters, one CTA per SM, persistent):
//  * Output tiles of 256 tokens x 256 features, one per CTA pair; with H*d a multiple of
//    256 a tile lies in one of the four outputs.  Tiles are visited in groups of 8 pair
//    rows (16 token blocks of 128), the token rows fastest, so the pairs working at one
//    time share a few weight panels and the x panel of the group stays in L2.
//  * The pair runs one M = 256 tcgen05.mma (cta_group::2, kind::f16, N = 256, K = 16,
//    fp32 accumulate): each CTA holds its 128 token rows of the x tile and 128 of the
//    256 weight rows, so a 64-wide K slice costs a CTA 32 KiB of shared memory instead
//    of 48, and six stages fit.  Warp 0 lane 0 of each CTA streams its two halves by
//    TMA (128B swizzle, cta_group::2) whose bytes complete on the even CTA's stage
//    barrier; only the even CTA announces the stage's bytes (both CTAs' share), since a
//    remote release-arrival from the odd CTA per stage measured 2x slower; warp 1 lane
//    0 of the even CTA issues the MMAs into one of two 256-column TMEM accumulators
//    (each CTA receives its 128 rows) and frees each stage in both CTAs with one commit.
//  * Warps 2-5 of each CTA drain the other accumulator while the next tile accumulates:
//    tcgen05.ld of 32 columns per thread (one token row each), SiLU for q, k, v, RNE to
//    bf16 and four 16-byte stores per row and slice, then a release arrival on the even
//    CTA's accumulator barrier.  Rows past T are not stored (loads past T or past hidden
//    read the tensor maps' zero fill, which adds nothing).
//  * SiLU(x) = x/2 (1 + tanh(x/2)) with the hardware tanh approximation, in fp32 on
//    the fp32 accumulator.
//  * Every wait is bounded (%globaltimer); a CTA that gives up records LA_ERR_TIMEOUT
//    in the status word, lets its copies and MMAs finish, frees TMEM and exits.
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

constexpr int BM = 128;                 // token rows per CTA (TMEM lanes); a pair: 256
constexpr int BN = 256;                 // output features per tile (TMEM columns)
constexpr int BNH = BN / 2;             // weight rows per CTA
constexpr int BK = 64;                  // K per stage: one 128-byte swizzle row
constexpr int kStages = 6;
constexpr int kThreads = 192;           // 6 warps
constexpr int kGroupM = 8;              // pair rows (256 tokens) per rasterisation group
constexpr uint32_t A_BYTES = BM * BK * 2;             // 16 KiB
constexpr uint32_t B_BYTES = BNH * BK * 2;            // 16 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KiB per CTA
constexpr uint32_t SMEM_DYN = kStages * STAGE_BYTES + 1024;  // + alignment slack
static_assert(SMEM_DYN + 1024 <= 227 * 1024, "shared memory budget");
constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN, 0, 0);  // M = 256, A and B K-major
constexpr uint64_t kTimeoutNs = 4000000000ull;  // 4 s
constexpr uint64_t kDrainNs = 200000000ull;     // 0.2 s

struct Params {
    __nv_bfloat16* out[4];  // q, k, v, g: [T][H*d]
    int* status;
    int T;                  // tokens
    int HD;                 // H * d
    int Mt, Nt, Kb;         // pair rows (256 tokens), feature blocks (all four outputs), K slices
    int tiles;              // Mt * Nt
    int activate;           // SiLU on q, k, v
};

struct Shared {
    // full, tempty, mmadone: used in the even CTA only
    uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], mmadone;
    uint32_t tmem_base;
    int abort_flag;
    int issued[2];          // per CTA of the pair: stage loads issued (even CTA's copy)
};

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float silu_t(float x) {
    const float h = 0.5f * x;
    return fmaf(h, tanh_approx(h), h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ bool abort_set(Shared& sh) {
    return *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0;
}
// Bounded wait for the phase of `bar` with `parity` (acquire at cluster scope when
// kCluster: the arrivals come from the other CTA); false when the CTA is aborting
// (honor_abort) or after `limit_ns`, in which case it raises the abort itself.
template <bool kCluster = false>
__device__ bool wait_bar(Shared& sh, int* status, uint64_t* bar, uint32_t parity,
                         bool honor_abort = true, uint64_t limit_ns = kTimeoutNs) {
    auto probe = [&]() {
        return kCluster ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (probe()) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (probe()) return true;
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

// Tile t -> (pair row m, feature block n): groups of kGroupM pair rows, the pair row
// fastest within a group.
__device__ __forceinline__ void tile_mn(const Params& p, int t, int& m, int& n) {
    const int per_group = kGroupM * p.Nt;
    const int grp = t / per_group;
    const int r = t - grp * per_group;
    const int m0 = grp * kGroupM;
    const int gm = p.Mt - m0 < kGroupM ? p.Mt - m0 : kGroupM;
    m = m0 + r % gm;
    n = r / gm;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_qkvg_proj(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                const Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Shared sh;
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);   // the even CTA's expect_tx for both CTAs' bytes
            mbar_init(&sh.empty[s], 1);  // the pair MMA's commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sh.tfull[a], 1);
            mbar_init(&sh.tempty[a], 8);  // one arrival per epilogue warp of both CTAs
        }
        mbar_init(&sh.mmadone, 1);
        sh.abort_flag = 0;
        sh.issued[0] = sh.issued[1] = 0;
        fence_mbar_init();
    }
    if (warp == 2) tmem_alloc_pair(&sh.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tm = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------------------- TMA producer
            // this CTA's 128 token rows and 128 weight rows of each stage, signalled on
            // the even CTA's stage barrier
            const uint32_t full0 = map_to_rank(smem_addr(&sh.full[0]), 0);
            int it = 0;
            bool ok = true;
            for (int t = pair; t < p.tiles && ok; t += npairs) {
                int m, n;
                tile_mn(p, t, m, n);
                for (int kb = 0; kb < p.Kb; ++kb) {
                    const int s = it % kStages;
                    const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                    if (!wait_bar(sh, p.status, &sh.empty[s], ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = sm + s * STAGE_BYTES;
                    const uint32_t fb = full0 + static_cast<uint32_t>(s) * 8u;
                    // the even CTA announces both CTAs' bytes; the odd CTA's copies only
                    // complete their share (a count that may run ahead of the announcement)
                    if (rank == 0) mbar_arrive_expect_tx(&sh.full[s], 2 * STAGE_BYTES);
                    tma_load_3d_pair(st, &tx, kb * BK, m * 2 * BM + static_cast<int>(rank) * BM, 0,
                                     fb);
                    tma_load_3d_pair(st + A_BYTES, &tw, kb * BK, n * BN + static_cast<int>(rank) * BNH,
                                     0, fb);
                    ++it;
                }
            }
            // the even CTA drains both producers' loads (its stage barriers count them)
            st_cluster_s32(map_to_rank(smem_addr(&sh.issued[rank]), 0), it);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------------------- MMA issuer (even CTA)
            int it = 0, ti = 0;
            bool ok = true;
            for (int t = pair; t < p.tiles && ok; t += npairs, ++ti) {
                const int a = ti & 1;
                const uint32_t aph = static_cast<uint32_t>(ti >> 1) & 1u;
                if (!wait_bar<true>(sh, p.status, &sh.tempty[a], aph ^ 1u)) break;
                tc_fence_after();
                const uint32_t acc = tm + static_cast<uint32_t>(a * BN);
                for (int kb = 0; kb < p.Kb; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                    if (!wait_bar<true>(sh, p.status, &sh.full[s], ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + s * STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks)
                        mma_ss_pair(acc, smem_desc_sw128(sa + ks * 32, 16, 1024),
                                    smem_desc_sw128(sb + ks * 32, 16, 1024), IDESC,
                                    (kb | ks) != 0 ? 1u : 0u);
                    mma_commit_pair(&sh.empty[s], static_cast<uint16_t>(3u));
                }
                if (!ok) break;
                mma_commit_pair(&sh.tfull[a], static_cast<uint16_t>(3u));
            }
            mma_commit_pair(&sh.mmadone, static_cast<uint16_t>(1u));
            wait_bar(sh, p.status, &sh.mmadone, 0, false, kDrainNs);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int quarter = warp & 3;  // TMEM lanes 32 quarter .. 32 quarter + 31
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tempty0 = map_to_rank(smem_addr(&sh.tempty[0]), 0);
        int ti = 0;
        for (int t = pair; t < p.tiles; t += npairs, ++ti) {
            const int a = ti & 1;
            const uint32_t aph = static_cast<uint32_t>(ti >> 1) & 1u;
            const bool got = wait_bar(sh, p.status, &sh.tfull[a], aph);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            int m, n;
            tile_mn(p, t, m, n);
            const int f0 = n * BN;            // feature of the fused output
            const int seg = f0 / p.HD;        // 0 q, 1 k, 2 v, 3 g
            const int col0 = f0 - seg * p.HD;
            const bool act = p.activate != 0 && seg < 3;
            const int64_t row = static_cast<int64_t>(m) * 2 * BM + static_cast<int>(rank) * BM +
                                quarter * 32 + lane;
            const bool live = row < p.T;
            __nv_bfloat16* base =
                seg == 0 ? p.out[0] : seg == 1 ? p.out[1] : seg == 2 ? p.out[2] : p.out[3];
            __nv_bfloat16* dst = base + row * p.HD + col0;
            const uint32_t tbase = tm + static_cast<uint32_t>(a * BN) + lane_base;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                LA_TMEM_LD32(tbase + c * 32, r);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float x0 = __uint_as_float(r[2 * j]), x1 = __uint_as_float(r[2 * j + 1]);
                    if (act) {
                        x0 = silu_t(x0);
                        x1 = silu_t(x1);
                    }
                    pk[j] = pack_bf16x2(x0, x1);
                }
                if (live) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tempty0 + static_cast<uint32_t>(a) * 8u);
        }
    }
    // teardown: the even CTA waits for any stage the producers filled but the MMAs did
    // not take (abort paths only), then both leave together
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both producers published their counts
    if (rank == 0 && tid == 0) {
        const int n = sh.issued[0] > sh.issued[1] ? sh.issued[0] : sh.issued[1];
        for (int it = n - kStages < 0 ? 0 : n - kStages; it < n; ++it)
            wait_bar(sh, p.status, &sh.full[it % kStages], static_cast<uint32_t>(it / kStages) & 1u,
                     false, kDrainNs);
    }
    __syncthreads();
    cluster_sync();  // no copy, MMA or arrival targets a CTA that has left
    tc_fence_after();
    if (warp == 2) tmem_dealloc_pair(tm, 512);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::mutex g_dev_mutex;
int g_sms[64];         // per device: co-resident two-CTA clusters (0 = not queried yet)
bool g_attr_set[64];   // per device: the kernel's shared-memory attribute is set

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

// A row-major [rows][cols] bf16 matrix as a 3-D tensor (x = column, y = row, z = 1),
// boxes of 64 columns x box_rows rows, 128B swizzle; reads past either edge give zeros.
bool encode_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                             static_cast<cuuint64_t>(cols) * 2 * static_cast<cuuint64_t>(rows)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Two-CTA clusters of the kernel that the current device holds at once, with the
// kernel's shared-memory attribute set; 0 on failure.
int prepare_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_attr_set[dev]) {
        if (cudaFuncSetAttribute(k_qkvg_proj, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SMEM_DYN)) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_attr_set[dev] = true;
    }
    if (!g_sms[dev]) {
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
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_qkvg_proj, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            return 0;
        }
        g_sms[dev] = n;
    }
    return g_sms[dev];
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

extern "C" int la_qkvg_projection(const void* x, const void* w, void* q, void* k, void* v,
                                  void* g, int64_t T, int hidden, int H, int d, unsigned flags,
                                  void* cuda_stream) {
    if (T < 0 || hidden <= 0 || H <= 0 || d <= 0) return LA_ERR_INVALID_ARG;
    if ((flags & ~LA_PROJ_SILU) != 0) return LA_ERR_INVALID_ARG;
    if (d != kHeadDim || (static_cast<int64_t>(H) * d) % BN != 0 || hidden % 8 != 0)
        return LA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(H) * d * 4 > (int64_t(1) << 30) || hidden > (1 << 24) ||
        T > (int64_t(1) << 30) ||
        ((T + BM - 1) / BM) * (static_cast<int64_t>(H) * d * 4 / BN) > (int64_t(1) << 30))
        return LA_ERR_UNSUPPORTED;
    if (!x || !w || !q || !k || !v || !g) return LA_ERR_INVALID_ARG;
    const void* ptrs[] = {x, w, q, k, v, g};
    for (const void* p : ptrs)
        if (!aligned16(p)) return LA_ERR_MISALIGNED;
    const int HD = H * d;
    const size_t out_bytes = static_cast<size_t>(T) * HD * 2;
    const size_t x_bytes = static_cast<size_t>(T) * hidden * 2;
    const size_t w_bytes = static_cast<size_t>(4) * HD * hidden * 2;
    void* outs[4] = {q, k, v, g};
    for (int i = 0; i < 4; ++i) {
        if (overlaps(outs[i], out_bytes, x, x_bytes) || overlaps(outs[i], out_bytes, w, w_bytes))
            return LA_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(outs[i], out_bytes, outs[j], out_bytes)) return LA_ERR_INVALID_ARG;
    }
    if (T == 0) return LA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    const int pairs = prepare_device();
    if (pairs <= 0) return LA_ERR_CUDA;
    Workspace ws;
    int rc = workspace_acquire(0, st, &ws);
    if (rc != LA_OK) return rc;
    CUtensorMap mx, mw;
    if (!encode_rows(&mx, x, T, hidden, BM) || !encode_rows(&mw, w, int64_t(4) * HD, hidden, BNH))
        return LA_ERR_UNSUPPORTED;
    Params prm;
    for (int i = 0; i < 4; ++i) prm.out[i] = static_cast<__nv_bfloat16*>(outs[i]);
    prm.status = ws.status;
    prm.T = static_cast<int>(T);
    prm.HD = HD;
    prm.Mt = static_cast<int>((T + 2 * BM - 1) / (2 * BM));
    prm.Nt = 4 * HD / BN;
    prm.Kb = (hidden + BK - 1) / BK;
    prm.tiles = prm.Mt * prm.Nt;
    prm.activate = (flags & LA_PROJ_SILU) ? 1 : 0;
    const int npairs = prm.tiles < pairs ? prm.tiles : pairs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * npairs), 1, 1);
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
    if (cudaLaunchKernelEx(&cfg, k_qkvg_proj, mx, mw, prm) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    note_launches(1);
    return LA_OK;
}
