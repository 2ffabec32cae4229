// la_prefill_tc.cu -- tensor-core prefill of the Lightning Attention layer (sm_103a).
//
// What it computes ("Hybrid Modeling", MiniMax-01 deep dive, Hugging Face blog,
// mechanism steps 2-4): q^,k^,v^ = SiLU(q,k,v); y_t = q^_t sum_{s<=t} k^_s^T v^_s;
// out = y / sqrt(mean over the H*d features of y^2 + eps) * sigmoid(g).  The causal
// product takes the blockwise O(d^2 n) route of the same section: per chunk c of 128
// tokens
//     Y_c = Q^_c S_{<c} + (Q^_c K^_c^T * M) V^_c ,    S_{<c+1} = S_{<c} + K^_c^T V^_c
// with M the inclusive lower-triangular mask and S the fp32 d x d state.
//
// Design (one B300 SM per CTA, 209 KiB shared memory, all 512 TMEM columns):
//  * A cluster of two CTAs owns one head h and runs through every chunk of every
//    sequence of the batch in order.  The pair splits the d_v columns: CTA r keeps the
//    state columns S[:, 64r, 64r+64) in TMEM and produces y and out for those columns.
//    Nothing on the state's chunk-to-chunk path crosses the pair.
//  * The activations are not duplicated: CTA 0 loads q and applies SiLU, CTA 1 does the
//    same for k, and each bulk-copies its activated 128 x 128 tile into the other's
//    shared memory.  Each CTA activates its own 64 columns of v.  Both then form the
//    full 128 x 128 score tile Q^ K^T (one N = 128 MMA chain: 64 tensor cycles per k-step
//    against 2 x 48 for two N = 64 halves on B300) and their halves of the products.
//  * Warp roles of a head's CTA (28 warps): warp 0 issues TMA loads (lane 0: q or k and
//    v; lane 1: g), warp 1 issues tcgen05 MMAs; warps 4-11 (2-4, 6-8, 10-11 on activated
//    inputs, keeping the MMA warp's sub-partition free of them) apply SiLU in shared memory
//    and push the activated tile to the peer; warps 12-15 convert the fp32 state to the
//    bf16 operand of Q^ S and mask each score half into the bf16 P operand (written in
//    place over it; a key block wholly below a warp's rows is converted without
//    selects); warps 16-19 post each chunk's per-token sums of squares; warps
//    20-23 and 24-27 finish every chunk together, each group half of y's columns
//    (norm, gate, TMA store).
//  * The RMSNorm spans all heads of a token.  The SMs the head pairs leave free run
//    reducer CTAs in the same co-resident grid: each head half posts its 128 per-token
//    sums of squares to a global slot and counts itself in; a reducer waits (bounded)
//    for all 2H halves of a chunk, sums them with all its threads in a fixed order
//    (deterministic) and publishes the chunk's 128 norm factors, whose slots hold an "empty" bit pattern
//    until written, so the finishing warps read their factor with one load.  A launch
//    resets the previous launch's counters and factors in the other of two banks.  y
//    stays in TMEM (five buffers) while the exchange is in flight.  The host checks
//    that the whole grid is co-resident before launching.
//  * q, k, v and g arrive by TMA in 128B-swizzled tiles, double-buffered; out leaves by
//    TMA store from the g tile it replaces (row by row for a partial chunk of a packed
//    batch, whose last rows belong to the next sequence).
//  * A batch is a list of (sequence, chunk) items run in order: B sequences of N tokens,
//    or sequences of any lengths packed back to back (the rows of a chunk past its
//    sequence's end are zeroed after loading, so they add nothing to any product).
//  * SiLU(x) = x/2 (1 + tanh(x/2)) and y r sigmoid(g) = a + a tanh(g/2) (a = y r / 2) with
//    the hardware tanh approximation: one SFU operation per element; x/2 and g/2 are
//    taken on the packed bf16 pair (exact), which saves an instruction per element on
//    an issue-bound path.
//  * Every wait is bounded (%globaltimer); a CTA that gives up records LA_ERR_TIMEOUT
//    in the status word, drains its in-flight copies and MMAs, frees TMEM and exits.
//
// TMEM columns: [0,128) scores, keys 0-63 then 64-127 (P of each half over its first 32) |
//               [128,192) S (fp32, this CTA's 64 columns) | [192,512) Y0 .. Y4.
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
constexpr int DV = 64;                // d_v columns per CTA
constexpr int kThreads = 896;         // 28 warps
constexpr int kYBufs = 5;             // y tiles in TMEM
constexpr int kMaxReducers = 16;      // reducer CTAs (on SMs the head pairs leave free)
constexpr int kGBufs = 2;             // g tiles in flight (TMA-loaded ahead of the epilogue)
constexpr int kPartRing = 16;         // chunks whose per-token partials are held at once
constexpr int kMinSegChunks = 64;     // segment mode: chunks per segment at least
constexpr uint32_t TILE = 32768;      // 128 x 128 bf16 = two swizzled 128 x 64 halves
constexpr uint32_t HALF = 16384;      // 128 x 64 bf16, one 128B-swizzled block
constexpr uint32_t OFF_QB = 0;                  // 2 stages: q^ tiles
constexpr uint32_t OFF_KB = OFF_QB + 2 * TILE;  // 2 stages: k^ tiles
constexpr uint32_t OFF_VB = OFF_KB + 2 * TILE;  // 2 stages: v^ (this CTA's 64 columns)
constexpr uint32_t OFF_SB = OFF_VB + 2 * HALF;  // bf16 state slice (MN-major B operand)
constexpr uint32_t OFF_GB = OFF_SB + HALF;      // kGBufs g tiles (this CTA's 64 columns)
constexpr uint32_t SMEM_USED = OFF_GB + kGBufs * HALF;  // 208 KiB
constexpr uint32_t SMEM_DYN = SMEM_USED + 1024; // + alignment slack
static_assert(SMEM_DYN + 6144 <= 227 * 1024, "shared memory budget");
constexpr uint32_t TM_A = 0, TM_S = 128, TM_Y = 192;
constexpr uint64_t kTimeoutNs = 4000000000ull;  // 4 s
constexpr uint64_t kDrainNs = 200000000ull;     // 0.2 s

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, 0, 0);  // A K-major, B K-major
constexpr uint32_t IDESC_QS = idesc_bf16_f32(128, DV, 0, 1);   // A K-major, B MN-major
constexpr uint32_t IDESC_KV = idesc_bf16_f32(128, DV, 1, 1);   // A MN-major, B MN-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, DV, 0, 1);   // A (TMEM), B MN-major

struct Params {
    __nv_bfloat16* out;  // partial chunks of packed batches are stored from here
    const float* S_in;
    float* S_out;
    float* y_dbg;
    unsigned* cnt;       // [B*Nc] head halves posted, from kXchEmpty
    float* rn;           // [B*Nc][CH] norm factors (kXchEmpty until written)
    float* part;         // [kPartRing][2H][CH] per-token sums of squares of each head half,
                         // chunk `it` in slot it % kPartRing
    uint4* xch_clear;    // the other bank's counters and factors of the previous launch
    int64_t n_clear4;    // ... as a count of 16-byte words
    int* status;
    const int4* items;   // per iteration {first row, valid rows, sequence, first chunk of it}
                         // (packed varlen batches), or nullptr: B sequences of N tokens
    int B, H;
    int64_t N;           // tokens per sequence (the packed token count for varlen)
    int Nc;              // chunks per sequence (uniform batches)
    uint64_t nc_magic;   // floor((2^64 - 1) / Nc): umulhi64(it, nc_magic) is it / Nc or one less
    int total;           // iterations: (sequence, chunk) items in order
    int nseg;            // segments of the item list, each run by its own head pairs (B == 1)
    int seg_items;       // items per segment (the last may have fewer)
    const float* S_seg;  // segment mode: [nseg][H][d][d] state before each segment
    float eps;
    float inv_width;     // 1 / (H * d)
};

// One (sequence, chunk) iteration: its tile rows start at token y of slab z of the
// [z][token][feature] tensor maps; rows >= nvalid are not part of the sequence.
struct Item {
    int y, z, nvalid, b, first;
};
template <bool kVarlen>
__device__ __forceinline__ Item item_at(const Params& p, int it) {
    Item r;
    if constexpr (kVarlen) {
        const int4 e = p.items[it];
        r.y = e.x;
        r.z = 0;
        r.nvalid = e.y;
        r.b = e.z;
        r.first = e.w;
    } else {
        int b = static_cast<int>(__umul64hi(static_cast<uint64_t>(it), p.nc_magic));
        int c = it - b * p.Nc;
        if (c >= p.Nc) {  // the estimate is at most one low
            ++b;
            c -= p.Nc;
        }
        const int64_t rem = p.N - static_cast<int64_t>(c) * CH;
        r.y = c * CH;
        r.z = b;
        r.nvalid = rem < CH ? static_cast<int>(rem) : CH;
        r.b = b;
        r.first = c == 0;
    }
    return r;
}

struct Shared {
    uint64_t rawqk[2], rawv[2], xin[2], actdone[2], qkempty[2], vempty[2];
    uint64_t afull[2], aempty[2], pfull[2], sdone, sready;
    uint64_t yfull[kYBufs], yempty[kYBufs], gfull[kGBufs], gempty[kGBufs], mmadone;
    uint32_t tmem_base;
    int abort_flag;
    int verdict[5];  // group-uniform wait results (SiLU, mask, post, finish 0, finish 1)
    int issued;      // iterations whose q or k loads the producer issued
    int xin_seen;    // iterations whose peer tile the MMA issuer consumed
    int g_issued;    // iterations whose g tile was issued
    float red[kThreads / 128][CH];  // reducer: per-token sums over ranges of head halves
};

// Per-stage timeline (a build with -DLA_TIMELINE only): %globaltimer stamps of the
// pipeline events of the first kTlChunks iterations of every CTA, read back with
// la_timeline_fetch.  Event numbers are listed in linear_attention_hybrid_fwd_b300/timeline.py.
#ifdef LA_TIMELINE
constexpr int kTlCtas = 160, kTlChunks = 64, kTlEvents = 32;
__device__ unsigned long long g_la_timeline[kTlCtas * kTlChunks * kTlEvents];
__device__ __forceinline__ void tl_stamp(int it, int e) {
    if (it >= 0 && it < kTlChunks && blockIdx.x < kTlCtas) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        g_la_timeline[(blockIdx.x * kTlChunks + it) * kTlEvents + e] = t;
    }
}
#define LA_TL(e) tl_stamp(it, (e))
#else
#define LA_TL(e) ((void)0)
#endif

// ------------------------------------------------------------------ numerics
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// SiLU(x) = x sigmoid(x) = h (1 + tanh(h)) with h = x/2.
__device__ __forceinline__ float silu_h(float h) { return fmaf(h, tanh_approx(h), h); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
// Both bf16 halves times 1/2 (exact: a power-of-two scaling of a bf16 value).
__device__ __forceinline__ uint32_t half_bf16x2(uint32_t u) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(u), "r"(0x3F003F00u));
    return r;
}
__device__ __forceinline__ uint32_t silu_bf16x2(uint32_t u) {
    const uint32_t hh = half_bf16x2(u);
    return pack_bf16x2(silu_h(bf_lo(hh)), silu_h(bf_hi(hh)));
}
__device__ __forceinline__ uint4 silu_chunk(uint4 v) {
    return make_uint4(silu_bf16x2(v.x), silu_bf16x2(v.y), silu_bf16x2(v.z), silu_bf16x2(v.w));
}

// Byte offset of the 16-byte chunk `c` (0..7) of row `r` in a 128B-swizzled block.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Smem descriptors.  K-major operand with K = 128 split into two 64-wide swizzled
// halves; k-step ks (16 elements = 32 bytes).  MN-major operand: k-step ks covers 16 rows
// (2048 bytes); `lbo` is the distance between 64-element MN blocks.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int ks) {
    return smem_desc_sw128(base + (ks >> 2) * HALF + (ks & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int ks) {
    return smem_desc_sw128(base + ks * 2048, HALF, 1024);
}
// A descriptor moved on by `off` bytes (a multiple of 16).  The start address is the
// low 14-bit field (address / 16) and every operand lies below 256 KiB, so the add stays
// in the low word.  The MMA issuer builds each stage's descriptors once per chunk and
// moves them by constants: it issues 32 MMAs per chunk, and their issue rate, not the
// tensor pipe, sets its pace.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off) {
    const uint32_t lo = static_cast<uint32_t>(d) + (off >> 4);
    return (d & 0xFFFFFFFF00000000ull) | lo;
}
// Offset of k-step ks (16 elements) in a K-major 128 x 128 tile of two swizzled halves.
__device__ __forceinline__ constexpr uint32_t kofs(int ks) {
    return static_cast<uint32_t>((ks >> 2) * HALF + (ks & 3) * 32);
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
// The spinning part of wait_bar, out of line: a wait that succeeds at once costs no
// instruction-cache lines at its call site.
template <bool kCluster>
__device__ __noinline__ bool wait_bar_spin(Shared& sh, int* status, uint64_t* bar,
                                           uint32_t parity, bool honor_abort,
                                           uint64_t limit_ns) {
    auto probe = [&]() {
        return kCluster ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (probe()) return true;
        if ((it & 15u) == 0) {
            if (honor_abort && abort_set(sh)) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                raise_abort(sh, status);
                return false;
            }
        }
    }
}
// Waits for the phase of `bar` with `parity` to complete.  Gives up (false) when the
// CTA is aborting (honor_abort) or after `limit_ns`, raising the abort itself.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(Shared& sh, int* status, uint64_t* bar,
                                         uint32_t parity, bool honor_abort = true,
                                         uint64_t limit_ns = kTimeoutNs) {
    const bool done =
        kCluster ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity);
    if (done) return true;
    return wait_bar_spin<kCluster>(sh, status, bar, parity, honor_abort, limit_ns);
}
// Group-uniform wait: thread `leader` waits (bounded), the group of `n` threads syncs on
// named barrier `id`, then every thread observes the completed phase itself.  No
// barrier used with it can complete a further phase before every thread of the group
// has observed this one (each next phase needs an arrival from this group).
template <bool kCluster = false>
__device__ bool group_wait(Shared& sh, int* status, uint64_t* bar, uint32_t parity, bool leader,
                           uint32_t id, uint32_t n, int slot) {
    if (leader) sh.verdict[slot] = wait_bar<kCluster>(sh, status, bar, parity) ? 1 : 0;
    named_bar_sync(id, n);
    const bool ok = *reinterpret_cast<volatile int*>(&sh.verdict[slot]) != 0;
    if (ok) {
        if (kCluster) {
            while (!mbar_try_wait_acq_cluster(bar, parity)) {
            }
        } else {
            while (!mbar_try_wait(bar, parity)) {
            }
        }
    }
    named_bar_sync(id, n);  // verdict slot may be rewritten only after everyone read it
    return ok;
}

// Write 32 fp32 values (columns 32*part .. +31 of row r, part 0 or 1) as bf16 into a
// 128B-swizzled 128 x 64 block.
__device__ __forceinline__ void store_row_bf16(uint8_t* blk, int r, int part,
                                               const uint32_t (&v)[32]) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(v[8 * cc + 0]), __uint_as_float(v[8 * cc + 1]));
        w.y = pack_bf16x2(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3]));
        w.z = pack_bf16x2(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5]));
        w.w = pack_bf16x2(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7]));
        *reinterpret_cast<uint4*>(blk + swz(r, part * 4 + cc)) = w;
    }
}

// A sequence's first chunk and last chunk: the conversion warps move this CTA's 64
// state columns of d_k row t between global memory and TMEM (out of line: once per
// sequence, kept out of the per-chunk code).
__device__ __noinline__ void state_rows_out(float* dst, uint32_t ts) {
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        uint32_t r[32];
        LA_TMEM_LD32(ts + 32 * part, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + 32 * part + j) =
                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
    }
}
__device__ __noinline__ void state_rows_in(const float* src, uint32_t ts, uint8_t* sbk, int t) {
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 f = src ? *reinterpret_cast<const float4*>(src + 32 * part + j)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            r[j] = __float_as_uint(f.x);
            r[j + 1] = __float_as_uint(f.y);
            r[j + 2] = __float_as_uint(f.z);
            r[j + 3] = __float_as_uint(f.w);
        }
        LA_TMEM_ST32(ts + 32 * part, r);
        store_row_bf16(sbk, t, part, r);
    }
    tmem_wait_st();
}

// Bounded spin until *cnt == target (unsigned compare); false after a timeout (raising
// the abort) or when the CTA is aborting.
__device__ bool spin_until(Shared& sh, int* status, const unsigned* cnt, unsigned target) {
    uint64_t t0 = 0;
    for (;;) {
        if (ld_acquire_gpu(cnt) == target) return true;
        if (abort_set(sh)) return false;
        const uint64_t now = global_timer_ns();
        if (t0 == 0) {
            t0 = now;
        } else if (now - t0 > kTimeoutNs) {
            raise_abort(sh, status);
            return false;
        }
        __nanosleep(200);
    }
}

// Bounded spin until the norm factor at `slot` is published (acquire); false after a
// timeout (raising the abort) or when the CTA is aborting.
__device__ bool spin_published(Shared& sh, int* status, const float* slot) {
    const unsigned* w = reinterpret_cast<const unsigned*>(slot);
    uint64_t t0 = 0;
    for (;;) {
        if (ld_acquire_gpu(w) != kXchEmpty) return true;
        if (abort_set(sh)) return false;
        const uint64_t now = global_timer_ns();
        if (t0 == 0) {
            t0 = now;
        } else if (now - t0 > kTimeoutNs) {
            raise_abort(sh, status);
            return false;
        }
        __nanosleep(200);
    }
}

// Reducer CTA: for its chunks (every R-th), waits for all 2H head halves' per-token sums
// of squares and publishes r_t = 1 / sqrt(mean + eps) for the chunk's 128 tokens.  Its
// kThreads / 128 groups of 128 threads (one per token) each add a fixed range of head
// halves in order; the ranges' sums are then added in range order (deterministic).
__device__ void reducer(Shared& sh, float (*red)[CH], const Params& p, int j, int R) {
    constexpr int G = kThreads / CH;  // 7 groups
    const int tid = threadIdx.x;
    const int t = tid & (CH - 1), gidx = tid >> 7;
    const bool leader = tid == 0;
    const int H2 = 2 * p.H, total = p.total;
    const int per = (H2 + G - 1) / G;
    const int lo = gidx * per, hi = lo + per < H2 ? lo + per : H2;
    const unsigned target = kXchEmpty + static_cast<unsigned>(H2);
    // chunks in the order the head pairs produce them: place li of every segment before
    // place li + 1 (one segment: chunk order)
    const int nseg = p.nseg, span = nseg * p.seg_items;
    for (int u = j; u < span; u += R) {
        const int li = u / nseg, sg = u - li * nseg;
        const int it = sg * p.seg_items + li;
        if (it >= total) continue;  // past the end of a shorter last segment
        if (leader) sh.verdict[0] = spin_until(sh, p.status, p.cnt + it, target) ? 1 : 0;
        __syncthreads();
        if (!*reinterpret_cast<volatile int*>(&sh.verdict[0])) break;
        if (tid == 0) LA_TL(25);
        // the chunk's partials slot: its segment's ring, its place in the segment mod the ring
        const float* src =
            p.part + (static_cast<size_t>(sg) * kPartRing + li % kPartRing) * H2 * CH + t;
        float acc = 0.f;
        for (int k0 = lo; k0 < hi; k0 += 8) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = k0 + k < hi ? __ldcg(src + static_cast<size_t>(k0 + k) * CH) : 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) acc += v[k];
        }
        red[gidx][t] = acc;
        __syncthreads();
        if (gidx == 0) {
            float tot = 0.f;
#pragma unroll
            for (int g = 0; g < G; ++g) tot += red[g][t];
            const float r = rsqrtf(tot * p.inv_width + p.eps);
            float* dst = p.rn + static_cast<size_t>(it) * CH + t;
            if (t == 0)  // after the barrier above: every read of the chunk's partials is done
                st_release_gpu_u32(reinterpret_cast<unsigned*>(dst), __float_as_uint(r));
            else
                __stcg(dst, r);
            if (t == 0) LA_TL(26);
        }
        __syncthreads();  // red is rewritten by the next chunk
    }
}

// ------------------------------------------------------------------ the kernel
// kVarlen: the items come from the packed batch's table (p.items) rather than from the
// uniform B x ceil(N / 128) grid of chunks; the uniform instance carries none of the
// packed batch's checks.  kAct: q, k, v arrive already SiLU-activated, and the
// activation warps only zero the rows past a packed sequence's end and forward tiles.
template <bool kVarlen, bool kAct>
__global__ void __launch_bounds__(kThreads, 1)
    k_prefill_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                 const __grid_constant__ CUtensorMap to, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Shared sh;
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int H = p.H;
    const int total = p.total;                               // (sequence, chunk) iterations
    const int cl = static_cast<int>(blockIdx.x >> 1);        // head pair index
    const int h = cl % H, seg = cl / H;                      // head, segment of the items
    const int it0 = seg * p.seg_items;                       // this pair's items: [it0, it0 + n_loc)
    const int n_loc = (total - it0 < p.seg_items ? total - it0 : p.seg_items);
    const int col0 = h * D + static_cast<int>(rank) * DV;    // first feature column owned
    const uint32_t own_off = rank == 0 ? OFF_QB : OFF_KB;    // the tile this CTA activates

    // the previous launch's counters and factors in the other bank become empty again
    {
        const uint4 e = make_uint4(kXchEmpty, kXchEmpty, kXchEmpty, kXchEmpty);
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + tid; i < p.n_clear4;
             i += static_cast<int64_t>(gridDim.x) * kThreads)
            p.xch_clear[i] = e;
    }
    const int heads2 = 2 * H * p.nseg;  // head CTAs; the reducer CTAs follow
    if (static_cast<int>(blockIdx.x) >= heads2) {  // a reducer CTA (no TMEM, no cluster traffic)
        if (tid == 0) {
            sh.abort_flag = 0;
            sh.verdict[0] = 0;
        }
        __syncthreads();
        reducer(sh, sh.red, p, static_cast<int>(blockIdx.x) - heads2,
                static_cast<int>(gridDim.x) - heads2);
        return;
    }

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.rawqk[s], 1);
            mbar_init(&sh.rawv[s], 1);
            mbar_init(&sh.xin[s], 1);
            mbar_init(&sh.actdone[s], 1);
            mbar_init(&sh.qkempty[s], 2);  // this CTA's MMAs and the peer's
            mbar_init(&sh.vempty[s], 1);
            mbar_init(&sh.afull[s], 1);
            mbar_init(&sh.aempty[s], 1);
            mbar_init(&sh.pfull[s], 1);
        }
        for (int y = 0; y < kYBufs; ++y) {
            mbar_init(&sh.yfull[y], 1);
            mbar_init(&sh.yempty[y], 2);  // both finishing groups
        }
        for (int i = 0; i < kGBufs; ++i) {
            mbar_init(&sh.gfull[i], 1);
            mbar_init(&sh.gempty[i], 1);
        }
        mbar_init(&sh.sdone, 1);
        mbar_init(&sh.sready, 1);
        mbar_init(&sh.mmadone, 1);
        sh.abort_flag = 0;
        for (int i = 0; i < 5; ++i) sh.verdict[i] = 0;
        sh.issued = 0;
        sh.xin_seen = 0;
        sh.g_issued = 0;
        fence_mbar_init();
    }
    if (warp == 2) tmem_alloc(&sh.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before anything reaches them
    tc_fence_after();
    const uint32_t tm = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------- TMA producer: q or k, and v
            const CUtensorMap* own_map = rank == 0 ? &tq : &tk;
            int issued = 0;
            for (int it = 0; it < n_loc; ++it) {
                const Item im = item_at<kVarlen>(p, it0 + it);
                const int s = it & 1;
                const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
                if (!wait_bar(sh, p.status, &sh.qkempty[s], ph ^ 1u)) break;
                uint8_t* own = sm + own_off + s * TILE;
                mbar_arrive_expect_tx(&sh.rawqk[s], TILE);
                tma_load_3d(own, own_map, h * D, im.y, im.z, &sh.rawqk[s]);
                tma_load_3d(own + HALF, own_map, h * D + 64, im.y, im.z, &sh.rawqk[s]);
                LA_TL(0);
                mbar_arrive_expect_tx(&sh.xin[s], TILE);  // the peer's activated tile
                issued = it + 1;
                if (!wait_bar(sh, p.status, &sh.vempty[s], ph ^ 1u)) break;
                mbar_arrive_expect_tx(&sh.rawv[s], HALF);
                tma_load_3d(sm + OFF_VB + s * HALF, &tv, col0, im.y, im.z, &sh.rawv[s]);
                LA_TL(1);
            }
            sh.issued = issued;
            // drain: the last loads land before this CTA may exit
            for (int it = issued - 2 < 0 ? 0 : issued - 2; it < issued; ++it) {
                const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
                wait_bar(sh, p.status, &sh.rawqk[it & 1], ph, false, kDrainNs);
                wait_bar(sh, p.status, &sh.rawv[it & 1], ph, false, kDrainNs);
            }
        } else if (lane == 1) {
            // -------------------------------------------- TMA producer: g
            int issued = 0;
            for (int it = 0; it < n_loc; ++it) {
                const Item im = item_at<kVarlen>(p, it0 + it);
                const int gs = it % kGBufs;
                const uint32_t gph = static_cast<uint32_t>(it / kGBufs) & 1u;
                if (!wait_bar(sh, p.status, &sh.gempty[gs], gph ^ 1u)) break;
                mbar_arrive_expect_tx(&sh.gfull[gs], HALF);
                tma_load_3d(sm + OFF_GB + gs * HALF, &tg, col0, im.y, im.z, &sh.gfull[gs]);
                LA_TL(2);
                issued = it + 1;
            }
            sh.g_issued = issued;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint64_t dq0 = desc_kmajor(sbase + OFF_QB, 0), dk0 = desc_kmajor(sbase + OFF_KB, 0);
            const uint64_t dkm0 = desc_mnmajor(sbase + OFF_KB, 0);
            const uint64_t dvm0 = desc_mnmajor(sbase + OFF_VB, 0);
            const uint64_t ds0 = desc_mnmajor(sbase + OFF_SB, 0);
            int seen = 0;
            for (int it = 0; it < n_loc; ++it) {
                const int s = it & 1;
                const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
                const uint32_t par = static_cast<uint32_t>(it) & 1u;
                const int yb = it % kYBufs;
                const uint32_t yph = static_cast<uint32_t>(it / kYBufs) & 1u;
                if (!wait_bar(sh, p.status, &sh.actdone[s], ph)) break;
                if (!wait_bar(sh, p.status, &sh.xin[s], ph)) break;
                seen = it + 1;
                LA_TL(7);
                const uint64_t dq = desc_add(dq0, s * TILE), dk = desc_add(dk0, s * TILE);
                const uint64_t dkm = desc_add(dkm0, s * TILE), dvm = desc_add(dvm0, s * HALF);
                const uint32_t tY = tm + TM_Y + yb * DV;
                bool ok = true;
                // scores A = Q^ K^T (128 x 128), once P V^ has read both halves of A
                if (!wait_bar(sh, p.status, &sh.aempty[0], par ^ 1u) ||
                    !wait_bar(sh, p.status, &sh.aempty[1], par ^ 1u))
                    break;
                LA_TL(27);
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tm + TM_A, desc_add(dq, kofs(ks)), desc_add(dk, kofs(ks)), IDESC_QK,
                           ks > 0);
                mma_commit(&sh.afull[0]);
                mma_commit(&sh.afull[1]);
                LA_TL(8);
                if (!wait_bar(sh, p.status, &sh.yempty[yb], yph ^ 1u)) break;
                LA_TL(28);
                if (!wait_bar(sh, p.status, &sh.sready, par)) break;
                LA_TL(29);
                tc_fence_after();
                // Y = Q^ S_{<c}  (this CTA's 64 columns)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tY, desc_add(dq, kofs(ks)), desc_add(ds0, ks * 2048), IDESC_QS, ks > 0);
                // S += K^T V  (fp32 in TMEM)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tm + TM_S, desc_add(dkm, ks * 2048), desc_add(dvm, ks * 2048), IDESC_KV,
                           1u);
                mma_commit(&sh.sdone);
                // q^ and k^ of this stage are no longer read (this CTA and the peer's copy)
                mma_commit_multicast(&sh.qkempty[s], static_cast<uint16_t>(3u));
                LA_TL(9);
                // Y += P_j V^_j, P_j = mask(A_j) in bf16 over the first 32 columns of A_j
                for (int j = 0; j < 2 && ok; ++j) {
                    if (!wait_bar(sh, p.status, &sh.pfull[j], par)) { ok = false; break; }
                    LA_TL(30 + j);
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ts(tY, tm + TM_A + 64 * j + ks * 8,
                               desc_add(dvm, 8192 * j + ks * 2048), IDESC_PV, 1u);
                    mma_commit(&sh.aempty[j]);
                }
                if (!ok) break;
                mma_commit(&sh.yfull[yb]);
                mma_commit(&sh.vempty[s]);
                LA_TL(10);
            }
            sh.xin_seen = seen;
            mma_commit(&sh.mmadone);
            wait_bar(sh, p.status, &sh.mmadone, 0, false, kDrainNs);
        }
    } else if (kAct ? (warp == 2 || warp == 3 || (warp >= 4 && warp < 12 && warp != 5 && warp != 9))
                    : (warp >= 4 && warp < 12)) {
        // ------------------------------------------------ SiLU (two warpgroups): the own
        // tile first (then pushed to the peer), then this CTA's v columns
        // Raw inputs: warps 4-11, two per sub-partition, which balances the SFU work.
        // Activated inputs (the warps only forward tiles): warps 2, 3, 4, 6, 7, 8, 10, 11,
        // none on the MMA warp's sub-partition (3% faster on activated inputs; on raw
        // inputs the uneven SFU load costs more than that).
        const int sidx = !kAct ? warp - 4
                         : warp < 4 ? warp - 2
                         : warp < 9 ? warp - 2 - (warp > 5 ? 1 : 0)
                                    : warp - 4;
        const int u = sidx * 32 + lane;
        const int t = u & 127;     // tile row (token)
        const int part = u >> 7;   // own-tile half; v chunks 4 part .. 4 part + 3
        const bool leader = u == 0;
        const uint32_t peer_own = map_to_rank(sbase + own_off, peer);
        const uint32_t peer_xin = map_to_rank(smem_addr(&sh.xin[0]), peer);
        for (int it = 0; it < n_loc; ++it) {
            const int s = it & 1;
            const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
            if (!group_wait(sh, p.status, &sh.rawqk[s], ph, leader, 1, 256, 0)) break;
            if (leader) LA_TL(3);
            // rows past a packed sequence's end hold the next sequence's tokens and become
            // zero; in a uniform batch the rows past N are already the tensor map's zero
            // fill, and SiLU(0) = 0
            const bool live = !kVarlen || t < p.items[it0 + it].y;
            uint8_t* blk = sm + own_off + s * TILE + part * HALF;
            uint4 x[4];
            if (kAct && live) {
                // already activated: nothing to do
            } else if (live) {
#pragma unroll 1
                for (int g4 = 0; g4 < 2; ++g4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        x[j] = *reinterpret_cast<const uint4*>(blk + swz(t, 4 * g4 + j));
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(blk + swz(t, 4 * g4 + j)) = silu_chunk(x[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(blk + swz(t, j)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (leader) LA_TL(4);
            if (leader)
                bulk_copy_to_peer(peer_own + s * TILE, sbase + own_off + s * TILE, TILE,
                                  peer_xin + s * 8);
            if (!group_wait(sh, p.status, &sh.rawv[s], ph, leader, 1, 256, 0)) break;
            if (leader) LA_TL(5);
            uint8_t* vt = sm + OFF_VB + s * HALF;
            if (kAct && live) {
            } else if (live) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    x[j] = *reinterpret_cast<const uint4*>(vt + swz(t, 4 * part + j));
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(vt + swz(t, 4 * part + j)) = silu_chunk(x[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(vt + swz(t, 4 * part + j)) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (leader) mbar_arrive(&sh.actdone[s]);
            if (leader) LA_TL(6);
        }
    } else if (warp >= 12 && warp < 16) {
        // ------------------------------------------------ state conversion + mask
        const int q4 = warp & 3;
        const int t = q4 * 32 + lane;  // token row (A, P) or d_k row (S)
        const bool leader = t == 0;
        const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
        uint8_t* sbk = sm + OFF_SB;
        for (int it = 0; it <= n_loc; ++it) {
            const Item im = item_at<kVarlen>(p, it0 + (it < n_loc ? it : n_loc - 1));
            // a sequence (or this pair's segment) ends before it, or one starts at it
            const bool first = it == n_loc || it == 0 || im.first;
            // (1) the bf16 operand S_{<c} for iteration it
            if (it > 0) {
                if (!group_wait(sh, p.status, &sh.sdone, static_cast<uint32_t>(it - 1) & 1u,
                                leader, 2, 128, 1))
                    break;
                tc_fence_after();
            }
            if (leader && it < n_loc) LA_TL(11);
            if (first) {
                if (it > 0 && p.S_out && seg == p.nseg - 1) {  // a finished sequence's state
                    const int pb = item_at<kVarlen>(p, it0 + it - 1).b;
                    state_rows_out(p.S_out + ((static_cast<size_t>(pb) * H + h) * D + t) * D +
                                       rank * DV,
                                   lb + TM_S);
                }
                if (it == n_loc) break;
                // segment mode: every segment starts from its prefix state (the first's is
                // a copy of S_in, so nothing reads S_in while the last segment writes S_out)
                const float* src =
                    p.S_seg  ? p.S_seg + ((static_cast<size_t>(seg) * H + h) * D + t) * D
                    : p.S_in ? p.S_in + ((static_cast<size_t>(im.b) * H + h) * D + t) * D
                             : nullptr;
                state_rows_in(src ? src + rank * DV : nullptr, lb + TM_S, sbk, t);
            } else {
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    uint32_t r[32];
                    LA_TMEM_LD32(lb + TM_S + 32 * part, r);
                    tmem_wait_ld();
                    store_row_bf16(sbk, t, part, r);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(2, 128);
            if (leader) mbar_arrive(&sh.sready);
            if (leader) LA_TL(12);
            // (2) P_j = A_j masked to s <= t, bf16, over the first 32 columns of A_j
            bool ok = true;
            for (int j = 0; j < 2; ++j) {
                if (!group_wait(sh, p.status, &sh.afull[j], static_cast<uint32_t>(it) & 1u,
                                leader, 2, 128, 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (leader) LA_TL(13 + 2 * j);
                const uint32_t tA = lb + TM_A + 64 * j;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const int sb0 = 64 * j + 32 * part;  // first key token of these columns
                    uint32_t pk[16];
                    if (sb0 + 31 < q4 * 32) {  // every key of these columns is <= every token
                        uint32_t r[32];
                        LA_TMEM_LD32(tA + 32 * part, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            pk[jj] = pack_bf16x2(__uint_as_float(r[2 * jj]),
                                                 __uint_as_float(r[2 * jj + 1]));
                    } else if (sb0 <= q4 * 32 + 31) {  // the warp's diagonal block
                        uint32_t r[32];
                        LA_TMEM_LD32(tA + 32 * part, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int s0 = sb0 + 2 * jj;
                            const float lo = s0 <= t ? __uint_as_float(r[2 * jj]) : 0.f;
                            const float hi = s0 + 1 <= t ? __uint_as_float(r[2 * jj + 1]) : 0.f;
                            pk[jj] = pack_bf16x2(lo, hi);
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) pk[jj] = 0u;
                    }
                    // columns [16 part, 16 part + 16) of A_j were read in this or an earlier part
                    LA_TMEM_ST16(tA + 16 * part, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                named_bar_sync(2, 128);
                if (leader) mbar_arrive(&sh.pfull[j]);
                if (leader) LA_TL(14 + 2 * j);
            }
            if (!ok) break;
        }
    } else if (warp >= 16 && warp < 20) {
        // ------------------------------------------------ post: this head half's per-token
        // sums of squares into the chunk's slot, then the chunk's counter
        const int q4 = warp & 3;
        const int t = q4 * 32 + lane;  // token row
        const bool leader = t == 0;
        const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
        float* const ring = p.part + static_cast<size_t>(seg) * kPartRing * 2 * H * CH;
        for (int it = 0; it < n_loc; ++it) {
            const int yb = it % kYBufs;
            const uint32_t yph = static_cast<uint32_t>(it / kYBufs) & 1u;
            const int gi = it0 + it;  // the chunk's index in the whole list
            if (it >= kPartRing) {
                // the partials slot is reused: chunk gi - kPartRing's reducer has read it
                // (the y ring makes this long done; the acquire orders the reuse)
                const bool ok =
                    !leader ||
                    spin_published(sh, p.status, p.rn + static_cast<size_t>(gi - kPartRing) * CH);
                if (!named_bar_and(3, 128, ok)) break;
            }
            if (!group_wait(sh, p.status, &sh.yfull[yb], yph, leader, 3, 128, 2)) break;
            if (leader) LA_TL(17);
            tc_fence_after();
            float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint32_t y[32];
                LA_TMEM_LD32(lb + TM_Y + yb * DV + 32 * part, y);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    ss0 = fmaf(__uint_as_float(y[j]), __uint_as_float(y[j]), ss0);
                    ss1 = fmaf(__uint_as_float(y[j + 1]), __uint_as_float(y[j + 1]), ss1);
                }
            }
            __stcg(ring + (static_cast<size_t>(it % kPartRing) * 2 * H + 2 * h + rank) * CH + t,
                   ss0 + ss1);
            named_bar_sync(3, 128);
            if (leader) red_release_gpu_add(p.cnt + gi, 1u);  // orders the group's stores
            if (leader) LA_TL(18);
        }
    } else if (warp >= 20) {
        // ------------------------------------------------ finish: norm, gate, store.  Both
        // groups take every iteration, group fg the columns [32 fg, 32 fg + 32) of y, so a
        // y tile is read (and its TMEM freed) in half the time one group would take.
        const int fg = (warp - 20) >> 2;
        const int q4 = warp & 3;
        const int t = q4 * 32 + lane;     // token row
        const bool leader = t == 0;
        const bool leader2 = leader && fg == 0;  // of both groups
        const uint32_t bar_id = 4 + fg;
        const int slot = 3 + fg;
        const uint32_t lb = tm + (static_cast<uint32_t>(q4 * 32) << 16);
        for (int it = 0; it < n_loc; ++it) {
            const Item im = item_at<kVarlen>(p, it0 + it);
            const int yb = it % kYBufs;
            const uint32_t yph = static_cast<uint32_t>(it / kYBufs) & 1u;
            const int gs = it % kGBufs;
            const uint32_t gph = static_cast<uint32_t>(it / kGBufs) & 1u;
            // r_t, published by the chunk's reducer (re-read, bounded, until written)
            float rn = 0.f;
            bool ready = false;
            {
                const float* src = p.rn + static_cast<size_t>(it0 + it) * CH + t;
                uint64_t t0 = 0;
                for (;;) {
                    rn = __ldcg(src);
                    if (__float_as_uint(rn) != kXchEmpty) {
                        ready = true;
                        break;
                    }
                    if (abort_set(sh)) break;
                    const uint64_t now = global_timer_ns();
                    if (t0 == 0) {
                        t0 = now;
                    } else if (now - t0 > kTimeoutNs) {
                        raise_abort(sh, p.status);
                        break;
                    }
                    __nanosleep(200);
                }
            }
            if (!named_bar_and(bar_id, 128, ready)) break;
            if (leader) LA_TL(19 + 3 * fg);
            // out = y (fp32, TMEM) * r_t * sigmoid(g), written over the g tile, then stored
            if (!group_wait(sh, p.status, &sh.gfull[gs], gph, leader, bar_id, 128, slot)) break;
            if (!group_wait(sh, p.status, &sh.yfull[yb], yph, leader, bar_id, 128, slot)) break;
            if (leader) LA_TL(20 + 3 * fg);
            tc_fence_after();
            uint8_t* gt = sm + OFF_GB + gs * HALF;
            const float hrn = 0.5f * rn;
            const bool valid = t < im.nvalid;
            const size_t grow =
                (static_cast<size_t>(im.z) * p.N + static_cast<size_t>(im.y) + t) * H * D + col0 +
                32 * fg;
            uint32_t y[32];
            LA_TMEM_LD32(lb + TM_Y + yb * DV + 32 * fg, y);
            tmem_wait_ld();
            tc_fence_before();
            named_bar_sync(bar_id, 128);
            if (leader) mbar_arrive(&sh.yempty[yb]);  // this group's half of y is read
            if (p.y_dbg && valid) {
                float4* yp = reinterpret_cast<float4*>(p.y_dbg + grow);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    yp[j] = make_float4(__uint_as_float(y[4 * j]), __uint_as_float(y[4 * j + 1]),
                                        __uint_as_float(y[4 * j + 2]), __uint_as_float(y[4 * j + 3]));
            }
            uint4 gv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                gv[j] = *reinterpret_cast<const uint4*>(gt + swz(t, 4 * fg + j));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t* gw = reinterpret_cast<uint32_t*>(&gv[j]);
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    // y r sigmoid(g) = a + a tanh(g/2) with a = y r / 2
                    const uint32_t hg = half_bf16x2(gw[k2]);
                    const float a0 = __uint_as_float(y[8 * j + 2 * k2]) * hrn;
                    const float a1 = __uint_as_float(y[8 * j + 2 * k2 + 1]) * hrn;
                    gw[k2] = pack_bf16x2(fmaf(a0, tanh_approx(bf_lo(hg)), a0),
                                         fmaf(a1, tanh_approx(bf_hi(hg)), a1));
                }
            }
            if (kVarlen && im.nvalid < CH) {
                // a partial chunk of a packed batch: its last rows are the next sequence's,
                // so only this sequence's rows are stored, each thread its half row from
                // registers.  The g tile is not written: a generic store to it could land
                // after the next TMA load into the same buffer.
                if (valid) {
                    uint4* orow = reinterpret_cast<uint4*>(p.out + grow);
#pragma unroll
                    for (int j = 0; j < 4; ++j) orow[j] = gv[j];
                }
                named_bar_sync(6, 256);  // both groups have read the g tile
                if (leader2) mbar_arrive(&sh.gempty[gs]);
                continue;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(gt + swz(t, 4 * fg + j)) = gv[j];
            fence_proxy_async_smem();
            named_bar_sync(6, 256);  // both halves of the tile are written
            if (leader) LA_TL(21 + 3 * fg);
            if (leader2) {
                tma_store_3d(&to, gt, col0, im.y, im.z);  // rows past N are dropped
                bulk_commit_group();
                bulk_wait_group_read0();  // the tile may take the next g once read
                mbar_arrive(&sh.gempty[gs]);
            }
        }
        if (leader2) bulk_wait_group0();
    }

    // ---------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        // abort paths only: copies that were announced but not consumed land first
        for (int it = sh.xin_seen; it < sh.issued; ++it)
            wait_bar(sh, p.status, &sh.xin[it & 1], static_cast<uint32_t>(it >> 1) & 1u, false,
                     kDrainNs);
        for (int it = sh.g_issued - kGBufs < 0 ? 0 : sh.g_issued - kGBufs; it < sh.g_issued; ++it)
            wait_bar(sh, p.status, &sh.gfull[it % kGBufs],
                     static_cast<uint32_t>(it / kGBufs) & 1u, false, kDrainNs);
    }
    __syncthreads();
    cluster_sync();  // no copy or remote arrival targets a CTA that has left
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
// 64 features x 128 tokens, 128B swizzle; loads past N read zeros, stores past N are
// dropped.
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

template <typename F>
bool set_smem_attr(F* f) {
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_DYN)) == cudaSuccess;
}

int max_active_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    if (g_max_clusters[dev] != 0) return g_max_clusters[dev];
    int n = -1;
    if (set_smem_attr(k_prefill_tc<false, false>) && set_smem_attr(k_prefill_tc<true, false>) &&
        set_smem_attr(k_prefill_tc<false, true>) && set_smem_attr(k_prefill_tc<true, true>)) {
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
        // the fewest co-resident clusters over the four instances
        n = 1 << 30;
        for (const void* f : {reinterpret_cast<const void*>(k_prefill_tc<false, false>),
                              reinterpret_cast<const void*>(k_prefill_tc<true, false>),
                              reinterpret_cast<const void*>(k_prefill_tc<false, true>),
                              reinterpret_cast<const void*>(k_prefill_tc<true, true>)}) {
            if (cudaOccupancyMaxActiveClusters(&m, f, &cfg) != cudaSuccess) {
                n = -1;
                break;
            }
            n = m < n ? m : n;
        }
    }
    cudaGetLastError();
    g_max_clusters[dev] = n > 0 ? n : -1;
    return g_max_clusters[dev];
}

// Flag bank layout for one launch of `total` items: [counters, padded to 4][factors].
size_t flag_cnt_words(int total) { return (static_cast<size_t>(total) + 3) & ~size_t(3); }
size_t flag_words_for(int total) {
    return flag_cnt_words(total) + static_cast<size_t>(total) * CH;
}

// Reducer CTAs for `pairs` head pairs: the clusters left over, at most kMaxReducers / 2.
int reducers_for(int pairs) {
    const int spare = max_active_clusters() - pairs;
    const int clusters = spare < kMaxReducers / 2 ? spare : kMaxReducers / 2;
    return clusters > 0 ? 2 * clusters : 0;
}

}  // namespace

bool encode_io_map_bf16(CUtensorMap* m, const void* base, int B, int H, int64_t N) {
    return encode_io_map(m, base, B, H, N);
}

int prefill_tc_supported(int B, int H, int64_t N) {
    if (N <= 0 || N > (int64_t(1) << 30)) return LA_ERR_UNSUPPORTED;
    const int64_t Nc = (N + CH - 1) / CH;
    if (static_cast<int64_t>(B) * Nc > (int64_t(1) << 30) / CH) return LA_ERR_UNSUPPORTED;
    if (!encoder()) return LA_ERR_UNSUPPORTED;
    // every head's pair and at least one reducer pair must be resident at once
    if (max_active_clusters() <= 0 || reducers_for(H) <= 0) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

size_t prefill_tc_flag_words(int items) { return flag_words_for(items); }

size_t prefill_tc_part_floats(int H, int nseg) {
    return static_cast<size_t>(nseg) * kPartRing * 2 * H * CH;
}

int prefill_tc_segment_plan(int B, int H, int64_t N, int* seg_items, int* fine) {
    *seg_items = 0;
    *fine = 1;
    if (B != 1 || N <= 0) return 1;
    const int64_t Nc = (N + CH - 1) / CH;
    const int clusters = max_active_clusters();
    if (clusters <= 1) return 1;
    // head pairs of all segments plus the reducer pairs resident at once (the full set
    // of kMaxReducers / 2 pairs when that still gives two segments, else one pair), and
    // segments of at least kMinSegChunks chunks
    int64_t nseg = (clusters - kMaxReducers / 2) / H;
    if (nseg < 2) nseg = (clusters - 1) / H;
    if (nseg > Nc / kMinSegChunks) nseg = Nc / kMinSegChunks;
    if (nseg < 2) return 1;
    // the state pass splits each prefix segment into m pieces so that it fills the SMs
    int64_t m = static_cast<int64_t>(2 * clusters) / (static_cast<int64_t>(H) * (nseg - 1));
    if (m < 1) m = 1;
    const int64_t cps = (Nc + nseg * m - 1) / (nseg * m);  // chunks per piece
    const int64_t per = cps * m;                            // chunks per segment
    const int64_t used = (Nc + per - 1) / per;              // non-empty segments
    if (used < 2) return 1;
    *seg_items = static_cast<int>(per);
    *fine = static_cast<int>(m);
    return static_cast<int>(used);
}

int prefill_tc_items(int B, int64_t N) {
    return static_cast<int>(static_cast<int64_t>(B) * ((N + CH - 1) / CH));
}

namespace {

// Launches the kernel over `total` items: B sequences of N tokens (items == nullptr) or
// a packed batch viewed as one slab of N tokens (items: the per-item table on device).
// nseg > 1 (B == 1, uniform): the items are cut into nseg runs of seg_items, each run by
// its own H head pairs from the state S_seg[seg].
int launch_items(const void* q, const void* k, const void* v, const void* g, void* out,
                 const float* S_in, float* S_out, float* y_debug, int B, int H, int64_t N,
                 int total, const int4* items, float eps, bool activated, const Workspace& ws,
                 const XchLease& xl, cudaStream_t st, int nseg = 1, int seg_items = 0,
                 const float* S_seg = nullptr) {
    if (nseg < 1 || (nseg > 1 && (B != 1 || items || !S_seg))) return LA_ERR_INVALID_ARG;
    if (nseg == 1) seg_items = total;
    if (seg_items < 1 || static_cast<int64_t>(nseg - 1) * seg_items >= total)
        return LA_ERR_INVALID_ARG;  // every segment holds at least one item
    const int R = reducers_for(H * nseg);
    if (R <= 0) return LA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv, mg, mo;
    if (!encode_io_map(&mq, q, B, H, N) || !encode_io_map(&mk, k, B, H, N) ||
        !encode_io_map(&mv, v, B, H, N) || !encode_io_map(&mg, g, B, H, N) ||
        !encode_io_map(&mo, out, B, H, N))
        return LA_ERR_UNSUPPORTED;
    Params prm;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.S_in = S_in;
    prm.S_out = S_out;
    prm.y_dbg = y_debug;
    prm.cnt = reinterpret_cast<unsigned*>(xl.use);
    prm.rn = xl.use + flag_cnt_words(total);
    prm.part = xl.part;
    prm.xch_clear = reinterpret_cast<uint4*>(xl.clear);
    prm.n_clear4 = static_cast<int64_t>(xl.clear_words / 4);
    prm.status = ws.status;
    prm.items = items;
    prm.B = B;
    prm.H = H;
    prm.N = N;
    prm.Nc = static_cast<int>((N + CH - 1) / CH);
    prm.nc_magic = ~0ull / static_cast<uint64_t>(prm.Nc);
    prm.total = total;
    prm.nseg = nseg;
    prm.seg_items = seg_items;
    prm.S_seg = S_seg;
    prm.eps = eps;
    prm.inv_width = 1.0f / static_cast<float>(H * D);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * H * nseg + R), 1, 1);
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
    const cudaError_t e =
        items ? (activated
                     ? cudaLaunchKernelEx(&cfg, k_prefill_tc<true, true>, mq, mk, mv, mg, mo, prm)
                     : cudaLaunchKernelEx(&cfg, k_prefill_tc<true, false>, mq, mk, mv, mg, mo,
                                          prm))
              : (activated
                     ? cudaLaunchKernelEx(&cfg, k_prefill_tc<false, true>, mq, mk, mv, mg, mo, prm)
                     : cudaLaunchKernelEx(&cfg, k_prefill_tc<false, false>, mq, mk, mv, mg, mo,
                                          prm));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    xch_commit(xl, flag_words_for(total));
    note_launches(1);
    return LA_OK;
}

}  // namespace

int launch_prefill_tc(const void* q, const void* k, const void* v, const void* g, void* out,
                      const float* S_in, float* S_out, float* y_debug, int B, int H, int64_t N,
                      float eps, bool activated, const Workspace& ws, const XchLease& xl,
                      cudaStream_t st, int nseg, int seg_items, const float* S_seg) {
    const int total = static_cast<int>(static_cast<int64_t>(B) * ((N + CH - 1) / CH));
    return launch_items(q, k, v, g, out, S_in, S_out, y_debug, B, H, N, total, nullptr, eps,
                        activated, ws, xl, st, nseg, seg_items, S_seg);
}

int launch_prefill_tc_varlen(const void* q, const void* k, const void* v, const void* g,
                             void* out, const float* S_in, float* S_out, float* y_debug, int H,
                             int64_t T, int total, const int4* items, float eps,
                             bool activated, const Workspace& ws, const XchLease& xl,
                             cudaStream_t st) {
    return launch_items(q, k, v, g, out, S_in, S_out, y_debug, 1, H, T, total, items, eps,
                        activated, ws, xl, st);
}

}  // namespace la

#ifdef LA_TIMELINE
// Timeline builds only (not part of the public interface): copy the stamps to host
// memory, or zero them.  Return a cudaError_t.
extern "C" int la_timeline_fetch(void* host, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, la::g_la_timeline, bytes));
}
extern "C" int la_timeline_clear() {
    static unsigned long long zeros[la::kTlCtas * la::kTlChunks * la::kTlEvents];
    return static_cast<int>(cudaMemcpyToSymbol(la::g_la_timeline, zeros, sizeof(zeros)));
}
#endif
