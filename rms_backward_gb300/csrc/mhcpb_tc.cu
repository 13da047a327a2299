// Tensor-core streaming kernel of the mHC projection/RMS backward (sm_103a).
//
// What it computes (cuDNN frontend page "DSv4.1 mHC projection/RMS backward",
// intro): for every token t and column k,
//   dX[t,k]          = sum_j P[t,j] W[j,k] + c[t] X[t,k],   c = grad_r / (r K)
//   partial[s][j][k] = sum_{t in chunk s} P[t,j] X[t,k]      (chunk: 512 tokens)
// with P = grad_proj[:, :24] and W rounded to TF32 (nearest, ties away) and
// FP32 accumulation.  The second kernel sums the partials in a fixed order.
//
// How, on GB300:
//  * The grid is persistent (one CTA per SM).  Work items are (128-column
//    strip, token chunk) pairs in strip-major order; a CTA takes a contiguous
//    range of them, so W for a strip is staged once per strip.  The chunking
//    depends only on T, so dW bits are the same on every SM count.
//  * One pipeline stage per 128-token tile, filled by TMA: the X tile
//    (128 x 128 BF16 as two 64-column boxes, 128-byte swizzle, read from HBM
//    exactly once, L2 evict-first), the tile's 24 used grad_proj columns and
//    its grad_r and r (L2 evict-last: every strip re-reads them), and with the
//    fused addend its BF16 addend tile.
//  * Both contractions run on the tensor cores (tcgen05.mma kind::f16, BF16
//    operands, FP32 accumulators in TMEM).  A TF32 value has 11 significant
//    bits, so it is exactly hi + lo with hi, lo BF16 (hi = bf16(v),
//    lo = v - hi).  With P = Ph + Pl and W = Wh + Wl, every product the MMA
//    forms is exact, exactly as a TF32 product would be:
//        dX tile  = [Ph Pl] x [Wh; Wh] + [Ph Pl] x [Wl; Wl]      (M128 N128 K96)
//        dW^T     = X^T x [Ph Pl]   (X used in place, MN-major; M128 N48 K128)
//    X itself is BF16, a subset of TF32, and needs no conversion.
//  * Epilogue warps read the dX accumulator from TMEM (double-buffered loads),
//    add c*X (FP32 FMA, X from the same shared-memory tile), round to BF16
//    (and add the optional BF16 addend the way a separate BF16 add would),
//    write the result over the X tile in place and TMA-store it.  At the end
//    of each chunk they write the chunk's dW partial (hi and lo halves summed)
//    to the workspace.
//  * Warp roles: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2-3 operand
//    preparation (TF32 rounding and BF16 hi/lo split of P and W into the
//    tensor-core operand layout, from shared memory), 4.. epilogue.
//  * Every mbarrier wait is bounded (wait_bar, mhcpb_wait.cuh): on timeout the kernel
//    records a status word, drains its own copies and MMAs and exits.
#include <cuda_bf16.h>

#include "mhcpb_check.cuh"
#include "mhcpb_internal.h"
#include "mhcpb_wait.cuh"
#include "ptx.cuh"

namespace mhcpb {
namespace tc {

namespace {

constexpr int kNJS = 2 * kNProj;                           // 48 split P columns
constexpr uint32_t kXTile = kTokenTile * kStrip * 2;       // 32 KiB of BF16
constexpr uint32_t kBoxBytes = kTokenTile * kBoxCols * 2;  // 16 KiB (one 64-column box)
constexpr uint32_t kPRaw = kTokenTile * kNProj * 4;        // 12 KiB: 128 rows x 24 FP32
constexpr uint32_t kPStage = kTokenTile * kNJS * 2;        // 12 KiB split P
constexpr uint32_t kWBytes = kStrip * 64 * 2;              // 16 KiB (8 blocks of 8 per column group)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDwCol = 256;                           // dW accumulators at 256 and 320
constexpr uint32_t kDwColStride = 64;

// Epilogue warps: one per (TMEM lane quarter, 64-column half of the strip).
constexpr int NEPI = 8;

template <bool ADD>
struct Cfg {
    static constexpr int NS = ADD ? 2 : 4;                 // pipeline stages
    static constexpr int NP = 2;                           // split-P stages
    static constexpr int threads = (4 + NEPI) * 32;
    // stage: X | raw P [128][24] | grad_r[128] | r[128] | addend (1 KiB-aligned parts)
    static constexpr uint32_t st_p = kXTile;
    static constexpr uint32_t st_gr = st_p + kPRaw;
    static constexpr uint32_t st_r = st_gr + kTokenTile * 4;
    static constexpr uint32_t st_add = st_r + kTokenTile * 4;
    static constexpr uint32_t stage_bytes = st_add + (ADD ? kXTile : 0u);
    static constexpr uint32_t off_p = NS * stage_bytes;
    static constexpr uint32_t off_w = off_p + NP * kPStage;
    static constexpr uint32_t off_bar = off_w + kWBytes;
    // barriers: x_full[NS] x_empty[NS] p_full[NP] p_empty[NP] acc_full[2]
    //           acc_empty[2] dw_empty[2] w_full w_empty fin side_full[NS]
    // (no dw_full: an item's dW accumulator is final when its last tile's
    // acc_full completes, which tracks the same MMAs)
    // (side_full: the stage's grad_proj rows, grad_r and r, which come from L2
    // and land well before the X tile, so P is converted while X is in flight)
    static constexpr int B_XF = 0, B_XE = NS, B_PF = 2 * NS, B_PE = 2 * NS + NP;
    static constexpr int B_AF = 2 * NS + 2 * NP, B_AE = B_AF + 2, B_DE = B_AF + 4,
                         B_WF = B_AF + 6, B_WE = B_AF + 7, B_FIN = B_AF + 8;
    static constexpr int B_SF = B_FIN + 1;
    static constexpr uint32_t side_bytes = kPRaw + 2 * kTokenTile * 4;
    static constexpr int n_bars = B_SF + NS;
    static constexpr uint32_t off_misc = off_bar + n_bars * 8;
    static constexpr uint32_t bytes = off_misc + 16;
    static constexpr uint32_t alloc = bytes + 1024;        // room to align the base to 1 KiB
    static_assert(st_add % 1024 == 0, "swizzled addend tile must be 1 KiB aligned");
    static_assert(stage_bytes % 1024 == 0, "stages must stay 1 KiB aligned");
    static_assert(alloc <= 232448, "shared memory budget");
};

// Timeline stamps for instrumented builds (MHCPB_TRACE); nothing otherwise.
#ifdef MHCPB_TRACE
#define TRACE(ev, n)                                                                        \
    do {                                                                                    \
        if (p.trace != nullptr && (n) < kTraceTiles)                                       \
            p.trace[((size_t)blockIdx.x * kTraceEvents + (ev)) * kTraceTiles + (n)] =      \
                ptx::globaltimer();                                                         \
    } while (0)
// the latest of several warps' stamps for one event, with the warp index in
// the low 3 bits (stamp << 3 | warp & 7)
#define TRACE_MAX(ev, n)                                                                    \
    do {                                                                                    \
        if (p.trace != nullptr && (n) < kTraceTiles)                                       \
            atomicMax(reinterpret_cast<unsigned long long*>(                               \
                          &p.trace[((size_t)blockIdx.x * kTraceEvents + (ev)) * kTraceTiles + (n)]), \
                      ((unsigned long long)ptx::globaltimer() << 3) | (unsigned long long)(warp & 7)); \
    } while (0)
#else
#define TRACE(ev, n) \
    do {             \
    } while (0)
#define TRACE_MAX(ev, n) \
    do {                 \
    } while (0)
#endif
enum TraceEvent {
    EV_PROD_ISSUE = 0, EV_MMA_XFULL, EV_MMA_PFULL, EV_MMA_ACCEMPTY, EV_MMA_ISSUED, EV_EPI_ACCFULL,
    EV_EPI_STORED, EV_EPI_RELEASE, EV_PREP_XFULL, EV_PREP_PEMPTY, EV_PREP_DONE, EV_PROD_XEMPTY,
    EV_CTA_START, EV_CTA_END, EV_DRAIN_START, EV_DRAIN_END,   // drains indexed by item
    EV_EPI_ACCFULL_LAST, EV_EPI_STORED_LAST, EV_EPI_RELEASE_LAST   // latest epilogue warp
};

__device__ __forceinline__ float tf32_rna(float v) {
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(v));
    return __uint_as_float(u & 0xFFFFE000u);
}

// TF32 value v -> (hi, lo) BF16 with hi + lo == v exactly (v finite), for two
// values at once, packed as BF16 pairs (first value in the low half):
// hi2 = {bf16(a), bf16(b)}, lo2 = {bf16(a - hi_a), bf16(b - hi_b)}; the
// remainders have at most 4 significant bits, so their rounding is exact.  A
// non-finite value keeps lo = 0 so that Inf stays Inf instead of Inf - Inf.
__device__ __forceinline__ void split_tf32x2(float a, float b, uint32_t& hi2, uint32_t& lo2) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    hi2 = *reinterpret_cast<uint32_t*>(&h);
    float ra = a - __uint_as_float(hi2 << 16);
    float rb = b - __uint_as_float(hi2 & 0xFFFF0000u);
    ra = isfinite(a) ? ra : 0.f;
    rb = isfinite(b) ? rb : 0.f;
    __nv_bfloat162 l = __floats2bfloat162_rn(ra, rb);
    lo2 = *reinterpret_cast<uint32_t*>(&l);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Work-item geometry shared by all roles.  A CTA owns the contiguous range
// [u_begin, u_end) of schedule units: whole items, or (p.half_units) halves of
// items (64 of the strip's 128 columns), in which case its first and last
// item may be half items (hmask 1 or 2).  Splitting an item by columns leaves
// every dW partial's bits unchanged: a column's partial depends only on that
// column's tokens, summed in the same tile order whichever CTA computes it.
struct Item {
    int strip, chunk, col0, t_begin, ntiles;
    uint32_t hmask;   // bit h set: 64-column half h of the strip belongs to this CTA
};
__device__ __forceinline__ Item item_at(const MainParams& p, int it, int u_begin, int u_end) {
    Item r;
    r.strip = it / p.S;
    r.chunk = it - r.strip * p.S;
    r.col0 = r.strip * kStrip;
    r.t_begin = r.chunk * p.chunk;
    const int t_end = min(p.T, r.t_begin + p.chunk);
    r.ntiles = (t_end - r.t_begin + kTokenTile - 1) / kTokenTile;
    r.hmask = !p.half_units ? 3u
                            : (2 * it >= u_begin ? 1u : 0u) | (2 * it + 1 < u_end ? 2u : 0u);
    return r;
}

// Shared-memory operand layouts written by the preparation warp (no swizzle,
// 8-row x 16-byte core matrices of 128 contiguous bytes):
//  P split  [token/8][jb 0..5][token%8][8 BF16]: jb 0,1 = Ph[0..15], 2,3 = Pl[0..15],
//           4 = Ph[16..23], 5 = Pl[16..23].  Read as the K-major A operand of the
//           dX MMA (M = token, K = split column) and as the MN-major B operand of
//           the dW MMA (N = split column, K = token).
//  W split  [col/8][wb 0..7][col%8][8 BF16]: wb 0,1 = Wh[0..15], 2 = 3 = Wh[16..23],
//           4,5 = Wl[0..15], 6 = 7 = Wl[16..23].  K-major B operand of the dX MMA.
// dX k-steps (16 split columns each) pair A blocks {0,2,4,0,2,4} with W blocks
// {0,0,2,4,4,6}: Ph.Wh + Pl.Wh + [Ph Pl]16..23.[Wh Wh] + the same with Wl.
__device__ __forceinline__ uint32_t p_off(int tok, int jb) {
    return (uint32_t)(((tok >> 3) * 6 + jb) * 128 + (tok & 7) * 16);
}
__device__ __forceinline__ uint32_t w_off(int col, int wb) {
    return (uint32_t)(((col >> 3) * 8 + wb) * 128 + (col & 7) * 16);
}

struct Maps {
    CUtensorMap x, dx, add, gp, gr, r;
};

// One 32-column chunk of the dX epilogue for this thread's row: acc (from
// TMEM) + c * x, BF16 rounding, optional BF16 addend, written over x in place.
template <bool ADD>
__device__ __forceinline__ void epi_chunk(const uint32_t (&v)[32], float c, uint8_t* xrow,
                                          const uint8_t* arow, int rr, int sub) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int ch = sub * 4 + i;
        const uint32_t off = (uint32_t)((ch ^ (rr & 7)) << 4);
        const uint4 xv = *reinterpret_cast<const uint4*>(xrow + off);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(xw[e] << 16);
            const float x1 = __uint_as_float(xw[e] & 0xFFFF0000u);
            const float d0 = fmaf(c, x0, __uint_as_float(v[i * 8 + 2 * e]));
            const float d1 = fmaf(c, x1, __uint_as_float(v[i * 8 + 2 * e + 1]));
            o[e] = pack_bf16x2(d0, d1);
        }
        if (ADD) {
            const uint4 av = *reinterpret_cast<const uint4*>(arow + off);
            const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float s0 = __uint_as_float(o[e] << 16) + __uint_as_float(aw[e] << 16);
                const float s1 =
                    __uint_as_float(o[e] & 0xFFFF0000u) + __uint_as_float(aw[e] & 0xFFFF0000u);
                o[e] = pack_bf16x2(s0, s1);
            }
        }
        *reinterpret_cast<uint4*>(xrow + off) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <bool ADD>
__global__ void __launch_bounds__(Cfg<ADD>::threads, 1)
    main_tc_kernel(const MainParams p, const __grid_constant__ Maps maps) {
    using C = Cfg<ADD>;
    constexpr int NS = C::NS, NP = C::NP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::off_misc);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::off_misc + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + C::off_bar + 8u * (uint32_t)i; };

    const int n_items = p.n_strips * p.S;
    const int n_units = p.half_units ? 2 * n_items : n_items;   // gridDim.x <= n_units (host)
    const int u_begin = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_end = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    const int it_begin = p.half_units ? u_begin >> 1 : u_begin;
    const int it_end = p.half_units ? ((u_end - 1) >> 1) + 1 : u_end;

    // Loads of one tile into stage st: side data first (L2-resident, lands
    // early) on its own barrier, then this CTA's 64-column halves of X (and of
    // the addend).  The tensor cores read the whole stage; the accumulator
    // rows/columns of a missing half are never used.
    auto issue_tile = [&](const Item& I, int tt, int st, uint64_t pol_stream, uint64_t pol_keep) {
        const int tok0 = I.t_begin + tt * kTokenTile;
        const uint32_t dst = sbase + (uint32_t)st * C::stage_bytes;
        const uint32_t fb = bar(C::B_XF + st);
        const uint32_t sb = bar(C::B_SF + st);
        ptx::mbar_arrive_expect_tx(sb, C::side_bytes);
        ptx::tma_load_2d(dst + C::st_p, &maps.gp, 0, tok0, sb, pol_keep);
        ptx::tma_load_2d(dst + C::st_gr, &maps.gr, tok0, 0, sb, pol_keep);
        ptx::tma_load_2d(dst + C::st_r, &maps.r, tok0, 0, sb, pol_keep);
        const uint32_t nbox = (I.hmask & 1u) + (I.hmask >> 1);
        ptx::mbar_arrive_expect_tx(fb, nbox * kBoxBytes * (ADD ? 2u : 1u));
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (I.hmask & (1u << h))
                ptx::tma_load_2d(dst + h * kBoxBytes, &maps.x, I.col0 + h * kBoxCols, tok0, fb,
                                 pol_stream);
        if (ADD) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (I.hmask & (1u << h))
                    ptx::tma_load_2d(dst + C::st_add + h * kBoxBytes, &maps.add,
                                     I.col0 + h * kBoxCols, tok0, fb, pol_stream);
        }
    };

    int npre = 0;   // tiles thread 0 (the producer lane) issued before the block-wide sync
    if (threadIdx.x == 0) {
        TRACE(EV_CTA_START, 0);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar(C::B_XF + s), 1);
            ptx::mbar_init(bar(C::B_XE + s), NEPI);
            ptx::mbar_init(bar(C::B_SF + s), 1);
        }
        for (int s = 0; s < NP; ++s) {
            ptx::mbar_init(bar(C::B_PF + s), 2);
            ptx::mbar_init(bar(C::B_PE + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(C::B_AF + b), 1);
            ptx::mbar_init(bar(C::B_AE + b), NEPI);
            ptx::mbar_init(bar(C::B_DE + b), NEPI);
        }
        ptx::mbar_init(bar(C::B_WF), 2);
        ptx::mbar_init(bar(C::B_WE), 1);
        ptx::mbar_init(bar(C::B_FIN), 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&maps.x);
        ptx::prefetch_tensormap(&maps.dx);
        ptx::prefetch_tensormap(&maps.gp);
        ptx::prefetch_tensormap(&maps.gr);
        ptx::prefetch_tensormap(&maps.r);
        if (ADD) ptx::prefetch_tensormap(&maps.add);
        // Launched as a programmatic dependent: everything above touches only
        // shared memory and the kernel parameters; no global memory is read or
        // written before the grids this one depends on have completed.
        ptx::grid_dependency_wait();
        // Fill every stage now (all start empty), so the first loads overlap
        // the TMEM allocation and the block-wide sync below.
        const uint64_t pol_stream = ptx::policy_evict_first();
        const uint64_t pol_keep = ptx::policy_evict_last();
        for (int it = it_begin; it < it_end && npre < NS; ++it) {
            const Item I = item_at(p, it, u_begin, u_end);
            for (int tt = 0; tt < I.ntiles && npre < NS; ++tt, ++npre)
                issue_tile(I, tt, npre, pol_stream, pol_keep);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    ptx::grid_dependency_wait();   // (returns at once: thread 0 waited above)
    ptx::grid_launch_dependents();

    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_stream = ptx::policy_evict_first();
            const uint64_t pol_keep = ptx::policy_evict_last();
            int st = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, last_par = 0;
            bool ok = true;
            int n = 0;   // tile counter of this CTA (trace index)
            for (int it = it_begin; it < it_end && ok; ++it) {
                const Item I = item_at(p, it, u_begin, u_end);
                for (int tt = 0; tt < I.ntiles; ++tt, ++n) {
                    if (n >= npre) {   // the first npre tiles went out before the sync
                        if (!wait_bar(bar(C::B_XE + st), ph ^ 1u, abort_flag, p.status, tmo,
                                      true)) {
                            ok = false;
                            break;
                        }
                        TRACE(EV_PROD_XEMPTY, n);
                        issue_tile(I, tt, st, pol_stream, pol_keep);
                    }
                    TRACE(EV_PROD_ISSUE, n);
                    issued |= 1u << st;
                    last_par = (last_par & ~(1u << st)) | (ph << st);
                    if (++st == NS) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            // drain: every load this thread issued has landed before the CTA exits
            for (int s = 0; s < NS; ++s)
                if (issued & (1u << s)) {
                    wait_bar(bar(C::B_SF + s), (last_par >> s) & 1u, abort_flag, p.status, tmo,
                             false);
                    wait_bar(bar(C::B_XF + s), (last_par >> s) & 1u, abort_flag, p.status, tmo,
                             false);
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_dx = ptx::idesc_bf16_f32(128, kStrip, false, false);
            constexpr uint32_t idesc_dw = ptx::idesc_bf16_f32(128, kNJS, true, true);
            const uint32_t a_blk[6] = {0, 2, 4, 0, 2, 4};
            const uint32_t b_blk[6] = {0, 0, 2, 4, 4, 6};
            const uint32_t w_base = sbase + C::off_w;
            int xs = 0, ps = 0, ab = 0;
            uint32_t xph = 0, pph = 0, aph = 0;
            int n_w = 0, prev_strip = -1, local = 0, n = 0;
            bool ok = true;
            // failure-detection test hook: nothing arrives on the final barrier
            // before the drain below, so this wait can only run out of time
            if (p.test_flags & kTestInjectStall)
                ok = wait_bar(bar(C::B_FIN), 0u, abort_flag, p.status, tmo, true);
            for (int it = it_begin; it < it_end && ok; ++it, ++local) {
                const Item I = item_at(p, it, u_begin, u_end);
                const int db = local & 1;
                const uint32_t dph = (uint32_t)(local >> 1) & 1u;
                if (I.strip != prev_strip) {
                    if (!wait_bar(bar(C::B_WF), (uint32_t)n_w & 1u, abort_flag, p.status, tmo,
                                  true)) {
                        ok = false;
                        break;
                    }
                    ++n_w;
                }
                if (!wait_bar(bar(C::B_DE + db), dph ^ 1u, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                const uint32_t d_dw = tmem + kDwCol + (uint32_t)db * kDwColStride;
                for (int tt = 0; tt < I.ntiles; ++tt, ++n) {
                    if (!wait_bar(bar(C::B_XF + xs), xph, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    TRACE(EV_MMA_XFULL, n);
                    if (!wait_bar(bar(C::B_PF + ps), pph, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    TRACE(EV_MMA_PFULL, n);
                    if (!wait_bar(bar(C::B_AE + ab), aph ^ 1u, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    TRACE(EV_MMA_ACCEMPTY, n);
                    ptx::tc_fence_after();
                    const uint32_t pA = sbase + C::off_p + (uint32_t)ps * kPStage;
                    const uint32_t xA = sbase + (uint32_t)xs * C::stage_bytes;
                    const uint32_t d_dx = tmem + (uint32_t)ab * kStrip;
                    // dX = [Ph Pl](x)[Wh;Wh] + [Ph Pl](x)[Wl;Wl]: M=128 tokens, N=128 cols
#pragma unroll
                    for (int k = 0; k < 6; ++k) {
                        const uint64_t da = ptx::smem_desc(pA + a_blk[k] * 128u, 128u, 768u,
                                                           ptx::kLayoutInterleave);
                        const uint64_t dbd = ptx::smem_desc(w_base + b_blk[k] * 128u, 128u, 1024u,
                                                            ptx::kLayoutInterleave);
                        ptx::mma_bf16(d_dx, da, dbd, idesc_dx, k > 0 ? 1u : 0u);
                    }
                    // dW^T += X^T [Ph Pl]: M=128 cols, N=48, K=128 tokens in 8 steps
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t da = ptx::smem_desc(xA + (uint32_t)k * 2048u, kBoxBytes,
                                                           1024u, ptx::kLayoutSwizzle128B);
                        const uint64_t dbd = ptx::smem_desc(pA + (uint32_t)k * 1536u, 768u, 128u,
                                                            ptx::kLayoutInterleave);
                        ptx::mma_bf16(d_dw, da, dbd, idesc_dw, (tt > 0 || k > 0) ? 1u : 0u);
                    }
                    ptx::tc_commit(bar(C::B_PE + ps));
                    ptx::tc_commit(bar(C::B_AF + ab));
                    TRACE(EV_MMA_ISSUED, n);
                    if (++xs == NS) { xs = 0; xph ^= 1u; }
                    if (++ps == NP) { ps = 0; pph ^= 1u; }
                    if (++ab == 2) { ab = 0; aph ^= 1u; }
                }
                if (!ok) break;
                const int next_strip = (it + 1 < it_end) ? (it + 1) / p.S : -1;
                if (next_strip != I.strip) ptx::tc_commit(bar(C::B_WE));
                prev_strip = I.strip;
            }
            // drain: all MMAs issued by this thread complete before TMEM/smem go away
            ptx::tc_commit(bar(C::B_FIN));
            wait_bar(bar(C::B_FIN), 0u, abort_flag, p.status, tmo, false);
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------------ operand preparation
        // two warps: each converts half of the strip's W columns and half of
        // every tile's tokens; P_FULL and W_FULL complete when both arrived
        const int pw = warp - 2;
        int xs = 0, ps = 0, n = 0;
        uint32_t xph = 0, pph = 0;
        int n_w = 0, prev_strip = -1;
        bool ok = true;
        // W columns of this lane for the next strip to stage.  They are fetched
        // a whole strip ahead (right after the current strip is staged), so a
        // strip change costs no global-memory round trip.
        float wv[2][kNProj];
        auto fetch_w = [&](int col0) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int col = col0 + pw * 64 + lane + 32 * q;
#pragma unroll
                for (int j = 0; j < kNProj; ++j)
                    wv[q][j] = col < p.K && check::in(p.w + (size_t)j * p.K + col, 4, p.w, (size_t)kNProj * p.K * 4, 0)
                                   ? __ldg(p.w + (size_t)j * p.K + col)
                                   : 0.f;
            }
        };
        fetch_w(item_at(p, it_begin, u_begin, u_end).col0);
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item I = item_at(p, it, u_begin, u_end);
            if (I.strip != prev_strip) {
                if (n_w > 0 && !wait_bar(bar(C::B_WE), (uint32_t)(n_w - 1) & 1u, abort_flag,
                                         p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                uint8_t* wsm = smem + C::off_w;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int cc = pw * 64 + lane + 32 * q;
                    uint32_t hw[kNProj / 2], lw[kNProj / 2];   // BF16 pairs (j, j+1)
#pragma unroll
                    for (int k = 0; k < kNProj / 2; ++k)
                        split_tf32x2(tf32_rna(wv[q][2 * k]), tf32_rna(wv[q][2 * k + 1]), hw[k], lw[k]);
                    // blocks: Wh 0-7, Wh 8-15, Wh 16-23 (twice), Wl 0-7, Wl 8-15, Wl 16-23 (twice)
                    const uint32_t* src[8] = {hw, hw + 4, hw + 8, hw + 8, lw, lw + 4, lw + 8, lw + 8};
#pragma unroll
                    for (int wb = 0; wb < 8; ++wb)
                        *reinterpret_cast<uint4*>(wsm + w_off(cc, wb)) =
                            make_uint4(src[wb][0], src[wb][1], src[wb][2], src[wb][3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(C::B_WF));
                ++n_w;
                prev_strip = I.strip;
                // items are strip-major: the next strip of this CTA, if any, starts
                // at item (strip + 1) * S
                if ((I.strip + 1) * p.S < it_end) fetch_w((I.strip + 1) * kStrip);
            }
            for (int tt = 0; tt < I.ntiles; ++tt, ++n) {
                if (!wait_bar(bar(C::B_SF + xs), xph, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                if (pw == 0) TRACE(EV_PREP_XFULL, n);
                if (!wait_bar(bar(C::B_PE + ps), pph ^ 1u, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                if (pw == 0) TRACE(EV_PREP_PEMPTY, n);
                const float* praw = reinterpret_cast<const float*>(smem + (uint32_t)xs * C::stage_bytes + C::st_p);
                uint8_t* psm = smem + C::off_p + ps * kPStage;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int tok = pw * 64 + lane + 32 * i;   // rows past T arrive as zeros (TMA fill)
                    float f[kNProj];
#pragma unroll
                    for (int q = 0; q < 6; ++q) {
                        const float4 v4 = *reinterpret_cast<const float4*>(praw + tok * kNProj + 4 * q);
                        f[4 * q] = v4.x; f[4 * q + 1] = v4.y; f[4 * q + 2] = v4.z; f[4 * q + 3] = v4.w;
                    }
                    uint32_t hw[kNProj / 2], lw[kNProj / 2];   // BF16 pairs (j, j+1)
#pragma unroll
                    for (int k = 0; k < kNProj / 2; ++k)
                        split_tf32x2(tf32_rna(f[2 * k]), tf32_rna(f[2 * k + 1]), hw[k], lw[k]);
                    // blocks: Ph 0-7, Ph 8-15, Pl 0-7, Pl 8-15, Ph 16-23, Pl 16-23
                    const uint32_t* src[6] = {hw, hw + 4, lw, lw + 4, hw + 8, lw + 8};
#pragma unroll
                    for (int jb = 0; jb < 6; ++jb)
                        *reinterpret_cast<uint4*>(psm + p_off(tok, jb)) =
                            make_uint4(src[jb][0], src[jb][1], src[jb][2], src[jb][3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(C::B_PF + ps));
                if (pw == 0) TRACE(EV_PREP_DONE, n);
                if (++xs == NS) { xs = 0; xph ^= 1u; }
                if (++ps == NP) { ps = 0; pph ^= 1u; }
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int e = warp - 4;
        const int q = warp & 3;                  // TMEM lane quarter = token rows 32q..32q+31
        const int h0 = e / 4;                    // the 64-column box of this warp
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int rr = q * 32 + lane;            // row within the token tile
        const float Kf = static_cast<float>(p.K);
        const uint64_t pol = ptx::policy_evict_first();
        const uint64_t pol_keep = ptx::policy_evict_last();   // partials: read back by the reduction
        int xs = 0, ab = 0, local = 0;
        uint32_t xph = 0, aph = 0;
        int n = 0;                               // tile counter (trace index)
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it, ++local) {
            const Item I = item_at(p, it, u_begin, u_end);
            const int db = local & 1;
            // dW partial of this item: this warp's lanes are strip columns
            // 32q..32q+31 (TMEM lane quarter q), i.e. half q / 2 of the strip
            const bool cols_mine = ((I.hmask >> (q >> 1)) & 1u) != 0u;
            const bool lo_part = cols_mine && h0 == 0;   // j 0..15
            const bool hi_part = cols_mine && h0 == 1;   // j 16..23
            const uint32_t dcol = tmem + lane_base + kDwCol + (uint32_t)db * kDwColStride;
            uint32_t d0[16], d1[16], d2[16];
            // Stores this thread's columns of the partial (after the last tile's
            // stage went back to the producer, so they delay no X load).
            auto store_partial = [&]() {
                if (e == 0 && lane == 0) TRACE(EV_DRAIN_START, local);
                const int col = I.col0 + q * 32 + lane;
                if (col < p.K) {
                    const size_t part_bytes = (size_t)p.S * kNProj * p.K * 4;   // checked builds
                    float* dst = p.partial + (size_t)I.chunk * kNProj * p.K + col;
                    // accumulator columns: 0-15 X^T Ph[0..15], 16-31 X^T Pl[0..15],
                    //                      32-39 X^T Ph[16..23], 40-47 X^T Pl[16..23]
                    if (lo_part) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (check::in(dst + (size_t)j * p.K, 4, p.partial, part_bytes, 1))
                                ptx::st_global_hint(dst + (size_t)j * p.K, __uint_as_float(d0[j]) + __uint_as_float(d1[j]), pol_keep);
                    }
                    if (hi_part) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (check::in(dst + (size_t)(16 + i) * p.K, 4, p.partial, part_bytes, 1))
                                ptx::st_global_hint(dst + (size_t)(16 + i) * p.K, __uint_as_float(d2[i]) + __uint_as_float(d2[8 + i]), pol_keep);
                    }
                }
                if (e == 0 && lane == 0) TRACE(EV_DRAIN_END, local);
            };
            for (int tt = 0; tt < I.ntiles; ++tt, ++n) {
                const int tok0 = I.t_begin + tt * kTokenTile;
                const bool last = tt == I.ntiles - 1;
                if (!wait_bar(bar(C::B_SF + xs), xph, abort_flag, p.status, tmo, true) ||
                    !wait_bar(bar(C::B_XF + xs), xph, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                uint8_t* xst = smem + (uint32_t)xs * C::stage_bytes;
                const float gr = reinterpret_cast<const float*>(xst + C::st_gr)[rr];
                const float rv = reinterpret_cast<const float*>(xst + C::st_r)[rr];
                const float c = (tok0 + rr < p.T) ? gr / (rv * Kf) : 0.f;
                if (!wait_bar(bar(C::B_AF + ab), aph, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                if (e == 0 && lane == 0) TRACE(EV_EPI_ACCFULL, n);
                if (lane == 0) TRACE_MAX(EV_EPI_ACCFULL_LAST, n);
                ptx::tc_fence_after();
                if (last) {
                    // the MMAs whose completion ACC_FULL signalled include the item's
                    // last dW MMAs: the dW accumulator is final; read it now, together
                    // with the first dX columns
                    if (lo_part) {
                        ptx::tmem_ld_32x32b_x16(dcol, d0);
                        ptx::tmem_ld_32x32b_x16(dcol + 16, d1);
                    }
                    if (hi_part) ptx::tmem_ld_32x32b_x16(dcol + 32, d2);
                }
                const bool mine = ((I.hmask >> h0) & 1u) != 0u;
                if (!mine) {
                    // none of this warp's dX columns belong to this CTA in this item:
                    // only hand the accumulator(s) and the stage back
                    if (last) {
                        ptx::tc_wait_ld();
                        ptx::reg_fence16(d0);
                        ptx::reg_fence16(d1);
                        ptx::reg_fence16(d2);
                        ptx::tc_fence_before();
                    }
                    __syncwarp();
                    if (lane == 0) {
                        ptx::mbar_arrive(bar(C::B_AE + ab));
                        ptx::mbar_arrive(bar(C::B_XE + xs));
                        if (last) ptx::mbar_arrive(bar(C::B_DE + db));
                    }
                    __syncwarp();
                    if (++xs == NS) { xs = 0; xph ^= 1u; }
                    if (++ab == 2) { ab = 0; aph ^= 1u; }
                    if (last) store_partial();
                    continue;
                }
                const uint32_t tcol = tmem + lane_base + (uint32_t)ab * kStrip + (uint32_t)(h0 * 64);
                uint32_t va[32], vb[32];
                ptx::tmem_ld_32x32b_x32(tcol, va);
                ptx::tc_wait_ld_regs(va);   // (and the dW columns)
                if (last) {
                    ptx::reg_fence16(d0);
                    ptx::reg_fence16(d1);
                    ptx::reg_fence16(d2);
                    // the dW accumulator is in registers: the MMA issuer may reuse it
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(C::B_DE + db));
                }
                constexpr int nch = 2;   // 32-column chunks of this warp
#pragma unroll
                for (int ch = 0; ch < nch; ++ch) {
                    const int h = h0 + (ch >> 1);
                    const int sub = ch & 1;
                    uint8_t* xrow = xst + h * kBoxBytes + rr * 128;
                    const uint8_t* arow = xst + C::st_add + h * kBoxBytes + rr * 128;
                    if (ch + 1 < nch) {
                        if (ch & 1) ptx::tmem_ld_32x32b_x32(tcol + (uint32_t)(ch + 1) * 32, va);
                        else ptx::tmem_ld_32x32b_x32(tcol + (uint32_t)(ch + 1) * 32, vb);
                    } else {
                        // every accumulator column of this warp is in registers:
                        // hand the TMEM buffer back to the MMA issuer
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(C::B_AE + ab));
                    }
                    const bool hv = ((I.hmask >> h) & 1u) != 0u;   // this half is the CTA's
                    if (hv) {
                        if (ch & 1) epi_chunk<ADD>(vb, c, xrow, arow, rr, sub);
                        else epi_chunk<ADD>(va, c, xrow, arow, rr, sub);
                    }
                    if (ch + 1 < nch) {
                        if (ch & 1) ptx::tc_wait_ld_regs(va);
                        else ptx::tc_wait_ld_regs(vb);
                    }
                    if (sub == 1) {
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && hv && tok0 + q * 32 < p.T && I.col0 + h * kBoxCols < p.K)
                            ptx::tma_store_2d(&maps.dx, ptx::smem_u32(xst + h * kBoxBytes + q * 32 * 128),
                                              I.col0 + h * kBoxCols, tok0 + q * 32, pol);
                    }
                }
                if (lane == 0) {
                    ptx::bulk_commit();
                    if (e == 0) TRACE(EV_EPI_STORED, n);
                    TRACE_MAX(EV_EPI_STORED_LAST, n);
                    ptx::bulk_wait_read<0>();          // this tile's stores have read smem
                    ptx::mbar_arrive(bar(C::B_XE + xs));
                    if (e == 0) TRACE(EV_EPI_RELEASE, n);
                    TRACE_MAX(EV_EPI_RELEASE_LAST, n);
                }
                __syncwarp();
                if (++xs == NS) { xs = 0; xph ^= 1u; }
                if (++ab == 2) { ab = 0; aph ^= 1u; }
                if (last) store_partial();
            }
        }
        // every dX store of this warp has read its shared memory (each tile
        // waited for that before releasing its stage); their global writes
        // complete with the grid, so the CTA need not wait for them
        if (lane == 0) ptx::bulk_wait_read<0>();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
        if (lane == 0) TRACE(EV_CTA_END, 0);
    }
}

template <bool ADD>
cudaError_t setup_one() {
    return cudaFuncSetAttribute(main_tc_kernel<ADD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Cfg<ADD>::alloc);
}

template <bool ADD>
cudaError_t launch_one(const MainParams& p, const Maps& m, int grid, cudaStream_t stream) {
    // programmatic dependent launch: the CTAs may be scheduled while the
    // previous kernel in the stream (e.g. the reduction of a previous
    // execute) finishes; they wait for it before touching global memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Cfg<ADD>::threads);
    cfg.dynamicSmemBytes = Cfg<ADD>::alloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, main_tc_kernel<ADD>, p, m);
}

}  // namespace

size_t smem_bytes(bool has_addend) { return has_addend ? Cfg<true>::alloc : Cfg<false>::alloc; }

cudaError_t setup(bool has_addend) { return has_addend ? setup_one<true>() : setup_one<false>(); }

cudaError_t checked_site(uint32_t* site) { return check::read_and_clear(site); }

cudaError_t launch(const MainParams& p, const CUtensorMap& x_map, const CUtensorMap& dx_map,
                   const CUtensorMap& add_map, const CUtensorMap& gp_map, const CUtensorMap& gr_map,
                   const CUtensorMap& r_map, int grid, cudaStream_t stream) {
    Maps m;
    m.x = x_map;
    m.dx = dx_map;
    m.add = add_map;
    m.gp = gp_map;
    m.gr = gr_map;
    m.r = r_map;
    return p.addend != nullptr ? launch_one<true>(p, m, grid, stream) : launch_one<false>(p, m, grid, stream);
}

}  // namespace tc
}  // namespace mhcpb
