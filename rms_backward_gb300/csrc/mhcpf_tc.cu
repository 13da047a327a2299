// Forward of the mHC projection stage on GB300 (sm_103a): in one read of X,
//
//   proj[t, j] = sum_k X[t, k] * W[j, k]        (j < 24; TF32 W, FP32 accumulation)
//   r[t]       = sqrt(sum_k X[t, k]^2 / K + eps)
//
// The prime-kernels PR #15 page describes its mhc_projection as the RMS and
// the projection logits, both from a single pass over X; the backward
// of this stage (cuDNN frontend page "DSv4.1 mHC projection/RMS backward",
// intro) takes the gradients of exactly these two outputs (its dX formula is
// their vector-Jacobian product).  proj is written FP32 [T, 32] with columns
// 24..31 zero, the layout the backward reads its gradient in.
//
// Kernel 1 (persistent, one CTA per SM).  Work unit = (512-column chunk,
// 128-token tile), chunk-major, contiguous unit ranges per CTA, so W of a
// chunk is prepared once per CTA.  Unit boundaries depend only on (T, K):
// proj and r are bitwise the same for every grid size.
//  * warp 0: TMA producer, four 64-column X boxes (128 rows, 128-byte
//    swizzle, 16 KiB each) per pipeline stage on one barrier, two stages, L2
//    evict-first.  One barrier per four boxes rather than per box: the MMA
//    warp's waits and commits, not the pipeline depth, limited this kernel
//    (7 one-box stages 51.8 us per step, 4 two-box stages 49.6, 2 four-box
//    stages 47.5);
//  * warp 1: TMEM allocation and MMA issue.  The X box is used in place as the
//    K-major A operand (M = 128 tokens, K = 64 columns); W of the chunk, split
//    into BF16 hi + lo (a TF32 value is exactly hi + lo, so every product is
//    the TF32 product), is the K-major B operand [Wh; Wl] (N = 48).  The
//    unit's 8 boxes accumulate into one TMEM accumulator (double-buffered
//    across units); proj = D[:, j] + D[:, 24 + j];
//  * warps 2-3: W preparation: each chunk of W is fetched by TMA (FP32) into
//    one of two W slots and converted there in place (TF32 rounding, hi/lo
//    split, 128-byte-swizzled K-major layout; a 64-column box is 6 KiB in
//    either form), so a CTA whose units span two chunks converts the second
//    while the MMAs still use the first (one slot converted after the first
//    chunk's MMAs: 41.2 us for this kernel; two slots: 39.7 us);
//  * warps 4-7: per token row, the sum of squares of the X box from shared
//    memory (eight 8-term partial sums, then their sum: a shallow FP32 sum),
//    and at the end of each unit the drain of the accumulator; they write
//    the unit's partials (24 projections and the sum of squares per token)
//    to the workspace.
// Kernel 2 (one of two layouts, the same bits) sums each token's partials
// over the chunks in ascending order and writes proj and r (programmatic
// dependent launch, like the backward's reduction), then drops the dead
// partial lines from L2.  Every mbarrier wait is bounded (wait_bar).
#include <cuda_bf16.h>

#include "mhcg_math.cuh"
#include "mhcpb_check.cuh"
#include "mhcpb_internal.h"
#include "mhcpb_wait.cuh"
#include "ptx.cuh"

namespace mhcpb {
namespace fwd {

namespace {

constexpr int kBoxes = kChunk / kBox;                 // 8 boxes per unit
constexpr uint32_t kBoxBytes = kTokenTile * kBox * 2;  // 16 KiB
constexpr uint32_t kWBoxBytes = 48 * kBox * 2;         // 6 KiB: [Wh; Wl] rows x 64 columns
constexpr int kBPS = 4;                                // X boxes per pipeline stage (one barrier)
constexpr uint32_t kStageBytes = kBPS * kBoxBytes;     // 64 KiB
constexpr int kNS = 2;                                 // X pipeline stages
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 128;                    // two accumulators of 64 columns
constexpr uint32_t kWRawBox = kNProj * kBox * 4;       // 6 KiB: FP32 W rows x 64 columns
static_assert(kWRawBox == kWBoxBytes, "a W box is converted in place");
constexpr uint32_t kWSlot = kBoxes * kWBoxBytes;       // 48 KiB: one chunk of W
constexpr uint32_t kOffW = kNS * kStageBytes;          // two W slots
constexpr uint32_t kOffBar = kOffW + 2 * kWSlot;
// barriers: x_full[NS] x_empty[NS] acc_full[2] acc_empty[2] w_empty[2] fin w_raw[2] w_full[2][8]
// (per W slot: w_raw, the chunk as stored (FP32) landed by TMA; w_full[b], box
// b converted in place, so the first MMAs of a chunk need not wait for all
// eight boxes; w_empty, the MMAs done with the slot)
constexpr int B_XF = 0, B_XE = kNS, B_AF = 2 * kNS, B_AE = 2 * kNS + 2, B_WE = 2 * kNS + 4,
              B_FIN = 2 * kNS + 6, B_WR = 2 * kNS + 7, B_WF = 2 * kNS + 9,
              kBars = 2 * kNS + 9 + 2 * kBoxes;
constexpr uint32_t kOffMisc = kOffBar + kBars * 8;
constexpr uint32_t kSmem = kOffMisc + 16 + 1024;        // + room to align the base to 1 KiB
static_assert(kSmem <= 232448, "shared memory budget");

// Timeline stamps for instrumented builds (MHCPB_TRACE); nothing otherwise.
#ifdef MHCPB_TRACE
#define FTRACE(ev, n)                                                                       \
    do {                                                                                    \
        if (p.trace != nullptr && (n) < kTraceTiles)                                       \
            p.trace[((size_t)blockIdx.x * kTraceEvents + (ev)) * kTraceTiles + (n)] =      \
                ptx::globaltimer();                                                         \
    } while (0)
#else
#define FTRACE(ev, n) \
    do {              \
    } while (0)
#endif
enum FwdTraceEvent {
    F_PROD_ISSUE = 0, F_MMA_XFULL, F_MMA_COMMIT, F_SS_XFULL, F_SS_DONE, F_PROD_XEMPTY,
    F_W_READY, F_DRAIN_START, F_DRAIN_END, F_CTA_START, F_CTA_END   // boxes; W by chunk; drains by unit
};

struct Unit {
    int fc, tt, nb;   // chunk, token tile, boxes inside K
};
__device__ __forceinline__ Unit unit_at(const FwdParams& p, int u) {
    Unit r;
    r.fc = u / p.n_tt;
    r.tt = u - r.fc * p.n_tt;
    const int rem = p.K - r.fc * kChunk;
    r.nb = min(kBoxes, (rem + kBox - 1) / kBox);
    return r;
}

__device__ __forceinline__ float tf32_rna(float v) {
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(v));
    return __uint_as_float(u & 0xFFFFE000u);
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap xmap,
                  const __grid_constant__ CUtensorMap wmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };

    const int n_units = p.n_fc * p.n_tt;   // gridDim.x <= n_units (host)
    const int u_begin = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_end = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    const uint64_t tmo = p.timeout_ns;
    // one chunk of W as stored (eight 64-column FP32 boxes, zero past K) into
    // W slot `slot`, L2 evict-last: every token tile re-reads W
    auto fetch_raw_w = [&](int fc, int slot) {
        const uint64_t pol_keep = ptx::policy_evict_last();
        ptx::mbar_arrive_expect_tx(bar(B_WR + slot), kBoxes * kWRawBox);
        for (int b = 0; b < kBoxes; ++b)
            ptx::tma_load_2d(sbase + kOffW + (uint32_t)slot * kWSlot + (uint32_t)b * kWRawBox, &wmap,
                             fc * kChunk + b * kBox, 0, bar(B_WR + slot), pol_keep);
    };

    if (threadIdx.x == 0) {
        FTRACE(F_CTA_START, 0);
        for (int s = 0; s < kNS; ++s) {
            ptx::mbar_init(bar(B_XF + s), 1);
            ptx::mbar_init(bar(B_XE + s), 1 + 4);   // the MMAs' commit + 4 sum-of-squares warps
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(B_AF + b), 1);
            ptx::mbar_init(bar(B_AE + b), 4);
        }
        for (int b = 0; b < 2 * kBoxes; ++b) ptx::mbar_init(bar(B_WF + b), 1);   // the converting warp
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(B_WE + s), 1);
            ptx::mbar_init(bar(B_WR + s), 1);
        }
        ptx::mbar_init(bar(B_FIN), 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&xmap);
        ptx::prefetch_tensormap(&wmap);
        // Launched as a programmatic dependent: no global memory is touched
        // before the grids this one depends on have completed.
        ptx::grid_dependency_wait();
        // the first chunk of W goes out before any X load: the MMAs cannot start
        // (nor release a stage) before it is converted
        if (u_begin < u_end) fetch_raw_w(unit_at(p, u_begin).fc, 0);
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

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol = ptx::policy_evict_first();
            int st = 0, n = 0;
            uint32_t ph = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int u = u_begin; u < u_end && ok; ++u) {
                const Unit U = unit_at(p, u);
                for (int b = 0; b < U.nb; b += kBPS, ++n) {
                    const int nbx = min(kBPS, U.nb - b);
                    if (n >= kNS &&
                        !wait_bar(bar(B_XE + st), ph ^ 1u, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    FTRACE(F_PROD_XEMPTY, n);
                    ptx::mbar_arrive_expect_tx(bar(B_XF + st), (uint32_t)nbx * kBoxBytes);
                    for (int i = 0; i < nbx; ++i)
                        ptx::tma_load_2d(sbase + (uint32_t)st * kStageBytes + (uint32_t)i * kBoxBytes, &xmap,
                                         U.fc * kChunk + (b + i) * kBox, U.tt * kTokenTile, bar(B_XF + st), pol);
                    FTRACE(F_PROD_ISSUE, n);
                    issued |= 1u << st;
                    last_par = (last_par & ~(1u << st)) | (ph << st);
                    if (++st == kNS) { st = 0; ph ^= 1u; }
                }
            }
            for (int s = 0; s < kNS; ++s)   // every load has landed before the CTA exits
                if (issued & (1u << s))
                    wait_bar(bar(B_XF + s), (last_par >> s) & 1u, abort_flag, p.status, tmo, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 48, false, false);
            int st = 0, ab = 0, n_w = 0, prev_fc = -1, n = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int u = u_begin; u < u_end && ok; ++u) {
                const Unit U = unit_at(p, u);
                const bool new_chunk = U.fc != prev_fc;   // W boxes: wait for each as it is needed
                if (new_chunk) {
                    ++n_w;
                    prev_fc = U.fc;
                }
                if (!wait_bar(bar(B_AE + ab), aph ^ 1u, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                const uint32_t d = tmem + (uint32_t)ab * 64u;
                const int wslot = (n_w - 1) & 1;   // chunk m of this CTA sits in slot m % 2
                const uint32_t w_base = sbase + kOffW + (uint32_t)wslot * kWSlot;
                for (int b = 0; b < U.nb; b += kBPS, ++n) {
                    const int nbx = min(kBPS, U.nb - b);
                    for (int i = 0; i < nbx && ok; ++i)
                        if (new_chunk && !wait_bar(bar(B_WF + wslot * kBoxes + b + i),
                                                   (uint32_t)((n_w - 1) >> 1) & 1u, abort_flag, p.status,
                                                   tmo, true))
                            ok = false;
                    if (!ok || !wait_bar(bar(B_XF + st), ph, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    FTRACE(F_MMA_XFULL, n);
                    ptx::tc_fence_after();
                    for (int i = 0; i < nbx; ++i) {
                        const uint32_t xa = sbase + (uint32_t)st * kStageBytes + (uint32_t)i * kBoxBytes;
                        const uint32_t wb = w_base + (uint32_t)(b + i) * kWBoxBytes;
                        // four K = 16 steps inside the 128-byte swizzle atom: +32 bytes each
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t da = ptx::smem_desc(xa + 32u * k, 16u, 1024u, ptx::kLayoutSwizzle128B);
                            const uint64_t db = ptx::smem_desc(wb + 32u * k, 16u, 1024u, ptx::kLayoutSwizzle128B);
                            ptx::mma_bf16(d, da, db, idesc, (b + i > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    ptx::tc_commit(bar(B_XE + st));
                    FTRACE(F_MMA_COMMIT, n);
                    if (++st == kNS) { st = 0; ph ^= 1u; }
                }
                if (!ok) break;
                ptx::tc_commit(bar(B_AF + ab));
                const bool next_fc_differs = (u + 1 >= u_end) || unit_at(p, u + 1).fc != U.fc;
                if (next_fc_differs) ptx::tc_commit(bar(B_WE + wslot));
                if (++ab == 2) { ab = 0; aph ^= 1u; }
            }
            ptx::tc_commit(bar(B_FIN));   // all MMAs complete before TMEM is freed
            wait_bar(bar(B_FIN), 0u, abort_flag, p.status, tmo, false);
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------- W preparation
        // Chunk m of this CTA's W goes to slot m % 2, arrives raw (FP32) by TMA
        // and is converted in place: a 64-column box is 6 KiB both as FP32 rows
        // and as the swizzled BF16 hi/lo operand.  Warp 2 converts the even
        // boxes, warp 3 the odd ones, each box read whole into registers before
        // it is overwritten.  Chunk 0 was fetched by thread 0 before the
        // block-wide sync, chunk 1 is fetched once chunk 0 is converted, chunk
        // m + 1 (m >= 1) once the MMAs of chunk m - 1 have left its slot; so a
        // chunk is converted while the MMAs still work on the previous one.
        const bool fetcher = warp == 2 && lane == 0;
        const int wq = warp - 2;   // boxes wq, wq + 2, ...
        int n_chunks = 0, fc_first = 0;
        if (u_begin < u_end) {
            fc_first = unit_at(p, u_begin).fc;
            n_chunks = unit_at(p, u_end - 1).fc - fc_first + 1;   // units are chunk-major
        }
        int n_raw = n_chunks > 0 ? 1 : 0;
        bool ok = true;
        int m = 0;
        for (; m < n_chunks && ok; ++m) {
            const int slot = m & 1;
            if (!wait_bar(bar(B_WR + slot), (uint32_t)(m >> 1) & 1u, abort_flag, p.status, tmo, true)) {
                ok = false;
                break;
            }
            uint8_t* wsm = smem + kOffW + (uint32_t)slot * kWSlot;
            for (int b = wq; b < kBoxes; b += 2) {
                uint8_t* box = wsm + b * kWBoxBytes;
                // 24 rows x 16 float4 = 384 float4, twelve per lane: all read first
                float4 v4[kNProj * (kBox / 4) / 32];
#pragma unroll
                for (int k = 0; k < kNProj * (kBox / 4) / 32; ++k)
                    v4[k] = reinterpret_cast<const float4*>(box)[lane + 32 * k];
                __syncwarp();
#pragma unroll
                for (int k = 0; k < kNProj * (kBox / 4) / 32; ++k) {
                    const int rem = lane + 32 * k;
                    const int j = rem >> 4, c4 = rem & 15;   // row, group of 4 columns
                    const float v[4] = {tf32_rna(v4[k].x), tf32_rna(v4[k].y), tf32_rna(v4[k].z),
                                        tf32_rna(v4[k].w)};
                    uint32_t hi[2], lo[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                        hi[e] = *reinterpret_cast<const uint32_t*>(&h);
                        const float r0 = isfinite(v[2 * e]) ? v[2 * e] - __low2float(h) : 0.f;
                        const float r1 = isfinite(v[2 * e + 1]) ? v[2 * e + 1] - __high2float(h) : 0.f;
                        const __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
                        lo[e] = *reinterpret_cast<const uint32_t*>(&l);
                    }
                    // 128-byte swizzle: 16-byte chunk c of row n sits at chunk c ^ (n & 7);
                    // four columns are 8 bytes, half a chunk
                    const int c16 = c4 >> 1, half = (c4 & 1) * 8;
                    const int nh = j, nl = kNProj + j;
                    *reinterpret_cast<uint2*>(box + nh * 128 + ((c16 ^ (nh & 7)) << 4) + half) = make_uint2(hi[0], hi[1]);
                    *reinterpret_cast<uint2*>(box + nl * 128 + ((c16 ^ (nl & 7)) << 4) + half) = make_uint2(lo[0], lo[1]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(B_WF + slot * kBoxes + b));
            }
            if (fetcher) FTRACE(F_W_READY, m);
            // chunk 1 is fetched only once chunk 0 is converted, not at the
            // start: then the first X boxes land without it in the way (at
            // K = 20480, T = 4096 the call is ~0.35 us faster)
            if (fetcher && m == 0 && n_chunks > 1) {
                fetch_raw_w(fc_first + 1, 1);
                n_raw = 2;
            }
            // chunk m + 1 goes to slot (m + 1) % 2 once the MMAs of chunk m - 1
            // (which also proves that chunk's conversion finished) have left it
            if (fetcher && m >= 1 && m + 1 < n_chunks) {
                const int ns = (m + 1) & 1;
                if (!wait_bar(bar(B_WE + ns), (uint32_t)((m - 1) >> 1) & 1u, abort_flag, p.status, tmo,
                              true)) {
                    ok = false;
                } else {
                    fetch_raw_w(fc_first + m + 1, ns);
                    n_raw = m + 2;
                }
            }
            __syncwarp();
        }
        // every raw W fetch has landed before the CTA exits
        if (fetcher)
            for (int c = m; c < n_raw; ++c)
                wait_bar(bar(B_WR + (c & 1)), (uint32_t)(c >> 1) & 1u, abort_flag, p.status, tmo, false);
        __syncwarp();
    } else {
        // ---------------------------------------------------------- sum of squares, drain
        const int q = warp & 3;                    // TMEM lane quarter = token rows 32q..32q+31
        const int rr = q * 32 + lane;              // row within the token tile
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const uint64_t pol_keep = ptx::policy_evict_last();
        int st = 0, ab = 0, n = 0, un = 0;
        uint32_t ph = 0, aph = 0;
        bool ok = true;
        for (int u = u_begin; u < u_end && ok; ++u, ++un) {
            const Unit U = unit_at(p, u);
            float ss = 0.f;
            for (int b0 = 0; b0 < U.nb; b0 += kBPS, ++n) {
                if (!wait_bar(bar(B_XF + st), ph, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                if (q == 0 && lane == 0) FTRACE(F_SS_XFULL, n);
                for (int i = 0; i < min(kBPS, U.nb - b0); ++i) {
                    const uint8_t* row = smem + (uint32_t)st * kStageBytes + (uint32_t)i * kBoxBytes + rr * 128;
                    float part[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (rr & 7)) << 4));
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                        float a = 0.f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = __uint_as_float(w4[e] << 16);
                            const float x1 = __uint_as_float(w4[e] & 0xFFFF0000u);
                            a = fmaf(x0, x0, a);
                            a = fmaf(x1, x1, a);
                        }
                        part[c] = a;
                    }
                    ss += ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(B_XE + st));
                if (q == 0 && lane == 0) FTRACE(F_SS_DONE, n);
                if (++st == kNS) { st = 0; ph ^= 1u; }
            }
            if (!ok) break;
            if (q == 0 && lane == 0) FTRACE(F_DRAIN_START, un);
            if (!wait_bar(bar(B_AF + ab), aph, abort_flag, p.status, tmo, true)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t d0[16], d1[16], d2[16];
            const uint32_t dcol = tmem + lane_base + (uint32_t)ab * 64u;
            ptx::tmem_ld_32x32b_x16(dcol, d0);        // X Wh^T, j 0..15
            ptx::tmem_ld_32x32b_x16(dcol + 16, d1);   // j 16..23, then X Wl^T j 0..7
            ptx::tmem_ld_32x32b_x16(dcol + 32, d2);   // X Wl^T j 8..23
            ptx::tc_wait_ld();
            ptx::reg_fence16(d0);
            ptx::reg_fence16(d1);
            ptx::reg_fence16(d2);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_AE + ab));
            const int t = U.tt * kTokenTile + rr;
            if (t < p.T) {
                // partial[fc][j][t] (token-contiguous rows: a warp writes 128 bytes per j)
                float* dst = p.partial + (size_t)U.fc * kPartRows * p.t_pad + t;
#pragma unroll
                const size_t part_bytes = (size_t)p.n_fc * kPartRows * p.t_pad * 4;   // checked builds
                for (int j = 0; j < kNProj; ++j) {
                    const float hi = __uint_as_float(j < 16 ? d0[j] : d1[j - 16]);
                    const float lo = __uint_as_float(j < 8 ? d1[8 + j] : d2[j - 8]);
                    if (check::in(dst + (size_t)j * p.t_pad, 4, p.partial, part_bytes, 0))
                        ptx::st_global_hint(dst + (size_t)j * p.t_pad, hi + lo, pol_keep);
                }
                if (check::in(dst + (size_t)kNProj * p.t_pad, 4, p.partial, part_bytes, 0))
                    ptx::st_global_hint(dst + (size_t)kNProj * p.t_pad, ss, pol_keep);
            }
            if (q == 0 && lane == 0) FTRACE(F_DRAIN_END, un);
            if (++ab == 2) { ab = 0; aph ^= 1u; }
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
        if (lane == 0) FTRACE(F_CTA_END, 0);
    }
}

// proj[t][j] = sum over chunks ascending of partial[fc][j][t]; r from the
// summed squares.  Two kernels with the same sums in the same order (so the
// same bits), chosen per call by the number of 32-token blocks:
//  * lines (at most one block per SM): block = 32 tokens, warp j' sums
//    partial row j' (lane = token, each load one 128-byte line), and the sums
//    leave through shared memory as whole proj rows (a token's 32 floats are
//    one 128-byte line).  64 registers x 800 threads: one block per SM.  With
//    the gate step fused in (mhcpb_forward_gates) it also runs the gates on
//    the sums, and is then taken at every T;
//  * outputs (more blocks than SMs): thread = (row j', token t), 256-thread
//    blocks, several per SM.  Its warps write 4-byte pieces of 32 proj rows
//    each, which costs ~1.7 us per call at T = 4096; but it keeps more loads
//    in flight per SM, and at T = 16384 it is ~1.7 us faster than lines in
//    3.4 waves.
constexpr int kGroup = 40;   // chunk partials loaded before they are summed (all of them at K = 20480)
constexpr int kLineTokens = 32;
constexpr int kLineThreads = kPartRows * 32;   // 800
constexpr int kOutThreads = 256;

// the ascending-order sum over the chunks of one partial element (src points
// at chunk 0; stride floats per chunk), every group's loads in flight together
__device__ __forceinline__ float sum_chunks(const float* src, int64_t stride, int n_fc, const float* part) {
    float a = 0.f;
    for (int f0 = 0; f0 < n_fc; f0 += kGroup) {
        float b[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g)
            if (f0 + g < n_fc && check::in(src + (int64_t)(f0 + g) * stride, 4, part, (size_t)n_fc * stride * 4, 1))
                b[g] = src[(int64_t)(f0 + g) * stride];
#pragma unroll
        for (int g = 0; g < kGroup; ++g)
            if (f0 + g < n_fc) a = (f0 + g == 0) ? b[g] : a + b[g];
    }
    return a;
}

template <bool GATES>
__global__ void __launch_bounds__(kLineThreads)
    fwd_reduce_lines_kernel(const float* __restrict__ part, float* __restrict__ proj,
                            float* __restrict__ r, int T, int t_pad, int n_fc, float kf, float eps,
                            int discard, GateArgs g) {
    __shared__ float sums[kPartRows][kLineTokens + 1];
    ptx::grid_launch_dependents();   // the next forward's kernel 1 may be scheduled
    ptx::grid_dependency_wait();
    const int row = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kLineTokens;   // gridDim.x = t_pad / 32: t0 + lane < t_pad
    const int64_t stride = (int64_t)kPartRows * t_pad;   // floats per chunk
    const float* src = part + (int64_t)row * t_pad + t0;
    sums[row][lane] = sum_chunks(src + lane, stride, n_fc, part);
    // the partials are dead once read: drop the warp's line of every chunk
    // from L2, spread over the lanes
    __syncwarp();
    if (discard)
        for (int f = lane; f < n_fc; f += 32)
            if (check::in(src + (int64_t)f * stride, 128, part, (size_t)n_fc * stride * 4, 4))
                ptx::discard_l2_line(src + (int64_t)f * stride);
    __syncthreads();
    if (threadIdx.x < kLineTokens * kProjCols / 4) {
        // 32 proj rows x 8 float4: columns 24..31 are the zero pad
        const int tt = threadIdx.x >> 3, c = (threadIdx.x & 7) * 4;
        const int t = t0 + tt;
        if (t < T) {
            float4 v;
            v.x = c + 0 < kNProj ? sums[c + 0][tt] : 0.f;
            v.y = c + 1 < kNProj ? sums[c + 1][tt] : 0.f;
            v.z = c + 2 < kNProj ? sums[c + 2][tt] : 0.f;
            v.w = c + 3 < kNProj ? sums[c + 3][tt] : 0.f;
            if (check::in(proj + (size_t)t * kProjCols + c, 16, proj, (size_t)T * kProjCols * 4, 2))
                *reinterpret_cast<float4*>(proj + (size_t)t * kProjCols + c) = v;
        }
    } else if (threadIdx.x < kLineTokens * kProjCols / 4 + kLineTokens) {
        const int tt = threadIdx.x - kLineTokens * kProjCols / 4;
        const int t = t0 + tt;
        if (t < T && check::in(r + t, 4, r, (size_t)T * 4, 3))
            r[t] = sqrtf(sums[kNProj][tt] / kf + eps);   // the mean of the squares, eps, root
    }
    if (GATES && threadIdx.x < kLineTokens * 16) {
        // the gate step on the values just stored: a half-warp per token,
        // token pairs per warp as in the gate kernels, and a token past T
        // given the gate kernels' inputs for it (r = 1, projections 0), so
        // every warp-wide choice and so every bit is the same as
        // mhcpb_gate_forward on the stored proj and r
        const int tt = threadIdx.x >> 4, l = threadIdx.x & 15;
        const int t = t0 + tt;
        const bool valid = t < T;
        const float rv = valid ? sqrtf(sums[kNProj][tt] / kf + eps) : 1.f;
        const float pres = valid ? sums[8 + l][tt] : 0.f;
        const float M = gatemath::sinkhorn(gatemath::res_logit(pres, rv, g.alpha, g.bias, l), g.n_iter, nullptr,
                                           nullptr, 0);
        if (valid) {
            const size_t h_bytes = (size_t)T * kNProj * 4;   // checked builds
            float* ht = g.h + (size_t)t * kNProj;
            if (check::in(ht + 8 + l, 4, g.h, h_bytes, 5)) ht[8 + l] = M;
            if (l < 8) {
                const float gv = gatemath::pre_post_gate(sums[l][tt], rv, g.alpha, g.bias, l);
                if (check::in(ht + l, 4, g.h, h_bytes, 5)) ht[l] = gv;
            }
        }
    }
}

__global__ void __launch_bounds__(kOutThreads)
    fwd_reduce_outputs_kernel(const float* __restrict__ part, float* __restrict__ proj,
                              float* __restrict__ r, int T, int t_pad, int n_fc, float kf,
                              float eps, int discard) {
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    const int64_t i = (int64_t)blockIdx.x * kOutThreads + threadIdx.x;
    const bool valid = i < (int64_t)kPartRows * t_pad;   // t_pad % 32 == 0: whole warps
    const int row = valid ? (int)(i / t_pad) : 0;       // j' (24 = sum of squares)
    const int t = valid ? (int)(i - (int64_t)row * t_pad) : 0;
    const int64_t stride = (int64_t)kPartRows * t_pad;
    const int64_t base = (int64_t)row * t_pad + t;
    const float a = valid ? sum_chunks(part + base, stride, n_fc, part) : 0.f;
    if (valid && t < T) {
        const size_t proj_bytes = (size_t)T * kProjCols * 4;   // checked builds
        if (row < kNProj) {
            if (check::in(proj + (size_t)t * kProjCols + row, 4, proj, proj_bytes, 2))
                proj[(size_t)t * kProjCols + row] = a;
        } else {
            if (check::in(r + t, 4, r, (size_t)T * 4, 3)) r[t] = sqrtf(a / kf + eps);
            float4* pad = reinterpret_cast<float4*>(proj + (size_t)t * kProjCols + kNProj);
            if (check::in(pad, 32, proj, proj_bytes, 2)) {
                pad[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                pad[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    // the warp's line of each chunk (32 tokens of one row), spread over the lanes
    __syncwarp();
    if (valid && discard) {
        const int64_t b0 = base - (t & 31);
        for (int f = t & 31; f < n_fc; f += 32)
            if (check::in(part + (int64_t)f * stride + b0, 128, part, (size_t)n_fc * stride * 4, 4))
                ptx::discard_l2_line(part + (int64_t)f * stride + b0);
    }
}

}  // namespace

size_t smem_bytes() { return kSmem; }

cudaError_t checked_site(uint32_t* site) { return check::read_and_clear(site); }

cudaError_t setup() {
    return cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
}

cudaError_t launch(const FwdParams& p, const CUtensorMap& x_map, const CUtensorMap& w_map, int grid,
                   cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1, cudaEvent_t ev2,
                   const GateArgs* gates) {
    cudaError_t e;
    if (ev0 && (e = cudaEventRecord(ev0, stream)) != cudaSuccess) return e;
    {
        // programmatic dependent launch, as for the backward's streaming kernel
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, fwd_tc_kernel, p, x_map, w_map)) != cudaSuccess) return e;
    }
    if (ev1 && (e = cudaEventRecord(ev1, stream)) != cudaSuccess) return e;
    // discard needs 128-byte lines: t_pad is a multiple of 32 floats
    const int discard = (reinterpret_cast<uintptr_t>(p.partial) & 127u) == 0 ? 1 : 0;
    // one wave of line blocks (kernel 1's grid is the SM count unless the
    // problem has fewer units, or a cap lowers it), else the output threads;
    // the gates need a token's sums together: always lines
    const bool lines = gates != nullptr || p.t_pad / kLineTokens <= grid;
    const GateArgs g = gates != nullptr ? *gates : GateArgs{nullptr, nullptr, 0, nullptr};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = lines ? dim3((unsigned)(p.t_pad / kLineTokens))
                        : dim3((unsigned)(((int64_t)kPartRows * p.t_pad + kOutThreads - 1) / kOutThreads));
    cfg.blockDim = dim3(lines ? kLineThreads : kOutThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* part = p.partial;
    if (gates != nullptr)
        e = cudaLaunchKernelEx(&cfg, fwd_reduce_lines_kernel<true>, part, p.proj, p.r, p.T, p.t_pad, p.n_fc,
                               (float)p.K, p.eps, discard, g);
    else if (lines)
        e = cudaLaunchKernelEx(&cfg, fwd_reduce_lines_kernel<false>, part, p.proj, p.r, p.T, p.t_pad, p.n_fc,
                               (float)p.K, p.eps, discard, g);
    else
        e = cudaLaunchKernelEx(&cfg, fwd_reduce_outputs_kernel, part, p.proj, p.r, p.T, p.t_pad, p.n_fc,
                               (float)p.K, p.eps, discard);
    if (e != cudaSuccess) return e;
    if (ev2 && (e = cudaEventRecord(ev2, stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace fwd
}  // namespace mhcpb
