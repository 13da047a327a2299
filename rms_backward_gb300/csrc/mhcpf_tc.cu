// Forward of the mHC projection stage on GB300 (sm_103a): in one read of X,
//
//   proj[t, j] = sum_k X[t, k] * W[j, k]        (j < 24; TF32 W, FP32 accumulation)
//   r[t]       = sqrt(sum_k X[t, k]^2 / K + eps)
//
// The prime-kernels PR #15 page describes its mhc_projection as the RMS and
// the projection logits computed in one read of the streams; the backward
// of this stage (cuDNN frontend page "DSv4.1 mHC projection/RMS backward",
// intro) takes the gradients of exactly these two outputs (its dX formula is
// their vector-Jacobian product).  proj is written FP32 [T, 32] with columns
// 24..31 zero, the layout the backward reads its gradient in.
//
// Kernel 1 (persistent, one CTA per SM).  Work unit = (512-column chunk,
// 128-token tile), chunk-major, contiguous unit ranges per CTA, so W of a
// chunk is prepared once per CTA.  Unit boundaries depend only on (T, K):
// proj and r are bitwise the same for every grid size.
//  * warp 0: TMA producer, one 64-column X box (128 rows, 128-byte swizzle,
//    16 KiB) per pipeline stage, L2 evict-first;
//  * warp 1: TMEM allocation and MMA issue.  The X box is used in place as the
//    K-major A operand (M = 128 tokens, K = 64 columns); W of the chunk, split
//    into BF16 hi + lo (a TF32 value is exactly hi + lo, so every product is
//    the TF32 product), is the K-major B operand [Wh; Wl] (N = 48).  The
//    unit's 8 boxes accumulate into one TMEM accumulator (double-buffered
//    across units); proj = D[:, j] + D[:, 24 + j];
//  * warps 2-3: W preparation (TF32 rounding, hi/lo split, 128-byte-swizzled
//    K-major layout);
//  * warps 4-7: per token row, the sum of squares of the X box from shared
//    memory (eight 8-term partial sums, then their sum: a shallow FP32 sum),
//    and at the end of each unit the drain of the accumulator; they write
//    the unit's partials (24 projections and the sum of squares per token)
//    to the workspace.
// Kernel 2 sums each token's partials over the chunks in ascending order and
// writes proj and r (programmatic dependent launch, like the backward's
// reduction).  Every mbarrier wait is bounded (wait_bar).
#include <cuda_bf16.h>

#include "mhcpb_internal.h"
#include "mhcpb_wait.cuh"
#include "ptx.cuh"

namespace mhcpb {
namespace fwd {

namespace {

constexpr int kBoxes = kChunk / kBox;                 // 8 boxes per unit
constexpr uint32_t kBoxBytes = kTokenTile * kBox * 2;  // 16 KiB
constexpr uint32_t kWBoxBytes = 48 * kBox * 2;         // 6 KiB: [Wh; Wl] rows x 64 columns
constexpr int kNS = 10;                                // X pipeline stages (one box each)
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 128;                    // two accumulators of 64 columns
constexpr uint32_t kOffW = kNS * kBoxBytes;
constexpr uint32_t kOffBar = kOffW + kBoxes * kWBoxBytes;
// barriers: x_full[NS] x_empty[NS] acc_full[2] acc_empty[2] w_full w_empty fin
constexpr int B_XF = 0, B_XE = kNS, B_AF = 2 * kNS, B_AE = 2 * kNS + 2, B_WF = 2 * kNS + 4,
              B_WE = 2 * kNS + 5, B_FIN = 2 * kNS + 6, kBars = 2 * kNS + 7;
constexpr uint32_t kOffMisc = kOffBar + kBars * 8;
constexpr uint32_t kSmem = kOffMisc + 16 + 1024;        // + room to align the base to 1 KiB
static_assert(kSmem <= 232448, "shared memory budget");

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
    fwd_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap xmap) {
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            ptx::mbar_init(bar(B_XF + s), 1);
            ptx::mbar_init(bar(B_XE + s), 1 + 4);   // the MMAs' commit + 4 sum-of-squares warps
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(B_AF + b), 1);
            ptx::mbar_init(bar(B_AE + b), 4);
        }
        ptx::mbar_init(bar(B_WF), 2);
        ptx::mbar_init(bar(B_WE), 1);
        ptx::mbar_init(bar(B_FIN), 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&xmap);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
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
                for (int b = 0; b < U.nb; ++b, ++n) {
                    if (n >= kNS &&
                        !wait_bar(bar(B_XE + st), ph ^ 1u, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(bar(B_XF + st), kBoxBytes);
                    ptx::tma_load_2d(sbase + (uint32_t)st * kBoxBytes, &xmap,
                                     U.fc * kChunk + b * kBox, U.tt * kTokenTile, bar(B_XF + st), pol);
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
            const uint32_t w_base = sbase + kOffW;
            int st = 0, ab = 0, n_w = 0, prev_fc = -1;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int u = u_begin; u < u_end && ok; ++u) {
                const Unit U = unit_at(p, u);
                if (U.fc != prev_fc) {
                    if (!wait_bar(bar(B_WF), (uint32_t)n_w & 1u, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    ++n_w;
                    prev_fc = U.fc;
                }
                if (!wait_bar(bar(B_AE + ab), aph ^ 1u, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                const uint32_t d = tmem + (uint32_t)ab * 64u;
                for (int b = 0; b < U.nb; ++b) {
                    if (!wait_bar(bar(B_XF + st), ph, abort_flag, p.status, tmo, true)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t xa = sbase + (uint32_t)st * kBoxBytes;
                    const uint32_t wb = w_base + (uint32_t)b * kWBoxBytes;
                    // four K = 16 steps inside the 128-byte swizzle atom: +32 bytes each
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t da = ptx::smem_desc(xa + 32u * k, 16u, 1024u, ptx::kLayoutSwizzle128B);
                        const uint64_t db = ptx::smem_desc(wb + 32u * k, 16u, 1024u, ptx::kLayoutSwizzle128B);
                        ptx::mma_bf16(d, da, db, idesc, (b > 0 || k > 0) ? 1u : 0u);
                    }
                    ptx::tc_commit(bar(B_XE + st));
                    if (++st == kNS) { st = 0; ph ^= 1u; }
                }
                if (!ok) break;
                ptx::tc_commit(bar(B_AF + ab));
                const bool next_fc_differs = (u + 1 >= u_end) || unit_at(p, u + 1).fc != U.fc;
                if (next_fc_differs) ptx::tc_commit(bar(B_WE));
                if (++ab == 2) { ab = 0; aph ^= 1u; }
            }
            ptx::tc_commit(bar(B_FIN));   // all MMAs complete before TMEM is freed
            wait_bar(bar(B_FIN), 0u, abort_flag, p.status, tmo, false);
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------- W preparation
        // thread = one of the chunk box's 64 columns; rows j (hi) and 24 + j (lo)
        const int col = (warp - 2) * 32 + lane;
        int n_w = 0, prev_fc = -1;
        bool ok = true;
        for (int u = u_begin; u < u_end && ok; ++u) {
            const Unit U = unit_at(p, u);
            if (U.fc == prev_fc) continue;
            prev_fc = U.fc;
            if (n_w > 0 &&
                !wait_bar(bar(B_WE), (uint32_t)(n_w - 1) & 1u, abort_flag, p.status, tmo, true)) {
                ok = false;
                break;
            }
            uint8_t* wsm = smem + kOffW;
            for (int b = 0; b < kBoxes; ++b) {
                const int k = U.fc * kChunk + b * kBox + col;
                uint8_t* box = wsm + b * kWBoxBytes;
                // 128-byte swizzle: 16-byte chunk c of row n sits at chunk c ^ (n & 7)
                const int c16 = col >> 3, within = (col & 7) * 2;
#pragma unroll 4
                for (int j = 0; j < kNProj; ++j) {
                    const float v = k < p.K ? tf32_rna(__ldg(p.w + (size_t)j * p.K + k)) : 0.f;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                    const float rem = isfinite(v) ? v - __bfloat162float(hi) : 0.f;
                    const __nv_bfloat16 lo = __float2bfloat16_rn(rem);
                    const int nh = j, nl = kNProj + j;
                    *reinterpret_cast<__nv_bfloat16*>(box + nh * 128 + ((c16 ^ (nh & 7)) << 4) + within) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(box + nl * 128 + ((c16 ^ (nl & 7)) << 4) + within) = lo;
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_WF));
            ++n_w;
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- sum of squares, drain
        const int q = warp & 3;                    // TMEM lane quarter = token rows 32q..32q+31
        const int rr = q * 32 + lane;              // row within the token tile
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const uint64_t pol_keep = ptx::policy_evict_last();
        int st = 0, ab = 0;
        uint32_t ph = 0, aph = 0;
        bool ok = true;
        for (int u = u_begin; u < u_end && ok; ++u) {
            const Unit U = unit_at(p, u);
            float ss = 0.f;
            for (int b = 0; b < U.nb; ++b) {
                if (!wait_bar(bar(B_XF + st), ph, abort_flag, p.status, tmo, true)) {
                    ok = false;
                    break;
                }
                const uint8_t* row = smem + (uint32_t)st * kBoxBytes + rr * 128;
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
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(B_XE + st));
                if (++st == kNS) { st = 0; ph ^= 1u; }
            }
            if (!ok) break;
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
                for (int j = 0; j < kNProj; ++j) {
                    const float hi = __uint_as_float(j < 16 ? d0[j] : d1[j - 16]);
                    const float lo = __uint_as_float(j < 8 ? d1[8 + j] : d2[j - 8]);
                    ptx::st_global_hint(dst + (size_t)j * p.t_pad, hi + lo, pol_keep);
                }
                ptx::st_global_hint(dst + (size_t)kNProj * p.t_pad, ss, pol_keep);
            }
            if (++ab == 2) { ab = 0; aph ^= 1u; }
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// proj[t][j] = sum over chunks ascending of partial[fc][j][t]; r from the
// summed squares.  Thread = (partial row j' in 0..24, four tokens).
constexpr int kReduceThreads = 256;
constexpr int kGroup = 8;

__global__ void __launch_bounds__(kReduceThreads)
    fwd_reduce_kernel(const float4* __restrict__ part, float* __restrict__ proj,
                      float* __restrict__ r, int T, int t4_count, int t_pad, int n_fc, float kf,
                      float eps, int discard) {
    ptx::grid_dependency_wait();
    const int64_t i = (int64_t)blockIdx.x * kReduceThreads + threadIdx.x;
    const bool valid = i < (int64_t)kPartRows * t4_count;
    const int row = valid ? (int)(i / t4_count) : 0;   // j' (24 = sum of squares)
    const int t4 = valid ? (int)(i - (int64_t)row * t4_count) : 0;
    const int64_t stride4 = (int64_t)kPartRows * (t_pad / 4);   // float4s per chunk
    const int64_t base4 = (int64_t)row * (t_pad / 4) + t4;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int f0 = 0; valid && f0 < n_fc; f0 += kGroup) {
        float4 b[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g)
            if (f0 + g < n_fc) b[g] = part[(int64_t)(f0 + g) * stride4 + base4];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            if (f0 + g < n_fc) {
                if (f0 + g == 0) {
                    a = b[g];
                } else {
                    a.x += b[g].x; a.y += b[g].y; a.z += b[g].z; a.w += b[g].w;
                }
            }
        }
    }
    if (valid) {
        const float v[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = t4 * 4 + e;
            if (t >= T) break;
            if (row < kNProj) {
                proj[(size_t)t * kProjCols + row] = v[e];
            } else {
                r[t] = sqrtf(v[e] / kf + eps);   // the mean of the squares, eps, root
#pragma unroll
                for (int c = kNProj; c < kProjCols; ++c) proj[(size_t)t * kProjCols + c] = 0.f;
            }
        }
    }
    // the partials are dead once read: drop their L2 lines (eight float4 of a
    // line belong to eight consecutive threads of this warp)
    __syncwarp();
    if (valid && discard && (t4 & 7) == 0) {
        for (int f = 0; f < n_fc; ++f) ptx::discard_l2_line(part + (int64_t)f * stride4 + base4);
    }
}

}  // namespace

size_t smem_bytes() { return kSmem; }

cudaError_t setup() {
    return cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
}

cudaError_t launch(const FwdParams& p, const CUtensorMap& x_map, int grid, cudaStream_t stream) {
    fwd_tc_kernel<<<grid, kThreads, kSmem, stream>>>(p, x_map);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int t4_count = p.t_pad / 4;
    const int64_t n = (int64_t)kPartRows * t4_count;
    // discard needs 128-byte lines: t_pad is a multiple of 32 floats
    const int discard = (reinterpret_cast<uintptr_t>(p.partial) & 127u) == 0 ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + kReduceThreads - 1) / kReduceThreads));
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fwd_reduce_kernel, reinterpret_cast<const float4*>(p.partial),
                              p.proj, p.r, p.T, t4_count, p.t_pad, p.n_fc, (float)p.K, p.eps,
                              discard);
}

}  // namespace fwd
}  // namespace mhcpb
