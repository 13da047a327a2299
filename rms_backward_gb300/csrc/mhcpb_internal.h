// Internal interface between the C-ABI host code and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mhcpb {

constexpr int kNProj = 24;          // projection columns used (P = grad_proj[:, :24])
constexpr int kGradProjCols = 32;   // stored width of grad_proj
// Tokens per dW partial: fixed (never a function of the GPU), so dW bits
// depend only on (T, K) and the inputs.  512 tokens keep the partials at 1/256
// of the streamed bytes; 256-token chunks balanced the persistent grid better
// but measured slower (twice the per-chunk dW drains and partial traffic).
constexpr int kMaxTokensPerPartial = 512;
inline int partial_tokens(int64_t /*T*/) { return 512; }

// Device status word values (match mhcpb_status_t).
constexpr uint32_t kDevOk = 0;
constexpr uint32_t kDevTimeout = 9;

// Everything the streaming kernels need besides the tensor maps.
struct MainParams {
    int32_t T;
    int32_t K;
    int32_t S;            // number of dW partials = ceil(T / chunk)
    int32_t chunk;        // tokens per dW partial (partial_tokens(T))
    int32_t n_strips;     // ceil(K / strip width) of the kernel in use
    int32_t half_units;   // tensor-core kernel: schedule in half items (64 columns)
    const uint16_t* x;    // BF16 [T, K] (FMA kernel reads it directly)
    const float* w;       // [24, K]
    const float* grad_proj;  // [T, 32]
    const float* grad_r;  // [T]
    const float* r;       // [T]
    uint16_t* dx;         // BF16 [T, K] (FMA kernel writes it directly)
    const uint16_t* addend;  // BF16 [T, K] or null
    float* partial;       // [S, 24, K]
    uint32_t* status;     // device status word
    uint64_t timeout_ns;  // bound on every wait inside the kernel
    uint32_t test_flags;  // kTestInjectStall: the MMA issuer waits on a barrier nothing completes
    uint64_t* trace;      // timeline stamps, only in builds with MHCPB_TRACE (else null)
};

// Timeline stamps of a traced build: [grid][kTraceEvents][kTraceTiles] u64.
constexpr int kTraceEvents = 19;
constexpr int kTraceTiles = 80;

constexpr uint32_t kTestInjectStall = 1u;

// Tensor-core (tcgen05 + TMA) streaming kernel: geometry and launch.
namespace tc {
constexpr int kTokenTile = 128;    // MMA M for dX; K-extent of one dW MMA group
constexpr int kStrip = 128;        // columns per strip: MMA N for dX, M for dW
constexpr int kBoxCols = 64;       // TMA box width (128 bytes of BF16)
// Schedule unit: half of a (strip, chunk) item (64 columns).  Whole-item
// units were measured slower at the training profile (69.1 vs 67.2 us): with
// half units the CTAs that get an extra unit move half an item's bytes more,
// not a whole item's.  The whole-item mode stays for comparison.
inline bool use_half_units(int64_t /*items*/, int /*sms*/) { return true; }
// Persistent grid: one CTA per SM, at most one per schedule unit, so every
// CTA has work.
inline int grid_size(int64_t items, int sms) {
    const int64_t units = use_half_units(items, sms) ? 2 * items : items;
    return (int)(units < sms ? units : sms);
}
size_t smem_bytes(bool has_addend);
cudaError_t setup(bool has_addend);
// checked builds: this unit's first out-of-range site (0: none), then cleared
cudaError_t checked_site(uint32_t* site);
// Tensor maps: x/dx/addend BF16 [T,K] boxes 64 x {128,32,128} (128-byte swizzle),
// grad_proj FP32 [T,32] box 24 x 128, grad_r and r FP32 [T] boxes of 128.
cudaError_t launch(const MainParams& p, const CUtensorMap& x_map, const CUtensorMap& dx_map,
                   const CUtensorMap& add_map, const CUtensorMap& gp_map, const CUtensorMap& gr_map,
                   const CUtensorMap& r_map, int grid, cudaStream_t stream);
}  // namespace tc

// FP32-FMA (CUDA core) streaming kernel: the measured control.
namespace fma {
constexpr int kStrip = 64;
constexpr int kThreads = 256;
size_t smem_bytes();
cudaError_t setup();
cudaError_t launch(const MainParams& p, cudaStream_t stream);
cudaError_t checked_site(uint32_t* site);
}  // namespace fma

// Forward of the stage (proj = X W^T over TF32 W, r = RMS of each row):
// tensor-core kernel plus a fixed-order reduction of per-chunk partials.
namespace fwd {
constexpr int kTokenTile = 128;   // MMA M
constexpr int kChunk = 512;       // columns per work unit (fixed: partials depend only on K)
constexpr int kBox = 64;          // TMA box width
constexpr int kPartRows = 25;     // per chunk and token: 24 projections + the sum of squares
constexpr int kProjCols = 32;     // stored width of proj (columns 24..31 written as zero)
struct FwdParams {
    int32_t T;
    int32_t K;
    int32_t n_tt;         // token tiles, ceil(T / 128)
    int32_t n_fc;         // column chunks, ceil(K / 512)
    int32_t t_pad;        // token stride of the partial rows, T rounded up to 32
    const float* w;       // [24, K]
    float* partial;       // [n_fc][25][t_pad]
    float* proj;          // [T, 32]
    float* r;             // [T]
    float eps;
    uint32_t* status;
    uint64_t timeout_ns;
    uint64_t* trace;      // timeline stamps, only in builds with MHCPB_TRACE (else null)
};
inline int64_t t_pad(int64_t T) { return (T + 31) / 32 * 32; }
inline int64_t n_chunks(int64_t K) { return (K + kChunk - 1) / kChunk; }
inline size_t workspace_bytes(int64_t T, int64_t K) {
    return (size_t)n_chunks(K) * kPartRows * (size_t)t_pad(T) * sizeof(float);
}
inline int grid_size(int64_t T, int64_t K, int sms) {
    const int64_t units = n_chunks(K) * ((T + kTokenTile - 1) / kTokenTile);
    return (int)(units < sms ? units : sms);
}
size_t smem_bytes();
cudaError_t setup();
cudaError_t checked_site(uint32_t* site);
// The gate step fused into the forward's reduction (mhcpb_forward_gates):
// h [T, 24] from the proj and r the reduction writes.
struct GateArgs {
    const float* alpha;   // [3]
    const float* bias;    // [24]
    int n_iter;
    float* h;             // [T, 24]
};
// launches both kernels on `stream`; x_map: X [T, K] BF16, boxes 64 x 128, 128-byte swizzle;
// w_map: W [24, K] FP32, boxes 64 x 24, no swizzle; non-null events are
// recorded before, between and after the two kernels; with `gates` the
// reduction also writes the gates
cudaError_t launch(const FwdParams& p, const CUtensorMap& x_map, const CUtensorMap& w_map, int grid,
                   cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1, cudaEvent_t ev2,
                   const GateArgs* gates = nullptr);
}  // namespace fwd

// Gate/normalisation step (mhcpb_gate_forward / mhcpb_gate_backward): a
// half-warp per token; log-domain iterations; the backward keeps the row- and
// column-normalised matrices of every iteration (2 n_iter per token) in shared
// memory.
namespace gates {
constexpr int kMaxIter = 64;
size_t backward_smem_bytes(int n_iter);
cudaError_t setup();
cudaError_t checked_site(uint32_t* site);
cudaError_t launch_forward(int64_t T, int n_iter, const float* proj, const float* r,
                           const float* alpha, const float* bias, float* h, cudaStream_t stream);
cudaError_t launch_backward(int64_t T, int n_iter, const float* proj, const float* r,
                            const float* alpha, const float* bias, const float* grad_h,
                            float* grad_proj, float* grad_r, float* dlogits, cudaStream_t stream);
}  // namespace gates

// Host helpers shared by the entry points (defined in mhcpb_api.cu).
// encode_tc_maps: the six tensor maps of the tensor-core kernel; returns the
// name of the map that failed, or null.  record_cuda_error: stores the
// thread's CUDA error text and returns MHCPB_ERR_CUDA.
const char* encode_tc_maps(CUtensorMap (&m)[6], int64_t T, int64_t K, const void* x,
                           const void* dx, const void* add, const void* gp, const void* gr,
                           const void* r);
int record_cuda_error(cudaError_t e, const char* what);

// Second kernel: dW[j,k] = sum over s ascending of partial[s][j][k]; with
// `compensated`, TwoSum at every addition and one final rounding; with
// `accumulate`, the result is added to dW's previous contents.
// `discard`: drop the partials' L2 lines after reading them (their contents
// are then undefined), only where nothing reads them again.
cudaError_t reduce_checked_site(uint32_t* site);
cudaError_t launch_reduce(const float* partial, float* dw, int S, int64_t n, bool compensated,
                          bool accumulate, bool discard, cudaStream_t stream);

}  // namespace mhcpb
