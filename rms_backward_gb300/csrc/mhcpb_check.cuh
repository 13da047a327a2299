// Bounds checks of a checked build (nvcc -DMHCPB_CHECKED).
//
// compute-sanitizer is not available to this library's tests, so a checked
// build stands in for its bounds checking: every global-memory access at a
// computed address (tensor-map copies are bounded by their maps already) is
// checked against the extent of the buffer it belongs to.  An access outside
// is skipped, and the first one records its site number in a word of the
// translation unit; mhcpb_debug_checked_sites reads and clears those words.
// In a normal build every check is the constant `true` and the word does not
// exist.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mhcpb {
namespace check {

#ifdef MHCPB_CHECKED
constexpr bool kEnabled = true;
// 0, or 1 + the site of the first access found outside its buffer (one word
// per translation unit: internal linkage)
static __device__ uint32_t g_first_site;

// true when [p, p + access) lies inside [base, base + bytes)
__device__ __forceinline__ bool in(const void* p, size_t access, const void* base, size_t bytes,
                                   uint32_t site) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
    if (a >= b && a - b <= bytes && access <= bytes - (a - b)) return true;
    atomicCAS(&g_first_site, 0u, 1u + site);
    return false;
}

// this translation unit's word, then cleared (current device)
static inline cudaError_t read_and_clear(uint32_t* site) {
    const uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(site, g_first_site, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_first_site, &zero, sizeof(uint32_t));
    return e;
}
#else
constexpr bool kEnabled = false;
__device__ __forceinline__ constexpr bool in(const void*, size_t, const void*, size_t, uint32_t) {
    return true;
}
static inline cudaError_t read_and_clear(uint32_t* site) {
    *site = 0;
    return cudaSuccess;
}
#endif

}  // namespace check
}  // namespace mhcpb
