// bsf8_noalloc.cu -- bsf8_gemm_static_scratch: the split-K GEMM for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace: a serving engine that reserves all of
// the GPU's memory up front for its own arena (weights, KV cache) has no allocation left to
// give, and a plugin or callback running inside such an engine may not call the allocator
// at all.  This entry point needs nothing from them but the inputs and the output: it runs
// the two-pass split-K GEMM (the fp32 partials pass, then the fixed-order reduce) with the
// partials in a buffer compiled into the library -- a file-scope device array that every
// GPU which loads the library holds until the process exits.
#include "bsf8.h"
#include "bsf8_internal.h"

#include <cstdint>

namespace {

constexpr size_t kScratchFloats = BSF8_STATIC_SCRATCH_BYTES / sizeof(float);

// The partials of every call live here.  Host code must not use this name as an address
// (on the host it is only a stand-in for the device symbol); the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_static_scratch[kScratchFloats];

// Device address of g_static_scratch on the current device, looked up once per device
// (on that device's first call).  Returns the CUDA error of the lookup, if any.
cudaError_t static_scratch_address(float **out) {
    static float *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    float *a = __atomic_load_n(&addr[dev], __ATOMIC_ACQUIRE);
    if (!a) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        a = static_cast<float *>(p);
        __atomic_store_n(&addr[dev], a, __ATOMIC_RELEASE);
    }
    *out = a;
    return cudaSuccess;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int status_of(cudaError_t e) {
    if (e == cudaSuccess) return BSF8_OK;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return BSF8_ERR_DEVICE;
    return BSF8_ERR_CUDA;
}

}  // namespace

extern "C" int bsf8_gemm_static_scratch(const void *x, const uint8_t *w8, const uint8_t *exp,
                                        void *y, int M, int N, int K, int G, int split_k,
                                        int64_t ldx, bsf8_stream_t stream) {
    // Argument rules of bsf8_gemm.
    if (!x || !w8 || !exp || !y) return BSF8_ERR_NULL;
    if (G < 1 || N < 32 || K < 32 || (N % 32) != 0 || (K % 32) != 0) return BSF8_ERR_SHAPE;
    if ((long long)G * N * (long long)K > (1LL << 46)) return BSF8_ERR_SHAPE;
    if (M < 1 || M > BSF8_MAX_M) return BSF8_ERR_SHAPE;
    if (split_k < 0 || split_k > K / 32) return BSF8_ERR_SHAPE;
    if (ldx < (int64_t)G * K) return BSF8_ERR_STRIDE;
    if (!aligned16(x) || (ldx % 8) != 0 || !aligned16(w8)) return BSF8_ERR_ALIGN;

    const int S = split_k == 0 ? bsf8::auto_split(M, N, K, G) : split_k;
    // The partials P[S][M][G][N] must fit the compiled-in buffer.
    if ((size_t)S * M * G * N > kScratchFloats) return BSF8_ERR_WORKSPACE;

    float *P = nullptr;
    cudaError_t e = static_scratch_address(&P);
    if (e != cudaSuccess) return status_of(e);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Every split writes all of its partials (an empty split writes +0) before the reduce
    // reads them, so nothing in the buffer needs clearing between calls.
    const bsf8::StreamPlan pl = bsf8::plan_stream(M, N, K, G, S, true);
    e = bsf8::launch_stream(pl, x, ldx, w8, exp, nullptr, P, M, N, K, G, s);
    if (e != cudaSuccess) return status_of(e);
    return status_of(bsf8::launch_splitk_reduce(P, y, S, (long long)M * G * N, s));
}
