// bsf8_noalloc.cu -- bsf8_gemm_static_scratch: the split-K GEMM for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace: a serving engine that reserves all of
// the GPU's memory up front for its own arena (weights, KV cache) has no allocation left to
// give, and a plugin or callback running inside such an engine may not call the allocator
// at all.  This entry point needs nothing from them but the inputs and the output.  Where
// bsf8_gemm needs no workspace for the call (its kernels sum the splits on chip) it is
// bsf8_gemm.  Otherwise it runs the two passes of the split-K GEMM -- bsf8_gemm_partials,
// then bsf8_splitk_reduce -- with the partials in a buffer compiled into the library, a
// file-scope device array that every GPU which loads the library holds until the process
// exits.  Those two passes run the kernel bsf8_gemm runs for the same sizes and split count
// and sum the splits in the same fixed order, so the result is bsf8_gemm's, bit for bit.
#include "bsf8.h"

#include <cuda_runtime.h>

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
    // Argument rules of bsf8_gemm (bsf8_gemm_partials checks the rest).
    if (!x || !w8 || !exp || !y) return BSF8_ERR_NULL;
    if (G < 1 || N < 32 || K < 32 || (N % 32) != 0 || (K % 32) != 0) return BSF8_ERR_SHAPE;
    if ((long long)G * N * (long long)K > (1LL << 46)) return BSF8_ERR_SHAPE;
    if (M < 1 || M > BSF8_MAX_M) return BSF8_ERR_SHAPE;
    if (split_k < 0 || split_k > K / 32) return BSF8_ERR_SHAPE;

    // the split count bsf8_gemm uses
    const int S = split_k == 0 ? bsf8_gemm_auto_split(M, N, K, G) : split_k;
    if (S < 1) return -S;
    // no workspace needed: bsf8_gemm itself
    if (bsf8_gemm_workspace_bytes(M, N, K, G, S) == 0)
        return bsf8_gemm(x, w8, exp, y, M, N, K, G, S, ldx, nullptr, 0, stream);
    // The partials P[S][M][G][N] must fit the compiled-in buffer.
    if ((size_t)S * M * G * N > kScratchFloats) return BSF8_ERR_WORKSPACE;

    float *P = nullptr;
    const cudaError_t e = static_scratch_address(&P);
    if (e != cudaSuccess) return status_of(e);
    // Every split writes all of its partials (an empty split writes +0) before the reduce
    // reads them, so nothing in the buffer needs clearing between calls.
    const int st = bsf8_gemm_partials(x, w8, exp, P, M, N, K, G, S, ldx, stream);
    if (st != BSF8_OK) return st;
    return bsf8_splitk_reduce(P, y, S, (int64_t)M * G * N, stream);
}
