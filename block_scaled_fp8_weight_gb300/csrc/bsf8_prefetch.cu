// bsf8_prefetch.cu -- bsf8_prefetch_l2: pull a twin (codes and exponents) into L2.
//
// Page: "recipes/docker-images/mia-tp4/docs/tp4-adapters.md", adapter table, l2_prefetch
// row: the upcoming layer's weights are warmed in L2 on a side stream while other work
// (the collectives between layers) runs, so that the GEMM then streams them from L2.
// The GEMM kernels already start their own weight copies before their dependency wait when
// the kernel before them allows it (programmatic dependent launch); this entry point
// serves the chains where it does not -- a kernel that is not this library's, a host
// synchronisation, a collective.
//
// Each thread issues one bulk L2 prefetch (cp.async.bulk.prefetch.L2) of up to kChunk
// bytes.  A prefetch is a hint: it reads nothing into the program and writes nothing, so
// it is safe on any stream at any time.
#include "bsf8.h"
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <cuda_runtime.h>

namespace {

constexpr unsigned kChunk = 16384;  // bytes one thread's prefetch covers
constexpr int kThreads = 128;

// Prefetches [base, base + bytes): base 16-byte aligned; a tail shorter than 16 bytes is
// left out (the L2 line holding it is pulled in by the chunk before it).
__global__ void __launch_bounds__(kThreads) prefetch_kernel(const uint8_t *a, unsigned long long a_bytes,
                                                            const uint8_t *b, unsigned long long b_bytes) {
    const unsigned long long na = (a_bytes + kChunk - 1) / kChunk;
    const unsigned long long nb = (b_bytes + kChunk - 1) / kChunk;
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < na + nb; i += stride) {
        const bool first = i < na;
        const unsigned long long j = first ? i : i - na;
        const unsigned long long total = first ? a_bytes : b_bytes;
        const unsigned long long off = j * kChunk;
        const unsigned long long len = total - off < kChunk ? total - off : kChunk;
        const unsigned long long len16 = len & ~15ull;
        if (len16) bsf8::prefetch_l2((first ? a : b) + off, (uint32_t)len16);
    }
}

}  // namespace

extern "C" int bsf8_prefetch_l2(const uint8_t *w8, const uint8_t *exp, int G, int N, int K,
                                bsf8_stream_t stream) {
    if (!w8 || !exp) return BSF8_ERR_NULL;
    if (G < 1 || N < 32 || K < 32 || (N % 32) != 0 || (K % 32) != 0) return BSF8_ERR_SHAPE;
    if ((long long)G * N * (long long)K > (1LL << 46)) return BSF8_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(w8) & 15u) || (reinterpret_cast<uintptr_t>(exp) & 15u))
        return BSF8_ERR_ALIGN;
    const unsigned long long wb = (unsigned long long)G * N * K;
    const unsigned long long eb = (unsigned long long)G * (N / 32) * (K / 32);
    const unsigned long long chunks = (wb + kChunk - 1) / kChunk + (eb + kChunk - 1) / kChunk;
    const unsigned long long blocks = (chunks + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(blocks < 1024 ? blocks : 1024);
    prefetch_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(w8, wb, exp, eb);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return BSF8_OK;
    return (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction) ? BSF8_ERR_DEVICE
                                                                                         : BSF8_ERR_CUDA;
}
