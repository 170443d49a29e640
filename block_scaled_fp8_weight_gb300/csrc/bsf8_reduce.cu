// bsf8_reduce.cu -- the fixed-order split-K sum (the second pass of a split GEMM) and the
// size-only split rule of the streaming kernel.
//
// Page: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- the reduce after
// _wo_a_partial_w8(): the module docstring's "Split-K partials are summed in a fixed order".
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <algorithm>

namespace bsf8 {

//   y[i] = bf16( ((P[0][i] + P[1][i]) + P[2][i]) + ... ),  fp32, left to right.
// Writes nothing while the device status word holds a timeout: the partials a first pass
// left after giving up a wait are incomplete (the status stays until the host reads it).
// OUT is uint16_t (bf16 y, one RNE) or float (the fp32 sums themselves: the head's fp32
// logits variant).
template <typename OUT>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ P,
                                                            OUT *__restrict__ y, int S,
                                                            long long count, const int *status) {
    pdl_trigger();
    pdl_wait();
    if (*(const volatile int *)status == kStatusTimeout) return;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
        float v = __ldcg(P + i);
        for (int s = 1; s < S; ++s) v = v + __ldcg(P + (size_t)s * count + i);
        if constexpr (sizeof(OUT) == 2)
            y[i] = f32_to_bf16_rn(v);
        else
            y[i] = v;
    }
}

// The split count of the streaming kernel when the caller leaves it to the library: the
// smallest S whose tiles of 64 weight rows (times groups and 32-token chunks) reach two
// blocks per SM of a 152-SM GB300, at most 8 and at most K/32.
int auto_split(int M, int N, int K, int G) {
    constexpr int kRowsPerTile = 64;
    constexpr long long kTargetBlocks = 2 * 152;
    const int nt8 = std::min(4, (M + 7) / 8);
    const int m_chunks = (M + 8 * nt8 - 1) / (8 * nt8);
    const long long tiles = (long long)((N + kRowsPerTile - 1) / kRowsPerTile) * G * m_chunks;
    const int smax = std::max(1, std::min(kMaxClusterSplits, K / 32));
    for (int S = 1; S <= smax; ++S)
        if (tiles * S >= kTargetBlocks) return S;
    return smax;
}

namespace {

template <typename OUT>
cudaError_t launch_reduce(const float *P, OUT *y, int S, long long count, cudaStream_t stream) {
    if (count == 0) return cudaSuccess;
    const Options opt = options();
    cudaLaunchConfig_t cfg = {};
    const long long blocks = std::min<long long>((count + 255) / 256, 152LL * 8);
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = opt.pdl ? 1 : 0;
    const int *status = status_word();
    if (!status) return cudaErrorInvalidSymbol;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<OUT>, P, y, S, count, status);
}

}  // namespace

cudaError_t launch_splitk_reduce(const float *P, void *y, int S, long long count, cudaStream_t stream) {
    return launch_reduce(P, static_cast<uint16_t *>(y), S, count, stream);
}

cudaError_t launch_splitk_reduce_f32(const float *P, float *y, int S, long long count, cudaStream_t stream) {
    return launch_reduce(P, y, S, count, stream);
}

}  // namespace bsf8
