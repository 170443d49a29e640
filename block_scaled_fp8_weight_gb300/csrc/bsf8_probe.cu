// bsf8_probe.cu -- bsf8_sm_clock_sample: a diagnostic for measurements (not on the path).
//
// Each block writes, for the SM it runs on, the global nanosecond timer and that SM's cycle
// counter.  Two samples on a stream, one before and one after a timed region, give every
// SM's average clock over the region: (cycles_after - cycles_before) / (ns_after - ns_before)
// per SM id, a figure taken inside the region rather than from an outside sampler whose
// period may exceed the region's length.
#include "bsf8.h"
#include "bsf8_device.cuh"

#include <cuda_runtime.h>

namespace {

__global__ void sm_clock_kernel(unsigned long long *out, int nsm) {
    unsigned int smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    if (threadIdx.x == 0 && (int)smid < nsm) {
        out[2 * smid] = bsf8::global_ns();
        out[2 * smid + 1] = clock64();
    }
}

}  // namespace

extern "C" int bsf8_sm_clock_sample(uint64_t *out, int nsm, bsf8_stream_t stream) {
    if (!out) return BSF8_ERR_NULL;
    if (nsm < 1 || nsm > 4096) return BSF8_ERR_SHAPE;
    sm_clock_kernel<<<2 * nsm, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<unsigned long long *>(out), nsm);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return BSF8_OK;
    return (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction) ? BSF8_ERR_DEVICE
                                                                                         : BSF8_ERR_CUDA;
}
