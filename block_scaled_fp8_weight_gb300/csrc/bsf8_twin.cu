// bsf8_twin.cu -- load-time kernels of libbsf8: the twin quantizer, the exact dequant
// and the K-padding of a twin and of an activation.
//
// Pages: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" (make_twin(),
// _dequant_kernel()) and "recipes/docker-images/mia-tp4/adapter/shared_pad_k.py"
// (_pad_weight(), _pad_input()).  All of them move every byte once: their roofline is
// HBM bandwidth.
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <algorithm>

namespace bsf8 {

namespace {

int grid_for(long long work, int threads) {
    const long long b = (work + threads - 1) / threads;
    return (int)std::max(1LL, std::min(b, 152LL * 16));
}

// Launches with programmatic dependent launch when enabled: a kernel may start while the
// previous one in the stream finishes; each kernel here waits (griddepcontrol.wait) before
// it touches memory, so only the launch overlaps.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), int grid, int block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)block, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = options().pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

}  // namespace

// ------------------------------------------------------------------ make_twin
//
// One warp per 32x32 block, lane r owns row r of the block (32 bf16 = 64 bytes).
//  amax:   integer max of |w| bit patterns (monotone in magnitude for non-NaN bf16);
//          a pattern >= 0x7F80 means Inf/NaN in the block.
//  e:      for amax = 2^E * (1 + f/128) (amax raised to 2^-126 first),
//          ceil(log2(amax/448)) = E - 8 + (f > 96), as 448 = 1.75 * 2^8 and
//          1 + 96/128 = 1.75; clamped to [-127, 127].
//  codes:  cvt.rn.satfinite.e4m3x2.f32 of w * 2^-e (a power-of-two scaling rounds
//          exactly like the division by 2^e; |w * 2^-e| <= 448, so saturation never
//          acts).
//  check:  the rebuild bf16(code * 2^e) -- the GEMM's own rebuild4 -- compared by value
//          with w (so -0 == +0).

__global__ void set_i32_kernel(int32_t *p, int32_t v) {
    pdl_trigger();
    pdl_wait();
    *p = v;
}

__device__ __forceinline__ uint16_t cvt_e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ bool bf16_pair_equal(uint32_t a, uint32_t b) {
    const uint32_t a0 = a & 0xFFFFu, a1 = a >> 16, b0 = b & 0xFFFFu, b1 = b >> 16;
    const bool e0 = (a0 == b0) || (((a0 | b0) & 0x7FFFu) == 0u);
    const bool e1 = (a1 == b1) || (((a1 | b1) & 0x7FFFu) == 0u);
    return e0 && e1;
}

__global__ void __launch_bounds__(256) make_twin_kernel(const uint16_t *__restrict__ w,
                                                        uint8_t *__restrict__ w8,
                                                        uint8_t *__restrict__ ex,
                                                        uint8_t *__restrict__ ok,
                                                        int32_t *__restrict__ accepted, int G,
                                                        int N, int K) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int nb = N / 32, kb = K / 32;
    const long long nblocks = (long long)G * nb * kb;
    const long long warps = (long long)gridDim.x * (blockDim.x / 32);
    for (long long b = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); b < nblocks;
         b += warps) {
        const long long rowblk = b / kb;  // g * nb + bi
        const int bj = (int)(b - rowblk * kb);
        const size_t row = (size_t)rowblk * 32 + lane;
        const uint16_t *src = w + row * K + (size_t)bj * 32;
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 u = *reinterpret_cast<const uint4 *>(src + 8 * i);
            v[4 * i + 0] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            amax = max(amax, max(v[i] & 0x7FFFu, (v[i] >> 16) & 0x7FFFu));
        amax = __reduce_max_sync(0xFFFFFFFFu, amax);

        uint8_t *dst = w8 + row * K + (size_t)bj * 32;
        if (amax >= 0x7F80u) {  // Inf or NaN in the block
            const uint4 nanq = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            reinterpret_cast<uint4 *>(dst)[0] = nanq;
            reinterpret_cast<uint4 *>(dst)[1] = nanq;
            if (lane == 0) {
                ex[b] = 0xFF;
                if (ok) ok[b] = 0;
                *accepted = 0;
            }
            continue;
        }
        int E, f;
        if (amax < 0x0080u) {  // below 2^-126 (zero or subnormal): the 2^-126 floor
            E = -126;
            f = 0;
        } else {
            E = (int)(amax >> 7) - 127;
            f = (int)(amax & 0x7Fu);
        }
        int e = E - 8 + (f > 0x60 ? 1 : 0);
        e = min(127, max(-127, e));
        const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, e <= 120
        const Scale sc = make_scale((uint32_t)(e + 127));
        uint32_t codes[8];
        bool good = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t p0 = v[2 * i], p1 = v[2 * i + 1];
            const float f0 = __uint_as_float(p0 << 16) * inv;
            const float f1 = __uint_as_float(p0 & 0xFFFF0000u) * inv;
            const float f2 = __uint_as_float(p1 << 16) * inv;
            const float f3 = __uint_as_float(p1 & 0xFFFF0000u) * inv;
            const uint32_t c = (uint32_t)cvt_e4m3x2(f1, f0) | ((uint32_t)cvt_e4m3x2(f3, f2) << 16);
            codes[i] = c;
            uint32_t lo, hi;
            rebuild4(c, sc, lo, hi);
            good = good && bf16_pair_equal(lo, p0) && bf16_pair_equal(hi, p1);
        }
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        const bool block_ok = __all_sync(0xFFFFFFFFu, good);
        if (lane == 0) {
            ex[b] = (uint8_t)(e + 127);
            if (ok) ok[b] = block_ok ? 1 : 0;
            if (!block_ok) *accepted = 0;
        }
    }
}

cudaError_t launch_make_twin(const void *w, uint8_t *w8, uint8_t *ex, uint8_t *ok,
                             int32_t *accepted, int G, int N, int K, cudaStream_t stream) {
    cudaError_t e = launch_pdl(set_i32_kernel, 1, 1, stream, accepted, 1);
    if (e != cudaSuccess) return e;
    const long long nblocks = (long long)G * (N / 32) * (K / 32);
    if (nblocks > 0)
        e = launch_pdl(make_twin_kernel, grid_for(nblocks * 32, 256), 256, stream, static_cast<const uint16_t *>(w),
                       w8, ex, ok, accepted, G, N, K);
    return e;
}

// ----------------------------------------------------- make_twin, 1 x 32 blocks
// The per-(row, 32-column) scale layout of the adapter table's draft_main_proj row: the
// same rule as make_twin with the block narrowed to one row of 32 columns; exponents and
// flags [G][N][K/32].  One thread a segment (64 bytes of bf16 in, 32 codes out), so a
// warp's loads cover 2 KB of consecutive columns.
__global__ void __launch_bounds__(256) make_twin_rows_kernel(const uint16_t *__restrict__ w,
                                                             uint8_t *__restrict__ w8,
                                                             uint8_t *__restrict__ ex,
                                                             uint8_t *__restrict__ ok,
                                                             int32_t *__restrict__ accepted,
                                                             long long nseg) {
    pdl_trigger();
    pdl_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long sg = (long long)blockIdx.x * blockDim.x + threadIdx.x; sg < nseg; sg += stride) {
        const uint16_t *src = w + sg * 32;
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 u = *reinterpret_cast<const uint4 *>(src + 8 * i);
            v[4 * i + 0] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = max(amax, max(v[i] & 0x7FFFu, (v[i] >> 16) & 0x7FFFu));
        uint4 *dst = reinterpret_cast<uint4 *>(w8 + sg * 32);
        if (amax >= 0x7F80u) {  // Inf or NaN in the segment
            const uint4 nanq = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            dst[0] = nanq;
            dst[1] = nanq;
            ex[sg] = 0xFF;
            if (ok) ok[sg] = 0;
            *accepted = 0;
            continue;
        }
        int E, f;
        if (amax < 0x0080u) {  // below 2^-126: the 2^-126 floor
            E = -126;
            f = 0;
        } else {
            E = (int)(amax >> 7) - 127;
            f = (int)(amax & 0x7Fu);
        }
        int e = E - 8 + (f > 0x60 ? 1 : 0);
        e = min(127, max(-127, e));
        const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
        const Scale sc = make_scale((uint32_t)(e + 127));
        uint32_t codes[8];
        bool good = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t p0 = v[2 * i], p1 = v[2 * i + 1];
            const float f0 = __uint_as_float(p0 << 16) * inv;
            const float f1 = __uint_as_float(p0 & 0xFFFF0000u) * inv;
            const float f2 = __uint_as_float(p1 << 16) * inv;
            const float f3 = __uint_as_float(p1 & 0xFFFF0000u) * inv;
            const uint32_t c = (uint32_t)cvt_e4m3x2(f1, f0) | ((uint32_t)cvt_e4m3x2(f3, f2) << 16);
            codes[i] = c;
            uint32_t lo, hi;
            rebuild4(c, sc, lo, hi);
            good = good && bf16_pair_equal(lo, p0) && bf16_pair_equal(hi, p1);
        }
        dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        ex[sg] = (uint8_t)(e + 127);
        if (ok) ok[sg] = good ? 1 : 0;
        if (!good) *accepted = 0;
    }
}

cudaError_t launch_make_twin_rows(const void *w, uint8_t *w8, uint8_t *ex, uint8_t *ok, int32_t *accepted,
                                  int G, int N, int K, cudaStream_t stream) {
    cudaError_t e = launch_pdl(set_i32_kernel, 1, 1, stream, accepted, 1);
    if (e != cudaSuccess) return e;
    const long long nseg = (long long)G * N * (K / 32);
    if (nseg > 0)
        e = launch_pdl(make_twin_rows_kernel, grid_for(nseg, 256), 256, stream, static_cast<const uint16_t *>(w),
                       w8, ex, ok, accepted, nseg);
    return e;
}

// -------------------------------------------------------------------- dequant
// One thread per 16 codes of a row: out = bf16(e4m3 * 2^(e-127)) via rebuild4 (the
// same rebuild the GEMM runs in registers), NaN codes patched to NaN.
// ROWS: one exponent byte per (row, 32 columns), [G][N][K/32]; else per 32 x 32 block.
template <bool ROWS>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ w8,
                                                      const uint8_t *__restrict__ ex,
                                                      uint16_t *__restrict__ out, int K,
                                                      long long chunks) {
    pdl_trigger();
    pdl_wait();
    const int kb = K / 32;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += stride) {
        const long long byte = c * 16;
        const long long row = byte / K;  // g * N + n
        const int k = (int)(byte - row * K);
        const uint32_t e = ex[(size_t)(ROWS ? row : row / 32) * kb + k / 32];
        const Scale sc = make_scale(e);
        const uint4 q = *reinterpret_cast<const uint4 *>(w8 + byte);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            rebuild4(qw[i], sc, o[2 * i], o[2 * i + 1]);
            if (nan_code_mask(qw[i])) patch_nan_codes(qw[i], o[2 * i], o[2 * i + 1]);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out + byte);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

cudaError_t launch_dequant(const uint8_t *w8, const uint8_t *ex, void *out, int G, int N, int K,
                           cudaStream_t stream) {
    const long long chunks = (long long)G * N * K / 16;
    if (chunks > 0)
        return launch_pdl(dequant_kernel<false>, grid_for(chunks, 256), 256, stream, w8, ex,
                          static_cast<uint16_t *>(out), K, chunks);
    return cudaSuccess;
}

cudaError_t launch_dequant_rows(const uint8_t *w8, const uint8_t *ex, void *out, int G, int N, int K,
                                cudaStream_t stream) {
    const long long chunks = (long long)G * N * K / 16;
    if (chunks > 0)
        return launch_pdl(dequant_kernel<true>, grid_for(chunks, 256), 256, stream, w8, ex,
                          static_cast<uint16_t *>(out), K, chunks);
    return cudaSuccess;
}

// ---------------------------------------------------------------------- pad-K
// One launch pads both arrays: threads 0 .. chunks-1 copy 16-byte pieces of the codes
// (zeros past K), the threads after them the exponent bytes (pad_exp past K/32).
__global__ void __launch_bounds__(256) pad_k_kernel(const uint8_t *__restrict__ w8,
                                                    uint8_t *__restrict__ w8_out,
                                                    const uint8_t *__restrict__ ex,
                                                    uint8_t *__restrict__ ex_out, int K, int Kp,
                                                    uint8_t pad_exp, long long chunks, long long n) {
    pdl_trigger();
    pdl_wait();
    const int cpr = Kp / 16, kb = K / 32, kbp = Kp / 32;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < chunks + n; c += stride) {
        if (c < chunks) {
            const long long row = c / cpr;
            const int k = (int)(c - row * cpr) * 16;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (k < K) v = *reinterpret_cast<const uint4 *>(w8 + (size_t)row * K + k);
            *reinterpret_cast<uint4 *>(w8_out + (size_t)row * Kp + k) = v;
        } else {
            const long long i = c - chunks;
            const long long row = i / kbp;
            const int j = (int)(i - row * kbp);
            ex_out[i] = j < kb ? ex[(size_t)row * kb + j] : pad_exp;
        }
    }
}

__global__ void __launch_bounds__(256) pad_x_kernel(const uint16_t *__restrict__ x, long long ldx,
                                                    uint16_t *__restrict__ x_out, int G, int K,
                                                    int Kp, long long chunks) {
    pdl_trigger();
    pdl_wait();
    const int cpg = Kp / 8;  // 16-byte chunks per group row
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += stride) {
        const long long mg = c / cpg;  // m * G + g
        const int k = (int)(c - mg * cpg) * 8;
        const long long m = mg / G;
        const int g = (int)(mg - m * G);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (k < K) v = *reinterpret_cast<const uint4 *>(x + (size_t)m * ldx + (size_t)g * K + k);
        *reinterpret_cast<uint4 *>(x_out + (size_t)mg * Kp + k) = v;
    }
}

cudaError_t launch_pad_k(const uint8_t *w8, const uint8_t *ex, uint8_t *w8_out, uint8_t *ex_out,
                         int G, int N, int K, int Kp, int pad_exp, cudaStream_t stream) {
    const long long chunks = (long long)G * N * (Kp / 16);
    const long long n = (long long)G * (N / 32) * (Kp / 32);
    if (chunks + n > 0)
        return launch_pdl(pad_k_kernel, grid_for(chunks + n, 256), 256, stream, w8, w8_out, ex, ex_out, K, Kp,
                          (uint8_t)pad_exp, chunks, n);
    return cudaSuccess;
}

cudaError_t launch_pad_x(const void *x, long long ldx, void *x_out, int M, int G, int K, int Kp,
                         cudaStream_t stream) {
    const long long chunks = (long long)M * G * (Kp / 8);
    if (chunks > 0)
        return launch_pdl(pad_x_kernel, grid_for(chunks, 256), 256, stream, static_cast<const uint16_t *>(x), ldx,
                          static_cast<uint16_t *>(x_out), G, K, Kp, chunks);
    return cudaSuccess;
}

}  // namespace bsf8
