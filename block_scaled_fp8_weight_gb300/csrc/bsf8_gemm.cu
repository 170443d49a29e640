// bsf8_gemm.cu -- the small-M block-scaled FP8 weight GEMM for GB300 (sm_103a).
//
//   y[m][g][n] = bf16( sum_s P[s][m][g][n] ),  P[s] = sum over split s of x * W,
//   W[g][n][k] = bf16( e4m3(w8[g][n][k]) * 2^(exp[g][n/32][k/32] - 127) ).
//
// Pages: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- _wo_a_partial_w8(),
// _wo_a_mid_kernel() and the fixed-order sum of their split-K partials.
//
// Design (weight-bandwidth bound at M <= 8: 2*M flops per weight byte):
//  * One CTA owns 64 weight rows x one split's columns of one group and up to 32 token
//    rows; larger M runs several token chunks (grid.y = G x chunks).
//  * A producer warp streams the weight rows into a shared-memory ring with 1-D bulk
//    copies (TMA), one copy per row per 256-column stage, completing on an mbarrier.
//    Before the programmatic-dependent-launch wait it only prefetches those rows into
//    L2, which is coherent, so the next layer's weights stream from HBM while the
//    previous kernel drains.
//  * Four consumer warps each take a 64-column slice of every stage for all 64 rows.
//    A thread reads 16 contiguous codes of a row (one 128-bit shared load), rebuilds
//    them exactly as bf16 with two byte permutes, a shift, a mask and one bf16x2
//    multiply per pair (see rebuild4), and feeds mma.sync m16n8k16 with the weight rows
//    as the MMA "M" side and the tokens as its "N" side.  The k order inside an MMA is
//    permuted the same way for both operands (thread t of a quad owns 16 contiguous
//    columns), so every operand load is a plain 128-bit load.
//  * The four warps' fp32 partials are summed in warp order, then the S splits of a
//    tile are summed s = 0..S-1: through distributed shared memory inside a cluster
//    (S <= 8), or as fp32 partials in global memory summed by a second kernel.
//  * Every wait is bounded; on timeout the kernel records BSF8_ERR_TIMEOUT, drains its
//    own copies in flight and skips its stores.
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <algorithm>

namespace bsf8 {

struct GemmParams {
    const uint16_t *x;
    long long ldx;
    const uint8_t *w8;
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S;
    int mode;
    int stages;
    int chunk_cols;
    unsigned long long timeout_ns;
    int skip_loads;
    int *status;
};

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ uint4 ld_cg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 lds_v4(const uint8_t *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

template <int NT8>
__global__ void __launch_bounds__(kGemmThreads) gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr int MT = NT8 * 8;
    extern __shared__ __align__(128) uint8_t smem[];

    const int ring_bytes = max(p.stages * kStageBytes, kConsumerWarps * kBN * MT * 4);
    const int nkb = p.chunk_cols / 32;
    const int exps_bytes = (2 * nkb + 15) & ~15;
    uint8_t *ring = smem;
    float *red = reinterpret_cast<float *>(smem);  // reused after the main loop
    float *part = reinterpret_cast<float *>(smem + ring_bytes);
    uint8_t *exps = smem + ring_bytes + kBN * MT * 4;
    uint64_t *full = reinterpret_cast<uint64_t *>(exps + exps_bytes);
    uint64_t *empty = full + kMaxStages;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kBN;
    const int g = blockIdx.y % p.G;
    const int mbase = (blockIdx.y / p.G) * MT;
    const int s = blockIdx.z;
    const int k_lo = min(p.K, s * p.chunk_cols);
    const int k_hi = min(p.K, k_lo + p.chunk_cols);
    const int T = (k_hi - k_lo + kStageK - 1) / kStageK;
    const int rows = min(kBN, p.N - n0);
    const int mrows = min(MT, p.M - mbase);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();

    int err = 0;
    int issued = 0;  // stages the producer has armed (meaningful in the producer warp)
    float acc[4][NT8][4];  // consumer accumulators: slab x token tile x fragment
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NT8; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.0f;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const uint8_t *wbase = p.w8 + ((size_t)g * p.N + n0) * p.K;
        if (!p.skip_loads) {
            const int pf = min(k_hi - k_lo, kPrefetchCols);
            if (pf > 0)
                for (int r = lane; r < rows; r += 32) prefetch_l2(wbase + (size_t)r * p.K + k_lo, pf);
        }
        pdl_wait();
        if (!p.skip_loads) {
            for (int t = 0; t < T; ++t) {
                const int slot = t % p.stages;
                if (t >= p.stages) {
                    int ok = 1;
                    if (lane == 0)
                        ok = mbar_wait_bounded(&empty[slot], ((t / p.stages) - 1) & 1, p.timeout_ns);
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok) {
                        err = 1;
                        break;
                    }
                }
                const int k0 = k_lo + t * kStageK;
                const int kw = min(kStageK, k_hi - k0);
                if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(rows * kw));
                __syncwarp();
                uint8_t *dst = ring + slot * kStageBytes;
                for (int r = lane; r < rows; r += 32)
                    bulk_g2s(dst + r * kRowPitch, wbase + (size_t)r * p.K + k0, (uint32_t)kw, &full[slot]);
                issued = t + 1;
            }
        }
    }
    else {
        // ------------------------------------------------------------ consumers
        pdl_wait();
        const int kb_lo = k_lo / 32;
        const int nkb_s = (k_hi - k_lo) / 32;
        const int nbr = (rows + 31) / 32;
        for (int i = threadIdx.x; i < nbr * nkb_s; i += kConsumerWarps * 32) {
            const int rb = i / nkb_s, j = i - rb * nkb_s;
            exps[rb * nkb + j] =
                p.ex[((size_t)g * (p.N / 32) + n0 / 32 + rb) * (p.K / 32) + kb_lo + j];
        }
        consumer_bar();

        const int q = lane & 3;
        const size_t xrow0 = (size_t)g * p.K;
        for (int t = 0; t < T; ++t) {
            const int slot = t % p.stages;
            const int wk0 = k_lo + t * kStageK + warp * 64;  // this warp's 64 columns
            const int kcol = wk0 + 16 * q;                   // this thread's 16 columns
            const bool valid = kcol < k_hi;

            // token operand: 16 bf16 of x[m][kcol .. kcol+15] per n8 tile (L2 only, so a
            // value written by the previous kernel is always seen)
            uint32_t xr[NT8][8];
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                const int m = mbase + j * 8 + (lane >> 2);
                uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
                if (valid && m < p.M) {
                    const uint16_t *src = p.x + (size_t)m * p.ldx + xrow0 + kcol;
                    a = ld_cg_v4(src);
                    b = ld_cg_v4(src + 8);
                }
                xr[j][0] = a.x; xr[j][1] = a.y; xr[j][2] = a.z; xr[j][3] = a.w;
                xr[j][4] = b.x; xr[j][5] = b.y; xr[j][6] = b.z; xr[j][7] = b.w;
            }

            const bool got = mbar_wait_bounded(&full[slot], (t / p.stages) & 1, p.timeout_ns);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                err = 1;
                break;
            }

            if (wk0 < k_hi) {
                const uint8_t *stage = ring + slot * kStageBytes + warp * 64 + 16 * q;
                const int kb_local = (kcol - k_lo) >> 5;
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    if (sl * 16 >= rows) break;
                    const int r = sl * 16 + (lane >> 2);
                    uint4 wa = make_uint4(0, 0, 0, 0), wb = make_uint4(0, 0, 0, 0);
                    uint32_t e_byte = 127;
                    if (valid) {
                        wa = lds_v4(stage + r * kRowPitch);
                        wb = lds_v4(stage + (r + 8) * kRowPitch);
                        e_byte = exps[(sl >> 1) * nkb + kb_local];
                    }
                    const Scale sc = make_scale(e_byte);
                    const uint32_t ua[4] = {wa.x, wa.y, wa.z, wa.w};
                    const uint32_t ub[4] = {wb.x, wb.y, wb.z, wb.w};
                    const uint32_t nanm = nan_code_mask(wa.x) | nan_code_mask(wa.y) |
                                          nan_code_mask(wa.z) | nan_code_mask(wa.w) |
                                          nan_code_mask(wb.x) | nan_code_mask(wb.y) |
                                          nan_code_mask(wb.z) | nan_code_mask(wb.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t alo, ahi, blo, bhi;
                        rebuild4(ua[j], sc, alo, ahi);  // row r:   columns 16q+4j+{0,1},{2,3}
                        rebuild4(ub[j], sc, blo, bhi);  // row r+8: same columns
                        if (nanm) {
                            patch_nan_codes(ua[j], alo, ahi);
                            patch_nan_codes(ub[j], blo, bhi);
                        }
#pragma unroll
                        for (int jj = 0; jj < NT8; ++jj)
                            mma_bf16_16816(acc[sl][jj], alo, blo, ahi, bhi, xr[jj][2 * j],
                                           xr[jj][2 * j + 1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }

    // ---------------------------------------------------------------- epilogue
    const int cta_err = __syncthreads_or(err);
    if (cta_err) {
        // Let every copy this CTA issued land before its shared memory is released,
        // then report; no output is written.
        if (warp == kConsumerWarps && lane == 0) {
            for (int slot = 0; slot < p.stages; ++slot) {
                int last = -1;
                for (int t = slot; t < issued; t += p.stages) last = t;
                if (last >= 0)
                    (void)mbar_wait_bounded(&full[slot], (last / p.stages) & 1, p.timeout_ns);
            }
            report_timeout(p.status);
        }
        __syncthreads();
        if (p.mode == kModeCluster) {  // the other CTAs of the cluster still meet here
            cluster_sync();
            cluster_sync();
        }
        return;
    }

    // Per-warp partial sums -> red[warp][row][token]; then summed in warp order.
    if (warp < kConsumerWarps) {
        const int q = lane & 3;
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
#pragma unroll
            for (int jj = 0; jj < NT8; ++jj) {
                const int row = sl * 16 + (lane >> 2);
                const int col = jj * 8 + 2 * q;
                float *d0 = red + ((size_t)warp * kBN + row) * MT + col;
                float *d1 = d0 + 8 * MT;
                *reinterpret_cast<float2 *>(d0) = make_float2(acc[sl][jj][0], acc[sl][jj][1]);
                *reinterpret_cast<float2 *>(d1) = make_float2(acc[sl][jj][2], acc[sl][jj][3]);
            }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kBN * MT; i += kGemmThreads) {
        float v = red[i];
        v = v + red[1 * kBN * MT + i];
        v = v + red[2 * kBN * MT + i];
        v = v + red[3 * kBN * MT + i];
        part[i] = v;
    }
    __syncthreads();

    // part[row][token] -> outputs.  Index i walks rows fastest so stores to y / P are
    // contiguous in n.
    const int total = rows * mrows;
    if (p.mode == kModeDirect) {
        for (int i = threadIdx.x; i < total; i += kGemmThreads) {
            const int m = i / rows, row = i - m * rows;
            p.y[((size_t)(mbase + m) * p.G + g) * p.N + n0 + row] = f32_to_bf16_rn(part[row * MT + m]);
        }
    } else if (p.mode == kModePartials) {
        for (int i = threadIdx.x; i < total; i += kGemmThreads) {
            const int m = i / rows, row = i - m * rows;
            p.partials[(((size_t)s * p.M + mbase + m) * p.G + g) * p.N + n0 + row] = part[row * MT + m];
        }
    } else {
        // Cluster of the S splits of this tile (cluster rank == split index): after all
        // partials are in shared memory, CTA s sums its share of the tile's outputs over
        // ranks 0, 1, ..., S-1 in that order, reading the others' shared memory.
        cluster_sync();
        const int per = (total + p.S - 1) / p.S;
        const int lo = s * per, hi = min(total, lo + per);
        for (int i = lo + (int)threadIdx.x; i < hi; i += kGemmThreads) {
            const int m = i / rows, row = i - m * rows;
            const float *src = part + row * MT + m;
            float v = ld_cluster_f32(map_to_rank(src, 0));
            for (int r = 1; r < p.S; ++r) v = v + ld_cluster_f32(map_to_rank(src, (uint32_t)r));
            p.y[((size_t)(mbase + m) * p.G + g) * p.N + n0 + row] = f32_to_bf16_rn(v);
        }
        cluster_sync();  // keep this CTA's shared memory alive until the others are done
    }
}

// -------------------------------------------------------- fixed-order split-K sum
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

// ------------------------------------------------------------------- host side

int auto_split(int M, int N, int K, int G) {
    const int nt8 = std::min(4, (M + 7) / 8);
    const int m_chunks = (M + 8 * nt8 - 1) / (8 * nt8);
    const long long tiles = (long long)((N + kBN - 1) / kBN) * G * m_chunks;
    const int smax = std::max(1, std::min(kMaxClusterSplits, K / 32));
    for (int S = 1; S <= smax; ++S)
        if (tiles * S >= kTargetCtas) return S;
    return smax;
}

GemmPlan plan_gemm(int M, int N, int K, int G, int S, int mode) {
    GemmPlan pl;
    pl.S = S;
    pl.mode = mode;
    pl.nt8 = std::min(4, (M + 7) / 8);
    pl.m_chunks = (M + 8 * pl.nt8 - 1) / (8 * pl.nt8);
    const int nkb = K / 32;
    pl.chunk_cols = ((nkb + S - 1) / S) * 32;
    pl.stages = std::max(1, std::min(kMaxStages, (pl.chunk_cols + kStageK - 1) / kStageK));
    const int MT = 8 * pl.nt8;
    const size_t ring = std::max((size_t)pl.stages * kStageBytes, (size_t)kConsumerWarps * kBN * MT * 4);
    const size_t exps = (size_t)((2 * (pl.chunk_cols / 32) + 15) & ~15);
    pl.smem_bytes = ring + (size_t)kBN * MT * 4 + exps + 2 * kMaxStages * sizeof(uint64_t);
    return pl;
}

namespace {

template <int NT8>
cudaError_t launch_nt8(const GemmPlan &pl, const GemmParams &prm, cudaStream_t stream,
                       const Options &opt) {
    static int configured[64] = {0};  // per device: dynamic shared memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(gemm_kernel<NT8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((prm.N + kBN - 1) / kBN), (unsigned)(prm.G * pl.m_chunks),
                       (unsigned)pl.S);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (pl.mode == kModeCluster) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = (unsigned)pl.S;
        ++na;
    }
    if (opt.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<NT8>, prm);
}

}  // namespace

cudaError_t launch_gemm(const GemmPlan &pl, const void *x, long long ldx, const uint8_t *w8,
                        const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                        cudaStream_t stream) {
    const Options opt = options();
    GemmParams prm;
    prm.x = static_cast<const uint16_t *>(x);
    prm.ldx = ldx;
    prm.w8 = w8;
    prm.ex = ex;
    prm.y = static_cast<uint16_t *>(y);
    prm.partials = partials;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.G = G;
    prm.S = pl.S;
    prm.mode = pl.mode;
    prm.stages = pl.stages;
    prm.chunk_cols = pl.chunk_cols;
    prm.timeout_ns = opt.timeout_ns;
    prm.skip_loads = opt.skip_loads;
    prm.status = status_word();
    if (!prm.status) return cudaErrorInvalidSymbol;
    switch (pl.nt8) {
        case 1: return launch_nt8<1>(pl, prm, stream, opt);
        case 2: return launch_nt8<2>(pl, prm, stream, opt);
        case 3: return launch_nt8<3>(pl, prm, stream, opt);
        default: return launch_nt8<4>(pl, prm, stream, opt);
    }
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
