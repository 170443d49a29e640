// bsf8_stream.cu -- the weight-streaming GEMM kernel for M <= 32 token rows per pass.
//
//   y[m][g][n] = bf16( sum_{s=0..S-1} P[s][m][g][n] ),  summed s = 0, 1, ... in fp32,
//   W[g][n][k] = bf16( e4m3(w8[g][n][k]) * 2^(exp[g][n/32][k/32] - 127) ).
//
// Page: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- _wo_a_partial_w8() and
// _wo_a_mid_kernel() with their fixed-order split-K sums.
//
// At M <= 8 the layer does 2*M flops per weight byte: it is bound by HBM bandwidth, and
// the work per byte (rebuild + MMA issue) must stay small enough for the SMs to keep up.
// Design:
//  * The unit of work is a warp task: one slab of 16 weight rows x a column range inside
//    one split.  A warp loads its rows with 128-bit global loads straight into registers
//    in the layout of the m16n8k16 A fragment (thread q of a quad owns 32 contiguous
//    columns of rows r and r+8 per 128-column step; the k order inside each MMA is
//    permuted identically for x), double-buffered over steps, so a call's bytes are in
//    flight at once across all warps; no shared-memory staging, no barriers.
//  * Codes are rebuilt exactly to bf16 in registers (rebuild4: two byte permutes, shift,
//    mask, one bf16x2 multiply per pair); e4m3 NaN codes are detected from the rebuilt
//    magnitude bits with one add per word and patched on a cold path.
//  * Before the programmatic-dependent-launch wait a warp only prefetches its rows into
//    L2 (coherent, so always safe); x is read and y written after the wait.
//  * Partial sums: per task in registers; the tasks of a split are summed in task order,
//    the splits in split order -- inside the CTA (shared memory) when a slab's tasks fit
//    in 8 warps, across a cluster of up to 8 CTAs (distributed shared memory) otherwise,
//    or written as fp32 partials P[s] for the separate fixed-order reduce.
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <algorithm>

namespace bsf8 {

struct StreamParams {
    const uint16_t *x;
    long long ldx;
    const uint8_t *w8;
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S;
    int chunk_cols;   // columns per split (multiple of 32)
    int kt;           // columns per task (multiple of the step width)
    int tps;          // tasks per split
    int spc;          // slabs per CTA (in-CTA mode)
    int cluster;      // CTAs per slab (cluster mode), else 1
    int spl;          // whole splits per CTA (partials mode)
    int cps;          // CTAs per slab (partials mode)
    int mode;         // kStreamInCta, kStreamCluster, kStreamPartials
};

constexpr int kStreamWarps = 8;
constexpr int kStreamThreads = kStreamWarps * 32;

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Rebuilds 4 codes and flags e4m3 NaN codes: after the shift-and-mask a NaN code has
// magnitude bits 0x07F0, the only pattern for which adding 0x0010 carries into bit 11.
__device__ __forceinline__ void rebuild4_flag(uint32_t w, const Scale &s, uint32_t &lo,
                                              uint32_t &hi, uint32_t &flag) {
    uint32_t t0, t1;
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w));
    t0 = (t0 << 4) & 0x87F087F0u;
    t1 = (t1 << 4) & 0x87F087F0u;
    flag |= (t0 + 0x00100010u) | (t1 + 0x00100010u);
    lo = bf16x2_mul(t0, s.s1);
    hi = bf16x2_mul(t1, s.s1);
    if (s.two) {
        lo = bf16x2_mul(lo, s.s2);
        hi = bf16x2_mul(hi, s.s2);
    }
}

// Step width: 128 columns (thread covers 32) for up to two token tiles, else 64 (16).
template <int NT8>
struct StepCfg {
    static constexpr int KS = NT8 <= 2 ? 128 : 64;
    static constexpr int TC = KS / 4;      // columns per thread per step
    static constexpr int WV = TC / 16;     // 16-byte weight vectors per row per step
    static constexpr int XV = TC / 8;      // 16-byte x vectors per token row per step
    static constexpr int MMAS = TC / 4;    // MMAs per step (each takes 4 columns/thread)
};

template <int NT8>
struct StepBuf {
    uint4 wa[StepCfg<NT8>::WV];           // row r
    uint4 wb[StepCfg<NT8>::WV];           // row r + 8
    uint4 xv[NT8][StepCfg<NT8>::XV];      // token rows of each n8 tile
    uint32_t e;                           // exponent byte of this thread's block
    bool valid;
};

template <int NT8>
__device__ __forceinline__ void load_step(StepBuf<NT8> &b, const StreamParams &p, int g, int n_r,
                                          int mbase, int lane, int kcol, int k1) {
    using C = StepCfg<NT8>;
    b.valid = kcol < k1;
    if (b.valid) {
        const uint8_t *ra = p.w8 + ((size_t)g * p.N + n_r) * p.K + kcol;
        const uint8_t *rb = ra + (size_t)8 * p.K;
#pragma unroll
        for (int v = 0; v < C::WV; ++v) {
            b.wa[v] = ldg_stream(ra + 16 * v);
            b.wb[v] = ldg_stream(rb + 16 * v);
        }
        b.e = ldg_u8(p.ex + ((size_t)g * (p.N / 32) + n_r / 32) * (p.K / 32) + kcol / 32);
#pragma unroll
        for (int j = 0; j < NT8; ++j) {
            const int m = mbase + j * 8 + (lane >> 2);
            if (m < p.M) {
                const uint16_t *src = p.x + (size_t)m * p.ldx + (size_t)g * p.K + kcol;
#pragma unroll
                for (int v = 0; v < C::XV; ++v) b.xv[j][v] = ldg_v4(src + 8 * v);
            } else {
#pragma unroll
                for (int v = 0; v < C::XV; ++v) b.xv[j][v] = make_uint4(0, 0, 0, 0);
            }
        }
    } else {
#pragma unroll
        for (int v = 0; v < C::WV; ++v) b.wa[v] = b.wb[v] = make_uint4(0, 0, 0, 0);
        b.e = 127;
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
            for (int v = 0; v < C::XV; ++v) b.xv[j][v] = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ uint32_t u4_word(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int NT8>
__device__ __forceinline__ void compute_step(const StepBuf<NT8> &b, float (&acc)[2][NT8][4]) {
    using C = StepCfg<NT8>;
    const Scale sc = make_scale(b.e);
    uint32_t flag = 0;
    uint32_t alo[C::MMAS], ahi[C::MMAS], blo[C::MMAS], bhi[C::MMAS];
#pragma unroll
    for (int j = 0; j < C::MMAS; ++j) {
        rebuild4_flag(u4_word(b.wa[j / 4], j % 4), sc, alo[j], ahi[j], flag);
        rebuild4_flag(u4_word(b.wb[j / 4], j % 4), sc, blo[j], bhi[j], flag);
    }
    if (flag & 0x08000800u) {  // an e4m3 NaN code is present (cold path)
#pragma unroll
        for (int j = 0; j < C::MMAS; ++j) {
            patch_nan_codes(u4_word(b.wa[j / 4], j % 4), alo[j], ahi[j]);
            patch_nan_codes(u4_word(b.wb[j / 4], j % 4), blo[j], bhi[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < C::MMAS; ++j)
#pragma unroll
        for (int t = 0; t < NT8; ++t) {
            // thread's x words: word i holds columns (2i, 2i+1) of its TC columns
            const uint32_t b0 = u4_word(b.xv[t][(2 * j) / 4], (2 * j) % 4);
            const uint32_t b1 = u4_word(b.xv[t][(2 * j + 1) / 4], (2 * j + 1) % 4);
            mma_bf16_16816(acc[j & 1][t], alo[j], blo[j], ahi[j], bhi[j], b0, b1);
        }
}

template <int NT8>
__global__ void __launch_bounds__(kStreamThreads) stream_kernel(const __grid_constant__ StreamParams p) {
    using C = StepCfg<NT8>;
    constexpr int MT = 8 * NT8;
    __shared__ __align__(16) float red[kStreamWarps][16][MT];  // per-warp task partials

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q = lane & 3;
    const int g = blockIdx.y % p.G;
    const int mbase = (blockIdx.y / p.G) * MT;
    const int nslabs = p.N / 16;
    const int tslab = p.S * p.tps;

    // ---- this warp's task: slab, split s, task u within the split
    int slab, s, u;
    bool active;
    if (p.mode == kStreamCluster) {
        slab = blockIdx.x / p.cluster;
        const int tau = (blockIdx.x % p.cluster) * kStreamWarps + warp;
        s = tau / p.tps;
        u = tau % p.tps;
        active = tau < tslab;
    } else if (p.mode == kStreamPartials) {
        slab = blockIdx.x / p.cps;
        s = (blockIdx.x % p.cps) * p.spl + warp / p.tps;
        u = warp % p.tps;
        active = warp < p.spl * p.tps && s < p.S;
    } else {
        slab = blockIdx.x * p.spc + warp / tslab;
        s = (warp % tslab) / p.tps;
        u = (warp % tslab) % p.tps;
        active = warp < p.spc * tslab && slab < nslabs;
    }
    int k0 = 0, k1 = 0;
    if (active) {
        const int s_lo = min(p.K, s * p.chunk_cols);
        const int s_hi = min(p.K, s_lo + p.chunk_cols);
        k0 = min(s_hi, s_lo + u * p.kt);
        k1 = min(s_hi, k0 + p.kt);
    }
    const int n_r = slab * 16 + (lane >> 2);  // this thread's rows: n_r and n_r + 8

    pdl_trigger();
    if (active && k1 > k0 && (lane >> 2) < 2) {
        // Lanes 0..7 prefetch the warp's 16 weight rows into L2 before the dependency wait.
        const int r = slab * 16 + lane * 2;
        const uint8_t *base = p.w8 + ((size_t)g * p.N + r) * p.K + k0;
        prefetch_l2(base, (uint32_t)(k1 - k0));
        prefetch_l2(base + p.K, (uint32_t)(k1 - k0));
    }
    pdl_wait();

    float acc[2][NT8][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int t = 0; t < NT8; ++t)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][t][c] = 0.0f;

    if (active && k1 > k0) {
        const int nsteps = (k1 - k0 + C::KS - 1) / C::KS;
        StepBuf<NT8> b0, b1;
        load_step<NT8>(b0, p, g, n_r, mbase, lane, k0 + q * C::TC, k1);
        int t = 0;
        for (; t + 2 <= nsteps; t += 2) {
            load_step<NT8>(b1, p, g, n_r, mbase, lane, k0 + (t + 1) * C::KS + q * C::TC, k1);
            compute_step<NT8>(b0, acc);
            if (t + 2 < nsteps)
                load_step<NT8>(b0, p, g, n_r, mbase, lane, k0 + (t + 2) * C::KS + q * C::TC, k1);
            compute_step<NT8>(b1, acc);
        }
        if (t < nsteps) compute_step<NT8>(b0, acc);
    }

    // ---- task partial -> shared memory (rows = weight rows, columns = tokens)
#pragma unroll
    for (int t = 0; t < NT8; ++t) {
        const int row = lane >> 2, col = t * 8 + 2 * q;
        *reinterpret_cast<float2 *>(&red[warp][row][col]) =
            make_float2(acc[0][t][0] + acc[1][t][0], acc[0][t][1] + acc[1][t][1]);
        *reinterpret_cast<float2 *>(&red[warp][row + 8][col]) =
            make_float2(acc[0][t][2] + acc[1][t][2], acc[0][t][3] + acc[1][t][3]);
    }
    const int mrows = min(MT, p.M - mbase);

    if (p.mode == kStreamInCta) {
        __syncthreads();
        // per output: P_s = sum_u task(s,u) in task order; y = sum_s P_s in split order
        const int per_slab = 16 * mrows;
        for (int i = threadIdx.x; i < p.spc * per_slab; i += kStreamThreads) {
            const int sl = i / per_slab, rem = i - sl * per_slab;
            const int m = rem / 16, row = rem - m * 16;
            const int sb = blockIdx.x * p.spc + sl;
            if (sb >= nslabs) continue;
            const int w0 = sl * tslab;
            float y = 0.0f;
            for (int ss = 0; ss < p.S; ++ss) {
                float ps = red[w0 + ss * p.tps][row][m];
                for (int uu = 1; uu < p.tps; ++uu) ps = ps + red[w0 + ss * p.tps + uu][row][m];
                y = ss == 0 ? ps : y + ps;
            }
            p.y[((size_t)(mbase + m) * p.G + g) * p.N + sb * 16 + row] = f32_to_bf16_rn(y);
        }
    } else if (p.mode == kStreamPartials) {
        __syncthreads();
        const int per_split = 16 * mrows;
        for (int i = threadIdx.x; i < p.spl * per_split; i += kStreamThreads) {
            const int ls = i / per_split, rem = i - ls * per_split;
            const int m = rem / 16, row = rem - m * 16;
            const int ss = (blockIdx.x % p.cps) * p.spl + ls;
            if (ss >= p.S) continue;
            float ps = red[ls * p.tps][row][m];
            for (int uu = 1; uu < p.tps; ++uu) ps = ps + red[ls * p.tps + uu][row][m];
            p.partials[(((size_t)ss * p.M + mbase + m) * p.G + g) * p.N + slab * 16 + row] = ps;
        }
    } else {
        // Cluster of the slab's CTAs (rank c holds tasks 8c .. 8c+7): each CTA sums a share
        // of the slab's outputs, reading every task partial in task order through DSMEM.
        cluster_sync();
        const int total = 16 * mrows;
        const int c = blockIdx.x % p.cluster;
        const int per = (total + p.cluster - 1) / p.cluster;
        const int lo = c * per, hi = min(total, lo + per);
        for (int i = lo + (int)threadIdx.x; i < hi; i += kStreamThreads) {
            const int m = i / 16, row = i - m * 16;
            float y = 0.0f;
            for (int ss = 0; ss < p.S; ++ss) {
                float ps = 0.0f;
                for (int uu = 0; uu < p.tps; ++uu) {
                    const int tau = ss * p.tps + uu;
                    const float v = ld_cluster_f32(
                        map_to_rank(&red[tau % kStreamWarps][row][m], (uint32_t)(tau / kStreamWarps)));
                    ps = uu == 0 ? v : ps + v;
                }
                y = ss == 0 ? ps : y + ps;
            }
            p.y[((size_t)(mbase + m) * p.G + g) * p.N + slab * 16 + row] = f32_to_bf16_rn(y);
        }
        cluster_sync();
    }
}

// ------------------------------------------------------------------- host side

StreamPlan plan_stream(int M, int N, int K, int G, int S, bool partials) {
    StreamPlan pl{};
    pl.nt8 = std::min(4, (M + 7) / 8);
    pl.m_chunks = (M + 8 * pl.nt8 - 1) / (8 * pl.nt8);
    const int ks = pl.nt8 <= 2 ? 128 : 64;
    const int nkb = K / 32;
    pl.S = S;
    pl.chunk_cols = ((nkb + S - 1) / S) * 32;
    // Task width: at least two steps, and at most 8 tasks per split.
    int kt = std::max(2 * ks, (pl.chunk_cols + 7) / 8);
    kt = (kt + ks - 1) / ks * ks;
    pl.kt = kt;
    pl.tps = (pl.chunk_cols + kt - 1) / kt;
    const int tslab = S * pl.tps;
    const int nslabs = N / 16;
    pl.spc = 1;
    pl.cluster = 1;
    pl.spl = 1;
    pl.cps = 1;
    if (partials || tslab > kStreamWarps * kMaxClusterSplits) {
        pl.mode = kStreamPartials;
        pl.spl = std::max(1, kStreamWarps / pl.tps);
        pl.cps = (S + pl.spl - 1) / pl.spl;
        pl.grid_x = nslabs * pl.cps;
    } else if (tslab <= kStreamWarps) {
        pl.mode = kStreamInCta;
        pl.spc = kStreamWarps / tslab;
        pl.grid_x = (nslabs + pl.spc - 1) / pl.spc;
    } else {
        pl.mode = kStreamCluster;
        pl.cluster = (tslab + kStreamWarps - 1) / kStreamWarps;
        pl.grid_x = nslabs * pl.cluster;
    }
    return pl;
}

namespace {
template <int NT8>
cudaError_t launch_stream_nt8(const StreamPlan &pl, const StreamParams &prm, cudaStream_t stream,
                              const Options &opt) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid_x, (unsigned)(prm.G * pl.m_chunks), 1);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (pl.mode == kStreamCluster) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)pl.cluster;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (opt.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, stream_kernel<NT8>, prm);
}
}  // namespace

cudaError_t launch_stream(const StreamPlan &pl, const void *x, long long ldx, const uint8_t *w8,
                          const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                          cudaStream_t stream) {
    const Options opt = options();
    StreamParams prm;
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
    prm.chunk_cols = pl.chunk_cols;
    prm.kt = pl.kt;
    prm.tps = pl.tps;
    prm.spc = pl.spc;
    prm.cluster = pl.cluster;
    prm.spl = pl.spl;
    prm.cps = pl.cps;
    prm.mode = pl.mode;
    switch (pl.nt8) {
        case 1: return launch_stream_nt8<1>(pl, prm, stream, opt);
        case 2: return launch_stream_nt8<2>(pl, prm, stream, opt);
        case 3: return launch_stream_nt8<3>(pl, prm, stream, opt);
        default: return launch_stream_nt8<4>(pl, prm, stream, opt);
    }
}

}  // namespace bsf8
