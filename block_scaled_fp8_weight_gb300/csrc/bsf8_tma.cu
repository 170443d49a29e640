// bsf8_tma.cu -- the default GEMM kernel for up to 16 token rows per pass.
//
//   y[m][g][n] = bf16( sum_{s=0..S-1} P[s][m][g][n] ),  summed s = 0, 1, ... in fp32,
//   W[g][n][k] = bf16( e4m3(w8[g][n][k]) * 2^(exp[g][n/32][k/32] - 127) ).
//
// Page: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- _wo_a_partial_w8() and
// _wo_a_mid_kernel() with their fixed-order split-K sums.
//
// Work decomposition as in bsf8_stream.cu: a warp task is 16 weight rows x a column range
// inside one split; a block holds 8 consumer warps (a group of tasks) and walks groups
// persistently.  What changes is how the weights arrive.  A producer warp issues, per
// pipeline stage, one 2-D TMA copy (cp.async.bulk.tensor) of 16 rows x 128 columns for
// each consumer warp into a shared-memory ring (128-byte swizzle, so the consumers'
// 128-bit reads are bank-conflict free), completing on the stage's mbarrier.  The
// consumer warps do no address arithmetic or copy issue for the weights: they wait for
// the stage, rebuild their 16 x 128 codes exactly in registers, run their MMAs and free
// the stage.  The twin is a static parameter, so the producer starts streaming at once,
// before the programmatic-dependent-launch wait; consumers read x and write y after it.
// Every wait is bounded: on timeout the block records BSF8_ERR_TIMEOUT, stores nothing and
// returns.
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <cuda.h>

#include <algorithm>
#include <mutex>

namespace bsf8 {

namespace {

constexpr int kConsumers = 8;
constexpr int kTmaThreads = (kConsumers + 1) * 32;
constexpr int kKS = 128;                    // columns per stage and task step
constexpr int kBoxBytes = 16 * kKS;         // one warp's box: 16 rows x 128 columns
constexpr int kStageBytes2 = kConsumers * kBoxBytes;
constexpr int kDepth = 6;                   // stages in the ring
constexpr int kRingBytes = kDepth * kStageBytes2;

struct TmaParams {
    CUtensorMap wmap;  // w8 as a [G*N rows][K columns] byte matrix, box 16 x 128
    const uint16_t *x;
    long long ldx;
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S;
    int chunk_cols, kt, tps, spc, cluster, spl, cps, mode;
    unsigned long long timeout_ns;
    int skip_loads;
    int *status;
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

__device__ __forceinline__ uint4 ldg_v4x(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u8x(const uint8_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t bf16x2_max_abs2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void spread4x(uint32_t w, uint32_t &t0, uint32_t &t1) {
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w));
    t0 = (t0 << 4) & 0x87F087F0u;
    t1 = (t1 << 4) & 0x87F087F0u;
}

__device__ __forceinline__ bool nan_code_seen(uint32_t mx) {
    return (mx & 0x7FFFu) >= 0x07F0u || ((mx >> 16) & 0x7FFFu) >= 0x07F0u;
}

// A warp's task: split s, task u of the split, columns [k0, k1), its slab in the block's
// first group (slab0) and the slab stride between groups; the block's group count.
struct Task {
    int s, u, k0, k1, slab0, slab_step, ngroups;
    bool active;
};

__device__ __forceinline__ Task task_of(const TmaParams &p, int w) {
    Task t;
    const int nslabs = p.N / 16;
    const int tslab = p.S * p.tps;
    t.ngroups = 1;
    t.slab_step = 0;
    if (p.mode == kStreamCluster) {
        t.slab0 = blockIdx.x / p.cluster;
        const int tau = (blockIdx.x % p.cluster) * kConsumers + w;
        t.s = tau / p.tps;
        t.u = tau % p.tps;
        t.active = tau < tslab;
    } else if (p.mode == kStreamPartials) {
        t.slab0 = blockIdx.x / p.cps;
        t.s = (blockIdx.x % p.cps) * p.spl + w / p.tps;
        t.u = w % p.tps;
        t.active = w < p.spl * p.tps && t.s < p.S;
    } else {
        const int groups_total = (nslabs + p.spc - 1) / p.spc;
        t.ngroups = (int)blockIdx.x < groups_total
                        ? (groups_total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        t.slab0 = blockIdx.x * p.spc + w / tslab;
        t.slab_step = gridDim.x * p.spc;
        t.s = (w % tslab) / p.tps;
        t.u = (w % tslab) % p.tps;
        t.active = w < p.spc * tslab;
    }
    t.k0 = t.k1 = 0;
    if (t.active) {
        const int s_lo = min(p.K, t.s * p.chunk_cols);
        const int s_hi = min(p.K, s_lo + p.chunk_cols);
        t.k0 = min(s_hi, s_lo + t.u * p.kt);
        t.k1 = min(s_hi, t.k0 + p.kt);
    }
    return t;
}

}  // namespace

namespace {

template <int NT8>
struct XTile {
    uint4 v[NT8][4];  // 32 bf16 of x per token row: this thread's columns of the step
    uint32_t e;       // exponent byte of the thread's 32x32 block
};

// Byte offsets of this thread's two 16-byte units of row r and r+8 in a 16 x 128 box
// written with the 128-byte swizzle (unit u of row r sits at unit u ^ (r % 8)).
struct BoxOffs {
    int a0, a1, b0, b1;
};

__device__ __forceinline__ BoxOffs box_offsets(int r, int q) {
    BoxOffs o;
    o.a0 = r * 128 + (((2 * q) ^ (r & 7)) << 4);
    o.a1 = r * 128 + (((2 * q + 1) ^ (r & 7)) << 4);
    o.b0 = o.a0 + 8 * 128;
    o.b1 = o.a1 + 8 * 128;
    return o;
}

// One 128-column step of a warp task: 8 MMAs per token tile.  mxa / mxb keep the largest
// rebuilt magnitude of rows r / r+8 (an e4m3 NaN code rebuilds to 0x07F0, above every
// finite code's 0x07E0; such rows are set to NaN at the end of the group).
template <int NT8, bool TWO>
__device__ __forceinline__ void tma_step(const uint8_t *box, const BoxOffs &o, bool valid,
                                         const XTile<NT8> &xt,
                                         float (&acc)[NT8 == 1 ? 2 : 1][NT8][4],
                                         uint32_t &mxa, uint32_t &mxb) {
    constexpr int ACC = NT8 == 1 ? 2 : 1;
    uint4 a[2], b[2];
    if (valid) {
        a[0] = *reinterpret_cast<const uint4 *>(box + o.a0);
        a[1] = *reinterpret_cast<const uint4 *>(box + o.a1);
        b[0] = *reinterpret_cast<const uint4 *>(box + o.b0);
        b[1] = *reinterpret_cast<const uint4 *>(box + o.b1);
    } else {
        a[0] = a[1] = b[0] = b[1] = make_uint4(0, 0, 0, 0);
    }
    const Scale sc = make_scale(xt.e);
    uint32_t s1 = sc.s1, s2 = sc.s2;
    if (TWO) {  // exact for every exponent byte: restore e4m3 * 1, then scale by 2^(e-127)
        s1 = 0x7B807B80u;
        const uint32_t bb = xt.e == 0 ? 0x0040u : (xt.e << 7);
        s2 = bb | (bb << 16);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 &av = a[j / 4], &bv = b[j / 4];
        const int i = j % 4;
        uint32_t t0, t1, u0, u1;
        spread4x(i == 0 ? av.x : i == 1 ? av.y : i == 2 ? av.z : av.w, t0, t1);
        spread4x(i == 0 ? bv.x : i == 1 ? bv.y : i == 2 ? bv.z : bv.w, u0, u1);
        mxa = bf16x2_max_abs2(mxa, bf16x2_max_abs2(t0, t1));
        mxb = bf16x2_max_abs2(mxb, bf16x2_max_abs2(u0, u1));
        uint32_t alo = bf16x2_mul(t0, s1), ahi = bf16x2_mul(t1, s1);
        uint32_t blo = bf16x2_mul(u0, s1), bhi = bf16x2_mul(u1, s1);
        if (TWO) {
            alo = bf16x2_mul(alo, s2);
            ahi = bf16x2_mul(ahi, s2);
            blo = bf16x2_mul(blo, s2);
            bhi = bf16x2_mul(bhi, s2);
        }
#pragma unroll
        for (int t = 0; t < NT8; ++t) {
            // x word 2j holds the thread's columns (4j, 4j+1), word 2j+1 holds (4j+2, 4j+3)
            const uint4 &xv = xt.v[t][j / 2];
            const uint32_t x0 = (j & 1) ? xv.z : xv.x;
            const uint32_t x1 = (j & 1) ? xv.w : xv.y;
            mma_bf16_16816(acc[j % ACC][t], alo, blo, ahi, bhi, x0, x1);
        }
    }
}

// End of a group (consumer threads only).  red[w] holds warp w's task partial; sums them in
// the fixed order (tasks of a split in task order, splits in split order) and stores y, or
// stores the per-split partials.  Stores are skipped when the block met an error.
template <int NT8>
__device__ __forceinline__ void tma_group_epilogue(const TmaParams &p, float (*red)[16][8 * NT8],
                                                   const volatile int *err, int g, int mbase,
                                                   int gslab) {
    constexpr int MT = 8 * NT8;
    const int nslabs = p.N / 16, tslab = p.S * p.tps;
    const int mrows = min(MT, p.M - mbase);
    const int tid = threadIdx.x;  // 0 .. 255
    if (p.mode == kStreamCluster) {
        cluster_sync();
        if (!*err) {
            const int total = 16 * mrows;
            const int c = blockIdx.x % p.cluster;
            const int per = (total + p.cluster - 1) / p.cluster;
            const int lo = c * per, hi = min(total, lo + per);
            for (int i = lo + tid; i < hi; i += kConsumers * 32) {
                const int m = i / 16, row = i - m * 16;
                float y = 0.0f;
                for (int ss = 0; ss < p.S; ++ss) {
                    float ps = 0.0f;
                    for (int uu = 0; uu < p.tps; ++uu) {
                        const int tau = ss * p.tps + uu;
                        const float v = ld_cluster_f32(
                            map_to_rank(&red[tau % kConsumers][row][m], (uint32_t)(tau / kConsumers)));
                        ps = uu == 0 ? v : ps + v;
                    }
                    y = ss == 0 ? ps : y + ps;
                }
                p.y[((size_t)(mbase + m) * p.G + g) * p.N + gslab * 16 + row] = f32_to_bf16_rn(y);
            }
        }
        cluster_sync();  // keep this block's shared memory alive until the others are done
        return;
    }
    consumer_sync();
    if (!*err) {
        if (p.mode == kStreamInCta) {
            const int per_slab = 16 * mrows;
            for (int i = tid; i < p.spc * per_slab; i += kConsumers * 32) {
                const int sl = i / per_slab, rem = i - sl * per_slab;
                const int m = rem / 16, row = rem - m * 16;
                const int sb = gslab + sl;
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
        } else {
            const int per_split = 16 * mrows;
            for (int i = tid; i < p.spl * per_split; i += kConsumers * 32) {
                const int ls = i / per_split, rem = i - ls * per_split;
                const int m = rem / 16, row = rem - m * 16;
                const int ss = (blockIdx.x % p.cps) * p.spl + ls;
                if (ss >= p.S) continue;
                float ps = red[ls * p.tps][row][m];
                for (int uu = 1; uu < p.tps; ++uu) ps = ps + red[ls * p.tps + uu][row][m];
                p.partials[(((size_t)ss * p.M + mbase + m) * p.G + g) * p.N + gslab * 16 + row] = ps;
            }
        }
    }
    consumer_sync();  // red is rewritten by the next group
}

}  // namespace

template <int NT8>
__global__ void __launch_bounds__(kTmaThreads, NT8 == 1 ? 2 : 1)
    tma_kernel(const __grid_constant__ TmaParams p) {
    constexpr int MT = 8 * NT8;
    constexpr int ACC = NT8 == 1 ? 2 : 1;
    extern __shared__ uint8_t dyn_smem[];
    // the swizzled boxes need 1024-byte alignment
    uint8_t *ring = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    __shared__ __align__(16) float red[kConsumers][16][MT];
    __shared__ __align__(8) uint64_t full[kDepth];
    __shared__ __align__(8) uint64_t empty[kDepth];
    __shared__ int s_err;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.y % p.G;
    const int mbase = (blockIdx.y / p.G) * MT;
    const int nslabs = p.N / 16;
    const int nst = p.kt / kKS;  // stages per group
    const Task me = task_of(p, warp < kConsumers ? warp : 0);
    const long long total = (long long)me.ngroups * nst;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDepth; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumers);
        }
        s_err = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();

    long long issued = 0;  // stages armed by the producer (its lane 0)
    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !p.skip_loads && total > 0) {
            Task tk[kConsumers];
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) tk[w] = task_of(p, w);
            int gi = 0, t = 0, slot = 0;
            for (long long T = 0; T < total; ++T) {
                if (T >= kDepth &&
                    !mbar_wait_bounded(&empty[slot], (uint32_t)(((T / kDepth) - 1) & 1), p.timeout_ns)) {
                    s_err = 1;
                    report_timeout(p.status);
                    break;
                }
                uint32_t bytes = 0;
#pragma unroll
                for (int w = 0; w < kConsumers; ++w) {
                    const int slab = tk[w].slab0 + gi * tk[w].slab_step;
                    if (tk[w].active && slab < nslabs && tk[w].k0 + t * kKS < tk[w].k1) bytes += kBoxBytes;
                }
                mbar_arrive_expect_tx(&full[slot], bytes);
                uint8_t *st = ring + slot * kStageBytes2;
#pragma unroll
                for (int w = 0; w < kConsumers; ++w) {
                    const int slab = tk[w].slab0 + gi * tk[w].slab_step;
                    const int col = tk[w].k0 + t * kKS;
                    if (tk[w].active && slab < nslabs && col < tk[w].k1)
                        tma_load_2d(st + w * kBoxBytes, &p.wmap, col, g * p.N + slab * 16, &full[slot]);
                }
                issued = T + 1;
                slot = slot + 1 == kDepth ? 0 : slot + 1;
                if (++t == nst) {
                    t = 0;
                    ++gi;
                }
            }
        }
        __syncwarp();
        if (p.mode == kStreamCluster) {  // the consumers' epilogue meets the cluster twice
            cluster_sync();
            cluster_sync();
        }
    } else {
        // ------------------------------------------------------------ consumers
        pdl_wait();
        const int q = lane & 3, r = lane >> 2;
        const BoxOffs bo = box_offsets(r, q);
        const uint16_t *xsrc[NT8];
#pragma unroll
        for (int tt = 0; tt < NT8; ++tt) {  // token rows >= M read row M-1 (never stored)
            const int m = min(mbase + tt * 8 + r, p.M - 1);
            xsrc[tt] = p.x + (size_t)m * p.ldx + (size_t)g * p.K + me.k0 + q * 32;
        }
        const size_t ebase = (size_t)g * (p.N / 32) * (p.K / 32) + (size_t)((me.k0 + q * 32) / 32);
        // The thread's 32 columns of step t are valid iff they start below k1 (tasks end on
        // a 32-column boundary); its box was loaded iff the step starts below k1.
        auto load_x = [&](XTile<NT8> &xt, int gi, int t) {
            const int slab = me.slab0 + gi * me.slab_step;
            if (me.active && gi < me.ngroups && slab < nslabs && me.k0 + t * kKS + q * 32 < me.k1) {
#pragma unroll
                for (int tt = 0; tt < NT8; ++tt)
#pragma unroll
                    for (int v = 0; v < 4; ++v) xt.v[tt][v] = ldg_v4x(xsrc[tt] + t * kKS + 8 * v);
                xt.e = ldg_u8x(p.ex + ebase + (size_t)(slab / 2) * (p.K / 32) + t * (kKS / 32));
            } else {
#pragma unroll
                for (int tt = 0; tt < NT8; ++tt)
#pragma unroll
                    for (int v = 0; v < 4; ++v) xt.v[tt][v] = make_uint4(0, 0, 0, 0);
                xt.e = 127;
            }
        };

        float acc[ACC][NT8][4];
#pragma unroll
        for (int a = 0; a < ACC; ++a)
#pragma unroll
            for (int tt = 0; tt < NT8; ++tt)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][tt][c] = 0.0f;
        uint32_t mxa = 0, mxb = 0;
        int err = 0;
        XTile<NT8> xa, xb;
        load_x(xa, 0, 0);
        int gi = 0, t = 0, slot = 0;
        for (long long T = 0; T < total; ++T) {
            const int ngi = t + 1 == nst ? gi + 1 : gi, nt = t + 1 == nst ? 0 : t + 1;
            const int slab = me.slab0 + gi * me.slab_step;
            const int col = me.k0 + t * kKS;
            const bool boxed = me.active && slab < nslabs && col < me.k1;   // box loaded for me
            const bool mine = boxed && col + q * 32 < me.k1;                // my 32 columns valid
            if (!err) {
                const bool got = mbar_wait_bounded(&full[slot], (uint32_t)((T / kDepth) & 1), p.timeout_ns);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    err = 1;
                    s_err = 1;
                    if (lane == 0) report_timeout(p.status);
                }
            }
            const uint8_t *box = ring + slot * kStageBytes2 + warp * kBoxBytes;
            if (T & 1) {
                load_x(xa, ngi, nt);
                if (!err && boxed) {
                    if (__any_sync(0xFFFFFFFFu, xb.e > 134u))
                        tma_step<NT8, true>(box, bo, mine, xb, acc, mxa, mxb);
                    else
                        tma_step<NT8, false>(box, bo, mine, xb, acc, mxa, mxb);
                }
            } else {
                load_x(xb, ngi, nt);
                if (!err && boxed) {
                    if (__any_sync(0xFFFFFFFFu, xa.e > 134u))
                        tma_step<NT8, true>(box, bo, mine, xa, acc, mxa, mxb);
                    else
                        tma_step<NT8, false>(box, bo, mine, xa, acc, mxa, mxb);
                }
            }
            __syncwarp();
            if (lane == 0 && !err) mbar_arrive(&empty[slot]);
            slot = slot + 1 == kDepth ? 0 : slot + 1;
            if (nt == 0) {
                // ---- end of group gi: every consumer warp runs this once per group
                uint32_t fa = nan_code_seen(mxa) ? 1u : 0u, fb = nan_code_seen(mxb) ? 1u : 0u;
                fa |= __shfl_xor_sync(0xFFFFFFFFu, fa, 1);
                fa |= __shfl_xor_sync(0xFFFFFFFFu, fa, 2);
                fb |= __shfl_xor_sync(0xFFFFFFFFu, fb, 1);
                fb |= __shfl_xor_sync(0xFFFFFFFFu, fb, 2);
                const float qnan = __uint_as_float(0x7FC00000u);
#pragma unroll
                for (int tt = 0; tt < NT8; ++tt) {
                    float v[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        v[c] = ACC == 2 ? acc[0][tt][c] + acc[ACC - 1][tt][c] : acc[0][tt][c];
                        if ((c < 2 && fa) || (c >= 2 && fb)) v[c] = qnan;
                    }
                    const int colx = tt * 8 + 2 * q;
                    *reinterpret_cast<float2 *>(&red[warp][r][colx]) = make_float2(v[0], v[1]);
                    *reinterpret_cast<float2 *>(&red[warp][r + 8][colx]) = make_float2(v[2], v[3]);
                }
#pragma unroll
                for (int a = 0; a < ACC; ++a)
#pragma unroll
                    for (int tt = 0; tt < NT8; ++tt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[a][tt][c] = 0.0f;
                mxa = mxb = 0;
                const int gslab = p.mode == kStreamInCta ? ((int)blockIdx.x + gi * (int)gridDim.x) * p.spc
                                                         : me.slab0;
                tma_group_epilogue<NT8>(p, red, &s_err, g, mbase, gslab);
            }
            gi = ngi;
            t = nt;
        }
    }

    // After an error, let every copy the producer armed land before the block exits.
    __syncthreads();
    if (s_err && warp == kConsumers && lane == 0) {
        for (int sl = 0; sl < kDepth; ++sl) {
            long long last = -1;
            for (long long T = sl; T < issued; T += kDepth) last = T;
            if (last >= 0) (void)mbar_wait_bounded(&full[sl], (uint32_t)((last / kDepth) & 1), p.timeout_ns);
        }
    }
}

// ------------------------------------------------------------------- host side

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Tensor maps of recently used weights (a map encodes only the address and the shape).
struct MapEntry {
    const void *ptr;
    long long rows;
    int K;
    CUtensorMap map;
};

cudaError_t weight_map(const uint8_t *w8, long long rows, int K, CUtensorMap *out) {
    static std::mutex mu;
    static MapEntry cache[64];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].ptr == w8 && cache[i].rows == rows && cache[i].K == K) {
            *out = cache[i].map;
            return cudaSuccess;
        }
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap m;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kKS, 16u};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w8), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    MapEntry &e = cache[next];
    e.ptr = w8;
    e.rows = rows;
    e.K = K;
    e.map = m;
    next = (next + 1) % 64;
    if (used < 64) ++used;
    *out = m;
    return cudaSuccess;
}

template <int NT8>
cudaError_t launch_tma_nt8(const StreamPlan &pl, const TmaParams &prm, cudaStream_t stream,
                           const Options &opt) {
    const size_t smem = (size_t)kRingBytes + 1024;
    static int configured[64] = {0};
    static int cap[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(tma_kernel<NT8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tma_kernel<NT8>, kTmaThreads, smem);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&cap[dev], std::max(1, sms * std::max(1, per_sm)), __ATOMIC_RELEASE);
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    int gx = pl.grid_x;
    if (pl.mode == kStreamInCta) gx = std::min(gx, __atomic_load_n(&cap[dev], __ATOMIC_ACQUIRE));
    cfg.gridDim = dim3((unsigned)gx, (unsigned)(prm.G * pl.m_chunks), 1);
    cfg.blockDim = dim3(kTmaThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
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
    return cudaLaunchKernelEx(&cfg, tma_kernel<NT8>, prm);
}

}  // namespace

StreamPlan plan_tma(int M, int N, int K, int G, int S, bool partials) {
    StreamPlan pl = plan_stream_ks(M, N, K, G, S, partials, kKS, 2);
    return pl;
}

cudaError_t launch_tma(const StreamPlan &pl, const void *x, long long ldx, const uint8_t *w8,
                       const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                       cudaStream_t stream) {
    const Options opt = options();
    TmaParams prm;
    cudaError_t e = weight_map(w8, (long long)G * N, K, &prm.wmap);
    if (e != cudaSuccess) return e;
    prm.x = static_cast<const uint16_t *>(x);
    prm.ldx = ldx;
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
    prm.timeout_ns = opt.timeout_ns;
    prm.skip_loads = opt.skip_loads;
    prm.status = status_word();
    if (!prm.status) return cudaErrorInvalidSymbol;
    return pl.nt8 == 1 ? launch_tma_nt8<1>(pl, prm, stream, opt) : launch_tma_nt8<2>(pl, prm, stream, opt);
}

}  // namespace bsf8
