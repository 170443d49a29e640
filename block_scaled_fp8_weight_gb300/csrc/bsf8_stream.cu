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

// 16-byte asynchronous copy global -> shared (L2 only); src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Shifted-and-masked codes (bf16 bits of e4m3 * 2^-120) for the four codes of w.
__device__ __forceinline__ void spread4(uint32_t w, uint32_t &t0, uint32_t &t1) {
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w));
    t0 = (t0 << 4) & 0x87F087F0u;
    t1 = (t1 << 4) & 0x87F087F0u;
}

// Step geometry: one weight row piece per thread per step.
//   NT8 == 1: 128-column steps, a thread owns 32 columns (8 MMAs per step);
//   NT8 >= 2: 64-column steps, a thread owns 16 columns (4 MMAs per step).
template <int NT8>
struct StepCfg {
    static constexpr int KS = NT8 == 1 ? 128 : 64;
    static constexpr int TC = KS / 4;                 // columns per thread per step
    static constexpr int WV = TC / 16;                // 16-byte vectors per row per thread
    static constexpr int XV = TC / 8;                 // 16-byte x vectors per token row
    static constexpr int MMAS = TC / 4;               // MMAs per step per token tile
    static constexpr int PITCH = KS == 128 ? 144 : 64;  // smem row pitch (conflict-free)
    static constexpr int STAGE = 16 * PITCH;          // one warp's stage: 16 rows
    static constexpr int DEPTH = KS == 128 ? 5 : 9;   // stages per warp ring
    static constexpr int CPL = 16 * KS / 16 / 32;    // 16-byte copies per lane per step
    static constexpr int ACC = NT8 == 1 ? 2 : 1;      // accumulator sets (MMA chain split)
};

template <int NT8>
struct XBuf {
    uint4 v[NT8][StepCfg<NT8>::XV];
    uint32_t e;
};

// One step of a warp task: rebuild the thread's codes of rows r and r+8 and feed each
// word straight into its MMAs.  mxa / mxb collect the largest rebuilt magnitude of rows r /
// r+8: an e4m3 NaN code rebuilds to the pattern 0x07F0, above every finite code's 0x07E0
// (448 * 2^-120), so the task's rows holding one are set to NaN once, at the end.
// ROWS: xb.e holds the exponent bytes of rows r (bits 0..7) and r + 8 (bits 8..15), the
// per-(row, 32-column) scale layout; else one byte for the thread's 32 x 32 block.
template <int NT8, bool TWO, bool ROWS>
__device__ __forceinline__ void compute_step(const uint8_t *stage, int r, int q, const XBuf<NT8> &xb,
                                             float (&acc)[StepCfg<NT8>::ACC][NT8][4],
                                             uint32_t &mxa, uint32_t &mxb) {
    using C = StepCfg<NT8>;
    const uint32_t ea = ROWS ? (xb.e & 0xFFu) : xb.e, eb = ROWS ? (xb.e >> 8) : xb.e;
    uint32_t s1a, s2a = 0, s1b, s2b = 0;
    if (TWO) {  // exact for every exponent byte: restore e4m3 * 1, then scale by 2^(e-127)
        s1a = s1b = 0x7B807B80u;
        const uint32_t ba = ea == 0 ? 0x0040u : (ea << 7), bb = eb == 0 ? 0x0040u : (eb << 7);
        s2a = ba | (ba << 16);
        s2b = bb | (bb << 16);
    } else {
        s1a = make_scale(ea).s1;
        s1b = ROWS ? make_scale(eb).s1 : s1a;
    }
#pragma unroll
    for (int v = 0; v < C::WV; ++v) {
        const uint4 a = *reinterpret_cast<const uint4 *>(stage + r * C::PITCH + q * C::TC + 16 * v);
        const uint4 b = *reinterpret_cast<const uint4 *>(stage + (r + 8) * C::PITCH + q * C::TC + 16 * v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = 4 * v + i;
            uint32_t t0, t1, u0, u1;
            spread4(i == 0 ? a.x : i == 1 ? a.y : i == 2 ? a.z : a.w, t0, t1);
            spread4(i == 0 ? b.x : i == 1 ? b.y : i == 2 ? b.z : b.w, u0, u1);
            mxa = bf16x2_max_abs(mxa, bf16x2_max_abs(t0, t1));
            mxb = bf16x2_max_abs(mxb, bf16x2_max_abs(u0, u1));
            uint32_t alo = bf16x2_mul(t0, s1a), ahi = bf16x2_mul(t1, s1a);
            uint32_t blo = bf16x2_mul(u0, s1b), bhi = bf16x2_mul(u1, s1b);
            if (TWO) {
                alo = bf16x2_mul(alo, s2a);
                ahi = bf16x2_mul(ahi, s2a);
                blo = bf16x2_mul(blo, s2b);
                bhi = bf16x2_mul(bhi, s2b);
            }
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                // x word i holds the thread's columns (2i, 2i+1); MMA j takes 4j .. 4j+3
                const uint4 &xv0 = xb.v[t][(2 * j) / 4];
                const uint32_t b0 = ((2 * j) % 4) == 0 ? xv0.x : xv0.z;
                const uint32_t b1 = ((2 * j) % 4) == 0 ? xv0.y : xv0.w;
                mma_bf16_16816(acc[j % C::ACC][t], alo, blo, ahi, bhi, b0, b1);
            }
        }
    }
}

__device__ __forceinline__ bool has_nan_code(uint32_t mx) {
    return (mx & 0x7FFFu) >= 0x07F0u || ((mx >> 16) & 0x7FFFu) >= 0x07F0u;
}

// End of a group: every warp has written its task partial to red[warp].  Sums them in the
// fixed order (tasks of a split in task order, splits in split order) and stores y, or
// stores the per-split partials P[s].  gslab is the first slab of the group.
template <int NT8>
__device__ __forceinline__ void group_epilogue(const StreamParams &p, float (*red)[16][8 * NT8], int g,
                                               int mbase, int nslabs, int tslab, int gslab) {
    constexpr int MT = 8 * NT8;
    const int mrows = min(MT, p.M - mbase);
    if (p.mode == kStreamInCta) {
        __syncthreads();
        const int per_slab = 16 * mrows;
        for (int i = threadIdx.x; i < p.spc * per_slab; i += kStreamThreads) {
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
        __syncthreads();  // red is rewritten by the next group
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
            p.partials[(((size_t)ss * p.M + mbase + m) * p.G + g) * p.N + gslab * 16 + row] = ps;
        }
        __syncthreads();
    } else {
        // Cluster of the slab's blocks (rank c holds tasks 8c .. 8c+7): each block sums a
        // share of the slab's outputs, reading every task partial in task order via DSMEM.
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
            p.y[((size_t)(mbase + m) * p.G + g) * p.N + gslab * 16 + row] = f32_to_bf16_rn(y);
        }
        cluster_sync();  // keep this block's shared memory alive until the others are done
    }
}

template <int NT8, bool ROWS>
__global__ void __launch_bounds__(kStreamThreads, NT8 <= 2 ? 2 : 1)
    stream_kernel(const __grid_constant__ StreamParams p) {
    using C = StepCfg<NT8>;
    constexpr int MT = 8 * NT8;
    __shared__ __align__(16) float red[kStreamWarps][16][MT];  // per-warp task partials

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q = lane & 3;
    const int r = lane >> 2;
    const int g = blockIdx.y % p.G;
    const int mbase = (blockIdx.y / p.G) * MT;
    const int nslabs = p.N / 16;
    const int tslab = p.S * p.tps;

    // ---- groups and this warp's task.  In-block mode: a group is spc slabs with all their
    // tasks, and a block walks groups blockIdx.x, blockIdx.x + gridDim.x, ... (persistent).
    // Partials / cluster mode: one group per block.  A warp's task (split s, task u, columns
    // [k0, k1)) is the same in every group; only the slab (its 16 rows) changes.
    int ngroups = 1, s, u, slab0, slab_step = 0;
    bool active;
    if (p.mode == kStreamCluster) {
        slab0 = blockIdx.x / p.cluster;
        const int tau = (blockIdx.x % p.cluster) * kStreamWarps + warp;
        s = tau / p.tps;
        u = tau % p.tps;
        active = tau < tslab;
    } else if (p.mode == kStreamPartials) {
        slab0 = blockIdx.x / p.cps;
        s = (blockIdx.x % p.cps) * p.spl + warp / p.tps;
        u = warp % p.tps;
        active = warp < p.spl * p.tps && s < p.S;
    } else {
        const int groups_total = (nslabs + p.spc - 1) / p.spc;
        ngroups = (int)blockIdx.x < groups_total
                      ? (groups_total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        slab0 = blockIdx.x * p.spc + warp / tslab;
        slab_step = gridDim.x * p.spc;
        s = (warp % tslab) / p.tps;
        u = (warp % tslab) % p.tps;
        active = warp < p.spc * tslab;
    }
    int k0 = 0, k1 = 0;
    if (active) {
        const int s_lo = min(p.K, s * p.chunk_cols);
        const int s_hi = min(p.K, s_lo + p.chunk_cols);
        k0 = min(s_hi, s_lo + u * p.kt);
        k1 = min(s_hi, k0 + p.kt);
    }
    // Steps per group; a warp without columns runs one all-zero step so that every warp
    // reaches each group's epilogue in the same loop.
    const int nst = active && k1 > k0 ? (k1 - k0 + C::KS - 1) / C::KS : 1;
    const long long total = (long long)ngroups * nst;

    pdl_trigger();

    float acc[C::ACC][NT8][4];
#pragma unroll
    for (int a = 0; a < C::ACC; ++a)
#pragma unroll
        for (int t = 0; t < NT8; ++t)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][t][c] = 0.0f;
    uint32_t mxa = 0, mxb = 0;  // largest rebuilt magnitudes of rows r and r+8

    extern __shared__ __align__(128) uint8_t ring_smem[];
    uint8_t *ring = ring_smem + warp * C::DEPTH * C::STAGE;
    // weight copies: lane copies 16-byte chunk (lane % cpr) of rows crow + i * rows_per
    constexpr int cpr = C::KS / 16;
    constexpr int rows_per = 32 / cpr;
    const int crow = lane / cpr, ccol = (lane % cpr) * 16;
    const size_t rstride = (size_t)rows_per * p.K;
    const size_t gbase = (size_t)g * p.N;

    // Issue cursor over the flattened (group, step) sequence of this warp.
    int is_gi = 0, is_t = 0, is_slot = 0;
    auto issue_next = [&]() {
        if (is_gi < ngroups) {
            const int slab = slab0 + is_gi * slab_step;
            const bool in = active && slab < nslabs && k0 + is_t * C::KS + ccol < k1;
            // a zero-fill copy reads nothing; it still gets a valid address
            const uint8_t *src = in ? p.w8 + (gbase + slab * 16 + crow) * p.K + k0 + ccol + (size_t)is_t * C::KS
                                    : p.w8;
            uint8_t *st = ring + is_slot * C::STAGE;
#pragma unroll
            for (int i = 0; i < C::CPL; ++i)
                cp_async16(st + (crow + i * rows_per) * C::PITCH + ccol, in ? src + i * rstride : src,
                           in ? 16u : 0u);
            if (++is_t == nst) {
                is_t = 0;
                ++is_gi;
            }
        }
        is_slot = is_slot + 1 == C::DEPTH ? 0 : is_slot + 1;
        cp_async_commit();
    };

    // The twin is a static parameter: the first DEPTH-1 steps of this warp's stream are
    // copied into its ring, and the rest of its first task prefetched into L2, before
    // waiting for the preceding kernel (whose outputs include x).
#pragma unroll
    for (int i = 0; i < C::DEPTH - 1; ++i) issue_next();
    if (active && ngroups > 0 && slab0 < nslabs && nst > C::DEPTH - 1 && lane < 16) {
        const int rest = (C::DEPTH - 1) * C::KS;
        if (k1 - k0 > rest)
            prefetch_l2(p.w8 + (gbase + slab0 * 16 + lane) * p.K + k0 + rest, (uint32_t)(k1 - k0 - rest));
    }
    pdl_wait();

    // token rows >= M read row M-1 instead: their outputs are never stored
    const uint16_t *xsrc[NT8];
#pragma unroll
    for (int t = 0; t < NT8; ++t) {
        const int m = min(mbase + t * 8 + r, p.M - 1);
        xsrc[t] = p.x + (size_t)m * p.ldx + (size_t)g * p.K + k0 + q * C::TC;
    }
    // exponent bytes: one per 32 x 32 block, or (ROWS) one per weight row and 32 columns
    const size_t ebase = (size_t)g * (ROWS ? p.N : p.N / 32) * (p.K / 32) + (size_t)((k0 + q * C::TC) / 32);
    auto load_x = [&](XBuf<NT8> &xb, int gi, int t) {
        const int slab = slab0 + gi * slab_step;
        if (active && gi < ngroups && slab < nslabs && k0 + t * C::KS + q * C::TC < k1) {
#pragma unroll
            for (int tt = 0; tt < NT8; ++tt)
#pragma unroll
                for (int v = 0; v < C::XV; ++v) xb.v[tt][v] = ldg_v4(xsrc[tt] + t * C::KS + 8 * v);
            if (ROWS) {
                const uint8_t *ea = p.ex + ebase + (size_t)(slab * 16 + r) * (p.K / 32) + t * (C::KS / 32);
                xb.e = ldg_u8(ea) | (ldg_u8(ea + (size_t)8 * (p.K / 32)) << 8);
            } else {
                xb.e = ldg_u8(p.ex + ebase + (size_t)(slab / 2) * (p.K / 32) + t * (C::KS / 32));
            }
        } else {
#pragma unroll
            for (int tt = 0; tt < NT8; ++tt)
#pragma unroll
                for (int v = 0; v < C::XV; ++v) xb.v[tt][v] = make_uint4(0, 0, 0, 0);
            xb.e = ROWS ? (127u | (127u << 8)) : 127u;
        }
    };
    auto compute = [&](const uint8_t *st, const XBuf<NT8> &cur) {
        const uint32_t emax = ROWS ? max(cur.e & 0xFFu, cur.e >> 8) : cur.e;
        if (__any_sync(0xFFFFFFFFu, emax > 134u))
            compute_step<NT8, true, ROWS>(st, r, q, cur, acc, mxa, mxb);
        else
            compute_step<NT8, false, ROWS>(st, r, q, cur, acc, mxa, mxb);
    };

    XBuf<NT8> xa, xb;
    int gi = 0, t = 0, slot = 0;
    load_x(xa, 0, 0);
    for (long long T = 0; T < total; ++T) {
        __syncwarp();  // every lane is done with the slot the next issue refills
        issue_next();
        const int ngi = t + 1 == nst ? gi + 1 : gi, nt = t + 1 == nst ? 0 : t + 1;
        const uint8_t *st = ring + slot * C::STAGE;
        if (T & 1) {
            load_x(xa, ngi, nt);
            cp_async_wait<C::DEPTH - 1>();
            __syncwarp();  // this step's slot has landed for every lane
            compute(st, xb);
        } else {
            load_x(xb, ngi, nt);
            cp_async_wait<C::DEPTH - 1>();
            __syncwarp();
            compute(st, xa);
        }
        slot = slot + 1 == C::DEPTH ? 0 : slot + 1;
        if (nt == 0) {
            // ---- end of group gi: the epilogue below runs once per group for every warp
            const int slab = slab0 + gi * slab_step;
            // A NaN code anywhere in row r (r+8) of the task makes that row's outputs NaN.
            uint32_t fa = has_nan_code(mxa) ? 1u : 0u, fb = has_nan_code(mxb) ? 1u : 0u;
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
                    v[c] = C::ACC == 2 ? acc[0][tt][c] + acc[C::ACC - 1][tt][c] : acc[0][tt][c];
                    if ((c < 2 && fa) || (c >= 2 && fb)) v[c] = qnan;
                }
                const int col = tt * 8 + 2 * q;
                *reinterpret_cast<float2 *>(&red[warp][r][col]) = make_float2(v[0], v[1]);
                *reinterpret_cast<float2 *>(&red[warp][r + 8][col]) = make_float2(v[2], v[3]);
            }
#pragma unroll
            for (int a = 0; a < C::ACC; ++a)
#pragma unroll
                for (int tt = 0; tt < NT8; ++tt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[a][tt][c] = 0.0f;
            mxa = mxb = 0;
            (void)slab;
            const int gslab = p.mode == kStreamInCta ? ((int)blockIdx.x + gi * (int)gridDim.x) * p.spc
                                                     : slab0;
            group_epilogue<NT8>(p, red, g, mbase, nslabs, tslab, gslab);
        }
        gi = ngi;
        t = nt;
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------- host side

StreamPlan plan_stream(int M, int N, int K, int G, int S, bool partials) {
    const int nt8 = std::min(4, (M + 7) / 8);
    return plan_stream_ks(M, N, K, G, S, partials, nt8 == 1 ? 128 : 64, 4);
}

StreamPlan plan_stream_ks(int M, int N, int K, int G, int S, bool partials, int ks, int max_nt8,
                          int max_kt) {
    StreamPlan pl{};
    pl.nt8 = std::min(max_nt8, (M + 7) / 8);
    pl.m_chunks = (M + 8 * pl.nt8 - 1) / (8 * pl.nt8);
    const int nkb = K / 32;
    pl.S = S;
    pl.chunk_cols = ((nkb + S - 1) / S) * 32;
    // Task width: at least 512 columns (every step of such a task is in the warp's ring
    // before the dependency wait), and at most 8 tasks per split.
    int kt = std::max(512, (pl.chunk_cols + 7) / 8);
    kt = (kt + ks - 1) / ks * ks;
    kt = std::min(kt, std::max(ks, max_kt / ks * ks));
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
        pl.grid_x = (nslabs + pl.spc - 1) / pl.spc;  // capped at the resident blocks at launch
    } else {
        pl.mode = kStreamCluster;
        pl.cluster = (tslab + kStreamWarps - 1) / kStreamWarps;
        pl.grid_x = nslabs * pl.cluster;
    }
    return pl;
}

namespace {
template <int NT8, bool ROWS>
cudaError_t launch_stream_nt8(const StreamPlan &pl, const StreamParams &prm, cudaStream_t stream,
                              const Options &opt) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid_x, (unsigned)(prm.G * pl.m_chunks), 1);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    const size_t smem = (size_t)kStreamWarps * StepCfg<NT8>::DEPTH * StepCfg<NT8>::STAGE;
    static int configured[64] = {0};  // per device: dynamic shared memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(stream_kernel<NT8, ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    cfg.dynamicSmemBytes = smem;
    if (pl.mode == kStreamInCta) {
        // Persistent: at most the blocks that are resident at once (groups are strided).
        static int cap[64] = {0};
        int c = __atomic_load_n(&cap[dev], __ATOMIC_ACQUIRE);
        if (c == 0) {
            int sms = 0, per_sm = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_kernel<NT8, ROWS>, kStreamThreads, smem);
            if (e != cudaSuccess) return e;
            c = std::max(1, sms * std::max(1, per_sm));
            __atomic_store_n(&cap[dev], c, __ATOMIC_RELEASE);
        }
        cfg.gridDim.x = (unsigned)std::min(pl.grid_x, c);
    }
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
    return cudaLaunchKernelEx(&cfg, stream_kernel<NT8, ROWS>, prm);
}
}  // namespace

cudaError_t launch_stream(const StreamPlan &pl, const void *x, long long ldx, const uint8_t *w8,
                          const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                          cudaStream_t stream, bool rows_exp) {
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
    if (rows_exp) switch (pl.nt8) {
            case 1: return launch_stream_nt8<1, true>(pl, prm, stream, opt);
            case 2: return launch_stream_nt8<2, true>(pl, prm, stream, opt);
            case 3: return launch_stream_nt8<3, true>(pl, prm, stream, opt);
            default: return launch_stream_nt8<4, true>(pl, prm, stream, opt);
        }
    switch (pl.nt8) {
        case 1: return launch_stream_nt8<1, false>(pl, prm, stream, opt);
        case 2: return launch_stream_nt8<2, false>(pl, prm, stream, opt);
        case 3: return launch_stream_nt8<3, false>(pl, prm, stream, opt);
        default: return launch_stream_nt8<4, false>(pl, prm, stream, opt);
    }
}

}  // namespace bsf8
