// bsf8_umma.cu -- the tensor-core (tcgen05) GEMM: weight rows stream in, are rebuilt to
// bf16 in shared memory and multiplied by the fifth-generation tensor cores.
//
//   y[m][g][n] = bf16( sum_{s=0..S-1} P[s][m][g][n] ),  summed s = 0, 1, ... in fp32,
//   W[g][n][k] = bf16( e4m3(w8[g][n][k]) * 2^(exp[g][n/32][k/32] - 127) ).
//
// Page: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- _wo_a_partial_w8() and
// _wo_a_mid_kernel() with their fixed-order split-K sums.
//
// A block owns 128 weight rows (a row block of one group), the columns of one split and a
// tile of up to 192 token rows (calls with more rows run one tile a grid z-index, each
// rebuilding the weights it streams: past a few hundred rows the product is bound by the
// tensor cores, not by the weight stream).
// Per 64-column step:
//   * the copy warp loads the step's codes (128 rows x 64 bytes, one TMA box; lane 0, up to
//     10 steps ahead, before the dependency wait too) and the step's x tile (lane 1: the M
//     token rows, zero-filled to a multiple of 16, x 64 columns, one box with the 128-byte
//     swizzle);
//   * eight rebuild warps (warp d rebuilds rows 16 d .. 16 d + 15) turn the codes into exact
//     bf16 weights -- the rebuild of bsf8_device.cuh -- and store them as the MMA's A
//     operand: K-major, 128-byte swizzle, 8-row atoms 1 KB apart;
//   * one thread of the MMA warp issues four tcgen05.mma (M = 128, N = tokens, K = 16) into
//     an fp32 accumulator in tensor memory and commits them to the barriers that free the
//     step's A and x slots.
// At the end the rebuild warps read the accumulators back (tcgen05.ld, thread = weight row;
// two warps a TMEM lane quarter split the token columns) and store y (one split) or the
// split's fp32 partials (the fixed-order reduce follows).
// Codes, A and x slots are rings with full/empty mbarriers; every wait is bounded, and on
// timeout the block records BSF8_ERR_TIMEOUT, stores nothing and returns.
//
// The weights are static, so their copies and the rebuild of the first steps run before the
// programmatic-dependent-launch wait; x is read and y written after it.
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <cuda.h>

#include <algorithm>
#include <mutex>

namespace bsf8 {

namespace {

constexpr int kRows = 128;           // weight rows a block (the MMA's M)
constexpr int kKB = 128;             // columns a step: 128-byte rows of codes
constexpr int kHalf = 64;            // columns of one 128-byte swizzle atom of bf16
constexpr int kCodesBytes = kRows * kKB;        // 16 KB of codes a step
constexpr int kAHalfBytes = kRows * kHalf * 2;  // 16 KB: A tile of one atom column
constexpr int kABytes = 2 * kAHalfBytes;        // 32 KB of bf16 a step
constexpr int kDaMax = 3, kDcMax = 8, kDxMax = 12;  // ring depths, set per call
// Dynamic shared memory a block: the A, x and codes rings, sized per call (x tiles grow
// with the tokens): x 2 .. 12 tiles within 48 KB unless two need more, A 2 steps of
// 32 KB, the codes ring the rest, 2 .. 8 steps.
constexpr int kSmemU = 208 * 1024;
constexpr int kRebuildWarps = 8;                // 16 weight rows each
constexpr int kThreadsU = (2 + kRebuildWarps) * 32;  // warp 0 copies, warp 1 MMA, 2.. rebuild
constexpr int kMaxTok = 192;  // tokens a block (a token tile; more rows take more tiles)
constexpr int kMaxRowsU = 16384;  // token rows a call (BSF8_MAX_M)
constexpr int kMaxSplitBlocks = 1024;  // 32-column exponent blocks of a split kept in smem
// The tensor core's fp32 accumulation into tensor memory loses accuracy with the number of
// products accumulated in place (measured: the error grows linearly with the steps
// accumulated, about eight times the fp32 index-order sum over 64 steps).  Each run of
// kChunkSteps steps therefore goes to its own accumulator, and the runs are summed in
// fp32 on the CUDA cores in run order: the error is then that of an ordinary fp32 sum.
constexpr int kChunkSteps = 4;  // 32 MMAs of K = 16 a run
constexpr int kTmemMax = 512;

struct UmmaParams {
    CUtensorMap cmap;  // w8 as [G*N rows][K columns] bytes, box 128 x 128, 128-byte swizzle
    CUtensorMap xmap;  // x as [M][G][K] bf16 (pitches ldx, K), box 64 x 1 x ntok, 128B swizzle
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S, chunk_cols, ntok;
    int to_partials;  // 1: store fp32 partials P[s] (even with one split), 0: store y
    int dx, dc, da;   // x, codes and A ring depths
    unsigned long long timeout_ns;
    int skip_loads;
    int *status;
};

__device__ __forceinline__ uint64_t evict_first_policy_u() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_2d_hint_u(void *dst, const CUtensorMap *map, int c0, int c1,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_3d_u(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile with the 128-byte swizzle: start
// address, leading offset unused (1), stride between 8-row atoms 1024 bytes, descriptor
// version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N columns, M = 128 rows.
__device__ __forceinline__ uint32_t mma_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc_u(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_u(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t max_xorsign_abs_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ bool nan_code_seen_u(uint32_t mx) {
    return (mx & 0x7FFFu) >= 0x07F0u || ((mx >> 16) & 0x7FFFu) >= 0x07F0u;
}

// Barrier of the rebuild warps only (named barrier 1).
__device__ __forceinline__ void named_sync_rebuild() {
    asm volatile("bar.sync 1, %0;" ::"n"(kRebuildWarps * 32) : "memory");
}

// Bounded wait on an mbarrier phase by every lane of a warp; false if any lane ran out.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
    const bool ok = mbar_wait_bounded(bar, parity, timeout_ns);
    return __all_sync(0xFFFFFFFFu, ok);
}

}  // namespace

__global__ void __launch_bounds__(kThreadsU, 2) umma_kernel(const __grid_constant__ UmmaParams p) {
    extern __shared__ uint8_t dyn_smem[];
    uint8_t *const base = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    uint8_t *const sA = base;                                   // da x 32 KB, 128B swizzle
    uint8_t *const sX = sA + p.da * kABytes;                    // dx x ntok x 256 B
    uint8_t *const sC = sX + p.dx * p.ntok * 256;                 // dc x 16 KB
    __shared__ __align__(8) uint64_t full_c[kDcMax], empty_c[kDcMax], full_a[kDaMax], empty_a[kDaMax];
    __shared__ __align__(8) uint64_t full_x[kDxMax], empty_x[kDxMax], d_full;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ uint32_t s_nan[4];  // per TMEM lane quarter: rows with an e4m3 NaN code
    __shared__ uint8_t s_exp[4][kMaxSplitBlocks];  // the split's exponents, per 32-row block

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y;
    const int rb = blockIdx.x / p.S, split = blockIdx.x % p.S;
    const int tok0 = blockIdx.z * p.ntok;  // first token row of this block's tile
    const int row0 = rb * kRows;  // first weight row of the block inside group g
    const int k0 = min(p.K, split * p.chunk_cols), k1 = min(p.K, k0 + p.chunk_cols);
    const int nkb = (k1 - k0 + kKB - 1) / kKB;
    const int nrun = (nkb + kChunkSteps - 1) / kChunkSteps;  // accumulators (runs of steps)
    uint32_t tcols = 32;
    while ((int)tcols < max(1, nrun) * p.ntok) tcols *= 2;   // the plan keeps this <= 512
    const int xbytes = p.ntok * 256;  // a step's x tile: two 64-column atoms
    const int kDx = p.dx, kDc = p.dc, kDa = p.da;  // ring depths of this call

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDcMax; ++i) {
            mbar_init(&full_c[i], 1);
            mbar_init(&empty_c[i], kRebuildWarps);
        }
        for (int i = 0; i < kDaMax; ++i) {
            mbar_init(&full_a[i], kRebuildWarps);
            mbar_init(&empty_a[i], 1);
        }
        for (int i = 0; i < kDxMax; ++i) {
            mbar_init(&full_x[i], 1);
            mbar_init(&empty_x[i], 1);
        }
        mbar_init(&d_full, 1);
        s_err = 0;
        for (int i = 0; i < 4; ++i) s_nan[i] = 0;
        fence_mbar_init();
        prefetch_tmap(&p.cmap);
        prefetch_tmap(&p.xmap);
    }
    if (warp == 1) tmem_alloc_u(&s_tmem, tcols);
    tc_before();
    __syncthreads();
    tc_after();
    pdl_trigger();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ copies
        if (lane == 0) {  // codes: static, streamed ahead from the start
            const uint64_t pol = evict_first_policy_u();
            int n = 0;
            bool bad = false;
            for (int kb = 0; kb < nkb; ++kb) {
                const int cs = kb % kDc;
                if (kb >= kDc && !mbar_wait_bounded(&empty_c[cs], (uint32_t)(((kb / kDc) - 1) & 1), p.timeout_ns)) {
                    bad = true;
                    break;
                }
                mbar_arrive_expect_tx(&full_c[cs], (uint32_t)kCodesBytes);
                if (!p.skip_loads)
                    tma_2d_hint_u(sC + cs * kCodesBytes, &p.cmap, k0 + kb * kKB, g * p.N + row0, &full_c[cs], pol);
                ++n;
            }
            if (bad) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
            if (*(volatile int *)&s_err && !p.skip_loads)  // let issued copies land (bounded)
                for (int i = max(0, n - kDc); i < n; ++i)
                    (void)mbar_wait_bounded(&full_c[i % kDc], (uint32_t)((i / kDc) & 1), p.timeout_ns);
        } else if (lane == 1) {  // x: after the dependency wait
            pdl_wait();
            int n = 0;
            bool bad = false;
            for (int kb = 0; kb < nkb; ++kb) {
                const int xs = kb % kDx;
                if (kb >= kDx && !mbar_wait_bounded(&empty_x[xs], (uint32_t)(((kb / kDx) - 1) & 1), p.timeout_ns)) {
                    bad = true;
                    break;
                }
                mbar_arrive_expect_tx(&full_x[xs], (uint32_t)xbytes);
                if (!p.skip_loads) {
                    tma_3d_u(sX + xs * xbytes, &p.xmap, k0 + kb * kKB, g, tok0, &full_x[xs]);
                    tma_3d_u(sX + xs * xbytes + xbytes / 2, &p.xmap, k0 + kb * kKB + kHalf, g, tok0, &full_x[xs]);
                }
                ++n;
            }
            if (bad) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
            if (*(volatile int *)&s_err && !p.skip_loads)
                for (int i = max(0, n - kDx); i < n; ++i)
                    (void)mbar_wait_bounded(&full_x[i % kDx], (uint32_t)((i / kDx) & 1), p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        const uint32_t idesc = mma_idesc(p.ntok);
        bool bad = false;
        const int tail = (k1 - k0) % kKB;  // columns of the last step inside the split (0: all)
        for (int kb = 0; kb < nkb; ++kb) {
            const int as = kb % kDa, xs = kb % kDx;
            if (!warp_wait(&full_a[as], (uint32_t)((kb / kDa) & 1), p.timeout_ns) ||
                !warp_wait(&full_x[xs], (uint32_t)((kb / kDx) & 1), p.timeout_ns)) {
                bad = true;
                break;
            }
            uint8_t *xt = sX + xs * xbytes;
            if (kb == nkb - 1 && tail != 0) {
                // x columns past the split's end belong to the next split: zero them (the
                // weights there are zero, and 0 * inf would be NaN); 16 units of 8 columns
                const int fu = tail / 8, units = 16 - fu;
                for (int i = lane; i < p.ntok * units; i += 32) {
                    const int r = i / units, u = fu + i % units;
                    *reinterpret_cast<uint4 *>(xt + (u >> 3) * (xbytes / 2) + (r >> 3) * 1024 + (r & 7) * 128 +
                                               (((u & 7) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            if (lane == 0) {
                tc_after();
                const uint32_t sa = smem_u32(sA + as * kABytes), sb = smem_u32(xt);
                const uint32_t dcol = (uint32_t)((kb / kChunkSteps) * p.ntok);  // this run's accumulator
#pragma unroll
                for (int ks = 0; ks < kKB / 16; ++ks) {  // atom column ks / 4, +32 bytes a K slice
                    const uint64_t ad = sw128_desc(sa + (ks >> 2) * kAHalfBytes) + 2 * (ks & 3);
                    const uint64_t bd = sw128_desc(sb + (ks >> 2) * (xbytes / 2)) + 2 * (ks & 3);
                    umma_f16(tmem + dcol, ad, bd, idesc, (kb % kChunkSteps > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(&empty_a[as]);
                umma_commit(&empty_x[xs]);
            }
            __syncwarp();
        }
        if (bad && lane == 0) {
            s_err = 1;
            report_timeout(p.status);
        }
        if (lane == 0) umma_commit(&d_full);  // completes once every MMA above has finished
        __syncwarp();
    } else {
        // ------------------------------------------------------------ rebuild + epilogue
        const int d = warp - 2;                // rows 16 d .. 16 d + 15 of the block
        const int rsub = lane >> 3, unit = lane & 7;  // rows 16 d + rsub + 4 i, 16 codes each
        const int n32 = row0 + 32 * (d >> 1);  // first row of the warp's exponent row block
        const bool rows_ok = n32 < p.N;
        {   // the split's exponent bytes of the block's four 32-row blocks (static: before the wait)
            const int kb0 = k0 / 32, nb = (k1 - k0) / 32;
            for (int i = threadIdx.x - 64; i < 4 * nb; i += kRebuildWarps * 32) {
                const int j = i / nb, b = i - j * nb;
                const int r32 = row0 / 32 + j;
                s_exp[j][b] = r32 < p.N / 32
                                  ? __ldg(p.ex + ((size_t)g * (p.N / 32) + r32) * (p.K / 32) + kb0 + b) : 127;
            }
            named_sync_rebuild();
        }
        const uint8_t *erow = s_exp[d >> 1];
        uint32_t mx[4] = {0, 0, 0, 0};
        bool bad = false;
        for (int kb = 0; kb < nkb; ++kb) {
            const int cs = kb % kDc, as = kb % kDa;
            if (!warp_wait(&full_c[cs], (uint32_t)((kb / kDc) & 1), p.timeout_ns) ||
                (kb >= kDa && !warp_wait(&empty_a[as], (uint32_t)(((kb / kDa) - 1) & 1), p.timeout_ns))) {
                bad = true;
                break;
            }
            const int kcol = k0 + kb * kKB + unit * 16;  // the lane's 16 columns
            const bool cols_ok = rows_ok && kcol < k1;
            const uint32_t e = cols_ok ? (uint32_t)erow[(kcol - k0) / 32] : 127u;
            const bool two = __any_sync(0xFFFFFFFFu, e > 134u);
            uint32_t s1, s2 = 0;
            if (two) {
                s1 = 0x7B807B80u;
                const uint32_t bb = e == 0 ? 0x0040u : (e << 7);
                s2 = bb | (bb << 16);
            } else {
                const uint32_t b = (e + 120u) << 7;
                s1 = b | (b << 16);
            }
            const uint8_t *cst = sC + cs * kCodesBytes;
            uint8_t *ast = sA + as * kABytes;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 16 * d + rsub + 4 * i;  // row inside the block
                // codes: 128-byte rows with the 128-byte swizzle (unit u of row r at u ^ r % 8)
                const uint4 c = cols_ok ? *reinterpret_cast<const uint4 *>(cst + row * 128 + ((unit ^ (row & 7)) << 4))
                                        : make_uint4(0, 0, 0, 0);
                uint32_t o[8];
                const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t t0, t1;
                    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w[j]));
                    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w[j]));
                    t0 = (t0 << 4) & 0x87F087F0u;
                    t1 = (t1 << 4) & 0x87F087F0u;
                    mx[i] = max_xorsign_abs_u(mx[i], max_xorsign_abs_u(t0, t1));
                    uint32_t lo = bf16x2_mul(t0, s1), hi = bf16x2_mul(t1, s1);
                    if (two) {
                        lo = bf16x2_mul(lo, s2);
                        hi = bf16x2_mul(hi, s2);
                    }
                    o[2 * j] = lo;
                    o[2 * j + 1] = hi;
                }
                // A: the lane's 16 columns are units 2 (unit % 4) and +1 of atom column unit / 4
                uint8_t *arow = ast + (unit >> 2) * kAHalfBytes + (row >> 3) * 1024 + (row & 7) * 128;
                const int u0 = 2 * (unit & 3);
                *reinterpret_cast<uint4 *>(arow + ((u0 ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4 *>(arow + (((u0 + 1) ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // A is read by the tensor core
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty_c[cs]);
                mbar_arrive(&full_a[as]);
            }
        }
        if (bad) {
            *(volatile int *)&s_err = 1;
            if (lane == 0) report_timeout(p.status);
        }
        // rows with an e4m3 NaN code, as bits of their TMEM lane quarter's mask
        uint32_t nmask = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (nan_code_seen_u(mx[i])) nmask |= 1u << ((16 * d + rsub + 4 * i) & 31);
        nmask = __reduce_or_sync(0xFFFFFFFFu, nmask);
        if (lane == 0 && nmask) atomicOr(&s_nan[d >> 1], nmask);

        pdl_wait();  // y may still be read by the kernels before this one
        const bool dok = warp_wait(&d_full, 0u, p.timeout_ns);
        named_sync_rebuild();  // every rebuild warp has posted its NaN rows
        tc_after();
        const int qd = warp & 3;               // TMEM lane quarter this warp may read
        const int half = (warp - 2) >> 2;      // warps of a quarter split the 16-column chunks
        const int n = row0 + 32 * qd + lane;   // this thread's weight row = its TMEM lane
        const bool store = dok && !*(volatile int *)&s_err && n < p.N;
        const bool poison = (s_nan[qd] >> lane) & 1u;
        for (int c0 = 16 * half; c0 < p.ntok; c0 += 32) {
            float acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
            for (int run = 0; run < nrun; ++run) {  // the runs' accumulators, in run order
                uint32_t r[16];
                tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(run * p.ntok + c0), r);
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = run == 0 ? __uint_as_float(r[j]) : acc[j] + __uint_as_float(r[j]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = tok0 + c0 + j;
                if (!store || m >= p.M) continue;
                float v = acc[j];
                if (poison) v = __uint_as_float(0x7FC00000u);
                if (p.to_partials)
                    p.partials[(((size_t)split * p.M + m) * p.G + g) * p.N + n] = v;
                else
                    p.y[((size_t)m * p.G + g) * p.N + n] = f32_to_bf16_rn(v);
            }
        }
        if (!dok && lane == 0) report_timeout(p.status);
    }

    tc_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA must be finished before its accumulator columns are freed (bounded)
        (void)mbar_wait_bounded(&d_full, 0u, p.timeout_ns);
        tc_after();
        tmem_dealloc_u(tmem, tcols);
    }
}

// ------------------------------------------------------------------- host side

namespace {

using EncodeTiledFnU = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnU encode_fn() {
    static EncodeTiledFnU fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnU>(f);
    });
    return fn;
}

// Tensor maps of recent operands (a map encodes only the address and the shape).
struct UKey {
    const void *ptr;
    long long a, b, c, d;
    bool operator==(const UKey &o) const {
        return ptr == o.ptr && a == o.a && b == o.b && c == o.c && d == o.d;
    }
};

cudaError_t umma_map(const UKey &key, bool codes, CUtensorMap *out) {
    static std::mutex mu;
    static UKey keys[64];
    static bool kind[64];
    static CUtensorMap maps[64];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (kind[i] == codes && keys[i] == key) {
            *out = maps[i];
            return cudaSuccess;
        }
    EncodeTiledFnU fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap m;
    CUresult r;
    if (codes) {  // [rows = a][K = b] bytes, box 128 x 128
        const cuuint64_t dims[2] = {(cuuint64_t)key.b, (cuuint64_t)key.a};
        const cuuint64_t strides[1] = {(cuuint64_t)key.b};
        const cuuint32_t box[2] = {(cuuint32_t)kKB, (cuuint32_t)kRows};
        const cuuint32_t es[2] = {1u, 1u};
        r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(key.ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {      // x: [M = a][G = b][K = c] bf16, row pitch d elements; box 64 x 1 x ntok (two a step)
        const cuuint64_t dims[3] = {(cuuint64_t)key.c, (cuuint64_t)key.b, (cuuint64_t)key.a};
        const cuuint64_t strides[2] = {(cuuint64_t)key.c * 2u, (cuuint64_t)key.d * 2u};
        const int ntok = (int)std::min<long long>(kMaxTok, (key.a + 15) / 16 * 16);  // a token tile
        const cuuint32_t box[3] = {(cuuint32_t)kHalf, 1u, (cuuint32_t)ntok};
        const cuuint32_t es[3] = {1u, 1u, 1u};
        r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(key.ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    keys[next] = key;
    kind[next] = codes;
    maps[next] = m;
    next = (next + 1) % 64;
    if (used < 64) ++used;
    *out = m;
    return cudaSuccess;
}

}  // namespace

UmmaPlan plan_umma(int M, int N, int K, int G, int S, bool partials) {
    UmmaPlan pl{};
    pl.S = S;
    pl.chunk_cols = ((K / 32 + S - 1) / S) * 32;
    pl.ntok = std::min(kMaxTok, (M + 15) / 16 * 16);  // tokens a tile
    pl.ttiles = (M + pl.ntok - 1) / std::max(1, pl.ntok);
    // the split's runs of steps each need ntok accumulator columns of tensor memory
    const int nrun = ((pl.chunk_cols + kKB - 1) / kKB + kChunkSteps - 1) / kChunkSteps;
    pl.tmem_ok = (long long)nrun * pl.ntok <= kTmemMax;
    pl.row_blocks = (N + kRows - 1) / kRows;
    pl.grid_x = pl.row_blocks * S;
    pl.partials = partials || S > 1;
    pl.ok = M >= 1 && M <= kMaxRowsU && (long long)G * N < (1LL << 31) && K < (1 << 30) && pl.tmem_ok &&
            pl.chunk_cols / 32 <= kMaxSplitBlocks;
    return pl;
}

// Splits for the tensor-core kernel: about one block an SM (the blocks stream, so more
// blocks than SMs add a wave), then enough that the runs' accumulators fit tensor memory.
int umma_auto_split(int M, int N, int K, int G, int sms) {
    const long long ttiles = (M + kMaxTok - 1) / kMaxTok;
    const long long blocks = (long long)((N + kRows - 1) / kRows) * G * ttiles;
    const int smax = std::max(1, K / 32);
    int S = (int)std::max(1LL, (sms + blocks / 2) / std::max(1LL, blocks));
    S = std::min(S, smax);
    while (S < smax && !plan_umma(M, N, K, G, S, false).ok) ++S;
    return S;
}

// Up to 16 tokens two blocks share an SM (rings within ~106 KB, accumulators within half of
// tensor memory): more blocks in flight to cover the per-step latency of one block's
// pipeline, and no second wave on large N.
bool umma_two_per_sm(const UmmaPlan &pl) {
    const int nrun = ((pl.chunk_cols + kKB - 1) / kKB + kChunkSteps - 1) / kChunkSteps;
    return pl.ntok <= 16 && nrun * pl.ntok <= kTmemMax / 2;
}

int umma_smem_budget(const UmmaPlan &pl) { return umma_two_per_sm(pl) ? 106 * 1024 : kSmemU; }

int umma_x_depth(const UmmaPlan &pl) {
    const int bytes = umma_two_per_sm(pl) ? 8 * 1024 : 48 * 1024;
    return std::max(2, std::min(kDxMax, bytes / (pl.ntok * 256)));
}

// A third A slot measured slower (the codes ring loses a step); two it is.
int umma_a_depth(const UmmaPlan &) { return 2; }

int umma_codes_depth(const UmmaPlan &pl) {
    const int left = umma_smem_budget(pl) - 1024 - umma_a_depth(pl) * kABytes - umma_x_depth(pl) * pl.ntok * 256;
    return std::min(kDcMax, left / kCodesBytes);
}

cudaError_t launch_umma(const UmmaPlan &pl, const void *x, long long ldx, const uint8_t *w8,
                        const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                        cudaStream_t stream) {
    if (!pl.ok) return cudaErrorInvalidValue;
    // the output the plan writes must be there (y for one split, the partials otherwise)
    if (pl.partials ? partials == nullptr : y == nullptr) return cudaErrorInvalidValue;
    const Options opt = options();
    UmmaParams prm;
    cudaError_t e = umma_map(UKey{w8, (long long)G * N, K, 0, 0}, true, &prm.cmap);
    if (e != cudaSuccess) return e;
    e = umma_map(UKey{x, M, G, K, ldx}, false, &prm.xmap);
    if (e != cudaSuccess) return e;
    prm.ex = ex;
    prm.y = static_cast<uint16_t *>(y);
    prm.partials = partials;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.G = G;
    prm.S = pl.S;
    prm.chunk_cols = pl.chunk_cols;
    prm.ntok = pl.ntok;
    prm.to_partials = pl.partials ? 1 : 0;
    prm.dx = umma_x_depth(pl);
    prm.dc = umma_codes_depth(pl);
    prm.da = umma_a_depth(pl);
    if (prm.dc < 2) return cudaErrorInvalidValue;
    prm.timeout_ns = opt.timeout_ns;
    prm.skip_loads = opt.skip_loads;
    prm.status = status_word();
    if (!prm.status) return cudaErrorInvalidSymbol;
    const size_t smem = (size_t)umma_smem_budget(pl);
    static int configured[64] = {0};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemU);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(umma_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid_x, (unsigned)G, (unsigned)pl.ttiles);
    cfg.blockDim = dim3(kThreadsU, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[1];
    int na = 0;
    if (opt.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, umma_kernel, prm);
}

}  // namespace bsf8
