// bsf8_ahead.cu -- the decode-ahead tensor-core GEMM for up to 32 token rows: the rebuilt
// weights wait in tensor memory as the MMA's A operand until x arrives.
//
//   y[m][g][n] = bf16( sum_{s=0..S-1} P[s][m][g][n] ),  summed s = 0, 1, ... in fp32,
//   W[g][n][k] = bf16( e4m3(w8[g][n][k]) * 2^(exp[g][n/32][k/32] - 127) )
//   (ROWS: exp[g][n][k/32], one exponent per weight row and 32 columns).
//
// Page: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- _wo_a_partial_w8() and
// _wo_a_mid_kernel() with their fixed-order split-K sums.
//
// A block owns 128 weight rows of one group and one task: at most 512 columns inside one
// split.  A cluster holds every task of its 128 rows (S splits x tps tasks, at most 16
// blocks; past 8 a non-portable cluster size, where the device schedules one), so the
// split-K sum never leaves the cluster.
//   before the wait (the weights are static):
//     * thread 0 loads the task's codes -- up to four 128-row x 128-byte boxes, 128-byte
//       swizzle -- on one mbarrier;
//     * thread = weight row (two threads a row, alternate 32-column blocks) rebuilds its
//       codes exactly to bf16: the first 128 columns into shared memory in the MMA's K-major
//       swizzled layout, the rest into tensor memory (lane = row, two bf16 a 32-bit column),
//       where tcgen05.mma reads A directly;
//   after griddepcontrol.wait:
//     * x (M rows x the task's columns) arrives by cp.async into a K-major swizzled tile of
//       16 or 32 token rows (rows >= M zero);
//     * the task's tcgen05.mma (M = 128, N = 16 or 32, K = 16; at most 32) go round robin
//       into 64 / N fp32 accumulators, each accumulator's MMAs issued by its own thread
//       (lane 0 of warps 0 .. 64/N - 1): a thread's tcgen05.mma issues ~100 cycles apart
//       however small N is (measured on a GB300), while MMAs issued by different warps
//       overlap;
//     * the accumulators come back (tcgen05.ld, thread = row) and are added in order; every
//       block pushes its rows' partials over DSMEM to the block of the cluster that folds
//       them (rank r folds rows [r L, r L + L), L = ceil(128 / C)), and after one cluster
//       barrier each block sums its rows' tasks in split order and stores y (or the splits'
//       fp32 partials).
// A block takes 256 TMEM columns (accumulators + A) and ~97 KB of shared memory, so two
// share an SM: the next call's blocks become resident and rebuild while this call
// finishes.  After the wait a call costs the x round trip, the MMA issue (a warp per
// accumulator), the accumulators' read and the reduction; the mma.sync decode-ahead kernel
// (bsf8_lowm.cu) spends 8x more MMA instructions there but issues them from all 8 warps,
// which is still faster up to 8 token rows.
//
// Every wait is bounded: on timeout the block records BSF8_ERR_TIMEOUT, stores nothing,
// lets its copies land and returns.
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <cuda.h>

#include <algorithm>
#include <mutex>

namespace bsf8 {

namespace {

constexpr int kThreadsA = 256;                          // 8 warps: 2 per TMEM lane quarter
constexpr int kRowsA = 128;                             // weight rows a block (the MMA's M)
constexpr int kBoxColsA = 128;                          // columns of a code box (128-byte rows)
constexpr int kBoxBytesA = kRowsA * kBoxColsA;          // 16 KB
constexpr int kMaxKtA = 512;                            // task columns (32 MMAs)
constexpr int kMaxBoxesA = kMaxKtA / kBoxColsA;
constexpr int kSmemColsA = 128;                         // task columns whose A is in shared memory
constexpr int kAtomBytesA = kRowsA * 64 * 2;            // 16 KB: 64 bf16 columns (one swizzle atom)
constexpr int kSmemABytes = kRowsA * kSmemColsA * 2;    // 32 KB
constexpr int kTmemColsA = 256;                         // accumulators (64) + A ((kt - 128) / 2)
constexpr int kAccColsA = 64;                           // 64 / ntok accumulators of ntok columns
constexpr int kMaxTokA = 32;
constexpr int kMaxPortableClusterA = 8;
constexpr int kMaxClusterA = 16;
// After the rebuild the codes' room holds the x tile (<= 8 chunks x 32 x 128 bytes) and the
// gather tiles: [C tasks][L rows][ntok] fp32 partials this block folds, C * ceil(128 / C) <= 140
// for C <= 16.
constexpr int kXTileBytesA = (kMaxKtA / 64) * kMaxTokA * 128;
constexpr int kGatherBytesA = 140 * kMaxTokA * 4;
constexpr int kSmemBytesA = kMaxBoxesA * kBoxBytesA + kSmemABytes + 1024;
static_assert(kXTileBytesA + kGatherBytesA <= kMaxBoxesA * kBoxBytesA, "x and gather fit the codes' room");
static_assert(kTmemColsA >= kAccColsA + (kMaxKtA - kSmemColsA) / 2, "accumulators and A fit");
static_assert(3 * (kSmemBytesA + 1024) > 228 * 1024, "at most two blocks an SM");
static_assert(2 * (kSmemBytesA + 2048) <= 228 * 1024, "two blocks fit an SM");

struct AheadParams {
    CUtensorMap wmap;  // w8 as a [G*N rows][K columns] byte matrix, box 128 x 128
    const uint16_t *x;  // [M][ldx] bf16
    long long ldx;
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S;
    int chunk_cols, kt, tps, ntok, nacc, cluster, rows_per_rank, partials_out;
    unsigned long long timeout_ns;
    int skip_loads;
    int *status;
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint64_t evict_first_policy_a() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_2d_a(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap_a(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 16-byte global -> shared copy through the load/store path.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all_a() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// First half of a split cluster barrier: arrive now, wait (cluster_wait_a) later.
__device__ __forceinline__ void cluster_arrive_relaxed_a() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_a() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc_a(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_a(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_before_a() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_a() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 registers of this thread -> columns [taddr, taddr + 16) of its TMEM lane.
__device__ __forceinline__ void tmem_st16_a(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16_a(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st_a() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major bf16 tile with the 128-byte swizzle: start
// address, leading offset unused (1), 8-row atoms 1024 bytes apart, descriptor version 1,
// layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc_a(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = n columns, M = 128 rows.
__device__ __forceinline__ uint32_t mma_idesc_a(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kRowsA >> 4) << 24);
}

// D (+)= A * B with A in shared memory (descriptor).
__device__ __forceinline__ void umma_ss_a(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (+)= A * B with A in tensor memory (lane = row of A, 8 columns = K 16 of bf16).
__device__ __forceinline__ void umma_ts_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit_a(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint32_t max_xorsign_abs_a(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Rebuilds the 32 codes of one 32-column block (c0 = columns 0..15, c1 = 16..31) to bf16:
// a[i] = bf16x2(column 2i, column 2i+1).  TWO: the two-multiply form, exact for every
// exponent byte; otherwise e <= 134 and one multiply by 2^(e-7).  mx keeps the largest
// magnitude pattern before scaling (an e4m3 NaN code spreads to 0x07F0, above every finite
// code's 0x07E0).
__device__ __forceinline__ void rebuild_block_a(const uint4 &c0, const uint4 &c1, uint32_t e, bool two,
                                                uint32_t (&a)[16], uint32_t &mx) {
    uint32_t s1, s2 = 0;
    if (two) {
        s1 = 0x7B807B80u;                         // 2^120: e4m3 * 2^-120 back to e4m3
        const uint32_t b = e == 0 ? 0x0040u : (e << 7);  // 2^(e-127) (byte 0: the subnormal 2^-127)
        s2 = b | (b << 16);
    } else {
        const uint32_t b = (e + 120u) << 7;       // 2^(e-7)
        s1 = b | (b << 16);
    }
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t t0, t1;
        asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w[i]));
        asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w[i]));
        t0 = (t0 << 4) & 0x87F087F0u;
        t1 = (t1 << 4) & 0x87F087F0u;
        mx = max_xorsign_abs_a(mx, max_xorsign_abs_a(t0, t1));
        uint32_t lo = bf16x2_mul(t0, s1), hi = bf16x2_mul(t1, s1);
        if (two) {
            lo = bf16x2_mul(lo, s2);
            hi = bf16x2_mul(hi, s2);
        }
        a[2 * i] = lo;
        a[2 * i + 1] = hi;
    }
}

__device__ __forceinline__ bool nan_code_seen_a(uint32_t mx) {
    return (mx & 0x7FFFu) >= 0x07F0u || ((mx >> 16) & 0x7FFFu) >= 0x07F0u;
}

}  // namespace

template <bool ROWS>
__global__ void __launch_bounds__(kThreadsA, 2) ahead_kernel(const __grid_constant__ AheadParams p) {
    extern __shared__ uint8_t dyn_smem[];
    // the swizzled tiles need 1024-byte alignment
    uint8_t *const codes = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    uint8_t *const xs = codes;  // after the rebuild the codes' room takes the x tile ...
    float *const gather = reinterpret_cast<float *>(codes + kXTileBytesA);  // ... and the gather tiles
    uint8_t *const sa = codes + kMaxBoxesA * kBoxBytesA;  // A of the task's first 128 columns
    __shared__ __align__(8) uint64_t wbar, dbar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ uint32_t s_nan[4];  // per TMEM lane quarter: rows with an e4m3 NaN code

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lq = warp & 3, h = warp >> 2;
    const int row = 32 * lq + lane;  // this thread's weight row in the block (= TMEM lane)
    const int g = blockIdx.y;
    const int C = p.cluster;
    const int tile = blockIdx.x / C, tau = blockIdx.x % C;  // rank in the cluster = task
    const int s = tau / p.tps, u = tau % p.tps;
    const int n0 = tile * kRowsA;
    const int s_lo = min(p.K, s * p.chunk_cols), s_hi = min(p.K, s_lo + p.chunk_cols);
    const int k0 = min(s_hi, s_lo + u * p.kt), k1 = min(s_hi, k0 + p.kt);
    const int nkb = (k1 - k0) / 32;
    const int nbox = (k1 - k0 + kBoxColsA - 1) / kBoxColsA;
    const int nsteps = (k1 - k0) / 16;
    const bool row_ok = n0 + row < p.N;

    const int nacc = min(p.nacc, nsteps);  // accumulators (and MMA-issuing warps) of the task
    if (threadIdx.x == 0) {
        mbar_init(&wbar, 1);
        mbar_init(&dbar, (uint32_t)max(1, nacc));
        fence_mbar_init();
        s_err = 0;
    }
    if (threadIdx.x < 4) s_nan[threadIdx.x] = 0u;
    if (threadIdx.x == 32) prefetch_tmap_a(&p.wmap);
    if (warp == 0) tmem_alloc_a(&s_tmem, kTmemColsA);
    tc_before_a();
    __syncthreads();
    tc_after_a();
    pdl_trigger();
    const uint32_t tmem = s_tmem;
    const uint32_t tlane = tmem + ((uint32_t)(32 * lq) << 16);  // this warp's lane quarter
    const uint32_t acol = (uint32_t)kAccColsA;                  // first A column

    // ---- weights (static): all of the task's boxes on one barrier.  The issuing lane's
    // warp-mates wait for it at __syncwarp, not in the barrier wait: a warp whose other
    // lanes sleep in mbarrier.try_wait lets the issuing lane run only between their sleeps.
    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&wbar, (uint32_t)(nbox * kBoxBytesA));
            if (!p.skip_loads) {
                const uint64_t pol = evict_first_policy_a();
                for (int b = 0; b < nbox; ++b)
                    tma_2d_a(codes + b * kBoxBytesA, &p.wmap, k0 + b * kBoxColsA, g * p.N + n0, &wbar, pol);
            }
        }
        __syncwarp();
    }
    // The task's x rows, pulled into L2 while the previous kernel runs (a hint: x is read
    // after the wait from L2, where the producer's writes land).
    if (threadIdx.x >= 64 && threadIdx.x < 64 + p.M && k1 > k0)
        prefetch_l2(p.x + (size_t)(threadIdx.x - 64) * p.ldx + (size_t)g * p.K + k0, (uint32_t)((k1 - k0) * 2));
    // exponent bytes of this thread's blocks j = 2 i + h (byte i)
    uint64_t ew = 0u;
    {
        const size_t kb = (size_t)(p.K / 32);
        const uint8_t *e0 = ROWS ? p.ex + ((size_t)g * p.N + (size_t)(n0 + row)) * kb + k0 / 32
                                 : p.ex + ((size_t)g * (p.N / 32) + (size_t)((n0 + row) / 32)) * kb + k0 / 32;
#pragma unroll
        for (int i = 0; i < kMaxKtA / 64; ++i) {
            const int j = 2 * i + h;
            const uint32_t e = row_ok && j < nkb ? (uint32_t)__ldg(e0 + j) : 127u;
            ew |= (uint64_t)e << (8 * i);
        }
    }

    // ---- before the wait: rebuild into shared and tensor memory
    int err = 0;
    {
        const bool ok = mbar_wait_bounded(&wbar, 0u, p.timeout_ns);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            err = 1;
            if (lane == 0) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
        }
    }
    uint32_t mx = 0;
    if (!err) {
#pragma unroll 1
        for (int i = 0; i < kMaxKtA / 64; ++i) {
            const int j = 2 * i + h;  // the warp's block (uniform)
            if (j >= nkb) break;
            const uint32_t e = (uint32_t)(ew >> (8 * i)) & 0xFFu;
            const bool two = __any_sync(0xFFFFFFFFu, e > 134u);
            const uint8_t *src = codes + (j >> 2) * kBoxBytesA + row * 128;
            const int u0 = 2 * (j & 3);
            const uint4 c0 = *reinterpret_cast<const uint4 *>(src + ((u0 ^ (row & 7)) << 4));
            const uint4 c1 = *reinterpret_cast<const uint4 *>(src + (((u0 + 1) ^ (row & 7)) << 4));
            uint32_t a[16];
            rebuild_block_a(c0, c1, e, two, a, mx);
            if (j < 4) {  // columns 0..127: the shared-memory A tiles (atom j / 2, units 4 (j % 2) ..)
                uint8_t *dst = sa + (j >> 1) * kAtomBytesA + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    *reinterpret_cast<uint4 *>(dst + (((4 * (j & 1) + v) ^ (row & 7)) << 4)) =
                        make_uint4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
            } else {      // columns 128..: tensor memory, 16 columns a block
                tmem_st16_a(tlane + acol + 16u * (uint32_t)(j - 4), a);
            }
        }
        if (nan_code_seen_a(mx)) atomicOr(&s_nan[lq], 1u << lane);
    }
    tmem_wait_st_a();
    fence_proxy_async();
    tc_before_a();
    __syncthreads();  // A is complete; the codes' room may take x and the gather tiles
    // Other blocks push into the gather tiles only after every block of the cluster got
    // here (the matching wait precedes the first DSMEM store).
    cluster_arrive_relaxed_a();
    const bool berr = *(volatile int *)&s_err != 0;
    // rows M .. ntok-1 of the x tile are zeros (a chunk of 64 columns is ntok x 128 bytes)
    const int xchunk = p.ntok * 128;
    {
        const int zr = p.ntok - p.M, nch = (k1 - k0 + 63) / 64;
        const int n = nch * zr * 8;
        for (int c = threadIdx.x; c < n; c += kThreadsA) {
            const int ch = c / (zr * 8), rem = c - ch * zr * 8;
            const int t = p.M + (rem >> 3);
            *reinterpret_cast<uint4 *>(xs + ch * xchunk + (t >> 3) * 1024 + (t & 7) * 128 + ((rem & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }

    // ---- the dependency wait: x (and y) belong to the kernels before this one
    pdl_wait();

    // ---- x: M rows x the task's columns, 16-byte copies into the swizzled tile
    {
        const int nu = (k1 - k0) / 8;  // 16-byte units a row
        const uint16_t *xg = p.x + (size_t)g * p.K + k0;
        for (int c = threadIdx.x; c < p.M * nu; c += kThreadsA) {
            const int t = c / nu, v = c - t * nu;
            cp_async_16(xs + (v >> 3) * xchunk + (t >> 3) * 1024 + (t & 7) * 128 + (((v & 7) ^ (t & 7)) << 4),
                        xg + (size_t)t * p.ldx + 8 * v);
        }
        cp_async_wait_all_a();
        fence_proxy_async();
        __syncthreads();
    }

    // ---- MMAs: warp a < nacc (lane 0; its warp-mates held at __syncwarp, as for the weight
    //      copies) issues steps a, a + nacc, ... into accumulator a (columns ntok a ..), in
    //      step order, and commits them to the barrier that waits for all issuers
    const bool mma = !berr && nsteps > 0;
    if (mma && warp < nacc) {
        if (lane == 0) {
            tc_after_a();
            const uint32_t idesc = mma_idesc_a(p.ntok);
            const uint32_t sa_addr = smem_u32(sa), xs_addr = smem_u32(xs);
            const uint32_t d = tmem + (uint32_t)(warp * p.ntok);
            for (int i = warp; i < nsteps; i += nacc) {
                const uint64_t bd = sw128_desc_a(xs_addr + (uint32_t)((i >> 2) * xchunk)) + 2 * (i & 3);
                const uint32_t acc = i >= nacc ? 1u : 0u;
                if (i < 8)
                    umma_ss_a(d, sw128_desc_a(sa_addr + (uint32_t)((i >> 2) * kAtomBytesA)) + 2 * (i & 3), bd,
                              idesc, acc);
                else
                    umma_ts_a(d, tmem + acol + 8u * (uint32_t)(i - 8), bd, idesc, acc);
            }
            umma_commit_a(&dbar);
        }
        __syncwarp();
    }

    // ---- the accumulators, added in order: thread = row, warp half h takes tokens 16 h ..
    float v[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) v[t] = 0.0f;
    bool dwait_ok = true;
    if (mma) {
        dwait_ok = mbar_wait_bounded(&dbar, 0u, p.timeout_ns);
        if (!__all_sync(0xFFFFFFFFu, dwait_ok)) {
            err = 1;
            if (lane == 0) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
        } else if (16 * h < p.ntok) {
            tc_after_a();
            for (int a = 0; a < nacc; ++a) {
                uint32_t r[16];
                tmem_ld16_a(tlane + (uint32_t)(a * p.ntok + 16 * h), r);
#pragma unroll
                for (int t = 0; t < 16; ++t) v[t] = a == 0 ? __uint_as_float(r[t]) : v[t] + __uint_as_float(r[t]);
            }
        }
    }
    if ((s_nan[lq] >> lane) & 1u) {
#pragma unroll
        for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(0x7FC00000u);
    }
    __syncthreads();
    const bool any_err = *(volatile int *)&s_err != 0;

    // ---- push the rows' partials to the blocks that fold them, then the fixed-order sum
    cluster_wait_a();  // every block of the cluster is past its rebuild
    const int L = p.rows_per_rank;
    if (any_err) {
        if (threadIdx.x == 0)  // the folding blocks must not store a sum with garbage in it
            for (int r = 0; r < C; ++r)
                asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(map_to_rank((const void *)&s_err, (uint32_t)r)),
                             "r"(1u)
                             : "memory");
    } else if (row_ok && 16 * h < p.ntok) {
        const int dst_rank = row / L, li = row - dst_rank * L;
        float *dst = gather + ((size_t)tau * L + li) * p.ntok + 16 * h;
        const int nt = min(16, p.M - 16 * h);
#pragma unroll
        for (int t = 0; t < 16; t += 4)
            if (t < nt)
                st_cluster_v4(map_to_rank(dst + t, (uint32_t)dst_rank), v[t], v[t + 1], v[t + 2], v[t + 3]);
    }
    cluster_sync();
    if (!*(volatile int *)&s_err) {
        const int r0 = tau * L;
        const size_t tstride = (size_t)L * p.ntok;  // one task's tile
        for (int c = threadIdx.x; c < p.M * L; c += kThreadsA) {
            const int t = c / L, i = c - t * L;
            const int rr = r0 + i;
            if (rr >= kRowsA || n0 + rr >= p.N) continue;
            const float *gp = gather + (size_t)i * p.ntok + t;
            float yv = 0.0f;
            for (int ss = 0; ss < p.S; ++ss) {
                float ps = gp[(size_t)(ss * p.tps) * tstride];
                for (int uu = 1; uu < p.tps; ++uu) ps = ps + gp[(size_t)(ss * p.tps + uu) * tstride];
                if (p.partials_out)
                    p.partials[(((size_t)ss * p.M + t) * p.G + g) * p.N + n0 + rr] = ps;
                else
                    yv = ss == 0 ? ps : yv + ps;
            }
            if (!p.partials_out) p.y[((size_t)t * p.G + g) * p.N + n0 + rr] = f32_to_bf16_rn(yv);
        }
    }

    // After an error, let the copies and MMAs this block issued finish before it exits.
    if (threadIdx.x == 0 && err) {
        if (nbox > 0 && !p.skip_loads) (void)mbar_wait_bounded(&wbar, 0u, p.timeout_ns);
        if (mma && !dwait_ok) (void)mbar_wait_bounded(&dbar, 0u, p.timeout_ns);
    }
    tc_before_a();
    __syncthreads();
    if (warp == 0) {
        tc_after_a();
        tmem_dealloc_a(tmem, kTmemColsA);
    }
}

// ------------------------------------------------------------------- host side

namespace {

using EncodeTiledFnA = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                    CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

EncodeTiledFnA encode_tiled_fn_a() {
    static EncodeTiledFnA fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnA>(f);
    });
    return fn;
}

// Tensor maps of recently used weights ([rows][K] bytes, box 128 x 128, 128-byte swizzle).
struct MapKeyA {
    const void *ptr;
    long long rows;
    int K;
};

cudaError_t codes_map_a(const uint8_t *w8, long long rows, int K, CUtensorMap *out) {
    static std::mutex mu;
    static MapKeyA keys[64];
    static CUtensorMap maps[64];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (keys[i].ptr == w8 && keys[i].rows == rows && keys[i].K == K) {
            *out = maps[i];
            return cudaSuccess;
        }
    EncodeTiledFnA fn = encode_tiled_fn_a();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap m;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kBoxColsA, (cuuint32_t)kRowsA};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult res = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w8), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return cudaErrorInvalidValue;
    keys[next] = MapKeyA{w8, rows, K};
    maps[next] = m;
    next = (next + 1) % 64;
    if (used < 64) ++used;
    *out = m;
    return cudaSuccess;
}

template <bool ROWS>
cudaError_t configure_ahead() {
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(ahead_kernel<ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytesA);
        if (e != cudaSuccess) return e;
        // two blocks an SM need the largest shared-memory carve-out
        e = cudaFuncSetAttribute(ahead_kernel<ROWS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(ahead_kernel<ROWS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    return cudaSuccess;
}

// Whether clusters of `size` blocks of this kernel can be scheduled on the current device
// (sizes up to 8 always can; larger ones depend on the GPU's cluster limits).  Asked once
// per device and size.
bool cluster_fits(int size) {
    if (size <= kMaxPortableClusterA) return true;
    static int known[64][kMaxClusterA + 1] = {};  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || size > kMaxClusterA) return false;
    int k = __atomic_load_n(&known[dev][size], __ATOMIC_ACQUIRE);
    if (k == 0) {
        k = 2;
        if (configure_ahead<false>() == cudaSuccess && configure_ahead<true>() == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)size, 1, 1);
            cfg.blockDim = dim3(kThreadsA, 1, 1);
            cfg.dynamicSmemBytes = kSmemBytesA;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = (unsigned)size;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, ahead_kernel<false>, &cfg) == cudaSuccess && n > 0) k = 1;
            else (void)cudaGetLastError();
        }
        __atomic_store_n(&known[dev][size], k, __ATOMIC_RELEASE);
    }
    return k == 1;
}

}  // namespace

AheadPlan plan_ahead(int M, int N, int K, int G, int S, bool partials) {
    AheadPlan pl{};
    pl.ok = false;
    if (M < 1 || M > kMaxTokA || S < 1 || N < 1 || K < 32 || G < 1) return pl;
    const int nkb = K / 32;
    pl.S = S;
    pl.chunk_cols = ((nkb + S - 1) / S) * 32;
    pl.tps = std::max(1, (pl.chunk_cols + kMaxKtA - 1) / kMaxKtA);
    pl.kt = ((pl.chunk_cols + pl.tps - 1) / pl.tps + 31) / 32 * 32;
    pl.cluster = S * pl.tps;
    pl.ntok = M <= 16 ? 16 : 32;
    pl.nacc = kAccColsA / pl.ntok;
    pl.rows_per_rank = (kRowsA + pl.cluster - 1) / pl.cluster;
    pl.grid_x = (N + kRowsA - 1) / kRowsA * pl.cluster;
    pl.partials = partials;
    pl.ok = pl.cluster <= kMaxClusterA && pl.kt <= kMaxKtA &&
            kAccColsA + std::max(0, pl.kt - kSmemColsA) / 2 <= kTmemColsA;
    if (pl.ok && pl.cluster > kMaxPortableClusterA) pl.ok = cluster_fits(pl.cluster);
    return pl;
}

cudaError_t launch_ahead(const AheadPlan &pl, const void *x, long long ldx, const uint8_t *w8, const uint8_t *ex,
                         void *y, float *partials, int M, int N, int K, int G, cudaStream_t stream,
                         bool rows_exp) {
    if (!pl.ok || M < 1 || M > kMaxTokA) return cudaErrorInvalidValue;
    if (pl.partials ? partials == nullptr : y == nullptr) return cudaErrorInvalidValue;
    const Options opt = options();
    AheadParams prm;
    cudaError_t e = codes_map_a(w8, (long long)G * N, K, &prm.wmap);
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
    prm.ntok = pl.ntok;
    prm.nacc = pl.nacc;
    prm.cluster = pl.cluster;
    prm.rows_per_rank = pl.rows_per_rank;
    prm.partials_out = pl.partials ? 1 : 0;
    prm.timeout_ns = opt.timeout_ns;
    prm.skip_loads = opt.skip_loads;
    prm.status = status_word();
    if (!prm.status) return cudaErrorInvalidSymbol;

    e = rows_exp ? configure_ahead<true>() : configure_ahead<false>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid_x, (unsigned)G, 1);
    cfg.blockDim = dim3(kThreadsA, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytesA;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (pl.cluster > 1) {
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
    return rows_exp ? cudaLaunchKernelEx(&cfg, ahead_kernel<true>, prm)
                    : cudaLaunchKernelEx(&cfg, ahead_kernel<false>, prm);
}

}  // namespace bsf8
