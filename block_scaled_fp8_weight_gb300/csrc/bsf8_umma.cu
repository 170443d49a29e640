// bsf8_umma.cu -- the tensor-core (tcgen05) GEMM: weight rows stream in, are rebuilt to
// bf16 straight into tensor memory and multiplied by the fifth-generation tensor cores.
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
// tensor cores, not by the weight stream).  The work moves in ring stages of one or two
// 128-column steps (two for 17..128 tokens where they fit: each barrier handoff then serves
// twice the work).  Per stage:
//   * one copy warp loads the stage's codes (per step 128 rows x 128 bytes, one TMA box; up
//     to 8 stages ahead, before the dependency wait too), another its x tiles (per step the
//     token rows, zero-filled to a multiple of 16, x 128 columns, two boxes of 64 with the
//     128-byte swizzle), each wait loop on a warp of its own;
//   * eight rebuild warps turn the codes into exact bf16 weights -- the rebuild of
//     bsf8_device.cuh -- and store them straight into tensor memory as the MMA's A operand
//     (thread = weight row = TMEM lane, two bf16 a column; the two warps of a TMEM lane
//     quarter take 64 columns of each step);
//   * one thread of the MMA warp issues eight tcgen05.mma a step (M = 128, N = tokens,
//     K = 16; A in tensor memory, x from shared memory) into an fp32 accumulator in tensor
//     memory and commits them to the barrier that frees the stage.
// A in tensor memory rather than shared memory: at 192 tokens a step moved ~190 KB through
// shared memory (the copies, the codes read, A written and read, x read), which bound the
// step at ~1500 cycles against 768 of tensor-core work; A in tensor memory takes 64 KB off.
// At the end the rebuild warps read the accumulators back (tcgen05.ld, thread = weight row;
// two warps a TMEM lane quarter split the token columns) and store y (one split), the
// split's sums into shared memory for the cluster of split blocks to fold (2..8 splits in
// one wave), or the split's fp32 partials (the fixed-order reduce follows).
// Codes and stages are rings with full/empty mbarriers; every wait is bounded, and on
// timeout the block records BSF8_ERR_TIMEOUT, stores nothing and returns.
//
// The weights are static, so their copies and the rebuild of the first stages run before
// the programmatic-dependent-launch wait; x is read and y written after it.
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
constexpr int kCodesBytes = kRows * kKB;  // 16 KB of codes a step
constexpr int kACols = kKB / 2;      // TMEM columns of a step's A (two bf16 a 32-bit column)
constexpr int kDsMax = 4, kDcMax = 8;  // ring depths, set per call
// Dynamic shared memory a block: the x tiles of the stage ring (a stage = one step's A slot
// in tensor memory and its x tile) and the codes ring, sized per call (x tiles grow with the
// tokens): 2 .. 4 stages, as many as tensor memory holds A slots for and 144 KB of x tiles
// unless two need more; the codes ring the rest, 2 .. 8 steps.
constexpr int kSmemU = 208 * 1024;
constexpr int kRebuildWarps = 8;     // two a TMEM lane quarter, 64 columns of a step each
// warp 0 copies codes, warp 1 issues MMAs, warps 2 .. 9 rebuild, warp 10 copies x
constexpr int kXWarp = 2 + kRebuildWarps;
constexpr int kThreadsU = (3 + kRebuildWarps) * 32;
constexpr int kMaxTok = 192;  // tokens a block (a token tile; more rows take more tiles)
constexpr int kMaxRowsU = 16384;  // token rows a call (BSF8_MAX_M)
constexpr int kMaxSplitBlocks = 1024;  // 32-column exponent blocks of a split kept in smem
// The tensor core's fp32 accumulation into tensor memory loses accuracy with the number of
// products accumulated in place (measured: the error grows linearly with the steps
// accumulated, about eight times the fp32 index-order sum over 64 steps).  Each run of
// 2^run_shift steps therefore goes to its own accumulator, and the runs are summed in
// fp32 on the CUDA cores in run order: the error is then that of an ordinary fp32 sum.
// Runs are 8 steps (64 MMAs of K = 16, still within the error of an fp32 sum by that
// measurement) past 16 tokens; up to 16 tokens 4 (32 MMAs), unless 4 would keep two blocks
// from sharing an SM or not fit tensor memory at all.
constexpr int kTmemMax = 512;
constexpr int kMaxFold = 8;  // splits a cluster sums in shared memory (the portable cluster size)

struct UmmaParams {
    CUtensorMap cmap;  // w8 as [G*N rows][K columns] bytes, box 128 x 128, 128-byte swizzle
    CUtensorMap xmap;  // x as [M][G][K] bf16 (pitches ldx, K), box 64 x 1 x ntok, 128B swizzle
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S, chunk_cols, ntok;
    int to_partials;  // 1: store fp32 partials P[s] (even with one split), 0: store y
    int ds, dc;       // stage (A slots + x tiles) and codes ring depths
    int sps;          // 128-column steps a stage (and a codes slot) holds: 1 or 2
    int run_shift;    // a run (one accumulator) is 2^run_shift steps
    int cluster_fold; // 1: the S split blocks of a row block form a cluster and sum their
                      // splits through distributed shared memory into y (no partials)
    int tcols;        // tensor memory columns a block allocates (A slots, then accumulators)
    unsigned long long timeout_ns;
    int skip_loads;
    int *status;
};

__device__ __forceinline__ uint64_t evict_first_policy_u() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t evict_normal_policy_u() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
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

// D (+)= A * B with A in tensor memory (lane = row of A, 8 columns = K 16 of bf16) and B in
// shared memory (descriptor).
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// 32 registers of this thread -> columns [taddr, taddr + 32) of its TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t max_xorsign_abs_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ bool nan_code_seen_u(uint32_t mx) {
    return (mx & 0x7FFFu) >= 0x07F0u || ((mx >> 16) & 0x7FFFu) >= 0x07F0u;
}

// Rebuilds one 32-column block of this thread's row (c0: columns 0..15, c1: 16..31) to bf16,
// a[i] = bf16x2(column 2i, column 2i + 1).  TWO: the scale 2^(e-127) in two multiplies (the
// first by 2^120, so that no intermediate leaves bf16's range), exact for every exponent
// byte; otherwise e <= 134 and one multiply by 2^(e-7).  mx keeps the largest magnitude
// pattern before scaling (an e4m3 NaN code spreads to 0x07F0, above every finite code's
// 0x07E0).  A template, so that the warp-uniform choice costs one branch a block.
template <bool TWO>
__device__ __forceinline__ void rebuild_block_u(const uint4 &c0, const uint4 &c1, uint32_t s1, uint32_t s2,
                                                uint32_t (&a)[16], uint32_t &mx) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t t0, t1;
        asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w[i]));
        asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w[i]));
        t0 = (t0 << 4) & 0x87F087F0u;
        t1 = (t1 << 4) & 0x87F087F0u;
        mx = max_xorsign_abs_u(mx, max_xorsign_abs_u(t0, t1));
        uint32_t lo = bf16x2_mul(t0, s1), hi = bf16x2_mul(t1, s1);
        if (TWO) {
            lo = bf16x2_mul(lo, s2);
            hi = bf16x2_mul(hi, s2);
        }
        a[2 * i] = lo;
        a[2 * i + 1] = hi;
    }
}

// Shared-memory address `a` of this CTA mapped into cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_u(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32_u(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cluster_v4_u(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
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

template <int SPS>  // 128-column steps a ring stage holds (1 or 2)
__global__ void __launch_bounds__(kThreadsU, 2) umma_kernel(const __grid_constant__ UmmaParams p) {
    extern __shared__ uint8_t dyn_smem[];
    uint8_t *const base = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    uint8_t *const sX = base;                                   // ds x ntok x 256 B
    uint8_t *const sC = sX + p.ds * p.sps * p.ntok * 256;       // dc x sps x 16 KB
    // full_c: a step's codes landed (TMA); empty_c: its rebuild read them (8 warps);
    // full_x: a step's x tile landed (TMA); full_s: the stage is ready for the MMAs (8 rebuild
    // warps, each after its part of A is in tensor memory; warp 2 after it also saw the x
    // tile land, and all of them on a ragged last step, after they zeroed the x tail);
    // empty_s: the stage's MMAs finished (commit); d_full: every MMA finished (commit).
    __shared__ __align__(8) uint64_t full_c[kDcMax], empty_c[kDcMax];
    __shared__ __align__(8) uint64_t full_x[kDsMax], full_s[kDsMax], empty_s[kDsMax], d_full;
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
    const int nrun = (nkb + (1 << p.run_shift) - 1) >> p.run_shift;  // accumulators (runs of steps)
    const int xbytes = p.ntok * 256;  // a step's x tile: two 64-column atoms
    const int kDs = p.ds, kDc = p.dc;  // ring depths of this call
    constexpr int sps = SPS;           // steps a stage
    const int nstg = (nkb + sps - 1) / sps;  // stages of the split
    const int cslot = sps * kCodesBytes, xslot = sps * xbytes;  // bytes of a codes slot, an x stage
    const uint32_t acols = (uint32_t)(sps * kACols);            // TMEM columns of a stage's A
    const uint32_t dbase = (uint32_t)kDs * acols;  // first accumulator column (A slots first)

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDcMax; ++i) {
            mbar_init(&full_c[i], 1);
            mbar_init(&empty_c[i], kRebuildWarps);
        }
        for (int i = 0; i < kDsMax; ++i) {
            mbar_init(&full_x[i], 1);
            mbar_init(&full_s[i], kRebuildWarps);
            mbar_init(&empty_s[i], 1);
        }
        mbar_init(&d_full, 1);
        s_err = 0;
        for (int i = 0; i < 4; ++i) s_nan[i] = 0;
        fence_mbar_init();
        prefetch_tmap(&p.cmap);
        prefetch_tmap(&p.xmap);
    }
    if (warp == 1) tmem_alloc_u(&s_tmem, (uint32_t)p.tcols);
    tc_before();
    __syncthreads();
    tc_after();
    pdl_trigger();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ codes
        if (lane == 0) {  // static, streamed ahead from the start
            // read once a call with one token tile (evict first); with more, every tile's blocks
            // read the same codes, so they stay (M = 1024: 79 MB from DRAM for 50 MB of operands)
            const uint64_t pol = gridDim.z > 1 ? evict_normal_policy_u() : evict_first_policy_u();
            int n = 0;
            bool bad = false;
            // ring slot and its use's parity by counters (a division by the run-time depth costs
            // a reciprocal sequence a step)
            int cs = 0;
            uint32_t ph = 0;
            for (int st = 0; st < nstg; ++st, cs = cs + 1 == kDc ? 0 : cs + 1, ph ^= cs == 0 ? 1u : 0u) {
                if (st >= kDc && !mbar_wait_bounded(&empty_c[cs], ph ^ 1u, p.timeout_ns)) {
                    bad = true;
                    break;
                }
                const int ns = min(sps, nkb - st * sps);  // steps of this stage
                mbar_arrive_expect_tx(&full_c[cs], (uint32_t)(ns * kCodesBytes));
                if (!p.skip_loads)
#pragma unroll
                    for (int j = 0; j < sps; ++j)
                        if (j < ns)
                            tma_2d_hint_u(sC + cs * cslot + j * kCodesBytes, &p.cmap, k0 + (st * sps + j) * kKB,
                                          g * p.N + row0, &full_c[cs], pol);
                ++n;
            }
            if (bad) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
            if (*(volatile int *)&s_err && !p.skip_loads)  // let issued copies land (bounded)
                for (int i = max(0, n - kDc); i < n; ++i)
                    (void)mbar_wait_bounded(&full_c[i % kDc], (uint32_t)((i / kDc) & 1), p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == kXWarp) {
        // ------------------------------------------------------------ x, after the dependency wait
        if (lane == 0) {
            pdl_wait();
            int n = 0;
            bool bad = false;
            int ss = 0;
            uint32_t ph = 0;
            for (int st = 0; st < nstg; ++st, ss = ss + 1 == kDs ? 0 : ss + 1, ph ^= ss == 0 ? 1u : 0u) {
                if (st >= kDs && !mbar_wait_bounded(&empty_s[ss], ph ^ 1u, p.timeout_ns)) {
                    bad = true;
                    break;
                }
                const int ns = min(sps, nkb - st * sps);
                mbar_arrive_expect_tx(&full_x[ss], (uint32_t)(ns * xbytes));
                if (!p.skip_loads)
#pragma unroll
                    for (int j = 0; j < sps; ++j) {
                        if (j >= ns) break;
                        uint8_t *xt = sX + ss * xslot + j * xbytes;
                        const int kc = k0 + (st * sps + j) * kKB;
                        tma_3d_u(xt, &p.xmap, kc, g, tok0, &full_x[ss]);
                        tma_3d_u(xt + xbytes / 2, &p.xmap, kc + kHalf, g, tok0, &full_x[ss]);
                    }
                ++n;
            }
            if (bad) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
            if (*(volatile int *)&s_err && !p.skip_loads)
                for (int i = max(0, n - kDs); i < n; ++i)
                    (void)mbar_wait_bounded(&full_x[i % kDs], (uint32_t)((i / kDs) & 1), p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue: one thread
        // One wait, eight MMAs and one commit a step, nothing else: every instruction of this
        // chain queues behind the rebuild warps' shared- and tensor-memory traffic (~100
        // cycles each when the loop also synchronised its warp).
        if (lane == 0) {
            const uint32_t idesc = mma_idesc(p.ntok);
            bool bad = false;
            int ss = 0;
            uint32_t ph = 0;
            for (int st = 0; st < nstg; ++st, ss = ss + 1 == kDs ? 0 : ss + 1, ph ^= ss == 0 ? 1u : 0u) {
                if (!mbar_wait_bounded(&full_s[ss], ph, p.timeout_ns)) {
                    bad = true;
                    break;
                }
                tc_after();
                const int ns = min(sps, nkb - st * sps);
#pragma unroll
                for (int j = 0; j < sps; ++j) {
                    if (j >= ns) break;
                    const int kb = st * sps + j;
                    const uint32_t sb = smem_u32(sX + ss * xslot + j * xbytes);
                    const uint32_t ta = tmem + (uint32_t)ss * acols + (uint32_t)(j * kACols);
                    const uint32_t dcol = tmem + dbase + (uint32_t)((kb >> p.run_shift) * p.ntok);  // this run's accumulator
                    const bool run_start = (kb & ((1 << p.run_shift) - 1)) == 0;
#pragma unroll
                    for (int ks = 0; ks < kKB / 16; ++ks) {  // x: atom column ks / 4, +32 bytes a K slice
                        const uint64_t bd = sw128_desc(sb + (ks >> 2) * (xbytes / 2)) + 2 * (ks & 3);
                        umma_ts(dcol, ta + 8u * (uint32_t)ks, bd, idesc, (!run_start || ks > 0) ? 1u : 0u);
                    }
                }
                umma_commit(&empty_s[ss]);
            }
            if (bad) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
            umma_commit(&d_full);  // completes once every MMA above has finished
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ rebuild + epilogue
        const int qd = warp & 3;               // TMEM lane quarter this warp may access
        const int part = (warp - 2) >> 2;      // 0, 1: the step's columns 64 part .. (rebuild),
                                               //       the token chunks 16 part + 32 i (epilogue)
        const int row = 32 * qd + lane;        // this thread's weight row in the block = TMEM lane
        const int n = row0 + row;
        const bool rows_ok = row0 + 32 * qd < p.N;  // warp-uniform (N is a multiple of 32)
        const int tail = (k1 - k0) % kKB;      // columns of the last step inside the split (0: all)
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
        const uint8_t *erow = s_exp[qd];
        const uint32_t tlane = tmem + ((uint32_t)(32 * qd) << 16);
        uint32_t mx = 0;
        bool bad = false;
        int cs = 0, ss = 0;          // ring slots, and the parities of their current uses
        uint32_t cph = 0, sph = 0;
        for (int st = 0; st < nstg; ++st, cs = cs + 1 == kDc ? 0 : cs + 1, cph ^= cs == 0 ? 1u : 0u,
                 ss = ss + 1 == kDs ? 0 : ss + 1, sph ^= ss == 0 ? 1u : 0u) {
            if (!warp_wait(&full_c[cs], cph, p.timeout_ns) ||
                (st >= kDs && !warp_wait(&empty_s[ss], sph ^ 1u, p.timeout_ns))) {
                bad = true;
                break;
            }
            tc_after();  // the MMAs that read this A slot have finished
            const int ns = min(sps, nkb - st * sps);
#pragma unroll
            for (int j = 0; j < sps; ++j) {
                if (j >= ns) break;
                const int kb = st * sps + j;
                const uint8_t *crow = sC + cs * cslot + j * kCodesBytes + row * 128;
                uint32_t a[32];
#pragma unroll
                for (int b = 0; b < 2; ++b) {  // the warp's two 32-column blocks of the step
                    const int cb = 2 * part + b;   // block inside the step
                    const int kcol = k0 + kb * kKB + 32 * cb;
                    uint32_t ab[16];
                    if (rows_ok && kcol < k1) {    // warp-uniform
                        // codes: 128-byte rows with the 128-byte swizzle (unit u of row r at u ^ r % 8)
                        const uint4 c0 = *reinterpret_cast<const uint4 *>(crow + (((2 * cb) ^ (row & 7)) << 4));
                        const uint4 c1 = *reinterpret_cast<const uint4 *>(crow + (((2 * cb + 1) ^ (row & 7)) << 4));
                        const uint32_t e = erow[(kcol - k0) / 32];  // one exponent a warp
                        if (e > 134u) {
                            const uint32_t bb = e << 7;  // 2^(e-127)
                            rebuild_block_u<true>(c0, c1, 0x7B807B80u, bb | (bb << 16), ab, mx);
                        } else {
                            const uint32_t bb = (e + 120u) << 7;  // 2^(e-7)
                            rebuild_block_u<false>(c0, c1, bb | (bb << 16), 0u, ab, mx);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) ab[i] = 0u;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) a[16 * b + i] = ab[i];
                }
                tmem_st32(tlane + (uint32_t)ss * acols + (uint32_t)(j * kACols + 32 * part), a);
            }
            tmem_wait_st();
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_c[cs]);
            // The stage's x tiles must have landed before the MMAs read them: one warp sees to
            // that (each wait costs its warp a few hundred cycles under the step's traffic),
            // all of them in the stage of a ragged last step, whose tail they zero.
            const bool tail_stage = st == nstg - 1 && tail != 0;
            if ((warp == 2 || tail_stage) && !warp_wait(&full_x[ss], sph, p.timeout_ns)) {
                bad = true;
                break;
            }
            if (tail_stage) {
                // x columns past the split's end belong to the next split: zero them (the
                // weights there are zero, and 0 * inf would be NaN); 16 units of 8 columns
                uint8_t *xt = sX + ss * xslot + (ns - 1) * xbytes;
                const int fu = tail / 8, units = 16 - fu;
                for (int i = threadIdx.x - 64; i < p.ntok * units; i += kRebuildWarps * 32) {
                    const int r = i / units, u = fu + i % units;
                    *reinterpret_cast<uint4 *>(xt + (u >> 3) * (xbytes / 2) + (r >> 3) * 1024 + (r & 7) * 128 +
                                               (((u & 7) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(&full_s[ss]);
        }
        if (bad) {
            *(volatile int *)&s_err = 1;
            if (lane == 0) report_timeout(p.status);
        }
        // rows with an e4m3 NaN code, as bits of their TMEM lane quarter's mask
        const uint32_t nmask = __ballot_sync(0xFFFFFFFFu, nan_code_seen_u(mx));
        if (lane == 0 && nmask) atomicOr(&s_nan[qd], nmask);

        pdl_wait();  // y may still be read by the kernels before this one
        const bool dok = warp_wait(&d_full, 0u, p.timeout_ns);
        named_sync_rebuild();  // every rebuild warp has posted its NaN rows
        tc_after();
        const bool store = dok && !*(volatile int *)&s_err && n < p.N;
        const bool poison = (s_nan[qd] >> lane) & 1u;
        // Uniform conditions are taken once a 16-token chunk, and the NaN rows by a select: a
        // branch per element (each with its reconvergence) cost ~3x the loads and stores.
        const int mrows = p.M - tok0;  // token rows of this tile that exist
        const size_t mstride = (size_t)p.G * p.N;  // one token row further in y or P[s]
        for (int c0 = 16 * part; store && c0 < p.ntok && c0 < mrows; c0 += 32) {
            float acc[16];
            if (nrun > 0) {
                uint32_t r[16];
                tmem_ld16(tlane + dbase + (uint32_t)c0, r);
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = __uint_as_float(r[j]);
            } else {  // a split past K's end (more splits than 32-column blocks fill): zeros
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
            }
            for (int run = 1; run < nrun; ++run) {  // the runs' accumulators, in run order
                uint32_t r[16];
                tmem_ld16(tlane + dbase + (uint32_t)(run * p.ntok + c0), r);
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] += __uint_as_float(r[j]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = poison ? __uint_as_float(0x7FC00000u) : acc[j];
            const size_t o0 = ((size_t)(tok0 + c0) * p.G + g) * p.N + n;
            const int mj = min(16, mrows - c0);
            if (p.cluster_fold) {  // the split's sums, token-major, in the freed stage memory
                float *f = reinterpret_cast<float *>(base) + c0 * kRows + row;
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j * kRows] = acc[j];
            } else if (p.to_partials) {
                float *dst = p.partials + (size_t)split * p.M * mstride + o0;
                if (mj == 16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[j * mstride] = acc[j];
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < mj) dst[j * mstride] = acc[j];
                }
            } else {
                uint16_t *dst = p.y + o0;
                if (mj == 16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[j * mstride] = f32_to_bf16_rn(acc[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < mj) dst[j * mstride] = f32_to_bf16_rn(acc[j]);
                }
            }
        }
        if (!dok && lane == 0) {
            *(volatile int *)&s_err = 1;
            report_timeout(p.status);
        }
    }

    tc_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA must be finished before its accumulator columns are freed (bounded)
        (void)mbar_wait_bounded(&d_full, 0u, p.timeout_ns);
        tc_after();
        tmem_dealloc_u(tmem, (uint32_t)p.tcols);
    }
    if (p.cluster_fold) {
        // The cluster holds the S splits of this row block (rank = split).  Every block has
        // put its split's sums in its shared memory; block `split` adds its slice of the
        // tokens over the ranks in split order -- ((P0 + P1) + P2) + ..., fp32, as the reduce
        // kernel does -- and stores y.  No block stores if any of them gave up a wait.
        __shared__ int s_fold_ok;
        cluster_sync();
        if (threadIdx.x == 0) {
            uint32_t bad = 0;
            for (int r = 0; r < p.S; ++r) bad |= ld_cluster_u32_u(mapa_u(smem_u32(&s_err), (uint32_t)r));
            s_fold_ok = bad == 0;
        }
        __syncthreads();
        if (s_fold_ok) {
            const int mrows = min(p.ntok, p.M - tok0);
            const int ts = (mrows + p.S - 1) / p.S;
            const int m_lo = min(mrows, split * ts), m_hi = min(mrows, m_lo + ts);
            const int q4 = min(kRows, p.N - row0) / 4;  // 4-row groups that exist
            const uint32_t fbase = smem_u32(base);
            for (int i = threadIdx.x; i < (m_hi - m_lo) * q4; i += blockDim.x) {
                const int ml = m_lo + i / q4, rr = 4 * (i % q4);
                const uint32_t a = fbase + (uint32_t)((ml * kRows + rr) * 4);
                float4 pv[kMaxFold];
#pragma unroll
                for (int r = 0; r < kMaxFold; ++r)
                    if (r < p.S) pv[r] = ld_cluster_v4_u(mapa_u(a, (uint32_t)r));
                float4 v = pv[0];
#pragma unroll
                for (int r = 1; r < kMaxFold; ++r)
                    if (r < p.S) {
                        v.x += pv[r].x;
                        v.y += pv[r].y;
                        v.z += pv[r].z;
                        v.w += pv[r].w;
                    }
                uint16_t *dst = p.y + ((size_t)(tok0 + ml) * p.G + g) * p.N + row0 + rr;
                const uint16_t b0 = f32_to_bf16_rn(v.x), b1 = f32_to_bf16_rn(v.y), b2 = f32_to_bf16_rn(v.z),
                               b3 = f32_to_bf16_rn(v.w);
                if ((reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {  // N, row0, rr: multiples of 4
                    *reinterpret_cast<uint2 *>(dst) =
                        make_uint2((uint32_t)b0 | ((uint32_t)b1 << 16), (uint32_t)b2 | ((uint32_t)b3 << 16));
                } else {
                    dst[0] = b0;
                    dst[1] = b1;
                    dst[2] = b2;
                    dst[3] = b3;
                }
            }
        }
        cluster_sync();  // no block leaves while another still reads its shared memory
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

namespace {

int umma_runs(const UmmaPlan &pl) {
    return ((pl.chunk_cols + kKB - 1) / kKB + (1 << pl.run_shift) - 1) >> pl.run_shift;
}

// Tensor memory a block's A slots (kACols columns each) and its runs' accumulators (ntok
// columns each) take.
int umma_tmem_need(const UmmaPlan &pl, int da) { return da * std::max(1, pl.sps) * kACols + umma_runs(pl) * pl.ntok; }

// SMs of the current device (0 without one), looked up once per device.
int sm_count_u() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = __atomic_load_n(&cached[dev], __ATOMIC_ACQUIRE);
    if (c == 0 && cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && c > 0)
        __atomic_store_n(&cached[dev], c, __ATOMIC_RELEASE);
    return c > 0 ? c : 0;
}

}  // namespace

UmmaPlan plan_umma(int M, int N, int K, int G, int S, bool partials) {
    UmmaPlan pl{};
    pl.S = S;
    pl.sps = 1;
    pl.chunk_cols = ((K / 32 + S - 1) / S) * 32;
    pl.ntok = std::min(kMaxTok, (M + 15) / 16 * 16);  // tokens a tile
    pl.ttiles = (M + pl.ntok - 1) / std::max(1, pl.ntok);
    // two A slots and the split's runs of steps (ntok accumulator columns each) in tensor
    // memory (half of it up to 16 tokens, so that two blocks share an SM).  Past 16 tokens,
    // runs of 8 steps: the room they leave takes more stages (mid rows at 128 / 192 tokens:
    // 14.8 / 16.4 -> 14.0 / 15.7 us), and at large M fewer splits (half the partials at 1024
    // rows); up to 16 tokens, runs of 8 only where 4 would not fit.
    pl.run_shift = pl.ntok > 16 ? 3 : 2;
    const int cap = pl.ntok <= 16 ? kTmemMax / 2 : kTmemMax;
    if (umma_tmem_need(pl, 2) > cap) {
        UmmaPlan p8 = pl;
        p8.run_shift = 3;
        if (umma_tmem_need(p8, 2) <= cap || umma_tmem_need(pl, 2) > kTmemMax) pl.run_shift = 3;
    }
    pl.tmem_ok = umma_tmem_need(pl, 2) <= kTmemMax;
    pl.row_blocks = (N + kRows - 1) / kRows;
    pl.grid_x = pl.row_blocks * S;
    // 2..8 splits of a call that wants y, all blocks in one wave: the split blocks of a row
    // block form a cluster and sum in shared memory (mid rows, G = 4, 1024 x 4096, S = 4:
    // 12.6 MB of partials and the reduce pass saved at 192 tokens, 15.5 -> 14.6 us).  Grids of
    // several waves keep the partials (each wave's blocks would wait for their cluster's
    // fold: head-like weight at 128 tokens 85.7 -> 89.0 us); not with two blocks an SM.
    const long long blocks = (long long)pl.row_blocks * S * G * pl.ttiles;
    pl.fold = !partials && S >= 2 && S <= kMaxFold && blocks <= sm_count_u() &&
              !(pl.ntok <= 16 && umma_tmem_need(pl, 2) <= kTmemMax / 2);
    // Two 128-column steps a stage for 17..128 tokens where two stages and two code slots of
    // that size fit: every barrier handoff of the step chain (~300-400 cycles each, traced)
    // then serves twice the work.
    if (pl.tmem_ok && pl.ntok > 16 && pl.ntok <= 128 && (pl.chunk_cols + kKB - 1) / kKB >= 2) {
        UmmaPlan p2 = pl;
        p2.sps = 2;
        if (umma_tmem_need(p2, 2) <= kTmemMax && 1024 + 2 * 2 * pl.ntok * 256 + 2 * 2 * kCodesBytes <= kSmemU)
            pl.sps = 2;
    }
    pl.partials = partials || (S > 1 && !pl.fold);
    pl.ok = M >= 1 && M <= kMaxRowsU && (long long)G * N < (1LL << 31) && K < (1 << 30) && pl.tmem_ok &&
            pl.chunk_cols / 32 <= kMaxSplitBlocks;
    return pl;
}

// Up to 16 tokens two blocks share an SM (rings within ~106 KB, A slots and accumulators
// within half of tensor memory): more blocks in flight to cover the per-step latency of one
// block's pipeline, and no second wave on large N.
bool umma_two_per_sm(const UmmaPlan &pl) { return pl.ntok <= 16 && umma_tmem_need(pl, 2) <= kTmemMax / 2; }

// Splits for the tensor-core kernel: as many as keep every block in one wave (the blocks an
// SM holds at once times the SMs; one block past that waits for a whole block's time -- 17
// splits of the 1152-row weight made 153 blocks on 152 SMs), then enough that the A slots
// and the runs' accumulators fit tensor memory.
int umma_auto_split(int M, int N, int K, int G, int sms) {
    const long long ttiles = (M + kMaxTok - 1) / kMaxTok;
    const long long blocks = (long long)((N + kRows - 1) / kRows) * G * ttiles;
    const int smax = std::max(1, K / 32);
    const int per_sm = umma_two_per_sm(plan_umma(M, N, K, G, 1, false)) ? 2 : 1;
    int S = (int)std::max(1LL, (long long)sms * per_sm / std::max(1LL, blocks));
    S = std::min(S, smax);
    while (S < smax && !plan_umma(M, N, K, G, S, false).ok) ++S;
    return S;
}

int umma_smem_budget(const UmmaPlan &pl) { return umma_two_per_sm(pl) ? 106 * 1024 : kSmemU; }

// Stages (a step's A slot in tensor memory and its x tile): 2 .. 4, as many as tensor memory
// leaves beside the accumulators and as 144 KB of x tiles hold (8 KB with two blocks an SM;
// the codes ring keeps 3 .. 8 slots beside them), at least two.
int umma_stage_depth(const UmmaPlan &pl) {
    const bool two = umma_two_per_sm(pl);
    const int cap = two ? kTmemMax / 2 : kTmemMax;
    const int xcap = std::max(2, (two ? 8 * 1024 : 144 * 1024) / (pl.sps * pl.ntok * 256));
    const int left2 = umma_smem_budget(pl) - 1024 - 2 * pl.sps * kCodesBytes;  // two code slots kept
    int ds = 2;
    while (ds < kDsMax && ds < xcap && umma_tmem_need(pl, ds + 1) <= cap &&
           (ds + 1) * pl.sps * pl.ntok * 256 <= left2)
        ++ds;
    return ds;
}

int umma_codes_depth(const UmmaPlan &pl) {
    const int left = umma_smem_budget(pl) - 1024 - umma_stage_depth(pl) * pl.sps * pl.ntok * 256;
    return std::min(kDcMax, left / (pl.sps * kCodesBytes));
}

// Tensor memory a block allocates: a power of two of at least 32 columns.
int umma_tmem_cols(const UmmaPlan &pl) {
    int c = 32;
    while (c < umma_tmem_need(pl, umma_stage_depth(pl))) c *= 2;
    return c;
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
    prm.cluster_fold = pl.fold ? 1 : 0;
    prm.ds = umma_stage_depth(pl);
    prm.sps = pl.sps;
    prm.run_shift = pl.run_shift;
    prm.dc = umma_codes_depth(pl);
    prm.tcols = umma_tmem_cols(pl);
    if (prm.dc < 2 || prm.tcols > (umma_two_per_sm(pl) ? kTmemMax / 2 : kTmemMax)) return cudaErrorInvalidValue;
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
        for (const void *fn : {(const void *)umma_kernel<1>, (const void *)umma_kernel<2>}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemU);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
        }
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid_x, (unsigned)G, (unsigned)pl.ttiles);
    cfg.blockDim = dim3(kThreadsU, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (opt.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (pl.fold) {  // grid x = row block * S + split: a cluster is one row block's splits
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)pl.S;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return pl.sps == 2 ? cudaLaunchKernelEx(&cfg, umma_kernel<2>, prm) : cudaLaunchKernelEx(&cfg, umma_kernel<1>, prm);
}

}  // namespace bsf8
