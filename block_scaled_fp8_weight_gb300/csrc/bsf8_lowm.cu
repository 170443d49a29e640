// bsf8_lowm.cu -- the decode-ahead GEMM kernel for up to 8 token rows.
//
//   y[m][g][n] = bf16( sum_{s=0..S-1} P[s][m][g][n] ),  summed s = 0, 1, ... in fp32,
//   W[g][n][k] = bf16( e4m3(w8[g][n][k]) * 2^(exp[g][n/32][k/32] - 127) ).
//
// Page: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- _wo_a_partial_w8() and
// _wo_a_mid_kernel() with their fixed-order split-K sums.
//
// A decode-step linear layer runs as one of a chain of dependent launches: its input x is
// written by the kernel just before it, so nothing that reads x can start before that
// kernel has finished (programmatic dependent launch, griddepcontrol.wait).  The weights
// and their exponents are static, so everything that touches only them runs before the
// wait, while the previous kernel is still working:
//
//   1. each warp streams its task's weight boxes (16 rows x 128 columns, up to 4) into
//      shared memory by TMA, rebuilds them exactly to bf16 MMA fragments in registers and
//      parks the fragments in tensor memory (tcgen05.st: 32 columns of the warp's 32 TMEM
//      lanes per box, 128 columns per warp, 256 per block);
//   2. griddepcontrol.wait;
//   3. x arrives (8 token rows x 128 columns per step, rows >= M zero-filled), the warp
//      reads its fragments back (tcgen05.ld) and runs the MMAs, and the block sums its
//      warps' partials in the fixed split order.
//
// After the wait a call costs its x round trip, a few MMAs and the reduction; the rebuild,
// the bulk of the instructions, overlaps the previous kernel.  Two blocks fit on an SM
// (256 TMEM columns each; the shared-memory request keeps a third out), so the next call's
// blocks become resident and rebuild while this call finishes.
//
// Work decomposition (bsf8_stream.cu) with tasks of at most 512 columns: a warp task is 16
// weight rows (one slab) x a column range inside one split; a block's 8 warps hold one
// group of tasks (in-block mode: the splits of its slabs summed in the block), or a block
// is one group of a cluster (cluster mode, the splits of a slab summed over DSMEM) or
// writes fp32 partials (partials mode).  Every block holds exactly one group.
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

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kKS = 128;           // columns per step
constexpr int kSlotBytes = 2048;   // a 16 x 128 weight box, or an 8 x 128 bf16 x tile
constexpr int kPre = 4;            // steps per task, all rebuilt ahead into tensor memory
constexpr int kMaxKt = kPre * kKS; // task columns
constexpr int kRegionBytes = kPre * kSlotBytes;  // a warp's slots
constexpr int kTmemCols = 256;     // per block: 128 columns for each of two warps a quarter
constexpr int kLowTasksPerBlock = 1;  // group mode: tasks of a slab a block holds (see plan_lowm)
// Shared-memory request: 8 warps x 4 slots, padded so that a third block never fits an SM
// (its tensor-memory allocation would wait for one of the other two to finish).
constexpr int kRingBytes = kWarps * kPre * kSlotBytes;  // the warps' slots
constexpr int kGatherTiles = 32;   // group mode: [16 rows][8 tokens] fp32 partial tiles a
                                   // block can receive for the slabs it reduces
constexpr int kSmemBytes = 84 * 1024;
static_assert(kRingBytes + kGatherTiles * 512 + 1024 <= kSmemBytes, "slots fit the request");
static_assert(3 * (kSmemBytes + 1024) > 228 * 1024, "at most two blocks an SM");
static_assert(2 * (kSmemBytes + 1024 + 8 * 1024) <= 228 * 1024, "two blocks fit an SM");

struct LowParams {
    CUtensorMap wmap;  // w8 as a [G*N rows][K columns] byte matrix, box 128 x 16
    const uint16_t *x;  // [M][ldx] bf16
    long long ldx;
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S;
    int chunk_cols, kt, tps, spc, cluster, spl, cps, mode, tpc, to_partials;
    unsigned long long timeout_ns;
    int skip_loads;
    int *status;
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_2d_hint(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 registers of this thread -> columns [taddr, taddr + 32) of its TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t max_xorsign_abs(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// e4m3 bytes -> bf16 patterns e4m3 * 2^-120 (sign-extending byte permute, shift, mask).
__device__ __forceinline__ void spread_codes(uint32_t w, uint32_t &t0, uint32_t &t1) {
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t0) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(t1) : "r"(w));
    t0 = (t0 << 4) & 0x87F087F0u;
    t1 = (t1 << 4) & 0x87F087F0u;
}

__device__ __forceinline__ bool nan_code_seen(uint32_t mx) {
    return (mx & 0x7FFFu) >= 0x07F0u || ((mx >> 16) & 0x7FFFu) >= 0x07F0u;
}

}  // namespace

namespace {

// A warp's task: split s, task u of the split, columns [k0, k1), its slab in the block's
// first group (slab0), the slab stride between groups and the block's group count.
struct Task {
    int s, u, k0, k1, slab0, slab_step, ngroups;
    bool active;
};

__device__ __forceinline__ Task task_of(const LowParams &p, int w) {
    Task t;
    const int tslab = p.S * p.tps;
    t.ngroups = 1;
    t.slab_step = 0;
    if (p.mode == kStreamPartials) {
        t.slab0 = blockIdx.x / p.cps;
        t.s = (blockIdx.x % p.cps) * p.spl + w / p.tps;
        t.u = w % p.tps;
        t.active = w < p.spl * p.tps && t.s < p.S;
    } else {  // group mode: a cluster of p.cluster blocks holds spc slabs x all their tasks
        const int spc = kWarps / p.tpc;
        const int rank = blockIdx.x % p.cluster;
        t.slab0 = (blockIdx.x / p.cluster) * spc + w / p.tpc;
        const int tau = rank * p.tpc + w % p.tpc;
        t.s = tau / p.tps;
        t.u = tau % p.tps;
        t.active = tau < tslab;
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

// Byte offsets of this thread's 16-byte units in a 16 x 128 weight box written with the
// 128-byte swizzle (unit u of row r sits at unit u ^ (r % 8)): row r units 2q, 2q+1 and
// row r+8 units 2q, 2q+1.
// Byte offset, in a 16 x 128 weight box written with the 128-byte swizzle (unit u of row r
// sits at unit u ^ (r % 8)), of row r's 8 codes at columns 32v + 8q .. 32v + 8q + 7.
__device__ __forceinline__ int piece_offset(int r, int q, int v) {
    return r * 128 + (((2 * v + (q >> 1)) ^ (r & 7)) << 4) + 8 * (q & 1);
}

// The column order inside a step.  Thread q of an MMA quad owns the step's columns
// 32v + 8q .. 32v + 8q + 7 for v = 0..3 -- one 8-column piece of each 32-column exponent
// block -- so that the quad's four threads read a token row's x in whole 64-byte runs.
// MMA j = 2v + h takes the piece's columns 4h .. 4h+3 as its k = {2q, 2q+1, 2q+8, 2q+9}
// (the same permutation on both operands leaves every product and every sum unchanged).
//
// Rebuilds this thread's share of one weight box into the A fragments of the step's 8
// MMAs: a[4j..4j+3] = (row r, piece columns 4h, 4h+1), (row r+8, same), (row r, 4h+2,
// 4h+3), (row r+8, same).  mxa / mxb keep the largest rebuilt magnitude of rows r / r+8
// before scaling (an e4m3 NaN code spreads to 0x07F0, above every finite code's 0x07E0).
// e[v]: the exponent byte of block v of the step; with ROWS (one exponent per weight row
// and 32 columns) e[v] is row r's and eb[v] row r+8's.  mine: bit v set where block v of
// the step lies inside the task.
template <bool TWO, bool ROWS>
__device__ __forceinline__ void decode_box(const uint8_t *box, int r, int q, uint32_t mine,
                                           const uint32_t (&e)[4], const uint32_t (&eb)[4],
                                           uint32_t (&a)[32], uint32_t &mxa, uint32_t &mxb) {
    uint2 pa[4], pb[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        if ((mine >> v) & 1u) {
            pa[v] = *reinterpret_cast<const uint2 *>(box + piece_offset(r, q, v));
            pb[v] = *reinterpret_cast<const uint2 *>(box + piece_offset(r + 8, q, v));
        } else {
            pa[v] = pb[v] = make_uint2(0, 0);
        }
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        uint32_t s1, s2 = 0, s1b, s2b = 0;
        if (TWO) {  // exact for every exponent byte: restore e4m3 * 1, then scale by 2^(e-127)
            s1 = s1b = 0x7B807B80u;
            const uint32_t bb = e[v] == 0 ? 0x0040u : (e[v] << 7);
            s2 = bb | (bb << 16);
            const uint32_t b8 = eb[v] == 0 ? 0x0040u : (eb[v] << 7);
            s2b = ROWS ? (b8 | (b8 << 16)) : s2;
        } else {    // e <= 134: one multiply by 2^(e-7)
            const uint32_t b = (e[v] + 120u) << 7;
            s1 = b | (b << 16);
            const uint32_t b8 = (eb[v] + 120u) << 7;
            s1b = ROWS ? (b8 | (b8 << 16)) : s1;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 2 * v + h;
            uint32_t t0, t1, u0, u1;
            spread_codes(h ? pa[v].y : pa[v].x, t0, t1);
            spread_codes(h ? pb[v].y : pb[v].x, u0, u1);
            mxa = max_xorsign_abs(mxa, max_xorsign_abs(t0, t1));
            mxb = max_xorsign_abs(mxb, max_xorsign_abs(u0, u1));
            uint32_t alo = bf16x2_mul(t0, s1), ahi = bf16x2_mul(t1, s1);
            uint32_t blo = bf16x2_mul(u0, s1b), bhi = bf16x2_mul(u1, s1b);
            if (TWO) {
                alo = bf16x2_mul(alo, s2);
                ahi = bf16x2_mul(ahi, s2);
                blo = bf16x2_mul(blo, s2b);
                bhi = bf16x2_mul(bhi, s2b);
            }
            a[4 * j + 0] = alo;
            a[4 * j + 1] = blo;
            a[4 * j + 2] = ahi;
            a[4 * j + 3] = bhi;
        }
    }
}

// The step's 8 MMAs (m16n8k16, rows r / r+8 of the slab, tokens 0..7) in the column order
// above: MMA j = 2v + h multiplies piece v's columns 4h .. 4h+3; xv[v] holds token r's 8
// columns of piece v.  Two accumulators break the dependency chain.
__device__ __forceinline__ void mma_step(const uint32_t (&a)[32], const uint4 (&xv)[4],
                                         float (&acc)[2][4]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 &x = xv[j / 2];
        mma_bf16_16816(acc[j & 1], a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3],
                       (j & 1) ? x.z : x.x, (j & 1) ? x.w : x.y);
    }
}

// 16 bytes of global memory, cached in L2 only (x is written by the kernel before this one;
// after the dependency wait L2 holds its values, while this SM's L1 might not).
__device__ __forceinline__ uint4 ld_cg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_cluster_v2f32(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// Parameters the block reads after the dependency wait, staged in shared memory before it.
// Kernel parameters read right after griddepcontrol.wait are slow to arrive (a measured
// ~0.5 us a call over a handful of reads on the decode-ahead tensor-core kernel), while
// shared memory answers at once.
struct PostParams {
    const uint16_t *x;
    uint16_t *y;
    float *partials;
    long long ldx;
    unsigned long long timeout_ns;
    int *status;
    int M, N, K, G, S, tps, tpc, cluster, mode, cps, spl, skip_loads, to_partials;
};

// Partials mode: red[w] holds warp w's task partial [16 rows][8 tokens]; the block stores
// its splits' fp32 partials (tasks of a split summed in task order).  Stores are skipped
// when the block met an error.
__device__ __forceinline__ void partials_epilogue(const PostParams &q, float (*red)[16][8],
                                                  const volatile int *err, int g) {
    const int mrows = min(8, q.M);
    __syncthreads();
    if (*err) return;
    const int slab = blockIdx.x / q.cps;
    const int per_split = 16 * mrows;
    for (int i = threadIdx.x; i < q.spl * per_split; i += kThreads) {
        const int ls = i / per_split, rem = i - ls * per_split;
        const int m = rem / 16, row = rem - m * 16;
        const int ss = (blockIdx.x % q.cps) * q.spl + ls;
        if (ss >= q.S) continue;
        float ps = red[ls * q.tps][row][m];
        for (int uu = 1; uu < q.tps; ++uu) ps = ps + red[ls * q.tps + uu][row][m];
        q.partials[(((size_t)ss * q.M + m) * q.G + g) * q.N + slab * 16 + row] = ps;
    }
}

// Keeps v in a register as an opaque value, so that the compiler cannot recompute it from
// kernel parameters after the dependency wait.
__device__ __forceinline__ int opaque(int v) {
    asm volatile("mov.b32 %0, %0;" : "+r"(v));
    return v;
}

}  // namespace

// One block: 8 warps.  Warp w owns an 8 KB region of shared memory (4 slots of 2 KB) and
// one mbarrier.  Its task has nst <= 4 steps of 128 columns.
//   before the wait: lane 0 arms the barrier with the task's weight bytes and issues one
//     TMA box (16 rows x 128 columns, 128-byte swizzle) per step into slot t; the warp
//     waits, rebuilds each box into its 32 fragment registers and parks steps 1.. in tensor
//     memory (step 0 stays in registers);
//   after the wait: every thread loads its token row's x for all of the task's steps
//     straight into registers (16-byte loads through L2; a quad's four threads read 64
//     contiguous bytes of a row, see the column order above), then step by step the warp
//     brings the fragments back from tensor memory (tcgen05.ld) and runs the MMAs.
// One barrier covers all of a warp's weight boxes: the copies complete in one transaction
// count, far faster than a barrier per box.
template <bool ROWS>
__global__ void __launch_bounds__(kThreads, 2) lowm_kernel(const __grid_constant__ LowParams p) {
    extern __shared__ uint8_t dyn_smem[];
    // the swizzled boxes need 1024-byte alignment
    uint8_t *ring = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    float *const gather = reinterpret_cast<float *>(ring + kRingBytes);  // group mode tiles
    __shared__ __align__(16) float red[kWarps][16][8];
    __shared__ __align__(8) uint64_t wbar[kWarps];
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ PostParams sp;
    __shared__ long long s_fold_y[kThreads];  // y element this thread folds (-1: none)
    __shared__ int s_fold_t[kThreads];        // its first partial tile (float index)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q = lane & 3, r = lane >> 2;
    const int g = blockIdx.y;
    const int nslabs = p.N / 16;
    const int nst = p.kt / kKS;  // steps of a task (<= kPre)
    const Task me = task_of(p, warp);
    uint8_t *const region = ring + warp * kRegionBytes;
    // every block holds exactly one group (the grid is the plan's, not capped)
    const int slab = me.slab0;
    const bool slab_ok = me.active && me.ngroups > 0 && slab < nslabs;

    if (lane == 0) {
        mbar_init(&wbar[warp], 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) s_err = 0;
    if (threadIdx.x == 32) prefetch_tensormap(&p.wmap);
    if (threadIdx.x == 64) {
        PostParams t;
        t.x = p.x;
        t.y = p.y;
        t.partials = p.partials;
        t.ldx = p.ldx;
        t.timeout_ns = p.timeout_ns;
        t.status = p.status;
        t.M = p.M;
        t.N = p.N;
        t.K = p.K;
        t.G = p.G;
        t.S = p.S;
        t.tps = p.tps;
        t.tpc = p.tpc;
        t.cluster = p.cluster;
        t.mode = p.mode;
        t.cps = p.cps;
        t.spl = p.spl;
        t.skip_loads = p.skip_loads;
        t.to_partials = p.to_partials;
        sp = t;
    }
    if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    // this warp's 128 TMEM columns in its lane quarter
    const uint32_t tbase = s_tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (warp >= 4 ? 128u : 0u);

    // ---- weights (static): all of the task's boxes on one barrier
    int nbox = 0;  // boxes issued (steps whose first column is inside the task)
    if (slab_ok)
        for (int t = 0; t < nst; ++t) nbox += me.k0 + t * kKS < me.k1 ? 1 : 0;
    if (lane == 0) {
        mbar_arrive_expect_tx(&wbar[warp], (uint32_t)(nbox * kSlotBytes));
        if (!p.skip_loads) {
            const uint64_t pol = evict_first_policy();
            for (int t = 0; t < nbox; ++t)
                tma_2d_hint(region + t * kSlotBytes, &p.wmap, me.k0 + t * kKS, g * p.N + slab * 16,
                            &wbar[warp], pol);
        }
    }
    // The task's x rows, pulled into L2 while the previous kernel runs.  They may still
    // change before the wait; a prefetch only moves lines into L2, where the producer's
    // writes land as well, and x is read after the wait through L2 only (ld.global.cg),
    // so the loads see the producer's values.  Where x is already in L2 this costs nothing.
    if (lane < p.M && lane < 8 && me.k1 > me.k0 && warp < p.tpc)
        prefetch_l2(p.x + (size_t)lane * p.ldx + (size_t)g * p.K + me.k0,
                    (uint32_t)((me.k1 - me.k0) * 2));
    // exponent bytes of the task: lane l holds block k0/32 + l of the slab's row block
    const int nkb = (me.k1 - me.k0) / 32;
    const uint32_t ereg =
        slab_ok && lane < nkb
            ? (uint32_t)__ldg(p.ex + (size_t)g * (p.N / 32) * (p.K / 32) +
                              (size_t)(slab / 2) * (p.K / 32) + me.k0 / 32 + lane)
            : 127u;
    // ROWS: the exponents of rows r and r+8 from their rows of exponents (block k0/32 + i)
    const uint8_t *er0 = p.ex + ((size_t)g * p.N + (size_t)slab * 16 + r) * (p.K / 32) + me.k0 / 32;
    const uint8_t *er8 = er0 + (size_t)8 * (p.K / 32);
    uint32_t emax = ereg;
    if (ROWS && slab_ok)
        for (int i = 0; i < nkb; ++i) emax = max(emax, max((uint32_t)__ldg(er0 + i), (uint32_t)__ldg(er8 + i)));
    const bool two = __any_sync(0xFFFFFFFFu, emax > 134u);

    // ---- before the wait: rebuild every step; steps 1.. into tensor memory, step 0 into
    //      registers (the first MMAs after the wait need no tensor-memory round trip)
    int err = 0;
    uint32_t mxa = 0, mxb = 0;
    {
        const bool ok = mbar_wait_bounded(&wbar[warp], 0u, p.timeout_ns);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            err = 1;
            *(volatile int *)&s_err = 1;
            if (lane == 0) report_timeout(p.status);
        }
    }
    auto step_exps = [&](int t, uint32_t (&e)[4], uint32_t (&eb)[4], uint32_t &mine) {
        mine = 0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int blk = 4 * t + v;  // block of the task
            const bool in = !err && slab_ok && blk < nkb;
            mine |= in ? 1u << v : 0u;
            const uint32_t eblk = __shfl_sync(0xFFFFFFFFu, ereg, blk & 31);
            e[v] = ROWS ? (in ? (uint32_t)__ldg(er0 + blk) : 127u) : eblk;
            eb[v] = ROWS ? (in ? (uint32_t)__ldg(er8 + blk) : 127u) : eblk;
        }
    };
    for (int t = 1; t < nst; ++t) {
        uint32_t e[4], eb[4], mine;
        step_exps(t, e, eb, mine);
        uint32_t a[32];
        if (two)
            decode_box<true, ROWS>(region + t * kSlotBytes, r, q, mine, e, eb, a, mxa, mxb);
        else
            decode_box<false, ROWS>(region + t * kSlotBytes, r, q, mine, e, eb, a, mxa, mxb);
        tmem_st32(tbase + 32u * t, a);
    }
    uint32_t cur[32];
    {
        uint32_t e[4], eb[4], mine;
        step_exps(0, e, eb, mine);
        if (two)
            decode_box<true, ROWS>(region, r, q, mine, e, eb, cur, mxa, mxb);
        else
            decode_box<false, ROWS>(region, r, q, mine, e, eb, cur, mxa, mxb);
    }
    tmem_wait_st();

    // ---- everything after the wait that depends only on the weights and the plan, done
    //      now: rows with an e4m3 NaN code, where this warp's partial tile goes, and which
    //      output this thread folds
    uint32_t fa = nan_code_seen(mxa) ? 1u : 0u, fb = nan_code_seen(mxb) ? 1u : 0u;
    fa |= __shfl_xor_sync(0xFFFFFFFFu, fa, 1);
    fa |= __shfl_xor_sync(0xFFFFFFFFu, fa, 2);
    fb |= __shfl_xor_sync(0xFFFFFFFFu, fb, 1);
    fb |= __shfl_xor_sync(0xFFFFFFFFu, fb, 2);
    const int C = p.cluster, spc = kWarps / p.tpc, tslab = p.S * p.tps;
    const int rank = blockIdx.x % C;
    // group mode: the partial tile of this warp's task sits at tile index li * tslab + tau of
    // block rr of the cluster (slab sl of the block group's spc reduced by rank sl % C)
    uint32_t tile_addr = 0;
    {
        const int sl = warp / p.tpc;
        const int rr = sl % C, li = sl / C;
        const int tau = rank * p.tpc + warp % p.tpc;
        float *tile = gather + (size_t)(li * tslab + tau) * 128 + r * 8 + 2 * q;
        tile_addr = C == 1 ? smem_u32(tile) : map_to_rank(tile, (uint32_t)rr);
    }
    // fold: output i of this block (i = thread, thread + 256, ...) is token m, row `row` of
    // local slab lj; fold_n outputs in all
    const int mrows = min(8, p.M), per_slab = 16 * mrows;
    const int nmine = (spc - rank + C - 1) / C;  // slabs rank, rank + C, ...
    const int fold_n = p.mode == kStreamPartials ? 0 : nmine * per_slab;
    long long fold_y = -1;   // y element of this thread's first output
    int fold_t = 0;          // its first tile, as a float index into gather
    if ((int)threadIdx.x < fold_n && fold_n > 0) {
        const int i = threadIdx.x;
        const int lj = i / per_slab, rem = i - lj * per_slab;
        const int m = rem / 16, row = rem - m * 16;
        const int sb = (blockIdx.x / C) * spc + lj * C + rank;
        if (sb < nslabs) {
            fold_y = ((long long)m * p.G + g) * p.N + sb * 16 + row;
            fold_t = lj * tslab * 128 + row * 8 + m;
        }
    }
    s_fold_y[threadIdx.x] = fold_y;  // read back after the wait (kept out of registers)
    s_fold_t[threadIdx.x] = fold_t;
    // held in registers as they are (not recomputed from kernel parameters after the wait)
    const int k0 = opaque(me.k0), k1 = opaque(me.k1);
    const int boxed_steps = opaque(slab_ok ? nbox : 0);
    const int nsteps = opaque(nst);
    const int active = opaque(me.active ? 1 : 0);
    tile_addr = (uint32_t)opaque((int)tile_addr);
    __syncthreads();  // the staged parameters are visible to every thread

    // ---- the dependency wait: x (and y) belong to the kernels before this one
    pdl_wait();
    const PostParams &prm = sp;  // read from shared memory where used

    // ---- x: token r's pieces of every step of the task, straight into registers (rows >= M
    //      and blocks past the task as zeros)
    uint4 xa[kPre][4];
    {
        const bool row_ok = r < prm.M && k1 > k0;
        const uint16_t *xrow = prm.x + (size_t)r * prm.ldx + (size_t)g * prm.K + 8 * q;
#pragma unroll
        for (int t = 0; t < kPre; ++t)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int col = k0 + t * kKS + 32 * v;  // the piece's block
                xa[t][v] = row_ok && t < boxed_steps && col < k1 ? ld_cg_v4(xrow + col) : make_uint4(0, 0, 0, 0);
            }
    }

    // ---- MMAs: step 0's fragments in cur, the others back from tensor memory a step at a time
    float acc[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.0f;
#pragma unroll
    for (int t = 0; t < kPre; ++t) {
        if (t < nsteps) {
            if (t > 0) {
                tmem_ld32(tbase + 32u * t, cur);
                tmem_wait_ld();
            }
            if (!err && t < boxed_steps) mma_step(cur, xa[t], acc);
        }
    }

    // ---- the fixed-order reduction and store
    {
        const float qnan = __uint_as_float(0x7FC00000u);
        float v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            v[c] = acc[0][c] + acc[1][c];
            if ((c < 2 && fa) || (c >= 2 && fb)) v[c] = qnan;
        }
        if (prm.mode == kStreamPartials) {
            *reinterpret_cast<float2 *>(&red[warp][r][2 * q]) = make_float2(v[0], v[1]);
            *reinterpret_cast<float2 *>(&red[warp][r + 8][2 * q]) = make_float2(v[2], v[3]);
            partials_epilogue(prm, red, &s_err, g);
        } else {
            // Group mode: every warp puts its partial tile in the block that reduces its
            // slab (this block when C = 1, else over DSMEM), then each block folds its
            // slabs' tiles in the fixed order.
            if (active) {
                if (prm.cluster == 1) {
                    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(tile_addr), "f"(v[0]), "f"(v[1]) : "memory");
                    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(tile_addr + 8 * 8 * 4), "f"(v[2]), "f"(v[3])
                                 : "memory");
                    if (err) s_err = 1;
                } else {
                    st_cluster_v2f32(tile_addr, v[0], v[1]);
                    st_cluster_v2f32(tile_addr + 8 * 8 * 4, v[2], v[3]);
                    if (err && lane == 0) {  // the reducer must not store a sum with garbage in it
                        const int sl = warp / prm.tpc;
                        const uint32_t ea = map_to_rank((const void *)&s_err, (uint32_t)(sl % prm.cluster));
                        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ea), "r"(1u) : "memory");
                    }
                }
            }
            if (prm.cluster > 1)
                cluster_sync();
            else
                __syncthreads();
            if (!s_err) {
                const int S = prm.S, tps = prm.tps;
                // partials: split ss of output (m, g, n) at P[ss][m][g][n], i.e. y's index
                // plus ss * M * G * N
                const long long mgn = (long long)prm.M * prm.G * prm.N;
                const long long fy = s_fold_y[threadIdx.x];
                if (fy >= 0) {
                    const float *tiles = gather + s_fold_t[threadIdx.x];
                    float y = 0.0f;
                    if (prm.to_partials) {
                        for (int ss = 0; ss < S; ++ss) {
                            float ps = tiles[(ss * tps) * 128];
                            for (int uu = 1; uu < tps; ++uu) ps = ps + tiles[(ss * tps + uu) * 128];
                            prm.partials[fy + ss * mgn] = ps;
                        }
                    } else {
#pragma unroll 8
                        for (int ss = 0; ss < S; ++ss) {
                            float ps = tiles[(ss * tps) * 128];
                            for (int uu = 1; uu < tps; ++uu) ps = ps + tiles[(ss * tps + uu) * 128];
                            y = ss == 0 ? ps : y + ps;
                        }
                        prm.y[fy] = f32_to_bf16_rn(y);
                    }
                }
                // outputs past the first 256 of the block (blocks of several slabs)
                const int nsl = prm.N / 16, C2 = prm.cluster, spc2 = kWarps / prm.tpc;
                const int mr = min(8, prm.M), ps_ = 16 * mr, ts = S * tps;
                for (int i = threadIdx.x + kThreads; i < fold_n; i += kThreads) {
                    const int lj = i / ps_, rem = i - lj * ps_;
                    const int m = rem / 16, row = rem - m * 16;
                    const int sb = (blockIdx.x / C2) * spc2 + lj * C2 + (blockIdx.x % C2);
                    if (sb >= nsl) continue;
                    const float *tiles = gather + (size_t)lj * ts * 128 + row * 8 + m;
                    const long long yi = ((long long)m * prm.G + g) * prm.N + sb * 16 + row;
                    float y = 0.0f;
                    for (int ss = 0; ss < S; ++ss) {
                        float ps = tiles[(ss * tps) * 128];
                        for (int uu = 1; uu < tps; ++uu) ps = ps + tiles[(ss * tps + uu) * 128];
                        if (prm.to_partials)
                            prm.partials[yi + ss * mgn] = ps;
                        else
                            y = ss == 0 ? ps : y + ps;
                    }
                    if (!prm.to_partials) prm.y[yi] = f32_to_bf16_rn(y);
                }
            }
        }
    }

    // After an error, let the weight boxes this warp issued land before the block exits.
    if (err && lane == 0 && nbox > 0 && !prm.skip_loads) (void)mbar_wait_bounded(&wbar[warp], 0u, prm.timeout_ns);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(s_tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------- host side

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
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

// Tensor maps of recently used weights ([rows][K] bytes, box 128 x 16, 128-byte swizzle).
// A map encodes only the address and the shape.
struct MapKey {
    const void *ptr;
    long long rows;
    int K;
};

cudaError_t weight_map(const uint8_t *w8, long long rows, int K, CUtensorMap *out) {
    static std::mutex mu;
    static MapKey keys[64];
    static CUtensorMap maps[64];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (keys[i].ptr == w8 && keys[i].rows == rows && keys[i].K == K) {
            *out = maps[i];
            return cudaSuccess;
        }
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap m;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kKS, 16u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult res = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w8), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return cudaErrorInvalidValue;
    keys[next] = MapKey{w8, rows, K};
    maps[next] = m;
    next = (next + 1) % 64;
    if (used < 64) ++used;
    *out = m;
    return cudaSuccess;
}

}  // namespace

StreamPlan plan_lowm(int M, int N, int K, int G, int S, bool partials) {
    // the same decomposition whether the caller wants y or the partials
    StreamPlan pl = plan_stream_ks(M, N, K, G, S, false, kKS, 1, kMaxKt);
    if (pl.mode == kStreamPartials) {
        pl.tpc = kWarps;
        return pl;
    }
    // Group mode.  A block holds tpc tasks of each of 8 / tpc slabs (the slabs' warps share
    // the tasks' x tiles) and a cluster of ceil(tslab / tpc) blocks holds all of the slabs'
    // tasks.  Where a slab has at most 8 tasks a block holds all of them (a cluster of one):
    // the splits are then summed in the block behind one __syncthreads, with no DSMEM push
    // and no cluster barrier after the wait.  Otherwise fewer tasks a block means less x to
    // fetch after the wait per block, but a larger cluster; kLowTasksPerBlock is the
    // balance, raised until the cluster fits 8.
    const int tslab = S * pl.tps;
    int tpc = kLowTasksPerBlock;
    if (tslab <= kWarps) {
        tpc = 1;
        while (tpc < tslab) tpc *= 2;
    }
    while (tpc < kWarps && (tslab + tpc - 1) / tpc > kMaxClusterSplits) tpc *= 2;
    while (tpc > 1 && tpc / 2 >= tslab) tpc /= 2;  // no more than the slab has
    const int spc = kWarps / tpc, cluster = (tslab + tpc - 1) / tpc;
    if ((spc + cluster - 1) / cluster * tslab > kGatherTiles) {  // too many tiles to gather
        StreamPlan pp = plan_stream_ks(M, N, K, G, S, true, kKS, 1, kMaxKt);
        pp.tpc = kWarps;
        return pp;
    }
    pl.tpc = tpc;
    pl.spc = spc;
    pl.cluster = cluster;
    pl.mode = kStreamGroup;
    pl.grid_x = (N / 16 + pl.spc - 1) / pl.spc * pl.cluster;
    pl.to_partials = partials ? 1 : 0;
    return pl;
}

// Partials mode sums a split's tasks inside one block of 8 warps; group mode clusters of
// at most 8 (the portable size) blocks.
bool lowm_fits(const StreamPlan &pl) {
    if (pl.mode == kStreamPartials) return pl.tps <= kWarps;
    return pl.mode == kStreamGroup && pl.cluster <= kMaxClusterSplits;
}

namespace {

// Shared-memory attributes of one instantiation, set once per device.
template <bool ROWS>
cudaError_t configure_lowm(size_t smem) {
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(lowm_kernel<ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        // two blocks an SM need the largest shared-memory carve-out
        e = cudaFuncSetAttribute(lowm_kernel<ROWS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_lowm(const StreamPlan &pl, const void *x, long long ldx, const uint8_t *w8,
                        const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                        cudaStream_t stream, bool rows_exp) {
    if (M < 1 || M > 8 || pl.nt8 != 1 || pl.m_chunks != 1 || pl.kt > kMaxKt || !lowm_fits(pl))
        return cudaErrorInvalidValue;
    if ((pl.mode == kStreamPartials || pl.to_partials) ? partials == nullptr : y == nullptr)
        return cudaErrorInvalidValue;
    const Options opt = options();
    LowParams prm;
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
    prm.tpc = pl.tpc;
    prm.to_partials = pl.to_partials;
    prm.timeout_ns = opt.timeout_ns;
    prm.skip_loads = opt.skip_loads;
    prm.status = status_word();
    if (!prm.status) return cudaErrorInvalidSymbol;

    const size_t smem = (size_t)kSmemBytes;
    e = rows_exp ? configure_lowm<true>(smem) : configure_lowm<false>(smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    // one group a block: the grid is the plan's (blocks beyond two an SM run in turn)
    cfg.gridDim = dim3((unsigned)pl.grid_x, (unsigned)G, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (pl.mode == kStreamGroup && pl.cluster > 1) {
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
    return rows_exp ? cudaLaunchKernelEx(&cfg, lowm_kernel<true>, prm) : cudaLaunchKernelEx(&cfg, lowm_kernel<false>, prm);
}

}  // namespace bsf8
