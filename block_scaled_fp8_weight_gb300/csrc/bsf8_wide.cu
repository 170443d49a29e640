// bsf8_wide.cu -- the wide-weight GEMM for up to 8 token rows: many 128-row blocks of
// weights streamed by TMA, with the codes widened to f16 by the hardware converter.
//
//   y[m][g][n] = bf16( sum_{s=0..S-1} P[s][m][g][n] ),  summed s = 0, 1, ... in fp32,
//   W[g][n][k] = bf16( e4m3(w8[g][n][k]) * 2^(exp[g][n/32][k/32] - 127) ).
//
// Page: "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- _wo_a_partial_w8() and its
// fixed-order split-K sum.
//
// At M <= 8 the layer does 2*M flops per weight byte; what decides whether the SMs keep
// up with HBM is the work spent per code.  Rebuilding bf16 weights costs about ten
// integer and bf16 instructions per four codes (bsf8_device.cuh).  This kernel forms the
// same products another way:
//  * every e4m3 value is an f16 value, and one cvt.rn.f16x2.e4m3x2 widens two codes
//    exactly (an e4m3 NaN code becomes an f16 NaN, which the MMA carries to its row);
//  * the activations of a split are converted once a block into shared memory as f16,
//    x' = x * 2^-s_m, with one power of two s_m per token row taken from the row's largest
//    magnitude (so that the row's largest x' lies in [2^15, 2^16));
//  * a pair of m16n8k16 f16 MMAs covers the 32 columns of one 32 x 32 exponent block (the
//    k order inside the MMAs is permuted identically for codes and x), and its fp32 sum is
//    scaled by 2^(e-127) with one FMA per accumulator; y = acc * 2^s_m at the end.
// For an exponent byte e in [16, 200] bf16(W) = e4m3 * 2^(e-127) holds without rounding,
// and every product code * x' is exact in the MMA, so the path computes the products
// bf16(W) * x exactly and differs from the rebuild only in the order of the fp32 sums
// (|x'| < 2^16 and |code| <= 448 keep a block's sum below 2^30 and a scaled sum below
// 2^103).  x' is exact where each non-zero |x| is at least 2^(s_m - 17): then its 8
// significant bits sit on or above f16's 2^-24 grid.  A block with an exponent byte
// outside [16, 200], or with an activation that misses that bound for some token row,
// takes the exact bf16 rebuild instead (its sums kept apart, in true units), and so does
// every block when a row's s_m falls outside [-100, 100] (activations near the ends of
// the bf16 range).
//
// Work: a task is (split s, group g, 32-row block); tasks are ordered by split, group and
// row block, and each block of the grid (one an SM) takes a contiguous range of them, so
// the x of a split is converted once for many tasks, and the SMs' shares differ by at most
// one 32-row task.  The codes stream into a ring of 16 KB TMA boxes -- 32 rows x 512
// columns, four 128-byte swizzled chunks through a 3-D view of the codes -- 4 to 12 deep,
// as many as the shared memory left by the f16 x of the M token rows holds (at one block an
// SM the bytes in flight set the bandwidth), by a copy warp that runs ahead of everything
// else: the weights are static, so it never waits for the preceding kernel.  Consumer warp
// w takes all 32 rows and the 64 columns 64w .. 64w + 63 of each box: codes by ldmatrix
// (conflict-free under the swizzle, already in the MMA's A layout), x' as one 16-byte load
// a block shared by both row tiles.  At the end of a task the last warp to post its sums
// adds the eight warps' sums of each row in column order.  x is read and y written after
// the programmatic-dependent-launch wait.  Every wait is bounded; on timeout the block
// records BSF8_ERR_TIMEOUT, stores nothing more and returns.
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <cuda.h>

#include <algorithm>
#include <mutex>

namespace bsf8 {

namespace {

constexpr int kWRows = 32;                   // weight rows a task
constexpr int kWChunk = 128;                 // columns of one 128-byte swizzled box row
constexpr int kWStepK = 512;                 // columns a step: four chunks
constexpr int kWBox = kWRows * kWStepK;      // 16 KB of codes a step
constexpr int kWWarps = 8;                   // consumer warps: two row halves x four chunks
constexpr int kWThreads = (kWWarps + 1) * 32;  // + the copy warp (three warps then share one
                                               // scheduler: at most 168 registers a thread)
constexpr int kWDepthMax = 12;               // ring depth: set per call from the room x leaves
constexpr int kWDepthMin = 4;
// Boxes a ring barrier covers: the copy warp arms one barrier for this many consecutive boxes
// of a task and each consumer warp waits on it and releases it once for all of them.  Every
// handoff costs a consumer warp a few hundred cycles whatever it covers; two boxes a barrier
// took the head-like weight (32768 x 5120) at M = 1 / 6 from 36.9 / 43.8 to 32.2 / 40.3 us.
constexpr int kWBoxesPerBar = 2;
constexpr int kWMaxChunk = 6144;             // columns of a split held as f16 x
constexpr int kWMaxBlocks = kWMaxChunk / 32;
constexpr int kWBadWords = kWMaxBlocks / 32;
constexpr int kWFastLo = 16, kWFastHi = 200;  // exponent bytes of the f16 path
constexpr int kWSmin = -100, kWSmax = 100;    // token scales of the f16 path
static_assert(kWMaxChunk / kWStepK <= 32, "one step word a lane");
// up to 8 token rows: one consumer warp a row in the x scan, tokens rotated mod 8 at a task's end
static_assert(kWWarps == 8, "eight consumer warps, eight token rows");
// dynamic shared memory at most (18 KB of the 227 KB are left to the static arrays):
// alignment slack, the ring and the f16 x of the token rows
constexpr size_t kWSmemMax = 227 * 1024 - 18 * 1024;
constexpr int kWRedSlots = 2;  // tasks whose warp sums may be pending at once

struct WideParams {
    CUtensorMap cmap;  // w8 as (128-column chunk, row, chunk index), box 128 x 32 x 4, 128B swizzle
    const uint16_t *x;
    long long ldx;
    const uint8_t *ex;
    uint16_t *y;
    float *partials;
    int M, N, K, G, S, chunk_cols;
    int tasks;        // S * G * N / 32
    int pitch;        // bytes a token row of f16 x in shared memory
    int depth;        // ring slots
    int to_partials;  // 1: store fp32 partials P[s] (even with one split), 0: store y
    unsigned long long timeout_ns;
    int skip_loads;
    int *status;
};

__device__ __forceinline__ uint64_t evict_first_policy_w() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_3d_w(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap_w(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16) from global src to shared address dst (both
// 16-byte aligned), completing that many bytes of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s_addr(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Four 8 x 16-byte matrices of shared memory (row addresses from lanes 8i .. 8i + 7 for
// matrix i); lane 4 r + q receives bytes 4q .. 4q + 3 of row r of each.
__device__ __forceinline__ uint4 ldsm_x4(uint32_t addr) {
    uint4 v;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 ldg64(const void *p) {
    uint2 v;
    asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u8_w(const uint8_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// The four codes of w as f16: lo = (code0, code1), hi = (code2, code3), exactly.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// D = A * B (first = true) or D += A * B for one m16n8k16 tile of f16 operands, fp32 sums.
__device__ __forceinline__ void mma_f16_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ void mma_f16_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// 2^s as a float for s in [-126, 127].
__device__ __forceinline__ float exp2_int(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// Barrier of the consumer warps only (named barrier 1).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kWWarps * 32) : "memory");
}

__device__ __forceinline__ bool warp_wait_w(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
    const bool ok = mbar_wait_bounded(bar, parity, timeout_ns);
    return __all_sync(0xFFFFFFFFu, ok);
}

// Exponent bytes of the two 32-column blocks blk0, blk0 + 1 (127 past the split's cb).
__device__ __forceinline__ uint32_t load_exp_word(const uint8_t *er, int blk0, int cb) {
    const uint32_t e0 = blk0 < cb ? ldg_u8_w(er + blk0) : 127u;
    const uint32_t e1 = blk0 + 1 < cb ? ldg_u8_w(er + blk0 + 1) : 127u;
    return e0 | (e1 << 8);
}

// s_m of a token row from the largest magnitude bits mx of its split: the largest x' in
// [2^15, 2^16); an all-zero row gets 0; inf / NaN give 113.  ok: s_m lies in the range of
// the f16 path.
__device__ __forceinline__ int row_scale(uint32_t mx, bool &ok) {
    int s = mx == 0 ? 0 : max((int)(mx >> 7), 1) - 142;
    ok = s >= kWSmin && s <= kWSmax;
    return ok ? s : 0;
}

// The 64-byte block at shared address base as 16 bf16 pairs: w[i] = columns (2i, 2i + 1).
__device__ __forceinline__ void load_block64(uint32_t base, uint32_t (&w)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 v = lds128(base + 16 * j);
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
    }
}

// Writes block blk of a token row (its bf16 pairs w, read from base) back to base as f16
// x' = x * 2^-s_m in the MMA B layout, s_m from the row's largest magnitude bits smax, and
// sets bit blk of bad when some non-zero |x| of the block is below 2^(s_m - 17) (x' not
// exact) or s_m is out of the f16 path's range.
__device__ __forceinline__ void convert_block64(const uint32_t (&w)[16], uint32_t base, uint32_t smax, int blk,
                                                uint32_t *bad) {
    bool rok;
    const int sm = row_scale(smax, rok);
    const float sc = exp2_int(-sm);
    const uint32_t thr1 = ((uint32_t)(sm + 110) << 7) - 1u;  // |x| >= 2^(s-17); s >= -100
    uint32_t o[16];
    uint32_t mn = 0xFFFFFFFFu;  // per half: smallest magnitude minus one (zero -> 0xFFFF)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        mn = min_u16x2(mn, ((w[i] | 0x80008000u) - 0x00010001u) ^ 0x80008000u);
        o[i] = pack_f16x2(__uint_as_float(w[i] << 16) * sc, __uint_as_float(w[i] & 0xFFFF0000u) * sc);
    }
    // the 16 bytes at 16q: columns 4q .. 4q + 3 (pairs 2q, 2q + 1) and 16 + 4q ..
    // 16 + 4q + 3 (pairs 8 + 2q, 9 + 2q)
#pragma unroll
    for (int q = 0; q < 4; ++q) sts128(base + 16 * q, o[2 * q], o[2 * q + 1], o[8 + 2 * q], o[9 + 2 * q]);
    if (!rok || min(mn & 0xFFFFu, mn >> 16) < thr1) atomicOr(&bad[blk >> 5], 1u << (blk & 31));
}

// Converts the split's x (token rows 0 .. M-1, columns [k0, k0 + 32 cb) of group g) into
// f16 x' at xh (rows pitch bytes apart; inside each 32-column block of 64 bytes, the 16
// bytes at 16q hold columns 4q .. 4q + 3 and 16 + 4q .. 16 + 4q + 3, the MMA B operand of
// lane quad q), sets s_sx[m] = s_m, and sets bit blk of s_bad for every 32-column block
// whose x' is not exact for some row.  Run by all consumer threads (tid 0 .. 255) between
// consumer barriers.  The rows first come into the same place as raw bf16 (one bulk copy
// a row on `xbar`, phase xphase; a bf16 row takes the bytes its f16 row will), so both
// passes read shared memory: loads from L2 in a loop took 2 to 5 us a conversion.  The
// second pass converts each 64-byte block in place, one thread a block.  Returns false when
// the copies did not land within the bound (nothing is converted then).
__device__ bool convert_x(const WideParams &p, uint32_t xh, int g, int k0, int cb, int tid,
                          uint32_t *s_max, uint32_t *s_bad, int *s_sx, uint64_t *xbar, uint32_t xphase,
                          int *s_xfail) {
    const int nvec = 4 * cb;  // 16-byte vectors of a row
    const int lane = tid & 31;
    if (tid < kWWarps) s_max[tid] = 0;
    if (tid < kWBadWords) s_bad[tid] = 0;
    if (tid == 0) *s_xfail = 0;
    // the previous x' was read by the generic proxy; the copies write through the async one
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    consumers_sync();
    if (tid == 0) {
        mbar_arrive_expect_tx(xbar, (uint32_t)(p.M * 64 * cb));
        const uint16_t *src0 = p.x + (size_t)g * p.K + k0;
        for (int m = 0; m < p.M; ++m)
            bulk_g2s_addr(xh + (uint32_t)(m * p.pitch), src0 + (size_t)m * p.ldx, (uint32_t)(64 * cb), xbar);
    }
    // every consumer thread sees the copies complete (or the bound run out), and the block
    // agrees on the outcome
    if (!mbar_wait_bounded(xbar, xphase, p.timeout_ns)) atomicOr(s_xfail, 1);
    consumers_sync();
    const bool landed = *(volatile int *)s_xfail == 0;
    if (!landed) {  // the copies must land before this memory is used again or freed (bounded)
        (void)mbar_wait_bounded(xbar, xphase, p.timeout_ns);
        consumers_sync();
        return false;
    }
    // pass 1: each row's largest magnitude (bf16 magnitudes order as integers), one warp a
    // row, so that the rows' loads and shuffle chains run side by side
    if ((tid >> 5) < p.M) {
        const uint32_t row = xh + (uint32_t)((tid >> 5) * p.pitch);
        uint32_t mx = 0;
#pragma unroll 4
        for (int v = lane; v < nvec; v += 32) {
            const uint4 u = lds128(row + 16u * (uint32_t)v);
            mx = max_u16x2(mx, max_u16x2(max_u16x2(u.x & 0x7FFF7FFFu, u.y & 0x7FFF7FFFu),
                                         max_u16x2(u.z & 0x7FFF7FFFu, u.w & 0x7FFF7FFFu)));
        }
        uint32_t v = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (lane == 0) s_max[tid >> 5] = v;
    }
    consumers_sync();
    // pass 2: convert each row's 64-byte blocks in place, one thread a (row, block); a block
    // is exact when each non-zero magnitude of every row is >= 2^(s_m - 17)
    if (tid < p.M) {  // a row whose s_m is out of range gets 0 here and every block marked below
        bool ok;
        s_sx[tid] = row_scale(s_max[tid], ok);
    }
    // Units u = tid + 256 j in pairs (j even, j + 1), both blocks' loads ahead of either's
    // arithmetic.
    const int nu = p.M * cb, ustride = kWWarps * 32;
    for (int u0 = tid; u0 < nu; u0 += 2 * ustride) {
        const int u1 = u0 + ustride;
        const int m0 = u0 / cb, b0 = u0 - m0 * cb;
        const uint32_t base0 = xh + (uint32_t)(m0 * p.pitch + 64 * b0);
        uint32_t w0[16], w1[16];
        load_block64(base0, w0);
        if (u1 < nu) {
            const int m1 = u1 / cb, b1 = u1 - m1 * cb;
            const uint32_t base1 = xh + (uint32_t)(m1 * p.pitch + 64 * b1);
            load_block64(base1, w1);
            convert_block64(w0, base0, s_max[m0], b0, s_bad);
            convert_block64(w1, base1, s_max[m1], b1, s_bad);
        } else {
            convert_block64(w0, base0, s_max[m0], b0, s_bad);
        }
    }
    if (tid >= p.M && tid < kWWarps) s_sx[tid] = 0;
    consumers_sync();
    return true;
}

// Step word of the warp's blocks blk0, blk0 + 1 (blk0 even): bit b = block blk0 + b lies
// inside the split, bit 2 + b = it takes the f16 path (exponent byte in range, x' exact in
// every token row).
__device__ __forceinline__ uint32_t step_code(uint32_t E, int blk0, int cb, const uint32_t *bad) {
    if (blk0 >= cb) return 0;
    const uint32_t anybad = bad[blk0 >> 5] >> (blk0 & 31);
    uint32_t code = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        if (blk0 + b >= cb) break;
        code |= 1u << b;
        const uint32_t e = (E >> (8 * b)) & 0xFFu;
        if (e >= (uint32_t)kWFastLo && e <= (uint32_t)kWFastHi && !((anybad >> b) & 1u)) code |= 4u << b;
    }
    return code;
}

// One 32-column block of one 16-row tile by the exact bf16 rebuild.  d: the codes as the
// ldmatrix operands (rows r, r + 8 of the first 16 columns, then of the second 16; lane
// quad q holds columns 4q .. 4q + 3 of each); xp: token row r's x at the block (nullptr: a
// zero row).  Returns the block's sums in true units.  Kept out of line: it runs only for
// blocks with an exponent byte or activations outside the f16 path.
__device__ __noinline__ float4 slow_block(uint4 d, uint32_t e, const uint16_t *xp, int q) {
    const Scale sc = make_scale(e);
    float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint32_t ra[2] = {d.x, d.z}, rb8[2] = {d.y, d.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint2 xv = xp ? ldg64(xp + 16 * h + 4 * q) : make_uint2(0, 0);
        uint32_t a0, a2, a1, a3;
        rebuild4(ra[h], sc, a0, a2);
        if (nan_code_mask(ra[h])) patch_nan_codes(ra[h], a0, a2);
        rebuild4(rb8[h], sc, a1, a3);
        if (nan_code_mask(rb8[h])) patch_nan_codes(rb8[h], a1, a3);
        mma_bf16_16816(t, a0, a1, a2, a3, xv.x, xv.y);
    }
    return make_float4(t[0], t[1], t[2], t[3]);
}

// One 32-column block of one 16-row tile on the f16 path: two MMAs (the block's first and
// second 16 columns) into t.
__device__ __forceinline__ void f16_block(float (&t)[4], uint4 d, uint4 xv) {
    uint32_t a0, a1, a2, a3;
    e4m3x4_to_f16(d.x, a0, a2);
    e4m3x4_to_f16(d.y, a1, a3);
    mma_f16_first(t, a0, a1, a2, a3, xv.x, xv.y);
    e4m3x4_to_f16(d.z, a0, a2);
    e4m3x4_to_f16(d.w, a1, a3);
    mma_f16_acc(t, a0, a1, a2, a3, xv.z, xv.w);
}

}  // namespace

__global__ void __launch_bounds__(kWThreads, 1) wide_kernel(const __grid_constant__ WideParams p) {
    extern __shared__ uint8_t dyn_smem[];
    uint8_t *const ring = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    const int D = p.depth;
    const int DB = D / kWBoxesPerBar;  // ring barriers (groups of kWBoxesPerBar boxes)
    uint8_t *const xh = ring + D * kWBox;  // f16 x of token rows 0 .. M-1
    __shared__ __align__(8) uint64_t full[kWDepthMax], empty[kWDepthMax], xbar;
    __shared__ int s_xfail;
    __shared__ uint32_t s_bad[kWBadWords];  // blocks of the split with an inexact x'
    __shared__ uint32_t s_max[kWWarps];     // per token row: largest magnitude bits
    __shared__ int s_sx[kWWarps];           // per token row: s_m
    __shared__ int s_err;
    // task-end slots: the chunk sums of a task's rows, the warps that have posted theirs,
    // and the laps of the slot already summed
    __shared__ __align__(16) float red[kWRedSlots][kWWarps][kWRows][kWWarps];
    __shared__ int red_cnt[kWRedSlots], red_done[kWRedSlots];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RB = p.N / kWRows;
    const int t_begin = (int)((long long)blockIdx.x * p.tasks / gridDim.x);
    const int t_end = (int)((long long)(blockIdx.x + 1) * p.tasks / gridDim.x);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWDepthMax; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWWarps);
        }
        mbar_init(&xbar, 1);
        s_err = 0;
        for (int i = 0; i < kWRedSlots; ++i) red_cnt[i] = red_done[i] = 0;
        fence_mbar_init();
        prefetch_tmap_w(&p.cmap);
    }
    __syncthreads();
    pdl_trigger();

    if (warp == kWWarps) {
        // ------------------------------------------------------------ codes
        if (lane == 0) {
            const uint64_t pol = evict_first_policy_w();
            int n = 0, slot = 0;
            uint32_t phase = 0;  // of the ring's current lap
            bool bad = false;
            for (int t = t_begin; t < t_end && !bad; ++t) {
                const int s = t / (p.G * RB), g = (t / RB) % p.G, rb = t % RB;
                const int k0 = min(p.K, s * p.chunk_cols), k1 = min(p.K, k0 + p.chunk_cols);
                const int nst = (k1 - k0 + kWStepK - 1) / kWStepK;
                for (int st0 = 0; st0 < nst; st0 += kWBoxesPerBar) {
                    // from the second lap on, the group's previous boxes must have been consumed
                    if (n >= DB && !mbar_wait_bounded(&empty[slot], phase ^ 1u, p.timeout_ns)) {
                        bad = true;
                        break;
                    }
                    const int nb = min(kWBoxesPerBar, nst - st0);  // boxes of this group
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(nb * kWBox));
                    if (!p.skip_loads)
                        for (int j = 0; j < nb; ++j)
                            tma_3d_w(ring + (kWBoxesPerBar * slot + j) * kWBox, &p.cmap, 0, g * p.N + rb * kWRows,
                                     (k0 + (st0 + j) * kWStepK) / kWChunk, &full[slot], pol);
                    ++n;
                    if (++slot == DB) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (bad) {
                *(volatile int *)&s_err = 1;
                report_timeout(p.status);
            }
            // every issued box lands before the block may exit (bounded)
            if (!p.skip_loads)
                for (int i = max(0, n - DB); i < n; ++i)
                    (void)mbar_wait_bounded(&full[i % DB], (uint32_t)((i / DB) & 1), p.timeout_ns);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Warp w takes all 32 rows of a box and its 32-column blocks 2w and 2w + 1 (blocks
    // 4 ch + 2 hb + {0, 1} of the box's chunk ch = w >> 1, hb = w & 1).
    const int tid = threadIdx.x, w = warp, r = lane >> 2, q = lane & 3;
    const int ch = w >> 1, hb = w & 1;
    const uint32_t ring_s = smem_u32(ring), xh_s = smem_u32(xh);
    // ldmatrix row addresses inside a box for row tile rt and block bb: lane 8i + rr gives
    // row 16 rt + rr + 8 (i & 1) of the block's 16-column half i >> 1 (128-byte swizzle)
    uint32_t lmo[2][2];
    {
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int row = 16 * rt + rr + 8 * (mi & 1);
                const int c16 = 2 * (2 * hb + bb) + (mi >> 1);
                lmo[rt][bb] = (uint32_t)(ch * (kWRows * 128) + row * 128 + ((c16 ^ rr) << 4));
            }
    }

    // exponent word of this warp's two blocks in step `lane` of task t
    auto task_exps = [&](int t) -> uint32_t {
        if (t >= t_end) return 0x7F7Fu;
        const int s = t / (p.G * RB), g = (t / RB) % p.G, rb = t % RB;
        const int k0 = min(p.K, s * p.chunk_cols), k1 = min(p.K, k0 + p.chunk_cols);
        const int cb = (k1 - k0) / 32;
        const uint8_t *er = p.ex + ((size_t)g * (p.N / 32) + rb) * (p.K / 32) + k0 / 32;
        return load_exp_word(er, 16 * lane + 2 * w, cb);
    };

    uint32_t En = task_exps(t_begin);  // static: before the dependency wait
    pdl_wait();

    int cur_gs = -1, slot = 0;
    uint32_t phase = 0, xphase = 0;  // ring and x-copy barrier phases
    bool bad = false;
    const bool xr = r < p.M;  // this thread's B-operand token row is held

    for (int t = t_begin; t < t_end; ++t) {
        const int s = t / (p.G * RB), g = (t / RB) % p.G, rb = t % RB;
        const int k0 = min(p.K, s * p.chunk_cols), k1 = min(p.K, k0 + p.chunk_cols);
        const int nst = (k1 - k0 + kWStepK - 1) / kWStepK, cb = (k1 - k0) / 32;
        const uint32_t E0 = En;
        En = task_exps(t + 1);  // the next task's exponents, in flight meanwhile

        const int gs = s * p.G + g;
        if (gs != cur_gs) {
            consumers_sync();  // every consumer warp is done with the previous x'
            if (!convert_x(p, xh_s, g, k0, cb, tid, s_max, s_bad, s_sx, &xbar, xphase, &s_xfail)) {
                bad = true;
                if (lane == 0) *(volatile int *)&s_err = 1;
            }
            xphase ^= 1u;
            cur_gs = gs;
        }
        const uint32_t C0 = step_code(E0, 16 * lane + 2 * w, cb, s_bad);

        float acc[2][4] = {};   // f16 path, in units of 2^-s_m; [row tile][fragment]
        float accs[2][4] = {};  // rebuild path, in true units
        // x' of token row r at this warp's first block of step 0
        const uint32_t xrow = xh_s + (uint32_t)(r * p.pitch + 128 * w + 16 * q);
        const uint16_t *xg = xr ? p.x + (size_t)r * p.ldx + (size_t)g * p.K + k0 + 64 * w : nullptr;
        for (int st0 = 0; st0 < nst; st0 += kWBoxesPerBar) {
          const int sl = slot;  // the group's barrier
          if (!bad) {
              bad = !warp_wait_w(&full[sl], phase, p.timeout_ns);
              if (bad && lane == 0) *(volatile int *)&s_err = 1;
          }
          for (int j = 0; j < kWBoxesPerBar; ++j) {  // the group's boxes
            const int st = st0 + j;
            if (st >= nst) break;
            if (!bad) {
                const uint32_t E = __shfl_sync(0xFFFFFFFFu, E0, st);
                const uint32_t C = __shfl_sync(0xFFFFFFFFu, C0, st);
                const uint32_t box = ring_s + (uint32_t)((kWBoxesPerBar * sl + j) * kWBox);
                const uint32_t xs = xrow + (uint32_t)(1024 * st);
                if (C == 0xFu) {
                    // the common step: both blocks on the f16 path, written out so that the
                    // loads and the four block-tiles' MMA chains overlap
                    uint4 d[2][2], xv[2];
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) {
                        d[0][bb] = ldsm_x4(box + lmo[0][bb]);
                        d[1][bb] = ldsm_x4(box + lmo[1][bb]);
                        xv[bb] = xr ? lds128(xs + 64 * bb) : make_uint4(0, 0, 0, 0);
                    }
                    float tb[2][2][4];
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb)
#pragma unroll
                        for (int rt = 0; rt < 2; ++rt) f16_block(tb[rt][bb], d[rt][bb], xv[bb]);
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) {
                        const float f = __uint_as_float(((E >> (8 * bb)) & 0xFFu) << 23);  // 2^(e-127)
#pragma unroll
                        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                            for (int c = 0; c < 4; ++c) acc[rt][c] = fmaf(tb[rt][bb][c], f, acc[rt][c]);
                    }
                } else {
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) {
                        if (!((C >> bb) & 1u)) continue;
                        const uint32_t e = (E >> (8 * bb)) & 0xFFu;
                        const uint4 d0 = ldsm_x4(box + lmo[0][bb]), d1 = ldsm_x4(box + lmo[1][bb]);
                        if ((C >> (2 + bb)) & 1u) {
                            const uint4 xv = xr ? lds128(xs + 64 * bb) : make_uint4(0, 0, 0, 0);
                            float t0[4], t1[4];
                            f16_block(t0, d0, xv);
                            f16_block(t1, d1, xv);
                            const float f = __uint_as_float(e << 23);
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                acc[0][c] = fmaf(t0[c], f, acc[0][c]);
                                acc[1][c] = fmaf(t1[c], f, acc[1][c]);
                            }
                        } else {
                            const uint16_t *xp = xg ? xg + kWStepK * st + 32 * bb : nullptr;
                            const float4 v0 = slow_block(d0, e, xp, q), v1 = slow_block(d1, e, xp, q);
                            accs[0][0] += v0.x;
                            accs[0][1] += v0.y;
                            accs[0][2] += v0.z;
                            accs[0][3] += v0.w;
                            accs[1][0] += v1.x;
                            accs[1][1] += v1.y;
                            accs[1][2] += v1.z;
                            accs[1][3] += v1.w;
                        }
                    }
                }
            }
          }
            __syncwarp();
            if (!bad && lane == 0) mbar_arrive(&empty[sl]);
            if (++slot == DB) {
                slot = 0;
                phase ^= 1u;
            }
        }

        // ---- task end: post this warp's sums; the last of the eight warps to post adds
        // the warps' sums of each row in warp (= column) order and stores the task's rows.
        const int li = t - t_begin, rs = li % kWRedSlots, lap = li / kWRedSlots;
        if (lap > 0 && lane == 0) {  // the slot's previous task must have been summed (bounded)
            const uint64_t t0 = global_ns();
            while (*(volatile int *)&red_done[rs] < lap)
                if (global_ns() - t0 > p.timeout_ns) {
                    *(volatile int *)&s_err = 1;
                    bad = true;
                    break;
                }
        }
        bad = __shfl_sync(0xFFFFFFFFu, bad ? 1 : 0, 0) != 0 || bad;
        {
            const int m0 = 2 * q;
            const float f0 = exp2_int(s_sx[m0]), f1 = exp2_int(s_sx[m0 + 1]);
#pragma unroll
            for (int rt = 0; rt < 2; ++rt) {
                *reinterpret_cast<float2 *>(&red[rs][w][16 * rt + r][m0]) =
                    make_float2(fmaf(acc[rt][0], f0, accs[rt][0]), fmaf(acc[rt][1], f1, accs[rt][1]));
                *reinterpret_cast<float2 *>(&red[rs][w][16 * rt + r + 8][m0]) =
                    make_float2(fmaf(acc[rt][2], f0, accs[rt][2]), fmaf(acc[rt][3], f1, accs[rt][3]));
            }
        }
        __syncwarp();
        __threadfence_block();
        int last = 0;
        if (lane == 0) last = atomicAdd(&red_cnt[rs], 1) == kWWarps - 1;
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        if (last) {
            __threadfence_block();
            if (!*(volatile int *)&s_err) {
                const int n = rb * kWRows + lane;  // lane = row of the task
                auto sum_store = [&](int m) {
                    float v = red[rs][0][lane][m];
#pragma unroll
                    for (int ww = 1; ww < kWWarps; ++ww) v += red[rs][ww][lane][m];
                    if (p.to_partials)
                        p.partials[(((size_t)s * p.M + m) * p.G + g) * p.N + n] = v;
                    else
                        p.y[((size_t)m * p.G + g) * p.N + n] = f32_to_bf16_rn(v);
                };
                if (p.M >= 4) {
                    // tokens in a lane-rotated order: in iteration j lane quad k takes token
                    // (j + k) mod 8, so an iteration's loads hit 32 distinct banks (token by
                    // token they hit four, eight ways each); the sum order is the same
#pragma unroll 1
                    for (int j = 0; j < kWWarps; ++j) {
                        const int m = (j + (lane >> 2)) & (kWWarps - 1);
                        if (m < p.M) sum_store(m);
                    }
                } else {
                    for (int m = 0; m < p.M; ++m) sum_store(m);
                }
            }
            __syncwarp();
            if (lane == 0) {
                red_cnt[rs] = 0;
                __threadfence_block();
                *(volatile int *)&red_done[rs] = lap + 1;
            }
        }
    }
    if (bad && lane == 0) report_timeout(p.status);
}

// ------------------------------------------------------------------- host side

namespace {

using EncodeTiledFnW = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnW encode_fn_w() {
    static EncodeTiledFnW fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnW>(f);
    });
    return fn;
}

// Tensor maps of recent code arrays (a map encodes only the address and the shape): the
// [rows][K] bytes viewed as (column within a 128-column chunk, row, chunk), so that one
// box of 128 x 32 x 4 brings 32 rows x 512 columns as four 128-byte swizzled chunks.
// K % 128 == 0: the view covers each row exactly.
cudaError_t codes_map_w(const void *ptr, long long rows, int K, CUtensorMap *out) {
    struct Key {
        const void *ptr;
        long long rows;
        int K;
    };
    static std::mutex mu;
    static Key keys[64];
    static CUtensorMap maps[64];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (keys[i].ptr == ptr && keys[i].rows == rows && keys[i].K == K) {
            *out = maps[i];
            return cudaSuccess;
        }
    EncodeTiledFnW fn = encode_fn_w();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)kWChunk, (cuuint64_t)rows, (cuuint64_t)(K / kWChunk)};
    const cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)kWChunk};
    const cuuint32_t box[3] = {(cuuint32_t)kWChunk, (cuuint32_t)kWRows, (cuuint32_t)(kWStepK / kWChunk)};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    CUtensorMap m;
    const CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    keys[next] = Key{ptr, rows, K};
    maps[next] = m;
    next = (next + 1) % 64;
    if (used < 64) ++used;
    *out = m;
    return cudaSuccess;
}

int sm_count_w() {
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return c;
}

}  // namespace

WidePlan plan_wide(int M, int N, int K, int G, int S, bool partials) {
    WidePlan pl{};
    pl.S = S;
    pl.chunk_cols = S >= 1 ? ((K / 32 + S - 1) / S) * 32 : 0;
    const int chunk_pad = (pl.chunk_cols + kWStepK - 1) / kWStepK * kWStepK;
    pl.pitch = 2 * chunk_pad + 64;  // 16-byte pieces of x land on distinct banks across rows
    const size_t xbytes = (size_t)std::max(1, std::min(M, kWWarps)) * pl.pitch;
    const size_t room = kWSmemMax - 1024 - std::min(xbytes, kWSmemMax - 1024);
    pl.depth = (int)std::min<size_t>(kWDepthMax, room / kWBox);
    pl.smem = 1024 + (size_t)pl.depth * kWBox + xbytes;
    const long long tasks = (long long)S * G * (N / kWRows);
    pl.tasks = tasks < (1LL << 30) ? (int)tasks : 0;
    pl.partials = partials || S > 1;
    // every split starts on a 128-column chunk of the 3-D view
    pl.ok = M >= 1 && M <= 8 && S >= 1 && K % kWChunk == 0 && pl.chunk_cols % kWChunk == 0 &&
            pl.chunk_cols <= kWMaxChunk && (long long)G * N < (1LL << 31) && pl.tasks > 0 &&
            pl.depth >= kWDepthMin && pl.smem <= kWSmemMax;
    return pl;
}

cudaError_t launch_wide(const WidePlan &pl, const void *x, long long ldx, const uint8_t *w8, const uint8_t *ex,
                        void *y, float *partials, int M, int N, int K, int G, cudaStream_t stream) {
    if (!pl.ok) return cudaErrorInvalidValue;
    if (pl.partials ? partials == nullptr : y == nullptr) return cudaErrorInvalidValue;
    const Options opt = options();
    WideParams prm;
    cudaError_t e = codes_map_w(w8, (long long)G * N, K, &prm.cmap);
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
    prm.tasks = pl.tasks;
    prm.pitch = pl.pitch;
    prm.depth = pl.depth;
    prm.to_partials = pl.partials ? 1 : 0;
    prm.timeout_ns = opt.timeout_ns;
    prm.skip_loads = opt.skip_loads;
    prm.status = status_word();
    if (!prm.status) return cudaErrorInvalidSymbol;
    static int configured[64] = {0};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmemMax);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(wide_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    const int sms = sm_count_w();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(pl.tasks, sms), 1, 1);
    cfg.blockDim = dim3(kWThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
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
    return cudaLaunchKernelEx(&cfg, wide_kernel, prm);
}

}  // namespace bsf8
