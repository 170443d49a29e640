// bsf8_abi.cu -- the extern "C" entry points of libbsf8 (declared in include/bsf8.h).
//
// Every entry point validates its arguments on the host before touching CUDA, so a bad
// call returns a status code without a GPU being involved; then it enqueues kernels on
// the caller's stream and returns.  Nothing here allocates memory.
#include "bsf8.h"
#include "bsf8_device.cuh"
#include "bsf8_internal.h"

#include <atomic>
#include <cstdint>

namespace bsf8 {

__device__ int g_status = 0;

namespace {
std::atomic<int> g_opt_pdl{1};
std::atomic<long long> g_opt_timeout_ns{2000000000LL};
std::atomic<int> g_opt_skip_loads{0};
std::atomic<int> g_opt_gemm_path{0};
}  // namespace

int *status_word() {
    static int *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    int *a = __atomic_load_n(&addr[dev], __ATOMIC_ACQUIRE);
    if (!a) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        a = static_cast<int *>(p);
        __atomic_store_n(&addr[dev], a, __ATOMIC_RELEASE);
    }
    return a;
}

Options options() {
    Options o;
    o.pdl = g_opt_pdl.load(std::memory_order_relaxed);
    o.timeout_ns = (unsigned long long)g_opt_timeout_ns.load(std::memory_order_relaxed);
    o.skip_loads = g_opt_skip_loads.load(std::memory_order_relaxed);
    o.gemm_path = g_opt_gemm_path.load(std::memory_order_relaxed);
    return o;
}

}  // namespace bsf8

using namespace bsf8;

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<int> g_last_cuda_error{0};

inline int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return BSF8_OK;
    g_last_cuda_error.store((int)e, std::memory_order_relaxed);
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction ||
        e == cudaErrorUnsupportedPtxVersion)
        return BSF8_ERR_DEVICE;
    return BSF8_ERR_CUDA;
}

// Common shape rules: sizes >= 1, N and K multiples of 32, element counts that fit.
inline int check_gnk(int G, int N, int K) {
    if (G < 1 || N < 32 || K < 32 || (N % 32) != 0 || (K % 32) != 0) return BSF8_ERR_SHAPE;
    if ((long long)G * N * (long long)K > (1LL << 46)) return BSF8_ERR_SHAPE;
    return BSF8_OK;
}

inline int check_gemm_args(const void *x, const uint8_t *w8, const uint8_t *exp, const void *out,
                           int M, int N, int K, int G, int split_k, int64_t ldx) {
    if (!x || !w8 || !exp || !out) return BSF8_ERR_NULL;
    int st = check_gnk(G, N, K);
    if (st) return st;
    if (M < 1 || M > BSF8_MAX_M) return BSF8_ERR_SHAPE;
    if (split_k < 0 || split_k > K / 32) return BSF8_ERR_SHAPE;
    if (ldx < (int64_t)G * K) return BSF8_ERR_STRIDE;
    if (!aligned16(x) || (ldx % 8) != 0 || !aligned16(w8)) return BSF8_ERR_ALIGN;
    return BSF8_OK;
}

// Kernel for a call.  The decode-ahead kernel pays off when each of its blocks holds one
// group of tasks, so that the group's weights are rebuilt before the dependency wait: up to
// 8 token rows and at most two blocks an SM.  Larger calls stream (the cp.async kernel
// sustains more bandwidth once the rebuild can no longer run ahead).  TMA coordinates are
// 32-bit, so the TMA kernels need G*N < 2^31.  The values are those of BSF8_OPT_GEMM_PATH
// and of bsf8_gemm_kernel.
enum MainKernel {
    kKernelNone = -1, kKernelStream = 2, kKernelLowM = 4, kKernelUmma = 5, kKernelWide = 6, kKernelAhead = 7
};

// Above this many token rows the tensor-core kernel (tcgen05) runs where the decode-ahead
// tensor-core kernel does not: its MMAs are cheap there, while the mma.sync kernels become
// bound by their MMA issue.  Measured on a GB300, mid rows (G = 4, 1024 x 4096): M = 20 / 24
// 10.7 us against 15.6 streaming, M = 64 12 against 35, M = 192 14.5 against 91; at M = 9 /
// 16 the streaming kernel is ahead (8.3 / 8.6 us against 11.7 / 10.6); the head-like weight
// (32768 x 5120) at M = 20 / 24: 64 against 120 us.
constexpr int kUmmaMinRows = 16;

// Token rows the decode-ahead tensor-core kernel (bsf8_ahead.cu) serves by default from 9 up.
constexpr int kAheadMaxRows = 32;

inline int sm_count() {
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = __atomic_load_n(&count[dev], __ATOMIC_ACQUIRE);
    if (c == 0 && cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        __atomic_store_n(&count[dev], c, __ATOMIC_RELEASE);
    return c;
}

// 9..32 rows whose one-split plan on the decode-ahead tensor-core kernel fits one block an
// SM: that kernel cuts the split into tasks anyway, so more splits would only add partials.
inline bool ahead_one_split(int M, int N, int K, int G) {
    if (M <= 8 || M > kAheadMaxRows) return false;
    const AheadPlan ap = plan_ahead(M, N, K, G, 1, false);
    return ap.ok && (long long)ap.grid_x * G <= sm_count();
}

// The split count when the caller leaves it to the library (split_k = 0).  Up to 8 token
// rows: 1 -- the decode-ahead and streaming kernels cut a split into tasks of at most 512
// (decode-ahead) or ~K/8 columns anyway, and more splits only add partial sums (measured:
// down_proj 4.0 us at one split against 5.4 at four); likewise 1 for 9..32 rows where the
// decode-ahead tensor-core kernel takes the call in one split.
inline int call_auto_split(int M, int N, int K, int G) {
    if (M <= 8) return 1;
    if (ahead_one_split(M, N, K, G)) return 1;
    // 9..16 rows elsewhere: the streaming kernel (or, on wide weights, the tensor-core kernel
    // at one split); the streaming kernel cuts a split into tasks, and extra splits measured
    // no faster (mid G = 4, 1024 x 4096, M = 16: 8.7 us at 1, 2, 4 and 8 splits, 19 us at
    // the five a blocks-per-SM target gave)
    if (M <= kUmmaMinRows) return 1;
    if (M > kUmmaMinRows && (long long)G * N < (1LL << 31)) {
        const int sms = sm_count();
        if (sms > 0) {
            const int S = umma_auto_split(M, N, K, G, sms);
            if (plan_umma(M, N, K, G, S, false).ok) return S;
        }
    }
    return auto_split(M, N, K, G);
}

// The kernel a call of these sizes runs.  It depends on the sizes, the split count and the
// options only -- not on whether the caller wants y or the fp32 partials -- so that
// bsf8_gemm and bsf8_gemm_partials + bsf8_splitk_reduce run the same kernel and give the
// same bits.  A kernel forced through BSF8_OPT_GEMM_PATH that cannot run the call gives
// kKernelNone (the entry points then return BSF8_ERR_VALUE).
inline MainKernel main_kernel(int M, int N, int K, int G, int S) {
    const bool tma_ok = (long long)G * N < (1LL << 31);
    switch (options().gemm_path) {  // a forced kernel
        case 2: return kKernelStream;
        case 4: return M <= 8 && tma_ok && lowm_fits(plan_lowm(M, N, K, G, S, false)) ? kKernelLowM : kKernelNone;
        case 5: return tma_ok && plan_umma(M, N, K, G, S, false).ok ? kKernelUmma : kKernelNone;
        case 6: return tma_ok && plan_wide(M, N, K, G, S, false).ok ? kKernelWide : kKernelNone;
        case 7: return tma_ok && plan_ahead(M, N, K, G, S, false).ok ? kKernelAhead : kKernelNone;
        default: break;
    }
    if (!tma_ok) return kKernelStream;
    if (M > 8 && M <= kAheadMaxRows) {
        // 9..32 rows where every 128-row block of the decode-ahead tensor-core plan holds
        // one block an SM (its cluster of <= 16 tasks a row block): wo_a (G = 2, 1024 x 4096)
        // at M = 16 takes 5.9 us against 7.5 us streaming, at M = 32 8.9 against 9.5 us for
        // the tensor-core kernel; gate_up (1152 x 5120) at M = 16 5.1 against 8.4.
        const AheadPlan ap = plan_ahead(M, N, K, G, S, false);
        if (ap.ok && (long long)ap.grid_x * G <= sm_count()) return kKernelAhead;
    }
    if (M > kUmmaMinRows) return plan_umma(M, N, K, G, S, false).ok ? kKernelUmma : kKernelStream;
    if (M > 8) {
        // 9..16 rows over an unsplit wide weight (a block of 128 rows for every SM, e.g. an
        // output head): the tensor-core kernel, two blocks an SM, measured 57 us against
        // 65 us for the streaming kernel at N = 32768, K = 5120.  Narrower weights stream.
        if (M <= 16 && S == 1 && (long long)G * ((N + 127) / 128) >= sm_count() &&
            plan_umma(M, N, K, G, S, false).ok)
            return kKernelUmma;
        return kKernelStream;
    }
    const StreamPlan pl = plan_lowm(M, N, K, G, S, false);
    if (lowm_fits(pl) && (long long)pl.grid_x * G <= 2LL * sm_count()) return kKernelLowM;
    // more weight than the decode-ahead grid holds: the wide-weight kernel streams it
    // (one split: more would add the reduce pass the streaming kernel does without)
    return S == 1 && plan_wide(M, N, K, G, S, false).ok ? kKernelWide : kKernelStream;
}

// How one call runs: the kernel, its plan, and whether it writes fp32 partials (then the
// fixed-order reduce follows, or the caller asked for the partials).
struct Call {
    MainKernel kernel;
    StreamPlan sp;
    UmmaPlan up;
    WidePlan wp;
    AheadPlan ap;
    bool partials_out;
};

inline Call plan_call(int M, int N, int K, int G, int S, bool partials) {
    Call c{};
    c.kernel = main_kernel(M, N, K, G, S);
    switch (c.kernel) {
        case kKernelNone: return c;
        case kKernelUmma:
            c.up = plan_umma(M, N, K, G, S, partials);
            c.partials_out = c.up.partials;
            return c;
        case kKernelWide:
            c.wp = plan_wide(M, N, K, G, S, partials);
            c.partials_out = c.wp.partials;
            return c;
        case kKernelAhead:
            c.ap = plan_ahead(M, N, K, G, S, partials);
            c.partials_out = c.ap.partials;
            return c;
        case kKernelLowM: c.sp = plan_lowm(M, N, K, G, S, partials); break;
        default: c.sp = plan_stream(M, N, K, G, S, partials); break;
    }
    c.partials_out = c.sp.mode == kStreamPartials || c.sp.to_partials;
    return c;
}

inline cudaError_t launch_call(const Call &c, const void *x, long long ldx, const uint8_t *w8,
                               const uint8_t *ex, void *y, float *P, int M, int N, int K, int G,
                               cudaStream_t s) {
    // the output the plan writes must be there (fp32 partials, or y)
    if (c.partials_out ? P == nullptr : y == nullptr) return cudaErrorInvalidValue;
    switch (c.kernel) {
        case kKernelUmma: return launch_umma(c.up, x, ldx, w8, ex, y, P, M, N, K, G, s);
        case kKernelWide: return launch_wide(c.wp, x, ldx, w8, ex, y, P, M, N, K, G, s);
        case kKernelAhead: return launch_ahead(c.ap, x, ldx, w8, ex, y, P, M, N, K, G, s);
        case kKernelLowM: return launch_lowm(c.sp, x, ldx, w8, ex, y, P, M, N, K, G, s);
        case kKernelStream: return launch_stream(c.sp, x, ldx, w8, ex, y, P, M, N, K, G, s);
        default: return cudaErrorInvalidValue;
    }
}

// The per-row-scale GEMM runs where the block layout's calls of the same shape do: on the
// decode-ahead kernel (M <= 8, its grid within two blocks an SM), on the decode-ahead
// tensor-core kernel (9..32 rows, its grid within one block an SM; with
// BSF8_OPT_GEMM_PATH 7 wherever its plan holds), else on the streaming kernel.
struct RowsCall {
    bool lowm, ahead;
    StreamPlan sp;
    AheadPlan ap;
};

inline RowsCall plan_rows(int M, int N, int K, int G, int S) {
    RowsCall c{};
    if (options().gemm_path == 7 || (M > 8 && M <= kAheadMaxRows)) {
        c.ap = plan_ahead(M, N, K, G, S, false);
        c.ahead = c.ap.ok && (options().gemm_path == 7 || (long long)c.ap.grid_x * G <= sm_count());
        if (c.ahead) return c;
    }
    if (M <= 8) {
        c.sp = plan_lowm(M, N, K, G, S, false);
        c.lowm = lowm_fits(c.sp) && (long long)c.sp.grid_x * G <= 2LL * sm_count();
        if (c.lowm) return c;
    }
    c.sp = plan_stream(M, N, K, G, S, false);
    return c;
}

}  // namespace

extern "C" {

const char *bsf8_strerror(int status) {
    switch (status) {
        case BSF8_OK: return "ok";
        case BSF8_ERR_SHAPE: return "invalid shape (sizes < 1, N or K not a multiple of 32, M or split_k out of range)";
        case BSF8_ERR_ALIGN: return "misaligned pointer or stride (16-byte rule)";
        case BSF8_ERR_STRIDE: return "row stride ldx smaller than G*K";
        case BSF8_ERR_WORKSPACE: return "workspace missing or too small";
        case BSF8_ERR_NULL: return "required pointer is NULL";
        case BSF8_ERR_CUDA: return "CUDA runtime error";
        case BSF8_ERR_TIMEOUT: return "a kernel gave up a bounded wait (outputs undefined)";
        case BSF8_ERR_DEVICE: return "device cannot run the sm_103a kernels";
        case BSF8_ERR_VALUE: return "option or scalar argument out of range";
        default: return "unknown status";
    }
}

int bsf8_version(void) { return 100; }

int bsf8_last_cuda_error(void) { return g_last_cuda_error.load(std::memory_order_relaxed); }

int bsf8_make_twin(const void *w, uint8_t *w8, uint8_t *exp, uint8_t *block_ok, int32_t *accepted,
                   int G, int N, int K, bsf8_stream_t stream) {
    if (!w || !w8 || !exp || !accepted) return BSF8_ERR_NULL;
    int st = check_gnk(G, N, K);
    if (st) return st;
    if (!aligned16(w) || !aligned16(w8)) return BSF8_ERR_ALIGN;
    return from_cuda(launch_make_twin(w, w8, exp, block_ok, accepted, G, N, K,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int bsf8_dequant(const uint8_t *w8, const uint8_t *exp, void *out, int G, int N, int K,
                 bsf8_stream_t stream) {
    if (!w8 || !exp || !out) return BSF8_ERR_NULL;
    int st = check_gnk(G, N, K);
    if (st) return st;
    if (!aligned16(w8) || !aligned16(out)) return BSF8_ERR_ALIGN;
    return from_cuda(launch_dequant(w8, exp, out, G, N, K, reinterpret_cast<cudaStream_t>(stream)));
}

int bsf8_gemm_auto_split(int M, int N, int K, int G) {
    int st = check_gnk(G, N, K);
    if (st) return -st;
    if (M < 1 || M > BSF8_MAX_M) return -BSF8_ERR_SHAPE;
    return call_auto_split(M, N, K, G);
}

size_t bsf8_gemm_workspace_bytes(int M, int N, int K, int G, int split_k) {
    if (check_gnk(G, N, K) || M < 1 || M > BSF8_MAX_M || split_k < 0 || split_k > K / 32) return 0;
    const int S = split_k == 0 ? call_auto_split(M, N, K, G) : split_k;
    const Call c = plan_call(M, N, K, G, S, false);
    if (c.kernel == kKernelNone || !c.partials_out) return 0;
    return (size_t)S * M * G * N * sizeof(float);
}

int bsf8_gemm(const void *x, const uint8_t *w8, const uint8_t *exp, void *y, int M, int N, int K,
              int G, int split_k, int64_t ldx, void *workspace, size_t workspace_bytes,
              bsf8_stream_t stream) {
    int st = check_gemm_args(x, w8, exp, y, M, N, K, G, split_k, ldx);
    if (st) return st;
    const int S = split_k == 0 ? call_auto_split(M, N, K, G) : split_k;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Call c = plan_call(M, N, K, G, S, false);
    if (c.kernel == kKernelNone) return BSF8_ERR_VALUE;
    if (!c.partials_out) return from_cuda(launch_call(c, x, ldx, w8, exp, y, nullptr, M, N, K, G, s));
    const size_t need = (size_t)S * M * G * N * sizeof(float);
    if (!workspace || workspace_bytes < need) return BSF8_ERR_WORKSPACE;
    if (!aligned16(workspace)) return BSF8_ERR_ALIGN;
    float *P = static_cast<float *>(workspace);
    st = from_cuda(launch_call(c, x, ldx, w8, exp, nullptr, P, M, N, K, G, s));
    if (st) return st;
    return from_cuda(launch_splitk_reduce(P, y, S, (long long)M * G * N, s));
}

int bsf8_gemm_kernel(int M, int N, int K, int G, int split_k) {
    int st = check_gnk(G, N, K);
    if (st) return -st;
    if (M < 1 || M > BSF8_MAX_M || split_k < 0 || split_k > K / 32) return -BSF8_ERR_SHAPE;
    const int S = split_k == 0 ? call_auto_split(M, N, K, G) : split_k;
    const MainKernel k = main_kernel(M, N, K, G, S);
    return k == kKernelNone ? -BSF8_ERR_VALUE : (int)k;
}

int bsf8_make_twin_rows(const void *w, uint8_t *w8, uint8_t *exp, uint8_t *block_ok, int32_t *accepted,
                        int G, int N, int K, bsf8_stream_t stream) {
    if (!w || !w8 || !exp || !accepted) return BSF8_ERR_NULL;
    int st = check_gnk(G, N, K);
    if (st) return st;
    if (!aligned16(w) || !aligned16(w8)) return BSF8_ERR_ALIGN;
    return from_cuda(launch_make_twin_rows(w, w8, exp, block_ok, accepted, G, N, K,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int bsf8_dequant_rows(const uint8_t *w8, const uint8_t *exp, void *out, int G, int N, int K,
                      bsf8_stream_t stream) {
    if (!w8 || !exp || !out) return BSF8_ERR_NULL;
    int st = check_gnk(G, N, K);
    if (st) return st;
    if (!aligned16(w8) || !aligned16(out)) return BSF8_ERR_ALIGN;
    return from_cuda(launch_dequant_rows(w8, exp, out, G, N, K, reinterpret_cast<cudaStream_t>(stream)));
}

size_t bsf8_gemm_rows_workspace_bytes(int M, int N, int K, int G, int split_k) {
    if (check_gnk(G, N, K) || M < 1 || M > BSF8_MAX_M || split_k < 0 || split_k > K / 32) return 0;
    const int S = split_k == 0 ? (M <= 8 || ahead_one_split(M, N, K, G) ? 1 : auto_split(M, N, K, G)) : split_k;
    const RowsCall c = plan_rows(M, N, K, G, S);
    if (c.ahead || c.sp.mode != kStreamPartials) return 0;
    return (size_t)S * M * G * N * sizeof(float);
}

int bsf8_gemm_rows(const void *x, const uint8_t *w8, const uint8_t *exp, void *y, int M, int N, int K, int G,
                   int split_k, int64_t ldx, void *workspace, size_t workspace_bytes, bsf8_stream_t stream) {
    int st = check_gemm_args(x, w8, exp, y, M, N, K, G, split_k, ldx);
    if (st) return st;
    const int S = split_k == 0 ? (M <= 8 || ahead_one_split(M, N, K, G) ? 1 : auto_split(M, N, K, G)) : split_k;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const RowsCall c = plan_rows(M, N, K, G, S);
    if (c.ahead) return from_cuda(launch_ahead(c.ap, x, ldx, w8, exp, y, nullptr, M, N, K, G, s, true));
    auto launch = [&](void *yy, float *P) {
        return c.lowm ? launch_lowm(c.sp, x, ldx, w8, exp, yy, P, M, N, K, G, s, true)
                      : launch_stream(c.sp, x, ldx, w8, exp, yy, P, M, N, K, G, s, true);
    };
    if (c.sp.mode != kStreamPartials) return from_cuda(launch(y, nullptr));
    const size_t need = (size_t)S * M * G * N * sizeof(float);
    if (!workspace || workspace_bytes < need) return BSF8_ERR_WORKSPACE;
    if (!aligned16(workspace)) return BSF8_ERR_ALIGN;
    float *P = static_cast<float *>(workspace);
    st = from_cuda(launch(nullptr, P));
    if (st) return st;
    return from_cuda(launch_splitk_reduce(P, y, S, (long long)M * G * N, s));
}

int bsf8_gemm_partials(const void *x, const uint8_t *w8, const uint8_t *exp, float *partials,
                       int M, int N, int K, int G, int split_k, int64_t ldx,
                       bsf8_stream_t stream) {
    int st = check_gemm_args(x, w8, exp, partials, M, N, K, G, split_k, ldx);
    if (st) return st;
    if (split_k < 1) return BSF8_ERR_SHAPE;
    if (!aligned16(partials)) return BSF8_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Call c = plan_call(M, N, K, G, split_k, true);
    if (c.kernel == kKernelNone) return BSF8_ERR_VALUE;
    return from_cuda(launch_call(c, x, ldx, w8, exp, nullptr, partials, M, N, K, G, s));
}

int bsf8_splitk_reduce(const float *partials, void *y, int S, int64_t count, bsf8_stream_t stream) {
    if (S < 1 || count < 0) return BSF8_ERR_SHAPE;
    if (count == 0) return BSF8_OK;
    if (!partials || !y) return BSF8_ERR_NULL;
    return from_cuda(launch_splitk_reduce(partials, y, S, (long long)count,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int bsf8_splitk_reduce_f32(const float *partials, float *y, int S, int64_t count, bsf8_stream_t stream) {
    if (S < 1 || count < 0) return BSF8_ERR_SHAPE;
    if (count == 0) return BSF8_OK;
    if (!partials || !y) return BSF8_ERR_NULL;
    return from_cuda(launch_splitk_reduce_f32(partials, y, S, (long long)count,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int bsf8_pad_k(const uint8_t *w8, const uint8_t *exp, uint8_t *w8_out, uint8_t *exp_out, int G,
               int N, int K, int Kp, int pad_exp, bsf8_stream_t stream) {
    if (!w8 || !exp || !w8_out || !exp_out) return BSF8_ERR_NULL;
    int st = check_gnk(G, N, K);
    if (st) return st;
    if (Kp < K || (Kp % 32) != 0 || check_gnk(G, N, Kp)) return BSF8_ERR_SHAPE;
    if (pad_exp < 0 || pad_exp > 255) return BSF8_ERR_VALUE;
    if (!aligned16(w8) || !aligned16(w8_out)) return BSF8_ERR_ALIGN;
    return from_cuda(launch_pad_k(w8, exp, w8_out, exp_out, G, N, K, Kp, pad_exp,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

int bsf8_pad_x(const void *x, int64_t ldx, void *x_out, int M, int G, int K, int Kp,
               bsf8_stream_t stream) {
    if (!x || !x_out) return BSF8_ERR_NULL;
    if (M < 1 || G < 1 || K < 32 || (K % 32) != 0 || Kp < K || (Kp % 32) != 0) return BSF8_ERR_SHAPE;
    if ((long long)M * G * (long long)Kp > (1LL << 46)) return BSF8_ERR_SHAPE;
    if (ldx < (int64_t)G * K) return BSF8_ERR_STRIDE;
    if (!aligned16(x) || (ldx % 8) != 0 || !aligned16(x_out)) return BSF8_ERR_ALIGN;
    return from_cuda(launch_pad_x(x, (long long)ldx, x_out, M, G, K, Kp,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

int bsf8_device_status(int *status, bsf8_stream_t stream) {
    if (!status) return BSF8_ERR_NULL;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (e != cudaSuccess) return from_cuda(e);
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof zero);
    if (e != cudaSuccess) return from_cuda(e);
    *status = v;
    return BSF8_OK;
}

int bsf8_set_option(int option, int64_t value) {
    if (value < 0) return BSF8_ERR_VALUE;
    switch (option) {
        case BSF8_OPT_PDL: g_opt_pdl.store(value ? 1 : 0); return BSF8_OK;
        case BSF8_OPT_WAIT_TIMEOUT_NS: g_opt_timeout_ns.store((long long)value); return BSF8_OK;
        case BSF8_OPT_DEBUG_SKIP_LOADS: g_opt_skip_loads.store(value ? 1 : 0); return BSF8_OK;
        case BSF8_OPT_GEMM_PATH:
            if (value > 7 || value == 1 || value == 3) return BSF8_ERR_VALUE;
            g_opt_gemm_path.store((int)value);
            return BSF8_OK;
        default: return BSF8_ERR_VALUE;
    }
}

int64_t bsf8_get_option(int option) {
    switch (option) {
        case BSF8_OPT_PDL: return g_opt_pdl.load();
        case BSF8_OPT_WAIT_TIMEOUT_NS: return g_opt_timeout_ns.load();
        case BSF8_OPT_DEBUG_SKIP_LOADS: return g_opt_skip_loads.load();
        case BSF8_OPT_GEMM_PATH: return g_opt_gemm_path.load();
        default: return -BSF8_ERR_VALUE;
    }
}

}  // extern "C"
