// bsf8_internal.h -- host-side interface between the C ABI (bsf8_abi.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bsf8 {

// Process-wide launch options (see BSF8_OPT_* in bsf8.h).
struct Options {
    int pdl;
    unsigned long long timeout_ns;
    int skip_loads;
    int gemm_path;  // 0: by shape; 2: streaming; 4: decode-ahead; 5: tensor-core;
                    // 6: wide-weight; 7: decode-ahead tensor-core
};
Options options();

// Device address of the library's status word on the current device (looked up once
// per device); nullptr if the lookup fails.
int *status_word();

// Largest cluster the streaming and decode-ahead kernels form to sum a slab's splits
// (the portable cluster size).
constexpr int kMaxClusterSplits = 8;

// Weight-streaming kernel (bsf8_stream.cu): warp tasks of 16 rows x a column range.
enum StreamMode { kStreamInCta = 0, kStreamCluster = 1, kStreamPartials = 2, kStreamGroup = 3 };

struct StreamPlan {
    int S, chunk_cols, kt, tps;  // splits, columns per split, per task, tasks per split
    int nt8, m_chunks;           // token tiles of 8 per pass, passes over the tokens
    int mode, spc, cluster, spl, cps, grid_x;
    int tpc;  // group mode (decode-ahead kernel): tasks of each slab a block holds
    int to_partials;  // group mode (decode-ahead kernel): the fold writes each split's fp32
                      // partial (tasks summed in order) instead of summing the splits into y
};

StreamPlan plan_stream(int M, int N, int K, int G, int S, bool partials);
// The same decomposition with an explicit step width, at most max_nt8 token tiles and
// tasks of at most max_kt columns.
StreamPlan plan_stream_ks(int M, int N, int K, int G, int S, bool partials, int ks, int max_nt8,
                          int max_kt = 1 << 30);

// Decode-ahead kernel (bsf8_lowm.cu) for up to 8 token rows; 128-column steps, tasks of
// at most 512 columns.  The plan's decomposition does not depend on `partials` (a call for
// the partials differs only in what the fold stores), so y and the partials summed by the
// fixed-order reduce agree bit for bit.  lowm_fits: the kernel can run the plan.
StreamPlan plan_lowm(int M, int N, int K, int G, int S, bool partials);
bool lowm_fits(const StreamPlan &plan);
cudaError_t launch_lowm(const StreamPlan &plan, const void *x, long long ldx, const uint8_t *w8,
                        const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                        cudaStream_t stream, bool rows_exp = false);

// Streaming kernel (bsf8_stream.cu).
// rows_exp: exponents per (weight row, 32 columns), [G][N][K/32], instead of per 32 x 32 block
cudaError_t launch_stream(const StreamPlan &plan, const void *x, long long ldx, const uint8_t *w8,
                          const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                          cudaStream_t stream, bool rows_exp = false);

// Tensor-core kernel (bsf8_umma.cu): 128-row blocks, one split and one token tile (up to 192
// rows) a block.  With more than one split the split blocks of a row block sum in a cluster
// (2..8 splits whose blocks fit one wave), else it writes fp32 partials (the fixed-order
// reduce follows).
struct UmmaPlan {
    int S, chunk_cols, ntok, row_blocks, grid_x, ttiles;  // ttiles: token tiles of ntok rows
    int run_shift;  // log2 of the steps a tensor-memory accumulator takes (2, or 3: see bsf8_umma.cu)
    bool fold;      // 2..8 splits summed inside a cluster of the split blocks (no partials)
    int sps;        // 128-column steps a ring stage holds (1 or 2)
    bool partials, tmem_ok, ok;  // ok: the kernel can run this call (else another kernel)
};
UmmaPlan plan_umma(int M, int N, int K, int G, int S, bool partials);
int umma_auto_split(int M, int N, int K, int G, int sms);
cudaError_t launch_umma(const UmmaPlan &plan, const void *x, long long ldx, const uint8_t *w8,
                        const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                        cudaStream_t stream);

// Wide-weight kernel (bsf8_wide.cu) for up to 8 token rows: tasks of 128 rows x one
// split, one block an SM; codes widened to f16, x converted once a split into shared memory.
// With more than one split it writes fp32 partials (the fixed-order reduce follows).
struct WidePlan {
    int S, chunk_cols, tasks, pitch, depth;
    size_t smem;
    bool partials, ok;  // ok: the kernel can run this call (else another kernel)
};
WidePlan plan_wide(int M, int N, int K, int G, int S, bool partials);
cudaError_t launch_wide(const WidePlan &plan, const void *x, long long ldx, const uint8_t *w8,
                        const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                        cudaStream_t stream);

// Decode-ahead tensor-core kernel (bsf8_ahead.cu) for up to 32 token rows: blocks of 128
// rows x one task (<= 512 columns of a split), a cluster per 128 rows holding all of their
// tasks (at most 16), the rebuilt weights in tensor memory before the dependency wait.
struct AheadPlan {
    int S, chunk_cols, kt, tps, ntok, nacc, cluster, rows_per_rank, grid_x;
    bool partials, ok;  // ok: the kernel can run this call (else another kernel)
};
AheadPlan plan_ahead(int M, int N, int K, int G, int S, bool partials);
cudaError_t launch_ahead(const AheadPlan &plan, const void *x, long long ldx, const uint8_t *w8,
                         const uint8_t *ex, void *y, float *partials, int M, int N, int K, int G,
                         cudaStream_t stream, bool rows_exp = false);

// The streaming kernel's split count for split_k = 0 (bsf8_reduce.cu; sizes only).
int auto_split(int M, int N, int K, int G);

// Launchers return a cudaError_t.
cudaError_t launch_splitk_reduce(const float *P, void *y, int S, long long count,
                                 cudaStream_t stream);
cudaError_t launch_splitk_reduce_f32(const float *P, float *y, int S, long long count, cudaStream_t stream);
cudaError_t launch_dequant(const uint8_t *w8, const uint8_t *ex, void *out, int G, int N, int K,
                           cudaStream_t stream);
cudaError_t launch_make_twin(const void *w, uint8_t *w8, uint8_t *ex, uint8_t *ok,
                             int32_t *accepted, int G, int N, int K, cudaStream_t stream);
// The per-(row, 32-column) scale layout: exponents and flags [G][N][K/32].
cudaError_t launch_make_twin_rows(const void *w, uint8_t *w8, uint8_t *ex, uint8_t *ok, int32_t *accepted,
                                  int G, int N, int K, cudaStream_t stream);
cudaError_t launch_dequant_rows(const uint8_t *w8, const uint8_t *ex, void *out, int G, int N, int K,
                                cudaStream_t stream);
cudaError_t launch_pad_k(const uint8_t *w8, const uint8_t *ex, uint8_t *w8_out, uint8_t *ex_out,
                         int G, int N, int K, int Kp, int pad_exp, cudaStream_t stream);
cudaError_t launch_pad_x(const void *x, long long ldx, void *x_out, int M, int G, int K, int Kp,
                         cudaStream_t stream);

}  // namespace bsf8
