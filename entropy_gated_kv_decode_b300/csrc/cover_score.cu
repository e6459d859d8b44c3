// COVER's stability-aware seed score ("Stop the Flip-Flop" (COVER), Italian
// technical summary, "Metodologia: COVER", item 2): five kernels over the
// per-item functions of cover_score.cuh, chained by programmatic dependent
// launch, and the C entry points of include/ec_cover.h.
//
// The work is a second pass of q . k over every key for the still-masked and
// candidate rows (the normalisers of their attention rows), then small sums.
// It is plain float32 SIMT arithmetic: a warp's 32 threads are 32 (row, head)
// pairs of one key-value head and walk the same key rows, so every key row is
// read once per warp and broadcast; no step waits on another CTA.
#include <math.h>

#include "cover_score.cuh"
#include "ec_cover.h"
#include "ec_internal.cuh"

namespace ec {
namespace {

constexpr int kThreads = 256;

template <int D>
__global__ void __launch_bounds__(kThreads) cover_partial_kernel(cover::Args A, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();  // inputs belong to the previous kernel until here
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < n) cover::partial_item<D>(A, t);
}

__global__ void __launch_bounds__(kThreads) cover_stats_kernel(cover::Args A, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < n) cover::stats_item(A, t);
}

template <int D>
__global__ void __launch_bounds__(kThreads) cover_din_kernel(cover::Args A, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < n) cover::din_item<D>(A, t);
}

__global__ void __launch_bounds__(kThreads) cover_final_kernel(cover::Args A, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < n) cover::final_item(A, t);
}

__global__ void __launch_bounds__(kThreads) cover_rank_kernel(cover::Args A, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < n) cover::rank_item(A, t);
}

inline dim3 grid_for(int64_t n) { return dim3(static_cast<unsigned>((n + kThreads - 1) / kThreads)); }

template <int D>
cudaError_t launch_all(const cover::Args &A, cudaStream_t stream)
{
    cudaError_t e = cudaSuccess;
    const int64_t n1 = cover::partial_items(A), n2 = cover::head_items(A), n4 = cover::final_items(A),
                  n5 = cover::rank_items(A);
    if (n1 > 0) e = launch(cover_partial_kernel<D>, grid_for(n1), dim3(kThreads), 0, stream, A, n1);
    if (e == cudaSuccess && n2 > 0)
        e = launch(cover_stats_kernel, grid_for(n2), dim3(kThreads), 0, stream, A, n2);
    if (e == cudaSuccess && n2 > 0)
        e = launch(cover_din_kernel<D>, grid_for(n2), dim3(kThreads), 0, stream, A, n2);
    if (e == cudaSuccess && n4 > 0)
        e = launch(cover_final_kernel, grid_for(n4), dim3(kThreads), 0, stream, A, n4);
    if (e == cudaSuccess && n5 > 0 && A.n_seed > 0)
        e = launch(cover_rank_kernel, grid_for(n5), dim3(kThreads), 0, stream, A, n5);
    return e;
}

struct Layout {
    size_t part, stat_m, stat_z, dout_h, din_h, total;
};

Layout layout(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads)
{
    int32_t n_chunks = 1, chunk_len = 1;
    cover::plan(batch, seq_len, r_max, n_heads, &n_chunks, &chunk_len);
    const size_t rows = static_cast<size_t>(batch) * r_max * n_heads;
    Layout w;
    w.part = kWsHeader;
    w.stat_m = align_up(w.part + rows * n_chunks * sizeof(cover::Part), 256);
    w.stat_z = align_up(w.stat_m + rows * sizeof(float), 256);
    w.dout_h = align_up(w.stat_z + rows * sizeof(float), 256);
    w.din_h = align_up(w.dout_h + rows * sizeof(float), 256);
    w.total = align_up(w.din_h + rows * sizeof(float), 256);
    return w;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace ec

extern "C" {

size_t ec_cover_score_workspace_size(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads)
{
    if (batch < 1 || seq_len < 1 || r_max < 0 || n_heads < 1) return ec::kWsHeader;
    return ec::layout(batch, seq_len, r_max, n_heads).total;
}

ec_status ec_cover_seed_score(const void *q, const void *k_cache, const int32_t *idx,
                              int64_t idx_stride, const int32_t *count, const uint8_t *role,
                              const uint8_t *drafted, const float *u, ec_dtype dtype, int32_t batch,
                              int32_t seq_len, int32_t r_max, int32_t n_heads, int32_t n_kv_heads,
                              int32_t head_dim, float scale, int32_t n_seed, float *d_in,
                              float *d_out, float *score, int32_t *seeds, void *workspace,
                              size_t workspace_bytes, ec_stream_t stream)
{
    if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_DTYPE;
    if (batch < 1 || seq_len < 1 || r_max < 0 || n_heads < 1 || n_kv_heads < 1 ||
        n_heads % n_kv_heads != 0 || idx_stride < r_max || n_seed < 0 || !isfinite(scale))
        return EC_ERR_SHAPE;
    if (dtype != EC_BF16 || (head_dim != 64 && head_dim != 128)) return EC_ERR_UNSUPPORTED;
    if (!count || !workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!q || !k_cache || !idx || !role || !drafted || !u || !d_in || !d_out || !score))
        return EC_ERR_NULL;
    if (n_seed > 0 && !seeds) return EC_ERR_NULL;
    if ((q && !ec::aligned16(q)) || (k_cache && !ec::aligned16(k_cache))) return EC_ERR_ALIGN;
    const ec::Layout w = ec::layout(batch, seq_len, r_max, n_heads);
    if ((reinterpret_cast<uintptr_t>(workspace) % EC_WORKSPACE_ALIGN) != 0 || workspace_bytes < w.total)
        return EC_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    ec::cover::Args A;
    A.q = static_cast<const uint16_t *>(q);
    A.k_cache = static_cast<const uint16_t *>(k_cache);
    A.idx = idx;
    A.idx_stride = idx_stride;
    A.count = count;
    A.role = role;
    A.drafted = drafted;
    A.u = u;
    A.B = batch;
    A.L = seq_len;
    A.R = r_max;
    A.H = n_heads;
    A.Hkv = n_kv_heads;
    ec::cover::plan(batch, seq_len, r_max, n_heads, &A.n_chunks, &A.chunk_len);
    A.n_seed = n_seed;
    A.scale = scale;
    A.part = reinterpret_cast<ec::cover::Part *>(ws + w.part);
    A.stat_m = reinterpret_cast<float *>(ws + w.stat_m);
    A.stat_z = reinterpret_cast<float *>(ws + w.stat_z);
    A.dout_h = reinterpret_cast<float *>(ws + w.dout_h);
    A.din_h = reinterpret_cast<float *>(ws + w.din_h);
    A.d_in = d_in;
    A.d_out = d_out;
    A.score = score;
    A.seeds = seeds;
    A.status = reinterpret_cast<uint32_t *>(ws);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = head_dim == 64 ? ec::launch_all<64>(A, s) : ec::launch_all<128>(A, s);
    return e == cudaSuccess ? EC_OK : EC_ERR_CUDA;
}

int32_t ec_cover_score_kernel_count(int32_t batch, int32_t r_max, int32_t n_seed)
{
    if (batch < 1 || r_max < 0 || n_seed < 0) return 0;
    if (r_max == 0) return n_seed > 0 ? 1 : 0;
    return n_seed > 0 ? 5 : 4;
}

}  // extern "C"
