// C ABI of libec: argument validation, workspace carving and kernel dispatch.
// Every check here runs on the host before anything is enqueued.
#include <math.h>

#include <atomic>
#include <mutex>

#include "ec_internal.cuh"
#include "tc_ptx.cuh"

namespace ec {

static std::atomic<long long> g_wait_limit{0};

long long wait_limit_cycles()
{
    const long long v = g_wait_limit.load(std::memory_order_relaxed);
    return v > 0 ? v : ptx::kWaitCycles;
}

cudaError_t configure_kernel(const void *kernel, int dynamic_smem)
{
    struct Done {
        const void *kernel;
        int dev;
    };
    static std::mutex mu;
    static Done done[256];
    static int n_done = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].kernel == kernel && done[i].dev == dev) return cudaSuccess;
    if (dynamic_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dynamic_smem);
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (n_done < 256) done[n_done++] = Done{kernel, dev};
    return cudaSuccess;
}

int device_sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev < 64) cached[dev] = n;
    return n;
}

}  // namespace ec

namespace {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline ec_status launched(cudaError_t e) { return e == cudaSuccess ? EC_OK : EC_ERR_CUDA; }

}  // namespace

extern "C" {

const char *ec_status_str(int s)
{
    switch (s) {
    case EC_OK: return "EC_OK";
    case EC_ERR_NULL: return "EC_ERR_NULL: a required pointer is NULL";
    case EC_ERR_SHAPE: return "EC_ERR_SHAPE: a size or scalar argument is out of range";
    case EC_ERR_DTYPE: return "EC_ERR_DTYPE: unsupported element type";
    case EC_ERR_ALIGN: return "EC_ERR_ALIGN: pointer or row stride breaks the 16-byte rule";
    case EC_ERR_WORKSPACE: return "EC_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case EC_ERR_CUDA: return "EC_ERR_CUDA: a CUDA call or kernel launch failed";
    case EC_ERR_UNSUPPORTED: return "EC_ERR_UNSUPPORTED: not implemented for these arguments";
    case EC_ERR_SCRATCH_LIMIT:
        return "EC_ERR_SCRATCH_LIMIT: request exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown ec_status";
    }
}

int ec_abi_version(void) { return EC_ABI_VERSION; }

ec_status ec_debug_set_wait_limit(int64_t cycles)
{
    if (cycles < 0) return EC_ERR_SHAPE;
    ec::g_wait_limit.store(static_cast<long long>(cycles), std::memory_order_relaxed);
    return EC_OK;
}

ec_status ec_workspace_init(void *workspace, size_t workspace_bytes, ec_stream_t stream)
{
    if (!workspace) return EC_ERR_NULL;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) || workspace_bytes < ec::kWsHeader)
        return EC_ERR_WORKSPACE;
    return launched(cudaMemsetAsync(workspace, 0, workspace_bytes, stream));
}

ec_status ec_read_device_status(void *workspace, uint32_t *bits, ec_stream_t stream)
{
    if (!workspace || !bits) return EC_ERR_NULL;
    uint32_t v = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return EC_ERR_CUDA;
    if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return EC_ERR_CUDA;
    if (cudaMemset(workspace, 0, sizeof v) != cudaSuccess) return EC_ERR_CUDA;
    *bits = v;
    return EC_OK;
}

size_t ec_decode_workspace_size(int32_t n_rows, int32_t batch)
{
    return ec::decode_workspace_bytes(n_rows, batch);
}

ec_status ec_decode_step(const void *logits, ec_dtype dtype, int64_t row_stride, int32_t n_rows,
                         int32_t vocab, const int32_t *seq_row_offsets, const int32_t *row_pos,
                         int32_t batch, int32_t seq_len, int32_t n_unmask, float tau,
                         int32_t step, int32_t *token_out, float *conf_out,
                         float *entropy_out, int32_t *unmask_rows, float *max_entropy,
                         uint8_t *refresh, uint8_t *is_masked, int32_t *seq_tokens,
                         int32_t *decode_step, void *workspace, size_t workspace_bytes,
                         ec_stream_t stream)
{
    if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_DTYPE;
    if (n_rows < 0 || vocab < 1 || batch < 1 || seq_len < 1 || n_unmask < 1 ||
        n_unmask > 1024 || row_stride < vocab || !isfinite(tau))
        return EC_ERR_SHAPE;
    if (!seq_row_offsets || !unmask_rows || !max_entropy || !refresh || !is_masked ||
        !seq_tokens || !decode_step || !workspace)
        return EC_ERR_NULL;
    if (n_rows > 0 && (!logits || !row_pos || !token_out || !conf_out || !entropy_out))
        return EC_ERR_NULL;
    const int elem = dtype == EC_BF16 ? 2 : 4;
    if (n_rows > 0 && (!aligned(logits, 16) || (row_stride * elem) % 16 != 0)) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) ||
        workspace_bytes < ec::decode_workspace_bytes(n_rows, batch))
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_decode_gate(
        logits, dtype, row_stride, n_rows, vocab, seq_row_offsets, row_pos, batch, seq_len,
        n_unmask, tau, step, token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
        is_masked, seq_tokens, decode_step, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

size_t ec_lmhead_workspace_size(int32_t n_rows, int32_t vocab, int32_t batch)
{
    return ec::lmhead_workspace_bytes(n_rows, vocab, batch);
}

ec_status ec_lmhead_decode_step(const void *hidden, const void *w_lm, int32_t n_rows,
                                int32_t hidden_dim, int32_t vocab, const int32_t *seq_row_offsets,
                                const int32_t *row_pos, int32_t batch, int32_t seq_len,
                                int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                                float *conf_out, float *entropy_out, int32_t *unmask_rows,
                                float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                                int32_t *seq_tokens, int32_t *decode_step, void *workspace,
                                size_t workspace_bytes, ec_stream_t stream)
{
    if (batch < 1 || seq_len < 1 || n_unmask < 1 || n_unmask > 1024 || !isfinite(tau) ||
        !ec::lmhead_shape_ok(n_rows, hidden_dim, vocab))
        return EC_ERR_SHAPE;
    if (!seq_row_offsets || !unmask_rows || !max_entropy || !refresh || !is_masked ||
        !seq_tokens || !decode_step || !workspace)
        return EC_ERR_NULL;
    if (n_rows > 0 && (!hidden || !w_lm || !row_pos || !token_out || !conf_out || !entropy_out))
        return EC_ERR_NULL;
    if ((hidden && !aligned(hidden, 16)) || (w_lm && !aligned(w_lm, 16))) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) ||
        workspace_bytes < ec::lmhead_workspace_bytes(n_rows, vocab, batch))
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_lmhead_gate(
        hidden, w_lm, n_rows, hidden_dim, vocab, seq_row_offsets, row_pos, batch, seq_len, n_unmask,
        tau, step, token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh, is_masked,
        seq_tokens, decode_step, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

ec_status ec_build_recompute_set(const uint8_t *is_masked, const int32_t *decode_step,
                                 const uint8_t *refresh, int32_t batch, int32_t seq_len,
                                 int32_t block_lo, int32_t block_hi, int32_t k, int32_t *idx,
                                 int32_t *count, ec_stream_t stream)
{
    if (!is_masked || !decode_step || !refresh || !idx || !count) return EC_ERR_NULL;
    if (batch < 1 || seq_len < 1 || k < 0 || block_lo < 0 || block_hi < block_lo ||
        block_hi > seq_len)
        return EC_ERR_SHAPE;
    return launched(ec::launch_recompute_set(is_masked, decode_step, refresh, batch, seq_len,
                                             block_lo, block_hi, k, idx, count,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

size_t ec_attention_workspace_size(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                   int32_t n_kv_heads, int32_t head_dim)
{
    return ec::attention_workspace_bytes(batch, seq_len, r_max, n_heads, n_kv_heads, head_dim);
}

int32_t ec_attention_kernel_count(ec_dtype dtype, int32_t batch, int32_t seq_len, int32_t r_max,
                                  int32_t n_heads, int32_t n_kv_heads, int32_t head_dim)
{
    if ((dtype != EC_F32 && dtype != EC_BF16) || batch < 1 || seq_len < 1 || r_max < 0 ||
        n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads != 0 ||
        (head_dim != 64 && head_dim != 128))
        return -1;
    if (r_max == 0) return 0;
    if (ec::attention_tc_supported(dtype, seq_len, head_dim))
        return ec::attention_tc_kernel_count(batch, seq_len, r_max, n_heads, n_kv_heads);
    return 2;
}

ec_status ec_selective_attention(const void *q, const void *k_new, const void *v_new,
                                 const int32_t *idx, int64_t idx_stride, const int32_t *count,
                                 void *k_cache, void *v_cache, void *out, ec_dtype dtype,
                                 int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                 int32_t n_kv_heads, int32_t head_dim, float scale,
                                 void *workspace, size_t workspace_bytes, ec_stream_t stream)
{
    if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_DTYPE;
    if (batch < 1 || seq_len < 1 || r_max < 0 || n_heads < 1 || n_kv_heads < 1 ||
        n_heads % n_kv_heads != 0 || (head_dim != 64 && head_dim != 128) || idx_stride < r_max ||
        !isfinite(scale))
        return EC_ERR_SHAPE;
    if (!count || !k_cache || !v_cache || !workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!q || !k_new || !v_new || !idx || !out)) return EC_ERR_NULL;
    const void *ptrs[] = {q, k_new, v_new, k_cache, v_cache, out};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) ||
        workspace_bytes <
            ec::attention_workspace_bytes(batch, seq_len, r_max, n_heads, n_kv_heads, head_dim))
        return EC_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t *status = static_cast<uint32_t *>(workspace);
    if (ec::attention_tc_supported(dtype, seq_len, head_dim))  // write-back, attention, merge
        return launched(ec::launch_attention_tc(q, k_new, v_new, idx, idx_stride, count, k_cache,
                                                v_cache, out, batch, seq_len, r_max, n_heads,
                                                n_kv_heads, head_dim, scale, workspace, s));
    cudaError_t e = ec::launch_scatter_kv(k_new, v_new, idx, idx_stride, count, k_cache, v_cache,
                                          dtype, batch, seq_len, r_max, n_kv_heads, head_dim,
                                          status, s);
    if (e != cudaSuccess) return EC_ERR_CUDA;
    return launched(ec::launch_attention_simt(q, k_cache, v_cache, out, count, dtype, batch,
                                              seq_len, r_max, n_heads, n_kv_heads, head_dim,
                                              scale, status, s));
}

ec_status ec_selective_attention_simsd(const void *q, const void *k_new, const void *v_new,
                                       const int32_t *idx, int64_t idx_stride,
                                       const int32_t *count, const uint8_t *section,
                                       const int32_t *tau, void *k_cache, void *v_cache,
                                       void *out, ec_dtype dtype, int32_t batch, int32_t seq_len,
                                       int32_t r_max, int32_t n_heads, int32_t n_kv_heads,
                                       int32_t head_dim, float scale, void *workspace,
                                       size_t workspace_bytes, ec_stream_t stream)
{
    if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_DTYPE;
    if (batch < 1 || seq_len < 1 || r_max < 0 || n_heads < 1 || n_kv_heads < 1 ||
        n_heads % n_kv_heads != 0 || (head_dim != 64 && head_dim != 128) || idx_stride < r_max ||
        !isfinite(scale))
        return EC_ERR_SHAPE;
    if (!count || !k_cache || !v_cache || !workspace || !section || !tau) return EC_ERR_NULL;
    if (r_max > 0 && (!q || !k_new || !v_new || !idx || !out)) return EC_ERR_NULL;
    if (!ec::attention_tc_supported(dtype, seq_len, head_dim)) return EC_ERR_UNSUPPORTED;
    const void *ptrs[] = {q, k_new, v_new, k_cache, v_cache, out};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) ||
        workspace_bytes <
            ec::attention_workspace_bytes(batch, seq_len, r_max, n_heads, n_kv_heads, head_dim))
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_attention_tc(q, k_new, v_new, idx, idx_stride, count, k_cache,
                                            v_cache, out, batch, seq_len, r_max, n_heads,
                                            n_kv_heads, head_dim, scale, workspace,
                                            reinterpret_cast<cudaStream_t>(stream), section, tau));
}

ec_status ec_selective_attention_cover(const void *q, const void *k_new, const void *v_new,
                                       const int32_t *idx, int64_t idx_stride,
                                       const int32_t *count, const uint8_t *seed, void *k_cache,
                                       void *v_cache, void *out, ec_dtype dtype, int32_t batch,
                                       int32_t seq_len, int32_t r_max, int32_t n_heads,
                                       int32_t n_kv_heads, int32_t head_dim, float scale,
                                       void *workspace, size_t workspace_bytes,
                                       ec_stream_t stream)
{
    if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_DTYPE;
    if (batch < 1 || seq_len < 1 || r_max < 0 || n_heads < 1 || n_kv_heads < 1 ||
        n_heads % n_kv_heads != 0 || (head_dim != 64 && head_dim != 128) || idx_stride < r_max ||
        !isfinite(scale))
        return EC_ERR_SHAPE;
    if (!count || !k_cache || !v_cache || !workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!q || !k_new || !v_new || !idx || !out || !seed)) return EC_ERR_NULL;
    if (!ec::attention_tc_supported(dtype, seq_len, head_dim)) return EC_ERR_UNSUPPORTED;
    const void *ptrs[] = {q, k_new, v_new, k_cache, v_cache, out};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) ||
        workspace_bytes <
            ec::attention_workspace_bytes(batch, seq_len, r_max, n_heads, n_kv_heads, head_dim))
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_attention_tc(q, k_new, v_new, idx, idx_stride, count, k_cache,
                                            v_cache, out, batch, seq_len, r_max, n_heads,
                                            n_kv_heads, head_dim, scale, workspace,
                                            reinterpret_cast<cudaStream_t>(stream), nullptr,
                                            nullptr, seed));
}

ec_status ec_qkv_projection(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                            int32_t hidden, const void *w_qkv, int32_t width, void *q, void *k,
                            void *v, void *workspace, size_t workspace_bytes, ec_stream_t stream)
{
    if (batch < 1 || r_max < 0 || !ec::qkv_shape_ok(hidden, width)) return EC_ERR_SHAPE;
    if (!workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!x || !w_qkv || !q || !k || !v)) return EC_ERR_NULL;
    const void *ptrs[] = {x, w_qkv, q, k, v};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) || workspace_bytes < ec::kWsHeader)
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_qkv_projection(x, count, batch, r_max, hidden, w_qkv, width, q, k,
                                              v, static_cast<uint32_t *>(workspace),
                                              reinterpret_cast<cudaStream_t>(stream)));
}

ec_status ec_embed_rows(const void *table, int64_t table_rows, int32_t hidden, const int32_t *idx,
                        int64_t idx_stride, const int32_t *count, const int32_t *seq_tokens,
                        const uint8_t *is_masked, int32_t mask_id, int32_t batch,
                        int32_t seq_len, int32_t r_max, void *x, void *workspace,
                        size_t workspace_bytes, ec_stream_t stream)
{
    if (batch < 1 || seq_len < 1 || r_max < 0 || table_rows < 1 || hidden < 8 || hidden % 8 ||
        idx_stride < r_max || mask_id < 0 || mask_id >= table_rows)
        return EC_ERR_SHAPE;
    if (!count || !workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!table || !idx || !seq_tokens || !is_masked || !x)) return EC_ERR_NULL;
    if ((table && !aligned(table, 16)) || (x && !aligned(x, 16))) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) || workspace_bytes < ec::kWsHeader)
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_embed_rows(table, table_rows, hidden, idx, idx_stride, count,
                                          seq_tokens, is_masked, mask_id, batch, seq_len, r_max, x,
                                          static_cast<uint32_t *>(workspace),
                                          reinterpret_cast<cudaStream_t>(stream)));
}


ec_status ec_rms_norm(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                      int32_t hidden, const void *weight, float eps, void *y, void *workspace,
                      size_t workspace_bytes, ec_stream_t stream)
{
    if (batch < 1 || r_max < 0 || !ec::rms_norm_shape_ok(hidden) || !(eps >= 0.f) || !isfinite(eps))
        return EC_ERR_SHAPE;
    if (!workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!x || !weight || !y)) return EC_ERR_NULL;
    const void *ptrs[] = {x, weight, y};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) || workspace_bytes < ec::kWsHeader)
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_rms_norm(x, count, batch, r_max, hidden, weight, eps, y,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

ec_status ec_rope(void *q, void *k, const int32_t *idx, int64_t idx_stride, const int32_t *count,
                  int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                  int32_t n_kv_heads, int32_t head_dim, double theta, void *workspace,
                  size_t workspace_bytes, ec_stream_t stream)
{
    if (batch < 1 || seq_len < 1 || r_max < 0 || n_heads < 1 || n_kv_heads < 1 ||
        !ec::rope_shape_ok(head_dim) || idx_stride < r_max || !(theta > 1.0) || !isfinite(theta))
        return EC_ERR_SHAPE;
    if (!count || !workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!q || !k || !idx)) return EC_ERR_NULL;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) || workspace_bytes < ec::kWsHeader)
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_rope(q, k, idx, idx_stride, count, batch, seq_len, r_max, n_heads,
                                    n_kv_heads, head_dim, theta,
                                    static_cast<uint32_t *>(workspace),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

ec_status ec_linear(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                    int32_t in_features, const void *w, int32_t out_features, int32_t mode,
                    const void *residual, void *y, void *workspace, size_t workspace_bytes,
                    ec_stream_t stream)
{
    if (batch < 1 || r_max < 0 || !ec::linear_shape_ok(in_features, out_features, mode))
        return EC_ERR_SHAPE;
    if (!workspace) return EC_ERR_NULL;
    if (r_max > 0 && (!x || !w || !y || (mode == 1 && !residual))) return EC_ERR_NULL;
    const void *ptrs[] = {x, w, y, mode == 1 ? residual : nullptr};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return EC_ERR_ALIGN;
    if (!aligned(workspace, EC_WORKSPACE_ALIGN) || workspace_bytes < ec::kWsHeader)
        return EC_ERR_WORKSPACE;
    return launched(ec::launch_linear(x, count, batch, r_max, in_features, w, out_features, mode,
                                      residual, y, static_cast<uint32_t *>(workspace),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
