// Internal declarations shared by the CUDA sources of libec (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "ec.h"

namespace ec {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Every workspace starts with a 256-byte header; its first word is the device
// status word (EC_DEV_* bits).
constexpr size_t kWsHeader = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__device__ __forceinline__ uint32_t ld_status(const uint32_t *status) { return __ldcg(status); }
__device__ __forceinline__ void flag_status(uint32_t *status, uint32_t bits)
{
    if (status) atomicOr(status, bits);
}

// 2^x on the SFU (ex2.approx, flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

int device_sm_count();  // SM count of the current device (cached per device)

// Cycles one in-kernel wait may take before it gives up (kernels carry it in
// their parameters): about 2 s, unless ec_debug_set_wait_limit lowered it.
long long wait_limit_cycles();

// ---- launches ----
// Every kernel of the library is launched with programmatic dependent launch:
// it may start while the previous kernel on the stream is still running.  Its
// CTAs first do their set-up that touches no global memory (barriers, TMEM,
// tensor-map prefetch), then pdl_wait() until the previous grid has completed
// and its writes are visible, and only then read or write global memory.  Each
// kernel calls pdl_launch_dependents() on entry so the next one can start early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Per (kernel, device), once: the dynamic shared-memory limit (when above the
// default) and the largest shared-memory carveout, so that SMs need no
// reconfiguration between the library's kernels.
cudaError_t configure_kernel(const void *kernel, int dynamic_smem);

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, Args &&...args)
{
    cudaError_t e = configure_kernel(reinterpret_cast<const void *>(kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- launchers (each returns cudaSuccess or the launch error) ----

// decode_gate.cu
size_t decode_workspace_bytes(int32_t n_rows, int32_t batch);
cudaError_t launch_decode_gate(const void *logits, int dtype, int64_t row_stride, int32_t n_rows,
                               int32_t vocab, const int32_t *seq_row_offsets,
                               const int32_t *row_pos, int32_t batch, int32_t seq_len,
                               int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                               float *conf_out, float *entropy_out, int32_t *unmask_rows,
                               float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                               int32_t *seq_tokens, int32_t *decode_step, void *workspace,
                               cudaStream_t stream);

// lmhead_gate.cu
bool lmhead_shape_ok(int32_t n_rows, int32_t hidden, int32_t vocab);
size_t lmhead_workspace_bytes(int32_t n_rows, int32_t vocab, int32_t batch);
cudaError_t launch_lmhead_gate(const void *hidden, const void *w_lm, int32_t n_rows,
                               int32_t hidden_dim, int32_t vocab, const int32_t *seq_row_offsets,
                               const int32_t *row_pos, int32_t batch, int32_t seq_len,
                               int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                               float *conf_out, float *entropy_out, int32_t *unmask_rows,
                               float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                               int32_t *seq_tokens, int32_t *decode_step, void *workspace,
                               cudaStream_t stream);

// recompute_set.cu
cudaError_t launch_recompute_set(const uint8_t *is_masked, const int32_t *decode_step,
                                 const uint8_t *refresh, int32_t batch, int32_t seq_len,
                                 int32_t block_lo, int32_t block_hi, int32_t k, int32_t *idx,
                                 int32_t *count, cudaStream_t stream);

// attention_simt.cu
size_t attention_workspace_bytes(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                 int32_t n_kv_heads, int32_t head_dim);
cudaError_t launch_scatter_kv(const void *k_new, const void *v_new, const int32_t *idx,
                              int64_t idx_stride, const int32_t *count, void *k_cache,
                              void *v_cache, int dtype, int32_t batch, int32_t seq_len,
                              int32_t r_max, int32_t n_kv_heads, int32_t head_dim,
                              uint32_t *status, cudaStream_t stream);
cudaError_t launch_attention_simt(const void *q, const void *k_cache, const void *v_cache,
                                  void *out, const int32_t *count, int dtype, int32_t batch,
                                  int32_t seq_len, int32_t r_max, int32_t n_heads,
                                  int32_t n_kv_heads, int32_t head_dim, float scale,
                                  uint32_t *status, cudaStream_t stream);

// attention_tc.cu
bool attention_tc_supported(int dtype, int32_t seq_len, int32_t head_dim);
int32_t attention_tc_kernel_count(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                  int32_t n_kv_heads);
size_t attention_tc_workspace_bytes(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                    int32_t n_kv_heads, int32_t head_dim);
cudaError_t launch_attention_tc(const void *q, const void *k_new, const void *v_new,
                                const int32_t *idx, int64_t idx_stride, const int32_t *count,
                                void *k_cache, void *v_cache, void *out, int32_t batch,
                                int32_t seq_len, int32_t r_max, int32_t n_heads,
                                int32_t n_kv_heads, int32_t head_dim, float scale,
                                void *workspace, cudaStream_t stream,
                                const uint8_t *section = nullptr, const int32_t *tau = nullptr,
                                const uint8_t *seed = nullptr);

// qkv_gemm.cu
bool qkv_shape_ok(int32_t hidden, int32_t width);
bool linear_shape_ok(int32_t in_features, int32_t out_features, int32_t mode);
cudaError_t launch_linear(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                          int32_t in_features, const void *w, int32_t out_features, int32_t mode,
                          const void *residual, void *out, uint32_t *status, cudaStream_t stream);

// layer_ops.cu
bool rms_norm_shape_ok(int32_t hidden);
cudaError_t launch_rms_norm(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                            int32_t hidden, const void *weight, float eps, void *out,
                            cudaStream_t stream);
bool rope_shape_ok(int32_t head_dim);
cudaError_t launch_rope(void *q, void *k, const int32_t *idx, int64_t idx_stride, const int32_t *count,
                        int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, double theta, uint32_t *status,
                        cudaStream_t stream);
cudaError_t launch_qkv_projection(const void *x, const int32_t *count, int32_t batch,
                                  int32_t r_max, int32_t hidden, const void *w_qkv, int32_t width,
                                  void *q, void *k, void *v, uint32_t *status, cudaStream_t stream);
cudaError_t launch_embed_rows(const void *table, int64_t table_rows, int32_t hidden,
                              const int32_t *idx, int64_t idx_stride, const int32_t *count,
                              const int32_t *seq_tokens, const uint8_t *is_masked, int32_t mask_id,
                              int32_t batch, int32_t seq_len, int32_t r_max, void *x,
                              uint32_t *status, cudaStream_t stream);

}  // namespace ec
