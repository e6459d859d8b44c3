// KV write-back and a CUDA-core (SIMT) selective bidirectional attention.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, section "1. Il Problema" (dLLM attention is
// bidirectional: every position attends to all others) and "Algoritmo di
// Funzionamento" step 2 (the partial forward recomputes K/V of the selected
// tokens only; the cache supplies all others).
//
// The SIMT kernel is the float32 path (its inputs cannot go through the bf16
// tensor cores without losing precision) and the reference kernel for the
// tensor-core path.  One warp owns one (sequence, query row, head): each lane
// holds head_dim/32 components of q, keys are visited in order with an online
// softmax in the log2 domain, and the output is normalised at the end.
#include <cuda_bf16.h>

#include <algorithm>

#include "ec_internal.cuh"

namespace ec {
namespace {

template <typename T, int P>
struct Lanes;

template <int P>
struct Lanes<float, P> {
    __device__ static __forceinline__ void load(const float *p, float (&x)[P])
    {
#pragma unroll
        for (int i = 0; i < P; ++i) x[i] = __ldg(p + i);
    }
    __device__ static __forceinline__ void store(float *p, const float (&x)[P])
    {
#pragma unroll
        for (int i = 0; i < P; ++i) p[i] = x[i];
    }
};

template <int P>
struct Lanes<__nv_bfloat16, P> {
    __device__ static __forceinline__ void load(const __nv_bfloat16 *p, float (&x)[P])
    {
#pragma unroll
        for (int i = 0; i < P; ++i) x[i] = __bfloat162float(p[i]);
    }
    __device__ static __forceinline__ void store(__nv_bfloat16 *p, const float (&x)[P])
    {
#pragma unroll
        for (int i = 0; i < P; ++i) p[i] = __float2bfloat16_rn(x[i]);
    }
};

// cache[b, idx[b, r]] = fresh[b, r] for r < count[b]; grid (r_max, batch).
__global__ void scatter_kv_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                  const int32_t *__restrict__ idx, int64_t idx_stride,
                                  const int32_t *__restrict__ count, uint4 *k_cache,
                                  uint4 *v_cache, int L, int r_max, int row_vec, uint32_t *status)
{
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.y, r = blockIdx.x;
    int c = __ldg(count + b);
    if (c < 0 || c > r_max) {
        if (threadIdx.x == 0 && r == 0) flag_status(status, EC_DEV_BAD_COUNT);
        c = max(0, min(c, r_max));
    }
    if (r >= c) return;
    const int32_t *row_idx = idx + static_cast<int64_t>(b) * idx_stride;
    const int p = __ldg(row_idx + r);
    const bool bad = p < 0 || p >= L || (r > 0 && __ldg(row_idx + r - 1) >= p);
    if (bad && threadIdx.x == 0) flag_status(status, EC_DEV_BAD_INDEX);
    if (p < 0 || p >= L) return;
    const int64_t src = (static_cast<int64_t>(b) * r_max + r) * row_vec;
    const int64_t dst = (static_cast<int64_t>(b) * L + p) * row_vec;
    for (int i = threadIdx.x; i < row_vec; i += blockDim.x) {
        k_cache[dst + i] = __ldg(k_new + src + i);
        v_cache[dst + i] = __ldg(v_new + src + i);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(128) attention_simt_kernel(
    const T *__restrict__ q, const T *__restrict__ k_cache, const T *__restrict__ v_cache,
    T *__restrict__ out, const int32_t *__restrict__ count, int L, int r_max, int H, int Hkv,
    float scale_log2)
{
    pdl_launch_dependents();
    pdl_wait();
    constexpr int P = D / 32;
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int r = w / H, h = w - (w / H) * H;
    const int c = max(0, min(__ldg(count + b), r_max));
    if (r >= c) return;
    const int g = h / (H / Hkv);

    float qv[P];
    Lanes<T, P>::load(q + ((static_cast<int64_t>(b) * r_max + r) * H + h) * D + lane * P, qv);
#pragma unroll
    for (int i = 0; i < P; ++i) qv[i] *= scale_log2;

    const int64_t key_stride = static_cast<int64_t>(Hkv) * D;
    const T *kp = k_cache + (static_cast<int64_t>(b) * L * Hkv + g) * D + lane * P;
    const T *vp = v_cache + (static_cast<int64_t>(b) * L * Hkv + g) * D + lane * P;
    float m = -INFINITY, l = 0.f, o[P];
#pragma unroll
    for (int i = 0; i < P; ++i) o[i] = 0.f;
    for (int j = 0; j < L; ++j) {
        float kv[P], vv[P];
        Lanes<T, P>::load(kp + j * key_stride, kv);
        Lanes<T, P>::load(vp + j * key_stride, vv);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < P; ++i) s = fmaf(qv[i], kv[i], s);
#pragma unroll
        for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (s > m) {
            const float alpha = ex2(m - s);
            l *= alpha;
#pragma unroll
            for (int i = 0; i < P; ++i) o[i] *= alpha;
            m = s;
        }
        const float pj = ex2(s - m);
        l += pj;
#pragma unroll
        for (int i = 0; i < P; ++i) o[i] = fmaf(pj, vv[i], o[i]);
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < P; ++i) o[i] *= inv;
    Lanes<T, P>::store(out + ((static_cast<int64_t>(b) * r_max + r) * H + h) * D + lane * P, o);
}

template <typename T>
cudaError_t launch_simt_typed(const void *q, const void *kc, const void *vc, void *out,
                              const int32_t *count, int32_t batch, int32_t L, int32_t r_max,
                              int32_t H, int32_t Hkv, int32_t d, float scale, cudaStream_t stream)
{
    const int64_t warps = static_cast<int64_t>(r_max) * H;
    const dim3 grid(static_cast<unsigned>((warps + 3) / 4), static_cast<unsigned>(batch));
    const float sl2 = scale * kLog2e;
    auto kernel = d == 128 ? attention_simt_kernel<T, 128> : attention_simt_kernel<T, 64>;
    return launch(kernel, grid, dim3(128), 0, stream, static_cast<const T *>(q),
                  static_cast<const T *>(kc), static_cast<const T *>(vc), static_cast<T *>(out),
                  count, L, r_max, H, Hkv, sl2);
}

}  // namespace

size_t attention_workspace_bytes(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                 int32_t n_kv_heads, int32_t head_dim)
{
    // the SIMT path needs only the status header; the tensor-core path also keeps
    // split-KV partials and its grid-barrier words
    return std::max(kWsHeader, attention_tc_workspace_bytes(batch, seq_len, r_max, n_heads,
                                                            n_kv_heads, head_dim));
}

cudaError_t launch_scatter_kv(const void *k_new, const void *v_new, const int32_t *idx,
                              int64_t idx_stride, const int32_t *count, void *k_cache,
                              void *v_cache, int dtype, int32_t batch, int32_t seq_len,
                              int32_t r_max, int32_t n_kv_heads, int32_t head_dim,
                              uint32_t *status, cudaStream_t stream)
{
    if (r_max == 0 || batch == 0) return cudaSuccess;
    const int elem = dtype == EC_BF16 ? 2 : 4;
    const int row_vec = n_kv_heads * head_dim * elem / 16;
    const dim3 grid(static_cast<unsigned>(r_max), static_cast<unsigned>(batch));
    return launch(scatter_kv_kernel, grid, dim3(128), 0, stream,
                  static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), idx,
                  idx_stride, count, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                  seq_len, r_max, row_vec, status);
}

cudaError_t launch_attention_simt(const void *q, const void *k_cache, const void *v_cache,
                                  void *out, const int32_t *count, int dtype, int32_t batch,
                                  int32_t seq_len, int32_t r_max, int32_t n_heads,
                                  int32_t n_kv_heads, int32_t head_dim, float scale,
                                  uint32_t *, cudaStream_t stream)
{
    if (r_max == 0 || batch == 0) return cudaSuccess;
    if (dtype == EC_BF16)
        return launch_simt_typed<__nv_bfloat16>(q, k_cache, v_cache, out, count, batch, seq_len,
                                                r_max, n_heads, n_kv_heads, head_dim, scale, stream);
    return launch_simt_typed<float>(q, k_cache, v_cache, out, count, batch, seq_len, r_max,
                                    n_heads, n_kv_heads, head_dim, scale, stream);
}

}  // namespace ec
