// The row-wise operations of a pre-norm transformer layer around the dense
// contractions: RMS normalisation and rotary position embedding of the
// recomputed rows.
//
// The pages' models (LLaDA-8B, Dream-7B) are pre-norm decoder stacks with RMSNorm
// and rotary embeddings; a partial forward ("Algoritmo di Funzionamento" step 2
// of the EntropyCache summary) runs them on the recomputed rows only, each row at
// its own position.
//   rms_norm   y = x / sqrt(mean(x^2) + eps) * g, float32 arithmetic, bf16 out;
//   rope       every query and key head of a row at position p: the pairs
//              (x_i, x_{i + d/2}), i < d/2, turned by p * theta^(-2 i / d)
//              (the rotate-half pairing), in place.
#include <cuda_bf16.h>

#include <algorithm>

#include "ec_internal.cuh"

namespace ec {
namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float lo_f(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float hi_f(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// One block per (row, sequence); 8 bf16 per uint4.
__global__ void __launch_bounds__(kNormThreads)
    rms_norm_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ g, int row_vec, float eps,
                    const int32_t *__restrict__ count, int r_max, uint4 *__restrict__ y)
{
    pdl_launch_dependents();
    pdl_wait();  // inputs belong to the previous kernel until here
    const int r = blockIdx.x, b = blockIdx.y;
    const int c = count ? max(0, min(__ldg(count + b), r_max)) : r_max;
    if (r >= c) return;
    const int64_t base = (static_cast<int64_t>(b) * r_max + r) * row_vec;
    float ss = 0.f;
    for (int i = threadIdx.x; i < row_vec; i += kNormThreads) {
        const uint4 v = x[base + i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ss = fmaf(lo_f(w[e]), lo_f(w[e]), ss);
            ss = fmaf(hi_f(w[e]), hi_f(w[e]), ss);
        }
    }
    __shared__ float part[kNormThreads / 32];
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
    const float inv = rsqrtf(tot / static_cast<float>(row_vec * 8) + eps);
    for (int i = threadIdx.x; i < row_vec; i += kNormThreads) {
        const uint4 v = x[base + i], s = __ldg(g + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w}, sw[4] = {s.x, s.y, s.z, s.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[e] = pack2(lo_f(w[e]) * inv * lo_f(sw[e]), hi_f(w[e]) * inv * hi_f(sw[e]));
        y[base + i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

constexpr int kRopeThreads = 128;

// One block per (row, sequence): the row's d/2 angles in double precision, then
// every (head, pair) of its query and key rows.
__global__ void __launch_bounds__(kRopeThreads)
    rope_kernel(__nv_bfloat16 *__restrict__ q, __nv_bfloat16 *__restrict__ k,
                const int32_t *__restrict__ idx, int64_t idx_stride, const int32_t *__restrict__ count,
                int r_max, int n_heads, int n_kv_heads, int head_dim, double theta, int seq_len,
                uint32_t *status)
{
    pdl_launch_dependents();
    pdl_wait();  // inputs belong to the previous kernel until here
    const int r = blockIdx.x, b = blockIdx.y;
    const int c = max(0, min(__ldg(count + b), r_max));
    if (r >= c) return;
    const int pos = __ldg(idx + b * idx_stride + r);
    if (pos < 0 || pos >= seq_len) {
        if (threadIdx.x == 0) flag_status(status, EC_DEV_BAD_INDEX);
        return;
    }
    const int half = head_dim / 2;
    __shared__ float cs[64], sn[64];  // head_dim <= 128
    for (int i = threadIdx.x; i < half; i += kRopeThreads) {
        const double a = static_cast<double>(pos) * pow(theta, -2.0 * i / head_dim);
        double sv, cv;
        sincos(a, &sv, &cv);
        cs[i] = static_cast<float>(cv);
        sn[i] = static_cast<float>(sv);
    }
    __syncthreads();
    const int total = (n_heads + n_kv_heads) * half;
    for (int t = threadIdx.x; t < total; t += kRopeThreads) {
        const int h = t / half, i = t - h * half;
        __nv_bfloat16 *row = h < n_heads
                                 ? q + ((static_cast<int64_t>(b) * r_max + r) * n_heads + h) * head_dim
                                 : k + ((static_cast<int64_t>(b) * r_max + r) * n_kv_heads + (h - n_heads)) *
                                           head_dim;
        const float x1 = __bfloat162float(row[i]), x2 = __bfloat162float(row[i + half]);
        row[i] = __float2bfloat16_rn(x1 * cs[i] - x2 * sn[i]);
        row[i + half] = __float2bfloat16_rn(x2 * cs[i] + x1 * sn[i]);
    }
}

}  // namespace

bool rms_norm_shape_ok(int32_t hidden) { return hidden >= 8 && hidden % 8 == 0; }

cudaError_t launch_rms_norm(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                            int32_t hidden, const void *weight, float eps, void *out,
                            cudaStream_t stream)
{
    if (r_max == 0) return cudaSuccess;
    return launch(rms_norm_kernel, dim3(static_cast<unsigned>(r_max), static_cast<unsigned>(batch)),
                  dim3(kNormThreads), 0, stream, static_cast<const uint4 *>(x),
                  static_cast<const uint4 *>(weight), hidden / 8, eps, count, r_max,
                  static_cast<uint4 *>(out));
}

bool rope_shape_ok(int32_t head_dim) { return head_dim >= 2 && head_dim <= 128 && head_dim % 2 == 0; }

cudaError_t launch_rope(void *q, void *k, const int32_t *idx, int64_t idx_stride, const int32_t *count,
                        int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, double theta, uint32_t *status,
                        cudaStream_t stream)
{
    if (r_max == 0) return cudaSuccess;
    return launch(rope_kernel, dim3(static_cast<unsigned>(r_max), static_cast<unsigned>(batch)),
                  dim3(kRopeThreads), 0, stream, static_cast<__nv_bfloat16 *>(q),
                  static_cast<__nv_bfloat16 *>(k), idx, idx_stride, count, r_max, n_heads, n_kv_heads,
                  head_dim, theta, seq_len, status);
}

}  // namespace ec
