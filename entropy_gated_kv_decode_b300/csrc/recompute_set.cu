// Recompute index set of the next forward, one CTA per sequence.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, "Algoritmo di Funzionamento" step 2 (a partial
// forward recomputes the currently masked tokens and the k most recently
// decoded tokens; E > tau recomputes everything), and the Arabic technical
// summary, "Algorithm workflow" phase 3 (a log of decode times; the top k by
// recency join the partial recompute window).
//
// Selection of the k most recent decoded positions without sorting: a binary
// search over decode-step values finds the threshold step s* (the k-th largest
// value); every decoded position with step > s* is taken, and of those with
// step == s* the lowest positions fill the remaining slots.  One packed block
// scan per tile of 1024 positions gives each taken position its output slot,
// so the output comes out in ascending position order.
#include <limits.h>

#include "ec_internal.cuh"

namespace ec {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int block_sum(int v, int *s_red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    int t = __reduce_add_sync(0xffffffffu, s_red[lane]);
    __syncthreads();
    return t;
}

__device__ __forceinline__ int block_max(int v, int *s_red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_max_sync(0xffffffffu, v);
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    int t = __reduce_max_sync(0xffffffffu, s_red[lane]);
    __syncthreads();
    return t;
}

__device__ __forceinline__ int block_min(int v, int *s_red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_min_sync(0xffffffffu, v);
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    int t = __reduce_min_sync(0xffffffffu, s_red[lane]);
    __syncthreads();
    return t;
}

// Exclusive prefix sum over the CTA of a packed pair of 16-bit counters.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *s_scan,
                                                         uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = s_scan[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        s_scan[lane] = w;
    }
    __syncthreads();
    const uint32_t excl = x - v + (warp > 0 ? s_scan[warp - 1] : 0u);
    total = s_scan[kWarps - 1];
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(kThreads) recompute_set_kernel(
    const uint8_t *__restrict__ is_masked, const int32_t *__restrict__ decode_step,
    const uint8_t *__restrict__ refresh, int L, int block_lo, int block_hi, int k,
    int32_t *__restrict__ idx, int32_t *__restrict__ count)
{
    __shared__ int s_red[kWarps];
    __shared__ uint32_t s_scan[kWarps];
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x, tid = threadIdx.x;
    const uint8_t *im = is_masked + static_cast<int64_t>(b) * L;
    const int32_t *ds = decode_step + static_cast<int64_t>(b) * L;
    int32_t *out = idx + static_cast<int64_t>(b) * L;

    if (refresh[b]) {  // full forward: every position
        for (int p = tid; p < L; p += kThreads) out[p] = p;
        if (tid == 0) count[b] = L;
        return;
    }

    // decoded, unmasked positions: how many, and the range of their steps
    int n = 0, hi = INT_MIN, lo = INT_MAX;
    for (int p = tid; p < L; p += kThreads) {
        const int d = __ldg(ds + p);
        if (d >= 0 && !__ldg(im + p)) {
            ++n;
            hi = max(hi, d);
            lo = min(lo, d);
        }
    }
    const int n_dec = block_sum(n, s_red);
    const int d_hi = block_max(hi, s_red);
    const int d_lo = block_min(lo, s_red);

    // take: steps > thr; of steps == thr, the first `need` positions
    bool take_recent = k > 0 && n_dec > 0;
    int thr = -1, need = 0;
    if (take_recent && n_dec > k) {
        int a = d_lo, z = d_hi;  // invariant: #(step >= a) >= k
        while (a < z) {
            const int mid = a + (z - a + 1) / 2;
            int c = 0;
            for (int p = tid; p < L; p += kThreads) {
                const int d = __ldg(ds + p);
                c += (d >= mid && !__ldg(im + p)) ? 1 : 0;
            }
            if (block_sum(c, s_red) >= k)
                a = mid;
            else
                z = mid - 1;
        }
        thr = a;
        int c = 0;
        for (int p = tid; p < L; p += kThreads) {
            const int d = __ldg(ds + p);
            c += (d > thr && !__ldg(im + p)) ? 1 : 0;
        }
        need = k - block_sum(c, s_red);
    }

    // ordered compaction, one tile of kThreads positions at a time
    int carry_a = 0, carry_t = 0;
    for (int base = 0; base < L; base += kThreads) {
        const int p = base + tid;
        bool plain = false, tie = false;
        if (p < L) {
            const int d = __ldg(ds + p);
            const bool masked = __ldg(im + p) != 0;
            const bool decoded = d >= 0 && !masked;
            plain = (masked && p >= block_lo && p < block_hi) || (take_recent && decoded && d > thr);
            tie = take_recent && decoded && d == thr && need > 0;
        }
        uint32_t total;
        const uint32_t ex = block_exclusive_scan((plain ? 0x10000u : 0u) | (tie ? 1u : 0u), s_scan,
                                                 total);
        const int before_plain = carry_a + static_cast<int>(ex >> 16);
        const int before_tie = carry_t + static_cast<int>(ex & 0xffffu);
        if (plain || (tie && before_tie < need)) out[before_plain + min(before_tie, need)] = p;
        carry_a += static_cast<int>(total >> 16);
        carry_t += static_cast<int>(total & 0xffffu);
    }
    const int c = carry_a + min(carry_t, need);
    for (int p = c + tid; p < L; p += kThreads) out[p] = -1;
    if (tid == 0) count[b] = c;
}

}  // namespace

cudaError_t launch_recompute_set(const uint8_t *is_masked, const int32_t *decode_step,
                                 const uint8_t *refresh, int32_t batch, int32_t seq_len,
                                 int32_t block_lo, int32_t block_hi, int32_t k, int32_t *idx,
                                 int32_t *count, cudaStream_t stream)
{
    return launch(recompute_set_kernel, dim3(batch), dim3(kThreads), 0, stream, is_masked,
                  decode_step, refresh, seq_len, block_lo, block_hi, k, idx, count);
}

}  // namespace ec
