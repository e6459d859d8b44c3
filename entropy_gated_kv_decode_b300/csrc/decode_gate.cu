// Decode-and-gate step of EntropyCache in one kernel launch.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, "Algoritmo di Funzionamento" steps 1-2, and the
// Arabic technical summary, "Algorithm workflow" phases 2-3 with the equation
// E_{t+1} = max_{i in D_{t+1}} ( -sum_j p_ij log p_ij ).
//
// Phase 1 (every CTA): stream one slice of one logits row once from HBM with
// 16-byte non-allocating loads and fold it into an online softmax state
//     m = max x,   a = first index of m,
//     S = sum 2^{y},  T = sum 2^{y} y,   y = (x - m) log2(e)
// so that for the whole row  H = ln S - ln2 * T / S  and  conf = p_a = 2^{y_a} / S.
// The state merges associatively (rescaling by 2^{(m' - m) log2 e}), so a row
// can be split across CTAs; warps merge with shuffles, the CTA through smem.
// Phase 2 (the last CTA of a row to finish, found with an atomic ticket — no
// CTA ever waits on another): merge the row's slices in a fixed order and write
// token / conf / entropy.
// Phase 3 (the last row of a sequence to finish): rank the sequence's rows by
// (confidence desc, position asc), take the first n_unmask, write them in rank
// order, E = max entropy over them, refresh = E > tau, and update the
// is_masked / token / decode-step state at their positions.
#include <float.h>
#include <limits.h>
#include <math.h>

#include "ec_internal.cuh"

namespace ec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;          // 16-byte vectors per thread per batch of loads
constexpr int kCtasPerSm = 4;       // resident CTAs per SM the grid is sized for
constexpr int kMaxSplits = 64;      // CTAs per row at most
constexpr int kMaxStagedRows = 2048;  // selection keys kept in smem up to this many rows
constexpr int kMaxUnmask = 1024;

struct __align__(16) Partial {
    float m;  // running maximum logit
    float s;  // sum 2^{(x - m) log2 e}
    float t;  // sum 2^{y} * y, y = (x - m) log2 e
    int idx;  // first index of the maximum
};

__device__ __forceinline__ Partial empty_partial()
{
    Partial p;
    p.m = -INFINITY;
    p.s = 0.f;
    p.t = 0.f;
    p.idx = INT_MAX;
    return p;
}

// a <- a (+) b.  The winner keeps the larger maximum (lower index on a tie).
__device__ __forceinline__ void merge(Partial &a, const Partial &b)
{
    if (b.s == 0.f) return;
    if (a.s == 0.f) {
        a = b;
        return;
    }
    const bool b_wins = b.m > a.m || (b.m == a.m && b.idx < a.idx);
    const Partial hi = b_wins ? b : a;
    const Partial lo = b_wins ? a : b;
    // The sums of a partial are relative to mb = fl(m * log2 e), the rounded value
    // its fold used; shifting between partials uses the same rounded values so the
    // merged sums stay exactly consistent with one reference point.
    const float d = lo.m * kLog2e - hi.m * kLog2e;  // <= 0
    const float f = ex2(d);
    a.m = hi.m;
    a.idx = hi.idx;
    a.s = fmaf(f, lo.s, hi.s);
    a.t = fmaf(f, fmaf(d, lo.s, lo.t), hi.t);
}

__device__ __forceinline__ Partial shfl_xor(const Partial &p, int off)
{
    Partial q;
    q.m = __shfl_xor_sync(0xffffffffu, p.m, off);
    q.s = __shfl_xor_sync(0xffffffffu, p.s, off);
    q.t = __shfl_xor_sync(0xffffffffu, p.t, off);
    q.idx = __shfl_xor_sync(0xffffffffu, p.idx, off);
    return q;
}

__device__ __forceinline__ void warp_merge(Partial &p)
{
#pragma unroll
    for (int off = 16; off; off >>= 1) merge(p, shfl_xor(p, off));
}

// ---- element types ----
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;
    static constexpr uint32_t kNegInfWord = 0xff800000u;
    __device__ static __forceinline__ void unpack(const uint4 &v, float *x)
    {
        x[0] = __uint_as_float(v.x);
        x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z);
        x[3] = __uint_as_float(v.w);
    }
    __device__ static __forceinline__ float scalar(const float *p) { return __ldg(p); }
};

// bfloat16 stored as raw uint16 bits; widening is a 16-bit shift.
template <>
struct Elem<uint16_t> {
    static constexpr int kPerVec = 8;
    static constexpr uint32_t kNegInfWord = 0xff80ff80u;
    __device__ static __forceinline__ void unpack(const uint4 &v, float *x)
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ float scalar(const uint16_t *p)
    {
        return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
    }
};

// Fold elements x[0..N) into (m, s0/s1, t0/t1, a); index_of(i) is the row index
// of x[i] (increasing in i), evaluated only when the maximum moves.
template <int N, typename IndexOf>
__device__ __forceinline__ void fold(const float (&x)[N], IndexOf index_of, float &m, float &s0,
                                     float &s1, float &t0, float &t1, int &a)
{
    float cm = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) cm = fmaxf(cm, x[i]);
    if (cm > m) {  // rare after the first batch: new maximum, rescale the sums
        int first = INT_MAX;
#pragma unroll
        for (int i = N - 1; i >= 0; --i)
            if (x[i] == cm) first = index_of(i);
        const float s = s0 + s1;
        if (s > 0.f) {
            const float d = m * kLog2e - cm * kLog2e;
            const float f = ex2(d);
            const float t = t0 + t1;
            t0 = f * fmaf(d, s, t);
            t1 = 0.f;
            s0 = f * s;
            s1 = 0.f;
        }
        m = cm;
        a = first;
    }
    const float mb = m * kLog2e;
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float y0 = fmaxf(fmaf(x[i], kLog2e, -mb), -1e30f);  // -inf logits -> weight 0
        const float e0 = ex2(y0);
        s0 += e0;
        t0 = fmaf(e0, y0, t0);
        if (i + 1 < N) {
            const float y1 = fmaxf(fmaf(x[i + 1], kLog2e, -mb), -1e30f);
            const float e1 = ex2(y1);
            s1 += e1;
            t1 = fmaf(e1, y1, t1);
        }
    }
}

struct Args {
    const void *logits;
    int64_t row_stride;
    int n_rows, vocab, splits;
    const int32_t *offsets, *row_pos;
    int batch, seq_len, n_unmask;
    float tau;
    int step;
    int32_t *token_out;
    float *conf_out, *entropy_out;
    int32_t *unmask_rows;
    float *max_entropy;
    uint8_t *refresh, *is_masked;
    int32_t *seq_tokens, *decode_step;
    uint32_t *status;
    unsigned *row_ctr, *seq_ctr;
    Partial *parts;
};

__device__ __forceinline__ unsigned long long select_key(float conf, int pos)
{
    // larger key = higher confidence, then lower position (conf > 0, so its bits order)
    return (static_cast<unsigned long long>(__float_as_uint(conf)) << 32) |
           static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(pos));
}

// Phase 3 for sequence b (whole CTA).
__device__ void finish_sequence(const Args &A, int b, int r0, int cnt)
{
    __shared__ unsigned long long s_key[kMaxStagedRows];
    __shared__ int s_sel[kMaxUnmask];
    __shared__ int s_nsel;
    __shared__ float s_wmax[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool staged = cnt <= kMaxStagedRows;
    if (staged)
        for (int i = tid; i < cnt; i += kThreads)
            s_key[i] = select_key(__ldcg(A.conf_out + r0 + i), __ldg(A.row_pos + r0 + i));
    __syncthreads();

    const int take = min(A.n_unmask, cnt);
    if (warp == 0) {
        unsigned long long prev = ~0ull;
        int nsel = 0;
        for (int s = 0; s < take; ++s) {
            unsigned long long best = 0ull;
            int bi = INT_MAX;
            for (int i = lane; i < cnt; i += 32) {
                const unsigned long long k =
                    staged ? s_key[i]
                           : select_key(__ldcg(A.conf_out + r0 + i), __ldg(A.row_pos + r0 + i));
                if (k < prev && k > best) {
                    best = k;
                    bi = i;
                }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                const unsigned long long ok = __shfl_xor_sync(0xffffffffu, best, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ok > best || (ok == best && oi < bi)) {
                    best = ok;
                    bi = oi;
                }
            }
            if (best == 0ull) break;  // only with duplicate positions (invalid input)
            if (lane == 0) s_sel[s] = bi;
            prev = best;
            ++nsel;
        }
        if (lane == 0) s_nsel = nsel;
    }
    __syncthreads();

    const int nsel = s_nsel;
    float h = -INFINITY;
    for (int s = tid; s < A.n_unmask; s += kThreads) {
        int32_t *slot = A.unmask_rows + static_cast<int64_t>(b) * A.n_unmask + s;
        if (s < nsel) {
            const int r = r0 + s_sel[s];
            h = fmaxf(h, __ldcg(A.entropy_out + r));
            const int tok = __ldcg(A.token_out + r);
            const int p = __ldg(A.row_pos + r);
            *slot = r;
            if (p >= 0 && p < A.seq_len) {
                const int64_t at = static_cast<int64_t>(b) * A.seq_len + p;
                A.is_masked[at] = 0;
                A.seq_tokens[at] = tok;
                A.decode_step[at] = A.step;
            }
        } else {
            *slot = -1;
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) h = fmaxf(h, __shfl_xor_sync(0xffffffffu, h, off));
    if (lane == 0) s_wmax[warp] = h;
    __syncthreads();
    if (tid == 0) {
        float e = s_wmax[0];
        for (int w = 1; w < kWarps; ++w) e = fmaxf(e, s_wmax[w]);
        A.max_entropy[b] = e;
        A.refresh[b] = e > A.tau ? 1 : 0;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_gate_kernel(const Args A)
{
    constexpr int E = Elem<T>::kPerVec;
    __shared__ Partial s_part[kWarps];
    __shared__ int s_seq, s_seq_lo, s_seq_cnt, s_row_last, s_seq_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // CTA 0 checks the offsets and finishes sequences that have no rows.
    if (blockIdx.x == 0) {
        for (int b = tid; b <= A.batch; b += kThreads) {
            const int o = __ldg(A.offsets + b);
            bool bad = (b == 0 && o != 0) || (b == A.batch && o != A.n_rows);
            if (b < A.batch) {
                const int o1 = __ldg(A.offsets + b + 1);
                bad |= o1 < o;
                if (o1 == o) {
                    for (int s = 0; s < A.n_unmask; ++s)
                        A.unmask_rows[static_cast<int64_t>(b) * A.n_unmask + s] = -1;
                    A.max_entropy[b] = -INFINITY;
                    A.refresh[b] = 0;
                }
            }
            if (bad) flag_status(A.status, EC_DEV_BAD_OFFSETS);
        }
    }
    if (A.n_rows == 0) return;

    const int row = blockIdx.x / A.splits;
    const int split = blockIdx.x - row * A.splits;

    // Which sequence owns this row (rows of a sequence are contiguous).
    if (tid == 0) s_seq = -1;
    __syncthreads();
    for (int b = tid; b < A.batch; b += kThreads) {
        const int o0 = __ldg(A.offsets + b), o1 = __ldg(A.offsets + b + 1);
        // only a well-formed range is trusted (keeps phase 3 inside [0, n_rows))
        if (o0 >= 0 && o1 <= A.n_rows && o0 <= row && row < o1) {
            atomicMax(&s_seq, b);
            s_seq_lo = o0;  // benign: only one b matches valid offsets
            s_seq_cnt = o1 - o0;
        }
    }

    // ---- phase 1: stream this CTA's slice of the row ----
    const T *row_ptr = static_cast<const T *>(A.logits) + static_cast<int64_t>(row) * A.row_stride;
    const int64_t nvec = A.vocab / E;
    const int64_t per = (nvec + A.splits - 1) / A.splits;
    const int64_t v0 = min(nvec, static_cast<int64_t>(split) * per);
    const int64_t v1 = min(nvec, v0 + per);
    const uint4 *vp = reinterpret_cast<const uint4 *>(row_ptr);

    float m = -INFINITY, s0 = 0.f, s1 = 0.f, t0 = 0.f, t1 = 0.f;
    int a = INT_MAX;
    for (int64_t base = v0 + tid; base < v1; base += kThreads * kUnroll) {
        uint4 raw[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = base + static_cast<int64_t>(u) * kThreads;
            const uint32_t w = Elem<T>::kNegInfWord;
            raw[u] = v < v1 ? ld_stream_v4(vp + v) : make_uint4(w, w, w, w);
        }
        float x[kUnroll * E];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) Elem<T>::unpack(raw[u], x + u * E);
        const int vb = static_cast<int>(base);
        fold(x, [vb](int i) { return (vb + (i / E) * kThreads) * E + (i % E); }, m, s0, s1, t0, t1, a);
    }
    // ragged tail (vocab % E elements) belongs to the last slice
    if (split == A.splits - 1) {
        const int tail0 = static_cast<int>(nvec * E);
        const int j = tail0 + tid;
        if (j < A.vocab) {
            float x[1] = {Elem<T>::scalar(row_ptr + j)};
            fold(x, [j](int) { return j; }, m, s0, s1, t0, t1, a);
        }
    }

    Partial p;
    p.m = m;
    p.s = s0 + s1;
    p.t = t0 + t1;
    p.idx = a;
    if (p.s == 0.f) p = empty_partial();
    warp_merge(p);
    if (lane == 0) s_part[warp] = p;
    __syncthreads();
    if (warp == 0) {
        p = lane < kWarps ? s_part[lane] : empty_partial();
        warp_merge(p);
    }

    // ---- phase 2: the last slice of the row to finish merges the slices ----
    if (A.splits > 1) {
        if (tid == 0) {
            __stcg(reinterpret_cast<float4 *>(A.parts + static_cast<int64_t>(row) * kMaxSplits + split),
                   make_float4(p.m, p.s, p.t, __int_as_float(p.idx)));
            __threadfence();
            const unsigned ticket = atomicInc(A.row_ctr + row, static_cast<unsigned>(A.splits - 1));
            s_row_last = ticket == static_cast<unsigned>(A.splits - 1);
        }
        __syncthreads();
        if (!s_row_last) return;
        __threadfence();
        if (warp == 0) {
            p = empty_partial();
            for (int i = lane; i < A.splits; i += 32) {
                const float4 q4 =
                    __ldcg(reinterpret_cast<const float4 *>(A.parts + static_cast<int64_t>(row) * kMaxSplits + i));
                Partial q;
                q.m = q4.x;
                q.s = q4.y;
                q.t = q4.z;
                q.idx = __float_as_int(q4.w);
                merge(p, q);
            }
            warp_merge(p);
        }
    }

    if (tid == 0) {
        // Sums are relative to mb = fl(m log2 e); for any reference point
        // H = ln S - ln2 * T / S, and the argmax's own term is 2^{m log2 e - mb}.
        const float S = p.s;
        const float H = logf(S) - kLn2 * (p.t / S);
        const float top = ex2(fmaf(p.m, kLog2e, -(p.m * kLog2e)));
        A.entropy_out[row] = fmaxf(H, 0.f);
        A.conf_out[row] = top / S;
        A.token_out[row] = p.idx;
        const int pos = __ldg(A.row_pos + row);
        if (pos < 0 || pos >= A.seq_len) flag_status(A.status, EC_DEV_BAD_ROW_POS);
        // ---- phase 3 ticket: is this the last row of its sequence? ----
        int last = 0;
        const int b = s_seq;
        if (b < 0) {
            flag_status(A.status, EC_DEV_BAD_OFFSETS);
        } else {
            __threadfence();
            const unsigned ticket = atomicInc(A.seq_ctr + b, static_cast<unsigned>(s_seq_cnt - 1));
            last = ticket == static_cast<unsigned>(s_seq_cnt - 1);
        }
        s_seq_last = last;
    }
    __syncthreads();
    if (!s_seq_last) return;
    __threadfence();
    finish_sequence(A, s_seq, s_seq_lo, s_seq_cnt);
}

}  // namespace

size_t decode_workspace_bytes(int32_t n_rows, int32_t batch)
{
    const size_t rows = n_rows > 0 ? static_cast<size_t>(n_rows) : 0;
    const size_t seqs = batch > 0 ? static_cast<size_t>(batch) : 0;
    size_t off = kWsHeader;
    off = align_up(off + rows * sizeof(unsigned), 16);
    off = align_up(off + seqs * sizeof(unsigned), 256);
    return off + rows * kMaxSplits * sizeof(Partial);
}

int decode_splits(int32_t n_rows, int32_t vocab, int elem_bytes)
{
    if (n_rows <= 0) return 1;
    const int64_t nvec = vocab / (16 / elem_bytes);
    const int slots = device_sm_count() * kCtasPerSm;
    int64_t s = slots / n_rows;
    s = std::min<int64_t>(s, nvec / (2 * kThreads));  // >= 2 vectors per thread per slice
    s = std::max<int64_t>(1, std::min<int64_t>(s, kMaxSplits));
    return static_cast<int>(s);
}

cudaError_t launch_decode_gate(const void *logits, int dtype, int64_t row_stride, int32_t n_rows,
                               int32_t vocab, const int32_t *seq_row_offsets,
                               const int32_t *row_pos, int32_t batch, int32_t seq_len,
                               int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                               float *conf_out, float *entropy_out, int32_t *unmask_rows,
                               float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                               int32_t *seq_tokens, int32_t *decode_step, void *workspace,
                               cudaStream_t stream)
{
    const int elem = dtype == EC_BF16 ? 2 : 4;
    Args A;
    A.logits = logits;
    A.row_stride = row_stride;
    A.n_rows = n_rows;
    A.vocab = vocab;
    A.splits = decode_splits(n_rows, vocab, elem);
    A.offsets = seq_row_offsets;
    A.row_pos = row_pos;
    A.batch = batch;
    A.seq_len = seq_len;
    A.n_unmask = n_unmask;
    A.tau = tau;
    A.step = step;
    A.token_out = token_out;
    A.conf_out = conf_out;
    A.entropy_out = entropy_out;
    A.unmask_rows = unmask_rows;
    A.max_entropy = max_entropy;
    A.refresh = refresh;
    A.is_masked = is_masked;
    A.seq_tokens = seq_tokens;
    A.decode_step = decode_step;
    char *ws = static_cast<char *>(workspace);
    A.status = reinterpret_cast<uint32_t *>(ws);
    size_t off = kWsHeader;
    A.row_ctr = reinterpret_cast<unsigned *>(ws + off);
    off = align_up(off + static_cast<size_t>(std::max(n_rows, 0)) * sizeof(unsigned), 16);
    A.seq_ctr = reinterpret_cast<unsigned *>(ws + off);
    off = align_up(off + static_cast<size_t>(batch) * sizeof(unsigned), 256);
    A.parts = reinterpret_cast<Partial *>(ws + off);

    const unsigned grid = n_rows > 0 ? static_cast<unsigned>(n_rows) * A.splits : 1u;
    if (dtype == EC_BF16)
        decode_gate_kernel<uint16_t><<<grid, kThreads, 0, stream>>>(A);
    else
        decode_gate_kernel<float><<<grid, kThreads, 0, stream>>>(A);
    return cudaGetLastError();
}

}  // namespace ec

// ---------------------------------------------------------------------------
// Allocation-free variant of ec_decode_step.
//
// For callers that cannot allocate device memory themselves (their device
// memory belongs to a host framework or a fixed pool, or a cudaMalloc, which
// may synchronise the device, is not acceptable in their decode loop).  The
// scratch that ec_decode_step takes as a workspace lives here in a fixed
// device array instead; every device that loads the library holds it until
// the process exits.

namespace ec {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
static cudaError_t decode_scratch_address(void **out)
{
    static void *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace ec

extern "C" ec_status ec_decode_step_noalloc(
    const void *logits, ec_dtype dtype, int64_t row_stride, int32_t n_rows, int32_t vocab,
    const int32_t *seq_row_offsets, const int32_t *row_pos, int32_t batch, int32_t seq_len,
    int32_t n_unmask, float tau, int32_t step, int32_t *token_out, float *conf_out,
    float *entropy_out, int32_t *unmask_rows, float *max_entropy, uint8_t *refresh,
    uint8_t *is_masked, int32_t *seq_tokens, int32_t *decode_step, ec_stream_t stream)
{
    if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_DTYPE;
    if (n_rows < 0 || vocab < 1 || batch < 1 || seq_len < 1 || n_unmask < 1 ||
        n_unmask > ec::kMaxUnmask || row_stride < vocab || !isfinite(tau))
        return EC_ERR_SHAPE;
    if (!seq_row_offsets || !unmask_rows || !max_entropy || !refresh || !is_masked ||
        !seq_tokens || !decode_step)
        return EC_ERR_NULL;
    if (n_rows > 0 && (!logits || !row_pos || !token_out || !conf_out || !entropy_out))
        return EC_ERR_NULL;
    const int elem = dtype == EC_BF16 ? 2 : 4;
    if (n_rows > 0 && ((reinterpret_cast<uintptr_t>(logits) & 15) != 0 ||
                       (row_stride * elem) % 16 != 0))
        return EC_ERR_ALIGN;
    const size_t need = ec::decode_workspace_bytes(n_rows, batch);
    if (need > ec::kNoAllocScratchBytes) return EC_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    if (ec::decode_scratch_address(&scratch) != cudaSuccess) return EC_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: clear the status word and the
    // tickets, which must start at zero (the per-slice partials need no clearing).
    const size_t zeroed = need - static_cast<size_t>(n_rows) * ec::kMaxSplits * sizeof(ec::Partial);
    if (cudaMemsetAsync(scratch, 0, zeroed, s) != cudaSuccess) return EC_ERR_CUDA;
    const cudaError_t e = ec::launch_decode_gate(
        logits, dtype, row_stride, n_rows, vocab, seq_row_offsets, row_pos, batch, seq_len,
        n_unmask, tau, step, token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
        is_masked, seq_tokens, decode_step, scratch, s);
    return e == cudaSuccess ? EC_OK : EC_ERR_CUDA;
}
