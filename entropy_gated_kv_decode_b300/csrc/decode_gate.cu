// Decode-and-gate step of EntropyCache in one kernel launch.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, "Algoritmo di Funzionamento" steps 1-2, and the
// Arabic technical summary, "Algorithm workflow" phases 2-3 with the equation
// E_{t+1} = max_{i in D_{t+1}} ( -sum_j p_ij log p_ij ).
//
// One pass over the logits folds every row into an online softmax state
//     m = max x,   a = first index of m,
//     S = sum 2^{y},  T = sum 2^{y} y,   y = (x - m) log2(e)
// so that for the whole row  H = ln S - ln2 * T / S  and  conf = p_a = 2^{y_a} / S.
// The state merges associatively (rescaling by 2^{(m' - m) log2 e}).
//
// Work split: the rows' 16-byte vectors (plus, per row, one "tail" unit holding
// the vocab % 8 (bf16) or % 4 (fp32) last elements) are laid end to end and cut
// into one contiguous, equal range per CTA of a persistent grid, so every CTA
// streams the same number of bytes whatever the row count.  A range covers
// pieces of one or more rows.
//   producer warp   one thread streams the range's bytes into a ring of
//                   shared-memory stages with bulk asynchronous copies (TMA,
//                   evict-first in L2), completing on mbarriers;
//   8 consumer warps fold each stage from shared memory, one 16-byte vector per
//                   thread at a time, and reduce a row piece to one partial
//                   state (warp shuffles, then shared memory);
//   row merge       each partial goes to the workspace slot (row, CTA); the last
//                   CTA of a row to finish (an atomic ticket — no CTA waits on
//                   another) merges the row's partials in slot order and writes
//                   token / conf / entropy;
//   sequence        the last row of a sequence to finish ranks the sequence's
//                   rows by (confidence desc, position asc), takes the first
//                   n_unmask, writes them in rank order, E = max entropy over
//                   them, refresh = E > tau, and updates the is_masked / token /
//                   decode-step state at their positions.
// Every wait is bounded (~2 s); a timeout sets EC_DEV_TIMEOUT and unwinds.
#include <float.h>
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "ec_internal.cuh"
#include "tc_ptx.cuh"

namespace ec {
namespace {

using ptx::Sync;

constexpr int kConsumers = 256;              // 8 folding warps
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 64;    // + producer warp + finisher warp
constexpr int kCtasPerSm = 3;
constexpr uint32_t kChunk = 16384;           // bytes per ring stage
constexpr int kStages = 3;
constexpr int kVecPerChunk = kChunk / 16;
constexpr int kVecPerThread = kVecPerChunk / kConsumers;  // 4
constexpr int kPieceSlots = 4;               // finished row pieces queued for the finisher
constexpr int kMaxSplits = 64;               // partial slots per row
constexpr int kMaxStagedRows = 1024;         // selection keys kept in smem up to this many rows
constexpr int kMaxUnmask = 1024;

enum : int {
    D_FULL = 0,                        // [kStages] stage landed
    D_EMPTY = D_FULL + kStages,        // [kStages] stage read by every consumer warp
    D_PFULL = D_EMPTY + kStages,       // [kPieceSlots] the 8 warp partials of a piece written
    D_PEMPTY = D_PFULL + kPieceSlots,  // [kPieceSlots] the finisher took them
    D_COUNT = D_PEMPTY + kPieceSlots
};
constexpr uint32_t kSmemDyn = kStages * kChunk + 1024 + 8 * D_COUNT;  // ring + align slack + barriers

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

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Running fold state of one thread (scalar sums for fp32 input, two-wide sums
// s2 / t2 for bf16 input; a partial adds both).
struct Fold {
    float m, s0, s1, t0, t1;
    uint64_t s2, t2;
    int a;
    __device__ void reset()
    {
        m = -INFINITY;
        s0 = s1 = t0 = t1 = 0.f;
        s2 = t2 = 0ull;
        a = INT_MAX;
    }
    // Fold elements x[0..N) with row indices index_of(i) (increasing in i;
    // evaluated only when the maximum moves).  Elements equal to -inf get weight 0.
    template <int N, typename IndexOf>
    __device__ __forceinline__ void add(const float (&x)[N], IndexOf index_of)
    {
        float cm = x[0];
#pragma unroll
        for (int i = 1; i < N; ++i) cm = fmaxf(cm, x[i]);
        if (cm > m) {  // rare after the first elements: new maximum, rescale the sums
            int first = INT_MAX;
#pragma unroll
            for (int i = N - 1; i >= 0; --i)
                if (x[i] == cm) first = index_of(i);
            float s_lo, s_hi, t_lo, t_hi;
            unpack2(s2, s_lo, s_hi);
            unpack2(t2, t_lo, t_hi);
            const float s = (s0 + s1) + (s_lo + s_hi);
            const float t = (t0 + t1) + (t_lo + t_hi);
            s1 = t1 = 0.f;
            s2 = t2 = 0ull;
            if (s > 0.f) {
                const float d = m * kLog2e - cm * kLog2e;
                const float f = ex2(d);
                t0 = f * fmaf(d, s, t);
                s0 = f * s;
            } else {
                s0 = t0 = 0.f;
            }
            m = cm;
            a = first;
        }
        const float mb = m * kLog2e;
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float y0 = fmaxf(fmaf(x[i], kLog2e, -mb), -1e30f);
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
    // bf16 words w[0..N) (element 2i in the low half of w[i], 2i+1 in the high
    // half), row index of element k = index_of(k).  Two-wide math: the batch
    // maximum on packed bf16 pairs, the exponent argument, S and T with f32x2
    // FMA / add.  -inf elements are clamped to -1e30 (an unsigned 16-bit minimum
    // on the bit patterns) only after a finite maximum exists, so their weights
    // 2^{(x - m) log2 e} underflow to exact zeros.
    template <int N, typename IndexOf>
    __device__ __forceinline__ void add_bf16(const uint32_t (&w)[N], IndexOf index_of)
    {
        uint32_t mw = w[0];
#pragma unroll
        for (int i = 1; i < N; ++i) mw = bf16x2_max(mw, w[i]);
        const float cm = fmaxf(__uint_as_float(mw << 16), __uint_as_float(mw & 0xffff0000u));
        if (cm > m) {  // rare after the first elements: new maximum, rescale the sums
            int first = INT_MAX;
#pragma unroll
            for (int i = N - 1; i >= 0; --i) {
                if (__uint_as_float(w[i] & 0xffff0000u) == cm) first = index_of(2 * i + 1);
                if (__uint_as_float(w[i] << 16) == cm) first = index_of(2 * i);
            }
            float s_lo, s_hi, t_lo, t_hi;
            unpack2(s2, s_lo, s_hi);
            unpack2(t2, t_lo, t_hi);
            const float s = s0 + s1 + s_lo + s_hi;
            float t = t0 + t1 + t_lo + t_hi;
            s0 = s1 = t0 = t1 = 0.f;
            if (s > 0.f) {
                const float d = m * kLog2e - cm * kLog2e;
                const float fct = ex2(d);
                t = fct * fmaf(d, s, t);
                s2 = pack2(fct * s, 0.f);
                t2 = pack2(t, 0.f);
            } else {
                s2 = t2 = 0ull;
            }
            m = cm;
            a = first;
        }
        if (m == -INFINITY) return;  // nothing but -inf so far: every weight is zero
        const float mb = m * kLog2e;
        const uint64_t l2e = pack2(kLog2e, kLog2e), nmb = pack2(-mb, -mb);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const uint32_t c = __vminu2(w[i], 0xf14af14au);  // -inf (0xff80) -> -1e30 (0xf14a)
            const uint64_t y2 = ffma2(pack2(__uint_as_float(c << 16), __uint_as_float(c & 0xffff0000u)),
                                      l2e, nmb);
            float y0, y1;
            unpack2(y2, y0, y1);
            const uint64_t e2 = pack2(ex2(y0), ex2(y1));
            s2 = fadd2(s2, e2);
            t2 = ffma2(e2, y2, t2);
        }
    }
    __device__ Partial partial() const
    {
        float s_lo, s_hi, t_lo, t_hi;
        unpack2(s2, s_lo, s_hi);
        unpack2(t2, t_lo, t_hi);
        Partial p;
        p.m = m;
        p.s = (s0 + s1) + (s_lo + s_hi);
        p.t = (t0 + t1) + (t_lo + t_hi);
        p.idx = a;
        if (p.s == 0.f) p = empty_partial();
        return p;
    }
};

struct Args {
    const void *logits;
    int64_t row_stride;  // elements
    int n_rows, vocab;
    int64_t nvec;        // whole 16-byte vectors per row
    int tail;            // elements after them
    int64_t units;       // per row: nvec + (tail > 0)
    int64_t total;       // n_rows * units
    int grid;
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
    long long wait_limit;  // cycles one in-kernel wait may take
    unsigned *row_ctr, *seq_ctr;
    Partial *parts;
};

// A piece: units [ua, ub) of row `row`, its partial slot (the row's pieces in CTA
// order) and the row's number of pieces.
struct Piece {
    int row;
    int64_t ua, ub;
    int slot, n_contrib;
};

// First unit of CTA c's range, and the CTA whose range holds unit u.
__device__ __forceinline__ int64_t range_begin(const Args &A, int c)
{
    return static_cast<int64_t>(c) * A.total / A.grid;
}
__device__ __forceinline__ int cta_of(const Args &A, int64_t u)
{
    return static_cast<int>(((u + 1) * A.grid - 1) / A.total);
}

// This CTA's piece of row i (its range [u_begin, u_end) meets the row).
__device__ __forceinline__ Piece row_piece(const Args &A, int i, int64_t u_begin, int64_t u_end)
{
    Piece p;
    const int64_t base = static_cast<int64_t>(i) * A.units;
    p.row = i;
    p.ua = max(u_begin, base) - base;
    p.ub = min(u_end, base + A.units) - base;
    const int c0 = cta_of(A, base);
    p.slot = static_cast<int>(blockIdx.x) - c0;
    p.n_contrib = cta_of(A, base + A.units - 1) - c0 + 1;
    return p;
}

__device__ __forceinline__ unsigned long long select_key(float conf, int pos)
{
    // larger key = higher confidence, then lower position (conf > 0, so its bits order)
    return (static_cast<unsigned long long>(__float_as_uint(conf)) << 32) |
           static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(pos));
}

// The sequence holding row i (rows of a sequence are contiguous), or -1 when the
// offsets do not place it in a well-formed range.  Whole warp: a 32-way search
// (one load per lane per round), the same answer in every lane.
__device__ int sequence_of(const Args &A, int i, int &lo, int &cnt)
{
    const int lane = threadIdx.x & 31;
    int a = 0, z = A.batch;  // the answer is the last b in [a, z) with offsets[b] <= i
    while (z - a > 1) {
        const int step = (z - a + 31) / 32;
        const int b = a + lane * step;
        const bool le = b < z && __ldg(A.offsets + b) <= i;
        const unsigned mask = __ballot_sync(0xffffffffu, le);
        const int k = mask ? 31 - __clz(static_cast<int>(mask)) : 0;
        a = a + k * step;
        z = min(z, a + step);
    }
    const int o0 = __ldg(A.offsets + a), o1 = __ldg(A.offsets + a + 1);
    if (o0 < 0 || o1 > A.n_rows || o0 > i || i >= o1) return -1;
    lo = o0;
    cnt = o1 - o0;
    return a;
}

// Ticket with release (publishes this thread's earlier writes) and acquire (the
// last taker sees every earlier taker's writes) at GPU scope; wraps to 0 after
// `last`, so the counter is ready for the next launch.
__device__ __forceinline__ unsigned ticket(unsigned *ctr, unsigned last)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(ctr), "r"(last)
                 : "memory");
    return old;
}

// Rank, gate and state update for sequence b, by one warp.
__device__ void finish_sequence(const Args &A, int b, int r0, int cnt)
{
    __shared__ unsigned long long s_key[kMaxStagedRows];
    __shared__ int s_sel[kMaxUnmask];
    const int lane = threadIdx.x & 31;
    const bool staged = cnt <= kMaxStagedRows;
    if (staged)  // eight rows per lane per round, every load issued before any is used
        for (int i0 = 0; i0 < cnt; i0 += 32 * 8) {
            float cf[8];
            int ps[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * 32 + lane;
                cf[u] = i < cnt ? __ldcg(A.conf_out + r0 + i) : 0.f;
                ps[u] = i < cnt ? __ldg(A.row_pos + r0 + i) : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * 32 + lane;
                if (i < cnt) s_key[i] = select_key(cf[u], ps[u]);
            }
        }
    __syncwarp();

    const int take = min(A.n_unmask, cnt);
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
    __syncwarp();
    // the selected rows' state updates and the maximum entropy, lanes in parallel
    float h = -INFINITY;
    for (int s = lane; s < A.n_unmask; s += 32) {
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
    if (lane == 0) {
        A.max_entropy[b] = h;
        A.refresh[b] = h > A.tau ? 1 : 0;
    }
    __syncwarp();  // s_key / s_sel are reused by the next call
}

// Finisher warp: for one finished piece (its CTA partial p, in every lane):
// publish it; the row's last contributor merges all of them and writes
// token / conf / entropy; the sequence's last row ranks and gates.
__device__ void finish_piece(const Args &A, const Piece &pc, Partial p)
{
    const int lane = threadIdx.x & 31;
    const int i = pc.row, n_contrib = pc.n_contrib, slot = pc.slot;
    int last = 1;
    if (n_contrib > 1) {
        if (lane == 0) {
            __stcg(reinterpret_cast<float4 *>(A.parts + static_cast<int64_t>(i) * kMaxSplits + slot),
                   make_float4(p.m, p.s, p.t, __int_as_float(p.idx)));
            last = ticket(A.row_ctr + i, static_cast<unsigned>(n_contrib - 1)) ==
                   static_cast<unsigned>(n_contrib - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) return;
        // the last contributor merges every slot in order
        p = empty_partial();
        for (int k = lane; k < n_contrib; k += 32) {
            const float4 q4 = __ldcg(
                reinterpret_cast<const float4 *>(A.parts + static_cast<int64_t>(i) * kMaxSplits + k));
            Partial q;
            q.m = q4.x;
            q.s = q4.y;
            q.t = q4.z;
            q.idx = __float_as_int(q4.w);
            merge(p, q);
        }
        warp_merge(p);
    }
    int lo = 0, cnt = 0, last_row = 0;
    const int b = sequence_of(A, i, lo, cnt);
    if (lane == 0) {
        // Sums are relative to mb = fl(m log2 e); for any reference point
        // H = ln S - ln2 * T / S, and the argmax's own term is 2^{m log2 e - mb}.
        const float S = p.s;
        const float H = logf(S) - kLn2 * (p.t / S);
        const float top = ex2(fmaf(p.m, kLog2e, -(p.m * kLog2e)));
        __stcg(A.entropy_out + i, fmaxf(H, 0.f));
        __stcg(A.conf_out + i, top / S);
        __stcg(A.token_out + i, p.idx);
        if (b < 0)
            flag_status(A.status, EC_DEV_BAD_OFFSETS);
        else
            last_row = ticket(A.seq_ctr + b, static_cast<unsigned>(cnt - 1)) ==
                       static_cast<unsigned>(cnt - 1);
    } else if (lane == 1) {
        const int pos = __ldg(A.row_pos + i);
        if (pos < 0 || pos >= A.seq_len) flag_status(A.status, EC_DEV_BAD_ROW_POS);
    }
    last_row = __shfl_sync(0xffffffffu, last_row, 0);
    if (!last_row) return;
    finish_sequence(A, b, lo, cnt);
}

// A consumer warp's partial of a piece (and, from warp 0, the piece itself) into
// the finisher's queue; a piece with row -1 tells the finisher that no more come.
__device__ __forceinline__ bool hand_over(const Sync &S, const Piece &pc, const Partial &p,
                                          uint32_t &n_pieces, Partial (*s_piece)[kConsumerWarps],
                                          Piece *s_info)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = n_pieces % kPieceSlots;
    if (n_pieces >= static_cast<uint32_t>(kPieceSlots) &&
        !__all_sync(0xffffffffu, S.wait(D_PEMPTY + slot, ((n_pieces / kPieceSlots) - 1) & 1)))
        return false;
    if (lane == 0) {
        s_piece[slot][warp] = p;
        if (warp == 0) s_info[slot] = pc;
        ptx::mbar_arrive(S.bar(D_PFULL + slot));  // release: the partial is visible
    }
    ++n_pieces;
    return true;
}

// Consumer side of one piece: fold its stages (and the tail unit when the piece
// ends the row) into the thread's state and hand the block's partial to the
// finisher.  Returns false after a failed wait.
struct RingPos {
    int s;         // stage index
    uint32_t ph;   // its phase parity
    __device__ void next()
    {
        if (++s == kStages) {
            s = 0;
            ph ^= 1u;
        }
    }
};

template <typename T>
__device__ bool fold_piece(const Args &A, const Sync &S, const uint8_t *ring, const Piece &pc,
                           RingPos &rp, uint32_t &n_pieces, Partial (*s_piece)[kConsumerWarps],
                           Piece *s_info)
{
    constexpr int E = Elem<T>::kPerVec;
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t vb = min(pc.ub, A.nvec);
    Fold f;
    f.reset();
    for (int64_t v = pc.ua; v < vb; v += kVecPerChunk, rp.next()) {
        const int s = rp.s;
        if (!__all_sync(0xffffffffu, S.wait(D_FULL + s, rp.ph))) return false;
        const uint4 *src = reinterpret_cast<const uint4 *>(ring + s * kChunk) + tid;
        uint4 raw[kVecPerThread];
        if (vb - v >= kVecPerChunk) {  // a full stage
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u) raw[u] = src[u * kConsumers];
        } else {
            const int nv = static_cast<int>(vb - v) - tid;
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u) {
                const uint32_t ni = Elem<T>::kNegInfWord;
                raw[u] = u * kConsumers < nv ? src[u * kConsumers] : make_uint4(ni, ni, ni, ni);
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(S.bar(D_EMPTY + s));
        const int vb0 = static_cast<int>(v) + tid;
        if constexpr (sizeof(T) == 2) {
            uint32_t wv[kVecPerThread * 4];
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u) {
                wv[4 * u] = raw[u].x;
                wv[4 * u + 1] = raw[u].y;
                wv[4 * u + 2] = raw[u].z;
                wv[4 * u + 3] = raw[u].w;
            }
            f.add_bf16(wv, [vb0](int k) { return (vb0 + (k / E) * kConsumers) * E + (k % E); });
        } else {
            float x[kVecPerThread * E];
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u) Elem<T>::unpack(raw[u], x + u * E);
            f.add(x, [vb0](int k) { return (vb0 + (k / E) * kConsumers) * E + (k % E); });
        }
    }
    // the tail unit (vocab % E last elements) belongs to the piece ending the row
    if (A.tail > 0 && pc.ub == A.units && tid < A.tail) {
        const int j = static_cast<int>(A.nvec * E) + tid;
        const T *row = static_cast<const T *>(A.logits) + static_cast<int64_t>(pc.row) * A.row_stride;
        float x[1] = {Elem<T>::scalar(row + j)};
        f.add(x, [j](int) { return j; });
    }
    Partial p = f.partial();
    warp_merge(p);
    return hand_over(S, pc, p, n_pieces, s_piece, s_info);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_gate_kernel(const Args A)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t ring_u32 = ptx::smem_u32(ring);
    __shared__ int s_abort;
    __shared__ Partial s_piece[kPieceSlots][kConsumerWarps];
    __shared__ Piece s_info[kPieceSlots];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Sync S{ring_u32 + kStages * kChunk, reinterpret_cast<volatile int *>(&s_abort), A.status,
           A.wait_limit};

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < D_COUNT; ++i) {
            uint32_t n = 1;
            if ((i >= D_EMPTY && i < D_EMPTY + kStages) || (i >= D_PFULL && i < D_PFULL + kPieceSlots))
                n = kConsumerWarps;
            ptx::mbar_init(S.bar(i), n);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // inputs and outputs belong to the previous kernel until here

    const int64_t u_begin = A.total ? range_begin(A, blockIdx.x) : 0;
    const int64_t u_end = A.total ? range_begin(A, blockIdx.x + 1) : 0;
    const int64_t su = A.units > 0 ? A.units : 1;
    const int row_first = static_cast<int>(u_begin / su);
    const int row_last = u_end > u_begin ? static_cast<int>((u_end - 1) / su) : row_first - 1;

    if (warp == kConsumerWarps) {
        // ---- producer: one thread streams the vector part of every piece ----
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int i = row_first; i <= row_last && ok; ++i) {
                const Piece pc = row_piece(A, i, u_begin, u_end);
                const char *row = static_cast<const char *>(A.logits) +
                                  static_cast<int64_t>(i) * A.row_stride * sizeof(T);
                const int64_t vb = min(pc.ub, A.nvec);
                for (int64_t v = pc.ua; v < vb && ok; v += kVecPerChunk, ++it) {
                    const int s = it % kStages;
                    if (it >= static_cast<uint32_t>(kStages))
                        ok = S.wait(D_EMPTY + s, ((it / kStages) - 1) & 1);
                    if (!ok) break;
                    const uint32_t bytes = static_cast<uint32_t>(std::min<int64_t>(kVecPerChunk, vb - v) * 16);
                    ptx::mbar_expect_tx(S.bar(D_FULL + s), bytes);
                    ptx::bulk_load_stream(ring_u32 + s * kChunk, row + v * 16, bytes, S.bar(D_FULL + s));
                }
            }
            if (!ok)  // let every copy already started land before the CTA exits
                for (uint32_t u = (it > kStages ? it - kStages : 0); u < it; ++u)
                    S.drain(D_FULL + u % kStages, (u / kStages) & 1);
        }
        return;
    }

    if (warp == kConsumerWarps + 1) {
        // ---- finisher: empty sequences (CTA 0), then every piece of this CTA ----
        if (blockIdx.x == 0) {
            for (int b = lane; b <= A.batch; b += 32) {
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
        for (uint32_t pc = 0;; ++pc) {
            const int slot = pc % kPieceSlots;
            if (!S.wait(D_PFULL + slot, (pc / kPieceSlots) & 1)) break;
            const Piece piece = s_info[slot];
            Partial p = lane < kConsumerWarps ? s_piece[slot][lane] : empty_partial();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(S.bar(D_PEMPTY + slot));
            if (piece.row < 0) break;  // the consumers' end marker
            warp_merge(p);
            finish_piece(A, piece, p);
        }
        return;
    }

    // ---- consumers: fold each stage, hand every finished piece to the finisher ----
    RingPos rp{0, 0u};
    uint32_t n_pieces = 0;
    bool ok = true;
    for (int i = row_first; i <= row_last && ok; ++i)
        ok = fold_piece<T>(A, S, ring, row_piece(A, i, u_begin, u_end), rp, n_pieces, s_piece,
                           s_info);
    // The next kernel may become resident once every CTA has streamed its bytes:
    // triggered earlier, its CTAs would take SM slots this grid's CTAs still need.
    pdl_launch_dependents();
    if (ok) {  // after a failure the finisher's wait gives up by itself
        Piece end;
        end.row = -1;
        end.ua = end.ub = 0;
        end.slot = end.n_contrib = 0;
        hand_over(S, end, empty_partial(), n_pieces, s_piece, s_info);
    }
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

// CTAs of the persistent grid: kCtasPerSm per SM, fewer when there are fewer
// units than that, and few enough that a row is split over at most
// kMaxSplits - 2 ranges (its partial slots).
int decode_grid(int32_t n_rows, int64_t units)
{
    if (n_rows <= 0) return 1;
    int64_t g = static_cast<int64_t>(device_sm_count()) * kCtasPerSm;
    g = std::min<int64_t>(g, static_cast<int64_t>(n_rows) * (kMaxSplits - 2));
    g = std::min<int64_t>(g, static_cast<int64_t>(n_rows) * units);
    return static_cast<int>(std::max<int64_t>(1, g));
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
    const int per_vec = 16 / elem;
    Args A;
    A.logits = logits;
    A.row_stride = row_stride;
    A.n_rows = n_rows;
    A.vocab = vocab;
    A.nvec = vocab / per_vec;
    A.tail = vocab - static_cast<int>(A.nvec) * per_vec;
    A.units = A.nvec + (A.tail > 0 ? 1 : 0);
    A.total = static_cast<int64_t>(n_rows) * A.units;
    A.grid = decode_grid(n_rows, A.units);
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
    A.wait_limit = wait_limit_cycles();
    size_t off = kWsHeader;
    A.row_ctr = reinterpret_cast<unsigned *>(ws + off);
    off = align_up(off + static_cast<size_t>(std::max(n_rows, 0)) * sizeof(unsigned), 16);
    A.seq_ctr = reinterpret_cast<unsigned *>(ws + off);
    off = align_up(off + static_cast<size_t>(batch) * sizeof(unsigned), 256);
    A.parts = reinterpret_cast<Partial *>(ws + off);

    const dim3 grid(static_cast<unsigned>(A.grid));
    if (dtype == EC_BF16)
        return launch(decode_gate_kernel<uint16_t>, grid, dim3(kThreads), kSmemDyn, stream, A);
    return launch(decode_gate_kernel<float>, grid, dim3(kThreads), kSmemDyn, stream, A);
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
