// The decode-and-gate finish shared by the kernels that fold logits rows: the
// online softmax state of a row slice and its associative merge, the row's
// outputs, and the sequence's confidence-ranked unmasking and entropy gate.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, "Algoritmo di Funzionamento" steps 1-2; Arabic
// technical summary, "Algorithm workflow" phases 2-3 and the equation
// E_{t+1} = max_{i in D_{t+1}} ( -sum_j p_ij log p_ij ).
//
// A slice of a row is folded into (m, S, T, a):
//     m = max x,  S = sum 2^{y},  T = sum 2^{y} y,  y = x log2(e) - fl(m log2(e)),
// a = where the maximum first occurs (its meaning is up to the kernel: an
// element index, or the 64-byte batch holding it).  For the whole row
//     H = ln S - ln2 T / S,   conf = p_argmax = 2^{m log2 e - fl(m log2 e)} / S.
#pragma once

#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "ec_internal.cuh"

namespace ec {
namespace gate {

constexpr int kMaxStagedRows = 1024;  // ranking keys kept in shared memory up to this many rows
constexpr int kMaxUnmask = 1024;

struct __align__(16) Partial {
    float m;  // maximum logit
    float s;  // sum 2^{y},  y = x log2 e - fl(m log2 e)
    float t;  // sum 2^{y} y
    int a;    // where the maximum first occurs
};

// 2^d for the shift between two references (d <= 0); exactly 1 when they are
// equal (the approximate exp2 need not return 1 for 0, and the sums of the
// partial holding the maximum must not move).
__device__ __forceinline__ float shift(float d) { return d == 0.f ? 1.f : ex2(d); }

// fl(lo log2 e) - fl(hi log2 e): the gap between two partials' reference points.
// Both products are rounded on their own (never contracted into one fma), so
// the gap is exactly 0 when the maxima are equal and the shift is exactly 1.
__device__ __forceinline__ float ref_gap(float lo, float hi)
{
    return __fmul_rn(lo, kLog2e) - __fmul_rn(hi, kLog2e);
}

__device__ __forceinline__ Partial empty_partial()
{
    Partial p;
    p.m = -INFINITY;
    p.s = 0.f;
    p.t = 0.f;
    p.a = INT_MAX;
    return p;
}

// a <- a (+) b.  The larger maximum wins (the earlier position on a tie).  The
// sums of a partial are relative to fl(m log2 e), the rounded value its fold
// used; shifting between partials uses the same rounded values, so the merged
// sums stay consistent with one reference point.
__device__ __forceinline__ void merge(Partial &a, const Partial &b)
{
    if (b.s == 0.f) return;
    if (a.s == 0.f) {
        a = b;
        return;
    }
    const bool b_wins = b.m > a.m || (b.m == a.m && b.a < a.a);
    const Partial hi = b_wins ? b : a;
    const Partial lo = b_wins ? a : b;
    const float d = ref_gap(lo.m, hi.m);  // <= 0
    const float f = shift(d);
    a.m = hi.m;
    a.a = hi.a;
    a.s = fmaf(f, lo.s, hi.s);
    a.t = fmaf(f, fmaf(d, lo.s, lo.t), hi.t);
}

__device__ __forceinline__ Partial shfl_xor(const Partial &p, int off)
{
    Partial q;
    q.m = __shfl_xor_sync(0xffffffffu, p.m, off);
    q.s = __shfl_xor_sync(0xffffffffu, p.s, off);
    q.t = __shfl_xor_sync(0xffffffffu, p.t, off);
    q.a = __shfl_xor_sync(0xffffffffu, p.a, off);
    return q;
}

__device__ __forceinline__ Partial shfl(const Partial &p, int src)
{
    Partial q;
    q.m = __shfl_sync(0xffffffffu, p.m, src);
    q.s = __shfl_sync(0xffffffffu, p.s, src);
    q.t = __shfl_sync(0xffffffffu, p.t, src);
    q.a = __shfl_sync(0xffffffffu, p.a, src);
    return q;
}

// Every lane ends with the merge of all 32 lanes' partials.
__device__ __forceinline__ void warp_merge(Partial &p)
{
#pragma unroll
    for (int off = 16; off; off >>= 1) merge(p, shfl_xor(p, off));
}

// Reduce the lanes' states to one: the warp maximum first, then every lane's
// sums shifted to it and added (no pairwise merges), and the earliest position
// among the lanes holding the maximum.  Every lane gets the result.
__device__ __forceinline__ Partial warp_reduce(const Partial &p)
{
    float M = p.m;
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float s = 0.f, t = 0.f;
    int a = INT_MAX;
    if (p.s > 0.f) {
        const float d = ref_gap(p.m, M);
        const float f = shift(d);
        s = f * p.s;
        t = f * fmaf(d, p.s, p.t);
        if (p.m == M) a = p.a;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, off);
        t += __shfl_xor_sync(0xffffffffu, t, off);
        a = min(a, __shfl_xor_sync(0xffffffffu, a, off));
    }
    Partial r;
    r.m = M;
    r.s = s;
    r.t = t;
    r.a = a;
    if (s == 0.f) r = empty_partial();
    return r;
}

__device__ __forceinline__ float4 to_f4(const Partial &p)
{
    return make_float4(p.m, p.s, p.t, __int_as_float(p.a));
}
__device__ __forceinline__ Partial from_f4(const float4 &v)
{
    Partial p;
    p.m = v.x;
    p.s = v.y;
    p.t = v.z;
    p.a = __float_as_int(v.w);
    return p;
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

// The outputs and decode state one step writes, and its sequence layout.
struct GateArgs {
    const int32_t *offsets, *row_pos;  // [batch + 1], [n_rows]
    int n_rows, batch, seq_len, n_unmask;
    float tau;
    int step;
    int32_t *token_out;
    float *conf_out, *entropy_out;
    int32_t *unmask_rows;
    float *max_entropy;
    uint8_t *refresh, *is_masked;
    int32_t *seq_tokens, *decode_step;
    uint32_t *status;
    unsigned *seq_ctr;  // [batch] rows of the sequence finished (wraps to 0)
};

__device__ __forceinline__ unsigned long long select_key(float conf, int pos)
{
    // larger key = higher confidence, then lower position (conf > 0, so its bits order)
    return (static_cast<unsigned long long>(__float_as_uint(conf)) << 32) |
           static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(pos));
}

// The sequence holding row i (rows of a sequence are contiguous), or -1 when the
// offsets do not place it in a well-formed range.  Whole warp: a 32-way search
// (one load per lane per round), the same answer in every lane.
__device__ __forceinline__ int sequence_of(const GateArgs &A, int i, int &lo, int &cnt)
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

// The ranking's view of a sequence's rows in shared memory (rows beyond
// kMaxStagedRows are read from the outputs in global memory instead).
struct SeqStage {
    unsigned long long key[kMaxStagedRows];
    float ent[kMaxStagedRows];
    int tok[kMaxStagedRows];
    int sel[kMaxUnmask];
};

// Stages sequence rows [r0, r0 + cnt) from the outputs in global memory, by one
// warp: every row's confidence, position, entropy and token in one round trip.
__device__ __forceinline__ void stage_sequence(const GateArgs &A, int r0, int cnt, SeqStage &st)
{
    const int lane = threadIdx.x & 31;
    if (cnt > kMaxStagedRows) return;
    for (int i0 = 0; i0 < cnt; i0 += 32 * 8) {  // eight rows per lane per round
        float cf[8], en[8];
        int ps[8], tk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * 32 + lane;
            cf[u] = i < cnt ? __ldcg(A.conf_out + r0 + i) : 0.f;
            en[u] = i < cnt ? __ldcg(A.entropy_out + r0 + i) : 0.f;
            tk[u] = i < cnt ? __ldcg(A.token_out + r0 + i) : 0;
            ps[u] = i < cnt ? __ldg(A.row_pos + r0 + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * 32 + lane;
            if (i < cnt) {
                st.key[i] = select_key(cf[u], ps[u]);
                st.ent[i] = en[u];
                st.tok[i] = tk[u];
            }
        }
    }
    __syncwarp();
}

// Rank, gate and state update for sequence b (rows [r0, r0 + cnt), staged in
// `st` when cnt <= kMaxStagedRows), by one warp.  A sequence with no rows gets
// no unmasked rows, E = -inf and no refresh.
__device__ __forceinline__ void rank_and_gate(const GateArgs &A, int b, int r0, int cnt, SeqStage &st)
{
    const int lane = threadIdx.x & 31;
    const bool staged = cnt <= kMaxStagedRows;
    const int take = min(A.n_unmask, cnt);
    unsigned long long prev = ~0ull;
    int nsel = 0;
    for (int s = 0; s < take; ++s) {
        unsigned long long best = 0ull;
        int bi = INT_MAX;
        for (int i = lane; i < cnt; i += 32) {
            const unsigned long long k =
                staged ? st.key[i]
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
        if (lane == 0) st.sel[s] = bi;
        prev = best;
        ++nsel;
    }
    __syncwarp();
    // the selected rows' state updates and the maximum entropy, lanes in parallel
    float h = -INFINITY;
    for (int s = lane; s < A.n_unmask; s += 32) {
        int32_t *slot = A.unmask_rows + static_cast<int64_t>(b) * A.n_unmask + s;
        if (s < nsel) {
            const int i = st.sel[s];
            const int r = r0 + i;
            h = fmaxf(h, staged ? st.ent[i] : __ldcg(A.entropy_out + r));
            const int tok = staged ? st.tok[i] : __ldcg(A.token_out + r);
            const int p = staged ? static_cast<int>(0xffffffffu - static_cast<uint32_t>(st.key[i]))
                                 : __ldg(A.row_pos + r);
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
    __syncwarp();  // the staged arrays are reused by the next call
}

// Stage, then rank and gate, sequence b from the rows' outputs in global memory.
__device__ __forceinline__ void finish_sequence(const GateArgs &A, int b, int r0, int cnt, SeqStage &st)
{
    stage_sequence(A, r0, cnt, st);
    rank_and_gate(A, b, r0, cnt, st);
}

// The outputs of row i from its merged state p: entropy, confidence and token.
__device__ __forceinline__ void store_row(const GateArgs &A, int i, const Partial &p, int token,
                                          float &conf, float &entropy)
{
    // Sums are relative to mb = fl(m log2 e); for any reference point
    // H = ln S - ln2 * T / S, and the argmax's own term is 2^{m log2 e - mb}.
    const float S = p.s;
    const float H = logf(S) - kLn2 * (p.t / S);
    const float top = ex2(fmaf(p.m, kLog2e, -(p.m * kLog2e)));
    entropy = fmaxf(H, 0.f);
    conf = top / S;
    __stcg(A.entropy_out + i, entropy);
    __stcg(A.conf_out + i, conf);
    __stcg(A.token_out + i, token);
}

// One thread, row i from its merged state p: the outputs, the row-position
// check and the sequence ticket.  Returns the sequence when this row was its
// last to finish (the caller then runs finish_sequence with a whole warp), else
// -1.  The sequence is found by a binary search over the offsets.
__device__ __forceinline__ int row_outputs(const GateArgs &A, int i, const Partial &p, int token,
                                           int &lo, int &cnt)
{
    int a = 0, z = A.batch;  // the last b in [a, z) with offsets[b] <= i
    while (z - a > 1) {
        const int mid = (a + z) / 2;
        if (__ldg(A.offsets + mid) <= i)
            a = mid;
        else
            z = mid;
    }
    const int o0 = __ldg(A.offsets + a), o1 = __ldg(A.offsets + a + 1);
    const bool ok = !(o0 < 0 || o1 > A.n_rows || o0 > i || i >= o1);
    float conf, entropy;
    store_row(A, i, p, token, conf, entropy);
    const int pos = __ldg(A.row_pos + i);
    if (pos < 0 || pos >= A.seq_len) flag_status(A.status, EC_DEV_BAD_ROW_POS);
    if (!ok) {
        flag_status(A.status, EC_DEV_BAD_OFFSETS);
        return -1;
    }
    lo = o0;
    cnt = o1 - o0;
    return ticket(A.seq_ctr + a, static_cast<unsigned>(cnt - 1)) == static_cast<unsigned>(cnt - 1)
               ? a
               : -1;
}

// Sequences without rows (CTA 0 at the start of a step): nothing unmasked,
// E = -inf, no refresh; malformed offsets are flagged.  Whole warp.
__device__ __forceinline__ void empty_sequences(const GateArgs &A)
{
    const int lane = threadIdx.x & 31;
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

}  // namespace gate
}  // namespace ec
