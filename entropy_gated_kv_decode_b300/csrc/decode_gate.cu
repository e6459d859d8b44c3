// Decode-and-gate step of EntropyCache: a streaming kernel and a finishing
// kernel, chained by programmatic dependent launch.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, "Algoritmo di Funzionamento" steps 1-2, and the
// Arabic technical summary, "Algorithm workflow" phases 2-3 with the equation
// E_{t+1} = max_{i in D_{t+1}} ( -sum_j p_ij log p_ij ).
//
// One pass over the logits folds every row into an online softmax state
//     m = max x,   S = sum 2^{y},  T = sum 2^{y} y,   y = x log2(e) - fl(m log2(e)),
// so that for the whole row  H = ln S - ln2 * T / S  and  conf = p_a = 2^{y_a} / S,
// a = the first index of m.  States merge associatively (rescaling by
// 2^{difference of the references}; on equal maxima the earlier index wins).
//
// Work split.  A row's 16-byte vectors form a head (about 95 %) and, for rows
// of 64 KB or more, a few tail chunks of at most 32 KB.  The heads of all rows,
// laid end to end, are cut into one equal contiguous range per CTA of a
// persistent grid (3 CTAs per SM); the tail chunks form a pool that CTAs claim
// from a global counter once their own range is done, so CTAs that streamed
// their range early take the remaining bytes and all finish together.  Every
// contiguous run of one row a CTA processes is a piece; a row's pieces fill
// fixed partial slots (its head pieces in CTA order, then its tail chunks), so
// the merge order, hence every result, is deterministic.
// Streaming kernel:
//   producer warp   one thread streams each piece into a ring of 16 KB stages
//                   with bulk asynchronous copies (evict-first in L2), a stage
//                   never crossing a row end, and writes a header per stage;
//   8 consumer warps each thread folds 4 contiguous vectors of every stage
//                   (64 bytes; read in a rotated order, free of bank conflicts)
//                   into its running state, which lives across the stages of a
//                   piece.  When the running maximum grows, the first index of
//                   the new maximum in the thread's batch is found at once.  At
//                   a piece end each warp reduces its lanes (maximum first, then
//                   rescaled sums) and hands its partial to the finisher;
//   finisher warp   merges the 8 warp partials of a piece into the piece's slot.
// Finishing kernel, one block per sequence: its rows' slots merged in parallel
// (token / conf / entropy written, ranking keys staged in shared memory), then
// one warp ranks the rows by (confidence desc, position asc), takes the first
// n_unmask, E = max entropy over them, refresh = E > tau, and updates
// is_masked / tokens / the decode-time log at their positions.  Finishing after
// the stream, all sequences at once, keeps the rows' last pieces, which all
// complete near the end of the stream, from queueing behind one another, and
// needs no ticket between blocks.
// The bf16 fold has no per-element guard for -inf: a -inf logit makes T NaN
// (0 * -inf), and the thread then refolds its share of that piece from global
// memory with -inf mapped to -1e30 (weight exactly 0), so rows without -inf pay
// nothing for the rare case.
// Every wait is bounded; a timeout sets EC_DEV_TIMEOUT and unwinds.
#include <float.h>
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "ec_internal.cuh"
#include "gate_common.cuh"
#include "tc_ptx.cuh"

namespace ec {
namespace {

using ptx::Sync;
using gate::Partial;
using gate::empty_partial;
using gate::merge;
using gate::shfl_xor;
using gate::shift;
using gate::ticket;
using gate::warp_merge;
using gate::warp_reduce;

constexpr int kConsumers = 256;              // 8 folding warps
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 64;    // + producer warp + finisher warp
constexpr int kCtasPerSm = 3;
constexpr uint32_t kStageBytes = 16384;      // bytes per ring stage
constexpr int kStages = 3;
constexpr int kVecPerStage = kStageBytes / 16;   // 1024 vectors
constexpr int kPieceSlots = 4;               // finished pieces queued for the finisher
constexpr int kMaxSplits = 64;               // partial slots per row
constexpr int kTailMinBytes = 65536;         // rows this long get a tail pool
constexpr int kTailPercent = 5;              // share of such a row in the pool
constexpr int kTailChunkVecs = 2048;         // 32 KB per pool chunk at most
constexpr int kMaxUnmask = gate::kMaxUnmask;
constexpr int kFinishThreads = 512;          // threads of a finishing block (one per sequence)

enum : int {
    D_FULL = 0,                        // [kStages] stage landed (and its header written)
    D_EMPTY = D_FULL + kStages,        // [kStages] stage read by every consumer warp
    D_PFULL = D_EMPTY + kStages,       // [kPieceSlots] the 8 warp partials of a piece written
    D_PEMPTY = D_PFULL + kPieceSlots,  // [kPieceSlots] the finisher took them
    D_COUNT = D_PEMPTY + kPieceSlots
};
constexpr uint32_t kSmemDyn = kStages * kStageBytes + 1024 + 8 * D_COUNT;  // ring + align + barriers

enum : int { H_FIRST = 1, H_TAIL = 2 };

// What a stage holds: vectors [v0, v0 + nv) of `row`.  The first stage of a
// piece also describes the piece: its slot, its end vector and whether it ends
// the row (then the vocab % per-vector elements after the last whole vector
// belong to it).  row < 0 marks the end of the CTA's work.
struct StageHdr {
    int row, v0, nv, flags, slot, pv1;
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

// One bf16 pair (element 2i in the low half) into the two-wide sums:
// y = x log2e - mb, e = 2^y, S += e, T += e y, in one block of f32x2 arithmetic.
__device__ __forceinline__ void fold_pair(uint32_t w, uint64_t l2e, uint64_t nmb, uint64_t &s2,
                                          uint64_t &t2)
{
    asm("{\n\t.reg .b32 lo, hi, e0, e1;\n\t.reg .b64 x2, y2, e2;\n\t"
        "shl.b32 lo, %2, 16;\n\tand.b32 hi, %2, 0xffff0000;\n\t"
        "mov.b64 x2, {lo, hi};\n\t"
        "fma.rn.f32x2 y2, x2, %3, %4;\n\t"
        "mov.b64 {lo, hi}, y2;\n\t"
        "ex2.approx.ftz.f32 e0, lo;\n\tex2.approx.ftz.f32 e1, hi;\n\t"
        "mov.b64 e2, {e0, e1};\n\t"
        "add.rn.f32x2 %0, %0, e2;\n\t"
        "fma.rn.f32x2 %1, e2, y2, %1;\n\t}"
        : "+l"(s2), "+l"(t2)
        : "r"(w), "l"(l2e), "l"(nmb));
}

// Running state of one thread over the batches of a piece.
struct Fold {
    float m;
    uint64_t s2, t2;  // two-wide sums (bf16 input)
    float s, t;       // scalar sums (float32 input, guarded elements)
    int a;
    __device__ __forceinline__ void reset()
    {
        m = -INFINITY;
        s2 = t2 = 0ull;
        s = t = 0.f;
        a = INT_MAX;
    }
    // A new maximum cm > everything folded so far, first seen in the 64-byte
    // batch starting at 16-byte vector `batch`: shift the sums to it.
    __device__ __forceinline__ void raise(float cm, int batch)
    {
        float s_lo, s_hi, t_lo, t_hi;
        unpack2(s2, s_lo, s_hi);
        unpack2(t2, t_lo, t_hi);
        const float ss = (s_lo + s_hi) + s;
        const float tt = (t_lo + t_hi) + t;
        s2 = t2 = 0ull;
        if (ss > 0.f) {
            const float d = gate::ref_gap(m, cm);
            const float f = shift(d);
            s = f * ss;
            t = f * fmaf(d, ss, tt);
        } else {
            s = t = 0.f;
        }
        m = cm;
        a = batch;
    }
    // One guarded element of the batch at vector `batch` (-inf has weight exactly 0).
    __device__ __forceinline__ void add_guarded(float x, int batch)
    {
        if (x > m) raise(x, batch);
        if (m == -INFINITY) return;
        const float y = fmaxf(fmaf(x, kLog2e, -(m * kLog2e)), -1e30f);
        const float e = ex2(y);
        s += e;
        t = fmaf(e, y, t);
    }
    // A batch of bf16 pairs (the thread's 64-byte batch starting at 16-byte
    // vector `batch`), the first nw of them valid (the others are -inf fill and
    // do not enter the sums).  No guard for -inf: see the file header.
    template <int N>
    __device__ __forceinline__ void add_bf16(const uint32_t (&w)[N], int nw, int batch)
    {
        uint32_t mw = w[0];
#pragma unroll
        for (int i = 1; i < N; ++i) mw = bf16x2_max(mw, w[i]);
        const float cm = fmaxf(__uint_as_float(mw << 16), __uint_as_float(mw & 0xffff0000u));
        if (cm > m) raise(cm, batch);
        if (m == -INFINITY) return;  // nothing but -inf so far: every weight is zero
        const float mb = m * kLog2e;
        const uint64_t l2e = pack2(kLog2e, kLog2e), nmb = pack2(-mb, -mb);
        if (nw == N) {
#pragma unroll
            for (int i = 0; i < N; ++i) fold_pair(w[i], l2e, nmb, s2, t2);
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i)
                if (i < nw) fold_pair(w[i], l2e, nmb, s2, t2);
        }
    }
    __device__ __forceinline__ Partial partial() const
    {
        float s_lo, s_hi, t_lo, t_hi;
        unpack2(s2, s_lo, s_hi);
        unpack2(t2, t_lo, t_hi);
        Partial p;
        p.m = m;
        p.s = (s_lo + s_hi) + s;
        p.t = (t_lo + t_hi) + t;
        p.a = a;
        if (!(p.s > 0.f)) p = empty_partial();
        return p;
    }
    __device__ __forceinline__ bool bad() const
    {
        float s_lo, s_hi, t_lo, t_hi;
        unpack2(s2, s_lo, s_hi);
        unpack2(t2, t_lo, t_hi);
        return isnan(((s_lo + s_hi) + (t_lo + t_hi)) + (s + t));
    }
};

// ---- element types: 16-byte vectors of 8 bf16 or 4 float32 ----
template <typename T>
struct Elem;
template <>
struct Elem<uint16_t> {
    static constexpr int kPerVec = 8;
    __device__ static __forceinline__ float at(const void *row, int64_t j)
    {
        return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const uint16_t *>(row) + j)) << 16);
    }
};
template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;
    __device__ static __forceinline__ float at(const void *row, int64_t j)
    {
        return __ldg(static_cast<const float *>(row) + j);
    }
};

struct Args {
    const void *logits;
    int64_t row_stride;  // elements
    int n_rows, vocab;
    int nvec;            // whole 16-byte vectors per row
    int tail;            // elements after them
    int head;            // vectors of a row in the static heads
    int n_tc;            // pool chunks per row (0: the whole row is head)
    int units;           // static units per row: head (+1 for the tail elements when n_tc == 0)
    int64_t total;       // n_rows * units
    int grid;
    gate::GateArgs g;    // outputs, decode state, sequences
    uint32_t *status;
    long long wait_limit;  // cycles one in-kernel wait may take
    unsigned *pool_ctr;  // [0] pool claims, [1] producers done
    Partial *parts;
};

// First static unit of CTA c's range, and the CTA whose range holds unit u.
__device__ __forceinline__ int64_t range_begin(const Args &A, int c)
{
    return static_cast<int64_t>(c) * A.total / A.grid;
}
__device__ __forceinline__ int cta_of(const Args &A, int64_t u)
{
    return static_cast<int>(((u + 1) * A.grid - 1) / A.total);
}
// Head pieces of row i (CTAs c0 .. c0 + n - 1, in CTA order); slots: those, then the tail chunks.
__device__ __forceinline__ int head_pieces(const Args &A, int i, int &c0)
{
    const int64_t base = static_cast<int64_t>(i) * A.units;
    c0 = cta_of(A, base);
    return cta_of(A, base + A.units - 1) - c0 + 1;
}
__device__ __forceinline__ int row_slots(const Args &A, int i)
{
    int c0;
    return head_pieces(A, i, c0) + A.n_tc;
}

template <typename T>
__device__ __forceinline__ const char *row_ptr(const Args &A, int i)
{
    return static_cast<const char *>(A.logits) + static_cast<int64_t>(i) * A.row_stride * sizeof(T);
}

// First index of the maximum M inside the 64-byte batch starting at 16-byte
// vector a (for a = nvec: among the elements after the last whole vector).
// Whole warp, one element per lane; elements past the vocabulary are not read.
template <typename T>
__device__ __forceinline__ int first_index_of(const Args &A, int row, int a, float M)
{
    constexpr int E = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int64_t j = static_cast<int64_t>(a) * E + lane;
    const bool hit = lane < 4 * E && j < A.vocab && Elem<T>::at(row_ptr<T>(A, row), j) == M;
    const unsigned mask = __ballot_sync(0xffffffffu, hit);
    return mask ? static_cast<int>(j - lane) + __ffs(mask) - 1 : a * E;
}

// ---- the consumer side ----
struct RingPos {
    int s;        // stage index
    uint32_t ph;  // its phase parity
    __device__ void next()
    {
        if (++s == kStages) {
            s = 0;
            ph ^= 1u;
        }
    }
};

struct PieceState {
    int row, slot, pv0, pv1, flags;
};

// The thread's 64-byte batch of a stage: vectors 4 tid + j, j = 0..3, read in
// the order j = (u + tid / 2) mod 4 so that each quarter-warp's 16-byte loads
// fall on distinct banks.  Returns how many of the 4 vectors are valid.
__device__ __forceinline__ int load_batch(const uint8_t *stage, int nv, uint32_t (&w)[16])
{
    const int tid = threadIdx.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(stage) + 4 * tid;
    const int nvalid = min(max(nv - 4 * tid, 0), 4);
    if (nvalid == 4) {
        // the order of the words inside the batch does not matter to the fold
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint4 v = src[(u + (tid >> 1)) & 3];
            w[4 * u] = v.x;
            w[4 * u + 1] = v.y;
            w[4 * u + 2] = v.z;
            w[4 * u + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = j < nvalid ? src[j] : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
        }
    }
    return nvalid;
}

// A thread's contribution to a piece, refolded from global memory with every
// element guarded (a -inf logit made the fast fold's T NaN).
template <typename T>
__device__ void refold_guarded(const Args &A, const PieceState &pc, Fold &f)
{
    constexpr int E = Elem<T>::kPerVec;
    const int tid = threadIdx.x;
    const char *row = row_ptr<T>(A, pc.row);
    f.reset();
    for (int v0 = pc.pv0; v0 < pc.pv1; v0 += kVecPerStage) {
        const int nv = min(kVecPerStage, pc.pv1 - v0);
        const int nvalid = min(max(nv - 4 * tid, 0), 4);
        const int batch = v0 + 4 * tid;
        for (int e = 0; e < nvalid * E; ++e)
            f.add_guarded(Elem<T>::at(row, static_cast<int64_t>(batch) * E + e), batch);
    }
}

// Folds the thread's batch of a float32 stage (guarded elements).
__device__ __forceinline__ void add_f32_batch(Fold &f, const uint32_t (&w)[16], int nvalid, int batch)
{
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (i < 4 * nvalid) cm = fmaxf(cm, __uint_as_float(w[i]));
    if (cm > f.m) f.raise(cm, batch);
    if (f.m == -INFINITY) return;
    const float mb = f.m * kLog2e;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (i < 4 * nvalid) {
            const float y = fmaxf(fmaf(__uint_as_float(w[i]), kLog2e, -mb), -1e30f);
            const float e = ex2(y);
            f.s += e;
            f.t = fmaf(e, y, f.t);
        }
}

// End of a piece: the row's last elements (when the piece ends the row), the
// guarded refold when -inf made the sums NaN, the warp reduction, and the
// hand-over of the warp partial (and, from warp 0, the piece) to the finisher.
template <typename T>
__device__ __forceinline__ bool end_piece(const Args &A, const Sync &S, const PieceState &pc, Fold &f,
                                          uint32_t &n_pieces, Partial (*s_piece)[kConsumerWarps],
                                          int2 *s_info)
{
    constexpr int E = Elem<T>::kPerVec;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (sizeof(T) == 2 && f.bad()) refold_guarded<T>(A, pc, f);
    if ((pc.flags & H_TAIL) && tid < A.tail)
        f.add_guarded(Elem<T>::at(row_ptr<T>(A, pc.row), static_cast<int64_t>(A.nvec) * E + tid),
                      A.nvec);
    const Partial p = warp_reduce(f.partial());
    const int slot = n_pieces % kPieceSlots;
    if (n_pieces >= static_cast<uint32_t>(kPieceSlots) &&
        !__all_sync(0xffffffffu, S.wait(D_PEMPTY + slot, ((n_pieces / kPieceSlots) - 1) & 1)))
        return false;
    if (lane == 0) {
        s_piece[slot][warp] = p;
        if (warp == 0) s_info[slot] = make_int2(pc.row, pc.slot);
        ptx::mbar_arrive(S.bar(D_PFULL + slot));  // release: the partial is visible
    }
    ++n_pieces;
    return true;
}

// Producer: the stages of one piece, vectors [pv0, pv1) of `row` (a piece with
// no whole vector, only the row's last elements, gets one empty stage).
template <typename T>
__device__ __forceinline__ bool issue_piece(const Args &A, const Sync &S, uint32_t ring_u32,
                                            StageHdr *hdr, uint32_t &it, int row, int pv0, int pv1,
                                            int slot, int flags)
{
    const char *base = row_ptr<T>(A, row);
    int v = pv0;
    bool first = true;
    do {
        const int nv = min(kVecPerStage, pv1 - v);
        const int s = it % kStages;
        if (it >= static_cast<uint32_t>(kStages) && !S.wait(D_EMPTY + s, ((it / kStages) - 1) & 1))
            return false;
        StageHdr h;
        h.row = row;
        h.v0 = v;
        h.nv = nv;
        h.flags = first ? (H_FIRST | flags) : 0;
        h.slot = slot;
        h.pv1 = pv1;
        hdr[s] = h;
        if (nv > 0) {
            const uint32_t bytes = static_cast<uint32_t>(nv) * 16u;
            ptx::mbar_expect_tx(S.bar(D_FULL + s), bytes);
            ptx::bulk_load_stream(ring_u32 + s * kStageBytes, base + static_cast<int64_t>(v) * 16, bytes,
                                  S.bar(D_FULL + s));
        } else {
            ptx::mbar_arrive(S.bar(D_FULL + s));
        }
        ++it;
        v += nv;
        first = false;
    } while (v < pv1);
    return true;
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
    __shared__ int2 s_info[kPieceSlots];
    __shared__ StageHdr s_hdr[kStages];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Sync S{ring_u32 + kStages * kStageBytes, reinterpret_cast<volatile int *>(&s_abort), A.status,
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

    if (warp == kConsumerWarps) {
        // ---- producer: this CTA's static range, then chunks of the pool ----
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            if (u_end > u_begin) {
                const int r_first = static_cast<int>(u_begin / A.units);
                const int r_last = static_cast<int>((u_end - 1) / A.units);
                for (int i = r_first; i <= r_last && ok; ++i) {
                    const int64_t base = static_cast<int64_t>(i) * A.units;
                    const int ua = static_cast<int>(max(u_begin, base) - base);
                    const int ub = static_cast<int>(min(u_end, base + A.units) - base);
                    const int c0 = cta_of(A, base);
                    const int flags = ub > A.head ? H_TAIL : 0;  // the unit after the head: last elements
                    ok = issue_piece<T>(A, S, ring_u32, s_hdr, it, i, ua, min(ub, A.head),
                                        static_cast<int>(blockIdx.x) - c0, flags);
                }
            }
            if (ok && A.n_tc > 0) {
                const unsigned n_pool = static_cast<unsigned>(A.n_rows) * static_cast<unsigned>(A.n_tc);
                unsigned next = atomicAdd(A.pool_ctr, 1u);
                while (ok && next < n_pool) {
                    const unsigned c = next;
                    next = atomicAdd(A.pool_ctr, 1u);  // the next claim travels while this one streams
                    const int i = static_cast<int>(c / A.n_tc), j = static_cast<int>(c % A.n_tc);
                    const int pv0 = A.head + j * kTailChunkVecs;
                    const int pv1 = min(A.nvec, pv0 + kTailChunkVecs);
                    int c0;
                    const int slot = head_pieces(A, i, c0) + j;
                    ok = issue_piece<T>(A, S, ring_u32, s_hdr, it, i, pv0, pv1, slot,
                                        (j == A.n_tc - 1 && A.tail > 0) ? H_TAIL : 0);
                }
                // the last producer to run out resets the pool for the next launch
                if (ok && ticket(A.pool_ctr + 1, static_cast<unsigned>(A.grid - 1)) ==
                              static_cast<unsigned>(A.grid - 1))
                    atomicExch(A.pool_ctr, 0u);
            }
            if (ok) {  // end marker
                const int s = it % kStages;
                if (it >= static_cast<uint32_t>(kStages)) ok = S.wait(D_EMPTY + s, ((it / kStages) - 1) & 1);
                if (ok) {
                    StageHdr h;
                    h.row = -1;
                    h.v0 = h.nv = h.flags = h.slot = h.pv1 = 0;
                    s_hdr[s] = h;
                    ptx::mbar_arrive(S.bar(D_FULL + s));
                    ++it;
                }
            }
            if (!ok)  // let every copy already started land before the CTA exits
                for (uint32_t u = (it > kStages ? it - kStages : 0); u < it; ++u)
                    S.drain(D_FULL + u % kStages, (u / kStages) & 1);
        }
        return;
    }

    if (warp == kConsumerWarps + 1) {
        // ---- finisher: the 8 warp partials of each piece merged into its slot ----
        for (uint32_t pc = 0;; ++pc) {
            const int slot = pc % kPieceSlots;
            if (!S.wait(D_PFULL + slot, (pc / kPieceSlots) & 1)) break;
            const int2 info = s_info[slot];
            Partial p = lane < kConsumerWarps ? s_piece[slot][lane] : empty_partial();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(S.bar(D_PEMPTY + slot));
            if (info.x < 0) break;  // the consumers' end marker
#pragma unroll
            for (int off = 4; off; off >>= 1) merge(p, shfl_xor(p, off));
            // the piece's maximum to its exact first index (the fold kept only
            // the 64-byte batch), off the consumers' path
            p = Partial{__shfl_sync(0xffffffffu, p.m, 0), __shfl_sync(0xffffffffu, p.s, 0),
                        __shfl_sync(0xffffffffu, p.t, 0), __shfl_sync(0xffffffffu, p.a, 0)};
            if (p.s > 0.f) p.a = first_index_of<T>(A, info.x, p.a, p.m);
            if (lane == 0)
                __stcg(reinterpret_cast<float4 *>(A.parts + static_cast<int64_t>(info.x) * kMaxSplits + info.y),
                       gate::to_f4(p));
        }
        return;
    }

    // ---- consumers: fold each stage; at every piece end hand the warp partial over ----
    RingPos rp{0, 0u};
    uint32_t n_pieces = 0;
    Fold f;
    f.reset();
    PieceState pc{-1, 0, 0, 0, 0};
    bool ok = true;
    for (;;) {
        const int s = rp.s;
        if (!__all_sync(0xffffffffu, S.wait(D_FULL + s, rp.ph))) {
            ok = false;
            break;
        }
        const StageHdr h = s_hdr[s];
        uint32_t w[16];
        int nvalid = 0;
        if (h.row >= 0) nvalid = load_batch(ring + s * kStageBytes, h.nv, w);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(S.bar(D_EMPTY + s));
        rp.next();
        if (h.row < 0 || (h.flags & H_FIRST)) {  // the previous piece is complete
            if (pc.row >= 0 && !end_piece<T>(A, S, pc, f, n_pieces, s_piece, s_info)) {
                ok = false;
                break;
            }
            if (h.row < 0) break;
            pc = PieceState{h.row, h.slot, h.v0, h.pv1, h.flags};
            f.reset();
        }
        if (nvalid > 0) {
            const int batch = h.v0 + 4 * tid;
            if constexpr (sizeof(T) == 2)
                f.add_bf16(w, 4 * nvalid, batch);
            else
                add_f32_batch(f, w, nvalid, batch);
        }
    }
    // The next kernel may become resident once every CTA has streamed its bytes:
    // triggered earlier, its CTAs would take SM slots this grid's CTAs still need.
    pdl_launch_dependents();
    if (ok) {  // end marker for the finisher (after a failure its wait gives up by itself)
        const int slot = n_pieces % kPieceSlots;
        if (n_pieces < static_cast<uint32_t>(kPieceSlots) ||
            __all_sync(0xffffffffu, S.wait(D_PEMPTY + slot, ((n_pieces / kPieceSlots) - 1) & 1))) {
            if (lane == 0) {
                if (warp == 0) s_info[slot] = make_int2(-1, 0);
                ptx::mbar_arrive(S.bar(D_PFULL + slot));
            }
        }
    }
}

// Second kernel, one block per sequence: groups of g lanes (g = 32 for short
// sequences, down to 1 for long ones) each merge one row's slots, write its
// token / conf / entropy and stage its ranking key in shared memory; then every
// row's rank is counted in parallel (one thread per row; sequences longer than
// the block are ranked by one warp, n_unmask selection rounds), the first
// n_unmask are unmasked, E = max entropy over them, refresh = E > tau, and the
// decode state is updated.  No block waits for another.  A stream kernel that gave up a wait left some slots unwritten: then
// nothing is finished (the status word reports the timeout).
__global__ void __launch_bounds__(kFinishThreads) decode_finish_kernel(const Args A)
{
    __shared__ gate::SeqStage st;
    const int b = static_cast<int>(blockIdx.x), tid = static_cast<int>(threadIdx.x);
    // The offsets, positions and slot counts are inputs, complete before the
    // streaming kernel began: read them while it still runs.
    const int lo = __ldg(A.g.offsets + b), hi = __ldg(A.g.offsets + b + 1);
    const bool seq_ok = !(lo < 0 || hi > A.n_rows || lo > hi);
    const int cnt = seq_ok ? hi - lo : 0;
    int g = 32;  // lanes per row: as many as the block holds for this sequence
    while (g > 1 && g * cnt > kFinishThreads) g >>= 1;
    const int j = tid % g;
    const int r_first = tid / g;
    const bool first_live = r_first < cnt;
    const int n_first = first_live ? row_slots(A, lo + r_first) : 0;
    const int pos_first = first_live ? __ldg(A.g.row_pos + lo + r_first) : 0;
    pdl_wait();  // the stream kernel's slots are complete and visible
    pdl_launch_dependents();
    // this lane's first slot of its first row travels with the status word (one
    // round trip for both); it is used only if no wait timed out
    const float4 *slots_first =
        reinterpret_cast<const float4 *>(A.parts + static_cast<int64_t>(lo + r_first) * kMaxSplits);
    float4 slot_first = make_float4(0.f, 0.f, 0.f, 0.f);
    if (seq_ok && first_live && j < n_first) slot_first = __ldcg(slots_first + j);
    if (ld_status(A.status) & EC_DEV_TIMEOUT) return;  // the whole block alike
    if (!seq_ok) {
        if (tid == 0) flag_status(A.status, EC_DEV_BAD_OFFSETS);
        return;
    }
    for (int r0 = 0; r0 < cnt; r0 += kFinishThreads / g) {
        const int r = r0 + r_first;
        const bool live = r < cnt;
        const int i = lo + r;
        Partial p = empty_partial();
        int pos = 0;
        if (live) {
            const float4 *slots =
                reinterpret_cast<const float4 *>(A.parts + static_cast<int64_t>(i) * kMaxSplits);
            const int n = r0 == 0 ? n_first : row_slots(A, i);
            pos = r0 == 0 ? pos_first : __ldg(A.g.row_pos + i);
            for (int k = j; k < n; k += g)
                merge(p, gate::from_f4(r0 == 0 && k == j ? slot_first : __ldcg(slots + k)));
        }
        for (int off = g >> 1; off; off >>= 1) merge(p, shfl_xor(p, off));
        if (live && j == 0) {
            float conf, entropy;
            const int token = p.s > 0.f ? p.a : 0;
            gate::store_row(A.g, i, p, token, conf, entropy);
            if (pos < 0 || pos >= A.g.seq_len) flag_status(A.status, EC_DEV_BAD_ROW_POS);
            if (r < gate::kMaxStagedRows) {
                st.key[r] = gate::select_key(conf, pos);
                st.ent[r] = entropy;
                st.tok[r] = token;
            }
        }
    }
    __syncthreads();  // every row's outputs written and staged
    if (cnt > kFinishThreads || cnt > gate::kMaxStagedRows) {
        if (tid < 32) gate::rank_and_gate(A.g, b, lo, cnt, st);
        return;
    }
    // Every row's rank by counting the rows ahead of it (confidence desc, then
    // position asc; equal keys, which only duplicate positions give, by row):
    // the n_unmask first are unmasked, in rank order.
    __shared__ int s_emax;  // max entropy of the unmasked rows, as bits (entropy >= 0)
    if (tid == 0) s_emax = INT_MIN;
    __syncthreads();
    const int take = min(A.g.n_unmask, cnt);
    if (tid < cnt) {
        const unsigned long long key = st.key[tid];
        int rank = 0;
        for (int q = 0; q < cnt; ++q) {
            const unsigned long long kq = st.key[q];
            rank += kq > key || (kq == key && q < tid);
        }
        if (rank < take) {
            const int r = lo + tid;
            const int p = static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
            A.g.unmask_rows[static_cast<int64_t>(b) * A.g.n_unmask + rank] = r;
            if (p >= 0 && p < A.g.seq_len) {
                const int64_t at = static_cast<int64_t>(b) * A.g.seq_len + p;
                A.g.is_masked[at] = 0;
                A.g.seq_tokens[at] = st.tok[tid];
                A.g.decode_step[at] = A.g.step;
            }
            atomicMax(&s_emax, __float_as_int(st.ent[tid]));
        }
    }
    for (int s2 = take + tid; s2 < A.g.n_unmask; s2 += kFinishThreads)
        A.g.unmask_rows[static_cast<int64_t>(b) * A.g.n_unmask + s2] = -1;
    __syncthreads();
    if (tid == 0) {
        const float h = take > 0 ? __int_as_float(s_emax) : -INFINITY;
        A.g.max_entropy[b] = h;
        A.g.refresh[b] = h > A.g.tau ? 1 : 0;
    }
}

}  // namespace

// Pool chunks per row of `nvec` 16-byte vectors and the row's head length.
static void row_split(int nvec, int *head, int *n_tc)
{
    if (static_cast<int64_t>(nvec) * 16 >= kTailMinBytes) {
        const int tail = static_cast<int>(static_cast<int64_t>(nvec) * kTailPercent / 100) / 4 * 4;
        *n_tc = (tail + kTailChunkVecs - 1) / kTailChunkVecs;
        *head = nvec - tail;
    } else {
        *n_tc = 0;
        *head = nvec;
    }
}

size_t decode_workspace_bytes(int32_t n_rows, int32_t batch)
{
    const size_t rows = n_rows > 0 ? static_cast<size_t>(n_rows) : 0;
    size_t off = kWsHeader;
    off = align_up(off + 2 * sizeof(unsigned), 256);  // pool claims, producers done
    return off + rows * kMaxSplits * sizeof(Partial);
}

size_t decode_workspace_zeroed_bytes(int32_t n_rows, int32_t batch)
{
    const size_t rows = n_rows > 0 ? static_cast<size_t>(n_rows) : 0;
    return decode_workspace_bytes(n_rows, batch) - rows * kMaxSplits * sizeof(Partial);
}

// CTAs of the persistent grid: kCtasPerSm per SM, fewer when there are fewer
// static units than that, and few enough that a row has at most kMaxSplits
// pieces (its head pieces and its pool chunks).
int decode_grid(int32_t n_rows, int64_t units, int n_tc)
{
    if (n_rows <= 0) return 1;
    int64_t g = static_cast<int64_t>(device_sm_count()) * kCtasPerSm;
    g = std::min<int64_t>(g, static_cast<int64_t>(n_rows) * (kMaxSplits - 2 - n_tc));
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
    A.tail = vocab - A.nvec * per_vec;
    row_split(A.nvec, &A.head, &A.n_tc);
    A.units = A.head + ((A.n_tc == 0 && A.tail > 0) ? 1 : 0);
    A.total = static_cast<int64_t>(n_rows) * A.units;
    A.grid = decode_grid(n_rows, A.units, A.n_tc);
    gate::GateArgs &g = A.g;
    g.offsets = seq_row_offsets;
    g.row_pos = row_pos;
    g.n_rows = n_rows;
    g.batch = batch;
    g.seq_len = seq_len;
    g.n_unmask = n_unmask;
    g.tau = tau;
    g.step = step;
    g.token_out = token_out;
    g.conf_out = conf_out;
    g.entropy_out = entropy_out;
    g.unmask_rows = unmask_rows;
    g.max_entropy = max_entropy;
    g.refresh = refresh;
    g.is_masked = is_masked;
    g.seq_tokens = seq_tokens;
    g.decode_step = decode_step;
    char *ws = static_cast<char *>(workspace);
    A.status = reinterpret_cast<uint32_t *>(ws);
    g.status = A.status;
    A.wait_limit = wait_limit_cycles();
    size_t off = kWsHeader;
    g.seq_ctr = nullptr;  // the finishing kernel takes a block per sequence: no tickets
    A.pool_ctr = reinterpret_cast<unsigned *>(ws + off);
    off = align_up(off + 2 * sizeof(unsigned), 256);
    A.parts = reinterpret_cast<Partial *>(ws + off);

    if (n_rows > 0) {
        const dim3 grid(static_cast<unsigned>(A.grid));
        const cudaError_t e =
            dtype == EC_BF16 ? launch(decode_gate_kernel<uint16_t>, grid, dim3(kThreads), kSmemDyn, stream, A)
                             : launch(decode_gate_kernel<float>, grid, dim3(kThreads), kSmemDyn, stream, A);
        if (e != cudaSuccess) return e;
    }
    return launch(decode_finish_kernel, dim3(static_cast<unsigned>(batch)), dim3(kFinishThreads), 0,
                  stream, A);
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
    // pool counters, which must start at zero (the partial slots are always
    // written before they are read).
    const size_t zeroed = ec::decode_workspace_zeroed_bytes(n_rows, batch);
    if (cudaMemsetAsync(scratch, 0, zeroed, s) != cudaSuccess) return EC_ERR_CUDA;
    const cudaError_t e = ec::launch_decode_gate(
        logits, dtype, row_stride, n_rows, vocab, seq_row_offsets, row_pos, batch, seq_len,
        n_unmask, tau, step, token_out, conf_out, entropy_out, unmask_rows, max_entropy, refresh,
        is_masked, seq_tokens, decode_step, scratch, s);
    return e == cudaSuccess ? EC_OK : EC_ERR_CUDA;
}

extern "C" ec_status ec_decode_noalloc_read_status(uint32_t *bits, ec_stream_t stream)
{
    if (!bits) return EC_ERR_NULL;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return EC_ERR_CUDA;
    uint32_t v = 0;
    // the status word is the first word of the scratch array; a copy from the
    // symbol allocates nothing
    if (cudaMemcpyFromSymbol(&v, ec::g_decode_scratch, sizeof v, 0, cudaMemcpyDeviceToHost) !=
        cudaSuccess)
        return EC_ERR_CUDA;
    *bits = v;
    return EC_OK;
}
