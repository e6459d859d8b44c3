// Selective-recompute bidirectional attention on the 5th-generation tensor
// cores (tcgen05 + TMEM), fed by TMA, with the KV write-back in the same call.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, section "1. Il Problema" (dLLM attention is
// bidirectional) and "Algoritmo di Funzionamento" step 2 (the partial forward
// recomputes K/V only for the selected tokens; the cache supplies the rest).
//
// Up to three launches, chained by programmatic dependent launch (PDL):
//   write_back_kernel   copies every fresh K/V row into the caches and at once
//                       lets the attention grid start;
//   attention_tc_kernel allocates TMEM, sets up its barriers and loads its first
//                       Q tile while the write-back runs, and waits for it
//                       (griddepcontrol.wait) only before its first K/V load;
//   merge_kernel        (only when some unit is split over several CTAs)
//                       combines the split units' partials into the output.
//
// Attention kernel: persistent, one CTA per SM.
//   units      up to 128 query rows of one (sequence b, KV head g): the
//              (recomputed row r, head h of g's group) pairs packed r-major, so
//              a GQA group shares each K/V tile.
//   pieces     the units' 128-key tiles are laid end to end and cut into one
//              equal contiguous range per CTA (stream-K), so every CTA does the
//              same number of tiles.  A range covers pieces of one or more
//              units.  A piece that is a whole unit writes its output directly;
//              otherwise it stores a partial (O, m, l) and moves on: no CTA
//              waits for another, and the merge kernel, spread over the whole
//              GPU, combines the partials afterwards.
//   warp 0     producer of Q (one tile per piece) and K tiles, warp 6 producer
//              of V tiles: TMA, 128-byte swizzle, rings of stages; a K stage is
//              released when its QK product completes, a V stage when its PV
//              product does;
//   warp 1     TMEM allocation; Q into TMEM (tcgen05.cp) and S = Q K^T into one
//              of two TMEM S buffers (tcgen05.mma) once the PV product that read
//              that buffer's P has completed;
//   warp 7     O += P V into the TMEM O accumulator: a second issuing thread, so
//              the next tile's QK never queues behind this tile's PV;
//   warps 2-5  one thread per query row: online softmax in the log2 domain on S
//              read by tcgen05.ld (the reference maximum moves only when it
//              grows by more than 8 in log2 units, rescaling O in TMEM when it
//              does), P as bf16 over the first half of the same S buffer (the
//              PV product takes its A operand from there), and the epilogue.
//              With P in its own S buffer the softmax never waits for the
//              previous tile's PV product, except to rescale O.
// Every wait is bounded (~2 s); a timeout sets EC_DEV_TIMEOUT and unwinds.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "ec_internal.cuh"
#include "tc_ptx.cuh"

namespace ec {
namespace {

using namespace ptx;

constexpr int kBlockM = 128;   // query rows per unit = TMEM lanes
constexpr int kBlockN = 128;   // keys per tile
constexpr int kThreads = 256;  // 8 warps
constexpr int kMaxContrib = 64;  // pieces a unit may be cut into

template <int D>
struct Cfg {
    static constexpr uint32_t kTile = kBlockM * D * 2;  // bytes of one Q / K / V tile
    static constexpr uint32_t kCol = kBlockM * 128;     // one 64-element column: 16 KB
    // stage counts at D = 128: 1 Q + 3 K + 3 V tiles fill 224 KB
    static constexpr int kQBufs = D == 128 ? 1 : 2;
    static constexpr int kKStages = D == 128 ? 3 : 4;
    static constexpr int kVStages = D == 128 ? 3 : 4;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kQBufs * kTile;
    static constexpr uint32_t kOffV = kOffK + kKStages * kTile;
    static constexpr uint32_t kOffBar = kOffV + kVStages * kTile;
    static constexpr uint32_t kOffMisc = kOffBar + 256;
    static constexpr uint32_t kBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t kTmemCols = 512;
    // two S buffers, columns [0, 128) and [128, 256); P (bf16 pairs) of a tile
    // overwrites the first 64 columns of its own S buffer
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = 256;  // O: columns [256, 256 + D)
    static constexpr uint32_t kColQ = 448;  // Q (bf16 pairs): columns [448, 448 + D / 2)
};

enum : int {
    B_KFULL = 0,    // [4] K tile landed
    B_KEMPTY = 4,   // [4] K stage consumed (its QK done)
    B_VFULL = 8,    // [4] V tile landed
    B_VEMPTY = 12,  // [4] V stage consumed (its PV done)
    B_QFULL = 16,   // [2] Q tile landed
    B_QEMPTY = 18,  // [2] Q tile copied into TMEM
    B_SFULL = 20,   // [2] S buffer written by its QK product
    B_PFULL = 22,   // [2] P written over its S buffer (and O corrected): 4 softmax warps
    B_SFREE = 24,   // [2] the PV product that read the buffer's P completed (O updated)
    B_DRAIN = 26,   // QK issuer's products all complete
    B_DRAIN2 = 27,  // PV issuer's products all complete
    B_COUNT = 28
};

struct Params {
    const __nv_bfloat16 *k_new, *v_new;
    __nv_bfloat16 *k_cache, *v_cache, *out;
    const int32_t *idx;
    int64_t idx_stride;
    const int32_t *count;
    int B, L, r_max, H, Hkv, G;
    int tok_per_tile;  // recomputed rows per unit: floor(128 / G)
    int n_mt;          // units per (b, g)
    int n_units, n_tiles, grid;
    int64_t total;     // n_units * n_tiles
    int slots;         // partial slots per unit (most pieces a unit is cut into)
    int n_split;       // > 0: split-major items (see piece_at); 0: stream-K ranges
    float scale_log2;
    uint32_t *status;   // workspace status word
    long long wait_limit;  // cycles one in-kernel wait may take
    float2 *part_ml;    // [n_units][slots][128] (m, l), m in raw score units
    float4 *part_o;     // [n_units][slots][D / 4][128] unnormalised O
};

// A piece: tiles [t0, t1) of one unit, processed by this CTA.
struct Piece {
    int unit, b, g, mt, t0, t1, cnt, slot, n_contrib;
};

__device__ __forceinline__ int64_t range_begin(const Params &P, int c)
{
    return static_cast<int64_t>(c) * P.total / P.grid;
}
__device__ __forceinline__ int cta_of(const Params &P, int64_t w)
{
    return static_cast<int>(((w + 1) * P.grid - 1) / P.total);
}

// The pieces of CTA blockIdx.x, in order.
//   stream-K (n_split == 0): the units' tiles laid end to end, one equal
//     contiguous range per CTA; the pieces are the units that range meets.
//   split-major items (n_split > 0): item i = ((b, g, split), mt) with mt
//     varying fastest is tiles [split * n_tiles / n_split, ...) of unit
//     (b, g, mt); items are dealt round-robin.  The CTAs working on the row
//     tiles of one KV head then read the same K/V tiles at the same time, so
//     each tile comes from HBM once and from L2 for the others (used when the
//     caches do not fit in L2).
struct Range {
    int64_t w0, w1;
    int u_first, count;
};
__device__ __forceinline__ Range my_range(const Params &P)
{
    Range r;
    if (P.n_split > 0) {
        const int n_items = P.n_units * P.n_split;
        r.w0 = r.w1 = 0;
        r.u_first = 0;
        r.count = static_cast<int>(blockIdx.x) < n_items
                      ? (n_items - 1 - static_cast<int>(blockIdx.x)) / P.grid + 1
                      : 0;
        return r;
    }
    r.w0 = range_begin(P, blockIdx.x);
    r.w1 = range_begin(P, blockIdx.x + 1);
    r.u_first = static_cast<int>(r.w0 / P.n_tiles);
    r.count = r.w1 > r.w0 ? static_cast<int>((r.w1 - 1) / P.n_tiles) - r.u_first + 1 : 0;
    return r;
}

__device__ __forceinline__ Piece piece_at(const Params &P, const Range &r, int k)
{
    Piece p;
    if (P.n_split > 0) {
        const int i = static_cast<int>(blockIdx.x) + k * P.grid;
        p.mt = i % P.n_mt;
        const int split = (i / P.n_mt) % P.n_split;
        const int bg = i / (P.n_mt * P.n_split);
        p.unit = bg * P.n_mt + p.mt;
        p.g = bg % P.Hkv;
        p.b = bg / P.Hkv;
        p.t0 = static_cast<int>(static_cast<int64_t>(P.n_tiles) * split / P.n_split);
        p.t1 = static_cast<int>(static_cast<int64_t>(P.n_tiles) * (split + 1) / P.n_split);
        p.slot = split;
        p.n_contrib = P.n_split;
    } else {
        const int u = r.u_first + k;
        p.unit = u;
        p.mt = u % P.n_mt;
        p.g = (u / P.n_mt) % P.Hkv;
        p.b = u / (P.n_mt * P.Hkv);
        const int64_t base = static_cast<int64_t>(u) * P.n_tiles;
        p.t0 = static_cast<int>(max(r.w0, base) - base);
        p.t1 = static_cast<int>(min(r.w1, base + P.n_tiles) - base);
        const int c0 = cta_of(P, base), c1 = cta_of(P, base + P.n_tiles - 1);
        p.slot = static_cast<int>(blockIdx.x) - c0;
        p.n_contrib = c1 - c0 + 1;
    }
    p.cnt = max(0, min(__ldg(P.count + p.b), P.r_max));
    return p;
}

// Units with no recomputed rows (mt beyond the sequence's count) are skipped by
// every role alike.
__device__ __forceinline__ bool piece_active(const Params &P, const Piece &p)
{
    return p.mt * P.tok_per_tile < p.cnt && p.t1 > p.t0;
}

static_assert(Cfg<128>::kColS + 2 * kBlockN <= Cfg<128>::kColO, "TMEM columns overlap");
static_assert(Cfg<128>::kColO + 128 <= Cfg<128>::kColQ, "TMEM columns overlap");
static_assert(Cfg<128>::kColQ + 128 / 2 <= Cfg<128>::kTmemCols, "TMEM columns overflow");
static_assert(Cfg<128>::kBytes <= 227 * 1024 && Cfg<64>::kBytes <= 227 * 1024, "shared memory");

// Q and K producer (one thread): per piece its Q tile, then its K tiles.
template <int D>
__device__ void producer_qk(const Params &P, const Sync &S, uint32_t sbase, const CUtensorMap *tm_q,
                            const CUtensorMap *tm_k)
{
    using C = Cfg<D>;
    const uint32_t q_bytes = static_cast<uint32_t>(P.tok_per_tile * P.G) * D * 2;
    const Range r = my_range(P);
    uint32_t T = 0, it = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        const int qb = it % C::kQBufs;
        if (it >= static_cast<uint32_t>(C::kQBufs))
            ok = S.wait(B_QEMPTY + qb, ((it / C::kQBufs) - 1) & 1);
        if (!ok) break;
        const uint32_t qdst = sbase + C::kOffQ + qb * C::kTile;
        mbar_expect_tx(S.bar(B_QFULL + qb), q_bytes);
        for (int c = 0; c < D / 64; ++c)
            tma_load_4d(qdst + c * C::kCol, tm_q, S.bar(B_QFULL + qb), c * 64, w.g * P.G,
                        w.mt * P.tok_per_tile, w.b);
        ++it;
        for (int t = w.t0; t < w.t1 && ok; ++t, ++T) {
            const int s = T % C::kKStages;
            if (T >= static_cast<uint32_t>(C::kKStages))
                ok = S.wait(B_KEMPTY + s, ((T / C::kKStages) - 1) & 1);
            if (!ok) break;
            const uint32_t kdst = sbase + C::kOffK + s * C::kTile;
            mbar_expect_tx(S.bar(B_KFULL + s), C::kTile);
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(kdst + c * C::kCol, tm_k, S.bar(B_KFULL + s), c * 64, w.g, t * kBlockN,
                            w.b);
        }
    }
    if (!ok) {  // let every copy this thread started land before the CTA exits
        for (uint32_t u = (T > C::kKStages ? T - C::kKStages : 0); u < T; ++u)
            S.drain(B_KFULL + u % C::kKStages, (u / C::kKStages) & 1);
        for (uint32_t u = (it > C::kQBufs ? it - C::kQBufs : 0); u < it; ++u)
            S.drain(B_QFULL + u % C::kQBufs, (u / C::kQBufs) & 1);
    }
}

// V producer (one thread): the V tiles of every piece, in the same order.
template <int D>
__device__ void producer_v(const Params &P, const Sync &S, uint32_t sbase, const CUtensorMap *tm_v)
{
    using C = Cfg<D>;
    const Range r = my_range(P);
    uint32_t T = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        for (int t = w.t0; t < w.t1 && ok; ++t, ++T) {
            const int s = T % C::kVStages;
            if (T >= static_cast<uint32_t>(C::kVStages))
                ok = S.wait(B_VEMPTY + s, ((T / C::kVStages) - 1) & 1);
            if (!ok) break;
            const uint32_t vdst = sbase + C::kOffV + s * C::kTile;
            mbar_expect_tx(S.bar(B_VFULL + s), C::kTile);
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(vdst + c * C::kCol, tm_v, S.bar(B_VFULL + s), c * 64, w.g, t * kBlockN,
                            w.b);
        }
    }
    if (!ok)
        for (uint32_t u = (T > C::kVStages ? T - C::kVStages : 0); u < T; ++u)
            S.drain(B_VFULL + u % C::kVStages, (u / C::kVStages) & 1);
}

// QK issuer (one thread): per piece Q into TMEM, then S = Q K^T for each tile
// into one of the two S buffers as soon as its K tile landed and the PV product
// of the tile two back (which read its P from that buffer) completed.  The next
// tile's scores are then ready while the softmax warps still work on this one.
template <int D>
__device__ void qk_issuer(const Params &P, const Sync &S, uint32_t sbase, uint32_t tmem)
{
    using C = Cfg<D>;
    constexpr uint32_t kIdescQK = idesc_bf16(kBlockM, kBlockN, false, false);
    const Range r = my_range(P);
    uint32_t T = 0, it = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        const int qb = it % C::kQBufs;
        ok = S.wait(B_QFULL + qb, (it / C::kQBufs) & 1);
        if (!ok) break;
        tc_fence_after();
        // Q into TMEM once per piece (after the previous piece's last QK, in issue
        // order); its shared-memory buffer is free for the next piece's Q after that
        const uint32_t qbase = sbase + C::kOffQ + qb * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            tmem_copy_128x256b(tmem + C::kColQ + kk * 8,
                               desc_sw128(qbase + (kk >> 2) * C::kCol + (kk & 3) * 32, 16, 1024));
        umma_commit(S.bar(B_QEMPTY + qb));
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int s = T % C::kKStages, sb = T & 1;
            ok = S.wait(B_KFULL + s, (T / C::kKStages) & 1);
            if (ok && T >= 2) ok = S.wait(B_SFREE + sb, ((T >> 1) - 1) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kbase = sbase + C::kOffK + s * C::kTile;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // Q from TMEM, K from shared memory
                const uint32_t off = (kk >> 2) * C::kCol + (kk & 3) * 32;
                umma_bf16_ts(tmem + C::kColS + sb * kBlockN, tmem + C::kColQ + kk * 8,
                             desc_sw128(kbase + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
            }
            umma_commit(S.bar(B_SFULL + sb));
            umma_commit(S.bar(B_KEMPTY + s));
        }
        ++it;
    }
    // everything issued has completed before TMEM is released
    umma_commit(S.bar(B_DRAIN));
    S.drain(B_DRAIN, 0);
}

// PV issuer (one thread): O (+)= P V for each tile once the softmax warps wrote
// P over its S buffer and its V tile landed; the first tile of a piece
// overwrites O.  Its completion frees the V stage and the S buffer.
template <int D>
__device__ void pv_issuer(const Params &P, const Sync &S, uint32_t sbase, uint32_t tmem)
{
    using C = Cfg<D>;
    constexpr uint32_t kIdescPV = idesc_bf16(kBlockM, D, false, true);
    const Range r = my_range(P);
    uint32_t T = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int s = T % C::kVStages, sb = T & 1;
            ok = S.wait(B_PFULL + sb, (T >> 1) & 1) && S.wait(B_VFULL + s, (T / C::kVStages) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t vbase = sbase + C::kOffV + s * C::kTile;
            const uint32_t pcol = tmem + C::kColS + sb * kBlockN;
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {  // P from TMEM, V from shared memory
                const uint64_t bd = desc_sw128(vbase + kk * 16 * 128, C::kCol, 1024);
                umma_bf16_ts(tmem + C::kColO, pcol + kk * 8, bd, kIdescPV,
                             (t > w.t0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(S.bar(B_VEMPTY + s));
            umma_commit(S.bar(B_SFREE + sb));
        }
    }
    umma_commit(S.bar(B_DRAIN2));
    S.drain(B_DRAIN2, 0);
}

__device__ __forceinline__ uint64_t f2x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void x2f(uint64_t v, float &lo, float &hi)
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
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int D>
__device__ void softmax_epilogue(const Params &P, const Sync &S, uint32_t tmem)
{
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = P.scale_log2;           // log2 units per raw score unit
    const float move = 8.f / c;             // raw-score growth that moves the reference
    const int kv_tail = P.L - (P.n_tiles - 1) * kBlockN;  // keys in the last tile
    const Range r = my_range(P);
    uint32_t T = 0;
    bool ok = true;
    // After a failed (timed-out) wait a warp skips all further work; every later
    // wait of any role returns at once (the abort flag is set).
    for (int k = 0; k < r.count; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        float m_run = -INFINITY, l_run = 0.f;  // m in raw score units
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int sb = T & 1;
            if (ok) ok = __all_sync(0xffffffffu, S.wait(B_SFULL + sb, (T >> 1) & 1));
            if (!ok) continue;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                tmem_ld32(tmem + lane_off + C::kColS + sb * kBlockN + cc * 32, sr[cc]);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_wait_ld(sr[cc]);

            if (t == P.n_tiles - 1 && kv_tail < kBlockN) {  // keys past L do not exist
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (cc * 32 + j >= kv_tail) sr[cc][j] = __float_as_uint(-INFINITY);
            }
            // row maximum of the raw scores (scale > 0 keeps the order)
            float mx4[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                float a = __uint_as_float(sr[cc][0]), b = __uint_as_float(sr[cc][1]);
#pragma unroll
                for (int j = 2; j < 32; j += 4) {
                    a = fmax3(a, __uint_as_float(sr[cc][j]), __uint_as_float(sr[cc][j + 1]));
                    b = fmax3(b, __uint_as_float(sr[cc][j + 2]), __uint_as_float(sr[cc][j + 3]));
                }
                mx4[cc] = fmaxf(a, b);
            }
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            float m_use = m_run, alpha = 1.f;
            bool rescale = false;
            if (mx > m_run + move) {  // p would exceed 2^8: move the reference
                m_use = mx;
                alpha = ex2((m_run - mx) * c);
                rescale = t > w.t0;
            }
            // p = 2^{(s - m) c}; two-wide FMA and adds, four partial sums
            const uint64_t c2 = f2x2(c, c);
            const float nmc = -m_use * c;
            const uint64_t nmc2 = f2x2(nmc, nmc);
            uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
            uint32_t pk[64];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const uint64_t y2 = ffma2(f2x2(__uint_as_float(sr[cc][j]), __uint_as_float(sr[cc][j + 1])),
                                              c2, nmc2);
                    float y0, y1;
                    x2f(y2, y0, y1);
                    const float p0 = ex2(y0), p1 = ex2(y1);
                    const uint64_t p2 = f2x2(p0, p1);
                    acc2[(j >> 1) & 3] = fadd2(acc2[(j >> 1) & 3], p2);
                    pk[(cc * 32 + j) >> 1] = pack_bf16x2(p0, p1);
                }
            float rs0, rs1, rs2, rs3, rs4, rs5, rs6, rs7;
            x2f(acc2[0], rs0, rs1);
            x2f(acc2[1], rs2, rs3);
            x2f(acc2[2], rs4, rs5);
            x2f(acc2[3], rs6, rs7);
            const float rowsum = ((rs0 + rs1) + (rs2 + rs3)) + ((rs4 + rs5) + (rs6 + rs7));
            l_run = l_run * alpha + rowsum;
            m_run = m_use;

            // O may be rescaled only after the previous tile's PV product completed
            // (the completion that freed the other S buffer)
            if (rescale) {
                const uint32_t Tp = T - 1;
                ok = __all_sync(0xffffffffu, S.wait(B_SFREE + (Tp & 1), (Tp >> 1) & 1));
                if (!ok) continue;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    const uint32_t ta = tmem + lane_off + C::kColO + cc * 32;
                    tmem_ld32(ta, o);
                    tmem_wait_ld(o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(ta, o);
                }
                tmem_wait_st();
            }
            // P (bf16 pairs) over the first half of this S buffer, in this row's
            // TMEM lane; the PV product reads it there
            const uint32_t pcol = tmem + lane_off + C::kColS + sb * kBlockN;
            tmem_st32(pcol, *reinterpret_cast<const uint32_t(*)[32]>(pk));
            tmem_st32(pcol + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.bar(B_PFULL + sb));
        }
        // ---- epilogue of the piece: O is final once the last PV product completed ----
        if (ok) {
            const uint32_t Tp = T - 1;
            ok = __all_sync(0xffffffffu, S.wait(B_SFREE + (Tp & 1), (Tp >> 1) & 1));
        }
        tc_fence_after();
        const int tok = w.mt * P.tok_per_tile + row / P.G;
        const bool valid = row < P.tok_per_tile * P.G && tok < w.cnt;
        const int h = w.g * P.G + row % P.G;
        __nv_bfloat16 *orow = P.out + ((static_cast<int64_t>(w.b) * P.r_max + tok) * P.H + h) * D;
        if (w.n_contrib == 1) {
            if (!ok) continue;
            const float inv = 1.f / l_run;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + C::kColO + cc * 32, o);
                tmem_wait_ld(o);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                        dst[q] = v;
                    }
                }
            }
            tc_fence_before();
            continue;
        }
        // part of a unit: store the partial (the merge kernel combines them)
        if (!ok) continue;
        float4 *po = P.part_o + (static_cast<int64_t>(w.unit) * P.slots + w.slot) * (D / 4) * kBlockM;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + C::kColO + cc * 32, o);
            tmem_wait_ld(o);
            if (valid) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    __stcg(po + (cc * 8 + q) * kBlockM + row,
                           make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                       __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3])));
            }
        }
        tc_fence_before();
        if (valid)
            __stcg(P.part_ml + (static_cast<int64_t>(w.unit) * P.slots + w.slot) * kBlockM + row,
                   make_float2(m_run, l_run));
    }
}

// Merge of the split units, a grid of its own after the attention grid.  For
// every valid row of a unit cut into n >= 2 pieces with partials (O_s, m_s, l_s):
//   out = sum_s 2^{(m_s - M) c} O_s / sum_s 2^{(m_s - M) c} l_s,   M = max_s m_s,
// the standard combination of softmax partials (m in raw score units, c the
// scale in log2 units).  Block (unit, 32-row group), thread (row, 8-column
// group): the partials keep rows innermost, so a warp reads 512 contiguous bytes
// per load.  Slots are taken eight at a time and every load of a batch, the
// sequence's row count included, is issued (volatile, in order) before any is
// used: a unit cut into up to eight pieces costs one round trip to L2.
__device__ __forceinline__ float4 ld_cg_v4(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float2 ld_cg_v2(const float2 *p)
{
    float2 v;
    asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

template <int D>
__global__ void __launch_bounds__(D * 4) merge_kernel(const Params P)
{
    constexpr int kBatch = 8;
    pdl_launch_dependents();
    pdl_wait();
    const int unit = blockIdx.x;
    const int row = blockIdx.y * 32 + (threadIdx.x & 31);
    const int grp = threadIdx.x >> 5;  // columns [8 grp, 8 grp + 8)
    const int mt = unit % P.n_mt, bg = unit / P.n_mt;
    const int g = bg % P.Hkv, b = bg / P.Hkv;
    int n = P.n_split;
    if (n == 0) {
        const int64_t base = static_cast<int64_t>(unit) * P.n_tiles;
        n = cta_of(P, base + P.n_tiles - 1) - cta_of(P, base) + 1;
    }
    // whole units were written by their piece; rows past r_max hold no token
    if (n < 2 || row >= P.tok_per_tile * P.G || mt * P.tok_per_tile + row / P.G >= P.r_max) return;
    const int count_b = __ldg(P.count + b);
    const float c = P.scale_log2;
    const int64_t s_base = static_cast<int64_t>(unit) * P.slots;
    float M = -INFINITY, l_sum = 0.f, acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    // rows past the sequence's count hold no partials; their loads stay inside the
    // workspace and their results are dropped below
    for (int s0 = 0; s0 < n; s0 += kBatch) {
        float2 ml[kBatch];
        float4 o[kBatch][2];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            ml[k] = make_float2(-INFINITY, 0.f);
            o[k][0] = o[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s0 + k < n) {  // uniform over the block
                const int64_t sl = s_base + s0 + k;
                ml[k] = ld_cg_v2(P.part_ml + sl * kBlockM + row);
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    o[k][q] = ld_cg_v4(P.part_o + (sl * (D / 4) + grp * 2 + q) * kBlockM + row);
            }
        }
        float mb = M;
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
            if (s0 + k < n) mb = fmaxf(mb, ml[k].x);
        const float alpha = ex2((M - mb) * c);  // 0 on the first batch
        l_sum *= alpha;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] *= alpha;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float e = s0 + k < n ? ex2((ml[k].x - mb) * c) : 0.f;
            l_sum = fmaf(e, ml[k].y, l_sum);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                acc[4 * q] = fmaf(e, o[k][q].x, acc[4 * q]);
                acc[4 * q + 1] = fmaf(e, o[k][q].y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(e, o[k][q].z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(e, o[k][q].w, acc[4 * q + 3]);
            }
        }
        M = mb;
    }
    const int cnt = max(0, min(count_b, P.r_max));
    const int tok = mt * P.tok_per_tile + row / P.G;
    if (tok >= cnt) return;
    const float inv = 1.f / l_sum;
    const int h = g * P.G + row % P.G;
    uint4 v;
    v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4 *>(P.out + ((static_cast<int64_t>(b) * P.r_max + tok) * P.H + h) * D +
                               grp * 8) = v;
}

// Fresh K/V rows into the caches.  Lets the attention grid launch at once.
template <int D>
__global__ void __launch_bounds__(256) write_back_kernel(const Params P)
{
    pdl_launch_dependents();
    pdl_wait();
    constexpr int kChunks = D / 8;
    const int64_t total = static_cast<int64_t>(P.B) * P.r_max * P.Hkv * kChunks;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(e % kChunks);
        const int64_t rg = e / kChunks;  // (b, r, g) flattened
        const int g = static_cast<int>(rg % P.Hkv);
        const int64_t br = rg / P.Hkv;
        const int r = static_cast<int>(br % P.r_max);
        const int b = static_cast<int>(br / P.r_max);
        const int c = __ldg(P.count + b);
        if (ch == 0 && g == 0 && r == 0 && (c < 0 || c > P.r_max))
            flag_status(P.status, EC_DEV_BAD_COUNT);
        if (r >= min(max(c, 0), P.r_max)) continue;
        const int32_t *idx = P.idx + static_cast<int64_t>(b) * P.idx_stride;
        const int p = __ldg(idx + r);
        if (p < 0 || p >= P.L) {
            if (ch == 0 && g == 0) flag_status(P.status, EC_DEV_BAD_INDEX);
            continue;
        }
        if (ch == 0 && g == 0 && r > 0 && __ldg(idx + r - 1) >= p)
            flag_status(P.status, EC_DEV_BAD_INDEX);
        const int64_t src = (br * P.Hkv + g) * D + ch * 8;
        const int64_t dst = ((static_cast<int64_t>(b) * P.L + p) * P.Hkv + g) * D + ch * 8;
        *reinterpret_cast<uint4 *>(P.k_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(P.k_new + src));
        *reinterpret_cast<uint4 *>(P.v_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(P.v_new + src));
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const Params P, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc + 16);
    Sync S{sbase + C::kOffBar, abort_flag, P.status, P.wait_limit};

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < B_COUNT; ++i)
            mbar_init(S.bar(i), (i == B_PFULL || i == B_PFULL + 1) ? 4u : 1u);
        fence_mbar_init();
    }
    // Q rows past tok_per_tile * G are never loaded: keep them zero
    for (uint32_t o = threadIdx.x * 16; o < C::kQBufs * C::kTile; o += kThreads * 16)
        st_shared_v4(sbase + C::kOffQ + o, 0u, 0u, 0u, 0u);
    fence_async_smem();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && (threadIdx.x & 31) == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the write-back grid (and everything before it) has completed

    if (warp == 0 || warp == 6) {
        if ((threadIdx.x & 31) == 0) {
            if (warp == 0)
                producer_qk<D>(P, S, sbase, &tm_q, &tm_k);
            else
                producer_v<D>(P, S, sbase, &tm_v);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 7) {
        if ((threadIdx.x & 31) == 0) {
            if (warp == 1)
                qk_issuer<D>(P, S, sbase, tmem);
            else
                pv_issuer<D>(P, S, sbase, tmem);
        }
        __syncwarp();
    } else {
        softmax_epilogue<D>(P, S, tmem);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [B, rows, heads, D] bf16 viewed as 4-D {D, heads, rows, B}; box {64, box_heads,
// box_rows, 1}, 128-byte swizzle, out-of-range elements read as zero.
bool encode_4d(CUtensorMap *map, const void *base, int B, int rows, int heads, int D,
               int box_heads, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(heads) * D * 2,
                                   static_cast<cuuint64_t>(rows) * heads * D * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_heads),
                               static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int G, tok_per_tile, n_mt, n_units, n_tiles, grid, slots, n_split;
    int64_t total;
    bool split;  // some unit is cut into several pieces: the merge kernel runs
};

// The work split, chosen by a cost model counted in tile times (one 128 x 128
// tile is about 1 us per SM at steady state):
//   whole units      split-major items with one split: no partials, no merge;
//   stream-K         equal contiguous tile ranges on every SM, plus the merge;
//   split-major      items of n_tiles / sp tiles dealt round-robin, plus the merge.
// A piece's epilogue costs about one tile and the merge kernel about five (its
// CTAs become resident while the attention grid runs; after it, one round trip
// to L2 and the writes).  Calibrated on whole decode steps: the single-sequence
// step (32 units of 8 tiles) is faster cut into 4 splits than in whole units.
// With several row tiles per KV head and caches larger than half of L2, stream-K
// would read each K/V tile from HBM once per row tile and is not taken.
Plan make_plan(int B, int L, int r_max, int H, int Hkv)
{
    constexpr double kPiece = 1.0, kMerge = 5.0;
    Plan p;
    p.G = H / Hkv;
    p.tok_per_tile = kBlockM / p.G;
    p.n_mt = (r_max + p.tok_per_tile - 1) / p.tok_per_tile;
    p.n_units = B * Hkv * p.n_mt;
    p.n_tiles = (L + kBlockN - 1) / kBlockN;
    p.total = static_cast<int64_t>(p.n_units) * p.n_tiles;
    const int n_sm = device_sm_count();
    auto ceil_div = [](int64_t a, int64_t b) { return (a + b - 1) / b; };

    // whole units
    double best = static_cast<double>(ceil_div(p.n_units, n_sm)) * (p.n_tiles + kPiece);
    p.n_split = 1;
    // split-major items
    for (int sp = 2; sp <= std::min(kMaxContrib, p.n_tiles / 2); ++sp) {
        const int64_t rounds = ceil_div(static_cast<int64_t>(p.n_units) * sp, n_sm);
        const double cost =
            static_cast<double>(rounds) * (ceil_div(p.n_tiles, sp) + kPiece) + kMerge;
        if (cost < best - 1e-9) {
            best = cost;
            p.n_split = sp;
        }
    }
    // stream-K
    const int64_t kv_bytes = 2LL * B * L * Hkv * 128 * 2;
    int64_t g = std::min<int64_t>(n_sm, p.total);
    g = std::max<int64_t>(1, std::min<int64_t>(g, static_cast<int64_t>(p.n_units) * (kMaxContrib - 2)));
    if (!(p.n_mt > 1 && kv_bytes > (64LL << 20))) {
        const int64_t per_cta = ceil_div(p.total, g);
        const double cost = static_cast<double>(per_cta) +
                            kPiece * static_cast<double>(ceil_div(per_cta, p.n_tiles) + 1) + kMerge;
        if (cost < best - 1e-9) {
            best = cost;
            p.n_split = 0;
        }
    }
    if (p.n_split == 0) {
        p.grid = static_cast<int>(g);
        // a unit of n_tiles tiles meets at most ceil(n_tiles * grid / total) + 1 ranges
        p.slots = static_cast<int>(std::min<int64_t>(
            kMaxContrib, ceil_div(static_cast<int64_t>(p.n_tiles) * p.grid, p.total) + 1));
        // a unit is split when a range boundary falls inside it
        auto cta = [&](int64_t w) { return ((w + 1) * p.grid - 1) / p.total; };
        p.split = false;
        for (int64_t u = 0; u < p.n_units && !p.split; ++u)
            p.split = cta(u * p.n_tiles) != cta(u * p.n_tiles + p.n_tiles - 1);
    } else {
        p.grid = static_cast<int>(std::min<int64_t>(n_sm, static_cast<int64_t>(p.n_units) * p.n_split));
        p.slots = p.n_split;
        p.split = p.n_split > 1;
    }
    return p;
}

size_t partial_offsets(const Plan &p, int D, size_t *off_ml, size_t *off_o)
{
    size_t off = kWsHeader;
    *off_ml = off;
    const size_t parts = p.split ? static_cast<size_t>(p.n_units) * p.slots : 0;
    off = align_up(off + parts * kBlockM * sizeof(float2), 256);
    *off_o = off;
    return off + parts * kBlockM * static_cast<size_t>(D) * sizeof(float);
}

template <int D>
cudaError_t launch_typed(const Params &p, const Plan &plan, const void *q, cudaStream_t stream)
{
    CUtensorMap tq, tk, tv;
    if (!encode_4d(&tq, q, p.B, p.r_max, p.H, D, p.G, p.tok_per_tile) ||
        !encode_4d(&tk, p.k_cache, p.B, p.L, p.Hkv, D, 1, kBlockN) ||
        !encode_4d(&tv, p.v_cache, p.B, p.L, p.Hkv, D, 1, kBlockN))
        return cudaErrorInvalidValue;
    // 1. write-back: a few CTAs per SM over the fresh rows
    const int64_t chunks = static_cast<int64_t>(p.B) * p.r_max * p.Hkv * (D / 8);
    const int wb_grid = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>((chunks + 255) / 256, 4 * static_cast<int64_t>(device_sm_count()))));
    cudaError_t e = launch(write_back_kernel<D>, dim3(wb_grid), dim3(256), 0, stream, p);
    if (e != cudaSuccess) return e;
    // 2. attention; its set-up overlaps the write-back (programmatic dependent launch)
    e = launch(attention_tc_kernel<D>, dim3(plan.grid), dim3(kThreads), Cfg<D>::kBytes, stream, p,
               tq, tk, tv);
    if (e != cudaSuccess || !plan.split) return e;
    // 3. merge of the split units: (unit, 32-row group) blocks over the rows a unit
    //    can hold (at most r_max tokens)
    const int row_groups = (std::min(kBlockM, std::min(p.tok_per_tile, p.r_max) * p.G) + 31) / 32;
    return launch(merge_kernel<D>, dim3(p.n_units, row_groups), dim3(D * 4), 0, stream, p);
}

}  // namespace

bool attention_tc_supported(int dtype, int32_t seq_len, int32_t head_dim)
{
    return dtype == EC_BF16 && (head_dim == 64 || head_dim == 128) && seq_len >= 1;
}

int32_t attention_tc_kernel_count(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                  int32_t n_kv_heads)
{
    return make_plan(batch, seq_len, r_max, n_heads, n_kv_heads).split ? 3 : 2;
}

size_t attention_tc_workspace_bytes(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                    int32_t n_kv_heads, int32_t head_dim)
{
    if (batch < 1 || seq_len < 1 || r_max < 1 || n_kv_heads < 1 || n_heads < n_kv_heads)
        return kWsHeader;
    const Plan p = make_plan(batch, seq_len, r_max, n_heads, n_kv_heads);
    size_t a, b;
    return partial_offsets(p, head_dim, &a, &b);
}

cudaError_t launch_attention_tc(const void *q, const void *k_new, const void *v_new,
                                const int32_t *idx, int64_t idx_stride, const int32_t *count,
                                void *k_cache, void *v_cache, void *out, int32_t batch,
                                int32_t seq_len, int32_t r_max, int32_t n_heads,
                                int32_t n_kv_heads, int32_t head_dim, float scale,
                                void *workspace, cudaStream_t stream)
{
    if (r_max == 0) return cudaSuccess;  // nothing to recompute, nothing to write back
    const Plan plan = make_plan(batch, seq_len, r_max, n_heads, n_kv_heads);
    Params p;
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    p.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.idx = idx;
    p.idx_stride = idx_stride;
    p.count = count;
    p.B = batch;
    p.L = seq_len;
    p.r_max = r_max;
    p.H = n_heads;
    p.Hkv = n_kv_heads;
    p.G = plan.G;
    p.tok_per_tile = plan.tok_per_tile;
    p.n_mt = plan.n_mt;
    p.n_units = plan.n_units;
    p.n_tiles = plan.n_tiles;
    p.grid = plan.grid;
    p.total = plan.total;
    p.slots = plan.slots;
    p.n_split = plan.n_split;
    p.scale_log2 = scale * kLog2e;
    char *ws = static_cast<char *>(workspace);
    size_t o_ml, o_o;
    partial_offsets(plan, head_dim, &o_ml, &o_o);
    p.status = reinterpret_cast<uint32_t *>(ws);
    p.wait_limit = wait_limit_cycles();
    p.part_ml = reinterpret_cast<float2 *>(ws + o_ml);
    p.part_o = reinterpret_cast<float4 *>(ws + o_o);
    return head_dim == 128 ? launch_typed<128>(p, plan, q, stream)
                           : launch_typed<64>(p, plan, q, stream);
}

}  // namespace ec
