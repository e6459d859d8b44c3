// Selective-recompute bidirectional attention on the 5th-generation tensor
// cores (tcgen05 + TMEM), fed by TMA, with the KV write-back in the same kernel.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, section "1. Il Problema" (dLLM attention is
// bidirectional) and "Algoritmo di Funzionamento" step 2 (the partial forward
// recomputes K/V only for the selected tokens; the cache supplies the rest).
//
// One launch.  Work is cut into
//   units    up to 128 query rows of one (sequence b, KV head g): the
//            (recomputed row r, head h of g's group) pairs packed r-major, so a
//            GQA group shares each K/V tile; a (b, g) has n_mt units;
//   groups   n_mt CTAs, one per unit of a (b, g).  The (b, g, 128-key tile)
//            pairs, laid end to end, are cut into one equal contiguous range per
//            group, and the n_mt CTAs of a group walk the same key tiles at the
//            same time: each tile comes from HBM once and from L2 for the others.
//   pieces   the (b, g)'s a range meets.  A piece that covers all of a unit's
//            tiles writes its output.  A unit cut over several groups is merged
//            in the kernel: the group holding its last tile owns it; the others
//            contribute a partial (O, m, l) and release a flag.  Every CTA runs
//            its pieces from the last (b, g) to the first, so a contribution
//            (the first piece a group runs) is done long before its owner (the
//            last piece of the next group) needs it.
// Write-back: the fresh K/V rows of a tile are patched into the tile in shared
// memory after its TMA load lands (so no CTA depends on another's global write);
// the cache is written from the fresh tensors by each CTA's softmax warps before
// their first tile, the CTA mt of a group taking every n_mt-th fresh row of the
// group's tiles.  A sequence that recomputes all L rows (count = L, so the index
// set is 0 .. L-1) loads its tiles from the fresh K/V directly, and its mt = 0
// CTAs store every tile to the cache with a TMA store.
// Instances: MODE_PLAIN; MODE_SIMSD (SimSD's temporal causal mask, label windows
// applied in the softmax); MODE_COVER (COVER's dual view: seed rows neither
// written back nor patched, a seed row's own column hidden and its masked-input
// term added in the epilogue).
//
// Warp roles (384 threads):
//   warp 0     TMA producer of Q (one tile per piece) and K tiles; warp 6 of V
//              tiles (128-byte swizzle, rings of stages);
//   warp 1     TMEM allocation; Q into TMEM (tcgen05.cp); per K tile the whole
//              warp patches the fresh rows into it (a TMA box for a tile of fresh
//              rows, else cp.async), or stores the tile for a full refresh; then one thread
//              issues S = Q K^T (tcgen05.mma) into one of two TMEM S buffers once
//              the PV product that read that buffer's P has completed;
//   warp 7     the same for V (patching), then O += P V into the TMEM O
//              accumulator: a second issuing thread, so the next tile's QK never
//              queues behind this tile's PV;
//   warps 2-5, 8-11  the write-back share, then the softmax, two warps per quarter
//              of the TMEM lanes: one row per thread and half a tile's score
//              columns per warp (the two halves
//              agree on the row maximum through shared memory); online softmax in
//              the log2 domain on S read by tcgen05.ld (the reference maximum moves
//              only when it grows by more than 8 in log2 units, rescaling O in
//              TMEM), P as bf16 over the first half of the same S buffer (the PV
//              product reads its A operand there), and the piece's epilogue.
// Every wait is bounded; a timeout sets EC_DEV_TIMEOUT and unwinds.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>

#include "ec_internal.cuh"
#include "tc_ptx.cuh"

namespace ec {
namespace {

using namespace ptx;

constexpr int kBlockM = 128;   // query rows per unit = TMEM lanes
constexpr int kBlockN = 128;   // keys per tile
constexpr int kThreads = 384;  // 12 warps
constexpr int kSoftmaxThreads = 256;  // 8 softmax warps
constexpr int kSoftmaxBarrier = 1;  // named barrier of the softmax warps
constexpr int kPairBarrier0 = 2;    // named barriers 2-5: the two softmax warps of a TMEM lane quarter
constexpr int kMaxContrib = 8;      // contributors merged by one owner at most

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
    static constexpr uint32_t kOffRows = kOffMisc + 64;   // [2][128] tile rows of a tile's fresh rows (K, V)
    static constexpr uint32_t kOffXchg = kOffRows + 256;  // [2][128] row maxima / sums of the two column halves
    static constexpr uint32_t kBytes = kOffXchg + 2 * 128 * 4 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t kTmemCols = 512;
    // two S buffers, columns [0, 128) and [128, 256); P (bf16 pairs) of a tile
    // overwrites the first 64 columns of its own S buffer
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = 256;  // O: columns [256, 256 + D)
    static constexpr uint32_t kColQ = 448;  // Q (bf16 pairs): columns [448, 448 + D / 2)
};

enum : int {
    B_KFULL = 0,     // [4] K tile landed
    B_KEMPTY = 4,    // [4] K stage consumed (its QK done)
    B_VFULL = 8,     // [4] V tile landed
    B_VEMPTY = 12,   // [4] V stage consumed (its PV done)
    B_QFULL = 16,    // [2] Q tile landed
    B_QEMPTY = 18,   // [2] Q tile copied into TMEM
    B_SFULL = 20,    // [2] S buffer written by its QK product
    B_PFULL = 22,    // [2] P written over its S buffer (and O corrected): 8 softmax warps
    B_SFREE = 24,    // [2] the PV product that read the buffer's P completed (O updated)
    B_DRAIN = 26,    // QK issuer's products all complete
    B_DRAIN2 = 27,   // PV issuer's products all complete
    B_KPATCH = 28,   // fresh K granules landed in the current K tile
    B_VPATCH = 29,   // fresh V granules landed in the current V tile
    B_COUNT = 30
};
static_assert(8 * B_COUNT <= 256, "barrier area");

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
    int grouped;       // 1: groups of n_mt CTAs over (b, g, tile) ranges; 0: whole units round-robin
    int n_groups;
    int64_t total;     // B * Hkv * n_tiles
    int slots;         // partial slots per unit (most contributors a unit can have)
    float scale_log2;
    uint32_t *status;     // workspace status word
    long long wait_limit; // cycles one in-kernel wait may take
    uint32_t *flags;      // [n_units] contributions released (the owner resets it to 0)
    float2 *part_ml;      // [n_units][slots][128] (m, l), m in raw score units
    float4 *part_o;       // [n_units][slots][D / 4][128] unnormalised O
    // SimSD's temporal causal mask (null without it): section (0 prompt, 1 data,
    // 2 mask slot) and step label of every position, [B, L] each
    const uint8_t *section;
    const int32_t *tau;
    // COVER's dual view (null without it): seed flag of every recomputed row,
    // [B, r_max]; the queries, read directly for the seeds' diagonal terms
    const uint8_t *seed;
    const __nv_bfloat16 *q;
};

enum : int { MODE_PLAIN = 0, MODE_SIMSD = 1, MODE_COVER = 2 };

// bf16 pairs (low half first) widened exactly to float, and a pair's dot product
// added to an accumulator
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t x)
{
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}
__device__ __forceinline__ float fmaf_bf16x2(uint32_t a, uint32_t b, float acc)
{
    const float2 fa = bf16x2_to_f2(a), fb = bf16x2_to_f2(b);
    return fmaf(fa.y, fb.y, fmaf(fa.x, fb.x, acc));
}

enum : int { ROLE_WHOLE = 0, ROLE_CONTRIB = 1, ROLE_OWNER = 2 };

// A piece: tiles [t0, t1) of unit (b, g, mt), processed by this CTA.
struct Piece {
    int unit, b, g, mt, t0, t1, cnt, role, slot, n_contrib;
};

__device__ __forceinline__ int group_of(const Params &P, int64_t w)
{
    return static_cast<int>(((w + 1) * P.n_groups - 1) / P.total);
}

// This CTA's share: `count` pieces, piece_at(k) for k in [0, count) in processing order.
struct Range {
    int64_t w0, w1;
    int bg_first, count, mt, group;
};
__device__ __forceinline__ Range my_range(const Params &P)
{
    Range r;
    r.w0 = r.w1 = 0;
    r.bg_first = 0;
    r.group = 0;
    r.mt = 0;
    r.count = 0;
    if (!P.grouped) {  // whole units dealt round-robin
        r.count = static_cast<int>(blockIdx.x) < P.n_units
                      ? (P.n_units - 1 - static_cast<int>(blockIdx.x)) / P.grid + 1
                      : 0;
        return r;
    }
    r.group = static_cast<int>(blockIdx.x) / P.n_mt;
    r.mt = static_cast<int>(blockIdx.x) % P.n_mt;
    if (r.group >= P.n_groups) return r;
    r.w0 = static_cast<int64_t>(r.group) * P.total / P.n_groups;
    r.w1 = static_cast<int64_t>(r.group + 1) * P.total / P.n_groups;
    if (r.w1 <= r.w0) return r;
    r.bg_first = static_cast<int>(r.w0 / P.n_tiles);
    r.count = static_cast<int>((r.w1 - 1) / P.n_tiles) - r.bg_first + 1;
    return r;
}

__device__ __forceinline__ Piece piece_at(const Params &P, const Range &r, int k)
{
    Piece p;
    if (!P.grouped) {
        p.unit = static_cast<int>(blockIdx.x) + k * P.grid;
        p.mt = p.unit % P.n_mt;
        const int bg = p.unit / P.n_mt;
        p.g = bg % P.Hkv;
        p.b = bg / P.Hkv;
        p.t0 = 0;
        p.t1 = P.n_tiles;
        p.role = ROLE_WHOLE;
        p.slot = p.n_contrib = 0;
    } else {
        const int bg = r.bg_first + r.count - 1 - k;  // the last (b, g) first
        p.mt = r.mt;
        p.unit = bg * P.n_mt + r.mt;
        p.g = bg % P.Hkv;
        p.b = bg / P.Hkv;
        const int64_t base = static_cast<int64_t>(bg) * P.n_tiles;
        p.t0 = static_cast<int>(max(r.w0, base) - base);
        p.t1 = static_cast<int>(min(r.w1, base + P.n_tiles) - base);
        const int k_first = group_of(P, base), k_last = group_of(P, base + P.n_tiles - 1);
        p.n_contrib = k_last - k_first;
        if (k_first == k_last) {
            p.role = ROLE_WHOLE;
            p.slot = 0;
        } else if (r.group == k_last) {
            p.role = ROLE_OWNER;
            p.slot = 0;
        } else {
            p.role = ROLE_CONTRIB;
            p.slot = r.group - k_first;
        }
    }
    p.cnt = max(0, min(__ldg(P.count + p.b), P.r_max));
    return p;
}

// Units with no recomputed rows (mt beyond the sequence's count) are skipped by
// every role alike (contributors and owner agree: count is one value).
__device__ __forceinline__ bool piece_active(const Params &P, const Piece &p)
{
    return p.mt * P.tok_per_tile < p.cnt && p.t1 > p.t0;
}

// Every position of sequence b is recomputed: the index set is 0 .. L-1.  (Not
// used with seeds, whose positions keep the cached K/V.)
__device__ __forceinline__ bool piece_dense(const Params &P, const Piece &p)
{
    return p.cnt == P.L && P.seed == nullptr;
}

static_assert(Cfg<128>::kColS + 2 * kBlockN <= Cfg<128>::kColO, "TMEM columns overlap");
static_assert(Cfg<128>::kColO + 128 <= Cfg<128>::kColQ, "TMEM columns overlap");
static_assert(Cfg<128>::kColQ + 128 / 2 <= Cfg<128>::kTmemCols, "TMEM columns overflow");
static_assert(Cfg<128>::kBytes <= 227 * 1024 && Cfg<64>::kBytes <= 227 * 1024, "shared memory");

// Q and K producer (one thread): per piece its Q tile, then its K tiles (from the
// fresh K of a fully recomputed sequence, else from the cache).
template <int D>
__device__ void producer_qk(const Params &P, const Sync &S, uint32_t sbase, const CUtensorMap *tm_q,
                            const CUtensorMap *tm_k, const CUtensorMap *tm_kn)
{
    using C = Cfg<D>;
    const uint32_t q_bytes = static_cast<uint32_t>(P.tok_per_tile * P.G) * D * 2;
    const Range r = my_range(P);
    uint32_t T = 0, it = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        const CUtensorMap *src = piece_dense(P, w) ? tm_kn : tm_k;
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
                tma_load_4d(kdst + c * C::kCol, src, S.bar(B_KFULL + s), c * 64, w.g, t * kBlockN, w.b);
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
__device__ void producer_v(const Params &P, const Sync &S, uint32_t sbase, const CUtensorMap *tm_v,
                           const CUtensorMap *tm_vn)
{
    using C = Cfg<D>;
    const Range r = my_range(P);
    uint32_t T = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        const CUtensorMap *src = piece_dense(P, w) ? tm_vn : tm_v;
        for (int t = w.t0; t < w.t1 && ok; ++t, ++T) {
            const int s = T % C::kVStages;
            if (T >= static_cast<uint32_t>(C::kVStages))
                ok = S.wait(B_VEMPTY + s, ((T / C::kVStages) - 1) & 1);
            if (!ok) break;
            const uint32_t vdst = sbase + C::kOffV + s * C::kTile;
            mbar_expect_tx(S.bar(B_VFULL + s), C::kTile);
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(vdst + c * C::kCol, src, S.bar(B_VFULL + s), c * 64, w.g, t * kBlockN, w.b);
        }
    }
    if (!ok)
        for (uint32_t u = (T > C::kVStages ? T - C::kVStages : 0); u < T; ++u)
            S.drain(B_VFULL + u % C::kVStages, (u / C::kVStages) & 1);
}

// TMA store of one 64-column block of a tile (rows past L are not stored).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
        : "memory");
}
// Wait until every bulk store this thread issued has finished reading shared memory.
__device__ __forceinline__ void bulk_commit_and_wait_read()
{
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every bulk store this thread issued is complete (before the CTA exits).
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// First r in [0, cnt) with idx[r] >= key (cnt when none), by the whole warp:
// 32 samples per round.  idx ascending; a non-ascending set still yields an
// index in [0, cnt].
__device__ __forceinline__ int lower_bound_warp(const int32_t *idx, int cnt, int key)
{
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = cnt;  // the answer lies in [lo, hi]
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        const int j = lo + lane * step;
        const bool below = j < hi && __ldg(idx + j) < key;
        const int n = __popc(__ballot_sync(0xffffffffu, below));  // samples below the key
        const int nlo = n > 0 ? lo + (n - 1) * step + 1 : lo;
        hi = min(hi, lo + n * step);
        lo = nlo;
    }
    const int j = lo + lane;
    const bool below = j < hi && __ldg(idx + j) < key;
    return lo + __popc(__ballot_sync(0xffffffffu, below));
}

// The fresh K or V rows of one piece, put into each landed tile by an MMA
// issuer warp before its product reads the tile.  The cursor walks the piece's
// ascending index set; a window of 128 of its entries (4 per lane) stays in
// registers and is refilled, off the critical path, after a tile used some.
// A tile made only of fresh rows comes in as one TMA box per column block; the
// rows of other tiles are copied by cp.async.  (Writing them back to the cache
// is done separately, see write_back_share.)
template <int D, bool kSeeds>
struct Patch {
    int cur, vbase, cnt;
    int v0, v1, v2, v3;  // entries vbase + lane + 32 k, INT_MAX past the set
    bool stored;         // a TMA store to the cache is in flight (full refresh)
    int bar;             // index of this warp's mbarrier for the granule loads
    uint32_t uses;       // its phases used so far
    const int32_t *idx;
    const uint8_t *sd;   // seed flags of the sequence's rows (null: no seeds)
    unsigned sflags;     // bit k: entry vbase + lane + 32 k is a seed (not patched)
    uint8_t *rows;       // shared [128]: tile rows of the current tile's fresh rows (255: none)
    const CUtensorMap *fresh128, *cache128;

    __device__ void init(int bar_, uint8_t *rows_smem, const CUtensorMap *f128, const CUtensorMap *c128)
    {
        stored = false;
        bar = bar_;
        uses = 0;
        rows = rows_smem;
        fresh128 = f128;
        cache128 = c128;
    }

    __device__ void load_window(int at)
    {
        const int lane = threadIdx.x & 31;
        vbase = at;
        v0 = at + lane < cnt ? __ldg(idx + at + lane) : INT_MAX;
        v1 = at + 32 + lane < cnt ? __ldg(idx + at + 32 + lane) : INT_MAX;
        v2 = at + 64 + lane < cnt ? __ldg(idx + at + 64 + lane) : INT_MAX;
        v3 = at + 96 + lane < cnt ? __ldg(idx + at + 96 + lane) : INT_MAX;
        sflags = 0;
        if constexpr (kSeeds)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (at + 32 * k + lane < cnt && __ldg(sd + at + 32 * k + lane)) sflags |= 1u << k;
    }

    // Whole warp, at a piece start.  The K side of one CTA per sequence also
    // checks the count and the whole index set.  The window starts as the set's
    // first 128 entries; the cursor (the first entry at or past the piece's first
    // key) is counted in it when it lies there, so a set of at most 128 entries
    // costs one round trip to global memory.
    __device__ void start(const Params &P, const Piece &w, bool check)
    {
        const int lane = threadIdx.x & 31;
        idx = P.idx + static_cast<int64_t>(w.b) * P.idx_stride;
        sd = kSeeds ? P.seed + static_cast<int64_t>(w.b) * P.r_max : nullptr;
        cnt = w.cnt;
        const bool checker = check && w.mt == 0 && w.g == 0 && w.t0 == 0;
        const bool dense = piece_dense(P, w);
        if (!dense || checker) load_window(0);
        if (checker) {
            const int c_raw = __ldg(P.count + w.b);
            if (lane == 0 && (c_raw < 0 || c_raw > P.r_max)) flag_status(P.status, EC_DEV_BAD_COUNT);
            // the window's entries against their predecessors, the rest by loads
            bool bad = false;
            const int vv[4] = {v0, v1, v2, v3};
            int carry = INT_MIN;  // entry 32 k - 1
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int up = __shfl_up_sync(0xffffffffu, vv[k], 1);
                const int prev = lane == 0 ? carry : up;
                const int e = 32 * k + lane;
                if (e < cnt) bad |= vv[k] < 0 || vv[k] >= P.L || (e > 0 && prev >= vv[k]);
                carry = __shfl_sync(0xffffffffu, vv[k], 31);
            }
            for (int j = 128 + lane; j < cnt; j += 32) {
                const int p = __ldg(idx + j);
                bad |= p < 0 || p >= P.L || __ldg(idx + j - 1) >= p;
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(P.status, EC_DEV_BAD_INDEX);
        }
        if (dense) {
            cur = vbase = 0;
            v0 = v1 = v2 = v3 = INT_MAX;
            sflags = 0;
            return;
        }
        const int lo = w.t0 * kBlockN;
        if (cnt <= 128 || __shfl_sync(0xffffffffu, v3, 31) >= lo) {  // entries are ascending
            cur = __popc(__ballot_sync(0xffffffffu, v0 < lo)) + __popc(__ballot_sync(0xffffffffu, v1 < lo)) +
                  __popc(__ballot_sync(0xffffffffu, v2 < lo)) + __popc(__ballot_sync(0xffffffffu, v3 < lo));
        } else {
            cur = lower_bound_warp(idx, w.cnt, lo);
            load_window(cur);
        }
    }

    // Whole warp, tile t of piece w landed at `tile`: the fresh rows that fall in
    // it into it, or for a fully recomputed sequence the tile stored to the cache
    // as it is (from the group's mt = 0 CTA).  Returns with the tile visible to
    // the tensor core, or false when a wait gave up.
    __device__ bool tile(const Params &P, const Sync &S, const Piece &w, int t, uint32_t tile, bool is_v)
    {
        using C = Cfg<D>;
        constexpr int kChunks = D / 8;  // 16-byte chunks per row and head
        constexpr int step = 32 / kChunks;
        const int lane = threadIdx.x & 31;
        if (piece_dense(P, w)) {
            if (w.mt == 0 && lane == 0) {  // the landed tile is the cache's new content
                fence_async_smem();
                for (int c = 0; c < D / 64; ++c)
                    tma_store_4d(cache128, tile + c * C::kCol, c * 64, w.g, t * kBlockN, w.b);
                bulk_commit_and_wait_read();  // read before the stage can be reused
                stored = true;
            }
            __syncwarp();
            return true;
        }
        const __nv_bfloat16 *fresh = is_v ? P.v_new : P.k_new;
        const int tile_end = (t + 1) * kBlockN;
        bool patched = false;
        for (;;) {
            // the entries cur .. cur + n - 1 of the window fall in this tile: their
            // rows in the tile to shared memory, in order
            int n = 0;
            bool seeded = false;  // a seed among them: its row keeps the cached K/V
            {
                const int vv[4] = {v0, v1, v2, v3};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = vbase + 32 * k + lane;
                    const bool in = e >= cur && vv[k] < tile_end;
                    const bool is_seed = kSeeds && ((sflags >> k) & 1u);
                    const unsigned m = __ballot_sync(0xffffffffu, in);
                    if constexpr (kSeeds) seeded |= __any_sync(0xffffffffu, in && is_seed);
                    if (in) {
                        const int rit = vv[k] - t * kBlockN;
                        rows[e - cur] = rit >= 0 && rit < kBlockN && !is_seed ? static_cast<uint8_t>(rit)
                                                                              : uint8_t(255);
                    }
                    n += __popc(m);
                }
            }
            __syncwarp();
            if (n > 0) {
                if (n == kBlockN && !seeded) {
                    // a whole tile of fresh rows (128 distinct positions inside it,
                    // so 128 consecutive fresh rows): one TMA box per column block
                    if (lane == 0) {
                        mbar_expect_tx(S.bar(bar), C::kTile);
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_4d(tile + c * C::kCol, fresh128, S.bar(bar), c * 64, w.g, cur, w.b);
                    }
                    const bool ok = __all_sync(0xffffffffu, S.wait(bar, uses & 1));
                    ++uses;
                    if (!ok) {
                        pending = true;  // the load may still land: drained on exit
                        return false;
                    }
                } else {
                    // every 16-byte chunk of those rows in flight at once (one round
                    // trip).  A lane always moves the same chunk c of rows q0,
                    // q0 + step, ..., four rows per step so that their addresses are
                    // computed together.
                    const int c = lane % kChunks, q0 = lane / kChunks;
                    const uint32_t col = tile + (c / 8) * C::kCol;
                    const int64_t row_elems = static_cast<int64_t>(P.Hkv) * D;
                    const int64_t src0 =
                        (static_cast<int64_t>(w.b) * P.r_max + cur) * row_elems + w.g * D + c * 8;
                    for (int qb = q0; qb < n; qb += 4 * step) {
                        int rq[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) rq[u] = qb + u * step < n ? rows[qb + u * step] : 255;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int rit = rq[u];
                            if (rit < kBlockN && t * kBlockN + rit < P.L)
                                cp_async_16(col + rit * 128 + (((c % 8) ^ (rit & 7)) << 4),
                                            fresh + src0 + (qb + u * step) * row_elems);
                        }
                    }
                    cp_async_wait_all();
                }
                __syncwarp();  // rows is rewritten by the next tile
                cur += n;
                patched = true;
            }
            // the window ran out inside this tile and the index set goes on: refill
            // it here and look again
            if (cur < vbase + 128 || cur >= cnt) break;
            load_window(cur);
        }
        if (patched) {
            fence_async_smem();  // the patched rows are visible to the tensor core
            // refill the window at the cursor for the next tiles; its loads travel
            // while this tile's product runs
            if (cur < cnt && cur > vbase) load_window(cur);
        }
        __syncwarp();
        return true;
    }

    // One thread, when the warp unwinds: let granule loads still in flight land.
    __device__ void drain(const Sync &S) const
    {
        if (pending) S.drain(bar, (uses - 1) & 1);
    }
    bool pending = false;
};

// Candidate rows of piece w for this CTA's write-back share: its rows
// j = mt, mt + n_mt, ... of the index set (none for a fully recomputed sequence,
// whose tiles are stored whole, see Patch::tile).
__device__ __forceinline__ int share_rows(const Params &P, const Piece &w)
{
    if (w.t1 <= w.t0 || w.cnt <= w.mt || piece_dense(P, w)) return 0;
    return (w.cnt - w.mt + P.n_mt - 1) / P.n_mt;
}

// Warps `part` of `n_parts` (whole warps), at the start of the kernel while the
// first tiles are in flight and before the first scores exist: this CTA's share
// of the KV write-back, both caches.  The CTAs of a group cover the same key
// tiles; the fresh rows whose positions fall in those tiles are written to the
// cache by the group's CTA mt = (row's rank mod n_mt).  The candidate rows of all
// pieces are laid end to end and dealt one per lane, so a round costs two round
// trips (the index, then the K and V rows, 16-byte chunks, a whole row per lane).
// Nothing in this kernel reads a fresh row from the cache (each landed tile is
// patched from the fresh tensor), so the copies need no ordering against the
// loads.
template <int D, bool kSeeds>
__device__ void write_back_share(const Params &P, int part, int n_parts)
{
    constexpr int kChunks = D / 8;
    const int lane = threadIdx.x & 31;
    const int64_t row_elems = static_cast<int64_t>(P.Hkv) * D;
    const Range r = my_range(P);
    for (int f0 = part * 32;; f0 += n_parts * 32) {
        // this lane's candidate: piece k, row j
        int f = f0 + lane, j = -1, k = 0;
        Piece w;
        for (; k < r.count; ++k) {
            w = piece_at(P, r, k);  // inactive pieces included: their rows are shared too
            const int n = share_rows(P, w);
            if (f < n) {
                j = w.mt + f * P.n_mt;
                break;
            }
            f -= n;
        }
        if (!__any_sync(0xffffffffu, j >= 0)) break;
        int p = -1;
        if (j >= 0) {
            p = __ldg(P.idx + static_cast<int64_t>(w.b) * P.idx_stride + j);
            if (p < w.t0 * kBlockN || p >= min(w.t1 * kBlockN, P.L)) p = -1;
            // a seed's position keeps the cached K/V (COVER's override)
            if constexpr (kSeeds)
                if (__ldg(P.seed + static_cast<int64_t>(w.b) * P.r_max + j)) p = -1;
        }
        if (p >= 0) {
            const int64_t src = (static_cast<int64_t>(w.b) * P.r_max + j) * row_elems + w.g * D;
            const int64_t dst = (static_cast<int64_t>(w.b) * P.L + p) * row_elems + w.g * D;
            const uint4 *ks = reinterpret_cast<const uint4 *>(P.k_new + src);
            const uint4 *vs = reinterpret_cast<const uint4 *>(P.v_new + src);
            uint4 xk[kChunks], xv[kChunks];
#pragma unroll
            for (int c = 0; c < kChunks; ++c) xk[c] = __ldg(ks + c);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) xv[c] = __ldg(vs + c);
            uint4 *kd = reinterpret_cast<uint4 *>(P.k_cache + dst);
            uint4 *vd = reinterpret_cast<uint4 *>(P.v_cache + dst);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) kd[c] = xk[c];
#pragma unroll
            for (int c = 0; c < kChunks; ++c) vd[c] = xv[c];
        }
    }
}

// QK issuer warp: per piece Q into TMEM; then per tile, once its K tile landed,
// the whole warp patches the fresh K rows into it, and one thread issues
// S = Q K^T into one of the two S buffers once the PV product of the tile two
// back (which read its P from that buffer) completed.
template <int D, bool kSeeds>
__device__ void qk_issuer(const Params &P, const Sync &S, uint32_t sbase, uint32_t tmem, uint8_t *rows,
                          const CUtensorMap *tm_kn, const CUtensorMap *tm_k)
{
    using C = Cfg<D>;
    constexpr uint32_t kIdescQK = idesc_bf16(kBlockM, kBlockN, false, false);
    const int lane = threadIdx.x & 31;
    const Range r = my_range(P);
    Patch<D, kSeeds> pt;
    pt.init(B_KPATCH, rows, tm_kn, tm_k);
    uint32_t T = 0, it = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        const int qb = it % C::kQBufs;
        if (lane == 0) {
            ok = S.wait(B_QFULL + qb, (it / C::kQBufs) & 1);
            if (ok) {
                tc_fence_after();
                // Q into TMEM once per piece (after the previous piece's last QK, in
                // issue order); its shared-memory buffer is free for the next
                // piece's Q after that
                const uint32_t qbase = sbase + C::kOffQ + qb * C::kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tmem_copy_128x256b(tmem + C::kColQ + kk * 8,
                                       desc_sw128(qbase + (kk >> 2) * C::kCol + (kk & 3) * 32, 16, 1024));
                umma_commit(S.bar(B_QEMPTY + qb));
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        pt.start(P, w, true);
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int s = T % C::kKStages, sb = T & 1;
            ok = __all_sync(0xffffffffu, S.wait(B_KFULL + s, (T / C::kKStages) & 1));
            if (!ok) break;
            const uint32_t kbase = sbase + C::kOffK + s * C::kTile;
            ok = pt.tile(P, S, w, t, kbase, false);
            if (!ok) break;
            if (lane == 0) {
                if (T >= 2) ok = S.wait(B_SFREE + sb, ((T >> 1) - 1) & 1);
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // Q from TMEM, K from shared memory
                        const uint32_t off = (kk >> 2) * C::kCol + (kk & 3) * 32;
                        umma_bf16_ts(tmem + C::kColS + sb * kBlockN, tmem + C::kColQ + kk * 8,
                                     desc_sw128(kbase + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(S.bar(B_SFULL + sb));
                    umma_commit(S.bar(B_KEMPTY + s));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
        ++it;
    }
    if (lane == 0) {
        // everything issued has completed before TMEM is released
        umma_commit(S.bar(B_DRAIN));
        S.drain(B_DRAIN, 0);
        pt.drain(S);
        if (pt.stored) bulk_wait_all();
    }
    __syncwarp();
}

// PV issuer warp: per tile, once its V tile landed the whole warp patches the
// fresh V rows into it, and one thread issues O (+)= P V once the softmax warps
// wrote P over its S buffer; the first tile of a piece overwrites O.  The
// product's completion frees the V stage and the S buffer.
template <int D, bool kSeeds>
__device__ void pv_issuer(const Params &P, const Sync &S, uint32_t sbase, uint32_t tmem, uint8_t *rows,
                          const CUtensorMap *tm_vn, const CUtensorMap *tm_v)
{
    using C = Cfg<D>;
    constexpr uint32_t kIdescPV = idesc_bf16(kBlockM, D, false, true);
    const int lane = threadIdx.x & 31;
    const Range r = my_range(P);
    Patch<D, kSeeds> pt;
    pt.init(B_VPATCH, rows, tm_vn, tm_v);
    uint32_t T = 0;
    bool ok = true;
    for (int k = 0; k < r.count && ok; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        pt.start(P, w, false);
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int s = T % C::kVStages, sb = T & 1;
            ok = __all_sync(0xffffffffu, S.wait(B_VFULL + s, (T / C::kVStages) & 1));
            if (!ok) break;
            const uint32_t vbase = sbase + C::kOffV + s * C::kTile;
            ok = pt.tile(P, S, w, t, vbase, true);
            if (!ok) break;
            if (lane == 0) {
                ok = S.wait(B_PFULL + sb, (T >> 1) & 1);
                if (ok) {
                    tc_fence_after();
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
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
    }
    if (lane == 0) {
        umma_commit(S.bar(B_DRAIN2));
        S.drain(B_DRAIN2, 0);
        pt.drain(S);
        if (pt.stored) bulk_wait_all();
    }
    __syncwarp();
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
__device__ __forceinline__ void softmax_sync()
{
    asm volatile("bar.sync %0, %1;" ::"n"(kSoftmaxBarrier), "n"(kSoftmaxThreads) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
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

// The owner of a split unit waits until its contributors released their
// partials (bounded; a timeout aborts the CTA like any other wait).  All four
// softmax warps call it, whatever their own state (`ok` false: a wait of this
// warp already gave up), so all of them reach the named barrier.
__device__ bool wait_contributions(const Params &P, const Sync &S, int unit, int n, bool ok_in)
{
    __shared__ int s_ok;
    if (threadIdx.x == 64) {
        const uint32_t *f = P.flags + unit;
        const long long t0 = clock64();
        bool ok = ok_in && !*S.abort_flag;
        while (ok && ld_acquire(f) < static_cast<uint32_t>(n)) {
            if (*S.abort_flag) {
                ok = false;
                break;
            }
            if (clock64() - t0 > P.wait_limit) {
                ok = S.give_up();
                break;
            }
            __nanosleep(64);
        }
        s_ok = ok;
        if (ok) P.flags[unit] = 0;  // ready for the next launch (no contributor touches it again)
    }
    softmax_sync();
    __threadfence();  // every thread reads the partials after the acquire
    return s_ok != 0;
}

// Softmax warps: 8 of them, two per quarter of the 128 TMEM lanes.  The warp of
// half 0 (warps 2-5) takes score columns 0-63 of its 32 rows, the warp of half 1
// (warps 8-11) columns 64-127, so two warps of each SM sub-partition share the
// exponentials and hide each other's latencies.  The two halves of a row agree on
// the row maximum through shared memory (one pair barrier per tile) and so keep
// the same reference m; each keeps its own partial row sum and its own half of
// O's columns, and the halves' sums are added at the end of a piece.
__device__ __forceinline__ void pair_sync(int quarter)
{
    asm volatile("bar.sync %0, 64;" ::"r"(kPairBarrier0 + quarter) : "memory");
}

// Row maximum of half a tile's raw scores (four independent chains).
__device__ __forceinline__ float row_max64(const uint32_t (&sr)[2][32])
{
    float mx2[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        float a = __uint_as_float(sr[cc][0]), b = __uint_as_float(sr[cc][1]);
#pragma unroll
        for (int j = 2; j < 32; j += 4) {
            a = fmax3(a, __uint_as_float(sr[cc][j]), __uint_as_float(sr[cc][j + 1]));
            b = fmax3(b, __uint_as_float(sr[cc][j + 2]), __uint_as_float(sr[cc][j + 3]));
        }
        mx2[cc] = fmaxf(a, b);
    }
    return fmaxf(mx2[0], mx2[1]);
}

// p = 2^{y}, y = s c - m c, for half a tile's 64 scores: two-wide FMA and adds
// into four partial sums, P packed as bf16 pairs.
__device__ __forceinline__ void exp_half(const uint32_t (&sr)[2][32], uint64_t c2, float nmc,
                                         uint64_t (&acc2)[4], uint32_t (&pk)[32])
{
    const uint64_t nmc2 = f2x2(nmc, nmc);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc2[k] = 0ull;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const uint64_t y2 =
                ffma2(f2x2(__uint_as_float(sr[cc][j]), __uint_as_float(sr[cc][j + 1])), c2, nmc2);
            float y0, y1;
            x2f(y2, y0, y1);
            const float p0 = ex2(y0), p1 = ex2(y1);
            acc2[(j >> 1) & 3] = fadd2(acc2[(j >> 1) & 3], f2x2(p0, p1));
            pk[(cc * 32 + j) >> 1] = pack_bf16x2(p0, p1);
        }
    }
}

// SimSD's temporal causal mask as label windows.  Every key gets one integer
// label and every query a closed window; the key is visible to the query when
// its label lies in the window:
//   key   prompt 0          data tau            mask slot tau - 2^30
//   query prompt [0, 0]      data [0, tau]       mask slot [tau - 2^30, tau - 1]
// A mask slot's window holds the prompt, the data labels below its own step and
// the slot labels of its step and later ones; a data token's holds the prompt and
// the data labels up to its own step; a prompt token's only the prompt.  Labels
// must lie in [1, 2^30): anything else marks the key hidden (and the query's
// window empty) and raises EC_DEV_BAD_LABEL.
constexpr int kSlotBase = 1 << 30;

__device__ __forceinline__ int simsd_key_label(const Params &P, int b, int j, bool &bad)
{
    const int64_t o = static_cast<int64_t>(b) * P.L + j;
    const int sec = __ldg(P.section + o);
    if (sec == 0) return 0;
    const int t = __ldg(P.tau + o);
    if (sec > 2 || t < 1 || t >= kSlotBase) {
        bad = true;
        return INT_MIN;
    }
    return sec == 1 ? t : t - kSlotBase;
}

__device__ __forceinline__ int2 simsd_window(const Params &P, int b, int pos, bool &bad)
{
    if (pos < 0 || pos >= P.L) return make_int2(1, 0);  // an index the K side flags
    const int64_t o = static_cast<int64_t>(b) * P.L + pos;
    const int sec = __ldg(P.section + o);
    if (sec == 0) return make_int2(0, 0);
    const int t = __ldg(P.tau + o);
    if (sec > 2 || t < 1 || t >= kSlotBase) {
        bad = true;
        return make_int2(1, 0);
    }
    return sec == 1 ? make_int2(0, t) : make_int2(t - kSlotBase, t - 1);
}

template <int D, int kMode>
__device__ void softmax_epilogue(const Params &P, const Sync &S, uint32_t tmem, float *xchg)
{
    constexpr bool kSimSD = kMode == MODE_SIMSD, kCover = kMode == MODE_COVER;
    constexpr bool kMasked = kMode != MODE_PLAIN;  // some score may be hidden
    using C = Cfg<D>;
    constexpr int kOChunks = D / 64;  // 32-column chunks of O per half
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = warp >= 8 ? 1 : 0;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float *x_own = xchg + half * kBlockM + row;
    const float *x_other = xchg + (1 - half) * kBlockM + row;
    const float c = P.scale_log2;  // log2 units per raw score unit
    const int kv_tail = P.L - (P.n_tiles - 1) * kBlockN;  // keys in the last tile
    const Range r = my_range(P);
    uint32_t T = 0;
    bool ok = true;
    // After a failed (timed-out) wait a warp skips all further work; every later
    // wait of any role returns at once (the abort flag is set).  Both warps of a
    // pair always reach the same pair barriers.
    for (int k = 0; k < r.count; ++k) {
        const Piece w = piece_at(P, r, k);
        if (!piece_active(P, w)) continue;
        float m_run = -INFINITY, l_run = 0.f;  // m in raw score units; l of this half
        int2 win = make_int2(INT_MIN, INT_MAX);  // rows past the unit's tokens see all
        bool bad_label = false;
        int own = -1;  // COVER: a seed row's own position, whose cached key it must not see
        if constexpr (kMasked) {
            const int tok = w.mt * P.tok_per_tile + row / P.G;
            if (row < P.tok_per_tile * P.G && tok < w.cnt) {
                const int pos = __ldg(P.idx + w.b * P.idx_stride + tok);
                if constexpr (kSimSD) win = simsd_window(P, w.b, pos, bad_label);
                if constexpr (kCover)
                    if (__ldg(P.seed + static_cast<int64_t>(w.b) * P.r_max + tok)) own = pos;
            }
        }
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int sb = T & 1;
            // the labels of this half's 64 keys (two per lane) and their range,
            // loaded while the product runs
            int lab0 = 0, lab1 = 0, lab_lo = 0, lab_hi = 0;
            if constexpr (kSimSD) {
                const int j0 = t * kBlockN + half * 64 + lane;
                const bool in0 = j0 < P.L, in1 = j0 + 32 < P.L;
                if (in0) lab0 = simsd_key_label(P, w.b, j0, bad_label);
                if (in1) lab1 = simsd_key_label(P, w.b, j0 + 32, bad_label);
                lab_lo = __reduce_min_sync(0xffffffffu, min(in0 ? lab0 : INT_MAX, in1 ? lab1 : INT_MAX));
                lab_hi = __reduce_max_sync(0xffffffffu, max(in0 ? lab0 : INT_MIN, in1 ? lab1 : INT_MIN));
            }
            if (ok) ok = __all_sync(0xffffffffu, S.wait(B_SFULL + sb, (T >> 1) & 1));
            tc_fence_after();
            const uint32_t scol = tmem + lane_off + C::kColS + sb * kBlockN + half * 64;
            uint32_t sr[2][32];
            float pmax = -INFINITY;
            if (ok) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) tmem_ld32(scol + cc * 32, sr[cc]);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) tmem_wait_ld(sr[cc]);
                const int live = kv_tail - half * 64;  // keys of this half in the last tile
                if (t == P.n_tiles - 1 && live < 64) {  // keys past L do not exist
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (cc * 32 + j >= live) sr[cc][j] = __float_as_uint(-INFINITY);
                }
                if constexpr (kCover) {
                    // a seed row hides the cached key at its own position (the
                    // diagonal term is added from its masked-input K/V at the end)
                    const int col = own - (t * kBlockN + half * 64);
                    if (col >= 0 && col < 64) {
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (cc * 32 + j == col) sr[cc][j] = __float_as_uint(-INFINITY);
                    }
                }
                if constexpr (kSimSD) {
                    // a row whose window misses part of the keys' label range
                    // hides those keys; the labels go round the warp
                    const bool all_in = win.x <= lab_lo && lab_hi <= win.y;
                    if (__any_sync(0xffffffffu, !all_in)) {
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int lab = __shfl_sync(0xffffffffu, cc ? lab1 : lab0, j);
                                if (lab < win.x || lab > win.y) sr[cc][j] = __float_as_uint(-INFINITY);
                            }
                    }
                }
                pmax = row_max64(sr);  // scale > 0 keeps the order
            }
            // the row maximum from both halves (the partner read our previous value
            // before the first barrier)
            pair_sync(quarter);
            *x_own = pmax;
            pair_sync(quarter);
            const float mx = fmaxf(pmax, *x_other);
            if (!ok) continue;
            // The reference m moves only when a score exceeds it by more than 8 in
            // log2 units (then O is rescaled once the previous PV product is done);
            // both halves take the same decision.
            float m_use = m_run, alpha = 1.f;
            bool rescale = false;
            if ((mx - m_run) * c > 8.f) {
                m_use = mx;
                alpha = ex2((m_run - mx) * c);
                rescale = t > w.t0;
            }
            uint64_t acc2[4];
            uint32_t pk[32];
            float nmc = -m_use * c;
            if constexpr (kMasked)
                if (m_use == -INFINITY) nmc = 0.f;  // every key so far hidden: all p = 0
            exp_half(sr, f2x2(c, c), nmc, acc2, pk);
            // P (bf16 pairs) over the first half of this S buffer, where the PV
            // product reads it: this half's 64 probabilities in 32 columns
            tmem_st32(tmem + lane_off + C::kColS + sb * kBlockN + half * 32, pk);
            float rs0, rs1, rs2, rs3, rs4, rs5, rs6, rs7;
            x2f(acc2[0], rs0, rs1);
            x2f(acc2[1], rs2, rs3);
            x2f(acc2[2], rs4, rs5);
            x2f(acc2[3], rs6, rs7);
            const float rowsum = ((rs0 + rs1) + (rs2 + rs3)) + ((rs4 + rs5) + (rs6 + rs7));
            l_run = l_run * alpha + rowsum;
            m_run = m_use;

            // O may be rescaled only after the previous tile's PV product completed
            // (the completion that freed the other S buffer); each half its columns
            if (rescale) {
                const uint32_t Tp = T - 1;
                ok = __all_sync(0xffffffffu, S.wait(B_SFREE + (Tp & 1), (Tp >> 1) & 1));
                if (!ok) continue;
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < kOChunks; ++cc) {
                    uint32_t o[32];
                    const uint32_t ta = tmem + lane_off + C::kColO + (half * kOChunks + cc) * 32;
                    tmem_ld32(ta, o);
                    tmem_wait_ld(o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(ta, o);
                }
            }
            // the P stores (and any O correction) complete before the PV product reads them
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
        if constexpr (kSimSD)
            if (__any_sync(0xffffffffu, bad_label) && lane == 0) flag_status(P.status, EC_DEV_BAD_LABEL);
        // the row sum of both halves (same reference m)
        pair_sync(quarter);
        *x_own = l_run;
        pair_sync(quarter);
        const float l_row = l_run + *x_other;
        const int tok = w.mt * P.tok_per_tile + row / P.G;
        const bool valid = row < P.tok_per_tile * P.G && tok < w.cnt;
        const int h = w.g * P.G + row % P.G;
        __nv_bfloat16 *orow = P.out + ((static_cast<int64_t>(w.b) * P.r_max + tok) * P.H + h) * D;
        if (w.role == ROLE_CONTRIB) {
            // a partial for the unit's owner: unnormalised O and (m, l), then the flag
            if (ok) {
                float4 *po = P.part_o + (static_cast<int64_t>(w.unit) * P.slots + w.slot) * (D / 4) * kBlockM;
#pragma unroll 1
                for (int cc = half * kOChunks; cc < (half + 1) * kOChunks; ++cc) {
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
                if (valid && half == 0)
                    __stcg(P.part_ml + (static_cast<int64_t>(w.unit) * P.slots + w.slot) * kBlockM + row,
                           make_float2(m_run, l_row));
                __threadfence();
            }
            tc_fence_before();
            softmax_sync();
            // released only when every softmax warp wrote its rows: a warp that gave
            // up raised the CTA's abort flag before the barrier
            if (ok && threadIdx.x == 64 && !*S.abort_flag) red_release_add(P.flags + w.unit, 1u);
            continue;
        }
        // whole unit or owner: out = (wo O + sum_s ws_s O_s) / (wo l + sum_s ws_s l_s),
        // every term scaled to M, the largest of the maxima; each half its columns
        int n = 0;
        if (w.role == ROLE_OWNER) {
            ok = wait_contributions(P, S, w.unit, w.n_contrib, ok);  // every softmax warp
            n = min(w.n_contrib, kMaxContrib);
        }
        if (!ok) continue;
        const float2 *mlp = P.part_ml + static_cast<int64_t>(w.unit) * P.slots * kBlockM + row;
        const float4 *pop = P.part_o + static_cast<int64_t>(w.unit) * P.slots * (D / 4) * kBlockM + row;
        auto weight = [&](int s, float M, float &ls) {  // contributor s's scale and its l
            const float2 v = valid ? ld_cg_v2(mlp + static_cast<int64_t>(s) * kBlockM)
                                   : make_float2(-INFINITY, 0.f);
            ls = v.y;
            return v.y > 0.f ? ex2((v.x - M) * c) : 0.f;
        };
        float M = m_run;
        for (int s = 0; s < n; ++s)
            if (valid) M = fmaxf(M, ld_cg_v2(mlp + static_cast<int64_t>(s) * kBlockM).x);
        const float wo = l_row > 0.f ? ex2((m_run - M) * c) : 0.f;
        float l = wo * l_row;
        for (int s = 0; s < n; ++s) {
            float ls;
            const float ws = weight(s, M, ls);
            l = fmaf(ws, ls, l);
        }
        // COVER: a seed row's diagonal term from its masked-input K/V, s = q . k_new
        // (raw units, both halves alike): O and l are rescaled to M2 = max(M, s)
        // and gain 2^{(s - M2) c} v_new and 2^{(s - M2) c}
        float f_old = 1.f, p_new = 0.f;
        const __nv_bfloat16 *vrow = nullptr;
        if constexpr (kCover) {
            if (valid && own >= 0) {
                const int64_t kv = ((static_cast<int64_t>(w.b) * P.r_max + tok) * P.Hkv + w.g) * D;
                const uint4 *qv = reinterpret_cast<const uint4 *>(P.q + ((static_cast<int64_t>(w.b) * P.r_max + tok) * P.H + h) * D);
                const uint4 *kn = reinterpret_cast<const uint4 *>(P.k_new + kv);
                float dot = 0.f;
#pragma unroll 4
                for (int u = 0; u < D / 8; ++u) {
                    const uint4 a = __ldg(qv + u), b = __ldg(kn + u);
                    dot = fmaf_bf16x2(a.x, b.x, dot);
                    dot = fmaf_bf16x2(a.y, b.y, dot);
                    dot = fmaf_bf16x2(a.z, b.z, dot);
                    dot = fmaf_bf16x2(a.w, b.w, dot);
                }
                const float M2 = fmaxf(M, dot);
                f_old = l > 0.f ? ex2((M - M2) * c) : 0.f;
                p_new = ex2((dot - M2) * c);
                l = fmaf(l, f_old, p_new);
                vrow = P.v_new + kv;
            }
        }
        const float inv = kMasked ? (l > 0.f ? 1.f / l : 0.f) : 1.f / l;  // no visible key: zeros
#pragma unroll 1
        for (int cc = half * kOChunks; cc < (half + 1) * kOChunks; ++cc) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + C::kColO + cc * 32, o);
            tmem_wait_ld(o);
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(o[j]) * wo;
            for (int s = 0; s < n; ++s) {
                float ls;
                const float ws = weight(s, M, ls);
                const float4 *po = pop + (static_cast<int64_t>(s) * (D / 4) + cc * 8) * kBlockM;
                if (valid) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 x = ld_cg_v4(po + q * kBlockM);
                        acc[4 * q] = fmaf(ws, x.x, acc[4 * q]);
                        acc[4 * q + 1] = fmaf(ws, x.y, acc[4 * q + 1]);
                        acc[4 * q + 2] = fmaf(ws, x.z, acc[4 * q + 2]);
                        acc[4 * q + 3] = fmaf(ws, x.w, acc[4 * q + 3]);
                    }
                }
            }
            if constexpr (kCover) {
                if (vrow) {
                    const uint4 *vv = reinterpret_cast<const uint4 *>(vrow + cc * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 x = __ldg(vv + q);
                        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = bf16x2_to_f2(xs[e]);
                            acc[8 * q + 2 * e] = fmaf(acc[8 * q + 2 * e], f_old, p_new * f.x);
                            acc[8 * q + 2 * e + 1] = fmaf(acc[8 * q + 2 * e + 1], f_old, p_new * f.y);
                        }
                    }
                }
            }
            if (valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 v;
                    v.x = pack_bf16x2(acc[8 * q] * inv, acc[8 * q + 1] * inv);
                    v.y = pack_bf16x2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv);
                    v.z = pack_bf16x2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv);
                    v.w = pack_bf16x2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv);
                    dst[q] = v;
                }
            }
        }
        tc_fence_before();
    }
}

template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const Params P, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_kn,
                        const __grid_constant__ CUtensorMap tm_vn)
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
            mbar_init(S.bar(i), (i == B_PFULL || i == B_PFULL + 1) ? 8u : 1u);
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
        prefetch_tmap(&tm_kn);
        prefetch_tmap(&tm_vn);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // inputs and outputs belong to the previous kernel until here

    if (warp == 0 || warp == 6) {
        if ((threadIdx.x & 31) == 0) {
            if (warp == 0)
                producer_qk<D>(P, S, sbase, &tm_q, &tm_k, &tm_kn);
            else
                producer_v<D>(P, S, sbase, &tm_v, &tm_vn);
        }
        __syncwarp();
    } else if (warp == 1) {
        qk_issuer<D, kMode == MODE_COVER>(P, S, sbase, tmem, smem + C::kOffRows, &tm_kn, &tm_k);
    } else if (warp == 7) {
        pv_issuer<D, kMode == MODE_COVER>(P, S, sbase, tmem, smem + C::kOffRows + 128, &tm_vn, &tm_v);
    } else {
        // the eight softmax warps: the write-back share while the first scores are
        // being produced, then the softmax
        write_back_share<D, kMode == MODE_COVER>(P, warp < 8 ? warp - 2 : warp - 4, 8);
        softmax_epilogue<D, kMode>(P, S, tmem, reinterpret_cast<float *>(smem + C::kOffXchg));
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

// [B, rows_alloc, heads, D] bf16 viewed as 4-D {D, heads, rows, B} with only the
// first `rows` rows of every batch entry addressable; box {64, box_heads,
// box_rows, 1}, 128-byte swizzle; out-of-range elements load as zero and are not
// stored.
bool encode_4d(CUtensorMap *map, const void *base, int B, int rows, int rows_alloc, int heads, int D,
               int box_heads, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(heads) * D * 2,
                                   static_cast<cuuint64_t>(rows_alloc) * heads * D * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_heads),
                               static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int G, tok_per_tile, n_mt, n_units, n_tiles, grid, slots, grouped, n_groups;
    int64_t total;
};

// The work split.  Groups of n_mt CTAs (one per unit of a (b, g)) take equal
// contiguous ranges of the (b, g, key tile) pairs, so every CTA does the same
// number of tiles and a group's CTAs share each K/V tile through L2.  When a
// (b, g) has more units than half the SMs, or a unit would need more than
// kMaxContrib contributors, whole units are dealt round-robin instead.
Plan make_plan(int B, int L, int r_max, int H, int Hkv)
{
    Plan p;
    p.G = H / Hkv;
    p.tok_per_tile = kBlockM / p.G;
    p.n_mt = (r_max + p.tok_per_tile - 1) / p.tok_per_tile;
    p.n_units = B * Hkv * p.n_mt;
    p.n_tiles = (L + kBlockN - 1) / kBlockN;
    p.total = static_cast<int64_t>(B) * Hkv * p.n_tiles;
    const int n_sm = device_sm_count();
    p.slots = 0;
    p.grouped = 0;
    p.n_groups = 0;
    if (p.n_mt >= 1 && 2 * p.n_mt <= n_sm) {
        const int n_groups = static_cast<int>(std::min<int64_t>(n_sm / p.n_mt, p.total));
        // most contributors of one (b, g): groups meeting it, its owner excluded
        auto grp = [&](int64_t w) { return ((w + 1) * n_groups - 1) / p.total; };
        int64_t worst = 0;
        for (int64_t bg = 0; bg < static_cast<int64_t>(B) * Hkv; ++bg)
            worst = std::max<int64_t>(worst, grp(bg * p.n_tiles + p.n_tiles - 1) - grp(bg * p.n_tiles));
        if (worst <= kMaxContrib) {
            p.grouped = 1;
            p.n_groups = n_groups;
            p.slots = static_cast<int>(worst);  // 0: no unit is cut, no partials
        }
    }
    p.grid = p.grouped ? p.n_groups * p.n_mt : std::max(1, std::min(n_sm, p.n_units));
    return p;
}

void partial_offsets(const Plan &p, int D, size_t *off_flags, size_t *off_ml, size_t *off_o,
                     size_t *end)
{
    size_t off = kWsHeader;
    *off_flags = off;
    off = align_up(off + static_cast<size_t>(p.n_units) * sizeof(uint32_t), 256);
    *off_ml = off;
    const size_t parts = p.grouped ? static_cast<size_t>(p.n_units) * p.slots : 0;
    off = align_up(off + parts * kBlockM * sizeof(float2), 256);
    *off_o = off;
    *end = off + parts * kBlockM * static_cast<size_t>(D) * sizeof(float);
}

template <int D>
cudaError_t launch_typed(const Params &p, const Plan &plan, const void *q, cudaStream_t stream)
{
    CUtensorMap tq, tk, tv, tkn, tvn;
    // the fresh K/V are viewed with at most L rows, so that rows at or past L
    // (present only when r_max > L) read as zero
    const int fresh_rows = std::min(p.L, p.r_max);
    if (!encode_4d(&tq, q, p.B, p.r_max, p.r_max, p.H, D, p.G, p.tok_per_tile) ||
        !encode_4d(&tk, p.k_cache, p.B, p.L, p.L, p.Hkv, D, 1, kBlockN) ||
        !encode_4d(&tv, p.v_cache, p.B, p.L, p.L, p.Hkv, D, 1, kBlockN) ||
        !encode_4d(&tkn, p.k_new, p.B, fresh_rows, p.r_max, p.Hkv, D, 1, kBlockN) ||
        !encode_4d(&tvn, p.v_new, p.B, fresh_rows, p.r_max, p.Hkv, D, 1, kBlockN))
        return cudaErrorInvalidValue;
    if (p.section)
        return launch(attention_tc_kernel<D, MODE_SIMSD>, dim3(plan.grid), dim3(kThreads),
                      Cfg<D>::kBytes, stream, p, tq, tk, tv, tkn, tvn);
    if (p.seed)
        return launch(attention_tc_kernel<D, MODE_COVER>, dim3(plan.grid), dim3(kThreads),
                      Cfg<D>::kBytes, stream, p, tq, tk, tv, tkn, tvn);
    return launch(attention_tc_kernel<D, MODE_PLAIN>, dim3(plan.grid), dim3(kThreads), Cfg<D>::kBytes,
                  stream, p, tq, tk, tv, tkn, tvn);
}

}  // namespace

bool attention_tc_supported(int dtype, int32_t seq_len, int32_t head_dim)
{
    return dtype == EC_BF16 && (head_dim == 64 || head_dim == 128) && seq_len >= 1;
}

int32_t attention_tc_kernel_count(int32_t, int32_t, int32_t, int32_t, int32_t) { return 1; }

size_t attention_tc_workspace_bytes(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                    int32_t n_kv_heads, int32_t head_dim)
{
    if (batch < 1 || seq_len < 1 || r_max < 1 || n_kv_heads < 1 || n_heads < n_kv_heads)
        return kWsHeader;
    const Plan p = make_plan(batch, seq_len, r_max, n_heads, n_kv_heads);
    size_t a, b, c, end;
    partial_offsets(p, head_dim, &a, &b, &c, &end);
    return end;
}

cudaError_t launch_attention_tc(const void *q, const void *k_new, const void *v_new,
                                const int32_t *idx, int64_t idx_stride, const int32_t *count,
                                void *k_cache, void *v_cache, void *out, int32_t batch,
                                int32_t seq_len, int32_t r_max, int32_t n_heads,
                                int32_t n_kv_heads, int32_t head_dim, float scale,
                                void *workspace, cudaStream_t stream, const uint8_t *section,
                                const int32_t *tau, const uint8_t *seed)
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
    p.grouped = plan.grouped;
    p.n_groups = plan.n_groups;
    p.total = plan.total;
    p.slots = plan.slots;
    p.scale_log2 = scale * kLog2e;
    char *ws = static_cast<char *>(workspace);
    size_t o_f, o_ml, o_o, end;
    partial_offsets(plan, head_dim, &o_f, &o_ml, &o_o, &end);
    p.status = reinterpret_cast<uint32_t *>(ws);
    p.wait_limit = wait_limit_cycles();
    p.flags = reinterpret_cast<uint32_t *>(ws + o_f);
    p.part_ml = reinterpret_cast<float2 *>(ws + o_ml);
    p.part_o = reinterpret_cast<float4 *>(ws + o_o);
    p.section = section;
    p.tau = tau;
    p.seed = seed;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    return head_dim == 128 ? launch_typed<128>(p, plan, q, stream)
                           : launch_typed<64>(p, plan, q, stream);
}

}  // namespace ec
