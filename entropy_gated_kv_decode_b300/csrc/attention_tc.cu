// Selective-recompute bidirectional attention on the 5th-generation tensor
// cores (tcgen05 + TMEM), fed by TMA, with the KV write-back fused into the
// kernel's prologue.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, section "1. Il Problema" (dLLM attention is
// bidirectional) and "Algoritmo di Funzionamento" step 2 (the partial forward
// recomputes K/V only for the selected tokens; the cache supplies the rest).
//
// Persistent cooperative kernel, one CTA per SM:
//   prologue   every CTA writes a share of the fresh K/V rows into the caches,
//              then one bounded grid barrier; afterwards the caches hold the
//              post-write-back state and every K/V tile is a plain TMA load.
//   work items a unit is up to 128 query rows of one (sequence b, KV head g): the
//              (recomputed row r, head h of g's group) pairs packed r-major, so a
//              GQA group shares each K/V tile.  A unit's keys are split into
//              `n_split` contiguous ranges of 128-key tiles; (unit, split) items
//              are dealt round-robin to the CTAs.  A split's partial (O, m, l)
//              goes to the workspace, and the last split of a unit to finish
//              (an atomic ticket: no CTA waits on another) merges them.
//   warp 0     producer of Q (one tile per item) and K tiles, warp 6 producer of
//              V tiles: TMA loads with 128-byte swizzle into rings of stages; a K
//              stage is released as soon as its QK product completes and a V
//              stage when its PV product does, so K loads run well ahead;
//   warp 1     TMEM allocation and tcgen05.mma issue: S = Q K^T into one of two
//              TMEM S buffers, O += P V into the TMEM O accumulator;
//   warps 2-5  one thread per query row: online softmax on S read by tcgen05.ld
//              in the log2 domain (the reference maximum only moves when it grows
//              by more than 8, rescaling O in TMEM when it does), P as bf16 into
//              shared memory, and the epilogue.
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
constexpr int kThreads = 224;  // 7 warps
constexpr int kMaxSplit = 32;

template <int D>
struct Cfg {
    static constexpr uint32_t kTile = kBlockM * D * 2;  // bytes of one Q / K / V tile
    static constexpr uint32_t kCol = kBlockM * 128;     // one 64-element column: 16 KB
    // stage counts: 1 Q + 3 K + 2 V (+ P) fill 224 KB at D = 128
    static constexpr int kQBufs = D == 128 ? 1 : 2;
    static constexpr int kKStages = D == 128 ? 3 : 4;
    static constexpr int kVStages = D == 128 ? 2 : 3;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kQBufs * kTile;
    static constexpr uint32_t kOffV = kOffK + kKStages * kTile;
    static constexpr uint32_t kOffP = kOffV + kVStages * kTile;
    static constexpr uint32_t kOffBar = kOffP + kBlockM * kBlockN * 2;
    static constexpr uint32_t kOffMisc = kOffBar + 256;
    static constexpr uint32_t kBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;    // two S buffers: columns [0, 128) and [128, 256)
    static constexpr uint32_t kColO = 256;  // O: columns [256, 256 + D)
};

enum : int {
    B_KFULL = 0,    // [4] K tile landed
    B_KEMPTY = 4,   // [4] K stage consumed (its QK done)
    B_VFULL = 8,    // [3] V tile landed
    B_VEMPTY = 11,  // [3] V stage consumed (its PV done)
    B_QFULL = 14,   // [2] Q tile landed
    B_QEMPTY = 16,  // [2] Q tile consumed (last QK of its item done)
    B_SFULL = 18,   // [2] S buffer written
    B_SFREE = 20,   // [2] S buffer read by the softmax warps
    B_PFULL = 22,   // P written, O corrected
    B_PVDONE = 23,
    B_DRAIN = 24,
    B_COUNT = 25
};

// Workspace header words (the first 256 bytes of the workspace).
constexpr int kHdrStatus = 0, kHdrBarCount = 2, kHdrBarGen = 3;

struct Params {
    const __nv_bfloat16 *k_new, *v_new;
    __nv_bfloat16 *k_cache, *v_cache, *out;
    const int32_t *idx;
    int64_t idx_stride;
    const int32_t *count;
    int B, L, r_max, H, Hkv, G;
    int tok_per_tile;  // recomputed rows per unit: floor(128 / G)
    int n_mt;          // units per (b, g)
    int n_units, n_split, n_items, n_tiles;
    float scale_log2;
    uint32_t *hdr;      // workspace header
    unsigned *tickets;  // [n_units]
    float2 *part_ml;    // [n_items][128] (m, l), log2 domain
    float4 *part_o;     // [n_items][D / 4][128] unnormalised O
};

struct Item {
    int unit, split, b, g, mt, t0, t1, cnt;
};

__device__ __forceinline__ Item decode_item(const Params &P, int i)
{
    Item it;
    it.unit = i % P.n_units;
    it.split = i / P.n_units;
    it.mt = it.unit % P.n_mt;
    it.g = (it.unit / P.n_mt) % P.Hkv;
    it.b = it.unit / (P.n_mt * P.Hkv);
    it.t0 = static_cast<int>(static_cast<int64_t>(P.n_tiles) * it.split / P.n_split);
    it.t1 = static_cast<int>(static_cast<int64_t>(P.n_tiles) * (it.split + 1) / P.n_split);
    it.cnt = max(0, min(__ldg(P.count + it.b), P.r_max));
    return it;
}

// Items with no recomputed rows (mt beyond the sequence's count) are skipped by
// every role alike.
__device__ __forceinline__ bool item_active(const Params &P, const Item &it)
{
    return it.mt * P.tok_per_tile < it.cnt && it.t1 > it.t0;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier for a cooperative launch (all CTAs co-resident).  Sense
// reversal on a generation word; bounded: returns false after ~2 s.
__device__ bool grid_barrier(uint32_t *hdr, unsigned n_ctas, volatile int *abort_flag)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t *count = hdr + kHdrBarCount;
        uint32_t *gen = hdr + kHdrBarGen;
        const uint32_t g0 = ld_acquire_u32(gen);
        __threadfence();
        const unsigned arrived = atomicAdd(count, 1u);
        int ok = 1;
        if (arrived == n_ctas - 1) {
            atomicExch(count, 0u);
            __threadfence();
            atomicAdd(gen, 1u);
        } else {
            const long long t0 = clock64();
            while (ld_acquire_u32(gen) == g0) {
                if (clock64() - t0 > kWaitCycles) {
                    flag_status(hdr + kHdrStatus, EC_DEV_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        s_ok = ok;
        if (!ok) *abort_flag = 1;
    }
    __syncthreads();
    return s_ok != 0;
}

// Q and K producer (one thread): per item its Q tile, then its K tiles.
template <int D>
__device__ void producer_qk(const Params &P, const Sync &S, uint32_t sbase, const CUtensorMap *tm_q,
                            const CUtensorMap *tm_k)
{
    using C = Cfg<D>;
    const uint32_t q_bytes = static_cast<uint32_t>(P.tok_per_tile * P.G) * D * 2;
    uint32_t T = 0, it = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < P.n_items && ok; i += gridDim.x) {
        const Item w = decode_item(P, i);
        if (!item_active(P, w)) continue;
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

// V producer (one thread): the V tiles of every item, in the same order.
template <int D>
__device__ void producer_v(const Params &P, const Sync &S, uint32_t sbase, const CUtensorMap *tm_v)
{
    using C = Cfg<D>;
    uint32_t T = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < P.n_items && ok; i += gridDim.x) {
        const Item w = decode_item(P, i);
        if (!item_active(P, w)) continue;
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

template <int D>
__device__ void mma_issuer(const Params &P, const Sync &S, uint32_t sbase, uint32_t tmem)
{
    using C = Cfg<D>;
    constexpr uint32_t kIdescQK = idesc_bf16(kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdescPV = idesc_bf16(kBlockM, D, false, true);
    uint32_t T = 0, it = 0;
    bool ok = true;
    // the PV product of the previous tile, issued after the next QK
    bool pv_pending = false, pv_first = false;
    uint32_t pv_T = 0;
    auto issue_pv = [&]() {
        const int s = pv_T % C::kVStages;
        ok = ok && S.wait(B_PFULL, pv_T & 1) && S.wait(B_VFULL + s, (pv_T / C::kVStages) & 1);
        if (!ok) return;
        tc_fence_after();
        const uint32_t vbase = sbase + C::kOffV + s * C::kTile;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
            const uint64_t a =
                desc_sw128(sbase + C::kOffP + (kk >> 2) * C::kCol + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = desc_sw128(vbase + kk * 16 * 128, C::kCol, 1024);
            umma_bf16(tmem + C::kColO, a, bd, kIdescPV, (!pv_first || kk > 0) ? 1u : 0u);
        }
        umma_commit(S.bar(B_VEMPTY + s));
        umma_commit(S.bar(B_PVDONE));
        pv_pending = false;
    };
    for (int i = blockIdx.x; i < P.n_items && ok; i += gridDim.x) {
        const Item w = decode_item(P, i);
        if (!item_active(P, w)) continue;
        const int qb = it % C::kQBufs;
        ok = S.wait(B_QFULL + qb, (it / C::kQBufs) & 1);
        if (!ok) break;
        const uint32_t qbase = sbase + C::kOffQ + qb * C::kTile;
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int s = T % C::kKStages, sb = T & 1;
            ok = S.wait(B_KFULL + s, (T / C::kKStages) & 1);
            if (ok && T >= 2) ok = S.wait(B_SFREE + sb, ((T >> 1) - 1) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kbase = sbase + C::kOffK + s * C::kTile;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * C::kCol + (kk & 3) * 32;
                umma_bf16(tmem + C::kColS + sb * kBlockN, desc_sw128(qbase + off, 16, 1024),
                          desc_sw128(kbase + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
            }
            umma_commit(S.bar(B_SFULL + sb));
            umma_commit(S.bar(B_KEMPTY + s));
            if (t == w.t1 - 1) umma_commit(S.bar(B_QEMPTY + qb));
            if (pv_pending) issue_pv();
            if (!ok) break;
            pv_pending = true;
            pv_first = t == w.t0;
            pv_T = T;
        }
        ++it;
    }
    if (ok && pv_pending) issue_pv();
    // everything issued has completed before TMEM is released
    umma_commit(S.bar(B_DRAIN));
    S.drain(B_DRAIN, 0);
}

template <int D>
__device__ void softmax_epilogue(const Params &P, const Sync &S, uint32_t sbase, uint32_t tmem)
{
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    __shared__ int s_last;
    uint32_t T = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < P.n_items && ok; i += gridDim.x) {
        const Item w = decode_item(P, i);
        if (!item_active(P, w)) continue;
        float m_run = -INFINITY, l_run = 0.f;
        for (int t = w.t0; t < w.t1; ++t, ++T) {
            const int sb = T & 1;
            ok = S.wait(B_SFULL + sb, (T >> 1) & 1);
            __syncwarp();  // reconverge before the warp-collective tcgen05.ld
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld32(tmem + lane_off + C::kColS + sb * kBlockN + c * 32, sr[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_wait_ld(sr[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.bar(B_SFREE + sb));

            const int kv_valid = min(kBlockN, P.L - t * kBlockN);
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float s = __uint_as_float(sr[c][j]) * P.scale_log2;
                    if (c * 32 + j >= kv_valid) s = -INFINITY;
                    sr[c][j] = __float_as_uint(s);
                    mx = fmaxf(mx, s);
                }
            float m_use = m_run, alpha = 1.f;
            bool rescale = false;
            if (mx > m_run + 8.f) {  // move the reference only when p could exceed 2^8
                m_use = mx;
                alpha = ex2(m_run - mx);
                rescale = t > w.t0;
            }
            float rowsum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float p0 = ex2(__uint_as_float(sr[c][j]) - m_use);
                    const float p1 = ex2(__uint_as_float(sr[c][j + 1]) - m_use);
                    rowsum += p0 + p1;
                    pk[(c * 32 + j) >> 1] = pack_bf16x2(p0, p1);
                }
            l_run = l_run * alpha + rowsum;
            m_run = m_use;

            // P buffer and O are free once the previous PV of this item completed
            // (for an item's first tile the previous epilogue already waited).
            if (t > w.t0) {
                ok = S.wait(B_PVDONE, (T - 1) & 1);
                __syncwarp();
                if (!ok) break;
            }
            tc_fence_after();
            if (rescale) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    const uint32_t ta = tmem + lane_off + C::kColO + c * 32;
                    tmem_ld32(ta, o);
                    tmem_wait_ld(o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(ta, o);
                }
                tmem_wait_st();
            }
#pragma unroll
            for (int ch = 0; ch < kBlockN / 8; ++ch)
                st_shared_v4(sbase + C::kOffP + sw128_offset(row, ch, C::kCol), pk[4 * ch],
                             pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.bar(B_PFULL));
        }
        if (!ok) break;

        // ---- epilogue of the item ----
        ok = S.wait(B_PVDONE, (T - 1) & 1);
        __syncwarp();
        if (!ok) break;
        tc_fence_after();
        const int tok = w.mt * P.tok_per_tile + row / P.G;
        const bool valid = row < P.tok_per_tile * P.G && tok < w.cnt;
        const int h = w.g * P.G + row % P.G;
        __nv_bfloat16 *orow = P.out + ((static_cast<int64_t>(w.b) * P.r_max + tok) * P.H + h) * D;
        if (P.n_split == 1) {
            const float inv = 1.f / l_run;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + C::kColO + c * 32, o);
                tmem_wait_ld(o);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
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
        // split item: store the partial, then the last split of the unit merges
        float4 *po = P.part_o + static_cast<int64_t>(i) * (D / 4) * kBlockM;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + C::kColO + c * 32, o);
            tmem_wait_ld(o);
            if (valid) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    __stcg(po + (c * 8 + q) * kBlockM + row,
                           make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                       __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3])));
            }
        }
        tc_fence_before();
        if (valid) __stcg(P.part_ml + static_cast<int64_t>(i) * kBlockM + row, make_float2(m_run, l_run));
        __threadfence();
        named_bar_sync(1, 128);
        if (warp == 2 && lane == 0) {
            const unsigned ticket = atomicInc(P.tickets + w.unit, static_cast<unsigned>(P.n_split - 1));
            s_last = ticket == static_cast<unsigned>(P.n_split - 1);
        }
        named_bar_sync(1, 128);
        if (!s_last) continue;
        __threadfence();
        if (valid) {
            // merge the n_split partials of this unit, in split order
            float m_all = -INFINITY;
            for (int s = 0; s < P.n_split; ++s) {
                const int item = s * P.n_units + w.unit;
                m_all = fmaxf(m_all, __ldcg(P.part_ml + static_cast<int64_t>(item) * kBlockM + row).x);
            }
            float scl[kMaxSplit];
            float l_tot = 0.f;
            for (int s = 0; s < P.n_split; ++s) {
                const int item = s * P.n_units + w.unit;
                const float2 ml = __ldcg(P.part_ml + static_cast<int64_t>(item) * kBlockM + row);
                scl[s] = ex2(ml.x - m_all);
                l_tot += scl[s] * ml.y;
            }
            const float inv = 1.f / l_tot;
#pragma unroll 1
            for (int c = 0; c < D / 8; ++c) {  // 8 output columns at a time
                float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
                for (int s = 0; s < P.n_split; ++s) {
                    const float4 *ps =
                        P.part_o + static_cast<int64_t>(s * P.n_units + w.unit) * (D / 4) * kBlockM;
                    const float4 x0 = __ldcg(ps + (2 * c) * kBlockM + row);
                    const float4 x1 = __ldcg(ps + (2 * c + 1) * kBlockM + row);
                    const float f = scl[s];
                    a0.x = fmaf(f, x0.x, a0.x);
                    a0.y = fmaf(f, x0.y, a0.y);
                    a0.z = fmaf(f, x0.z, a0.z);
                    a0.w = fmaf(f, x0.w, a0.w);
                    a1.x = fmaf(f, x1.x, a1.x);
                    a1.y = fmaf(f, x1.y, a1.y);
                    a1.z = fmaf(f, x1.z, a1.z);
                    a1.w = fmaf(f, x1.w, a1.w);
                }
                uint4 v;
                v.x = pack_bf16x2(a0.x * inv, a0.y * inv);
                v.y = pack_bf16x2(a0.z * inv, a0.w * inv);
                v.z = pack_bf16x2(a1.x * inv, a1.y * inv);
                v.w = pack_bf16x2(a1.z * inv, a1.w * inv);
                *reinterpret_cast<uint4 *>(orow + c * 8) = v;
            }
        }
        __syncwarp();
    }
}

// Prologue: every fresh row of every (b, KV head) is written into the caches.
template <int D>
__device__ void write_back(const Params &P)
{
    constexpr int kChunks = D / 8;
    const int64_t total = static_cast<int64_t>(P.B) * P.r_max * P.Hkv * kChunks;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int ch = static_cast<int>(e % kChunks);
        const int64_t rg = e / kChunks;  // (b, r, g) flattened
        const int g = static_cast<int>(rg % P.Hkv);
        const int64_t br = rg / P.Hkv;
        const int r = static_cast<int>(br % P.r_max);
        const int b = static_cast<int>(br / P.r_max);
        const int c = __ldg(P.count + b);
        if (ch == 0 && g == 0 && r == 0 && (c < 0 || c > P.r_max))
            flag_status(P.hdr + kHdrStatus, EC_DEV_BAD_COUNT);
        if (r >= min(max(c, 0), P.r_max)) continue;
        const int32_t *idx = P.idx + static_cast<int64_t>(b) * P.idx_stride;
        const int p = __ldg(idx + r);
        if (p < 0 || p >= P.L) {
            if (ch == 0 && g == 0) flag_status(P.hdr + kHdrStatus, EC_DEV_BAD_INDEX);
            continue;
        }
        if (ch == 0 && g == 0 && r > 0 && __ldg(idx + r - 1) >= p)
            flag_status(P.hdr + kHdrStatus, EC_DEV_BAD_INDEX);
        const int64_t src = (br * P.Hkv + g) * D + ch * 8;
        const int64_t dst = ((static_cast<int64_t>(b) * P.L + p) * P.Hkv + g) * D + ch * 8;
        *reinterpret_cast<uint4 *>(P.k_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(P.k_new + src));
        *reinterpret_cast<uint4 *>(P.v_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(P.v_new + src));
    }
    // generic-proxy writes, read next by the TMA (async proxy) of other CTAs
    asm volatile("fence.proxy.async.global;" ::: "memory");
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
    Sync S{sbase + C::kOffBar, abort_flag, P.hdr + kHdrStatus};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < B_COUNT; ++i)
            mbar_init(S.bar(i), (i == B_SFREE || i == B_SFREE + 1 || i == B_PFULL) ? 4u : 1u);
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
    write_back<D>(P);
    const bool ok = grid_barrier(P.hdr, gridDim.x, abort_flag);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (ok) {
        if (warp == 0 || warp == 6) {
            if ((threadIdx.x & 31) == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                if (warp == 0) {
                    prefetch_tmap(&tm_q);
                    prefetch_tmap(&tm_k);
                    producer_qk<D>(P, S, sbase, &tm_q, &tm_k);
                } else {
                    prefetch_tmap(&tm_v);
                    producer_v<D>(P, S, sbase, &tm_v);
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            if ((threadIdx.x & 31) == 0) mma_issuer<D>(P, S, sbase, tmem);
            __syncwarp();
        } else {
            softmax_epilogue<D>(P, S, sbase, tmem);
        }
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
    int G, tok_per_tile, n_mt, n_units, n_tiles, n_split, n_items, n_ctas;
};

Plan make_plan(int B, int L, int r_max, int H, int Hkv)
{
    Plan p;
    p.G = H / Hkv;
    p.tok_per_tile = kBlockM / p.G;
    p.n_mt = (r_max + p.tok_per_tile - 1) / p.tok_per_tile;
    p.n_units = B * Hkv * p.n_mt;
    p.n_tiles = (L + kBlockN - 1) / kBlockN;
    const int n_sm = device_sm_count();
    // Pick the split that minimises (rounds of items per CTA) x (tiles per item +
    // fixed per-item cost); a split keeps at least two tiles.
    double best = 1e30;
    p.n_split = 1;
    const int max_split = std::max(1, std::min(kMaxSplit, p.n_tiles / 2));
    for (int s = 1; s <= max_split; ++s) {
        const int64_t items = static_cast<int64_t>(p.n_units) * s;
        const int64_t rounds = (items + n_sm - 1) / n_sm;
        const double per_item =
            std::ceil(static_cast<double>(p.n_tiles) / s) + 1.5 + (s > 1 ? 0.5 : 0.0);
        const double cost = static_cast<double>(rounds) * per_item;
        if (cost < best - 1e-9) {
            best = cost;
            p.n_split = s;
        }
    }
    p.n_items = p.n_units * p.n_split;
    p.n_ctas = std::min(p.n_items, n_sm);
    return p;
}

size_t partial_offsets(const Plan &p, int D, size_t *off_tickets, size_t *off_ml, size_t *off_o)
{
    size_t off = kWsHeader;
    *off_tickets = off;
    off = align_up(off + static_cast<size_t>(p.n_units) * sizeof(unsigned), 256);
    *off_ml = off;
    const size_t parts = p.n_split > 1 ? static_cast<size_t>(p.n_items) : 0;
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
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<D>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(Cfg<D>::kBytes));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.n_ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<D>::kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: the grid barrier is safe
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attention_tc_kernel<D>, p, tq, tk, tv);
}

}  // namespace

bool attention_tc_supported(int dtype, int32_t seq_len, int32_t head_dim)
{
    return dtype == EC_BF16 && (head_dim == 64 || head_dim == 128) && seq_len >= 1;
}

size_t attention_tc_workspace_bytes(int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                    int32_t n_kv_heads, int32_t head_dim)
{
    if (batch < 1 || seq_len < 1 || r_max < 1 || n_kv_heads < 1 || n_heads < n_kv_heads)
        return kWsHeader;
    const Plan p = make_plan(batch, seq_len, r_max, n_heads, n_kv_heads);
    size_t a, b, c;
    return partial_offsets(p, head_dim, &a, &b, &c);
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
    p.n_split = plan.n_split;
    p.n_items = plan.n_items;
    p.n_tiles = plan.n_tiles;
    p.scale_log2 = scale * kLog2e;
    char *ws = static_cast<char *>(workspace);
    size_t o_t, o_ml, o_o;
    partial_offsets(plan, head_dim, &o_t, &o_ml, &o_o);
    p.hdr = reinterpret_cast<uint32_t *>(ws);
    p.tickets = reinterpret_cast<unsigned *>(ws + o_t);
    p.part_ml = reinterpret_cast<float2 *>(ws + o_ml);
    p.part_o = reinterpret_cast<float4 *>(ws + o_o);
    return head_dim == 128 ? launch_typed<128>(p, plan, q, stream)
                           : launch_typed<64>(p, plan, q, stream);
}

}  // namespace ec
