// Selective-recompute bidirectional attention on the 5th-generation tensor
// cores (tcgen05 + TMEM), fed by TMA, with the KV write-back fused in.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, section "1. Il Problema" (dLLM attention is
// bidirectional) and "Algoritmo di Funzionamento" step 2 (the partial forward
// recomputes K/V only for the selected tokens; the cache supplies the rest).
//
// One CTA owns one tile of 128 query rows of one (sequence b, KV head g): the
// rows are the (recomputed row r, head h in g's group) pairs packed r-major, so
// a GQA group shares every K/V tile it loads.  Warp roles:
//   warp 0     producer: per 128-key tile, a TMA load of K and V (128B swizzle)
//              from the cache; where the tile holds recomputed positions, the
//              fresh rows are written over the loaded rows in shared memory
//              (tiles made only of fresh rows are loaded straight from the
//              fresh K/V);
//   warp 1     allocates TMEM and issues tcgen05.mma: S = Q K^T into one of two
//              TMEM S buffers, O += P V into the TMEM O accumulator;
//   warps 2-5  one thread per query row: online softmax on S read with
//              tcgen05.ld (log2 domain, the running maximum only moves when it
//              grows by more than 2^8, rescaling O in TMEM when it does), P as
//              bf16 into shared memory, and the normalised output at the end.
// Write-back: every CTA of (b, g) copies an equal share of the fresh rows into
// the global caches.  No CTA reads what another writes in this launch: any
// tile holding a fresh position gets that row from the fresh K/V, so no grid
// barrier is needed.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "ec_internal.cuh"
#include "tc_ptx.cuh"

namespace ec {
namespace {

using namespace ptx;

constexpr int kBlockM = 128;  // query rows per CTA = TMEM lanes
constexpr int kBlockN = 128;  // keys per tile
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr int kMaxTiles = 1024;                   // keys per sequence up to 131072
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s: a wait this long is a fault

template <int D>
struct Cfg {
    static constexpr uint32_t kTile = kBlockM * D * 2;   // bytes of one Q / K / V tile
    static constexpr uint32_t kCol = kBlockM * 128;      // one 64-element column: 16 KB
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kTile;
    static constexpr uint32_t kOffV = kOffK + kStages * kTile;
    static constexpr uint32_t kOffP = kOffV + kStages * kTile;
    static constexpr uint32_t kOffBar = kOffP + kBlockM * kBlockN * 2;
    static constexpr uint32_t kOffTable = kOffBar + 256;
    static constexpr uint32_t kOffMisc = kOffTable + (kMaxTiles + 1) * 4;
    static constexpr uint32_t kBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;    // two S buffers: columns [0, 128) and [128, 256)
    static constexpr uint32_t kColO = 256;  // O: columns [256, 256 + D)
};

enum : int {
    B_KFULL = 0,  // [2] K tile ready for the MMA
    B_VFULL = 2,  // [2] V tile ready
    B_KLOAD = 4,  // [2] TMA of a K tile that still needs fresh rows patched in
    B_VLOAD = 6,  // [2]
    B_EMPTY = 8,  // [2] K/V stage consumed
    B_Q = 10,
    B_SFULL = 11,  // [2]
    B_SFREE = 13,  // [2]
    B_PFULL = 15,
    B_PVDONE = 16,
    B_DRAIN = 17,
    B_COUNT = 18
};

struct Params {
    const __nv_bfloat16 *q, *k_new, *v_new;
    __nv_bfloat16 *k_cache, *v_cache, *out;
    const int32_t *idx;
    int64_t idx_stride;
    const int32_t *count;
    int L, r_max, H, Hkv, G, n_mtiles;
    float scale_log2;
    uint32_t *status;
};

struct Sync {
    uint32_t bars;
    volatile int *abort_flag;
    uint32_t *status;
    __device__ uint32_t bar(int i) const { return bars + 8u * static_cast<uint32_t>(i); }
    // Bounded wait: gives up (and raises the abort flag) after ~2 s.
    __device__ bool wait(int i, uint32_t parity) const
    {
        const uint32_t b = bar(i);
        if (mbar_try_wait(b, parity)) return true;
        const long long t0 = clock64();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try_wait(b, parity)) return true;
            if ((it & 127u) == 0u) {
                if (*abort_flag) return false;
                if (clock64() - t0 > kWaitCycles) {
                    *abort_flag = 1;
                    flag_status(status, EC_DEV_TIMEOUT);
                    return false;
                }
            }
        }
    }
    __device__ bool drain(int i, uint32_t parity) const
    {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar(i), parity))
            if (clock64() - t0 > kWaitCycles / 4) return false;
        return true;
    }
};

template <int D>
__device__ void producer(const Params &P, const Sync &S, uint32_t sbase, int *table, int b, int g,
                         int cnt, int n_tiles, const CUtensorMap *tm_kc, const CUtensorMap *tm_vc,
                         const CUtensorMap *tm_kn, const CUtensorMap *tm_vn)
{
    using C = Cfg<D>;
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const int lane = threadIdx.x & 31;
    const int32_t *idx = P.idx + static_cast<int64_t>(b) * P.idx_stride;
    // table[t] = first recomputed row whose position is >= 128 t (idx is ascending)
    for (int t = lane; t <= n_tiles; t += 32) {
        const int key = t * kBlockN;
        int lo = 0, hi = cnt;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(idx + mid) < key)
                lo = mid + 1;
            else
                hi = mid;
        }
        table[t] = lo;
    }
    __syncwarp();
    if (lane == 0) {
        prefetch_tmap(tm_kc);
        prefetch_tmap(tm_vc);
        prefetch_tmap(tm_kn);
        prefetch_tmap(tm_vn);
    }
    uint32_t full_uses[kStages] = {0, 0}, load_uses[kStages] = {0, 0};
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j % kStages;
        if (j >= kStages) ok = S.wait(B_EMPTY + s, ((j / kStages) - 1) & 1);
        if (!ok) break;
        const int rlo = table[j], rhi = table[j + 1], nf = rhi - rlo;
        const uint32_t kdst = sbase + C::kOffK + s * C::kTile;
        const uint32_t vdst = sbase + C::kOffV + s * C::kTile;
        ++full_uses[s];
        if (nf == 0 || nf == kBlockN) {
            // untouched tile from the cache, or a tile made only of fresh rows
            const CUtensorMap *mk = nf ? tm_kn : tm_kc;
            const CUtensorMap *mv = nf ? tm_vn : tm_vc;
            const int row0 = nf ? rlo : j * kBlockN;
            if (lane == 0) {
                mbar_expect_tx(S.bar(B_KFULL + s), C::kTile);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(kdst + c * C::kCol, mk, S.bar(B_KFULL + s), c * 64, g, row0, b);
                mbar_expect_tx(S.bar(B_VFULL + s), C::kTile);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(vdst + c * C::kCol, mv, S.bar(B_VFULL + s), c * 64, g, row0, b);
            }
            __syncwarp();
            continue;
        }
        // mixed tile: load from the cache, then overwrite the fresh rows
        const uint32_t par = load_uses[s] & 1u;
        ++load_uses[s];
        if (lane == 0) {
            mbar_expect_tx(S.bar(B_KLOAD + s), C::kTile);
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(kdst + c * C::kCol, tm_kc, S.bar(B_KLOAD + s), c * 64, g, j * kBlockN, b);
            mbar_expect_tx(S.bar(B_VLOAD + s), C::kTile);
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(vdst + c * C::kCol, tm_vc, S.bar(B_VLOAD + s), c * 64, g, j * kBlockN, b);
        }
        __syncwarp();
        for (int pass = 0; pass < 2 && ok; ++pass) {
            ok = S.wait((pass ? B_VLOAD : B_KLOAD) + s, par);
            if (!ok) break;
            const __nv_bfloat16 *src = pass ? P.v_new : P.k_new;
            const uint32_t dst = pass ? vdst : kdst;
            for (int i = lane; i < nf * kChunks; i += 32) {
                const int r = rlo + i / kChunks, ch = i % kChunks;
                const int row = __ldg(idx + r) - j * kBlockN;
                if (row < 0 || row >= kBlockN) {
                    flag_status(P.status, EC_DEV_BAD_INDEX);
                    continue;
                }
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(
                    src + ((static_cast<int64_t>(b) * P.r_max + r) * P.Hkv + g) * D + ch * 8));
                st_shared_v4(dst + sw128_offset(row, ch, C::kCol), v.x, v.y, v.z, v.w);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.bar((pass ? B_VFULL : B_KFULL) + s));
        }
    }
    if (!ok && lane == 0) {  // let every copy this warp started land before the CTA exits
        for (int s = 0; s < kStages; ++s) {
            if (full_uses[s]) {
                S.drain(B_KFULL + s, (full_uses[s] - 1) & 1);
                S.drain(B_VFULL + s, (full_uses[s] - 1) & 1);
            }
            if (load_uses[s]) {
                S.drain(B_KLOAD + s, (load_uses[s] - 1) & 1);
                S.drain(B_VLOAD + s, (load_uses[s] - 1) & 1);
            }
        }
    }
}

template <int D>
__device__ void mma_issuer(const Sync &S, uint32_t sbase, uint32_t tmem, int n_tiles)
{
    using C = Cfg<D>;
    constexpr uint32_t kIdescQK = idesc_bf16(kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdescPV = idesc_bf16(kBlockM, D, false, true);
    bool ok = S.wait(B_Q, 0);
    tc_fence_after();
    auto issue_pv = [&](int t) {
        const int s = t % kStages;
        ok = ok && S.wait(B_PFULL, t & 1) && S.wait(B_VFULL + s, (t / kStages) & 1);
        if (!ok) return;
        tc_fence_after();
        const uint32_t vbase = sbase + C::kOffV + s * C::kTile;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
            const uint64_t a = desc_sw128(sbase + C::kOffP + (kk >> 2) * C::kCol + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = desc_sw128(vbase + kk * 16 * 128, C::kCol, 1024);
            umma_bf16(tmem + C::kColO, a, bd, kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(S.bar(B_EMPTY + s));
        umma_commit(S.bar(B_PVDONE));
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j % kStages, sb = j & 1;
        ok = S.wait(B_KFULL + s, (j / kStages) & 1);
        if (ok && j >= 2) ok = S.wait(B_SFREE + sb, ((j >> 1) - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kbase = sbase + C::kOffK + s * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kCol + (kk & 3) * 32;
            umma_bf16(tmem + C::kColS + sb * kBlockN, desc_sw128(sbase + C::kOffQ + off, 16, 1024),
                      desc_sw128(kbase + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
        }
        umma_commit(S.bar(B_SFULL + sb));
        if (j >= 1) issue_pv(j - 1);
    }
    if (ok) issue_pv(n_tiles - 1);
    // everything issued has completed before TMEM is released
    umma_commit(S.bar(B_DRAIN));
    S.drain(B_DRAIN, 0);
}

template <int D>
__device__ void softmax_epilogue(const Params &P, const Sync &S, uint32_t sbase, uint32_t tmem,
                                 int b, int g, int mt, int rows_valid, int n_tiles)
{
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const int m = mt * kBlockM + row;
    const bool valid = m < rows_valid;
    const int r = m / P.G, h = g * P.G + (m - r * P.G);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;

    // Q tile (rows past the valid count are zero)
    const __nv_bfloat16 *qrow = P.q + ((static_cast<int64_t>(b) * P.r_max + r) * P.H + h) * D;
#pragma unroll
    for (int ch = 0; ch < D / 8; ++ch) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (valid) v = __ldg(reinterpret_cast<const uint4 *>(qrow + ch * 8));
        st_shared_v4(sbase + C::kOffQ + sw128_offset(row, ch, C::kCol), v.x, v.y, v.z, v.w);
    }
    fence_async_smem();
    named_bar_sync(1, 128);
    if (warp == 2 && lane == 0) mbar_arrive(S.bar(B_Q));

    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
        const int sb = j & 1;
        ok = S.wait(B_SFULL + sb, (j >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + C::kColS + sb * kBlockN + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_wait_ld(sr[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(S.bar(B_SFREE + sb));

        const int kv_valid = min(kBlockN, P.L - j * kBlockN);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float s = __uint_as_float(sr[c][i]) * P.scale_log2;
                if (c * 32 + i >= kv_valid) s = -INFINITY;
                sr[c][i] = __float_as_uint(s);
                mx = fmaxf(mx, s);
            }
        float m_use = m_run, alpha = 1.f;
        bool rescale = false;
        if (mx > m_run + 8.f) {  // move the reference only when p could exceed 2^8
            m_use = mx;
            alpha = ex2(m_run - mx);
            rescale = j > 0;
        }
        float rowsum = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float p0 = ex2(__uint_as_float(sr[c][i]) - m_use);
                const float p1 = ex2(__uint_as_float(sr[c][i + 1]) - m_use);
                rowsum += p0 + p1;
                pk[(c * 32 + i) >> 1] = pack_bf16x2(p0, p1);
            }
        l_run = l_run * alpha + rowsum;
        m_run = m_use;

        // the P buffer and O are free once PV(j-1) has completed
        if (j >= 1) {
            ok = S.wait(B_PVDONE, (j - 1) & 1);
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
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st32(ta, o);
            }
            tmem_wait_st();
        }
#pragma unroll
        for (int ch = 0; ch < kBlockN / 8; ++ch)
            st_shared_v4(sbase + C::kOffP + sw128_offset(row, ch, C::kCol), pk[4 * ch], pk[4 * ch + 1],
                         pk[4 * ch + 2], pk[4 * ch + 3]);
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(S.bar(B_PFULL));
    }
    if (!ok) return;
    ok = S.wait(B_PVDONE, (n_tiles - 1) & 1);
    if (!ok) return;
    tc_fence_after();
    const float inv = 1.f / l_run;
    __nv_bfloat16 *orow = P.out + ((static_cast<int64_t>(b) * P.r_max + r) * P.H + h) * D;
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
                v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                dst[q] = v;
            }
        }
    }
    tc_fence_before();
}

// Copy this CTA's share of the fresh rows of KV head g into the caches.
template <int D>
__device__ void write_back_share(const Params &P, int b, int g, int mt, int cnt)
{
    constexpr int kChunks = D / 8;
    const int r0 = static_cast<int>(static_cast<int64_t>(cnt) * mt / P.n_mtiles);
    const int r1 = static_cast<int>(static_cast<int64_t>(cnt) * (mt + 1) / P.n_mtiles);
    const int32_t *idx = P.idx + static_cast<int64_t>(b) * P.idx_stride;
    for (int i = threadIdx.x; i < (r1 - r0) * kChunks; i += kThreads) {
        const int r = r0 + i / kChunks, ch = i % kChunks;
        const int p = __ldg(idx + r);
        if (p < 0 || p >= P.L || (r > 0 && __ldg(idx + r - 1) >= p)) {
            if (ch == 0) flag_status(P.status, EC_DEV_BAD_INDEX);
            if (p < 0 || p >= P.L) continue;
        }
        const int64_t src = ((static_cast<int64_t>(b) * P.r_max + r) * P.Hkv + g) * D + ch * 8;
        const int64_t dst = ((static_cast<int64_t>(b) * P.L + p) * P.Hkv + g) * D + ch * 8;
        *reinterpret_cast<uint4 *>(P.k_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(P.k_new + src));
        *reinterpret_cast<uint4 *>(P.v_cache + dst) = __ldg(reinterpret_cast<const uint4 *>(P.v_new + src));
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const Params P, const __grid_constant__ CUtensorMap tm_kc,
                        const __grid_constant__ CUtensorMap tm_vc,
                        const __grid_constant__ CUtensorMap tm_kn,
                        const __grid_constant__ CUtensorMap tm_vn)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int mt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    int cnt = __ldg(P.count + b);
    if (cnt < 0 || cnt > P.r_max) {
        if (threadIdx.x == 0 && mt == 0 && g == 0) flag_status(P.status, EC_DEV_BAD_COUNT);
        cnt = max(0, min(cnt, P.r_max));
    }
    write_back_share<D>(P, b, g, mt, cnt);
    const int rows_valid = cnt * P.G;
    if (mt * kBlockM >= rows_valid) return;  // uniform: this tile has no query rows
    const int n_tiles = (P.L + kBlockN - 1) / kBlockN;

    int *table = reinterpret_cast<int *>(smem + C::kOffTable);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc + 16);
    Sync S{sbase + C::kOffBar, abort_flag, P.status};
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            const bool four = i == B_SFREE || i == B_SFREE + 1 || i == B_PFULL;
            mbar_init(S.bar(i), four ? 4u : 1u);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        producer<D>(P, S, sbase, table, b, g, cnt, n_tiles, &tm_kc, &tm_vc, &tm_kn, &tm_vn);
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) mma_issuer<D>(S, sbase, tmem, n_tiles);
        __syncwarp();
    } else {
        softmax_epilogue<D>(P, S, sbase, tmem, b, g, mt, rows_valid, n_tiles);
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

// [B, rows, Hkv, D] bf16 viewed as 4-D {D, Hkv, rows, B}; box {64, 1, 128, 1}, 128B swizzle.
bool encode_rows(CUtensorMap *map, const void *base, int B, int rows, int Hkv, int D)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                                static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(Hkv) * D * 2,
                                   static_cast<cuuint64_t>(rows) * Hkv * D * 2};
    const cuuint32_t box[4] = {64, 1, kBlockN, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_typed(const Params &p, int batch, cudaStream_t stream)
{
    CUtensorMap kc, vc, kn, vn;
    const int rows_new = p.r_max > 0 ? p.r_max : 1;
    if (!encode_rows(&kc, p.k_cache, batch, p.L, p.Hkv, D) ||
        !encode_rows(&vc, p.v_cache, batch, p.L, p.Hkv, D) ||
        !encode_rows(&kn, p.k_new, batch, rows_new, p.Hkv, D) ||
        !encode_rows(&vn, p.v_new, batch, rows_new, p.Hkv, D))
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
    const dim3 grid(static_cast<unsigned>(p.n_mtiles), static_cast<unsigned>(p.Hkv),
                    static_cast<unsigned>(batch));
    attention_tc_kernel<D><<<grid, kThreads, Cfg<D>::kBytes, stream>>>(p, kc, vc, kn, vn);
    return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(int dtype, int32_t seq_len, int32_t head_dim)
{
    return dtype == EC_BF16 && (head_dim == 64 || head_dim == 128) &&
           seq_len <= kMaxTiles * kBlockN;
}

cudaError_t launch_attention_tc(const void *q, const void *k_new, const void *v_new,
                                const int32_t *idx, int64_t idx_stride, const int32_t *count,
                                void *k_cache, void *v_cache, void *out, int32_t batch,
                                int32_t seq_len, int32_t r_max, int32_t n_heads,
                                int32_t n_kv_heads, int32_t head_dim, float scale,
                                uint32_t *status, cudaStream_t stream)
{
    if (r_max == 0) return cudaSuccess;  // nothing to recompute, nothing to write back
    Params p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    p.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.idx = idx;
    p.idx_stride = idx_stride;
    p.count = count;
    p.L = seq_len;
    p.r_max = r_max;
    p.H = n_heads;
    p.Hkv = n_kv_heads;
    p.G = n_heads / n_kv_heads;
    p.n_mtiles = static_cast<int>((static_cast<int64_t>(r_max) * p.G + kBlockM - 1) / kBlockM);
    p.scale_log2 = scale * kLog2e;
    p.status = status;
    return head_dim == 128 ? launch_typed<128>(p, batch, stream) : launch_typed<64>(p, batch, stream);
}

}  // namespace ec
