// Q/K/V projection of the recomputed rows on the 5th-generation tensor cores,
// and the embedding gather that feeds the first layer.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, "Algoritmo di Funzionamento" step 2: a partial
// forward recomputes only the selected tokens (their queries, keys and values),
// a full forward all of them.  The projection is the one dense contraction of
// that forward besides attention:
//     [Q | K | V][b, r, :] = X[b, r, :] W^T,   W = [W_q; W_k; W_v]  ([3 width, hidden])
// for the count[b] recomputed rows r of every sequence b.
//
// Persistent kernel, one CTA per SM, 128 x BN output tiles (BN = 64, 128 or
// 256), K in steps of 64:
//   warp 0      TMA producer: X tile [128 x 64] and W tile [BN x 64], 128-byte
//               swizzle, into a ring of stages;
//   warp 1      TMEM allocation and tcgen05.mma issue (M = 128, N = BN, K = 16
//               per instruction), fp32 accumulation in one of two TMEM buffers so
//               the epilogue of a tile overlaps the main loop of the next;
//   warps 2-5   epilogue: one thread per output row, tcgen05.ld of 32 columns at
//               a time, rounded to bf16 and stored into Q, K or V.
// Tiles are dealt round-robin with the (sequence, row-tile) index varying
// fastest, so the CTAs running at one time share weight tiles through L2.
//
// The same kernel serves the other dense contractions of a transformer layer
// (a pre-norm block: output projection and gated MLP), with one of four
// epilogues:
//   QKV       the three column segments of W into Q, K and V;
//   STORE     Y = X W^T;
//   RESIDUAL  Y = R + X W^T (R may be Y itself);
//   SWIGLU    W = [W_gate; W_up] ([2F, hidden]); a tile's B operand holds BN/2
//             gate rows and the BN/2 up rows of the same outputs (two TMA boxes),
//             and Y[:, j] = silu(g_j) u_j, g and u the two halves of the tile.
// Row tiles at or past count[b] are skipped by every role alike.  Every wait is
// bounded (~2 s); a timeout sets EC_DEV_TIMEOUT and unwinds.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "ec_internal.cuh"
#include "tc_ptx.cuh"

namespace ec {
namespace {

using namespace ptx;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;  // 6 warps
constexpr uint32_t kSmemBudget = 200 * 1024;

template <int BN>
struct GemmCfg {
    static constexpr uint32_t kA = kBM * kBK * 2;  // 16 KB
    static constexpr uint32_t kB = BN * kBK * 2;
    static constexpr uint32_t kStage = kA + kB;
    static constexpr int kStages = static_cast<int>(kSmemBudget / kStage) > 8
                                       ? 8
                                       : static_cast<int>(kSmemBudget / kStage);
    static constexpr uint32_t kOffBar = kStages * kStage;
    static constexpr uint32_t kOffMisc = kOffBar + 256;
    static constexpr uint32_t kBytes = kOffMisc + 64 + 1024;
    static constexpr uint32_t kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
};

enum : int {
    G_FULL = 0,        // [8] stage landed
    G_EMPTY = 8,       // [8] stage consumed by its MMAs
    G_ACC_FULL = 16,   // [2] accumulator complete
    G_ACC_EMPTY = 18,  // [2] accumulator read by the epilogue
    G_DRAIN = 20,
    G_COUNT = 21
};

enum : int { EPI_QKV = 0, EPI_STORE = 1, EPI_RESIDUAL = 2, EPI_SWIGLU = 3 };

struct GemmParams {
    const int32_t *count;  // [batch] rows present per sequence, or null (= r_max)
    __nv_bfloat16 *out[3];
    const __nv_bfloat16 *res;  // RESIDUAL: R, [batch, r_max, width]
    int mode;
    int batch, r_max, hidden, width, n_mt, n_nt, n_tiles;
    int w_half;  // SWIGLU: F, the row where W_up starts
    uint32_t *status;
    long long wait_limit;  // cycles one in-kernel wait may take
};

struct Tile {
    int b, mt, nt, rows;
};

__device__ __forceinline__ Tile decode_tile(const GemmParams &P, int t)
{
    Tile w;
    const int bm = t % (P.batch * P.n_mt);
    w.nt = t / (P.batch * P.n_mt);
    w.b = bm / P.n_mt;
    w.mt = bm - w.b * P.n_mt;
    const int c = P.count ? __ldg(P.count + w.b) : P.r_max;
    w.rows = max(0, min(c, P.r_max));
    return w;
}

__device__ __forceinline__ bool tile_active(const Tile &w) { return w.mt * kBM < w.rows; }

template <int BN>
__device__ void gemm_producer(const GemmParams &P, const Sync &S, uint32_t sbase,
                              const CUtensorMap *tm_x, const CUtensorMap *tm_w)
{
    using C = GemmCfg<BN>;
    const int nk = P.hidden / kBK;
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < P.n_tiles && ok; t += gridDim.x) {
        const Tile w = decode_tile(P, t);
        if (!tile_active(w)) continue;
        for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % C::kStages;
            if (it >= static_cast<uint32_t>(C::kStages))
                ok = S.wait(G_EMPTY + s, ((it / C::kStages) - 1) & 1);
            if (!ok) break;
            const uint32_t dst = sbase + s * C::kStage;
            mbar_expect_tx(S.bar(G_FULL + s), C::kStage);
            tma_load_3d(dst, tm_x, S.bar(G_FULL + s), kb * kBK, w.mt * kBM, w.b);
            if (P.mode == EPI_SWIGLU) {  // BN/2 gate rows, then the same outputs' up rows
                tma_load_2d(dst + C::kA, tm_w, S.bar(G_FULL + s), kb * kBK, w.nt * (BN / 2));
                tma_load_2d(dst + C::kA + (BN / 2) * kBK * 2, tm_w, S.bar(G_FULL + s), kb * kBK,
                            P.w_half + w.nt * (BN / 2));
            } else {
                tma_load_2d(dst + C::kA, tm_w, S.bar(G_FULL + s), kb * kBK, w.nt * BN);
            }
        }
    }
    if (!ok)  // let every copy already started land before the CTA exits
        for (uint32_t u = (it > C::kStages ? it - C::kStages : 0); u < it; ++u)
            S.drain(G_FULL + u % C::kStages, (u / C::kStages) & 1);
}

template <int BN>
__device__ void gemm_mma(const GemmParams &P, const Sync &S, uint32_t sbase, uint32_t tmem)
{
    using C = GemmCfg<BN>;
    constexpr uint32_t kIdesc = idesc_bf16(kBM, BN, false, false);
    const int nk = P.hidden / kBK;
    uint32_t it = 0, tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < P.n_tiles && ok; t += gridDim.x) {
        const Tile w = decode_tile(P, t);
        if (!tile_active(w)) continue;
        const uint32_t a = tl & 1;
        if (tl >= 2) ok = S.wait(G_ACC_EMPTY + a, ((tl >> 1) - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc = tmem + a * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % C::kStages;
            ok = S.wait(G_FULL + s, (it / C::kStages) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t xa = sbase + s * C::kStage;
            const uint32_t wb = xa + C::kA;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
                umma_bf16(acc, desc_sw128(xa + k * 32, 16, 1024), desc_sw128(wb + k * 32, 16, 1024),
                          kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
            umma_commit(S.bar(G_EMPTY + s));
        }
        if (!ok) break;
        umma_commit(S.bar(G_ACC_FULL + a));
        ++tl;
    }
    // everything issued has completed before TMEM is released
    umma_commit(S.bar(G_DRAIN));
    S.drain(G_DRAIN, 0);
}

template <int BN>
__device__ void gemm_epilogue(const GemmParams &P, const Sync &S, uint32_t tmem)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t tl = 0;
    for (int t = blockIdx.x; t < P.n_tiles; t += gridDim.x) {
        const Tile w = decode_tile(P, t);
        if (!tile_active(w)) continue;
        const uint32_t a = tl & 1;
        const bool ok = S.wait(G_ACC_FULL + a, (tl >> 1) & 1);
        __syncwarp();
        if (!ok) break;
        tc_fence_after();
        const int r = w.mt * kBM + row;
        const bool valid = r < w.rows;
        const bool swiglu = P.mode == EPI_SWIGLU;
        const int n0 = swiglu ? w.nt * (BN / 2) : w.nt * BN;  // first output column
        const int seg = P.mode == EPI_QKV ? n0 / P.width : 0;
        const int64_t off = (static_cast<int64_t>(w.b) * P.r_max + r) * P.width + (n0 - seg * P.width);
        __nv_bfloat16 *dst = P.out[seg] + off;
#pragma unroll 1
        for (int c = 0; c < (swiglu ? BN / 64 : BN / 32); ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + a * BN + c * 32, v);
            tmem_wait_ld(v);
            if (swiglu) {  // v = gate columns; the up columns sit BN/2 further
                uint32_t u[32];
                tmem_ld32(tmem + lane_off + a * BN + BN / 2 + c * 32, u);
                tmem_wait_ld(u);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float g = __uint_as_float(v[j]);
                    v[j] = __float_as_uint(g / (1.f + __expf(-g)) * __uint_as_float(u[j]));
                }
            } else if (P.mode == EPI_RESIDUAL && valid) {
                const uint4 *r4 = reinterpret_cast<const uint4 *>(P.res + off + c * 32);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 x = r4[q];
                    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * q + 2 * e] = __float_as_uint(__uint_as_float(v[8 * q + 2 * e]) +
                                                           __uint_as_float(xs[e] << 16));
                        v[8 * q + 2 * e + 1] = __float_as_uint(__uint_as_float(v[8 * q + 2 * e + 1]) +
                                                               __uint_as_float(xs[e] & 0xffff0000u));
                    }
                }
            }
            if (valid) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 o;
                    o.x = pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1]));
                    o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
                    o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
                    o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
                    d4[q] = o;
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(S.bar(G_ACC_EMPTY + a));
        ++tl;
    }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_kernel(const GemmParams P, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_w)
{
    using C = GemmCfg<BN>;
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
        for (int i = 0; i < G_COUNT; ++i) mbar_init(S.bar(i), (i == G_ACC_EMPTY || i == G_ACC_EMPTY + 1) ? 4u : 1u);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && (threadIdx.x & 31) == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // inputs and outputs belong to the previous kernel until here

    if (warp == 0) {
        if ((threadIdx.x & 31) == 0) gemm_producer<BN>(P, S, sbase, &tm_x, &tm_w);
        __syncwarp();
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) gemm_mma<BN>(P, S, sbase, tmem);
        __syncwarp();
    } else {
        gemm_epilogue<BN>(P, S, tmem);
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

// bf16 tensor of `rank` dims (innermost first), 128-byte swizzled box.
bool encode(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides_bytes, const cuuint32_t *box)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims,
              strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile width: minimise (rounds of tiles per CTA) x (per-tile cost ~ BN + 64),
// among the widths that tile the output (`segs` segments of `width` columns;
// SWIGLU: BN/2 must divide F).
int choose_bn(int batch, int r_max, int width, int segs = 3, bool swiglu = false)
{
    const int n_sm = device_sm_count();
    const int n_mt = (r_max + kBM - 1) / kBM;
    int best_bn = 0;
    double best = 1e30;
    for (int bn : {256, 128, 64}) {
        if (swiglu ? width % (bn / 2) : width % bn) continue;
        const int64_t tiles = static_cast<int64_t>(batch) * n_mt * (segs * width / bn);
        const double cost = static_cast<double>((tiles + n_sm - 1) / n_sm) * (bn + 64);
        if (cost < best - 1e-9) {
            best = cost;
            best_bn = bn;
        }
    }
    return best_bn;
}

template <int BN>
cudaError_t launch_bn(GemmParams p, const void *x, const void *w, cudaStream_t stream)
{
    using C = GemmCfg<BN>;
    const int w_rows = p.mode == EPI_QKV ? 3 * p.width : (p.mode == EPI_SWIGLU ? 2 * p.width : p.width);
    p.n_nt = w_rows / BN;
    p.n_tiles = p.batch * p.n_mt * p.n_nt;
    CUtensorMap tx, tw;
    const cuuint64_t xd[3] = {static_cast<cuuint64_t>(p.hidden), static_cast<cuuint64_t>(p.r_max),
                              static_cast<cuuint64_t>(p.batch)};
    const cuuint64_t xs[2] = {static_cast<cuuint64_t>(p.hidden) * 2,
                              static_cast<cuuint64_t>(p.r_max) * p.hidden * 2};
    const cuuint32_t xb[3] = {kBK, kBM, 1};
    const cuuint64_t wd[2] = {static_cast<cuuint64_t>(p.hidden), static_cast<cuuint64_t>(w_rows)};
    const cuuint64_t ws[1] = {static_cast<cuuint64_t>(p.hidden) * 2};
    const cuuint32_t wbx[2] = {kBK, static_cast<cuuint32_t>(p.mode == EPI_SWIGLU ? BN / 2 : BN)};
    if (!encode(&tx, x, 3, xd, xs, xb) || !encode(&tw, w, 2, wd, ws, wbx)) return cudaErrorInvalidValue;
    const int grid = std::min(p.n_tiles, device_sm_count());
    return launch(qkv_gemm_kernel<BN>, dim3(grid), dim3(kThreads), C::kBytes, stream, p, tx, tw);
}

// ---- embedding gather ----
// x[b, r, :] = table[token of position idx[b, r]] for r < count[b]: the token
// decoded there, or mask_id while the position is still masked.
__global__ void embed_rows_kernel(const uint4 *__restrict__ table, int64_t table_rows, int row_vec,
                                  const int32_t *__restrict__ idx, int64_t idx_stride,
                                  const int32_t *__restrict__ count,
                                  const int32_t *__restrict__ seq_tokens,
                                  const uint8_t *__restrict__ is_masked, int32_t mask_id, int L,
                                  int r_max, uint4 *__restrict__ x, uint32_t *status)
{
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.y;
    const int c = max(0, min(__ldg(count + b), r_max));
    for (int r = blockIdx.x; r < c; r += gridDim.x) {
        const int p = __ldg(idx + static_cast<int64_t>(b) * idx_stride + r);
        if (p < 0 || p >= L) {
            if (threadIdx.x == 0) flag_status(status, EC_DEV_BAD_INDEX);
            continue;
        }
        const int64_t at = static_cast<int64_t>(b) * L + p;
        int tok = __ldg(is_masked + at) ? mask_id : __ldg(seq_tokens + at);
        if (tok < 0 || tok >= table_rows) {
            if (threadIdx.x == 0) flag_status(status, EC_DEV_BAD_INDEX);
            continue;
        }
        const uint4 *src = table + static_cast<int64_t>(tok) * row_vec;
        uint4 *dst = x + (static_cast<int64_t>(b) * r_max + r) * row_vec;
        for (int i = threadIdx.x; i < row_vec; i += blockDim.x) dst[i] = __ldg(src + i);
    }
}

}  // namespace

bool qkv_shape_ok(int32_t hidden, int32_t width)
{
    return hidden >= kBK && hidden % kBK == 0 && width >= 64 && width % 64 == 0;
}

cudaError_t launch_qkv_projection(const void *x, const int32_t *count, int32_t batch,
                                  int32_t r_max, int32_t hidden, const void *w_qkv, int32_t width,
                                  void *q, void *k, void *v, uint32_t *status, cudaStream_t stream)
{
    if (r_max == 0) return cudaSuccess;
    GemmParams p;
    p.count = count;
    p.out[0] = static_cast<__nv_bfloat16 *>(q);
    p.out[1] = static_cast<__nv_bfloat16 *>(k);
    p.out[2] = static_cast<__nv_bfloat16 *>(v);
    p.batch = batch;
    p.r_max = r_max;
    p.hidden = hidden;
    p.width = width;
    p.n_mt = (r_max + kBM - 1) / kBM;
    p.status = status;
    p.wait_limit = wait_limit_cycles();
    p.mode = EPI_QKV;
    p.res = nullptr;
    p.w_half = 0;
    switch (choose_bn(batch, r_max, width)) {
    case 256: return launch_bn<256>(p, x, w_qkv, stream);
    case 128: return launch_bn<128>(p, x, w_qkv, stream);
    default: return launch_bn<64>(p, x, w_qkv, stream);
    }
}

bool linear_shape_ok(int32_t in_features, int32_t out_features, int32_t mode)
{
    return in_features >= kBK && in_features % kBK == 0 && out_features >= 64 &&
           out_features % (mode == 2 ? 32 : 64) == 0 && mode >= 0 && mode <= 2;
}

cudaError_t launch_linear(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                          int32_t in_features, const void *w, int32_t out_features, int32_t mode,
                          const void *residual, void *out, uint32_t *status, cudaStream_t stream)
{
    if (r_max == 0) return cudaSuccess;
    GemmParams p;
    p.count = count;
    p.out[0] = p.out[1] = p.out[2] = static_cast<__nv_bfloat16 *>(out);
    p.res = static_cast<const __nv_bfloat16 *>(residual);
    p.mode = mode == 0 ? EPI_STORE : (mode == 1 ? EPI_RESIDUAL : EPI_SWIGLU);
    p.batch = batch;
    p.r_max = r_max;
    p.hidden = in_features;
    p.width = out_features;
    p.w_half = mode == 2 ? out_features : 0;
    p.n_mt = (r_max + kBM - 1) / kBM;
    p.status = status;
    p.wait_limit = wait_limit_cycles();
    const bool sw = p.mode == EPI_SWIGLU;
    switch (choose_bn(batch, r_max, out_features, sw ? 2 : 1, sw)) {
    case 256: return launch_bn<256>(p, x, w, stream);
    case 128: return launch_bn<128>(p, x, w, stream);
    default: return launch_bn<64>(p, x, w, stream);
    }
}

cudaError_t launch_embed_rows(const void *table, int64_t table_rows, int32_t hidden,
                              const int32_t *idx, int64_t idx_stride, const int32_t *count,
                              const int32_t *seq_tokens, const uint8_t *is_masked, int32_t mask_id,
                              int32_t batch, int32_t seq_len, int32_t r_max, void *x,
                              uint32_t *status, cudaStream_t stream)
{
    if (r_max == 0) return cudaSuccess;
    const int row_vec = hidden * 2 / 16;
    const dim3 grid(static_cast<unsigned>(std::min(r_max, 4 * device_sm_count())),
                    static_cast<unsigned>(batch));
    return launch(embed_rows_kernel, grid, dim3(256), 0, stream,
                  static_cast<const uint4 *>(table), table_rows, row_vec, idx, idx_stride, count,
                  seq_tokens, is_masked, mask_id, seq_len, r_max, static_cast<uint4 *>(x), status);
}

}  // namespace ec
