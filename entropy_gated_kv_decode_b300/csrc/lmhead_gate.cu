// Decode-and-gate fused into the LM-head GEMM: the logits of the masked rows
// are produced on the 5th-generation tensor cores and folded into each row's
// online softmax state in the GEMM's epilogue, so the [N, V] logits never reach
// HBM.
//
// "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion Language
// Models" — Italian summary, section "2. Metodologia", observation 1 (the
// decision needs only an O(V) operation per decoded token) and "Algoritmo di
// Funzionamento" point 3 (constant overhead); section "4. Risultati" (the
// decision logic takes 0.5 % of inference time).  The step's outputs are those
// of the decode-and-gate step: token, confidence and entropy per row, the
// confidence-ranked unmasking, E = max entropy of the unmasked rows and the
// E > tau refresh decision.
//
// Persistent kernel, one CTA per SM, output tiles of 128 rows x 256 vocabulary
// columns, K (the hidden size) in steps of 64:
//   warp 0      TMA producer: hidden-state tile [128 x 64] and W_lm tile
//               [256 x 64], 128-byte swizzle, into a ring of stages;
//   warp 1      TMEM allocation and tcgen05.mma issue (M = 128, N = 256, K = 16),
//               float32 accumulation in one of two TMEM buffers, so the epilogue
//               of a tile overlaps the main loop of the next;
//   warps 2-5   epilogue, one thread per row: the tile's 256 logits (tcgen05.ld,
//               32 columns at a time) folded into the row's running state
//               (m, S, T, first index of m).
// The grid is a whole number of groups of n_mt CTAs (n_mt = row tiles); a CTA
// keeps one row tile and walks every (grid / n_mt)-th vocabulary tile, so the
// row states stay in registers for the whole kernel.  At the end each CTA
// publishes its rows' states to fixed slots; the last CTA of a row tile (an
// acq_rel ticket, no waiting) merges the slots in order, and each row's outputs
// and its sequence's ranking and gate follow as in the decode-and-gate step.
// Every wait is bounded; a timeout sets EC_DEV_TIMEOUT and unwinds.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "ec_internal.cuh"
#include "gate_common.cuh"
#include "tc_ptx.cuh"

namespace ec {
namespace {

using namespace ptx;
using gate::Partial;

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kThreads = 192;  // 6 warps
constexpr int kStages = 4;
constexpr uint32_t kA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kB = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kStage = kA + kB;
constexpr uint32_t kOffBar = kStages * kStage;
constexpr uint32_t kOffMisc = kOffBar + 256;
constexpr uint32_t kBytes = kOffMisc + 64 + 1024;
constexpr uint32_t kTmemCols = 2 * kBN;

enum : int {
    L_FULL = 0,        // [4] stage landed
    L_EMPTY = 4,       // [4] stage consumed by its MMAs
    L_ACC_FULL = 8,    // [2] accumulator complete
    L_ACC_EMPTY = 10,  // [2] accumulator read by the epilogue
    L_DRAIN = 12,
    L_COUNT = 13
};

struct LmParams {
    int n_rows, hidden, vocab;
    int n_mt, n_nt;       // row tiles, vocabulary tiles
    int grid, per_mt;     // CTAs; CTAs per row tile (grid / n_mt)
    gate::GateArgs g;
    uint32_t *status;
    long long wait_limit;
    unsigned *mt_ctr;     // [n_mt] CTAs of the row tile done (wraps to 0)
    float4 *parts;        // [n_rows][per_mt] row states
};

// The k-th vocabulary tile of this CTA (or -1 past the last).
__device__ __forceinline__ int vocab_tile(const LmParams &P, int k)
{
    const int nt = static_cast<int>(blockIdx.x) / P.n_mt + k * P.per_mt;
    return nt < P.n_nt ? nt : -1;
}

__device__ void lm_producer(const LmParams &P, const Sync &S, uint32_t sbase, const CUtensorMap *tm_x,
                            const CUtensorMap *tm_w)
{
    const int mt = static_cast<int>(blockIdx.x) % P.n_mt;
    const int nk = P.hidden / kBK;
    uint32_t it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        const int nt = vocab_tile(P, k);
        if (nt < 0) break;
        for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % kStages;
            if (it >= static_cast<uint32_t>(kStages)) ok = S.wait(L_EMPTY + s, ((it / kStages) - 1) & 1);
            if (!ok) break;
            const uint32_t dst = sbase + s * kStage;
            mbar_expect_tx(S.bar(L_FULL + s), kStage);
            tma_load_2d(dst, tm_x, S.bar(L_FULL + s), kb * kBK, mt * kBM);
            tma_load_2d(dst + kA, tm_w, S.bar(L_FULL + s), kb * kBK, nt * kBN);
        }
    }
    if (!ok)  // let every copy already started land before the CTA exits
        for (uint32_t u = (it > kStages ? it - kStages : 0); u < it; ++u)
            S.drain(L_FULL + u % kStages, (u / kStages) & 1);
}

__device__ void lm_mma(const LmParams &P, const Sync &S, uint32_t sbase, uint32_t tmem)
{
    constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN, false, false);
    const int nk = P.hidden / kBK;
    uint32_t it = 0, tl = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
        if (vocab_tile(P, k) < 0) break;
        const uint32_t a = tl & 1;
        if (tl >= 2) ok = S.wait(L_ACC_EMPTY + a, ((tl >> 1) - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc = tmem + a * kBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = it % kStages;
            ok = S.wait(L_FULL + s, (it / kStages) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t xa = sbase + s * kStage;
            const uint32_t wb = xa + kA;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                umma_bf16(acc, desc_sw128(xa + kk * 32, 16, 1024), desc_sw128(wb + kk * 32, 16, 1024),
                          kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
            umma_commit(S.bar(L_EMPTY + s));
        }
        if (!ok) break;
        umma_commit(S.bar(L_ACC_FULL + a));
        ++tl;
    }
    // everything issued has completed before TMEM is released
    umma_commit(S.bar(L_DRAIN));
    S.drain(L_DRAIN, 0);
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// One row's running state over float32 logits.
struct RowFold {
    float m, s, t;
    int a;
    __device__ void reset()
    {
        m = -INFINITY;
        s = t = 0.f;
        a = INT_MAX;
    }
    // 32 consecutive logits, columns j0 .. j0 + 31, the first n of them real.
    __device__ __forceinline__ void add32(const uint32_t (&v)[32], int j0, int n)
    {
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = j < n ? __uint_as_float(v[j]) : -INFINITY;
        float cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; j += 2) cm = fmax3(cm, x[j], x[j + 1]);
        if (cm > m) {  // new maximum: its first column, the sums shifted to it
            int first = INT_MAX;
#pragma unroll
            for (int j = 31; j >= 0; --j)
                if (x[j] == cm) first = j0 + j;
            if (s > 0.f) {
                const float d = gate::ref_gap(m, cm);
                const float f = gate::shift(d);
                t = f * fmaf(d, s, t);
                s = f * s;
            }
            m = cm;
            a = first;
        }
        if (m == -INFINITY) return;
        const float mb = m * kLog2e;
        float s0 = 0.f, s1 = 0.f, t0 = 0.f, t1 = 0.f;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float y0 = fmaxf(fmaf(x[j], kLog2e, -mb), -1e30f);
            const float y1 = fmaxf(fmaf(x[j + 1], kLog2e, -mb), -1e30f);
            const float e0 = ex2(y0), e1 = ex2(y1);
            s0 += e0;
            s1 += e1;
            t0 = fmaf(e0, y0, t0);
            t1 = fmaf(e1, y1, t1);
        }
        s += s0 + s1;
        t += t0 + t1;
    }
    __device__ __forceinline__ Partial partial() const
    {
        Partial p;
        p.m = m;
        p.s = s;
        p.t = t;
        p.a = a;
        if (!(s > 0.f)) p = gate::empty_partial();
        return p;
    }
};

// Epilogue warps: fold every tile's logits into the row states; at the end
// publish them, and the row tile's last CTA merges and finishes the rows.
__device__ void lm_epilogue(const LmParams &P, const Sync &S, uint32_t tmem)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row_in = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int mt = static_cast<int>(blockIdx.x) % P.n_mt;
    const int row = mt * kBM + row_in;
    const bool valid = row < P.n_rows;
    RowFold f;
    f.reset();
    bool ok = true;
    uint32_t tl = 0;
    for (int k = 0;; ++k) {
        const int nt = vocab_tile(P, k);
        if (nt < 0) break;
        const uint32_t a = tl & 1;
        ok = __all_sync(0xffffffffu, S.wait(L_ACC_FULL + a, (tl >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + a * kBN + c * 32, v);
            tmem_wait_ld(v);
            const int j0 = nt * kBN + c * 32;
            f.add32(v, j0, min(32, P.vocab - j0));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(S.bar(L_ACC_EMPTY + a));
        ++tl;
    }
    // This CTA's states to its slot of the row tile; then the row tile's last CTA
    // (a ticket) merges every slot.  All four epilogue warps reach both named
    // barriers whatever happened; a CTA that gave up a wait takes no ticket, so
    // its row tile is left unfinished (the status word reports the timeout).
    __shared__ int s_last, s_n_done;
    __shared__ int s_done[kBM];
    __shared__ gate::SeqStage s_stage;
    const int slot = static_cast<int>(blockIdx.x) / P.n_mt;
    if (ok && valid)
        __stcg(P.parts + static_cast<int64_t>(row) * P.per_mt + slot, gate::to_f4(f.partial()));
    __threadfence();
    if (threadIdx.x == 64) s_n_done = 0;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (threadIdx.x == 64)
        s_last = !*S.abort_flag &&
                 gate::ticket(P.mt_ctr + mt, static_cast<unsigned>(P.per_mt - 1)) ==
                     static_cast<unsigned>(P.per_mt - 1);
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (!s_last) return;
    __threadfence();  // every thread reads the other CTAs' states after the acquire
    if (valid) {
        Partial p = gate::empty_partial();
        for (int s = 0; s < P.per_mt; ++s)
            gate::merge(p, gate::from_f4(__ldcg(P.parts + static_cast<int64_t>(row) * P.per_mt + s)));
        int lo = 0, cnt = 0;
        const int b = gate::row_outputs(P.g, row, p, p.s > 0.f ? p.a : 0, lo, cnt);
        if (b >= 0) s_done[atomicAdd(&s_n_done, 1)] = b;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    // the sequences whose last row finished here, ranked and gated by one warp
    if (warp != 2) return;
    __threadfence();
    for (int k = 0; k < s_n_done; ++k) {
        const int b = s_done[k];
        const int lo = __ldg(P.g.offsets + b);
        gate::finish_sequence(P.g, b, lo, __ldg(P.g.offsets + b + 1) - lo, s_stage);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    lmhead_gate_kernel(const LmParams P, const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc + 16);
    Sync S{sbase + kOffBar, abort_flag, P.status, P.wait_limit};

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < L_COUNT; ++i)
            mbar_init(S.bar(i), (i == L_ACC_EMPTY || i == L_ACC_EMPTY + 1) ? 4u : 1u);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
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
        if ((threadIdx.x & 31) == 0) lm_producer(P, S, sbase, &tm_x, &tm_w);
        __syncwarp();
        if (blockIdx.x == 0) gate::empty_sequences(P.g);
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) lm_mma(P, S, sbase, tmem);
        __syncwarp();
    } else {
        lm_epilogue(P, S, tmem);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
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

// [rows, cols] bf16, row-major, as a 2-D map {cols, rows} with a {64, box_rows} box.
bool encode_2d(CUtensorMap *map, const void *base, int rows, int cols, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row tiles, and CTAs per row tile: a whole number of groups on the SMs.
void lm_plan(int n_rows, int vocab, int *n_mt, int *n_nt, int *per_mt)
{
    *n_mt = std::max(1, (n_rows + kBM - 1) / kBM);
    *n_nt = (vocab + kBN - 1) / kBN;
    const int n_sm = device_sm_count();
    *per_mt = std::max(1, std::min(n_sm / *n_mt, *n_nt));
}

}  // namespace

bool lmhead_shape_ok(int32_t n_rows, int32_t hidden, int32_t vocab)
{
    return n_rows >= 0 && hidden >= kBK && hidden % kBK == 0 && vocab >= 1 &&
           n_rows <= device_sm_count() * kBM;
}

size_t lmhead_workspace_bytes(int32_t n_rows, int32_t vocab, int32_t batch)
{
    int n_mt, n_nt, per_mt;
    lm_plan(std::max(n_rows, 0), std::max(vocab, 1), &n_mt, &n_nt, &per_mt);
    size_t off = kWsHeader;
    off = align_up(off + static_cast<size_t>(std::max(batch, 0)) * sizeof(unsigned), 16);  // sequences
    off = align_up(off + static_cast<size_t>(n_mt) * sizeof(unsigned), 256);             // row tiles
    return off + static_cast<size_t>(std::max(n_rows, 0)) * per_mt * sizeof(float4);
}

cudaError_t launch_lmhead_gate(const void *hidden, const void *w_lm, int32_t n_rows,
                               int32_t hidden_dim, int32_t vocab, const int32_t *seq_row_offsets,
                               const int32_t *row_pos, int32_t batch, int32_t seq_len,
                               int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                               float *conf_out, float *entropy_out, int32_t *unmask_rows,
                               float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                               int32_t *seq_tokens, int32_t *decode_step, void *workspace,
                               cudaStream_t stream)
{
    LmParams P;
    P.n_rows = n_rows;
    P.hidden = hidden_dim;
    P.vocab = vocab;
    lm_plan(n_rows, vocab, &P.n_mt, &P.n_nt, &P.per_mt);
    P.grid = P.n_mt * P.per_mt;
    gate::GateArgs &g = P.g;
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
    P.status = reinterpret_cast<uint32_t *>(ws);
    g.status = P.status;
    P.wait_limit = wait_limit_cycles();
    size_t off = kWsHeader;
    g.seq_ctr = reinterpret_cast<unsigned *>(ws + off);
    off = align_up(off + static_cast<size_t>(batch) * sizeof(unsigned), 16);
    P.mt_ctr = reinterpret_cast<unsigned *>(ws + off);
    off = align_up(off + static_cast<size_t>(P.n_mt) * sizeof(unsigned), 256);
    P.parts = reinterpret_cast<float4 *>(ws + off);
    CUtensorMap tx = {}, tw = {};
    if (n_rows == 0) {
        P.n_nt = 0;  // no GEMM: only the sequences' empty outputs
    } else if (!encode_2d(&tx, hidden, n_rows, hidden_dim, kBM) ||
               !encode_2d(&tw, w_lm, vocab, hidden_dim, kBN)) {
        return cudaErrorInvalidValue;
    }
    return launch(lmhead_gate_kernel, dim3(P.grid), dim3(kThreads), kBytes, stream, P, tx, tw);
}

}  // namespace ec
