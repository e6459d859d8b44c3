// Test-only host build of the seed-score kernels' per-item code
// (entropy_gated_kv_decode_b300/csrc/cover_score.cuh): every item of each of
// the five kernels, in launch order, on the CPU.  The items of one kernel never
// read what another item of the same kernel writes, so running them one after
// another computes what the grid computes.  It checks the kernels' index
// arithmetic and their float32 results against the oracle on a machine without
// a GPU; the library itself runs these functions only on the GPU.
#include <vector>

#include "cover_score.cuh"

using namespace ec::cover;

extern "C" int cover_score_on_host(const uint16_t *q, const uint16_t *k_cache, const int32_t *idx,
                                   int64_t idx_stride, const int32_t *count, const uint8_t *role,
                                   const uint8_t *drafted, const float *u, int32_t batch,
                                   int32_t seq_len, int32_t r_max, int32_t n_heads,
                                   int32_t n_kv_heads, int32_t head_dim, float scale,
                                   int32_t n_seed, float *d_in, float *d_out, float *score,
                                   int32_t *seeds, uint32_t *status)
{
    if (head_dim != 64 && head_dim != 128) return -1;
    Args A;
    A.q = q;
    A.k_cache = k_cache;
    A.idx = idx;
    A.idx_stride = idx_stride;
    A.count = count;
    A.role = role;
    A.drafted = drafted;
    A.u = u;
    A.B = batch;
    A.L = seq_len;
    A.R = r_max;
    A.H = n_heads;
    A.Hkv = n_kv_heads;
    plan(batch, seq_len, r_max, n_heads, &A.n_chunks, &A.chunk_len);
    A.n_seed = n_seed;
    A.scale = scale;
    const size_t rows = static_cast<size_t>(batch) * r_max * n_heads;
    std::vector<Part> part(rows * A.n_chunks);
    std::vector<float> stat_m(rows), stat_z(rows), dout_h(rows), din_h(rows);
    A.part = part.data();
    A.stat_m = stat_m.data();
    A.stat_z = stat_z.data();
    A.dout_h = dout_h.data();
    A.din_h = din_h.data();
    A.d_in = d_in;
    A.d_out = d_out;
    A.score = score;
    A.seeds = seeds;
    A.status = status;
    for (int64_t t = 0; t < partial_items(A); ++t)
        head_dim == 64 ? partial_item<64>(A, t) : partial_item<128>(A, t);
    for (int64_t t = 0; t < head_items(A); ++t) stats_item(A, t);
    for (int64_t t = 0; t < head_items(A); ++t)
        head_dim == 64 ? din_item<64>(A, t) : din_item<128>(A, t);
    for (int64_t t = 0; t < final_items(A); ++t) final_item(A, t);
    if (n_seed > 0)
        for (int64_t t = 0; t < rank_items(A); ++t) rank_item(A, t);
    return A.n_chunks;
}
