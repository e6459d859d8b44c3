/*
 * ec_cover.h — COVER's stability-aware seed score, beside the hot path of ec.h
 * (same conventions: caller-owned device buffers, asynchronous work on
 * `stream`, argument errors returned before any launch, device-side index
 * errors reported in the workspace's status word).
 *
 * "Stop the Flip-Flop: Verifica Preservante il Contesto per una Decodifica di
 * Diffusione Veloce e Revocabile" (COVER), Italian technical summary
 * (gist.science/it/paper/2602.06161), section "Metodologia: COVER", item 2
 * "Selezione dei Seed Sensibile alla Stabilità": the decoded tokens to verify
 * (the seeds of ec_selective_attention_cover) are chosen by
 *     Score = u (1 + d_in) / (1 + d_out),
 * u the entropy of the token's current assignment, d_in how much the positions
 * still masked rely on the token as context, d_out how strongly the token
 * attends to the positions drafted at this step.
 */
#ifndef ENTROPY_GATED_KV_DECODE_EC_COVER_H
#define ENTROPY_GATED_KV_DECODE_EC_COVER_H

#include "ec.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace ec_cover_seed_score needs (EC_WORKSPACE_ALIGN-
 * aligned, status word first): the status header, one 16-byte running softmax
 * state per (row, head, key range) and four floats per (row, head).  Sizes out
 * of range (batch or seq_len or n_heads below 1, r_max below 0) give the header's
 * 256 bytes; the call itself rejects them. */
size_t ec_cover_score_workspace_size(int32_t batch, int32_t seq_len, int32_t r_max,
                                     int32_t n_heads);

/*
 * The seed score of every candidate row and the seed set, from one layer's
 * attention (the page gives no formula for d_in and d_out; this is the plain
 * reading over that layer's head-averaged attention probabilities):
 *
 *   a^h_{r,j} = softmax over j < seq_len of scale * q[b,r,h,:] . k_cache[b,j,g,:],
 *               g = h / (n_heads / n_kv_heads)   (the bidirectional attention of
 *               ec_selective_attention, over the cache as it stands)
 *   d_in(c)   = (1/H) sum_h sum_{r < count[b], role[b,r] & 1} a^h_{r, idx[b,c]}
 *   d_out(c)  = (1/H) sum_h sum_{j : drafted[b,j] != 0} a^h_{c, j}
 *   score(c)  = u[b,c] (1 + d_in(c)) / (1 + d_out(c))
 *   seeds[b, 0..n_seed): the positions idx[b,c] of the candidates ranked by
 *               score descending, ties to the lower position (NaN last), -1
 *               where the sequence has fewer candidates.
 *
 * q bf16 device [batch, r_max, n_heads, head_dim]: the recomputed rows'
 * queries (rows r < count[b], at positions idx[b*idx_stride + r], as for
 * ec_selective_attention); k_cache bf16 device [batch, seq_len, n_kv_heads,
 * head_dim] after the step's write-back; head_dim 64 or 128; q and k_cache
 * 16-byte aligned.  role uint8 device [batch, r_max]: bit 0 = the row's
 * position is still masked after this step's unmasking (its query counts toward
 * d_in), bit 1 = the row is a candidate (a decoded token that may be verified);
 * a row may carry both; other bits are ignored.  Positions are distinct within a
 * sequence (as ec_build_recompute_set produces them); two candidate rows at one
 * position tie on both keys and share a seed slot, so the list then ends early
 * (-1).  drafted uint8 device [batch, seq_len]: nonzero at the
 * positions unmasked at this step.  u float32 device [batch, r_max]: a
 * candidate row's entropy (the entropy output of ec_decode_step for the logits
 * row of that position).  Outputs float32 device [batch, r_max]: d_in, d_out,
 * score, written at the candidate rows r < count[b] only (other rows are left
 * unchanged); seeds int32 device [batch, n_seed] (may be NULL when n_seed == 0).
 *
 * Arithmetic: float32 dot products and sums, expf, one softmax normaliser per
 * (row, head) over all keys; the ranking compares the float32 scores.
 * Errors: EC_ERR_DTYPE for an unknown dtype, EC_ERR_UNSUPPORTED for float32 or
 * another head_dim, EC_ERR_SHAPE for sizes out of range (n_heads not a
 * multiple of n_kv_heads, idx_stride < r_max, n_seed < 0, a non-finite scale),
 * EC_ERR_NULL, EC_ERR_ALIGN, EC_ERR_WORKSPACE (ec_cover_score_workspace_size
 * bytes, zeroed once).  A count outside [0, r_max] is clamped; a row index
 * outside [0, seq_len) drops the row and sets EC_DEV_BAD_INDEX.  Calls on the
 * same workspace must not overlap.  Up to five kernel launches
 * (ec_cover_score_kernel_count), none of which waits on another CTA.
 */
ec_status ec_cover_seed_score(const void *q, const void *k_cache, const int32_t *idx,
                              int64_t idx_stride, const int32_t *count, const uint8_t *role,
                              const uint8_t *drafted, const float *u, ec_dtype dtype,
                              int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                              int32_t n_kv_heads, int32_t head_dim, float scale, int32_t n_seed,
                              float *d_in, float *d_out, float *score, int32_t *seeds,
                              void *workspace, size_t workspace_bytes, ec_stream_t stream);

/* Kernel launches one ec_cover_seed_score call makes with these sizes. */
int32_t ec_cover_score_kernel_count(int32_t batch, int32_t r_max, int32_t n_seed);

#ifdef __cplusplus
}
#endif

#endif
