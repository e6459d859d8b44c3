// COVER's stability-aware seed score: the arithmetic of its kernels, one work
// item (one thread) at a time.
//
// "Stop the Flip-Flop: Verifica Preservante il Contesto per una Decodifica di
// Diffusione Veloce e Revocabile" (COVER), Italian technical summary, section
// "Metodologia: COVER", item 2 "Selezione dei Seed Sensibile alla Stabilità":
// a decoded token is scored by u (1 + d_in) / (1 + d_out), u the entropy of its
// current assignment, d_in how much the still-masked positions rely on it as
// context, d_out how strongly it attends to the positions drafted at this step;
// the seeds to verify are the best scores.  With one layer's attention
// probabilities a^h_{r,j} = softmax_j(scale q_{r,h} . k_{j,g(h)}) over all L keys:
//   d_in(c)  = (1/H) sum_h sum_{still-masked rows r} a^h_{r, p_c}
//   d_out(c) = (1/H) sum_h sum_{drafted positions j} a^h_{c, j}
//
// Five steps, each a kernel over independent items:
//   partial  (b, key range, kv head, row, head in group): the row's running
//            maximum m, sum z of e^{s - m} and the drafted keys' share zd over
//            one range of keys (the threads of a warp share the key rows);
//   stats    (b, row, head): the ranges merged: M, Z, and ZD / Z, the head's
//            part of d_out;
//   din      (b, candidate, head): the candidate's key against every
//            still-masked query of the head: sum e^{s - M} / Z;
//   final    (b, candidate): the head means, the score, and -1 in every seed slot;
//   rank     (b, candidate): its place by (score desc, position asc) among the
//            sequence's candidates, written to the seed slot of that place.
// The functions are plain C++ usable from host and device code; the library
// runs them only in its kernels.
#pragma once

#include <math.h>
#include <stdint.h>
#include <string.h>

#include "ec.h"

#if defined(__CUDACC__)
#define EC_HD __host__ __device__ __forceinline__
#else
#define EC_HD inline
#endif
#if defined(__CUDA_ARCH__)
#define EC_UNROLL _Pragma("unroll")
#else
#define EC_UNROLL
#endif

namespace ec {
namespace cover {

struct alignas(16) Vec16 {
    uint32_t w[4];
};

// A key range's running softmax state for one (row, head).
struct alignas(16) Part {
    float m, z, zd, pad;
};

struct Args {
    const uint16_t *q;        // bf16 [B, R, H, D]
    const uint16_t *k_cache;  // bf16 [B, L, Hkv, D]
    const int32_t *idx;       // [B, idx_stride] positions of the rows
    int64_t idx_stride;
    const int32_t *count;     // [B]
    const uint8_t *role;      // [B, R]: bit 0 still masked, bit 1 candidate
    const uint8_t *drafted;   // [B, L]: nonzero = drafted at this step
    const float *u;           // [B, R]
    int32_t B, L, R, H, Hkv, n_chunks, chunk_len, n_seed;
    float scale;
    Part *part;                             // [B, R, H, n_chunks]
    float *stat_m, *stat_z, *dout_h, *din_h;  // [B, R, H]
    float *d_in, *d_out, *score;            // [B, R]
    int32_t *seeds;                         // [B, n_seed]
    uint32_t *status;
};

EC_HD float as_float(uint32_t x)
{
#if defined(__CUDA_ARCH__)
    return __uint_as_float(x);
#else
    float f;
    memcpy(&f, &x, sizeof f);
    return f;
#endif
}

// bf16 pair (low half first) widened exactly
EC_HD float lo_f(uint32_t x) { return as_float(x << 16); }
EC_HD float hi_f(uint32_t x) { return as_float(x & 0xffff0000u); }

EC_HD Vec16 load16(const uint16_t *p)
{
#if defined(__CUDA_ARCH__)
    return *reinterpret_cast<const Vec16 *>(p);
#else
    Vec16 v;
    memcpy(&v, p, sizeof v);
    return v;
#endif
}

EC_HD void flag(uint32_t *status, uint32_t bits)
{
#if defined(__CUDA_ARCH__)
    if (status) atomicOr(status, bits);
#else
    if (status) *status |= bits;
#endif
}

template <int D>
EC_HD void load_row(const uint16_t *p, uint32_t (&w)[D / 2])
{
    EC_UNROLL
    for (int i = 0; i < D / 8; ++i) {
        const Vec16 v = load16(p + 8 * i);
        EC_UNROLL
        for (int e = 0; e < 4; ++e) w[4 * i + e] = v.w[e];
    }
}

// sum_e a_e b_e in float32: four running sums (element pairs 4i + e go to sum
// e), added as (s0 + s1) + (s2 + s3); a held in registers, b read from memory.
// Both operand orders give the same bits.
template <int D>
EC_HD float dot_row(const uint32_t (&a)[D / 2], const uint16_t *b)
{
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    EC_UNROLL
    for (int i = 0; i < D / 8; ++i) {
        const Vec16 v = load16(b + 8 * i);
        EC_UNROLL
        for (int e = 0; e < 4; ++e) {
            s[e] = fmaf(lo_f(a[4 * i + e]), lo_f(v.w[e]), s[e]);
            s[e] = fmaf(hi_f(a[4 * i + e]), hi_f(v.w[e]), s[e]);
        }
    }
    return (s[0] + s[1]) + (s[2] + s[3]);
}

// Position of row r of sequence b, or -1 when the row is past count (clamped
// to [0, R]) or its index is outside [0, L).
EC_HD int32_t row_pos(const Args &A, int32_t b, int32_t r)
{
    int32_t c = A.count[b];
    c = c < 0 ? 0 : (c > A.R ? A.R : c);
    if (r >= c) return -1;
    const int32_t p = A.idx[b * A.idx_stride + r];
    return (p >= 0 && p < A.L) ? p : -1;
}

EC_HD uint8_t role_of(const Args &A, int32_t b, int32_t r) { return A.role[(int64_t)b * A.R + r]; }

EC_HD int64_t partial_items(const Args &A) { return (int64_t)A.B * A.n_chunks * A.R * A.H; }
EC_HD int64_t head_items(const Args &A) { return (int64_t)A.B * A.R * A.H; }
EC_HD int32_t final_span(const Args &A) { return A.R > A.n_seed ? A.R : A.n_seed; }
EC_HD int64_t final_items(const Args &A) { return (int64_t)A.B * final_span(A); }
EC_HD int64_t rank_items(const Args &A) { return (int64_t)A.B * A.R; }

// item t -> (b, key range, kv head g, row r, head in group hg), hg fastest
template <int D>
EC_HD void partial_item(const Args &A, int64_t t)
{
    const int32_t G = A.H / A.Hkv;
    const int32_t hg = static_cast<int32_t>(t % G);
    t /= G;
    const int32_t r = static_cast<int32_t>(t % A.R);
    t /= A.R;
    const int32_t g = static_cast<int32_t>(t % A.Hkv);
    t /= A.Hkv;
    const int32_t ch = static_cast<int32_t>(t % A.n_chunks);
    const int32_t b = static_cast<int32_t>(t / A.n_chunks);
    if (row_pos(A, b, r) < 0 || !(role_of(A, b, r) & 3)) return;
    const int64_t row = ((int64_t)b * A.R + r) * A.H + g * G + hg;
    uint32_t qw[D / 2];
    load_row<D>(A.q + row * D, qw);
    const int32_t j0 = ch * A.chunk_len;
    const int32_t j1 = j0 + A.chunk_len < A.L ? j0 + A.chunk_len : A.L;
    float m = -INFINITY, z = 0.f, zd = 0.f;
    for (int32_t j = j0; j < j1; ++j) {
        const float s = A.scale * dot_row<D>(qw, A.k_cache + (((int64_t)b * A.L + j) * A.Hkv + g) * D);
        const float dr = A.drafted[(int64_t)b * A.L + j] ? 1.f : 0.f;
        if (s > m) {
            const float c = expf(m - s);
            z = z * c + 1.f;
            zd = zd * c + dr;
            m = s;
        } else {
            const float e = expf(s - m);
            z += e;
            zd += dr * e;
        }
    }
    Part P;
    P.m = m;
    P.z = z;
    P.zd = zd;
    P.pad = 0.f;
    A.part[row * A.n_chunks + ch] = P;
}

// item t -> (b, r, h), h fastest
EC_HD void stats_item(const Args &A, int64_t t)
{
    const int32_t h = static_cast<int32_t>(t % A.H);
    t /= A.H;
    const int32_t r = static_cast<int32_t>(t % A.R);
    const int32_t b = static_cast<int32_t>(t / A.R);
    if (row_pos(A, b, r) < 0 || !(role_of(A, b, r) & 3)) return;
    const int64_t row = ((int64_t)b * A.R + r) * A.H + h;
    const Part *P = A.part + row * A.n_chunks;
    float M = -INFINITY;
    for (int32_t k = 0; k < A.n_chunks; ++k)
        if (P[k].z > 0.f && P[k].m > M) M = P[k].m;
    float Z = 0.f, ZD = 0.f;
    for (int32_t k = 0; k < A.n_chunks; ++k)
        if (P[k].z > 0.f) {  // an empty range holds nothing
            const float c = expf(P[k].m - M);
            Z += P[k].z * c;
            ZD += P[k].zd * c;
        }
    A.stat_m[row] = M;
    A.stat_z[row] = Z;
    A.dout_h[row] = ZD / Z;
}

// item t -> (b, candidate row c, h), h fastest
template <int D>
EC_HD void din_item(const Args &A, int64_t t)
{
    const int32_t h = static_cast<int32_t>(t % A.H);
    t /= A.H;
    const int32_t c = static_cast<int32_t>(t % A.R);
    const int32_t b = static_cast<int32_t>(t / A.R);
    const int32_t pc = row_pos(A, b, c);
    if (pc < 0 || !(role_of(A, b, c) & 2)) return;
    const int32_t g = h / (A.H / A.Hkv);
    uint32_t kw[D / 2];
    load_row<D>(A.k_cache + (((int64_t)b * A.L + pc) * A.Hkv + g) * D, kw);
    float acc = 0.f;
    for (int32_t r = 0; r < A.R; ++r) {
        if (row_pos(A, b, r) < 0 || !(role_of(A, b, r) & 1)) continue;
        const int64_t row = ((int64_t)b * A.R + r) * A.H + h;
        const float s = A.scale * dot_row<D>(kw, A.q + row * D);
        acc += expf(s - A.stat_m[row]) / A.stat_z[row];
    }
    A.din_h[((int64_t)b * A.R + c) * A.H + h] = acc;
}

// item t -> (b, c) for c < max(R, n_seed)
EC_HD void final_item(const Args &A, int64_t t)
{
    const int32_t span = final_span(A);
    const int32_t c = static_cast<int32_t>(t % span);
    const int32_t b = static_cast<int32_t>(t / span);
    if (c < A.n_seed) A.seeds[(int64_t)b * A.n_seed + c] = -1;
    if (c >= A.R) return;
    int32_t cnt = A.count[b];
    cnt = cnt < 0 ? 0 : (cnt > A.R ? A.R : cnt);
    if (c < cnt) {
        const int32_t p = A.idx[b * A.idx_stride + c];
        if (p < 0 || p >= A.L) flag(A.status, EC_DEV_BAD_INDEX);
    }
    if (row_pos(A, b, c) < 0 || !(role_of(A, b, c) & 2)) return;
    const int64_t row = ((int64_t)b * A.R + c) * A.H;
    float din = 0.f, dout = 0.f;
    for (int32_t h = 0; h < A.H; ++h) {
        din += A.din_h[row + h];
        dout += A.dout_h[row + h];
    }
    din /= static_cast<float>(A.H);
    dout /= static_cast<float>(A.H);
    const int64_t o = (int64_t)b * A.R + c;
    A.d_in[o] = din;
    A.d_out[o] = dout;
    A.score[o] = A.u[o] * (1.f + din) / (1.f + dout);
}

// ranking key: the score, NaN below everything
EC_HD float rank_key(float s) { return s == s ? s : -INFINITY; }

// item t -> (b, c), c fastest
EC_HD void rank_item(const Args &A, int64_t t)
{
    const int32_t c = static_cast<int32_t>(t % A.R);
    const int32_t b = static_cast<int32_t>(t / A.R);
    const int32_t pc = row_pos(A, b, c);
    if (pc < 0 || !(role_of(A, b, c) & 2)) return;
    const float key = rank_key(A.score[(int64_t)b * A.R + c]);
    int32_t rank = 0;
    for (int32_t o = 0; o < A.R; ++o) {
        const int32_t po = row_pos(A, b, o);
        if (o == c || po < 0 || !(role_of(A, b, o) & 2)) continue;
        const float ko = rank_key(A.score[(int64_t)b * A.R + o]);
        if (ko > key || (ko == key && po < pc)) ++rank;
    }
    if (rank < A.n_seed) A.seeds[(int64_t)b * A.n_seed + rank] = pc;
}

// Key ranges per (row, head): about 2^21 partial items in all, ranges of at
// least 64 keys where the rows alone give fewer.
EC_HD void plan(int32_t B, int32_t L, int32_t R, int32_t H, int32_t *n_chunks, int32_t *chunk_len)
{
    int64_t rows = (int64_t)B * R * H;
    if (rows < 1) rows = 1;
    int64_t n = (L + 63) / 64;
    const int64_t want = (((int64_t)1 << 21) + rows - 1) / rows;
    if (want < n) n = want;
    if (n < 1) n = 1;
    *n_chunks = static_cast<int32_t>(n);
    *chunk_len = static_cast<int32_t>((L + n - 1) / n);
}

}  // namespace cover
}  // namespace ec
