/*
 * ec.h — C ABI of the EntropyCache per-step hot path on one B300 (sm_103a).
 *
 * The method: "EntropyCache: Decoded Token Entropy Guided KV Caching for
 * Diffusion Language Models".  Passages cited below by page and section:
 *   [EC-it] Italian summary (gist.science/it/paper/2603.18489), section
 *           "2. Metodologia", subsection "Algoritmo di Funzionamento", steps 1-3;
 *           section "1. Il Problema" for the bidirectional attention.
 *   [EC-ar] Arabic technical summary (gist.science/ar/paper/2603.18489), section
 *           "2. Methodology", subsection "Algorithm workflow", phases 1-3 and the
 *           equation E_{t+1} = max_{i in D_{t+1}} ( -sum_j p_ij log p_ij ).
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" are CUDA device pointers; every buffer is owned by
 *     the caller, the library allocates nothing and keeps no host-side state
 *     (beyond per-device lookups it caches, such as the address of the fixed
 *     scratch array of ec_decode_step_noalloc).
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and runs asynchronously; nothing synchronises the host except
 *     ec_read_device_status().
 *   - Argument errors (null pointers, shapes, dtypes, alignment, workspace size)
 *     are detected on the host and returned before anything is launched.  A
 *     failed launch returns EC_ERR_CUDA.  Inconsistent device-resident indices
 *     (a row position outside [0, L), a count above its bound, an unsorted index
 *     set) cannot be seen from the host: the kernels keep every access in bounds,
 *     skip the offending item and set a bit in the workspace's status word, which
 *     ec_read_device_status() returns.
 *   - Floating-point work is float32 on float32 or bfloat16 inputs; NaN inputs
 *     are outside the contract.
 */
#ifndef ENTROPY_GATED_KV_DECODE_EC_H
#define ENTROPY_GATED_KV_DECODE_EC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *ec_stream_t;

typedef enum {
    EC_OK = 0,
    EC_ERR_NULL = -1,        /* a required pointer is NULL */
    EC_ERR_SHAPE = -2,       /* a size or scalar argument is out of range */
    EC_ERR_DTYPE = -3,       /* unsupported element type */
    EC_ERR_ALIGN = -4,       /* a pointer or row stride breaks the 16-byte rule */
    EC_ERR_WORKSPACE = -5,   /* workspace missing, misaligned or too small */
    EC_ERR_CUDA = -6,        /* a CUDA runtime call or launch failed */
    EC_ERR_UNSUPPORTED = -7, /* valid request this library does not implement */
    EC_ERR_SCRATCH_LIMIT = -8 /* request needs more than the fixed built-in scratch */
} ec_status;

typedef enum { EC_F32 = 0, EC_BF16 = 1 } ec_dtype;

/* Bits of the device status word (first 4 bytes of every workspace). */
#define EC_DEV_BAD_OFFSETS 0x1u  /* seq_row_offsets not 0 .. n_rows non-decreasing */
#define EC_DEV_BAD_ROW_POS 0x2u  /* a row position outside [0, seq_len) */
#define EC_DEV_BAD_COUNT 0x4u    /* a recompute count above r_max or seq_len */
#define EC_DEV_BAD_INDEX 0x8u    /* an index outside [0, seq_len) or not ascending */
#define EC_DEV_TIMEOUT 0x10u     /* a bounded wait inside a kernel gave up */
#define EC_DEV_BAD_LABEL 0x20u   /* a SimSD section or step label out of range */

/* Human-readable name of a status code (static string). */
const char *ec_status_str(int status);

/* ABI revision of this header; bumped on any incompatible change. */
#define EC_ABI_VERSION 1
int ec_abi_version(void);

/*
 * Test hook for the device-side timeout path.  Every wait inside the kernels
 * (a ring stage landing, a tensor-core product completing) is bounded: by
 * default it gives up after about 2 s, sets EC_DEV_TIMEOUT in the workspace's
 * status word, lets the copies and tensor-core operations it already started
 * complete, releases its tensor memory and returns, leaving the context usable.
 * This sets that limit, in SM clock cycles, for launches made afterwards by any
 * thread of the process (0 restores the default); a limit of a few hundred
 * cycles makes the first wait on data give up.  After a call that timed out,
 * zero its workspace (ec_workspace_init) before the next call.  Not for use in
 * production: it changes no result of a call that does not time out.
 * Returns EC_ERR_SHAPE for a negative value.
 */
ec_status ec_debug_set_wait_limit(int64_t cycles);

/* Alignment, in bytes, that every workspace pointer must have. */
#define EC_WORKSPACE_ALIGN 256

/*
 * Zero a workspace (cudaMemsetAsync).  Every workspace must be zeroed once
 * before its first use; the kernels leave their counters at zero on exit, so
 * later calls need no further reset.  After a call whose device status reports
 * EC_DEV_TIMEOUT the counters may not be back at zero: zero the workspace again.
 * Returns EC_ERR_CUDA if the memset fails.
 */
ec_status ec_workspace_init(void *workspace, size_t workspace_bytes, ec_stream_t stream);

/*
 * Read, and clear, the device status word of `workspace`.  Synchronises
 * `stream` first.  *bits receives the EC_DEV_* flags set since the last read.
 */
ec_status ec_read_device_status(void *workspace, uint32_t *bits, ec_stream_t stream);

/* ------------------------------------------------------------------------- */
/* (a) decode and gate                                                        */
/* ------------------------------------------------------------------------- */

/* Bytes of device workspace ec_decode_step needs for this many rows/sequences. */
size_t ec_decode_workspace_size(int32_t n_rows, int32_t batch);

/*
 * One denoising step's decode and gate ([EC-it] steps 1-2; [EC-ar] phases 2-3).
 *
 * Inputs
 *   logits        device, [n_rows, vocab] row-major with `row_stride` elements
 *                 between rows, `dtype` EC_F32 or EC_BF16.  The base pointer must be
 *                 16-byte aligned and row_stride * element size a multiple of 16.
 *                 Each row holds the logits of one currently masked position.
 *   seq_row_offsets device int32 [batch + 1]: the rows of sequence b are
 *                 [seq_row_offsets[b], seq_row_offsets[b+1]); offsets[0] = 0,
 *                 non-decreasing, offsets[batch] = n_rows.
 *   row_pos       device int32 [n_rows]: position in [0, seq_len) of each row
 *                 (distinct within a sequence).
 *   n_unmask      tokens unmasked per sequence this step (1 .. 1024).
 *   tau           entropy threshold in nats (finite).
 *   step          index of this denoising step, written to the decode-time log.
 * Outputs (device)
 *   token_out, conf_out, entropy_out  [n_rows]: greedy token (first index of the
 *                 maximum logit), its softmax probability, and the Shannon entropy
 *                 -sum_j p_j ln p_j of the row's softmax, in nats.
 *   unmask_rows   int32 [batch, n_unmask]: per sequence, the rows unmasked this
 *                 step in rank order (confidence descending, position ascending
 *                 on ties), at most the sequence's row count; the rest -1.
 *   max_entropy   float [batch]: E = max entropy over the rows unmasked this
 *                 step ([EC-ar] E_{t+1}); -inf for a sequence with no rows.
 *   refresh       uint8 [batch]: 1 when E > tau (strict), i.e. the next forward
 *                 must recompute the whole KV cache; 0 when E <= tau.
 * State (device, in/out, [batch, seq_len] each)
 *   is_masked     uint8: cleared at every unmasked position.
 *   seq_tokens    int32: receives the decoded token at every unmasked position.
 *   decode_step   int32: receives `step` at every unmasked position (the
 *                 decode-time log of [EC-ar] phase 3; -1 = never decoded).
 * Workspace: device, EC_WORKSPACE_ALIGN-aligned, at least
 *   ec_decode_workspace_size(n_rows, batch) bytes, zeroed before first use (its
 *   counters return to zero after every call).
 * Calls on the same workspace must not overlap in time.
 * Launches: a streaming kernel and a finishing kernel chained by programmatic
 * dependent launch (the finishing kernel alone when n_rows == 0).  When the
 * status word reports EC_DEV_TIMEOUT (a bounded wait ran out) no per-row output
 * of that call is written; zero the workspace again (ec_workspace_init) before
 * reusing it.
 */
ec_status ec_decode_step(const void *logits, ec_dtype dtype, int64_t row_stride,
                         int32_t n_rows, int32_t vocab, const int32_t *seq_row_offsets,
                         const int32_t *row_pos, int32_t batch, int32_t seq_len,
                         int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                         float *conf_out, float *entropy_out, int32_t *unmask_rows,
                         float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                         int32_t *seq_tokens, int32_t *decode_step, void *workspace,
                         size_t workspace_bytes, ec_stream_t stream);

/*
 * ec_decode_step without a caller-provided workspace: it allocates nothing.
 *
 * The paper has no counterpart; this is a deployment convenience.  Some callers
 * cannot allocate device memory on their own: their device memory is owned by a
 * host framework or a fixed-size pool that hands out only the tensors of the
 * model, or they run in a latency-critical decode loop where a cudaMalloc (which
 * may synchronise the device) is not acceptable.  This entry point takes the same
 * inputs, outputs and state as ec_decode_step and keeps its scratch (counters and
 * per-slice partial results) in a fixed array compiled into the library.
 *
 *   - Limit: ec_decode_workspace_size(n_rows, batch) must not exceed 2 MiB
 *     (about 2000 logits rows); larger requests return EC_ERR_SCRATCH_LIMIT
 *     before anything is enqueued.
 *   - Every device that loads the library holds those 2 MiB until the process exits.
 *   - The first call on a device looks the array's device address up (with that
 *     device current); make that first call before any stream capture.
 *   - All calls share the one array: each call first clears the part that must
 *     start at zero, on `stream`.  Calls whose kernels can overlap on the GPU
 *     (different streams, no ordering between them) race on the array and give
 *     undefined results; serialise them.
 *   - The call's device status bits (bad offsets or positions, EC_DEV_TIMEOUT when
 *     a bounded wait ran out and the step was left unfinished) stay in the array:
 *     read them with ec_decode_noalloc_read_status.  The return value of this call
 *     reports only what the host checks and the launch found.
 */
ec_status ec_decode_step_noalloc(const void *logits, ec_dtype dtype, int64_t row_stride,
                                 int32_t n_rows, int32_t vocab, const int32_t *seq_row_offsets,
                                 const int32_t *row_pos, int32_t batch, int32_t seq_len,
                                 int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                                 float *conf_out, float *entropy_out, int32_t *unmask_rows,
                                 float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                                 int32_t *seq_tokens, int32_t *decode_step, ec_stream_t stream);

/*
 * Status bits (EC_DEV_* flags, 0 = clean) of the last ec_decode_step_noalloc call
 * on the current device: synchronizes `stream` (the stream of that call), then
 * copies the status word out of the library's scratch array, allocating nothing.
 * The next ec_decode_step_noalloc call clears it.  EC_ERR_NULL for a null `bits`.
 */
ec_status ec_decode_noalloc_read_status(uint32_t *bits, ec_stream_t stream);

/* Bytes of device workspace ec_lmhead_decode_step needs (depends on the
 * current device's SM count). */
size_t ec_lmhead_workspace_size(int32_t n_rows, int32_t vocab, int32_t batch);

/*
 * The decode-and-gate step with the logits computed inside it: the LM head's
 * product hidden x W_lm^T on the tensor cores, each row's logits folded into its
 * softmax statistics as they leave the accumulator, so the [n_rows, vocab] logits
 * are never written to memory ([EC-it] section 2, observation 1: the decision is
 * an O(V) operation per decoded token; "Algoritmo di Funzionamento" point 3 and
 * section 4: it costs a constant, negligible share of inference).
 *
 *   logits[i, j] = sum_e hidden[i, e] * w_lm[j, e]   (float32 accumulation of the
 *   bf16 products), then everything ec_decode_step computes from those logits.
 *
 * hidden  bf16 device [n_rows, hidden_dim], rows contiguous, 16-byte aligned;
 * w_lm    bf16 device [vocab, hidden_dim] (one vocabulary entry's weights per row,
 *         as a linear layer stores them), 16-byte aligned.
 * hidden_dim a multiple of 64; n_rows at most 128 x the SM count (18944 on a
 * B300).  Every other argument, output and state buffer is as in
 * ec_decode_step; the token is the first index of the largest float32 logit.
 * Workspace: ec_lmhead_workspace_size bytes, EC_WORKSPACE_ALIGN-aligned, zeroed
 * before first use (counters return to zero after every call; zero it again
 * after a call whose status reports EC_DEV_TIMEOUT).
 */
ec_status ec_lmhead_decode_step(const void *hidden, const void *w_lm, int32_t n_rows,
                                int32_t hidden_dim, int32_t vocab, const int32_t *seq_row_offsets,
                                const int32_t *row_pos, int32_t batch, int32_t seq_len,
                                int32_t n_unmask, float tau, int32_t step, int32_t *token_out,
                                float *conf_out, float *entropy_out, int32_t *unmask_rows,
                                float *max_entropy, uint8_t *refresh, uint8_t *is_masked,
                                int32_t *seq_tokens, int32_t *decode_step, void *workspace,
                                size_t workspace_bytes, ec_stream_t stream);

/*
 * Recompute index set of the next forward ([EC-it] step 2; [EC-ar] phase 1 and
 * phase 3 "token selection").
 *
 *   refresh[b] != 0: idx[b, :] = 0 .. seq_len-1, count[b] = seq_len (full forward).
 *   otherwise:       the masked positions of the active block [block_lo, block_hi)
 *                    together with the min(k, #decoded) decoded positions of largest
 *                    decode_step (ties: lower position first), ascending.
 * Inputs: is_masked uint8 / decode_step int32 device [batch, seq_len] (state
 * after ec_decode_step), refresh uint8 device [batch].  0 <= block_lo <= block_hi
 * <= seq_len, k >= 0.
 * Outputs: idx int32 device [batch, seq_len] (ascending, the unused tail -1),
 * count int32 device [batch].  No workspace.
 */
ec_status ec_build_recompute_set(const uint8_t *is_masked, const int32_t *decode_step,
                                 const uint8_t *refresh, int32_t batch, int32_t seq_len,
                                 int32_t block_lo, int32_t block_hi, int32_t k, int32_t *idx,
                                 int32_t *count, ec_stream_t stream);

/* ------------------------------------------------------------------------- */
/* (b) selective-recompute attention                                          */
/* ------------------------------------------------------------------------- */

/* Bytes of device workspace ec_selective_attention needs on the current device
 * (the split of the keys across CTAs, hence the partial-result storage, depends
 * on its SM count). */
size_t ec_attention_workspace_size(int32_t batch, int32_t seq_len, int32_t r_max,
                                   int32_t n_heads, int32_t n_kv_heads, int32_t head_dim);

/* Kernels one ec_selective_attention call with these arguments launches on the
 * current device (for launch accounting): bf16 with head_dim 64/128 runs one
 * tensor-core kernel (the KV write-back and the merge of units split over
 * several CTAs happen inside it); float32 runs a write-back and the CUDA-core
 * attention.  0 when r_max == 0; -1 for arguments the call rejects. */
int32_t ec_attention_kernel_count(ec_dtype dtype, int32_t batch, int32_t seq_len, int32_t r_max,
                                  int32_t n_heads, int32_t n_kv_heads, int32_t head_dim);

/*
 * Write the freshly projected K/V rows into the caches and run bidirectional
 * attention of the recomputed query rows over every cached key ([EC-it] step 2:
 * recompute only the selected tokens, reuse the cache for the others; [EC-it]
 * section 1 and [EC-ar] section 1: dLLM attention is non-causal).
 *
 *   for b, r < count[b]:  K[b, idx[b*idx_stride + r]] = k_new[b, r]  (same for V)
 *   then for every such r and head h (kv head g = h / (n_heads / n_kv_heads)):
 *     out[b, r, h, :] = softmax_j( scale * q[b,r,h,:] . K[b,j,g,:] ) V[b,j,g,:]
 *   over all j < seq_len.
 *
 * Layouts (contiguous, `dtype` elements): q and out [batch, r_max, n_heads, head_dim];
 * k_new, v_new [batch, r_max, n_kv_heads, head_dim]; k_cache, v_cache (in/out)
 * [batch, seq_len, n_kv_heads, head_dim].  idx int32 device with row stride
 * idx_stride >= r_max; the first count[b] entries of row b are distinct positions in
 * [0, seq_len), strictly ascending (the output of ec_build_recompute_set).
 * count int32 device [batch], 0 <= count[b] <= r_max.  Rows r >= count[b] of
 * `out` are left unchanged.  head_dim 64 or 128; n_heads % n_kv_heads == 0;
 * 16-byte aligned pointers.  Workspace: ec_attention_workspace_size bytes, zeroed
 * before first use.  Calls on the same workspace or caches must not overlap.
 */
ec_status ec_selective_attention(const void *q, const void *k_new, const void *v_new,
                                 const int32_t *idx, int64_t idx_stride, const int32_t *count,
                                 void *k_cache, void *v_cache, void *out, ec_dtype dtype,
                                 int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                 int32_t n_kv_heads, int32_t head_dim, float scale,
                                 void *workspace, size_t workspace_bytes, ec_stream_t stream);

/*
 * ec_selective_attention under SimSD's token-level temporal causal mask
 * ("SimSD - Simple Speculative Decoding in Diffusion Language Models", Italian
 * technical summary, section "Metodologia: SimSD", items 1 and 2).
 *
 * The sequence is a prompt followed by a data section D of reference tokens and
 * a mask section of prediction slots; section[b, j] is 0 (prompt), 1 (data) or 2
 * (mask slot) and tau[b, j] the step label of a data or mask position (the step
 * map; a data token and its paired slot carry the same label; ignored for the
 * prompt).  The write-back and the attention are those of ec_selective_attention
 * except that the softmax of query row r (position i = idx[b*idx_stride + r])
 * runs over the keys j visible to it:
 *   - every prompt key;
 *   - for a mask slot i: data keys with tau[j] < tau[i] and slots with
 *     tau[j] >= tau[i] (the page's rule);
 *   - for a data token i: data keys with tau[j] <= tau[i] (reading: no slot);
 *   - for a prompt token i: nothing more (reading).
 * A row that sees no key is written as zeros.
 *
 * section uint8 and tau int32, device, [batch, seq_len] contiguous; labels of data
 * and mask positions in [1, 2^30).  A label out of range (or a section above 2)
 * hides that key, empties the window of a query at that position and sets
 * EC_DEV_BAD_LABEL.  Every other argument, the workspace (same size as
 * ec_attention_workspace_size) and the errors are those of ec_selective_attention,
 * but only bf16 with head_dim 64 or 128 is implemented (EC_ERR_UNSUPPORTED
 * otherwise); one kernel launch.
 */
ec_status ec_selective_attention_simsd(const void *q, const void *k_new, const void *v_new,
                                       const int32_t *idx, int64_t idx_stride,
                                       const int32_t *count, const uint8_t *section,
                                       const int32_t *tau, void *k_cache, void *v_cache,
                                       void *out, ec_dtype dtype, int32_t batch, int32_t seq_len,
                                       int32_t r_max, int32_t n_heads, int32_t n_kv_heads,
                                       int32_t head_dim, float scale, void *workspace,
                                       size_t workspace_bytes, ec_stream_t stream);

/*
 * ec_selective_attention with COVER's dual view: the KV-cache override and the
 * diagonal correction ("Stop the Flip-Flop: Verifica Preservante il Contesto per
 * una Decodifica di Diffusione Veloce e Revocabile", Italian technical summary,
 * section "Metodologia: COVER", item 1).
 *
 * seed uint8, device, [batch, r_max]: seed[b*r_max + r] != 0 marks recomputed row
 * r as a seed, a decoded token under verification whose input was [MASK], so its
 * k_new / v_new rows are the masked-input K/V.  Then:
 *   - only the non-seed rows are written back: a seed's position keeps the K/V
 *     the cache held before the call (the previous step's), which every other
 *     query attends to;
 *   - a seed row's own column uses its masked-input k_new / v_new instead of the
 *     cached K/V at its position (no self-leakage), and the softmax is taken over
 *     the row so corrected:
 *       out[b, r, h] = softmax_j(scale * q . K'_j) V'_j,  K'_j = cache after the
 *       write-back, except K'_{idx[r]} = k_new[b, r] (and V') when r is a seed.
 * No seeds: the same results as ec_selective_attention.  A fully recomputed
 * sequence (count == seq_len) takes the general path.  Every other argument, the
 * workspace (ec_attention_workspace_size bytes) and the errors are those of
 * ec_selective_attention, but only bf16 with head_dim 64 or 128 is implemented
 * (EC_ERR_UNSUPPORTED otherwise); one kernel launch.
 */
ec_status ec_selective_attention_cover(const void *q, const void *k_new, const void *v_new,
                                       const int32_t *idx, int64_t idx_stride,
                                       const int32_t *count, const uint8_t *seed, void *k_cache,
                                       void *v_cache, void *out, ec_dtype dtype, int32_t batch,
                                       int32_t seq_len, int32_t r_max, int32_t n_heads,
                                       int32_t n_kv_heads, int32_t head_dim, float scale,
                                       void *workspace, size_t workspace_bytes,
                                       ec_stream_t stream);

/* ------------------------------------------------------------------------- */
/* the forward that produces the recomputed rows' queries, keys and values    */
/* ------------------------------------------------------------------------- */

/*
 * Rows of the first layer's input for the recomputed positions ([EC-it] step 2:
 * the partial forward runs only the selected tokens; [EC-it] section 1: a
 * masked diffusion model starts every position as [MASK] and replaces it by
 * the decoded token).
 *
 *   for b, r < count[b], p = idx[b*idx_stride + r]:
 *     x[b, r, :] = table[is_masked[b, p] ? mask_id : seq_tokens[b, p], :]
 *
 * table bf16 device [table_rows, hidden] (hidden a multiple of 8, 16-byte
 * aligned); idx / count as produced by ec_build_recompute_set; seq_tokens int32
 * and is_masked uint8 device [batch, seq_len]; x bf16 device [batch, r_max,
 * hidden].  Rows r >= count[b] of x are left unchanged.  An index outside
 * [0, seq_len) or a token outside [0, table_rows) skips the row and sets
 * EC_DEV_BAD_INDEX.  Workspace: at least EC_WORKSPACE_ALIGN bytes (the status
 * word), aligned, zeroed once.
 */
ec_status ec_embed_rows(const void *table, int64_t table_rows, int32_t hidden, const int32_t *idx,
                        int64_t idx_stride, const int32_t *count, const int32_t *seq_tokens,
                        const uint8_t *is_masked, int32_t mask_id, int32_t batch,
                        int32_t seq_len, int32_t r_max, void *x, void *workspace,
                        size_t workspace_bytes, ec_stream_t stream);

/*
 * Query, key and value projection of the recomputed rows ([EC-it] step 2: the
 * partial forward recomputes Q/K/V of the selected tokens only; a full forward
 * does it for all of them).  bf16 operands, float32 accumulation on the tensor
 * cores, bf16 results:
 *
 *   for b, r < count[b], j < width:
 *     q[b, r, j] = sum_e x[b, r, e] * w_qkv[j, e]
 *     k[b, r, j] = sum_e x[b, r, e] * w_qkv[width + j, e]
 *     v[b, r, j] = sum_e x[b, r, e] * w_qkv[2 width + j, e]
 *
 * x bf16 device [batch, r_max, hidden]; w_qkv bf16 device [3 width, hidden]
 * (each output feature's weights contiguous, as a linear layer stores them);
 * q, k, v bf16 device [batch, r_max, width] each (with width = heads x head_dim
 * they are the [batch, r_max, heads, head_dim] operands of
 * ec_selective_attention).  count int32 device [batch] or NULL (every one of the
 * r_max rows); rows r >= count[b] are left unchanged.  hidden and width are
 * multiples of 64; pointers 16-byte aligned.  Workspace: at least
 * EC_WORKSPACE_ALIGN bytes (the status word), aligned, zeroed once.
 */
ec_status ec_qkv_projection(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                            int32_t hidden, const void *w_qkv, int32_t width, void *q, void *k,
                            void *v, void *workspace, size_t workspace_bytes, ec_stream_t stream);

/* ------------------------------------------------------------------------- */
/* the rest of a pre-norm transformer layer over the recomputed rows          */
/* ------------------------------------------------------------------------- */
/*
 * The models the pages run (LLaDA-8B, Dream-7B) stack pre-norm layers:
 *   a = rms_norm(x, g1);  [q|k|v] = a W_qkv^T;  rope(q, k);  o = attention;
 *   h = x + o W_o^T;  b = rms_norm(h, g2);  y = h + W_down (silu(b W_gate^T) * b W_up^T)
 * and a partial forward ([EC-it] step 2) runs them on the recomputed rows only.
 * These three calls, with ec_qkv_projection and ec_selective_attention, make that
 * layer; each works on rows r < count[b] of [batch, r_max, ...] bf16 tensors and
 * leaves the others unchanged.  Workspace: at least EC_WORKSPACE_ALIGN bytes (the
 * status word), aligned, zeroed once.
 */

/* y = x / sqrt(mean_j x_j^2 + eps) * weight, float32 arithmetic, bf16 out.  x, y
 * [batch, r_max, hidden] (may alias), weight [hidden]; hidden a multiple of 8;
 * count may be NULL (all r_max rows); 16-byte aligned pointers. */
ec_status ec_rms_norm(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                      int32_t hidden, const void *weight, float eps, void *y, void *workspace,
                      size_t workspace_bytes, ec_stream_t stream);

/* Rotary position embedding in place: for row r of sequence b at rotary position
 * p = idx[b*idx_stride + r] (normally the row's sequence position, the recompute
 * set itself; SimSD's prediction slots take their data token's position, see
 * entropy_gated_kv_decode_b300/simsd.py) and every head of q ([batch, r_max, n_heads,
 * head_dim]) and k ([batch, r_max, n_kv_heads, head_dim]), the pairs
 * (x_i, x_{i + head_dim/2}), i < head_dim/2, turn by the angle
 * p * theta^(-2 i / head_dim) (computed in double precision):
 *   x_i' = x_i cos - x_{i+d/2} sin,   x_{i+d/2}' = x_{i+d/2} cos + x_i sin.
 * head_dim even, at most 128; a position outside [0, seq_len) leaves its row
 * unchanged and sets EC_DEV_BAD_INDEX. */
ec_status ec_rope(void *q, void *k, const int32_t *idx, int64_t idx_stride, const int32_t *count,
                  int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_heads,
                  int32_t n_kv_heads, int32_t head_dim, double theta, void *workspace,
                  size_t workspace_bytes, ec_stream_t stream);

/* Linear layer of the recomputed rows on the tensor cores (bf16 operands, float32
 * accumulation, bf16 out), x [batch, r_max, in_features]:
 *   mode 0  y = x W^T,               W [out_features, in_features]
 *   mode 1  y = residual + x W^T     (residual may be y itself)
 *   mode 2  y = silu(x W_g^T) * (x W_u^T), W = [W_g; W_u] [2 out_features, in_features],
 *           silu(z) = z / (1 + e^-z)
 * y and residual [batch, r_max, out_features].  in_features a multiple of 64;
 * out_features a multiple of 64 (mode 2: of 32, at least 64); count may be NULL;
 * 16-byte aligned pointers. */
ec_status ec_linear(const void *x, const int32_t *count, int32_t batch, int32_t r_max,
                    int32_t in_features, const void *w, int32_t out_features, int32_t mode,
                    const void *residual, void *y, void *workspace, size_t workspace_bytes,
                    ec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ENTROPY_GATED_KV_DECODE_EC_H */
