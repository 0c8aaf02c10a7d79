/*
 * csa2.h -- C ABI of the CSA2 global-attention step on one GPU (sm_103a).
 *
 * The step, per query batch (one decode token per sequence, or a prefill
 * chunk of causal queries):
 *   1. indexer scoring of each query against the compressed indexer keys,
 *      over the whole visible context (Full mode) or over the hierarchical
 *      candidate pool only (Reindex mode);
 *   2. per-query top-k selection;
 *   3. a gather of the selected 512-wide main-KV latents from an FP4 cache
 *      (E2M1 values, one E4M3 scale per 16 channels), dequantised and
 *      concatenated with the sliding-window KV;
 *   4. multi-head softmax attention over that set.
 * Reuse mode skips 1-2 and takes the index list of an earlier layer.
 *
 * Sources (page title and section):
 *   [Notes]     "DeepSeek-V4.1-Flash KV-Cache Compression" reading notes:
 *               section 2 (CSA2 modes, block compression by m), section 3
 *               (hierarchical sparse indexer, 2,048 blocks x 8 positions),
 *               section 4 (FP4 main KV, E4M3 scale per 16 channels, range
 *               448 x 6 = 2688), section 5 (window [max(s, i - n_win + 1), i]).
 *   [Deep read] "DeepSeek-V4.1-Flash: reading a model through its three memory
 *               costs", section 03 (what each mode computes and reuses).
 *   [Thread]    threadnavigator notes, item 4 (select main KV, concatenate with
 *               the windowed KV, then attend).
 *
 * Readings where the pages are silent (the test oracle uses the same ones):
 *   score(q, j) = sum_h w_h * ReLU(q_h . k_j), one indexer key per entry shared
 *   by all indexer heads; FP8 = E4M3 with a power-of-two scale per vector; FP4
 *   scale = smallest E4M3 s with 6 s >= amax, codes round-to-nearest-even;
 *   top-k ties go to the lower position and the list is ascending; attention
 *   uses the dequantised latent as key and value, logits sm_scale * q . v.
 *
 * Conventions for every entry point:
 *   - Every pointer is a DEVICE pointer unless stated otherwise, owned by the
 *     caller; the library never allocates or frees memory.  Temporary space
 *     comes from a caller-provided workspace whose size the *_workspace_size
 *     functions give.
 *   - Bulk arrays (cache rows, key scales, queries, scores, block maxima,
 *     window KV, outputs, workspace) must be 16-byte aligned; small index
 *     arrays (seq_base, seq_len, q_seq, q_pos, idx, cnt, n_valid, pool_blk,
 *     pool_n, win_start, lse) need only their natural alignment.  A violation
 *     returns CSA2_ERR_ALIGN.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = default).
 *     The returned status covers host-side argument checks and the launch
 *     (cudaGetLastError); it does not wait for the GPU.
 *   - Problems only the GPU can see (a query position past the cached
 *     entries, an index out of range, a full sequence, FP4 saturation, a
 *     pipeline wait that exceeded its limit) are counted in the optional
 *     `counters` array (uint32 [CSA2_NUM_COUNTERS], device), never trapped.
 *     An offending row or query is skipped (its scores/outputs are left
 *     unspecified); the rest of the batch is computed normally.
 *   - A pointer that a mode must not touch may be NULL.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CSA2_OK = 0,
    CSA2_ERR_INVALID_ARG = -1,  /* a size, count or NULL pointer out of contract */
    CSA2_ERR_ALIGN = -2,        /* an array pointer not 16-byte aligned */
    CSA2_ERR_CAPACITY = -3,     /* workspace or output too small */
    CSA2_ERR_UNSUPPORTED = -4,  /* shape outside the compiled kernels (e.g. d_idx) */
    CSA2_ERR_CUDA = -5          /* a CUDA launch or driver call failed */
} csa2_status;

typedef enum { CSA2_FULL = 0, CSA2_REINDEX = 1, CSA2_REUSE = 2 } csa2_mode;

/* Device counter slots (uint32 each). */
enum {
    CSA2_CNT_FP4_SATURATED = 0,   /* 16-channel groups whose amax exceeded 2688 */
    CSA2_CNT_CAPACITY = 1,        /* append batches refused: sequence full */
    CSA2_CNT_BAD_INPUT = 2,       /* query past the cache, index out of range, mixed group */
    CSA2_CNT_TIMEOUT = 3,         /* a pipeline wait exceeded its limit (kernel returned) */
    CSA2_NUM_COUNTERS = 4
};

#define CSA2_D 512              /* latent width [Notes] section 4 */
#define CSA2_CODE_BYTES 256     /* E2M1 codes per entry: channel 2i in the low nibble of byte i */
#define CSA2_SCALE_BYTES 32     /* E4M3 scales per entry: byte g covers channels 16g..16g+15 */
#define CSA2_POOL_BLOCK 8       /* positions per candidate-pool block [Notes] section 3 */

/* One FP4 main-KV cache with its FP8 indexer keys (the cache a Full layer
 * owns; Reindex and Reuse layers read it).  Sequence b owns the rows
 * seq_base[b] .. seq_base[b+1]-1; its entry j (0-based, in compressed units)
 * is row seq_base[b] + j.  seq_len[b] counts the entries written so far and
 * is advanced on the device by csa2_quantize_append. */
typedef struct {
    uint8_t *codes;            /* [cap][256] E2M1 codes */
    uint8_t *scales;           /* [cap][32]  E4M3 scales */
    uint8_t *kidx;             /* [cap][d_idx] E4M3 indexer keys */
    float *kscale;             /* [cap] power-of-two key scales */
    const int64_t *seq_base;   /* [batch + 1], seq_base[batch] <= cap */
    int32_t *seq_len;          /* [batch] entries held */
    int64_t cap;               /* rows allocated (host value) */
    int32_t batch;             /* sequences */
    int32_t d_idx;             /* indexer key width: 64 or 128 */
    int32_t m;                 /* block-compression factor (entries = tokens / m) */
} csa2_cache;

/* A query batch.  Query i belongs to sequence q_seq[i] and sits at token
 * position q_pos[i] (0-based); it sees the entries j < floor((q_pos+1)/m).
 * group > 1 declares that each run of `group` consecutive queries shares one
 * sequence (a prefill chunk); the indexer then scores them together. */
typedef struct {
    const int32_t *q_seq;      /* [nq] */
    const int32_t *q_pos;      /* [nq] */
    int32_t nq;
    int32_t group;             /* 1 (decode) or a divisor of nq with group * h_idx <= 256 */
} csa2_queries;

/* ---- 1. append ------------------------------------------------------------
 * Compress n_tok new tokens per sequence into n_tok/m entries and store them:
 * entry e of sequence b = sum over its m tokens i of softmax_i(Z[b][i][c]) *
 * C[b][i][c] per channel c ([Notes] sections 1-2: disjoint blocks, no
 * positional term; m = 1 stores C itself), then FP4-encode it and FP8-encode
 * its indexer key.  Rows seq_base[b] + seq_len[b] + e are written and
 * seq_len[b] grows by n_tok/m.  A sequence without room is left unchanged and
 * counted in CSA2_CNT_CAPACITY.
 *   C   [batch][n_tok][512] fp32;  Z same shape, NULL when m == 1;
 *   key [batch][n_tok/m][d_idx] fp32 (the indexer-key projection of each entry).
 * n_tok must be a positive multiple of m. */
csa2_status csa2_quantize_append(const csa2_cache *cache, const float *C, const float *Z,
                                 const float *key, int32_t n_tok, uint32_t *counters,
                                 void *stream);

/* The same append with the indexer key projected from the stored entry
 * instead of passed in ([Notes] section 1: the indexer key is a linear
 * projection of the main KV; this library's reading: of the dequantised FP4
 * entry, so that every key can be rebuilt from the cache alone):
 *   key[b][e][d] = sum_c value(entry)[c] * w_ik[c][d], then FP8-encoded as in
 *   csa2_quantize_append; the sum runs in fp32 over c = 0..511 in order.
 *   w_ik [512][d_idx] bf16 (bit patterns), row c = latent channel c, device
 *   memory, 16-byte aligned, owned by the caller and only read.
 * One launch when n_tok / m <= 8 (decode: one CTA per sequence appends its
 * entries and advances seq_len itself), two otherwise (the appends, then the
 * sequence-length update); each CTA stages w_ik (64 or 128 KB) in shared
 * memory.  Same status and counters as csa2_quantize_append.  If a CTA's wait
 * for its copy of w_ik runs past its time limit (CSA2_CNT_TIMEOUT), the keys
 * of its remaining entries are not written: in the one-launch form that
 * sequence's seq_len is not advanced; in the two-launch form the entries are
 * committed all the same and their keys are unspecified, so a cache that saw
 * CSA2_CNT_TIMEOUT from this call must not be scored. */
csa2_status csa2_quantize_append_project(const csa2_cache *cache, const float *C,
                                         const float *Z, const uint16_t *w_ik, int32_t n_tok,
                                         uint32_t *counters, void *stream);

/* ---- 2. Full-mode indexer -------------------------------------------------
 * scores[i][j] = sum_h w[i][h] * ReLU(q_h . k_j) for the visible entries
 * j < N_i = floor((q_pos[i]+1)/m) of query i ([Notes] section 2: a Full
 * layer scores every entry the query can see), with q_h FP8-quantised per head
 * by the library.  Entries j >= N_i are not written.  If blockmax is not NULL it also
 * receives, for each aligned 8-entry block b holding a visible entry, the max
 * score over the block's visible entries ([Notes] section 3, step 1).
 * n_valid[i] (nullable) receives N_i.
 *   q_idx [nq][h_idx][d_idx] fp32, w [nq][h_idx] fp32, h_idx <= 16;
 *   scores [nq][ld_scores] fp32, ld_scores >= max_n;
 *   blockmax [nq][ld_blockmax], ld_blockmax >= ceil(max_n / 8);
 *   max_n: host bound on every N_i (queries beyond it are counted as bad). */
csa2_status csa2_index_full(const csa2_cache *cache, const csa2_queries *queries,
                            const float *q_idx, const float *w, int32_t h_idx, int64_t max_n,
                            float *scores, int64_t ld_scores, float *blockmax,
                            int64_t ld_blockmax, int32_t *n_valid, void *workspace,
                            size_t ws_bytes, uint32_t *counters, void *stream);

/* ---- 3. Reindex-mode indexer ----------------------------------------------
 * Same score as the Full indexer, at the pool positions only ([Notes] section
 * 3, step 3; [Deep read] section 03, Reindex computes its own indexer Q):
 * candidate p < pool_n[i] is entry 8 * pool_blk[i][p / 8] + p % 8.
 *   pool_blk [nq][pool_blocks] ascending block ids, pool_n [nq];
 *   scores [nq][ld_scores] in pool order, ld_scores >= 8 * pool_blocks.
 * group must be 1 (one pool per query). */
csa2_status csa2_index_reindex(const csa2_cache *cache, const csa2_queries *queries,
                               const float *q_idx, const float *w, int32_t h_idx,
                               const int32_t *pool_blk, const int32_t *pool_n,
                               int32_t pool_blocks, float *scores, int64_t ld_scores,
                               int32_t *n_valid, void *workspace, size_t ws_bytes,
                               uint32_t *counters, void *stream);

/* ---- 4. top-k ------------------------------------------------------------
 * For each query i, the positions of the min(k, n_valid[i]) largest of
 * scores[i][0 .. n_valid[i]), ties to the lower position, written ascending
 * to idx_out[i][0 .. cnt_out[i]).  If pool_blk is not NULL, candidate p stands
 * for position 8 * pool_blk[i][p / 8] + p % 8 (a Reindex score row).  -0.0
 * equals +0.0; NaN scores are outside the contract.
 *   scores [nq][ld_scores]; n_valid [nq] (<= max_n); idx_out [nq][ld_idx]. */
csa2_status csa2_topk(const float *scores, int64_t ld_scores, const int32_t *n_valid,
                      const int32_t *pool_blk, int32_t pool_blocks, int32_t nq, int64_t max_n,
                      int32_t k, int32_t *idx_out, int64_t ld_idx, int32_t *cnt_out,
                      void *workspace, size_t ws_bytes, void *stream);

/* ---- 4b. top-k that allocates nothing ---------------------------------------
 * The same selection as csa2_topk, for callers that cannot get device memory
 * for a workspace: for instance a plugin running inside a host program that
 * owns every device allocation, or a serving loop that forbids allocating once
 * it has started.  The pages have no counterpart to this call; it is a
 * convenience of this library.
 *
 * Scratch: a fixed 4 MiB array of device memory inside the library, held by
 * every GPU that loads it until the process exits (its size is
 * csa2_topk_noalloc_max_scratch()).  A problem whose
 * csa2_topk_workspace_size(nq, max_n) exceeds it is refused with
 * CSA2_ERR_CAPACITY and nothing is launched.  The call never allocates or
 * frees memory.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress; make that first call
 * before any stream capture.  A failed lookup returns CSA2_ERR_CUDA.
 * Sharing: every call on a device uses the same array, which keeps what the
 * last call left in it (each call clears what it needs before use).  Calls
 * whose kernels overlap on the GPU (different streams with no ordering) race
 * on the array and give undefined results: order them on one stream.
 * Arguments, outputs and errors are otherwise those of csa2_topk. */
csa2_status csa2_topk_noalloc(const float *scores, int64_t ld_scores, const int32_t *n_valid,
                              const int32_t *pool_blk, int32_t pool_blocks, int32_t nq,
                              int64_t max_n, int32_t k, int32_t *idx_out, int64_t ld_idx,
                              int32_t *cnt_out, void *stream);
size_t csa2_topk_noalloc_max_scratch(void);

/* ---- 5. candidate pool ----------------------------------------------------
 * From a Full layer's block maxima: the pool_blocks blocks with the largest
 * block max among the ceil(N_i / 8) visible blocks (ties to the lower block),
 * ascending in pool_blk[i], and pool_n[i] = the visible positions they hold
 * ([Notes] section 3: 2,048 blocks x 8 = 16,384 positions).
 *   blockmax [nq][ld_blockmax]; n_valid [nq] = N_i (entries, from the indexer). */
csa2_status csa2_pool_select(const float *blockmax, int64_t ld_blockmax, const int32_t *n_valid,
                             int32_t nq, int64_t max_n, int32_t pool_blocks, int32_t *pool_blk,
                             int32_t *pool_n, void *workspace, size_t ws_bytes, void *stream);

/* ---- 6. sparse attention --------------------------------------------------
 * For query i of sequence b at position t: the row set is the dequantised
 * entries idx[i][0 .. cnt[i]) followed by the window rows of the positions
 * max(s_b, t - n_win + 1, 0) .. t, where s_b = win_start[b] (0 if NULL) and
 * position p lives at win[b][p mod wcap] ([Notes] section 5; [Thread] item 4:
 * concatenation, no de-duplication).  For every head h:
 *   out[i][h] = sum_r softmax_r(sm_scale * q[i][h] . v_r) v_r,
 *   lse[i][h] = log sum_r exp(sm_scale * q[i][h] . v_r)   (nullable).
 *   idx [nq][ld_idx] entry numbers < N_i (others are skipped and counted);
 *   q [nq][H][512] bf16 bits; 1 <= H <= 64;
 *   win [batch][wcap][512] bf16 bits (NULL allowed when n_win == 0);
 *   out [nq][H][512] fp32; k_max >= every cnt[i].
 * Arithmetic: the tensor-core products take f16 operands.  The dequantised
 * FP4 values are exact in f16; q and the window rows are converted from bf16
 * to f16, which is exact for magnitudes in [2^-14, 65504] (smaller ones become
 * f16 subnormals with an absolute error below 2^-25; 65504 and above are
 * outside the contract); the softmax weights P are stored as f16 (at most 256
 * before normalisation, relative error 2^-11).  Logits, the softmax and every
 * sum are fp32.
 * The attention needs no workspace (csa2_attn_workspace_size() is 0; the
 * argument may be NULL): a query's row tiles are divided over at most 16 CTAs
 * of one thread-block cluster (8 where the GPU does not schedule clusters of
 * 16), which merge on chip. */
csa2_status csa2_sparse_attn(const csa2_cache *cache, const csa2_queries *queries,
                             const int32_t *idx, int64_t ld_idx, const int32_t *cnt,
                             int32_t k_max, const uint16_t *q, int32_t H, const uint16_t *win,
                             int32_t wcap, const int32_t *win_start, int32_t n_win,
                             float sm_scale, float *out, float *lse, void *workspace,
                             size_t ws_bytes, uint32_t *counters, void *stream);

/* ---- 7. one layer ---------------------------------------------------------
 * Full:    index_full (+ block max and pool when build_pool) -> top-k -> attention.
 * Reindex: index_reindex over pool_blk/pool_n -> top-k -> attention.
 * Reuse:   attention with idx/cnt as given (kidx, q_idx, w, pool untouched).
 * ([Notes] section 2; [Deep read] section 03 mode table.) */
typedef struct {
    csa2_mode mode;
    const csa2_cache *cache;
    const csa2_queries *queries;
    /* indexer (Full, Reindex) */
    const float *q_idx;        /* [nq][h_idx][d_idx] */
    const float *w;            /* [nq][h_idx] */
    int32_t h_idx;
    int64_t max_n;             /* bound on visible entries of any query */
    int32_t k;                 /* top-k */
    int32_t build_pool;        /* Full only: also produce pool_blk/pool_n */
    int32_t pool_blocks;       /* 2048 in the pages */
    int32_t *pool_blk;         /* [nq][pool_blocks]: output (Full+pool), input (Reindex) */
    int32_t *pool_n;           /* [nq] */
    /* selection: output of Full/Reindex, input of Reuse */
    int32_t *idx;              /* [nq][k] */
    int32_t *cnt;              /* [nq] */
    /* attention */
    const uint16_t *q;         /* [nq][H][512] bf16 */
    int32_t H;
    const uint16_t *win;       /* [batch][wcap][512] bf16 */
    int32_t wcap;
    const int32_t *win_start;  /* [batch] or NULL */
    int32_t n_win;
    float sm_scale;
    float *out;                /* [nq][H][512] */
    float *lse;                /* [nq][H] or NULL */
    void *workspace;
    size_t ws_bytes;
    uint32_t *counters;        /* [CSA2_NUM_COUNTERS] or NULL */
} csa2_layer_args;

csa2_status csa2_layer_step(const csa2_layer_args *args, void *stream);

/* ---- workspace sizes (host-only, no GPU work) ------------------------------ */
size_t csa2_index_workspace_size(int32_t nq, int32_t group, int32_t h_idx, int32_t d_idx);
size_t csa2_topk_workspace_size(int32_t nq, int64_t max_n);
size_t csa2_attn_workspace_size(int32_t nq, int32_t H, int32_t k_max, int32_t n_win);
size_t csa2_layer_workspace_size(const csa2_layer_args *args);

/* ---- misc ------------------------------------------------------------------ */
const char *csa2_status_string(csa2_status s);
/* Kernels this library has launched since it was loaded (host counter). */
uint64_t csa2_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
