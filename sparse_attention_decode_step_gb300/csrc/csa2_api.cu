// csa2_api.cu -- the C ABI: argument checks, workspace sizing, launches, and
// the per-layer driver (Full / Reindex / Reuse).  Host code only.
#include <atomic>
#include <mutex>

#include "csa2_internal.h"

namespace csa2 {

static std::atomic<uint64_t> g_launches{0};

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int device_sm_count()
{
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

cudaError_t make_tmap_rows_u8(CUtensorMap *map, const void *base, int64_t rows, int row_bytes,
                              int box_rows, int swizzle_bytes)
{
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)row_bytes, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                 : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- attention plan
// Rows of a query are processed in 128-row tiles; a query's tiles are divided
// over `splits` CTAs (one thread-block cluster: at most 16 where the GPU
// schedules clusters of 16, else 8; 13 .. 15 are not used) so that the grid
// fills the SMs in one wave (one CTA per SM: the kernel uses ~220 KB of shared
// memory and all 512 TMEM columns), with as few splits as give the same
// number of tiles per split.
int attn_plan(int nq, int k_max, int n_win)
{
    const int rows = k_max + n_win > 0 ? k_max + n_win : 1;
    const int tiles = (rows + 127) / 128;
    const int sms = device_sm_count();
    const int cap = attn_max_splits();
    int s = sms / (nq > 0 ? nq : 1);
    if (s > tiles) s = tiles;
    if (s > cap) s = cap;                  // the splits of a query merge within one cluster
    if (s > 12 && s < 16) s = 12;
    if (s < 1) s = 1;
    const int tps = (tiles + s - 1) / s;
    s = (tiles + tps - 1) / tps;
    if (s > 12 && s < 16) s = 16;          // (16 splits give at most tps tiles each too)
    return s;
}

// The splits of a query merge on chip (distributed shared memory): the
// attention needs no workspace.
size_t attn_workspace_bytes(int nq, int H, int k_max, int n_win)
{
    (void)nq; (void)H; (void)k_max; (void)n_win;
    return 0;
}

}  // namespace csa2

using namespace csa2;

// ---------------------------------------------------------------- checks
namespace {

inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool al8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

#define CSA2_REQUIRE(cond, code) \
    do {                         \
        if (!(cond)) return (code); \
    } while (0)

csa2_status check_cache(const csa2_cache *c, bool need_keys)
{
    CSA2_REQUIRE(c != nullptr, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(c->codes && c->scales && c->seq_base && c->seq_len, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(c->batch > 0 && c->m >= 1 && c->cap > 0, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(c->cap % 8 == 0 && c->cap < (1LL << 31), CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(c->codes) && al16(c->scales) && al8(c->seq_base) && al4(c->seq_len),
                 CSA2_ERR_ALIGN);
    if (need_keys) {
        CSA2_REQUIRE(c->kidx && c->kscale, CSA2_ERR_INVALID_ARG);
        CSA2_REQUIRE(al16(c->kidx) && al16(c->kscale), CSA2_ERR_ALIGN);
        CSA2_REQUIRE(c->d_idx == 64 || c->d_idx == 128, CSA2_ERR_UNSUPPORTED);
    }
    return CSA2_OK;
}

csa2_status check_queries(const csa2_queries *q)
{
    CSA2_REQUIRE(q != nullptr && q->nq >= 0, CSA2_ERR_INVALID_ARG);
    if (q->nq == 0) return CSA2_OK;
    CSA2_REQUIRE(q->q_seq && q->q_pos, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al4(q->q_seq) && al4(q->q_pos), CSA2_ERR_ALIGN);
    CSA2_REQUIRE(q->group >= 1 && q->nq % q->group == 0, CSA2_ERR_INVALID_ARG);
    return CSA2_OK;
}

csa2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

csa2_status check_index_args(const csa2_cache *cache, const csa2_queries *qs, const float *q_idx,
                             const float *w, int32_t h_idx, const float *scores, int64_t ld,
                             const void *ws)
{
    csa2_status s = check_cache(cache, true);
    if (s != CSA2_OK) return s;
    s = check_queries(qs);
    if (s != CSA2_OK) return s;
    CSA2_REQUIRE(q_idx && w && scores && ws, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(q_idx) && al16(w) && al16(scores) && al16(ws), CSA2_ERR_ALIGN);
    CSA2_REQUIRE(h_idx >= 1 && h_idx <= 16, CSA2_ERR_UNSUPPORTED);
    CSA2_REQUIRE(qs->group * h_idx <= 256, CSA2_ERR_UNSUPPORTED);
    if (qs->group > 1) CSA2_REQUIRE(16 % h_idx == 0, CSA2_ERR_UNSUPPORTED);
    CSA2_REQUIRE(ld > 0 && ld % 4 == 0, CSA2_ERR_INVALID_ARG);
    return CSA2_OK;
}

}  // namespace

extern "C" {

size_t csa2_index_workspace_size(int32_t nq, int32_t group, int32_t h_idx, int32_t d_idx)
{
    if (nq <= 0 || group <= 0 || nq % group) return 0;
    return index_workspace_bytes(nq, group, h_idx, d_idx);
}

size_t csa2_topk_workspace_size(int32_t nq, int64_t max_n)
{
    if (nq <= 0) return 0;
    return topk_workspace_bytes(nq, max_n < 1 ? 1 : max_n);
}

size_t csa2_attn_workspace_size(int32_t nq, int32_t H, int32_t k_max, int32_t n_win)
{
    if (nq <= 0) return 0;
    return attn_workspace_bytes(nq, H, k_max, n_win);
}

csa2_status csa2_quantize_append(const csa2_cache *cache, const float *C, const float *Z,
                                 const float *key, int32_t n_tok, uint32_t *counters,
                                 void *stream)
{
    csa2_status s = check_cache(cache, true);
    if (s != CSA2_OK) return s;
    CSA2_REQUIRE(n_tok > 0 && n_tok % cache->m == 0, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(C && key && (cache->m == 1 || Z), CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(C) && al16(key) && (Z == nullptr || al16(Z)), CSA2_ERR_ALIGN);
    CSA2_REQUIRE(counters == nullptr || al16(counters), CSA2_ERR_ALIGN);
    return cuda_status(launch_append(*cache, C, Z, key, n_tok, counters,
                                     static_cast<cudaStream_t>(stream)));
}

csa2_status csa2_quantize_append_project(const csa2_cache *cache, const float *C,
                                         const float *Z, const uint16_t *w_ik, int32_t n_tok,
                                         uint32_t *counters, void *stream)
{
    csa2_status s = check_cache(cache, true);
    if (s != CSA2_OK) return s;
    CSA2_REQUIRE(n_tok > 0 && n_tok % cache->m == 0, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(C && w_ik && (cache->m == 1 || Z), CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(C) && al16(w_ik) && (Z == nullptr || al16(Z)), CSA2_ERR_ALIGN);
    CSA2_REQUIRE(counters == nullptr || al16(counters), CSA2_ERR_ALIGN);
    return cuda_status(launch_append_project(*cache, C, Z, w_ik, n_tok, counters,
                                             static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The entry points' bodies (shared with csa2_layer_step).
csa2_status index_full_impl(const csa2_cache *cache, const csa2_queries *queries,
                            const float *q_idx, const float *w, int32_t h_idx, int64_t max_n,
                            float *scores, int64_t ld_scores, float *blockmax,
                            int64_t ld_blockmax, int32_t *n_valid, void *workspace,
                            size_t ws_bytes, uint32_t *counters, void *stream)
{
    csa2_status s = check_index_args(cache, queries, q_idx, w, h_idx, scores, ld_scores, workspace);
    if (s != CSA2_OK) return s;
    if (queries->nq == 0) return CSA2_OK;
    CSA2_REQUIRE(max_n >= 1 && ld_scores >= max_n, CSA2_ERR_INVALID_ARG);
    if (blockmax) {
        CSA2_REQUIRE(al16(blockmax), CSA2_ERR_ALIGN);
        CSA2_REQUIRE(ld_blockmax >= (max_n + 7) / 8 && ld_blockmax % 4 == 0, CSA2_ERR_INVALID_ARG);
    }
    CSA2_REQUIRE(n_valid == nullptr || al4(n_valid), CSA2_ERR_ALIGN);
    CSA2_REQUIRE(ws_bytes >= index_workspace_bytes(queries->nq, queries->group, h_idx,
                                                   cache->d_idx),
                 CSA2_ERR_CAPACITY);
    return cuda_status(launch_index(*cache, *queries, q_idx, w, h_idx, max_n, nullptr, nullptr, 0,
                                    scores, ld_scores, blockmax, ld_blockmax, n_valid, workspace,
                                    counters, static_cast<cudaStream_t>(stream)));
}

csa2_status index_reindex_impl(const csa2_cache *cache, const csa2_queries *queries,
                               const float *q_idx, const float *w, int32_t h_idx,
                               const int32_t *pool_blk, const int32_t *pool_n,
                               int32_t pool_blocks, float *scores, int64_t ld_scores,
                               int32_t *n_valid, void *workspace, size_t ws_bytes,
                               uint32_t *counters, void *stream)
{
    csa2_status s = check_index_args(cache, queries, q_idx, w, h_idx, scores, ld_scores, workspace);
    if (s != CSA2_OK) return s;
    if (queries->nq == 0) return CSA2_OK;
    CSA2_REQUIRE(queries->group == 1, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(pool_blk && pool_n && pool_blocks >= 1, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al4(pool_blk) && al4(pool_n), CSA2_ERR_ALIGN);
    CSA2_REQUIRE(ld_scores >= 8LL * pool_blocks, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(n_valid == nullptr || al4(n_valid), CSA2_ERR_ALIGN);
    CSA2_REQUIRE(ws_bytes >= index_workspace_bytes(queries->nq, 1, h_idx, cache->d_idx),
                 CSA2_ERR_CAPACITY);
    return cuda_status(launch_index(*cache, *queries, q_idx, w, h_idx, 8LL * pool_blocks, pool_blk,
                                    pool_n, pool_blocks, scores, ld_scores, nullptr, 0, n_valid,
                                    workspace, counters, static_cast<cudaStream_t>(stream)));
}

csa2_status topk_impl(const float *scores, int64_t ld_scores, const int32_t *n_valid,
                      const int32_t *pool_blk, int32_t pool_blocks, int32_t nq, int64_t max_n,
                      int32_t k, int32_t *idx_out, int64_t ld_idx, int32_t *cnt_out,
                      void *workspace, size_t ws_bytes, void *stream)
{
    CSA2_REQUIRE(nq >= 0, CSA2_ERR_INVALID_ARG);
    if (nq == 0) return CSA2_OK;
    CSA2_REQUIRE(scores && n_valid && idx_out && cnt_out && workspace, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(scores) && al4(n_valid) && al4(idx_out) && al4(cnt_out) &&
                     al16(workspace),
                 CSA2_ERR_ALIGN);
    CSA2_REQUIRE(k >= 1 && max_n >= 1 && ld_scores >= max_n && ld_scores % 4 == 0 && ld_idx >= k,
                 CSA2_ERR_INVALID_ARG);
    if (pool_blk) {
        CSA2_REQUIRE(al4(pool_blk), CSA2_ERR_ALIGN);
        CSA2_REQUIRE(pool_blocks >= 1 && max_n <= 8LL * pool_blocks, CSA2_ERR_INVALID_ARG);
    }
    CSA2_REQUIRE(max_n < (1LL << 31), CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(ws_bytes >= topk_workspace_bytes(nq, max_n), CSA2_ERR_CAPACITY);
    return cuda_status(launch_topk(scores, ld_scores, n_valid, 0, pool_blk, pool_blocks, nq, max_n,
                                   k, idx_out, ld_idx, cnt_out, workspace,
                                   static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

csa2_status csa2_index_full(const csa2_cache *cache, const csa2_queries *queries,
                            const float *q_idx, const float *w, int32_t h_idx, int64_t max_n,
                            float *scores, int64_t ld_scores, float *blockmax,
                            int64_t ld_blockmax, int32_t *n_valid, void *workspace,
                            size_t ws_bytes, uint32_t *counters, void *stream)
{
    return index_full_impl(cache, queries, q_idx, w, h_idx, max_n, scores, ld_scores, blockmax,
                           ld_blockmax, n_valid, workspace, ws_bytes, counters, stream);
}

csa2_status csa2_index_reindex(const csa2_cache *cache, const csa2_queries *queries,
                               const float *q_idx, const float *w, int32_t h_idx,
                               const int32_t *pool_blk, const int32_t *pool_n,
                               int32_t pool_blocks, float *scores, int64_t ld_scores,
                               int32_t *n_valid, void *workspace, size_t ws_bytes,
                               uint32_t *counters, void *stream)
{
    return index_reindex_impl(cache, queries, q_idx, w, h_idx, pool_blk, pool_n, pool_blocks,
                              scores, ld_scores, n_valid, workspace, ws_bytes, counters, stream);
}

csa2_status csa2_topk(const float *scores, int64_t ld_scores, const int32_t *n_valid,
                      const int32_t *pool_blk, int32_t pool_blocks, int32_t nq, int64_t max_n,
                      int32_t k, int32_t *idx_out, int64_t ld_idx, int32_t *cnt_out,
                      void *workspace, size_t ws_bytes, void *stream)
{
    return topk_impl(scores, ld_scores, n_valid, pool_blk, pool_blocks, nq, max_n, k, idx_out,
                     ld_idx, cnt_out, workspace, ws_bytes, stream);
}

csa2_status csa2_pool_select(const float *blockmax, int64_t ld_blockmax, const int32_t *n_valid,
                             int32_t nq, int64_t max_n, int32_t pool_blocks, int32_t *pool_blk,
                             int32_t *pool_n, void *workspace, size_t ws_bytes, void *stream)
{
    CSA2_REQUIRE(nq >= 0, CSA2_ERR_INVALID_ARG);
    if (nq == 0) return CSA2_OK;
    CSA2_REQUIRE(blockmax && n_valid && pool_blk && pool_n && workspace, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(blockmax) && al4(n_valid) && al4(pool_blk) && al4(pool_n) &&
                     al16(workspace),
                 CSA2_ERR_ALIGN);
    CSA2_REQUIRE(max_n >= 1 && pool_blocks >= 1, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(ld_blockmax >= (max_n + 7) / 8 && ld_blockmax % 4 == 0, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(ws_bytes >= topk_workspace_bytes(nq, (max_n + 7) / 8), CSA2_ERR_CAPACITY);
    return cuda_status(launch_pool(blockmax, ld_blockmax, n_valid, nq, max_n, pool_blocks,
                                   pool_blk, pool_n, workspace,
                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// early: the kernel launched just before on the stream (this library's top-k
// inside csa2_layer_step) writes none of q, win or the cache, so the attention
// may load q before its programmatic dependent-launch wait.
csa2_status sparse_attn_impl(const csa2_cache *cache, const csa2_queries *queries,
                             const int32_t *idx, int64_t ld_idx, const int32_t *cnt,
                             int32_t k_max, const uint16_t *q, int32_t H, const uint16_t *win,
                             int32_t wcap, const int32_t *win_start, int32_t n_win,
                             float sm_scale, float *out, float *lse, void *workspace,
                             size_t ws_bytes, uint32_t *counters, int early, void *stream)
{
    csa2_status s = check_cache(cache, false);
    if (s != CSA2_OK) return s;
    s = check_queries(queries);
    if (s != CSA2_OK) return s;
    if (queries->nq == 0) return CSA2_OK;
    CSA2_REQUIRE(k_max >= 0 && n_win >= 0 && k_max + n_win >= 1, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(H >= 1 && H <= 64, CSA2_ERR_UNSUPPORTED);
    CSA2_REQUIRE(q && out, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(k_max == 0 || (idx && cnt && ld_idx >= k_max), CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(n_win == 0 || (win && wcap >= n_win), CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(q) && al16(out) && (idx == nullptr || al4(idx)) &&
                     (cnt == nullptr || al4(cnt)) && (win == nullptr || al16(win)) &&
                     (win_start == nullptr || al4(win_start)) && (lse == nullptr || al4(lse)),
                 CSA2_ERR_ALIGN);
    CSA2_REQUIRE(ws_bytes >= attn_workspace_bytes(queries->nq, H, k_max, n_win), CSA2_ERR_CAPACITY);
    AttnParams p{};
    p.codes = cache->codes;
    p.scales = cache->scales;
    p.seq_base = cache->seq_base;
    p.seq_len = cache->seq_len;
    p.m = cache->m;
    p.batch = cache->batch;
    p.q_seq = queries->q_seq;
    p.q_pos = queries->q_pos;
    p.nq = queries->nq;
    p.idx = idx;
    p.ld_idx = ld_idx;
    p.cnt = cnt;
    p.k_max = k_max;
    p.q = q;
    p.H = H;
    p.win = (n_win > 0) ? win : nullptr;
    p.wcap = wcap > 0 ? wcap : 1;
    p.win_start = win_start;
    p.n_win = n_win;
    p.sm_scale = sm_scale;
    p.out = out;
    p.lse = lse;
    p.splits = attn_plan(p.nq, k_max, n_win);
    (void)workspace;
    p.counters = counters;
    p.early = early;
    return cuda_status(launch_attn_tc(p, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

csa2_status csa2_sparse_attn(const csa2_cache *cache, const csa2_queries *queries,
                             const int32_t *idx, int64_t ld_idx, const int32_t *cnt,
                             int32_t k_max, const uint16_t *q, int32_t H, const uint16_t *win,
                             int32_t wcap, const int32_t *win_start, int32_t n_win,
                             float sm_scale, float *out, float *lse, void *workspace,
                             size_t ws_bytes, uint32_t *counters, void *stream)
{
    return sparse_attn_impl(cache, queries, idx, ld_idx, cnt, k_max, q, H, win, wcap, win_start,
                            n_win, sm_scale, out, lse, workspace, ws_bytes, counters, 0, stream);
}

// ---------------------------------------------------------------- layer driver
namespace {

struct LayerPlan {
    int64_t max_n, ld, ld_bm;
    int chunk;                    // queries per indexer/top-k chunk
    size_t off_scores, off_bm, off_nv, off_idx_ws, off_topk_ws, off_attn_ws, total;
};

bool plan_layer(const csa2_layer_args *a, LayerPlan *pl)
{
    const csa2_queries *qs = a->queries;
    const int nq = qs->nq;
    const int group = qs->group;
    pl->max_n = (a->mode == CSA2_REINDEX) ? 8LL * a->pool_blocks : a->max_n;
    if (pl->max_n < 1) pl->max_n = 1;
    pl->ld = align_up((size_t)pl->max_n, 4);
    pl->ld_bm = align_up((size_t)(pl->max_n + 7) / 8, 4);
    // keep one chunk's score rows near 256 MB
    int64_t chunk = (64LL << 20) / pl->ld;
    if (chunk < group) chunk = group;
    chunk = chunk / group * group;
    if (chunk > nq) chunk = nq;
    if (chunk < 1) chunk = 1;
    pl->chunk = (int)chunk;
    size_t o = 0;
    if (a->mode != CSA2_REUSE) {
        pl->off_scores = o;
        o += align_up((size_t)chunk * pl->ld * 4, 256);
        pl->off_bm = o;
        if (a->mode == CSA2_FULL && a->build_pool) o += align_up((size_t)chunk * pl->ld_bm * 4, 256);
        pl->off_nv = o;
        o += align_up((size_t)nq * 4, 256);
        pl->off_idx_ws = o;
        o += align_up(index_workspace_bytes((int)chunk, a->mode == CSA2_FULL ? group : 1, a->h_idx,
                                            a->cache->d_idx),
                      256);
        pl->off_topk_ws = o;
        size_t tk = topk_workspace_bytes((int)chunk, pl->max_n);
        if (a->mode == CSA2_FULL && a->build_pool) {
            size_t tp = topk_workspace_bytes((int)chunk, (pl->max_n + 7) / 8);
            if (tp > tk) tk = tp;
        }
        o += align_up(tk, 256);
    }
    pl->off_attn_ws = o;
    o += align_up(attn_workspace_bytes(nq, a->H, a->k, a->n_win), 256);
    pl->total = o;
    return true;
}

}  // namespace

size_t csa2_layer_workspace_size(const csa2_layer_args *a)
{
    if (a == nullptr || a->queries == nullptr || a->cache == nullptr || a->queries->nq <= 0)
        return 0;
    LayerPlan pl;
    plan_layer(a, &pl);
    return pl.total;
}

csa2_status csa2_layer_step(const csa2_layer_args *a, void *stream)
{
    CSA2_REQUIRE(a != nullptr, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(a->mode == CSA2_FULL || a->mode == CSA2_REINDEX || a->mode == CSA2_REUSE,
                 CSA2_ERR_INVALID_ARG);
    csa2_status s = check_cache(a->cache, a->mode != CSA2_REUSE);
    if (s != CSA2_OK) return s;
    s = check_queries(a->queries);
    if (s != CSA2_OK) return s;
    const int nq = a->queries->nq;
    if (nq == 0) return CSA2_OK;
    CSA2_REQUIRE(a->idx && a->cnt && a->k >= 1 && a->workspace, CSA2_ERR_INVALID_ARG);
    CSA2_REQUIRE(al16(a->workspace) && al4(a->idx) && al4(a->cnt), CSA2_ERR_ALIGN);
    if (a->mode == CSA2_REINDEX || (a->mode == CSA2_FULL && a->build_pool))
        CSA2_REQUIRE(a->pool_blk && a->pool_n && a->pool_blocks >= 1, CSA2_ERR_INVALID_ARG);
    if (a->mode == CSA2_REINDEX) CSA2_REQUIRE(a->queries->group == 1, CSA2_ERR_INVALID_ARG);
    LayerPlan pl;
    plan_layer(a, &pl);
    CSA2_REQUIRE(a->ws_bytes >= pl.total, CSA2_ERR_CAPACITY);
    uint8_t *ws = static_cast<uint8_t *>(a->workspace);

    if (a->mode != CSA2_REUSE) {
        float *scores = reinterpret_cast<float *>(ws + pl.off_scores);
        float *bm = reinterpret_cast<float *>(ws + pl.off_bm);
        int32_t *nv = reinterpret_cast<int32_t *>(ws + pl.off_nv);
        void *iws = ws + pl.off_idx_ws;
        void *tws = ws + pl.off_topk_ws;
        const size_t iws_bytes = pl.off_topk_ws - pl.off_idx_ws;
        const size_t tws_bytes = pl.off_attn_ws - pl.off_topk_ws;
        for (int q0 = 0; q0 < nq; q0 += pl.chunk) {
            const int nc = (nq - q0 < pl.chunk) ? nq - q0 : pl.chunk;
            csa2_queries sub = *a->queries;
            sub.q_seq = a->queries->q_seq + q0;
            sub.q_pos = a->queries->q_pos + q0;
            sub.nq = nc;
            const float *qi = a->q_idx + (int64_t)q0 * a->h_idx * a->cache->d_idx;
            const float *wi = a->w + (int64_t)q0 * a->h_idx;
            int32_t *pblk = a->pool_blk ? a->pool_blk + (int64_t)q0 * a->pool_blocks : nullptr;
            int32_t *pn = a->pool_n ? a->pool_n + q0 : nullptr;
            if (a->mode == CSA2_FULL) {
                s = index_full_impl(a->cache, &sub, qi, wi, a->h_idx, pl.max_n, scores, pl.ld,
                                    a->build_pool ? bm : nullptr, pl.ld_bm, nv + q0, iws,
                                    iws_bytes, a->counters, stream);
            } else {
                s = index_reindex_impl(a->cache, &sub, qi, wi, a->h_idx, pblk, pn, a->pool_blocks,
                                       scores, pl.ld, nv + q0, iws, iws_bytes, a->counters,
                                       stream);
            }
            if (s != CSA2_OK) return s;
            s = topk_impl(scores, pl.ld, nv + q0, a->mode == CSA2_REINDEX ? pblk : nullptr,
                          a->pool_blocks, nc, pl.max_n, a->k, a->idx + (int64_t)q0 * a->k, a->k,
                          a->cnt + q0, tws, tws_bytes, stream);
            if (s != CSA2_OK) return s;
            if (a->mode == CSA2_FULL && a->build_pool) {
                s = csa2_pool_select(bm, pl.ld_bm, nv + q0, nc, pl.max_n, a->pool_blocks, pblk, pn,
                                     tws, tws_bytes, stream);
                if (s != CSA2_OK) return s;
            }
        }
    }
    // after this call's own top-k, the attention may load its queries early
    return sparse_attn_impl(a->cache, a->queries, a->idx, a->k, a->cnt, a->k, a->q, a->H, a->win,
                            a->wcap, a->win_start, a->n_win, a->sm_scale, a->out, a->lse,
                            ws + pl.off_attn_ws, pl.total - pl.off_attn_ws, a->counters,
                            a->mode != CSA2_REUSE ? 1 : 0, stream);
}

const char *csa2_status_string(csa2_status s)
{
    switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_ALIGN: return "pointer not 16-byte aligned";
    case CSA2_ERR_CAPACITY: return "workspace or output too small";
    case CSA2_ERR_UNSUPPORTED: return "shape not supported by the compiled kernels";
    case CSA2_ERR_CUDA: return "CUDA launch or driver error";
    }
    return "unknown status";
}

uint64_t csa2_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
