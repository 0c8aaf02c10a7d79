// csa2_internal.h -- declarations shared by the library's translation units
// (launchers, parameter blocks, host utilities).  Not part of the C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Host-side count of kernel launches (csa2_launch_count).
void note_launch(int n = 1);

// Launch with programmatic stream serialization (see pdl_wait in
// csa2_device.cuh) and, if cluster_x > 0, a runtime cluster shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, unsigned cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    unsigned n = 0;
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 0) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = cluster_x;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    note_launch();
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Number of SMs of the current device (cached per device).
int device_sm_count();

// 2-D tensor map over a row-major uint8 array [rows][row_bytes] with a box of
// [box_rows][row_bytes] and the given swizzle width (64 or 128 bytes).
cudaError_t make_tmap_rows_u8(CUtensorMap *map, const void *base, int64_t rows, int row_bytes,
                              int box_rows, int swizzle_bytes);

// ---- append
cudaError_t launch_append(const csa2_cache &c, const float *C, const float *Z, const float *key,
                          int n_tok, uint32_t *counters, cudaStream_t st);
cudaError_t launch_append_project(const csa2_cache &c, const float *C, const float *Z,
                                  const uint16_t *w_ik, int n_tok, uint32_t *counters,
                                  cudaStream_t st);

// ---- indexer
size_t index_workspace_bytes(int nq, int group, int h_idx, int d_idx);
cudaError_t launch_index(const csa2_cache &c, const csa2_queries &qs, const float *q_idx,
                         const float *w, int h_idx, int64_t max_n, const int32_t *pool_blk,
                         const int32_t *pool_n, int pool_blocks, float *scores, int64_t ld,
                         float *blockmax, int64_t ld_bm, int32_t *n_valid, void *ws,
                         uint32_t *counters, cudaStream_t st);

// ---- top-k and pool
size_t topk_workspace_bytes(int nq, int64_t max_n);
cudaError_t launch_topk(const float *scores, int64_t ld, const int32_t *n_valid, int n_div8,
                        const int32_t *pool_blk, int pool_blocks, int nq, int64_t max_n, int k,
                        int32_t *idx_out, int64_t ld_idx, int32_t *cnt_out, void *ws,
                        cudaStream_t st);
cudaError_t launch_pool(const float *blockmax, int64_t ld_bm, const int32_t *n_valid, int nq,
                        int64_t max_n, int pool_blocks, int32_t *pool_blk, int32_t *pool_n,
                        void *ws, cudaStream_t st);

// ---- attention
struct AttnParams {
    const uint8_t *codes, *scales;
    const int64_t *seq_base;
    const int32_t *seq_len;
    int m, batch;
    const int32_t *q_seq, *q_pos;
    int nq;
    const int32_t *idx;
    int64_t ld_idx;
    const int32_t *cnt;
    int k_max;
    const uint16_t *q;
    int H;
    const uint16_t *win;
    int wcap;
    const int32_t *win_start;
    int n_win;
    float sm_scale;
    float *out, *lse;
    int splits;         // CTAs per query; its tiles are divided evenly over them
    uint32_t *counters;
    // 1: q (and the window and the cache) are not written by the kernel launched
    // just before on the stream, so they may be read before the programmatic
    // dependent-launch wait (csa2_layer_step after its own top-k)
    int early;
};

// Splits (CTAs, at most 8 = one cluster) per query, and the workspace (none).
int attn_plan(int nq, int k_max, int n_win);
size_t attn_workspace_bytes(int nq, int H, int k_max, int n_win);
// The largest cluster of attention CTAs (splits of a query) this GPU schedules.
int attn_max_splits();
cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st);

}  // namespace csa2
