// csa2_index.cu -- indexer scoring (Full and Reindex modes) on tcgen05.
//
// score(q, j) = sum_h w_h * ReLU(q_h . k_j), q_h and k_j in E4M3 with
// power-of-two scales ([Notes] section 2: Full mode scores the whole visible
// context and Reindex rescores a shared key with its own query; section 3:
// the block-max pool and the Reindex search inside it).
//
// Layout of the contraction (swap-AB): the M = 128 rows of one MMA are 128
// cache entries (a TMA-loaded tile of the FP8 key cache, K-major, 128-byte
// swizzle), the N columns are the indexer heads of one query group (group *
// h_idx rows of FP8 query, padded to a multiple of 16) and K = d_idx.  The
// accumulator (128 lanes x N fp32) lives in tensor memory; each epilogue
// thread owns one entry (one TMEM lane) and turns its N dot products into
// `group` scores with the ReLU-weighted head sum, then reduces 8 lanes for the
// block max.  At decode the kernel is bound by the key stream from HBM
// (132 B per entry): one CTA per SM keeps ~200 KB of TMA loads in flight.
// With query groups (prefill: group 32, N = 256) the epilogue's ReLU-weighted
// head sums on the CUDA cores are the bound: a second instance runs two CTAs
// per SM with eight epilogue warps each, so that four epilogue warps per
// scheduler interleave; the two column halves of its accumulator are separate
// MMAs with their own TMEM barriers.
//
// Warp roles: warp 0 = TMA producer (the whole warp: in Reindex mode lane i
// fetches pool block i of a tile), warp 1 = MMA issuer and TMEM owner, warps
// 2.. = epilogue (warp w reads TMEM lanes 32 (w % 4) ..); 192 threads (four
// epilogue warps) at decode, 320 (eight) with query groups.
// Units of work are (query group, 128-entry tile); each CTA takes a contiguous
// range of units so the query tile (B operand) is reloaded only when the group
// changes.  Every wait is bounded in time (csa2::kWaitNs) and sets an abort flag.
#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

constexpr int kIdxThreads = 192;          // one CTA per SM: 4 epilogue warps
constexpr int kIdxThreadsGrouped = 320;   // two CTAs per SM: 8 epilogue warps each
constexpr int kIdxThreadsMax = kIdxThreadsGrouped;
constexpr int kTile = 128;
constexpr int kEpiBatch = 4;          // tiles the epilogue takes per pass (decode)
constexpr int kMaxGroupCols = 256;     // group * h_idx (the MMA's N) is at most 256
// the epilogue warps (2 ..) only
template <int kEpiThreads>
__device__ __forceinline__ void named_sync_epilogue()
{
    asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory");
}

struct IndexParams {
    const float *kscale;
    const int64_t *seq_base;
    const int32_t *seq_len;
    int64_t cap;
    int batch, d_idx, m;
    const int32_t *q_seq, *q_pos;
    const float *q_idx, *w;
    int nq, group, n_groups, h_idx, n_pad;
    int64_t max_n;
    // reindex (pool_blk != nullptr)
    const int32_t *pool_blk, *pool_n;
    int pool_blocks;
    // workspace
    uint8_t *q8img;    // [n_groups][n_pad][d_idx], swizzled like the smem tile
    float *ws;         // [nq][h_idx] = w * q scale
    int32_t *nt;       // [nq] candidates of each query
    int32_t *gtiles;   // [n_groups] tiles of each group
    // outputs
    float *scores;
    int64_t ld;
    float *blockmax;
    int64_t ld_bm;
    int32_t *n_valid;
    uint32_t *counters;
};

// Byte offset of (row r, byte c) in a K-major tile with `rowb`-byte rows under
// the matching TMA/UMMA swizzle (128 B rows: SW128, 64 B rows: SW64).
__device__ __forceinline__ uint32_t swz_off(uint32_t r, uint32_t c, uint32_t rowb)
{
    uint32_t chunk = c >> 4;
    uint32_t x = (rowb == 128) ? (r & 7u) : ((r >> 1) & 3u);
    return r * rowb + ((chunk ^ x) << 4) + (c & 15u);
}

// ---------------------------------------------------------------- prologue
// One CTA per query group: candidate counts, tiles per group, the FP8 query
// image (the smem B operand, pre-swizzled) and w * q scale.
__global__ void __launch_bounds__(256) index_prep_kernel(IndexParams p)
{
    pdl_wait();
    pdl_trigger();
    const int g = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = g * p.group;
    __shared__ int s_bad;
    __shared__ int s_maxn;
    if (threadIdx.x == 0) { s_bad = 0; s_maxn = 0; }
    __syncthreads();
    const int b = p.q_seq[q0];   // validated per query below before any use
    if (threadIdx.x < p.group) {
        const int q = q0 + threadIdx.x;
        int bad = 0;
        int64_t n = 0;
        if (p.q_seq[q] != b || b < 0 || b >= p.batch) bad = 1;
        if (!bad) {
            const int64_t base = p.seq_base[b];
            const int64_t room = p.seq_base[b + 1] - base;
            const int64_t len = p.seq_len[b];
            if ((base & 7) != 0 || base + room > p.cap || len > room) bad = 1;
            if (p.pool_blk == nullptr) {
                n = ((int64_t)p.q_pos[q] + 1) / p.m;
                if (n > len || n > p.max_n || p.q_pos[q] < 0) { bad = 1; n = 0; }
            } else {
                n = p.pool_n[q];
                if (n < 0 || n > 8LL * p.pool_blocks) { bad = 1; n = 0; }
            }
        }
        if (bad) { atomicOr(&s_bad, 1); n = 0; }
        p.nt[q] = (int32_t)n;
        if (p.n_valid) p.n_valid[q] = (int32_t)n;
        atomicMax(&s_maxn, (int)n);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (s_bad) count_event(p.counters, CSA2_CNT_BAD_INPUT);
        p.gtiles[g] = s_bad ? 0 : (s_maxn + kTile - 1) / kTile;
    }
    // FP8 query rows: row r = (query in group) * h_idx + head; padding rows = 0
    uint8_t *img = p.q8img + (int64_t)g * p.n_pad * p.d_idx;
    for (int r = warp; r < p.n_pad; r += blockDim.x / 32) {
        const int qq = r / p.h_idx, h = r % p.h_idx;
        const bool real = qq < p.group;
        const float *src = p.q_idx + ((int64_t)(q0 + qq) * p.h_idx + h) * p.d_idx;
        if (p.d_idx == 128) {
            float4 v = real ? __ldg(reinterpret_cast<const float4 *>(src) + lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
            float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const float s = fp8_pow2_scale(a);
            uint32_t word = e4m3_byte(v.x / s) | (e4m3_byte(v.y / s) << 8) |
                            (e4m3_byte(v.z / s) << 16) | (e4m3_byte(v.w / s) << 24);
            *reinterpret_cast<uint32_t *>(img + swz_off(r, lane * 4, 128)) = word;
            if (real && lane == 0) p.ws[(int64_t)(q0 + qq) * p.h_idx + h] =
                __ldg(p.w + (int64_t)(q0 + qq) * p.h_idx + h) * s;
        } else {
            float2 v = real ? __ldg(reinterpret_cast<const float2 *>(src) + lane)
                            : make_float2(0.f, 0.f);
            float a = fmaxf(fabsf(v.x), fabsf(v.y));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const float s = fp8_pow2_scale(a);
            uint16_t word = (uint16_t)(e4m3_byte(v.x / s) | (e4m3_byte(v.y / s) << 8));
            *reinterpret_cast<uint16_t *>(img + swz_off(r, lane * 2, 64)) = word;
            if (real && lane == 0) p.ws[(int64_t)(q0 + qq) * p.h_idx + h] =
                __ldg(p.w + (int64_t)(q0 + qq) * p.h_idx + h) * s;
        }
    }
}

// Scores of the queries in one 32-column pass of a group tile: query qq's HQ
// head columns, ReLU, weighted sum with its w * scale, times the key scale.
// (HQ a multiple of 4: the weights are read 4 at a time, sWg being 16-byte
// aligned, and the even and odd heads are summed in the two halves of a packed
// f32x2 FMA, then added.)
template <int HQ>
__device__ __forceinline__ void group_scores(const IndexParams &p, const float (&v)[32],
                                             const float *sWg, const int32_t *sNg, int c0, int nqp,
                                             int q0, int64_t j, float sk, int lane)
{
#pragma unroll
    for (int k2 = 0; k2 < 32 / HQ; ++k2) {
        if (k2 >= nqp) break;
        const int qq = c0 / HQ + k2;
        const float *wq = sWg + qq * HQ;
        float sc = 0.f;
        if constexpr (HQ % 4 == 0) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int h = 0; h < HQ; h += 4) {
                const float4 w4 = *reinterpret_cast<const float4 *>(wq + h);
                const float *x = v + k2 * HQ + h;
                acc = fma_f32x2(make_float2(w4.x, w4.y), make_float2(fmaxf(x[0], 0.f), fmaxf(x[1], 0.f)), acc);
                acc = fma_f32x2(make_float2(w4.z, w4.w), make_float2(fmaxf(x[2], 0.f), fmaxf(x[3], 0.f)), acc);
            }
            sc = acc.x + acc.y;
        } else {
#pragma unroll
            for (int h = 0; h < HQ; ++h) sc = fmaf(wq[h], fmaxf(v[k2 * HQ + h], 0.f), sc);
        }
        sc *= sk;
        const bool valid = j < sNg[qq];
        const int q = q0 + qq;
        if (valid) p.scores[(int64_t)q * p.ld + j] = sc;
        if (p.blockmax != nullptr) {
            float bm = valid ? sc : -INFINITY;
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
            if ((lane & 7) == 0 && valid) p.blockmax[(int64_t)q * p.ld_bm + (j >> 3)] = bm;
        }
    }
}

// ---------------------------------------------------------------- main kernel
// Position in this CTA's unit range: group g, tile t of it, and gt = tiles of
// group g (kept in a register: the global copy is read only on a group change).
struct UnitIter {
    int g, t, gt;
    int64_t u, u1;
};

__device__ __forceinline__ void unit_next(UnitIter &it, const int32_t *gtiles, int n_groups)
{
    ++it.u;
    ++it.t;
    while (it.g < n_groups && it.t >= it.gt) {
        ++it.g;
        it.t = 0;
        it.gt = it.g < n_groups ? gtiles[it.g] : 0;
    }
}

// kTwoPerSm: query groups run two CTAs per SM (registers capped to fit), each
// with eight epilogue warps (two per TMEM lane quarter, each taking half of the
// group's columns), so that the epilogues, the bottleneck there, have four
// warps per scheduler to interleave; decode runs one CTA with four.
template <int D_IDX, bool kTwoPerSm>
__global__ void __launch_bounds__(kTwoPerSm ? kIdxThreadsGrouped : kIdxThreads, kTwoPerSm ? 2 : 1)
    index_main_kernel(const __grid_constant__ CUtensorMap tmap, IndexParams p, int stages, int nacc)
{
    constexpr int kThreads = kTwoPerSm ? kIdxThreadsGrouped : kIdxThreads;
    constexpr int kEpiWarps = kThreads / 32 - 2;
    constexpr uint32_t kABytes = kTile * D_IDX;
    constexpr uint32_t kSbo = 8 * D_IDX;
    constexpr uint32_t kLayout = (D_IDX == 128) ? kLayoutSW128 : kLayoutSW64;
    const uint32_t b_bytes = (uint32_t)p.n_pad * D_IDX;
    const uint32_t b_stride = (b_bytes + 1023u) & ~1023u;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~(uintptr_t)1023);
    uint8_t *sA = smem;                                      // stages x kABytes
    float *sK = reinterpret_cast<float *>(sA + stages * kABytes);     // stages x 128 key scales
    uint8_t *sB = reinterpret_cast<uint8_t *>(sK + stages * kTile);   // 2 x b_stride (1024-aligned)
    sB = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sB) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + 2 * b_stride);
    uint64_t *full = bars, *empty = bars + stages;
    uint64_t *bfull = empty + stages, *bempty = bfull + 2;
    // kTwoPerSm: one TMEM accumulator whose two column halves (see csplit) each
    // have their own full / empty barrier pair
    const int nbar = kTwoPerSm ? 2 : nacc;
    uint64_t *tfull = bempty + 2, *tempty = tfull + nbar;
    uint64_t *done = tempty + nbar;
    int *sI = reinterpret_cast<int *>(done + 1);             // misc ints
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sI + 8);
    int64_t *s_scan = reinterpret_cast<int64_t *>(s_tmem + 2);  // kThreads
    float *sWg = reinterpret_cast<float *>(                              // [group * h_idx] (group > 1)
        (reinterpret_cast<uintptr_t>(s_scan + kIdxThreadsMax) + 15) & ~(uintptr_t)15);
    int32_t *sNg = reinterpret_cast<int32_t *>(sWg + kMaxGroupCols); // [group]

    volatile int *abort_flag = sI;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t ncols_acc = (uint32_t)p.n_pad;
    uint32_t tm_cols = 32;
    while (tm_cols < ncols_acc * nacc) tm_cols <<= 1;
    // column split between the two epilogue halves (a multiple of 32, so whole
    // queries on each side; used with eight epilogue warps)
    const int ncols_q = p.group * p.h_idx;
    const int csplit = min(ncols_q, (ncols_q + 63) / 64 * 32);

    if (tid == 0) {
        sI[0] = 0;
        for (int s = 0; s < stages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1 + kEpiWarps); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bfull[i], 1); mbar_init(&bempty[i], 1); }
        for (int i = 0; i < nbar; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kTwoPerSm ? kEpiWarps / 2 : kEpiWarps);
        }
        mbar_init(done, 1);
        fence_barrier_init();
        prefetch_tmap(&tmap);
    }
    if (warp == 1) { tmem_alloc(s_tmem, tm_cols); tmem_relinquish(); }
    // everything above touched no global memory that an earlier kernel writes.
    // No early trigger here: the top-k clusters that follow would be placed on
    // the first SMs this kernel frees, several per SM, and run ~1.5x slower
    // than when they are spread over the whole GPU at once.
    pdl_wait();

    // ---- this CTA's unit range [u0, u1) and its first (group, tile)
    {
        const int per = (p.n_groups + kThreads - 1) / kThreads;
        const int gs = min(tid * per, p.n_groups), ge = min(gs + per, p.n_groups);
        int64_t mine = 0;
        for (int g = gs; g < ge; ++g) mine += p.gtiles[g];
        // exclusive prefix of the per-thread counts: shuffles within each warp,
        // then the 6 warp totals
        int64_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_scan[warp] = incl;                // warp totals
        __syncthreads();
        int64_t before = 0, T = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int64_t v = s_scan[w];
            before += (w < warp) ? v : 0;
            T += v;
        }
        __syncthreads();                                     // the warp totals are read
        s_scan[tid] = before + incl - mine;
        if (tid == 0) {
            const int64_t u0 = T * blockIdx.x / gridDim.x, u1 = T * (blockIdx.x + 1) / gridDim.x;
            reinterpret_cast<int64_t *>(sI + 2)[0] = u0;
            reinterpret_cast<int64_t *>(sI + 2)[1] = u1;
            sI[1] = p.n_groups;   // start group (n_groups = none)
            sI[6] = 0;
        }
        __syncthreads();
        const int64_t u0 = reinterpret_cast<int64_t *>(sI + 2)[0];
        const int64_t u1 = reinterpret_cast<int64_t *>(sI + 2)[1];
        int64_t acc = s_scan[tid];
        if (u0 < u1 && acc <= u0 && u0 < acc + mine) {
            for (int g = gs; g < ge; ++g) {
                const int64_t n = p.gtiles[g];
                if (u0 < acc + n) { sI[1] = g; sI[6] = (int)(u0 - acc); break; }
                acc += n;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    UnitIter it0;
    it0.g = sI[1];
    it0.t = sI[6];
    it0.gt = it0.g < p.n_groups ? p.gtiles[it0.g] : 0;
    it0.u = reinterpret_cast<int64_t *>(sI + 2)[0];
    it0.u1 = reinterpret_cast<int64_t *>(sI + 2)[1];

    if (warp == 0) {
        // ================================================= TMA producer (whole warp:
        // lane 0 issues the Full-mode copies; in Reindex mode lane i fetches the
        // tile's pool block i)
        if (it0.u < it0.u1) {
            UnitIter it = it0;
            int stage = 0;
            uint32_t phase = 0;
            int prev_g = -1, bidx = 1;
            uint32_t buse[2] = {0, 0};
            int64_t n_issued = 0;
            int b = 0, pn = 0;
            const uint64_t l2_once = l2_evict_first_policy();
            int64_t base = 0, room = 0;
            // Reindex: lane i's pool block of the tiles 0..3 ahead, loaded 4 tiles
            // early so that these dependent reads overlap (rotated each tile)
            const bool reindex = p.pool_blk != nullptr;
            UnitIter la = it;
            auto pool_load = [&](const UnitIter &u) -> int {
                if (u.u >= u.u1) return -1;
                const int qq = u.g * p.group;
                const int nbq = min(kTile / 8, (p.nt[qq] + 7) / 8 - u.t * (kTile / 8));
                return lane < nbq ? p.pool_blk[(int64_t)qq * p.pool_blocks + u.t * (kTile / 8) + lane] : -1;
            };
            int pb0 = -1, pb1 = -1, pb2 = -1, pb3 = -1;
            if (reindex) {
                pb0 = pool_load(la); unit_next(la, p.gtiles, p.n_groups);
                pb1 = pool_load(la); unit_next(la, p.gtiles, p.n_groups);
                pb2 = pool_load(la); unit_next(la, p.gtiles, p.n_groups);
                pb3 = pool_load(la); unit_next(la, p.gtiles, p.n_groups);
            }
            while (it.u < it.u1) {
                const int g = it.g, t = it.t;
                const int q0 = g * p.group;
                if (g != prev_g) {
                    b = p.q_seq[q0];
                    base = p.seq_base[b];
                    room = p.seq_base[b + 1] - base;
                    if (p.pool_blk != nullptr) pn = p.nt[q0];     // group == 1 in Reindex mode
                    bidx ^= 1;
                    if (!__all_sync(0xffffffffu, mbar_wait<kTwoPerSm>(&bempty[bidx], (buse[bidx] & 1u) ^ 1u, abort_flag)))
                        break;
                    ++buse[bidx];
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bfull[bidx], b_bytes);
                        bulk_load(sB + bidx * b_stride, p.q8img + (int64_t)g * b_bytes, b_bytes,
                                  &bfull[bidx]);
                    }
                    prev_g = g;
                }
                if (!__all_sync(0xffffffffu, mbar_wait<kTwoPerSm>(&empty[stage], phase ^ 1u, abort_flag))) break;
                uint8_t *dstA = sA + stage * kABytes;
                float *dstK = sK + stage * kTile;
                if (p.pool_blk == nullptr) {
                    if (lane == 0) {
                        const int64_t r0 = base + (int64_t)t * kTile;
                        int64_t nk = p.cap - r0;
                        nk = nk > kTile ? kTile : nk;               // cap % 8 == 0, r0 % 8 == 0
                        mbar_arrive_expect_tx(&full[stage], kABytes + (uint32_t)nk * 4u);
                        if (kTwoPerSm) {
                            // query groups re-read the key tiles: default L2 policy
                            tma_load_2d(dstA, &tmap, 0, (int32_t)r0, &full[stage]);
                            bulk_load(dstK, p.kscale + r0, (uint32_t)nk * 4u, &full[stage]);
                        } else {
                            // decode streams each key once: evict it first, keep the scores
                            tma_load_2d_hint(dstA, &tmap, 0, (int32_t)r0, &full[stage], l2_once);
                            bulk_load_hint(dstK, p.kscale + r0, (uint32_t)nk * 4u, &full[stage], l2_once);
                        }
                    }
                } else {
                    const int nblk = (pn + 7) / 8;
                    const int bb0 = t * (kTile / 8);
                    const int nb = min(kTile / 8, nblk - bb0);
                    const int blk = pb0;
                    pb0 = pb1; pb1 = pb2; pb2 = pb3;
                    pb3 = pool_load(la);
                    unit_next(la, p.gtiles, p.n_groups);
                    const bool ok_blk = lane < nb && blk >= 0 && 8LL * blk + 8 <= room;
                    const uint32_t vmask = __ballot_sync(0xffffffffu, ok_blk);
                    const uint32_t nvalid = (uint32_t)__popc(vmask);
                    if (lane == 0) {
                        if ((int)nvalid < nb) count_event(p.counters, CSA2_CNT_BAD_INPUT);
                        mbar_arrive_expect_tx(&full[stage], nvalid * (8u * D_IDX + 32u));
                    }
                    __syncwarp();
                    if (ok_blk) {
                        const int64_t r = base + 8LL * blk;
                        tma_load_2d_hint(dstA + lane * 8 * D_IDX, &tmap, 0, (int32_t)r, &full[stage], l2_once);
                        bulk_load_hint(dstK + lane * 8, p.kscale + r, 32u, &full[stage], l2_once);
                    }
                }
                ++n_issued;
                if (++stage == stages) { stage = 0; phase ^= 1u; }
                unit_next(it, p.gtiles, p.n_groups);
            }
            if (lane == 0 && it.u < it.u1) { *abort_flag = 1; count_event(p.counters, CSA2_CNT_TIMEOUT); }
            // no copy of ours may still be landing when the CTA exits: wait (bounded)
            // for the last arming of every stage (issue i used stage i % stages, its
            // (i / stages)-th arming) and of every query buffer
            if (lane == 0) {
                volatile int no_abort = 0;
                for (int s = 0; s < stages; ++s) {
                    if (n_issued <= s) continue;
                    const int64_t last = s + (n_issued - 1 - s) / stages * stages;
                    mbar_wait(&full[s], (uint32_t)((last / stages) & 1), &no_abort);
                }
                for (int i = 0; i < 2; ++i)
                    if (buse[i]) mbar_wait(&bfull[i], (buse[i] - 1u) & 1u, &no_abort);
            }
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (lane == 0 && it0.u < it0.u1) {
            UnitIter it = it0;
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            int prev_g = -1, bidx = 1;
            uint32_t buse[2] = {0, 0};
            const uint32_t idesc = instr_desc(128, (uint32_t)p.n_pad, 0, 0, 0, 0);
            while (it.u < it.u1) {
                const int g = it.g;
                if (g != prev_g) {
                    if (prev_g >= 0) mma_commit(&bempty[bidx]);
                    bidx ^= 1;
                    if (!mbar_wait<kTwoPerSm>(&bfull[bidx], buse[bidx] & 1u, abort_flag)) break;
                    ++buse[bidx];
                    prev_g = g;
                }
                if (!mbar_wait<kTwoPerSm>(&full[stage], phase, abort_flag)) break;
                const uint32_t a0 = smem_u32(sA + stage * kABytes);
                const uint32_t b0 = smem_u32(sB + bidx * b_stride);
                if constexpr (kTwoPerSm) {
                    // columns [0, csplit) and [csplit, n_pad): separate MMAs and
                    // barriers, so each epilogue half waits only for its own columns
                    bool ok = true;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (!mbar_wait<true>(&tempty[h], aphase ^ 1u, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t c0 = h ? (uint32_t)csplit : 0u;
                        const uint32_t n = h ? (uint32_t)(p.n_pad - csplit) : (uint32_t)csplit;
                        const uint32_t id = instr_desc(128, n, 0, 0, 0, 0);
#pragma unroll
                        for (int k = 0; k < D_IDX / 32; ++k) {
                            mma_f8f6f4(tmem_base + c0, smem_desc(a0 + 32 * k, 16, kSbo, kLayout),
                                       smem_desc(b0 + c0 * D_IDX + 32 * k, 16, kSbo, kLayout), id, k > 0);
                        }
                        mma_commit(&tfull[h]);
                    }
                    if (!ok) break;
                    mma_commit(&empty[stage]);
                } else {
                    if (!mbar_wait<kTwoPerSm>(&tempty[acc], aphase ^ 1u, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)acc * ncols_acc;
#pragma unroll
                    for (int k = 0; k < D_IDX / 32; ++k) {
                        mma_f8f6f4(d, smem_desc(a0 + 32 * k, 16, kSbo, kLayout),
                                   smem_desc(b0 + 32 * k, 16, kSbo, kLayout), idesc, k > 0);
                    }
                    mma_commit(&empty[stage]);
                    mma_commit(&tfull[acc]);
                }
                if (++stage == stages) { stage = 0; phase ^= 1u; }
                if (++acc == nacc) { acc = 0; aphase ^= 1u; }
                unit_next(it, p.gtiles, p.n_groups);
            }
            if (it.u < it.u1) { *abort_flag = 1; count_event(p.counters, CSA2_CNT_TIMEOUT); }
            // all MMAs of this thread complete before TMEM is released
            mma_commit(done);
            if (!mbar_wait(done, 0, abort_flag)) count_event(p.counters, CSA2_CNT_TIMEOUT);
        }
    } else {
        // ================================================= epilogue (128 threads)
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int row = (int)(quarter * 32 + lane);        // TMEM lane = entry within tile
        UnitIter it = it0;
        int stage = 0, acc = 0;
        uint32_t aphase = 0, sphase = 0;
        int prev_g = -1;
        float wsr[16];
        int ntq = 0;
        while (it.u < it.u1) {
            const int g = it.g, t = it.t;
            const int q0 = g * p.group;
            // (kTwoPerSm is only launched for groups of more than 64 / h_idx queries)
            if (!kTwoPerSm && g != prev_g && p.group == 1) {
                for (int h = 0; h < 16; ++h) wsr[h] = (h < p.h_idx) ? p.ws[(int64_t)q0 * p.h_idx + h] : 0.f;
                ntq = p.nt[q0];
                prev_g = g;
            }
            if (!kTwoPerSm && p.group == 1) {
                // up to kEpiBatch consecutive tiles of this query per pass: all their
                // TMEM loads are in flight together, one wait, one release each
                int nb = 0, bt[kEpiBatch], bs[kEpiBatch], ba[kEpiBatch];
                bool ok = true;
                {
                    UnitIter pk = it;
                    while (nb < kEpiBatch && pk.u < pk.u1 && pk.g == g) {
                        ok = ok && mbar_wait(&tfull[acc], aphase, abort_flag);
                        // the stage's TMA data (key scales) is complete: observe it directly
                        ok = ok && mbar_wait(&full[stage], sphase, abort_flag);
                        bt[nb] = pk.t; bs[nb] = stage; ba[nb] = acc; ++nb;
                        if (++stage == stages) { stage = 0; sphase ^= 1u; }
                        if (++acc == nacc) { acc = 0; aphase ^= 1u; }
                        unit_next(pk, p.gtiles, p.n_groups);
                    }
                    it = pk;
                }
                // warp-uniform: the TMEM loads below are .sync.aligned
                if (!__all_sync(0xffffffffu, ok)) {
                    *abort_flag = 1;
                    if (lane == 0) count_event(p.counters, CSA2_CNT_TIMEOUT);
                    break;
                }
                tc_fence_after();
                float v[kEpiBatch][16];
#pragma unroll
                for (int b = 0; b < kEpiBatch; ++b)
                    if (b < nb)
                        tmem_ld16(tmem_base + ((quarter * 32u) << 16) + (uint32_t)ba[b] * ncols_acc, v[b]);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    for (int b = 0; b < nb; ++b) mbar_arrive(&tempty[ba[b]]);
#pragma unroll
                for (int b = 0; b < kEpiBatch; ++b) {
                    if (b >= nb) break;
                    const int64_t j = (int64_t)bt[b] * kTile + row;
                    float sc = 0.f;
#pragma unroll
                    for (int h = 0; h < 16; ++h) sc = fmaf(wsr[h], fmaxf(v[b][h], 0.f), sc);
                    sc *= sK[bs[b] * kTile + row];
                    const bool valid = j < ntq;
                    if (valid) p.scores[(int64_t)q0 * p.ld + j] = sc;
                    if (p.blockmax != nullptr) {
                        float bm = valid ? sc : -INFINITY;
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
                        if ((lane & 7) == 0 && valid) p.blockmax[(int64_t)q0 * p.ld_bm + (j >> 3)] = bm;
                    }
                }
                // this warp is done with the stages' key scales: its share of their release
                __syncwarp();
                if (lane == 0)
                    for (int b = 0; b < nb; ++b) mbar_arrive(&empty[bs[b]]);
                continue;
            }
            // warp-uniform waits: the TMEM loads below are .sync.aligned
            const int tb = kTwoPerSm ? (warp >= 6 ? 1 : 0) : acc;   // this warp's TMEM barrier pair
            bool ok = mbar_wait<kTwoPerSm>(&tfull[tb], aphase, abort_flag);
            // the stage's TMA data (key scales) is complete: observe it directly
            // (already complete, and it cannot be re-armed before this warp releases it)
            ok = ok && mbar_wait<kTwoPerSm>(&full[stage], sphase, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                *abort_flag = 1;
                if (lane == 0) count_event(p.counters, CSA2_CNT_TIMEOUT);
                break;
            }
            // a new query group: its w * scale and candidate counts into shared
            // memory, once, by the four epilogue warps together
            if (g != prev_g) {
                named_sync_epilogue<32 * kEpiWarps>();   // the previous group's values are no longer read
                const int etid = tid - 64;
                for (int i = etid; i < p.group * p.h_idx; i += 32 * kEpiWarps)
                    sWg[i] = p.ws[(int64_t)q0 * p.h_idx + i];
                for (int i = etid; i < p.group; i += 32 * kEpiWarps) sNg[i] = p.nt[q0 + i];
                named_sync_epilogue<32 * kEpiWarps>();
                prev_g = g;
            }
            tc_fence_after();
            const int64_t j = (int64_t)t * kTile + row;
            const float sk = sK[stage * kTile + row];
            const uint32_t tbase = tmem_base + ((quarter * 32u) << 16) + (uint32_t)acc * ncols_acc;
            {
                // h_idx columns per query, 32 columns per pass (h_idx divides 16, so
                // a pass holds whole queries); the next pass's TMEM loads are in
                // flight while this pass is summed.  With eight epilogue warps, warps
                // 2..5 take the columns below `split` (a multiple of 32) and 6..9 the rest.
                const int hq = p.h_idx, hq_sh = __ffs(hq) - 1;    // h_idx is a power of two
                const int ncols = p.group * hq;
                int c_lo = 0, c_hi = ncols;
                if (kEpiWarps == 8) {
                    if (warp >= 6) c_lo = csplit; else c_hi = csplit;
                }
                auto load32 = [&](int c, float (&v)[32]) {
                    tmem_ld16(tbase + (uint32_t)c, *reinterpret_cast<float(*)[16]>(v));
                    if (c + 16 < c_hi) tmem_ld16(tbase + (uint32_t)c + 16, *reinterpret_cast<float(*)[16]>(v + 16));
                };
                auto sum32 = [&](int c, const float (&v)[32]) {
                    const int nqp = min(32, c_hi - c) >> hq_sh;       // queries in this pass
                    switch (hq) {
                    case 1: group_scores<1>(p, v, sWg, sNg, c, nqp, q0, j, sk, lane); break;
                    case 2: group_scores<2>(p, v, sWg, sNg, c, nqp, q0, j, sk, lane); break;
                    case 4: group_scores<4>(p, v, sWg, sNg, c, nqp, q0, j, sk, lane); break;
                    case 8: group_scores<8>(p, v, sWg, sNg, c, nqp, q0, j, sk, lane); break;
                    default: group_scores<16>(p, v, sWg, sNg, c, nqp, q0, j, sk, lane); break;
                    }
                };
                if constexpr (kEpiWarps == 8) {
                    // (registers are capped for two CTAs per SM: one pass in flight;
                    // the other three warps of this scheduler hide the load)
                    for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
                        float va[32];
                        if (c0 + 16 < c_hi) {
                            tmem_ld32(tbase + (uint32_t)c0, va);
                        } else {
                            tmem_ld16(tbase + (uint32_t)c0, *reinterpret_cast<float(*)[16]>(va));
                        }
                        tmem_wait_ld();
                        sum32(c0, va);
                    }
                } else {
                    float va[32], vb[32];
                    if (c_lo < c_hi) {
                        load32(c_lo, va);
                        tmem_wait_ld();
                    }
                    for (int c0 = c_lo; c0 < c_hi; c0 += 64) {
                        const bool has_b = c0 + 32 < c_hi, has_a = c0 + 64 < c_hi;
                        if (has_b) load32(c0 + 32, vb);
                        sum32(c0, va);
                        if (!has_b) break;
                        tmem_wait_ld();
                        if (has_a) load32(c0 + 64, va);
                        sum32(c0 + 32, vb);
                        if (has_a) tmem_wait_ld();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[tb]);
            }
            // this warp is done with the stage's key scales: its share of the release
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == stages) { stage = 0; sphase ^= 1u; }
            if (++acc == nacc) { acc = 0; aphase ^= 1u; }
            unit_next(it, p.gtiles, p.n_groups);
        }
        if (it.u < it.u1) *abort_flag = 1;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tm_cols);
    }
}

// ---------------------------------------------------------------- host side
static size_t index_smem_bytes(int d_idx, int n_pad, int stages, int nacc)
{
    const size_t a = (size_t)stages * kTile * d_idx;
    const size_t k = (size_t)stages * kTile * 4;
    const size_t b = 2 * (((size_t)n_pad * d_idx + 1023) & ~(size_t)1023);
    const size_t bars = (size_t)(2 * stages + 4 + 2 * (nacc > 2 ? nacc : 2) + 1) * 8;
    return 1024 /*align*/ + a + k + 1024 /*align B*/ + b + bars + 64 + kIdxThreadsMax * 8 + 16 +
           kMaxGroupCols * 4 + kMaxGroupCols * 4;
}

size_t index_workspace_bytes(int nq, int group, int h_idx, int d_idx)
{
    const int n_groups = nq / group;
    int n_pad = ((group * h_idx + 15) / 16) * 16;
    size_t s = align_up((size_t)n_groups * n_pad * d_idx, 256);
    s += align_up((size_t)nq * h_idx * 4, 256);
    s += align_up((size_t)nq * 4, 256);
    s += align_up((size_t)n_groups * 4, 256);
    return s;
}

cudaError_t launch_index(const csa2_cache &c, const csa2_queries &qs, const float *q_idx,
                         const float *w, int h_idx, int64_t max_n, const int32_t *pool_blk,
                         const int32_t *pool_n, int pool_blocks, float *scores, int64_t ld,
                         float *blockmax, int64_t ld_bm, int32_t *n_valid, void *ws,
                         uint32_t *counters, cudaStream_t st)
{
    IndexParams p{};
    p.kscale = c.kscale;
    p.seq_base = c.seq_base;
    p.seq_len = c.seq_len;
    p.cap = c.cap;
    p.batch = c.batch;
    p.d_idx = c.d_idx;
    p.m = c.m;
    p.q_seq = qs.q_seq;
    p.q_pos = qs.q_pos;
    p.q_idx = q_idx;
    p.w = w;
    p.nq = qs.nq;
    p.group = qs.group;
    p.n_groups = qs.nq / qs.group;
    p.h_idx = h_idx;
    p.n_pad = ((qs.group * h_idx + 15) / 16) * 16;
    p.max_n = max_n;
    p.pool_blk = pool_blk;
    p.pool_n = pool_n;
    p.pool_blocks = pool_blocks;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    p.q8img = wsb;
    wsb += align_up((size_t)p.n_groups * p.n_pad * c.d_idx, 256);
    p.ws = reinterpret_cast<float *>(wsb);
    wsb += align_up((size_t)qs.nq * h_idx * 4, 256);
    p.nt = reinterpret_cast<int32_t *>(wsb);
    wsb += align_up((size_t)qs.nq * 4, 256);
    p.gtiles = reinterpret_cast<int32_t *>(wsb);
    p.scores = scores;
    p.ld = ld;
    p.blockmax = blockmax;
    p.ld_bm = ld_bm;
    p.n_valid = n_valid;
    p.counters = counters;

    CUtensorMap tmap;
    cudaError_t e = make_tmap_rows_u8(&tmap, c.kidx, c.cap, c.d_idx,
                                      pool_blk ? 8 : kTile, c.d_idx == 128 ? 128 : 64);
    if (e != cudaSuccess) return e;

    e = launch_k(index_prep_kernel, dim3(p.n_groups), dim3(256), 0, st, 0, p);
    if (e != cudaSuccess) return e;

    // decode (N <= 64): one CTA per SM with a deep key pipeline (HBM-bound);
    // query groups (N up to 256): two CTAs per SM, each with a shallow pipeline
    // and one accumulator, whose MMAs and epilogues interleave
    const bool grouped = p.n_pad > 64;
    const int stages = grouped ? 2 : (c.d_idx == 128 ? 12 : 16);
    const int nacc = grouped ? 1 : 8;
    const size_t smem = index_smem_bytes(c.d_idx, p.n_pad, stages, nacc);
    const int grid = device_sm_count() * (grouped ? 2 : 1);
    auto run = [&](auto k) {
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return launch_k(k, dim3(grid), dim3(grouped ? kIdxThreadsGrouped : kIdxThreads), smem, st, 0,
                        tmap, p, stages, nacc);
    };
    if (c.d_idx == 128)
        e = grouped ? run(index_main_kernel<128, true>) : run(index_main_kernel<128, false>);
    else
        e = grouped ? run(index_main_kernel<64, true>) : run(index_main_kernel<64, false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csa2

