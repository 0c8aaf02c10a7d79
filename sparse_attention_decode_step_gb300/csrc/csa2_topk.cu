// csa2_topk.cu -- per-query top-k by radix select, and the candidate pool.
//
// Top-k: the k largest scores, ties to the lower position, listed ascending
// (the tie rule is this library's reading; the pages give none).
// Scores become order-preserving uint32 keys (-0 == +0).  Three histogram
// rounds (11 + 11 + 10 bits) find the exact k-th key T and how many keys equal
// to T are taken; a final ordered compaction writes every key > T and the
// first (lowest-position) keys == T.  Up to 256K candidates a query is one
// cluster of 8 CTAs (keys in shared memory, cluster barriers between rounds);
// above that the work is split into 4096-candidate chunks over many CTAs in
// separate launches, histograms merged with global atomics (no CTA ever waits
// on another).
//
// Pool ([Notes] section 3): the same selection over the block maxima of a Full
// layer (k = 2,048 blocks), then the count of visible positions they hold.
#include <cooperative_groups.h>
#include <mutex>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

constexpr int kChunk = 4096;
constexpr int kTkThreads = 256;
constexpr int kPerThread = kChunk / kTkThreads;   // 16
constexpr int kBins = 2048;

struct TopkState {
    uint32_t prefix;   // key bits fixed so far
    int32_t k_rem;     // elements still to take among those matching prefix
    int32_t n;         // candidates of this query
    int32_t all;       // n <= k: every candidate is taken
};

struct TopkParams {
    const float *scores;
    int64_t ld;
    const int32_t *n_valid;
    int n_div8;                 // candidates = ceil(n_valid / 8) (block maxima)
    const int32_t *pool_blk;    // candidate -> position map, or null
    int pool_blocks;
    int nq, k, n_chunks;
    int64_t max_n;              // bound on every query's candidate count (smem sizing)
    int32_t *idx_out;
    int64_t ld_idx;
    int32_t *cnt_out;
    // workspace
    uint32_t *hist;             // [3][nq][kBins]
    TopkState *state;           // [nq]
    uint32_t *ccount;           // [nq][n_chunks][2]  (gt, eq)
    uint32_t *coff;             // [nq][n_chunks][2]  (out offset, eq before)
    const uint32_t *hist0;      // [nq][kBins] first-digit histogram from the indexer, or null
};

__device__ __forceinline__ int round_shift(int r) { return r == 0 ? 21 : (r == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t round_bins(int r) { return r == 2 ? 1024u : 2048u; }

__global__ void topk_init_kernel(TopkParams p)
{
    pdl_wait();
    pdl_trigger();
    const int q = blockIdx.x;
    for (int i = threadIdx.x; i < 3 * kBins; i += blockDim.x) {
        const int r = i / kBins, b = i % kBins;
        p.hist[((int64_t)r * p.nq + q) * kBins + b] = 0u;
    }
    if (threadIdx.x == 0) {
        int n = p.n_valid[q];
        if (p.n_div8) n = (n + 7) / 8;
        if (n < 0) n = 0;
        TopkState s;
        s.prefix = 0u;
        s.n = n;
        s.all = (n <= p.k) ? 1 : 0;
        s.k_rem = s.all ? n : p.k;
        p.state[q] = s;
        p.cnt_out[q] = s.all ? n : p.k;
    }
}

__global__ void __launch_bounds__(kTkThreads) topk_hist_kernel(TopkParams p, int r)
{
    pdl_wait();
    pdl_trigger();
    const int q = blockIdx.y, c = blockIdx.x;
    const TopkState st = p.state[q];
    if (st.all) return;
    const int64_t i0 = (int64_t)c * kChunk;
    if (i0 >= st.n) return;
    __shared__ uint32_t h[kBins];
    for (int i = threadIdx.x; i < kBins; i += kTkThreads) h[i] = 0u;
    __syncthreads();
    const float *row = p.scores + (int64_t)q * p.ld;
    const int sh = round_shift(r);
    const uint32_t mask = round_bins(r) - 1u;
    for (int e = 0; e < kPerThread; ++e) {
        const int64_t i = i0 + e * kTkThreads + threadIdx.x;
        if (i < st.n) {
            const uint32_t key = score_key(row[i]);
            bool match = (r == 0) || ((key >> (sh + (r == 1 ? 11 : 10))) == st.prefix);
            if (match) atomicAdd(&h[(key >> sh) & mask], 1u);
        }
    }
    __syncthreads();
    uint32_t *gh = p.hist + ((int64_t)r * p.nq + q) * kBins;
    for (int i = threadIdx.x; i < (int)round_bins(r); i += kTkThreads)
        if (h[i]) atomicAdd(gh + i, h[i]);
}

// Block-wide exclusive scan of one value per thread (kTkThreads threads).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *s_warp, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = (lane < kTkThreads / 32) ? s_warp[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kTkThreads / 32) s_warp[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before = (warp > 0) ? s_warp[warp - 1] : 0u;
    if (total) *total = s_warp[kTkThreads / 32 - 1];
    __syncthreads();
    return before + x - v;
}

// Picks the digit of round r: bins are scanned from the top; the digit d has
// count(> d) < k_rem <= count(>= d).
__global__ void __launch_bounds__(kTkThreads) topk_scan_kernel(TopkParams p, int r)
{
    pdl_wait();
    pdl_trigger();
    const int q = blockIdx.x;
    TopkState st = p.state[q];
    if (st.all) return;
    const uint32_t nb = round_bins(r);
    const uint32_t per = nb / kTkThreads;      // 8 or 4 bins per thread, descending digits
    const uint32_t *gh = p.hist + ((int64_t)r * p.nq + q) * kBins;
    uint32_t cnt[8];
    uint32_t mine = 0;
    for (uint32_t i = 0; i < per; ++i) {
        const uint32_t d = nb - 1u - (threadIdx.x * per + i);
        cnt[i] = gh[d];
        mine += cnt[i];
    }
    __shared__ uint32_t s_warp[kTkThreads / 32];
    __shared__ uint32_t s_digit, s_above;
    if (threadIdx.x == 0) { s_digit = 0; s_above = 0; }
    __syncthreads();
    uint32_t before = block_excl_scan(mine, s_warp, nullptr);
    const uint32_t need = (uint32_t)st.k_rem;
    if (before < need && need <= before + mine) {
        uint32_t acc = before;
        for (uint32_t i = 0; i < per; ++i) {
            if (need <= acc + cnt[i]) {
                s_digit = nb - 1u - (threadIdx.x * per + i);
                s_above = acc;
                break;
            }
            acc += cnt[i];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int bits = (r == 2) ? 10 : 11;
        st.prefix = (st.prefix << bits) | s_digit;
        st.k_rem -= (int32_t)s_above;
        p.state[q] = st;
    }
}

__device__ __forceinline__ void load16(const float *row, int64_t i0, int64_t n, uint32_t (&key)[16],
                                       bool (&ok)[16])
{
    // 16 consecutive candidates i0..i0+15 of this thread
    if (i0 + 16 <= n) {
        const float4 *v4 = reinterpret_cast<const float4 *>(row + i0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 v = v4[j];
            key[4 * j] = score_key(v.x);
            key[4 * j + 1] = score_key(v.y);
            key[4 * j + 2] = score_key(v.z);
            key[4 * j + 3] = score_key(v.w);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) ok[j] = true;
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            ok[j] = (i0 + j) < n;
            key[j] = ok[j] ? score_key(row[i0 + j]) : 0u;
        }
    }
}

__global__ void __launch_bounds__(kTkThreads) topk_count_kernel(TopkParams p)
{
    pdl_wait();
    pdl_trigger();
    const int q = blockIdx.y, c = blockIdx.x;
    const TopkState st = p.state[q];
    const int64_t i0 = (int64_t)c * kChunk + threadIdx.x * kPerThread;
    uint32_t gt = 0, eq = 0;
    if (!st.all) {
        uint32_t key[16];
        bool ok[16];
        load16(p.scores + (int64_t)q * p.ld, i0, st.n, key, ok);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            gt += (ok[j] && key[j] > st.prefix);
            eq += (ok[j] && key[j] == st.prefix);
        }
    } else {
        gt = (uint32_t)max((int64_t)0, min((int64_t)kPerThread, (int64_t)st.n - i0));
    }
    __shared__ uint32_t s_warp[kTkThreads / 32];
    uint32_t tgt, teq;
    block_excl_scan(gt, s_warp, &tgt);
    block_excl_scan(eq, s_warp, &teq);
    if (threadIdx.x == 0) {
        uint32_t *cc = p.ccount + ((int64_t)q * p.n_chunks + c) * 2;
        cc[0] = tgt;
        cc[1] = teq;
    }
}

__global__ void __launch_bounds__(kTkThreads) topk_offsets_kernel(TopkParams p)
{
    pdl_wait();
    pdl_trigger();
    const int q = blockIdx.x;
    const TopkState st = p.state[q];
    const int32_t k_eq = st.all ? 0 : st.k_rem;
    __shared__ uint32_t s_warp[kTkThreads / 32];
    __shared__ uint32_t s_carry_out, s_carry_eq;
    if (threadIdx.x == 0) { s_carry_out = 0; s_carry_eq = 0; }
    __syncthreads();
    for (int c0 = 0; c0 < p.n_chunks; c0 += kTkThreads) {
        const int c = c0 + threadIdx.x;
        uint32_t gt = 0, eq = 0;
        if (c < p.n_chunks) {
            const uint32_t *cc = p.ccount + ((int64_t)q * p.n_chunks + c) * 2;
            gt = cc[0];
            eq = cc[1];
        }
        uint32_t eq_tot;
        const uint32_t eq_before = s_carry_eq + block_excl_scan(eq, s_warp, &eq_tot);
        int64_t take = (int64_t)k_eq - (int64_t)eq_before;
        take = take < 0 ? 0 : (take > eq ? eq : take);
        uint32_t out_tot;
        const uint32_t out_before = s_carry_out + block_excl_scan(gt + (uint32_t)take, s_warp, &out_tot);
        if (c < p.n_chunks) {
            uint32_t *co = p.coff + ((int64_t)q * p.n_chunks + c) * 2;
            co[0] = out_before;
            co[1] = eq_before;
        }
        __syncthreads();
        if (threadIdx.x == 0) { s_carry_out += out_tot; s_carry_eq += eq_tot; }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kTkThreads) topk_write_kernel(TopkParams p)
{
    pdl_wait();
    pdl_trigger();
    const int q = blockIdx.y, c = blockIdx.x;
    const TopkState st = p.state[q];
    const int64_t i0 = (int64_t)c * kChunk + threadIdx.x * kPerThread;
    if ((int64_t)c * kChunk >= st.n) return;
    const uint32_t *co = p.coff + ((int64_t)q * p.n_chunks + c) * 2;
    const uint32_t out0 = co[0], eqb = co[1];
    uint32_t key[16];
    bool ok[16];
    uint32_t sel_mask = 0, eq_mask = 0;
    if (st.all) {
#pragma unroll
        for (int j = 0; j < 16; ++j) if (i0 + j < st.n) sel_mask |= 1u << j;
    } else {
        load16(p.scores + (int64_t)q * p.ld, i0, st.n, key, ok);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (ok[j] && key[j] > st.prefix) sel_mask |= 1u << j;
            if (ok[j] && key[j] == st.prefix) eq_mask |= 1u << j;
        }
    }
    __shared__ uint32_t s_warp[kTkThreads / 32];
    const uint32_t eq_rank0 = eqb + block_excl_scan(__popc(eq_mask), s_warp, nullptr);
    uint32_t r = eq_rank0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (eq_mask & (1u << j)) {
            if ((int64_t)r < (int64_t)st.k_rem) sel_mask |= 1u << j;
            ++r;
        }
    }
    uint32_t slot = out0 + block_excl_scan(__popc(sel_mask), s_warp, nullptr);
    int32_t *out = p.idx_out + (int64_t)q * p.ld_idx;
    const int32_t *pb = p.pool_blk ? p.pool_blk + (int64_t)q * p.pool_blocks : nullptr;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (sel_mask & (1u << j)) {
            const int64_t i = i0 + j;
            const int32_t pos = pb ? 8 * pb[i >> 3] + (int32_t)(i & 7) : (int32_t)i;
            if (slot < (uint32_t)p.k) out[slot] = pos;   // exactly min(k, n) slots exist
            ++slot;
        }
    }
}

// ---------------------------------------------------------------- one cluster per query
// Up to kClusterMax candidates: a cluster of 8 CTAs per query.  Each CTA keeps
// its eighth of the keys in shared memory (one pass over the scores) and
// builds a shared-memory histogram of each round; the non-empty bins go to the
// query's histogram in the workspace with global atomics, and after a cluster
// barrier every CTA reads it back and takes the same digit decision.  The
// ordered compaction exchanges per-CTA counts the same way.  One launch; the
// cluster barriers are hardware barriers reached by every CTA equally often.
constexpr int kClusterCtas = 8;
constexpr int kClThreads = 512;
constexpr int64_t kClusterMax = 262144;
constexpr int kClChunkMax = (int)(kClusterMax / kClusterCtas);   // keys per CTA

// Block-wide exclusive scan (512 threads); *total gets the block sum.
__device__ __forceinline__ uint32_t scan512(uint32_t v, uint32_t *s_warp, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kClThreads / 32 ? s_warp[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kClThreads / 32) s_warp[lane] = w;       // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before = warp > 0 ? s_warp[warp - 1] : 0u;
    if (total) *total = s_warp[kClThreads / 32 - 1];
    __syncthreads();
    return before + x - v;
}

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kClThreads)
    topk_cluster_kernel(TopkParams p)
{
    pdl_wait();
    pdl_trigger();
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int q = blockIdx.y, rank = (int)cluster.block_rank(), tid = threadIdx.x;
    extern __shared__ __align__(16) uint32_t s_keys[];          // [chunk]
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t s_warp[kClThreads / 32];
    __shared__ uint32_t s_digit, s_above;

    int n = p.n_valid[q];
    if (p.n_div8) n = (n + 7) / 8;
    if (n < 0) n = 0;
    if (n > p.max_n) n = (int)p.max_n;                           // shared memory was sized for max_n
    const int chunk = ((n + kClusterCtas - 1) / kClusterCtas + 3) & ~3;
    const int lo = min(rank * chunk, n), hi = min(lo + chunk, n);
    const int len = hi - lo;
    const float *row = p.scores + (int64_t)q * p.ld;
    const bool all = n <= p.k;
    uint32_t prefix = 0;
    int32_t k_rem = all ? n : p.k;
    // per-query global histograms (one per round) and per-CTA counts, in the workspace
    uint32_t *ghist = p.hist + (int64_t)q * 3 * kBins;
    uint32_t *gcnt = p.ccount + (int64_t)q * kClusterCtas * 2;
    if (rank == 0) {
        if (tid == 0) p.cnt_out[q] = all ? n : p.k;
        for (int i = tid; i < 3 * kBins; i += kClThreads) ghist[i] = 0u;
    }
    for (int i = tid; i < kBins; i += kClThreads) hist[i] = 0u;   // re-cleared by each merge
    __syncthreads();

    // keys of this CTA's candidates into shared memory (lo is a multiple of 4),
    // with the first round's histogram (top 11 bits) built on the way; a
    // thread's loads of one pass (up to kLoadUnroll float4) are all in flight
    // before the first is used
    constexpr int kLoadUnroll = 4;
    for (int i0 = tid * 4; i0 < len; i0 += kClThreads * 4 * kLoadUnroll) {
        float4 f[kLoadUnroll];
#pragma unroll
        for (int u = 0; u < kLoadUnroll; ++u) {
            const int i = i0 + u * kClThreads * 4;
            if (i + 4 <= len) f[u] = *reinterpret_cast<const float4 *>(row + lo + i);
        }
#pragma unroll
        for (int u = 0; u < kLoadUnroll; ++u) {
            const int i = i0 + u * kClThreads * 4;
            if (i + 4 <= len) {
                const uint32_t k0 = score_key(f[u].x), k1 = score_key(f[u].y);
                const uint32_t k2 = score_key(f[u].z), k3 = score_key(f[u].w);
                *reinterpret_cast<uint4 *>(s_keys + i) = make_uint4(k0, k1, k2, k3);
                if (!all) {
                    atomicAdd(&hist[k0 >> 21], 1u);
                    atomicAdd(&hist[k1 >> 21], 1u);
                    atomicAdd(&hist[k2 >> 21], 1u);
                    atomicAdd(&hist[k3 >> 21], 1u);
                }
            } else if (i < len) {
                for (int j = i; j < len; ++j) {
                    const uint32_t kj = score_key(row[lo + j]);
                    s_keys[j] = kj;
                    if (!all) atomicAdd(&hist[kj >> 21], 1u);
                }
            }
        }
    }
    cluster.sync();                                              // histograms zeroed, keys loaded

    if (!all) {
        for (int r = 0; r < 3; ++r) {
            const int sh = r == 0 ? 21 : (r == 1 ? 10 : 0);
            const int pbits = r == 0 ? 0 : (r == 1 ? 11 : 22);
            const uint32_t nb = r == 2 ? 1024u : 2048u;
            if (r > 0) {                                         // round 0 was built with the load
#pragma unroll 4
                for (int i = tid; i < len; i += kClThreads) {
                    const uint32_t key = s_keys[i];
                    if ((key >> (32 - pbits)) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1u)], 1u);
                }
            }
            __syncthreads();
            uint32_t *gh = ghist + r * kBins;
            for (int i = tid; i < (int)nb; i += kClThreads) {
                const uint32_t h = hist[i];
                if (h) { atomicAdd(gh + i, h); hist[i] = 0u; }
            }
            cluster.sync();                                      // the query's histogram is complete
            // digit d with count(> d) < k_rem <= count(>= d); bins from the top, 4 per thread
            uint32_t c[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int b = kBins - 1 - tid * 4 - j;
                c[j] = b < (int)nb ? __ldcg(gh + b) : 0u;
            }
            if (tid == 0) { s_digit = 0; s_above = 0; }
            const uint32_t mine = c[0] + c[1] + c[2] + c[3];
            const uint32_t before = scan512(mine, s_warp, nullptr);
            const uint32_t need = (uint32_t)k_rem;
            if (before < need && need <= before + mine) {
                uint32_t acc = before;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (need <= acc + c[j]) { s_digit = kBins - 1 - tid * 4 - j; s_above = acc; break; }
                    acc += c[j];
                }
            }
            __syncthreads();
            prefix = (prefix << (r == 2 ? 10 : 11)) | s_digit;
            k_rem -= (int32_t)s_above;
        }
    }

    // ---- ordered compaction: keys > T, then the lowest-position keys == T.
    // Warp w owns a contiguous segment of this CTA's keys and walks it 32 keys
    // at a time with ballots: one pass counts, the other writes.  Output slot
    // of a chosen key = (keys > T before it) + min(keys == T before it, k_rem).
    const uint32_t T = prefix;
    const int lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kClThreads / 32;
    const int seg = (((len + kWarps - 1) / kWarps) + 31) & ~31;
    const int s0 = min(len, warp * seg), s1 = min(len, s0 + seg);
    __shared__ uint32_t s_wgt[kWarps], s_weq[kWarps], s_base[2];
    uint32_t wgt = 0, weq = 0;
#pragma unroll 4
    for (int b = s0; b < s1; b += 32) {
        const int i = b + lane;
        const uint32_t key = i < s1 ? s_keys[i] : 0u;
        wgt += __popc(__ballot_sync(0xffffffffu, i < s1 && (all || key > T)));
        weq += __popc(__ballot_sync(0xffffffffu, i < s1 && !all && key == T));
    }
    if (lane == 0) { s_wgt[warp] = wgt; s_weq[warp] = weq; }
    __syncthreads();
    if (tid == 0) {
        uint32_t g = 0, e = 0;
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t a = s_wgt[w], c = s_weq[w];
            s_wgt[w] = g; s_weq[w] = e;            // exclusive prefixes within the CTA
            g += a; e += c;
        }
        gcnt[2 * rank] = g;
        gcnt[2 * rank + 1] = e;
    }
    cluster.sync();                                              // every CTA's counts are out
    if (tid == 0) {
        uint32_t g = 0, e = 0;
        for (int rr = 0; rr < rank; ++rr) { g += __ldcg(gcnt + 2 * rr); e += __ldcg(gcnt + 2 * rr + 1); }
        s_base[0] = g; s_base[1] = e;
    }
    __syncthreads();
    uint32_t g = s_base[0] + s_wgt[warp], e = s_base[1] + s_weq[warp];
    const uint32_t kr = all ? 0u : (uint32_t)k_rem;
    const uint32_t lt = (1u << lane) - 1u;
    int32_t *out = p.idx_out + (int64_t)q * p.ld_idx;
    const int32_t *pb = p.pool_blk ? p.pool_blk + (int64_t)q * p.pool_blocks : nullptr;
#pragma unroll 4
    for (int b = s0; b < s1; b += 32) {
        const int i = b + lane;
        const uint32_t key = i < s1 ? s_keys[i] : 0u;
        const bool is_gt = i < s1 && (all || key > T);
        const bool is_eq = i < s1 && !all && key == T;
        const uint32_t mg = __ballot_sync(0xffffffffu, is_gt);
        const uint32_t me = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t my_g = g + __popc(mg & lt), my_e = e + __popc(me & lt);
        uint32_t slot = 0xffffffffu;
        if (is_gt) slot = my_g + min(my_e, kr);
        else if (is_eq && my_e < kr) slot = my_g + my_e;
        if (slot < (uint32_t)p.k) {
            const int64_t ii = lo + i;
            out[slot] = pb ? 8 * pb[ii >> 3] + (int32_t)(ii & 7) : (int32_t)ii;
        }
        g += __popc(mg);
        e += __popc(me);
    }
}

// ---------------------------------------------------------------- decode: one cluster per query
// For a decode layer whose indexer counted the histogram of the top 11 key bits
// (hist0), with up to kSelMaxN candidates: one cluster of C CTAs (1024 threads
// each) per query, every CTA a contiguous slice of the score row (read from
// L2, where the indexer left it) and each of its warps a contiguous segment of
// the slice, all of whose 16-byte loads are in flight together.  From hist0
// every CTA knows the bin d0 (top 11 bits) that holds the k-th key, with fewer
// than k keys above it.  One pass marks the keys above bin d0 in a bitmap of
// the slice and lists the keys in bin d0 (the candidates), counted by their
// next 11 bits; the cluster's summed counts give the 22-bit bin m1 of the
// k-th key.  Candidates above m1 join the bitmap.  The few keys inside m1 are
// copied to every CTA of the cluster, so that each finds the exact k-th key T
// and its own place in the output by itself: keys above T are all taken, and
// of the keys equal to T the lowest positions (slices in order).  Each CTA
// writes the set bits of its bitmap, ascending, at its offset in the output.
// When bin m1 is too full to copy (heavy ties), the last 10 bits are counted
// over the cluster as well, which costs one more cluster barrier.  Order never
// depends on the candidate list, so a slice whose candidates overflow the list
// re-reads them from the score row.
constexpr int kSelThreads = 1024;
constexpr int kSelSlice = 16384;                       // positions per CTA, nominal
constexpr int kSelMaxSlice = 32768;                    // bitmap words: 1024 (one per thread)
constexpr int kSelMaxCtas = 8;
constexpr int kSelCand = 4096;                         // candidates listed per CTA
constexpr int kSelWarpCand = kSelCand / (kSelThreads / 32);   // 128 per warp
constexpr int kSelCopy = 4096;                         // keys of bin m1 copied to a CTA, all slices
constexpr int kSelLoads = 5;                           // 16-byte loads per lane and step
constexpr int kSelStep = 128 * kSelLoads;              // positions per warp and step
constexpr int64_t kSelMaxN = (int64_t)kSelMaxSlice * kSelMaxCtas;   // 262,144

// Block-wide exclusive scan of one 32-bit value per thread (1024 threads).
__device__ __forceinline__ uint32_t scan_sel(uint32_t v, uint32_t *s_warp, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;                                  // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before = warp > 0 ? s_warp[warp - 1] : 0u;
    if (total) *total = s_warp[31];
    __syncthreads();
    return before + x - v;
}

// Digit of a round: bins `nb` (descending from nb - 1), counts in h; the digit
// d has count(> d) < need <= count(>= d).  Every thread returns d and count(> d).
__device__ __forceinline__ void pick_digit(const uint32_t *h, int nb, uint32_t need,
                                           uint32_t *s_warp, uint32_t *s_res, uint32_t &d,
                                           uint32_t &above)
{
    const int per = (nb + kSelThreads - 1) / kSelThreads;    // 1 or 2
    uint32_t c[2] = {0u, 0u}, mine = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int b = nb - 1 - (threadIdx.x * per + i);
        if (i < per && b >= 0) c[i] = h[b];
        mine += c[i];
    }
    if (threadIdx.x == 0) { s_res[0] = 0u; s_res[1] = 0u; }
    const uint32_t before = scan_sel(mine, s_warp, nullptr);
    if (before < need && need <= before + mine) {
        uint32_t acc = before;
        for (int i = 0; i < per; ++i) {
            if (need <= acc + c[i]) {
                s_res[0] = (uint32_t)(nb - 1 - (threadIdx.x * per + i));
                s_res[1] = acc;
                break;
            }
            acc += c[i];
        }
    }
    __syncthreads();
    d = s_res[0];
    above = s_res[1];
    __syncthreads();
}

struct SelShared {
    uint32_t bits[kSelMaxSlice / 32];      // taken positions of the slice
    uint32_t ties[kSelMaxSlice / 32];      // positions of the slice whose key equals T
    uint32_t h1[2048];                     // bin-d0 keys of the slice by bits 10..20 (read by the cluster)
    uint32_t h2[1024];                     // bin-m1 keys of the slice by bits 0..9 (read by the cluster)
    uint32_t hs[2048];                     // counts summed over the cluster
    uint32_t cand_key[kSelCand];
    int32_t cand_pos[kSelCand];            // (positions relative to the slice)
    uint32_t copy_key[kSelCopy];           // keys of bin m1: source slice r at [r * cap, ..)  (peers write)
    uint32_t pub[3][kSelMaxCtas];          // per source slice (peers write): taken so far, keys in m1, ties
    uint32_t stat[2][kSelMaxCtas];         // per source slice: copied keys above T, equal to T
    uint32_t cnt[4];                       // list overflow, keys in m1, ties
    uint32_t wcnt[kSelThreads / 32];       // candidates found by each warp
    uint32_t s_warp[kSelThreads / 32];
    uint32_t s_res[2];
};

__global__ void __launch_bounds__(kSelThreads, 1) topk_select_kernel(TopkParams p, int slice)
{
    pdl_wait();
    pdl_trigger();
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
    extern __shared__ __align__(16) uint8_t sel_smem[];
    SelShared &sh = *reinterpret_cast<SelShared *>(sel_smem);
    const int q = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int n = p.n_valid[q];
    if (p.n_div8) n = (n + 7) / 8;
    if (n < 0) n = 0;
    if (n > p.max_n) n = (int)p.max_n;
    const float *row = p.scores + (int64_t)q * p.ld;
    int32_t *out = p.idx_out + (int64_t)q * p.ld_idx;
    const int32_t *pb = p.pool_blk ? p.pool_blk + (int64_t)q * p.pool_blocks : nullptr;
    auto pos_of = [&](int i) { return pb ? 8 * __ldg(pb + (i >> 3)) + (i & 7) : i; };
    if (n <= p.k) {                                          // (the same for the whole cluster)
        if (rank == 0) {
            for (int i = tid; i < n; i += kSelThreads) out[i] = pos_of(i);
            if (tid == 0) p.cnt_out[q] = n;
        }
        return;
    }
    if (rank == 0 && tid == 0) p.cnt_out[q] = p.k;
    const int lo = min(n, rank * slice), hi = min(n, lo + slice);
    const int nwords = (hi - lo + 31) >> 5;
    const int wseg = slice / 32;                             // a multiple of 128
    const int s0 = min(hi, lo + warp * wseg), s1 = min(hi, s0 + wseg);

    // a step's loads: lane l of load u holds positions st + 128 u + 4 l .. + 3
    float4 f[kSelLoads];
    auto load_step = [&](int st) {
#pragma unroll
        for (int u = 0; u < kSelLoads; ++u) {
            const int i0 = st + 128 * u + 4 * lane;
            if (i0 + 4 <= s1) {
                f[u] = __ldcg(reinterpret_cast<const float4 *>(row + i0));
            } else {
                f[u].x = i0 < s1 ? __ldcg(row + i0) : 0.f;
                f[u].y = i0 + 1 < s1 ? __ldcg(row + i0 + 1) : 0.f;
                f[u].z = i0 + 2 < s1 ? __ldcg(row + i0 + 2) : 0.f;
                f[u].w = 0.f;
            }
        }
    };
    if (s0 < s1) load_step(s0);                              // in flight while d0 is found

    for (int i = tid; i < kSelMaxSlice / 32; i += kSelThreads) { sh.bits[i] = 0u; sh.ties[i] = 0u; }
    for (int i = tid; i < 2048; i += kSelThreads) {
        sh.h1[i] = 0u;
        sh.hs[i] = __ldcg(p.hist0 + (int64_t)q * kBins + i);
    }
    for (int i = tid; i < 1024; i += kSelThreads) sh.h2[i] = 0u;
    if (tid < 2 * kSelMaxCtas) (&sh.stat[0][0])[tid] = 0u;
    if (tid < 4) sh.cnt[tid] = 0u;
    __syncthreads();
    uint32_t d0, above0;
    pick_digit(sh.hs, kBins, (uint32_t)p.k, sh.s_warp, sh.s_res, d0, above0);
    uint32_t k_rem = (uint32_t)p.k - above0;

    // ---- the pass: keys above bin d0 into the bitmap, keys in bin d0 listed
    // (each warp in its own region) and counted by bits 10..20
    uint32_t wc = 0;                                         // this warp's candidates
    for (int st = s0; st < s1; st += kSelStep) {
        if (st != s0) load_step(st);
#pragma unroll
        for (int u = 0; u < kSelLoads; ++u) {
            const int i0 = st + 128 * u + 4 * lane;
            const uint32_t kk[4] = {score_key(f[u].x), score_key(f[u].y), score_key(f[u].z),
                                    score_key(f[u].w)};
            uint32_t fa = 0, fb = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool in = i0 + j < s1;
                const uint32_t b = kk[j] >> 21;
                fa |= (uint32_t)(in && b > d0) << j;
                fb |= (uint32_t)(in && b == d0) << j;
            }
            // bitmap word (i0 - lo) / 32: the nibbles of 8 lanes
            uint32_t wbits = fa << (4 * (lane & 7));
            wbits |= __shfl_xor_sync(0xffffffffu, wbits, 1);
            wbits |= __shfl_xor_sync(0xffffffffu, wbits, 2);
            wbits |= __shfl_xor_sync(0xffffffffu, wbits, 4);
            if ((lane & 7) == 0 && i0 < s1 && wbits) sh.bits[(i0 - lo) >> 5] = wbits;
            // candidates: slots of this warp's region of the list, in lane order
            const uint32_t b0 = __ballot_sync(0xffffffffu, fb & 1u), b1 = __ballot_sync(0xffffffffu, fb & 2u);
            const uint32_t b2 = __ballot_sync(0xffffffffu, fb & 4u), b3 = __ballot_sync(0xffffffffu, fb & 8u);
            if (b0 | b1 | b2 | b3) {
                const uint32_t lt = (1u << lane) - 1u;
                uint32_t slot = wc + __popc(b0 & lt) + __popc(b1 & lt) + __popc(b2 & lt) + __popc(b3 & lt);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (fb & (1u << j)) {
                        atomicAdd(&sh.h1[(kk[j] >> 10) & 2047u], 1u);
                        if (slot < (uint32_t)kSelWarpCand) {
                            sh.cand_key[warp * kSelWarpCand + slot] = kk[j];
                            sh.cand_pos[warp * kSelWarpCand + slot] = i0 + j - lo;
                        }
                        ++slot;
                    }
                }
                wc += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
            }
        }
    }
    if (lane == 0) {
        sh.wcnt[warp] = wc;
        if (wc > (uint32_t)kSelWarpCand) sh.cnt[0] = 1u;     // a region overflowed
    }
    __syncthreads();
    const bool listed = sh.cnt[0] == 0u;
    // this slice's candidates, from the list or (overflow) from the score row
    auto for_cand = [&](auto &&fn) {
        if (listed) {
            for (int c = tid; c < kSelCand; c += kSelThreads)
                if ((c & (kSelWarpCand - 1)) < (int)sh.wcnt[c / kSelWarpCand]) fn(sh.cand_key[c], sh.cand_pos[c]);
        } else {
            for (int i = lo + tid; i < hi; i += kSelThreads) {
                const uint32_t key = score_key(__ldcg(row + i));
                if ((key >> 21) == d0) fn(key, i - lo);
            }
        }
    };
    // the sum over the cluster of a per-slice count table (all loads in flight together)
    auto cluster_sum = [&](const uint32_t *tab, int i) {
        uint32_t v[kSelMaxCtas];
#pragma unroll
        for (int r = 0; r < kSelMaxCtas; ++r) v[r] = r < C ? cluster.map_shared_rank(tab, r)[i] : 0u;
        return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    };
    cluster.sync();                                          // every slice's h1 is complete

    // ---- bin m1 from the cluster's counts
    const uint32_t g0 = cluster_sum(sh.h1, tid), g1 = cluster_sum(sh.h1, tid + 1024);
    sh.hs[tid] = g0;                                         // (pick_digit above has finished with hs)
    sh.hs[tid + 1024] = g1;
    __syncthreads();
    uint32_t d1, above1;
    pick_digit(sh.hs, 2048, k_rem, sh.s_warp, sh.s_res, d1, above1);
    k_rem -= above1;
    const uint32_t m1 = (d0 << 11) | d1;
    const int cap = kSelCopy / C;                            // copied keys per source slice
    const bool copy = sh.hs[d1] <= (uint32_t)cap;            // the same in every CTA
    // candidates above m1 join the bitmap; those in m1 are copied to every CTA
    // (or, heavy ties, counted by their last 10 bits)
    for_cand([&](uint32_t key, int rp) {
        const uint32_t b = key >> 10;
        if (b > m1) {
            atomicOr(&sh.bits[rp >> 5], 1u << (rp & 31));
        } else if (b == m1) {
            if (copy) {
                const uint32_t slot = atomicAdd(&sh.cnt[1], 1u);
                if (slot < (uint32_t)cap)
                    for (int r = 0; r < C; ++r) cluster.map_shared_rank(sh.copy_key, r)[rank * cap + slot] = key;
            } else {
                atomicAdd(&sh.h2[key & 1023u], 1u);
            }
        }
    });
    __syncthreads();
    uint32_t T, out_base = 0, my_take = 0;
    if (copy) {
        uint32_t n_taken;
        scan_sel(tid < nwords ? __popc(sh.bits[tid]) : 0u, sh.s_warp, &n_taken);
        if (tid < C) {
            uint32_t *t = cluster.map_shared_rank(&sh.pub[0][0], tid);
            t[rank] = n_taken;                               // pub[0][rank]
            t[kSelMaxCtas + rank] = sh.cnt[1];               // pub[1][rank]
        }
        cluster.sync();                                      // every slice's keys of m1 and counts are here
        // T from the copied keys; per source slice, those above and equal to T
        for (int i = tid; i < 1024; i += kSelThreads) sh.hs[i] = 0u;
        __syncthreads();
        for (int e = tid; e < C * cap; e += kSelThreads) {
            const int r = e / cap;
            if (e - r * cap < (int)sh.pub[1][r]) atomicAdd(&sh.hs[sh.copy_key[e] & 1023u], 1u);
        }
        __syncthreads();
        uint32_t d2, above2;
        pick_digit(sh.hs, 1024, k_rem, sh.s_warp, sh.s_res, d2, above2);
        k_rem -= above2;
        T = (m1 << 10) | d2;
        for (int e = tid; e < C * cap; e += kSelThreads) {
            const int r = e / cap;
            if (e - r * cap < (int)sh.pub[1][r]) {
                const uint32_t key = sh.copy_key[e];
                if (key > T) atomicAdd(&sh.stat[0][r], 1u);
                else if (key == T) atomicAdd(&sh.stat[1][r], 1u);
            }
        }
        __syncthreads();
        // this slice's keys above T and ties
        for_cand([&](uint32_t key, int rp) {
            if (key > T) atomicOr(&sh.bits[rp >> 5], 1u << (rp & 31));
            else if (key == T) atomicOr(&sh.ties[rp >> 5], 1u << (rp & 31));
        });
        // ties are taken slice by slice in position order
        uint32_t eq_acc = 0;
        for (int r = 0; r < C; ++r) {
            const uint32_t eq_r = sh.stat[1][r];
            const uint32_t take_r = min(eq_r, k_rem > eq_acc ? k_rem - eq_acc : 0u);
            if (r < rank) out_base += sh.pub[0][r] + sh.stat[0][r] + take_r;
            if (r == rank) my_take = take_r;
            eq_acc += eq_r;
        }
    } else {
        cluster.sync();                                      // every slice's h2 is complete
        sh.hs[tid] = cluster_sum(sh.h2, tid);
        __syncthreads();
        uint32_t d2, above2;
        pick_digit(sh.hs, 1024, k_rem, sh.s_warp, sh.s_res, d2, above2);
        k_rem -= above2;
        T = (m1 << 10) | d2;
        for_cand([&](uint32_t key, int rp) {
            if ((key >> 10) == m1) {
                if (key > T) {
                    atomicOr(&sh.bits[rp >> 5], 1u << (rp & 31));
                } else if (key == T) {
                    atomicOr(&sh.ties[rp >> 5], 1u << (rp & 31));
                    atomicAdd(&sh.cnt[2], 1u);
                }
            }
        });
        __syncthreads();
        uint32_t n_taken;
        scan_sel(tid < nwords ? __popc(sh.bits[tid]) : 0u, sh.s_warp, &n_taken);
        if (tid < C) {
            uint32_t *t = cluster.map_shared_rank(&sh.pub[0][0], tid);
            t[rank] = n_taken;                               // pub[0][rank]
            t[2 * kSelMaxCtas + rank] = sh.cnt[2];           // pub[2][rank]
        }
        cluster.sync();                                      // every slice's counts are here
        uint32_t eq_acc = 0;
        for (int r = 0; r < C; ++r) {
            const uint32_t eq_r = sh.pub[2][r];
            const uint32_t take_r = min(eq_r, k_rem > eq_acc ? k_rem - eq_acc : 0u);
            if (r < rank) out_base += sh.pub[0][r] + take_r;
            if (r == rank) my_take = take_r;
            eq_acc += eq_r;
        }
    }
    // (no shared memory of a peer is touched past the last cluster barrier)
    __syncthreads();
    // this slice's first my_take ties join its taken positions, which are
    // written ascending from out_base
    const uint32_t wt = tid < nwords ? sh.ties[tid] : 0u;
    const uint32_t tb = scan_sel(__popc(wt), sh.s_warp, nullptr);
    uint32_t w = tid < nwords ? sh.bits[tid] : 0u;
    if (tb < my_take) {
        uint32_t need = my_take - tb, x = wt;
        while (x && need) {
            const uint32_t lowbit = x & (~x + 1u);
            w |= lowbit;
            x ^= lowbit;
            --need;
        }
    }
    uint32_t o = out_base + scan_sel(__popc(w), sh.s_warp, nullptr);
    while (w) {
        const int b = __ffs(w) - 1;
        w &= w - 1u;
        if (o < (uint32_t)p.k) out[o] = pos_of(lo + 32 * tid + b);
        ++o;
    }
}

// Pool size: 8 per chosen block, minus the invisible tail of the newest block
// when it is partial and was chosen.
__global__ void pool_count_kernel(const int32_t *n_valid, const int32_t *pool_blk, int pool_blocks,
                                  const int32_t *cnt, int32_t *pool_n, int nq)
{
    pdl_wait();
    pdl_trigger();
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= nq) return;
    const int n = n_valid[q];
    const int c = cnt[q];
    int pn = 8 * c;
    if (c > 0) {
        const int last = pool_blk[(int64_t)q * pool_blocks + c - 1];
        const int end = 8 * last + 8;
        if (end > n) pn -= end - n;
    }
    pool_n[q] = pn;
}

// ---------------------------------------------------------------- host side
size_t topk_workspace_bytes(int nq, int64_t max_n)
{
    int64_t n_chunks = (max_n + kChunk - 1) / kChunk;
    if (n_chunks < kClusterCtas) n_chunks = kClusterCtas;      // the cluster path's per-CTA counts
    size_t s = align_up((size_t)3 * nq * kBins * 4, 256);
    s += align_up((size_t)nq * sizeof(TopkState), 256);
    s += align_up((size_t)nq * n_chunks * 8, 256) * 2;
    return s;
}

cudaError_t launch_topk(const float *scores, int64_t ld, const int32_t *n_valid, int n_div8,
                        const int32_t *pool_blk, int pool_blocks, int nq, int64_t max_n, int k,
                        int32_t *idx_out, int64_t ld_idx, int32_t *cnt_out, void *ws,
                        const uint32_t *hist0, cudaStream_t st)
{
    TopkParams p{};
    p.hist0 = hist0;
    p.scores = scores;
    p.ld = ld;
    p.n_valid = n_valid;
    p.n_div8 = n_div8;
    p.pool_blk = pool_blk;
    p.pool_blocks = pool_blocks;
    p.nq = nq;
    p.k = k;
    p.max_n = max_n;
    p.n_chunks = (int)((max_n + kChunk - 1) / kChunk);
    if (p.n_chunks < 1) p.n_chunks = 1;
    const int64_t ws_chunks = p.n_chunks < kClusterCtas ? kClusterCtas : p.n_chunks;
    p.idx_out = idx_out;
    p.ld_idx = ld_idx;
    p.cnt_out = cnt_out;
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.hist = reinterpret_cast<uint32_t *>(w);
    w += align_up((size_t)3 * nq * kBins * 4, 256);
    p.state = reinterpret_cast<TopkState *>(w);
    w += align_up((size_t)nq * sizeof(TopkState), 256);
    p.ccount = reinterpret_cast<uint32_t *>(w);
    w += align_up((size_t)nq * ws_chunks * 8, 256);
    p.coff = reinterpret_cast<uint32_t *>(w);

    if (hist0 != nullptr && topk_select_fits(max_n, k)) {
        // C CTAs per query (a power of two, at most 8, about 16K positions each),
        // each a slice of a multiple of 4,096 positions (warp segments of a
        // multiple of 128), at most 32,768 (one bitmap word per thread)
        int C = 1;
        while (C < kSelMaxCtas && (int64_t)(2 * C) * kSelSlice <= max_n) C *= 2;
        const int64_t per = (max_n + C - 1) / C;
        const int slice = (int)((per + 4095) / 4096 * 4096);
        static_assert(kSelMaxSlice / 32 <= kSelThreads, "one bitmap word per thread");
        const size_t smem = sizeof(SelShared);
        cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const cudaError_t e = launch_k(topk_select_kernel, dim3(C, nq), dim3(kSelThreads), smem, st,
                                       (unsigned)C, p, slice);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    if (max_n <= kClusterMax) {
        const int chunk = (int)(((max_n + kClusterCtas - 1) / kClusterCtas + 3) & ~3);
        const size_t smem = (size_t)chunk * 4;
        cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kClChunkMax * 4));
        // the cluster shape comes from the kernel's __cluster_dims__
        const cudaError_t e = launch_k(topk_cluster_kernel, dim3(kClusterCtas, nq), dim3(kClThreads),
                                       smem, st, 0, p);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const dim3 grid2(p.n_chunks, nq);
    cudaError_t e = launch_k(topk_init_kernel, dim3(nq), dim3(256), 0, st, 0, p);
    for (int r = 0; r < 3 && e == cudaSuccess; ++r) {
        e = launch_k(topk_hist_kernel, grid2, dim3(kTkThreads), 0, st, 0, p, r);
        if (e == cudaSuccess) e = launch_k(topk_scan_kernel, dim3(nq), dim3(kTkThreads), 0, st, 0, p, r);
    }
    if (e == cudaSuccess) e = launch_k(topk_count_kernel, grid2, dim3(kTkThreads), 0, st, 0, p);
    if (e == cudaSuccess) e = launch_k(topk_offsets_kernel, dim3(nq), dim3(kTkThreads), 0, st, 0, p);
    if (e == cudaSuccess) e = launch_k(topk_write_kernel, grid2, dim3(kTkThreads), 0, st, 0, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

bool topk_select_fits(int64_t max_n, int k) { return max_n <= kSelMaxN && k >= 1; }

cudaError_t launch_pool(const float *blockmax, int64_t ld_bm, const int32_t *n_valid, int nq,
                        int64_t max_n, int pool_blocks, int32_t *pool_blk, int32_t *pool_n,
                        void *ws, cudaStream_t st)
{
    // the counts of chosen blocks go to pool_n first, then become positions
    const int64_t max_blocks = (max_n + 7) / 8;
    cudaError_t e = launch_topk(blockmax, ld_bm, n_valid, 1, nullptr, 0, nq, max_blocks,
                                pool_blocks, pool_blk, pool_blocks, pool_n, ws, nullptr, st);
    if (e != cudaSuccess) return e;
    e = launch_k(pool_count_kernel, dim3((nq + 127) / 128), dim3(128), 0, st, 0,
                 (const int32_t *)n_valid, (const int32_t *)pool_blk, pool_blocks,
                 (const int32_t *)pool_n, pool_n, nq);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa2

// ---------------------------------------------------------------- allocation-free top-k
// csa2_topk_noalloc keeps its scratch in a fixed array of device global memory
// that lives as long as the library is loaded.  In host code the array's name
// is only a stand-in, never a device address: the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
namespace csa2 {

constexpr size_t kNoallocScratchBytes = 4u << 20;   // 4 MiB
static __device__ __align__(256) uint8_t g_topk_scratch[kNoallocScratchBytes];

static std::mutex g_scratch_mu;
static void *g_scratch_addr[64] = {nullptr};

// Device address of the scratch array on the current device; the first call
// on a device looks it up.  nullptr if the lookup fails.
static void *noalloc_scratch()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_topk_scratch) != cudaSuccess || ptr == nullptr)
            return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace csa2

extern "C" size_t csa2_topk_noalloc_max_scratch(void) { return csa2::kNoallocScratchBytes; }

extern "C" csa2_status csa2_topk_noalloc(const float *scores, int64_t ld_scores,
                                         const int32_t *n_valid, const int32_t *pool_blk,
                                         int32_t pool_blocks, int32_t nq, int64_t max_n, int32_t k,
                                         int32_t *idx_out, int64_t ld_idx, int32_t *cnt_out,
                                         void *stream)
{
    using namespace csa2;
    auto al = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    if (nq < 0) return CSA2_ERR_INVALID_ARG;
    if (nq == 0) return CSA2_OK;
    if (!scores || !n_valid || !idx_out || !cnt_out) return CSA2_ERR_INVALID_ARG;
    if (!al(scores, 16) || !al(n_valid, 4) || !al(idx_out, 4) || !al(cnt_out, 4) ||
        (pool_blk && !al(pool_blk, 4)))
        return CSA2_ERR_ALIGN;
    if (k < 1 || max_n < 1 || max_n >= (1LL << 31) || ld_scores < max_n || ld_scores % 4 != 0 ||
        ld_idx < k)
        return CSA2_ERR_INVALID_ARG;
    if (pool_blk && (pool_blocks < 1 || max_n > 8LL * pool_blocks)) return CSA2_ERR_INVALID_ARG;
    if (topk_workspace_bytes(nq, max_n) > kNoallocScratchBytes) return CSA2_ERR_CAPACITY;
    void *scratch = noalloc_scratch();
    if (scratch == nullptr) return CSA2_ERR_CUDA;
    // launch_topk's first kernel clears the histograms and state it reads later
    const cudaError_t e = launch_topk(scores, ld_scores, n_valid, 0, pool_blk, pool_blocks, nq,
                                      max_n, k, idx_out, ld_idx, cnt_out, scratch, nullptr,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}
