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

// ---------------------------------------------------------------- one CTA per query
// One CTA of 512 threads per query (rows up to kRsMaxN candidates), no
// cluster: used when a launch has enough queries to fill the GPU, or few
// enough rows that one CTA each finishes before a cluster would.  A strided
// sample of about 4,096 keys gives, by two radix rounds over the sample, a
// 22-bit threshold with about 1.5 k / stride + 16 sampled keys above it; one
// pass over the row lists every key at or above it with its position, in
// per-warp regions of the list.  That list holds the top k whenever it holds
// at least k keys; three radix rounds over the list alone give the exact k-th
// key T, the list's keys above T go to a bitmap of positions and its keys
// equal to T to a tie bitmap, of which the lowest positions are taken, and the
// set bits are written in ascending order.  With stride 1 (rows up to 4,096)
// the threshold is exact.  When the list overflows a region or holds fewer
// than k keys (heavy ties, an unlucky sample), an exact path takes over: a full
// count of the top 11 bits, a pass that marks the keys above that bin and
// lists the bin's keys, two rounds over that list (or over the row again when
// it overflows).
constexpr int kRsThreads = 512;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kRsMaxN = 262144;
constexpr int kRsWords = kRsMaxN / 32;              // 8,192 bitmap words: 512 per warp
constexpr int kRsCand = 8192;                       // list entries: 512 per warp
constexpr int kRsWarpCand = kRsCand / kRsWarps;
constexpr int kRsSample = 4096;
constexpr int kRsMinQueries = 96;
constexpr int kRsLoads = 8;                         // 16-byte loads per lane in flight

struct RsShared {
    uint32_t bits[kRsWords];      // taken positions
    uint32_t ties[kRsWords];      // positions whose key equals T
    uint32_t cand_key[kRsCand];
    int32_t cand_pos[kRsCand];
    uint32_t hist[kBins];
    uint32_t wcnt[kRsWarps];      // list entries of each warp (fast path)
    uint32_t s_warp[kRsWarps];
    uint32_t s_res[2];
    uint32_t n_cand;
    uint32_t flag;                // a warp's list region overflowed
};

// The digit d of a round over bins h[0 .. nb) (from the top): count(> d) < need
// <= count(>= d); every thread gets d and count(> d) (0, 0 when the bins hold
// fewer than need).  512 threads, 4 bins each.
__device__ __forceinline__ void rs_pick(const uint32_t *h, int nb, uint32_t need, uint32_t *s_warp,
                                        uint32_t *s_res, uint32_t &d, uint32_t &above)
{
    const int tid = threadIdx.x;
    uint32_t c[4], mine = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = nb - 1 - 4 * tid - j;
        c[j] = b >= 0 ? h[b] : 0u;
        mine += c[j];
    }
    if (tid == 0) { s_res[0] = 0u; s_res[1] = 0u; }
    const uint32_t before = scan512(mine, s_warp, nullptr);
    if (before < need && need <= before + mine) {
        uint32_t acc = before;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (need <= acc + c[j]) { s_res[0] = (uint32_t)(nb - 1 - 4 * tid - j); s_res[1] = acc; break; }
            acc += c[j];
        }
    }
    __syncthreads();
    d = s_res[0];
    above = s_res[1];
    __syncthreads();
}

// Warp-inclusive scan
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

__global__ void __launch_bounds__(kRsThreads, 1) topk_rowselect_kernel(TopkParams p)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t rs_smem[];
    RsShared &sh = *reinterpret_cast<RsShared *>(rs_smem);
    const int q = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int n = p.n_valid[q];
    if (p.n_div8) n = (n + 7) / 8;
    if (n < 0) n = 0;
    if (n > p.max_n) n = (int)p.max_n;
    const float *row = p.scores + (int64_t)q * p.ld;
    int32_t *out = p.idx_out + (int64_t)q * p.ld_idx;
    const int32_t *pb = p.pool_blk ? p.pool_blk + (int64_t)q * p.pool_blocks : nullptr;
    auto pos_of = [&](int i) { return pb ? 8 * __ldg(pb + (i >> 3)) + (i & 7) : i; };
    if (n <= p.k) {
        for (int i = tid; i < n; i += kRsThreads) out[i] = pos_of(i);
        if (tid == 0) p.cnt_out[q] = n;
        return;
    }
    if (tid == 0) p.cnt_out[q] = p.k;
    for (int i = tid; i < kRsWords; i += kRsThreads) { sh.bits[i] = 0u; sh.ties[i] = 0u; }
    for (int i = tid; i < kBins; i += kRsThreads) sh.hist[i] = 0u;
    if (tid == 0) { sh.n_cand = 0u; sh.flag = 0u; }
    // a warp's pieces of the row (below): the first one's loads go out now
    auto load_piece = [&](float4 (&f)[kRsLoads], int base) {
#pragma unroll
        for (int u = 0; u < kRsLoads; ++u) {
            const int i0 = base + 128 * u + 4 * lane;
            if (i0 + 4 <= n) {
                f[u] = __ldcg(reinterpret_cast<const float4 *>(row + i0));
            } else {
                f[u].x = i0 < n ? __ldcg(row + i0) : 0.f;
                f[u].y = i0 + 1 < n ? __ldcg(row + i0 + 1) : 0.f;
                f[u].z = i0 + 2 < n ? __ldcg(row + i0 + 2) : 0.f;
                f[u].w = 0.f;
            }
        }
    };
    constexpr int kStride = 1024 * kRsWarps;
    float4 fa[kRsLoads], fb[kRsLoads];
    if (1024 * warp < n) load_piece(fa, 1024 * warp);

    // ---- the sample: positions st * m, m < n_s (8 per thread at most)
    const int st = (n + kRsSample - 1) / kRsSample;
    const int n_s = (n + st - 1) / st;
    uint32_t smp[kRsSample / kRsThreads];
#pragma unroll
    for (int j = 0; j < kRsSample / kRsThreads; ++j) {
        const int m = tid + kRsThreads * j;
        smp[j] = m < n_s ? score_key(__ldcg(row + (int64_t)m * st)) : 0u;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRsSample / kRsThreads; ++j)
        if (tid + kRsThreads * j < n_s) atomicAdd(&sh.hist[smp[j] >> 21], 1u);
    __syncthreads();
    // keys above the threshold, counted in the sample: k exactly when the sample
    // is the row, else about 1.5 k / st + 16
    const uint32_t t_s = st == 1 ? (uint32_t)p.k : min((uint32_t)n_s, (uint32_t)((3LL * p.k) / (2LL * st)) + 16u);
    uint32_t da, above;
    rs_pick(sh.hist, kBins, t_s, sh.s_warp, sh.s_res, da, above);
    for (int i = tid; i < kBins; i += kRsThreads) sh.hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRsSample / kRsThreads; ++j)
        if (tid + kRsThreads * j < n_s && (smp[j] >> 21) == da) atomicAdd(&sh.hist[(smp[j] >> 10) & 2047u], 1u);
    __syncthreads();
    uint32_t db;
    rs_pick(sh.hist, kBins, t_s - above, sh.s_warp, sh.s_res, db, above);
    const uint32_t key_lo = (da << 21) | (db << 10);   // list: keys >= key_lo

    // ---- the list pass: warp w takes the 1,024-position pieces w, w + 16, ...
    // (lane l of load u: positions 128 u + 4 l .. + 3), the next piece's loads in
    // flight while one is processed.  A lane's 32 decisions of a piece form one
    // mask (bit 4u + j), one warp scan gives the lane its slots in the warp's
    // region, and the positions of its keys >= key_lo are stored (their keys are
    // read back from the row after the pass)
    uint32_t wc = 0;
    auto list_piece = [&](const float4 (&f)[kRsLoads], int base) {
        uint32_t mask = 0;
#pragma unroll
        for (int u = 0; u < kRsLoads; ++u) {
            const int i0 = base + 128 * u + 4 * lane;
            mask |= (uint32_t)(i0 < n && score_key(f[u].x) >= key_lo) << (4 * u);
            mask |= (uint32_t)(i0 + 1 < n && score_key(f[u].y) >= key_lo) << (4 * u + 1);
            mask |= (uint32_t)(i0 + 2 < n && score_key(f[u].z) >= key_lo) << (4 * u + 2);
            mask |= (uint32_t)(i0 + 3 < n && score_key(f[u].w) >= key_lo) << (4 * u + 3);
        }
        const uint32_t cb = __popc(mask);
        const uint32_t incl = warp_incl_scan(cb, lane);
        uint32_t slot = wc + incl - cb;
        while (mask) {
            const int bit = __ffs(mask) - 1;
            mask &= mask - 1u;
            if (slot < (uint32_t)kRsWarpCand)
                sh.cand_pos[warp * kRsWarpCand + slot] = base + 128 * (bit >> 2) + 4 * lane + (bit & 3);
            ++slot;
        }
        wc += __shfl_sync(0xffffffffu, incl, 31);
    };
    for (int base = 1024 * warp; base < n; base += 2 * kStride) {
        if (base + kStride < n) load_piece(fb, base + kStride);
        list_piece(fa, base);
        if (base + 2 * kStride < n) load_piece(fa, base + 2 * kStride);
        if (base + kStride < n) list_piece(fb, base + kStride);
    }
    // the listed keys, read back from the row (one load each, all in flight)
    for (int s2 = lane; s2 < (int)min(wc, (uint32_t)kRsWarpCand); s2 += 32)
        sh.cand_key[warp * kRsWarpCand + s2] = score_key(__ldcg(row + sh.cand_pos[warp * kRsWarpCand + s2]));
    if (lane == 0) {
        sh.wcnt[warp] = wc;
        if (wc > (uint32_t)kRsWarpCand) sh.flag = 1u;
    }
    __syncthreads();
    uint32_t c_total = 0;
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) c_total += sh.wcnt[w];
    const bool fast = sh.flag == 0u && c_total >= (uint32_t)p.k;
    uint32_t T, k_rem, d0, d1, d2;
    if (fast) {
        // ---- three radix rounds over the list alone
        auto for_list = [&](auto &&fn) {
            for (int e = tid; e < kRsCand; e += kRsThreads)
                if ((e % kRsWarpCand) < (int)sh.wcnt[e / kRsWarpCand]) fn(sh.cand_key[e], sh.cand_pos[e]);
        };
        for (int i = tid; i < kBins; i += kRsThreads) sh.hist[i] = 0u;
        __syncthreads();
        for_list([&](uint32_t key, int) { atomicAdd(&sh.hist[key >> 21], 1u); });
        __syncthreads();
        rs_pick(sh.hist, kBins, (uint32_t)p.k, sh.s_warp, sh.s_res, d0, above);
        k_rem = (uint32_t)p.k - above;
        for (int i = tid; i < kBins; i += kRsThreads) sh.hist[i] = 0u;
        __syncthreads();
        for_list([&](uint32_t key, int) {
            if ((key >> 21) == d0) atomicAdd(&sh.hist[(key >> 10) & 2047u], 1u);
        });
        __syncthreads();
        rs_pick(sh.hist, kBins, k_rem, sh.s_warp, sh.s_res, d1, above);
        k_rem -= above;
        const uint32_t m1 = (d0 << 11) | d1;
        for (int i = tid; i < 1024; i += kRsThreads) sh.hist[i] = 0u;
        __syncthreads();
        for_list([&](uint32_t key, int) {
            if ((key >> 10) == m1) atomicAdd(&sh.hist[key & 1023u], 1u);
        });
        __syncthreads();
        rs_pick(sh.hist, 1024, k_rem, sh.s_warp, sh.s_res, d2, above);
        k_rem -= above;                                  // keys equal to T that are taken
        T = (m1 << 10) | d2;
        for_list([&](uint32_t key, int pos) {
            if (key > T) atomicOr(&sh.bits[pos >> 5], 1u << (pos & 31));
            else if (key == T) atomicOr(&sh.ties[pos >> 5], 1u << (pos & 31));
        });
    } else {
        // ---- exact path.  Pass 1: count of the top 11 key bits
        for (int i = tid; i < kBins; i += kRsThreads) sh.hist[i] = 0u;
        __syncthreads();
        for (int i0 = 4 * tid; i0 < n; i0 += 4 * kRsThreads * kRsLoads) {
            float4 f[kRsLoads];
#pragma unroll
            for (int u = 0; u < kRsLoads; ++u) {
                const int i = i0 + 4 * kRsThreads * u;
                if (i + 4 <= n) f[u] = __ldcg(reinterpret_cast<const float4 *>(row + i));
            }
#pragma unroll
            for (int u = 0; u < kRsLoads; ++u) {
                const int i = i0 + 4 * kRsThreads * u;
                if (i + 4 <= n) {
                    atomicAdd(&sh.hist[score_key(f[u].x) >> 21], 1u);
                    atomicAdd(&sh.hist[score_key(f[u].y) >> 21], 1u);
                    atomicAdd(&sh.hist[score_key(f[u].z) >> 21], 1u);
                    atomicAdd(&sh.hist[score_key(f[u].w) >> 21], 1u);
                } else {
                    for (int j = i; j < n; ++j) atomicAdd(&sh.hist[score_key(__ldcg(row + j)) >> 21], 1u);
                }
            }
        }
        __syncthreads();
        rs_pick(sh.hist, kBins, (uint32_t)p.k, sh.s_warp, sh.s_res, d0, above);
        k_rem = (uint32_t)p.k - above;
        for (int i = tid; i < kBins; i += kRsThreads) sh.hist[i] = 0u;
        __syncthreads();
        // pass 2: keys above bin d0 into the bitmap (lanes 8j .. 8j + 7 make one
        // word), keys in bin d0 listed (shared slot counter) and counted by bits 10..20
        for (int base = 1024 * warp; base < n; base += 1024 * kRsWarps) {
            float4 f[kRsLoads];
#pragma unroll
            for (int u = 0; u < kRsLoads; ++u) {
                const int i0 = base + 128 * u + 4 * lane;
                if (i0 + 4 <= n) {
                    f[u] = __ldcg(reinterpret_cast<const float4 *>(row + i0));
                } else {
                    f[u].x = i0 < n ? __ldcg(row + i0) : 0.f;
                    f[u].y = i0 + 1 < n ? __ldcg(row + i0 + 1) : 0.f;
                    f[u].z = i0 + 2 < n ? __ldcg(row + i0 + 2) : 0.f;
                    f[u].w = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kRsLoads; ++u) {
                const int i0 = base + 128 * u + 4 * lane;
                const uint32_t kk[4] = {score_key(f[u].x), score_key(f[u].y), score_key(f[u].z),
                                        score_key(f[u].w)};
                uint32_t fa = 0, fb = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = i0 + j < n;
                    fa |= (uint32_t)(in && (kk[j] >> 21) > d0) << j;
                    fb |= (uint32_t)(in && (kk[j] >> 21) == d0) << j;
                }
                uint32_t wbits = fa << (4 * (lane & 7));
                wbits |= __shfl_xor_sync(0xffffffffu, wbits, 1);
                wbits |= __shfl_xor_sync(0xffffffffu, wbits, 2);
                wbits |= __shfl_xor_sync(0xffffffffu, wbits, 4);
                if ((lane & 7) == 0 && i0 < n && wbits) sh.bits[i0 >> 5] = wbits;
                if (__ballot_sync(0xffffffffu, fb != 0u)) {
                    const uint32_t cb = __popc(fb);
                    const uint32_t incl = warp_incl_scan(cb, lane);
                    uint32_t slot = 0;
                    if (lane == 31) slot = atomicAdd(&sh.n_cand, incl);
                    slot = __shfl_sync(0xffffffffu, slot, 31) + incl - cb;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (fb & (1u << j)) {
                            atomicAdd(&sh.hist[(kk[j] >> 10) & 2047u], 1u);
                            if (slot < (uint32_t)kRsCand) {
                                sh.cand_key[slot] = kk[j];
                                sh.cand_pos[slot] = i0 + j;
                            }
                            ++slot;
                        }
                    }
                }
            }
        }
        __syncthreads();
        const bool listed = sh.n_cand <= (uint32_t)kRsCand;
        const int n_cand = listed ? (int)sh.n_cand : 0;
        // the keys of bin d0, from the list or (overflow) from the row
        auto for_cand = [&](auto &&fn) {
            if (listed) {
                for (int c = tid; c < n_cand; c += kRsThreads) fn(sh.cand_key[c], sh.cand_pos[c]);
            } else {
                for (int i = tid; i < n; i += kRsThreads) {
                    const uint32_t key = score_key(__ldcg(row + i));
                    if ((key >> 21) == d0) fn(key, i);
                }
            }
        };
        rs_pick(sh.hist, kBins, k_rem, sh.s_warp, sh.s_res, d1, above);
        k_rem -= above;
        const uint32_t m1 = (d0 << 11) | d1;
        for (int i = tid; i < 1024; i += kRsThreads) sh.hist[i] = 0u;
        __syncthreads();
        for_cand([&](uint32_t key, int) {
            if ((key >> 10) == m1) atomicAdd(&sh.hist[key & 1023u], 1u);
        });
        __syncthreads();
        rs_pick(sh.hist, 1024, k_rem, sh.s_warp, sh.s_res, d2, above);
        k_rem -= above;
        T = (m1 << 10) | d2;
        for_cand([&](uint32_t key, int pos) {
            if (key > T) atomicOr(&sh.bits[pos >> 5], 1u << (pos & 31));
            else if (key == T) atomicOr(&sh.ties[pos >> 5], 1u << (pos & 31));
        });
    }
    __syncthreads();

    // ---- output.  Thread t owns bitmap words 16t .. 16t + 15 (ascending
    // positions; four 16-byte reads).  Ties are taken in position order: the
    // threads before it take theirs first.
    const int w0 = 16 * tid;
    uint32_t bw[16], tw[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 b4 = reinterpret_cast<const uint4 *>(sh.bits + w0)[v];
        const uint4 t4 = reinterpret_cast<const uint4 *>(sh.ties + w0)[v];
        bw[4 * v] = b4.x; bw[4 * v + 1] = b4.y; bw[4 * v + 2] = b4.z; bw[4 * v + 3] = b4.w;
        tw[4 * v] = t4.x; tw[4 * v + 1] = t4.y; tw[4 * v + 2] = t4.z; tw[4 * v + 3] = t4.w;
    }
    uint32_t n_tie = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) n_tie += __popc(tw[j]);
    const uint32_t ties_before = scan512(n_tie, sh.s_warp, nullptr);
    uint32_t keep = k_rem > ties_before ? min(n_tie, k_rem - ties_before) : 0u;
    uint32_t n_sel = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        uint32_t t = tw[j];
        while (t && keep) {
            const uint32_t low = t & (~t + 1u);
            bw[j] |= low;
            t ^= low;
            --keep;
        }
        n_sel += __popc(bw[j]);
    }
    uint32_t o = scan512(n_sel, sh.s_warp, nullptr);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        uint32_t x = bw[j];
        while (x) {
            const int bit = __ffs(x) - 1;
            x &= x - 1u;
            if (o < (uint32_t)p.k) out[o] = pos_of(32 * (w0 + j) + bit);
            ++o;
        }
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
                        cudaStream_t st)
{
    TopkParams p{};
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

    if (nq >= kRsMinQueries && max_n <= kRsMaxN) {
        const size_t smem = sizeof(RsShared);
        cudaFuncSetAttribute(topk_rowselect_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const cudaError_t e = launch_k(topk_rowselect_kernel, dim3(nq), dim3(kRsThreads), smem, st, 0, p);
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

cudaError_t launch_pool(const float *blockmax, int64_t ld_bm, const int32_t *n_valid, int nq,
                        int64_t max_n, int pool_blocks, int32_t *pool_blk, int32_t *pool_n,
                        void *ws, cudaStream_t st)
{
    // the counts of chosen blocks go to pool_n first, then become positions
    const int64_t max_blocks = (max_n + 7) / 8;
    cudaError_t e = launch_topk(blockmax, ld_bm, n_valid, 1, nullptr, 0, nq, max_blocks,
                                pool_blocks, pool_blk, pool_blocks, pool_n, ws, st);
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
                                      max_n, k, idx_out, ld_idx, cnt_out, scratch,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}
