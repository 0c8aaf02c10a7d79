// csa2_append.cu -- FP4 append of new main-KV entries and their FP8 indexer keys.
//
// [Notes] section 1 (C_l, Z_l projected per layer), section 2 (sequence-block
// compression by m: disjoint blocks, no absolute positional embedding) and
// section 4 (E2M1 values with one E4M3 scale per 16 channels, range 2688).
//
// One warp per new entry; lane l owns the 16-channel group 16l..16l+15, so a
// group's amax, scale and codes never leave the lane.  Loads are 64 B per lane
// (warp-contiguous 2 KB per token), stores are 8 B of codes and 1 B of scale
// per lane.  The encode is division-free and exact: the scale is the smallest
// E4M3 s with 6 s >= amax (found by bisection over the E4M3 bytes), and each
// code is chosen by comparing |x| with the exact midpoints m_k * s.
#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

// Smallest positive E4M3 byte b with 6 * value(b) >= amax (amax > 0); 0x7E and
// *sat when even 6 * 448 is too small.
__device__ __forceinline__ uint32_t fp4_scale_byte(float amax, bool *sat)
{
    if (6.0f * 448.0f < amax) { *sat = true; return 0x7Eu; }
    uint32_t lo = 0, hi = 0x7E;       // value(hi) * 6 >= amax, value(lo) * 6 < amax (lo = 0 -> 0)
    while (hi - lo > 1) {
        uint32_t mid = (lo + hi) >> 1;
        if (6.0f * e4m3_pos_value(mid) >= amax) hi = mid; else lo = mid;
    }
    return hi;
}

// E2M1 code of x under scale s: round to nearest, ties to the even code.
// Midpoints between magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} are {.25, .75,
// 1.25, 1.75, 2.5, 3.5, 5}; at a tie with midpoint k the result goes up when
// code k + 1 is even (k odd).  Every m_k * s is exact in fp32.
__device__ __forceinline__ uint32_t fp4_code(float x, float s)
{
    float a = fabsf(x);
    uint32_t c = 0;
    c += (a > 0.25f * s);
    c += (a >= 0.75f * s);
    c += (a > 1.25f * s);
    c += (a >= 1.75f * s);
    c += (a > 2.5f * s);
    c += (a >= 3.5f * s);
    c += (a > 5.0f * s);
    if (c != 0 && x < 0.0f) c |= 8u;
    return c;
}

// Value of E2M1 code `code` (sign bit 3) under scale s: magnitudes 0, 0.5, 1,
// 1.5, 2, 3, 4, 6 built as fp32 bit patterns (index i >= 2: exponent
// 126 + i / 2, mantissa bit i & 1; index 1: 0.5).
__device__ __forceinline__ float fp4_value(uint32_t code, float s)
{
    const uint32_t i = code & 7u;
    const uint32_t bits = (i >= 2u) ? (((126u + (i >> 1)) << 23) | ((i & 1u) << 22))
                                    : (i == 1u ? (126u << 23) : 0u);
    const float v = __uint_as_float(bits) * s;
    return (code & 8u) ? -v : v;
}

// FP4 part of entry e of sequence b (warp = b * n_ent + e), one 16-channel
// group per lane: block compression, encode, store of codes and scale.
// Returns the cache row, or -1 when the entry is not stored (past the batch,
// or the sequence has no room).  kDequant: v = the stored values of this
// lane's channels 16 lane .. 16 lane + 15 (code value x scale, exact in fp32).
template <bool kDequant>
__device__ __forceinline__ int64_t append_fp4(const csa2_cache &cache, const float *__restrict__ C,
                                              const float *__restrict__ Z, int n_tok, int n_ent,
                                              uint32_t *counters, int64_t warp, int lane,
                                              float (&v)[16])
{
    if (warp >= (int64_t)cache.batch * n_ent) return -1;
    const int b = (int)(warp / n_ent), e = (int)(warp % n_ent);
    const int64_t base = cache.seq_base[b];
    const int64_t room = cache.seq_base[b + 1] - base;
    const int64_t len = cache.seq_len[b];
    if (len + n_ent > room || len < 0) {
        if (e == 0 && lane == 0) count_event(counters, CSA2_CNT_CAPACITY);
        return -1;
    }
    const int64_t row = base + len + e;
    const int m = cache.m;

    // ---- block compression of this lane's 16 channels
    float x[16];
    const int64_t tok0 = (int64_t)b * n_tok + (int64_t)e * m;
    const float4 *c4 = reinterpret_cast<const float4 *>(C + tok0 * CSA2_D + lane * 16);
    if (m == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 v = __ldg(c4 + i);
            x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
        }
    } else {
        const float4 *z4 = reinterpret_cast<const float4 *>(Z + tok0 * CSA2_D + lane * 16);
        float zmax[16], num[16], den[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) { zmax[c] = -INFINITY; num[c] = 0.f; den[c] = 0.f; }
        for (int t = 0; t < m; ++t) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float4 v = __ldg(z4 + t * (CSA2_D / 4) + i);
                zmax[4 * i] = fmaxf(zmax[4 * i], v.x);
                zmax[4 * i + 1] = fmaxf(zmax[4 * i + 1], v.y);
                zmax[4 * i + 2] = fmaxf(zmax[4 * i + 2], v.z);
                zmax[4 * i + 3] = fmaxf(zmax[4 * i + 3], v.w);
            }
        }
        for (int t = 0; t < m; ++t) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float4 zv = __ldg(z4 + t * (CSA2_D / 4) + i);
                float4 cv = __ldg(c4 + t * (CSA2_D / 4) + i);
                float zz[4] = {zv.x, zv.y, zv.z, zv.w}, cc[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float w = expf(zz[j] - zmax[4 * i + j]);
                    den[4 * i + j] += w;
                    num[4 * i + j] = fmaf(w, cc[j], num[4 * i + j]);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) x[c] = num[c] / den[c];
    }

    // ---- FP4: one scale byte and 16 codes
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) amax = fmaxf(amax, fabsf(x[c]));
    uint32_t sb = 0;
    uint32_t packed[2] = {0u, 0u};
    if constexpr (kDequant) {
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = 0.f;
    }
    if (amax > 0.f) {
        bool sat = false;
        sb = fp4_scale_byte(amax, &sat);
        if (sat) count_event(counters, CSA2_CNT_FP4_SATURATED);
        const float s = e4m3_pos_value(sb);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint32_t code = fp4_code(x[c], s);
            packed[c >> 3] |= code << (4 * (c & 7));
            if constexpr (kDequant) v[c] = fp4_value(code, s);
        }
    }
    *reinterpret_cast<uint2 *>(cache.codes + row * CSA2_CODE_BYTES + lane * 8) =
        make_uint2(packed[0], packed[1]);
    cache.scales[row * CSA2_SCALE_BYTES + lane] = (uint8_t)sb;
    return row;
}

// Entry e of sequence b (warp = b * n_ent + e): the FP4 entry, then the FP8
// indexer key given by the caller.
__device__ __forceinline__ void append_entry(const csa2_cache &cache, const float *__restrict__ C,
                                             const float *__restrict__ Z,
                                             const float *__restrict__ key, int n_tok, int n_ent,
                                             uint32_t *counters, int64_t warp, int lane)
{
    float unused[16];
    const int64_t row = append_fp4<false>(cache, C, Z, n_tok, n_ent, counters, warp, lane, unused);
    if (row < 0) return;
    const int b = (int)(warp / n_ent), e = (int)(warp % n_ent);

    // ---- FP8 indexer key: power-of-two scale per entry
    const float *kr = key + ((int64_t)b * n_ent + e) * cache.d_idx;
    if (cache.d_idx == 128) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(kr) + lane);
        float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float s = fp8_pow2_scale(a);
        uint32_t w = e4m3_byte(v.x / s) | (e4m3_byte(v.y / s) << 8) | (e4m3_byte(v.z / s) << 16) |
                     (e4m3_byte(v.w / s) << 24);
        *reinterpret_cast<uint32_t *>(cache.kidx + row * 128 + lane * 4) = w;
        if (lane == 0) cache.kscale[row] = s;
    } else {  // 64
        float2 v = __ldg(reinterpret_cast<const float2 *>(kr) + lane);
        float a = fmaxf(fabsf(v.x), fabsf(v.y));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float s = fp8_pow2_scale(a);
        uint16_t w = (uint16_t)(e4m3_byte(v.x / s) | (e4m3_byte(v.y / s) << 8));
        *reinterpret_cast<uint16_t *>(cache.kidx + row * 64 + lane * 2) = w;
        if (lane == 0) cache.kscale[row] = s;
    }
}

__global__ void __launch_bounds__(256) append_kernel(csa2_cache cache, const float *__restrict__ C,
                                                    const float *__restrict__ Z,
                                                    const float *__restrict__ key, int n_tok,
                                                    int n_ent, uint32_t *counters)
{
    pdl_wait();
    pdl_trigger();
    append_entry(cache, C, Z, key, n_tok, n_ent, counters,
                 ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5, threadIdx.x & 31);
}

// Small appends (n_ent <= 8, e.g. one decode token): CTA b writes the entries
// of sequence b, one warp each, then advances seq_len[b] itself (same room
// test as append_entry), so no second launch is needed.
__global__ void __launch_bounds__(256) append_commit_fused_kernel(csa2_cache cache,
                                                                  const float *__restrict__ C,
                                                                  const float *__restrict__ Z,
                                                                  const float *__restrict__ key,
                                                                  int n_tok, int n_ent,
                                                                  uint32_t *counters)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    append_entry(cache, C, Z, key, n_tok, n_ent, counters,
                 (int64_t)b * n_ent + (threadIdx.x >> 5), threadIdx.x & 31);
    __syncthreads();                           // every warp has read seq_len[b] and written
    if (threadIdx.x == 0) {
        const int64_t room = cache.seq_base[b + 1] - cache.seq_base[b];
        const int64_t len = cache.seq_len[b];
        if (len >= 0 && len + n_ent <= room) cache.seq_len[b] = (int32_t)(len + n_ent);
    }
}

// Advances seq_len after every entry of the batch was written (same room test
// as append_kernel, so refused sequences stay unchanged).
__global__ void append_commit_kernel(csa2_cache cache, int n_ent)
{
    pdl_wait();
    pdl_trigger();
    for (int b = threadIdx.x; b < cache.batch; b += blockDim.x) {
        const int64_t room = cache.seq_base[b + 1] - cache.seq_base[b];
        const int64_t len = cache.seq_len[b];
        if (len >= 0 && len + n_ent <= room) cache.seq_len[b] = (int32_t)(len + n_ent);
    }
}

// Append whose FP8 indexer key is projected from the stored entry: key =
// (dequantised FP4 entry) x W_IK, W_IK bf16 [512][d_idx] (this library's
// reading of the key as a linear projection of the main KV: of the stored
// entry, so that keys can be rebuilt from the cache alone).  Each CTA copies
// W_IK into shared memory with asynchronous bulk copies that land while its
// warps compress and encode their entries; one warp per entry: the entry's
// 512 stored values go to a per-warp buffer, then lane l sums key components
// (d_idx / 32) l .. + d_idx / 32 - 1 over the channels in order (fp32 FMA).
// kFused (at most 8 entries per sequence, e.g. one decode token): CTA b
// appends sequence b's entries and advances seq_len[b] itself.
constexpr int kProjThreads = 256;
constexpr int kProjWarps = kProjThreads / 32;
constexpr uint32_t kProjChunk = 32768;     // bytes per bulk copy of W_IK

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Key components of the entry staged in vb, FP8-encoded into cache row `row`.
__device__ __forceinline__ void project_key(const csa2_cache &cache, const uint16_t *sW,
                                            const float *vb, int64_t row, int lane)
{
    if (cache.d_idx == 128) {
        float k0 = 0.f, k1 = 0.f, k2 = 0.f, k3 = 0.f;   // components 4 lane .. 4 lane + 3
#pragma unroll 2
        for (int c = 0; c < CSA2_D; c += 4) {
            const float4 x4 = *reinterpret_cast<const float4 *>(vb + c);
            const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint2 w = *reinterpret_cast<const uint2 *>(sW + (c + u) * 128 + 4 * lane);
                k0 = fmaf(xs[u], bf16_lo(w.x), k0);
                k1 = fmaf(xs[u], bf16_hi(w.x), k1);
                k2 = fmaf(xs[u], bf16_lo(w.y), k2);
                k3 = fmaf(xs[u], bf16_hi(w.y), k3);
            }
        }
        float a = fmaxf(fmaxf(fabsf(k0), fabsf(k1)), fmaxf(fabsf(k2), fabsf(k3)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float s = fp8_pow2_scale(a);
        const uint32_t w = e4m3_byte(k0 / s) | (e4m3_byte(k1 / s) << 8) | (e4m3_byte(k2 / s) << 16) |
                           (e4m3_byte(k3 / s) << 24);
        *reinterpret_cast<uint32_t *>(cache.kidx + row * 128 + lane * 4) = w;
        if (lane == 0) cache.kscale[row] = s;
    } else {                                          // 64: components 2 lane, 2 lane + 1
        float k0 = 0.f, k1 = 0.f;
#pragma unroll 2
        for (int c = 0; c < CSA2_D; c += 4) {
            const float4 x4 = *reinterpret_cast<const float4 *>(vb + c);
            const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(sW + (c + u) * 64 + 2 * lane);
                k0 = fmaf(xs[u], bf16_lo(w), k0);
                k1 = fmaf(xs[u], bf16_hi(w), k1);
            }
        }
        float a = fmaxf(fabsf(k0), fabsf(k1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float s = fp8_pow2_scale(a);
        const uint16_t w = (uint16_t)(e4m3_byte(k0 / s) | (e4m3_byte(k1 / s) << 8));
        *reinterpret_cast<uint16_t *>(cache.kidx + row * 64 + lane * 2) = w;
        if (lane == 0) cache.kscale[row] = s;
    }
}

template <bool kFused>
__global__ void __launch_bounds__(kProjThreads) append_project_kernel(
    csa2_cache cache, const float *__restrict__ C, const float *__restrict__ Z,
    const uint16_t *__restrict__ w_ik, int n_tok, int n_ent, uint32_t *counters)
{
    extern __shared__ __align__(16) uint8_t smem_proj[];
    __shared__ __align__(8) uint64_t bar_w;
    __shared__ int s_timeout;             // a warp gave up waiting for W_IK
    const int d_idx = cache.d_idx;
    const uint32_t w_bytes = (uint32_t)CSA2_D * (uint32_t)d_idx * 2u;
    uint16_t *sW = reinterpret_cast<uint16_t *>(smem_proj);                   // [512][d_idx]
    float *sVal = reinterpret_cast<float *>(smem_proj + w_bytes);             // [warps][512]
    if (threadIdx.x == 0) {
        mbar_init(&bar_w, 1);
        fence_barrier_init();
        s_timeout = 0;
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar_w, w_bytes);
        for (uint32_t off = 0; off < w_bytes; off += kProjChunk)
            bulk_load(reinterpret_cast<uint8_t *>(sW) + off,
                      reinterpret_cast<const uint8_t *>(w_ik) + off,
                      min(kProjChunk, w_bytes - off), &bar_w);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *vb = sVal + warp * CSA2_D;
    volatile int no_abort = 0;
    bool w_ready = false;
    const int64_t total = (int64_t)cache.batch * n_ent;
    const int64_t first = kFused ? (int64_t)blockIdx.x * n_ent + warp
                                 : (int64_t)blockIdx.x * kProjWarps + warp;
    const int64_t stride = kFused ? total : (int64_t)gridDim.x * kProjWarps;
    for (int64_t ent = first; ent < total && (!kFused || warp < n_ent); ent += stride) {
        float v[16];
        const int64_t row = append_fp4<true>(cache, C, Z, n_tok, n_ent, counters, ent, lane, v);
        if (row < 0) continue;                       // the same for the whole warp
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
            reinterpret_cast<float4 *>(vb + 16 * lane)[c4] =
                make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
        __syncwarp();
        if (!w_ready) {
            // W_IK has landed (bounded wait; on expiry the key is not written)
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_w, 0, &no_abort));
            if (!ok) {
                if (lane == 0) {
                    count_event(counters, CSA2_CNT_TIMEOUT);
                    s_timeout = 1;
                }
                break;
            }
            w_ready = true;
        }
        project_key(cache, sW, vb, row, lane);
        __syncwarp();                                // vb is refilled by the next entry
    }
    __syncthreads();
    // no copy of this CTA may still be landing when it exits (bounded)
    if (threadIdx.x == 0) mbar_wait(&bar_w, 0, &no_abort);
    // a sequence whose keys were not all written keeps its length (fused path;
    // the two-launch path advances every sequence with room)
    if (kFused && threadIdx.x == 0 && s_timeout == 0) {
        const int b = blockIdx.x;
        const int64_t room = cache.seq_base[b + 1] - cache.seq_base[b];
        const int64_t len = cache.seq_len[b];
        if (len >= 0 && len + n_ent <= room) cache.seq_len[b] = (int32_t)(len + n_ent);
    }
}

cudaError_t launch_append_project(const csa2_cache &c, const float *C, const float *Z,
                                  const uint16_t *w_ik, int n_tok, uint32_t *counters,
                                  cudaStream_t st)
{
    const int n_ent = n_tok / c.m;
    const size_t w_bytes = (size_t)CSA2_D * c.d_idx * 2;
    if (n_ent <= kProjWarps) {
        // one CTA per sequence, one warp per entry, seq_len advanced in the same launch
        const size_t smem = w_bytes + (size_t)n_ent * CSA2_D * 4;
        cudaFuncSetAttribute(append_project_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const cudaError_t e = launch_k(append_project_kernel<true>, dim3((unsigned)c.batch),
                                       dim3(32 * n_ent), smem, st, 0, c, C, Z, w_ik, n_tok, n_ent,
                                       counters);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int64_t warps = (int64_t)c.batch * n_ent;
    int64_t blocks = (warps + kProjWarps - 1) / kProjWarps;
    if (blocks > device_sm_count()) blocks = device_sm_count();
    if (blocks < 1) blocks = 1;
    const size_t smem = w_bytes + (size_t)kProjWarps * CSA2_D * 4;
    cudaFuncSetAttribute(append_project_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    cudaError_t e = launch_k(append_project_kernel<false>, dim3((unsigned)blocks),
                             dim3(kProjThreads), smem, st, 0, c, C, Z, w_ik, n_tok, n_ent, counters);
    if (e != cudaSuccess) return e;
    e = launch_k(append_commit_kernel, dim3(1), dim3(256), 0, st, 0, c, n_ent);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_append(const csa2_cache &c, const float *C, const float *Z, const float *key,
                          int n_tok, uint32_t *counters, cudaStream_t st)
{
    const int n_ent = n_tok / c.m;
    if (n_ent <= 8) {
        const cudaError_t e = launch_k(append_commit_fused_kernel, dim3((unsigned)c.batch),
                                       dim3(32 * n_ent), 0, st, 0, c, C, Z, key, n_tok, n_ent, counters);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int64_t warps = (int64_t)c.batch * n_ent;
    const int64_t blocks = (warps * 32 + 255) / 256;
    cudaError_t e = launch_k(append_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 0, c, C, Z,
                             key, n_tok, n_ent, counters);
    if (e != cudaSuccess) return e;
    e = launch_k(append_commit_kernel, dim3(1), dim3(256), 0, st, 0, c, n_ent);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csa2
