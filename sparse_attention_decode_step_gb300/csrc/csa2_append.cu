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

// Entry e of sequence b (warp = b * n_ent + e), one 16-channel group per lane.
__device__ __forceinline__ void append_entry(const csa2_cache &cache, const float *__restrict__ C,
                                             const float *__restrict__ Z,
                                             const float *__restrict__ key, int n_tok, int n_ent,
                                             uint32_t *counters, int64_t warp, int lane)
{
    if (warp >= (int64_t)cache.batch * n_ent) return;
    const int b = (int)(warp / n_ent), e = (int)(warp % n_ent);
    const int64_t base = cache.seq_base[b];
    const int64_t room = cache.seq_base[b + 1] - base;
    const int64_t len = cache.seq_len[b];
    if (len + n_ent > room || len < 0) {
        if (e == 0 && lane == 0) count_event(counters, CSA2_CNT_CAPACITY);
        return;
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
    if (amax > 0.f) {
        bool sat = false;
        sb = fp4_scale_byte(amax, &sat);
        if (sat) count_event(counters, CSA2_CNT_FP4_SATURATED);
        const float s = e4m3_pos_value(sb);
#pragma unroll
        for (int c = 0; c < 16; ++c) packed[c >> 3] |= fp4_code(x[c], s) << (4 * (c & 7));
    }
    *reinterpret_cast<uint2 *>(cache.codes + row * CSA2_CODE_BYTES + lane * 8) =
        make_uint2(packed[0], packed[1]);
    cache.scales[row * CSA2_SCALE_BYTES + lane] = (uint8_t)sb;

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
