// csa2_attn_simt.cu -- sparse attention over selected FP4 entries + window KV,
// CUDA-core version (also the reference the tensor-core kernel is checked
// against on the GPU).
//
// [Thread] item 4: the selected main-KV entries are concatenated with the
// windowed KV, then attended; [Deep read] section 03: each layer brings its own
// query and window; [Notes] section 4: value = E2M1 code x E4M3 scale (exact in
// fp32); [Notes] section 5: window [max(s, t - n_win + 1), t].
//
// Grid (splits, nq); each CTA runs an online softmax over a contiguous slice
// of the query's rows (32-row tiles dequantised into shared memory) and
// leaves unnormalised partials (O, running max, running sum) per head; the
// combine kernel merges the splits.
#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

constexpr int kAtThreads = 256;
constexpr int kTR = 32;          // rows per tile
constexpr int kQStride = 520;    // bf16 per smem query row (pad: conflict-free 16 B reads)

// Row set of one query: cnt selected entries, then the window positions lo..t.
struct RowSet {
    int b, cnt, nw;
    int64_t base, lo, nt;
    bool bad;
};

__device__ __forceinline__ RowSet row_set(const AttnParams &p, int q)
{
    RowSet rs;
    rs.b = p.q_seq[q];
    rs.bad = (rs.b < 0 || rs.b >= p.batch);
    if (rs.bad) {           // unknown sequence: no rows, counted by the caller
        rs.b = 0; rs.cnt = 0; rs.nw = 0; rs.base = 0; rs.lo = 0; rs.nt = 0;
        return rs;
    }
    const int64_t t = p.q_pos[q];
    rs.base = p.seq_base[rs.b];
    int64_t nt = (t + 1) / p.m;
    const int64_t len = p.seq_len[rs.b];
    if (nt > len) nt = len;
    rs.nt = nt;
    rs.cnt = (p.cnt != nullptr && p.k_max > 0) ? min(p.cnt[q], p.k_max) : 0;
    if (rs.cnt < 0) rs.cnt = 0;
    int64_t nw = 0, lo = 0;
    if (p.win != nullptr && p.n_win > 0 && t >= 0) {
        lo = t - p.n_win + 1;
        const int64_t s = p.win_start ? (int64_t)p.win_start[rs.b] : 0;
        if (lo < s) lo = s;
        if (lo < 0) lo = 0;
        nw = (t >= lo) ? t - lo + 1 : 0;
    }
    rs.lo = lo;
    rs.nw = (int)nw;
    return rs;
}

// Dequantise 64 channels (c0..c0+63) of one FP4 entry into fp32.
__device__ __forceinline__ void dequant64(const uint8_t *codes, const uint8_t *scales, int c0,
                                          float *dst)
{
    const uint4 *c4 = reinterpret_cast<const uint4 *>(codes + c0 / 2);
    const uint32_t sc4 = *reinterpret_cast<const uint32_t *>(scales + c0 / 16);
    const float lut[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 v = __ldg(c4 + h);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int cbase = h * 32 + i * 8;          // channel offset within the 64
            const float s = e4m3_pos_value((sc4 >> (8 * (cbase / 16))) & 0x7Fu);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t nib = (w[i] >> (4 * j)) & 15u;
                const float mag = lut[nib & 7u] * s;
                dst[cbase + j] = (nib & 8u) ? -mag : mag;
            }
        }
    }
}

__global__ void __launch_bounds__(kAtThreads, 1) attn_simt_kernel(AttnParams p)
{
    const int q = blockIdx.y, split = blockIdx.x;
    const int tid = threadIdx.x;
    const RowSet rs = row_set(p, q);
    const int n_rows = rs.cnt + rs.nw;
    const int r_begin = split * p.rows_per_split;
    const int r_end = min(n_rows, r_begin + p.rows_per_split);
    const int H = p.H;

    extern __shared__ __align__(16) uint8_t smem_raw[];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem_raw);            // [H][kQStride]
    float *sV = reinterpret_cast<float *>(sQ + 64 * kQStride);                  // [kTR][512]
    float *sP = sV + kTR * CSA2_D;                                              // [kTR][64]
    float *sAlpha = sP + kTR * 64;                                              // [64]
    float *sM = sAlpha + 64;                                                    // [64]
    float *sL = sM + 64;                                                        // [64]
    int *sRowOk = reinterpret_cast<int *>(sL + 64);                             // [kTR]
    int *sBad = sRowOk + kTR;

    // query rows
    const uint16_t *qg = p.q + (int64_t)q * H * CSA2_D;
    for (int i = tid; i < H * CSA2_D / 8; i += kAtThreads) {
        const int h = i / (CSA2_D / 8), c8 = i % (CSA2_D / 8);
        *reinterpret_cast<uint4 *>(sQ + h * kQStride + c8 * 8) =
            __ldg(reinterpret_cast<const uint4 *>(qg + h * CSA2_D + c8 * 8));
    }
    if (tid < 64) { sM[tid] = -INFINITY; sL[tid] = 0.f; }
    if (tid == 0) *sBad = rs.bad ? 1 : 0;

    float acc[64][2];
#pragma unroll
    for (int h = 0; h < 64; ++h) { acc[h][0] = 0.f; acc[h][1] = 0.f; }
    __syncthreads();

    const float l2scale = p.sm_scale * 1.4426950408889634f;   // logits in base 2
    for (int r0 = r_begin; r0 < r_end; r0 += kTR) {
        // ---- dequantise / copy the tile's rows (8 threads per row, 64 channels each)
        {
            const int rr = tid >> 3, c0 = (tid & 7) * 64;
            const int r = r0 + rr;
            float *dst = sV + rr * CSA2_D + c0;
            bool ok = r < r_end;
            if (ok && r < rs.cnt) {
                const int j = p.idx[(int64_t)q * p.ld_idx + r];
                if (j < 0 || j >= rs.nt) {
                    ok = false;
                    if ((tid & 7) == 0) atomicOr(sBad, 1);
                } else {
                    const int64_t row = rs.base + j;
                    dequant64(p.codes + row * CSA2_CODE_BYTES, p.scales + row * CSA2_SCALE_BYTES,
                              c0, dst);
                }
            } else if (ok) {
                const int64_t pos = rs.lo + (r - rs.cnt);
                const uint16_t *wr = p.win + ((int64_t)rs.b * p.wcap + pos % p.wcap) * CSA2_D + c0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint4 v = __ldg(reinterpret_cast<const uint4 *>(wr) + i);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        dst[i * 8 + 2 * j] = __uint_as_float(w4[j] << 16);
                        dst[i * 8 + 2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
                    }
                }
            }
            if (!ok) {
#pragma unroll
                for (int i = 0; i < 64; ++i) dst[i] = 0.f;
            }
            if ((tid & 7) == 0) sRowOk[rr] = ok ? 1 : 0;
        }
        __syncthreads();
        // ---- logits: thread = (head h = tid / 4, rows tid % 4 + 4 i)
        {
            const int h = tid >> 2, rsub = tid & 3;
            float lg[8];
            bool rok[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lg[i] = 0.f;
                rok[i] = sRowOk[rsub + 4 * i] != 0;
            }
            if (h < H) {
                const __nv_bfloat16 *qh = sQ + h * kQStride;
                for (int c = 0; c < CSA2_D; c += 8) {
                    uint4 qv = *reinterpret_cast<const uint4 *>(qh + c);
                    const uint32_t q4[4] = {qv.x, qv.y, qv.z, qv.w};
                    float qf[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        qf[2 * j] = __uint_as_float(q4[j] << 16);
                        qf[2 * j + 1] = __uint_as_float(q4[j] & 0xFFFF0000u);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 *v4 = reinterpret_cast<const float4 *>(sV + (rsub + 4 * i) * CSA2_D + c);
                        float4 a = v4[0], bq = v4[1];
                        lg[i] = fmaf(qf[0], a.x, lg[i]);
                        lg[i] = fmaf(qf[1], a.y, lg[i]);
                        lg[i] = fmaf(qf[2], a.z, lg[i]);
                        lg[i] = fmaf(qf[3], a.w, lg[i]);
                        lg[i] = fmaf(qf[4], bq.x, lg[i]);
                        lg[i] = fmaf(qf[5], bq.y, lg[i]);
                        lg[i] = fmaf(qf[6], bq.z, lg[i]);
                        lg[i] = fmaf(qf[7], bq.w, lg[i]);
                    }
                }
            }
            // online softmax per head (4 lanes share a head)
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lg[i] = rok[i] ? lg[i] * l2scale : -INFINITY;
                mx = fmaxf(mx, lg[i]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_old = (h < 64) ? sM[h] : 0.f;
            const float m_new = fmaxf(m_old, mx);
            float psum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float pv = (m_new == -INFINITY) ? 0.f : exp2f(lg[i] - m_new);
                psum += pv;
                sP[(rsub + 4 * i) * 64 + h] = pv;
            }
            psum += __shfl_xor_sync(0xffffffffu, psum, 1);
            psum += __shfl_xor_sync(0xffffffffu, psum, 2);
            __syncthreads();
            if (rsub == 0 && h < H) {
                const float alpha = (m_old == -INFINITY) ? (m_new == -INFINITY ? 1.f : 0.f)
                                                         : exp2f(m_old - m_new);
                sAlpha[h] = alpha;
                sM[h] = m_new;
                sL[h] = sL[h] * alpha + psum;
            }
        }
        __syncthreads();
        // ---- O += P V: thread owns channels 2 tid, 2 tid + 1 of every head
        {
            const int c = 2 * tid;
#pragma unroll
            for (int h = 0; h < 64; ++h) {
                if (h < H) { const float a = sAlpha[h]; acc[h][0] *= a; acc[h][1] *= a; }
            }
            const int nr = min(kTR, r_end - r0);
            for (int r = 0; r < nr; ++r) {
                const float2 v = *reinterpret_cast<const float2 *>(sV + r * CSA2_D + c);
                const float4 *pr = reinterpret_cast<const float4 *>(sP + r * 64);
#pragma unroll
                for (int h4 = 0; h4 < 16; ++h4) {
                    if (4 * h4 < H) {
                        const float4 pp = pr[h4];
                        acc[4 * h4][0] = fmaf(pp.x, v.x, acc[4 * h4][0]);
                        acc[4 * h4][1] = fmaf(pp.x, v.y, acc[4 * h4][1]);
                        acc[4 * h4 + 1][0] = fmaf(pp.y, v.x, acc[4 * h4 + 1][0]);
                        acc[4 * h4 + 1][1] = fmaf(pp.y, v.y, acc[4 * h4 + 1][1]);
                        acc[4 * h4 + 2][0] = fmaf(pp.z, v.x, acc[4 * h4 + 2][0]);
                        acc[4 * h4 + 2][1] = fmaf(pp.z, v.y, acc[4 * h4 + 2][1]);
                        acc[4 * h4 + 3][0] = fmaf(pp.w, v.x, acc[4 * h4 + 3][0]);
                        acc[4 * h4 + 3][1] = fmaf(pp.w, v.y, acc[4 * h4 + 3][1]);
                    }
                }
            }
        }
        __syncthreads();
    }
    if (tid == 0 && *sBad) count_event(p.counters, CSA2_CNT_BAD_INPUT);

    // ---- partials: O (unnormalised), m (base 2), l
    const int64_t pbase = ((int64_t)q * p.splits + split) * H;
    float *po = p.part_o + pbase * CSA2_D;
    for (int h = 0; h < H; ++h)
        *reinterpret_cast<float2 *>(po + h * CSA2_D + 2 * tid) = make_float2(acc[h][0], acc[h][1]);
    if (tid < H) {
        p.part_ml[(pbase + tid) * 2] = sM[tid];
        p.part_ml[(pbase + tid) * 2 + 1] = sL[tid];
    }
}

// out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s ;  lse = (M + log2 L) ln 2
__global__ void attn_combine_kernel(AttnParams p)
{
    const int q = blockIdx.y, h = blockIdx.x;
    const int H = p.H;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s)
        M = fmaxf(M, p.part_ml[(((int64_t)q * p.splits + s) * H + h) * 2]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    const int c = threadIdx.x * 4;
    for (int s = 0; s < p.splits; ++s) {
        const int64_t i = ((int64_t)q * p.splits + s) * H + h;
        const float ms = p.part_ml[i * 2];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - M);
        L = fmaf(p.part_ml[i * 2 + 1], f, L);
        const float4 v = *reinterpret_cast<const float4 *>(p.part_o + i * CSA2_D + c);
        o.x = fmaf(v.x, f, o.x);
        o.y = fmaf(v.y, f, o.y);
        o.z = fmaf(v.z, f, o.z);
        o.w = fmaf(v.w, f, o.w);
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
    *reinterpret_cast<float4 *>(p.out + ((int64_t)q * H + h) * CSA2_D + c) = o;
    if (p.lse != nullptr && threadIdx.x == 0)
        p.lse[(int64_t)q * H + h] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

cudaError_t launch_attn_simt(const AttnParams &p, cudaStream_t st)
{
    const size_t smem = (size_t)64 * kQStride * 2 + (size_t)kTR * CSA2_D * 4 + kTR * 64 * 4 +
                        3 * 64 * 4 + kTR * 4 + 16;
    cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attn_simt_kernel<<<dim3(p.splits, p.nq), kAtThreads, smem, st>>>(p);
    attn_combine_kernel<<<dim3(p.H, p.nq), 128, 0, st>>>(p);
    note_launch(2);
    return cudaGetLastError();
}

}  // namespace csa2
