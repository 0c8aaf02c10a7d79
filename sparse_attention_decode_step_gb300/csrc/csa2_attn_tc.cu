// csa2_attn_tc.cu -- sparse attention on tcgen05 (tensor cores, TMEM accumulators).
//
// [Thread] item 4: selected main-KV entries are concatenated with the windowed
// KV and attended; [Deep read] section 03: every layer brings its own query
// and window; [Notes] section 4: value = E2M1 code x E4M3 scale; [Notes]
// section 5: window [max(s, t - n_win + 1), t].
//
// One CTA = one query x a contiguous range of 128-row tiles of its row set.
// All heads share each gathered row (the latent is both key and value), so
// the contraction is laid out with the ROWS as the MMA's M = 128:
//     S^T [128 rows x 64 heads]   = V [128 x 512] . Q^T          (K = 512)
//     O^T [512 ch x 64 heads]    += V^T [512 x 128] . P^T        (K = 128 rows)
// V is dequantised once into shared memory as f16 in the 128-byte-swizzled
// K-major layout; the PV product reads the very same bytes as an MN-major
// operand.  E2M1 x E4M3 has at most 6 significant bits and lies in
// [2^-10, 2688], so it is exact in f16 (hardware cvt.rn.f16x2.e2m1x2, then one
// f16x2 multiply by the group scale).  Q (bf16 in) and the window rows (bf16
// in) are converted to f16, P is stored as f16; S and O accumulate in fp32 in
// tensor memory (64 + 256 columns).  Online softmax in base 2 with lazy
// rescaling: the reference max of a head moves only when a tile exceeds it by
// more than 8 (P <= 256 stays exact enough in f16), and O^T is then rescaled
// in TMEM.
//
// Warps: 0 = MMA issuer / TMEM owner; 1..4 = row workers (thread = tile row:
// gather + dequant, then softmax of that row; epilogue: thread = channel).
// Partials (O unnormalised, reference max, sum) go to the workspace; the
// split-combine kernel merges them.
#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace csa2 {

constexpr int kTcThreads = 160;
constexpr int kRows = 128;           // rows per tile (MMA M)
constexpr int kHeads = 64;           // MMA N (heads padded to 64)
constexpr uint32_t kVBytes = kRows * CSA2_D * 2;          // 128 KB
constexpr uint32_t kQBytes = kHeads * CSA2_D * 2;         // 64 KB
constexpr uint32_t kPBytes = kRows * kHeads * 2;          // 16 KB
constexpr uint32_t kVAtom = kRows * 128;                  // one 64-channel atom column of V
constexpr uint32_t kQAtom = kHeads * 128;
constexpr float kRescaleThreshold = 8.0f;                 // log2 units

__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_sync_workers()
{
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// 8 E2M1 codes (one 32-bit word, channel 2i in the low nibble of byte i) ->
// 4 x f16x2, multiplied by the f16x2 scale pair {s, s}.
__device__ __forceinline__ uint4 fp4x8_to_f16(uint32_t w, uint32_t s2)
{
    uint32_t o0, o1, o2, o3;
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}\n"
        : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
        : "r"(w));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o0) : "r"(s2));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o1) : "r"(s2));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o2) : "r"(s2));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o3) : "r"(s2));
    return make_uint4(o0, o1, o2, o3);
}

// E4M3 scale byte -> f16x2 {s, s}
__device__ __forceinline__ uint32_t scale_pair(uint32_t byte)
{
    uint32_t r;
    const uint16_t two = (uint16_t)(byte | (byte << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
    return r;
}

// two bf16 (one 32-bit word) -> f16x2
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// byte offset of the 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled atom column
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c)
{
    return r * 128u + ((c ^ (r & 7u)) << 4);
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64])
{
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
          "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
          "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
          "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
          "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const float (&v)[64])
{
    uint32_t r[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(v[i]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
        "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
        "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]),
        "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]),
        "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]),
        "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]),
        "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Transposed warp reduction: 64 values per lane -> lane l holds the reduction
// over the warp of values 2l and 2l+1 (in v[0], v[1]).
template <bool kMax>
__device__ __forceinline__ void warp_reduce64(float (&v)[64], int lane)
{
#pragma unroll
    for (int n = 64, o = 16; n > 2; n >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
}

// Row set of one query (selected entries, then window positions).
struct TcRowSet {
    int b, cnt, nw;
    int64_t base, lo, nt;
    bool bad;
};

__device__ __forceinline__ TcRowSet tc_row_set(const AttnParams &p, int q)
{
    TcRowSet rs{};
    rs.b = p.q_seq[q];
    rs.bad = (rs.b < 0 || rs.b >= p.batch);
    if (rs.bad) { rs.b = 0; return rs; }
    const int64_t t = p.q_pos[q];
    rs.base = p.seq_base[rs.b];
    int64_t nt = (t + 1) / p.m;
    const int64_t len = p.seq_len[rs.b];
    if (nt > len) nt = len;
    rs.nt = nt;
    rs.cnt = (p.cnt != nullptr && p.k_max > 0) ? min(p.cnt[q], p.k_max) : 0;
    if (rs.cnt < 0) rs.cnt = 0;
    if (p.win != nullptr && p.n_win > 0 && t >= 0) {
        int64_t lo = t - p.n_win + 1;
        const int64_t s = p.win_start ? (int64_t)p.win_start[rs.b] : 0;
        if (lo < s) lo = s;
        if (lo < 0) lo = 0;
        rs.lo = lo;
        rs.nw = (t >= lo) ? (int)(t - lo + 1) : 0;
    }
    return rs;
}

__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(AttnParams p)
{
    const int q = blockIdx.y, split = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~(uintptr_t)1023);
    uint8_t *sV = smem;                       // [8 atoms][128 rows][128 B]
    uint8_t *sQ = sV + kVBytes;               // [8 atoms][64 heads][128 B]
    uint8_t *sP = sQ + kQBytes;               // [128 rows][64 heads] f16, 128 B rows
    float *sRed = reinterpret_cast<float *>(sP + kPBytes);   // [4][64]
    float *sM = sRed + 4 * 64;                // reference max per head (log2 units)
    float *sL = sM + 64;                      // running sum per head
    float *sAlpha = sL + 64;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sAlpha + 64);
    uint64_t *bar_v = bars, *bar_s = bars + 1, *bar_p = bars + 2, *bar_o = bars + 3;
    uint64_t *bar_done = bars + 4;
    int *sFlag = reinterpret_cast<int *>(bars + 5);          // [0] abort, [1] rescale, [2] bad
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(sFlag + 4);
    volatile int *abort_flag = sFlag;

    const TcRowSet rs = tc_row_set(p, q);
    const int n_rows = rs.cnt + rs.nw;
    const int r_begin = split * p.rows_per_split;
    const int r_end = min(n_rows, r_begin + p.rows_per_split);
    const int n_tiles = (r_end > r_begin) ? (r_end - r_begin + kRows - 1) / kRows : 0;

    if (tid == 0) {
        mbar_init(bar_v, 4);
        mbar_init(bar_s, 1);
        mbar_init(bar_p, 4);
        mbar_init(bar_o, 1);
        mbar_init(bar_done, 1);
        sFlag[0] = 0;
        sFlag[1] = 0;
        sFlag[2] = rs.bad ? 1 : 0;
        fence_barrier_init();
    }
    if (tid < 64) { sM[tid] = -INFINITY; sL[tid] = 0.f; sAlpha[tid] = 1.f; }
    if (warp == 0) { tmem_alloc(sTmem, 512); tmem_relinquish(); }

    // ---- Q: bf16 -> f16, K-major 128-byte swizzle, heads >= H are zero
    {
        const uint16_t *qg = p.q + (int64_t)q * H * CSA2_D;
        for (int i = tid; i < kHeads * (CSA2_D / 8); i += kTcThreads) {
            const int h = i / (CSA2_D / 8), c8 = i % (CSA2_D / 8);   // 8 channels per chunk
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < H) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(qg + h * CSA2_D + c8 * 8));
                v = make_uint4(bf16x2_to_f16x2(raw.x), bf16x2_to_f16x2(raw.y),
                               bf16x2_to_f16x2(raw.z), bf16x2_to_f16x2(raw.w));
            }
            *reinterpret_cast<uint4 *>(sQ + (c8 >> 3) * kQAtom + sw128(h, c8 & 7)) = v;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t tS = tmem;                  // S^T: columns 0..63
    const uint32_t tO = tmem + 64;             // O^T block mb: columns 64 + 64 mb

    if (warp == 0) {
        // ============================================== MMA issuer
        if (lane == 0 && n_tiles > 0) {
            const uint32_t id_qk = instr_desc(128, kHeads, 0, 0, 0, 0);
            const uint32_t id_pv = instr_desc(128, kHeads, 0, 0, 1, 1);
            const uint32_t v0 = smem_u32(sV), q0 = smem_u32(sQ), p0 = smem_u32(sP);
            for (int i = 0; i < n_tiles; ++i) {
                if (!mbar_wait(bar_v, i & 1, abort_flag)) { *abort_flag = 1; break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < CSA2_D / 16; ++ks) {
                    const uint32_t a = v0 + (ks >> 2) * kVAtom + (ks & 3) * 32;
                    const uint32_t b = q0 + (ks >> 2) * kQAtom + (ks & 3) * 32;
                    mma_f16(tS, smem_desc(a, 16, 1024, kLayoutSW128),
                            smem_desc(b, 16, 1024, kLayoutSW128), id_qk, ks > 0);
                }
                mma_commit(bar_s);
                if (!mbar_wait(bar_p, i & 1, abort_flag)) { *abort_flag = 1; break; }
                tc_fence_after();
#pragma unroll
                for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
                    for (int ks = 0; ks < kRows / 16; ++ks) {
                        const uint32_t a = v0 + 2 * mb * kVAtom + ks * 2048;
                        const uint32_t b = p0 + ks * 2048;
                        mma_f16(tO + 64 * mb, smem_desc(a, kVAtom, 1024, kLayoutSW128),
                                smem_desc(b, kVAtom, 1024, kLayoutSW128), id_pv,
                                (i > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                mma_commit(bar_o);
            }
            if (*abort_flag) count_event(p.counters, CSA2_CNT_TIMEOUT);
            // every MMA of this thread has completed before TMEM is released
            volatile int no_abort = 0;
            mma_commit(bar_done);
            mbar_wait(bar_done, 0, &no_abort);
        }
    } else {
        // ============================================== row workers (128 threads)
        const int t = tid - 32;                           // tile row / TMEM lane in softmax
        const uint32_t quarter = (uint32_t)(warp & 3);   // TMEM lanes 32 quarter ..
        const int row = (int)(quarter * 32 + lane);      // TMEM lane owned by this thread
        const float l2s = p.sm_scale * 1.4426950408889634f;
        // prefetch registers: one FP4 row (256 B codes + 32 B scales)
        uint4 rc[16], rsc[2];
        int kind = 0;                                    // 0 empty, 1 fp4, 2 window
        int64_t wrow = 0;
        auto fetch = [&](int tile) {
            const int g = r_begin + tile * kRows + row;
            kind = 0;
            if (g < r_end) {
                if (g < rs.cnt) {
                    const int j = p.idx[(int64_t)q * p.ld_idx + g];
                    if (j >= 0 && j < rs.nt) {
                        kind = 1;
                        const int64_t r = rs.base + j;
                        const uint4 *c4 = reinterpret_cast<const uint4 *>(p.codes + r * CSA2_CODE_BYTES);
                        const uint4 *s4 = reinterpret_cast<const uint4 *>(p.scales + r * CSA2_SCALE_BYTES);
#pragma unroll
                        for (int k = 0; k < 16; ++k) rc[k] = __ldg(c4 + k);
                        rsc[0] = __ldg(s4);
                        rsc[1] = __ldg(s4 + 1);
                    } else {
                        sFlag[2] = 1;
                    }
                } else {
                    kind = 2;
                    const int64_t pos = rs.lo + (g - rs.cnt);
                    wrow = ((int64_t)rs.b * p.wcap + pos % p.wcap) * CSA2_D;
                }
            }
        };
        auto store_v = [&]() {
            if (kind == 1) {
                const uint32_t sw[8] = {rsc[0].x, rsc[0].y, rsc[0].z, rsc[0].w,
                                        rsc[1].x, rsc[1].y, rsc[1].z, rsc[1].w};
#pragma unroll
                for (int a = 0; a < 8; ++a) {            // atom column: channels 64a..64a+63
#pragma unroll
                    for (int c = 0; c < 8; ++c) {        // 8 channels = 4 code bytes
                        const int word = a * 8 + c;      // 32-bit word of the codes
                        const uint4 &u = rc[word >> 2];
                        const uint32_t w = (word & 3) == 0 ? u.x : (word & 3) == 1 ? u.y
                                         : (word & 3) == 2 ? u.z : u.w;
                        const int grp = (64 * a + 8 * c) >> 4;       // scale group
                        const uint32_t sb = (sw[grp >> 2] >> (8 * (grp & 3))) & 0xFFu;
                        *reinterpret_cast<uint4 *>(sV + a * kVAtom + sw128(row, c)) =
                            fp4x8_to_f16(w, scale_pair(sb));
                    }
                }
            } else if (kind == 2) {
                const uint4 *src = reinterpret_cast<const uint4 *>(p.win + wrow);
#pragma unroll 4
                for (int k = 0; k < 64; ++k) {
                    const uint4 raw = __ldg(src + k);
                    *reinterpret_cast<uint4 *>(sV + (k >> 3) * kVAtom + sw128(row, k & 7)) =
                        make_uint4(bf16x2_to_f16x2(raw.x), bf16x2_to_f16x2(raw.y),
                                   bf16x2_to_f16x2(raw.z), bf16x2_to_f16x2(raw.w));
                }
            } else {
#pragma unroll
                for (int k = 0; k < 64; ++k)
                    *reinterpret_cast<uint4 *>(sV + (k >> 3) * kVAtom + sw128(row, k & 7)) =
                        make_uint4(0, 0, 0, 0);
            }
        };

        if (n_tiles > 0) fetch(0);
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
            if (i > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar_o, (i - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
            }
            const bool valid = kind != 0;
            store_v();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_v);
            if (i + 1 < n_tiles) fetch(i + 1);

            // ---- softmax of this thread's row
            ok = __all_sync(0xffffffffu, mbar_wait(bar_s, i & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            float x[64];
            tmem_ld64(tS + ((quarter * 32u) << 16), x);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 64; ++h) x[h] = valid ? x[h] * l2s : -INFINITY;
            float r[64];
#pragma unroll
            for (int h = 0; h < 64; ++h) r[h] = x[h];
            warp_reduce64<true>(r, lane);
            sRed[quarter * 64 + 2 * lane] = r[0];
            sRed[quarter * 64 + 2 * lane + 1] = r[1];
            named_sync_workers();
            if (t < 64) {
                const float tmax = fmaxf(fmaxf(sRed[t], sRed[64 + t]), fmaxf(sRed[128 + t], sRed[192 + t]));
                const float m_old = sM[t];
                float alpha = 1.f;
                if (tmax > m_old + kRescaleThreshold || (m_old == -INFINITY && tmax > -INFINITY)) {
                    alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - tmax);
                    sM[t] = tmax;
                    if (i > 0) sFlag[1] = 1;
                }
                sAlpha[t] = alpha;
            }
            named_sync_workers();
            // P = 2^(x - m) as f16 into sP (row = this thread's tile row)
            float mh[64];
#pragma unroll
            for (int h4 = 0; h4 < 16; ++h4) {
                const float4 m4 = reinterpret_cast<const float4 *>(sM)[h4];
                mh[4 * h4] = m4.x; mh[4 * h4 + 1] = m4.y; mh[4 * h4 + 2] = m4.z; mh[4 * h4 + 3] = m4.w;
            }
#pragma unroll
            for (int h = 0; h < 64; ++h) x[h] = (mh[h] == -INFINITY) ? 0.f : exp2f(x[h] - mh[h]);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = make_uint4(f32x2_to_f16x2(x[8 * c], x[8 * c + 1]),
                                           f32x2_to_f16x2(x[8 * c + 2], x[8 * c + 3]),
                                           f32x2_to_f16x2(x[8 * c + 4], x[8 * c + 5]),
                                           f32x2_to_f16x2(x[8 * c + 6], x[8 * c + 7]));
                *reinterpret_cast<uint4 *>(sP + sw128(row, c)) = v;
            }
            warp_reduce64<false>(x, lane);
            sRed[quarter * 64 + 2 * lane] = x[0];
            sRed[quarter * 64 + 2 * lane + 1] = x[1];
            named_sync_workers();
            if (t < 64) sL[t] = sL[t] * sAlpha[t] + ((sRed[t] + sRed[64 + t]) + (sRed[128 + t] + sRed[192 + t]));
            const bool rescale = sFlag[1] != 0;
            named_sync_workers();
            if (rescale) {
                // O^T *= alpha per head (column); PV of the previous tile has completed
                float al[64];
#pragma unroll
                for (int h4 = 0; h4 < 16; ++h4) {
                    const float4 a4 = reinterpret_cast<const float4 *>(sAlpha)[h4];
                    al[4 * h4] = a4.x; al[4 * h4 + 1] = a4.y; al[4 * h4 + 2] = a4.z; al[4 * h4 + 3] = a4.w;
                }
#pragma unroll 1
                for (int mb = 0; mb < 4; ++mb) {
                    float o[64];
                    const uint32_t ta = tO + 64 * mb + ((quarter * 32u) << 16);
                    tmem_ld64(ta, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 64; ++h) o[h] *= al[h];
                    tmem_st64(ta, o);
                }
                tmem_wait_st();
                named_sync_workers();
                if (t == 0) sFlag[1] = 0;
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p);
        }
        if (!ok) *abort_flag = 1;

        // ---- epilogue: O^T (unnormalised) -> partials; thread = channel within block
        if (ok && n_tiles > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar_o, (n_tiles - 1) & 1, abort_flag));
            tc_fence_after();
        }
        const int64_t pbase = ((int64_t)q * p.splits + split) * H;
        if (ok) {
            float *po = p.part_o + pbase * CSA2_D;
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
                float o[64];
                if (n_tiles > 0) {
                    tmem_ld64(tO + 64 * mb + ((quarter * 32u) << 16), o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int h = 0; h < 64; ++h) o[h] = 0.f;
                }
                const int c = 128 * mb + row;
#pragma unroll
                for (int h = 0; h < 64; ++h)
                    if (h < H) po[(int64_t)h * CSA2_D + c] = o[h];
            }
            if (t < H) {
                p.part_ml[(pbase + t) * 2] = (n_tiles > 0) ? sM[t] : -INFINITY;
                p.part_ml[(pbase + t) * 2 + 1] = (n_tiles > 0) ? sL[t] : 0.f;
            }
        }
        if (t == 0 && sFlag[2]) count_event(p.counters, CSA2_CNT_BAD_INPUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st)
{
    const size_t smem = 1024 + kVBytes + kQBytes + kPBytes + (4 * 64 + 3 * 64) * 4 + 5 * 8 + 64;
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attn_tc_kernel<<<dim3(p.splits, p.nq), kTcThreads, smem, st>>>(p);
    attn_combine_kernel<<<dim3(p.H, p.nq), 128, 0, st>>>(p);
    note_launch(2);
    return cudaGetLastError();
}

}  // namespace csa2
