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
// tensor memory (64 + 256 columns, 64 more for the running row sums).  Online
// softmax in base 2 with lazy rescaling: the reference max of a head moves
// only when a tile exceeds it by more than 8 (P <= 256 stays exact enough in
// f16), and O^T is then rescaled in TMEM.
//
// Warps: 0..15 = workers (warp 0 also owns TMEM), 16 = MMA issuer (the
// issuing thread stalls while the tensor pipe's queue is full, so it must not
// hold up the workers).  Sixteen workers keep four warps on each scheduler; a
// 17-warp CTA gets at most 96 registers per thread.  V is gathered with 8 lanes
// per row (128 contiguous code bytes = one 128-byte line per row, 4 rows per
// warp load, 8 rows per warp and tile) and dequantised in two 256-channel
// chunks, each with its own barrier.  The chunks are pipelined across tiles:
// the PV product of tile i releases chunk 0 of the V tile after its first two
// channel blocks, so the workers store chunk 0 of tile i + 1 while PV
// finishes, and the QK product of tile i + 1 over chunk 0 runs while chunk 1
// is stored.  The next tile's codes are loaded in two halves, chunk 0 while
// this tile's QK product finishes and chunk 1 once its P is stored (while its
// PV product starts); the rows of the tile after that are asked of L2 one tile
// earlier.  In the softmax a worker owns a quarter of a tile row (16 heads),
// four per TMEM lane quarter.  The cross-row max reduction runs only when a
// logit exceeds its head's reference max by more than 8 (always on the first
// tile); each thread keeps its row's sums in TMEM and they are reduced once,
// at the end.  The workers' votes and barriers leave the MMA warp out, whose
// waits are bounded and end when the workers raise the abort flag.  The
// splits of a query (at most 8) form a thread-block cluster: every CTA sends
// its reference max and sum to all peers, scales its O^T by 2^(m_s - M) / L
// and stores each 32-channel chunk into the shared memory of the CTA that owns
// the chunk ([64 heads][32 channels]; a 4 x 4 transpose within each group of 4
// lanes gives a lane 4 channels of one head, so a warp store writes four
// contiguous 128-byte head rows in 16-byte words), which sums the splits'
// chunks and writes the output 16 bytes at a time.  Nothing
// goes through global memory between splits.  The set-up that reads nothing
// the previous kernel writes (barriers, TMEM, and inside a layer step the
// query block and the query's metadata) runs before the
// programmatic-dependent-launch wait.
#include <cooperative_groups.h>

#include "csa2_device.cuh"
#include "csa2_internal.h"

namespace cg = cooperative_groups;

namespace csa2 {

constexpr int kTcThreads = 544;       // warps 0..15 workers, warp 16 MMA issuer
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

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x (hardware approximation, relative error near 2^-22; 2^-inf = 0)
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// Transposed warp reduction of 16 values per lane: afterwards lanes l and
// l + 16 hold, in v[0], the reduction over all 32 lanes of value l & 15.
template <bool kMax>
__device__ __forceinline__ void warp_reduce16(float (&v)[16], int lane)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float recv = __shfl_xor_sync(0xffffffffu, v[i], 16);
        v[i] = kMax ? fmaxf(v[i], recv) : v[i] + recv;
    }
#pragma unroll
    for (int n = 16, o = 8; n > 1; n >>= 1, o >>= 1) {
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

constexpr int kWorkerWarps = 16;                     // four per TMEM lane quarter
constexpr int kWorkers = 32 * kWorkerWarps;

// CTA barrier of the worker warps alone (the MMA warp never takes part)
__device__ __forceinline__ void workers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory");
}

// The same barrier, returning whether v holds for every worker thread
__device__ __forceinline__ bool workers_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n"
        ".reg .pred pin, pout;\n"
        "setp.ne.u32 pin, %1, 0;\n"
        "bar.red.and.pred pout, 1, %2, pin;\n"
        "selp.u32 %0, 1, 0, pout;\n"
        "}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kWorkers)
        : "memory");
    return r != 0;
}

// Row set of one query (selected entries, then window positions).  The
// metadata part reads only the caller's query and cache descriptors; the
// count of selected entries (written by a top-k just before) is read apart.
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

__device__ __forceinline__ int tc_row_count(const AttnParams &p, int q)
{
    const int c = (p.cnt != nullptr && p.k_max > 0) ? min(p.cnt[q], p.k_max) : 0;
    return c < 0 ? 0 : c;
}

// Cluster merge: a block of the receive area is one 32-channel chunk of one
// split, [64 heads][32 channels] fp32 (8 KB), so that a warp (lane = channel)
// writes and reads 128 contiguous bytes per head.
constexpr int kXBlock = 64 * 32;

// 4 x 4 transpose within each group of 4 lanes: lane 4g + j holds a[i] =
// element (row j, column i) before and element (row i, column j) after.
__device__ __forceinline__ void transpose4(float (&a)[4], int lane)
{
    const bool b0 = (lane & 1) != 0, b1 = (lane & 2) != 0;
    float x0 = b0 ? a[0] : a[1], x1 = b0 ? a[2] : a[3];
    float r0 = __shfl_xor_sync(0xffffffffu, x0, 1), r1 = __shfl_xor_sync(0xffffffffu, x1, 1);
    if (b0) { a[0] = r0; a[2] = r1; } else { a[1] = r0; a[3] = r1; }
    x0 = b1 ? a[0] : a[2];
    x1 = b1 ? a[1] : a[3];
    r0 = __shfl_xor_sync(0xffffffffu, x0, 2);
    r1 = __shfl_xor_sync(0xffffffffu, x1, 2);
    if (b1) { a[0] = r0; a[1] = r1; } else { a[2] = r0; a[3] = r1; }
}
constexpr int kMaxClusterSplits = 16;   // 1 .. 12 or 16 (the receive area, below)

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
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
    float *sRed = reinterpret_cast<float *>(sP + kPBytes);   // [4 quarters][64 heads]
    float *sM = sRed + 4 * 64;                // reference max per head (log2 units)
    float *sAlpha = sM + 64;                  // rescale factor of the current tile
    float *sL = sAlpha + 64;                  // running sum per head
    float *sRedL = sL + 64;                   // [4 quarters][64 heads] tile row sums
    float *sML = sRedL + 4 * 64;              // cluster merge: [split][m | l][64 heads]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sML + kMaxClusterSplits * 2 * 64);
    uint64_t *bar_v = bars;                   // [2]: V channel chunk h (256 channels) stored
    uint64_t *bar_o = bars + 2;               // [2]: PV channel blocks 2h, 2h + 1 done (chunk h free)
    uint64_t *bar_s = bars + 4, *bar_p = bars + 5;   // S^T complete; P stored
    uint64_t *bar_done = bars + 6, *bar_q = bars + 7;
    int *sFlag = reinterpret_cast<int *>(bars + 8);   // [0] abort [1] rescale [2] bad [3] need max
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(sFlag + 4);
    volatile int *abort_flag = sFlag;

    // ---- set-up that reads nothing an earlier kernel writes: barriers, TMEM, and
    // (p.early) the query block, whose bulk copy lands in the still-free V tile,
    // and the query's row-set metadata
    if (tid == 0) {
        for (int c = 0; c < 2; ++c) {
            mbar_init(&bar_v[c], kWorkerWarps);
            mbar_init(&bar_o[c], 1);
        }
        mbar_init(bar_s, 1);
        mbar_init(bar_p, kWorkerWarps);
        mbar_init(bar_done, 1);
        mbar_init(bar_q, 1);
        sFlag[0] = 0;
        sFlag[1] = 0;
        sFlag[2] = 0;
        sFlag[3] = 0;
        fence_barrier_init();
    }
    if (tid < 64) { sM[tid] = -INFINITY; sAlpha[tid] = 1.f; sL[tid] = 0.f; }
    // a CTA's shared memory may be written by its cluster peers only once it runs:
    // arrive now, wait before the first remote store (the merge at the end)
    cluster_arrive();
    __syncthreads();
    auto load_q = [&]() {
        const uint32_t qbytes = (uint32_t)H * CSA2_D * 2;
        mbar_arrive_expect_tx(bar_q, qbytes);
        bulk_load(sV, p.q + (int64_t)q * H * CSA2_D, qbytes, bar_q);
    };
    // ---- Q: the raw bf16 block [H][512] lands in the V tile, then bf16 -> f16 into
    // the K-major 128-byte-swizzled sQ (heads >= H are zero): inside a layer
    // step while the top-k finishes, otherwise while the first tile's rows are
    // in flight (the first tile's stores into the V tile come after a barrier)
    auto convert_q = [&]() {
        volatile int no_abort = 0;
        if (!mbar_wait(bar_q, 0, &no_abort)) sFlag[0] = 1;
        for (int i = tid; i < kHeads * (CSA2_D / 8); i += kTcThreads) {
            const int h = i / (CSA2_D / 8), c8 = i % (CSA2_D / 8);   // 8 channels per chunk
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < H) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(sV + h * 1024 + c8 * 16);
                v = make_uint4(bf16x2_to_f16x2(raw.x), bf16x2_to_f16x2(raw.y),
                               bf16x2_to_f16x2(raw.z), bf16x2_to_f16x2(raw.w));
            }
            *reinterpret_cast<uint4 *>(sQ + (c8 >> 3) * kQAtom + sw128(h, c8 & 7)) = v;
        }
    };
    if (tid == 0 && p.early) load_q();
    if (warp == 0) { tmem_alloc(sTmem, 512); tmem_relinquish(); }
    TcRowSet rs{};
    if (p.early) {
        rs = tc_row_set(p, q);
        convert_q();
    }
    pdl_wait();
    pdl_trigger();
    if (tid == 0 && !p.early) load_q();
    if (!p.early) rs = tc_row_set(p, q);
    if (!rs.bad) rs.cnt = tc_row_count(p, q);
    if (tid == 0 && rs.bad) sFlag[2] = 1;
    const int n_rows = rs.cnt + rs.nw;
    // this query's tiles, ceil(tiles / splits) per split: the last split, which
    // holds the window rows (the slower tile), gets the remainder
    const int q_tiles = (n_rows + kRows - 1) / kRows;
    const int tps = (q_tiles + p.splits - 1) / p.splits;
    const int t_begin = min(q_tiles, split * tps);
    const int t_end = min(q_tiles, t_begin + tps);
    const int r_begin = t_begin * kRows;
    const int r_end = min(n_rows, t_end * kRows);
    const int n_tiles = t_end - t_begin;

    // ---- a worker thread's places: softmax row (= TMEM lane) and heads; gather rows
    const uint32_t quarter = (uint32_t)(warp & 3);    // TMEM lanes 32 quarter ..
    const int row = (int)(quarter * 32 + lane);       // tile row == TMEM lane of this thread
    const int h0 = 16 * (warp >> 2);                  // heads h0 .. h0 + 15 of its softmax

    // ---- gather.  Warp w fills tile rows 8w .. 8w + 7.  A warp load covers 4
    // rows with 8 lanes each: lane l takes row 8w + 4x + (l >> 3) and, in channel
    // chunk h (channels 256h ..), the 32 channels 256h + 32 sub .. (sub = l & 7):
    // 16 contiguous code bytes and 2 scale bytes, so that each row's 8 lanes read
    // one 128-byte line.  Register slot t = 2h + x.
    const int sub = lane & 7;
    const int rho = sub >> 1;                          // store rotation (bank groups)
    uint4 gc[4];                  // codes of slot t
    uint32_t gsc[4];              // the two scale bytes of those channels
    uint32_t gkind = 0;           // bit t: FP4 row with data; bit 4 + t: window row
    int gj = -1;                  // lanes 0-7: entry of row 8 warp + lane of the tile loaded next
    auto tile_row = [&](int tile, int r) { return r_begin + tile * kRows + r; };
    // entry of tile row r (-1 for window rows and rows past the end)
    auto entry = [&](int tile, int r) {
        const int g = tile_row(tile, r);
        return (g < r_end && g < rs.cnt) ? __ldg(p.idx + (int64_t)q * p.ld_idx + g) : -1;
    };
    // the register slots of channel chunk h (slots 2h, 2h + 1) with tile `tile`
    auto load_half = [&](int tile, int h) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int t = 2 * h + x;
            gkind &= ~((1u << t) | (1u << (4 + t)));
            const int rw = 4 * x + (lane >> 3);
            const int g = tile_row(tile, 8 * warp + rw);
            const int j = __shfl_sync(0xffffffffu, gj, rw);
            if (g < r_end && g < rs.cnt) {
                if (j >= 0 && j < rs.nt) {
                    const int64_t r = rs.base + j;
                    gc[t] = __ldg(reinterpret_cast<const uint4 *>(p.codes + r * CSA2_CODE_BYTES) + 8 * h + sub);
                    gsc[t] = __ldg(reinterpret_cast<const uint16_t *>(p.scales + r * CSA2_SCALE_BYTES) + 8 * h + sub);
                    gkind |= 1u << t;
                } else {
                    sFlag[2] = 1;
                }
            } else if (g < r_end) {
                gkind |= 1u << (4 + t);
            }
        }
    };
    // Chunk h of this warp's rows into sV.  A lane's 32 channels are the 16-byte
    // pieces 4 (sub & 1) .. + 3 of atom column 4h + (sub >> 1).  A 16-byte store is
    // served 8 lanes (one row) at a time; lane sub writes, in its m-th store, piece
    // 4 (sub & 1) + ((m + rho) & 3), so that the 8 lanes of a row hit 8 different
    // 16-byte bank groups (the source words are rotated to match).
    auto store_chunk = [&](int tile, int h) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int t = 2 * h + x;
            const int r = 8 * warp + 4 * x + (lane >> 3);
            uint4 v[4];
            if (gkind & (1u << t)) {
                const uint32_t p0 = scale_pair(gsc[t] & 0xFFu), p1 = scale_pair((gsc[t] >> 8) & 0xFFu);
                uint32_t w[4] = {gc[t].x, gc[t].y, gc[t].z, gc[t].w};
                uint32_t sp[4] = {p0, p0, p1, p1};
                if (rho & 1) {
                    const uint32_t w0 = w[0], s0 = sp[0];
                    w[0] = w[1]; w[1] = w[2]; w[2] = w[3]; w[3] = w0;
                    sp[0] = sp[1]; sp[1] = sp[2]; sp[2] = sp[3]; sp[3] = s0;
                }
                if (rho & 2) {
                    uint32_t a = w[0], b = w[1];
                    w[0] = w[2]; w[1] = w[3]; w[2] = a; w[3] = b;
                    a = sp[0]; b = sp[1];
                    sp[0] = sp[2]; sp[1] = sp[3]; sp[2] = a; sp[3] = b;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) v[m] = fp4x8_to_f16(w[m], sp[m]);
            } else if (gkind & (1u << (4 + t))) {
                const int64_t pos = rs.lo + (tile_row(tile, r) - rs.cnt);
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    p.win + ((int64_t)rs.b * p.wcap + pos % p.wcap) * CSA2_D) + 32 * h + 4 * sub;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint4 raw = __ldg(src + ((m + rho) & 3));
                    v[m] = make_uint4(bf16x2_to_f16x2(raw.x), bf16x2_to_f16x2(raw.y),
                                      bf16x2_to_f16x2(raw.z), bf16x2_to_f16x2(raw.w));
                }
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m) v[m] = make_uint4(0, 0, 0, 0);
            }
            uint8_t *dst = sV + (4 * h + (sub >> 1)) * kVAtom;
#pragma unroll
            for (int m = 0; m < 4; ++m)
                *reinterpret_cast<uint4 *>(
                    dst + sw128((uint32_t)r, (uint32_t)(4 * (sub & 1) + ((m + rho) & 3)))) = v[m];
        }
    };
    // The rows of the tile after the next one are asked of L2 one tile before
    // their loads (lanes 0-7: row 8 warp + lane, entry j; gj2 holds the entries
    // of that tile)
    int gj2 = -1;
    auto prefetch_rows = [&](int tile, int j) {
        const int g = tile_row(tile, 8 * warp + (lane & 7));
        if (lane < 8 && g < r_end && g < rs.cnt && j >= 0 && j < rs.nt) {
            const int64_t r = rs.base + j;
            const uint8_t *c = p.codes + r * CSA2_CODE_BYTES;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(c));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(c + 128));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p.scales + r * CSA2_SCALE_BYTES));
        }
    };
    auto rows_entry = [&](int tile) { return lane < 8 ? entry(tile, 8 * warp + (lane & 7)) : -1; };
    int my_j = -1;                // entry of this thread's softmax row in the current tile
    if (warp < kWorkerWarps && n_tiles > 0) {
        gj = rows_entry(0);
        my_j = entry(0, row);
        load_half(0, 0);
        load_half(0, 1);
        if (n_tiles > 1) gj = rows_entry(1);
        if (n_tiles > 2) gj2 = rows_entry(2);
    }
    // (p.early: the query was converted before the dependent-launch wait)
    if (!p.early) convert_q();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t tS = tmem;                  // S^T: columns 0..63
    const uint32_t tO = tmem + 64;             // O^T block mb: columns 64 + 64 mb
    const uint32_t tLsum = tmem + 320;         // running sums: columns 320 .. 383
    const uint32_t lane_q = (quarter * 32u) << 16;

    const uint32_t tL = tLsum + (uint32_t)h0 + lane_q;   // (workers) running sums, see below
    if (warp == kWorkerWarps) {
        // ============================================== MMA issuer
        if (lane == 0 && n_tiles > 0) {
            const uint32_t id_qk = instr_desc(128, kHeads, 0, 0, 0, 0);
            const uint32_t id_pv = instr_desc(128, kHeads, 0, 0, 1, 1);
            const uint32_t v0 = smem_u32(sV), q0 = smem_u32(sQ), p0 = smem_u32(sP);
            for (int i = 0; i < n_tiles; ++i) {
                bool run = true;
                for (int h = 0; h < 2 && run; ++h) {
                    // the K range of chunk h (channels 256h ..) as soon as it is stored
                    if (!mbar_wait<true>(&bar_v[h], i & 1, abort_flag)) { run = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int k16 = 0; k16 < 16; ++k16) {
                        const int ks = 16 * h + k16;
                        const uint32_t a = v0 + (ks >> 2) * kVAtom + (ks & 3) * 32;
                        const uint32_t b = q0 + (ks >> 2) * kQAtom + (ks & 3) * 32;
                        mma_f16(tS, smem_desc(a, 16, 1024, kLayoutSW128),
                                smem_desc(b, 16, 1024, kLayoutSW128), id_qk, ks > 0);
                    }
                }
                if (!run) { *abort_flag = 1; break; }
                mma_commit(bar_s);
                if (!mbar_wait<true>(bar_p, i & 1, abort_flag)) { *abort_flag = 1; break; }
                tc_fence_after();
                // channel blocks 0, 1 (chunk 0 of V) then 2, 3 (chunk 1); each pair's
                // completion releases its chunk of the V tile
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
                    if (mb & 1) mma_commit(&bar_o[mb >> 1]);
                }
            }
            // completes once every MMA issued above has completed
            mma_commit(bar_done);
        }
    } else {
        // ============================================== 16 worker warps
        const float l2s = p.sm_scale * 1.4426950408889634f;
        // this thread's share of the running sums, its row's P for heads h0 .. h0+15,
        // accumulates in TMEM columns 320 + h0 .. (its lane = its row): rescaled with
        // the reference max, reduced over the rows once, at the end
        {
            float z[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) z[h] = 0.f;
            tmem_st16(tL, z);
            tmem_wait_st();
        }
        bool ok = !sFlag[0];
        for (int i = 0; i < n_tiles && ok; ++i) {
            if (i + 2 < n_tiles) prefetch_rows(i + 2, gj2);
            const int g_row = tile_row(i, row);
            const bool valid = g_row < r_end && (g_row >= rs.cnt || (my_j >= 0 && my_j < rs.nt));
            // chunk h of this tile goes where the previous tile's PV product has
            // released it (its channel blocks 2h, 2h + 1 done); a warp that gives
            // up on a wait still arrives, and the vote below stops every worker
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                bool got = true;
                if (i > 0) {
                    got = __all_sync(0xffffffffu, mbar_wait<true>(&bar_o[h], (i - 1) & 1, abort_flag));
                    tc_fence_after();
                }
                if (got) store_chunk(i, h);
                else ok = false;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_v[h]);
            }
            // the next tile's codes: chunk 0 while the QK product finishes, chunk 1
            // (below) while the PV product of this tile starts
            const bool more = i + 1 < n_tiles;
            int my_j_next = -1;
            if (more) load_half(i + 1, 0);

            // ---- softmax of this row, heads h0 .. h0+15
            const bool got_s = ok && mbar_wait<true>(bar_s, i & 1, abort_flag);
            tc_fence_after();
            float x[16];
            if (got_s) {
                tmem_ld16(tS + lane_q + (uint32_t)h0, x);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int h = 0; h < 16; ++h) x[h] = 0.f;
            }
            bool over = false;
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) {
                const float4 m4 = reinterpret_cast<const float4 *>(sM + h0)[h4];
                const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int h = 4 * h4 + j;
                    x[h] = valid ? x[h] * l2s : -INFINITY;
                    over |= x[h] > mm[j] + kRescaleThreshold;
                }
            }
            // the reference max moves only when some logit is more than 8 above it;
            // the flag holds the number of the last tile that needed it (no reset)
            if (over) sFlag[3] = i + 1;
            ok = workers_and(got_s);
            if (!ok) {
                if (tid == 0) *abort_flag = 1;     // (the issuer stops waiting)
                break;
            }
            if (sFlag[3] == i + 1) {
                float r[16];
#pragma unroll
                for (int h = 0; h < 16; ++h) r[h] = x[h];
                warp_reduce16<true>(r, lane);
                if (lane < 16) sRed[quarter * 64 + h0 + lane] = r[0];
                workers_sync();
                if (tid < 64) {
                    const float tmax = fmaxf(fmaxf(sRed[tid], sRed[64 + tid]),
                                             fmaxf(sRed[128 + tid], sRed[192 + tid]));
                    const float m_old = sM[tid];
                    float alpha = 1.f;
                    if (tmax > m_old + kRescaleThreshold) {
                        alpha = (m_old == -INFINITY) ? 0.f : fast_exp2(m_old - tmax);
                        sM[tid] = tmax;
                        if (i > 0) sFlag[1] = 1;
                    }
                    sAlpha[tid] = alpha;
                }
                workers_sync();
                if (sFlag[1] != 0) {
                    // O^T and the running sums *= alpha per head; PV of the previous
                    // tile has completed (both of its chunk barriers were waited above)
                    float al[16];
#pragma unroll
                    for (int h4 = 0; h4 < 4; ++h4) {
                        const float4 a4 = reinterpret_cast<const float4 *>(sAlpha + h0)[h4];
                        al[4 * h4] = a4.x; al[4 * h4 + 1] = a4.y; al[4 * h4 + 2] = a4.z; al[4 * h4 + 3] = a4.w;
                    }
                    {
                        float o[16];
                        tmem_ld16(tL, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int h = 0; h < 16; ++h) o[h] *= al[h];
                        tmem_st16(tL, o);
                    }
#pragma unroll 1
                    for (int mb = 0; mb < 4; ++mb) {
                        float o[16];
                        const uint32_t ta = tO + 64 * mb + (uint32_t)h0 + lane_q;
                        tmem_ld16(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int h = 0; h < 16; ++h) o[h] *= al[h];
                        tmem_st16(ta, o);
                    }
                    tmem_wait_st();
                }
                workers_sync();
                if (tid == 0) sFlag[1] = 0;
            }
            // P = 2^(x - m) as f16 into sP (pieces h0 / 8, h0 / 8 + 1 of its row)
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) {
                const float4 m4 = reinterpret_cast<const float4 *>(sM + h0)[h4];
                const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int h = 4 * h4 + j;
                    x[h] = (mm[j] == -INFINITY) ? 0.f : fast_exp2(x[h] - mm[j]);
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint4 v = make_uint4(f32x2_to_f16x2(x[8 * c], x[8 * c + 1]),
                                           f32x2_to_f16x2(x[8 * c + 2], x[8 * c + 3]),
                                           f32x2_to_f16x2(x[8 * c + 4], x[8 * c + 5]),
                                           f32x2_to_f16x2(x[8 * c + 6], x[8 * c + 7]));
                *reinterpret_cast<uint4 *>(sP + sw128(row, h0 / 8 + c)) = v;
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p);
            if (more) {
                load_half(i + 1, 1);
                gj = gj2;
                if (i + 3 < n_tiles) gj2 = rows_entry(i + 3);
                my_j_next = entry(i + 1, row);
            }
            {
                float o[16];
                tmem_ld16(tL, o);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 16; ++h) o[h] += x[h];
                tmem_st16(tL, o);
                tmem_wait_st();
            }
            my_j = my_j_next;
        }
        if (!ok) *abort_flag = 1;
    }
    // every MMA issued has completed before O^T is read and TMEM released
    if (n_tiles > 0) {
        volatile int no_abort = 0;
        if (!mbar_wait<true>(bar_done, 0, &no_abort)) *abort_flag = 1;
        tc_fence_after();
    }
    // the running sums: over the warp's 32 rows, then the 4 quarters
    if (warp < kWorkerWarps) {
        float lsum[16];
        tmem_ld16(tL, lsum);
        tmem_wait_ld();
        warp_reduce16<false>(lsum, lane);
        if (lane < 16) sRedL[quarter * 64 + h0 + lane] = lsum[0];
    }
    __syncthreads();
    if (tid < 64) sL[tid] = (sRedL[tid] + sRedL[64 + tid]) + (sRedL[128 + tid] + sRedL[192 + tid]);
    if (tid == 0 && sFlag[2]) count_event(p.counters, CSA2_CNT_BAD_INPUT);
    if (tid == 0 && *abort_flag) count_event(p.counters, CSA2_CNT_TIMEOUT);

    {
        // ---- merge of the cluster's splits.  Every thread of every CTA reaches
        // each cluster barrier exactly once, whatever happened above.
        cg::cluster_group cluster = cg::this_cluster();
        const int S = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
        float *sFac = reinterpret_cast<float *>(sP);          // [split][head]
        float *sX = reinterpret_cast<float *>(sV);            // receive area (V and Q tiles)
        cluster_wait();              // (arrived at the start) every CTA of the cluster runs
        // this split's reference max and sum go to every CTA's own table (a peer's
        // V, Q and P tiles may still be in use)
        if (tid < 64) {
            const bool any = !*abort_flag && n_tiles > 0;
            const float m = any ? sM[tid] : -INFINITY, l = any ? sL[tid] : 0.f;
            for (int s = 0; s < S; ++s) {
                float *t = cluster.map_shared_rank(sML, s);
                t[rank * 128 + tid] = m;
                t[rank * 128 + 64 + tid] = l;
            }
        }
        cluster.sync();              // every split has finished its tiles; all m, l delivered
        if (tid < 64) {
            float M = -INFINITY;
            for (int s = 0; s < S; ++s) M = fmaxf(M, sML[s * 128 + tid]);
            float L = 0.f;
            for (int s = 0; s < S; ++s) {
                const float ms = sML[s * 128 + tid];
                const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
                sFac[s * 64 + tid] = w;
                L = fmaf(sML[s * 128 + 64 + tid], w, L);
            }
            const float inv = (L > 0.f) ? 1.f / L : 0.f;
            for (int s = 0; s < S; ++s) sFac[s * 64 + tid] *= inv;
            if (p.lse != nullptr && rank == 0 && tid < H)
                p.lse[(int64_t)q * H + tid] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
        }
        __syncthreads();
        if (warp < kWorkerWarps) {
            const bool any = !*abort_flag && n_tiles > 0;
            float f[16];
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) {
                const float4 a4 = reinterpret_cast<const float4 *>(sFac + rank * 64 + h0)[h4];
                f[4 * h4] = a4.x; f[4 * h4 + 1] = a4.y; f[4 * h4 + 2] = a4.z; f[4 * h4 + 3] = a4.w;
            }
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
                float o[16];
                if (any) {
                    tmem_ld16(tO + 64 * mb + (uint32_t)h0 + lane_q, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int h = 0; h < 16; ++h) o[h] = 0.f;
                }
                const int c = 4 * mb + (int)quarter;
                // lane 4g + j: channels 32c + 4g .. + 3 of head h0 + 4k + j, one
                // 16-byte word (8 lanes write one head's 128 contiguous bytes)
                const int g4 = 4 * (lane >> 2), j = lane & 3;
                float *dst = S == 1 ? nullptr
                                    : cluster.map_shared_rank(sX, c % S) + ((c / S) * S + rank) * kXBlock;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float a[4] = {o[4 * k] * f[4 * k], o[4 * k + 1] * f[4 * k + 1],
                                  o[4 * k + 2] * f[4 * k + 2], o[4 * k + 3] * f[4 * k + 3]};
                    transpose4(a, lane);
                    const int h = h0 + 4 * k + j;
                    const float4 v = make_float4(a[0], a[1], a[2], a[3]);
                    if (S == 1) {
                        // a single split: its scaled O^T is the output
                        if (h < H)
                            *reinterpret_cast<float4 *>(p.out + ((int64_t)q * H + h) * CSA2_D + 32 * c + g4) = v;
                    } else {
                        *reinterpret_cast<float4 *>(dst + h * 32 + g4) = v;
                    }
                }
            }
        }
        if (S > 1) cluster.sync();   // every block has arrived at its owner (S is uniform)
        // chunks rank, rank + S, ...: a warp sums 4 heads of the chunk per item,
        // lane 8j + g4 / 4 the channels g4 .. g4 + 3 of head hb + j (one 16-byte
        // load per split, all in flight; one 16-byte store)
        const int n_own = S > 1 ? (16 - rank + S - 1) / S : 0;
        for (int it = warp; it < n_own * 16; it += kTcThreads / 32) {
            const int k = it >> 4, c = rank + k * S;
            const int h = 4 * (it & 15) + (lane >> 3), g4 = 4 * (lane & 7);
            if (h >= H) continue;
            const float *src = sX + k * S * kXBlock + h * 32 + g4;
            float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < S; s0 += 4) {
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    v[j] = (s0 + j < S) ? *reinterpret_cast<const float4 *>(src + (s0 + j) * kXBlock)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                r.x += (v[0].x + v[1].x) + (v[2].x + v[3].x);
                r.y += (v[0].y + v[1].y) + (v[2].y + v[3].y);
                r.z += (v[0].z + v[1].z) + (v[2].z + v[3].z);
                r.w += (v[0].w + v[1].w) + (v[2].w + v[3].w);
            }
            *reinterpret_cast<float4 *>(p.out + ((int64_t)q * H + h) * CSA2_D + 32 * c + g4) = r;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The largest cluster of attention CTAs this GPU schedules: 16 when a cluster
// of 16 (non-portable size) fits, else the portable 8 (asked once).
int attn_max_splits()
{
    static int cached = 0;
    if (cached) return cached;
    int m = 8;
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        const size_t smem = 1024 + kVBytes + kQBytes + kPBytes + (8 * 64 + 3 * 64) * 4 +
                            kMaxClusterSplits * 2 * 64 * 4 + 9 * 8 + 64;
        cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1);
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel, &cfg) == cudaSuccess && n > 0) m = 16;
    }
    cudaGetLastError();
    cached = m;
    return m;
}

cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st)
{
    // receive area: ceil(16 / S) chunk slots x S senders blocks, at most 24 (S = 12)
    // for S in 1 .. 12 and 16 blocks at S = 16; S in 13 .. 15 would need 26 .. 30
    static_assert(24 * kXBlock * 4 <= kVBytes + kQBytes, "merge area fits in the V and Q tiles");
    static_assert(kMaxClusterSplits * 64 * 4 <= kPBytes, "merge weights fit in the P tile");
    if (p.splits < 1 || p.splits > kMaxClusterSplits || (p.splits > 12 && p.splits < 16))
        return cudaErrorInvalidValue;
    if (p.splits > 8) cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    const size_t smem = 1024 + kVBytes + kQBytes + kPBytes + (8 * 64 + 3 * 64) * 4 +
                        kMaxClusterSplits * 2 * 64 * 4 + 9 * 8 + 64;
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const cudaError_t e = launch_k(attn_tc_kernel, dim3(p.splits, p.nq), dim3(kTcThreads), smem, st,
                                   (unsigned)p.splits, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa2
