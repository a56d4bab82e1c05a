// verify.cu -- multi-token verify attention over the quantized paged cache
// (a block of draft positions per request, causal within the block), on the
// fifth-generation tensor cores (tcgen05).
//
// The Lynx reading, section 4: decoding runs speculatively on the anchor-only
// draft cache, and once the residuals land a verify pass re-reads the refined
// cache for the drafted positions. Here that pass is attention of T_q query
// positions per request over the full (or anchor-only) reconstruction, where
// the last T_q tokens of the context are the drafted ones: position i sees the
// context up to and including draft token i. Dequantization stays on chip
// ("KV-cache quantization" explainer, "Bottom-right").
//
// With T_q x G query rows per KV head, Q.K^T and P.V are dense contractions.
// A CTA owns 128 query rows (the MMA's M) and a range of pages; per 32-token
// chunk:
//  - 16 decode warps expand the chunk's K and V codes (x = a + b L in fp32, split
//    into fp16 hi + lo) into shared-memory operand tiles in the tensor cores'
//    K-major swizzled layouts (K: rows of 128 channels, 128-byte swizzle; V
//    transposed: rows of 32 tokens, 64-byte swizzle);
//  - one thread issues the Q.K^T MMAs and another the P.V MMAs (tcgen05.mma):
//    S = Q.K^T into tensor memory with Q hi/lo
//    resident in tensor memory as the A operand (three products hi.hi + hi.lo
//    + lo.hi keep fp32-level accuracy), and after the softmax O += P.V with P
//    hi/lo in tensor memory as the A operand; only K and V^T are read from
//    shared memory by the tensor cores;
//  - softmax warps own one query row per thread: they read the row's 32
//    scores from tensor memory, apply the causal mask and the online softmax
//    (the reference moves only when a score passes it by 2^8; then O is
//    rescaled in tensor memory), and write P hi/lo back to tensor memory.
// Chunk codes arrive by bulk copy into a ring of slots, where the producer
// warp also turns each chunk's metadata into its affines once; every wait is
// bounded and sleeps in hardware.
// Split-K partials are merged by the decode path's combine kernel.
#include <cstddef>
#include <cuda_fp16.h>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr int kRow = kD / 2;                  // code bytes per token
constexpr int kPart = kD + 2;
constexpr int kRows = 128;                    // query rows per CTA (MMA M)
constexpr int kSoftWarps = 4, kDecWarps = 16;
constexpr int kMmaWarp = kSoftWarps + kDecWarps;      // issues the Q.K^T MMAs, owns the tensor memory
constexpr int kProdWarp = kMmaWarp + 1;                // issues the bulk copies, computes the chunk affines
constexpr int kPvWarp = kProdWarp + 1;                 // issues the P.V MMAs (kMmaWarp issues Q.K^T)
constexpr int kThreads = (kPvWarp + 1) * 32;
constexpr int kRing = 6;                      // chunk slots of codes in flight
constexpr int kBufs = 3;                      // K / V operand tiles and S buffers
constexpr int kPBufs = 2;                     // P buffers
constexpr uint32_t kWaitLimit = 1u << 18;   // waits of up to kSleepNs each: about 1 s in all
constexpr uint32_t kSleepNs = 4096;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kLevCopies = 32;                // one level-table copy per lane: conflict-free lookups
// tensor memory columns (fp32 / f16x2 words; lane = query row)
constexpr uint32_t kColS = 0;                           // S [buffer][Q.K_hi 32 tokens, Q_hi.K_lo 32 tokens]
constexpr uint32_t kColP = kColS + 64 * kBufs;          // P [buffer][hi 16 words, lo 16 words]
constexpr uint32_t kColO = kColP + 32 * kPBufs;         // O [128 channels]
constexpr uint32_t kColQ = kColO + kD;                  // Q hi [64 words], Q lo [64 words]
constexpr uint32_t kColsUsed = kColQ + kD;
constexpr uint32_t kTmemCols = 512;
static_assert(kColsUsed <= kTmemCols, "tensor memory columns");

// One chunk of K and V as it arrives (codes of 32 tokens, page and chunk metadata).
template <bool FULL>
struct Slot {
    uint8_t ka[kChunk * kRow], va[kChunk * kRow];
    uint8_t kr[FULL ? kChunk * kRow : 16], vr[FULL ? kChunk * kRow : 16];
    float kpm[2 * kD], vpm[2 * kD];           // page min, range
    uint16_t kcm[2 * kD], vcm[2 * kD];        // chunk mean, scale
    // chunk affines a = mn + rng mu and b = rng s, computed once per chunk:
    // K as [part][group][4] (channel 8 group + 4 part + i), V in channel order
    float kaf[2][16][4], kbf[2][16][4], vaf[kD], vbf[kD];
};

// Operand tiles. 128-byte swizzle: 16-byte piece c of a 128-byte row r sits at
// piece c ^ (r & 7), atoms of 8 rows x 128 bytes; 64-byte swizzle: piece c of
// a 64-byte row r at c ^ ((r >> 1) & 3). Every tile starts on 1024 bytes.
template <bool FULL>
struct Smem {
    uint8_t k[kBufs][2][2][kChunk * 128];     // K [buffer][k-atom][hi, lo][token][64 channels] (128B): per
                                              // k-atom, the hi rows then the lo rows form one 64-row operand
    uint8_t v[kBufs][2][kD * 64];             // V [buffer][hi, lo][channel][32 tokens] (64B)
    Slot<FULL> slot[kRing];
    float lev[256 * kLevCopies];              // level of a code byte (anchor: of a nibble), entry-major
    int slot_page[kRing];                     // physical page of the chunk in each slot (-1: invalid)
    uint32_t tmem;
    alignas(8) uint64_t ring_full[kRing], slot_free[kRing];
    uint64_t k_full[kBufs], v_full[kBufs], s_full[kBufs], s_free[kBufs], pv_done[kBufs], p_full[kPBufs];
    uint64_t drained, drained_pv;
    uint64_t aff_ready[kRing];                // the slot's chunk affines are written
};

__device__ __forceinline__ uint32_t sw128(int row, int byte)
{
    return (uint32_t)(row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15)));
}
__device__ __forceinline__ uint32_t sw64(int row, int byte)
{
    return (uint32_t)(row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3)) << 4) | (byte & 15)));
}

// Shared-memory matrix descriptor of a K-major swizzled operand (SBO = bytes
// between 8-row groups; layout 2 = 128-byte swizzle, 4 = 64-byte swizzle).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t sbo, uint32_t layout)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)layout << 61);
}

// Instruction descriptor: f32 accumulator, f16 A and B, both K-major, N, M.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) (+)= A (tensor memory: row i in lane i, two f16 per
// column) x B (shared-memory descriptor).
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Bounded wait that sleeps in hardware: each try_wait suspends the thread
// until the phase completes or the hinted time (ns) passes, so waiting
// threads take no issue slots from the ones doing work.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(ok)
                     : "r"(smem_u32(bar)), "r"(parity), "r"(kSleepNs)
                     : "memory");
        if (ok)
            return true;
    }
    return false;
}


__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7F800000); }

__device__ __forceinline__ float exp2_sm(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (x0, x1) -> fp16 pairs hi and lo with hi + lo = (x0, x1) to ~22 bits. The
// remainders x - hi are exact in fp32; each comes from one mixed-precision
// multiply-add (fp16 operands, fp32 addend and result), with no separate
// widening of hi.
__device__ __forceinline__ void split2(float2 x, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(x.x, x.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    float r0, r1;
    asm("{\n\t.reg .b16 h0, h1, m1;\n\tmov.b32 {h0, h1}, %2;\n\tmov.b16 m1, 0xBC00;\n\t"
        "fma.rn.f32.f16 %0, h0, m1, %3;\n\tfma.rn.f32.f16 %1, h1, m1, %4;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "r"(hi), "f"(x.x), "f"(x.y));
    const __half2 l = __floats2half2_rn(r0, r1);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Chunk affines a = mn + rng mu and b = rng s of the four channels d .. d + 3
// (two packed pairs; each lane of the packed operations is one IEEE operation).
__device__ __forceinline__ void affine4(const float *pm, const uint16_t *cm, int d, float4 &a, float4 &b)
{
    const float4 mn = *reinterpret_cast<const float4 *>(pm + d), rg = *reinterpret_cast<const float4 *>(pm + kD + d);
    const uint2 mu = *reinterpret_cast<const uint2 *>(cm + d), sc = *reinterpret_cast<const uint2 *>(cm + kD + d);
    const float2 a01 = __ffma2_rn(make_float2(rg.x, rg.y), __half22float2(*reinterpret_cast<const __half2 *>(&mu.x)),
                                  make_float2(mn.x, mn.y));
    const float2 a23 = __ffma2_rn(make_float2(rg.z, rg.w), __half22float2(*reinterpret_cast<const __half2 *>(&mu.y)),
                                  make_float2(mn.z, mn.w));
    const float2 b01 = __fmul2_rn(make_float2(rg.x, rg.y), __half22float2(*reinterpret_cast<const __half2 *>(&sc.x)));
    const float2 b23 = __fmul2_rn(make_float2(rg.z, rg.w), __half22float2(*reinterpret_cast<const __half2 *>(&sc.y)));
    a = make_float4(a01.x, a01.y, a23.x, a23.y);
    b = make_float4(b01.x, b01.y, b23.x, b23.y);
}

// Levels of the two channels of a code byte (anchor byte a8, residual byte
// r8), the channel in the nibble at bit `sh` first (sh = 0: low channel
// first; sh = 4: high channel first). Full: entry (anchor nibble << 4) |
// residual nibble. Anchor: every entry e holds the level of nibble e & 15, so
// a byte shifted right indexes its upper nibble's channel directly. Table
// copies interleave: entry e of this lane's copy is lv[kLevCopies e].
template <bool FULL>
__device__ __forceinline__ float2 levels(const float *lv, uint32_t a8, uint32_t r8, uint32_t sh = 0)
{
    const uint32_t sh2 = 4u - sh;
    if (FULL)
        return make_float2(lv[kLevCopies * ((((a8 >> sh) & 0x0Fu) << 4) | ((r8 >> sh) & 0x0Fu))],
                           lv[kLevCopies * ((((a8 >> sh2) & 0x0Fu) << 4) | ((r8 >> sh2) & 0x0Fu))]);
    return make_float2(lv[kLevCopies * (a8 >> sh)], lv[kLevCopies * (a8 >> sh2)]);
}

// K of one chunk into the tiles kt[k-atom][hi/lo] (rows = tokens, 128-byte
// rows of 64 channels). Decode thread u (0..511) takes the 16-byte piece of
// channels 8 g .. 8 g + 7, g = u % 16, of token u / 16: one 32-bit code load
// per plane and one 16-byte store per tile (the 8 lanes of a store phase
// write one whole row).
template <bool FULL>
__device__ __forceinline__ void decode_k(const Slot<FULL> &sl, bool valid, const float *lv,
                                         uint8_t (&kt)[2][2][kChunk * 128], int u)
{
    const int g = u & 15, t = u >> 4, ka = g >> 3, piece = g & 7;
    const float4 a0 = *reinterpret_cast<const float4 *>(sl.kaf[0][g]), a1 = *reinterpret_cast<const float4 *>(sl.kaf[1][g]);
    const float4 b0 = *reinterpret_cast<const float4 *>(sl.kbf[0][g]), b1 = *reinterpret_cast<const float4 *>(sl.kbf[1][g]);
    const float2 aa[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(a1.x, a1.y), make_float2(a1.z, a1.w)};
    const float2 bb[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
    uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
    if (valid) {
        const uint32_t a4 = *reinterpret_cast<const uint32_t *>(sl.ka + t * kRow + 4 * g);
        const uint32_t r4 = FULL ? *reinterpret_cast<const uint32_t *>(sl.kr + t * kRow + 4 * g) : 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            split2(__ffma2_rn(bb[i], levels<FULL>(lv, (a4 >> (8 * i)) & 0xFFu, (r4 >> (8 * i)) & 0xFFu), aa[i]), hi[i],
                   lo[i]);
    }
    const uint32_t off = sw128(t, 16 * piece);
    *reinterpret_cast<uint4 *>(&kt[ka][0][off]) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4 *>(&kt[ka][1][off]) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// V of one chunk, transposed, into the tiles vt[hi/lo] (rows = channels,
// 64-byte rows of 32 tokens). Decode thread u takes channel pair pr = u % 64
// of the four tokens 4 o .. 4 o + 3, where o is the warp's quad u / 64,
// exchanged with its neighbour (o ^ 1) by lanes with bit 3 of pr set; lanes
// with bit 2 of pr set store row 2 pr + 1 first. Together the 16 lanes of an
// 8-byte store phase cover all 32 banks.
template <bool FULL>
__device__ __forceinline__ void decode_v(const Slot<FULL> &sl, bool valid, const float *lv, uint8_t (&vt)[2][kD * 64],
                                         int u)
{
    const int pr = u & 63, sw = (pr >> 2) & 1, o = (u >> 6) ^ ((pr >> 3) & 1);
    const uint32_t sh = 4u * (uint32_t)sw;
    float2 aa = *reinterpret_cast<const float2 *>(sl.vaf + 2 * pr), bb = *reinterpret_cast<const float2 *>(sl.vbf + 2 * pr);
    if (sw) {
        aa = make_float2(aa.y, aa.x);
        bb = make_float2(bb.y, bb.x);
    }
    float2 x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int t = 4 * o + e;
        x[e] = make_float2(0.0f, 0.0f);
        if (valid) {
            const uint32_t a8 = sl.va[t * kRow + pr];
            const uint32_t r8 = FULL ? sl.vr[t * kRow + pr] : 0u;
            x[e] = __ffma2_rn(bb, levels<FULL>(lv, a8, r8, sh), aa);
        }
    }
    uint32_t h0[2], h1[2], l0[2], l1[2];     // rows 2 pr + sw and 2 pr + 1 - sw; word j = tokens 4 o + 2 j, + 1
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        split2(make_float2(x[2 * j].x, x[2 * j + 1].x), h0[j], l0[j]);
        split2(make_float2(x[2 * j].y, x[2 * j + 1].y), h1[j], l1[j]);
    }
    const uint32_t o0 = sw64(2 * pr + sw, 8 * o), o1 = sw64(2 * pr + 1 - sw, 8 * o);
    *reinterpret_cast<uint2 *>(&vt[0][o0]) = make_uint2(h0[0], h0[1]);
    *reinterpret_cast<uint2 *>(&vt[0][o1]) = make_uint2(h1[0], h1[1]);
    *reinterpret_cast<uint2 *>(&vt[1][o0]) = make_uint2(l0[0], l0[1]);
    *reinterpret_cast<uint2 *>(&vt[1][o1]) = make_uint2(l1[0], l1[1]);
}

template <bool FULL>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(VerifyArgs a, LevelTable levt)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem<FULL> &sm = *reinterpret_cast<Smem<FULL> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, kvh = blockIdx.y / a.RB, rb = blockIdx.y % a.RB, b = blockIdx.z;
    const int G = a.G, Tq = a.Tq;
    const int64_t T = (int64_t)a.pool_pages * kPage;
    if (smem_u32(smem_raw) & 1023u) {        // the swizzled tiles need a 1024-byte aligned window
        if (a.dev_err && tid == 0)
            atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
        return;
    }

    // ---- set-up: level table, barriers, tensor memory ---------------------
    for (int i = tid; i < 256 * kLevCopies; i += kThreads) {
        const int e = i / kLevCopies;
        sm.lev[i] = FULL ? levt.full[e] : levt.anchor[e & 15];
    }
    if (tid == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&sm.ring_full[s], 1);
            mbar_init(&sm.slot_free[s], kDecWarps);
        }
        for (int s = 0; s < kBufs; ++s) {
            mbar_init(&sm.k_full[s], kDecWarps);
            mbar_init(&sm.v_full[s], kDecWarps);
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.s_free[s], kSoftWarps);
            mbar_init(&sm.pv_done[s], 1);
        }
        for (int s = 0; s < kPBufs; ++s)
            mbar_init(&sm.p_full[s], kSoftWarps);
        mbar_init(&sm.drained, 1);
        mbar_init(&sm.drained_pv, 1);
        for (int s = 0; s < kRing; ++s)
            mbar_init(&sm.aff_ready[s], 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {                  // the MMA warp owns the tensor memory
        tmem_alloc(&sm.tmem, kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    int ctx = a.ctx[b];
    if (ctx < 0 || ctx > a.max_pages * kPage) {
        if (a.dev_err && split == 0 && blockIdx.y == 0 && tid == 0)
            atomicOr(a.dev_err, LYNX_DEVERR_CTX);
        ctx = min(max(ctx, 0), a.max_pages * kPage);
    }
    // softmax thread: query row rl of this block (draft position pos, head h)
    const int rl = 32 * (warp & 3) + lane, r = rb * kRows + rl;
    const bool rowok = warp < kSoftWarps && r < Tq * G;
    const int pos = rowok ? r / G : 0, h = kvh * G + (rowok ? r % G : 0);
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    if (warp < kSoftWarps) {                 // Q (scaled to log2 units) hi / lo and O = 0 into tensor memory
        const float qscale = a.sm_scale * kLog2e;
        const uint16_t *qrow = a.q + (((int64_t)b * Tq + pos) * a.Hq + h) * kD;
#pragma unroll 1
        for (int grp = 0; grp < 8; ++grp) {  // 16 channels (8 words) at a time
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int w8 = 0; w8 < 2; ++w8) {
                const uint4 w = rowok ? *reinterpret_cast<const uint4 *>(qrow + 16 * grp + 8 * w8) : make_uint4(0, 0, 0, 0);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    split2(make_float2(bf16_lo(ws[i]) * qscale, bf16_hi(ws[i]) * qscale), hi[4 * w8 + i], lo[4 * w8 + i]);
            }
            tmem_st8(trow + kColQ + 8 * grp, hi);
            tmem_st8(trow + kColQ + 64 + 8 * grp, lo);
        }
        float z[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            z[k] = 0.0f;
#pragma unroll 1
        for (int k = 0; k < 8; ++k)
            tmem_st16f(trow + kColO + 16 * k, z);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const int p_begin = split * a.pages_per_split;
    const int p_end = min(p_begin + a.pages_per_split, a.max_pages);
    const int p_live = min(p_end, (ctx + kPage - 1) / kPage);
    const int np = max(p_live - p_begin, 0);
    const int nch = kNChunk * np;
    auto phys_of = [&](int i) -> int {
        const int p = a.page_table[(int64_t)b * a.max_pages + p_begin + i];
        return (p >= 0 && p < a.pool_pages) ? p : -1;
    };
    bool timed_out = false;

    if (warp == kProdWarp) {
        // ---- producer: chunk codes into the ring of slots by bulk copy (lane
        // 0), and the affines of the chunk before (whole warp, once the copies
        // of that chunk have landed) --------------------------------------------
        int cur_i = -1, cur_p = -1;
        auto affines = [&](int c) -> bool {  // whole warp; lane l takes channels 4 l .. 4 l + 3
            const int s = c % kRing;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_sleep(&sm.ring_full[s], (uint32_t)((c / kRing) & 1), kWaitLimit)))
                return false;
            Slot<FULL> &sl = sm.slot[s];
            float4 ka4, kb4, va4, vb4;
            affine4(sl.kpm, sl.kcm, 4 * lane, ka4, kb4);
            affine4(sl.vpm, sl.vcm, 4 * lane, va4, vb4);
            *reinterpret_cast<float4 *>(sl.kaf[lane & 1][lane >> 1]) = ka4;
            *reinterpret_cast<float4 *>(sl.kbf[lane & 1][lane >> 1]) = kb4;
            *reinterpret_cast<float4 *>(sl.vaf + 4 * lane) = va4;
            *reinterpret_cast<float4 *>(sl.vbf + 4 * lane) = vb4;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.aff_ready[s]);
            return true;
        };
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int s = c % kRing, i = c >> 3, j = c & 7;
            // slot s was last decoded for chunk c - kRing
            if (c >= kRing &&
                !__all_sync(0xFFFFFFFFu,
                            mbar_wait_sleep(&sm.slot_free[s], (uint32_t)(((c - kRing) / kRing) & 1), kWaitLimit))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                if (i != cur_i) {            // one page-table read a page
                    cur_i = i;
                    cur_p = phys_of(i);
                    if (cur_p < 0 && a.dev_err)
                        atomicOr(a.dev_err, LYNX_DEVERR_PAGE);
                }
                Slot<FULL> &sl = sm.slot[s];
                uint64_t *bar = &sm.ring_full[s];
                sm.slot_page[s] = cur_p;
                if (cur_p < 0) {
                    mbar_arrive(bar);
                } else {
                    fence_proxy_async_smem();    // the decoders' reads of the slot come before the copies' writes
                    const int64_t rows = ((int64_t)kvh * T + (int64_t)cur_p * kPage + j * kChunk) * kRow;
                    const int64_t pmo = ((int64_t)kvh * a.pool_pages + cur_p) * (2 * kD);
                    const int64_t cmo = (((int64_t)kvh * a.pool_pages + cur_p) * kNChunk + j) * (2 * kD);
                    mbar_arrive_expect_tx(bar, (FULL ? 4u : 2u) * kChunk * kRow + 2 * (2 * kD * 4) + 2 * (2 * kD * 2));
                    bulk_g2s(sl.ka, a.ka + rows, kChunk * kRow, bar);
                    bulk_g2s(sl.va, a.va + rows, kChunk * kRow, bar);
                    if (FULL) {
                        bulk_g2s(sl.kr, a.kr + rows, kChunk * kRow, bar);
                        bulk_g2s(sl.vr, a.vr + rows, kChunk * kRow, bar);
                    }
                    bulk_g2s(sl.kpm, a.kpm + pmo, 2 * kD * 4, bar);
                    bulk_g2s(sl.vpm, a.vpm + pmo, 2 * kD * 4, bar);
                    bulk_g2s(sl.kcm, a.kcm + cmo, 2 * kD * 2, bar);
                    bulk_g2s(sl.vcm, a.vcm + cmo, 2 * kD * 2, bar);
                }
            }
            __syncwarp();
            if (c >= 1 && !(ok = affines(c - 1)))
                break;
        }
        // the last chunk's affines; every copy issued has then landed (bounded)
        if (ok && nch > 0)
            ok = affines(nch - 1);
        timed_out = !ok;
    } else if (warp >= kSoftWarps && warp < kMmaWarp) {
        // ---- decode warps ----------------------------------------------------
        const int u = 32 * (warp - kSoftWarps) + lane;
        const float *lv = sm.lev + lane;
        for (int c = 0; c < nch; ++c) {
            const int s = c % kRing, buf = c % kBufs;
            const uint32_t prev = (uint32_t)(((c - kBufs) / kBufs) & 1);
            // codes in; K tile `buf` last read by the Q.K^T of chunk c - kBufs
            bool ok = mbar_wait_sleep(&sm.ring_full[s], (uint32_t)((c / kRing) & 1), kWaitLimit) &&
                      mbar_wait_sleep(&sm.aff_ready[s], (uint32_t)((c / kRing) & 1), kWaitLimit);
            if (ok && c >= kBufs)
                ok = mbar_wait_sleep(&sm.s_full[buf], prev, kWaitLimit);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const bool valid = sm.slot_page[s] >= 0;
            decode_k<FULL>(sm.slot[s], valid, lv, sm.k[buf], u);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.k_full[buf]);
            // V tile `buf` last read by the P.V of chunk c - kBufs
            if (c >= kBufs && !__all_sync(0xFFFFFFFFu, mbar_wait_sleep(&sm.pv_done[buf], prev, kWaitLimit))) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            decode_v<FULL>(sm.slot[s], valid, lv, sm.v[buf], u);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.v_full[buf]);
                mbar_arrive(&sm.slot_free[s]);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---- Q.K^T issuer: S of chunk c as soon as its K tile is decoded and
        // S buffer c % kBufs has been read by the softmax
        if (lane == 0 && nch > 0) {
            // Q_hi against the stacked [K_hi; K_lo] (64 rows) gives both cross
            // terms in one product: columns 0-31 Q_hi.K_hi, 32-63 Q_hi.K_lo;
            // Q_lo.K_hi accumulates into columns 0-31
            constexpr uint32_t id64 = idesc_f16(kRows, 2 * kChunk), id32 = idesc_f16(kRows, kChunk);
            const uint32_t tQh = tmem + kColQ, tQl = tmem + kColQ + kD / 2;
            const uint32_t k0 = smem_u32(sm.k);
            for (int c = 0; c < nch; ++c) {
                const int buf = c % kBufs;
                if (!mbar_wait_sleep(&sm.k_full[buf], (uint32_t)((c / kBufs) & 1), kWaitLimit) ||
                    (c >= kBufs &&
                     !mbar_wait_sleep(&sm.s_free[buf], (uint32_t)(((c - kBufs) / kBufs) & 1), kWaitLimit))) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t tS = tmem + kColS + 64u * buf;
                const uint32_t kb = k0 + (uint32_t)buf * (uint32_t)sizeof(sm.k[0]);
#pragma unroll
                for (int st = 0; st < 8; ++st) {  // 16 channels a step: 8 columns of Q, 32 bytes of a K row
                    const uint64_t kd = sdesc(kb + (uint32_t)(st >> 2) * (uint32_t)sizeof(sm.k[0][0]) + 32 * (st & 3), 1024, 2);
                    umma_ts(tS, tQh + 8 * st, kd, id64, st > 0 ? 1u : 0u);
                    umma_ts(tS, tQl + 8 * st, kd, id32, 1u);
                }
                umma_commit(&sm.s_full[buf]);
            }
            // every MMA this thread issued must finish before the tensor memory
            // is freed (the commit tracks all of them; bounded)
            umma_commit(&sm.drained);
            mbar_wait_sleep(&sm.drained, 0u, kWaitLimit);
        }
    } else if (warp == kPvWarp) {
        // ---- P.V issuer: O += P.V of chunk c as soon as its P is written and
        // its V tile decoded
        if (lane == 0 && nch > 0) {
            constexpr uint32_t idpv = idesc_f16(kRows, kD);
            const uint32_t tO = tmem + kColO, v0 = smem_u32(sm.v);
            for (int c = 0; c < nch; ++c) {
                const int buf = c % kBufs, pb = c % kPBufs;
                if (!mbar_wait_sleep(&sm.p_full[pb], (uint32_t)((c / kPBufs) & 1), kWaitLimit) ||
                    !mbar_wait_sleep(&sm.v_full[buf], (uint32_t)((c / kBufs) & 1), kWaitLimit)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t tPh = tmem + kColP + 32u * pb, tPl = tPh + 16;
                const uint32_t vb = v0 + (uint32_t)buf * (uint32_t)sizeof(sm.v[0]);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {  // 16 tokens a step: 8 columns of P, 32 bytes of a V^T row
                    const uint64_t vh = sdesc(vb + 32 * kk, 512, 4);
                    const uint64_t vl = sdesc(vb + (uint32_t)sizeof(sm.v[0][0]) + 32 * kk, 512, 4);
                    umma_ts(tO, tPh + 8 * kk, vh, idpv, 1u);
                    umma_ts(tO, tPh + 8 * kk, vl, idpv, 1u);
                    umma_ts(tO, tPl + 8 * kk, vh, idpv, 1u);
                }
                umma_commit(&sm.pv_done[buf]);
            }
            umma_commit(&sm.drained_pv);
            mbar_wait_sleep(&sm.drained_pv, 0u, kWaitLimit);
        }
    } else {
        // ---- softmax warps: one query row per thread -------------------------
        const int nvis = rowok ? ctx - Tq + pos + 1 : 0;           // tokens this draft position sees
        // chunks wholly inside every row's view need no mask
        const int vis_all = ctx - Tq + 1;
        int vpage = -1;
        bool pvalid = false;
        float m_run = neg_inf(), l_run = 0.0f;
        for (int c = 0; c < nch; ++c) {
            const int buf = c % kBufs, pb = c % kPBufs;
            if (!mbar_wait_sleep(&sm.s_full[buf], (uint32_t)((c / kBufs) & 1), kWaitLimit)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            float S[32];                     // Q_hi.K_hi + Q_lo.K_hi, plus Q_hi.K_lo, 16 columns at a time
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float s0[16], s1[16];
                tmem_ld16(trow + kColS + 64 * buf + 16 * hf, s0);
                tmem_ld16(trow + kColS + 64 * buf + 32 + 16 * hf, s1);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    S[16 * hf + k] = s0[k] + s1[k];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.s_free[buf]);
            const int t0 = (p_begin + (c >> 3)) * kPage + (c & 7) * kChunk;
            if ((c >> 3) != vpage) {         // one page-table read a page
                vpage = c >> 3;
                pvalid = phys_of(vpage) >= 0;
            }
            const bool valid = pvalid;
            float mx = neg_inf();
            if (valid && t0 + kChunk <= vis_all) {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    mx = fmaxf(mx, S[k]);
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    S[k] = (!valid || t0 + k >= nvis) ? neg_inf() : S[k];
                    mx = fmaxf(mx, S[k]);
                }
            }
            // the reference moves only when a score passes it by 2^8 (weights
            // up to 2^8 are exact in fp32 and fine in fp16)
            const bool up = mx > m_run + 8.0f;
            if (__any_sync(0xFFFFFFFFu, up)) {
                // rare: rescale this row's output, complete up to chunk c - 1
                if (c >= 1 && !mbar_wait_sleep(&sm.pv_done[(c - 1) % kBufs], (uint32_t)(((c - 1) / kBufs) & 1),
                                                  kWaitLimit)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const float alpha = up ? (m_run == neg_inf() ? 0.0f : exp2_sm(m_run - mx)) : 1.0f;
                if (up) {
                    m_run = mx;
                    l_run *= alpha;
                }
#pragma unroll 1
                for (int k = 0; k < 8; ++k) {    // 16 columns at a time (the scores stay live)
                    float o[16];
                    tmem_ld16(trow + kColO + 16 * k, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[e] *= alpha;
                    tmem_st16f(trow + kColO + 16 * k, o);
                }
                tmem_wait_st();
            }
            // P buffer `pb` was last read by the P.V of chunk c - kPBufs
            if (c >= kPBufs && !mbar_wait_sleep(&sm.pv_done[(c - kPBufs) % kBufs],
                                                  (uint32_t)(((c - kPBufs) / kBufs) & 1), kWaitLimit)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            // m_run is -inf only while every score so far (this chunk's too) is
            // masked: then every weight is exp2(-inf) = 0
            const float m_eff = m_run == neg_inf() ? 0.0f : m_run;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {     // P hi words 8 hf .. + 7, then the lo words
                uint32_t ph[8], pl[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int c2 = 2 * (8 * hf + k);
                    const float p0 = exp2_sm(S[c2] - m_eff), p1 = exp2_sm(S[c2 + 1] - m_eff);
                    l_run += p0 + p1;
                    split2(make_float2(p0, p1), ph[k], pl[k]);
                }
                tmem_st8(trow + kColP + 32 * pb + 8 * hf, ph);
                tmem_st8(trow + kColP + 32 * pb + 16 + 8 * hf, pl);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.p_full[pb]);
        }
        // ---- this range's partial of the row
        if (!timed_out && nch > 0 &&
            !mbar_wait_sleep(&sm.pv_done[(nch - 1) % kBufs], (uint32_t)(((nch - 1) / kBufs) & 1), kWaitLimit))
            timed_out = true;
        tc_fence_after();
        float *part = a.part + ((((int64_t)b * Tq + pos) * a.Hq + h) * a.n_splits + split) * kPart;
#pragma unroll 1
        for (int k = 0; k < 8; ++k) {
            float o[16];
            tmem_ld16(trow + kColO + 16 * k, o);
            tmem_wait_ld();
            if (rowok)                       // a partial is 130 floats: 8-byte aligned
#pragma unroll
                for (int e = 0; e < 16; e += 2)
                    *reinterpret_cast<float2 *>(part + 16 * k + e) = make_float2(o[e], o[e + 1]);
        }
        if (rowok) {
            part[kD] = m_run;
            part[kD + 1] = l_run;
        }
    }
    if (timed_out && a.dev_err)
        atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool FULL>
cudaError_t run(const VerifyArgs &a, cudaStream_t s)
{
    static_assert(sizeof(Smem<FULL>) <= 227 * 1024, "shared memory per CTA");
    // bulk copies land on 16-byte boundaries; swizzled tiles start on 1024 bytes
    static_assert(sizeof(Slot<FULL>) % 16 == 0 && offsetof(Slot<FULL>, kpm) % 16 == 0 &&
                      offsetof(Slot<FULL>, vpm) % 16 == 0 && offsetof(Slot<FULL>, kcm) % 16 == 0 &&
                      offsetof(Slot<FULL>, vcm) % 16 == 0 && offsetof(Slot<FULL>, vr) % 16 == 0,
                  "slot layout");
    static_assert(offsetof(Smem<FULL>, k) % 1024 == 0 && offsetof(Smem<FULL>, v) % 1024 == 0 &&
                      offsetof(Smem<FULL>, slot) % 16 == 0,
                  "tile layout");
    const size_t smem = sizeof(Smem<FULL>);
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<FULL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)a.n_splits, (unsigned)(a.H * a.RB), (unsigned)a.B);
    verify_kernel<FULL><<<grid, kThreads, smem, s>>>(a, host_tables().lev);
    return cudaGetLastError();
}

} // namespace

int verify_row_blocks(int draft, int G) { return (draft * G + kRows - 1) / kRows; }

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s)
{
    if (a.B == 0 || a.Hq == 0 || a.Tq == 0)
        return cudaSuccess;
    cudaError_t e = a.full ? run<true>(a, s) : run<false>(a, s);
    if (e != cudaSuccess)
        return e;
    AttnArgs c = {};
    c.part = a.part;
    c.out = a.out;
    c.B = a.B * a.Tq;
    c.Hq = a.Hq;
    c.n_splits = a.n_splits;
    return launch_attn_combine(c, s);
}

} // namespace lynx
