// attn_mma.cu -- fused-dequant paged decode attention on the tensor cores
// (K4, groups of up to 16 query heads per KV head).
//
// One decode step over the quantized paged cache ("KV-cache quantization"
// explainer, "Bottom-right": the compact cache is read as is and expanded
// only in registers, inside Q.K^T and P.V). Anchor mode reads the anchor
// planes only (the draft cache of the Lynx reading, section 4); full mode adds
// the residual planes.
//
// Factorisation. Every element of chunk j (32 tokens) and channel d decodes
// as x = a_jd + b_jd * L(code) with a = mn + rng mu, b = rng s and L an exact
// fp16 level value. Hence, per chunk,
//   s_t  = beta_j + sum_d (q_d b_jd) L_td,         beta_j = sum_d q_d a_jd
//   o_d += sum_j [ a_jd sum_{t in j} p_t + b_jd sum_{t in j} p_t L_td ],
// so the tensor-core operands on the cache side are the level values
// themselves (no rounding), and the dense operand (q b, or p) is split into an
// fp16 hi/lo pair to keep fp32-level accuracy (mma.sync m16n8k16, fp32
// accumulation).
//
// Work: a CTA per (page range, KV head, request). Pages arrive by bulk copy
// into two shared-memory stages; V codes are re-laid out once per page with an
// 8x8 nibble transpose (token pairs per byte, swizzled) so that each P.V B
// fragment is one 16-bit load. Two variants:
//  - groups of up to 8 query heads: 8 warps, warp j owns chunk j of every
//    page; the MMA rows are the 8 heads' hi parts over their lo parts, so one
//    MMA carries both halves of the split;
//  - groups of up to 16: 16 warps, warps j and j + 8 share chunk j and each
//    decodes half of the channels (Q.K^T halves are summed through shared
//    memory, P.V covers its own channels); MMA rows are the 16 heads, hi and lo
//    in two MMAs; each warp runs the softmax of one head row and the pair swaps
//    the resulting P fragments.
// The chunks' running (max, sum, output) are merged in shared memory into one
// partial per query head; a second kernel merges the partials of the ranges.
#include <cuda_fp16.h>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr uint32_t kPlane = kPage * kD / 2;   // 16 KiB
constexpr int kPart = kD + 2;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <bool FULL>
struct Stage {
    uint8_t ka[kPlane];
    uint8_t va[kPlane];
    uint8_t kr[FULL ? kPlane : 16];
    uint8_t vr[FULL ? kPlane : 16];
    float kpm[2 * kD];
    float vpm[2 * kD];
    uint16_t kcm[kNChunk * 2 * kD];
    uint16_t vcm[kNChunk * 2 * kD];
};

template <bool FULL>
struct Smem {
    Stage<FULL> st[2];
    uint8_t vta[kD * (kPage / 2)];            // V anchors: byte k of channel c holds tokens 2k, 2k+1 (swizzled)
                                              // (V residuals, same layout, go to the stage's va slot)
    // chunk affines of channel pairs: (a_2i, a_2i+1, b_2i, b_2i+1), K's b times 2^-guard
    float4 kab[kNChunk][kD / 2];
    float4 vab[kNChunk][kD / 2];
    float qs[16][kD + 8];                     // the group's queries times sm_scale log2(e); unused rows 0
                                              // (rows padded: 8 heads x 4 lanes read distinct banks)
    float xch[kNChunk][19][32];               // Q.K^T halves exchanged between the two warps of a chunk;
                                              // row 18: per quad, each warp's sum of P and rescale
                                              // (the P fragments are swapped through the stage's consumed
                                              // V plane: 8 pairs x 2 warps x 8 words x 32 lanes = 16 KiB)
    // level table, one copy per lane (conflict-free lookups): anchor mode maps a
    // byte of two anchors to the half2 of their levels, full mode a code byte
    // (A << 4 | r) to the fp16 level
    uint32_t lut[FULL ? 256 * 32 / 2 : 256 * 32];
    int guard;                                // exponent keeping q b inside fp16 for this page
    float qmax;
    alignas(8) uint64_t bar[2];
};

struct Merge {                                // overlays the stages after the page loop
    float m[kNChunk][16];                     // per chunk (warp or warp pair) and query head
    float l[kNChunk][16];
    float o[kNChunk][16][kD];
};

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x0, x1) -> fp16 pairs hi and lo with hi + lo = (x0, x1) to ~22 bits.
__device__ __forceinline__ void split2(float2 x, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(x.x, x.y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x.x - hf.x, x.y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Transposed V planes: channel c owns 128 bytes; its 8-byte group g holds the
// token pairs 8g + {0, 4, 1, 5, 2, 6, 3, 7} (so pairs k and k+4 are adjacent),
// and the groups of each channel are rotated by c + c/8 so that 8 consecutive
// channels (a P.V fragment load) and 16 channels 8 apart (a transpose store)
// fall in distinct banks. vt_group() is the byte offset of group g of channel c.
__device__ __forceinline__ int vt_group(int c, int g)
{
    return c * (kPage / 2) + (((g + c + (c >> 3)) & 15) << 3);
}

// 8x8 transpose of 4-bit elements: w[r] nibble i  ->  w[i] nibble r.
__device__ __forceinline__ void transpose8x8_nibbles(uint32_t (&w)[8])
{
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint32_t a = w[r], b = w[r + 4];
        w[r] = __byte_perm(a, b, 0x5410u);
        w[r + 4] = __byte_perm(a, b, 0x7632u);
    }
#pragma unroll
    for (int r = 0; r < 8; r += (r & 1) ? 3 : 1) {   // r = 0, 1, 4, 5
        const uint32_t a = w[r], b = w[r + 2];
        w[r] = __byte_perm(a, b, 0x6240u);
        w[r + 2] = __byte_perm(a, b, 0x7351u);
    }
#pragma unroll
    for (int r = 0; r < 8; r += 2) {
        const uint32_t a = w[r], b = w[r + 1];
        w[r] = (a & 0x0F0F0F0Fu) | ((b << 4) & 0xF0F0F0F0u);
        w[r + 1] = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
    }
}

// One plane of V codes ([256 tokens][64 bytes]) into the transposed layout:
// block (word wp = channels 8wp..8wp+7, group g, half) = 8 rows x 8 channels.
template <int NT>
__device__ __forceinline__ void transpose_v(const uint8_t *src, uint8_t *dst, int tid)
{
    constexpr int kRow[8] = {0, 1, 8, 9, 2, 3, 10, 11};
    for (int blk = tid; blk < 512; blk += NT) {
        const int wp = blk & 15, half = (blk >> 4) & 1, g = blk >> 5;
        const int base = 16 * g + 4 * half;
        uint32_t w[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            w[r] = *reinterpret_cast<const uint32_t *>(src + (base + kRow[r]) * (kD / 2) + 4 * wp);
        transpose8x8_nibbles(w);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint32_t *>(dst + vt_group(8 * wp + i, g) + 4 * half) = w[i];
    }
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7F800000); }

__device__ __forceinline__ void pair_sync(int j)
{
    asm volatile("bar.sync %0, 64;" ::"r"(1 + j) : "memory");
}

template <int NW, bool FULL>
__global__ void __launch_bounds__(NW * 32, 1) attn_mma_kernel(AttnArgs a, LevelTable lev)
{
    constexpr int NT = NW * 32;
    constexpr bool PAIR = NW == 16;         // two warps per chunk, split by channels
    constexpr int NH = PAIR ? 2 : 1;        // query heads (MMA row pairs) per lane
    constexpr int NTO = PAIR ? 8 : 16;      // output n-tiles per warp
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<FULL> &sm = *reinterpret_cast<Smem<FULL> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = lane >> 2, q = lane & 3;
    const int j = warp & 7;                 // chunk of this warp
    const int hc = warp >> 3;               // PAIR: channels 64hc .. 64hc + 63, softmax of head row n + 8hc
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = a.G;
    const int64_t T = (int64_t)a.pool_pages * kPage;

    // ---- per-CTA set-up ------------------------------------------------
    if (FULL) {
        uint16_t *lut16 = reinterpret_cast<uint16_t *>(sm.lut);
        for (int i = tid; i < 256 * 32; i += NT)
            lut16[i] = __half_as_ushort(__float2half_rn(lev.full[i >> 5]));
    } else {
        for (int i = tid; i < 256 * 32; i += NT) {
            const int e = i >> 5;
            const __half2 h = __floats2half2_rn(lev.anchor[e & 15], lev.anchor[e >> 4]);
            sm.lut[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
    }
    const float qscale = a.sm_scale * kLog2e;
    float lq = 0.0f;
    for (int i = tid; i < 16 * kD; i += NT) {
        const int h = i / kD, d = i % kD;
        float v = 0.0f;
        if (h < G)
            v = __uint_as_float((uint32_t)a.q[((int64_t)b * a.Hq + g * G + h) * kD + d] << 16) * qscale;
        sm.qs[h][d] = v;
        lq = fmaxf(lq, fabsf(v));
    }
    if (tid == 0) {
        sm.qmax = 0.0f;
        sm.guard = 0;
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    atomicMax(reinterpret_cast<int *>(&sm.qmax), __float_as_int(lq));

    int ctx = a.ctx[b];
    if (ctx < 0 || ctx > a.max_pages * kPage) {
        if (a.dev_err && split == 0 && g == 0 && tid == 0)
            atomicOr(a.dev_err, LYNX_DEVERR_CTX);
        ctx = min(max(ctx, 0), a.max_pages * kPage);
    }
    const uint8_t *ka = a.ka + (int64_t)g * T * (kD / 2);
    const uint8_t *va = a.va + (int64_t)g * T * (kD / 2);
    const uint8_t *kr = FULL ? a.kr + (int64_t)g * T * (kD / 2) : nullptr;
    const uint8_t *vr = FULL ? a.vr + (int64_t)g * T * (kD / 2) : nullptr;
    const float *kpm = a.kpm + (int64_t)g * a.pool_pages * (2 * kD);
    const float *vpm = a.vpm + (int64_t)g * a.pool_pages * (2 * kD);
    const uint16_t *kcm = a.kcm + (int64_t)g * a.pool_pages * (kNChunk * 2 * kD);
    const uint16_t *vcm = a.vcm + (int64_t)g * a.pool_pages * (kNChunk * 2 * kD);
    const int64_t score_stride = (int64_t)a.max_pages * kPage;
    const int64_t qrow0 = (int64_t)b * a.Hq + g * G;

    const int p_begin = split * a.pages_per_split;
    const int p_end = min(p_begin + a.pages_per_split, a.max_pages);
    const int p_live = min(p_end, (ctx + kPage - 1) / kPage);   // pages holding context
    const int np = max(p_live - p_begin, 0);

    // physical page of the i-th live page of this range, or -1 (flagged)
    auto phys_of = [&](int i) -> int {
        const int p = a.page_table[(int64_t)b * a.max_pages + p_begin + i];
        return (p >= 0 && p < a.pool_pages) ? p : -1;
    };
    auto issue = [&](int i, int s) {
        const int p = phys_of(i);
        if (p < 0)
            return;
        Stage<FULL> &st = sm.st[s];
        const uint32_t bytes = (FULL ? 4u : 2u) * kPlane + 2u * (2 * kD * 4) + 2u * (kNChunk * 2 * kD * 2);
        mbar_arrive_expect_tx(&sm.bar[s], bytes);
        bulk_g2s(st.ka, ka + (int64_t)p * kPlane, kPlane, &sm.bar[s]);
        bulk_g2s(st.va, va + (int64_t)p * kPlane, kPlane, &sm.bar[s]);
        if (FULL) {
            bulk_g2s(st.kr, kr + (int64_t)p * kPlane, kPlane, &sm.bar[s]);
            bulk_g2s(st.vr, vr + (int64_t)p * kPlane, kPlane, &sm.bar[s]);
        }
        bulk_g2s(st.kpm, kpm + (int64_t)p * (2 * kD), 2 * kD * 4, &sm.bar[s]);
        bulk_g2s(st.vpm, vpm + (int64_t)p * (2 * kD), 2 * kD * 4, &sm.bar[s]);
        bulk_g2s(st.kcm, kcm + (int64_t)p * (kNChunk * 2 * kD), kNChunk * 2 * kD * 2, &sm.bar[s]);
        bulk_g2s(st.vcm, vcm + (int64_t)p * (kNChunk * 2 * kD), kNChunk * 2 * kD * 2, &sm.bar[s]);
    };
    if (tid == 0) {
        if (np > 0)
            issue(0, 0);
        if (np > 1)
            issue(1, 1);
    }

    // pages of the range past the context: scores -inf
    if (a.scores) {
        for (int lp = max(p_live, p_begin); lp < p_end; ++lp)
            for (int i = tid; i < G * kPage; i += NT)
                a.scores[(qrow0 + i / kPage) * score_stride + (int64_t)lp * kPage + i % kPage] = neg_inf();
    }

    // Running softmax state. STACK: head n. PAIR: head row n + 8hc (this warp's
    // softmax); the output of both head rows n and n + 8 for its channels.
    float m_run = neg_inf(), l_run = 0.0f;
    float2 O[NTO][NH];
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt)
#pragma unroll
        for (int i2 = 0; i2 < NH; ++i2)
            O[nt][i2] = make_float2(0.0f, 0.0f);
    const uint32_t *lut_lane = sm.lut + (FULL ? 0 : lane);
    const uint16_t *lut16_lane = reinterpret_cast<const uint16_t *>(sm.lut) + lane;

    uint32_t phase[2] = {0u, 0u};
    for (int i = 0; i < np; ++i) {
        const int s = i & 1;
        const int lp = p_begin + i;
        const int phys = phys_of(i);
        const int nvalid = min(kPage, ctx - lp * kPage);
        if (phys < 0) {
            if (a.dev_err && tid == 0)
                atomicOr(a.dev_err, LYNX_DEVERR_PAGE);
            if (a.scores)
                for (int e = tid; e < G * kPage; e += NT)
                    a.scores[(qrow0 + e / kPage) * score_stride + (int64_t)lp * kPage + e % kPage] = neg_inf();
            __syncthreads();
            if (tid == 0 && i + 2 < np)
                issue(i + 2, s);
            continue;
        }
        const bool ok = mbar_wait_bounded(&sm.bar[s], phase[s], kWaitLimit);
        if (__syncthreads_or(!ok)) {
            // a copy never completed: let what is in flight land (bounded), then stop
            if (tid == 0) {
                mbar_wait_bounded(&sm.bar[s], phase[s], kWaitLimit);
                if (i + 1 < np && phys_of(i + 1) >= 0)
                    mbar_wait_bounded(&sm.bar[s ^ 1], phase[s ^ 1], kWaitLimit);
                if (a.dev_err)
                    atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
            }
            __syncthreads();
            break;
        }
        phase[s] ^= 1u;
        const Stage<FULL> &st = sm.st[s];

        // ---- per-page preparation: chunk affines, V transpose, fp16 guard ----
        {
            float rmax = 0.0f;
            for (int e = tid; e < kNChunk * (kD / 2); e += NT) {
                const int jj = e >> 6, d = 2 * (e & 63);
                const float2 kmn = *reinterpret_cast<const float2 *>(st.kpm + d);
                const float2 krg = *reinterpret_cast<const float2 *>(st.kpm + kD + d);
                const float2 vmn = *reinterpret_cast<const float2 *>(st.vpm + d);
                const float2 vrg = *reinterpret_cast<const float2 *>(st.vpm + kD + d);
                const float2 kmu = __half22float2(*reinterpret_cast<const __half2 *>(st.kcm + (jj * 2) * kD + d));
                const float2 ksc = __half22float2(*reinterpret_cast<const __half2 *>(st.kcm + (jj * 2 + 1) * kD + d));
                const float2 vmu = __half22float2(*reinterpret_cast<const __half2 *>(st.vcm + (jj * 2) * kD + d));
                const float2 vsc = __half22float2(*reinterpret_cast<const __half2 *>(st.vcm + (jj * 2 + 1) * kD + d));
                const float2 kb = __fmul2_rn(krg, ksc), vb = __fmul2_rn(vrg, vsc);
                const float2 ka2 = __ffma2_rn(krg, kmu, kmn), va2 = __ffma2_rn(vrg, vmu, vmn);
                sm.kab[jj][e & 63] = make_float4(ka2.x, ka2.y, kb.x, kb.y);
                sm.vab[jj][e & 63] = make_float4(va2.x, va2.y, vb.x, vb.y);
                rmax = fmaxf(rmax, fmaxf(fabsf(kb.x), fabsf(kb.y)));
            }
            transpose_v<NT>(st.va, sm.vta, tid);
            // q b must stay a finite fp16 pair: if qmax * max|b| reaches 2^14 on
            // this page, scale K's b by 2^-e (and the scores back by 2^e)
            const bool need_guard = __syncthreads_or(rmax * sm.qmax >= 16384.0f);
            if (FULL) {   // the residual plane goes where the anchor plane was
                transpose_v<NT>(st.vr, sm.st[s].va, tid);
                __syncthreads();
            }
            if (need_guard) {
                if (rmax * sm.qmax >= 16384.0f) {
                    int e2;
                    frexpf(rmax * sm.qmax, &e2);
                    atomicMax(&sm.guard, e2 - 14);
                }
                __syncthreads();
                const float sc = exp2f((float)-sm.guard);
                for (int e = tid; e < kNChunk * (kD / 2); e += NT) {
                    float4 &kk = sm.kab[e >> 6][e & 63];
                    kk.z *= sc;
                    kk.w *= sc;
                }
                __syncthreads();
            }
        }
        const float gscale = exp2f((float)sm.guard);

        // ---- this warp's chunk -------------------------------------------------
        const int nv = min(max(nvalid - j * kChunk, 0), kChunk);
        if (nv > 0) {
            // B fragments of K for k-steps kk = 2m, 2m+1 and n-tile nt (tokens 8nt + n):
            // bytes q of the four words of the 16-byte block m of the token's row
            auto k_frag = [&](int nt, int m, uint32_t (&bq)[4]) {
                const int row = j * kChunk + nt * 8 + n;
                const int off = row * (kD / 2) + (PAIR ? 32 * hc : 0) + 16 * m;
                const uint4 aw = *reinterpret_cast<const uint4 *>(st.ka + off);
                if (FULL) {
                    const uint4 rw = *reinterpret_cast<const uint4 *>(st.kr + off);
                    const uint32_t awv[4] = {aw.x, aw.y, aw.z, aw.w};
                    const uint32_t rwv[4] = {rw.x, rw.y, rw.z, rw.w};
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        const uint32_t ev = ((awv[w4] << 4) & 0xF0F0F0F0u) | (rwv[w4] & 0x0F0F0F0Fu);
                        const uint32_t od = (awv[w4] & 0xF0F0F0F0u) | ((rwv[w4] >> 4) & 0x0F0F0F0Fu);
                        const uint32_t le = lut16_lane[__byte_perm(ev, 0u, 0x4440u | q) * 32];
                        const uint32_t lo = lut16_lane[__byte_perm(od, 0u, 0x4440u | q) * 32];
                        bq[w4] = __byte_perm(le, lo, 0x5410u);
                    }
                } else {
                    bq[0] = lut_lane[__byte_perm(aw.x, 0u, 0x4440u | q) * 32];
                    bq[1] = lut_lane[__byte_perm(aw.y, 0u, 0x4440u | q) * 32];
                    bq[2] = lut_lane[__byte_perm(aw.z, 0u, 0x4440u | q) * 32];
                    bq[3] = lut_lane[__byte_perm(aw.w, 0u, 0x4440u | q) * 32];
                }
            };
            // B fragments of V for channel column c and k-step ks (tokens 16ks ..)
            auto v_frag = [&](int c, int ks, uint32_t &b0, uint32_t &b1) {
                const int pos = vt_group(c, 2 * j + ks) + 2 * q;
                const uint32_t a16 = *reinterpret_cast<const uint16_t *>(sm.vta + pos);
                if (FULL) {
                    const uint32_t r16 = *reinterpret_cast<const uint16_t *>(st.va + pos);
                    const uint32_t ev = ((a16 << 4) & 0xF0F0u) | (r16 & 0x0F0Fu);
                    const uint32_t od = (a16 & 0xF0F0u) | ((r16 >> 4) & 0x0F0Fu);
                    b0 = __byte_perm(lut16_lane[(ev & 0xFFu) * 32], lut16_lane[(od & 0xFFu) * 32], 0x5410u);
                    b1 = __byte_perm(lut16_lane[(ev >> 8) * 32], lut16_lane[(od >> 8) * 32], 0x5410u);
                } else {
                    b0 = lut_lane[(a16 & 0xFFu) * 32];
                    b1 = lut_lane[(a16 >> 8) * 32];
                }
            };

            // Q.K^T. STACK: rows = (8 heads hi | their lo), all 128 channels.
            // PAIR: rows = 16 heads, hi and lo as two MMAs, this warp's 64 channels.
            float S[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.0f;
            float2 beta2[NH];
#pragma unroll
            for (int i2 = 0; i2 < NH; ++i2)
                beta2[i2] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int m = 0; m < (PAIR ? 2 : 4); ++m) {
                uint32_t Ahi[2][4], Alo[2][4];
#pragma unroll
                for (int kx = 0; kx < 2; ++kx) {
                    const int c0 = (PAIR ? 64 * hc : 0) + 32 * m + 16 * kx + 2 * q;
                    const float4 k01 = sm.kab[j][c0 >> 1];          // channels c0, c0 + 1
                    const float4 k89 = sm.kab[j][(c0 >> 1) + 4];    // channels c0 + 8, c0 + 9
                    float2 x[NH][2];
#pragma unroll
                    for (int i2 = 0; i2 < NH; ++i2) {
                        const float2 q01 = *reinterpret_cast<const float2 *>(&sm.qs[n + 8 * i2][c0]);
                        const float2 q89 = *reinterpret_cast<const float2 *>(&sm.qs[n + 8 * i2][c0 + 8]);
                        beta2[i2] = __ffma2_rn(q01, make_float2(k01.x, k01.y), beta2[i2]);
                        beta2[i2] = __ffma2_rn(q89, make_float2(k89.x, k89.y), beta2[i2]);
                        x[i2][0] = __fmul2_rn(q01, make_float2(k01.z, k01.w));
                        x[i2][1] = __fmul2_rn(q89, make_float2(k89.z, k89.w));
                    }
                    if (PAIR) {
                        split2(x[0][0], Ahi[kx][0], Alo[kx][0]);
                        split2(x[NH - 1][0], Ahi[kx][1], Alo[kx][1]);
                        split2(x[0][1], Ahi[kx][2], Alo[kx][2]);
                        split2(x[NH - 1][1], Ahi[kx][3], Alo[kx][3]);
                    } else {
                        split2(x[0][0], Ahi[kx][0], Ahi[kx][1]);
                        split2(x[0][1], Ahi[kx][2], Ahi[kx][3]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    uint32_t bq[4];
                    k_frag(nt, m, bq);
#pragma unroll
                    for (int kx = 0; kx < 2; ++kx) {
                        mma16816(S[nt], Ahi[kx], bq[2 * kx], bq[2 * kx + 1]);
                        if (PAIR)
                            mma16816(S[nt], Alo[kx], bq[2 * kx], bq[2 * kx + 1]);
                    }
                }
            }
            float beta[NH];
#pragma unroll
            for (int i2 = 0; i2 < NH; ++i2) {
                beta[i2] = beta2[i2].x + beta2[i2].y;
                beta[i2] += __shfl_xor_sync(0xFFFFFFFFu, beta[i2], 1);
                beta[i2] += __shfl_xor_sync(0xFFFFFFFFu, beta[i2], 2);
            }
            if (PAIR) {
                // sum the two channel halves: the upper warp hands its half over,
                // the lower warp adds and hands the total back, so both warps hold
                // the same scores bit for bit
                float *xc = &sm.xch[j][0][lane];
                if (hc == 1) {
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            xc[(nt * 4 + e) * 32] = S[nt][e];
                    xc[16 * 32] = beta[0];
                    xc[17 * 32] = beta[NH - 1];
                }
                pair_sync(j);
                if (hc == 0) {
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            S[nt][e] += xc[(nt * 4 + e) * 32];
                            xc[(nt * 4 + e) * 32] = S[nt][e];
                        }
                    beta[0] += xc[16 * 32];
                    beta[NH - 1] += xc[17 * 32];
                    xc[16 * 32] = beta[0];
                    xc[17 * 32] = beta[NH - 1];
                }
                pair_sync(j);
                if (hc == 1) {
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            S[nt][e] = xc[(nt * 4 + e) * 32];
                    beta[0] = xc[16 * 32];
                    beta[NH - 1] = xc[17 * 32];
                }
            }

            // scores of this warp's softmax head (base-2 log domain), masking, online softmax
            const int sh = PAIR ? hc : 0;          // head row: n + 8 sh
            const float bsh = PAIR ? (hc ? beta[NH - 1] : beta[0]) : beta[0];
            float P[4][2];
            float mx = neg_inf();
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tt = nt * 8 + 2 * q + e;
                    const float raw = PAIR ? S[nt][2 * sh + e] : S[nt][e] + S[nt][e + 2];
                    const float v = tt < nv ? fmaf(raw, gscale, bsh) : neg_inf();
                    P[nt][e] = v;
                    mx = fmaxf(mx, v);
                }
            if (a.scores && n + 8 * sh < G) {
                float *srow = a.scores + (qrow0 + n + 8 * sh) * score_stride + (int64_t)lp * kPage + j * kChunk;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    *reinterpret_cast<float2 *>(srow + nt * 8 + 2 * q) = make_float2(P[nt][0] * kLn2, P[nt][1] * kLn2);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = exp2f(m_run - m_new);
            m_run = m_new;
            float ps = 0.0f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pv = exp2f(P[nt][e] - m_new);
                    P[nt][e] = pv;
                    ps += pv;
                }
            l_run = fmaf(l_run, alpha, ps);
            ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 1);
            ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 2);

            // this head row's P as hi/lo fp16 pairs for n-tiles 0..3 (tokens 8nt + 2q + e)
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                split2(make_float2(P[nt][0], P[nt][1]), ph[nt], pl[nt]);

            // PAIR: swap P fragments, sums and rescales with the partner warp
            uint32_t oph[4], opl[4];
            float ops = ps, oalpha = alpha;
            if (PAIR) {
                // the V plane this page's transpose consumed (the anchor plane in
                // anchor mode, the residual plane in full mode) is free until the
                // end of the page
                uint32_t *xpb = reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(FULL ? st.vr : st.va));
                uint32_t *mine = xpb + ((j * 2 + hc) * 8) * 32 + lane;
                const uint32_t *theirs = xpb + ((j * 2 + (hc ^ 1)) * 8) * 32 + lane;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    mine[nt * 32] = ph[nt];
                    mine[(4 + nt) * 32] = pl[nt];
                }
                float *qrow = &sm.xch[j][18][0];
                if (q == 0) {
                    qrow[n * 4 + hc * 2] = ps;
                    qrow[n * 4 + hc * 2 + 1] = alpha;
                }
                pair_sync(j);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    oph[nt] = theirs[nt * 32];
                    opl[nt] = theirs[(4 + nt) * 32];
                }
                ops = qrow[n * 4 + (hc ^ 1) * 2];
                oalpha = qrow[n * 4 + (hc ^ 1) * 2 + 1];
            }
            // per output head row i2 (row n + 8 i2): its sum of P and rescale
            float psum[NH], alph[NH];
            psum[0] = (PAIR && hc == 1) ? ops : ps;
            alph[0] = (PAIR && hc == 1) ? oalpha : alpha;
            if (PAIR) {
                psum[NH - 1] = hc == 1 ? ps : ops;
                alph[NH - 1] = hc == 1 ? alpha : oalpha;
            }
#pragma unroll
            for (int i2 = 0; i2 < NH; ++i2) {
                if (alph[i2] != 1.0f) {
                    const float2 al = make_float2(alph[i2], alph[i2]);
#pragma unroll
                    for (int nt = 0; nt < NTO; ++nt)
                        O[nt][i2] = __fmul2_rn(O[nt][i2], al);
                }
            }

            // P as A fragments (k = tokens of n-tiles 2ks, 2ks + 1)
            uint32_t Phi[2][4], Plo[2][4];
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                if (PAIR) {
                    const bool lower = hc == 0;   // this warp's softmax row is n (else n + 8)
                    Phi[ks][0] = lower ? ph[2 * ks] : oph[2 * ks];
                    Phi[ks][1] = lower ? oph[2 * ks] : ph[2 * ks];
                    Phi[ks][2] = lower ? ph[2 * ks + 1] : oph[2 * ks + 1];
                    Phi[ks][3] = lower ? oph[2 * ks + 1] : ph[2 * ks + 1];
                    Plo[ks][0] = lower ? pl[2 * ks] : opl[2 * ks];
                    Plo[ks][1] = lower ? opl[2 * ks] : pl[2 * ks];
                    Plo[ks][2] = lower ? pl[2 * ks + 1] : opl[2 * ks + 1];
                    Plo[ks][3] = lower ? opl[2 * ks + 1] : pl[2 * ks + 1];
                } else {
                    Phi[ks][0] = ph[2 * ks];
                    Phi[ks][1] = pl[2 * ks];
                    Phi[ks][2] = ph[2 * ks + 1];
                    Phi[ks][3] = pl[2 * ks + 1];
                }
            }

            // P.L over this warp's output channels, then o += b (P.L) + a sum(P)
#pragma unroll
            for (int nt = 0; nt < NTO; ++nt) {
                const int cb = (PAIR ? 64 * hc : 0) + nt * 8;
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t b0, b1;
                    v_frag(cb + n, ks, b0, b1);
                    mma16816(acc, Phi[ks], b0, b1);
                    if (PAIR)
                        mma16816(acc, Plo[ks], b0, b1);
                }
                const float4 vv = sm.vab[j][(cb >> 1) + q];    // channels cb + 2q, cb + 2q + 1
                const float2 va2 = make_float2(vv.x, vv.y), vb2 = make_float2(vv.z, vv.w);
#pragma unroll
                for (int i2 = 0; i2 < NH; ++i2) {
                    const float2 dd = PAIR ? make_float2(acc[2 * i2], acc[2 * i2 + 1])
                                           : make_float2(acc[0] + acc[2], acc[1] + acc[3]);
                    O[nt][i2] = __ffma2_rn(vb2, dd, __ffma2_rn(make_float2(psum[i2], psum[i2]), va2, O[nt][i2]));
                }
            }
        } else if (a.scores && hc == 0) {
            for (int e = lane; e < G * kChunk; e += 32)
                a.scores[(qrow0 + e / kChunk) * score_stride + (int64_t)lp * kPage + j * kChunk + e % kChunk] =
                    neg_inf();
        }
        __syncthreads();   // stage s, transposed V and affines free again
        if (tid == 0 && i + 2 < np) {
            fence_proxy_async_smem();
            issue(i + 2, s);
        }
    }

    // ---- merge the chunks' states, write this range's partial ------------
    __syncthreads();
    Merge &mg = *reinterpret_cast<Merge *>(smem_raw);
    {
        float l = l_run;
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
        if (q == 0) {
            const int h = n + (PAIR ? 8 * hc : 0);
            mg.m[j][h] = m_run;
            mg.l[j][h] = l;
        }
    }
#pragma unroll
    for (int i2 = 0; i2 < NH; ++i2)
#pragma unroll
        for (int nt = 0; nt < NTO; ++nt)
            *reinterpret_cast<float2 *>(&mg.o[j][n + 8 * i2][(PAIR ? 64 * hc : 0) + nt * 8 + 2 * q]) = O[nt][i2];
    __syncthreads();
    for (int e = tid; e < G * kD; e += NT) {
        const int h = e / kD, d = e % kD;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kNChunk; ++w)
            M = fmaxf(M, mg.m[w][h]);
        float L = 0.0f, o = 0.0f;
        if (M > neg_inf()) {
#pragma unroll
            for (int w = 0; w < kNChunk; ++w) {
                const float sc = exp2f(mg.m[w][h] - M);
                L = fmaf(mg.l[w][h], sc, L);
                o = fmaf(mg.o[w][h][d], sc, o);
            }
        }
        float *pp = a.part + ((qrow0 + h) * a.n_splits + split) * kPart;
        pp[d] = o;
        if (d == 0) {
            pp[kD] = M;
            pp[kD + 1] = L;
        }
    }
}

template <int NW, bool FULL>
cudaError_t run(const AttnArgs &a, cudaStream_t s)
{
    static_assert(sizeof(Merge) <= sizeof(Stage<FULL>) * 2, "merge area overlays the stages");
    static_assert(sizeof(Smem<FULL>) <= 227 * 1024, "shared memory per CTA");
    const size_t smem = sizeof(Smem<FULL>);
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<NW, FULL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)a.n_splits, (unsigned)a.H, (unsigned)a.B);
    attn_mma_kernel<NW, FULL><<<grid, NW * 32, smem, s>>>(a, host_tables().lev);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_attn_mma(const AttnArgs &a, cudaStream_t s)
{
    if (a.G <= 8)
        return a.full ? run<8, true>(a, s) : run<8, false>(a, s);
    return a.full ? run<16, true>(a, s) : run<16, false>(a, s);
}

} // namespace lynx
