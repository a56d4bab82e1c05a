// attn_mma.cu -- fused-dequant paged decode attention on the tensor cores
// (K4, groups of up to 16 query heads per KV head).
//
// One decode step over the quantized paged cache ("KV-cache quantization"
// explainer, "Bottom-right": the compact cache is read as is and expanded
// only on chip, inside Q.K^T and P.V). Anchor mode reads the anchor planes only
// (the draft cache of the Lynx reading, section 4); full mode adds the residual
// planes.
//
// Factorisation. Every element of chunk j (32 tokens) and channel d decodes
// as x = a_jd + b_jd * L(code) with a = mn + rng mu, b = rng s and L an exact
// fp16 level value. Hence, per chunk,
//   s_t  = beta_j + sum_d (q_d b_jd) L_td,         beta_j = sum_d q_d a_jd
//   o_d += sum_j [ a_jd sum_{t in j} p_t + b_jd sum_{t in j} p_t L_td ],
// so the tensor-core operands on the cache side are the level values
// themselves (no rounding), and the dense operand (q b, or p) is split into an
// fp16 hi/lo pair to keep fp32-level accuracy (mma.sync m16n8k16, fp32
// accumulation). The MMA rows are 8 query heads' hi parts over the same heads'
// lo parts, so one MMA carries both halves of the split.
//
// Work: a CTA per (page range, KV head, request) with 8 warps per group of 8
// query heads; warp w owns chunk w % 8 for head group w / 8. A page's K planes
// and V planes arrive by bulk copy into their own buffers. Per page:
//   K phase: the warps of chunk j turn its 32 x 128 K codes into fp16 levels
//            in a swizzled shared-memory tile (one table lookup per code byte),
//            then each warp runs Q.K^T on it (B fragments by ldmatrix) and the
//            online softmax of its 8 heads;
//   V phase: the same warps overwrite the tile with the chunk's V levels and
//            run P.V (B fragments by ldmatrix.trans).
// Each code is decoded once per CTA; a K or V buffer is refilled with a later
// page as soon as its codes are decoded. The chunks' running (max, sum, output)
// are merged in shared memory into one partial per query head; a second
// kernel merges the partials of the ranges.
#include <cuda_fp16.h>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr uint32_t kPlane = kPage * kD / 2;   // 16 KiB: one page of one plane
constexpr int kRow = kD / 2;                  // code bytes per token
constexpr int kTileRow = kD * 2;              // bytes per token of an fp16 tile
constexpr int kPart = kD + 2;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One tensor's page as it arrives.
template <bool FULL>
struct Raw {
    uint8_t a[kPlane];
    uint8_t r[FULL ? kPlane : 16];
    float pm[2 * kD];
    uint16_t cm[kNChunk * 2 * kD];
};

template <bool FULL, int NB>
struct Smem {
    Raw<FULL> rk[NB], rv[NB];
    // fp16 levels of chunk j ([32 tokens][128 channels], K then V); the
    // 16-byte slot s of token t sits at slot s ^ (t & 7) so that 8 rows of one
    // slot column (an ldmatrix 8x8 matrix) fall in distinct banks
    uint16_t dec[kNChunk][kChunk * kD];
    // chunk affines of channel pairs: (a_2i, a_2i+1, b_2i, b_2i+1)
    float4 kab[kNChunk][kD / 2];
    float4 vab[kNChunk][kD / 2];
    float qs[16][kD + 8];                     // the group's queries times sm_scale log2(e); unused rows 0
    // level table, one copy per lane (conflict-free lookups): anchor mode maps a
    // byte of two anchors to the half2 of their levels, full mode a code byte
    // (A << 4 | r) to the fp16 level
    uint32_t lut[FULL ? 256 * 32 / 2 : 256 * 32];
    float rmaxw[16];                          // per warp: max |b| of K in its chunk
    float qmax;
    alignas(8) uint64_t bar_k[NB];
    uint64_t bar_v[NB];
};

struct Merge {                                // overlays the raw buffers after the page loop
    float m[kNChunk][16];                     // per chunk and query head
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

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
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

// Byte offset of 16-byte slot `slot` of token `t` in a chunk tile.
__device__ __forceinline__ uint32_t tile_off(int t, int slot)
{
    return (uint32_t)(t * kTileRow + ((slot ^ (t & 7)) << 4));
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7F800000); }

// Barrier of the HG warps that share a chunk.
template <int HG>
__device__ __forceinline__ void chunk_sync(int j)
{
    if (HG == 1)
        __syncwarp();
    else
        asm volatile("bar.sync %0, %1;" ::"r"(1 + j), "r"(HG * 32) : "memory");
}

// Codes of one chunk (32 token rows of 64 bytes per plane) -> fp16 levels in
// the chunk tile. Unit u = (token u / 16, channels 8 (u % 16) .. + 7): one
// 4-byte read per plane, four table lookups, one 16-byte store.
template <bool FULL, int PT>
__device__ __forceinline__ void decode_chunk(const uint8_t *pa, const uint8_t *pr, uint8_t *tile, int pt,
                                             const uint32_t *lut_lane, const uint16_t *lut16_lane)
{
#pragma unroll 4
    for (int u = pt; u < kChunk * 16; u += PT) {
        const int t = u >> 4, c8 = u & 15;
        const uint32_t aw = *reinterpret_cast<const uint32_t *>(pa + t * kRow + c8 * 4);
        uint4 v;
        if (FULL) {
            const uint32_t rw = *reinterpret_cast<const uint32_t *>(pr + t * kRow + c8 * 4);
            // byte i of ev / od: code (A << 4 | r) of channel 8 c8 + 2i / 2i + 1
            const uint32_t ev = ((aw << 4) & 0xF0F0F0F0u) | (rw & 0x0F0F0F0Fu);
            const uint32_t od = (aw & 0xF0F0F0F0u) | ((rw >> 4) & 0x0F0F0F0Fu);
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t le = lut16_lane[__byte_perm(ev, 0u, 0x4440u | i) * 32];
                const uint32_t lo = lut16_lane[__byte_perm(od, 0u, 0x4440u | i) * 32];
                w[i] = __byte_perm(le, lo, 0x5410u);
            }
            v = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            v = make_uint4(lut_lane[__byte_perm(aw, 0u, 0x4440u) * 32], lut_lane[__byte_perm(aw, 0u, 0x4441u) * 32],
                           lut_lane[__byte_perm(aw, 0u, 0x4442u) * 32], lut_lane[__byte_perm(aw, 0u, 0x4443u) * 32]);
        }
        *reinterpret_cast<uint4 *>(tile + tile_off(t, c8)) = v;
    }
}

// Chunk affine (a, b) of channel pair c from one tensor's page metadata.
__device__ __forceinline__ float4 chunk_affine(const float *pm, const uint16_t *cm, int j, int c)
{
    const int d = 2 * c;
    const float2 mn = *reinterpret_cast<const float2 *>(pm + d);
    const float2 rg = *reinterpret_cast<const float2 *>(pm + kD + d);
    const float2 mu = __half22float2(*reinterpret_cast<const __half2 *>(cm + (j * 2) * kD + d));
    const float2 sc = __half22float2(*reinterpret_cast<const __half2 *>(cm + (j * 2 + 1) * kD + d));
    const float2 b = __fmul2_rn(rg, sc), a = __ffma2_rn(rg, mu, mn);
    return make_float4(a.x, a.y, b.x, b.y);
}

template <int HG, bool FULL, int NB>
__global__ void __launch_bounds__(HG * 256, 1) attn_mma_kernel(AttnArgs a, LevelTable lev)
{
    constexpr int NW = 8 * HG;
    constexpr int NT = NW * 32;
    constexpr int PT = HG * 32;             // threads per chunk
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<FULL, NB> &sm = *reinterpret_cast<Smem<FULL, NB> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = lane >> 2, q = lane & 3;
    const int j = warp & 7;                 // chunk of this warp
    const int hg = warp >> 3;               // head group: query heads 8 hg .. 8 hg + 7 of the KV head's group
    const int pt = hg * 32 + lane;          // index among the chunk's threads
    const int hrow = hg * 8 + n;            // this lane's query head (MMA rows n and n + 8)
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
        for (int s = 0; s < NB; ++s) {
            mbar_init(&sm.bar_k[s], 1);
            mbar_init(&sm.bar_v[s], 1);
        }
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
    const uint8_t *ka = a.ka + (int64_t)g * T * kRow;
    const uint8_t *va = a.va + (int64_t)g * T * kRow;
    const uint8_t *kr = FULL ? a.kr + (int64_t)g * T * kRow : nullptr;
    const uint8_t *vr = FULL ? a.vr + (int64_t)g * T * kRow : nullptr;
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
    // copies of page i into buffer s; `pend` (thread 0) marks buffers with a copy in flight
    uint32_t pend = 0;
    auto issue = [&](int i, int s, bool is_v) {
        const int p = phys_of(i);
        if (p < 0)
            return;
        Raw<FULL> &r = is_v ? sm.rv[s] : sm.rk[s];
        uint64_t *bar = is_v ? &sm.bar_v[s] : &sm.bar_k[s];
        const uint8_t *pa = is_v ? va : ka;
        const uint8_t *pr = is_v ? vr : kr;
        const float *pm = is_v ? vpm : kpm;
        const uint16_t *cm = is_v ? vcm : kcm;
        mbar_arrive_expect_tx(bar, (FULL ? 2u : 1u) * kPlane + 2 * kD * 4 + kNChunk * 2 * kD * 2);
        bulk_g2s(r.a, pa + (int64_t)p * kPlane, kPlane, bar);
        if (FULL)
            bulk_g2s(r.r, pr + (int64_t)p * kPlane, kPlane, bar);
        bulk_g2s(r.pm, pm + (int64_t)p * (2 * kD), 2 * kD * 4, bar);
        bulk_g2s(r.cm, cm + (int64_t)p * (kNChunk * 2 * kD), kNChunk * 2 * kD * 2, bar);
        pend |= 1u << (is_v ? NB + s : s);
    };
    if (tid == 0)
        for (int i = 0; i < NB && i < np; ++i) {
            issue(i, i, false);
            issue(i, i, true);
        }

    // pages of the range past the context: scores -inf
    if (a.scores) {
        for (int lp = max(p_live, p_begin); lp < p_end; ++lp)
            for (int i = tid; i < G * kPage; i += NT)
                a.scores[(qrow0 + i / kPage) * score_stride + (int64_t)lp * kPage + i % kPage] = neg_inf();
    }

    float m_run = neg_inf(), l_run = 0.0f;
    float2 O[16];                           // head hrow, channels 8 nt + 2q, + 1
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
        O[nt] = make_float2(0.0f, 0.0f);
    const uint32_t *lut_lane = sm.lut + lane;
    const uint16_t *lut16_lane = reinterpret_cast<const uint16_t *>(sm.lut) + lane;
    uint8_t *tile = reinterpret_cast<uint8_t *>(sm.dec[j]);
    const uint32_t tile_s = smem_u32(tile);
    // ldmatrix: this lane gives the address of row lane % 8 of matrix lane / 8
    const int lm = lane >> 3, lr = lane & 7;

    uint32_t phk[NB], phv[NB];
#pragma unroll
    for (int s = 0; s < NB; ++s)
        phk[s] = phv[s] = 0u;
    bool timed_out = false;
    for (int i = 0; i < np; ++i) {
        const int s = i % NB;
        const int lp = p_begin + i;
        const int nvalid = min(kPage, ctx - lp * kPage);
        if (phys_of(i) < 0) {
            if (a.dev_err && tid == 0)
                atomicOr(a.dev_err, LYNX_DEVERR_PAGE);
            if (a.scores)
                for (int e = tid; e < G * kPage; e += NT)
                    a.scores[(qrow0 + e / kPage) * score_stride + (int64_t)lp * kPage + e % kPage] = neg_inf();
            __syncthreads();
            if (tid == 0 && i + NB < np) {
                issue(i + NB, s, false);
                issue(i + NB, s, true);
            }
            continue;
        }
        const int nv = min(max(nvalid - j * kChunk, 0), kChunk);   // valid tokens of chunk j

        // ---- K phase: decode chunk j's K, Q.K^T and softmax ----------------
        bool ok = mbar_wait_bounded(&sm.bar_k[s], phk[s], kWaitLimit);
        if (ok && nv > 0) {
            const Raw<FULL> &rk = sm.rk[s];
            float rmax = 0.0f;
            for (int c = pt; c < kD / 2; c += PT) {
                const float4 ab = chunk_affine(rk.pm, rk.cm, j, c);
                sm.kab[j][c] = ab;
                rmax = fmaxf(rmax, fmaxf(fabsf(ab.z), fabsf(ab.w)));
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                rmax = fmaxf(rmax, __shfl_xor_sync(0xFFFFFFFFu, rmax, o));
            if (lane == 0)
                sm.rmaxw[warp] = rmax;
            decode_chunk<FULL, PT>(rk.a + j * kChunk * kRow, FULL ? rk.r + j * kChunk * kRow : nullptr, tile, pt,
                                   lut_lane, lut16_lane);
        }
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        phk[s] ^= 1u;
        if (tid == 0) {
            pend &= ~(1u << s);
            if (i + NB < np) {
                fence_proxy_async_smem();
                issue(i + NB, s, false);
            }
        }

        uint32_t Phi[2][4];
        float psum = 0.0f;
        if (nv > 0) {
            // q b must stay a finite fp16 pair: if qmax * max|b| reaches 2^14 in
            // this chunk, q b is scaled by 2^-e and the scores back by 2^e
            float rm = sm.rmaxw[j];
            if (HG == 2)
                rm = fmaxf(rm, sm.rmaxw[j + 8]);
            int ge = 0;
            if (rm * sm.qmax >= 16384.0f) {
                frexpf(rm * sm.qmax, &ge);
                ge -= 14;
            }
            const float gdown = exp2f((float)-ge), gscale = exp2f((float)ge);

            // Q.K^T: rows = 8 heads' hi parts over their lo parts
            float S[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.0f;
            float2 beta2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int c0 = ks * 16 + 2 * q;
                const float4 k01 = sm.kab[j][c0 >> 1];          // channels c0, c0 + 1
                const float4 k89 = sm.kab[j][(c0 >> 1) + 4];    // channels c0 + 8, c0 + 9
                const float2 q01 = *reinterpret_cast<const float2 *>(&sm.qs[hrow][c0]);
                const float2 q89 = *reinterpret_cast<const float2 *>(&sm.qs[hrow][c0 + 8]);
                beta2 = __ffma2_rn(q01, make_float2(k01.x, k01.y), beta2);
                beta2 = __ffma2_rn(q89, make_float2(k89.x, k89.y), beta2);
                float2 x0 = __fmul2_rn(q01, make_float2(k01.z, k01.w));
                float2 x1 = __fmul2_rn(q89, make_float2(k89.z, k89.w));
                if (ge) {
                    x0 = __fmul2_rn(x0, make_float2(gdown, gdown));
                    x1 = __fmul2_rn(x1, make_float2(gdown, gdown));
                }
                uint32_t A[4];
                split2(x0, A[0], A[1]);
                split2(x1, A[2], A[3]);
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    // n-tiles 2p, 2p + 1: matrices (n-tile 2p + m / 2, slot 2ks + m % 2)
                    uint32_t bb[4];
                    const int t = 8 * (2 * p + (lm >> 1)) + lr;
                    ldsm_x4(tile_s + tile_off(t, 2 * ks + (lm & 1)), bb);
                    mma16816(S[2 * p], A, bb[0], bb[1]);
                    mma16816(S[2 * p + 1], A, bb[2], bb[3]);
                }
            }
            float beta = beta2.x + beta2.y;
            beta += __shfl_xor_sync(0xFFFFFFFFu, beta, 1);
            beta += __shfl_xor_sync(0xFFFFFFFFu, beta, 2);

            // scores of head hrow (base-2 log domain), masking, online softmax
            float P[4][2];
            float mx = neg_inf();
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tt = nt * 8 + 2 * q + e;
                    const float v = tt < nv ? fmaf(S[nt][e] + S[nt][e + 2], gscale, beta) : neg_inf();
                    P[nt][e] = v;
                    mx = fmaxf(mx, v);
                }
            if (a.scores && hrow < G) {
                float *srow = a.scores + (qrow0 + hrow) * score_stride + (int64_t)lp * kPage + j * kChunk;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    *reinterpret_cast<float2 *>(srow + nt * 8 + 2 * q) = make_float2(P[nt][0] * kLn2, P[nt][1] * kLn2);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = exp2f(m_run - m_new);
            m_run = m_new;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pv = exp2f(P[nt][e] - m_new);
                    P[nt][e] = pv;
                    psum += pv;
                }
            l_run = fmaf(l_run, alpha, psum);
            psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 1);
            psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 2);
            if (alpha != 1.0f) {
                const float2 al = make_float2(alpha, alpha);
#pragma unroll
                for (int nt = 0; nt < 16; ++nt)
                    O[nt] = __fmul2_rn(O[nt], al);
            }
            // P as A fragments: k = tokens of n-tiles 2ks, 2ks + 1; rows hi over lo
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                split2(make_float2(P[2 * ks][0], P[2 * ks][1]), Phi[ks][0], Phi[ks][1]);
                split2(make_float2(P[2 * ks + 1][0], P[2 * ks + 1][1]), Phi[ks][2], Phi[ks][3]);
            }
        } else if (a.scores && hrow < G) {
            for (int e = q; e < kChunk; e += 4)
                a.scores[(qrow0 + hrow) * score_stride + (int64_t)lp * kPage + j * kChunk + e] = neg_inf();
        }
        chunk_sync<HG>(j);   // the chunk's warps are done with its K tile

        // ---- V phase: decode chunk j's V, P.V --------------------------------
        ok = mbar_wait_bounded(&sm.bar_v[s], phv[s], kWaitLimit);
        if (ok && nv > 0) {
            const Raw<FULL> &rv = sm.rv[s];
            for (int c = pt; c < kD / 2; c += PT)
                sm.vab[j][c] = chunk_affine(rv.pm, rv.cm, j, c);
            decode_chunk<FULL, PT>(rv.a + j * kChunk * kRow, FULL ? rv.r + j * kChunk * kRow : nullptr, tile, pt,
                                   lut_lane, lut16_lane);
        }
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        phv[s] ^= 1u;
        if (tid == 0) {
            pend &= ~(1u << (NB + s));
            if (i + NB < np) {
                fence_proxy_async_smem();
                issue(i + NB, s, true);
            }
        }
        if (nv > 0) {
            const float2 ps2 = make_float2(psum, psum);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                // n-tiles 2p, 2p + 1 (channels 16p ..); k-steps = tokens 0..15, 16..31:
                // matrices (tokens 16 ks + 8 (m % 2) .., slot 2p + m / 2), transposed
                float accA[4] = {0.0f, 0.0f, 0.0f, 0.0f}, accB[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t bb[4];
                    const int t = 16 * ks + 8 * (lm & 1) + lr;
                    ldsm_x4_trans(tile_s + tile_off(t, 2 * p + (lm >> 1)), bb);
                    mma16816(accA, Phi[ks], bb[0], bb[1]);
                    mma16816(accB, Phi[ks], bb[2], bb[3]);
                }
                // o += b (P.L) + a sum(P), channels 8 nt + 2q, + 1
                const float4 vA = sm.vab[j][(2 * p) * 4 + q];
                const float4 vB = sm.vab[j][(2 * p + 1) * 4 + q];
                O[2 * p] = __ffma2_rn(make_float2(vA.z, vA.w), make_float2(accA[0] + accA[2], accA[1] + accA[3]),
                                      __ffma2_rn(ps2, make_float2(vA.x, vA.y), O[2 * p]));
                O[2 * p + 1] = __ffma2_rn(make_float2(vB.z, vB.w), make_float2(accB[0] + accB[2], accB[1] + accB[3]),
                                          __ffma2_rn(ps2, make_float2(vB.x, vB.y), O[2 * p + 1]));
            }
        }
        chunk_sync<HG>(j);   // the chunk's warps are done with its V tile
    }
    if (timed_out) {
        // a copy never completed: let the ones in flight land (bounded), then stop
        if (tid == 0) {
            for (int s = 0; s < NB; ++s) {
                if (pend & (1u << s))
                    mbar_wait_bounded(&sm.bar_k[s], phk[s], kWaitLimit);
                if (pend & (1u << (NB + s)))
                    mbar_wait_bounded(&sm.bar_v[s], phv[s], kWaitLimit);
            }
            if (a.dev_err)
                atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
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
            mg.m[j][hrow] = m_run;
            mg.l[j][hrow] = l;
        }
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2 *>(&mg.o[j][hrow][nt * 8 + 2 * q]) = O[nt];
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

template <int HG, bool FULL, int NB>
cudaError_t run(const AttnArgs &a, cudaStream_t s)
{
    static_assert(sizeof(Merge) <= sizeof(Raw<FULL>) * 2 * NB, "merge area overlays the raw buffers");
    static_assert(sizeof(Smem<FULL, NB>) <= 227 * 1024, "shared memory per CTA");
    const size_t smem = sizeof(Smem<FULL, NB>);
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<HG, FULL, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)a.n_splits, (unsigned)a.H, (unsigned)a.B);
    attn_mma_kernel<HG, FULL, NB><<<grid, HG * 256, smem, s>>>(a, host_tables().lev);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_attn_mma(const AttnArgs &a, cudaStream_t s)
{
    // anchor pages are small enough for two buffers per tensor; full pages get one
    if (a.G <= 8)
        return a.full ? run<1, true, 1>(a, s) : run<1, false, 2>(a, s);
    return a.full ? run<2, true, 1>(a, s) : run<2, false, 2>(a, s);
}

} // namespace lynx
