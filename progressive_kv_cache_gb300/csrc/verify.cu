// verify.cu -- multi-token verify attention over the quantized paged cache
// (a block of draft positions per request, causal within the block).
//
// The Lynx reading, section 4: decoding runs speculatively on the anchor-only
// draft cache, and once the residuals land a verify pass re-reads the refined
// cache for the drafted positions. Here that pass is attention of T_q query
// positions per request over the full (or anchor-only) reconstruction, where
// the last T_q tokens of the context are the drafted ones: position i sees the
// context up to and including draft token i. Dequantization stays on chip
// ("KV-cache quantization" explainer, "Bottom-right").
//
// With T_q x G query rows per KV head, Q.K^T and P.V are dense contractions:
// each 32-token chunk of K and V is decoded once per CTA (x = a + b L, fp32)
// into shared-memory fp16 hi/lo tiles, and every warp runs 16 query rows over
// them on the tensor cores (mma.sync m16n8k16, fp32 accumulation) with the
// three-product split (hi.hi + hi.lo + lo.hi) that keeps fp32-level accuracy.
// Softmax is online per row; split-K partials are merged by the decode path's
// combine kernel.
#include <cuda_fp16.h>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr uint32_t kPlane = kPage * kD / 2;   // 16 KiB: one page of one plane
constexpr int kRow = kD / 2;                  // code bytes per token
constexpr int kTileRow = kD * 2;              // bytes per token of an fp16 tile
constexpr int kTile = kChunk * kTileRow;      // 8 KiB
constexpr int kPart = kD + 2;
constexpr int kWarps = 8;                     // 16 query rows each
constexpr int kRows = kWarps * 16;            // rows per CTA
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;

template <bool FULL>
struct Page {                                 // one tensor's page as it arrives
    uint8_t a[kPlane];
    uint8_t r[FULL ? kPlane : 16];
    float pm[2 * kD];
    uint16_t cm[kNChunk * 2 * kD];
};

template <bool FULL>
struct Smem {
    Page<FULL> k[2], v[2];                    // double-buffered pages
    uint8_t tile[2][4][kTile];                // per chunk buffer: K hi, K lo, V hi, V lo
    float lev[256 * 8];                       // level of a code byte (anchor: of an anchor nibble), 8 copies
    alignas(8) uint64_t bar[2];
};

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
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
    const float2 r = __ffma2_rn(__half22float2(h), make_float2(-1.0f, -1.0f), x);
    const __half2 l = __floats2half2_rn(r.x, r.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7F800000); }

__device__ __forceinline__ float exp2_sm(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte slot `slot` of token `t` in a chunk tile: the slots
// of 8 consecutive tokens (an ldmatrix 8x8 matrix) fall in distinct banks.
__device__ __forceinline__ uint32_t tile_off(int t, int slot)
{
    return (uint32_t)(t * kTileRow + ((slot ^ (t & 7)) << 4));
}

// Decode chunk j of one tensor's page into fp16 hi/lo tiles. Thread u takes
// channel pair p = u % 64 (channels 2p, 2p + 1) of tokens 8 (u / 64) .. + 7:
// its affines are computed once, consecutive threads read consecutive code
// bytes and metadata and write consecutive 4-byte words of a tile row. The
// level table is replicated 8 times (copy u % 8).
template <bool FULL>
__device__ __forceinline__ void decode_chunk(const Page<FULL> &pg, int j, const float *lev, uint8_t *hi_tile,
                                             uint8_t *lo_tile, int tid)
{
    const int p = tid & 63, t0 = (tid >> 6) * 8;
    const int d = 2 * p;
    const float2 mn = *reinterpret_cast<const float2 *>(pg.pm + d);
    const float2 rg = *reinterpret_cast<const float2 *>(pg.pm + kD + d);
    const float2 mu = __half22float2(*reinterpret_cast<const __half2 *>(pg.cm + (2 * j) * kD + d));
    const float2 sc = __half22float2(*reinterpret_cast<const __half2 *>(pg.cm + (2 * j + 1) * kD + d));
    const float2 a = __ffma2_rn(rg, mu, mn), b = __fmul2_rn(rg, sc);
    const float *lv = lev + (tid & 7);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int t = t0 + k;
        const int row = j * kChunk + t;
        const uint32_t a8 = pg.a[row * kRow + p];
        float L0, L1;
        if (FULL) {
            const uint32_t r8 = pg.r[row * kRow + p];
            L0 = lv[8 * (((a8 & 0x0Fu) << 4) | (r8 & 0x0Fu))];
            L1 = lv[8 * ((a8 & 0xF0u) | (r8 >> 4))];
        } else {
            L0 = lv[8 * (a8 & 0x0Fu)];
            L1 = lv[8 * (a8 >> 4)];
        }
        uint32_t hi, lo;
        split2(__ffma2_rn(b, make_float2(L0, L1), a), hi, lo);
        // word p % 4 of 16-byte slot p / 4 of token t's row
        const uint32_t off = tile_off(t, p >> 2) + 4 * (p & 3);
        *reinterpret_cast<uint32_t *>(hi_tile + off) = hi;
        *reinterpret_cast<uint32_t *>(lo_tile + off) = lo;
    }
}

template <bool FULL>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(VerifyArgs a, LevelTable levt)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<FULL> &sm = *reinterpret_cast<Smem<FULL> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int lm = lane >> 3, lr = lane & 7;   // ldmatrix: this lane addresses row lr of matrix lm
    const int split = blockIdx.x, kvh = blockIdx.y / a.RB, rb = blockIdx.y % a.RB, b = blockIdx.z;
    const int G = a.G, Tq = a.Tq;
    const int64_t T = (int64_t)a.pool_pages * kPage;

    for (int i = tid; i < 256 * 8; i += kThreads)
        sm.lev[i] = FULL ? levt.full[i >> 3] : levt.anchor[(i >> 3) & 15];
    if (tid == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
    }

    int ctx = a.ctx[b];
    if (ctx < 0 || ctx > a.max_pages * kPage) {
        if (a.dev_err && split == 0 && blockIdx.y == 0 && tid == 0)
            atomicOr(a.dev_err, LYNX_DEVERR_CTX);
        ctx = min(max(ctx, 0), a.max_pages * kPage);
    }

    // this lane's two query rows (r = position * G + head in group); a row past
    // the block is padding: zero query, nothing visible, never written
    int rowi[2], rowh[2], nvis[2];
    bool rowok[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = rb * kRows + warp * 16 + g + 8 * e;
        rowok[e] = r < Tq * G;
        rowi[e] = rowok[e] ? r / G : 0;
        rowh[e] = kvh * G + (rowok[e] ? r % G : 0);
        nvis[e] = rowok[e] ? ctx - Tq + rowi[e] + 1 : 0;   // draft position i sees tokens < nvis
    }
    // query fragments (hi and lo), scaled by sm_scale log2(e)
    const float qscale = a.sm_scale * kLog2e;
    uint32_t QH[8][4], QL[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            const int e = f & 1, coff = (f >> 1) * 8;
            float2 x = make_float2(0.0f, 0.0f);
            if (rowok[e]) {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(
                    a.q + (((int64_t)b * Tq + rowi[e]) * a.Hq + rowh[e]) * kD + 16 * ks + coff + 2 * q);
                x = make_float2(bf16_lo(w) * qscale, bf16_hi(w) * qscale);
            }
            split2(x, QH[ks][f], QL[ks][f]);
        }

    const int p_begin = split * a.pages_per_split;
    const int p_end = min(p_begin + a.pages_per_split, a.max_pages);
    const int p_live = min(p_end, (ctx + kPage - 1) / kPage);
    const int np = max(p_live - p_begin, 0);
    const uint8_t *ka = a.ka + (int64_t)kvh * T * kRow, *va = a.va + (int64_t)kvh * T * kRow;
    const uint8_t *kr = FULL ? a.kr + (int64_t)kvh * T * kRow : nullptr;
    const uint8_t *vr = FULL ? a.vr + (int64_t)kvh * T * kRow : nullptr;
    const float *kpm = a.kpm + (int64_t)kvh * a.pool_pages * (2 * kD);
    const float *vpm = a.vpm + (int64_t)kvh * a.pool_pages * (2 * kD);
    const uint16_t *kcm = a.kcm + (int64_t)kvh * a.pool_pages * (kNChunk * 2 * kD);
    const uint16_t *vcm = a.vcm + (int64_t)kvh * a.pool_pages * (kNChunk * 2 * kD);

    auto phys_of = [&](int i) -> int {
        const int p = a.page_table[(int64_t)b * a.max_pages + p_begin + i];
        return (p >= 0 && p < a.pool_pages) ? p : -1;
    };
    // page i of the range into buffer i & 1 (thread 0); an invalid page
    // completes the phase without data and is skipped
    int last_issued = -1;           // thread 0: the last page whose copies were issued
    auto issue = [&](int i) {
        const int buf = i & 1, p = phys_of(i);
        uint64_t *bar = &sm.bar[buf];
        if (p < 0) {
            if (a.dev_err)
                atomicOr(a.dev_err, LYNX_DEVERR_PAGE);
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
            return;
        }
        last_issued = i;
        if (i >= 2)
            fence_proxy_async_smem();   // the buffer's previous page was read through the generic proxy
        mbar_arrive_expect_tx(bar, 2u * ((FULL ? 2u : 1u) * kPlane + 2 * kD * 4 + kNChunk * 2 * kD * 2));
        const int64_t off = (int64_t)p * kPlane;
        bulk_g2s(sm.k[buf].a, ka + off, kPlane, bar);
        bulk_g2s(sm.v[buf].a, va + off, kPlane, bar);
        if (FULL) {
            bulk_g2s(sm.k[buf].r, kr + off, kPlane, bar);
            bulk_g2s(sm.v[buf].r, vr + off, kPlane, bar);
        }
        bulk_g2s(sm.k[buf].pm, kpm + (int64_t)p * (2 * kD), 2 * kD * 4, bar);
        bulk_g2s(sm.v[buf].pm, vpm + (int64_t)p * (2 * kD), 2 * kD * 4, bar);
        bulk_g2s(sm.k[buf].cm, kcm + (int64_t)p * (kNChunk * 2 * kD), kNChunk * 2 * kD * 2, bar);
        bulk_g2s(sm.v[buf].cm, vcm + (int64_t)p * (kNChunk * 2 * kD), kNChunk * 2 * kD * 2, bar);
    };
    __syncthreads();
    if (tid == 0 && np > 0)
        issue(0);

    float m_run[2] = {neg_inf(), neg_inf()}, l_run[2] = {0.0f, 0.0f};
    float O[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
        O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.0f;

    // chunk c = chunk c % 8 of page c / 8: decode chunk c + 1 into tile buffer
    // (c + 1) & 1 while the warps run chunk c from buffer c & 1
    const int nchunks = kNChunk * np;
    bool timed_out = false;
    bool pvalid = false;            // whether the page of the chunk being decoded holds data
    auto decode = [&](int c) -> bool {
        const int i = c >> 3, j = c & 7;
        if (j == 0) {
            if (tid == 0 && i + 1 < np)
                issue(i + 1);       // its buffer held page i - 1, fully decoded by now
            const bool ok = mbar_wait_bounded(&sm.bar[i & 1], (uint32_t)((i >> 1) & 1), kWaitLimit);
            if (__syncthreads_or(!ok))
                return false;
            pvalid = phys_of(i) >= 0;
        }
        if (pvalid) {
            uint8_t(&tl)[4][kTile] = sm.tile[c & 1];
            decode_chunk<FULL>(sm.k[i & 1], j, sm.lev, tl[0], tl[1], tid);
            decode_chunk<FULL>(sm.v[i & 1], j, sm.lev, tl[2], tl[3], tid);
        }
        return true;
    };
    bool cvalid_next = false;
    if (nchunks > 0) {
        timed_out = !decode(0);
        cvalid_next = pvalid;
    }
    __syncthreads();
    for (int c = 0; c < nchunks && !timed_out; ++c) {
        const bool cvalid = cvalid_next;
        if (c + 1 < nchunks) {
            timed_out = !decode(c + 1);
            cvalid_next = pvalid;
            if (timed_out)
                break;
        }
        const int t0 = (p_begin + (c >> 3)) * kPage + (c & 7) * kChunk;   // first token of chunk c
        // a warp none of whose rows sees the chunk skips it
        const bool seen = __any_sync(0xFFFFFFFFu, t0 < max(nvis[0], nvis[1]));
        if (cvalid && seen) {
            const uint32_t kh = smem_u32(sm.tile[c & 1][0]), kl = smem_u32(sm.tile[c & 1][1]);
            const uint32_t vh = smem_u32(sm.tile[c & 1][2]), vl = smem_u32(sm.tile[c & 1][3]);
            // ---- S = Q.K^T over the chunk's 32 tokens (four n-tiles of 8)
            float S[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.0f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    // matrices (n-tile 2pp + m / 2, k-half m % 2) of 8 tokens x 8 channels
                    const uint32_t off = tile_off(8 * (2 * pp + (lm >> 1)) + lr, 2 * ks + (lm & 1));
                    uint32_t bh[4], bl[4];
                    ldsm_x4(kh + off, bh);
                    ldsm_x4(kl + off, bl);
                    mma16816(S[2 * pp], QH[ks], bh[0], bh[1]);
                    mma16816(S[2 * pp + 1], QH[ks], bh[2], bh[3]);
                    mma16816(S[2 * pp], QH[ks], bl[0], bl[1]);
                    mma16816(S[2 * pp + 1], QH[ks], bl[2], bl[3]);
                    mma16816(S[2 * pp], QL[ks], bh[0], bh[1]);
                    mma16816(S[2 * pp + 1], QL[ks], bh[2], bh[3]);
                }
            // ---- causal mask and online softmax of rows g (e = 0) and g + 8 (e = 1)
            float mx[2] = {neg_inf(), neg_inf()};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const int e = f >> 1;
                    const int tok = t0 + 8 * nt + 2 * q + (f & 1);
                    if (tok >= nvis[e])
                        S[nt][f] = neg_inf();
                    mx[e] = fmaxf(mx[e], S[nt][f]);
                }
            float scale[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xFFFFFFFFu, mx[e], 1));
                mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xFFFFFFFFu, mx[e], 2));
                // the reference moves only when a score passes it by 2^8
                const bool up = mx[e] > m_run[e] + 8.0f;
                const float m_new = up ? mx[e] : m_run[e];
                scale[e] = up ? exp2_sm(m_run[e] - m_new) : 1.0f;
                m_run[e] = m_new;
                l_run[e] *= scale[e];
            }
            if (__any_sync(0xFFFFFFFFu, scale[0] != 1.0f || scale[1] != 1.0f)) {
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    O[nt][0] *= scale[0];
                    O[nt][1] *= scale[0];
                    O[nt][2] *= scale[1];
                    O[nt][3] *= scale[1];
                }
            }
            uint32_t PH[2][4], PL[2][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                float p[4];
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const int e = f >> 1;
                    p[f] = m_run[e] == neg_inf() ? 0.0f : exp2_sm(S[nt][f] - m_run[e]);
                    l_run[e] += p[f];
                }
                // A fragment of k-step nt / 2: rows g, g + 8 and tokens 2q (+8 for odd nt)
                const int kk = nt >> 1, hf = (nt & 1) * 2;
                split2(make_float2(p[0], p[1]), PH[kk][hf], PL[kk][hf]);
                split2(make_float2(p[2], p[3]), PH[kk][hf + 1], PL[kk][hf + 1]);
            }
            // ---- O += P.V (sixteen n-tiles of 8 channels)
#pragma unroll
            for (int pp = 0; pp < 8; ++pp)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    // matrices (tokens 16 kk + 8 (m % 2) .., channels of n-tile 2pp + m / 2), transposed
                    const uint32_t off = tile_off(16 * kk + 8 * (lm & 1) + lr, 2 * pp + (lm >> 1));
                    uint32_t bh[4], bl[4];
                    ldsm_x4_trans(vh + off, bh);
                    ldsm_x4_trans(vl + off, bl);
                    mma16816(O[2 * pp], PH[kk], bh[0], bh[1]);
                    mma16816(O[2 * pp + 1], PH[kk], bh[2], bh[3]);
                    mma16816(O[2 * pp], PH[kk], bl[0], bl[1]);
                    mma16816(O[2 * pp + 1], PH[kk], bl[2], bl[3]);
                    mma16816(O[2 * pp], PL[kk], bh[0], bh[1]);
                    mma16816(O[2 * pp + 1], PL[kk], bh[2], bh[3]);
                }
        }
        __syncthreads();   // chunk c's tiles are free for chunk c + 2
    }
    if (timed_out) {
        if (tid == 0) {
            // let a copy still in flight land (bounded) before the CTA ends
            if (last_issued >= 0)
                mbar_wait_bounded(&sm.bar[last_issued & 1], (uint32_t)((last_issued >> 1) & 1), kWaitLimit);
            if (a.dev_err)
                atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
        }
    }

    // ---- this range's partial of each row
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        float l = l_run[e];
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
        if (!rowok[e])
            continue;
        float *part = a.part + ((((int64_t)b * Tq + rowi[e]) * a.Hq + rowh[e]) * a.n_splits + split) * kPart;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
            *reinterpret_cast<float2 *>(part + 8 * nt + 2 * q) = make_float2(O[nt][2 * e], O[nt][2 * e + 1]);
        if (q == 0) {
            part[kD] = m_run[e];
            part[kD + 1] = l;
        }
    }
}

template <bool FULL>
cudaError_t run(const VerifyArgs &a, cudaStream_t s)
{
    static_assert(sizeof(Smem<FULL>) <= 227 * 1024, "shared memory per CTA");
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
