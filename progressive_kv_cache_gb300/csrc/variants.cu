// variants.cu -- the quantizer with every knob that section 7 of the Lynx
// reading ("What the paper does not establish") lists as unmeasured: other
// anchor/residual splits, chunk size C in {16, 32, 64}, the alpha of the map
// (0: the linear grid), each stage switched off on its own, and the uniform
// INTb comparator. One pass over a page writes the codes (optional), the
// metadata (optional) and the page's squared errors of the anchor-only and the
// full reconstruction, so a quality study reads the bf16 cache once.
//
// Stages as in section 3 ("The quantizer"): page normalisation, chunk
// isolation (fp16 chunk mean rounded to nearest, fp16 scale rounded up, the
// chunk sum by a stride-halving tree), the level count q = #{k : |w| >= T_k}
// with the sign-aware mapping, the bias 2^(r-1) - 1 and the r-bit cut. Every
// fp32 step rounds to nearest with no fused multiply-add, so the codes are
// those of the written definition. A split (a, r) gives 2^(a+r-1) - 1 levels.
//
// A CTA encodes one page (256 tokens x 128 channels); thread (d, half) owns
// channel d over tokens 128 half .. 128 half + 127 and reads it straight from
// global memory (a warp reads 64 contiguous bytes a token; the passes after
// the first hit in L1), so occupancy is set by registers, not by a page
// buffer.
#include <cfloat>
#include <cmath>
#include <cuda_fp16.h>

#include "lynx_internal.cuh"

namespace lynx {
namespace {

constexpr int kThreadsV = 256;
constexpr int kMaxQ = 127;

struct VariantArgs {
    const uint16_t *x;            // [pages][256][128] bf16
    int16_t *codes;               // [pages][256][128] or null
    int8_t *anchor;               // [pages][256][128] or null
    uint8_t *resid;               // [pages][256][128] or null
    float *page_meta;             // [pages][2][128] or null
    uint16_t *chunk_meta;         // [pages][256 / C][2][128] or null
    double *err;                  // [pages][3] or null
    float *x_anchor, *x_full;     // [pages][256][128] fp32 reconstructions, or null
    int qmax, rbits, bias, flags, ubits;
    float thr[kMaxQ + 1];         // thr[k], k = 1..qmax, increasing; +inf above qmax (thr[0] unused)
    float lv[kMaxQ + 2];          // level value of |code| k = 0..qmax + 1 (fp16-exact)
};

struct SmemV {
    float thr[kMaxQ + 1];
    float lv[kMaxQ + 2];
    float mn[2][kD], mx[2][kD];
    int nan[2][kD];
    double red[kThreadsV / 32][3];
};

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Floor division by 2^r of a signed integer.
__device__ __forceinline__ int floor_shift(int b, int r) { return b >= 0 ? (b >> r) : -((-b + (1 << r) - 1) >> r); }

// Each thread's channel minimum and maximum over its half of the page (read
// straight from global memory: consecutive threads read consecutive
// channels), combined through shared memory; returns (mn, rng) of the channel
// over the page, NaN if it holds a NaN.
__device__ __forceinline__ void page_range(SmemV &sm, const uint16_t *__restrict__ xp, int d, int half, float &mn,
                                           float &rng)
{
    float lo = __int_as_float(0x7F800000), hi = -lo;
    int nan = 0;
    for (int t = 128 * half; t < 128 * half + 128; ++t) {
        const float v = bf16f(__ldg(xp + t * kD + d));
        if (v != v) {
            nan = 1;
            continue;
        }
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
    }
    sm.mn[half][d] = lo;
    sm.mx[half][d] = hi;
    sm.nan[half][d] = nan;
    __syncthreads();
    lo = fminf(sm.mn[0][d], sm.mn[1][d]) + 0.0f;    // a zero extreme is +0
    hi = fmaxf(sm.mx[0][d], sm.mx[1][d]) + 0.0f;
    rng = __fsub_rn(hi, lo);
    mn = lo;
    if (sm.nan[0][d] | sm.nan[1][d])
        mn = rng = __int_as_float(0x7FC00000);
    if (rng != rng)
        rng = __int_as_float(0x7FC00000);
}

// Deterministic block sum of three per-thread fp32 partials into err[0..2].
__device__ __forceinline__ void block_err(SmemV &sm, float e0, float e1, float e2, double *err)
{
    double v[3] = {e0, e1, e2};
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            v[k] += __shfl_xor_sync(0xFFFFFFFFu, v[k], o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        for (int k = 0; k < 3; ++k)
            sm.red[warp][k] = v[k];
    __syncthreads();
    if (threadIdx.x == 0 && err) {
        double s[3] = {0.0, 0.0, 0.0};
        for (int w = 0; w < kThreadsV / 32; ++w)
            for (int k = 0; k < 3; ++k)
                s[k] += sm.red[w][k];
        for (int k = 0; k < 3; ++k)
            err[k] = s[k];
    }
}

// RECON: the launch writes a reconstruction (the stores cost the errors-only
// study about 9 %, so that path is compiled without them)
template <int C, bool RECON>
__global__ void __launch_bounds__(kThreadsV) variant_kernel(const __grid_constant__ VariantArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SmemV &sm = *reinterpret_cast<SmemV *>(smem_raw);
    const int64_t page = blockIdx.x;
    const int d = threadIdx.x & (kD - 1), half = threadIdx.x >> 7;
    for (int i = threadIdx.x; i <= kMaxQ + 1; i += kThreadsV) {
        if (i <= a.qmax + 1)
            sm.lv[i] = a.lv[i];
        if (i <= kMaxQ)
            sm.thr[i] = a.thr[i];
    }
    const bool page_norm = !(a.flags & LYNX_VAR_NO_PAGE_NORM);
    const bool iso = !(a.flags & LYNX_VAR_NO_CHUNK_ISOLATION);
    const bool sign_aware = !(a.flags & LYNX_VAR_NO_SIGN_AWARE);
    float mn, rng;
    page_range(sm, a.x + page * kPage * kD, d, half, mn, rng);
    if (!page_norm) {
        mn = 0.0f;
        rng = 1.0f;
    }
    const float inv = rng > 0.0f ? __fdiv_rn(1.0f, rng) : 0.0f;
    const bool degenerate = page_norm && (!(rng <= FLT_MAX) || !(inv <= FLT_MAX));
    if (a.page_meta && half == 0) {
        a.page_meta[(page * 2 + 0) * kD + d] = mn;
        a.page_meta[(page * 2 + 1) * kD + d] = rng;
    }
    const uint16_t *__restrict__ xp = a.x + page * kPage * kD;
    auto u_of = [&](int t) -> float {    // stage 1 value of token t
        const float x = bf16f(__ldg(xp + t * kD + d));
        if (!page_norm)
            return x;
        return degenerate ? 0.0f : __fmul_rn(__fsub_rn(x, mn), inv);
    };
    float e0 = 0.0f, e1 = 0.0f, e2 = 0.0f;
    constexpr int nch = kPage / C;
    for (int j = (128 / C) * half; j < (128 / C) * (half + 1); ++j) {
        const int t0 = j * C;
        // stage 2: chunk mean (stride-halving tree) and max-abs scale
        uint16_t mu_b = 0x3800u, s_b = 0x3800u;    // 1/2, 1/2: the page's own centre
        float mu = 0.5f, sf = 0.5f, inv_s = 2.0f;
        if (iso) {
            float sl[C];
#pragma unroll
            for (int i = 0; i < C; ++i)
                sl[i] = u_of(t0 + i);
#pragma unroll
            for (int h = C / 2; h >= 1; h >>= 1)
#pragma unroll
                for (int i = 0; i < h; ++i)
                    sl[i] = __fadd_rn(sl[i], sl[i + h]);
            const __half mh = __float2half_rn(__fdiv_rn(sl[0], (float)C));
            mu = __half2float(mh);
            mu_b = __half_as_ushort(mh);
            float s = 0.0f;
            for (int i = 0; i < C; ++i)
                s = fmaxf(s, fabsf(__fsub_rn(u_of(t0 + i), mu)));
            const __half sh = __float2half_ru(s);
            sf = __half2float(sh);
            s_b = __half_as_ushort(sh);
            inv_s = sf > 0.0f ? __fdiv_rn(1.0f, sf) : 0.0f;
        }
        if (a.chunk_meta) {
            a.chunk_meta[((page * nch + j) * 2 + 0) * kD + d] = mu_b;
            a.chunk_meta[((page * nch + j) * 2 + 1) * kD + d] = s_b;
        }
        const float am = __fmaf_rn(rng, mu, mn), bm = __fmul_rn(rng, sf);   // decoder affines
        for (int i = 0; i < C; ++i) {
            const int t = t0 + i;
            const float w = __fmul_rn(__fsub_rn(u_of(t), mu), inv_s);
            // stage 3: level count #{k : |w| >= T_k}, by a fixed seven-step
            // search of the increasing thresholds (+inf past qmax; a NaN
            // compares false and counts 0)
            const float aw = fabsf(w);
            int lo = 0;
#pragma unroll
            for (int step = 64; step >= 1; step >>= 1)
                lo += aw >= sm.thr[lo + step] ? step : 0;
            const int c = w < 0.0f ? -(sign_aware ? max(lo, 1) : lo) : lo;
            // stage 4: bias and cut
            const int b = c + a.bias;
            const int A = floor_shift(b, a.rbits), r = b - (A << a.rbits);
            const int ca = A << a.rbits;
            const int64_t o = (page * kPage + t) * kD + d;
            if (a.codes)
                a.codes[o] = (int16_t)c;
            if (a.anchor)
                a.anchor[o] = (int8_t)A;
            if (a.resid)
                a.resid[o] = (uint8_t)r;
            const int kf = min(abs(c), a.qmax + 1), ka = min(abs(ca), a.qmax + 1);
            const float lf = c > 0 ? sm.lv[kf] : (c < 0 ? -sm.lv[kf] : 0.0f);
            const float la = ca > 0 ? sm.lv[ka] : (ca < 0 ? -sm.lv[ka] : 0.0f);
            const float x = bf16f(__ldg(xp + t * kD + d));
            const float xf = __fmaf_rn(bm, lf, am), xa = __fmaf_rn(bm, la, am);
            if (RECON && a.x_full)
                a.x_full[o] = xf;
            if (RECON && a.x_anchor)
                a.x_anchor[o] = xa;
            const float ef = __fsub_rn(xf, x), ea = __fsub_rn(xa, x);
            e0 = __fmaf_rn(x, x, e0);
            e1 = __fmaf_rn(ea, ea, e1);
            e2 = __fmaf_rn(ef, ef, e2);
        }
    }
    block_err(sm, e0, e1, e2, a.err ? a.err + page * 3 : nullptr);
}

// The uniform INTb comparator: per (page, channel) min-max grid of 2^b levels,
// code = floor((x - mn) * ((2^b - 1) / rng) + 1/2), every step in fp32.
template <bool RECON>
__global__ void __launch_bounds__(kThreadsV) uniform_kernel(const __grid_constant__ VariantArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SmemV &sm = *reinterpret_cast<SmemV *>(smem_raw);
    const int64_t page = blockIdx.x;
    const int d = threadIdx.x & (kD - 1), half = threadIdx.x >> 7;
    const uint16_t *__restrict__ xp = a.x + page * kPage * kD;
    float mn, rng;
    page_range(sm, xp, d, half, mn, rng);
    if (a.page_meta && half == 0) {
        const bool tok = a.flags & LYNX_VAR_UNIFORM_PER_TOKEN;   // no per-(page, channel) grid: zeros
        a.page_meta[(page * 2 + 0) * kD + d] = tok ? 0.0f : mn;
        a.page_meta[(page * 2 + 1) * kD + d] = tok ? 0.0f : rng;
    }
    const float top = (float)((1 << a.ubits) - 1);
    float e0 = 0.0f, e1 = 0.0f;
    if (a.flags & LYNX_VAR_UNIFORM_PER_TOKEN) {
        // per token: thread t owns token t, its grid over the 128 channels;
        // channel (j + t) mod 128 at step j keeps a warp on distinct banks
        const int t = threadIdx.x;
        float lo = __int_as_float(0x7F800000), hi = -lo;
        int nan = 0;
        for (int j = 0; j < kD; ++j) {
            const float v = bf16f(__ldg(xp + t * kD + ((j + t) & (kD - 1))));
            if (v != v) {
                nan = 1;
                continue;
            }
            lo = fminf(lo, v);
            hi = fmaxf(hi, v);
        }
        float tmn = lo + 0.0f, trg = __fsub_rn(hi + 0.0f, tmn);
        if (nan)
            tmn = trg = __int_as_float(0x7FC00000);
        const float inv_step = trg > 0.0f ? __fdiv_rn(top, trg) : 0.0f;
        const float step = __fdiv_rn(trg, top);
        for (int j = 0; j < kD; ++j) {
            const int dd = (j + t) & (kD - 1);
            const float x = bf16f(__ldg(xp + t * kD + dd));
            float q = floorf(__fadd_rn(__fmul_rn(__fsub_rn(x, tmn), inv_step), 0.5f));
            q = q != q ? 0.0f : fminf(fmaxf(q, 0.0f), top);
            if (a.codes)
                a.codes[(page * kPage + t) * kD + dd] = (int16_t)q;
            const float xr = __fmaf_rn(q, step, tmn);
            if (RECON && a.x_full)
                a.x_full[(page * kPage + t) * kD + dd] = xr;
            if (RECON && a.x_anchor)
                a.x_anchor[(page * kPage + t) * kD + dd] = xr;
            const float e = __fsub_rn(xr, x);
            e0 = __fmaf_rn(x, x, e0);
            e1 = __fmaf_rn(e, e, e1);
        }
        block_err(sm, e0, e1, e1, a.err ? a.err + page * 3 : nullptr);
        return;
    }
    const float inv_step = rng > 0.0f ? __fdiv_rn(top, rng) : 0.0f;
    const float step = __fdiv_rn(rng, top);
    for (int t = 128 * half; t < 128 * half + 128; ++t) {
        const float x = bf16f(__ldg(xp + t * kD + d));
        float q = floorf(__fadd_rn(__fmul_rn(__fsub_rn(x, mn), inv_step), 0.5f));
        q = q != q ? 0.0f : fminf(fmaxf(q, 0.0f), top);
        if (a.codes)
            a.codes[(page * kPage + t) * kD + d] = (int16_t)q;
        const float xr = __fmaf_rn(q, step, mn);
        if (RECON && a.x_full)
            a.x_full[(page * kPage + t) * kD + d] = xr;
        if (RECON && a.x_anchor)
            a.x_anchor[(page * kPage + t) * kD + d] = xr;
        const float e = __fsub_rn(xr, x);
        e0 = __fmaf_rn(x, x, e0);
        e1 = __fmaf_rn(e, e, e1);
    }
    block_err(sm, e0, e1, e1, a.err ? a.err + page * 3 : nullptr);
}

template <typename K>
cudaError_t launch_one(K kernel, const VariantArgs &a, dim3 grid, size_t smem, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kernel<<<grid, kThreadsV, smem, s>>>(a);
    return cudaGetLastError();
}

template <int C>
cudaError_t launch_variant(const VariantArgs &a, dim3 grid, size_t smem, cudaStream_t s, bool recon)
{
    return recon ? launch_one(variant_kernel<C, true>, a, grid, smem, s)
                 : launch_one(variant_kernel<C, false>, a, grid, smem, s);
}

} // namespace

cudaError_t launch_quantize_variant(const uint16_t *x, int64_t pages, const lynx_variant &v, int16_t *codes,
                                    int8_t *anchor, uint8_t *resid, float *page_meta, uint16_t *chunk_meta,
                                    double *err, float *x_anchor, float *x_full, cudaStream_t s)
{
    if (pages == 0)
        return cudaSuccess;
    VariantArgs a{};
    a.x = x;
    a.codes = codes;
    a.anchor = anchor;
    a.resid = resid;
    a.page_meta = page_meta;
    a.chunk_meta = chunk_meta;
    a.err = err;
    a.x_anchor = x_anchor;
    a.x_full = x_full;
    a.flags = (int)v.flags;
    a.ubits = v.uniform_bits;
    const size_t smem = sizeof(SmemV);
    const dim3 grid((unsigned)pages);
    const bool recon = x_anchor || x_full;
    if (v.uniform_bits > 0)
        return recon ? launch_one(uniform_kernel<true>, a, grid, smem, s)
                     : launch_one(uniform_kernel<false>, a, grid, smem, s);
    // Tables from the written map, in fp64 (thresholds where the map crosses
    // k - 1/2, levels at k), rounded to fp32 and fp16.
    const int qm = (1 << (v.anchor_bits + v.residual_bits - 2)) - 1;
    const double al = v.alpha;
    a.qmax = qm;
    a.rbits = v.residual_bits;
    a.bias = (v.flags & LYNX_VAR_NO_BIAS) ? 0 : (1 << (v.residual_bits - 1)) - 1;
    for (int k = 1; k <= qm; ++k)
        a.thr[k] = (float)(al > 0.0 ? (std::pow(1.0 + al, (k - 0.5) / qm) - 1.0) / al : (k - 0.5) / qm);
    for (int k = qm + 1; k <= kMaxQ; ++k)
        a.thr[k] = INFINITY;                    // never reached: the count stops at qmax
    for (int k = 0; k <= qm + 1; ++k)
        a.lv[k] = __half2float(__double2half(al > 0.0 ? (std::pow(1.0 + al, (double)k / qm) - 1.0) / al
                                                      : (double)k / qm));
    switch (v.chunk) {
    case 16:
        return launch_variant<16>(a, grid, smem, s, recon);
    case 32:
        return launch_variant<32>(a, grid, smem, s, recon);
    default:
        return launch_variant<64>(a, grid, smem, s, recon);
    }
}

} // namespace lynx
