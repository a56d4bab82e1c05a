// attn.cu -- fused-dequant paged decode attention (K4) for sm_103a, CUDA-core
// version.
//
// One decode step over the quantized paged cache: for request b and query head
// h (KV head g = h / G), scores s_t = sm_scale * q . K_t for t < ctx_b, softmax,
// output sum_t p_t V_t. K and V are never materialised: each element is decoded
// from its nibble(s) in registers (x = a + b * Ls(code), a and b per chunk and
// channel) right where Q.K^T or P.V consumes it ("KV-cache quantization"
// explainer, "Bottom-right": the fused kernel reads the compact cache and
// expands it only in registers). Anchor-only mode reads the anchor planes only
// (the draft cache of the Lynx reading, section 4); full mode adds the
// residual planes.
//
// Split-K: the pages of each (request, KV head) are cut into n_splits ranges,
// one CTA per (range, KV head, request); a CTA keeps a running (max, sum,
// output) per query head of its group and writes the partial triple, and a
// second kernel merges the triples with a log-sum-exp combine.
#include <cuda_fp16.h>

#include "lynx_internal.cuh"

namespace lynx {
namespace {

constexpr int kThreads = 256;
constexpr int kPart = kD + 2;     // floats per partial: o[128], m, l

template <int GMAX>
struct Smem {
    float q[GMAX][kD];
    float s[GMAX][kPage];
    uint8_t vc[kPage * kD / 2];
    uint8_t vr[kPage * kD / 2];
    float2 kab[kNChunk][kD];
    float2 vab[kNChunk][kD];
    float m[GMAX], l[GMAX], alpha[GMAX];
    float lut[256];
    int flag;
};

__device__ __forceinline__ void load_ab(float2 (*ab)[kD], const float *pm, const uint16_t *cm, int tid)
{
    for (int i = tid; i < kNChunk * kD; i += kThreads) {
        const int j = i / kD, d = i % kD;
        const float mn = pm[d], rg = pm[kD + d];
        const float mu = __half2float(__ushort_as_half(cm[(j * 2) * kD + d]));
        const float sc = __half2float(__ushort_as_half(cm[(j * 2 + 1) * kD + d]));
        ab[j][d] = make_float2(fmaf(rg, mu, mn), rg * sc);
    }
}

template <int GMAX, bool FULL>
__global__ void __launch_bounds__(kThreads, 1) attn_split_kernel(AttnArgs a, LevelTable lev)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<GMAX> &sm = *reinterpret_cast<Smem<GMAX> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = a.G;
    const int64_t T = (int64_t)a.pool_pages * kPage;

    for (int i = tid; i < 256; i += kThreads)
        sm.lut[i] = FULL ? lev.full[i] : lev.anchor[i & 15];
    for (int i = tid; i < GMAX * kD; i += kThreads) {
        const int h = i / kD, d = i % kD;
        float v = 0.0f;
        if (h < G) {
            const uint16_t bits = a.q[((int64_t)b * a.Hq + g * G + h) * kD + d];
            v = __uint_as_float((uint32_t)bits << 16);
        }
        sm.q[h][d] = v;
    }
    if (tid < GMAX) {
        sm.m[tid] = -__int_as_float(0x7F800000);
        sm.l[tid] = 0.0f;
    }

    int ctx = a.ctx[b];
    if (ctx < 0 || ctx > a.max_pages * kPage) {
        if (a.dev_err && split == 0 && g == 0 && tid == 0)
            atomicOr(a.dev_err, LYNX_DEVERR_CTX);
        ctx = min(max(ctx, 0), a.max_pages * kPage);
    }
    const uint8_t *ka = a.ka + (int64_t)g * T * (kD / 2);
    const uint8_t *kr = FULL ? a.kr + (int64_t)g * T * (kD / 2) : nullptr;
    const uint8_t *va = a.va + (int64_t)g * T * (kD / 2);
    const uint8_t *vr = FULL ? a.vr + (int64_t)g * T * (kD / 2) : nullptr;
    const float *kpm = a.kpm + (int64_t)g * a.pool_pages * (2 * kD);
    const float *vpm = a.vpm + (int64_t)g * a.pool_pages * (2 * kD);
    const uint16_t *kcm = a.kcm + (int64_t)g * a.pool_pages * (kNChunk * 2 * kD);
    const uint16_t *vcm = a.vcm + (int64_t)g * a.pool_pages * (kNChunk * 2 * kD);
    const int64_t score_stride = (int64_t)a.max_pages * kPage;

    // PV ownership: channel d, heads h = hh, hh + 2, ...
    const int d = tid & (kD - 1), hh = tid >> 7;
    float acc[GMAX / 2];
#pragma unroll
    for (int i = 0; i < GMAX / 2; ++i)
        acc[i] = 0.0f;

    const int p_begin = split * a.pages_per_split;
    const int p_end = min(p_begin + a.pages_per_split, a.max_pages);
    for (int lp = p_begin; lp < p_end; ++lp) {
        const int t0 = lp * kPage;
        const int nvalid = min(kPage, ctx - t0);
        int phys = -1;
        if (nvalid > 0) {
            phys = a.page_table[(int64_t)b * a.max_pages + lp];
            if (phys < 0 || phys >= a.pool_pages) {
                if (a.dev_err && tid == 0)
                    atomicOr(a.dev_err, LYNX_DEVERR_PAGE);
                phys = -1;
            }
        }
        if (phys < 0) {
            if (a.scores)
                for (int i = tid; i < G * kPage; i += kThreads)
                    a.scores[((int64_t)b * a.Hq + g * G + i / kPage) * score_stride + t0 + i % kPage] =
                        -__int_as_float(0x7F800000);
            continue;
        }
        __syncthreads();   // previous page fully consumed
        load_ab(sm.kab, kpm + (int64_t)phys * (2 * kD), kcm + (int64_t)phys * (kNChunk * 2 * kD), tid);
        load_ab(sm.vab, vpm + (int64_t)phys * (2 * kD), vcm + (int64_t)phys * (kNChunk * 2 * kD), tid);
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(va + (int64_t)phys * kPage * (kD / 2));
            uint4 *dst = reinterpret_cast<uint4 *>(sm.vc);
            for (int i = tid; i < kPage * kD / 32; i += kThreads)
                dst[i] = src[i];
            if (FULL) {
                const uint4 *src2 = reinterpret_cast<const uint4 *>(vr + (int64_t)phys * kPage * (kD / 2));
                uint4 *dst2 = reinterpret_cast<uint4 *>(sm.vr);
                for (int i = tid; i < kPage * kD / 32; i += kThreads)
                    dst2[i] = src2[i];
            }
        }
        __syncthreads();

        // scores: thread = token
        {
            const int t = tid;
            float s[GMAX];
#pragma unroll
            for (int h = 0; h < GMAX; ++h)
                s[h] = 0.0f;
            if (t < nvalid) {
                const int jc = t / kChunk;
                const uint4 *krow = reinterpret_cast<const uint4 *>(ka + ((int64_t)phys * kPage + t) * (kD / 2));
                const uint4 *rrow =
                    FULL ? reinterpret_cast<const uint4 *>(kr + ((int64_t)phys * kPage + t) * (kD / 2)) : nullptr;
#pragma unroll 1
                for (int blk = 0; blk < 4; ++blk) {
                    const uint4 av = krow[blk];
                    uint4 rv = make_uint4(0, 0, 0, 0);
                    if (FULL)
                        rv = rrow[blk];
                    const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
                    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                    for (int wv = 0; wv < 4; ++wv) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int dd = blk * 32 + wv * 8 + c;
                            const uint32_t an = (aw[wv] >> (4 * c)) & 15u;
                            const uint32_t idx = FULL ? ((an << 4) | ((rw[wv] >> (4 * c)) & 15u)) : an;
                            const float2 ab = sm.kab[jc][dd];
                            const float kv = fmaf(ab.y, sm.lut[idx], ab.x);
#pragma unroll
                            for (int h = 0; h < GMAX; ++h)
                                s[h] = fmaf(sm.q[h][dd], kv, s[h]);
                        }
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                if (h < G) {
                    const float v = t < nvalid ? s[h] * a.sm_scale : -__int_as_float(0x7F800000);
                    sm.s[h][t] = v;
                    if (a.scores)
                        a.scores[((int64_t)b * a.Hq + g * G + h) * score_stride + t0 + t] = v;
                }
            }
        }
        __syncthreads();

        // online softmax per head: warp w owns heads w, w + 8, ...
        for (int h = warp; h < G; h += kThreads / 32) {
            float mx = -__int_as_float(0x7F800000);
            for (int t = lane; t < nvalid; t += 32)
                mx = fmaxf(mx, sm.s[h][t]);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            const float m_old = sm.m[h];
            const float m_new = fmaxf(m_old, mx);
            float sum = 0.0f;
            for (int t = lane; t < nvalid; t += 32) {
                const float pv = expf(sm.s[h][t] - m_new);
                sm.s[h][t] = pv;
                sum += pv;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
            if (lane == 0) {
                const float al = expf(m_old - m_new);
                sm.alpha[h] = al;
                sm.l[h] = sm.l[h] * al + sum;
                sm.m[h] = m_new;
            }
        }
        __syncthreads();

        // P.V: thread = (channel d, heads of parity hh)
        {
#pragma unroll
            for (int i = 0; i < GMAX / 2; ++i)
                if (2 * i + hh < G)
                    acc[i] *= sm.alpha[2 * i + hh];
            const int sh = 4 * (d & 1);
            for (int t = 0; t < nvalid; ++t) {
                const uint32_t an = (sm.vc[t * (kD / 2) + (d >> 1)] >> sh) & 15u;
                const uint32_t idx = FULL ? ((an << 4) | ((sm.vr[t * (kD / 2) + (d >> 1)] >> sh) & 15u)) : an;
                const float2 ab = sm.vab[t / kChunk][d];
                const float vv = fmaf(ab.y, sm.lut[idx], ab.x);
#pragma unroll
                for (int i = 0; i < GMAX / 2; ++i)
                    if (2 * i + hh < G)
                        acc[i] = fmaf(sm.s[2 * i + hh][t], vv, acc[i]);
            }
        }
    }
    __syncthreads();

    // partial triples
    float *part = a.part;
#pragma unroll
    for (int i = 0; i < GMAX / 2; ++i) {
        const int h = 2 * i + hh;
        if (h < G)
            part[(((int64_t)b * a.Hq + g * G + h) * a.n_splits + split) * kPart + d] = acc[i];
    }
    if (tid < G) {
        float *pp = part + (((int64_t)b * a.Hq + g * G + tid) * a.n_splits + split) * kPart;
        pp[kD] = sm.m[tid] * 1.4426950408889634f;   // partials carry m in the base-2 log domain
        pp[kD + 1] = sm.l[tid];
    }
}

// Log-sum-exp merge of the page ranges' partials (base-2 log domain): one block
// per (request, query head), thread d owns channel d. One online pass over the
// partials, 16 at a time: their loads are all issued before any is used, so a
// merge of n ranges waits on about n / 16 rounds of memory latency.
__global__ void __launch_bounds__(kD) attn_combine_kernel(const float *__restrict__ part, int n_splits,
                                                          float *__restrict__ out)
{
    constexpr int U = 16;
    // launched as a programmatic dependent of the split kernel: everything
    // above this point overlaps its tail; the partials are read only after it
    // has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t bh = blockIdx.x;
    const int d = threadIdx.x;
    const float *pp = part + bh * n_splits * kPart;
    const float ninf = -__int_as_float(0x7F800000);

    float M = ninf, L = 0.0f, o = 0.0f;
    for (int s0 = 0; s0 < n_splits; s0 += U) {
        float mv[U], lv[U], ov[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool in = s0 + u < n_splits;
            const float *r = pp + (int64_t)(s0 + u) * kPart;
            mv[u] = in ? r[kD] : ninf;
            lv[u] = in ? r[kD + 1] : 0.0f;
            ov[u] = in ? r[d] : 0.0f;
        }
        float Mb = M;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (lv[u] > 0.0f)
                Mb = fmaxf(Mb, mv[u]);
        if (Mb > ninf) {
            const float c = M > ninf ? exp2f(M - Mb) : 0.0f;   // earlier ranges, to the new maximum
            L *= c;
            o *= c;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float w = lv[u] > 0.0f ? exp2f(mv[u] - Mb) : 0.0f;
                L = fmaf(lv[u], w, L);
                o = fmaf(ov[u], w, o);
            }
            M = Mb;
        }
    }
    out[bh * kD + d] = L > 0.0f ? o / L : 0.0f;
}

template <int GMAX, bool FULL>
cudaError_t run(const AttnArgs &a, cudaStream_t s)
{
    const size_t smem = sizeof(Smem<GMAX>);
    cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<GMAX, FULL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)a.n_splits, (unsigned)a.H, (unsigned)a.B);
    attn_split_kernel<GMAX, FULL><<<grid, kThreads, smem, s>>>(a, host_tables().lev);
    return cudaGetLastError();
}

} // namespace

void attn_split_plan(int batch, int kv_heads, int max_pages, int sms, int *n_splits, int *pages_per_split)
{
    // One CTA per SM runs at a time. When the (request, KV head) pairs are
    // fewer than the SMs, cut each context into as many ranges as fill one
    // wave; otherwise use short ranges so that many waves balance ragged
    // context lengths.
    const long units = (long)(batch > 0 ? batch : 1) * (kv_heads > 0 ? kv_heads : 1);
    int pps;
    if (units <= sms) {
        const int want = (int)(sms / units);
        pps = (max_pages + want - 1) / want;
    } else {
        pps = 8;
    }
    if (pps < 1)
        pps = 1;
    if (max_pages / pps > 8192)   // at most 8192 ranges (bounds the workspace and the combine)
        pps = (max_pages + 8191) / 8192;
    if (pps > max_pages)
        pps = max_pages > 0 ? max_pages : 1;
    *pages_per_split = pps;
    *n_splits = max_pages > 0 ? (max_pages + pps - 1) / pps : 1;
}

int attn_max_splits(int batch, int q_heads, int max_pages, int sms)
{
    int best = 1;
    for (int h = 1; h <= q_heads; ++h) {
        if (q_heads % h || q_heads / h > 32)
            continue;
        int n = 1, pps = 1;
        attn_split_plan(batch, h, max_pages, sms, &n, &pps);
        if (n > best)
            best = n;
    }
    return best;
}

size_t attn_workspace_bytes(int batch, int q_heads, int n_splits)
{
    return (size_t)batch * (size_t)q_heads * (size_t)n_splits * kPart * sizeof(float);
}

cudaError_t launch_attn_combine(const AttnArgs &a, cudaStream_t s)
{
    // programmatic dependent launch: the combine is scheduled while the split
    // kernel's last CTAs finish and waits for their results on the device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * a.Hq));
    cfg.blockDim = dim3(kD);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel, (const float *)a.part, a.n_splits, a.out);
}

cudaError_t launch_decode_attn(const AttnArgs &a, cudaStream_t s)
{
    if (a.B == 0 || a.Hq == 0)
        return cudaSuccess;
    cudaError_t e;
    if (a.G <= 16)
        e = launch_attn_mma(a, s);
    else
        e = a.full ? run<32, true>(a, s) : run<32, false>(a, s);
    if (e != cudaSuccess)
        return e;
    return launch_attn_combine(a, s);
}

} // namespace lynx
