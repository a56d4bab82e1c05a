// quantize.cu -- per-page Lynx encoder (K1) for sm_103a.
//
// "Lynx: the KV cache does not have to arrive whole" (aigenapps reading),
// section 3 "The quantizer": per 256-token page and channel, (1) page-level
// normalisation to [0,1]; (2) chunk-wise outlier isolation over C = 32 tokens,
// centring by the local mean and dividing by the local max-abs; (3) an
// alpha-law log map onto 127 levels with sign-aware mapping of negatives;
// (4) the +7 round-half-down bias and the 4-bit anchor / 4-bit residual cut.
//
// Layout of the work: a persistent CTA (one per SM) walks pages; each page
// (256 x 128 bf16 = 64 KiB, contiguous in [L][H][T][128]) is prefetched into
// one of two shared-memory buffers with a single bulk copy while the previous
// page is encoded. Warp j owns chunk j (32 tokens); lane l owns channels
// 4l..4l+3, so the chunk reduction tree of the numeric contract runs inside one
// thread's registers. The packed planes are staged in shared memory and leave
// with two 16 KiB bulk stores; the metadata goes out with direct 8/16-byte
// stores.
#include <cuda_fp16.h>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kPageBytes = kPage * kD * 2;       // 64 KiB of bf16
constexpr uint32_t kPlaneBytes = kPage * kD / 2;      // 16 KiB per plane and page
constexpr uint32_t kWaitLimit = 1u << 22;

struct Smem {
    uint16_t x[2][kPage * kD];         // double-buffered input page
    uint8_t anc[kPage * kD / 2];       // staged anchor plane of the page
    uint8_t res[kPage * kD / 2];       // staged residual plane of the page
    float pmin[kNChunk][kD];
    float pmax[kNChunk][kD];
    uint2 tab[kNBucket + 1];
    alignas(8) uint64_t bar[2];
};

struct Params {
    const uint16_t *x;
    const int32_t *page_valid;
    uint8_t *anc, *res;
    float *pm;
    uint16_t *cm;
    int64_t pages;  // L * H * P
    int P;          // pages per (layer, head)
};

// Stage 3: level count by bucket lookup plus one compare (equal to the count
// #{k : |w| >= T_k} for every finite w), then the sign-aware code.
__device__ __forceinline__ int level_code(float w, const uint2 *tab)
{
    const uint32_t ab = __float_as_uint(w) & 0x7FFFFFFFu;
    const uint32_t idx = min((ab >> 19) - kBucketBase, (uint32_t)kNBucket);
    const uint2 e = tab[idx];
    const int q = (int)e.y + (ab >= e.x ? 1 : 0);
    return (w < 0.0f) ? -max(q, 1) : q;
}

// Stages 2-4 for one channel of one chunk held in registers u[0..31].
// NC = 32 for a full chunk; otherwise nc valid tokens (runtime).
template <bool FULL>
__device__ __forceinline__ void chunk_channel(const float (&u)[kChunk], int nc, const uint2 *tab, int shift,
                                              uint32_t (&packed)[kChunk], __half &mu_out, __half &s_out)
{
    // chunk mean: stride-halving pairwise tree over 32 slots, absent slots +0
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = (FULL || i < nc) ? u[i] : 0.0f;
        const float b = (FULL || i + 16 < nc) ? u[i + 16] : 0.0f;
        t[i] = __fadd_rn(a, b);
    }
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i)
            t[i] = __fadd_rn(t[i], t[i + h]);
    const float mean = FULL ? __fdiv_rn(t[0], 32.0f) : __fdiv_rn(t[0], (float)nc);
    const __half mu_h = __float2half_rn(mean);
    const float mu = __half2float(mu_h);

    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
        if (FULL || i < nc)
            s = fmaxf(s, fabsf(__fsub_rn(u[i], mu)));
    const __half s_h = __float2half_ru(s);
    const float sf = __half2float(s_h);
    const float inv_s = sf > 0.0f ? __frcp_rn(sf) : 0.0f;

#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
        int c = 0;
        if (FULL || i < nc)
            c = level_code(__fmul_rn(__fsub_rn(u[i], mu), inv_s), tab);
        const uint32_t b = (uint32_t)(c + kBias) & 0xFFu;   // anchor nibble high, residual low
        // bits 0..15: anchor nibbles of the thread's 4 channels; 16..31: residual nibbles
        packed[i] |= ((b >> 4) << shift) | ((b & 15u) << (16 + shift));
    }
    mu_out = mu_h;
    s_out = s_h;
}

__global__ void __launch_bounds__(kThreads, 1) quantize_kernel(Params p, MapTable map)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const int j = tid >> 5;         // chunk of this warp
    const int lane = tid & 31;
    const int d0 = lane * 4;        // first of this thread's 4 channels

    for (int i = tid; i <= kNBucket; i += kThreads)
        sm.tab[i] = map.e[i];
    if (tid == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t first = blockIdx.x, stride = gridDim.x;
    if (tid == 0 && first < p.pages) {
        mbar_arrive_expect_tx(&sm.bar[0], kPageBytes);
        bulk_g2s(sm.x[0], p.x + first * (int64_t)(kPage * kD), kPageBytes, &sm.bar[0]);
    }

    int k = 0;
    bool prefetched = false;
    for (int64_t page = first; page < p.pages; page += stride, ++k) {
        const int buf = k & 1;
        const int64_t next = page + stride;
        prefetched = false;
        if (tid == 0 && next < p.pages) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sm.bar[buf ^ 1], kPageBytes);
            bulk_g2s(sm.x[buf ^ 1], p.x + next * (int64_t)(kPage * kD), kPageBytes, &sm.bar[buf ^ 1]);
            prefetched = true;
        }
        const bool ok = mbar_wait_bounded(&sm.bar[buf], (uint32_t)(k >> 1) & 1u, kWaitLimit);
        if (__syncthreads_or(!ok)) {
            // the copy never landed: stop, after letting any copy in flight finish
            if (tid == 0 && prefetched)
                mbar_wait_bounded(&sm.bar[buf ^ 1], (uint32_t)((k + 1) >> 1) & 1u, kWaitLimit);
            break;
        }

        int n = p.page_valid ? p.page_valid[page % p.P] : kPage;
        n = min(max(n, 0), kPage);
        const int nc = min(max(n - j * kChunk, 0), kChunk);

        // (a) this thread's 32 tokens x 4 channels
        const uint16_t *xs = sm.x[buf];
        uint2 xr[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            xr[i] = *reinterpret_cast<const uint2 *>(xs + (j * kChunk + i) * kD + d0);

        // (b) stage 1 statistics: chunk-local min/max, then across the page
        {
            float lmin[4], lmax[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                lmin[c] = __int_as_float(0x7F800000);
                lmax[c] = -__int_as_float(0x7F800000);
            }
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                if (i < nc) {
                    const float v0 = bf16_lo(xr[i].x), v1 = bf16_hi(xr[i].x);
                    const float v2 = bf16_lo(xr[i].y), v3 = bf16_hi(xr[i].y);
                    lmin[0] = fminf(lmin[0], v0); lmax[0] = fmaxf(lmax[0], v0);
                    lmin[1] = fminf(lmin[1], v1); lmax[1] = fmaxf(lmax[1], v1);
                    lmin[2] = fminf(lmin[2], v2); lmax[2] = fmaxf(lmax[2], v2);
                    lmin[3] = fminf(lmin[3], v3); lmax[3] = fmaxf(lmax[3], v3);
                }
            }
            *reinterpret_cast<float4 *>(&sm.pmin[j][d0]) = make_float4(lmin[0], lmin[1], lmin[2], lmin[3]);
            *reinterpret_cast<float4 *>(&sm.pmax[j][d0]) = make_float4(lmax[0], lmax[1], lmax[2], lmax[3]);
        }
        if (tid == 0)
            bulk_wait_read_all();   // the previous page's planes have left the staging tile
        __syncthreads();

        float mn[4], rng[4], inv_r[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float a = sm.pmin[0][d0 + c], b = sm.pmax[0][d0 + c];
#pragma unroll
            for (int jj = 1; jj < kNChunk; ++jj) {
                a = fminf(a, sm.pmin[jj][d0 + c]);
                b = fmaxf(b, sm.pmax[jj][d0 + c]);
            }
            if (n == 0)
                a = b = 0.0f;
            a = __fadd_rn(a, 0.0f);   // a zero minimum or maximum is +0
            b = __fadd_rn(b, 0.0f);
            mn[c] = a;
            rng[c] = __fsub_rn(b, a);
            inv_r[c] = rng[c] > 0.0f ? __frcp_rn(rng[c]) : 0.0f;
        }

        // stages 2-4, channel by channel; codes packed per token
        uint32_t packed[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            packed[i] = 0;
        __half mu_h[4], s_h[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float u[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const uint32_t w = (c < 2) ? xr[i].x : xr[i].y;
                const float x = (c & 1) ? bf16_hi(w) : bf16_lo(w);
                u[i] = __fmul_rn(__fsub_rn(x, mn[c]), inv_r[c]);
            }
            if (nc == kChunk) {
                chunk_channel<true>(u, nc, sm.tab, 4 * c, packed, mu_h[c], s_h[c]);
            } else if (nc > 0) {
                chunk_channel<false>(u, nc, sm.tab, 4 * c, packed, mu_h[c], s_h[c]);
            } else {
#pragma unroll
                for (int i = 0; i < kChunk; ++i)
                    packed[i] |= (uint32_t)kBias << (16 + 4 * c);   // code 0: anchor 0, residual 7
                mu_h[c] = __ushort_as_half(0);
                s_h[c] = __ushort_as_half(0);
            }
        }

        // stage the planes: anchor bytes (d0, d0+1), (d0+2, d0+3) of each token
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const int row = j * kChunk + i;
            *reinterpret_cast<uint16_t *>(&sm.anc[row * (kD / 2) + lane * 2]) = (uint16_t)(packed[i] & 0xFFFFu);
            *reinterpret_cast<uint16_t *>(&sm.res[row * (kD / 2) + lane * 2]) = (uint16_t)(packed[i] >> 16);
        }

        // metadata: page (min, range) from warp 0; chunk (mean, scale) from every thread
        if (j == 0) {
            float *pm = p.pm + page * (int64_t)(2 * kD);
            *reinterpret_cast<float4 *>(pm + d0) = make_float4(mn[0], mn[1], mn[2], mn[3]);
            *reinterpret_cast<float4 *>(pm + kD + d0) = make_float4(rng[0], rng[1], rng[2], rng[3]);
        }
        {
            uint16_t *cm = p.cm + (page * kNChunk + j) * (int64_t)(2 * kD);
            uint2 mu2, s2;
            mu2.x = (uint32_t)__half_as_ushort(mu_h[0]) | ((uint32_t)__half_as_ushort(mu_h[1]) << 16);
            mu2.y = (uint32_t)__half_as_ushort(mu_h[2]) | ((uint32_t)__half_as_ushort(mu_h[3]) << 16);
            s2.x = (uint32_t)__half_as_ushort(s_h[0]) | ((uint32_t)__half_as_ushort(s_h[1]) << 16);
            s2.y = (uint32_t)__half_as_ushort(s_h[2]) | ((uint32_t)__half_as_ushort(s_h[3]) << 16);
            *reinterpret_cast<uint2 *>(cm + d0) = mu2;
            *reinterpret_cast<uint2 *>(cm + kD + d0) = s2;
        }
        __syncthreads();
        if (tid == 0) {
            fence_proxy_async_smem();
            bulk_s2g(p.anc + page * (int64_t)kPlaneBytes, sm.anc, kPlaneBytes);
            bulk_s2g(p.res + page * (int64_t)kPlaneBytes, sm.res, kPlaneBytes);
            bulk_commit();
        }
    }
    if (tid == 0)
        bulk_wait_all();
}

__global__ void level_codes_kernel(const float *__restrict__ w, int64_t n, int8_t *__restrict__ codes,
                                   MapTable map)
{
    __shared__ uint2 tab[kNBucket + 1];
    for (int i = threadIdx.x; i <= kNBucket; i += blockDim.x)
        tab[i] = map.e[i];
    __syncthreads();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        codes[i] = (int8_t)level_code(w[i], tab);
}

} // namespace

cudaError_t launch_quantize(const uint16_t *x, const int32_t *page_valid, const lynx_qkv &o, cudaStream_t s)
{
    const int P = o.tokens / kPage;
    const int64_t pages = (int64_t)o.layers * o.kv_heads * P;
    if (pages == 0)
        return cudaSuccess;
    const int sms = device_sm_count();
    if (sms <= 0)
        return cudaErrorNoDevice;
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    Params p{x, page_valid, o.anchor, o.residual, o.page_meta, o.chunk_meta, pages, P};
    const int64_t grid = pages < sms ? pages : sms;
    quantize_kernel<<<(unsigned)grid, kThreads, smem, s>>>(p, host_tables().map);
    return cudaGetLastError();
}

cudaError_t launch_level_codes(const float *w, int64_t n, int8_t *codes, cudaStream_t s)
{
    if (n == 0)
        return cudaSuccess;
    const int sms = device_sm_count();
    if (sms <= 0)
        return cudaErrorNoDevice;
    int64_t blocks = (n + 255) / 256;
    if (blocks > (int64_t)sms * 8)
        blocks = (int64_t)sms * 8;
    level_codes_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, n, codes, host_tables().map);
    return cudaGetLastError();
}

} // namespace lynx
