// dequant.cu -- anchor-only reconstruction (K2) and in-place residual
// refinement (K3) for sm_103a.
//
// "Lynx: the KV cache does not have to arrive whole" (aigenapps reading),
// section 4: the anchor planes alone give the draft cache that decoding starts
// from; once the residual planes are in, the cache is refined to the full
// quantization. Both are streaming decodes of the planes: per element one nibble
// (pair) lookup and one fused multiply-add,
//   x = a + b * Ls(code),  a = mn + rng * mu,  b = rng * s  (per chunk, channel).
// Refinement rewrites the dense cache written by the anchor pass with the full
// reconstruction, reading only the planes (1.16 B/element instead of the 2
// B/element of the dense draft).
//
// Work: persistent CTAs (two or four per SM) walk pages. A page's planes and metadata
// arrive by bulk copy into one of two shared-memory stages while the previous
// page is decoded, so reads never wait in the compute loop. Warp w decodes
// chunk w (32 tokens): lane l owns channels 8(l%16)..+7 of rows 2i + l/16 and
// writes them with one 16-byte store (bf16) or two (fp32); a warp's store
// covers 512 contiguous bytes. Code bytes are assembled four at a time with
// word-wide nibble masks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kPlane = kPage * kD / 2;   // 16 KiB
constexpr uint32_t kWaitLimit = 1u << 22;

template <bool FULL>
struct Stage {
    uint8_t anc[kPlane];
    uint8_t res[FULL ? kPlane : 16];
    float pm[2 * kD];
    uint16_t cm[kNChunk * 2 * kD];
};

template <bool FULL>
struct Smem {
    Stage<FULL> st[2];
    // full mode: 256 signed levels, one copy per lane (conflict-free lookups);
    // anchor mode: 16 levels, one word per bank already
    float lut[FULL ? 256 * 32 : 16];
    alignas(8) uint64_t bar[2];
};

struct Params {
    const uint8_t *anc, *res;
    const float *pm;
    const uint16_t *cm;
    void *out;
    int64_t pages;   // L * H * P
};

template <bool FULL>
constexpr int ctas_per_sm() { return FULL ? 2 : 4; }   // bounded by shared memory (full) and registers

template <bool FULL, bool F32>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<FULL>()) dequant_kernel(Params p, LevelTable lev)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<FULL> &sm = *reinterpret_cast<Smem<FULL> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, j = tid >> 5;
    const int cg = lane & 15;        // channel group: channels 8cg..8cg+7
    const int rp = lane >> 4;        // row parity

    for (int i = tid; i < (FULL ? 256 * 32 : 16); i += kThreads)
        sm.lut[i] = FULL ? lev.full[i >> 5] : lev.anchor[i];
    if (tid == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const float *lut_lane = FULL ? sm.lut + lane : sm.lut;

    auto issue = [&](int64_t page, int s) {
        Stage<FULL> &st = sm.st[s];
        const uint32_t bytes = (FULL ? 2u : 1u) * kPlane + 2 * kD * 4 + kNChunk * 2 * kD * 2;
        mbar_arrive_expect_tx(&sm.bar[s], bytes);
        bulk_g2s(st.anc, p.anc + page * kPlane, kPlane, &sm.bar[s]);
        if (FULL)
            bulk_g2s(st.res, p.res + page * kPlane, kPlane, &sm.bar[s]);
        bulk_g2s(st.pm, p.pm + page * (2 * kD), 2 * kD * 4, &sm.bar[s]);
        bulk_g2s(st.cm, p.cm + page * (kNChunk * 2 * kD), kNChunk * 2 * kD * 2, &sm.bar[s]);
    };

    const int64_t first = blockIdx.x, stride = gridDim.x;
    if (tid == 0) {
        if (first < p.pages)
            issue(first, 0);
        if (first + stride < p.pages)
            issue(first + stride, 1);
    }
    uint32_t phase[2] = {0u, 0u};
    int k = 0;
    for (int64_t page = first; page < p.pages; page += stride, ++k) {
        const int s = k & 1;
        const bool ok = mbar_wait_bounded(&sm.bar[s], phase[s], kWaitLimit);
        if (__syncthreads_or(!ok)) {
            // a copy never landed: let the one in flight land (bounded), then stop
            if (tid == 0 && page + stride < p.pages)
                mbar_wait_bounded(&sm.bar[s ^ 1], phase[s ^ 1], kWaitLimit);
            break;
        }
        phase[s] ^= 1u;
        const Stage<FULL> &st = sm.st[s];

        // chunk affine of this lane's 8 channels
        float a[8], b[8];
        {
            const float4 mn0 = *reinterpret_cast<const float4 *>(st.pm + cg * 8);
            const float4 mn1 = *reinterpret_cast<const float4 *>(st.pm + cg * 8 + 4);
            const float4 rg0 = *reinterpret_cast<const float4 *>(st.pm + kD + cg * 8);
            const float4 rg1 = *reinterpret_cast<const float4 *>(st.pm + kD + cg * 8 + 4);
            const uint4 mu8 = *reinterpret_cast<const uint4 *>(st.cm + (j * 2) * kD + cg * 8);
            const uint4 s8 = *reinterpret_cast<const uint4 *>(st.cm + (j * 2 + 1) * kD + cg * 8);
            const float mn[8] = {mn0.x, mn0.y, mn0.z, mn0.w, mn1.x, mn1.y, mn1.z, mn1.w};
            const float rg[8] = {rg0.x, rg0.y, rg0.z, rg0.w, rg1.x, rg1.y, rg1.z, rg1.w};
            const uint32_t muw[4] = {mu8.x, mu8.y, mu8.z, mu8.w};
            const uint32_t sw[4] = {s8.x, s8.y, s8.z, s8.w};
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint16_t mub = (uint16_t)(muw[c >> 1] >> (16 * (c & 1)));
                const uint16_t sb = (uint16_t)(sw[c >> 1] >> (16 * (c & 1)));
                a[c] = fmaf(rg[c], __half2float(__ushort_as_half(mub)), mn[c]);
                b[c] = rg[c] * __half2float(__ushort_as_half(sb));
            }
        }

        const int64_t row0 = page * kPage + j * kChunk + rp;
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
            const int r = j * kChunk + rp + 2 * it;   // row within the page
            const uint32_t aw = *reinterpret_cast<const uint32_t *>(st.anc + r * (kD / 2) + cg * 4);
            // code bytes of the even and of the odd channels, four per word:
            // full (A << 4 | r), anchor-only A
            uint32_t ev, od;
            if (FULL) {
                const uint32_t rw = *reinterpret_cast<const uint32_t *>(st.res + r * (kD / 2) + cg * 4);
                ev = ((aw << 4) & 0xF0F0F0F0u) | (rw & 0x0F0F0F0Fu);
                od = (aw & 0xF0F0F0F0u) | ((rw >> 4) & 0x0F0F0F0Fu);
            } else {
                ev = aw & 0x0F0F0F0Fu;
                od = (aw >> 4) & 0x0F0F0F0Fu;
            }
            float x[8];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t ie = __byte_perm(ev, 0u, 0x4440u | kk);
                const uint32_t io = __byte_perm(od, 0u, 0x4440u | kk);
                x[2 * kk] = fmaf(b[2 * kk], lut_lane[FULL ? ie * 32 : ie], a[2 * kk]);
                x[2 * kk + 1] = fmaf(b[2 * kk + 1], lut_lane[FULL ? io * 32 : io], a[2 * kk + 1]);
            }
            const int64_t row = row0 + 2 * it;
            if (F32) {
                float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * kD + cg * 8);
                o[0] = make_float4(x[0], x[1], x[2], x[3]);
                o[1] = make_float4(x[4], x[5], x[6], x[7]);
            } else {
                uint4 v;
                __nv_bfloat162 h0 = __floats2bfloat162_rn(x[0], x[1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(x[2], x[3]);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(x[4], x[5]);
                __nv_bfloat162 h3 = __floats2bfloat162_rn(x[6], x[7]);
                v.x = *reinterpret_cast<uint32_t *>(&h0);
                v.y = *reinterpret_cast<uint32_t *>(&h1);
                v.z = *reinterpret_cast<uint32_t *>(&h2);
                v.w = *reinterpret_cast<uint32_t *>(&h3);
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + row * kD + cg * 8) = v;
            }
        }
        __syncthreads();   // stage s consumed
        if (tid == 0 && page + 2 * stride < p.pages) {
            fence_proxy_async_smem();
            issue(page + 2 * stride, s);
        }
    }
}

template <bool FULL, bool F32>
cudaError_t run(const Params &p, cudaStream_t s)
{
    const int sms = device_sm_count();
    if (sms <= 0)
        return cudaErrorNoDevice;
    const size_t smem = sizeof(Smem<FULL>);
    cudaError_t e =
        cudaFuncSetAttribute(dequant_kernel<FULL, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int64_t blocks = (int64_t)ctas_per_sm<FULL>() * sms;
    if (blocks > p.pages)
        blocks = p.pages;
    dequant_kernel<FULL, F32><<<(unsigned)blocks, kThreads, smem, s>>>(p, host_tables().lev);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_dequant(const lynx_qkv &in, void *out, bool full, bool f32, cudaStream_t s)
{
    const int64_t pages = (int64_t)in.layers * in.kv_heads * (in.tokens / kPage);
    if (pages == 0)
        return cudaSuccess;
    Params p{in.anchor, in.residual, in.page_meta, in.chunk_meta, out, pages};
    if (full)
        return f32 ? run<true, true>(p, s) : run<true, false>(p, s);
    return f32 ? run<false, true>(p, s) : run<false, false>(p, s);
}

} // namespace lynx
