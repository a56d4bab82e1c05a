// dequant.cu -- anchor-only reconstruction (K2) and in-place residual
// refinement (K3) for sm_103a.
//
// "Lynx: the KV cache does not have to arrive whole" (aigenapps reading),
// section 4: the anchor stream alone is the draft cache ("Anchor stream lands,
// decoding starts"); when the residual lands "the kernel refines the cache to
// Q_full". Both are streaming decodes of the planes: per element one nibble (or
// nibble pair) lookup and one fused multiply-add,
//   x = a + b * Ls(code),  a = mn + rng * mu,  b = rng * s  (per chunk, channel).
// Refinement rewrites the dense cache written by the anchor pass with the full
// reconstruction, reading only the planes (1.16 B/element instead of the 2
// B/element of the dense draft).
//
// Work unit: one 32-token chunk of one (layer, head, page) = 4096 elements,
// owned by one warp; lane l decodes channels 8(l%16)..+7 of rows 2i + l/16.
// Code bytes are assembled four at a time with word-wide nibble masks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lynx_internal.cuh"

namespace lynx {
namespace {

constexpr int kThreads = 256;

struct Params {
    const uint8_t *anc, *res;
    const float *pm;
    const uint16_t *cm;
    void *out;
    int64_t units;   // L * H * P * 8 chunks
};

template <bool FULL, bool F32>
__global__ void __launch_bounds__(kThreads) dequant_kernel(Params p, LevelTable lev)
{
    // Full mode: 256 signed level values, replicated 32 times so that lane l
    // reads only bank l (random codes would otherwise conflict); anchor mode:
    // 16 values, one word per bank already.
    constexpr int kLut = FULL ? 256 * 32 : 16;
    __shared__ float lut[kLut];
    for (int i = threadIdx.x; i < kLut; i += kThreads)
        lut[i] = FULL ? lev.full[i >> 5] : lev.anchor[i];
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int cg = lane & 15;        // channel group: channels 8cg..8cg+7
    const int rp = lane >> 4;        // row parity
    const float *lut_lane = FULL ? lut + lane : lut;
    const int64_t wstride = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t u = blockIdx.x * (int64_t)(kThreads / 32) + (threadIdx.x >> 5); u < p.units; u += wstride) {
        const int64_t page = u >> 3;
        const int j = (int)(u & 7);
        const float *pm = p.pm + page * (2 * kD) + cg * 8;
        const float4 mn0 = *reinterpret_cast<const float4 *>(pm);
        const float4 mn1 = *reinterpret_cast<const float4 *>(pm + 4);
        const float4 rg0 = *reinterpret_cast<const float4 *>(pm + kD);
        const float4 rg1 = *reinterpret_cast<const float4 *>(pm + kD + 4);
        const uint16_t *cm = p.cm + (page * kNChunk + j) * (2 * kD) + cg * 8;
        const uint4 mu8 = *reinterpret_cast<const uint4 *>(cm);
        const uint4 s8 = *reinterpret_cast<const uint4 *>(cm + kD);
        const float mn[8] = {mn0.x, mn0.y, mn0.z, mn0.w, mn1.x, mn1.y, mn1.z, mn1.w};
        const float rg[8] = {rg0.x, rg0.y, rg0.z, rg0.w, rg1.x, rg1.y, rg1.z, rg1.w};
        const uint32_t muw[4] = {mu8.x, mu8.y, mu8.z, mu8.w};
        const uint32_t sw[4] = {s8.x, s8.y, s8.z, s8.w};
        float a[8], b[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint16_t mub = (uint16_t)(muw[c >> 1] >> (16 * (c & 1)));
            const uint16_t sb = (uint16_t)(sw[c >> 1] >> (16 * (c & 1)));
            a[c] = fmaf(rg[c], __half2float(__ushort_as_half(mub)), mn[c]);
            b[c] = rg[c] * __half2float(__ushort_as_half(sb));
        }

        const int64_t row0 = page * kPage + j * kChunk + rp;
        uint32_t aw[16], rw[16];
#pragma unroll
        for (int it = 0; it < 16; ++it) {
            const int64_t row = row0 + 2 * it;
            aw[it] = __ldg(reinterpret_cast<const uint32_t *>(p.anc + row * (kD / 2) + cg * 4));
            rw[it] = FULL ? __ldg(reinterpret_cast<const uint32_t *>(p.res + row * (kD / 2) + cg * 4)) : 0u;
        }
#pragma unroll
        for (int it = 0; it < 16; ++it) {
            const int64_t row = row0 + 2 * it;
            // code bytes of the even and of the odd channels, four per word:
            // full (A << 4 | r), anchor-only A
            uint32_t ev, od;
            if (FULL) {
                ev = ((aw[it] << 4) & 0xF0F0F0F0u) | (rw[it] & 0x0F0F0F0Fu);
                od = (aw[it] & 0xF0F0F0F0u) | ((rw[it] >> 4) & 0x0F0F0F0Fu);
            } else {
                ev = aw[it] & 0x0F0F0F0Fu;
                od = (aw[it] >> 4) & 0x0F0F0F0Fu;
            }
            float x[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t ie = __byte_perm(ev, 0u, 0x4440u | k);
                const uint32_t io = __byte_perm(od, 0u, 0x4440u | k);
                x[2 * k] = fmaf(b[2 * k], lut_lane[FULL ? ie * 32 : ie], a[2 * k]);
                x[2 * k + 1] = fmaf(b[2 * k + 1], lut_lane[FULL ? io * 32 : io], a[2 * k + 1]);
            }
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
    }
}

template <bool FULL, bool F32>
cudaError_t run(const Params &p, cudaStream_t s)
{
    const int sms = device_sm_count();
    if (sms <= 0)
        return cudaErrorNoDevice;
    int64_t blocks = (p.units + 7) / 8;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap)
        blocks = cap;
    dequant_kernel<FULL, F32><<<(unsigned)blocks, kThreads, 0, s>>>(p, host_tables().lev);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_dequant(const lynx_qkv &in, void *out, bool full, bool f32, cudaStream_t s)
{
    const int64_t units = (int64_t)in.layers * in.kv_heads * (in.tokens / kPage) * kNChunk;
    if (units == 0)
        return cudaSuccess;
    Params p{in.anchor, in.residual, in.page_meta, in.chunk_meta, out, units};
    if (full)
        return f32 ? run<true, true>(p, s) : run<true, false>(p, s);
    return f32 ? run<false, true>(p, s) : run<false, false>(p, s);
}

} // namespace lynx
