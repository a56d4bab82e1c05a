// synth.cu -- GPU side of the seeded synthetic-input generator.
//
// Same definition as lynx_synth/__init__.py (SplitMix64 counter hash, Exp(1)
// quantile table, random sign, per-channel fp32 scale, bf16 nearest-even).
// Input generation only: none of the quantizer's arithmetic is here.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t z)
{
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t bf16_rn(float f)
{
    uint32_t u = __float_as_uint(f);
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    return (uint16_t)u;
}

// out: [rows_lh][T][D] bf16 bits; scales: [rows_lh][D]; each thread writes 8
// consecutive channels (one 16-byte store).
__global__ void fill_kernel(uint4 *__restrict__ out, uint64_t key, const float *__restrict__ scales,
                            const float *__restrict__ table, int64_t n_vec, int64_t T, int64_t D)
{
    const int64_t vec_per_row = D / 8;
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n_vec;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i0 = v * 8;
        const int64_t lh = v / (vec_per_row * T);
        const int64_t d0 = (v % vec_per_row) * 8;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            uint16_t b[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint64_t h = splitmix64(key + (uint64_t)(i0 + e + k));
                float mag = table[(h >> 47) & 0xFFFFu];
                float val = (h >> 63) ? -mag : mag;
                b[k] = bf16_rn(__fmul_rn(val, scales[lh * D + d0 + e + k]));
            }
            w[e / 2] = (uint32_t)b[0] | ((uint32_t)b[1] << 16);
        }
        out[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

} // namespace

extern "C" int synth_fill_laplace_bf16(void *out, uint64_t key, const float *scales,
                                       const float *table, int64_t rows_lh, int64_t T, int64_t D,
                                       void *stream)
{
    if (!out || !scales || !table || D % 8 || rows_lh < 0 || T < 0)
        return 1;
    const int64_t n_vec = rows_lh * T * D / 8;
    if (n_vec == 0)
        return 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (n_vec + 255) / 256;
    if (blocks > (int64_t)sms * 16)
        blocks = (int64_t)sms * 16;
    fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>((uint4 *)out, key, scales, table,
                                                                   n_vec, T, D);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
