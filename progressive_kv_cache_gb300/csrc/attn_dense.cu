// attn_dense.cu -- decode attention over a dense fp32 cache, a diagnostic for
// quality studies: the attention output of a reconstruction set against the
// same attention over the original values ("vNMSE of the attention output",
// section 5 of the Lynx reading). It is not part of the method's path.
//
// out[b][h] = sum_t softmax_t(sm_scale q[b][h] . k[g][t]) v[g][t], g = h / (Hq / H),
// every request attending to all `T` tokens. One CTA per (request, query
// head): the row's scores live in shared memory (T <= kMaxTokens), then one
// max, the weights and their sum, and an output pass in which thread
// (channel, half) sums its channel over half of the tokens. fp32 throughout.
#include <cuda_bf16.h>

#include "lynx_internal.cuh"

namespace lynx {
namespace {

constexpr int kThreadsA = 256;
constexpr int kMaxTokens = 49152;             // 192 KiB of scores

__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = is_max ? fmaxf(v, w) : v + w;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();                         // earlier readers of `red` are done
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < kThreadsA / 32; ++w)
        r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

__global__ void __launch_bounds__(kThreadsA) dense_attn_kernel(const uint16_t *__restrict__ q,
                                                              const float *__restrict__ k,
                                                              const float *__restrict__ v, int Hq, int H, int T,
                                                              float scale2, float *__restrict__ out)
{
    extern __shared__ float sc[];            // T scores, then T weights
    __shared__ float red[kThreadsA / 32];
    __shared__ float qs[kD];
    __shared__ float half_o[kD];
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int kvh = h / (Hq / H);
    if (tid < kD)
        qs[tid] = __uint_as_float((uint32_t)q[((int64_t)b * Hq + h) * kD + tid] << 16) * scale2;
    __syncthreads();
    const float *kb = k + (int64_t)kvh * T * kD, *vb = v + (int64_t)kvh * T * kD;
    float mx = -__int_as_float(0x7F800000);
    for (int t = tid; t < T; t += kThreadsA) {
        const float4 *kr = reinterpret_cast<const float4 *>(kb + (int64_t)t * kD);
        float s = 0.0f;
#pragma unroll 8
        for (int i = 0; i < kD / 4; ++i) {
            const float4 kv = __ldg(kr + i);
            s = fmaf(qs[4 * i], kv.x, s);
            s = fmaf(qs[4 * i + 1], kv.y, s);
            s = fmaf(qs[4 * i + 2], kv.z, s);
            s = fmaf(qs[4 * i + 3], kv.w, s);
        }
        sc[t] = s;
        mx = fmaxf(mx, s);
    }
    mx = block_reduce(mx, true, red);
    float l = 0.0f;
    for (int t = tid; t < T; t += kThreadsA) {
        const float p = exp2f(sc[t] - mx);
        sc[t] = p;
        l += p;
    }
    l = block_reduce(l, false, red);         // also orders the weights before the output pass
    const int ch = tid & (kD - 1), hf = tid >> 7;
    float o = 0.0f;
    for (int t = hf; t < T; t += 2)
        o = fmaf(sc[t], __ldg(vb + (int64_t)t * kD + ch), o);
    if (hf == 1)
        half_o[ch] = o;
    __syncthreads();
    if (hf == 0)
        out[((int64_t)b * Hq + h) * kD + ch] = (o + half_o[ch]) / l;
}

} // namespace

cudaError_t launch_dense_attn(const uint16_t *q, const float *k, const float *v, int B, int Hq, int H, int T,
                              float sm_scale, float *out, cudaStream_t s)
{
    if (B == 0 || Hq == 0)
        return cudaSuccess;
    const size_t smem = (size_t)T * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(dense_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kMaxTokens * sizeof(float)));
    if (e != cudaSuccess)
        return e;
    dense_attn_kernel<<<dim3((unsigned)Hq, (unsigned)B), kThreadsA, smem, s>>>(q, k, v, Hq, H, T,
                                                                               sm_scale * 1.4426950408889634f, out);
    return cudaGetLastError();
}

int dense_attn_max_tokens() { return kMaxTokens; }

} // namespace lynx
