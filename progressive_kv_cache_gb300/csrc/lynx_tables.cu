// lynx_tables.cu -- host-built tables of the Lynx quantizer, and device queries.
//
// Thresholds and level values come from section 3 of the aigenapps reading of
// Lynx (a logarithmic alpha-law map of |w| onto 127 levels, whose reconstructed
// magnitude grows geometrically as (1+alpha)^q), evaluated in double on the
// host and rounded once: thresholds to fp32, levels to fp16.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda_fp16.h>

#include "lynx_internal.cuh"

namespace lynx {

namespace {

uint32_t f32_bits(float f)
{
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

float f32_from_bits(uint32_t u)
{
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

uint16_t half_bits(__half h)
{
    uint16_t u;
    std::memcpy(&u, &h, 2);
    return u;
}

void build(HostTables &t)
{
    t.ok = true;
    t.thr[0] = 0.0f;
    for (int k = 1; k <= kQMax; ++k)
        t.thr[k] = (float)((std::pow(1.0 + kAlpha, (k - 0.5) / kQMax) - 1.0) / kAlpha);
    float lvf[65];
    for (int k = 0; k <= 64; ++k) {
        __half h = __double2half((std::pow(1.0 + kAlpha, (double)k / kQMax) - 1.0) / kAlpha);
        t.lv[k] = half_bits(h);
        lvf[k] = __half2float(h);
    }

    // stage-3 buckets: bucket of each threshold under the encoder's index
    // function, evaluated in fp32 exactly as on the device
    int tb[kQMax + 1];
    for (int k = 1; k <= kQMax; ++k) {
        volatile float sum = t.thr[k] + f32_from_bits(kBucketOffsetBits);
        tb[k] = (int)(f32_bits(sum) >> 19) - (int)kBucketBase;
        if (tb[k] < 0 || tb[k] >= kNBucket || !(t.thr[k] > 0.0f) || (k > 1 && !(t.thr[k] > t.thr[k - 1])))
            t.ok = false;
    }
    auto byte_of = [](int c) { return (uint32_t)(c + kBias) & 0xFFu; };
    for (int i = 0; i < kNBucket; ++i) {
        int q0 = 0, inside = 0, kin = 0;
        for (int k = 1; k <= kQMax; ++k) {
            if (tb[k] < i)
                ++q0;
            else if (tb[k] == i) {
                ++inside;
                kin = k;
            }
        }
        if (inside > 1)
            t.ok = false;   // would break the one-compare lookup
        const int q1 = q0 + 1 > kQMax ? kQMax : q0 + 1;
        const int n0 = -(q0 > 1 ? q0 : 1), n1 = -(q1 > 1 ? q1 : 1);
        const uint32_t bytes = byte_of(q0) | (byte_of(q1) << 8) | (byte_of(n0) << 16) | (byte_of(n1) << 24);
        // 2^30 - bits(T*) > 0 since T* <= 1 (bits below 2^30)
        const uint32_t k_add = inside ? (1u << 30) - f32_bits(t.thr[kin]) : 0u;
        if (inside && !(f32_bits(t.thr[kin]) < (1u << 30)))
            t.ok = false;
        t.code.e[i] = make_uint2(k_add, bytes);
    }

    // decoder levels
    for (int an = 0; an < 16; ++an) {
        int A = an >= 8 ? an - 16 : an;
        for (int r = 0; r < 16; ++r) {
            int c = 16 * A + r - kBias;
            int m = c < 0 ? -c : c;
            if (m > 64)
                m = 64;
            float v = lvf[m];
            t.lev.full[(an << 4) | r] = c < 0 ? -v : v;
        }
        int c = 16 * A;
        int m = c < 0 ? -c : c;
        if (m > 64)
            m = 64;
        t.lev.anchor[an] = c < 0 ? -lvf[m] : lvf[m];
    }
}

} // namespace

const HostTables &host_tables()
{
    static HostTables t;
    static std::once_flag once;
    std::call_once(once, [] { build(t); });
    return t;
}

int device_sm_count()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 0;
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64 && cache[dev])
        return cache[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev < 64)
        cache[dev] = sms;
    return sms;
}

} // namespace lynx
