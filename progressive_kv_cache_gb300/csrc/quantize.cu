// quantize.cu -- per-page Lynx encoder (K1) for sm_103a.
//
// "Lynx: the KV cache does not have to arrive whole" (aigenapps reading),
// section 3 "The quantizer": per 256-token page and channel, (1) page-level
// normalisation to [0,1]; (2) chunk-wise outlier isolation over C = 32 tokens,
// centring by the local mean and dividing by the local max-abs; (3) an
// alpha-law log map onto 127 levels with sign-aware mapping of negatives;
// (4) the +7 round-half-down bias and the 4-bit anchor / 4-bit residual cut.
//
// Layout of the work: the unit of work is one channel half of a page (256
// tokens x 64 channels; the statistics are per channel, so the two halves of
// a page are independent). Persistent CTAs of 8 warps, two per SM, walk the
// units; a unit arrives by one 2D tensor copy (TMA, rows of 128 bytes out of
// the page's 256) into a single input buffer, which is refilled with the next
// unit (already on its way to L2) as soon as the current one is in registers,
// and the two CTAs of an SM run out of step, so that one's barriers and
// latency-bound stretches overlap the other's stage 3 (one 16-warp CTA per
// page with a double-buffered input keeps all warps in the same phase and
// runs 1.8 % slower). Warp w owns chunk
// w (32 tokens); lane l owns one channel pair, so the chunk reduction tree
// of the numeric contract runs inside one thread's registers. Stage 3 is one
// lookup in a 16-way replicated bucket table (a conflict-free 8-byte load per
// element) whose entry carries the four possible stored bytes, then one
// integer add and one byte permute; the odd channel of a pair reads a second
// table with the nibbles of each byte swapped, so that one more permute
// merges the pair and the two plane bytes are a shift and a logic operation
// away. The packed planes are staged in shared memory and leave with two 2D
// tensor stores of 8 KiB (256 rows of 32 bytes); the metadata goes out with
// direct 4/8-byte stores. Two barriers a unit: after the chunk extremes (which
// also carries the outcome of the bounded wait for the unit) and before the
// tensor stores.
//
// The kernel is bound by instruction issue, so the per-element work is kept
// short: the bucket index needs no clamp (|w| + 2^-13 always lands in the
// table), the threshold test and the sign of w come out of one integer add
// as the byte index, and the chunk's max |v| comes from its two extremes
// instead of a max over all elements (v is a monotone function of x, so the
// extremes of x give the extremes of v). Storing the planes straight to
// global memory (no staging, one barrier a page) needs fewer instructions
// but stalls on the load/store unit and runs slower.
// Codes are computed for a group of tokens before the group's stores: a table
// load may not move above an earlier store to shared memory, so interleaving
// them would serialise the tokens.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr int kHalf = kD / 2;                          // channels of one work unit
constexpr int kRowB = kHalf / 2;                       // plane bytes of one token in a unit
constexpr int kThreads = kNChunk * 32;                 // a warp per chunk, a lane per channel pair
constexpr int kCopies = 16;                            // table replicas (one per half-warp lane)
constexpr uint32_t kUnitBytes = kPage * kHalf * 2;    // 32 KiB of bf16
constexpr uint32_t kTabBytes = kNBucket * kCopies * 8; // one replicated table
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kQNaN = 0x7FC00000u;
constexpr int kGroup = 16;                           // tokens whose codes are computed before their stores
                                                     // (measured: 16 runs 0.7 % faster than 8, 0.5 % than 32
                                                     // and 3.2 % than 4)
static_assert(kGroup > 0 && kChunk % kGroup == 0, "groups must tile the chunk");
constexpr float kF32Max = 3.40282347e38f;


struct Smem {
    uint16_t x[kPage * kHalf];         // the unit's input: 256 tokens x 64 channels
    uint8_t anc[kPage * kRowB];        // staged anchor plane of the unit
    uint8_t res[kPage * kRowB];        // staged residual plane of the unit
    uint2 pmm[kNChunk][kHalf / 2];     // bf16x2 chunk (minima, maxima) of channel pairs
    // [0]: the stored bytes; [1]: the same bytes with their nibbles swapped
    // (the odd channel of a pair)
    uint2 tab[2][kNBucket * kCopies];
    alignas(8) uint64_t bar;
};

struct Params {
    const uint16_t *x;            // source pages, one after another
    const int32_t *page_valid;
    uint8_t *anc, *res;
    float *pm;
    uint16_t *cm;
    int64_t pages;                // source pages: L * H * P, or n * L * H when appending
    int P;                        // pages per (layer, head) of the destination
    // appending: source page i = (tail i / LH, layer-head i % LH) is encoded
    // into physical page dst_page[i / LH] of that layer-head, with
    // tail_valid[i / LH] valid tokens; NULL for the whole-tensor encoder
    const int32_t *dst_page;
    const int32_t *tail_valid;
    int LH;
    uint32_t *dev_err;
};

// Destination page of source page i (-1: outside the pool, flagged).
__device__ __forceinline__ int64_t dst_of(const Params &p, int64_t i)
{
    if (!p.dst_page)
        return i;
    const int d = p.dst_page[i / p.LH];
    return (d >= 0 && d < p.P) ? (i % p.LH) * (int64_t)p.P + d : -1;
}

// Valid tokens of source page i (clamped to 0..256).
__device__ __forceinline__ int valid_of(const Params &p, int64_t i)
{
    const int n = p.dst_page ? p.tail_valid[i / p.LH] : (p.page_valid ? p.page_valid[i % p.P] : kPage);
    return min(max(n, 0), kPage);
}

__device__ __forceinline__ uint2 lds_u2(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// Bucket-table entry of w (|w| < 2) in table TAB. `tab_base` is the shared
// address of this lane's replica of table 0, offset so that the bucket number
// indexes it directly; `stride` is the byte distance between buckets
// (kCopies * 8). It arrives as a kernel argument so that the address is one
// integer multiply-add, which runs on the FMA pipe: with the constant in view
// the compiler forms it with a shift and an add on the ALU pipe, the busier one.
template <int TAB>
__device__ __forceinline__ uint2 entry_of(float w, uint32_t tab_base, uint32_t stride)
{
    const uint32_t bucket = __float_as_uint(__fadd_rn(fabsf(w), __uint_as_float(kBucketOffsetBits))) >> 19;
    return lds_u2(bucket * stride + tab_base + TAB * kTabBytes);
}

// Index of the stored byte in the entry: bits 31-30 of bits(w) + K, which are
// 2 * sign(w) + (|w| >= T*). `one` is 1, a kernel argument for the same reason
// as the stride: the add is then a multiply-add on the FMA pipe.
__device__ __forceinline__ uint32_t byte_index(float w, uint32_t k, uint32_t one)
{
    return (__float_as_uint(w) * one + k) >> 30;
}

// Stage 3 + the +7 bias for one value w (|w| < 2, never -0): a word whose low
// byte is the stored byte (c + 7) & 0xFF, anchor in the high nibble and
// residual in the low one (bits 8-31 are not defined).
__device__ __forceinline__ uint32_t code_byte(float w, uint32_t tab_base, uint32_t stride, uint32_t one)
{
    const uint2 e = entry_of<0>(w, tab_base, stride);
    return __byte_perm(e.y, 0u, byte_index(w, e.x, one));
}

// The same for the pair (w0, w1) of channels 2pi, 2pi + 1: byte 0 of the
// result is the stored byte of w0 (A0 << 4 | r0) and byte 1 that of w1 with
// its nibbles swapped (r1 << 4 | A1), read from the second table; the second
// permute merges the two (selector nibble 1 = 4 takes byte 0 of b1). Then the
// anchor byte A1 << 4 | A0 is the result shifted right by 4, and the residual
// byte r1 << 4 | r0 one logic operation away (bits 16-31 are not defined).
__device__ __forceinline__ uint32_t code_pair(float w0, float w1, uint32_t tab_base, uint32_t stride, uint32_t one)
{
    // both buckets' sums |w| + 2^-13 in one packed add (each lane one IEEE add)
    const float off = __uint_as_float(kBucketOffsetBits);
    const float2 sum = __fadd2_rn(make_float2(fabsf(w0), fabsf(w1)), make_float2(off, off));
    const uint2 e0 = lds_u2((__float_as_uint(sum.x) >> 19) * stride + tab_base);
    const uint2 e1 = lds_u2((__float_as_uint(sum.y) >> 19) * stride + tab_base + kTabBytes);
    const uint32_t b1 = __byte_perm(e1.y, 0u, byte_index(w1, e1.x, one));
    return __byte_perm(e0.y, b1, byte_index(w0, e0.x, one) + 0x40u);
}

// bf16x2 min / max that propagate NaN (a NaN value marks its channel)
__device__ __forceinline__ uint32_t bf2_min(uint32_t a, uint32_t b)
{
    __nv_bfloat162 r = __hmin2_nan(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b)
{
    __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// (x0 - m0, x1 - m1) for the bf16 pair x, each one fp32 operation rounded to
// nearest: x * 1 + (-m) with bf16 operands and an fp32 addend, whose product is
// exact, so the result is the rounded difference itself; the bf16 values need
// no separate widening.
__device__ __forceinline__ float2 sub_bf2(uint32_t x, float2 negm)
{
    float r0, r1;
    asm("{\n\t.reg .b16 l, h, one;\n\tmov.b32 {l, h}, %2;\n\tmov.b16 one, 0x3F80;\n\t"
        "fma.rn.f32.bf16 %0, l, one, %3;\n\tfma.rn.f32.bf16 %1, h, one, %4;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "r"(x), "f"(negm.x), "f"(negm.y));
    return make_float2(r0, r1);
}

// 1/s, correctly rounded, for the chunk scale s: an fp16 value (an 11-bit
// significand, 2^-24 <= s < 2). The hardware approximation r, then one Newton
// step written as two fused multiply-adds, r + r (1 - s r). With an 11-bit
// significand the exact 1/s = 2^k / M (M < 2^11) lies at least 2^-35
// (relative) from any midpoint between two fp32 values, while the step leaves
// an error near (1 - s r)^2 <= 2^-44, so the final rounding is the correct
// one (checked exhaustively for every positive fp16 value and every starting
// point within 2 ulp).
__device__ __forceinline__ float rcp_of_fp16(float s)
{
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
    return __fmaf_rn(r, __fmaf_rn(-s, r, 1.0f), r);
}

// Stages 2-4 for this thread's two channels of one chunk, held as float2
// lanes (x = channel 2pi, y = channel 2pi + 1) so that each packed fp32
// instruction performs the contract's operation for both channels (every lane
// of __fadd2_rn / __fmul2_rn is one IEEE round-to-nearest operation, and
// x - y is computed as x + (-y), which is the same operation). `full` chunks
// have 32 valid tokens, others nc; ulo / uhi are u at the chunk's smallest and
// largest valid x. Writes the staged plane bytes and returns the chunk
// metadata (mean, scale) of both channels as fp16x2 words.
template <bool FULL>
__device__ __forceinline__ void encode_chunk(const float2 (&u)[kChunk], int nc, float2 ulo, float2 uhi,
                                             uint32_t tab_base, uint32_t stride, uint32_t one, uint8_t *anc_row0,
                                             uint8_t *res_row0, uint32_t &mu2, uint32_t &s2)
{
    // chunk mean: stride-halving pairwise tree over 32 slots, absent slots +0
    const float2 zero = make_float2(0.0f, 0.0f);
    float2 t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        t[i] = __fadd2_rn((FULL || i < nc) ? u[i] : zero, (FULL || i + 16 < nc) ? u[i + 16] : zero);
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i)
            t[i] = __fadd2_rn(t[i], t[i + h]);
    float2 mean;
    if (FULL) {
        mean = __fmul2_rn(t[0], make_float2(0.03125f, 0.03125f));   // exact: division by 32
    } else {
        const float ncf = (float)nc;
        mean = make_float2(__fdiv_rn(t[0].x, ncf), __fdiv_rn(t[0].y, ncf));
    }
    const __half2 mh = __floats2half2_rn(mean.x, mean.y);   // one packed conversion
    const __half mh0 = __low2half(mh), mh1 = __high2half(mh);
    const float2 negmu = make_float2(-__half2float(mh0), -__half2float(mh1));

    // max |v| over the chunk: v = u - mu is non-decreasing in u, so it is
    // reached at the chunk's extremes
    const float2 vlo = __fadd2_rn(ulo, negmu), vhi = __fadd2_rn(uhi, negmu);
    const float s0 = fmaxf(fabsf(vlo.x), fabsf(vhi.x)), s1 = fmaxf(fabsf(vlo.y), fabsf(vhi.y));
    const __half sh0 = __float2half_ru(s0), sh1 = __float2half_ru(s1);
    const float sf0 = __half2float(sh0), sf1 = __half2float(sh1);
    const float2 inv_s = make_float2(sf0 > 0.0f ? rcp_of_fp16(sf0) : 0.0f, sf1 > 0.0f ? rcp_of_fp16(sf1) : 0.0f);

    // groups of kGroup tokens: all lookups of a group, then its stores (a
    // table load may not move above an earlier store to shared memory, so
    // interleaving them would serialise the tokens)
#pragma unroll
    for (int g0 = 0; g0 < kChunk; g0 += kGroup) {
        uint32_t ab[kGroup], rb[kGroup];
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            const int i = g0 + k;
            ab[k] = 0x00u;                               // code 0: anchor 0, residual 7
            rb[k] = 0x77u;
            if (FULL || i < nc) {
                // w = v * inv_s, as one rounding of the product plus +0, which
                // turns a -0 product into +0 (both code 0) and changes nothing else
                const float2 w = __ffma2_rn(__fadd2_rn(u[i], negmu), inv_s, zero);
                const uint32_t z = code_pair(w.x, w.y, tab_base, stride, one);
                // low bytes: the anchors and the residuals of the pair (bits
                // 8-31 are not stored)
                ab[k] = z >> 4;
                rb[k] = (z & 0x0Fu) | ((z >> 8) & ~0x0Fu);
            }
        }
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            anc_row0[(g0 + k) * kRowB] = (uint8_t)ab[k];
            res_row0[(g0 + k) * kRowB] = (uint8_t)rb[k];
        }
    }
    mu2 = (uint32_t)__half_as_ushort(mh0) | ((uint32_t)__half_as_ushort(mh1) << 16);
    s2 = (uint32_t)__half_as_ushort(sh0) | ((uint32_t)__half_as_ushort(sh1) << 16);
}

// One 2D tiled tensor copy global -> shared, completing on an mbarrier
// (coordinates: innermost first, in elements).
__device__ __forceinline__ void tile_g2s(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3}], [%4];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
                 : "memory");
}

// Prefetch one 2D tile into L2.
__device__ __forceinline__ void tile_prefetch_l2(const CUtensorMap *map, int c0, int c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// One 2D tiled tensor copy shared -> global, tracked by the issuing thread's
// bulk groups.
__device__ __forceinline__ void tile_s2g(const CUtensorMap *map, int c0, int c1, const void *src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

// Work unit u = (page u / 2, channel half u % 2). A CTA of 8 warps takes
// units blockIdx.x, blockIdx.x + gridDim.x, ...; two CTAs share an SM and run
// out of step, so that one's barrier and latency-bound stretches (the chunk
// extremes, the page statistics) overlap the other's stage 3. The input
// buffer is refilled with the next unit as soon as every value of the current
// one is in registers (after the first barrier).
// tab_stride: kCopies * 8, and one: 1, passed at run time (see code_byte)
__global__ void __launch_bounds__(kThreads, 2) quantize_kernel(Params p, const __grid_constant__ CUtensorMap xmap,
                                                               const __grid_constant__ CUtensorMap amap,
                                                               const __grid_constant__ CUtensorMap rmap,
                                                               CodeTable table, uint32_t tab_stride, uint32_t one)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int j = warp;                            // chunk of this warp; lane: channel pair of the half

    for (int i = tid; i < kNBucket * kCopies; i += kThreads) {
        const uint2 e = table.e[i / kCopies];
        sm.tab[0][i] = e;
        sm.tab[1][i] = make_uint2(e.x, ((e.y >> 4) & 0x0F0F0F0Fu) | ((e.y << 4) & 0xF0F0F0F0u));
    }
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t tab_base = smem_u32(&sm.tab[0][lane & (kCopies - 1)]) - kBucketBase * (kCopies * 8);

    const int64_t units = 2 * p.pages;
    const int64_t first = blockIdx.x, stride = gridDim.x;
    if (tid == 0 && first < units) {
        mbar_arrive_expect_tx(&sm.bar, kUnitBytes);
        tile_g2s(sm.x, &xmap, (int)(first & 1) * kHalf, (int)(first >> 1) * kPage, &sm.bar);
    }

    int k = 0;
    for (int64_t unit = first; unit < units; unit += stride, ++k) {
        const int64_t page = unit >> 1, next = unit + stride;
        const int half = (int)(unit & 1);
        const int pi = half * (kHalf / 2) + lane;  // channel pair of the page: channels 2pi, 2pi+1
        // the next unit's tile heads for L2 now; its copy into shared memory
        // follows after this unit's first barrier (0.4 % faster)
        if (warp == 0 && lane == 0 && next < units)
            tile_prefetch_l2(&xmap, (int)(next & 1) * kHalf, (int)(next >> 1) * kPage);
        const bool ok = mbar_wait_bounded(&sm.bar, (uint32_t)k & 1u, kWaitLimit);

        const int n = valid_of(p, page);
        const int64_t dst = dst_of(p, page);
        if (dst < 0 && p.dev_err && tid == 0)
            atomicOr(p.dev_err, LYNX_DEVERR_PAGE);
        const int nc = min(max(n - j * kChunk, 0), kChunk);

        // (a) this thread's 32 tokens x 2 channels, and their chunk min/max
        const uint16_t *xs = sm.x + j * kChunk * kHalf + 2 * lane;
        uint32_t xw[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            xw[i] = *reinterpret_cast<const uint32_t *>(xs + i * kHalf);
        uint32_t cmn2 = 0x7F807F80u, cmx2 = 0xFF80FF80u;   // +inf, -inf pairs
        if (nc == kChunk) {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                cmn2 = bf2_min(cmn2, xw[i]);
                cmx2 = bf2_max(cmx2, xw[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kChunk; ++i)
                if (i < nc) {
                    cmn2 = bf2_min(cmn2, xw[i]);
                    cmx2 = bf2_max(cmx2, xw[i]);
                }
        }
        sm.pmm[j][lane] = make_uint2(cmn2, cmx2);
        if (warp == 0 && lane == 0)
            bulk_wait_read_all();   // the previous unit's planes have left the staging tile
        // (a thread whose wait gave up read a unit that never landed; nothing
        // of it is used)
        if (__syncthreads_or(!ok)) {
            // the copy never landed: report it (appending), and stop after
            // waiting once more for it
            if (tid == 0) {
                if (p.dev_err)
                    atomicOr(p.dev_err, LYNX_DEVERR_TIMEOUT);
                mbar_wait_bounded(&sm.bar, (uint32_t)k & 1u, kWaitLimit);
            }
            break;
        }
        // every value of the unit is in registers: refill the buffer with the
        // next unit (the reads reach thread 0 through the barrier; its proxy
        // fence orders them before the copy's writes)
        if (warp == 0 && lane == 0 && next < units) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sm.bar, kUnitBytes);
            tile_g2s(sm.x, &xmap, (int)(next & 1) * kHalf, (int)(next >> 1) * kPage, &sm.bar);
        }

        // (b) stage 1 over the unit's page
        uint32_t mn2 = sm.pmm[0][lane].x, mx2 = sm.pmm[0][lane].y;
#pragma unroll
        for (int jj = 1; jj < kNChunk; ++jj) {
            const uint2 e = sm.pmm[jj][lane];
            mn2 = bf2_min(mn2, e.x);
            mx2 = bf2_max(mx2, e.y);
        }
        float mn0 = bf16_lo(mn2), mn1 = bf16_hi(mn2), mx0 = bf16_lo(mx2), mx1 = bf16_hi(mx2);
        if (n == 0)
            mn0 = mn1 = mx0 = mx1 = 0.0f;
        // a zero extreme is +0 (each lane of the packed operations is one
        // IEEE operation, and x - y is x + (-y))
        const float2 mnz = __fadd2_rn(make_float2(mn0, mn1), make_float2(0.0f, 0.0f));
        const float2 mxz = __fadd2_rn(make_float2(mx0, mx1), make_float2(0.0f, 0.0f));
        mn0 = mnz.x;
        mn1 = mnz.y;
        const float2 rg2 = __fadd2_rn(mxz, make_float2(-mnz.x, -mnz.y));
        float rg0 = rg2.x, rg1 = rg2.y;
        // a NaN value (min and max NaN) stores min and range as the quiet NaN;
        // so does any NaN range
        if (mn0 != mn0)
            mn0 = __uint_as_float(kQNaN);
        if (mn1 != mn1)
            mn1 = __uint_as_float(kQNaN);
        if (rg0 != rg0)
            rg0 = __uint_as_float(kQNaN);
        if (rg1 != rg1)
            rg1 = __uint_as_float(kQNaN);
        float ir0 = rg0 > 0.0f ? __frcp_rn(rg0) : 0.0f;
        float ir1 = rg1 > 0.0f ? __frcp_rn(rg1) : 0.0f;
        // statistics fp32 cannot carry (range or reciprocal not finite): the
        // channel is coded as constant, every u = 0 (x and min taken as 0)
        const bool bad0 = !(rg0 <= kF32Max) || !(ir0 <= kF32Max);
        const bool bad1 = !(rg1 <= kF32Max) || !(ir1 <= kF32Max);
        float2 negmn = make_float2(-mn0, -mn1);
        if (bad0 | bad1) {
            const uint32_t keep = (bad0 ? 0xFFFF0000u : 0xFFFFFFFFu) & (bad1 ? 0x0000FFFFu : 0xFFFFFFFFu);
#pragma unroll
            for (int i = 0; i < kChunk; ++i)
                xw[i] &= keep;
            cmn2 &= keep;
            cmx2 &= keep;
            if (bad0)
                negmn.x = ir0 = 0.0f;
            if (bad1)
                negmn.y = ir1 = 0.0f;
        }

        float2 u[kChunk], ulo, uhi;
        {
            const float2 ir = make_float2(ir0, ir1);
#pragma unroll
            for (int i = 0; i < kChunk; ++i)
                u[i] = __fmul2_rn(sub_bf2(xw[i], negmn), ir);
            ulo = __fmul2_rn(sub_bf2(cmn2, negmn), ir);
            uhi = __fmul2_rn(sub_bf2(cmx2, negmn), ir);
        }

        // (c) stages 2-4
        uint8_t *anc_row0 = sm.anc + j * kChunk * kRowB + lane;
        uint8_t *res_row0 = sm.res + j * kChunk * kRowB + lane;
        uint32_t mu2 = 0, s2 = 0;
        if (nc == kChunk) {
            encode_chunk<true>(u, nc, ulo, uhi, tab_base, tab_stride, one, anc_row0, res_row0, mu2, s2);
        } else if (nc > 0) {
            encode_chunk<false>(u, nc, ulo, uhi, tab_base, tab_stride, one, anc_row0, res_row0, mu2, s2);
        } else {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                anc_row0[i * kRowB] = 0x00u;
                res_row0[i * kRowB] = 0x77u;
            }
        }

        // metadata: page (min, range) from chunk 0's warp; chunk (mean, scale) from every thread
        if (j == 0 && dst >= 0) {
            float *pm = p.pm + dst * (int64_t)(2 * kD) + 2 * pi;
            *reinterpret_cast<float2 *>(pm) = make_float2(mn0, mn1);
            *reinterpret_cast<float2 *>(pm + kD) = make_float2(rg0, rg1);
        }
        if (dst >= 0) {
            uint16_t *cm = p.cm + (dst * kNChunk + j) * (int64_t)(2 * kD) + 2 * pi;
            *reinterpret_cast<uint32_t *>(cm) = mu2;
            *reinterpret_cast<uint32_t *>(cm + kD) = s2;
        }
        // every thread's plane bytes reach thread 0 through the barrier, and
        // its proxy fence then orders them before the tensor copies' reads
        // (the fence lies on the causality path from each write to the copy)
        __syncthreads();
        if (warp == 0 && lane == 0 && dst >= 0) {
            fence_proxy_async_smem();
            tile_s2g(&amap, half * kRowB, (int)dst * kPage, sm.anc);
            tile_s2g(&rmap, half * kRowB, (int)dst * kPage, sm.res);
            bulk_commit();
        }
    }
    if (tid == 0)
        bulk_wait_all();
}

// The encoder's stage-3 path on arbitrary values (a diagnostic): the same
// table and code_byte(), with |w| clamped to 1.5 (every |w| >= T_63 < 1 has
// the same code), -0 turned into +0 and NaN into 0 first, so that any input
// stays inside the table (the encoder itself sees only finite w with
// |w| <= 1 + 2^-23, never -0).
__global__ void level_codes_kernel(const float *__restrict__ w, int64_t n, int8_t *__restrict__ codes,
                                   CodeTable table)
{
    __shared__ uint2 tab[kNBucket * kCopies];
    for (int i = threadIdx.x; i < kNBucket * kCopies; i += blockDim.x)
        tab[i] = table.e[i / kCopies];
    __syncthreads();
    const uint32_t tab_base = smem_u32(&tab[threadIdx.x & (kCopies - 1)]) - kBucketBase * (kCopies * 8);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = w[i];
        const float c = v == v ? __fadd_rn(copysignf(fminf(fabsf(v), 1.5f), v), 0.0f) : 0.0f;
        codes[i] = (int8_t)((int)(int8_t)code_byte(c, tab_base, kCopies * 8, 1u) - kBias);
    }
}

// cuTensorMapEncodeTiled, through the runtime's driver entry point (no link
// against the driver library); NULL when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A 2D row-major map of `rows` rows of `width` elements, copied in boxes of
// box_w x 256 rows (no swizzle, no interleave).
bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap *m, CUtensorMapDataType dt, const void *base,
                 uint64_t width, uint64_t row_bytes, uint64_t rows, uint32_t box_w)
{
    const cuuint64_t dims[2] = {width, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_w, (cuuint32_t)kPage};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs per SM the encoder runs at (2 when shared memory and registers allow).
int quantize_ctas_per_sm(size_t smem)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_kernel, kThreads, smem) != cudaSuccess)
        return 0;
    return n;
}

// dst_pages: pages of the destination planes (one after another)
cudaError_t run_quantize(const Params &p, int64_t dst_pages, cudaStream_t s)
{
    if (p.pages == 0)
        return cudaSuccess;
    // tile coordinates are 32-bit row numbers
    if (p.pages > INT32_MAX / kPage || dst_pages > INT32_MAX / kPage)
        return cudaErrorNotSupported;
    const int sms = device_sm_count();
    if (sms <= 0)
        return cudaErrorNoDevice;
    const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn)
        return cudaErrorNotSupported;
    // an empty pool (appending into 0 pages: every tail is outside it, skipped
    // and flagged) still needs well-formed plane maps; no store ever uses them
    const uint64_t plane_rows = (uint64_t)(dst_pages > 0 ? dst_pages : 1) * kPage;
    CUtensorMap xmap, amap, rmap;
    if (!encode_rows(fn, &xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.x, kD, kD * 2, (uint64_t)p.pages * kPage, kHalf) ||
        !encode_rows(fn, &amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.anc, kD / 2, kD / 2, plane_rows, kRowB) ||
        !encode_rows(fn, &rmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.res, kD / 2, kD / 2, plane_rows, kRowB))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess)
        return e;
    const int per_sm = quantize_ctas_per_sm(smem);
    if (per_sm <= 0)
        return cudaErrorNotSupported;
    const int64_t units = 2 * p.pages, cap = (int64_t)sms * per_sm;
    const int64_t grid = units < cap ? units : cap;
    quantize_kernel<<<(unsigned)grid, kThreads, smem, s>>>(p, xmap, amap, rmap, host_tables().code,
                                                           (uint32_t)kCopies * 8u, 1u);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_quantize(const uint16_t *x, const int32_t *page_valid, const lynx_qkv &o, cudaStream_t s)
{
    const int P = o.tokens / kPage;
    const int64_t pages = (int64_t)o.layers * o.kv_heads * P;
    Params p{x, page_valid, o.anchor, o.residual, o.page_meta, o.chunk_meta, pages, P, nullptr, nullptr, 1, nullptr};
    return run_quantize(p, pages, s);
}

cudaError_t launch_quantize_append(const uint16_t *tail, const int32_t *dst_page, const int32_t *valid, int n,
                                   const lynx_qkv &o, uint32_t *dev_err, cudaStream_t s)
{
    const int LH = o.layers * o.kv_heads;
    Params p{tail, nullptr, o.anchor, o.residual, o.page_meta, o.chunk_meta,
             (int64_t)n * LH, o.tokens / kPage, dst_page, valid, LH > 0 ? LH : 1, dev_err};
    return run_quantize(p, (int64_t)LH * (o.tokens / kPage), s);
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
    level_codes_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, n, codes, host_tables().code);
    return cudaGetLastError();
}

} // namespace lynx
