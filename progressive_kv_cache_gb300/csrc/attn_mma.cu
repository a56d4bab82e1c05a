// attn_mma.cu -- fused-dequant paged decode attention on the tensor cores
// (K4, groups of up to 16 query heads per KV head).
//
// One decode step over the quantized paged cache ("KV-cache quantization"
// explainer, "Bottom-right": the compact cache is read as is and expanded
// only on chip, inside Q.K^T and P.V). Anchor mode reads the anchor planes only
// (the draft cache of the Lynx reading, section 4); full mode adds the residual
// planes.
//
// Factorisation. Every element of chunk j (32 tokens) and channel d decodes
// as x = a_jd + b_jd * L(code) with a = mn + rng mu, b = rng s and L an exact
// fp16 level value. Hence, per chunk,
//   s_t  = beta_j + sum_d (q_d b_jd) L_td,         beta_j = sum_d q_d a_jd
//   o_d += sum_j [ a_jd sum_{t in j} p_t + b_jd sum_{t in j} p_t L_td ],
// so the tensor-core operands on the cache side are the level values
// themselves (no rounding), and the dense operand (q b, or p) is split into an
// fp16 hi/lo pair to keep fp32-level accuracy (mma.sync m16n8k16, fp32
// accumulation).
//
// Register-direct operands. A code byte holds two channels of one token, and
// the MMA's B fragment wants two adjacent k-indices of one column in one
// register. Q.K^T contracts over channels, so the channel order inside the
// contraction is free: lane (g, q) of the warp reads 16 code bytes of token g
// of an 8-token tile (channels 32q .. 32q + 31) and every byte, through one
// table lookup, is a finished B register; the A fragments (q b) follow the
// same channel order. P.V contracts over tokens: the nibbles of one channel of
// two tokens are merged into one byte (two logic operations per four bytes),
// whose lookup is again a finished B register. No decoded value touches shared
// memory. The lookup table is replicated per lane (conflict-free) with entries
// 256 bytes apart, so that one byte permute forms the whole address.
//
// Work: a CTA per (page range, KV head, request) of 16 warps. The pages' K
// and V planes and metadata arrive by bulk copy in a ring of slots (one
// tensor's page per slot); the warp that releases the last chunk of a slot
// refills it. Warp w takes chunks w, w + 16, ... of the range, each for all
// query heads of the group: with up to 8 heads the MMA rows are the heads' hi
// parts over their lo parts; with up to 16 the rows are the heads and hi and
// lo go through two MMAs into the same accumulators. The chunks' running (max,
// sum, output) are merged in shared memory into one partial per query head; a
// second kernel merges the partials of the ranges.
//
// Tensor memory as a register file extension. A warp's running output (16
// heads x 128 channels, 64 fp32 values a lane) lives in tensor memory between
// chunks and comes into registers half at a time for the P.V update. This
// keeps the warp under 128 registers, so 16 warps (four per scheduler) fit.
#include <cuda_fp16.h>

#include <mutex>

#include "lynx_internal.cuh"
#include "lynx_ptx.cuh"

namespace lynx {
namespace {

constexpr uint32_t kPlane = kPage * kD / 2;   // 16 KiB: one page of one plane
constexpr int kRow = kD / 2;                  // code bytes per token
constexpr int kPart = kD + 2;
constexpr int kWarps = 16;                    // four per scheduler
constexpr uint32_t kTmemCols = 256;           // per warp 64 columns of its lane quarter: the running output
constexpr int kThreads = kWarps * 32;
constexpr int kAff = kD + 16;                 // channel c stored at c + 4 (c / 32): no bank conflicts
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// The system reserves shared memory ahead of a kernel's dynamic window (1 KiB
// on this part family). With that base the level table below starts at shared
// address 0x10000, and the shared address of a table word is one byte permute
// of the code byte and a per-lane constant. The base is measured once per
// device (table_aligned()); a device whose window starts elsewhere is refused
// (the call returns LYNX_ERR_UNSUPPORTED), and the kernel checks it again.
constexpr uint32_t kDynBase = 1024;
constexpr uint32_t kPre = 0x10000 - kDynBase;

// One tensor's page metadata as it arrives.
struct SlotMeta {
    float pm[2 * kD];
    uint16_t cm[kNChunk * 2 * kD];
};

template <int NS>
struct Head {
    // the group's queries times sm_scale log2(e), as this lane's A-fragment
    // channels: qf[s][r][lane] = q[row g + 8 r][32 q + 4 s .. + 3]
    float4 qf[8][2][32];
    float aff[kWarps][2][kAff];               // per warp: chunk affines a, b (K, then V)
    SlotMeta meta[NS];
    float qmax;
    int rel[NS];                              // releases of the slot's current item
    int last[NS];                             // last item issued into each slot (its tag)
    uint32_t tmem;                            // tensor-memory base of the running outputs
    alignas(16) uint16_t qstage[16 * kD];     // the group's query rows as they arrive (bf16)
    alignas(8) uint64_t q_bar;
    alignas(8) uint64_t full_bar[NS];
};

template <bool FULL, int NS>
struct Smem {
    Head<NS> h;
    unsigned char pad[kPre - sizeof(Head<NS>)];
    // level table: entry e (a code byte) at byte 256 e; anchor mode: word
    // `lane` = half2 of the levels of the two anchor nibbles of e; full mode:
    // word 32 + `lane` = fp16 level of the code byte e (A << 4 | r) in its low half
    uint32_t lut[256 * 64];
    uint8_t plane[NS][FULL ? 2 : 1][kPlane];  // per slot: anchor (and residual) codes
};

constexpr int kMrow = 4 * 34;                 // a merge row: four 32-channel blocks, each padded by 2
struct Merge {                                // overlays the table and the planes after the page loop
    float m[kWarps][16];                      // per warp and query head
    float l[kWarps][16];
    float o4[4][16][kMrow];                   // per lane quarter: its four warps' weighted sum; channel d at 34 (d / 32) + d % 32
    float sc[16][kWarps];                     // per query head: each warp's weight 2^(m_w - M)
    float M[16], L[16];                       // per query head: the range's max and sum
};

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with a zero accumulator in.
__device__ __forceinline__ void mma16816_z(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%10,%10,%10,%10};"
                 : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// (x0, x1) -> fp16 pairs hi and lo with hi + lo = (x0, x1) to ~22 bits. The
// remainders x - hi are exact in fp32; each comes from one mixed-precision
// multiply-add (fp16 operands, fp32 addend and result), with no separate
// widening of hi.
__device__ __forceinline__ void split2(float2 x, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(x.x, x.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    float r0, r1;
    asm("{\n\t.reg .b16 h0, h1, m1;\n\tmov.b32 {h0, h1}, %2;\n\tmov.b16 m1, 0xBC00;\n\t"
        "fma.rn.f32.f16 %0, h0, m1, %3;\n\tfma.rn.f32.f16 %1, h1, m1, %4;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "r"(hi), "f"(x.x), "f"(x.y));
    const __half2 l = __floats2half2_rn(r0, r1);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7F800000); }

// 2^x for the softmax weights (x <= 0): the hardware approximation, results
// below 2^-126 flushed to zero.
__device__ __forceinline__ float exp2_sm(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Table word of code byte I of w: lanebase = the table's shared address |
// this lane's column, and one permute puts the code byte in bits 8-15.
template <int I>
__device__ __forceinline__ uint32_t lut_ld(uint32_t w, uint32_t lanebase)
{
    const uint32_t addr = __byte_perm(w, lanebase, 0x7604u | (I << 4));
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// Low halves of x and y as one half2 (x's in the low half).
__device__ __forceinline__ uint32_t pack_lo(uint32_t x, uint32_t y) { return __byte_perm(x, y, 0x5410u); }

// Full-mode code bytes (A << 4 | r) of the even / odd channels of a word of
// anchor nibbles aw and residual nibbles rw.
__device__ __forceinline__ uint32_t codes_even(uint32_t aw, uint32_t rw)
{
    return ((aw << 4) & 0xF0F0F0F0u) | (rw & 0x0F0F0F0Fu);
}
__device__ __forceinline__ uint32_t codes_odd(uint32_t aw, uint32_t rw)
{
    return (aw & 0xF0F0F0F0u) | ((rw >> 4) & 0x0F0F0F0Fu);
}

// Byte i of the result holds nibble 2i of x (low) and nibble 2i of y (high),
// resp. nibble 2i + 1: one channel of two tokens.
__device__ __forceinline__ uint32_t nib_even(uint32_t x, uint32_t y)
{
    return (x & 0x0F0F0F0Fu) | ((y << 4) & 0xF0F0F0F0u);
}
__device__ __forceinline__ uint32_t nib_odd(uint32_t x, uint32_t y)
{
    return ((x >> 4) & 0x0F0F0F0Fu) | (y & 0xF0F0F0F0u);
}

// Chunk affines a = mn + rng mu and b = rng s of channels 4l .. 4l + 3 of one
// tensor's page into the warp's buffers; returns max |b| of those channels.
__device__ __forceinline__ float chunk_affines(const float *pm, const uint16_t *cm, int j, int lane, float *fa,
                                               float *fb)
{
    const int d = 4 * lane;
    const float4 mn = *reinterpret_cast<const float4 *>(pm + d);
    const float4 rg = *reinterpret_cast<const float4 *>(pm + kD + d);
    const uint2 mu2 = *reinterpret_cast<const uint2 *>(cm + (2 * j) * kD + d);
    const uint2 sc2 = *reinterpret_cast<const uint2 *>(cm + (2 * j + 1) * kD + d);
    const float2 mu01 = __half22float2(*reinterpret_cast<const __half2 *>(&mu2.x));
    const float2 mu23 = __half22float2(*reinterpret_cast<const __half2 *>(&mu2.y));
    const float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(&sc2.x));
    const float2 s23 = __half22float2(*reinterpret_cast<const __half2 *>(&sc2.y));
    const float2 a01 = __ffma2_rn(make_float2(rg.x, rg.y), mu01, make_float2(mn.x, mn.y));
    const float2 a23 = __ffma2_rn(make_float2(rg.z, rg.w), mu23, make_float2(mn.z, mn.w));
    const float2 b01 = __fmul2_rn(make_float2(rg.x, rg.y), s01);
    const float2 b23 = __fmul2_rn(make_float2(rg.z, rg.w), s23);
    const int p = d + 4 * (d >> 5);
    *reinterpret_cast<float4 *>(fa + p) = make_float4(a01.x, a01.y, a23.x, a23.y);
    *reinterpret_cast<float4 *>(fb + p) = make_float4(b01.x, b01.y, b23.x, b23.y);
    return fmaxf(fmaxf(fabsf(b01.x), fabsf(b01.y)), fmaxf(fabsf(b23.x), fabsf(b23.y)));
}


__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <bool G16, bool FULL, int NS>
__global__ void __launch_bounds__(kThreads, 1) attn_mma_kernel(AttnArgs a, LevelTable lev)
{
    constexpr int R = G16 ? 2 : 1;          // query-head rows per lane: g (and g + 8)
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<FULL, NS> &sm = *reinterpret_cast<Smem<FULL, NS> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int G = a.G;
    const int64_t T = (int64_t)a.pool_pages * kPage;

    if (smem_u32(smem_raw) != kDynBase) {    // the table layout needs this window base (checked on the host too)
        if (a.dev_err && tid == 0)
            atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
        return;
    }

    int ctx = a.ctx[b];
    if (ctx < 0 || ctx > a.max_pages * kPage) {
        if (a.dev_err && split == 0 && kvh == 0 && tid == 0)
            atomicOr(a.dev_err, LYNX_DEVERR_CTX);
        ctx = min(max(ctx, 0), a.max_pages * kPage);
    }
    const int64_t score_stride = (int64_t)a.max_pages * kPage;
    const int p_begin = split * a.pages_per_split;
    const int p_end = min(p_begin + a.pages_per_split, a.max_pages);
    const int p_live = min(p_end, (ctx + kPage - 1) / kPage);   // pages holding context
    const int np = max(p_live - p_begin, 0);

    // physical page of the i-th live page of this range, or -1 (flagged)
    auto phys_of = [&](int i) -> int {
        const int p = a.page_table[(int64_t)b * a.max_pages + p_begin + i];
        return (p >= 0 && p < a.pool_pages) ? p : -1;
    };

    // ---- the ring: page i's K is item 2i, its V item 2i + 1; item x goes
    // to slot x % NS. Each of the 8 chunks of an item releases it once its
    // codes and metadata are in registers; the warp giving the 8th release
    // refills the slot with item x + NS at once.
    auto issue = [&](int x) {
        const int s = x % NS;
        const int t = x & 1;
        const int p = phys_of(x >> 1);
        SlotMeta &mt = sm.h.meta[s];
        uint64_t *bar = &sm.h.full_bar[s];
        *reinterpret_cast<volatile int *>(&sm.h.last[s]) = x;
        if (p < 0) {
            mbar_arrive(bar);   // completes the phase with no data: consumers skip the page
            return;
        }
        const int64_t off = (int64_t)kvh * T * kRow + (int64_t)p * kPlane;
        const int64_t pmo = ((int64_t)kvh * a.pool_pages + p) * (2 * kD);
        const int64_t cmo = ((int64_t)kvh * a.pool_pages + p) * (kNChunk * 2 * kD);
        mbar_arrive_expect_tx(bar, (FULL ? 2u : 1u) * kPlane + 2 * kD * 4 + kNChunk * 2 * kD * 2);
        bulk_g2s(sm.plane[s][0], (t ? a.va : a.ka) + off, kPlane, bar);
        if (FULL)
            bulk_g2s(sm.plane[s][FULL ? 1 : 0], (t ? a.vr : a.kr) + off, kPlane, bar);
        bulk_g2s(mt.pm, (t ? a.vpm : a.kpm) + pmo, 2 * kD * 4, bar);
        bulk_g2s(mt.cm, (t ? a.vcm : a.kcm) + cmo, kNChunk * 2 * kD * 2, bar);
    };

    // ---- per-CTA set-up ------------------------------------------------
    const int64_t qrow0 = (int64_t)b * a.Hq + (int64_t)kvh * G;
    if (tid == 0) {
        // the group's G query rows are contiguous: one copy, landing while the
        // tables are set up
        mbar_init(&sm.h.q_bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&sm.h.q_bar, (uint32_t)G * kD * 2);
        bulk_g2s(sm.h.qstage, a.q + qrow0 * kD, (uint32_t)G * kD * 2, &sm.h.q_bar);
        sm.h.qmax = 0.0f;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sm.h.full_bar[s], 1);
            sm.h.rel[s] = 0;
            sm.h.last[s] = -1;
        }
        fence_mbar_init();
        for (int x = 0; x < NS && x < 2 * np; ++x)   // the first pages arrive while the tables are set up
            issue(x);
    }
    for (int i = tid; i < 256 * 32; i += kThreads) {
        const int e = i >> 5, l = i & 31;
        uint32_t v;
        if (FULL) {
            v = (uint32_t)__half_as_ushort(__float2half_rn(lev.full[e]));
        } else {
            const __half2 h = __floats2half2_rn(lev.anchor[e & 15], lev.anchor[e >> 4]);
            v = *reinterpret_cast<const uint32_t *>(&h);
        }
        sm.lut[e * 64 + (FULL ? 32 : 0) + l] = v;
    }
    const float qscale = a.sm_scale * kLog2e;
    float lq = 0.0f;
    __syncthreads();                         // the query barrier is initialised
    const bool q_ok = mbar_wait_bounded(&sm.h.q_bar, 0u, kWaitLimit);
    if (!q_ok && a.dev_err)
        atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
    for (int i = tid; i < 8 * 2 * 32 * 4; i += kThreads) {
        // element c of qf[s][r][l]
        const int c = i & 3, l = (i >> 2) & 31, r = (i >> 7) & 1, s = i >> 8;
        const int row = (l >> 2) + 8 * r;
        const int d = 32 * (l & 3) + 4 * s + c;
        float v = 0.0f;
        if (row < G && (G16 || r == 0))
            v = __uint_as_float((uint32_t)sm.h.qstage[row * kD + d] << 16) * qscale;
        reinterpret_cast<float *>(&sm.h.qf[s][r][l])[c] = v;
        lq = fmaxf(lq, fabsf(v));
    }
    if (warp == 0)
        tmem_alloc(&sm.h.tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    atomicMax(reinterpret_cast<int *>(&sm.h.qmax), __float_as_int(lq));   // non-negative floats order as ints
    // this warp's running outputs: lane quarter warp % 4, columns 64 (warp / 4) ..
    // + 63; column 16 r + 4 mm + 2 side + e of half hf (32 hf + ..) holds row g + 8 r,
    // channel 32 q + 16 side + 2 (4 hf + mm) + e
    const uint32_t tO = sm.h.tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64u * (uint32_t)(warp >> 2);

    // pages of the range past the context: scores -inf
    if (a.scores) {
        for (int lp = max(p_live, p_begin); lp < p_end; ++lp)
            for (int i = tid; i < G * kPage; i += kThreads)
                a.scores[(qrow0 + i / kPage) * score_stride + (int64_t)lp * kPage + i % kPage] = neg_inf();
    }
    __syncthreads();   // qmax complete

    float m_run[R], l_run[R];                // per row: running max (base 2) and this lane's sum
#pragma unroll
    for (int r = 0; r < R; ++r) {
        m_run[r] = neg_inf();
        l_run[r] = 0.0f;
    }
    {
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            z[i] = 0.0f;
        tmem_st32f(tO, z);
        tmem_st32f(tO + 32, z);
    }

    // lane 0, after the warp's last read of item x's slot
    auto release = [&](int x) {
        const int s = x % NS;
        __threadfence_block();
        if (atomicAdd(&sm.h.rel[s], 1) == kNChunk - 1) {
            sm.h.rel[s] = 0;
            __threadfence_block();
            if (x + NS < 2 * np) {
                fence_proxy_async_smem();
                issue(x + NS);
            }
        }
    };
    // A warp skips the pages other warps take, so a slot's barrier may still
    // be in the phase of an item this warp never saw, whose parity equals
    // that of the one it waits for; the slot's tag (the item last issued into
    // it) tells the two apart: once it reads x, the phase of x is current or
    // complete.
    auto wait_item = [&](int x) -> bool {
        const int s = x % NS;
        const volatile int *tag = &sm.h.last[s];
        uint32_t it = 0;
        while (*tag != x) {
            if (++it == kWaitLimit)
                return false;
            __nanosleep(32);
        }
        return mbar_wait_bounded(&sm.h.full_bar[s], (uint32_t)((x / NS) & 1), kWaitLimit);
    };

    // ---- warp w: chunks w, w + kWarps, ... of the range (chunk c = chunk
    // c % 8 of page c / 8) ------------------------------------------------
    const uint32_t lane4 = (uint32_t)lane << 2;
    const uint32_t lut_s = smem_u32(sm.lut);
    const uint32_t lb = (FULL ? 128u : 0u) + lane4 + lut_s;   // this lane's table column
    float *kaf = sm.h.aff[warp][0], *kbf = sm.h.aff[warp][1];             // K's, then V's
    float *vaf = kaf, *vbf = kbf;
    const float qmax = sm.h.qmax;
    bool timed_out = false;
    for (int c = warp; c < kNChunk * np; c += kWarps) {
        const int i = c >> 3, j = c & 7;
        const int xk = 2 * i, sK = xk % NS, sV = (xk + 1) % NS;
        const int lp = p_begin + i;
        const bool valid = phys_of(i) >= 0;
        const int nv = min(max(ctx - lp * kPage - j * kChunk, 0), kChunk);   // valid tokens of chunk j
        if (__any_sync(0xFFFFFFFFu, !wait_item(xk))) {   // warp-uniform: the whole warp leaves together
            timed_out = true;
            break;
        }
        if (!valid || nv == 0) {
            if (!valid && a.dev_err && j == 0 && lane == 0)
                atomicOr(a.dev_err, LYNX_DEVERR_PAGE);
            if (a.scores)
                for (int e = lane; e < G * kChunk; e += 32)
                    a.scores[(qrow0 + e / kChunk) * score_stride + (int64_t)lp * kPage + j * kChunk + e % kChunk] =
                        neg_inf();
            __syncwarp();
            if (lane == 0)
                release(xk);
            if (__any_sync(0xFFFFFFFFu, !wait_item(xk + 1))) {
                timed_out = true;
                break;
            }
            __syncwarp();
            if (lane == 0)
                release(xk + 1);
            continue;
        }

        // ---- K: affines and codes of chunk j, then release the slot -------
        float gscale, gdown;
        int ge = 0;
        uint4 kc[4], kr4[4];
        {
            const SlotMeta &mt = sm.h.meta[sK];
            float bm = chunk_affines(mt.pm, mt.cm, j, lane, kaf, kbf);
            const uint8_t *ca = sm.plane[sK][0] + (j * kChunk + g) * kRow + 16 * q;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                kc[nt] = *reinterpret_cast<const uint4 *>(ca + nt * 8 * kRow);
            if (FULL) {
                const uint8_t *cr = sm.plane[sK][FULL ? 1 : 0] + (j * kChunk + g) * kRow + 16 * q;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    kr4[nt] = *reinterpret_cast<const uint4 *>(cr + nt * 8 * kRow);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, o));
            // q b must stay a finite fp16 pair: past 2^14 it is scaled by
            // 2^-e and the scores back by 2^e
            if (bm * qmax >= 16384.0f) {
                frexpf(bm * qmax, &ge);
                ge -= 14;
            }
            gdown = exp2f((float)-ge);
            gscale = exp2f((float)ge);
            if (ge != 0) {                   // rare: fold 2^-e into this lane's b values
                float4 *bv = reinterpret_cast<float4 *>(kbf + 4 * lane + 4 * (lane >> 3));
                const float4 v = *bv;
                *bv = make_float4(v.x * gdown, v.y * gdown, v.z * gdown, v.w * gdown);
            }
            __syncwarp();
            if (lane == 0)
                release(xk);
        }

        // ---- Q.K^T ------------------------------------------------------------
        float S[4][4];
        float2 beta2[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            beta2[r] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int cp = 36 * q + 4 * s;   // channels 32q + 4s .. + 3 (padded index)
            const float4 bb = *reinterpret_cast<const float4 *>(kbf + cp);
            const float4 aa = *reinterpret_cast<const float4 *>(kaf + cp);
            uint32_t A0[4], A1[4];           // G16: hi and lo fragments; else A0 = hi rows over lo rows
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float4 qv = sm.h.qf[s][r][lane];
                beta2[r] = __ffma2_rn(make_float2(qv.x, qv.y), make_float2(aa.x, aa.y), beta2[r]);
                beta2[r] = __ffma2_rn(make_float2(qv.z, qv.w), make_float2(aa.z, aa.w), beta2[r]);
                float2 x01 = __fmul2_rn(make_float2(qv.x, qv.y), make_float2(bb.x, bb.y));
                float2 x23 = __fmul2_rn(make_float2(qv.z, qv.w), make_float2(bb.z, bb.w));
                if (G16) {
                    split2(x01, A0[r], A1[r]);
                    split2(x23, A0[2 + r], A1[2 + r]);
                } else {
                    split2(x01, A0[0], A0[1]);
                    split2(x23, A0[2], A0[3]);
                }
            }
            const int wi = s >> 1;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const uint32_t aw = wi == 0 ? kc[nt].x : wi == 1 ? kc[nt].y : wi == 2 ? kc[nt].z : kc[nt].w;
                uint32_t b0, b1;
                if (FULL) {
                    const uint32_t rw = wi == 0 ? kr4[nt].x : wi == 1 ? kr4[nt].y : wi == 2 ? kr4[nt].z : kr4[nt].w;
                    const uint32_t ev = codes_even(aw, rw), od = codes_odd(aw, rw);
                    if (s & 1) {
                        b0 = pack_lo(lut_ld<2>(ev, lb), lut_ld<2>(od, lb));
                        b1 = pack_lo(lut_ld<3>(ev, lb), lut_ld<3>(od, lb));
                    } else {
                        b0 = pack_lo(lut_ld<0>(ev, lb), lut_ld<0>(od, lb));
                        b1 = pack_lo(lut_ld<1>(ev, lb), lut_ld<1>(od, lb));
                    }
                } else {
                    if (s & 1) {
                        b0 = lut_ld<2>(aw, lb);
                        b1 = lut_ld<3>(aw, lb);
                    } else {
                        b0 = lut_ld<0>(aw, lb);
                        b1 = lut_ld<1>(aw, lb);
                    }
                }
                if (s == 0)
                    mma16816_z(S[nt], A0, b0, b1);
                else
                    mma16816(S[nt], A0, b0, b1);
                if (G16)
                    mma16816(S[nt], A1, b0, b1);
            }
        }

        // ---- scores (base-2 log domain) relative to the running reference
        // m_run (0 before the first chunk), masking, online softmax --------
        // The reference moves only when a score passes it by more than 2^8
        // (weights up to 2^8 are exact in fp32 and fine in fp16), so the
        // running output is rarely rescaled.
        float P[R][4][2];                    // row r, n-tile nt: tokens 8 nt + 2q, + 1
        float mref[R], mx[R], psum[R], oscale[R];
        bool up = false;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float bt = beta2[r].x + beta2[r].y;
            bt += __shfl_xor_sync(0xFFFFFFFFu, bt, 1);
            bt += __shfl_xor_sync(0xFFFFFFFFu, bt, 2);
            mref[r] = m_run[r] == neg_inf() ? 0.0f : m_run[r];
            const float bm = bt - mref[r];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float acc = G16 ? S[nt][2 * r + e] : S[nt][e] + S[nt][2 + e];
                    P[r][nt][e] = fmaf(acc, gscale, bm);
                }
        }
        if (nv < kChunk) {                   // ragged chunk: tokens past the context
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (8 * nt + 2 * q + e >= nv)
                            P[r][nt][e] = neg_inf();
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float m = fmaxf(fmaxf(fmaxf(P[r][0][0], P[r][0][1]), fmaxf(P[r][1][0], P[r][1][1])),
                            fmaxf(fmaxf(P[r][2][0], P[r][2][1]), fmaxf(P[r][3][0], P[r][3][1])));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            mx[r] = m;
            up |= m_run[r] == neg_inf() || m > 8.0f;
            const int h = g + 8 * r;
            if (a.scores && h < G) {
                float *srow = a.scores + (qrow0 + h) * score_stride + (int64_t)lp * kPage + j * kChunk;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    *reinterpret_cast<float2 *>(srow + nt * 8 + 2 * q) =
                        make_float2((P[r][nt][0] + mref[r]) * kLn2, (P[r][nt][1] + mref[r]) * kLn2);
            }
        }
        const bool rescale = __any_sync(0xFFFFFFFFu, up);
        if (rescale) {                       // rare: move the reference to this chunk's maximum
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const bool first = m_run[r] == neg_inf();
                const bool u = first || mx[r] > 8.0f;
                const float shift = u ? mx[r] : 0.0f;
                const float alpha = first ? 0.0f : exp2_sm(-shift);
                m_run[r] = mref[r] + shift;
                l_run[r] *= alpha;
                oscale[r] = alpha;           // applied to the outputs as they are loaded below
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    P[r][nt][0] -= shift;
                    P[r][nt][1] -= shift;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float ps = 0.0f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pv = exp2_sm(P[r][nt][e]);
                    P[r][nt][e] = pv;
                    ps += pv;
                }
            l_run[r] += ps;
            ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 1);
            ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 2);
            psum[r] = ps;
        }
        // P as A fragments; k-step kk = tokens 16 kk .. 16 kk + 15
        uint32_t PA0[2][4], PA1[2][4];       // G16: hi, lo; else PA0 = hi rows over lo rows
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            if (G16) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    split2(make_float2(P[r][2 * kk][0], P[r][2 * kk][1]), PA0[kk][r], PA1[kk][r]);
                    split2(make_float2(P[r][2 * kk + 1][0], P[r][2 * kk + 1][1]), PA0[kk][2 + r], PA1[kk][2 + r]);
                }
            } else {
                split2(make_float2(P[0][2 * kk][0], P[0][2 * kk][1]), PA0[kk][0], PA0[kk][1]);
                split2(make_float2(P[0][2 * kk + 1][0], P[0][2 * kk + 1][1]), PA0[kk][2], PA0[kk][3]);
            }
        }

        // ---- V: affines and codes of chunk j, then release the slot -------
        if (__any_sync(0xFFFFFFFFu, !wait_item(xk + 1))) {
            timed_out = true;
            break;
        }
        uint2 vc[2][4], vr4[2][4];           // [k-step][tokens 2q, 2q + 1, 2q + 8, 2q + 9], bytes 8g .. 8g + 7
        {
            const SlotMeta &mt = sm.h.meta[sV];
            __syncwarp();                    // every lane is done with K's affines
            chunk_affines(mt.pm, mt.cm, j, lane, vaf, vbf);
            const uint8_t *ca = sm.plane[sV][0] + (j * kChunk + 2 * q) * kRow + 8 * g;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    vc[kk][u] = *reinterpret_cast<const uint2 *>(ca + (16 * kk + (u & 1) + 8 * (u >> 1)) * kRow);
            if (FULL) {
                const uint8_t *cr = sm.plane[sV][FULL ? 1 : 0] + (j * kChunk + 2 * q) * kRow + 8 * g;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        vr4[kk][u] = *reinterpret_cast<const uint2 *>(cr + (16 * kk + (u & 1) + 8 * (u >> 1)) * kRow);
            }
            __syncwarp();
            if (lane == 0)
                release(xk + 1);
        }

        // ---- P.V: n-tile 2m + e holds channel 16 n + 2m + e of column n ------
        float4 vb4l, vb4h, va4l, va4h;       // affines of this lane's channels for m, m + 1
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {     // the running outputs of m = 4 hf .. 4 hf + 3, from tensor memory
        float o[32];
        tmem_wait_st();
        tmem_ld32f(tO + 32 * hf, o);
        tmem_wait_ld();
        if (rescale) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    o[16 * r + i] *= oscale[r];
        }
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const int m = 4 * hf + mm;
            const int wi = m >> 2;
            float C[2][4];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t bl0, bl1, bo0, bo1;   // (b0, b1) of n-tiles 2m and 2m + 1
                const uint32_t x0 = wi ? vc[kk][0].y : vc[kk][0].x, x1 = wi ? vc[kk][1].y : vc[kk][1].x;
                const uint32_t x2 = wi ? vc[kk][2].y : vc[kk][2].x, x3 = wi ? vc[kk][3].y : vc[kk][3].x;
                if (FULL) {
                    const uint32_t r0 = wi ? vr4[kk][0].y : vr4[kk][0].x, r1 = wi ? vr4[kk][1].y : vr4[kk][1].x;
                    const uint32_t r2 = wi ? vr4[kk][2].y : vr4[kk][2].x, r3 = wi ? vr4[kk][3].y : vr4[kk][3].x;
                    const uint32_t e0 = codes_even(x0, r0), e1 = codes_even(x1, r1);
                    const uint32_t e2 = codes_even(x2, r2), e3 = codes_even(x3, r3);
                    const uint32_t o0 = codes_odd(x0, r0), o1 = codes_odd(x1, r1);
                    const uint32_t o2 = codes_odd(x2, r2), o3 = codes_odd(x3, r3);
                    switch (m & 3) {
#define LYNX_V_FULL(I)                                                                                                 \
case I:                                                                                                            \
    bl0 = pack_lo(lut_ld<I>(e0, lb), lut_ld<I>(e1, lb));                                      \
    bl1 = pack_lo(lut_ld<I>(e2, lb), lut_ld<I>(e3, lb));                                      \
    bo0 = pack_lo(lut_ld<I>(o0, lb), lut_ld<I>(o1, lb));                                      \
    bo1 = pack_lo(lut_ld<I>(o2, lb), lut_ld<I>(o3, lb));                                      \
    break;
                        LYNX_V_FULL(0)
                        LYNX_V_FULL(1)
                        LYNX_V_FULL(2)
                        default:
                        LYNX_V_FULL(3)
#undef LYNX_V_FULL
                    }
                } else {
                    const uint32_t e01 = nib_even(x0, x1), e23 = nib_even(x2, x3);
                    const uint32_t o01 = nib_odd(x0, x1), o23 = nib_odd(x2, x3);
                    switch (m & 3) {
#define LYNX_V_ANCHOR(I)                                                                                               \
case I:                                                                                                            \
    bl0 = lut_ld<I>(e01, lb);                                                                          \
    bl1 = lut_ld<I>(e23, lb);                                                                          \
    bo0 = lut_ld<I>(o01, lb);                                                                          \
    bo1 = lut_ld<I>(o23, lb);                                                                          \
    break;
                        LYNX_V_ANCHOR(0)
                        LYNX_V_ANCHOR(1)
                        LYNX_V_ANCHOR(2)
                        default:
                        LYNX_V_ANCHOR(3)
#undef LYNX_V_ANCHOR
                    }
                }
                if (kk == 0) {
                    mma16816_z(C[0], PA0[kk], bl0, bl1);
                    mma16816_z(C[1], PA0[kk], bo0, bo1);
                } else {
                    mma16816(C[0], PA0[kk], bl0, bl1);
                    mma16816(C[1], PA0[kk], bo0, bo1);
                }
                if (G16) {
                    mma16816(C[0], PA1[kk], bl0, bl1);
                    mma16816(C[1], PA1[kk], bo0, bo1);
                }
            }
            // o += b (P.L) + a sum(P): column 2q -> channels 32q + 2m, + 1;
            // column 2q + 1 -> channels 32q + 16 + 2m, + 1
            if ((m & 1) == 0) {
                vb4l = *reinterpret_cast<const float4 *>(vbf + 36 * q + 2 * m);
                vb4h = *reinterpret_cast<const float4 *>(vbf + 36 * q + 16 + 2 * m);
                va4l = *reinterpret_cast<const float4 *>(vaf + 36 * q + 2 * m);
                va4h = *reinterpret_cast<const float4 *>(vaf + 36 * q + 16 + 2 * m);
            }
            const float2 bl = (m & 1) ? make_float2(vb4l.z, vb4l.w) : make_float2(vb4l.x, vb4l.y);
            const float2 bh = (m & 1) ? make_float2(vb4h.z, vb4h.w) : make_float2(vb4h.x, vb4h.y);
            const float2 al = (m & 1) ? make_float2(va4l.z, va4l.w) : make_float2(va4l.x, va4l.y);
            const float2 ah = (m & 1) ? make_float2(va4h.z, va4h.w) : make_float2(va4h.x, va4h.y);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float2 cl, ch;
                if (G16) {
                    cl = make_float2(C[0][2 * r], C[1][2 * r]);
                    ch = make_float2(C[0][2 * r + 1], C[1][2 * r + 1]);
                } else {
                    cl = make_float2(C[0][0] + C[0][2], C[1][0] + C[1][2]);
                    ch = make_float2(C[0][1] + C[0][3], C[1][1] + C[1][3]);
                }
                const float2 ps2 = make_float2(psum[r], psum[r]);
                float *ol = o + 16 * r + 4 * mm;
                const float2 nl = __ffma2_rn(bl, cl, __ffma2_rn(al, ps2, make_float2(ol[0], ol[1])));
                const float2 nh = __ffma2_rn(bh, ch, __ffma2_rn(ah, ps2, make_float2(ol[2], ol[3])));
                ol[0] = nl.x;
                ol[1] = nl.y;
                ol[2] = nh.x;
                ol[3] = nh.y;
            }
        }
        tmem_st32f(tO + 32 * hf, o);
        }
    }
    if (timed_out && a.dev_err && lane == 0)
        atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
    __syncthreads();
    if (tid == 0) {
        // every copy issued must land before the merge reuses the slots
        // (after a timeout some may still be in flight; bounded)
        bool ok = mbar_wait_bounded(&sm.h.q_bar, 0u, kWaitLimit);
        for (int s = 0; s < NS; ++s)
            if (sm.h.last[s] >= 0 && !mbar_wait_bounded(&sm.h.full_bar[s], (uint32_t)((sm.h.last[s] / NS) & 1), kWaitLimit))
                ok = false;
        if (!ok && a.dev_err)
            atomicOr(a.dev_err, LYNX_DEVERR_TIMEOUT);
    }

    // the combine kernel that follows may be scheduled now (it waits for
    // this grid's completion before reading the partials)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- merge the chunks' states, write this range's partial ------------
    __syncthreads();   // every copy has landed and every table and plane read is done: the merge area overlays them
    Merge &mg = *reinterpret_cast<Merge *>(sm.lut);
#pragma unroll
    for (int r = 0; r < R; ++r) {            // (1) every warp's (max, sum) per query head
        const int h = g + 8 * r;
        float l = l_run[r];
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
        if (q == 0) {
            mg.m[warp][h] = m_run[r];
            mg.l[warp][h] = l;
        }
    }
    __syncthreads();
    static_assert(kWarps == 16, "one 16-lane group per query head below");
    if (tid < 16 * kWarps) {                 // (2) lane group h: warp w's weight for query head h
        const int h = tid >> 4, w = tid & 15;
        const float mw = mg.m[w][h];
        float M = mw;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        const float sc = M > neg_inf() ? exp2f(mw - M) : 0.0f;
        float L = mg.l[w][h] * sc;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
            L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
        mg.sc[h][w] = sc;
        if (w == 0) {
            mg.M[h] = M;
            mg.L[h] = L;
        }
    }
    tmem_wait_st();                          // this warp's last output stores are done
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    {
        // (3) inside each lane quarter: warp (quarter q4, part cb) sums slice cb
        // (16 columns) of the quarter's four warps' blocks, weighted. A lane holds
        // the same (g, q) positions in every warp of its quarter; slice cb is
        // half cb / 2 and row group cb % 2 of the block layout above
        const int q4 = warp & 3, cb = warp >> 2, hf = cb >> 1, r = cb & 1, h = g + 8 * r;
        if (G16 || r == 0) {
            const uint32_t tq = sm.h.tmem + ((uint32_t)(32 * q4) << 16) + 16u * (uint32_t)cb;
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                acc[i] = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {    // warp q4 + 4k: its block starts at column 64k
                float v[16];
                tmem_ld16(tq + 64u * (uint32_t)k, v);
                tmem_wait_ld();
                const float s = mg.sc[h][q4 + 4 * k];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[i] = fmaf(v[i], s, acc[i]);
            }
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) { // column 4 mm + 2 side + e: channel 32 q + 16 side + 2 (4 hf + mm) + e
                const int m = 4 * hf + mm;
                *reinterpret_cast<float2 *>(&mg.o4[q4][h][34 * q + 2 * m]) = make_float2(acc[4 * mm], acc[4 * mm + 1]);
                *reinterpret_cast<float2 *>(&mg.o4[q4][h][34 * q + 16 + 2 * m]) =
                    make_float2(acc[4 * mm + 2], acc[4 * mm + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {                         // every warp's tensor-memory reads are done
        tc_fence_after();
        tmem_dealloc(sm.h.tmem, kTmemCols);
    }
    for (int e = tid; e < G * kD; e += kThreads) {   // (4) the four quarters' sums
        const int h = e / kD, d = e % kD, c = 34 * (d >> 5) + (d & 31);
        const float o = (mg.o4[0][h][c] + mg.o4[1][h][c]) + (mg.o4[2][h][c] + mg.o4[3][h][c]);
        float *pp = a.part + ((qrow0 + h) * a.n_splits + split) * kPart;
        pp[d] = o;
        if (d == 0) {
            pp[kD] = mg.M[h];
            pp[kD + 1] = mg.L[h];
        }
    }
}

template <bool G16, bool FULL, int NS>
cudaError_t run(const AttnArgs &a, cudaStream_t s)
{
    static_assert(sizeof(Head<NS>) <= kPre, "everything ahead of the table fits below 0x10000");
    static_assert(sizeof(Merge) <= sizeof(uint32_t) * 256 * 64 + NS * (FULL ? 2 : 1) * kPlane,
                  "merge area overlays the table and the planes");
    static_assert(sizeof(Smem<FULL, NS>) <= 227 * 1024, "shared memory per CTA");
    const size_t smem = sizeof(Smem<FULL, NS>);
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<G16, FULL, NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)a.n_splits, (unsigned)a.H, (unsigned)a.B);
    attn_mma_kernel<G16, FULL, NS><<<grid, kThreads, smem, s>>>(a, host_tables().lev);
    return cudaGetLastError();
}

__device__ uint32_t g_dyn_base;

__global__ void dyn_base_probe()
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    g_dyn_base = smem_u32(smem_raw);
}

// Whether the dynamic shared window of this device starts at kDynBase, so
// that the attention kernel's level table sits at shared address 0x10000.
// Measured by a one-thread kernel at the first call on each device (a
// synchronous step: that first call must not be inside a stream capture).
bool table_aligned()
{
    static std::mutex mu;
    static int state[64] = {};   // 0 unknown, 1 aligned, 2 not
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    if (state[dev] == 0) {
        uint32_t base = 0;
        dyn_base_probe<<<1, 1, 16>>>();
        const bool ok = cudaGetLastError() == cudaSuccess &&
                        cudaMemcpyFromSymbol(&base, g_dyn_base, sizeof(base)) == cudaSuccess;
        state[dev] = ok && base == kDynBase ? 1 : 2;
    }
    return state[dev] == 1;
}

} // namespace

cudaError_t launch_attn_mma(const AttnArgs &a, cudaStream_t s)
{
    // slots hold one tensor's page: 16 KiB of codes in anchor mode, 32 KiB in full mode
    if (!table_aligned())
        return cudaErrorNotSupported;
    if (a.G <= 8)
        return a.full ? run<false, true, 3>(a, s) : run<false, false, 6>(a, s);
    return a.full ? run<true, true, 3>(a, s) : run<true, false, 6>(a, s);
}

} // namespace lynx
