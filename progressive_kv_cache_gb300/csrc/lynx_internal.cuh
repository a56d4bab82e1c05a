// lynx_internal.cuh -- types shared by the library's translation units.
//
// The tables below are built once on the host (lynx_tables.cu) from the
// written definitions of the Lynx quantizer (section 3 "The quantizer" of the
// aigenapps reading) and passed to kernels by value, so the library holds no
// device-global state and needs no initialisation call.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/lynx.h"

namespace lynx {

constexpr int kPage = 256;     // tokens per page
constexpr int kChunk = 32;     // C = 32 tokens per chunk
constexpr int kNChunk = kPage / kChunk;
constexpr int kD = 128;        // head dimension
constexpr int kQMax = 63;      // codes -63..63 (127 levels)
constexpr int kBias = 7;       // +7 before the 4-bit cut
constexpr double kAlpha = 255.0;

// Stage-3 bucket table. The code of w depends only on |w| through the count
// q = #{k : |w| >= T_k}, and the table finds q with one lookup and one
// integer add: the bucket of |w| is bits(fp32(|w| + 2^-13)) >> 19, a monotone
// function of |w| with 16 buckets per octave of |w| + 2^-13, each narrower
// than the gap between two consecutive thresholds, so at most one threshold
// T* lies in a bucket (the builder checks this). |w| in [0, 2 - 2^-13) gives
// buckets kBucketBase .. kBucketBase + kNBucket - 1 with no clamp. Each entry holds
// K = 2^30 - bits(T*) (0 when the bucket holds none) and the four possible
// stored bytes (c + 7) & 0xFF. For |w| < 2, bits(|w|) < 2^30, and for
// non-negative floats bits(|w|) >= bits(T*) exactly when |w| >= T*, so
// bits(w) + K never carries into bit 31 and its bits 31-30 are
// 2 * sign(w) + (|w| >= T*), the index of the stored byte:
//   byte 0: w >= 0 below T*   byte 1: w >= 0 at or above T*
//   byte 2: w < 0 below T*    byte 3: w < 0 at or above T*
// (sign(w) is the sign bit: the encoder turns -0 into +0 first).
constexpr uint32_t kBucketBase = (127u - 13u) << 4;   // bucket of 2^-13
constexpr int kNBucket = 14 * 16;                      // |w| + 2^-13 in [2^-13, 2)
constexpr uint32_t kBucketOffsetBits = (127u - 13u) << 23;   // 2^-13

struct CodeTable {
    uint2 e[kNBucket];
};

// Signed level values used by the decoders:
//   full[(A & 15) << 4 | r] = sgn(c) * Lv[min(|c|, 64)], c = 16A + r - 7
//   anchor[A & 15]          = sgn(16A) * Lv[min(|16A|, 64)]
struct LevelTable {
    float full[256];
    float anchor[16];
};

struct HostTables {
    float thr[64];
    uint16_t lv[65];
    CodeTable code;
    LevelTable lev;
    bool ok;
};

const HostTables &host_tables();   // built once, thread-safe

int device_sm_count();             // SM count of the current device (cached per device)

// ---- launchers (one per translation unit) -------------------------------
cudaError_t launch_quantize(const uint16_t *x, const int32_t *page_valid, const lynx_qkv &o,
                            cudaStream_t s);
cudaError_t launch_quantize_append(const uint16_t *tail, const int32_t *dst_page, const int32_t *valid, int n,
                                   const lynx_qkv &o, uint32_t *dev_err, cudaStream_t s);
cudaError_t launch_level_codes(const float *w, int64_t n, int8_t *codes, cudaStream_t s);
cudaError_t launch_dequant(const lynx_qkv &in, void *out, bool full, bool f32, cudaStream_t s);
cudaError_t launch_quantize_variant(const uint16_t *x, int64_t pages, const lynx_variant &v, int16_t *codes,
                                    int8_t *anchor, uint8_t *resid, float *page_meta, uint16_t *chunk_meta,
                                    double *err, float *x_anchor, float *x_full, cudaStream_t s);
cudaError_t launch_dense_attn(const uint16_t *q, const float *k, const float *v, int B, int Hq, int H, int T,
                              float sm_scale, float *out, cudaStream_t s);
int dense_attn_max_tokens();

struct AttnArgs {
    const uint16_t *q;
    const uint8_t *ka, *kr, *va, *vr;
    const float *kpm, *vpm;
    const uint16_t *kcm, *vcm;
    const int32_t *page_table, *ctx;
    float *out, *scores, *part;
    uint32_t *dev_err;
    int B, Hq, H, G, max_pages, pool_pages, n_splits, pages_per_split;
    float sm_scale;
    bool full;
};
// Split-K plan: pages of each (request, KV head) are cut into n_splits ranges
// of pages_per_split pages. Partials are (o[128], m, l) with m in the base-2
// log domain (scores pre-multiplied by log2(e)).
void attn_split_plan(int batch, int kv_heads, int max_pages, int sms, int *n_splits, int *pages_per_split);
int attn_max_splits(int batch, int q_heads, int max_pages, int sms);   // over every valid kv_heads
size_t attn_workspace_bytes(int batch, int q_heads, int n_splits);
cudaError_t launch_decode_attn(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_attn_mma(const AttnArgs &a, cudaStream_t s);        // tensor-core path, G <= 16
cudaError_t launch_attn_combine(const AttnArgs &a, cudaStream_t s);

struct VerifyArgs {
    const uint16_t *q;                        // [B][Tq][Hq][128] bf16
    const uint8_t *ka, *kr, *va, *vr;         // planes of one layer (all KV heads)
    const float *kpm, *vpm;
    const uint16_t *kcm, *vcm;
    const int32_t *page_table, *ctx;
    float *out, *part;                        // out [B][Tq][Hq][128]; partials [B*Tq*Hq][n_splits][130]
    uint32_t *dev_err;
    int B, Tq, Hq, H, G, RB, max_pages, pool_pages, n_splits, pages_per_split;
    float sm_scale;
    bool full;
};
int verify_row_blocks(int draft, int G);      // CTAs across the T_q * G query rows of a KV head
cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s);

// ---- device helpers ------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

} // namespace lynx
