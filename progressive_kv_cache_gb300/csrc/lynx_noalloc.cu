// lynx_noalloc.cu -- decode attention for callers that cannot allocate.
//
// lynx_decode_attn asks its caller for a workspace (the split-K partial
// results). Some callers have no way to provide one: a serving engine whose
// memory pool has already reserved all free device memory for the KV cache,
// a plugin that is handed only its input and output buffers, or a
// latency-critical path where cudaMalloc (which can synchronise the device)
// is not allowed. lynx_decode_attn_noalloc serves them: its scratch lives in
// the fixed-size device array below, which every GPU that loads this library
// holds from module load until process exit.
#include <mutex>

#include "lynx_internal.cuh"

namespace {

// 16 MiB of split-K partials (LYNX_NOALLOC_SCRATCH_BYTES): enough for batch 1 x
// 64 query heads x 512 pages (a 128K-token context) and for 32 requests x 64
// query heads x 64 pages.
constexpr size_t kNoAllocScratchBytes = LYNX_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device. In host code the array's name is only a host-side stand-in;
// the device address has to come from cudaGetSymbolAddress.
lynx_status scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return LYNX_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return LYNX_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return LYNX_OK;
}

} // namespace

extern "C" lynx_status lynx_decode_attn_noalloc(const void *q_bf16, const lynx_qkv *k, const lynx_qkv *v,
                                                int32_t layer, const int32_t *page_table, const int32_t *ctx_lens,
                                                int32_t batch, int32_t q_heads, int32_t max_pages, float sm_scale,
                                                lynx_mode mode, float *out, float *scores, uint32_t *dev_err,
                                                void *stream)
{
    // The scratch is offered to lynx_decode_attn as a workspace of
    // kNoAllocScratchBytes: its own checks (arguments first, then the split
    // plan of this very shape against the workspace size) run before anything
    // is launched, so a shape whose partials do not fit is refused there with
    // LYNX_ERR_WORKSPACE.
    void *scratch = nullptr;
    if (batch > 0 && q_heads > 0) {
        lynx_status st = scratch_for_current_device(&scratch);
        if (st != LYNX_OK)
            return st;
    }
    return lynx_decode_attn(q_bf16, k, v, layer, page_table, ctx_lens, batch, q_heads, max_pages, sm_scale, mode,
                            out, scores, scratch, scratch ? kNoAllocScratchBytes : 0, dev_err, stream);
}
