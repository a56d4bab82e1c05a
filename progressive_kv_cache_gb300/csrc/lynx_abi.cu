// lynx_abi.cu -- the extern "C" entry points declared in include/lynx.h:
// argument checks on the host, then one launch sequence per call. Nothing is
// allocated here; every buffer belongs to the caller.
#include <cstdint>
#include <cstring>

#include "lynx_internal.cuh"

using namespace lynx;

namespace {

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

lynx_status check_qkv(const lynx_qkv *t, bool need_residual)
{
    if (!t || !t->anchor || !t->page_meta || !t->chunk_meta || (need_residual && !t->residual))
        return LYNX_ERR_NULL;
    if (t->layers < 0 || t->kv_heads < 0 || t->tokens < 0 || t->tokens % kPage || t->head_dim != kD)
        return LYNX_ERR_SHAPE;
    if (!aligned(t->anchor, 16) || !aligned(t->page_meta, 16) || !aligned(t->chunk_meta, 16) ||
        (t->residual && !aligned(t->residual, 16)))
        return LYNX_ERR_ALIGN;
    if (!host_tables().ok)
        return LYNX_ERR_UNSUPPORTED;
    return LYNX_OK;
}

lynx_status from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? LYNX_OK : e == cudaErrorNotSupported ? LYNX_ERR_UNSUPPORTED : LYNX_ERR_CUDA;
}

} // namespace

extern "C" {

const char *lynx_status_string(lynx_status s)
{
    switch (s) {
    case LYNX_OK: return "ok";
    case LYNX_ERR_NULL: return "a required pointer is NULL";
    case LYNX_ERR_SHAPE: return "invalid or unsupported shape";
    case LYNX_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
    case LYNX_ERR_UNSUPPORTED: return "unsupported configuration";
    case LYNX_ERR_WORKSPACE: return "workspace too small";
    case LYNX_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

void lynx_host_tables(float *thr, uint16_t *lv)
{
    const HostTables &t = host_tables();
    if (thr)
        std::memcpy(thr, t.thr, sizeof t.thr);
    if (lv)
        std::memcpy(lv, t.lv, sizeof t.lv);
}

lynx_status lynx_quantize_pages(const void *x_bf16, const int32_t *page_valid, const lynx_qkv *out, void *stream)
{
    lynx_status st = check_qkv(out, true);
    if (st != LYNX_OK)
        return st;
    if (!x_bf16)
        return LYNX_ERR_NULL;
    if (!aligned(x_bf16, 16) || (page_valid && !aligned(page_valid, 4)))
        return LYNX_ERR_ALIGN;
    return from_cuda(launch_quantize(static_cast<const uint16_t *>(x_bf16), page_valid, *out, (cudaStream_t)stream));
}

lynx_status lynx_quantize_append(const void *tail_bf16, const int32_t *phys_page, const int32_t *valid,
                                 int32_t n, const lynx_qkv *out, uint32_t *dev_err, void *stream)
{
    lynx_status st = check_qkv(out, true);
    if (st != LYNX_OK)
        return st;
    if (n < 0 || (int64_t)out->layers * out->kv_heads > INT32_MAX)
        return LYNX_ERR_SHAPE;
    if (n == 0 || out->layers == 0 || out->kv_heads == 0)
        return LYNX_OK;
    if (!tail_bf16 || !phys_page || !valid)
        return LYNX_ERR_NULL;
    if (!aligned(tail_bf16, 16) || !aligned(phys_page, 4) || !aligned(valid, 4) || (dev_err && !aligned(dev_err, 4)))
        return LYNX_ERR_ALIGN;
    return from_cuda(launch_quantize_append(static_cast<const uint16_t *>(tail_bf16), phys_page, valid, n, *out,
                                            dev_err, (cudaStream_t)stream));
}

lynx_status lynx_dequant_anchor(const lynx_qkv *in, void *out, lynx_out_dtype dt, void *stream)
{
    lynx_status st = check_qkv(in, false);
    if (st != LYNX_OK)
        return st;
    if (!out)
        return LYNX_ERR_NULL;
    if (!aligned(out, 16))
        return LYNX_ERR_ALIGN;
    if (dt != LYNX_OUT_BF16 && dt != LYNX_OUT_F32)
        return LYNX_ERR_UNSUPPORTED;
    return from_cuda(launch_dequant(*in, out, false, dt == LYNX_OUT_F32, (cudaStream_t)stream));
}

lynx_status lynx_refine_residual(const lynx_qkv *in, void *inout, lynx_out_dtype dt, void *stream)
{
    lynx_status st = check_qkv(in, true);
    if (st != LYNX_OK)
        return st;
    if (!inout)
        return LYNX_ERR_NULL;
    if (!aligned(inout, 16))
        return LYNX_ERR_ALIGN;
    if (dt != LYNX_OUT_BF16 && dt != LYNX_OUT_F32)
        return LYNX_ERR_UNSUPPORTED;
    return from_cuda(launch_dequant(*in, inout, true, dt == LYNX_OUT_F32, (cudaStream_t)stream));
}

size_t lynx_decode_attn_workspace(int32_t batch, int32_t q_heads, int32_t max_pages)
{
    if (batch <= 0 || q_heads <= 0 || max_pages <= 0)
        return 0;
    const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
    return attn_workspace_bytes(batch, q_heads, attn_max_splits(batch, q_heads, max_pages, sms));
}

lynx_status lynx_decode_attn(const void *q_bf16, const lynx_qkv *k, const lynx_qkv *v, int32_t layer,
                             const int32_t *page_table, const int32_t *ctx_lens, int32_t batch, int32_t q_heads,
                             int32_t max_pages, float sm_scale, lynx_mode mode, float *out, float *scores,
                             void *workspace, size_t ws_bytes, uint32_t *dev_err, void *stream)
{
    const bool full = mode == LYNX_MODE_FULL;
    if (mode != LYNX_MODE_ANCHOR && mode != LYNX_MODE_FULL)
        return LYNX_ERR_UNSUPPORTED;
    lynx_status st = check_qkv(k, full);
    if (st != LYNX_OK)
        return st;
    if ((st = check_qkv(v, full)) != LYNX_OK)
        return st;
    if (!q_bf16 || !page_table || !ctx_lens || !out)
        return LYNX_ERR_NULL;
    if (batch < 0 || q_heads < 0 || max_pages <= 0 || k->kv_heads <= 0)
        return LYNX_ERR_SHAPE;
    if (k->layers != v->layers || k->kv_heads != v->kv_heads || k->tokens != v->tokens)
        return LYNX_ERR_SHAPE;
    if (layer < 0 || layer >= k->layers || q_heads % k->kv_heads)
        return LYNX_ERR_SHAPE;
    const int G = q_heads / k->kv_heads;
    if (batch > 0 && G > 32)
        return LYNX_ERR_UNSUPPORTED;
    if (!aligned(q_bf16, 16) || !aligned(out, 16) || (scores && !aligned(scores, 16)) ||
        !aligned(page_table, 4) || !aligned(ctx_lens, 4) || (dev_err && !aligned(dev_err, 4)) ||
        (workspace && !aligned(workspace, 16)))
        return LYNX_ERR_ALIGN;
    if (batch == 0 || q_heads == 0)
        return LYNX_OK;
    const int sms = device_sm_count();
    if (sms <= 0)
        return LYNX_ERR_CUDA;
    int n_splits = 1, pps = 1;
    attn_split_plan(batch, k->kv_heads, max_pages, sms, &n_splits, &pps);
    if (!workspace)
        return LYNX_ERR_NULL;
    if (ws_bytes < attn_workspace_bytes(batch, q_heads, n_splits))
        return LYNX_ERR_WORKSPACE;

    const int64_t H = k->kv_heads, T = k->tokens, P = T / kPage;
    const int64_t plane_off = (int64_t)layer * H * T * (kD / 2);
    const int64_t pm_off = (int64_t)layer * H * P * (2 * kD);
    const int64_t cm_off = (int64_t)layer * H * P * (kNChunk * 2 * kD);
    AttnArgs a{};
    a.q = static_cast<const uint16_t *>(q_bf16);
    a.ka = k->anchor + plane_off;
    a.kr = full ? k->residual + plane_off : nullptr;
    a.va = v->anchor + plane_off;
    a.vr = full ? v->residual + plane_off : nullptr;
    a.kpm = k->page_meta + pm_off;
    a.vpm = v->page_meta + pm_off;
    a.kcm = k->chunk_meta + cm_off;
    a.vcm = v->chunk_meta + cm_off;
    a.page_table = page_table;
    a.ctx = ctx_lens;
    a.out = out;
    a.scores = scores;
    a.part = static_cast<float *>(workspace);
    a.dev_err = dev_err;
    a.B = batch;
    a.Hq = q_heads;
    a.H = (int)H;
    a.G = G;
    a.max_pages = max_pages;
    a.pool_pages = (int)P;
    a.n_splits = n_splits;
    a.pages_per_split = pps;
    a.sm_scale = sm_scale;
    a.full = full;
    return from_cuda(launch_decode_attn(a, (cudaStream_t)stream));
}

// Split plan of the verify pass: the (request, row block) pairs play the part
// of the requests of the decode plan.
static void verify_plan(int batch, int draft, int kv_heads, int G, int max_pages, int sms, int *rb, int *n_splits,
                        int *pps)
{
    *rb = verify_row_blocks(draft, G);
    attn_split_plan(batch * *rb, kv_heads, max_pages, sms, n_splits, pps);
}

size_t lynx_verify_attn_workspace(int32_t batch, int32_t draft, int32_t q_heads, int32_t max_pages)
{
    if (batch <= 0 || draft <= 0 || draft > 64 || q_heads <= 0 || max_pages <= 0)
        return 0;
    const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
    int best = 1;
    for (int h = 1; h <= q_heads; ++h) {      // every kv_heads the call may pass
        if (q_heads % h)
            continue;
        int rb = 1, n = 1, pps = 1;
        verify_plan(batch, draft, h, q_heads / h, max_pages, sms, &rb, &n, &pps);
        best = n > best ? n : best;
    }
    return attn_workspace_bytes(batch * draft, q_heads, best);
}

lynx_status lynx_verify_attn(const void *q_bf16, const lynx_qkv *k, const lynx_qkv *v, int32_t layer,
                             const int32_t *page_table, const int32_t *ctx_lens, int32_t batch, int32_t draft,
                             int32_t q_heads, int32_t max_pages, float sm_scale, lynx_mode mode, float *out,
                             void *workspace, size_t ws_bytes, uint32_t *dev_err, void *stream)
{
    const bool full = mode == LYNX_MODE_FULL;
    if (mode != LYNX_MODE_ANCHOR && mode != LYNX_MODE_FULL)
        return LYNX_ERR_UNSUPPORTED;
    lynx_status st = check_qkv(k, full);
    if (st != LYNX_OK)
        return st;
    if ((st = check_qkv(v, full)) != LYNX_OK)
        return st;
    if (!q_bf16 || !page_table || !ctx_lens || !out)
        return LYNX_ERR_NULL;
    if (batch < 0 || draft < 1 || draft > 64 || q_heads < 0 || max_pages <= 0 || k->kv_heads <= 0)
        return LYNX_ERR_SHAPE;
    if (k->layers != v->layers || k->kv_heads != v->kv_heads || k->tokens != v->tokens)
        return LYNX_ERR_SHAPE;
    if (layer < 0 || layer >= k->layers || q_heads % k->kv_heads)
        return LYNX_ERR_SHAPE;
    if (!aligned(q_bf16, 16) || !aligned(out, 16) || !aligned(page_table, 4) || !aligned(ctx_lens, 4) ||
        (dev_err && !aligned(dev_err, 4)) || (workspace && !aligned(workspace, 16)))
        return LYNX_ERR_ALIGN;
    if (batch == 0 || q_heads == 0)
        return LYNX_OK;
    const int sms = device_sm_count();
    if (sms <= 0)
        return LYNX_ERR_CUDA;
    const int G = q_heads / k->kv_heads;
    int rb = 1, n_splits = 1, pps = 1;
    verify_plan(batch, draft, k->kv_heads, G, max_pages, sms, &rb, &n_splits, &pps);
    if (!workspace)
        return LYNX_ERR_NULL;
    if (ws_bytes < attn_workspace_bytes(batch * draft, q_heads, n_splits))
        return LYNX_ERR_WORKSPACE;

    const int64_t H = k->kv_heads, T = k->tokens, P = T / kPage;
    const int64_t plane_off = (int64_t)layer * H * T * (kD / 2);
    const int64_t pm_off = (int64_t)layer * H * P * (2 * kD);
    const int64_t cm_off = (int64_t)layer * H * P * (kNChunk * 2 * kD);
    VerifyArgs a{};
    a.q = static_cast<const uint16_t *>(q_bf16);
    a.ka = k->anchor + plane_off;
    a.kr = full ? k->residual + plane_off : nullptr;
    a.va = v->anchor + plane_off;
    a.vr = full ? v->residual + plane_off : nullptr;
    a.kpm = k->page_meta + pm_off;
    a.vpm = v->page_meta + pm_off;
    a.kcm = k->chunk_meta + cm_off;
    a.vcm = v->chunk_meta + cm_off;
    a.page_table = page_table;
    a.ctx = ctx_lens;
    a.out = out;
    a.part = static_cast<float *>(workspace);
    a.dev_err = dev_err;
    a.B = batch;
    a.Tq = draft;
    a.Hq = q_heads;
    a.H = (int)H;
    a.G = G;
    a.RB = rb;
    a.max_pages = max_pages;
    a.pool_pages = (int)P;
    a.n_splits = n_splits;
    a.pages_per_split = pps;
    a.sm_scale = sm_scale;
    a.full = full;
    return from_cuda(launch_verify(a, (cudaStream_t)stream));
}

lynx_status lynx_level_codes(const float *w, int64_t n, int8_t *codes, void *stream)
{
    if (n < 0)
        return LYNX_ERR_SHAPE;
    if (n > 0 && (!w || !codes))
        return LYNX_ERR_NULL;
    if (!host_tables().ok)
        return LYNX_ERR_UNSUPPORTED;
    return from_cuda(launch_level_codes(w, n, codes, (cudaStream_t)stream));
}

lynx_status lynx_quantize_variant(const void *x_bf16, int32_t n, int32_t tokens, const lynx_variant *v,
                                  int16_t *codes, int8_t *anchor, uint8_t *residual, float *page_meta,
                                  uint16_t *chunk_meta, double *err, float *x_anchor, float *x_full,
                                  void *stream)
{
    if (!v)
        return LYNX_ERR_NULL;
    if (n < 0 || tokens < 0 || tokens % kPage)
        return LYNX_ERR_SHAPE;
    if (v->uniform_bits < 0 || v->uniform_bits > 8)
        return LYNX_ERR_UNSUPPORTED;
    if (v->uniform_bits > 0 && (v->flags & ~LYNX_VAR_UNIFORM_PER_TOKEN))
        return LYNX_ERR_UNSUPPORTED;
    if (v->uniform_bits == 0) {
        if (v->chunk != 16 && v->chunk != 32 && v->chunk != 64)
            return LYNX_ERR_UNSUPPORTED;
        if (v->anchor_bits < 1 || v->anchor_bits > 6 || v->residual_bits < 1 || v->residual_bits > 4 ||
            v->anchor_bits + v->residual_bits > 8 || v->anchor_bits + v->residual_bits < 3)
            return LYNX_ERR_UNSUPPORTED;
        if (!(v->alpha >= 0.0f) || !(v->alpha <= 3.0e38f))
            return LYNX_ERR_UNSUPPORTED;
        if (v->flags & ~(LYNX_VAR_NO_PAGE_NORM | LYNX_VAR_NO_CHUNK_ISOLATION | LYNX_VAR_NO_BIAS | LYNX_VAR_NO_SIGN_AWARE))
            return LYNX_ERR_UNSUPPORTED;
    }
    const int64_t pages = (int64_t)n * (tokens / kPage);
    if (pages == 0)
        return LYNX_OK;
    if (!x_bf16)
        return LYNX_ERR_NULL;
    const void *ptrs[] = {x_bf16, codes, anchor, residual, page_meta, chunk_meta, err, x_anchor, x_full};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16))
            return LYNX_ERR_ALIGN;
    return from_cuda(launch_quantize_variant(static_cast<const uint16_t *>(x_bf16), pages, *v, codes, anchor,
                                             residual, page_meta, chunk_meta, err, x_anchor, x_full,
                                             (cudaStream_t)stream));
}

lynx_status lynx_dense_attn(const void *q_bf16, const float *k, const float *v, int32_t batch, int32_t q_heads,
                            int32_t kv_heads, int32_t tokens, float sm_scale, float *out, void *stream)
{
    if (batch < 0 || q_heads < 0 || kv_heads < 0 || tokens < 0)
        return LYNX_ERR_SHAPE;
    if (batch == 0 || q_heads == 0)
        return LYNX_OK;
    if (kv_heads == 0 || q_heads % kv_heads || tokens == 0 || tokens > dense_attn_max_tokens())
        return LYNX_ERR_SHAPE;
    if (!q_bf16 || !k || !v || !out)
        return LYNX_ERR_NULL;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(q_bf16, 2) || !aligned(out, 4))
        return LYNX_ERR_ALIGN;
    return from_cuda(launch_dense_attn(static_cast<const uint16_t *>(q_bf16), k, v, batch, q_heads, kv_heads, tokens,
                                       sm_scale, out, (cudaStream_t)stream));
}

} // extern "C"
