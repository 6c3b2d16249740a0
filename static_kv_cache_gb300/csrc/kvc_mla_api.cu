// kvc_mla_api.cu -- host side of the MLA latent cache: argument checks, the
// workspace layout, tensor maps and the three launches of a decode step.
#include <cmath>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>

#include "../../include/kvc.h"
#include "kvc_internal.cuh"
#include "kvc_mla.cuh"

struct kvc_mla_cache {
    kvc_mla_config cfg;
    const kvc::MlaKernelInfo *info;
    uint8_t *c_base;
    uint8_t *ws;
    uint64_t ws_bytes;
    uint64_t off_qt, off_ml, off_acc;  // workspace sections; the error word is at 0
    int num_sms;
    int n_stages;
    int smem_bytes;
    int num_splits;                    // 0: automatic
    CUtensorMap tm64, tm16;
};

namespace {

uint64_t round256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool mla_shape_ok(const kvc_mla_config *c) {
    return c && c->n_layers > 0 && c->batch > 0 && c->n_heads > 0 && c->d_head > 0 && c->d_latent > 0 &&
           c->max_context > 0 && (c->dtype == KVC_BF16 || c->dtype == KVC_FP16 || c->dtype == KVC_FP32 ||
                                  c->dtype == KVC_INT8);
}

const kvc::MlaKernelInfo *find_mla(const kvc_mla_config *c) {
    if (c->d_head % 16 != 0 || c->d_head < 16 || c->d_head > 256) return nullptr;
    // 8 or 16 heads: one kernel instance; 32 to 128 heads (a multiple of 16):
    // the 16-head kernel over head groups
    const int Hk = c->n_heads <= 16 ? c->n_heads : (c->n_heads % 16 == 0 && c->n_heads <= 128 ? 16 : 0);
    if (c->dtype == KVC_BF16) return kvc::mla_kernel_bf16(c->d_latent, Hk);
    if (c->dtype == KVC_FP16) return kvc::mla_kernel_f16(c->d_latent, Hk);
    return nullptr;
}

struct MlaLayout {
    uint64_t qt, ml, acc, total;
};

MlaLayout mla_layout(const kvc_mla_config *c) {
    const uint64_t slots = uint64_t(kvc::MLA_MAX_CTAS) + uint64_t(c->batch);
    MlaLayout l;
    l.qt = 256;
    l.ml = round256(l.qt + uint64_t(c->batch) * c->n_heads * c->d_latent * 2);
    l.acc = round256(l.ml + slots * c->n_heads * 2 * 4);
    l.total = round256(l.acc + slots * c->n_heads * uint64_t(c->d_latent) * 4);
    return l;
}

uint64_t layer_slab(const kvc_mla_cache *h) {
    const kvc_mla_config &c = h->cfg;
    return uint64_t(c.batch) * uint64_t(c.max_context) * c.d_latent * 2;
}

// The whole latent cache as [L*B][max_ctx][d_c]: boxes of 64 columns x rows.
bool encode_latent_map(const kvc_mla_config *c, void *base, uint32_t rows, CUtensorMap *out) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!encode) return false;
    const CUtensorMapDataType dt =
        c->dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[3] = {cuuint64_t(c->d_latent), cuuint64_t(c->max_context),
                                cuuint64_t(c->n_layers) * cuuint64_t(c->batch)};
    const cuuint64_t strides[2] = {cuuint64_t(c->d_latent) * 2, cuuint64_t(c->max_context) * c->d_latent * 2};
    const cuuint32_t box[3] = {64, rows, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    return encode(out, dt, 3, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

kvc_status mla_launch(kvc_mla_cache *h, int32_t layer, const void *q, const void *c_new, const void *w_uk,
                      const void *w_uv, const int32_t *valid_len, int32_t hint, void *out, void *stream) {
    if (!h || layer < 0 || layer >= h->cfg.n_layers || !q || !w_uk || !w_uv || !valid_len || !out)
        return KVC_ERR_INVALID;
    if (hint < 0 || hint > h->cfg.max_context) return KVC_ERR_INVALID;
    if (!aligned16(q) || !aligned16(w_uk) || !aligned16(w_uv) || (c_new && !aligned16(c_new)))
        return KVC_ERR_ALIGNMENT;
    const kvc_mla_config &c = h->cfg;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *slab = h->c_base + layer_slab(h) * layer;
    int32_t *err = reinterpret_cast<int32_t *>(h->ws);

    // 1. absorbed queries (and the step's latent row)
    kvc::MlaAbsorbArgs ab;
    ab.q = q;
    ab.w_uk = w_uk;
    ab.qt = h->ws + h->off_qt;
    ab.c_new = c_new;
    ab.cache = slab;
    ab.valid_len = valid_len;
    ab.err = err;
    ab.B = c.batch;
    ab.H = c.n_heads;
    ab.d_h = c.d_head;
    ab.d_c = c.d_latent;
    ab.max_ctx = c.max_context;
    ab.scale = float(1.4426950408889634 / std::sqrt(double(c.d_head)));
    if (h->info->absorb(ab, s) != cudaSuccess) return KVC_ERR_CUDA;

    // 2. attention over the latents: the same even split of the flattened
    // rows as the GQA decode, at most one CTA per SM
    // Head groups of one split run side by side: nsplit splits x groups CTAs.
    const int groups = c.n_heads > 16 ? c.n_heads / 16 : 1;
    int64_t grid = h->num_splits;
    if (grid == 0) {
        const int64_t upper = int64_t(c.batch) * (hint > 0 ? hint : c.max_context);
        grid = (upper + 4 * 64 - 1) / (4 * 64);
        if (grid > h->num_sms / groups) grid = h->num_sms / groups;
    }
    if (grid > kvc::MLA_MAX_CTAS) grid = kvc::MLA_MAX_CTAS;
    if (grid < 1) grid = 1;
    kvc::MlaArgs a;
    a.H_all = c.n_heads;
    a.groups = groups;
    a.B = c.batch;
    a.H_kv = 1;
    a.max_ctx = c.max_context;
    a.gran = 1;
    a.err = err;
    a.valid_len = valid_len;
    a.qt = h->ws + h->off_qt;
    a.part_ml = reinterpret_cast<float *>(h->ws + h->off_ml);
    a.part_acc = reinterpret_cast<float *>(h->ws + h->off_acc);
    a.n_stages = h->n_stages;
    a.seg_base = layer * c.batch;
    a.timeout_ns = kvc::WAIT_TIMEOUT_NS;
    a.tm64 = h->tm64;
    a.tm16 = h->tm16;
    if (h->info->launch(a, int(grid * groups), h->smem_bytes, s) != cudaSuccess) return KVC_ERR_CUDA;

    // 3. fold the splits, apply W_UV
    kvc::MlaCombineArgs cb;
    cb.part_ml = a.part_ml;
    cb.part_acc = a.part_acc;
    cb.valid_len = valid_len;
    cb.w_uv = w_uv;
    cb.out = out;
    cb.B = c.batch;
    cb.H = c.n_heads;
    cb.d_h = c.d_head;
    cb.d_c = c.d_latent;
    cb.max_ctx = c.max_context;
    cb.grid = int(grid);
    if (h->info->combine(cb, s) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

}  // namespace

extern "C" {

uint64_t kvc_mla_cache_bytes(const kvc_mla_config *cfg) {
    if (!mla_shape_ok(cfg)) return 0;
    const int eb = cfg->dtype == KVC_FP32 ? 4 : cfg->dtype == KVC_INT8 ? 1 : 2;
    return uint64_t(cfg->n_layers) * uint64_t(cfg->d_latent) * uint64_t(cfg->max_context) * uint64_t(cfg->batch) *
           uint64_t(eb);
}

uint64_t kvc_mla_workspace_bytes(const kvc_mla_config *cfg) {
    if (!mla_shape_ok(cfg)) return 0;
    return mla_layout(cfg).total;
}

kvc_status kvc_mla_alloc(const kvc_mla_config *cfg, void *c_base, void *workspace, uint64_t ws_bytes,
                         kvc_mla_cache **out) {
    if (!out) return KVC_ERR_INVALID;
    *out = nullptr;
    if (!mla_shape_ok(cfg) || !c_base) return KVC_ERR_INVALID;
    const kvc::MlaKernelInfo *info = find_mla(cfg);
    if (!info) return KVC_ERR_UNSUPPORTED;
    if (!aligned16(c_base)) return KVC_ERR_ALIGNMENT;
    const MlaLayout l = mla_layout(cfg);
    if (!workspace || ws_bytes < l.total) return KVC_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVC_ERR_ALIGNMENT;
    int dev = 0, sms = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return KVC_ERR_CUDA;
    const int budget = optin < kvc::SMEM_BUDGET ? optin : kvc::SMEM_BUDGET;
    int ns = (budget - info->fixed_smem) / info->stage_bytes;
    if (ns > 16) ns = 16;
    if (ns < info->min_stages) return KVC_ERR_UNSUPPORTED;
    // the error word starts at 0 (nothing else in the workspace is read before it is written)
    if (cudaMemsetAsync(workspace, 0, 256, 0) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaStreamSynchronize(0) != cudaSuccess) return KVC_ERR_CUDA;
    kvc_mla_cache *h = new (std::nothrow) kvc_mla_cache;
    if (!h) return KVC_ERR_CUDA;
    h->cfg = *cfg;
    h->info = info;
    h->c_base = static_cast<uint8_t *>(c_base);
    h->ws = static_cast<uint8_t *>(workspace);
    h->ws_bytes = ws_bytes;
    h->off_qt = l.qt;
    h->off_ml = l.ml;
    h->off_acc = l.acc;
    h->num_sms = sms;
    h->n_stages = ns;
    h->smem_bytes = info->fixed_smem + ns * info->stage_bytes;
    h->num_splits = 0;
    if (!encode_latent_map(cfg, c_base, 64, &h->tm64) || !encode_latent_map(cfg, c_base, 16, &h->tm16) ||
        info->set_max_smem(h->smem_bytes) != cudaSuccess) {
        delete h;
        return KVC_ERR_CUDA;
    }
    *out = h;
    return KVC_OK;
}

void kvc_mla_free(kvc_mla_cache *h) { delete h; }

kvc_status kvc_mla_set_num_splits(kvc_mla_cache *h, int32_t n) {
    if (!h || n < 0 || n > kvc::MLA_MAX_CTAS) return KVC_ERR_INVALID;
    h->num_splits = n;
    return KVC_OK;
}

kvc_status kvc_mla_append(kvc_mla_cache *h, int32_t layer, const void *c_new, const int32_t *cache_index,
                          int32_t T_new, void *stream) {
    if (!h || layer < 0 || layer >= h->cfg.n_layers || T_new < 0) return KVC_ERR_INVALID;
    if (T_new == 0) return KVC_OK;
    if (!c_new || !cache_index) return KVC_ERR_INVALID;
    if (T_new > h->cfg.max_context) return KVC_ERR_CAPACITY;
    if (!aligned16(c_new)) return KVC_ERR_ALIGNMENT;
    const cudaError_t e = kvc::launch_append(h->c_base + layer_slab(h) * layer, nullptr,
                                             static_cast<const uint8_t *>(c_new), nullptr, cache_index, 0,
                                             h->cfg.batch, 1, T_new, h->cfg.max_context, h->cfg.d_latent * 2,
                                             reinterpret_cast<int32_t *>(h->ws), h->num_sms,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status kvc_mla_decode_attn(kvc_mla_cache *h, int32_t layer, const void *q, const void *w_uk, const void *w_uv,
                               const int32_t *valid_len, int32_t max_valid_hint, void *out, void *stream) {
    return mla_launch(h, layer, q, nullptr, w_uk, w_uv, valid_len, max_valid_hint, out, stream);
}

kvc_status kvc_mla_decode_step(kvc_mla_cache *h, int32_t layer, const void *q, const void *c_new,
                               const void *w_uk, const void *w_uv, const int32_t *valid_len,
                               int32_t max_valid_hint, void *out, void *stream) {
    if (!c_new) return KVC_ERR_INVALID;
    return mla_launch(h, layer, q, c_new, w_uk, w_uv, valid_len, max_valid_hint, out, stream);
}

kvc_status kvc_mla_get_error(kvc_mla_cache *h, void *stream) {
    if (!h) return KVC_ERR_INVALID;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, h->ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return KVC_ERR_CUDA;
    if (word != 0 && cudaMemset(h->ws, 0, sizeof word) != cudaSuccess) return KVC_ERR_CUDA;
    return static_cast<kvc_status>(word);
}

}  // extern "C"
