// kvc_api.cu -- host side of libkvc.so: argument checks, launch planning and
// the extern "C" entry points declared in include/kvc.h.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>

#include "../../include/kvc.h"
#include "kvc_internal.cuh"

struct kvc_cache {
    kvc_config cfg;
    int device;
    int num_sms;
    int max_smem;            // opt-in dynamic shared memory per block
    int elem_bytes;
    int group;               // n_heads / n_kv_heads
    int num_splits;          // 0: automatic
    uint64_t flag_timeout_ns;  // limit of the split combine's wait for the other splits
    uint8_t *k_base;
    uint8_t *v_base;
    uint8_t *k_scale;        // int8 caches: per-row fp32 scales [L, B, H_kv, T_max]; else null
    uint8_t *v_scale;
    const int32_t *block_table;  // paged caches: [B, max_blocks]; else null
    int32_t num_blocks;          // paged: physical blocks per layer pool
    int32_t kv_pair;             // paged: KV heads read per tile (1, or 2 with the pair kernel)
    uint8_t *ws;
    uint64_t ws_bytes;
    kvc::WorkspaceLayout wl;
    const kvc::DecodeKernelInfo *decode;
    const kvc::PrefillKernelInfo *prefill;  // nullptr where chunked prefill is not built
    int n_stages;
    int smem_bytes;
    CUtensorMap tm_k32, tm_k8, tm_v32, tm_v8;  // used by kernels with info->tensor_maps
    CUtensorMap pf_k32, pf_k8, pf_v32, pf_v8;  // the chunked prefill's (64-column blocks)
    CUtensorMap pf_k128, pf_v128;             // and its whole-tile boxes (128 rows)
    CUtensorMap rb_k64, rb_v64, rb_k32, rb_v32;  // kernels with info->ragged_maps: 64- and 32-row boxes
};

namespace {

int elem_bytes_of(int32_t dtype) {
    switch (dtype) {
        case KVC_BF16: return 2;
        case KVC_FP16: return 2;
        case KVC_FP32: return 4;
        case KVC_INT8: return 1;
        default: return 0;
    }
}

bool shape_ok(const kvc_config *c) {
    return c && c->n_layers > 0 && c->batch > 0 && c->n_heads > 0 && c->n_kv_heads > 0 &&
           c->d_head > 0 && c->max_context > 0 && c->n_heads % c->n_kv_heads == 0 &&
           elem_bytes_of(c->dtype) > 0;
}

// Kernel for a contiguous cache bound to a handle: 16- and 32-head groups of
// 16-bit caches at d_h = 128 take the tcgen05 kernel, which reads its tiles
// through the handle's 128-row tensor maps; the rest the kernel table.
const kvc::DecodeKernelInfo *find_decode(const kvc_config *c) {
    const int G = c->n_heads / c->n_kv_heads;
    if (c->d_head == 128 && (G == 16 || G == 32)) {
        if (c->dtype == KVC_BF16) return kvc::decode_kernel_tc_bf16_128(G);
        if (c->dtype == KVC_FP16) return kvc::decode_kernel_tc_f16_128(G);
    }
    return kvc::find_decode_kernel(c->dtype, c->d_head, G);
}

// Paged pools with 2 or 4 query heads per KV head and an even number of KV
// heads (16-bit, d_h 64 or 128) are read two KV heads per tile: a block
// stores the heads' rows one after another, so one box brings both.
bool paged_pair_ok(const kvc_config *c) {
    const int G = c->n_heads / c->n_kv_heads;
    return (c->dtype == KVC_BF16 || c->dtype == KVC_FP16) && (c->d_head == 64 || c->d_head == 128) &&
           (G == 2 || G == 4) && c->n_kv_heads % 2 == 0;
}

// Kernel for a paged pool: the tensor-core kernel (16-bit, 2 to 8 query heads
// per KV head, or 16, 32, 64); the pair kernel where paged_pair_ok holds;
// else for d_h = 128 the variant whose consumers read the half-row tile
// layout the paged producer writes, for d_h = 64 the contiguous cache's
// kernel (the layouts coincide).  Null otherwise.
const kvc::DecodeKernelInfo *find_decode_paged(const kvc_config *c) {
    const int G = c->n_heads / c->n_kv_heads;
    if (paged_pair_ok(c)) {
        const bool bf = c->dtype == KVC_BF16;
        if (c->d_head == 128) return bf ? kvc::decode_kernel_pair_bf16_128(2 * G) : kvc::decode_kernel_pair_f16_128(2 * G);
        return bf ? kvc::decode_kernel_pair_bf16_64(2 * G) : kvc::decode_kernel_pair_f16_64(2 * G);
    }
    if (G < 2 || (G > 8 && G != 16 && G != 32 && G != 64)) return nullptr;
    if (c->d_head == 128) {
        if (c->dtype == KVC_BF16) return kvc::decode_kernel_paged_bf16_128(G);
        if (c->dtype == KVC_FP16) return kvc::decode_kernel_paged_f16_128(G);
        return nullptr;
    }
    if (c->d_head == 64 && (c->dtype == KVC_BF16 || c->dtype == KVC_FP16)) return find_decode(c);
    return nullptr;
}

// Chunked-prefill kernel: 16-bit caches with d_h 64 or 128.
const kvc::PrefillKernelInfo *find_prefill(const kvc_config *c) {
    const int G = c->n_heads / c->n_kv_heads;
    const int D = c->d_head;
    if (c->dtype == KVC_BF16) {
        if (D == 64) return kvc::prefill_kernel_bf16_64(G);
        if (D == 128) return kvc::prefill_kernel_bf16_128(G);
    } else if (c->dtype == KVC_FP16) {
        if (D == 64) return kvc::prefill_kernel_f16_64(G);
        if (D == 128) return kvc::prefill_kernel_f16_128(G);
    }
    return nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t layer_scale_bytes(const kvc_cache *h) {
    const kvc_config &c = h->cfg;
    return uint64_t(c.batch) * c.n_kv_heads * uint64_t(c.max_context) * 4;
}

uint64_t layer_slab_bytes(const kvc_cache *h) {
    const kvc_config &c = h->cfg;
    if (h->block_table)  // paged: one pool of num_blocks blocks of 16 rows per KV head
        return uint64_t(h->num_blocks) * c.n_kv_heads * 16ull * c.d_head * h->elem_bytes;
    return uint64_t(c.batch) * c.n_kv_heads * uint64_t(c.max_context) * c.d_head * h->elem_bytes;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

const kvc::DecodeKernelInfo *kvc::find_decode_kernel(int32_t dtype, int D, int G) {
#define KVC_PICK(TAG, DD) \
    if (D == DD) return kvc::decode_kernel_##TAG##_##DD(G);
    switch (dtype) {
        case KVC_BF16:
            KVC_PICK(bf16, 32) KVC_PICK(bf16, 64) KVC_PICK(bf16, 128) KVC_PICK(bf16, 256) break;
        case KVC_FP16:
            KVC_PICK(f16, 32) KVC_PICK(f16, 64) KVC_PICK(f16, 128) KVC_PICK(f16, 256) break;
        case KVC_FP32:
            KVC_PICK(f32, 32) KVC_PICK(f32, 64) KVC_PICK(f32, 128) KVC_PICK(f32, 256) break;
        case KVC_INT8:
            KVC_PICK(q8, 128) break;
        default: break;
    }
#undef KVC_PICK
    return nullptr;
}

int kvc::decode_stage_count(const DecodeKernelInfo *info, int smem_optin) {
    const int budget = smem_optin < SMEM_BUDGET ? smem_optin : SMEM_BUDGET;
    int n = (budget - info->fixed_smem) / info->stage_bytes;
    if (n > 32) n = 32;
    return n < info->consumer_warps + 1 ? 0 : n;
}

int kvc::decode_grid(const DecodeKernelInfo *info, int B, int H_kv, int D, int elem_bytes, int max_ctx,
                     int max_valid_hint, int num_sms, int forced) {
    // Splits: every SM streams an equal share of the live rows; small
    // problems use fewer CTAs so that each still gets several tiles.  When
    // the problem is small and every segment (sequence, KV head) holds at
    // most 64 KB per tensor, one CTA per segment: the step is latency there,
    // and a CTA that owns a whole segment needs no split combine.
    int64_t want = forced;
    if (want == 0) {
        const int64_t seg_rows = max_valid_hint > 0 ? max_valid_hint : max_ctx;
        const int64_t segs = int64_t(B) * H_kv;
        const int64_t min_rows = 4 * int64_t(info->tile_rows);
        want = (segs * seg_rows + min_rows - 1) / min_rows;
        if (want < num_sms && segs <= num_sms && seg_rows * D * elem_bytes <= 65536) want = segs;
        if (want > num_sms) want = num_sms;
        if (want < 1) want = 1;
    }
    if (want > MAX_CTAS) want = MAX_CTAS;
    return int(want);
}

bool kvc::encode_cache_maps(int32_t dtype, int D, int max_ctx, int64_t n_segs, const void *k_base,
                            const void *v_base, CUtensorMap *k32, CUtensorMap *k8, CUtensorMap *v32,
                            CUtensorMap *v8, bool tile_box) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    // 16-bit caches: boxes of 64 elements (128 bytes) per row; int8 codes:
    // 128 elements (128 bytes).
    const bool q8 = dtype == KVC_INT8;
    const int eb = q8 ? 1 : 2;
    const CUtensorMapDataType dt = q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                      : dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (tile_box && (q8 || D % 64 != 0)) return false;
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(max_ctx), cuuint64_t(n_segs)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * eb, cuuint64_t(max_ctx) * D * eb};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    struct Job { const void *base; cuuint32_t rows; CUtensorMap *out; };
    // the larger box covers a whole decode tile (int8: 128 rows; 16-bit: 32)
    const cuuint32_t r32 = q8 ? 128 : 32;
    if (tile_box) {
        // (64 columns, rows, column blocks, segments); a block is 128 bytes
        // further along the row, so the box lands block after block
        const cuuint64_t dims4[4] = {64, cuuint64_t(max_ctx), cuuint64_t(D / 64), cuuint64_t(n_segs)};
        const cuuint64_t strides4[3] = {cuuint64_t(D) * eb, 128, cuuint64_t(max_ctx) * D * eb};
        const cuuint32_t box4[4] = {64, 32, cuuint32_t(D / 64), 1};
        const Job tiles[2] = {{k_base, 32, k32}, {v_base, 32, v32}};
        for (const Job &j : tiles)
            if (encode(j.out, dt, 4, const_cast<void *>(j.base), dims4, strides4, box4, elem,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
    }
    const Job jobs[4] = {{k_base, r32, k32}, {k_base, 8, k8}, {v_base, r32, v32}, {v_base, 8, v8}};
    for (const Job &j : jobs) {
        if (tile_box && j.rows != 8) continue;  // encoded above
        const cuuint32_t box[3] = {cuuint32_t(128 / eb), j.rows, 1};
        if (encode(j.out, dt, 3, const_cast<void *>(j.base), dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool kvc::encode_row_box_maps(int32_t dtype, int D, int max_ctx, int64_t n_segs, const void *k_base,
                              const void *v_base, int rows, CUtensorMap *k, CUtensorMap *v) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode || (dtype != KVC_BF16 && dtype != KVC_FP16 && dtype != KVC_INT8) || rows < 1 || rows > 256)
        return false;
    // 128 bytes of a row per box: 64 16-bit elements or 128 int8 codes
    const int eb = dtype == KVC_INT8 ? 1 : 2;
    const CUtensorMapDataType dt = dtype == KVC_INT8   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(max_ctx), cuuint64_t(n_segs)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * eb, cuuint64_t(max_ctx) * D * eb};
    const cuuint32_t box[3] = {cuuint32_t(128 / eb), cuuint32_t(rows), 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    const void *bases[2] = {k_base, v_base};
    CUtensorMap *outs[2] = {k, v};
    for (int i = 0; i < 2; ++i)
        if (encode(outs[i], dt, 3, const_cast<void *>(bases[i]), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    return true;
}

bool kvc::encode_pool_maps(int32_t dtype, int D, int64_t n_blocks_total, const void *k_pool, const void *v_pool,
                           CUtensorMap *k16, CUtensorMap *k8, CUtensorMap *v16, CUtensorMap *v8) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode || (dtype != KVC_BF16 && dtype != KVC_FP16)) return false;
    const CUtensorMapDataType dt = dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // each block of one KV head (16 rows of D elements) viewed as HR rows of
    // 128 bytes: a box of 64 columns x HR covers the whole block with one copy
    const cuuint32_t HR = cuuint32_t(16 * (D / 64));
    const cuuint64_t dims[3] = {64, HR, cuuint64_t(n_blocks_total)};
    const cuuint64_t strides[2] = {128, cuuint64_t(HR) * 128};
    const cuuint32_t elem[3] = {1, 1, 1};
    struct Job { const void *base; cuuint32_t rows; CUtensorMap *out; };
    const Job jobs[4] = {{k_pool, HR, k16}, {k_pool, HR / 2, k8}, {v_pool, HR, v16}, {v_pool, HR / 2, v8}};
    for (const Job &j : jobs) {
        const cuuint32_t box[3] = {64, j.rows, 1};
        if (encode(j.out, dt, 3, const_cast<void *>(j.base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool kvc::encode_pool_pair_maps(int32_t dtype, int D, int H_kv, int64_t blocks_total, const void *k_pool,
                                const void *v_pool, CUtensorMap *k16, CUtensorMap *k8, CUtensorMap *v16,
                                CUtensorMap *v8) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode || (dtype != KVC_BF16 && dtype != KVC_FP16) || D % 64 != 0 || H_kv < 2) return false;
    const CUtensorMapDataType dt = dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t row = cuuint64_t(D) * 2;  // bytes of one row
    // (64 columns, 16 rows, column blocks, heads, blocks): a column block is
    // 128 bytes further along the row, so a box lands block after block
    const cuuint64_t dims[5] = {64, 16, cuuint64_t(D / 64), cuuint64_t(H_kv), cuuint64_t(blocks_total)};
    const cuuint64_t strides[4] = {row, 128, 16 * row, cuuint64_t(H_kv) * 16 * row};
    const cuuint32_t elem[5] = {1, 1, 1, 1, 1};
    const cuuint32_t pair_box[5] = {64, 16, cuuint32_t(D / 64), 2, 1};
    const cuuint32_t half_box[5] = {64, 8, 1, 1, 1};
    struct Job { const void *base; const cuuint32_t *box; CUtensorMap *out; };
    const Job jobs[4] = {{k_pool, pair_box, k16}, {k_pool, half_box, k8}, {v_pool, pair_box, v16}, {v_pool, half_box, v8}};
    for (const Job &j : jobs) {
        if (encode(j.out, dt, 5, const_cast<void *>(j.base), dims, strides, j.box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

extern "C" {

int32_t kvc_abi_version(void) { return KVC_ABI_VERSION; }

const char *kvc_status_str(int32_t s) {
    switch (s) {
        case KVC_OK: return "ok";
        case KVC_ERR_INVALID: return "invalid argument";
        case KVC_ERR_CAPACITY: return "append would pass max_context";
        case KVC_ERR_CUDA: return "CUDA runtime error";
        case KVC_ERR_WORKSPACE: return "workspace missing or too small";
        case KVC_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
        case KVC_ERR_DEVICE_INDEX: return "device-resident cache_index or valid_len out of range";
        case KVC_ERR_UNSUPPORTED: return "configuration not supported by the compiled kernels";
        case KVC_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        default: return "unknown status";
    }
}

kvc_status kvc_check_config(const kvc_config *cfg) {
    if (!shape_ok(cfg)) return KVC_ERR_INVALID;
    if (!find_decode(cfg)) return KVC_ERR_UNSUPPORTED;
    return KVC_OK;
}

uint64_t kvc_cache_bytes(const kvc_config *c) {
    if (!shape_ok(c)) return 0;
    return 2ull * uint64_t(c->n_layers) * uint64_t(c->n_kv_heads) * uint64_t(c->d_head) *
           uint64_t(c->max_context) * uint64_t(c->batch) * uint64_t(elem_bytes_of(c->dtype));
}

uint64_t kvc_bytes_per_token(const kvc_config *c) {
    if (!shape_ok(c)) return 0;
    return 2ull * uint64_t(c->n_layers) * uint64_t(c->n_kv_heads) * uint64_t(c->d_head) *
           uint64_t(elem_bytes_of(c->dtype));
}

uint64_t kvc_workspace_bytes(const kvc_config *c) {
    if (!shape_ok(c)) return 0;
    const int G = c->n_heads / c->n_kv_heads;
    const uint64_t one = kvc::workspace_layout(c->batch, c->n_kv_heads, G, c->d_head).total;
    // a paged pool read two KV heads per tile: half the segments, twice the heads each
    const uint64_t pair =
        paged_pair_ok(c) ? kvc::workspace_layout(c->batch, c->n_kv_heads / 2, 2 * G, c->d_head).total : 0;
    return one > pair ? one : pair;
}

uint64_t kvc_scale_bytes(const kvc_config *c) {
    if (!shape_ok(c) || c->dtype != KVC_INT8) return 0;
    return uint64_t(c->n_layers) * uint64_t(c->batch) * uint64_t(c->n_kv_heads) * uint64_t(c->max_context) * 4;
}

}  // extern "C"

namespace {

kvc_status alloc_impl(const kvc_config *cfg, void *k_base, void *v_base, void *k_scale, void *v_scale,
                      void *workspace, uint64_t ws_bytes, kvc_cache **out, const int32_t *block_table = nullptr,
                      int32_t num_blocks = 0) {
    if (!out || !shape_ok(cfg) || !k_base || !v_base) return KVC_ERR_INVALID;
    if (k_scale && (!aligned16(k_scale) || !aligned16(v_scale))) return KVC_ERR_ALIGNMENT;
    const kvc::DecodeKernelInfo *info = block_table ? find_decode_paged(cfg) : find_decode(cfg);
    if (!info) return KVC_ERR_UNSUPPORTED;
    // the 128- and 32-row maps are encoded with the chunked prefill's
    const kvc::PrefillKernelInfo *pinfo = block_table ? nullptr : find_prefill(cfg);
    if (info->row_box_maps && !pinfo) info = kvc::find_decode_kernel(cfg->dtype, cfg->d_head, cfg->n_heads / cfg->n_kv_heads);
    if (!info) return KVC_ERR_UNSUPPORTED;
    if (!aligned16(k_base) || !aligned16(v_base) || (workspace && !aligned16(workspace)))
        return KVC_ERR_ALIGNMENT;
    const uint64_t need = kvc_workspace_bytes(cfg);
    if (!workspace || ws_bytes < need) return KVC_ERR_WORKSPACE;

    int dev = 0, sms = 0, smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVC_ERR_CUDA;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return KVC_ERR_CUDA;

    // As many pipeline stages as shared memory holds (at most 32), but at
    // least one more than there are consumer warps.
    const int n_stages = kvc::decode_stage_count(info, smem);
    if (n_stages == 0) return KVC_ERR_UNSUPPORTED;
    const int smem_bytes = info->fixed_smem + n_stages * info->stage_bytes;
    if (info->set_max_smem(smem_bytes) != cudaSuccess) return KVC_ERR_CUDA;
    if (pinfo && pinfo->set_max_smem(pinfo->smem) != cudaSuccess) return KVC_ERR_CUDA;

    // Zero the workspace: error word and per-segment counters start at 0.
    if (cudaMemsetAsync(workspace, 0, need, 0) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaStreamSynchronize(0) != cudaSuccess) return KVC_ERR_CUDA;

    kvc_cache *h = new (std::nothrow) kvc_cache;
    if (!h) return KVC_ERR_INVALID;
    h->cfg = *cfg;
    h->device = dev;
    h->num_sms = sms;
    h->max_smem = smem;
    h->elem_bytes = elem_bytes_of(cfg->dtype);
    h->group = cfg->n_heads / cfg->n_kv_heads;
    h->num_splits = 0;
    h->flag_timeout_ns = kvc::WAIT_TIMEOUT_NS;
    h->k_base = static_cast<uint8_t *>(k_base);
    h->v_base = static_cast<uint8_t *>(v_base);
    h->k_scale = static_cast<uint8_t *>(k_scale);
    h->v_scale = static_cast<uint8_t *>(v_scale);
    h->block_table = block_table;
    h->num_blocks = num_blocks;
    h->kv_pair = block_table && paged_pair_ok(cfg) ? 2 : 1;
    h->ws = static_cast<uint8_t *>(workspace);
    h->ws_bytes = ws_bytes;
    h->wl = kvc::workspace_layout(cfg->batch, cfg->n_kv_heads / h->kv_pair, h->group * h->kv_pair, cfg->d_head);
    h->decode = info;
    h->prefill = pinfo;
    h->n_stages = n_stages;
    h->smem_bytes = smem_bytes;
    if (block_table) {
        h->prefill = nullptr;  // chunked prefill reads contiguous caches only
        const bool maps_ok =
            h->kv_pair == 2
                ? kvc::encode_pool_pair_maps(cfg->dtype, cfg->d_head, cfg->n_kv_heads,
                                             int64_t(cfg->n_layers) * num_blocks, k_base, v_base, &h->tm_k32,
                                             &h->tm_k8, &h->tm_v32, &h->tm_v8)
                : kvc::encode_pool_maps(cfg->dtype, cfg->d_head, int64_t(cfg->n_layers) * num_blocks * cfg->n_kv_heads,
                                        k_base, v_base, &h->tm_k32, &h->tm_k8, &h->tm_v32, &h->tm_v8);
        if (!maps_ok) {
            delete h;
            return KVC_ERR_CUDA;
        }
    } else {
        const int64_t n_segs = int64_t(cfg->n_layers) * cfg->batch * cfg->n_kv_heads;
        if ((info->tensor_maps || pinfo) &&
            !kvc::encode_cache_maps(cfg->dtype, cfg->d_head, cfg->max_context, n_segs, k_base, v_base,
                                    &h->tm_k32, &h->tm_k8, &h->tm_v32, &h->tm_v8, info->tile_box)) {
            delete h;
            return KVC_ERR_CUDA;
        }
        h->pf_k32 = h->tm_k32;
        h->pf_k8 = h->tm_k8;
        h->pf_v32 = h->tm_v32;
        h->pf_v8 = h->tm_v8;
        if (pinfo && info->tile_box &&
            !kvc::encode_cache_maps(cfg->dtype, cfg->d_head, cfg->max_context, n_segs, k_base, v_base,
                                    &h->pf_k32, &h->pf_k8, &h->pf_v32, &h->pf_v8)) {
            delete h;
            return KVC_ERR_CUDA;
        }
        if (pinfo && !kvc::encode_row_box_maps(cfg->dtype, cfg->d_head, cfg->max_context, n_segs, k_base, v_base,
                                               128, &h->pf_k128, &h->pf_v128)) {
            delete h;
            return KVC_ERR_CUDA;
        }
        if (info->ragged_maps &&
            (!kvc::encode_row_box_maps(cfg->dtype, cfg->d_head, cfg->max_context, n_segs, k_base, v_base, 64,
                                       &h->rb_k64, &h->rb_v64) ||
             !kvc::encode_row_box_maps(cfg->dtype, cfg->d_head, cfg->max_context, n_segs, k_base, v_base, 32,
                                       &h->rb_k32, &h->rb_v32))) {
            delete h;
            return KVC_ERR_CUDA;
        }
    }
    *out = h;
    return KVC_OK;
}

}  // namespace

extern "C" {

kvc_status kvc_alloc(const kvc_config *cfg, void *k_base, void *v_base, void *workspace,
                     uint64_t ws_bytes, kvc_cache **out) {
    if (cfg && cfg->dtype == KVC_INT8) return KVC_ERR_INVALID;  // needs its scale arrays
    return alloc_impl(cfg, k_base, v_base, nullptr, nullptr, workspace, ws_bytes, out);
}

kvc_status kvc_alloc_scaled(const kvc_config *cfg, void *k_base, void *v_base, void *k_scale, void *v_scale,
                            void *workspace, uint64_t ws_bytes, kvc_cache **out) {
    if (!cfg || cfg->dtype != KVC_INT8 || !k_scale || !v_scale) return KVC_ERR_INVALID;
    return alloc_impl(cfg, k_base, v_base, k_scale, v_scale, workspace, ws_bytes, out);
}

uint64_t kvc_pool_bytes(const kvc_config *cfg, int32_t num_blocks) {
    if (!shape_ok(cfg) || num_blocks <= 0 || cfg->dtype == KVC_INT8) return 0;
    return uint64_t(cfg->n_layers) * uint64_t(num_blocks) * uint64_t(cfg->n_kv_heads) * 16ull *
           uint64_t(cfg->d_head) * uint64_t(elem_bytes_of(cfg->dtype));
}

kvc_status kvc_alloc_paged(const kvc_config *cfg, void *k_pool, void *v_pool, int32_t num_blocks,
                           const int32_t *block_table, void *workspace, uint64_t ws_bytes, kvc_cache **out) {
    if (!cfg || !block_table || num_blocks <= 0 || cfg->max_context % 16 != 0) return KVC_ERR_INVALID;
    if (cfg->dtype == KVC_INT8) return KVC_ERR_UNSUPPORTED;
    if (shape_ok(cfg) && !find_decode_paged(cfg)) return KVC_ERR_UNSUPPORTED;  // the paged producer is the TMA kernel's
    if (!aligned16(block_table)) return KVC_ERR_ALIGNMENT;
    return alloc_impl(cfg, k_pool, v_pool, nullptr, nullptr, workspace, ws_bytes, out, block_table, num_blocks);
}

void kvc_free(kvc_cache *h) { delete h; }

kvc_status kvc_set_num_splits(kvc_cache *h, int32_t n) {
    if (!h || n < 0 || n > kvc::MAX_CTAS) return KVC_ERR_INVALID;
    h->num_splits = n;
    return KVC_OK;
}

kvc_status kvc_set_wait_timeout_ns(kvc_cache *h, uint64_t ns) {
    if (!h) return KVC_ERR_INVALID;
    h->flag_timeout_ns = ns == 0 ? kvc::WAIT_TIMEOUT_NS : ns;
    return KVC_OK;
}

kvc_status kvc_append(kvc_cache *h, int32_t layer, const void *k_new, const void *v_new,
                      const int32_t *cache_index, int32_t T_new, void *stream) {
    if (!h || layer < 0 || layer >= h->cfg.n_layers || T_new < 0) return KVC_ERR_INVALID;
    if (T_new == 0) return KVC_OK;
    if (!k_new || !v_new || !cache_index) return KVC_ERR_INVALID;
    if (T_new > h->cfg.max_context) return KVC_ERR_CAPACITY;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVC_ERR_ALIGNMENT;
    const uint64_t slab = layer_slab_bytes(h);
    if (h->cfg.dtype == KVC_INT8) {
        const uint64_t ss = layer_scale_bytes(h);
        const cudaError_t e = kvc::launch_append_q8(
            h->k_base + slab * layer, h->v_base + slab * layer, reinterpret_cast<float *>(h->k_scale + ss * layer),
            reinterpret_cast<float *>(h->v_scale + ss * layer), static_cast<const uint8_t *>(k_new),
            static_cast<const uint8_t *>(v_new), cache_index, 0, h->cfg.batch, h->cfg.n_kv_heads, T_new,
            h->cfg.max_context, h->cfg.d_head, reinterpret_cast<int32_t *>(h->ws), h->num_sms,
            static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
    }
    const cudaError_t e = kvc::launch_append(
        h->k_base + slab * layer, h->v_base + slab * layer, static_cast<const uint8_t *>(k_new),
        static_cast<const uint8_t *>(v_new), cache_index, 0, h->cfg.batch, h->cfg.n_kv_heads, T_new,
        h->cfg.max_context, h->cfg.d_head * h->elem_bytes, reinterpret_cast<int32_t *>(h->ws),
        h->num_sms, static_cast<cudaStream_t>(stream), h->block_table, h->cfg.max_context / 16, h->num_blocks);
    return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // extern "C"

namespace {

// Launch the decode kernel of one layer; k_new / v_new non-null make it the
// fused step.  Arguments are already validated.
kvc_status launch_decode(kvc_cache *h, int32_t layer, const void *q, const int32_t *valid_len,
                         int32_t max_valid_hint, void *out, void *stream, const void *k_new,
                         const void *v_new) {
    const kvc_config &c = h->cfg;

    // a pair kernel's segment is (sequence, KV-head pair): half the segments, twice the row bytes
    const int kp = h->kv_pair;
    const int grid = kvc::decode_grid(h->decode, c.batch, c.n_kv_heads / kp, c.d_head * kp, h->elem_bytes,
                                      c.max_context, max_valid_hint, h->num_sms, h->num_splits);

    const uint64_t slab = layer_slab_bytes(h);
    kvc::DecodeArgs a{};
    a.K = h->k_base + slab * layer;
    a.V = h->v_base + slab * layer;
    a.q = q;
    a.out = out;
    a.k_new = static_cast<const uint8_t *>(k_new);
    a.v_new = static_cast<const uint8_t *>(v_new);
    a.k_scale = h->k_scale ? reinterpret_cast<const float *>(h->k_scale + layer_scale_bytes(h) * layer) : nullptr;
    a.v_scale = h->v_scale ? reinterpret_cast<const float *>(h->v_scale + layer_scale_bytes(h) * layer) : nullptr;
    a.valid_len = valid_len;
    a.part_ml = reinterpret_cast<float *>(h->ws + h->wl.part_ml);
    a.part_acc = reinterpret_cast<float *>(h->ws + h->wl.part_acc);
    a.tickets = reinterpret_cast<int32_t *>(h->ws + h->wl.tickets);
    a.ready = reinterpret_cast<int32_t *>(h->ws + h->wl.ready);
    a.err = reinterpret_cast<int32_t *>(h->ws);
    a.B = c.batch;
    a.H_kv = c.n_kv_heads;
    a.max_ctx = c.max_context;
    a.n_stages = h->n_stages;
    a.scale_log2 = float(1.4426950408889634 / std::sqrt(double(c.d_head)));
    a.timeout_ns = kvc::WAIT_TIMEOUT_NS;
    a.flag_timeout_ns = h->flag_timeout_ns;
    a.seg_base = layer * c.batch * c.n_kv_heads;
    a.block_table = h->block_table;
    a.max_blocks = c.max_context / 16;
    a.num_blocks = h->num_blocks;
    a.gran = h->block_table ? 16 : h->decode->split_gran > 1 ? h->decode->split_gran : 1;
    if (h->block_table) a.seg_base = layer * h->num_blocks * c.n_kv_heads;
    if (kp == 2) {  // segments are head pairs; the pair maps address blocks
        a.H_kv = c.n_kv_heads / 2;
        a.seg_base = layer * h->num_blocks;
    }
    if (h->decode->tensor_maps) {
        a.tm_k32 = h->tm_k32;
        a.tm_k8 = h->tm_k8;
        a.tm_v32 = h->tm_v32;
        a.tm_v8 = h->tm_v8;
        a.tm_k128 = h->pf_k128;  // encoded with the chunked prefill's maps
        a.tm_v128 = h->pf_v128;
        a.tm_kr32 = h->pf_k32;
        a.tm_vr32 = h->pf_v32;
        if (h->decode->ragged_maps && !h->block_table) {
            a.tm_k64 = h->rb_k64;
            a.tm_v64 = h->rb_v64;
            a.tm_kr32 = h->rb_k32;
            a.tm_vr32 = h->rb_v32;
        }
    }
    const cudaError_t e = h->decode->launch(a, grid, h->smem_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace

extern "C" {

kvc_status kvc_decode_attn(kvc_cache *h, int32_t layer, const void *q, const int32_t *valid_len,
                           int32_t max_valid_hint, void *out, void *stream) {
    if (!h || layer < 0 || layer >= h->cfg.n_layers || !q || !valid_len || !out)
        return KVC_ERR_INVALID;
    if (max_valid_hint < 0 || max_valid_hint > h->cfg.max_context) return KVC_ERR_INVALID;
    if (!aligned16(q)) return KVC_ERR_ALIGNMENT;
    return launch_decode(h, layer, q, valid_len, max_valid_hint, out, stream, nullptr, nullptr);
}

kvc_status kvc_decode_step(kvc_cache *h, int32_t layer, const void *q, const void *k_new, const void *v_new,
                           const int32_t *valid_len, int32_t max_valid_hint, void *out, void *stream) {
    if (!h || layer < 0 || layer >= h->cfg.n_layers || !q || !k_new || !v_new || !valid_len || !out)
        return KVC_ERR_INVALID;
    if (max_valid_hint < 0 || max_valid_hint > h->cfg.max_context) return KVC_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new)) return KVC_ERR_ALIGNMENT;
    // one launch: every decode kernel appends (an int8 cache: quantises) the
    // step's new rows as it streams
    return launch_decode(h, layer, q, valid_len, max_valid_hint, out, stream, k_new, v_new);
}

kvc_status kvc_prefill_attn(kvc_cache *h, int32_t layer, const void *q, const int32_t *cache_index,
                            int32_t T_new, void *out, void *stream) {
    if (!h || layer < 0 || layer >= h->cfg.n_layers || !q || !cache_index || !out || T_new < 0)
        return KVC_ERR_INVALID;
    if (T_new == 0) return KVC_OK;
    if (T_new > h->cfg.max_context) return KVC_ERR_CAPACITY;
    if (!h->prefill) return KVC_ERR_UNSUPPORTED;
    if (!aligned16(q)) return KVC_ERR_ALIGNMENT;
    const kvc_config &c = h->cfg;
    // work items of rows / g chunk tokens of one (sequence, KV head); the
    // kernel is persistent, one CTA per SM (or per item when there are fewer)
    const int64_t tokens_per_item = h->prefill->rows / h->group;  // >= 1: find_prefill checked the group
    const int64_t q_blocks = (T_new + tokens_per_item - 1) / tokens_per_item;
    const int64_t items = int64_t(c.batch) * c.n_kv_heads * q_blocks;
    if (items > 0x7fffffff) return KVC_ERR_UNSUPPORTED;
    const int64_t grid = items < h->num_sms ? items : h->num_sms;
    const uint64_t slab = layer_slab_bytes(h);
    kvc::PrefillArgs a{};
    a.K = h->k_base + slab * layer;
    a.V = h->v_base + slab * layer;
    a.q = q;
    a.out = out;
    a.cache_index = cache_index;
    a.err = reinterpret_cast<int32_t *>(h->ws);
    a.B = c.batch;
    a.H_kv = c.n_kv_heads;
    a.max_ctx = c.max_context;
    a.T_new = T_new;
    a.group = h->group;
    a.q_blocks = int(q_blocks);
    a.scale_log2 = float(1.4426950408889634 / std::sqrt(double(c.d_head)));
    a.timeout_ns = kvc::WAIT_TIMEOUT_NS;
    a.seg_base = layer * c.batch * c.n_kv_heads;
    a.tm_k128 = h->pf_k128;
    a.tm_v128 = h->pf_v128;
    a.tm_k32 = h->pf_k32;
    a.tm_k8 = h->pf_k8;
    a.tm_v32 = h->pf_v32;
    a.tm_v8 = h->pf_v8;
    const cudaError_t e = h->prefill->launch(a, int(grid), h->prefill->smem, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status kvc_get_error(kvc_cache *h, void *stream) {
    if (!h) return KVC_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, h->ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return KVC_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(h->ws, 0, sizeof word) != cudaSuccess) return KVC_ERR_CUDA;
        if (word == KVC_ERR_TIMEOUT) {
            // an aborted launch can leave counters and publish flags set
            const uint64_t n = h->wl.part_ml - h->wl.tickets;
            if (cudaMemset(h->ws + h->wl.tickets, 0, n) != cudaSuccess) return KVC_ERR_CUDA;
        }
        if (cudaDeviceSynchronize() != cudaSuccess) return KVC_ERR_CUDA;
    }
    return static_cast<kvc_status>(word);
}

}  // extern "C"
