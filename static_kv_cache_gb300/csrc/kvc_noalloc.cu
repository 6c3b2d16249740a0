// kvc_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// kvc_decode_attn needs a workspace buffer (split partials, per-segment
// counters, the error word) that the caller allocates and binds with
// kvc_alloc.  Some callers cannot do that: their device memory is owned by
// someone else -- a host framework that budgets every byte itself, or a plugin
// interface that hands the library only the tensors of the call -- so they
// can neither call cudaMalloc nor give the library a workspace.  For them,
// kvc_decode_attn_static runs the same decode kernel with its scratch in a
// fixed-size array that lives in this library's device memory image.  Nothing
// is allocated at call time.
//
// Costs of that choice, which the caller accepts:
//   * every GPU that loads the library holds KVC_STATIC_SCRATCH_BYTES of
//     device memory for the array until the process exits;
//   * all calls share the one array: calls that overlap on the GPU (different
//     streams without ordering between them) race and produce garbage; order
//     them on one stream;
//   * a configuration whose scratch does not fit the array is rejected.
#include <cmath>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.cuh"

namespace {

// The scratch array.  Its size is the library's stated maximum.
static __device__ __align__(256) uint8_t g_static_scratch[KVC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    uint8_t *scratch = nullptr;  // device address of g_static_scratch on this device
    int num_sms = 0;
    int smem_optin = 0;
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Shared-memory attribute already set for (device, kernel); the kernels are
// few, so a short list per device suffices.
constexpr int kMaxKernelsPerDevice = 128;
const kvc::DecodeKernelInfo *g_smem_set[kMaxDevices][kMaxKernelsPerDevice];
int g_smem_set_count[kMaxDevices];

int elem_bytes(int32_t dtype) {
    switch (dtype) {
        case KVC_BF16: return 2;
        case KVC_FP16: return 2;
        case KVC_FP32: return 4;
        default: return 0;
    }
}

// One-time set-up for the current device: the scratch array's device
// address, the SM count and the shared-memory limit.
kvc_status setup_device(int dev, DeviceSetup **out) {
    if (dev < 0 || dev >= kMaxDevices) return KVC_ERR_UNSUPPORTED;
    DeviceSetup &s = g_setup[dev];
    if (!s.ready) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) return KVC_ERR_CUDA;
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return KVC_ERR_CUDA;
        if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return KVC_ERR_CUDA;
        s.scratch = static_cast<uint8_t *>(ptr);
        s.num_sms = sms;
        s.smem_optin = smem;
        s.ready = true;
    }
    *out = &s;
    return KVC_OK;
}

kvc_status ensure_smem_attribute(int dev, const kvc::DecodeKernelInfo *info, int smem_bytes) {
    for (int i = 0; i < g_smem_set_count[dev]; ++i)
        if (g_smem_set[dev][i] == info) return KVC_OK;
    if (g_smem_set_count[dev] >= kMaxKernelsPerDevice) return KVC_ERR_UNSUPPORTED;
    if (info->set_max_smem(smem_bytes) != cudaSuccess) return KVC_ERR_CUDA;
    g_smem_set[dev][g_smem_set_count[dev]++] = info;
    return KVC_OK;
}

uint64_t round256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

}  // namespace

extern "C" kvc_status kvc_decode_attn_static(const kvc_config *cfg, int32_t layer, const void *k_base,
                                             const void *v_base, const void *q,
                                             const int32_t *valid_len, int32_t max_valid_hint,
                                             void *out, void *stream) {
    if (!cfg || !k_base || !v_base || !q || !valid_len || !out) return KVC_ERR_INVALID;
    if (cfg->dtype == KVC_INT8) return KVC_ERR_UNSUPPORTED;  // no scale arrays on this call
    const int eb = elem_bytes(cfg->dtype);
    if (eb == 0 || cfg->n_layers <= 0 || cfg->batch <= 0 || cfg->n_heads <= 0 || cfg->n_kv_heads <= 0 ||
        cfg->d_head <= 0 || cfg->max_context <= 0 || cfg->n_heads % cfg->n_kv_heads != 0)
        return KVC_ERR_INVALID;
    if (layer < 0 || layer >= cfg->n_layers) return KVC_ERR_INVALID;
    if (max_valid_hint < 0 || max_valid_hint > cfg->max_context) return KVC_ERR_INVALID;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(k_base) | reinterpret_cast<uintptr_t>(v_base) |
                          reinterpret_cast<uintptr_t>(q);
    if (mis & 15u) return KVC_ERR_ALIGNMENT;
    const int G = cfg->n_heads / cfg->n_kv_heads;
    const kvc::DecodeKernelInfo *info = kvc::find_decode_kernel(cfg->dtype, cfg->d_head, G);
    if (!info) return KVC_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
    DeviceSetup *ds = nullptr;
    int n_stages = 0, smem_bytes = 0;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        kvc_status st = setup_device(dev, &ds);
        if (st != KVC_OK) return st;
        n_stages = kvc::decode_stage_count(info, ds->smem_optin);
        if (n_stages == 0) return KVC_ERR_UNSUPPORTED;
        smem_bytes = info->fixed_smem + n_stages * info->stage_bytes;
        st = ensure_smem_attribute(dev, info, smem_bytes);
        if (st != KVC_OK) return st;
    }

    // Grid: the choice kvc_decode_attn makes, at most one CTA per SM.
    const int grid = kvc::decode_grid(info, cfg->batch, cfg->n_kv_heads, cfg->d_head, eb, cfg->max_context,
                                      max_valid_hint, ds->num_sms, 0);

    // Scratch layout inside the array: error word, one counter per
    // (sequence, KV head), one publish flag per split slot, then the split
    // partials.  Split c of segment s uses slot c + s, so grid + B * H_kv
    // slots suffice.
    const uint64_t segs = uint64_t(cfg->batch) * cfg->n_kv_heads;
    const uint64_t slots = uint64_t(grid) + segs;
    const uint64_t off_tickets = 256;
    const uint64_t off_ready = round256(off_tickets + segs * 4);
    const uint64_t off_ml = round256(off_ready + slots * 4);
    const uint64_t off_acc = round256(off_ml + slots * G * 2 * 4);
    const uint64_t total = round256(off_acc + slots * G * uint64_t(cfg->d_head) * 4);
    if (total > KVC_STATIC_SCRATCH_BYTES) return KVC_ERR_WORKSPACE;

    // Tensor maps of the caches for kernels that read through them (host
    // computation only).
    CUtensorMap maps[4];
    if (info->tensor_maps &&
        !kvc::encode_cache_maps(cfg->dtype, cfg->d_head, cfg->max_context,
                                int64_t(cfg->n_layers) * cfg->batch * cfg->n_kv_heads, k_base, v_base,
                                &maps[0], &maps[1], &maps[2], &maps[3], info->tile_box))
        return KVC_ERR_CUDA;

    // The array keeps the previous call's contents: the counters and the
    // publish flags must start at zero.  The error word is left alone: it
    // keeps the first error any call recorded until kvc_static_get_error
    // reads and clears it.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ds->scratch + off_tickets, 0, off_ml - off_tickets, s) != cudaSuccess) return KVC_ERR_CUDA;

    const uint64_t slab = uint64_t(cfg->batch) * cfg->n_kv_heads * uint64_t(cfg->max_context) *
                          cfg->d_head * eb;
    kvc::DecodeArgs a{};
    a.K = static_cast<const uint8_t *>(k_base) + slab * layer;
    a.V = static_cast<const uint8_t *>(v_base) + slab * layer;
    a.q = q;
    a.out = out;
    a.k_new = nullptr;
    a.v_new = nullptr;
    a.k_scale = nullptr;
    a.v_scale = nullptr;
    a.valid_len = valid_len;
    a.part_ml = reinterpret_cast<float *>(ds->scratch + off_ml);
    a.part_acc = reinterpret_cast<float *>(ds->scratch + off_acc);
    a.tickets = reinterpret_cast<int32_t *>(ds->scratch + off_tickets);
    a.ready = reinterpret_cast<int32_t *>(ds->scratch + off_ready);
    a.err = reinterpret_cast<int32_t *>(ds->scratch);
    a.B = cfg->batch;
    a.H_kv = cfg->n_kv_heads;
    a.max_ctx = cfg->max_context;
    a.n_stages = n_stages;
    a.scale_log2 = float(1.4426950408889634 / std::sqrt(double(cfg->d_head)));
    a.timeout_ns = kvc::WAIT_TIMEOUT_NS;
    a.flag_timeout_ns = kvc::WAIT_TIMEOUT_NS;
    a.seg_base = layer * cfg->batch * cfg->n_kv_heads;
    a.block_table = nullptr;
    a.max_blocks = a.num_blocks = 0;
    a.gran = 1;
    if (info->tensor_maps) {
        a.tm_k32 = maps[0];
        a.tm_k8 = maps[1];
        a.tm_v32 = maps[2];
        a.tm_v8 = maps[3];
    }
    const cudaError_t e = info->launch(a, int(grid), smem_bytes, s);
    return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

extern "C" kvc_status kvc_static_get_error(void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
    DeviceSetup *ds = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        const kvc_status st = setup_device(dev, &ds);
        if (st != KVC_OK) return st;
    }
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
    int32_t word = 0;  // host stack: the read allocates nothing
    if (cudaMemcpy(&word, ds->scratch, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return KVC_ERR_CUDA;
    if (word != 0 && cudaMemset(ds->scratch, 0, sizeof word) != cudaSuccess) return KVC_ERR_CUDA;
    if (word != 0 && cudaDeviceSynchronize() != cudaSuccess) return KVC_ERR_CUDA;
    return static_cast<kvc_status>(word);
}
