// kvc_internal.cuh -- definitions shared by the kernels and the host API of
// libkvc.so.  Not part of the public ABI (see include/kvc.h).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace kvc {

// Device error codes written to the workspace error word (match kvc_status).
constexpr int32_t ERR_TIMEOUT = 5;
constexpr int32_t ERR_DEVICE_INDEX = 6;

// Upper bound on the CTAs of one decode launch; sizes the split partials.
constexpr int MAX_CTAS = 1024;

// Dynamic shared memory a decode CTA may use (stages + scratch): the whole
// opt-in limit of one block (227 KB on sm_100-class GPUs).
constexpr int SMEM_BUDGET = 227 * 1024;

// Default bound on any single wait inside a kernel.
constexpr unsigned long long WAIT_TIMEOUT_NS = 1000ull * 1000ull * 1000ull;  // 1 s

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)            error word (int32) + padding
//   tickets             int32 [B * H_kv]         arrivals per (sequence, KV head)
//   ready               int32 [slots]            split partial published (1) or not (0)
//   part_ml             float [slots][G][2]      (running max, sum) per split
//   part_acc            float [slots][G][D]      unnormalised output per split
// slots = MAX_CTAS + B * H_kv: split c of segment s uses slot c + s, which is
// unique because the splits and the segments are both contiguous ranges of
// one flattened row space (every new piece starts a new split, a new
// segment, or both).
// ---------------------------------------------------------------------------
struct WorkspaceLayout {
    uint64_t tickets, ready, part_ml, part_acc, total;
};

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

inline WorkspaceLayout workspace_layout(int B, int H_kv, int G, int D) {
    WorkspaceLayout w;
    const uint64_t segs = uint64_t(B) * H_kv;
    const uint64_t slots = uint64_t(MAX_CTAS) + segs;
    w.tickets = 256;
    w.ready = align256(w.tickets + segs * 4);
    w.part_ml = align256(w.ready + slots * 4);
    w.part_acc = align256(w.part_ml + slots * G * 2 * 4);
    w.total = align256(w.part_acc + slots * G * uint64_t(D) * 4);
    return w;
}

// Arguments of the decode kernel (passed by value as a grid constant).
struct DecodeArgs {
    const uint8_t *K;          // layer slab of the K cache, [B, H_kv, max_ctx, D]
    const uint8_t *V;          // layer slab of the V cache
    const void *q;             // [B, H, D]
    void *out;                 // [B, H, D]
    // Fused decode step (tensor-core kernel): the new rows [B, H_kv, D] that
    // this launch appends at valid_len - 1 and attends with; null otherwise.
    const uint8_t *k_new;
    const uint8_t *v_new;
    // int8 caches: one fp32 scale per cache row, [B, H_kv, max_ctx] per layer
    const float *k_scale;
    const float *v_scale;
    // Paged caches (tensor-core kernel): K and V are this layer's pools
    // [num_blocks, H_kv, 16, D], block_table [B, max_blocks] maps a sequence's
    // logical block to a physical one; null for contiguous caches.
    const int32_t *block_table;
    int32_t max_blocks, num_blocks;
    // Rows of the flattened split space per segment are rounded up to a
    // multiple of gran (16 for paged caches, so every tile starts on a block).
    int32_t gran;
    const int32_t *valid_len;  // [B]
    float *part_ml;
    float *part_acc;
    int32_t *tickets;
    int32_t *ready;            // [slots], zero between launches
    int32_t *err;
    int32_t B, H_kv, max_ctx;
    int32_t n_stages;
    float scale_log2;          // log2(e) / sqrt(D)
    unsigned long long timeout_ns;
    // Limit of the last split's wait for the other splits' partials (the
    // split combine's ready flags); every other wait keeps timeout_ns.
    unsigned long long flag_timeout_ns;
    // Tensor maps of the whole K and V caches viewed as [L*B*H_kv][T_max][D]
    // (16-bit caches, tensor-core kernel only): boxes of 64 columns x 32 or
    // x 8 rows with the 128-byte swizzle.  seg_base = layer * B * H_kv.
    int32_t seg_base;
    CUtensorMap tm_k32, tm_k8, tm_v32, tm_v8;  // the type carries its own alignment
    // The tcgen05 kernel of large head groups: boxes of 64 columns x 128 and
    // x 32 rows over the same caches (one column block per box); it takes
    // its 8-row boxes from tm_k8 / tm_v8.  The int8 kernel: boxes of 128
    // codes x 32 rows in tm_kr32 / tm_vr32 and x 64 rows in tm_k64 / tm_v64,
    // for the tile that holds a fused step's new row.
    CUtensorMap tm_k128, tm_v128, tm_kr32, tm_vr32;
    CUtensorMap tm_k64, tm_v64;
};

// One compiled decode kernel and what the host needs to launch it.
struct DecodeKernelInfo {
    int tile_rows;       // rows of K (and of V) per pipeline stage
    int consumer_warps;  // warps that compute; one more warp issues the copies
    int stage_bytes;     // K tile + V tile
    int fixed_smem;      // dynamic shared memory besides the stages
    cudaError_t (*set_max_smem)(int bytes);
    cudaError_t (*launch)(const DecodeArgs &a, int grid, int smem, cudaStream_t s);
    bool tensor_maps;    // reads K/V through the tensor maps in DecodeArgs
    bool tile_box;       // its full-tile map is the 4-D one of encode_cache_maps
    bool row_box_maps;   // also reads through the 128- and 32-row maps (tm_k128 ...)
    // Split points fall on multiples of this many rows of a segment (0: any
    // row).  A kernel's tile: then only a segment's last tile is ragged, not
    // also the last tile of every piece that ends inside a segment (each
    // ragged tile costs the copy issuer several small boxes).
    int split_gran;
    // Also reads a ragged tile through boxes of 128-byte row slices x 64 and
    // x 32 rows (tm_k64 / tm_v64, tm_kr32 / tm_vr32; contiguous caches).
    bool ragged_maps;
};

// Registry of compiled decode kernels, one lookup per (element type, D);
// each returns nullptr for an unsupported group size.
#define KVC_DECLARE_DECODE_TABLE(TAG, D) \
    const DecodeKernelInfo *decode_kernel_##TAG##_##D(int G);
KVC_DECLARE_DECODE_TABLE(bf16, 32)
KVC_DECLARE_DECODE_TABLE(bf16, 64)
KVC_DECLARE_DECODE_TABLE(bf16, 128)
KVC_DECLARE_DECODE_TABLE(bf16, 256)
KVC_DECLARE_DECODE_TABLE(f16, 32)
KVC_DECLARE_DECODE_TABLE(f16, 64)
KVC_DECLARE_DECODE_TABLE(f16, 128)
KVC_DECLARE_DECODE_TABLE(f16, 256)
KVC_DECLARE_DECODE_TABLE(f32, 32)
KVC_DECLARE_DECODE_TABLE(f32, 64)
KVC_DECLARE_DECODE_TABLE(f32, 128)
KVC_DECLARE_DECODE_TABLE(f32, 256)
KVC_DECLARE_DECODE_TABLE(q8, 128)
#undef KVC_DECLARE_DECODE_TABLE
// paged pools with d_h = 128: the tensor-core kernel in the half-row tile layout
const DecodeKernelInfo *decode_kernel_paged_bf16_128(int G);
const DecodeKernelInfo *decode_kernel_paged_f16_128(int G);
// contiguous caches with 16 or 32 query heads per KV head at d_h = 128: the
// tcgen05 kernel (keys on M = 128, the group's heads on N)
const DecodeKernelInfo *decode_kernel_tc_bf16_128(int G);
const DecodeKernelInfo *decode_kernel_tc_f16_128(int G);
// paged pools read two KV heads per tile (G2 = query heads of both: 4 or 8)
const DecodeKernelInfo *decode_kernel_pair_bf16_64(int G2);
const DecodeKernelInfo *decode_kernel_pair_bf16_128(int G2);
const DecodeKernelInfo *decode_kernel_pair_f16_64(int G2);
const DecodeKernelInfo *decode_kernel_pair_f16_128(int G2);

// Launch planning shared by every decode entry point (kvc_api.cu).
// The kernel for a contiguous cache of this element type, head width and
// query-head group; nullptr where none is compiled.
const DecodeKernelInfo *find_decode_kernel(int32_t dtype, int D, int G);
// Pipeline stages that fit the shared memory a block may opt into (at most
// 32, at least one more than the consumer warps); 0 if that many do not fit.
int decode_stage_count(const DecodeKernelInfo *info, int smem_optin);
// CTAs of one decode launch: `forced` when non-zero, otherwise one CTA per SM
// with at least four tiles each, or one CTA per (sequence, KV head) segment
// when the problem is small and every segment holds at most 64 KB per tensor.
int decode_grid(const DecodeKernelInfo *info, int B, int H_kv, int D, int elem_bytes, int max_ctx,
                int max_valid_hint, int num_sms, int forced);

// Arguments of the chunked-prefill kernel (grid constant).
struct PrefillArgs {
    const uint8_t *K;            // layer slab of the K cache, [B, H_kv, max_ctx, D]
    const uint8_t *V;            // layer slab of the V cache
    const void *q;               // [B, H, T_new, D]
    void *out;                   // [B, H, T_new, D]
    const int32_t *cache_index;  // [B]: row of each sequence's first chunk token
    int32_t *err;
    int32_t B, H_kv, max_ctx, T_new;
    int32_t group;               // g = H / H_kv query heads per KV head
    int32_t q_blocks;            // CTAs per (sequence, KV head): ceil(T_new / (rows / g))
    float scale_log2;            // log2(e) / sqrt(D)
    unsigned long long timeout_ns;
    int32_t seg_base;            // layer * B * H_kv (tensor-map segment of this layer)
    // the cache viewed as [L*B*H_kv][T_max][D]: boxes of 64 columns x 128,
    // 32 and 8 rows, 128-byte swizzle
    CUtensorMap tm_k128, tm_v128, tm_k32, tm_k8, tm_v32, tm_v8;
};

// One compiled prefill kernel.
struct PrefillKernelInfo {
    int rows;    // query rows per work item: rows / g chunk tokens of the g heads of a KV head
    int smem;    // dynamic shared memory per CTA
    cudaError_t (*set_max_smem)(int bytes);
    cudaError_t (*launch)(const PrefillArgs &a, int grid, int smem, cudaStream_t s);
};

// Registry of prefill kernels (16-bit caches, D = 64 or 128); nullptr for an
// unsupported group size (more query heads per KV head than rows per CTA).
#define KVC_DECLARE_PREFILL_TABLE(TAG, D) \
    const PrefillKernelInfo *prefill_kernel_##TAG##_##D(int G);
KVC_DECLARE_PREFILL_TABLE(bf16, 64)
KVC_DECLARE_PREFILL_TABLE(bf16, 128)
KVC_DECLARE_PREFILL_TABLE(f16, 64)
KVC_DECLARE_PREFILL_TABLE(f16, 128)
#undef KVC_DECLARE_PREFILL_TABLE

// Tensor maps of a K and a V cache [n_segs][max_ctx][D] (n_segs = L * B *
// H_kv), 128-byte swizzle.  16-bit elements: boxes of 64 columns x 32 rows and
// x 8 rows (one 64-column block of a tile each).  With tile_box the 32-row
// map is 4-D instead, (64 columns, rows, D / 64 column blocks, segments) with
// the blocks 128 bytes apart, so one box brings a whole 32-row tile laid out
// block after block.  int8 codes: boxes of 128 columns x 128
// rows (a whole int8 decode tile) and x 8 rows.  Host only; returns false if
// the driver refuses.
bool encode_cache_maps(int32_t dtype, int D, int max_ctx, int64_t n_segs, const void *k_base,
                       const void *v_base, CUtensorMap *k32, CUtensorMap *k8, CUtensorMap *v32,
                       CUtensorMap *v8, bool tile_box = false);

// Tensor maps of K and V caches [n_segs][max_ctx][D] with boxes of 128 bytes
// of a row (64 16-bit elements or 128 int8 codes) x `rows` rows (at most
// 256), 128-byte swizzle.  Host only.
bool encode_row_box_maps(int32_t dtype, int D, int max_ctx, int64_t n_segs, const void *k_base,
                         const void *v_base, int rows, CUtensorMap *k, CUtensorMap *v);

// Quantising append for int8 caches (kvc_append.cu): bf16 rows -> one fp32
// scale per row and int8 codes, written at cache_index[b] + index_offset.
cudaError_t launch_append_q8(uint8_t *K_layer, uint8_t *V_layer, float *ks_layer, float *vs_layer,
                             const uint8_t *k_new, const uint8_t *v_new, const int32_t *cache_index,
                             int index_offset, int B, int H_kv, int T_new, int max_ctx, int D, int32_t *err,
                             int num_sms, cudaStream_t stream);

// Append launcher (kvc_append.cu): rows go to cache_index[b] + index_offset;
// with a block table, K_layer / V_layer are the layer's pools [num_blocks,
// H_kv, 16, D] and the rows go to their slots in the mapped blocks.
cudaError_t launch_append(uint8_t *K_layer, uint8_t *V_layer, const uint8_t *k_new,
                          const uint8_t *v_new, const int32_t *cache_index, int index_offset,
                          int B, int H_kv, int T_new, int max_ctx, int row_bytes, int32_t *err,
                          int num_sms, cudaStream_t stream, const int32_t *table = nullptr,
                          int max_blocks = 0, int num_blocks = 0);

// Launch `kernel` with programmatic stream serialization, so that its CTAs may
// be scheduled while the previous kernel on the stream drains (the kernel
// calls dev::grid_dependency_wait before touching global memory).
#ifdef __CUDACC__
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, int smem, cudaStream_t s, const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
#endif

// Tensor maps of paged pools [n_blocks_total][16][D] (n_blocks_total = L *
// num_blocks * H_kv), each block viewed as 16 * D/64 rows of 128 bytes: boxes
// of 64 columns x all of them (a whole block, in the *32 slots) and x half of
// them (its first 8 rows), 128-byte swizzle.  Host only.
bool encode_pool_maps(int32_t dtype, int D, int64_t n_blocks_total, const void *k_pool, const void *v_pool,
                      CUtensorMap *k16, CUtensorMap *k8, CUtensorMap *v16, CUtensorMap *v8);
// Tensor maps of paged pools read two KV heads at a time: the pools as 5-D
// arrays (64 columns, 16 rows, D/64 column blocks, H_kv heads, blocks_total =
// L * num_blocks blocks), boxes of (64, 16, D/64, 2, 1) -- a block's rows of
// two heads -- and of (64, 8, 1, 1, 1), 128-byte swizzle.  Host only.
bool encode_pool_pair_maps(int32_t dtype, int D, int H_kv, int64_t blocks_total, const void *k_pool,
                           const void *v_pool, CUtensorMap *k16, CUtensorMap *k8, CUtensorMap *v16, CUtensorMap *v8);

}  // namespace kvc

// ---------------------------------------------------------------------------
// Device helpers: inline PTX for mbarriers, bulk (TMA) copies and timers.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
namespace kvc {
namespace dev {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test: has the phase of `bar` with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when *abort becomes non-zero, after timeout_ns of wall
// time, or after 2^30 polls, whichever comes first.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int *abort,
                                                  unsigned long long timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// 16-byte asynchronous copy global -> shared (L2 only), tracked by the
// issuing thread's cp.async group.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// 4-byte asynchronous copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed; the
// barrier's pending count is raised first, so the phase cannot complete
// before then.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Wait until the global flag *p becomes non-zero (acquire at GPU scope).
// Gives up like mbar_wait_bounded.
__device__ __forceinline__ bool flag_wait_bounded(const int32_t *p, const volatile int *abort,
                                                  unsigned long long timeout_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v != 0) return true;
        if (*abort) return false;
        if (it == 0) {
            t0 = global_timer_ns();
        } else if (global_timer_ns() - t0 > timeout_ns) {
            return false;
        }
    }
    return false;
}

// Store to a global flag that other CTAs poll (after a fence that orders the
// data it publishes).
__device__ __forceinline__ void flag_store(int32_t *p, int32_t v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 1-D bulk copy global -> shared through the TMA unit; completion is
// signalled on `bar` as transaction bytes.  dst, src and bytes must be
// multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// The same copy with an L2 cache policy (l2_evict_first_policy ...).
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Four 8x8 matrices of 16-bit elements from shared memory; lane l supplies
// the address of row (l % 8) of matrix (l / 8).  Lane l receives, from each
// matrix, the 32-bit pair (row l/4, columns 2*(l%4) and 2*(l%4)+1); with
// .trans it receives (rows 2*(l%4) and 2*(l%4)+1, column l/4) instead.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// d[16x8] += A[16x16] * B[16x8] with fp32 accumulation on the warp's tensor
// core path; A row-major, B column-major, both bf16 (or both fp16).
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit elements held as a warp fragment: lane
// l holds the pair (row l/4, columns 2*(l%4), 2*(l%4)+1) before and after.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// One box of a 3-D tensor map (coordinates innermost first) into shared
// memory through the TMA unit, completion signalled on `bar`.
// L2 policies for the cache hint of a copy.  evict_first: the lines a copy
// brings in are the first to go, for K/V (or latent) tiles that a decode
// launch reads exactly once; they then do not push the small arrays that
// every launch reuses (queries, lengths, block tables, split partials) out
// of L2 on their way through.  evict_normal: the default behaviour.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// The same copy with an L2 cache policy (l2_evict_first_policy ...).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                           uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// The same for a 4-D tensor map.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, int w,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// The same copy with an L2 cache policy (l2_evict_first_policy ...).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, int w,
                                           uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
        : "memory");
}

// The same for a 5-D tensor map.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, int w, int u,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(u), "r"(bar)
        : "memory");
}

// The same copy with an L2 cache policy (l2_evict_first_policy ...).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, int w, int u,
                                           uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(u), "r"(bar), "l"(policy)
        : "memory");
}

// Bring a tensor map's descriptor close to the TMA unit before its first use.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Order this thread's earlier generic-proxy shared-memory writes before
// later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void record_error(int32_t *err, int32_t code) {
    atomicCAS(err, 0, code);
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream drains;
// grid_dependency_wait blocks until that kernel has completed and its memory
// operations are visible (immediately when there is no such kernel), so it
// comes before the first global-memory access.  allow_dependents lets the
// next such kernel be scheduled once every CTA of this grid has issued it.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The int8 cache's quantisation of one row ("10.3 -- KV cache implementation
// details", section 4.4: the cache stored as int8, p = 1), taken by a whole
// warp: lane l holds elements [l * EPL, (l + 1) * EPL) of the row in fp32.
// scale = absmax / 127 and code = rint(x * (127 / absmax)) in fp32 (IEEE
// division and product, round half to even), codes clamped to [-127, 127]; a
// row of zeros gets scale 0.  Returns the lane's EPL codes packed little-end
// first; every caller (the append and the fused decode step) goes through
// this one function, so their codes agree bit for bit.
template <int EPL>
__device__ __forceinline__ uint32_t quantise_row_q8(const float (&x)[EPL], float &scale) {
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) am = fmaxf(am, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    scale = am / 127.0f;
    const float inv = am > 0.f ? 127.0f / am : 0.f;
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        int c = __float2int_rn(x[e] * inv);
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        packed |= (uint32_t(c) & 0xffu) << (8 * e);
    }
    return packed;
}

}  // namespace dev
}  // namespace kvc
#endif
