// kvc_append.cu -- in-place append of new K/V rows into the static cache.
//
// "KV Cache Optimization: GQA Audit, In-Place Buffers, Persistent Prompts",
// #2 In-place KV cache updates (After): rows [valid, valid + T_new) of the
// pre-allocated [B, H, capacity, D] buffer are slice-assigned; nothing is
// concatenated or reallocated.  "10.3 -- KV cache implementation details",
// section 5: appending k_t, v_t is the only cache write of a decode step.
//
// For every (sequence b, KV head j) the T_new source rows k_new[b, j, :, :]
// and the destination rows K[b, j, cache_index[b] : cache_index[b] + T_new, :]
// are both contiguous runs of T_new * row_bytes bytes, so the whole append is
// a set of contiguous copies.  One thread moves one 16-byte vector;
// consecutive threads move consecutive vectors of a run (coalesced on both
// sides).  K and V are handled by the same launch.
#include <cuda_bf16.h>

#include "kvc_internal.cuh"

namespace kvc {

__global__ void __launch_bounds__(256) append_kernel(uint8_t *__restrict__ K, uint8_t *__restrict__ V,
                                                     const uint8_t *__restrict__ k_new,
                                                     const uint8_t *__restrict__ v_new,
                                                     const int32_t *__restrict__ cache_index, int index_offset,
                                                     int B, int H_kv, int T_new, int max_ctx, int row_vecs,
                                                     const int32_t *__restrict__ table, int max_blocks,
                                                     int num_blocks, int32_t *err) {
    dev::grid_dependency_wait();   // the previous kernel on the stream has completed
    dev::allow_dependents();
    const int64_t run = int64_t(T_new) * row_vecs;   // vectors per (b, j)
    const int64_t per_tensor = int64_t(B) * H_kv * run;
    const int64_t total = V ? 2 * per_tensor : per_tensor;   // V null: one tensor (a latent cache)
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const bool is_v = i >= per_tensor;
        const int64_t r = is_v ? i - per_tensor : i;
        const int64_t seg = r / run;                 // b * H_kv + j
        const int64_t off = r - seg * run;           // vector within the run
        const int b = int(seg / H_kv);
        const int ci = __ldg(cache_index + b) + index_offset;
        if (ci < 0 || ci > max_ctx - T_new) {
            if (off == 0 && seg % H_kv == 0 && !is_v) atomicCAS(err, 0, ERR_DEVICE_INDEX);
            continue;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(is_v ? v_new : k_new) + seg * run + off;
        int64_t row;  // destination row, in rows of the layer's cache or pool
        if (table) {  // paged: the position's slot in its physical block of 16 rows
            const int pos = ci + int(off / row_vecs);
            const int phys = __ldg(table + int64_t(b) * max_blocks + pos / 16);
            if (phys < 0 || phys >= num_blocks) {
                atomicCAS(err, 0, ERR_DEVICE_INDEX);
                continue;
            }
            row = (int64_t(phys) * H_kv + seg % H_kv) * 16 + pos % 16;
        } else {
            row = seg * max_ctx + ci + off / row_vecs;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(is_v ? V : K) + row * row_vecs + off % row_vecs;
        *dst = __ldg(src);
    }
}

// int8 cache ("10.3", section 4.4: the cache stored as int8, p = 1): each
// appended row of d_h bf16 elements is quantised symmetrically with one fp32
// scale, scale = absmax / 127 and code = rint(x * (127 / absmax)) in fp32
// (IEEE division and product, round half to even); a row of zeros gets
// scale 0.  One warp per (row, K or V): lane l holds elements
// [l * D/32, (l + 1) * D/32).
template <int D>
__global__ void __launch_bounds__(256) append_q8_kernel(uint8_t *__restrict__ K, uint8_t *__restrict__ V,
                                                        float *__restrict__ ks, float *__restrict__ vs,
                                                        const uint8_t *__restrict__ k_new,
                                                        const uint8_t *__restrict__ v_new,
                                                        const int32_t *__restrict__ cache_index,
                                                        int index_offset, int B, int H_kv, int T_new, int max_ctx,
                                                        int32_t *err) {
    constexpr int EPL = D / 32;  // bf16 elements per lane (2 or 4)
    dev::grid_dependency_wait();   // the previous kernel on the stream has completed
    dev::allow_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t rows = int64_t(B) * H_kv * T_new;       // rows per tensor
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t wi = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); wi < 2 * rows; wi += warps) {
        const bool is_v = wi >= rows;
        const int64_t r = is_v ? wi - rows : wi;              // (b * H_kv + j) * T_new + t
        const int64_t seg = r / T_new;
        const int t = int(r - seg * T_new);
        const int b = int(seg / H_kv);
        const int ci = __ldg(cache_index + b) + index_offset;
        if (ci < 0 || ci > max_ctx - T_new) {
            if (lane == 0 && t == 0 && seg % H_kv == 0 && !is_v) atomicCAS(err, 0, ERR_DEVICE_INDEX);
            continue;
        }
        const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(is_v ? v_new : k_new) + r * D + lane * EPL;
        float x[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] = __bfloat162float(src[e]);
        float scale;
        const uint32_t packed = dev::quantise_row_q8<EPL>(x, scale);
        const int64_t row = seg * max_ctx + ci + t;          // cache row within the layer
        uint8_t *dst = (is_v ? V : K) + row * D + lane * EPL;
        if constexpr (EPL == 4)
            *reinterpret_cast<uint32_t *>(dst) = packed;
        else
            *reinterpret_cast<uint16_t *>(dst) = uint16_t(packed);
        if (lane == 0) (is_v ? vs : ks)[row] = scale;
    }
}

cudaError_t launch_append_q8(uint8_t *K_layer, uint8_t *V_layer, float *ks_layer, float *vs_layer,
                             const uint8_t *k_new, const uint8_t *v_new, const int32_t *cache_index,
                             int index_offset, int B, int H_kv, int T_new, int max_ctx, int D, int32_t *err,
                             int num_sms, cudaStream_t stream) {
    const int64_t warps = 2 * int64_t(B) * H_kv * T_new;
    if (warps == 0) return cudaSuccess;
    const int64_t want = (warps + 7) / 8;                   // 8 warps per 256-thread block
    const int64_t cap = int64_t(num_sms) * 8;
    const int grid = int(want < cap ? want : cap);
    if (D == 128)
        return launch_pdl(append_q8_kernel<128>, dim3(grid), dim3(256), 0, stream, K_layer, V_layer, ks_layer, vs_layer,
                          k_new, v_new, cache_index, index_offset, B, H_kv, T_new, max_ctx, err);
    if (D == 64)
        return launch_pdl(append_q8_kernel<64>, dim3(grid), dim3(256), 0, stream, K_layer, V_layer, ks_layer, vs_layer,
                          k_new, v_new, cache_index, index_offset, B, H_kv, T_new, max_ctx, err);
    return cudaErrorInvalidValue;
}

cudaError_t launch_append(uint8_t *K_layer, uint8_t *V_layer, const uint8_t *k_new,
                          const uint8_t *v_new, const int32_t *cache_index, int index_offset, int B,
                          int H_kv, int T_new, int max_ctx, int row_bytes, int32_t *err, int num_sms,
                          cudaStream_t stream, const int32_t *table, int max_blocks, int num_blocks) {
    const int row_vecs = row_bytes / 16;
    const int64_t total = (V_layer ? 2 : 1) * int64_t(B) * H_kv * T_new * row_vecs;
    if (total == 0) return cudaSuccess;
    const int64_t want = (total + 255) / 256;
    const int64_t cap = int64_t(num_sms) * 8;
    const int grid = int(want < cap ? want : cap);
    return launch_pdl(append_kernel, dim3(grid), dim3(256), 0, stream, K_layer, V_layer, k_new, v_new, cache_index,
                      index_offset, B, H_kv, T_new, max_ctx, row_vecs, table, max_blocks, num_blocks, err);
}

}  // namespace kvc
