// kvc_prefill.cuh -- chunked-prefill attention over the static cache.
//
// "KV-Cache Mechanics", AR Static KV-Cache: prefill is a forward pass over
// the prompt that fills the pre-allocated cache from cache_index; decoding
// continues where it stopped.  "10.3 -- KV cache implementation details",
// section 3: prefill processes the prompt's positions together (compute
// bound), decode one position per step.  With the chunk's T_new rows already
// appended at cache_index c, the query of chunk position t attends causally
// over cache rows [0, c + t]; the mask is implicit on the pages and the
// causal reading is the one under which prefill, chunked prefill and decode
// agree.
//
// Unlike decode, this is a dense contraction: T_new * g query rows of one KV
// head against the same keys.  One CTA takes 64 query rows of one (sequence,
// KV head), ordered token-major inside the head group (row r = t * g + i),
// and every key row the last of them can see.  Four consumer warps own 16
// query rows each and keep Q in registers as mma.sync m16n8k16 A fragments;
// a producer warp streams K and V tiles through the same TMA tensor maps,
// 128-byte swizzle and live-range-only boxes as the tensor-core decode
// kernel; every consumer reads every tile (the stage is released when all
// four have).  Per tile and warp:
//   S[16 x 32] = Q . K^T (B = K rows by ldmatrix), causal mask on the tiles
//   that cross a row's limit, online softmax per row (two shuffles), and
//   O[16 x D] += P . V with P taken from the S accumulator as the A operand
//   and V by ldmatrix .trans.
// Each CTA covers its rows' whole key range, so no split combine is needed.
#pragma once

#include "kvc_decode_mma.cuh"

namespace kvc {

template <typename T, int D, int G>
struct PrefillCfg {
    using M = MmaCfg<T, D, G>;                       // tile geometry and swizzle
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int TILE = M::TILE;             // keys per tile (32)
    static constexpr int TILE_BYTES = M::TILE_BYTES;
    static constexpr int STAGE_BYTES = M::STAGE_BYTES;
    static constexpr int CHUNKS = M::CHUNKS;
    static constexpr int KSTEPS = D / 16;
    static constexpr int NTD = D / 8;
    static constexpr int NWQ = 4;                    // consumer warps, 16 query rows each
    static constexpr int QROWS = 16 * NWQ;
    static constexpr int THREADS = (NWQ + 1) * 32;
    static constexpr int N_STAGES = 4;
    // alignment slack, barriers, abort flag
    static constexpr int FIXED_SMEM = 1024 + 16 * N_STAGES + 16;
    static constexpr int SMEM = FIXED_SMEM + N_STAGES * STAGE_BYTES;
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(PrefillCfg<T, D, G>::THREADS, 2)
    prefill_kernel(const __grid_constant__ PrefillArgs a) {
    using C = PrefillCfg<T, D, G>;
    using Ops = MmaOps<T>;
    using E = ElemOps<T>;
    constexpr int TILE = C::TILE, KSTEPS = C::KSTEPS, NTD = C::NTD, NS = C::N_STAGES, NWQ = C::NWQ;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t stage0 = dev::smem_addr(smem);
    const uint32_t bar0 = stage0 + NS * C::STAGE_BYTES;  // full[NS], then empty[NS]
    volatile int *flags = reinterpret_cast<volatile int *>(smem + NS * C::STAGE_BYTES + 16 * NS);

    const int seg = int(blockIdx.x) / a.q_blocks;       // b * H_kv + kv
    const int qb = int(blockIdx.x) % a.q_blocks;
    const int b = seg / a.H_kv, kv = seg % a.H_kv;
    dev::grid_dependency_wait();   // the previous kernel on the stream (the chunk's append) has completed
    dev::allow_dependents();
    const int c = __ldg(a.cache_index + b);
    if (c < 0 || c > a.max_ctx - a.T_new) {             // uniform over the CTA
        if (threadIdx.x == 0 && qb == 0 && kv == 0) dev::record_error(a.err, ERR_DEVICE_INDEX);
        return;
    }
    const int rows = a.T_new * G;                        // query rows of this (b, kv)
    const int r_first = qb * C::QROWS;
    const int r_end = min(rows, r_first + C::QROWS);
    const int kend = c + (r_end - 1) / G + 1;            // keys the last row can see

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&a.tm_k32);
        dev::prefetch_tensormap(&a.tm_v32);
        for (int s = 0; s < NS; ++s) {
            dev::mbar_init(bar0 + 8 * s, 1);
            dev::mbar_init(bar0 + 8 * (NS + s), NWQ);
        }
        flags[0] = 0;
        dev::fence_mbar_init();
    }
    __syncthreads();
    const int ntiles = (kend + TILE - 1) / TILE;

    // ---------------------------------------------------------------- producer
    if (warp == 0) {
        constexpr int CB = C::ROW_BYTES / 128;
        const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;
        const uint8_t *kseg = a.K + int64_t(seg) * kv_slab;
        const uint8_t *vseg = a.V + int64_t(seg) * kv_slab;
        const int z = a.seg_base + seg;
        uint32_t generic_written = 0, issued = 0;
        for (int t = 0; t < ntiles; ++t) {
            const int stage = t % NS;
            const uint32_t round = uint32_t(t / NS);
            if (round > 0) {
                const bool w = dev::mbar_wait_bounded(bar0 + 8 * (NS + stage), (round - 1) & 1, flags, a.timeout_ns);
                if (!__all_sync(FULL, w)) {
                    if (lane == 0) {
                        if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                        flags[0] = 1;
                    }
                    break;
                }
            }
            const int row0 = t * TILE, nr = min(TILE, kend - row0);
            const uint32_t full = bar0 + 8 * stage;
            const uint32_t kdst = stage0 + uint32_t(stage) * C::STAGE_BYTES, vdst = kdst + C::TILE_BYTES;
            const int q = nr >> 3, rem = nr & 7;
            if (lane == 0) {
                if (generic_written & (1u << stage)) dev::fence_proxy_async_smem();
                dev::mbar_expect_tx(full, 2u * uint32_t(8 * q) * C::ROW_BYTES);
                if (q == 4) {
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb) {
                        dev::tma_load_3d(kdst + cb * C::M::BLOCK_BYTES, &a.tm_k32, cb * 64, row0, z, full);
                        dev::tma_load_3d(vdst + cb * C::M::BLOCK_BYTES, &a.tm_v32, cb * 64, row0, z, full);
                    }
                } else {
                    for (int j = 0; j < q; ++j)
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb) {
                            const uint32_t off = cb * C::M::BLOCK_BYTES + j * 8 * 128;
                            dev::tma_load_3d(kdst + off, &a.tm_k8, cb * 64, row0 + 8 * j, z, full);
                            dev::tma_load_3d(vdst + off, &a.tm_v8, cb * 64, row0 + 8 * j, z, full);
                        }
                }
            }
            if (rem) {
                const int per = rem * C::CHUNKS;
                for (int i = lane; i < 2 * per; i += 32) {
                    const bool is_v = i >= per;
                    const int j = is_v ? i - per : i;
                    const int r = 8 * q + j / C::CHUNKS, c16 = j % C::CHUNKS;
                    const uint8_t *src = (is_v ? vseg : kseg) + int64_t(row0 + r) * C::ROW_BYTES + c16 * 16;
                    dev::cp_async_16(C::M::swz(is_v ? vdst : kdst, r, c16 * 8), src);
                }
                dev::cp_async_arrive(full);
                generic_written |= 1u << stage;
            } else {
                generic_written &= ~(1u << stage);
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(full);
            ++issued;
        }
        __syncwarp();
        dev::named_barrier_sync(1, C::THREADS);
        if (lane == 0 && flags[0]) drain_copies(bar0, NS, issued, a.timeout_ns);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int gr = lane >> 2, tq = lane & 3;
    const int H = a.H_kv * G;
    const int k_key = ((lane >> 4) & 1) * 8 + (lane & 7);   // K as B: matrices (k0, d0) (k0, d8) (k8, d0) (k8, d8)
    const int k_col = ((lane >> 3) & 1) * 8;
    const int v_key = ((lane >> 3) & 1) * 8 + (lane & 7);   // V as B (.trans): (k0, d0) (k8, d0) (k0, d8) (k8, d8)
    const int v_col = ((lane >> 4) & 1) * 8;

    // this lane's two query rows (fragment rows gr and gr + 8 of the warp's 16)
    const int rA = r_first + cw * 16 + gr, rB = rA + 8;
    const bool okA = rA < r_end, okB = rB < r_end;
    const int tA = rA / G, iA = rA % G, tB = rB / G, iB = rB % G;
    const int limA = okA ? c + tA + 1 : 1, limB = okB ? c + tB + 1 : 1;  // keys < lim are visible
    const int lim_min = min(limA, limB);
    const T *q = reinterpret_cast<const T *>(a.q);
    const T *qA = q + ((int64_t(b) * H + kv * G + iA) * a.T_new + tA) * D;
    const T *qB = q + ((int64_t(b) * H + kv * G + iB) * a.T_new + tB) * D;
    uint32_t qa[KSTEPS][4];
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        const int col = ks * 16 + 2 * tq;
        qa[ks][0] = okA ? __ldg(reinterpret_cast<const uint32_t *>(qA + col)) : 0u;
        qa[ks][1] = okB ? __ldg(reinterpret_cast<const uint32_t *>(qB + col)) : 0u;
        qa[ks][2] = okA ? __ldg(reinterpret_cast<const uint32_t *>(qA + col + 8)) : 0u;
        qa[ks][3] = okB ? __ldg(reinterpret_cast<const uint32_t *>(qB + col + 8)) : 0u;
    }
    float o[NTD][4];
#pragma unroll
    for (int n = 0; n < NTD; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    // Tiles wholly past the limits of all 16 of this warp's rows contribute
    // nothing (the bound is warp-uniform: the tile work is warp-collective);
    // the warp still releases every stage of the CTA's range.
    const int rw0 = r_first + cw * 16;
    const int my_kend = rw0 < r_end ? c + (min(rw0 + 15, r_end - 1) / G) + 1 : 0;
    for (int t = 0; t < ntiles; ++t) {
        const int stage = t % NS;
        const uint32_t round = uint32_t(t / NS);
        bool ok = !flags[0] && dev::mbar_wait_bounded(bar0 + 8 * stage, round & 1, flags, a.timeout_ns);
        ok = __all_sync(FULL, ok);
        if (!ok) {
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
            break;
        }
        const int row0 = t * TILE, nr = min(TILE, kend - row0);
        if (row0 < my_kend) {
            const uint32_t ks_base = stage0 + uint32_t(stage) * C::STAGE_BYTES;
            const uint32_t vs_base = ks_base + C::TILE_BYTES;
            float s[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[4];
                    dev::ldsm_x4(C::M::swz(ks_base, half * 16 + k_key, ks * 16 + k_col), r);
                    Ops::mma(s[2 * half], qa[ks], r[0], r[1]);
                    Ops::mma(s[2 * half + 1], qa[ks], r[2], r[3]);
                }
            }
            if (row0 + TILE > lim_min) {  // the tile crosses a row's causal limit
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = row0 + n * 8 + 2 * tq + e;
                        if (key >= limA) s[n][e] = -INFINITY;
                        if (key >= limB) s[n][2 + e] = -INFINITY;
                    }
            }
            float xA = -INFINITY, xB = -INFINITY;
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                xA = fmaxf(xA, fmaxf(s[n][0], s[n][1]));
                xB = fmaxf(xB, fmaxf(s[n][2], s[n][3]));
            }
            xA = fmaxf(xA, __shfl_xor_sync(FULL, xA, 1));
            xA = fmaxf(xA, __shfl_xor_sync(FULL, xA, 2));
            xB = fmaxf(xB, __shfl_xor_sync(FULL, xB, 1));
            xB = fmaxf(xB, __shfl_xor_sync(FULL, xB, 2));
            // a row with every key of the tile masked keeps its state
            const float mnA = xA == -INFINITY ? mA : fmaxf(mA, xA * a.scale_log2);
            const float mnB = xB == -INFINITY ? mB : fmaxf(mB, xB * a.scale_log2);
            const float cA = mnA == -INFINITY ? 1.f : exp2f(mA - mnA);
            const float cB = mnB == -INFINITY ? 1.f : exp2f(mB - mnB);
            mA = mnA;
            mB = mnB;
            float pA = 0.f, pB = 0.f;
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                s[n][0] = exp2f(fmaf(s[n][0], a.scale_log2, -mnA));
                s[n][1] = exp2f(fmaf(s[n][1], a.scale_log2, -mnA));
                s[n][2] = exp2f(fmaf(s[n][2], a.scale_log2, -mnB));
                s[n][3] = exp2f(fmaf(s[n][3], a.scale_log2, -mnB));
                pA += s[n][0] + s[n][1];
                pB += s[n][2] + s[n][3];
            }
            lA = fmaf(lA, cA, pA);
            lB = fmaf(lB, cB, pB);
            if (__any_sync(FULL, (cA != 1.f) || (cB != 1.f))) {
#pragma unroll
                for (int n = 0; n < NTD; ++n) {
                    o[n][0] *= cA;
                    o[n][1] *= cA;
                    o[n][2] *= cB;
                    o[n][3] *= cB;
                }
            }
            uint32_t pa[2][4];
#pragma unroll
            for (int kst = 0; kst < 2; ++kst) {
                pa[kst][0] = Ops::pack(s[2 * kst][0], s[2 * kst][1]);
                pa[kst][1] = Ops::pack(s[2 * kst][2], s[2 * kst][3]);
                pa[kst][2] = Ops::pack(s[2 * kst + 1][0], s[2 * kst + 1][1]);
                pa[kst][3] = Ops::pack(s[2 * kst + 1][2], s[2 * kst + 1][3]);
            }
#pragma unroll
            for (int kst = 0; kst < 2; ++kst) {
#pragma unroll
                for (int dn = 0; dn < NTD / 2; ++dn) {
                    uint32_t r[4];
                    dev::ldsm_x4_trans(C::M::swz(vs_base, kst * 16 + v_key, dn * 16 + v_col), r);
                    if (nr < TILE) {  // stale rows past the copied ones
                        const int k0 = kst * 16 + 2 * tq;
                        r[0] = live_pair(r[0], k0, nr);
                        r[1] = live_pair(r[1], k0 + 8, nr);
                        r[2] = live_pair(r[2], k0, nr);
                        r[3] = live_pair(r[3], k0 + 8, nr);
                    }
                    Ops::mma(o[2 * dn], pa[kst], r[0], r[1]);
                    Ops::mma(o[2 * dn + 1], pa[kst], r[2], r[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(bar0 + 8 * (NS + stage));
    }

    // ---- normalise and write this lane's rows
    lA += __shfl_xor_sync(FULL, lA, 1);
    lA += __shfl_xor_sync(FULL, lA, 2);
    lB += __shfl_xor_sync(FULL, lB, 1);
    lB += __shfl_xor_sync(FULL, lB, 2);
    if (!flags[0]) {
        T *out = reinterpret_cast<T *>(a.out);
        T *oA = out + ((int64_t(b) * H + kv * G + iA) * a.T_new + tA) * D;
        T *oB = out + ((int64_t(b) * H + kv * G + iB) * a.T_new + tB) * D;
        const float invA = 1.f / lA, invB = 1.f / lB;
#pragma unroll
        for (int n = 0; n < NTD; ++n) {
            const int col = n * 8 + 2 * tq;
            if (okA) {
                oA[col] = E::round(o[n][0] * invA);
                oA[col + 1] = E::round(o[n][1] * invA);
            }
            if (okB) {
                oB[col] = E::round(o[n][2] * invB);
                oB[col + 1] = E::round(o[n][3] * invB);
            }
        }
    }
    dev::named_barrier_sync(1, C::THREADS);
}

template <typename T, int D, int G>
cudaError_t set_prefill_max_smem(int bytes) {
    return cudaFuncSetAttribute(prefill_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T, int D, int G>
cudaError_t launch_prefill(const PrefillArgs &a, int grid, int smem, cudaStream_t s) {
    return launch_pdl(prefill_kernel<T, D, G>, dim3(grid), dim3(PrefillCfg<T, D, G>::THREADS), smem, s, a);
}

template <typename T, int D, int G>
const PrefillKernelInfo *prefill_info() {
    using C = PrefillCfg<T, D, G>;
    static const PrefillKernelInfo info = {C::QROWS, C::SMEM, &set_prefill_max_smem<T, D, G>,
                                           &launch_prefill<T, D, G>};
    return &info;
}

}  // namespace kvc
