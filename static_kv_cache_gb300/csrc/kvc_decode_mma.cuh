// kvc_decode_mma.cuh -- the decode attention of kvc_decode.cuh with the two
// contractions on the warp tensor-core path, for 16-bit caches and head
// groups of 2 to 8.
//
// Same mathematics, decomposition, pipeline protocol and merge as
// decode_split_kernel ("10.3 -- KV cache implementation details", section 5,
// attention bullet; GQA per section 4.2): only the per-tile arithmetic of a
// consumer warp changes.  With g query heads sharing a KV head, the tile of
// scores is a g x TILE product and P.V a g x d_h one.  On CUDA cores every
// cached element costs a widening instruction plus g/2 packed FMAs per
// contraction, which at g >= 2 keeps the SM busy issuing arithmetic rather
// than streaming; the mma.sync m16n8k16 tile (M = the g query rows, padded to
// 16) does the same work in a few instructions per 16 keys, with fp32
// accumulation exactly as before.
//
// Per 32-key tile a consumer warp (lane = 4 * gr + tq):
//   S[16 x 32] = Q[16 x D] . K^T : A = Q fragments (rows gr < g, loaded once
//     per piece), B = K rows via ldmatrix (K is row-major [key][d], which is
//     the column-major B operand), 4 n-tiles x D/16 k-steps.
//   softmax on the accumulator fragments: lane (gr, tq) holds scores of head
//     gr for keys 8n + 2tq + {0, 1}; a head's row lives in 4 lanes, so the
//     tile maximum takes two shuffles; scores are scaled by log2(e)/sqrt(D)
//     in fp32 after the product.
//   O[16 x D] += P . V : the S accumulator layout is the A-operand layout, so
//     P is rounded to the cache's 16-bit type in place; B = V via ldmatrix
//     .trans; 2 k-steps x D/8 n-tiles.
// K and V tiles reach shared memory through TMA tensor copies with the
// 128-byte swizzle (16-byte chunk c of row r of each 64-column block stored at
// chunk c ^ (r mod 8)), which makes every ldmatrix conflict-free.  A box only
// ever covers 8-row groups inside the live range (32 rows for a full tile, 8
// for the groups of a tail tile); the last (rows mod 8) rows of a tail tile
// are loaded by the producer warp's other lanes with plain 16-byte loads and
// stored at their swizzled positions, so rows past valid_len are never read.
// Rows past the copied ones in a tail tile hold stale bytes: their scores are
// replaced by -inf and their V fragments are zeroed in registers.
#pragma once

#include "kvc_decode.cuh"

namespace kvc {

template <typename T>
struct MmaOps;

template <>
struct MmaOps<__nv_bfloat16> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    __device__ __forceinline__ static void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        dev::mma_16816_bf16(d, a, b0, b1);
    }
};

template <>
struct MmaOps<__half> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        const __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    __device__ __forceinline__ static void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        dev::mma_16816_f16(d, a, b0, b1);
    }
};

template <typename T, int D, int G>
struct MmaCfg {
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int TILE = 32;                     // keys per tile
    static constexpr int BLOCK_BYTES = TILE * 128;      // one 64-column block of a tile
    static constexpr int TILE_BYTES = TILE * ROW_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
    static constexpr int CHUNKS = ROW_BYTES / 16;       // 16-byte chunks of a row
    static constexpr int KSTEPS = D / 16;               // k-steps of the score product
    static constexpr int NTD = D / 8;                   // n-tiles of the P.V product
    static constexpr int NW = 7;                        // consumer warps (+1 producer)
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr int SCR_ACC_FLOATS = NW * G * D;
    static constexpr int SCR_ML_FLOATS = NW * G * 2;
    // 1 KB of slack to align the stages to the 1024-byte swizzle atom
    static constexpr int FIXED_SMEM = 1024 + 4 * (SCR_ACC_FLOATS + SCR_ML_FLOATS) + 16;

    static_assert(sizeof(T) == 2, "the tensor-core path takes 16-bit caches");
    static_assert(G >= 1 && G <= 8, "the query group must fit the 8 live rows of an m16 tile");
    static_assert(D % 64 == 0, "head width must be a multiple of 64 (128-byte swizzle blocks)");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the swizzle-atom alignment");

    // Shared-memory address of (row r, element col) in a swizzled tile; col
    // is a multiple of 8 (one 16-byte chunk).
    __device__ __forceinline__ static uint32_t swz(uint32_t tile, int r, int col) {
        return tile + uint32_t(col >> 6) * BLOCK_BYTES + uint32_t(r) * 128 +
               uint32_t((((col >> 3) & 7) ^ (r & 7)) << 4);
    }
};

// The producer warp: walks the CTA's pieces; for each tile one lane issues
// the TMA boxes and the other lanes load the tail rows no box may cover.
template <typename C>
__device__ __forceinline__ uint32_t produce_tiles_tma(const DecodeArgs &a, Walker walk, uint32_t stage0,
                                                      uint32_t bar0, int ns, int64_t kv_slab,
                                                      volatile int *flags, int lane) {
    constexpr int TILE = C::TILE, CB = C::ROW_BYTES / 128;
    uint32_t issued = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    Piece pc;
    while (ok && walk.next(a, pc)) {
        const int seg = pc.b * a.H_kv + pc.kv;
        const int z = a.seg_base + seg;  // tensor-map segment coordinate
        const uint8_t *kseg = a.K + int64_t(seg) * kv_slab;
        const uint8_t *vseg = a.V + int64_t(seg) * kv_slab;
        for (int row0 = pc.lo; row0 < pc.hi; row0 += TILE) {
            const int nr = min(TILE, pc.hi - row0);
            if (round > 0) {
                const bool w =
                    dev::mbar_wait_bounded(bar0 + 8 * (ns + stage), (round - 1) & 1, flags, a.timeout_ns);
                if (!__all_sync(0xffffffffu, w)) {
                    if (lane == 0) {
                        if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                        flags[0] = 1;
                    }
                    ok = false;
                    break;
                }
            }
            const uint32_t full = bar0 + 8 * stage;
            const uint32_t kdst = stage0 + uint32_t(stage) * C::STAGE_BYTES;
            const uint32_t vdst = kdst + C::TILE_BYTES;
            const int q = nr >> 3, rem = nr & 7;  // 8-row groups, rows after them
            if (lane == 0) {
                dev::mbar_expect_tx(full, 2u * uint32_t(8 * q) * C::ROW_BYTES);
                if (q == 4) {
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb) {
                        dev::tma_load_3d(kdst + cb * C::BLOCK_BYTES, &a.tm_k32, cb * 64, row0, z, full);
                        dev::tma_load_3d(vdst + cb * C::BLOCK_BYTES, &a.tm_v32, cb * 64, row0, z, full);
                    }
                } else {
                    for (int j = 0; j < q; ++j)
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb) {
                            const uint32_t off = cb * C::BLOCK_BYTES + j * 8 * 128;
                            dev::tma_load_3d(kdst + off, &a.tm_k8, cb * 64, row0 + 8 * j, z, full);
                            dev::tma_load_3d(vdst + off, &a.tm_v8, cb * 64, row0 + 8 * j, z, full);
                        }
                }
            }
            if (rem) {
                const int per = rem * C::CHUNKS;  // 16-byte chunks per tensor
                for (int i = lane; i < 2 * per; i += 32) {
                    const bool is_v = i >= per;
                    const int j = is_v ? i - per : i;
                    const int r = 8 * q + j / C::CHUNKS, c16 = j % C::CHUNKS;
                    const uint8_t *src = (is_v ? vseg : kseg) + int64_t(row0 + r) * C::ROW_BYTES + c16 * 16;
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
                    dev::st_shared_v4(C::swz(is_v ? vdst : kdst, r, c16 * 8), v);
                }
                dev::fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(full);
            ++issued;
            if (++stage == ns) {
                stage = 0;
                ++round;
            }
        }
    }
    return issued;
}

// Zero the halves of a 32-bit pair of keys (k, k + 1) that are not live.
__device__ __forceinline__ uint32_t live_pair(uint32_t r, int k, int nr) {
    return r & ((k < nr ? 0x0000ffffu : 0u) | (k + 1 < nr ? 0xffff0000u : 0u));
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(MmaCfg<T, D, G>::THREADS, 1)
    decode_mma_kernel(const __grid_constant__ DecodeArgs a) {
    using C = MmaCfg<T, D, G>;
    using Ops = MmaOps<T>;
    constexpr int NW = C::NW, TILE = C::TILE, KSTEPS = C::KSTEPS, NTD = C::NTD;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int ns = a.n_stages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t stage0 = dev::smem_addr(smem);
    const uint32_t bar0 = stage0 + uint32_t(ns) * C::STAGE_BYTES;  // full[ns], then empty[ns]
    float *scr_acc = reinterpret_cast<float *>(smem + size_t(ns) * C::STAGE_BYTES + 16 * size_t(ns));
    float *scr_ml = scr_acc + C::SCR_ACC_FLOATS;
    volatile int *flags = reinterpret_cast<volatile int *>(scr_ml + C::SCR_ML_FLOATS);  // abort, last

    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            dev::mbar_init(bar0 + 8 * s, 1);
            dev::mbar_init(bar0 + 8 * (ns + s), 1);
        }
        flags[0] = 0;
        flags[1] = 0;
        dev::fence_mbar_init();
    }
    __syncthreads();

    const Plan plan = make_plan(a, lane);
    if (plan.r0 >= plan.r1 || plan.b >= a.B) return;  // uniform over the CTA

    Walker walk;
    walk.init(a, plan);
    const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;

    // ---------------------------------------------------------------- producer
    if (warp == 0) {
        const uint32_t issued = produce_tiles_tma<C>(a, walk, stage0, bar0, ns, kv_slab, flags, lane);
        __syncwarp();
        dev::named_barrier_sync(2, C::THREADS);  // every warp is done
        if (lane == 0 && flags[0]) drain_copies(bar0, ns, issued, a.timeout_ns);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int ctid = threadIdx.x - 32;
    const int gr = lane >> 2;  // row of the m16 tile = query head within the group
    const int tq = lane & 3;   // quad lane
    const int H = a.H_kv * G;
    // ldmatrix row addresses (see the layouts above)
    const int k_key = ((lane >> 4) & 1) * 8 + (lane & 7);   // score B: matrices (k0, d0) (k0, d8) (k8, d0) (k8, d8)
    const int k_col = ((lane >> 3) & 1) * 8;
    const int v_key = ((lane >> 3) & 1) * 8 + (lane & 7);   // P.V B: matrices (k0, d0) (k8, d0) (k0, d8) (k8, d8)
    const int v_col = ((lane >> 4) & 1) * 8;

    uint32_t qa[KSTEPS][2];
    float o[NTD][4];
    float m, l;
    uint32_t t = 0;
    int stage = 0;
    uint32_t round = 0;
    Piece pc;
    while (walk.next(a, pc)) {
        {
            const T *qrow = reinterpret_cast<const T *>(a.q) + (int64_t(pc.b) * H + pc.kv * G + gr) * D;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                qa[ks][0] = gr < G ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * tq)) : 0u;
                qa[ks][1] = gr < G ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + 2 * tq)) : 0u;
            }
#pragma unroll
            for (int n = 0; n < NTD; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            m = -INFINITY;
            l = 0.f;
        }

        for (int row0 = pc.lo; row0 < pc.hi; row0 += TILE, ++t) {
            const int cur_stage = stage;
            const uint32_t cur_round = round;
            if (++stage == ns) {
                stage = 0;
                ++round;
            }
            if (int(t % NW) != cw) continue;
            const int nr = min(TILE, pc.hi - row0);
            // Wait for the previous release of this stage first, then for its
            // data: the reasoning is the one in decode_split_kernel.
            const uint32_t full_bar = bar0 + 8 * cur_stage;
            const uint32_t empty_bar = bar0 + 8 * (ns + cur_stage);
            bool ok = !flags[0] &&
                      (cur_round == 0 ||
                       dev::mbar_wait_bounded(empty_bar, (cur_round - 1) & 1, flags, a.timeout_ns)) &&
                      dev::mbar_wait_bounded(full_bar, cur_round & 1, flags, a.timeout_ns);
            ok = __all_sync(FULL, ok);
            if (!ok) {
                if (lane == 0) {
                    if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                    flags[0] = 1;
                }
                continue;
            }
            const uint32_t ks_base = stage0 + uint32_t(cur_stage) * C::STAGE_BYTES;
            const uint32_t vs_base = ks_base + C::TILE_BYTES;

            // ---- scores S = Q . K^T for 32 keys (4 n-tiles of 8)
            float sacc[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const uint32_t afr[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[4];
                    dev::ldsm_x4(C::swz(ks_base, half * 16 + k_key, ks * 16 + k_col), r);
                    Ops::mma(sacc[2 * half], afr, r[0], r[1]);
                    Ops::mma(sacc[2 * half + 1], afr, r[2], r[3]);
                }
            }

            // ---- online softmax for head gr (row gr of the tile, held by 4 lanes)
            float p[8];
            float tmax = -INFINITY;
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = n * 8 + 2 * tq + e;
                    p[n * 2 + e] = key < nr ? sacc[n][e] * a.scale_log2 : -INFINITY;
                    tmax = fmaxf(tmax, p[n * 2 + e]);
                }
            tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, 1));
            tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, 2));
            const float mn = fmaxf(m, tmax);
            const float corr = exp2f(m - mn);
            m = mn;
            float psum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                p[i] = exp2f(p[i] - mn);
                psum += p[i];
            }
            l = fmaf(l, corr, psum);
            if (__any_sync(FULL, corr != 1.f)) {
#pragma unroll
                for (int n = 0; n < NTD; ++n) {
                    o[n][0] *= corr;
                    o[n][1] *= corr;
                }
            }
            uint32_t pa[4];
#pragma unroll
            for (int n = 0; n < 4; ++n) pa[n] = Ops::pack(p[2 * n], p[2 * n + 1]);

            // ---- O += P . V over the tile's two 16-key steps
#pragma unroll
            for (int kst = 0; kst < 2; ++kst) {
                const uint32_t afr[4] = {pa[2 * kst], 0u, pa[2 * kst + 1], 0u};
#pragma unroll
                for (int dn = 0; dn < NTD / 2; ++dn) {
                    uint32_t r[4];
                    dev::ldsm_x4_trans(C::swz(vs_base, kst * 16 + v_key, dn * 16 + v_col), r);
                    if (nr < TILE) {  // stale rows past the copied ones
                        const int k0 = kst * 16 + 2 * tq;
                        r[0] = live_pair(r[0], k0, nr);
                        r[1] = live_pair(r[1], k0 + 8, nr);
                        r[2] = live_pair(r[2], k0, nr);
                        r[3] = live_pair(r[3], k0 + 8, nr);
                    }
                    Ops::mma(o[2 * dn], afr, r[0], r[1]);
                    Ops::mma(o[2 * dn + 1], afr, r[2], r[3]);
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(empty_bar);
        }

        // ---- end of piece: this warp's state to shared memory, then merge
        l += __shfl_xor_sync(FULL, l, 1);
        l += __shfl_xor_sync(FULL, l, 2);
        if (gr < G) {
#pragma unroll
            for (int n = 0; n < NTD; ++n)
                *reinterpret_cast<float2 *>(scr_acc + (cw * G + gr) * D + n * 8 + 2 * tq) =
                    make_float2(o[n][0], o[n][1]);
            if (tq == 0) {
                scr_ml[(cw * G + gr) * 2] = m;
                scr_ml[(cw * G + gr) * 2 + 1] = l;
            }
        }
        dev::named_barrier_sync(1, NW * 32);
        merge_piece<T, D, G, NW>(a, plan, pc, scr_acc, scr_ml, flags, ctid);
    }
    dev::named_barrier_sync(2, C::THREADS);
}

template <typename T, int D, int G>
cudaError_t set_mma_max_smem(int bytes) {
    return cudaFuncSetAttribute(decode_mma_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                bytes);
}

template <typename T, int D, int G>
cudaError_t launch_mma(const DecodeArgs &a, int grid, int smem, cudaStream_t s) {
    decode_mma_kernel<T, D, G><<<grid, MmaCfg<T, D, G>::THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int D, int G>
const DecodeKernelInfo *mma_decode_info() {
    using C = MmaCfg<T, D, G>;
    static const DecodeKernelInfo info = {C::TILE, C::NW, C::STAGE_BYTES + 16, C::FIXED_SMEM,
                                          &set_mma_max_smem<T, D, G>, &launch_mma<T, D, G>, true};
    return &info;
}

}  // namespace kvc
