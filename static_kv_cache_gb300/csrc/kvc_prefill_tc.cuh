// kvc_prefill_tc.cuh -- chunked-prefill attention on the fifth-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// "KV-Cache Mechanics", AR Static KV-Cache: prefill is a forward pass over
// the prompt that fills the pre-allocated cache from cache_index; decoding
// continues where it stopped.  "10.3 -- KV cache implementation details",
// section 3: prefill processes the prompt's positions together and is
// compute-bound.  With the chunk's T_new rows already appended at
// cache_index c, the query of chunk position t attends causally over cache
// rows [0, c + t] (the causal reading: the one under which one pass, chunks
// and decode steps agree).
//
// One CTA takes BM = 128 query rows of one (sequence, KV head): the g heads
// of the group for TB = 128 / g consecutive chunk tokens, head-major (row
// r = i * TB + tt is head i, token t0 + tt), and every key its last token
// can see, in tiles of BN = 128 keys.  Per key tile j:
//   S_j = Q . K_j^T      tcgen05.mma, M = 128 rows, N = 128 keys, K = d_h;
//                        A = Q and B = K_j K-major in shared memory, S in
//                        tensor memory (two buffers, so S_{j+1} is computed
//                        while the softmax works on S_j)
//   softmax              thread r of the four softmax warps owns row r (its
//                        TMEM lane): tcgen05.ld of the row, causal mask on
//                        the tiles that cross a row's limit, running max and
//                        sum in fp32 (log2 domain); P rounded to the cache
//                        type into shared memory (K-major, 128-byte swizzle)
//   O += P_j . V_j       tcgen05.mma, N = d_h; B = V_j as stored ([key][d]:
//                        the N dimension contiguous, an MN-major operand); O
//                        stays in tensor memory for the whole key range.
// The running max is only raised when a tile's maximum exceeds it by more
// than 2^8 (probabilities stay <= 256, no loss in fp32 or in P); only then
// is the row of O in tensor memory rescaled (tcgen05.ld, multiply,
// tcgen05.st), after the previous P.V has completed.  The final O / l is
// rounded once to the cache type.
//
// Warps: 0-3 softmax and epilogue, 4 producer (TMA boxes of 128 keys x 64
// columns, 128-byte swizzle, two stages of K and V), 5 MMA issuer (one
// thread) and tensor-memory owner.  Rows past the chunk's last visible key
// are never read: a partial last tile is boxed in 32- and 8-row groups, its
// remaining live rows copied by the producer's lanes, the rest zeroed.  Every
// wait is bounded; a timeout records KVC_ERR_TIMEOUT, every role leaves its
// loop, the MMA issuer waits for its MMAs, the producer for its copies, and
// tensor memory is freed before the CTA exits.
#pragma once

#include <type_traits>

#include "kvc_decode_mma.cuh"
#include "kvc_tcgen05.cuh"

namespace kvc {

template <typename T, int D>
struct TcPrefillCfg {
    static constexpr int BM = 128;                 // query rows per CTA (TMEM lanes)
    static constexpr int BN = 128;                 // keys per tile
    static constexpr int CB = D / 64;              // 128-byte column blocks of a row
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int CHUNKS = ROW_BYTES / 16;  // 16-byte chunks of a row
    static constexpr int BLK = 128 * 128;          // one column block of a 128-row tile
    static constexpr int Q_BYTES = CB * BLK;
    static constexpr int P_BYTES = (BN / 64) * BLK;
    static constexpr int KT_BYTES = CB * BLK;
    static constexpr int STAGE_BYTES = 2 * KT_BYTES;  // K tile, then V tile
    static constexpr int NS = D == 64 ? 4 : 2;
    // full[NS], empty[NS], s_full[2], p_full, p_free, q_full, mma_done
    static constexpr int NBAR = 2 * NS + 6;
    static constexpr int BAR_OFF = Q_BYTES + P_BYTES + NS * STAGE_BYTES;
    static constexpr int SMEM = 1024 + BAR_OFF + 8 * NBAR + 32;  // + TMEM address, abort flag
    static constexpr int THREADS = 192;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL = 256;
    static constexpr float RESCALE_LOG2 = 8.f;

    static_assert(D == 64 || D == 128, "head width 64 or 128");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");

    // Address of 16-byte chunk c of row r in a swizzled 128-row tile.
    __device__ __forceinline__ static uint32_t swz(uint32_t tile, int r, int c) {
        return tile + uint32_t(c >> 3) * BLK + uint32_t(r) * 128 + (uint32_t((c & 7) ^ (r & 7)) << 4);
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(TcPrefillCfg<T, D>::THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
    using C = TcPrefillCfg<T, D>;
    using Ops = MmaOps<T>;
    constexpr int BM = C::BM, BN = C::BN, CB = C::CB, NS = C::NS, BLK = C::BLK;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t IDESC_S = tc::idesc_f16_f32acc(BF16, BM, BN, false, false);
    constexpr uint32_t IDESC_O = tc::idesc_f16_f32acc(BF16, BM, D, false, true);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = dev::smem_addr(smem);
    const uint32_t q_s = sb, p_s = sb + C::Q_BYTES, st_s = p_s + C::P_BYTES;
    const uint32_t bar = sb + C::BAR_OFF;  // full[NS], empty[NS], then the single barriers
    const uint32_t s_full = bar + 16 * NS, p_full = s_full + 16, p_free = p_full + 8, q_full = p_free + 8,
                   mma_done = q_full + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + 8 * C::NBAR);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::BAR_OFF + 8 * C::NBAR + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int G = a.group;
    const int TB = BM / G;                         // chunk tokens per CTA
    const int nseg = a.B * a.H_kv;
    const int qb = a.q_blocks - 1 - int(blockIdx.x) / nseg;  // the longest key ranges first
    const int seg = int(blockIdx.x) % nseg;
    const int b = seg / a.H_kv, kv = seg % a.H_kv;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&a.tm_k128);
        dev::prefetch_tensormap(&a.tm_v128);
        for (int s = 0; s < NS; ++s) {
            dev::mbar_init(bar + 8 * s, 1);         // TMA bytes (+ the producer's arrival)
            dev::mbar_init(bar + 8 * (NS + s), 1);  // released by the commit after P.V
        }
        dev::mbar_init(s_full, 1);
        dev::mbar_init(s_full + 8, 1);
        dev::mbar_init(p_full, 4);   // one arrival per softmax warp
        dev::mbar_init(p_free, 1);
        dev::mbar_init(q_full, 4);
        dev::mbar_init(mma_done, 1);
        flags[0] = 0;
        dev::fence_mbar_init();
    }
    if (warp == 5) {
        tc::tmem_alloc(dev::smem_addr(tmem_slot), C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    // everything above overlaps the previous kernel on the stream (the chunk's
    // append); nothing below runs before it has completed
    dev::grid_dependency_wait();
    dev::allow_dependents();
    const int c = __ldg(a.cache_index + b);
    const bool bad = c < 0 || c > a.max_ctx - a.T_new;
    if (bad && threadIdx.x == 0 && kv == 0 && qb == 0) dev::record_error(a.err, ERR_DEVICE_INDEX);
    const int t0 = qb * TB;
    const int ntok = min(TB, a.T_new - t0);
    const int kend = c + t0 + ntok;  // keys [0, kend) are visible to some row of the CTA
    const int ntiles = bad ? 0 : (kend + BN - 1) / BN;

    int issued = 0;  // tiles whose copies the producer issued
    if (warp == 4) {
        // ------------------------------------------------------------ producer
        const int z = a.seg_base + seg;
        const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;
        const uint8_t *kseg = a.K + int64_t(seg) * kv_slab;
        const uint8_t *vseg = a.V + int64_t(seg) * kv_slab;
        uint32_t generic_written = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int s = j % NS;
            const uint32_t round = uint32_t(j / NS);
            if (round > 0) {
                const bool w = dev::mbar_wait_bounded(bar + 8 * (NS + s), (round - 1) & 1, flags, a.timeout_ns);
                if (!__all_sync(FULL, w)) {
                    if (lane == 0) {
                        if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                        flags[0] = 1;
                    }
                    break;
                }
            }
            const int row0 = j * BN, nr = min(BN, kend - row0);
            const uint32_t full = bar + 8 * s;
            const uint32_t kdst = st_s + uint32_t(s) * C::STAGE_BYTES, vdst = kdst + C::KT_BYTES;
            // the stage's last fill had generic-proxy stores: order them
            // before the TMA unit writes it again
            if (generic_written & (1u << s)) dev::fence_proxy_async_smem();
            if (nr == BN) {
                if (lane == 0) {
                    dev::mbar_arrive_expect_tx(full, 2u * BN * C::ROW_BYTES);
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb) {
                        dev::tma_load_3d(kdst + cb * BLK, &a.tm_k128, cb * 64, row0, z, full);
                        dev::tma_load_3d(vdst + cb * BLK, &a.tm_v128, cb * 64, row0, z, full);
                    }
                }
                generic_written &= ~(1u << s);
            } else {
                // a partial tile: 32-row, then 8-row boxes over the live rows,
                // the remaining live rows by 16-byte loads, zeros after them
                const int n32 = nr >> 5, n8 = (nr >> 3) & 3, boxed = 32 * n32 + 8 * n8;
                if (lane == 0) {
                    dev::mbar_expect_tx(full, 2u * uint32_t(boxed) * C::ROW_BYTES);
                    for (int g = 0; g < n32; ++g)
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb) {
                            const uint32_t off = cb * BLK + g * 32 * 128;
                            dev::tma_load_3d(kdst + off, &a.tm_k32, cb * 64, row0 + 32 * g, z, full);
                            dev::tma_load_3d(vdst + off, &a.tm_v32, cb * 64, row0 + 32 * g, z, full);
                        }
                    for (int g = 0; g < n8; ++g)
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb) {
                            const int r = 32 * n32 + 8 * g;
                            const uint32_t off = cb * BLK + r * 128;
                            dev::tma_load_3d(kdst + off, &a.tm_k8, cb * 64, row0 + r, z, full);
                            dev::tma_load_3d(vdst + off, &a.tm_v8, cb * 64, row0 + r, z, full);
                        }
                }
                const int per = (BN - boxed) * C::CHUNKS;  // 16-byte chunks per tensor after the boxes
                for (int i = lane; i < 2 * per; i += 32) {
                    const bool is_v = i >= per;
                    const int jj = is_v ? i - per : i;
                    const int r = boxed + jj / C::CHUNKS, c16 = jj % C::CHUNKS;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (r < nr)
                        v = __ldg(reinterpret_cast<const uint4 *>((is_v ? vseg : kseg) +
                                                                  int64_t(row0 + r) * C::ROW_BYTES) + c16);
                    dev::st_shared_v4(C::swz(is_v ? vdst : kdst, r, c16), v);
                }
                dev::fence_proxy_async_smem();  // the tensor core reads these rows
                generic_written |= 1u << s;
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(full);
            }
            issued = j + 1;
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = dev::mbar_wait_bounded(q_full, 0, flags, a.timeout_ns);
            tc::fence_after();
            const uint32_t o_t = tmem + C::O_COL;
            for (int j = 0; ok && j <= ntiles; ++j) {
                if (j < ntiles) {
                    // S_j = Q . K_j^T into S buffer j % 2 (free: the softmax of
                    // tile j - 2 was waited for before P.V of tile j - 2)
                    const int s = j % NS;
                    ok = dev::mbar_wait_bounded(bar + 8 * s, uint32_t(j / NS) & 1, flags, a.timeout_ns);
                    if (!ok) break;
                    tc::fence_after();
                    const uint32_t kt = st_s + uint32_t(s) * C::STAGE_BYTES;
                    const uint32_t s_t = tmem + ((j & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * BLK + (ks & 3) * 32;
                        tc::mma_f16_ss(s_t, tc::smem_desc_sw128(q_s + off, 16, 1024),
                                       tc::smem_desc_sw128(kt + off, 16, 1024), IDESC_S, ks > 0);
                    }
                    tc::commit(s_full + 8 * (j & 1));
                }
                if (j > 0) {
                    // O += P_{j-1} . V_{j-1}, once the softmax has written P
                    const int jp = j - 1, sp = jp % NS;
                    ok = dev::mbar_wait_bounded(p_full, uint32_t(jp) & 1, flags, a.timeout_ns);
                    if (!ok) break;
                    tc::fence_after();
                    const uint32_t vt = st_s + uint32_t(sp) * C::STAGE_BYTES + C::KT_BYTES;
#pragma unroll
                    for (int ks = 0; ks < BN / 16; ++ks) {
                        tc::mma_f16_ss(o_t, tc::smem_desc_sw128(p_s + (ks >> 2) * BLK + (ks & 3) * 32, 16, 1024),
                                       tc::smem_desc_sw128(vt + ks * 2048, BLK, 1024), IDESC_O, (jp > 0 || ks > 0));
                    }
                    tc::commit(bar + 8 * (NS + sp));  // K/V stage free
                    tc::commit(p_free);               // P buffer free, O up to date
                }
            }
            if (!ok) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
            // every MMA issued here has completed before tensor memory is freed
            tc::commit(mma_done);
            const volatile int never = 0;
            dev::mbar_wait_bounded(mma_done, 0, &never, a.timeout_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int r = threadIdx.x;              // query row = TMEM lane
        const int i = r / TB, tt = r - i * TB;  // head of the group, token of the block
        const bool row_ok = !bad && i < G && tt < ntok;
        const int t = t0 + tt;
        const int H = a.H_kv * G;
        const int64_t row_elem = ((int64_t(b) * H + kv * G + i) * a.T_new + t) * D;
        {
            // Q row into shared memory (K-major, swizzled); unused rows zero
            const uint4 *qrow = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.q) + row_elem);
#pragma unroll
            for (int c16 = 0; c16 < C::CHUNKS; ++c16) {
                const uint4 v = row_ok ? __ldg(qrow + c16) : make_uint4(0u, 0u, 0u, 0u);
                dev::st_shared_v4(C::swz(q_s, r, c16), v);
            }
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(q_full);
        }
        const int limit = row_ok ? c + t : c;  // last visible key (unused rows: any finite range)
        const int lim_min = c + t0;            // smallest limit of the CTA's rows
        const uint32_t lane_base = uint32_t(warp * 32) << 16;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            ok = !flags[0] && dev::mbar_wait_bounded(s_full + 8 * (j & 1), uint32_t(j >> 1) & 1, flags, a.timeout_ns);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc::fence_after();
            uint32_t sr[4][32];
            const uint32_t s_t = tmem + lane_base + ((j & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(s_t + 32 * q4, sr[q4]);
            tc::tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tc::reg_fence(sr[q4]);
            const int key0 = j * BN;
            if (key0 + BN - 1 > lim_min) {  // the tile crosses some row's causal limit
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (key0 + 32 * q4 + e > limit) sr[q4][e] = __float_as_uint(-INFINITY);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sr[q4][e]));
            const float m_tile = mx * a.scale_log2;
            // raise the reference max only when the tile's exceeds it by 2^8
            const float m_new = m_tile > m_run + C::RESCALE_LOG2 ? m_tile : m_run;
            const float corr = m_new == m_run ? 1.f : exp2f(m_run - m_new);
            m_run = m_new;
            const float neg = m_run == -INFINITY ? 0.f : -m_run;
            float psum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float p0 = exp2f(fmaf(__uint_as_float(sr[q4][e]), a.scale_log2, neg));
                    const float p1 = exp2f(fmaf(__uint_as_float(sr[q4][e + 1]), a.scale_log2, neg));
                    psum += p0 + p1;
                    pk[16 * q4 + e / 2] = Ops::pack(p0, p1);
                }
            l_run = fmaf(l_run, corr, psum);
            if (j > 0) {
                // P.V of the previous tile has read P and written O
                ok = !flags[0] && dev::mbar_wait_bounded(p_free, uint32_t(j - 1) & 1, flags, a.timeout_ns);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc::fence_after();
                if (__any_sync(FULL, corr != 1.f)) {
#pragma unroll
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        uint32_t o[32];
                        const uint32_t o_t = tmem + lane_base + C::O_COL + 32 * q4;
                        tc::tmem_ld32(o_t, o);
                        tc::tmem_ld_wait();
                        tc::reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                        tc::tmem_st32(o_t, o);
                    }
                    tc::tmem_st_wait();
                }
            }
            // P row into shared memory: the A operand of O += P . V
#pragma unroll
            for (int c16 = 0; c16 < BN / 8; ++c16)
                dev::st_shared_v4(C::swz(p_s, r, c16),
                                  make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]));
            dev::fence_proxy_async_smem();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(p_full);
        }
        if (!ok) {
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
        } else if (ntiles > 0) {
            // ---- epilogue: out = O / l, once the last P.V has completed
            ok = !flags[0] && dev::mbar_wait_bounded(p_free, uint32_t(ntiles - 1) & 1, flags, a.timeout_ns);
            ok = __all_sync(FULL, ok);
            if (ok) {
                tc::fence_after();
                const float inv = 1.f / l_run;
                uint4 *orow = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(a.out) + row_elem);
#pragma unroll
                for (int q4 = 0; q4 < D / 32; ++q4) {
                    uint32_t o[32];
                    tc::tmem_ld32(tmem + lane_base + C::O_COL + 32 * q4, o);
                    tc::tmem_ld_wait();
                    tc::reg_fence(o);
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        const uint4 v = make_uint4(
                            Ops::pack(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                            Ops::pack(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                            Ops::pack(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                            Ops::pack(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
                        if (row_ok) orow[(32 * q4 + e) / 8] = v;
                    }
                }
            } else if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
        }
    }

    // ---- teardown: every role is done; the MMAs have completed
    tc::fence_before();
    __syncthreads();
    if (warp == 5) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (warp == 4 && lane == 0 && flags[0]) {
        // after an abort, wait (bounded) for the copies that may still land
        const volatile int never = 0;
        for (int j = issued > NS ? issued - NS : 0; j < issued; ++j)
            dev::mbar_wait_bounded(bar + 8 * (j % NS), uint32_t(j / NS) & 1, &never, a.timeout_ns);
    }
}

template <typename T, int D>
cudaError_t set_prefill_tc_max_smem(int bytes) {
    return cudaFuncSetAttribute(prefill_tc_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T, int D>
cudaError_t launch_prefill_tc(const PrefillArgs &a, int grid, int smem, cudaStream_t s) {
    return launch_pdl(prefill_tc_kernel<T, D>, dim3(grid), dim3(TcPrefillCfg<T, D>::THREADS), smem, s, a);
}

template <typename T, int D>
const PrefillKernelInfo *prefill_tc_info() {
    using C = TcPrefillCfg<T, D>;
    static const PrefillKernelInfo info = {C::BM, C::SMEM, &set_prefill_tc_max_smem<T, D>, &launch_prefill_tc<T, D>};
    return &info;
}

}  // namespace kvc
