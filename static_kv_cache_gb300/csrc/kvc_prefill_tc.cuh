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
//   softmax              two threads own row r (its TMEM lane), one per half
//                        of the key tile (64 keys): tcgen05.ld of that half
//                        row, causal mask on the tiles that cross the row's
//                        limit, a running max and sum in fp32 (log2 domain)
//                        per half; P rounded to the cache type into shared
//                        memory (K-major, 128-byte swizzle)
//   O_h += P_h . V_h     tcgen05.mma per half h of the keys, N = d_h, into
//                        one tensor-memory accumulator per half; B = V_j as
//                        stored ([key][d]: the N dimension contiguous, an
//                        MN-major operand).  O_0 and O_1 stay in tensor memory
//                        for the whole key range.
// Each half raises its reference max only when a tile's maximum exceeds it
// by more than 2^8 (probabilities stay <= 256, no loss in fp32 or in P);
// only then is its accumulator rescaled in tensor memory (tcgen05.ld,
// multiply, tcgen05.st), after its previous P.V has completed.  The halves
// never wait for each other: the epilogue swaps their (max, sum) once and
// writes (O_0 e_0 + O_1 e_1) / (l_0 e_0 + l_1 e_1), e_h = 2^(m_h - max),
// rounded once to the cache type.
//
// Warps: 0-7 softmax and epilogue (two per TMEM lane quarter), 8 producer
// (TMA boxes of 128 keys x 64 columns, 128-byte swizzle; a ring of K tiles,
// released as soon as S has read them, and a ring of V tiles, released after
// P.V), 9 MMA issuer (one thread) and tensor-memory owner.  Rows past the chunk's last visible key
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
    static constexpr int KT_BYTES = CB * BLK;        // one K (or V) tile
    // K tiles are released as soon as S = Q.K^T has used them, V tiles only
    // after P.V: separate rings, the K ring the deeper
    static constexpr int NSK = D == 64 ? 4 : 2;
    static constexpr int NSV = D == 64 ? 4 : 2;
    // kfull[NSK], kempty[NSK], vfull[NSV], vempty[NSV], s_full[2],
    // p_full[2], p_free[2], q_full, mma_done, pair[4]
    static constexpr int NBAR = 2 * NSK + 2 * NSV + 12;
    static constexpr int BAR_OFF = Q_BYTES + P_BYTES + (NSK + NSV) * KT_BYTES;
    // the two softmax threads of a row swap their halves' running maxima and
    // sums here at the end: [2][half][row]
    static constexpr int XCH_OFF = BAR_OFF + 8 * NBAR + 32;  // after the TMEM address and the abort flag
    static constexpr int SMEM = 1024 + XCH_OFF + 2 * 2 * BM * 4;
    static constexpr int NSW = 8;                  // softmax warps: two per TMEM lane quarter
    static constexpr int THREADS = (NSW + 2) * 32;
    static constexpr uint32_t TMEM_COLS = 512;
    // two S buffers, then one O accumulator per half of the key tile
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL = 256;
    static_assert(O_COL + 2 * D <= TMEM_COLS, "two S buffers and two O accumulators in tensor memory");
    static constexpr float RESCALE_LOG2 = 8.f;

    static_assert(D == 64 || D == 128, "head width 64 or 128");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");

    // Address of 16-byte chunk c of row r in a swizzled 128-row tile.
    __device__ __forceinline__ static uint32_t swz(uint32_t tile, int r, int c) {
        return tile + uint32_t(c >> 3) * BLK + uint32_t(r) * 128 + (uint32_t((c & 7) ^ (r & 7)) << 4);
    }
};

// 2^x on the special-function unit (the PTX instruction; flushes subnormal
// results to zero, which only affects probabilities below 2^-126).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

template <typename T, int D>
__global__ void __launch_bounds__(TcPrefillCfg<T, D>::THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
    using C = TcPrefillCfg<T, D>;
    using Ops = MmaOps<T>;
    constexpr int BM = C::BM, BN = C::BN, CB = C::CB, NSK = C::NSK, NSV = C::NSV, BLK = C::BLK;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t IDESC_S = tc::idesc_f16_f32acc(BF16, BM, BN, false, false);
    constexpr uint32_t IDESC_O = tc::idesc_f16_f32acc(BF16, BM, D, false, true);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = dev::smem_addr(smem);
    const uint32_t q_s = sb, p_s = sb + C::Q_BYTES, k_s = p_s + C::P_BYTES, v_s = k_s + NSK * C::KT_BYTES;
    const uint32_t kfull = sb + C::BAR_OFF, kempty = kfull + 8 * NSK, vfull = kempty + 8 * NSK,
                   vempty = vfull + 8 * NSV;
    const uint32_t s_full = vempty + 8 * NSV, p_full = s_full + 16, p_free = p_full + 16, q_full = p_free + 16,
                   mma_done = q_full + 8, pair_bar = mma_done + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + 8 * C::NBAR);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::BAR_OFF + 8 * C::NBAR + 16);
    float *xch = reinterpret_cast<float *>(smem + C::XCH_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int PRODUCER = C::NSW, ISSUER = C::NSW + 1;  // the two single warps after the softmax warps

    const int G = a.group;
    const int TB = BM / G;                         // chunk tokens per CTA
    const int nseg = a.B * a.H_kv;
    const int qb = a.q_blocks - 1 - int(blockIdx.x) / nseg;  // the longest key ranges first
    const int seg = int(blockIdx.x) % nseg;
    const int b = seg / a.H_kv, kv = seg % a.H_kv;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&a.tm_k128);
        dev::prefetch_tensormap(&a.tm_v128);
        for (int s = 0; s < NSK; ++s) {
            dev::mbar_init(kfull + 8 * s, 1);   // TMA bytes (+ the producer's arrival)
            dev::mbar_init(kempty + 8 * s, 1);  // released by the commit after S = Q.K^T
        }
        for (int s = 0; s < NSV; ++s) {
            dev::mbar_init(vfull + 8 * s, 1);
            dev::mbar_init(vempty + 8 * s, 1);  // released by the commit after P.V
        }
        dev::mbar_init(s_full, 1);
        dev::mbar_init(s_full + 8, 1);
        for (int hf = 0; hf < 2; ++hf) {
            dev::mbar_init(p_full + 8 * hf, C::NSW / 2);  // the four softmax warps of a half
            dev::mbar_init(p_free + 8 * hf, 1);
        }
        dev::mbar_init(q_full, C::NSW);
        dev::mbar_init(mma_done, 1);
        for (int qd = 0; qd < 4; ++qd) dev::mbar_init(pair_bar + 8 * qd, 2);  // the two warps of a lane quarter
        flags[0] = 0;
        dev::fence_mbar_init();
    }
    if (warp == ISSUER) {
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

    int issued_k = 0, issued_v = 0;  // tiles whose copies the producer issued
    if (warp == PRODUCER) {
        // ------------------------------------------------------------ producer
        // K of tile j + 1 goes out before V of tile j: S needs K a whole
        // softmax earlier than P.V needs V.
        const int z = a.seg_base + seg;
        const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;
        const uint8_t *kseg = a.K + int64_t(seg) * kv_slab;
        const uint8_t *vseg = a.V + int64_t(seg) * kv_slab;
        uint32_t generic_k = 0, generic_v = 0;  // stages whose last fill had generic-proxy stores
        bool ok = true;
        // one tile of one tensor into one stage
        auto load = [&](bool is_v, int j, uint32_t dst, uint32_t full, uint32_t &generic, int s) {
            const int row0 = j * BN, nr = min(BN, kend - row0);
            const CUtensorMap *m128 = is_v ? &a.tm_v128 : &a.tm_k128;
            const CUtensorMap *m32 = is_v ? &a.tm_v32 : &a.tm_k32;
            const CUtensorMap *m8 = is_v ? &a.tm_v8 : &a.tm_k8;
            // generic-proxy stores of the stage's last fill come before the
            // TMA unit writes it again
            if (generic & (1u << s)) dev::fence_proxy_async_smem();
            if (nr == BN) {
                if (lane == 0) {
                    dev::mbar_arrive_expect_tx(full, uint32_t(BN) * C::ROW_BYTES);
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb) dev::tma_load_3d(dst + cb * BLK, m128, cb * 64, row0, z, full);
                }
                generic &= ~(1u << s);
                return;
            }
            // a partial tile: 32-row, then 8-row boxes over the live rows, the
            // remaining live rows by 16-byte loads, zeros after them
            const int n32 = nr >> 5, n8 = (nr >> 3) & 3, boxed = 32 * n32 + 8 * n8;
            if (lane == 0) {
                dev::mbar_expect_tx(full, uint32_t(boxed) * C::ROW_BYTES);
                for (int g = 0; g < n32; ++g)
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb)
                        dev::tma_load_3d(dst + cb * BLK + g * 32 * 128, m32, cb * 64, row0 + 32 * g, z, full);
                for (int g = 0; g < n8; ++g)
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb) {
                        const int r = 32 * n32 + 8 * g;
                        dev::tma_load_3d(dst + cb * BLK + r * 128, m8, cb * 64, row0 + r, z, full);
                    }
            }
            const uint8_t *src = (is_v ? vseg : kseg) + int64_t(row0) * C::ROW_BYTES;
            for (int i = lane; i < (BN - boxed) * C::CHUNKS; i += 32) {
                const int r = boxed + i / C::CHUNKS, c16 = i % C::CHUNKS;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < nr) v = __ldg(reinterpret_cast<const uint4 *>(src + int64_t(r) * C::ROW_BYTES) + c16);
                dev::st_shared_v4(C::swz(dst, r, c16), v);
            }
            dev::fence_proxy_async_smem();  // the tensor core reads these rows
            generic |= 1u << s;
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(full);
        };
        auto wait_free = [&](uint32_t empty, int j, int ns) {
            if (j < ns) return true;
            const bool w = dev::mbar_wait_bounded(empty, uint32_t(j / ns - 1) & 1, flags, a.timeout_ns);
            if (__all_sync(FULL, w)) return true;
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
            return false;
        };
        for (int j = 0; ok && j <= ntiles; ++j) {
            if (j < ntiles) {
                const int s = j % NSK;
                ok = wait_free(kempty + 8 * s, j, NSK);
                if (!ok) break;
                load(false, j, k_s + uint32_t(s) * C::KT_BYTES, kfull + 8 * s, generic_k, s);
                issued_k = j + 1;
            }
            if (j > 0) {
                const int jv = j - 1, s = jv % NSV;
                ok = wait_free(vempty + 8 * s, jv, NSV);
                if (!ok) break;
                load(true, jv, v_s + uint32_t(s) * C::KT_BYTES, vfull + 8 * s, generic_v, s);
                issued_v = jv + 1;
            }
        }
    } else if (warp == ISSUER) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = dev::mbar_wait_bounded(q_full, 0, flags, a.timeout_ns);
            tc::fence_after();
            for (int j = 0; ok && j <= ntiles; ++j) {
                if (j < ntiles) {
                    // S_j = Q . K_j^T into S buffer j % 2 (free: the softmax of
                    // tile j - 2 was waited for before P.V of tile j - 2)
                    const int s = j % NSK;
                    ok = dev::mbar_wait_bounded(kfull + 8 * s, uint32_t(j / NSK) & 1, flags, a.timeout_ns);
                    if (!ok) break;
                    tc::fence_after();
                    const uint32_t kt = k_s + uint32_t(s) * C::KT_BYTES;
                    const uint32_t s_t = tmem + ((j & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * BLK + (ks & 3) * 32;
                        tc::mma_f16_ss(s_t, tc::smem_desc_sw128(q_s + off, 16, 1024),
                                       tc::smem_desc_sw128(kt + off, 16, 1024), IDESC_S, ks > 0);
                    }
                    tc::commit(s_full + 8 * (j & 1));
                    tc::commit(kempty + 8 * s);  // K stage free
                }
                if (j > 0) {
                    // O_h += P_h . V_h for the two halves h of tile j - 1 (keys
                    // [64 h, 64 h + 64)), each once its softmax warps have
                    // written their half of P
                    const int jp = j - 1, sp = jp % NSV;
                    ok = dev::mbar_wait_bounded(vfull + 8 * sp, uint32_t(jp / NSV) & 1, flags, a.timeout_ns);
                    if (!ok) break;
                    const uint32_t vt = v_s + uint32_t(sp) * C::KT_BYTES;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        ok = dev::mbar_wait_bounded(p_full + 8 * hf, uint32_t(jp) & 1, flags, a.timeout_ns);
                        if (!ok) break;
                        tc::fence_after();
                        const uint32_t o_t = tmem + C::O_COL + uint32_t(hf) * D;
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_f16_ss(o_t, tc::smem_desc_sw128(p_s + hf * BLK + ks * 32, 16, 1024),
                                           tc::smem_desc_sw128(vt + hf * 8192 + ks * 2048, BLK, 1024), IDESC_O,
                                           (jp > 0 || ks > 0));
                        tc::commit(p_free + 8 * hf);  // this half of P free, O_h up to date
                    }
                    if (!ok) break;
                    tc::commit(vempty + 8 * sp);  // V stage free
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
        // Two warps per TMEM lane quarter: thread (qd, hf) owns row r of the
        // quarter and keys [64 hf, 64 hf + 64) of every tile, with its own
        // running max and sum and its own accumulator O_hf in tensor memory.
        // The halves never wait for each other; the epilogue combines them.
        const int qd = warp & 3, hf = warp >> 2;
        const int r = 32 * qd + lane;           // query row = TMEM lane
        const int i = r / TB, tt = r - i * TB;  // head of the group, token of the block
        const bool row_ok = !bad && i < G && tt < ntok;
        const int t = t0 + tt;
        const int H = a.H_kv * G;
        const int64_t row_elem = ((int64_t(b) * H + kv * G + i) * a.T_new + t) * D;
        const uint32_t pbar = pair_bar + 8 * qd;
        constexpr int QC = C::CHUNKS / 2;       // 16-byte chunks of Q (and of the output) per half row
        {
            // this half of the Q row into shared memory (K-major, swizzled)
            const uint4 *qrow = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.q) + row_elem);
#pragma unroll
            for (int c16 = hf * QC; c16 < (hf + 1) * QC; ++c16) {
                const uint4 v = row_ok ? __ldg(qrow + c16) : make_uint4(0u, 0u, 0u, 0u);
                dev::st_shared_v4(C::swz(q_s, r, c16), v);
            }
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(q_full);
        }
        const int limit = row_ok ? c + t : c;  // last visible key (unused rows: any finite range)
        const int lim_min = c + t0;            // smallest limit of the CTA's rows
        const uint32_t lane_base = uint32_t(qd * 32) << 16;
        const uint32_t o_t = tmem + lane_base + C::O_COL + uint32_t(hf) * D;  // this half's accumulator
        const uint32_t pf = p_free + 8 * hf;
        const float2 scale2 = make_float2(a.scale_log2, a.scale_log2);
        float m_run = -INFINITY;
        float2 l2 = make_float2(0.f, 0.f);     // running sum, two partial lanes
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            ok = !flags[0] && dev::mbar_wait_bounded(s_full + 8 * (j & 1), uint32_t(j >> 1) & 1, flags, a.timeout_ns);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc::fence_after();
            uint32_t sr[2][32];
            const uint32_t s_t = tmem + lane_base + ((j & 1) ? C::S_COL1 : C::S_COL0) + 64 * hf;
            tc::tmem_ld32(s_t, sr[0]);
            tc::tmem_ld32(s_t + 32, sr[1]);
            tc::tmem_ld_wait();
            tc::reg_fence(sr[0]);
            tc::reg_fence(sr[1]);
            const int key0 = j * BN + 64 * hf;
            if (key0 + 63 > lim_min) {  // this half tile crosses some row's causal limit
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (key0 + 32 * h2 + e > limit) sr[h2][e] = __float_as_uint(-INFINITY);
            }
            // maximum over four independent chains (no long dependency chain)
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(sr[h2][e]), __uint_as_float(sr[h2][e + 1]));
            const float m_tile = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * a.scale_log2;
            // raise the reference max only when the tile's exceeds it by 2^8
            const float m_new = m_tile > m_run + C::RESCALE_LOG2 ? m_tile : m_run;
            const float corr = m_new == m_run ? 1.f : ex2_approx(m_run - m_new);
            m_run = m_new;
            const float negm = m_run == -INFINITY ? 0.f : -m_run;
            const float2 neg2 = make_float2(negm, negm);
            float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 y = __ffma2_rn(make_float2(__uint_as_float(sr[h2][e]), __uint_as_float(sr[h2][e + 1])),
                                                scale2, neg2);
                    const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
                    ps[(e >> 1) & 3] = __fadd2_rn(ps[(e >> 1) & 3], make_float2(p0, p1));
                    pk[16 * h2 + e / 2] = Ops::pack(p0, p1);
                }
            l2 = __ffma2_rn(l2, make_float2(corr, corr), __fadd2_rn(__fadd2_rn(ps[0], ps[1]), __fadd2_rn(ps[2], ps[3])));
            if (j > 0) {
                // this half's P.V of the previous tile has read P and written O_hf
                ok = !flags[0] && dev::mbar_wait_bounded(pf, uint32_t(j - 1) & 1, flags, a.timeout_ns);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc::fence_after();
                if (__any_sync(FULL, corr != 1.f)) {
                    const float2 c2 = make_float2(corr, corr);
#pragma unroll
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        uint32_t o[32];
                        tc::tmem_ld32(o_t + 32 * q4, o);
                        tc::tmem_ld_wait();
                        tc::reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), c2);
                            o[e] = __float_as_uint(v.x);
                            o[e + 1] = __float_as_uint(v.y);
                        }
                        tc::tmem_st32(o_t + 32 * q4, o);
                    }
                    tc::tmem_st_wait();
                }
            }
            // this half of the P row into shared memory: the A operand of
            // O_hf += P_hf . V_hf (P block hf, keys [64 hf, 64 hf + 64))
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
                dev::st_shared_v4(C::swz(p_s, r, 8 * hf + cc),
                                  make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]));
            dev::fence_proxy_async_smem();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(p_full + 8 * hf);
        }
        if (!ok) {
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
        } else if (ntiles > 0) {
            // ---- epilogue: both halves' last P.V have completed; swap the
            // halves' (max, sum), then out = (O_0 e_0 + O_1 e_1) / (l_0 e_0 +
            // l_1 e_1) with e_h = 2^(m_h - max(m_0, m_1)), this thread taking
            // output columns [hf D/2, (hf + 1) D/2)
            ok = !flags[0] && dev::mbar_wait_bounded(p_free, uint32_t(ntiles - 1) & 1, flags, a.timeout_ns) &&
                 dev::mbar_wait_bounded(p_free + 8, uint32_t(ntiles - 1) & 1, flags, a.timeout_ns);
            ok = __all_sync(FULL, ok);
            const float l_me = l2.x + l2.y;
            if (ok) {
                xch[hf * BM + r] = m_run;
                xch[2 * BM + hf * BM + r] = l_me;
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(pbar);
                ok = __all_sync(FULL, dev::mbar_wait_bounded(pbar, 0, flags, a.timeout_ns));
            }
            if (ok) {
                tc::fence_after();
                const float m_ot = xch[(hf ^ 1) * BM + r], l_ot = xch[2 * BM + (hf ^ 1) * BM + r];
                const float m0 = hf ? m_ot : m_run, m1 = hf ? m_run : m_ot;
                const float l0 = hf ? l_ot : l_me, l1 = hf ? l_me : l_ot;
                const float M = fmaxf(m0, m1);  // finite: key 0 is visible to every row
                const float e0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - M);
                const float e1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - M);
                const float inv = 1.f / (l0 * e0 + l1 * e1);
                const float f0 = e0 * inv, f1 = e1 * inv;
                uint4 *orow = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(a.out) + row_elem) + hf * QC;
                const uint32_t oc = tmem + lane_base + C::O_COL + uint32_t(hf) * (D / 2);  // column hf D/2 of O_0
#pragma unroll
                for (int q4 = 0; q4 < D / 64; ++q4) {
                    uint32_t u[32], v[32];
                    tc::tmem_ld32(oc + 32 * q4, u);
                    tc::tmem_ld32(oc + D + 32 * q4, v);
                    tc::tmem_ld_wait();
                    tc::reg_fence(u);
                    tc::reg_fence(v);
                    float y[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        y[e] = fmaf(__uint_as_float(u[e]), f0, __uint_as_float(v[e]) * f1);
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        const uint4 w = make_uint4(Ops::pack(y[e], y[e + 1]), Ops::pack(y[e + 2], y[e + 3]),
                                                   Ops::pack(y[e + 4], y[e + 5]), Ops::pack(y[e + 6], y[e + 7]));
                        if (row_ok) orow[(32 * q4 + e) / 8] = w;
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
    if (warp == ISSUER) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (warp == PRODUCER && lane == 0 && flags[0]) {
        // after an abort, wait (bounded) for the copies that may still land
        const volatile int never = 0;
        for (int j = issued_k > NSK ? issued_k - NSK : 0; j < issued_k; ++j)
            dev::mbar_wait_bounded(kfull + 8 * (j % NSK), uint32_t(j / NSK) & 1, &never, a.timeout_ns);
        for (int j = issued_v > NSV ? issued_v - NSV : 0; j < issued_v; ++j)
            dev::mbar_wait_bounded(vfull + 8 * (j % NSV), uint32_t(j / NSV) & 1, &never, a.timeout_ns);
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
