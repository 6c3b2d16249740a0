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
// Work item: BM = 128 query rows of one (sequence, KV head) -- the g heads
// of the group for TB = 128 / g consecutive chunk tokens, head-major (row
// r = i * TB + tt is head i, token t0 + tt) -- and every key its last token
// can see, in tiles of BN = 128 keys.  Per key tile j:
//   S_j = Q . K_j^T      tcgen05.mma, M = 128 rows, N = 128 keys, K = d_h;
//                        A = Q and B = K_j K-major in shared memory, S in
//                        tensor memory (two buffers, so S_{j+1} is computed
//                        while the softmax works on S_j)
//   softmax              two threads own row r (its TMEM lane), one per half
//                        of the key tile (64 keys): tcgen05.ld of that half
//                        row, causal mask on the tiles that cross the row's
//                        limit, a running max and sum in fp32 (log2 domain)
//                        per half; P rounded to the cache type and stored
//                        back into tensor memory over the S columns already
//                        read (tcgen05.st)
//   O_h += P_h . V_h     tcgen05.mma per half h of the keys, N = d_h, A = P_h
//                        from tensor memory, into one tensor-memory
//                        accumulator per half; B = V_j as stored ([key][d]:
//                        the N dimension contiguous, an MN-major operand).
// Each half raises its reference max only when a tile's maximum exceeds it
// by more than 2^8 (probabilities stay <= 256, no loss in fp32 or in P);
// only then is its accumulator rescaled in tensor memory (tcgen05.ld,
// multiply, tcgen05.st), after its previous P.V has completed.  The halves
// never wait for each other during the item: its epilogue swaps their (max,
// sum) once and writes (O_0 e_0 + O_1 e_1) / (l_0 e_0 + l_1 e_1), e_h =
// 2^(m_h - max), rounded once to the cache type.
//
// The kernel is persistent: one CTA per SM walks its share of the items
// (heaviest first, dealt out in a snake order so every CTA gets a similar
// number of key tiles).  K and V tiles stream through their rings across
// item boundaries; the next item's Q is copied as soon as the current item's
// last S has read the Q buffer; its first S tiles are computed while the
// current item's epilogue reads the accumulators, which the next P.V only
// overwrites once the epilogue has released them.
//
// Warps: 0-7 softmax and epilogue (two per TMEM lane quarter); 8 and 11
// producers of K and of V (TMA boxes of 128 keys x 64 columns, 128-byte
// swizzle; a ring of K tiles, released as soon as S has read them, and a ring
// of V tiles, released after P.V); 9 and 10 MMA issuers (one thread each: S,
// and P.V), warp 9 also the tensor-memory owner.  Rows past an
// item's last visible key are never read: a partial last tile is boxed in
// 32- and 8-row groups, its remaining live rows copied by the producer's
// lanes, the rest zeroed.  Every wait is bounded; a timeout records
// KVC_ERR_TIMEOUT, every role leaves its loop, the MMA issuer waits for its
// MMAs, the producer and the softmax warps for their copies, and tensor
// memory is freed before the CTA exits.
#pragma once

#include <type_traits>

#include "kvc_decode_mma.cuh"
#include "kvc_tcgen05.cuh"

namespace kvc {

template <typename T, int D>
struct TcPrefillCfg {
    static constexpr int BM = 128;                 // query rows per item (TMEM lanes)
    static constexpr int BN = 128;                 // keys per tile
    static constexpr int CB = D / 64;              // 128-byte column blocks of a row
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int CHUNKS = ROW_BYTES / 16;  // 16-byte chunks of a row
    static constexpr int BLK = 128 * 128;          // one column block of a 128-row tile
    static constexpr int Q_BYTES = CB * BLK;
    static constexpr int KT_BYTES = CB * BLK;      // one K (or V) tile
    // K tiles are released as soon as S = Q.K^T has used them, V tiles only
    // after P.V: separate rings
    static constexpr int NSK = D == 64 ? 4 : 3;
    static constexpr int NSV = D == 64 ? 4 : 2;
    // kfull[NSK], kempty[NSK], vfull[NSV], vempty[NSV], s_full[2],
    // p_full[2 buffers][2 halves], p_free[2 buffers][2 halves], q_full,
    // q_empty, o_free, mma_done, pair[4], s_free[2].  Every barrier whose
    // phases follow the key tiles is kept per S buffer, so that no waiter is
    // ever two phases away from it (the softmax may run two tiles ahead of
    // P.V).
    static constexpr int NBAR = 2 * NSK + 2 * NSV + 20;
    static constexpr int BAR_OFF = Q_BYTES + (NSK + NSV) * KT_BYTES;
    // the two softmax threads of a row swap their halves' running maxima and
    // sums here at the end of an item: per lane quarter [half][max, sum][32]
    static constexpr int XCH_OFF = BAR_OFF + 8 * NBAR + 32;  // after the TMEM address and the abort flag
    static constexpr int SMEM = 1024 + XCH_OFF + 4 * 2 * 2 * 32 * 4;
    static constexpr int NSW = 8;                  // softmax warps: two per TMEM lane quarter
    static constexpr int THREADS = (NSW + 4) * 32; // + K producer, S issuer, P.V issuer, V producer
    static constexpr uint32_t TMEM_COLS = 512;
    // two S buffers, then one O accumulator per half of the key tile; the
    // probabilities P of a tile overwrite the first 32 columns of each half
    // of its S buffer (64 keys as 16-bit pairs)
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

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One work item: a block of chunk tokens of segment seg (= b * H_kv + kv)
// and the key range its rows see.  Every role of the CTA derives the same
// items in the same order.
struct PrefillItem {
    int b, kv, seg, qb, t0, ntok, c, kend, ntiles;
};

// The k-th item of this CTA (false past the last): items are numbered
// heaviest first (the last token blocks of every segment see the most keys)
// and dealt to the CTAs in a snake order, row k of the deal running forward
// for even k and backward for odd k.
template <class A>
__device__ __forceinline__ bool prefill_item(const A &a, int k, int tokens_per_item, PrefillItem &it) {
    const int P = int(gridDim.x), cta = int(blockIdx.x);
    const int nseg = a.B * a.H_kv;
    const int64_t idx = int64_t(k) * P + ((k & 1) ? P - 1 - cta : cta);
    if (idx >= int64_t(nseg) * a.q_blocks) return false;
    it.qb = a.q_blocks - 1 - int(idx / nseg);
    it.seg = int(idx % nseg);
    it.b = it.seg / a.H_kv;
    it.kv = it.seg % a.H_kv;
    it.t0 = it.qb * tokens_per_item;
    it.ntok = min(tokens_per_item, a.T_new - it.t0);
    it.c = __ldg(a.cache_index + it.b);
    const bool bad = it.c < 0 || it.c > a.max_ctx - a.T_new;
    it.kend = it.c + it.t0 + it.ntok;  // keys [0, kend) are visible to some row of the item
    it.ntiles = bad ? 0 : (it.kend + 127) / 128;
    return true;
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
    // the single warps after the softmax warps
    constexpr int PRODUCER = C::NSW, ISSUER = C::NSW + 1, PV_ISSUER = C::NSW + 2, V_PRODUCER = C::NSW + 3;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = dev::smem_addr(smem);
    const uint32_t q_s = sb, k_s = sb + C::Q_BYTES, v_s = k_s + NSK * C::KT_BYTES;
    const uint32_t kfull = sb + C::BAR_OFF, kempty = kfull + 8 * NSK, vfull = kempty + 8 * NSK,
                   vempty = vfull + 8 * NSV;
    const uint32_t s_full = vempty + 8 * NSV, p_full = s_full + 16, p_free = p_full + 32, q_full = p_free + 32,
                   q_empty = q_full + 8, o_free = q_empty + 8, mma_done = o_free + 8, pair_bar = mma_done + 8,
                   s_free = pair_bar + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + 8 * C::NBAR);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::BAR_OFF + 8 * C::NBAR + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int G = a.group;
    const int TB = BM / G;  // chunk tokens per item

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
        for (int x = 0; x < 2; ++x) {
            dev::mbar_init(s_full + 8 * x, 1);
            dev::mbar_init(s_free + 8 * x, 1);           // the P.V of the buffer's tile has completed
        }
        for (int x = 0; x < 4; ++x) {                    // [buffer][half]
            dev::mbar_init(p_full + 8 * x, C::NSW / 2);  // the half's four softmax warps
            dev::mbar_init(p_free + 8 * x, 1);           // the half's P.V has completed
        }
        dev::mbar_init(q_full, C::NSW);                  // every softmax warp copied its rows of Q
        dev::mbar_init(q_empty, 1);                      // the item's last S has read its Q
        dev::mbar_init(o_free, C::NSW);                  // the epilogue has read the accumulators
        dev::mbar_init(mma_done, 2);                     // one commit per issuing thread
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

    int issued = 0;  // tiles whose copies this producer issued
    if (warp == PRODUCER || warp == V_PRODUCER) {
        // ------------------------------------------------------------ producers
        // One warp streams the K tiles, one the V tiles, each as far ahead as
        // its ring allows (S needs K a whole softmax earlier than P.V needs V).
        const bool is_v = warp == V_PRODUCER;
        const int ns = is_v ? NSV : NSK;
        const uint32_t ring = is_v ? v_s : k_s, full0 = is_v ? vfull : kfull, empty0 = is_v ? vempty : kempty;
        uint32_t generic = 0;  // stages whose last fill had generic-proxy stores
        bool ok = true;
        PrefillItem it{};
        // one tile of this producer's tensor of the current item into one stage
        auto load = [&](int j, uint32_t dst, uint32_t full, int s) {
            const int z = a.seg_base + it.seg;
            const int row0 = j * BN, nr = min(BN, it.kend - row0);
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
            const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;
            const uint8_t *src = (is_v ? a.V : a.K) + int64_t(it.seg) * kv_slab + int64_t(row0) * C::ROW_BYTES;
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
        // the stage of the n-th tile of a ring is free again
        auto wait_free = [&](uint32_t empty, int n, int ns) {
            if (n < ns) return true;
            const bool w = dev::mbar_wait_bounded(empty, uint32_t(n / ns - 1) & 1, flags, a.timeout_ns);
            if (__all_sync(FULL, w)) return true;
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
            return false;
        };
        for (int k = 0; ok && prefill_item(a, k, TB, it); ++k) {
            for (int j = 0; ok && j < it.ntiles; ++j) {
                const int s = issued % ns;
                ok = wait_free(empty0 + 8 * s, issued, ns);
                if (!ok) break;
                load(j, ring + uint32_t(s) * C::KT_BYTES, full0 + 8 * s, s);
                ++issued;
            }
        }
    } else if (warp == ISSUER || warp == PV_ISSUER) {
        // ------------------------------------------------------------ MMA issuers
        // Two threads in two warps issue the two streams of MMAs, so that a
        // thread busy issuing one product never holds back the other.
        if (lane == 0) {
            bool ok = true;
            int gs = 0, nk = 0;  // tiles and items issued so far
            PrefillItem it;
            for (int k = 0; ok && prefill_item(a, k, TB, it); ++k) {
                if (it.ntiles == 0) continue;
                if (warp == ISSUER) {
                    // S = Q . K_j^T into S buffer gs % 2, once the P.V of tile
                    // gs - 2 has read its probabilities from that buffer
                    const uint32_t qt = q_s;
                    ok = dev::mbar_wait_bounded(q_full, uint32_t(nk) & 1, flags, a.timeout_ns);
                    for (int j = 0; ok && j < it.ntiles; ++j, ++gs) {
                        const int s = gs % NSK;
                        ok = dev::mbar_wait_bounded(kfull + 8 * s, uint32_t(gs / NSK) & 1, flags, a.timeout_ns);
                        if (ok && gs >= 2)
                            ok = dev::mbar_wait_bounded(s_free + 8 * (gs & 1), uint32_t((gs >> 1) - 1) & 1, flags,
                                                        a.timeout_ns);
                        if (!ok) break;
                        tc::fence_after();
                        const uint32_t kt = k_s + uint32_t(s) * C::KT_BYTES;
                        const uint32_t s_t = tmem + ((gs & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t off = (ks >> 2) * BLK + (ks & 3) * 32;
                            tc::mma_f16_ss(s_t, tc::smem_desc_sw128(qt + off, 16, 1024),
                                           tc::smem_desc_sw128(kt + off, 16, 1024), IDESC_S, ks > 0);
                        }
                        tc::commit(s_full + 8 * (gs & 1));
                        tc::commit(kempty + 8 * s);                                   // K stage free
                        if (j == it.ntiles - 1) tc::commit(q_empty);  // the item's Q read
                    }
                } else {
                    // O_h += P_h . V_h for the two halves h of every tile
                    // (keys [64 h, 64 h + 64)), each once its softmax warps
                    // have written their half of P; the item's first P.V
                    // overwrites the accumulators once the previous item's
                    // epilogue has read them
                    for (int j = 0; ok && j < it.ntiles; ++j, ++gs) {
                        const int s = gs % NSV;
                        ok = dev::mbar_wait_bounded(vfull + 8 * s, uint32_t(gs / NSV) & 1, flags, a.timeout_ns);
                        if (ok && j == 0 && nk > 0)
                            ok = dev::mbar_wait_bounded(o_free, uint32_t(nk - 1) & 1, flags, a.timeout_ns);
                        if (!ok) break;
                        const uint32_t vt = v_s + uint32_t(s) * C::KT_BYTES;
                        const int buf = gs & 1;
                        const uint32_t pt = tmem + (buf ? C::S_COL1 : C::S_COL0);  // P in the tile's S buffer
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            ok = dev::mbar_wait_bounded(p_full + 8 * (2 * buf + hf), uint32_t(gs >> 1) & 1, flags,
                                                        a.timeout_ns);
                            if (!ok) break;
                            tc::fence_after();
                            const uint32_t o_t = tmem + C::O_COL + uint32_t(hf) * D;
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                tc::mma_f16_ts(o_t, pt + 64 * hf + 8 * ks,
                                               tc::smem_desc_sw128(vt + hf * 8192 + ks * 2048, BLK, 1024), IDESC_O,
                                               (j > 0 || ks > 0));
                            tc::commit(p_free + 8 * (2 * buf + hf));  // O_h up to date
                        }
                        if (!ok) break;
                        tc::commit(s_free + 8 * buf);  // the S buffer (and its P) free
                        if (!ok) break;
                        tc::commit(vempty + 8 * s);  // V stage free
                    }
                }
                ++nk;
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
        const int qd = warp & 3, hf = warp >> 2;
        const int r = 32 * qd + lane;           // query row = TMEM lane
        const int i = r / TB, tt = r - i * TB;  // head of the group, token of the item
        const int H = a.H_kv * G;
        const uint32_t pbar = pair_bar + 8 * qd;
        constexpr int QC = C::CHUNKS / 2;       // 16-byte chunks of Q (and of the output) per half row
        float *xch = reinterpret_cast<float *>(smem + C::XCH_OFF) + qd * 4 * 32;  // this lane quarter's slots
        const uint32_t lane_base = uint32_t(qd * 32) << 16;
        const float2 scale2 = make_float2(a.scale_log2, a.scale_log2);
        // this thread's half of an item's Q row into the Q buffer
        auto copy_q = [&](const PrefillItem &x, bool async) {
            const bool valid = x.ntiles > 0 && i < G && tt < x.ntok;
            const uint32_t qt = q_s;
            const uint4 *qrow = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const T *>(a.q) + ((int64_t(x.b) * H + x.kv * G + i) * a.T_new + x.t0 + tt) * D);
#pragma unroll
            for (int c16 = hf * QC; c16 < (hf + 1) * QC; ++c16) {
                if (!valid)
                    dev::st_shared_v4(C::swz(qt, r, c16), make_uint4(0u, 0u, 0u, 0u));
                else if (async)
                    dev::cp_async_16(C::swz(qt, r, c16), qrow + c16);
                else
                    dev::st_shared_v4(C::swz(qt, r, c16), __ldg(qrow + c16));
            }
        };
        bool ok = true;
        int gt = 0, nk = 0, kn = 0;  // tiles and items processed so far, items enumerated so far
        PrefillItem it, nx;
        bool have = prefill_item(a, kn++, TB, it);
        while (have && it.ntiles == 0) {
            if (threadIdx.x == 0 && it.kv == 0 && it.qb == 0) dev::record_error(a.err, ERR_DEVICE_INDEX);
            have = prefill_item(a, kn++, TB, it);
        }
        if (have) {
            copy_q(it, false);
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(q_full);
        }
        while (have) {
            // the next item with work (its enumeration index kx); its Q is
            // copied into the Q buffer as soon as this item's last S has read
            // it -- polled between tiles, so the copy hides behind the
            // item's last tiles
            int kx = -1;
            {
                bool hn = prefill_item(a, kn, TB, nx);
                while (hn && nx.ntiles == 0) {
                    if (threadIdx.x == 0 && nx.kv == 0 && nx.qb == 0) dev::record_error(a.err, ERR_DEVICE_INDEX);
                    hn = prefill_item(a, ++kn, TB, nx);
                }
                if (hn) kx = kn++;
            }
            const bool have_nx = kx >= 0;
            bool q_copied = !have_nx;
            const bool row_ok = i < G && tt < it.ntok;
            const int limit = row_ok ? it.c + it.t0 + tt : it.c;  // last visible key (unused rows: any finite range)
            const int lim_min = it.c + it.t0;                     // smallest limit of the item's rows
            const uint32_t o_t = tmem + lane_base + C::O_COL + uint32_t(hf) * D;  // this half's accumulator
            const uint32_t pf = p_free + 8 * hf;
            float m_run = -INFINITY;
            float2 l2 = make_float2(0.f, 0.f);  // running sum, two partial lanes
            for (int j = 0; j < it.ntiles; ++j, ++gt) {
                if (!q_copied && __all_sync(FULL, dev::mbar_test_wait(q_empty, uint32_t(nk) & 1))) {
                    copy_q(nx, true);
                    q_copied = true;
                }
                ok = !flags[0] &&
                     dev::mbar_wait_bounded(s_full + 8 * (gt & 1), uint32_t(gt >> 1) & 1, flags, a.timeout_ns);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc::fence_after();
                uint32_t sr[2][32];
                const uint32_t s_t = tmem + lane_base + ((gt & 1) ? C::S_COL1 : C::S_COL0) + 64 * hf;
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
                // maximum over four independent chains
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        m4[(e >> 1) & 3] =
                            fmax3(m4[(e >> 1) & 3], __uint_as_float(sr[h2][e]), __uint_as_float(sr[h2][e + 1]));
                const float m_tile = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * a.scale_log2;
                // raise the reference max only when the tile's exceeds it by 2^8
                const float m_new = m_tile > m_run + C::RESCALE_LOG2 ? m_tile : m_run;
                const float corr = m_new == m_run ? 1.f : ex2_approx(m_run - m_new);
                m_run = m_new;
                const float negm = m_run == -INFINITY ? 0.f : -m_run;
                const float2 neg2 = make_float2(negm, negm);
                float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                uint32_t pk[32];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 y = __ffma2_rn(
                            make_float2(__uint_as_float(sr[h2][e]), __uint_as_float(sr[h2][e + 1])), scale2, neg2);
                        const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
                        ps[(e >> 1) & 3] = __fadd2_rn(ps[(e >> 1) & 3], make_float2(p0, p1));
                        pk[16 * h2 + e / 2] = Ops::pack(p0, p1);
                    }
                l2 = __ffma2_rn(l2, make_float2(corr, corr),
                                __fadd2_rn(__fadd2_rn(ps[0], ps[1]), __fadd2_rn(ps[2], ps[3])));
                if (j > 0 && __any_sync(FULL, corr != 1.f)) {
                    // rescale O_hf once this half's P.V of the previous tile has
                    // completed (its next P.V waits for this tile's P)
                    ok = !flags[0] && dev::mbar_wait_bounded(pf + 16 * ((gt - 1) & 1), uint32_t((gt - 1) >> 1) & 1,
                                                             flags, a.timeout_ns);
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                    tc::fence_after();
                    const float2 c2 = make_float2(corr, corr);
#pragma unroll 1
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        uint32_t o[32];
                        tc::tmem_ld32(o_t + 32 * q4, o);
                        tc::tmem_ld_wait();
                        tc::reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 v =
                                __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), c2);
                            o[e] = __float_as_uint(v.x);
                            o[e + 1] = __float_as_uint(v.y);
                        }
                        tc::tmem_st32(o_t + 32 * q4, o);
                    }
                }
                // this half of the P row into the tile's S buffer (columns
                // [64 hf, 64 hf + 32)): the A operand of O_hf += P_hf . V_hf
                tc::tmem_st32(s_t, pk);
                tc::tmem_st_wait();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(p_full + 8 * (2 * (gt & 1) + hf));
            }
            if (!ok) break;
            if (have_nx) {
                if (!q_copied) {
                    ok = __all_sync(FULL, !flags[0] && dev::mbar_wait_bounded(q_empty, uint32_t(nk) & 1, flags,
                                                                               a.timeout_ns));
                    if (!ok) break;
                    copy_q(nx, true);
                }
                // the next item's Q has landed: hand it to the S issuer
                cp_async_wait_all();
                dev::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(q_full);
            }
            // ---- epilogue: both halves' last P.V have completed; swap the
            // halves' (max, sum), then out = (O_0 e_0 + O_1 e_1) / (l_0 e_0 +
            // l_1 e_1) with e_h = 2^(m_h - max(m_0, m_1)), this thread taking
            // output columns [hf D/2, (hf + 1) D/2)
            const uint32_t pl = p_free + 16 * ((gt - 1) & 1);  // the last tile's buffer
            ok = !flags[0] && dev::mbar_wait_bounded(pl, uint32_t((gt - 1) >> 1) & 1, flags, a.timeout_ns) &&
                 dev::mbar_wait_bounded(pl + 8, uint32_t((gt - 1) >> 1) & 1, flags, a.timeout_ns);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            const float l_me = l2.x + l2.y;
            xch[(hf * 2 + 0) * 32 + lane] = m_run;
            xch[(hf * 2 + 1) * 32 + lane] = l_me;
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(pbar);
            ok = __all_sync(FULL, dev::mbar_wait_bounded(pbar, 0, flags, a.timeout_ns));  // phase 2 nk
            if (!ok) break;
            const float m_ot = xch[((hf ^ 1) * 2 + 0) * 32 + lane], l_ot = xch[((hf ^ 1) * 2 + 1) * 32 + lane];
            // both threads of the row read before either writes these rows again
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(pbar);
            tc::fence_after();
            const float m0 = hf ? m_ot : m_run, m1 = hf ? m_run : m_ot;
            const float l0 = hf ? l_ot : l_me, l1 = hf ? l_me : l_ot;
            const float M = fmaxf(m0, m1);  // finite: key 0 is visible to every row
            const float e0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - M);
            const float e1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - M);
            const float inv = 1.f / (l0 * e0 + l1 * e1);
            const float f0 = e0 * inv, f1 = e1 * inv;
            uint4 *orow = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(a.out) +
                                                    ((int64_t(it.b) * H + it.kv * G + i) * a.T_new + it.t0 + tt) * D) +
                          hf * QC;
            const uint32_t oc = tmem + lane_base + C::O_COL + uint32_t(hf) * (D / 2);  // column hf D/2 of O_0
#pragma unroll 1
            for (int q4 = 0; q4 < D / 64; ++q4) {
                uint32_t u[32], v[32];
                tc::tmem_ld32(oc + 32 * q4, u);
                tc::tmem_ld32(oc + D + 32 * q4, v);
                tc::tmem_ld_wait();
                tc::reg_fence(u);
                tc::reg_fence(v);
                if (q4 == D / 64 - 1) {
                    // the accumulators are read: the next item's P.V may overwrite them
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(o_free);
                }
#pragma unroll
                for (int e = 0; e < 32; e += 2) {  // combined pair -> u[e / 2], packed in place
                    const float y0 = fmaf(__uint_as_float(u[e]), f0, __uint_as_float(v[e]) * f1);
                    const float y1 = fmaf(__uint_as_float(u[e + 1]), f0, __uint_as_float(v[e + 1]) * f1);
                    u[e / 2] = Ops::pack(y0, y1);
                }
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4) orow[(32 * q4) / 8 + e / 4] = make_uint4(u[e], u[e + 1], u[e + 2], u[e + 3]);
                }
            }
            ok = __all_sync(FULL, dev::mbar_wait_bounded(pbar, 1, flags, a.timeout_ns));  // phase 2 nk + 1
            if (!ok) break;
            ++nk;
            have = have_nx && prefill_item(a, kx, TB, it);
        }
        if (!ok && lane == 0) {
            if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
            flags[0] = 1;
        }
    }

    // ---- teardown: every role is done; the MMAs have completed
    tc::fence_before();
    __syncthreads();
    if (warp == ISSUER) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if ((warp == PRODUCER || warp == V_PRODUCER) && lane == 0 && flags[0]) {
        // after an abort, wait (bounded) for the copies that may still land
        const volatile int never = 0;
        const int ns = warp == V_PRODUCER ? NSV : NSK;
        const uint32_t full0 = warp == V_PRODUCER ? vfull : kfull;
        for (int j = issued > ns ? issued - ns : 0; j < issued; ++j)
            dev::mbar_wait_bounded(full0 + 8 * (j % ns), uint32_t(j / ns) & 1, &never, a.timeout_ns);
    }
    if (warp < C::NSW) cp_async_wait_all();  // no copy of this thread lands after the CTA exits
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
