// kvc_decode_tc.cuh -- decode attention for large query-head groups on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// "10.3 -- KV cache implementation details", section 4.1: under multi-query
// and grouped-query attention the g query heads of a KV head share its cached
// K and V; section 5: one decode step attends the new query over every live
// row.  With g = 16 or 32 the product of a key tile with the group's queries
// is a real dense tile, which the 5th-generation tensor cores take whole:
//   S^T = K_t . Q^T     tcgen05.mma M = 128 keys, N = g heads, K = d_h = 128;
//                       A = the K tile, B = the group's queries (both
//                       K-major in shared memory), S^T in tensor memory (two
//                       buffers: S of the next tile while the softmax reads
//                       this one)
//   softmax             two threads own key k of the tile (its TMEM lane),
//                       each reading the scores of half of the g heads; each
//                       head's tile maximum is a transpose-reduction over a
//                       warp's 32 keys, then over the four lane quarters
//                       through shared memory; probabilities P^T[head][key]
//                       are written to
//                       shared memory in the B-operand layout of
//   O^T += V^T . P^T    tcgen05.mma M = d_h = 128, N = g, K = 128 keys; A =
//                       the V tile as stored ([key][d]: M contiguous, an
//                       MN-major operand), O^T in tensor memory.
// The running max of each head is raised only when a tile's maximum exceeds
// it by more than 2^8 (P stays <= 256); O^T and the partial sums are then
// rescaled, after the previous P.V has completed.
//
// The split of the live rows over the CTAs, the pieces and the ticket-first
// split combine are those of decode_mma_kernel; the softmax warps run the
// combine themselves at the end of a piece, on O^T read straight from tensor
// memory, so no shared-memory copy of the state is needed and the K and V
// rings get that space.
//
// Warps: 0 and 1 copy the K and V tiles (TMA boxes of 64 columns x 128, 32 or
// 8 rows with the 128-byte swizzle; rows past a box-aligned range and the
// step's new row by 16-byte loads; rows past the piece's end zeroed); 2 issues
// S (and owns tensor memory), 3 issues P.V (one thread each); 4-11 softmax
// and the piece epilogue (split combine included), two per TMEM lane quarter
// (one per half of the heads).  Every wait is bounded; a timeout records
// KVC_ERR_TIMEOUT, every role leaves its loop, the issuers wait for their MMAs
// and tensor memory is freed before the CTA exits.
#pragma once

#include <type_traits>

#include "kvc_decode_mma.cuh"
#include "kvc_tcgen05.cuh"

namespace kvc {

template <typename T, int G>
struct TcDecodeCfg {
    static constexpr int D = 128;                  // head width
    static constexpr int TK = 128;                 // keys per tile (TMEM lanes of S^T)
    static constexpr int CB = D / 64;              // 128-byte column blocks of a row
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int CHUNKS = ROW_BYTES / 16;  // 16-byte chunks of a row
    static constexpr int BLK = TK * 128;           // one column block of a tile
    static constexpr int KT_BYTES = CB * BLK;      // a K (or V) tile
    // K tiles are released after S, V tiles only after P.V: the deeper V ring
    static constexpr int NSK = 2, NSV = 4;
    static constexpr int QB = G * 128;             // one 64-column block of Q^T (G rows)
    static constexpr int Q_BYTES = CB * QB;
    static constexpr int P_BYTES = (TK / 64) * G * 128;  // P^T of one tile: two 64-key blocks of G rows
    static constexpr int K_OFF = 0, V_OFF = NSK * KT_BYTES, Q_OFF = V_OFF + NSV * KT_BYTES,
                         P_OFF = Q_OFF + Q_BYTES, RED_OFF = P_OFF + 2 * P_BYTES;
    // the softmax warps' exchange slots, [2 phases][2 halves][4 quarters][32]:
    // tile maxima, or at a piece's end the partial sums
    static constexpr int RED_BYTES = 4 * (2 * 2 * 4 * 32);
    // kfull[NSK] kempty[NSK] vfull[NSV] vempty[NSV] s_full[2] s_free[2] p_full[2]
    // p_free[2] q_full q_empty o_free mx st_full st_free mma_done
    static constexpr int NBAR = 2 * NSK + 2 * NSV + 15;
    static constexpr int BAR_OFF = RED_OFF + RED_BYTES;
    static constexpr int SMEM = 1024 + BAR_OFF + 8 * NBAR + 32;  // + the TMEM address and the flags
    // softmax warps: two per TMEM lane quarter, one per half of the heads
    static constexpr int NSOFT = 8, GH = G / 2;
    static constexpr int THREADS = 13 * 32;
    static constexpr int K_PRODUCER = 0, V_PRODUCER = 1, S_ISSUER = 2, O_ISSUER = 3, SOFT0 = 4, MERGER = 12;
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 64, O_COL = 128;  // S^T buffers and O^T, G columns each
    static constexpr float RESCALE_LOG2 = 8.f;
    static_assert(G == 16 || G == 32, "16 or 32 query heads per KV head");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    static_assert(KT_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0 && P_BYTES % 1024 == 0, "swizzle-atom alignment");

    // 16-byte chunk c of row r of a swizzled tile (column blocks BLK apart).
    __device__ __forceinline__ static uint32_t swz(uint32_t tile, int r, int c) {
        return tile + uint32_t(c >> 3) * BLK + uint32_t(r) * 128 + (uint32_t((c & 7) ^ (r & 7)) << 4);
    }
};

namespace tcd {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Reduce v[0..G) of every lane of the warp with max (SUM = false) or + (SUM =
// true); afterwards lane l holds, in v[0], the result for element l mod G.
// The halves of the vector are exchanged between lane pairs (a transpose
// reduction: 16 + 8 + 4 + 2 + 1 shuffles for 32 elements).
template <int G, bool SUM>
__device__ __forceinline__ void transpose_reduce(float (&v)[G], int lane) {
#pragma unroll
    for (int s = G / 2; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = up ? v[i] : v[i + s];
            const float keep = up ? v[i + s] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s);
            v[i] = SUM ? keep + recv : fmaxf(keep, recv);
        }
    }
#pragma unroll
    for (int s = G; s < 32; s <<= 1) {
        const float recv = __shfl_xor_sync(0xffffffffu, v[0], s);
        v[0] = SUM ? v[0] + recv : fmaxf(v[0], recv);
    }
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, uint32_t (&r)[32]) {
    tc::tmem_ld32(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_st_cols<8>(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_cols<32>(uint32_t taddr, const uint32_t (&r)[32]) {
    tc::tmem_st32(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_st_cols<16>(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// keep uses of the loaded registers behind tcgen05.wait::ld
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// x rounded to the cache's 16-bit type, as its bits.
template <typename T>
__device__ __forceinline__ uint16_t bits16(float x);
template <>
__device__ __forceinline__ uint16_t bits16<__nv_bfloat16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <>
__device__ __forceinline__ uint16_t bits16<__half>(float x) {
    return __half_as_ushort(__float2half_rn(x));
}

}  // namespace tcd

// The merge warp of decode_tc_kernel: for each split piece of the CTA, once
// the softmax warps have written its state to its partial slot (CTA +
// segment), the split combine of merge_pieces_chunked on that global state:
// a split takes its ticket -- every split but the last publishes (fence,
// ready flag), the last waits for the others' flags, folds all the segment's
// partials (eight heads at a time, every split's loads in flight together)
// and writes the output, then resets the counter and the flags.  (A piece
// that is a whole segment was written by the softmax warps.)
template <typename T, int D, int G>
__device__ __forceinline__ void merge_pieces_tc(const DecodeArgs &a, const Plan &plan, Walker walk, uint32_t st_full,
                                                uint32_t st_free, volatile int *flags, int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(D == 128, "four output columns per lane");
    const int H = a.H_kv * G;
    const int me = int(blockIdx.x);
    uint32_t piece = 0;
    Piece pc;
    while (walk.next(a, pc)) {
        bool ok = !flags[0] && dev::mbar_wait_bounded(st_full, piece & 1, flags, a.timeout_ns);
        ok = __all_sync(FULL, ok);
        if (!ok) {
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
            return;
        }
        const int seg = pc.b * a.H_kv + pc.kv;
        const int c0 = int(pc.seg_start / plan.chunk), c1 = int((pc.seg_start + pc.len - 1) / plan.chunk);
        if (c0 != c1) {  // whole segments were written by the softmax warps
            int ticket = 0;
            if (lane == 0) ticket = atomicAdd(a.tickets + seg, 1);
            ticket = __shfl_sync(FULL, ticket, 0);
            if (ticket < c1 - c0) {
                // not the last split: publish the partial
                __threadfence();
                __syncwarp();
                if (lane == 0) dev::flag_store(a.ready + me + seg, 1);
            } else {
                // the last split: wait for the others' flags, then fold every
                // split's partial (this CTA's included)
                bool pub = true;
                for (int c = c0 + lane; c <= c1; c += 32)
                    if (c != me) pub = pub && dev::flag_wait_bounded(a.ready + c + seg, flags, a.flag_timeout_ns);
                pub = __all_sync(FULL, pub);
                if (!pub) {
                    if (lane == 0) {
                        if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                        flags[0] = 1;
                    }
                    return;
                }
                __threadfence();
                // lane h < G: head h's max and sum over the splits
                const float *mlp = a.part_ml + (int64_t(c0) + seg) * G * 2;
                float Mh = -INFINITY, Lh = 0.f;
                if (lane < G) {
                    for (int c = 0; c <= c1 - c0; ++c) Mh = fmaxf(Mh, __ldcg(mlp + (c * G + lane) * 2));
                    for (int c = 0; c <= c1 - c0; ++c)
                        Lh = fmaf(__ldcg(mlp + (c * G + lane) * 2 + 1), tcd::ex2(__ldcg(mlp + (c * G + lane) * 2) - Mh), Lh);
                }
                const float invh = lane < G ? 1.f / Lh : 0.f;
                // eight heads at a time, lane l: output columns [4 l, 4 l + 4)
#pragma unroll 1
                for (int h0 = 0; h0 < G; h0 += 8) {
                    float4 acc[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int c = 0; c <= c1 - c0; ++c) {
                        const float e_lane = lane < G ? tcd::ex2(__ldcg(mlp + (c * G + lane) * 2) - Mh) : 0.f;
                        const float4 *src = reinterpret_cast<const float4 *>(a.part_acc + ((int64_t(c0) + c + seg) * G + h0) * D) + lane;
                        float4 v[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) v[k] = __ldcg(src + k * (D / 4));
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float e = __shfl_sync(FULL, e_lane, h0 + k);
                            acc[k].x = fmaf(v[k].x, e, acc[k].x);
                            acc[k].y = fmaf(v[k].y, e, acc[k].y);
                            acc[k].z = fmaf(v[k].z, e, acc[k].z);
                            acc[k].w = fmaf(v[k].w, e, acc[k].w);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float inv = __shfl_sync(FULL, invh, h0 + k);
                        uint16_t *ob = reinterpret_cast<uint16_t *>(a.out) + (int64_t(pc.b) * H + pc.kv * G + h0 + k) * D + 4 * lane;
                        const uint32_t lo = uint32_t(tcd::bits16<T>(acc[k].x * inv)) | (uint32_t(tcd::bits16<T>(acc[k].y * inv)) << 16);
                        const uint32_t hi = uint32_t(tcd::bits16<T>(acc[k].z * inv)) | (uint32_t(tcd::bits16<T>(acc[k].w * inv)) << 16);
                        *reinterpret_cast<uint2 *>(ob) = make_uint2(lo, hi);
                    }
                }
                for (int c = c0 + lane; c <= c1; c += 32)  // ready for the next launch
                    if (c != me) dev::flag_store(a.ready + c + seg, 0);
                if (lane == 0) a.tickets[seg] = 0;
            }
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(st_free);
        ++piece;
    }
}

template <typename T, int G>
// 13 warps: four run on one scheduler, whose 16,384 registers cap them at 128
__global__ void __maxnreg__(128) decode_tc_kernel(const __grid_constant__ DecodeArgs a) {
    using C = TcDecodeCfg<T, G>;
    constexpr int D = C::D, TK = C::TK, CB = C::CB, NSK = C::NSK, NSV = C::NSV, BLK = C::BLK;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t IDESC_S = tc::idesc_f16_f32acc(BF16, TK, G, false, false);  // K-major A and B
    constexpr uint32_t IDESC_O = tc::idesc_f16_f32acc(BF16, D, G, true, false);    // A = V^T MN-major

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = dev::smem_addr(smem);
    const uint32_t k_s = sb + C::K_OFF, v_s = sb + C::V_OFF, q_s = sb + C::Q_OFF, p_s = sb + C::P_OFF;
    float *red = reinterpret_cast<float *>(smem + C::RED_OFF);        // [2 phases][2 halves][4 quarters][32]
    const uint32_t kfull = sb + C::BAR_OFF, kempty = kfull + 8 * NSK, vfull = kempty + 8 * NSK,
                   vempty = vfull + 8 * NSV, s_full = vempty + 8 * NSV, s_free = s_full + 16, p_full = s_free + 16,
                   p_free = p_full + 16, q_full = p_free + 16, q_empty = q_full + 8, o_free = q_empty + 8,
                   mx_bar = o_free + 8, st_full = mx_bar + 8, st_free = st_full + 8, mma_done = st_free + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + 8 * C::NBAR);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + C::BAR_OFF + 8 * C::NBAR + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&a.tm_k128);
        dev::prefetch_tensormap(&a.tm_v128);
        for (int s = 0; s < NSK; ++s) {
            dev::mbar_init(kfull + 8 * s, 1);   // TMA bytes and the producer's arrival
            dev::mbar_init(kempty + 8 * s, 1);  // the commit after S
        }
        for (int s = 0; s < NSV; ++s) {
            dev::mbar_init(vfull + 8 * s, 1);
            dev::mbar_init(vempty + 8 * s, 1);  // the commit after P.V
        }
        for (int x = 0; x < 2; ++x) {
            dev::mbar_init(s_full + 8 * x, 1);        // S^T of the buffer's tile is in tensor memory
            dev::mbar_init(s_free + 8 * x, C::NSOFT);  // the softmax warps have read it
            dev::mbar_init(p_full + 8 * x, C::NSOFT);  // P^T written (and O^T rescaled)
            dev::mbar_init(p_free + 8 * x, 1);        // the P.V that read it has completed
        }
        dev::mbar_init(q_full, C::NSOFT);    // the piece's queries are in shared memory
        dev::mbar_init(q_empty, 1);          // the piece's last S has read them
        dev::mbar_init(o_free, C::NSOFT);    // the piece's O^T has been read
        dev::mbar_init(st_full, C::NSOFT);   // the piece's state is in its partial slot
        dev::mbar_init(st_free, 1);          // the merge warp is done with it
        dev::mbar_init(mx_bar, C::NSOFT);    // the four softmax warps' tile maxima
        dev::mbar_init(mma_done, 2);         // one commit per issuing thread
        flags[0] = 0;
        dev::fence_mbar_init();
    }
    if (warp == C::S_ISSUER) {
        tc::tmem_alloc(dev::smem_addr(tmem_slot), C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    // everything above overlaps the previous kernel on the stream; nothing
    // below runs before it has completed
    dev::grid_dependency_wait();
    dev::allow_dependents();

    const Plan plan = make_plan(a, a.valid_len, lane);
    bool any = plan.r0 < plan.r1 && plan.b < a.B;  // uniform over the CTA
    Walker walk;
    if (any) walk.init(a, plan, a.valid_len);
    const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;

    int issued = 0;  // tiles whose copies this producer issued
    if (!any) {
        // no rows for this CTA
    } else if (warp == C::K_PRODUCER || warp == C::V_PRODUCER) {
        // ------------------------------------------------------------ producers
        const bool is_v = warp == C::V_PRODUCER;
        const int ns = is_v ? NSV : NSK;
        const uint32_t ring = is_v ? v_s : k_s, full0 = is_v ? vfull : kfull, empty0 = is_v ? vempty : kempty;
        const CUtensorMap *m128 = is_v ? &a.tm_v128 : &a.tm_k128;
        const CUtensorMap *m32 = is_v ? &a.tm_vr32 : &a.tm_kr32;
        const CUtensorMap *m8 = is_v ? &a.tm_v8 : &a.tm_k8;
        const uint64_t pol = dev::l2_evict_first_policy();  // K/V rows are read once per launch
        uint32_t generic = 0;  // stages whose last fill had generic-proxy stores
        bool ok = true;
        Piece pc;
        while (ok && walk.next(a, pc)) {
            const int seg = pc.b * a.H_kv + pc.kv;
            const int z = a.seg_base + seg;
            const uint8_t *src_seg = (is_v ? a.V : a.K) + int64_t(seg) * kv_slab;
            const uint8_t *new_src = a.k_new ? (is_v ? a.v_new : a.k_new) + int64_t(seg) * C::ROW_BYTES : nullptr;
            const int new_row = a.k_new ? pc.n - 1 : -1;
            for (int row0 = pc.lo; row0 < pc.hi; row0 += TK) {
                const int nr = min(TK, pc.hi - row0);
                const int s = issued % ns;
                if (issued >= ns) {
                    const bool w = dev::mbar_wait_bounded(empty0 + 8 * s, uint32_t(issued / ns - 1) & 1, flags,
                                                          a.timeout_ns);
                    if (!__all_sync(FULL, w)) {
                        if (lane == 0) {
                            if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                            flags[0] = 1;
                        }
                        ok = false;
                        break;
                    }
                }
                const uint32_t dst = ring + uint32_t(s) * C::KT_BYTES, full = full0 + 8 * s;
                // generic-proxy stores of the stage's last fill come before the
                // TMA unit writes it again
                if (generic & (1u << s)) dev::fence_proxy_async_smem();
                // rows a box may cover: those before the step's new row
                const int nb = (new_row >= row0 && new_row < row0 + nr) ? new_row - row0 : nr;
                if (nb == TK) {
                    if (lane == 0) {
                        dev::mbar_arrive_expect_tx(full, uint32_t(TK) * C::ROW_BYTES);
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb) dev::tma_load_3d(dst + cb * BLK, m128, cb * 64, row0, z, full, pol);
                    }
                    generic &= ~(1u << s);
                } else {
                    // 32-row, then 8-row boxes over the rows before the new
                    // row, the remaining live rows by 16-byte loads (the new
                    // row from k_new / v_new), zeros after them
                    const int n32 = nb >> 5, n8 = (nb >> 3) & 3, boxed = 32 * n32 + 8 * n8;
                    if (lane == 0) {
                        dev::mbar_expect_tx(full, uint32_t(boxed) * C::ROW_BYTES);
                        for (int g = 0; g < n32; ++g)
#pragma unroll
                            for (int cb = 0; cb < CB; ++cb)
                                dev::tma_load_3d(dst + cb * BLK + g * 32 * 128, m32, cb * 64, row0 + 32 * g, z, full, pol);
                        for (int g = 0; g < n8; ++g)
#pragma unroll
                            for (int cb = 0; cb < CB; ++cb) {
                                const int r = 32 * n32 + 8 * g;
                                dev::tma_load_3d(dst + cb * BLK + r * 128, m8, cb * 64, row0 + r, z, full, pol);
                            }
                    }
                    for (int i = lane; i < (TK - boxed) * C::CHUNKS; i += 32) {
                        const int r = boxed + i / C::CHUNKS, c16 = i % C::CHUNKS;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (r < nr) {
                            const uint8_t *src = row0 + r == new_row
                                                     ? new_src
                                                     : src_seg + int64_t(row0 + r) * C::ROW_BYTES;
                            v = __ldg(reinterpret_cast<const uint4 *>(src) + c16);
                        }
                        dev::st_shared_v4(C::swz(dst, r, c16), v);
                    }
                    dev::fence_proxy_async_smem();  // the tensor core reads these rows
                    generic |= 1u << s;
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(full);
                }
                ++issued;
            }
        }
    } else if (warp == C::S_ISSUER || warp == C::O_ISSUER) {
        // ------------------------------------------------------------ MMA issuers
        if (lane == 0) {
            bool ok = true;
            int t = 0, np = 0;  // tiles and pieces so far
            Piece pc;
            while (ok && walk.next(a, pc)) {
                const int ntiles = (pc.hi - pc.lo + TK - 1) / TK;
                if (warp == C::S_ISSUER) {
                    // S^T = K_t . Q^T into S buffer t % 2 once the softmax
                    // warps have read that buffer's previous tile
                    ok = dev::mbar_wait_bounded(q_full, uint32_t(np) & 1, flags, a.timeout_ns);
                    for (int j = 0; ok && j < ntiles; ++j, ++t) {
                        const int s = t % NSK;
                        ok = dev::mbar_wait_bounded(kfull + 8 * s, uint32_t(t / NSK) & 1, flags, a.timeout_ns);
                        if (ok && t >= 2)
                            ok = dev::mbar_wait_bounded(s_free + 8 * (t & 1), uint32_t((t >> 1) - 1) & 1, flags,
                                                        a.timeout_ns);
                        if (!ok) break;
                        tc::fence_after();
                        const uint32_t kt = k_s + uint32_t(s) * C::KT_BYTES;
                        const uint32_t s_t = tmem + ((t & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            tc::mma_f16_ss(s_t,
                                           tc::smem_desc_sw128(kt + (ks >> 2) * BLK + (ks & 3) * 32, 16, 1024),
                                           tc::smem_desc_sw128(q_s + (ks >> 2) * C::QB + (ks & 3) * 32, 16, 1024),
                                           IDESC_S, ks > 0);
                        tc::commit(s_full + 8 * (t & 1));
                        tc::commit(kempty + 8 * s);                 // K stage free
                        if (j == ntiles - 1) tc::commit(q_empty);  // the piece's queries read
                    }
                } else {
                    // O^T += V_t^T . P_t^T once the softmax warps have
                    // written P_t; a piece's first P.V overwrites O^T once the
                    // previous piece's epilogue has read it
                    for (int j = 0; ok && j < ntiles; ++j, ++t) {
                        const int s = t % NSV;
                        ok = dev::mbar_wait_bounded(vfull + 8 * s, uint32_t(t / NSV) & 1, flags, a.timeout_ns);
                        if (ok && j == 0 && np > 0)
                            ok = dev::mbar_wait_bounded(o_free, uint32_t(np - 1) & 1, flags, a.timeout_ns);
                        if (ok)
                            ok = dev::mbar_wait_bounded(p_full + 8 * (t & 1), uint32_t(t >> 1) & 1, flags,
                                                        a.timeout_ns);
                        if (!ok) break;
                        tc::fence_after();
                        const uint32_t vt = v_s + uint32_t(s) * C::KT_BYTES;
                        const uint32_t pt = p_s + uint32_t(t & 1) * C::P_BYTES;
#pragma unroll
                        for (int ks = 0; ks < TK / 16; ++ks)  // keys [16 ks, 16 ks + 16)
                            tc::mma_f16_ss(tmem + C::O_COL, tc::smem_desc_sw128(vt + ks * 2048, BLK, 1024),
                                           tc::smem_desc_sw128(pt + (ks >> 2) * (G * 128) + (ks & 3) * 32, 16, 1024),
                                           IDESC_O, (j > 0 || ks > 0));
                        tc::commit(p_free + 8 * (t & 1));  // O^T up to date, P buffer free
                        tc::commit(vempty + 8 * s);        // V stage free
                    }
                }
                ++np;
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
    } else if (warp == C::MERGER) {
        // ------------------------------------------------------------ merger
        merge_pieces_tc<T, D, G>(a, plan, walk, st_full, st_free, flags, lane);
    } else {
        // ------------------------------------------------------------ softmax
        // Thread (w, hh, lane) owns key 32 w + lane of every tile (S^T lane)
        // and row d = 32 w + lane of O^T, for the heads [hh GH, hh GH + GH);
        // lane l also keeps head (hh GH + l mod GH)'s running max.
        constexpr int GH = C::GH;
        const int w = (warp - C::SOFT0) & 3, hh = (warp - C::SOFT0) >> 2;  // TMEM lane quarter: warp mod 4 == w
        const int key = 32 * w + lane;
        const int sid = (warp - C::SOFT0) * 32 + lane;  // 0 .. 255
        const uint32_t lane_base = uint32_t(w * 32) << 16;
        const uint32_t o_row = tmem + lane_base + C::O_COL + uint32_t(hh * GH);  // this thread's columns of O^T
        const int H = a.H_kv * G;
        bool ok = true;
        int t = 0, np = 0, mxp = 0;  // tiles, pieces, phases of the softmax warps' exchange barrier
        Piece pc;
        while (ok && walk.next(a, pc)) {
            const int ntiles = (pc.hi - pc.lo + TK - 1) / TK;
            // the piece's queries into Q^T ([64-column block][head][128 B],
            // swizzled), once the previous piece's last S has read the buffer
            if (np > 0) {
                ok = __all_sync(FULL, dev::mbar_wait_bounded(q_empty, uint32_t(np - 1) & 1, flags, a.timeout_ns));
                if (!ok) break;
            }
            {
                const uint4 *qg = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.q) +
                                                                  (int64_t(pc.b) * H + pc.kv * G) * D);
                for (int i = sid; i < G * C::CHUNKS; i += C::NSOFT * 32) {
                    const int h = i / C::CHUNKS, c16 = i % C::CHUNKS;
                    dev::st_shared_v4(q_s + uint32_t(c16 >> 3) * C::QB + uint32_t(h) * 128 +
                                          (uint32_t((c16 & 7) ^ (h & 7)) << 4),
                                      __ldg(qg + i));
                }
                dev::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(q_full);
            }
            float m_run = -INFINITY;  // head (hh GH + lane mod GH)'s running max, log2 domain
            float lsum[GH];           // this key's share of the running sums of this thread's heads
#pragma unroll
            for (int h = 0; h < GH; ++h) lsum[h] = 0.f;
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int nr = min(TK, pc.hi - (pc.lo + j * TK));
                ok = !flags[0] &&
                     dev::mbar_wait_bounded(s_full + 8 * (t & 1), uint32_t(t >> 1) & 1, flags, a.timeout_ns);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc::fence_after();
                uint32_t sr[GH];
                tcd::tmem_ld_cols<GH>(tmem + lane_base + ((t & 1) ? C::S_COL1 : C::S_COL0) + uint32_t(hh * GH), sr);
                tc::tmem_ld_wait();
                tcd::reg_fence<GH>(sr);
                tc::fence_before();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(s_free + 8 * (t & 1));  // S buffer read
                float v[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) v[h] = key < nr ? __uint_as_float(sr[h]) : -INFINITY;
                // each head's maximum over the tile: over the warp's keys,
                // then over the four lane quarters (lane l: head hh GH + l mod GH)
                float mv[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) mv[h] = v[h];
                tcd::transpose_reduce<GH, false>(mv, lane);
                float *rt = red + ((mxp & 1) * 2 + hh) * 4 * 32;
                rt[w * 32 + lane] = mv[0];
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(mx_bar);
                // (the next phase needs this warp's arrival: no waiter is two
                // phases behind; the slots of phase p are rewritten at p + 2,
                // after every warp has passed phase p + 1)
                ok = __all_sync(FULL, dev::mbar_wait_bounded(mx_bar, uint32_t(mxp) & 1, flags, a.timeout_ns));
                ++mxp;
                if (!ok) break;
                const float m_tile =
                    fmaxf(fmaxf(rt[lane], rt[32 + lane]), fmaxf(rt[64 + lane], rt[96 + lane])) * a.scale_log2;
                // raise the reference max only when the tile's exceeds it by 2^8
                const float m_new = m_tile > m_run + C::RESCALE_LOG2 ? m_tile : m_run;
                const float corr = m_new == m_run ? 1.f : tcd::ex2(m_run - m_new);
                m_run = m_new;
                const float negm = m_run == -INFINITY ? 0.f : -m_run;
                // P^T of this key for this thread's heads into P buffer t % 2,
                // once the P.V of tile t - 2 has read it
                if (t >= 2) {
                    ok = __all_sync(FULL, !flags[0] && dev::mbar_wait_bounded(p_free + 8 * (t & 1),
                                                                               uint32_t((t >> 1) - 1) & 1, flags,
                                                                               a.timeout_ns));
                    if (!ok) break;
                }
                const bool rescale = __any_sync(FULL, corr != 1.f);
                const uint32_t pb = p_s + uint32_t(t & 1) * C::P_BYTES + uint32_t(key >> 6) * (G * 128);
                const int kc = (key & 63) >> 3, kb2 = (key & 7) * 2;
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const int hg = hh * GH + h;  // head within the group
                    const float mh = __shfl_sync(FULL, negm, h);
                    const float p = tcd::ex2(fmaf(v[h], a.scale_log2, mh));
                    if (rescale) lsum[h] *= __shfl_sync(FULL, corr, h);
                    lsum[h] += p;
                    tcd::st_shared_u16(pb + uint32_t(hg) * 128 + (uint32_t(kc ^ (hg & 7)) << 4) + kb2,
                                       tcd::bits16<T>(p));
                }
                if (rescale && j > 0) {
                    // O^T *= corr per head (column), after the previous tile's P.V
                    ok = __all_sync(FULL, !flags[0] && dev::mbar_wait_bounded(p_free + 8 * ((t - 1) & 1),
                                                                               uint32_t((t - 1) >> 1) & 1, flags,
                                                                               a.timeout_ns));
                    if (!ok) break;
                    tc::fence_after();
                    uint32_t o[GH];
                    tcd::tmem_ld_cols<GH>(o_row, o);
                    tc::tmem_ld_wait();
                    tcd::reg_fence<GH>(o);
#pragma unroll
                    for (int h = 0; h < GH; ++h)
                        o[h] = __float_as_uint(__uint_as_float(o[h]) * __shfl_sync(FULL, corr, h));
                    tcd::tmem_st_cols<GH>(o_row, o);
                    tc::tmem_st_wait();
                }
                dev::fence_proxy_async_smem();  // P^T is read by the tensor core
                tc::fence_before();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(p_full + 8 * (t & 1));
            }
            if (!ok) break;
            // ---- piece epilogue: every head's sum over the piece's keys; a
            // whole segment's output, or a split's state (O^T from tensor
            // memory, each head's max and sum) into its partial slot (CTA +
            // segment) for the merge warp, which runs the split combine.  The
            // previous piece's combine must be done first: the two barriers
            // between these warps and the merge warp then never run more than
            // one phase apart.
            tcd::transpose_reduce<GH, true>(lsum, lane);
            float *lr = red + (mxp & 1) * 256;  // this phase's slots: [2 halves][4 quarters][32]
            lr[(hh * 4 + w) * 32 + lane] = lsum[0];
            const int seg = pc.b * a.H_kv + pc.kv;
            ok = !flags[0] &&
                 dev::mbar_wait_bounded(p_free + 8 * ((t - 1) & 1), uint32_t((t - 1) >> 1) & 1, flags, a.timeout_ns) &&
                 (np == 0 || dev::mbar_wait_bounded(st_free, uint32_t(np - 1) & 1, flags, a.timeout_ns));
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc::fence_after();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(mx_bar);  // sums written (one more phase of mx)
            ok = __all_sync(FULL, dev::mbar_wait_bounded(mx_bar, uint32_t(mxp) & 1, flags, a.timeout_ns));
            ++mxp;
            if (!ok) break;
            {
                uint32_t o[GH];
                tcd::tmem_ld_cols<GH>(o_row, o);
                tc::tmem_ld_wait();
                tcd::reg_fence<GH>(o);
                tc::fence_before();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(o_free);  // O^T read: the next piece may overwrite it
                const float *lh = lr + hh * 4 * 32;
                const float l_lane = (lh[lane] + lh[32 + lane]) + (lh[64 + lane] + lh[96 + lane]);  // head hh GH + lane mod GH
                const int c0 = int(pc.seg_start / plan.chunk), c1 = int((pc.seg_start + pc.len - 1) / plan.chunk);
                if (c0 == c1) {
                    // the piece is the whole segment: its output, normalised
                    uint16_t *ob = reinterpret_cast<uint16_t *>(a.out) + (int64_t(pc.b) * H + pc.kv * G + hh * GH) * D + key;
#pragma unroll
                    for (int h = 0; h < GH; ++h)
                        ob[h * D] = tcd::bits16<T>(__uint_as_float(o[h]) / __shfl_sync(FULL, l_lane, h));
                } else {
                    // a split: its partial, combined by the merge warp
                    const int64_t slot = int64_t(blockIdx.x) + seg;
                    float *pa = a.part_acc + (slot * G + hh * GH) * D + key;
#pragma unroll
                    for (int h = 0; h < GH; ++h) pa[h * D] = __uint_as_float(o[h]);
                    if (w == 0 && lane < GH) {
                        a.part_ml[(slot * G + hh * GH + lane) * 2] = m_run;
                        a.part_ml[(slot * G + hh * GH + lane) * 2 + 1] = l_lane;
                    }
                    __threadfence();
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(st_full);
            }
            // fused step: the CTA holding the segment's last row stores the
            // step's new K and V rows into the cache (nobody in this launch
            // reads them back from there)
            if (a.k_new && pc.hi == pc.n && sid < 2 * C::CHUNKS) {
                const bool is_v = sid >= C::CHUNKS;
                const int c16 = is_v ? sid - C::CHUNKS : sid;
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.v_new : a.k_new) +
                                                                       int64_t(seg) * C::ROW_BYTES) + c16);
                uint8_t *cache = const_cast<uint8_t *>(is_v ? a.V : a.K);  // the caller's writable cache
                reinterpret_cast<uint4 *>(cache + int64_t(seg) * kv_slab + int64_t(pc.n - 1) * C::ROW_BYTES)[c16] = v;
            }
            ++np;
        }
        if (!ok && lane == 0) {
            if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
            flags[0] = 1;
        }
    }

    // ---- teardown: every role is done; the MMAs have completed
    tc::fence_before();
    __syncthreads();
    if (warp == C::S_ISSUER) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if ((warp == C::K_PRODUCER || warp == C::V_PRODUCER) && lane == 0 && flags[0]) {
        // after an abort, wait (bounded) for the copies that may still land
        const volatile int never = 0;
        const int ns = warp == C::V_PRODUCER ? NSV : NSK;
        const uint32_t full0 = warp == C::V_PRODUCER ? vfull : kfull;
        for (int j = issued > ns ? issued - ns : 0; j < issued; ++j)
            dev::mbar_wait_bounded(full0 + 8 * (j % ns), uint32_t(j / ns) & 1, &never, a.timeout_ns);
    }
}

template <typename T, int G>
cudaError_t set_tc_decode_max_smem(int bytes) {
    return cudaFuncSetAttribute(decode_tc_kernel<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T, int G>
cudaError_t launch_tc_decode(const DecodeArgs &a, int grid, int smem, cudaStream_t s) {
    return launch_pdl(decode_tc_kernel<T, G>, dim3(grid), dim3(TcDecodeCfg<T, G>::THREADS), smem, s, a);
}

// The kernel's whole shared memory is its fixed part; one "stage" of zero
// bytes keeps the host's stage rule satisfied.
template <typename T, int G>
const DecodeKernelInfo *tc_decode_info() {
    using C = TcDecodeCfg<T, G>;
    static const DecodeKernelInfo info = {C::TK, 0, 1, C::SMEM, &set_tc_decode_max_smem<T, G>,
                                          &launch_tc_decode<T, G>, true, true, true, C::TK};
    return &info;
}

}  // namespace kvc
