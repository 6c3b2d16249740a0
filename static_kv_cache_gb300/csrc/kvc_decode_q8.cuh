// kvc_decode_q8.cuh -- decode attention over an int8 cache with one fp32
// scale per row ("10.3 -- KV cache implementation details", section 4.4: the
// cache stored as int8, p = 1, half the bytes of a 16-bit cache; section 5:
// the decode attention).  The attention reads the dequantised rows
// x_hat = code * scale; q and the output are bf16.
//
// Same decomposition, stage ring, merge warp and split combine as
// decode_mma_kernel; the tiles hold int8 codes (128 rows of d_h bytes, TMA
// boxes with the 128-byte swizzle) and the row scales arrive by 4-byte
// cp.async beside them.  The per-row scale factors out of both products
// exactly:
//   S^T[key][head] = scale_k[key] * sum_d code_k[key][d] * q[head][d]
//   O^T[d][head]  += sum_key code_v[key][d] * (p[key][head] * scale_v[key])
// so the MMAs run on the raw codes.  An int8 code converts exactly to fp16
// (byte into the mantissa of 1024 + u, minus 1152), so both products use
// mma.sync m16n8k16 in fp16 with fp32 accumulation; q is converted bf16 ->
// fp16 once per piece (exact for values of normal fp16 magnitude) and the
// scaled probabilities are rounded to fp16 where the 16-bit kernel rounds
// them to the cache type.
//
// Fragments.  The tiles are read with ldmatrix on 16-bit pairs of codes.
//   K (non-.trans): lane (gq, tq) gets 4 codes of one key, d = 4tq..4tq+3 of
//     a 16-byte chunk; codes (0, 1) feed one MMA and (2, 3) another, which
//     permutes the contraction index d identically in A and in the q
//     fragments (loaded with the same permutation), so S is unchanged.
//   V (.trans): lane (gq, tq) gets codes (key 2tq, 2tq+1) x (d 2gq, 2gq+1) of
//     a chunk; bytes (0, 2) are the A pair of row d = 2gq, bytes (1, 3) of
//     row d = 2gq + 1, so each ldmatrix feeds an "even" and an "odd" MMA
//     whose accumulator rows map to d = 32cp + 2gq + e and 32cp + 16 + 2gq + e.
// Stale rows past a tail tile's copied ones are masked in S (-inf) and their
// scaled probabilities are set to 0, so their codes and scales never reach
// the sums.
#pragma once

#include "kvc_decode_mma.cuh"

namespace kvc {

template <int D, int G>
struct Q8Cfg {
    static constexpr int ROW_BYTES = D;                 // one int8 code per element
    // 128 keys per tile: a stage (K and V codes) is 32 KB, one 16 KB box
    // per tensor.  The copy issue costs about the same per box whatever its
    // size, so the largest tiles that leave enough stages (six here, for
    // four streams) carry the most bytes per box (64-row tiles: 41.9 us per
    // layer call, 128-row tiles: 40.3 us).
    static constexpr int TILE = 128;
    static constexpr int MT = TILE / 16;                 // 16-key m-tiles of a tile
    // Two consumer warps share each tile, one per half of its keys, each with
    // its own softmax state: a warp's work per tile (and the time the tile's
    // stage stays occupied) is halved.  The warps form NW / WPT streams that
    // take the tiles round robin.
    static constexpr int WPT = 2;                        // consumer warps per tile
    static constexpr int KW = TILE / WPT;                // keys of a tile per warp
    static constexpr int MTW = KW / 16;                  // m-tiles of S^T = k-steps of P.V per warp
    static constexpr int TILE_BYTES = TILE * ROW_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K codes, V codes
    static constexpr int CHUNKS = ROW_BYTES / 16;
    static constexpr int CPAIRS = D / 32;                // 32-code blocks of a row
    static constexpr int NW = 8;
    // Warps: 0 issues the copies, 4 merges, 8 only takes part in the
    // set-up, the other eight compute.  A warp runs on scheduler (SMSP)
    // warp mod 4, so the copy-issuing warp shares its scheduler with no
    // consumer: consumers there delay its issue and, with it, the stream.
    static constexpr int THREADS = (NW + 3) * 32;
    static constexpr int ACTIVE_THREADS = (NW + 2) * 32;  // all but the idle warp
    static constexpr int PRODUCER_WARP = 0, MERGER_WARP = 4, IDLE_WARP = 8;
    static constexpr int SCR_ACC_FLOATS = NW * G * D;
    static constexpr int SCR_ML_FLOATS = NW * G * 2;
    static constexpr int VL_CACHE = 256;
    static constexpr int N_FLAGS = 8;
    // per stage besides the codes: TILE K scales + TILE V scales (in their own array)
    static constexpr int SCALE_BYTES = 2 * TILE * 4;
    static constexpr int FIXED_SMEM =
        1024 + 16 + 4 * (SCR_ACC_FLOATS + SCR_ML_FLOATS) + 4 * N_FLAGS + 4 * VL_CACHE;
    static_assert(D == 128, "the int8 kernel reads whole 128-byte rows");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the swizzle-atom alignment");

    // Shared-memory address of 16-byte chunk c of row r of a swizzled tile.
    __device__ __forceinline__ static uint32_t swz(uint32_t tile, int r, int c) {
        return tile + uint32_t(r) * 128 + uint32_t(((c & 7) ^ (r & 7)) << 4);
    }
};

namespace q8 {

// Two int8 codes, picked from a 32-bit word by a byte selector for the low
// bytes of each 16-bit half, as an fp16 pair: (1024 + (code ^ 0x80)) - 1152.
__device__ __forceinline__ uint32_t to_f16x2(uint32_t flipped, uint32_t sel) {
    const uint32_t w = __byte_perm(flipped, 0x64646464u, sel);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&w), __halves2half2(__ushort_as_half(0x6480),
                                                                                     __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t f16x2_from_bf16x2(uint32_t b) {
    const float lo = __uint_as_float(b << 16), hi = __uint_as_float(b & 0xffff0000u);
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

}  // namespace q8

// Producer: codes through the tensor maps (one box of 128 codes x 128 rows
// for a whole tile, boxes of x 8 rows in a tail tile), the tail's last rows
// and every row scale by cp.async; in a fused step the new row is quantised
// by the warp itself (the append's own quantise_row_q8).
template <typename C>
__device__ __forceinline__ uint32_t produce_tiles_q8(const DecodeArgs &a, Walker walk, uint32_t stage0,
                                                     uint32_t scale0, uint32_t bar0, int ns, int64_t kv_slab,
                                                     volatile int *flags, int lane) {
    constexpr int TILE = C::TILE;
    uint32_t issued = 0, generic_written = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    const uint64_t pol = dev::l2_evict_first_policy();  // codes are read once per launch
    Piece pc;
    while (ok && walk.next(a, pc)) {
        const int seg = pc.b * a.H_kv + pc.kv;
        const int z = a.seg_base + seg;
        const uint8_t *kseg = a.K + int64_t(seg) * kv_slab;
        const uint8_t *vseg = a.V + int64_t(seg) * kv_slab;
        const float *kss = a.k_scale + int64_t(seg) * a.max_ctx;
        const float *vss = a.v_scale + int64_t(seg) * a.max_ctx;
        // In a fused step the segment's last row is this step's new row: the
        // warp quantises it from k_new / v_new into the stage and the cache;
        // no box or copy reads it from the stale cache.
        const int new_row = a.k_new ? pc.n - 1 : -1;
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
            const uint32_t kdst = stage0 + uint32_t(stage) * C::STAGE_BYTES, vdst = kdst + C::TILE_BYTES;
            const uint32_t sdst = scale0 + uint32_t(stage) * C::SCALE_BYTES;
            // A tile without the new row comes as one 128-row box per tensor,
            // a segment's ragged last tile included: its rows past nr are
            // copied but never used (their scores are -inf and their scaled
            // probabilities 0, both by selection, and a code is always a
            // finite integer).  Only a box that would run past max_ctx, and
            // the tile holding a fused step's new row, take boxes of 64, 32
            // and 8 rows over the rows before that row, and cp.async for the
            // last few.
            const bool has_new = new_row >= row0 && new_row < row0 + nr;
            const int nb = has_new ? new_row - row0 : nr;  // rows read from the cache
            const bool whole = !has_new && row0 + TILE <= a.max_ctx;
            const int boxed = whole ? TILE : (nb & ~7);    // rows the boxes bring
            if (lane == 0) {
                if (generic_written & (1u << stage)) dev::fence_proxy_async_smem();
                dev::mbar_expect_tx(full, 2u * uint32_t(boxed) * C::ROW_BYTES);
                if (whole) {
                    dev::tma_load_3d(kdst, &a.tm_k32, 0, row0, z, full, pol);
                    dev::tma_load_3d(vdst, &a.tm_v32, 0, row0, z, full, pol);
                } else {
                    int r = 0;
                    if (boxed - r >= 64) {
                        dev::tma_load_3d(kdst, &a.tm_k64, 0, row0, z, full, pol);
                        dev::tma_load_3d(vdst, &a.tm_v64, 0, row0, z, full, pol);
                        r += 64;
                    }
                    if (boxed - r >= 32) {
                        dev::tma_load_3d(kdst + r * 128, &a.tm_kr32, 0, row0 + r, z, full, pol);
                        dev::tma_load_3d(vdst + r * 128, &a.tm_vr32, 0, row0 + r, z, full, pol);
                        r += 32;
                    }
                    for (; r < boxed; r += 8) {
                        dev::tma_load_3d(kdst + r * 128, &a.tm_k8, 0, row0 + r, z, full, pol);
                        dev::tma_load_3d(vdst + r * 128, &a.tm_v8, 0, row0 + r, z, full, pol);
                    }
                }
            }
            // row scales: lane l takes rows l and l + 32 of K and of V
#pragma unroll
            for (int h = 0; h < TILE / 32; ++h) {
                const int r = lane + 32 * h;
                if (r < nb) {
                    dev::cp_async_4(sdst + 4 * r, kss + row0 + r);
                    dev::cp_async_4(sdst + 4 * (TILE + r), vss + row0 + r);
                }
            }
            if (!whole) {
                const int per = (nb - boxed) * C::CHUNKS;  // rows after the boxes, before a new row
                for (int i = lane; i < 2 * per; i += 32) {
                    const bool is_v = i >= per;
                    const int j = is_v ? i - per : i;
                    const int r = boxed + j / C::CHUNKS, c16 = j % C::CHUNKS;
                    const uint8_t *src = (is_v ? vseg : kseg) + int64_t(row0 + r) * C::ROW_BYTES + c16 * 16;
                    dev::cp_async_16(C::swz(is_v ? vdst : kdst, r, c16), src);
                }
                if (has_new) {
                    // the new row, K then V: lane l quantises elements
                    // [4l, 4l + 4) and stores their codes in the stage (16-byte
                    // chunk l / 4 of the swizzled row) and in the cache, with
                    // the row's scale beside them
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint8_t *src = (t ? a.v_new : a.k_new) + int64_t(seg) * (2 * C::ROW_BYTES) + 8 * lane;
                        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(src));
                        const float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                                            __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
                        float scale;
                        const uint32_t codes = dev::quantise_row_q8<4>(x, scale);
                        dev::st_shared_u32(C::swz(t ? vdst : kdst, nb, lane >> 2) + 4 * (lane & 3), codes);
                        uint8_t *cache = const_cast<uint8_t *>(t ? a.V : a.K);  // the caller's writable cache
                        reinterpret_cast<uint32_t *>(cache + int64_t(seg) * kv_slab +
                                                     int64_t(new_row) * C::ROW_BYTES)[lane] = codes;
                        if (lane == 0) {
                            dev::st_shared_f32(sdst + 4 * (t * TILE + nb), scale);
                            const_cast<float *>(t ? a.v_scale : a.k_scale)[int64_t(seg) * a.max_ctx + new_row] =
                                scale;
                        }
                    }
                }
                generic_written |= 1u << stage;
            } else {
                generic_written &= ~(1u << stage);
            }
            dev::cp_async_arrive(full);
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

template <int D, int G>
__global__ void __launch_bounds__(Q8Cfg<D, G>::THREADS, 1) decode_q8_kernel(const __grid_constant__ DecodeArgs a) {
    using C = Q8Cfg<D, G>;
    using T = __nv_bfloat16;  // q and output
    constexpr int NW = C::NW, TILE = C::TILE, CPAIRS = C::CPAIRS, MT = C::MTW, NSTREAM = NW / C::WPT;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int ns = a.n_stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t stage0 = dev::smem_addr(smem);
    const uint32_t bar0 = stage0 + uint32_t(ns) * C::STAGE_BYTES;  // full[ns], empty[ns]
    const uint32_t scr_full = bar0 + 16 * uint32_t(ns);
    const uint32_t scr_free = scr_full + 8;
    const uint32_t scale0 = scr_free + 8;                           // [ns][2][TILE] floats
    const float *scales = reinterpret_cast<const float *>(smem + (scale0 - stage0));
    float *scr_acc = reinterpret_cast<float *>(smem + (scale0 - stage0) + size_t(ns) * C::SCALE_BYTES);
    float *scr_ml = scr_acc + C::SCR_ACC_FLOATS;
    volatile int *flags = reinterpret_cast<volatile int *>(scr_ml + C::SCR_ML_FLOATS);
    int32_t *vl_cache = reinterpret_cast<int32_t *>(scr_ml + C::SCR_ML_FLOATS) + C::N_FLAGS;
    const int32_t *vl = a.B <= C::VL_CACHE ? vl_cache : a.valid_len;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&a.tm_k32);
        dev::prefetch_tensormap(&a.tm_v32);
        for (int s = 0; s < ns; ++s) {
            dev::mbar_init(bar0 + 8 * s, 1);
            dev::mbar_init(bar0 + 8 * (ns + s), C::WPT);  // released by both warps of a stream
        }
        dev::mbar_init(scr_full, NW);
        dev::mbar_init(scr_free, 1);
        flags[0] = 0;
        dev::fence_mbar_init();
    }
    // the set-up above overlaps the previous kernel on the stream; nothing
    // below runs before it has completed
    dev::grid_dependency_wait();
    dev::allow_dependents();
    if (a.B <= C::VL_CACHE)
        for (int b = threadIdx.x; b < a.B; b += C::THREADS) vl_cache[b] = __ldg(a.valid_len + b);
    __syncthreads();

    if (warp == C::IDLE_WARP) return;
    const Plan plan = make_plan(a, vl, lane);
    if (plan.r0 >= plan.r1 || plan.b >= a.B) return;  // uniform over the CTA
    Walker walk;
    walk.init(a, plan, vl);
    const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;

    float *fin_acc = reinterpret_cast<float *>(smem);   // the drained ring, for the final combine
    float *fin_ml = fin_acc + (NW + 1) * G * D;
    constexpr int FOLD_U = fold_batch<D, G>();

    // ---------------------------------------------------------------- producer
    if (warp == C::PRODUCER_WARP) {
        const uint32_t issued = produce_tiles_q8<C>(a, walk, stage0, scale0, bar0, ns, kv_slab, flags, lane);
        __syncwarp();
        dev::named_barrier_sync(2, C::ACTIVE_THREADS);
        if (lane == 0 && flags[0]) drain_copies(bar0, ns, issued, a.timeout_ns);
        __syncwarp();
        return;
    }
    // ---------------------------------------------------------------- merger
    if (warp == C::MERGER_WARP) {
        LaneState<D, G> st;
        FinalCombine job;
        const bool help = merge_pieces<T, D, G, NW, 1, false>(a, plan, walk, scr_acc, scr_ml, scr_full, scr_free,
                                                              flags, lane, st, job);
        if (lane == 0) {
            flags[1] = help;
            flags[2] = job.seg;
            flags[3] = job.c0;
            flags[4] = job.c1;
            flags[5] = job.me;
        }
        __syncwarp();
        dev::named_barrier_sync(3, (NW + 1) * 32);
        if (help) {
            st.template fold_partials<FOLD_U>(a, job.seg, job.c0 + NW, job.c1, NW + 1, job.me, lane);
            st.store_slot(fin_acc, fin_ml, NW, lane);
            dev::named_barrier_sync(3, (NW + 1) * 32);
            st.reduce_slots(fin_acc, fin_ml, NW + 1, lane);
            st.template write_output<T>(a, job.b, job.kv, lane);
            for (int c = job.c0 + lane; c <= job.c1; c += 32)
                if (c != job.me) dev::flag_store(a.ready + c + job.seg, 0);
            if (lane == 0) a.tickets[job.seg] = 0;
        }
        __syncwarp();
        dev::named_barrier_sync(2, C::ACTIVE_THREADS);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1 - (warp > C::MERGER_WARP) - (warp > C::IDLE_WARP);  // 0 .. NW - 1
    const int strm = cw / C::WPT;            // tiles strm, strm + NSTREAM, ...
    const int kofs = (cw % C::WPT) * C::KW;  // this warp's keys of a tile: [kofs, kofs + KW)
    const int gq = lane >> 2, tq = lane & 3;
    const int H = a.H_kv * G;
    // ldmatrix lanes.  K (non-.trans): matrices (keys 0-7, chunk c) (keys 8-15,
    // chunk c) (keys 0-7, chunk c+1) (keys 8-15, chunk c+1).  V (.trans):
    // (keys 0-7, chunk c) (keys 0-7, chunk c+1) (keys 8-15, chunk c) (keys 8-15, chunk c+1).
    const int k_row = ((lane >> 3) & 1) * 8 + (lane & 7), k_chunk = (lane >> 4) & 1;
    const int v_row = ((lane >> 4) & 1) * 8 + (lane & 7), v_chunk = (lane >> 3) & 1;

    uint32_t qb[CPAIRS][4];   // fp16 Q^T fragments, d permuted as the K codes are
    float o[CPAIRS][2][4];    // O^T accumulators: [32-d block][even/odd d][fragment]
    float m0, m1, l0, l1;     // heads 2tq and 2tq + 1
    uint32_t t = 0, piece = 0;
    int stage = 0;
    uint32_t round = 0;
    Piece pc;
    while (walk.next(a, pc)) {
        {
            const T *qrow = reinterpret_cast<const T *>(a.q) + (int64_t(pc.b) * H + pc.kv * G + gq) * D;
#pragma unroll
            for (int cp = 0; cp < CPAIRS; ++cp) {
                const int d0 = 32 * cp + 4 * tq;
                auto ld = [&](int d) {
                    return gq < G ? q8::f16x2_from_bf16x2(__ldg(reinterpret_cast<const uint32_t *>(qrow + d))) : 0u;
                };
                qb[cp][0] = ld(d0);
                qb[cp][1] = ld(d0 + 16);
                qb[cp][2] = ld(d0 + 2);
                qb[cp][3] = ld(d0 + 18);
            }
#pragma unroll
            for (int cp = 0; cp < CPAIRS; ++cp)
#pragma unroll
                for (int e = 0; e < 2; ++e) o[cp][e][0] = o[cp][e][1] = o[cp][e][2] = o[cp][e][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }

        for (int row0 = pc.lo; row0 < pc.hi; row0 += TILE, ++t) {
            const int cur_stage = stage;
            const uint32_t cur_round = round;
            if (++stage == ns) {
                stage = 0;
                ++round;
            }
            if (int(t % NSTREAM) != strm) continue;
            const int nr = min(TILE, pc.hi - row0);
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
            const float *ksc = scales + cur_stage * 2 * TILE, *vsc = ksc + TILE;
            if (kofs >= nr) {  // a tail tile with no live key in this warp's half
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(empty_bar);
                continue;
            }

            // ---- S^T = K . Q^T on the codes, then the K row scales
            float s[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int cp = 0; cp < CPAIRS; ++cp) {
                    uint32_t r[4];
                    dev::ldsm_x4(C::swz(ks_base, kofs + mt * 16 + k_row, 2 * cp + k_chunk), r);
                    uint32_t lo[4], hi[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t f = r[i] ^ 0x80808080u;
                        lo[i] = q8::to_f16x2(f, 0x5140);
                        hi[i] = q8::to_f16x2(f, 0x7362);
                    }
                    dev::mma_16816_f16(s[mt], lo, qb[cp][0], qb[cp][1]);
                    dev::mma_16816_f16(s[mt], hi, qb[cp][2], qb[cp][3]);
                }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int k = kofs + 16 * mt + gq;
                const float sa = ksc[k], sb = ksc[k + 8];   // rows past nr hold stale scales
                s[mt][0] = k < nr ? s[mt][0] * sa : -INFINITY;
                s[mt][1] = k < nr ? s[mt][1] * sa : -INFINITY;
                s[mt][2] = k + 8 < nr ? s[mt][2] * sb : -INFINITY;
                s[mt][3] = k + 8 < nr ? s[mt][3] * sb : -INFINITY;
            }

            // ---- online softmax per head column
            float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                x0 = fmaxf(x0, fmaxf(s[mt][0], s[mt][2]));
                x1 = fmaxf(x1, fmaxf(s[mt][1], s[mt][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, off));
                x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, off));
            }
            const float mn0 = fmaxf(m0, x0 * a.scale_log2), mn1 = fmaxf(m1, x1 * a.scale_log2);
            const float corr0 = exp2f(m0 - mn0), corr1 = exp2f(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float p[MT][4];
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                p[mt][0] = exp2f(fmaf(s[mt][0], a.scale_log2, -mn0));
                p[mt][1] = exp2f(fmaf(s[mt][1], a.scale_log2, -mn1));
                p[mt][2] = exp2f(fmaf(s[mt][2], a.scale_log2, -mn0));
                p[mt][3] = exp2f(fmaf(s[mt][3], a.scale_log2, -mn1));
                ps0 += p[mt][0] + p[mt][2];
                ps1 += p[mt][1] + p[mt][3];
            }
            l0 = fmaf(l0, corr0, ps0);
            l1 = fmaf(l1, corr1, ps1);
            if (__any_sync(FULL, (corr0 != 1.f) || (corr1 != 1.f))) {
#pragma unroll
                for (int cp = 0; cp < CPAIRS; ++cp)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        o[cp][e][0] *= corr0;
                        o[cp][e][1] *= corr1;
                        o[cp][e][2] *= corr0;
                        o[cp][e][3] *= corr1;
                    }
            }
            // ---- scaled probabilities P'[key][head] = p * scale_v[key] -> B fragments
            uint32_t pb[MT][2];
#pragma unroll
            for (int kst = 0; kst < MT; ++kst) {
                const int k = kofs + 16 * kst + gq;
                const float va = k < nr ? vsc[k] : 0.f, vb = k + 8 < nr ? vsc[k + 8] : 0.f;
                pb[kst][0] = dev::movmatrix_trans(q8::pack_f16(p[kst][0] * va, p[kst][1] * va));
                pb[kst][1] = dev::movmatrix_trans(q8::pack_f16(p[kst][2] * vb, p[kst][3] * vb));
            }
            // ---- O^T += V^T . P'^T on the codes
#pragma unroll
            for (int kst = 0; kst < MT; ++kst)
#pragma unroll
                for (int cp = 0; cp < CPAIRS; ++cp) {
                    uint32_t r[4];
                    dev::ldsm_x4_trans(C::swz(vs_base, kofs + kst * 16 + v_row, 2 * cp + v_chunk), r);
                    uint32_t ev[4], od[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t f = r[i] ^ 0x80808080u;
                        ev[i] = q8::to_f16x2(f, 0x6240);
                        od[i] = q8::to_f16x2(f, 0x7351);
                    }
                    dev::mma_16816_f16(o[cp][0], ev, pb[kst][0], pb[kst][1]);
                    dev::mma_16816_f16(o[cp][1], od, pb[kst][0], pb[kst][1]);
                }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(empty_bar);
        }

        // ---- end of piece: hand this warp's state to the merge warp
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(FULL, l0, off);
            l1 += __shfl_xor_sync(FULL, l1, off);
        }
        bool ok = !flags[0] &&
                  (piece == 0 || dev::mbar_wait_bounded(scr_free, (piece - 1) & 1, flags, a.timeout_ns));
        ok = __all_sync(FULL, ok);
        if (ok) {
            const int h0 = 2 * tq, h1 = 2 * tq + 1;
#pragma unroll
            for (int cp = 0; cp < CPAIRS; ++cp)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int d = 32 * cp + 2 * gq + e;
                    if (h0 < G) {
                        scr_acc[(cw * G + h0) * D + d] = o[cp][e][0];
                        scr_acc[(cw * G + h0) * D + d + 16] = o[cp][e][2];
                    }
                    if (h1 < G) {
                        scr_acc[(cw * G + h1) * D + d] = o[cp][e][1];
                        scr_acc[(cw * G + h1) * D + d + 16] = o[cp][e][3];
                    }
                }
            if (gq == 0) {
                if (h0 < G) {
                    scr_ml[(cw * G + h0) * 2] = m0;
                    scr_ml[(cw * G + h0) * 2 + 1] = l0;
                }
                if (h1 < G) {
                    scr_ml[(cw * G + h1) * 2] = m1;
                    scr_ml[(cw * G + h1) * 2 + 1] = l1;
                }
            }
        } else if (lane == 0) {
            if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
            flags[0] = 1;
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(scr_full);
        ++piece;
    }

    // ---- the final combine, when the merger asks for it
    dev::named_barrier_sync(3, (NW + 1) * 32);
    if (flags[1]) {
        const int seg = flags[2], c0 = flags[3], c1 = flags[4], me = flags[5];
        LaneState<D, G> st;
        st.clear();
        st.template fold_partials<FOLD_U>(a, seg, c0 + cw, c1, NW + 1, me, lane);
        st.store_slot(fin_acc, fin_ml, cw, lane);
        dev::named_barrier_sync(3, (NW + 1) * 32);
    }
    dev::named_barrier_sync(2, C::ACTIVE_THREADS);
}

template <int D, int G>
cudaError_t set_q8_max_smem(int bytes) {
    return cudaFuncSetAttribute(decode_q8_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, int G>
cudaError_t launch_q8(const DecodeArgs &a, int grid, int smem, cudaStream_t s) {
    return launch_pdl(decode_q8_kernel<D, G>, dim3(grid), dim3(Q8Cfg<D, G>::THREADS), smem, s, a);
}

template <int D, int G>
const DecodeKernelInfo *q8_decode_info() {
    using C = Q8Cfg<D, G>;
    // one stage per stream in use, one more being filled
    static const DecodeKernelInfo info = {C::TILE, C::NW / C::WPT, C::STAGE_BYTES + 16 + C::SCALE_BYTES, C::FIXED_SMEM,
                                          &set_q8_max_smem<D, G>, &launch_q8<D, G>, true, false, false, C::TILE,
                                          true};
    return &info;
}

}  // namespace kvc
