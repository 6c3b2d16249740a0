// kvc_decode.cuh -- split-context single-query decode attention for sm_103a.
//
// What it computes ("10.3 -- KV cache implementation details", section 5,
// attention bullet; "KV Cache Optimization: GQA Audit, In-Place Buffers,
// Persistent Prompts", #2 After, reads sliced to the live length):
//   out[b, j*G + h, :] = softmax_t(q[b, j*G + h, :] . K[b, j, t, :] / sqrt(D))
//                        . V[b, j, t, :]          for t < valid_len[b]
// where j is a KV head and G = H / H_kv query heads share it ("10.3",
// section 4.2; contiguous grouping).
//
// Decomposition.  The live rows of all (sequence, KV head) segments form one
// flattened row space of R = H_kv * sum_b valid_len[b] rows (segment s =
// b * H_kv + j holds valid_len[b] rows).  CTA c takes the contiguous range
// [c * chunk, (c + 1) * chunk) of it, chunk = ceil(R / gridDim.x), so every
// CTA streams the same number of K/V bytes whatever the length mix.  The
// range splits into pieces at segment boundaries.  For each piece the CTA
// produces the softmax state (running max m, sum l, unnormalised
// accumulator) of its G query heads; a piece that is a whole segment is
// normalised and written out directly, otherwise it is stored as a split
// partial and the last CTA to finish a segment (an atomic counter per
// segment) merges its partials with the log-sum-exp rule.
//
// Inside a CTA: warp 0 is the producer, one elected lane issuing 1-D bulk
// (TMA) copies of [tile_rows, D] K and V slabs -- contiguous in the cache
// layout -- into a ring of shared-memory stages guarded by mbarriers.  Only
// live rows are copied, so padded rows are never read from HBM.  NW consumer
// warps take the tiles round robin; each keeps its own online-softmax state
// (fp32, scores in the log2 domain: q is prescaled by log2(e) / sqrt(D)) and
// the warps' states are merged through shared memory at the end of a piece.
// Every K/V byte is read from HBM once for all G query heads.
//
// Lane mapping inside a warp for one tile: LPR = D / 8 lanes share a row
// (each owns 8 elements = one 16-byte chunk for 16-bit types, two for fp32),
// RPW = 32 / LPR rows are in flight per pass.  Scores are partial dot
// products over each lane's 8 elements, completed by a reduce-scatter over
// the LPR lanes that leaves every lane with the full scores of one row: lane
// `sub` accumulates pass i into slot i ^ (sub >> SHIFT), which makes the
// exchange at every level a plain shuffle of a fixed slot.  The probabilities
// go through a small per-warp shared buffer to the P.V pass, where each lane
// accumulates its 8 output dimensions for its rows; the row groups are
// summed at the end of a piece.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvc_internal.cuh"

namespace kvc {

template <typename T>
struct ElemOps;

template <>
struct ElemOps<__nv_bfloat16> {
    static constexpr int EPC = 8;  // elements per 16-byte chunk
    // bf16 is the top half of a binary32: widening is a shift / mask.
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x << 16);
        f[1] = __uint_as_float(v.x & 0xffff0000u);
        f[2] = __uint_as_float(v.y << 16);
        f[3] = __uint_as_float(v.y & 0xffff0000u);
        f[4] = __uint_as_float(v.z << 16);
        f[5] = __uint_as_float(v.z & 0xffff0000u);
        f[6] = __uint_as_float(v.w << 16);
        f[7] = __uint_as_float(v.w & 0xffff0000u);
    }
    // Widened pairs (element 2i, element 2i+1) for the packed fp32 FMA.
    __device__ __forceinline__ static void unpack2(const uint4 &v, float2 *f) {
        f[0] = make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
        f[1] = make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
        f[2] = make_float2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
        f[3] = make_float2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
    }
    __device__ __forceinline__ static __nv_bfloat16 round(float x) { return __float2bfloat16_rn(x); }
};

template <>
struct ElemOps<__half> {
    static constexpr int EPC = 8;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ __forceinline__ static void unpack2(const uint4 &v, float2 *f) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __half22float2(h[i]);
    }
    __device__ __forceinline__ static __half round(float x) { return __float2half_rn(x); }
};

template <>
struct ElemOps<float> {
    static constexpr int EPC = 4;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static void unpack2(const uint4 &v, float2 *f) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ __forceinline__ static float round(float x) { return x; }
};

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int pow2floor(int x) { return x >= 2 ? 2 * pow2floor(x / 2) : 1; }
constexpr int ilog2(int x) { return x >= 2 ? 1 + ilog2(x / 2) : 0; }

template <typename T, int D, int G>
struct DecodeCfg {
    static constexpr int EB = sizeof(T);
    static constexpr int EPC = 16 / EB;
    static constexpr int E = 8;              // elements of a row per lane
    static constexpr int CPL = E / EPC;      // 16-byte chunks of a row per lane
    static constexpr int LPR = D / E;        // lanes per row
    static constexpr int RPW = 32 / LPR;     // rows per warp pass
    static constexpr int ROW_BYTES = D * EB;
    // passes per tile: at most LPR (one row per lane after the reduction),
    // about 8 KB of K per tile, at most 64 score registers per lane
    static constexpr int NPASS =
        cmin(LPR, cmin(pow2floor(cmax(1, 8192 / (ROW_BYTES * RPW))), pow2floor(cmax(1, 64 / G))));
    static constexpr int TILE = RPW * NPASS;  // rows per tile
    static constexpr int SHIFT = ilog2(LPR / NPASS);
    static constexpr int TILE_BYTES = TILE * ROW_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
    static constexpr int NW = 7;                        // consumer warps (+1 producer = 256 threads)
    static constexpr int E2 = E / 2;                    // element pairs of a row per lane
    static constexpr int PC = EPC / 2;                  // pairs per 16-byte chunk
    static constexpr int GP = 2 * ((G + 1) & ~1);       // per row: (p, p) for each head, 16-byte padded
    static constexpr int PBUF_FLOATS = NW * TILE * GP;
    static constexpr int SCR_ACC_FLOATS = NW * G * D;
    static constexpr int SCR_ML_FLOATS = NW * G * 2;
    static constexpr int FIXED_SMEM = 4 * (PBUF_FLOATS + SCR_ACC_FLOATS + SCR_ML_FLOATS) + 16;
    static constexpr int THREADS = (NW + 1) * 32;

    static_assert(D % E == 0 && LPR >= 1 && LPR <= 32, "unsupported head width");
    static_assert(CPL >= 1 && E % EPC == 0, "bad chunking");
    static_assert(LPR % NPASS == 0, "passes must divide the lanes of a row");
    static_assert(TILE_BYTES % 128 == 0, "tiles must keep 128-byte alignment");
};

// --------------------------------------------------------------------------
// Planning: the CTA's range of the flattened row space and where it starts.
// Every warp computes it independently (no shared state, no block barrier).
// --------------------------------------------------------------------------
struct Plan {
    int64_t chunk, r0, r1;
    int b;        // sequence holding row r0
    int64_t pb;   // flattened offset of sequence b's first segment
    int n;        // valid_len[b]
};

// Live rows of sequence b, 0 for an out-of-range length.  `vl` is the
// valid_len array or a shared-memory copy of it.
template <class A>
__device__ __forceinline__ int live_len(const A &a, const int32_t *vl, int b) {
    const int v = vl[b];
    return (v >= 1 && v <= a.max_ctx) ? v : 0;
}

__device__ __forceinline__ int64_t warp_sum_i64(int64_t v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// A segment's rows in the flattened split space: its live rows rounded up to
// the granularity.
template <class A>
__device__ __forceinline__ int round_len(const A &a, int n) { return (n + a.gran - 1) / a.gran * a.gran; }

// The CTA's range as split `split` of `nsplit` (by default the CTA's index
// in the grid and the grid's size).
template <class A>
__device__ __forceinline__ Plan make_plan(const A &a, const int32_t *vl, int lane, int split, int nsplit) {
    Plan p;
    int64_t total = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        int n = 0;
        if (b < a.B) {
            n = live_len(a, vl, b);
            if (n == 0 && blockIdx.x == 0 && threadIdx.x < 32) dev::record_error(a.err, ERR_DEVICE_INDEX);
        }
        total += warp_sum_i64(round_len(a, n));
    }
    const int64_t R = total * a.H_kv;
    p.chunk = (R + nsplit - 1) / nsplit;
    p.chunk = (p.chunk + a.gran - 1) / a.gran * a.gran;  // split points fall on multiples of gran
    p.r0 = min(R, int64_t(split) * p.chunk);
    p.r1 = min(R, p.r0 + p.chunk);
    p.b = a.B;
    p.pb = 0;
    p.n = 0;
    if (p.r0 >= p.r1) return p;
    int64_t base = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        const int n = (b < a.B) ? live_len(a, vl, b) : 0;
        const int64_t w = int64_t(round_len(a, n)) * a.H_kv;
        int64_t incl = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int64_t excl = incl - w;
        const unsigned hit =
            __ballot_sync(0xffffffffu, n > 0 && base + excl <= p.r0 && p.r0 < base + incl);
        if (hit) {
            const int src = __ffs(hit) - 1;
            p.b = b0 + src;
            p.pb = base + __shfl_sync(0xffffffffu, excl, src);
            p.n = __shfl_sync(0xffffffffu, n, src);
            return p;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    return p;
}

template <class A>
__device__ __forceinline__ Plan make_plan(const A &a, const int32_t *vl, int lane) {
    return make_plan(a, vl, lane, int(blockIdx.x), int(gridDim.x));
}

// One maximal run of rows of one segment inside the CTA's range: live rows
// [lo, hi) of the segment; len is the segment's length in the split space.
struct Piece {
    int b, kv, lo, hi, n, len;
    int64_t seg_start;
};

struct Walker {
    const int32_t *vl;
    int b, kv, n;
    int64_t seg_start, r, r1;

    int len;  // round_len of n

    template <class A>
    __device__ __forceinline__ void init(const A &a, const Plan &p, const int32_t *lengths) {
        vl = lengths;
        b = p.b;
        n = p.n;
        len = round_len(a, n);
        r = p.r0;
        r1 = p.r1;
        kv = (len > 0) ? int((p.r0 - p.pb) / len) : 0;
        seg_start = p.pb + int64_t(kv) * len;
    }

    template <class A>
    __device__ __forceinline__ bool next(const A &a, Piece &pc) {
        if (r >= r1 || b >= a.B) return false;
        while (r >= seg_start + len) {
            seg_start += len;
            if (++kv == a.H_kv) {
                kv = 0;
                do {
                    ++b;
                    n = (b < a.B) ? live_len(a, vl, b) : 0;
                } while (b < a.B && n == 0);
                if (b >= a.B) return false;
                len = round_len(a, n);
            }
        }
        pc.b = b;
        pc.kv = kv;
        pc.n = n;
        pc.len = len;
        pc.seg_start = seg_start;
        pc.lo = int(r - seg_start);
        const int end = int(min(int64_t(len), r1 - seg_start));
        pc.hi = min(end, n);  // rounding rows hold no data
        r = seg_start + end;
        return true;
    }
};

// The producer: one thread walks the CTA's pieces and streams every tile of
// K and V into the stage ring with 1-D bulk copies.
template <typename C>
__device__ __forceinline__ uint32_t produce_tiles(const DecodeArgs &a, Walker walk, uint32_t stage0,
                                                  uint32_t bar0, int ns, int64_t kv_slab,
                                                  volatile int *flags) {
    constexpr int TILE = C::TILE;
    uint32_t issued = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    const uint64_t pol = dev::l2_evict_first_policy();  // K/V rows are read once per launch
    Piece pc;
    while (ok && walk.next(a, pc)) {
        const int64_t seg = int64_t(pc.b) * a.H_kv + pc.kv;
        const uint8_t *kseg = a.K + seg * kv_slab;
        const uint8_t *vseg = a.V + seg * kv_slab;
        // In a fused step the segment's last row is this step's new row: it
        // is copied from k_new / v_new, never from the stale cache row.
        const int new_row = a.k_new ? pc.n - 1 : -1;
        for (int row = pc.lo; row < pc.hi; row += TILE) {
            const int nr = min(TILE, pc.hi - row);
            if (round > 0 &&
                !dev::mbar_wait_bounded(bar0 + 8 * (ns + stage), (round - 1) & 1, flags, a.timeout_ns)) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
                ok = false;
                break;
            }
            const uint32_t bytes = uint32_t(nr) * C::ROW_BYTES;
            const uint32_t full = bar0 + 8 * stage;
            const uint32_t dst = stage0 + uint32_t(stage) * C::STAGE_BYTES;
            dev::mbar_arrive_expect_tx(full, 2 * bytes);
            if (new_row >= row && new_row < row + nr) {  // the new row is the tile's last
                const uint32_t old_bytes = uint32_t(new_row - row) * C::ROW_BYTES;
                if (old_bytes) {
                    dev::bulk_copy_g2s(dst, kseg + int64_t(row) * C::ROW_BYTES, old_bytes, full, pol);
                    dev::bulk_copy_g2s(dst + C::TILE_BYTES, vseg + int64_t(row) * C::ROW_BYTES, old_bytes, full, pol);
                }
                dev::bulk_copy_g2s(dst + old_bytes, a.k_new + seg * C::ROW_BYTES, C::ROW_BYTES, full);
                dev::bulk_copy_g2s(dst + C::TILE_BYTES + old_bytes, a.v_new + seg * C::ROW_BYTES, C::ROW_BYTES, full);
            } else {
                dev::bulk_copy_g2s(dst, kseg + int64_t(row) * C::ROW_BYTES, bytes, full, pol);
                dev::bulk_copy_g2s(dst + C::TILE_BYTES, vseg + int64_t(row) * C::ROW_BYTES, bytes, full, pol);
            }
            ++issued;
            if (++stage == ns) {
                stage = 0;
                ++round;
            }
        }
    }
    return issued;
}

// After an abort, wait (bounded) for the copies of the last ns issued tiles,
// the only ones that can still be in flight, before shared memory is freed.
__device__ __forceinline__ void drain_copies(uint32_t bar0, int ns, uint32_t issued,
                                             unsigned long long timeout_ns) {
    const volatile int never = 0;
    const uint32_t first = issued > uint32_t(ns) ? issued - ns : 0;
    for (uint32_t t = first; t < issued; ++t)
        dev::mbar_wait_bounded(bar0 + 8 * (t % ns), (t / ns) & 1, &never, timeout_ns);
}

// End of a piece, after every consumer warp has written its softmax state
// (max m, sum l, unnormalised accumulator) for the piece's G heads to
// scr_ml [NW][G][2] and scr_acc [NW][G][D]: merge the warps' states, then
// either normalise and write the output (the piece is a whole segment) or
// store a split partial; the last CTA to finish a segment merges its
// partials and writes the output.  Called by the NW consumer warps only.
template <typename T, int D, int G, int NW>
__device__ __forceinline__ void merge_piece(const DecodeArgs &a, const Plan &plan, const Piece &pc,
                                            const float *scr_acc, const float *scr_ml,
                                            volatile int *flags, int ctid) {
    using Ops = ElemOps<T>;
    const int H = a.H_kv * G;

    const int seg = pc.b * a.H_kv + pc.kv;
    if (a.k_new && pc.hi == pc.n) {
        // fused step: this CTA holds the segment's last row; store the new K
        // and V rows into the cache (nobody in this launch reads them there)
        constexpr int VECS = D * int(sizeof(T)) / 16;  // 16-byte vectors of a row
        const int64_t row_off = (int64_t(seg) * a.max_ctx + pc.n - 1) * (D * int64_t(sizeof(T)));
        for (int i = ctid; i < 2 * VECS; i += NW * 32) {
            const bool is_v = i >= VECS;
            const int v = is_v ? i - VECS : i;
            const uint4 x = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.v_new : a.k_new) +
                                                                  int64_t(seg) * D * int64_t(sizeof(T))) + v);
            reinterpret_cast<uint4 *>(const_cast<uint8_t *>(is_v ? a.V : a.K) + row_off)[v] = x;
        }
    }
    const int c0 = int(pc.seg_start / plan.chunk);
    const int c1 = int((pc.seg_start + pc.len - 1) / plan.chunk);
    const bool whole = (c0 == c1);
    T *ob = reinterpret_cast<T *>(a.out) + (int64_t(pc.b) * H + pc.kv * G) * D;
    const bool aborted = flags[0] != 0;
    if (!aborted) {
        for (int idx = ctid; idx < G * D; idx += NW * 32) {
            const int h = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, scr_ml[(w * G + h) * 2]);
            float L = 0.f, A = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float e = exp2f(scr_ml[(w * G + h) * 2] - M);
                L = fmaf(scr_ml[(w * G + h) * 2 + 1], e, L);
                A = fmaf(scr_acc[(w * G + h) * D + d], e, A);
            }
            if (whole) {
                ob[h * D + d] = Ops::round(A / L);
            } else {
                const int slot = int(blockIdx.x) + seg;
                a.part_acc[(int64_t(slot) * G + h) * D + d] = A;
                if (d == 0) {
                    a.part_ml[(int64_t(slot) * G + h) * 2] = M;
                    a.part_ml[(int64_t(slot) * G + h) * 2 + 1] = L;
                }
            }
        }
    }
    if (!whole) {
        __threadfence();
        dev::named_barrier_sync(1, NW * 32);
        if (ctid == 0) {
            int last = 0;
            if (!flags[0]) last = atomicAdd(a.tickets + seg, 1) == c1 - c0;
            flags[1] = last;
        }
        dev::named_barrier_sync(1, NW * 32);
        if (flags[1]) {
            __threadfence();
            for (int idx = ctid; idx < G * D; idx += NW * 32) {
                const int h = idx / D, d = idx % D;
                float M = -INFINITY;
                for (int c = c0; c <= c1; ++c)
                    M = fmaxf(M, __ldcg(a.part_ml + (int64_t(c + seg) * G + h) * 2));
                float L = 0.f, A = 0.f;
                for (int c = c0; c <= c1; ++c) {
                    const int64_t sl = int64_t(c + seg) * G + h;
                    const float e = exp2f(__ldcg(a.part_ml + sl * 2) - M);
                    L = fmaf(__ldcg(a.part_ml + sl * 2 + 1), e, L);
                    A = fmaf(__ldcg(a.part_acc + sl * D + d), e, A);
                }
                ob[h * D + d] = Ops::round(A / L);
            }
            if (ctid == 0) a.tickets[seg] = 0;
        }
    }
    dev::named_barrier_sync(1, NW * 32);
}

// --------------------------------------------------------------------------
// The kernel.
// --------------------------------------------------------------------------
template <typename T, int D, int G>
__global__ void __launch_bounds__(DecodeCfg<T, D, G>::THREADS, 1)
    decode_split_kernel(const __grid_constant__ DecodeArgs a) {
    using C = DecodeCfg<T, D, G>;
    using Ops = ElemOps<T>;
    constexpr int NW = C::NW, LPR = C::LPR, RPW = C::RPW, EPC = C::EPC, CPL = C::CPL;
    constexpr int NPASS = C::NPASS, TILE = C::TILE, SHIFT = C::SHIFT;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(1024) uint8_t smem[];
    const int ns = a.n_stages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t stage0 = dev::smem_addr(smem);
    const uint32_t bar0 = stage0 + uint32_t(ns) * C::STAGE_BYTES;  // full[ns], then empty[ns]
    float *pbuf = reinterpret_cast<float *>(smem + size_t(ns) * C::STAGE_BYTES + 16 * size_t(ns));
    float *scr_acc = pbuf + C::PBUF_FLOATS;
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
    // the set-up above overlaps the previous kernel on the stream; nothing
    // below runs before it has completed
    dev::grid_dependency_wait();
    dev::allow_dependents();
    __syncthreads();

    const Plan plan = make_plan(a, a.valid_len, lane);
    if (plan.r0 >= plan.r1 || plan.b >= a.B) return;  // uniform over the CTA

    Walker walk;
    walk.init(a, plan, a.valid_len);
    const int64_t kv_slab = int64_t(a.max_ctx) * C::ROW_BYTES;  // bytes per (b, kv)

    // ---------------------------------------------------------------- producer
    if (warp == 0) {
        uint32_t issued = 0;
        if (lane == 0) issued = produce_tiles<C>(a, walk, stage0, bar0, ns, kv_slab, flags);
        __syncwarp();
        dev::named_barrier_sync(2, C::THREADS);  // every warp is done
        if (lane == 0 && flags[0]) drain_copies(bar0, ns, issued, a.timeout_ns);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int ctid = threadIdx.x - 32;
    const int grp = lane / LPR;
    const int sub = lane % LPR;
    const int my_row = (sub >> SHIFT) * RPW + grp;            // row held after the reduction
    const bool owner = (sub & ((1 << SHIFT) - 1)) == 0;       // one lane per row counts it
    float *pb = pbuf + cw * TILE * C::GP;
    const int H = a.H_kv * G;

    constexpr int E2 = C::E2, PC = C::PC, GP = C::GP;
    float2 qr[G][E2], acc[G][E2];
    float m[G], l[G];
    uint32_t t = 0;
    int stage = 0;
    uint32_t round = 0;
    Piece pc;
    while (walk.next(a, pc)) {
        // Query rows of this segment's G heads, prescaled into the log2 domain.
        {
            const T *qb = reinterpret_cast<const T *>(a.q) + (int64_t(pc.b) * H + pc.kv * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(qb + h * D) + sub + c * LPR);
                    Ops::unpack2(raw, &qr[h][c * PC]);
                }
#pragma unroll
                for (int e = 0; e < E2; ++e) {
                    qr[h][e].x *= a.scale_log2;
                    qr[h][e].y *= a.scale_log2;
                    acc[h][e] = make_float2(0.f, 0.f);
                }
                m[h] = -INFINITY;
                l[h] = 0.f;
            }
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
            // The previous use of this stage (tile t - ns) belongs to another
            // warp and copies may land out of order, so when this warp gets
            // here the full barrier may be in phase r-1 (t - ns still landing),
            // r, or r+1 (t already landed): r-1 and r+1 share a parity.  So
            // first wait until tile t - ns has been released (empty barrier,
            // phase r-1).  That barrier can only be in phase r-1 or r: t - ns
            // was issued before this warp's previous tile, and only this warp
            // can release t.  Once t - ns is released its data had landed, so
            // the full barrier is in phase r or r+1 and its parity wait is exact.
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
            const uint8_t *ks = smem + size_t(cur_stage) * C::STAGE_BYTES;
            const uint8_t *vs = ks + C::TILE_BYTES;

            // ---- scores: partial dot products, then reduce-scatter over the row's lanes
            float s[NPASS][G];
#pragma unroll
            for (int j = 0; j < NPASS; ++j) {
                const int row = (j ^ (sub >> SHIFT)) * RPW + grp;
                const uint8_t *rp = ks + row * C::ROW_BYTES;
                float2 kf[E2];
#pragma unroll
                for (int c = 0; c < CPL; ++c)
                    Ops::unpack2(*reinterpret_cast<const uint4 *>(rp + (sub + c * LPR) * 16), &kf[c * PC]);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    // even and odd elements in the two halves of a packed FMA
                    float2 d = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < E2; ++e) d = __ffma2_rn(qr[h][e], kf[e], d);
                    s[j][h] = d.x + d.y;
                }
            }
#pragma unroll
            for (int lv = NPASS / 2; lv >= 1; lv >>= 1) {
#pragma unroll
                for (int j = 0; j < lv; ++j)
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        s[j][h] += __shfl_xor_sync(FULL, s[j + lv][h], lv << SHIFT);
            }
#pragma unroll
            for (int bm = (1 << SHIFT) >> 1; bm >= 1; bm >>= 1)
#pragma unroll
                for (int h = 0; h < G; ++h) s[0][h] += __shfl_xor_sync(FULL, s[0][h], bm);

            // ---- online softmax (warp-uniform running max per head)
            const bool live = my_row < nr;
            float corr[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float sc = live ? s[0][h] : -INFINITY;
                float tm = sc;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(FULL, tm, o));
                const float mn = fmaxf(m[h], tm);
                corr[h] = exp2f(m[h] - mn);
                m[h] = mn;
                const float p = exp2f(sc - mn);
                l[h] = fmaf(l[h], corr[h], owner ? p : 0.f);
                if (owner) *reinterpret_cast<float2 *>(pb + my_row * GP + 2 * h) = make_float2(p, p);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 c2 = make_float2(corr[h], corr[h]);
#pragma unroll
                for (int e = 0; e < E2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], c2);
            }
            __syncwarp();

            // ---- P.V: each lane accumulates its 8 dimensions over its rows
            if (nr == TILE) {
#pragma unroll
                for (int i = 0; i < NPASS; ++i) {
                    const int row = i * RPW + grp;
                    float2 pw[G], vf[E2];
#pragma unroll
                    for (int h = 0; h < G; ++h) pw[h] = *reinterpret_cast<const float2 *>(pb + row * GP + 2 * h);
                    const uint8_t *rp = vs + row * C::ROW_BYTES;
#pragma unroll
                    for (int c = 0; c < CPL; ++c)
                        Ops::unpack2(*reinterpret_cast<const uint4 *>(rp + (sub + c * LPR) * 16), &vf[c * PC]);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < E2; ++e) acc[h][e] = __ffma2_rn(pw[h], vf[e], acc[h][e]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NPASS; ++i) {
                    const int row = i * RPW + grp;
                    if (row < nr) {  // rows past the copied ones hold stale bytes
                        float2 pw[G], vf[E2];
#pragma unroll
                        for (int h = 0; h < G; ++h)
                            pw[h] = *reinterpret_cast<const float2 *>(pb + row * GP + 2 * h);
                        const uint8_t *rp = vs + row * C::ROW_BYTES;
#pragma unroll
                        for (int c = 0; c < CPL; ++c)
                            Ops::unpack2(*reinterpret_cast<const uint4 *>(rp + (sub + c * LPR) * 16),
                                         &vf[c * PC]);
#pragma unroll
                        for (int h = 0; h < G; ++h)
#pragma unroll
                            for (int e = 0; e < E2; ++e) acc[h][e] = __ffma2_rn(pw[h], vf[e], acc[h][e]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(bar0 + 8 * (ns + cur_stage));
        }

        // ---- end of piece: merge the warps' states
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) l[h] += __shfl_xor_sync(FULL, l[h], o);
        }
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < E2; ++e) {
                    acc[h][e].x += __shfl_xor_sync(FULL, acc[h][e].x, o);
                    acc[h][e].y += __shfl_xor_sync(FULL, acc[h][e].y, o);
                }
        if (grp == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int c = 0; c < CPL; ++c)
#pragma unroll
                    for (int i = 0; i < PC; ++i)
                        *reinterpret_cast<float2 *>(scr_acc + (cw * G + h) * D + (sub + c * LPR) * EPC + 2 * i) =
                            acc[h][c * PC + i];
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                scr_ml[(cw * G + h) * 2] = m[h];
                scr_ml[(cw * G + h) * 2 + 1] = l[h];
            }
        }
        dev::named_barrier_sync(1, NW * 32);
        merge_piece<T, D, G, NW>(a, plan, pc, scr_acc, scr_ml, flags, ctid);
    }
    dev::named_barrier_sync(2, C::THREADS);
}

template <typename T, int D, int G>
cudaError_t set_decode_max_smem(int bytes) {
    return cudaFuncSetAttribute(decode_split_kernel<T, D, G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T, int D, int G>
cudaError_t launch_decode(const DecodeArgs &a, int grid, int smem, cudaStream_t s) {
    return launch_pdl(decode_split_kernel<T, D, G>, dim3(grid), dim3(DecodeCfg<T, D, G>::THREADS), smem, s, a);
}

template <typename T, int D, int G>
const DecodeKernelInfo *decode_info() {
    using C = DecodeCfg<T, D, G>;
    static const DecodeKernelInfo info = {C::TILE, C::NW, C::STAGE_BYTES + 16, C::FIXED_SMEM,
                                          &set_decode_max_smem<T, D, G>, &launch_decode<T, D, G>, false};
    return &info;
}

}  // namespace kvc
