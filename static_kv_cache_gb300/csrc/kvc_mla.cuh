// kvc_mla.cuh -- decode attention over an MLA latent cache.
//
// "10.3 -- KV cache implementation details", section 4.3 (Multi-head Latent
// Attention): the cache holds one latent c of width d_c per token; head h
// rebuilds its key and value rows as W_UK[h] c and W_UV[h] c (W of shape
// [d_h, d_c]).  "KV-Cache Mechanics" (MHA vs GQA vs MLA) names the decode
// cost of doing so the "absorb" overhead.  The absorbed order computes the
// same attention without rebuilding any row:
//
//   q~[b, h]    = W_UK[h]^T q[b, h]                 (mla_absorb_kernel)
//   s[b, h, t]  = q~[b, h] . c[b, t] / sqrt(d_h)
//   o~[b, h]    = sum_t softmax_t(s) c[b, t]        (mla_decode_kernel, per split)
//   out[b, h]   = W_UV[h] o~[b, h]                  (mla_combine_kernel)
//
// so every latent row is read once and serves as both the key and the value
// of all H heads.  Per row that is 4 H d_c FLOPs on d_c * p bytes, 2H FLOP/B
// (32 at H = 16 in bf16): the contractions run on the warp tensor-core path
// (mma.sync m16n8k16), keys or latent columns on the M side and the H heads on
// the N side, with fp32 accumulation.
//
// mla_decode_kernel: the flattened row space of the B sequences (one segment
// per sequence) is split evenly over the CTAs like the GQA decode kernels.
// A producer warp streams 64-row tiles of latents into a ring of stages with
// TMA (128-byte swizzle, one box per 64-column block; 16-row boxes for a
// tile's tail).  Four consumer warps share each tile: warp w forms the scores
// of keys [16w, 16w + 16) against all heads over the whole width, the four
// warps exchange per-head tile maxima and the bf16 probabilities through
// shared memory, then warp w accumulates columns [w d_c/4, (w+1) d_c/4) of the
// attended latent for all keys of the tile.  Every piece (one sequence's rows
// inside one CTA's range) leaves an fp32 partial (m, l, o~) in the workspace;
// mla_combine_kernel folds the partials of each sequence and applies W_UV.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvc_decode.cuh"

namespace kvc {

// Most CTAs the MLA decode launch uses; the workspace holds grid + B partial
// slots.
constexpr int MLA_MAX_CTAS = 256;

struct MlaArgs {
    // split planning (make_plan / Walker): one segment per sequence
    int32_t B, H_kv, max_ctx, gran;
    int32_t *err;
    const int32_t *valid_len;  // [B]
    const void *qt;            // absorbed queries [B, H_all, d_c], prescaled by log2(e) / sqrt(d_h)
    float *part_ml;            // [slots, H_all, 2]: running max (log2 domain) and sum
    float *part_acc;           // [slots, H_all, d_c]: unnormalised attended latent
    // More heads than one kernel instance takes: the grid is nsplit splits
    // x groups head groups of the kernel's H heads, CTA c taking split
    // c / groups for heads [(c % groups) H, (c % groups + 1) H) -- the
    // groups of one split are neighbours in the grid, so they run at the same
    // time and read the split's latent rows once from memory between them.
    int32_t H_all, groups;
    int32_t n_stages;
    int32_t seg_base;          // layer * B: the layer's first row block in the tensor maps
    unsigned long long timeout_ns;
    // the whole latent cache viewed as [L*B][max_ctx][d_c]: boxes of 64
    // columns x 64 rows and x 16 rows, 128-byte swizzle
    CUtensorMap tm64, tm16;
};

struct MlaAbsorbArgs {
    const void *q;        // [B, H, d_h]
    const void *w_uk;     // [H, d_h, d_c]
    void *qt;             // [B, H, d_c]
    const void *c_new;    // [B, d_c]: the step's latent row, appended at valid_len - 1; null: none
    void *cache;          // the layer's latent slab [B, max_ctx, d_c]
    const int32_t *valid_len;
    int32_t *err;
    int32_t B, H, d_h, d_c, max_ctx;
    float scale;          // log2(e) / sqrt(d_h)
};

struct MlaCombineArgs {
    const float *part_ml;
    const float *part_acc;
    const int32_t *valid_len;
    const void *w_uv;     // [H, d_h, d_c]
    void *out;            // [B, H, d_h]
    int32_t B, H, d_h, d_c, max_ctx;
    int32_t grid;         // CTAs of the decode launch whose partials these are
};

template <typename T>
struct MlaElem;
template <>
struct MlaElem<__nv_bfloat16> {
    __device__ __forceinline__ static float load(const __nv_bfloat16 &x) { return __bfloat162float(x); }
    __device__ __forceinline__ static __nv_bfloat16 store(float x) { return __float2bfloat16_rn(x); }
    __device__ __forceinline__ static void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        dev::mma_16816_bf16(d, a, b0, b1);
    }
};
template <>
struct MlaElem<__half> {
    __device__ __forceinline__ static float load(const __half &x) { return __half2float(x); }
    __device__ __forceinline__ static __half store(float x) { return __float2half_rn(x); }
    __device__ __forceinline__ static void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        dev::mma_16816_f16(d, a, b0, b1);
    }
};

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}

template <typename T, int DC, int H>
struct MlaCfg {
    static constexpr int TILE = 64;                       // latent rows per stage
    static constexpr int NW = 4;                          // consumer warps
    static constexpr int THREADS = (NW + 1) * 32;         // + the producer warp
    static constexpr int CB = DC / 64;                    // 128-byte column blocks of a row
    static constexpr int BLOCK_BYTES = TILE * 128;        // one column block of a tile
    static constexpr int STAGE_BYTES = CB * BLOCK_BYTES;
    static constexpr int NT = H / 8;                      // n-tiles of heads
    static constexpr int KS = DC / 16;                    // k-steps of the scores
    static constexpr int MTW = DC / NW / 16;              // P.V m-tiles (16 latent columns) per warp
    static constexpr int QS = DC + 8;                     // q~ row stride, elements (conflict-free ldmatrix)
    static constexpr int PS = TILE + 8;                   // probability row stride, elements
    // after the stages: 2 barriers per stage, q~ [H][QS], P [2][H][PS],
    // tile maxima [2][NW][H], sums [NW][H], abort votes [2], the abort flag
    static constexpr int FIXED_SMEM = 1024 + H * QS * 2 + 2 * H * PS * 2 + 4 * (2 * NW * H + NW * H) + 16;
    static constexpr int BARRIER_BYTES_PER_STAGE = 16;

    static_assert(H == 8 || H == 16, "heads on the N side: one or two n-tiles");
    static_assert(DC % 64 == 0 && DC >= 128 && DC <= 512, "latent width: 128-byte column blocks, 4 warps");
    static_assert(STAGE_BYTES % 1024 == 0, "stages keep the swizzle-atom alignment");
};

// ---------------------------------------------------------------------------
// Absorb: q~[b, h, j] = scale * sum_i q[b, h, i] W_UK[h, i, j], rounded once
// to the cache type; with c_new, also the step's latent row into the cache.
// Per head this is a [B x d_h] . [d_h x d_c] product, taken on mma.sync with
// fp32 accumulation.  Grid (H, DC / 64, ceil(B / 64)), 128 threads: block
// (h, y, z) computes columns [64 y, 64 y + 64) for sequences
// [64 z, 64 z + 64); warp w takes the 16 sequences 64 z + 16 w + [0, 16) and
// all 8 column n-tiles.  q rows and the W_UK[h] slice reach shared memory
// by cp.async (row strides padded by 16 bytes, so every ldmatrix is
// conflict-free); the W slice is [d][j], read transposed into B fragments.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int DH_MAX>
struct MlaAbsorbSmem {
    static constexpr int QS = DH_MAX + 8;                 // q row stride, elements
    static constexpr int WS = 64 + 8;                     // W slice row stride, elements
    static constexpr int BYTES = 64 * QS * 2 + DH_MAX * WS * 2;
};

template <typename T, int DC>
__global__ void __launch_bounds__(128) mla_absorb_kernel(const MlaAbsorbArgs a) {
    using E = MlaElem<T>;
    using S = MlaAbsorbSmem<256>;
    extern __shared__ __align__(16) uint8_t abs_smem[];
    T *qs = reinterpret_cast<T *>(abs_smem);                  // [64][QS]
    T *wsl = qs + 64 * S::QS;                                 // [d_h][WS]
    const int h = blockIdx.x, j0 = blockIdx.y * 64, b0 = blockIdx.z * 64;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int dh = a.d_h, vq = dh / 8;                        // 16-byte vectors per q row
    dev::grid_dependency_wait();   // the previous kernel on the stream has completed
    dev::allow_dependents();
    const T *q = static_cast<const T *>(a.q);
    const T *w = static_cast<const T *>(a.w_uk) + int64_t(h) * dh * DC + j0;
    for (int v = t; v < 64 * vq; v += 128) {
        const int r = v / vq, c = (v - r * vq) * 8;
        const uint32_t dst = dev::smem_addr(qs + r * S::QS + c);
        if (b0 + r < a.B) dev::cp_async_16(dst, q + (int64_t(b0 + r) * a.H + h) * dh + c);
        else *reinterpret_cast<uint4 *>(qs + r * S::QS + c) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int v = t; v < dh * 8; v += 128) {
        const int r = v >> 3, c = (v & 7) * 8;
        dev::cp_async_16(dev::smem_addr(wsl + r * S::WS + c), w + int64_t(r) * DC + c);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    cp_async_wait_all();
    __syncthreads();

    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int l7 = lane & 7, j8 = lane >> 3;
    // A (q rows x d): lane supplies row 16 w + (j8 & 1) * 8 + l7, columns (j8 >> 1) * 8
    const uint32_t a_addr = dev::smem_addr(qs + (16 * warp + (j8 & 1) * 8 + l7) * S::QS + (j8 >> 1) * 8);
    // B (d x columns) from W rows via .trans: lane supplies d row (j8 & 1) * 8 + l7, columns (j8 >> 1) * 8
    const uint32_t b_addr = dev::smem_addr(wsl + ((j8 & 1) * 8 + l7) * S::WS + (j8 >> 1) * 8);
    for (int ks = 0; ks < dh / 16; ++ks) {
        uint32_t af[4];
        dev::ldsm_x4(a_addr + ks * 32, af);
#pragma unroll
        for (int np = 0; np < 4; ++np) {     // pairs of n-tiles
            uint32_t bf[4];
            dev::ldsm_x4_trans(b_addr + (ks * 16 * S::WS + np * 16) * 2, bf);
            E::mma(acc[2 * np], af, bf[0], bf[1]);
            E::mma(acc[2 * np + 1], af, bf[2], bf[3]);
        }
    }
    T *qt = static_cast<T *>(a.qt);
    const int rb = b0 + 16 * warp + (lane >> 2);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const int j = j0 + nt * 8 + 2 * (lane & 3);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int b = rb + 8 * hf;
            if (b < a.B) {
                T pair[2] = {E::store(acc[nt][2 * hf] * a.scale), E::store(acc[nt][2 * hf + 1] * a.scale)};
                *reinterpret_cast<uint32_t *>(qt + (int64_t(b) * a.H + h) * DC + j) = *reinterpret_cast<uint32_t *>(pair);
            }
        }
    }
    if (a.c_new && h == 0) {
        // the step's latent rows of the block's sequences and columns: 64 x 64
        const T *cn = static_cast<const T *>(a.c_new);
        T *cache = static_cast<T *>(a.cache);
        for (int i = t; i < 64 * 8; i += 128) {
            const int bb = i >> 3, c = (i & 7) * 8, b = b0 + bb;
            if (b >= a.B) break;
            const int v = __ldg(a.valid_len + b);
            if (v >= 1 && v <= a.max_ctx)
                *reinterpret_cast<uint4 *>(cache + (int64_t(b) * a.max_ctx + v - 1) * DC + j0 + c) =
                    __ldg(reinterpret_cast<const uint4 *>(cn + int64_t(b) * DC + j0 + c));
            else if (c == 0 && blockIdx.y == 0)
                dev::record_error(a.err, ERR_DEVICE_INDEX);
        }
    }
}

// ---------------------------------------------------------------------------
template <typename T, int DC, int H>
__global__ void __launch_bounds__(MlaCfg<T, DC, H>::THREADS, 1) mla_decode_kernel(const __grid_constant__ MlaArgs a) {
    using C = MlaCfg<T, DC, H>;
    using E = MlaElem<T>;
    constexpr int TILE = C::TILE, NW = C::NW, NT = C::NT, MTW = C::MTW, BB = C::BLOCK_BYTES;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int ns = a.n_stages;
    const uint32_t stage0 = dev::smem_addr(smem);
    const uint32_t bar0 = stage0 + uint32_t(ns) * C::STAGE_BYTES;  // full[ns], then empty[ns]
    uint8_t *rest = smem + size_t(ns) * (C::STAGE_BYTES + C::BARRIER_BYTES_PER_STAGE);
    T *q_s = reinterpret_cast<T *>(rest);                           // [H][QS]
    T *p_s = q_s + H * C::QS;                                       // [2][H][PS]
    float *red = reinterpret_cast<float *>(p_s + 2 * H * C::PS);    // [2][NW][H]
    float *lsum = red + 2 * NW * H;                                 // [NW][H]
    volatile int *vote = reinterpret_cast<volatile int *>(lsum + NW * H);  // [2]
    volatile int *flags = vote + 2;                                 // [0]: abort
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            dev::mbar_init(bar0 + 8 * s, 1);
            dev::mbar_init(bar0 + 8 * (ns + s), NW);
        }
        vote[0] = vote[1] = 0;
        flags[0] = 0;
        dev::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        dev::prefetch_tensormap(&a.tm64);
        dev::prefetch_tensormap(&a.tm16);
    }
    __syncthreads();  // the barriers are initialised for every role
    // The set-up above overlaps the previous kernel on the stream: the absorb
    // launch of the same call.  The consumers touch nothing before it has
    // completed; the producer starts earlier (below).
    if (warp != 0) {
        dev::grid_dependency_wait();
        dev::allow_dependents();
    }

    const int split = int(blockIdx.x) / a.groups, head0 = (int(blockIdx.x) % a.groups) * H;
    const Plan plan = make_plan(a, a.valid_len, lane, split, int(gridDim.x) / a.groups);
    if (plan.r0 >= plan.r1 || plan.b >= a.B) return;  // uniform over the CTA
    Walker walk;
    walk.init(a, plan, a.valid_len);

    // ---------------------------------------------------------------- producer
    if (warp == 0) {
        // The producer plans and copies before its dependency wait.  This
        // launch can only start once every CTA of the absorb launch has passed
        // its own wait for the kernel before it (the absorb signals its
        // dependents right after that wait), so the valid lengths and every
        // latent row but each sequence's last live one (the new row, which
        // the absorb itself writes) are in place.  Tiles that do not hold a
        // sequence's last live row go ahead; the wait comes before the first
        // tile that does, or before the ring's first reuse, whichever is
        // first.
        bool waited = false;
        uint32_t t = 0;
        bool ok = true;
        // one head group: the latent rows are read once per launch; several:
        // the split's other groups read the same rows from L2 alongside
        const uint64_t pol = a.groups > 1 ? dev::l2_evict_normal_policy() : dev::l2_evict_first_policy();
        Piece pc;
        while (ok && walk.next(a, pc)) {
            const int z = a.seg_base + pc.b;
            for (int row0 = pc.lo; row0 < pc.hi; row0 += TILE, ++t) {
                const int nr = min(TILE, pc.hi - row0);
                const int s = int(t % uint32_t(ns));
                const uint32_t r = t / uint32_t(ns);
                if (!waited && (r > 0 || row0 + nr == pc.n)) {
                    dev::grid_dependency_wait();
                    dev::allow_dependents();
                    waited = true;
                }
                if (r > 0) {
                    const bool w = dev::mbar_wait_bounded(bar0 + 8 * (ns + s), (r - 1) & 1, flags, a.timeout_ns);
                    if (!__all_sync(FULL, w)) {
                        if (lane == 0) {
                            if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                            flags[0] = 1;
                        }
                        ok = false;
                        break;
                    }
                }
                if (lane == 0) {
                    const uint32_t full = bar0 + 8 * s;
                    const uint32_t dst = stage0 + uint32_t(s) * C::STAGE_BYTES;
                    if (nr == TILE) {
                        dev::mbar_arrive_expect_tx(full, C::STAGE_BYTES);
#pragma unroll
                        for (int cb = 0; cb < C::CB; ++cb) dev::tma_load_3d(dst + cb * BB, &a.tm64, cb * 64, row0, z, full, pol);
                    } else {
                        const int nb = (nr + 15) >> 4;
                        dev::mbar_arrive_expect_tx(full, uint32_t(nb) * C::CB * 16 * 128);
                        for (int j = 0; j < nb; ++j)
#pragma unroll
                            for (int cb = 0; cb < C::CB; ++cb)
                                dev::tma_load_3d(dst + cb * BB + j * 2048, &a.tm16, cb * 64, row0 + 16 * j, z, full, pol);
                    }
                }
                __syncwarp();
            }
        }
        if (!waited) {
            dev::grid_dependency_wait();
            dev::allow_dependents();
        }
        __syncwarp();
        dev::named_barrier_sync(2, C::THREADS);  // every warp is done
        if (lane == 0 && flags[0]) drain_copies(bar0, ns, t, a.timeout_ns);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int ctid = threadIdx.x - 32;
    const int l7 = lane & 7, j8 = lane >> 3;
    // ldmatrix row offsets.  Scores, A = latent rows (keys) x columns: lane
    // supplies key 16cw + (j8 & 1) * 8 + l7, columns (j8 >> 1) * 8 of a k-step.
    uint32_t a_off[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        a_off[kk] = uint32_t(16 * cw + (j8 & 1) * 8 + l7) * 128 + uint32_t(((2 * kk + (j8 >> 1)) ^ l7) << 4);
    // P.V, A = latent columns x keys (ldmatrix .trans): lane supplies key
    // (j8 >> 1) * 8 + l7 of a 16-key step, columns 16 mt + (j8 & 1) * 8.
    uint32_t v_off[MTW];
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) {
        const int col = 16 * (cw * MTW + mt) + (j8 & 1) * 8;
        v_off[mt] = uint32_t(col >> 6) * BB + uint32_t((j8 >> 1) * 8 + l7) * 128 + uint32_t((((col >> 3) & 7) ^ l7) << 4);
    }
    // B fragments: rows of q~ (heads) and of P (heads), 8 elements each.
    const int b_row = (j8 >> 1) * 8 + l7, b_col = (j8 & 1) * 8;
    const uint32_t q_addr = dev::smem_addr(q_s) + uint32_t(b_row * C::QS + b_col) * 2;
    const uint32_t p_addr0 = dev::smem_addr(p_s) + uint32_t(b_row * C::PS + b_col) * 2;

    const int key0 = 16 * cw + (lane >> 2);  // keys of this lane's score rows: key0, key0 + 8
    const int hq = 2 * (lane & 3);           // heads of this lane's columns: nt*8 + hq + {0, 1}
    uint32_t t = 0;
    bool ok = true;
    Piece pc;
    while (ok && walk.next(a, pc)) {
        // the sequence's absorbed queries into shared memory
        dev::named_barrier_sync(1, NW * 32);
        {
            const uint4 *src =
                reinterpret_cast<const uint4 *>(static_cast<const T *>(a.qt) + (int64_t(pc.b) * a.H_all + head0) * DC);
            for (int i = ctid; i < H * DC / 8; i += NW * 32) {
                const int h = i / (DC / 8), c = i - h * (DC / 8);
                *reinterpret_cast<uint4 *>(q_s + h * C::QS + c * 8) = __ldg(src + i);
            }
        }
        dev::named_barrier_sync(1, NW * 32);

        float o[MTW][NT][4];
        float m_run[NT][2], l_run[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_run[nt][0] = m_run[nt][1] = -INFINITY;
            l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        }

        for (int row0 = pc.lo; row0 < pc.hi; row0 += TILE, ++t) {
            const int nr = min(TILE, pc.hi - row0);
            const int s = int(t % uint32_t(ns));
            const uint32_t r = t / uint32_t(ns);
            const int buf = int(t & 1);
            // the four warps consume every tile together, so round r - 1 of
            // this stage was theirs and its full phase has completed
            bool w_ok = dev::mbar_wait_bounded(bar0 + 8 * s, r & 1, flags, a.timeout_ns);
            w_ok = __all_sync(FULL, w_ok);
            const uint32_t stage = stage0 + uint32_t(s) * C::STAGE_BYTES;
            float sc[NT][4];
            if (w_ok) {
                if (nr < TILE) {
                    // rows past the tile's live rows: zero (they may hold
                    // anything, and P.V multiplies them by 0)
                    const int z0 = max(nr, 16 * cw), z1 = 16 * cw + 16;
                    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
                    for (int i = lane; i < (z1 - z0) * C::CB * 8; i += 32) {
                        const int row = z0 + i / (C::CB * 8), rr = i % (C::CB * 8);
                        dev::st_shared_v4(stage + uint32_t(rr >> 3) * BB + uint32_t(row) * 128 + uint32_t(rr & 7) * 16, zero);
                    }
                    dev::fence_proxy_async_smem();
                    __syncwarp();
                }
                // scores of keys [16cw, 16cw + 16) for all heads, two chains
                float sa[2][NT][4];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) sa[c2][nt][0] = sa[c2][nt][1] = sa[c2][nt][2] = sa[c2][nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    uint32_t af[4];
                    dev::ldsm_x4(stage + uint32_t(ks >> 2) * BB + a_off[ks & 3], af);
                    if constexpr (NT == 2) {
                        uint32_t bf[4];
                        dev::ldsm_x4(q_addr + ks * 32, bf);
                        E::mma(sa[ks & 1][0], af, bf[0], bf[1]);
                        E::mma(sa[ks & 1][1], af, bf[2], bf[3]);
                    } else {
                        uint32_t b0, b1;
                        ldsm_x2(q_addr + ks * 32, b0, b1);
                        E::mma(sa[ks & 1][0], af, b0, b1);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] = sa[0][nt][e] + sa[1][nt][e];
            } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = -INFINITY;
                if (lane == 0) {
                    vote[buf] = 1;
                    if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                    flags[0] = 1;
                }
            }
            // mask keys past the tile's live rows; per-head maxima of the tile
            float mx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (key0 >= nr) sc[nt][0] = sc[nt][1] = -INFINITY;
                if (key0 + 8 >= nr) sc[nt][2] = sc[nt][3] = -INFINITY;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float v = fmaxf(sc[nt][e], sc[nt][e + 2]);
                    v = fmaxf(v, __shfl_xor_sync(FULL, v, 4));
                    v = fmaxf(v, __shfl_xor_sync(FULL, v, 8));
                    v = fmaxf(v, __shfl_xor_sync(FULL, v, 16));
                    mx[nt][e] = v;
                }
            }
            if (lane < 4) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    red[(buf * NW + cw) * H + nt * 8 + hq] = mx[nt][0];
                    red[(buf * NW + cw) * H + nt * 8 + hq + 1] = mx[nt][1];
                }
            }
            dev::named_barrier_sync(1, NW * 32);  // maxima and abort votes visible
            if (vote[buf]) {  // set only by a failed wait, never cleared: all warps leave at this tile
                ok = false;
                break;
            }
            T *pb = p_s + buf * H * C::PS;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float alpha[2], mn[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int head = nt * 8 + hq + e;
                    float tm = red[(buf * NW + 0) * H + head];
#pragma unroll
                    for (int w = 1; w < NW; ++w) tm = fmaxf(tm, red[(buf * NW + w) * H + head]);
                    mn[e] = fmaxf(m_run[nt][e], tm);
                    alpha[e] = exp2f(m_run[nt][e] - mn[e]);
                    m_run[nt][e] = mn[e];
                }
                const float p0 = exp2f(sc[nt][0] - mn[0]), p1 = exp2f(sc[nt][1] - mn[1]);
                const float p2 = exp2f(sc[nt][2] - mn[0]), p3 = exp2f(sc[nt][3] - mn[1]);
                l_run[nt][0] = l_run[nt][0] * alpha[0] + p0 + p2;
                l_run[nt][1] = l_run[nt][1] * alpha[1] + p1 + p3;
                const int h0 = nt * 8 + hq;
                pb[h0 * C::PS + key0] = E::store(p0);
                pb[(h0 + 1) * C::PS + key0] = E::store(p1);
                pb[h0 * C::PS + key0 + 8] = E::store(p2);
                pb[(h0 + 1) * C::PS + key0 + 8] = E::store(p3);
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    o[mt][nt][0] *= alpha[0];
                    o[mt][nt][1] *= alpha[1];
                    o[mt][nt][2] *= alpha[0];
                    o[mt][nt][3] *= alpha[1];
                }
            }
            dev::named_barrier_sync(1, NW * 32);  // probabilities and zeroed rows visible
            // P.V: latent columns of this warp x all keys of the tile
            const uint32_t p_addr = p_addr0 + uint32_t(buf * H * C::PS) * 2;
#pragma unroll
            for (int kst = 0; kst < TILE / 16; ++kst) {
                uint32_t pf[NT][2];
                if constexpr (NT == 2) {
                    uint32_t r4[4];
                    dev::ldsm_x4(p_addr + kst * 32, r4);
                    pf[0][0] = r4[0];
                    pf[0][1] = r4[1];
                    pf[1][0] = r4[2];
                    pf[1][1] = r4[3];
                } else {
                    ldsm_x2(p_addr + kst * 32, pf[0][0], pf[0][1]);
                }
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    uint32_t af[4];
                    dev::ldsm_x4_trans(stage + v_off[mt] + kst * 2048, af);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) E::mma(o[mt][nt], af, pf[nt][0], pf[nt][1]);
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(bar0 + 8 * (ns + s));
        }
        if (!ok) break;

        // the piece's partial: m and l per head, and this warp's columns of o~
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = l_run[nt][e];
                v += __shfl_xor_sync(FULL, v, 4);
                v += __shfl_xor_sync(FULL, v, 8);
                v += __shfl_xor_sync(FULL, v, 16);
                l_run[nt][e] = v;
            }
        if (lane < 4) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                lsum[cw * H + nt * 8 + hq] = l_run[nt][0];
                lsum[cw * H + nt * 8 + hq + 1] = l_run[nt][1];
            }
        }
        dev::named_barrier_sync(1, NW * 32);
        const int64_t slot = int64_t(split) + pc.b;
        if (cw == 0 && lane < 4) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int head = nt * 8 + hq + e;
                    float L = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) L += lsum[w * H + head];
                    a.part_ml[(slot * a.H_all + head0 + head) * 2] = m_run[nt][e];
                    a.part_ml[(slot * a.H_all + head0 + head) * 2 + 1] = L;
                }
        }
        float *acc = a.part_acc + (slot * a.H_all + head0) * DC;
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = 16 * (cw * MTW + mt) + (lane >> 2);
                const int h0 = nt * 8 + hq;
                acc[h0 * DC + col] = o[mt][nt][0];
                acc[(h0 + 1) * DC + col] = o[mt][nt][1];
                acc[h0 * DC + col + 8] = o[mt][nt][2];
                acc[(h0 + 1) * DC + col + 8] = o[mt][nt][3];
            }
    }
    dev::named_barrier_sync(2, C::THREADS);
}

// ---------------------------------------------------------------------------
// Combine and up-project: for each sequence b and head h, fold the partials
// of b's splits (slots [c0 + b, c1 + b], the CTAs whose ranges meet b's rows)
// into o~ = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), round it once to
// the cache type, then out[b, h] = W_UV[h] o~ on mma.sync (fp32
// accumulation), rounded once.  Grid (H, ceil(B / 16), ceil(d_h / 64)), 512
// threads.  The block's 64 rows of W_UV[h] start towards shared memory
// (cp.async) first; meanwhile warp k folds sequence 16 y + k (its lanes over
// the splits, then over the columns, every split's loads issued together);
// then warps 0-7 each take one 8-row n-tile of the block's rows against the
// 16 sequences over all of d_c.  The d_h / 64 blocks of a (head, 16
// sequences) pair fold the same partials.
// A sequence with an out-of-range length has no partials and keeps its out.
template <int DC>
struct MlaCombineSmem {
    static constexpr int AS = DC + 8;                     // row stride of o~ and of W rows, elements
    static constexpr int A = 16 * AS * 2;                 // o~ of 16 sequences
    static constexpr int W = 64 * AS * 2;                 // 64 rows of W_UV[h]
    static constexpr int WTS = 16 * MLA_MAX_CTAS * 4;     // split weights
    static constexpr int BYTES = A + W + WTS + 128;
};

template <typename T, int DC>
__global__ void __launch_bounds__(512) mla_combine_kernel(const MlaCombineArgs a) {
    using E = MlaElem<T>;
    using S = MlaCombineSmem<DC>;
    extern __shared__ __align__(16) uint8_t cmb[];
    T *os = reinterpret_cast<T *>(cmb);                               // [16][AS]
    T *wrows = reinterpret_cast<T *>(cmb + S::A);                      // [64][AS]
    float *wts = reinterpret_cast<float *>(cmb + S::A + S::W);        // [16][MLA_MAX_CTAS]
    int *s_c0 = reinterpret_cast<int *>(cmb + S::A + S::W + S::WTS);   // [16]
    int *s_c1 = s_c0 + 16;                                             // [16]
    const int h = blockIdx.x;
    const int b0 = blockIdx.y * 16;
    const int i0 = blockIdx.z * 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr unsigned FULL = 0xffffffffu;
    const int rows = min(64, a.d_h - i0);
    {
        // W_UV rows start towards shared memory before the dependency wait:
        // this launch follows the attention launch of the same call, which
        // signals its dependents only after its own wait for the absorb,
        // which had waited for everything before the call; W_UV is in place.
        const T *w = static_cast<const T *>(a.w_uv) + (int64_t(h) * a.d_h + i0) * DC;
        for (int v = threadIdx.x; v < rows * (DC / 8); v += 512) {
            const int r = v / (DC / 8), c = (v - r * (DC / 8)) * 8;
            dev::cp_async_16(dev::smem_addr(wrows + r * S::AS + c), w + int64_t(r) * DC + c);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    dev::grid_dependency_wait();   // the attention launch has completed: its partials are in place
    dev::allow_dependents();
    if (warp == 0) {
        // the decode launch's plan: flattened offsets of the sequences and the split length
        int64_t base = 0, mine = 0;
        int my_n = 0;
        for (int c0 = 0; c0 < a.B; c0 += 64) {   // two loads per lane in flight together
            int n2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int b = c0 + 32 * e + lane;
                const int v = b < a.B ? a.valid_len[b] : 0;
                n2[e] = (v >= 1 && v <= a.max_ctx) ? v : 0;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int n = n2[e], cb = c0 + 32 * e;
                int64_t incl = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int64_t y = __shfl_up_sync(FULL, incl, o);
                    if (lane >= o) incl += y;
                }
                for (int k = 0; k < 16; ++k) {
                    const int want = b0 + k;
                    if (want >= cb && want < cb + 32) {
                        const int src = want - cb;
                        const int64_t ex = base + __shfl_sync(FULL, incl - n, src);
                        const int nn = __shfl_sync(FULL, n, src);
                        if (lane == k) {
                            mine = ex;
                            my_n = nn;
                        }
                    }
                }
                base += __shfl_sync(FULL, incl, 31);
            }
        }
        const int64_t chunk = (base + a.grid - 1) / a.grid;
        if (lane < 16) {
            const bool live = my_n > 0 && b0 + lane < a.B;
            s_c0[lane] = live ? int(mine / chunk) : 0;
            s_c1[lane] = live ? int((mine + my_n - 1) / chunk) : -1;
        }
    }
    __syncthreads();
    {
        // warp k folds sequence b0 + k
        const int s16 = warp, b = b0 + s16, c0 = s_c0[s16], ns = s_c1[s16] - c0 + 1;
        T *orow = os + s16 * S::AS;
        if (b >= a.B || ns <= 0) {   // no live rows: a zero row (its output is not written)
            for (int c = lane * 8; c < DC; c += 256) *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0u, 0u, 0u, 0u);
        } else {
            const float *ml = a.part_ml + ((int64_t(c0) + b) * a.H + h) * 2;
            const int64_t ml_stride = int64_t(a.H) * 2;       // next slot
            float *wk_s = wts + s16 * MLA_MAX_CTAS;
            float M = -INFINITY, L = 0.f;
            for (int k0 = 0; k0 < ns; k0 += 32) {             // one pass for up to 32 splits
                const int k = k0 + lane;
                const float2 v = k < ns ? *reinterpret_cast<const float2 *>(ml + k * ml_stride) : make_float2(-INFINITY, 0.f);
                if (k < ns) wk_s[k] = v.x;                    // each split's running max, for now
                if (v.y > 0.f) M = fmaxf(M, v.x);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
            __syncwarp();
            for (int k0 = 0; k0 < ns; k0 += 32) {
                const int k = k0 + lane;
                if (k < ns) {
                    const float l = ml[k * ml_stride + 1];
                    const float wk = l > 0.f ? exp2f(wk_s[k] - M) : 0.f;
                    wk_s[k] = wk;
                    L += l * wk;
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(FULL, L, o);
            const float inv = 1.f / L;
            __syncwarp();
            const float *acc = a.part_acc + ((int64_t(c0) + b) * a.H + h) * DC + lane * 4;
            const int64_t acc_stride = int64_t(a.H) * DC;
            constexpr int R4 = DC / 128;      // float4 columns per lane
            constexpr int KB = 4;             // splits whose loads are in flight together
            float4 sum[R4];
#pragma unroll
            for (int r = 0; r < R4; ++r) sum[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k0 = 0; k0 < ns; k0 += KB) {
                float4 x[KB][R4];
                float wk[KB];
#pragma unroll
                for (int kk = 0; kk < KB; ++kk) {
                    const int k = k0 + kk;
                    wk[kk] = k < ns ? wk_s[k] : 0.f;
#pragma unroll
                    for (int r = 0; r < R4; ++r)
                        x[kk][r] = wk[kk] != 0.f ? __ldg(reinterpret_cast<const float4 *>(acc + k * acc_stride + r * 128))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int kk = 0; kk < KB; ++kk)
#pragma unroll
                    for (int r = 0; r < R4; ++r) {
                        sum[r].x = fmaf(wk[kk], x[kk][r].x, sum[r].x);
                        sum[r].y = fmaf(wk[kk], x[kk][r].y, sum[r].y);
                        sum[r].z = fmaf(wk[kk], x[kk][r].z, sum[r].z);
                        sum[r].w = fmaf(wk[kk], x[kk][r].w, sum[r].w);
                    }
            }
#pragma unroll
            for (int r = 0; r < R4; ++r) {
                T v4[4] = {E::store(sum[r].x * inv), E::store(sum[r].y * inv), E::store(sum[r].z * inv),
                           E::store(sum[r].w * inv)};
                *reinterpret_cast<uint2 *>(orow + r * 128 + lane * 4) = *reinterpret_cast<uint2 *>(v4);
            }
        }
    }
    cp_async_wait_all();
    __syncthreads();
    // out[b0 + m, h, i0 + 8 warp + n] for warps 0-7: A = o~ [16 x d_c], B = W rows [8 x d_c]
    if (warp < 8 && 8 * warp < rows) {
        const int l7 = lane & 7, j8 = lane >> 3;
        const uint32_t a_addr = dev::smem_addr(os + ((j8 & 1) * 8 + l7) * S::AS + (j8 >> 1) * 8);
        const uint32_t b_addr = dev::smem_addr(wrows + (8 * warp + l7) * S::AS + (j8 & 1) * 8 + (j8 >> 1) * 16);
        float c2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // two chains over k
#pragma unroll
        for (int ks = 0; ks < DC / 16; ks += 2) {
            uint32_t af[4], bf[4];
            dev::ldsm_x4(a_addr + ks * 32, af);
            dev::ldsm_x4(b_addr + ks * 32, bf);          // lanes 16-31 supply the next k-step
            E::mma(c2[0], af, bf[0], bf[1]);
            uint32_t af2[4];
            dev::ldsm_x4(a_addr + (ks + 1) * 32, af2);
            E::mma(c2[1], af2, bf[2], bf[3]);
        }
        T *out = static_cast<T *>(a.out);
        const int i = i0 + 8 * warp + 2 * (lane & 3);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int m = (lane >> 2) + 8 * hf, b = b0 + m;
            if (b < a.B && s_c1[m] >= s_c0[m]) {
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    if (i + e < i0 + rows)
                        out[(int64_t(b) * a.H + h) * a.d_h + i + e] = E::store(c2[0][2 * hf + e] + c2[1][2 * hf + e]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
struct MlaKernelInfo {
    int stage_bytes;
    int fixed_smem;       // besides the stages and their barriers
    int min_stages;
    cudaError_t (*set_max_smem)(int bytes);   // the decode kernel's, and the combine kernel's fixed size
    cudaError_t (*launch)(const MlaArgs &a, int grid, int smem, cudaStream_t s);
    cudaError_t (*absorb)(const MlaAbsorbArgs &a, cudaStream_t s);
    cudaError_t (*combine)(const MlaCombineArgs &a, cudaStream_t s);
};

template <typename T, int DC, int H>
const MlaKernelInfo *mla_info() {
    using C = MlaCfg<T, DC, H>;
    static const MlaKernelInfo info = {
        C::STAGE_BYTES + C::BARRIER_BYTES_PER_STAGE,
        C::FIXED_SMEM,
        2,
        [](int bytes) {
            cudaError_t e = cudaFuncSetAttribute(mla_combine_kernel<T, DC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 MlaCombineSmem<DC>::BYTES);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(mla_absorb_kernel<T, DC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     MlaAbsorbSmem<256>::BYTES);
            if (e != cudaSuccess) return e;
            return cudaFuncSetAttribute(mla_decode_kernel<T, DC, H>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        },
        [](const MlaArgs &a, int grid, int smem, cudaStream_t s) {
            return launch_pdl(mla_decode_kernel<T, DC, H>, dim3(grid), dim3(C::THREADS), smem, s, a);
        },
        [](const MlaAbsorbArgs &a, cudaStream_t s) {
            const dim3 grid(a.H, DC / 64, (a.B + 63) / 64);
            return launch_pdl(mla_absorb_kernel<T, DC>, grid, dim3(128), MlaAbsorbSmem<256>::BYTES, s, a);
        },
        [](const MlaCombineArgs &a, cudaStream_t s) {
            const dim3 grid(a.H, (a.B + 15) / 16, (a.d_h + 63) / 64);
            return launch_pdl(mla_combine_kernel<T, DC>, grid, dim3(512), MlaCombineSmem<DC>::BYTES, s, a);
        },
    };
    return &info;
}

// Tables, one per element type (kvc_mla_inst.cu): the kernel for (d_c, H),
// or null.
const MlaKernelInfo *mla_kernel_bf16(int d_c, int H);
const MlaKernelInfo *mla_kernel_f16(int d_c, int H);

}  // namespace kvc
