// kvc_decode_mma.cuh -- the decode attention of kvc_decode.cuh with the two
// contractions on the warp tensor-core path, for 16-bit caches and head
// groups of 2 to 8, 16, 32 and 64 (multi-query attention: "10.3", section
// 4.1, one KV head shared by every query head).
//
// Same mathematics, decomposition and pipeline protocol as
// decode_split_kernel ("10.3 -- KV cache implementation details", section 5,
// attention bullet; GQA per section 4.2).  With g query heads sharing a KV
// head, the tile of scores is a g x TILE product and P.V a g x d_h one.  On
// CUDA cores every cached element costs a widening instruction plus g/2
// packed FMAs per contraction, which at g >= 2 keeps the SM busy issuing
// arithmetic rather than streaming; the mma.sync m16n8k16 tile does the same
// work in a few instructions per 16 keys, with fp32 accumulation.
//
// Both products are taken transposed, so that the cached rows fill the M = 16
// side of the tile and the g query heads the N = 8 side (g <= 8, no padding to
// 16).  Per 32-key tile a consumer warp (lane = 4 * gq + tq):
//   S^T[32 x 8] = K[32 x D] . Q^T : A = K rows via ldmatrix (row-major
//     [key][d]), B = Q^T fragments (head gq, loaded once per piece); 2 m-tiles
//     x D/16 k-steps.  Lane (gq, tq) holds the scores of heads 2tq, 2tq+1 for
//     keys 16 mt + gq and 16 mt + gq + 8.
//   softmax per head over the keys: a head's column lives in the 8 lanes of
//     one tq, so the tile maximum takes three shuffles; the running sum stays
//     per lane until the end of the piece.  Scores are scaled by
//     log2(e)/sqrt(D) in fp32 after the product.
//   O^T[D x 8] += V^T . P^T : A = V^T via ldmatrix .trans on the same [key][d]
//     rows, B = P^T.  The S^T accumulator holds P^T with the keys along the
//     rows; one movmatrix.trans per 8x8 block turns it into the B-operand
//     layout (keys along the columns).  D/16 m-tiles x 2 k-steps.
// K and V tiles reach shared memory through TMA tensor copies with the
// 128-byte swizzle (16-byte chunk c of row r of each 64-column block stored at
// chunk c ^ (r mod 8)), which makes every ldmatrix conflict-free.  A box only
// ever covers 8-row groups inside the live range (32 rows for a full tile, 8
// for the groups of a tail tile); the last (rows mod 8) rows of a tail tile
// are loaded by the producer warp's other lanes with plain 16-byte loads and
// stored at their swizzled positions, so rows past valid_len are never read.
// Rows past the copied ones in a tail tile hold stale bytes: their scores are
// replaced by -inf and their V fragments are zeroed in registers.
//
// Merging is taken off the consumers: at the end of a piece each consumer
// warp leaves its softmax state in shared memory and goes on with the next
// piece; a merge warp combines the NW states, then writes the output or the
// split partial (and, for the last CTA of a segment, combines the partials)
// while the consumers keep the stage ring draining.
//
// Groups of 16, 32 or 64 query heads take the heads in chunks of 16, one
// chunk per consumer warp, as two N = 8 column tiles that share every K and
// V fragment the warp loads: the NW consumers form NW / NC streams of
// NC = G / 16 warps, the streams take the tiles round robin, and the NC
// warps of a stream all read the same tile, each for its own 16 heads (the
// tile's empty barrier completes after NC arrivals).  Every K/V byte is still
// read from HBM once for the whole group.  The merge warp combines the
// streams' states one 8-head chunk at a time.
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
    static constexpr int KSTEPS = D / 16;               // k-steps of S^T, m-tiles of O^T
    static constexpr int NW = 8;                        // consumer warps (+ producer + merger)
    // Warps: 0 issues the copies, 4 merges, 8 only takes part in the
    // set-up, the other eight compute.  A warp runs on scheduler (SMSP)
    // warp mod 4, so the copy-issuing warp shares its scheduler with no
    // consumer: consumers there delay its issue and, with it, the stream
    // (measured so for every group size, the compute-heavy 32-head group
    // included).
    static constexpr int PRODUCER_WARP = 0, MERGER_WARP = 4, IDLE_WARP = 8;
    static constexpr int THREADS = (NW + 3) * 32;
    static constexpr int ACTIVE_THREADS = (NW + 2) * 32;  // all but the idle warp
    // Groups of 16 or more heads: each consumer warp takes 16 heads (two
    // N = 8 column tiles, so every K and V fragment it loads serves both), and
    // the NC = G / 16 warps of a stream share each tile.
    static constexpr int NT = G >= 16 ? 2 : 1;          // 8-head column tiles per consumer warp
    static constexpr int GW = G >= 16 ? 16 : G;         // heads of one consumer warp
    static constexpr int NC = G >= 16 ? G / 16 : 1;     // warps sharing a tile
    static constexpr bool CHUNKED = G > 8;              // merged 8 heads at a time
    static constexpr int NSTREAM = NW / NC;             // streams of NC warps taking tiles round robin
    static constexpr int SCR_ACC_FLOATS = NSTREAM * G * D;
    static constexpr int SCR_ML_FLOATS = NSTREAM * G * 2;
    static constexpr int VL_CACHE = 256;                // valid lengths kept in shared memory
    static constexpr int N_FLAGS = 8;                   // abort flag, then the final-combine job
    // 1 KB of slack to align the stages to the 1024-byte swizzle atom, the two
    // merge barriers, the consumers' states, the flags, the valid lengths
    static constexpr int FIXED_SMEM =
        1024 + 16 + 4 * (SCR_ACC_FLOATS + SCR_ML_FLOATS) + 4 * N_FLAGS + 4 * VL_CACHE;
    // A final piece whose segment has more than this many other splits is
    // combined by every warp of the CTA instead of the merge warp alone.
    static constexpr int HELP_MIN_OTHERS = 4;

    static_assert(sizeof(T) == 2, "the tensor-core path takes 16-bit caches");
    static_assert(G >= 1 && (G <= 8 || (G % 16 == 0 && NW % NC == 0)),
                  "a group of more than 8 heads is taken in whole 16-head chunks, one per consumer warp");
    static_assert(D % 64 == 0, "head width must be a multiple of 64 (128-byte swizzle blocks)");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the swizzle-atom alignment");

    // Shared-memory address of (row r, element col) in a swizzled tile; col
    // is a multiple of 8 (one 16-byte chunk).
    __device__ __forceinline__ static uint32_t swz(uint32_t tile, int r, int col) {
        return tile + uint32_t(col >> 6) * BLOCK_BYTES + uint32_t(r) * 128 +
               uint32_t((((col >> 3) & 7) ^ (r & 7)) << 4);
    }
    // The same for a tile filled from a paged pool: rows of D elements kept
    // whole, i.e. 128-byte half-rows hr = r * (D / 64) + col / 64 in order, the
    // swizzle keyed on hr.  For D = 64 both layouts coincide.
    __device__ __forceinline__ static uint32_t swz_pg(uint32_t tile, int r, int col) {
        const uint32_t hr = uint32_t(r) * (D / 64) + uint32_t(col >> 6);
        return tile + hr * 128 + uint32_t((((col >> 3) & 7) ^ int(hr & 7)) << 4);
    }
};

// The producer warp: walks the CTA's pieces; for each tile one lane issues
// the TMA boxes and the other lanes load the tail rows no box may cover.  A
// full tile is one box of K and one of V (the 4-D map: all 64-column blocks);
// a tail tile takes one 8-row box per 64-column block.
template <typename C>
__device__ __forceinline__ uint32_t produce_tiles_tma(const DecodeArgs &a, Walker walk, uint32_t stage0,
                                                      uint32_t bar0, int ns, int64_t kv_slab,
                                                      volatile int *flags, int lane) {
    constexpr int TILE = C::TILE, CB = C::ROW_BYTES / 128;
    uint32_t issued = 0;
    int stage = 0;
    uint32_t round = 0;
    uint32_t generic_written = 0;  // stages whose last fill used cp.async
    bool ok = true;
    const uint64_t pol = dev::l2_evict_first_policy();  // K/V rows are read once per launch
    Piece pc;
    while (ok && walk.next(a, pc)) {
        const int seg = pc.b * a.H_kv + pc.kv;
        const int z = a.seg_base + seg;  // tensor-map segment coordinate
        const uint8_t *kseg = a.K + int64_t(seg) * kv_slab;
        const uint8_t *vseg = a.V + int64_t(seg) * kv_slab;
        // In a fused step the segment's last row is this step's new row: it
        // comes from k_new / v_new, never through a box over the stale cache.
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
            const uint32_t kdst = stage0 + uint32_t(stage) * C::STAGE_BYTES;
            const uint32_t vdst = kdst + C::TILE_BYTES;
            const int nb = (new_row >= row0 && new_row < row0 + nr) ? new_row - row0 : nr;  // rows boxes may cover
            const int q = nb >> 3, rem = nr - 8 * q;  // 8-row groups, rows after them
            if (lane == 0) {
                // the stage's previous rows came through the generic proxy:
                // order them before the TMA unit overwrites the stage
                if (generic_written & (1u << stage)) dev::fence_proxy_async_smem();
                dev::mbar_expect_tx(full, 2u * uint32_t(8 * q) * C::ROW_BYTES);
                if (q == 4) {
                    dev::tma_load_4d(kdst, &a.tm_k32, 0, row0, 0, z, full, pol);
                    dev::tma_load_4d(vdst, &a.tm_v32, 0, row0, 0, z, full, pol);
                } else {
                    for (int j = 0; j < q; ++j)
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb) {
                            const uint32_t off = cb * C::BLOCK_BYTES + j * 8 * 128;
                            dev::tma_load_3d(kdst + off, &a.tm_k8, cb * 64, row0 + 8 * j, z, full, pol);
                            dev::tma_load_3d(vdst + off, &a.tm_v8, cb * 64, row0 + 8 * j, z, full, pol);
                        }
                }
            }
            if (rem) {
                // rows no box may cover: 16-byte asynchronous copies, each
                // lane's completion counted on the stage's barrier
                const int per = rem * C::CHUNKS;  // 16-byte chunks per tensor
                for (int i = lane; i < 2 * per; i += 32) {
                    const bool is_v = i >= per;
                    const int j = is_v ? i - per : i;
                    const int r = 8 * q + j / C::CHUNKS, c16 = j % C::CHUNKS;
                    const uint8_t *src =
                        row0 + r == new_row
                            ? (is_v ? a.v_new : a.k_new) + int64_t(seg) * C::ROW_BYTES + c16 * 16
                            : (is_v ? vseg : kseg) + int64_t(row0 + r) * C::ROW_BYTES + c16 * 16;
                    dev::cp_async_16(C::swz(is_v ? vdst : kdst, r, c16 * 8), src);
                }
                dev::cp_async_arrive(full);
                generic_written |= 1u << stage;
            } else {
                generic_written &= ~(1u << stage);
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

// The producer for a paged cache: a tile of 32 rows starts on a block
// boundary (the split space is rounded to 16 rows per segment), so it is the
// first 16 rows of two logical blocks.  Their physical blocks come from the
// block table, 32 entries at a time (one per lane, shared by shuffles, the
// next 32 loaded ahead); a full block arrives as one box of K and one of V
// (the pool viewed as 128-byte half-rows), a partial one as an 8-row box and
// 16-byte cp.async copies.  A table entry
// outside [0, num_blocks) is recorded as a device-index error and its block
// is not copied.
template <typename C>
__device__ __forceinline__ uint32_t produce_tiles_paged(const DecodeArgs &a, Walker walk, uint32_t stage0,
                                                        uint32_t bar0, int ns, volatile int *flags, int lane) {
    constexpr int TILE = C::TILE, BS = 16;
    static_assert(TILE == 2 * BS, "a tile is two blocks");
    constexpr unsigned FULL = 0xffffffffu;
    const int64_t block_bytes = int64_t(BS) * C::ROW_BYTES;  // one KV head's rows of a block
    uint32_t issued = 0, generic_written = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    const uint64_t pol = dev::l2_evict_first_policy();  // K/V rows are read once per launch
    Piece pc;
    while (ok && walk.next(a, pc)) {
        const int32_t *trow = a.block_table + int64_t(pc.b) * a.max_blocks;
        const int new_row = a.k_new ? pc.n - 1 : -1;
        // Table entries in windows of 32 (lane l: logical block base + l), one
        // window ahead: tile t of the piece needs blocks first + 2t and
        // first + 2t + 1, both in window t / 16; window k + 1 is loaded when
        // window k comes into use, so its latency hides behind 16 tiles.
        const int first = pc.lo / BS;
        auto load_window = [&](int base) { return base + lane < a.max_blocks ? __ldg(trow + base + lane) : -1; };
        int32_t cached = load_window(first);
        int32_t ahead = load_window(first + 32);
        int cached_base = first;
        for (int row0 = pc.lo; row0 < pc.hi; row0 += TILE) {
            const int nr = min(TILE, pc.hi - row0);
            // the tile's blocks first: none of this needs the stage, so it
            // stays off the path from the stage's release to its refill
            const int blk0 = row0 / BS;
            if (blk0 >= cached_base + 32) {   // the next window: already loaded
                cached_base += 32;
                cached = ahead;
                ahead = load_window(cached_base + 32);
            }
            int phys[2], rows[2], boxed[2];
            uint32_t tx_rows = 0;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                phys[jj] = __shfl_sync(FULL, cached, blk0 + jj - cached_base);
                rows[jj] = max(0, min(BS, nr - BS * jj));
                const int first = row0 + BS * jj;
                const int nb = (new_row >= first && new_row < first + rows[jj]) ? new_row - first : rows[jj];
                boxed[jj] = nb == BS ? BS : (nb >= 8 ? 8 : 0);
                if (rows[jj] > 0 && (phys[jj] < 0 || phys[jj] >= a.num_blocks)) {
                    if (lane == 0) dev::record_error(a.err, ERR_DEVICE_INDEX);
                    rows[jj] = boxed[jj] = 0;  // not copied: its rows stay stale
                }
                tx_rows += uint32_t(boxed[jj]);
            }
            if (round > 0) {
                const bool w =
                    dev::mbar_wait_bounded(bar0 + 8 * (ns + stage), (round - 1) & 1, flags, a.timeout_ns);
                if (!__all_sync(FULL, w)) {
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
            if (generic_written & (1u << stage)) dev::fence_proxy_async_smem();  // every issuing lane
            if (lane == 0) dev::mbar_expect_tx(full, 2u * tx_rows * C::ROW_BYTES);
            __syncwarp();
            if (lane < 4) {
                // lanes 0-3: (block 0, K) (block 0, V) (block 1, K) (block 1, V),
                // all in one instruction.  One box covers the block's 16 (or
                // first 8) whole rows: the pool viewed as 128-byte half-rows.
                const int jj = lane >> 1;
                const bool is_v = lane & 1;
                const int bx = jj ? boxed[1] : boxed[0];
                if (bx) {
                    const int z = a.seg_base + (jj ? phys[1] : phys[0]) * a.H_kv + pc.kv;
                    const CUtensorMap *m = bx == BS ? (is_v ? &a.tm_v32 : &a.tm_k32) : (is_v ? &a.tm_v8 : &a.tm_k8);
                    dev::tma_load_3d((is_v ? vdst : kdst) + jj * BS * C::ROW_BYTES, m, 0, 0, z, full, pol);
                }
            }
            bool generic = false;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int rem = rows[jj] - boxed[jj];
                if (rem <= 0) continue;
                generic = true;
                const int64_t blk_off = (int64_t(phys[jj]) * a.H_kv + pc.kv) * block_bytes;
                const int per = rem * C::CHUNKS;
                for (int i = lane; i < 2 * per; i += 32) {
                    const bool is_v = i >= per;
                    const int j = is_v ? i - per : i;
                    const int r = boxed[jj] + j / C::CHUNKS, c16 = j % C::CHUNKS;  // row within the block
                    const int logical = row0 + BS * jj + r;
                    const uint8_t *src =
                        logical == new_row
                            ? (is_v ? a.v_new : a.k_new) + (int64_t(pc.b) * a.H_kv + pc.kv) * C::ROW_BYTES + c16 * 16
                            : (is_v ? a.V : a.K) + blk_off + int64_t(r) * C::ROW_BYTES + c16 * 16;
                    dev::cp_async_16(C::swz_pg(is_v ? vdst : kdst, BS * jj + r, c16 * 8), src);
                }
            }
            if (generic) {
                dev::cp_async_arrive(full);
                generic_written |= 1u << stage;
            } else {
                generic_written &= ~(1u << stage);
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

// The producer for a paged pool read two KV heads at a time.  One block of
// the pool holds the 16 rows of every KV head of a sequence, head after head
// ([H_kv, 16, D]), so the rows of KV heads 2j and 2j + 1 are one contiguous
// run of 2 x 16 rows: one box of each tensor brings both (8 KB at d_h = 128,
// the size of the contiguous cache's tile boxes), where one head per box
// takes twice the boxes for the same bytes.  A segment is (sequence, head
// pair) and a tile is one block: stage rows [16 z, 16 z + 16) hold head
// 2j + z, laid out [head][64-column block][16 rows][128 bytes] with the
// 128-byte swizzle (the 5-D box of the pair maps writes exactly that).  A
// partial last block is boxed in 8 rows per (head, column block) and
// finished with 16-byte cp.async copies; the new row of a fused step comes
// from k_new / v_new.  A table entry outside [0, num_blocks) is recorded as a
// device-index error and its block is not copied.  a.H_kv counts head pairs,
// a.seg_base is the layer's first block in the pools.
template <typename C>
__device__ __forceinline__ uint32_t produce_tiles_paged_pair(const DecodeArgs &a, Walker walk, uint32_t stage0,
                                                             uint32_t bar0, int ns, volatile int *flags,
                                                             int lane) {
    constexpr int BS = 16, CB = C::ROW_BYTES / 128;
    constexpr int HEAD_BYTES = BS * C::ROW_BYTES;  // one head's rows of a stage tile
    static_assert(C::TILE_BYTES == 2 * HEAD_BYTES, "a tile is one block of two heads");
    constexpr unsigned FULL = 0xffffffffu;
    const int H_all = 2 * a.H_kv;  // KV heads of the pool
    uint32_t issued = 0, generic_written = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    const uint64_t pol = dev::l2_evict_first_policy();  // K/V rows are read once per launch
    Piece pc;
    while (ok && walk.next(a, pc)) {
        const int32_t *trow = a.block_table + int64_t(pc.b) * a.max_blocks;
        const int new_row = a.k_new ? pc.n - 1 : -1;
        const int first = pc.lo / BS;
        // the tile's table entry, loaded one tile ahead (a warp-uniform load
        // from the table's cached lines) so that its latency hides behind
        // the previous tile's copies
        int phys_next = __ldg(trow + first);
        for (int row0 = pc.lo; row0 < pc.hi; row0 += BS) {
            const int nr = min(BS, pc.hi - row0);
            const int blk = row0 / BS;
            const int phys = phys_next;
            const int nb = (new_row >= row0 && new_row < row0 + nr) ? new_row - row0 : nr;
            int rows = nr;
            int boxed = nb == BS ? BS : (nb >= 8 ? 8 : 0);
            if (phys < 0 || phys >= a.num_blocks) {
                if (lane == 0) dev::record_error(a.err, ERR_DEVICE_INDEX);
                rows = boxed = 0;  // not copied: its rows stay stale
            }
            if (round > 0) {
                const bool w =
                    dev::mbar_wait_bounded(bar0 + 8 * (ns + stage), (round - 1) & 1, flags, a.timeout_ns);
                if (!__all_sync(FULL, w)) {
                    if (lane == 0) {
                        if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                        flags[0] = 1;
                    }
                    ok = false;
                    break;
                }
            }
            phys_next = blk + 1 < a.max_blocks ? __ldg(trow + blk + 1) : -1;
            const uint32_t full = bar0 + 8 * stage;
            const uint32_t kdst = stage0 + uint32_t(stage) * C::STAGE_BYTES;
            const uint32_t vdst = kdst + C::TILE_BYTES;
            if (generic_written & (1u << stage)) dev::fence_proxy_async_smem();  // every issuing lane
            if (lane == 0) dev::mbar_expect_tx(full, 4u * uint32_t(boxed) * C::ROW_BYTES);
            __syncwarp();
            const int wblk = a.seg_base + phys;
            if (boxed == BS) {
                // lane 0: K, lane 1: V, both heads in one box each
                if (lane < 2)
                    dev::tma_load_5d(lane ? vdst : kdst, lane ? &a.tm_v32 : &a.tm_k32, 0, 0, 0, 2 * pc.kv, wblk,
                                     full, pol);
            } else if (boxed == 8 && lane < 4 * CB) {
                // one 8-row box per (tensor, head, column block)
                const bool is_v = lane & 1;
                const int z = (lane >> 1) & 1, cb = lane >> 2;
                dev::tma_load_5d((is_v ? vdst : kdst) + z * HEAD_BYTES + cb * 2048, is_v ? &a.tm_v8 : &a.tm_k8, 0, 0,
                                 cb, 2 * pc.kv + z, wblk, full, pol);
            }
            const int rem = rows - boxed;
            if (rem > 0) {
                // rows no box covers: (tensor, head, row, 16-byte chunk) per lane
                const int per = rem * C::CHUNKS;
                for (int i = lane; i < 4 * per; i += 32) {
                    const bool is_v = i >= 2 * per;
                    const int j = is_v ? i - 2 * per : i;
                    const int z = j / per, jj = j - z * per;
                    const int r = boxed + jj / C::CHUNKS, c16 = jj % C::CHUNKS;
                    const int kvh = 2 * pc.kv + z;
                    const uint8_t *src =
                        row0 + r == new_row
                            ? (is_v ? a.v_new : a.k_new) + (int64_t(pc.b) * H_all + kvh) * C::ROW_BYTES + c16 * 16
                            : (is_v ? a.V : a.K) + ((int64_t(phys) * H_all + kvh) * BS + r) * C::ROW_BYTES + c16 * 16;
                    const uint32_t dst = (is_v ? vdst : kdst) + uint32_t(z * HEAD_BYTES + (c16 >> 3) * 2048 + r * 128) +
                                         (uint32_t((c16 & 7) ^ (r & 7)) << 4);
                    dev::cp_async_16(dst, src);
                }
                dev::cp_async_arrive(full);
                generic_written |= 1u << stage;
            } else {
                generic_written &= ~(1u << stage);
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

// Byte offset, inside a swizzled tile, of the 16-byte chunk that lane-row
// `row` (row mod 8 == lane mod 8) reads at column 16 * step + 8 * half, for
// step mod 4 == j: the chunk index (2 j + half) is XOR-ed with (row mod 8).
__device__ __forceinline__ uint32_t swz_lane_offset(int row, int half, int lane, int j) {
    return uint32_t(row) * 128 + ((uint32_t(2 * j) ^ uint32_t(half ^ (lane & 7))) << 4);
}

// A softmax state over a set of keys for G heads of one KV head, as the
// merge lanes hold it: lane l owns columns [l * D/32, (l + 1) * D/32).  The
// G heads are heads [h0, h0 + G) of a group of GS (the arrays below are laid
// out per GS heads); for groups of up to 8 heads GS = G and h0 = 0.
template <int D, int G, int GS = G>
struct LaneState {
    static constexpr int DPL = D / 32;
    float acc[G][DPL];  // unnormalised output
    float m[G];         // running maximum (log2 domain)
    float l[G];         // running sum

    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[h][i] = 0.f;
        }
    }

    // Combine the states of slots [0, n) of a shared-memory array laid out
    // [slot][G][D] (acc) and [slot][G][2] (max, sum) into this state, which
    // it replaces.
    __device__ __forceinline__ void reduce_slots(const float *sacc, const float *sml, int n, int lane,
                                                 int h0 = 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float M = -INFINITY;
            for (int w = 0; w < n; ++w) M = fmaxf(M, sml[(w * GS + h0 + h) * 2]);
            float L = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[h][i] = 0.f;
            for (int w = 0; w < n; ++w) {
                const float e = exp2f(sml[(w * GS + h0 + h) * 2] - M);
                L = fmaf(sml[(w * GS + h0 + h) * 2 + 1], e, L);
                const float *src = sacc + (w * GS + h0 + h) * D + lane * DPL;
                if constexpr (DPL == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    acc[h][0] = fmaf(v.x, e, acc[h][0]);
                    acc[h][1] = fmaf(v.y, e, acc[h][1]);
                    acc[h][2] = fmaf(v.z, e, acc[h][2]);
                    acc[h][3] = fmaf(v.w, e, acc[h][3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    acc[h][0] = fmaf(v.x, e, acc[h][0]);
                    acc[h][1] = fmaf(v.y, e, acc[h][1]);
                }
            }
            m[h] = M;
            l[h] = L;
        }
    }

    // Store this state as slot `slot` of such an array.
    __device__ __forceinline__ void store_slot(float *sacc, float *sml, int slot, int lane) const {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float *dst = sacc + (slot * G + h) * D + lane * DPL;
            if constexpr (DPL == 4)
                *reinterpret_cast<float4 *>(dst) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
            else
                *reinterpret_cast<float2 *>(dst) = make_float2(acc[h][0], acc[h][1]);
        }
        if (lane < G) {
            float mv = m[0], lv = l[0];
#pragma unroll
            for (int h = 1; h < G; ++h)
                if (lane == h) {
                    mv = m[h];
                    lv = l[h];
                }
            *reinterpret_cast<float2 *>(sml + (slot * G + lane) * 2) = make_float2(mv, lv);
        }
    }

    // Fold split partials c = first, first + step, ... <= last of segment
    // `seg` (all but `skip`) from the workspace into this state.  U partials'
    // loads are issued together.
    template <int U>
    __device__ __forceinline__ void fold_partials(const DecodeArgs &a, int seg, int first, int last, int step,
                                                  int skip, int lane, int h0 = 0) {
        for (int c = first; c <= last; c += U * step) {
            float pm[U][G], pl[U][G], pa[U][G][DPL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cu = c + u * step;
                const bool use = cu <= last && cu != skip;
                const int64_t sl = int64_t(cu + seg) * GS + h0;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    pm[u][h] = -INFINITY;
                    pl[u][h] = 0.f;
#pragma unroll
                    for (int i = 0; i < DPL; ++i) pa[u][h][i] = 0.f;
                    if (use) {
                        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.part_ml + (sl + h) * 2));
                        pm[u][h] = ml.x;
                        pl[u][h] = ml.y;
                        const float *src = a.part_acc + (sl + h) * D + lane * DPL;
                        if constexpr (DPL == 4) {
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                            pa[u][h][0] = v.x;
                            pa[u][h][1] = v.y;
                            pa[u][h][2] = v.z;
                            pa[u][h][3] = v.w;
                        } else {
                            const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                            pa[u][h][0] = v.x;
                            pa[u][h][1] = v.y;
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    if (pm[u][h] == -INFINITY) continue;  // no partial (every split has a finite max)
                    const float Mn = fmaxf(m[h], pm[u][h]);
                    const float so = exp2f(m[h] - Mn), sn = exp2f(pm[u][h] - Mn);
                    l[h] = fmaf(l[h], so, pl[u][h] * sn);
#pragma unroll
                    for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(acc[h][i], so, pa[u][h][i] * sn);
                    m[h] = Mn;
                }
        }
    }

    // Publish this state as the split partial of slot `slot`.
    __device__ __forceinline__ void store_partial(const DecodeArgs &a, int64_t slot, int lane, int h0 = 0) const {
        const int64_t sl = slot * GS + h0;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float *dst = a.part_acc + (sl + h) * D + lane * DPL;
            if constexpr (DPL == 4)
                *reinterpret_cast<float4 *>(dst) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
            else
                *reinterpret_cast<float2 *>(dst) = make_float2(acc[h][0], acc[h][1]);
        }
        if (lane < G) {
            float mv = m[0], lv = l[0];
#pragma unroll
            for (int h = 1; h < G; ++h)
                if (lane == h) {
                    mv = m[h];
                    lv = l[h];
                }
            *reinterpret_cast<float2 *>(a.part_ml + (sl + lane) * 2) = make_float2(mv, lv);
        }
    }

    // out[b, kv*G + h, :] = acc / l, rounded once.
    template <typename T>
    __device__ __forceinline__ void write_output(const DecodeArgs &a, int b, int kv, int lane, int h0 = 0) const {
        using Ops = ElemOps<T>;
        const int H = a.H_kv * GS;
        T *ob = reinterpret_cast<T *>(a.out) + (int64_t(b) * H + kv * GS + h0) * D + lane * DPL;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float inv = 1.f / l[h];
#pragma unroll
            for (int i = 0; i < DPL; ++i) ob[h * D + i] = Ops::round(acc[h][i] * inv);
        }
    }
};

// Partials the fold issues together: bounded by the registers they take.
template <int D, int G>
__host__ __device__ constexpr int fold_batch() {
    return (G * (D / 32 + 2)) <= 24 ? 4 : (G * (D / 32 + 2)) <= 36 ? 2 : 1;
}

// The combine that the final piece of a CTA still owes when its segment has
// many splits: done by every warp of the CTA after the stream has ended.
struct FinalCombine {
    int seg, c0, c1, me, b, kv;
};

// The merge warp: for each piece of the CTA, wait for the NW consumer states,
// combine them and free the states.  A piece that is a whole segment writes
// its output.  A split takes a ticket on the segment's counter first: every
// split but the last publishes its partial (data, fence, then its ready
// flag); the last one waits for the others' flags -- their CTAs are past their
// tickets, so the wait is short and needs no co-residency -- and folds their
// partials into its own state, then writes the output and resets the counter
// and the flags for the next launch.  When that last split is the CTA's final
// piece and the segment has more than HELP_MIN_OTHERS other splits, the fold
// is left to the whole CTA: the function returns true with the job in `job`
// and the CTA's own partial in `st`.  In a fused step it also stores the new
// 16-bit K and V rows into the cache (NEW_ROWS false: the caller's producer
// stores them itself, as the int8 cache's quantising producer does).
template <typename T, int D, int G, int NW, int KH = 1, bool NEW_ROWS = true>
__device__ __forceinline__ bool merge_pieces(const DecodeArgs &a, const Plan &plan, Walker walk,
                                             const float *scr_acc, const float *scr_ml, uint32_t scr_full,
                                             uint32_t scr_free, volatile int *flags, int lane,
                                             LaneState<D, G> &st, FinalCombine &job) {
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int HELP_MIN_OTHERS = MmaCfg<T, D, G>::HELP_MIN_OTHERS;
    uint32_t piece = 0;
    Piece pc;
    constexpr int ROW_BYTES = D * 2, CHUNKS = ROW_BYTES / 16;
    static_assert(2 * CHUNKS <= 32, "one 16-byte chunk of the new rows per lane");
    const int64_t kv_slab = int64_t(a.max_ctx) * ROW_BYTES;
    while (walk.next(a, pc)) {
        Walker peek = walk;
        Piece next_pc;
        const bool final_piece = !peek.next(a, next_pc);
        if (NEW_ROWS && a.k_new && pc.hi == pc.n && lane < 2 * CHUNKS) {
            // fused step: this CTA holds the segment's last row; store the
            // new K and V rows of its KH KV heads into the cache (nobody in
            // this launch reads them back from there)
            const bool is_v = lane >= CHUNKS;
            const int c16 = is_v ? lane - CHUNKS : lane;
            uint8_t *cache = const_cast<uint8_t *>(is_v ? a.V : a.K);  // the caller's writable cache
#pragma unroll
            for (int z = 0; z < KH; ++z) {
                const int kvh = pc.kv * KH + z;  // KV head
                const int64_t seg = int64_t(pc.b) * a.H_kv * KH + kvh;
                const uint4 v =
                    __ldg(reinterpret_cast<const uint4 *>((is_v ? a.v_new : a.k_new) + seg * ROW_BYTES) + c16);
                int64_t row_off = seg * kv_slab + int64_t(pc.n - 1) * ROW_BYTES;
                if (a.block_table) {  // paged: the row's slot in its physical block
                    const int p = pc.n - 1;
                    const int phys = __ldg(a.block_table + int64_t(pc.b) * a.max_blocks + p / 16);
                    row_off = phys >= 0 && phys < a.num_blocks
                                  ? ((int64_t(phys) * a.H_kv * KH + kvh) * 16 + p % 16) * ROW_BYTES
                                  : -1;  // reported by the producer
                }
                if (row_off >= 0) reinterpret_cast<uint4 *>(cache + row_off)[c16] = v;
            }
        }
        bool ok = !flags[0] && dev::mbar_wait_bounded(scr_full, piece & 1, flags, a.timeout_ns);
        ok = __all_sync(FULL, ok);
        if (!ok) {
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
            return false;
        }
        st.reduce_slots(scr_acc, scr_ml, NW, lane);
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(scr_free);
        ++piece;

        const int seg = pc.b * a.H_kv + pc.kv;
        const int c0 = int(pc.seg_start / plan.chunk);
        const int c1 = int((pc.seg_start + pc.len - 1) / plan.chunk);
        const int me = int(blockIdx.x);
        if (c0 != c1) {
            int ticket = 0;
            if (lane == 0) ticket = atomicAdd(a.tickets + seg, 1);
            ticket = __shfl_sync(FULL, ticket, 0);
            if (ticket < c1 - c0) {
                // not the last split: publish the partial
                st.store_partial(a, me + seg, lane);
                __threadfence();
                __syncwarp();
                if (lane == 0) dev::flag_store(a.ready + me + seg, 1);
                continue;
            }
            // the last split: wait for the others' partials
            bool pub = true;
            for (int c = c0 + lane; c <= c1; c += 32)
                if (c != me) pub = pub && dev::flag_wait_bounded(a.ready + c + seg, flags, a.flag_timeout_ns);
            pub = __all_sync(FULL, pub);
            if (!pub) {
                if (lane == 0) {
                    if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                    flags[0] = 1;
                }
                return false;
            }
            __threadfence();
            if (final_piece && c1 - c0 > HELP_MIN_OTHERS && !flags[0]) {
                job = FinalCombine{seg, c0, c1, me, pc.b, pc.kv};
                return true;
            }
            st.template fold_partials<fold_batch<D, G>()>(a, seg, c0, c1, 1, me, lane);
            for (int c = c0 + lane; c <= c1; c += 32)
                if (c != me) dev::flag_store(a.ready + c + seg, 0);
            if (lane == 0) a.tickets[seg] = 0;
        }
        st.template write_output<T>(a, pc.b, pc.kv, lane);
    }
    return false;
}

// The merge warp for groups of more than 8 heads: the same protocol as
// merge_pieces, with the streams' states combined one 8-head chunk at a time
// (a lane holds one chunk's state, as for an 8-head group).  The ticket is
// taken once per piece, before any chunk is published; a split publishes
// every chunk, then its ready flag; the last split waits for the others'
// flags, then folds their partials and writes the output chunk by chunk.
// The consumers' states are released once every chunk has been read.  The
// final combine is never handed to the whole CTA.
template <typename T, int D, int G, int NSLOT>
__device__ __forceinline__ void merge_pieces_chunked(const DecodeArgs &a, const Plan &plan, Walker walk,
                                                     const float *scr_acc, const float *scr_ml, uint32_t scr_full,
                                                     uint32_t scr_free, volatile int *flags, int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int NC = G / 8;
    constexpr int ROW_BYTES = D * 2, CHUNKS = ROW_BYTES / 16;
    static_assert(G % 8 == 0 && NC > 1, "for groups of whole 8-head chunks");
    static_assert(2 * CHUNKS <= 32, "one 16-byte chunk of the new rows per lane");
    const int64_t kv_slab = int64_t(a.max_ctx) * ROW_BYTES;
    LaneState<D, 8, G> st;
    uint32_t piece = 0;
    Piece pc;
    while (walk.next(a, pc)) {
        if (a.k_new && pc.hi == pc.n && lane < 2 * CHUNKS) {
            // fused step: store the new K and V rows into the cache (as merge_pieces)
            const int64_t seg = int64_t(pc.b) * a.H_kv + pc.kv;
            const bool is_v = lane >= CHUNKS;
            const int c16 = is_v ? lane - CHUNKS : lane;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.v_new : a.k_new) + seg * ROW_BYTES) + c16);
            uint8_t *cache = const_cast<uint8_t *>(is_v ? a.V : a.K);
            int64_t row_off = seg * kv_slab + int64_t(pc.n - 1) * ROW_BYTES;
            if (a.block_table) {
                const int p = pc.n - 1;
                const int phys = __ldg(a.block_table + int64_t(pc.b) * a.max_blocks + p / 16);
                row_off = phys >= 0 && phys < a.num_blocks
                              ? ((int64_t(phys) * a.H_kv + pc.kv) * 16 + p % 16) * ROW_BYTES
                              : -1;
            }
            if (row_off >= 0) reinterpret_cast<uint4 *>(cache + row_off)[c16] = v;
        }
        bool ok = !flags[0] && dev::mbar_wait_bounded(scr_full, piece & 1, flags, a.timeout_ns);
        ok = __all_sync(FULL, ok);
        if (!ok) {
            if (lane == 0) {
                if (!flags[0]) dev::record_error(a.err, ERR_TIMEOUT);
                flags[0] = 1;
            }
            return;
        }
        const int seg = pc.b * a.H_kv + pc.kv;
        const int c0 = int(pc.seg_start / plan.chunk);
        const int c1 = int((pc.seg_start + pc.len - 1) / plan.chunk);
        const int me = int(blockIdx.x);
        int mode = 0;  // 0: the piece is the whole segment, 1: publish a partial, 2: last split
        if (c0 != c1) {
            int ticket = 0;
            if (lane == 0) ticket = atomicAdd(a.tickets + seg, 1);
            ticket = __shfl_sync(FULL, ticket, 0);
            mode = ticket < c1 - c0 ? 1 : 2;
        }
        if (mode == 2) {
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
        }
#pragma unroll 1
        for (int hc = 0; hc < NC; ++hc) {
            st.reduce_slots(scr_acc, scr_ml, NSLOT, lane, 8 * hc);
            if (mode == 1) {
                st.store_partial(a, me + seg, lane, 8 * hc);
            } else {
                if (mode == 2) st.template fold_partials<fold_batch<D, 8>()>(a, seg, c0, c1, 1, me, lane, 8 * hc);
                st.template write_output<T>(a, pc.b, pc.kv, lane, 8 * hc);
            }
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(scr_free);
        ++piece;
        if (mode == 1) {
            __threadfence();
            __syncwarp();
            if (lane == 0) dev::flag_store(a.ready + me + seg, 1);
        } else if (mode == 2) {
            for (int c = c0 + lane; c <= c1; c += 32)
                if (c != me) dev::flag_store(a.ready + c + seg, 0);
            if (lane == 0) a.tickets[seg] = 0;
        }
    }
}

// PG: the tiles come from a paged pool in the half-row layout (MmaCfg::swz_pg);
// only the d_h = 128 kernels need it (for d_h = 64 the layouts coincide).
// PAIR: the tiles come from a paged pool two KV heads at a time
// (produce_tiles_paged_pair): a segment is (sequence, head pair), G counts
// the query heads of both KV heads (query head c belongs to KV head
// c / (G / 2)), a tile is 16 keys of each head, stage rows [16 z, 16 z + 16)
// hold head z; the products of one head's keys with the other head's
// queries are masked out of the softmax.
template <typename T, int D, int G, bool PG = false, bool PAIR = false>
__global__ void __launch_bounds__(MmaCfg<T, D, G>::THREADS, 1)
    decode_mma_kernel(const __grid_constant__ DecodeArgs a) {
    using C = MmaCfg<T, D, G>;
    constexpr bool PAGED_OK = PG || D == 64;         // the paged producer's layout is this kernel's
    constexpr bool PGL = PG && D != 64 && !PAIR;     // consumers address the half-row layout
    using Ops = MmaOps<T>;
    constexpr int NW = C::NW, TILE = C::TILE, KSTEPS = C::KSTEPS;
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(!PAIR || (G == 4 || G == 8), "head pairs of 2 or 4 query heads per KV head");
    constexpr int TK = PAIR ? 16 : TILE;  // keys of a segment per tile
    constexpr int KH = PAIR ? 2 : 1;      // KV heads per segment
    // tile addressing: the 16-row m-tile and the 64-column block strides
    constexpr uint32_t MT_STRIDE = PAIR ? 16u * C::ROW_BYTES : 2048u;
    constexpr uint32_t CB_STRIDE = PAIR ? 2048u : uint32_t(C::BLOCK_BYTES);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int ns = a.n_stages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t stage0 = dev::smem_addr(smem);
    const uint32_t bar0 = stage0 + uint32_t(ns) * C::STAGE_BYTES;  // full[ns], then empty[ns]
    const uint32_t scr_full = bar0 + 16 * uint32_t(ns);             // consumer states written
    const uint32_t scr_free = scr_full + 8;                         // consumer states read
    float *scr_acc = reinterpret_cast<float *>(smem + size_t(ns) * C::STAGE_BYTES + 16 * size_t(ns) + 16);
    float *scr_ml = scr_acc + C::SCR_ACC_FLOATS;
    // flags[0]: abort; flags[1]: final combine wanted; flags[2..7]: its job
    volatile int *flags = reinterpret_cast<volatile int *>(scr_ml + C::SCR_ML_FLOATS);
    int32_t *vl_cache = reinterpret_cast<int32_t *>(scr_ml + C::SCR_ML_FLOATS) + C::N_FLAGS;
    const int32_t *vl = a.B <= C::VL_CACHE ? vl_cache : a.valid_len;

    if (threadIdx.x == 0) {
        dev::prefetch_tensormap(&a.tm_k32);
        dev::prefetch_tensormap(&a.tm_v32);
        dev::prefetch_tensormap(&a.tm_k8);
        dev::prefetch_tensormap(&a.tm_v8);
        for (int s = 0; s < ns; ++s) {
            dev::mbar_init(bar0 + 8 * s, 1);
            dev::mbar_init(bar0 + 8 * (ns + s), C::NC);  // released by the NC warps of a stream
        }
        dev::mbar_init(scr_full, NW);
        dev::mbar_init(scr_free, 1);
        flags[0] = 0;
        dev::fence_mbar_init();
    }
    // everything above overlaps the previous kernel on the stream; nothing
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

    // ---------------------------------------------------------------- producer
    if (warp == C::PRODUCER_WARP) {
        uint32_t issued;
        if constexpr (PAIR)
            issued = produce_tiles_paged_pair<C>(a, walk, stage0, bar0, ns, flags, lane);
        else if constexpr (PAGED_OK)
            issued = a.block_table ? produce_tiles_paged<C>(a, walk, stage0, bar0, ns, flags, lane)
                                   : produce_tiles_tma<C>(a, walk, stage0, bar0, ns, kv_slab, flags, lane);
        else
            issued = produce_tiles_tma<C>(a, walk, stage0, bar0, ns, kv_slab, flags, lane);
        __syncwarp();
        dev::named_barrier_sync(2, C::ACTIVE_THREADS);  // every warp is done
        if (lane == 0 && flags[0]) drain_copies(bar0, ns, issued, a.timeout_ns);
        __syncwarp();
        return;
    }
    // The stage ring is idle once every consumer has handed over its final
    // state; the final combine keeps its per-warp states there.
    float *fin_acc = reinterpret_cast<float *>(smem);
    float *fin_ml = fin_acc + (NW + 1) * G * D;
    constexpr int FOLD_U = fold_batch<D, G>();
    constexpr int NC = C::NC, NSTREAM = C::NSTREAM, NT = C::NT;

    // ---------------------------------------------------------------- merger
    if constexpr (C::CHUNKED) {
        if (warp == C::MERGER_WARP) {
            merge_pieces_chunked<T, D, G, NSTREAM>(a, plan, walk, scr_acc, scr_ml, scr_full, scr_free, flags, lane);
            __syncwarp();
            dev::named_barrier_sync(2, C::ACTIVE_THREADS);
            return;
        }
    } else if (warp == C::MERGER_WARP) {
        LaneState<D, G> st;
        FinalCombine job;
        const bool help = merge_pieces<T, D, G, NW, KH>(a, plan, walk, scr_acc, scr_ml, scr_full, scr_free, flags,
                                                    lane, st, job);
        if (lane == 0) {
            flags[1] = help;
            flags[2] = job.seg;
            flags[3] = job.c0;
            flags[4] = job.c1;
            flags[5] = job.me;
        }
        __syncwarp();
        dev::named_barrier_sync(3, (NW + 1) * 32);  // consumers and merger
        if (help) {
            // the merger's share of the final combine starts from the CTA's own partial
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
    const int strm = cw / NC;  // this warp's stream: tiles strm, strm + NSTREAM, ...
    const int h0 = (cw % NC) * C::GW;  // first head of this warp's chunk (0 for groups up to 8)
    const int gq = lane >> 2;  // fragment row group: query head of B / C columns
    const int tq = lane & 3;   // quad lane
    const int H = a.H_kv * G;
    // ldmatrix lanes.  S^T operand A from K rows: matrices (keys 0-7, d 0-7)
    // (keys 8-15, d 0-7) (keys 0-7, d 8-15) (keys 8-15, d 8-15).  O^T operand
    // A from V rows with .trans: matrices (d 0-7, keys 0-7) (d 8-15, keys 0-7)
    // (d 0-7, keys 8-15) (d 8-15, keys 8-15).
    const int k_row = ((lane >> 3) & 1) * 8 + (lane & 7), k_half = (lane >> 4) & 1;
    const int v_row = ((lane >> 4) & 1) * 8 + (lane & 7), v_half = (lane >> 3) & 1;
    uint32_t koff[4], voff[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        koff[j] = swz_lane_offset(k_row, k_half, lane, j);
        voff[j] = swz_lane_offset(v_row, v_half, lane, j);
    }
    // the half-row layout of a paged tile: row r of the tile is D / 64
    // half-rows hr = r * D/64 + col / 64, the swizzle keyed on hr mod 8
    constexpr int CBK = PGL ? D / 64 : 1;
    uint32_t koffp[CBK][4], voffp[CBK][4];
    if constexpr (PGL) {
#pragma unroll
        for (int cb = 0; cb < CBK; ++cb)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                koffp[cb][j] = uint32_t(k_row * C::ROW_BYTES + cb * 128) +
                               (uint32_t((2 * j + k_half) ^ ((k_row * CBK + cb) & 7)) << 4);
                voffp[cb][j] = uint32_t(v_row * C::ROW_BYTES + cb * 128) +
                               (uint32_t((2 * j + v_half) ^ ((v_row * CBK + cb) & 7)) << 4);
            }
    }

    // Per 8-head column tile nt of this warp: Q^T fragments, O^T, and the
    // running max / sum of the lane's two heads h0 + 8 nt + 2 tq (+ 1).
    uint32_t qb[KSTEPS][NT][2];
    float o[KSTEPS][NT][4];
    float mx[NT][2], lx[NT][2];
    uint32_t t = 0, piece = 0;
    int stage = 0;
    uint32_t round = 0;
    Piece pc;
    while (walk.next(a, pc)) {
        {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hq = h0 + 8 * nt + gq;
                const T *qrow = reinterpret_cast<const T *>(a.q) + (int64_t(pc.b) * H + pc.kv * G + hq) * D;
                const bool qv = hq < G;
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    qb[ks][nt][0] = qv ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * tq)) : 0u;
                    qb[ks][nt][1] = qv ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + 2 * tq)) : 0u;
                }
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
                mx[nt][0] = mx[nt][1] = -INFINITY;
                lx[nt][0] = lx[nt][1] = 0.f;
            }
        }

        for (int row0 = pc.lo; row0 < pc.hi; row0 += TK, ++t) {
            const int cur_stage = stage;
            const uint32_t cur_round = round;
            if (++stage == ns) {
                stage = 0;
                ++round;
            }
            if (int(t % NSTREAM) != strm) continue;
            const int nr = min(TK, pc.hi - row0);
            // Wait for the previous release of this stage first, then for its
            // data: the reasoning is the one in decode_split_kernel, with a
            // stream's NC warps in place of one warp (tile t - ns needs all of
            // its stream's arrivals; t can only be released with this warp's).
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

            // ---- S^T = K . Q^T for 32 keys (2 m-tiles of 16), NT column tiles
            float s[2][NT][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) s[mt][nt][0] = s[mt][nt][1] = s[mt][nt][2] = s[mt][nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t r[4];
                    if constexpr (PGL)
                        dev::ldsm_x4(ks_base + mt * 16 * C::ROW_BYTES + koffp[ks >> 2][ks & 3], r);
                    else
                        dev::ldsm_x4(ks_base + (ks >> 2) * CB_STRIDE + mt * MT_STRIDE + koff[ks & 3], r);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) Ops::mma(s[mt][nt], r, qb[ks][nt][0], qb[ks][nt][1]);
                }
            }

            // ---- online softmax per head column (keys along the rows)
            if (nr < TK) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int k = (PAIR ? 0 : 16 * mt) + gq;  // key of the rows gq, gq + 8
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (k >= nr) s[mt][nt][0] = s[mt][nt][1] = -INFINITY;
                        if (k + 8 >= nr) s[mt][nt][2] = s[mt][nt][3] = -INFINITY;
                    }
                }
            }
            if constexpr (PAIR) {
                // m-tile z holds KV head z's keys: only its own query heads
                // (columns [z G/2, (z + 1) G/2)) see them; padding columns
                // past G keep their zero products
                const int cz = (2 * tq) / (G / 2);  // KV head of this lane's two columns
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
                    if (cz < 2 && cz != mt) s[mt][0][0] = s[mt][0][1] = s[mt][0][2] = s[mt][0][3] = -INFINITY;
            }
            float corr[NT][2];
            float p[2][NT][4];
            bool any_corr = false;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float x0 = fmaxf(fmaxf(s[0][nt][0], s[0][nt][2]), fmaxf(s[1][nt][0], s[1][nt][2]));
                float x1 = fmaxf(fmaxf(s[0][nt][1], s[0][nt][3]), fmaxf(s[1][nt][1], s[1][nt][3]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, off));
                    x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, off));
                }
                const float mn0 = fmaxf(mx[nt][0], x0 * a.scale_log2), mn1 = fmaxf(mx[nt][1], x1 * a.scale_log2);
                corr[nt][0] = exp2f(mx[nt][0] - mn0);
                corr[nt][1] = exp2f(mx[nt][1] - mn1);
                mx[nt][0] = mn0;
                mx[nt][1] = mn1;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    p[mt][nt][0] = exp2f(fmaf(s[mt][nt][0], a.scale_log2, -mn0));
                    p[mt][nt][1] = exp2f(fmaf(s[mt][nt][1], a.scale_log2, -mn1));
                    p[mt][nt][2] = exp2f(fmaf(s[mt][nt][2], a.scale_log2, -mn0));
                    p[mt][nt][3] = exp2f(fmaf(s[mt][nt][3], a.scale_log2, -mn1));
                }
                lx[nt][0] = fmaf(lx[nt][0], corr[nt][0], (p[0][nt][0] + p[0][nt][2]) + (p[1][nt][0] + p[1][nt][2]));
                lx[nt][1] = fmaf(lx[nt][1], corr[nt][1], (p[0][nt][1] + p[0][nt][3]) + (p[1][nt][1] + p[1][nt][3]));
                any_corr = any_corr || (corr[nt][0] != 1.f) || (corr[nt][1] != 1.f);
            }
            if (__any_sync(FULL, any_corr)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float2 cc = make_float2(corr[nt][0], corr[nt][1]);
#pragma unroll
                    for (int mt = 0; mt < KSTEPS; ++mt) {
                        const float2 lo = __fmul2_rn(make_float2(o[mt][nt][0], o[mt][nt][1]), cc);
                        const float2 hi = __fmul2_rn(make_float2(o[mt][nt][2], o[mt][nt][3]), cc);
                        o[mt][nt][0] = lo.x;
                        o[mt][nt][1] = lo.y;
                        o[mt][nt][2] = hi.x;
                        o[mt][nt][3] = hi.y;
                    }
                }
            }
            // P^T blocks (keys x heads) -> B fragments (keys along k)
            uint32_t pb[2][NT][2];
#pragma unroll
            for (int kst = 0; kst < 2; ++kst)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    pb[kst][nt][0] = dev::movmatrix_trans(Ops::pack(p[kst][nt][0], p[kst][nt][1]));
                    pb[kst][nt][1] = dev::movmatrix_trans(Ops::pack(p[kst][nt][2], p[kst][nt][3]));
                }

            // ---- O^T += V^T . P^T over the tile's two 16-key steps
#pragma unroll
            for (int kst = 0; kst < 2; ++kst) {
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    uint32_t r[4];
                    if constexpr (PGL)
                        dev::ldsm_x4_trans(vs_base + kst * 16 * C::ROW_BYTES + voffp[mt >> 2][mt & 3], r);
                    else
                        dev::ldsm_x4_trans(vs_base + (mt >> 2) * CB_STRIDE + kst * MT_STRIDE + voff[mt & 3], r);
                    if (nr < TK) {  // stale rows past the copied ones
                        const int k0 = (PAIR ? 0 : kst * 16) + 2 * tq;
                        r[0] = live_pair(r[0], k0, nr);
                        r[1] = live_pair(r[1], k0, nr);
                        r[2] = live_pair(r[2], k0 + 8, nr);
                        r[3] = live_pair(r[3], k0 + 8, nr);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) Ops::mma(o[mt][nt], r, pb[kst][nt][0], pb[kst][nt][1]);
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(empty_bar);
        }

        // ---- end of piece: hand this warp's state to the merge warp
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                lx[nt][0] += __shfl_xor_sync(FULL, lx[nt][0], off);
                lx[nt][1] += __shfl_xor_sync(FULL, lx[nt][1], off);
            }
        bool ok = !flags[0] &&
                  (piece == 0 || dev::mbar_wait_bounded(scr_free, (piece - 1) & 1, flags, a.timeout_ns));
        ok = __all_sync(FULL, ok);
        if (ok) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int ha = h0 + 8 * nt + 2 * tq, hb = ha + 1;  // heads of this lane's two columns
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    const int d = 16 * mt + gq;
                    if (ha < G) {
                        scr_acc[(strm * G + ha) * D + d] = o[mt][nt][0];
                        scr_acc[(strm * G + ha) * D + d + 8] = o[mt][nt][2];
                    }
                    if (hb < G) {
                        scr_acc[(strm * G + hb) * D + d] = o[mt][nt][1];
                        scr_acc[(strm * G + hb) * D + d + 8] = o[mt][nt][3];
                    }
                }
                if (gq == 0) {
                    if (ha < G) {
                        scr_ml[(strm * G + ha) * 2] = mx[nt][0];
                        scr_ml[(strm * G + ha) * 2 + 1] = lx[nt][0];
                    }
                    if (hb < G) {
                        scr_ml[(strm * G + hb) * 2] = mx[nt][1];
                        scr_ml[(strm * G + hb) * 2 + 1] = lx[nt][1];
                    }
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

    // ---- the final combine, when the merger asks for it (groups up to 8 heads)
    if constexpr (!C::CHUNKED) {
        dev::named_barrier_sync(3, (NW + 1) * 32);
        if (flags[1]) {
            const int seg = flags[2], c0 = flags[3], c1 = flags[4], me = flags[5];
            LaneState<D, G> st;
            st.clear();
            st.template fold_partials<FOLD_U>(a, seg, c0 + cw, c1, NW + 1, me, lane);
            st.store_slot(fin_acc, fin_ml, cw, lane);
            dev::named_barrier_sync(3, (NW + 1) * 32);
        }
    }
    dev::named_barrier_sync(2, C::ACTIVE_THREADS);
}

template <typename T, int D, int G, bool PG, bool PAIR>
cudaError_t set_mma_max_smem(int bytes) {
    return cudaFuncSetAttribute(decode_mma_kernel<T, D, G, PG, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                bytes);
}

template <typename T, int D, int G, bool PG, bool PAIR>
cudaError_t launch_mma(const DecodeArgs &a, int grid, int smem, cudaStream_t s) {
    return launch_pdl(decode_mma_kernel<T, D, G, PG, PAIR>, dim3(grid), dim3(MmaCfg<T, D, G>::THREADS), smem, s, a);
}

// PG: the kernel for paged pools with d_h = 128 (the half-row tile layout).
// PAIR: the kernel for paged pools read two KV heads per tile (G counts the
// query heads of both); a tile is 16 keys of each head.
template <typename T, int D, int G, bool PG = false, bool PAIR = false>
const DecodeKernelInfo *mma_decode_info() {
    using C = MmaCfg<T, D, G>;
    static const DecodeKernelInfo info = {PAIR ? 16 : C::TILE, C::NW, C::STAGE_BYTES + 16, C::FIXED_SMEM,
                                          &set_mma_max_smem<T, D, G, PG, PAIR>, &launch_mma<T, D, G, PG, PAIR>,
                                          true, true, false, PAIR ? 16 : C::TILE};
    return &info;
}

}  // namespace kvc
