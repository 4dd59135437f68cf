// Tile-packed CSF on sm_103a: the same per-row bases and codes as a CSF stack,
// stored in the order of the block-scaled GEMM scale tiles so that every
// 128 x 4 tile decodes on its own (stage-readable storage), plus the
// conversion from a CSF stack and the decode into the tiled scale layout.
//
// Pages followed (cited by title and paragraph; they have no numbered
// sections):
//   "NVFP4-CSF: expand_scales() for ahead-of-call scale expansion (canonical
//     twin of #477)": commit message on packed experts prepared from CSF
//     checkpoints that keep their scales as stage-readable compressed
//     storage, which each pipeline stage rebuilds in shared memory (no record
//     layout given: the layout below is this library's).
//   "finegrained-kernels: decode losslessly compressed NVFP4 scales (CSF)":
//     format paragraph (base byte per row, 4-bit offsets, exception stream).
//
// Layout (per expert: nrb = ceil(R/128) row blocks, ncb = ceil(C/4) column
// blocks, T = nrb*ncb tiles, tile t = rb*ncb + cb; global tile = e*T + t):
//   codes   NVFP4 256 bytes a tile, MXFP4 128 (offset plane, then escape
//           plane, 64 bytes each); position q = 16*b + 4*a + c of a tile is
//           row 128*rb + b + 32*a, column 4*cb + c; padding positions code 0.
//   bases   128 bytes a row block, byte 4*b + a = base of row b + 32*a.
//   tile_index  E*T + 1 u32, exclusive prefix of the tiles' exception counts.
//   exc_bytes   each tile's exceptions in position order.
// Lane b of a warp owns line b of a tile (positions 16b .. 16b+15): 8 code
// bytes (NVFP4) and 4 base bytes, exactly the 16 bytes of line b of the tile
// in the block-scaled layout, which sits at byte 512*(global tile) + 16*b.
#include "csf_device.cuh"
#include "csf_internal.cuh"
#include "csf_tile.cuh"

namespace csfk {
namespace {

using dev::flag;
using dev::kFull;
using dev::lanemask_lt;

constexpr int kTlWarps = 4;
constexpr int kTlThreads = 32 * kTlWarps;

__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, int lane, uint32_t &total) {
    uint32_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, d);
        if (lane >= d) x += y;
    }
    total = __shfl_sync(kFull, x, 31);
    return x - v;
}

// Bits [pos, pos + 64) of an LSB-first packed plane of `bytes` bytes (8-byte
// aligned, `bytes` a multiple of 8); words past the end read as 0.
__device__ __forceinline__ uint64_t plane_bits(const uint8_t *plane, uint64_t pos, uint64_t bytes) {
    const uint64_t w = pos >> 6;
    const uint32_t sh = (uint32_t)pos & 63u;
    const unsigned long long *p = reinterpret_cast<const unsigned long long *>(plane);
    const uint64_t a = (w + 1) * 8 <= bytes ? __ldg(p + w) : 0ull;
    const uint64_t b = (sh != 0 && (w + 2) * 8 <= bytes) ? __ldg(p + w + 1) : 0ull;
    return sh ? (a >> sh) | (b << (64 - sh)) : a;
}

struct Geo {
    uint32_t R, C, nrb, ncb, T;
};

__device__ __forceinline__ Geo geo_of(const DecStack &S) {
    Geo g;
    g.R = (uint32_t)S.R;
    g.C = (uint32_t)S.C;
    g.nrb = (g.R + kTileRows - 1) / kTileRows;
    g.ncb = (g.C + 3) / 4;
    g.T = g.nrb * g.ncb;
    return g;
}

// ------------------------------------------------------------------ pack

// The CSF codes of columns [4cb, 4cb+4) of one row: NVFP4 four nibbles in
// bits 0..15 and their escape flags in bits 16..19; MXFP4 four offset bits
// in bits 0..3 and four escape bits in 16..19.  Columns past C read 0.
template <int KIND>
__device__ __forceinline__ uint32_t csf_cols4(const DecStack &S, uint64_t row, uint32_t cb, uint32_t C) {
    const uint64_t el = row * C + 4u * cb;
    const uint32_t cv = min(4u, C - 4u * cb);
    if (KIND == CSF_NVFP4) {
        uint32_t n = (uint32_t)plane_bits(S.offsets, 4 * el, S.off_bytes) & 0xFFFFu;
        n &= cv >= 4 ? 0xFFFFu : (1u << (4 * cv)) - 1;
        const uint32_t f = n & (n >> 1) & (n >> 2) & (n >> 3) & 0x1111u;      // nibble == 15 -> bit 4j
        const uint32_t e4 = (f & 1u) | ((f >> 3) & 2u) | ((f >> 6) & 4u) | ((f >> 9) & 8u);
        return n | (e4 << 16);
    }
    const uint32_t m = cv >= 4 ? 0xFu : (1u << cv) - 1;
    const uint32_t o4 = (uint32_t)plane_bits(S.offsets, el, S.off_bytes) & m;
    const uint32_t x4 = (uint32_t)plane_bits(S.escapes, el, S.off_bytes) & m;
    return o4 | (x4 << 16);
}

// One warp per (expert, row block), walking its column tiles in order.  A
// row block is a run of consecutive rows, so its exceptions fill the same
// range of the tile-ordered stream as of the row-major CSF stream, starting
// at the CSF index of its first row; within it the tiles follow one another
// (a running sum over the walk), so no scan pass is needed.
template <int KIND>
__global__ void __launch_bounds__(kTlThreads) tiled_pack_kernel(const __grid_constant__ DecStack S,
                                                                 const __grid_constant__ TiledOut O) {
    const int lane = threadIdx.x & 31;
    const Geo g = geo_of(S);
    const uint64_t items = (uint64_t)S.rows / g.R * g.nrb;                 // E * nrb
    const uint64_t nw = (uint64_t)gridDim.x * kTlWarps;
    const uint32_t nexc = (uint32_t)S.num_exc;
    if (blockIdx.x == 0 && threadIdx.x == 0) O.tile_index[items * g.ncb] = __ldg(S.exc_index + S.rows);
    for (uint64_t it = (uint64_t)blockIdx.x * kTlWarps + (threadIdx.x >> 5); it < items; it += nw) {
        const uint64_t e = it / g.nrb;
        const uint32_t rb = (uint32_t)(it - e * g.nrb);
        uint64_t row[4];
        bool ok[4];
        uint32_t X[4] = {0, 0, 0, 0};
        uint32_t bw = 0;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const uint32_t rl = rb * kTileRows + (uint32_t)lane + 32u * a;
            ok[a] = rl < g.R;
            row[a] = e * g.R + rl;
            if (ok[a]) {
                X[a] = __ldg(S.exc_index + row[a]);
                bw |= (uint32_t)__ldg(S.base + row[a]) << (8 * a);
            }
        }
        reinterpret_cast<uint32_t *>(O.bases)[it * 32 + lane] = bw;
        uint32_t run = __shfl_sync(kFull, X[0], 0);                          // index of the block's first row
        bool bad = false;
        for (uint32_t cb = 0; cb < g.ncb; ++cb) {
            const uint64_t tile = it * g.ncb + cb;
            uint32_t v[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) v[a] = ok[a] ? csf_cols4<KIND>(S, row[a], cb, g.C) : 0u;
            uint32_t cnt = 0;
#pragma unroll
            for (int a = 0; a < 4; ++a) cnt += __popc(v[a] >> 16);
            uint32_t tot;
            const uint32_t pre = warp_excl_scan(cnt, lane, tot);
            if (lane == 0) O.tile_index[tile] = run;
            if (KIND == CSF_NVFP4) {
                const uint64_t code = (uint64_t)(v[0] & 0xFFFFu) | ((uint64_t)(v[1] & 0xFFFFu) << 16) |
                                      ((uint64_t)(v[2] & 0xFFFFu) << 32) | ((uint64_t)(v[3] & 0xFFFFu) << 48);
                reinterpret_cast<unsigned long long *>(O.codes + tile * 256)[lane] = code;
            } else {
                const uint32_t ob = (v[0] & 0xFu) | ((v[1] & 0xFu) << 4) | ((v[2] & 0xFu) << 8) |
                                    ((v[3] & 0xFu) << 12);
                const uint32_t xb = ((v[0] >> 16) & 0xFu) | (((v[1] >> 16) & 0xFu) << 4) |
                                    (((v[2] >> 16) & 0xFu) << 8) | (((v[3] >> 16) & 0xFu) << 12);
                reinterpret_cast<uint16_t *>(O.codes + tile * 128)[lane] = (uint16_t)ob;
                reinterpret_cast<uint16_t *>(O.codes + tile * 128 + 64)[lane] = (uint16_t)xb;
            }
            // Exceptions in position order: row a, then column; the CSF byte of
            // a row's k-th exception in this tile is at X[a] + k.
            uint64_t dst = (uint64_t)run + pre;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                uint32_t f = v[a] >> 16;
                while (f) {
                    uint32_t byte = 0;
                    if (X[a] < nexc) byte = __ldg(S.exc_bytes + X[a]);
                    else bad = true;
                    if (dst < O.exc_capacity) O.exc_bytes[dst] = (uint8_t)byte;
                    else flag(O.err, CSF_DEV_ERR_CAPACITY);
                    ++X[a];
                    ++dst;
                    f &= f - 1;
                }
            }
            run += tot;
        }
        // every row's exceptions accounted for: the index and the codes agree
#pragma unroll
        for (int a = 0; a < 4; ++a)
            if (ok[a] && X[a] != __ldg(S.exc_index + row[a] + 1)) bad = true;
        if (__any_sync(kFull, bad) && lane == 0) flag(S.err, CSF_DEV_ERR_CORRUPT);
    }
}

// ---------------------------------------------------------------- decode
//
// The per-tile decode is the public device API of include/csf_tile.cuh
// (csf_tile_load, csf_tile_expand, csf_tile_patch, csf_tile_mask_edge), so
// this kernel and any consumer kernel that rebuilds tiles in shared memory
// run the same code.

__device__ __forceinline__ csf_tile_src tile_src(const DecStack &S, const TiledIn &I) {
    csf_tile_src s;
    s.codes = I.codes;
    s.bases = I.bases;
    s.tile_index = I.tile_index;
    s.exc_bytes = I.exc_bytes;
    s.num_exc = (uint32_t)I.num_exc;
    s.kind = S.kind;
    s.R = S.R;
    s.C = S.C;
    return s;
}

// One tile from its raw inputs, whole warp.  `line` is the lane's own
// 16-byte shared-memory slot, where lanes with exceptions patch them byte by
// byte; `edge` says that the tile holds padding (rows past R or columns past
// C), which is written as 0.  STAGE = false: lane b writes line b (16 bytes)
// at dst + 16*b.  STAGE = true: the warp's 32 slots hold the rebuilt tile (512
// bytes, block-scaled order) in shared memory, as a pipeline stage would
// consume it, and lane 0 writes the tile's checksum to *sum (the sum of its
// 128 little-endian words w_i times 2i + 1, mod 2^32).  Returns true when the
// tile's index disagrees with its codes.
template <int KIND, bool STAGE>
__device__ __forceinline__ bool tile_finish(const csf_tile_src &src, uint32_t rb, uint32_t cb, bool edge,
                                            const csf_tile_line &L, const csf_tile_raw &r, uint8_t *dst,
                                            uint32_t *sum, uint4 *line, int lane) {
    uint32_t w0 = L.w0, w1 = L.w1, w2 = L.w2, w3 = L.w3;
    if (STAGE || L.cnt) *line = make_uint4(w0, w1, w2, w3);
    const bool bad = csf_tile_patch<KIND>(src, r, L, reinterpret_cast<uint8_t *>(line), lane);
    if (L.cnt) {
        const uint4 q = *line;
        w0 = q.x; w1 = q.y; w2 = q.z; w3 = q.w;
    }
    if (edge) csf_tile_mask_edge(src, rb, cb, lane, w0, w1, w2, w3);
    if (STAGE) {
        if (edge) *line = make_uint4(w0, w1, w2, w3);
        __syncwarp();   // the whole tile is in shared memory
        const uint32_t k = 8u * (uint32_t)lane + 1u;   // 2 * (4 lane) + 1
        const uint32_t part = w0 * k + w1 * (k + 2u) + w2 * (k + 4u) + w3 * (k + 6u);
        const uint32_t tsum = __reduce_add_sync(kFull, part);
        if (lane == 0) *sum = tsum;
        __syncwarp();   // the slots may be reused for the next tile
    } else {
        *reinterpret_cast<uint4 *>(dst + 16u * (uint32_t)lane) = make_uint4(w0, w1, w2, w3);
    }
    return bad;
}

// The experts to decode, compacted into `act` in shared memory with ballots
// (whole block; routing read on the device).  Returns how many; without
// routing every expert, and `act` is not used.
__device__ uint32_t active_experts(const TiledIn &I, uint32_t E, uint32_t *act, uint32_t *s_cnt) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (I.expert_start == nullptr) return E;
    uint32_t n_act = 0;
    for (uint32_t e0 = 0; e0 < E; e0 += kTlThreads) {
        const uint32_t e = e0 + threadIdx.x;
        bool a = false;
        if (e < E) {
            if (I.es64) {
                const long long *st = static_cast<const long long *>(I.expert_start);
                a = __ldg(st + e + 1) > __ldg(st + e);
            } else {
                const int *st = static_cast<const int *>(I.expert_start);
                a = __ldg(st + e + 1) > __ldg(st + e);
            }
        }
        const uint32_t bal = __ballot_sync(kFull, a);
        if (lane == 0) s_cnt[warp] = __popc(bal);
        __syncthreads();
        uint32_t bn = n_act, tn = 0;
#pragma unroll
        for (int w = 0; w < kTlWarps; ++w) {
            if (w < warp) bn += s_cnt[w];
            tn += s_cnt[w];
        }
        if (a) act[bn + __popc(bal & lanemask_lt())] = e;
        n_act += tn;
        __syncthreads();
    }
    return n_act;
}

// Decode (STAGE = false: into the block-scaled workspace S.ws) or stage-read
// (STAGE = true: each tile rebuilt in shared memory, one checksum per tile
// written to sums[e * T + t]) the tiles of the selected experts.
template <int KIND, bool STAGE>
__global__ void __launch_bounds__(kTlThreads) tiled_decode_kernel(const __grid_constant__ DecStack S,
                                                                   const __grid_constant__ TiledIn I,
                                                                   uint32_t *sums) {
    extern __shared__ __align__(16) uint32_t act[];
    __shared__ uint32_t s_cnt[kTlWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const Geo g = geo_of(S);
    const uint32_t n_act = active_experts(I, (uint32_t)(S.rows / g.R), act, s_cnt);
    const uint64_t total = (uint64_t)n_act * g.T;
    const uint64_t nw = (uint64_t)gridDim.x * kTlWarps;
    const uint64_t w = (uint64_t)blockIdx.x * kTlWarps + warp;
    // A contiguous range of tiles per warp, walked with running counters
    // (active expert j, tile t = rb*ncb + cb, global tile and row block); the
    // next tile's inputs are fetched while the current one is expanded.
    __shared__ uint4 s_line[kTlWarps][32];
    uint4 *line = &s_line[warp][lane];
    const uint32_t full_rb = g.R / kTileRows, full_cb = g.C / 4;  // row / column blocks without padding
    const csf_tile_src src = tile_src(S, I);
    bool bad = false;
    const uint64_t it0 = total * w / nw;
    uint32_t n = (uint32_t)(total * (w + 1) / nw - it0);
    uint32_t j = (uint32_t)(it0 / g.T);
    uint32_t t = (uint32_t)(it0 - (uint64_t)j * g.T);
    uint32_t rb = t / g.ncb, cb = t - rb * g.ncb;
    uint64_t e = I.expert_start != nullptr && n ? act[j] : j;
    uint64_t tile = e * g.T + t, rbg = e * g.nrb + rb;
    csf_tile_raw cur;
    if (n) cur = csf_tile_load<KIND>(src, tile, rbg, lane);
    for (; n; --n) {
        uint32_t jn = j, tn = t + 1, rbn = rb, cbn = cb + 1;
        uint64_t tilen = tile + 1, rbgn = rbg;
        if (cbn == g.ncb) { cbn = 0; ++rbn; ++rbgn; }
        if (tn == g.T) {
            tn = 0; rbn = 0; cbn = 0; ++jn;
            if (I.expert_start != nullptr && n > 1) {
                const uint64_t en = act[jn];
                tilen = en * g.T;
                rbgn = en * g.nrb;
            }
        }
        // expand this tile, then load the next one into the registers the
        // expansion has read (the patch needs only the index entries)
        const csf_tile_line L = csf_tile_expand<KIND>(cur);
        csf_tile_raw idx;
        idx.code = 0;
        idx.bw = 0;
        idx.x0 = cur.x0;
        idx.x1 = cur.x1;
        if (n > 1) cur = csf_tile_load<KIND>(src, tilen, rbgn, lane);
        const bool edge = rb >= full_rb || cb >= full_cb;
        bad |= tile_finish<KIND, STAGE>(src, rb, cb, edge, L, idx, STAGE ? nullptr : S.ws + tile * 512,
                                        STAGE ? sums + tile : nullptr, line, lane);
        j = jn; t = tn; rb = rbn; cb = cbn; tile = tilen; rbg = rbgn;
    }
    if (__any_sync(kFull, bad) && lane == 0) flag(S.err, CSF_DEV_ERR_CORRUPT);
}

}  // namespace

cudaError_t launch_tiled_checksum(const DecStack &S, const TiledIn &I, uint32_t *sums, int grid, size_t smem,
                                  cudaStream_t s) {
    if (S.kind == CSF_NVFP4)
        tiled_decode_kernel<CSF_NVFP4, true><<<grid, kTlThreads, smem, s>>>(S, I, sums);
    else
        tiled_decode_kernel<CSF_MXFP4, true><<<grid, kTlThreads, smem, s>>>(S, I, sums);
    return cudaGetLastError();
}

cudaError_t tiled_checksum_occupancy(int kind, size_t smem, int *blocks_per_sm) {
    if (kind == CSF_NVFP4)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, tiled_decode_kernel<CSF_NVFP4, true>,
                                                             kTlThreads, smem);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, tiled_decode_kernel<CSF_MXFP4, true>,
                                                         kTlThreads, smem);
}

cudaError_t launch_tiled_pack(const DecStack &S, const TiledOut &O, int grid, cudaStream_t s) {
    if (S.kind == CSF_NVFP4)
        tiled_pack_kernel<CSF_NVFP4><<<grid, kTlThreads, 0, s>>>(S, O);
    else
        tiled_pack_kernel<CSF_MXFP4><<<grid, kTlThreads, 0, s>>>(S, O);
    return cudaGetLastError();
}

cudaError_t tiled_decode_occupancy(int kind, size_t smem, int *blocks_per_sm) {
    if (kind == CSF_NVFP4)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, tiled_decode_kernel<CSF_NVFP4, false>,
                                                             kTlThreads, smem);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, tiled_decode_kernel<CSF_MXFP4, false>,
                                                         kTlThreads, smem);
}

cudaError_t launch_tiled_decode(const DecStack &S, const TiledIn &I, int grid, size_t smem, cudaStream_t s) {
    if (S.kind == CSF_NVFP4)
        tiled_decode_kernel<CSF_NVFP4, false><<<grid, kTlThreads, smem, s>>>(S, I, nullptr);
    else
        tiled_decode_kernel<CSF_MXFP4, false><<<grid, kTlThreads, smem, s>>>(S, I, nullptr);
    return cudaGetLastError();
}

}  // namespace csfk
