// CSF decode into the scale-operand layout of Blackwell block-scaled GEMMs
// (sm_103a): the 128 x 4 tiled layout that tcgen05 block scaling and
// cuBLASLt's VEC16_UE4M3 / VEC32_UE8M0 scale factors read, so that no layout
// pass runs between the decode and the GEMM.  This kernel works line by line
// in registers and serves rows wider than the shared-memory buffers of
// decode_blocks_kernel (csf_decode.cu) allow.
//
// Pages followed (cited by title and paragraph; they have no numbered
// sections):
//   "finegrained-kernels: decode losslessly compressed NVFP4 scales (CSF)":
//     format paragraph (base byte per row, 4-bit offsets, exception stream,
//     exact bytes); measurement paragraph (decode staging before the GEMM is
//     the cost to remove); helpers paragraph (routed experts only, no CPU
//     sync).
//   "NVFP4-CSF: expand_scales() for ahead-of-call scale expansion (canonical
//     twin of #477)": commit messages on one-bit MXFP4 / four-bit NVFP4
//     offsets, on zero padding of partial atoms, on both routing integer
//     types.
// The tiled layout itself is NVIDIA's documented block-scaling-factor
// layout: per expert, the R x C scales padded to 128-row / 4-column
// multiples, 128 x 4 tiles of 512 bytes in row-block-major order, line
// r % 32 of a tile holding rows r, r+32, r+64, r+96 with four columns each.
#include "csf_device.cuh"
#include "csf_internal.cuh"

namespace csfk {
namespace {

using dev::add_base;
using dev::flag;
using dev::kFull;
using dev::lanemask_lt;

constexpr int kTileWarps = kTileBlockWarps;
constexpr int kTileThreads = 32 * kTileWarps;

#ifndef CSF_TILES_MIN_BLOCKS
#define CSF_TILES_MIN_BLOCKS 8
#endif

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

// The 16 columns of round k of the lane's four rows (NVFP4: 64 nibble bits;
// MXFP4: offset bits in bits 0..15, escape bits in bits 32..47).
template <int KIND>
__device__ __forceinline__ uint64_t row_bits(const DecStack &S, uint32_t row, bool ok, uint32_t C, uint32_t k) {
    if (!ok) return 0;
    const uint64_t el = (uint64_t)row * C + 16u * k;
    if (KIND == CSF_NVFP4) return plane_bits(S.offsets, 4 * el, S.off_bytes);
    return (plane_bits(S.offsets, el, S.off_bytes) & 0xFFFFull) |
           ((plane_bits(S.escapes, el, S.off_bytes) & 0xFFFFull) << 32);
}

template <int KIND>
__device__ __forceinline__ void fetch_round(const DecStack &S, const uint32_t (&row)[4], const bool (&ok)[4],
                                            uint32_t C, uint32_t k, uint64_t &n0, uint64_t &n1, uint64_t &n2,
                                            uint64_t &n3) {
    n0 = row_bits<KIND>(S, row[0], ok[0], C, k);
    n1 = row_bits<KIND>(S, row[1], ok[1], C, k);
    n2 = row_bits<KIND>(S, row[2], ok[2], C, k);
    n3 = row_bits<KIND>(S, row[3], ok[3], C, k);
}

// Byte j (0..15) of the 16-byte group (w0, w1, w2, w3) becomes v.
__device__ __forceinline__ void put_byte4(uint32_t &w0, uint32_t &w1, uint32_t &w2, uint32_t &w3, uint32_t j,
                                          uint32_t v) {
    const uint32_t sh = 8 * (j & 3);
    const uint32_t m = 0xFFu << sh, x = v << sh;
    const uint32_t q = j >> 2;
    w0 = q == 0 ? (w0 & ~m) | x : w0;
    w1 = q == 1 ? (w1 & ~m) | x : w1;
    w2 = q == 2 ? (w2 & ~m) | x : w2;
    w3 = q == 3 ? (w3 & ~m) | x : w3;
}

// One round of one row: 16 columns from `bits` expanded on base A, the row's
// exceptions patched in column order from stream position X, the columns
// past the row (cv of 16 lie inside) and rows past R set to 0.
template <int KIND>
__device__ __forceinline__ void tile_row(const DecStack &S, uint64_t bits, uint32_t A, bool ok, uint32_t cv,
                                         uint32_t nexc, uint32_t &X, bool &bad, uint32_t &w0, uint32_t &w1,
                                         uint32_t &w2, uint32_t &w3) {
    const uint32_t A4 = A * 0x01010101u;
    uint32_t f0, f1;                                           // escape flags
    if (KIND == CSF_NVFP4) {
        const uint32_t x0 = (uint32_t)bits, x1 = (uint32_t)(bits >> 32);
        const uint32_t l0 = x0 & 0x0F0F0F0Fu, h0 = (x0 >> 4) & 0x0F0F0F0Fu;
        const uint32_t l1 = x1 & 0x0F0F0F0Fu, h1 = (x1 >> 4) & 0x0F0F0F0Fu;
        const uint32_t o0 = __byte_perm(l0, h0, 0x5140), o1 = __byte_perm(l0, h0, 0x7362);
        const uint32_t o2 = __byte_perm(l1, h1, 0x5140), o3 = __byte_perm(l1, h1, 0x7362);
        if (A <= 240u) {
            w0 = A4 + o0; w1 = A4 + o1; w2 = A4 + o2; w3 = A4 + o3;
        } else {
            w0 = add_base(A4, o0); w1 = add_base(A4, o1); w2 = add_base(A4, o2); w3 = add_base(A4, o3);
        }
        // nibble == 15 -> bit 4j (column j); columns past the row masked
        const uint64_t cm = cv >= 16 ? ~0ull : (1ull << (4 * cv)) - 1;
        f0 = x0 & (x0 >> 1) & (x0 >> 2) & (x0 >> 3) & 0x11111111u & (uint32_t)cm;
        f1 = x1 & (x1 >> 1) & (x1 >> 2) & (x1 >> 3) & 0x11111111u & (uint32_t)(cm >> 32);
    } else {
        const uint32_t o16 = (uint32_t)bits & 0xFFFFu;
        // bit i of each nibble -> byte i
        const uint32_t o0 = ((o16 & 0xFu) * 0x00204081u) & 0x01010101u;
        const uint32_t o1 = (((o16 >> 4) & 0xFu) * 0x00204081u) & 0x01010101u;
        const uint32_t o2 = (((o16 >> 8) & 0xFu) * 0x00204081u) & 0x01010101u;
        const uint32_t o3 = ((o16 >> 12) * 0x00204081u) & 0x01010101u;
        if (A <= 254u) {
            w0 = A4 + o0; w1 = A4 + o1; w2 = A4 + o2; w3 = A4 + o3;
        } else {
            w0 = add_base(A4, o0); w1 = add_base(A4, o1); w2 = add_base(A4, o2); w3 = add_base(A4, o3);
        }
        f0 = (uint32_t)(bits >> 32) & (cv >= 16 ? 0xFFFFu : (1u << cv) - 1);
        f1 = 0;
    }
    // Exceptions of the round, in column order, from the row's stream position.
    while (f0 | f1) {
        uint32_t j;
        if (KIND == CSF_NVFP4) {
            if (f0) { j = (uint32_t)(__ffs(f0) - 1) >> 2; f0 &= f0 - 1; }
            else    { j = 8 + ((uint32_t)(__ffs(f1) - 1) >> 2); f1 &= f1 - 1; }
        } else {
            j = (uint32_t)(__ffs(f0) - 1);
            f0 &= f0 - 1;
        }
        uint32_t v = 0;
        if (X < nexc) v = __ldg(S.exc_bytes + X);
        else bad = true;
        ++X;
        put_byte4(w0, w1, w2, w3, j, v);
    }
    // Padding: columns past C and rows past R are 0.
    const uint32_t m0 = cv >= 4 ? 0xFFFFFFFFu : (1u << (8 * cv)) - 1;
    const uint32_t m1 = cv >= 8 ? 0xFFFFFFFFu : (cv > 4 ? (1u << (8 * (cv - 4))) - 1 : 0u);
    const uint32_t m2 = cv >= 12 ? 0xFFFFFFFFu : (cv > 8 ? (1u << (8 * (cv - 8))) - 1 : 0u);
    const uint32_t m3 = cv >= 16 ? 0xFFFFFFFFu : (cv > 12 ? (1u << (8 * (cv - 12))) - 1 : 0u);
    w0 = ok ? w0 & m0 : 0u;
    w1 = ok ? w1 & m1 : 0u;
    w2 = ok ? w2 & m2 : 0u;
    w3 = ok ? w3 & m3 : 0u;
}

// One warp writes every tile of one 128-row block of expert e: lane b owns
// rows b, b+32, b+64, b+96 of the block, which are exactly the rows of line
// b in each 128 x 4 tile.  The lane reads 16 columns of each of its rows a
// round (the next round's bits are fetched ahead), expands them, patches
// its own rows' exceptions in order (each row's position starts at its
// index entry, so no scan is needed), and stores line b of four tiles; the
// warp's 32 lines make each tile one coalesced 512-byte store.
template <int KIND>
__device__ void tile_block(const DecStack &S, uint64_t e, uint32_t rl0, int lane) {
    const uint32_t R = (uint32_t)S.R, C = (uint32_t)S.C;
    const uint32_t ncb = (C + 3) / 4;
    const uint32_t nrounds = (ncb + 3) / 4;
    const uint64_t RP = ((uint64_t)R + kTileRows - 1) / kTileRows * kTileRows;
    uint8_t *line = S.ws + e * RP * (4ull * ncb) + (uint64_t)(rl0 / kTileRows) * ncb * 512 + 16u * (uint32_t)lane;
    const uint32_t nexc = (uint32_t)S.num_exc;
    uint32_t row[4], A[4], X[4], Xend[4];
    bool ok[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const uint32_t rl = rl0 + (uint32_t)lane + 32u * a;
        ok[a] = rl < R;
        row[a] = (uint32_t)(e * R) + rl;
        A[a] = ok[a] ? (uint32_t)__ldg(S.base + row[a]) : 0u;
        X[a] = ok[a] ? __ldg(S.exc_index + row[a]) : 0u;
        Xend[a] = ok[a] ? __ldg(S.exc_index + row[a] + 1) : 0u;
    }
    bool bad = false;
    uint64_t n0, n1, n2, n3;
    fetch_round<KIND>(S, row, ok, C, 0, n0, n1, n2, n3);
    for (uint32_t k = 0; k < nrounds; ++k) {
        const uint64_t cur[4] = {n0, n1, n2, n3};
        if (k + 1 < nrounds) fetch_round<KIND>(S, row, ok, C, k + 1, n0, n1, n2, n3);
        const uint32_t cv = min(16u, C - 16u * k);             // columns of the round inside the row
        uint32_t w[4][4];
        tile_row<KIND>(S, cur[0], A[0], ok[0], cv, nexc, X[0], bad, w[0][0], w[0][1], w[0][2], w[0][3]);
        tile_row<KIND>(S, cur[1], A[1], ok[1], cv, nexc, X[1], bad, w[1][0], w[1][1], w[1][2], w[1][3]);
        tile_row<KIND>(S, cur[2], A[2], ok[2], cv, nexc, X[2], bad, w[2][0], w[2][1], w[2][2], w[2][3]);
        tile_row<KIND>(S, cur[3], A[3], ok[3], cv, nexc, X[3], bad, w[3][0], w[3][1], w[3][2], w[3][3]);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t cb = 4 * k + g;
            if (cb < ncb)
                *reinterpret_cast<uint4 *>(line + (uint64_t)cb * 512) = make_uint4(w[0][g], w[1][g], w[2][g], w[3][g]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
        if (ok[a] && X[a] != Xend[a]) bad = true;
    if (__any_sync(kFull, bad) && lane == 0) flag(S.err, CSF_DEV_ERR_CORRUPT);
}

__global__ void __launch_bounds__(kTileThreads, CSF_TILES_MIN_BLOCKS) decode_tiles_kernel(const __grid_constant__ DecParams P) {
    extern __shared__ __align__(16) uint32_t act[];
    __shared__ uint32_t s_cnt[kTileWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint32_t n_act = (uint32_t)P.E;
    if (P.expert_start != nullptr) {
        n_act = 0;
        for (int e0 = 0; e0 < P.E; e0 += kTileThreads) {
            const int e = e0 + threadIdx.x;
            bool a = false;
            if (e < P.E) {
                if (P.es64) {
                    const long long *st = static_cast<const long long *>(P.expert_start);
                    a = __ldg(st + e + 1) > __ldg(st + e);
                } else {
                    const int *st = static_cast<const int *>(P.expert_start);
                    a = __ldg(st + e + 1) > __ldg(st + e);
                }
            }
            const uint32_t bal = __ballot_sync(kFull, a);
            if (lane == 0) s_cnt[warp] = __popc(bal);
            __syncthreads();
            uint32_t bn = n_act, tn = 0;
#pragma unroll
            for (int w = 0; w < kTileWarps; ++w) {
                if (w < warp) bn += s_cnt[w];
                tn += s_cnt[w];
            }
            if (a) act[bn + __popc(bal & lanemask_lt())] = (uint32_t)e;
            n_act += tn;
            __syncthreads();
        }
    }
    const uint32_t B0 = (uint32_t)(P.st[0].r_hi - P.st[0].r_lo + kTileRows - 1) / kTileRows;
    const uint32_t B1 = P.nstacks > 1 ? (uint32_t)(P.st[1].r_hi - P.st[1].r_lo + kTileRows - 1) / kTileRows : 0u;
    const uint64_t it0 = (uint64_t)n_act * B0;
    const uint64_t total = it0 + (uint64_t)n_act * B1;
    const uint64_t nw = (uint64_t)gridDim.x * kTileWarps;
    for (uint64_t it = (uint64_t)blockIdx.x * kTileWarps + warp; it < total; it += nw) {
        const int s = it < it0 ? 0 : 1;
        const DecStack &S = P.st[s];
        const uint32_t Bs = s ? B1 : B0;
        const uint64_t li = s ? it - it0 : it;
        const uint32_t j = (uint32_t)(li / Bs);
        const uint32_t t = (uint32_t)(li - (uint64_t)j * Bs);
        const uint64_t e = P.expert_start != nullptr ? act[j] : j;
        const uint32_t rl0 = (uint32_t)S.r_lo + t * kTileRows;
        if (S.kind == CSF_NVFP4) tile_block<CSF_NVFP4>(S, e, rl0, lane);
        else tile_block<CSF_MXFP4>(S, e, rl0, lane);
    }
}

}  // namespace

cudaError_t decode_tiles_occupancy(size_t smem, int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_tiles_kernel, kTileThreads, smem);
}

cudaError_t launch_decode_tiles(const DecParams &p, int grid, size_t smem, cudaStream_t s) {
    decode_tiles_kernel<<<grid, kTileThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace csfk
