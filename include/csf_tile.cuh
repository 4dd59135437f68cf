/*
 * csf_tile.cuh -- device-side decoder of one tile of a tile-packed CSF stack
 * (csf_tiled, see csf.h), for CUDA kernels that read scales per pipeline
 * stage.  Header only; include it in a .cu file compiled for sm_103a.
 *
 * Source: [B478] "NVFP4-CSF: expand_scales() for ahead-of-call scale
 * expansion (canonical twin of #477)", commit message on packed experts whose
 * scales stay compressed and are rebuilt by each GEMM pipeline stage in
 * shared memory.  The pages give no record layout; the tile-packed form of
 * csf.h is this library's.  A stage that is about to consume the scales of
 * one 128-row x 4-column block calls csf_tile_decode_warp with that tile's
 * coordinates: one warp rebuilds the 512 scale bytes in shared memory, in the
 * 128 x 4 block-scaled layout (CSF_LAYOUT_BLOCKED order), and nothing is
 * written to global memory.
 *
 * Layout read (csf.h, csf_tiled): per expert nrb = ceil(R/128) row blocks and
 * ncb = ceil(C/4) column blocks, tile t = rb * ncb + cb, global tile
 * e * nrb * ncb + t; lane b of the warp owns line b of the tile (rows
 * 128 rb + b + 32 a, a = 0..3, columns 4 cb .. 4 cb + 3):
 *   codes  NVFP4 256 bytes a tile (lane b: bytes 8b .. 8b+7, position
 *          q = 16b + 4a + c in nibble q, nibble 15 = exception); MXFP4 128
 *          bytes (offset bits of lane b in bytes 2b, 2b+1; escape bits in
 *          64 + 2b, 64 + 2b + 1).
 *   bases  128 bytes per expert and row block: word b = the bases of rows
 *          b, b+32, b+64, b+96.
 *   tile_index  exclusive prefix of the tiles' exception counts; a tile's
 *          exceptions are in position order.
 * Decoded byte = base + offset (mod 256), or the next exception byte.
 * Padding positions (rows >= R, columns >= C) decode to 0.
 */
#ifndef CSF_TILE_CUH
#define CSF_TILE_CUH

#include <stdint.h>

#include "csf.h"

/* The device view of a tile-packed stack (plain pointers and sizes). */
struct csf_tile_src {
    const uint8_t *codes;
    const uint8_t *bases;
    const uint32_t *tile_index;
    const uint8_t *exc_bytes;
    uint32_t num_exc;   /* exceptions in the stream (bounds every read) */
    int32_t kind;       /* CSF_NVFP4 or CSF_MXFP4 */
    int32_t R;          /* rows per expert */
    int32_t C;          /* scale columns per row */
};

/* The device view of a csf_tiled (host or device code). */
__host__ __device__ inline csf_tile_src csf_tile_src_of(const csf_tiled &t) {
    csf_tile_src s;
    s.codes = t.codes;
    s.bases = t.bases;
    s.tile_index = t.tile_index;
    s.exc_bytes = t.exc_bytes;
    s.num_exc = (uint32_t)t.num_exc;
    s.kind = t.g.kind;
    s.R = t.g.rows;
    s.C = t.g.cols;
    return s;
}

__host__ __device__ inline uint32_t csf_tile_row_blocks(const csf_tile_src &s) { return ((uint32_t)s.R + 127u) / 128u; }
__host__ __device__ inline uint32_t csf_tile_col_blocks(const csf_tile_src &s) { return ((uint32_t)s.C + 3u) / 4u; }

/* Lane b's raw inputs of one tile: its 8 code bytes (NVFP4) or 2 + 2 plane
 * bytes (MXFP4), its 4 row bases, and (lane 0) the tile's index entries. */
struct csf_tile_raw {
    uint64_t code;
    uint32_t bw;
    uint32_t x0, x1;
};

/* Lane b's line of a tile before exceptions: 16 bytes (word a = row
 * 128 rb + b + 32 a, byte c = column 4 cb + c), the escape flags (NVFP4: bit
 * 4j for byte j of the line; MXFP4: bit j) and their count. */
struct csf_tile_line {
    uint32_t w0, w1, w2, w3;
    uint64_t f;
    uint32_t cnt;
};

namespace csf_tile_detail {

/* base + offset byte-wise mod 256 for offsets below 0x80: the low 7 bits are
 * added, bit 7 is folded back with XOR, so no carry crosses a byte. */
__device__ __forceinline__ uint32_t add_base(uint32_t bw, uint32_t off) {
    return ((bw & 0x7F7F7F7Fu) + off) ^ (bw & 0x80808080u);
}

/* One step of a warp inclusive scan: the shuffle's predicate (the source lane
 * exists) guards the add, so no lane-index compare is needed. */
template <int D>
__device__ __forceinline__ void scan_step(uint32_t &x) {
    asm("{\n .reg .b32 y;\n .reg .pred p;\n shfl.sync.up.b32 y|p, %0, %1, 0, -1;\n @p add.u32 %0, %0, y;\n}"
        : "+r"(x)
        : "n"(D));
}

__device__ __forceinline__ uint32_t excl_scan(uint32_t v, int lane, uint32_t &total) {
    (void)lane;
    uint32_t x = v;
    scan_step<1>(x);
    scan_step<2>(x);
    scan_step<4>(x);
    scan_step<8>(x);
    scan_step<16>(x);
    total = __shfl_sync(0xFFFFFFFFu, x, 31);
    return x - v;
}

}  // namespace csf_tile_detail

/* Lane's inputs of global tile `tile`, whose row block is `rbg` (expert *
 * nrb + rb).  All 32 lanes call it. */
template <int KIND>
__device__ __forceinline__ csf_tile_raw csf_tile_load(const csf_tile_src &s, uint64_t tile, uint64_t rbg, int lane) {
    csf_tile_raw r;
    r.bw = __ldg(reinterpret_cast<const uint32_t *>(s.bases) + rbg * 32 + lane);
    if (KIND == CSF_NVFP4) {
        r.code = __ldg(reinterpret_cast<const unsigned long long *>(s.codes + tile * 256) + lane);
    } else {
        const uint16_t *c16 = reinterpret_cast<const uint16_t *>(s.codes + tile * 128);
        r.code = (uint64_t)__ldg(c16 + lane) | ((uint64_t)__ldg(c16 + 32 + lane) << 32);
    }
    r.x0 = r.x1 = 0;
    if (lane == 0) {
        r.x0 = __ldg(s.tile_index + tile);
        r.x1 = __ldg(s.tile_index + tile + 1);
    }
    return r;
}

/* Lane's line from its raw inputs: offsets expanded to bytes and the row
 * bases added (no exceptions yet). */
template <int KIND>
__device__ __forceinline__ csf_tile_line csf_tile_expand(const csf_tile_raw &r) {
    using csf_tile_detail::add_base;
    csf_tile_line L;
    if (KIND == CSF_NVFP4) {
        const uint32_t x0 = (uint32_t)r.code, x1 = (uint32_t)(r.code >> 32);
        const uint32_t l0 = x0 & 0x0F0F0F0Fu, h0 = (x0 >> 4) & 0x0F0F0F0Fu;
        const uint32_t l1 = x1 & 0x0F0F0F0Fu, h1 = (x1 >> 4) & 0x0F0F0F0Fu;
        L.w0 = __byte_perm(l0, h0, 0x5140);
        L.w1 = __byte_perm(l0, h0, 0x7362);
        L.w2 = __byte_perm(l1, h1, 0x5140);
        L.w3 = __byte_perm(l1, h1, 0x7362);
        const uint32_t f0 = x0 & (x0 >> 1) & (x0 >> 2) & (x0 >> 3) & 0x11111111u;   /* nibble 15 -> bit 4j */
        const uint32_t f1 = x1 & (x1 >> 1) & (x1 >> 2) & (x1 >> 3) & 0x11111111u;
        L.cnt = __popc(f0) + __popc(f1);
        L.f = (uint64_t)f0 | ((uint64_t)f1 << 32);
    } else {
        const uint32_t o16 = (uint32_t)r.code & 0xFFFFu, x16 = (uint32_t)(r.code >> 32) & 0xFFFFu;
        L.w0 = ((o16 & 0xFu) * 0x00204081u) & 0x01010101u;                            /* bit i -> byte i */
        L.w1 = (((o16 >> 4) & 0xFu) * 0x00204081u) & 0x01010101u;
        L.w2 = (((o16 >> 8) & 0xFu) * 0x00204081u) & 0x01010101u;
        L.w3 = ((o16 >> 12) * 0x00204081u) & 0x01010101u;
        L.f = x16;
        L.cnt = __popc(x16);
    }
    /* row bases, byte a of bw for word a, added byte by byte modulo 256 */
    L.w0 = add_base(__byte_perm(r.bw, 0, 0x0000), L.w0);
    L.w1 = add_base(__byte_perm(r.bw, 0, 0x1111), L.w1);
    L.w2 = add_base(__byte_perm(r.bw, 0, 0x2222), L.w2);
    L.w3 = add_base(__byte_perm(r.bw, 0, 0x3333), L.w3);
    return L;
}

/* The tile's exceptions, whole warp: lane b's ones are written in place into
 * `line`, the 16 bytes of shared memory that hold its expanded line (no other
 * lane touches them).  Returns true on every lane when the tile's index and
 * its escape codes disagree or an index points past the stream (those bytes
 * read as 0). */
template <int KIND>
__device__ __forceinline__ bool csf_tile_patch(const csf_tile_src &s, const csf_tile_raw &r, const csf_tile_line &L,
                                               uint8_t *line, int lane) {
    uint32_t tot;
    const uint32_t pre = csf_tile_detail::excl_scan(L.cnt, lane, tot);
    const uint32_t X = __shfl_sync(0xFFFFFFFFu, r.x0, 0);
    bool bad = false;
    uint64_t f = L.f;
    uint32_t k = X + pre;
    while (f) {
        const uint32_t bit = (uint32_t)(__ffsll((long long)f) - 1);
        const uint32_t j = KIND == CSF_NVFP4 ? bit >> 2 : bit;
        f &= f - 1;
        uint8_t v = 0;
        if (k < s.num_exc) v = __ldg(s.exc_bytes + k);
        else bad = true;
        ++k;
        line[j] = v;
    }
    if (lane == 0 && X + tot != r.x1) bad = true;
    return __any_sync(0xFFFFFFFFu, bad);
}

/* Padding of an edge tile (rows >= R, columns >= C) to 0: lane b's line of
 * row block rb, column block cb. */
__device__ __forceinline__ void csf_tile_mask_edge(const csf_tile_src &s, uint32_t rb, uint32_t cb, int lane,
                                                   uint32_t &w0, uint32_t &w1, uint32_t &w2, uint32_t &w3) {
    const uint32_t R = (uint32_t)s.R, C = (uint32_t)s.C;
    const uint32_t rl = rb * 128u + (uint32_t)lane;
    const uint32_t cv = min(4u, C - 4u * cb);
    const uint32_t cm = cv >= 4 ? 0xFFFFFFFFu : (1u << (8 * cv)) - 1;
    w0 = rl < R ? w0 & cm : 0u;
    w1 = rl + 32 < R ? w1 & cm : 0u;
    w2 = rl + 64 < R ? w2 & cm : 0u;
    w3 = rl + 96 < R ? w3 & cm : 0u;
}

/* Decode tile (expert, rb, cb) into `dst`: 512 bytes of shared memory,
 * 16-byte aligned, in the block-scaled order (byte 16 b + 4 a + c = row
 * 128 rb + b + 32 a, column 4 cb + c).  Called by all 32 lanes of one warp;
 * the tile is complete in `dst` for the whole warp on return.  Returns true
 * (every lane) when the tile's index disagrees with its codes. */
template <int KIND>
__device__ __forceinline__ bool csf_tile_decode_warp(const csf_tile_src &s, uint64_t expert, uint32_t rb, uint32_t cb,
                                                     uint8_t *dst) {
    const int lane = (int)(threadIdx.x & 31u);
    const uint64_t nrb = csf_tile_row_blocks(s), ncb = csf_tile_col_blocks(s);
    const uint64_t rbg = expert * nrb + rb;
    const uint64_t tile = rbg * ncb + cb;
    const csf_tile_raw r = csf_tile_load<KIND>(s, tile, rbg, lane);
    const csf_tile_line L = csf_tile_expand<KIND>(r);
    uint4 *line = reinterpret_cast<uint4 *>(dst) + lane;
    *line = make_uint4(L.w0, L.w1, L.w2, L.w3);
    const bool bad = csf_tile_patch<KIND>(s, r, L, reinterpret_cast<uint8_t *>(line), lane);
    if (128u * (rb + 1) > (uint32_t)s.R || 4u * (cb + 1) > (uint32_t)s.C) {
        uint4 q = *line;
        csf_tile_mask_edge(s, rb, cb, lane, q.x, q.y, q.z, q.w);
        *line = q;
    }
    __syncwarp();
    return bad;
}

#endif /* CSF_TILE_CUH */
