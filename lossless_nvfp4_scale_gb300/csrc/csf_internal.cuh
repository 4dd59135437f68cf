// Internal declarations shared by the CSF library's translation units.
// Nothing here is part of the C ABI (include/csf.h is).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "csf.h"

namespace csfk {

constexpr int kThreads = 256;               // threads per block, every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRoutedExperts = 8192;     // routed decode keeps the active list in smem

// Prepare tiles start where the packed planes start a 16-byte piece:
// 32 elements (NVFP4 nibbles), 128 elements (MXFP4 bits).
constexpr int kChunkNv = 32;
constexpr int kChunkMx = 128;
// Decode lane chunks: NVFP4 64 elements (32 offset bytes -> 64 dense bytes),
// MXFP4 128 elements (16 bytes of each plane -> 128 dense bytes).  Decode
// segments start on lane-chunk boundaries.
constexpr int kLaneNv = 64;
constexpr int kLaneMx = 128;

// One stack as the decode kernel sees it.
struct DecStack {
    const uint8_t *base;
    const uint8_t *offsets;
    const uint8_t *escapes;
    const uint32_t *exc_index;
    const uint8_t *exc_bytes;
    uint8_t *ws;
    uint32_t *err;        // may be null
    uint64_t num_exc;
    uint64_t rows;        // E*R
    uint64_t n;           // E*R*C
    int32_t R;
    int32_t C;
    int32_t kind;
    int32_t rb;           // rows per work unit: smallest count whose elements fill whole chunks
    uint32_t step_r;      // (32 lane chunks of elements) / C
    uint32_t step_q;      // (32 lane chunks of elements) % C
    int32_t ws_align;     // alignment of ws in bytes (32, 16, 4 or 1)
    int32_t off_align32;  // offsets pointer is 32-byte aligned (256-bit loads)
    uint64_t off_bytes;   // readable bytes at offsets (packed length rounded up to 16)
    uint64_t max_units;   // units per segment so that a segment stays below 2^30 elements
    int32_t r_lo;         // rows [r_lo, r_hi) of each expert are written (0, R: all)
    int32_t r_hi;
    uint32_t upe;         // units per expert when R % rb == 0 (every expert alike), else 0
    uint32_t pad_;
};

struct DecParams {
    DecStack st[2];
    int32_t nstacks;
    int32_t E;
    const void *expert_start;   // null: every expert
    int32_t es64;
    int32_t uniform;            // every stack has R % rb == 0: unit -> expert is a division
    uint32_t buf_off;           // scale-operand layout by blocks: dynamic smem offset of the 128-row buffer
    uint32_t buf_bytes;         // bytes of that buffer
};

struct PrepParams {
    const uint8_t *dense;
    uint8_t *base;
    uint8_t *offsets;
    uint8_t *escapes;
    uint32_t *exc_index;
    uint8_t *exc_bytes;
    uint32_t *err;               // may be null
    unsigned int *ticket;        // scratch: tile ticket counter (zeroed)
    unsigned long long *status;  // scratch: one look-back word per tile (zeroed; wide rows)
    uint32_t *tile_total;        // scratch: exception total of each tile (row path)
    uint64_t exc_capacity;
    uint64_t rows;
    uint64_t n;
    uint64_t num_tiles;
    uint64_t magic;              // ceil(2^40 / C): tile-local element -> row
    int32_t C;
    int32_t kind;
    int32_t tr;                  // rows per tile
    int32_t dense_aligned;       // dense pointer is 16-byte aligned
    uint32_t smem_dense;         // byte sizes of the dynamic smem regions
    uint32_t smem_planes;
    int32_t stride;              // row stride of the staged tile (row-wise kernel)
    int32_t stage;               // row-wise kernel: how the tile is staged (plain loads, one bulk copy, a copy per row)
    uint32_t spin_limit;         // polls before a bounded wait gives up (CSF_DEV_ERR_TIMEOUT)
    uint32_t smem_hist;          // row-wise kernel: bytes of the bins / exception staging region
    int32_t nbuf;                // base kernel: tile staging buffers (2: the next tile loads during this one)
    int32_t nbuf_enc;            // encode kernel: the same
    uint32_t exc_stage;          // encode kernel: bytes of the shared-memory exception stage
    uint32_t slot_bytes;         // fused path: bytes of a tile's exception slot in the scratch
    uint8_t *slot;               // fused path: the slots (scratch), one per tile
    int32_t fused;               // row path in one pass per tile plus a placing kernel
    int32_t pad4_;
};

// Rows per unit so that a unit's first element starts a whole chunk.
inline int32_t unit_rows(int32_t C, int chunk) {
    int32_t g = C;
    int32_t a = chunk;
    while (a) { int32_t t = g % a; g = a; a = t; }   // gcd(C, chunk)
    return chunk / g;
}

// Which segment decoders a row-major decode launch compiles in: NVFP4 only,
// MXFP4 only, or both (a pair of stacks of different kinds).
enum DecodeKinds { kKindsNv = 0, kKindsMx = 1, kKindsBoth = 2 };
inline int decode_kinds(const DecParams &p) {
    const int k0 = p.st[0].kind;
    if (p.nstacks > 1 && p.st[1].kind != k0) return kKindsBoth;
    return k0 == CSF_NVFP4 ? kKindsNv : kKindsMx;
}
cudaError_t launch_decode(const DecParams &p, int grid, size_t smem, bool routed, cudaStream_t s);
cudaError_t decode_occupancy(bool routed, int kinds, size_t smem, int *blocks_per_sm);
// Decode into the 128 x 4 tiled scale-operand layout of block-scaled GEMMs
// (one warp per 128-row block of an expert).
constexpr int kTileRows = 128;
constexpr int kTileBlockWarps = 4;   // warps per block
// Same layout, one thread block per 128-row block, decoded by the row-major
// segment code into a shared-memory buffer (csf_decode.cu).
#ifndef CSF_BLK_WARPS
#define CSF_BLK_WARPS 2
#endif
constexpr int kBlkWarps = CSF_BLK_WARPS;
constexpr int kBlkThreads = 32 * kBlkWarps;
cudaError_t launch_decode_blocks(const DecParams &p, int grid, size_t smem, cudaStream_t s);
cudaError_t decode_blocks_occupancy(const DecParams &p, size_t smem, int *blocks_per_sm);
cudaError_t launch_decode_tiles(const DecParams &p, int grid, size_t smem, cudaStream_t s);
cudaError_t decode_tiles_occupancy(size_t smem, int *blocks_per_sm);

// Tile-packed CSF (csf_tiled.cu).
struct TiledOut {
    uint8_t *codes;
    uint8_t *bases;
    uint32_t *tile_index;
    uint8_t *exc_bytes;
    uint64_t exc_capacity;
    uint32_t *err;          // may be null
};

struct TiledIn {
    const uint8_t *codes;
    const uint8_t *bases;
    const uint32_t *tile_index;
    const uint8_t *exc_bytes;
    uint64_t num_exc;
    const void *expert_start;   // null: every expert
    int32_t es64;
    int32_t pad_;
};

cudaError_t launch_tiled_pack(const DecStack &S, const TiledOut &O, int grid, cudaStream_t s);
cudaError_t tiled_decode_occupancy(int kind, size_t smem, int *blocks_per_sm);
cudaError_t launch_tiled_decode(const DecStack &S, const TiledIn &I, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_tiled_checksum(const DecStack &S, const TiledIn &I, uint32_t *sums, int grid, size_t smem,
                                  cudaStream_t s);
cudaError_t tiled_checksum_occupancy(int kind, size_t smem, int *blocks_per_sm);

// Geometry checks shared by every entry point: sets N = E*R*C and rows = E*R.
csf_status check_geometry(const csf_geometry *g, uint64_t *n, uint64_t *rows);

// A checked prepare, shared by csf_prepare and csf_prepare_static:
// prepare_check makes the host-only argument checks and sizes the look-back
// scratch (no CUDA call); prepare_configure picks the launch configuration
// (it may query the device); prepare_enqueue clears the scratch on `s` and
// launches the kernel.
struct PrepPlan {
    uint64_t n;
    uint64_t rows;
    uint64_t scratch_bytes;   // the least scratch: per-tile totals or look-back words
    uint64_t fused_bytes;     // scratch of the fused row path (0: not available)
    bool fused;               // the caller's scratch takes the fused row path
    bool staged;
    size_t smem;
};
csf_status prepare_check(const uint8_t *dense, const csf_stack *out, uint64_t exc_capacity, PrepPlan *plan);
csf_status prepare_configure(const uint8_t *dense, const csf_geometry &g, PrepPlan *plan);
csf_status prepare_enqueue(const uint8_t *dense, const csf_stack &out, uint64_t exc_capacity, void *scratch,
                           const PrepPlan &plan, cudaStream_t s);

cudaError_t launch_prepare(const PrepParams &p, size_t smem, cudaStream_t s);
void make_prep_params(PrepParams &p, const uint8_t *dense, const csf_stack &out, uint64_t exc_capacity,
                      void *scratch, uint64_t rows, uint64_t n, bool staged, bool fused);
// Scratch bytes of the fused row path (rows of up to 255 bytes; 0 for wider
// rows, which have no fused path).
uint64_t prepare_fused_scratch_bytes(int32_t kind, int32_t C, uint64_t rows);
size_t prepare_smem_bytes(int32_t kind, int32_t C, int32_t tr, bool staged);
bool prepare_stages_rows(int32_t kind, int32_t C, const void *dense);
bool prepare_needs_cleared_scratch(int32_t C);
int32_t prepare_tile_rows(int32_t kind, int32_t C);

}  // namespace csfk
