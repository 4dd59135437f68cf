/*
 * csf.h -- C ABI of the GB300 (sm_103a) CSF scale codec library (libcsf.so).
 *
 * CSF stores the FP8 scale bytes of FP4 MoE expert weights losslessly: one
 * base byte per row, most scales as small offsets from that base, and the
 * bytes outside the offset range in an exception stream found through a
 * per-row prefix index.  Decoding rebuilds the original bytes exactly.
 *
 * Sources (web pages, cited by title and paragraph; they have no numbered
 * sections):
 *   [FK]   "finegrained-kernels: decode losslessly compressed NVFP4 scales
 *           (CSF)": format paragraph (base byte per row, 4-bit offsets,
 *           exception stream, exact bytes); strategy table (decode once, or
 *           keep compressed and decode into one shared workspace before each
 *           GEMM); helpers paragraph (a prepare helper that keeps the input
 *           device, a GPU decoder into caller-owned reusable workspace, the
 *           grouped-routing expert_start tensor skipping inactive experts in
 *           both the fixed-stream and exception passes, no CPU sync);
 *           validation paragraph (reusable odd-offset workspace).
 *   [B478] "NVFP4-CSF: expand_scales() for ahead-of-call scale expansion
 *           (canonical twin of #477)": commit messages on one-bit MXFP4 and
 *           four-bit NVFP4 offsets from a row base byte, on pairing gate/up
 *           and down scales without extra streams, on both routing integer
 *           types, and on caller-owned scratch.
 *   [B477] "NVFP4-CSF: expand_scales() for ahead-of-call scale expansion":
 *           body (expansion into the shared scratch ahead of the call, on a
 *           side stream, with the caller ordering the streams).
 *   [V964] "Load native FP4 experts with optional lossless CSF scales":
 *           GPU encoding plus exception index at preparation time.
 *
 * Byte layout of a stack of E experts x R rows x C scale bytes
 * (N = E*R*C elements, rows = E*R; element i = (e*R + r)*C + c):
 *   base[rows]            one byte per row.
 *   NVFP4 offsets         flat nibble stream over all N elements: element i
 *                         in byte i/2, even i in the low nibble.  Nibble
 *                         0..14 = offset from the row base, 15 = exception.
 *   MXFP4 offsets/escapes two flat LSB-first bit planes (element i in byte
 *                         i/8, bit i%8): offset bit, and escape bit (1 =
 *                         exception; its offset bit is 0).
 *   exc_index[rows+1]     uint32 exclusive prefix of per-row exception
 *                         counts; exc_index[rows] = total exceptions.
 *   exc_bytes[total]      exception bytes, row-major.
 * Decoded byte: base[row] + offset (mod 256), or, for an exception, the byte
 * at exc_index[row] + (number of earlier exceptions in the same row).
 * Encoding is canonical: the base is the smallest byte present in the row
 * whose window [base, base+w] (w = 14 NVFP4, 1 MXFP4) holds the most of the
 * row's bytes; pad nibbles/bits past N are 0.
 *
 * Conventions shared by every call:
 *   - All buffer pointers are DEVICE pointers owned by the caller; the library
 *     never allocates or frees device memory.  Calls are asynchronous on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream) and never
 *     synchronise the host.  The one exception is the self-test
 *     csf_selftest_lookback_timeout, which allocates, runs and synchronises
 *     on its own.
 *   - The return value reports argument and launch errors only.  Data errors
 *     found on the device (a corrupt index, a full exception buffer, a bounded
 *     wait that gave up) are OR-ed into the optional device word
 *     `error_word` as CSF_DEV_ERR_* bits; kernels never trap, and their reads
 *     and writes stay inside the buffers described here.
 *   - Packed streams are read in 16-byte pieces: `offsets` and `escapes` must
 *     be 16-byte aligned and allocated to the lengths csf_sizes() reports
 *     (the packed length rounded up to 16 bytes).
 */
#ifndef CSF_H
#define CSF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSF_ABI_VERSION 5

typedef enum {
    CSF_OK = 0,
    CSF_ERR_ARG = 1,         /* NULL/unaligned pointer, bad kind, host pointer where a device one is needed */
    CSF_ERR_SIZE = 2,        /* a buffer or scratch smaller than the geometry needs */
    CSF_ERR_UNSUPPORTED = 3, /* geometry beyond the library's limits (see csf_sizes) */
    CSF_ERR_CUDA = 4         /* a CUDA runtime call or a launch failed */
} csf_status;

/* Device error-word bits (OR-ed, never cleared by the library). */
#define CSF_DEV_ERR_CORRUPT  0x1u /* index disagrees with the escape codes, or points past the stream */
#define CSF_DEV_ERR_CAPACITY 0x2u /* prepare: more exceptions than exc_capacity (exc_index still complete) */
#define CSF_DEV_ERR_TIMEOUT  0x4u /* prepare: a bounded inter-block wait gave up */

typedef enum {
    CSF_NVFP4 = 0, /* UE4M3 scales, one per 16 weights: 4-bit offsets, escape nibble 15 */
    CSF_MXFP4 = 1  /* UE8M0 scales, one per 32 weights: 1-bit offset plane + 1-bit escape plane */
} csf_kind;

typedef struct {
    int32_t kind;        /* csf_kind */
    int32_t num_experts; /* E >= 1 */
    int32_t rows;        /* R >= 1 rows (output channels) per expert */
    int32_t cols;        /* C >= 1 scale bytes per row (K/16 NVFP4, K/32 MXFP4) */
} csf_geometry;

/* Allocation sizes in bytes for one geometry (csf_sizes). */
typedef struct {
    uint64_t dense;           /* E*R*C: the dense stack and a decode workspace */
    uint64_t base;            /* rows */
    uint64_t offsets;         /* packed offsets rounded up to 16 */
    uint64_t escapes;         /* MXFP4 escape plane rounded up to 16; 0 for NVFP4 */
    uint64_t exc_index;       /* 4*(rows+1) */
    uint64_t prepare_scratch; /* scratch for csf_prepare's fastest path */
    uint64_t blocked;         /* a workspace in CSF_LAYOUT_BLOCKED: E * (R up to 128) * (C up to 4) */
    uint64_t tiled_codes;     /* csf_tiled codes: 256 (NVFP4) or 128 (MXFP4) bytes a tile */
    uint64_t tiled_bases;     /* csf_tiled bases: 128 bytes per expert and 128-row block */
    uint64_t tiled_index;     /* csf_tiled tile_index: 4 * (tiles + 1) */
} csf_sizes_t;

/*
 * A compressed stack: device buffers owned by the caller.  csf_prepare fills
 * them; csf_decode, csf_decode_pair and csf_decode_rows read them.  `num_exc`
 * is the host copy of exc_index[rows] (the caller reads it once after
 * prepare); `exc_bytes` must be readable for num_exc bytes rounded up to a
 * multiple of 16.
 */
typedef struct {
    csf_geometry g;
    uint8_t *base;
    uint8_t *offsets;
    uint8_t *escapes;     /* MXFP4 only; NULL for NVFP4 */
    uint32_t *exc_index;
    uint8_t *exc_bytes;
    uint64_t num_exc;
    uint32_t *error_word; /* optional device word for CSF_DEV_ERR_* bits; may be NULL */
} csf_stack;

/* Human-readable name of a status code. */
const char *csf_status_string(csf_status status);

/* CSF_ABI_VERSION of the loaded library. */
int csf_abi_version(void);

/*
 * Allocation sizes for a geometry.  Host only, no CUDA calls.  Returns
 * CSF_ERR_ARG for a bad kind or non-positive sizes, CSF_ERR_UNSUPPORTED when
 * N >= 2^40 or rows >= 2^31.
 */
csf_status csf_sizes(const csf_geometry *g, csf_sizes_t *out);

/*
 * Encode a dense stack on the GPU: base bytes, offset (and escape) planes,
 * the exception index and the exception stream, in one pass over the dense
 * bytes ([FK] format and helpers paragraphs; [V964] encoding plus index).
 *
 *   dense          device, E*R*C bytes, row-major [E][R][C], any alignment.
 *   out            geometry and destination buffers (base, offsets,
 *                  escapes for MXFP4, exc_index, exc_bytes, error_word).
 *                  out->num_exc is not written (read exc_index[rows]).
 *   exc_capacity   bytes available at out->exc_bytes.  Exceptions past it are
 *                  dropped and CSF_DEV_ERR_CAPACITY is set; exc_index is
 *                  complete either way, so the caller can re-run with a
 *                  buffer of exc_index[rows] bytes.  E*R*C always suffices.
 *   scratch        device, 8-byte aligned, scratch_bytes long; needs no
 *                  initialisation.  Calls that share a scratch buffer must
 *                  not overlap on the GPU.  csf_sizes().prepare_scratch is
 *                  the size that takes the fastest path; the least accepted
 *                  size is 16 bytes plus 8 per tile of rows (128-row tiles
 *                  for rows of up to 255 bytes).
 * Rows of up to 255 bytes (tiles of 128 rows, one thread per row):
 *   - with at least csf_sizes().prepare_scratch bytes of scratch, and up to
 *     8192 tiles (1 M rows), one pass per tile picks each row's base,
 *     writes the planes, each row's place inside its tile in exc_index and
 *     the tile's exception bytes to its slot in the scratch (128 * C bytes
 *     a tile: the scratch is about the size of the dense stack); a second
 *     kernel adds each tile's offset in the stream (the sum of the earlier
 *     tiles' totals) to the exc_index entries and copies the slots into the
 *     stream;
 *   - with less, two kernels: the first picks the bases and counts the
 *     exceptions (per-tile totals in the scratch), the second places each
 *     tile in the stream from the totals before it and encodes.
 * No block waits on another.  Wider rows take one kernel whose blocks pass
 * exception-count prefixes to later blocks through the scratch (a decoupled
 * look-back, cleared by this call on `stream`); every wait is bounded and
 * sets CSF_DEV_ERR_TIMEOUT rather than hang.
 * Errors: CSF_ERR_ARG (NULL, misaligned planes, dense not in device memory),
 * CSF_ERR_SIZE (scratch smaller than the least accepted size), CSF_ERR_CUDA.
 */
csf_status csf_prepare(const uint8_t *dense, csf_stack *out, uint64_t exc_capacity,
                       void *scratch, size_t scratch_bytes, void *stream);

/* Size of the device scratch array built into the library for
 * csf_prepare_static (held on every GPU that loads the library). */
#define CSF_STATIC_SCRATCH_BYTES (256u * 1024u)

/*
 * csf_prepare without a scratch argument, for callers that cannot allocate
 * device memory.  The pages have no counterpart; this is a convenience of this
 * library.  Some callers cannot call cudaMalloc: a plugin inside a host
 * process whose caching allocator owns all device memory, code that runs
 * where an allocation would implicitly synchronise the device or disturb a
 * stream capture, code with a fixed memory budget.  This entry point
 * allocates nothing: its scratch (the per-tile exception totals of rows up
 * to 255 bytes; a ticket counter and one look-back word per tile of wider
 * rows) is a CSF_STATIC_SCRATCH_BYTES device array inside the library.
 * The caller still passes `dense` and every output buffer, as for csf_prepare,
 * and the results are the same bytes.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it under the id of the current CUDA
 * context; make that first call before any stream capture.  A device reset
 * (cudaDeviceReset) destroys the context and the array with it: the next call
 * runs in a new context and looks the address up again, as a first call.
 * Every call shares the one array (rows wider than 255 bytes clear the part
 * they use on `stream` first): calls that overlap on the GPU race, so order
 * them.
 * Errors: as csf_prepare, plus CSF_ERR_SIZE when the geometry needs more than
 * CSF_STATIC_SCRATCH_BYTES of scratch (16 + 8 bytes per tile of rows; tiles
 * are 128 rows when C <= 255, so about 4 million rows).
 */
csf_status csf_prepare_static(const uint8_t *dense, csf_stack *out, uint64_t exc_capacity, void *stream);

/*
 * Decode a stack into a dense workspace ([FK] format, strategy table and
 * helpers paragraphs).
 *
 *   s              the stack (num_exc set).
 *   ws, ws_bytes   device workspace of at least E*R*C bytes, any byte
 *                  alignment (odd offsets allowed), row-major [E][R][C].
 *   expert_start   NULL: decode every expert.  Else a device array of E+1
 *                  int32 (expert_start_is_int64 == 0) or int64 entries, the
 *                  grouped-routing prefix: expert e is decoded iff
 *                  expert_start[e+1] > expert_start[e]; the workspace planes
 *                  of the other experts are not touched.  The routing is read
 *                  on the device: no host sync, no selection buffer.
 * One kernel launch; no host synchronisation.
 * Errors: CSF_ERR_ARG, CSF_ERR_SIZE (ws_bytes < E*R*C),
 * CSF_ERR_UNSUPPORTED (routed decode with E > 8192), CSF_ERR_CUDA.
 */
csf_status csf_decode(const csf_stack *s, uint8_t *ws, size_t ws_bytes,
                      const void *expert_start, int expert_start_is_int64, void *stream);

/*
 * Decode a gate(/up) stack and a down stack in ONE launch with the same
 * routing ([B478] pairing commit message): same semantics as two csf_decode
 * calls.  The stacks must have the same number of experts; kinds, rows and
 * columns may differ.  Errors as csf_decode, plus CSF_ERR_ARG when the
 * expert counts differ.
 */
csf_status csf_decode_pair(const csf_stack *gate, uint8_t *gate_ws, size_t gate_ws_bytes,
                           const csf_stack *down, uint8_t *down_ws, size_t down_ws_bytes,
                           const void *expert_start, int expert_start_is_int64, void *stream);

/*
 * Workspace layouts of csf_decode_rows and csf_expand.
 *   CSF_LAYOUT_ROWS     row-major [E][R][C], the layout of csf_decode.
 *   CSF_LAYOUT_BLOCKED  the scale-operand layout that Blackwell block-scaled
 *       GEMMs (tcgen05 block scaling, cuBLASLt VEC16_UE4M3 / VEC32_UE8M0
 *       scales) read, written directly so that no layout pass runs before
 *       the GEMM ([FK] measurement paragraph: decode staging before the GEMM
 *       is the cost).  Per expert, its R x C scales padded to RP = R rounded
 *       up to 128 rows and CP = C rounded up to 4 columns, cut into 128 x 4
 *       tiles of 512 bytes; tiles in row-block-major order (column blocks
 *       innermost); scale (r, c) of a tile at byte
 *       (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.  Experts follow each
 *       other, RP * CP bytes apart.  Padding bytes are written 0.  Needs a
 *       16-byte aligned workspace of csf_sizes().blocked bytes and row
 *       ranges on 128-row boundaries (row_hi may also be R).
 */
#define CSF_LAYOUT_ROWS 0
#define CSF_LAYOUT_BLOCKED 1

/* One stack of a csf_decode_rows call and the rows of each expert it writes. */
typedef struct {
    const csf_stack *stack; /* num_exc set */
    uint8_t *ws;            /* device workspace: ROWS >= E*R*C bytes, [E][R][C], any byte alignment;
                               BLOCKED >= csf_sizes().blocked bytes, 16-byte aligned */
    size_t ws_bytes;
    int32_t row_lo;         /* rows row_lo <= r < row_hi of each selected expert are written; */
    int32_t row_hi;         /* 0 <= row_lo < row_hi <= R */
    int32_t layout;         /* CSF_LAYOUT_ROWS or CSF_LAYOUT_BLOCKED; every part of a call alike */
} csf_decode_part;

/*
 * Decode only a range of rows of each expert ([B478] pairing commit message:
 * decode only the gate halves that a fused gate/up consumer reads).  For a
 * fused gate/up stack with R = 2*I rows per expert, the gate half is rows
 * [0, I).  The workspace keeps its whole-stack layout (row-major [E][R][C],
 * or the blocked layout below, chosen per call by `layout`): rows outside the
 * range, and the planes of experts that expert_start leaves inactive, are not
 * touched.  One or two parts (for example the gate half of a gate/up stack
 * and the whole down stack) decode in ONE launch with the same routing.
 *
 *   parts, num_parts  1 or 2 parts; every part must have the same number of
 *                     experts.
 *   expert_start      as csf_decode (NULL: every expert).
 * Errors: CSF_ERR_ARG (bad part count, NULL stack, empty or out-of-range
 * rows, differing expert counts or layouts, an unknown layout, a blocked
 * workspace not 16-byte aligned or rows off its 128-row boundaries, and the
 * csf_decode cases), CSF_ERR_SIZE, CSF_ERR_UNSUPPORTED (E > 8192 with
 * routing, or with a partial row range in the row-major layout: the
 * per-expert work list lives in shared memory), CSF_ERR_CUDA.
 */
csf_status csf_decode_rows(const csf_decode_part *parts, int num_parts,
                           const void *expert_start, int expert_start_is_int64, void *stream);

/*
 * Ahead-of-call expansion ([B477] body and [B478] commit message on
 * expand_scales): expand every expert of one layer's stacks into their shared
 * workspaces before the call that reads them, typically on a side stream
 * while other work (that layer's attention) runs, so the expansion leaves the
 * critical path.  The caller orders the streams; this call takes the two
 * events that do it:
 *
 *   parts, num_parts  as csf_decode_rows; every expert is written (the
 *                     routing is not known yet), rows [row_lo, row_hi) of
 *                     each.
 *   after          optional cudaEvent_t recorded by the previous user of the
 *                  workspaces (the call that read them last); `stream` waits
 *                  for it before the expansion writes.  NULL: no wait.
 *   done           optional cudaEvent_t recorded on `stream` once the
 *                  expansion is complete; the consumer's stream waits for it
 *                  before its first read.  NULL: not recorded.
 *   stream         the (side) stream that runs the expansion.
 * Same bytes as csf_decode_rows with expert_start NULL; no host
 * synchronisation.  Arguments are checked before anything is enqueued.
 * The expansion uses the full persistent grid: it overlaps well with work
 * that leaves SMs idle (latency-bound kernels), not with kernels that fill
 * every SM.
 * Errors: as csf_decode_rows; CSF_ERR_CUDA when the wait or the record fails
 * (a wait may already be enqueued when the launch or the record fails).
 */
csf_status csf_expand(const csf_decode_part *parts, int num_parts, void *after, void *done, void *stream);

/*
 * Tile-packed CSF: a stage-readable form of a CSF stack ([B478] commit message
 * on packed experts prepared from CSF checkpoints, whose scales stay as
 * compressed storage that each GEMM pipeline stage rebuilds in shared memory;
 * the pages give no record layout, so this one is the library's).  The same
 * per-row bases and codes, stored in the order of the block-scaled GEMM scale
 * tiles (CSF_LAYOUT_BLOCKED), so that any 128 x 4 tile decodes on its own with
 * no walk along its rows.  Per expert: nrb = ceil(R/128) row blocks, ncb =
 * ceil(C/4) column blocks, T = nrb * ncb tiles, tile t = rb * ncb + cb.
 *   codes       NVFP4: 256 bytes a tile; position q = 16*b + 4*a + c (row
 *               128*rb + b + 32*a, column 4*cb + c) in byte q/2, even q in the
 *               low nibble; nibble 0..14 = offset, 15 = exception.  MXFP4:
 *               128 bytes a tile, offset bits (bytes 0..63, position q at bit
 *               q%8 of byte q/8) then escape bits (bytes 64..127).  Padding
 *               positions (row >= R or column >= C) code 0.
 *   bases       128 bytes per expert and row block, byte 4*b + a = base of
 *               row 128*rb + b + 32*a (0 past R).
 *   tile_index  E*T + 1 uint32: exclusive prefix of the tiles' exception
 *               counts, the total last.
 *   exc_bytes   each tile's exceptions in position order (num_exc bytes,
 *               readable rounded up to 16).
 * Sizes: csf_sizes().tiled_codes / tiled_bases / tiled_index.
 */
typedef struct {
    csf_geometry g;
    uint8_t *codes;       /* 16-byte aligned */
    uint8_t *bases;       /* 16-byte aligned */
    uint32_t *tile_index;
    uint8_t *exc_bytes;
    uint64_t num_exc;     /* host copy: the CSF stack's num_exc (same exceptions, tile order) */
    uint32_t *error_word; /* optional device word for CSF_DEV_ERR_* bits; may be NULL */
} csf_tiled;

/*
 * Convert a CSF stack to its tile-packed form on the GPU (one kernel, one
 * warp per expert and 128-row block).  A row block's exceptions take the same
 * range of the stream as in the CSF stack, from the CSF index of its first
 * row, so tile_index follows from that index and a running count over the
 * block's tiles.  `exc_capacity` = bytes at dst->exc_bytes (src->num_exc
 * suffices); exceptions past it are dropped and CSF_DEV_ERR_CAPACITY set.  A
 * CSF index that disagrees with the escape codes sets CSF_DEV_ERR_CORRUPT.
 * dst->num_exc is not written (it equals src->num_exc).  The stacks must have
 * the same geometry.
 * Errors: CSF_ERR_ARG (NULL or misaligned buffers, geometries differ),
 * CSF_ERR_UNSUPPORTED (more than 2^32 - 1 exceptions), CSF_ERR_CUDA.
 */
csf_status csf_tiled_pack(const csf_stack *src, csf_tiled *dst, uint64_t exc_capacity, void *stream);

/*
 * Decode a tile-packed stack into the block-scaled GEMM scale layout
 * (CSF_LAYOUT_BLOCKED, same bytes as csf_decode_rows of the CSF stack with
 * that layout); each warp decodes a contiguous range of tiles, one tile at a
 * time, every tile on its own.  ws: 16-byte aligned, csf_sizes().blocked
 * bytes.  expert_start as csf_decode: tiles of inactive experts are not
 * touched.  Errors: CSF_ERR_ARG, CSF_ERR_SIZE, CSF_ERR_UNSUPPORTED (routing
 * with E > 8192), CSF_ERR_CUDA.
 */
csf_status csf_tiled_decode(const csf_tiled *t, uint8_t *ws, size_t ws_bytes,
                            const void *expert_start, int expert_start_is_int64, void *stream);

/*
 * Stage-read check of a tile-packed stack ([B478] commit message on packed
 * experts whose scales each GEMM pipeline stage rebuilds in shared memory):
 * every tile of the selected experts is rebuilt in shared memory by the
 * device decoder of csf_tile.cuh (csf_tile_decode_warp), as a stage would
 * before consuming it, and only a 32-bit checksum per tile is written -- no
 * decoded scales reach global memory.  Checksum of a tile = sum over its 128
 * little-endian 32-bit words w_i, in the CSF_LAYOUT_BLOCKED order of the
 * tile's 512 bytes, of w_i * (2i + 1), modulo 2^32.
 *
 *   sums, sums_count  device array of at least E * T uint32, T = tiles per
 *                     expert (ceil(R/128) * ceil(C/4)); sums[e*T + t].
 *   expert_start      as csf_decode: entries of inactive experts are not
 *                     written.
 * A tile whose index disagrees with its codes sets CSF_DEV_ERR_CORRUPT.
 * Errors: CSF_ERR_ARG, CSF_ERR_SIZE (sums_count < E*T), CSF_ERR_UNSUPPORTED
 * (routing with E > 8192), CSF_ERR_CUDA.
 */
csf_status csf_tiled_checksum(const csf_tiled *t, uint32_t *sums, size_t sums_count, const void *expert_start,
                              int expert_start_is_int64, void *stream);

/*
 * Failure-detection self-test of the prepare's bounded waits, synchronous.
 * Runs the single-pass prepare kernel of wide rows on a small internal stack
 * (512 x 300 NVFP4, 48-row tiles) whose first tile no block ever takes, so
 * the next tiles' decoupled look-backs wait on a status word that nothing
 * writes; with a poll limit of 4096 the waits give up, the kernel finishes,
 * and the device error word of the run is written to *error_word
 * (CSF_DEV_ERR_TIMEOUT expected).
 * Nothing faults or hangs, and the context stays usable.  Allocates and frees
 * its own device memory on its own stream.
 * Errors: CSF_ERR_ARG (NULL), CSF_ERR_CUDA.
 */
csf_status csf_selftest_lookback_timeout(uint32_t *error_word);

#ifdef __cplusplus
}
#endif

#endif /* CSF_H */
