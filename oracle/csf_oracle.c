/*
 * CSF scale-codec oracle: plain, slow, single-threaded CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * It restates, loop by loop, what the following web pages say the method
 * computes (cited by page title and paragraph; the pages have no numbered
 * sections):
 *   [FK]   "finegrained-kernels: decode losslessly compressed NVFP4 scales
 *           (CSF)" -- format paragraph (one base byte per row, most scales as
 *           4-bit offsets from it, the rest in an exception stream, exact
 *           reconstruction); helpers paragraph (decode of the whole stack, or
 *           only of experts with routed tokens, inactive planes untouched).
 *   [B478] "NVFP4-CSF: expand_scales() for ahead-of-call scale expansion
 *           (canonical twin of #477)" -- commit message documenting one-bit
 *           MXFP4 and four-bit NVFP4 offsets from a row base byte.
 *   [V964] "Load native FP4 experts with optional lossless CSF scales" --
 *           encoding plus exception index at preparation time.
 *
 * The pages print no byte layout.  The layout below is the plainest reading
 * consistent with them:
 *   - dense stack: row-major [E][R][C] bytes; a row is one output channel's
 *     C scale bytes; row index = e*R + r; element index i = row*C + c.
 *   - NVFP4: window width w = 14; offsets are a flat nibble stream over all
 *     N = E*R*C elements, element i in byte i>>1, even i in the low nibble;
 *     nibble 0..14 is an offset, nibble 15 marks an exception.
 *   - MXFP4: w = 1; two flat LSB-first bit planes: offset bit and escape bit
 *     (escape bit 1 = exception, its offset bit is written 0).
 *   - base: smallest byte value present in the row whose window
 *     [v, v+w] holds the most of the row's bytes.
 *   - exceptions: bytes outside [base, base+w], appended in row-major order;
 *     exc_index[row] = number of exceptions in earlier rows (length rows+1,
 *     last entry = total).
 *   - decode: dense = base + offset (mod 256), or the exception byte at
 *     exc_index[row] + (number of earlier escapes in the same row).
 *   - routed decode: expert e is active iff start[e+1] > start[e]; planes of
 *     inactive experts are not written.
 *   - row-range decode: only rows [row_lo, row_hi) of each written expert are
 *     written (the gate half of a fused gate/up expert is rows [0, R/2)).
 *   - blocked decode: the same bytes placed in the 128 x 4 tiled scale-operand
 *     layout of block-scaled GEMMs (see blocked_offset), padding written 0.
 *   - tile-packed form: the same bases, codes and exception bytes reordered so
 *     that each 128 x 4 tile of that layout decodes on its own ([B478] commit
 *     message on stage-readable compressed scales; layout in csfo_tiled_pack),
 *     and its decode into the blocked layout.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { CSFO_NVFP4 = 0, CSFO_MXFP4 = 1 };
enum { CSFO_OK = 0, CSFO_ERR_ARG = 1, CSFO_ERR_CAPACITY = 2, CSFO_ERR_CORRUPT = 3 };

/* Width of the offset window: 4-bit offsets 0..14 (15 is the escape code)
 * for NVFP4, 1-bit offsets 0..1 for MXFP4 ([B478] offsets commit message). */
static int window_width(int kind) { return kind == CSFO_NVFP4 ? 14 : 1; }

static unsigned nibble_get(const uint8_t *s, uint64_t i)
{
    return (s[i / 2] >> (4 * (i % 2))) & 0xFu;
}

static void nibble_put(uint8_t *s, uint64_t i, unsigned v)
{
    s[i / 2] = (uint8_t)(s[i / 2] | (v << (4 * (i % 2))));
}

static unsigned bit_get(const uint8_t *s, uint64_t i)
{
    return (s[i / 8] >> (i % 8)) & 1u;
}

static void bit_put(uint8_t *s, uint64_t i, unsigned v)
{
    s[i / 8] = (uint8_t)(s[i / 8] | (v << (i % 8)));
}

/* Byte lengths of the packed streams for one geometry. */
void csfo_stream_bytes(int kind, int64_t E, int64_t R, int64_t C,
                       uint64_t *offsets_bytes, uint64_t *escapes_bytes,
                       uint64_t *base_bytes, uint64_t *index_entries)
{
    uint64_t n = (uint64_t)E * (uint64_t)R * (uint64_t)C;
    uint64_t rows = (uint64_t)E * (uint64_t)R;
    if (kind == CSFO_NVFP4) {
        *offsets_bytes = (n + 1) / 2;
        *escapes_bytes = 0;
    } else {
        *offsets_bytes = (n + 7) / 8;
        *escapes_bytes = (n + 7) / 8;
    }
    *base_bytes = rows;
    *index_entries = rows + 1;
}

/* Base byte of one row ([FK] format paragraph: one base byte per row, most
 * scales as offsets from it).  Reading: the smallest value that occurs in the
 * row among those whose window [v, v+w] covers the most bytes of the row. */
static unsigned choose_base(const uint8_t *x, int64_t C, int w)
{
    uint64_t hist[256];
    memset(hist, 0, sizeof hist);
    for (int64_t c = 0; c < C; ++c)
        hist[x[c]] += 1;
    unsigned best = 0;
    int64_t best_count = -1;
    for (int v = 0; v < 256; ++v) {
        if (hist[v] == 0)
            continue;
        int64_t count = 0;
        for (int u = v; u <= v + w && u < 256; ++u)
            count += (int64_t)hist[u];
        if (count > best_count) {
            best_count = count;
            best = (unsigned)v;
        }
    }
    return best;
}

/*
 * Encode a dense stack ([FK] format paragraph; [V964] encoding plus index).
 * Writes base[rows], offsets (and escapes for MXFP4) -- zeroed here first --,
 * exc_index[rows+1] and up to exc_capacity exception bytes.  *num_exc gets
 * the total.  Returns CSFO_ERR_CAPACITY if the exceptions did not fit.
 */
int csfo_encode(int kind, int64_t E, int64_t R, int64_t C, const uint8_t *dense,
                uint8_t *base, uint8_t *offsets, uint8_t *escapes,
                uint32_t *exc_index, uint8_t *exc_bytes, uint64_t exc_capacity,
                uint64_t *num_exc)
{
    if ((kind != CSFO_NVFP4 && kind != CSFO_MXFP4) || E < 0 || R < 0 || C < 1)
        return CSFO_ERR_ARG;
    uint64_t ob, eb, bb, ie;
    csfo_stream_bytes(kind, E, R, C, &ob, &eb, &bb, &ie);
    memset(offsets, 0, ob);
    if (kind == CSFO_MXFP4)
        memset(escapes, 0, eb);
    int w = window_width(kind);
    uint64_t rows = (uint64_t)E * (uint64_t)R;
    uint64_t total = 0;
    int status = CSFO_OK;
    for (uint64_t row = 0; row < rows; ++row) {
        const uint8_t *x = dense + row * (uint64_t)C;
        unsigned b = choose_base(x, C, w);
        base[row] = (uint8_t)b;
        if (total > 0xFFFFFFFFull)
            return CSFO_ERR_ARG;
        exc_index[row] = (uint32_t)total;
        for (int64_t c = 0; c < C; ++c) {
            uint64_t i = row * (uint64_t)C + (uint64_t)c;
            int d = (int)x[c] - (int)b;
            int inside = d >= 0 && d <= w;
            if (kind == CSFO_NVFP4) {
                nibble_put(offsets, i, inside ? (unsigned)d : 0xFu);
            } else {
                bit_put(offsets, i, inside ? (unsigned)d : 0u);
                bit_put(escapes, i, inside ? 0u : 1u);
            }
            if (!inside) {
                if (total < exc_capacity)
                    exc_bytes[total] = x[c];
                else
                    status = CSFO_ERR_CAPACITY;
                total += 1;
            }
        }
    }
    if (total > 0xFFFFFFFFull)
        return CSFO_ERR_ARG;
    exc_index[rows] = (uint32_t)total;
    *num_exc = total;
    return status;
}

/* Escape test of element i ([FK] exception stream; [B478] offsets). */
static int is_escape(int kind, const uint8_t *offsets, const uint8_t *escapes, uint64_t i)
{
    if (kind == CSFO_NVFP4)
        return nibble_get(offsets, i) == 0xFu;
    return bit_get(escapes, i) == 1u;
}

static unsigned offset_of(int kind, const uint8_t *offsets, uint64_t i)
{
    if (kind == CSFO_NVFP4)
        return nibble_get(offsets, i);
    return bit_get(offsets, i);
}

/*
 * Decode one row (global row index `row`) into out_row[0..C) ([FK] format
 * paragraph): base + offset mod 256, or the next exception byte of the row.
 * An exception reference past num_exc writes 0 and returns CSFO_ERR_CORRUPT.
 */
static int decode_row(int kind, int64_t C, const uint8_t *base, const uint8_t *offsets,
                      const uint8_t *escapes, const uint32_t *exc_index, const uint8_t *exc_bytes,
                      uint64_t num_exc, uint64_t row, uint8_t *out_row)
{
    int status = CSFO_OK;
    uint64_t rank = 0;
    for (int64_t c = 0; c < C; ++c) {
        uint64_t i = row * (uint64_t)C + (uint64_t)c;
        if (is_escape(kind, offsets, escapes, i)) {
            uint64_t pos = (uint64_t)exc_index[row] + rank;
            rank += 1;
            if (pos < num_exc) {
                out_row[c] = exc_bytes[pos];
            } else {
                out_row[c] = 0;
                status = CSFO_ERR_CORRUPT;
            }
        } else {
            out_row[c] = (uint8_t)((base[row] + offset_of(kind, offsets, i)) & 0xFFu);
        }
    }
    return status;
}

/*
 * Decode ([FK] format and helpers paragraphs).  expert_start is NULL for the
 * whole stack, else E+1 int64 entries; only experts with start[e+1] > start[e]
 * are written.  Within each written expert only rows row_lo <= r < row_hi are
 * written ([B478] pairing commit message: decode only the gate half that a
 * fused gate/up consumer reads; 0 and R give every row).  An exception
 * reference past num_exc writes 0 and returns CSFO_ERR_CORRUPT.
 */
int csfo_decode(int kind, int64_t E, int64_t R, int64_t C,
                const uint8_t *base, const uint8_t *offsets, const uint8_t *escapes,
                const uint32_t *exc_index, const uint8_t *exc_bytes, uint64_t num_exc,
                const int64_t *expert_start, int64_t row_lo, int64_t row_hi, uint8_t *out)
{
    if ((kind != CSFO_NVFP4 && kind != CSFO_MXFP4) || E < 0 || R < 0 || C < 1)
        return CSFO_ERR_ARG;
    if (row_lo < 0 || row_hi > R || row_lo > row_hi)
        return CSFO_ERR_ARG;
    int status = CSFO_OK;
    for (int64_t e = 0; e < E; ++e) {
        if (expert_start != NULL && !(expert_start[e + 1] > expert_start[e]))
            continue;
        for (int64_t r = row_lo; r < row_hi; ++r) {
            uint64_t row = (uint64_t)e * (uint64_t)R + (uint64_t)r;
            if (decode_row(kind, C, base, offsets, escapes, exc_index, exc_bytes, num_exc, row,
                           out + row * (uint64_t)C) != CSFO_OK)
                status = CSFO_ERR_CORRUPT;
        }
    }
    return status;
}

/*
 * Byte position of scale (r, c) of expert e in the scale-operand layout of
 * Blackwell block-scaled GEMMs (the 128 x 4 tiled layout NVIDIA documents for
 * cuBLASLt block scaling, "32_4_4" swizzle).  Each expert's R x C scale
 * matrix is padded to RP = R rounded up to 128 rows and CP = C rounded up to
 * 4 columns and cut into 128 x 4 tiles of 512 bytes, stored row-block by
 * row-block, column blocks innermost.  Inside a tile, the 16-byte line
 * r % 32 holds rows r % 32, +32, +64, +96, four columns each:
 *   offset = (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.
 * Experts follow each other, RP * CP bytes apart.
 */
static uint64_t blocked_offset(int64_t R, int64_t C, int64_t e, int64_t r, int64_t c)
{
    uint64_t RP = (uint64_t)((R + 127) / 128) * 128;
    uint64_t CP = (uint64_t)((C + 3) / 4) * 4;
    uint64_t tile = (uint64_t)(r / 128) * (CP / 4) + (uint64_t)(c / 4);
    return (uint64_t)e * RP * CP + tile * 512 + (uint64_t)(r % 32) * 16 + (uint64_t)((r % 128) / 32) * 4
           + (uint64_t)(c % 4);
}

/* Bytes of one stack in the scale-operand layout. */
uint64_t csfo_blocked_bytes(int64_t E, int64_t R, int64_t C)
{
    return (uint64_t)E * (uint64_t)((R + 127) / 128) * 128 * (uint64_t)((C + 3) / 4) * 4;
}

/*
 * Decode straight into the scale-operand layout (the decode-into-the-GEMM's
 * operand idea of the [FK] measurement paragraph, which puts the staging cost
 * of a separate layout pass before the GEMM).  Writes every tile of the
 * 128-row blocks that cover rows [row_lo, row_hi) of each selected expert:
 * row_lo must be a multiple of 128 and row_hi a multiple of 128 or R.  Tile
 * positions past the expert's rows or columns (the padding) are written 0.
 * Other tiles, and inactive experts, are left alone.
 */
int csfo_decode_blocked(int kind, int64_t E, int64_t R, int64_t C,
                        const uint8_t *base, const uint8_t *offsets, const uint8_t *escapes,
                        const uint32_t *exc_index, const uint8_t *exc_bytes, uint64_t num_exc,
                        const int64_t *expert_start, int64_t row_lo, int64_t row_hi, uint8_t *out)
{
    if ((kind != CSFO_NVFP4 && kind != CSFO_MXFP4) || E < 0 || R < 1 || C < 1)
        return CSFO_ERR_ARG;
    if (row_lo < 0 || row_hi > R || row_lo >= row_hi || row_lo % 128 != 0 || (row_hi % 128 != 0 && row_hi != R))
        return CSFO_ERR_ARG;
    uint8_t *row_bytes = (uint8_t *)malloc((size_t)C);
    if (!row_bytes)
        return CSFO_ERR_ARG;
    int64_t CP = (C + 3) / 4 * 4;
    int64_t r_end = (row_hi + 127) / 128 * 128;
    int status = CSFO_OK;
    for (int64_t e = 0; e < E; ++e) {
        if (expert_start != NULL && !(expert_start[e + 1] > expert_start[e]))
            continue;
        for (int64_t r = row_lo; r < r_end; ++r) {
            if (r < R) {
                uint64_t row = (uint64_t)e * (uint64_t)R + (uint64_t)r;
                if (decode_row(kind, C, base, offsets, escapes, exc_index, exc_bytes, num_exc, row,
                               row_bytes) != CSFO_OK)
                    status = CSFO_ERR_CORRUPT;
            }
            for (int64_t c = 0; c < CP; ++c)
                out[blocked_offset(R, C, e, r, c)] = (r < R && c < C) ? row_bytes[c] : 0;
        }
    }
    free(row_bytes);
    return status;
}

/*
 * Tile-packed CSF: the same per-row bases and codes, stored in the order of
 * the block-scaled GEMM scale layout so that any 128 x 4 tile decodes on its
 * own (the stage-readable packed storage that the expand_scales commit
 * message describes for pipeline stages; its layout is not on the pages, so
 * this one is a design of this library).  Per expert, tiles as in
 * blocked_offset: tile t = row block rb * (CP/4) + column block cb.  Inside a
 * tile, position q = 16*b + 4*a + c (line b, row r = 128*rb + b + 32*a,
 * column 4*cb + c), the same order as the tile's bytes in the blocked layout.
 *   codes   NVFP4: 256 bytes per tile, position q in byte q/2 (even q in the
 *           low nibble), nibble = offset 0..14 or 15 for an exception.
 *           MXFP4: 128 bytes per tile, an offset bit plane (bytes 0..63,
 *           position q at bit q%8 of byte q/8) then an escape bit plane
 *           (bytes 64..127).  Padding positions (r >= R or c >= C) code 0.
 *   bases   128 bytes per row block, byte 4*b + a = base of row
 *           128*rb + b + 32*a (0 for padding rows).
 *   tile_index  E*T + 1 u32: exclusive prefix of the tiles' exception counts.
 *   exc_bytes   each tile's exceptions in position order.
 * Packed from a CSF stack: decoded first, then every position recoded against
 * its row's base, so the codes equal the CSF codes of the same elements.
 */
uint64_t csfo_tiled_code_bytes(int kind, int64_t E, int64_t R, int64_t C)
{
    uint64_t T = (uint64_t)((R + 127) / 128) * (uint64_t)((C + 3) / 4);
    return (uint64_t)E * T * (kind == CSFO_NVFP4 ? 256u : 128u);
}

int csfo_tiled_pack(int kind, int64_t E, int64_t R, int64_t C,
                    const uint8_t *base, const uint8_t *offsets, const uint8_t *escapes,
                    const uint32_t *exc_index, const uint8_t *exc_bytes, uint64_t num_exc,
                    uint8_t *codes, uint8_t *bases, uint32_t *tile_index, uint8_t *t_exc,
                    uint64_t t_exc_capacity, uint64_t *t_num_exc)
{
    if ((kind != CSFO_NVFP4 && kind != CSFO_MXFP4) || E < 1 || R < 1 || C < 1)
        return CSFO_ERR_ARG;
    int w = window_width(kind);
    int64_t nrb = (R + 127) / 128, ncb = (C + 3) / 4;
    uint64_t per_tile = kind == CSFO_NVFP4 ? 256u : 128u;
    uint8_t *dense = (uint8_t *)malloc((size_t)(E * R * C));
    if (!dense)
        return CSFO_ERR_ARG;
    int status = csfo_decode(kind, E, R, C, base, offsets, escapes, exc_index, exc_bytes, num_exc, NULL, 0, R,
                             dense);
    memset(codes, 0, (size_t)csfo_tiled_code_bytes(kind, E, R, C));
    memset(bases, 0, (size_t)(E * nrb * 128));
    uint64_t n = 0;        /* exceptions written so far */
    uint64_t tile = 0;
    for (int64_t e = 0; e < E; ++e) {
        for (int64_t rb = 0; rb < nrb; ++rb) {
            for (int64_t b = 0; b < 32; ++b)
                for (int64_t a = 0; a < 4; ++a) {
                    int64_t r = 128 * rb + b + 32 * a;
                    if (r < R)
                        bases[(e * nrb + rb) * 128 + 4 * b + a] = base[e * R + r];
                }
            for (int64_t cb = 0; cb < ncb; ++cb, ++tile) {
                tile_index[tile] = (uint32_t)n;
                uint8_t *tc = codes + tile * per_tile;
                for (int64_t q = 0; q < 512; ++q) {
                    int64_t b = q / 16, a = (q / 4) % 4, c = 4 * cb + q % 4;
                    int64_t r = 128 * rb + b + 32 * a;
                    if (r >= R || c >= C)
                        continue;                          /* padding: code 0 */
                    uint64_t row = (uint64_t)e * (uint64_t)R + (uint64_t)r;
                    unsigned v = dense[row * (uint64_t)C + (uint64_t)c], bs = base[row];
                    int inside = v >= bs && v - bs <= (unsigned)w;
                    if (!inside) {
                        if (n < t_exc_capacity)
                            t_exc[n] = (uint8_t)v;
                        else
                            status = CSFO_ERR_CAPACITY;
                        n += 1;
                    }
                    if (kind == CSFO_NVFP4) {
                        nibble_put(tc, (uint64_t)q, inside ? v - bs : 15u);
                    } else {
                        bit_put(tc, (uint64_t)q, inside ? v - bs : 0u);
                        bit_put(tc + 64, (uint64_t)q, inside ? 0u : 1u);
                    }
                }
            }
        }
    }
    tile_index[tile] = (uint32_t)n;
    *t_num_exc = n;
    free(dense);
    return status;
}

/*
 * Decode a tile-packed stack into the block-scaled GEMM scale layout (same
 * bytes as csfo_decode_blocked of the CSF stack it was packed from).
 * expert_start as in csfo_decode.  An exception reference past num_exc
 * writes 0 and returns CSFO_ERR_CORRUPT.
 */
int csfo_tiled_decode(int kind, int64_t E, int64_t R, int64_t C,
                      const uint8_t *codes, const uint8_t *bases, const uint32_t *tile_index,
                      const uint8_t *t_exc, uint64_t num_exc, const int64_t *expert_start, uint8_t *out)
{
    if ((kind != CSFO_NVFP4 && kind != CSFO_MXFP4) || E < 1 || R < 1 || C < 1)
        return CSFO_ERR_ARG;
    int64_t nrb = (R + 127) / 128, ncb = (C + 3) / 4;
    uint64_t per_tile = kind == CSFO_NVFP4 ? 256u : 128u;
    int status = CSFO_OK;
    for (int64_t e = 0; e < E; ++e) {
        if (expert_start != NULL && !(expert_start[e + 1] > expert_start[e]))
            continue;
        for (int64_t rb = 0; rb < nrb; ++rb) {
            for (int64_t cb = 0; cb < ncb; ++cb) {
                uint64_t tile = ((uint64_t)e * (uint64_t)nrb + (uint64_t)rb) * (uint64_t)ncb + (uint64_t)cb;
                const uint8_t *tc = codes + tile * per_tile;
                uint64_t k = tile_index[tile];
                for (int64_t q = 0; q < 512; ++q) {
                    int64_t b = q / 16, a = (q / 4) % 4, c = 4 * cb + q % 4;
                    int64_t r = 128 * rb + b + 32 * a;
                    uint8_t v = 0;
                    int esc = kind == CSFO_NVFP4 ? nibble_get(tc, (uint64_t)q) == 15u
                                                 : bit_get(tc + 64, (uint64_t)q) == 1u;
                    if (esc) {
                        if (k < num_exc) {
                            v = t_exc[k];
                        } else {
                            status = CSFO_ERR_CORRUPT;
                        }
                        k += 1;
                    } else {
                        unsigned off = kind == CSFO_NVFP4 ? nibble_get(tc, (uint64_t)q) : bit_get(tc, (uint64_t)q);
                        v = (uint8_t)((bases[(e * nrb + rb) * 128 + 4 * b + a] + off) & 0xFFu);
                    }
                    out[blocked_offset(R, C, e, r, c)] = (r < R && c < C) ? v : 0;
                }
                if (k != tile_index[tile + 1])
                    status = CSFO_ERR_CORRUPT;
            }
        }
    }
    return status;
}

/*
 * Well-formedness of a stack's index: exc_index[0] == 0, each row's index
 * step equals the number of escapes in that row, and the last entry equals
 * num_exc.  Returns CSFO_OK or CSFO_ERR_CORRUPT.
 */
int csfo_check(int kind, int64_t E, int64_t R, int64_t C,
               const uint8_t *offsets, const uint8_t *escapes,
               const uint32_t *exc_index, uint64_t num_exc)
{
    if ((kind != CSFO_NVFP4 && kind != CSFO_MXFP4) || E < 0 || R < 0 || C < 1)
        return CSFO_ERR_ARG;
    uint64_t rows = (uint64_t)E * (uint64_t)R;
    if (exc_index[0] != 0)
        return CSFO_ERR_CORRUPT;
    for (uint64_t row = 0; row < rows; ++row) {
        uint64_t count = 0;
        for (int64_t c = 0; c < C; ++c)
            count += (uint64_t)is_escape(kind, offsets, escapes, row * (uint64_t)C + (uint64_t)c);
        if ((uint64_t)exc_index[row + 1] != (uint64_t)exc_index[row] + count)
            return CSFO_ERR_CORRUPT;
    }
    if ((uint64_t)exc_index[rows] != num_exc)
        return CSFO_ERR_CORRUPT;
    return CSFO_OK;
}
