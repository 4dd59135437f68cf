// CSF decode kernel for sm_103a: rebuilds dense FP8 scale bytes from a
// compressed stack, row-major, for the whole stack or only for routed
// experts, for every row of an expert or only a row range (the gate half of a
// fused gate/up expert), and for one stack or a gate/down pair in the same
// launch.  (csf_tiles.cu writes the tiled scale-operand layout instead.)
//
// Pages followed (cited by title and paragraph; they have no numbered
// sections):
//   "finegrained-kernels: decode losslessly compressed NVFP4 scales (CSF)":
//     format paragraph (base byte per row, 4-bit offsets, exception stream,
//     exact bytes); helpers paragraph (a fixed-stream pass and an exception
//     pass that both skip experts without routed tokens, leaving their
//     workspace planes untouched, with no selection buffer and no CPU sync);
//     measurement paragraph (contiguous work instead of padded row tiles).
//   "NVFP4-CSF: expand_scales() for ahead-of-call scale expansion (canonical
//     twin of #477)": commit messages on one-bit MXFP4 / four-bit NVFP4
//     offsets, on pairing gate/up and down scales without extra streams,
//     on both routing integer types, on decoding only the gate halves a
//     consumer reads, and on vectorised indexed reconstruction and
//     exception lookup.
//
// Design (GB300 first; HBM-bound byte work, no tensor cores):
//   * Work unit = a run of `rb` rows whose elements fill whole lane chunks
//     (64 elements = 32 offset bytes for NVFP4; 128 elements = 16 bytes of
//     each bit plane for MXFP4).  Every warp of a persistent grid takes one
//     contiguous range of units (balanced to one unit), reads one exc_index
//     entry where each contiguous segment starts, and walks the exception
//     stream in order: exceptions of consecutive rows are consecutive, so an
//     escape's position is the segment's first index plus the escapes before
//     it (a warp scan of per-lane popcounts).  The index entry at the segment
//     end is checked against the running position.
//   * Lanes read 256-bit pieces of the offset stream (coalesced across the
//     warp), prefetching the next piece while the current one is expanded
//     with byte permutes (NVFP4) or a bit-to-byte spreading multiply (MXFP4)
//     and the row bases added byte by byte.  A segment whose bases cannot
//     carry out of a byte, with row boundaries on word boundaries, runs a
//     loop instance that holds only the word-wise expansion (one base select
//     and a plain 32-bit add per word); other segments run the general loop.
//     Chunks spanning three rows (32 <= C < 64) take each word's bases with
//     one byte permute of the three packed bases.
//   * Escapes are patched in a lane-private, bank-swizzled shared-memory slot
//     (one byte store each); each 32 dense bytes leave with one 256-bit store.
//   * Per-expert mode (routing and/or row ranges): every block compacts the
//     active experts of `expert_start` (all experts without it) into shared
//     memory with ballots and prefix sums, each with the units that hold its
//     rows [r_lo, r_hi); units of inactive experts and of rows outside the
//     range never exist, so those workspace bytes are never written.  With a
//     partial row range every expert gets whole warps.
//   * The kernel is instantiated per kind (NVFP4, MXFP4, or both for a
//     mixed pair), so a launch carries only the decoders it uses.
//   * A unit whose rows straddle an expert or range boundary (R*C not a
//     multiple of the lane chunk) is decoded whole but stored only inside the
//     selected rows.
#include <type_traits>

#include "csf_device.cuh"
#include "csf_internal.cuh"

namespace csfk {
namespace {

using dev::add_base;
using dev::flag;
using dev::kFull;
using dev::lanemask_lt;

constexpr int kStageBytes = 4096;   // per warp: 32 lanes x 128 bytes

// Exclusive warp prefix sum of v (and the warp total).  Each step's shuffle
// also yields whether the source lane exists (PTX shfl.sync.up's predicate),
// which guards the add: no lane-index compare per step.
template <int D>
__device__ __forceinline__ void scan_step(uint32_t &x) {
    asm("{\n .reg .b32 y;\n .reg .pred p;\n shfl.sync.up.b32 y|p, %0, %1, 0, -1;\n @p add.u32 %0, %0, y;\n}"
        : "+r"(x)
        : "n"(D));
}
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, int lane, uint32_t &total) {
    (void)lane;
    uint32_t x = v;
    scan_step<1>(x);
    scan_step<2>(x);
    scan_step<4>(x);
    scan_step<8>(x);
    scan_step<16>(x);
    total = __shfl_sync(kFull, x, 31);
    return x - v;
}

__device__ __forceinline__ void ld_v8(const uint8_t *p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                   "=r"(w[7])
                 : "l"(p));
}

__device__ __forceinline__ void st_v8(uint8_t *p, const uint32_t *w) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Store 32 decoded bytes of local elements [p, p+32) at ws + p, keeping only
// the bytes inside [lo, hi).  `align` = byte alignment of ws (p % 32 == 0).
__device__ __forceinline__ void store32(uint8_t *ws, int align, uint32_t p, const uint32_t *w, uint32_t lo,
                                        uint32_t hi) {
    uint8_t *d = ws + p;
    if (p >= lo && p + 32 <= hi) {
        if (align >= 32) {
            st_v8(d, w);
        } else if (align >= 16) {
            reinterpret_cast<uint4 *>(d)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4 *>(d)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else if (align >= 4) {
#pragma unroll
            for (int k = 0; k < 8; ++k) reinterpret_cast<uint32_t *>(d)[k] = w[k];
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) d[j] = (uint8_t)(w[j >> 2] >> (8 * (j & 3)));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t q = p + j;
            if (q >= lo && q < hi) d[j] = (uint8_t)(w[j >> 2] >> (8 * (j & 3)));
        }
    }
}

__device__ __forceinline__ void sts_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void sts_u8(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Shared-memory twin of store32: local elements [p, p+32) at shared address
// sa0 + p (16-byte aligned), only the bytes inside [lo, hi).
__device__ __forceinline__ void sstore32(uint32_t sa0, uint32_t p, const uint32_t *w, uint32_t lo, uint32_t hi) {
    const uint32_t a = sa0 + p;
    if (p >= lo && p + 32 <= hi) {
        sts_v4(a, w[0], w[1], w[2], w[3]);
        sts_v4(a + 16, w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t q = p + j;
            if (q >= lo && q < hi) sts_u8(a + j, (w[j >> 2] >> (8 * (j & 3))) & 0xFFu);
        }
    }
}

// Mask of the bytes of word k (elements 4k..4k+3 of a run) that lie at or
// after element b of the run.
__device__ __forceinline__ uint32_t bytes_from(int b, int k) {
    const uint32_t s = (uint32_t)max(8 * (b - 4 * k), 0);
    return __funnelshift_lc(0u, 0xFFFFFFFFu, s);   // shift >= 32 gives 0
}

// Escape flags of the 8 elements of one offset word, in element order in
// bits 0..7 (higher bits are garbage).  lo4 / hi4 hold the even / odd
// elements' nibbles as bytes; nibble 15 + 1 carries into bit 4 of its byte.
__device__ __forceinline__ uint32_t escape_flags8(uint32_t lo4, uint32_t hi4) {
    const uint32_t zl = (lo4 + 0x01010101u) & 0x10101010u;   // element 2m -> bit 8m+4
    const uint32_t zh = (hi4 + 0x01010101u) & 0x10101010u;   // element 2m+1 -> bit 8m+4
    // bits 8m+4 / 8m+5 -> bits 2m / 2m+1 of the high product word
    return __umulhi(zl + 2u * zh, 0x10410400u);
}

// Replicated row bases for NW words (4*NW elements) starting at a run whose
// first row has base `first`; `b` = elements to the next row start; rows after
// the first are read from base[rn], base[rn+1], ... (rn = that next row).
template <int NW>
__device__ __forceinline__ void base_words_general(uint32_t (&bw)[NW], uint32_t first, int b,
                                                   const uint8_t *__restrict__ base, uint64_t rn, uint64_t rows,
                                                   uint32_t C) {
    const uint32_t a = first * 0x01010101u;
#pragma unroll
    for (int k = 0; k < NW; ++k) bw[k] = a;
    while (b < 4 * NW) {
        const uint32_t nb = (rn < rows ? (uint32_t)__ldg(base + rn) : 0u) * 0x01010101u;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const uint32_t m = bytes_from(b, k);
            bw[k] = (bw[k] & ~m) | (nb & m);
        }
        b += (int)C;
        ++rn;
    }
}

// ------------------------------------------------------------------ NVFP4

// True when rows [row_a, row_b) can take the word-wise expansion: C a multiple
// of 4 and at least one lane chunk (so a chunk holds at most one row boundary,
// on a word boundary), and no base above `limit` (240 for NVFP4, 254 for
// MXFP4: base + largest code <= 255, so a plain 32-bit add cannot carry from
// one byte into the next).  Whole warp; the bases are read again by the decode
// itself, from L1.
__device__ __forceinline__ bool words_case(const DecStack &S, uint64_t row_a, uint64_t row_b, int lane, int chunk,
                                           uint32_t limit) {
    if ((S.C & 3) != 0 || S.C < chunk) return false;
    // The decode also reads the base of the row after a chunk's last row
    // (row_b, when it exists): include it.
    const uint64_t end = min(row_b + 1, (uint64_t)S.rows);
    bool high = false;
    for (uint64_t r = row_a + (uint64_t)lane; r < end; r += 32) high |= __ldg(S.base + r) > limit;
    return !__any_sync(kFull, high);
}

// Decode rows [row_a, row_b) of an NVFP4 stack (row_a*C a multiple of 64),
// storing only global elements in [lo, hi).  Whole warp.  SMEM: the bytes go
// to shared memory instead, element row_a*C + p at shared address sdst + p
// (16-byte aligned for p % 32 == 0), and exceptions are patched there in
// place (no staging); `stage` is then unused.  The loop is compiled twice:
// once with only the word-wise expansion, taken when words_case() holds for
// the segment, and once general; WORDS_OK = false (no stack of the launch
// can take the word-wise loop) compiles the general loop alone.
template <bool SMEM, bool WORDS_OK>
__device__ void segment_nvfp4(const DecStack &S, uint64_t row_a, uint64_t row_b, uint64_t lo, uint64_t hi,
                              int lane, uint8_t *stage, uint32_t sdst) {
    const uint32_t C = (uint32_t)S.C;
    const uint64_t sa = row_a * C;
    const uint32_t nel = (uint32_t)(row_b * C - sa);
    const uint32_t nch = (nel + kLaneNv - 1) / kLaneNv;
    const uint8_t *offs = S.offsets + sa / 2;
    const uint64_t avail64 = S.off_bytes - sa / 2;
    const uint32_t avail = avail64 > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)avail64;
    const uint8_t *bases = S.base + row_a;
    const uint64_t rows_left = S.rows - row_a;
    uint8_t *ws = S.ws + sa;
    const uint32_t lo_l = (uint32_t)(lo - sa);
    const uint32_t hi_l = (uint32_t)(hi - sa);
    const bool fast = lo_l == 0 && hi_l == nel && S.ws_align >= 32;
    const bool v8ok = S.off_align32 != 0;
    const uint32_t nexc = (uint32_t)S.num_exc;
    bool bad = false;
    const uint32_t gs = (((uint32_t)lane >> 1) & 3u) << 4;   // 16-byte slot swizzle (bank spread)
    uint8_t *my = stage + lane * 64;

    uint32_t rr = ((uint32_t)lane * kLaneNv) / C;
    uint32_t q = ((uint32_t)lane * kLaneNv) % C;
    uint32_t w[8], bA = 0, bB = 0, bD = 0;

    // chunks below nch8 are whole 32-byte pieces that one 256-bit load reads
    const uint32_t nch8 = v8ok ? min(nch, avail / 32) : 0u;
    auto load = [&](uint32_t c, uint32_t r) {
        if (c < nch) {
            const uint8_t *p = offs + (size_t)c * 32;
            if (c < nch8) {
                ld_v8(p, w);
            } else {
                const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
                w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
                if (c * 32 + 32 <= avail) {
                    const uint4 b2 = __ldg(reinterpret_cast<const uint4 *>(p + 16));
                    w[4] = b2.x; w[5] = b2.y; w[6] = b2.z; w[7] = b2.w;
                } else {
                    w[4] = w[5] = w[6] = w[7] = 0;
                }
            }
            bA = __ldg(bases + r);
            bB = (r + 1 < rows_left) ? (uint32_t)__ldg(bases + r + 1) : 0u;
            if (C < kLaneNv) bD = (r + 2 < rows_left) ? (uint32_t)__ldg(bases + r + 2) : 0u;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0;
            bA = bB = bD = 0;
        }
    };
    load((uint32_t)lane, rr);
    // The index entries at both ends of the segment travel with the first
    // piece: one memory round trip before the first expand.  Lane 1 keeps the
    // end entry for the final check.
    uint32_t X = 0, Xend = 0;
    if (lane == 0) X = __ldg(S.exc_index + row_a);
    if (lane == 1) Xend = __ldg(S.exc_index + row_b);
    // The base check's loads leave together with the first piece as well.
    const bool words = WORDS_OK && words_case(S, row_a, row_b, lane, kLaneNv, 240u);
    X = __shfl_sync(kFull, X, 0);

    auto run = [&](auto words_tag) {
        constexpr bool WORDS = decltype(words_tag)::value;
        for (uint32_t cb = 0; cb < nch; cb += 32) {
            const uint32_t cc = cb + lane;
            // this step's piece and bases, read in place: the next piece is
            // loaded into the same registers once the expansion has used them
            const uint32_t(&cw)[8] = w;
            const uint32_t &cA = bA, &cB = bB, &cD = bD, &cq = q, &crr = rr;

            const uint32_t p = cc * kLaneNv;
            const int nv = cc < nch ? (int)min(nel - p, (uint32_t)kLaneNv) : 0;
            const int b = (int)(C - cq);                           // elements to the next row start
            uint32_t out[16], fl[8];
            if constexpr (WORDS) {
                // Row boundaries fall on whole words and base + 15 <= 255 for every
                // row of the segment: one base select and a plain add per word.
                const uint32_t A = cA * 0x01010101u, B = cB * 0x01010101u;
                const int kb = b >> 2;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t x = cw[i];
                    const uint32_t lo4 = x & 0x0F0F0F0Fu, hi4 = (x >> 4) & 0x0F0F0F0Fu;
                    fl[i] = escape_flags8(lo4, hi4);
                    out[2 * i] = (2 * i >= kb ? B : A) + __byte_perm(lo4, hi4, 0x5140);
                    out[2 * i + 1] = (2 * i + 1 >= kb ? B : A) + __byte_perm(lo4, hi4, 0x7362);
                }
            } else if (C >= kLaneNv) {
                // At most one row boundary in the 64 elements: bytes at or after
                // element b take row B's base.
                const uint32_t A = cA * 0x01010101u, B = cB * 0x01010101u;
                if (cA <= 240u && cB <= 240u && (C & 3u) == 0) {
                    // Row boundaries fall on whole words (C % 4 == 0) and base + 15
                    // <= 255 (a plain add cannot carry between bytes).
                    const int kb = b >> 2;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t x = cw[i];
                        const uint32_t lo4 = x & 0x0F0F0F0Fu, hi4 = (x >> 4) & 0x0F0F0F0Fu;
                        fl[i] = escape_flags8(lo4, hi4);
                        out[2 * i] = (2 * i >= kb ? B : A) + __byte_perm(lo4, hi4, 0x5140);
                        out[2 * i + 1] = (2 * i + 1 >= kb ? B : A) + __byte_perm(lo4, hi4, 0x7362);
                    }
                } else if (cA <= 240u && cB <= 240u) {
                    // base + 15 <= 255: a plain add cannot carry between bytes.
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t x = cw[i];
                        const uint32_t lo4 = x & 0x0F0F0F0Fu, hi4 = (x >> 4) & 0x0F0F0F0Fu;
                        fl[i] = escape_flags8(lo4, hi4);
                        const uint32_t m0 = bytes_from(b, 2 * i), m1 = bytes_from(b, 2 * i + 1);
                        out[2 * i] = ((A & ~m0) | (B & m0)) + __byte_perm(lo4, hi4, 0x5140);
                        out[2 * i + 1] = ((A & ~m1) | (B & m1)) + __byte_perm(lo4, hi4, 0x7362);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t x = cw[i];
                        const uint32_t lo4 = x & 0x0F0F0F0Fu, hi4 = (x >> 4) & 0x0F0F0F0Fu;
                        fl[i] = escape_flags8(lo4, hi4);
                        const uint32_t m0 = bytes_from(b, 2 * i), m1 = bytes_from(b, 2 * i + 1);
                        out[2 * i] = add_base((A & ~m0) | (B & m0), __byte_perm(lo4, hi4, 0x5140));
                        out[2 * i + 1] = add_base((A & ~m1) | (B & m1), __byte_perm(lo4, hi4, 0x7362));
                    }
                }
            } else if (C >= 32) {
                // At most two row boundaries in the 64 elements (at b and b + C).
                // The three row bases sit in bytes 0..2 of P3.  For 8 elements
                // at a time, nibble j of `rows` is the row (0, 1 or 2) of
                // element j: a 1 from each boundary at or before it, as clamped
                // funnel shifts of 0x11111111; a byte permute of P3 by it gives
                // a word's four bases.
                const uint32_t P3 = cA | (cB << 8) | (cD << 16);
                const int s1 = 4 * b, s2 = 4 * (b + (int)C);
                // One branch per chunk (bases above 240 are rare): plain adds,
                // or carry-free byte adds.
                auto two_rows = [&](auto plain) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t x = cw[i];
                        const uint32_t lo4 = x & 0x0F0F0F0Fu, hi4 = (x >> 4) & 0x0F0F0F0Fu;
                        fl[i] = escape_flags8(lo4, hi4);
                        const uint32_t rows = __funnelshift_lc(0u, 0x11111111u, (uint32_t)max(s1 - 32 * i, 0)) +
                                              __funnelshift_lc(0u, 0x11111111u, (uint32_t)max(s2 - 32 * i, 0));
                        const uint32_t bw0 = __byte_perm(P3, 0, rows), bw1 = __byte_perm(P3, 0, rows >> 16);
                        const uint32_t o0 = __byte_perm(lo4, hi4, 0x5140), o1 = __byte_perm(lo4, hi4, 0x7362);
                        out[2 * i] = decltype(plain)::value ? bw0 + o0 : add_base(bw0, o0);
                        out[2 * i + 1] = decltype(plain)::value ? bw1 + o1 : add_base(bw1, o1);
                    }
                };
                if (cA <= 240u && cB <= 240u && cD <= 240u)
                    two_rows(std::true_type{});
                else
                    two_rows(std::false_type{});
            } else {
                uint32_t bw[16];
                base_words_general<16>(bw, cA, b, S.base, row_a + crr + 1, S.rows, C);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t x = cw[i];
                    const uint32_t lo4 = x & 0x0F0F0F0Fu, hi4 = (x >> 4) & 0x0F0F0F0Fu;
                    fl[i] = escape_flags8(lo4, hi4);
                    out[2 * i] = add_base(bw[2 * i], __byte_perm(lo4, hi4, 0x5140));
                    out[2 * i + 1] = add_base(bw[2 * i + 1], __byte_perm(lo4, hi4, 0x7362));
                }
            }
            q += S.step_q;
            rr += S.step_r;
            if (q >= C) { q -= C; ++rr; }
            if (cb + 32 < nch) load(cc + 32, rr);                // the next piece, while this one is patched
            // Element-ordered escape masks: bit j of f_h <-> element 32h + j.
            uint32_t f0 = __byte_perm(__byte_perm(fl[0], fl[1], 0x0040), __byte_perm(fl[2], fl[3], 0x0040), 0x5410);
            uint32_t f1 = __byte_perm(__byte_perm(fl[4], fl[5], 0x0040), __byte_perm(fl[6], fl[7], 0x0040), 0x5410);
            if (nv < kLaneNv) {
                f0 &= nv >= 32 ? 0xFFFFFFFFu : (nv == 0 ? 0u : 0xFFFFFFFFu >> (32 - nv));
                f1 &= nv <= 32 ? 0u : 0xFFFFFFFFu >> (64 - nv);
            }
            const uint32_t cnt = __popc(f0) + __popc(f1);
            uint32_t tot;
            uint32_t xl = X + warp_excl_scan(cnt, lane, tot);
            X += tot;
            if constexpr (SMEM) {
                // Write the chunk, then patch its exceptions in place.
                if (nv > 0) {
                    sstore32(sdst, p, out, lo_l, hi_l);
                    if (nv > 32) sstore32(sdst, p + 32, out + 8, lo_l, hi_l);
                }
                if (cnt) {
                    if (xl <= nexc && cnt <= nexc - xl) {
                        const uint8_t *ep = S.exc_bytes + xl;
                        uint32_t f = f0;
                        while (f) {
                            const uint32_t j = p + (uint32_t)(__ffs(f) - 1);
                            const uint32_t v = __ldg(ep++);
                            if (j >= lo_l && j < hi_l) sts_u8(sdst + j, v);
                            f &= f - 1;
                        }
                        f = f1;
                        while (f) {
                            const uint32_t j = p + (uint32_t)(__ffs(f) + 31);
                            const uint32_t v = __ldg(ep++);
                            if (j >= lo_l && j < hi_l) sts_u8(sdst + j, v);
                            f &= f - 1;
                        }
                    } else {
                        bad = true;
                    }
                }
                continue;
            }
            if (__any_sync(kFull, cnt != 0)) {
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    *reinterpret_cast<uint4 *>(my + ((16 * s) ^ gs)) =
                        make_uint4(out[4 * s], out[4 * s + 1], out[4 * s + 2], out[4 * s + 3]);
                // The lane's exceptions are consecutive in the stream.  An index
                // that points past it leaves the bytes and is reported.  (No
                // branch around the loops: they do nothing on empty masks, and
                // fewer divergent regions cost fewer instructions.)
                if (cnt && !(xl <= nexc && cnt <= nexc - xl)) {
                    bad = true;
                    f0 = f1 = 0;
                }
                const uint8_t *ep = S.exc_bytes + xl;
                uint32_t f = f0;
                while (f) {
                    my[(uint32_t)(__ffs(f) - 1) ^ gs] = __ldg(ep++);
                    f &= f - 1;
                }
                f = f1;
                while (f) {
                    my[(uint32_t)(__ffs(f) + 31) ^ gs] = __ldg(ep++);
                    f &= f - 1;
                }
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(my + ((16 * s) ^ gs));
                    out[4 * s] = v.x; out[4 * s + 1] = v.y; out[4 * s + 2] = v.z; out[4 * s + 3] = v.w;
                }
            }
            if (nv == kLaneNv && fast) {
                st_v8(ws + p, out);
                st_v8(ws + p + 32, out + 8);
            } else if (nv > 0) {
                store32(ws, S.ws_align, p, out, lo_l, hi_l);
                if (nv > 32) store32(ws, S.ws_align, p + 32, out + 8, lo_l, hi_l);
            }
        }
    };
    if constexpr (WORDS_OK) {
        if (words)
            run(std::true_type{});
        else
            run(std::false_type{});
    } else {
        run(std::false_type{});
    }
    if (lane == 1 && Xend != X) bad = true;
    if (__any_sync(kFull, bad) && lane == 0) flag(S.err, CSF_DEV_ERR_CORRUPT);
}

// ------------------------------------------------------------------ MXFP4

// Patch the escapes flagged in f (bit i -> staged element jb + i) with the
// next bytes of the exception stream, two per trip: the two loads are
// independent.  Used where exceptions are dense (MXFP4); with a few per lane
// chunk (NVFP4) the one-per-trip loop is faster.
__device__ __forceinline__ void patch_two(uint8_t *my, uint32_t gs, uint32_t jb, uint32_t f, const uint8_t *&ep) {
    while (f) {
        const uint32_t j0 = jb + (uint32_t)(__ffs(f) - 1);
        f &= f - 1;
        const bool two = f != 0;
        const uint32_t j1 = jb + (uint32_t)(__ffs(f) - 1);   // unused unless two
        f &= f - 1;
        const uint8_t v0 = __ldg(ep);
        uint8_t v1 = 0;
        if (two) v1 = __ldg(ep + 1);
        my[j0 ^ gs] = v0;
        if (two) my[j1 ^ gs] = v1;
        ep += two ? 2 : 1;
    }
}

// Decode rows [row_a, row_b) of an MXFP4 stack (row_a*C a multiple of 128);
// SMEM, sdst and WORDS_OK as in segment_nvfp4 (word-wise: C % 4 == 0, C >= 128
// and no base above 254).
template <bool SMEM, bool WORDS_OK>
__device__ void segment_mxfp4(const DecStack &S, uint64_t row_a, uint64_t row_b, uint64_t lo, uint64_t hi,
                              int lane, uint8_t *stage, uint32_t sdst) {
    const uint32_t C = (uint32_t)S.C;
    const uint64_t sa = row_a * C;
    const uint32_t nel = (uint32_t)(row_b * C - sa);
    const uint32_t nch = (nel + kLaneMx - 1) / kLaneMx;
    const uint8_t *offs = S.offsets + sa / 8;
    const uint8_t *escs = S.escapes + sa / 8;
    const uint8_t *bases = S.base + row_a;
    const uint64_t rows_left = S.rows - row_a;
    uint8_t *ws = S.ws + sa;
    const uint32_t lo_l = (uint32_t)(lo - sa);
    const uint32_t hi_l = (uint32_t)(hi - sa);
    const bool fast = lo_l == 0 && hi_l == nel && S.ws_align >= 32;
    const uint32_t nexc = (uint32_t)S.num_exc;
    bool bad = false;
    const uint32_t gs = ((uint32_t)lane & 7u) << 4;          // 16-byte slot swizzle (bank spread)
    uint8_t *my = stage + lane * 128;

    uint32_t rr = ((uint32_t)lane * kLaneMx) / C;
    uint32_t q = ((uint32_t)lane * kLaneMx) % C;
    uint4 ov = make_uint4(0, 0, 0, 0), xv = make_uint4(0, 0, 0, 0);
    uint32_t bA = 0, bB = 0;
    auto load = [&](uint32_t c, uint32_t r) {
        if (c < nch) {
            ov = __ldg(reinterpret_cast<const uint4 *>(offs + (size_t)c * 16));
            xv = __ldg(reinterpret_cast<const uint4 *>(escs + (size_t)c * 16));
            bA = __ldg(bases + r);
            bB = (r + 1 < rows_left) ? (uint32_t)__ldg(bases + r + 1) : 0u;
        } else {
            ov = xv = make_uint4(0, 0, 0, 0);
            bA = bB = 0;
        }
    };
    load((uint32_t)lane, rr);
    uint32_t X = 0, Xend = 0;                                  // as in segment_nvfp4
    if (lane == 0) X = __ldg(S.exc_index + row_a);
    if (lane == 1) Xend = __ldg(S.exc_index + row_b);
    const bool words = WORDS_OK && words_case(S, row_a, row_b, lane, kLaneMx, 254u);
    X = __shfl_sync(kFull, X, 0);

    auto run = [&](auto words_tag) {
    constexpr bool WORDS = decltype(words_tag)::value;
    for (uint32_t cb = 0; cb < nch; cb += 32) {
        const uint32_t cc = cb + lane;
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
        uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t cA = bA, cB = bB, cq = q, crr = rr;

        const uint32_t p = cc * kLaneMx;
        const int nv = cc < nch ? (int)min(nel - p, (uint32_t)kLaneMx) : 0;
        if (nv < kLaneMx) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int nvg = min(max(nv - 32 * k, 0), 32);
                if (nvg < 32) xw[k] &= nvg == 0 ? 0u : (0xFFFFFFFFu >> (32 - nvg));
            }
        }
        const uint32_t cnt = __popc(xw[0]) + __popc(xw[1]) + __popc(xw[2]) + __popc(xw[3]);
        uint32_t tot;
        uint32_t xl = X + warp_excl_scan(cnt, lane, tot);
        X += tot;
        if (nv > 0) {
            uint32_t rg = crr, qg = cq;                        // row / column of the group start
#pragma unroll
            for (int gi = 0; gi < 4; ++gi) {
                uint32_t out[8];
                if constexpr (WORDS) {
                    // Row B starts at word kb of the chunk (none when kb >= 32).
                    const uint32_t A4 = cA * 0x01010101u, B4 = cB * 0x01010101u;
                    const int kb = (int)(C - cq) >> 2;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t nib = (ow[gi] >> (4 * k)) & 0xFu;
                        out[k] = (8 * gi + k >= kb ? B4 : A4) + ((nib * 0x00204081u) & 0x01010101u);
                    }
                } else {
                const int bg = (int)(C - qg);                  // elements to the next row start
                const uint32_t A = rg == crr ? cA
                                 : (rg == crr + 1 ? cB : (rg < rows_left ? (uint32_t)__ldg(bases + rg) : 0u));
                if (C >= 32 || bg >= 32) {
                    // At most one row boundary in the group: bytes at or after
                    // element bg take row B's base.
                    uint32_t B = A;
                    if (bg < 32) {
                        const uint32_t rn = rg + 1;
                        B = rn == crr + 1 ? cB : (rn < rows_left ? (uint32_t)__ldg(bases + rn) : 0u);
                    }
                    const uint32_t A4 = A * 0x01010101u, B4 = B * 0x01010101u;
                    if (A <= 254u && B <= 254u) {
                        // base + 1 <= 255: a plain add cannot carry between bytes.
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t nib = (ow[gi] >> (4 * k)) & 0xFu;
                            const uint32_t m = bytes_from(bg, k);
                            out[k] = ((A4 & ~m) | (B4 & m)) + ((nib * 0x00204081u) & 0x01010101u);  // bit j -> byte j
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t nib = (ow[gi] >> (4 * k)) & 0xFu;
                            const uint32_t m = bytes_from(bg, k);
                            out[k] = add_base((A4 & ~m) | (B4 & m), (nib * 0x00204081u) & 0x01010101u);
                        }
                    }
                } else {
                    uint32_t bw[8];
                    base_words_general<8>(bw, A, bg, S.base, row_a + rg + 1, S.rows, C);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t nib = (ow[gi] >> (4 * k)) & 0xFu;
                        out[k] = add_base(bw[k], (nib * 0x00204081u) & 0x01010101u);
                    }
                }
                }
                if constexpr (SMEM) {
                    if (32 * gi < nv) sstore32(sdst, p + 32u * gi, out, lo_l, hi_l);
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int s = 2 * gi + h;
                        *reinterpret_cast<uint4 *>(my + ((16 * s) ^ gs)) =
                            make_uint4(out[4 * h], out[4 * h + 1], out[4 * h + 2], out[4 * h + 3]);
                    }
                }
                qg += 32;
                while (qg >= C) { qg -= C; ++rg; }
            }
        }
        // the next piece, into the registers the expansion has just read
        q += S.step_q;
        rr += S.step_r;
        if (q >= C) { q -= C; ++rr; }
        if (cb + 32 < nch) load(cc + 32, rr);
        if (nv > 0) {
            if (cnt) {
                if (xl <= nexc && cnt <= nexc - xl) {
                    const uint8_t *ep = S.exc_bytes + xl;
#pragma unroll
                    for (int gi = 0; gi < 4; ++gi) {
                        uint32_t f = xw[gi];
                        if constexpr (SMEM) {
                            while (f) {
                                const uint32_t j = p + 32u * gi + (uint32_t)(__ffs(f) - 1);
                                const uint32_t v = __ldg(ep++);
                                if (j >= lo_l && j < hi_l) sts_u8(sdst + j, v);   // patched in place
                                f &= f - 1;
                            }
                        } else {
                            patch_two(my, gs, 32u * gi, f, ep);
                        }
                    }
                } else {
                    bad = true;
                }
            }
            if constexpr (!SMEM) {
                // reload the patched lane chunk and store it
#pragma unroll
                for (int gi = 0; gi < 4; ++gi) {
                    uint32_t out[8];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(my + ((16 * (2 * gi + h)) ^ gs));
                        out[4 * h] = v.x; out[4 * h + 1] = v.y; out[4 * h + 2] = v.z; out[4 * h + 3] = v.w;
                    }
                    const uint32_t pg = p + 32u * gi;
                    if (nv == kLaneMx && fast) st_v8(ws + pg, out);
                    else if (32 * gi < nv) store32(ws, S.ws_align, pg, out, lo_l, hi_l);
                }
            }
        }
    }
    };
    if constexpr (WORDS_OK) {
        if (words)
            run(std::true_type{});
        else
            run(std::false_type{});
    } else {
        run(std::false_type{});
    }
    if (lane == 1 && Xend != X) bad = true;
    if (__any_sync(kFull, bad) && lane == 0) flag(S.err, CSF_DEV_ERR_CORRUPT);
}

// Units that hold rows [r_lo, r_hi) of expert e.
// Rows stay below 2^31, so 32-bit arithmetic holds.
__device__ __forceinline__ uint32_t units_of_expert(const DecStack &S, uint32_t e) {
    const uint32_t r0 = e * (uint32_t)S.R + (uint32_t)S.r_lo;
    const uint32_t r1 = e * (uint32_t)S.R + (uint32_t)S.r_hi;
    const uint32_t rb = (uint32_t)S.rb;
    return (r1 + rb - 1) / rb - r0 / rb;
}

#ifndef CSF_DECODE_MIN_BLOCKS
#define CSF_DECODE_MIN_BLOCKS 3
#endif

// PER_EXPERT: the work list is built per selected expert (routing, row
// ranges); otherwise it covers the whole stacks.  KINDS (DecodeKinds): the
// segment decoders compiled in, so that a launch of one kind carries no code
// of the other.
template <bool PER_EXPERT, int KINDS>
__global__ void __launch_bounds__(kThreads, CSF_DECODE_MIN_BLOCKS) decode_kernel(const __grid_constant__ DecParams P) {
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ __align__(16) uint8_t s_stage[kWarps][kStageBytes];
    __shared__ uint32_t s_wsum[3][kWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint64_t T0, T1;
    uint32_t n_act = 0;
    uint32_t *act = smem;
    uint32_t *up0 = smem + P.E;
    uint32_t *up1 = up0 + P.E + 1;
    if (PER_EXPERT && P.uniform) {
        // Every expert has upe units: only the active ids are needed (none
        // without routing: expert j is entry j).
        uint32_t run_n = (uint32_t)P.E;
        if (P.expert_start != nullptr) {
            run_n = 0;
            for (int e0 = 0; e0 < P.E; e0 += kThreads) {
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
                if (lane == 0) s_wsum[0][warp] = __popc(bal);
                __syncthreads();
                uint32_t bn = run_n, tn = 0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    if (w < warp) bn += s_wsum[0][w];
                    tn += s_wsum[0][w];
                }
                if (a) act[bn + __popc(bal & lanemask_lt())] = (uint32_t)e;
                run_n += tn;
                __syncthreads();
            }
        }
        n_act = run_n;
        T0 = (uint64_t)n_act * P.st[0].upe;
        T1 = P.nstacks > 1 ? (uint64_t)n_act * P.st[1].upe : 0;
    } else if (PER_EXPERT) {
        // Active-expert compaction: expert e is active iff start[e+1] > start[e]
        // (every expert without routing), with each stack's unit prefix.
        uint32_t run_n = 0, run0 = 0, run1 = 0;
        for (int e0 = 0; e0 < P.E; e0 += kThreads) {
            const int e = e0 + threadIdx.x;
            bool a = false;
            if (e < P.E) {
                if (P.expert_start == nullptr) {
                    a = true;
                } else if (P.es64) {
                    const long long *s = static_cast<const long long *>(P.expert_start);
                    a = __ldg(s + e + 1) > __ldg(s + e);
                } else {
                    const int *s = static_cast<const int *>(P.expert_start);
                    a = __ldg(s + e + 1) > __ldg(s + e);
                }
            }
            const uint32_t u0 = a ? units_of_expert(P.st[0], (uint32_t)e) : 0u;
            const uint32_t u1 = (a && P.nstacks > 1) ? units_of_expert(P.st[1], (uint32_t)e) : 0u;
            const uint32_t bal = __ballot_sync(kFull, a);
            uint32_t t0, t1;
            const uint32_t x0 = warp_excl_scan(u0, lane, t0);
            const uint32_t x1 = warp_excl_scan(u1, lane, t1);
            if (lane == 0) {
                s_wsum[0][warp] = __popc(bal);
                s_wsum[1][warp] = t0;
                s_wsum[2][warp] = t1;
            }
            __syncthreads();
            uint32_t bn = run_n, b0 = run0, b1 = run1;
            uint32_t tn = 0, tt0 = 0, tt1 = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                if (w < warp) { bn += s_wsum[0][w]; b0 += s_wsum[1][w]; b1 += s_wsum[2][w]; }
                tn += s_wsum[0][w]; tt0 += s_wsum[1][w]; tt1 += s_wsum[2][w];
            }
            if (a) {
                const uint32_t j = bn + __popc(bal & lanemask_lt());
                act[j] = (uint32_t)e;
                up0[j] = b0 + x0;
                up1[j] = b1 + x1;
            }
            run_n += tn; run0 += tt0; run1 += tt1;
            __syncthreads();
        }
        if (threadIdx.x == 0) { up0[run_n] = run0; up1[run_n] = run1; }
        __syncthreads();
        n_act = run_n;
        T0 = run0;
        T1 = run1;
    } else {
        T0 = (P.st[0].rows + P.st[0].rb - 1) / P.st[0].rb;
        T1 = P.nstacks > 1 ? (P.st[1].rows + P.st[1].rb - 1) / P.st[1].rb : 0;
    }
    uint8_t *stage = s_stage[warp];
    const uint64_t T = T0 + T1;
    const uint64_t W = (uint64_t)gridDim.x * kWarps;
    const uint64_t w = (uint64_t)blockIdx.x * kWarps + warp;
    uint64_t u = T * w / W;
    uint64_t ub = T * (w + 1) / W;
    if (PER_EXPERT && P.uniform && P.nstacks == 1 && n_act > 0 && W >= n_act && W < (1u << 13) &&
        P.st[0].upe < (1u << 19) && !(P.st[0].r_lo == 0 && P.st[0].r_hi == P.st[0].R)) {
        // A row range of every selected expert (segments cannot run on from
        // one expert to the next): whole warps per expert, so that no warp's
        // range straddles two experts and pays a second segment start.  With
        // fewer than 2^13 warps and 2^19 units per expert every product below
        // fits in 32 bits.
        const uint32_t U = P.st[0].upe, wpe = (uint32_t)W / n_act, j = (uint32_t)w / wpe;
        if (j >= n_act) {
            u = ub = 0;
        } else {
            const uint32_t k = (uint32_t)w - j * wpe;
            u = (uint64_t)j * U + U * k / wpe;
            ub = (uint64_t)j * U + U * (k + 1) / wpe;
        }
    }
    while (u < ub) {
        const int s = (u < T0) ? 0 : 1;
        const DecStack &S = P.st[s];
        const uint64_t base_u = s ? T0 : 0;
        const uint64_t lu = u - base_u;
        const uint64_t lend = (s ? ub : min(ub, T0)) - base_u;
        uint64_t row_a, row_b, lo, hi, cnt;
        const uint64_t rb = (uint64_t)S.rb;
        const uint64_t C = (uint64_t)S.C;
        if (!PER_EXPERT) {
            cnt = min(lend - lu, S.max_units);
            row_a = lu * rb;
            row_b = min((lu + cnt) * rb, S.rows);
            lo = row_a * C;
            hi = row_b * C;
        } else {
            // Entry jl of the active list holds unit lu; the segment ends at
            // the unit `u_end` where entry je starts.
            uint32_t jl, je;
            uint64_t k, u_end;
            const bool routed = P.expert_start != nullptr;
            // With whole experts that start on unit boundaries, the units of
            // consecutive active experts are consecutive in the stack: one
            // segment runs on through them.
            const bool run_on = S.r_lo == 0 && S.r_hi == S.R && S.R % S.rb == 0;
            if (P.uniform) {
                const uint32_t U = S.upe;
                jl = (uint32_t)(lu / U);
                k = lu - (uint64_t)jl * U;
                je = jl + 1;
                if (run_on && routed)
                    while (je < n_act && act[je] == act[je - 1] + 1 && (uint64_t)je * U < lend) ++je;
                u_end = (uint64_t)je * U;
            } else {
                const uint32_t *up = s ? up1 : up0;
                uint32_t jh = n_act - 1;            // largest jl with up[jl] <= lu
                jl = 0;
                while (jl < jh) {
                    const uint32_t mid = (jl + jh + 1) >> 1;
                    if ((uint64_t)up[mid] <= lu) jl = mid; else jh = mid - 1;
                }
                k = lu - up[jl];
                je = jl + 1;
                if (run_on)
                    while (je < n_act && act[je] == act[je - 1] + 1 && (uint64_t)up[je] < lend) ++je;
                u_end = up[je];
            }
            const uint64_t e = routed || !P.uniform ? act[jl] : jl;
            const uint64_t e_last = routed || !P.uniform ? act[je - 1] : je - 1;
            const uint64_t R = (uint64_t)S.R;
            cnt = min(min(lend, u_end) - lu, S.max_units);
            const uint64_t r0 = e * R + (uint64_t)S.r_lo;
            const uint64_t r1 = e_last * R + (uint64_t)S.r_hi;
            const uint64_t first_unit = r0 / rb;
            row_a = (first_unit + k) * rb;
            row_b = min((first_unit + k + cnt) * rb, S.rows);
            lo = max(row_a, r0) * C;
            hi = min(row_b, r1) * C;
        }
        if (KINDS == kKindsNv || (KINDS == kKindsBoth && S.kind == CSF_NVFP4)) {
            segment_nvfp4<false, true>(S, row_a, row_b, lo, hi, lane, stage, 0u);
        } else {
            segment_mxfp4<false, true>(S, row_a, row_b, lo, hi, lane, stage, 0u);
        }
        u += cnt;
    }
}

// ------------------------------ scale-operand layout, a 128-row block per block

#ifndef CSF_BLOCKS_MIN_BLOCKS
#define CSF_BLOCKS_MIN_BLOCKS 12
#endif

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Decode into the 128 x 4 tiled scale-operand layout of block-scaled GEMMs
// (see csf_tiles.cu for the layout): a block of kBlkWarps warps takes one
// 128-row block of an expert; each warp decodes its share of the rows with
// the row-major segment code into the block's shared-memory buffer
// (exceptions patched in place); then the warps write the block's tiles,
// lane b assembling line b of a tile from rows b, b+32, b+64, b+96, so every
// tile leaves as one coalesced 512-byte warp store.  Rows whose first unit
// starts before the warp's share are decoded whole and clipped.
// KINDS (DecodeKinds) and WORDS_OK as for decode_kernel and segment_nvfp4.
template <int KINDS, bool WORDS_OK>
__global__ void __launch_bounds__(kBlkThreads, CSF_BLOCKS_MIN_BLOCKS)
    decode_blocks_kernel(const __grid_constant__ DecParams P) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ uint32_t s_cnt[kBlkWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint32_t *act = reinterpret_cast<uint32_t *>(dsm);
    uint8_t *buf = dsm + P.buf_off;
    const uint32_t buf_sa = (uint32_t)__cvta_generic_to_shared(buf);

    uint32_t n_act = (uint32_t)P.E;
    if (P.expert_start != nullptr) {
        n_act = 0;
        for (int e0 = 0; e0 < P.E; e0 += kBlkThreads) {
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
            for (int w = 0; w < kBlkWarps; ++w) {
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
    constexpr uint32_t kShare = kTileRows / kBlkWarps;                     // rows decoded per warp
    for (uint64_t it = blockIdx.x; it < total; it += gridDim.x) {
        const int s = it < it0 ? 0 : 1;
        const DecStack &S = P.st[s];
        const uint32_t Bs = s ? B1 : B0;
        const uint64_t li = s ? it - it0 : it;
        const uint32_t j = (uint32_t)(li / Bs);
        const uint32_t t = (uint32_t)(li - (uint64_t)j * Bs);
        const uint64_t e = P.expert_start != nullptr ? act[j] : j;
        const uint64_t R = (uint64_t)S.R, C = (uint64_t)S.C, rb = (uint64_t)S.rb;
        const uint32_t rl0 = (uint32_t)S.r_lo + t * kTileRows;          // expert-local first row
        const uint64_t r0 = e * R + rl0;
        const uint64_t r1 = min(r0 + kTileRows, e * R + (uint64_t)S.r_hi);
        // Element x of the stack lands at buf + (x - x0); 32-byte pieces of the
        // flat stream stay 32-byte aligned.
        const uint64_t x0 = (r0 * C) & ~31ull;
        const uint64_t rs = r0 + (uint64_t)warp * kShare;
        const uint64_t re = min(rs + kShare, r1);
        if (rs < re) {
            const uint64_t row_a = rs / rb * rb, row_b = min((re + rb - 1) / rb * rb, S.rows);
            const uint32_t sdst = buf_sa + (uint32_t)(row_a * C - x0);  // modulo 2^32
            if (KINDS == kKindsNv || (KINDS == kKindsBoth && S.kind == CSF_NVFP4))
                segment_nvfp4<true, WORDS_OK>(S, row_a, row_b, rs * C, re * C, lane, buf, sdst);
            else
                segment_mxfp4<true, WORDS_OK>(S, row_a, row_b, rs * C, re * C, lane, buf, sdst);
        }
        __syncthreads();

        const uint32_t Ci = (uint32_t)C;
        const uint32_t ncb = (Ci + 3) / 4;
        const uint32_t nrow = (uint32_t)(r1 - r0);
        const uint64_t RP = (R + kTileRows - 1) / kTileRows * kTileRows;
        uint8_t *line = S.ws + e * RP * (4ull * ncb) + (uint64_t)(rl0 / kTileRows) * ncb * 512 + 16u * (uint32_t)lane;
        const uint32_t src = buf_sa + (uint32_t)(r0 * C - x0) + (uint32_t)lane * Ci;
        for (uint32_t cb = (uint32_t)warp; cb < ncb; cb += kBlkWarps) {
            uint32_t w[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                uint32_t v = 0;
                if ((uint32_t)lane + 32u * a < nrow) {
                    const uint32_t off = src + 32u * a * Ci + 4 * cb;
                    if ((Ci & 3) == 0) {
                        v = lds_u32(off);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (4 * cb + q < Ci) v |= lds_u8(off + q) << (8 * q);
                    }
                }
                w[a] = v;
            }
            *reinterpret_cast<uint4 *>(line + (uint64_t)cb * 512) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
    }
}

}  // namespace

// The blocked-layout instance a launch needs: its kinds, and whether any
// stack of it can take the word-wise loop (C % 4 == 0 and C at least the
// lane chunk: 64 NVFP4, 128 MXFP4).
template <int KINDS, bool WORDS_OK>
cudaError_t blocks_of(const DecParams *p, int grid, size_t smem, cudaStream_t s, int *blocks_per_sm) {
    cudaError_t e = cudaFuncSetAttribute(decode_blocks_kernel<KINDS, WORDS_OK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (blocks_per_sm)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_blocks_kernel<KINDS, WORDS_OK>,
                                                             kBlkThreads, smem);
    decode_blocks_kernel<KINDS, WORDS_OK><<<grid, kBlkThreads, smem, s>>>(*p);
    return cudaGetLastError();
}

cudaError_t blocks_dispatch(const DecParams &p, int grid, size_t smem, cudaStream_t s, int *blocks_per_sm) {
    const int k = decode_kinds(p);
    bool words = false;
    for (int i = 0; i < p.nstacks; ++i)
        if (p.st[i].C % 4 == 0 && p.st[i].C >= (p.st[i].kind == CSF_NVFP4 ? kLaneNv : kLaneMx)) words = true;
    if (k == kKindsMx)
        return words ? blocks_of<kKindsMx, true>(&p, grid, smem, s, blocks_per_sm)
                     : blocks_of<kKindsMx, false>(&p, grid, smem, s, blocks_per_sm);
    if (k == kKindsNv)
        return words ? blocks_of<kKindsNv, true>(&p, grid, smem, s, blocks_per_sm)
                     : blocks_of<kKindsNv, false>(&p, grid, smem, s, blocks_per_sm);
    return words ? blocks_of<kKindsBoth, true>(&p, grid, smem, s, blocks_per_sm)
                 : blocks_of<kKindsBoth, false>(&p, grid, smem, s, blocks_per_sm);
}

cudaError_t decode_blocks_occupancy(const DecParams &p, size_t smem, int *blocks_per_sm) {
    return blocks_dispatch(p, 0, smem, nullptr, blocks_per_sm);
}

cudaError_t launch_decode_blocks(const DecParams &p, int grid, size_t smem, cudaStream_t s) {
    return blocks_dispatch(p, grid, smem, s, nullptr);
}

// Dynamic shared memory beyond the default window (48 KB with the static
// part) needs an opt-in, before the occupancy query as well as the launch.
template <typename K>
cudaError_t allow_smem(K kernel, size_t smem) {
    if (smem == 0) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <bool PER_EXPERT, int KINDS>
cudaError_t occupancy_of(size_t smem, int *blocks_per_sm) {
    cudaError_t e = allow_smem(decode_kernel<PER_EXPERT, KINDS>, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel<PER_EXPERT, KINDS>, kThreads,
                                                         smem);
}

template <bool PER_EXPERT>
cudaError_t occupancy_kinds(int kinds, size_t smem, int *blocks_per_sm) {
    if (kinds == kKindsNv) return occupancy_of<PER_EXPERT, kKindsNv>(smem, blocks_per_sm);
    if (kinds == kKindsMx) return occupancy_of<PER_EXPERT, kKindsMx>(smem, blocks_per_sm);
    return occupancy_of<PER_EXPERT, kKindsBoth>(smem, blocks_per_sm);
}

cudaError_t decode_occupancy(bool per_expert, int kinds, size_t smem, int *blocks_per_sm) {
    return per_expert ? occupancy_kinds<true>(kinds, smem, blocks_per_sm)
                      : occupancy_kinds<false>(kinds, smem, blocks_per_sm);
}

template <bool PER_EXPERT, int KINDS>
cudaError_t launch_of(const DecParams &p, int grid, size_t smem, cudaStream_t s) {
    cudaError_t e = allow_smem(decode_kernel<PER_EXPERT, KINDS>, smem);
    if (e != cudaSuccess) return e;
    decode_kernel<PER_EXPERT, KINDS><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <bool PER_EXPERT>
cudaError_t launch_kinds(const DecParams &p, int grid, size_t smem, cudaStream_t s) {
    const int k = decode_kinds(p);
    if (k == kKindsNv) return launch_of<PER_EXPERT, kKindsNv>(p, grid, smem, s);
    if (k == kKindsMx) return launch_of<PER_EXPERT, kKindsMx>(p, grid, smem, s);
    return launch_of<PER_EXPERT, kKindsBoth>(p, grid, smem, s);
}

cudaError_t launch_decode(const DecParams &p, int grid, size_t smem, bool per_expert, cudaStream_t s) {
    return per_expert ? launch_kinds<true>(p, grid, smem, s) : launch_kinds<false>(p, grid, smem, s);
}

}  // namespace csfk
