// CSF decode kernel for sm_103a: rebuilds dense FP8 scale bytes from a
// compressed stack, for the whole stack or only for routed experts, and for
// one stack or a gate/down pair in the same launch.
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
//     on both routing integer types, and on vectorised indexed
//     reconstruction and exception lookup.
//
// Design (GB300 first; HBM-bound byte work, no tensor cores):
//   * Work unit = a run of `rb` rows whose elements fill whole chunks
//     (32 elements = 16 offset bytes for NVFP4, 128 elements = 16 bytes of
//     each bit plane for MXFP4).  Every warp of a persistent grid takes one
//     contiguous range of units (balanced to one unit), so it reads a single
//     exc_index entry at the start of each contiguous segment and then walks
//     the exception stream in order: exceptions of consecutive rows are
//     consecutive, so the running position is the segment's first index plus
//     the escapes met so far (warp ballot-free scan of per-lane popcounts).
//     The per-row index is checked against that position at the segment end.
//   * Lanes read 16-byte pieces of the offset stream (coalesced), expand them
//     with byte permutes and carry-free byte adds, patch escapes in registers
//     from the exception stream, and write each 32-byte piece with one
//     256-bit store (full sectors, no read-for-ownership).
//   * Routed mode: every block compacts the active experts of `expert_start`
//     into shared memory with ballots and prefix sums; the units of inactive
//     experts never exist, so their workspace planes are never written.
//   * A unit whose rows straddle an expert boundary (R*C not a multiple of the
//     chunk) is decoded whole but stored only inside its expert's rows.
#include "csf_internal.cuh"

namespace csfk {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, int lane, uint32_t &total) {
    uint32_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t y = __shfl_up_sync(kFull, x, d);
        if (lane >= d) x += y;
    }
    total = __shfl_sync(kFull, x, 31);
    return x - v;
}

__device__ __forceinline__ uint4 ldg16(const uint8_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void st_v8(uint8_t *p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Store 32 decoded bytes for elements [p, p+32) to ws + p, keeping only the
// bytes inside [lo, hi).  `align` is the byte alignment of ws (p is a
// multiple of 32).
__device__ __forceinline__ void store32(uint8_t *ws, int align, uint64_t p, const uint32_t (&w)[8],
                                        uint64_t lo, uint64_t hi) {
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
            uint64_t q = p + j;
            if (q >= lo && q < hi) d[j] = (uint8_t)(w[j >> 2] >> (8 * (j & 3)));
        }
    }
}

// Bytes [j] of bw = base byte of the row of element (start + j), for NW words
// (4*NW elements).  `b` = elements from `start` to the next row start;
// `second` = base of that next row; rows after it are loaded here.
template <int NW>
__device__ __forceinline__ void base_words(uint32_t (&bw)[NW], uint32_t first, uint32_t second, int b,
                                           const uint8_t *__restrict__ base, uint64_t row_after_next,
                                           uint64_t rows, uint32_t C) {
    const uint32_t a = first * 0x01010101u;
#pragma unroll
    for (int k = 0; k < NW; ++k) bw[k] = a;
    if (b < 4 * NW) {
        uint32_t nb = second * 0x01010101u;
        uint64_t rn = row_after_next;
        while (true) {
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                int d8 = 8 * (b - 4 * k);
                uint32_t s = (uint32_t)min(max(d8, 0), 32);
                uint32_t m = __funnelshift_lc(0u, 0xFFFFFFFFu, s);  // bytes at or after the boundary
                bw[k] = (bw[k] & ~m) | (nb & m);
            }
            b += (int)C;
            if (b >= 4 * NW) break;
            nb = (rn < rows ? (uint32_t)__ldg(base + rn) : 0u) * 0x01010101u;
            ++rn;
        }
    }
}

// base + offset, byte-wise mod 256, for offsets below 0x80 (no carry between
// bytes: the low 7 bits are added, bit 7 is folded back with XOR).
__device__ __forceinline__ uint32_t add_base(uint32_t bw, uint32_t off) {
    return ((bw & 0x7F7F7F7Fu) + off) ^ (bw & 0x80808080u);
}

__device__ __forceinline__ uint32_t exc_at(const DecStack &S, uint64_t x, bool &bad) {
    if (x < S.num_exc) return (uint32_t)__ldg(S.exc_bytes + x);
    bad = true;
    return 0u;
}

__device__ __forceinline__ void flag(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// Insert exception bytes into one output word for the set escape bits of
// `m` (bit 4j <-> byte j for NVFP4, bit j <-> byte j for MXFP4).
template <int STRIDE>
__device__ __forceinline__ void patch_word(uint32_t &w, uint32_t m, const DecStack &S, uint64_t &x, bool &bad) {
    while (m) {
        const uint32_t b = (uint32_t)(__ffs(m) - 1);
        m &= m - 1;
        const uint32_t sh = 8u * (b / STRIDE);
        const uint32_t e = exc_at(S, x, bad);
        ++x;
        w = (w & ~(0xFFu << sh)) | (e << sh);
    }
}

// Decode rows [row_a, row_b) of an NVFP4 stack (row_a*C a multiple of 32),
// storing only elements in [lo, hi).  Whole warp; U chunks per lane per step.
template <int U>
__device__ void segment_nvfp4(const DecStack &S, uint64_t row_a, uint64_t row_b, uint64_t lo, uint64_t hi,
                              int lane) {
    const uint32_t C = (uint32_t)S.C;
    const uint64_t sa = row_a * C;
    const uint64_t sb = row_b * C;
    const uint64_t c_begin = sa / kChunkNv;
    const uint64_t c_end = (sb + kChunkNv - 1) / kChunkNv;
    uint64_t X = 0;
    if (lane == 0) X = __ldg(S.exc_index + row_a);
    X = __shfl_sync(kFull, X, 0);
    bool bad = false;
    const uint32_t lane_el = (uint32_t)lane * kChunkNv;
    uint64_t r = row_a + lane_el / C;
    uint32_t q = lane_el % C;
    for (uint64_t cb = c_begin; cb < c_end; cb += 32 * U) {
        uint4 off[U];
        uint32_t bA[U], bB[U], qu[U];
        uint64_t ru[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t c = cb + 32 * u + lane;
            ru[u] = r;
            qu[u] = q;
            if (c < c_end) {
                off[u] = ldg16(S.offsets + c * 16);
                bA[u] = __ldg(S.base + r);
                bB[u] = (r + 1 < S.rows) ? (uint32_t)__ldg(S.base + r + 1) : 0u;
            } else {
                off[u] = make_uint4(0, 0, 0, 0);
                bA[u] = bB[u] = 0;
            }
            q += S.step_q;
            r += S.step_r;
            if (q >= C) { q -= C; ++r; }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t c = cb + 32 * u + lane;
            const uint64_t p = c * kChunkNv;
            const int nv = c < c_end ? (int)min(sb - p, (uint64_t)kChunkNv) : 0;
            uint32_t bw[8];
            base_words<8>(bw, bA[u], bB[u], (int)(C - qu[u]), S.base, ru[u] + 2, S.rows, C);
            const uint32_t wv[4] = {off[u].x, off[u].y, off[u].z, off[u].w};
            uint32_t out[8], t[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = wv[i];
                const uint32_t lo4 = w & 0x0F0F0F0Fu;
                const uint32_t hi4 = (w >> 4) & 0x0F0F0F0Fu;
                out[2 * i] = add_base(bw[2 * i], __byte_perm(lo4, hi4, 0x5140));
                out[2 * i + 1] = add_base(bw[2 * i + 1], __byte_perm(lo4, hi4, 0x7362));
                uint32_t esc = w & (w >> 1) & (w >> 2) & (w >> 3) & 0x11111111u;  // nibble == 15
                const int nvi = min(max(nv - 8 * i, 0), 8);
                if (nvi < 8) esc &= (1u << (4 * nvi)) - 1u;
                t[i] = esc;
            }
            const uint32_t cnt = __popc(t[0]) + __popc(t[1]) + __popc(t[2]) + __popc(t[3]);
            uint32_t tot;
            const uint32_t ex = warp_excl_scan(cnt, lane, tot);
            uint64_t xl = X + ex;
            X += tot;
            if (cnt) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    patch_word<4>(out[k], (t[k >> 1] >> (16 * (k & 1))) & 0x1111u, S, xl, bad);
            }
            if (nv > 0) store32(S.ws, S.ws_align, p, out, lo, hi);
        }
    }
    if (lane == 0) {
        const uint64_t expect = __ldg(S.exc_index + row_b);
        if (expect != X) bad = true;
    }
    if (__any_sync(kFull, bad) && lane == 0) flag(S.err, CSF_DEV_ERR_CORRUPT);
}

// Decode rows [row_a, row_b) of an MXFP4 stack (row_a*C a multiple of 128).
template <int U>
__device__ void segment_mxfp4(const DecStack &S, uint64_t row_a, uint64_t row_b, uint64_t lo, uint64_t hi,
                              int lane) {
    const uint32_t C = (uint32_t)S.C;
    const uint64_t sa = row_a * C;
    const uint64_t sb = row_b * C;
    const uint64_t c_begin = sa / kChunkMx;
    const uint64_t c_end = (sb + kChunkMx - 1) / kChunkMx;
    uint64_t X = 0;
    if (lane == 0) X = __ldg(S.exc_index + row_a);
    X = __shfl_sync(kFull, X, 0);
    bool bad = false;
    const uint32_t lane_el = (uint32_t)lane * kChunkMx;
    uint64_t r = row_a + lane_el / C;
    uint32_t q = lane_el % C;
    for (uint64_t cb = c_begin; cb < c_end; cb += 32 * U) {
        uint4 ov[U], xv[U];
        uint32_t bA[U], bB[U], qu[U];
        uint64_t ru[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t c = cb + 32 * u + lane;
            ru[u] = r;
            qu[u] = q;
            if (c < c_end) {
                ov[u] = ldg16(S.offsets + c * 16);
                xv[u] = ldg16(S.escapes + c * 16);
                bA[u] = __ldg(S.base + r);
                bB[u] = (r + 1 < S.rows) ? (uint32_t)__ldg(S.base + r + 1) : 0u;
            } else {
                ov[u] = xv[u] = make_uint4(0, 0, 0, 0);
                bA[u] = bB[u] = 0;
            }
            q += S.step_q;
            r += S.step_r;
            if (q >= C) { q -= C; ++r; }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t c = cb + 32 * u + lane;
            const uint64_t p = c * kChunkMx;
            const int nv = c < c_end ? (int)min(sb - p, (uint64_t)kChunkMx) : 0;
            const uint32_t ow[4] = {ov[u].x, ov[u].y, ov[u].z, ov[u].w};
            uint32_t xw[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int nvg = min(max(nv - 32 * g, 0), 32);
                if (nvg < 32) xw[g] &= (nvg == 0) ? 0u : (0xFFFFFFFFu >> (32 - nvg));
            }
            const uint32_t cnt = __popc(xw[0]) + __popc(xw[1]) + __popc(xw[2]) + __popc(xw[3]);
            uint32_t tot;
            const uint32_t ex = warp_excl_scan(cnt, lane, tot);
            uint64_t xl = X + ex;
            X += tot;
            if (nv == 0) continue;
            uint64_t rg = ru[u];
            uint32_t qg = qu[u];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                if (32 * g < nv) {
                    const uint32_t first = (rg == ru[u]) ? bA[u] : (rg == ru[u] + 1 ? bB[u] : (uint32_t)__ldg(S.base + rg));
                    const int bnd = (int)(C - qg);
                    uint32_t second = 0;
                    if (bnd < 32) {
                        const uint64_t rs = rg + 1;
                        second = (rs == ru[u] + 1) ? bB[u] : (rs < S.rows ? (uint32_t)__ldg(S.base + rs) : 0u);
                    }
                    uint32_t bw[8];
                    base_words<8>(bw, first, second, bnd, S.base, rg + 2, S.rows, C);
                    uint32_t out[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t nib = (ow[g] >> (4 * k)) & 0xFu;
                        out[k] = add_base(bw[k], (nib * 0x00204081u) & 0x01010101u);  // bit j -> byte j
                    }
                    if (xw[g]) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) patch_word<1>(out[k], (xw[g] >> (4 * k)) & 0xFu, S, xl, bad);
                    }
                    store32(S.ws, S.ws_align, p + 32 * g, out, lo, hi);
                }
                qg += 32;
                while (qg >= C) { qg -= C; ++rg; }
            }
        }
    }
    if (lane == 0) {
        const uint64_t expect = __ldg(S.exc_index + row_b);
        if (expect != X) bad = true;
    }
    if (__any_sync(kFull, bad) && lane == 0) flag(S.err, CSF_DEV_ERR_CORRUPT);
}

__device__ __forceinline__ uint64_t units_of_expert(const DecStack &S, uint64_t e) {
    const uint64_t R = (uint64_t)S.R;
    const uint64_t rb = (uint64_t)S.rb;
    return ((e + 1) * R + rb - 1) / rb - (e * R) / rb;
}

template <bool ROUTED>
__global__ void __launch_bounds__(kThreads, 4) decode_kernel(const __grid_constant__ DecParams P) {
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ uint32_t s_wsum[3][kWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint64_t T0, T1;
    uint32_t n_act = 0;
    uint32_t *act = smem;
    uint32_t *up0 = smem + P.E;
    uint32_t *up1 = up0 + P.E + 1;
    if (ROUTED) {
        // Active-expert compaction: expert e is active iff start[e+1] > start[e].
        uint32_t run_n = 0, run0 = 0, run1 = 0;
        for (int e0 = 0; e0 < P.E; e0 += kThreads) {
            const int e = e0 + threadIdx.x;
            bool a = false;
            if (e < P.E) {
                if (P.es64) {
                    const long long *s = static_cast<const long long *>(P.expert_start);
                    a = __ldg(s + e + 1) > __ldg(s + e);
                } else {
                    const int *s = static_cast<const int *>(P.expert_start);
                    a = __ldg(s + e + 1) > __ldg(s + e);
                }
            }
            const uint32_t u0 = a ? (uint32_t)units_of_expert(P.st[0], (uint64_t)e) : 0u;
            const uint32_t u1 = (a && P.nstacks > 1) ? (uint32_t)units_of_expert(P.st[1], (uint64_t)e) : 0u;
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
    const uint64_t T = T0 + T1;
    const uint64_t W = (uint64_t)gridDim.x * kWarps;
    const uint64_t w = (uint64_t)blockIdx.x * kWarps + warp;
    uint64_t u = T * w / W;
    const uint64_t ub = T * (w + 1) / W;
    while (u < ub) {
        const int s = (u < T0) ? 0 : 1;
        const DecStack &S = P.st[s];
        const uint64_t base_u = s ? T0 : 0;
        const uint64_t lu = u - base_u;
        const uint64_t lend = (s ? ub : min(ub, T0)) - base_u;
        uint64_t row_a, row_b, lo, hi, cnt;
        const uint64_t rb = (uint64_t)S.rb;
        const uint64_t C = (uint64_t)S.C;
        if (!ROUTED) {
            cnt = lend - lu;
            row_a = lu * rb;
            row_b = min(lend * rb, S.rows);
            lo = row_a * C;
            hi = row_b * C;
        } else {
            const uint32_t *up = s ? up1 : up0;
            uint32_t jl = 0, jh = n_act - 1;   // largest j with up[j] <= lu
            while (jl < jh) {
                const uint32_t mid = (jl + jh + 1) >> 1;
                if ((uint64_t)up[mid] <= lu) jl = mid; else jh = mid - 1;
            }
            const uint64_t e = act[jl];
            const uint64_t R = (uint64_t)S.R;
            const uint64_t k = lu - up[jl];
            cnt = min(lend, (uint64_t)up[jl + 1]) - lu;
            const uint64_t first_unit = (e * R) / rb;
            row_a = (first_unit + k) * rb;
            row_b = min((first_unit + k + cnt) * rb, S.rows);
            lo = max(row_a, e * R) * C;
            hi = min(row_b, (e + 1) * R) * C;
        }
        if (S.kind == CSF_NVFP4)
            segment_nvfp4<2>(S, row_a, row_b, lo, hi, lane);
        else
            segment_mxfp4<1>(S, row_a, row_b, lo, hi, lane);
        u += cnt;
    }
}

}  // namespace

cudaError_t decode_occupancy(bool routed, size_t smem, int *blocks_per_sm) {
    if (routed)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel<true>, kThreads, smem);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel<false>, kThreads, smem);
}

cudaError_t launch_decode(const DecParams &p, int grid, size_t smem, bool routed, cudaStream_t s) {
    if (routed) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
        }
        decode_kernel<true><<<grid, kThreads, smem, s>>>(p);
    } else {
        decode_kernel<false><<<grid, kThreads, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace csfk
