// CSF prepare kernels for sm_103a: encode a dense stack (base byte per row,
// offset / escape planes, exception index, exception stream).
//
// Pages followed (cited by title and paragraph; no numbered sections):
//   "finegrained-kernels: decode losslessly compressed NVFP4 scales (CSF)":
//     format paragraph (base byte per row, most scales as 4-bit offsets,
//     out-of-range values in an exception stream); helpers paragraph
//     (preparation keeps the input device).
//   "Load native FP4 experts with optional lossless CSF scales": encoding plus
//     exception index built on the GPU at preparation time.
//   "NVFP4-CSF: expand_scales() for ahead-of-call scale expansion (canonical
//     twin of #477)": commit message on one-bit MXFP4 and four-bit NVFP4
//     offsets from a row base byte.
//
// Base rule (the pages do not give one; plainest reading that minimises the
// exception stream): the smallest byte value present in the row whose window
// [v, v+w] (w = 14 NVFP4, 1 MXFP4) holds the most of the row's bytes.
//
// Rows of up to 255 bytes (every workload of the pages) take one pass per
// 128-row tile that writes each tile's exception bytes to a slot of the
// scratch, then a kernel that places the slots in the stream; with a smaller
// scratch, a base kernel and an encode kernel (see the row-wise section
// below).  No block waits on another.  Wider rows take one single-pass kernel
// (prepare_kernel): per tile of rows, one warp per row picks the base from a
// 256-bin histogram, all threads pack the planes, and a block scan of the
// exception counts is chained to the earlier tiles by a decoupled look-back
// (Merrill & Garland, "Single-pass Parallel Prefix Scan with Decoupled
// Look-back", 2016) over per-tile status words in caller scratch; tiles take
// ids from a ticket counter in start order, so a block only waits on blocks
// already running, and every wait is bounded and reports
// CSF_DEV_ERR_TIMEOUT instead of hanging.
#include <cstring>

#include "csf_internal.cuh"

namespace csfk {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr unsigned long long kFlagAgg = 1ull << 62;
constexpr unsigned long long kFlagIncl = 2ull << 62;
constexpr unsigned long long kValMask = (1ull << 62) - 1;
constexpr uint32_t kSpinLimit = 1u << 22;   // polls before a look-back wait gives up (default)

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

__device__ __forceinline__ unsigned long long warp_sum64(unsigned long long v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void flag(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}


// Decoupled look-back (whole warp): publish this tile's exception total, then
// walk back over earlier tiles' status words until an inclusive prefix is
// found; publish this tile's inclusive prefix and return its exclusive one.
// Tiles take ids from a ticket counter in start order, so every tile waited on
// belongs to a block that is already running; each wait is bounded and sets
// CSF_DEV_ERR_TIMEOUT instead of hanging.
__device__ unsigned long long lookback_exclusive(const PrepParams &P, uint64_t tile, unsigned long long total,
                                                 int lane) {
    unsigned long long excl = 0;
    bool timed_out = false;
    if (lane == 0) st_release(&P.status[tile], (tile == 0 ? kFlagIncl : kFlagAgg) | total);
    if (tile > 0) {
        long long j = (long long)tile - 1;
        while (true) {
            const long long idx = j - lane;
            unsigned long long v = kFlagIncl;   // before tile 0: inclusive zero
            if (idx >= 0) {
                v = ld_acquire(&P.status[idx]);
                uint32_t spins = 0;
                while ((v >> 62) == 0) {
                    if (++spins > P.spin_limit) { timed_out = true; v = kFlagAgg; break; }
                    __nanosleep(64);
                    v = ld_acquire(&P.status[idx]);
                }
            }
            const uint32_t incl = __ballot_sync(kFull, (v >> 62) == 2);
            unsigned long long val = v & kValMask;
            if (incl) {
                const int first = __ffs(incl) - 1;
                if (lane > first) val = 0;
                excl += warp_sum64(val);
                break;
            }
            excl += warp_sum64(val);
            j -= 32;
        }
        if (lane == 0) st_release(&P.status[tile], kFlagIncl | (excl + total));
    }
    if (__any_sync(kFull, timed_out) && lane == 0) flag(P.err, CSF_DEV_ERR_TIMEOUT);
    return excl;
}

__global__ void __launch_bounds__(kThreads) prepare_kernel(const __grid_constant__ PrepParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ unsigned int s_tile;
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_wsum[kWarps];
    __shared__ uint32_t s_total;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int tr = P.tr;
    const uint32_t C = (uint32_t)P.C;
    const bool nv = P.kind == CSF_NVFP4;
    const int wwin = nv ? 14 : 1;

    uint8_t *s_dense = smem;
    uint8_t *s_planes = smem + P.smem_dense;
    uint32_t *s_hist = reinterpret_cast<uint32_t *>(s_planes + P.smem_planes);
    uint32_t *s_cnt = s_hist + kWarps * 256;
    uint8_t *s_base = reinterpret_cast<uint8_t *>(s_cnt + tr);

    if (tid == 0) s_tile = atomicAdd(P.ticket, 1u);
    __syncthreads();
    const uint64_t tile = s_tile;
    if (tile >= P.num_tiles) return;   // grid == num_tiles, so every ticket is a tile
    const uint64_t r0 = tile * (uint64_t)tr;
    const uint64_t r1 = min(r0 + (uint64_t)tr, P.rows);
    const int nr = (int)(r1 - r0);
    const uint64_t e0 = r0 * C;
    const uint32_t ne = (uint32_t)nr * C;

    // 1. Stage the tile's dense bytes.
    {
        const uint8_t *src = P.dense + e0;
        uint32_t done = 0;
        if (P.dense_aligned) {
            const uint32_t n16 = ne / 16;
            for (uint32_t i = tid; i < n16; i += kThreads)
                reinterpret_cast<uint4 *>(s_dense)[i] = __ldg(reinterpret_cast<const uint4 *>(src) + i);
            done = n16 * 16;
        }
        for (uint32_t i = done + tid; i < ne; i += kThreads) s_dense[i] = __ldg(src + i);
    }
    __syncthreads();

    // 2. Base byte and exception count of each row (one warp per row).
    uint32_t *hist = s_hist + warp * 256;
    for (int k = warp; k < nr; k += kWarps) {
        const uint8_t *x = s_dense + (uint32_t)k * C;
        reinterpret_cast<uint4 *>(hist)[2 * lane] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(hist)[2 * lane + 1] = make_uint4(0, 0, 0, 0);
        __syncwarp();
        for (uint32_t c = lane; c < C; c += 32) atomicAdd(&hist[x[c]], 1u);
        __syncwarp();
        uint32_t h[8];
        {
            const uint4 a = reinterpret_cast<const uint4 *>(hist)[2 * lane];
            const uint4 b = reinterpret_cast<const uint4 *>(hist)[2 * lane + 1];
            h[0] = a.x; h[1] = a.y; h[2] = a.z; h[3] = a.w;
            h[4] = b.x; h[5] = b.y; h[6] = b.z; h[7] = b.w;
        }
        uint32_t key = 0;
        if (nv) {
            // Inclusive prefix over the 256 bins; window count of v is
            // P[min(v+14, 255)] - P[v] + h[v].
            uint32_t pre[8];
            uint32_t run = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { run += h[j]; pre[j] = run; }
            uint32_t tot;
            const uint32_t ex = warp_excl_scan(run, lane, tot);
#pragma unroll
            for (int j = 0; j < 8; ++j) pre[j] += ex;
            __syncwarp();
            reinterpret_cast<uint4 *>(hist)[2 * lane] = make_uint4(pre[0], pre[1], pre[2], pre[3]);
            reinterpret_cast<uint4 *>(hist)[2 * lane + 1] = make_uint4(pre[4], pre[5], pre[6], pre[7]);
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t v = 8u * lane + j;
                const uint32_t top = min(v + 14u, 255u);
                const uint32_t wcount = hist[top] - (pre[j] - h[j]);
                if (h[j]) key = max(key, (wcount << 8) | (255u - v));
            }
        } else {
            uint32_t nxt = __shfl_down_sync(kFull, h[0], 1);
            if (lane == 31) nxt = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t v = 8u * lane + j;
                const uint32_t wcount = h[j] + (j < 7 ? h[j + 1] : nxt);
                if (h[j]) key = max(key, (wcount << 8) | (255u - v));
            }
        }
        key = __reduce_max_sync(kFull, key);
        if (lane == 0) {
            s_base[k] = (uint8_t)(255u - (key & 0xFFu));
            s_cnt[k] = C - (key >> 8);
        }
        __syncwarp();
    }
    __syncthreads();

    // 3. Pack the planes of the tile (pad bits past the stack end are 0).
    if (nv) {
        const uint32_t nbytes = ((ne + 1) / 2 + 15) & ~15u;
        for (uint32_t wi = tid; wi < nbytes / 4; wi += kThreads) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t el = wi * 8 + j;
                if (el < ne) {
                    const uint32_t row = (uint32_t)(((uint64_t)el * P.magic) >> 40);
                    const uint32_t b = s_base[row];
                    const uint32_t xv = s_dense[el];
                    const uint32_t d = xv - b;
                    const uint32_t nib = (xv >= b && d <= 14u) ? d : 15u;
                    word |= nib << (4 * j);
                }
            }
            reinterpret_cast<uint32_t *>(s_planes)[wi] = word;
        }
    } else {
        const uint32_t nbytes = ((ne + 7) / 8 + 15) & ~15u;
        uint32_t *po = reinterpret_cast<uint32_t *>(s_planes);
        uint32_t *pe = reinterpret_cast<uint32_t *>(s_planes + nbytes);
        for (uint32_t wi = tid; wi < nbytes / 4; wi += kThreads) {
            uint32_t ow = 0, xw = 0;
            const uint32_t el0 = wi * 32;
            if (el0 < ne) {
                uint32_t row = (uint32_t)(((uint64_t)el0 * P.magic) >> 40);
                uint32_t next = (row + 1) * C;
                uint32_t b = s_base[row];
#pragma unroll 4
                for (int j = 0; j < 32; ++j) {
                    const uint32_t el = el0 + j;
                    if (el < ne) {
                        if (el == next) { ++row; next += C; b = s_base[row]; }
                        const uint32_t xv = s_dense[el];
                        const uint32_t d = xv - b;
                        const bool inside = xv >= b && d <= 1u;
                        ow |= (inside ? d : 0u) << j;
                        xw |= (inside ? 0u : 1u) << j;
                    }
                }
            }
            po[wi] = ow;
            pe[wi] = xw;
        }
    }

    // 4a. Block-wide exclusive scan of the per-row counts (in place).
    const int per = (nr + kThreads - 1) / kThreads;
    const int k0 = min(tid * per, nr);
    const int k1 = min(k0 + per, nr);
    uint32_t local = 0;
    for (int k = k0; k < k1; ++k) local += s_cnt[k];
    uint32_t wtot;
    const uint32_t wex = warp_excl_scan(local, lane, wtot);
    if (lane == 0) s_wsum[warp] = wtot;
    __syncthreads();
    uint32_t boff = 0, btot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) boff += s_wsum[w];
        btot += s_wsum[w];
    }
    {
        uint32_t run = boff + wex;
        for (int k = k0; k < k1; ++k) {
            const uint32_t c = s_cnt[k];
            s_cnt[k] = run;
            run += c;
        }
    }
    if (tid == 0) s_total = btot;

    // 4b. Decoupled look-back across tiles (warp 0).
    if (warp == 0) {
        const unsigned long long excl = lookback_exclusive(P, tile, btot, lane);
        if (lane == 0) s_excl = excl;
    }
    __syncthreads();
    const unsigned long long excl = s_excl;

    // 5. Outputs.
    for (int k = tid; k < nr; k += kThreads) {
        const unsigned long long v = excl + s_cnt[k];
        P.exc_index[r0 + k] = (uint32_t)v;
        P.base[r0 + k] = s_base[k];
    }
    if (tile == P.num_tiles - 1 && tid == 0) {
        const unsigned long long all = excl + s_total;
        P.exc_index[P.rows] = (uint32_t)all;
        if (all > 0xFFFFFFFFull) flag(P.err, CSF_DEV_ERR_CAPACITY);
    }
    if (nv) {
        const uint32_t nbytes = ((ne + 1) / 2 + 15) & ~15u;
        uint4 *dst = reinterpret_cast<uint4 *>(P.offsets + e0 / 2);
        for (uint32_t i = tid; i < nbytes / 16; i += kThreads) dst[i] = reinterpret_cast<const uint4 *>(s_planes)[i];
    } else {
        const uint32_t nbytes = ((ne + 7) / 8 + 15) & ~15u;
        uint4 *dso = reinterpret_cast<uint4 *>(P.offsets + e0 / 8);
        uint4 *dse = reinterpret_cast<uint4 *>(P.escapes + e0 / 8);
        for (uint32_t i = tid; i < nbytes / 16; i += kThreads) {
            dso[i] = reinterpret_cast<const uint4 *>(s_planes)[i];
            dse[i] = reinterpret_cast<const uint4 *>(s_planes + nbytes)[i];
        }
    }
    // Exception bytes, row-major, at excl + row prefix + rank in row.
    bool over = false;
    for (int k = warp; k < nr; k += kWarps) {
        const uint8_t *x = s_dense + (uint32_t)k * C;
        const uint32_t b = s_base[k];
        unsigned long long run = excl + s_cnt[k];
        for (uint32_t c0 = 0; c0 < C; c0 += 32) {
            const uint32_t c = c0 + lane;
            bool esc = false;
            uint32_t xv = 0;
            if (c < C) {
                xv = x[c];
                const uint32_t d = xv - b;
                esc = !(xv >= b && d <= (uint32_t)wwin);
            }
            const uint32_t bal = __ballot_sync(kFull, esc);
            if (esc) {
                const unsigned long long pos = run + __popc(bal & lanemask_lt());
                if (pos < P.exc_capacity) P.exc_bytes[pos] = (uint8_t)xv;
                else over = true;
            }
            run += __popc(bal);
        }
    }
    if (__any_sync(kFull, over) && lane == 0) flag(P.err, CSF_DEV_ERR_CAPACITY);
}


// ---------------------------------------------------------------- row-wise
//
// Rows of C <= 255 bytes are prepared without any wait between blocks.  The
// exception stream needs every tile's position, which depends on the
// exception counts of all earlier tiles; a single pass would make each tile
// wait for the slowest of the hundreds of tiles in flight before it (a
// decoupled look-back measured 20 us of the gate stack's 78 us this way).
// Fused path (the scratch holds a slot of 128 * C bytes per tile):
//   fused kernel   per tile: each row's base, the planes, each row's place
//                  inside the tile (exc_index[]), the tile's exception bytes
//                  in its slot and its total.
//   place kernel   per tile: its offset in the stream (the sum of the
//                  earlier totals) added to its rows' exc_index entries, and
//                  its slot copied into the stream.
// Two-kernel path (a scratch of 8 bytes per tile):
//   base kernel    per row: base byte and exception count (into base[] and,
//                  for now, exc_index[]); per tile: its exception total.
//   encode kernel  per tile: its offset in the exception stream (the sum of
//                  the earlier tiles' totals), the rows' exc_index entries
//                  (offset + block scan of the counts), the offset / escape
//                  planes, and the exception bytes written straight to their
//                  final positions.
// The fused, base and encode kernels are persistent: block b takes tiles b,
// b + G, b + 2G, ... (G = grid), staging each tile in shared memory with bulk
// copies while it works on the one before.

// Rows (and threads) per block; a multiple of every chunk-alignment row count
// (it divides into 32 and 128-element pieces), so each tile's planes start on
// a 16-byte boundary.
constexpr int kRowTile = 128;
// NVFP4 base search: a relative histogram of the row, with bins for the
// values [a, a + 32) around the row's anchor a = median - 16 and one bin for
// every byte outside them (windows span 15 values: 32 bins hold them with
// room on both sides).  MXFP4 windows span 2 values: the row's counts of
// the three values a, a + 1, a + 2 around a = median - 1 decide it (no bins).
template <int KIND> struct Bins {
    static constexpr int n = KIND == CSF_NVFP4 ? 32 : 8;
    static constexpr int lead = KIND == CSF_NVFP4 ? 16 : 1;   // anchor = median - lead
};
constexpr uint32_t kH = 0x80808080u;   // bit 7 of each byte

// How a thread reads its row's 4-byte words from the staged tile.
enum RowRead { kRdWord = 0, kRdVec = 1, kRdShift = 2 };
// How a tile is staged in shared memory.
enum Stage { kStagePlain = 0, kStageTile = 1 };

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// One bulk copy global -> this block's shared memory (both 16-byte aligned,
// `bytes` a multiple of 16), completing on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// its later bulk copies into it.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Polls of a staging buffer's barrier before the wait gives up, and how long
// each poll may suspend the thread (ns) while the copies are in flight, so
// that waiting threads sleep instead of spinning.
constexpr uint32_t kMbarPolls = 1u << 16;
constexpr uint32_t kMbarSuspendNs = 20000;

__device__ __forceinline__ bool mbar_done(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kMbarSuspendNs)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase `parity` of a staging buffer's barrier; false
// when the polls ran out (about a second).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kMbarPolls; ++i)
        if (mbar_done(bar, parity)) return true;
    return false;
}

// Median of five bytes: the two middle values of the first four are
// max(min(p0,p1), min(p2,p3)) and min(max(p0,p1), max(p2,p3)); the median of
// all five is the median of those two and p4.
__device__ __forceinline__ uint32_t median5(uint32_t p0, uint32_t p1, uint32_t p2, uint32_t p3, uint32_t p4) {
    const uint32_t e = max(min(p0, p1), min(p2, p3));
    const uint32_t f = min(max(p0, p1), max(p2, p3));
    return max(min(p4, e), min(max(p4, e), f));
}

// 0xFF in each byte whose bit 7 is set in `f`, 0x00 in the others (the other
// bits of f are ignored): a byte permute whose selector nibbles 8..B pick
// bytes 0..3 and replicate their sign bit.  (PTX prmt; CUDA's __byte_perm
// keeps only the low 3 bits of each selector nibble, so it cannot do this.)
__device__ __forceinline__ uint32_t byte_mask(uint32_t f) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(f), "r"(0xBA98u));
    return r;
}

// Byte-wise x - b (mod 256 in each byte, no borrow across bytes) and, in bit
// 7 of each byte of `below`, whether that byte of x is below b.
__device__ __forceinline__ uint32_t sub_bytes(uint32_t x, uint32_t B, uint32_t &below) {
    const uint32_t d = ((x | kH) - (B & ~kH)) ^ ((x ^ ~B) & kH);
    below = (~x & B) | (~(x ^ B) & d);   // borrow out of bit 7 of each byte
    return d;
}

// The row's 4-byte words, read from its staged copy in shared memory.
template <int RD>
struct RowWords {
    const uint32_t *w;   // kRdShift: the aligned word at or below the row start
    uint32_t sh;         // kRdShift: 8 * (row start % 4)
    __device__ __forceinline__ explicit RowWords(const uint8_t *r) {
        // rounded down by pointer arithmetic (not through an integer), so the
        // loads stay shared-memory loads
        const uint32_t m = (uint32_t)reinterpret_cast<uintptr_t>(r) & 3u;
        w = reinterpret_cast<const uint32_t *>(r - m);
        sh = 8u * m;
    }
    // word k (bytes 4k .. 4k+3 of the row); kRdShift reads one word past them
    __device__ __forceinline__ uint32_t word(uint32_t k) const {
        if (RD == kRdShift) return __funnelshift_r(w[k], w[k + 1], sh);
        return w[k];
    }
    // words 8g .. 8g+7
    __device__ __forceinline__ void group(uint32_t g, uint32_t (&x)[8]) const {
        if (RD == kRdVec) {
            const uint4 a = reinterpret_cast<const uint4 *>(w)[2 * g];
            const uint4 b = reinterpret_cast<const uint4 *>(w)[2 * g + 1];
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        } else if (RD == kRdWord) {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = w[8 * g + j];
        } else {
            uint32_t y[9];
#pragma unroll
            for (int j = 0; j < 9; ++j) y[j] = w[8 * g + j];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = __funnelshift_r(y[j], y[j + 1], sh);
        }
    }
};

// The row's relative histogram: four bytes of a word into the bins of this
// thread's column (word-sized counters, bank = thread, no conflicts).
template <int NB>
__device__ __forceinline__ void hist_word(uint32_t *hcol, uint32_t x, uint32_t A4) {
    constexpr uint32_t kNB4 = (uint32_t)NB * 0x01010101u;
    uint32_t below;
    const uint32_t d = sub_bytes(x, A4, below);
    // d >= NB in a byte (bit 7): outside [a, a + NB) (bytes below a wrap past NB, a <= 256 - NB)
    const uint32_t out = ((d | kH) - kNB4) | d;
    const uint32_t m = byte_mask(out);                            // 0xFF in each outside byte
    const uint32_t bins = (d & ~m) | (kNB4 & m);                  // bin NB = outside
    atomicAdd(hcol + (bins & 0xFFu) * kRowTile, 1u);
    atomicAdd(hcol + __byte_perm(bins, 0, 0x4441) * kRowTile, 1u);
    atomicAdd(hcol + __byte_perm(bins, 0, 0x4442) * kRowTile, 1u);
    atomicAdd(hcol + (bins >> 24) * kRowTile, 1u);
}

template <int NB>
__device__ __forceinline__ void hist_byte(uint32_t *hcol, uint32_t v, uint32_t a) {
    const uint32_t d = v - a;   // below a: wraps far above NB
    atomicAdd(hcol + min(d, (uint32_t)NB) * kRowTile, 1u);
}

// MXFP4: counts of the row's bytes in [a, a + 1), [a, a + 2) and [a, a + 3)
// from one word (A4 = a in every byte).  Bytes below a wrap to at least
// 256 - a >= 3 (a <= 253), so they are never counted.
__device__ __forceinline__ void count3_word(uint32_t x, uint32_t A4, uint32_t &n1, uint32_t &n2, uint32_t &n3) {
    uint32_t below;
    const uint32_t d = sub_bytes(x, A4, below);
    const uint32_t dh = d | kH;
    // d < k in a byte: bit 7 clear both in d and in (d | 0x80) - k
    n1 += __popc(~(dh - 0x01010101u) & ~d & kH);
    n2 += __popc(~(dh - 0x02020202u) & ~d & kH);
    n3 += __popc(~(dh - 0x03030303u) & ~d & kH);
}

// MXFP4 base rule from the counts c0, c1, c2 of the values a, a + 1, a + 2
// (a <= 253): the better of the windows [a, a + 1] and [a + 1, a + 2] (each
// only if its first value is present), when a bound proves it the best of
// the row.  Windows [v, v + 1] with v < a hold at most one of the counted
// values, a: at most C - c1 - c2 bytes, which must be fewer than the best
// (ties go to the smaller value); windows with v > a + 1 hold at most a + 2:
// at most C - c0 - c1, which may equal it.  Returns the packed key
// (count << 8) | (255 - base), 0 when the proof fails.
__device__ __forceinline__ uint32_t count3_key(uint32_t C, uint32_t a, uint32_t c0, uint32_t c1, uint32_t c2) {
    uint32_t best = 0;
    if (c0) best = ((c0 + c1) << 8) | (255u - a);
    if (c1) best = max(best, ((c1 + c2) << 8) | (254u - a));
    const uint32_t M = best >> 8;
    const bool ok_low = a == 0 || C - c1 - c2 < M;
    const bool ok_high = C - c0 - c1 <= M;
    return ok_low && ok_high ? best : 0u;
}

// Base rule on the relative histogram h[0..n] (h[n] = bytes outside
// [a, a + n)): the best window among those lying inside the bins, and
// whether that is provably the best window of the whole row.  Returns the
// packed key (count << 8) | (255 - base), 0 when the proof fails.
//   Windows [v, v + w] with v < a hold at most out + (bytes in [a, a + w))
//   (they reach at most w - 1 values into the bins); windows past the bins'
//   exact range hold at most out + (bytes in the last w bins).  A lower
//   window must hold strictly fewer bytes than the best (ties go to the
//   smaller value), a higher one at most as many.
template <int KIND>
__device__ __forceinline__ uint32_t window_key(const uint32_t *hcol, uint32_t a) {
    constexpr int w = KIND == CSF_NVFP4 ? 14 : 1;
    constexpr int kBins = Bins<KIND>::n;
    constexpr int jmax = kBins - 1 - w;               // last window that lies inside the bins
    uint32_t h[Bins<KIND>::n + 1];
#pragma unroll
    for (int i = 0; i <= Bins<KIND>::n; ++i) h[i] = hcol[i * kRowTile];
    const uint32_t out = h[kBins];
    const bool top = a + kBins == 256;                // the bins reach 255: every window is exact
    uint32_t best = 0, S = 0, low = 0, hi = 0;
#pragma unroll
    for (int i = 0; i <= w; ++i) S += h[i];
#pragma unroll
    for (int i = 0; i < w; ++i) low += h[i];
#pragma unroll
    for (int i = kBins - w; i < kBins; ++i) hi += h[i];
#pragma unroll
    for (int j = 0; j <= jmax; ++j) {
        if (h[j]) best = max(best, (S << 8) | (255u - a - (uint32_t)j));
        if (j < jmax) S += h[j + w + 1] - h[j];
    }
    if (top) {
        // windows truncated at 255
        S -= h[jmax];
#pragma unroll
        for (int j = jmax + 1; j < kBins; ++j) {
            if (h[j]) best = max(best, (S << 8) | (255u - a - (uint32_t)j));
            S -= h[j];
        }
    }
    const uint32_t M = best >> 8;
    const bool ok_low = a == 0 || out + low < M;
    const bool ok_high = top || out + hi <= M;
    return ok_low && ok_high ? best : 0u;
}

// Exact base rule over all 256 values for one row, whole warp (the fallback
// when the relative histogram cannot prove its answer), in the warp's own
// columns of the bins; the row is read from global memory, so the staged
// tile may already be refilled.  Returns the packed key
// (count << 8) | (255 - base).
template <int KIND>
__device__ uint32_t exact_key(const uint8_t *__restrict__ row, uint32_t C, uint32_t *hist, int warp, int lane) {
    constexpr uint32_t w = KIND == CSF_NVFP4 ? 14u : 1u;
    auto at = [&](uint32_t v) -> uint32_t * { return hist + (v >> 5) * kRowTile + 32u * warp + (v & 31u); };
#pragma unroll
    for (int i = 0; i < 8; ++i) *at((uint32_t)lane + 32u * i) = 0;
    __syncwarp();
    for (uint32_t c = lane; c < C; c += 32) atomicAdd(at(__ldg(row + c)), 1u);
    __syncwarp();
    uint32_t hv[8], pre[8], run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        hv[j] = *at(8u * lane + j);
        run += hv[j];
        pre[j] = run;
    }
    uint32_t tot;
    const uint32_t ex = warp_excl_scan(run, lane, tot);
#pragma unroll
    for (int j = 0; j < 8; ++j) pre[j] += ex;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) *at(8u * lane + j) = pre[j];   // inclusive prefix P[v]
    __syncwarp();
    uint32_t key = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t v = 8u * lane + j;
        const uint32_t cnt = *at(min(v + w, 255u)) - (pre[j] - hv[j]);   // P[v + w] - P[v - 1]
        if (hv[j]) key = max(key, (cnt << 8) | (255u - v));
    }
    key = __reduce_max_sync(kFull, key);
    __syncwarp();
    return key;
}

// Tile staging shared by the two row kernels: rows of tile t land in a buffer
// at row * stride.  The bulk copy of a tile is issued by lane 0 of warp 0;
// with plain staging every thread loads.
__device__ __forceinline__ uint32_t tile_rows(const PrepParams &P, uint64_t t) {
    const uint64_t r0 = t * (uint64_t)kRowTile;
    return (uint32_t)(min(r0 + (uint64_t)kRowTile, P.rows) - r0);
}

__device__ __forceinline__ void stage_issue(const PrepParams &P, uint64_t t, uint8_t *dst, uint64_t *bar, int lane) {
    const uint32_t C = (uint32_t)P.C;
    const uint32_t nb = (tile_rows(P, t) * C) & ~15u;   // the last tile's tail (< 16 bytes) is loaded plainly
    if (lane == 0) {
        fence_proxy_async();
        mbar_expect(bar, nb);
        if (nb) bulk_load(dst, P.dense + t * (uint64_t)kRowTile * C, nb, bar);
    }
}

// Makes tile t's rows available in `dst` (whole block): plain loads, or the
// bulk copies' completion (phase `parity` of `bar`) plus the tail of a packed
// last tile.
__device__ __forceinline__ void stage_wait(const PrepParams &P, uint64_t t, uint8_t *dst, uint64_t *bar,
                                           uint32_t parity, int tid) {
    const uint32_t C = (uint32_t)P.C;
    const uint32_t ne = tile_rows(P, t) * C;
    const uint8_t *src = P.dense + t * (uint64_t)kRowTile * C;
    if (P.stage == kStagePlain) {
        uint32_t done = 0;
        if (P.dense_aligned) {
            const uint32_t n16 = ne / 16;
            for (uint32_t i = tid; i < n16; i += kRowTile)
                reinterpret_cast<uint4 *>(dst)[i] = __ldg(reinterpret_cast<const uint4 *>(src) + i);
            done = n16 * 16;
        }
        for (uint32_t i = done + tid; i < ne; i += kRowTile) dst[i] = __ldg(src + i);
        __syncthreads();
        return;
    }
    if (P.stage == kStageTile && (ne & 15u) != 0) {
        for (uint32_t i = (ne & ~15u) + tid; i < ne; i += kRowTile) dst[i] = __ldg(src + i);
        __syncthreads();
    }
    if (!mbar_wait(bar, parity)) {
        flag(P.err, CSF_DEV_ERR_TIMEOUT);
        mbar_wait(bar, parity);   // let copies in flight land before going on
    }
}

// First pass over a staged row for its base: NVFP4 rows are histogrammed
// into 32 bins around the median of five of their bytes (bins in the
// thread's column `hcol`); MXFP4 rows count the three values around that
// median (n1, n2, n3: bytes in [a, a+1), [a, a+2), [a, a+3)).  Returns the
// anchor a.
template <int KIND, int RD>
__device__ __forceinline__ uint32_t row_scan(const uint8_t *rowb, uint32_t C, uint32_t *hcol, uint32_t &n1,
                                             uint32_t &n2, uint32_t &n3) {
    constexpr int NB = Bins<KIND>::n;
    const uint32_t nw = C / 4;   // whole words of the row
    const uint32_t med = median5(rowb[0], rowb[C / 4], rowb[C / 2], rowb[(3 * C) / 4], rowb[C - 1]);
    const RowWords<RD> rw(rowb);
    uint32_t a;
    if constexpr (KIND == CSF_NVFP4) {
#pragma unroll
        for (int i = 0; i <= Bins<KIND>::n; ++i) hcol[i * kRowTile] = 0;
        a = min(max((int)med - Bins<KIND>::lead, 0), 256 - NB);
        const uint32_t A4 = a * 0x01010101u;
        for (uint32_t g = 0; g < nw / 8; ++g) {
            uint32_t x[8];
            rw.group(g, x);
#pragma unroll
            for (int j = 0; j < 8; ++j) hist_word<NB>(hcol, x[j], A4);
        }
        for (uint32_t q = nw & ~7u; q < nw; ++q) hist_word<NB>(hcol, rw.word(q), A4);
        for (uint32_t c = 4 * nw; c < C; ++c) hist_byte<NB>(hcol, rowb[c], a);
    } else {
        a = min(max((int)med - Bins<KIND>::lead, 0), 253);
        const uint32_t A4 = a * 0x01010101u;
        for (uint32_t g = 0; g < nw / 8; ++g) {
            uint32_t x[8];
            rw.group(g, x);
#pragma unroll
            for (int j = 0; j < 8; ++j) count3_word(x[j], A4, n1, n2, n3);
        }
        for (uint32_t q = nw & ~7u; q < nw; ++q) count3_word(rw.word(q), A4, n1, n2, n3);
        for (uint32_t c = 4 * nw; c < C; ++c) {
            const uint32_t d = (uint32_t)rowb[c] - a;   // below a: wraps far above 3
            n1 += d < 1u;
            n2 += d < 2u;
            n3 += d < 3u;
        }
    }
    return a;
}

// The row's base key (count << 8) | (255 - base) from its first pass when a
// bound proves it (window_key, count3_key), else 0.
template <int KIND>
__device__ __forceinline__ uint32_t row_fast_key(const uint32_t *hcol, uint32_t C, uint32_t a, uint32_t n1,
                                                 uint32_t n2, uint32_t n3) {
    if constexpr (KIND == CSF_NVFP4) return window_key<KIND>(hcol, a);
    else return count3_key(C, a, n1, n2 - n1, n3 - n2);
}

// Rows of the warp whose key is 0 (no proof): their warp applies the exact
// rule over all 256 values, one row at a time, reading the row from global
// memory (row0 = the row of lane 0).  Whole warp; uses the warp's columns of
// the bins.
template <int KIND>
__device__ __forceinline__ uint32_t settle_keys(const PrepParams &P, uint32_t key, bool mine, uint64_t row0,
                                                uint32_t *s_hist, int warp, int lane) {
    const uint32_t C = (uint32_t)P.C;
    uint32_t redo = __ballot_sync(kFull, mine && key == 0);
    while (redo) {
        const int src_lane = __ffs(redo) - 1;
        redo &= redo - 1;
        const uint32_t k2 = exact_key<KIND>(P.dense + (row0 + (uint64_t)src_lane) * C, C, s_hist, warp, lane);
        if (lane == src_lane) key = k2;
    }
    return key;
}

// Encodes one staged row against its base: its codes go into the tile's
// planes in shared memory (s_planes: NVFP4 nibbles, or MXFP4 offset bits
// then escape bits in the second half; the row starts at tile element el0)
// and its exception bytes to positions pos, pos + 1, ... of `stage` (shared
// memory) when `staged`, else of `gdst` (global memory, `gcap` bytes
// available: later bytes are dropped and `over` set).  Word by word:
// byte-wise subtract, range test, nibble or bit gather; escape positions are
// taken 8 words at a time and walked in element order.  LOW: the base is at
// most 241 (NVFP4) or 254 (MXFP4), so a byte below it wraps to at least
// w + 1 in the byte-wise subtract and needs no test of its own.  Returns the
// position after the row's last exception.
template <int KIND, int RD, bool LOW>
__device__ __forceinline__ uint32_t encode_row(const uint8_t *rowb, uint32_t C, uint32_t base, uint32_t el0,
                                               uint8_t *s_planes, uint32_t planes_bytes, uint8_t *stage, bool staged,
                                               uint8_t *gdst, uint64_t gcap, uint32_t pos, bool &over) {
    const uint32_t nw = C / 4;                       // whole words of the row
    const uint32_t tailn = C & 3u;                   // kRdShift only
    const uint32_t B4 = base * 0x01010101u;
    const RowWords<RD> rw(rowb);
    uint32_t *pw = reinterpret_cast<uint32_t *>(s_planes);
    uint32_t *px = reinterpret_cast<uint32_t *>(s_planes + planes_bytes / 2);
    // the exception bytes of the 8 words from word k0 on: bit 4j + i of
    // `em` = byte i of word j (bit order = element order)
    auto emit = [&](uint32_t em, uint32_t k0) {
        const uint8_t *src = rowb + 4 * k0;
        if (staged && KIND == CSF_MXFP4) {
            // dense exceptions: two a trip, their loads issued together
            while (em) {
                const uint32_t i0 = (uint32_t)(__ffs(em) - 1);
                em &= em - 1;
                const bool two_more = em != 0;
                const uint32_t i1 = two_more ? (uint32_t)(__ffs(em) - 1) : i0;
                em &= em - 1;
                const uint8_t v0 = src[i0], v1 = src[i1];
                stage[pos] = v0;
                if (two_more) stage[pos + 1] = v1;
                pos += two_more ? 2u : 1u;
            }
        } else if (staged) {
            while (em) {
                const uint32_t i = (uint32_t)(__ffs(em) - 1);
                em &= em - 1;
                stage[pos++] = src[i];
            }
        } else {
            while (em) {
                const uint32_t i = (uint32_t)(__ffs(em) - 1);
                em &= em - 1;
                if (pos < gcap) gdst[pos] = src[i];
                else over = true;
                ++pos;
            }
        }
    };
    constexpr uint32_t kW1 = KIND == CSF_NVFP4 ? 0x0F0F0F0Fu : 0x02020202u;   // (w + 1) per byte
    // codes of word k (bytes x; `valid` masks the bytes of a tail word)
    // and its escape nibble (bit i = byte i outside [b, b + w])
    auto code = [&](uint32_t x, uint32_t valid, uint32_t &ob4) -> uint32_t {
        uint32_t below;
        const uint32_t d = sub_bytes(x, B4, below);
        const uint32_t wrapped = LOW ? 0u : below;
        const uint32_t o = ((((d | kH) - kW1) | d | wrapped) & kH) & valid;
        const uint32_t m = byte_mask(o);
        if (KIND == CSF_NVFP4) {
            const uint32_t c = ((d & ~m) | (0x0F0F0F0Fu & m)) & valid;
            const uint32_t t = c | (c >> 4);
            ob4 = __byte_perm(t, 0, 0x4420);                                // 4 nibbles
        } else {
            ob4 = (((d & ~m) & 0x01010101u & valid) * 0x10204080u) >> 28;  // 4 offset bits
        }
        return (o * 0x00204081u) >> 28;
    };
    auto store_nv = [&](uint32_t k, uint32_t cd) {
        const uint32_t el = el0 + 4 * k;
        if (RD != kRdShift) {
            reinterpret_cast<uint16_t *>(s_planes)[el >> 2] = (uint16_t)cd;
        } else {
            const uint32_t sh = 4 * (el & 7u);
            atomicOr(pw + (el >> 3), cd << sh);
            if (sh > 16 && (cd >> (32 - sh)) != 0) atomicOr(pw + (el >> 3) + 1, cd >> (32 - sh));
        }
    };
    auto store_mx = [&](uint32_t el, uint32_t o, uint32_t e, uint32_t bits) {   // `bits` bits at element el
        const uint32_t sh = el & 31u;
        if (o) atomicOr(pw + (el >> 5), o << sh);
        if (e) atomicOr(px + (el >> 5), e << sh);
        if (sh + bits > 32) {
            if (o >> (32 - sh)) atomicOr(pw + (el >> 5) + 1, o >> (32 - sh));
            if (e >> (32 - sh)) atomicOr(px + (el >> 5) + 1, e >> (32 - sh));
        }
    };
    for (uint32_t g = 0; g < nw / 8; ++g) {
        uint32_t x[8];
        rw.group(g, x);
        uint32_t em = 0, ow = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t cd;
            const uint32_t e4 = code(x[j], 0xFFFFFFFFu, cd);
            em |= e4 << (4 * j);
            if (KIND == CSF_NVFP4) store_nv(8 * g + j, cd);
            else ow |= cd << (4 * j);
        }
        if (KIND == CSF_MXFP4) {
            const uint32_t el = el0 + 32 * g;
            if (RD != kRdShift && (el & 31u) == 0) {
                pw[el >> 5] = ow;
                px[el >> 5] = em;
            } else {
                store_mx(el, ow, em, 32);
            }
        }
        if (em) emit(em, 8 * g);
    }
    // remaining whole words and the tail word, in one last group
    uint32_t em = 0;
    const uint32_t k0 = nw & ~7u;
    for (uint32_t q = k0; q < nw + (tailn ? 1u : 0u); ++q) {
        const uint32_t valid = q < nw ? 0xFFFFFFFFu : 0xFFFFFFFFu >> (32 - 8 * tailn);
        uint32_t cd;
        const uint32_t e4 = code(rw.word(q), valid, cd);
        em |= e4 << (4 * (q - k0));
        if (KIND == CSF_NVFP4) store_nv(q, cd);
        else store_mx(el0 + 4 * q, cd, e4, 4);
    }
    emit(em, k0);
    return pos;
}

// Highest base for which no byte below it can wrap into its window in the
// byte-wise subtract (base + w + 1 <= 256).
template <int KIND>
__device__ __forceinline__ constexpr uint32_t low_base() { return KIND == CSF_NVFP4 ? 241u : 254u; }

// Writes the tile's planes from shared memory to the stack (16-byte pieces;
// the tile starts at element e0 on a 16-byte boundary of each plane) and,
// when `clear`, zeroes them for the next tile.  Whole block.
template <int KIND>
__device__ __forceinline__ void write_planes(const PrepParams &P, uint8_t *s_planes, uint64_t e0, uint32_t nr,
                                             bool clear, int tid) {
    const uint32_t C = (uint32_t)P.C;
    if (KIND == CSF_NVFP4) {
        const uint32_t nbytes = ((nr * C + 1) / 2 + 15) & ~15u;
        uint4 *dst = reinterpret_cast<uint4 *>(P.offsets + e0 / 2);
        for (uint32_t i = tid; i < nbytes / 16; i += kRowTile) {
            dst[i] = reinterpret_cast<const uint4 *>(s_planes)[i];
            if (clear) reinterpret_cast<uint4 *>(s_planes)[i] = make_uint4(0, 0, 0, 0);
        }
    } else {
        const uint32_t nbytes = ((nr * C + 7) / 8 + 15) & ~15u;
        const uint32_t pbytes = P.smem_planes / 2;
        uint4 *dso = reinterpret_cast<uint4 *>(P.offsets + e0 / 8);
        uint4 *dse = reinterpret_cast<uint4 *>(P.escapes + e0 / 8);
        for (uint32_t i = tid; i < nbytes / 16; i += kRowTile) {
            dso[i] = reinterpret_cast<const uint4 *>(s_planes)[i];
            dse[i] = reinterpret_cast<const uint4 *>(s_planes + pbytes)[i];
            if (clear) {
                reinterpret_cast<uint4 *>(s_planes)[i] = make_uint4(0, 0, 0, 0);
                reinterpret_cast<uint4 *>(s_planes + pbytes)[i] = make_uint4(0, 0, 0, 0);
            }
        }
    }
}

// Base kernel (two-kernel path): one thread per row.  Each row's base comes
// from row_scan and row_fast_key, or from the exact rule when no bound
// proves it.  Writes base[row], the row's exception count into
// exc_index[row] (until the encode kernel replaces it) and the tile's total
// into the scratch.
template <int KIND, int RD>
__global__ void __launch_bounds__(kRowTile) prepare_base_kernel(const __grid_constant__ PrepParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t s_wsum[2][kRowTile / 32];
    __shared__ __align__(8) uint64_t s_bar[2];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t C = (uint32_t)P.C;
    const uint32_t stride = (uint32_t)P.stride;
    const bool bulk = P.stage != kStagePlain;
    const bool two = bulk && P.nbuf == 2;
    const uint64_t G = gridDim.x;

    uint32_t *s_hist = reinterpret_cast<uint32_t *>(smem);          // bins x kRowTile words (8 x 128 at least)
    uint8_t *s_dense0 = smem + P.smem_hist;                          // nbuf staging buffers

    if (tid == 0 && bulk) {
        mbar_init(&s_bar[0]);
        mbar_init(&s_bar[1]);
    }
    __syncthreads();
    if (bulk && warp == 0 && blockIdx.x < P.num_tiles) stage_issue(P, blockIdx.x, s_dense0, &s_bar[0], lane);

    const uint32_t ntiles = (uint32_t)P.num_tiles;
    for (uint32_t k = 0, tile = blockIdx.x; tile < ntiles; ++k, tile += (uint32_t)G) {
        // buffer and barrier of this tile: with two buffers they alternate;
        // with one, the barrier alternates so that its phases stay in step
        const int buf = two ? (int)(k & 1u) : 0;
        const int bar = (int)(k & 1u);
        uint8_t *s_dense = s_dense0 + (uint32_t)buf * P.smem_dense;
        if (two && warp == 0 && tile + G < ntiles)
            stage_issue(P, tile + G, s_dense0 + (uint32_t)(buf ^ 1) * P.smem_dense, &s_bar[bar ^ 1], lane);
        stage_wait(P, tile, s_dense, &s_bar[bar], (k >> 1) & 1u, tid);

        const uint32_t r0 = tile * (uint32_t)kRowTile;
        const int nr = (int)tile_rows(P, tile);
        const bool mine = tid < nr;
        const uint8_t *rowb = s_dense + (uint32_t)tid * stride;
        uint32_t *hcol = s_hist + tid;
        uint32_t a = 0, n1 = 0, n2 = 0, n3 = 0;
        if (mine) a = row_scan<KIND, RD>(rowb, C, hcol, n1, n2, n3);
        if (!two) {
            // every row is read: with one buffer, refill it now
            __syncthreads();
            if (bulk && warp == 0 && tile + G < ntiles) stage_issue(P, tile + G, s_dense0, &s_bar[bar ^ 1], lane);
        }
        uint32_t key = mine ? row_fast_key<KIND>(hcol, C, a, n1, n2, n3) : 0u;
        key = settle_keys<KIND>(P, key, mine, r0 + 32u * (uint32_t)warp, s_hist, warp, lane);
        const uint32_t count = mine ? C - (key >> 8) : 0u;
        const uint32_t wsum = __reduce_add_sync(kFull, count);
        if (lane == 0) s_wsum[k & 1u][warp] = wsum;
        if (mine) {
            P.base[r0 + tid] = (uint8_t)(255u - (key & 0xFFu));
            P.exc_index[r0 + tid] = count;
        }
        __syncthreads();   // the tile's rows are read: its buffer may be refilled
        if (tid == 0) {
            uint32_t t = 0;
#pragma unroll
            for (int w = 0; w < kRowTile / 32; ++w) t += s_wsum[k & 1u][w];
            P.tile_total[tile] = t;
        }
    }
}

// Encode kernel (two-kernel path): one thread per row.  The tile's offset in
// the exception stream is the sum of the earlier tiles' totals (each block
// keeps a running sum over its tiles); exc_index entries follow from a block
// scan of the counts; each thread encodes its row (encode_row) into the
// tile's planes and writes its exception bytes to their positions in the
// stream, through a shared-memory stage when the tile's exceptions fit it.
template <int KIND, int RD>
__global__ void __launch_bounds__(kRowTile) prepare_encode_kernel(const __grid_constant__ PrepParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t s_wsum[2][kRowTile / 32];
    __shared__ uint32_t s_part[2][kRowTile / 32];
    __shared__ __align__(8) uint64_t s_bar[2];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t C = (uint32_t)P.C;
    const uint32_t stride = (uint32_t)P.stride;
    const bool bulk = P.stage != kStagePlain;
    const bool two = bulk && P.nbuf_enc == 2;
    const uint64_t G = gridDim.x;

    uint8_t *s_dense0 = smem;                                        // nbuf staging buffers
    uint8_t *s_planes = smem + (uint32_t)P.nbuf_enc * P.smem_dense;
    uint8_t *s_exc = s_planes + P.smem_planes;                       // the tile's exception bytes, in order

    if (tid == 0 && bulk) {
        mbar_init(&s_bar[0]);
        mbar_init(&s_bar[1]);
    }
    for (uint32_t i = tid; i < P.smem_planes / 16; i += kRowTile)
        reinterpret_cast<uint4 *>(s_planes)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (bulk && warp == 0 && blockIdx.x < P.num_tiles) stage_issue(P, blockIdx.x, s_dense0, &s_bar[0], lane);

    const uint32_t ntiles = (uint32_t)P.num_tiles;
    unsigned long long off = 0;                      // exceptions of the tiles before this one
    bool bad = false, over = false;
    // The next tile's row counts and bases, and this thread's share of the
    // totals of the tiles between it and the previous one, are loaded one
    // tile ahead (tile totals of one window of G tiles fit 32 bits).
    uint32_t nx_count = 0, nx_base = 0, nx_part = 0;
    auto prefetch = [&](uint32_t t, uint32_t from) {
        nx_count = nx_base = nx_part = 0;
        if (t >= ntiles) return;
        const uint32_t r = t * (uint32_t)kRowTile + tid;
        if (tid < (int)tile_rows(P, t)) {
            nx_count = P.exc_index[r];
            nx_base = P.base[r];
        }
        for (uint32_t j = from + tid; j < t; j += kRowTile) nx_part += P.tile_total[j];
    };
    prefetch(blockIdx.x, 0);
    for (uint32_t k = 0, tile = blockIdx.x; tile < ntiles; ++k, tile += (uint32_t)G) {
        const int buf = two ? (int)(k & 1u) : 0;
        const int bar = (int)(k & 1u);
        uint8_t *s_dense = s_dense0 + (uint32_t)buf * P.smem_dense;
        if (two && warp == 0 && tile + G < ntiles)
            stage_issue(P, tile + G, s_dense0 + (uint32_t)(buf ^ 1) * P.smem_dense, &s_bar[bar ^ 1], lane);

        const uint32_t count = nx_count, base = nx_base;
        const uint32_t part = __reduce_add_sync(kFull, nx_part);
        if (lane == 0) s_part[k & 1u][warp] = part;
        const uint32_t r0 = tile * (uint32_t)kRowTile;
        const int nr = (int)tile_rows(P, tile);
        const bool mine = tid < nr;
        uint32_t wtot;
        const uint32_t wex = warp_excl_scan(count, lane, wtot);
        if (lane == 0) s_wsum[k & 1u][warp] = wtot;
        stage_wait(P, tile, s_dense, &s_bar[bar], (k >> 1) & 1u, tid);
        __syncthreads();
        uint32_t boff = 0, btot = 0;
#pragma unroll
        for (int w = 0; w < kRowTile / 32; ++w) {
            if (w < warp) boff += s_wsum[k & 1u][w];
            btot += s_wsum[k & 1u][w];
            off += s_part[k & 1u][w];
        }
        prefetch(tile + (uint32_t)G, tile);
        const uint32_t pre = boff + wex;
        if (mine) P.exc_index[r0 + tid] = (uint32_t)(off + pre);
        if (tile == ntiles - 1 && tid == 0) {
            const unsigned long long all = off + btot;
            P.exc_index[P.rows] = (uint32_t)all;
            if (all > 0xFFFFFFFFull) flag(P.err, CSF_DEV_ERR_CAPACITY);
        }
        // the tile's exceptions are staged in shared memory unless they
        // overflow the stage; then they go straight to the stream
        const bool staged = btot <= P.exc_stage;
        const bool low = __all_sync(kFull, !mine || base <= low_base<KIND>());
        if (mine) {
            const uint64_t gcap = off < P.exc_capacity ? P.exc_capacity - off : 0;
            const uint8_t *rowb = s_dense + (uint32_t)tid * stride;
            const uint32_t end =
                low ? encode_row<KIND, RD, true>(rowb, C, base, (uint32_t)tid * C, s_planes, P.smem_planes, s_exc,
                                                 staged, P.exc_bytes + off, gcap, pre, over)
                    : encode_row<KIND, RD, false>(rowb, C, base, (uint32_t)tid * C, s_planes, P.smem_planes, s_exc,
                                                  staged, P.exc_bytes + off, gcap, pre, over);
            if (end != pre + count) bad = true;           // the two kernels must agree on the count
        }
        __syncthreads();   // planes and exceptions staged; the tile's rows are read
        if (!two && bulk && warp == 0 && tile + G < ntiles)
            stage_issue(P, tile + G, s_dense0, &s_bar[bar ^ 1], lane);
        // planes of the tile, cleared again for the next one
        write_planes<KIND>(P, s_planes, (uint64_t)r0 * C, (uint32_t)nr, true, tid);
        if (staged) {
            for (uint32_t i = tid; i < btot; i += kRowTile) {
                const unsigned long long g = off + i;
                if (g < P.exc_capacity) P.exc_bytes[g] = s_exc[i];
                else over = true;
            }
        }
    }
    if (__any_sync(kFull, over) && lane == 0) flag(P.err, CSF_DEV_ERR_CAPACITY);
    if (__any_sync(kFull, bad) && lane == 0) flag(P.err, CSF_DEV_ERR_CORRUPT);
}

// Fused kernel (one pass per tile; the scratch holds a slot of 128 * C bytes
// per tile): one thread per row.  Base search as in the base kernel, then a
// block scan of the counts gives each row's exceptions' place inside the
// tile, and each thread encodes its row from the same staged copy: planes to
// the stack, exception bytes to the tile's slot (through a shared-memory
// stage when they fit it), exc_index[row] = the row's place inside the tile,
// the tile's total to the scratch.  The bins, and after them the planes and
// the exception stage, share one region of shared memory.
template <int KIND, int RD>
__global__ void __launch_bounds__(kRowTile, 7) prepare_fused_kernel(const __grid_constant__ PrepParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t s_wsum[kRowTile / 32];
    __shared__ __align__(8) uint64_t s_bar[2];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t C = (uint32_t)P.C;
    const uint32_t stride = (uint32_t)P.stride;
    const bool bulk = P.stage != kStagePlain;
    const bool two = bulk && P.nbuf == 2;
    const uint64_t G = gridDim.x;

    uint32_t *s_hist = reinterpret_cast<uint32_t *>(smem);          // the bins, during the base search
    uint8_t *s_planes = smem;                                        // then the tile's planes
    uint8_t *s_exc = smem + P.smem_planes;                           // and its exception bytes, in order
    uint8_t *s_dense0 = smem + P.smem_hist;                          // nbuf staging buffers

    if (tid == 0 && bulk) {
        mbar_init(&s_bar[0]);
        mbar_init(&s_bar[1]);
    }
    __syncthreads();
    if (bulk && warp == 0 && blockIdx.x < P.num_tiles) stage_issue(P, blockIdx.x, s_dense0, &s_bar[0], lane);
    // The placing kernel may be scheduled now: it waits for this grid to
    // complete before it reads anything (the grid is persistent, so all its
    // blocks are already resident).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const uint32_t ntiles = (uint32_t)P.num_tiles;
    bool bad = false, over = false;
    for (uint32_t k = 0, tile = blockIdx.x; tile < ntiles; ++k, tile += (uint32_t)G) {
        const int buf = two ? (int)(k & 1u) : 0;
        const int bar = (int)(k & 1u);
        uint8_t *s_dense = s_dense0 + (uint32_t)buf * P.smem_dense;
        if (two && warp == 0 && tile + G < ntiles)
            stage_issue(P, tile + G, s_dense0 + (uint32_t)(buf ^ 1) * P.smem_dense, &s_bar[bar ^ 1], lane);
        stage_wait(P, tile, s_dense, &s_bar[bar], (k >> 1) & 1u, tid);

        const uint32_t r0 = tile * (uint32_t)kRowTile;
        const int nr = (int)tile_rows(P, tile);
        const bool mine = tid < nr;
        const uint8_t *rowb = s_dense + (uint32_t)tid * stride;
        uint32_t *hcol = s_hist + tid;
        uint32_t a = 0, n1 = 0, n2 = 0, n3 = 0;
        if (mine) a = row_scan<KIND, RD>(rowb, C, hcol, n1, n2, n3);
        uint32_t key = mine ? row_fast_key<KIND>(hcol, C, a, n1, n2, n3) : 0u;
        key = settle_keys<KIND>(P, key, mine, r0 + 32u * (uint32_t)warp, s_hist, warp, lane);
        const uint32_t count = mine ? C - (key >> 8) : 0u;
        const uint32_t base = 255u - (key & 0xFFu);
        uint32_t wtot;
        const uint32_t wex = warp_excl_scan(count, lane, wtot);
        if (lane == 0) s_wsum[warp] = wtot;
        __syncthreads();   // the bins are read: their space takes the planes
        for (uint32_t i = tid; i < P.smem_planes / 16; i += kRowTile)
            reinterpret_cast<uint4 *>(s_planes)[i] = make_uint4(0, 0, 0, 0);
        uint32_t boff = 0, btot = 0;
#pragma unroll
        for (int w = 0; w < kRowTile / 32; ++w) {
            if (w < warp) boff += s_wsum[w];
            btot += s_wsum[w];
        }
        const uint32_t pre = boff + wex;
        const bool staged = btot <= P.exc_stage;
        uint8_t *slot = P.slot + (uint64_t)tile * P.slot_bytes;
        __syncthreads();   // planes cleared
        const bool low = __all_sync(kFull, !mine || base <= low_base<KIND>());
        if (mine) {
            const uint32_t end =
                low ? encode_row<KIND, RD, true>(rowb, C, base, (uint32_t)tid * C, s_planes, P.smem_planes, s_exc,
                                                 staged, slot, P.slot_bytes, pre, over)
                    : encode_row<KIND, RD, false>(rowb, C, base, (uint32_t)tid * C, s_planes, P.smem_planes, s_exc,
                                                  staged, slot, P.slot_bytes, pre, over);
            if (end != pre + count) bad = true;
            P.base[r0 + tid] = (uint8_t)base;
            P.exc_index[r0 + tid] = pre;
        }
        __syncthreads();   // planes and exceptions staged; the tile's rows are read
        if (!two && bulk && warp == 0 && tile + G < ntiles)
            stage_issue(P, tile + G, s_dense0, &s_bar[bar ^ 1], lane);
        write_planes<KIND>(P, s_planes, (uint64_t)r0 * C, (uint32_t)nr, false, tid);
        if (staged) {
            // whole 16-byte pieces (the slot is 16-byte aligned and private
            // to the tile; bytes past the total are never read)
            for (uint32_t i = tid; i < (btot + 15) / 16; i += kRowTile)
                reinterpret_cast<uint4 *>(slot)[i] = reinterpret_cast<const uint4 *>(s_exc)[i];
        }
        if (tid == 0) P.tile_total[tile] = btot;
        __syncthreads();   // the shared region is read before the next tile's bins
    }
    if (__any_sync(kFull, over) && lane == 0) flag(P.err, CSF_DEV_ERR_CORRUPT);   // a slot holds a whole tile
    if (__any_sync(kFull, bad) && lane == 0) flag(P.err, CSF_DEV_ERR_CORRUPT);
}

// Copies a tile's n exception bytes from its slot (16-byte aligned) to
// stream position o (whole warp).  Whole 4-byte words of the stream take
// one funnel-shifted word store each, the partial words at both ends byte
// stores.  The slot is read 8 words a lane per round, loaded together; the
// slot word before each comes from the next lower lane (lane 0: lane 31 of
// the step before).  `first` holds the first round's words, loaded by the
// caller.
__device__ __forceinline__ void place_words(uint32_t *d32, const uint32_t *__restrict__ s32, uint32_t a,
                                            uint32_t n, const uint32_t (&first)[8], int lane) {
    const uint32_t nwords = (a + n + 3) / 4;   // stream word j holds slot bytes 4j - a .. 4j - a + 3
    uint32_t carry = 0;
    for (uint32_t jb = 0; jb < nwords; jb += 8 * 32) {
        uint32_t hi[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t j = jb + 32u * (uint32_t)k + (uint32_t)lane;
            hi[k] = jb == 0 ? first[k] : (4 * j < n ? __ldg(s32 + j) : 0u);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t j = jb + 32u * (uint32_t)k + (uint32_t)lane;
            uint32_t lo = __shfl_up_sync(kFull, hi[k], 1);
            const uint32_t top = __shfl_sync(kFull, hi[k], 31);
            if (lane == 0) lo = carry;
            carry = top;
            if (j >= nwords) continue;
            const uint32_t v = a == 0 ? hi[k] : __funnelshift_r(lo, hi[k], 8u * (4u - a));
            const uint32_t b0 = 4 * j;                     // stream bytes o - a + b0 .. + 3
            if (b0 >= a && b0 + 4 <= a + n) {
                d32[j] = v;
            } else {
                uint8_t *d8 = reinterpret_cast<uint8_t *>(d32 + j);
#pragma unroll
                for (uint32_t q = 0; q < 4; ++q)
                    if (b0 + q >= a && b0 + q < a + n) d8[q] = (uint8_t)(v >> (8 * q));
            }
        }
    }
}

// Second kernel of the fused path: each warp places one tile, tile
// 4 * block + warp.  Everything that does not depend on the tile's offset
// is loaded first, in one round trip: the tile's total and its rows'
// exc_index entries (each row's place inside the tile), the first 256 words
// of its slot, and the block's share of the totals of all earlier tiles.
// Then the offset (the block's sum plus a scan of its four totals) is added
// to the entries and the slot is copied to its place in the stream.  With
// the stream pointer not 4-byte aligned, or a slot that would pass the
// capacity, the bytes are copied one by one (bytes past the capacity are
// dropped and CSF_DEV_ERR_CAPACITY set).
__global__ void __launch_bounds__(kRowTile) prepare_place_kernel(const __grid_constant__ PrepParams P) {
    __shared__ unsigned long long s_red[kRowTile / 32];
    __shared__ uint32_t s_tot[kRowTile / 32];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint64_t ntiles = P.num_tiles;
    const uint64_t t0 = (uint64_t)blockIdx.x * (kRowTile / 32);
    const uint64_t tile = t0 + (uint64_t)warp;
    const bool have = tile < ntiles;
    // Launched as a programmatic dependent of the fused kernel: wait until
    // that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // loads that need no offset
    const uint32_t n = have ? __ldg(P.tile_total + tile) : 0u;
    const uint64_t r_lo = tile * kRowTile, r_hi = have ? min(r_lo + (uint64_t)kRowTile, P.rows) : r_lo;
    uint32_t e[kRowTile / 32];
#pragma unroll
    for (int i = 0; i < kRowTile / 32; ++i) {
        const uint64_t r = r_lo + (uint64_t)(lane + 32 * i);
        e[i] = r < r_hi ? P.exc_index[r] : 0u;
    }
    const uint8_t *slot = P.slot + tile * (uint64_t)P.slot_bytes;
    const uint32_t *s32 = reinterpret_cast<const uint32_t *>(slot);
    uint32_t first[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t j = 32u * (uint32_t)k + (uint32_t)lane;
        first[k] = have && 4 * j < P.slot_bytes ? __ldg(s32 + j) : 0u;
    }
    // totals of the tiles before the block: eight loads in flight a thread
    unsigned long long run = 0;
    uint64_t j = tid;
    for (; j + 7 * kRowTile < t0; j += 8 * kRowTile) {
        uint32_t v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __ldg(P.tile_total + j + i * kRowTile);
#pragma unroll
        for (int i = 0; i < 8; ++i) run += v[i];
    }
    for (; j < t0; j += kRowTile) run += __ldg(P.tile_total + j);
    run = warp_sum64(run);
    if (lane == 0) {
        s_red[warp] = run;
        s_tot[warp] = n;
    }
    __syncthreads();
    unsigned long long o = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kRowTile / 32; ++w) {
        o += s_red[w];
        all += s_tot[w];
    }
    all += o;
#pragma unroll
    for (int w = 0; w < kRowTile / 32; ++w) o += w < warp ? s_tot[w] : 0u;

    if (have) {
#pragma unroll
        for (int i = 0; i < kRowTile / 32; ++i) {
            const uint64_t r = r_lo + (uint64_t)(lane + 32 * i);
            if (r < r_hi) P.exc_index[r] = (uint32_t)(o + e[i]);
        }
        uint8_t *dst = P.exc_bytes;
        if ((reinterpret_cast<uintptr_t>(dst) & 3u) == 0 && o + n <= P.exc_capacity) {
            place_words(reinterpret_cast<uint32_t *>(dst) + (o >> 2), s32, (uint32_t)(o & 3u), n, first, lane);
        } else {
            bool over = false;
            for (uint32_t i = lane; i < n; i += 32) {
                if (o + i < P.exc_capacity) dst[o + i] = __ldg(slot + i);
                else over = true;
            }
            if (__any_sync(kFull, over) && lane == 0) flag(P.err, CSF_DEV_ERR_CAPACITY);
        }
    }
    if (t0 + kRowTile / 32 >= ntiles && tid == 0) {
        P.exc_index[P.rows] = (uint32_t)all;
        if (all > 0xFFFFFFFFull) flag(P.err, CSF_DEV_ERR_CAPACITY);
    }
}

}  // namespace

static bool rows_path(int32_t C) { return C <= 255; }

static int row_read(int32_t C) {
    if (C % 16 == 0) return kRdVec;
    if (C % 4 == 0) return kRdWord;
    return kRdShift;
}

// Smem row stride of the staged tile: the rows stay packed, as in global
// memory, so that one bulk copy stages a whole tile.  (Padding rows to an
// odd number of 16-byte slots made quarter-warp vector reads conflict-free,
// but a copy per row cost more: MXFP4's 160-byte rows took 128 bulk copies
// per tile.)
static int32_t rows_stride(int32_t C) { return C; }

int32_t prepare_tile_rows(int32_t kind, int32_t C) {
    if (rows_path(C)) return kRowTile;
    const int32_t rbp = unit_rows(C, kind == CSF_NVFP4 ? kChunkNv : kChunkMx);
    const int64_t per = (int64_t)rbp * C;
    int64_t k = 16384 / per;
    if (k < 1) k = 1;
    return (int32_t)(k * rbp);
}

static uint32_t round16(uint64_t v) { return (uint32_t)((v + 15) & ~15ull); }

static uint32_t planes_bytes(int32_t kind, uint64_t te) {
    return kind == CSF_NVFP4 ? round16((te + 1) / 2) : 2 * round16((te + 7) / 8);
}

// Whether the row kernels stage tiles with bulk copies (one per tile): the
// dense pointer must be 16-byte aligned.  Otherwise every thread loads part
// of the tile.
static int rows_stage(int32_t C, const void *dense) {
    (void)C;
    return (reinterpret_cast<uintptr_t>(dense) & 15u) != 0 ? kStagePlain : kStageTile;
}

static uint32_t rows_dense_bytes(int32_t C) { return round16((uint64_t)kRowTile * rows_stride(C) + 16); }
// Bins of the base kernel: 33 words a row for NVFP4; MXFP4 keeps none, but
// every kind needs the 8 x 32 words a warp's exact fallback uses.
static uint32_t rows_hist_bytes(int32_t kind) { return 4u * (kind == CSF_NVFP4 ? 33u : 8u) * kRowTile; }
// Shared-memory stage of the encode kernel's exception bytes: a tile with
// more exceptions writes them straight to the stream instead.
static uint32_t rows_exc_stage(int32_t C) {
    const uint32_t all = round16((uint64_t)kRowTile * C);
    return all < 4096u ? all : 4096u;
}
// Two staging buffers (the next tile loading while one is worked on) only
// while the base kernel keeps 8 blocks per SM (24 KB with the bins); else one
// buffer, refilled as soon as its rows have been read: more resident blocks
// hide the copies better (gate 53.7 -> 52.2 us, MXFP4 122.5 -> 117.7 us).
static int rows_nbuf(int32_t kind, int32_t C, bool bulk) {
    return bulk && rows_hist_bytes(kind) + 2u * rows_dense_bytes(C) <= 24u * 1024u ? 2 : 1;
}
static int rows_nbuf_enc(int32_t kind, int32_t C, bool bulk) {
    const uint32_t rest = planes_bytes(kind, (uint64_t)kRowTile * C) + rows_exc_stage(C);
    return bulk && 2u * rows_dense_bytes(C) + rest <= 40u * 1024u ? 2 : 1;
}
// Fused kernel: one region for the bins and, after them, the planes and the
// exception stage; staging buffers as the base kernel's.
static uint32_t fused_region_bytes(int32_t kind, int32_t C) {
    const uint32_t enc = planes_bytes(kind, (uint64_t)kRowTile * C) + rows_exc_stage(C);
    const uint32_t h = rows_hist_bytes(kind);
    return h > enc ? h : enc;
}
static int fused_nbuf(int32_t kind, int32_t C, bool bulk) {
    return bulk && fused_region_bytes(kind, C) + 2u * rows_dense_bytes(C) <= 24u * 1024u ? 2 : 1;
}
// A tile's exception slot in the scratch: room for every byte of the tile.
static uint32_t slot_bytes(int32_t C) { return round16((uint64_t)kRowTile * C); }
// Fused scratch: 16 bytes, a 4-byte total per tile, then the slots (256-byte
// aligned).
static uint64_t slots_offset(uint64_t tiles) { return (16 + 4 * tiles + 255) & ~255ull; }

// Tiles up to which the fused path runs: each block of its placing kernel
// sums the totals of all tiles before it, which costs tiles^2 / 8 loads in
// all (8.4 M at this limit of 1 M rows); larger stacks take the two-kernel
// path, whose running sums cost a few loads per tile.
constexpr uint64_t kFusedMaxTiles = 8192;

uint64_t prepare_fused_scratch_bytes(int32_t kind, int32_t C, uint64_t rows) {
    (void)kind;
    const uint64_t tiles = (rows + kRowTile - 1) / kRowTile;
    if (!rows_path(C) || tiles > kFusedMaxTiles) return 0;
    return slots_offset(tiles) + tiles * slot_bytes(C);
}

// Dynamic shared memory of a launch.  Row path: the base kernel holds the
// bins and the staging buffers, the encode kernel the buffers, the planes
// and the exception stage; `staged` = bulk staging.  The larger of the two
// is reported.  Wide rows: the single-pass kernel.
size_t prepare_smem_bytes(int32_t kind, int32_t C, int32_t tr, bool staged) {
    const uint64_t te = (uint64_t)tr * C;
    if (rows_path(C)) {
        const size_t base = rows_hist_bytes(kind) + (uint32_t)rows_nbuf(kind, C, staged) * rows_dense_bytes(C);
        const size_t enc = (uint32_t)rows_nbuf_enc(kind, C, staged) * rows_dense_bytes(C) + planes_bytes(kind, te) +
                           rows_exc_stage(C);
        return base > enc ? base : enc;
    }
    return (size_t)round16(te) + planes_bytes(kind, te) + kWarps * 256 * 4 + (size_t)tr * 4 + round16(tr);
}

// true: the row kernels stage tiles with bulk copies.
bool prepare_stages_rows(int32_t kind, int32_t C, const void *dense) {
    (void)kind;
    return rows_path(C) && rows_stage(C, dense) != kStagePlain;
}

// The row path sums tile totals (4 bytes a tile, written before they are
// read); the single-pass wide-row kernel needs its ticket and look-back
// words zeroed.
bool prepare_needs_cleared_scratch(int32_t C) { return !rows_path(C); }

void make_prep_params(PrepParams &p, const uint8_t *dense, const csf_stack &out, uint64_t exc_capacity,
                      void *scratch, uint64_t rows, uint64_t n, bool staged, bool fused) {
    (void)staged;   // implied by the geometry and the dense pointer (prepare_stages_rows)
    const csf_geometry &g = out.g;
    const int32_t tr = prepare_tile_rows(g.kind, g.cols);
    std::memset(&p, 0, sizeof p);
    p.dense = dense;
    p.base = out.base;
    p.offsets = out.offsets;
    p.escapes = out.escapes;
    p.exc_index = out.exc_index;
    p.exc_bytes = out.exc_bytes;
    p.err = out.error_word;
    p.ticket = static_cast<unsigned int *>(scratch);
    p.status = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(scratch) + 16);
    p.tile_total = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) + 16);
    p.exc_capacity = exc_capacity;
    p.rows = rows;
    p.n = n;
    p.num_tiles = (rows + tr - 1) / tr;
    p.magic = ((1ull << 40) + (uint64_t)g.cols - 1) / (uint64_t)g.cols;
    p.C = g.cols;
    p.kind = g.kind;
    p.tr = tr;
    p.dense_aligned = (reinterpret_cast<uintptr_t>(dense) & 15u) == 0 ? 1 : 0;
    const uint64_t te = (uint64_t)tr * g.cols;
    p.spin_limit = kSpinLimit;
    p.smem_planes = planes_bytes(g.kind, te);
    if (rows_path(g.cols)) {
        p.stride = rows_stride(g.cols);
        p.smem_hist = rows_hist_bytes(g.kind);
        p.smem_dense = rows_dense_bytes(g.cols);
        p.stage = rows_stage(g.cols, dense);
        p.nbuf = rows_nbuf(g.kind, g.cols, p.stage != kStagePlain);
        p.nbuf_enc = rows_nbuf_enc(g.kind, g.cols, p.stage != kStagePlain);
        p.exc_stage = rows_exc_stage(g.cols);
        if (fused) {
            p.fused = 1;
            p.smem_hist = fused_region_bytes(g.kind, g.cols);
            p.nbuf = fused_nbuf(g.kind, g.cols, p.stage != kStagePlain);
            p.slot_bytes = slot_bytes(g.cols);
            p.slot = static_cast<uint8_t *>(scratch) + slots_offset(p.num_tiles);
        }
    } else {
        p.stride = g.cols;
        p.smem_dense = round16(te);
        p.stage = kStagePlain;
    }
}

// Persistent grid of one of the row kernels: as many blocks as stay resident.
template <typename K>
static cudaError_t launch_persistent(K kernel, const PrepParams &p, size_t smem, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, occ = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kRowTile, smem)) != cudaSuccess)
        return e;
    uint64_t grid = (uint64_t)sms * (uint64_t)(occ > 0 ? occ : 1);
    if (grid > p.num_tiles) grid = p.num_tiles;
    kernel<<<(unsigned)grid, kRowTile, smem, s>>>(p);
    return cudaGetLastError();
}

template <int KIND, int RD>
static cudaError_t launch_rows_rd(const PrepParams &p, cudaStream_t s) {
    cudaError_t e = launch_persistent(prepare_base_kernel<KIND, RD>, p, p.smem_hist + (uint32_t)p.nbuf * p.smem_dense, s);
    if (e != cudaSuccess) return e;
    return launch_persistent(prepare_encode_kernel<KIND, RD>, p,
                             (uint32_t)p.nbuf_enc * p.smem_dense + p.smem_planes + p.exc_stage, s);
}

// Fused path: the one-pass kernel, then the placing kernel: a block per 4
// tiles (one per warp).
template <int KIND, int RD>
static cudaError_t launch_fused_rd(const PrepParams &p, cudaStream_t s) {
    cudaError_t e = launch_persistent(prepare_fused_kernel<KIND, RD>, p, p.smem_hist + (uint32_t)p.nbuf * p.smem_dense, s);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the placing grid is scheduled while the
    // fused grid runs and starts as soon as it completes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.num_tiles + 3) / 4));
    cfg.blockDim = dim3(kRowTile);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, prepare_place_kernel, p) == cudaSuccess) return cudaSuccess;
    cudaGetLastError();
    prepare_place_kernel<<<cfg.gridDim, kRowTile, 0, s>>>(p);   // without the programmatic edge
    return cudaGetLastError();
}

template <int KIND>
static cudaError_t launch_rows(const PrepParams &p, cudaStream_t s) {
    const int rd = row_read(p.C);
    if (p.fused) {
        if (rd == kRdVec) return launch_fused_rd<KIND, kRdVec>(p, s);
        if (rd == kRdWord) return launch_fused_rd<KIND, kRdWord>(p, s);
        return launch_fused_rd<KIND, kRdShift>(p, s);
    }
    if (rd == kRdVec) return launch_rows_rd<KIND, kRdVec>(p, s);
    if (rd == kRdWord) return launch_rows_rd<KIND, kRdWord>(p, s);
    return launch_rows_rd<KIND, kRdShift>(p, s);
}

cudaError_t launch_prepare(const PrepParams &p, size_t smem, cudaStream_t s) {
    if (rows_path(p.C)) return p.kind == CSF_NVFP4 ? launch_rows<CSF_NVFP4>(p, s) : launch_rows<CSF_MXFP4>(p, s);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    prepare_kernel<<<(unsigned)p.num_tiles, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace csfk
