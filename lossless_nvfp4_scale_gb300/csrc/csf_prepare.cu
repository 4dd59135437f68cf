// CSF prepare kernel for sm_103a: encodes a dense stack (base byte per row,
// offset / escape planes, exception index, exception stream) in one pass over
// the dense bytes.
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
// Per block = one tile of `tr` rows (a whole number of chunk-aligned row
// groups, so output planes start on 16-byte boundaries):
//   1. stage the tile's dense bytes in shared memory (one HBM read);
//   2. one warp per row: 256-bin histogram in shared memory, window counts
//      (prefix sums for NVFP4, neighbour sums for MXFP4), warp max-reduce of
//      (count, -value) picks the base; the row's exception count is C minus
//      the winning window count;
//   3. all threads pack offset nibbles / bit planes from the staged bytes;
//   4. block scan of the per-row counts; the tile total is chained to earlier
//      tiles by a decoupled look-back (Merrill & Garland, "Single-pass
//      Parallel Prefix Scan with Decoupled Look-back", 2016) over per-tile
//      status words in caller scratch; tiles take ids from a ticket counter in
//      start order, so a block only waits on blocks already running; every
//      wait is bounded and reports CSF_DEV_ERR_TIMEOUT instead of hanging;
//   5. write base bytes, planes, exc_index and the exception bytes at their
//      global positions.
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

// Rows (and threads) per block in the row-wise kernel; a multiple of every
// chunk-alignment row count (it divides into 32 and 128-element pieces).
constexpr int kRowTile = 128;

// Row-wise prepare for C <= 255 (byte counters cannot overflow).  One thread
// per row: a thread-private 256-bin histogram of byte counters (word k of
// thread t at hist[k * kRowTile + t], so a warp's accesses hit 32 banks), an
// occupancy mask of 8-bin groups, window counts for the occupied words only
// (byte prefix sums for NVFP4, neighbour sums for MXFP4), and the packed
// 16-bit key (count << 8 | 255 - value) whose maximum is the most bytes with
// the smallest value.  The histogram area is reused to stage the tile's
// exception bytes in row-major order for one coalesced copy-out.  The tile's
// dense rows are staged in shared memory with one coalesced read, unless that
// would leave fewer than 4 blocks per SM (prepare_stages_rows): then each
// thread reads its row in place, as 4-byte words through L1.
template <bool STAGE>
__global__ void __launch_bounds__(kRowTile) prepare_rows_kernel(const __grid_constant__ PrepParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ unsigned int s_tile;
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_wsum[kRowTile / 32];
    __shared__ uint32_t s_total;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t C = (uint32_t)P.C;
    const bool nv = P.kind == CSF_NVFP4;
    const uint32_t stride = (uint32_t)P.stride;

    uint32_t *s_hist = reinterpret_cast<uint32_t *>(smem);            // 64 x kRowTile words
    uint8_t *s_exc = smem;                                             // after the base pass
    uint8_t *s_dense = smem + 256 * kRowTile;
    uint8_t *s_planes = s_dense + P.smem_dense;
    uint8_t *s_base = s_planes + P.smem_planes;
    uint32_t *s_pre = reinterpret_cast<uint32_t *>(s_base + kRowTile);

    if (tid == 0) s_tile = atomicAdd(P.ticket, 1u);
    __syncthreads();
    const uint64_t tile = s_tile;
    if (tile >= P.num_tiles) return;
    const uint64_t r0 = tile * (uint64_t)kRowTile;
    const uint64_t r1 = min(r0 + (uint64_t)kRowTile, P.rows);
    const int nr = (int)(r1 - r0);
    const uint64_t e0 = r0 * C;
    const uint32_t ne = (uint32_t)nr * C;

    // 1. Zero the histograms and planes; stage the rows at `stride` (unless
    //    the rows are read in place: C % 4 == 0, 4-byte aligned dense).
    for (int i = tid; i < 64 * kRowTile / 4; i += kRowTile)
        reinterpret_cast<uint4 *>(s_hist)[i] = make_uint4(0, 0, 0, 0);
    for (uint32_t i = tid; i < P.smem_planes / 16; i += kRowTile)
        reinterpret_cast<uint4 *>(s_planes)[i] = make_uint4(0, 0, 0, 0);
    if (STAGE) {
        const uint8_t *src = P.dense + e0;
        if (stride == C) {
            uint32_t done = 0;
            if (P.dense_aligned) {
                const uint32_t n16 = ne / 16;
                for (uint32_t i = tid; i < n16; i += kRowTile)
                    reinterpret_cast<uint4 *>(s_dense)[i] = __ldg(reinterpret_cast<const uint4 *>(src) + i);
                done = n16 * 16;
            }
            for (uint32_t i = done + tid; i < ne; i += kRowTile) s_dense[i] = __ldg(src + i);
        } else {
            // C % 4 == 0 here: 4-byte words never straddle rows.
            auto put = [&](uint32_t e, uint32_t w) {
                const uint32_t row = (uint32_t)(((uint64_t)e * P.magic) >> 40);
                *reinterpret_cast<uint32_t *>(s_dense + row * stride + (e - row * C)) = w;
            };
            uint32_t done = 0;
            if (P.dense_aligned) {
                const uint32_t n16 = ne / 16;
                for (uint32_t i = tid; i < n16; i += kRowTile) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + i);
                    put(16 * i, v.x); put(16 * i + 4, v.y); put(16 * i + 8, v.z); put(16 * i + 12, v.w);
                }
                done = n16 * 16;
            }
            for (uint32_t e = done + 4 * tid; e < ne; e += 4 * kRowTile) {
                const uint32_t w = (uint32_t)__ldg(src + e) | ((uint32_t)__ldg(src + e + 1) << 8) |
                                   ((uint32_t)__ldg(src + e + 2) << 16) | ((uint32_t)__ldg(src + e + 3) << 24);
                put(e, w);
            }
        }
    }
    __syncthreads();

    // 2. Base byte and exception count of this thread's row.
    uint32_t base = 0, count = 0;
    if (tid < nr) {
        const uint8_t *row = STAGE ? s_dense + tid * stride : P.dense + (r0 + (uint64_t)tid) * C;
        uint32_t *h = s_hist + tid;
        uint32_t occ = 0;
        // Shared-memory reductions (no returned value): increments of the same
        // word need no read-after-write chain through this thread.
        auto add = [&](uint32_t v) {
            atomicAdd(h + (v >> 2) * kRowTile, 1u << ((v & 3u) << 3));
            occ |= 1u << (v >> 3);
        };
        if (!STAGE || (stride & 3u) == 0) {
            const uint32_t *rw = reinterpret_cast<const uint32_t *>(row);
            for (uint32_t k = 0; k < C / 4; ++k) {
                const uint32_t x = rw[k];
                add(x & 0xFFu); add((x >> 8) & 0xFFu); add((x >> 16) & 0xFFu); add(x >> 24);
            }
            for (uint32_t c = C & ~3u; c < C; ++c) add(row[c]);
        } else {
            for (uint32_t c = 0; c < C; ++c) add(row[c]);
        }
        uint32_t best = 0;
        while (occ) {
            const uint32_t g = (uint32_t)(__ffs(occ) - 1);
            occ &= occ - 1;
#pragma unroll
            for (uint32_t m = 2 * g; m < 2 * g + 2; ++m) {
                const uint32_t hm = h[m * kRowTile];
                if (hm == 0) continue;
                uint32_t W;
                if (nv) {
                    // window [v, v+14]: byte prefix sums over words m..m+4
                    const uint32_t q0 = hm * 0x01010101u;
                    uint32_t c = q0 >> 24;
                    uint32_t q[4];
#pragma unroll
                    for (int i = 1; i <= 4; ++i) {
                        const uint32_t hw = (m + i < 64) ? h[(m + i) * kRowTile] : 0u;
                        q[i - 1] = hw * 0x01010101u + c * 0x01010101u;
                        c = q[i - 1] >> 24;
                    }
                    W = __byte_perm(q[2], q[3], 0x5432) - (q0 << 8);
                } else {
                    // window [v, v+1]
                    const uint32_t hn = (m + 1 < 64) ? h[(m + 1) * kRowTile] : 0u;
                    W = hm + __byte_perm(hm, hn, 0x4321);
                }
                const uint32_t f = (((hm & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | hm) & 0x80808080u;
                const uint32_t Wm = W & (f | (f - (f >> 7)));               // present values only
                const uint32_t cm = 4u * m;
                const uint32_t kE = (Wm & 0x00FF00FFu) * 256u + (0x00FD00FFu - cm * 0x00010001u);
                const uint32_t kO = ((Wm >> 8) & 0x00FF00FFu) * 256u + (0x00FC00FEu - cm * 0x00010001u);
                best = __vmaxu2(best, __vmaxu2(kE, kO));
            }
        }
        const uint32_t key = max(best & 0xFFFFu, best >> 16);
        base = 255u - (key & 0xFFu);
        count = C - (key >> 8);
        s_base[tid] = (uint8_t)base;
    }

    // 3. Block scan of the per-row counts.
    uint32_t wtot;
    const uint32_t wex = warp_excl_scan(count, lane, wtot);
    if (lane == 0) s_wsum[warp] = wtot;
    __syncthreads();   // also ends every histogram read: s_exc may overwrite it
    uint32_t boff = 0, btot = 0;
#pragma unroll
    for (int w = 0; w < kRowTile / 32; ++w) {
        if (w < warp) boff += s_wsum[w];
        btot += s_wsum[w];
    }
    const uint32_t pre = boff + wex;
    if (tid < nr) s_pre[tid] = pre;
    if (tid == 0) s_total = btot;

    // 4. Look-back across tiles (warp 0), overlapping the packing below.
    if (warp == 0) {
        const unsigned long long excl = lookback_exclusive(P, tile, btot, lane);
        if (lane == 0) s_excl = excl;
    }

    // 5. Pack this row's planes; stage its exceptions at their tile position.
    if (tid < nr) {
        const uint8_t *row = STAGE ? s_dense + tid * stride : P.dense + (r0 + (uint64_t)tid) * C;
        uint32_t pos = pre;
        uint32_t el = (uint32_t)tid * C;   // tile-local element index
        const uint32_t w = nv ? 14u : 1u;
        uint32_t *po = reinterpret_cast<uint32_t *>(s_planes);
        uint32_t *px = reinterpret_cast<uint32_t *>(s_planes + P.smem_planes / 2);
        // Codes of 4 elements: NVFP4 nibbles in bits 0..15, MXFP4 offset bits in
        // bits 0..3 and escape bits in 4..7.
        auto code4 = [&](uint32_t x, uint32_t nb) {
            uint32_t cd = 0;
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j) {
                if (j < nb) {
                    const uint32_t v = (x >> (8 * j)) & 0xFFu;
                    const uint32_t d = v - base;
                    const bool inside = v >= base && d <= w;
                    if (!inside) s_exc[pos++] = (uint8_t)v;
                    if (nv) cd |= (inside ? d : 15u) << (4 * j);
                    else cd |= (inside ? (d << j) : (0x10u << j));
                }
            }
            return cd;
        };
        // The same codes for a whole word at once (SWAR): per byte d = x - base
        // without borrows between bytes, and bit 7 of `o` set for the bytes
        // outside [base, base + w] (d > w, or x below base: the byte's borrow).
        const uint32_t B4 = base * 0x01010101u, W1 = (w + 1) * 0x01010101u;
        auto code4w = [&](uint32_t x) {
            const uint32_t H = 0x80808080u;
            const uint32_t d = ((x | H) - (B4 & ~H)) ^ ((x ^ ~B4) & H);
            const uint32_t bo = ((~x & B4) | (~(x ^ B4) & d)) & H;
            const uint32_t o = ((((d | H) - W1) | d) | bo) & H;
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j)               // exceptions, in element order
                if (o & (0x80u << (8 * j))) s_exc[pos++] = (uint8_t)(x >> (8 * j));
            const uint32_t ob = o >> 7;                    // 1 in each outside byte
            if (nv) {
                const uint32_t c = (d & ~(ob * 0xFFu)) | (ob * 0x0Fu);    // outside -> escape code 15
                const uint32_t t = c | (c >> 4);
                return __byte_perm(t, 0u, 0x4420);         // nibble j = element j
            }
            // bit 0 of each byte -> bits 0..3 (offset bits, 0 for exceptions), escape bits -> 4..7
            const uint32_t ofb = (((d & ~ob) & 0x01010101u) * 0x01020408u) >> 24;
            const uint32_t esb = (ob * 0x01020408u) >> 24;
            return ofb | (esb << 4);
        };
        uint32_t acc = 0, ax = 0;
        auto flush = [&](bool force) {
            if (nv) {
                if ((el & 7u) == 0 || force) {
                    if (acc) atomicOr(po + ((el - 1) >> 3), acc);
                    acc = 0;
                }
            } else if ((el & 31u) == 0 || force) {
                if (acc) atomicOr(po + ((el - 1) >> 5), acc);
                if (ax) atomicOr(px + ((el - 1) >> 5), ax);
                acc = ax = 0;
            }
        };
        if ((!STAGE || (stride & 3u) == 0) && (el & 3u) == 0) {
            // Whole words; groups of 4 never straddle an output word.
            const uint32_t *rw = reinterpret_cast<const uint32_t *>(row);
            for (uint32_t k = 0; k < C / 4; ++k) {
                const uint32_t cd = code4w(rw[k]);
                if (nv) acc |= cd << (4 * (el & 7u));
                else { acc |= (cd & 0xFu) << (el & 31u); ax |= (cd >> 4) << (el & 31u); }
                el += 4;
                flush(k == C / 4 - 1 && (C & 3u) == 0);
            }
            for (uint32_t c = C & ~3u; c < C; ++c) {
                const uint32_t cd = code4(row[c], 1);
                if (nv) acc |= cd << (4 * (el & 7u));
                else { acc |= (cd & 1u) << (el & 31u); ax |= ((cd >> 4) & 1u) << (el & 31u); }
                ++el;
                flush(c == C - 1);
            }
        } else {
            for (uint32_t c = 0; c < C; ++c) {
                const uint32_t cd = code4(row[c], 1);
                if (nv) acc |= cd << (4 * (el & 7u));
                else { acc |= (cd & 1u) << (el & 31u); ax |= ((cd >> 4) & 1u) << (el & 31u); }
                ++el;
                flush(c == C - 1);
            }
        }
    }
    __syncthreads();
    const unsigned long long excl = s_excl;
    const uint32_t total = s_total;

    // 6. Outputs.
    for (int k = tid; k < nr; k += kRowTile) {
        P.exc_index[r0 + k] = (uint32_t)(excl + s_pre[k]);
        P.base[r0 + k] = s_base[k];
    }
    if (tile == P.num_tiles - 1 && tid == 0) {
        const unsigned long long all = excl + total;
        P.exc_index[P.rows] = (uint32_t)all;
        if (all > 0xFFFFFFFFull) flag(P.err, CSF_DEV_ERR_CAPACITY);
    }
    if (nv) {
        const uint32_t nbytes = ((ne + 1) / 2 + 15) & ~15u;
        uint4 *dst = reinterpret_cast<uint4 *>(P.offsets + e0 / 2);
        for (uint32_t i = tid; i < nbytes / 16; i += kRowTile) dst[i] = reinterpret_cast<const uint4 *>(s_planes)[i];
    } else {
        const uint32_t nbytes = ((ne + 7) / 8 + 15) & ~15u;
        const uint32_t pbytes = P.smem_planes / 2;
        uint4 *dso = reinterpret_cast<uint4 *>(P.offsets + e0 / 8);
        uint4 *dse = reinterpret_cast<uint4 *>(P.escapes + e0 / 8);
        for (uint32_t i = tid; i < nbytes / 16; i += kRowTile) {
            dso[i] = reinterpret_cast<const uint4 *>(s_planes)[i];
            dse[i] = reinterpret_cast<const uint4 *>(s_planes + pbytes)[i];
        }
    }
    bool over = false;
    for (uint32_t i = tid; i < total; i += kRowTile) {
        const unsigned long long pos = excl + i;
        if (pos < P.exc_capacity) P.exc_bytes[pos] = s_exc[i];
        else over = true;
    }
    if (over) flag(P.err, CSF_DEV_ERR_CAPACITY);
}

}  // namespace

static bool rows_path(int32_t C) { return C <= 255; }

// Smem row stride of the staged tile in the row-wise kernel: rows of C % 4 == 0
// bytes are read as words, so their word stride is made odd (conflict-free).
static int32_t rows_stride(int32_t C) {
    if (C % 4 != 0) return C;
    return ((C / 4) % 2 == 1) ? C : C + 4;
}

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

size_t prepare_smem_bytes(int32_t kind, int32_t C, int32_t tr, bool staged) {
    const uint64_t te = (uint64_t)tr * C;
    if (rows_path(C))
        return 256u * kRowTile + (staged ? round16((uint64_t)kRowTile * rows_stride(C)) : 0u) +
               planes_bytes(kind, te) + kRowTile + 4u * kRowTile;
    return (size_t)round16(te) + planes_bytes(kind, te) + kWarps * 256 * 4 + (size_t)tr * 4 + round16(tr);
}

// The row-wise kernel stages its tile in shared memory (one coalesced read of
// the dense rows) when 4 or more blocks per SM still fit; otherwise, and only
// for rows it can read as aligned 4-byte words, each thread reads its row in
// place.  Measured on the gate (C = 100: 4 blocks staged) staging is faster
// (121 against 139 us); on MXFP4 384 x 2048 x 160 (3 blocks staged, 5 not)
// reading in place is (272 against 343 us).
bool prepare_stages_rows(int32_t kind, int32_t C, const void *dense) {
    if (!rows_path(C)) return true;
    if (C % 4 != 0 || (reinterpret_cast<uintptr_t>(dense) & 3u) != 0) return true;
    const size_t smem = prepare_smem_bytes(kind, C, kRowTile, true);
    int occ = 0;
    if (cudaFuncSetAttribute(prepare_rows_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, prepare_rows_kernel<true>, kRowTile, smem) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return occ >= 4;
}

void make_prep_params(PrepParams &p, const uint8_t *dense, const csf_stack &out, uint64_t exc_capacity,
                      void *scratch, uint64_t rows, uint64_t n, bool staged) {
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
    p.stride = rows_path(g.cols) ? rows_stride(g.cols) : g.cols;
    p.stage = staged ? 1 : 0;
    p.spin_limit = kSpinLimit;
    p.smem_dense = rows_path(g.cols) ? (staged ? round16((uint64_t)kRowTile * p.stride) : 0u) : round16(te);
    p.smem_planes = planes_bytes(g.kind, te);
}

cudaError_t launch_prepare(const PrepParams &p, size_t smem, cudaStream_t s) {
    if (rows_path(p.C)) {
        const auto kernel = p.stage ? prepare_rows_kernel<true> : prepare_rows_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kernel<<<(unsigned)p.num_tiles, kRowTile, smem, s>>>(p);
        return cudaGetLastError();
    }
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    prepare_kernel<<<(unsigned)p.num_tiles, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace csfk
