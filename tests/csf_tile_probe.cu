/*
 * A consumer kernel of the public device decoder include/csf_tile.cuh, built
 * by tests/test_gpu_tile_device.py: each warp rebuilds tiles of a tile-packed
 * stack in a shared-memory buffer of its own with csf_tile_decode_warp -- the
 * way a GEMM pipeline stage would -- and then copies the 512 bytes out, only
 * so that the test can compare them with the oracle.  Tiles of experts that
 * the grouped-routing prefix leaves inactive are skipped.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "csf_tile.cuh"

template <int KIND>
__global__ void __launch_bounds__(128) probe_kernel(csf_tile_src s, uint32_t E, const void *expert_start, int es64,
                                                    uint8_t *out, uint32_t *bad) {
    __shared__ __align__(16) uint8_t stage[4][512];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t nrb = csf_tile_row_blocks(s), ncb = csf_tile_col_blocks(s), T = nrb * ncb;
    const uint64_t total = (uint64_t)E * T;
    for (uint64_t i = (uint64_t)blockIdx.x * 4 + warp; i < total; i += (uint64_t)gridDim.x * 4) {
        const uint32_t e = (uint32_t)(i / T), t = (uint32_t)(i % T);
        if (expert_start) {
            const bool active = es64 ? static_cast<const long long *>(expert_start)[e + 1] >
                                           static_cast<const long long *>(expert_start)[e]
                                     : static_cast<const int *>(expert_start)[e + 1] >
                                           static_cast<const int *>(expert_start)[e];
            if (!active) continue;   // warp-uniform
        }
        if (csf_tile_decode_warp<KIND>(s, e, t / ncb, t % ncb, stage[warp]) && lane == 0) atomicOr(bad, 1u);
        reinterpret_cast<uint4 *>(out + i * 512)[lane] = reinterpret_cast<const uint4 *>(stage[warp])[lane];
        __syncwarp();
    }
}

extern "C" int csf_tile_probe(const uint8_t *codes, const uint8_t *bases, const uint32_t *tile_index,
                              const uint8_t *exc_bytes, uint32_t num_exc, int kind, int E, int R, int C,
                              const void *expert_start, int es64, uint8_t *out, uint32_t *bad) {
    csf_tile_src s;
    s.codes = codes;
    s.bases = bases;
    s.tile_index = tile_index;
    s.exc_bytes = exc_bytes;
    s.num_exc = num_exc;
    s.kind = kind;
    s.R = R;
    s.C = C;
    if (kind == CSF_NVFP4)
        probe_kernel<CSF_NVFP4><<<120, 128>>>(s, (uint32_t)E, expert_start, es64, out, bad);
    else
        probe_kernel<CSF_MXFP4><<<120, 128>>>(s, (uint32_t)E, expert_start, es64, out, bad);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return (int)e;
}
