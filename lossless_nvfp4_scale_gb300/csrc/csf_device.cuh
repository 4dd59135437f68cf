// Small device helpers shared by the decode kernels (csf_decode.cu,
// csf_tiles.cu).  Internal to the library.
#pragma once

#include <cstdint>

namespace csfk {
namespace dev {

constexpr uint32_t kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// base + offset, byte-wise mod 256, for offsets below 0x80 (the low 7 bits
// are added, bit 7 is folded back with XOR, so no carry crosses a byte).
__device__ __forceinline__ uint32_t add_base(uint32_t bw, uint32_t off) {
    return ((bw & 0x7F7F7F7Fu) + off) ^ (bw & 0x80808080u);
}

__device__ __forceinline__ void flag(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

}  // namespace dev
}  // namespace csfk
