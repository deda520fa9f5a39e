// Shared device helpers of the paged KV-cache library (sm_103a).
#pragma once

#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

#define PK_DEV __device__ __forceinline__

namespace pk {

// ---------------------------------------------------------------------------
// bf16 <-> fp32.  A bf16 word is the top half of a binary32 word, so widening
// is a shift; narrowing rounds to nearest-even with cvt.rn.bf16x2.f32.
// ---------------------------------------------------------------------------
PK_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
PK_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

PK_DEV void unpack8(const uint4 &u, float f[8]) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
    f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

// Pack two fp32 into a bf16x2 word (lo in the low half), round-to-nearest-even.
PK_DEV uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^x with the SFU instruction (ex2.approx.ftz.f32: relative error ~2^-22,
// 2^-inf = 0).
PK_DEV float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Rescale factor 2^(m_old - m_new) that also handles the empty state
// (m_old = -inf gives 0 even when m_new is -inf too).
PK_DEV float rescale(float m_old, float m_new) {
    return m_old == -INFINITY ? 0.f : fast_exp2(m_old - m_new);
}

// Read-only 16-byte global load that does not allocate in L1.
PK_DEV uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

PK_DEV void set_error(unsigned int *err, unsigned int bit) {
    if (err) atomicOr(err, bit);
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace pk

// Host-side helpers shared by the translation units (defined in errors.cu).
namespace pk {
// Device address of the current device's error word (nullptr on failure).
unsigned int *error_word_ptr();
// Multiprocessor count of the current device (0 on failure).
int sm_count();
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Raise the dynamic shared memory limit of `func` to `bytes` on the current
// device.  The attribute is per device, so it is set once for every (device,
// kernel) pair; thread-safe.
cudaError_t set_max_dynamic_smem(const void *func, int bytes);
}  // namespace pk
