// common.cuh -- small device/host helpers shared by the libacache kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "acache.h"

#define ACACHE_DEVFN __device__ __forceinline__

namespace acache {

// OR a flag into the caller's status word (nullable).
ACACHE_DEVFN void flag(int32_t* dev_status, int32_t bit) {
    if (dev_status) atomicOr(dev_status, bit);
}

template <typename T> ACACHE_DEVFN float to_f32(T x);
template <> ACACHE_DEVFN float to_f32<float>(float x) { return x; }
template <> ACACHE_DEVFN float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> ACACHE_DEVFN T from_f32(float x);
template <> ACACHE_DEVFN float from_f32<float>(float x) { return x; }
template <> ACACHE_DEVFN __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// 2^x on the MUFU unit (hardware ex2, ~2 ulp; -inf -> 0).
ACACHE_DEVFN float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input form of max.f32 on sm_100 and later)
ACACHE_DEVFN float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic: two FMAs / adds per instruction slot).
ACACHE_DEVFN uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
ACACHE_DEVFN void f2unpack(uint64_t v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
ACACHE_DEVFN uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
ACACHE_DEVFN uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

ACACHE_DEVFN float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

ACACHE_DEVFN float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// log2(e): softmax logits are carried in the base-2 domain, exp(x) = 2^(x*log2 e).
constexpr float kLog2e = 1.4426950408889634f;

}  // namespace acache

// ---- host side ------------------------------------------------------------------
namespace acache {
int sm_count();                   // SMs of the current device (cached per device)
int launch_status();              // ACACHE_OK or ACACHE_ERR_CUDA after a launch
long long wait_budget();          // cycles a kernel's pipeline wait may take (acache_wait_budget)
}  // namespace acache
