// common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a only).
//
// Format (NVFP4 as used by the pages; block size, scale type and grid are the
// NVFP4 definition, which the pages leave unstated): 16-element blocks along a
// row, one E4M3 scale byte per block, one FP32 tensor scale, E2M1 codes on
// {0,.5,1,1.5,2,3,4,6} with the sign in bit 3, two codes per byte with the
// even element in the low nibble ("Scale-QLoRA", rit.work, format paragraph:
// each weight is an E2M1 code plus a shared block scale).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// ---------------------------------------------------------------- workspace
// The first 256 bytes of every workspace are a control block of u32 words.
enum CtlWord : int {
    CTL_STATUS = 0,       // first device-side error code (0 = none)
    CTL_AMAX = 1,         // running max of |w| bf16 magnitude bits
    CTL_AMAX_COUNT = 2,   // blocks of the amax kernel that have finished
    CTL_BAR_COUNT = 3,    // grid barrier: arrivals
    CTL_BAR_GEN = 4,      // grid barrier: generation
    CTL_DIRTY = 5,        // kTilesDirty: a wait gave up while tile counters were in use
    CTL_WORDS_USED = 6,
};
constexpr size_t kCtlBytes = 256;
constexpr uint32_t kTilesDirty = 0x7D17u;
// After the control block: arrival counters at a fixed place, so that calls
// of any shape find them at zero (every kernel that counts resets its
// counters before it returns).  Per-call scratch starts after them.
// The words count arrivals per output tile (decode GEMMs: the last block to
// arrive at a tile adds up the shares of the others).
constexpr int kTileCounters = 8192;
constexpr size_t kWsHeaderBytes = kCtlBytes + 4 * (size_t)kTileCounters;

// Spin limit of every device-side wait: about a second of polling, after
// which the kernel records NVFP4_ERR_TIMEOUT and gives up instead of hanging.
constexpr uint32_t kSpinLimit = 1u << 24;

__device__ __forceinline__ void record_status(uint32_t *ctl, nvfp4_status s)
{
    atomicCAS(&ctl[CTL_STATUS], 0u, (uint32_t)s);
}

// A bounded wait gave up in a kernel that counts arrivals per output tile:
// the counters may be left non-zero, so besides the status the workspace is
// marked, and nvfp4_get_device_status clears them when it reports the timeout.
__device__ __forceinline__ void record_timeout_tiles(uint32_t *ctl)
{
    record_status(ctl, NVFP4_ERR_TIMEOUT);
    atomicExch(&ctl[CTL_DIRTY], kTilesDirty);
}

// ---------------------------------------------------------------- scalars
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// E4M3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte)
{
    uint32_t h2;
    uint16_t pair = (uint16_t)(byte & 0xFF);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

// E4M3 byte -> f16x2 holding the value twice (exact).
__device__ __forceinline__ uint32_t e4m3_to_h2_dup(uint32_t byte)
{
    uint32_t h2;
    uint16_t pair = (uint16_t)((byte & 0xFF) | ((byte & 0xFF) << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    return h2;
}

// Non-negative float -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_encode_nonneg(float x)
{
    uint16_t r;
    x = fminf(x, 448.0f);  // +inf and huge values saturate
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
    return r & 0xFF;
}


// Byte with two E2M1 codes -> f16x2 (low nibble -> low half), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte_in_low8)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h2) : "r"(byte_in_low8));
    return h2;
}

// All four bytes of a word -> four f16x2 (byte i -> out[i]).
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t out[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3]) : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 2^e as a float for e in [-149, 127] (exact, subnormal below -126).
__device__ __forceinline__ float exp2i(int e)
{
    if (e >= -126)
        return __uint_as_float((uint32_t)(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}

// x * 2^e exactly for x with |x * 2^e| in the normal range; e in [-254, 254].
__device__ __forceinline__ float scale_pow2(float x, int e)
{
    if (e > 127) {
        x = __fmul_rn(x, exp2i(127));
        e -= 127;
    } else if (e < -126) {
        x = __fmul_rn(x, exp2i(-126));
        e += 126;
    }
    return __fmul_rn(x, exp2i(e));
}

// ---------------------------------------------------------------- memory
// L2 eviction-priority hints for loads (per instruction; no device setting).
__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ld_hint_u4(const void *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// 16-byte global -> shared copy that bypasses registers (cp.async); src_bytes
// 0 writes zeros and reads nothing.  Completion: cp_async_commit groups the
// copies issued so far, cp_async_wait<n> waits until at most n groups are
// still in flight.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *src, uint32_t src_bytes, uint64_t pol)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(d), "l"(src),
                 "r"(src_bytes), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue / wait until every prerequisite grid has finished and its memory
// is visible.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream_u2(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- tensor core
// D = A * B + C, m16n8k16, f16 inputs, f32 accumulate (legacy warp-level MMA;
// the A operand is produced in registers by the dequantiser).
__device__ __forceinline__ void mma_f16_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with C = 0 (the first product of an accumulator chain).
__device__ __forceinline__ void mma_f16_16816_z(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    const float z = 0.0f;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

__device__ __forceinline__ void mma_bf16_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- grid barrier
// Barrier across all blocks of a cooperative launch.  Waits are bounded:
// after kSpinLimit polls the block records NVFP4_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool grid_barrier(uint32_t *ctl, uint32_t nblocks)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        volatile uint32_t *gen = &ctl[CTL_BAR_GEN];
        uint32_t my_gen = *gen;
        __threadfence();
        uint32_t arrived = atomicAdd(&ctl[CTL_BAR_COUNT], 1u);
        if (arrived == nblocks - 1) {
            ctl[CTL_BAR_COUNT] = 0;
            __threadfence();
            atomicAdd(&ctl[CTL_BAR_GEN], 1u);
        } else {
            uint32_t it = 0;
            while (*gen == my_gen) {
                if (++it > kSpinLimit) {
                    record_status(ctl, NVFP4_ERR_TIMEOUT);
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

}  // namespace nvfp4
