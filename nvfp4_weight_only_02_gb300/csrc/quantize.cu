// quantize.cu -- NVFP4 quantiser, dequantiser and scale-only update (sm_103a).
//
// Quantisation is weight-only ("RL with NVFP4 + LoRA" post, section "Метод");
// the tensor scale is either recomputed from the current tensor (dynamic,
// "max" calibration) or kept frozen (Nemotron NVFP4/QAD page, section 03
// "Dynamic vs Frozen").  The scale-only update follows the Scale-QLoRA page
// (codes frozen; trained block scales rounded onto the E4M3 grid; merge writes
// only scale bytes).
//
// Layout: W bf16 N x K row-major; codes N x K/2 bytes (even element in the low
// nibble); scales N x K/16 bytes.  Because K % 16 == 0, the flattened tensor
// is a sequence of 16-element blocks, each 32 bytes of bf16, 8 bytes of codes
// and 1 scale byte, so the kernels index blocks linearly and never need the
// row/column split.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

// ------------------------------------------------------------------ amax
__device__ __forceinline__ uint32_t absmax8(uint4 a, uint4 b)
{
    // per-halfword max of the bf16 magnitude bits of 16 elements
    const uint32_t m = 0x7FFF7FFFu;
    uint32_t x = __vimax3_u16x2(a.x & m, a.y & m, a.z & m);
    uint32_t y = __vimax3_u16x2(a.w & m, b.x & m, b.y & m);
    uint32_t z = __vimax3_u16x2(b.z & m, b.w & m, x);
    return __vmaxu2(y, z);
}

// Pass 1 of the dynamic mode: a = max |w| over the tensor, exact (integer max
// of bf16 magnitude bits; NaN/inf patterns sort above every finite value and
// are reported).  The last block to finish turns a into s_t = a / 2688 and
// writes it to *tensor_scale, then leaves the control words at zero.
__global__ void __launch_bounds__(256) amax_kernel(const uint4 *__restrict__ w, int64_t nvec,
                                                   float *__restrict__ tensor_scale,
                                                   uint32_t *__restrict__ ctl)
{
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < nvec; i += 4 * stride) {  // four 16-byte loads in flight
        uint4 a = ld_stream_u4(w + i);
        uint4 b = ld_stream_u4(w + i + stride);
        uint4 c = ld_stream_u4(w + i + 2 * stride);
        uint4 d = ld_stream_u4(w + i + 3 * stride);
        m = __vmaxu2(m, __vmaxu2(absmax8(a, b), absmax8(c, d)));
    }
    for (; i < nvec; i += stride) {
        uint4 a = ld_stream_u4(w + i);
        m = __vmaxu2(m, absmax8(a, make_uint4(0, 0, 0, 0)));
    }
    m = max(m & 0xFFFFu, m >> 16);
    m = __reduce_max_sync(0xffffffffu, m);
    __shared__ uint32_t s_m[8];
    __shared__ bool s_last;
    if ((threadIdx.x & 31) == 0)
        s_m[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int k = 0; k < (int)(blockDim.x >> 5); k++)
            b = max(b, s_m[k]);
        atomicMax(&ctl[CTL_AMAX], b);
        __threadfence();
        s_last = atomicAdd(&ctl[CTL_AMAX_COUNT], 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last && threadIdx.x == 0) {
        __threadfence();
        uint32_t a_bits = atomicExch(&ctl[CTL_AMAX], 0u);
        ctl[CTL_AMAX_COUNT] = 0;
        if (a_bits >= 0x7F80u) {
            record_status(ctl, NVFP4_ERR_NONFINITE);
            *tensor_scale = __uint_as_float(0x7FC00000u);
        } else {
            // 2688 = 6 (largest E2M1 value) * 448 (largest E4M3 value)
            *tensor_scale = __fdiv_rn(bf16_bits_to_f32(a_bits), 2688.0f);
        }
    }
}

// ------------------------------------------------------------------ quantise
// x / S without a division: with r = RN(1/S), q0 = RN(x r) is within two ulps
// of x/S, the remainder q0 S - x is exact in one FMA, and one FMA correction
// q0 - rem r gives the correctly rounded quotient (Markstein's correction
// step, P. Markstein, IBM J. Res. Dev. 34(1), 1990).  Written so that the
// sign of a zero quotient follows x.  Used for S in [2^-96, 2^96] and
// |x / S| < 2^20 (no overflow or underflow in the steps); nvfp4_quotient_check
// compares it with IEEE division for every fp32 significand of S, every bf16
// significand of x, both signs and quotient exponents -13 .. 9, which covers
// every quotient whose E2M1 or E4M3 rounding it decides.
__device__ __forceinline__ float quotient(float x, float S, float r)
{
    const float q0 = __fmul_rn(x, r);
    const float rem = __fmaf_rn(q0, S, -x);
    return __fmaf_rn(-rem, r, q0);
}

__device__ __forceinline__ bool fast_quotient_domain(float S)
{
    return S >= 0x1p-96f && S <= 0x1p96f;
}

// Max of the eight bf16 magnitudes of a vector, as magnitude bits (packed pair).
__device__ __forceinline__ uint32_t absmax_vec2(uint4 v)
{
    const uint32_t m = 0x7FFF7FFFu;
    return __vmaxu2(__vimax3_u16x2(v.x & m, v.y & m, v.z & m), v.w & m);
}

// Four packed E2M1 bytes from eight signed quotients (element 2i in the low
// nibble of byte i); round to nearest even, saturating, sign kept (-0 -> 0x8).
__device__ __forceinline__ uint32_t e2m1x8_pack(const float q[8])
{
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return w;
}

// Codes of 8 elements (4 bf16 pairs) with block scale S > 0.
__device__ __forceinline__ uint32_t encode8(uint4 v, float S, float r, bool fast)
{
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    float q[8];
    if (fast) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            q[2 * i] = quotient(__uint_as_float(words[i] << 16), S, r);
            q[2 * i + 1] = quotient(__uint_as_float(words[i] & 0xFFFF0000u), S, r);
        }
    } else {
        // rare: scale outside the fast domain, or quotients beyond 2^20
        const float S8 = __fmul_rn(8.0f, S);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float lo = __uint_as_float(words[i] << 16);
            const float hi = __uint_as_float(words[i] & 0xFFFF0000u);
            q[2 * i] = copysignf(__fdiv_rn(fminf(fabsf(lo), S8), S), lo);
            q[2 * i + 1] = copysignf(__fdiv_rn(fminf(fabsf(hi), S8), S), hi);
        }
    }
    return e2m1x8_pack(q);
}

// Pass 2: one thread per 16-element block (two 16-byte loads).  Every block
// scale byte e has a fixed S = fl32(dec(e) s_t) and RN(1/S) for the whole
// tensor, so both are tabulated once per CTA in shared memory.  Blocks are
// visited from the end of the tensor towards the start, so that the tail
// pass 1 left in L2 is re-read first.
__global__ void __launch_bounds__(256) quantize_kernel(const uint4 *__restrict__ w, int64_t nblocks,
                                                       const float *__restrict__ tensor_scale,
                                                       uint2 *__restrict__ codes,
                                                       uint8_t *__restrict__ scales,
                                                       uint32_t *__restrict__ ctl)
{
    __shared__ float s_S[128], s_R[128];
    float s_t = *tensor_scale;
    if (!(s_t >= 0.0f && s_t <= FLT_MAX)) {  // NaN, inf or negative frozen scale
        if (blockIdx.x == 0 && threadIdx.x == 0)
            record_status(ctl, NVFP4_ERR_NONFINITE);
        s_t = 0.0f;
    }
    for (int e = threadIdx.x; e < 128; e += blockDim.x) {
        const float S = __fmul_rn(e4m3_to_f32((uint32_t)e), s_t);
        s_S[e] = S;
        s_R[e] = fast_quotient_domain(S) ? __frcp_rn(S) : 0.0f;
    }
    const float d = __fmul_rn(6.0f, s_t);
    const bool d_fast = fast_quotient_domain(d);
    const float rd = d_fast ? __frcp_rn(d) : 0.0f;
    __syncthreads();

    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t b = nblocks - 1 - ((int64_t)blockIdx.x * blockDim.x + threadIdx.x); b >= 0; b -= nthreads) {
        const uint4 v0 = ld_stream_u4(w + 2 * b);
        const uint4 v1 = ld_stream_u4(w + 2 * b + 1);
        uint32_t m = absmax8(v0, v1);
        m = max(m & 0xFFFFu, m >> 16);
        uint32_t e = 0;
        uint2 cw = make_uint2(0u, 0u);
        if (m >= 0x7F80u) {
            record_status(ctl, NVFP4_ERR_NONFINITE);
        } else if (s_t != 0.0f) {
            const float a_b = bf16_bits_to_f32(m);
            if (!d_fast)
                e = e4m3_encode_nonneg(__fdiv_rn(a_b, d));
            else if (__fmul_rn(a_b, rd) >= 1024.0f)
                e = 0x7E;  // far beyond 448: saturates
            else
                e = e4m3_encode_nonneg(quotient(a_b, d, rd));
            const float S = s_S[e];
            if (S != 0.0f) {
                const float r = s_R[e];
                const bool fast = r != 0.0f && __fmul_rn(a_b, r) < 0x1p20f;
                cw.x = encode8(v0, S, r, fast);
                cw.y = encode8(v1, S, r, fast);
            }
        }
        codes[b] = cw;
        scales[b] = (uint8_t)e;
    }
}

// ------------------------------------------------------------------ fused dynamic quantise
// Dynamic mode in one persistent cooperative kernel: pass 1 reads the block's
// contiguous share of W once for the tensor amax -- consecutive lanes on
// consecutive 16-byte vectors, six loads in flight per thread -- and keeps
// the last kFusedCacheBlocks 16-element blocks of the share in shared memory;
// its other loads ask L2 to keep their lines (evict-last), since pass 2 reads
// them again.  After one grid barrier, pass 2 quantises the share from its
// end backwards, one 16-element block per thread and two blocks in flight, so
// it starts with the blocks held in shared memory and continues with those
// pass 1 read last, which are the likeliest still to be in L2 (those loads
// are the last use: evict-first).
constexpr int kFusedThreads = 1024;
constexpr int kFusedCacheBlocks = 6144;  // 192 KB of bf16 per block
constexpr int kFusedInFlight = 6;

__device__ __forceinline__ void quantize_block(uint4 v0, uint4 v1, float s_t, float d, bool d_fast, float rd,
                                               const float *s_S, const float *s_R, uint2 &cw_out,
                                               uint32_t &e_out, uint32_t *ctl)
{
    uint32_t m = absmax8(v0, v1);
    m = max(m & 0xFFFFu, m >> 16);
    uint32_t e = 0;
    uint2 cw = make_uint2(0u, 0u);
    if (m >= 0x7F80u) {
        record_status(ctl, NVFP4_ERR_NONFINITE);
    } else if (s_t != 0.0f) {
        const float a_b = bf16_bits_to_f32(m);
        if (!d_fast)
            e = e4m3_encode_nonneg(__fdiv_rn(a_b, d));
        else if (__fmul_rn(a_b, rd) >= 1024.0f)
            e = 0x7E;
        else
            e = e4m3_encode_nonneg(quotient(a_b, d, rd));
        const float S = s_S[e];
        if (S != 0.0f) {
            const float r = s_R[e];
            const bool fast = r != 0.0f && __fmul_rn(a_b, r) < 0x1p20f;
            cw.x = encode8(v0, S, r, fast);
            cw.y = encode8(v1, S, r, fast);
        }
    }
    cw_out = cw;
    e_out = e;
}

__global__ void __launch_bounds__(kFusedThreads, 1)
    quantize_fused_kernel(const uint4 *__restrict__ w, int64_t nblocks, float *__restrict__ tensor_scale,
                          uint2 *__restrict__ codes, uint8_t *__restrict__ scales, uint32_t *__restrict__ ctl)
{
    extern __shared__ __align__(16) uint4 s_cache[];  // [kFusedCacheBlocks][2]
    __shared__ float s_S[128], s_R[128];
    __shared__ uint32_t s_m[kFusedThreads / 32];
    __shared__ bool s_last;
    const int P = gridDim.x, bid = blockIdx.x, tid = threadIdx.x;
    const int64_t b0 = (int64_t)bid * nblocks / P, b1 = (int64_t)(bid + 1) * nblocks / P;
    const int64_t cache_from = max(b0, b1 - (int64_t)kFusedCacheBlocks);

    // pass 1: amax of the share; keep its tail in shared memory
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    const int64_t v0 = 2 * b0, v1 = 2 * b1, cache_vfrom = 2 * cache_from;
    uint32_t m = 0;
    for (int64_t i = v0 + tid; i < v1; i += (int64_t)kFusedThreads * kFusedInFlight) {
        uint4 v[kFusedInFlight];
#pragma unroll
        for (int k = 0; k < kFusedInFlight; k++) {
            const int64_t ik = i + (int64_t)k * kFusedThreads;
            v[k] = ik < v1 ? ld_hint_u4(w + ik, ik >= cache_vfrom ? drop : keep) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kFusedInFlight; k++) {
            const int64_t ik = i + (int64_t)k * kFusedThreads;
            m = __vmaxu2(m, absmax_vec2(v[k]));
            if (ik >= cache_vfrom && ik < v1)
                s_cache[ik - cache_vfrom] = v[k];
        }
    }
    m = max(m & 0xFFFFu, m >> 16);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((tid & 31) == 0)
        s_m[tid >> 5] = m;
    __syncthreads();
    if (tid == 0) {
        uint32_t bm = 0;
        for (int k = 0; k < kFusedThreads / 32; k++)
            bm = max(bm, s_m[k]);
        atomicMax(&ctl[CTL_AMAX], bm);
    }
    if (!grid_barrier(ctl, P))
        return;

    // s_t = amax / 2688, identical in every block
    const uint32_t a_bits = *(volatile uint32_t *)&ctl[CTL_AMAX];
    float s_t;
    if (a_bits >= 0x7F80u) {
        if (bid == 0 && tid == 0) {
            record_status(ctl, NVFP4_ERR_NONFINITE);
            *tensor_scale = __uint_as_float(0x7FC00000u);
        }
        s_t = 0.0f;
    } else {
        s_t = __fdiv_rn(bf16_bits_to_f32(a_bits), 2688.0f);
        if (bid == 0 && tid == 0)
            *tensor_scale = s_t;
    }
    for (int e = tid; e < 128; e += kFusedThreads) {
        const float S = __fmul_rn(e4m3_to_f32((uint32_t)e), s_t);
        s_S[e] = S;
        s_R[e] = fast_quotient_domain(S) ? __frcp_rn(S) : 0.0f;
    }
    const float d = __fmul_rn(6.0f, s_t);
    const bool d_fast = fast_quotient_domain(d);
    const float rd = d_fast ? __frcp_rn(d) : 0.0f;
    __syncthreads();

    // pass 2, from the end of the share backwards.  First the tail kept in
    // shared memory (kFusedCacheBlocks is a whole number of strides, so each
    // thread's last cached block is followed by block cache_from - 1 - tid),
    // two blocks per step per thread.
    int64_t bb = b1 - 1 - tid;
    for (; bb >= cache_from; bb -= 2 * kFusedThreads) {
        const int64_t bc = bb - kFusedThreads;
        uint2 cw;
        uint32_t e;
        quantize_block(s_cache[2 * (bb - cache_from)], s_cache[2 * (bb - cache_from) + 1], s_t, d, d_fast, rd,
                       s_S, s_R, cw, e, ctl);
        codes[bb] = cw;
        scales[bb] = (uint8_t)e;
        if (bc >= cache_from) {
            quantize_block(s_cache[2 * (bc - cache_from)], s_cache[2 * (bc - cache_from) + 1], s_t, d, d_fast,
                           rd, s_S, s_R, cw, e, ctl);
            codes[bc] = cw;
            scales[bc] = (uint8_t)e;
        }
    }
    // Then the rest of the share from L2 and DRAM (read once: evict-first), two
    // blocks per step per thread; the next step's two blocks are requested
    // before this step's are quantised (up to four blocks in flight).  A block
    // before b0 is neither loaded nor quantised.
    bb = cache_from - 1 - tid;
    auto fetch = [&](int64_t b, uint4 &v0, uint4 &v1) {
        if (b >= b0) {
            v0 = ld_hint_u4(w + 2 * b, drop);
            v1 = ld_hint_u4(w + 2 * b + 1, drop);
        }
    };
    uint4 v0a = make_uint4(0u, 0u, 0u, 0u), v1a = v0a, v0b = v0a, v1b = v0a;
    uint4 n0a = v0a, n1a = v0a, n0b = v0a, n1b = v0a;
    fetch(bb, v0a, v1a);
    fetch(bb - kFusedThreads, v0b, v1b);
    for (; bb >= b0; bb -= 2 * kFusedThreads) {
        const int64_t bc = bb - kFusedThreads;
        fetch(bb - 2 * kFusedThreads, n0a, n1a);
        fetch(bc - 2 * kFusedThreads, n0b, n1b);
        uint2 cw;
        uint32_t e;
        quantize_block(v0a, v1a, s_t, d, d_fast, rd, s_S, s_R, cw, e, ctl);
        codes[bb] = cw;
        scales[bb] = (uint8_t)e;
        if (bc >= b0) {
            quantize_block(v0b, v1b, s_t, d, d_fast, rd, s_S, s_R, cw, e, ctl);
            codes[bc] = cw;
            scales[bc] = (uint8_t)e;
        }
        v0a = n0a;
        v1a = n1a;
        v0b = n0b;
        v1b = n1b;
    }

    // the last block out leaves the amax word at zero for the next call
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&ctl[CTL_AMAX_COUNT], 1u) == (uint32_t)P - 1;
        if (s_last) {
            ctl[CTL_AMAX] = 0;
            ctl[CTL_AMAX_COUNT] = 0;
        }
    }
}

// ------------------------------------------------------------------ dequantise
__global__ void __launch_bounds__(256) dequantize_kernel(const uint32_t *__restrict__ codes,
                                                         const uint8_t *__restrict__ scales,
                                                         const float *__restrict__ tensor_scale,
                                                         int64_t nhalves, void *__restrict__ out,
                                                         int out_fp32)
{
    const float s_t = *tensor_scale;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; h < nhalves; h += stride) {
        const uint32_t cw = codes[h];
        const float dec = e4m3_to_f32(scales[h >> 1]);
        uint32_t h2[4];
        e2m1x8_to_h2x4(cw, h2);
        float o[8];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            __half2 p = *reinterpret_cast<__half2 *>(&h2[i]);
            o[2 * i] = __fmul_rn(__fmul_rn(__low2float(p), dec), s_t);
            o[2 * i + 1] = __fmul_rn(__fmul_rn(__high2float(p), dec), s_t);
        }
        if (out_fp32) {
            float4 *dst = reinterpret_cast<float4 *>(out) + 2 * h;
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
        } else {
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
                p[i] = *reinterpret_cast<uint32_t *>(&b);
            }
            reinterpret_cast<uint4 *>(out)[h] = make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
}

// ------------------------------------------------------------------ scale-only update
__global__ void __launch_bounds__(256) round_scales_kernel(const float *__restrict__ param,
                                                           const float *__restrict__ tensor_scale,
                                                           int64_t n, uint8_t *__restrict__ out,
                                                           uint32_t *__restrict__ ctl)
{
    const float s_t = *tensor_scale;
    const bool st_ok = s_t >= 0.0f && s_t <= FLT_MAX;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float p = param[i];
        uint32_t e = 0;
        if (!st_ok || !(fabsf(p) <= FLT_MAX)) {
            record_status(ctl, NVFP4_ERR_NONFINITE);
        } else if (s_t != 0.0f && p > 0.0f) {
            e = e4m3_encode_nonneg(__fdiv_rn(p, s_t));
        }
        out[i] = (uint8_t)e;
    }
}

// ------------------------------------------------------------------ diagnostics
__global__ void encode_debug_kernel(const float *__restrict__ x, int64_t n, int which,
                                    uint8_t *__restrict__ out)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float v = x[i];
        uint32_t b;
        if (which == 0) {
            const float q[8] = {v, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            b = e2m1x8_pack(q) & 0xFu;
        } else {
            b = e4m3_encode_nonneg(v);
        }
        out[i] = (uint8_t)b;
    }
}

__global__ void quotient_check_kernel(uint32_t sig_lo, uint32_t sig_hi,
                                      unsigned long long *__restrict__ mismatches)
{
    const uint32_t sig = sig_lo + blockIdx.x * blockDim.x + threadIdx.x;
    if (sig >= sig_hi)
        return;
    const float S = __uint_as_float((127u << 23) | sig);  // [1, 2)
    const float r = __frcp_rn(S);
    unsigned long long bad = 0;
    for (int e = -13; e <= 9; e++)
        for (uint32_t ws = 0; ws < 256; ws++) {
            // bf16 significand (7 bits) with both signs
            const uint32_t bits = ((ws & 128u) << 24) | ((uint32_t)(127 + e) << 23) | ((ws & 127u) << 16);
            const float x = __uint_as_float(bits);
            bad += __float_as_uint(quotient(x, S, r)) != __float_as_uint(__fdiv_rn(x, S));
        }
    if (bad)
        atomicAdd(mismatches, bad);
}

// ------------------------------------------------------------------ launchers
static int grid_for(int64_t work_items, int per_block, int max_blocks)
{
    int64_t g = (work_items + per_block - 1) / per_block;
    if (g > max_blocks)
        g = max_blocks;
    return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_quantize(const void *w, int64_t N, int64_t K, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, bool given, uint32_t *ctl, cudaStream_t s,
                            const DeviceInfo &dev)
{
    const int64_t nelem = N * K;
    if (!given && dev.fused_quant_blocks > 0) {
        const uint4 *wp = reinterpret_cast<const uint4 *>(w);
        int64_t nblocks = nelem / 16;
        float *tsp = tensor_scale;
        uint2 *cp = reinterpret_cast<uint2 *>(codes);
        uint8_t *sp = scales;
        uint32_t *ctlp = ctl;
        void *args[] = {&wp, &nblocks, &tsp, &cp, &sp, &ctlp};
        return cudaLaunchCooperativeKernel((const void *)quantize_fused_kernel, dim3(dev.fused_quant_blocks),
                                           dim3(kFusedThreads), args, kFusedCacheBlocks * 32, s);
    }
    if (!given) {
        const int64_t nvec = nelem / 8;
        amax_kernel<<<grid_for(nvec, 256 * 4, dev.num_sms * 8), 256, 0, s>>>(
            reinterpret_cast<const uint4 *>(w), nvec, tensor_scale, ctl);
    }
    const int64_t nblocks = nelem / 16;
    quantize_kernel<<<grid_for(nblocks, 256, dev.num_sms * 8), 256, 0, s>>>(
        reinterpret_cast<const uint4 *>(w), nblocks, tensor_scale,
        reinterpret_cast<uint2 *>(codes), scales, ctl);
    return cudaGetLastError();
}

void query_quantize_occupancy(DeviceInfo &dev)
{
    int b = 0;
    if (cudaFuncSetAttribute(quantize_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFusedCacheBlocks * 32) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, quantize_fused_kernel, kFusedThreads,
                                                      kFusedCacheBlocks * 32) != cudaSuccess)
        b = 0;
    dev.fused_quant_blocks = b >= 1 ? dev.num_sms : 0;
}

cudaError_t launch_dequantize(const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                              int64_t N, int64_t K, void *out, bool fp32, cudaStream_t s,
                              const DeviceInfo &dev)
{
    const int64_t nhalves = N * K / 8;
    dequantize_kernel<<<grid_for(nhalves, 256, dev.num_sms * 8), 256, 0, s>>>(
        reinterpret_cast<const uint32_t *>(codes), scales, tensor_scale, nhalves, out, fp32 ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_round_scales(const float *param, const float *tensor_scale, int64_t n,
                                uint8_t *out, uint32_t *ctl, cudaStream_t s, const DeviceInfo &dev)
{
    round_scales_kernel<<<grid_for(n, 256, dev.num_sms * 8), 256, 0, s>>>(param, tensor_scale, n,
                                                                          out, ctl);
    return cudaGetLastError();
}

cudaError_t launch_encode_debug(const float *x, int64_t n, int which, uint8_t *out, cudaStream_t s,
                                const DeviceInfo &dev)
{
    encode_debug_kernel<<<grid_for(n, 256, dev.num_sms * 16), 256, 0, s>>>(x, n, which, out);
    return cudaGetLastError();
}

cudaError_t launch_quotient_check(uint32_t lo, uint32_t hi, unsigned long long *mismatches,
                                  cudaStream_t s)
{
    if (hi <= lo)
        return cudaSuccess;
    const uint32_t n = hi - lo;
    quotient_check_kernel<<<(n + 255) / 256, 256, 0, s>>>(lo, hi, mismatches);
    return cudaGetLastError();
}

}  // namespace nvfp4
